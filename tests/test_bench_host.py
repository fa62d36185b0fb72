"""Host-side logic of bench.py on CPU: the counting rules behind the roofline figures, the
comment-insensitive source hash that gates the committed DRAM traffic, and the reference arm on
the decode workload."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gated_deltanet_chunkwise_gdn_gb300 import workloads as wl  # noqa: E402


def test_decode_algorithmic_bytes_are_states_plus_inputs():
    w = wl.BY_NAME["decode"]
    lengths = wl.sequence_lengths(w)
    acct = bench.kernel_accounting(w, lengths)
    B = len(lengths)
    states = B * w.HV * w.V * w.K * 4 * 2                  # each state read and written once, fp32
    inputs = B * (2 * w.H * w.K * 2 + 2 * w.HV * w.V * 2 + 2 * w.HV * 4)  # q, k; v, o; a, b
    assert acct["decode"]["bytes"] == states + inputs == 1080098816
    assert set(acct) == {"decode", "path"}


def test_long_prefill_path_bytes_per_token_head():
    """1032 B per token-head at K = V = 128 (q, k, v, o, a, b), plus the one state read and written."""
    w = wl.BY_NAME["long"]
    lengths = wl.sequence_lengths(w)
    acct = bench.kernel_accounting(w, lengths)
    T = sum(lengths)
    per_token = 2 * w.H * w.K * 2 + 2 * w.HV * w.V * 2 + 8 * w.HV
    assert per_token / w.HV == 1032
    assert acct["path"]["bytes"] == T * per_token + w.HV * w.V * w.K * 8


def test_source_hash_ignores_comments_and_whitespace():
    a = "int f(int x) {  // one\n  return x + 1; /* two */ }\n"
    b = "int f(int x){return x+1;}  // other words\n"
    c = 'int f(int x) { return x + 2; }'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only('char* s = "// kept";') == 'char*s="// kept";'


def test_committed_traffic_is_reported_only_for_the_sources_it_was_taken_on():
    """A committed DRAM figure is reported while its kernel's code hash matches, else null."""
    tab = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    for workload, kernels in tab.items():
        for kernel, ent in kernels.items():
            got = bench.measured_traffic(kernel, workload)
            if ent["source_hash"] == bench.kernel_source_hash(kernel):
                assert got == ent["dram_bytes_per_launch"], (workload, kernel)
            else:
                assert got is None, (workload, kernel)


@pytest.mark.timeout(300)
def test_reference_arm_on_the_decode_workload():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "decode",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert "decode" in line["metric"] and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
