"""GB300-native chunkwise Gated DeltaNet prefill (placeholder, binding added with the C-ABI)."""
