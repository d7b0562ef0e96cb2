"""GB300-native Gated DeltaNet causal core (placeholder; filled in with the CUDA binding)."""
