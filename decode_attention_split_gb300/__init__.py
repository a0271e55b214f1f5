"""GB300-native split-KV decode attention (placeholder; the binding is added with the CUDA library)."""
