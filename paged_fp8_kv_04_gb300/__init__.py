"""GB300-native paged decode attention over an FP8 (e4m3) KV cache."""
