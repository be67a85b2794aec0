"""GB300-native quantized paged KV-cache decode attention (INT4 + TurboQuant FP8 layouts)."""
