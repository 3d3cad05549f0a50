"""GB300-native quantization-aware attention (QAT attention)."""
