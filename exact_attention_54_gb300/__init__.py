"""GB300-native exact attention (FlashAttention-2 forward, varlen, split-KV decode)."""
