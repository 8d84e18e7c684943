"""GB300-native FP8 / BF16 causal prefill FlashAttention (placeholder binding)."""
