"""FlashAttention forward (prefill + paged decode) for GB300."""
