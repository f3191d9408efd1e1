"""attnfuse-gb300: fused RoPE + variant attention for GB300 (sm_103a)."""
