"""fp8_token_group_bf16_b300: fused FP8 per-group quantisation epilogues for B300 (sm_103a)."""
