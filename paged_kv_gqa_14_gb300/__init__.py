"""paged_kv_gqa_14_gb300: paged grouped-query attention and fused RoPE-and-append for GB300."""
