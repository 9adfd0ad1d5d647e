"""paged_kv_gqa_block_gb300: single-token paged-KV GQA decode attention for GB300 (sm_103a)."""
