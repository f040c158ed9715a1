"""Batched paged-KV decode attention for GB300 (sm_103a)."""
