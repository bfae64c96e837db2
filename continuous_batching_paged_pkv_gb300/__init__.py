"""Paged-KV attention step for continuous batching, native to GB300 (sm_103a)."""
