"""ResidualKV cache-write and sparse-read path for GB300 (sm_103a)."""
