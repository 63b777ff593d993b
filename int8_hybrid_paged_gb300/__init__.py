"""GB300-native KV4-RL decode hot path: paged INT4 KV cache with a bounded INT8 side cache."""
