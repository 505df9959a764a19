"""GB300-native bf16 allreduce over R virtual ranks held as HBM buffers."""
