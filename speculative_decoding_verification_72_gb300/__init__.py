"""GB300 (sm_103a) library for batched speculative-decoding verification."""
