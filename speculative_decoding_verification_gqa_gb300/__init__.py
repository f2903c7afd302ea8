"""GB300-native speculative-decoding verification: GQA verify attention and greedy
acceptance as hand-written sm_103a CUDA kernels behind a C ABI (libspecverify.so)."""
