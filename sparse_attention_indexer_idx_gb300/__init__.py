"""GB300-native sparse-attention indexer hot path.

libidx.so (CUDA kernels for sm_103a behind a C ABI, include/idx.h) computes the
DSA indexer score and its exact top-K, DoSA safe-upper-bound pruning, the
segment-witness covering merge and MiniMax block-max selection.  `binding`
is the thin ctypes layer over it; `workloads` makes seeded synthetic inputs.
"""
