"""libcsa2: the CSA2 long-context attention step (FP4 KV cache, lightning indexer,
top-k, sparse MLA-style attention) as hand-written CUDA for sm_103a behind a
C ABI, with a thin ctypes binding."""
