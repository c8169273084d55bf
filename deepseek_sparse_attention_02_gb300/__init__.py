"""DeepSeek Sparse Attention decode hot path for GB300 (sm_103a).

The compute lives in libdsa.so (CUDA kernels behind the C ABI of
include/dsa.h); ``deepseek_sparse_attention_02_gb300.dsa`` is its Python
binding and ``deepseek_sparse_attention_02_gb300.workloads`` the seeded input
generators.  Nothing is imported eagerly so the generators stay usable on a
machine without the built library.
"""
