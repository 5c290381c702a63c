"""QUOKA per-chunk KV selection plus sparse attention on GB300 (sm_103a).

The compute path is the C-ABI library ``libquoka.so`` (CUDA kernels); the
Python side only marshals tensors into it.  Import the binding with
``from sparse_attention_chunked_gb300 import quoka``.
"""
