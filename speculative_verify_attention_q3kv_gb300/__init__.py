"""q3kv: speculative-verify attention over a 3-bit, Hadamard-rotated, paged KV
cache, as hand-written CUDA for sm_103a behind a small C ABI (``include/q3kv.h``).

Python surface (argument marshalling only):
  api.make_desc, api.pool_bytes, api.workspace_bytes, api.Allocator,
  api.append, api.verify_attn
The CUDA library is built in-tree by ``build.build()``; nothing here falls back
to another implementation when it is missing.
"""
__all__ = ["api", "build"]
