"""CPU oracle for the q3kv verify step -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the hot path computes:

* ``wht``       -- the Walsh-Hadamard rotation of K, V and Q head vectors;
* ``codec``     -- the 3-bit block codec (fp16 absmax/3.5 scale, round-half-even codes);
* ``packing``   -- the byte layout of a coded vector and of a cache page;
* ``attention`` -- multi-token causal verify attention in float64 over the
                   exactly dequantised values, GQA group by group;
* ``cache``     -- an oracle-side paged cache: append and read back;
* ``accept``    -- greedy acceptance of a verify step's drafts and the commit
                   (rollback) of the cache length;
* ``fp8``       -- the fp8 E4M3 comparison format (saturating, unscaled,
                   unrotated), its paged cache and plain-basis attention;
* ``turbo5k``   -- the turbo5k-style cache: 5-bit Lloyd-Max K (root-mean-square
                   scale per 128 dims) with the 3-bit V, its paged cache.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never imports, links or runs anything here, and nothing here imports
the product.

Source: the "Quasar" (q27) engine wiki -- "turbo3 3-bit KV cache" and
"Self-speculation as the whole design" bullets, and the "KV cache" bullet of the
stack list (WHT-rotated 3-bit blocks, symmetric K+V, one shared-KV verify).  The
pages give no bit-level codec; the codec here is this library's stated one
(head_dim 256, fp32 Walsh-Hadamard rotation, 32-element blocks, fp16 scale
absmax/3.5, codes clamp(rint(x/s + 3.5), 0, 7), 112 bytes per vector).

Parity status: every function is pinned by tests under ``tests/`` against
closed forms, brute force, library routines and hand-derived examples.  The
codec as a whole is *parity unpinned* against the pages' own turbo3 format,
which the pages never specify bit by bit.
"""
