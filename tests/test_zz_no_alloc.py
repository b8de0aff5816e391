"""The fixed-scratch verify entry point (q3kv_verify_attn_noalloc).

It serves callers that cannot hand the library a device workspace; it must
give the same results as q3kv_verify_attn with a caller workspace, on
consecutive calls that reuse (and so inherit the contents of) its scratch.
This file is collected last on purpose, and also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import q3kv_inputs as qi
from gpu_harness import GpuCache, slot_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_attention_q3kv_gb300 import _lib
    return _lib.load()


def _case(seed):
    w = qi.Workload(2, "noalloc", seed, 3, 2, (0, 0), (0, 0), 1, "bf16", "loguniform10", "normal")
    ctx, T = [3000, 700, 5000], [6, 3, 8]
    L = [n + t for n, t in zip(ctx, T)]
    c = GpuCache(w, L)
    kvs = [slot_kv(w, b, 1, 0, L[b]) for b in range(3)]
    c.append_rows(1, [0, 1, 2], [0, 0, 0], kvs)
    return w, c, L, T


def _call_noalloc(lib, c, L, T, q, impl, split):
    from speculative_verify_attention_q3kv_gb300 import _lib
    # keep every device argument referenced until the call has run
    offs = torch.tensor(np.concatenate([[0], np.cumsum(T)]).astype(np.int32)).cuda()
    ctx_len = torch.tensor(L, dtype=torch.int32).cuda()
    n_q = torch.tensor(T, dtype=torch.int32).cuda()
    out = torch.full((q.shape[0], 16, 256), float("nan"), dtype=torch.float32, device="cuda")
    rc = lib.q3kv_verify_attn_noalloc(
        torch.cuda.current_stream().cuda_stream, ctypes.byref(c.desc), c.pool.data_ptr(), c.page_table.data_ptr(),
        c.page_table.shape[1], ctx_len.data_ptr(), n_q.data_ptr(), offs.data_ptr(), 3, max(L), max(T), 1,
        q.data_ptr(), _lib.Q3KV_BF16, out.data_ptr(), impl, split, c.status.data_ptr())
    torch.cuda.synchronize()
    assert rc == 0, _lib.strerror(rc)
    return out.cpu().numpy()


@pytest.mark.parametrize("impl,split", [(2, 512), (1, 512), (0, 0)])
def test_noalloc_matches_workspace_call_twice(lib, impl, split):
    """Same kernels on the same inputs: the two calls must agree bit for bit.

    (0, 0) is the default a caller uses: automatic leg and split policy.
    """
    w, c, L, T = _case(21)
    for call in range(2):                       # the second call inherits the first call's scratch
        qs = [qi.q_rows(w, b, 1, call, T[b]) for b in range(3)]
        want = c.verify(1, L, T, qs, impl=impl, split_positions=split)     # caller workspace
        qd = torch.from_numpy(np.concatenate(qs)).to(torch.bfloat16).cuda()
        got = _call_noalloc(lib, c, L, T, qd, impl, split)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, want)
    assert int(c.status.item()) == 0


def test_noalloc_rejects_oversized_scratch(lib):
    from speculative_verify_attention_q3kv_gb300 import _lib, api
    d = api.make_desc(1, 2, 4)
    # 64 slots x 2 heads x 2 row chunks x 2561 splits of partials is far beyond the fixed scratch
    need = api.workspace_bytes(d, 64, 655360, 16, 2, 256)
    assert need > _lib.Q3KV_NOALLOC_SCRATCH_BYTES
    args = [None, ctypes.byref(d), 16, 16, 4, 16, 16, 16, 64, 655360, 16, 0, 16, _lib.Q3KV_BF16, 16, 2, 256, None]
    assert lib.q3kv_verify_attn_noalloc(*args) == _lib.Q3KV_ERR_WORKSPACE_TOO_SMALL
