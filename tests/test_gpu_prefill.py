"""GPU parity of prefill attention over the 3-bit cache (q3kv_prefill_attn).

A prefill is the verify step with many new tokens: the oracle is the same
float64 causal attention (``oracle.attention.verify_attention``), the tolerance
the same max-abs 2e-3 / relative L2 1e-3.  Cases: a fresh prefill, a prefill
onto an existing context, ragged slots mixing prefill and verify widths, and
the token bound of each call.

Every case, on both legs, is held to the same max-abs 2e-3 / relative L2
1e-3, including queries and cache that both carry 10x outlier channels (the
inputs with the largest scores, where the tensor-core leg's dropped lo.lo
product of the key contraction matters most).  At the call's bound of 8,192
new tokens the oracle computes sampled query tokens one by one.
"""
import numpy as np
import pytest
import torch

import q3kv_inputs as qi
from gpu_harness import GpuCache, check_close, oracle_verify, slot_kv, tdtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_attention_q3kv_gb300 import _lib
    _lib.load()


def _prefill(c, layer, ctx_len, n_new, q_rows, impl=0, split_positions=0):
    from speculative_verify_attention_q3kv_gb300 import api
    w = c.w
    offs = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    q = torch.from_numpy(np.concatenate(q_rows)).to(tdtype(w)).cuda()
    out = torch.full((q.shape[0], w.num_q_heads, 256), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = api.prefill_workspace_bytes(c.desc, w.num_slots, max(ctx_len), max(n_new), impl, split_positions)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    api.prefill_attn(c.desc, c.pool, c.page_table, torch.tensor(np.asarray(ctx_len, np.int32)).cuda(),
                     torch.tensor(np.asarray(n_new, np.int32)).cuda(), torch.from_numpy(offs).cuda(), max(ctx_len),
                     max(n_new), layer, q, out, ws, impl, split_positions, c.status)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _small(dtype, dist, slots):
    base = qi.WORKLOADS[1]
    return qi.Workload(base.key, "small", 17, slots, 2, (0, 0), (0, 0), 1, dtype, dist, dist)


@pytest.mark.parametrize("impl,dtype,dist", [(1, "bf16", "loguniform10"), (2, "f32", "outlier8"),
                                             (2, "bf16", "outlier8")])
def test_fresh_prefill(impl, dtype, dist):
    w = _small(dtype, dist, 1)
    T = 300
    c = GpuCache(w, [T])
    k, v = slot_kv(w, 0, 0, 0, T)
    c.append_rows(0, [0], [0], [(k, v)])
    q = qi.q_rows(w, 0, 0, 0, T)
    got = _prefill(c, 0, [T], [T], [q], impl=impl)
    check_close(got, oracle_verify(w, 0, 0, 0, q, k, v))
    assert int(c.status.item()) == 0


def test_prefill_onto_context():
    w = _small("f32", "outlier8", 1)
    N, T = 700, 1000
    c = GpuCache(w, [N + T])
    k, v = slot_kv(w, 0, 0, 0, N + T)
    c.append_rows(0, [0], [0], [(k[:N], v[:N])])
    c.append_rows(0, [0], [N], [(k[N:], v[N:])])
    q = qi.q_rows(w, 0, 0, 0, T)
    got = _prefill(c, 0, [N + T], [T], [q], impl=2)
    check_close(got, oracle_verify(w, 0, 0, N, q, k, v))
    assert int(c.status.item()) == 0


@pytest.mark.parametrize("split", [0, 256])
def test_ragged_prefill_and_verify_widths(split):
    w = _small("bf16", "outlier8", 3)
    ctx = [0, 256, 1000]
    T = [64, 129, 8]
    c = GpuCache(w, [n + t for n, t in zip(ctx, T)], num_layers=2)
    kvs = [slot_kv(w, b, 1, 0, ctx[b] + T[b]) for b in range(3)]
    c.append_rows(1, [1, 2], [0, 0], [(kvs[b][0][:ctx[b]], kvs[b][1][:ctx[b]]) for b in (1, 2)])
    c.append_rows(1, [0, 1, 2], ctx, [(k[ctx[b]:], v[ctx[b]:]) for b, (k, v) in enumerate(kvs)])
    qs = [qi.q_rows(w, b, 1, 0, T[b]) for b in range(3)]
    want = np.concatenate([oracle_verify(w, b, 1, ctx[b], qs[b], *kvs[b]) for b in range(3)])
    got = _prefill(c, 1, [n + t for n, t in zip(ctx, T)], T, qs, impl=2, split_positions=split)
    check_close(got, want)
    assert int(c.status.item()) == 0


def test_token_bounds():
    from speculative_verify_attention_q3kv_gb300 import _lib, api
    d = api.make_desc(1, 2, 64)
    assert api.prefill_workspace_bytes(d, 1, 8192, 8192, 2) > 0
    with pytest.raises(_lib.Q3KVError):
        api.prefill_workspace_bytes(d, 1, 9000, 8193, 2)
    with pytest.raises(_lib.Q3KVError):
        api.workspace_bytes(d, 1, 1000, 17, 2)            # the verify call keeps its 16-token bound


@pytest.mark.parametrize("impl", [1, 2])
def test_outlier_heavy_queries_and_cache(impl):
    w = _small("bf16", "loguniform10", 1)
    T = 300
    c = GpuCache(w, [T])
    k, v = slot_kv(w, 0, 0, 0, T)
    c.append_rows(0, [0], [0], [(k, v)])
    q = qi.q_rows(w, 0, 0, 0, T)
    got = _prefill(c, 0, [T], [T], [q], impl=impl)
    check_close(got, oracle_verify(w, 0, 0, 0, q, k, v))
    assert int(c.status.item()) == 0


@pytest.mark.parametrize("impl,dist", [(0, "loguniform10"), (2, "outlier8")])
def test_prefill_at_the_token_bound_sampled_rows(impl, dist):
    """8,192 new tokens (the call's bound) onto 700 cached positions; sampled tokens checked."""
    from oracle.attention import verify_attention
    from oracle.cache import encode_dequantized
    w = _small("bf16", dist, 1)
    N, T = 700, 8192
    c = GpuCache(w, [N + T])
    k, v = slot_kv(w, 0, 0, 0, N + T)
    c.append_rows(0, [0], [0], [(k[:N], v[:N])])
    c.append_rows(0, [0], [N], [(k[N:], v[N:])])
    q = qi.q_rows(w, 0, 0, 0, T)
    got = _prefill(c, 0, [N + T], [T], [q], impl=impl)
    assert int(c.status.item()) == 0
    assert np.all(np.isfinite(got))
    kh = np.stack([encode_dequantized(k[:, g]) for g in range(w.num_kv_heads)])
    vh = np.stack([encode_dequantized(v[:, g]) for g in range(w.num_kv_heads)])
    ts = [0, 1, 7, 8, 63, 64, 1000, 4095, 4096, 6001, 8190, 8191]
    want = np.concatenate([verify_attention(q[t:t + 1], kh[:, :N + t + 1], vh[:, :N + t + 1], N + t, w.group)
                           for t in ts])
    check_close(got[ts], want)
