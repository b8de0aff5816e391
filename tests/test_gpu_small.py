"""GPU parity on small cases: codes bit-exact, outputs within tolerance of the
fp64 oracle, plus the layout, batching, split and error-status properties.

Tolerance (fixed for this library): max-abs 2e-3 and relative L2 1e-3 over the
compared output tensor, against the oracle's float64 result on the same
dequantised values.  Codes and scales: bit-exact record bytes.
"""
import numpy as np
import pytest
import torch

import q3kv_inputs as qi
from gpu_harness import GpuCache, check_close, oracle_records, oracle_verify, slot_kv

pytestmark = pytest.mark.gpu

IMPLS = [1, 2]   # Q3KV_IMPL_FMA, Q3KV_IMPL_MMA


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_attention_q3kv_gb300 import _lib
    _lib.load()


def _impl_or_skip(impl):
    from speculative_verify_attention_q3kv_gb300 import _lib
    w = qi.WORKLOADS[1]
    from speculative_verify_attention_q3kv_gb300 import api
    try:
        api.workspace_bytes(api.make_desc(1, 2, 8), 1, 1024, 4, impl, 256)
    except _lib.Q3KVError as e:
        if e.code == _lib.Q3KV_ERR_UNSUPPORTED:
            pytest.skip(f"impl {impl} not built")
        raise


def _small(dtype="f32", dist="outlier8", slots=3, key=1):
    base = qi.WORKLOADS[key]
    return qi.Workload(base.key, "small", 11, slots, 2, (0, 0), (0, 0), 1, dtype, dist, dist)


@pytest.mark.parametrize("impl", IMPLS)
def test_workload1_full(impl):
    _impl_or_skip(impl)
    w = qi.WORKLOADS[1]
    N, T = 1024, 4
    c = GpuCache(w, [N + T])
    k, v = slot_kv(w, 0, 0, 0, N + T)
    c.append_rows(0, [0], [0], [(k[:N], v[:N])])     # the cached context
    c.append_rows(0, [0], [N], [(k[N:], v[N:])])     # the step's 1 + 3 new tokens
    for g in range(2):
        for kv, x in ((0, k), (1, v)):
            assert np.array_equal(c.records(0, 0, g, kv, 0, N + T), oracle_records(x[:, g]))
    q = qi.q_rows(w, 0, 0, 0, T)
    out = c.verify(0, [N + T], [T], [q], impl=impl)
    check_close(out, oracle_verify(w, 0, 0, N, q, k, v))
    assert int(c.status.item()) == 0


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("dtype,dist", [("f32", "outlier8"), ("bf16", "loguniform10")])
def test_ragged_slots_with_splits(impl, dtype, dist):
    _impl_or_skip(impl)
    w = _small(dtype, dist, slots=4)
    ctx = [5, 300, 777, 1500]          # cached positions before the step
    T = [1, 4, 8, 16]                  # 8..128 query rows per kv head
    c = GpuCache(w, [n + t for n, t in zip(ctx, T)], num_layers=2)
    kvs = [slot_kv(w, b, 1, 0, ctx[b] + T[b]) for b in range(4)]
    c.append_rows(1, list(range(4)), [0] * 4, [(k[:ctx[b]], v[:ctx[b]]) for b, (k, v) in enumerate(kvs)])
    c.append_rows(1, list(range(4)), ctx, [(k[ctx[b]:], v[ctx[b]:]) for b, (k, v) in enumerate(kvs)])
    for b in range(4):
        for g in range(2):
            assert np.array_equal(c.records(b, 1, g, 0, 0, ctx[b] + T[b]), oracle_records(kvs[b][0][:, g]))
            assert np.array_equal(c.records(b, 1, g, 1, 0, ctx[b] + T[b]), oracle_records(kvs[b][1][:, g]))
    qs = [qi.q_rows(w, b, 1, 0, T[b]) for b in range(4)]
    want = np.concatenate([oracle_verify(w, b, 1, ctx[b], qs[b], *kvs[b]) for b in range(4)])
    for split in (256, 512, 0):
        out = c.verify(1, [n + t for n, t in zip(ctx, T)], T, qs, impl=impl, split_positions=split)
        check_close(out, want)
    assert int(c.status.item()) == 0


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("split", [0, 256])
def test_outlier_heavy_queries_and_cache_verify_shapes(impl, split):
    """Verify widths 6..16 over 4K+ positions; queries and cache both with 10x channels."""
    _impl_or_skip(impl)
    w = _small("bf16", "loguniform10", slots=3)
    ctx, T = [4096, 6000, 4500], [6, 11, 16]
    L = [n + t for n, t in zip(ctx, T)]
    c = GpuCache(w, L, num_layers=1)
    kvs = [slot_kv(w, b, 0, 0, L[b]) for b in range(3)]
    c.append_rows(0, [0, 1, 2], [0, 0, 0], kvs)
    qs = [qi.q_rows(w, b, 0, 0, T[b]) for b in range(3)]
    want = np.concatenate([oracle_verify(w, b, 0, ctx[b], qs[b], *kvs[b]) for b in range(3)])
    out = c.verify(0, L, T, qs, impl=impl, split_positions=split)
    check_close(out, want)
    assert int(c.status.item()) == 0


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("split", [0, 256])
def test_score_jump_around_the_lagged_maximum_threshold(impl, split):
    """One late key whose score for query row (token 0, head 0) exceeds every earlier score by
    delta log2 units, per slot delta from 4 to 20: around 14 the tensor-core leg either keeps
    its running maximum (P up to 2^14 in the fp16 hi/lo split) or rescales; both must hold."""
    _impl_or_skip(impl)
    deltas = [4.0, 12.0, 13.5, 13.9, 14.1, 14.5, 16.0, 20.0]
    S, N, T = len(deltas), 1000, 4
    w = _small("f32", "outlier8", slots=S)
    L = [N + T] * S
    c = GpuCache(w, L, num_layers=1)
    kvs, qs = [], []
    log2e = 1.4426950408889634
    for b, delta in enumerate(deltas):
        k, v = slot_kv(w, b, 0, 0, N + T)
        q = qi.q_rows(w, b, 0, 0, T)
        p_star = N - 50                              # in the context's last tile
        u = q[0, 0].astype(np.float64)
        prev = float(np.max(k[:p_star, 0].astype(np.float64) @ u)) / 16.0 * log2e
        scale = (prev + delta) * 16.0 / (log2e * float(u @ u))
        k = k.copy()
        k[p_star, 0] = (scale * u).astype(np.float32)
        kvs.append((k, v))
        qs.append(q)
    c.append_rows(0, list(range(S)), [0] * S, kvs)
    want = np.concatenate([oracle_verify(w, b, 0, N, qs[b], *kvs[b]) for b in range(S)])
    out = c.verify(0, L, [T] * S, qs, impl=impl, split_positions=split)
    check_close(out, want)
    assert int(c.status.item()) == 0


@pytest.mark.parametrize("impl", IMPLS)
def test_batched_equals_solo_bitwise(impl):
    _impl_or_skip(impl)
    w = _small("bf16", "loguniform10", slots=3)
    ctx, T = [600, 41, 1300], [6, 3, 8]
    L = [n + t for n, t in zip(ctx, T)]
    c = GpuCache(w, L, num_layers=1)
    kvs = [slot_kv(w, b, 0, 0, L[b]) for b in range(3)]
    c.append_rows(0, [0, 1, 2], [0, 0, 0], kvs)
    qs = [qi.q_rows(w, b, 0, 0, T[b]) for b in range(3)]
    batched = c.verify(0, L, T, qs, impl=impl, split_positions=512)
    rows = np.concatenate([[0], np.cumsum(T)])
    for b in range(3):
        solo_ctx = [0, 0, 0]
        solo_T = [0, 0, 0]
        solo_ctx[b], solo_T[b] = L[b], T[b]
        solo_q = [qs[i] if i == b else np.zeros((0, 16, 256), np.float32) for i in range(3)]
        solo = c.verify(0, solo_ctx, solo_T, solo_q, impl=impl, split_positions=512)
        assert np.array_equal(solo, batched[rows[b]:rows[b + 1]])


@pytest.mark.parametrize("impl", IMPLS)
def test_paged_equals_contiguous_bitwise(impl):
    _impl_or_skip(impl)
    w = _small("f32", "outlier8", slots=2)
    L, T = [900, 513], [5, 2]
    outs, recs = [], []
    for contiguous in (False, True):
        c = GpuCache(w, L, num_layers=1, extra_pages=3, contiguous=contiguous)
        kvs = [slot_kv(w, b, 0, 0, L[b]) for b in range(2)]
        c.append_rows(0, [0, 1], [0, 0], kvs)
        qs = [qi.q_rows(w, b, 0, 0, T[b]) for b in range(2)]
        outs.append(c.verify(0, L, T, qs, impl=impl, split_positions=256))
        recs.append([c.records(b, 0, g, kv, 0, L[b]) for b in range(2) for g in range(2) for kv in range(2)])
    assert np.array_equal(outs[0], outs[1])
    for a, b in zip(*recs):
        assert np.array_equal(a, b)


def test_rollback_overwrites():
    w = _small("f32", "outlier8", slots=1)
    c = GpuCache(w, [20], num_layers=1)
    k, v = slot_kv(w, 0, 0, 0, 13)
    c.append_rows(0, [0], [0], [(k, v)])
    # drafts at 8..12 rejected; three different tokens appended at 8..10
    rng = np.random.default_rng(0)
    k2 = rng.standard_normal((3, 2, 256)).astype(np.float32)
    v2 = rng.standard_normal((3, 2, 256)).astype(np.float32)
    c.append_rows(0, [0], [8], [(k2, v2)])
    kk = np.concatenate([k[:8], k2])
    vv = np.concatenate([v[:8], v2])
    for g in range(2):
        assert np.array_equal(c.records(0, 0, g, 0, 0, 11), oracle_records(kk[:, g]))
        assert np.array_equal(c.records(0, 0, g, 1, 0, 11), oracle_records(vv[:, g]))
    q = qi.q_rows(w, 0, 0, 0, 3)
    out = c.verify(0, [11], [3], [q], impl=1)
    check_close(out, oracle_verify(w, 0, 0, 8, q, kk, vv))


def test_status_bad_page_and_length():
    w = _small("f32", "outlier8", slots=1)
    c = GpuCache(w, [300], num_layers=1)
    k, v = slot_kv(w, 0, 0, 0, 300)
    c.append_rows(0, [0], [0], [(k, v)])
    assert int(c.status.item()) == 0
    # a page id beyond the pool: the verify skips it and flags BAD_PAGE
    c.page_table[0, 1] = c.num_pages + 5
    c.page_table_np[0, 1] = c.num_pages + 5
    q = qi.q_rows(w, 0, 0, 0, 2)
    c.verify(0, [300], [2], [q], impl=1, split_positions=256)
    assert int(c.status.item()) & 4
    # an append into that page is skipped and flagged too
    c.status.zero_()
    c.append_rows(0, [0], [290], [(k[:2], v[:2])])
    assert int(c.status.item()) & 4
    # a context longer than the page table: BAD_LENGTH, output untouched (NaN fill stays)
    c.status.zero_()
    out = c.verify(0, [c.page_table_np.shape[1] * 256 + 1], [2], [q], impl=1, split_positions=256)
    assert int(c.status.item()) & 8
    assert np.all(np.isnan(out))
    # more query tokens than positions: BAD_LENGTH
    c.status.zero_()
    c.verify(0, [1], [2], [q], impl=1, split_positions=256)
    assert int(c.status.item()) & 8


def test_status_nonfinite_and_overflow():
    w = _small("f32", "outlier8", slots=1)
    c = GpuCache(w, [4], num_layers=1)
    k = np.zeros((2, 2, 256), np.float32)
    v = np.zeros((2, 2, 256), np.float32)
    k[0, 0, 3] = np.nan
    c.append_rows(0, [0], [0], [(k, v)])
    assert int(c.status.item()) == 1
    c.status.zero_()
    k[0, 0, 3] = 0.0
    v[1, 1, 0] = 4.0e6
    c.append_rows(0, [0], [0], [(k, v)])
    assert int(c.status.item()) == 2


@pytest.mark.parametrize("scale_value,flagged", [(4.0e5, True), (1.0e5, False)])
def test_status_range_of_the_tensor_core_leg(scale_value, flagged):
    """A block scale above 65504 / 12 (one input channel at 4e5 rotates to 25,000 in every dim:
    s = 7,143) is flagged by the tensor-core leg and read by the CUDA-core leg; 1e5 (s = 1,786)
    is read by both."""
    w = _small("f32", "outlier8", slots=1)
    N, T = 40, 2
    c = GpuCache(w, [N + T], num_layers=1)
    k, v = slot_kv(w, 0, 0, 0, N + T)
    k[5, 1, 17] = scale_value
    c.append_rows(0, [0], [0], [(k, v)])
    assert int(c.status.item()) == 0
    q = qi.q_rows(w, 0, 0, 0, T)
    want = oracle_verify(w, 0, 0, N, q, k, v)
    check_close(c.verify(0, [N + T], [T], [q], impl=1), want)
    assert int(c.status.item()) == 0
    out = c.verify(0, [N + T], [T], [q], impl=2)
    if flagged:
        assert int(c.status.item()) & 32
    else:
        assert int(c.status.item()) == 0
        check_close(out, want)


def test_empty_calls():
    w = _small("f32", "outlier8", slots=2)
    c = GpuCache(w, [10, 10], num_layers=1)
    # no new tokens anywhere: nothing happens
    c.append_rows(0, [0, 1], [0, 0], [(np.zeros((0, 2, 256), np.float32),) * 2] * 2)
    assert int(c.status.item()) == 0
    # one slot with no query tokens, the other with one
    k, v = slot_kv(w, 1, 0, 0, 10)
    c.append_rows(0, [1], [0], [(k, v)])
    q = qi.q_rows(w, 1, 0, 0, 1)
    out = c.verify(0, [0, 10], [0, 1], [np.zeros((0, 16, 256), np.float32), q], impl=1)
    check_close(out, oracle_verify(w, 1, 0, 9, q, k, v))


@pytest.mark.parametrize("impl", IMPLS)
def test_merge_beyond_preloaded_split_rows(impl):
    """256-position splits over ~30K positions: 120 splits per unit (the merge preloads 96)."""
    _impl_or_skip(impl)
    w = _small("bf16", "loguniform10", slots=1)
    N, T = 30_700, 3
    c = GpuCache(w, [N + T], num_layers=1)
    k, v = slot_kv(w, 0, 0, 0, N + T)
    c.append_rows(0, [0], [0], [(k, v)])
    q = qi.q_rows(w, 0, 0, 0, T)
    out = c.verify(0, [N + T], [T], [q], impl=impl, split_positions=256)
    check_close(out, oracle_verify(w, 0, 0, N, q, k, v))
    assert int(c.status.item()) == 0


@pytest.mark.parametrize("impl", IMPLS)
def test_merge_beyond_one_weight_chunk(impl):
    """2,050 splits of 256 positions (the merge stages 2,048 split weights at a time).

    Every page holds the same 256 K/V vectors and the context is a whole number
    of pages, so each position's weight appears 2,050 times and the attention
    equals that of the single page (the oracle over one page).
    """
    _impl_or_skip(impl)
    from speculative_verify_attention_q3kv_gb300 import api
    w = qi.Workload(1, "repeat", 13, 1, 1, (0, 0), (0, 0), 1, "bf16", "outlier8", "outlier8",
                    num_kv_heads=1, num_q_heads=8)
    pages = 2050
    L, T = pages * 256, 1
    c = GpuCache(w, [L], num_layers=1)
    k1, v1 = slot_kv(w, 0, 0, 0, 256)
    dt = torch.bfloat16
    kd = torch.from_numpy(k1).to(dt).cuda().repeat(pages, 1, 1)
    vd = torch.from_numpy(v1).to(dt).cuda().repeat(pages, 1, 1)
    zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.append(c.desc, c.pool, c.page_table, zero, torch.tensor([L], dtype=torch.int32).cuda(),
               torch.tensor([0, L], dtype=torch.int32).cuda(), L, 0, kd, vd, c.status)
    q = qi.q_rows(w, 0, 0, 0, T)
    out = c.verify(0, [L], [T], [q], impl=impl, split_positions=256)
    check_close(out, oracle_verify(w, 0, 0, 256 - T, q, k1, v1))
    assert int(c.status.item()) == 0
