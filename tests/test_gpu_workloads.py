"""GPU parity at the five workloads' full sizes, in the launch configuration the
benchmark uses (default implementation, library split policy).

Each test populates sampled layers of the workload with the seeded inputs,
checks the stored records bit for bit against the oracle's encoding (every
position of the sampled units, or sampled pages of the 655,360-position one)
and the verify outputs against the oracle's float64 attention within max-abs
2e-3 / relative L2 1e-3.  The oracle re-encodes each sampled unit from the raw
inputs itself; nothing it compares with comes from the CUDA path.
"""
import numpy as np
import pytest
import torch

import q3kv_inputs as qi
from gpu_harness import GpuCache, check_close, oracle_records, oracle_verify, slot_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _prefill_and_step(c, w, layer, slots, ctx, T, chunk=65536):
    """Append positions [0, ctx) then the step's T tokens, per slot; returns raw K, V per slot."""
    kvs = [slot_kv(w, b, layer, 0, ctx[b] + T[b]) for b in slots]
    starts = {b: 0 for b in slots}
    while True:
        rows, idx, st = [], [], []
        for i, b in enumerate(slots):
            n = min(chunk, ctx[b] - starts[b])
            if n > 0:
                k, v = kvs[i]
                rows.append((k[starts[b]:starts[b] + n], v[starts[b]:starts[b] + n]))
                idx.append(b)
                st.append(starts[b])
                starts[b] += n
        if not rows:
            break
        c.append_rows(layer, idx, st, rows)
    c.append_rows(layer, list(slots), [ctx[b] for b in slots],
                  [(kvs[i][0][ctx[b]:], kvs[i][1][ctx[b]:]) for i, b in enumerate(slots)])
    return kvs


def _check_unit_records(c, w, b, layer, k, v, positions=None):
    for g in range(w.num_kv_heads):
        for kv, x in ((0, k), (1, v)):
            if positions is None:
                got = c.records(b, layer, g, kv, 0, x.shape[0])
                assert np.array_equal(got, oracle_records(x[:, g])), (b, layer, g, kv)
            else:
                for p0, n in positions:
                    got = c.records(b, layer, g, kv, p0, n)
                    assert np.array_equal(got, oracle_records(x[p0:p0 + n, g])), (b, layer, g, kv, p0)


def test_workload2_layers_0_and_15():
    w = qi.WORKLOADS[2]
    sh = qi.draw_shapes(w)
    ctx, T = sh.ctx, sh.n_new[0]
    c = GpuCache(w, [ctx[0] + T[0]], contiguous=True)
    for layer in (0, 15):
        (k, v), = _prefill_and_step(c, w, layer, [0], ctx, T)
        _check_unit_records(c, w, 0, layer, k, v)
        q = qi.q_rows(w, 0, layer, 0, T[0])
        out = c.verify(layer, [ctx[0] + T[0]], T, [q])
        check_close(out, oracle_verify(w, 0, layer, ctx[0], q, k, v))
    assert int(c.status.item()) == 0


def test_workload3_ragged_slots_layer_7():
    w = qi.WORKLOADS[3]
    sh = qi.draw_shapes(w)
    ctx, T = sh.ctx, sh.n_new[0]
    c = GpuCache(w, [n + t for n, t in zip(ctx, T)])
    layer = 7
    kvs = _prefill_and_step(c, w, layer, list(range(w.num_slots)), ctx, T)
    qs = [qi.q_rows(w, b, layer, 0, T[b]) for b in range(w.num_slots)]
    out = c.verify(layer, [n + t for n, t in zip(ctx, T)], T, qs)
    want = np.concatenate([oracle_verify(w, b, layer, ctx[b], qs[b], *kvs[b]) for b in range(w.num_slots)])
    check_close(out, want)
    for b in range(w.num_slots):
        k, v = kvs[b]
        pages = [(p0, 256) for p0 in range(0, ctx[b] - 256, 256 * 37)] + [(ctx[b] + T[b] - 40, 40)]
        _check_unit_records(c, w, b, layer, k, v, pages)
    assert int(c.status.item()) == 0


def test_workload4_continuous_batching_layer_3():
    w = qi.WORKLOADS[4]
    sh = qi.draw_shapes(w)
    layer = 3
    total = [sh.ctx[b] + sum(sh.n_new[s][b] for s in range(w.steps)) for b in range(w.num_slots)]
    c = GpuCache(w, total)
    S = w.num_slots
    kall = [slot_kv(w, b, layer, 0, total[b]) for b in range(S)]
    # prefill the starting contexts
    c.append_rows(layer, list(range(S)), [0] * S, [(kall[b][0][:sh.ctx[b]], kall[b][1][:sh.ctx[b]]) for b in range(S)])
    lens = list(sh.ctx)
    for step in range(w.steps):
        T = sh.n_new[step]
        c.append_rows(layer, list(range(S)), lens,
                      [(kall[b][0][lens[b]:lens[b] + T[b]], kall[b][1][lens[b]:lens[b] + T[b]]) for b in range(S)])
        qs = [qi.q_rows(w, b, layer, step, T[b]) for b in range(S)]
        out = c.verify(layer, [l + t for l, t in zip(lens, T)], T, qs)
        if step in (0, 13, w.steps - 1):
            want = np.concatenate([oracle_verify(w, b, layer, lens[b], qs[b], kall[b][0][:lens[b] + T[b]],
                                                 kall[b][1][:lens[b] + T[b]]) for b in range(S)])
            check_close(out, want)
        lens = [l + t for l, t in zip(lens, T)]
    for b in range(S):
        # every position appended during the 32 steps, bit for bit
        s0 = sh.ctx[b]
        _check_unit_records(c, w, b, layer, kall[b][0], kall[b][1], [(s0, lens[b] - s0)])
    assert int(c.status.item()) == 0


def test_workload5_655360_positions_layer_0():
    w = qi.WORKLOADS[5]
    sh = qi.draw_shapes(w)
    ctx, T = sh.ctx, sh.n_new[0]
    c = GpuCache(w, [ctx[0] + T[0]], contiguous=True)
    layer = 0
    (k, v), = _prefill_and_step(c, w, layer, [0], ctx, T, chunk=131072)
    q = qi.q_rows(w, 0, layer, 0, T[0])
    out = c.verify(layer, [ctx[0] + T[0]], T, [q])
    check_close(out, oracle_verify(w, 0, layer, ctx[0], q, k, v))
    rng = np.random.default_rng(0)
    pages = [(int(p) * 256, 256) for p in rng.choice(ctx[0] // 256, 12, replace=False)] + [(ctx[0] - 56, 64)]
    _check_unit_records(c, w, 0, layer, k, v, pages)
    assert int(c.status.item()) == 0
