"""GPU parity of the fp8 E4M3 comparison cache (q3kv_fp8_append / q3kv_fp8_verify_attn).

Record bytes bit-exact against ``oracle.fp8``; verify outputs within max-abs
2e-3 and relative L2 1e-3 of the oracle's float64 attention over the decoded
values (plain basis, no rotation); ragged slots, split counts, masks and the
status bits of the format.
"""
import numpy as np
import pytest
import torch

import q3kv_inputs as qi
from gpu_harness import check_close, slot_kv, tdtype
from oracle import fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_attention_q3kv_gb300 import _lib
    _lib.load()


class Fp8Cache:
    def __init__(self, w, max_positions, num_layers=None, seed=5):
        from speculative_verify_attention_q3kv_gb300 import api
        self.api = api
        self.w = w
        self.num_layers = num_layers or w.num_layers
        pages = [(n + 255) // 256 for n in max_positions]
        self.num_pages = sum(pages)
        self.desc = api.make_desc(self.num_layers, w.num_kv_heads, self.num_pages)
        self.pool = torch.zeros(api.fp8_pool_bytes(self.desc), dtype=torch.uint8, device="cuda")
        pt = qi.random_page_table(w.num_slots, pages, self.num_pages, seed)
        self.page_table_np = pt
        self.page_table = torch.from_numpy(pt).cuda()
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def append(self, layer, starts, kv_rows):
        w = self.w
        n_new = np.array([k.shape[0] for k, _ in kv_rows], np.int32)
        offs = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
        dt = tdtype(w)
        k = torch.from_numpy(np.concatenate([k for k, _ in kv_rows])).to(dt).cuda()
        v = torch.from_numpy(np.concatenate([v for _, v in kv_rows])).to(dt).cuda()
        self.api.fp8_append(self.desc, self.pool, self.page_table, torch.tensor(np.asarray(starts, np.int32)).cuda(),
                            torch.from_numpy(n_new).cuda(), torch.from_numpy(offs).cuda(), int(n_new.max()), layer,
                            k, v, self.status)

    def verify(self, layer, ctx_len, n_q, q_rows, split_positions=0, impl=0):
        w = self.w
        offs = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int32)
        q = torch.from_numpy(np.concatenate(q_rows)).to(tdtype(w)).cuda()
        out = torch.full((q.shape[0], w.num_q_heads, 256), float("nan"), dtype=torch.float32, device="cuda")
        nbytes = self.api.workspace_bytes(self.desc, w.num_slots, max(ctx_len), max(n_q), 2, split_positions)
        ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        self.api.fp8_verify_attn(self.desc, self.pool, self.page_table, torch.tensor(np.asarray(ctx_len, np.int32)).cuda(),
                                 torch.tensor(np.asarray(n_q, np.int32)).cuda(), torch.from_numpy(offs).cuda(),
                                 max(ctx_len), max(n_q), layer, q, out, ws, impl, split_positions, self.status)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def records(self, slot, layer, g, kv, count):
        pos = np.arange(count)
        pages = self.page_table_np[slot][pos // 256].astype(np.int64)
        offs = ((((pages * self.num_layers + layer) * self.w.num_kv_heads + g) * 2 + kv) * 256 + pos % 256) * 256
        idx = torch.from_numpy(offs[:, None] + np.arange(256)[None, :]).cuda()
        return self.pool[idx].cpu().numpy()


def _bf16_exact(x, w):
    return torch.from_numpy(x).to(tdtype(w)).float().numpy()


def _oracle(w, n_ctx, q, k, v):
    kh = np.stack([fp8.decode(fp8.encode(_bf16_exact(k[:, g], w))[0]) for g in range(w.num_kv_heads)])
    vh = np.stack([fp8.decode(fp8.encode(_bf16_exact(v[:, g], w))[0]) for g in range(w.num_kv_heads)])
    return fp8.attention(_bf16_exact(q, w), kh, vh, n_ctx, w.group)


def _small(dtype, dist, slots):
    base = qi.WORKLOADS[1]
    return qi.Workload(base.key, "small", 13, slots, 2, (0, 0), (0, 0), 1, dtype, dist, dist)


def test_fp8_records_bit_exact_and_verify():
    w = qi.WORKLOADS[1]
    N, T = 1024, 4
    c = Fp8Cache(w, [N + T])
    k, v = slot_kv(w, 0, 0, 0, N + T)
    c.append(0, [0], [(k[:N], v[:N])])
    c.append(0, [N], [(k[N:], v[N:])])
    for g in range(2):
        for kv, x in ((0, k), (1, v)):
            assert np.array_equal(c.records(0, 0, g, kv, N + T), fp8.encode(_bf16_exact(x[:, g], w))[0])
    q = qi.q_rows(w, 0, 0, 0, T)
    out = c.verify(0, [N + T], [T], [q])
    check_close(out, _oracle(w, N, q, k, v))
    assert int(c.status.item()) == 0


@pytest.mark.parametrize("dtype,dist", [("f32", "outlier8"), ("bf16", "loguniform10")])
def test_fp8_ragged_slots_with_splits(dtype, dist):
    w = _small(dtype, dist, 4)
    ctx = [5, 300, 777, 1500]
    T = [1, 4, 8, 16]
    c = Fp8Cache(w, [n + t for n, t in zip(ctx, T)], num_layers=2)
    kvs = [slot_kv(w, b, 1, 0, ctx[b] + T[b]) for b in range(4)]
    c.append(1, [0] * 4, [(k[:ctx[b]], v[:ctx[b]]) for b, (k, v) in enumerate(kvs)])
    c.append(1, ctx, [(k[ctx[b]:], v[ctx[b]:]) for b, (k, v) in enumerate(kvs)])
    for b in range(4):
        for g in range(2):
            assert np.array_equal(c.records(b, 1, g, 1, ctx[b] + T[b]),
                                  fp8.encode(_bf16_exact(kvs[b][1][:, g], w))[0])
    qs = [qi.q_rows(w, b, 1, 0, T[b]) for b in range(4)]
    want = np.concatenate([_oracle(w, ctx[b], qs[b], *kvs[b]) for b in range(4)])
    for split in (256, 512, 0):
        got = c.verify(1, [n + t for n, t in zip(ctx, T)], T, qs, split_positions=split)
        check_close(got, want)
    assert int(c.status.item()) == 0


def test_fp8_saturation_and_non_finite_flag():
    w = _small("f32", "outlier8", 1)
    n = 300
    k, v = slot_kv(w, 0, 0, 0, n)
    k = k.copy()
    v = v.copy()
    k[3, 0, :8] = [500.0, -1e6, 448.0, 464.0, -470.0, 2.0 ** -10, -2.0 ** -10, 1e-9]
    c = Fp8Cache(w, [n])
    c.append(0, [0], [(k, v)])
    rec = c.records(0, 0, 0, 0, n)
    assert list(rec[3, :8]) == [0x7E, 0xFE, 0x7E, 0x7E, 0xFE, 0x00, 0x80, 0x00]
    assert np.array_equal(rec, fp8.encode(k[:, 0])[0])
    assert int(c.status.item()) == 0
    q = qi.q_rows(w, 0, 0, 0, 4)
    check_close(c.verify(0, [n], [4], [q]), _oracle(w, n - 4, q, k, v))
    k[7, 1, 5] = np.inf
    c.append(0, [0], [(k, v)])
    assert int(c.status.item()) & 1


def test_fp8_cuda_core_leg_is_unsupported():
    from speculative_verify_attention_q3kv_gb300 import _lib
    w = _small("f32", "outlier8", 1)
    c = Fp8Cache(w, [260])
    k, v = slot_kv(w, 0, 0, 0, 260)
    c.append(0, [0], [(k, v)])
    with pytest.raises(_lib.Q3KVError) as e:
        c.verify(0, [260], [4], [qi.q_rows(w, 0, 0, 0, 4)], impl=1)
    assert e.value.code == _lib.Q3KV_ERR_UNSUPPORTED
