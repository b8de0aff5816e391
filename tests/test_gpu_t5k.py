"""GPU parity of the turbo5k-style cache (q3kv_t5k_append / q3kv_t5k_verify_attn).

K records (5-bit Lloyd-Max codes, nibble and 5th-bit planes, two fp16 scales)
and V records (the 3-bit codec) bit-exact against ``oracle.turbo5k``; verify
outputs of both legs within max-abs 2e-3 / relative L2 1e-3 of the float64
attention over the decoded values (the tensor-core leg reads K_hat rounded to
float32 and split into fp16 hi/lo).
"""
import numpy as np
import pytest
import torch

import q3kv_inputs as qi
from gpu_harness import check_close, slot_kv, tdtype
from oracle import codec as q3codec
from oracle import packing as q3packing
from oracle import turbo5k as t
from oracle.attention import verify_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_attention_q3kv_gb300 import _lib
    _lib.load()


class T5kCache:
    def __init__(self, w, max_positions, num_layers=None, seed=9):
        from speculative_verify_attention_q3kv_gb300 import api
        self.api, self.w = api, w
        self.num_layers = num_layers or w.num_layers
        pages = [(n + 255) // 256 for n in max_positions]
        self.num_pages = sum(pages)
        self.desc = api.make_desc(self.num_layers, w.num_kv_heads, self.num_pages)
        self.pool = torch.zeros(api.t5k_pool_bytes(self.desc), dtype=torch.uint8, device="cuda")
        self.pt = qi.random_page_table(w.num_slots, pages, self.num_pages, seed)
        self.page_table = torch.from_numpy(self.pt).cuda()
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def append(self, layer, starts, kv_rows):
        n_new = np.array([k.shape[0] for k, _ in kv_rows], np.int32)
        offs = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
        dt = tdtype(self.w)
        k = torch.from_numpy(np.concatenate([k for k, _ in kv_rows])).to(dt).cuda()
        v = torch.from_numpy(np.concatenate([v for _, v in kv_rows])).to(dt).cuda()
        self.api.t5k_append(self.desc, self.pool, self.page_table, torch.tensor(np.asarray(starts, np.int32)).cuda(),
                            torch.from_numpy(n_new).cuda(), torch.from_numpy(offs).cuda(), int(n_new.max()), layer,
                            k, v, self.status)

    def verify(self, layer, ctx_len, n_q, q_rows, split_positions=0, impl=1):
        w = self.w
        offs = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int32)
        q = torch.from_numpy(np.concatenate(q_rows)).to(tdtype(w)).cuda()
        out = torch.full((q.shape[0], w.num_q_heads, 256), float("nan"), dtype=torch.float32, device="cuda")
        nbytes = self.api.workspace_bytes(self.desc, w.num_slots, max(ctx_len), max(n_q), impl, split_positions)
        ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        self.api.t5k_verify_attn(self.desc, self.pool, self.page_table, torch.tensor(np.asarray(ctx_len, np.int32)).cuda(),
                                 torch.tensor(np.asarray(n_q, np.int32)).cuda(), torch.from_numpy(offs).cuda(),
                                 max(ctx_len), max(n_q), layer, q, out, ws, impl, split_positions, self.status)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def records(self, slot, layer, g, kv, count):
        pos = np.arange(count)
        pages = self.pt[slot][pos // 256].astype(np.int64)
        size = t.K_RECORD_BYTES if kv == 0 else t.V_RECORD_BYTES
        fn = t.k_offset if kv == 0 else t.v_offset
        offs = fn(self.num_layers, self.w.num_kv_heads, pages, layer, g, pos % 256)
        idx = torch.from_numpy(offs[:, None] + np.arange(size)[None, :]).cuda()
        return self.pool[idx].cpu().numpy()


def _oracle(w, n_ctx, q, k, v):
    kh = np.stack([t.encode_dequantized_k(k[:, g]) for g in range(w.num_kv_heads)])
    vh = np.stack([q3codec.dequantize(*q3codec.encode(v[:, g])[:2]) for g in range(w.num_kv_heads)])
    return verify_attention(q, kh, vh, n_ctx, w.group)


def _small(dtype, dist, slots):
    base = qi.WORKLOADS[1]
    return qi.Workload(base.key, "small", 19, slots, 2, (0, 0), (0, 0), 1, dtype, dist, dist)


@pytest.mark.parametrize("impl", [1, 2])
@pytest.mark.parametrize("dtype,dist", [("f32", "outlier8"), ("bf16", "loguniform10")])
def test_t5k_records_bit_exact_and_verify(dtype, dist, impl):
    w = _small(dtype, dist, 1)
    N, T = 700, 6
    c = T5kCache(w, [N + T])
    k, v = slot_kv(w, 0, 0, 0, N + T)
    c.append(0, [0], [(k[:N], v[:N])])
    c.append(0, [N], [(k[N:], v[N:])])
    for g in range(2):
        kc, ks, _ = t.encode_k(k[:, g])
        assert np.array_equal(c.records(0, 0, g, 0, N + T), t.pack_k(kc, ks))
        vc, vs, _ = q3codec.encode(v[:, g])
        assert np.array_equal(c.records(0, 0, g, 1, N + T), q3packing.pack_records(vc, vs))
    q = qi.q_rows(w, 0, 0, 0, T)
    for split in (256, 0):
        check_close(c.verify(0, [N + T], [T], [q], split_positions=split, impl=impl), _oracle(w, N, q, k, v))
    assert int(c.status.item()) == 0


@pytest.mark.parametrize("impl", [1, 2])
def test_t5k_ragged_slots(impl):
    w = _small("bf16", "outlier8", 3)
    ctx = [5, 300, 1500]
    T = [1, 8, 16]
    c = T5kCache(w, [n + t_ for n, t_ in zip(ctx, T)], num_layers=2)
    kvs = [slot_kv(w, b, 1, 0, ctx[b] + T[b]) for b in range(3)]
    c.append(1, [0] * 3, [(k[:ctx[b]], v[:ctx[b]]) for b, (k, v) in enumerate(kvs)])
    c.append(1, ctx, [(k[ctx[b]:], v[ctx[b]:]) for b, (k, v) in enumerate(kvs)])
    qs = [qi.q_rows(w, b, 1, 0, T[b]) for b in range(3)]
    want = np.concatenate([_oracle(w, ctx[b], qs[b], *kvs[b]) for b in range(3)])
    check_close(c.verify(1, [n + t_ for n, t_ in zip(ctx, T)], T, qs, impl=impl), want)
    assert int(c.status.item()) == 0


def test_t5k_outlier_heavy_verify_shapes_tensor_core_leg():
    """Verify widths 6..16 over 4K+ positions, queries and cache both with 10x channels."""
    w = _small("bf16", "loguniform10", 2)
    ctx, T = [4096, 5000], [6, 16]
    L = [n + t_ for n, t_ in zip(ctx, T)]
    c = T5kCache(w, L, num_layers=1)
    kvs = [slot_kv(w, b, 0, 0, L[b]) for b in range(2)]
    c.append(0, [0, 0], kvs)
    qs = [qi.q_rows(w, b, 0, 0, T[b]) for b in range(2)]
    want = np.concatenate([_oracle(w, ctx[b], qs[b], *kvs[b]) for b in range(2)])
    for split in (0, 256):
        check_close(c.verify(0, L, T, qs, split_positions=split, impl=2), want)
    assert int(c.status.item()) == 0
