"""Helpers shared by the GPU tests (not collected by pytest itself).

They drive the CUDA path only through the Python binding of the C ABI
(``speculative_verify_attention_q3kv_gb300.api``) and compute expectations only
with ``oracle``; both sides take their inputs from ``q3kv_inputs``.
"""
from __future__ import annotations

import numpy as np
import torch

import q3kv_inputs as qi
from oracle import codec, packing
from oracle.attention import verify_attention
from oracle.cache import encode_dequantized
from speculative_verify_attention_q3kv_gb300 import api

MAX_ABS = 2e-3
REL_L2 = 1e-3


def tdtype(w: qi.Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


class GpuCache:
    """A device pool plus its page table for the slots of one workload."""

    def __init__(self, w: qi.Workload, max_positions, num_layers=None, extra_pages=0, seed=7, contiguous=False):
        self.w = w
        self.num_layers = num_layers or w.num_layers
        pages = [(n + qi.PAGE_SIZE - 1) // qi.PAGE_SIZE for n in max_positions]
        self.num_pages = sum(pages) + extra_pages
        self.desc = api.make_desc(self.num_layers, w.num_kv_heads, self.num_pages)
        self.pool = torch.zeros(api.pool_bytes(self.desc), dtype=torch.uint8, device="cuda")
        if contiguous:
            pt = np.full((w.num_slots, max(pages)), -1, np.int32)
            k = 0
            for b, n in enumerate(pages):
                pt[b, :n] = np.arange(k, k + n)
                k += n
        else:
            pt = qi.random_page_table(w.num_slots, pages, self.num_pages, seed)
        self.page_table_np = pt
        self.page_table = torch.from_numpy(pt).cuda()
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def append_rows(self, layer, slots, starts, kv_rows, layer_index=None):
        """Append raw K/V rows (per slot: float32 [n, Hkv, 256] pairs) at the given start positions."""
        w = self.w
        n_new = [k.shape[0] for k, _ in kv_rows]
        offs = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
        full_len = np.zeros(w.num_slots, np.int32)
        full_new = np.zeros(w.num_slots, np.int32)
        full_off = np.zeros(w.num_slots + 1, np.int32)
        # rows are laid out in slot order of `slots`; map to a dense per-slot table
        row_starts = np.zeros(w.num_slots, np.int32)
        for i, b in enumerate(slots):
            full_len[b] = starts[i]
            full_new[b] = n_new[i]
            row_starts[b] = offs[i]
        full_off[:-1] = row_starts
        full_off[-1] = offs[-1]
        k = np.concatenate([k for k, _ in kv_rows]) if kv_rows else np.zeros((0, w.num_kv_heads, 256), np.float32)
        v = np.concatenate([v for _, v in kv_rows]) if kv_rows else np.zeros((0, w.num_kv_heads, 256), np.float32)
        dt = tdtype(w)
        kd = torch.from_numpy(np.ascontiguousarray(k)).to(dt).cuda()
        vd = torch.from_numpy(np.ascontiguousarray(v)).to(dt).cuda()
        api.append(self.desc, self.pool, self.page_table, torch.from_numpy(full_len).cuda(),
                   torch.from_numpy(full_new).cuda(), torch.from_numpy(full_off).cuda(), max(n_new + [0]),
                   layer if layer_index is None else layer_index, kd, vd, self.status)

    def verify(self, layer, ctx_len, n_q, q_rows, impl=0, split_positions=0, layer_index=None):
        """Run q3kv_verify_attn; q_rows per slot float32 [T_b, Hq, 256]. Returns float32 [sum T, Hq, 256]."""
        w = self.w
        offs = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int32)
        q = np.concatenate(q_rows) if q_rows else np.zeros((0, w.num_q_heads, 256), np.float32)
        qd = torch.from_numpy(np.ascontiguousarray(q)).to(tdtype(w)).cuda()
        out = torch.full((max(q.shape[0], 1), w.num_q_heads, 256), float("nan"), dtype=torch.float32, device="cuda")
        max_ctx = int(max(ctx_len)) if len(ctx_len) else 0
        max_nq = int(max(n_q)) if len(n_q) else 0
        nbytes = api.workspace_bytes(self.desc, w.num_slots, max_ctx, max_nq, impl, split_positions)
        ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        api.verify_attn(self.desc, self.pool, self.page_table,
                        torch.tensor(np.asarray(ctx_len, np.int32)).cuda(), torch.tensor(np.asarray(n_q, np.int32)).cuda(),
                        torch.from_numpy(offs).cuda(), max_ctx, max_nq,
                        layer if layer_index is None else layer_index, qd, out, ws, impl, split_positions, self.status)
        torch.cuda.synchronize()
        return out[: q.shape[0]].cpu().numpy()

    def records(self, slot, layer, kv_head, kv, start, count, layer_index=None):
        """Bytes of records [count, 112] of positions [start, start+count) of a slot (read back for comparison)."""
        pool = self.pool
        li = layer if layer_index is None else layer_index
        out = []
        pos = np.arange(start, start + count)
        pages = self.page_table_np[slot][pos // 256]
        offs = ((((pages.astype(np.int64) * self.num_layers + li) * self.w.num_kv_heads + kv_head) * 2 + kv) * 256
                + pos % 256) * 112
        idx = torch.from_numpy(offs[:, None] + np.arange(112)[None, :]).cuda()
        return pool[idx].cpu().numpy()


def oracle_records(x_raw):
    codes, s16, _ = codec.encode(x_raw)
    return packing.pack_records(codes, s16)


def check_close(got, want, max_abs=MAX_ABS, rel_l2=REL_L2):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - want)
    ma = float(err.max()) if err.size else 0.0
    rl = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)) if err.size else 0.0
    assert ma <= max_abs and rl <= rel_l2, f"max_abs {ma:.3e} rel_l2 {rl:.3e}"
    return ma, rl


def slot_kv(w, slot, layer, start, count):
    """Raw K and V [count, Hkv, 256] of a slot."""
    k = np.stack([qi.kv_rows(w, slot, layer, g, 0, start, count) for g in range(w.num_kv_heads)], axis=1)
    v = np.stack([qi.kv_rows(w, slot, layer, g, 1, start, count) for g in range(w.num_kv_heads)], axis=1)
    return k, v


def oracle_verify(w, slot, layer, n_ctx, q, k_all=None, v_all=None):
    """fp64 verify output of one slot, from raw inputs (encodes positions [0, n_ctx + T))."""
    T = q.shape[0]
    if k_all is None:
        k_all, v_all = slot_kv(w, slot, layer, 0, n_ctx + T)
    kh = np.stack([encode_dequantized(k_all[:, g]) for g in range(w.num_kv_heads)])
    vh = np.stack([encode_dequantized(v_all[:, g]) for g in range(w.num_kv_heads)])
    return verify_attention(q, kh, vh, n_ctx, w.group)
