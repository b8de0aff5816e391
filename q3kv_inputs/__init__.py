"""Seeded synthetic inputs for the q3kv verify step.

This module only draws random numbers and describes workload shapes.  It holds
none of the method's arithmetic (no rotation, no quantisation, no attention),
so both the CPU oracle and the CUDA path can take their inputs from it without
sharing any code that computes a result.

Workloads
---------
Five synthetic workloads stand in for the agentic traffic the source pages
measure on (the q27 wiki, "Self-speculation as the whole design" and "KV cache"
bullets: head_dim 256, 16 full-attention layers, verify widths up to 12,
contexts up to 655,360 positions).  No dataset item is reproduced.

Every value is addressed by what it is -- (slot, layer, kv head, K|V, page) for
cached keys and values, (slot, layer, step) for queries -- and drawn from its own
PCG64 stream, so any page of any workload can be regenerated on its own.  That
is what lets a test check a sampled unit of a full-size workload without
generating the rest.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np

HEAD_DIM = 256
PAGE_SIZE = 256

# spawn-key tags: keep streams for different roles apart
_TAG_SHAPE = 1
_TAG_KV = 2
_TAG_KV_CHANNEL = 3
_TAG_Q = 4
_TAG_Q_CHANNEL = 5
_TAG_LOGITS = 6
_TAG_TOKENS = 7

# Vocabulary size of the acceptance inputs: the padded vocabulary the pages
# quote for their model family (a synthetic stand-in; no weights are used).
VOCAB = 248_320


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic verify workload."""

    key: int                 # 1..5
    name: str
    seed: int
    num_slots: int
    num_layers: int
    ctx_range: Tuple[int, int]      # inclusive uniform range of cached positions N_b
    draft_range: Tuple[int, int]    # inclusive uniform range of d (T_b = 1 + d)
    steps: int                      # continuous-batching steps (append + verify each)
    dtype: str                      # 'f32' or 'bf16' for K, V and Q inputs
    kv_dist: str                    # 'outlier8' or 'loguniform10'
    q_dist: str                     # 'outlier8' or 'normal'
    num_kv_heads: int = 2
    num_q_heads: int = 16
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS: Dict[int, Workload] = {
    1: Workload(1, "1slot_1layer_ctx1024_t4_f32", 0, 1, 1, (1024, 1024), (3, 3), 1,
                "f32", "outlier8", "outlier8"),
    2: Workload(2, "1slot_16layer_ctx32768_t6_bf16", 1, 1, 16, (32768, 32768), (5, 5), 1,
                "bf16", "loguniform10", "normal"),
    3: Workload(3, "4slot_16layer_ragged8k-128k_t3-8_bf16", 2, 4, 16, (8192, 131072), (2, 7), 1,
                "bf16", "loguniform10", "normal"),
    4: Workload(4, "8slot_16layer_32step_ctx2k-64k_t4-8_bf16", 3, 8, 16, (2048, 65536), (3, 7), 32,
                "bf16", "loguniform10", "normal"),
    5: Workload(5, "1slot_16layer_ctx655360_t8_bf16", 4, 1, 16, (655360, 655360), (7, 7), 1,
                "bf16", "outlier8", "normal"),
}


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(key))))


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), kept as float32.

    Inputs of the bf16 workloads are drawn in float32 and rounded once here;
    that exact array is what both sides are given.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).reshape(x.shape)


@dataclasses.dataclass
class Shapes:
    """Drawn ragged shapes of a workload.

    ctx[b]     -- cached positions of slot b before the first step
    n_new[s][b] -- tokens slot b appends and verifies at step s (T = 1 + d)
    """

    ctx: List[int]
    n_new: List[List[int]]

    def ctx_before(self, step: int) -> List[int]:
        out = list(self.ctx)
        for s in range(step):
            out = [c + t for c, t in zip(out, self.n_new[s])]
        return out


def draw_shapes(w: Workload) -> Shapes:
    rng = _rng(w.seed, _TAG_SHAPE)
    lo, hi = w.ctx_range
    ctx = [int(rng.integers(lo, hi + 1)) for _ in range(w.num_slots)]
    dlo, dhi = w.draft_range
    n_new = [[1 + int(rng.integers(dlo, dhi + 1)) for _ in range(w.num_slots)] for _ in range(w.steps)]
    return Shapes(ctx, n_new)


def kv_channel_scale(w: Workload, layer: int, kv_head: int, which: int) -> np.ndarray:
    """Per-channel multiplier of K (which=0) or V (which=1) for one (layer, kv head).

    'outlier8': four distinct channels scaled x8, the rest x1.
    'loguniform10': every channel scaled by 10**U(0,1).
    The same multiplier applies to every slot and position.
    """
    rng = _rng(w.seed, _TAG_KV_CHANNEL, layer, kv_head, which)
    return _channel_scale(rng, w.kv_dist, w.head_dim)


def q_channel_scale(w: Workload, layer: int, q_head: int) -> np.ndarray:
    rng = _rng(w.seed, _TAG_Q_CHANNEL, layer, q_head)
    return _channel_scale(rng, w.q_dist, w.head_dim)


def _channel_scale(rng: np.random.Generator, dist: str, d: int) -> np.ndarray:
    if dist == "outlier8":
        s = np.ones(d, dtype=np.float32)
        s[rng.choice(d, size=4, replace=False)] = np.float32(8.0)
        return s
    if dist == "loguniform10":
        return (10.0 ** rng.uniform(0.0, 1.0, size=d)).astype(np.float32)
    if dist == "normal":
        return np.ones(d, dtype=np.float32)
    raise ValueError(dist)


def kv_page(w: Workload, slot: int, layer: int, kv_head: int, which: int, page: int) -> np.ndarray:
    """Raw (unrotated) K or V head vectors of positions [page*P, (page+1)*P) of a slot, float32 [P, D]."""
    rng = _rng(w.seed, _TAG_KV, slot, layer, kv_head, which, page)
    x = rng.standard_normal((w.page_size, w.head_dim), dtype=np.float32)
    x *= kv_channel_scale(w, layer, kv_head, which)[None, :]
    if w.dtype == "bf16":
        x = round_to_bf16(x)
    return x


def kv_rows(w: Workload, slot: int, layer: int, kv_head: int, which: int, start: int, count: int) -> np.ndarray:
    """Raw K or V vectors of positions [start, start+count) of a slot, float32 [count, D]."""
    out = np.empty((count, w.head_dim), dtype=np.float32)
    p = start
    while p < start + count:
        page = p // w.page_size
        base = page * w.page_size
        hi = min(start + count, base + w.page_size)
        out[p - start:hi - start] = kv_page(w, slot, layer, kv_head, which, page)[p - base:hi - base]
        p = hi
    return out


def q_rows(w: Workload, slot: int, layer: int, step: int, n_q: int) -> np.ndarray:
    """Raw (unrotated) queries of one slot at one step and layer, float32 [n_q, Hq, D]."""
    rng = _rng(w.seed, _TAG_Q, slot, layer, step)
    x = rng.standard_normal((n_q, w.num_q_heads, w.head_dim), dtype=np.float32)
    for h in range(w.num_q_heads):
        x[:, h, :] *= q_channel_scale(w, layer, h)[None, :]
    if w.dtype == "bf16":
        x = round_to_bf16(x)
    return x


def logits_rows(seed: int, rows: int, vocab: int, kind: str = "normal", bf16: bool = False) -> np.ndarray:
    """Synthetic logits float32 [rows, vocab] for the acceptance step.

    kind "normal": N(0, 4) values (distinct maxima); "ties": small integers in
    [-3, 3] (many equal maxima).  bf16=True rounds them once to bfloat16; that
    exact array is what both sides are given.
    """
    rng = _rng(seed, _TAG_LOGITS, rows, vocab)
    if kind == "ties":
        x = rng.integers(-3, 4, size=(rows, vocab)).astype(np.float32)
    else:
        x = (2.0 * rng.standard_normal((rows, vocab), dtype=np.float32)).astype(np.float32)
    return round_to_bf16(x) if bf16 else x


def random_tokens(seed: int, rows: int, vocab: int) -> np.ndarray:
    """Uniform random token ids int32 [rows] (query tokens that are not planted)."""
    return _rng(seed, _TAG_TOKENS, rows, vocab).integers(0, vocab, size=rows).astype(np.int32)


def random_page_table(num_slots: int, pages_per_slot: List[int], num_pages: int, seed: int) -> np.ndarray:
    """A scattered page table: distinct page ids drawn without replacement.

    Returned as int32 [num_slots, max(pages_per_slot)], unused entries -1.
    Tests use it so that the paged layout is exercised with non-contiguous pages.
    """
    need = int(sum(pages_per_slot))
    if need > num_pages:
        raise ValueError("not enough pages")
    rng = _rng(seed, 99)
    ids = rng.permutation(num_pages)[:need].astype(np.int32)
    width = max(1, max(pages_per_slot))
    pt = np.full((num_slots, width), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(pages_per_slot):
        pt[b, :n] = ids[k:k + n]
        k += n
    return pt


def torch_fill_kv_(x, w: Workload, layer: int, kv_head: int, which: int, generator) -> None:
    """Fill a device tensor [n, D] with raw K or V values of the workload's distribution.

    Used by the benchmark to populate large caches quickly on the device; the
    draws come from a seeded torch generator and are not the numpy streams
    above, so they serve timing, never parity.
    """
    import torch

    scale = torch.from_numpy(kv_channel_scale(w, layer, kv_head, which)).to(x.device)
    tmp = torch.randn(x.shape, generator=generator, device=x.device, dtype=torch.float32)
    tmp.mul_(scale)
    x.copy_(tmp.to(x.dtype))
