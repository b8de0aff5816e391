"""Thin Python layer over the C ABI: torch tensors in, raw pointers out.

Argument marshalling only -- every step of the hot path runs in the CUDA
library.  Names follow ``include/q3kv.h``.  Device buffers are torch tensors the
caller owns; the library never allocates device memory.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np
import torch

from . import _lib
from ._lib import CacheDesc, Q3KVError, check  # noqa: F401  (re-exported)

HEAD_DIM = 256
PAGE_SIZE = 256
GROUP = 8


def make_desc(num_layers: int, num_kv_heads: int, num_pages: int) -> CacheDesc:
    return CacheDesc(num_layers, num_kv_heads, GROUP * num_kv_heads, HEAD_DIM, PAGE_SIZE, num_pages)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to q3kv must be contiguous")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return _lib.Q3KV_F32
    if t.dtype == torch.bfloat16:
        return _lib.Q3KV_BF16
    raise TypeError(f"q3kv inputs must be float32 or bfloat16, got {t.dtype}")


def _on_gpu(name: str, t: Optional[torch.Tensor], dev: int, dtype=None, min_numel: int = 0,
            optional: bool = False) -> None:
    """Refuse, before any launch, a tensor the kernels could not address safely.

    The C ABI takes raw device pointers; a host tensor, a tensor on another
    device, a wrong element type or a buffer shorter than the call's counts
    would be read or written out of bounds on the GPU.  Values inside device
    arrays (lengths, offsets, page ids) are checked by the kernels.
    """
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    idx = _device_index(t)
    if idx is None:
        raise ValueError(f"{name} must be a CUDA tensor")
    if idx != dev:
        raise ValueError(f"{name} is on cuda:{idx}, the current device is cuda:{dev}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements, the call needs at least {min_numel}")


def _device_index(t: torch.Tensor) -> Optional[int]:
    """CUDA device index of a tensor; None for a tensor in host (or any other) memory."""
    return t.device.index if t.is_cuda else None


def _current_device() -> int:
    return torch.cuda.current_device() if torch.cuda.is_available() else -1


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _check_cache_args(desc: CacheDesc, pool: torch.Tensor, need_pool_bytes: int, page_table: torch.Tensor,
                      lens: torch.Tensor, counts: torch.Tensor, offsets: torch.Tensor,
                      status: Optional[torch.Tensor], dev: int) -> int:
    """Common checks of the append / verify / prefill calls; returns num_slots."""
    _on_gpu("pool", pool, dev)
    if _nbytes(pool) < need_pool_bytes:
        raise ValueError(f"pool holds {_nbytes(pool)} bytes, the cache needs {need_pool_bytes}")
    _on_gpu("lengths", lens, dev, torch.int32)
    if lens.dim() != 1:
        raise ValueError("per-slot lengths must be one-dimensional")
    n = lens.shape[0]
    _on_gpu("page_table", page_table, dev, torch.int32)
    if page_table.dim() != 2 or page_table.shape[1] < 1 or (n > 0 and page_table.shape[0] < n):
        raise ValueError(f"page_table must be int32 [num_slots >= {n}, max_pages_per_slot >= 1], "
                         f"got {tuple(page_table.shape)}")
    _on_gpu("per-slot token counts", counts, dev, torch.int32, n)
    _on_gpu("row offsets", offsets, dev, torch.int32, n)
    _on_gpu("status", status, dev, torch.int32, 1, optional=True)
    return n


def _check_rows(name: str, t: torch.Tensor, heads: int, dev: int) -> None:
    _on_gpu(name, t, dev)
    if t.dim() != 3 or t.shape[1] != heads or t.shape[2] != HEAD_DIM:
        raise ValueError(f"{name} must be [rows, {heads}, {HEAD_DIM}], got {tuple(t.shape)}")


def _check_append(desc, pool, pool_bytes_fn, page_table, slot_len, n_new, row_offsets, k, v, status) -> None:
    dev = _current_device()
    _check_cache_args(desc, pool, pool_bytes_fn(desc), page_table, slot_len, n_new, row_offsets, status, dev)
    if k.dtype != v.dtype:
        raise TypeError("k and v must share a dtype")
    _check_rows("k", k, desc.num_kv_heads, dev)
    _check_rows("v", v, desc.num_kv_heads, dev)
    if k.shape != v.shape:
        raise ValueError(f"k and v differ in shape: {tuple(k.shape)} vs {tuple(v.shape)}")


def _check_verify(desc, pool, pool_bytes_fn, page_table, ctx_len, n_q, q_offsets, q, out, workspace,
                  status) -> None:
    dev = _current_device()
    _check_cache_args(desc, pool, pool_bytes_fn(desc), page_table, ctx_len, n_q, q_offsets, status, dev)
    _check_rows("q", q, desc.num_q_heads, dev)
    if out.dtype != torch.float32:
        raise TypeError("out must be float32")
    _check_rows("out", out, desc.num_q_heads, dev)
    if out.shape[0] < q.shape[0]:
        raise ValueError(f"out has {out.shape[0]} rows, q has {q.shape[0]}")
    _on_gpu("workspace", workspace, dev, optional=True)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pool_bytes(desc: CacheDesc) -> int:
    n = ctypes.c_size_t()
    check(_lib.load().q3kv_pool_bytes(ctypes.byref(desc), ctypes.byref(n)), "q3kv_pool_bytes")
    return n.value


def workspace_bytes(desc: CacheDesc, num_slots: int, max_ctx_len: int, max_n_q: int,
                    impl: int = _lib.Q3KV_IMPL_AUTO, split_positions: int = 0) -> int:
    n = ctypes.c_size_t()
    check(_lib.load().q3kv_workspace_bytes(ctypes.byref(desc), num_slots, max_ctx_len, max_n_q, impl,
                                           split_positions, ctypes.byref(n)), "q3kv_workspace_bytes")
    return n.value


class Allocator:
    """Host free-list page allocator (q3kv_allocator_*)."""

    def __init__(self, num_pages: int, num_slots: int, max_pages_per_slot: int):
        self._lib = _lib.load()
        h = ctypes.c_void_p()
        check(self._lib.q3kv_allocator_create(num_pages, num_slots, max_pages_per_slot, ctypes.byref(h)),
              "q3kv_allocator_create")
        self._h = h
        self.max_pages_per_slot = max_pages_per_slot

    def alloc_pages(self, slot: int, n_positions: int) -> np.ndarray:
        row = np.full(self.max_pages_per_slot, -1, dtype=np.int32)
        n = ctypes.c_int32()
        check(self._lib.q3kv_alloc_pages(self._h, slot, n_positions,
                                         row.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), ctypes.byref(n)),
              "q3kv_alloc_pages")
        return row

    def free_slot(self, slot: int) -> None:
        check(self._lib.q3kv_free_slot(self._h, slot), "q3kv_free_slot")

    def free_pages(self) -> int:
        n = ctypes.c_int32()
        check(self._lib.q3kv_free_pages(self._h, ctypes.byref(n)), "q3kv_free_pages")
        return n.value

    def close(self) -> None:
        if self._h:
            self._lib.q3kv_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def append(desc: CacheDesc, pool: torch.Tensor, page_table: torch.Tensor, slot_len: torch.Tensor,
           n_new: torch.Tensor, row_offsets: torch.Tensor, max_n_new: int, layer: int,
           k: torch.Tensor, v: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_append: quantise and store k, v [rows, kv_heads, 256] for each slot."""
    _check_append(desc, pool, pool_bytes, page_table, slot_len, n_new, row_offsets, k, v, status)
    rc = _lib.load().q3kv_append(_stream(stream), ctypes.byref(desc), _ptr(pool), _ptr(page_table),
                                 page_table.shape[1], _ptr(slot_len), _ptr(n_new), _ptr(row_offsets),
                                 slot_len.shape[0], max_n_new, layer, _ptr(k), _ptr(v), _dtype_code(k),
                                 _ptr(status))
    check(rc, "q3kv_append")


def verify_attn(desc: CacheDesc, pool: torch.Tensor, page_table: torch.Tensor, ctx_len: torch.Tensor,
                n_q: torch.Tensor, q_offsets: torch.Tensor, max_ctx_len: int, max_n_q: int, layer: int,
                q: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                impl: int = _lib.Q3KV_IMPL_AUTO, split_positions: int = 0,
                status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_verify_attn: out[rows, q_heads, 256] (float32) for every slot's query tokens."""
    _check_verify(desc, pool, pool_bytes, page_table, ctx_len, n_q, q_offsets, q, out, workspace, status)
    rc = _lib.load().q3kv_verify_attn(_stream(stream), ctypes.byref(desc), _ptr(pool), _ptr(page_table),
                                      page_table.shape[1], _ptr(ctx_len), _ptr(n_q), _ptr(q_offsets),
                                      ctx_len.shape[0], max_ctx_len, max_n_q, layer, _ptr(q), _dtype_code(q),
                                      _ptr(out), impl, split_positions, _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _ptr(status))
    check(rc, "q3kv_verify_attn")


def verify_attn_noalloc(desc: CacheDesc, pool: torch.Tensor, page_table: torch.Tensor, ctx_len: torch.Tensor,
                        n_q: torch.Tensor, q_offsets: torch.Tensor, max_ctx_len: int, max_n_q: int, layer: int,
                        q: torch.Tensor, out: torch.Tensor, impl: int = _lib.Q3KV_IMPL_AUTO,
                        split_positions: int = 0, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_verify_attn_noalloc: verify_attn with the library's fixed scratch instead of a workspace.

    For callers that cannot provide device scratch memory; calls that overlap
    on the GPU share that scratch and must not run concurrently.
    """
    _check_verify(desc, pool, pool_bytes, page_table, ctx_len, n_q, q_offsets, q, out, None, status)
    rc = _lib.load().q3kv_verify_attn_noalloc(_stream(stream), ctypes.byref(desc), _ptr(pool), _ptr(page_table),
                                              page_table.shape[1], _ptr(ctx_len), _ptr(n_q), _ptr(q_offsets),
                                              ctx_len.shape[0], max_ctx_len, max_n_q, layer, _ptr(q),
                                              _dtype_code(q), _ptr(out), impl, split_positions, _ptr(status))
    check(rc, "q3kv_verify_attn_noalloc")


def prefill_workspace_bytes(desc: CacheDesc, num_slots: int, max_ctx_len: int, max_n_new: int,
                            impl: int = _lib.Q3KV_IMPL_AUTO, split_positions: int = 0) -> int:
    n = ctypes.c_size_t()
    check(_lib.load().q3kv_prefill_workspace_bytes(ctypes.byref(desc), num_slots, max_ctx_len, max_n_new, impl,
                                                   split_positions, ctypes.byref(n)), "q3kv_prefill_workspace_bytes")
    return n.value


def prefill_attn(desc: CacheDesc, pool: torch.Tensor, page_table: torch.Tensor, ctx_len: torch.Tensor,
                 n_new: torch.Tensor, q_offsets: torch.Tensor, max_ctx_len: int, max_n_new: int, layer: int,
                 q: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                 impl: int = _lib.Q3KV_IMPL_AUTO, split_positions: int = 0,
                 status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_prefill_attn: causal attention of up to 8192 appended tokens per slot over the 3-bit cache."""
    _check_verify(desc, pool, pool_bytes, page_table, ctx_len, n_new, q_offsets, q, out, workspace, status)
    rc = _lib.load().q3kv_prefill_attn(_stream(stream), ctypes.byref(desc), _ptr(pool), _ptr(page_table),
                                       page_table.shape[1], _ptr(ctx_len), _ptr(n_new), _ptr(q_offsets),
                                       ctx_len.shape[0], max_ctx_len, max_n_new, layer, _ptr(q), _dtype_code(q),
                                       _ptr(out), impl, split_positions, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(status))
    check(rc, "q3kv_prefill_attn")


def t5k_pool_bytes(desc: CacheDesc) -> int:
    """q3kv_t5k_pool_bytes: bytes of a turbo5k-style pool (164-byte K, 112-byte V records)."""
    n = ctypes.c_size_t()
    check(_lib.load().q3kv_t5k_pool_bytes(ctypes.byref(desc), ctypes.byref(n)), "q3kv_t5k_pool_bytes")
    return n.value


def t5k_append(desc: CacheDesc, pool: torch.Tensor, page_table: torch.Tensor, slot_len: torch.Tensor,
               n_new: torch.Tensor, row_offsets: torch.Tensor, max_n_new: int, layer: int,
               k: torch.Tensor, v: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_t5k_append: 5-bit Lloyd-Max K and 3-bit V records for k, v [rows, kv_heads, 256]."""
    _check_append(desc, pool, t5k_pool_bytes, page_table, slot_len, n_new, row_offsets, k, v, status)
    rc = _lib.load().q3kv_t5k_append(_stream(stream), ctypes.byref(desc), _ptr(pool), _ptr(page_table),
                                     page_table.shape[1], _ptr(slot_len), _ptr(n_new), _ptr(row_offsets),
                                     slot_len.shape[0], max_n_new, layer, _ptr(k), _ptr(v), _dtype_code(k),
                                     _ptr(status))
    check(rc, "q3kv_t5k_append")


def t5k_verify_attn(desc: CacheDesc, pool: torch.Tensor, page_table: torch.Tensor, ctx_len: torch.Tensor,
                    n_q: torch.Tensor, q_offsets: torch.Tensor, max_ctx_len: int, max_n_q: int, layer: int,
                    q: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                    impl: int = _lib.Q3KV_IMPL_FMA, split_positions: int = 0,
                    status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_t5k_verify_attn: verify attention over the turbo5k-style cache (CUDA-core leg)."""
    _check_verify(desc, pool, t5k_pool_bytes, page_table, ctx_len, n_q, q_offsets, q, out, workspace, status)
    rc = _lib.load().q3kv_t5k_verify_attn(_stream(stream), ctypes.byref(desc), _ptr(pool), _ptr(page_table),
                                          page_table.shape[1], _ptr(ctx_len), _ptr(n_q), _ptr(q_offsets),
                                          ctx_len.shape[0], max_ctx_len, max_n_q, layer, _ptr(q), _dtype_code(q),
                                          _ptr(out), impl, split_positions, _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _ptr(status))
    check(rc, "q3kv_t5k_verify_attn")


def fp8_pool_bytes(desc: CacheDesc) -> int:
    """q3kv_fp8_pool_bytes: bytes of an fp8 E4M3 comparison pool (256-byte records)."""
    n = ctypes.c_size_t()
    check(_lib.load().q3kv_fp8_pool_bytes(ctypes.byref(desc), ctypes.byref(n)), "q3kv_fp8_pool_bytes")
    return n.value


def fp8_append(desc: CacheDesc, pool: torch.Tensor, page_table: torch.Tensor, slot_len: torch.Tensor,
               n_new: torch.Tensor, row_offsets: torch.Tensor, max_n_new: int, layer: int,
               k: torch.Tensor, v: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_fp8_append: store k, v [rows, kv_heads, 256] as E4M3 records (the comparison cache)."""
    _check_append(desc, pool, fp8_pool_bytes, page_table, slot_len, n_new, row_offsets, k, v, status)
    rc = _lib.load().q3kv_fp8_append(_stream(stream), ctypes.byref(desc), _ptr(pool), _ptr(page_table),
                                     page_table.shape[1], _ptr(slot_len), _ptr(n_new), _ptr(row_offsets),
                                     slot_len.shape[0], max_n_new, layer, _ptr(k), _ptr(v), _dtype_code(k),
                                     _ptr(status))
    check(rc, "q3kv_fp8_append")


def fp8_verify_attn(desc: CacheDesc, pool: torch.Tensor, page_table: torch.Tensor, ctx_len: torch.Tensor,
                    n_q: torch.Tensor, q_offsets: torch.Tensor, max_ctx_len: int, max_n_q: int, layer: int,
                    q: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                    impl: int = _lib.Q3KV_IMPL_AUTO, split_positions: int = 0,
                    status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_fp8_verify_attn: verify attention over the fp8 comparison cache (tensor-core leg)."""
    _check_verify(desc, pool, fp8_pool_bytes, page_table, ctx_len, n_q, q_offsets, q, out, workspace, status)
    rc = _lib.load().q3kv_fp8_verify_attn(_stream(stream), ctypes.byref(desc), _ptr(pool), _ptr(page_table),
                                          page_table.shape[1], _ptr(ctx_len), _ptr(n_q), _ptr(q_offsets),
                                          ctx_len.shape[0], max_ctx_len, max_n_q, layer, _ptr(q), _dtype_code(q),
                                          _ptr(out), impl, split_positions, _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _ptr(status))
    check(rc, "q3kv_fp8_verify_attn")


def _check_accept(logits, q_offsets, n_q, tokens, ctx_len, n_accepted, next_token, committed_len, workspace,
                  status):
    """Checks common to the acceptance calls; returns (rows, vocab) of the logits."""
    dev = _current_device()
    _on_gpu("logits", logits, dev)
    if logits.dim() != 2:
        raise ValueError(f"logits must be [rows, vocab], got {tuple(logits.shape)}")
    _dtype_code(logits)
    rows, vocab = logits.shape
    _on_gpu("n_q", n_q, dev, torch.int32)
    if n_q.dim() != 1:
        raise ValueError("n_q must be one-dimensional")
    n = n_q.shape[0]
    for name, t in (("q_offsets", q_offsets), ("ctx_len", ctx_len), ("n_accepted", n_accepted),
                    ("next_token", next_token), ("committed_len", committed_len)):
        _on_gpu(name, t, dev, torch.int32, n)
    _on_gpu("tokens", tokens, dev, torch.int32, rows)
    _on_gpu("workspace", workspace, dev, optional=True)
    _on_gpu("status", status, dev, torch.int32, 1, optional=True)
    return rows, vocab


def accept_workspace_bytes(num_rows: int, vocab: int) -> int:
    n = ctypes.c_size_t()
    check(_lib.load().q3kv_accept_workspace_bytes(num_rows, vocab, ctypes.byref(n)), "q3kv_accept_workspace_bytes")
    return n.value


def accept_greedy(logits: torch.Tensor, q_offsets: torch.Tensor, n_q: torch.Tensor, tokens: torch.Tensor,
                  max_n_q: int, ctx_len: torch.Tensor, n_accepted: torch.Tensor, next_token: torch.Tensor,
                  committed_len: torch.Tensor, workspace: Optional[torch.Tensor],
                  status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_accept_greedy: logits [rows, vocab] (f32 or bf16); int32 per-slot outputs."""
    rows, vocab = _check_accept(logits, q_offsets, n_q, tokens, ctx_len, n_accepted, next_token, committed_len,
                                workspace, status)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.load().q3kv_accept_greedy(_stream(stream), _ptr(logits), _dtype_code(logits), vocab, _ptr(q_offsets),
                                        _ptr(n_q), _ptr(tokens), n_q.shape[0], rows, max_n_q, _ptr(ctx_len),
                                        _ptr(n_accepted), _ptr(next_token), _ptr(committed_len), _ptr(workspace),
                                        nbytes, _ptr(status))
    check(rc, "q3kv_accept_greedy")


def accept_sample(logits: torch.Tensor, q_offsets: torch.Tensor, n_q: torch.Tensor, tokens: torch.Tensor,
                  max_n_q: int, ctx_len: torch.Tensor, temperature: float, uniforms: torch.Tensor, seed: int,
                  n_accepted: torch.Tensor, next_token: torch.Tensor, committed_len: torch.Tensor,
                  workspace: Optional[torch.Tensor], status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_accept_sample: rejection-sampled acceptance; uniforms float32 [rows]."""
    rows, vocab = _check_accept(logits, q_offsets, n_q, tokens, ctx_len, n_accepted, next_token, committed_len,
                                workspace, status)
    _on_gpu("uniforms", uniforms, _current_device(), torch.float32, rows)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.load().q3kv_accept_sample(_stream(stream), _ptr(logits), _dtype_code(logits), vocab, _ptr(q_offsets),
                                        _ptr(n_q), _ptr(tokens), n_q.shape[0], rows, max_n_q, _ptr(ctx_len),
                                        float(temperature), _ptr(uniforms), int(seed) & ((1 << 64) - 1),
                                        _ptr(n_accepted), _ptr(next_token), _ptr(committed_len), _ptr(workspace),
                                        nbytes, _ptr(status))
    check(rc, "q3kv_accept_sample")


def accept_sample_nucleus(logits: torch.Tensor, q_offsets: torch.Tensor, n_q: torch.Tensor, tokens: torch.Tensor,
                          max_n_q: int, ctx_len: torch.Tensor, temperature: float, top_p: float,
                          uniforms: torch.Tensor, seed: int, n_accepted: torch.Tensor, next_token: torch.Tensor,
                          committed_len: torch.Tensor, workspace: Optional[torch.Tensor],
                          status: Optional[torch.Tensor] = None, stream=None) -> None:
    """q3kv_accept_sample_nucleus: rejection-sampled acceptance with the top-p nucleus."""
    rows, vocab = _check_accept(logits, q_offsets, n_q, tokens, ctx_len, n_accepted, next_token, committed_len,
                                workspace, status)
    _on_gpu("uniforms", uniforms, _current_device(), torch.float32, rows)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.load().q3kv_accept_sample_nucleus(_stream(stream), _ptr(logits), _dtype_code(logits), vocab,
                                                _ptr(q_offsets), _ptr(n_q), _ptr(tokens), n_q.shape[0], rows,
                                                max_n_q, _ptr(ctx_len), float(temperature), float(top_p),
                                                _ptr(uniforms), int(seed) & ((1 << 64) - 1), _ptr(n_accepted),
                                                _ptr(next_token), _ptr(committed_len), _ptr(workspace), nbytes,
                                                _ptr(status))
    check(rc, "q3kv_accept_sample_nucleus")
