"""Operand-precision ladder of the tensor-core verify leg, emulated in numpy.

The tensor-core leg multiplies fp16 operands (tcgen05 ``kind::f16``) and
accumulates in fp32.  This module emulates the operand choices such a kernel
can make -- every operand rounded once to fp16, or split into fp16 hi/lo pairs
with the leading cross products -- and measures each against the float64
oracle on the seeded workloads.  Products are summed exactly here: what is
studied is the rounding of the operands, which decided the kernel's design
before the kernel existed (a single fp16 operand per side misses the 2e-3 /
1e-3 tolerance on the outlier-heavy workloads; exact K/V pairs and
round-to-nearest Q/P pairs with three products meet it with a wide margin).

The tensor-core leg's own choices, as emulated by ``kernel_q3`` and
``kernel_fp8``:

* Q is rotated and scaled into log2 units (H q / 16 * log2 e), then split into
  round-to-nearest fp16 hi/lo;
* the 3-bit K/V values (c - 3.5) s are split exactly: s_hi = s with its fp16
  mantissa cut to 8 significant bits, s_lo = s - s_hi, so (c - 3.5) s_hi and
  (c - 3.5) s_lo are both exact in fp16;
* S = Qhi.Khi + Qlo.Khi + Qhi.Klo (the Qlo.Klo product is dropped: below
  2^-20 of the scores with the 8-bit K split; a 6-bit K split left it at
  2^-18, which on outlier-heavy queries and keys costs up to 2e-3 of output,
  the ``kernel_q3_k6`` row);
* P = 2^(S - max) in fp32; the row sum is taken from that fp32 P; P is split
  into round-to-nearest fp16 hi/lo and O = Phi.Vhi + Phi.Vlo + Plo.Vhi;
* fp8 E4M3 values are exact in fp16, so that format needs two products per
  contraction (Qhi.K + Qlo.K, Phi.V + Plo.V) and no rotation.

Workloads 3 and 4 draw K, V and Q from workload 2's distributions, so the
ladder runs workloads 1, 2 and 5.  Run it as a script for their full sizes
(minutes of CPU):

    python tests/precision_ladder.py
"""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import q3kv_inputs as qi  # noqa: E402
from oracle import codec, fp8  # noqa: E402
from oracle.wht import rotate_f64  # noqa: E402

LOG2E = 1.0 / np.log(2.0)


def f16(x):
    """Round to fp16 (nearest, ties to even), back to float64."""
    return np.asarray(x, np.float64).astype(np.float16).astype(np.float64)


def split16(x):
    """Round-to-nearest fp16 hi/lo pair of x."""
    hi = f16(x)
    return hi, f16(np.asarray(x, np.float64) - hi)


K_HI_MASK = 0xFFF8   # fp16 bits of s kept in s_hi: 8 significant bits (K and V)
V_HI_MASK = K_HI_MASK
K6_HI_MASK = 0xFFE0  # 6 significant bits: the earlier key split, kept as a ladder row


def exact_split_q3(x_raw, hi_mask=V_HI_MASK):
    """3-bit K or V of raw vectors -> (value, hi, lo) with hi + lo == value exactly.

    s_hi keeps the fp16 bits of the block scale selected by ``hi_mask``.
    """
    codes, s16, _ = codec.encode(x_raw)
    c = codes.astype(np.float64) - 3.5
    s = np.repeat(s16.astype(np.float64), 32, axis=-1)
    s_hi = np.repeat((s16.view(np.uint16) & np.uint16(hi_mask)).view(np.float16).astype(np.float64), 32, axis=-1)
    return c * s, c * s_hi, c * (s - s_hi)


class Case:
    """One (layer, kv head) of a workload's first slot: raw Q rows of the group, K, V."""

    def __init__(self, wkey, layer: int, g: int, n_ctx: int, T: int):
        w = qi.WORKLOADS[wkey] if isinstance(wkey, int) else wkey
        L = n_ctx + T
        self.k_raw = qi.kv_rows(w, 0, layer, g, 0, 0, L)
        self.v_raw = qi.kv_rows(w, 0, layer, g, 1, 0, L)
        q = qi.q_rows(w, 0, layer, 0, T)[:, 8 * g:8 * g + 8, :]
        self.q_raw = q.reshape(T * 8, 256).astype(np.float64)
        tt = np.repeat(np.arange(T), 8)
        self.masked = np.arange(L)[None, :] > (n_ctx + tt)[:, None]


def _softmax_pv(s, masked, v_parts, p_mode):
    """Scores s (log2 units) -> O for one P treatment.

    p_mode "exact": float64 P times v_parts["exact"]; "f16": P rounded once to
    fp16 (row sum of the rounded P) times v_parts["single"]; "split": float32
    P, its row sum, and Phi.Vhi + Plo.Vhi (+ Phi.Vlo when v_parts["lo"] is
    given).
    """
    s = np.where(masked, -np.inf, s)
    p = np.exp2(s - s.max(axis=1, keepdims=True))
    if p_mode == "exact":
        return (p @ v_parts["exact"]) / p.sum(axis=1, keepdims=True)
    p = p.astype(np.float32).astype(np.float64)      # the kernel's P is float32
    if p_mode == "f16":                         # one rounding, row sum of the rounded P
        pr = f16(p)
        return (pr @ v_parts["single"]) / pr.sum(axis=1, keepdims=True)
    phi, plo = split16(p)                       # kernel: fp32 row sum, split P
    o = phi @ v_parts["hi"] + plo @ v_parts["hi"]
    if v_parts.get("lo") is not None:
        o = o + phi @ v_parts["lo"]
    return o / p.sum(axis=1, keepdims=True)


def ladder_q3(case: Case) -> dict:
    """Error of every scheme on the 3-bit cache (rotated basis in, unrotated out)."""
    kv, khi, klo = exact_split_q3(case.k_raw, K_HI_MASK)
    _, khi6, klo6 = exact_split_q3(case.k_raw, K6_HI_MASK)
    vv, vhi, vlo = exact_split_q3(case.v_raw, V_HI_MASK)
    q = rotate_f64(case.q_raw) / 16.0 * LOG2E
    qhi, qlo = split16(q)
    V = {"exact": vv, "single": f16(vv), "hi": vhi, "lo": vlo}
    Vexact = {"exact": vv, "single": vv}
    schemes = {
        "reference": lambda: _softmax_pv(q @ kv.T, case.masked, Vexact, "exact"),
        "all_f16": lambda: _softmax_pv(f16(q) @ f16(kv).T, case.masked, V, "f16"),
        "q_f16": lambda: _softmax_pv(f16(q) @ kv.T, case.masked, Vexact, "exact"),
        "k_f16": lambda: _softmax_pv(q @ f16(kv).T, case.masked, Vexact, "exact"),
        "p_f16": lambda: _softmax_pv(q @ kv.T, case.masked, Vexact, "f16"),
        "v_f16": lambda: _softmax_pv(q @ kv.T, case.masked, {"exact": f16(vv)}, "exact"),
        "kernel_q3": lambda: _softmax_pv(qhi @ khi.T + qlo @ khi.T + qhi @ klo.T, case.masked, V, "split"),
        # the same with K split at 6 significant bits
        "kernel_q3_k6": lambda: _softmax_pv(qhi @ khi6.T + qlo @ khi6.T + qhi @ klo6.T, case.masked, V, "split"),
        # the same with the fourth product Qlo.Klo: what dropping it costs
        "q3_4prod": lambda: _softmax_pv((qhi + qlo) @ kv.T, case.masked, V, "split"),
    }
    return {name: rotate_f64(fn()) for name, fn in schemes.items()}


def ladder_fp8(case: Case) -> dict:
    """Error of the fp8 leg's scheme (plain basis) next to the float64 attention."""
    kv = fp8.decode(fp8.encode_vectors(case.k_raw)[0])
    vv = fp8.decode(fp8.encode_vectors(case.v_raw)[0])
    q = case.q_raw / 16.0 * LOG2E
    qhi, qlo = split16(q)
    return {
        "reference": _softmax_pv(q @ kv.T, case.masked, {"exact": vv}, "exact"),
        "kernel_fp8": _softmax_pv(qhi @ kv.T + qlo @ kv.T, case.masked, {"hi": vv, "lo": None}, "split"),
    }


def errors(results: dict) -> dict:
    """name -> (max-abs, relative L2) against results['reference']."""
    ref = results["reference"]
    out = {}
    for name, o in results.items():
        if name == "reference":
            continue
        e = o - ref
        out[name] = (float(np.abs(e).max()), float(np.linalg.norm(e) / np.linalg.norm(ref)))
    return out


def main():
    """Per workload: layers 0-2, both kv heads; max-abs over them and relative L2 over all rows."""
    for wkey, n_ctx, T in ((1, 1024, 4), (2, 32768, 6), (5, 65536, 8)):
        diffs, refs = {}, []
        for layer in range(3 if qi.WORKLOADS[wkey].num_layers >= 3 else 1):
            for g in range(2):
                case = Case(wkey, layer, g, n_ctx, T)
                for res in (ladder_q3(case), ladder_fp8(case)):
                    ref = res["reference"]
                    if "kernel_q3" in res:
                        refs.append(ref)
                    for name, o in res.items():
                        if name != "reference":
                            diffs.setdefault(name, []).append((o - ref, ref))
        print(f"workload {wkey}, context {n_ctx}, T {T} ({len(refs)} (layer, kv head) cases)")
        for name, pairs in diffs.items():
            e = np.concatenate([d.ravel() for d, _ in pairs])
            r = np.concatenate([x.ravel() for _, x in pairs])
            print(f"  {name:12s} max-abs {np.abs(e).max():.2e}  rel-L2 {np.linalg.norm(e) / np.linalg.norm(r):.2e}")


if __name__ == "__main__":
    main()
