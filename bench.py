"""Benchmark of the q3kv verify step (quantise-append + verify attention).

One step = for each of the workload's layers: q3kv_append of every slot's 1+d
new K/V, then q3kv_verify_attn of the same tokens over the slot's whole cache;
for the continuous-batching workload (--workload 4) one benchmark step is its
whole schedule of 32 such steps over 8 slots, each with its own lengths.
Default workload: the largest one-GPU configuration, 1 slot, 16 layers, 2 kv /
16 q heads, head_dim 256, 655,360 cached positions, 8 query tokens (1 + 7
drafts), bf16 inputs.

Prints one JSON line.  ``value`` = verified tokens/s (sum over slots of 1+d per
step / device time of a step) with the cache and the step's inputs resident on
the device; ``e2e`` = the same metric through the same C-ABI calls with the
step's inputs copied from pinned host memory and the outputs copied back inside
the timed region.  ``roofline`` describes the verify kernel: algorithmic KV
bytes per launch (224 bytes per attended position per kv head; 512 with
``--kv fp8``, the fp8 E4M3 comparison cache) over its mean CUDA-event duration.
``--impl reference`` times the CPU oracle instead.

Multi-GPU: replicas only (one independent replica per rank, no collective on
the data path); ``value`` sums all ranks' tokens over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import q3kv_inputs as qi  # noqa: E402

METRIC = "verified tokens/s and KV HBM GB/s (fraction of GB300 peak) for 3-bit verify attn"
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes (read + write) of the verify kernel per attended position and kv head,
# from ncu captures of the current kernel in this benchmark's launch configuration
# (profiles/); the roofline's traffic is this times the launch's positions.
# Workloads without a capture of the current kernel report null.
NCU_TRAFFIC_BYTES_PER_POSITION = {5: 226.61, 4: 232.06, 3: 228.80, 2: 227.56}
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling captures only: run the workload with this many layers (the line says so)")
    ap.add_argument("--verify-impl", default="auto", choices=["auto", "fma", "mma"])
    ap.add_argument("--split", type=int, default=0, help="positions per split (0 = library policy)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", type=int, default=0,
                    help="instead of the verify step: a fresh prefill of this many tokens (append + prefill "
                         "attention over the 3-bit cache, every layer of the workload, one slot)")
    ap.add_argument("--kv", default="q3", choices=["q3", "fp8", "t5k"],
                    help="cache format: the 3-bit rotated codec, the fp8 E4M3 comparison format, or the "
                         "turbo5k-style 5-bit K / 3-bit V format")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed plumbing
def dist_init(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
        pg = dist
    return rank, world, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x):
    if pg is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.mark_at = 0

    def mark(self):
        """Samples from the one just before this point on describe the timed region."""
        self.mark_at = max(len(self.lines) - 1, 0)

    def wait_samples(self, n, busy, timeout_s=3.0):
        """Call busy() (untimed GPU work that it waits for) until n samples arrived after the mark.

        nvidia-smi reports every 200 ms, longer than a short timed region: keeping
        the GPU loaded until samples arrive makes them describe the clocks under
        the benchmark's own load.  Bounded by timeout_s; never raises.
        """
        if self.proc is None:
            return
        t0 = time.monotonic()
        try:
            while len(self.lines) - self.mark_at < n and time.monotonic() - t0 < timeout_s:
                busy()
        except Exception:
            pass

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.mark_at:]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "200 ms samples from the last one before the timed region through untimed replays "
                          "of the same step right after it"}


_HBM_KEYS = ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs")


def _find_hbm(d, depth=0):
    """First positive HBM copy bandwidth (GB/s) in a peaks record: top-level keys first, then nested ones."""
    if not isinstance(d, dict) or depth > 3:
        return None
    for key in _HBM_KEYS:
        if key in d:
            v = d[key]
            v = v.get("value", v.get("gbs")) if isinstance(v, dict) else v
            try:
                v = float(v)
            except (TypeError, ValueError):
                continue
            if v > 0:
                return v
    for v in d.values():
        found = _find_hbm(v, depth + 1)
        if found is not None:
            return found
    return None


def measured_peak_hbm():
    """(GB/s, "measured") from MEASURED_PEAKS.json next to this file, else the fallback figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                v = _find_hbm(json.load(f))
            if v is not None:
                return v, "measured"
        except (ValueError, OSError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- our arm
class Cache:
    """The workload's paged cache on the device: pool, page table, the slots' cached contexts."""

    def __init__(self, w, device, kv="q3", layers=None):
        import torch

        from speculative_verify_attention_q3kv_gb300 import api

        self.torch, self.api, self.w, self.device = torch, api, w, device
        self.shapes = qi.draw_shapes(w)
        self.S = w.num_slots
        self.layers = layers or w.num_layers
        final = self.shapes.ctx_before(w.steps)            # lengths after the last step
        pages = [(n + 255) // 256 for n in final]
        self.desc = api.make_desc(self.layers, w.num_kv_heads, sum(pages))
        self.kv = kv
        # bytes per position and kv head, K and V together
        self.position_bytes = {"q3": 224, "fp8": 512, "t5k": 164 + 112}[kv]
        self.append_fn = {"q3": api.append, "fp8": api.fp8_append, "t5k": api.t5k_append}[kv]
        self.verify_fn = {"q3": api.verify_attn, "fp8": api.fp8_verify_attn, "t5k": api.t5k_verify_attn}[kv]
        pool_bytes = {"q3": api.pool_bytes, "fp8": api.fp8_pool_bytes, "t5k": api.t5k_pool_bytes}[kv](self.desc)
        self.pool = torch.zeros(pool_bytes, dtype=torch.uint8, device=device)
        pt = np.full((self.S, max(pages)), -1, np.int32)
        k = 0
        for b, n in enumerate(pages):
            pt[b, :n] = np.arange(k, k + n)
            k += n
        self.page_table = torch.from_numpy(pt).to(device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        g = torch.Generator(device=device)
        g.manual_seed(1000 + w.seed)
        self._prefill(g)

    def _prefill(self, g):
        """The slots' cached contexts before the first step (set-up, not timed)."""
        torch, w = self.torch, self.w
        chunk = 32768
        zero = torch.zeros(self.S, dtype=torch.int32, device=self.device)
        for l in range(self.layers):
            for b in range(self.S):
                for start in range(0, self.shapes.ctx[b], chunk):
                    n = min(chunk, self.shapes.ctx[b] - start)
                    kk = torch.empty((n, w.num_kv_heads, w.head_dim), dtype=self.dt, device=self.device)
                    vv = torch.empty_like(kk)
                    for h in range(w.num_kv_heads):
                        qi.torch_fill_kv_(kk[:, h], w, l, h, 0, g)
                        qi.torch_fill_kv_(vv[:, h], w, l, h, 1, g)
                    lens = zero.clone()
                    lens[b] = start
                    nn = zero.clone()
                    nn[b] = n
                    offs = torch.zeros(self.S + 1, dtype=torch.int32, device=self.device)
                    offs[b + 1:] = n
                    self.append_fn(self.desc, self.pool, self.page_table, lens, nn, offs, n, l, kk, vv, self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0, "prefill flagged a device status"


class Step:
    """Inputs and the per-layer append + verify calls of one step (step index s of the workload)."""

    def __init__(self, cache, s, verify_impl, split, ws=None):
        torch, api, w = cache.torch, cache.api, cache.w
        self.torch, self.api, self.w, self.c = torch, api, w, cache
        device = cache.device
        self.ctx = cache.shapes.ctx_before(s)
        self.n_new = cache.shapes.n_new[s]
        self.S = w.num_slots
        self.Ltot = [c + t for c, t in zip(self.ctx, self.n_new)]
        i32 = dict(dtype=torch.int32, device=device)
        self.slot_len = torch.tensor(self.ctx, **i32)
        self.n_new_d = torch.tensor(self.n_new, **i32)
        offs = np.concatenate([[0], np.cumsum(self.n_new)]).astype(np.int32)
        self.row_off = torch.from_numpy(offs).to(device)
        self.ctx_len = torch.tensor(self.Ltot, **i32)
        self.rows = int(offs[-1])
        self.max_new = max(self.n_new)
        self.max_ctx = max(self.Ltot)
        self.impl = {"auto": 0, "fma": 1, "mma": 2}[verify_impl]
        self.split = split
        self.ws = ws if ws is not None else torch.zeros(
            api.workspace_bytes(cache.desc, self.S, self.max_ctx, self.max_new, self.impl, split),
            dtype=torch.uint8, device=device)
        self.status = cache.status
        H, Hq, D, Ly = w.num_kv_heads, w.num_q_heads, w.head_dim, cache.layers
        g = torch.Generator(device=device)
        g.manual_seed(3000 + 97 * w.seed + s)
        # step inputs: new K, V [layers, rows, H, D]; Q [layers, rows, Hq, D]
        self.k_new = torch.empty((Ly, self.rows, H, D), dtype=cache.dt, device=device)
        self.v_new = torch.empty_like(self.k_new)
        self.q = (torch.randn((Ly, self.rows, Hq, D), generator=g, device=device)).to(cache.dt)
        for l in range(Ly):
            for h in range(H):
                qi.torch_fill_kv_(self.k_new[l, :, h], w, l, h, 0, g)
                qi.torch_fill_kv_(self.v_new[l, :, h], w, l, h, 1, g)
        self.out = torch.empty((Ly, self.rows, Hq, D), dtype=torch.float32, device=device)

    def kv_bytes_per_layer(self):
        return sum(self.Ltot) * self.w.num_kv_heads * self.c.position_bytes

    def run(self, append=True, verify=True):
        """One step: for every layer, append the new K/V then verify the new tokens."""
        c = self.c
        for l in range(c.layers):
            if append:
                c.append_fn(c.desc, c.pool, c.page_table, self.slot_len, self.n_new_d, self.row_off,
                            self.max_new, l, self.k_new[l], self.v_new[l], self.status)
            if verify:
                c.verify_fn(c.desc, c.pool, c.page_table, self.ctx_len, self.n_new_d, self.row_off,
                            self.max_ctx, self.max_new, l, self.q[l], self.out[l], self.ws, self.impl,
                            self.split, self.status)

    def launches_per_layer(self):
        """Our kernels per layer: append; for the tensor-core leg the query kernel and the verify
        kernel (the CUDA-core leg: the verify kernel); the split merge when the context is split,
        which is when the workspace holds split partials beyond the tensor-core leg's queries."""
        mma = self.impl != 1
        units = self.S * self.w.num_kv_heads * ((8 * self.max_new + 63) // 64)
        query_bytes = units * 2 * 64 * 256 * 2 if mma else 0
        need = self.api.workspace_bytes(self.c.desc, self.S, self.max_ctx, self.max_new, self.impl, self.split)
        return 1 + (2 if mma else 1) + (1 if need > query_bytes else 0)


class Acceptance:
    """Synthetic logits of one step's query tokens and the acceptance calls (a Qwen-class vocabulary)."""

    def __init__(self, st):
        torch, api, w = st.torch, st.api, st.w
        device = st.c.device
        self.st, self.api = st, api
        i32 = dict(dtype=torch.int32, device=device)
        g = torch.Generator(device=device)
        g.manual_seed(5000 + w.seed)
        self.vocab = qi.VOCAB
        self.rows = st.rows
        self.logits = torch.randn((st.rows, self.vocab), generator=g, device=device).to(torch.bfloat16)
        self.tokens = torch.from_numpy(qi.random_tokens(w.seed, st.rows, self.vocab)).to(device)
        # outputs kept apart so the lengths stay fixed between steps
        self.n_acc = torch.zeros(st.S, **i32)
        self.next_tok = torch.zeros(st.S, **i32)
        self.committed = torch.zeros(st.S, **i32)
        self.ws = torch.empty(max(api.accept_workspace_bytes(st.rows, self.vocab), 8), dtype=torch.uint8,
                              device=device)
        self.uniforms = torch.rand(st.rows, generator=g, device=device)

    def greedy(self):
        st = self.st
        self.api.accept_greedy(self.logits, st.row_off, st.n_new_d, self.tokens, st.max_new, st.ctx_len,
                               self.n_acc, self.next_tok, self.committed, self.ws, st.status)

    def nucleus(self, temperature=1.0, top_p=0.95):
        """Sampled acceptance with the top-p nucleus (the model card's temperature 1.0, top-p 0.95)."""
        st = self.st
        self.api.accept_sample_nucleus(self.logits, st.row_off, st.n_new_d, self.tokens, st.max_new,
                                       st.ctx_len, temperature, top_p, self.uniforms, 1234, self.n_acc,
                                       self.next_tok, self.committed, self.ws, st.status)


def capture(fn):
    """fn's launches as one CUDA graph (no host launch gaps when replayed)."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                                   # warm the launch path on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    torch.cuda.synchronize()
    return graph


def _timed(stream, reps, body, flush):
    """Device milliseconds of body() per repetition, L2 flushed before each (outside the events)."""
    import torch

    out = []
    for _ in range(reps):
        flush.zero_()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        body()
        b_.record(stream)
        out.append((a, b_))
    return out


def run_ours(args, rank, world, local, pg):
    import torch

    from speculative_verify_attention_q3kv_gb300 import build as b

    b.build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = qi.WORKLOADS[args.workload]
    cache = Cache(w, device, kv=args.kv, layers=args.layers)
    Ly = cache.layers
    # one benchmark step = the workload's whole schedule: one verify step, or (continuous
    # batching) every one of its append + verify steps in order, each with its own lengths
    last = Step(cache, w.steps - 1, args.verify_impl, args.split)
    steps = [Step(cache, s, args.verify_impl, args.split, ws=last.ws) for s in range(w.steps - 1)] + [last]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    tokens_per_step = sum(sum(st.n_new) for st in steps)

    for _ in range(max(args.warmup, 3)):
        for st in steps:
            st.run()
    torch.cuda.synchronize()
    # each step, and its verify calls alone (for the per-launch roofline), as CUDA graphs
    g_steps = [capture(st.run) for st in steps]
    g_verify = [capture(lambda st=st: st.run(append=False)) for st in steps]
    acc = Acceptance(steps[0])
    g_accept = capture(acc.greedy)
    g_nucleus = capture(acc.nucleus)

    def whole_step():
        for g_ in g_steps:
            g_.replay()

    def whole_verify():
        for g_ in g_verify:
            g_.replay()

    for _ in range(max(args.warmup, 3)):
        whole_step()
        whole_verify()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)

    def busy():                             # untimed load while the clock samples arrive
        for _ in range(max(1, 8 // len(g_steps))):
            whole_step()
        torch.cuda.synchronize()

    clocks.start()
    clocks.wait_samples(1, busy)
    barrier(pg)
    torch.cuda.synchronize()
    clocks.mark()
    ev = _timed(stream, args.steps, whole_step, flush)
    vev = _timed(stream, args.steps, whole_verify, flush)     # the steps' verify calls back to back
    aev = _timed(stream, args.steps, g_accept.replay, flush)  # acceptance (argmax + acceptance kernels)
    nev = _timed(stream, args.steps, g_nucleus.replay, flush)  # sampled acceptance with the top-p nucleus
    torch.cuda.synchronize()
    clocks.wait_samples(3, busy)
    clock_info = clocks.stop()
    barrier(pg)
    step_ms = [a.elapsed_time(b_) for a, b_ in ev]
    accept_us = statistics.mean(a.elapsed_time(b_) for a, b_ in aev) * 1e3
    nucleus_us = statistics.mean(a.elapsed_time(b_) for a, b_ in nev) * 1e3
    n_verify = Ly * len(steps)                                 # verify calls per benchmark step
    verify_ms = [a.elapsed_time(b_) for a, b_ in vev]
    total_s = max_over_ranks(pg, sum(step_ms) / 1e3)
    assert int(cache.status.item()) == 0, "device status flagged during the benchmark"

    # ---- end to end: inputs from pinned host memory, outputs back to host, inside the timed region
    e2e = None
    if not args.no_e2e:
        host = [(st.k_new.cpu().pin_memory(), st.v_new.cpu().pin_memory(), st.q.cpu().pin_memory(),
                 torch.empty(st.out.shape, dtype=torch.float32).pin_memory()) for st in steps]
        e_ms = []
        for s in range(max(args.warmup, 3) + args.steps):
            flush.zero_()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for st, g_, (hk, hv, hq, ho) in zip(steps, g_steps, host):
                # the step's inputs arrive from pinned host memory into the buffers the graph reads
                st.k_new.copy_(hk, non_blocking=True)
                st.v_new.copy_(hv, non_blocking=True)
                st.q.copy_(hq, non_blocking=True)
                g_.replay()
                ho.copy_(st.out, non_blocking=True)
            b_.record(stream)
            torch.cuda.synchronize()
            if s >= max(args.warmup, 3):
                e_ms.append(a.elapsed_time(b_))
        e2e_s = max_over_ranks(pg, sum(e_ms) / 1e3)
        h2d = sum(t.numel() * t.element_size() for hk, hv, hq, _ in host for t in (hk, hv, hq))
        d2h = sum(ho.numel() * ho.element_size() for *_, ho in host)
        e2e = {"value": world * tokens_per_step * args.steps / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    if rank != 0:
        return
    peak, peak_kind = measured_peak_hbm()
    kv_bytes_step = sum(st.kv_bytes_per_layer() for st in steps) * Ly      # per benchmark step, all layers
    mean_verify_s = statistics.mean(verify_ms) / 1e3 / n_verify               # per verify call
    kv_bytes = kv_bytes_step / n_verify                                        # per verify call (mean)
    achieved = kv_bytes / mean_verify_s / 1e9
    cpu = None
    if not args.no_cpu_baseline and world == 1 and args.kv == "q3" and args.layers is None:
        cpu = cpu_baseline(w, budget_s=20.0)
    traffic = None
    if args.verify_impl == "auto" and args.kv == "q3" and args.split == 0:
        per_pos = NCU_TRAFFIC_BYTES_PER_POSITION.get(w.key)
        if per_pos is not None:
            traffic = per_pos * kv_bytes / 224.0          # kv_bytes / 224 = attended (position, kv head) pairs
    ctxs = [st.ctx for st in steps]
    news = [st.n_new for st in steps]
    line = {
        "metric": METRIC,
        "value": world * tokens_per_step * args.steps / total_s,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": total_s * 1e3 / args.steps,
        "ms_per_step_median": statistics.median(step_ms),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; K,V per-channel 10^U(0,1) outliers, Q N(0,1))" if w.kv_dist == "loguniform10"
                else "synthetic (seeded; K,V N(0,1) with 4 outlier channels x8)",
        "config": {"workload": (w.name if args.kv == "q3" else w.name + "_" + args.kv + "kv")
                               + ("" if args.layers is None else f"_profile{Ly}layer"),
                   "kv_format": {"q3": "q3kv 3-bit WHT, 112 B per head vector",
                                 "fp8": "fp8 e4m3, 256 B per head vector",
                                 "t5k": "turbo5k-style: 5-bit Lloyd-Max K 164 B + 3-bit V 112 B"}[args.kv],
                   "slots": w.num_slots, "layers": Ly, "kv_heads": w.num_kv_heads,
                   "q_heads": w.num_q_heads, "head_dim": w.head_dim,
                   "ctx": ctxs[0] if len(steps) == 1 else ctxs,
                   "query_tokens": news[0] if len(steps) == 1 else news,
                   "steps_per_benchmark_step": len(steps),
                   "page_size": 256, "verify_impl": args.verify_impl, "split_positions": args.split,
                   "l2": "flushed between timed steps (256 MiB write)", "launch": "CUDA graph per step",
                   "parallelism": f"replicas{world}"},
        "kv_gbs": kv_bytes_step * args.steps / (sum(verify_ms) / 1e3) / 1e9,
        "verify_only_tokens_per_s": tokens_per_step * args.steps / (sum(verify_ms) / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "q3kv_verify_attn per layer (query + verify + split-merge kernels)",
                     "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": kv_bytes,
                     "mean_launch_us": mean_verify_s * 1e6},
        "accept": {"us": accept_us, "vocab": acc.vocab, "logits_bytes": acc.rows * acc.vocab * 2,
                   "gbs": acc.rows * acc.vocab * 2 / (accept_us * 1e-6) / 1e9,
                   "kernel": "q3kv_accept_greedy (argmax + acceptance kernels), bf16 logits, once per step",
                   "sampled_top_p_us": nucleus_us,
                   "sampled_top_p_kernel": "q3kv_accept_sample_nucleus (temperature 1.0, top-p 0.95): max, "
                                           "radix select of the cut (2 levels), nucleus Gumbel-max, acceptance"},
        "clocks": clock_info,
        "gpu_launches": args.steps * Ly * sum(st.launches_per_layer() for st in steps),
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- oracle (CPU) arm
ORACLE_WINDOW = 16384          # cached positions per slot the oracle's timed sample attends over
_ORACLE_SETUP = {}


def _oracle_setup(w, layer, step, window):
    """Untimed set-up of the oracle's sample: each slot's last min(N, window) cached positions.

    Positions keep their own seeded values (the slot's streams at [N - n, N)); they sit at
    positions [0, n) of a small paged cache, so the timed part appends the step's tokens at n.
    """
    from oracle.cache import PagedCache

    key = (w.key, layer, step, window)
    if key in _ORACLE_SETUP:
        return _ORACLE_SETUP[key]
    _ORACLE_SETUP.clear()
    shapes = qi.draw_shapes(w)
    ctx, news = shapes.ctx_before(step), shapes.n_new[step]
    held = [min(n, window) for n in ctx]
    pages = [(h + t + 255) // 256 for h, t in zip(held, news)]
    pt = np.full((w.num_slots, max(pages)), -1, np.int32)
    k = 0
    for b, n in enumerate(pages):
        pt[b, :n] = np.arange(k, k + n)
        k += n
    cache = PagedCache(sum(pages), 1, w.num_kv_heads)
    for b in range(w.num_slots):
        kk = np.stack([qi.kv_rows(w, b, layer, g, 0, ctx[b] - held[b], held[b]) for g in range(w.num_kv_heads)], axis=1)
        vv = np.stack([qi.kv_rows(w, b, layer, g, 1, ctx[b] - held[b], held[b]) for g in range(w.num_kv_heads)], axis=1)
        cache.append(pt[b], 0, 0, kk, vv)
    out = (cache, pt, ctx, news, held)
    _ORACLE_SETUP[key] = out
    return out


def _oracle_step_sample(w, layer, step=0, window=ORACLE_WINDOW):
    """The oracle's append + verify of one layer of one step, every slot: (tokens, seconds, scaled).

    The append of the step's tokens is timed as it is; each slot's verify attends over its
    held window plus the new tokens and its time is scaled by (N + T) / (held + T), the ratio of
    attended positions (the verify's cost is linear in them).
    """
    cache, pt, ctx, news, held = _oracle_setup(w, layer, step, window)
    total = 0.0
    for b in range(w.num_slots):
        n, T, h = ctx[b], news[b], held[b]
        kk = np.stack([qi.kv_rows(w, b, layer, g, 0, n, T) for g in range(w.num_kv_heads)], axis=1)
        vv = np.stack([qi.kv_rows(w, b, layer, g, 1, n, T) for g in range(w.num_kv_heads)], axis=1)
        q = qi.q_rows(w, b, layer, step, T)
        t0 = time.perf_counter()
        cache.append(pt[b], h, 0, kk, vv)
        t1 = time.perf_counter()
        cache.verify(pt[b], 0, h, q, w.group)
        t2 = time.perf_counter()
        total += (t1 - t0) + (t2 - t1) * (n + T) / (h + T)
    return sum(news), total


def _sample_text(w, window):
    scaled = any(n > window for n in qi.draw_shapes(w).ctx_before(w.steps - 1))
    return (f"one layer of {'step 0 of the ' + str(w.steps) + '-step schedule' if w.steps > 1 else 'the step'} "
            f"(append + verify of every slot); " +
            (f"each slot's verify attends over its last {window} cached positions plus the new tokens and "
             f"its time is scaled by the ratio of attended positions; " if scaled else "") +
            f"counted for all {w.num_layers} layers" + (f" and {w.steps} steps" if w.steps > 1 else "") +
            "; set-up (encoding the cached context) not timed")


def cpu_baseline(w, budget_s=20.0):
    spent, n = 0.0, 0
    while spent < budget_s and n < 8:
        tok, dt = _oracle_step_sample(w, 0)
        spent += dt
        n += 1
    per_layer = spent / n
    return {"value": tok / (per_layer * w.num_layers), "unit": "tokens/s", "cores": _threads(),
            "host_cpus": os.cpu_count(), "blas_threads": _blas_threads(), "kind": "oracle",
            "sample": _sample_text(w, ORACLE_WINDOW) + f"; mean of {n} repetitions"}


def _blas_threads():
    """Threads of the BLAS numpy calls into (None where threadpoolctl is not installed)."""
    try:
        import threadpoolctl

        return int(max((p.get("num_threads", 1) for p in threadpoolctl.threadpool_info()), default=1))
    except Exception:
        return None


def _threads():
    n = _blas_threads()
    return n if n is not None else (os.cpu_count() or 1)


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = qi.WORKLOADS[args.workload]
    shapes = qi.draw_shapes(w)
    times = []
    for s in range(max(args.warmup, 3) + args.steps):
        tok, dt = _oracle_step_sample(w, 0)
        if s >= max(args.warmup, 3):
            # one sampled layer of one step stands for all layers and all steps of the schedule
            times.append(dt * w.num_layers * w.steps)
    tok_step = sum(sum(t) for t in shapes.n_new)
    total = sum(times)
    value = tok_step * args.steps / total
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": total * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "slots": w.num_slots, "layers": w.num_layers, "ctx": shapes.ctx,
                       "query_tokens": shapes.n_new[0] if w.steps == 1 else shapes.n_new,
                       "steps_per_benchmark_step": w.steps},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _threads(), "host_cpus": os.cpu_count(),
                             "blas_threads": _blas_threads(), "kind": "oracle",
                             "sample": _sample_text(w, ORACLE_WINDOW)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_prefill(args, rank, world, local, pg):
    """A fresh prefill of args.prefill tokens per layer: quantise-append, then causal attention."""
    import torch

    from speculative_verify_attention_q3kv_gb300 import api
    from speculative_verify_attention_q3kv_gb300 import build as b

    b.build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = qi.WORKLOADS[args.workload]
    T, Ly, H, Hq = args.prefill, w.num_layers, w.num_kv_heads, w.num_q_heads
    pages = (T + 255) // 256
    desc = api.make_desc(Ly, H, pages)
    pool = torch.zeros(api.pool_bytes(desc), dtype=torch.uint8, device=device)
    i32 = dict(dtype=torch.int32, device=device)
    pt = torch.arange(pages, **i32)[None]
    zero, n_new, offs, ctx = (torch.tensor([0], **i32), torch.tensor([T], **i32), torch.tensor([0, T], **i32),
                              torch.tensor([T], **i32))
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(2000 + w.seed)
    k = torch.empty((Ly, T, H, 256), dtype=dt, device=device)
    v = torch.empty_like(k)
    for l in range(Ly):
        for h in range(H):
            qi.torch_fill_kv_(k[l, :, h], w, l, h, 0, g)
            qi.torch_fill_kv_(v[l, :, h], w, l, h, 1, g)
    q = torch.randn((Ly, T, Hq, 256), generator=g, device=device).to(dt)
    out = torch.empty((Ly, T, Hq, 256), dtype=torch.float32, device=device)
    impl = {"auto": 0, "fma": 1, "mma": 2}[args.verify_impl]
    ws = torch.zeros(max(api.prefill_workspace_bytes(desc, 1, T, T, impl, args.split), 16), dtype=torch.uint8,
                     device=device)
    status = torch.zeros(1, **i32)

    def step(append=True):
        for l in range(Ly):
            if append:
                api.append(desc, pool, pt, zero, n_new, offs, T, l, k[l], v[l], status)
            api.prefill_attn(desc, pool, pt, ctx, n_new, offs, T, T, l, q[l], out[l], ws, impl, args.split, status)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    aev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)

    def busy():                             # untimed load while the clock samples arrive
        step()
        torch.cuda.synchronize()

    clocks.start()
    clocks.wait_samples(1, busy)
    barrier(pg)
    torch.cuda.synchronize()
    clocks.mark()
    for s_ in range(args.steps):
        flush.zero_()
        ev[s_][0].record()
        step()
        ev[s_][1].record()
    for s_ in range(args.steps):
        flush.zero_()
        aev[s_][0].record()
        step(append=False)
        aev[s_][1].record()
    torch.cuda.synchronize()
    clocks.wait_samples(3, busy)
    clock_info = clocks.stop()
    barrier(pg)
    assert int(status.item()) == 0, "device status flagged during the prefill benchmark"
    total_s = max_over_ranks(pg, sum(a.elapsed_time(b_) for a, b_ in ev) / 1e3)
    attn_s = sum(a.elapsed_time(b_) for a, b_ in aev) / 1e3
    if rank != 0:
        return
    # causal rows: token t reads t + 1 positions of 224 bytes per kv head
    attended = H * T * (T + 1) // 2
    line = {"metric": "prefill tokens/s (append + causal prefill attention over the 3-bit cache, all layers)",
            "value": world * T * args.steps / total_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": total_s * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
            "data": "synthetic (seeded, the workload's K/V distributions)",
            "config": {"workload": f"prefill{T}_{Ly}layer", "layers": Ly, "kv_heads": H, "q_heads": Hq,
                       "new_tokens": T, "context_before": 0, "verify_impl": args.verify_impl,
                       "l2": "flushed between timed steps (256 MiB write)", "launch": "stream (no graph)"},
            "attention_us_per_layer": attn_s * 1e6 / (args.steps * Ly),
            "attention_only_tokens_per_s": T * args.steps / attn_s,
            "attended_kv_bytes_per_layer": attended * 224,
            "clocks": clock_info, "e2e": None, "cpu_baseline": None}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local, pg = dist_init(args.gpus)
    if args.prefill and args.impl != "reference":
        run_prefill(args, rank, world, local, pg)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
