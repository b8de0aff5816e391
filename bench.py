"""Benchmark of the q3kv verify step (quantise-append + verify attention).

One step = for each of the workload's layers: q3kv_append of every slot's 1+d
new K/V, then q3kv_verify_attn of the same tokens over the slot's whole cache.
Default workload: 1 slot, 16 layers, 2 kv / 16 q heads, head_dim 256, 32,768
cached positions, 6 query tokens (1 + 5 drafts), bf16 inputs.

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
# DRAM bytes (read + write) of one verify-kernel launch, from one ncu capture of
# this benchmark's launch configuration (profiles/verify_mma_workload2_ctx32768_t6.md);
# workloads without a capture of the current kernel report null.
NCU_TRAFFIC_BYTES = {2: 14988288}
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 5])
    ap.add_argument("--verify-impl", default="auto", choices=["auto", "fma", "mma"])
    ap.add_argument("--split", type=int, default=0, help="positions per split (0 = library policy)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", type=int, default=0,
                    help="instead of the verify step: a fresh prefill of this many tokens (append + prefill "
                         "attention over the 3-bit cache, every layer of the workload, one slot)")
    ap.add_argument("--kv", default="q3", choices=["q3", "fp8", "t5k"],
                    help="cache format: the 3-bit rotated codec, the fp8 E4M3 comparison format, or the "
                         "turbo5k-style 5-bit K / 3-bit V format (CUDA-core leg)")
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
class Step:
    """Device buffers and the per-layer append + verify calls of one workload step."""

    def __init__(self, w, verify_impl, split, device, kv="q3"):
        import torch

        from speculative_verify_attention_q3kv_gb300 import api

        self.torch = torch
        self.api = api
        self.w = w
        shapes = qi.draw_shapes(w)
        self.ctx = shapes.ctx
        self.n_new = shapes.n_new[0]
        self.S = w.num_slots
        self.Ltot = [c + t for c, t in zip(self.ctx, self.n_new)]
        pages = [(n + 255) // 256 for n in self.Ltot]
        self.num_pages = sum(pages)
        self.desc = api.make_desc(w.num_layers, w.num_kv_heads, self.num_pages)
        self.fp8 = kv == "fp8"
        # bytes per position and kv head, K and V together
        self.position_bytes = {"q3": 224, "fp8": 512, "t5k": 164 + 112}[kv]
        self._append = {"q3": api.append, "fp8": api.fp8_append, "t5k": api.t5k_append}[kv]
        self._verify = {"q3": api.verify_attn, "fp8": api.fp8_verify_attn, "t5k": api.t5k_verify_attn}[kv]
        pool_bytes = {"q3": api.pool_bytes, "fp8": api.fp8_pool_bytes, "t5k": api.t5k_pool_bytes}[kv](self.desc)
        self.pool = torch.zeros(pool_bytes, dtype=torch.uint8, device=device)
        pt = np.full((self.S, max(pages)), -1, np.int32)
        k = 0
        for b, n in enumerate(pages):
            pt[b, :n] = np.arange(k, k + n)
            k += n
        self.page_table = torch.from_numpy(pt).to(device)
        i32 = dict(dtype=torch.int32, device=device)
        self.slot_len = torch.tensor(self.ctx, **i32)
        self.n_new_d = torch.tensor(self.n_new, **i32)
        offs = np.concatenate([[0], np.cumsum(self.n_new)]).astype(np.int32)
        self.row_off = torch.from_numpy(offs).to(device)
        self.ctx_len = torch.tensor(self.Ltot, **i32)
        self.rows = int(offs[-1])
        self.max_new = max(self.n_new)
        self.max_ctx = max(self.Ltot)
        self.dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        self.impl = {"auto": 0, "fma": 1, "mma": 2}[verify_impl]
        if kv == "t5k":
            self.impl = 1                      # the turbo5k-style cache is read by the CUDA-core leg
        self.split = split
        self.ws = torch.zeros(api.workspace_bytes(self.desc, self.S, self.max_ctx, self.max_new, self.impl, split),
                              dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, **i32)
        self.device = device
        H, Hq, D, Ly = w.num_kv_heads, w.num_q_heads, w.head_dim, w.num_layers
        g = torch.Generator(device=device)
        g.manual_seed(1000 + w.seed)
        # step inputs: new K, V [layers, rows, H, D]; Q [layers, rows, Hq, D]
        self.k_new = torch.empty((Ly, self.rows, H, D), dtype=self.dt, device=device)
        self.v_new = torch.empty_like(self.k_new)
        self.q = (torch.randn((Ly, self.rows, Hq, D), generator=g, device=device)).to(self.dt)
        for l in range(Ly):
            for h in range(H):
                qi.torch_fill_kv_(self.k_new[l, :, h], w, l, h, 0, g)
                qi.torch_fill_kv_(self.v_new[l, :, h], w, l, h, 1, g)
        self.out = torch.empty((Ly, self.rows, Hq, D), dtype=torch.float32, device=device)
        # acceptance after the step: synthetic logits of the step's query tokens, a
        # Qwen-class vocabulary; outputs kept apart so the lengths stay fixed between steps
        self.vocab = qi.VOCAB
        self.logits = torch.randn((self.rows, self.vocab), generator=g, device=device).to(torch.bfloat16)
        self.tokens = torch.from_numpy(qi.random_tokens(w.seed, self.rows, self.vocab)).to(device)
        self.n_acc = torch.zeros(self.S, **i32)
        self.next_tok = torch.zeros(self.S, **i32)
        self.committed = torch.zeros(self.S, **i32)
        self.accept_ws = torch.empty(max(api.accept_workspace_bytes(self.rows, self.vocab), 8), dtype=torch.uint8,
                                     device=device)
        self.uniforms = torch.rand(self.rows, generator=g, device=device)
        self._prefill(g)

    def _prefill(self, g):
        torch, api, w = self.torch, self.api, self.w
        chunk = 32768
        zero = torch.zeros(self.S, dtype=torch.int32, device=self.device)
        for l in range(w.num_layers):
            for b in range(self.S):
                for start in range(0, self.ctx[b], chunk):
                    n = min(chunk, self.ctx[b] - start)
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
                    self._append(self.desc, self.pool, self.page_table, lens, nn, offs, n, l, kk, vv, self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0, "prefill flagged a device status"

    def kv_bytes_per_layer(self):
        return sum(self.Ltot) * self.w.num_kv_heads * self.position_bytes

    def run(self, append=True, verify=True):
        """One step: for every layer, append the new K/V then verify the new tokens."""
        api = self.api
        for l in range(self.w.num_layers):
            if append:
                self._append(self.desc, self.pool, self.page_table, self.slot_len, self.n_new_d, self.row_off,
                             self.max_new, l, self.k_new[l], self.v_new[l], self.status)
            if verify:
                self._verify(self.desc, self.pool, self.page_table, self.ctx_len, self.n_new_d, self.row_off,
                             self.max_ctx, self.max_new, l, self.q[l], self.out[l], self.ws, self.impl,
                             self.split, self.status)

    def accept(self):
        """Greedy acceptance of the step's drafts and the committed lengths (once per step)."""
        self.api.accept_greedy(self.logits, self.row_off, self.n_new_d, self.tokens, self.max_new, self.ctx_len,
                               self.n_acc, self.next_tok, self.committed, self.accept_ws, self.status)

    def accept_nucleus(self, temperature=1.0, top_p=0.95):
        """Sampled acceptance with the top-p nucleus (the model card's temperature 1.0, top-p 0.95)."""
        self.api.accept_sample_nucleus(self.logits, self.row_off, self.n_new_d, self.tokens, self.max_new,
                                       self.ctx_len, temperature, top_p, self.uniforms, 1234, self.n_acc,
                                       self.next_tok, self.committed, self.accept_ws, self.status)

    def launches_per_layer(self):
        """Our kernels per layer: append; for the tensor-core leg the query kernel and the verify
        kernel (the CUDA-core leg: the verify kernel); the split merge when the context is split,
        which is when the workspace holds split partials beyond the tensor-core leg's queries."""
        mma = self.impl != 1
        units = self.S * self.w.num_kv_heads * ((8 * self.max_new + 63) // 64)
        query_bytes = units * 2 * 64 * 256 * 2 if mma else 0
        split = self.ws.numel() > query_bytes
        return 1 + (2 if mma else 1) + (1 if split else 0)

    def capture(self, fn=None, **kw):
        """The step's launches (or fn's) as one CUDA graph (no host launch gaps when replayed)."""
        torch = self.torch
        fn = fn or (lambda: self.run(**kw))
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()                               # warm the launch path on the capture stream
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        torch.cuda.synchronize()
        return graph


def run_ours(args, rank, world, local, pg):
    import torch

    from speculative_verify_attention_q3kv_gb300 import build as b

    b.build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = qi.WORKLOADS[args.workload]
    st = Step(w, args.verify_impl, args.split, device, kv=args.kv)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    tokens_per_step = sum(st.n_new)
    Ly = w.num_layers

    for _ in range(max(args.warmup, 3)):
        st.run()
    torch.cuda.synchronize()
    # the step, and its verify calls alone (for the per-launch roofline), as CUDA graphs
    g_step = st.capture()
    g_verify = st.capture(append=False)
    g_accept = st.capture(st.accept)
    g_nucleus = st.capture(st.accept_nucleus)
    for _ in range(max(args.warmup, 3)):
        g_step.replay()
        g_verify.replay()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    vev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)

    def busy():                             # untimed load while the clock samples arrive
        for _ in range(8):
            g_step.replay()
        torch.cuda.synchronize()

    clocks.start()
    clocks.wait_samples(1, busy)
    barrier(pg)
    torch.cuda.synchronize()
    clocks.mark()
    for s in range(args.steps):
        flush.zero_()                       # L2 flush between timed steps (outside the events)
        ev[s][0].record(stream)
        g_step.replay()
        ev[s][1].record(stream)
    for s in range(args.steps):
        flush.zero_()
        vev[s][0].record(stream)
        g_verify.replay()                   # the step's Ly verify calls back to back
        vev[s][1].record(stream)
    aev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for s in range(args.steps):
        flush.zero_()
        aev[s][0].record(stream)
        g_accept.replay()                   # the step's acceptance (argmax + acceptance kernels)
        aev[s][1].record(stream)
    nev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for s in range(args.steps):
        flush.zero_()
        nev[s][0].record(stream)
        g_nucleus.replay()                  # sampled acceptance with the top-p nucleus
        nev[s][1].record(stream)
    torch.cuda.synchronize()
    clocks.wait_samples(3, busy)
    clock_info = clocks.stop()
    barrier(pg)
    step_ms = [a.elapsed_time(b_) for a, b_ in ev]
    accept_us = statistics.mean(a.elapsed_time(b_) for a, b_ in aev) * 1e3
    nucleus_us = statistics.mean(a.elapsed_time(b_) for a, b_ in nev) * 1e3
    verify_ms = [a.elapsed_time(b_) / Ly for a, b_ in vev for _ in range(Ly)]   # per verify call
    total_s = max_over_ranks(pg, sum(step_ms) / 1e3)
    assert int(st.status.item()) == 0, "device status flagged during the benchmark"

    # ---- end to end: inputs from pinned host memory, outputs back to host, inside the timed region
    e2e = None
    if not args.no_e2e:
        hk = st.k_new.cpu().pin_memory()
        hv = st.v_new.cpu().pin_memory()
        hq = st.q.cpu().pin_memory()
        ho = torch.empty(st.out.shape, dtype=torch.float32).pin_memory()
        e_ms = []
        for s in range(max(args.warmup, 3) + args.steps):
            flush.zero_()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            # the step's inputs arrive from pinned host memory into the buffers the graph reads
            st.k_new.copy_(hk, non_blocking=True)
            st.v_new.copy_(hv, non_blocking=True)
            st.q.copy_(hq, non_blocking=True)
            g_step.replay()
            ho.copy_(st.out, non_blocking=True)
            b_.record(stream)
            torch.cuda.synchronize()
            if s >= max(args.warmup, 3):
                e_ms.append(a.elapsed_time(b_))
        e2e_s = max_over_ranks(pg, sum(e_ms) / 1e3)
        h2d = hk.numel() * hk.element_size() + hv.numel() * hv.element_size() + hq.numel() * hq.element_size()
        d2h = ho.numel() * ho.element_size()
        e2e = {"value": world * tokens_per_step * args.steps / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    if rank != 0:
        return
    peak, peak_kind = measured_peak_hbm()
    mean_verify_s = statistics.mean(verify_ms) / 1e3
    kv_bytes = st.kv_bytes_per_layer()
    achieved = kv_bytes / mean_verify_s / 1e9
    cpu = None
    if not args.no_cpu_baseline and world == 1 and args.kv == "q3":
        cpu = cpu_baseline(w, budget_s=20.0)
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
        "config": {"workload": w.name if args.kv == "q3" else w.name + "_" + args.kv + "kv",
                   "kv_format": {"q3": "q3kv 3-bit WHT, 112 B per head vector",
                                 "fp8": "fp8 e4m3, 256 B per head vector",
                                 "t5k": "turbo5k-style: 5-bit Lloyd-Max K 164 B + 3-bit V 112 B"}[args.kv],
                   "slots": w.num_slots, "layers": Ly, "kv_heads": w.num_kv_heads,
                   "q_heads": w.num_q_heads, "head_dim": w.head_dim, "ctx": st.ctx, "query_tokens": st.n_new,
                   "page_size": 256, "verify_impl": args.verify_impl, "split_positions": args.split,
                   "l2": "flushed between timed steps (256 MiB write)", "launch": "CUDA graph per step",
                   "parallelism": f"replicas{world}"},
        "kv_gbs": kv_bytes * Ly * args.steps / (sum(verify_ms) / 1e3) / 1e9,
        "verify_only_tokens_per_s": tokens_per_step * args.steps / (sum(verify_ms) / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": NCU_TRAFFIC_BYTES.get(w.key) if args.verify_impl == "auto" and args.kv == "q3" else None,
                     "kernel": "q3kv_verify_attn per layer (query + verify + split-merge kernels)",
                     "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": kv_bytes,
                     "mean_launch_us": mean_verify_s * 1e6},
        "accept": {"us": accept_us, "vocab": st.vocab, "logits_bytes": st.rows * st.vocab * 2,
                   "gbs": st.rows * st.vocab * 2 / (accept_us * 1e-6) / 1e9,
                   "kernel": "q3kv_accept_greedy (argmax + acceptance kernels), bf16 logits, once per step",
                   "sampled_top_p_us": nucleus_us,
                   "sampled_top_p_kernel": "q3kv_accept_sample_nucleus (temperature 1.0, top-p 0.95): max, "
                                           "radix select of the cut (2 levels), nucleus Gumbel-max, acceptance"},
        "clocks": clock_info,
        "gpu_launches": args.steps * Ly * st.launches_per_layer(),
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- oracle (CPU) arm
_PREFILLED = {}


def _oracle_layer_sample(w, layer, shapes):
    """Run the oracle's append + verify for one layer of every slot; returns (tokens, seconds of the step part)."""
    from oracle.cache import PagedCache

    S = w.num_slots
    Ltot = [c + t for c, t in zip(shapes.ctx, shapes.n_new[0])]
    pages = [(n + 255) // 256 for n in Ltot]
    pt = np.full((S, max(pages)), -1, np.int32)
    k = 0
    for b, n in enumerate(pages):
        pt[b, :n] = np.arange(k, k + n)
        k += n
    if (w.key, layer) not in _PREFILLED:
        cache = PagedCache(sum(pages), 1, w.num_kv_heads)
        for b in range(S):                             # prefill (set-up, not timed)
            kk = np.stack([qi.kv_rows(w, b, layer, g, 0, 0, shapes.ctx[b]) for g in range(w.num_kv_heads)], axis=1)
            vv = np.stack([qi.kv_rows(w, b, layer, g, 1, 0, shapes.ctx[b]) for g in range(w.num_kv_heads)], axis=1)
            cache.append(pt[b], 0, 0, kk, vv)
        _PREFILLED[(w.key, layer)] = cache
    cache = _PREFILLED[(w.key, layer)]
    t0 = time.perf_counter()
    for b in range(S):                                 # the step: append the new tokens, verify them
        n, T = shapes.ctx[b], shapes.n_new[0][b]
        kk = np.stack([qi.kv_rows(w, b, layer, g, 0, n, T) for g in range(w.num_kv_heads)], axis=1)
        vv = np.stack([qi.kv_rows(w, b, layer, g, 1, n, T) for g in range(w.num_kv_heads)], axis=1)
        cache.append(pt[b], n, 0, kk, vv)
        cache.verify(pt[b], 0, n, qi.q_rows(w, b, layer, 0, T), w.group)
    return sum(shapes.n_new[0]), time.perf_counter() - t0


def cpu_baseline(w, budget_s=20.0):
    shapes = qi.draw_shapes(w)
    spent, layers = 0.0, 0
    while spent < budget_s and layers < w.num_layers:
        _, dt = _oracle_layer_sample(w, layers, shapes)
        spent += dt
        layers += 1
    per_layer = spent / layers
    tokens = sum(shapes.n_new[0])
    return {"value": tokens / (per_layer * w.num_layers), "unit": "tokens/s", "cores": _threads(),
            "host_cpus": os.cpu_count(), "blas_threads": _blas_threads(), "kind": "oracle",
            "sample": f"{layers} of {w.num_layers} layers of one step (append + verify, every slot), "
                      f"scaled to {w.num_layers} layers; prefill not timed"}


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
        tok, dt = _oracle_layer_sample(w, s % w.num_layers, shapes)
        if s >= max(args.warmup, 3):
            times.append(dt * w.num_layers)           # one sampled layer stands for all layers
    total = sum(times)
    value = tok * args.steps / total
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": total * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "slots": w.num_slots, "layers": w.num_layers, "ctx": shapes.ctx,
                       "query_tokens": shapes.n_new[0]},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _threads(), "host_cpus": os.cpu_count(),
                             "blas_threads": _blas_threads(), "kind": "oracle",
                             "sample": "each step runs one layer of the step (append + verify of every slot) "
                                       "and counts it for all layers"},
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
