#!/usr/bin/env python3
"""Decode-attention benchmark over a quantized paged KV cache.

Metric: decode-attention microseconds per step and effective cache GB/s (as a
fraction of the GB300's measured HBM bandwidth) against context length.  One
step = kvq_append of the step's new token(s) + kvq_decode + kvq_combine, all
inputs resident in HBM.  Default workload: GQA 6:1, int8 per-row absmax,
B=1, Hq=24, Hkv=4, D=256, block 256, context 262,144 (the kv-quant-attn
page's geometry); the context sweep 1K..262,144 is reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent
replica (the path does not shard); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention µs/step and cache GB/s (% of GB300 HBM peak) vs context length"
SWEEP = [1024, 4096, 16384, 65536, 262144]
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
EARLY_CACHE = True  # the decode steps' KVQ_DECODE_EARLY_CACHE (see --no-early-cache)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="gqa", choices=["tiny", "gqa", "paged", "spec", "mixed"])
    p.add_argument("--ctx", type=int, default=None, help="context length (gqa: 262144, spec: 32768, tiny: 256)")
    p.add_argument("--reps", type=int, default=0, help="cache replicas rotated per step (0: enough for 4x L2)")
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prologue", action="store_true", help="skip the QK-RMSNorm + RoPE prologue timing")
    p.add_argument("--no-prefill", action="store_true", help="skip the chunked-prefill timing")
    p.add_argument("--no-group", action="store_true", help="skip the group-wise-scale decode timing")
    p.add_argument("--no-latent", action="store_true", help="skip the head_dim 576 latent-cache timing")
    p.add_argument("--no-early-cache", action="store_true",
                   help="decode without KVQ_DECODE_EARLY_CACHE (cache reads wait for the step's append)")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads (tiny, paged, spec, mixed) beside the default line")
    return p.parse_args()


# --------------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_tensor_peak():
    """Dense 16-bit tensor throughput (TFLOP/s): the measured bf16 GEMM burst
    figure (f16 runs at the same rate), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, r in rows for n, v in zip(names, r) if v.lower().startswith("active")})
        busy = [s for s, _, _ in rows]
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(m for _, m, _ in rows),
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def describe(w, window=0):
    names = {1: "int8", 2: "fp8-e4m3", 3: "int4"}
    modes = {1: "per-row", 2: "per-tensor", 3: "per-channel"}
    L = w.seq_lens
    ctx = f"ctx={int(L[0])}" if (L == L[0]).all() else f"ctx=ragged[{int(L.min())}..{int(L.max())}] sum={int(L.sum())}"
    s = (f"{w.name}: {names[w.dtype]} K {modes[w.k_mode]} / V {modes[w.v_mode]}, B={w.batch} Hq={w.num_q_heads} "
         f"Hkv={w.num_kv_heads} D={w.head_dim} T={w.q_tokens} block={w.block_size} {ctx}")
    if w.softcap:
        s += f" softcap={w.softcap:g}"
    if w.use_sink:
        s += " head_sink"
    if window:
        s += f" window={window}"
    return s


def make_workload(args):
    from decode_attention_quantized_gb300 import synth
    ctx = args.ctx
    if ctx is None and args.workload == "gqa":
        ctx = 262144
    if args.workload in ("tiny", "gqa", "spec"):
        return synth.make(args.workload, ctx=ctx)
    return synth.make(args.workload, max_ctx=ctx)


# --------------------------------------------------------------------------- GPU arm

class Rig:
    """Workload w on the current GPU: one cache filled through kvq_append and
    replicated so that consecutive launches read different memory and the
    replicas together exceed 4x the L2 size (inputs larger than L2); decode
    buffers per window; eight query draws."""

    def __init__(self, w, windows=(0,), reps=0):
        import torch
        from decode_attention_quantized_gb300 import kvq, synth
        from decode_attention_quantized_gb300.workload import GpuWorkload

        self.w, self.windows = w, tuple(windows)
        dev = torch.cuda.current_device()
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        kv_bytes = synth.step_bytes(w)["kv"]
        if reps <= 0:
            reps = min(512, max(2, math.ceil(4 * self.l2 / max(kv_bytes, 1))))
        self.reps = reps
        gws = [GpuWorkload(w, device=f"cuda:{dev}", gen_device="cuda")]
        gws[0].fill_history()
        for _ in range(reps - 1):
            g = GpuWorkload.__new__(GpuWorkload)
            g.__dict__.update(gws[0].__dict__)
            src = gws[0].cache
            c = kvq.QuantizedPagedCache.__new__(kvq.QuantizedPagedCache)
            c.__dict__.update(src.__dict__)
            c.k_codes, c.v_codes = src.k_codes.clone(), src.v_codes.clone()
            c.k_scale, c.v_scale = src.k_scale.clone(), src.v_scale.clone()
            g.cache = c
            gws.append(g)
        self.gws = gws
        self.k_new, self.v_new, self.slots = gws[0].new_tokens()
        self.qs = [w.q("cuda", i).to(f"cuda:{dev}") for i in range(8)]
        # q, the block table and seq_lens are never written by the kernel before
        # kvq_decode (kvq_append), which writes only the new tokens' cache rows:
        # the decode may read the inputs and the older rows while append finishes
        flags = kvq.DECODE_EARLY_INPUTS | (kvq.DECODE_EARLY_CACHE if EARLY_CACHE else 0)
        self.plist = [gws[0].params(window=wd, flags=flags) for wd in self.windows]
        self.bufs = [gws[0].buffers(p) for p in self.plist]
        self.stream = torch.cuda.current_stream()

    def _args(self, i, j=None):
        j = i % len(self.windows) if j is None else j
        return self.gws[i % self.reps], self.plist[j], self.bufs[j], self.qs[i % len(self.qs)]

    def append(self, i, j=None):
        from decode_attention_quantized_gb300 import kvq
        g, p, b, q = self._args(i, j)
        kvq.kvq_append(g.cache, self.k_new, self.v_new, self.slots)

    def decode(self, i, j=None):
        from decode_attention_quantized_gb300 import kvq
        g, p, b, q = self._args(i, j)
        kvq.kvq_decode(g.cache, p, q, g.block_table, g.seq_lens, b.workspace)

    def combine(self, i, j=None):
        from decode_attention_quantized_gb300 import kvq
        g, p, b, q = self._args(i, j)
        kvq.kvq_combine(g.cache, p, b.workspace, g.head_sink, b.out, b.lse)

    def step(self, i):
        self.append(i)
        self.decode(i)
        self.combine(i)

    def graph_ms(self, fn, steps, first):
        """Total ms of `steps` launches fn(first), fn(first + 1), ... captured
        once in a CUDA graph (the ABI is capture-safe) and replayed between
        CUDA events on the launching stream."""
        import torch
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for i in range(steps):
                fn(first + i)
        gr.replay()  # warm replay
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        gr.replay()
        t1.record(self.stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    def per_launch_ms(self, n, first, j=None):
        """n decode launches, each bracketed by its own pair of CUDA events.  A
        sleep kernel ahead of them keeps the GPU busy while the host enqueues
        them all, so no launch waits on the host; consecutive launches read
        different cache replicas (L2-cold)."""
        import torch
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e5 * n + 2e6))  # about 0.1 ms per launch at 2 GHz: longer than their enqueue
        for i in range(n):
            ev[i][0].record(self.stream)
            self.decode(first + i, j)
            ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]


def pct(xs, q):
    """q-th percentile (linear interpolation) of a list."""
    xs = sorted(xs)
    k = (len(xs) - 1) * q / 100.0
    f = math.floor(k)
    c = min(f + 1, len(xs) - 1)
    return xs[f] + (xs[c] - xs[f]) * (k - f)


def measure(w, steps, warmup, *, windows=(0,), e2e=False, reps=0, per_launch=0):
    """Time `steps` decode steps of workload w on the current GPU (graphs of K
    launches), and optionally `per_launch` decode launches one by one per
    window (median and p10 / p90)."""
    import torch
    from decode_attention_quantized_gb300 import kvq, synth

    rig = Rig(w, windows, reps)
    for i in range(warmup):  # eager warm-up: per-device set-up, plan cache, smem limits
        rig.step(i)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0, "device error flags set during warm-up"
    total_ms = rig.graph_ms(rig.step, steps, warmup)
    dec_ms = rig.graph_ms(rig.decode, steps, warmup) / steps
    app_ms = rig.graph_ms(rig.append, steps, warmup) / steps
    comb_ms = rig.graph_ms(rig.combine, steps, warmup) / steps
    assert kvq.kvq_get_device_error() == 0, "device error flags set during the timed steps"
    res = dict(total_ms=total_ms, steps=steps, decode_ms=[dec_ms], append_ms=[app_ms], combine_ms=[comb_ms],
               launches=3 * steps, reps=rig.reps, l2=rig.l2)
    sb = [synth.step_bytes(w, wd) for wd in windows]
    res["step_bytes"] = sum(sum(sb[i % len(windows)].values()) for i in range(warmup, warmup + steps))
    res["decode_bytes"] = [synth.decode_bytes(w, windows[i % len(windows)]) for i in range(warmup, warmup + steps)]
    if per_launch:
        res["per_launch"] = []
        for j, wd in enumerate(windows):
            for i in range(3):  # warm the per-launch path (events, sleep)
                rig.decode(i, j)
            ms = rig.per_launch_ms(per_launch, warmup + steps, j)
            res["per_launch"].append(dict(window=wd, ms=ms, bytes=synth.decode_bytes(w, wd)))
        assert kvq.kvq_get_device_error() == 0, "device error flags set during the per-launch timing"
    if e2e:
        res["e2e"] = measure_e2e(w, rig.gws, rig.plist, windows, steps, warmup, rig.k_new, rig.v_new, rig.slots,
                                 rig.qs)
    del rig
    torch.cuda.empty_cache()
    return res


def launch_stats(pl, peak):
    """Median and p10 / p90 of per-launch decode times, with GB/s and the
    fraction of the HBM peak at the median."""
    ms = pl["ms"]
    med = statistics.median(ms)
    gbs = pl["bytes"] / (med * 1e-3) / 1e9
    return {"decode_us_median": round(1e3 * med, 2), "decode_us_p10": round(1e3 * pct(ms, 10), 2),
            "decode_us_p90": round(1e3 * pct(ms, 90), 2), "launches": len(ms),
            "decode_gbs_at_median": round(gbs, 1), "frac_of_hbm_at_median": round(gbs / peak, 3),
            "algorithmic_bytes_per_launch": int(pl["bytes"])}


def measure_configs(names, steps, warmup, peak, per_launch):
    """The other workloads of the benchmark at full size, each with its
    graph-mean decode time and per-launch percentiles (the mixed workload's
    full and windowed calls separately)."""
    import torch
    from decode_attention_quantized_gb300 import synth
    out = []
    for name in names:
        w = synth.make(name)
        windows = (w.window_for_call(0), w.window_for_call(1)) if w.window else (0,)
        r = measure(w, steps, warmup, windows=windows, per_launch=per_launch)
        for j, pl in enumerate(r["per_launch"]):
            ent = {"name": name if len(windows) == 1 else f"{name}-{'window' if pl['window'] else 'full'}",
                   "workload": describe(w, pl["window"]), "replicas": r["reps"]}
            ent.update(launch_stats(pl, peak))
            if name == "tiny":
                ent["roofline"] = "latency-bound: no bandwidth claim"
            out.append(ent)
        out[-1]["graph_mean_decode_us_all_calls"] = round(1e3 * statistics.mean(r["decode_ms"]), 2)
        out[-1]["graph_mean_step_us_all_calls"] = round(1e3 * r["total_ms"] / r["steps"], 2)
        del r
        torch.cuda.empty_cache()
    return out


def measure_e2e(w, gws, plist, windows, steps, warmup, k_new, v_new, slots, qs):
    """Same steps through the public API with host buffers: every step copies
    its inputs (q, new K/V rows, slot_mapping, seq_lens) from pinned host memory,
    runs append + decode + combine, reads the output and LSE back, and the host
    waits for it.  The inputs of a step sit in one pinned staging buffer (each
    at a 256-byte aligned offset) and travel in one copy; the output and LSE
    are written into one device buffer and come back in one copy.  Each step's
    calls (the two copies and the three kvq calls) are captured once into a
    CUDA graph of their own, as a serving loop would, and every timed step
    replays its graph and synchronizes; the same steps issued call by call are
    reported beside it."""
    import torch
    from decode_attention_quantized_gb300 import kvq

    dev = torch.cuda.current_device()
    stream = torch.cuda.current_stream()
    seq_lens = gws[0].seq_lens

    def layout(tensors):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, off

    ins = [qs[0], k_new, v_new, slots, seq_lens]
    in_offs, in_bytes = layout(ins)
    # one pinned host buffer per query draw; K/V rows, slots and lengths are the same in each
    h_in = []
    for q in qs:
        h = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        for t, o in zip([q, k_new, v_new, slots, seq_lens], in_offs):
            n = t.numel() * t.element_size()
            h[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        h_in.append(h)
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=f"cuda:{dev}")

    def view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    d_q, d_k, d_v, d_s, d_l = (view(d_in, o, t) for t, o in zip(ins, in_offs))
    bufs = [gws[0].buffers(p) for p in plist]
    outs = [bufs[0].out, bufs[0].lse]
    out_offs, out_bytes = layout(outs)
    d_outbuf = torch.empty(out_bytes, dtype=torch.uint8, device=f"cuda:{dev}")
    d_out, d_lse = (view(d_outbuf, o, t) for t, o in zip(outs, out_offs))
    h_outbuf = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    reps = len(gws)

    def calls(i):  # on torch's current stream (the capture stream inside a graph capture)
        g = gws[i % reps]
        j = i % len(windows)
        d_in.copy_(h_in[i % len(h_in)], non_blocking=True)
        kvq.kvq_append(g.cache, d_k, d_v, d_s)
        kvq.kvq_decode(g.cache, plist[j], d_q, g.block_table, d_l, bufs[j].workspace)
        kvq.kvq_combine(g.cache, plist[j], bufs[j].workspace, g.head_sink, d_out, d_lse)
        h_outbuf.copy_(d_outbuf, non_blocking=True)

    def eager(i):
        calls(i)
        stream.synchronize()

    for i in range(warmup):
        eager(i)
    torch.cuda.synchronize()
    t = time.perf_counter()
    for i in range(steps):
        eager(warmup + i)
    torch.cuda.synchronize()
    wall_eager = time.perf_counter() - t

    graphs = []
    for i in range(steps):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            calls(warmup + i)
        graphs.append(gr)
    for gr in graphs[:3]:  # warm replays
        gr.replay()
    torch.cuda.synchronize()
    t = time.perf_counter()
    for gr in graphs:
        gr.replay()
        torch.cuda.current_stream().synchronize()
    wall = time.perf_counter() - t
    h2d = (qs[0].numel() * 2 + k_new.numel() * 2 + v_new.numel() * 2 + slots.numel() * 8 + seq_lens.numel() * 4)
    d2h = d_out.numel() * 2 + d_lse.numel() * 4
    return dict(wall_s=wall, wall_eager_s=wall_eager, h2d=h2d, d2h=d2h)


def measure_prologue(w, steps, warmup, peak):
    """The fused QK-RMSNorm + RoPE prologue (kvq_append_norm_rope on the new
    K/V rows, kvq_norm_rope_apply on the queries) at the step's sizes, next to
    the plain kvq_append, each as a graph of `steps` launches; and a bulk
    kvq_append_norm_rope over enough tokens that its bf16 inputs exceed L2,
    reported against the HBM peak (algorithmic bytes: bf16 K/V read, codes and
    per-row scales written, slots, positions and the tables' rows read)."""
    import torch
    from decode_attention_quantized_gb300 import kvq, synth

    dev = torch.cuda.current_device()
    D, Hkv, Hq = w.head_dim, w.num_kv_heads, w.num_q_heads
    max_pos = 8192  # table rows; positions are taken modulo this
    cos, sin = synth.rope_tables(max_pos, D)
    pro = kvq.NormRope(norm_weight=synth.norm_weight_bf16(D, f"cuda:{dev}", "bench", "norm"), eps=1e-6,
                       rotary_dim=D, cos=torch.from_numpy(cos).cuda(), sin=torch.from_numpy(sin).cuda())
    qmax = {kvq.INT8: 127.0, kvq.INT4: 7.0, kvq.FP8_E4M3: 448.0}[w.dtype]

    def cache_for(n_tokens):
        bs = 256
        nb = (n_tokens + bs - 1) // bs
        def static(mode):
            if mode == kvq.PER_TENSOR:
                return torch.full((1,), 4.0 / qmax)
            if mode == kvq.PER_CHANNEL:
                return torch.full((Hkv, D), 4.0 / qmax)
            return None
        return kvq.QuantizedPagedCache(w.dtype, w.k_mode, w.v_mode, nb, bs, Hkv, D, device=f"cuda:{dev}",
                                       k_static=static(w.k_mode), v_static=static(w.v_mode))

    def timed_graph(fn, n):
        for _ in range(max(3, warmup)):
            fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for _ in range(n):
                fn()
        gr.replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        gr.replay()
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    N = w.batch * w.q_tokens
    cache = cache_for(N)
    k = synth.randn_bf16((N, Hkv, D), f"cuda:{dev}", "bench", "pro-k")
    v = synth.randn_bf16((N, Hkv, D), f"cuda:{dev}", "bench", "pro-v")
    q = synth.randn_bf16((N, Hq, D), f"cuda:{dev}", "bench", "pro-q")
    qo = torch.empty_like(q)
    slots = torch.arange(N, dtype=torch.int64, device=f"cuda:{dev}")
    pos = (torch.arange(N, dtype=torch.int64, device=f"cuda:{dev}") * 7) % max_pos
    us_app = 1e3 * timed_graph(lambda: kvq.kvq_append(cache, k, v, slots), steps)
    us_fused = 1e3 * timed_graph(lambda: kvq.kvq_append_norm_rope(cache, pro, k, v, slots, pos), steps)
    us_q = 1e3 * timed_graph(lambda: kvq.kvq_norm_rope_apply(pro, q, qo, pos), steps)
    pro_h = kvq.NormRope(norm_weight=pro.norm_weight, eps=pro.eps, rotary_dim=D, cos=pro.cos, sin=pro.sin,
                         hadamard=True)
    us_fused_h = 1e3 * timed_graph(lambda: kvq.kvq_append_norm_rope(cache, pro_h, k, v, slots, pos), steps)
    del cache, k, v, q, qo

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nb_tok = max(1024, int(2 * l2 // (2 * Hkv * D * 2)))  # bf16 K + V twice the L2 size
    cache = cache_for(nb_tok)
    k = synth.randn_bf16((nb_tok, Hkv, D), f"cuda:{dev}", "bench", "pro-bulk-k")
    v = synth.randn_bf16((nb_tok, Hkv, D), f"cuda:{dev}", "bench", "pro-bulk-v")
    slots = torch.arange(nb_tok, dtype=torch.int64, device=f"cuda:{dev}")
    pos = slots % max_pos
    ms = timed_graph(lambda: kvq.kvq_append_norm_rope(cache, pro, k, v, slots, pos), 5)
    assert kvq.kvq_get_device_error() == 0, "device error flags set in the prologue timing"
    dp = D // 2 if w.dtype == kvq.INT4 else D
    rows = nb_tok * Hkv
    nbytes = (2 * rows * D * 2 + 2 * rows * dp + 4 * rows * ((w.k_mode == kvq.PER_ROW) + (w.v_mode == kvq.PER_ROW))
              + nb_tok * (8 + 8 + 2 * 4 * (D // 2)))
    gbs = nbytes / (ms * 1e-3) / 1e9
    del cache, k, v
    torch.cuda.empty_cache()
    return {"step_tokens": N, "append_us": round(us_app, 2), "append_norm_rope_us": round(us_fused, 2),
            "norm_rope_q_us": round(us_q, 2), "append_norm_rope_hadamard_us": round(us_fused_h, 2),
            "bulk": {"tokens": nb_tok, "append_norm_rope_us": round(1e3 * ms, 1), "gbs": round(gbs, 1),
                     "frac_of_hbm": round(gbs / peak, 3), "bytes": int(nbytes)},
            "prologue": f"RMSNorm (bf16 weight, eps 1e-6) + RoPE on all {D} channels (half split), fixed-order fp32"}


def measure_prefill(w, steps, warmup, peak, chunk=64):
    """kvq_prefill of a chunk of `chunk` query tokens per sequence at the end of
    the workload's sequences (the chunk's rows already in the cache), as a
    graph of `steps` calls.  Reported against the bytes a single pass over
    the cache would read: kvq_prefill re-reads each prefix once per group of
    up to 8 chunk tokens, so the fraction shows that cost."""
    import torch
    from decode_attention_quantized_gb300 import kvq, synth
    from decode_attention_quantized_gb300.workload import GpuWorkload

    dev = torch.cuda.current_device()
    gw = GpuWorkload(w, device=f"cuda:{dev}", gen_device="cuda")
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    kvq.kvq_append(gw.cache, k_new, v_new, slots)
    C = chunk
    params = kvq.make_params(w.batch, w.num_q_heads, C, w.max_blocks, max_seq_len=gw.max_seq_len,
                             softcap=w.softcap)
    q = synth.randn_bf16((w.batch, C, w.num_q_heads, w.head_dim), f"cuda:{dev}", "bench", "prefill-q")
    out = torch.empty_like(q)
    lse = torch.empty((w.batch, C, w.num_q_heads), dtype=torch.float32, device=f"cuda:{dev}")
    ws = torch.empty(kvq.kvq_prefill_workspace_size(gw.cache, params) // 4 + 64, dtype=torch.int32,
                     device=f"cuda:{dev}")

    def call():
        kvq.kvq_prefill(gw.cache, params, q, gw.block_table, gw.seq_lens, gw.head_sink, out, lse, ws)

    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for _ in range(steps):
            call()
    gr.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    gr.replay()
    t1.record()
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0, "device error flags set in the prefill timing"
    ms = t0.elapsed_time(t1) / steps
    one_pass = synth.decode_bytes(w)
    # attention FLOPs of the chunk: 4 D per (query row, visible key)
    seen = sum(min(int(L), max(0, int(L) - C + t + 1)) for L in w.seq_lens for t in range(C))
    flops = 4.0 * w.head_dim * w.num_q_heads * seen
    G = w.group
    qt = w.head_dim in (128, 256) and w.k_mode != synth.PER_GROUP and w.v_mode != synth.PER_GROUP
    tq = 0
    if qt:
        tq = min(128 // G, C)
        while C % tq:
            tq -= 1
        qt = tq * G >= 64
    T = tq if qt else max(t for t in (8, 4, 2, 1) if C % t == 0)
    tpeak, tkind = load_tensor_peak()
    del gw, q, out, lse, ws
    torch.cuda.empty_cache()
    return {"chunk_tokens": C, "us_per_chunk": round(1e3 * ms, 2),
            "tokens_per_s": round(w.batch * C / (ms * 1e-3), 1),
            "kernel": ("query tiles of %d tokens x %d heads (tcgen05, rows as M)" % (T, G)) if qt
                      else "virtual decode sequences of %d tokens" % T,
            "groups_per_sequence": C // T,
            "attention_tflops": round(flops / (ms * 1e-3) / 1e12, 1),
            "frac_of_tensor_peak": round(flops / (ms * 1e-3) / 1e12 / tpeak, 3),
            "tensor_peak_tflops": tpeak, "tensor_peak_kind": f"of {tkind} (bf16 dense GEMM; f16 same rate)",
            "single_pass_gbs": round(one_pass / (ms * 1e-3) / 1e9, 1),
            "single_pass_frac_of_hbm": round(one_pass / (ms * 1e-3) / 1e9 / peak, 3)}


def measure_group(w, steps, warmup, peak, group_size=64):
    """The same workload with group-wise scales on both sides (PER_GROUP, one
    fp32 scale per group_size channels of each K and V row): decode timed as
    a graph of K launches, like the main line's roofline figure.  Its
    algorithmic bytes include the group scales."""
    import dataclasses
    import torch
    from decode_attention_quantized_gb300 import synth

    wg = dataclasses.replace(w, k_mode=synth.PER_GROUP, v_mode=synth.PER_GROUP, group_size=group_size)
    r = measure(wg, steps, warmup)
    dec_ms = statistics.mean(r["decode_ms"])
    dec_bytes = statistics.mean(r["decode_bytes"])
    gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    del r
    torch.cuda.empty_cache()
    return {"group_size": group_size, "modes": "K and V per-group", "decode_us": round(1e3 * dec_ms, 2),
            "decode_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 3),
            "algorithmic_bytes_per_launch": int(dec_bytes)}


def measure_latent(steps, warmup, peak, *, B=4, Hq=8, T=1, ctx=32768, bs=64):
    """A LATENT cache at the pages' absorbed-MLA shape (head_dim 576 = 512
    latent + 64 rotary channels, v_head_size 512; one kv head shared by Hq
    query heads), int8 per-row scales: decode timed as a graph of K launches
    over rotated cache replicas (inputs larger than L2), and per launch.  Each
    cached row is read once (V is its leading 512 channels): algorithmic bytes
    per key = 576 codes + 4 scale bytes."""
    import torch
    from decode_attention_quantized_gb300 import kvq, synth

    dev = torch.cuda.current_device()
    D, Dv, Hkv = 576, 512, 1
    mb = (ctx + bs - 1) // bs
    NB = B * mb
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    cache_bytes = NB * bs * Hkv * (D + 4)
    reps = min(64, max(2, math.ceil(4 * l2 / cache_bytes)))
    table = torch.arange(NB, dtype=torch.int32, device=f"cuda:{dev}").reshape(B, mb)
    lens = torch.full((B,), ctx, dtype=torch.int32, device=f"cuda:{dev}")
    caches = []
    base = kvq.QuantizedPagedCache(kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, NB, bs, Hkv, D, device=f"cuda:{dev}",
                                   latent=True, v_head_size=Dv)
    chunk = 1 << 15
    for t0 in range(0, B * ctx, chunk):
        n = min(chunk, B * ctx - t0)
        k = synth.randn_bf16((n, Hkv, D), f"cuda:{dev}", "bench", "mla-k", t0)
        slots = torch.arange(t0, t0 + n, dtype=torch.int64, device=f"cuda:{dev}")  # table is in order
        kvq.kvq_append(base, k, None, slots)
    caches.append(base)
    for _ in range(reps - 1):
        c = kvq.QuantizedPagedCache.__new__(kvq.QuantizedPagedCache)
        c.__dict__.update(base.__dict__)
        c.k_codes = base.k_codes.clone()
        c.v_codes = c.k_codes
        c.k_scale = base.k_scale.clone()
        c.v_scale = c.k_scale
        caches.append(c)
    q = synth.randn_bf16((B, T, Hq, D), f"cuda:{dev}", "bench", "mla-q")
    params = kvq.make_params(B, Hq, T, mb, max_seq_len=ctx, flags=kvq.DECODE_EARLY_INPUTS)
    bufs = kvq.alloc_decode_buffers(base, params)

    def dec(i):
        kvq.kvq_decode(caches[i % reps], params, q, table, lens, bufs.workspace)

    for i in range(max(3, warmup)):
        dec(i)
        kvq.kvq_combine(caches[i % reps], params, bufs.workspace, None, bufs.out, bufs.lse)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for i in range(steps):
            dec(i)
    gr.replay()
    torch.cuda.synchronize()
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0e.record()
    gr.replay()
    t1e.record()
    torch.cuda.synchronize()
    ms = t0e.elapsed_time(t1e) / steps
    n = max(50, steps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e5 * n + 2e6))
    for i in range(n):
        ev[i][0].record()
        dec(i)
        ev[i][1].record()
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev]
    assert kvq.kvq_get_device_error() == 0, "device error flags set in the latent timing"
    nbytes = B * ctx * Hkv * (D + 4) + B * T * Hq * D * 2 + B * mb * 4 + B * 4
    del caches, base, bufs
    torch.cuda.empty_cache()
    gbs = nbytes / (ms * 1e-3) / 1e9
    med = statistics.median(per)
    return {"workload": f"latent int8 per-row, head_dim {D} (v_head_size {Dv}), B={B} Hq={Hq} Hkv={Hkv} T={T} "
                        f"block={bs} ctx={ctx}", "decode_us": round(1e3 * ms, 2), "decode_gbs": round(gbs, 1),
            "frac_of_hbm": round(gbs / peak, 3), "decode_us_median": round(1e3 * med, 2),
            "decode_us_p10": round(1e3 * pct(per, 10), 2), "decode_us_p90": round(1e3 * pct(per, 90), 2),
            "algorithmic_bytes_per_launch": int(nbytes), "bytes_per_key": D + 4, "replicas": reps}


def decode_kernel_name(w):
    """The decode kernel a workload runs on: the tensor-memory kernel for
    17..48 query rows per kv head at head_dim 256 (17..64 at 128), else the
    mma.sync kernel."""
    rows = w.group * w.q_tokens
    tc = 17 <= rows <= (48 if w.head_dim == 256 else 64) and w.head_dim in (128, 256)
    return "decode_tc_kernel" if tc else "decode_kernel"


def traffic_from_profiles(kernel_tag: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    from decode_attention_quantized_gb300 import build as b
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel_tag)
        if ent and ent.get("source_stamp") == b._stamp():
            return ent["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


def run_ours(args):
    import torch
    from decode_attention_quantized_gb300 import build as cuda_build
    from decode_attention_quantized_gb300 import kvq, synth

    global EARLY_CACHE
    EARLY_CACHE = not args.no_early_cache

    world, rank, local = dist_setup()
    cuda_build.build()
    kvq.load()
    peak, peak_kind = load_peaks()
    w = make_workload(args)
    windows = (w.window_for_call(0), w.window_for_call(1)) if w.window else (0,)

    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    n_pl = max(50, args.steps)
    res = measure(w, args.steps, args.warmup, windows=windows, e2e=not args.no_e2e, reps=args.reps,
                  per_launch=n_pl)
    clk = clocks.stop()
    barrier(world)
    total_ms = max_over_ranks(res["total_ms"], world)

    sweep = []
    if not args.no_sweep and args.workload == "gqa" and world == 1:
        for ctx in SWEEP:
            if ctx == w.seq_lens[0]:
                r = res
                wc = w
            else:
                wc = synth.make("gqa", ctx=ctx)
                r = measure(wc, max(10, args.steps), max(3, args.warmup), per_launch=n_pl)
            dec_ms = statistics.mean(r["decode_ms"])
            kvb = synth.decode_bytes(wc)
            ent = {"ctx": ctx, "us_per_step": round(1e3 * r["total_ms"] / r["steps"], 2),
                   "decode_us": round(1e3 * dec_ms, 2),
                   "decode_gbs": round(kvb / (dec_ms * 1e-3) / 1e9, 1),
                   "frac_of_hbm": round(kvb / (dec_ms * 1e-3) / 1e9 / peak, 3),
                   "cache_mb": round(synth.step_bytes(wc)["kv"] / 1e6, 2),
                   "replicas": r["reps"]}
            ent["per_launch"] = {k: v for k, v in launch_stats(r["per_launch"][0], peak).items()
                                 if k.startswith("decode_us") or k.startswith("frac")}
            sweep.append(ent)
            del r
            torch.cuda.empty_cache()

    K = args.steps
    step_bytes = res["step_bytes"] * world
    value = step_bytes / (total_ms * 1e-3) / 1e9
    dec_mean_ms = statistics.mean(res["decode_ms"])
    dec_bytes = statistics.mean(res["decode_bytes"])
    achieved = dec_bytes / (dec_mean_ms * 1e-3) / 1e9
    tag = f"{args.workload}-{int(w.seq_lens.max())}"
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 4),
        "us_per_step": round(1e3 * total_ms / K, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded torch generators; no dataset)",
        "config": {
            "workload": describe(w),
            "cache_dtype": {1: "int8", 2: "fp8-e4m3", 3: "int4"}[w.dtype],
            "compute": "f16 x f16 -> f32 tensor-core mma, fp32 softmax",
            "step": "kvq_append (new tokens) + kvq_decode (flags KVQ_DECODE_EARLY_INPUTS%s) + kvq_combine"
                    % (" | KVQ_DECODE_EARLY_CACHE" if EARLY_CACHE else ""),
            "timing": "K steps captured once in a CUDA graph and replayed between CUDA events; per-kernel "
                      "times from graphs of K launches of that kernel alone; decode_per_launch and configs: "
                      f"{n_pl} decode launches each bracketed by its own CUDA events (median, p10, p90)",
            "windows_per_call": list(windows),
            "l2": f"inputs larger than L2: {res['reps']} cache replicas rotated per step, "
                  f"{res['reps'] * synth.step_bytes(w)['kv'] / 1e6:.0f} MB total vs L2 {res['l2'] / 1e6:.0f} MB",
            "parallelism": "replicas" if world > 1 else "single-gpu",
        },
        "step_breakdown_us_mean": {
            "append": round(1e3 * statistics.mean(res["append_ms"]), 2),
            "decode": round(1e3 * statistics.mean(res["decode_ms"]), 2),
            "combine": round(1e3 * statistics.mean(res["combine_ms"]), 2),
        },
        "decode_per_launch": [dict(window=pl["window"], **launch_stats(pl, peak)) for pl in res["per_launch"]],
        "roofline": {
            "kernel": decode_kernel_name(w),
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"of {peak_kind}",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic_from_profiles(tag),
            "algorithmic_bytes_per_launch": int(dec_bytes),
            "timing": "mean over a CUDA graph of K decode launches back to back; consecutive launches "
                      "overlap (the next one's plan, copies and tiles run during the previous one's tail), "
                      "so this is a period per launch; decode_per_launch has single launches",
        },
        "gpu_launches": res["launches"],
        "clocks": clk,
    }
    if sweep:
        line["sweep"] = sweep
    if "e2e" in res:
        e = res["e2e"]
        e2e_wall = max_over_ranks(e["wall_s"], world)
        e2e_eager = max_over_ranks(e["wall_eager_s"], world)
        line["e2e"] = {"value": round(step_bytes / e2e_wall / 1e9, 1), "unit": "GB/s",
                       "us_per_step": round(1e6 * e2e_wall / K, 2),
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "mode": "per step: H2D copy of the inputs from pinned memory, kvq_append, kvq_decode, "
                               "kvq_combine, D2H copy of out and LSE, captured once as one CUDA graph per step, "
                               "replayed and host-synchronized every step",
                       "eager": {"value": round(step_bytes / e2e_eager / 1e9, 1),
                                 "us_per_step": round(1e6 * e2e_eager / K, 2),
                                 "mode": "the same calls issued one by one every step"}}
    if rank == 0 and world == 1 and args.workload == "gqa" and not args.no_configs:
        head = {"name": f"gqa-{int(w.seq_lens.max())}", "workload": describe(w), "replicas": res["reps"]}
        head.update(launch_stats(res["per_launch"][0], peak))
        line["configs"] = [head] + measure_configs(["tiny", "paged", "spec", "mixed"], args.steps, args.warmup,
                                                   peak, n_pl)
    if rank == 0 and world == 1 and args.workload == "gqa" and not args.no_latent:
        line["latent"] = measure_latent(args.steps, args.warmup, peak)
    if rank == 0 and world == 1 and not args.no_prologue:
        line["prologue"] = measure_prologue(w, args.steps, args.warmup, peak)
    if rank == 0 and world == 1 and not args.no_prefill:
        line["prefill"] = measure_prefill(w, max(3, args.steps // 3), args.warmup, peak)
    if rank == 0 and world == 1 and not args.no_group:
        line["group_scales"] = measure_group(w, args.steps, args.warmup, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, windows[0], budget_s=12.0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# --------------------------------------------------------------------------- oracle (CPU) arm

def oracle_sample(w, window, kv_heads):
    """Oracle cache of sequence 0 restricted to the given kv heads' query rows;
    returns a callable that runs one timed sample and its algorithmic bytes."""
    import numpy as np
    import torch
    from decode_attention_quantized_gb300 import synth
    from oracle import oracle

    def bits(t):
        return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    gen = "cuda" if torch.cuda.is_available() else "cpu"
    b = int(np.argmax(w.seq_lens))
    L = int(w.seq_lens[b])
    bs = w.block_size
    nbk = max(1, math.ceil(L / bs))
    ks = synth.calibrate_static(w, gen, "k")
    vs = synth.calibrate_static(w, gen, "v")
    oc = oracle.OracleCache(w.dtype, w.k_mode, w.v_mode, nbk, bs, w.num_kv_heads, w.head_dim,
                            None if ks is None else ks.cpu().numpy(), None if vs is None else vs.cpu().numpy())
    k, v = w.seq_kv(b, gen)
    table = np.arange(nbk, dtype=np.int32)[None, :]
    oc.append(bits(k), bits(v), np.arange(L, dtype=np.int64))
    q = bits(w.q(gen))[b:b + 1]
    sink = w.head_sink(gen)
    sink = None if sink is None else sink.cpu().numpy()
    G, T = w.group, w.q_tokens
    rows = np.array([(0, t, h * G + g) for h in kv_heads for t in range(T) for g in range(G)], np.int32)
    lens = np.array([L], np.int32)
    cores = os.cpu_count() or 1
    per_key = 2 * w.row_bytes() + (4 if w.k_mode == 1 else 0) + (4 if w.v_mode == 1 else 0)
    lo = max(0, L - T + 1 - window) if window else 0
    nbytes = (L - lo) * per_key * len(kv_heads) + len(rows) * w.head_dim * 2 * 2

    def run():
        t = time.perf_counter()
        oc.attend(q, table, lens, q_tokens=T, softcap=w.softcap, window=window, head_sink=sink, rows=rows,
                  nthreads=cores)
        return time.perf_counter() - t

    desc = (f"sequence {b} (L={L}), {len(rows)} query rows of kv head(s) {list(kv_heads)} "
            f"of {w.batch * T * w.num_q_heads} in the step; oracle dequantizes each row's keys in fp64")
    return run, nbytes, cores, desc


def cpu_baseline(w, window, budget_s=12.0):
    run, nbytes, cores, desc = oracle_sample(w, window, kv_heads=list(range(w.num_kv_heads)))
    t = run()
    reps = 1
    while t * (reps + 1) / reps < budget_s and reps < 3:
        t += run()
        reps += 1
    return {"value": round(nbytes * reps / t / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": desc + f"; {reps} run(s), {t:.1f} s"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from decode_attention_quantized_gb300 import synth
    from oracle import oracle
    oracle.build()
    w = make_workload(args)
    run, nbytes, cores, desc = oracle_sample(w, w.window_for_call(0), kv_heads=[0])
    for _ in range(args.warmup):
        run()
    times = [run() for _ in range(args.steps)]
    total = sum(times)
    value = nbytes * args.steps / total / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded torch generators; no dataset)",
        "config": {"workload": describe(w), "note": "the CPU fp64 oracle, one bounded sample per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
