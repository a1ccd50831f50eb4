#!/usr/bin/env python
"""Decode throughput of the batched step on GB300: tok/s vs the
(W + B*A)/beta HBM roofline.

Workload (default): the 7B-shaped decoder (32 layers, d 4096, 32 q / 8 KV
heads, head_dim 128, FFN 14336, vocab 65536, bf16 random-init weights) in a
pure-decode step of B = 32 rows whose cached contexts are drawn from
U[256, 4096] (seeded), 32-position KV blocks on a randomly permuted
placement, KV filled with seeded random bf16, every row sampled with
temperature 1, top_p 0.3, frequency penalty 1, decay 0.996.  One "step" is
one pass of the whole step (embedding, 32 layers, LM head, sampler) for all
B rows; the weights (14.5 GB) and KV (~9 GB) are far larger than L2, so no
flush is needed between steps.

value  = B * n_gpus / step time, inputs resident on the device (Batch API),
         each step replayed as one CUDA graph of the same kernels
         (cbd_batch_set_graph); the launch-by-launch time is reported in
         "graph".
e2e    = the same through cbd_step with host arrays: the step's rows, block
         tables and sampling parameters go host->device and the sampled
         tokens come back device->host inside every timed step (steps run as
         cached graphs, cbd_engine_set_step_graph; the launch-by-launch time
         is reported beside).
Multi-GPU: independent replicas (one engine per GPU, no collective on the
data path); barrier + max-over-ranks timing.

sweep  = the same step at every B in --sweep (default 1, 2, 4, 8, 16, 64,
         128; contexts U[256, 4096], one pool sized for the largest B, each B
         the first B rows), tok/s and the roofline fraction per B.
cpu_baseline = one whole step of the CPU oracle (every layer, every row, the
         LM head) on this workload's shapes, timed once.

--impl reference times the CPU oracle (no GPU): every step is one whole
oracle step of the same workload.

--gpus N without a torchrun environment re-launches this script under
torch.distributed.run with N ranks (one engine per GPU).

--trace serves a continuous-batching request trace instead (7B shape, 64
slots, Poisson arrivals, prompts from {20, 50, 200, 1000}, outputs
min(Geometric(1/128), 512), 512-token chunks, <= 2048 rows per step, a
128-token answer reservation) through the C++ scheduler and the engine
(continuous_batching_decode_gb300.serve) and prints one line per policy:
generated tok/s over the wall clock, time to first token, steps and rows.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s on 1 GB300 vs batch B; step HBM GB/s vs (W+B·A)/β roofline"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="cbd", choices=["cbd", "reference"])
    ap.add_argument("--shape", default="7b")
    ap.add_argument("--B", type=int, default=32)
    ap.add_argument("--ctx-lo", type=int, default=256)
    ap.add_argument("--ctx-hi", type=int, default=4096)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0, help="override layer count (profiling cases only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", default="1,2,4,8,16,64,128",
                    help="comma-separated B values timed after the headline step ('' = none)")
    ap.add_argument("--gemm-path", type=int, default=0, help="0 auto, 1 CUDA-core GEMV, 2 tcgen05")
    ap.add_argument("--attn-path", type=int, default=0, help="0 streaming mma.sync, 1 CUDA cores, 2 per-chunk mma.sync")
    ap.add_argument("--gemm-chain", action="store_true",
                    help="decode contractions of a layer as one persistent chain instead of one launch each")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="KV pool element type (fp8: E4M3; skips the CPU baseline)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "int8"],
                    help="streamed weight type (int8: per-row scales; the CPU baseline runs the int8 oracle)")
    ap.add_argument("--rows-gemm", type=int, default=256,
                    help="steps of at least this many rows may run the 128-row-tile GEMM (0 = never)")
    ap.add_argument("--rows-gemm-force", action="store_true",
                    help="... on every GEMM of such a step (default: where it fills the GPU well)")
    ap.add_argument("--no-prefill-attn", action="store_true",
                    help="mixed step: prompt rows on the streaming attention kernel")
    ap.add_argument("--mixed", type=int, default=0,
                    help="prefill rows (512-row chunks) added to the B decode rows: one mixed-step line")
    ap.add_argument("--trace", action="store_true", help="serve the request trace (see the module docstring)")
    ap.add_argument("--trace-requests", type=int, default=2000)
    ap.add_argument("--trace-rate", type=float, default=0.0, help="requests/s (0: all arrive at t = 0)")
    ap.add_argument("--trace-blocks", type=int, default=4096, help="KV pool blocks (4096 = ample)")
    ap.add_argument("--policy", default="both", choices=["forma", "albatross", "both"])
    ap.add_argument("--l2-prefetch-mb", type=int, default=0,
                    help="MiB of the next weight contraction each kernel prefetches into L2 (0: off)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def shape_of(args):
    from continuous_batching_decode_gb300 import synth
    s = dict(synth.MODEL_SHAPES[args.shape])
    if args.layers:
        s["n_layers"] = args.layers
    return s


def weight_bytes(s, int8=False):
    """W: every weight streamed once per step (embedding excluded); int8:
    one byte per weight plus an fp32 scale per matrix row."""
    d, hq, hkv, hd, F, V, L = (s["d_model"], s["n_heads"], s["n_kv_heads"], s["head_dim"], s["ffn_dim"],
                               s["vocab"], s["n_layers"])
    wb = 1 if int8 else 2
    rows = (hq + 2 * hkv) * hd + d + 2 * F + d
    per_layer = ((hq + 2 * hkv) * hd * d + d * hq * hd + 2 * F * d + d * F) * wb + 2 * d * 2 + (rows * 4 if int8 else 0)
    return L * per_layer + V * d * wb + (V * 4 if int8 else 0) + d * 2


def kv_pos_bytes(s, eb=2):
    """K and V bytes of one cached position over all layers (eb bytes per element)."""
    return 2 * s["n_layers"] * s["n_kv_heads"] * s["head_dim"] * eb


def config_of(args, s, wl, world):
    """The workload description both arms print."""
    return {"workload": (f"{args.shape}-shaped pure-decode step, B={args.B}, ctx U[{args.ctx_lo},{args.ctx_hi}], "
                         "32-position blocks, top_p 0.3 sampling"),
            "B": args.B, "shape": args.shape, "layers": s["n_layers"], "mean_ctx": float(np.mean(wl["ctx"])),
            "kv": "e4m3" if args.kv == "fp8" else "bf16",
            "weights": args.weights,
            "l2": "inputs larger than L2 (weights 7.2-14.5 GB + KV); no flush",
            "parallelism": f"replicas x{world}"}


def workload(s, B, lo, hi, seed):
    from continuous_batching_decode_gb300 import synth
    db = synth.decode_batch(B, lo, hi, s["vocab"], seed)
    ctx, toks = db["contexts"], db["tokens"]
    need = {i: (c + 1 + 31) // 32 for i, c in enumerate(ctx)}
    mbps = (hi + 1 + 31) // 32
    n_pool = sum(need.values()) + 8
    tables, nbps = synth.permuted_tables(need, n_pool, mbps, np.random.default_rng(seed + 1))
    rows = [(i, toks[i], ctx[i], 0, 1) for i in range(B)]
    samp = [dict(temperature=1.0, top_p=0.3, top_k=0, frequency_penalty=1.0, penalty_decay=0.996, seed=seed,
                 request_id=i, token_index=0) for i in range(B)]
    return dict(ctx=ctx, rows=rows, tables=tables, nbps=nbps, samp=samp, mbps=mbps, n_pool=n_pool)


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.dev, self.lines, self.proc = dev, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_bytes(cls, s, B, ctx, eb=2, wb=2):
    """Algorithmic bytes one launch of a kernel class must move (7B: see the
    design notes for the per-unit figures); wb = bytes per weight (int8
    weights add an fp32 scale per row)."""
    d, hq, hkv, hd, F, V = s["d_model"], s["n_heads"], s["n_kv_heads"], s["head_dim"], s["ffn_dim"], s["vocab"]
    act = lambda k: B * k * 2 * 2            # hi + lo bf16 activations read
    sc = lambda rows: rows * 4 if wb == 1 else 0
    if cls == "gemm_qkv":
        return (hq + 2 * hkv) * hd * d * wb + sc((hq + 2 * hkv) * hd) + act(d) + B * hq * hd * 4 + B * 2 * hkv * hd * eb
    if cls == "gemm_o":
        return d * hq * hd * wb + sc(d) + act(hq * hd) + 2 * B * d * 4
    if cls == "gemm_gate_up":
        return 2 * F * d * wb + sc(2 * F) + act(d) + B * F * 2 * 2
    if cls == "gemm_down":
        return d * F * wb + sc(d) + act(F) + 2 * B * d * 4
    if cls == "gemm_chain":
        # one launch per layer: O, gate/up and down, plus the next layer's
        # QKV in all but the last layer's; the mean over the layers
        L = s["n_layers"]
        per = sum(kernel_bytes(k, s, B, ctx, eb, wb) for k in ("gemm_o", "gemm_gate_up", "gemm_down"))
        return (L * per + (L - 1) * kernel_bytes("gemm_qkv", s, B, ctx, eb, wb)) / L
    if cls == "gemm_lm_head":
        return V * d * wb + sc(V) + act(d) + B * V * 4
    if cls == "attention":
        return sum(c + 1 for c in ctx) * hkv * hd * 2 * eb + B * hq * hd * 4 + B * hq * hd * 2 * 2
    if cls == "sampler":
        return B * V * 4 * 4
    return None


def measured_traffic(cls, args):
    """DRAM bytes per launch of a kernel class from a committed ncu summary
    under profiles/ (dram__bytes_read + dram__bytes_write), when it was taken
    on this workload and the kernel's source is unchanged since; else None."""
    import hashlib
    files = {"attention": ("attn_stream_7b_B32_2layer.md", ("k_attn.cu", "attn_stream.cuh"))}
    if cls not in files or (args.shape, args.B, args.ctx_lo, args.ctx_hi, args.seed, args.kv) != \
            ("7b", 32, 256, 4096, 0, "bf16"):
        return None
    prof, srcs = files[cls]
    try:
        text = open(os.path.join(ROOT, "profiles", prof)).read()
        cur = hashlib.sha256()
        for src in srcs:
            cur.update(open(os.path.join(ROOT, "continuous_batching_decode_gb300", "csrc", src), "rb").read())
    except OSError:
        return None
    key = "source_sha256 " + "+".join(srcs) + ":"
    val = sha = None
    for line in text.splitlines():
        if line.startswith("traffic_per_launch_bytes:"):
            val = int(line.split(":")[1])
        if line.startswith(key):
            sha = line.split(":")[1].strip()
    return val if val is not None and sha == cur.hexdigest() else None


def host_mem_available_gb():
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    return int(ln.split()[1]) / 2**20
    except OSError:
        pass
    return 0.0


def oracle_kv(s, ctx, seed):
    """KV state of the oracle for the timed step: random bf16 values (the
    device pool holds random bf16 too), one [c+2, H_kv, hd] array per row and
    per K / V, shared by every layer -- each layer reads and writes the same
    shapes as with distinct arrays, and the host holds 1/L of the bytes."""
    from oracle import model as om
    cfg = om.ModelConfig(**s)
    rng = np.random.default_rng(seed)
    kv = {}
    for i, c in enumerate(ctx):
        q = om.SequenceKV(om.ModelConfig(**dict(s, n_layers=1)), c + 2)
        shp = (c + 2, s["n_kv_heads"], s["head_dim"])
        K = om.round_to_bf16(rng.standard_normal(shp, dtype=np.float32).astype(np.float64) * 1.3)
        V = om.round_to_bf16(rng.standard_normal(shp, dtype=np.float32).astype(np.float64) * 1.3)
        q.K = [K] * cfg.n_layers
        q.V = [V] * cfg.n_layers
        q.length = c
        kv[i] = q
    return kv


def oracle_model(s, weights, cache, int8=False):
    from oracle import model as om
    return om.OracleModel(om.ModelConfig(**s), weights, cache=cache, weight_format="int8" if int8 else "bf16")


def oracle_step_seconds(model, kv, rows):
    """Wall time of one oracle step over `rows` (all layers, the LM head)."""
    from oracle import model as om
    t0 = time.perf_counter()
    om.step(model, kv, rows)
    return time.perf_counter() - t0


def host_weight_bits(s, seed):
    """The workload's weights generated on the host (the same seeded draw the
    device weights come from), as bf16 bit arrays."""
    from continuous_batching_decode_gb300 import synth
    w = synth.make_weights(s, seed=seed, device="cpu")
    return {k: synth.bf16_bits(v) for k, v in w.items()}


def run_reference(args):
    """CPU oracle arm on the host cores: every step runs the oracle over a
    bounded sample of the workload's rows (all layers, the LM head)."""
    s = shape_of(args)
    B = args.B
    wl = workload(s, B, args.ctx_lo, args.ctx_hi, args.seed)
    bits = host_weight_bits(s, args.seed)
    # fp64 copies of every layer stay cached across steps when the host has
    # room for them (~8 bytes per parameter), else each step upcasts per layer
    cache = host_mem_available_gb() > 1.5 * 8 * sum(v.size for v in bits.values()) / 2**30
    model = oracle_model(s, bits, cache, args.weights == "int8")
    kv = oracle_kv(s, wl["ctx"], args.seed + 2)
    rows = [(r[0], r[1], r[2], 1) for r in wl["rows"]]
    # Each step is a bounded sample of the workload so that the whole
    # --steps K --warmup W run ends within ~150 s of host time: b of the B
    # rows (a rotating window, all layers and the LM head), b chosen from two
    # one-row calibration steps (the first also fills the weight cache); the
    # rate is rows run / time.  The decode rows are independent, so a step of
    # b rows is b/B of the step's work.
    budget_s = 150.0
    oracle_step_seconds(model, kv, rows[:1])
    t_row = oracle_step_seconds(model, kv, rows[1:2] if B > 1 else rows[:1])
    n_left = max(1, args.warmup + args.steps - 2)
    b = int(max(1, min(B, budget_s / n_left / max(t_row, 1e-6))))
    ts = []
    for i in range(max(0, args.warmup - 2) + args.steps):
        j0 = (i * b) % B
        sub = [rows[(j0 + j) % B] for j in range(b)]
        t = oracle_step_seconds(model, kv, sub)
        if i >= max(0, args.warmup - 2):
            ts.append(t)
    t = sum(ts) / len(ts)
    value = b / t
    cores = len(os.sched_getaffinity(0))
    sample = (f"{b} of the {B} rows per step (a rotating window; {s['n_layers']} layers and the LM head), each "
              f"step timed, {'whole steps' if b == B else 'rate = rows run / time'}; fp64 weights "
              f"{'cached after the first calibration step' if cache else 'upcast per layer every step'}; KV random "
              "bf16 per row, shared by the layers")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1000 * B / b, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(args, s, wl, args.gpus),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_cbd(args):
    if args.kv == "fp8":
        args.no_cpu_baseline = True      # the oracle sample reads a bf16 pool
    import torch
    import continuous_batching_decode_gb300 as cbd
    from continuous_batching_decode_gb300 import build, replicas, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    if rank == 0 or world == 1:
        build.build()
    if dist:
        dist.barrier()
    cbd.lib()
    dev = torch.cuda.current_device()
    s = shape_of(args)
    B = args.B
    wl = workload(s, B, args.ctx_lo, args.ctx_hi, args.seed)
    w = synth.make_weights(s, seed=args.seed, device="cuda")
    fp8 = args.kv == "fp8"
    eb = 1 if fp8 else 2
    sweep = [int(x) for x in args.sweep.split(",") if x.strip()]
    b_cap = max([B] + sweep)
    i8 = args.weights == "int8"
    wb = 1 if i8 else 2
    cfg = cbd.make_config(s, max_rows=max(b_cap, 64), max_slots=max(b_cap, 8), max_blocks_per_seq=wl["mbps"],
                          kv_fp8=fp8, weights_int8=i8)
    e = cbd.engine_create(cfg, w)
    cbd.engine_set_gemm_path(e, args.gemm_path)
    cbd.engine_set_rows_gemm(e, args.rows_gemm, args.rows_gemm_force)
    cbd.engine_set_attention_path(e, args.attn_path)
    cbd.engine_set_l2_prefetch(e, args.l2_prefetch_mb << 20)
    cbd.engine_set_gemm_chain(e, args.gemm_chain)
    host_bits = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host_bits = {k: synth.bf16_bits(v) for k, v in w.items()}
    del w
    torch.cuda.empty_cache()

    def make_pool(n_pool):
        p = cbd.kv_pool_create(e, n_pool)
        base, nbytes, nb = cbd.kv_pool_data(p)
        # [L][n_blocks][H_kv][K|V][32 * hd]: each tile in 128-byte-swizzled order
        view = cbd.device_view(base, (s["n_layers"], nb, s["n_kv_heads"], 2, 32 * s["head_dim"]),
                               "u8" if fp8 else "bf16")
        gen = torch.Generator(device="cuda").manual_seed(args.seed + 3)
        for l in range(s["n_layers"]):
            r = torch.randn(view[l].shape, generator=gen, device="cuda") * 1.3
            view[l].copy_(r.to(torch.float8_e4m3fn).view(torch.uint8) if fp8 else r.to(torch.bfloat16))
        return p
    pool = make_pool(wl["n_pool"])
    stream = torch.cuda.current_stream()
    b = cbd.batch_create(e, pool, wl["rows"], wl["tables"], wl["nbps"], wl["samp"])
    out = torch.zeros(B, dtype=torch.int32, device="cuda")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # launch by launch (the PDL chain enqueued kernel by kernel): reported beside
    for _ in range(args.warmup):
        cbd.batch_run(e, pool, b, out)
    torch.cuda.synchronize()
    ev0.record(stream)
    th0 = time.perf_counter()
    for _ in range(args.steps):
        cbd.batch_run(e, pool, b, out)
    lbl_host_us = (time.perf_counter() - th0) / args.steps * 1e6
    ev1.record(stream)
    torch.cuda.synchronize()
    lbl = {"ms_per_step": round(ev0.elapsed_time(ev1) / args.steps, 4),
           "host_enqueue_us_per_step": round(lbl_host_us, 1)}
    cbd.engine_check(e)
    # the timed steps replay the step as one CUDA graph (cbd_batch_set_graph:
    # the same kernels and programmatic edges, one host launch per step)
    cbd.batch_set_graph(b, True)
    for _ in range(args.warmup):
        cbd.batch_run(e, pool, b, out)
    torch.cuda.synchronize()
    cbd.engine_check(e)

    clk = Clocks(dev)
    clk.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    th0 = time.perf_counter()
    for _ in range(args.steps):
        cbd.batch_run(e, pool, b, out)
    host_us = (time.perf_counter() - th0) / args.steps * 1e6
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = clk.stop()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    cbd.engine_check(e)
    # replicas: the units all ranks processed / the slowest rank's time
    ms = replicas.max_over_ranks(ms_local, dist, "cuda")
    value = replicas.job_throughput(float(B), ms_local / 1000.0, dist, "cuda")
    launches = cbd.batch_launches(b) * args.steps

    graph = {"replay": True, "host_enqueue_us_per_step": round(host_us, 1), "captures": cbd.batch_captures(b),
             "launch_by_launch": lbl}
    cbd.batch_set_graph(b, False)

    # per-kernel live timing (same batch, same stream, CUDA events per launch)
    cbd.engine_profile(e, True)
    for _ in range(args.steps):
        cbd.batch_run(e, pool, b, out)
    prof = cbd.engine_profile_read(e)
    cbd.engine_profile(e, False)
    peak, peak_kind = peaks()
    dom = max(prof, key=lambda k: prof[k][1])
    ranked = sorted(((v[1], k) for k, v in prof.items()), reverse=True)
    roof = None
    for _, k in ranked:
        byt = kernel_bytes(k, s, B, wl["ctx"], eb, wb)
        if byt:
            n_l, tot = prof[k]
            avg_s = tot / n_l / 1000.0
            ach = byt / avg_s / 1e9
            roof = {"kernel": k, "bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(ach / peak, 4), "traffic": measured_traffic(k, args), "peak_kind": peak_kind,
                    "bytes_per_launch": byt, "avg_launch_us": round(avg_s * 1e6, 2)}
            break
    W = weight_bytes(s, i8)
    A = sum(c + 1 for c in wl["ctx"]) * kv_pos_bytes(s, eb)
    step_bytes = W + A
    step_roof = {"W_bytes": W, "BA_bytes": A, "bytes_per_step": step_bytes,
                 "achieved_GBs": round(step_bytes / (ms / 1000.0) / 1e9, 1),
                 "frac_of_measured": round(step_bytes / (ms / 1000.0) / 1e9 / peak, 4),
                 "frac_of_8TBs": round(step_bytes / (ms / 1000.0) / 8e12, 4),
                 "roofline_tok_s_8TBs": round(B / (step_bytes / 8e12), 1)}
    kernels = {k: {"launches": v[0], "ms_per_step": round(v[1] / args.steps, 4),
                   "share": round(v[1] / sum(x[1] for x in prof.values()), 4)} for k, v in prof.items()}

    # end to end through cbd_step: host arrays in, tokens out, every step.
    # The inputs are marshalled once into the C layout (cbd.rows_table /
    # sampling_table); every step then writes the tokens the previous step
    # drew into the rows, as a decode loop does (positions stay fixed, so
    # every step does the same work).
    e2e = None
    if not args.no_e2e:
        host_tok = torch.zeros(B, dtype=torch.int32).pin_memory()
        rows_t = cbd.rows_table(wl["rows"])
        samp_t = cbd.sampling_table(wl["samp"])
        tables_t = np.ascontiguousarray(wl["tables"], dtype=np.int32)
        nbps_t = np.ascontiguousarray(wl["nbps"], dtype=np.int32)
        tok_np = host_tok.numpy()

        def one_step():
            cbd.step(e, pool, rows_t, tables_t, nbps_t, samp_t, None, out)
            host_tok.copy_(out, non_blocking=True)
            stream.synchronize()
            rows_t["token"] = tok_np
            samp_t["token_index"] += 1

        def e2e_ms():
            for _ in range(3):
                one_step()
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            ev0.record(stream)
            for _ in range(args.steps):
                one_step()
            ev1.record(stream)
            torch.cuda.synchronize()
            wall = (time.perf_counter() - t0) / args.steps * 1000.0
            return replicas.max_over_ranks(max(ev0.elapsed_time(ev1) / args.steps, wall), dist, "cuda")
        lbl_ms = e2e_ms()                       # launch by launch
        cbd.engine_set_step_graph(e, True)      # each cbd_step as one cached graph
        sync_ms = e2e_ms()

        # Pipelined decode loop: rows carry CBD_TOKEN_LAST (each slot's
        # last drawn token, read on the device), so the host enqueues step
        # k + 1 without waiting for step k's tokens; every step's tokens are
        # still copied back, asynchronously, into a pinned ring.
        rows_last = rows_t.copy()
        rows_last["token"] = cbd.TOKEN_LAST
        ring = torch.zeros(args.steps, B, dtype=torch.int32).pin_memory()

        def pipelined_ms():
            for _ in range(3):
                one_step()                      # explicit tokens: every slot has a last token
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            ev0.record(stream)
            for k in range(args.steps):
                cbd.step(e, pool, rows_last, tables_t, nbps_t, samp_t, None, out)
                ring[k].copy_(out, non_blocking=True)
                samp_t["token_index"] += 1
            ev1.record(stream)
            torch.cuda.synchronize()
            wall = (time.perf_counter() - t0) / args.steps * 1000.0
            return replicas.max_over_ranks(max(ev0.elapsed_time(ev1) / args.steps, wall), dist, "cuda")
        e_ms = pipelined_ms()
        cbd.engine_set_step_graph(e, False)
        h2d = len(wl["rows"]) * 20 + wl["tables"].nbytes + wl["nbps"].nbytes + len(wl["samp"]) * 48
        e2e = {"value": B * world / (e_ms / 1000.0), "unit": "tok/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": B * 4, "ms_per_step": round(e_ms, 4), "step_graph": True,
               "loop": "pipelined: each step's rows take the slot's last drawn token on the device "
                       "(CBD_TOKEN_LAST) and its tokens are copied back asynchronously; positions fixed",
               "sync_loop": {"value": B * world / (sync_ms / 1000.0), "ms_per_step": round(sync_ms, 4),
                             "loop": "tokens read back and fed in from the host before the next step"},
               "launch_by_launch_ms_per_step": round(lbl_ms, 4)}
        cbd.engine_check(e)

    cbd.batch_destroy(b)
    cbd.kv_pool_destroy(pool)

    # B sweep ("20.3 服务、批处理与流式" section 20.3.2: throughput grows with B
    # while the weight stream is shared): one pool for the largest B, each B
    # the first B rows of that draw, every step replayed as a graph
    sweep_out = {}
    if sweep:
        wls = workload(s, b_cap, args.ctx_lo, args.ctx_hi, args.seed)
        pool = make_pool(wls["n_pool"])
        outs = torch.zeros(b_cap, dtype=torch.int32, device="cuda")
        for Bs in sorted(set(sweep + [B])):
            b2 = cbd.batch_create(e, pool, wls["rows"][:Bs], wls["tables"], wls["nbps"], wls["samp"][:Bs])
            cbd.batch_set_graph(b2, True)
            for _ in range(args.warmup):
                cbd.batch_run(e, pool, b2, outs)
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            ev0.record(stream)
            for _ in range(args.steps):
                cbd.batch_run(e, pool, b2, outs)
            ev1.record(stream)
            torch.cuda.synchronize()
            ms2 = replicas.max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dist, "cuda")
            by = W + sum(c + 1 for c in wls["ctx"][:Bs]) * kv_pos_bytes(s, eb)
            sweep_out[str(Bs)] = {"ms_per_step": round(ms2, 4), "tok_s": round(Bs * world / ms2 * 1000, 1),
                                  "mean_ctx": round(float(np.mean(wls["ctx"][:Bs])), 1),
                                  "GBs": round(by / ms2 / 1e6, 1), "frac_of_measured": round(by / ms2 / 1e6 / peak, 4),
                                  "frac_of_8TBs": round(by / ms2 / 1e6 / 8000, 4)}
            cbd.batch_destroy(b2)
        cbd.engine_check(e)
        cbd.kv_pool_destroy(pool)

    # the CPU oracle, one whole step of this workload on the host cores
    cpu = None
    if host_bits is not None:
        model = oracle_model(s, host_bits, cache=False, int8=i8)
        okv = oracle_kv(s, wl["ctx"], args.seed + 2)
        t_step = oracle_step_seconds(model, okv, [(r[0], r[1], r[2], 1) for r in wl["rows"]])
        del okv, model, host_bits
        cpu = {"value": round(B / t_step, 4), "unit": "tok/s", "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle", "step_s": round(t_step, 2),
               "sample": (f"one whole step timed: {s['n_layers']} layers for all {B} rows plus the LM head, fp64 "
                          f"weights upcast per layer{' (quantised to int8 and back)' if i8 else ''}; KV random bf16 "
                          "per row, shared by the layers")}

    line = {"metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 (int8 weights)" if i8 else "bf16", "data": "synthetic (seeded random-init weights, random bf16 KV)",
            "config": dict(config_of(args, s, wl, world), gemm_path=args.gemm_path, attn_path=args.attn_path,
                           l2_prefetch_mb=args.l2_prefetch_mb, gemm_chain=args.gemm_chain),
            "roofline": roof, "step_roofline": step_roof, "kernels": kernels, "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks, "cpu_baseline": cpu, "graph": graph, "sweep": sweep_out}
    if rank == 0:
        print(json.dumps(line), flush=True)
    cbd.engine_destroy(e)
    if dist:
        dist.destroy_process_group()


def run_mixed(args):
    """A mixed step ("20.3 服务、批处理与流式" section 20.3.2: prefill chunks
    share the step with decode rows): the B decode rows of the default
    workload plus `--mixed` prefill rows, as 512-row chunks at positions
    0..511 of new slots.  Reports the step time and the weight contractions'
    algorithmic throughput (2 x parameters x rows) against the measured bf16
    tensor peak (the contraction is compute-bound at this many rows)."""
    import torch
    import continuous_batching_decode_gb300 as cbd
    from continuous_batching_decode_gb300 import build, synth

    torch.cuda.set_device(0)
    build.build()
    s = shape_of(args)
    B, P = args.B, args.mixed
    nch = (P + 511) // 512
    db = synth.decode_batch(B, args.ctx_lo, args.ctx_hi, s["vocab"], args.seed)
    ctx = db["contexts"]
    need = {i: (c + 1 + 31) // 32 for i, c in enumerate(ctx)}
    for j in range(nch):
        need[B + j] = 16
    mbps = max((args.ctx_hi + 1 + 31) // 32, 16)
    n_pool = sum(need.values()) + 8
    tables, nbps = synth.permuted_tables(need, n_pool, mbps, np.random.default_rng(args.seed + 1))
    rng = np.random.default_rng(args.seed + 2)
    rows = [(i, db["tokens"][i], ctx[i], 0, 1) for i in range(B)]
    for j in range(nch):
        n = min(512, P - 512 * j)
        toks = synth.random_tokens(rng, n, s["vocab"])
        rows += [(B + j, toks[i], i, 1, 1 if i == n - 1 else 0) for i in range(n)]
    m = sum(1 for r in rows if r[4])
    samp = [dict(temperature=1.0, top_p=0.3, frequency_penalty=1.0, penalty_decay=0.996, seed=args.seed,
                 request_id=i) for i in range(m)]
    w = synth.make_weights(s, seed=args.seed, device="cuda")
    fp8 = args.kv == "fp8"
    e = cbd.engine_create(cbd.make_config(s, max_rows=len(rows), max_slots=B + nch, max_blocks_per_seq=mbps,
                                          kv_fp8=fp8), w)
    del w
    torch.cuda.empty_cache()
    cbd.engine_set_rows_gemm(e, args.rows_gemm, args.rows_gemm_force)
    cbd.engine_set_prefill_attention(e, not args.no_prefill_attn)
    pool = cbd.kv_pool_create(e, n_pool)
    base, nbytes, nb = cbd.kv_pool_data(pool)
    kv = cbd.device_view(base, (s["n_layers"], nb, s["n_kv_heads"], 2, 32 * s["head_dim"]), "u8" if fp8 else "bf16")
    gen = torch.Generator(device="cuda").manual_seed(args.seed + 3)
    for l in range(s["n_layers"]):
        r = torch.randn(kv[l].shape, generator=gen, device="cuda") * 1.3
        kv[l].copy_(r.to(torch.float8_e4m3fn).view(torch.uint8) if fp8 else r.to(torch.bfloat16))
    b = cbd.batch_create(e, pool, rows, tables, nbps, samp)
    out = torch.zeros(m, dtype=torch.int32, device="cuda")
    cbd.batch_set_graph(b, True)
    for _ in range(args.warmup):
        cbd.batch_run(e, pool, b, out)
    torch.cuda.synchronize()
    cbd.engine_check(e)
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        cbd.batch_run(e, pool, b, out)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / args.steps
    cbd.batch_set_graph(b, False)
    cbd.engine_profile(e, True)
    for _ in range(args.steps):
        cbd.batch_run(e, pool, b, out)
    prof = cbd.engine_profile_read(e)
    cbd.engine_profile(e, False)
    cbd.engine_check(e)
    d, hq, hkv, hd, F, V, L = (s[k] for k in ("d_model", "n_heads", "n_kv_heads", "head_dim", "ffn_dim", "vocab",
                                             "n_layers"))
    layer_params = (hq + 2 * hkv) * hd * d + d * hq * hd + 3 * F * d
    n = len(rows)
    flops = 2.0 * (L * layer_params * n + V * d * m)
    gemm_ms = sum(v[1] for k, v in prof.items() if k.startswith("gemm")) / args.steps
    try:
        peak_tf = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"])
        kind = "measured"
    except Exception:
        peak_tf, kind = 1900.0, "fallback"
    ach = flops / (gemm_ms / 1000.0) / 1e12
    line = {"metric": "mixed step: rows/s and weight-contraction TFLOP/s", "impl": "cbd",
            "value": round(n / (ms / 1000.0), 1), "unit": "rows/s", "ms_per_step": round(ms, 4),
            "rows": n, "decode_rows": B, "prefill_rows": P, "sampled_rows": m,
            "gemm": {"bound": "tensor", "achieved": round(ach, 1), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(ach / peak_tf, 4), "peak_kind": kind, "algorithmic_flops": flops,
                     "ms_per_step": round(gemm_ms, 4),
                     "note": "2 x params x rows; the MMAs also multiply the lo half of each activation (2x issued)"},
            "kernels": {k: round(v[1] / args.steps, 4) for k, v in prof.items()},
            "config": {"workload": f"{args.shape}-shaped mixed step: {B} decode rows (ctx U[{args.ctx_lo},"
                                   f"{args.ctx_hi}]) + {P} prefill rows in 512-row chunks", "shape": args.shape,
                       "rows_gemm_min": args.rows_gemm, "rows_gemm_force": args.rows_gemm_force,
                       "kv": "e4m3" if fp8 else "bf16", "prefill_attention": not args.no_prefill_attn},
            "data": "synthetic (seeded random-init weights, random bf16 KV, random prompt ids)"}
    print(json.dumps(line), flush=True)
    cbd.batch_destroy(b)
    cbd.kv_pool_destroy(pool)
    cbd.engine_destroy(e)


def run_trace(args):
    import torch
    import continuous_batching_decode_gb300 as cbd
    from continuous_batching_decode_gb300 import build, serve, synth

    torch.cuda.set_device(0)
    build.build()
    s = shape_of(args)
    slots, rows, mbps = 64, 2048, 64
    w = synth.make_weights(s, seed=args.seed, device="cuda")
    fp8 = args.kv == "fp8"
    e = cbd.engine_create(cbd.make_config(s, max_rows=rows, max_slots=slots, max_blocks_per_seq=mbps, kv_fp8=fp8), w)
    del w
    torch.cuda.empty_cache()
    reqs = synth.request_trace(args.trace_requests, s["vocab"], seed=args.seed,
                               rate=args.trace_rate if args.trace_rate > 0 else None)
    samp = dict(temperature=1.0, top_p=0.3, top_k=0, frequency_penalty=1.0, penalty_decay=0.996)
    for r in reqs:
        r["sampling"] = dict(samp, seed=args.seed + 11)
    policies = ["forma", "albatross"] if args.policy == "both" else [args.policy]
    for pol in policies:
        pool = cbd.kv_pool_create(e, args.trace_blocks)
        srv = serve.Server(e, pool, n_blocks=args.trace_blocks, max_slots=slots, max_rows=rows,
                           max_blocks_per_seq=mbps, vocab=s["vocab"], chunk=512, answer_budget=128, policy=pol)
        try:
            res = srv.run(reqs)
        finally:
            srv.close()
            cbd.kv_pool_destroy(pool)
        ttft = res["ttft"]
        line = dict(metric="trace generated tok/s (wall clock, host loop included)", impl="cbd",
                    value=round(res["tok_s"], 1), unit="tok/s", policy=pol, requests=len(reqs),
                    generated=res["generated"], wall_s=round(res["wall_s"], 3), steps=res["steps"],
                    rows_per_step=round(res["rows"] / max(res["steps"], 1), 1),
                    ttft_s=dict(mean=round(float(ttft.mean()), 4), p50=round(float(np.median(ttft)), 4),
                                p99=round(float(np.quantile(ttft, 0.99)), 4)),
                    stalled_rows=res["stats"]["stalled_rows"], fallback_stops=res["stats"]["fallback_stops"],
                    host_sched_us_per_step=round(res["sched_us_per_step"], 1),
                    config=dict(workload="7b-shaped continuous-batching trace", slots=slots, max_rows=rows,
                                chunk=512, answer_budget=128, pool_blocks=args.trace_blocks,
                                rate=args.trace_rate or "all at t=0", kv="e4m3" if fp8 else "bf16"),
                    data="synthetic (seeded random-init weights, random prompt ids)")
        print(json.dumps(line), flush=True)


def spawn_ranks(n):
    """Re-run this command under torch.distributed.run with n ranks on this
    node (127.0.0.1 rendezvous); returns its exit status."""
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    args = parse()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and not (args.trace or args.mixed):
        sys.exit(spawn_ranks(args.gpus))
    if "WORLD_SIZE" in os.environ:
        print(f"bench rank {os.environ.get('RANK', '0')} of {os.environ['WORLD_SIZE']}", file=sys.stderr, flush=True)
    if args.trace:
        run_trace(args)
        return
    if args.mixed:
        run_mixed(args)
        return
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args)
        return
    run_cbd(args)


if __name__ == "__main__":
    main()
