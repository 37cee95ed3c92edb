#!/usr/bin/env python
"""Benchmark of the FlashAttention forward hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * prefill  fa_fwd, causal, B=4 H=32 Sq=Sk=4096 d=128 bf16, Q,K,V ~ N(0,1)
  * decode   fa_decode_paged, B=32 H=32 d=128 fp16, ctx ~ U[1,8192], 256-token
             pages scattered over a pool of 1200 pages by a random permutation
`value` is the prefill throughput in TFLOP/s (4*B*H*d * visible pairs, masked pairs
not counted), timed with CUDA events around each prefill launch; the decode
throughput (algorithmic HBM bytes / time) is reported beside it under "decode".
Inputs are larger than L2 (prefill Q+K+V 402 MB, decode K/V 2.2 GB), so no flush
is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload default|causal2k|causal4k|noncausal4k|window32k|decode|sweep]
With --gpus N > 1 run under torchrun: every rank runs the same workload on its own
GPU (replicas; no collective on the data path), value = N * units / max rank time.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense FP16/BF16 tensor-core rate of one GB300: NVIDIA's GB300 NVL72 figure, 360
# PFLOPS FP16/BF16 for 72 GPUs, which NVIDIA quotes with 2:4 sparsity, halved for dense math.
# A chain of tcgen05 128x128x16 bf16 MMAs on this GPU runs one MMA per 65 SM cycles, about
# 8050 FLOP per cycle per SM, i.e. 2.53 PFLOP/s at 2070 MHz on 152 SMs: the same figure.
NOMINAL_BF16_TFLOPS = 2500.0
NOMINAL_SOURCE = ("NVIDIA GB300 NVL72 spec: FP16/BF16 tensor core 360 PFLOPS per 72 GPUs with "
                  "2:4 sparsity = 2.5 PFLOP/s dense per GPU (a tcgen05 MMA chain measures 2.53 at "
                  "2070 MHz)")
# Untimed steps run back to back while the clock sampler is on, just before the timed
# ones, so that the sampled clocks show the kernels under sustained load even when the
# timed region itself is short.
CLOCK_SOAK_S = 1.5

PREFILL = {
    "causal2k": dict(B=4, H=32, S=2048, d=128, dtype="f16", mode=1, window=0, n_global=0,
                     factor=0.5),
    "causal4k": dict(B=4, H=32, S=4096, d=128, dtype="bf16", mode=1, window=0, n_global=0,
                     factor=1.0),
    "noncausal4k": dict(B=4, H=32, S=4096, d=128, dtype="bf16", mode=0, window=0, n_global=0,
                        factor=1.0),
    "window32k": dict(B=1, H=32, S=32768, d=128, dtype="bf16", mode=2, window=2048,
                      n_global=64, factor=1.0),
    # the pages give no width for these two masks: band +-512 keys, a 1024-key prefix
    "band4k": dict(B=4, H=32, S=4096, d=128, dtype="bf16", mode=3, window=512, n_global=0,
                   factor=1.0),
    "prefixlm4k": dict(B=4, H=32, S=4096, d=128, dtype="bf16", mode=4, window=0, n_global=1024,
                       factor=1.0),
    # BigBird-shaped layout of 128 x 128 blocks (the pages give none): local +-1 block,
    # 1 global block row and column, 2 random blocks per row, seeded
    "blocksparse4k": dict(B=4, H=32, S=4096, d=128, dtype="bf16", mode=5, window=0, n_global=0,
                          factor=1.0, layout=dict(local=1, n_global=1, n_random=2)),
    # FP32 inputs and output (each product formed from bf16 high and low parts)
    "causal4k_f32": dict(B=4, H=32, S=4096, d=128, dtype="f32", mode=1, window=0, n_global=0,
                         factor=1.0),
}
DECODE = dict(B=32, H=32, d=128, page=256, pool=1200, max_ctx=8192, dtype="f16")
PREFIX_WORKLOADS = ("default", "decode", "causal2k", "causal4k", "causal4k_f32", "noncausal4k",
                    "window32k",
                    "band4k", "prefixlm4k")
MODE_NAME = {0: "none", 1: "causal", 2: "causal_window", 3: "band", 4: "prefix_lm",
             5: "block_sparse"}

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# capture of each kernel, with the workloads it holds for and the SHA-256 of the kernel
# sources it was taken on; the figure is reported only for those workloads and only while
# those sources are unchanged. Summaries: profiles/.
NCU_TRAFFIC = {
    # prefill_bm256_kernel, causal 4k B4 H16 capture: 213.7 MB read + 47.4 MB written,
    # scaled x2 to B4 H32
    "prefill": {"bytes": 522.13e6, "workloads": ("default", "causal4k"),
                "sources": ['fa_prefill.cu', 'fa_mma.cuh', 'fa_ptx.cuh', 'fa_plan.h', 'fa_internal.h'],
                "sha256": "c1b9809d6f61876576f34769600da90cb7e0305adedb690f307a790ba94d7552"},
    # paged decode B8 capture: 547.5 MB read + 4.9 MB written for 547.5 MB algorithmic,
    # scaled to the bench call's 2410.7 MB algorithmic
    "decode": {"workloads": ("default", "decode"), "bytes": 2.4321e9, "sources": ['fa_decode.cu', 'fa_ptx.cuh', 'fa_internal.h'],
               "sha256": "8cb2b4a6b72f7981946d2f596fca13eefd0d352127ef81533f9ce99792534363"},
    # FP32 inputs, causal 4k B4 H16 capture of one call: split_bf16_kernel 402.7 MB read +
    # 345.3 MB written, prefill_bm256_kernel (split) 409.0 MB read + 110.4 MB written;
    # scaled x2 to B4 H32
    "prefill_f32": {"bytes": 2534.8e6, "workloads": ("causal4k_f32",),
                    "sources": ['fa_prefill.cu', 'fa_prefill_split.cu', 'fa_mma.cuh', 'fa_ptx.cuh',
                                'fa_plan.h', 'fa_internal.h'],
                    "sha256": "38ee28e9d1c5bcc0f491957be24204c5a35718fa816be5b62740ffacfc4b37b1"},
}


def sources_sha(names):
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "tiled_attention_06_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic(kind, workload, override):
    if override is not None:
        return override
    t = NCU_TRAFFIC[kind]
    if t["bytes"] is None or workload not in t["workloads"] or \
            t["sha256"] != sources_sha(t["sources"]):
        return None
    return t["bytes"]


# --------------------------------------------------------------------------- accounting
def row_visible(pos, Sk, mode, window=0, n_global=0):
    """Keys visible to the query at key position `pos` (closed form of the mask)."""
    if mode == 0:
        return Sk
    if mode == 3:  # |pos - j| <= window
        return max(0, min(pos + window, Sk - 1) - max(pos - window, 0) + 1)
    if mode == 4:  # j <= pos or j < n_global
        return max(0, min(max(pos + 1, n_global), Sk))
    if pos < 0:
        return 0
    hi = min(pos, Sk - 1) + 1
    if mode == 1:
        return hi
    lo = max(0, pos - window + 1)
    return max(0, hi - lo) + max(0, min(n_global, hi, lo))


def visible_pairs(Sq, Sk, mode, window=0, n_global=0):
    """Number of (query, key) pairs the mask leaves visible."""
    delta = Sk - Sq
    return sum(row_visible(i + delta, Sk, mode, window, n_global) for i in range(Sq))


def layout_pairs(layout, Sq, Sk, block=128, heads=None):
    """Visible (query, key) pairs of a block layout [H, nqb, nkb], summed over its heads
    (or the listed ones): each set block counts its rows x keys, clipped at Sq and Sk."""
    lay = np.asarray(layout, dtype=np.int64)
    if heads is not None:
        lay = lay[list(heads)]
    rows = np.minimum(block, Sq - block * np.arange(lay.shape[1]))
    keys = np.minimum(block, Sk - block * np.arange(lay.shape[2]))
    return int(np.einsum("hij,i,j->", lay, rows, keys))


def make_layout(cfg):
    from tiled_attention_06_gb300 import inputs
    return inputs.block_layout(cfg["H"], cfg["S"], cfg["S"], **cfg["layout"])


def prefill_flops(cfg, layout=None):
    if cfg["mode"] == 5:
        if layout is None:
            layout = make_layout(cfg)
        return 4.0 * cfg["B"] * cfg["d"] * layout_pairs(layout, cfg["S"], cfg["S"])
    return 4.0 * cfg["B"] * cfg["H"] * cfg["d"] * visible_pairs(cfg["S"], cfg["S"], cfg["mode"],
                                                                cfg["window"], cfg["n_global"])


def decode_bytes(ctx_lens, B, H, d, max_pages, elem=2):
    kv = int(sum(int(c) for c in ctx_lens)) * H * d * elem * 2
    return kv + 2 * B * H * d * elem + B * H * 4 + B * max_pages * 4 + B * 4


def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return pk, "measured"
    return FALLBACK, "fallback"


# --------------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        rank = dist.get_rank()
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
        return rank, world
    return 0, 1


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest value of x across ranks (host collective; not on the data path)."""
    if world == 1:
        return float(x)
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank, max_seconds, world):
    """Whole-job throughput: every rank processed units_per_rank in at most max_seconds."""
    return units_per_rank * world / max_seconds


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    # where the raw samples go: --clock-log PATH, else the system's temporary directory
    log_path = None

    def __init__(self, device_index):
        import tempfile
        self.idx = device_index
        self.proc = None
        self.path = ClockSampler.log_path or os.path.join(tempfile.gettempdir(),
                                                          f"fa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}",
                                          f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sms, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1].split()[0]))
                mx = float(parts[2].split()[0])
                power.append(float(parts[3].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms),
                "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------- our arm
def make_prefill(cfg, dev, seed=0):
    from tiled_attention_06_gb300 import inputs
    dt = inputs.DTYPES[cfg["dtype"]]
    q, k, v = inputs.prefill_inputs(cfg["B"], cfg["H"], cfg["S"], cfg["S"], cfg["d"], dt,
                                    factor=cfg["factor"], seed=seed)
    return q, k, v


def make_decode(dev, seed=0):
    from tiled_attention_06_gb300 import inputs
    c = DECODE
    return inputs.decode_inputs(B=c["B"], H=c["H"], d=c["d"], page_size=c["page"],
                                num_pages=c["pool"], max_ctx=c["max_ctx"],
                                dtype=inputs.DTYPES[c["dtype"]], seed=seed)


def run_ours(args, rank, world):
    import tiled_attention_06_gb300 as fa
    from tiled_attention_06_gb300 import build
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks, peak_kind = load_peaks()
    stream = torch.cuda.current_stream()
    workload = "default" if args.workload == "default" else args.workload
    if workload in ("chunked", "multimodal"):
        return run_next_rows(args, fa, workload, peaks, peak_kind, stream, world)
    if workload in ("bwd4k", "bwd_blocksparse4k"):
        return run_backward(args, fa, peaks, stream, world, workload)
    pcfg = PREFILL["causal4k" if workload in ("default", "sweep") else workload] \
        if workload != "decode" else None
    with_decode = workload in ("default", "decode")

    # ---- inputs, resident in HBM before timing
    layout = lay_d = None
    if pcfg:
        q, k, v = make_prefill(pcfg, dev)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        od = torch.empty_like(qd)
        ld = torch.empty(qd.shape[:3], dtype=torch.float32, device=dev)
        if pcfg["mode"] == 5:
            layout = make_layout(pcfg)
            lay_d = layout.to(dev)
        pflops = prefill_flops(pcfg, layout)
        scale = 1 / math.sqrt(pcfg["d"])
        f32 = pcfg["dtype"] == "f32"
        ws32 = torch.empty(max(fa.fa_fwd_workspace_size(pcfg["B"], pcfg["H"], pcfg["S"], pcfg["S"],
                                                        pcfg["d"], fa.FA_F32), 16),
                           dtype=torch.uint8, device=dev) if f32 else None
    if with_decode:
        di = make_decode(dev)
        dq, dk, dv = di.q.to(dev), di.k_pages.to(dev), di.v_pages.to(dev)
        dbt, dcl = di.block_table.to(dev), di.ctx_lens.to(dev)
        do = torch.empty_like(dq)
        dl = torch.empty(dq.shape[:2], dtype=torch.float32, device=dev)
        mp = dbt.shape[1]
        ws = torch.empty(fa.fa_decode_workspace_size(DECODE["B"], DECODE["H"], DECODE["d"], mp,
                                                     DECODE["page"]), dtype=torch.uint8,
                         device=dev)
        dbytes = decode_bytes(di.ctx_lens.tolist(), DECODE["B"], DECODE["H"], DECODE["d"], mp)
        dscale = 1 / math.sqrt(DECODE["d"])

    def prefill_call(host_layout=True, **ex):
        if args.block_m and "block_m" not in ex:
            ex["block_m"] = args.block_m
        if lay_d is not None:
            ex["block_layout"] = lay_d
            if host_layout:  # the layout also on the host, for the work plan
                ex["block_layout_host"] = layout
        if ws32 is not None:
            ex["workspace"] = ws32
        if ex:
            fa.fa_fwd_ex(qd, kd, vd, od, ld, scale, pcfg["mode"], pcfg["window"],
                         pcfg["n_global"], stream=stream, **ex)
        else:
            fa.fa_fwd(qd, kd, vd, od, ld, scale, pcfg["mode"], pcfg["window"], pcfg["n_global"],
                      stream=stream)

    def decode_call():
        if args.pages_per_split:
            fa.fa_decode_paged_ex(dq, dk, dv, dbt, dcl, do, dl, dscale, ws,
                                  pages_per_split=args.pages_per_split, stream=stream)
        else:
            fa.fa_decode_paged(dq, dk, dv, dbt, dcl, do, dl, dscale, ws, stream=stream)

    if workload == "sweep":
        return run_sweep(args, fa, prefill_call, pflops, peaks, peak_kind, pcfg)

    K, W = args.steps, args.warmup
    for _ in range(W):
        if pcfg:
            prefill_call()
        if with_decode:
            decode_call()
    torch.cuda.synchronize()
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("device status after warm-up: " + fa.fa_last_error_string())

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    soak, t_soak = 0, time.perf_counter()
    while time.perf_counter() - t_soak < args.clock_soak:
        for _ in range(8):
            if pcfg:
                prefill_call()
            if with_decode:
                decode_call()
        soak += 8
        torch.cuda.synchronize()
    t_soak = time.perf_counter() - t_soak
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        ev[i][0].record(stream)
        if pcfg:
            prefill_call()
        ev[i][1].record(stream)
        if with_decode:
            decode_call()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("device status after timing: " + fa.fa_last_error_string())
    p_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    d_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    total_ms = max_over_ranks(total_ms, world)
    # an FP32 prefill is two launches: the split into bf16 planes and the prefill kernel
    launches = K * ((0 if not pcfg else 2 if f32 else 1) + (2 if with_decode else 0))

    clk["soak"] = {"steps": soak, "seconds": round(t_soak, 3),
                   "note": "clocks sampled over untimed back-to-back steps just before the "
                           "timed ones, and during them"}
    res = {"n_gpus": world, "steps": K, "warmup": W, "ms_per_step": total_ms / K,
           "scaling": "weak", "vs_baseline": None, "data": "synthetic (seeded N(0,1), "
           "shapes of the pages' workloads; no dataset)", "gpu_launches": launches,
           "clocks": clk}
    hbm_peak = float(peaks["hbm_gbs"])
    # captured traffic holds for the workloads' own shapes only
    tkey = None if (args.batch or args.heads or args.pool or args.dtype) else workload
    if pcfg:
        p_sum = max_over_ranks(sum(p_ms) / 1e3, world)
        p_avg = sum(p_ms) / K / 1e3
        value = aggregate(pflops * K, p_sum, world) / 1e12
        tc_peak = float(peaks["bf16_tflops"])
        achieved = pflops / p_avg / 1e12
        res.update({"metric": "attention fwd TFLOP/s (% BF16 TC peak); paged decode HBM GB/s "
                              "(% of 8 TB/s)",
                    "value": value, "unit": "TFLOP/s", "higher_is_better": True,
                    "dtype": pcfg["dtype"]})
        bm = args.block_m or fa.fa_fwd_default_block_m(pcfg["mode"])
        kname = (f"split_bf16_kernel + prefill_bm256_kernel<{pcfg['d']},64,bf16 split> "
                 "(timed together: one fa_fwd_ex call)" if f32 else
                 f"prefill_bm{bm}_kernel<{pcfg['d']},128,{pcfg['dtype']}>")
        res["roofline"] = {"kernel": kname,
                           "bound": "tensor",
                           "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                           "frac": achieved / tc_peak,
                           "frac_of_sustained": achieved / float(
                               peaks.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"])),
                           "peak_source": f"{peak_kind} bf16 burst (MEASURED_PEAKS.json)"
                           if peak_kind == "measured" else "fallback 1.9 PFLOP/s",
                           "traffic": ncu_traffic("prefill_f32" if f32 else "prefill",
                                                  tkey, args.prefill_traffic),
                           "algorithmic_flops": pflops,
                           "ms_per_launch": p_avg * 1e3,
                           "peak_nominal": NOMINAL_BF16_TFLOPS,
                           "frac_nominal": achieved / NOMINAL_BF16_TFLOPS,
                           "nominal_source": NOMINAL_SOURCE}
        if f32:  # the tensor cores run three bf16 products per product of the method
            res["roofline"]["tensor_flops_executed"] = 3 * pflops
            res["roofline"]["tensor_frac"] = 3 * achieved / tc_peak
    if with_decode:
        d_sum = max_over_ranks(sum(d_ms) / 1e3, world)
        d_avg = sum(d_ms) / K / 1e3
        dval = aggregate(dbytes * K, d_sum, world) / 1e9
        dec = {"value": dval, "unit": "GB/s", "frac_of_8TBs": dval / world / 8000.0,
               "roofline": {"kernel": "decode_split_kernel + decode_merge_kernel",
                            "bound": "hbm", "achieved": dbytes / d_avg / 1e9, "peak": hbm_peak,
                            "unit": "GB/s", "frac": dbytes / d_avg / 1e9 / hbm_peak,
                            "peak_source": f"{peak_kind} copy bandwidth",
                            "traffic": ncu_traffic("decode", tkey, args.decode_traffic), "algorithmic_bytes": dbytes,
                            "ms_per_call": d_avg * 1e3}}
        if pcfg:
            res["decode"] = dec
        else:
            res.update({"metric": "paged decode HBM GB/s (% of 8 TB/s)", "value": dval,
                        "unit": "GB/s", "higher_is_better": True, "dtype": "f16",
                        "roofline": dec["roofline"]})
    if lay_d is not None:  # the same calls planned without the host copy of the layout
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            prefill_call(host_layout=False)
        e1.record(stream)
        torch.cuda.synchronize()
        res["without_host_layout"] = {"value": pflops * K / (e0.elapsed_time(e1) / 1e3) / 1e12,
                                      "unit": "TFLOP/s",
                                      "api": "fa_fwd_ex without block_layout_host (every item "
                                             "planned as dense)"}
    res["config"] = workload_config(pcfg, with_decode, world)

    # ---- end to end through the public API with host buffers
    res["e2e"] = e2e_prefill(fa, pcfg, q, k, v, pflops, scale, stream, world, args, layout,
                             ws32) \
        if pcfg \
        else e2e_decode(fa, di, dbytes, dscale, ws, dk, dv, stream, world, args)
    # ---- CPU baseline: the oracle on a bounded sample, rank 0 only
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(pcfg, q if pcfg else None, k if pcfg else None,
                                           v if pcfg else None,
                                           di if with_decode else None)
    return res


def workload_config(pcfg, with_decode, world):
    cfg = {}
    if pcfg:
        cfg["workload"] = (f"prefill {MODE_NAME[pcfg['mode']]} B{pcfg['B']} H{pcfg['H']} "
                           f"S{pcfg['S']} d{pcfg['d']} {pcfg['dtype']}"
                           + (f" window {pcfg['window']} global {pcfg['n_global']}"
                              if pcfg["mode"] == 2 else ""))
    if with_decode:
        d = DECODE
        dec = (f"paged decode B{d['B']} H{d['H']} d{d['d']} {d['dtype']} ctx~U[1,{d['max_ctx']}] "
               f"page {d['page']} pool {d['pool']}")
        cfg["workload"] = (cfg["workload"] + " + " + dec) if pcfg else dec
    cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
    cfg["l2"] = "inputs larger than L2 (no flush)"
    return cfg


def measure_link(h2d_bytes, d2h_bytes, dev, reps=3):
    """Pinned host <-> device copy bandwidth on this machine, the limit of an end-to-end call:
    one cudaMemcpyAsync (tensor.copy_) of the step's input bytes host to device, one of its
    output bytes device to host, and both directions at once on two streams; CUDA events,
    best of `reps`. GB/s = bytes moved / time."""
    hin = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    hout = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    din = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    dout = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def best(fn):
        t = []
        for _ in range(reps + 1):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s1)
            fn()
            s1.wait_stream(s2)
            e1.record(s1)
            torch.cuda.synchronize()
            t.append(e0.elapsed_time(e1) / 1e3)
        return min(t[1:])

    def h2d():
        with torch.cuda.stream(s1):
            din.copy_(hin, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s1):
            hout.copy_(dout, non_blocking=True)

    def both():
        s2.wait_stream(s1)
        with torch.cuda.stream(s1):
            din.copy_(hin, non_blocking=True)
        with torch.cuda.stream(s2):
            hout.copy_(dout, non_blocking=True)

    t_in, t_out, t_both = best(h2d), best(d2h), best(both)
    del hin, hout, din, dout
    return {"h2d_gbs": h2d_bytes / t_in / 1e9, "d2h_gbs": d2h_bytes / t_out / 1e9,
            "both_ms": t_both * 1e3, "h2d_ms": t_in * 1e3, "d2h_ms": t_out * 1e3,
            "how": "pinned tensor.copy_ (one cudaMemcpyAsync) of the step's input bytes H2D "
                   "and output bytes D2H, alone and both at once on two streams; best of "
                   f"{reps}, CUDA events"}


def e2e_prefill(fa, pcfg, q, k, v, pflops, scale, stream, world, args, layout=None, ws32=None):
    """The prefill end to end through the public API: every step copies its Q, K, V (and
    layout) from pinned host memory to the device, runs the call and copies O and LSE back.
    Steps are pipelined over two device buffer sets and three streams (copies in, the call,
    copies out), so the copies of one step overlap the call of the previous one; each step
    still moves all of its own bytes inside the timed region."""
    dev = torch.device("cuda", torch.cuda.current_device())
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ins = [hq, hk, hv]
    hlay = layout.pin_memory() if layout is not None else None
    if hlay is not None:
        ins.append(hlay)
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    hl = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
    NB = 2
    bufs = []
    for _ in range(NB):
        bufs.append(dict(q=torch.empty_like(hq, device=dev), k=torch.empty_like(hk, device=dev),
                         v=torch.empty_like(hv, device=dev),
                         o=torch.empty(q.shape, dtype=q.dtype, device=dev),
                         l=torch.empty(q.shape[:3], dtype=torch.float32, device=dev),
                         lay=torch.empty_like(hlay, device=dev) if hlay is not None else None))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(NB)]
    comp_done = [torch.cuda.Event() for _ in range(NB)]
    out_done = [torch.cuda.Event() for _ in range(NB)]
    used = [False] * NB

    def step(i):
        b = bufs[i % NB]
        n = i % NB
        if used[n]:
            s_in.wait_event(comp_done[n])  # the call that read this set's inputs is done
        with torch.cuda.stream(s_in):
            b["q"].copy_(hq, non_blocking=True)
            b["k"].copy_(hk, non_blocking=True)
            b["v"].copy_(hv, non_blocking=True)
            if hlay is not None:
                b["lay"].copy_(hlay, non_blocking=True)
        in_ready[n].record(s_in)
        stream.wait_event(in_ready[n])
        if used[n]:
            stream.wait_event(out_done[n])  # this set's O and LSE have been copied out
        if hlay is not None:
            fa.fa_fwd_ex(b["q"], b["k"], b["v"], b["o"], b["l"], scale, pcfg["mode"],
                         block_layout=b["lay"], block_layout_host=hlay, stream=stream)
        elif ws32 is not None:
            fa.fa_fwd_ex(b["q"], b["k"], b["v"], b["o"], b["l"], scale, pcfg["mode"],
                         pcfg["window"], pcfg["n_global"], workspace=ws32, stream=stream)
        else:
            fa.fa_fwd(b["q"], b["k"], b["v"], b["o"], b["l"], scale, pcfg["mode"], pcfg["window"],
                      pcfg["n_global"], stream=stream)
        comp_done[n].record(stream)
        s_out.wait_event(comp_done[n])
        with torch.cuda.stream(s_out):
            ho.copy_(b["o"], non_blocking=True)
            hl.copy_(b["l"], non_blocking=True)
        out_done[n].record(s_out)
        used[n] = True

    K = max(3, min(args.steps, args.e2e_steps))
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(s_in)
    for i in range(K):
        step(3 + i)
    s_out.wait_event(comp_done[(3 + K - 1) % NB])
    e1.record(s_out)  # after the last copy out, which follows every call and copy in
    torch.cuda.synchronize()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = ho.numel() * ho.element_size() + hl.numel() * 4
    api = ("tiled_attention_06_gb300.fa_fwd_ex (C ABI fa_fwd_ex)" if ws32 is not None
           or layout is not None else "tiled_attention_06_gb300.fa_fwd (C ABI fa_fwd)")
    link = measure_link(h2d, d2h, dev)
    # with copies in, the call and copies out overlapped, a step can be no shorter than
    # the copies of its bytes both ways at once
    step_ms = secs / K * 1e3
    link["step_ms"] = step_ms
    link["frac_of_link"] = link["both_ms"] / step_ms
    return {"value": aggregate(pflops * K, secs, world) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "h2d_gbs_achieved": h2d / (step_ms / 1e3) / 1e9, "link": link,
            "api": api + " with pinned host buffers; steps pipelined over two device buffer "
                         "sets (copies in / call / copies out on three streams)"}


def e2e_decode(fa, di, dbytes, dscale, ws, dk, dv, stream, world, args):
    dev = torch.device("cuda", torch.cuda.current_device())
    hq, hbt, hcl = di.q.pin_memory(), di.block_table.pin_memory(), di.ctx_lens.pin_memory()
    ho = torch.empty(di.q.shape, dtype=di.q.dtype).pin_memory()
    hl = torch.empty(di.q.shape[:2], dtype=torch.float32).pin_memory()
    qd, btd, cld = (torch.empty_like(t, device=dev) for t in (hq, hbt, hcl))
    od = torch.empty_like(qd)
    ld = torch.empty(hl.shape, dtype=torch.float32, device=dev)

    def step():
        qd.copy_(hq, non_blocking=True)
        btd.copy_(hbt, non_blocking=True)
        cld.copy_(hcl, non_blocking=True)
        fa.fa_decode_paged(qd, dk, dv, btd, cld, od, ld, dscale, ws, stream=stream)
        ho.copy_(od, non_blocking=True)
        hl.copy_(ld, non_blocking=True)

    K = max(3, min(args.steps, args.e2e_steps))
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    return {"value": aggregate(dbytes * K, secs, world) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hq, hbt, hcl)),
            "d2h_bytes_per_step": ho.numel() * ho.element_size() + hl.numel() * 4, "steps": K,
            "api": "tiled_attention_06_gb300.fa_decode_paged; the paged KV cache stays resident"}


# --------------------------------------------------------------------------- oracle timing
def oracle_prefill_sample(pcfg, q, k, v, n_heads):
    """Time the FP64 oracle on every row of the first n_heads (batch 0) of the prefill."""
    import numpy as np

    import oracle
    S = pcfg["S"]
    rows = np.arange(n_heads * S, dtype=np.int64)
    t0 = time.perf_counter()
    if pcfg["mode"] == 5:  # the first n_heads (batch, head) pairs: heads 0.. of batch 0, ...
        layout = make_layout(pcfg)
        pairs = layout_pairs(layout, S, S, heads=[bh % pcfg["H"] for bh in range(n_heads)])
        t0 = time.perf_counter()
        oracle.attention_layout(q, k, v, 1 / math.sqrt(pcfg["d"]), layout, rows=rows)
    else:
        pairs = n_heads * visible_pairs(S, S, pcfg["mode"], pcfg["window"], pcfg["n_global"])
        oracle.attention(q, k, v, 1 / math.sqrt(pcfg["d"]), pcfg["mode"], pcfg["window"],
                         pcfg["n_global"], rows=rows)
    secs = time.perf_counter() - t0
    return 4.0 * pairs * pcfg["d"], secs, oracle.threads_used()


def visible_pairs_row(pos, Sk, pcfg):
    return row_visible(pos, Sk, pcfg["mode"], pcfg["window"], pcfg["n_global"])


def oracle_decode_sample(di, n_seq):
    """Time the FP64 oracle on the first n_seq sequences (all heads) of the decode."""
    import numpy as np

    import oracle
    bh = np.arange(n_seq * di.H, dtype=np.int64)
    nbytes = decode_bytes(di.ctx_lens[:n_seq].tolist(), n_seq, di.H, di.d,
                          di.block_table.shape[1])
    t0 = time.perf_counter()
    oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens,
                        1 / math.sqrt(di.d), bh_list=bh)
    return nbytes, time.perf_counter() - t0, oracle.threads_used()


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(pcfg, q, k, v, di):
    out = {"kind": "oracle", "cpu": cpu_model()}
    if pcfg:
        n_heads = pcfg["B"] * pcfg["H"] if pcfg["S"] <= 4096 else 4  # ~10 s on 16 cores
        flops, secs, cores = oracle_prefill_sample(pcfg, q, k, v, n_heads)
        out.update({"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": cores,
                    "seconds": secs,
                    "sample": f"FP64 oracle, all {pcfg['S']} rows of {n_heads} of "
                              f"{pcfg['B'] * pcfg['H']} (batch, head) pairs"})
    if di is not None:
        nbytes, secs, cores = oracle_decode_sample(di, di.B)
        dec = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": cores, "seconds": secs,
               "sample": f"FP64 oracle, all {di.B} sequences, all {di.H} heads"}
        if pcfg:
            out["decode"] = dec
        else:
            out.update(dec)
    return out


# --------------------------------------------------------------------------- next rows
CHUNKED = dict(B=8, H=32, d=128, page=256, pool=600, chunk=512, max_ctx0=7680, dtype="f16")
MULTIMODAL = dict(B=4, H=32, d=128, V=576, T=2048, dtype="bf16")


def timed(calls, K, W, stream, soak_s=CLOCK_SOAK_S):
    """Run each zero-argument call per step; CUDA-event milliseconds of each, summed, and
    the SM clocks sampled during the timed steps."""
    for _ in range(W):
        for c in calls:
            c()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(K)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    soak, t_soak = 0, time.perf_counter()
    while time.perf_counter() - t_soak < soak_s:
        for c in calls:
            c()
        soak += 1
        if soak % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    t_soak = time.perf_counter() - t_soak
    for i in range(K):
        ev[i][0].record(stream)
        for j, c in enumerate(calls):
            c()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    clk["soak"] = {"steps": soak, "seconds": round(t_soak, 3)}
    return [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K))
            for j in range(len(calls))], clk


def run_next_rows(args, fa, workload, peaks, peak_kind, stream, world):
    """chunked: append a 512-token chunk to each of 8 paged sequences (contexts up to
    7.7k, 256-token pages, fp16) and run its causal prefill through the block table, with
    the lengths also given on the host for the work plan (the call without them is timed
    beside it).
    multimodal: LLaVA-shaped vision 576 + text 2048 tokens (B=4, H=32, d=128, bf16) as
    three calls (vision full, text causal, text-to-vision) plus the LSE merge; beside it,
    the text rows as one causal call over [vision; text] keys, and the whole layer as one
    prefix-LM call over [vision; text] with the vision tokens as the prefix."""
    from tiled_attention_06_gb300 import inputs
    dev = torch.device("cuda", torch.cuda.current_device())
    K, W = args.steps, args.warmup
    tc_peak = float(peaks["bf16_tflops"])
    res = {"n_gpus": world, "steps": K, "warmup": W, "scaling": "weak", "vs_baseline": None,
           "higher_is_better": True, "data": "synthetic (seeded N(0,1))"}
    if workload == "chunked":
        c = CHUNKED
        dt = inputs.DTYPES[c["dtype"]]
        g = torch.Generator().manual_seed(0)
        ctx0 = torch.randint(0, c["max_ctx0"] + 1, (c["B"],), generator=g)
        total = (ctx0 + c["chunk"]).tolist()
        npages = [-(-t // c["page"]) for t in total]
        perm = torch.randperm(c["pool"], generator=g)
        table = torch.full((c["B"], max(npages)), -1, dtype=torch.int32)
        off = 0
        for b in range(c["B"]):
            table[b, :npages[b]] = perm[off:off + npages[b]].to(torch.int32)
            off += npages[b]
        B, H, d, T = c["B"], c["H"], c["d"], c["chunk"]
        kp = torch.randn(c["pool"], H, c["page"], d, generator=g).to(dt).to(dev)
        vp = torch.randn(c["pool"], H, c["page"], d, generator=g).to(dt).to(dev)
        kn = torch.randn(B, H, T, d, generator=g).to(dt).to(dev)
        vn = torch.randn(B, H, T, d, generator=g).to(dt).to(dev)
        q = torch.randn(B, H, T, d, generator=g).to(dt).to(dev)
        tab, c0 = table.to(dev), ctx0.to(torch.int32).to(dev)
        ctx = torch.tensor(total, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        scale = 1 / math.sqrt(d)
        # every step appends the same chunk at the same place, then runs its prefill; the
        # lengths are also given on the host, for the work plan
        ctx_host = torch.tensor(total, dtype=torch.int32)
        ms, clk = timed([lambda: fa.fa_kv_append(kn, vn, kp, vp, tab, c0, stream=stream),
                         lambda: fa.fa_fwd_paged(q, kp, vp, tab, ctx, o, lse, scale,
                                                 fa.FA_MASK_CAUSAL, stream=stream,
                                                 ctx_lens_host=ctx_host)], K, W, stream,
                        args.clock_soak)
        unplanned, _ = timed([lambda: fa.fa_fwd_paged(q, kp, vp, tab, ctx, o, lse, scale,
                                                      fa.FA_MASK_CAUSAL, stream=stream)],
                             K, W, stream, 0.0)
        assert fa.fa_get_device_status() == fa.FA_OK
        pairs = sum(visible_pairs(T, t, 1) for t in total)
        flops = 4.0 * H * d * pairs
        app_bytes = 2 * 2 * B * H * T * d * 2  # read k/v chunk, write into pages
        pf = flops * K / (ms[1] / 1e3) / 1e12
        res.update({"metric": "chunked prefill through a paged KV cache TFLOP/s",
                    "value": pf, "unit": "TFLOP/s", "dtype": c["dtype"],
                    "ms_per_step": (ms[0] + ms[1]) / K, "gpu_launches": 2 * K, "clocks": clk,
                    "roofline": {"kernel": "prefill_bm%d_kernel (paged)"
                                           % fa.fa_fwd_default_block_m(fa.FA_MASK_CAUSAL),
                                 "bound": "tensor",
                                 "achieved": pf, "peak": tc_peak, "unit": "TFLOP/s",
                                 "frac": pf / tc_peak, "traffic": None,
                                 "algorithmic_flops": flops},
                    "append": {"value": app_bytes * K / (ms[0] / 1e3) / 1e9, "unit": "GB/s",
                               "ms_per_call": ms[0] / K},
                    "without_host_lengths": {"value": flops * K / (unplanned[0] / 1e3) / 1e12,
                                             "unit": "TFLOP/s",
                                             "api": "fa_fwd_paged (every item weighed by the "
                                                    "pool capacity)"},
                    "api": "fa_fwd_paged_host_lens (lengths also on the host for the plan)",
                    "config": {"workload": f"append {T} tokens + causal chunked prefill, B{B} "
                                           f"H{H} d{d} {c['dtype']}, ctx0~U[0,{c['max_ctx0']}], "
                                           f"page {c['page']}, pool {c['pool']}"}})
    else:
        c = MULTIMODAL
        dt = inputs.DTYPES[c["dtype"]]
        B, H, d, V, T = c["B"], c["H"], c["d"], c["V"], c["T"]
        q, k, v = inputs.prefill_inputs(B, H, V + T, V + T, d, dt, seed=0)
        q, k, v = q.to(dev), k.to(dev), v.to(dev)
        qv, qt = q[:, :, :V].contiguous(), q[:, :, V:].contiguous()
        kv_, kt = k[:, :, :V].contiguous(), k[:, :, V:].contiguous()
        vv, vt = v[:, :, :V].contiguous(), v[:, :, V:].contiguous()
        scale = 1 / math.sqrt(d)
        ov, lv = torch.empty_like(qv), torch.empty(B, H, V, device=dev)
        ott, ltt = torch.empty_like(qt), torch.empty(B, H, T, device=dev)
        otv, ltv = torch.empty_like(qt), torch.empty(B, H, T, device=dev)
        ot, lt = torch.empty_like(qt), torch.empty(B, H, T, device=dev)
        o1, l1 = torch.empty_like(qt), torch.empty(B, H, T, device=dev)
        split = [lambda: fa.fa_fwd(qv, kv_, vv, ov, lv, scale, fa.FA_MASK_NONE, stream=stream),
                 lambda: fa.fa_fwd(qt, kt, vt, ott, ltt, scale, fa.FA_MASK_CAUSAL, stream=stream),
                 lambda: fa.fa_fwd(qt, kv_, vv, otv, ltv, scale, fa.FA_MASK_NONE, stream=stream),
                 lambda: fa.fa_merge_partials(ott, ltt, otv, ltv, ot, lt, stream=stream)]
        ms, clk = timed(split, K, W, stream, args.clock_soak)
        one, _ = timed([lambda: fa.fa_fwd(qt, k, v, o1, l1, scale, fa.FA_MASK_CAUSAL,
                                          stream=stream)], K, W, stream, 0.0)
        oa, la = torch.empty_like(q), torch.empty(B, H, V + T, device=dev)
        plm, _ = timed([lambda: fa.fa_fwd(q, k, v, oa, la, scale, fa.FA_MASK_PREFIX_LM,
                                          n_global=V, stream=stream)], K, W, stream, 0.0)
        assert fa.fa_get_device_status() == fa.FA_OK
        pairs = V * V + T * (T + 1) // 2 + T * V
        flops = 4.0 * B * H * d * pairs
        total_ms = sum(ms)
        val = flops * K / (total_ms / 1e3) / 1e12
        res.update({"metric": "multimodal attention layer TFLOP/s (three-call split + merge)",
                    "value": val, "unit": "TFLOP/s", "dtype": c["dtype"],
                    "ms_per_step": total_ms / K, "gpu_launches": 4 * K, "clocks": clk,
                    "roofline": {"kernel": "prefill_bm256_kernel x3 + merge_kernel",
                                 "bound": "tensor",
                                 "achieved": val, "peak": tc_peak, "unit": "TFLOP/s",
                                 "frac": val / tc_peak, "traffic": None,
                                 "algorithmic_flops": flops},
                    "calls_ms": {"vision": ms[0] / K, "text_causal": ms[1] / K,
                                 "text_to_vision": ms[2] / K, "merge": ms[3] / K},
                    "text_rows_one_call_ms": one[0] / K,
                    "prefix_lm_one_call": {"ms": plm[0] / K,
                                           "value": flops * K / (plm[0] / 1e3) / 1e12,
                                           "unit": "TFLOP/s"},
                    "config": {"workload": f"vision {V} + text {T} tokens, B{B} H{H} d{d} "
                                           f"{c['dtype']}"}})
    return res


def run_backward(args, fa, peaks, stream, world, workload="bwd4k"):
    """Backward of the causal 4k bf16 prefill (B4 H32 S4096 d128), or of the block-sparse 4k
    one (the BigBird-shaped layout of blocksparse4k): fa_bwd after one forward call, timed
    with CUDA events. Work counted: the five products of the backward (S recomputed, dP, dV,
    dK, dQ) over the visible pairs, 2.5x the forward's; each is computed once."""
    from tiled_attention_06_gb300 import inputs
    sparse = workload == "bwd_blocksparse4k"
    cfg = PREFILL["blocksparse4k" if sparse else "causal4k"]
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v = (t.to(dev) for t in make_prefill(cfg, dev))
    dout = inputs.prefill_inputs(cfg["B"], cfg["H"], cfg["S"], cfg["S"], cfg["d"],
                                 inputs.DTYPES[cfg["dtype"]], seed=1)[0].to(dev)
    scale = 1 / math.sqrt(cfg["d"])
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    layout = make_layout(cfg) if sparse else None
    lay_d = layout.to(dev) if sparse else None
    if sparse:
        fa.fa_fwd_ex(q, k, v, o, lse, scale, cfg["mode"], block_layout=lay_d, stream=stream)
    else:
        fa.fa_fwd(q, k, v, o, lse, scale, cfg["mode"], stream=stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(cfg["B"], cfg["H"], cfg["S"]), dtype=torch.uint8,
                     device=dev)
    K, W = args.steps, args.warmup
    ms, clk = timed([lambda: fa.fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, ws, scale, cfg["mode"],
                                       stream=stream, block_layout=lay_d)], K, W, stream,
                    args.clock_soak)
    ms = ms[0]
    assert fa.fa_get_device_status() == fa.FA_OK
    flops = 2.5 * prefill_flops(cfg, layout)
    val = aggregate(flops * K, max_over_ranks(ms / 1e3, world), world) / 1e12
    tc_peak = float(peaks["bf16_tflops"])
    achieved = flops * K / (ms / 1e3) / 1e12
    return {"n_gpus": world, "steps": K, "warmup": W, "scaling": "weak", "vs_baseline": None,
            "higher_is_better": True, "data": "synthetic (seeded N(0,1))",
            "metric": "attention backward TFLOP/s (5 products over visible pairs)",
            "value": val, "unit": "TFLOP/s", "dtype": cfg["dtype"], "ms_per_step": ms / K,
            "gpu_launches": 3 * K, "clocks": clk,
            "roofline": {"kernel": "bwd_dkdv_kernel (+ bwd_prep_kernel, bwd_dq_convert_kernel)",
                         "bound": "tensor", "achieved": achieved, "peak": tc_peak,
                         "unit": "TFLOP/s", "frac": achieved / tc_peak, "traffic": None,
                         "algorithmic_flops": flops},
            "config": {"workload": ("backward of block-sparse (BigBird layout) prefill"
                                    if sparse else "backward of causal prefill")
                                   + " B4 H32 S4096 d128 bf16"}}


# --------------------------------------------------------------------------- reference arm
def reference_rows(S, n_bh, rows_per_bh, seed=0):
    """Seeded query rows for the reference arm: rows_per_bh distinct rows of every one of
    the n_bh (batch, head) pairs, as flat ids bh * S + i, and the rows' positions."""
    g = torch.Generator().manual_seed(seed)
    pos = torch.randperm(S, generator=g)[:min(rows_per_bh, S)].sort().values.numpy()
    flat = (np.arange(n_bh, dtype=np.int64)[:, None] * S + pos[None, :]).reshape(-1)
    return flat, pos


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, on the workload of our arm.

    Each step is a bounded sample of that workload. Prefill: the same seeded 512 query
    rows of every (batch, head) pair (the oracle parallelises over (batch, head) pairs, so
    every core has pairs to work on); decode (when our arm's step has one): every
    sequence with all its heads. Prefill and decode are timed apart, like our arm's."""
    import oracle
    workload = args.workload if args.workload in PREFIX_WORKLOADS else "default"
    pcfg = None if workload == "decode" else PREFILL["causal4k" if workload == "default"
                                                     else workload]
    with_decode = workload in ("default", "decode")
    res = {"impl": "reference", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "scaling": "weak", "vs_baseline": None, "data": "synthetic (seeded N(0,1))",
           "gpu_launches": 0}
    cores = oracle.threads_used()
    if pcfg:
        q, k, v = make_prefill(pcfg, None)
        S, BH = pcfg["S"], pcfg["B"] * pcfg["H"]
        rows, pos = reference_rows(S, BH, 512)
        pflops_step = 4.0 * pcfg["d"] * BH * sum(visible_pairs_row(int(i), S, pcfg) for i in pos)
        psample = (f"FP64 oracle, the same {len(pos)} seeded query rows of each of the {BH} "
                   "(batch, head) pairs per step")

        def pstep():
            oracle.attention(q, k, v, 1 / math.sqrt(pcfg["d"]), pcfg["mode"], pcfg["window"],
                             pcfg["n_global"], rows=rows)
    if with_decode:
        di = make_decode(None)
        dbytes_step = decode_bytes(di.ctx_lens.tolist(), di.B, di.H, di.d,
                                   di.block_table.shape[1])
        dsample = f"FP64 oracle, all {di.B} sequences with all {di.H} heads per step"

        def dstep():
            oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens,
                                1 / math.sqrt(di.d))
    for _ in range(args.warmup):
        if pcfg:
            pstep()
        if with_decode:
            dstep()
    p_s = d_s = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        if pcfg:
            pstep()
        t1 = time.perf_counter()
        if with_decode:
            dstep()
        t2 = time.perf_counter()
        p_s += t1 - t0
        d_s += t2 - t1
    K = args.steps
    if pcfg:
        value = pflops_step * K / p_s / 1e12
        res.update({"metric": "attention fwd TFLOP/s (% BF16 TC peak); paged decode HBM GB/s "
                              "(% of 8 TB/s)",
                    "value": value, "unit": "TFLOP/s", "dtype": pcfg["dtype"]})
        res["cpu_baseline"] = {"kind": "oracle", "value": value, "unit": "TFLOP/s",
                               "cores": cores, "sample": psample, "cpu": cpu_model(),
                               "seconds": p_s}
    if with_decode:
        dval = dbytes_step * K / d_s / 1e9
        dec = {"value": dval, "unit": "GB/s", "cores": cores, "sample": dsample, "seconds": d_s}
        if pcfg:
            res["decode"] = {"value": dval, "unit": "GB/s"}
            res["cpu_baseline"]["decode"] = dec
        else:
            res.update({"metric": "paged decode HBM GB/s (% of 8 TB/s)", "value": dval,
                        "unit": "GB/s", "dtype": "f16"})
            res["cpu_baseline"] = dict(kind="oracle", cpu=cpu_model(), **dec)
    res.update({"higher_is_better": True, "ms_per_step": (p_s + d_s) / K * 1e3,
                "config": workload_config(pcfg, with_decode, 1)})
    res["e2e"] = {"value": res["value"], "unit": res["unit"], "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}
    return res


# --------------------------------------------------------------------------- tile sweep
def run_sweep(args, fa, prefill_call, pflops, peaks, peak_kind, pcfg):
    """Tile-size sweep of the causal 4k prefill: query rows per work item (BLOCK_M 64, 128
    or 256; 64 runs tcgen05 MMAs with M = 64, 256 two 128-row tiles per item) x key-block
    size (BLOCK_N 64 or 128)."""
    lines = []
    for bm in (64, 128, 256):
        for bn in (64, 128):
            for _ in range(3):
                prefill_call(block_n=bn, block_m=bm)
            torch.cuda.synchronize()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = max(5, args.steps // 4)
            s.record()
            for _ in range(n):
                prefill_call(block_n=bn, block_m=bm)
            e.record()
            torch.cuda.synchronize()
            ms = s.elapsed_time(e) / n
            lines.append({"block_m": bm, "block_n": bn, "ms": ms, "tflops": pflops / ms / 1e9,
                          "frac": pflops / ms / 1e9 / float(peaks["bf16_tflops"])})
    return {"metric": "attention fwd TFLOP/s tile sweep", "value": max(l["tflops"] for l in lines),
            "unit": "TFLOP/s", "sweep": lines, "config": workload_config(pcfg, False, 1),
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "ms_per_step": min(l["ms"] for l in lines), "dtype": pcfg["dtype"],
            "gpu_launches": 6 * (3 + max(5, args.steps // 4))}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="default",
                    choices=["default", "causal2k", "causal4k", "causal4k_f32", "noncausal4k",
                             "window32k",
                             "band4k", "prefixlm4k", "blocksparse4k", "chunked", "multimodal",
                             "bwd4k", "bwd_blocksparse4k",
                             "decode", "sweep"])
    ap.add_argument("--batch", type=int, default=None, help="override B (small profiling cases)")
    ap.add_argument("--heads", type=int, default=None, help="override H (small profiling cases)")
    ap.add_argument("--pool", type=int, default=None, help="override the decode page pool size")
    ap.add_argument("--dtype", choices=["f16", "bf16"], default=None,
                    help="override the prefill input dtype")
    ap.add_argument("--block-m", type=int, default=0,
                    help="prefill query rows per work item (128 or 256; 0 = library default)")
    ap.add_argument("--pages-per-split", type=int, default=0,
                    help="decode pages per split-K partial (0 = library default)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--clock-soak", type=float, default=CLOCK_SOAK_S,
                    help="seconds of untimed steps run while the clocks are sampled, just "
                         "before the timed ones (0 = none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-log", default=None,
                    help="file for the raw nvidia-smi clock samples (default: a temporary file)")
    ap.add_argument("--prefill-traffic", type=float, default=None,
                    help="DRAM bytes per prefill launch from an ncu capture of this kernel")
    ap.add_argument("--decode-traffic", type=float, default=None,
                    help="DRAM bytes per decode call from an ncu capture")
    args = ap.parse_args(argv)
    ClockSampler.log_path = args.clock_log
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    for cfg in list(PREFILL.values()) + [DECODE]:
        if args.batch:
            cfg["B"] = args.batch
        if args.heads:
            cfg["H"] = args.heads
        if args.dtype and cfg is not DECODE:
            cfg["dtype"] = args.dtype
    if args.pool:
        DECODE["pool"] = args.pool
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        if rank != 0:
            return 0
        res = run_reference(args, rank, 1)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
        res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
