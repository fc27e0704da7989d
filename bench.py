"""Benchmark of the NVFP4 Attn-QAT hot path on GB300.

One step = one Attn-QAT forward + straight-through backward (all kernels of the
path: the Q/K/V quantization pass, two-pass forward, delta pre-pass, key-outer
dK/dV kernel, query-outer dQ kernel; the backward reads the quantized operands
the forward saved, as api.AttnQAT does) on the Wan2.1-T2V-1.3B self-attention shape
B=1, H=12, N=25088, D=128 (16x28x56 latent tokens), seeded synthetic bf16
inputs resident in HBM.  Counted FLOPs: forward 4*B*H*N^2*D, backward 2.5x that.

The roofline object describes the kernel with the largest share of the step,
timed live inside the timed region with CUDA events that the library records
around each of its launches on the launching stream (nvq_timing_*).

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun, one process per GPU)
are independent replicas of the same step: weak scaling, no data-path
collective; the barrier and the max-over-ranks time use torch.distributed.

--impl reference runs the CPU oracle (float64, the baseline here) on a bounded
slice of the same workload: query rows [0, R) of one head against all keys.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Attn-QAT fwd+bwd TFLOPS and % of GB300 BF16 peak at N=25088,H=12,D=128"
WORKLOAD = ("Wan2.1-1.3B self-attention at 448x896x61 frames: B=1, H=12, N=25088 "
            "(16x28x56 latent tokens), D=128, non-causal, scale 1/sqrt(128); Q,K per-(token,head) "
            "unit-RMS N(0,1), V,dO N(0,1) bf16 (seed 2); NVFP4 fake-quant on Q,K,V,P")
SHAPE = dict(b=1, n=25088, h=12, d=128)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def flops_fwd(b, nq, nkv, h, d):
    return 4.0 * b * h * nq * nkv * d


def kernel_work(kind, b, n, h, d):
    """Algorithmic work of one launch of a kernel kind: (amount, unit, bound).
    Attention kernels count the contractions they execute (the forward's row-max
    pass included); HBM-bound passes count the bytes they must move."""
    gemm = 2.0 * b * h * n * n * d  # one N x N x D contraction per (batch, head)
    rows = b * n * h * d * 2.0      # one bf16 [B, N, H, D] tensor
    table = {
        "attn_fwd": (3 * gemm, "flop", "tensor"),   # S (pass 1), S (pass 2) on FP4 UMMAs, P~ V~
        "bwd_dkdv": (4 * gemm, "flop", "tensor"),   # S, dP, dV, dK
        "bwd_dq": (3 * gemm, "flop", "tensor"),     # S (FP4 UMMAs), dP, dQ
        # q, k, v read once; written as codes + scale blocks + bf16 (q, k) and f16 + bf16 (v)
        "quantize": (rows * (3 + 2 * (0.25 + 1 / 32 + 1) + 2), "byte", "hbm"),
        "bwd_delta": (2 * rows + b * h * n * 4.0, "byte", "hbm"),  # o, dO in, delta out
    }
    return table[kind]


# DRAM traffic per launch of a kernel (dram__bytes_read.sum + dram__bytes_write.sum)
# from one single-pass ncu capture at the Wan 25088 shape
# (profiles/traffic_attn_kernels_wan25088.md), with the SHA-256 of the kernel's
# sources at the time: a changed source reports null.
TRAFFIC = {
    "bwd_dkdv": {"bytes": 417985280, "sources": ['nvfp4_fake_quant_gb300/csrc/attn_bwd.cu', 'nvfp4_fake_quant_gb300/csrc/nvq_ptx.cuh', 'nvfp4_fake_quant_gb300/csrc/nvq_quant.cuh', 'nvfp4_fake_quant_gb300/csrc/nvq_internal.h'],
                "sha256": "ea393c1143a70d924af307f7d64dcf10bebd6ca49bb0143a087dbe387c27d304"},
}


def traffic_for(kind):
    t = TRAFFIC.get(kind)
    if t is None or (SHAPE["n"], SHAPE["h"]) != (25088, 12):
        return None
    import hashlib
    m = hashlib.sha256()
    try:
        for f in t["sources"]:
            with open(os.path.join(ROOT, f), "rb") as fh:
                m.update(fh.read())
    except OSError:
        return None
    return t["bytes"] if m.hexdigest() == t["sha256"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


def dist_setup(n_gpus: int):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        return rank, ws, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x: float, dist, dev) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(ms_local: float, flops_local: float, dist, dev):
    """Whole-job figures of a replica run: the slowest rank's time and the
    total work of all ranks (replicas, no data-path collective).
    Returns (ms, tflops)."""
    ms = max_over_ranks(ms_local, dist, dev)
    flops = flops_local
    if dist is not None:
        import torch
        t = torch.tensor([flops_local], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        flops = float(t.item())
    return ms, flops / (ms * 1e-3) / 1e12


def host_info():
    """The host the oracle runs on: usable cores, CPU model, torch's CPU threads."""
    import platform

    import torch
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"cores": len(os.sched_getaffinity(0)), "cpu_model": model or platform.machine(),
            "torch_threads": torch.get_num_threads(), "arch": platform.machine()}


# The oracle's sample of the headline workload, the same in both arms: query
# rows [0, CPU_ROWS) of head 0 against all 25088 keys, forward + backward.
CPU_ROWS = 4096


def _timed(fn, repeats):
    t0 = time.perf_counter()
    for _ in range(repeats):
        fn()
    return (time.perf_counter() - t0) / repeats


def cpu_baseline(rows: int = CPU_ROWS, head: int = 0, repeats: int = 1):
    """The oracle, as it stands, on query rows [0, rows) of one head (all keys)."""
    from nvfp4_fake_quant_gb300 import workloads
    from oracle import attention as oa
    inp = workloads.wan25088()
    q = inp.q[:, :rows, head:head + 1]
    k = inp.k[:, :, head:head + 1]
    v = inp.v[:, :, head:head + 1]
    do = inp.do[:, :rows, head:head + 1]

    def one():
        o, _, _ = oa.attn_fwd(q, k, v, inp.scale)
        oa.attn_bwd(q, k, v, o, do, inp.scale)
    dt = _timed(one, repeats)
    fl = 3.5 * flops_fwd(1, rows, SHAPE["n"], 1, SHAPE["d"])
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", **host_info(), "kind": "oracle",
            "seconds": dt * repeats, "repeats": repeats,
            "sample": f"query rows 0..{rows - 1} of head {head} (of 12) against all "
                      f"{SHAPE['n']} keys, fwd+bwd in float64; value = counted FLOPs of that "
                      "slice / its time"}


def cpu_quantizer():
    """The oracle's quantizer over the whole 4096x4096 workload (unit and static
    global scale), in GB/s of the same algorithmic bytes as the GPU figure."""
    from nvfp4_fake_quant_gb300 import workloads
    from oracle import nvfp4 as onv
    x = workloads.quant_matrix()
    g = onv.global_sf(x)
    out = {}
    for name, gsf in (("unit_gsf", 1.0), ("static_gsf", g)):
        dt = _timed(lambda: onv.quantizer_outputs(x, gsf), 1)
        out[name] = {"value": x.numel() * 4.0625 / dt / 1e9, "seconds": dt}
    return {**out, "unit": "GB/s", **host_info(), "kind": "oracle",
            "sample": "the whole 4096x4096 matrix, codes + scales + dequantized bf16"}


def cpu_sparse(rows: int = 2048, head: int = 0):
    """The oracle's block selection and block-sparse fwd+bwd on query rows
    [0, rows) (whole cubes) of one head of the block-sparse workload."""
    from nvfp4_fake_quant_gb300 import api, workloads
    from oracle import attention as oa
    from oracle import vsa as ov
    inp = workloads.vsa25088()
    t, hh, w = workloads.VSA_GRID
    b, n, _, _, d = inp.shape
    topk = api.vsa_effective_topk(0.9, n // 128)
    sl = slice(head, head + 1)
    qc, kc, vc, doc = (ov.to_cubes(x[:, :, sl], t, hh, w) for x in (inp.q, inp.k, inp.v, inp.do))

    def one():
        tiles = ov.select_tiles(qc, kc, topk)[:, :, :rows // 128]
        o, _, _ = oa.attn_fwd(qc[:, :rows], kc, vc, inp.scale, kv_tiles=tiles)
        oa.attn_bwd(qc[:, :rows], kc, vc, o, doc[:, :rows], inp.scale, kv_tiles=tiles)
    dt = _timed(one, 1)
    fl = 3.5 * 4.0 * rows * topk * 128 * d
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", **host_info(), "kind": "oracle",
            "seconds": dt,
            "sample": f"head {head}: cube order, selection of all query cubes, fine attention "
                      f"fwd+bwd of query cubes 0..{rows // 128 - 1} (float64); value = counted "
                      "sparse FLOPs of that slice / its time"}


def cpu_hp(rows: int = CPU_ROWS, head: int = 0):
    """The oracle's auxiliary-output forward and the backward with delta from it,
    on the headline sample."""
    from nvfp4_fake_quant_gb300 import workloads
    from oracle import attention as oa
    inp = workloads.wan25088()
    q = inp.q[:, :rows, head:head + 1]
    k, v = inp.k[:, :, head:head + 1], inp.v[:, :, head:head + 1]
    do = inp.do[:, :rows, head:head + 1]

    def one():
        o, _, _ = oa.attn_fwd(q, k, v, inp.scale)
        oa.attn_fwd_hp(q, k, v, inp.scale)
        oa.attn_bwd(q, k, v, o, do, inp.scale, delta_mode="hp")
    dt = _timed(one, 1)
    fl = 3.5 * flops_fwd(1, rows, SHAPE["n"], 1, SHAPE["d"])
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", **host_info(), "kind": "oracle",
            "seconds": dt,
            "sample": f"query rows 0..{rows - 1} of head {head} against all keys: forward, "
                      "auxiliary output and backward with delta from it (float64)"}


def cpu_linear(rows: int = 2048):
    """The oracle's NVFP4 linear forward and backward on rows [0, rows) of x."""
    from nvfp4_fake_quant_gb300 import workloads
    from oracle import linear as ol
    inp = workloads.wan_ffn_up()
    x, g = inp.x[:rows], inp.grad[:rows]

    def one():
        ol.linear_fwd(x, inp.w, inp.bias)
        ol.linear_bwd(g, x, inp.w)
    dt = _timed(one, 1)
    fl = 6.0 * rows * inp.w.shape[0] * inp.w.shape[1]
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", **host_info(), "kind": "oracle",
            "seconds": dt,
            "sample": f"rows 0..{rows - 1} of x: quantized forward (weight quantized whole) and "
                      "the three straight-through gradients (float64); value = 6*rows*N*K / time"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    rows = CPU_ROWS
    vals = []
    for _ in range(args.warmup):
        cpu_baseline(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(rows))
    total = time.perf_counter() - t0
    fl = 3.5 * flops_fwd(1, rows, SHAPE["n"], 1, SHAPE["d"]) * args.steps
    value = fl / total / 1e12
    cb = dict(vals[-1])
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": cb["sample"]},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_events(fn, iters, stream):
    import torch
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(iters):
        fn()
    e.record(stream)
    e.synchronize()
    return s.elapsed_time(e) / iters


def quantizer_bench(peaks, stream, iters=20):
    """nvfp4_fake_quant on the 4096x4096 workload, L2 defeated by rotating
    buffer sets whose total exceeds twice the L2 size.  "us" is the time per
    launch of a CUDA graph holding iters x sets launches back to back (no host
    gaps; events around the graph replay); "wall_us" the back-to-back rate of
    the Python calls, which on a host slower than the kernel includes gaps."""
    import torch

    from nvfp4_fake_quant_gb300 import api, workloads
    x = workloads.quant_matrix().cuda()
    l2 = torch.cuda.get_device_properties(x.device).L2_cache_size
    per_set = x.numel() * 2 * 2 + x.numel() // 16
    nsets = max(4, math.ceil(2 * l2 / per_set) + 1)
    xs = [x.clone() for _ in range(nsets)]
    outs = [torch.empty_like(x) for _ in range(nsets)]
    scs = [torch.empty(x.shape[0], x.shape[1] // 16, dtype=torch.uint8, device=x.device)
           for _ in range(nsets)]
    gsf = api.nvfp4_global_sf(x)
    res = {}
    alg_bytes = x.numel() * 4.0625
    for name, g in (("unit", None), ("static", gsf)):
        state = {"i": 0}

        def one():
            i = state["i"] % nsets
            state["i"] += 1
            api.nvfp4_fake_quant(xs[i], g, out=outs[i], scales=scs[i])
        for _ in range(nsets):
            one()
        torch.cuda.synchronize()
        wall_ms = time_events(one, iters * nsets, stream)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(nsets):
                one()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(iters * nsets):
                one()
        graph.replay()
        torch.cuda.synchronize()
        us = time_events(graph.replay, 3, stream) / (iters * nsets) * 1e3
        gbs = alg_bytes / (us * 1e-6) / 1e9
        res[name] = {"us": us, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"],
                     "wall_us": wall_ms * 1e3, "launches_per_graph": iters * nsets}
    res["algorithmic_bytes"] = alg_bytes
    res["workload"] = ("bf16 4096x4096, N(0,1), 1% entries x50, 2% zero 16-blocks (seed 1); "
                       f"{nsets} rotating buffer sets to defeat L2")
    res["peak_GB/s"] = peaks["hbm_gbs"]
    return res


def sparse_bench(peaks, stream, steps, warmup):
    """The block-sparse workload (Wan latent 16x28x56, B=1, H=12, D=128, 196 cubes
    of 4x4x8 tokens, top-20 key cubes per query cube): one step = raster -> cube
    order of q, k, v, dO, block selection, sparse forward and backward (from the
    operands the forward saved), cube ->
    raster order of o, dq, dk, dv.  Counted FLOPs: forward 4*H*N*(20*128)*D,
    backward 2.5x that."""
    import torch

    from nvfp4_fake_quant_gb300 import api, workloads
    inp = workloads.vsa25088()
    grid = workloads.VSA_GRID
    b, n, _, h, d = inp.shape
    topk = api.vsa_effective_topk(0.9, n // api.VSA_TILE)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    qc, kc, vc, doc = (torch.empty_like(q) for _ in range(4))
    o_c, dq_c, dk_c, dv_c = (torch.empty_like(q) for _ in range(4))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    stats = torch.empty((b, h, 2, n), dtype=torch.float32, device=q.device)
    wsf = torch.empty(api.attn_qat_fwd_workspace(b, n, n, h, d), dtype=torch.uint8, device=q.device)
    wsb = torch.empty(api.attn_qat_bwd_sparse_saved_workspace(b, n, h, d, topk),
                      dtype=torch.uint8, device=q.device)

    def step():
        for src, dst in ((q, qc), (k, kc), (v, vc), (do, doc)):
            api.vsa_reorder(src, grid, out=dst)
        tiles = api.vsa_select_tiles(qc, kc, topk)
        api.attn_qat_fwd_sparse(qc, kc, vc, tiles, inp.scale, o=o_c, stats=stats, workspace=wsf)
        # the backward reads the quantized operands the forward left in wsf
        api.attn_qat_bwd_sparse_saved(wsf, o_c, stats, doc, tiles, inp.scale, dq=dq_c, dk=dk_c,
                                      dv=dv_c, workspace=wsb)
        for src, dst in ((o_c, o), (dq_c, dq), (dk_c, dk), (dv_c, dv)):
            api.vsa_reorder(src, grid, to_cubes=False, out=dst)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    api.timing_enable(True)
    ms_eager = time_events(step, steps, stream)
    kt = api.timing_read()
    api.timing_enable(False)
    if api.device_status() != 0:
        raise RuntimeError("a bounded device wait timed out (block-sparse)")
    # The step's kernels are short (the reorders ~20 us each), so issuing them
    # one call at a time leaves the GPU waiting for the host; a training loop
    # would replay the step as one CUDA graph.  Same calls, same buffers.
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    ms = time_events(graph.replay, steps, stream)
    if api.device_status() != 0:
        raise RuntimeError("a bounded device wait timed out (block-sparse, graph)")
    f_fwd = 4.0 * b * h * n * (topk * api.VSA_TILE) * d
    total = sum(t for _, t in kt.values())
    return {"workload": "Wan latent 16x28x56 (N=25088), B=1, H=12, D=128, q,k,v,dO N(0,1) "
                        "(seed 4); 196 cubes of 4x4x8, top-20 key cubes per query cube",
            "ms_per_step": ms, "launch": "one CUDA graph per step (the calls captured once)",
            "ms_per_step_eager": ms_eager, "TFLOP/s": 3.5 * f_fwd / (ms * 1e-3) / 1e12,
            "flops_counting": "fwd 4*B*H*N*(topk*128)*D + bwd 2.5x fwd",
            "pct_of_bf16_peak": 3.5 * f_fwd / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "kernels": {name: {"launches": c, "avg_ms": t / c, "share": t / total}
                        for name, (c, t) in kt.items() if c}}


def hp_bench(peaks, stream, steps, inp, q, k, v, do, wsf, wsb):
    """The Wan step with the auxiliary high-precision output: forward with O_hp =
    P V~ / l next to O, backward with delta from O_hp.  Same counted FLOPs as the
    headline step (the extra P V~ product is not counted)."""
    import torch

    from nvfp4_fake_quant_gb300 import api
    b, n, h, d = q.shape
    o, o_hp = torch.empty_like(q), torch.empty_like(q)
    stats = torch.empty((b, h, 2, n), dtype=torch.float32, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def fwd():
        api.attn_qat_fwd_hp(q, k, v, inp.scale, False, o=o, o_hp=o_hp, stats=stats, workspace=wsf)

    def step():
        fwd()
        api.attn_qat_bwd_saved(wsf, o_hp, stats, do, inp.scale, False, dq=dq, dk=dk, dv=dv,
                               workspace=wsb)

    step()
    torch.cuda.synchronize()
    api.timing_enable(True)
    ms = time_events(step, steps, stream)
    kt = api.timing_read()
    api.timing_enable(False)
    fwd_ms = time_events(fwd, steps, stream)
    if api.device_status() != 0:
        raise RuntimeError("a bounded device wait timed out (auxiliary output)")
    f_fwd = flops_fwd(b, n, n, h, d)
    total = sum(t for _, t in kt.values())
    return {"ms_per_step": ms, "TFLOP/s": 3.5 * f_fwd / (ms * 1e-3) / 1e12,
            "pct_of_bf16_peak": 3.5 * f_fwd / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "fwd_ms": fwd_ms, "fwd_tflops_executed": 2.0 * f_fwd / (fwd_ms * 1e-3) / 1e12,
            "flops_counting": "as the headline step; executed forward work is S twice and "
                              "two P V~ products (4 * 2*N^2*D per head)",
            "kernels": {name: {"launches": c, "avg_ms": t / c, "share": t / total}
                        for name, (c, t) in kt.items() if c}}


def linear_bench(peaks, stream, steps):
    """The NVFP4 linear on the Wan FFN up-projection (x [25088, 1536], w [8960, 1536],
    bias): forward = the weight's global scale, tiled quantization of x (under its
    calibrated global scale) and w, FP4
    block-scaled GEMM with bias; backward = grad_x, grad_w (BF16 GEMMs) and the bias
    gradient.  The FP4 GEMM is measured against 6x the measured BF16 peak (the
    nominal FP4:BF16 dense ratio 13.5:2.25)."""
    import torch

    from nvfp4_fake_quant_gb300 import api, workloads
    inp = workloads.wan_ffn_up()
    x, w, b, g = (t.cuda() for t in (inp.x, inp.w, inp.bias, inp.grad))
    m, k = x.shape
    n = w.shape[0]
    out = torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    wsf = torch.empty(api._lib.load().nvfp4_linear_workspace(m, n, k), dtype=torch.uint8,
                      device=x.device)
    wsb = torch.empty(api._lib.load().nvfp4_linear_bwd_workspace(m, n, k), dtype=torch.uint8,
                      device=x.device)

    # the input's global scale is a calibrated constant (computed once, as the
    # reference's input_global_sf); the weight's is taken from w at every call
    x_sf = api.nvfp4_global_sf(x)

    def fwd():
        api.nvfp4_linear_fwd(x, w, b, x_global_sf=x_sf, out=out, workspace=wsf)

    def bwd():
        api.nvfp4_linear_bwd(g, x, w, workspace=wsb)

    for _ in range(3):
        fwd()
        bwd()
    torch.cuda.synchronize()
    api.timing_enable(True)
    fwd_ms = time_events(fwd, steps, stream)
    kt_f = api.timing_read()
    api.timing_enable(False)
    api.timing_enable(True)
    bwd_ms = time_events(bwd, steps, stream)
    kt_b = api.timing_read()
    api.timing_enable(False)
    if api.device_status() != 0:
        raise RuntimeError("device error (linear)")
    flops = 2.0 * m * n * k
    fp4_peak = 6.0 * peaks["bf16_tflops"]
    gemm_f = kt_f["linear"][1] / kt_f["linear"][0]
    quant_f = kt_f["quantize"][1] / max(1, kt_f["quantize"][0])
    gemm_b = kt_b["linear"][1] / steps
    return {"workload": "Wan FFN up-projection: x [25088, 1536], w [8960, 1536], bias; "
                        "N(0,1) inputs, w N(0, 1/1536) (seed 6)",
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_tflops": flops / (fwd_ms * 1e-3) / 1e12,
            "bwd_tflops": 2 * flops / (bwd_ms * 1e-3) / 1e12,
            "fp4_gemm_ms": gemm_f, "fp4_gemm_tflops": flops / (gemm_f * 1e-3) / 1e12,
            "fp4_gemm_frac_of_fp4_peak": flops / (gemm_f * 1e-3) / 1e12 / fp4_peak,
            "fp4_peak_tflops": fp4_peak, "fp4_peak_source": "6 x measured bf16 (nominal ratio)",
            "quantize_ms_per_launch": quant_f,
            "bwd_gemm_tflops": 2 * flops / (gemm_b * 1e-3) / 1e12,
            "kernels_fwd": {name: {"launches": c / steps, "avg_ms": t / c}
                            for name, (c, t) in kt_f.items() if c},
            "kernels_bwd": {name: {"launches": c / steps, "avg_ms": t / c}
                            for name, (c, t) in kt_b.items() if c}}


def gpu_local_cpus(dev):
    """The CPUs sysfs lists as local to the GPU's PCI device (its NUMA node), or None."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(dev)
        path = "/sys/bus/pci/devices/%04x:%02x:%02x.0/local_cpulist" % (
            pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        cpus = set()
        with open(path) as f:
            for part in f.read().strip().split(","):
                if "-" in part:
                    a, b_ = part.split("-")
                    cpus.update(range(int(a), int(b_) + 1))
                elif part:
                    cpus.add(int(part))
        allowed = os.sched_getaffinity(0)
        cpus &= allowed
        return cpus if cpus and cpus != allowed else None
    except Exception:
        return None


def pinned_near(dev, make):
    """make() run with this process's threads on the CPUs local to the GPU (when
    sysfs names a proper subset of the allowed CPUs), so that the pinned host
    pages it touches first sit on the GPU's NUMA node; the affinity is restored
    afterwards.  Returns (result, the CPUs used or None)."""
    cpus = gpu_local_cpus(dev)
    if cpus is None:
        return make(), None
    old = os.sched_getaffinity(0)
    try:
        os.sched_setaffinity(0, cpus)
        return make(), sorted(cpus)
    finally:
        os.sched_setaffinity(0, old)


def run_ours(args):
    import torch

    from nvfp4_fake_quant_gb300 import _lib, api, workloads
    rank, ws, local, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _lib.load()
    peaks, peak_src = load_peaks()
    b, n, h, d = SHAPE["b"], SHAPE["n"], SHAPE["h"], SHAPE["d"]
    if (n, h) == (25088, 12):
        inp = workloads.wan25088()
    else:  # profiling cases: same recipe at another size
        inp = workloads.attn_inputs(b, n, n, h, d, seed=2, dist="unit_rms")
    q, k, v, do = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.do))
    stream = torch.cuda.current_stream(dev)
    o = torch.empty_like(q)
    stats = torch.empty((b, h, 2, n), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsf = torch.empty(api.attn_qat_fwd_workspace(b, n, n, h, d), dtype=torch.uint8, device=dev)
    wsb = torch.empty(int(api._lib.load().attn_qat_bwd_saved_workspace(b, n, n, h, d)),
                      dtype=torch.uint8, device=dev)

    def fwd():
        api.attn_qat_fwd(q, k, v, inp.scale, False, o=o, stats=stats, workspace=wsf)

    def bwd():
        # the backward reads the quantized operands the forward left in wsf (the
        # path of api.AttnQAT): no quantizer launch in the backward
        api.attn_qat_bwd_saved(wsf, o, stats, do, inp.scale, False, dq=dq, dk=dk, dv=dv,
                               workspace=wsb)

    def step():
        fwd()
        bwd()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if api.device_status(dev) != 0:
        raise RuntimeError("a bounded device wait timed out during warm-up")

    # ---- timed region: K steps, barrier + synchronize on both sides
    barrier(dist)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    api.timing_enable(True)  # per-launch events on the launching stream, for the roofline
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist)
    ktimes = api.timing_read()
    api.timing_enable(False)
    clocks = clk.summary()
    f_fwd = flops_fwd(b, n, n, h, d)
    f_step = 3.5 * f_fwd
    ms, value = aggregate(ev0.elapsed_time(ev1) / args.steps, f_step, dist, dev)

    # ---- per-call durations (fwd, bwd) on the launching stream
    fwd_ms = time_events(fwd, max(2, args.steps), stream)
    bwd_ms = time_events(bwd, max(2, args.steps), stream)
    bwd_tflops = 2.5 * f_fwd / (bwd_ms * 1e-3) / 1e12
    fwd_tflops = f_fwd / (fwd_ms * 1e-3) / 1e12
    if api.device_status(dev) != 0:
        raise RuntimeError("a bounded device wait timed out")

    # ---- end to end through the public API with pinned host buffers.  Every step
    # copies its q, k, v, dO in from pinned host memory and its dq, dk, dv out to
    # pinned host memory.  The copies run on two copy streams over two device
    # buffer sets: step j+1's inputs arrive and step j's gradients leave while the
    # GPU computes, the way a training loop overlaps its transfers.
    def make_host():
        ins = tuple(t.pin_memory() for t in (inp.q, inp.k, inp.v, inp.do))
        outs = tuple(torch.zeros_like(t).pin_memory() for t in (inp.q, inp.k, inp.v))
        return ins + outs

    (hq, hk, hv, hdo, hdq, hdk, hdv), host_cpus = pinned_near(dev, make_host)
    e2e_sets = []
    if not args.skip_e2e:
        for _ in range(2):
            e2e_sets.append({"q": torch.empty_like(q), "k": torch.empty_like(k),
                             "v": torch.empty_like(v), "do": torch.empty_like(do),
                             "o": torch.empty_like(o), "stats": torch.empty_like(stats),
                             "dq": torch.empty_like(dq), "dk": torch.empty_like(dk),
                             "dv": torch.empty_like(dv)})
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(steps):
        done = [torch.cuda.Event() for _ in range(steps)]
        out = [torch.cuda.Event() for _ in range(steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for j in range(steps):
            st = e2e_sets[j % 2]
            with torch.cuda.stream(s_in):
                if j >= 2:  # the set's inputs are free once step j-2 has been computed
                    s_in.wait_event(done[j - 2])
                for name, src in (("q", hq), ("k", hk), ("v", hv), ("do", hdo)):
                    st[name].copy_(src, non_blocking=True)
                arrived = torch.cuda.Event()
                arrived.record(s_in)
            stream.wait_event(arrived)
            if j >= 2:  # the set's gradients of step j-2 have left
                stream.wait_event(out[j - 2])
            api.attn_qat_fwd(st["q"], st["k"], st["v"], inp.scale, False, o=st["o"],
                             stats=st["stats"], workspace=wsf)
            api.attn_qat_bwd_saved(wsf, st["o"], st["stats"], st["do"], inp.scale, False,
                                   dq=st["dq"], dk=st["dk"], dv=st["dv"], workspace=wsb)
            done[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[j])
                for dst, name in ((hdq, "dq"), (hdk, "dk"), (hdv, "dv")):
                    dst.copy_(st[name], non_blocking=True)
                out[j].record(s_out)
        stream.wait_event(out[steps - 1])
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end) / steps

    e2e_ms = e2e_value = float("nan")
    if not args.skip_e2e:
        e2e_run(2)
        torch.cuda.synchronize(dev)
        barrier(dist)
        e2e_ms, e2e_value = aggregate(e2e_run(args.steps), f_step, dist, dev)
        if not torch.equal(hdq, e2e_sets[(args.steps - 1) % 2]["dq"].cpu()):
            raise RuntimeError("end-to-end run: dq on the host differs from the device's")
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in (hdq, hdk, hdv))

    quant = quantizer_bench(peaks, stream) if rank == 0 and not args.skip_quantizer else None
    sparse = (sparse_bench(peaks, stream, max(3, args.steps), args.warmup)
              if rank == 0 and not args.skip_sparse and (n, h) == (25088, 12) else None)
    hp = (hp_bench(peaks, stream, max(3, args.steps), inp, q, k, v, do, wsf, wsb)
          if rank == 0 and not args.skip_hp else None)
    lin = linear_bench(peaks, stream, max(3, args.steps)) \
        if rank == 0 and not args.skip_linear else None

    peak_t = peaks["bf16_tflops"]
    k_total = sum(ms for _, ms in ktimes.values())
    kernels = {name: {"launches": cnt, "avg_ms": ms / cnt, "share": ms / k_total}
               for name, (cnt, ms) in ktimes.items() if cnt}
    dom = max(kernels, key=lambda name: ktimes[name][1])
    amount, unit, bound = kernel_work(dom, b, n, h, d)
    dom_ms = kernels[dom]["avg_ms"]
    if unit == "flop":
        achieved, peak, r_unit = amount / (dom_ms * 1e-3) / 1e12, peak_t, "TFLOP/s"
        p_name = "bf16_tflops (burst)"
    else:
        achieved, peak, r_unit = amount / (dom_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
        p_name = "hbm_gbs"
    roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak,
                "unit": r_unit, "frac": achieved / peak, "traffic": traffic_for(dom),
                "algorithmic_per_launch": amount, "launch_ms": dom_ms,
                "peak_source": f"{peak_src} {p_name}"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp4+bf16", "data": "synthetic",
        "precision": ("Q~/K~/V~/P~ NVFP4 (E2M1 codes, E4M3 scale per 16, unit global scale); "
                      "S on block-scaled FP4 UMMAs (exact products), P~V~ on F16 UMMAs, backward "
                      "contractions on BF16 UMMAs; fp32 accumulation; bf16 outputs"),
        "config": {"workload": WORKLOAD if (n, h) == (25088, 12) else
                   f"profiling case B=1, H={h}, N={n}, D=128 (Wan recipe, seed 2)",
                   "flops_per_step": f_step,
                   "flops_counting": "fwd 4*B*H*N^2*D + bwd 2.5x fwd",
                   "l2": "inputs larger than L2 (q,k,v,dO 77 MB each + workspaces)",
                   "parallelism": f"replicas x{ws}"},
        "pct_of_bf16_peak": value / ws / peak_t,
        "peaks": {"bf16_tflops": peak_t, "hbm_gbs": peaks["hbm_gbs"], "source": peak_src},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
        "roofline": roofline,
        "kernels": kernels,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "method": "per step: q, k, v, dO copied in from pinned host memory and dq, dk, "
                          "dv copied out to it, on two copy streams over two device buffer "
                          "sets overlapping the neighbouring steps' compute",
                "pinned_first_touch_cpus": (f"{host_cpus[0]}-{host_cpus[-1]} (local to the GPU)"
                                            if host_cpus else "all allowed (sysfs named no "
                                            "narrower GPU-local set)")},
        "gpu_launches": sum(k["launches"] for k in kernels.values()),
        "clocks": clocks,
    }
    cpu = rank == 0 and not args.skip_cpu_baseline
    if quant is not None:
        if cpu:
            quant["cpu_baseline"] = cpu_quantizer()
        line["quantizer"] = quant
    if sparse is not None:
        if cpu:
            sparse["cpu_baseline"] = cpu_sparse()
        line["block_sparse"] = sparse
    if hp is not None:
        if cpu:
            hp["cpu_baseline"] = cpu_hp()
        line["aux_output"] = hp
    if lin is not None:
        if cpu:
            lin["cpu_baseline"] = cpu_linear()
        line["nvfp4_linear"] = lin
    if cpu:
        line["cpu_baseline"] = cpu_baseline(CPU_ROWS, repeats=args.cpu_repeats)
    # compact figures of every report, last on the line (read from its tail)
    summ = {"step_ms": ms, "pct_of_bf16_peak": line["pct_of_bf16_peak"],
            "roofline_frac": roofline["frac"], "e2e_ms": e2e_ms}
    if quant is not None:
        summ["quantizer_frac"] = {m: quant[m]["frac"] for m in ("unit", "static")}
        if "cpu_baseline" in quant:
            summ["quantizer_cpu_GB/s"] = {m: quant["cpu_baseline"][m + "_gsf"]["value"]
                                          for m in ("unit", "static")}
    for key, rep in (("block_sparse", sparse), ("aux_output", hp)):
        if rep is not None:
            summ[key] = {"ms_per_step": rep["ms_per_step"], "TFLOP/s": rep["TFLOP/s"],
                         "pct_of_bf16_peak": rep["pct_of_bf16_peak"]}
            if "cpu_baseline" in rep:
                summ[key]["cpu_TFLOP/s"] = rep["cpu_baseline"]["value"]
    if lin is not None:
        summ["nvfp4_linear"] = {"fwd_ms": lin["fwd_ms"], "bwd_ms": lin["bwd_ms"],
                                "fp4_gemm_tflops": lin["fp4_gemm_tflops"],
                                "bwd_gemm_tflops": lin["bwd_gemm_tflops"]}
        if "cpu_baseline" in lin:
            summ["nvfp4_linear"]["cpu_TFLOP/s"] = lin["cpu_baseline"]["value"]
    if "cpu_baseline" in line:
        summ["cpu_TFLOP/s"] = line["cpu_baseline"]["value"]
        summ["cpu_cores"] = line["cpu_baseline"]["cores"]
    line["summary"] = summ
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-repeats", type=int, default=4,
                    help="repeats of the oracle's sample in the cpu_baseline object")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-quantizer", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-sparse", action="store_true",
                    help="skip the block-sparse (VSA) workload's extra measurement")
    ap.add_argument("--skip-linear", action="store_true",
                    help="skip the NVFP4 linear (Wan FFN up-projection) measurement")
    ap.add_argument("--skip-hp", action="store_true",
                    help="skip the measurement of the step with the auxiliary output")
    ap.add_argument("--quantizer-only", action="store_true",
                    help="time only the standalone quantizer (profiling of that kernel)")
    ap.add_argument("--linear-only", action="store_true",
                    help="time only the NVFP4 linear (profiling of its GEMMs)")
    ap.add_argument("--n", type=int, default=None,
                    help="override N (profiling of smaller cases; not the headline workload)")
    ap.add_argument("--heads", type=int, default=None, help="override H (profiling only)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.n is not None:
        SHAPE["n"] = args.n
    if args.heads is not None:
        SHAPE["h"] = args.heads
    if args.impl == "reference":
        return run_reference(args)
    if args.quantizer_only:
        import torch
        from nvfp4_fake_quant_gb300 import _lib
        _lib.load()
        peaks, _ = load_peaks()
        print(json.dumps({"quantizer": quantizer_bench(peaks, torch.cuda.current_stream(),
                                                       iters=args.steps)}), flush=True)
        return 0
    if args.linear_only:
        import torch
        from nvfp4_fake_quant_gb300 import _lib
        _lib.load()
        peaks, _ = load_peaks()
        print(json.dumps({"nvfp4_linear": linear_bench(peaks, torch.cuda.current_stream(),
                                                       max(3, args.steps))}), flush=True)
        return 0
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
