#!/usr/bin/env python
"""Throughput of the MaskLLM 2:4 mask layer on GB300.

One step = one pass of the whole hot path over the seven linears of a
LLaMA-2-7B block (202,375,168 weights, inputs resident in HBM):
magnitude prior -> forward (W', row sum of squares) -> backward (dlogits)
-> hard mask + 2:4 compression, each kernel over all seven matrices.

Prints one JSON line (rank 0).  `value` is whole-job weights per second
(all ranks); `e2e` is the same step through the C ABI with the inputs copied
from pinned host memory and every output copied back inside the timed region;
`roofline` is the dominant kernel's algorithmic bytes per launch over its
CUDA-event launch time against the measured HBM copy bandwidth;
`cpu_baseline` times the CPU oracle on a bounded sample of the same workload.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl gpu|reference]
For N > 1 launch one process per GPU with torch.distributed.run; each rank
processes its own block (a different layer's tensors: weak scaling, no
collective on the data path).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# Algorithmic bytes per weight of each kernel (what the method must move).
BYTES_PER_WEIGHT = {"prior": 8.0, "forward": 10.0, "backward": 16.0, "hard_compress": 9.125}
KERNELS = ("prior", "forward", "backward", "hard_compress")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal (context beside the measured peak)
METRIC = "weights/s (prior + forward + backward + hard-compress step)"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gpu", "reference"), default="gpu")
    ap.add_argument("--workload", default="llama2_7b_block")
    ap.add_argument("--e2e-steps", type=int, default=16)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other weight sets (full LLaMA-2-7B, Nemotron-4-15B layers, "
                         "near-one-hot compress)")
    ap.add_argument("--spmm-tile-n", type=int, default=0,
                    help="force the sparse product's tile width (128..256, a multiple of 32) "
                         "for the spmm extra; 0 = the width the library picks per call")
    ap.add_argument("--only", default=None,
                    help="comma-separated matrix names of the workload to run (e.g. 'down'); "
                         "for small profiling runs")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------

class Ranks:
    def __init__(self, backend_gpu: bool):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            backend = "nccl" if backend_gpu else "gloo"
            if backend_gpu:
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        return reduce_max(self.pg, x)

    def sum(self, x: float) -> float:
        return reduce_sum(self.pg, x)

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def _reduce(pg, x: float, op_name: str) -> float:
    if pg is None:
        return x
    import torch
    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=getattr(pg.ReduceOp, op_name))
    return float(t.item())


def reduce_max(pg, x: float) -> float:
    """Max of a per-rank value (the job's time is its slowest rank's)."""
    return _reduce(pg, x, "MAX")


def reduce_sum(pg, x: float) -> float:
    return _reduce(pg, x, "SUM")


def job_value(weights_per_rank: int, world: int, max_seconds: float, steps: int) -> float:
    """Whole-job throughput: the weights all ranks processed over the slowest rank's time."""
    return weights_per_rank * world * steps / max_seconds


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def traffic_table():
    """Per-launch DRAM bytes from the committed ncu summary, keyed by kernel
    and matrix shape, valid only for the kernel source it was taken on."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    try:
        with open(path) as f:
            for line in f:
                p = line.split()
                if len(p) == 5 and p[0] == "traffic":
                    out[(p[1], p[2])] = (float(p[3]), p[4])
    except OSError:
        pass
    return out


# the sources compiled into the timed stream kernels; a stored traffic
# figure is valid only for the digest it was taken with
STREAM_SOURCES = ("device_common.cuh", "kernels_stream.cu", "pipeline.cuh")


def _code_only(text: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed
    (string literals in these sources hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_digest() -> str:
    """Digest of the code compiled into the stream kernels (comments and
    whitespace excluded: they change no instruction)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "semi_structured_sparsity_gb300", "csrc")
    for fn in STREAM_SOURCES:
        with open(os.path.join(csrc, fn)) as f:
            h.update(fn.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:12]


# ---------------------------------------------------------------------------
# the step
# ---------------------------------------------------------------------------

class Block:
    """Resident inputs and outputs of one block of matrices on one GPU, with
    the C-ABI matrix descriptors built once."""

    def __init__(self, wl, layer, device, only=None):
        import torch

        from semi_structured_sparsity_gb300 import binding as mk
        from semi_structured_sparsity_gb300 import workloads as W
        self.mk, self.wl, self.dev = mk, wl, device
        self.mats = []
        for m in range(len(wl.matrices)):
            if only and wl.matrices[m][0] not in only:
                continue
            x = W.matrix_inputs(wl, layer, m, device=device)
            if x.L is None:   # logits = magnitude prior + noise
                x.L = mk.maskllm_prior_init(x.W, wl.prior_scale) + x.L_noise
                x.L_noise = None
            r, c = x.rows, x.cols
            self.mats.append({
                "x": x, "W": x.W, "logits": x.L, "grad_W_out": x.G, "tensor_id": x.tensor_id,
                "logits_out": torch.empty((r, c // 4, 6), dtype=torch.float32, device=device),
                "W_out": torch.empty((r, c), dtype=torch.bfloat16, device=device),
                "row_sq_out": torch.empty((r,), dtype=torch.float32, device=device),
                "dlogits_out": torch.empty((r, c // 4, 6), dtype=torch.float32, device=device),
                "values_out": torch.empty((r, c // 2), dtype=torch.bfloat16, device=device),
                "meta_out": torch.empty((r, c // 32), dtype=torch.int32, device=device),
            })
        torch.cuda.synchronize(device)
        self.arr = mk.matrix_array(self.mats)
        self.n = len(self.mats)
        self.weights = sum(m["x"].rows * m["x"].cols for m in self.mats)
        self.launches_per_call = (self.n + mk.MAX_BATCH - 1) // mk.MAX_BATCH
        self.launches = 0

    def outputs(self, m):
        return (m["logits_out"], m["W_out"], m["row_sq_out"], m["dlogits_out"], m["values_out"],
                m["meta_out"])

    def run(self, step: int, events=None):
        """One step: each kernel once over all matrices (batched launch);
        events[k] = (start, end) CUDA events bracketing kernel k (optional)."""
        import torch
        mk, wl, L = self.mk, self.wl, self.mk.lib()
        s = torch.cuda.current_stream(self.dev).cuda_stream
        for k in KERNELS:
            if events is not None:
                events[k][0].record()
            if k == "prior":
                st = L.maskllm_prior_init_batched(self.arr, self.n, wl.prior_scale or 1.0, s)
            elif k == "forward":
                st = L.maskllm_forward_batched(self.arr, self.n, wl.tau, wl.kappa, 0, step, s)
            elif k == "backward":
                st = L.maskllm_backward_batched(self.arr, self.n, wl.tau, wl.kappa, 0, step,
                                                0.0, s)
            else:
                st = L.maskllm_hard_compress_batched(self.arr, self.n, s)
            if st != 0:
                raise mk.MaskLLMError("maskllm_%s_batched" % k, st)
            self.launches += self.launches_per_call
            if events is not None:
                events[k][1].record()


def run_gpu(args):
    import torch

    from semi_structured_sparsity_gb300 import _build
    from semi_structured_sparsity_gb300 import workloads as W
    _build.build()
    ranks = Ranks(backend_gpu=True)
    dev = torch.device("cuda", ranks.local)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    only = set(args.only.split(",")) if args.only else None
    blk = Block(wl, layer=ranks.rank % max(wl.layers, 1), device=dev, only=only)
    stream = torch.cuda.current_stream(dev)

    for s in range(args.warmup):
        blk.run(s)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    ev = {k: [] for k in KERNELS}
    ranks.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = blk.launches
    t0.record(stream)
    for s in range(args.steps):
        e = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for k in KERNELS}
        blk.run(args.warmup + s, events=e)
        for k in KERNELS:
            ev[k].append(e[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ranks.barrier()
    clk = clocks.stop()
    launches = blk.launches - launches0
    sec = t0.elapsed_time(t1) / 1e3
    sec_max = ranks.max(sec)
    per_kernel_s = {k: sum(a.elapsed_time(b) for a, b in ev[k]) / 1e3 / args.steps
                    for k in KERNELS}
    value = job_value(blk.weights, ranks.world, sec_max, args.steps)

    peak, peak_kind = hbm_peak()
    kernels = {}
    for k in KERNELS:
        gbs = BYTES_PER_WEIGHT[k] * blk.weights / per_kernel_s[k] / 1e9
        kernels[k] = {"us_per_step": round(per_kernel_s[k] * 1e6, 2),
                      "weights_per_s": blk.weights / per_kernel_s[k],
                      "GB_per_s": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4),
                      "frac_of_nominal_hbm": round(gbs / NOMINAL_HBM_GBS, 4)}
    dominant = max(KERNELS, key=lambda k: per_kernel_s[k])
    # the dominant kernel's algorithmic bytes over its CUDA-event time (one
    # batched launch per step covers the whole block)
    ach = BYTES_PER_WEIGHT[dominant] * blk.weights / per_kernel_s[dominant] / 1e9
    # ncu DRAM bytes per launch (read + write) of each kernel, valid only for
    # the kernel source they were captured on
    tt = traffic_table()
    digest = kernel_source_digest()
    shape_key = "%s" % args.workload
    for k in KERNELS:
        hit = tt.get((k, shape_key))
        kernels[k]["traffic"] = hit[0] if hit is not None and hit[1] == digest else None
        kernels[k]["algorithmic_bytes"] = BYTES_PER_WEIGHT[k] * blk.weights
    traffic = kernels[dominant]["traffic"]

    extras = run_extras(blk, peak, dev, spmm_tile_n=args.spmm_tile_n)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, blk, ranks, dev, only=only)

    if not args.no_configs and ranks.world == 1 and not args.only:
        extras["configs"] = run_configs(dev, peak)

    cpu = None
    if not args.no_cpu_baseline and ranks.rank == 0 and ranks.world == 1:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "weights/s",
        "n_gpus": ranks.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec_max / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 weights, fp32 logits",
        "data": "synthetic (seeded; LLaMA-2-7B block shapes, W~N(0,0.02), logits = magnitude "
                "prior(300) + N(0,0.1), G~N(0,1e-3))",
        "config": {"workload": args.workload + ("[%s]" % args.only if args.only else ""),
                   "weights_per_gpu": blk.weights,
                   "matrices": [[m["x"].rows, m["x"].cols] for m in blk.mats], "tau": wl.tau,
                   "kappa": wl.kappa, "parallelism": "dp%d (independent blocks)" % ranks.world,
                   "l2": "inputs larger than L2 (per-kernel sweep reads >= 1.6 GB)"},
        "kernels": kernels,
        "roofline": {"kernel": dominant, "bound": "hbm", "achieved": round(ach, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(ach / peak, 4), "traffic": traffic,
                     "bytes_per_weight": BYTES_PER_WEIGHT[dominant],
                     "bytes_per_launch": BYTES_PER_WEIGHT[dominant] * blk.weights
                     / blk.launches_per_call,
                     "launches_per_step": blk.launches_per_call},
        "extras": extras,
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)
    ranks.close()


def run_extras(blk, peak, dev, reps=20, spmm_tile_n=0):
    """The entry points beyond the step, on the same resident block: logits
    from a given mask (6.125 B/weight: codes in, logits out; one batched
    launch), the convergence
    diagnostics (6.5 B/weight: logits and previous draws in, draws out) and
    the forward with the diagnostics in the same pass (10.5 B/weight) and
    the backward with them (16.5 B/weight), each over all matrices in one
    batched launch, CUDA-event timed."""
    import torch
    mk, wl = blk.mk, blk.wl
    L = mk.lib()
    s = torch.cuda.current_stream(dev).cuda_stream
    draws = [torch.zeros((m["x"].rows, m["x"].cols // 4), dtype=torch.uint8, device=dev)
             for m in blk.mats]
    nxt = [torch.empty_like(d) for d in draws]
    l1 = [torch.empty((m["x"].rows,), dtype=torch.int32, device=dev) for m in blk.mats]
    mp = [torch.empty((m["x"].rows,), dtype=torch.float32, device=dev) for m in blk.mats]

    # logits from the step's compressed masks: one batched launch per block
    pfm_arr = mk.matrix_array([{"meta": m["meta_out"], "logits_out": m["logits_out"]}
                               for m in blk.mats])

    def prior_from_mask():
        st = L.maskllm_prior_from_mask_batched(pfm_arr, len(blk.mats), 1.0, 0.0, s)
        assert st == 0

    # the diagnostics over the block: one batched launch per call
    ms_arr = mk.matrix_array([{"W": None, "logits": m["logits"], "tensor_id": m["tensor_id"],
                               "prev_idx": draws[i], "idx_out": nxt[i], "l1_row_out": l1[i],
                               "maxprob_row_out": mp[i]} for i, m in enumerate(blk.mats)])

    def mask_stats(step):
        st = L.maskllm_mask_stats_batched(ms_arr, len(blk.mats), wl.tau, wl.kappa, 0, step, s)
        assert st == 0

    w_out = [torch.empty_like(m["x"].W) for m in blk.mats]
    row_sq = [torch.empty((m["x"].rows,), dtype=torch.float32, device=dev) for m in blk.mats]
    fs_arr = mk.matrix_array([{"W": m["W"], "logits": m["logits"], "tensor_id": m["tensor_id"],
                               "prev_idx": draws[i], "W_out": w_out[i], "row_sq_out": row_sq[i],
                               "idx_out": nxt[i], "l1_row_out": l1[i], "maxprob_row_out": mp[i]}
                              for i, m in enumerate(blk.mats)])

    def forward_stats(step):
        st = L.maskllm_forward_stats_batched(fs_arr, len(blk.mats), wl.tau, wl.kappa, 0, step, s)
        assert st == 0

    # the backward with the diagnostics (dlogits into the step's own buffers)
    bs_arr = mk.matrix_array([{"W": m["W"], "logits": m["logits"], "grad_W_out": m["grad_W_out"],
                               "tensor_id": m["tensor_id"], "prev_idx": draws[i],
                               "dlogits_out": m["dlogits_out"], "idx_out": nxt[i],
                               "l1_row_out": l1[i], "maxprob_row_out": mp[i]}
                              for i, m in enumerate(blk.mats)])

    def backward_stats(step):
        st = L.maskllm_backward_stats_batched(bs_arr, len(blk.mats), wl.tau, wl.kappa, 0, step,
                                              0.0, s)
        assert st == 0

    out = {}
    for name, fn, bpw in (("prior_from_mask", lambda i: prior_from_mask(), 6.125),
                          ("mask_stats", mask_stats, 6.5),
                          ("forward_stats", forward_stats, 10.5),
                          ("backward_stats", backward_stats, 16.5)):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(reps):
            fn(i)
        b.record()
        torch.cuda.synchronize(dev)
        sec = a.elapsed_time(b) / 1e3 / reps
        gbs = bpw * blk.weights / sec / 1e9
        out[name] = {"us_per_block": round(sec * 1e6, 2), "GB_per_s": round(gbs, 1),
                     "frac_of_hbm": round(gbs / peak, 4), "bytes_per_weight": bpw,
                     "launches_per_block": -(-len(blk.mats) // mk.MAX_BATCH)}
    out["perm_search"] = run_perm_search(blk, dev)
    blk.mk.maskllm_test_spmm_tile_n(spmm_tile_n)
    try:
        out["spmm"] = run_spmm(blk, dev)
    finally:
        blk.mk.maskllm_test_spmm_tile_n(0)
    out["spmm"]["tile_n"] = spmm_tile_n if spmm_tile_n else "chosen per call"
    return out


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def run_spmm(blk, dev, n_tokens=4096, reps=20):
    """2:4 sparse x dense product: the block's q projection as the hard mask
    compressed it in the step, times n_tokens seeded bf16 activation rows
    (C = A B^T, fp32 out), CUDA-event timed (median of reps).  Reported as
    dense-equivalent TFLOP/s (2 M N K / t) against the sparse tensor peak,
    twice the measured dense bf16 peak (the 2x math rate of the sparse tensor
    cores); cuBLAS's dense product of the same (decompressed) matrix and, when
    torch has it, cuSPARSELt's sparse product are timed beside it."""
    import torch
    from semi_structured_sparsity_gb300 import workloads as WL
    mk = blk.mk
    q = blk.mats[0]
    vals, meta = q["values_out"], q["meta_out"]
    M, half = vals.shape
    K = 2 * half
    Bt = WL.normal_bf16(n_tokens, K, 1.0, 4242, device=dev)
    C = torch.empty((M, n_tokens), dtype=torch.float32, device=dev)

    def med(fn):
        # back-to-back launches (operands stay in L2, as in any GEMM
        # benchmark): median over 5 runs of the mean of `reps` launches
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(5):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) / 1e3 / reps)
        return statistics.median(ts)

    flops = 2.0 * M * n_tokens * K
    t = med(lambda: mk.maskllm_spmm(vals, meta, Bt, C=C))
    peak, kind = bf16_peak()
    out = {"M": M, "K": K, "N": n_tokens, "us": round(t * 1e6, 2),
           "dense_equiv_tflops": round(flops / t / 1e12, 1),
           "roofline": {"bound": "tensor", "peak": round(2 * peak, 1), "peak_kind":
                        kind + " (2 x dense bf16)", "frac": round(flops / t / 1e12 / (2 * peak), 4)}}
    Wd = mk.maskllm_decompress(vals, meta, M, K)
    td = med(lambda: torch.matmul(Wd, Bt.t()))
    out["cublas_dense_us"] = round(td * 1e6, 2)
    try:
        comp = torch._cslt_compress(Wd)
        tc = med(lambda: torch._cslt_sparse_mm(comp, Bt.t()))
        out["cusparselt_us"] = round(tc * 1e6, 2)
    except Exception as e:   # torch built without cuSPARSELt
        out["cusparselt_us"] = None
        out["cusparselt_note"] = type(e).__name__
    return out


def run_perm_search(blk, dev, steps=256, reps=3):
    """Channel-permutation search on the block's first matrix (the q
    projection): the call with 0 steps (set-up and the [cols, cols] swap-gain
    table, an integer max-plus product over the rows: cols^2 * rows
    max-and-add evaluations), and with `steps` steps, CUDA-event timed on the
    launching stream (best of `reps`)."""
    import torch
    mk = blk.mk
    L = mk.lib()
    s = torch.cuda.current_stream(dev).cuda_stream
    Wq = blk.mats[0]["x"].W
    rows, cols = Wq.shape
    ws = torch.empty((mk.maskllm_perm_workspace_bytes(rows, cols),), dtype=torch.uint8,
                     device=dev)
    ident = torch.arange(cols, dtype=torch.int32, device=dev)
    perm = ident.clone()
    swaps = torch.zeros((steps, 2), dtype=torch.int32, device=dev)
    gains = torch.zeros((steps,), dtype=torch.int64, device=dev)
    small = torch.zeros((8,), dtype=torch.int32, device=dev)

    def timed(n):
        best = None
        for _ in range(reps):
            perm.copy_(ident)
            torch.cuda.synchronize(dev)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            st = L.maskllm_perm_search(Wq.data_ptr(), rows, cols, perm.data_ptr(), n,
                                       ws.data_ptr(), ws.numel(), swaps.data_ptr(),
                                       gains.data_ptr(), small.data_ptr(),
                                       small.data_ptr() + 16, s)
            b.record()
            torch.cuda.synchronize(dev)
            assert st == 0
            t = a.elapsed_time(b) / 1e3
            best = t if best is None else min(best, t)
        return best

    timed(0)
    t0 = timed(0)
    tn = timed(steps)
    n = int(small[0].item())
    shift = int(small[4].item())
    shift_t = torch.tensor([shift, 0, 0, 0], dtype=torch.int32, device=dev)
    m_start = int(mk.maskllm_perm_metric(Wq, ident, shift_t).item())
    m_end = int(mk.maskllm_perm_metric(Wq, perm, shift_t).item())
    evals = float(cols) * cols * rows
    return {"matrix": [rows, cols], "table_build_us": round(t0 * 1e6, 1),
            "table_evals_per_s": round(evals / t0, 1),
            "steps": n, "us_per_step": round((tn - t0) / max(n, 1) * 1e6, 2),
            "kept_magnitude_gain": round((m_end - m_start) / max(m_start, 1), 6),
            "note": "evals = cols^2 * rows max-and-add; table_build includes the scan and "
                    "set-up kernels"}


def _config_block(wl, layer, dev, outputs):
    """Resident inputs and the requested outputs of one layer of workload wl
    (logits built as the step builds them); matrix descriptors for the
    batched calls."""
    import torch

    from semi_structured_sparsity_gb300 import binding as mk
    from semi_structured_sparsity_gb300 import workloads as W
    mats = []
    for m in range(len(wl.matrices)):
        x = W.matrix_inputs(wl, layer, m, device=dev, with_grad="backward" in outputs)
        if x.L is None:
            x.L = mk.maskllm_prior_init(x.W, wl.prior_scale) + x.L_noise
            x.L_noise = None
        r, c = x.rows, x.cols
        d = {"W": x.W, "logits": x.L, "grad_W_out": x.G, "tensor_id": x.tensor_id}
        if "forward" in outputs:
            d["W_out"] = torch.empty_like(x.W)
            d["row_sq_out"] = torch.empty((r,), dtype=torch.float32, device=dev)
        if "backward" in outputs:
            d["dlogits_out"] = torch.empty_like(x.L)
        if "hard_compress" in outputs:
            d["values_out"] = torch.empty((r, c // 2), dtype=torch.bfloat16, device=dev)
            d["meta_out"] = torch.empty((r, c // 32), dtype=torch.int32, device=dev)
        mats.append(d)
    return mats


def _timed_calls(fn, dev, reps):
    """Mean seconds of one fn() over `reps` back-to-back calls (after one
    untimed call), CUDA events on the current stream."""
    import torch
    fn()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / 1e3 / reps


def _kernel_line(weights, seconds, op, peak, launches):
    gbs = BYTES_PER_WEIGHT[op] * weights / seconds / 1e9
    return {"us": round(seconds * 1e6, 1), "weights_per_s": weights / seconds,
            "GB_per_s": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4),
            "launches": launches}


def run_configs(dev, peak, reps=5):
    """The other weight sets of the mask layer, CUDA-event timed on this GPU
    (each config's buffers are freed before the next):
      * llama2_7b_full: one forward and one backward mask step over all 32
        layers x 7 matrices (6,476,005,376 weights) with every layer's logits
        and dlogits resident (tau 0.5), as batched calls of 16 matrices;
      * nemotron4_15b: forward and backward of each of the 32 layers (6
        matrices, 390,070,272 weights per layer), layer by layer, each
        layer's inputs generated, timed and freed in turn (tau 0.2, kappa 500);
      * compress_7b: hard mask + 2:4 compression of the LLaMA-2-7B block
        with near-one-hot logits and 1% exact ties."""
    import torch

    from semi_structured_sparsity_gb300 import binding as mk
    from semi_structured_sparsity_gb300 import workloads as W
    L = mk.lib()
    s = torch.cuda.current_stream(dev).cuda_stream
    out = {}

    def batched(op, wl, arr, n):
        if op == "forward":
            st = L.maskllm_forward_batched(arr, n, wl.tau, wl.kappa, 0, 0, s)
        elif op == "backward":
            st = L.maskllm_backward_batched(arr, n, wl.tau, wl.kappa, 0, 0, 0.0, s)
        else:
            st = L.maskllm_hard_compress_batched(arr, n, s)
        if st != 0:
            raise mk.MaskLLMError("maskllm_%s_batched" % op, st)

    # config 3: the full model, all layers resident
    wl = W.WORKLOADS["llama2_7b_full"]
    mats = [d for layer in range(wl.layers)
            for d in _config_block(wl, layer, dev, ("forward", "backward"))]
    torch.cuda.synchronize(dev)
    arr = mk.matrix_array(mats)
    weights = sum(d["W"].numel() for d in mats)
    launches = (len(mats) + mk.MAX_BATCH - 1) // mk.MAX_BATCH
    k3 = {op: _kernel_line(weights, _timed_calls(lambda: batched(op, wl, arr, len(mats)), dev,
                                                 reps), op, peak, launches)
          for op in ("forward", "backward")}
    step = sum(v["us"] for v in k3.values()) / 1e6
    out["llama2_7b_full"] = {"weights": weights, "matrices": len(mats), "tau": wl.tau,
                             "kappa": wl.kappa, "kernels": k3,
                             "step_ms": round(step * 1e3, 3), "weights_per_s": weights / step,
                             "resident_GB": round(sum(t.numel() * t.element_size()
                                                      for d in mats for t in d.values()
                                                      if torch.is_tensor(t)) / 1e9, 1)}
    del mats, arr
    torch.cuda.empty_cache()

    # config 4: Nemotron-4-15B shapes, 32 layers one at a time
    wl = W.WORKLOADS["nemotron4_15b"]
    tot = {"forward": 0.0, "backward": 0.0}
    weights = 0
    launches = 0
    for layer in range(wl.layers):
        mats = _config_block(wl, layer, dev, ("forward", "backward"))
        torch.cuda.synchronize(dev)
        arr = mk.matrix_array(mats)
        for op in tot:
            tot[op] += _timed_calls(lambda: batched(op, wl, arr, len(mats)), dev, 2)
        weights += sum(d["W"].numel() for d in mats)
        launches += 1
        del mats, arr
    torch.cuda.empty_cache()
    k4 = {op: _kernel_line(weights, sec, op, peak, launches) for op, sec in tot.items()}
    step = sum(tot.values())
    out["nemotron4_15b"] = {"weights": weights, "layers": wl.layers, "tau": wl.tau,
                            "kappa": wl.kappa, "kernels": k4,
                            "step_ms": round(step * 1e3, 3), "weights_per_s": weights / step,
                            "note": "per-kernel time summed over the 32 layers (one batched "
                                    "launch per layer and kernel)"}

    # config 5: hard mask + compression of near-one-hot logits with ties
    wl = W.WORKLOADS["compress_7b"]
    mats = _config_block(wl, 0, dev, ("hard_compress",))
    torch.cuda.synchronize(dev)
    arr = mk.matrix_array(mats)
    weights = sum(d["W"].numel() for d in mats)
    sec = _timed_calls(lambda: batched("hard_compress", wl, arr, len(mats)), dev, 20)
    out["compress_7b"] = {"weights": weights, "kernels": {
        "hard_compress": _kernel_line(weights, sec, "hard_compress", peak, 1)}}
    del mats, arr
    torch.cuda.empty_cache()
    return out


def run_e2e(args, blk, ranks, dev, only=None):
    """The same step through the C ABI with host buffers: every step copies
    W, logits and G from pinned host memory, runs the four kernels, and copies
    every output back to pinned host memory.  Steps are pipelined the way a
    caller streaming many steps would: two sets of device buffers, the inputs
    of step s + 1 copied in (one stream) while step s computes (a second) and
    the outputs of step s - 1 are copied out (a third), ordered by events.
    Every step's copies are inside the timed region."""
    import torch
    sets = [blk, Block(blk.wl, layer=ranks.rank % max(blk.wl.layers, 1), device=dev, only=only)]
    host_in, host_out = [], []
    for m in blk.mats:
        x = m["x"]
        host_in.append([t.cpu().pin_memory() for t in (x.W, x.L, x.G)])
        host_out.append([torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                         for t in blk.outputs(m)])
    h2d = sum(t.numel() * t.element_size() for h in host_in for t in h)
    d2h = sum(t.numel() * t.element_size() for h in host_out for t in h)
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
    # per step: (start, end) events around its H2D copies and its D2H copies,
    # recorded after the waits, so each pair spans the copies alone
    copy_ev = {"h2d": [], "d2h": []}

    def timing_pair():
        return (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))

    def one(step, timed=False):
        x_i = step % 2
        b = sets[x_i]
        with torch.cuda.stream(s_in):
            if step >= 2:
                s_in.wait_event(ev["comp"][x_i])      # step - 2 has read these inputs
            if timed:
                copy_ev["h2d"].append(timing_pair())
                copy_ev["h2d"][-1][0].record(s_in)
            for m, hin in zip(b.mats, host_in):
                x = m["x"]
                for dst, src in zip((x.W, x.L, x.G), hin):
                    dst.copy_(src, non_blocking=True)
            if timed:
                copy_ev["h2d"][-1][1].record(s_in)
            ev["in"][x_i].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev["in"][x_i])
            if step >= 2:
                s_comp.wait_event(ev["out"][x_i])     # step - 2's outputs are out
            b.run(step)
            ev["comp"][x_i].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][x_i])
            if timed:
                copy_ev["d2h"].append(timing_pair())
                copy_ev["d2h"][-1][0].record(s_out)
            for m, hout in zip(b.mats, host_out):
                for dst, src in zip(hout, b.outputs(m)):
                    dst.copy_(src, non_blocking=True)
            if timed:
                copy_ev["d2h"][-1][1].record(s_out)
            ev["out"][x_i].record(s_out)

    for w in range(2):
        one(w)
    torch.cuda.synchronize(dev)
    ranks.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    s_comp.wait_event(t0)
    s_out.wait_event(t0)
    for st in range(args.e2e_steps):
        one(st + 2, timed=True)
    t1.record(s_out)
    torch.cuda.synchronize(dev)
    ranks.barrier()
    sec = ranks.max(t0.elapsed_time(t1) / 1e3)
    # achieved host-link rates of the timed steps: bytes over the summed
    # durations of each step's copies (the copies of one direction are
    # serialised on their stream, so the sum is that direction's busy time)
    h2d_s = sum(a.elapsed_time(b) for a, b in copy_ev["h2d"]) / 1e3
    d2h_s = sum(a.elapsed_time(b) for a, b in copy_ev["d2h"]) / 1e3
    del sets[1]
    return {"value": job_value(blk.weights, ranks.world, sec, args.e2e_steps),
            "unit": "weights/s", "steps": args.e2e_steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_gbs": round(h2d * args.e2e_steps / h2d_s / 1e9, 1),
            "d2h_gbs": round(d2h * args.e2e_steps / d2h_s / 1e9, 1),
            "ms_per_step": round(sec / args.e2e_steps * 1e3, 3),
            "pipelining": "2 device buffer sets; H2D, kernels and D2H of consecutive steps on "
                          "3 streams"}


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def oracle_sample_step(wl, rows_per_matrix: int, layer: int = 0):
    """CPU inputs of `rows_per_matrix` rows of every matrix of the workload,
    drawn with the workload's distributions and per-tensor seeds."""
    from semi_structured_sparsity_gb300 import workloads as W
    import oracle as orc
    out = []
    for m, (name, rows, cols) in enumerate(wl.matrices):
        n = min(rows_per_matrix, rows)
        seed = lambda role: W.tensor_seed(wl.index, layer, m, role)
        Wb = W.bf16_bits(W.normal_bf16(n, cols, wl.w_sigma, seed(W.ROLE_W)))
        Gb = W.bf16_bits(W.normal_bf16(n, cols, wl.g_sigma, seed(W.ROLE_G)))
        if wl.logits == "prior":
            noise = W.normal_f32((n, cols // 4, 6), wl.l_sigma, seed(W.ROLE_L)).numpy()
            L = orc.prior_init(Wb, wl.prior_scale) + noise
        elif wl.logits == "onehot":
            L = W.onehot_logits(n, cols, seed(W.ROLE_L)).numpy()
        else:
            L = W.normal_f32((n, cols // 4, 6), wl.l_sigma, seed(W.ROLE_L)).numpy()
        out.append((Wb, L.astype("float32"), Gb, W.noise_tensor_id(layer, m)))
    return out


def oracle_step(wl, sample, step: int):
    import oracle as orc
    for Wb, L, Gb, tid in sample:
        orc.prior_init(Wb, wl.prior_scale or 1.0)
        orc.forward(Wb, L, wl.tau, wl.kappa, 0, step, tid)
        orc.backward(Wb, L, Gb, wl.tau, wl.kappa, 0, step, tid)
        orc.hard_compress(Wb, L)


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86 "model name"; on Arm the
    implementer and part codes)."""
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return "implementer %s part %s" % (fields.get("CPU implementer", "?"), fields["CPU part"])
    import platform
    return platform.machine()


def oracle_step_sharded(wl, sample, step: int, threads: int):
    """One oracle pass over the sample with every matrix split into `threads`
    row shards, one task per shard on a pool of `threads` threads (the
    oracle's compiled calls release the interpreter lock; row_begin keeps each
    shard's noise counters those of the whole matrix)."""
    import oracle as orc
    from concurrent.futures import ThreadPoolExecutor
    orc.gumbel_noise(0, 0, 0, 0, 1)   # the oracle's table, built once before the threads
    tasks = []
    for Wb, L, Gb, tid in sample:
        rows = Wb.shape[0]
        for i in range(threads):
            a, b = rows * i // threads, rows * (i + 1) // threads
            if b > a:
                tasks.append((Wb[a:b], L[a:b], Gb[a:b], tid, a))

    def run(task):
        Wb, L, Gb, tid, r0 = task
        orc.prior_init(Wb, wl.prior_scale or 1.0)
        orc.forward(Wb, L, wl.tau, wl.kappa, 0, step, tid, row_begin=r0)
        orc.backward(Wb, L, Gb, wl.tau, wl.kappa, 0, step, tid, row_begin=r0)
        orc.hard_compress(Wb, L)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, tasks))


def cpu_baseline(wl, target_seconds: float):
    """The oracle, as it stands, single-threaded, on a bounded sample: the
    first k rows of every matrix of the block, k grown until the timed pass
    takes about `target_seconds`.  The same sample is then run row-sharded
    over every host core (`all_cores`)."""
    k = 1
    while True:
        sample = oracle_sample_step(wl, k)
        t = time.perf_counter()
        oracle_step(wl, sample, 0)
        dt = time.perf_counter() - t
        if dt >= target_seconds or k >= 4096:
            break
        k = min(4096, max(k + 1, int(k * min(8.0, 1.2 * target_seconds / max(dt, 1e-3)))))
    weights = sum(s[0].size for s in sample)
    cores = os.cpu_count() or 1
    t = time.perf_counter()
    oracle_step_sharded(wl, sample, 0, cores)
    dt_all = time.perf_counter() - t
    return {"value": weights / dt, "unit": "weights/s", "cores": 1, "kind": "oracle",
            "sample": "first %d rows of each of the %d matrices (%d weights), one full "
                      "prior+forward+backward+compress pass, %.1f s" % (
                          k, len(sample), weights, dt),
            "cpu_model": cpu_model(),
            "all_cores": {"value": weights / dt_all, "unit": "weights/s", "cores": cores,
                          "sample": "the same sample, every matrix in %d row shards, one "
                                    "thread per shard, %.2f s" % (cores, dt_all)}}


def run_reference(args):
    """The oracle as the reference arm: each step runs prior, forward,
    backward and compress on a bounded sample (the first k rows of every
    matrix), sized so the whole --warmup + --steps run stays within minutes."""
    ranks_world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from semi_structured_sparsity_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    total_steps = args.warmup + args.steps
    budget = 120.0 / max(total_steps, 1)       # seconds of CPU per step
    k = 1
    while True:
        sample = oracle_sample_step(wl, k)
        t = time.perf_counter()
        oracle_step(wl, sample, 0)
        dt = time.perf_counter() - t
        if dt >= 0.5 * budget or k >= 4096:
            break
        k *= 2
    for s in range(args.warmup):
        oracle_step(wl, sample, s)
    t = time.perf_counter()
    for s in range(args.steps):
        oracle_step(wl, sample, args.warmup + s)
    sec = time.perf_counter() - t
    weights = sum(x[0].size for x in sample)
    value = weights * args.steps / sec
    desc = "first %d rows of each of the %d matrices (%d weights) per step" % (
        k, len(sample), weights)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "weights/s",
        "n_gpus": ranks_world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 weights, fp32 logits (oracle computes in fp64)",
        "data": "synthetic (seeded, same recipe as the GPU arm)",
        "config": {"workload": args.workload, "weights_per_step": weights},
        "cpu_baseline": {"value": value, "unit": "weights/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "weights/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
