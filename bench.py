"""Benchmark of the ConvRot W8A8 linear on GB300.

One step = one pass of the runtime path over one batch: the fused
rotate + row-absmax + quantize kernel on X, then the int8 GEMM with the
fused dequant/bias/bf16 epilogue for every linear that shares the packed
activation; for 8-bit codes both through one public call
(convrot_int8_linear), for 4-bit codes through the quantize and linear
calls. Weights are prepared once before timing (the offline path).
`--workload dit_block` chains the linears of one DiT block instead.

Timing: W warm-up steps, then K timed steps; each step is bracketed by CUDA
events on the launching stream (the GEMM is a programmatic dependent launch
of the rotate+quantize, so nothing is recorded between them; each of the two
kernels is then timed alone the same way for the per-kernel figures), and L2
is flushed between steps, outside
the events: a 256 MiB write, then a 256 MiB read, so that the flush's own
dirty lines are written back before the step starts. Clocks are sampled
with nvidia-smi during the timed region. The e2e figure repeats the step
through the public API with host buffers: pinned X copied in, Y copied
back, inside the timed region.

Default workload: the large-M qkv linear (X bf16 [32700, 3072], three
3072-wide linears sharing one packed activation, G = 256), the largest
single-GPU configuration; `--secondary` adds the DiT 4096x6144x6144 step,
GEMM and rotate+quantize times to the same line. The line also carries the
integer tensor-path probe (cuBLASLt int8 and this library's int8 warp-MMA
GEMM at 8192^3, beside torch's fp16 matmul) that the roofline's denominator
choice rests on, and, from the CPU-baseline leg, the GPU codes compared with
the oracle's on the sampled rows.

`--impl reference` times the CPU oracle (fp64 numpy) on a bounded row
sample of the same workload, on the host cores.
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
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as WL  # noqa: E402

METRIC = "ConvRot W8A8 linear int8 TOPS and rotate+quant GB/s, % of roofline"
L2_FLUSH_BYTES = 256 << 20
# GPU-side pause before each timed step (~150 us at 2 GHz) so that the host
# has enqueued the whole step before it starts: the events then time the
# kernels, not the host's launch latency.
PRE_STEP_SLEEP_CYCLES = 300_000

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the step's dominant kernel, from one ncu capture of `bench.py --profile` on
# GB300 (summaries in profiles/), keyed by kernel and workload, with the
# SHA-256 of the kernel's source code (comments aside, see code_sha256) at
# capture time: once the code has changed the figure no longer applies and
# the line reports null.
NCU_TRAFFIC = {
    ("gemm_tc_kernel", "qkv_32700x3072x(3x3072)_G256"): {
        "bytes": 699_902_208 + 580_496_384,
        "source": "int8_convrot_w8a8_gb300/csrc/gemm_tc.cu",
        "sha256": "8cce6a3df0f8969540d9248fb6015864c5adc50dad74cdcf4c11f5cf37bcbf74",
    },
    ("gemm_tc_kernel", "dit_linear_4096x6144x6144_G256"): {
        "bytes": 239_336_192 + 43_612_160,
        "source": "int8_convrot_w8a8_gb300/csrc/gemm_tc.cu",
        "sha256": "8cce6a3df0f8969540d9248fb6015864c5adc50dad74cdcf4c11f5cf37bcbf74",
    },
}


def code_sha256(path: str) -> str:
    """SHA-256 of a C++/CUDA source with its // comments and blank lines
    removed, so that only code changes change it."""
    import hashlib
    import re
    lines = []
    with open(path) as f:
        for line in f:
            line = re.sub(r"//.*", "", line).strip()
            if line:
                lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def ncu_traffic(kernel: str, workload: str):
    rec = NCU_TRAFFIC.get((kernel, workload))
    if rec is None:
        return None
    if code_sha256(os.path.join(ROOT, rec["source"])) != rec["sha256"]:
        return None
    return rec["bytes"]


WORKLOADS = {
    "dit6144": lambda: WL.dit6144(),
    "dit6144_rht128": lambda: WL.dit6144_variant("rht", 128),
    "dit6144_rht256": lambda: WL.dit6144_variant("rht", 256),
    "dit6144_none": lambda: WL.dit6144_variant("none", 0),
    "dit6144_w4": lambda: _w4(WL.dit6144()),
    "qkv32700_w4": lambda: _w4(WL.qkv32700()),
    "gsweep256_w4": lambda: _w4(WL.gsweep(256)),
    "k2688_w4": lambda: _w4(WL.k2688()),
    "qkv32700": lambda: WL.qkv32700(),
    "qkv32700_cat": lambda: _concat(WL.qkv32700()),
    "ffn_pair": lambda: WL.ffn_pair(),
    "gsweep16": lambda: WL.gsweep(16),
    "gsweep64": lambda: WL.gsweep(64),
    "gsweep256": lambda: WL.gsweep(256),
    "gsweep1024": lambda: WL.gsweep(1024),
    "k2688": lambda: WL.k2688(),
    "tiny": lambda: WL.tiny(),
}


def rq_kernel_name(wl) -> str:
    """The rotate+quantize kernel the library picks for this workload (bf16,
    aligned torch buffers)."""
    lines = wl.K // 64
    parts = (lines + 255) // 256
    boxes = wl.K % 64 == 0 and lines % parts == 0 and (parts == 1 or (lines // parts) % 8 == 0)
    if (boxes and wl.transform == "h4" and wl.group in (4, 16, 64, 256, 1024)
            and wl.K % max(256, wl.group) == 0):
        return "rq_mma_kernel"
    # K a multiple of 64 but not of 256: tiles of 2 or 4 rows, groups within a line
    r0 = 2 if lines % 2 == 0 else 4
    if (wl.transform == "h4" and wl.group in (4, 16, 64) and wl.K % 64 == 0 and wl.K >= 256
            and parts == 1 and r0 * wl.K * 2 <= 48 * 1024):
        return "rq_mma_kernel"
    lane = (boxes and K_LANE_MAX >= wl.K and
            ((wl.transform == "h4" and wl.group in (4, 16, 64, 256, 1024)) or
             (wl.transform == "rht" and 2 <= wl.group <= 256) or wl.transform == "none"))
    return "rq_lane_kernel" if lane else "rq_generic_kernel"


K_LANE_MAX = 64 * 384  # the register kernel takes rows of up to 384 lines (in up to two TMA boxes)


def _w4(wl):
    """The same inputs through the 4-bit ConvRot path (codes in [-7, 7])."""
    wl.bits = 4
    wl.name = wl.name + "_W4A4"
    return wl


def _concat(wl):
    wl.weights = [torch.cat(wl.weights)]
    wl.biases = [torch.cat(wl.biases)]
    wl.name = wl.name.replace("(3x3072)", "9216cat")
    return wl


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ------------------------------------------------------------------ oracle ---

def oracle_sample(wl, rows: int, seed: int = 0):
    """Times the CPU oracle on a seeded sample of `rows` rows (full K, all N)."""
    import oracle as O
    sg = None if wl.signs is None else wl.signs.numpy()
    qmax = O.QMAX4 if getattr(wl, "bits", 8) == 4 else O.QMAX
    Ws = [O.prepare_weights(W.numpy().astype(np.float64), wl.group, wl.transform, sg, qmax) for W in wl.weights]
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(wl.M, size=min(rows, wl.M), replace=False))
    X64 = wl.X[torch.from_numpy(idx)].float().numpy().astype(np.float64)
    t0 = time.perf_counter()
    Qx, sx, v = O.quantize_act(X64, wl.group, wl.transform, sg, qmax)
    t1 = time.perf_counter()
    for (Qw, sw, _), b in zip(Ws, wl.biases):
        O.round_to_bf16(O.reconstruct(O.int_gemm(Qx, Qw), sx, sw, b.numpy()))
    t2 = time.perf_counter()
    ops = 2.0 * len(idx) * sum(wl.Ns) * wl.K
    return {"rows": len(idx), "seconds": t2 - t0, "quant_seconds": t1 - t0, "ops": ops,
            "idx": idx, "Qx": Qx, "sx": sx, "v": v}


def code_parity(ref, q_gpu, s_gpu, bits: int):
    """The GPU's codes and scales on the oracle's sampled rows: code flips
    (|dQ| = 1 near a rounding boundary is the tolerated case), the largest
    distance of a flipped code's fp64 value to its boundary, and the largest
    relative scale error."""
    import oracle as O
    q = q_gpu[ref["idx"]]
    if bits == 4:
        q = O.unpack_int4(q)
    d = q.astype(np.int64) - ref["Qx"].astype(np.int64)
    flips = d != 0
    dist = O.boundary_distance(ref["v"][flips])
    s_ref = ref["sx"].astype(np.float64)
    s_err = np.abs(s_gpu[ref["idx"]].astype(np.float64) - s_ref) / np.where(s_ref > 0, s_ref, 1.0)
    return {"rows": int(len(ref["idx"])), "elements": int(d.size), "flips": int(flips.sum()),
            "max_abs_dq": int(np.abs(d).max(initial=0)),
            "code_flip_max_boundary_distance": float(dist.max()) if dist.size else None,
            "scale_max_rel_err": float(s_err.max(initial=0.0))}


def reference_main(args, world, rank):
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]()
    rows = args.ref_rows
    res = []
    for _ in range(args.warmup):
        oracle_sample(wl, max(8, rows // 8))
    for s in range(args.steps):
        res.append(oracle_sample(wl, rows, seed=s))
    secs = sum(r["seconds"] for r in res)
    ops = sum(r["ops"] for r in res)
    value = ops / secs / 1e12
    cores = blas_threads()
    sample = f"{rows} seeded rows of {wl.M} per step (full K={wl.K}, all N={sum(wl.Ns)}), fp64 numpy"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TOPS", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- GPU ---

def _best_ms(fn, reps: int = 5, warm: int = 2) -> float:
    for _ in range(warm):
        fn()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1)
        best = t if best is None else min(best, t)
    return best


def int8_peak_probe(cr, dev, n: int = 8192) -> dict:
    """The integer tensor paths this chip offers, at n^3: cuBLASLt's int8
    GEMM (torch._int_mm, measurement only) and this library's int8 warp-MMA
    GEMM, beside torch's fp16 matmul. sm_103a has no integer tcgen05 MMA, so
    the library feeds the int8 codes to the fp16 tensor cores (exact); its
    roofline is the bf16/fp16 dense peak, the fastest exact path there is."""
    g = torch.Generator(device="cpu").manual_seed(11)
    a8 = torch.randint(-127, 128, (n, n), dtype=torch.int8, generator=g).to(dev)
    b8 = torch.randint(-127, 128, (n, n), dtype=torch.int8, generator=g).to(dev)
    ops = 2.0 * n ** 3
    res = {"shape": f"{n}x{n}x{n}"}
    try:
        bt = b8.t()
        res["int_mm_tops"] = ops / _best_ms(lambda: torch._int_mm(a8, bt)) / 1e9
    except RuntimeError as e:  # not every torch build has it for this arch
        res["int_mm_tops"] = None
        res["int_mm_error"] = str(e).splitlines()[0][:120]
    ones_x = torch.ones(n, dtype=torch.float32, device=dev)
    act = cr.PackedAct(a8, ones_x, None, 0, cr.TRANSFORMS["none"])
    w = cr.PackedWeight(b8, ones_x.clone(), None, 0, cr.TRANSFORMS["none"])
    y = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
    res["int8_mma_sync_tops"] = ops / _best_ms(lambda: cr.convrot_linear(act, w, out=y, int8_mma=True)) / 1e9
    h = a8.to(torch.float16)
    ht = b8.to(torch.float16).t()
    res["fp16_matmul_tflops"] = ops / _best_ms(lambda: torch.matmul(h, ht)) / 1e9
    if cr.convrot_get_device_status() != 0:
        raise RuntimeError("device status after the int8 probe")
    best_int = max(v for v in (res["int_mm_tops"], res["int8_mma_sync_tops"]) if v is not None)
    res["best_integer_path_tops"] = best_int
    res["denominator"] = ("bf16 dense burst peak (MEASURED_PEAKS.json): the int8 codes run exactly on the "
                          "fp16 tensor cores, whose rate equals bf16's; the integer paths above are "
                          "the dense INT8 figures this chip offers")
    return res


def read_floor(dev, nbytes: int, flush_l2, steps: int, warmup: int) -> dict:
    """A plain read of nbytes from HBM (torch amax over an fp32 buffer of that
    size) and a plain copy of them, timed like a step (L2 flushed, GPU-side
    pause): the practical floor for streaming that many bytes once."""
    src = torch.zeros(max(1, nbytes // 4), dtype=torch.float32, device=dev)
    dst = torch.empty_like(src)
    out = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        marks = []
        for i in range(warmup + steps):
            flush_l2()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= warmup:
                marks.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in marks) * 1e3

    return {"bytes": 4 * src.numel(), "read_us": timed(lambda: torch.amax(src, dim=0, out=out)),
            "copy_us": timed(lambda: dst.copy_(src))}


def l2_flusher(dev):
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one: the written
        # lines leave L2 (and reach DRAM) here, not inside the next timed step
        flush.zero_()
        torch.sum(flush_rd, dim=0, out=flush_sink)

    return flush_l2



def secondary_figures(cr, args, name, dev, flush_l2) -> dict:
    """Step, GEMM and rotate+quantize (int8 contract) times of a second 8-bit
    workload, same protocol as the main line (L2 flushed, GPU-side pause,
    CUDA events on the launching stream)."""
    wl = WORKLOADS[name]()
    stream = torch.cuda.current_stream()
    sg = None if wl.signs is None else wl.signs.to(dev)
    use_f16 = wl.M > 64
    ws = [cr.convrot_prepare_weights(W.to(dev), wl.group, wl.transform, sg, with_f16=use_f16) for W in wl.weights]
    bs = [b.to(dev) for b in wl.biases]
    X = wl.X.to(dev)
    outs = [torch.empty((wl.M, n), dtype=torch.bfloat16, device=dev) for n in wl.Ns]
    gws = cr.gemm_workspace(dev)
    scratch = cr.int8_linear_scratch(wl.M, wl.K, dev)
    act = cr.convrot_quantize_act(X, wl.group, wl.transform, sg, with_f16=use_f16)
    act8 = cr.convrot_quantize_act(X, wl.group, wl.transform, sg, with_f16=False)

    def timed(fn):
        marks = []
        for i in range(args.warmup + args.steps):
            flush_l2()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                marks.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in marks) / 1e3

    step_s = timed(lambda: cr.convrot_int8_linear(X, ws, bs, signs=sg, outs=outs, scratch=scratch, workspace=gws))
    gemm_s = timed(lambda: cr.convrot_linear_multi(act, ws, bs, outs=outs, workspace=gws))
    q_s = timed(lambda: cr.convrot_quantize_act(X, wl.group, wl.transform, sg, with_f16=False, out=act8))
    floor = read_floor(dev, (3 * wl.M * wl.K + 4 * wl.M) // 2, flush_l2, args.steps, args.warmup)
    if cr.convrot_get_device_status() != 0:
        raise RuntimeError(f"device status after the {name} figures")
    pk = peaks()
    M, K, Ns = wl.M, wl.K, wl.Ns
    ops = 2.0 * M * sum(Ns) * K
    q_bytes = 3 * M * K + 4 * M
    gemm_tflops = ops / gemm_s / 1e12
    return {"workload": wl.name, "step_us": step_s * 1e6, "step_tops": ops / step_s / 1e12,
            "gemm_us": gemm_s * 1e6, "gemm_tflops": gemm_tflops,
            "gemm_frac": gemm_tflops / pk["bf16_tflops"] if use_f16 else None,
            "rotate_quant": {"kernel": rq_kernel_name(wl), "us": q_s * 1e6, "algorithmic_bytes": q_bytes,
                             "gbs": q_bytes / q_s / 1e9, "frac": q_bytes / q_s / 1e9 / pk["hbm_gbs"],
                             "copy_floor_us": floor["copy_us"], "frac_of_copy_floor": floor["copy_us"] / (q_s * 1e6)}}


def gpu_main(args, world, rank, local):
    import int8_convrot_w8a8_gb300 as cr

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = WORKLOADS[args.workload]()
    stream = torch.cuda.current_stream()
    sg = None if wl.signs is None else wl.signs.to(dev)
    bits = getattr(wl, "bits", 8)
    # the tensor-core operand copies: fp16 (8-bit codes, M > 64) or e4m3 (4-bit codes, always)
    use_f16 = wl.M > 64 or bits == 4
    if bits == 4:
        def quant(Xq, with_f16, out=None, stream=None):
            return cr.convrot_quantize_act4(Xq, wl.group, wl.transform, sg, with_f8=with_f16, out=out, stream=stream)

        def lin(a, outs_, workspace, stream=None):
            cr.convrot_linear4_multi(a, ws, bs, outs=outs_, stream=stream, workspace=workspace)

        ws = [cr.convrot_prepare_weights4(W.to(dev), wl.group, wl.transform, sg) for W in wl.weights]
    else:
        def quant(Xq, with_f16, out=None, stream=None):
            return cr.convrot_quantize_act(Xq, wl.group, wl.transform, sg, with_f16=with_f16, out=out, stream=stream)

        def lin(a, outs_, workspace, stream=None):
            if len(ws) == 1:
                cr.convrot_linear(a, ws[0], bs[0], out=outs_[0], stream=stream, workspace=workspace)
            else:
                cr.convrot_linear_multi(a, ws, bs, outs=outs_, stream=stream, workspace=workspace)

        ws = [cr.convrot_prepare_weights(W.to(dev), wl.group, wl.transform, sg, with_f16=use_f16)
              for W in wl.weights]
    bs = [b.to(dev) for b in wl.biases]
    X = wl.X.to(dev)
    M, K, Ns = wl.M, wl.K, wl.Ns
    act = quant(X, use_f16)
    outs = [torch.empty((M, n), dtype=torch.bfloat16, device=dev) for n in Ns]
    gws = cr.gemm_workspace(dev)  # lets the GEMM split a mostly idle last round of tiles
    flush_l2 = l2_flusher(dev)
    # 8-bit steps go through the one-call linear (rotate+quantize, then the
    # GEMM as its programmatic dependent)
    one_call = None
    if bits == 8:
        scratch = cr.int8_linear_scratch(M, K, dev)

        def one_call(Xq, outs_, scratch_, workspace, stream=None):
            cr.convrot_int8_linear(Xq, ws, bs, signs=sg, outs=outs_, scratch=scratch_, workspace=workspace,
                                   stream=stream)

    def step():
        if one_call is not None:
            one_call(X, outs, scratch, gws)
        else:
            # nothing between the two launches: the GEMM is a programmatic
            # dependent of the rotate+quantize and may start while it finishes
            quant(X, use_f16, out=act)
            lin(act, outs, gws)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    assert cr.convrot_get_device_status() == 0
    if args.profile:
        # a short, fixed launch list for ncu: one more step, then one int8-only
        # rotate+quantize, the same on the register butterfly kernel where the
        # library runs the tensor-core one, and (where supported) one
        # matmul-form rotate+quantize
        step()
        quant(X, False)
        if bits == 8 and rq_kernel_name(wl) == "rq_mma_kernel":
            cr.convrot_quantize_act_kernel(X, wl.group, wl.transform, sg, kernel="butterfly", with_f16=False)
        if bits == 8 and wl.transform == "h4" and wl.group in (16, 64, 256) and K % max(wl.group, 64) == 0 \
                and K // max(wl.group, 64) <= 128:
            cr.convrot_quantize_act_hmatmul(X, wl.group, with_f16=False)
        torch.cuda.synchronize()
        return

    barrier(world)
    torch.cuda.synchronize()
    host_us = []
    with ClockSampler(local) as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush_l2()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            e0, e1 = ev[i]
            h0 = time.perf_counter()
            e0.record(stream)
            step()
            e1.record(stream)
            host_us.append(1e6 * (time.perf_counter() - h0))
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
    barrier(world)
    status = cr.convrot_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    def timed(fn):
        """Per-launch times (ms) of fn alone, same flush and pause as a step."""
        marks = []
        for i in range(args.warmup + args.steps):
            flush_l2()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            fn()
            b1.record(stream)
            if i >= args.warmup:
                marks.append((b0, b1))
        torch.cuda.synchronize()
        return [b0.elapsed_time(b1) for b0, b1 in marks]

    # the step's two kernels timed alone: the GEMM (the roofline kernel) and
    # the rotate+quantize with its operand copy
    gemm_ms = timed(lambda: lin(act, outs, gws))
    quant_ms = timed(lambda: quant(X, use_f16, out=act))
    # the rotate+quantize contract alone (bf16 in, codes + fp32 scales out, no
    # operand copy), for the GB/s figure
    act8 = quant(X, False)
    q_only_ms = timed(lambda: quant(X, False, out=act8))
    # the same contract with the rotation applied as a dense tensor-core matmul
    hm_ms = None
    if bits == 8 and wl.transform == "h4" and wl.group in (16, 64, 256) and K % max(wl.group, 64) == 0 \
            and K // max(wl.group, 64) <= 128:
        hm_ms = []
        for i in range(args.warmup + args.steps):
            flush_l2()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            cr.convrot_quantize_act_hmatmul(X, wl.group, with_f16=False)
            b1.record(stream)
            if i >= args.warmup:
                hm_ms.append((b0, b1))
        torch.cuda.synchronize()
        hm_ms = [b0.elapsed_time(b1) for b0, b1 in hm_ms]
    # the same contract on the all-fp32 register butterfly kernel, where the
    # library runs the tensor-core stage instead
    bf_ms = None
    if bits == 8 and rq_kernel_name(wl) == "rq_mma_kernel":
        actb = quant(X, False)
        bf_ms = timed(lambda: cr.convrot_quantize_act_kernel(X, wl.group, wl.transform, sg, kernel="butterfly",
                                                             with_f16=False, out=actb))
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)

    ops_step = 2.0 * M * sum(Ns) * K
    value = world * ops_step * args.steps / total_s / 1e12
    pk = peaks()
    gemm_s = statistics.mean(gemm_ms) / 1e3
    quant_s = statistics.mean(quant_ms) / 1e3
    gemm_tflops = ops_step / gemm_s / 1e12
    # algorithmic bytes of rotate+quantize: bf16 in, int8 out, fp32 scales
    # 4-bit codes are packed two per byte; their e4m3 copy is one byte per code
    q_bytes = 2 * M * K + (M * K if bits == 8 else M * K // 2) + 4 * M
    q_bytes_f16 = q_bytes + (2 if bits == 8 else 1) * M * K if use_f16 else q_bytes
    quant_only_s = statistics.mean(q_only_ms) / 1e3
    quant_gbs = q_bytes / quant_only_s / 1e9
    # the floor for moving the contract's bytes once in this protocol: a plain
    # torch copy of half of them (it reads and writes each byte once)
    q_floor = read_floor(dev, q_bytes // 2, flush_l2, args.steps, args.warmup)
    if bits == 4:
        # e4m3 dense rate: the measured bf16 burst x the nominal fp8 / bf16 ratio (4.5 / 2.25)
        peak8 = 2.0 * pk["bf16_tflops"]
        dominant = {"kernel": "gemm_tc_kernel", "bound": "tensor", "achieved": gemm_tflops,
                    "peak": peak8, "unit": "TFLOP/s", "frac": gemm_tflops / peak8,
                    "traffic": ncu_traffic("gemm_tc_kernel", wl.name),
                    "peak_note": f"{pk['source']} bf16 dense burst x 2 (nominal fp8/bf16 ratio 4.5/2.25)"}
    elif use_f16:
        dominant = {"kernel": "gemm_tc_kernel", "bound": "tensor", "achieved": gemm_tflops,
                    "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": gemm_tflops / pk["bf16_tflops"],
                    "traffic": ncu_traffic("gemm_tc_kernel", wl.name),
                    "peak_note": f"{pk['source']} bf16 dense burst; the fp16 tensor rate is the same (nominal ratio 1)"}
    else:
        w_bytes = sum(n * K + 4 * n for n in Ns) + M * K + 4 * M + 2 * M * sum(Ns)
        gbs = w_bytes / gemm_s / 1e9
        floor = read_floor(dev, w_bytes, flush_l2, args.steps, args.warmup)
        dominant = {"kernel": "gemm_small_tc_kernel" if M > 16 and K % 128 == 0 else "gemm_small_kernel",
                    "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": gbs / pk["hbm_gbs"], "traffic": None,
                    "peak_note": f"{pk['source']} HBM copy bandwidth",
                    "read_floor": dict(floor, gemm_us=gemm_s * 1e6,
                                       ratio_to_read=gemm_s * 1e6 / floor["read_us"],
                                       ratio_to_copy=gemm_s * 1e6 / floor["copy_us"],
                                       note="the weight-stream GEMM against a plain torch read (amax) and copy "
                                            "of the same number of bytes, same flush and pause")}

    secondary = None
    if args.secondary != "none" and args.secondary != args.workload and bits == 8:
        secondary = secondary_figures(cr, args, args.secondary, dev, flush_l2)
    probe = None if args.no_int8_probe else int8_peak_probe(cr, dev)
    if probe is not None and use_f16 and bits == 8:
        probe["gemm_over_best_integer_path"] = gemm_tflops / probe["best_integer_path_tops"]
        probe["gemm_frac_of_fp16_matmul"] = gemm_tflops / probe["fp16_matmul_tflops"]

    # ---- end to end through the public API with host buffers: every step
    # copies its X in from pinned host memory and its Y back out; three streams
    # with their own device buffers keep consecutive steps in flight, so one
    # step's copies overlap another's kernels (no L2 flush here: each step's
    # input arrives from the host).
    Xh = wl.X.pin_memory()
    nbuf = 3
    e2e_streams = [torch.cuda.Stream() for _ in range(nbuf)]
    bufs = []
    for _ in range(nbuf):
        Xd = torch.empty_like(X)
        bufs.append({"X": Xd,
                     "act": quant(Xd.zero_(), use_f16),
                     "scratch": cr.int8_linear_scratch(M, K, dev) if one_call is not None else None,
                     "Y": [torch.empty((M, n), dtype=torch.bfloat16, device=dev) for n in Ns],
                     "ws": cr.gemm_workspace(dev),
                     "Yh": [torch.empty((M, n), dtype=torch.bfloat16).pin_memory() for n in Ns]})

    def e2e_step(i):
        b, s = bufs[i % nbuf], e2e_streams[i % nbuf]
        with torch.cuda.stream(s):
            b["X"].copy_(Xh, non_blocking=True)
            if one_call is not None:
                one_call(b["X"], b["Y"], b["scratch"], b["ws"], stream=s)
            else:
                quant(b["X"], use_f16, out=b["act"], stream=s)
                lin(b["act"], b["Y"], b["ws"], stream=s)
            for y, yh in zip(b["Y"], b["Yh"]):
                yh.copy_(y, non_blocking=True)

    torch.cuda.synchronize()
    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for s in e2e_streams:
        s.wait_event(a0)
    for i in range(args.steps):
        e2e_step(i)
    for s in e2e_streams:
        stream.wait_stream(s)
    a1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(a0.elapsed_time(a1) / 1e3, world)
    e2e_value = world * ops_step * args.steps / e2e_s / 1e12
    e2e_ms = [1e3 * e2e_s / args.steps]

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(step_ms), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8" if bits == 8 else "int4", "data": "synthetic",
        "config": {"workload": wl.name, "M": M, "K": K, "N": Ns, "group": wl.group, "transform": wl.transform,
                   "seed": wl.seed, "l2": "flushed between steps outside the events: 256 MiB write, then 256 MiB read",
                   "inputs": wl.description,
                   "gemm_path": ("tcgen05 e4m3-exact (kind::f8f6f4)" if bits == 4 else
                                 "tcgen05 fp16-exact" if use_f16 else "int8 weight stream (TMA + mma.sync s8)"),
                   "step": ("convrot_int8_linear" if one_call is not None else
                            "convrot_quantize_act4 + convrot_linear4_multi")},
        "roofline": dominant,
        "rotate_quant": {"kernel": rq_kernel_name(wl),
                         "us": quant_only_s * 1e6, "gbs": quant_gbs, "peak_gbs": pk["hbm_gbs"],
                         "frac": quant_gbs / pk["hbm_gbs"], "algorithmic_bytes": q_bytes,
                         "note": ("packed 4-bit codes + scales only; in the step the kernel also writes the e4m3 copy"
                                  if bits == 4 else
                                  "int8 codes + scales only; in the step the kernel also writes the fp16 operand copy"),
                         "in_step_us": quant_s * 1e6, "in_step_bytes": q_bytes_f16,
                         "in_step_gbs": q_bytes_f16 / quant_s / 1e9,
                         "copy_floor_us": q_floor["copy_us"],
                         "frac_of_copy_floor": q_floor["copy_us"] / (quant_only_s * 1e6),
                         "copy_floor_note": "a torch copy reading and writing the contract's algorithmic bytes "
                                            "once, same flush and pause (event-timed launches carry a fixed "
                                            "cost of a few microseconds on this GPU)"},
        "rotate_quant_hmatmul": None if hm_ms is None else {
            "kernel": "hmatmul_kernel", "us": statistics.mean(hm_ms) * 1e3,
            "gbs": q_bytes / (statistics.mean(hm_ms) / 1e3) / 1e9,
            "frac": q_bytes / (statistics.mean(hm_ms) / 1e3) / 1e9 / pk["hbm_gbs"],
            "tensor_tflops": 2.0 * M * K * max(wl.group, 64) / (statistics.mean(hm_ms) / 1e3) / 1e12},
        "rotate_quant_butterfly": None if bf_ms is None else {
            "kernel": "rq_lane_kernel", "us": statistics.mean(bf_ms) * 1e3,
            "gbs": q_bytes / (statistics.mean(bf_ms) / 1e3) / 1e9,
            "frac": q_bytes / (statistics.mean(bf_ms) / 1e3) / 1e9 / pk["hbm_gbs"]},
        "gemm_us": gemm_s * 1e6,
        "int8_peak_probe": probe,
        "secondary": secondary,
        "gpu_launches": 2 * args.steps,
        "e2e": {"value": e2e_value, "unit": "TOPS", "h2d_bytes_per_step": 2 * M * K,
                "d2h_bytes_per_step": 2 * M * sum(Ns), "ms_per_step": statistics.mean(e2e_ms),
                "pipelining": "3 streams, copies of one step overlap kernels of the others"},
        "clocks": clocks.summary(),
        "wall_s_timed": wall1 - wall0,
        "host_us_per_step": statistics.median(host_us),
    }
    if world == 1 and not args.no_cpu_baseline:
        # about 10 s of oracle work: seeded row samples of the same workload;
        # the first sample's codes are also compared with the GPU's int8-only
        # launch on the same rows
        secs, ops, rows, reps = 0.0, 0.0, 0, 0
        q_gpu = (act8.q4 if bits == 4 else act8.q).cpu().numpy()
        s_gpu = act8.scale.cpu().numpy()
        parity = None
        while secs < args.cpu_seconds:
            ref = oracle_sample(wl, args.ref_rows, seed=100 + reps)
            secs += ref["seconds"]
            ops += ref["ops"]
            rows += ref["rows"]
            if parity is None:
                parity = code_parity(ref, q_gpu, s_gpu, bits)
            reps += 1
        cores = blas_threads()
        line["cpu_baseline"] = {"value": ops / secs / 1e12, "unit": "TOPS", "cores": cores, "kind": "oracle",
                                "sample": f"{reps} x {args.ref_rows} seeded rows of {M} ({rows} rows, full K, "
                                          f"all N), fp64 numpy, {secs:.1f} s"}
        line["code_parity"] = dict(parity, tolerance="|dQ| <= 1 on <= 1e-4 of elements, flips within "
                                                     "1e-6 * 127 code units of a rounding boundary")
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ DiT block ---

BLOCKS = {"dit_block": lambda: WL.dit_block()}


def block_main(args, world, rank, local):
    """The linears of one DiT block, each group one library call from its bf16
    input (rotate + quantize, then the GEMM as its programmatic dependent):
    qkv (three linears sharing one packed activation), the output projection,
    fc1 on the projection's output, fc2 on fc1's output."""
    import int8_convrot_w8a8_gb300 as cr

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    blk = BLOCKS[args.workload]()
    G, T = blk.group, blk.transform
    M, D, H = blk.M, blk.D, blk.fc1.shape[0]

    def prep(W):
        return cr.convrot_prepare_weights(W.to(dev), G, T)

    qkv_w, qkv_b = [prep(W) for W in blk.qkv], [b.to(dev) for b in blk.qkv_b]
    out_w, out_b = prep(blk.out), blk.out_b.to(dev)
    fc1_w, fc1_b = prep(blk.fc1), blk.fc1_b.to(dev)
    fc2_w, fc2_b = prep(blk.fc2), blk.fc2_b.to(dev)
    X, A = blk.X.to(dev), blk.A.to(dev)
    Yqkv = [torch.empty((M, D), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    Yo = torch.empty((M, D), dtype=torch.bfloat16, device=dev)
    Yh = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    Y2 = torch.empty((M, D), dtype=torch.bfloat16, device=dev)
    scratch = cr.int8_linear_scratch(M, max(D, H), dev)  # one scratch, reused in stream order
    gws = cr.gemm_workspace(dev)
    flush_l2 = l2_flusher(dev)
    # (name, input, weights, biases, outputs)
    layers = [("qkv", X, qkv_w, qkv_b, Yqkv), ("out_proj", A, [out_w], [out_b], [Yo]),
              ("fc1", Yo, [fc1_w], [fc1_b], [Yh]), ("fc2", Yh, [fc2_w], [fc2_b], [Y2])]

    def run(layer, s=None):
        _, x, w, b, y = layer
        cr.convrot_int8_linear(x, w, b, outs=y, scratch=scratch, workspace=gws, stream=s)

    def step():
        for layer in layers:
            run(layer)

    def timed(fn):
        marks = []
        for i in range(args.warmup + args.steps):
            flush_l2()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                marks.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in marks) / 1e3

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if cr.convrot_get_device_status() != 0:
        raise RuntimeError("device status after warm-up")
    barrier(world)
    with ClockSampler(local) as clocks:
        step_s = timed(step)
    total_s = max_over_ranks(step_s * args.steps, world)
    # each group alone: the whole call, its GEMM on a packed activation made
    # beforehand, and its rotate+quantize (with the fp16 operand copy)
    per = []
    for layer in layers:
        name, x, w, b, y = layer
        a = cr.convrot_quantize_act(x, G, T, with_f16=True)
        gemm_s = timed(lambda: cr.convrot_linear_multi(a, w, b, outs=y, workspace=gws))
        quant_s = timed(lambda: cr.convrot_quantize_act(x, G, T, with_f16=True, out=a))
        call_s = timed(lambda: run(layer))
        K = x.shape[1]
        ops = 2.0 * M * K * sum(ww.N for ww in w)
        per.append({"layer": name, "K": K, "N": [ww.N for ww in w], "call_us": call_s * 1e6,
                    "rotate_quant_kernel": rq_kernel_name(types.SimpleNamespace(K=K, transform=T, group=G)),
                    "gemm_us": gemm_s * 1e6, "gemm_tflops": ops / gemm_s / 1e12,
                    "rotate_quant_us": quant_s * 1e6,
                    "rotate_quant_gbs": (5.0 * M * K + 4 * M) / quant_s / 1e9, "ops": ops})
        del a
    torch.cuda.synchronize()
    if cr.convrot_get_device_status() != 0:
        raise RuntimeError("device status after the timed region")
    ops_step = sum(p_["ops"] for p_ in per)
    value = world * ops_step * args.steps / total_s / 1e12
    pk = peaks()
    gemm_tflops = ops_step / sum(p_["gemm_us"] for p_ in per) * 1e-6
    q_bytes = sum(5.0 * M * p_["K"] + 4 * M for p_ in per)
    q_s = sum(p_["rotate_quant_us"] for p_ in per) / 1e6

    # end to end through the public API: X and A in from pinned host memory,
    # the qkv outputs and the block output back, every step, one stream
    Xh, Ah = blk.X.pin_memory(), blk.A.pin_memory()
    Yqkv_h = [torch.empty((M, D), dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    Y2_h = torch.empty((M, D), dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        X.copy_(Xh, non_blocking=True)
        A.copy_(Ah, non_blocking=True)
        step()
        for y, yh in zip(Yqkv + [Y2], Yqkv_h + [Y2_h]):
            yh.copy_(y, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(timed(e2e_step) * args.steps, world)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": blk.name, "M": M, "D": D, "mlp_width": H, "group": G, "transform": T,
                   "seed": blk.seed, "inputs": blk.description,
                   "l2": "flushed between steps outside the events: 256 MiB write, then 256 MiB read",
                   "calls": "4 x convrot_int8_linear (rotate+quantize, then the GEMM as its programmatic dependent)"},
        "roofline": {"kernel": "gemm_tc_kernel", "bound": "tensor", "achieved": gemm_tflops,
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": gemm_tflops / pk["bf16_tflops"],
                     "traffic": None,
                     "peak_note": f"{pk['source']} bf16 dense burst; the four GEMMs' flops over their summed times"},
        "rotate_quant": {"kernel": "+".join(sorted({p_["rotate_quant_kernel"] for p_ in per})),
                         "us": q_s * 1e6, "gbs": q_bytes / q_s / 1e9,
                         "peak_gbs": pk["hbm_gbs"], "frac": q_bytes / q_s / 1e9 / pk["hbm_gbs"],
                         "algorithmic_bytes": q_bytes,
                         "note": "the four rotate+quantize launches with their fp16 operand copies (5 bytes per element)"},
        "layers": per,
        "gpu_launches": 8 * args.steps,
        "e2e": {"value": world * ops_step * args.steps / e2e_s / 1e12, "unit": "TOPS",
                "h2d_bytes_per_step": 2 * 2 * M * D, "d2h_bytes_per_step": 4 * 2 * M * D,
                "ms_per_step": 1e3 * e2e_s / args.steps, "pipelining": "none: one stream"},
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


ROWPAR = {"qkv32700_rowpar2": lambda: (WL.qkv32700(), 2)}


def rowpar_main(args, world, rank, local):
    """One rank of a row-parallel (K-sharded) linear group (sglang digest,
    "风险与影响": each rank holds whole groups of every row): the qkv linears
    with their 3072 input features split over two ranks. Each rank runs the
    row maxima of its slice, the quantization of its slice against the
    all-reduced maxima, its partial int32 accumulators (one launch for the
    three weights), and after the all-reduced sum the dequant. This GPU runs
    rank 0's launches, each timed alone and all four back to back; the two
    all-reduces are exchanges between GPUs and are not part of the time."""
    import int8_convrot_w8a8_gb300 as cr

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    wl, ranks = ROWPAR[args.workload]()
    M, K, G, T = wl.M, wl.K, wl.group, wl.transform
    Kr = K // ranks
    Xf = wl.X.to(dev)
    slices = [Xf[:, r * Kr:(r + 1) * Kr] for r in range(ranks)]  # views, row pitch K
    X = slices[rank % ranks]
    ws = [cr.convrot_prepare_weights(W.to(dev), G, T) for W in wl.weights]  # offline, whole K
    cols = slice((rank % ranks) * Kr, (rank % ranks + 1) * Kr)
    qw = torch.cat([w.q[:, cols] for w in ws]).contiguous()
    w_cat = cr.PackedWeight(qw, torch.cat([w.scale for w in ws]), qw.to(torch.float16), G, ws[0].transform)
    b_cat = torch.cat([b.to(dev) for b in wl.biases])
    N = w_cat.N
    # the two exchanges, done once outside the timed launches
    amax_all = torch.stack([cr.convrot_rotate_absmax(x, G, T) for x in slices]).amax(dim=0)
    amax = torch.empty(M, dtype=torch.float32, device=dev)
    act = cr.convrot_quantize_act_given_max(X, amax_all, G, T)
    A = torch.empty((M, N), dtype=torch.int32, device=dev)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush_l2 = l2_flusher(dev)

    def s_absmax():
        cr.convrot_rotate_absmax(X, G, T, out=amax)

    def s_quant():
        cr.convrot_quantize_act_given_max(X, amax_all, G, T, out=act)

    def s_gemm():
        cr.convrot_gemm_s32(act, w_cat, out=A)

    def s_dequant():
        cr.convrot_dequant(A, act.scale, w_cat.scale, b_cat, out=Y)

    def s_all():
        s_absmax()
        s_quant()
        s_gemm()
        s_dequant()

    def timed(fn):
        marks = []
        for i in range(args.warmup + args.steps):
            flush_l2()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                marks.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in marks) / 1e3

    if args.profile:
        # a short, fixed launch list for ncu: the four launches, twice
        for _ in range(2):
            s_all()
        torch.cuda.synchronize()
        return
    barrier(world)
    with ClockSampler(local) as clocks:
        step_s = timed(s_all)
    total_s = max_over_ranks(step_s * args.steps, world)
    parts = {name: timed(fn) for name, fn in
             (("rotate_absmax", s_absmax), ("quantize_given_max", s_quant), ("gemm_s32", s_gemm),
              ("dequant", s_dequant))}
    torch.cuda.synchronize()
    if cr.convrot_get_device_status() != 0:
        raise RuntimeError("device status after the timed region")
    if rank != 0:
        return
    pk = peaks()
    ops = 2.0 * M * N * Kr
    bytes_ = {"rotate_absmax": 2.0 * M * Kr + 4 * M,
              "quantize_given_max": 2.0 * M * Kr + 4 * M + 1.0 * M * Kr + 4 * M,
              "dequant": 4.0 * M * N + 2.0 * M * N + 4 * M + 8 * N}
    steps = {}
    for name, t in parts.items():
        d = {"us": t * 1e6}
        if name in bytes_:
            d.update({"algorithmic_bytes": bytes_[name], "gbs": bytes_[name] / t / 1e9,
                      "frac_of_hbm": bytes_[name] / t / 1e9 / pk["hbm_gbs"]})
            if name == "quantize_given_max":
                d["note"] = "int8 codes + scales; the launch also writes the fp16 operand copy the GEMM reads"
        else:
            d.update({"tflops": ops / t / 1e12, "frac_of_bf16": ops / t / 1e12 / pk["bf16_tflops"]})
        steps[name] = d
    g = parts["gemm_s32"]
    line = {
        "metric": METRIC, "value": ops * args.steps / total_s / 1e12, "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": wl.name + f"_rowparallel{ranks}_rank0", "M": M, "K": K, "K_per_rank": Kr, "N": N,
                   "group": G, "transform": T, "seed": wl.seed, "ranks": ranks,
                   "l2": "flushed between steps outside the events: 256 MiB write, then 256 MiB read",
                   "exchanges": "the all-reduce (max) of the row maxima and the all-reduce (sum) of the int32 "
                                "partial accumulators run between GPUs and are not in the time (one GPU)",
                   "value": "this rank's 2*M*N*K_per_rank int ops over its four launches back to back"},
        "roofline": {"kernel": "gemm_tc_kernel", "bound": "tensor", "achieved": ops / g / 1e12,
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": ops / g / 1e12 / pk["bf16_tflops"],
                     "traffic": None, "peak_note": f"{pk['source']} bf16 dense burst (raw int32 output)"},
        "steps_alone": steps,
        "gpu_launches": 4 * args.steps,
        "e2e": None,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="qkv32700", choices=sorted(WORKLOADS) + sorted(BLOCKS) + sorted(ROWPAR))
    ap.add_argument("--secondary", default="dit6144", choices=["none"] + sorted(WORKLOADS),
                    help="a second 8-bit workload whose step, GEMM and rotate+quantize times go in the same line")
    ap.add_argument("--no-int8-probe", action="store_true",
                    help="skip the integer tensor-path probe (torch._int_mm, the int8 warp-MMA GEMM)")
    ap.add_argument("--ref-rows", type=int, default=1024)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", action="store_true",
                    help="prepare, warm up, run one more step and exit (for ncu captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            if args.workload in BLOCKS or args.workload in ROWPAR:
                ap.error("the reference arm times single-linear workloads")
            reference_main(args, world, rank)
        elif args.workload in BLOCKS:
            block_main(args, world, rank, local)
        elif args.workload in ROWPAR:
            rowpar_main(args, world, rank, local)
        else:
            gpu_main(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
