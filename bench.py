"""Benchmark of the GB300 GEMM library.

Headline: BF16 NT GEMM at the Qwen-2B-shaped MLP gate/up size
(M=5120, N=11008, K=2048), TFLOP/s per GPU (whole job over all ranks).  A
step is one gemm_bf16_nt call (tile scheduler, TMA staging, tcgen05 MMA and
BF16 epilogue) over one batch of synthetic inputs already resident in HBM.
Consecutive steps rotate over several copies of the inputs and outputs so
that the working set (> 2x L2) is never served from L2.  The other shapes of
the same metric (down, qkv, gqa, their split-K / stream-K schedules, the
NN layout, the W4A16 GEMM, the LoRA fold, the router and the NVFP4 GEMM)
are measured the same way and reported under "shapes".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s and % of GB300 dense BF16/FP4 tensor peak, per shape"
L2_BYTES = 129 * 1024 * 1024
E2E_CHUNKS = 4  # row chunks of the e2e pipeline
E2E_COPY_STREAMS = 1  # two measured no faster: device-to-host bandwidth bounds the step
# nominal dense FP4 / dense BF16 tensor rate on GB300 (15 / 2.25 PFLOP/s)
FP4_PEAK_RATIO = 15.0 / 2.25
# The block-scaled 256x256x64 MMA of a CTA pair takes the same 162.3 cycles
# as the BF16 256x256x16 one (bench.py --tensor-rate), so the tensor pipe's
# own FP4 ceiling is 4x the BF16 rate.
FP4_MMA_RATIO = 4.0
SM_MAX_MHZ = 2070.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-shapes", action="store_true", help="headline shape only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--clock-warm-s", type=float, default=0.6,
                    help="extra warm-up seconds so that clock samples cover the load")
    ap.add_argument("--shapes",
                    default="down,qkv,gqa,gateup_nn,gqa_splitk,down_streamk,qkv_streamk,w4a16,lora,"
                            "router,nvfp4,nvfp4_decode",
                    help="comma list of the extra shapes to measure")
    ap.add_argument("--no-headline", action="store_true",
                    help="profiling aid: measure only --shapes and print them")
    ap.add_argument("--tensor-rate", action="store_true",
                    help="measure the tcgen05 MMA issue rate (BF16 and block-scaled FP4) with "
                         "the probe library and print it, instead of the GEMM benchmark")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampler running while the GPU is under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        win = [p for (t, p) in self.samples if t0 - 0.06 <= t <= t1 + 0.06]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        smax = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        power = [num(p[3]) for p in win if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "power_w_max": max(power) if power else None, "samples": len(win)}


# ----------------------------------------------------------------- timing
def time_launches(torch, stream, fn, n_sets, warmup, steps, min_warm_s=0.0):
    """Run `fn(i % n_sets)` warmup + steps times on `stream`; time the steps
    with CUDA events recorded on that stream.  Returns (seconds per step,
    wall-clock window of the timed region)."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn(i % n_sets)
        stream.synchronize()
        if min_warm_s > 0:  # keep the GPU busy long enough for clock samples
            t_end = time.time() + min_warm_s
            i = 0
            while time.time() < t_end:
                for _ in range(20):
                    fn(i % n_sets)
                    i += 1
                stream.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        start.record(stream)
        for i in range(steps):
            fn(i % n_sets)
        end.record(stream)
        end.synchronize()
        t1 = time.time()
    return start.elapsed_time(end) / 1e3 / steps, (t0, t1)


def reduce_max(torch, dist, value: float, device) -> float:
    """Max of `value` over the ranks of the default process group (identity
    when torch.distributed is not initialised)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def n_sets_for(bytes_per_set: int) -> int:
    return max(2, -(-2 * L2_BYTES // max(1, bytes_per_set)) + 1)


def headline_config(w, world: int) -> dict:
    """The headline workload as both arms name it: the gate/up GEMM and the
    GPU arm's L2 rule (rotating input/output sets larger than 2x L2)."""
    set_bytes = (w.M * w.K + w.N * w.K + w.M * w.N) * 2
    nsets = n_sets_for(set_bytes)
    return {"workload": "bf16 NT GEMM M=5120 N=11008 K=2048 (Qwen-2B-shaped MLP gate/up)",
            "M": w.M, "N": w.N, "K": w.K, "parallelism": f"replicas x{world}",
            "l2": f"rotating {nsets} input/output sets ({nsets * set_bytes / 2**20:.0f} MiB "
                  f"> 2x L2) between steps"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_tcgen05_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- CPU oracle
def cpu_baseline(seconds: float):
    """The oracle, as it stands, on whole sampled rows of the gate/up GEMM."""
    import oracle
    from nvfp4_block_scaled_tcgen05_gb300 import synth
    w = synth.BF16_WORKLOADS["gateup"]
    A, B = synth.gemm_inputs(w)
    threads = oracle.default_threads()
    rng = np.random.default_rng(0)
    rows_done, t_spent, chunk = 0, 0.0, max(threads, 16)
    while t_spent < seconds and rows_done < w.M:
        rows = rng.integers(0, w.M, size=chunk)
        t0 = time.perf_counter()
        oracle.gemm_bf16_nt(A, B, rows=rows, threads=threads)
        t_spent += time.perf_counter() - t0
        rows_done += chunk
        chunk = min(chunk * 2, 4 * threads * 8)
    flops = 2.0 * rows_done * w.N * w.K
    return {"value": flops / t_spent / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{rows_done} sampled rows of the 5120x11008x2048 BF16 GEMM "
                      f"({flops / 1e9:.1f} GFLOP in {t_spent:.1f} s)"}


def run_reference(args):
    """Reference arm: the CPU oracle, timed as it stands on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from nvfp4_block_scaled_tcgen05_gb300 import synth
    w = synth.BF16_WORKLOADS["gateup"]
    A, B = synth.gemm_inputs(w)
    threads = oracle.default_threads()
    rows_per_step = 4 * threads
    rng = np.random.default_rng(1)
    for _ in range(args.warmup):
        oracle.gemm_bf16_nt(A, B, rows=rng.integers(0, w.M, rows_per_step), threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm_bf16_nt(A, B, rows=rng.integers(0, w.M, rows_per_step), threads=threads)
    dt = (time.perf_counter() - t0) / args.steps
    value = 2.0 * rows_per_step * w.N * w.K / dt / 1e12
    sample = f"{rows_per_step} sampled rows of the 5120x11008x2048 BF16 GEMM per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(w, args.gpus),
        "cpu_baseline": {"kind": "oracle", "cores": threads, "sample": sample, "value": value,
                         "unit": "TFLOP/s"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


# ----------------------------------------------------------------- tensor rate
def tensor_rate(torch, dev, local, n_mma=8192):
    """SM cycles per CTA-pair MMA issued back to back by one thread (zero
    operands in shared memory), for kind::f16 256xNx16 and kind::mxf4nvf4
    256xNx64 (N = 256: the square tiles; N = 128: the decode tiles), alone on
    one CTA pair and on every SM pair, and with tcgen05.cp scale copies
    issued by two other warps at the same time (per 4 MMAs: `copies`
    32x128b.warpx4 and `wide` 128x256b; the decode kernel's mix is 4 + 2).
    With `commit_every` the issuers also commit per stage as the GEMM
    kernel does (the MMA thread every 4 MMAs; the copy warps after each
    group); `flags` place waiting threads beside the MMAs (bit meanings in
    probe/tensor_rate.cu: 1 multicast commits, 2 a polling thread on the
    peer CTA, 4 that poll sleeps, 8/16 one lane / a whole warp of the MMA
    CTA polling, 32 that poll sleeps, 64 / 128 commits in a fixed pattern
    after each group of 4 MMAs / after the next group's first MMA).
    Whole-GPU rates use CUDA events around
    the launch and the SM clock sampled meanwhile."""
    import ctypes
    from nvfp4_block_scaled_tcgen05_gb300 import build as _b
    lib = ctypes.CDLL(_b.PROBE_LIB)
    f = lib.probe_tensor_rate
    f.argtypes = [ctypes.c_int] * 8 + [ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    props = torch.cuda.get_device_properties(dev)
    pairs = props.multi_processor_count // 2
    out = torch.zeros(2 * pairs, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    rows = []
    kdepth = {0: 16, 1: 64}
    cases = ((0, 256, 0, 0, 0, 0), (1, 256, 0, 0, 0, 0), (1, 256, 8, 0, 0, 0),
             (1, 256, 12, 0, 0, 0), (1, 256, 0, 0, 0, 2), (1, 256, 0, 0, 0, 24),
             (1, 256, 0, 0, 4, 0), (1, 256, 0, 0, 64, 0), (1, 256, 0, 0, 4096, 0),
             (1, 256, 0, 0, 4, 64), (1, 256, 0, 0, 4, 128), (1, 256, 0, 0, 4, 65),
             (1, 256, 0, 0, 4, 129), (1, 256, 8, 0, 4, 129), (0, 256, 0, 0, 4, 64),
             (0, 192, 0, 0, 0, 0), (0, 192, 0, 0, 4, 64), (0, 128, 0, 0, 0, 0),
             (1, 128, 0, 0, 0, 0), (1, 128, 4, 2, 0, 0),
             (1, 128, 4, 2, 4, 64), (1, 128, 4, 2, 4, 129))
    for kind, mma_n, copies, wide, commit_every, flags in cases:
        flops = 2.0 * 256 * mma_n * kdepth[kind]
        for clusters in (1, pairs):
            for _ in range(2):  # warm-up launch, then the measured one
                rc = f(kind, mma_n, clusters, n_mma, copies, wide, commit_every, flags,
                       out.data_ptr(), stream)
                if rc:
                    raise RuntimeError(f"probe_tensor_rate rc={rc}")
            clocks = ClockSampler(local)
            clocks.start()
            time.sleep(0.15)
            t0 = time.time()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 20 if clusters > 1 else 3
            e0.record()
            for _ in range(reps):
                f(kind, mma_n, clusters, n_mma, copies, wide, commit_every, flags, out.data_ptr(),
                  stream)
            e1.record()
            e1.synchronize()
            t1 = time.time()
            clocks.stop()
            clk = clocks.summary(t0, t1)
            v = out.view(pairs, 2)[:clusters].cpu().numpy()
            cyc = v[:, 0].astype(np.float64) / n_mma
            sec = e0.elapsed_time(e1) / 1e3 / reps
            rows.append({"kind": (f"bf16 kind::f16 256x{mma_n}x16" if kind == 0
                                  else f"nvfp4 kind::mxf4nvf4 4X 256x{mma_n}x64"),
                         "copies_per_4_mma": copies, "wide_copies_per_4_mma": wide,
                         "commit_every": commit_every, "flags": flags,
                         "cta_pairs": clusters,
                         "cycles_per_mma_median": float(np.median(cyc)),
                         "cycles_per_mma_max": float(cyc.max()),
                         "flop_per_sm_per_cycle": flops / 2 / float(np.median(cyc)),
                         "tflops_whole_launch": clusters * n_mma * flops / sec / 1e12,
                         "sm_mhz_median": clk.get("sm_mhz")})
    return rows


def probe_fp4_mma_rate(torch, dev, n_mma=8192, reps=20):
    """The block-scaled MMA's own rate on this GPU now: the issue-rate probe
    (kind::mxf4nvf4 256x256x64 back to back from zeroed shared memory, no
    scale copies or commits) on every CTA pair, TFLOP/s by CUDA events."""
    import ctypes
    from nvfp4_block_scaled_tcgen05_gb300 import build as _b
    lib = ctypes.CDLL(_b.PROBE_LIB)
    f = lib.probe_tensor_rate
    f.argtypes = [ctypes.c_int] * 8 + [ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    pairs = torch.cuda.get_device_properties(dev).multi_processor_count // 2
    out = torch.zeros(2 * pairs, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(2):
        if f(1, 256, pairs, n_mma, 0, 0, 0, 0, out.data_ptr(), stream):
            raise RuntimeError("probe_tensor_rate failed")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        f(1, 256, pairs, n_mma, 0, 0, 0, 0, out.data_ptr(), stream)
    e1.record()
    e1.synchronize()
    sec = e0.elapsed_time(e1) / 1e3 / reps
    return pairs * n_mma * 2.0 * 256 * 256 * 64 / sec / 1e12


# ----------------------------------------------------------------- our arm
def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.tensor_rate:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        print(json.dumps({"tensor_rate": tensor_rate(torch, torch.device("cuda", local), local)}))
        return
    import torch
    import torch.distributed as dist

    import __graft_entry__
    import nvfp4_block_scaled_tcgen05_gb300 as g
    from nvfp4_block_scaled_tcgen05_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    __graft_entry__.build()
    lib = g.load()
    pk = peaks()
    stream = torch.cuda.Stream(device=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x: float) -> float:
        return reduce_max(torch, dist, x, dev)

    def up(x, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(x))
        if dtype is not None:
            t = t.view(dtype)
        return t.to(dev)

    if args.no_headline:
        shapes = measure_shapes(torch, lib, synth, up, stream, dev, pk, max(3, args.warmup),
                                args.steps, args.shapes.split(","), args.clock_warm_s)
        if rank == 0:
            print(json.dumps({"shapes": shapes}))
        return

    # ------------------------------------------------ headline: gate/up
    w = synth.BF16_WORKLOADS["gateup"]
    A_h, B_h = synth.gemm_inputs(w, seed_offset=rank)
    set_bytes = (w.M * w.K + w.N * w.K + w.M * w.N) * 2
    nsets = n_sets_for(set_bytes)
    A0, B0 = up(A_h, torch.bfloat16), up(B_h, torch.bfloat16)
    As = [A0] + [A0.clone() for _ in range(nsets - 1)]
    Bs = [B0] + [B0.clone() for _ in range(nsets - 1)]
    Cs = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev) for _ in range(nsets)]
    sp = stream.cuda_stream

    def step(i):
        rc = lib.gemm_bf16_nt(As[i].data_ptr(), Bs[i].data_ptr(), Cs[i].data_ptr(), w.M, w.N, w.K, sp)
        if rc:
            raise RuntimeError(g.status_string(rc))

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    t_load0 = time.time()
    sec, (t0, t1) = time_launches(torch, stream, step, nsets, max(3, args.warmup), args.steps,
                                  min_warm_s=args.clock_warm_s)
    barrier()
    clocks.stop()
    clk = clocks.summary(t_load0, t1)
    sec = max_over_ranks(sec)
    flops = 2.0 * w.M * w.N * w.K
    per_gpu_tflops = flops / sec / 1e12
    value = world * per_gpu_tflops
    assert lib.gemm_get_device_status(sp) == 0
    # The timed steps above follow >= clock_warm_s of back-to-back load; about
    # 50 ms into such load the power cap lowers the SM clock (measured: 129 us
    # per step at 2070 MHz, then ~140 us at ~1730 MHz), so they are compared
    # with the sustained peak.  The same steps after 1 s without load run at
    # the boost clock: that figure is compared with the burst peak.
    sustained_region = args.clock_warm_s >= 0.1
    time.sleep(1.0)
    burst_sec, _ = time_launches(torch, stream, step, nsets, 3, args.steps)
    burst_sec = max_over_ranks(burst_sec)
    burst_tflops = flops / burst_sec / 1e12

    # ------------------------------------------------ e2e through host buffers
    # Every step copies that step's A and B from pinned host memory and reads
    # C back to pinned host memory.  The step is pipelined over E2E_CHUNKS
    # row chunks of A/C (each chunk one gemm_bf16_nt call on 256-row-aligned
    # rows, so results equal the one-call GEMM bit for bit): host-to-device
    # copies, GEMMs and device-to-host copies run on three streams, and two
    # device buffer sets let step i+1's copies and GEMMs proceed while step
    # i's result is still being read back.  The timed region runs the steps
    # back to back and ends after the last step's read-back.
    A_pin = torch.from_numpy(A_h.view(np.int16)).pin_memory()
    B_pin = torch.from_numpy(B_h.view(np.int16)).pin_memory()
    C_pin = torch.empty((w.M, w.N), dtype=torch.int16).pin_memory()
    bufs = [(As[j].view(torch.int16), Bs[j].view(torch.int16), Cs[j].view(torch.int16))
            for j in range(min(2, nsets))]
    # copies alternate over E2E_COPY_STREAMS streams per direction (each
    # stream's copies can go to a different copy engine)
    s_h2ds = [torch.cuda.Stream(device=dev) for _ in range(E2E_COPY_STREAMS)]
    s_d2hs = [torch.cuda.Stream(device=dev) for _ in range(E2E_COPY_STREAMS)]
    nch = E2E_CHUNKS if w.M % (256 * E2E_CHUNKS) == 0 else 1
    rows = w.M // nch
    done_gemm = [None] * len(bufs)   # last GEMM event per buffer set
    done_d2h = [None] * len(bufs)    # last device-to-host event per buffer set
    e2e_count = [0]

    def e2e_step(_):
        j = e2e_count[0] % len(bufs)
        e2e_count[0] += 1
        A_d, B_d, C_d = bufs[j]
        loaded = []
        if done_gemm[j] is not None:
            for sh in s_h2ds:
                sh.wait_event(done_gemm[j])  # the GEMMs that read this set are done
        nb_rows = w.N // len(s_h2ds)
        b_done = []
        for k, sh in enumerate(s_h2ds):  # B split over the copy streams
            with torch.cuda.stream(sh):
                r1 = w.N if k == len(s_h2ds) - 1 else (k + 1) * nb_rows
                B_d[k * nb_rows:r1].copy_(B_pin[k * nb_rows:r1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(sh)
                b_done.append(ev)
        for c in range(nch):
            sh = s_h2ds[c % len(s_h2ds)]
            with torch.cuda.stream(sh):
                A_d[c * rows:(c + 1) * rows].copy_(A_pin[c * rows:(c + 1) * rows], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(sh)
                loaded.append(ev)
        for ev in b_done:
            stream.wait_event(ev)
        computed = []
        for c in range(nch):
            stream.wait_event(loaded[c])
            if c == 0 and done_d2h[j] is not None:
                stream.wait_event(done_d2h[j])  # C of this set was read back
            rc = lib.gemm_bf16_nt(A_d[c * rows:].data_ptr(), B_d.data_ptr(),
                                  C_d[c * rows:].data_ptr(), rows, w.N, w.K, sp)
            if rc:
                raise RuntimeError(g.status_string(rc))
            ev = torch.cuda.Event()
            ev.record(stream)
            computed.append(ev)
        done_gemm[j] = computed[-1]
        ends = []
        for c in range(nch):
            sd = s_d2hs[c % len(s_d2hs)]
            with torch.cuda.stream(sd):
                sd.wait_event(computed[c])
                C_pin[c * rows:(c + 1) * rows].copy_(C_d[c * rows:(c + 1) * rows], non_blocking=True)
                if c >= nch - len(s_d2hs):
                    ev = torch.cuda.Event()
                    ev.record(sd)
                    ends.append(ev)
        # one event for "C of this set has been read back"; the compute
        # stream waits on it only before it next writes this set, so step
        # i+1's GEMMs overlap step i's device-to-host copies
        s0 = s_d2hs[0]
        for ev in ends[1:]:
            s0.wait_event(ev)
        done = torch.cuda.Event()
        done.record(s0)
        done_d2h[j] = done
        last_d2h[0] = done

    last_d2h = [None]

    def e2e_timed(nsteps):
        """nsteps pipelined steps, timed on `stream` from before the first
        copy to after the last step's device-to-host copies."""
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for s_ in s_h2ds + s_d2hs:
            s_.wait_event(start)
        for i in range(nsteps):
            e2e_step(i)
        stream.wait_event(last_d2h[0])
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end) / 1e3 / nsteps

    e2e_steps = max(3, min(args.steps, 20))
    for i in range(2):  # warm-up steps
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_sec = max_over_ranks(e2e_timed(e2e_steps))
    h2d = (w.M * w.K + w.N * w.K) * 2
    d2h = w.M * w.N * 2
    # the e2e output must equal the device-resident result bit for bit
    torch.cuda.synchronize()
    e2e_ok = bool(torch.equal(C_pin.to(dev), Cs[0].view(torch.int16))) if nsets > 0 else False

    del As, Bs, Cs
    torch.cuda.empty_cache()

    # ------------------------------------------------ other shapes
    shapes = []
    if not args.no_shapes:
        shapes = measure_shapes(torch, lib, synth, up, stream, dev, pk, max(3, args.warmup),
                                30, args.shapes.split(","), args.clock_warm_s)

    peak_used = pk["bf16_tflops_sustained"] if sustained_region else pk["bf16_tflops"]
    peak_source = (f"{pk['source']} cuBLAS bf16 sustained (the timed steps follow "
                   f"{args.clock_warm_s:g} s of load, past the point where the power cap "
                   f"lowers the SM clock)" if sustained_region
                   else f"{pk['source']} cuBLAS bf16 burst")
    result = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": headline_config(w, world),
        "roofline": {"bound": "tensor", "achieved": per_gpu_tflops, "peak": peak_used,
                     "unit": "TFLOP/s", "frac": per_gpu_tflops / peak_used,
                     "peak_source": peak_source,
                     "burst": {"achieved": burst_tflops, "ms_per_step": burst_sec * 1e3,
                               "peak": pk["bf16_tflops"],
                               "frac": burst_tflops / pk["bf16_tflops"],
                               "note": "the same steps after 1 s without load (boost clock), "
                                       f"against the {pk['source']} cuBLAS bf16 burst"},
                     "kernel": "tcgen05_gemm_kernel<TileCfg<bf16, CTA pair, 256x256 tile, 3 x 128-deep stages>, StoreBF16>",
                     "traffic": recorded_traffic("gemm_bf16_gateup")},
        "e2e": {"value": world * flops / e2e_sec / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_sec * 1e3, "matches_device_result": e2e_ok,
                "pipeline": f"{nch} row chunks; GEMMs on one stream, copies on "
                            f"{E2E_COPY_STREAMS} streams per direction; 2 device buffer sets"},
        "gpu_launches": args.steps,
        "clocks": clk,
        "shapes": shapes,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def measure_shapes(torch, lib, synth, up, stream, dev, pk, warmup, reps, which,
                   clock_warm_s=0.6):
    sp = stream.cuda_stream
    which = {w.strip() for w in which if w.strip()}
    out = []
    bf16_peak = pk["bf16_tflops"]
    fp4_peak = bf16_peak * FP4_PEAK_RATIO

    def check(rc):
        if rc:
            raise RuntimeError(f"status {rc}")

    # plain BF16 shapes
    for name in ("down", "qkv", "gqa", "gateup"):
        if name not in which:
            continue
        w = synth.BF16_WORKLOADS[name]
        A_h, B_h = synth.gemm_inputs(w)
        set_bytes = (w.M * w.K + w.N * w.K + w.M * w.N) * 2
        n = n_sets_for(set_bytes)
        A0, B0 = up(A_h, torch.bfloat16), up(B_h, torch.bfloat16)
        As = [A0] + [A0.clone() for _ in range(n - 1)]
        Bs = [B0] + [B0.clone() for _ in range(n - 1)]
        Cs = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev) for _ in range(n)]
        fn = lambda i: check(lib.gemm_bf16_nt(As[i].data_ptr(), Bs[i].data_ptr(), Cs[i].data_ptr(),
                                              w.M, w.N, w.K, sp))
        sec, _ = time_launches(torch, stream, fn, n, warmup, reps)
        tf = 2.0 * w.M * w.N * w.K / sec / 1e12
        out.append({"shape": name, "M": w.M, "N": w.N, "K": w.K, "us": sec * 1e6, "TFLOP/s": tf,
                    "frac_bf16_peak": tf / bf16_peak})
        del As, Bs, Cs

    if "gateup_nn" in which:
        # NN layout (B stored [K][N]) on the gate/up shape
        w = synth.BF16_WORKLOADS["gateup"]
        A_h, B_h = synth.gemm_inputs(w)
        Bkn_h = np.ascontiguousarray(B_h.T)
        set_bytes = (w.M * w.K + w.N * w.K + w.M * w.N) * 2
        n = n_sets_for(set_bytes)
        A0, B0 = up(A_h, torch.bfloat16), up(Bkn_h, torch.bfloat16)
        As = [A0] + [A0.clone() for _ in range(n - 1)]
        Bs = [B0] + [B0.clone() for _ in range(n - 1)]
        Cs = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev) for _ in range(n)]
        fn = lambda i: check(lib.gemm_bf16_nn(As[i].data_ptr(), Bs[i].data_ptr(), Cs[i].data_ptr(),
                                              w.M, w.N, w.K, sp))
        sec, _ = time_launches(torch, stream, fn, n, warmup, reps)
        tf = 2.0 * w.M * w.N * w.K / sec / 1e12
        out.append({"shape": "gateup_nn", "M": w.M, "N": w.N, "K": w.K, "us": sec * 1e6,
                    "TFLOP/s": tf, "frac_bf16_peak": tf / bf16_peak})
        del As, Bs, Cs

    if "gqa_splitk" in which:
        out.append(measure_splitk(torch, lib, synth, up, stream, dev, warmup, reps, check,
                                  bf16_peak, "gqa", 4))
    for name in ("down", "qkv", "gateup"):
        if f"{name}_streamk" in which:
            out.append(measure_streamk(torch, lib, synth, up, stream, dev, warmup, reps, check,
                                       bf16_peak, name))
    for name in sorted(synth.W4A16):
        if name in which or "w4a16" in which:
            out.append(measure_w4a16(torch, lib, synth, up, stream, dev, warmup, reps, check,
                                     bf16_peak, name))
    if "lora" in which:
        out.append(measure_lora(torch, lib, synth, up, stream, dev, pk, warmup, reps, check))
    if "router" in which:
        out.append(measure_router(torch, lib, synth, up, stream, dev, warmup, reps, check))
    if "nvfp4" in which:
        out.append(measure_nvfp4(torch, lib, synth, up, stream, dev, warmup, reps, check, fp4_peak,
                                 sustained_s=0.4 if clock_warm_s > 0 else 0.0))
    if "nvfp4_decode" in which:
        for name in sorted(synth.NVFP4_DECODE):
            out.append(measure_nvfp4_decode(torch, lib, synth, up, stream, dev, pk, warmup, reps,
                                            check, fp4_peak, name))
    assert lib.gemm_get_device_status(sp) == 0
    return out


def measure_splitk(torch, lib, synth, up, stream, dev, warmup, reps, check, bf16_peak, name,
                   splits):
    """Split-K GEMM (both kernels: FP32 partials + ordered reduce) on one shape."""
    import ctypes
    sp = stream.cuda_stream
    w = synth.BF16_WORKLOADS[name]
    A_h, B_h = synth.gemm_inputs(w)
    ws_bytes = int(lib.gemm_bf16_nt_splitk_workspace_bytes(w.M, w.N, w.K, splits))
    set_bytes = (w.M * w.K + w.N * w.K + w.M * w.N) * 2 + ws_bytes
    n = n_sets_for(set_bytes)
    A0, B0 = up(A_h, torch.bfloat16), up(B_h, torch.bfloat16)
    As = [A0] + [A0.clone() for _ in range(n - 1)]
    Bs = [B0] + [B0.clone() for _ in range(n - 1)]
    Cs = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev) for _ in range(n)]
    Ws = [torch.empty(ws_bytes, dtype=torch.uint8, device=dev) for _ in range(n)]
    fn = lambda i: check(lib.gemm_bf16_nt_splitk(As[i].data_ptr(), Bs[i].data_ptr(),
                                                 Cs[i].data_ptr(), Ws[i].data_ptr(),
                                                 ctypes.c_size_t(ws_bytes), w.M, w.N, w.K,
                                                 splits, sp))
    sec, _ = time_launches(torch, stream, fn, n, warmup, reps)
    tf = 2.0 * w.M * w.N * w.K / sec / 1e12
    del As, Bs, Cs, Ws
    return {"shape": f"{name}_splitk{splits}", "M": w.M, "N": w.N, "K": w.K, "us": sec * 1e6,
            "TFLOP/s": tf, "frac_bf16_peak": tf / bf16_peak}


def measure_streamk(torch, lib, synth, up, stream, dev, warmup, reps, check, bf16_peak, name):
    """Stream-K GEMM (GEMM with FP32 partial tiles + ordered fixup) on one shape;
    the 160-tile shapes leave 8 tiles for a third round on 76 CTA pairs, the
    860-tile gate/up shape 24 tiles for a twelfth."""
    import ctypes
    sp = stream.cuda_stream
    w = synth.BF16_WORKLOADS[name]
    A_h, B_h = synth.gemm_inputs(w)
    ws_bytes = int(lib.gemm_bf16_nt_streamk_workspace_bytes())
    set_bytes = (w.M * w.K + w.N * w.K + w.M * w.N) * 2
    n = n_sets_for(set_bytes)
    A0, B0 = up(A_h, torch.bfloat16), up(B_h, torch.bfloat16)
    As = [A0] + [A0.clone() for _ in range(n - 1)]
    Bs = [B0] + [B0.clone() for _ in range(n - 1)]
    Cs = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev) for _ in range(n)]
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)  # stream-ordered reuse
    fn = lambda i: check(lib.gemm_bf16_nt_streamk(As[i].data_ptr(), Bs[i].data_ptr(),
                                                  Cs[i].data_ptr(), ws.data_ptr(),
                                                  ctypes.c_size_t(ws_bytes), w.M, w.N, w.K, sp))
    sec, _ = time_launches(torch, stream, fn, n, warmup, reps)
    tf = 2.0 * w.M * w.N * w.K / sec / 1e12
    del As, Bs, Cs, ws
    return {"shape": f"{name}_streamk", "M": w.M, "N": w.N, "K": w.K, "us": sec * 1e6,
            "TFLOP/s": tf, "frac_bf16_peak": tf / bf16_peak}


def measure_lora(torch, lib, synth, up, stream, dev, pk, warmup, reps, check):
    """LoRA fold: fused scaled-acc vs the unfused pair; HBM-bound."""
    sp = stream.cuda_stream
    w = synth.LORA
    X_h, W_h = synth.gemm_inputs(w)
    O_h = synth.scaled_acc_out(w.M, w.N, w.seed)
    Xd, Wd = up(X_h, torch.bfloat16), up(W_h, torch.bfloat16)
    n = n_sets_for(w.M * w.N * 2)
    Os = [up(O_h, torch.bfloat16) for _ in range(n)]
    scratch = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
    import ctypes
    sc = ctypes.c_float(synth.LORA_SCALE)
    fused = lambda i: check(lib.gemm_bf16_nt_scaled_acc(Xd.data_ptr(), Wd.data_ptr(), Os[i].data_ptr(),
                                                        w.M, w.N, w.K, sc, sp))
    def unfused(i):
        check(lib.gemm_bf16_nt(Xd.data_ptr(), Wd.data_ptr(), scratch.data_ptr(), w.M, w.N, w.K, sp))
        check(lib.bf16_scaled_add(Os[i].data_ptr(), scratch.data_ptr(), sc, w.M * w.N, sp))
    sec_f, _ = time_launches(torch, stream, fused, n, warmup, reps)
    sec_u, _ = time_launches(torch, stream, unfused, n, warmup, reps)
    bytes_fused = 2 * w.M * w.N * 2 + (w.M + w.N) * w.K * 2
    res = {"shape": "lora_fold", "M": w.M, "N": w.N, "K": w.K, "us": sec_f * 1e6,
           "GB/s": bytes_fused / sec_f / 1e9,
           "frac_hbm_peak": bytes_fused / sec_f / 1e9 / pk["hbm_gbs"],
           "unfused_us": sec_u * 1e6, "fused_speedup": sec_u / sec_f,
           "TFLOP/s": 2.0 * w.M * w.N * w.K / sec_f / 1e12}
    del Os, scratch
    return res


def measure_router(torch, lib, synth, up, stream, dev, warmup, reps, check):
    """Ordered router GEMM on CUDA cores: 2 flops per (multiply, add) pair,
    against the FP32 pipe's one fused multiply-add (2 flops) per lane per
    clock, which the kernel issues where the products are exact."""
    sp = stream.cuda_stream
    w = synth.ROUTER
    A_h, B_h = synth.gemm_inputs(w)
    n = n_sets_for((w.M * w.K + w.N * w.K) * 2 + w.M * w.N * 4)
    A0, B0 = up(A_h, torch.bfloat16), up(B_h, torch.bfloat16)
    Ad = [A0] + [A0.clone() for _ in range(n - 1)]
    Bd = [B0] + [B0.clone() for _ in range(n - 1)]
    Cr = [torch.empty((w.M, w.N), dtype=torch.float32, device=dev) for _ in range(n)]
    fn = lambda i: check(lib.gemm_bf16_nt_ordered(Ad[i].data_ptr(), Bd[i].data_ptr(),
                                                  Cr[i].data_ptr(), w.M, w.N, w.K, sp))
    sec, _ = time_launches(torch, stream, fn, n, warmup, reps)
    props = torch.cuda.get_device_properties(dev)
    alu_peak = props.multi_processor_count * 128 * 2 * 2070e6 / 1e12  # FMA TFLOP/s, max SM clock
    tf = 2.0 * w.M * w.N * w.K / sec / 1e12
    res = {"shape": "router", "M": w.M, "N": w.N, "K": w.K, "us": sec * 1e6, "TFLOP/s": tf,
           "frac_alu_peak": tf / alu_peak, "alu_peak_tflops": alu_peak}
    del Ad, Bd, Cr
    return res


def measure_nvfp4(torch, lib, synth, up, stream, dev, warmup, reps, check, fp4_peak,
                  sustained_s=0.4):
    """NVFP4 block-scaled GEMM at L=1, 4096 x 7168 x 16384; with sustained_s > 0
    also back to back for that long with the SM clock sampled."""
    sp = stream.cuda_stream
    w = synth.NVFP4
    a_h, b_h, sfa_h, sfb_h = synth.nvfp4_inputs(w)
    set_bytes = a_h.size + b_h.size + sfa_h.size + sfb_h.size + w.L * w.M * w.N * 2
    n = n_sets_for(set_bytes)
    a0, b0, sa0, sb0 = up(a_h), up(b_h), up(sfa_h), up(sfb_h)
    sets = [(a0, b0, sa0, sb0)] + [(a0.clone(), b0.clone(), sa0.clone(), sb0.clone())
                                   for _ in range(n - 1)]
    cs = [torch.empty((w.L, w.M, w.N), dtype=torch.float16, device=dev) for _ in range(n)]
    fn = lambda i: check(lib.gemm_nvfp4_bs(sets[i][0].data_ptr(), sets[i][1].data_ptr(),
                                           sets[i][2].data_ptr(), sets[i][3].data_ptr(),
                                           cs[i].data_ptr(), w.L, w.M, w.N, w.K, sp))
    # the MMA's own rate, measured by the issue-rate probe just before
    probe_rate = probe_fp4_mma_rate(torch, dev)
    sec, _ = time_launches(torch, stream, fn, n, warmup, reps)
    flops = 2.0 * w.L * w.M * w.N * w.K
    tf = flops / sec / 1e12
    mma_rate = fp4_peak * FP4_MMA_RATIO / FP4_PEAK_RATIO  # 4 x measured BF16 burst
    res = {"shape": "nvfp4", "L": w.L, "M": w.M, "N": w.N, "K": w.K, "us": sec * 1e6,
           "TFLOP/s": tf, "frac_fp4_peak": tf / fp4_peak, "fp4_peak_tflops": fp4_peak,
           "fp4_peak_source": "measured bf16 burst x nominal fp4/bf16 ratio 15/2.25",
           "fp4_mma_rate_tflops": mma_rate,
           "frac_fp4_mma_rate": tf / mma_rate,
           "fp4_probe_mma_rate_tflops": probe_rate,
           "frac_fp4_probe_mma_rate": tf / probe_rate}
    # The same launches back to back for ~0.5 s with the SM clock sampled:
    # real FP4 operands draw enough power for the power cap to lower the
    # clock, and the MMA rate scales with it.
    if sustained_s > 0:
        clocks = ClockSampler(dev.index if dev.index is not None else 0)
        clocks.start()
        time.sleep(0.1)
        t0 = time.time()
        sec_s, (_, t1) = time_launches(torch, stream, fn, n, 0, reps, min_warm_s=sustained_s)
        clocks.stop()
        clk = clocks.summary(t0, t1)
        tf_s = flops / sec_s / 1e12
        sus = {"us": sec_s * 1e6, "TFLOP/s": tf_s, "sm_mhz": clk.get("sm_mhz"),
               "reasons": clk.get("reasons")}
        if clk.get("sm_mhz"):
            sus["frac_fp4_mma_rate_at_sm_mhz"] = tf_s / (mma_rate * clk["sm_mhz"] / SM_MAX_MHZ)
        res["sustained"] = sus
    del sets, cs
    return res


def measure_w4a16(torch, lib, synth, up, stream, dev, warmup, reps, check, bf16_peak, name):
    """W4A16 (BF16 activations x NVFP4 weights, converted on chip) on one shape.
    The MMAs are BF16: reported against the BF16 tensor peak."""
    sp = stream.cuda_stream
    w = synth.W4A16[name]
    A_h, b_h, sfb_h, scale2 = synth.w4a16_inputs(w)
    set_bytes = A_h.size * 2 + b_h.size + sfb_h.size + w.M * w.N * 2
    n = n_sets_for(set_bytes)
    A0, b0, s0 = up(A_h, torch.bfloat16), up(b_h), up(sfb_h)
    sets = [(A0, b0, s0)] + [(A0.clone(), b0.clone(), s0.clone()) for _ in range(n - 1)]
    cs = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev) for _ in range(n)]
    fn = lambda i: check(lib.gemm_w4a16(sets[i][0].data_ptr(), sets[i][1].data_ptr(),
                                        sets[i][2].data_ptr(), scale2, cs[i].data_ptr(),
                                        w.M, w.N, w.K, sp))
    sec, _ = time_launches(torch, stream, fn, n, warmup, reps)
    # the two-pass form (weights converted into a workspace, then the dense GEMM)
    import ctypes
    ws_bytes = int(lib.gemm_w4a16_ws_workspace_bytes(w.N, w.K))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    fn2 = lambda i: check(lib.gemm_w4a16_ws(sets[i][0].data_ptr(), sets[i][1].data_ptr(),
                                            sets[i][2].data_ptr(), scale2, cs[i].data_ptr(),
                                            ws.data_ptr(), ctypes.c_size_t(ws_bytes),
                                            w.M, w.N, w.K, sp))
    sec2, _ = time_launches(torch, stream, fn2, n, warmup, reps)
    # the same weights in the transposed layout (codes [K/2][ldb], scales
    # [K/16][ldb], ldb = N rounded up to 128)
    ldb = -(-w.N // 128) * 128
    bt_h = np.zeros((w.K // 2, ldb), dtype=np.uint8)
    st_h = np.zeros((w.K // 16, ldb), dtype=np.uint8)
    bt_h[:, :w.N] = b_h.T
    st_h[:, :w.N] = sfb_h.T
    bt0, st0 = up(bt_h), up(st_h)
    tsets = [(sets[0][0], bt0, st0)] + [(sets[i][0], bt0.clone(), st0.clone()) for i in range(1, n)]
    fn3 = lambda i: check(lib.gemm_w4a16_t(tsets[i][0].data_ptr(), tsets[i][1].data_ptr(),
                                           tsets[i][2].data_ptr(), scale2, cs[i].data_ptr(),
                                           w.M, w.N, w.K, ldb, sp))
    sec3, _ = time_launches(torch, stream, fn3, n, warmup, reps)
    tf = 2.0 * w.M * w.N * w.K / sec / 1e12
    del sets, tsets, cs, ws
    return {"shape": name, "M": w.M, "N": w.N, "K": w.K, "us": sec * 1e6, "TFLOP/s": tf,
            "frac_bf16_peak": tf / bf16_peak,
            "weight_bytes": int(b_h.size + sfb_h.size),
            "two_pass_us": sec2 * 1e6,
            "transposed_layout_us": sec3 * 1e6}


def measure_nvfp4_decode(torch, lib, synth, up, stream, dev, pk, warmup, reps, check, fp4_peak,
                         name):
    """NVFP4 at decode-like M = 128 with split-K (FP32 partials + ordered reduce).
    Weight-bandwidth bound: reported against HBM as well as the FP4 peak."""
    sp = stream.cuda_stream
    w, k_splits = synth.NVFP4_DECODE[name]
    a_h, b_h, sfa_h, sfb_h = synth.nvfp4_inputs(w)
    ws_bytes = lib.gemm_nvfp4_bs_splitk_workspace_bytes(w.M, w.N, w.K, k_splits)
    set_bytes = a_h.size + b_h.size + sfa_h.size + sfb_h.size + w.M * w.N * 2
    n = n_sets_for(set_bytes)
    a0, b0, sa0, sb0 = up(a_h), up(b_h), up(sfa_h), up(sfb_h)
    sets = [(a0, b0, sa0, sb0)] + [(a0.clone(), b0.clone(), sa0.clone(), sb0.clone())
                                   for _ in range(n - 1)]
    cs = [torch.empty((1, w.M, w.N), dtype=torch.float16, device=dev) for _ in range(n)]
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    fn = lambda i: check(lib.gemm_nvfp4_bs_splitk(
        sets[i][0].data_ptr(), sets[i][1].data_ptr(), sets[i][2].data_ptr(), sets[i][3].data_ptr(),
        cs[i].data_ptr(), ws.data_ptr(), ws_bytes, 1, w.M, w.N, w.K, k_splits, sp))
    sec, _ = time_launches(torch, stream, fn, n, warmup, reps)
    # the same calls replayed from one CUDA graph, the way a decode loop runs
    # them (the launch gaps of the host are gone; the kernels and their
    # programmatic dependent launches are the same)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(reps):
            fn(i % n)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        graph.replay()
        stream.synchronize()
        g0.record(stream)
        graph.replay()
        g1.record(stream)
    g1.synchronize()
    gsec = g0.elapsed_time(g1) / 1e3 / reps
    del graph
    tf = 2.0 * w.M * w.N * w.K / sec / 1e12
    gbs = set_bytes / sec / 1e9
    res = {"shape": name, "L": 1, "M": w.M, "N": w.N, "K": w.K, "k_splits": k_splits,
           "us": sec * 1e6, "TFLOP/s": tf, "frac_fp4_peak": tf / fp4_peak,
           "GB/s": gbs, "frac_hbm_peak": gbs / pk["hbm_gbs"],
           "graph_us": gsec * 1e6, "graph_frac_hbm_peak": set_bytes / gsec / 1e9 / pk["hbm_gbs"],
           "bytes": int(set_bytes), "note": "operands + scales + fp16 output; split-K workspace "
           "traffic (L2-resident) not counted"}
    del sets, cs, ws
    return res


if __name__ == "__main__":
    main()
