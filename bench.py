#!/usr/bin/env python3
"""Benchmark of the chunkwise Gated DeltaNet forward (and the decode step).

One step = one ldn_chunk_fwd over the workload
gdn_bf16_b4_t2048_h16_d128 (B=4, T=2048, H=16, dk=dv=128, chunk 64, bf16
q/k/v/out, fp32 beta/gates/state), inputs resident in HBM.  L2 is flushed
(a 512 MiB device write, then a 512 MiB read of another buffer, so no dirty
lines are left to write back) before every timed launch; each launch is timed with
CUDA events on the stream it runs on.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference this method
has) on the host cores over a bounded sample of the same workload.
Under torchrun each rank runs the same per-GPU workload (independent
sequences: weak scaling) and the max time over ranks is reported.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s chunkwise GDN fwd (H=16,dk=dv=128) + % roofline; decode GB/s"
WORKLOAD = "gdn_bf16_b4_t2048_h16_d128"
EXTRA_WORKLOADS = ("kda_bf16_b8_t4096_h16_d128", "gdn_bf16_long_b1_t8192_h16_d128",
                   "gdn_bf16_long_b1_t32768_h16_d128", "gdn_bf16_long_b1_t65536_h16_d128",
                   "deltanet_fp32_b1_t256_h1_d64", "gdn2_bf16_b8_t4096_h16_d128")
PROLOGUE_WORKLOADS = ("gdn_prologue_bf16_b4_t2048_h16_d128_w4", "kda_prologue_bf16_b8_t4096_h16_d128_w4")
RLA_WORKLOADS = ("rla_bf16_b4_t2048_h16_d128", "rdn_bf16_b4_t2048_h16_d128")
BACKWARD_WORKLOADS = ("gdn_bf16_b4_t2048_h16_d128", "kda_bf16_b8_t4096_h16_d128")
DECODE_WORKLOADS = ("gdn_decode_b64_h16_dk128_dv128_steps1000", "gdn_decode_b64_h16_dk64_dv128_steps1000",
                    "gdn2_decode_b64_h16_dk128_dv128_steps1000")
FLUSH_BYTES = 512 << 20          # > 129 MB L2
FALLBACK_HBM_GBS = 6800.0
MODE_NAME = {0: "deltanet", 1: "gdn", 2: "kda", 3: "gdn2"}
KERNEL_NAME = {2: "tcgen05", 3: "split", 4: "pair", 5: "presolved"}   # LDN_VARIANT_* -> kernel family in the JSON line
TWO_LAUNCH = (3, 5)   # variants that make two launches per call (split, pre-solved)


def noalloc_pieces(B, T, H, dv, chosen):
    """Pieces a call with S_final through the library's 256 MiB array is cut into (groups
    of whole sequences, or runs of chunks of one sequence), as the C header states for the
    no-allocation entry and Gated DeltaNet-2."""
    cap = 256 << 20
    unit = 32768 + (dv // 64) * 16384 + 16896 if chosen == 3 else 16384
    nch = (T + 63) // 64
    per_seq = H * nch * unit
    if per_seq <= cap:
        nb = min(B, cap // per_seq)
        return (B + nb - 1) // nb
    tpc = cap // (H * unit)   # runs of chunks (S_final given: the state is carried in it)
    return B * ((nch + tpc - 1) // tpc)


def chunk_launches(chosen, B, T, H, dk, dv, mode, dt, ws_bytes):
    """Kernel launches of one chunkwise forward call: the split variant makes four when it
    cuts long sequences into segments (maps, scan, outputs after the preparation)."""
    import gated_delta_rule_chunkwise_gb300 as ldn
    if chosen == 3 and ldn.ldn_chunk_fwd_split_segments(B, T, H, dk, dv, 64, mode, dt, ws_bytes) >= 3:
        return 4
    return 2 if chosen in TWO_LAUNCH else 1
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------
# algorithmic work
def chunk_bytes(B, T, H, dk, dv, el_bytes, mode, s0, s_final):
    """Bytes a chunk forward must move at least: q, k, v read, o written,
    beta and gate read (fp32; Gated DeltaNet-2: erase, write and gate), initial /
    final state (fp32)."""
    n = B * T * H
    gates = {0: 4, 1: 8, 2: 4 + 4 * dk, 3: 8 * dk + 4 * dv}[mode]
    b = n * (el_bytes * (2 * dk + 2 * dv) + gates)
    st = B * H * dk * dv * 4
    return b + (st if s0 else 0) + (st if s_final else 0)


def chunk_flops(B, T, H, dk, dv, C=64):
    """Algorithmic flops of the chunk form per token-head, causal halves counted
    once: 6 dk dv (state read/write products) + C (3 dk + 2 dv) + C^2 / 3."""
    return B * T * H * (6 * dk * dv + C * (3 * dk + 2 * dv) + C * C / 3)


def el_bytes_of(dtype):
    return 2 if dtype == "bf16" else 4


def prologue_bytes(B, T, H, dk, dv, el_bytes, mode, width):
    """Algorithmic bytes of ldn_prologue: q, k, v read and written once, beta logit
    and beta, the gate input and output, the convolution weights."""
    n = B * T * H
    qkv = 2 * n * (2 * dk + dv) * el_bytes
    gate = 0 if mode == 0 else 2 * n * 4 * (dk if mode == 2 else 1)
    return qkv + 2 * n * 4 + gate + 4 * H * (2 * dk + dv) * width


def rmsnorm_bytes(B, T, H, dv, el_bytes):
    """Algorithmic bytes of ldn_rmsnorm_gated: o and the gate read, y written."""
    return 3 * B * T * H * dv * el_bytes + 4 * dv


def backward_bytes(B, T, H, dk, dv, el_bytes, mode):
    """Bytes ldn_backward must move at least: q, k, v and dout read (el_bytes),
    beta and gate read, dq, dk, dv, dbeta and dgate written (fp32), dS_final read
    and dS0 written (fp32)."""
    n = B * T * H
    gw = {0: 0, 1: 1, 2: dk}[mode]
    per = el_bytes * (2 * dk + 2 * dv) + 4 * (1 + gw) + 4 * (2 * dk + dv + 1 + gw)
    return n * per + 2 * B * H * dk * dv * 4


def rla_bytes(B, T, H, dk, dv, el_bytes):
    """Bytes ldn_rla_fwd must move at least: q, k, v read and o written (el_bytes),
    beta, gamma and the gate read (fp32), both final states written (fp32)."""
    return B * T * H * (el_bytes * (2 * dk + 2 * dv) + 12) + 2 * B * H * dk * dv * 4


def decode_bytes(B, H, dk, dv, mode):
    """State read and written, q, k, v, out (fp32) and the gates of one step."""
    gates = {0: 4, 1: 8, 2: 4 + 4 * dk, 3: 8 * dk + 4 * dv}[mode]
    return B * H * (2 * dk * dv * 4 + 2 * dk * 4 + 2 * dv * 4 + gates)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gated_delta_rule_chunkwise_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key, src_hash):
    """dram bytes per launch from a committed ncu summary, only if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("source_hash") == src_hash:
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            self.out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(self.out)):
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                smax.append(float(row[2]))
            except ValueError:
                continue
            for nm, val in zip(names, row[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# multi-rank host logic (one process per GPU; no data-path collective)
L2_NOTE = ("GPU arm: flushed before every timed launch (512 MiB write, then 512 MiB read of another buffer: "
           "cold and clean); CPU oracle arm: not applicable")


def run_config(w, workload, world):
    """The workload's `config` object, the same keys and values in both arms."""
    return {"workload": workload, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv, "chunk": 64,
            "mode": MODE_NAME[w.mode], "l2": L2_NOTE,
            "parallelism": f"replica x{world} (independent sequences per GPU)"}


def rank_seed(rank: int) -> int:
    """Each rank draws its own independent sequences: the workload is sharded
    by batch (weak scaling), rank r uses seed r."""
    return int(rank)


def reduce_max(x: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (the timed region is as slow as
    the slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
def run_reference(args):
    """fp64 CPU oracle, timed on this host's cores over a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from gated_delta_rule_chunkwise_gb300 import workloads as wl
    w = wl.make_chunk(args.workload)
    threads = oracle.default_threads()
    # calibrate one (b, h) chain, then size the per-step sample to ~1.5 s of wall time
    t0 = time.perf_counter()
    oracle.fwd(w.q[:1, :, :1], w.k[:1, :, :1], w.v[:1, :, :1], w.beta[:1, :, :1],
               None if w.gate is None else w.gate[:1, :, :1], None, mode=w.mode, nthreads=1)
    t1 = time.perf_counter() - t0
    units = int(max(1, min(w.B * w.H, round(1.5 * threads / max(t1, 1e-6)))))
    nb = max(1, min(w.B, units // w.H)) if units >= w.H else 1
    nh = w.H if units >= w.H else units
    sub = lambda a: None if a is None else np.ascontiguousarray(a[:nb, :, :nh])
    q, k, v, beta, gate = sub(w.q), sub(w.k), sub(w.v), sub(w.beta), sub(w.gate)
    used = threads
    for _ in range(args.warmup):
        oracle.fwd(q, k, v, beta, gate, None, mode=w.mode, want_state=True)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _, _, used = oracle.fwd(q, k, v, beta, gate, None, mode=w.mode, want_state=True, return_threads=True)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    tokens = nb * w.T * nh              # token-heads of the sample, expressed per H heads below
    value = (nb * w.T) * (nh / w.H) / (ms / 1e3)
    sample = (f"{nb} of {w.B} sequences x {nh} of {w.H} heads x T={w.T} per step "
              f"({tokens} token-heads; tokens/s scaled to H={w.H} heads)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded recipe, no dataset)",
            "config": run_config(w, args.workload, int(os.environ.get("WORLD_SIZE", "1"))),
            "kernel": "fp64 CPU oracle (token-by-token recurrence)",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def parity_record(got, ref, bf16, tol):
    """Both forms of the parity metric on one tensor: plain max|gpu - oracle| /
    RMS(oracle), and (bf16-stored results) the error in excess of the 2^-8 |oracle|
    storage rounding, with the count of elements that are within tol only
    through that allowance."""
    import numpy as np
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = max(float(np.sqrt(np.mean(ref * ref))), 1e-30)
    err = np.abs(got - ref)
    exc = np.maximum(err - (2.0 ** -8 if bf16 else 0.0) * np.abs(ref), 0.0)
    return {"plain": float(err.max()) / rms, "excess_over_bf16_rounding": float(exc.max()) / rms,
            "n_within_tol_only_through_allowance": int(np.count_nonzero((err > tol * rms) & (exc <= tol * rms))),
            "n_elements": int(ref.size), "tol": tol}


def cpu_baseline(w, out=None, S_final=None):
    """The oracle as it stands, on this host's cores, over ~10-20 s of work.
    Given the GPU's output and final state for the same workload, also returns
    their parity against the oracle's result on the same sample (both forms of
    the metric), else None."""
    import numpy as np
    import oracle
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.fwd(w.q[:1, :, :1], w.k[:1, :, :1], w.v[:1, :, :1], w.beta[:1, :, :1],
               None if w.gate is None else w.gate[:1, :, :1], None, mode=w.mode, nthreads=1)
    t1 = time.perf_counter() - t0
    units = int(max(1, min(w.B * w.H, round(12.0 * threads / max(t1, 1e-6)))))
    nb = max(1, min(w.B, units // w.H)) if units >= w.H else 1
    nh = w.H if units >= w.H else units
    sub = lambda a: None if a is None else np.ascontiguousarray(a[:nb, :, :nh])
    t0 = time.perf_counter()
    ro, rs, used = oracle.fwd(sub(w.q), sub(w.k), sub(w.v), sub(w.beta), sub(w.gate),
                              None if w.S0 is None else np.ascontiguousarray(w.S0[:nb, :nh]), mode=w.mode,
                              return_threads=True)
    dt = time.perf_counter() - t0
    value = (nb * w.T) * (nh / w.H) / dt
    sample = f"{nb} of {w.B} sequences x {nh} of {w.H} heads x T={w.T}"
    base = {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"{sample} ({nb * nh * w.T} token-heads, {dt:.1f} s wall); tokens/s scaled to H={w.H} heads"}
    par = None
    if out is not None:
        tol = 2e-2 if w.dtype == "bf16" else 1e-4
        par = {"sample": f"{sample}: the timed launch's output and final state against the oracle's",
               "output": parity_record(out[:nb, :, :nh], ro, w.dtype == "bf16", tol),
               "final_state": parity_record(S_final[:nb, :nh], rs, False, tol)}
    return base, par


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    from gated_delta_rule_chunkwise_gb300 import build as ldn_build
    ldn_build.build()
    import gated_delta_rule_chunkwise_gb300 as ldn
    from gated_delta_rule_chunkwise_gb300 import workloads as wl

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x):
        return reduce_max(x, world, "cuda")

    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush_l2():
        """Write 512 MiB (evicts everything), then read another 512 MiB (the
        dirty lines of the write are written back now, not inside the next
        timed launch): the timed kernel starts with a cold, clean L2."""
        flush_w.zero_()
        flush_r.sum()

    # ---------------- chunk forward (the headline) ----------------
    w = wl.make_chunk(args.workload, seed=rank_seed(rank))
    t = w.torch_inputs("cuda")
    el = 2 if w.dtype == "bf16" else 4
    dtype_code = ldn.LDN_BF16 if w.dtype == "bf16" else ldn.LDN_F32
    out = torch.empty((w.B, w.T, w.H, w.dv), dtype=t["q"].dtype, device="cuda")
    S_final = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    P = lambda x: 0 if x is None else x.data_ptr()
    args_ptrs = (P(t["q"]), P(t["k"]), P(t["v"]), P(t["beta"]), P(t["gate"]), P(t["S0"]), P(out), P(S_final))
    # workspace of the split variant (allocated by torch; the library allocates nothing)
    ws_bytes = ldn.ldn_chunk_fwd_workspace_size(w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, dtype_code)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    chosen = args.variant if args.variant != ldn.LDN_VARIANT_AUTO else \
        ldn.ldn_chunk_fwd_select_ws(w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, dtype_code, ws_bytes)

    def step():
        st = ldn.ldn_chunk_fwd_ws(*args_ptrs, w.B, w.T, w.H, w.dk, w.dv, 64, w.mode, dtype_code,
                                  args.variant, ws.data_ptr(), ws_bytes, sh)
        if st != ldn.LDN_OK:
            raise ldn.LdnError(st, "ldn_chunk_fwd_ws")

    for _ in range(max(3, args.warmup)):
        flush_l2()
        step()
    if ldn.device_status() != ldn.LDN_OK:
        raise RuntimeError("device status not ok after warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    wall0 = time.perf_counter()
    for e0, e1 in evs:
        flush_l2()
        e0.record(stream)
        step()
        e1.record(stream)
    barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    per_call = chunk_launches(chosen, w.B, w.T, w.H, w.dk, w.dv, w.mode, dtype_code, ws_bytes)
    launches = args.steps * per_call
    if ldn.device_status() != ldn.LDN_OK:
        raise RuntimeError("device status not ok after the timed region")
    per = [e0.elapsed_time(e1) for e0, e1 in evs]
    ms = max_over_ranks(statistics.mean(per))
    # the timed launches' result, kept for the parity record of the CPU-baseline leg
    keep = rank == 0 and world == 1 and not args.no_cpu_baseline
    head_out = out.float().cpu().numpy() if keep else None
    head_sf = S_final.cpu().numpy() if keep else None
    tokens = w.B * w.T
    value = world * tokens / (ms / 1e3)
    nbytes = chunk_bytes(w.B, w.T, w.H, w.dk, w.dv, el, w.mode, False, True)
    flops = chunk_flops(w.B, w.T, w.H, w.dk, w.dv)
    achieved_gbs = nbytes / (ms / 1e3) / 1e9
    from_variant = KERNEL_NAME.get(chosen, "simt")
    src = {"tcgen05": ["chunk_tc.cu"], "pair": ["chunk_tc.cu"], "presolved": ["chunk_tc.cu"],
           "split": ["chunk_tc.cu", "chunk_state.cu"]}.get(from_variant, ["chunk_simt.cu"])
    kernel_key = f"chunk_{from_variant}:{args.workload}"
    src_hash = kernel_source_hash(src)
    traffic = recorded_traffic(kernel_key, src_hash)
    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved_gbs / hbm_peak, "traffic": traffic,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback",
                "algorithmic_bytes_per_launch": nbytes, "kernel": f"chunk_{from_variant}",
                "tensor": {"achieved_tflops": flops / (ms / 1e3) / 1e12, "peak_tflops": bf16_peak,
                           "frac": flops / (ms / 1e3) / 1e12 / bf16_peak, "algorithmic_flops_per_launch": flops},
                "roofline_time_us": 1e6 * max(nbytes / (hbm_peak * 1e9), flops / (bf16_peak * 1e12)),
                "frac_of_roofline_time": 1e6 * max(nbytes / (hbm_peak * 1e9), flops / (bf16_peak * 1e12)) / (ms * 1e3)}

    # ---------------- end to end through the public API, host buffers ----------------
    # Every step copies its inputs from pinned host memory and reads its output and
    # final state back.  As a serving loop would, the steps are pipelined: the inputs
    # of step i + 1 go up (copy stream) and the results of step i come down (a second
    # copy stream) while step i computes, on two sets of device tensors.
    e2e = None
    if not args.no_e2e:
        names = [k_ for k_, v_ in t.items() if v_ is not None]
        host = {k_: t[k_].cpu().pin_memory() for k_ in names}
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        sf_h = torch.empty(S_final.shape, dtype=S_final.dtype).pin_memory()
        dev = [{k_: torch.empty_like(t[k_]) for k_ in names} for _ in range(2)]
        dout_ = [torch.empty_like(out) for _ in range(2)]
        dsf_ = [torch.empty_like(S_final) for _ in range(2)]
        h2d = sum(v_.numel() * v_.element_size() for v_ in host.values())
        d2h = out.numel() * out.element_size() + S_final.numel() * 4
        s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
        up_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        down_done = [torch.cuda.Event() for _ in range(2)]

        def e2e_run(n):
            for i in range(n):
                b_ = i & 1
                with torch.cuda.stream(s_up):
                    if i >= 2:
                        s_up.wait_event(comp_done[b_])          # step i - 2 has read these inputs
                    for k_ in names:
                        dev[b_][k_].copy_(host[k_], non_blocking=True)
                    up_done[b_].record(s_up)
                stream.wait_event(up_done[b_])
                if i >= 2:
                    stream.wait_event(down_done[b_])            # step i - 2's results are read out
                d_ = dev[b_]
                st_ = ldn.ldn_chunk_fwd_ws(P(d_["q"]), P(d_["k"]), P(d_["v"]), P(d_["beta"]), P(d_.get("gate")),
                                           P(d_.get("S0")), P(dout_[b_]), P(dsf_[b_]), w.B, w.T, w.H, w.dk, w.dv,
                                           64, w.mode, dtype_code, args.variant, ws.data_ptr(), ws_bytes, sh)
                if st_ != ldn.LDN_OK:
                    raise ldn.LdnError(st_, "ldn_chunk_fwd_ws")
                comp_done[b_].record(stream)
                with torch.cuda.stream(s_down):
                    s_down.wait_event(comp_done[b_])
                    out_h.copy_(dout_[b_], non_blocking=True)
                    sf_h.copy_(dsf_[b_], non_blocking=True)
                    down_done[b_].record(s_down)

        e2e_run(max(3, args.warmup))
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_up)
        e2e_run(args.steps)
        s_down.wait_stream(stream)
        e1.record(s_down)
        torch.cuda.synchronize()
        barrier()
        launches += args.steps * per_call
        ems = max_over_ranks(e0.elapsed_time(e1) / args.steps)
        e2e = {"value": world * tokens / (ems / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems,
               "overlap": "pipelined: step i+1 uploads and step i downloads on two copy streams while step i "
                          "computes (two sets of device tensors)"}
        del host, out_h, sf_h, dev, dout_, dsf_

    # ---------------- the other chunkwise workloads (secondary lines) ----------------
    others = None
    if not args.no_extra:
        others = {}
        for name in EXTRA_WORKLOADS:
            ow = wl.make_chunk(name, seed=rank)
            ot = ow.torch_inputs("cuda")
            oel = 2 if ow.dtype == "bf16" else 4
            oout = torch.empty((ow.B, ow.T, ow.H, ow.dv), dtype=ot["q"].dtype, device="cuda")
            osf = torch.empty((ow.B, ow.H, ow.dk, ow.dv), dtype=torch.float32, device="cuda")
            optr = (P(ot["q"]), P(ot["k"]), P(ot["v"]), P(ot["beta"]), P(ot["gate"]), P(ot["S0"]), P(oout), P(osf))
            odt = ldn.LDN_BF16 if ow.dtype == "bf16" else ldn.LDN_F32
            g2 = ow.mode == wl.MODE_GDN2

            ows_bytes = 0 if g2 else ldn.ldn_chunk_fwd_workspace_size(ow.B, ow.T, ow.H, ow.dk, ow.dv, 64, ow.mode, odt)
            ows = torch.empty(max(ows_bytes, 256), dtype=torch.uint8, device="cuda")
            ochosen = ldn.ldn_chunk_fwd_select_ws(ow.B, ow.T, ow.H, ow.dk, ow.dv, 64, ow.mode, odt,
                                                  (1 << 64) - 1 if g2 else ows_bytes)

            def ostep():
                if g2:
                    st_ = ldn.ldn_chunk_fwd_gdn2(optr[0], optr[1], optr[2], P(ot["erase"]), P(ot["write"]), optr[4],
                                                 optr[5], optr[6], optr[7], ow.B, ow.T, ow.H, ow.dk, ow.dv, 64, odt,
                                                 ldn.LDN_VARIANT_AUTO, sh)
                else:
                    st_ = ldn.ldn_chunk_fwd_ws(*optr, ow.B, ow.T, ow.H, ow.dk, ow.dv, 64, ow.mode, odt,
                                               ldn.LDN_VARIANT_AUTO, ows.data_ptr(), ows_bytes, sh)
                if st_ != ldn.LDN_OK:
                    raise ldn.LdnError(st_, "ldn_chunk_fwd_gdn2" if g2 else "ldn_chunk_fwd_ws")

            ostep()
            oev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
            for e0, e1 in oev:
                flush_l2()
                e0.record(stream)
                ostep()
                e1.record(stream)
            barrier()
            onl = ((2 * noalloc_pieces(ow.B, ow.T, ow.H, ow.dv, ochosen) if ochosen in TWO_LAUNCH else 1) if g2
                   else chunk_launches(ochosen, ow.B, ow.T, ow.H, ow.dk, ow.dv, ow.mode, odt, ows_bytes))
            launches += 4 * onl
            oms = max_over_ranks(statistics.mean(e0.elapsed_time(e1) for e0, e1 in oev))
            ob = chunk_bytes(ow.B, ow.T, ow.H, ow.dk, ow.dv, oel, ow.mode, ow.S0 is not None, True)
            kern = KERNEL_NAME.get(ochosen, "simt")
            osrc = {"tcgen05": ["chunk_tc.cu"], "pair": ["chunk_tc.cu"], "presolved": ["chunk_tc.cu"],
                    "split": ["chunk_tc.cu", "chunk_state.cu"]}.get(kern, ["chunk_simt.cu"])
            otraffic = recorded_traffic(f"chunk_{kern}:{name}", kernel_source_hash(osrc))
            others[name] = {"tokens_per_s": world * ow.B * ow.T / (oms / 1e3), "ms_per_launch": oms,
                            "kernel": f"chunk_{kern}", "launches_per_call": onl, "algorithmic_bytes": ob,
                            "hbm_frac": ob / (oms / 1e3) / 1e9 / hbm_peak, "traffic": otraffic,
                            "traffic_over_algorithmic": None if otraffic is None else otraffic / ob}
            del ot, oout, osf, ows
        if ldn.device_status() != ldn.LDN_OK:
            raise RuntimeError("other workloads: device status not ok")

    # ---------------- prologue and epilogue around the path (bandwidth) ----------------
    around = None
    if not args.no_extra:
        around = {}
        for name in PROLOGUE_WORKLOADS:
            p = wl.make_prologue(name, seed=rank)
            el = torch.bfloat16 if p["dtype"] == "bf16" else torch.float32
            dev = lambda x, dt=torch.float32: None if x is None else torch.from_numpy(x).to("cuda", dt)
            pi = {k_: dev(p[k_], el) for k_ in ("q_in", "k_in", "v_in", "o", "g")}
            pf = {k_: dev(p[k_]) for k_ in ("conv_q", "conv_k", "conv_v", "beta_logit", "gate_z", "gate_a", "gate_b", "gain")}
            B_, T_, H_, dk_, dv_ = p["B"], p["T"], p["H"], p["dk"], p["dv"]
            qo = torch.empty((B_, T_, H_, dk_), dtype=el, device="cuda")
            ko, vo = torch.empty_like(qo), torch.empty((B_, T_, H_, dv_), dtype=el, device="cuda")
            bo = torch.empty((B_, T_, H_), dtype=torch.float32, device="cuda")
            go_ = torch.empty(tuple(p["gate_z"].shape), dtype=torch.float32, device="cuda")
            yo = torch.empty_like(pi["o"])
            dt_ = ldn.LDN_BF16 if p["dtype"] == "bf16" else ldn.LDN_F32
            P_ = lambda x: 0 if x is None else x.data_ptr()

            def pro():
                st_ = ldn.ldn_prologue(P_(pi["q_in"]), P_(pi["k_in"]), P_(pi["v_in"]), P_(pf["conv_q"]),
                                       P_(pf["conv_k"]), P_(pf["conv_v"]), p["width"], P_(pf["beta_logit"]),
                                       P_(pf["gate_z"]), P_(pf["gate_a"]), P_(pf["gate_b"]), P_(qo), P_(ko), P_(vo),
                                       P_(bo), P_(go_), B_, T_, H_, dk_, dv_, p["mode"], dt_, 1e-6, sh)
                if st_ != ldn.LDN_OK:
                    raise ldn.LdnError(st_, "ldn_prologue")

            def epi():
                st_ = ldn.ldn_rmsnorm_gated(P_(pi["o"]), P_(pi["g"]), P_(pf["gain"]), P_(yo), B_, T_, H_, dv_, dt_,
                                            1e-6, sh)
                if st_ != ldn.LDN_OK:
                    raise ldn.LdnError(st_, "ldn_rmsnorm_gated")

            res = {}
            for what, fn, nb_, nl in (("prologue", pro, prologue_bytes(B_, T_, H_, dk_, dv_, el_bytes_of(p["dtype"]),
                                                                       p["mode"], p["width"]),
                                                                       (1 if dk_ == dv_ else 2) + (p["mode"] == 2)),
                                      ("rmsnorm_gated", epi, rmsnorm_bytes(B_, T_, H_, dv_, el_bytes_of(p["dtype"])), 1)):
                for _ in range(3):
                    fn()
                barrier()
                evs_ = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
                for e0, e1 in evs_:
                    flush_l2()
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                barrier()
                ms_ = max_over_ranks(statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs_))
                launches += nl * (3 + len(evs_))
                res[what] = {"us_per_call": ms_ * 1e3, "algorithmic_bytes": nb_, "GB/s": nb_ / (ms_ / 1e3) / 1e9,
                             "frac_hbm": nb_ / (ms_ / 1e3) / 1e9 / hbm_peak, "launches_per_call": nl}
            around[name] = res
            del pi, pf, qo, ko, vo, bo, go_, yo
        if ldn.device_status() != ldn.LDN_OK:
            raise RuntimeError("prologue / epilogue: device status not ok")

    # ---------------- backward (gradients of the forward) ----------------
    backward = None
    if not args.no_extra:
        backward = {}
        for name in BACKWARD_WORKLOADS:
            bw = wl.make_chunk(name, seed=rank)
            bt = bw.torch_inputs("cuda")
            dout_np, dsf_np = wl.make_upstream(bw, seed=rank + 1)
            bdo = torch.from_numpy(dout_np).to("cuda", bt["q"].dtype)
            bdsf = torch.from_numpy(dsf_np).cuda()
            f32 = dict(dtype=torch.float32, device="cuda")
            B_, T_, H_, dk_, dv_ = bw.B, bw.T, bw.H, bw.dk, bw.dv
            gq, gk = torch.empty((B_, T_, H_, dk_), **f32), torch.empty((B_, T_, H_, dk_), **f32)
            gv, gb = torch.empty((B_, T_, H_, dv_), **f32), torch.empty((B_, T_, H_), **f32)
            gg = torch.empty(tuple(bt["gate"].shape), **f32)
            gs0 = torch.empty((B_, H_, dk_, dv_), **f32)
            bdt = ldn.LDN_BF16 if bw.dtype == "bf16" else ldn.LDN_F32
            need = ldn.ldn_backward_workspace_size(B_, T_, H_, dk_, dv_, bw.mode, bdt)
            bws = torch.empty(need, dtype=torch.uint8, device="cuda")
            chunked = bdt == ldn.LDN_BF16 and dk_ == 128 and dv_ == 128 and bw.mode in (0, 1)

            def bstep():
                st_ = ldn.ldn_backward(P(bt["q"]), P(bt["k"]), P(bt["v"]), P(bt["beta"]), P(bt["gate"]), P(bt["S0"]),
                                       P(bdo), P(bdsf), P(gq), P(gk), P(gv), P(gb), P(gg), P(gs0), B_, T_, H_, dk_,
                                       dv_, bw.mode, bdt, bws.data_ptr(), need, sh)
                if st_ != ldn.LDN_OK:
                    raise ldn.LdnError(st_, "ldn_backward")

            bstep()
            bev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
            for e0, e1 in bev:
                flush_l2()
                e0.record(stream)
                bstep()
                e1.record(stream)
            barrier()
            launches += (5 if chunked else 3) * (1 + len(bev))
            bms = max_over_ranks(statistics.mean(e0.elapsed_time(e1) for e0, e1 in bev))
            bb = backward_bytes(B_, T_, H_, dk_, dv_, el_bytes_of(bw.dtype), bw.mode)
            kernels = ("chunk_tc_kernel<prep-X> + chunk_tc_kernel<fed> (forward with chunk states) + "
                       "bwd_prep_kernel + bwd_chain_kernel + bwd_chunk_kernel" if chunked else
                       "bwd_kernel<phase 1> + bwd_kernel<phase 2> + bwd_reduce_kernel")
            backward[name] = {"ms_per_call": bms, "tokens_per_s": world * B_ * T_ / (bms / 1e3),
                              "form": "chunkwise" if chunked else "recurrent", "kernels": kernels,
                              "algorithmic_bytes": bb, "hbm_frac": bb / (bms / 1e3) / 1e9 / hbm_peak,
                              "workspace_bytes": need}
            del bt, bdo, bdsf, gq, gk, gv, gb, gg, gs0, bws
        if ldn.device_status() != ldn.LDN_OK:
            raise RuntimeError("backward: device status not ok")

    # ---------------- Residual Linear Attention / Residual DeltaNet ----------------
    rla = None
    if not args.no_extra:
        rla = {}
        for name in RLA_WORKLOADS:
            rp = wl.make_rla(name, seed=rank)
            rel = torch.bfloat16 if rp["dtype"] == "bf16" else torch.float32
            rd = lambda a, dt=torch.float32: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dt)
            rq, rk, rv = rd(rp["q"], rel), rd(rp["k"], rel), rd(rp["v"], rel)
            rb, rgm, rgt = rd(rp["beta"]), rd(rp["gamma"]), rd(rp["gate"])
            B_, T_, H_, dk_, dv_ = rp["B"], rp["T"], rp["H"], rp["dk"], rp["dv"]
            rout = torch.empty((B_, T_, H_, dv_), dtype=rel, device="cuda")
            rsf = torch.empty((B_, H_, dk_, dv_), dtype=torch.float32, device="cuda")
            rrf = torch.empty_like(rsf)
            rdt = ldn.LDN_BF16 if rp["dtype"] == "bf16" else ldn.LDN_F32
            rneed = ldn.ldn_rla_fwd_workspace_size(B_, T_, H_, dk_, dv_, int(rp["delta"]), rdt)
            rws = torch.empty(max(rneed, 1), dtype=torch.uint8, device="cuda")
            rchunk = rdt == ldn.LDN_BF16 and dk_ == 128 and dv_ == 128

            def rstep():
                st_ = ldn.ldn_rla_fwd_ws(P(rq), P(rk), P(rv), P(rb), P(rgm), P(rgt), rp["clip"], 0, 0, P(rout),
                                         P(rsf), P(rrf), B_, T_, H_, dk_, dv_, int(rp["delta"]), rdt,
                                         rws.data_ptr() if rneed else 0, rneed, sh)
                if st_ != ldn.LDN_OK:
                    raise ldn.LdnError(st_, "ldn_rla_fwd_ws")

            rstep()
            rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
            for e0, e1 in rev:
                flush_l2()
                e0.record(stream)
                rstep()
                e1.record(stream)
            barrier()
            nrl = (3 if rp["delta"] else 1) if rchunk else 1
            launches += nrl * (1 + len(rev))
            rms = max_over_ranks(statistics.mean(e0.elapsed_time(e1) for e0, e1 in rev))
            rbytes = rla_bytes(B_, T_, H_, dk_, dv_, el_bytes_of(rp["dtype"]))
            rkern = ("chunk_tc_kernel<prep-X> x 2 (the solves for beta and gamma) + rla_chunk_kernel<RDN>"
                     if rp["delta"] else "rla_chunk_kernel<RLA>") if rchunk else "rla_kernel (both states in one pass)"
            rla[name] = {"ms_per_call": rms, "tokens_per_s": world * B_ * T_ / (rms / 1e3),
                         "form": "chunkwise" if rchunk else "recurrent", "kernels": rkern, "workspace_bytes": rneed,
                         "algorithmic_bytes": rbytes, "hbm_frac": rbytes / (rms / 1e3) / 1e9 / hbm_peak}
            del rq, rk, rv, rb, rgm, rgt, rout, rsf, rrf, rws
        if ldn.device_status() != ldn.LDN_OK:
            raise RuntimeError("rla: device status not ok")

    # ---------------- decode step (bandwidth) ----------------
    decode = None
    if not args.no_decode:
        decode = {}
        del t, out, S_final
        for name in DECODE_WORKLOADS:
            d = wl.make_decode(name, seed=rank)
            td = d.torch_inputs("cuda")
            S = td["S0"].clone()
            o = torch.empty((d.B, d.H, d.dv), dtype=torch.float32, device="cuda")
            steps = d.T
            g2 = d.mode == wl.MODE_GDN2
            ptr = [(td["q"][i].data_ptr(), td["k"][i].data_ptr(), td["v"][i].data_ptr(),
                    td["erase"][i].data_ptr() if g2 else td["beta"][i].data_ptr(), td["gate"][i].data_ptr(),
                    td["write"][i].data_ptr() if g2 else 0) for i in range(steps)]

            def dstep(i):
                qp, kp, vp, bp, gp, wp = ptr[i]
                if g2:
                    st = ldn.ldn_decode_step_gdn2(qp, kp, vp, bp, wp, gp, S.data_ptr(), o.data_ptr(), d.B, d.H, d.dk,
                                                  d.dv, ldn.LDN_F32, sh)
                else:
                    st = ldn.ldn_decode_step(qp, kp, vp, bp, gp, S.data_ptr(), o.data_ptr(), d.B, d.H, d.dk, d.dv,
                                             d.mode, ldn.LDN_F32, sh)
                if st != ldn.LDN_OK:
                    raise ldn.LdnError(st, "ldn_decode_step")

            for i in range(5):
                dstep(i)
            S.copy_(td["S0"])
            barrier()
            cold = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for i, (e0, e1) in enumerate(cold):
                flush_l2()
                e0.record(stream)
                dstep(i)
                e1.record(stream)
            barrier()
            cold_ms = max_over_ranks(statistics.mean(e0.elapsed_time(e1) for e0, e1 in cold))
            S.copy_(td["S0"])
            barrier()
            w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            w0.record(stream)
            for i in range(steps):
                dstep(i)
            w1.record(stream)
            barrier()
            warm_ms = max_over_ranks(w0.elapsed_time(w1) / steps)
            # the same steps captured once in a CUDA graph and replayed (no host launch cost)
            cg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(cg, capture_error_mode="thread_local"):
                gsh = torch.cuda.current_stream().cuda_stream
                for i in range(steps):
                    qp, kp, vp, bp, gp, wp = ptr[i]
                    if g2:
                        st = ldn.ldn_decode_step_gdn2(qp, kp, vp, bp, wp, gp, S.data_ptr(), o.data_ptr(), d.B, d.H,
                                                      d.dk, d.dv, ldn.LDN_F32, gsh)
                    else:
                        st = ldn.ldn_decode_step(qp, kp, vp, bp, gp, S.data_ptr(), o.data_ptr(), d.B, d.H, d.dk, d.dv,
                                                 d.mode, ldn.LDN_F32, gsh)
                    if st != ldn.LDN_OK:
                        raise ldn.LdnError(st, "ldn_decode_step (capture)")
            S.copy_(td["S0"])
            cg.replay()
            S.copy_(td["S0"])
            barrier()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            cg.replay()
            g1.record(stream)
            barrier()
            graph_ms = max_over_ranks(g0.elapsed_time(g1) / steps)
            del cg
            launches += 3 * steps
            # the same steps in one ldn_decode_steps call (state read and written once per call)
            multi = None
            if not g2:
                mo = torch.empty((steps, d.B, d.H, d.dv), dtype=torch.float32, device="cuda")

                def mstep():
                    st = ldn.ldn_decode_steps(td["q"].data_ptr(), td["k"].data_ptr(), td["v"].data_ptr(),
                                              td["beta"].data_ptr(), td["gate"].data_ptr(), S.data_ptr(), mo.data_ptr(),
                                              steps, d.B, d.H, d.dk, d.dv, d.mode, ldn.LDN_F32, sh)
                    if st != ldn.LDN_OK:
                        raise ldn.LdnError(st, "ldn_decode_steps")

                S.copy_(td["S0"])
                mstep()
                mev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
                for e0, e1 in mev:
                    S.copy_(td["S0"])
                    flush_l2()
                    e0.record(stream)
                    mstep()
                    e1.record(stream)
                barrier()
                m_ms = max_over_ranks(statistics.mean(e0.elapsed_time(e1) for e0, e1 in mev))
                launches += 1 + len(mev)
                per_tok = d.B * d.H * (2 * d.dk * 4 + 2 * d.dv * 4 + {0: 4, 1: 8, 2: 4 + 4 * d.dk}[d.mode])
                mbytes = 2 * d.B * d.H * d.dk * d.dv * 4 + steps * per_tok
                multi = {"steps_per_call": steps, "ms_per_call": m_ms, "us_per_step": m_ms * 1e3 / steps,
                         "tokens_per_s": world * d.B * steps / (m_ms / 1e3), "kernels": "decode_steps_kernel",
                         "algorithmic_bytes": mbytes, "hbm_frac": mbytes / (m_ms / 1e3) / 1e9 / hbm_peak,
                         "note": "ldn_decode_steps (opt-in): all steps in one launch, the state on chip between "
                                 "steps; bound by the per-step barriers, not HBM; L2 flushed before each call"}
                del mo
            if ldn.device_status() != ldn.LDN_OK:
                raise RuntimeError("decode: device status not ok")
            db = decode_bytes(d.B, d.H, d.dk, d.dv, d.mode)
            decode[name] = {"steps": steps, "bytes_per_step": db,
                            "cold_l2": {"us_per_step": cold_ms * 1e3, "GB/s": db / (cold_ms / 1e3) / 1e9,
                                        "frac_hbm": db / (cold_ms / 1e3) / 1e9 / hbm_peak},
                            "warm_back_to_back": {"us_per_step": warm_ms * 1e3, "GB/s": db / (warm_ms / 1e3) / 1e9},
                            "cuda_graph": {"us_per_step": graph_ms * 1e3, "GB/s": db / (graph_ms / 1e3) / 1e9,
                                           "note": "all steps replayed from one captured graph, L2 not flushed"},
                            "tokens_per_s": world * d.B / (cold_ms / 1e3), "multi_step": multi}
            del td, S, o, ptr

    line = {"impl": "ours", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded numpy recipe: L2-normalised Gaussian q,k; Gaussian v; sigmoid beta; "
                    "-0.1*softplus log-decay); no dataset",
            "config": run_config(w, args.workload, world), "kernel": f"chunk_{from_variant}",
            "roofline": roofline, "e2e": e2e, "clocks": clk, "gpu_launches": launches,
            "other_workloads": others, "prologue_epilogue": around, "backward": backward, "rla": rla,
            "wall_s_timed_region": wall, "decode": decode}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = cpu_baseline(w, head_out, head_sf)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile_case(args):
    """Two untimed calls of one operation on a given shape (a small case for an
    ncu capture): gdn (ldn_chunk_fwd_ws, the variant the cost model picks, as
    the timed step runs it), backward-gdn / backward-kda (ldn_backward), gdn2
    (ldn_chunk_fwd_gdn2), kda (ldn_chunk_fwd_noalloc), rla / rdn
    (ldn_rla_fwd_ws), automatic variant, bf16, d = 128, the workload recipe of
    the named mode."""
    import numpy as np
    import torch
    import gated_delta_rule_chunkwise_gb300 as ldn
    from gated_delta_rule_chunkwise_gb300 import workloads as wl
    ldn.load()
    B, T, H = (int(x) for x in args.shape.split(","))
    if args.profile in ("rla", "rdn"):
        p = wl.make_rla(f"{args.profile}_bf16_b4_t2048_h16_d128", B=B, T=T, H=H)
        d = lambda a, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dt)
        for _ in range(2):
            ldn.rla_fwd(d(p["q"], torch.bfloat16), d(p["k"], torch.bfloat16), d(p["v"], torch.bfloat16), d(p["beta"]),
                        d(p["gamma"]), d(p["gate"]), clip=p["clip"], delta=p["delta"])
        torch.cuda.synchronize()
        st = ldn.device_status()
        print(json.dumps({"profile_case": args.profile, "shape": [B, T, H], "status": st}))
        return 0 if st == ldn.LDN_OK else 1
    name = {"backward-gdn": "gdn_bf16_b4_t2048_h16_d128", "backward-kda": "kda_bf16_b8_t4096_h16_d128",
            "gdn2": "gdn2_bf16_b8_t4096_h16_d128", "kda": "kda_bf16_b8_t4096_h16_d128",
            "gdn": "gdn_bf16_b4_t2048_h16_d128"}[args.profile]
    w = wl.make_chunk(name, B=B, T=T, H=H)
    t = w.torch_inputs("cuda")
    if args.profile == "gdn":
        out = torch.empty_like(t["v"])
        wsb = ldn.ldn_chunk_fwd_workspace_size(B, T, H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16)
        wsp = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
        var = ldn.ldn_chunk_fwd_select_ws(B, T, H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16, wsb)
        for _ in range(2):
            st = ldn.ldn_chunk_fwd_ws(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["beta"].data_ptr(),
                                      t["gate"].data_ptr(), 0, out.data_ptr(), 0, B, T, H, w.dk, w.dv, 64, w.mode,
                                      ldn.LDN_BF16, var, wsp.data_ptr(), wsb, torch.cuda.current_stream().cuda_stream)
            if st != ldn.LDN_OK:
                raise ldn.LdnError(st, "ldn_chunk_fwd_ws")
    elif args.profile.startswith("backward"):
        dout, dsf = wl.make_upstream(w)
        d = torch.from_numpy(dout).to("cuda", t["q"].dtype)
        f = torch.from_numpy(dsf).cuda()
        for _ in range(2):
            ldn.backward(t["q"], t["k"], t["v"], t["beta"], t["gate"], t["S0"], d, f, mode=w.mode)
    elif args.profile == "gdn2":
        for _ in range(2):
            ldn.chunk_fwd_gdn2(t["q"], t["k"], t["v"], t["erase"], t["write"], t["gate"], t["S0"])
    else:
        out = torch.empty_like(t["v"])
        for _ in range(2):
            st = ldn.ldn_chunk_fwd_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                                           t["beta"].data_ptr(), t["gate"].data_ptr(), 0, out.data_ptr(), 0,
                                           B, T, H, w.dk, w.dv, 64, w.mode, ldn.LDN_BF16, ldn.LDN_VARIANT_AUTO,
                                           torch.cuda.current_stream().cuda_stream)
            if st != ldn.LDN_OK:
                raise ldn.LdnError(st, "ldn_chunk_fwd_noalloc")
    torch.cuda.synchronize()
    st = ldn.device_status()
    print(json.dumps({"profile_case": args.profile, "shape": [B, T, H], "status": st}))
    return 0 if st == ldn.LDN_OK else 1


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--variant", type=int, default=0,
                    help="0 auto, 1 SIMT fp32, 2 tcgen05 fused, 3 split, 4 tcgen05 cluster pair, 5 pre-solved")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workload lines")
    ap.add_argument("--profile", choices=["gdn", "backward-gdn", "backward-kda", "gdn2", "kda", "rla", "rdn"],
                    help="run one operation twice, untimed, on --shape (a small case for ncu) and exit")
    ap.add_argument("--shape", default="1,2048,16", help="B,T,H for --profile")
    args = ap.parse_args()
    if args.profile:
        return run_profile_case(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
