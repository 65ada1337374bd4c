#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300: chunked prefill and decode step.

Prints ONE JSON line (rank 0).  The headline workload is the bf16 batch
prefill B=4, H=32, T=8192, d=128, C=64 (fp32 log-decay and beta, zero initial
state): `value` is prefill tokens/s over all ranks.  One step = one
kda_chunk_fwd call over the whole batch.  The decode workload (N=256, H=32,
d=128, fp32 state, 1000 consecutive steps) is reported beside it in
`decode` as state GB/s and sequence-steps/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the fp64 CPU oracle (the correctness reference, not a
tuned CPU implementation) on the host cores, on a bounded sample of the same
workload, and prints the same line with "impl": "reference".

Under torchrun each rank runs its own copy of the workload (independent
problems: weak scaling, no collective in the data path); the step time is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (H=32,d=128) & decode state GB/s vs roofline, 1×GB300"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_SRC = os.path.join(ROOT, "hybrid_linear_attention_chunk_gb300", "csrc", "kda_chunk_tc.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "kda_chunk_tc_prefill_B4_H32_T8192.traffic.txt")


# ------------------------------------------------------------------ helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _cudart():
    """The CUDA runtime torch loaded (found by its soname), for pitched host <-> device copies;
    None when it cannot be loaded."""
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            lib = ctypes.CDLL(name)
        except OSError:
            continue
        if hasattr(lib, "cudaMemcpy2DAsync"):
            lib.cudaMemcpy2DAsync.restype = ctypes.c_int
            return lib
    return None


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def source_sha(path: str) -> str:
    """sha256[:16] of a source file's code: line comments and blank lines are
    left out, so that a comment edit does not void a capture of the same code."""
    with open(path, "rb") as f:
        lines = f.read().decode("utf-8").splitlines()
    code = []
    for ln in lines:
        cut = ln.split("//", 1)[0].rstrip()
        if cut:
            code.append(cut)
    return hashlib.sha256("\n".join(code).encode("utf-8")).hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the prefill kernel from the committed ncu
    summary, or None when the kernel source changed since the capture."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    k, v = line.strip().split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha") != source_sha(PREFILL_SRC):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while work runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ workload sizes

def prefill_bytes(B, T, H, dk, dv, qkv_bytes=2, gate_bytes=4, out_bytes=2, state_in=False):
    tok = B * T * H
    b = tok * (2 * dk + dv) * qkv_bytes + tok * dk * gate_bytes + tok * gate_bytes + tok * dv * out_bytes
    b += B * H * dk * dv * 4 * (2 if state_in else 1)
    return b


def prefill_flops(B, T, H, d, C):
    # 6 d^2 + 10 C d per (token, head): the dense contractions of the chunk form
    return B * T * H * (6 * d * d + 10 * C * d)


def decode_bytes(N, H, dk, dv):
    nh = N * H
    return nh * dk * dv * 4 * 2 + nh * (2 * dk + dv) * 2 + nh * dk * 4 + nh * 4 + nh * dv * 2


# ------------------------------------------------------------------ GPU arm

def run_gpu(args):
    import numpy as np
    import torch
    import hybrid_linear_attention_chunk_gb300 as kda
    from hybrid_linear_attention_chunk_gb300 import inputs

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    kda.load()
    hbm_peak, tc_peak, peak_kind = load_peaks()

    w = inputs.PREFILL_B4_T8K
    x = inputs.make_prefill(w, device=dev, seed=inputs.SEED_BASE + w.seed_index + 1000 * rank)
    q, k, v, g, beta = x["q"], x["k"], x["v"], x["log_alpha"], x["beta"]
    out = torch.empty(w.B * w.T, w.H, w.dv, dtype=torch.bfloat16, device=dev)
    sT = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.kda_chunk_fwd(q, k, v, g, beta, None, None, out, sT, B=w.B, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index)
    clocks.start()
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    ms_local = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    ms = reduce_max(ms_local, world, dev)
    ms_step = ms / args.steps
    tokens = w.B * w.T
    value = world * tokens / (ms_step * 1e-3)

    # roofline of the prefill kernel (one launch per step, events on its stream)
    alg_bytes = prefill_bytes(w.B, w.T, w.H, w.dk, w.dv)
    achieved = alg_bytes / (ms_local / args.steps * 1e-3) / 1e9
    traffic = profiled_traffic()
    flops = prefill_flops(w.B, w.T, w.H, w.dk, w.chunk)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                "peak_source": f"{peak_kind} hbm_gbs",
                "kernel": "chunk_tc_kernel", "algorithmic_bytes_per_launch": alg_bytes,
                "tensor_tflops": round(flops / (ms_local / args.steps * 1e-3) / 1e12, 1),
                "tensor_frac_of_bf16_peak": round(flops / (ms_local / args.steps * 1e-3) / 1e12 / tc_peak, 4)}

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hg, hb = (t.cpu().pin_memory() for t in (q, k, v, g, beta))
        ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hs = torch.empty(sT.shape, dtype=sT.dtype).pin_memory()
        e2e_steps = max(20, min(50, args.steps // 20))  # a timed region of ~0.15 s or more

        # The batch goes through in P token ranges of every sequence: range p
        # of all B sequences is one kda_chunk_fwd call that resumes from the
        # states range p - 1 left (initial_state = final_state, in place), so
        # every call keeps all B x H chains busy.  The host-to-device copy of
        # range p + 1 and the device-to-host copy of range p - 1 overlap the
        # call for range p (three streams; events keep a buffer from being
        # refilled or read back while a call still uses it).
        P = 8 if w.T % (8 * w.chunk) == 0 else 1
        Tp = w.T // P
        pieces = [tuple(torch.empty((w.B * Tp,) + tuple(t.shape[1:]), dtype=t.dtype, device=dev)
                        for t in (q, k, v, g, beta, out)) for _ in range(P)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(P)]
        ev_done = [torch.cuda.Event() for _ in range(P)]
        ev_back = [torch.cuda.Event() for _ in range(P)]

        def rows(b, p):  # host rows of sequence b, range p; device rows of sequence b in a piece
            return slice(b * w.T + p * Tp, b * w.T + (p + 1) * Tp), slice(b * Tp, (b + 1) * Tp)

        # Range p of all B sequences is one pitched block of each host tensor (B rows of Tp
        # tokens, T tokens apart): one cudaMemcpy2DAsync per tensor and range.
        cudart = _cudart()

        def copy_range(dst, src, p, h2d, strm):
            rb = src[0].numel() * src.element_size()  # bytes per token row
            if cudart is None:
                for b in range(w.B):
                    hr, dr = rows(b, p)
                    if h2d:
                        dst[dr].copy_(src[hr], non_blocking=True)
                    else:
                        dst[hr].copy_(src[dr], non_blocking=True)
                return
            if h2d:  # host [B*T] rows -> device [B*Tp] rows
                args = (dst.data_ptr(), Tp * rb, src.data_ptr() + p * Tp * rb, w.T * rb, 1)
            else:    # device [B*Tp] rows -> host [B*T] rows
                args = (dst.data_ptr() + p * Tp * rb, w.T * rb, src.data_ptr(), Tp * rb, 2)
            rc = cudart.cudaMemcpy2DAsync(ctypes.c_void_p(args[0]), ctypes.c_size_t(args[1]),
                                          ctypes.c_void_p(args[2]), ctypes.c_size_t(args[3]),
                                          ctypes.c_size_t(Tp * rb), ctypes.c_size_t(w.B), ctypes.c_int(args[4]),
                                          ctypes.c_void_p(strm.cuda_stream))
            if rc != 0:
                raise RuntimeError(f"cudaMemcpy2DAsync failed ({rc})")

        def e2e_step(first, order_in=False):
            # Consecutive steps overlap: step i + 1's input copies follow step i's on s_in as soon
            # as each piece's previous call has read it (ev_done); only the warm-up step and the
            # first timed step order their copies after the work already on `stream`.
            if first or order_in:
                s_in.wait_stream(stream)
            for p in range(P):
                dq, dk_, dv_, dg, db, do_ = pieces[p]
                if not first:
                    s_in.wait_event(ev_done[p])  # the previous step's call has read this piece
                with torch.cuda.stream(s_in):
                    for d_, h_ in ((dq, hq), (dk_, hk), (dv_, hv), (dg, hg), (db, hb)):
                        copy_range(d_, h_, p, True, s_in)
                    ev_in[p].record(s_in)
                stream.wait_event(ev_in[p])
                if not first:
                    stream.wait_event(ev_back[p])  # the previous step's output piece is back on the host
                kda.kda_chunk_fwd(dq, dk_, dv_, dg, db, sT if p > 0 else None, None, do_, sT, B=w.B,
                                  stream=stream)
                ev_done[p].record(stream)
                s_out.wait_event(ev_done[p])
                with torch.cuda.stream(s_out):
                    copy_range(ho, do_, p, False, s_out)
                    if p == P - 1:
                        hs.copy_(sT, non_blocking=True)
                    ev_back[p].record(s_out)
            stream.wait_stream(s_out)

        e2e_step(True)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        t0 = time.perf_counter()
        ev0.record(stream)
        for i in range(e2e_steps):
            e2e_step(False, order_in=i == 0)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = reduce_max(ev0.elapsed_time(ev1), world, dev) / e2e_steps
        h2d = sum(t.numel() * t.element_size() for t in (q, k, v, g, beta))
        d2h = out.numel() * out.element_size() + sT.numel() * sT.element_size()
        # the host output of the ranged, resumed calls against the single device-path call
        e2e_diff = float((ho.float() - out.float().cpu()).abs().max())
        e2e = {"value": round(world * tokens / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps, "max_abs_diff_vs_device_path": e2e_diff,
               "api": "kda_chunk_fwd via ctypes on 8 token ranges of the batch (each resuming from the previous "
                      "range's states), pinned host buffers, one pitched copy per tensor and range ("
                      + ("cudaMemcpy2DAsync" if cudart is not None else "per-sequence copies")
                      + "), copies overlapped on two streams, consecutive steps pipelined"}
        del hq, hk, hv, hg, hb, pieces

    # decode: 1000 consecutive steps of the N=256 workload
    dw = inputs.DECODE_N256
    dsteps = args.decode_steps
    dec = None
    if dsteps > 0:
        dx = inputs.make_decode(dw, steps=dsteps, device=dev, seed=inputs.SEED_BASE + dw.seed_index + 1000 * rank)
        state = dx["state"]
        dout = torch.empty(dsteps, dw.N, dw.H, dw.dv, dtype=torch.bfloat16, device=dev)
        views = [tuple(dx[n][t] for n in ("q", "k", "v", "log_alpha", "beta")) for t in range(dsteps)]

        def dstep(t):
            kda.kda_decode_step(*views[t], state, dout[t], stream=stream)

        for t in range(min(3, dsteps)):
            dstep(t)
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        ev0.record(stream)
        for t in range(dsteps):
            dstep(t)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        dms_local = ev0.elapsed_time(ev1)
        dms = reduce_max(dms_local, world, dev)
        per = dms / dsteps
        db_ = decode_bytes(dw.N, dw.H, dw.dk, dw.dv)
        gbs = db_ / (dms_local / dsteps * 1e-3) / 1e9
        dec = {"workload": dw.name, "steps": dsteps, "us_per_step": round(per * 1e3, 2),
               "state_gbs": round(world * db_ / (per * 1e-3) / 1e9, 1),
               "seq_steps_per_s": round(world * dw.N / (per * 1e-3), 1),
               "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                            "frac": round(gbs / hbm_peak, 4), "kernel": "decode_d128_half_kernel",
                            "algorithmic_bytes_per_launch": db_},
               "launches": dsteps}
        del dx, views

    # the long-context and varlen workloads, reported beside the headline
    extra = {}
    for key, wl, nsteps in (("long_context", inputs.LONG_T1M, args.long_steps),
                            ("varlen", inputs.VARLEN_64, args.varlen_steps)):
        if nsteps > 0:
            extra[key] = time_prefill_workload(kda, inputs, wl, nsteps, dev, stream, world, rank, hbm_peak,
                                               0.0 if args.no_cpu_baseline else args.cpu_seconds / 2)

    if world > 1 and args.cp_steps > 0:
        extra["cp"] = time_cp(kda, inputs, args.cp_steps, dev, world, rank)
    if args.ckpt_steps > 0:
        extra["checkpoints"] = time_checkpoints(kda, x, w, args.ckpt_steps, 512, ms_step, dev, stream, world)
    if args.bwd_steps > 0:
        extra["backward"] = time_backward(kda, x, w, args.bwd_steps, ms_step, dev, stream, world)
    if args.layer_steps > 0:
        extra["layer_form"] = time_layer(kda, inputs, x, w, args.layer_steps, ms_step, dev, stream, world, rank,
                                         hbm_peak)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), log_alpha U[ln0.5,-1e-3], beta sigmoid(N(0,1)))",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                       "chunk": w.chunk, "qkv": "bf16", "gates": "fp32", "state": "fp32, zero initial",
                       "out": "bf16", "kernel": "tcgen05 chunk_tc_kernel",
                       "l2": "inputs 1.62 GB per step > 129 MB L2: no flush"},
            "roofline": roofline,
            "gpu_launches": args.steps,
            "e2e": e2e,
            "decode": dec,
            "clocks": clk,
            **extra,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, x, seconds=args.cpu_seconds)
            if dec is not None:
                line["decode"]["cpu_baseline"] = cpu_baseline_decode(inputs.DECODE_N256, dev)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def time_prefill_workload(kda, inputs, w, steps, dev, stream, world, rank, hbm_peak, cpu_seconds=0.0):
    """Times one more prefill workload (one kda_chunk_fwd call per step); with
    cpu_seconds > 0 (rank 0) the oracle is timed beside it on a bounded sample."""
    import numpy as np
    import torch
    x = inputs.make_prefill(w, device=dev, seed=inputs.SEED_BASE + w.seed_index + 1000 * rank)
    varlen = w.varlen_seqs > 0
    cu = x["cu_seqlens"] if varlen else None
    B = None if varlen else w.B
    out = torch.empty(x["T_total"], w.H, w.dv, dtype=torch.bfloat16, device=dev)
    sT = torch.empty(x["N"], w.H, w.dk, w.dv, dtype=torch.float32, device=dev)
    d = kda.chunk_desc(x["q"], x["v"], cu_seqlens=cu, gate_dtype=0, B=B)
    ws_bytes = kda.kda_chunk_fwd_workspace_size(d)

    def step():
        kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["initial_state"], cu, out, sT,
                          B=B, stream=stream)

    step()
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms_local = ev0.elapsed_time(ev1) / steps
    ms = reduce_max(ms_local, world, dev)
    tokens = x["T_total"]
    lens = np.asarray(x["lengths"])
    alg = prefill_bytes(1, tokens, w.H, w.dk, w.dv, state_in=x["initial_state"] is not None)
    alg += (x["N"] - 1) * w.H * w.dk * w.dv * 4 * (2 if x["initial_state"] is not None else 1)
    gbs = alg / (ms_local * 1e-3) / 1e9
    res = {"workload": w.name, "steps": steps, "ms_per_step": round(ms, 3),
           "tokens_per_s": round(world * tokens / (ms * 1e-3), 1), "tokens": int(tokens),
           "sequences": int(x["N"]), "longest": int(lens.max()),
           "split_workspace_bytes": int(ws_bytes),
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                        "frac": round(gbs / hbm_peak, 4), "algorithmic_bytes_per_step": int(alg)}}
    if cpu_seconds > 0 and rank == 0:
        res["cpu_baseline"] = cpu_baseline_sample(w, x, cpu_seconds)
    del x, out, sT
    torch.cuda.empty_cache()
    return res


def time_cp(kda, inputs, steps, dev, world, rank, w=None, backend=None, all_gather=None, seed_base=None):
    """The long-context workload over the ranks by tokens, through the
    context-parallel path (kda_chunk_fwd_cp): rank r holds tokens
    [r L, (r + 1) L) of every sequence, forms its affine pair, one all-gather
    moves every rank's pair (and rank 0's initial state), the entry states are
    composed and the local segment rerun.  Total work is fixed (strong
    scaling); the pairs are the only data that crosses devices.  `backend` and
    `all_gather` default to the library and torch.distributed; on a CPU device
    the steps are timed with the host clock."""
    import time
    import torch
    from hybrid_linear_attention_chunk_gb300.cp import LibraryBackend, kda_chunk_fwd_cp

    w = w or inputs.LONG_T1M
    if w.T % world:
        return {"workload": w.name, "skipped": f"{w.T} tokens do not split evenly over {world} ranks"}
    L = w.T // world
    wl = inputs.scaled(w, T=L)
    seed = (inputs.SEED_BASE if seed_base is None else seed_base) + w.seed_index + 1000 * rank
    x = inputs.make_prefill(wl, device=dev, seed=seed)
    s0 = x["initial_state"] if rank == 0 else None
    backend = backend or LibraryBackend(kda)

    def step():
        return kda_chunk_fwd_cp(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], s0, rank=rank, world=world,
                                B=w.B, all_gather=all_gather, backend=backend)

    cuda = dev.type == "cuda"
    sync = (lambda: torch.cuda.synchronize(dev)) if cuda else (lambda: None)
    step()
    sync()
    barrier(world, dev if cuda else None)
    if cuda:
        stream = torch.cuda.current_stream(dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        sync()
        ms_local = ev0.elapsed_time(ev1) / steps
    else:
        t0 = time.perf_counter()
        for _ in range(steps):
            step()
        ms_local = (time.perf_counter() - t0) * 1e3 / steps
    per_rank = [ms_local]
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
        parts = [torch.zeros_like(t) for _ in range(world)]
        dist.all_gather(parts, t)
        per_rank = [float(p.item()) for p in parts]
    ms = max(per_rank)
    tokens = w.B * w.T
    pair_bytes = 3 * w.B * w.H * w.dk * w.dv * 4
    res = {"workload": w.name, "path": "kda_chunk_fwd_cp", "ranks": world, "tokens_per_rank": L,
           "steps": steps, "ms_per_step": round(ms, 3), "tokens_per_s": round(tokens / (ms * 1e-3), 1),
           "scaling": "strong", "per_rank_ms": [round(v, 3) for v in per_rank],
           "allgather_bytes_per_rank": pair_bytes}
    del x
    if cuda:
        torch.cuda.empty_cache()
    return res


def time_checkpoints(kda, x, w, steps, every, ms_headline, dev, stream, world):
    """The headline batch through kda_chunk_fwd_ckpt, keeping the state every
    `every` tokens (the prefix cache's 512-token hash block)."""
    import torch
    slots = w.B * (w.T // every)
    ck = torch.empty(slots, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)
    out = torch.empty(w.B * w.T, w.H, w.dv, dtype=torch.bfloat16, device=dev)
    sT = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)

    def step():
        kda.kda_chunk_fwd_ckpt(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], every, out=out,
                               final_state=sT, ckpt=ck, B=w.B, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = reduce_max(ev0.elapsed_time(ev1) / steps, world, dev)
    res = {"workload": w.name, "every": every, "slots": slots, "steps": steps, "ms_per_step": round(ms, 4),
           "checkpoint_bytes_per_step": int(ck.numel() * 4),
           "time_vs_headline": round(ms / ms_headline, 4)}
    del ck, out, sT
    torch.cuda.empty_cache()
    return res


def time_backward(kda, x, w, steps, ms_headline, dev, stream, world):
    """kda_chunk_bwd on the headline batch (the forward recomputed inside),
    with a random d_out and a caller workspace."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(123)
    dO = torch.randn(w.B * w.T, w.H, w.dv, generator=gen, device=dev).to(torch.bfloat16)
    d = kda.chunk_desc(x["q"], x["v"], out_dtype=dO.dtype, gate_dtype=0, B=w.B)
    ws_bytes = kda.kda_chunk_bwd_workspace_size(d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    f = dict(dtype=torch.float32, device=dev)
    grads = dict(dq=torch.empty(x["q"].shape, **f), dk=torch.empty(x["k"].shape, **f),
                 dv=torch.empty(x["v"].shape, **f), dlog_alpha=torch.empty(x["log_alpha"].shape, **f),
                 dbeta=torch.empty(x["beta"].shape, **f), d_initial_state=None)

    def step():
        kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], dO, B=w.B, stream=stream,
                          workspace=ws, grads=grads)

    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms_local = ev0.elapsed_time(ev1) / steps
    ms = reduce_max(ms_local, world, dev)
    tok = w.B * w.T
    # algorithmic bytes: the forward's inputs and dO read once, the five fp32
    # gradients written once (no initial state, no final-state gradient here)
    th = tok * w.H
    qkv_b = x["q"].element_size()
    alg = th * ((2 * w.dk + w.dv) * qkv_b + w.dk * 4 + 4 + w.dv * dO.element_size()) \
        + th * ((2 * w.dk + w.dv + w.dk) * 4 + 4)
    gbs = alg / (ms_local * 1e-3) / 1e9
    res = {"workload": w.name, "api": "kda_chunk_bwd (fp32, 16-token chunks; gradient products on mma.sync split-tf32)", "steps": steps,
           "ms_per_step": round(ms, 3), "tokens_per_s": round(world * tok / (ms * 1e-3), 1),
           "time_vs_forward": round(ms / ms_headline, 3), "workspace_bytes": int(ws_bytes),
           "launches_per_step": 4,
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": load_peaks()[0], "unit": "GB/s",
                        "frac": round(gbs / load_peaks()[0], 4), "algorithmic_bytes_per_step": int(alg),
                        "note": "the per-chunk states the backward keeps (workspace) are not algorithmic bytes"}}
    del dO, ws, grads
    torch.cuda.empty_cache()
    return res


def time_layer(kda, inputs, x, w, steps, ms_headline, dev, stream, world, rank, hbm_peak):
    """The headline batch in the layer form (kda_layer_fwd): log-decay from
    bf16 decay logits inside the kernel, output RMSNorm and sigmoid gate in its
    epilogue.  Beside it, the same layer unfused: torch forms the fp32
    log-decay, kda_chunk_fwd runs, torch applies the norm and the gate."""
    import torch
    gt = inputs.make_layer_gates(w.B * w.T, w.H, w.dk, w.dv, w.qkv_dtype, device=dev,
                                 seed=inputs.SEED_BASE + 100 + 1000 * rank)
    out = torch.empty(w.B * w.T, w.H, w.dv, dtype=torch.bfloat16, device=dev)
    sT = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)

    def fused():
        kda.kda_layer_fwd(x["q"], x["k"], x["v"], gt["z"], x["beta"], gt["A_log"], -5.0, out_gate=gt["out_gate"],
                          norm_weight=gt["norm_weight"], norm_eps=1e-6, out=out, final_state=sT, B=w.B,
                          stream=stream)

    def unfused():
        g = -5.0 * torch.sigmoid(torch.exp(gt["A_log"])[None, :, None] * gt["z"].float())
        o, _ = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], g, x["beta"], None, None, out, sT, B=w.B, stream=stream)
        of = o.float()
        y = of * torch.rsqrt(of.pow(2).mean(-1, keepdim=True) + 1e-6) * gt["norm_weight"]
        return (y * torch.sigmoid(gt["out_gate"].float())).to(torch.bfloat16)

    def timed(fn, n):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        torch.cuda.synchronize(dev)
        barrier(world, dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(n):
                fn()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return reduce_max(ev0.elapsed_time(ev1) / n, world, dev)

    ms = timed(fused, steps)
    ms_unfused = timed(unfused, max(steps // 5, 3))
    tok = w.B * w.T
    # per (token, head): q, k, v, z, out_gate and out in bf16, beta fp32
    alg = tok * w.H * ((2 * w.dk + w.dv) * 2 + w.dk * 2 + 4 + w.dv * 2 + w.dv * 2) + w.B * w.H * w.dk * w.dv * 4
    gbs = alg / (ms * 1e-3) / 1e9
    res = {"workload": w.name, "api": "kda_layer_fwd (decay logits bf16, out_gate bf16, RMSNorm weight fp32)",
           "steps": steps, "ms_per_step": round(ms, 4), "tokens_per_s": round(world * tok / (ms * 1e-3), 1),
           "time_vs_headline": round(ms / ms_headline, 4),
           "unfused_ms_per_step": round(ms_unfused, 4),
           "unfused": "torch log-decay + kda_chunk_fwd + torch RMSNorm/gate",
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                        "frac": round(gbs / hbm_peak, 4), "algorithmic_bytes_per_step": int(alg)}}
    del gt, out, sT
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------- oracle on the host

def cpu_baseline(w, x, seconds=12.0):
    """The fp64 oracle (as it stands) on host cores over a bounded sample of the
    workload: whole (sequence, head) chains of T tokens."""
    import numpy as np
    import oracle
    from hybrid_linear_attention_chunk_gb300 import inputs

    cores = os.cpu_count() or 1
    T = w.T

    def run_chains(nchains):
        # chains 0..nchains-1 in (sequence, head) order; host copies of just those
        nh = min(w.H, nchains)
        ns = (nchains + w.H - 1) // w.H
        hs = {name: inputs.host_f32(x[name][: ns * T, :nh].contiguous())
              for name in ("q", "k", "v", "log_alpha", "beta")}
        cu = np.arange(ns + 1, dtype=np.int64) * T
        t0 = time.perf_counter()
        oracle.recurrent(hs["q"], hs["k"], hs["v"], hs["log_alpha"], hs["beta"], None, cu,
                         chains=list(range(nchains)), nthreads=cores, want_o=True)
        return time.perf_counter() - t0

    # calibrate with one chain, then fill ~`seconds` across all cores
    t1 = run_chains(1)
    nchains = int(max(1, min(w.B * w.H, round(seconds / max(t1, 1e-3) * cores))))
    if nchains > w.H:
        nchains = (nchains // w.H) * w.H
    dt = run_chains(nchains)
    tok_equiv = nchains * T / w.H  # tokens (all heads) of work done
    res = {"value": round(tok_equiv / dt, 2), "unit": "tokens/s", "cores": min(cores, nchains),
           "kind": "oracle",
           "sample": f"{nchains} of {w.B * w.H} (sequence, head) chains of {w.name}, full length {T}; "
                     f"value = chains*T/H tokens per second; {dt:.1f} s"}
    # the same oracle on one thread: the first L tokens of one chain
    h1 = {name: inputs.host_f32(x[name][:T, :1].contiguous()) for name in ("q", "k", "v", "log_alpha", "beta")}

    def one_thread(L):
        t0 = time.perf_counter()
        oracle.recurrent(*(h1[n][:L] for n in ("q", "k", "v", "log_alpha", "beta")), None,
                         np.array([0, L], dtype=np.int64), nthreads=1)
        return time.perf_counter() - t0

    L = min(T, max(64, int(512 * min(4.0, seconds / 3) / max(one_thread(512), 1e-4))))
    d1 = one_thread(L)
    res["one_thread"] = {"value": round(L / w.H / d1, 2), "unit": "tokens/s", "cores": 1,
                         "sample": f"tokens [0, {L}) of chain (0, 0) on one thread; value = L/H tokens per second; "
                                   f"{d1:.1f} s"}
    return res


def cpu_baseline_sample(w, x, seconds=6.0):
    """The fp64 oracle (as it stands) on host cores over a bounded sample of a
    prefill workload: the first L tokens of sequence 0, every head in parallel,
    from the sequence's initial state, L calibrated to about `seconds`."""
    import numpy as np
    import oracle
    from hybrid_linear_attention_chunk_gb300 import inputs

    cores = os.cpu_count() or 1
    names = ("q", "k", "v", "log_alpha", "beta")
    len0 = int(x["lengths"][0])
    s0 = x["initial_state"]
    s0h = None if s0 is None else inputs.host_f32(s0[:1])

    def run(L):
        hs = [inputs.host_f32(x[n][:L]) for n in names]
        t0 = time.perf_counter()
        oracle.recurrent(*hs, s0h, np.array([0, L], dtype=np.int64), nthreads=cores, want_o=True)
        return time.perf_counter() - t0

    L0 = min(len0, 256)
    t_cal = run(L0)
    L = int(min(len0, max(L0, L0 * seconds / max(t_cal, 1e-4))))
    dt = run(L)
    return {"value": round(L / dt, 2), "unit": "tokens/s", "cores": min(cores, w.H), "kind": "oracle",
            "sample": f"tokens [0, {L}) of sequence 0 of {w.name}, all {w.H} heads in parallel"
                      f"{'' if s0 is None else ' from its initial state'}; value = tokens (every head) per "
                      f"second; {dt:.1f} s"}


def cpu_baseline_decode(dw, dev, seconds=8.0):
    """The fp64 oracle's decode step on host cores over the whole decode state
    (N=256, H=32, d=128, every head), for as many consecutive steps as fill
    about `seconds`."""
    import numpy as np
    import oracle
    from hybrid_linear_attention_chunk_gb300 import inputs

    cores = os.cpu_count() or 1
    K = 64
    dx = inputs.make_decode(dw, steps=K, device=dev)
    names = ("q", "k", "v", "log_alpha", "beta")
    S = inputs.host_f32(dx["state"]).astype(np.float64)
    steps = [[inputs.host_f32(dx[n][t]) for n in names] for t in range(K)]
    del dx
    t0 = time.perf_counter()
    done = 0
    while done < K and (done < 2 or time.perf_counter() - t0 < seconds):
        _, S = oracle.decode_step(*steps[done], S, nthreads=cores)
        done += 1
    dt = time.perf_counter() - t0
    per = dt / done
    return {"value": round(dw.N / per, 2), "unit": "seq*steps/s",
            "state_gbs": round(decode_bytes(dw.N, dw.H, dw.dk, dw.dv) / per / 1e9, 3), "cores": cores,
            "kind": "oracle",
            "sample": f"{done} consecutive steps of {dw.name} over all {dw.N * dw.H} heads; {dt:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    import torch
    from hybrid_linear_attention_chunk_gb300 import inputs

    w = inputs.PREFILL_B4_T8K
    cores = os.cpu_count() or 1
    # a bounded slice of the workload: `cores` heads of sequence 0, first L tokens
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    L0 = 512
    xs = inputs.make_prefill(inputs.scaled(w, B=1, H=min(cores, w.H)), device=dev)
    hs = {n: inputs.host_f32(xs[n]) for n in ("q", "k", "v", "log_alpha", "beta")}

    def one(L):
        cu = np.array([0, L], dtype=np.int64)
        t0 = time.perf_counter()
        oracle.recurrent(hs["q"][:L], hs["k"][:L], hs["v"][:L], hs["log_alpha"][:L], hs["beta"][:L],
                         None, cu, nthreads=cores)
        return time.perf_counter() - t0

    t_cal = one(L0)
    budget = 90.0 / max(1, args.steps + args.warmup)  # whole run within ~2 minutes
    L = int(min(w.T, max(16, L0 * budget / max(t_cal, 1e-4))))
    for _ in range(args.warmup):
        one(L)
    times = [one(L) for _ in range(args.steps)]
    dt = sum(times)
    heads = hs["q"].shape[1]
    tokens = args.steps * L * heads / w.H
    value = tokens / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                       "chunk": w.chunk},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step: {heads} heads x {L} tokens of sequence 0 "
                                       f"(value = tokens*heads/H per second)"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--long-steps", type=int, default=3, help="steps of the 2^20-token workload (0: skip)")
    ap.add_argument("--varlen-steps", type=int, default=5, help="steps of the 64-sequence varlen workload")
    ap.add_argument("--bwd-steps", type=int, default=10,
                    help="steps of the backward on the headline batch (0: skip)")
    ap.add_argument("--layer-steps", type=int, default=100,
                    help="steps of the headline batch in the layer form (0: skip)")
    ap.add_argument("--ckpt-steps", type=int, default=100,
                    help="steps of the headline batch with 512-token state checkpoints (0: skip)")
    ap.add_argument("--cp-steps", type=int, default=3,
                    help="with N > 1: steps of the 2^20-token workload split over the ranks by tokens "
                         "(context-parallel path; 0: skip)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
