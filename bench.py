"""Benchmark of the quantized GEMM / implicit-GEMM conv path on one GB300.

A step is one quantized GEMM (u8 activations with zero point x s8 per-channel
weights, int32 accumulation, fused requant to int8) on the ViT-B MLP fc1
layer: M = 64 x 197 tokens = 12608, K = 768, N = 3072 -- one qgemm_s8 call with
a workspace (the A pre-pass kernel, then the GEMM kernel).  A second loop runs
the two kernels as separate calls with events around each, for the roofline
line (the GEMM kernel alone) and the pre-pass figures.
Inputs are resident in HBM; L2 is flushed (a 256 MiB write) between timed
steps, outside the timed events.  The line also carries the quantize GB/s of a 1 GiB fp32 -> s8
per-row quantize and the other layer shapes as extras.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --impl reference the CPU oracle is timed on a bounded sample of the same
workload (the reference arm).  Under torchrun every rank runs its own replica
(weak scaling, no collective on the data path); rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "int8 TOPS and % of GB300 dense-INT8 peak (GEMM/conv); quantize GB/s vs HBM"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the headline GEMM kernel, taken from a kept ncu capture of this workload (not
# measured in this run); valid only for the sources that kernel is built from
# (hash of HEADLINE_SOURCES) and reported as null otherwise.
TRAFFIC_NCU = {"csrc_sha256_16": "27f01dc14f452274", "bytes": 24317696 + 901120}


HEADLINE_SOURCES = ("qnn_gemm.cu", "qnn_gemm_layout.h", "qnn_internal.h", "qnn_mma_kernel.cuh", "qnn_ptx.cuh")


def csrc_hash():
    import hashlib
    h = hashlib.sha256()
    for name in HEADLINE_SOURCES:
        f = os.path.join(ROOT, "integer_quantized_nn_gb300", "csrc", name)
        h.update(name.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return dict(FALLBACK), "fallback"


# ------------------------------------------------------------------ dist utils
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Dist:
    def __init__(self, backend):
        self.ws, self.rank, self.local = dist_env()
        self.pg = None
        if self.ws > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([float(v)], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"qnn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(1.0)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        if not isinstance(rows, list) or not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


# ------------------------------------------------------------------ GPU arm
def gpu_setup_gemm(torch, qnn, w, a_dt, device, ptf=None):
    A = torch.from_numpy(np.ascontiguousarray(w["A"])).to(device)
    B = torch.from_numpy(np.ascontiguousarray(w["B"])).to(device)
    N, K = w["B"].shape
    nb = qnn.qnn_gemm_packed_b_bytes(N, K)
    buf = torch.empty(nb + 1024, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 1024
    Bp = buf[off:off + nb]
    colsum = torch.empty(N, dtype=torch.int32, device=device)
    if ptf is None:
        qnn.qgemm_prepack_b(B, Bp, colsum)
    else:
        qnn.qgemm_prepack_b_ptf(B, ptf, Bp, colsum)
    sw = torch.from_numpy(np.asarray(w["s_w"], np.float32)).to(device)
    bias = None if w.get("bias") is None else torch.from_numpy(w["bias"]).to(device)
    zp = torch.empty(N, dtype=torch.int32, device=device)
    Mv = torch.empty(N, dtype=torch.float32, device=device)
    Bq = torch.empty(N, dtype=torch.float32, device=device)
    qnn.q_fold_epilogue(N, a_dt, w["z_a"], colsum, w["s_a"], sw, w["s_o"], bias=bias, zp_term=zp,
                        M=Mv, Bq=Bq)
    return dict(A=A, Bp=Bp, zp=zp, M=Mv, Bq=Bq, keep=(buf, B, colsum, sw, bias))


def time_steps(torch, fn, steps, warmup, flush, stream):
    """Per-step CUDA events around fn() on `stream`; L2 flushed between steps
    outside the events.  Returns list of ms."""
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_split(torch, fns, steps, warmup, flush, stream):
    """Like time_steps for a step made of several calls: events before, between
    and after the calls of fns.  Returns (whole-step ms list, per-call ms lists)."""
    for _ in range(warmup):
        flush()
        for f in fns:
            f()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)] for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        for j, f in enumerate(fns):
            f()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    whole = [e[0].elapsed_time(e[-1]) for e in ev]
    parts = [[e[j].elapsed_time(e[j + 1]) for e in ev] for j in range(len(fns))]
    return whole, parts


def run_gpu(args):
    import torch
    dist = Dist("nccl")
    torch.cuda.set_device(dist.local)
    device = torch.device("cuda", dist.local)
    from integer_quantized_nn_gb300 import qnn, workloads
    qnn.load()
    pk, pk_kind = peaks()
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def flush():
        flush_buf.fill_(1)

    # ---- headline workload: ViT-B fc1
    M, K, N = 12608, 768, 3072
    w = workloads.vit_fc1(M=M, K=K, N=N)
    g = gpu_setup_gemm(torch, qnn, w, "u8", device)
    C = torch.empty((M, N), dtype=torch.uint8, device=device)
    epi = qnn.epilogue("requant", zp_term=g["zp"], M=g["M"], Bq=g["Bq"], out_dt="s8")
    ws_buf = torch.empty(qnn.qnn_gemm_workspace_bytes(M, K), dtype=torch.uint8, device=device)

    # a step: one qgemm_s8 call with the workspace -- the A pre-pass kernel, then the GEMM
    # kernel launched as its programmatic dependent (its launch overlaps the pre-pass tail)
    def step():
        qnn.qgemm_s8(g["A"], "u8", g["Bp"], M, N, K, epi, C, workspace=ws_buf, stream=stream)

    # the same two kernels as separate calls, for each kernel's own duration
    def pack():
        qnn.qgemm_pack_a(g["A"], "u8", M, K, ws_buf, stream=stream)

    def gemm():
        qnn.qgemm_s8_packed(ws_buf, "u8", g["Bp"], M, N, K, epi, C, stream=stream)

    flops = 2.0 * M * N * K
    dist.barrier()
    clk = ClockSampler(dist.local)
    clk.start()
    torch.cuda.synchronize()
    dist.barrier()
    t_wall0 = time.time()
    times = time_steps(torch, step, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    dist.barrier()
    t_wall1 = time.time()
    # second loop, same steps and flushes: events around each kernel (the event between them
    # also stops the dependent-launch overlap, so this loop's steps are a little longer)
    _, (t_pack, t_gemm) = time_split(torch, [pack, gemm], args.steps, 1, flush, stream)
    torch.cuda.synchronize()
    t_wall2 = time.time()
    clocks = ClockSampler.summarize(clk.stop(), t_wall0, t_wall2)
    st = qnn.qnn_check_device_error()
    if st != qnn.QNN_OK:
        raise RuntimeError(f"device status: {qnn.status_string(st)}")
    total_ms = sum(times)
    total_ms_max = dist.max(total_ms)
    value = dist.ws * args.steps * flops / (total_ms_max * 1e-3) / 1e12
    gemm_ms = sum(t_gemm) / args.steps
    achieved = flops / (gemm_ms * 1e-3) / 1e12
    pack_ms = sum(t_pack) / args.steps
    pack_bytes = M * K + qnn.qnn_gemm_workspace_bytes(M, K)

    # ---- e2e: host buffers, every step's copies inside the timed region.  Steps are
    # pipelined as a server would run them: step i's H2D copy (its own pinned input
    # buffer), its qgemm_s8 call and its D2H copy of the result run on three streams,
    # so step i's GEMM overlaps step i-1's D2H and step i+1's H2D (two device buffer
    # sets); an L2 flush (160 MiB write) precedes every GEMM on the compute stream and
    # counts inside the timed region.
    e2e_steps = max(3, min(args.steps, 200))
    A_h = [torch.from_numpy(np.ascontiguousarray(w["A"])).pin_memory() for _ in range(2)]
    C_h = [torch.empty((M, N), dtype=torch.uint8).pin_memory() for _ in range(2)]
    A_d = [torch.empty_like(g["A"]) for _ in range(2)]
    C_d = [torch.empty((M, N), dtype=torch.uint8, device=device) for _ in range(2)]
    e2e_flush = torch.empty(160 << 20, dtype=torch.uint8, device=device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("h2d", "gemm", "d2h")}

    def e2e_loop(n):
        for i in range(n):
            b = i % 2
            s_in.wait_event(ev["gemm"][b])        # A_d[b] free again
            with torch.cuda.stream(s_in):
                A_d[b].copy_(A_h[b], non_blocking=True)
            ev["h2d"][b].record(s_in)
            stream.wait_event(ev["h2d"][b])
            stream.wait_event(ev["d2h"][b])       # C_d[b] free again
            e2e_flush.fill_(i & 255)
            qnn.qgemm_s8(A_d[b], "u8", g["Bp"], M, N, K, epi, C_d[b], workspace=ws_buf, stream=stream)
            ev["gemm"][b].record(stream)
            s_out.wait_event(ev["gemm"][b])
            with torch.cuda.stream(s_out):
                C_h[b].copy_(C_d[b], non_blocking=True)
            ev["d2h"][b].record(s_out)

    e2e_loop(max(2, args.warmup))
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    s_in.wait_event(t_start)
    s_out.wait_event(t_start)
    e2e_loop(e2e_steps)
    stream.wait_stream(s_out)
    stream.wait_stream(s_in)
    t_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = dist.max(t_start.elapsed_time(t_end)) / e2e_steps
    e2e_value = dist.ws * flops / (e2e_ms * 1e-3) / 1e12
    st = qnn.qnn_check_device_error()
    if st != qnn.QNN_OK:
        raise RuntimeError(f"device status: {qnn.status_string(st)}")
    if not torch.equal(C_h[(e2e_steps - 1) % 2], C.cpu()):
        raise RuntimeError("end-to-end output differs from the device-timed output")

    extras = {}
    if not args.no_extras and dist.rank == 0:
        extras = run_extras(torch, qnn, workloads, device, flush, stream, pk, args)

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1), and the
    # oracle's single-thread / all-core times for every workload
    cpu = None
    otab = None
    if dist.rank == 0 and dist.ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_gemm(w, target_s=args.cpu_seconds)
        if not args.no_oracle_table:
            gms = {k: v["ms"] for k, v in extras.items() if isinstance(v, dict) and "ms" in v}
            gms["vit_fc1"] = round(total_ms_max / args.steps, 5)
            otab = oracle_table(gms)

    dtype_str = "u8 x s8 -> s32 (exact on the f16 tensor pipe), requant to s8"
    peak = float(pk["bf16_tflops"])
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TOPS", "n_gpus": dist.ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_str,
        "data": "synthetic (seeded numpy PCG64; no dataset or trained weights)",
        "config": {"workload": "ViT-B MLP fc1 qgemm_s8: u8 (Z=128) x s8 per-channel -> s8",
                   "M": M, "K": K, "N": N, "tokens": "64 x 197", "l2": "flushed between steps "
                   "(256 MiB write, outside the timed events)", "parallelism": f"replicas x{dist.ws}"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": (TRAFFIC_NCU["bytes"] if csrc_hash() == TRAFFIC_NCU["csrc_sha256_16"]
                                 else None),
                     "traffic_unit": "bytes per launch (ncu DRAM read + write); a constant from a "
                                     "kept ncu capture of the same kernel sources, not measured in this run",
                     "peak_kind": f"{pk_kind} bf16 dense burst (the f16 MMA kind runs at the bf16 rate)",
                     "kernel": "qmma_kernel<GemmPackedOp,256,false>",
                     "kernel_ms": round(gemm_ms, 5),
                     "kernel_timing": "CUDA events around the GEMM kernel alone, in a second loop of "
                                      "the same steps right after the timed one (same L2 flushes)",
                     "algorithmic": "2*M*N*K int ops per launch"},
        "prepass": {"kernel": "pack_a_kernel<false>", "ms": round(pack_ms, 5),
                    "bytes": pack_bytes, "GB/s": round(pack_bytes / (pack_ms * 1e-3) / 1e9, 1),
                    "frac_hbm": round(pack_bytes / (pack_ms * 1e-3) / 1e9 / float(pk["hbm_gbs"]), 4),
                    "algorithmic": "M*K code bytes read + the fp16 image written"},
        "cpu_baseline": cpu,
        "oracle_cpu": otab,
        "e2e": {"value": round(e2e_value, 3), "unit": "TOPS", "h2d_bytes_per_step": M * K,
                "d2h_bytes_per_step": M * N, "ms_per_step": round(e2e_ms, 5),
                "pipelining": "H2D / qgemm_s8 / D2H on three streams, two buffer sets; an L2 flush "
                              "before every GEMM inside the timed region"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "extras": extras,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def _aligned_1024(torch, nbytes, device):
    buf = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 1024
    return buf[off:off + nbytes]


def setup_conv_u8zw(torch, qnn, workloads, device, stream):
    """ResNet-50 stage-1 3x3 Conv_Add_Relu, u8 activations x u8 filters with
    per-filter zero points (qconv_prepack_w_u8 + qconv_u8u8).  Returns the call
    and its op / byte counts."""
    wc = workloads.conv_u8()
    Nb, H, W, C, OC = 64, 56, 56, 64, 64
    g = qnn.conv_geom(Nb, H, W, C, OC, 3, 3, (1, 1), (1, 1))
    Wp = _aligned_1024(torch, qnn.qnn_conv_packed_w_bytes(g, "u8"), device)
    cs = torch.empty(OC, dtype=torch.int32, device=device)
    qnn.qconv_prepack_w_u8(torch.from_numpy(wc["W"]).to(device), torch.from_numpy(wc["z_w"]).to(device), g, Wp, cs)
    zp = torch.empty(OC, dtype=torch.int32, device=device)
    Mv = torch.empty(OC, dtype=torch.float32, device=device)
    Bq = torch.empty(OC, dtype=torch.float32, device=device)
    qnn.q_fold_epilogue(OC, "u8", wc["z_in"], cs, wc["s_a"], torch.from_numpy(wc["s_w"]).to(device), wc["s_o"],
                        bias=torch.from_numpy(wc["bias"]).to(device), zp_term=zp, M=Mv, Bq=Bq, w_per_channel=True)
    I8 = torch.from_numpy(wc["I"]).to(device)
    res8 = torch.from_numpy(wc["res"]).to(device)
    R = float(np.float32(np.float32(wc["s_r"]) / np.float32(wc["s_o"])))
    epi = qnn.epilogue("requant", relu=True, out_dt="u8", zp_term=zp, M=Mv, Bq=Bq, residual=res8, res_dt="u8",
                       z_res=wc["z_res"], R=R)
    O8 = torch.empty((Nb, g.OH, g.OW, OC), dtype=torch.uint8, device=device)
    ws8 = torch.empty(qnn.qnn_conv_workspace_bytes(g, "u8"), dtype=torch.uint8, device=device)
    keep = (Wp, cs, zp, Mv, Bq, I8, res8, O8, epi, ws8)

    def fn():
        qnn.qconv_u8u8(keep[5], wc["z_in"], keep[0], g, keep[8], keep[7], workspace=keep[9], stream=stream)

    return fn, {"ops": 2.0 * Nb * g.OH * g.OW * OC * C * 9,
                "bytes": I8.numel() + O8.numel() + res8.numel() + OC * C * 9}


def setup_gemm_zw(torch, qnn, workloads, device, stream):
    """ViT-B fc1 with u8 weights carrying per-channel zero points
    (qgemm_prepack_b_u8 + qgemm_zw with its workspace)."""
    wz = workloads.vit_fc1_zw()
    Mm, Kk = wz["A"].shape
    Nn = wz["B"].shape[0]
    Bp = _aligned_1024(torch, qnn.qnn_gemm_packed_b_bytes(Nn, Kk), device)
    cs = torch.empty(Nn, dtype=torch.int32, device=device)
    zwd = torch.from_numpy(wz["z_w"]).to(device)
    qnn.qgemm_prepack_b_u8(torch.from_numpy(wz["B"]).to(device), zwd, Bp, cs)
    zp = torch.empty(Nn, dtype=torch.int32, device=device)
    Mv = torch.empty(Nn, dtype=torch.float32, device=device)
    Bq = torch.empty(Nn, dtype=torch.float32, device=device)
    qnn.q_fold_epilogue(Nn, "u8", wz["z_a"], cs, wz["s_a"], torch.from_numpy(wz["s_w"]).to(device), wz["s_o"],
                        bias=torch.from_numpy(wz["bias"]).to(device), zp_term=zp, M=Mv, Bq=Bq, w_per_channel=True)
    A = torch.from_numpy(wz["A"]).to(device)
    C = torch.empty((Mm, Nn), dtype=torch.uint8, device=device)
    epi = qnn.epilogue("requant", out_dt="s8", zp_term=zp, M=Mv, Bq=Bq)
    ws = torch.empty(qnn.qnn_gemm_zw_workspace_bytes(Mm, Kk), dtype=torch.uint8, device=device)
    keep = (Bp, cs, zp, Mv, Bq)

    def fn():
        qnn.qgemm_zw(A, "u8", keep[0], zwd, Mm, Nn, Kk, epi, C, workspace=ws, stream=stream)

    return fn, {"ops": 2.0 * Mm * Nn * Kk, "M": Mm, "N": Nn, "K": Kk}


def square_16384(torch, qnn, workloads, device, flush, stream, peak, steps, out):
    """qgemm_s8 at M = N = K = 16384 (8.80 T int ops per call), operands drawn on
    the device; requant multiplier 2^-21 (2^-(ceil(log2 K) + 7)), s8 out."""
    n = 16384
    A = workloads.device_uniform_s8((n, n), 5160, device)
    B = workloads.device_uniform_s8((n, n), 5161, device)
    Bp = _aligned_1024(torch, qnn.qnn_gemm_packed_b_bytes(n, n), device)
    cs = torch.empty(n, dtype=torch.int32, device=device)
    qnn.qgemm_prepack_b(B, Bp, cs)
    del B
    zp = torch.empty(n, dtype=torch.int32, device=device)
    Mv = torch.empty(n, dtype=torch.float32, device=device)
    Bq = torch.empty(n, dtype=torch.float32, device=device)
    qnn.q_fold_epilogue(n, "s8", 0, cs, 1.0, torch.ones(n, dtype=torch.float32, device=device), 2.0 ** 21,
                        zp_term=zp, M=Mv, Bq=Bq)
    C = torch.empty((n, n), dtype=torch.uint8, device=device)
    epi = qnn.epilogue("requant", zp_term=zp, M=Mv, Bq=Bq, out_dt="s8")
    ws = torch.empty(qnn.qnn_gemm_workspace_bytes(n, n), dtype=torch.uint8, device=device)
    t = time_steps(torch, lambda: qnn.qgemm_s8(A, "s8", Bp, n, n, n, epi, C, workspace=ws, stream=stream),
                   max(3, min(steps, 10)), 3, flush, stream)
    ms = statistics.median(t)
    tops = 2.0 * n ** 3 / (ms * 1e-3) / 1e12
    out["square_16384"] = {"M": n, "N": n, "K": n, "ms": round(ms, 4), "TOPS": round(tops, 2),
                           "frac_f16_peak": round(tops / peak, 4)}
    del A, Bp, C, ws


def run_extras(torch, qnn, workloads, device, flush, stream, pk, args):
    out = {}
    hbm = float(pk["hbm_gbs"])
    peak = float(pk["bf16_tflops"])
    steps = max(3, min(args.steps, args.extra_steps))

    # quantize fp32 -> s8, per row, 1 GiB
    R = Cc = 16384
    x = workloads.device_normal_f32((R, Cc), 505, device)
    scale = (x.abs().amax(dim=1) / 127.0).contiguous()
    q = torch.empty((R, Cc), dtype=torch.uint8, device=device)
    p = qnn.qparams("sym", scale=scale, per_channel=True, axis=0)
    t = time_steps(torch, lambda: qnn.q_quantize(x, q, "s8", p, stream=stream), steps, 3, flush,
                   stream)
    ms = statistics.median(t)
    gbs = 5.0 * R * Cc / (ms * 1e-3) / 1e9
    out["quantize_rows_1GiB"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                 "frac_hbm": round(gbs / hbm, 4), "bytes": "5 B/elem"}
    # dequantize s8 -> fp32
    t = time_steps(torch, lambda: qnn.q_dequantize(q, "s8", x, p, stream=stream), steps, 3, flush,
                   stream)
    ms = statistics.median(t)
    gbs = 5.0 * R * Cc / (ms * 1e-3) / 1e9
    out["dequantize_rows_1GiB"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                   "frac_hbm": round(gbs / hbm, 4)}
    # pack fp32 -> u4 (asymmetric, zero point 8, per row), two codes per byte: 4.5 B/elem
    q4 = torch.empty((R, Cc // 2), dtype=torch.uint8, device=device)
    s4 = (scale * (127.0 / 7.5)).contiguous()
    z4 = torch.full((R,), 8, dtype=torch.int32, device=device)
    p4 = qnn.qparams("asym", scale=s4, zero_point=z4, per_channel=True, axis=0)
    t = time_steps(torch, lambda: qnn.q_quantize(x, q4, "u4", p4, stream=stream), steps, 3, flush,
                   stream)
    ms = statistics.median(t)
    gbs = 4.5 * R * Cc / (ms * 1e-3) / 1e9
    out["pack_u4_rows_1GiB"] = {"ms": round(ms, 4), "GB/s": round(gbs, 1),
                                "frac_hbm": round(gbs / hbm, 4), "bytes": "4.5 B/elem (4 read, 0.5 write)"}
    del x, q, q4, scale, s4, z4

    def gemm_entry(name, w, a_dt, alpha=None, ptf_in_weights=False):
        Mm, Kk = w["A"].shape
        Nn = w["B"].shape[0]
        al = None
        if alpha is not None:
            al = torch.from_numpy(alpha.astype(np.uint8)).to(device)
        g = gpu_setup_gemm(torch, qnn, w, a_dt, device, ptf=al if ptf_in_weights else None)
        C = torch.empty((Mm, Nn), dtype=torch.uint8, device=device)
        epi = qnn.epilogue("requant", zp_term=None if al is not None else g["zp"], M=g["M"],
                           Bq=g["Bq"], ptf_shift=None if ptf_in_weights else al,
                           ptf_max_shift=0 if alpha is None else int(alpha.max()))
        ws = torch.empty(qnn.qnn_gemm_workspace_bytes(Mm, Kk), dtype=torch.uint8, device=device)
        t = time_steps(torch, lambda: qnn.qgemm_s8(g["A"], a_dt, g["Bp"], Mm, Nn, Kk, epi, C,
                                                   workspace=ws, stream=stream), steps, 3, flush, stream)
        ms = statistics.median(t)
        tf = time_steps(torch, lambda: qnn.qgemm_s8(g["A"], a_dt, g["Bp"], Mm, Nn, Kk, epi, C,
                                                    stream=stream), steps, 3, flush, stream)
        ms_fused = statistics.median(tf)
        tops = 2.0 * Mm * Nn * Kk / (ms * 1e-3) / 1e12
        out[name] = {"M": Mm, "N": Nn, "K": Kk, "ms": round(ms, 4), "TOPS": round(tops, 2),
                     "frac_f16_peak": round(tops / peak, 4),
                     "ms_no_workspace": round(ms_fused, 4)}

    gemm_entry("gemm_sym_256", workloads.gemm_sym(), "s8")
    for nm, (Kk, Nn) in workloads.VITL_SHAPES.items():
        w = workloads.vitl_ptf(M=12608, K=Kk, N=Nn)
        xq = torch.from_numpy(w["x"]).to(device)
        Aq = torch.empty(w["x"].shape, dtype=torch.uint8, device=device)
        qnn.q_quantize(xq, Aq, "s8", qnn.qparams("sym", scale=torch.from_numpy(w["in_scale"]).to(device),
                                                 per_channel=True, axis=1))
        w2 = dict(A=Aq.cpu().numpy(), B=w["B"], s_w=w["s_w"], bias=w["bias"], s_a=w["s"],
                  s_o=w["s_o"], z_a=0)
        # the layer's PTF factors folded into its weights at prepack (qgemm_prepack_b_ptf)
        gemm_entry(f"vitl_{nm}_ptf", w2, "s8", alpha=w["alpha"], ptf_in_weights=True)
        if nm == "fc2":
            # the same factors applied to the activations by the A pre-pass
            gemm_entry(f"vitl_{nm}_ptf_on_activations", w2, "s8", alpha=w["alpha"])
        del xq, Aq
    for n in (2048, 4096, 8192):
        gemm_entry(f"square_{n}", workloads.gemm_square(n), "s8")
    square_16384(torch, qnn, workloads, device, flush, stream, peak, steps, out)

    def relayout_u4(packed, shape, layout):
        """Packed NHWC nibbles -> the same codes packed in `layout` (data movement only)."""
        if layout == "nhwc":
            return packed
        Nb, H, W, C = shape
        codes = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
        codes[..., 0::2] = packed & 15
        codes[..., 1::2] = packed >> 4
        codes = codes.reshape(Nb, H, W, C)
        if layout == "nchw":
            codes = codes.transpose(0, 3, 1, 2)
        else:
            codes = codes.reshape(Nb, H, W, C // 64, 64).transpose(0, 3, 1, 2, 4)
        flat = np.ascontiguousarray(codes).reshape(-1)
        return (flat[0::2] | (flat[1::2] << 4)).astype(np.uint8)

    def conv_entry(name, w, geom, layout="nhwc"):
        Nb, H, W, C, OC, F, pad, st = geom
        g = qnn.conv_geom(Nb, H, W, C, OC, F, F, (pad, pad), (st, st), layout=layout)
        Wd = torch.from_numpy(w["W"]).to(device)
        nb = qnn.qnn_conv_packed_w_bytes(g, "s4")
        buf = torch.empty(nb + 1024, dtype=torch.uint8, device=device)
        off = (-buf.data_ptr()) % 1024
        Wp = buf[off:off + nb]
        cs = torch.empty(OC, dtype=torch.int32, device=device)
        qnn.qconv_prepack_w(Wd, "s4", g, Wp, cs)
        sw = torch.from_numpy(w["s_w"]).to(device)
        bias = torch.from_numpy(w["bias"]).to(device)
        zp = torch.empty(OC, dtype=torch.int32, device=device)
        Mv = torch.empty(OC, dtype=torch.float32, device=device)
        Bq = torch.empty(OC, dtype=torch.float32, device=device)
        qnn.q_fold_epilogue(OC, "u4", w["z_in"], cs, w["s_a"], sw, w["s_o"], bias=bias, zp_term=zp,
                            M=Mv, Bq=Bq)
        I = torch.from_numpy(relayout_u4(w["I"], (Nb, H, W, C), layout)).to(device)
        res = None if w["res"] is None else torch.from_numpy(
            relayout_u4(w["res"], (Nb, g.OH, g.OW, OC), layout)).to(device)
        R = float(np.float32(np.float32(w["s_r"]) / np.float32(w["s_o"])))
        epi = qnn.epilogue("requant", relu=True, out_dt="u4", zp_term=zp, M=Mv, Bq=Bq, residual=res,
                           res_dt="u4", z_res=w["z_res"], R=R)
        O = torch.empty((Nb, g.OH, g.OW, OC // 2), dtype=torch.uint8, device=device)
        ws = torch.empty(qnn.qnn_conv_workspace_bytes(g, "u4"), dtype=torch.uint8, device=device)
        t = time_steps(torch, lambda: qnn.qconv_u4s4(I, w["z_in"], Wp, g, epi, O, workspace=ws,
                                                     stream=stream), steps, 3, flush, stream)
        ms = statistics.median(t)
        ms_fused = None
        if layout != "nchw":
            tf = time_steps(torch, lambda: qnn.qconv_u4s4(I, w["z_in"], Wp, g, epi, O, stream=stream),
                            steps, 3, flush, stream)
            ms_fused = statistics.median(tf)
        ops = 2.0 * Nb * g.OH * g.OW * OC * C * F * F
        tops = ops / (ms * 1e-3) / 1e12
        byts = I.numel() + O.numel() + (0 if res is None else res.numel()) + Wd.numel()
        out[name] = {"ms": round(ms, 4), "TOPS": round(tops, 2),
                     "frac_fp8_peak": round(tops / (2.0 * peak), 4),
                     "ms_no_workspace": None if ms_fused is None else round(ms_fused, 4),
                     "GB/s": round(byts / (ms * 1e-3) / 1e9, 1),
                     "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / hbm, 4)}

    conv_entry("conv3x3_u4s4_add_relu", workloads.conv_u4(), (64, 56, 56, 64, 64, 3, 1, 1))
    conv_entry("conv1x1_u4s4_relu", workloads.conv_u4(C=256, OC=64, F=1, pad=0, residual=False, tag=1),
               (64, 56, 56, 256, 64, 1, 0, 1))
    # the same 3x3 Conv_Add_Relu with input, residual and output in NCHW and NCHW64
    conv_entry("conv3x3_u4s4_add_relu_nchw", workloads.conv_u4(), (64, 56, 56, 64, 64, 3, 1, 1), layout="nchw")
    conv_entry("conv3x3_u4s4_add_relu_nchw64", workloads.conv_u4(), (64, 56, 56, 64, 64, 3, 1, 1), layout="nchw64")

    # weight zero points: ResNet-50 3x3 with u8 activations x u8 filters (zero point taken
    # out at prepack), and ViT-B fc1 with u8 weights (the run-time row-sum term)
    fn, info = setup_conv_u8zw(torch, qnn, workloads, device, stream)
    t = time_steps(torch, fn, steps, 3, flush, stream)
    ms = statistics.median(t)
    tops = info["ops"] / (ms * 1e-3) / 1e12
    out["conv3x3_u8u8_zw_add_relu"] = {"ms": round(ms, 4), "TOPS": round(tops, 2),
                                       "frac_f16_peak": round(tops / peak, 4),
                                       "GB/s": round(info["bytes"] / (ms * 1e-3) / 1e9, 1),
                                       "frac_hbm": round(info["bytes"] / (ms * 1e-3) / 1e9 / hbm, 4)}
    del fn, info
    fn, info = setup_gemm_zw(torch, qnn, workloads, device, stream)
    t = time_steps(torch, fn, steps, 3, flush, stream)
    ms = statistics.median(t)
    tops = info["ops"] / (ms * 1e-3) / 1e12
    out["vit_fc1_zw"] = {"M": info["M"], "N": info["N"], "K": info["K"], "ms": round(ms, 4),
                         "TOPS": round(tops, 2), "frac_f16_peak": round(tops / peak, 4)}
    del fn, info

    # Log-Int-Softmax over ViT-B attention maps at batch 64, then the shift product with V
    Bh, Lt, dh = 64 * 12, 197, 64
    rows = Bh * Lt
    xl = workloads.device_attention_logits(rows, Lt, 1234, device)
    codes = torch.empty((rows, Lt), dtype=torch.uint8, device=device)
    t = time_steps(torch, lambda: qnn.q_log_int_softmax(xl, rows, Lt, workloads.ATTN_S, 4, codes,
                                                        stream=stream), steps, 3, flush, stream)
    ms = statistics.median(t)
    gbs = 5.0 * rows * Lt / (ms * 1e-3) / 1e9
    out["log_int_softmax_vitb_b64"] = {"rows": rows, "L": Lt, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                                       "frac_hbm": round(gbs / hbm, 4), "bytes": "4 B in + 1 B out /elem"}
    vq = workloads.device_uniform_s8((Bh, Lt, dh), 77, device)
    ov = torch.empty((Bh, Lt, dh), dtype=torch.int32, device=device)
    t = time_steps(torch, lambda: qnn.q_attn_shift_v(codes, vq, Bh, Lt, Lt, dh, 4, ov, stream=stream),
                   steps, 3, flush, stream)
    ms = statistics.median(t)
    byts = Bh * Lt * Lt + Bh * Lt * dh + 4 * Bh * Lt * dh
    out["attn_shift_v_vitb_b64"] = {"heads": Bh, "Lq": Lt, "Lk": Lt, "d": dh, "ms": round(ms, 4),
                                    "GMAC/s": round(Bh * Lt * Lt * dh / (ms * 1e-3) / 1e9, 1),
                                    "GB/s": round(byts / (ms * 1e-3) / 1e9, 1),
                                    "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / hbm, 4)}
    # the same two steps in one kernel (codes kept in shared memory)
    t = time_steps(torch, lambda: qnn.q_lis_attn_v(xl, workloads.ATTN_S, vq, Bh, Lt, Lt, dh, 4, ov, stream=stream),
                   steps, 3, flush, stream)
    ms = statistics.median(t)
    byts = 4 * Bh * Lt * Lt + Bh * Lt * dh + 4 * Bh * Lt * dh
    out["lis_attn_v_fused_vitb_b64"] = {"ms": round(ms, 4), "GB/s": round(byts / (ms * 1e-3) / 1e9, 1),
                                        "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / hbm, 4),
                                        "bytes": "int32 logits + V + int32 out"}
    del xl, codes, vq, ov

    # integer LayerNorm over ViT-B activations at batch 64 (PTF factors), s8 out
    wl = workloads.vit_layernorm()
    lx = torch.from_numpy(wl["x"]).to(device)
    la = torch.from_numpy(wl["alpha"]).to(device)
    lg, lb, lo = (torch.from_numpy(wl[k]).to(device) for k in ("gamma", "beta", "o"))
    R, C = wl["x"].shape
    ly = torch.empty((R, C), dtype=torch.int8, device=device)
    t = time_steps(torch, lambda: qnn.q_int_layernorm(lx, R, C, wl["s"], lg, lb, lo, ly, alpha=la,
                                                      alpha_max=int(wl["alpha"].max()), stream=stream),
                   steps, 3, flush, stream)
    ms = statistics.median(t)
    gbs = 2.0 * R * C / (ms * 1e-3) / 1e9
    out["int_layernorm_vitb_b64"] = {"rows": R, "C": C, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                                     "frac_hbm": round(gbs / hbm, 4), "bytes": "1 B in + 1 B out /elem"}

    # standalone quantized add (shared scale) on the ViT-B residual stream, and the
    # dynamic per-token quantize of the same fp32 activations
    ea = workloads.device_uniform_s8((R, C), 91, device)
    eb = workloads.device_uniform_s8((R, C), 92, device)
    eo = torch.empty((R, C), dtype=torch.int8, device=device)
    t = time_steps(torch, lambda: qnn.q_eltwise_s8("add", ea, eb, R * C, 0.5, eo, stream=stream), steps, 3,
                   flush, stream)
    ms = statistics.median(t)
    gbs = 3.0 * R * C / (ms * 1e-3) / 1e9
    out["eltwise_add_s8_vitb_b64"] = {"n": R * C, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                                      "frac_hbm": round(gbs / hbm, 4), "bytes": "3 B /elem"}
    xf = workloads.device_normal_f32((R, C), 93, device)
    dsc = torch.empty(R, dtype=torch.float32, device=device)
    t = time_steps(torch, lambda: qnn.q_quantize_rows_dynamic(xf, R, C, eo, dsc, stream=stream), steps, 3,
                   flush, stream)
    ms = statistics.median(t)
    gbs = 5.0 * R * C / (ms * 1e-3) / 1e9
    out["quantize_rows_dynamic_vitb_b64"] = {"rows": R, "cols": C, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                                             "frac_hbm": round(gbs / hbm, 4), "bytes": "4 B in + 1 B out /elem"}
    return out


def run_case(args):
    """One workload only, for profiling: warmup + steps launches of its kernel
    (L2 flushed before each), then a one-line JSON with the median time."""
    import torch
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    from integer_quantized_nn_gb300 import qnn, workloads
    qnn.load()
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def flush():
        flush_buf.fill_(1)

    case = args.case
    if case == "dequantize":
        R = Cc = 16384
        x = workloads.device_normal_f32((R, Cc), 505, device)
        scale = (x.abs().amax(dim=1) / 127.0).contiguous()
        q = torch.empty((R, Cc), dtype=torch.uint8, device=device)
        p = qnn.qparams("sym", scale=scale, per_channel=True, axis=0)
        qnn.q_quantize(x, q, "s8", p, stream=stream)
        fn = lambda: qnn.q_dequantize(q, "s8", x, p, stream=stream)  # noqa: E731
    elif case == "quantize":
        R = Cc = 16384
        x = workloads.device_normal_f32((R, Cc), 505, device)
        scale = (x.abs().amax(dim=1) / 127.0).contiguous()
        q = torch.empty((R, Cc), dtype=torch.uint8, device=device)
        p = qnn.qparams("sym", scale=scale, per_channel=True, axis=0)
        fn = lambda: qnn.q_quantize(x, q, "s8", p, stream=stream)  # noqa: E731
    elif case in ("vit_fc1", "square_4096", "vitl_fc2") or case.startswith("gemm:"):
        if case.startswith("gemm:"):
            Mg, Ng, Kg = (int(v) for v in case.split(":")[1:4])
            w, a_dt, alpha = workloads.vit_fc1(M=Mg, K=Kg, N=Ng), "u8", None
        elif case == "vit_fc1":
            w, a_dt, alpha = workloads.vit_fc1(), "u8", None
        elif case == "square_4096":
            w, a_dt, alpha = workloads.gemm_square(4096), "s8", None
        else:
            v = workloads.vitl_ptf(M=12608, K=4096, N=1024)
            xq = torch.from_numpy(v["x"]).to(device)
            Aq = torch.empty(v["x"].shape, dtype=torch.uint8, device=device)
            qnn.q_quantize(xq, Aq, "s8", qnn.qparams("sym", scale=torch.from_numpy(v["in_scale"]).to(device),
                                                     per_channel=True, axis=1))
            w = dict(A=Aq.cpu().numpy(), B=v["B"], s_w=v["s_w"], bias=v["bias"], s_a=v["s"], s_o=v["s_o"], z_a=0)
            a_dt, alpha = "s8", v["alpha"]
        Mm, Kk = w["A"].shape
        Nn = w["B"].shape[0]
        al = None if alpha is None else torch.from_numpy(alpha.astype(np.uint8)).to(device)
        g = gpu_setup_gemm(torch, qnn, w, a_dt, device, ptf=al)
        C = torch.empty((Mm, Nn), dtype=torch.uint8, device=device)
        epi = qnn.epilogue("requant", zp_term=None if al is not None else g["zp"], M=g["M"], Bq=g["Bq"],
                           ptf_max_shift=0 if alpha is None else int(alpha.max()))
        ws = None if getattr(args, "fused", False) else torch.empty(qnn.qnn_gemm_workspace_bytes(Mm, Kk), dtype=torch.uint8,
                                                 device=device)
        fn = lambda: qnn.qgemm_s8(g["A"], a_dt, g["Bp"], Mm, Nn, Kk, epi, C, workspace=ws,  # noqa: E731
                                  stream=stream)
    elif case in ("conv3x3", "conv1x1"):
        if case == "conv3x3":
            w, geom = workloads.conv_u4(), (64, 56, 56, 64, 64, 3, 1, 1)
        else:
            w = workloads.conv_u4(C=256, OC=64, F=1, pad=0, residual=False, tag=1)
            geom = (64, 56, 56, 256, 64, 1, 0, 1)
        Nb, H, W, C, OC, F, pad, st = geom
        gg = qnn.conv_geom(Nb, H, W, C, OC, F, F, (pad, pad), (st, st))
        Wd = torch.from_numpy(w["W"]).to(device)
        nb = qnn.qnn_conv_packed_w_bytes(gg, "s4")
        buf = torch.empty(nb + 1024, dtype=torch.uint8, device=device)
        off = (-buf.data_ptr()) % 1024
        Wp = buf[off:off + nb]
        cs = torch.empty(OC, dtype=torch.int32, device=device)
        qnn.qconv_prepack_w(Wd, "s4", gg, Wp, cs)
        zp = torch.empty(OC, dtype=torch.int32, device=device)
        Mv = torch.empty(OC, dtype=torch.float32, device=device)
        Bq = torch.empty(OC, dtype=torch.float32, device=device)
        qnn.q_fold_epilogue(OC, "u4", w["z_in"], cs, w["s_a"], torch.from_numpy(w["s_w"]).to(device),
                            w["s_o"], bias=torch.from_numpy(w["bias"]).to(device), zp_term=zp, M=Mv, Bq=Bq)
        I = torch.from_numpy(w["I"]).to(device)
        res = None if w["res"] is None else torch.from_numpy(w["res"]).to(device)
        R = float(np.float32(np.float32(w["s_r"]) / np.float32(w["s_o"])))
        epi = qnn.epilogue("requant", relu=True, out_dt="u4", zp_term=zp, M=Mv, Bq=Bq, residual=res,
                           res_dt="u4", z_res=w["z_res"], R=R)
        O = torch.empty((Nb, gg.OH, gg.OW, OC // 2), dtype=torch.uint8, device=device)
        ws = None if getattr(args, "fused", False) else torch.empty(qnn.qnn_conv_workspace_bytes(gg, "u4"),
                                                                     dtype=torch.uint8, device=device)
        fn = lambda: qnn.qconv_u4s4(I, w["z_in"], Wp, gg, epi, O, workspace=ws, stream=stream)  # noqa: E731
    elif case == "conv_u8zw":
        fn, _ = setup_conv_u8zw(torch, qnn, workloads, device, stream)
    elif case == "gemm_zw":
        fn, _ = setup_gemm_zw(torch, qnn, workloads, device, stream)
    elif case == "eltwise":
        R, C = 64 * 197, 768
        ea = workloads.device_uniform_s8((R, C), 91, device)
        eb = workloads.device_uniform_s8((R, C), 92, device)
        eo = torch.empty((R, C), dtype=torch.int8, device=device)
        fn = lambda: qnn.q_eltwise_s8("add", ea, eb, R * C, 0.5, eo, stream=stream)  # noqa: E731
    elif case == "dynquant":
        R, C = 64 * 197, 768
        xf = workloads.device_normal_f32((R, C), 93, device)
        eo = torch.empty((R, C), dtype=torch.int8, device=device)
        dsc = torch.empty(R, dtype=torch.float32, device=device)
        fn = lambda: qnn.q_quantize_rows_dynamic(xf, R, C, eo, dsc, stream=stream)  # noqa: E731
    elif case == "layernorm":
        wl = workloads.vit_layernorm()
        lx = torch.from_numpy(wl["x"]).to(device)
        la = torch.from_numpy(wl["alpha"]).to(device)
        lg, lb, lo = (torch.from_numpy(wl[k]).to(device) for k in ("gamma", "beta", "o"))
        R, C = wl["x"].shape
        ly = torch.empty((R, C), dtype=torch.int8, device=device)
        fn = lambda: qnn.q_int_layernorm(lx, R, C, wl["s"], lg, lb, lo, ly, alpha=la,  # noqa: E731
                                         alpha_max=int(wl["alpha"].max()), stream=stream)
    elif case in ("lis", "shift", "attn", "fused"):
        Bh, Lt, dh = 64 * 12, 197, 64
        xl = workloads.device_attention_logits(Bh * Lt, Lt, 1234, device)
        codes = torch.empty((Bh * Lt, Lt), dtype=torch.uint8, device=device)
        qnn.q_log_int_softmax(xl, Bh * Lt, Lt, workloads.ATTN_S, 4, codes, stream=stream)
        if case == "lis":
            fn = lambda: qnn.q_log_int_softmax(xl, Bh * Lt, Lt, workloads.ATTN_S, 4, codes,  # noqa: E731
                                               stream=stream)
        else:
            vq = workloads.device_uniform_s8((Bh, Lt, dh), 77, device)
            ov = torch.empty((Bh, Lt, dh), dtype=torch.int32, device=device)

            def fn():
                if case == "fused":
                    qnn.q_lis_attn_v(xl, workloads.ATTN_S, vq, Bh, Lt, Lt, dh, 4, ov, stream=stream)
                    return
                if case == "attn":
                    qnn.q_log_int_softmax(xl, Bh * Lt, Lt, workloads.ATTN_S, 4, codes, stream=stream)
                qnn.q_attn_shift_v(codes, vq, Bh, Lt, Lt, dh, 4, ov, stream=stream)
    else:
        raise SystemExit(f"unknown case {case}")
    t = time_steps(torch, fn, args.steps, args.warmup, flush, stream)
    st = qnn.qnn_check_device_error()
    print(json.dumps({"case": case, "steps": args.steps, "median_ms": statistics.median(t),
                      "status": qnn.status_string(st)}), flush=True)
    if st != qnn.QNN_OK:
        raise SystemExit(1)


def cpu_baseline_gemm(w, target_s=15.0):
    """The oracle (plain C, OpenMP over rows) on a sample of rows of the same GEMM."""
    from oracle import oracle
    oracle.build()
    A = w["A"].astype(np.int32)
    B = w["B"].astype(np.int32)
    N, K = B.shape
    cs = oracle.colsum(B)
    _, Mo, Bqo, _ = oracle.fold(cs, w["z_a"], w["s_a"], w["s_w"], w["s_o"], w["bias"])
    rows = 64
    t0 = time.perf_counter()
    acc = oracle.gemm_acc(A[:rows], B, w["z_a"])
    oracle.requant(acc, Mo, Bqo, "s8")
    dt = time.perf_counter() - t0
    rows = int(min(A.shape[0], max(64, rows * target_s / max(dt, 1e-6))))
    t0 = time.perf_counter()
    acc = oracle.gemm_acc(A[:rows], B, w["z_a"])
    oracle.requant(acc, Mo, Bqo, "s8")
    dt = time.perf_counter() - t0
    tops = 2.0 * rows * N * K / dt / 1e12
    return {"value": round(tops, 6), "unit": "TOPS", "cores": oracle.get_threads(), "kind": "oracle",
            "sample": f"first {rows} of {A.shape[0]} rows (x all {N} columns, K={K}), "
                      f"{dt:.1f} s; scaled to the metric's unit"}


def oracle_table(gpu_ms):
    """The oracle on the host cores for each workload: single-threaded and with
    OpenMP on every core available to the process (over output rows, pixels or
    channels).  Timed in full where the run is short enough; the largest GEMMs
    run on a leading sample of output rows and the time is scaled by the row
    count ("extrapolated").  gpu_ms: the GPU's time per call for the speedup."""
    from oracle import oracle
    from integer_quantized_nn_gb300 import workloads
    oracle.build()
    ncores = oracle.get_threads()
    out = {"cores": ncores, "entries": {}}

    def timed(fn, threads):
        oracle.set_threads(threads)
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    def record(name, work, unit, fn_rows, total_rows, rows_1, rows_n):
        e = {"work": work, "unit": unit}
        for tag, threads, rows in (("1thread", 1, rows_1), ("ncore", ncores, rows_n)):
            rows = min(rows, total_rows)
            dt = timed(lambda: fn_rows(rows), threads) * total_rows / rows
            e[f"s_{tag}"] = round(dt, 3)
            e[f"{unit}_{tag}"] = round(work / dt / (1e12 if unit == "TOPS" else 1e9), 6)
            e[f"timed_{tag}"] = ("full" if rows == total_rows else
                                 f"extrapolated from the first {rows} of {total_rows} output rows")
        if name in gpu_ms:
            e["gpu_ms"] = gpu_ms[name]
            e["gpu_speedup_vs_ncore"] = round(e["s_ncore"] * 1e3 / gpu_ms[name], 1)
        out["entries"][name] = e

    def gemm(name, A, B, z_a, alpha, s_a, s_w, s_o, bias, rows_1, rows_n):
        B32 = B.astype(np.int32)
        _, Mo, Bqo, _ = oracle.fold(oracle.colsum(B32), z_a, s_a, s_w, s_o, bias)

        def fn(r):
            oracle.requant(oracle.gemm_acc(A[:r], B32, z_a, alpha), Mo, Bqo, "s8")
        record(name, 2.0 * A.shape[0] * B.shape[0] * B.shape[1], "TOPS", fn, A.shape[0], rows_1, rows_n)

    w = workloads.gemm_sym()
    gemm("gemm_sym_256", w["A"].astype(np.int32), w["B"], 0, None, 1.0, w["s_w"], 1024.0, None, 256, 256)
    w = workloads.vit_fc1()
    gemm("vit_fc1", w["A"].astype(np.int32), w["B"], 128, None, w["s_a"], w["s_w"], w["s_o"], w["bias"],
         1024, 12608)
    for nm, (Kk, Nn) in workloads.VITL_SHAPES.items():
        v = workloads.vitl_ptf(M=12608, K=Kk, N=Nn)
        A = oracle.quantize(v["x"], oracle.SYM, "s8", scale=v["in_scale"], per_channel=True, axis=1)
        full = nm == "proj"
        gemm(f"vitl_{nm}_ptf", A, v["B"], 0, v["alpha"], v["s"], v["s_w"], v["s_o"], v["bias"],
             12608 if full else 64, 12608 if full else 64)
        del v, A
    for n, r1 in ((2048, 64), (4096, 64), (8192, 16), (16384, 8)):
        if n <= 8192:
            w = workloads.gemm_square(n)
            A, B = w["A"][:64].astype(np.int32), w["B"]
        else:
            g = np.random.default_rng(5160)
            A = g.integers(-128, 128, size=(64, n), dtype=np.int8).astype(np.int32)
            B = g.integers(-128, 128, size=(n, n), dtype=np.int8)
        e = int(math.ceil(math.log2(n))) + 7
        B32 = B.astype(np.int32)
        _, Mo, Bqo, _ = oracle.fold(oracle.colsum(B32), 0, 1.0, np.ones(n, np.float32), float(2.0 ** e))

        def fn(r, A=A, B32=B32, Mo=Mo, Bqo=Bqo):
            oracle.requant(oracle.gemm_acc(A[:r], B32, 0), Mo, Bqo, "s8")
        record(f"square_{n}", 2.0 * n ** 3, "TOPS", fn, n, r1, 64)
        del A, B, B32

    def conv(name, w, geom):
        Nb, H, W, C, OC, F, pad, st = geom
        Ic = oracle.unpack_nibbles(w["I"], signed=False)
        Wc = oracle.unpack_nibbles(w["W"], signed=True)
        _, Mo, Bqo, _ = oracle.fold(oracle.colsum(Wc.reshape(OC, -1)), w["z_in"], w["s_a"], w["s_w"], w["s_o"],
                                    w["bias"])
        OH = (H + 2 * pad - F) // st + 1
        OW = (W + 2 * pad - F) // st + 1
        res = None if w["res"] is None else oracle.unpack_nibbles(w["res"], signed=False).reshape(-1, OC)
        R = float(np.float32(np.float32(w["s_r"]) / np.float32(w["s_o"])))

        def fn(nimg):
            acc = oracle.conv_acc_direct(Ic[:nimg], Wc, w["z_in"], (pad, pad), (st, st))
            rr = None if res is None else res[:nimg * OH * OW]
            oracle.requant(acc, Mo, Bqo, "u4", relu=True, res=rr, z_res=w["z_res"], R=R)
        record(name, 2.0 * Nb * OH * OW * OC * C * F * F, "TOPS", fn, Nb, Nb, Nb)

    conv("conv3x3_u4s4_add_relu", workloads.conv_u4(), (64, 56, 56, 64, 64, 3, 1, 1))
    conv("conv1x1_u4s4_relu", workloads.conv_u4(C=256, OC=64, F=1, pad=0, residual=False, tag=1),
         (64, 56, 56, 256, 64, 1, 0, 1))

    q = workloads.quant_rows()
    record("quantize_rows_1GiB", 5.0 * q["x"].size, "GB/s",
           lambda r: oracle.quantize(q["x"][:r], oracle.SYM, "s8", scale=q["scale"][:r], per_channel=True, axis=0),
           q["x"].shape[0], q["x"].shape[0], q["x"].shape[0])
    oracle.set_threads(ncores)
    return out


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from integer_quantized_nn_gb300 import workloads
    from oracle import oracle
    oracle.build()
    M, K, N = 12608, 768, 3072
    w = workloads.vit_fc1(M=M, K=K, N=N)
    A = w["A"].astype(np.int32)
    B = w["B"].astype(np.int32)
    cs = oracle.colsum(B)
    _, Mo, Bqo, _ = oracle.fold(cs, w["z_a"], w["s_a"], w["s_w"], w["s_o"], w["bias"])
    # size the per-step sample so warmup + steps take about args.cpu_seconds * 4
    t0 = time.perf_counter()
    oracle.requant(oracle.gemm_acc(A[:16], B, w["z_a"]), Mo, Bqo, "s8")
    per_row = (time.perf_counter() - t0) / 16
    budget = 4.0 * args.cpu_seconds
    rows = int(max(1, min(M, budget / max(per_row, 1e-9) / max(1, args.steps + args.warmup))))
    rng = np.random.default_rng(0)

    def step(i):
        r0 = int(rng.integers(0, M - rows + 1))
        acc = oracle.gemm_acc(A[r0:r0 + rows], B, w["z_a"])
        oracle.requant(acc, Mo, Bqo, "s8")

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    ops = 2.0 * rows * N * K * args.steps
    v = ops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TOPS", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8 x s8 -> s32 (int64 C loops), requant to s8", "data": "synthetic",
        "config": {"workload": "ViT-B MLP fc1 qgemm_s8: u8 (Z=128) x s8 per-channel -> s8",
                   "M": M, "K": K, "N": N, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(v, 6), "unit": "TOPS", "cores": oracle.get_threads(),
                         "kind": "oracle",
                         "sample": f"{rows} consecutive rows per step (x all {N} columns, K={K})"},
        "e2e": {"value": round(v, 6), "unit": "TOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--extra-steps", type=int, default=20)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-oracle-table", action="store_true",
                    help="skip the per-workload single-thread / all-core oracle timings")
    ap.add_argument("--fused", action="store_true",
                    help="--case GEMMs / convs: no workspace (A re-encoded inside the kernel)")
    ap.add_argument("--case", default=None,
                    help="run one workload only (profiling): quantize, dequantize, vit_fc1, square_4096, "
                         "vitl_fc2, conv3x3, conv1x1, gemm:M:N:K (u8 x s8 -> s8), lis, shift, "
                         "attn (ViT-B b64 Log-Int-Softmax, shift product, both), fused (both in one kernel), layernorm, "
                         "eltwise, dynquant, conv_u8zw (3x3 u8 x u8 filters with zero points), "
                         "gemm_zw (ViT-B fc1 with u8 weights and zero points)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
