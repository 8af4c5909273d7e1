"""Benchmark of the 4-bit-weight GEMM hot path on GB300.

Workload (one "step"): the QQQ-style W4A8 per-channel sweep at N=8192,
K=21760 — one GEMM for each M in {1, 8, 32, 128, 512, 1024} (int8
activations with per-token fp32 scales, int4 weights with per-channel fp32
scales, fp16 output), the shape of the pytorch/ao PR #1113 "support W4A8
Marlin kernel" speedup sweep.  Weights are prepacked once (offline step,
timed separately under "prepack").  Every GEMM of a step reads its own
weight copy: ROTATE copies of the weights and activations rotate GEMM by
GEMM, so a copy is read again only after ROTATE - 1 other 89 MB copies
(more than 2x the 129 MB L2) have streamed through.

metric: TFLOP/s of the whole sweep (sum 2*M*N*K / step time).  The timed
region is `--steps` steps between barriers; it is repeated until at least
MIN_TIMED_S seconds of timed regions have run (so that the clocks sampled
during them mean something), and the step time is the median over repeats.
"sweep" has the per-M breakdown (isolated graph replays of one GEMM: us,
TFLOP/s, weight GB/s, roofline fraction against the burst peaks); "extra"
has the same for the other workloads: W4A8 g128 (N=8192, K=21760), W4A16
decode on the Llama-3-8B linear shapes and W4A16 prefill on the Llama-3-70B
MLP shapes.  --impl reference times the CPU oracle (plain fp64/int64 C) on a
bounded sample of the same workload.

Multi-GPU (torchrun): replicas only; every rank runs the same sweep on its
own GPU and value = all ranks' flops / the slowest rank's time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import w4synth  # noqa: E402

N, K = w4synth.QQQ_N, w4synth.QQQ_K
M_SWEEP = w4synth.QQQ_CH_M
ROTATE = 8            # weight + activation copies of the step, rotated GEMM by GEMM
L2_BYTES = 129 * 2 ** 20
MIN_TIMED_S = 2.0     # repeat the K-step timed region until this much has run
METRIC = "int4-weight GEMM TFLOP/s & weight GB/s vs M (N=8192,K=21760), % roofline"
UNIT = "TFLOP/s"
WORKLOAD = "W4A8 QQQ per-channel sweep M in {1,8,32,128,512,1024}, N=8192, K=21760"


def flops(M, n=N, k=K):
    return 2.0 * M * n * k


def weight_bytes():
    return K * N // 2 + 4 * N  # packed int4 + fp32 channel scales


def algo_bytes(M):
    # weights + int8 activations + token scales + fp16 output
    return weight_bytes() + M * K + 4 * M + 2 * M * N


def w4a8_g128_bytes(M, n=N, k=K):
    """W4A8 per-group: packed int4 + int8 group scales + fp32 channel scales,
    int8 activations + token scales, fp16 output."""
    return k * n // 2 + (k // 128) * n + 4 * n + M * k + 4 * M + 2 * M * n


def w4a16_bytes(M, n, k, zeros, gs=128):
    """W4A16: packed int4 + 16-bit scales (+ zero-points), 16-bit activations
    and output."""
    G = k // gs
    return k * n // 2 + G * n * 2 * (2 if zeros else 1) + M * k * 2 + M * n * 2


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"],
                    bf16_sus=p.get("bf16_tflops_sustained", p["bf16_tflops"]), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def roofline_entry(us, fl, nbytes, pk, tc_ratio=1.0):
    """Roofline of one isolated launch: the larger of the HBM time of its
    algorithmic bytes and the tensor time of its flops (burst bf16 peak,
    times tc_ratio for other MMA kinds: 2 for fp8, the nominal 4.5 / 2.25
    PFLOP/s ratio), over the measured time."""
    t_hbm = nbytes / (pk["hbm"] * 1e9)
    t_tc = fl / (pk["bf16"] * tc_ratio * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    return {"us": round(us, 2), "tflops": round(fl / (us * 1e-6) / 1e12, 1),
            "gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "bound": bound,
            "roofline_frac": round(max(t_hbm, t_tc) / (us * 1e-6), 3)}


def measured_traffic(kernel, M):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
        if not rec or rec.get("M") != M:
            return None
        with open(os.path.join(ROOT, rec["src"]), "rb") as f:
            sha = hashlib.sha1(f.read()).hexdigest()
        return rec["dram_bytes_per_launch"] if sha.startswith(rec["src_sha1_prefix"]) else None
    except (OSError, ValueError, KeyError):
        return None


def slowest_rank_ms(local_ms, world, device):
    """The job's time: the slowest rank's (ms), returned on every rank."""
    if world <= 1:
        return local_ms
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(step_flops, world, ms_per_step):
    """Whole-job throughput: every rank's flops over the slowest rank's time."""
    return step_flops * world / (ms_per_step * 1e-3) / 1e12


def rotation(step, j, nper=len(M_SWEEP), copies=ROTATE):
    """Copy read by GEMM j of step `step`: consecutive GEMMs read different
    copies, and a copy comes back only after copies - 1 others."""
    return (step * nper + j) % copies


def rotation_period(nper=len(M_SWEEP), copies=ROTATE):
    """Steps after which the rotation pattern repeats (graphs to capture)."""
    return copies // math.gcd(nper, copies)


def copies_for(nbytes, minimum=2):
    """Copies of a problem whose rotation streams more than 2x L2 between two
    reads of the same copy."""
    return max(minimum, 2 * L2_BYTES // max(nbytes, 1) + 2)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen between t0 and t1
        (time.time() values; all samples when not given)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clocks(out, t0, t1)


def parse_clocks(text, t0=None, t1=None):
    """Median SM clock, the largest max clock, the largest power draw and the
    throttle reasons seen in nvidia-smi CSV lines (FIELDS order) between t0
    and t1."""
    import datetime

    sms, maxes, power, reasons = [], [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            sm, mx = float(parts[1]), float(parts[2])
        except ValueError:
            continue
        if t0 is not None and not (t0 <= ts <= t1):
            continue
        sms.append(sm)
        maxes.append(mx)
        try:
            power.append(float(parts[3]))
        except ValueError:
            pass
        for nm, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(nm)
    if not sms:
        return None
    return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
            "reasons": sorted(reasons), "samples": len(sms),
            "power_w_max": max(power) if power else None}


def make_inputs(dev):
    """ROTATE copies of every input of the step, resident in HBM: one seeded
    weight (prepacked) and one set of activations per M, cloned so that each
    copy lives at its own addresses."""
    import int4_weight_mixed_gb300 as w4

    e = w4synth.gen_w4a8(1, N, K, group_size=-1, seed=100)
    w_dev = e["w"].to(dev)
    b0 = w4.prepack_B(w_dev, e["wtype"], e["layout"], K, N)
    del w_dev
    acts0 = {}
    for M in M_SWEEP:
        x = w4synth.gen_w4a8(M, 8, K, seed=1000 + M)  # its a [M,K] and s_tok [M]
        acts0[M] = (x["a"].to(dev), x["s_tok"].to(dev))
    s_ch = e["s_ch"].to(dev)
    sets = []
    for r in range(ROTATE):
        b = b0 if r == 0 else b0.clone()
        acts = acts0 if r == 0 else {M: (a.clone(), s.clone()) for M, (a, s) in acts0.items()}
        sets.append(dict(b=b, s_ch=s_ch if r == 0 else s_ch.clone(), acts=acts, wq=e["w"],
                         wtype=e["wtype"]))
    return sets


def launches_per_gemm(name):
    """Kernels of this library one GEMM launches: the streamed skinny-M
    schedule three (activation staging, GEMM, reduction); the tensor-core W4A8
    schedule two (int8->bf16 staging, GEMM); the others one."""
    return 3 if name.startswith("ds") else 2 if name.startswith("tc") else 1


def launches_per_step(w4):
    names = w4.schedule_names()
    return sum(launches_per_gemm(names[w4.default_schedule(M, N, K, torch.int8, -1)])
               for M in M_SWEEP)


def capture(fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


CHAIN = 16  # GEMMs per timing graph


def time_isolated(fns, reps, stream, eager=False):
    """Microseconds per GEMM of one shape: one graph holding CHAIN (or more)
    back-to-back launches that cycle through the rotated copies, as a decode
    step runs them (launch gaps between graphs and host launch costs stay out
    of the figure), replayed between CUDA events on the launching stream;
    `reps` GEMMs in all (at least two replays)."""
    for f in fns:  # eager first: kernel attributes are set outside any capture
        f()
    torch.cuda.synchronize()
    L = max(CHAIN, len(fns))
    seq = [fns[i % len(fns)] for i in range(L)]
    if eager:  # plain launches (profilers); host-bound for small GEMMs
        run = lambda: [f() for f in seq]
    else:
        g = capture(lambda: [f() for f in seq])
        run = g.replay
    run()
    torch.cuda.synchronize()
    n_rep = max(2, reps // L)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(n_rep):
        run()
    a1.record(stream)
    torch.cuda.synchronize()
    return a0.elapsed_time(a1) * 1e3 / (n_rep * L)


def extra_workloads(w4, dev, stream, pk, reps, eager=False):
    """The other configurations, one isolated GEMM at a time (default
    schedule), each with its roofline fraction: W4A8 per-group g128 at N=8192,
    K=21760; W4A16 decode on the Llama-3-8B linear shapes (uint4 + bf16
    zero-points); W4A16 prefill on the Llama-3-70B MLP shapes at M=4096."""
    names = w4.schedule_names()
    out = {"w4a8_g128_n8192_k21760": [], "w4a16_decode_llama3_8b": [],
           "w4a16_prefill_llama3_70b": []}

    # W4A8 g128
    e = w4synth.gen_w4a8(1, N, K, group_size=128, seed=200)
    b = w4.prepack_B(e["w"].to(dev), e["wtype"], e["layout"], K, N)
    sg, s_ch = e["sg"].to(dev), e["s_ch"].to(dev)
    for M in w4synth.QQQ_G128_M:
        x = w4synth.gen_w4a8(M, 8, K, seed=300 + M)
        R = copies_for(w4a8_g128_bytes(M))
        cp = [(b, sg, s_ch, x["a"].to(dev), x["s_tok"].to(dev))]
        cp += [tuple(t.clone() for t in cp[0]) for _ in range(R - 1)]
        o = torch.empty((M, N), dtype=torch.float16, device=dev)
        ws = w4.workspace(dev, w4.workspace_size(M, N, K, torch.int8, 128))
        fns = [lambda c=c, M=M: w4.gemm(c[3], c[0], e["wtype"], N, scales=c[1], group_size=128,
                                       token_scales=c[4], channel_scales=c[2], out=o, ws=ws)
               for c in cp]
        us = time_isolated(fns, reps, stream, eager)
        ent = roofline_entry(us, flops(M), w4a8_g128_bytes(M), pk)
        ent.update(M=M, schedule=names[w4.default_schedule(M, N, K, torch.int8, 128)])
        out["w4a8_g128_n8192_k21760"].append(ent)
        del cp, fns
    del b, sg, s_ch

    # W4A8 with fp8 (E4M3) activations, per-channel, at the QQQ sweep shape
    out["w4a8_fp8_n8192_k21760"] = []
    e = w4synth.gen_w4a8_fp8(1, N, K, seed=250)
    b = w4.prepack_B(e["w"].to(dev), e["wtype"], e["layout"], K, N)
    s_ch = e["s_ch"].to(dev)
    for M in M_SWEEP:
        x = w4synth.gen_w4a8_fp8(M, 8, K, seed=260 + M)
        nb = algo_bytes(M)
        R = copies_for(nb)
        cp = [(b, x["a"].to(dev).view(torch.float8_e4m3fn), x["s_tok"].to(dev))]
        cp += [tuple(t.clone() for t in cp[0]) for _ in range(R - 1)]
        o = torch.empty((M, N), dtype=torch.float16, device=dev)
        ws = w4.workspace(dev, w4.workspace_size(M, N, K, torch.float8_e4m3fn, -1))
        fns = [lambda c=c: w4.gemm(c[1], c[0], e["wtype"], N, group_size=-1, token_scales=c[2],
                                   channel_scales=s_ch, out=o, ws=ws) for c in cp]
        us = time_isolated(fns, reps, stream, eager)
        sch = names[w4.default_schedule(M, N, K, torch.float8_e4m3fn, -1)]
        # kind::f8f6f4 on the tensor-core schedule; the clustered decode
        # schedule runs fp16 mma.sync
        ent = roofline_entry(us, flops(M), nb, pk, tc_ratio=2.0 if sch.startswith("tc") else 1.0)
        ent.update(M=M, schedule=sch)
        out["w4a8_fp8_n8192_k21760"].append(ent)
        del cp, fns
    del b, s_ch

    # W4A16 decode, Llama-3-8B shapes (uint4 + pre-scaled bf16 zero-points, g128)
    for (n, k) in w4synth.DECODE_SHAPES:
        d = w4synth.gen_w4a16(max(w4synth.DECODE_M), n, k, act_dtype=torch.bfloat16,
                              wtype=w4synth.UINT4, layout=w4synth.NK_EXLLAMA, group_size=128,
                              zeros=True, seed=n + k)
        b = w4.prepack_B(d["w"].to(dev), d["wtype"], d["layout"], k, n)
        s, z, a_all = d["s"].to(dev), d["z"].to(dev), d["a"].to(dev)
        for M in w4synth.DECODE_M:
            nb = w4a16_bytes(M, n, k, zeros=True)
            R = copies_for(nb)
            base = (b, s, z, a_all[:M].contiguous())
            cp = [base] + [tuple(t.clone() for t in base) for _ in range(R - 1)]
            o = torch.empty((M, n), dtype=torch.bfloat16, device=dev)
            ws = w4.workspace(dev, w4.workspace_size(M, n, k, torch.bfloat16, 128))
            fns = [lambda c=c: w4.gemm(c[3], c[0], d["wtype"], n, scales=c[1], zeros=c[2],
                                       group_size=128, out=o, ws=ws) for c in cp]
            us = time_isolated(fns, reps, stream, eager)
            ent = roofline_entry(us, flops(M, n, k), nb, pk)
            ent.update(M=M, N=n, K=k, copies=R,
                       schedule=names[w4.default_schedule(M, n, k, torch.bfloat16, 128)])
            out["w4a16_decode_llama3_8b"].append(ent)
            del cp, fns
        del b, s, z, a_all

    # W4A16 prefill, Llama-3-70B MLP shapes at M=4096 (uint4b8, bf16 scales, g128)
    M = 4096
    for (n, k) in w4synth.PREFILL_SHAPES:
        d = w4synth.gen_w4a16(M, n, k, act_dtype=torch.bfloat16, wtype=w4synth.UINT4B8,
                              layout=w4synth.NK_EXLLAMA, group_size=128, zeros=False,
                              seed=n + k)
        b = w4.prepack_B(d["w"].to(dev), d["wtype"], d["layout"], k, n)
        base = (b, d["s"].to(dev), d["a"].to(dev))
        cp = [base, tuple(t.clone() for t in base)]
        o = torch.empty((M, n), dtype=torch.bfloat16, device=dev)
        ws = w4.workspace(dev, w4.workspace_size(M, n, k, torch.bfloat16, 128))
        fns = [lambda c=c: w4.gemm(c[2], c[0], d["wtype"], n, scales=c[1], group_size=128, out=o,
                                   ws=ws)
               for c in cp]
        us = time_isolated(fns, max(5, reps // 4), stream, eager)
        ent = roofline_entry(us, flops(M, n, k), w4a16_bytes(M, n, k, zeros=False), pk)
        ent.update(M=M, N=n, K=k, schedule=names[w4.default_schedule(M, n, k, torch.bfloat16, 128)])
        out["w4a16_prefill_llama3_70b"].append(ent)
        del cp, fns, b, base
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import int4_weight_mixed_gb300 as w4

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w4.load()
    pk = peaks()
    sets = make_inputs(dev)
    outs = {M: torch.empty((M, N), dtype=torch.float16, device=dev) for M in M_SWEEP}
    ws = w4.workspace(dev, w4.workspace_size(max(M_SWEEP), N, K, torch.int8, -1))
    stream = torch.cuda.current_stream(dev)

    def gemm(r, M):
        st = sets[r]
        a, s_tok = st["acts"][M]
        w4.gemm(a, st["b"], st["wtype"], N, scales=None, group_size=-1, token_scales=s_tok,
                channel_scales=st["s_ch"], out=outs[M], ws=ws)

    def step(i):
        for j, M in enumerate(M_SWEEP):
            gemm(rotation(i, j), M)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # prepack timing (offline step, not part of a step)
    wq = sets[0]["wq"].to(dev)
    pre_b = torch.empty_like(sets[0]["b"])
    for _ in range(3):
        w4.prepack_B(wq, sets[0]["wtype"], w4synth.NK_EXLLAMA, K, N, out=pre_b)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(10):
        w4.prepack_B(wq, sets[0]["wtype"], w4synth.NK_EXLLAMA, K, N, out=pre_b)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    prepack_us = e0.elapsed_time(e1) * 1e3 / 10
    del wq, pre_b

    # per-token int8 quantization of fp16 activations at the largest sweep M
    # (the step before a W4A8 GEMM; timed beside the step, not inside it):
    # 4 input copies > L2, 2 bytes read + 1 written per element
    qm = max(M_SWEEP)
    qa = [w4synth.gen_act16(qm, K, torch.float16, seed=50 + r).to(dev) for r in range(4)]
    qo = [(torch.empty(qm, K, dtype=torch.int8, device=dev),
           torch.empty(qm, dtype=torch.float32, device=dev)) for _ in range(4)]
    for r in range(3):
        w4.quantize_per_token(qa[r % 4], out=qo[r % 4][0], scales=qo[r % 4][1])
    e0.record(stream)
    for r in range(20):
        w4.quantize_per_token(qa[r % 4], out=qo[r % 4][0], scales=qo[r % 4][1])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    quant_us = e0.elapsed_time(e1) * 1e3 / 20
    quant_gbs = (3 * qm * K + 4 * qm) / (quant_us * 1e-6) / 1e9
    # the same for E4M3 codes
    qo8 = [(torch.empty(qm, K, dtype=torch.float8_e4m3fn, device=dev), qo[r][1]) for r in range(4)]
    for r in range(3):
        w4.quantize_per_token_fp8(qa[r % 4], out=qo8[r % 4][0], scales=qo8[r % 4][1])
    e0.record(stream)
    for r in range(20):
        w4.quantize_per_token_fp8(qa[r % 4], out=qo8[r % 4][0], scales=qo8[r % 4][1])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    quant8_us = e0.elapsed_time(e1) * 1e3 / 20
    # W4A8 with the per-token quantization inside the call (fp16 activations
    # in), against quantize + gemm, at the largest sweep M
    dyn = {}
    b0, sch0 = sets[0]["b"], sets[0]["s_ch"]
    o_d = torch.empty((qm, N), dtype=torch.float16, device=dev)
    ws_d = w4.workspace(dev, int(w4.load().w4_gemm_dynamic_workspace_size(qm, N, K, w4.S8, -1)))
    for name, fn in (
            ("fused", lambda r: w4.gemm_dynamic(qa[r % 4], sets[r % ROTATE]["b"], sets[0]["wtype"],
                                                N, torch.int8, group_size=-1,
                                                channel_scales=sch0, out=o_d, ws=ws_d)),
            ("two_step", lambda r: w4.gemm(*w4.quantize_per_token(qa[r % 4], out=qo[r % 4][0],
                                                                  scales=qo[r % 4][1])[:1],
                                           sets[r % ROTATE]["b"], sets[0]["wtype"], N,
                                           group_size=-1, token_scales=qo[r % 4][1],
                                           channel_scales=sch0, out=o_d, ws=ws_d))):
        for r in range(3):
            fn(r)
        e0.record(stream)
        for r in range(10):
            fn(r)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        dyn[name] = round(e0.elapsed_time(e1) * 1e3 / 10, 1)
    del qa, qo, qo8, o_d

    # eager warm-up (sets kernel attributes), then one graph per step of the
    # rotation pattern
    period = rotation_period()
    for i in range(args.warmup):
        step(i)
    barrier()
    if args.eager:  # plain launches (for profilers that do not follow graphs)
        class _Eager:
            def __init__(self, i):
                self.i = i

            def replay(self):
                step(self.i)
        step_graphs = [_Eager(i) for i in range(period)]
    else:
        step_graphs = [capture(lambda i=i: step(i)) for i in range(period)]
    for i in range(args.warmup):
        step_graphs[i % period].replay()
    barrier()

    # timed region: K steps of the whole sweep, graph replays on one stream,
    # repeated until MIN_TIMED_S of timed regions have run
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    rep_ms = []
    timed_s = 0.0
    wall0 = time.time()
    while True:
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        t_start.record(stream)
        for i in range(args.steps):
            step_graphs[i % period].replay()
        t_end.record(stream)
        barrier()
        ms = t_start.elapsed_time(t_end)
        rep_ms.append(ms)
        timed_s += ms * 1e-3
        if timed_s >= args.min_timed_s or len(rep_ms) >= 100000:
            break
    wall1 = time.time()
    time.sleep(0.2)
    clk = clocks.stop(wall0, wall1)
    total_ms = slowest_rank_ms(statistics.median(rep_ms), world, dev)

    # per-M launch durations: graphs of one GEMM per rotated copy, events on
    # the launching stream around `reps` replays
    per_m = {}
    reps = max(8, min(args.steps, 100))
    for M in M_SWEEP:
        per_m[M] = time_isolated([lambda r=r, M=M: gemm(r, M) for r in range(ROTATE)], reps,
                                 stream, args.eager)
    if w4.check_status(ws) != w4.OK:
        raise RuntimeError("a device-side wait timed out during the benchmark")

    extra = None
    if not args.skip_extra:
        extra = extra_workloads(w4, dev, stream, pk, reps, args.eager)

    # end-to-end through the public API from pinned host buffers
    e2e = None
    if rank == 0 or world > 1:
        host_a = {M: sets[0]["acts"][M][0].cpu().pin_memory() for M in M_SWEEP}
        host_s = {M: sets[0]["acts"][M][1].cpu().pin_memory() for M in M_SWEEP}
        host_o = {M: torch.empty((M, N), dtype=torch.float16).pin_memory() for M in M_SWEEP}
        h2d = sum(host_a[M].numel() + 4 * host_s[M].numel() for M in M_SWEEP)
        d2h = sum(2 * M * N for M in M_SWEEP)
        e2e_steps = max(3, min(args.steps, 50))
        # Copies on two more streams (one per direction, so that both copy
        # engines run) overlap the GEMMs: the inputs of the next M go in while
        # the current GEMM runs, and each result comes back while the next GEMM
        # runs. Two sets of device buffers, used by alternate steps, let a
        # step's GEMMs start while the previous step's last result is still
        # being copied back (allocated once, outside the timing).  The weights
        # rotate GEMM by GEMM as in the device-timed step.
        h2d_stream = torch.cuda.Stream(device=dev)
        d2h_stream = torch.cuda.Stream(device=dev)
        bufs = [dict(a={M: torch.empty_like(host_a[M], device=dev) for M in M_SWEEP},
                     s={M: torch.empty_like(host_s[M], device=dev) for M in M_SWEEP},
                     o={M: torch.empty((M, N), dtype=torch.float16, device=dev) for M in M_SWEEP},
                     free=None)
                for _ in range(2)]
        ev_in = {M: torch.cuda.Event() for M in M_SWEEP}
        ev_out = {M: torch.cuda.Event() for M in M_SWEEP}
        step_no = [0]

        def e2e_step():
            i = step_no[0]
            b = bufs[i % 2]
            step_no[0] += 1
            with torch.cuda.stream(h2d_stream):
                if b["free"] is not None:  # this set's previous GEMMs and copies are done
                    h2d_stream.wait_event(b["free"])
                for M in M_SWEEP:
                    b["a"][M].copy_(host_a[M], non_blocking=True)
                    b["s"][M].copy_(host_s[M], non_blocking=True)
                    ev_in[M].record(h2d_stream)
            for j, M in enumerate(M_SWEEP):
                wset = sets[rotation(i, j)]
                stream.wait_event(ev_in[M])
                w4.gemm(b["a"][M], wset["b"], wset["wtype"], N, scales=None,
                        group_size=-1, token_scales=b["s"][M], channel_scales=wset["s_ch"],
                        out=b["o"][M], ws=ws)
                ev_out[M].record(stream)
            with torch.cuda.stream(d2h_stream):
                for M in M_SWEEP:
                    d2h_stream.wait_event(ev_out[M])
                    host_o[M].copy_(b["o"][M], non_blocking=True)
                b["free"] = torch.cuda.Event()
                b["free"].record(d2h_stream)

        for _ in range(3):
            e2e_step()
        barrier()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        h0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        host_ms = (time.perf_counter() - h0) * 1e3 / e2e_steps  # enqueueing, on the host
        stream.wait_stream(d2h_stream)  # the last results are back on the host
        x1.record(stream)
        barrier()
        e2e_ms = slowest_rank_ms(x0.elapsed_time(x1) / e2e_steps, world, dev)
        e2e = {"value": job_tflops(sum(flops(M) for M in M_SWEEP), world, e2e_ms),
               "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "host_enqueue_ms_per_step": round(host_ms, 4)}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    names = w4.schedule_names()
    step_flops = sum(flops(M) for M in M_SWEEP)
    ms_per_step = total_ms / args.steps
    value = job_tflops(step_flops, world, ms_per_step)
    sweep = []
    for M in M_SWEEP:
        ent = roofline_entry(per_m[M], flops(M), algo_bytes(M), pk)
        ent["weight_gbs"] = round(weight_bytes() / (per_m[M] * 1e-6) / 1e9, 1)
        ent["M"] = M
        ent["schedule"] = names[w4.default_schedule(M, N, K, torch.int8, -1)]
        sweep.append(ent)
    # dominant kernel: the largest share of the step
    dom = max(M_SWEEP, key=lambda M: per_m[M])
    dom_us = per_m[dom]
    dom_ent = next(e for e in sweep if e["M"] == dom)
    pair = dom_ent["schedule"].startswith("tc") and "p_" in dom_ent["schedule"]
    kname = (f"tc_gemm_kernel<W4A8{', CTA pairs' if pair else ''}> ({dom_ent['schedule']}, "
             "+ its int8->bf16 staging launch)"
             if dom_ent["schedule"].startswith("tc") else f"{dom_ent['schedule']} launches")
    if dom_ent["bound"] == "tensor":
        roofline = {"kernel": kname, "M": dom, "bound": "tensor",
                    "achieved": round(flops(dom) / (dom_us * 1e-6) / 1e12, 1),
                    "peak": pk["bf16"], "unit": "TFLOP/s",
                    "peak_source": f"{pk['src']} bf16 dense, burst (isolated graph replays of "
                                   "this GEMM, ~30 ms each)"}
    else:
        roofline = {"kernel": kname, "M": dom, "bound": "hbm",
                    "achieved": round(algo_bytes(dom) / (dom_us * 1e-6) / 1e9, 1),
                    "peak": pk["hbm"], "unit": "GB/s", "peak_source": f"{pk['src']} HBM copy"}
    roofline["traffic"] = measured_traffic(
        "tc_gemm_kernel<W4A8, CTA pairs>" if pair else "tc_gemm_kernel<W4A8>", dom)
    roofline["frac"] = round(roofline["achieved"] / roofline["peak"], 3)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "l2": f"{ROTATE} weight+activation copies rotated GEMM by GEMM "
                         f"({ROTATE - 1} x 89 MB between two reads of a copy > 2x L2)",
                   "timing": f"{len(rep_ms)} repeats of the {args.steps}-step timed region "
                             f"({timed_s:.2f} s timed); median repeat",
                   "arith": "int8 x int4 exact on bf16 tensor cores, fp32 chunks drained "
                            "to int32, fp16 epilogue",
                   "parallelism": f"replicas x{world}"},
        "sweep": sweep, "roofline": roofline, "e2e": e2e, "extra": extra,
        "prepack": {"us": round(prepack_us, 1),
                    "gbs": round(2 * K * N // 2 / (prepack_us * 1e-6) / 1e9, 1)},
        "quantize": {"kernel": "quant2_kernel<fp16, int8>", "M": qm, "K": K,
                     "us": round(quant_us, 2), "gbs": round(quant_gbs, 1), "bound": "hbm",
                     "frac": round(quant_gbs / pk["hbm"], 3),
                     "fp8_us": round(quant8_us, 2),
                     "fp8_frac": round((3 * qm * K + 4 * qm) / (quant8_us * 1e-6) / 1e9 / pk["hbm"], 3)},
        "dynamic_w4a8_m1024_us": dyn,
        "gpu_launches": launches_per_step(w4) * args.steps * len(rep_ms),
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(target_s=args.cpu_seconds)
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_single(args):
    """One GEMM (M = args.single) of the sweep shape or of --shape N,K, eager
    launches: the small case for ncu captures (one weight copy).  --act
    int8: W4A8 (per-channel, or --group-size); fp8: W4A8 with E4M3
    activations; bf16: W4A16 uint4 with bf16 zero-points, group 128."""
    import int4_weight_mixed_gb300 as w4

    dev = torch.device("cuda", 0)
    M = args.single
    n, k = (int(x) for x in args.shape.split(","))
    gs = args.group_size
    if args.act == "bf16":
        d = w4synth.gen_w4a16(M, n, k, act_dtype=torch.bfloat16, wtype=w4synth.UINT4,
                              group_size=128, zeros=True, seed=0)
        b = w4.prepack_B(d["w"].to(dev), d["wtype"], d["layout"], k, n)
        a, s, z = d["a"].to(dev), d["s"].to(dev), d["z"].to(dev)
        ws = w4.workspace(dev, w4.workspace_size(M, n, k, torch.bfloat16, 128))
        out = torch.empty((M, n), dtype=torch.bfloat16, device=dev)
        call = lambda: w4.gemm(a, b, d["wtype"], n, scales=s, zeros=z, group_size=128, out=out,
                               ws=ws, schedule=args.schedule)
    else:
        fp8 = args.act == "fp8"
        e = (w4synth.gen_w4a8_fp8(M, n, k, seed=0) if fp8
             else w4synth.gen_w4a8(M, n, k, group_size=gs, seed=0))
        b = w4.prepack_B(e["w"].to(dev), e["wtype"], e["layout"], k, n)
        a = e["a"].to(dev).view(torch.float8_e4m3fn) if fp8 else e["a"].to(dev)
        s_tok, s_ch = e["s_tok"].to(dev), e["s_ch"].to(dev)
        sg = None if fp8 or e["sg"] is None else e["sg"].to(dev)
        ws = w4.workspace(dev, w4.workspace_size(M, n, k, a.dtype, gs))
        out = torch.empty((M, n), dtype=torch.float16, device=dev)
        call = lambda: w4.gemm(a, b, e["wtype"], n, scales=sg, group_size=gs, token_scales=s_tok,
                               channel_scales=s_ch, out=out, ws=ws, schedule=args.schedule)
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    st = w4.check_status(ws)
    print(json.dumps({"single_M": M, "N": n, "K": k, "act": args.act, "group_size": gs,
                      "launches": args.warmup + args.steps, "status": st}))
    if st != w4.OK:
        sys.exit(1)


def run_launch_list(args):
    """Only the step: W warm-up then K steps of the sweep, eager launches
    (for an ncu launch list: 15 launches of this library per step)."""
    import int4_weight_mixed_gb300 as w4

    dev = torch.device("cuda", 0)
    w4.load()
    sets = make_inputs(dev)
    outs = {M: torch.empty((M, N), dtype=torch.float16, device=dev) for M in M_SWEEP}
    ws = w4.workspace(dev, w4.workspace_size(max(M_SWEEP), N, K, torch.int8, -1))
    for i in range(args.warmup + args.steps):
        for j, M in enumerate(M_SWEEP):
            st = sets[rotation(i, j)]
            a, s_tok = st["acts"][M]
            w4.gemm(a, st["b"], st["wtype"], N, scales=None, group_size=-1, token_scales=s_tok,
                    channel_scales=st["s_ch"], out=outs[M], ws=ws)
    torch.cuda.synchronize()
    print(json.dumps({"launch_list_steps": args.steps, "warmup": args.warmup,
                      "launches_per_step": launches_per_step(w4)}))


def run_quant_single(args):
    """Per-token int8 quantization of fp16 activations [M = args.quant_single,
    K], eager launches: the small case for ncu captures (one input copy)."""
    import int4_weight_mixed_gb300 as w4

    dev = torch.device("cuda", 0)
    M = args.quant_single
    a = w4synth.gen_act16(M, K, torch.float16, seed=50).to(dev)
    q = torch.empty(M, K, dtype=torch.int8, device=dev)
    s = torch.empty(M, dtype=torch.float32, device=dev)
    for _ in range(args.warmup + args.steps):
        w4.quantize_per_token(a, out=q, scales=s)
    torch.cuda.synchronize()
    print(json.dumps({"quant_M": M, "K": K, "launches": args.warmup + args.steps}))


def oracle_sample(rows_per_m, cols, seed=0):
    """Time the oracle on rows_per_m sampled rows x `cols` columns of every
    M of the sweep (full K).  Returns (seconds, flops)."""
    import oracle

    e = w4synth.gen_w4a8(1, N, K, group_size=-1, seed=seed)
    total_flops, total_s = 0.0, 0.0
    for M in M_SWEEP:
        g = torch.Generator().manual_seed(M)
        rows_n = min(rows_per_m, M)
        a = torch.randint(-127, 128, (rows_n, K), generator=g, dtype=torch.int32).to(torch.int8)
        rows = np.repeat(np.arange(rows_n), cols.size)
        cc = np.tile(cols, rows_n)
        t0 = time.perf_counter()
        acc = oracle.w4a8_elems(a, e["w"], e["layout"], e["wtype"], None, -1, K, N, rows, cc)
        oracle.w4a8_scale(acc, rows, cc, np.ones(rows_n), e["s_ch"])
        total_s += time.perf_counter() - t0
        total_flops += 2.0 * K * rows.size
    return total_s, total_flops


def cpu_baseline(target_s=10.0):
    """The oracle, as it stands, on a bounded sample sized to ~target_s."""
    import oracle

    cols = np.arange(0, N, 64, dtype=np.int64)  # 128 columns
    s, f = oracle_sample(1, cols)
    rate = f / max(s, 1e-6)
    per_row = 2.0 * K * N  # flops of one row x all columns
    rows = 1
    while rows < 64 and (rows * 2) * per_row * 5 / rate <= target_s:
        rows *= 2
    cols2 = np.arange(N, dtype=np.int64)
    s2, f2 = oracle_sample(rows, cols2)
    return {"value": f2 / s2 / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"min(M,{rows}) rows of each M x all {N} columns x full K={K} "
                      f"({f2 / 2:.3g} MACs in {s2:.1f} s)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    cols = np.arange(0, N, 512, dtype=np.int64)  # 16 columns per M per step
    for _ in range(args.warmup):
        oracle_sample(1, cols[:2])
    times, fl = [], 0.0
    for i in range(args.steps):
        s, f = oracle_sample(1, cols, seed=i % 2)
        times.append(s)
        fl = f
    ms = 1e3 * sum(times) / len(times)
    value = fl / (ms * 1e-3) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": "per step: 1 row of "
                                            "each M x 16 columns x full K"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": "1 row of each M x 16 columns x full K per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--min-timed-s", type=float, default=MIN_TIMED_S,
                    help="repeat the K-step timed region until this many seconds have run")
    ap.add_argument("--skip-extra", action="store_true",
                    help="leave out the other workloads (shorter launch lists)")
    ap.add_argument("--single", type=int, default=0, help="run only the GEMM with this M")
    ap.add_argument("--group-size", type=int, default=-1, help="group size of --single")
    ap.add_argument("--act", default="int8", choices=["int8", "fp8", "bf16"],
                    help="activations of --single")
    ap.add_argument("--shape", default=f"{N},{K}", help="N,K of --single")
    ap.add_argument("--launch-list", action="store_true",
                    help="run only warm-up + K eager steps (ncu launch lists)")
    ap.add_argument("--schedule", type=int, default=-1)
    ap.add_argument("--quant-single", type=int, default=0,
                    help="run only the per-token quantization of this many rows")
    ap.add_argument("--eager", action="store_true",
                    help="launch the step without CUDA graphs (profiler launch lists)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.launch_list:
        run_launch_list(args)
    elif args.single:
        run_single(args)
    elif args.quant_single:
        run_quant_single(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
