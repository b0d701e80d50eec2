"""Throughput of the chunked gated-delta forward on one GB300 (JSON line out).

One step = the whole hot path over one batch: the chunkwise forward of the
Gated DeltaNet workload B=4, T=4096, H=16, d_k=d_v=128 (bf16 inputs, fp32
state, random initial state, final state returned), then one decode step per
(sequence, head) continuing from that final state. Unit: token-heads per
second (prefill B*T*H plus decode B*H per step). Other workloads are selected
with --workload (1..5; the decode phase applies where the workload has one).

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream with the L2 flushed (a 256 MiB write) before every
step, outside the events. Per-kernel events give the roofline of the chunk
kernel. Under torchrun each rank runs its own copy of the workload (weak
scaling; no collective on the data path) and the time is the max over ranks.

--impl reference times the float64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_rule_10_gb300 import workloads as wl  # noqa: E402

METRIC = "gated-delta chunk fwd tokens·heads/s at 1 GB300; % of bf16 tensor/HBM roofline"
UNIT = "token-heads/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5])
    p.add_argument("--decode-steps", type=int, default=1)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-value-beta", action="store_true",
                   help="skip the per-value-channel write strength measurement")
    p.add_argument("--no-split", action="store_true",
                   help="skip the sequence-split measurement")
    p.add_argument("--no-backward", action="store_true",
                   help="skip the backward measurement")
    p.add_argument("--no-pipelined", action="store_true",
                   help="skip the long-sequence (pipelined call) measurement")
    p.add_argument("--pipeline", type=int, default=None,
                   help="time segments of the pipelined forward (default: the library's "
                        "recommendation for the workload; 1: the plain call)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, device=None):
    """The largest of a per-rank value over all ranks of the process group (the
    slowest rank's time); x itself without a group or with one rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank_step, steps, world, total_ms):
    """Units per second of the whole job: each of `world` ranks ran `steps` steps
    of `units_per_rank_step` units, the slowest in `total_ms` milliseconds."""
    return units_per_rank_step * steps * world / (total_ms / 1e3)


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


# DRAM bytes (read + write) of one gdr_chunk_fwd call as ncu counted them
# (dram__bytes_read.sum + dram__bytes_write.sum summed over chunk_prep_kernel
# and chunk_scan_kernel), per workload, with the hash of the kernel sources they
# were taken on: a changed kernel reports null traffic until it is profiled
# again. Source: profiles/chunk_fwd_two_kernel_gdn_b4_t4096_h16_d128.md.
TRAFFIC = {2: {"bytes": 835.4e6, "sources": "23b49c3cb85400d5"}}
KERNEL_SOURCES = ("chunk_prep.cu", "chunk_scan.cu", "packet.h", "tc.cuh", "tri_inverse.cuh",
                  "common.cuh")


def kernel_sources_hash():
    import hashlib
    h = hashlib.sha1()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gated_delta_rule_10_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload):
    t = TRAFFIC.get(workload)
    if t is None or t["sources"] != kernel_sources_hash():
        return None
    return t["bytes"]


def algorithmic_flops_per_th(dk, dv, C=64):
    """Minimal FLOPs per token-head of the chunk algorithm (triangles counted once):
    6 dk dv (Y S, Q_gamma S, K_tail^T W) + (C-1)(2 dk + dv) (T, Y, U strictly lower)
    + (C+1)(dk + dv) (A_qk and A_qk W with the diagonal) + C^2/3 (substitution)."""
    return 6 * dk * dv + (C - 1) * (2 * dk + dv) + (C + 1) * (dk + dv) + C * C / 3.0


def tensor_bytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts if t is not None)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed loop runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def make_step_inputs(cfg_id, rank, dev):
    c = wl.CONFIGS[cfg_id]
    x = wl.config_inputs(cfg_id, seed=c["seed"] + 1000 * rank)
    N, H = c["B"], c["H"]
    if "decode" in c:
        N = c["decode"]["N"]
    y = wl.make_inputs(c["variant"], N, 1, H, c["dk"], c["dv"], c["dtype"],
                       seed=c["seed"] + 1000 * rank + 1, q_prescaled=c["q_prescaled"])
    return c, x, y


def squeeze_t(t):
    return None if t is None else t[:, 0].contiguous()


def run_ours(args):
    import gated_delta_rule_10_gb300 as gdr

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    c, x, y = make_step_inputs(args.workload, rank, dev)
    xd = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
    yd = {k: (squeeze_t(v).to(dev) if torch.is_tensor(v) else v) for k, v in y.items()}
    B, T, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
    N = y["q"].shape[0]
    has_decode = args.decode_steps > 0
    o = torch.empty(B, T, H, dv, dtype=c["dtype"], device=dev)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    # decode state: the prefill's final state when the batch matches, else its own
    if N == B:
        state = hT
    else:
        gen = torch.Generator().manual_seed(99 + rank)
        state = (torch.randn(N, H, dk, dv, generator=gen) * c.get("decode", {}).get("h_std", 0.02)
                 ).to(dev)
    o_dec = torch.empty(N, H, dv, dtype=c["dtype"], device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    shape = gdr.make_shape(B, T, H, dk, dv, c["dtype"], x["flags"], x["scale"])
    # long sequences with few (batch, head) pairs: the pipelined call overlaps the
    # preparation of one time segment with the state pass of the previous one
    pipe = args.pipeline if args.pipeline is not None else gdr.pipeline_segments(shape)
    ws_bytes = (gdr.chunk_fwd_pipelined_workspace_bytes(shape, pipe) if pipe > 1
                else gdr.chunk_fwd_workspace_bytes(shape))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None

    def step():
        gdr.chunk_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["lam"], xd["b"],
                      xd["w"], xd["h0"], scale=x["scale"], flags=x["flags"], o=o, hT=hT,
                      workspace=ws, pipeline=pipe)
        for _ in range(args.decode_steps if has_decode else 0):
            gdr.recurrent_step(yd["q"], yd["k"], yd["v"], yd["g"], state, yd["beta"], yd["lam"],
                               yd["b"], yd["w"], scale=y["scale"], flags=y["flags"], o=o_dec)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.1)
    for i in range(K):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        gdr.chunk_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["lam"], xd["b"],
                      xd["w"], xd["h0"], scale=x["scale"], flags=x["flags"], o=o, hT=hT,
                      workspace=ws, pipeline=pipe)
        ev[i][1].record(stream)
        for _ in range(args.decode_steps if has_decode else 0):
            gdr.recurrent_step(yd["q"], yd["k"], yd["v"], yd["g"], state, yd["beta"], yd["lam"],
                               yd["b"], yd["w"], scale=y["scale"], flags=y["flags"], o=o_dec)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    chunk_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    step_ms = [a + b for a, b in zip(chunk_ms, dec_ms)]
    total_ms = max_over_ranks(sum(step_ms), device=dev)

    th_prefill = B * T * H
    th_decode = N * H * (args.decode_steps if has_decode else 0)
    th_step = th_prefill + th_decode
    value = whole_job_value(th_step, K, world, total_ms)

    # roofline of the dominant kernel (the chunked forward), algorithmic bytes
    pk, pk_kind = peaks()
    chunk_bytes = tensor_bytes(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["lam"],
                               xd["b"], xd["w"], xd["h0"], o, hT)
    mean_chunk_s = statistics.mean(chunk_ms) / 1e3
    gbs = chunk_bytes / mean_chunk_s / 1e9
    flops = algorithmic_flops_per_th(dk, dv) * th_prefill
    tflops = flops / mean_chunk_s / 1e12
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    bound = "hbm" if flops / chunk_bytes < ridge else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / pk["hbm_gbs"], 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(tflops, 2), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(tflops / pk["bf16_tflops"], 4)}
    roof.update({"traffic": measured_traffic(args.workload),
                 "kernel": ("gdr_chunk_fwd: chunk_prep_kernel + chunk_scan_kernel (one call)"
                            if pipe <= 1 else
                            "gdr_chunk_fwd_pipelined: %d x (chunk_prep_kernel + chunk_scan_kernel)"
                            ", one call" % pipe),
                 "pipeline_segments": pipe,
                 "peak_source": pk_kind,
                 "algorithmic_bytes_per_launch": chunk_bytes,
                 "algorithmic_flops_per_launch": flops,
                 "tensor_tflops_achieved": round(tflops, 2),
                 "tensor_frac_of_bf16_peak": round(tflops / pk["bf16_tflops"], 4),
                 "launch_ms_mean": round(statistics.mean(chunk_ms), 4)})
    dec_bytes = tensor_bytes(yd["q"], yd["k"], yd["v"], yd["g"], yd["beta"], yd["lam"],
                             yd["b"], yd["w"], o_dec) + 2 * tensor_bytes(state)
    decode_info = None
    if has_decode and statistics.mean(dec_ms) > 0:
        dgbs = dec_bytes * args.decode_steps / (statistics.mean(dec_ms) / 1e3) / 1e9
        decode_info = {"kernel": "recurrent_step_kernel", "N": N, "H": H,
                       "ms_mean": round(statistics.mean(dec_ms), 4),
                       "achieved_gbs": round(dgbs, 1), "frac_hbm": round(dgbs / pk["hbm_gbs"], 4)}

    epilogue_info = measure_epilogue(gdr, o, c, dev, stream, flush, K, pk)
    value_beta_info = None if args.no_value_beta else measure_value_beta(gdr, dev, stream, flush,
                                                                         K, pk, clk)
    split_info = None if args.no_split else measure_split(gdr, dev, stream, flush, K, pk)
    pipe_info = None if args.no_pipelined else measure_pipelined(gdr, dev, stream, flush,
                                                                 min(K, 10), pk)
    backward_info = None if args.no_backward else measure_backward(gdr, xd, c, dev, stream, flush,
                                                                   min(K, 10), pk, clk)

    e2e = None if args.no_e2e else measure_e2e(gdr, x, y, c, dev, args, B, T, H, dk, dv, N)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if c["dtype"] == torch.bfloat16
        else "f32", "data": "synthetic",
        "config": {"workload": c["name"] + (" + %d decode step(s) at N=%d" %
                                            (args.decode_steps, N) if has_decode else ""),
                   "variant": c["variant"], "B": B, "T": T, "H": H, "dk": dk, "dv": dv,
                   "chunk": 64, "token_heads_per_step": th_step,
                   "l2": "flushed before every timed step (256 MiB write, outside the events)",
                   "parallelism": "replica per GPU" if world > 1 else "single GPU"},
        "roofline": roof,
        "decode": decode_info,
        "epilogue": epilogue_info,
        "value_beta": value_beta_info,
        "sequence_split": split_info,
        "pipelined": pipe_info,
        "backward": backward_info,
        # this library's kernels per timed step: the two-kernel chunked forward
        # (bf16 with the full workspace) or one fused kernel (fp32), then the
        # decode steps
        "gpu_launches": K * ((2 * max(pipe, 1) if ws is not None else 1) +
                             (args.decode_steps if has_decode else 0)),
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(x, y if N == B else None, th_step)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_epilogue(gdr, o, c, dev, stream, flush, K, pk, eps=1e-6):
    """The output epilogue (RMSNorm, gain, SiLU output gate) on the step's
    read-out o, timed alone: K launches, L2 flushed before each, CUDA events on
    the launching stream. Not part of the step or its metric."""
    from gated_delta_rule_10_gb300 import workloads as wl
    rows = o.numel() // c["dv"]
    e = wl.epilogue_inputs(rows, c["dv"], c["dtype"], seed=11, device=dev)
    y = torch.empty_like(e["z"])
    o2 = o.reshape(rows, c["dv"])
    for _ in range(3):
        gdr.rmsnorm_gate(o2, e["z"], e["weight"], eps, out=y)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        gdr.rmsnorm_gate(o2, e["z"], e["weight"], eps, out=y)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    nbytes = tensor_bytes(o2, e["z"], y, e["weight"])
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"kernel": "rmsnorm_gate_kernel", "rows": rows, "dv": c["dv"], "launches": K,
            "ms_mean": round(ms, 4), "algorithmic_bytes_per_launch": nbytes,
            "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
            "l2": "flushed before every launch"}


def fp32_alu_peak_tflops(sm_mhz):
    """FP32 (non-tensor) FMA peak of one GB300: 152 SMs x 128 FP32 lanes x 2 flops
    per FMA x the SM clock seen under load."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


def measure_value_beta(gdr, dev, stream, flush, K, pk, clk):
    """The write strength per value channel (flag BETA_CHANNEL) on the 4 x 4096 x 16
    x 128 bf16 workload, both paths timed alone like the step: K calls, L2 flushed
    before each, CUDA events on the launching stream. Not part of the step or its
    metric. The chunked two-kernel path (full workspace) is reported against HBM
    with the algorithmic bytes; the token-order scan (empty workspace) against the
    FP32 pipe with 7 d_k d_v flops per token-head (decay, two column sums, the
    rank-1 write)."""
    from gated_delta_rule_10_gb300 import workloads as wl
    c = wl.CONFIGS["vbeta"]
    x = wl.config_inputs("vbeta", device=dev)
    B, T, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
    o = torch.empty(B, T, H, dv, dtype=c["dtype"], device=dev)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    shape = gdr.make_shape(B, T, H, dk, dv, c["dtype"], x["flags"], x["scale"])
    th = B * T * H
    flops = 7.0 * dk * dv * th
    nbytes = tensor_bytes(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], o, hT)
    sm_mhz = (clk or {}).get("sm_mhz") or 2070.0
    alu_peak = fp32_alu_peak_tflops(sm_mhz)
    out = {"workload": c["name"], "launches": K, "l2": "flushed before every call",
           "algorithmic_flops_per_call": flops, "algorithmic_bytes_per_call": nbytes}
    paths = (("chunked", torch.empty(gdr.chunk_fwd_workspace_bytes(shape), dtype=torch.uint8,
                                     device=dev)),
             ("token_scan", torch.empty(0, dtype=torch.uint8, device=dev)))
    for name, ws in paths:
        def call():
            gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"],
                          scale=x["scale"], flags=x["flags"], o=o, hT=hT, workspace=ws)

        for _ in range(3):
            call()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        torch.cuda.synchronize()
        for i in range(K):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
        gbs = nbytes / (ms / 1e3) / 1e9
        tf = flops / (ms / 1e3) / 1e12
        r = {"ms_mean": round(ms, 4), "token_heads_per_s": round(th / (ms / 1e3), 1),
             "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4)}
        if name == "chunked":
            r["kernels"] = "chunk_prep_kernel + chunk_scan_kernel (substitution variant)"
            r["roofline"] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                             "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4)}
        else:
            r["kernels"] = "value_beta_scan_kernel"
            r["roofline"] = {"bound": "alu", "achieved": round(tf, 2), "peak": round(alu_peak, 2),
                             "unit": "TFLOP/s", "frac": round(tf / alu_peak, 4),
                             "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x SM clock"}
        out[name] = r
    return out


def measure_split(gdr, dev, stream, flush, K, pk, H=4):
    """The sequence split where it engages: the GDN-2 recipe of workload 5 (65536
    tokens, d = 128) with B * H = 4, through gdr_chunk_fwd's default (split into
    runs) and with one run (the plain two-kernel path), each timed alone: K calls,
    L2 flushed before each, CUDA events on the launching stream. Not part of the
    step or its metric."""
    from gated_delta_rule_10_gb300 import workloads as wl
    c = dict(wl.CONFIGS[5], H=H)
    x = wl.config_inputs(5, device=dev, H=H)
    B, T, dk, dv = c["B"], c["T"], c["dk"], c["dv"]
    o = torch.empty(B, T, H, dv, dtype=c["dtype"], device=dev)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    shape = gdr.make_shape(B, T, H, dk, dv, c["dtype"], x["flags"], x["scale"])
    ws = torch.empty(gdr.chunk_fwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    plain = gdr.chunk_fwd_workspace_bytes(shape, segments=1)
    out = {"workload": "gdn2_bf16_b1_t65536_h%d_d128" % H}
    for name, segments in (("split", None), ("one_run", 1)):
        def call():
            gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"], x["w"],
                          x["h0"], scale=x["scale"], flags=x["flags"], o=o, hT=hT, workspace=ws,
                          segments=segments)
        for _ in range(3):
            call()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        torch.cuda.synchronize()
        for i in range(K):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
        nbytes = tensor_bytes(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"], x["w"],
                              x["h0"], o, hT)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"ms_mean": round(ms, 4), "token_heads_per_s": round(B * T * H / (ms / 1e3), 1),
                     "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4)}
    out["runs_per_sequence"] = next(P for P in (64, 32, 16, 8, 4, 2, 1)
                                    if gdr.chunk_fwd_workspace_bytes(shape, segments=P) == ws.numel()
                                    ) if ws.numel() > plain else 1
    out["launches_per_call"] = {"split": 4, "one_run": 2}
    out["l2"] = "flushed before every call"
    return out


def measure_pipelined(gdr, dev, stream, flush, K, pk):
    """The Gated DeltaNet-2 prefill (1 x 65536 x 32 x 128 bf16: B * H = 32, the
    state pass on 64 SMs) through the plain call and through the pipelined call
    with the library's recommended time segments, K calls each, L2 flushed
    before every call, CUDA events on the launching stream."""
    x = wl.config_inputs(5)
    x = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
    B, T, H, dk = x["q"].shape
    dv = x["v"].shape[-1]
    shape = gdr.make_shape(B, T, H, dk, dv, x["q"].dtype, x["flags"], x["scale"])
    o = torch.empty(B, T, H, dv, dtype=x["q"].dtype, device=dev)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    seg = gdr.pipeline_segments(shape)
    nbytes = tensor_bytes(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"], x["w"],
                          x["h0"], o, hT)
    out = {"workload": "gdn2_bf16_b1_t65536_h32_d128", "segments": seg, "launches": K,
           "algorithmic_bytes_per_call": nbytes, "l2": "flushed before every call"}
    for name, pipe in (("plain", 1), ("pipelined", seg)):
        ws = torch.empty(gdr.chunk_fwd_pipelined_workspace_bytes(shape, pipe) if pipe > 1
                         else gdr.chunk_fwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)

        def call():
            gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"], x["w"],
                          x["h0"], scale=x["scale"], flags=x["flags"], o=o, hT=hT, workspace=ws,
                          pipeline=pipe)
        for _ in range(2):
            call()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        torch.cuda.synchronize()
        for i in range(K):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"ms_mean": round(ms, 4), "token_heads_per_s": round(B * T * H / (ms / 1e3), 1),
                     "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4)}
        del ws
    return out


def bwd_flops_per_th(dk, dv, C=64):
    """Multiply-adds x 2 per token-head of the chunk backward as built: the chunk's
    forward quantities (T, A, Y, U, A_qk), the forward and reverse state passes
    (W, S', dW, dS: 6 dk dv), and the per-chunk gradient products (dA_qk, dQ_gamma,
    dK_bar, dK_tail, dY, dA, dZ, dE_bar, dT)."""
    d = max(dk, dv)
    return 2.0 * (8 * dk * dv + 12 * C * d + C * C)


def measure_backward(gdr, xd, c, dev, stream, flush, K, pk, clk):
    """gdr_chunk_bwd on the step's workload (gradients of <dO, o> + <dhT, hT>), timed
    alone: K calls, L2 flushed before each, CUDA events on the launching stream.
    Not part of the step or its metric; fp32 arithmetic on the FP32 pipe."""
    B, T, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
    gen = torch.Generator().manual_seed(7)
    dO = torch.randn(B, T, H, dv, generator=gen).to(c["dtype"]).to(dev)
    dhT = (torch.randn(B, H, dk, dv, generator=gen) * 0.1).to(dev)
    shape = gdr.make_shape(B, T, H, dk, dv, c["dtype"], xd["flags"], xd["scale"])
    ws = torch.empty(gdr.chunk_bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)

    def call():
        return gdr.chunk_bwd(xd["q"], xd["k"], xd["v"], xd["g"], dO, xd["beta"], xd["lam"],
                             xd["b"], xd["w"], xd["h0"], dhT, scale=xd["scale"],
                             flags=xd["flags"], workspace=ws)

    for _ in range(2):
        grads = call()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    th = B * T * H
    flops = bwd_flops_per_th(dk, dv) * th
    tf = flops / (ms / 1e3) / 1e12
    peak = fp32_alu_peak_tflops((clk or {}).get("sm_mhz") or 2070.0)
    nbytes = tensor_bytes(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["lam"], xd["b"],
                          xd["w"], xd["h0"], dO, dhT, *[t for t in grads.values() if t is not None])
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"kernels": "bwd_chunk_prep, bwd_state_pass, bwd_dstate_pass, bwd_chunk_grad",
            "workload": c["name"], "launches": K, "ms_mean": round(ms, 4),
            "token_heads_per_s": round(th / (ms / 1e3), 1),
            "roofline": {"bound": "alu", "achieved": round(tf, 2), "peak": round(peak, 2),
                         "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                         "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x SM clock"},
            "algorithmic_flops_per_call": flops, "algorithmic_bytes_per_call": nbytes,
            "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
            "workspace_bytes": ws.numel(), "l2": "flushed before every call"}


def measure_e2e(gdr, x, y, c, dev, args, B, T, H, dk, dv, N, steps=8, n_up=1):
    """Same metric through the public API with pinned host buffers: every step
    copies its inputs host->device, runs the path, and copies o, the decode
    output and the final state back. The steps are pipelined the way a server
    would run them: inputs of step i+1 go up on a copy stream while step i
    computes, and step i's results come down on another while step i+1
    computes (device buffers double-buffered); every copy of every step is
    inside the timed region. The upload bounds the step (~180 GB/s host to
    device here); two to four upload streams measured no faster than one."""
    names = ("q", "k", "v", "g", "beta", "lam", "b", "w", "h0")
    hx = {n: x[n].pin_memory() for n in names if x[n] is not None}
    hy = {n: squeeze_t(y[n]).pin_memory() for n in ("q", "k", "v", "g", "beta", "lam", "b", "w")
          if y[n] is not None}
    nb = 2
    dx = [{n: torch.empty_like(t, device=dev) for n, t in hx.items()} for _ in range(nb)]
    dy = [{n: torch.empty_like(t, device=dev) for n, t in hy.items()} for _ in range(nb)]
    o = [torch.empty(B, T, H, dv, dtype=c["dtype"], device=dev) for _ in range(nb)]
    hT = [torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev) for _ in range(nb)]
    state = [hT[i] if N == B else torch.zeros(N, H, dk, dv, device=dev) for i in range(nb)]
    o_dec = [torch.empty(N, H, dv, dtype=c["dtype"], device=dev) for _ in range(nb)]
    ho = torch.empty_like(o[0], device="cpu").pin_memory()
    hhT = torch.empty_like(state[0], device="cpu").pin_memory()
    ho_dec = torch.empty_like(o_dec[0], device="cpu").pin_memory()
    shape = gdr.make_shape(B, T, H, dk, dv, c["dtype"], x["flags"], x["scale"])
    nws = gdr.chunk_fwd_workspace_bytes(shape)
    ws = [torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None for _ in range(nb)]
    comp = torch.cuda.current_stream(dev)
    ups = [torch.cuda.Stream(dev) for _ in range(n_up)]
    down = torch.cuda.Stream(dev)
    g = lambda d, n: d.get(n)
    # the input tensors dealt over the upload streams, largest first
    order = sorted(list(hx.items()) + [("y." + n, t) for n, t in hy.items()],
                   key=lambda kv: -kv[1].numel() * kv[1].element_size())
    lanes = [[] for _ in range(n_up)]
    load = [0] * n_up
    for n, t in order:
        j = load.index(min(load))
        lanes[j].append(n)
        load[j] += t.numel() * t.element_size()

    def run(steps_n):
        up_done = [[torch.cuda.Event() for _ in range(n_up)] for _ in range(steps_n)]
        comp_done = [torch.cuda.Event() for _ in range(steps_n)]
        down_done = [torch.cuda.Event() for _ in range(steps_n)]
        for i in range(steps_n):
            s = i % nb
            # inputs of step i: after step i - nb has finished reading buffer s
            for j, up in enumerate(ups):
                with torch.cuda.stream(up):
                    if i >= nb:
                        up.wait_event(comp_done[i - nb])
                    for n in lanes[j]:
                        if n.startswith("y."):
                            dy[s][n[2:]].copy_(hy[n[2:]], non_blocking=True)
                        else:
                            dx[s][n].copy_(hx[n], non_blocking=True)
                    up_done[i][j].record(up)
                comp.wait_event(up_done[i][j])
            if i >= nb:
                comp.wait_event(down_done[i - nb])   # results of step i - nb are down
            d, e = dx[s], dy[s]
            gdr.chunk_fwd(g(d, "q"), g(d, "k"), g(d, "v"), g(d, "g"), g(d, "beta"), g(d, "lam"),
                          g(d, "b"), g(d, "w"), g(d, "h0"), scale=x["scale"], flags=x["flags"],
                          o=o[s], hT=hT[s], workspace=ws[s])
            for _ in range(args.decode_steps):
                gdr.recurrent_step(g(e, "q"), g(e, "k"), g(e, "v"), g(e, "g"), state[s],
                                   g(e, "beta"), g(e, "lam"), g(e, "b"), g(e, "w"),
                                   scale=y["scale"], flags=y["flags"], o=o_dec[s])
            comp_done[i].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(comp_done[i])
                ho.copy_(o[s], non_blocking=True)
                ho_dec.copy_(o_dec[s], non_blocking=True)
                hhT.copy_(state[s], non_blocking=True)
                down_done[i].record(down)
        comp.wait_event(down_done[steps_n - 1])
        for up in ups:
            up.wait_stream(comp)
        down.wait_stream(comp)

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    for up in ups:
        up.wait_event(e0)
    run(steps)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    th = B * T * H + N * H * args.decode_steps
    h2d = sum(t.numel() * t.element_size() for t in hx.values()) + \
        sum(t.numel() * t.element_size() for t in hy.values()) * args.decode_steps
    d2h = tensor_bytes(ho, ho_dec, hhT)
    return {"value": round(th / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "steps": steps,
            "pipelined": "inputs of step i+1 up (%d copy streams) and results of step i-1 down "
                         "while step i computes" % n_up}


def oracle_step(x, y, seqs, nthreads):
    """The oracle on `seqs` (batch, head) sequences of the step's workload: the
    prefill tokens followed by the decode token (same math as the GPU step)."""
    import numpy as np
    from oracle import native

    f64 = lambda t: None if t is None else t.double().numpy()
    out_th = 0
    t_total = 0.0
    for (b, h) in seqs:
        def pick(n):
            t = x[n]
            if t is None:
                return None
            t = t[b:b + 1, :, h:h + 1]
            if y is not None and y[n] is not None:
                t = torch.cat([t, y[n][b:b + 1, :, h:h + 1]], dim=1)
            return f64(t.contiguous())
        args = [pick(n) for n in ("q", "k", "v", "g", "beta", "lam", "b", "w")]
        h0 = None if x["h0"] is None else f64(x["h0"][b:b + 1, h:h + 1].contiguous())
        t0 = time.perf_counter()
        native.recurrence(*args[:4], beta=args[4], lam=args[5], b=args[6], w=args[7], h0=h0,
                          scale=x["scale"], flags=x["flags"], nthreads=1)
        t_total += time.perf_counter() - t0
        out_th += args[0].shape[1]
    return out_th, t_total


def cpu_baseline(x, y, th_step, budget_s=20.0):
    """The oracle as it stands, timed on the host cores: every (batch, head)
    sequence of the workload (each the prefill plus the decode token), spread
    over all cores with OpenMP, repeated until ~budget_s or one pass."""
    import numpy as np
    from oracle import native

    f64 = lambda t: None if t is None else t.double().numpy()
    cat = lambda n: (torch.cat([x[n], y[n]], dim=1) if (y is not None and x[n] is not None)
                     else x[n])
    arrs = {n: f64(cat(n)) for n in ("q", "k", "v", "g", "beta", "lam", "b", "w")}
    h0 = f64(x["h0"])
    cores = native.max_threads()
    th = arrs["q"].shape[0] * arrs["q"].shape[1] * arrs["q"].shape[2]
    reps, t_total = 0, 0.0
    while reps == 0 or (t_total < budget_s and reps < 3):
        t0 = time.perf_counter()
        native.recurrence(arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"], arrs["lam"],
                          arrs["b"], arrs["w"], h0, x["scale"], x["flags"], nthreads=cores)
        t_total += time.perf_counter() - t0
        reps += 1
    return {"value": round(th * reps / t_total, 1), "unit": UNIT, "cores": cores,
            "kind": "oracle", "sample": "whole workload (%d token-heads incl. decode tokens), "
            "%d pass(es), C fp64 token recurrence, OpenMP over (batch, head)" % (th, reps),
            "seconds": round(t_total, 3)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import native
    c, x, y = make_step_inputs(args.workload, 0, "cpu")
    N = y["q"].shape[0]
    yy = y if N == c["B"] else None
    B, H = c["B"], c["H"]
    # bounded sample per step: 2 sequences (each ~0.5 GFLOP at T=4096)
    seqs_all = [(b, h) for b in range(B) for h in range(H)]
    per_step = 2
    for i in range(args.warmup):
        oracle_step(x, yy, seqs_all[:1], 1)
    th_total, t_total = 0, 0.0
    steps = max(1, min(args.steps, 8))
    for i in range(steps):
        seqs = [seqs_all[(i * per_step + j) % len(seqs_all)] for j in range(per_step)]
        th, t = oracle_step(x, yy, seqs, 1)
        th_total += th
        t_total += t
    value = th_total / t_total
    res = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
           "steps": steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_total / steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": {"workload": c["name"], "variant": c["variant"], "B": c["B"], "T": c["T"],
                      "H": c["H"], "dk": c["dk"], "dv": c["dv"]},
           "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": "%d (batch, head) sequences per step (prefill plus "
                                      "decode token), single thread" % per_step},
           "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
