"""Throughput of the gated-delta hot path on one GB300 (one JSON line out).

One step = the whole hot path over one batch of the Gated DeltaNet-2 workload:
the chunkwise forward of B=1, T=65536, H=32, d_k=d_v=128 (bf16 inputs, fp32
state, final state returned), then its decode phase, 256 single-token steps
at batch N=256 (H=32) from random fp32 states, one gdr_recurrent_step call per
token. Unit: token-heads per second (prefill B*T*H plus decode N*H per decode
step). --workload 1..4 selects another workload as the step (then one decode
step per (batch, head) from the prefill's final state); every run also times
the other workloads' chunked forwards alone (`configs`).

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream with the L2 flushed (a 256 MiB write) and the decode
states reset before every step, outside the events. The `roofline` object is
the chunked forward's (the metric's subject): algorithmic bytes over its
event-timed duration against the measured HBM copy bandwidth; the decode
phase, the standalone gate cumsum and every other workload carry their own.
Under torchrun each rank runs its own copy of the workload (weak scaling; no
collective on the data path) and the time is the max over ranks.

--impl reference times the float64 CPU oracle on the host cores instead (a
bounded sample of the same workload's recipe per step).
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
    p.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5])
    p.add_argument("--decode-steps", type=int, default=None,
                   help="decode steps per step (default: the workload's decode phase, else 1)")
    p.add_argument("--no-configs", action="store_true",
                   help="skip timing the other workloads")
    p.add_argument("--seq-len", type=int, default=None,
                   help="override the workload's T (a shortened case for profiler runs; "
                        "the line then does not describe the named workload)")
    p.add_argument("--minimal", action="store_true",
                   help="the step alone: no other workloads, epilogue, gate cumsum, e2e, CPU "
                        "baseline or side measurements (for profiler runs)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-value-beta", action="store_true",
                   help="skip the per-value-channel write strength measurement")
    p.add_argument("--no-split", action="store_true",
                   help="skip the sequence-split measurement")
    p.add_argument("--no-graph", action="store_true",
                   help="launch the decode steps one by one instead of replaying a CUDA graph")
    p.add_argument("--no-backward", action="store_true",
                   help="skip the backward measurement")
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
# and chunk_scan_kernel, from one capture of the plain two-kernel call), per
# workload, with the hash of the kernel sources they were taken on: a changed
# kernel reports null traffic until it is profiled again. The Gated DeltaNet-2
# prefill (1 x 65536 x 32 x 128) is too large to capture whole: its figure is
# the capture of the same call at T = 8192 (1185.2 MB for 128 chunks per
# sequence, the chunk count of each of its 8 pipelined segments) times 8, since
# every term of the traffic (inputs, packets, outputs) grows with the chunks.
TRAFFIC = {2: {"bytes": 849.6e6, "sources": "720d4711722d2517"},
           3: {"bytes": 1771.9e6, "sources": "720d4711722d2517"},
           4: {"bytes": 4091.1e6, "sources": "720d4711722d2517"},
           5: {"bytes": 8 * 1185.2e6, "sources": "720d4711722d2517",
               "scaled": "ncu DRAM bytes of the call at T = 8192 (1185.2 MB) x 8, the ratio of the chunks"}}
KERNEL_SOURCES = ("chunk_prep.cu", "chunk_scan.cu", "chunk_scan_t.cu", "packet.h", "tc.cuh",
                  "tri_inverse.cuh", "common.cuh")


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


def traffic_fields(workload):
    """The roofline object's traffic keys: the bytes (or None) and, for a figure
    scaled from a shortened capture, how it was scaled."""
    b = measured_traffic(workload)
    out = {"traffic": b}
    if b is not None and "scaled" in TRAFFIC[workload]:
        out["traffic_scaled_from"] = TRAFFIC[workload]["scaled"]
    return out


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


def decode_of(cfg_id, N_default):
    """(steps, N) of the workload's decode phase: its own, else one decode step
    per (batch, head) continuing from the prefill's final state."""
    c = wl.CONFIGS[cfg_id]
    if "decode" in c:
        return c["decode"]["steps"], c["decode"]["N"]
    return 1, N_default


def prefill_bytes(x, o, hT):
    """Algorithmic bytes of one chunked forward: every input read once, o and the
    final state written once."""
    return tensor_bytes(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"], x["w"],
                        x["h0"], o, hT)


def roofline_obj(nbytes, flops, ms, pk, pk_kind):
    """HBM or tensor roofline of one launch from its algorithmic bytes / flops and
    its mean event-timed duration."""
    s = ms / 1e3
    gbs = nbytes / s / 1e9
    tflops = flops / s / 1e12
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if flops / max(nbytes, 1) < ridge:
        r = {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
             "frac": round(gbs / pk["hbm_gbs"], 4)}
    else:
        r = {"bound": "tensor", "achieved": round(tflops, 2), "peak": pk["bf16_tflops"],
             "unit": "TFLOP/s", "frac": round(tflops / pk["bf16_tflops"], 4)}
    r.update({"peak_source": pk_kind, "algorithmic_bytes_per_launch": nbytes,
              "algorithmic_flops_per_launch": flops,
              "tensor_tflops_achieved": round(tflops, 2),
              "tensor_frac_of_bf16_peak": round(tflops / pk["bf16_tflops"], 4),
              "launch_ms_mean": round(ms, 4)})
    return r


def time_calls(call, K, stream, flush, warm=3, before=None):
    """Mean milliseconds of `call` over K calls, each bracketed by CUDA events on
    `stream`, the L2 flushed (and `before` run) ahead of each outside the events."""
    for _ in range(warm):
        if before is not None:
            before()
        call()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(float(i))
        if before is not None:
            before()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))


def fwd_launches(gdr, shape, pipe, ws):
    """This library's kernel launches in one chunked forward call."""
    if ws is None:
        return 1                       # fp32: one fused kernel
    if pipe > 1:
        return 2 * pipe                # preparation + state pass per time segment
    return 2                           # the five workloads never split (B * H >= 32)


def run_ours(args):
    import gated_delta_rule_10_gb300 as gdr

    if args.minimal:
        args.no_configs = args.no_e2e = args.no_cpu_baseline = True
        args.no_value_beta = args.no_split = args.no_backward = True

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = args.workload
    c = dict(wl.CONFIGS[cfg])
    if args.seq_len:
        c["T"] = args.seq_len
        c["name"] = c["name"] + "_T%d" % args.seq_len
    # inputs drawn on the device (seeded CUDA generator), resident in HBM
    x = wl.config_inputs(cfg, gen_device=dev, seed=c["seed"] + 1000 * rank, T=c["T"])
    B, T, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
    dec_steps, N = decode_of(cfg, B)
    if args.decode_steps is not None:
        dec_steps = args.decode_steps
    if "decode" in c:
        y = wl.decode_phase_inputs(cfg, seed=c["seed"] + 500 + 1000 * rank, gen_device=dev,
                                   steps=max(dec_steps, 1))
    else:   # one token per (batch, head) after the prefill, from its final state
        y = wl.make_inputs(c["variant"], max(dec_steps, 1), B, H, dk, dv, c["dtype"],
                           seed=c["seed"] + 1000 * rank + 1, gen_device=dev)
        y["h0"] = None
    o = torch.empty(B, T, H, dv, dtype=c["dtype"], device=dev)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    state = hT if y["h0"] is None else torch.empty_like(y["h0"])
    o_dec = torch.empty(max(dec_steps, 1), N, H, dv, dtype=c["dtype"], device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    shape = gdr.make_shape(B, T, H, dk, dv, c["dtype"], x["flags"], x["scale"])
    # long sequences with few (batch, head) pairs: the pipelined call overlaps the
    # preparation of one time segment with the state pass of the previous one
    pipe = args.pipeline if args.pipeline is not None else gdr.pipeline_segments(shape)
    ws_bytes = (gdr.chunk_fwd_pipelined_workspace_bytes(shape, pipe) if pipe > 1
                else gdr.chunk_fwd_workspace_bytes(shape))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    yg = lambda n, s: None if y[n] is None else y[n][s]

    def prefill():
        gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"], x["w"],
                      x["h0"], scale=x["scale"], flags=x["flags"], o=o, hT=hT, workspace=ws,
                      pipeline=pipe)

    def decode():
        for s in range(dec_steps):
            gdr.recurrent_step(yg("q", s), yg("k", s), yg("v", s), yg("g", s), state,
                               yg("beta", s), yg("lam", s), yg("b", s), yg("w", s),
                               scale=y["scale"], flags=y["flags"], o=o_dec[s])

    def reset():
        # the decode phase starts from its own random states (outside the events)
        if y["h0"] is not None:
            state.copy_(y["h0"])

    for _ in range(args.warmup):
        reset()
        prefill()
        decode()
    torch.cuda.synchronize()
    # the decode phase's launches, recorded once into a CUDA graph and replayed
    # every step (the same kernels, without one host launch per token)
    graph = None
    if dec_steps > 0 and not args.no_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            decode()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            decode()
        torch.cuda.synchronize()

    def decode_phase():
        if graph is not None:
            graph.replay()
        else:
            decode()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.1)
    for i in range(K):
        flush.fill_(float(i))
        reset()
        ev[i][0].record(stream)
        prefill()
        ev[i][1].record(stream)
        decode_phase()
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
    th_decode = N * H * dec_steps
    th_step = th_prefill + th_decode
    value = whole_job_value(th_step, K, world, total_ms)

    # roofline of the chunked forward (the metric's subject), algorithmic bytes
    pk, pk_kind = peaks()
    mean_chunk = statistics.mean(chunk_ms)
    roof = roofline_obj(prefill_bytes(x, o, hT), algorithmic_flops_per_th(dk, dv) * th_prefill,
                        mean_chunk, pk, pk_kind)
    roof.update(traffic_fields(None if args.seq_len else cfg))
    roof.update({"kernel": ("gdr_chunk_fwd: chunk_prep_kernel + chunk_scan_kernel (one call)"
                            if pipe <= 1 else
                            "gdr_chunk_fwd_pipelined: %d x (chunk_prep_kernel + chunk_scan_kernel)"
                            ", one call" % pipe),
                 "pipeline_segments": pipe,
                 "token_heads_per_s": round(th_prefill / (mean_chunk / 1e3), 1)})
    decode_info = None
    if dec_steps > 0:
        per = statistics.mean(dec_ms) / dec_steps
        dbytes = (tensor_bytes(*(yg(n, 0) for n in ("q", "k", "v", "g", "beta", "lam", "b",
                                                      "w")), o_dec[0]) + 2 * tensor_bytes(state))
        droof = roofline_obj(dbytes, 5.0 * dk * dv * N * H, per, pk, pk_kind)
        decode_info = {"kernel": "recurrent_step_kernel", "steps": dec_steps, "N": N, "H": H,
                       "launch": ("one CUDA graph of the steps' launches, replayed"
                                  if graph is not None else "one launch per step"),
                       "from": "random fp32 states" if y["h0"] is not None else
                               "the prefill's final state",
                       "ms_per_phase": round(statistics.mean(dec_ms), 4),
                       "ms_per_decode_step": round(per, 5),
                       "token_heads_per_s": round(th_decode / (statistics.mean(dec_ms) / 1e3), 1),
                       "roofline": droof}
    plain_ms = None
    if pipe > 1 and not args.minimal:   # the same inputs through the plain two-kernel call
        ws1 = torch.empty(gdr.chunk_fwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
        plain_ms = time_calls(lambda: gdr.chunk_fwd(
            x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"], x["w"], x["h0"],
            scale=x["scale"], flags=x["flags"], o=o, hT=hT, workspace=ws1, pipeline=1),
            min(K, 10), stream, flush)
        del ws1
        roof["plain_call_ms"] = round(plain_ms, 4)

    cumsum_info = epilogue_info = None
    if not args.minimal:
        cumsum_info = measure_gate_cumsum(gdr, x, c, dev, stream, flush, min(K, 20), pk,
                                          pk_kind)
        epilogue_info = measure_epilogue(gdr, o, c, dev, stream, flush, min(K, 20), pk)
        if c["dtype"] == torch.bfloat16:
            epilogue_info["fused"] = measure_fused_epilogue(gdr, x, c, dev, stream, flush,
                                                            min(K, 10), pk, pk_kind, pipe)
    e2e = None if args.no_e2e else measure_e2e(gdr, x, y, c, dev, pipe, dec_steps, N)
    # the other workloads, each timed alone in its default launch configuration
    configs_info = None
    if not args.no_configs:
        configs_info = {}
        del ws
        for other in (1, 2, 3, 4, 5):
            if other != cfg:
                configs_info[str(other)] = measure_config(gdr, other, dev, stream, flush,
                                                          min(K, 20), pk, pk_kind)
    value_beta_info = None if args.no_value_beta else measure_value_beta(gdr, dev, stream, flush,
                                                                         min(K, 10), pk, clk)
    split_info = None if args.no_split else measure_split(gdr, dev, stream, flush, min(K, 10), pk)
    backward_info = None if args.no_backward else measure_backward(gdr, dev, stream, flush,
                                                                   min(K, 10), pk, clk)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if c["dtype"] == torch.bfloat16
        else "f32", "data": "synthetic",
        "config": dict(config_obj(c, dec_steps, N, world),
                       l2="flushed before every timed step (256 MiB write, outside the events)",
                       inputs="drawn on the device with a seeded CUDA generator, resident in HBM"),
        "roofline": roof,
        "decode": decode_info,
        "gate_cumsum": cumsum_info,
        "configs": configs_info,
        "epilogue": epilogue_info,
        "value_beta": value_beta_info,
        "sequence_split": split_info,
        "backward": backward_info,
        # this library's kernels per timed step: the chunked forward's launches,
        # then one per decode step
        "gpu_launches": K * (fwd_launches(gdr, shape, pipe, ws_bytes or None) + dec_steps),
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(x, y, dec_steps)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_config(gdr, cfg, dev, stream, flush, K, pk, pk_kind):
    """One workload's chunked forward timed alone in the launch configuration the
    library picks for it (pipelined where it recommends time segments): K calls,
    L2 flushed before each, CUDA events on the launching stream."""
    c = wl.CONFIGS[cfg]
    x = wl.config_inputs(cfg, gen_device=dev)
    B, T, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
    o = torch.empty(B, T, H, dv, dtype=c["dtype"], device=dev)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    shape = gdr.make_shape(B, T, H, dk, dv, c["dtype"], x["flags"], x["scale"])
    pipe = gdr.pipeline_segments(shape)
    nws = (gdr.chunk_fwd_pipelined_workspace_bytes(shape, pipe) if pipe > 1
           else gdr.chunk_fwd_workspace_bytes(shape))
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None

    def call():
        gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"], x["w"],
                      x["h0"], scale=x["scale"], flags=x["flags"], o=o, hT=hT, workspace=ws,
                      pipeline=pipe)

    ms = time_calls(call, K, stream, flush)
    th = B * T * H
    roof = roofline_obj(prefill_bytes(x, o, hT), algorithmic_flops_per_th(dk, dv) * th, ms, pk,
                        pk_kind)
    roof.update(traffic_fields(cfg))
    out = {"workload": c["name"], "dtype": "bf16" if c["dtype"] == torch.bfloat16 else "f32",
           "launches": K, "ms_mean": round(ms, 4), "token_heads_per_s": round(th / (ms / 1e3), 1),
           "pipeline_segments": pipe, "roofline": roof, "l2": "flushed before every call",
           "kernels": ("chunk_fwd_kernel (fp32)" if ws is None else
                       "chunk_prep_kernel + chunk_scan_kernel" +
                       (" x %d time segments" % pipe if pipe > 1 else ""))}
    del x, o, hT, ws
    torch.cuda.empty_cache()
    return out


def measure_gate_cumsum(gdr, x, c, dev, stream, flush, K, pk, pk_kind):
    """The standalone chunk-local log-decay cumsum (gdr_gate_cumsum) on the
    workload's gate tensor (per key channel for the channel-decay variants), timed
    alone: K launches, L2 flushed before each. Bytes: g read once, G written once."""
    g = x["g"]
    G = torch.empty_like(g)
    ms = time_calls(lambda: gdr.gate_cumsum(g, out=G), K, stream, flush)
    nbytes = tensor_bytes(g, G)
    roof = roofline_obj(nbytes, float(g.numel()), ms, pk, pk_kind)
    del G
    return {"kernel": "gate_cumsum_vec4" if g.dim() == 4 else "gate_cumsum_scalar",
            "shape": list(g.shape), "launches": K, "ms_mean": round(ms, 4),
            "roofline": roof, "l2": "flushed before every launch"}


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


def measure_fused_epilogue(gdr, x, c, dev, stream, flush, K, pk, pk_kind, pipe, eps=1e-6):
    """The step's chunked forward with the output epilogue fused into its state
    pass (gdr_chunk_fwd_gated[_pipelined]), against the same forward followed by
    the standalone epilogue kernel: K calls each, L2 flushed before every call,
    CUDA events on the launching stream. Bytes of the fused call: the forward's
    inputs, z and the gain read, y and the final state written."""
    B, T, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
    e = wl.epilogue_inputs(B * T * H, dv, c["dtype"], seed=11, device=dev)
    z, weight = e["z"].reshape(B, T, H, dv), e["weight"]
    y = torch.empty(B, T, H, dv, dtype=c["dtype"], device=dev)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    shape = gdr.make_shape(B, T, H, dk, dv, c["dtype"], x["flags"], x["scale"])
    ws = torch.empty(gdr.chunk_fwd_pipelined_workspace_bytes(shape, pipe) if pipe > 1
                     else gdr.chunk_fwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    fwd = lambda gate: gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["lam"], x["b"],
                                     x["w"], x["h0"], scale=x["scale"], flags=x["flags"], o=y,
                                     hT=hT, workspace=ws, pipeline=pipe, out_gate=gate)
    fused_ms = time_calls(lambda: fwd((z, weight, eps)), K, stream, flush)
    yy = y.reshape(-1, dv)

    def separate():
        fwd(None)
        gdr.rmsnorm_gate(yy, z.reshape(-1, dv), weight, eps, out=yy)

    sep_ms = time_calls(separate, K, stream, flush)
    nbytes = prefill_bytes(x, y, hT) + tensor_bytes(z, weight)
    th = B * T * H
    roof = roofline_obj(nbytes, algorithmic_flops_per_th(dk, dv) * th, fused_ms, pk, pk_kind)
    del ws, y, z, e
    torch.cuda.empty_cache()
    return {"workload": c["name"], "fused_ms_mean": round(fused_ms, 4),
            "forward_then_epilogue_ms_mean": round(sep_ms, 4),
            "fused_token_heads_per_s": round(th / (fused_ms / 1e3), 1),
            "kernels": "chunk_prep_kernel + chunk_scan_t_kernel with the epilogue in its output "
                       "role" + (" x %d time segments" % pipe if pipe > 1 else ""),
            "launches": K, "roofline": roof, "l2": "flushed before every call"}


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
    x = wl.config_inputs("vbeta", gen_device=dev)
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
    # the backward of the same workload (the token-order backward with chunk
    # checkpoints: a forward pass, then every chunk re-run and walked back);
    # against the FP32 pipe with about 3 x 7 + 12 d_k d_v flops per token-head
    gen = torch.Generator(device=dev).manual_seed(11)
    dO = torch.randn(B, T, H, dv, generator=gen, device=dev).to(c["dtype"])
    dhT = torch.randn(B, H, dk, dv, generator=gen, device=dev) * 0.1
    bws = torch.empty(gdr.chunk_bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)

    def bwd():
        gdr.chunk_bwd(x["q"], x["k"], x["v"], x["g"], dO, x["beta"], h0=x["h0"], dhT=dhT,
                      scale=x["scale"], flags=x["flags"], workspace=bws)

    for _ in range(2):
        bwd()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        bwd()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    bflops = 33.0 * dk * dv * th
    tf = bflops / (ms / 1e3) / 1e12
    out["backward"] = {"ms_mean": round(ms, 4), "token_heads_per_s": round(th / (ms / 1e3), 1),
                       "kernels": "value_beta_bwd_kernel", "workspace_bytes": bws.numel(),
                       "roofline": {"bound": "alu", "achieved": round(tf, 2),
                                    "peak": round(alu_peak, 2), "unit": "TFLOP/s",
                                    "frac": round(tf / alu_peak, 4),
                                    "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x SM clock"}}
    return out


def measure_split(gdr, dev, stream, flush, K, pk, H=4):
    """The sequence split where it engages: the GDN-2 recipe of workload 5 (65536
    tokens, d = 128) with B * H = 4, through gdr_chunk_fwd's default (split into
    runs) and with one run (the plain two-kernel path), each timed alone: K calls,
    L2 flushed before each, CUDA events on the launching stream. Not part of the
    step or its metric."""
    from gated_delta_rule_10_gb300 import workloads as wl
    c = dict(wl.CONFIGS[5], H=H)
    x = wl.config_inputs(5, gen_device=dev, H=H)
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


def bwd_flops_per_th(dk, dv, C=64):
    """Multiply-adds x 2 per token-head of the chunk backward as built: the chunk's
    forward quantities (T, A, Y, U, A_qk), the forward and reverse state passes
    (W, S', dW, dS: 6 dk dv), and the per-chunk gradient products (dA_qk, dQ_gamma,
    dK_bar, dK_tail, dY, dA, dZ, dE_bar, dT)."""
    d = max(dk, dv)
    return 2.0 * (8 * dk * dv + 12 * C * d + C * C)


def measure_backward(gdr, dev, stream, flush, K, pk, clk, cfg=2):
    """gdr_chunk_bwd on the Gated DeltaNet workload (4 x 4096 x 16 x 128 bf16;
    gradients of <dO, o> + <dhT, hT>), timed alone: K calls, L2 flushed before
    each, CUDA events on the launching stream. Not part of the step or its
    metric; fp32 accumulation (bf16 inputs: single tf32 products in the per-chunk
    kernels)."""
    c = wl.CONFIGS[cfg]
    xd = wl.config_inputs(cfg, gen_device=dev)
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


def measure_e2e(gdr, x, y, c, dev, pipe, dec_steps, N, steps=6):
    """Same metric through the public API with pinned host buffers: every step
    copies its inputs host->device (the prefill's tensors, the decode phase's
    per-token tensors and its starting states), runs the path, and copies o, the
    prefill's final state, every decode output and the decode's final states
    back. The steps are pipelined the way a server would run them: inputs of step
    i+1 go up on a copy stream while step i computes, and step i's results come
    down on another while step i+1 computes (device buffers double-buffered);
    every copy of every step is inside the timed region."""
    B, T, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
    names = ("q", "k", "v", "g", "beta", "lam", "b", "w", "h0")
    hx = {n: x[n].cpu().pin_memory() for n in names if x[n] is not None}
    hy = {n: y[n][:max(dec_steps, 1)].cpu().pin_memory() for n in names[:-1]
          if y[n] is not None}
    if y["h0"] is not None:
        hy["h0"] = y["h0"].cpu().pin_memory()
    nb = 2
    dx = [{n: torch.empty_like(t, device=dev) for n, t in hx.items()} for _ in range(nb)]
    dy = [{n: torch.empty_like(t, device=dev) for n, t in hy.items()} for _ in range(nb)]
    o = [torch.empty(B, T, H, dv, dtype=c["dtype"], device=dev) for _ in range(nb)]
    hT = [torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev) for _ in range(nb)]
    o_dec = [torch.empty(max(dec_steps, 1), N, H, dv, dtype=c["dtype"], device=dev)
             for _ in range(nb)]
    ho = torch.empty_like(o[0], device="cpu").pin_memory()
    hhT = torch.empty_like(hT[0], device="cpu").pin_memory()
    ho_dec = torch.empty_like(o_dec[0], device="cpu").pin_memory()
    hstate = (torch.empty_like(hy["h0"]).pin_memory() if "h0" in hy else None)
    shape = gdr.make_shape(B, T, H, dk, dv, c["dtype"], x["flags"], x["scale"])
    nws = (gdr.chunk_fwd_pipelined_workspace_bytes(shape, pipe) if pipe > 1
           else gdr.chunk_fwd_workspace_bytes(shape))
    ws = [torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None for _ in range(nb)]
    comp = torch.cuda.current_stream(dev)
    up = torch.cuda.Stream(dev)
    down = torch.cuda.Stream(dev)
    g = lambda d, n: d.get(n)
    gs = lambda d, n, s: None if d.get(n) is None else d[n][s]

    def run(steps_n):
        up_done = [torch.cuda.Event() for _ in range(steps_n)]
        comp_done = [torch.cuda.Event() for _ in range(steps_n)]
        down_done = [torch.cuda.Event() for _ in range(steps_n)]
        for i in range(steps_n):
            s = i % nb
            # inputs of step i: after step i - nb has finished reading buffer s
            with torch.cuda.stream(up):
                if i >= nb:
                    up.wait_event(comp_done[i - nb])
                for n, t in hx.items():
                    dx[s][n].copy_(t, non_blocking=True)
                for n, t in hy.items():
                    dy[s][n].copy_(t, non_blocking=True)
                up_done[i].record(up)
            comp.wait_event(up_done[i])
            if i >= nb:
                comp.wait_event(down_done[i - nb])   # results of step i - nb are down
            d, e = dx[s], dy[s]
            gdr.chunk_fwd(g(d, "q"), g(d, "k"), g(d, "v"), g(d, "g"), g(d, "beta"), g(d, "lam"),
                          g(d, "b"), g(d, "w"), g(d, "h0"), scale=x["scale"], flags=x["flags"],
                          o=o[s], hT=hT[s], workspace=ws[s], pipeline=pipe)
            state = e["h0"] if "h0" in e else hT[s]
            for t in range(dec_steps):
                gdr.recurrent_step(gs(e, "q", t), gs(e, "k", t), gs(e, "v", t), gs(e, "g", t),
                                   state, gs(e, "beta", t), gs(e, "lam", t), gs(e, "b", t),
                                   gs(e, "w", t), scale=y["scale"], flags=y["flags"],
                                   o=o_dec[s][t])
            comp_done[i].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(comp_done[i])
                ho.copy_(o[s], non_blocking=True)
                hhT.copy_(hT[s], non_blocking=True)
                ho_dec.copy_(o_dec[s], non_blocking=True)
                if hstate is not None:
                    hstate.copy_(e["h0"], non_blocking=True)
                down_done[i].record(down)
        comp.wait_event(down_done[steps_n - 1])
        up.wait_stream(comp)
        down.wait_stream(comp)

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    up.wait_event(e0)
    run(steps)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    th = B * T * H + N * H * dec_steps
    h2d = tensor_bytes(*hx.values()) + tensor_bytes(*hy.values())
    d2h = tensor_bytes(ho, hhT, ho_dec, hstate)
    out = {"value": round(th / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "steps": steps,
           "pipelined": "inputs of step i+1 up and results of step i-1 down while step i "
                        "computes (one copy stream each way)"}
    del dx, dy, o, hT, o_dec, ws
    torch.cuda.empty_cache()
    return out


def config_obj(c, dec_steps, N, world):
    """The `config` object of the JSON line (shared by both arms)."""
    B, T, H = c["B"], c["T"], c["H"]
    return {"workload": c["name"] + (" + %d decode step(s) at N=%d" % (dec_steps, N)
                                     if dec_steps else ""),
            "variant": c["variant"], "B": B, "T": T, "H": H, "dk": c["dk"], "dv": c["dv"],
            "chunk": 64, "token_heads_per_step": B * T * H + N * H * dec_steps,
            "prefill_token_heads": B * T * H, "decode_token_heads": N * H * dec_steps,
            "parallelism": "replica per GPU" if world > 1 else "single GPU"}


def oracle_sample(xp, yd, nthreads):
    """The float64 oracle (C token recurrence, OpenMP over (batch, head)) on a
    sample of a workload: prefill sequences xp ([B, T, H, d] tensors, each from
    its h0 or zero) and decode sequences yd ([steps, N, H, d] per-token tensors
    from their starting states yd["h0"]), the latter run as N sequences of
    `steps` tokens. Returns (token-heads, seconds)."""
    from oracle import native

    f64 = lambda t: None if t is None else t.detach().double().cpu().numpy()
    names = ("q", "k", "v", "g", "beta", "lam", "b", "w")
    jobs = [(({n: f64(xp[n]) for n in names}), f64(xp["h0"]))]
    if yd is not None:
        jobs.append(({n: (None if yd[n] is None else f64(yd[n].transpose(0, 1)))
                      for n in names}, f64(yd["h0"])))
    th, secs = 0, 0.0
    for arrs, h0 in jobs:
        t0 = time.perf_counter()
        native.recurrence(arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"], arrs["lam"],
                          arrs["b"], arrs["w"], h0, xp["scale"], xp["flags"], nthreads=nthreads)
        secs += time.perf_counter() - t0
        th += arrs["q"].shape[0] * arrs["q"].shape[1] * arrs["q"].shape[2]
    return th, secs


def cpu_baseline(x, y, dec_steps, budget_s=12.0):
    """The oracle as it stands, timed on all host cores on a bounded sample of the
    step's workload: the prefill of batch row 0 for up to 16 heads over every
    token, and (where the decode phase starts from its own states) the decode
    of every sequence for up to 4 heads over all its steps; repeated until
    ~budget_s or three passes."""
    from oracle import native

    H = x["q"].shape[2]
    hs = slice(0, min(H, 16))
    sel = lambda t, hsl: None if t is None else t[0:1, :, hsl]
    xp = {n: sel(x[n], hs) for n in ("q", "k", "v", "g", "beta", "lam", "b", "w")}
    xp.update(h0=None if x["h0"] is None else x["h0"][0:1, hs], scale=x["scale"],
              flags=x["flags"])
    yd = None
    if y.get("h0") is not None and dec_steps > 0:
        hd = slice(0, min(H, 4))
        yd = {n: (None if y[n] is None else y[n][:dec_steps, :, hd])
              for n in ("q", "k", "v", "g", "beta", "lam", "b", "w")}
        yd["h0"] = y["h0"][:, hd]
    cores = native.max_threads()
    reps, th_total, t_total = 0, 0, 0.0
    while reps == 0 or (t_total < budget_s and reps < 3):
        th, t = oracle_sample(xp, yd, cores)
        th_total += th
        t_total += t
        reps += 1
    npre = xp["q"].shape[1] * xp["q"].shape[2]
    what = "prefill of %d (batch, head) sequences x %d tokens" % (xp["q"].shape[2],
                                                                xp["q"].shape[1])
    if yd is not None:
        what += " + decode of %d sequences x %d heads x %d steps from their states" % (
            yd["q"].shape[1], yd["q"].shape[2], yd["q"].shape[0])
    return {"value": round(th_total / t_total, 1), "unit": UNIT, "cores": cores,
            "kind": "oracle", "sample": what + "; %d token-heads per pass (%d prefill), %d "
            "pass(es); C fp64 token recurrence, OpenMP over (batch, head)" % (
                th_total // reps, npre, reps), "seconds": round(t_total, 3)}


def run_reference(args):
    """The float64 oracle, as it stands, on the host cores, on the same workload's
    recipe at a bounded sample size per step: the prefill of 16 heads over 8192
    tokens and the decode of every sequence of 2 heads over 128 steps (where the
    workload has a decode phase from its own states)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import native
    cfg = args.workload
    c = wl.CONFIGS[cfg]
    dec_steps, N = decode_of(cfg, c["B"])
    if args.decode_steps is not None:
        dec_steps = args.decode_steps
    xp = wl.config_inputs(cfg, B=1, T=min(c["T"], 8192), H=min(c["H"], 16))
    yd = None
    if "decode" in c and dec_steps > 0:
        yd = wl.decode_phase_inputs(cfg, steps=min(dec_steps, 128), H=min(c["H"], 2))
    cores = native.max_threads()
    for _ in range(args.warmup):
        oracle_sample(dict(xp, q=xp["q"][:, :64], k=xp["k"][:, :64], v=xp["v"][:, :64],
                           g=xp["g"][:, :64],
                           **{n: (None if xp[n] is None else xp[n][:, :64])
                              for n in ("beta", "lam", "b", "w")}), None, cores)
    th_total, t_total = 0, 0.0
    for _ in range(args.steps):
        th, t = oracle_sample(xp, yd, cores)
        th_total += th
        t_total += t
    value = th_total / t_total
    sample = "prefill of %d sequences x %d tokens" % (xp["q"].shape[2], xp["q"].shape[1])
    if yd is not None:
        sample += " + decode of %d sequences x %d heads x %d steps" % (
            yd["q"].shape[1], yd["q"].shape[2], yd["q"].shape[0])
    res = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * t_total / args.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": config_obj(c, dec_steps, N, world),
           "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cores,
                            "kind": "oracle",
                            "sample": sample + " per step (same recipe as the workload, "
                                      "%d token-heads), all host cores" % (th_total //
                                                                          args.steps)},
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
