"""Throughput of the P-EAGLE parallel draft pass on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  draft (fc + input fusion, N decoder layers, LM head + argmax + d2t; peagle_draft),
  greedy verification (peagle_verify_greedy), KV commit of the NTP row plus the accepted
  drafts (peagle_append_kv), and a reset of seq_lens so every step drafts from the same
  committed context.  The metric is draft tokens per second (batch x K per step) for the
  decode-shaped bf16 drafter: H=2880, 4 layers, 64/8 heads of 64, I=7680, Vd=32000 ->
  Vt=201088, batch 1, 4096 cached positions, K=8.  The step is captured in a CUDA graph
  and replayed; each replay streams 1.04 GB (weights + KV), far more than the 129 MB L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload decode_b1|decode_b2|ragged_b16]

Five extra objects on the line: decode_configs (the draft pass on the concurrency-2 and
the ragged batch-16 workloads, each with its HBM roofline), train_fwd (the training-style
masked forward, n=2048, K=8, COD 0.8), train_step (the same rows: forward, mean cross-entropy and every parameter
gradient), sliding_window (the concurrency-2 workload with and without a 4096-position
drafter attention window) and efficient_head (the headline workload with the rank-128 /
top-128 LM head and with the full head, on the 32000-entry draft vocabulary and on the
whole 201088-entry vocabulary); --no-configs / --no-train-fwd / --no-train-step /
--no-window / --no-head skip them, and --only NAME runs one of them alone (a short driver
for profilers).

--impl reference times the fp64 oracle on the host cores instead (a deliberately slow
plain program; see the cpu_baseline object).  Under torchrun each rank runs an
independent replica on its own GPU (the pass shards by request: no collective).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

DEFAULT_WORKLOAD = "decode_b1"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=["decode_b1", "decode_b2", "ragged_b16"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other decode workloads (decode_b2, ragged_b16)")
    ap.add_argument("--no-train-fwd", action="store_true",
                    help="skip the training-style masked forward measurement")
    ap.add_argument("--no-window", action="store_true",
                    help="skip the sliding-window attention measurement")
    ap.add_argument("--no-head", action="store_true",
                    help="skip the efficient LM head measurement")
    ap.add_argument("--no-train-step", action="store_true",
                    help="skip the training step measurement")
    ap.add_argument("--train-seq", type=int, default=0,
                    help="with --only train_step: a shorter sequence than the workload's "
                         "(a small case for profiler captures)")
    ap.add_argument("--train-layers", type=int, default=0,
                    help="with --only train_step: fewer decoder layers (profiler captures)")
    ap.add_argument("--only", choices=["train_fwd", "train_step", "window", "head_draft_vocab",
                                       "head_full_vocab", "decode_b2", "ragged_b16"],
                    help="run one of the extra measurements alone and print its object "
                         "(a short driver for profilers)")
    return ap.parse_args()


# ---------------------------------------------------------------------------- helpers


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.5)  # let the sampler start before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# DRAM bytes (read + write) of one pass-kernel launch on decode_b1: dram__bytes_read.sum +
# dram__bytes_write.sum of one ncu capture of the current pass kernel (None when the kernel
# has changed since the counters were taken)
PASS_KERNEL_DECODE_B1_DRAM_BYTES = 1_052_764_160


def gemm_weight_bytes(dims) -> int:
    """Weight bytes one draft pass streams through the projections."""
    H, I, Vd = dims.hidden, dims.intermediate, dims.draft_vocab
    qkv = dims.qkv_out
    p = H * 3 * H + Vd * H
    for layer in range(dims.n_layers):
        din = 2 * H if layer == 0 else H
        p += qkv * din + H * dims.n_q_heads * dims.head_dim + 2 * I * H + H * I
    return p * 2


def kv_bytes(dims, lens, K) -> int:
    """KV-cache bytes the attention reads per pass (committed context + draft block)."""
    per_pos = dims.n_layers * dims.n_kv_heads * dims.head_dim * 2 * 2
    return int(sum(int(L) + K for L in lens)) * per_pos


def masked_pairs(rp, rd) -> int:
    """Allowed (query, key) pairs of the training mask over retained rows (p, d): every
    row sees the depth-1 keys at positions 0 .. p-d+1 and the d-1 deeper rows of its own
    chain, plus itself."""
    import numpy as np

    p, d = np.asarray(rp, np.int64), np.asarray(rd, np.int64)
    return int(((p - d + 1) + 1).sum() + (d - 1).sum())


def forward_flops(dims, rp, rd) -> float:
    """Algorithmic FLOPs of the training-style forward over the retained rows: 2 per
    multiply-add of every projection for every row that needs it (fc only for the depth-1
    rows -- the deeper rows share the constant fc(h_shared); every layer and the LM head
    for all rows) plus 4 * nq * hd per allowed (query, key) pair in each of the N layers
    (the score and the value products)."""
    import numpy as np

    M = len(rp)
    n1 = int((np.asarray(rd) == 1).sum())
    params = gemm_weight_bytes(dims) // 2
    fc = dims.hidden * 3 * dims.hidden
    gemm = 2.0 * (M * (params - fc) + n1 * fc)
    attn = 4.0 * dims.n_layers * dims.n_q_heads * dims.head_dim * masked_pairs(rp, rd)
    return gemm, attn


def whole_job(dist, ms_step, units_per_rank, world, device):
    """Whole-job throughput of `world` independent replicas (weak scaling): the units all
    ranks processed over the slowest rank's step time, the max taken over ranks by a
    collective when `dist` is given.  Returns (max ms per step, units per second)."""
    import torch

    ms_max = float(ms_step)
    if dist:
        t = torch.tensor([ms_max], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
    return ms_max, world * units_per_rank / (ms_max * 1e-3)


# ---------------------------------------------------------------------------- our arm


def run_ours(args, rank, world, dist):
    import torch

    import drafting_eagle_draft_gb300 as pk

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS[args.workload]
    dims = wl.dims
    w = synth.make_weights(dims, 1234)
    inp = synth.make_decode_inputs(wl, 99)
    B, K, cap = wl.batch, wl.K, inp["capacity"]
    R = B * K
    ctx = pk.peagle_create(w, pk.make_dims(dims, B, K, cap))
    del w
    ck = inp["cache_k"].to(dev)
    cv = inp["cache_v"].to(dev)
    kv = pk.kv_struct(ck, cv, cap, B)
    sl0 = torch.from_numpy(inp["seq_lens"]).to(dev)
    sl = sl0.clone()
    th = inp["target_hidden"].to(dev)
    nt = torch.from_numpy(inp["new_token"]).to(dev)
    toks = torch.zeros(B, K, dtype=torch.int32, device=dev)
    acc = torch.zeros(B, dtype=torch.int32, device=dev)
    bonus = torch.zeros(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # target argmax agreeing with the drafts on a geometric(0.7) prefix
    with torch.cuda.stream(stream):
        pk.peagle_draft(ctx, B, kv, sl, th, nt, K, toks, None, stream)
    stream.synchronize()
    tgt_np, _ = synth.geometric_target_argmax(toks.cpu().numpy(), dims.target_vocab, 0.7, 6)
    tgt = torch.from_numpy(tgt_np).to(dev)

    # the step commits the draft block's NTP row (the new token's K/V; the accepted drafts'
    # own K/V come from a catch-up pass with their target hidden states)
    ntp_only = torch.zeros(B, dtype=torch.int32, device=dev)

    def step():
        sl.copy_(sl0)
        pk.peagle_draft(ctx, B, kv, sl, th, nt, K, toks, None, stream)
        pk.peagle_verify_greedy(B, K, toks, tgt, acc, bonus, stream)
        pk.peagle_append_kv(ctx, B, kv, sl, ntp_only, stream=stream, n_extra=1)

    # warm-up (eager), then capture one step in a CUDA graph
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    assert pk.peagle_status(ctx) == pk.PEAGLE_OK
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    ms_step = ms / args.steps
    assert pk.peagle_status(ctx) == pk.PEAGLE_OK

    # the draft pass alone, as its own CUDA graph, timed with events on its stream: the
    # duration of the dominant kernel (the persistent pass kernel, or the multi-kernel
    # sequence when that is disabled)
    sl.copy_(sl0)
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph, stream=stream):
        pk.peagle_draft(ctx, B, kv, sl, th, nt, K, toks, None, stream)
    reps_d = max(args.steps, 20)
    with torch.cuda.stream(stream):
        for _ in range(3):
            dgraph.replay()
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(reps_d):
            dgraph.replay()
        d1.record(stream)
    d1.synchronize()
    draft_ms = d0.elapsed_time(d1) / reps_d

    # per-stage timing of the same step (the pass kernel's phase trace, or CUDA events
    # around each launch of the multi-kernel path)
    pk.peagle_set_timing(ctx, True)
    stage_ms = {k: 0.0 for k in pk.STAGES}
    stage_n = {k: 0 for k in pk.STAGES}
    reps = 5
    with torch.cuda.stream(stream):
        step()
        pk.peagle_read_timing(ctx)
        for _ in range(reps):
            step()
            t = pk.peagle_read_timing(ctx)
            for k, (m_, n_) in t.items():
                stage_ms[k] += m_ / reps
                stage_n[k] = n_
    pass_kernel = pk.peagle_read_pass_trace(ctx) is not None
    pk.peagle_set_timing(ctx, False)
    if pass_kernel:
        launches_per_step = 3  # pass kernel, verify, KV commit
    else:
        launches_per_step = sum(stage_n.values()) + 1  # + verify (context-free)

    # end to end through the public API with host buffers (pinned), copies in the region:
    # one packed host->device copy of the step's inputs (target hidden states, new tokens,
    # seq_lens) and one packed device->host copy of its results (draft tokens, accepted
    # lengths, bonus tokens)
    th_b = inp["target_hidden"].numel() * inp["target_hidden"].element_size()
    h2d = th_b + 4 * B + 4 * B
    in_h = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    in_h[:th_b].copy_(inp["target_hidden"].contiguous().view(-1).view(torch.uint8))
    in_h[th_b:th_b + 4 * B].copy_(torch.from_numpy(inp["new_token"]).view(torch.uint8))
    in_h[th_b + 4 * B:].copy_(torch.from_numpy(inp["seq_lens"]).view(torch.uint8))
    in_d = torch.empty(h2d, dtype=torch.uint8, device=dev)
    th_e = in_d[:th_b].view(th.dtype).view(th.shape)
    nt_e = in_d[th_b:th_b + 4 * B].view(torch.int32)
    sl_e = in_d[th_b + 4 * B:].view(torch.int32)
    out_d = torch.empty(B * K + 2 * B, dtype=torch.int32, device=dev)
    toks_e = out_d[:B * K].view(B, K)
    acc_e, bonus_e = out_d[B * K:B * K + B], out_d[B * K + B:]
    out_h = torch.empty(B * K + 2 * B, dtype=torch.int32).pin_memory()
    d2h = out_h.numel() * 4

    def e2e_step():
        in_d.copy_(in_h, non_blocking=True)
        pk.peagle_draft(ctx, B, kv, sl_e, th_e, nt_e, K, toks_e, None, stream)
        pk.peagle_verify_greedy(B, K, toks_e, tgt, acc_e, bonus_e, stream)
        pk.peagle_append_kv(ctx, B, kv, sl_e, ntp_only, stream=stream, n_extra=1)
        out_h.copy_(out_d, non_blocking=True)
        stream.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        t1 = time.perf_counter()
    e2e_ms = (t1 - t0) * 1e3 / args.e2e_steps

    # roofline of the dominant kernel: algorithmic bytes of one draft pass (every weight
    # once, the KV cache of the committed context and the draft block) over its duration
    wbytes = gemm_weight_bytes(dims)
    pk_ = peaks()
    lens = inp["seq_lens"]
    total_bytes = wbytes + kv_bytes(dims, lens, K)
    roofline_us = total_bytes / (pk_["hbm_gbs"] * 1e9) * 1e6
    traffic = None
    if pass_kernel:
        kern = "pass_kernel (the whole draft pass, one launch)"
        kern_bytes, kern_ms, kern_launches = total_bytes, draft_ms, 1
        if wl.name == "decode_b1":
            traffic = PASS_KERNEL_DECODE_B1_DRAM_BYTES
    else:
        gemm_stages = ("fc", "qkv", "oproj", "gate_up", "down", "lm_head")
        kern = "tc_gemm_kernel (all projection launches)"
        kern_bytes = wbytes
        kern_ms = sum(stage_ms[k] for k in gemm_stages)
        kern_launches = sum(stage_n[k] for k in gemm_stages)
    achieved = kern_bytes / (kern_ms * 1e-3) / 1e9

    # whole job: tokens of all ranks / max time over ranks
    ms_max, total_tok_s = whole_job(dist, ms_step, R, world, dev)

    out = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(wl, inp, budget_s=12.0)
        out = {
            "metric": "draft tokens/s", "value": round(total_tok_s, 2), "unit": "tok/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_max, 5), "us_per_pass": round(ms_max * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded; random-init weights)",
            "config": {"workload": wl.name, "batch": B, "K": K, "kv_len": [int(x) for x in lens],
                       "hidden": dims.hidden, "layers": dims.n_layers,
                       "heads": [dims.n_q_heads, dims.n_kv_heads, dims.head_dim],
                       "intermediate": dims.intermediate,
                       "vocab": [dims.draft_vocab, dims.target_vocab],
                       "l2": "inputs larger than L2: %.2f GB streamed per step vs 129 MB L2"
                             % (total_bytes / 1e9),
                       "parallelism": f"replicas x{world}", "graph": "CUDA graph per step"},
            "roofline": {"bound": "hbm", "kernel": kern,
                         "achieved": round(achieved, 1), "peak": pk_["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / pk_["hbm_gbs"], 4), "traffic": traffic,
                         "bytes_per_launch": kern_bytes, "launches_per_step": kern_launches,
                         "kernel_ms_per_step": round(kern_ms, 4),
                         "peak_source": pk_["source"] + " (burst copy)",
                         "pass_roofline_us": round(roofline_us, 2),
                         "pass_frac": round(roofline_us / (ms_max * 1e3), 4)},
            "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "e2e": {"value": round(R / (e2e_ms * 1e-3), 2), "unit": "tok/s",
                    "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h)},
            "gpu_launches": int(launches_per_step * args.steps),
            "clocks": clk,
        }
        if cpu:
            out["cpu_baseline"] = cpu
    ctx.close()
    if rank == 0 and world == 1 and not args.no_configs:
        out["decode_configs"] = {nm: decode_config_measure(dev, nm)
                                 for nm in ("decode_b2", "ragged_b16") if nm != wl.name}
    if rank == 0 and world == 1 and not args.no_train_fwd:
        out["train_fwd"] = train_fwd_measure(dev)
    if rank == 0 and world == 1 and not args.no_window:
        out["sliding_window"] = window_measure(dev)
    if rank == 0 and world == 1 and not args.no_head:
        out["efficient_head"] = head_measure(dev)
    if rank == 0 and world == 1 and not args.no_train_step:
        out["train_step"] = train_step_measure(dev)
    return out


def _pass_us(dev, wl, dims, w, inp, reps=20):
    """Draft-pass time of one context on `inp`, replayed as a CUDA graph (microseconds)."""
    import torch

    import drafting_eagle_draft_gb300 as pk

    B, K, cap = wl.batch, wl.K, inp["capacity"]
    ck, cv = inp["cache_k"].to(dev), inp["cache_v"].to(dev)
    kv = pk.kv_struct(ck, cv, cap, B)
    sl = torch.from_numpy(inp["seq_lens"]).to(dev)
    th = inp["target_hidden"].to(dev)
    nt = torch.from_numpy(inp["new_token"]).to(dev)
    ctx = pk.peagle_create(w, pk.make_dims(dims, B, K, cap))
    toks = torch.zeros(B, K, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for _ in range(3):
            pk.peagle_draft(ctx, B, kv, sl, th, nt, K, toks, None, s)
    s.synchronize()
    assert pk.peagle_status(ctx) == pk.PEAGLE_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pk.peagle_draft(ctx, B, kv, sl, th, nt, K, toks, None, s)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    e1.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    out = toks.cpu().numpy()
    ctx.close()
    return us, out


def decode_config_measure(dev, name):
    """Draft-pass time of another decode workload (decode_b2: concurrency 2, contexts 8192 /
    10240, K=8; ragged_b16: the H=4096 drafter, 16 requests with contexts U[1024, 8192],
    K=5) as a CUDA graph, with its HBM roofline: algorithmic bytes (every weight once, the
    committed KV context and the draft block) over the pass time, against the measured
    copy bandwidth."""
    wl = synth.WORKLOADS[name]
    dims = wl.dims
    w = synth.make_weights(dims, 1234)
    inp = synth.make_decode_inputs(wl, 99)
    us, _ = _pass_us(dev, wl, dims, w, inp)
    del w
    lens = [int(x) for x in inp["seq_lens"]]
    nbytes = gemm_weight_bytes(dims) + kv_bytes(dims, lens, wl.K)
    pk_ = peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    R = wl.batch * wl.K
    return {"workload": name, "batch": wl.batch, "K": wl.K,
            "kv_len": lens if len(lens) <= 2 else {"min": min(lens), "max": max(lens),
                                                  "mean": round(sum(lens) / len(lens), 1)},
            "us_per_pass": round(us, 2), "draft_tok_s": round(R / (us * 1e-6), 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk_["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / pk_["hbm_gbs"], 4),
                         "bytes_per_pass": nbytes,
                         "pass_roofline_us": round(nbytes / (pk_["hbm_gbs"] * 1e3), 2),
                         "peak_source": pk_["source"] + " (burst copy)"}}


def window_measure(dev, window=4096):
    """Sliding-window drafter attention on the concurrency-2 workload (contexts 8192 and
    10240, K=8): draft-pass time as a CUDA graph with a 4096-position window and with full
    attention on the same inputs, and the cached keys / values each pass reads."""
    wl = synth.WORKLOADS["decode_b2"]
    w = synth.make_weights(wl.dims, 1234)
    inp = synth.make_decode_inputs(wl, 99)
    K = wl.K
    res = {name: _pass_us(dev, wl, synth.shrink(wl.dims, attn_window=W), w, inp)[0]
           for name, W in (("window", window), ("full", 0))}
    lens = [int(x) for x in inp["seq_lens"]]
    kvb = lambda span: sum(span(L) for L in lens) * wl.dims.n_kv_heads * wl.dims.head_dim * 2 * 2 \
        * wl.dims.n_layers
    return {"workload": "decode_b2 (contexts %s, K=%d)" % ("/".join(map(str, lens)), K),
            "window": window, "us_per_pass": round(res["window"], 2),
            "us_per_pass_full": round(res["full"], 2),
            "kv_bytes_per_pass": kvb(lambda L: min(L + K, window + K - 1)),
            "kv_bytes_per_pass_full": kvb(lambda L: L + K)}


def head_measure(dev, rank=128, topk=128, vocabs=("draft_vocab", "full_vocab")):
    """Efficient LM head on the headline workload (batch 1, 4096 cached positions, K=8):
    draft-pass time as a CUDA graph with the rank-128 scoring projection and the full head
    on its 128 best candidates, against the full head on the same weights and inputs, the
    head bytes each pass reads (candidate rows counted once per draft row), and how many
    of the K drafted tokens the two agree on.  Measured on the 32000-entry draft vocabulary
    and on the whole 201088-entry target vocabulary as the draft vocabulary (no d2t), the
    setting the efficient head is meant for."""
    wl = synth.WORKLOADS["decode_b1"]
    inp = synth.make_decode_inputs(wl, 99)
    out = {}
    for name, vocab in (("draft_vocab", None), ("full_vocab", wl.dims.target_vocab)):
        if name not in vocabs:
            continue
        d = synth.shrink(wl.dims, lm_rank=rank, lm_topk=topk)
        if vocab:
            d = synth.shrink(d, draft_vocab=vocab, d2t="identity")
        w = synth.make_weights(d, 1234)
        eff, t_eff = _pass_us(dev, wl, d, w, inp)
        full, t_full = _pass_us(dev, wl, synth.shrink(d, lm_rank=0, lm_topk=0), w, inp)
        H, Vd, R = d.hidden, d.draft_vocab, wl.batch * wl.K
        out[name] = {
            "workload": "decode_b1 (context 4096, K=8), Vd %d, rank %d, top %d" % (Vd, rank, topk),
            "us_per_pass": round(eff, 2), "us_per_pass_full_head": round(full, 2),
            "head_bytes_per_pass": 2 * (rank * H + Vd * rank + R * topk * H),
            "head_bytes_per_pass_full_head": 2 * Vd * H,
            "tokens_equal_full_head": int((t_eff == t_full).sum()), "tokens": int(t_eff.size)}
        del w
    return out


def train_fwd_measure(dev, reps=3):
    """Training-style masked forward of the decode drafter (n=2048, K=8, COD 0.8): time per
    forward with CUDA events, and the tensor-core roofline of its algorithmic FLOPs
    (forward_flops) against the measured bf16 burst peak."""
    import torch

    import drafting_eagle_draft_gb300 as pk

    wl = synth.WORKLOADS["train_fwd"]
    dims = wl.dims
    w = synth.make_weights(dims, 1234)
    ti = synth.make_train_inputs(wl, 21)
    n, K = wl.n_seq, wl.K
    rp, rd = pk.peagle_cod_rows(n, K, wl.cod_ratio, ti["cod_u"])
    M = len(rp)
    ctx = pk.peagle_create(w, pk.make_dims(dims, 1, K, n, max_rows=M, max_seq=n))
    del w
    tok = torch.from_numpy(ti["tokens"]).to(dev)
    hid = ti["hidden"].to(dev)
    rpd = torch.from_numpy(rp).to(dev)
    rdd = torch.from_numpy(rd).to(dev)
    am = torch.empty(M, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream(device=dev)

    def fwd():
        pk.peagle_forward_parallel(ctx, n, K, tok, hid, rpd, rdd, M, am, None, s)

    with torch.cuda.stream(s):
        fwd()
    s.synchronize()
    assert pk.peagle_status(ctx) == pk.PEAGLE_OK
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(reps):
            fwd()
        e1.record(s)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    pk.peagle_set_timing(ctx, True)
    with torch.cuda.stream(s):
        fwd()
    st = pk.peagle_read_timing(ctx)
    ctx.close()
    gemm_flops, attn_flops = forward_flops(dims, rp, rd)
    pk_ = peaks()
    tflops = (gemm_flops + attn_flops) / (ms * 1e-3) / 1e12
    return {"workload": wl.name, "rows": M, "ms": round(ms, 3),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1),
                         "peak": pk_["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tflops / pk_["bf16_tflops"], 4),
                         "peak_source": pk_["source"] + " bf16 burst (a forward of ~15 ms)",
                         "flops": "projections 2 x rows x params (fc for depth-1 rows only) "
                                  "+ attention 4 x N x nq x hd x allowed pairs"},
            "algorithmic_tflop": round((gemm_flops + attn_flops) / 1e12, 3),
            "gemm_tflop": round(gemm_flops / 1e12, 3), "attn_tflop": round(attn_flops / 1e12, 3),
            "stages_ms": {k: round(v[0], 3) for k, v in st.items()}}


def train_step_measure(dev, reps=3, n_seq=0, n_layers=0):
    """Training step without optimizer on the training workload (decode drafter, n=2048,
    K=8, COD 0.8): ms per step (forward with kept activations, mean cross-entropy, every
    parameter gradient) with CUDA events, and its algorithmic FLOPs against the TF32 peak
    (the GEMMs run on TF32 tensor cores): three times the forward's (forward_flops: every
    projection forward, dX and dW; attention forward 2 products, backward 4)."""
    import numpy as np
    import torch

    import drafting_eagle_draft_gb300 as pk

    wl = synth.WORKLOADS["train_fwd"]
    if n_seq or n_layers:  # a reduced case (profiler captures), never a bench line
        wl = dataclasses.replace(wl, n_seq=n_seq or wl.n_seq,
                                 dims=synth.shrink(wl.dims, n_layers=n_layers or wl.dims.n_layers))
    dims = wl.dims
    w = synth.make_weights(dims, 1234)
    ti = synth.make_train_inputs(wl, 21)
    n, K = wl.n_seq, wl.K
    rp, rd = pk.peagle_cod_rows(n, K, wl.cod_ratio, ti["cod_u"])
    M = len(rp)
    ctx = pk.peagle_create(w, pk.make_dims(dims, 1, K, n, max_rows=M, max_seq=n, train=True))
    del w
    H, I, nq, nkv, hd, L = (dims.hidden, dims.intermediate, dims.n_q_heads, dims.n_kv_heads,
                            dims.head_dim, dims.n_layers)
    z = lambda *shape: torch.empty(shape, dtype=torch.float32, device=dev)  # noqa: E731
    qo = (nq + 2 * nkv) * hd
    g = {"embed": None, "emb_mask": z(H), "h_shared": z(3 * H), "fc": z(H, 3 * H),
         "input_norm": z(H), "hidden_norm": z(H), "final_norm": z(H),
         "lm_head": z(dims.draft_vocab, H),
         "qkv": [z(qo, 2 * H if l == 0 else H) for l in range(L)],
         "o": [z(H, nq * hd) for _ in range(L)], "attn_norm": [z(H) for _ in range(L)],
         "post_norm": [z(H) for _ in range(L)], "gate": [z(I, H) for _ in range(L)],
         "up": [z(I, H) for _ in range(L)], "down": [z(H, I) for _ in range(L)]}
    gs = pk.grads_struct(g, L)
    tok = torch.from_numpy(ti["tokens"]).to(dev)
    hid = ti["hidden"].to(dev)
    rpd = torch.from_numpy(rp).to(dev)
    rdd = torch.from_numpy(rd).to(dev)
    lab = torch.from_numpy(
        np.random.default_rng(5).integers(0, dims.draft_vocab, M).astype(np.int32)).to(dev)
    loss = torch.zeros(1, device=dev)
    s = torch.cuda.Stream(device=dev)

    def step():
        pk.peagle_train_step(ctx, n, K, tok, hid, rpd, rdd, M, lab, loss, gs, s)

    with torch.cuda.stream(s):
        step()
        step()
    s.synchronize()
    assert pk.peagle_status(ctx) == pk.PEAGLE_OK
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(reps):
            step()
        e1.record(s)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    ctx.close()
    gemm_f, attn_f = forward_flops(dims, rp, rd)
    flops = 3.0 * gemm_f + 3.0 * attn_f  # forward, then two products per forward product
    pk_ = peaks()
    # TF32 peak: the measured bf16 burst peak times GB300's nominal dense TF32 / bf16 ratio
    peak = pk_["bf16_tflops"] * 1.1 / 2.25
    tflops = flops / (ms * 1e-3) / 1e12
    return {"workload": wl.name, "n_seq": n, "layers": dims.n_layers, "rows": M,
            "ms": round(ms, 3), "loss": round(loss.item(), 5),
            "tflops": round(tflops, 1), "peak_tflops": round(peak, 1),
            "peak_source": "measured bf16 burst x GB300 nominal dense TF32/bf16 ratio "
                           "(1.1 / 2.25 PFLOP/s)",
            "frac": round(tflops / peak, 4), "algorithmic_tflop": round(flops / 1e12, 3)}


# ---------------------------------------------------------------------------- oracle arm


def cpu_baseline(wl, inp, budget_s=12.0):
    """The fp64 oracle (as it stands) on the host cores: full draft passes of the same
    workload until about budget_s seconds of work have run."""
    from oracle import peagle_oracle as O

    dims = wl.dims
    w = synth.make_weights(dims, 1234)
    W = O.Weights64.from_synth(w, lazy=True)
    K = wl.K
    n = 0
    t0 = time.perf_counter()
    while True:
        O.draft_pass(W, dims, inp["cache_k"], inp["cache_v"], inp["seq_lens"],
                     inp["target_hidden"], inp["new_token"], K, bf16=O.DRAFT_BF16_CASTS)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = (time.perf_counter() - t0) / n
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(wl.batch * K / dt, 3), "unit": "tok/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n} full fp64 draft passes of {wl.name} (all rows, all layers), "
                      f"{dt:.2f} s each; numpy BLAS threads over {cores} cores"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from oracle import peagle_oracle as O

    wl = synth.WORKLOADS[args.workload]
    dims = wl.dims
    w = synth.make_weights(dims, 1234)
    W = O.Weights64.from_synth(w, lazy=True)
    inp = synth.make_decode_inputs(wl, 99)
    K = wl.K

    def step():
        r = O.draft_pass(W, dims, inp["cache_k"], inp["cache_v"], inp["seq_lens"],
                         inp["target_hidden"], inp["new_token"], K, bf16=O.DRAFT_BF16_CASTS)
        tgt, _ = synth.geometric_target_argmax(r.tokens, dims.target_vocab, 0.7, 6)
        acc, _ = O.verify_greedy(r.tokens, tgt)
        return acc

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    v = wl.batch * K / dt
    return {"impl": "reference", "metric": "draft tokens/s", "value": round(v, 3), "unit": "tok/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; random-init weights)",
            "config": {"workload": wl.name, "batch": wl.batch, "K": K,
                       "kv_len": [int(x) for x in inp["seq_lens"]]},
            "cpu_baseline": {"value": round(v, 3), "unit": "tok/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"each step one full fp64 oracle draft pass of {wl.name} "
                                       "plus greedy verification"},
            "e2e": {"value": round(v, 3), "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------- main


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    dist = None
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    elif args.only:
        import torch

        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        if args.only == "train_fwd":
            out = {"train_fwd": train_fwd_measure(dev)}
        elif args.only == "train_step":
            out = {"train_step": train_step_measure(dev, n_seq=args.train_seq,
                                                    n_layers=args.train_layers)}
        elif args.only == "window":
            out = {"sliding_window": window_measure(dev)}
        elif args.only in ("decode_b2", "ragged_b16"):
            out = {"decode_configs": {args.only: decode_config_measure(dev, args.only)}}
        else:
            out = {"efficient_head": head_measure(dev, vocabs=(args.only[5:],))}
    else:
        if world > 1:
            import torch
            import torch.distributed as tdist

            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            tdist.init_process_group("nccl")
            dist = tdist
        out = run_ours(args, rank, world, dist)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
