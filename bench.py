"""Benchmark of one decoder-block forward pass on GB300, as one JSON line.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                [--no-sub-configs] [--no-cpu-baseline]

A step is one blk_forward over the workload's synthetic batch (all stages of the
block). Default workload: the largest configuration, the Apertus-shape bf16
prefill block (batch 2 x 4096 tokens, q/k-norm, xIELU 16384). The same process
then times the Llama-7B-shape prefill (1 x 2048), the Arcee-shape prefill
(4 x 2048) and the decode step (64 sequences over 4096 cached positions) the same
way, each as its own record under "configs". Inputs and weights are resident in
HBM before timing; L2 is flushed between timed steps, outside the timed events:
a 256 MiB buffer is written and then read, so the flush's own dirty lines are
written back before the step starts and the step begins with none of its
operands in L2. value is whole-job tokens/s; e2e repeats the measurement with
the input copied from pinned host memory and the output read back inside each
step, pipelined as a serving loop runs it: two input/output buffer pairs, the
next step's upload and the previous step's read-back on their own copy streams
beside each forward. e2e_serial does each step's upload, forward and read-back
in turn on one stream.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload, one sample per step (the only other place this script runs the oracle
is the cpu_baseline leg of our own line, which repeats that same sample).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decoder-block tokens/s (bf16, 1×GB300) and % of BF16 tensor-core / HBM roofline"
DEFAULT_WORKLOAD = "apertus_qknorm_bf16_B2_T4096"
# timed after the headline in the same process, each as its own record under "configs"
SUB_CONFIGS = ("llama7b_bf16_B1_T2048", "arcee_gqa_bf16_B4_T2048", "llama7b_decode_bf16_B64_L4096")
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu capture, or None when the
    kernel's source changed since the capture (or none exists for this workload)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[kernel].get(workload)  # {kernel: {workload: record}}
        if t is None:
            return None
        src = open(os.path.join(ROOT, t["source"]), "rb").read()
        if hashlib.sha256(src).hexdigest()[:16] != t["sha256_16"]:
            return None
        return t["dram_bytes"]
    except Exception:
        return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 50 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def wait_first_sample(self, timeout=3.0):
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < timeout:
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.02)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- work counts

def work_counts(wl):
    """Algorithmic FLOPs and bytes of the block and of each stage (one step)."""
    B, T, D, H, Hkv, d, F = wl.batch, wl.seq, wl.hidden_size, wl.num_heads, wl.num_kv_heads, wl.head_dim, \
        wl.intermediate_size
    M = B * T
    es = 2 if wl.dtype == "bf16" else 4
    n_up = 2 * F if wl.hidden_act == "silu" else F
    n_qkv = (2 * H if wl.attn_gate else H) + 2 * Hkv  # heads of the fused projection (+ the attention gate)
    W = wl.sliding_window

    def keys_seen(first_pos, n):  # keys visible to the queries at positions first_pos .. first_pos + n - 1
        return float(sum(min(p + 1, W) if W else p + 1 for p in range(first_pos, first_pos + n)))

    g = {"qkv": 2.0 * M * D * n_qkv * d, "o": 2.0 * M * H * d * D, "up": 2.0 * M * D * n_up,
         "down": 2.0 * M * F * D}
    if wl.cache_len and T == 1:
        L = keys_seen(wl.cache_len, 1)
        g["attn"] = 4.0 * B * H * d * L
        kv_bytes = 2.0 * B * Hkv * L * d * es
    elif wl.cache_len:  # a prefill chunk: query t sees the keys up to position cache_len + t
        g["attn"] = 4.0 * B * H * d * keys_seen(wl.cache_len, T)
        first = max(0, wl.cache_len - W + 1) if W else 0
        kv_bytes = 2.0 * B * Hkv * (wl.cache_len + T - first) * d * es
    else:
        g["attn"] = 4.0 * B * H * d * keys_seen(0, T)
        kv_bytes = 0.0
    weight_bytes = es * (D * n_qkv * d + H * d * D + n_up * D + F * D + (4 if wl.sandwich_norm else 2) * D)
    if wl.n_layers:  # the model: every layer, plus lm_head
        g = {k: v * wl.n_layers for k, v in g.items()}
        g["lm_head"] = 2.0 * M * D * wl.vocab
        weight_bytes = weight_bytes * wl.n_layers + es * (2 * wl.vocab * D + D)
    return g, weight_bytes, kv_bytes


# ---------------------------------------------------------------- oracle (CPU)

def cpu_sample_cap(wl):
    """Tokens (prefill) or sequences (decode) of one bounded oracle sample, the same on both arms."""
    return 2 if (wl.cache_len and wl.seq == 1) else min(wl.seq, 1024)


def oracle_tokens_per_s(wl, w_cpu, x_cpu, cache_cpu, tokens_cap):
    """fp64 oracle on a bounded sample of the workload; returns (tokens/s, sample text, seconds)."""
    import numpy as np

    import oracle
    cfg = oracle.BlockConfig(wl.hidden_size, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.intermediate_size,
                             wl.hidden_act, wl.rms_norm_eps, wl.rope_theta, wl.qk_norm, wl.xielu_alpha_p,
                             wl.xielu_alpha_n,
                             rope_scaling=oracle.RopeScaling(*wl.rope_scaling) if wl.rope_scaling else None,
                             sliding_window=wl.sliding_window, use_rope=wl.use_rope, attn_gate=wl.attn_gate,
                             sandwich_norm=wl.sandwich_norm)
    wn = {k: v.double().numpy() for k, v in w_cpu.items()}
    t0 = time.perf_counter()
    if wl.cache_len and wl.seq > 1:
        n = min(wl.seq, tokens_cap)
        kc, vc = cache_cpu
        oracle.prefill_with_cache(cfg, wn, x_cpu[:1, :n].double().numpy(), kc[:1].double().numpy(),
                                  vc[:1].double().numpy(), np.full(1, wl.cache_len))
        ntok = n
        sample = f"sequence 0, first {n} of {wl.seq} chunk tokens after a {wl.cache_len}-position cache"
    elif wl.cache_len:
        nb = max(1, min(wl.batch, tokens_cap))
        kc, vc = cache_cpu
        lens = np.full(nb, wl.cache_len)
        oracle.decode_step(cfg, wn, x_cpu[:nb, 0].double().numpy(), kc[:nb].double().numpy(),
                           vc[:nb].double().numpy(), lens)
        ntok = nb
        sample = f"{nb} of {wl.batch} sequences, one decode token each over a {wl.cache_len}-position cache"
    else:
        T = min(wl.seq, tokens_cap)
        oracle.block_forward(cfg, wn, x_cpu[:1, :T].double().numpy())
        ntok = T
        sample = f"sequence 0, first {T} of {wl.seq} tokens (full block, causal prefix)"
    dt = time.perf_counter() - t0
    if wl.n_layers:  # the model: one layer timed, counted once per layer (embedding and lm_head left out)
        dt *= wl.n_layers
        sample += f"; one layer timed and counted {wl.n_layers} times (embedding and lm_head not included)"
    return ntok / dt, sample, dt


def cpu_baseline(wl, w_cpu, x_cpu, cache_cpu, min_seconds):
    """The oracle on repeated bounded samples (the reference arm's per-step sample) for at
    least min_seconds of host time; tokens/s over all repetitions."""
    cap = cpu_sample_cap(wl)
    reps, secs, ntok, sample = 0, 0.0, 0.0, ""
    while reps == 0 or secs < min_seconds:
        tps, sample, dt = oracle_tokens_per_s(wl, w_cpu, x_cpu, cache_cpu, cap)
        reps += 1
        secs += dt
        ntok += tps * dt
    return {"value": ntok / secs, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{sample}; {reps} repetition(s), {secs:.1f} s of host time", "seconds": secs}


def run_reference(args, wl):
    """--impl reference: the fp64 oracle on the host cores, same metric/unit/config."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from llama_family_decoder_gb300.synth import make_input, make_kv_cache, make_weights
    w = make_weights(wl)
    x = make_input(wl)
    cache = make_kv_cache(wl) if wl.cache_len else None
    cap = cpu_sample_cap(wl)  # per step: a bounded sample (about a second or two)
    times, sample, ntok = [], "", 0.0
    for i in range(args.warmup + args.steps):
        tps, sample, dt = oracle_tokens_per_s(wl, w, x, cache, cap)
        if i >= args.warmup:
            times.append(dt)
            ntok += tps * dt
    value = ntok / sum(times)
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl, args.gpus),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{sample}, one per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def config_of(wl, n):
    c = {"workload": wl.name, "batch": wl.batch, "seq": wl.seq, "hidden": wl.hidden_size, "heads": wl.num_heads,
         "kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "ffn": wl.intermediate_size, "act": wl.hidden_act,
         "qk_norm": wl.qk_norm, "l2": "flushed between timed steps (256 MiB written, then read back so that "
                                                       "its dirty lines are written back before the step)",
         "weights": "bf16, with fp16 copies of q/k/v(/gate)/o_proj/gate/up prepared once, outside the timed region",
         "parallelism": "replicas" if n > 1 else "single"}
    if wl.cache_len:
        c["cache_len"] = wl.cache_len
    return c


# ---------------------------------------------------------------- replicas (N > 1)

def rank_seed(wl, rank):
    """Each replica draws its own synthetic batch and weights."""
    return wl.seed + 17 * rank


def max_over_ranks(x, device):
    """The slowest rank's value (the job's time); x itself on one rank."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_step, steps, total_ms):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_step * steps / (total_ms / 1e3)


# ---------------------------------------------------------------- our arm

# Stage names of blk_profile_* -> (roofline kernel name, work key of work_counts)
PREFILL_STAGES = {
    "qkv_gemm_rope": ("tc_gemm_kernel (QKV + q/k-norm + RoPE)", "qkv"),
    "attention": ("attn_tc_kernel (causal flash attention)", "attn"),
    "o_proj_gemm_resid_norm2": ("tc_gemm_kernel (o_proj + residual + norm-2 fold)", "o"),
    "mlp_up_gemm_act": ("tc_gemm_kernel (MLP up/gate + activation)", "up"),
    "down_gemm_resid": ("tc_gemm_kernel (down + residual)", "down"),
}

SPEC_BF16_TFLOPS = 2250.0
SPEC_HBM_GBS = 8000.0


def measure(args, wl, dev, world, rank, cpu_seconds):
    """Times wl.steps graph replays of one forward of workload wl on this rank; returns the
    record of one bench line (without the job-level keys)."""
    import torch
    import torch.distributed as dist

    from llama_family_decoder_gb300 import DecoderBlock
    from llama_family_decoder_gb300.synth import make_input, make_kv_cache, make_weights

    local = dev.index
    w_cpu = make_weights(wl, seed=rank_seed(wl, rank))
    x_cpu = make_input(wl, seed=rank_seed(wl, rank))
    w = {k: v.to(dev) for k, v in w_cpu.items()}
    x = x_cpu.to(dev)
    cached = wl.cache_len > 0  # T new tokens after cache_len positions: a decode step (T == 1) or a chunk
    decode = cached and wl.seq == 1
    cache = None
    cache_cpu = None
    if cached:
        cache_cpu = make_kv_cache(wl)
        kc, vc = (t.to(dev) for t in cache_cpu)
        lens0 = torch.full((wl.batch,), wl.cache_len, dtype=torch.int32, device=dev)
        cache = {"k": kc, "v": vc, "lens": lens0.clone()}
    blk = DecoderBlock.from_workload(wl)
    if wl.dtype == "bf16":
        w = blk.prepare(w)  # one-time load step: fp16 copies of the weights the GEMMs read
    out = torch.empty_like(x)
    ws = torch.empty(blk.workspace_bytes(wl.batch, wl.seq, cached), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # Write a buffer larger than L2, then read it: the read evicts the
        # write's dirty lines, so their write-back happens here and not inside
        # the next timed step. L2 is left holding clean lines of this buffer.
        flush.zero_()
        flush.amax()
    stream = torch.cuda.current_stream(dev)

    def step():
        if cached:
            cache["lens"].copy_(lens0)  # every step processes the same positions
        blk.forward(x, w, cache=cache, out=out, workspace=ws, stream=stream,
                    host_lens_max=wl.cache_len if cached else -1)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if args.ncu:  # one more forward for a profiler to capture, nothing timed
        step()
        torch.cuda.synchronize()
        blk.close()
        return None

    # Every timed step replays one CUDA graph of the whole forward (captured once).
    # The headline times a graph without profiling events; a second graph, with
    # the per-stage events recorded inside it, is replayed for the stage times.
    hl = wl.cache_len if cached else -1
    graph = blk.forward_graph(x, w, out, ws, cache=cache, host_lens_max=hl)
    blk.profile(True)
    pgraph = blk.forward_graph(x, w, out, ws, cache=cache, host_lens_max=hl)
    for g in (graph, pgraph, graph, pgraph):
        if cached:
            cache["lens"].copy_(lens0)
        g.launch(stream)
    torch.cuda.synchronize()
    blk.profile_collect()
    blk.profile_reset()

    def timed(g, collect):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2()
            if cached:
                cache["lens"].copy_(lens0)
            starts[i].record(stream)
            g.launch(stream)
            ends[i].record(stream)
            if collect:
                blk.profile_collect()  # waits for this step; adds its per-stage event times
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local if world > 1 else 0]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_index) as clk:
        clk.wait_first_sample()
        step_ms = timed(graph, False)
        prof_ms = timed(pgraph, True)
    if world > 1:
        dist.barrier()
    stages = blk.profile_collect()
    pgraph.close()
    blk.profile(False)  # the profiled graph recorded these events: drop them after it
    total_ms = max_over_ranks(sum(step_ms), dev)
    ms_per_step = total_ms / args.steps
    tokens = wl.batch * wl.seq
    value = job_tokens_per_s(world, tokens, args.steps, total_ms)

    # ---- end to end with host buffers: the input copied from pinned host memory and the
    # output read back inside every timed step
    x_host = x_cpu.pin_memory()
    out_host = torch.empty_like(x_cpu).pin_memory()
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush_l2()
        if cached:
            cache["lens"].copy_(lens0)
        e_starts[i].record(stream)
        x.copy_(x_host, non_blocking=True)
        graph.launch(stream)
        out_host.copy_(out, non_blocking=True)
        e_ends[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(e_starts, e_ends)) / args.steps, dev)
    nbytes = x_cpu.numel() * x_cpu.element_size()

    # ---- end to end, pipelined as a serving loop runs it: two input/output buffer pairs,
    # each with its forward graph; step i's input is uploaded from pinned host memory on one
    # copy stream while step i - 1 computes, and its output read back to pinned host memory
    # on another while step i + 1 computes. Every step still moves its own input and output;
    # the timed region runs from the first upload to the last read-back. No L2 flush inside
    # it: each configuration's weights and activations exceed L2.
    x2, out2 = torch.empty_like(x), torch.empty_like(out)
    graph2 = blk.forward_graph(x2, w, out2, ws, cache=cache, host_lens_max=hl)
    xs, outs, graphs = (x, x2), (out, out2), (graph, graph2)
    host_in = (x_host, x_cpu.clone().pin_memory())
    host_out = (out_host, torch.empty_like(x_cpu).pin_memory())
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    up_done = [torch.cuda.Event() for _ in range(args.steps)]
    fw_done = [torch.cuda.Event() for _ in range(args.steps)]
    rd_done = [torch.cuda.Event() for _ in range(args.steps)]
    t_first, t_last = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_first.record(h2d_s)
    for i in range(args.steps):
        bsel = i % 2
        if i >= 2:
            h2d_s.wait_event(fw_done[i - 2])  # the forward two steps back has read this input buffer
        with torch.cuda.stream(h2d_s):
            xs[bsel].copy_(host_in[bsel], non_blocking=True)
        up_done[i].record(h2d_s)
        stream.wait_event(up_done[i])
        if i >= 2:
            stream.wait_event(rd_done[i - 2])  # this output buffer has been read back
        if cached:
            cache["lens"].copy_(lens0)
        graphs[bsel].launch(stream)
        fw_done[i].record(stream)
        d2h_s.wait_event(fw_done[i])
        with torch.cuda.stream(d2h_s):
            host_out[bsel].copy_(outs[bsel], non_blocking=True)
        rd_done[i].record(d2h_s)
    t_last.record(d2h_s)
    torch.cuda.synchronize()
    graph.close()
    graph2.close()
    e2e_pipe_ms = max_over_ranks(t_first.elapsed_time(t_last) / args.steps, dev)

    # ---- roofline of the dominant kernel (its live event times, on the forward's stream).
    # Every kernel here runs for well under a second inside a sub-second step, so a
    # tensor-bound kernel is held to the burst bf16 peak (the fp16 kind runs at the same rate).
    peaks = _peaks()
    g, weight_bytes, kv_bytes = work_counts(wl)
    launches = sum(n for _, n in stages.values())
    stage_ms = {k: v[0] / args.steps for k, v in stages.items()}
    if decode:
        name = "attention_splitkv"
        ms = stage_ms[name]
        es = 2 if wl.dtype == "bf16" else 4
        algo = kv_bytes + wl.batch * wl.num_heads * wl.head_dim * es * 2
        achieved = algo / (ms / 1e3) / 1e9
        kname = "attn_decode_kernel (split-KV)"
        roof = {"bound": "hbm", "kernel": kname, "stage": name, "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "frac_of_spec_8000": achieved / SPEC_HBM_GBS, "traffic": _traffic(kname, wl.name),
                "algorithmic_bytes": algo, "stage_us": ms * 1e3,
                "peak_source": f"{peaks['source']} copy bandwidth"}
    else:
        name = max((s for s in PREFILL_STAGES if s in stage_ms), key=lambda s: stage_ms[s])
        kname, key = PREFILL_STAGES[name]
        ms = stage_ms[name]
        achieved = g[key] / (ms / 1e3) / 1e12
        pk = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "kernel": kname, "stage": name, "achieved": achieved,
                "peak": pk, "unit": "TFLOP/s", "frac": achieved / pk,
                "frac_of_spec_2250": achieved / SPEC_BF16_TFLOPS, "traffic": _traffic(kname, wl.name),
                "algorithmic_flops": g[key], "stage_us": ms * 1e3,
                "peak_source": f"{peaks['source']} burst bf16 (sustained {peaks['bf16_tflops_sustained']})"}
    total_flops = sum(g.values())
    step_s = ms_per_step / 1e3
    block = {"tflops": total_flops / step_s / 1e12,
             "frac_of_bf16_burst": total_flops / step_s / 1e12 / peaks["bf16_tflops"],
             "frac_of_bf16_spec_2250": total_flops / step_s / 1e12 / SPEC_BF16_TFLOPS,
             "hbm_gbs_weights_plus_kv": (weight_bytes + kv_bytes) / step_s / 1e9}
    if decode:
        step_bytes = weight_bytes + kv_bytes + 2.0 * wl.batch * wl.hidden_size * 2
        block.update({"step_us": ms_per_step * 1e3, "step_bytes": step_bytes,
                      "frac_of_hbm_measured": step_bytes / step_s / 1e9 / peaks["hbm_gbs"],
                      "frac_of_hbm_spec_8000": step_bytes / step_s / 1e9 / SPEC_HBM_GBS,
                      "target_us_at_70pct_of_8000": step_bytes / (0.7 * SPEC_HBM_GBS * 1e9) * 1e6})
    stage_roof = {}
    for s, (kn, key) in PREFILL_STAGES.items():
        if s in stage_ms and not decode:
            a = g[key] / (stage_ms[s] / 1e3) / 1e12
            stage_roof[s] = {"us": stage_ms[s] * 1e3, "tflops": a, "frac_of_bf16_burst": a / peaks["bf16_tflops"]}

    rec = {"value": value, "unit": "tokens/s", "ms_per_step": ms_per_step, "dtype": wl.dtype,
           "config": config_of(wl, world), "roofline": roof,
           "e2e": {"value": job_tokens_per_s(world, tokens, 1, e2e_pipe_ms), "unit": "tokens/s",
                   "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "ms_per_step": e2e_pipe_ms,
                   "mode": "pipelined: two buffer pairs, the next input's upload and the previous output's "
                           "read-back on their own streams beside each forward"},
           "e2e_serial": {"value": job_tokens_per_s(world, tokens, 1, e2e_ms), "unit": "tokens/s",
                          "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "ms_per_step": e2e_ms,
                          "mode": "each step: upload, forward, read-back in turn on one stream"},
           "gpu_launches": launches, "clocks": clk.summary(), "stages_ms": stage_ms,
           "stage_roofline": stage_roof,
           "ms_per_step_with_stage_events": sum(prof_ms) / args.steps, "block": block}
    blk.close()
    del w, x, out, ws, flush, cache
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and cpu_seconds > 0:
        rec["cpu_baseline"] = cpu_baseline(wl, w_cpu, x_cpu, cache_cpu, cpu_seconds)
    return rec


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    from llama_family_decoder_gb300.synth import WORKLOADS

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    __graft_entry__.build()

    cpu_s = 0.0 if args.no_cpu_baseline else 10.0
    head = measure(args, wl, dev, world, rank, cpu_s)
    if head is None:  # --ncu: nothing timed
        if world > 1:
            dist.destroy_process_group()
        return
    line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) input)"}
    line.update({k: v for k, v in head.items() if k not in line and k != "unit"})
    subs = [] if (args.workload != DEFAULT_WORKLOAD or args.no_sub_configs) else SUB_CONFIGS
    if subs:
        line["configs"] = {}
        for name in subs:  # the other configurations, timed the same way in this process
            line["configs"][name] = measure(args, WORKLOADS[name], dev, world, rank, 0.0 if cpu_s == 0 else 2.0)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_model(args, wl):
    """The model around the block: embedding, wl.n_layers blocks, final norm, lm_head, one
    blk_model_forward per step, replayed from a CUDA graph. Weights are drawn on the device
    (N(0, 0.02) projections, unit gains, N(0, 1) embeddings): at 32 layers they are ~13 GB."""
    import torch

    from llama_family_decoder_gb300 import DecoderBlock
    from llama_family_decoder_gb300.synth import make_input, make_weights

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import __graft_entry__
    __graft_entry__.build()

    D, H, Hkv, d, F, V = wl.hidden_size, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.intermediate_size, wl.vocab
    gen = torch.Generator(device=dev).manual_seed(rank_seed(wl, rank))
    bf = torch.bfloat16

    def rnd(*shape, std=0.02):
        return (torch.randn(*shape, generator=gen, device=dev) * std).to(bf)

    blk = DecoderBlock.from_workload(wl)
    layers = []
    for _ in range(wl.n_layers):
        w = {"input_layernorm": torch.ones(D, dtype=bf, device=dev), "q_proj": rnd(H * d, D),
             "k_proj": rnd(Hkv * d, D), "v_proj": rnd(Hkv * d, D), "o_proj": rnd(D, H * d),
             "post_attention_layernorm": torch.ones(D, dtype=bf, device=dev), "up_proj": rnd(F, D),
             "down_proj": rnd(D, F)}
        if wl.hidden_act == "silu":
            w["gate_proj"] = rnd(F, D)
        layers.append(blk.prepare(w))  # the one-time load step of each layer
    embed, lm_head = rnd(V, D, std=1.0), rnd(V, D)
    norm_g = torch.ones(D, dtype=bf, device=dev)
    tokens = torch.randint(0, V, (wl.batch, wl.seq), generator=gen, device=dev, dtype=torch.int32)
    logits = torch.empty(wl.batch, wl.seq, V, dtype=bf, device=dev)
    ws = torch.empty(blk.model_workspace_bytes(wl.batch, wl.seq), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        flush.amax()

    def fwd():
        blk.model_forward(tokens, layers, embed, norm_g, lm_head, logits=logits, workspace=ws)

    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize()
    if args.ncu:
        fwd()
        torch.cuda.synchronize()
        return
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fwd()  # one more warm-up on the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            fwd()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local if world > 1 else 0]
    with ClockSampler(gpu_index) as clk:
        clk.wait_first_sample()
        for i in range(args.steps):
            flush_l2()
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
        torch.cuda.synchronize()
    total_ms = max_over_ranks(sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)), dev)
    ms_per_step = total_ms / args.steps
    ntok = wl.batch * wl.seq
    value = job_tokens_per_s(world, ntok, args.steps, total_ms)
    # end to end: token ids from pinned host memory, the last position's logits back (the next-token scores)
    tok_host = tokens.cpu().pin_memory()
    last_host = torch.empty(wl.batch, V, dtype=bf).pin_memory()
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush_l2()
        e_s[i].record(stream)
        tokens.copy_(tok_host, non_blocking=True)
        graph.replay()
        last_host.copy_(logits[:, -1], non_blocking=True)
        e_e[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(s_.elapsed_time(e_) for s_, e_ in zip(e_s, e_e)) / args.steps, dev)
    peaks = _peaks()
    g, weight_bytes, _ = work_counts(wl)
    flops = sum(g.values())
    achieved = flops / (ms_per_step / 1e3) / 1e12
    pk = peaks["bf16_tflops_sustained"]
    roof = {"bound": "tensor", "kernel": "whole model step (every launch of the forward)", "achieved": achieved,
            "peak": pk, "unit": "TFLOP/s", "frac": achieved / pk, "traffic": None, "algorithmic_flops": flops,
            "peak_source": f"{peaks['source']} sustained bf16 (burst {peaks['bf16_tflops']})"}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (N(0,0.02) projections drawn on the device, N(0,1) embeddings, random token ids)",
            "config": dict(config_of(wl, world), n_layers=wl.n_layers, vocab=V), "roofline": roof,
            "e2e": {"value": job_tokens_per_s(world, ntok, 1, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": tok_host.numel() * 4, "d2h_bytes_per_step": last_host.numel() * 2},
            "gpu_launches": 1 + 6 * wl.n_layers + 2, "clocks": clk.summary(),
            "block": {"tflops": achieved, "frac_of_bf16_spec_2250": achieved / 2250.0,
                      "weight_bytes": weight_bytes}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, sample, dt = oracle_tokens_per_s(wl, make_weights(wl), make_input(wl), None, 64)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": sample, "seconds": dt}
    if rank == 0:
        print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-configs", action="store_true", help="time the headline workload only")
    ap.add_argument("--ncu", action="store_true", help="warm up, run one more forward for a profiler, exit")
    args = ap.parse_args()
    from llama_family_decoder_gb300.synth import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    elif wl.n_layers:
        run_model(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
