#!/usr/bin/env python3
"""ResidualAttention decode throughput on GB300 (tokens/s and achieved HBM GB/s).

Headline workload: the Llama-3-70B-shaped two-level fork tree (64 q / 8 kv
heads, head_dim 128, rank 16; 64 agents under a 131072-token root, 4 trunks of
8192 tokens, 16 agents per trunk with U[1,4096] private tokens; 1 query per
agent), the largest decode workload, seeded and synthetic.  Each pool set
(layer) holds 1.8 GB, so two sets already keep every call's inputs out of the
129 MB L2.

One step = one decode step over every timed layer: per layer, the new token's
rows are scattered into the pools (forkkv_write_rows) and ResidualAttention
decode runs (forkkv_residual_attn_decode: split-KV kernel + combine kernel).
The writes of a step and the decodes of a step are each captured in a CUDA
graph; the timed region replays them K times, with CUDA events around each
step's decodes (the roofline's launch time).  tokens/s counts one (agent,
layer) attention as one token, i.e. A * layers / step time.  The same step
through the library's one-graph call (forkkv_step_graph_launch, every layer's
write and decode in one CUDA graph) is timed too ("step_graph"), and the e2e
figure runs through it with host copies in and out.

The same line carries "per_config" (the Llama-3-8B-shaped and Qwen2.5-7B-shaped
decode fan-outs, each with its own roofline) and "prefill" (the Qwen2.5-14B-
shaped chunked prefill against the dense bf16 tensor peak), timed in the same
run.  --config picks another headline workload; --fill times the residual fill.

--impl reference times the fp64 CPU oracle instead (the only reference this
method has), on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ResidualAttention decode tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# kernels launched per layer and step: the row write, the split-KV kernel, the combine kernel
GPU_LAUNCHES_PER_LAYER = 3


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def percentiles(xs, qs=(10, 50, 90)):
    """Nearest-rank percentiles of a list of timings ({"p10": ..., "p50": ..., "p90": ...})."""
    v = sorted(xs)
    out = {}
    for q in qs:
        k = max(0, min(len(v) - 1, math.ceil(q / 100 * len(v)) - 1))
        out[f"p{q}"] = v[k]
    return out


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks of the initialised process group (x itself on one
    rank): the job's time is that of its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, agents: int, layers: int, seconds_per_step: float) -> float:
    """Whole-job throughput of `world` independent replicas (weak scaling): every replica
    attends `agents` x `layers` (agent, layer) tokens per step, and a step of the job lasts as
    long as its slowest replica's (seconds_per_step, already the maximum over ranks)."""
    return world * agents * layers / seconds_per_step


def _traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu capture (scaled to a full
    launch where the capture was of a smaller case), if the kernel source is unchanged since."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)[kernel][workload]
        sources = d.get("sources") or [d["source"]]
        h = hashlib.sha256()
        for src in sources:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        return d["dram_bytes_per_launch"] if h.hexdigest() == d.get("sources_sha256", d.get("source_sha256")) else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.idx = device_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_figures(w, layers: int):
    """Algorithmic bytes and flops of one decode call (one layer), from the drawn lengths."""
    cfg = w.cfg
    A, Hq, Hkv, D, r, G = cfg.n_agents, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rank, cfg.group
    unique_rows = sum(w.node_tokens)            # every base row once, shared prefix included once
    lens = [int(x) for x in w.seq_lens]
    base = unique_rows * Hkv * D * 2 * 2         # K and V, bf16
    res = sum(lens) * 2 * r * 2                  # k_res and v_res, bf16
    qo = 2 * A * Hq * D * 2                      # q in, out
    adapters = A * 2 * r * Hkv * D * 2           # B_k, B_v
    tables = sum(2 * math.ceil(L / 16) * 4 for L in lens) + A * 8
    flops = sum(lens) * Hkv * (2 * D * (r + 2 * G) + 2 * G * r)
    return {"bytes": base + res + qo + adapters + tables, "base_bytes": base, "res_bytes": res, "flops": flops}


def run_oracle_sample(w, agent: int, kv_head: int):
    from oracle import residual_attention as ra
    import torch
    kb, vb = w.agent_base(agent)
    f = lambda t: t.to(torch.float64).numpy()
    G = w.cfg.group
    heads = list(range(kv_head * G, (kv_head + 1) * G))
    ra.residual_attention(f(w.q[agent]), w.positions[agent].numpy(), f(kb), f(vb), f(w.k_res[agent]),
                          f(w.v_res[agent]), f(w.B_k[agent]), f(w.B_v[agent]), w.cfg.rope_theta, q_heads=heads)
    return len(heads) / w.cfg.n_q_heads  # fraction of one (agent, layer) token


def cpu_baseline(w, seconds: float = 12.0) -> dict:
    """The oracle, as it stands, on a bounded sample: (agent, KV head) units of one layer call."""
    t0 = time.perf_counter()
    tokens, units = 0.0, 0
    while time.perf_counter() - t0 < seconds:
        a = units % w.cfg.n_agents
        h = (units // w.cfg.n_agents) % w.cfg.n_kv_heads
        tokens += run_oracle_sample(w, a, h)
        units += 1
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{units} (agent, KV head) units of one layer call ({w.cfg.group} query heads each, "
                      f"fp64 NumPy, default BLAS threading) in {dt:.1f} s; one unit = "
                      f"{1 / w.cfg.n_kv_heads:.3f} of an (agent, layer) token",
            "machine": platform.machine()}


def prefill_flops(w) -> int:
    """Algorithmic flops of one prefill-chunk call: per (query row, visible key) the score, value and
    residual-value products; per (key, head) the up-projection; per query row the B_v epilogue."""
    cfg = w.cfg
    D, r, G, Hkv = cfg.head_dim, cfg.rank, cfg.group, cfg.n_kv_heads
    total = 0
    for a in range(cfg.n_agents):
        L = int(w.seq_lens[a])
        vis = sum(min(int(p) + 1, L) for p in w.positions[a].tolist())
        total += Hkv * (G * vis * (2 * D + 2 * D + 2 * r) + L * 2 * r * D + cfg.q_len * G * 2 * r * D)
    return total


def bench_prefill(args, cfg) -> dict:
    """Prefill-chunk throughput (TFLOP/s against the dense bf16 tensor peak), one layer per call;
    returns the JSON line as a dict."""
    import torch
    from disaggregated_kv_attention_gb300 import build as _build
    from disaggregated_kv_attention_gb300 import forkkv as fk
    from disaggregated_kv_attention_gb300 import paged
    from disaggregated_kv_attention_gb300 import workload as wl
    _build.build()
    w = wl.generate(cfg)
    dev = torch.device("cuda", 0)
    P = paged.place(w, device=dev)
    rope = fk.rope_table(cfg.rope_theta, P.max_seq_len, device=dev)
    out = torch.empty_like(P.q)
    p, keep = paged.params(P, out, rope=rope, prefill=True)
    fk.forkkv_residual_attn_prefill_chunk(p)
    torch.cuda.synchronize()
    if fk.forkkv_get_device_status():
        raise RuntimeError("device status set by the prefill kernel")
    for _ in range(args.warmup):
        fk.forkkv_residual_attn_prefill_chunk(p)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    time.sleep(0.3)
    for k in range(args.steps):
        ev[2 * k].record(stream)
        fk.forkkv_residual_attn_prefill_chunk(p)
        ev[2 * k + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if fk.forkkv_get_device_status():
        raise RuntimeError("device status set by the prefill kernel")
    ms = [ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(args.steps)]
    t = statistics.median(ms) / 1000
    flops = prefill_flops(w)
    hbm, tf, tf_sus, src = _peaks()
    achieved = flops / t / 1e12
    tokens = cfg.n_agents * cfg.q_len
    return {
        "metric": "ResidualAttention prefill-chunk TFLOP/s (% of dense bf16 tensor peak), 1 GPU",
        "value": achieved, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * t, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": f"{cfg.name}: {cfg.description}", "layers": 1,
                                        "l2": "inputs larger than L2 (q and out alone are 336 MB)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tf, "unit": "TFLOP/s", "frac": achieved / tf,
                     "traffic": _traffic("prefill_kernel", cfg.name),
                     "peak_source": f"{src} bf16_tflops burst (of {src})",
                     "alg_flops_per_launch": flops, "launch_ms_median": 1000 * t},
        "tokens_per_s": tokens / t, "gpu_launches": args.steps, "clocks": clk}


def bench_fill(args, cfg) -> int:
    """Residual fill of a fan-out: every agent's xA rows of every shared-prefix token, one call
    (forkkv_residual_fill), for the decode configuration's agents and prefix (hidden size of the
    model named by the configuration).  Four copies of x are cycled so the inputs exceed L2."""
    import torch
    from disaggregated_kv_attention_gb300 import build as _build
    from disaggregated_kv_attention_gb300 import forkkv as fk
    _build.build()
    n_ag = cfg.n_agents
    n_tok = cfg.nodes[0].tokens[0]  # the root's (shared prefix's) tokens
    hidden = cfg.hidden
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(1000 + cfg.index)
    reps = 4
    xs = [torch.randn(n_tok, hidden, generator=g).to(torch.bfloat16).to(dev) for _ in range(reps)]
    A = (0.02 * torch.randn(n_ag, 2, 16, hidden, generator=g)).to(torch.bfloat16).to(dev)
    n_res = n_ag * ((n_tok + 15) // 16)
    pools = fk.Pools(8, n_res, cfg.n_kv_heads, n_layers=1, device=dev, fill=0)
    t = torch.arange(n_tok)
    slots = torch.stack([((t // 16) * n_ag + a) * 16 + t % 16 for a in range(n_ag)]).to(torch.int32).to(dev)
    fk.forkkv_residual_fill(pools, 0, xs[0], A, slots)
    torch.cuda.synchronize()
    if fk.forkkv_get_device_status():
        raise RuntimeError("device status set by the residual fill")
    for k in range(args.warmup):
        fk.forkkv_residual_fill(pools, 0, xs[k % reps], A, slots)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    time.sleep(0.3)
    for k in range(args.steps):
        ev[2 * k].record(stream)
        fk.forkkv_residual_fill(pools, 0, xs[k % reps], A, slots)
        ev[2 * k + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    us = [1000 * ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(args.steps)]
    t_us = statistics.mean(us)
    alg_bytes = n_tok * hidden * 2 + A.numel() * 2 + n_ag * n_tok * 2 * 16 * 2 + slots.numel() * 4
    flops = 2 * n_tok * hidden * 32 * n_ag
    hbm, tf, tf_sus, src = _peaks()
    gbs = alg_bytes / (t_us * 1e-6) / 1e9
    tfs = flops / (t_us * 1e-6) / 1e12
    hbm_bound = alg_bytes / (hbm * 1e9) >= flops / (tf * 1e12)
    print(json.dumps({
        "metric": "Residual fill GB/s (% of HBM peak), 1 GPU", "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_us / 1000, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name} fan-out fill: {n_ag} agents x {n_tok} prefix tokens, hidden {hidden}, "
                               f"rank 16 (k and v), x cycled over {reps} copies (inputs > L2)"},
        "roofline": {"bound": "hbm" if hbm_bound else "tensor", "achieved": gbs if hbm_bound else tfs,
                     "peak": hbm if hbm_bound else tf, "unit": "GB/s" if hbm_bound else "TFLOP/s",
                     "frac": (gbs / hbm) if hbm_bound else (tfs / tf), "traffic": _traffic("residual_fill_kernel", cfg.name),
                     "peak_source": f"{src} ({'hbm_gbs' if hbm_bound else 'bf16_tflops burst'})",
                     "alg_bytes_per_launch": alg_bytes, "alg_flops_per_launch": flops},
        "achieved_tflops": tfs, "tensor_frac": tfs / tf, "hbm_frac": gbs / hbm,
        "gpu_launches": args.steps, "clocks": clk}))
    return 0


# decode workloads reported beside the headline, and the prefill-chunk workload
PER_CONFIG = ("llama3_8b_decode", "qwen25_7b_mapreduce_decode")
PREFILL_CONFIG = "qwen25_14b_prefill"
L2_BYTES = 129e6


def pool_sets(cfg, fig, requested: int) -> int:
    """Pool sets (layers) timed: `requested`, else enough that the sets together hold at least four
    times the L2 (so a call never finds its inputs there), at least two, at most the model's layers."""
    if requested:
        return requested
    return int(min(cfg.model_layers, max(2, math.ceil(4 * L2_BYTES / fig["bytes"]))))


def decode_run(cfg, w, layers, steps, warmup, dev, world, full):
    """Time `steps` decode steps over `layers` pool sets of workload w (one step = every layer's row write
    and decode, each captured in a CUDA graph); with `full`, also the one-graph step API and the e2e leg."""
    import torch
    from disaggregated_kv_attention_gb300 import forkkv as fk
    from disaggregated_kv_attention_gb300 import paged

    fig = workload_figures(w, layers)
    P = paged.place(w, device=dev, n_layers=layers)
    A, Hkv = cfg.n_agents, cfg.n_kv_heads
    lens = [int(x) for x in w.seq_lens]
    rope = fk.rope_table(cfg.rope_theta, P.max_seq_len, device=dev)
    plan, info = fk.forkkv_plan_build(P.bpt_np, w.seq_lens.numpy(), Hkv)
    plan_d = torch.from_numpy(plan).to(dev)

    # per-layer step inputs: q, and the new token's rows (the workload's own last rows)
    q_all = P.q.unsqueeze(0).repeat(layers, 1, 1, 1, 1).contiguous()
    out_all = torch.empty_like(q_all)
    kb_last = torch.stack([w.agent_base(a)[0][lens[a] - 1] for a in range(A)])
    vb_last = torch.stack([w.agent_base(a)[1][lens[a] - 1] for a in range(A)])
    kr_last = torch.stack([w.k_res[a][lens[a] - 1] for a in range(A)])
    vr_last = torch.stack([w.v_res[a][lens[a] - 1] for a in range(A)])
    kb_new = kb_last.unsqueeze(0).repeat(layers, 1, 1, 1).to(dev).contiguous()
    vb_new = vb_last.unsqueeze(0).repeat(layers, 1, 1, 1).to(dev).contiguous()
    kr_new = kr_last.unsqueeze(0).repeat(layers, 1, 1).to(dev).contiguous()
    vr_new = vr_last.unsqueeze(0).repeat(layers, 1, 1).to(dev).contiguous()
    slot_b = torch.tensor([int(P.bpt_np[a, (lens[a] - 1) // 16]) * 16 + (lens[a] - 1) % 16 for a in range(A)],
                          dtype=torch.int32, device=dev)
    slot_r = torch.tensor([int(P.rpt_np[a, (lens[a] - 1) // 16]) * 16 + (lens[a] - 1) % 16 for a in range(A)],
                          dtype=torch.int32, device=dev)

    params = []
    for l in range(layers):
        p = fk.attn_params(P.pools, l, q_all[l], out_all[l], P.bpt, P.rpt, P.seq_lens, P.positions, P.max_seq_len,
                           P.B_k, P.B_v, rope=rope, plan=plan_d, plan_info=info)
        params.append(p)
    ws = fk.workspace_for(params[0], device=dev)
    for p in params:
        fk.set_workspace(p, ws)

    def writes():
        for l in range(layers):
            fk.forkkv_write_rows(P.pools, l, slot_b, slot_r, kb_new[l], vb_new[l], kr_new[l], vr_new[l])

    def decodes():
        for p in params:
            fk.forkkv_residual_attn_decode(p)

    # eager once (sets kernel attributes), check status, then capture
    writes()
    decodes()
    torch.cuda.synchronize()
    st = fk.forkkv_get_device_status()
    if st:
        raise RuntimeError(f"device status {st} after the first step")
    g_w, g_d = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g_w, stream=s):
            writes()
        with torch.cuda.graph(g_d, stream=s):
            decodes()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        g_w.replay()
        g_d.replay()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    time.sleep(0.3)
    e_start.record(stream)
    for k in range(steps):
        g_w.replay()
        ev0[k].record(stream)
        g_d.replay()
        ev1[k].record(stream)
    e_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(e_start.elapsed_time(e_end), dev)
    dec_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    call_us = 1000 * statistics.mean(dec_ms) / layers
    call_pct = {k: 1000 * v / layers for k, v in percentiles(dec_ms).items()}
    ms_step = total_ms / steps
    hbm, tf, tf_sus, src = _peaks()
    achieved = fig["bytes"] / (call_us * 1e-6) / 1e9
    res = {
        "fig": fig, "layers": layers, "ms_per_step": ms_step, "call_us": call_us, "call_pct": call_pct,
        "value": job_tokens_per_s(world, A, layers, ms_step / 1000), "clocks": clk,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": _traffic("decode_split_kernel", cfg.name),
                     "peak_source": f"{src} hbm_gbs (of {src})",
                     "kernel": "forkkv_residual_attn_decode (split-KV kernel + combine kernel), per layer call",
                     "alg_bytes_per_launch": fig["bytes"], "launch_us": call_us},
        "achieved_tflops": fig["flops"] / (call_us * 1e-6) / 1e12,
        "tensor_frac": fig["flops"] / (call_us * 1e-6) / 1e12 / tf,
    }
    if not full:
        st = fk.forkkv_get_device_status()
        if st:
            raise RuntimeError(f"device status {st} after the timed region")
        return res

    # the same step through the public one-graph API (forkkv_step_graph_*: every layer's row
    # write and decode in one CUDA graph), device-timed over the same number of steps
    rows = [(slot_b, slot_r, kb_new[l], vb_new[l], kr_new[l], vr_new[l]) for l in range(layers)]
    sg = fk.forkkv_step_graph_create(params, rows)
    for _ in range(warmup):
        fk.forkkv_step_graph_launch(sg, stream)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(steps):
        fk.forkkv_step_graph_launch(sg, stream)
    g1.record(stream)
    torch.cuda.synchronize()
    sg_ms = g0.elapsed_time(g1) / steps

    # end to end through the public API: pinned host inputs in, the one-graph step, result out,
    # every step
    q_h = q_all.cpu().pin_memory()
    kbh, vbh = kb_new.cpu().pin_memory(), vb_new.cpu().pin_memory()
    krh, vrh = kr_new.cpu().pin_memory(), vr_new.cpu().pin_memory()
    bpt_h, rpt_h = P.bpt.cpu().pin_memory(), P.rpt.cpu().pin_memory()
    lens_h, pos_h = P.seq_lens.cpu().pin_memory(), P.positions.cpu().pin_memory()
    out_h = torch.empty_like(out_all, device="cpu").pin_memory()
    h2d = [(q_all, q_h), (kb_new, kbh), (vb_new, vbh), (kr_new, krh), (vr_new, vrh), (P.bpt, bpt_h),
           (P.rpt, rpt_h), (P.seq_lens, lens_h), (P.positions, pos_h)]
    h2d_bytes = sum(h.numel() * h.element_size() for _, h in h2d)
    d2h_bytes = out_h.numel() * out_h.element_size()
    e2e_steps = max(10, steps // 4)

    def e2e_step():
        for d, h in h2d:
            d.copy_(h, non_blocking=True)
        fk.forkkv_step_graph_launch(sg, stream)
        out_h.copy_(out_all, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, dev)
    torch.cuda.synchronize()
    fk.forkkv_step_graph_destroy(sg)
    st = fk.forkkv_get_device_status()
    if st:
        raise RuntimeError(f"device status {st} after the timed region")
    res["step_graph"] = {"ms_per_step": sg_ms, "tokens_per_s": world * A * layers / (sg_ms / 1000),
                         "api": "forkkv_step_graph_launch: one CUDA graph per step (every timed layer)"}
    res["e2e"] = {"value": job_tokens_per_s(world, A, layers, e2e_s), "unit": "tokens/s",
                  "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "steps": e2e_steps,
                  "api": "forkkv_step_graph_launch"}
    return res


def decode_config(cfg, w, layers):
    return {"workload": f"{cfg.name}: {cfg.description}", "layers": layers, "model_layers": cfg.model_layers,
            "agents": cfg.n_agents, "q_heads": cfg.n_q_heads, "kv_heads": cfg.n_kv_heads,
            "head_dim": cfg.head_dim, "rank": cfg.rank, "page": cfg.page_size,
            "seq_lens": [int(x) for x in w.seq_lens], "seed": cfg.seed}


def _free_device():
    import gc
    import torch
    gc.collect()
    torch.cuda.empty_cache()


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="forkkv", choices=["forkkv", "reference"])
    ap.add_argument("--config", default="llama3_70b_stress_decode")
    ap.add_argument("--layers", type=int, default=0, help="pool sets timed (0: enough to hold 4x the L2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline only: no per_config / prefill lines")
    ap.add_argument("--fill", action="store_true", help="time the residual fill of the configuration's fan-out")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from disaggregated_kv_attention_gb300 import workload as wl
    cfg = wl.CONFIGS[args.config]
    if args.fill:
        return bench_fill(args, cfg)
    if cfg.q_len != 1:
        print(json.dumps(bench_prefill(args, cfg)))
        return 0
    w = wl.generate(cfg)
    layers = pool_sets(cfg, workload_figures(w, 1), args.layers)
    fig = workload_figures(w, layers)
    config = decode_config(cfg, w, layers)
    config["l2"] = "inputs larger than L2: %d pool sets (layers), %.2f GB in total" % (
        layers, layers * fig["bytes"] / 1e9)

    if args.impl == "reference":
        if rank != 0:
            return 0
        samples = []
        for k in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            frac = run_oracle_sample(w, k % cfg.n_agents, (k // cfg.n_agents) % cfg.n_kv_heads)
            dt = time.perf_counter() - t0
            if k >= args.warmup:
                samples.append((frac, dt))
            if k >= args.warmup and sum(d for _, d in samples) > 120:
                break  # bounded: the whole run stays within a few minutes
        tok = sum(f for f, _ in samples)
        sec = sum(d for _, d in samples)
        value = tok / sec
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": len(samples), "warmup": args.warmup, "ms_per_step": 1000 * sec / len(samples),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                                 "kind": "oracle",
                                 "sample": f"each step: one (agent, KV head) unit of one layer call "
                                           f"({cfg.group} query heads, fp64 NumPy), rotating over agents and "
                                           f"heads; {len(samples)} steps timed (capped at 120 s of CPU work)"},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from disaggregated_kv_attention_gb300 import build as _build
    _build.build()
    dev = torch.device("cuda", local)

    r = decode_run(cfg, w, layers, args.steps, args.warmup, dev, world, full=True)
    A = cfg.n_agents
    line = {
        "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
        "roofline": r["roofline"],
        "decode_call_us": r["call_us"],
        "decode_call_us_percentiles": r["call_pct"],
        "model_step_tokens_per_s": world * A / (cfg.model_layers * r["call_us"] * 1e-6),
        "model_step_note": f"agents / ({cfg.model_layers} layers x the mean layer-call time)",
        "step_graph": r["step_graph"],
        "achieved_tflops": r["achieved_tflops"], "tensor_frac": r["tensor_frac"],
        "alg_flops_per_call": fig["flops"],
        "e2e": r["e2e"],
        "gpu_launches": args.steps * layers * GPU_LAUNCHES_PER_LAYER,
        "clocks": r["clocks"],
    }
    del r
    _free_device()
    if world == 1 and not args.no_extra:
        # the other decode workloads and the prefill chunk, timed in the same run
        per = {}
        for name in PER_CONFIG:
            c = wl.CONFIGS[name]
            wc = wl.generate(c)
            lc = pool_sets(c, workload_figures(wc, 1), 0)
            rc = decode_run(c, wc, lc, min(args.steps, 200), args.warmup, dev, world, full=False)
            per[name] = {"config": decode_config(c, wc, lc), "decode_call_us": rc["call_us"],
                         "decode_call_us_percentiles": rc["call_pct"], "tokens_per_s": rc["value"],
                         "roofline": rc["roofline"], "achieved_tflops": rc["achieved_tflops"],
                         "tensor_frac": rc["tensor_frac"], "clocks": rc["clocks"]}
            del wc, rc
            _free_device()
        line["per_config"] = per
        pf = bench_prefill(argparse.Namespace(steps=min(args.steps, 20), warmup=args.warmup),
                           wl.CONFIGS[PREFILL_CONFIG])
        line["prefill"] = {k: pf[k] for k in ("value", "unit", "ms_per_step", "config", "roofline",
                                              "tokens_per_s", "clocks", "steps")}
        _free_device()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
