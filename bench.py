"""Verify-step benchmark: one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c1] [--impl reference]

A step is one pass of the whole hot path on one synthetic batch: gated NoPE
MLA verify attention (with its split-KV LSE merge) followed by the greedy
verify (argmax, accepted prefix, trimmed kv_lens).  The default workload is
the C=1 verify batch (1 request, k=7, 64 heads, context 1536, 163840-token
vocabulary).  Inputs sit in HBM before timing; L2 (129 MB) is flushed before
every timed step, outside the timed events, by writing a 512 MB buffer and
then reading a 256 MB one (so the flush's own dirty lines are written back
before the step starts).

--impl reference times the float64 CPU oracle on the same workload (host
cores).  Under torchrun (N > 1) every rank runs an independent replica (the
verify step has no exchange between requests); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-step µs & attention TFLOP/s (frac of peak); greedy-verify GB/s, 1×GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="c1")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(times_ms, device, world):
    """Mean of this rank's per-step times, then the maximum over all ranks
    (all_reduce MAX over the default process group when world > 1)."""
    m = statistics.mean(times_ms)
    if world > 1:
        import torch
        t = torch.tensor([m], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        m = float(t.item())
    return m


def replica_throughput(step_ms, world):
    """Steps per second of the whole job: every rank runs its own replica."""
    return world * 1000.0 / step_ms


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_figures(inp):
    """Algorithmic work of one step (counted on visible rows only)."""
    H = inp["H"]
    sum_b = int(inp["kv_bounds"].astype("int64").sum())
    attn_flops = 4.0 * 512 * H * sum_b
    k1 = inp["k"] + 1
    kv_rows = 0
    for r in range(inp["R"]):
        kv_rows += int(inp["kv_bounds"][r * k1:(r + 1) * k1].max())
    T = inp["T"]
    attn_bytes = 1024.0 * kv_rows + T * H * (3 * 1024 + 4)
    logits_bytes = 4.0 * T * inp["cfg"].vocab
    return attn_flops, attn_bytes, logits_bytes


# the sources that compile into the attention kernel whose DRAM traffic the
# committed ncu summary records
ATTENTION_SOURCES = ("mla_verify_decode.cu", "sv_ptx.cuh")


def kernel_source_hash():
    """Hash of the attention kernel's code: comments and whitespace are
    dropped first, so that a comment edit keeps recorded counters valid."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verify_mla_gb300", "csrc")
    for fn in ATTENTION_SOURCES:
        with open(os.path.join(csrc, fn)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(fn.encode() + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(config_name):
    """DRAM bytes per attention launch from a committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(config_name)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
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
        os.unlink(self.path)
        if not sm:
            return None
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(config_name: str, min_seconds: float = 10.0, max_steps: int = 1000):
    """Time the float64 oracle on the host cores in a fresh process."""
    cores = len(os.sched_getaffinity(0))
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
from workloads import make_inputs
from oracle import ref_verify_step
inp = make_inputs({config_name!r}, seed=0)
ts = []
t_end = time.perf_counter() + {min_seconds}
while len(ts) < {max_steps} and (len(ts) < 2 or time.perf_counter() < t_end):
    t0 = time.perf_counter(); ref_verify_step(inp); ts.append(time.perf_counter() - t0)
print(json.dumps({{"per_step_s": sorted(ts)[len(ts)//2], "n": len(ts)}}))
"""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=600)
    if res.returncode != 0:
        return {"error": res.stderr.strip().splitlines()[-1:] or ["failed"]}
    d = json.loads(res.stdout.strip().splitlines()[-1])
    return {"value": d["per_step_s"] * 1e6, "unit": "us", "cores": cores, "kind": "oracle",
            "sample": f"the whole {config_name} verify step (attention for all tokens and heads + "
                      f"greedy verify), median of {d['n']} runs"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from workloads import CONFIGS
    cfg = CONFIGS[args.config]
    base = cpu_baseline(args.config, min_seconds=max(5.0, 0.5 * args.steps), max_steps=args.steps)
    if "error" in base:
        print(json.dumps({"impl": "reference", "unavailable": f"oracle run failed: {base['error']}"}))
        return
    v = base["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "us", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1000.0,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{cfg.name}: {cfg.description}"},
        "cpu_baseline": base,
        "e2e": {"value": v, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    import numpy as np
    import torch

    import speculative_decoding_verify_mla_gb300 as sv
    from workloads import CONFIGS, make_inputs

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    sv.load_library()

    cfg = CONFIGS[args.config]
    inp = make_inputs(cfg, seed=rank)
    R, k, H, T, V = inp["R"], inp["k"], inp["H"], inp["T"], cfg.vocab
    attn_flops, attn_bytes, logits_bytes = workload_figures(inp)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    def i32(x):
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(device)

    q, kv, gate = bf16(inp["q_bits"]), bf16(inp["kv_bits"]), bf16(inp["gate_bits"])
    bt, bounds = i32(inp["block_table"]), i32(inp["kv_bounds"])
    logits = torch.from_numpy(inp["logits"]).to(device)
    drafts, kv_in = i32(inp["draft_tokens"]), i32(inp["kv_lens_in"])
    step = sv.VerifyStep(device, R, k, H, V, inp["max_pages"], num_splits=args.splits)
    # L2 (129 MB) flush before every timed step: write 512 MB, then read
    # 256 MB of another buffer so that the write-back of the dirty flush
    # lines happens here and not inside the timed step
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=device)
    flush_sink = torch.empty((), dtype=torch.float32, device=device)

    def flush_l2():
        flush.zero_()
        torch.sum(flush_rd, dim=0, out=flush_sink)

    def run_step():
        return step(q, kv, bt, bounds, gate, inp["softmax_scale"], logits, drafts, kv_in)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def timed(fn, n):
        """Per-call device time (ms) of fn, L2 flushed before each call."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            flush_l2()
            starts[i].record()
            fn()
            ends[i].record()
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    for _ in range(max(3, args.warmup)):
        run_step()
    barrier()

    sampler = ClockSampler(local)
    if not args.no_clocks:
        sampler.start()
    barrier()
    step_ms = timed(run_step, args.steps)
    barrier()
    attn_ms = timed(lambda: sv.mla_verify_decode(q, kv, bt, bounds, gate, k + 1, inp["softmax_scale"],
                                                 num_splits=step.num_splits, workspace=step.attn_ws,
                                                 out=step.out, lse=step.lse, status=step.status),
                    args.steps)
    greedy_ms = timed(lambda: sv.spec_verify_greedy(logits, drafts, kv_in, k, workspace=step.greedy_ws,
                                                    argmax_ids=step.argmax, accepted=step.accepted,
                                                    next_tokens=step.next_tokens,
                                                    kv_lens_out=step.kv_lens_out), args.steps)
    # the same step replayed from a CUDA graph (launch overheads removed)
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=device)
        cap.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                run_step()
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        graph_ms = timed(g.replay, args.steps)
    except RuntimeError as e:  # capture unsupported by this torch/driver: reported, not hidden
        graph_error = str(e).splitlines()[0][:120]
    barrier()
    # paged latent KV append of the k+1 verify rows (the step just before the
    # attention); it rewrites the rows the pool already holds at those
    # positions, so the attention inputs stay the same
    pos_np = np.concatenate([np.arange(L - (k + 1), L) for L in inp["kv_lens_in"]]).astype(np.int32)
    rows = [int(inp["block_table"][t // (k + 1)][p // 64]) * 64 + p % 64 for t, p in enumerate(pos_np)]
    kv_new = kv.view(-1, 512)[torch.tensor(rows, dtype=torch.long, device=device)].contiguous()
    positions = i32(pos_np)
    append_ms = timed(lambda: sv.mla_kv_append(kv_new, positions, bt, kv, k + 1, status=step.status),
                      args.steps)
    # sampled (rejection-sampling) verification on the same logits shape, with
    # seeded draft distributions and uniforms
    from workloads import make_sampled_inputs
    sinp = make_sampled_inputs(cfg, seed=rank)
    s_logits = torch.from_numpy(sinp["logits"]).to(device)
    s_drafts, s_kv = i32(sinp["draft_tokens"]), i32(sinp["kv_lens_in"])
    s_probs = torch.from_numpy(sinp["draft_probs"]).to(device)
    s_uni = torch.from_numpy(sinp["uniforms"]).to(device)
    s_ws = sv.sampled_workspace(device, R, k, V)
    s_out = [torch.empty(R, dtype=torch.int32, device=device) for _ in range(3)]
    sampled_ms = timed(lambda: sv.spec_verify_sampled(s_logits, s_drafts, s_probs, s_uni, s_kv, k,
                                                      temperature=sinp["temperature"], workspace=s_ws,
                                                      accepted=s_out[0], next_tokens=s_out[1],
                                                      kv_lens_out=s_out[2]), args.steps)
    # the same attention over an fp8 (E4M3 + scale) copy of the KV pool
    from workloads import fp8_kv_pool
    codes, kv_scale = fp8_kv_pool(inp)
    kv8 = torch.from_numpy(codes).to(device)
    out8 = torch.empty_like(step.out)
    lse8 = torch.empty_like(step.lse)
    kv8_ms = timed(lambda: sv.mla_verify_decode(q, kv8, bt, bounds, gate, k + 1, inp["softmax_scale"],
                                                num_splits=step.num_splits, workspace=step.attn_ws,
                                                out=out8, lse=lse8, status=step.status, kv_scale=kv_scale),
                   args.steps)
    del kv8
    # per-head W_UV value up-projection of the attention output (v_dim 128,
    # seeded bf16 weights), the step after the merge
    from workloads import f32_to_bf16_bits
    w_np = f32_to_bf16_bits(np.random.default_rng(rank + 7).standard_normal((H, 128, 512), dtype=np.float32)
                            / np.float32(16.0))
    w_uv = torch.from_numpy(w_np.view(np.int16)).view(torch.bfloat16).to(device)
    out_v = torch.empty((T, H, 128), dtype=torch.bfloat16, device=device)
    wuv_ms = timed(lambda: sv.mla_wuv_project(step.out, w_uv, out_v=out_v), args.steps)
    # the LSE merge + gate on its own (the public entry point, fp32 partials
    # read from HBM after the flush), over the step's split count (4 when the
    # step does not split)
    s_comb = step.num_splits if step.num_splits > 1 else 4
    g_comb = torch.Generator(device=device).manual_seed(rank + 11)
    part_o = torch.randn((s_comb, T, H, 512), generator=g_comb, device=device)
    part_lse = torch.randn((s_comb, T, H), generator=g_comb, device=device)
    comb_out, comb_lse = torch.empty_like(step.out), torch.empty_like(step.lse)
    comb_ms = timed(lambda: sv.mla_lse_combine(part_o, part_lse, gate, out=comb_out, lse=comb_lse), args.steps)
    comb_bytes = s_comb * T * H * (2048 + 4) + T * H * (1024 + 1024 + 4)
    del part_o, part_lse
    barrier()
    clocks = sampler.stop() if not args.no_clocks else None

    # end to end through the public API: the step's inputs from pinned host
    # memory (two staged groups: attention inputs on the main stream, logits
    # and drafts on the greedy verify's stream), the step, the results back
    att = sv.StagedInputs(device, {"q_latent": (tuple(q.shape), q.dtype),
                                   "gate": (tuple(gate.shape), gate.dtype),
                                   "block_table": (tuple(bt.shape), bt.dtype),
                                   "kv_bounds": (tuple(bounds.shape), bounds.dtype)})
    ver = sv.StagedInputs(device, {"logits": (tuple(logits.shape), logits.dtype),
                                   "draft_tokens": (tuple(drafts.shape), drafts.dtype),
                                   "kv_lens_in": (tuple(kv_in.shape), kv_in.dtype)})
    for grp, items in ((att, (("q_latent", q), ("gate", gate), ("block_table", bt), ("kv_bounds", bounds))),
                       (ver, (("logits", logits), ("draft_tokens", drafts), ("kv_lens_in", kv_in)))):
        for kk, v in items:
            grp.host[kk].copy_(v.cpu())
    host_out = torch.empty((3, R), dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for g in (att, ver) for t in g.host.values())
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        res = step.run_staged(att, ver, kv, inp["softmax_scale"])
        host_out.copy_(res, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e2e_ms = timed(e2e_step, args.steps)
    barrier()

    # max over ranks
    def agg(xs):
        return max_over_ranks(xs, device, world)

    step_mean, attn_mean, greedy_mean, e2e_mean = (agg(step_ms), agg(attn_ms), agg(greedy_ms), agg(e2e_ms))
    append_mean = agg(append_ms)
    sampled_mean = agg(sampled_ms)
    wuv_mean = agg(wuv_ms)
    kv8_mean = agg(kv8_ms)
    comb_mean = agg(comb_ms)
    graph_mean = agg(graph_ms) if graph_ms else None
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peaks, peak_kind = load_peaks()
    attn_tflops = attn_flops / (attn_mean * 1e-3) / 1e12
    greedy_gbps = logits_bytes / (greedy_mean * 1e-3) / 1e9
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tensor_bound = attn_flops / attn_bytes > ridge
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": attn_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        ach = attn_bytes / (attn_mean * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(args.config)
    roof["kernel"] = "mla_verify_decode call (" + {3: "plan + attention + LSE combine kernels",
                                                   2: "attention + LSE combine kernels",
                                                   1: "attention kernel"}[step.attention_launches] + ")"
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json burst)" if peak_kind == "measured" else "fallback"
    roof["algorithmic_per_launch"] = {"flops": attn_flops, "bytes": attn_bytes}

    base = None
    if not args.no_cpu_baseline:
        base = cpu_baseline(args.config)

    line = {
        "metric": METRIC,
        "value": step_mean * 1000.0,
        "unit": "us",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_mean,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{cfg.name}: {cfg.description}", "R": R, "k": k, "H": H, "T": T,
                   "vocab": V, "latent": 512, "page": 64, "num_splits": step.num_splits,
                   "l2": "flushed before every timed step (512 MB write, then 256 MB read), outside the events",
                   "parallelism": f"replicas x{world}"},
        "attention_us": attn_mean * 1000.0,
        "attention_tflops": attn_tflops,
        "greedy_us": greedy_mean * 1000.0,
        "greedy_gbps": greedy_gbps,
        "greedy_hbm_frac": greedy_gbps / peaks["hbm_gbs"],
        "kv_append_us": append_mean * 1000.0,
        "kv_append_gbps": T * 2 * 1024 / (append_mean * 1e-3) / 1e9,
        "sampled_verify_us": sampled_mean * 1000.0,
        "sampled_verify_gbps": (T + 2 * R) * V * 4 / (sampled_mean * 1e-3) / 1e9,
        "step_graph_replay_us": graph_mean * 1000.0 if graph_mean else None,
        "attention_kv8_us": kv8_mean * 1000.0,
        "attention_kv8_tflops": attn_flops / (kv8_mean * 1e-3) / 1e12,
        "wuv_project_us": wuv_mean * 1000.0,
        "wuv_project_tflops": 2.0 * T * H * 128 * 512 / (wuv_mean * 1e-3) / 1e12,
        "combine_us": comb_mean * 1000.0,
        "combine_splits": s_comb,
        "combine_gbps": comb_bytes / (comb_mean * 1e-3) / 1e9,
        "combine_hbm_frac": comb_bytes / (comb_mean * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "steps_per_s_all_gpus": replica_throughput(step_mean, world),
        "roofline": roof,
        "cpu_baseline": base,
        "e2e": {"value": e2e_mean * 1000.0, "unit": "us", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * step.launches_per_step,
        "gpu_launches_all_timed_loops": args.steps * (3 * step.launches_per_step + step.attention_launches
                                                       + 1 + 1 + 2 + 1 + step.attention_launches + 1),
        "clocks": clocks,
        "status_word": int(step.status.item()),
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
