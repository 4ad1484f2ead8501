"""Verify-step benchmark: one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c4] [--impl reference]
                    [--extra-configs c1,c2,c3]

A step is one pass of the whole hot path on one synthetic batch: gated NoPE
MLA verify attention (with its split-KV LSE merge) followed by the greedy
verify (argmax, accepted prefix, trimmed kv_lens).  The default workload is
the long-context split-KV verify batch (16 requests, k=7, 64 heads, contexts
8K-32K with straddling groups and 10% bound-0 tokens, 163840-token
vocabulary), the largest of the verify-step configurations; the C=1, C=32
and C=64 batches are measured after it with the same method and reported
under "extra_configs".  Inputs sit in HBM before timing; L2 (129 MB) is
flushed before every timed step, outside the timed events, by writing a
512 MB buffer and then reading a 256 MB one (so the flush's own dirty lines
are written back before the step starts).  Every timed quantity is reported
as the median over the timed steps, with p10 / p90 / mean beside it.

--impl reference times the float64 CPU oracle on the same workload (host
cores), each step on a bounded sample of the batch's requests scaled to the
whole batch.  Under torchrun (N > 1) every rank runs an independent replica
(the verify step has no exchange between requests); rank 0 prints.
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
# nominal GB300 figures (dense bf16 tensor rate, HBM3e bandwidth), for context
NOMINAL_PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="c4")
    ap.add_argument("--extra-configs", default="c1,c2,c3",
                    help="comma-separated configurations measured after the main one ('' for none)")
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


def step_stats(times_ms):
    """Median, p10, p90 and mean (ms) of one rank's per-step times."""
    xs = sorted(times_ms)
    n = len(xs)

    def pct(p):
        # nearest-rank percentile
        return xs[min(n - 1, max(0, int(round(p / 100.0 * (n - 1)))))]
    return {"median": statistics.median(xs), "p10": pct(10), "p90": pct(90), "mean": statistics.mean(xs)}


def max_over_ranks(times_ms, device, world, stat="median"):
    """One statistic (median by default) of this rank's per-step times, then
    the maximum over all ranks (all_reduce MAX over the default process group
    when world > 1)."""
    m = step_stats(times_ms)[stat]
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


_ORACLE_SAMPLE_CODE = """
import json, math, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from workloads import make_inputs
from oracle import ref_greedy_verify, ref_verify_attention
inp = make_inputs({name!r}, seed=0)
R, k = inp["R"], inp["k"]
k1 = k + 1
n = R if R <= 2 else max(1, math.ceil(R / 8))
work_all = int(inp["kv_bounds"].astype(np.int64).sum())
ests = []
t_end = time.perf_counter() + {min_seconds}
s = 0
while s < {warmup} + {max_steps} and (s < {warmup} + {min_steps} or time.perf_counter() < t_end):
    reqs = [(s * n + i) % R for i in range(n)]
    toks = np.concatenate([np.arange(r * k1, (r + 1) * k1) for r in reqs])
    t0 = time.perf_counter()
    ref_verify_attention(inp["q_bits"][toks], inp["kv_bits"], inp["block_table"][reqs], inp["kv_bounds"][toks],
                         inp["gate_bits"][toks], k1, inp["softmax_scale"])
    ta = time.perf_counter() - t0
    t0 = time.perf_counter()
    ref_greedy_verify(inp["logits"][toks], inp["draft_tokens"][reqs], inp["kv_lens_in"][reqs], k)
    tg = time.perf_counter() - t0
    work = int(inp["kv_bounds"][toks].astype(np.int64).sum())
    scale_a = work_all / work if work > 0 else R / n
    if s >= {warmup}:
        ests.append(ta * scale_a + tg * R / n)
    s += 1
print(json.dumps({{"per_step_s": sorted(ests)[len(ests) // 2], "n": len(ests), "reqs": n, "R": R}}))
"""


def cpu_baseline(config_name: str, min_seconds: float = 10.0, min_steps: int = 3, max_steps: int = 1000,
                 warmup: int = 0):
    """Time the float64 oracle on the host cores in a fresh process (BLAS
    threads = the cores this process may use).  Each step runs the oracle on a
    bounded sample of the batch -- a rotating subset of its requests (all of
    them for batches of <= 2 requests) -- and scales the attention time by the
    attention work (sum of kv_bounds) and the greedy time by the number of
    logits rows to the whole batch; the median of those per-step estimates is
    reported."""
    cores = len(os.sched_getaffinity(0))
    code = _ORACLE_SAMPLE_CODE.format(root=ROOT, name=config_name, min_seconds=min_seconds,
                                      min_steps=min_steps, max_steps=max_steps, warmup=warmup)
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=1800)
    if res.returncode != 0:
        return {"error": res.stderr.strip().splitlines()[-1:] or ["failed"]}
    d = json.loads(res.stdout.strip().splitlines()[-1])
    if d["reqs"] >= d["R"]:
        how = "the whole batch each step"
    else:
        how = (f"{d['reqs']} of the batch's {d['R']} requests each step (rotating), attention time scaled "
               f"by the batch's sum of kv_bounds and greedy time by its logits rows")
    return {"value": d["per_step_s"] * 1e6, "unit": "us", "cores": cores, "kind": "oracle",
            "sample": f"{config_name} verify step (attention for every token and head + greedy verify) "
                      f"on {how}; median of {d['n']} steps"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from workloads import CONFIGS
    cfg = CONFIGS[args.config]
    base = cpu_baseline(args.config, min_seconds=0.0, min_steps=args.steps, max_steps=args.steps,
                        warmup=args.warmup)
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


def roofline(attn_flops, attn_bytes, attn_ms, peaks, peak_kind):
    """Attention roofline: tensor-bound when its arithmetic intensity is above
    the measured ridge point, else HBM-bound; fractions of the measured and
    of the nominal peak."""
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if attn_flops / attn_bytes > ridge:
        ach = attn_flops / (attn_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "peak_nominal": NOMINAL_PEAKS["bf16_tflops"]}
    else:
        ach = attn_bytes / (attn_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "peak_nominal": NOMINAL_PEAKS["hbm_gbs"]}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["frac_nominal"] = roof["achieved"] / roof["peak_nominal"]
    roof["peak_source"] = (f"{peak_kind} (MEASURED_PEAKS.json burst)" if peak_kind == "measured"
                           else "fallback")
    return roof


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
    peaks, peak_kind = load_peaks()

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    def i32(x):
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(device)

    # L2 (129 MB) flush before every timed step: write 512 MB, then read
    # 256 MB of another buffer so that the write-back of the dirty flush
    # lines happens here and not inside the timed step
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
    flush_rd = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=device)
    flush_sink = torch.empty((), dtype=torch.float32, device=device)

    def flush_l2():
        flush.zero_()
        torch.sum(flush_rd, dim=0, out=flush_sink)

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

    def measure(name, full):
        """Timed loops of one configuration: the step (eager and replayed
        from a CUDA graph), the attention call and the greedy verify alone;
        with `full`, also the neighbouring kernels and the end-to-end step."""
        cfg = CONFIGS[name]
        inp = make_inputs(cfg, seed=rank)
        R, k, H, T, V = inp["R"], inp["k"], inp["H"], inp["T"], cfg.vocab
        attn_flops, attn_bytes, logits_bytes = workload_figures(inp)
        q, kv, gate = bf16(inp["q_bits"]), bf16(inp["kv_bits"]), bf16(inp["gate_bits"])
        bt, bounds = i32(inp["block_table"]), i32(inp["kv_bounds"])
        logits = torch.from_numpy(inp["logits"]).to(device)
        drafts, kv_in = i32(inp["draft_tokens"]), i32(inp["kv_lens_in"])
        step = sv.VerifyStep(device, R, k, H, V, inp["max_pages"], num_splits=args.splits)
        res = {"cfg": cfg, "inp_figures": (attn_flops, attn_bytes, logits_bytes), "R": R, "k": k, "H": H,
               "T": T, "V": V, "num_splits": step.num_splits, "attention_launches": step.attention_launches,
               "launches_per_step": step.launches_per_step}

        def run_step():
            return step(q, kv, bt, bounds, gate, inp["softmax_scale"], logits, drafts, kv_in)

        for _ in range(max(3, args.warmup)):
            run_step()
        barrier()
        res["step"] = timed(run_step, args.steps)
        barrier()
        res["attn"] = timed(lambda: sv.mla_verify_decode(q, kv, bt, bounds, gate, k + 1, inp["softmax_scale"],
                                                         num_splits=step.num_splits, workspace=step.attn_ws,
                                                         out=step.out, lse=step.lse, status=step.status),
                            args.steps)
        res["greedy"] = timed(lambda: sv.spec_verify_greedy(logits, drafts, kv_in, k, workspace=step.greedy_ws,
                                                            argmax_ids=step.argmax, accepted=step.accepted,
                                                            next_tokens=step.next_tokens,
                                                            kv_lens_out=step.kv_lens_out), args.steps)
        # the same step replayed from a CUDA graph (launch overheads removed)
        res["graph"] = None
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
            res["graph"] = timed(g.replay, args.steps)
        except RuntimeError as e:  # capture unsupported by this torch/driver: reported, not hidden
            res["graph_error"] = str(e).splitlines()[0][:120]
        barrier()
        if not full:
            res["status_word"] = int(step.status.item())
            return res
        # paged latent KV append of the k+1 verify rows (the step just before
        # the attention); it rewrites the rows the pool already holds at those
        # positions, so the attention inputs stay the same
        pos_np = np.concatenate([np.arange(L - (k + 1), L) for L in inp["kv_lens_in"]]).astype(np.int32)
        rows = [int(inp["block_table"][t // (k + 1)][p // 64]) * 64 + p % 64 for t, p in enumerate(pos_np)]
        kv_new = kv.view(-1, 512)[torch.tensor(rows, dtype=torch.long, device=device)].contiguous()
        positions = i32(pos_np)
        res["append"] = timed(lambda: sv.mla_kv_append(kv_new, positions, bt, kv, k + 1, status=step.status),
                              args.steps)
        # sampled (rejection-sampling) verification on the same logits shape,
        # with seeded draft distributions and uniforms
        from workloads import make_sampled_inputs
        sinp = make_sampled_inputs(cfg, seed=rank)
        s_logits = torch.from_numpy(sinp["logits"]).to(device)
        s_drafts, s_kv = i32(sinp["draft_tokens"]), i32(sinp["kv_lens_in"])
        s_probs = torch.from_numpy(sinp["draft_probs"]).to(device)
        s_uni = torch.from_numpy(sinp["uniforms"]).to(device)
        s_ws = sv.sampled_workspace(device, R, k, V)
        s_out = [torch.empty(R, dtype=torch.int32, device=device) for _ in range(3)]
        res["sampled"] = timed(lambda: sv.spec_verify_sampled(s_logits, s_drafts, s_probs, s_uni, s_kv, k,
                                                              temperature=sinp["temperature"], workspace=s_ws,
                                                              accepted=s_out[0], next_tokens=s_out[1],
                                                              kv_lens_out=s_out[2]), args.steps)
        del s_logits, s_probs
        # the same attention over an fp8 (E4M3 + scale) copy of the KV pool
        from workloads import fp8_kv_pool
        codes, kv_scale = fp8_kv_pool(inp)
        kv8 = torch.from_numpy(codes).to(device)
        out8 = torch.empty_like(step.out)
        lse8 = torch.empty_like(step.lse)
        res["kv8"] = timed(lambda: sv.mla_verify_decode(q, kv8, bt, bounds, gate, k + 1, inp["softmax_scale"],
                                                        num_splits=step.num_splits, workspace=step.attn_ws,
                                                        out=out8, lse=lse8, status=step.status,
                                                        kv_scale=kv_scale), args.steps)
        del kv8
        # per-head W_UV value up-projection of the attention output (v_dim 128,
        # seeded bf16 weights), the step after the merge
        from workloads import f32_to_bf16_bits
        w_np = f32_to_bf16_bits(np.random.default_rng(rank + 7).standard_normal((H, 128, 512), dtype=np.float32)
                                / np.float32(16.0))
        w_uv = torch.from_numpy(w_np.view(np.int16)).view(torch.bfloat16).to(device)
        out_v = torch.empty((T, H, 128), dtype=torch.bfloat16, device=device)
        res["wuv"] = timed(lambda: sv.mla_wuv_project(step.out, w_uv, out_v=out_v), args.steps)
        # the LSE merge + gate on its own (the public entry point, fp32
        # partials read from HBM after the flush), over the step's split
        # count (4 when the step does not split or uses the balanced plan)
        s_comb = step.num_splits if step.num_splits > 1 else 4
        g_comb = torch.Generator(device=device).manual_seed(rank + 11)
        part_o = torch.randn((s_comb, T, H, 512), generator=g_comb, device=device)
        part_lse = torch.randn((s_comb, T, H), generator=g_comb, device=device)
        comb_out, comb_lse = torch.empty_like(step.out), torch.empty_like(step.lse)
        res["comb"] = timed(lambda: sv.mla_lse_combine(part_o, part_lse, gate, out=comb_out, lse=comb_lse),
                            args.steps)
        res["comb_splits"] = s_comb
        res["comb_bytes"] = s_comb * T * H * (2048 + 4) + T * H * (1024 + 1024 + 4)
        del part_o, part_lse
        barrier()
        # end to end through the public API: the step's inputs from pinned
        # host memory (two staged groups: attention inputs on the main stream,
        # logits and drafts on the greedy verify's stream), the step, the
        # results back
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
        res["h2d"] = sum(t.numel() * t.element_size() for g_ in (att, ver) for t in g_.host.values())
        res["d2h"] = host_out.numel() * host_out.element_size()

        def e2e_step():
            out = step.run_staged(att, ver, kv, inp["softmax_scale"])
            host_out.copy_(out, non_blocking=True)

        for _ in range(3):
            e2e_step()
        barrier()
        res["e2e"] = timed(e2e_step, args.steps)
        barrier()
        res["status_word"] = int(step.status.item())
        return res

    sampler = ClockSampler(local)
    if not args.no_clocks:
        sampler.start()
    barrier()
    main_res = measure(args.config, full=True)
    extra_names = [c for c in args.extra_configs.split(",") if c and c != args.config]
    extra_res = {}
    for name in extra_names:
        torch.cuda.empty_cache()
        extra_res[name] = measure(name, full=False)
    barrier()
    clocks = sampler.stop() if not args.no_clocks else None

    # max over ranks (the median of each timed loop, and p10 / p90 / mean)
    def agg(xs, stat="median"):
        return max_over_ranks(xs, device, world, stat)

    def dist_of(xs):
        return {s: agg(xs, s) * 1000.0 for s in ("median", "p10", "p90", "mean")}

    def summary(res):
        attn_flops, attn_bytes, logits_bytes = res["inp_figures"]
        step_d, attn_d, greedy_d = dist_of(res["step"]), dist_of(res["attn"]), dist_of(res["greedy"])
        graph_d = dist_of(res["graph"]) if res.get("graph") else None
        attn_ms = attn_d["median"] / 1000.0
        greedy_gbps = logits_bytes / (greedy_d["median"] * 1e-6) / 1e9
        roof = roofline(attn_flops, attn_bytes, attn_ms, peaks, peak_kind)
        return {
            "workload": f"{res['cfg'].name}: {res['cfg'].description}",
            "num_splits": res["num_splits"],
            "step_us": step_d, "step_graph_replay_us": graph_d,
            "attention_us": attn_d, "attention_tflops": attn_flops / (attn_ms * 1e-3) / 1e12,
            "attention_roofline": roof,
            "greedy_us": greedy_d, "greedy_gbps": greedy_gbps,
            "greedy_hbm_frac": greedy_gbps / peaks["hbm_gbs"],
            "greedy_hbm_frac_nominal": greedy_gbps / NOMINAL_PEAKS["hbm_gbs"],
            "status_word": res["status_word"],
        }

    main_sum = summary(main_res)
    extra_sum = {name: summary(r) for name, r in extra_res.items()}
    m = main_res
    append_us = agg(m["append"]) * 1000.0
    sampled_us = agg(m["sampled"]) * 1000.0
    wuv_us = agg(m["wuv"]) * 1000.0
    kv8_us = agg(m["kv8"]) * 1000.0
    comb_us = agg(m["comb"]) * 1000.0
    e2e_us = agg(m["e2e"]) * 1000.0
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    attn_flops, attn_bytes, logits_bytes = m["inp_figures"]
    R, k, H, T, V = m["R"], m["k"], m["H"], m["T"], m["V"]
    roof = dict(main_sum["attention_roofline"])
    roof["traffic"] = recorded_traffic(args.config)
    if roof["traffic"] is not None:
        roof["traffic_scope"] = ("dram__bytes_read.sum + dram__bytes_write.sum of the attention kernel "
                                 "(mla_verify_kernel) per launch, one ncu capture "
                                 f"(profiles/mla_verify_kernel_{args.config}.md)")
    roof["kernel"] = "mla_verify_decode call (" + {3: "plan + attention + LSE combine kernels",
                                                   2: "attention + LSE combine kernels",
                                                   1: "attention kernel"}[m["attention_launches"]] + ")"
    roof["timing"] = "median CUDA-event duration of the call over the timed steps, L2 flushed before each"
    roof["algorithmic_per_launch"] = {"flops": attn_flops, "bytes": attn_bytes}

    base = None
    if not args.no_cpu_baseline:
        base = cpu_baseline(args.config)

    step_med = main_sum["step_us"]["median"]
    line = {
        "metric": METRIC,
        "value": step_med,
        "unit": "us",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_med / 1000.0,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": main_sum["workload"], "R": R, "k": k, "H": H, "T": T,
                   "vocab": V, "latent": 512, "page": 64, "num_splits": m["num_splits"],
                   "l2": "flushed before every timed step (512 MB write, then 256 MB read), outside the events",
                   "statistic": "median of the timed steps (p10 / p90 / mean under step_us)",
                   "parallelism": f"replicas x{world}"},
        "step_us": main_sum["step_us"],
        "step_graph_replay_us": main_sum["step_graph_replay_us"],
        "attention_us": main_sum["attention_us"],
        "attention_tflops": main_sum["attention_tflops"],
        "greedy_us": main_sum["greedy_us"],
        "greedy_gbps": main_sum["greedy_gbps"],
        "greedy_hbm_frac": main_sum["greedy_hbm_frac"],
        "greedy_hbm_frac_nominal": main_sum["greedy_hbm_frac_nominal"],
        "kv_append_us": append_us,
        "kv_append_gbps": T * 2 * 1024 / (append_us * 1e-6) / 1e9,
        "sampled_verify_us": sampled_us,
        "sampled_verify_gbps": (T + 2 * R) * V * 4 / (sampled_us * 1e-6) / 1e9,
        "attention_kv8_us": kv8_us,
        "attention_kv8_tflops": attn_flops / (kv8_us * 1e-6) / 1e12,
        "wuv_project_us": wuv_us,
        "wuv_project_tflops": 2.0 * T * H * 128 * 512 / (wuv_us * 1e-6) / 1e12,
        "combine_us": comb_us,
        "combine_splits": m["comb_splits"],
        "combine_gbps": m["comb_bytes"] / (comb_us * 1e-6) / 1e9,
        "combine_hbm_frac": m["comb_bytes"] / (comb_us * 1e-6) / 1e9 / peaks["hbm_gbs"],
        "steps_per_s_all_gpus": replica_throughput(step_med / 1000.0, world),
        "roofline": roof,
        "cpu_baseline": base,
        "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"]},
        "gpu_launches": args.steps * m["launches_per_step"],
        "gpu_launches_all_timed_loops": args.steps * (3 * m["launches_per_step"] + m["attention_launches"]
                                                       + 1 + 1 + 2 + 1 + m["attention_launches"] + 1)
                                        + sum(args.steps * (3 * r["launches_per_step"] + r["attention_launches"]
                                                            + 1) for r in extra_res.values()),
        "extra_configs": extra_sum,
        "clocks": clocks,
        "status_word": main_sum["status_word"],
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
