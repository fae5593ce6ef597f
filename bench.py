"""Benchmark of the fused verify step (spec_verify_step) on the bass_b8 workload.

`--path draft` measures the draft side instead: K consecutive draft positions
per step (single-row attention, append, draft-token draw).

Default: 1 GPU.  Under torchrun, one rank per GPU, each with its own batch of
8 sequences (global sequence ids offset by rank): weak scaling, no data-path
collective; the barrier and the max-over-ranks timing use torch.distributed.

Prints one JSON line (rank 0).  `value` = verify steps/s of the whole job with
inputs resident in HBM (CUDA-graph replays of the C-ABI call, three rotating
input sets so every step reads ~157 MB > L2; exactly --steps calls timed);
`e2e` = the same metric through the C-ABI call with pinned host buffers copied
in and results copied out every step; `roofline` = the attention kernel (the
dominant one) timed alone; `cpu_baseline` = the CPU oracle timed on a bounded
sample with one thread, `cpu_baseline_all_cores` with every core of the
affinity mask.  Draft tokens are drawn from the processed draft rows p_hat on
the device (the draft model's sampler) unless --gumbel-drafts; the oracle
draws its own from the same rows and counters.  `oracle_check` compares the
GPU step's outputs with the oracle's on these inputs, `ties` counts the
decisions inside the near-tie windows, `acceptance` sets the measured mean
accepted drafts per sequence (over --acc-seeds Philox seeds) beside the closed
form sum_j prod_t sum_x min(p_hat, q_hat); `padded` (with --padded) times the
same batch padded to its longest cache and largest K.
`--impl reference` times the CPU oracle alone (the reference arm).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "verify steps/s & accepted tok/s at B=8 7.8B-shape; achieved HBM GB/s vs peak"
UNIT = "steps/s"
WORKLOAD = "bass_b8"
FALLBACK_HBM_GBS = 6800.0


def workload_desc(w):
    K = f"K={w.K_lo}" if w.K_lo == w.K_hi else f"K in [{w.K_lo},{w.K_hi}]"
    pre = f", shared prefix {w.prefix_len}" if w.prefix_len else ""
    kv = f", K/V {w.kv_dtype} (scale {w.kv_scale})" if w.kv_dtype else ""
    return (f"{w.name}: B={w.B}, Hq={w.Hq}, Hkv={w.Hkv}, D={w.D}, KV len {w.L_dist} "
            f"[{w.L_lo},{w.L_hi}]{pre}, {K}, V={w.V}, {w.dtype}{kv}, T={w.temperature}, "
            f"top_p={w.top_p}, top_k={w.top_k}")


def kernels_per_step(w):
    """Kernels one fused step launches: the attention (prefix row-blocks,
    decode partials and their merge with a shared prefix) and the sampler (one
    cluster kernel without processing beyond a temperature, else statistics +
    draw kernels)."""
    attn = 3 if w.prefix_len or w.prefix_lens else 1
    cluster = w.top_p >= 1.0 and w.top_k == 0 and w.temperature > 0.0
    return attn + (1 if cluster else 2)


def compute_dtype(w):
    """What the path computes in: bf16 / fp32 operands, or E4M3 K/V codes
    widened to f16 tensor-core operands (fp32 accumulation throughout)."""
    return "e4m3 K/V -> f16 mma, bf16 q/out" if w.kv_dtype == "e4m3" else w.dtype


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm_gb_s"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def traffic_record(kernel_src_sha, workload=WORKLOAD):
    """DRAM bytes per attention launch from a committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    for ln in open(p):
        f = ln.split()
        if len(f) == 4 and f[0] == "attention" and f[1] == workload and f[2] == kernel_src_sha:
            return float(f[3])
    return None


def src_sha():
    """Hash of the attention kernel's sources with comments and whitespace
    removed (a comment edit leaves the compiled kernel, and so its recorded
    DRAM traffic, unchanged)."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verify_09_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("attention") or f.endswith((".cuh", ".h")):
            text = open(os.path.join(csrc, f)).read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            h.update(f.encode() + b"\0" + "".join(text.split()).encode())
    return h.hexdigest()[:12]


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in open(self.path):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def cpu_baseline(inp, budget_s=12.0, cores=1):
    """The oracle, as it stands, on whole steps of the workload until the
    budget is used (at least one step); BLAS/OMP threads as the process was
    started with (`cores`)."""
    import oracle
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.verify_step(inp)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": n / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} whole {inp['workload'].name} steps (attention + sampling + append), "
                      f"{el:.1f} s, OMP/BLAS threads {cores}"}


def cpu_baseline_all_cores(argv, budget_s=10.0):
    """The same timing in a child process whose BLAS/OMP threads are all the
    cores of this process's affinity mask (the thread count is fixed when numpy
    loads, hence the child)."""
    ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    env = dict(os.environ, OMP_NUM_THREADS=str(ncores), OPENBLAS_NUM_THREADS=str(ncores),
               MKL_NUM_THREADS=str(ncores), CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), *argv, "--cpu-child",
                            str(ncores), "--cpu-budget", str(budget_s)],
                           capture_output=True, text=True, env=env, timeout=budget_s * 6 + 120)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:        # reported, never fatal to the GPU measurement
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


def overrides(args):
    """Workload overrides from the command line (sampling parameters, K)."""
    over = {k: v for k, v in (("temperature", args.temperature), ("top_k", args.top_k),
                              ("top_p", args.top_p)) if v is not None}
    if args.k is not None:
        over.update(K_lo=args.k, K_hi=args.k, K_fixed=())
    if args.kv_dtype is not None:
        over.update(kv_dtype=args.kv_dtype)
    if args.draft_noise is not None:
        over.update(draft_noise=args.draft_noise)
    return over


def run_reference(args, rank):
    if rank != 0:
        return
    over = overrides(args)
    w = W.workload(args.workload, **over)
    import oracle
    if args.path == "draft":
        P = args.positions or w.K_hi
        base, dsteps = W.make_draft_inputs(w, positions=P)

        def one():
            inp = dict(base)
            for st in dsteps:
                inp.update(st)
                r = oracle.draft_step(inp)
                inp.update(k_cache=r["k_cache"], v_cache=r["v_cache"], kv_len=r["new_kv_len"])
        metric = DRAFT_METRIC
    else:
        inp = W.make_inputs(w)
        if not args.gumbel_drafts:      # the oracle's own draws from p_hat (untimed setup)
            inp["draft_tokens"], _ = oracle_drafts(inp)

        def one():
            oracle.verify_step(inp)
        metric = METRIC
    for _ in range(min(args.warmup, 3)):          # (bounded: the oracle takes ~0.5 s a step)
        one()
    steps = max(1, min(args.steps, 3))
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    el = time.perf_counter() - t0
    v = steps / el
    line = {"impl": "reference", "metric": metric, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "warmup": min(args.warmup, 3), "ms_per_step": 1e3 * el / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(w)},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{steps} whole steps (the requested count, capped at 3)"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def timed_replays(torch, sets, fn, n_launch, stream, dist, shard, no_graph, percentiles):
    """Time exactly n_launch calls of fn over the rotating input sets with CUDA
    events on the launching stream: full replays of one CUDA graph holding one
    call per set, then (when n_launch is not a multiple of the sets) one replay
    of a graph holding the first n_launch % len(sets) calls (unless no_graph);
    the barrier and max over ranks make it the job's time.  Returns (ms, calls,
    pct): pct (with percentiles) holds p10 / p50 / p90 of the time per call over
    200 single full replays, each bracketed by its own events."""
    n_launch = max(1, int(n_launch))
    reps, rem = divmod(n_launch, len(sets))
    graph = graph_rem = None
    if not no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for d in sets:
                fn(d)
        if rem:
            graph_rem = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph_rem):
                for d in sets[:rem]:
                    fn(d)
        torch.cuda.synchronize()
    for _ in range(2):
        graph.replay() if graph else [fn(d) for d in sets]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(reps):
        if graph:
            graph.replay()
        else:
            for d in sets:
                fn(d)
    if rem:
        if graph_rem is not None:
            graph_rem.replay()
        else:
            for d in sets[:rem]:
                fn(d)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = shard.max_over_ranks(ev0.elapsed_time(ev1), dist, device="cuda")
    pct = None
    if percentiles and graph is not None:
        n = 200
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
        for i in range(n):
            evs[2 * i].record(stream)
            graph.replay()
            evs[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        per = np.array([evs[2 * i].elapsed_time(evs[2 * i + 1]) * 1e3 / len(sets)
                        for i in range(n)])
        pct = {"p10": float(np.percentile(per, 10)), "p50": float(np.percentile(per, 50)),
               "p90": float(np.percentile(per, 90)), "unit": "us per call",
               "replays": n, "calls_per_replay": len(sets)}
    return ms, n_launch, pct


def draft_rows(inp, j):
    """Sequences with a draft j + 1 and the index of their draft row j."""
    cu = np.asarray(inp["cu_q"], dtype=np.int64)
    K = np.diff(cu) - 1
    seqs = np.flatnonzero(K > j)
    return seqs, cu[seqs] - seqs + j


def draw_drafts_on_device(torch, api, d, inp, seed=None):
    """Replace the draft tokens of StepBuffers `d` by draws from the processed
    draft rows (spec_draft_sample: temperature / top-k / top-p, Philox stream
    1): draft j + 1 of sequence i is drawn from its draft row j, at token index
    kv_len[i] + j + 1, as the draft model's sampler draws it.  Setup only
    (untimed).  Returns the tokens as a host array."""
    K = np.diff(np.asarray(inp["cu_q"])) - 1
    for j in range(int(K.max()) if K.size else 0):
        seqs, rows = draft_rows(inp, j)
        idx = torch.from_numpy(rows).cuda()
        logits = d.drf.index_select(0, idx).contiguous()
        kv = torch.from_numpy((np.asarray(inp["kv_len"])[seqs] + j).astype(np.int32)).cuda()
        sid = d.seq_ids.index_select(0, torch.from_numpy(seqs).cuda()).contiguous()
        out = torch.empty(len(seqs), dtype=torch.int32, device="cuda")
        args = api.draft_args(logits, kv, out, temperature=inp["temperature"],
                              top_p=inp["top_p"], seed=inp["seed"] if seed is None else seed,
                              seq_ids=sid, dev_status=d.status, top_k=inp.get("top_k", 0))
        ws = api.Workspace(api.draft_workspace_bytes(args))
        api.spec_draft_sample(args, ws)
        d.drafts.index_copy_(0, idx, out)
        torch.cuda.synchronize()
    return d.drafts.cpu().numpy()


def oracle_drafts(inp):
    """The oracle's own draws of the same drafts (same rows, indices and
    Philox stream 1 counters as draw_drafts_on_device); returns (tokens, set of
    draft rows inside the oracle's draw tie window)."""
    import oracle
    toks = np.array(inp["draft_tokens"], copy=True)
    tied = set()
    K = np.diff(np.asarray(inp["cu_q"])) - 1
    for j in range(int(K.max()) if K.size else 0):
        seqs, rows = draft_rows(inp, j)
        r = oracle.draft_sample(inp["draft_logits"][rows], np.asarray(inp["kv_len"])[seqs] + j,
                                inp["temperature"], inp["top_p"], inp["seed"],
                                np.asarray(inp["seq_ids"])[seqs], inp.get("top_k", 0))
        toks[rows] = r["tokens"]
        tied |= {int(x) for x in rows[r["tie"]]}
    return toks, tied


def oracle_check(inp_oracle, gpu_drafts, drafts_tied, num_accepted, out_tokens):
    """The oracle's step on its own drafts against the GPU's outputs: sequences
    equal bit for bit, inside a near-tie window (a draft draw or a step
    decision), or different (must be 0), and the tie counts by clause."""
    import oracle
    ref = oracle.verify_step(inp_oracle, attention=False)
    cu = np.asarray(inp_oracle["cu_q"])
    exact = tied = bad = 0
    draft_ties = 0
    for i in range(len(cu) - 1):
        r0, r1 = int(cu[i]), int(cu[i + 1])
        rows = range(r0 - i, r1 - i - 1)
        if any(r in drafts_tied for r in rows):
            draft_ties += 1
            tied += 1
            continue
        if any(int(gpu_drafts[r]) != int(inp_oracle["draft_tokens"][r]) for r in rows):
            bad += 1
            continue
        if ref["tie_kind"][i]:
            tied += 1
            continue
        same = int(num_accepted[i]) == int(ref["num_accepted"][i]) and \
            list(out_tokens[r0:r1]) == list(ref["out_tokens"][r0:r1])
        exact += same
        bad += not same
    return ({"sequences": len(cu) - 1, "exact": exact, "tied": tied, "different": bad},
            {"sequences": int(ref["tie_count"]) + draft_ties,
             "positions": int(ref["tie_positions"]) + len(drafts_tied),
             "clauses": dict(ref["tie_clauses"], draft_draw=draft_ties)})


def acceptance_closed_form(inp):
    """Expected accepted drafts per sequence with drafts drawn from p_hat:
    sum_j prod_{t <= j} beta_t, beta_t = sum_x min(p_hat_t, q_hat_t) (the
    speculative-sampling paper's acceptance rate, appendix "Proof")."""
    from oracle.sampling import process_row, to_f64
    cu = np.asarray(inp["cu_q"])
    tot = []
    for i in range(len(cu) - 1):
        r0, K = int(cu[i]), int(cu[i + 1] - cu[i] - 1)
        e, run = 0.0, 1.0
        for j in range(K):
            q = process_row(to_f64(inp["target_logits"][r0 + j]), inp["temperature"],
                            inp["top_p"], inp.get("top_k", 0)).probs
            p = process_row(to_f64(inp["draft_logits"][r0 - i + j]), inp["temperature"],
                            inp["top_p"], inp.get("top_k", 0)).probs
            run *= float(np.minimum(p, q).sum())
            e += run
        tot.append(e)
    return float(np.mean(tot))


DRAFT_METRIC = ("draft-side steps/s (K positions of single-row attention + append + draft "
                "draw) at B=8 7.8B-shape; achieved HBM GB/s vs peak")


def draft_cpu_baseline(base, steps, budget_s=12.0):
    """The oracle's draft positions, as they stand, until the budget is used
    (at least one whole draft-side step of len(steps) positions)."""
    import oracle
    n, t0 = 0, time.perf_counter()
    while True:
        inp = dict(base)
        for st in steps:
            inp.update(st)
            r = oracle.draft_step(inp)
            inp.update(k_cache=r["k_cache"], v_cache=r["v_cache"], kv_len=r["new_kv_len"])
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": n / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} whole draft-side steps of {len(steps)} positions, {el:.1f} s, "
                      "OMP/BLAS threads 1"}


def run_draft(args, w, api, shard, dist, world, rank, local_rank):
    """The draft side of the loop: K consecutive draft positions per step."""
    import torch
    from speculative_decoding_verify_09_gb300.buffers import DraftBuffers
    P = args.positions or w.K_hi
    base, steps = W.make_draft_inputs(w, positions=P)
    lo, _ = shard.rank_range(world * w.B, rank, world)
    base["seq_ids"] = base["seq_ids"] + lo
    sets = [DraftBuffers(base, api, positions=P, steps=steps) for _ in range(args.sets)]
    stream = torch.cuda.current_stream()
    per_pos = W.draft_step_bytes(base)
    esz = 4 if w.dtype == "f32" else 2
    attn_bytes = per_pos - w.B * w.V * esz - 2 * w.B * 2 * w.Hkv * w.D * esz

    def timed(fn, n_launch, percentiles=False):
        return timed_replays(torch, sets, fn, n_launch, stream, dist, shard, args.no_graph,
                             percentiles)

    for k in range(max(args.warmup, 3)):
        sets[k % len(sets)].run_all(fused=True)
        sets[k % len(sets)].run_all()
    torch.cuda.synchronize()
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0] \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else str(local_rank)
    clk = Clocks(gpu_index)
    time.sleep(0.3)
    # a position as one call (spec_draft_step: draw and append beside the
    # attention); the three separate calls are timed after it for comparison
    ms_step, n_steps, pct = timed(lambda d: d.run_all(fused=True), args.steps, percentiles=True)
    clocks = clk.stop()
    ms_3, n_3, _ = timed(lambda d: d.run_all(), args.steps)

    def attn0(d):
        api.spec_verify_attn(d.attn[0], d.ws_attn)

    ms_attn, n_attn, _ = timed(attn0, args.attn_steps)
    attn_us = 1e3 * ms_attn / n_attn
    peak, peak_kind = peaks()
    achieved = attn_bytes / (attn_us * 1e-6) / 1e9
    sha = src_sha()
    per_step_ms = ms_step / n_steps
    step_total = P * per_pos

    # end to end: every step uploads all positions' inputs (one pinned arena),
    # runs the positions and downloads their outputs (one pinned arena)
    d = sets[0]
    d.stage(steps)
    for it in range(3 + args.e2e_steps):
        if it == 3:
            if dist:
                dist.barrier()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        d.upload()
        d.run_all(fused=True)
        d.download()
        stream.synchronize()
    e2e_s = shard.max_over_ranks(time.perf_counter() - t0, dist, device="cuda")
    e2e = {"value": world * args.e2e_steps / e2e_s, "unit": UNIT,
           "h2d_bytes_per_step": d.in_bytes, "d2h_bytes_per_step": d.out_bytes}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = draft_cpu_baseline(base, steps)
    if rank == 0:
        line = {
            "metric": DRAFT_METRIC, "value": world * n_steps / (ms_step / 1e3), "unit": UNIT,
            "n_gpus": world, "steps": n_steps, "warmup": max(args.warmup, 3),
            "ms_per_step": per_step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": compute_dtype(w),
            "data": "synthetic (seeded; random-init tensors of the workload's shapes)",
            "config": {"workload": workload_desc(w) + f"; draft side: {P} positions of one "
                       "query row per sequence (draft attention layer of the same shape)",
                       "parallelism": f"dp{world} (sequence shards)", "global_batch": world * w.B,
                       "l2": f"{len(sets)} rotating input sets; each position reads "
                             f"{per_pos / 1e6:.0f} MB (the K positions of a step re-read one "
                             "cache, as a draft model does)",
                       "launch": "CUDA graph of the C-ABI calls per input set"
                       if not args.no_graph else "direct launches"},
            "draft_tok_s": world * w.B * P * n_steps / (ms_step / 1e3),
            "step_time_percentiles": pct,
            "three_calls_per_position": {"ms_per_step": ms_3 / n_3, "steps": n_3,
                                         "how": "spec_verify_attn, kv_append_ragged and "
                                                "spec_draft_sample per position, serialized"},
            "step_bytes": step_total,
            "step_hbm_gbs": step_total / (per_step_ms * 1e-3) / 1e9,
            "step_frac_of_peak": step_total / (per_step_ms * 1e-3) / 1e9 / peak,
            "roofline": {"kernel": "attention, one query row per sequence", "bound": "hbm",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                         "traffic": traffic_record(sha, "draft_" + args.workload),
                         "algorithmic_bytes_per_launch": attn_bytes,
                         "avg_launch_us": attn_us, "kernel_src": sha},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": kernels_per_step(w) * P * n_steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--sets", type=int, default=3, help="rotating input sets (L2 defeat)")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--attn-steps", type=int, default=3000,
                    help="attention-only launches timed for the roofline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch directly (profiling)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(W.WORKLOADS),
                    help="input shapes (default: the headline bass_b8)")
    ap.add_argument("--temperature", type=float, default=None, help="override (0 = greedy)")
    ap.add_argument("--top-k", type=int, default=None, help="override (0 = off)")
    ap.add_argument("--top-p", type=float, default=None, help="override")
    ap.add_argument("--kv-dtype", default=None, choices=["e4m3"],
                    help="override: E4M3 K/V (8-bit cache, per-tensor scales)")
    ap.add_argument("--k", type=int, default=None,
                    help="override: every sequence drafts K tokens (K sweep)")
    ap.add_argument("--path", default="verify", choices=["verify", "draft"],
                    help="verify: the fused verify step (default); draft: the draft side "
                         "(K single-row positions per step)")
    ap.add_argument("--positions", type=int, default=None,
                    help="draft positions per draft-side step (default: the workload's K)")
    ap.add_argument("--draft-noise", type=float, default=None,
                    help="override: std of the draft logits' noise around the target logits")
    ap.add_argument("--padded", action="store_true",
                    help="also time the same batch padded (every cache to the longest, every "
                         "block to the largest K), as a padded multi-sample step would run")
    ap.add_argument("--gumbel-drafts", action="store_true",
                    help="keep the generator's stand-in drafts (Gumbel-max over the unprocessed "
                         "draft row) instead of drawing them from p_hat on the device")
    ap.add_argument("--acc-seeds", type=int, default=64,
                    help="Philox seeds of the measured acceptance (drafts redrawn per seed)")
    ap.add_argument("--cpu-child", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help=argparse.SUPPRESS)
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.cpu_child:                  # the oracle timed with all cores (no GPU)
        inp = W.make_inputs(W.workload(args.workload, **overrides(args)))
        if not args.gumbel_drafts:
            inp["draft_tokens"], _ = oracle_drafts(inp)
        print(json.dumps(cpu_baseline(inp, args.cpu_budget, cores=args.cpu_child)), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import speculative_decoding_verify_09_gb300 as pkg
    from speculative_decoding_verify_09_gb300 import shard
    pkg.build()
    api = pkg.load()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    # weak scaling: rank r owns global sequences [r*B, (r+1)*B) of a batch of
    # world*B sequences (the same shapes on every rank, uniforms keyed by the
    # global sequence id); no exchange on the data path
    over = overrides(args)
    w = W.workload(args.workload, **over)
    if args.path == "draft":
        run_draft(args, w, api, shard, dist, world, rank, local_rank)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return
    inp = W.make_inputs(w)
    lo, _ = shard.rank_range(world * w.B, rank, world)
    inp["seq_ids"] = inp["seq_ids"] + lo
    from speculative_decoding_verify_09_gb300.buffers import StepBuffers
    sets = [StepBuffers(inp, api) for _ in range(args.sets)]
    if not args.gumbel_drafts:        # drafts from p_hat, as the draft model draws them
        for d in sets:
            gpu_drafts = draw_drafts_on_device(torch, api, d, inp)
        inp["draft_tokens"] = gpu_drafts
    nbytes = W.step_bytes(inp)
    stream = torch.cuda.current_stream()

    def step(d):
        api.spec_verify_step(d.attn, d.sample, d.kv_cap, d.new_kv_len, d.ws)

    def attn_only(d):
        api.spec_verify_attn(d.attn, d.ws)

    # warm-up (also settles the accepted counts used for the append bytes)
    for k in range(max(args.warmup, 3)):
        step(sets[k % len(sets)])
    torch.cuda.synchronize()
    n_acc = sets[0].num_accepted.cpu().numpy()
    emitted = int(np.sum(n_acc + 1))
    esz = 4 if w.dtype == "f32" else 2
    kvsz = 1 if w.kv_dtype == "e4m3" else esz
    append_bytes = 2 * 2 * emitted * w.Hkv * w.D * kvsz       # K and V, read + write
    step_total = nbytes["attention"] + nbytes["sampler"] + append_bytes

    def timed(fn, n_launch, percentiles=False):
        return timed_replays(torch, sets, fn, n_launch, stream, dist, shard, args.no_graph,
                             percentiles)

    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0] \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else str(local_rank)
    clk = Clocks(gpu_index)
    time.sleep(0.3)
    ms_step, n_steps, pct = timed(step, args.steps, percentiles=True)
    clocks = clk.stop()
    ms_attn, n_attn, _ = timed(attn_only, args.attn_steps)

    emitted_all = int(shard.sum_over_ranks(emitted, dist, device="cuda"))
    per_step_ms = ms_step / n_steps
    value = world * n_steps / (ms_step / 1e3)
    attn_us = 1e3 * ms_attn / n_attn
    peak, peak_kind = peaks()
    achieved = nbytes["attention"] / (attn_us * 1e-6) / 1e9
    sha = src_sha()
    traffic = traffic_record(sha, args.workload + ("_e4m3" if w.kv_dtype == "e4m3" else ""))

    # end to end through the C ABI: every step copies its inputs (one pinned
    # host arena -> one device arena), runs the fused call and copies its
    # results back (one device arena -> pinned host).  Serial: the host waits
    # for each step.  Two batches in flight (a two-micro-batch serving loop):
    # the host waits for a batch's previous result before issuing its next
    # step, while the other batch's copies and step run.
    from speculative_decoding_verify_09_gb300.buffers import StagedStep
    if len(sets) < 2:
        sets.append(StepBuffers(inp, api))
    staged = [StagedStep(sets[0]), StagedStep(sets[1])]
    for x in staged:
        x.pack(inp)
    h2d, d2h = staged[0].in_bytes, staged[0].out_bytes

    def e2e_run(pipelined):
        # uploads and downloads on their own streams: a batch's upload never
        # waits behind the other batch's download (which waits for its step)
        cs_up, cs_dn = torch.cuda.Stream(), torch.cuda.Stream()
        up = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        dl = [torch.cuda.Event() for _ in range(2)]

        def issue(i):
            b = i % 2 if pipelined else 0
            x, d = staged[b], sets[b]
            if pipelined:
                with torch.cuda.stream(cs_up):
                    x.upload()
                    up[b].record(cs_up)
                stream.wait_event(up[b])
            else:
                x.upload()
            api.spec_verify_step(x.attn, x.sample, d.kv_cap, d.new_kv_len, d.ws)
            if pipelined:
                done[b].record(stream)
                with torch.cuda.stream(cs_dn):
                    cs_dn.wait_event(done[b])
                    x.download()
                    dl[b].record(cs_dn)
            else:
                x.download()
                stream.synchronize()

        for i in range(4):
            issue(i)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t0 = time.perf_counter()
        for i in range(args.e2e_steps):
            if pipelined:
                dl[i % 2].synchronize()        # this batch's previous result is on the host
            issue(i)
        torch.cuda.synchronize()
        el = shard.max_over_ranks(time.perf_counter() - t0, dist, device="cuda")
        return {"value": world * args.e2e_steps / el, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h}

    e2e_serial = e2e_run(False)
    e2e = e2e_run(True)
    e2e["mode"] = "two independent batches in flight (copies of one overlap the other's step)"
    e2e_serial["mode"] = "one step at a time, host waits for each"

    # measured acceptance (untimed): per Philox seed, redraw the drafts from
    # p_hat and run the sampler; mean accepted drafts per sequence
    acc = None
    if not args.gumbel_drafts and args.acc_seeds > 0:
        dacc = StepBuffers(inp, api)
        tot = 0.0
        for sd in range(args.acc_seeds):
            draw_drafts_on_device(torch, api, dacc, inp, seed=1000 + sd)
            dacc.sample.seed = 1000 + sd
            api.spec_reject_sample(dacc.sample, dacc.ws)
            tot += float(dacc.num_accepted.float().mean())
        acc = {"measured_accepted_per_seq": tot / args.acc_seeds, "seeds": args.acc_seeds,
               "drafts": "drawn from p_hat per seed (Philox stream 1)"}

    padded = None
    if args.padded:
        Lmax, Kmax = int(np.max(inp["kv_len"])), int(np.max(np.diff(inp["cu_q"]))) - 1
        wp = W.workload(args.workload, **dict(over, L_dist="fixed", L_fixed=(Lmax,) * w.B,
                                              K_lo=Kmax, K_hi=Kmax, K_fixed=(Kmax,) * w.B))
        inp_p = W.make_inputs(wp)
        inp_p["seq_ids"] = inp_p["seq_ids"] + lo
        sets_p = [StepBuffers(inp_p, api) for _ in range(args.sets)]
        if not args.gumbel_drafts:
            for d in sets_p:
                draw_drafts_on_device(torch, api, d, inp_p)
        for k in range(3):
            step(sets_p[k % len(sets_p)])
        ms_p, n_p, _ = timed_replays(torch, sets_p, step, args.steps, stream, dist, shard,
                                     args.no_graph, False)
        bytes_p = W.padded_step_bytes(inp)["total"]
        padded = {"ms_per_step": ms_p / n_p, "steps": n_p, "step_bytes": bytes_p,
                  "padding_free_ms_per_step": per_step_ms,
                  "padding_free_step_bytes": step_total,
                  "time_ratio": (ms_p / n_p) / per_step_ms, "bytes_ratio": bytes_p / step_total,
                  "how": f"the same shapes with every cache at the longest ({Lmax}) and every "
                         f"block at the largest K ({Kmax}); the fused step timed on it"}
        del sets_p

    cpu = cpu_all = oracle_agree = ties = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp_o = dict(inp)
        drafts_tied = set()
        if not args.gumbel_drafts:
            inp_o["draft_tokens"], drafts_tied = oracle_drafts(inp)
        oracle_agree, ties = oracle_check(inp_o, inp["draft_tokens"], drafts_tied,
                                          sets[0].num_accepted.cpu().numpy(),
                                          sets[0].out_tokens.cpu().numpy())
        if acc is not None:
            acc["closed_form_accepted_per_seq"] = acceptance_closed_form(inp_o)
        cpu = cpu_baseline(inp_o)
        cpu_all = cpu_baseline_all_cores(sys.argv[1:])

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n_steps,
            "warmup": max(args.warmup, 3), "ms_per_step": per_step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": compute_dtype(w),
            "data": "synthetic (seeded; random-init tensors of the workload's shapes)",
            "config": {"workload": workload_desc(w), "parallelism": f"dp{world} (sequence shards)",
                       "global_batch": world * w.B,
                       "l2": f"inputs larger than L2: {len(sets)} rotating input sets of "
                             f"{step_total / 1e6:.0f} MB per step",
                       "launch": "CUDA graph of the C-ABI call per input set" if not args.no_graph
                       else "direct launches"},
            "accepted_tok_s": emitted_all * n_steps / (ms_step / 1e3),
            "step_time_percentiles": pct,
            "mean_accepted_per_seq": float(np.mean(n_acc)),
            "step_bytes": step_total,
            "step_hbm_gbs": step_total / (per_step_ms * 1e-3) / 1e9,
            "step_frac_of_peak": step_total / (per_step_ms * 1e-3) / 1e9 / peak,
            "roofline": {"kernel": "attention (split-KV, stream-K)", "bound": "hbm",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                         "traffic": traffic, "algorithmic_bytes_per_launch": nbytes["attention"],
                         "avg_launch_us": attn_us, "kernel_src": sha},
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "e2e": e2e,
            "e2e_serial": e2e_serial,
            "gpu_launches": kernels_per_step(w) * n_steps,
            "clocks": clocks,
            "drafts": "Gumbel-max stand-in" if args.gumbel_drafts else
                      "drawn from p_hat on the device (spec_draft_sample, Philox stream 1)",
            "acceptance": acc,
            "oracle_check": oracle_agree,
            "ties": ties,
            "padded": padded,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
