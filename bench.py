#!/usr/bin/env python
"""Throughput of the speculative-tree hot path: verified trees/s and logit GB/s.

One step = spec_tree_build (support selection + dual-identity expansion of
every draft row, then top-R ranking) + spec_tree_verify over one batch of
trees whose draft and target logits are resident in HBM.  Prints one JSON
line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs one process per GPU under torchrun: each rank owns its own batch of
trees (weak scaling); the only collectives are the barrier around the timed
region and the max over ranks of its duration.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified trees/sec and logit GB/s (fraction of GB300 HBM peak) at 128K vocab"
DENSE = 0x40000000  # support = the whole vocabulary
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_b64")
    ap.add_argument("--batch", type=int, default=None, help="override trees per GPU (also of --sweep lines)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="one JSON line per configuration: the workloads, the batch sweep with both builders, "
                         "the wide supports (single GPU; not the contract line)")
    ap.add_argument("--only", default=None,
                    help="--sweep: configurations whose name contains one of these comma-separated texts")
    return ap.parse_args()


def workload(args):
    from dynamic_tree_speculative_gb300 import workloads as WL
    wl = WL.BENCH_WORKLOAD if args.workload == "llama3_b64" else WL.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.with_(B=args.batch)
    return wl


def describe(wl) -> str:
    return (f"{wl.name}: V={wl.V} {wl.dtype} logits, {wl.B} trees per GPU, K={wl.K}, m={wl.m}, W={wl.W}, "
            f"depth {wl.depth}, R={wl.R}, T={wl.temperature}, builder {wl.builder}, top-{wl.support} support")


def config_of(wl, n_gpus):
    return {"workload": describe(wl), "trees_per_gpu": wl.B, "global_batch": wl.B * n_gpus, "vocab": wl.V,
            "K": wl.K, "m": wl.m, "W": wl.W, "depth": wl.depth, "R": wl.R, "temperature": wl.temperature,
            "builder": wl.builder, "support": wl.support, "zipf_a": wl.zipf_a, "sigma_draft": wl.sigma_draft,
            "parallelism": f"trees sharded over {n_gpus} GPU(s), no collective on the data path",
            "l2": "inputs larger than L2: every step streams all draft rows and the accepted target rows"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks ---

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the GPU works."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, window=None):
        """Summary of the samples; `window` = (t0, t1) host times keeps those taken inside it."""
        if self.proc is None:
            return {"error": "nvidia-smi unavailable"}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"error": "no samples"}
        where = "warm-up + timed steps"
        if window is not None:
            inside = []
            for r in rows:
                try:
                    ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + r[0].split(".")[1]) if "." in r[0] else 0.0
                except Exception:
                    continue
                if window[0] - 0.01 <= ts <= window[1] + 0.01:
                    inside.append(r)
            if inside:
                rows, where = inside, "timed steps"
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[6 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "interval_ms": 20,
                "window": where}


# ------------------------------------------------------------ CPU oracle ---

def oracle_trees(wl, seed, tree_ids, budget_s, warm=0):
    """Build + verify trees of the workload through the float64 oracle; returns (trees, seconds)."""
    import numpy as np
    import torch
    from dynamic_tree_speculative_gb300 import workloads as WL
    from oracle import spec_tree_oracle as O
    op = O.Params(K=wl.K, m=wl.m, W=wl.W, depth=wl.depth, R=wl.R, temperature=wl.temperature,
                  support=wl.support, builder=wl.builder, lam=wl.lam, beta=wl.beta, gamma=wl.gamma,
                  delta=wl.delta, rho=wl.rho, eta=wl.eta, alpha=wl.alpha)
    n_rows = wl.n_exp
    u_probe = WL.build_uniforms(wl, seed, n_rows)
    uv, ub = WL.verify_uniforms(wl, seed)
    done, spent = 0, 0.0
    for i, b in enumerate(tree_ids):
        draft, latent = WL.draft_logits(wl, seed, n_rows=n_rows, trees=[b])
        rows = WL.to_numpy_f64(draft[0])
        t0 = time.perf_counter()
        tree = O.build(rows, u_probe[b].numpy().astype(np.float64), op)
        t1 = time.perf_counter()
        exp_row = torch.full((1, wl.R + 1), -1, dtype=torch.int32)
        exp_row[0, :tree.n_nodes] = torch.from_numpy(tree.exp_row.astype(np.int32))
        target = WL.to_numpy_f64(WL.target_logits(wl, seed, latent, exp_row, trees=[b])[0])
        t2 = time.perf_counter()
        O.verify(tree, target, uv[b].numpy(), float(ub[b]), op)
        t3 = time.perf_counter()
        if i >= warm:
            done += 1
            spent += (t1 - t0) + (t3 - t2)
        if budget_s is not None and spent >= budget_s:
            break
    return done, spent


def _oracle_tree_job(job):
    """One tree of the workload through the oracle (build + verify), in a worker process; returns the
    seconds spent in the oracle (input generation excluded)."""
    wl, seed, b = job
    done, spent = oracle_trees(wl, seed, [b], None)
    return spent


def _worker_init():
    os.environ["OMP_NUM_THREADS"] = "1"
    os.environ["OPENBLAS_NUM_THREADS"] = "1"


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


class OraclePool:
    """The oracle, unchanged, on every host core: one process per core (spawned, so that a process
    that already holds a CUDA context can start it), one tree per process and round."""

    def __init__(self, cores=None):
        import multiprocessing as mp
        self.cores = cores or os.cpu_count() or 1
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS")}
        os.environ["OMP_NUM_THREADS"] = os.environ["OPENBLAS_NUM_THREADS"] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_worker_init)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def round(self, wl, seed, tree_ids):
        """Build + verify `tree_ids` concurrently; returns the round's time (the slowest process)."""
        spent = self.pool.map(_oracle_tree_job, [(wl, seed, b) for b in tree_ids], chunksize=1)
        return max(spent)

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_all_cores(wl, seed, rounds, warm=1, pool=None):
    """Trees/s of the oracle on every host core: `rounds` rounds of one tree per core."""
    own = pool is None
    pool = pool or OraclePool()
    try:
        k = 0
        for _ in range(warm):
            pool.round(wl, seed, [(k + i) % wl.B for i in range(pool.cores)])
            k += pool.cores
        done, spent = 0, 0.0
        for _ in range(rounds):
            spent += pool.round(wl, seed, [(k + i) % wl.B for i in range(pool.cores)])
            k += pool.cores
            done += pool.cores
        return done, spent, pool.cores
    finally:
        if own:
            pool.close()


def run_reference(args):
    """The CPU oracle, as it stands, on every host core: each step one tree per core, concurrently."""
    from dynamic_tree_speculative_gb300 import ranks as R
    info = R.rank_info()
    if not info.is_root:
        return 0
    wl = workload(args)
    done, spent, cores = oracle_all_cores(wl, args.seed, args.steps, warm=args.warmup)
    value = done / spent
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "trees/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spent / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl, args.gpus),
            "cpu_baseline": {"value": value, "unit": "trees/s", "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"each step one tree of the workload per host core, build + verify, "
                                       f"{cores} processes ({done} trees timed)"},
            "e2e": {"value": value, "unit": "trees/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- our arm ---

def select_expand_traffic(V):
    """DRAM bytes per select_expand launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "select_expand_traffic.json")
    src = os.path.join(ROOT, "dynamic_tree_speculative_gb300", "csrc", "select_expand.cu")
    try:
        with open(path) as f:
            d = json.load(f)
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if d.get("source_sha256") != h:
            return None
        return d
    except Exception:
        return None


def run_ours(args):
    import torch
    from dynamic_tree_speculative_gb300 import binding as B
    from dynamic_tree_speculative_gb300 import ranks as R
    from dynamic_tree_speculative_gb300 import workloads as WL

    info = R.rank_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device(f"cuda:{info.local_rank}")
    torch.cuda.set_device(dev)
    R.init(info, "nccl")
    wl = workload(args)
    seed = R.rank_seed(args.seed, info.rank)
    params = B.Params.from_workload(wl)
    cparams = params.c()
    n_rows = B.rows_needed(params)
    V = wl.V

    draft, latent = WL.draft_logits(wl, seed, n_rows=n_rows, device=dev)
    u_probe = WL.build_uniforms(wl, seed, n_rows, device=dev)
    uv, ub = WL.verify_uniforms(wl, seed, device=dev)
    tree = B.TreeBuffers(params, wl.B, device=dev)
    out = B.VerifyOutputs(params, wl.B, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.spec_tree_build(cparams, V, draft, u_probe, tree, status)
    torch.cuda.synchronize()
    target = WL.target_logits(wl, seed, latent, tree.node_exp_row, device=dev)
    del latent
    torch.cuda.empty_cache()
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        B.spec_tree_select_expand(cparams, V, draft, u_probe, tree, status, stream)
        if ev is not None:
            ev[1].record(stream)
        B.spec_tree_rank(cparams, V, tree, status, stream)
        B.spec_tree_verify(cparams, V, target, tree, uv, ub, out.accept_len, out.out_tok, out.out_node, None,
                           status, stream)

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else info.local_rank)
    clocks.start()
    for _ in range(args.warmup):
        step()
    K = args.steps
    # the headline: K steps with no event between them (the three launches of a step chain as they
    # would in a serving loop)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    R.barrier(info, dev)
    torch.cuda.synchronize()
    host_t0 = time.time()
    t_start.record(stream)
    for k in range(K):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    host_t1 = time.time()
    R.barrier(info, dev)
    clk = clocks.stop((host_t0, host_t1))
    elapsed = t_start.elapsed_time(t_end) / 1e3
    # the dominant kernel's launch time: the same steps again with events around select_expand
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    for k in range(K):
        step(evs[k])
    torch.cuda.synchronize()
    k1_s = statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3
    st = int(status.item())

    acc = out.accept_len.cpu()
    trees_rate = R.whole_job_rate(wl.B * K, elapsed, info, dev)
    slowest = R.max_over_ranks(elapsed, info, dev)
    S = min(wl.support, V)
    es = 2 if wl.dtype == "bf16" else 4
    draft_bytes = wl.B * n_rows * V * es
    sup_bytes = wl.B * n_rows * (S * 12 + 12)
    target_bytes = int((acc.long() + 1).sum()) * V * es
    step_bytes = draft_bytes + sup_bytes + target_bytes
    logit_gbs = R.sum_over_ranks(step_bytes * K, info, dev) / slowest / 1e9
    hbm, peak_kind = peaks()
    k1_bytes = draft_bytes + sup_bytes + wl.B * n_rows * 4
    achieved = k1_bytes / k1_s / 1e9
    trf = select_expand_traffic(V)

    result = {
        "metric": METRIC, "value": trees_rate, "unit": "trees/s", "n_gpus": info.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": 1e3 * slowest / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic", "config": config_of(wl, info.world),
        "logit_gbs": logit_gbs, "logit_frac_of_peak": logit_gbs / (hbm * info.world),
        "peak_kind": peak_kind, "status": st,
        "accept_len_mean": float(acc.float().mean()),
        "roofline": {"kernel": "select_expand", "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "traffic": None if trf is None else trf["dram_bytes_per_launch_scaled"],
                     "algorithmic_bytes_per_launch": k1_bytes, "avg_launch_ms": 1e3 * k1_s},
        "gpu_launches": 3 * K, "clocks": clk,
    }

    if info.is_root and info.world == 1 and not args.no_cpu_baseline:
        done1, spent1 = oracle_trees(wl, seed, list(range(wl.B)), args.cpu_seconds / 2)
        pool = OraclePool()
        rounds = max(1, int(args.cpu_seconds / 2 / max(spent1 / done1, 1e-3)))
        done, spent, cores = oracle_all_cores(wl, seed, rounds, warm=1, pool=pool)
        pool.close()
        result["cpu_baseline"] = {
            "value": done / spent, "unit": "trees/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{done} trees of this workload (build + verify), float64 numpy, {cores} processes "
                      f"(one per host core, one tree each per round, {rounds} rounds)",
            "single_thread": {"value": done1 / spent1, "unit": "trees/s", "cores": 1,
                              "sample": f"{done1} trees of this workload, one thread"}}

    if not args.no_e2e:
        result["e2e"] = e2e(args, wl, cparams, draft, target, u_probe, uv, ub, tree, out, status, info, dev, K)
    if info.is_root:
        print(json.dumps(result), flush=True)
    if info.world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def e2e(args, wl, cparams, draft, target, u_probe, uv, ub, tree, out, status, info, dev, K):
    """Same metric through the public API with inputs in pinned host memory and results read back."""
    import torch
    from dynamic_tree_speculative_gb300 import binding as B
    from dynamic_tree_speculative_gb300 import ranks as R
    # inputs copied to HBM every step; the target logits stay in pinned host memory and verify reads
    # only the accepted path's rows from there (unified addressing over NVLink-C2C)
    hosts = [x.cpu().pin_memory() for x in (draft, u_probe, uv, ub)]
    devs = [draft, u_probe, uv, ub]
    target_h = target.cpu().pin_memory()
    res_h = [torch.empty(out.accept_len.shape, dtype=torch.int32).pin_memory(),
             torch.empty(out.out_tok.shape, dtype=torch.int32).pin_memory()]
    stream = torch.cuda.current_stream()
    V = wl.V

    def step():
        for d, h in zip(devs, hosts):
            d.copy_(h, non_blocking=True)
        B.spec_tree_build(cparams, V, draft, u_probe, tree, status, stream)
        B.spec_tree_verify(cparams, V, target_h, tree, uv, ub, out.accept_len, out.out_tok, out.out_node, None,
                           status, stream)
        res_h[0].copy_(out.accept_len, non_blocking=True)
        res_h[1].copy_(out.out_tok, non_blocking=True)

    for _ in range(min(args.warmup, 2)):
        step()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    R.barrier(info, dev)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(K):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    R.barrier(info, dev)
    el = R.max_over_ranks(a.elapsed_time(b) / 1e3, info, dev)
    acc = res_h[0].long()
    target_read = int((acc + 1).sum()) * target_h.shape[-1] * target_h.element_size()
    h2d = sum(h.numel() * h.element_size() for h in hosts) + target_read
    d2h = sum(h.numel() * h.element_size() for h in res_h)
    return {"value": R.sum_over_ranks(wl.B * K, info, dev) / el, "unit": "trees/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "target_rows_read_from_host_bytes": target_read,
            "path": "draft logits and uniforms copied pinned host -> HBM, spec_tree_build, spec_tree_verify "
                    "reading the accepted path's target rows from pinned host memory, results -> host"}


def sweep_configs():
    from dynamic_tree_speculative_gb300 import workloads as WL
    base = WL.WORKLOADS["sweep_smart"]
    cfgs = [WL.WORKLOADS["vicuna"], WL.WORKLOADS["llama3"], WL.WORKLOADS["rl"]]
    for builder in ("topr", "smart"):
        for b in (1, 2, 4, 8, 16, 32, 64, 128, 256):
            cfgs.append(base.with_(name=f"sweep_{builder}_b{b}", B=b, builder=builder))
    for sup in (256, 512, 1024):
        cfgs.append(WL.BENCH_WORKLOAD.with_(name=f"llama3_b64_support{sup}", support=sup))
    # the dense support (|S| = V)
    cfgs.append(WL.BENCH_WORKLOAD.with_(name="llama3_b64_dense", support=DENSE))
    cfgs.append(WL.BENCH_WORKLOAD.with_(name="llama3_b8_dense", B=8, support=DENSE))
    return cfgs


def run_sweep(args):
    """Build + verify throughput per configuration, inputs resident in HBM, CUDA-event timed."""
    import torch
    from dynamic_tree_speculative_gb300 import binding as B
    from dynamic_tree_speculative_gb300 import workloads as WL
    dev = torch.device("cuda")
    hbm, peak_kind = peaks()
    steps = min(args.steps, 200)
    only = [x for x in args.only.split(",") if x] if args.only else None

    def wanted(name: str) -> bool:
        return only is None or any(x in name for x in only)

    for wl in sweep_configs():
        if not wanted(wl.name):
            continue
        if args.batch:
            wl = wl.with_(B=args.batch)
        params = B.Params.from_workload(wl)
        cp = params.c()
        n_rows = B.rows_needed(params)
        draft, latent = WL.draft_logits(wl, args.seed, n_rows=n_rows, device=dev)
        u_probe = WL.build_uniforms(wl, args.seed, n_rows, device=dev)
        uv, ub = WL.verify_uniforms(wl, args.seed, device=dev)
        tree = B.TreeBuffers(params, wl.B, device=dev, V=wl.V)
        out = B.VerifyOutputs(params, wl.B, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        B.spec_tree_build(cp, wl.V, draft, u_probe, tree, status)
        torch.cuda.synchronize()
        target = WL.target_logits(wl, args.seed, latent, tree.node_exp_row, device=dev)
        del latent
        stream = torch.cuda.current_stream()
        dense = B.is_dense(params, wl.V)

        def step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            B.spec_tree_select_expand(cp, wl.V, draft, u_probe, tree, status, stream)
            if ev is not None:
                ev[1].record(stream)
            B.spec_tree_rank(cp, wl.V, tree, status, stream)
            if dense:
                B.spec_tree_verify_dense(cp, wl.V, target, draft, tree, uv, ub, out.accept_len, out.out_tok,
                                         out.out_node, None, status, stream)
            else:
                B.spec_tree_verify(cp, wl.V, target, tree, uv, ub, out.accept_len, out.out_tok, out.out_node, None,
                                   status, stream)

        for _ in range(max(args.warmup, 3)):
            step()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for k in range(steps):
            step(evs[k])
        b.record(stream)
        torch.cuda.synchronize()
        el = a.elapsed_time(b) / 1e3
        sel_s = statistics.mean(x.elapsed_time(y) for x, y in evs) / 1e3
        acc = out.accept_len.cpu()
        es = 2 if wl.dtype == "bf16" else 4
        S = min(wl.support, wl.V)
        if dense:
            S = wl.K + 1  # ranks 0..K-1 and the probe are written
        draft_bytes = wl.B * n_rows * wl.V * es
        sup_bytes = wl.B * n_rows * (S * 12 + 12)
        step_bytes = draft_bytes + sup_bytes + int((acc.long() + 1).sum()) * wl.V * es
        sel_bytes = draft_bytes + sup_bytes + wl.B * n_rows * 4
        line = {"sweep": wl.name, "config": config_of(wl, 1), "trees_per_s": wl.B * steps / el,
                "ms_per_step": 1e3 * el / steps, "logit_gbs": step_bytes * steps / el / 1e9,
                "logit_frac_of_peak": step_bytes * steps / el / 1e9 / hbm,
                "select_expand_ms": 1e3 * sel_s, "select_expand_frac": sel_bytes / sel_s / 1e9 / hbm,
                "peak_gbs": hbm, "peak_kind": peak_kind, "accept_len_mean": float(acc.float().mean()),
                "tree_nodes_mean": float((tree.n_nodes.cpu().float() - 1).mean()), "status": int(status.item()),
                "steps": steps}
        print(json.dumps(line), flush=True)
        del draft, target, tree, out
        torch.cuda.empty_cache()
    for b in (8, 64):
        if not wanted(f"layer_mode_b{b}"):
            continue
        print(json.dumps(sweep_layer_mode(WL.BENCH_WORKLOAD.with_(name=f"layer_mode_b{b}", B=b), args)), flush=True)
    return 0


def sweep_layer_mode(wl, args):
    """The layer-by-layer build (one spec_tree_layer call per layer, then spec_tree_finish) against the
    one-shot spec_tree_build on the same draft rows; each layer's rows are a slice of the same tensor."""
    import torch
    from dynamic_tree_speculative_gb300 import binding as B
    from dynamic_tree_speculative_gb300 import workloads as WL
    dev = torch.device("cuda")
    params = B.Params.from_workload(wl)
    cp = params.c()
    n_rows = B.rows_needed(params)
    draft, _ = WL.draft_logits(wl, args.seed, n_rows=n_rows, device=dev)
    u_probe = WL.build_uniforms(wl, args.seed, n_rows, device=dev)
    tree = B.TreeBuffers(params, wl.B, device=dev)
    state = B.LayerState(params, wl.B, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    layers = []
    for layer in range(wl.depth):
        rows = B.spec_tree_layer_rows(params, layer)
        r0 = 0 if layer == 0 else 1 + (layer - 1) * wl.W
        layers.append((layer, draft[:, r0:r0 + rows].contiguous(), u_probe[:, r0:r0 + rows].contiguous()))

    def one_shot():
        B.spec_tree_build(cp, wl.V, draft, u_probe, tree, status)

    def layered():
        for layer, d, u in layers:
            B.spec_tree_layer(cp, wl.V, layer, d, u, tree, state, status)
        B.spec_tree_finish(cp, wl.V, tree, state, status)

    res = {}
    for name, fn in (("one_shot_build_us", one_shot), ("layer_by_layer_build_us", layered)):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(20):
            fn()
        b.record()
        torch.cuda.synchronize()
        res[name] = a.elapsed_time(b) / 20 * 1e3
    return {"sweep": wl.name, "config": config_of(wl, 1), **res, "layer_calls": wl.depth + 1,
            "status": int(status.item())}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
