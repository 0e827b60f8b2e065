"""Benchmark of the CSA decode hot path at 1M-token context on B300.

One step = one decode step of a batch of 4 sequences with 2^20 cached tokens
each (262144 compressed entries, m = 4): append one token per sequence
(softmax-gated pooling + window ring), lightning-indexer scores over every
entry (64 heads x 128 dims, e4m3 keys), top-2048 selection, and sparse
shared-KV attention (64 heads x 512 dims, e4m3 + bf16 rope entries) over the
selected entries, the 128-token window and the sink.  Metric: decode
queries/s (one query per sequence per step) plus the HBM roofline of the
dominant kernel (the indexer).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

--impl reference times the CPU oracle (plain fp64 numpy, single thread) on a
bounded sample of the same workload; under torchrun only rank 0 does that.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = ("csa_decode_1m", "hca_decode_128k", "stack_decode_paged", "csa_prefill_8k")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6400.0, 1800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in (self.out or "").splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _workload(name, steps_total):
    from long_context_attention_05_b300 import synthetic as S
    extra = steps_total // 4 + 16
    if name == "csa_decode_1m":
        return [S.config2(extra_entries=extra)]
    if name == "hca_decode_128k":
        return [S.config1(extra_entries=extra)]
    if name == "stack_decode_paged":
        return S.config4_layers(extra_entries=extra)
    if name == "csa_prefill_8k":
        return [S.config3()]
    raise SystemExit(f"unknown workload {name}")


def _alg_bytes(w):
    """Algorithmic HBM bytes of one step: (indexer bytes, whole-step bytes)."""
    n_e = np.asarray(w.n_entries, dtype=np.int64)
    B, nq = w.batch, w.n_new
    entry = (w.d - w.d_rope) + 2 * w.d_rope + 4 if w.kv_dtype == "e4m3" else 4 * w.d
    tok = 2 if w.tok_dtype == "bf16" else 4
    q_bytes = B * nq * w.heads * w.d * tok
    out_bytes = B * nq * w.heads * (w.d * tok + 4)
    new_tok = B * nq * 2 * (w.d + w.d_idx) * tok
    win = B * nq * w.n_win * w.d * tok
    if w.kind == "csa":
        key = w.d_idx + 4 if w.kv_dtype == "e4m3" else 4 * w.d_idx
        idx_bytes = int(n_e.sum()) * nq * key + B * nq * w.heads_idx * (w.d_idx * tok + 4)
        att = B * nq * w.k * entry
    else:
        idx_bytes = 0
        att = int(n_e.sum()) * nq * entry
    return idx_bytes, idx_bytes + att + q_bytes + out_bytes + new_tok + win


def _oracle_rows_inproc(workload, budget_s, n_layers, steps=1, warmup=0):
    """Times the oracle on whole query rows (one sequence's query at a time):
    `warmup` untimed rows, then `steps` sample steps of at least one row each,
    together about budget_s seconds.  Inputs are generated once."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import harness as H
    from long_context_attention_05_b300 import synthetic as S
    wl = _workload(workload, 0)[:n_layers]
    data = []
    for w in wl:
        inp = S.step_inputs(w)
        arrs = S.seeded_cache(w, inp.get("q_idx"), inp.get("w_idx"))
        rows = [(b, 0) for b in range(w.batch)] if w.mode == "decode" else [(0, i) for i in range(w.n_new)]
        data.append((w, inp, arrs, rows))
    order = [(li, r) for r in range(max(len(d[3]) for d in data)) for li in range(len(data)) if r < len(data[li][3])]
    pos = 0

    def one_row():
        nonlocal pos
        li, r = order[pos % len(order)]
        pos += 1
        w, inp, arrs, rows = data[li]
        b, i = rows[r]
        t0 = time.perf_counter()
        H.oracle_seeded_step(w, arrs, inp, b, i)
        return time.perf_counter() - t0

    for _ in range(warmup):
        one_row()
    per_step = budget_s / max(steps, 1)
    n_rows, t_total = 0, 0.0
    for _ in range(steps):
        t_step = 0.0
        while True:
            t_step += one_row()
            n_rows += 1
            if t_step >= per_step:
                break
        t_total += t_step
    return n_rows, t_total


def _oracle_rows(workload, budget_s, n_layers=1, steps=1, warmup=0):
    """Runs the oracle sample in a fresh single-threaded process (BLAS and OpenMP
    pinned to one thread; spawned, never forked from a CUDA process)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", workload, str(budget_s),
                        str(n_layers), str(steps), str(warmup)], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed:\n" + r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["rows"], d["seconds"]


def run_reference(args):
    wl = _workload(args.workload, 0)
    n_layers = 2 if args.workload == "stack_decode_paged" else 1
    per_step = args.budget / max(args.steps, 1)
    rows_total, t_total = _oracle_rows(args.workload, args.budget, n_layers, args.steps, args.warmup)
    qps = rows_total / t_total
    if n_layers == 2:   # a query of the stack is one row in each of its 4 layers (2 CSA, 2 HCA)
        qps /= 2.0
    sample = (f"{rows_total} oracle query rows of {wl[0].name} (fp64 numpy, 1 thread, "
              f"{args.steps} steps of >= 1 row and ~{per_step:.2f} s)")
    line = {"metric": "CSA/HCA decode queries/s at 1M ctx; achieved HBM GB/s vs B300 peak", "value": qps,
            "unit": "queries/s", "impl": "reference", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * t_total / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded caches, no weights)",
            "config": {"workload": wl[0].name if n_layers == 1 else args.workload},
            "cpu_baseline": {"value": qps, "unit": "queries/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": qps, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import long_context_attention_05_b300 as L
    from long_context_attention_05_b300 import synthetic as S
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    total_steps = args.steps * 2 + args.warmup + 8
    wl = _workload(args.workload, total_steps)
    nsets = 4
    layers = []
    for li, w in enumerate(wl):
        sets = [S.step_inputs(w, step=s) for s in range(nsets)]
        arrs = S.seeded_cache(w, sets[0].get("q_idx"), sets[0].get("w_idx"))
        cache = L.Cache.from_host(w, arrs, device=dev)
        kv_bytes = S.cache_bytes(arrs)
        del arrs
        dsets = [{k: L.to_device(v, dev) for k, v in s.items()} for s in sets]
        hsets = [{k: torch.from_numpy(np.ascontiguousarray(v.view(np.int16) if v.dtype == np.uint16 else v))
                  .pin_memory() for k, v in s.items()} for s in sets]
        B, nq = w.batch, w.n_new
        ws = L.alloc_workspace(cache, B, nq, w.heads, w.k, device=dev)
        bufs = {"out": torch.empty((B, nq, w.heads, w.d), dtype=torch.bfloat16, device=dev),
                "lse": torch.empty((B, nq, w.heads), dtype=torch.float32, device=dev)}
        if w.kind == "csa":
            bufs["idx"] = torch.empty((B, nq, w.k), dtype=torch.int32, device=dev)
            bufs["cnt"] = torch.empty((B, nq), dtype=torch.int32, device=dev)
            bufs["scores"] = torch.empty((B * nq, cache.entry_cap), dtype=torch.float32, device=dev)
        layers.append(dict(w=w, cache=cache, dsets=dsets, hsets=hsets, ws=ws, bufs=bufs, kv_bytes=kv_bytes))

    stream = torch.cuda.current_stream(dev)
    ev_pairs = []

    def step(s, timed=False):
        for ly in layers:
            w, c, gi, b = ly["w"], ly["cache"], ly["dsets"][s % nsets], ly["bufs"]
            L.csa_compress(c, gi["x"], gi["gate"], gi["pos_bias"], gi.get("idx_x"), gi.get("idx_gate"),
                           gi.get("idx_pos_bias"))
            if w.kind == "csa":
                if timed and ly is layers[0]:
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                L.csa_index_scores(c, gi["q_idx"], gi["w_idx"], b["scores"], ly["ws"])
                if timed and ly is layers[0]:
                    e1.record(stream)
                    ev_pairs.append((e0, e1))
                L.csa_topk(c, b["scores"], w.batch, w.n_new, w.k, b["idx"], b["cnt"], ly["ws"])
                L.csa_sparse_attend(c, gi["q"], gi["sink"], b["idx"], b["out"], b["lse"], ly["ws"])
            else:
                L.hca_attend(c, gi["q"], gi["sink"], b["out"], b["lse"], ly["ws"])

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        t0.record(stream)
        for s in range(args.steps):
            step(args.warmup + s, timed=True)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1)
    idx_ms = float(np.mean([a.elapsed_time(b) for a, b in ev_pairs])) if ev_pairs else None

    # end to end through the public API: pinned host inputs -> device, step, result -> host
    h_out = torch.empty(layers[-1]["bufs"]["out"].shape, dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty(layers[-1]["bufs"]["lse"].shape, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for ly in layers for v in ly["hsets"][0].values())
    d2h = h_out.numel() * 2 + h_lse.numel() * 4
    torch.cuda.synchronize(dev)
    barrier()
    w0 = time.perf_counter()
    for s in range(args.steps):
        k = (args.warmup + args.steps + s) % nsets
        for ly in layers:
            for name, hv in ly["hsets"][k].items():
                dv = ly["dsets"][k][name]
                dv.view(hv.dtype).copy_(hv, non_blocking=True) if dv.dtype == torch.bfloat16 \
                    else dv.copy_(hv, non_blocking=True)
        step(args.warmup + args.steps + s)
        h_out.copy_(layers[-1]["bufs"]["out"], non_blocking=True)
        h_lse.copy_(layers[-1]["bufs"]["lse"], non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - w0
    barrier()

    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([ms, e2e_s], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms, e2e_s = float(tt[0]), float(tt[1])
    w0l = layers[0]["w"]
    queries_per_step = w0l.batch * w0l.n_new
    value = world * queries_per_step * args.steps / (ms / 1000.0)
    e2e = world * queries_per_step * args.steps / e2e_s
    hbm_peak, bf16_peak, peak_kind = _peaks()
    idx_bytes, step_bytes = _alg_bytes(w0l)
    step_bytes_all = sum(_alg_bytes(ly["w"])[1] for ly in layers)
    roofline = None
    if idx_ms:
        ach = idx_bytes / (idx_ms / 1000.0) / 1e9
        roofline = {"bound": "hbm", "kernel": "k_index (lightning indexer scores)", "achieved": round(ach, 1),
                    "peak": hbm_peak, "unit": "GB/s", "frac": round(ach / hbm_peak, 4), "traffic": None,
                    "peak_kind": f"{peak_kind} hbm_gbs", "avg_launch_us": round(idx_ms * 1000, 2),
                    "alg_bytes_per_launch": int(idx_bytes)}
    step_ach = step_bytes_all / (ms / args.steps / 1000.0) / 1e9
    launches_per_step = sum((3 + 2) if ly["w"].kind == "csa" else 3 for ly in layers)
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        nl = 2 if args.workload == "stack_decode_paged" else 1
        n, t = _oracle_rows(args.workload, args.budget, nl)
        qps = n / t / float(nl)
        cpu = {"value": qps, "unit": "queries/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} oracle query rows of {w0l.name} (fp64 numpy, 1 thread), {t:.1f} s"}
    gqa8 = 8 * 128 * 2 * 2
    line = {
        "metric": "CSA/HCA decode queries/s at 1M ctx; achieved HBM GB/s vs B300 peak",
        "value": value, "unit": "queries/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3/bf16 storage, f32 accumulate", "data": "synthetic (seeded caches, no weights)",
        "config": {"workload": w0l.name if len(layers) == 1 else args.workload, "batch_per_gpu": w0l.batch,
                   "ctx_tokens": int(max(w0l.ctx)), "entries_per_seq": int(max(w0l.n_entries)), "m": w0l.m,
                   "heads": w0l.heads, "d": w0l.d, "indexer": f"{w0l.heads_idx}x{w0l.d_idx} e4m3", "top_k": w0l.k,
                   "window": w0l.n_win, "layers": len(layers),
                   "l2": "inputs larger than L2 (cache >> 126 MB)",
                   "kv_bytes_per_token_vs_bf16_gqa8": round(sum(ly["kv_bytes"] for ly in layers) /
                                                            (len(layers) * w0l.batch * max(w0l.ctx)) / gqa8, 4)},
        "roofline": roofline,
        "step_roofline": {"bound": "hbm", "achieved": round(step_ach, 1), "peak": hbm_peak, "unit": "GB/s",
                          "frac": round(step_ach / hbm_peak, 4), "alg_bytes_per_step": int(step_bytes_all)},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e, "unit": "queries/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    if len(sys.argv) > 1 and sys.argv[1] == "--oracle-sample":
        n, t = _oracle_rows_inproc(sys.argv[2], float(sys.argv[3]), int(sys.argv[4]), int(sys.argv[5]),
                                   int(sys.argv[6]))
        print(json.dumps({"rows": n, "seconds": t}))
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default="csa_decode_1m")
    ap.add_argument("--budget", type=float, default=12.0, help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
