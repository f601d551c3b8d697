#!/usr/bin/env python3
"""Benchmark: paged FP8 MLA split-KV decode on one GB300 (or N replicas).

One step = one full decode call (split-KV kernel + merge) over one batch of
synthetic, seeded inputs: H = 12 heads, q = 1, B = 16 requests of 1,048,576
KV tokens each (latent 512 + rope 64 E4M3, page size 32, random page
permutation), the long-context workload of TensorRT-LLM issue #20510.  The
KV cache (9.66 GB) is far larger than L2, so no flush is needed between steps.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 MLA split-KV decode us/call; KV-read HBM GB/s as fraction of GB300 peak"
UNIT = "us/call"
DEFAULT_WORKLOAD = "long_h12_q1_l1m_b16"
# Published time for this exact workload (H12 q1 B16 1M, issue #20510 "Repro 1",
# kernel before #19338, on an unspecified Blackwell SM10x GPU): context only.
PUBLISHED_US = {"long_h12_q1_l1m_b16": 1095.5}
L2_ROTATE_BYTES = 2 * 126 * 1024 * 1024  # rotate inputs below 2x the 126 MB L2
# Sources of the split-KV kernel a workload runs (recorded ncu traffic is
# valid only for the source it was taken on).
_COMMON_SOURCES = ["split_kv_mla_paged_gb300/csrc/mla_device.cuh",
                   "split_kv_mla_paged_gb300/csrc/mla_internal.h",
                   "split_kv_mla_paged_gb300/csrc/sm103_ptx.cuh"]
KERNEL_SOURCES = {
    "e4m3": ["split_kv_mla_paged_gb300/csrc/mla_decode.cu"] + _COMMON_SOURCES,
    "bf16": ["split_kv_mla_paged_gb300/csrc/mla_decode_bf16.cu",
             "split_kv_mla_paged_gb300/csrc/mla_decode.cu"] + _COMMON_SOURCES,
}


def kernel_hash(dtype: str = "e4m3") -> str:
    """Hash of the kernel sources' code (comments and blank lines excluded)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[dtype]:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def algorithmic_flops(lens, H: int, q_len: int, causal: bool, sel=None) -> int:
    """QK over 576 dims and PV over 512 for every visible (row, key) pair:
    2 * 1088 flop each.  A causal MTP row (query token qi of q) sees the
    first L - q + qi + 1 keys; with a page selection, only the selected keys
    among them."""
    pairs = 0
    for b, L in enumerate(lens):
        for qi in range(q_len):
            n_tok = L - q_len + qi + 1 if causal else L
            keys = selected_keys(sel[b], L, n_tok) if sel is not None else min(L, n_tok)
            pairs += H * keys
    return 2 * 1088 * pairs


def recorded_traffic(workload: str):
    """DRAM bytes per split-KV launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "split_kv_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(workload)
    from synth import WORKLOADS
    dtype = WORKLOADS.get(workload, {}).get("dtype", "e4m3")
    if not entry or entry.get("kernel_sha") != kernel_hash(dtype):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank value over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def selected_keys(sel_row, L: int, n_tok: int) -> int:
    """Keys of the selected pages (one request's block_idx row) below n_tok."""
    n = 0
    for p in sel_row:
        p = int(p)
        if p >= 0:
            n += max(0, min(32, min(L, n_tok) - 32 * p))
    return n


def cpu_oracle_sample(inp, w, rows_per_sample: int, softmax_scale: float, tokens: int = 0,
                      selection=None):
    """Time the oracle on the first `rows_per_sample` rows, each over its first
    `tokens` keys (0 = the full KV length; with a page selection `selection`
    [B, topk], only the selected keys among them).  Returns (seconds, row-keys
    done, threads); the work per (row, key) is uniform, so time scales by
    row-keys."""
    import numpy as np
    import torch
    import oracle
    H, q_len = inp.num_heads, inp.q_len
    per_req = H * q_len
    n_req = max(1, -(-rows_per_sample // per_req))
    rows = np.arange(min(rows_per_sample, inp.rows), dtype=np.int64)
    # Host copies of only the sampled requests' pages (prepared outside the timing).
    batches = []
    for b in range(n_req):
        L = int(inp.kv_lens[b])
        n_tok = L if tokens <= 0 else min(L, tokens)
        n_pages = (n_tok + 31) // 32
        pages = inp.page_table[b, :n_pages].to(torch.int64).to(inp.kv.device)
        kv_b = inp.kv[pages].cpu().numpy()
        q_b = inp.q[b:b + 1].cpu().numpy()
        table = np.arange(n_pages, dtype=np.int32)[None, :]
        sel = rows[(rows // per_req) == b] - b * per_req
        # Causal rows see up to L - q_len + qi + 1 keys; the sample keeps the
        # first n_tok of them (all visible when n_tok <= L - q_len + 1).
        batches.append((q_b, kv_b, table, np.array([L], dtype=np.int32), sel, n_tok))
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    done = 0
    for b, (q_b, kv_b, table, lens, rsel, n_tok) in enumerate(batches):
        blk = None if selection is None else selection[b:b + 1]
        oracle.decode_rows(q_b, kv_b, table, lens, q_len=q_len, num_heads=H, causal=w["causal"],
                           softmax_scale=softmax_scale, rows=rsel, tok_begin=0,
                           tok_end=n_tok if n_tok < int(lens[0]) else -1, block_idx=blk)
        keys = n_tok if selection is None else selected_keys(selection[b], int(lens[0]), n_tok)
        done += len(rsel) * keys
    return time.perf_counter() - t0, done, threads


def run_reference(args, w, world, rank):
    """The oracle, as it stands, on the host cores: each step a bounded sample
    (one row per host thread, over a prefix of the KV range sized so that the
    whole run takes about --ref-budget-s seconds), scaled by row-tokens."""
    import torch
    from synth import SOFTMAX_SCALE, workload_inputs
    import oracle
    if world > 1 and rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if dev == "cpu":
        # Only the sampled request is needed on the host.
        from synth import decode_inputs
        inp = decode_inputs(1, w["num_heads"], w["q_len"], w["kv_lens"][:1], w["seed"])
    else:
        inp = workload_inputs(args.workload, device=dev)
    sel = None
    if w.get("topk"):
        from synth import page_selection
        sel = page_selection(w["kv_lens"], w["topk"], seed=w["seed"] + 100)
        total_row_tokens = (sum(selected_keys(sel[b], int(L), int(L))
                                for b, L in enumerate(w["kv_lens"]))
                            * w["num_heads"] * w["q_len"])
    else:
        total_row_tokens = sum(int(L) for L in w["kv_lens"]) * w["num_heads"] * w["q_len"]
    threads = oracle.max_threads()
    rows = min(threads, w["num_heads"] * w["q_len"])
    L0 = int(w["kv_lens"][0])
    cal_tokens = min(L0, 16384)
    t_cal, _, _ = cpu_oracle_sample(inp, w, rows, SOFTMAX_SCALE, tokens=cal_tokens,
                                    selection=sel)
    per_step = args.ref_budget_s / (args.steps + args.warmup)
    tokens = int(max(1024, min(L0, cal_tokens * per_step / max(t_cal, 1e-6))))
    times = []
    for k in range(args.warmup + args.steps):
        t, done, threads = cpu_oracle_sample(inp, w, rows, SOFTMAX_SCALE, tokens=tokens,
                                             selection=sel)
        if k >= args.warmup:
            times.append(t / done * total_row_tokens * 1e6)
    value = statistics.mean(times)
    sample = (f"{rows} rows of request 0 over their first {tokens} of {L0} keys per step"
              f"{' (selected pages only)' if sel is not None else ''}; "
              f"time scaled by row-keys to the whole call")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": ("synthetic (seeded N(0,0.5^2) cast to "
                 f"{'BF16' if w.get('dtype') == 'bf16' else 'E4M3'})"),
        "config": {"workload": args.workload, "batch": w["batch"], "num_heads": w["num_heads"],
                   "q_len": w["q_len"], "kv_len": w["kv_lens"][0], "causal": w["causal"],
                   "parallelism": "replicas" if world > 1 else "single"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def kv_append_bench(args):
    """The FP8 paged KV append (quantise BF16 latent rows, scatter through the
    page table): 16 requests x 8 new tokens (an MTP decode step) and 16 x 65,536
    (a prefill chunk), positions in random pages of a larger pool, with a
    power-of-two kv_scale (1.0) and a calibrated-looking one (0.37).
    Algorithmic bytes per row: 1152 read + 576 written + 8 of indices.  Prints
    one JSON line with every case against the measured copy bandwidth."""
    import numpy as np
    import torch
    import split_kv_mla_paged_gb300 as mla
    from split_kv_mla_paged_gb300 import build as mla_build
    mla_build.build()
    mla.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    peaks = measured_peaks()
    K = max(10, min(args.steps, 100))
    cases = []
    for (name, per_req), kv_scale in itertools.product(
            (("mtp_step_b16_q8", 8), ("prefill_b16_64k", 65536)), (1.0, 0.37)):
        B = 16
        n = B * per_req
        pages_per_req = (per_req + 31) // 32 + 1
        n_pages = B * pages_per_req * 2
        g = torch.Generator(device="cpu").manual_seed(7)
        table = torch.randperm(n_pages, generator=g)[:B * pages_per_req].reshape(
            B, pages_per_req).to(torch.int32)
        start = torch.randint(0, 32, (B,), generator=g)
        req = torch.arange(B, dtype=torch.int32).repeat_interleave(per_req)
        pos = (start.repeat_interleave(per_req) + torch.arange(per_req).repeat(B)).to(torch.int32)
        rows = (torch.randn(n, 576, generator=g) * 0.5).to(torch.bfloat16)
        kv = torch.zeros((n_pages, 32, 576), dtype=torch.uint8, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        args_d = (rows.to(dev), n, req.to(dev), pos.to(dev), table.to(dev), pages_per_req, B,
                  kv, n_pages, kv_scale, st)
        with torch.cuda.stream(stream):
            mla.mla_kv_append(*args_d, stream=stream)
        torch.cuda.synchronize(dev)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for _ in range(K):
                mla.mla_kv_append(*args_d)
        with torch.cuda.stream(stream):
            gr.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / K
        assert int(st.item()) == 0
        nbytes = n * (1152 + 576 + 8)
        gbs = nbytes / (us * 1e-6) / 1e9
        cases.append({"case": name, "kv_scale": kv_scale, "rows": n, "us": us, "bytes": nbytes, "gbs": gbs,
                      "frac": gbs / peaks["hbm_gbs"]})
        del gr
    line = {"metric": "FP8 paged KV append us/call", "unit": "us/call", "n_gpus": 1, "steps": K,
            "higher_is_better": False, "dtype": "bf16->e4m3", "data": "synthetic",
            "peak_gbs": peaks["hbm_gbs"], "cases": cases}
    print(json.dumps(line), flush=True)


def merge_sweep(args):
    """The merge alone on seeded partials: rows = B*q*H in {12 .. 192}, splits
    {6 .. 128}, KvSplit {1 .. 16} (10 % empty slots), CUDA graphs of K calls
    per point, rotating over partial sets larger than 2x L2 in total.  Prints
    one JSON line: the per-point times, the partial bytes read per call and the
    graph floor of a one-element kernel."""
    import numpy as np
    import torch
    import split_kv_mla_paged_gb300 as mla
    from split_kv_mla_paged_gb300 import build as mla_build
    from synth import merge_partials
    mla_build.build()
    mla.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    K = max(10, min(args.steps, 200))
    tiny = torch.zeros(1, device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(K):
            tiny.add_(1.0)

    def time_graph(graph):
        with torch.cuda.stream(stream):
            graph.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / K

    floor = time_graph(g)
    points = []
    # rows = B*q*H of the workloads (12 .. 192; 768 = H96 q8 B1), splits of
    # the pages' and the GB300 planner's plans, every KvSplit.
    for rows in (12, 96, 192, 768):
        for S in (6, 12, 19, 25, 50, 100, 128, 152):
            plan_ks = mla.mla_decode_plan([S * 128], 1, 1, sm_count=S).kv_split
            for ks in (1, 2, 4, 8, 16):
                if ks > S:
                    continue
                o, ml = merge_partials(rows, S, seed=rows * 1000 + S)
                part_bytes = o.nbytes + ml.nbytes
                n_sets = max(1, min(16, -(-L2_ROTATE_BYTES // part_bytes)))
                sets = []
                for k in range(n_sets):
                    o_d = torch.from_numpy(np.roll(o, k, axis=0)).to(dev)
                    ml_d = torch.from_numpy(np.roll(ml, k, axis=0)).to(dev)
                    out = torch.empty((rows, 512), dtype=torch.bfloat16, device=dev)
                    lse = torch.empty((rows,), dtype=torch.float32, device=dev)
                    sets.append((o_d, ml_d, out, lse))
                with torch.cuda.stream(stream):
                    mla.mla_merge(*sets[0][:2], rows, S, ks, sets[0][2], sets[0][3], None, stream)
                torch.cuda.synchronize(dev)
                gm = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gm, stream=stream):
                    for k in range(K):
                        o_d, ml_d, out, lse = sets[k % n_sets]
                        mla.mla_merge(o_d, ml_d, rows, S, ks, out, lse, None)
                us = time_graph(gm)
                points.append({"rows": rows, "splits": S, "kv_split": ks, "us": us,
                               "planner_kv_split": plan_ks,
                               "partial_bytes": part_bytes,
                               "gbs": part_bytes / (us * 1e-6) / 1e9})
                del gm, sets
    line = {"metric": "MLA merge us/call (merge-only sweep)", "unit": "us/call", "n_gpus": 1,
            "steps": K, "higher_is_better": False, "dtype": "f32", "data": "synthetic partials",
            "floor_us_per_call": floor, "points": points}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--plan", choices=["gb300", "pages"], default="gb300")
    ap.add_argument("--target", type=int, default=0,
                    help="CTA target of the pages' planner formula (overrides --plan)")
    ap.add_argument("--persistent", type=int, default=0,
                    help="run the plan's CTA item list with this many persistent CTAs (FP8)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--kv-append", action="store_true",
                    help="time the FP8 paged KV append (decode-sized and prefill-sized batches)")
    ap.add_argument("--merge-sweep", action="store_true",
                    help="time the merge alone over the merge-only sweep (rows x splits x KvSplit)")
    ap.add_argument("--replays", type=int, default=10,
                    help="further replays of the K-call graph for p10/median/p90")
    ap.add_argument("--cpu-rows", type=int, default=192,
                    help="rows of the oracle CPU baseline sample (0 disables it)")
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="wall-clock budget of the whole --impl reference run")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from synth import SOFTMAX_SCALE, WORKLOADS, workload_inputs
    w = WORKLOADS[args.workload]
    world, rank, local = dist_env()
    if args.merge_sweep:
        merge_sweep(args)
        return
    if args.kv_append:
        kv_append_bench(args)
        return

    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        run_reference(args, w, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import numpy as np
    import torch
    import split_kv_mla_paged_gb300 as mla
    from split_kv_mla_paged_gb300 import build as mla_build

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(mla_build.LIB_PATH):
        mla_build.build()
    if world > 1:
        dist.barrier()
    mla.load_library()

    inp = workload_inputs(args.workload, device=dev)
    B, H, q_len = inp.batch, inp.num_heads, inp.q_len
    lens = inp.kv_lens.tolist()
    topk = w.get("topk")
    is_sparse = topk is not None
    # A sparse decode is planned over the compact range of its selection.
    plan_lens = [32 * topk] * B if is_sparse else lens
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    if args.target > 0:
        plan = mla.mla_decode_plan(plan_lens, H, q_len, sm_count=sm_count,
                                   target_ctas=args.target)
    elif args.plan == "pages" and w["target"] is not None:
        plan = mla.mla_decode_plan(plan_lens, H, q_len, target_ctas=w["target"])
    else:
        plan = mla.mla_decode_plan(plan_lens, H, q_len, sm_count=sm_count)
    ws_bytes = mla.mla_decode_workspace_size(B, q_len, H, plan.max_splits)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    splits_d = torch.from_numpy(plan.splits).to(dev)
    chunks_d = torch.from_numpy(plan.chunks).to(dev)
    # Inputs larger than L2 need no flush.  Smaller ones rotate over enough
    # distinct seeded pools (with their own workspaces and outputs) that
    # consecutive steps never find their KV in L2.
    sels = []
    if is_sparse:
        # One KV pool; the steps rotate over distinct page selections of it, so
        # consecutive steps read different pages (L2 is cold for each).
        from synth import page_selection
        sel0 = page_selection(lens, topk, seed=w["seed"] + 100)
        kv_bytes = sum(selected_keys(sel0[b], L, L) for b, L in enumerate(lens)) * 576
        n_pools = 1 if kv_bytes >= L2_ROTATE_BYTES else min(64, -(-L2_ROTATE_BYTES // kv_bytes))
        sels = [torch.from_numpy(sel0).to(dev)] + [
            torch.from_numpy(page_selection(lens, topk, seed=w["seed"] + 100 + k)).to(dev)
            for k in range(1, n_pools)]
        pools = [inp] * n_pools
    else:
        kv_bytes = inp.kv_bytes()
        n_pools = 1 if kv_bytes >= L2_ROTATE_BYTES else min(64, -(-L2_ROTATE_BYTES // kv_bytes))
        pools = [inp] + [workload_inputs(args.workload, device=dev, seed_offset=k)
                         for k in range(1, n_pools)]
    calls = []
    for k, pool in enumerate(pools):
        ws_k = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        mla.mla_decode_workspace_init(ws_k, ws_bytes)
        out_k = torch.empty((B, q_len, H, 512), dtype=torch.bfloat16, device=dev)
        lse_k = torch.empty((B, q_len, H), dtype=torch.float32, device=dev)
        calls.append((pool.q, pool.kv, pool.num_pages, pool.page_table, pool.max_pages, lens_d,
                      splits_d, chunks_d, plan.max_splits, plan.kv_split, B, q_len, H,
                      w["causal"], 1.0, 1.0, SOFTMAX_SCALE, ws_k, ws_bytes, out_k, lse_k, None)
                     + ((sels[k],) if is_sparse else ()))
    args_common = calls[0]
    ws, out, lse = args_common[17], args_common[19], args_common[20]
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    is_bf16 = inp.q.dtype == torch.bfloat16

    # A plan with empty split slots (a skewed or ragged batch) launches the FP8
    # kernel over its CTA item list: exactly the CTAs that have work.
    use_items = (not is_bf16) and (bool(np.any(plan.splits < plan.max_splits))
                                   or args.persistent > 0)
    items_h = mla.mla_decode_plan_items(plan.splits, H, q_len) if use_items else None
    items_d = torch.from_numpy(items_h).to(dev) if use_items else None

    def decode_call(*a, items=None, phases=mla.PHASE_ALL):
        # a = one call's 22 arguments (+ the page selection), then the stream
        c, s = a[:-1], a[-1]
        it = items_d if items is None else items
        if is_sparse:
            mla.mla_decode_sparse(*c[:6], c[22], topk, *c[6:22], cta_items=it,
                                  persistent_ctas=args.persistent, phases=phases, stream=s)
        elif is_bf16:  # BF16 Q and KV: no q/kv scales
            if phases == mla.PHASE_ALL:
                mla.mla_decode_bf16(*c[:14], *c[16:22], s)
            else:
                mla.mla_decode_bf16_ex(*c[:14], *c[16:22], phases=phases, stream=s)
        elif use_items:
            mla.mla_decode_ex(*c[:22], cta_items=it, persistent_ctas=args.persistent,
                              phases=phases, stream=s)
        else:
            mla.mla_decode(*c[:22], s)

    # The two phases of the same calls alone, for per-kernel durations: the
    # split-KV kernel, then the merge of the partials it left (the phase entry
    # points for plain calls, the options' phases for the others).
    def split_call(*a):
        if is_bf16 or is_sparse or use_items:
            decode_call(*a, phases=mla.PHASE_SPLIT)
        else:
            mla.mla_decode_splitkv(*a[:22], a[-1])

    def merge_call(*a):
        if is_bf16 or is_sparse or use_items:
            decode_call(*a, phases=mla.PHASE_MERGE)
        else:
            mla.mla_decode_merge(*a[:22], a[-1])

    phases = (("full", decode_call), ("split", split_call), ("merge", merge_call))

    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            decode_call(*calls[k % n_pools], stream)
    torch.cuda.synchronize(dev)
    mla.mla_decode_status(ws, stream)

    # ---- timed region: K steps replayed from a CUDA graph ----
    # One graph holds the K decode calls (split-KV kernel + merge); two more
    # hold the same K calls of each phase alone, for per-kernel durations.
    K = args.steps
    graphs = {}
    for name, fn in phases:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(K):
                fn(*calls[k % n_pools], None)
        graphs[name] = g
    for g in graphs.values():  # one untimed replay each
        g.replay()
    torch.cuda.synchronize(dev)
    ev = {n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for n in graphs}
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        for n in ("full", "split", "merge"):
            ev[n][0].record(stream)
            graphs[n].replay()
            ev[n][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    total_ms = ev["full"][0].elapsed_time(ev["full"][1])
    split_us = ev["split"][0].elapsed_time(ev["split"][1]) * 1e3 / K
    merge_us = ev["merge"][0].elapsed_time(ev["merge"][1]) * 1e3 / K
    us_per_call = max_over_ranks(total_ms * 1e3 / K, dev)
    mla.mla_decode_status(ws, stream)

    # ---- spread over further replays, and the graph-launch floor ----
    # p10 / median / p90 of the per-call time over further replays of the
    # K-call graph (reported beside `value`, which is the bracketed run above).
    rep_us = []
    with torch.cuda.stream(stream):
        for _ in range(max(0, args.replays)):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graphs["full"].replay()
            e1.record(stream)
            e1.synchronize()
            rep_us.append(e0.elapsed_time(e1) * 1e3 / K)
    # Trivial-kernel floor: K one-element kernels through the same graph path.
    tiny = torch.zeros(1, device=dev)
    with torch.cuda.stream(stream):
        tiny.add_(1.0)
    torch.cuda.synchronize(dev)
    g_floor = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_floor, stream=stream):
        for _ in range(K):
            tiny.add_(1.0)
    with torch.cuda.stream(stream):
        g_floor.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g_floor.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    floor_us = e0.elapsed_time(e1) * 1e3 / K
    # Warm L2 (reported beside the cold number when the inputs rotate): the
    # same K calls on the first pool only.
    warm_us = None
    if n_pools > 1:
        g_warm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_warm, stream=stream):
            for _ in range(K):
                decode_call(*calls[0], None)
        with torch.cuda.stream(stream):
            g_warm.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g_warm.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        warm_us = e0.elapsed_time(e1) * 1e3 / K
        del g_warm
    mla.mla_decode_status(ws, stream)
    del graphs, g_floor

    # ---- end to end through the public API with host buffers ----
    # Each call copies its inputs (Q, page table, plan arrays, selection or
    # item list) from pinned host memory and reads its output and LSE back.
    # Two schedules are timed: "serial" (copies and call in order on one
    # stream) and "overlapped" (the copies of call k + 1 on a second stream
    # into the other of two device input sets while call k computes, the
    # double buffering of a serving loop: call k waits for its own copies, and
    # copies into a set wait until the call that last read it is done).  The
    # second costs more host work per call, so it pays only where the call's
    # device time hides it; the line reports the faster and both values.
    q_h = inp.q.cpu().pin_memory()
    pt_h = inp.page_table.cpu().pin_memory()
    meta_h = torch.tensor(np.stack([np.asarray(lens, np.int32), plan.splits, plan.chunks]),
                          dtype=torch.int32).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    sel_h = sels[0].cpu().pin_memory() if is_sparse else None
    it_h = torch.from_numpy(items_h).pin_memory() if use_items else None
    h2d = q_h.numel() * q_h.element_size() + pt_h.numel() * 4 + meta_h.numel() * 4
    if is_sparse:
        h2d += sel_h.numel() * 4
    if use_items:
        h2d += it_h.numel() * 4
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    sets = []
    for _ in range(2):
        st = {"q": torch.empty_like(inp.q), "pt": torch.empty_like(inp.page_table),
              "meta": torch.empty_like(meta_h, device=dev),
              "sel": torch.empty_like(sels[0]) if is_sparse else None,
              "it": torch.empty_like(items_d) if use_items else None,
              "copied": torch.cuda.Event(), "used": torch.cuda.Event()}
        a_ = list(args_common)
        a_[0], a_[3] = st["q"], st["pt"]
        a_[5], a_[6], a_[7] = st["meta"][0], st["meta"][1], st["meta"][2]
        if is_sparse:
            a_[22] = st["sel"]
        st["args"] = a_
        sets.append(st)
    copy_stream = torch.cuda.Stream(device=dev)
    n_e2e = [0]

    def e2e_step_serial():
        st = sets[0]
        p = (mla.mla_decode_plan(plan_lens, H, q_len, sm_count=sm_count)
             if args.plan == "gb300" else plan)
        del p
        if use_items:
            mla.mla_decode_plan_items(plan.splits, H, q_len)  # host cost of the item list
        st["q"].copy_(q_h, non_blocking=True)
        st["pt"].copy_(pt_h, non_blocking=True)
        st["meta"].copy_(meta_h, non_blocking=True)
        if is_sparse:
            st["sel"].copy_(sel_h, non_blocking=True)
        if use_items:
            st["it"].copy_(it_h, non_blocking=True)
        decode_call(*st["args"], stream, items=st["it"] if use_items else None)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    def e2e_step_overlapped():
        st = sets[n_e2e[0] & 1]
        p = (mla.mla_decode_plan(plan_lens, H, q_len, sm_count=sm_count)
             if args.plan == "gb300" else plan)
        del p
        if use_items:
            mla.mla_decode_plan_items(plan.splits, H, q_len)  # host cost of the item list
        with torch.cuda.stream(copy_stream):
            if n_e2e[0] >= 2:
                copy_stream.wait_event(st["used"])
            st["q"].copy_(q_h, non_blocking=True)
            st["pt"].copy_(pt_h, non_blocking=True)
            st["meta"].copy_(meta_h, non_blocking=True)
            if is_sparse:
                st["sel"].copy_(sel_h, non_blocking=True)
            if use_items:
                st["it"].copy_(it_h, non_blocking=True)
            st["copied"].record(copy_stream)
        stream.wait_event(st["copied"])
        decode_call(*st["args"], stream, items=st["it"] if use_items else None)
        st["used"].record(stream)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        n_e2e[0] += 1

    e2e_sched = {}
    for name, step in (("serial", e2e_step_serial), ("overlapped", e2e_step_overlapped)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            for _ in range(args.e2e_steps):
                step()
            torch.cuda.synchronize(dev)
        e2e_sched[name] = max_over_ranks((time.perf_counter() - t0) * 1e6 / args.e2e_steps, dev)
    e2e_best = min(e2e_sched, key=e2e_sched.get)
    e2e_us = e2e_sched[e2e_best]

    # ---- roofline of the dominant kernel (split-KV) ----
    # HBM-bound unless the flop per KV byte is above the ridge of the MMA
    # type's peak (E4M3: twice the measured bf16 burst, the nominal ratio of
    # the dense rates), as for H96 q8 (768 rows per request).
    split_avg_s = split_us * 1e-6
    achieved = kv_bytes / split_avg_s / 1e9
    peaks = measured_peaks()
    traffic = recorded_traffic(args.workload)
    flops = algorithmic_flops(lens, H, q_len, w["causal"], sel0 if is_sparse else None)
    mma_peak = peaks["bf16_tflops"] * (1.0 if is_bf16 else 2.0)
    ridge = mma_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    intensity = flops / kv_bytes
    tflops = flops / split_avg_s / 1e12
    hbm_line = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"]}
    tensor_line = {"bound": "tensor", "achieved": tflops, "peak": mma_peak, "unit": "TFLOP/s",
                   "frac": tflops / mma_peak,
                   "peak_note": ("measured bf16 burst" if is_bf16 else
                                 "2 x measured bf16 burst (nominal E4M3 / bf16 dense ratio)")}
    roof = dict(tensor_line if intensity >= ridge else hbm_line)
    roof.update({"traffic": traffic, "peak_source": peaks["source"],
                 "flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                 "other": {k: v for k, v in (hbm_line if intensity >= ridge else tensor_line).items()
                           if k in ("bound", "achieved", "peak", "unit", "frac")},
                 "kernel": ("mla_split_kv_bf16_kernel (timed with its merge)"
                            if is_bf16 else "mla_split_kv_kernel")})

    cpu = None
    if rank == 0 and world == 1 and args.cpu_rows > 0:
        sel_np = sels[0].cpu().numpy() if is_sparse else None
        t, done, threads = cpu_oracle_sample(inp, w, args.cpu_rows, SOFTMAX_SCALE,
                                             selection=sel_np)
        total = kv_bytes // (576 * inp.kv.element_size()) * H * q_len  # row-keys
        cpu = {"value": t / done * total * 1e6, "unit": UNIT, "cores": threads,
               "kind": "oracle",
               "sample": f"first {args.cpu_rows} of {inp.rows} rows over their full KV length "
                         f"({t:.1f} s); time scaled by row-keys to the whole call"}

    if rank == 0:
        pub = PUBLISHED_US.get(args.workload)
        line = {
            "metric": METRIC, "value": us_per_call, "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": us_per_call / 1e3,
            "higher_is_better": False, "scaling": "weak",
            "vs_baseline": (us_per_call / pub) if pub else None,
            "dtype": "bf16" if is_bf16 else "e4m3",
            "data": ("synthetic (seeded N(0,0.5^2) cast to "
                     f"{'BF16' if is_bf16 else 'E4M3'}, random pages)"),
            "config": {"workload": args.workload, "batch": B, "num_heads": H, "q_len": q_len,
                       "kv_len": lens[0], "causal": w["causal"],
                       "plan": f"target {args.target}" if args.target > 0 else args.plan,
                       "persistent_ctas": args.persistent,
                       "splits": plan.splits.tolist()[:4] + (["..."] if B > 4 else []),
                       "kv_split": plan.kv_split, "kv_bytes": kv_bytes,
                       "cta_items": use_items,
                       "l2": ("inputs larger than L2 (no flush)" if n_pools == 1 else
                              f"{n_pools} rotating input pools ({n_pools * kv_bytes} B > 2x L2)"),
                       "timing": "CUDA graph of K calls, CUDA events",
                       "parallelism": f"replicas x{world}" if world > 1 else "single"},
            "kv_gbs": kv_bytes / (us_per_call * 1e-6) / 1e9,
            "aggregate_kv_gbs": world * kv_bytes / (us_per_call * 1e-6) / 1e9,
            "split_kernel_us": split_us,
            "merge_kernel_us": merge_us,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "schedule": e2e_best, "serial_us": e2e_sched["serial"],
                    "overlapped_us": e2e_sched["overlapped"]},
            "gpu_launches": K * (2 if plan.max_splits > 1 else 1),
            "replays": ({"n": len(rep_us), "p10_us": float(np.percentile(rep_us, 10)),
                         "median_us": float(np.median(rep_us)),
                         "p90_us": float(np.percentile(rep_us, 90))} if rep_us else None),
            "floor_us_per_call": floor_us,
            "warm_l2_us_per_call": warm_us,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
