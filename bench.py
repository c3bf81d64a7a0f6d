"""Benchmark: paged decode-attention KV GB/s and tokens/s on GB300.

A step is one pass of the whole hot path over one batch:
  copy_blocks (if the step has copy-on-write pairs) -> slot mapping ->
  reshape_and_cache of the new tokens -> paged decode attention (+ merge).
Default workload: the LLaMA-7B-shaped layer -- 64 sequences, 32 heads x 128,
fp16, block size 16, context ~ U{128..2048}, pool = need + 10 %, shuffled
placement, one new token per sequence.

value  = logical KV bytes read per step (sum ctx * H * D * 2 * 2 B) / step time
e2e    = the same metric with each step's inputs and output in pinned host
         memory and every host<->device transfer inside the timed region (one
         upload of the integer inputs; the kernels read the tokens and write
         the output over the host link)
--impl reference times the fp64 CPU oracle on the host cores instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs its own batch (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attn KV GB/s (% of GB300 HBM peak) and tokens/s at 1 GPU"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ["paged_kv_cache_162_gb300/csrc/decode.cu",
                  "paged_kv_cache_162_gb300/csrc/pkv_device.cuh"]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="llama7b_batch64")
    p.add_argument("--partition-tokens", type=int, default=0)
    p.add_argument("--shared-prefix", action="store_true",
                   help="shared_prefix workloads (and --measure beam_search): decode with each "
                        "prompt's prefix read once")
    p.add_argument("--block-size", type=int, default=0,
                   help="llama7b_batch64 only: another block size (8, 16, 32, 64)")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--prefix-kernel", choices=["mma", "tcgen05"], default="mma",
                   help="with --shared-prefix: the prefix kernel (tcgen05: head_dim 128)")
    p.add_argument("--unfused", action="store_true",
                   help="time the step as four separate calls instead of pkv_decode_step")
    p.add_argument("--measure", choices=["step", "swap_blocks", "beam_search"], default="step",
                   help="swap_blocks: GPU <-> pinned-host block copies; beam_search: fork + "
                        "copy-on-write every step")
    return p.parse_args(argv)


# ------------------------------------------------------------------ helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and with blank runs collapsed, so
    that an edit to a comment leaves the digest of the code unchanged.
    String and character literals are kept as they are."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest(paths=DECODE_SOURCES) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if the
    decode sources are unchanged since that capture; else None."""
    path = os.path.join(ROOT, "profiles", f"decode_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    d = re.search(r"decode_source_digest:\s*([0-9a-f]+)", text)
    if not m or not d or d.group(1) != source_digest():
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9], float(f[3])))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        # samples under load: power within half of the highest seen
        pmax = max(r[3] for r in rows)
        load = [r for r in rows if r[3] >= 0.5 * pmax] or rows
        sms = sorted(r[0] for r in load)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[2]) if v == "Active"})
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(load), "power_w_max": pmax}


def reduce_max(values, world, device=None):
    """Max over ranks of each value (all_reduce MAX); identity at world 1."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def weak_value(bytes_per_rank, world, step_ms):
    """Whole-job GB/s: every rank moves bytes_per_rank per step, and the
    slowest rank's step time bounds the job."""
    return world * bytes_per_rank / (step_ms * 1e-3) / 1e9


# ------------------------------------------------------------- workloads
def describe(w):
    import numpy as np
    ctx = w.context_lens.astype(np.int64)
    blocks = -(-ctx // w.bs)
    return {"workload": w.name, "seqs": w.S, "heads": w.H, "head_dim": w.D, "block_size": w.bs,
            "pool_blocks": w.NB, "context_min": int(ctx.min()), "context_max": int(ctx.max()),
            "context_sum": int(ctx.sum()), "new_tokens": w.T,
            "kv_bytes_per_step": w.kv_bytes(),
            # the block-size trade-off: table entries vs unfilled slots in last blocks
            "table_entries": int(blocks.sum()),
            "unfilled_slot_fraction": float((blocks * w.bs - ctx).sum() / (blocks * w.bs).sum())}


def make_workload(name, rank, block_size=0):
    import workloads as W
    seed_shift = 7919 * rank  # each rank its own batch
    if name == "llama7b_batch64":
        return W.llama7b_batch64(seed=1001 + seed_shift, bs=block_size or 16)
    if name == "continuous_batching_bf16":
        return W.continuous_batching_bf16(seed=1002 + seed_shift)
    if name == "shared_prefix":
        return W.shared_prefix(seed=1003 + seed_shift)
    if name == "shared_prefix_cow":
        return W.shared_prefix(seed=1003 + seed_shift, cow=True)
    if name.startswith("long_context_bs"):
        return W.long_context(bs=int(name[len("long_context_bs"):]), seed=1004 + seed_shift)
    if name == "tiny":
        return W.tiny(seed=1000 + seed_shift)
    raise SystemExit(f"unknown workload {name}")


# --------------------------------------------------------- oracle timing
def time_oracle(w, seconds_per_step=2.0, threads=None):
    """Times one oracle step (slot mapping, cache write, fp64 decode) over a
    bounded sample of the workload: the first n (sequence, head) pairs in
    sequence order, n calibrated so that the step takes about
    `seconds_per_step`.  Returns (seconds, sample_bytes, sample_seqs,
    threads, fn) where fn() re-runs the same sample."""
    import numpy as np
    from oracle import kernels as K
    from oracle import step as OS
    import workloads as W

    if threads is None:
        threads = K.default_threads()
    a, tables, nb, pairs = OS.plan(w)
    ids, rob, k_pool, v_pool = OS.build_pool(w, tables, pairs, W.POISON[w.dtype])
    ctx = w.context_lens.astype(np.int64)
    per_tok = w.D * 2 * 2  # K and V bytes of one token of one head
    all_items = np.array([[s, h] for s in range(w.S) for h in range(w.H)], dtype=np.int32)
    item_bytes = ctx[all_items[:, 0]] * per_tok

    def run_items(items, tok):
        K.copy_blocks(k_pool, v_pool, pairs, row_of_block=rob)
        slots = K.slot_mapping(tables, w.seq_idx[tok], w.pos[tok], w.bs)
        K.reshape_and_cache(k_pool, v_pool, w.new_k[tok], w.new_v[tok], slots, row_of_block=rob)
        K.decode(w.q, k_pool, v_pool, tables, w.context_lens, w.scale, w.dtype == W.BF16,
                 row_of_block=rob, items=items, nthreads=threads)

    # calibrate on about 1 % of the workload (at least one item per thread)
    n_cal = int(min(len(all_items), max(threads, len(all_items) // 100)))
    t0 = time.perf_counter()
    run_items(all_items[:n_cal], np.zeros(len(w.seq_idx), dtype=bool))
    rate = item_bytes[:n_cal].sum() / max(time.perf_counter() - t0, 1e-6)
    cum = np.cumsum(item_bytes)
    n = int(np.searchsorted(cum, rate * seconds_per_step)) + 1
    n = max(1, min(n, len(all_items)))
    items = all_items[:n]
    seqs = np.unique(items[:, 0])
    tok = np.isin(w.seq_idx, seqs)
    sample_bytes = int(item_bytes[:n].sum())

    def one():
        run_items(items, tok)

    reps, t0 = 0, time.perf_counter()
    while True:
        one()
        reps += 1
        if time.perf_counter() - t0 >= min(1.0, seconds_per_step):
            break
    dt = (time.perf_counter() - t0) / reps
    return dt, sample_bytes, n / w.H, threads, one


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = make_workload(args.workload, 0)
    # each step a bounded sample, so that warmup + steps take ~2.5 minutes
    per_step = min(2.0, max(0.02, 150.0 / (args.steps + args.warmup + 1)))
    dt, sample_bytes, nseq, threads, one = time_oracle(w, per_step)
    for _ in range(max(0, args.warmup)):
        one()
    times = []
    for _ in range(max(1, args.steps)):
        t0 = time.perf_counter()
        one()
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    gbs = sample_bytes / t / 1e9
    tok_s = nseq / t
    sample = (f"first {int(round(nseq * w.H))} (sequence, head) pairs of {w.name} in sequence "
              f"order ({nseq:.2f} of {w.S} sequences), {sample_bytes / 1e6:.1f} MB of logical "
              f"KV per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": describe(w), "tokens_per_s": tok_s,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- our path
def run_ours(args):
    if args.prefix_kernel == "tcgen05":
        os.environ["PKV_PREFIX_KERNEL"] = "tcgen05"
    else:
        os.environ.pop("PKV_PREFIX_KERNEL", None)
    import numpy as np
    import torch
    import torch.distributed as dist

    import workloads as W
    from paged_kv_cache_162_gb300 import _lib as L
    from paged_kv_cache_162_gb300.engine import DecodeStep, dtype_code

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        # one rank per GPU: bind the group to this rank's device
        dist.init_process_group("nccl", device_id=dev)

    w = make_workload(args.workload, rank, args.block_size)
    st = DecodeStep(dtype=w.dtype, S=w.S, H=w.H, D=w.D, bs=w.bs, NB=w.NB, MB=w.MB, scale=w.scale,
                    ctx_before=w.ctx_before, n_new=w.n_new, tables_pre=w.tables_pre,
                    nblocks_pre=w.nblocks_pre, initial_free=w.initial_free, blocks=w.blocks,
                    k_blocks=w.k_blocks, v_blocks=w.v_blocks, q=w.q, new_k=w.new_k,
                    new_v=w.new_v, seq_idx=w.seq_idx, pos=w.pos,
                    fill_bits=int(W.POISON[w.dtype]), partition_tokens=args.partition_tokens,
                    device=dev)
    st.plan()
    stream = torch.cuda.Stream(device=dev)
    kv_bytes = w.kv_bytes()
    # algorithmic bytes of one decode launch: KV rows + q + out + table entries
    dec_bytes = (kv_bytes + 2 * w.S * w.H * w.D * 2
                 + int(np.ceil(w.context_lens / w.bs).sum()) * 4)
    # the step: copy_blocks (if any pairs), then pkv_decode_step (slot
    # mapping + cache write + plan in one kernel, then decode); --unfused and
    # shared-prefix decode use the separate calls
    fused = not args.unfused
    decode_kernels = 3 if args.shared_prefix else 2   # plan or prologue, [prefix,] decode
    launches_per_step = ((1 if len(st.pairs_host) else 0) +
                         (decode_kernels if fused else (2 if w.T else 0) + decode_kernels))

    from paged_kv_cache_162_gb300.engine import (StepGraph, compute_slot_mapping, copy_blocks,
                                                 reshape_and_cache)
    has_pairs = len(st.pairs_host) > 0
    if args.shared_prefix:
        if not w.name.startswith("shared_prefix"):
            raise SystemExit("--shared-prefix needs a shared_prefix workload")
        from paged_kv_cache_162_gb300.engine import paged_attention_decode_shared_prefix
        samples = w.notes["samples"]
        groups = torch.tensor([[p * samples, samples, 1024] for p in range(w.S // samples)],
                              dtype=torch.int32, device=dev)
        from paged_kv_cache_162_gb300 import _lib as _L
        ws_sp = torch.empty(_L.pkv_decode_shared_prefix_workspace_size(
            w.S, w.H, w.D, groups.shape[0], st.max_context_len, args.partition_tokens),
            dtype=torch.uint8, device=dev)
        st.decode = lambda stream=None: paged_attention_decode_shared_prefix(
            st.out, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, groups,
            st.scale, st.max_context_len, args.partition_tokens, workspace=ws_sp, stream=stream)
        st.prefix_groups, st.workspace = groups, ws_sp   # for the fused step

    def step():
        if fused:
            st.run(stream, fused=True)
            return
        if has_pairs:
            copy_blocks(st.k_cache, st.v_cache, st.pairs, stream)
        if w.T:
            compute_slot_mapping(st.slot_mapping, st.block_tables, st.seq_idx, st.pos, w.bs,
                                 stream)
            reshape_and_cache(st.new_k, st.new_v, st.k_cache, st.v_cache, st.slot_mapping, stream)
        st.decode(stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    stream.synchronize()
    L.pkv_sync_check(stream)

    def barrier():
        if world > 1:
            dist.barrier(device_ids=[local])

    # ---- the timed region: K whole steps, events only at its two ends
    K = max(1, args.steps)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        # warm up again after the sampler's start-up pause, so that a short
        # timed region does not begin on a GPU that has just idled for 0.3 s
        # (measured: 20 timed steps 171.5 us per step after the pause, 168.4
        # us with this, 168.8 us over 5000 steps).  It runs for at least
        # 0.25 s, so the sampler (one sample per 100 ms) also records the
        # clocks under this load right before a timed region that may be
        # only a few milliseconds long.
        t_warm = time.perf_counter()
        n_warm = 0
        with torch.cuda.stream(stream):
            while n_warm < max(3, args.warmup) or time.perf_counter() - t_warm < 0.25:
                step()
                n_warm += 1
                if n_warm % 32 == 0:
                    stream.synchronize()  # keep the host within 32 steps of the GPU
        stream.synchronize()
        barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for _ in range(K):
                step()
            t_end.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier()
    total_ms = t_start.elapsed_time(t_end)
    L.pkv_sync_check(stream)
    errs = L.pkv_get_device_errors()
    if errs:
        raise SystemExit(f"device error word set: {errs:#x}")

    # ---- the same steps again with an event pair around every kernel call:
    # each kernel's duration in the step's own cache state (the events cost
    # the step its launch overlap, so the step time comes from region A)
    KB = min(K, 500)
    names = (["copy_blocks"] if has_pairs else []) + (["slot_mapping", "reshape_and_cache"]
                                                      if w.T else []) + ["decode"]
    evs = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(KB)] for n in names}
    calls = {
        "copy_blocks": lambda: copy_blocks(st.k_cache, st.v_cache, st.pairs, stream),
        "slot_mapping": lambda: compute_slot_mapping(st.slot_mapping, st.block_tables, st.seq_idx,
                                                     st.pos, w.bs, stream),
        "reshape_and_cache": lambda: reshape_and_cache(st.new_k, st.new_v, st.k_cache, st.v_cache,
                                                       st.slot_mapping, stream),
        "decode": lambda: st.decode(stream),
    }
    with torch.cuda.stream(stream):
        for i in range(KB):
            for n in names:
                evs[n][i][0].record(stream)
                calls[n]()
                evs[n][i][1].record(stream)
    stream.synchronize()
    elem = 2
    nbytes = {"decode": dec_bytes,
              "slot_mapping": w.T * (4 + 4 + 4 + 8),   # seq_idx, pos, table entry; slot
              "reshape_and_cache": w.T * (2 * 2 * w.H * w.D * elem + 8),  # K, V rows in and out
              "copy_blocks": len(st.pairs_host) * 2 * 2 * w.bs * w.H * w.D * elem}
    kernels = {}
    for n in names:
        ms = sum(a.elapsed_time(b) for a, b in evs[n]) / KB
        kernels[n] = {"ms": ms, "bytes": nbytes[n], "gbs": nbytes[n] / (ms * 1e-3) / 1e9}
    dec_ms = kernels["decode"]["ms"]

    # ---- end to end: every input and the output in pinned host memory,
    # all host<->device traffic inside the timed region, one CUDA graph per
    # step, then a sync.  The integer inputs (tables, lengths, positions,
    # copy pairs) are uploaded by one copy; the kernels read q and the new
    # K/V where the host wrote them and write the output straight into host
    # memory (GB300: over the coherent NVLink-C2C link), which replaced the
    # copies of those bytes
    ref_out = st.out.clone()
    dev_in, host_in, (up_dev, up_host) = st.pack_inputs(on_host=("q", "new_k", "new_v"))
    host_out = st.pin_output()
    h2d = host_in.numel()
    d2h = host_out.numel() * host_out.element_size()
    g = StepGraph(st, stream, h2d=[(up_dev, up_host)], d2h=[], fused=fused)

    def e2e_step():
        g.replay()          # on `stream`
        stream.synchronize()

    E = max(1, args.e2e_steps)
    for _ in range(3):
        e2e_step()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        e2e_step()
    e1.record(stream)
    stream.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / E
    # the graph's output must equal the eager, device-resident step's
    assert torch.equal(host_out.view(torch.int16), ref_out.cpu().view(torch.int16))

    # ---- max over ranks
    step_ms = total_ms / K
    step_ms, e2e_ms, dec_ms = reduce_max([step_ms, e2e_ms, dec_ms], world, dev)
    peak, peak_kind = measured_peak()
    value = weak_value(kv_bytes, world, step_ms)
    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
    traffic = profiled_traffic(args.workload)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        dt, sample_bytes, nseq, threads, _ = time_oracle(w)
        dt1, bytes1, nseq1, _, _ = time_oracle(w, 1.0, threads=1)
        cpu = {"value": sample_bytes / dt / 1e9, "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "sample": f"one oracle step (slot mapping, cache write, fp64 decode) over the "
                         f"first {int(round(nseq * w.H))} (sequence, head) pairs in sequence "
                         f"order ({nseq:.2f} of {w.S} sequences, "
                         f"{sample_bytes / 1e6:.1f} MB logical KV), {dt:.2f} s",
               "one_thread": {"value": bytes1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"the first {int(round(nseq1 * w.H))} (sequence, head) "
                                        f"pairs, {bytes1 / 1e6:.1f} MB logical KV, "
                                        f"{dt1:.2f} s"}}

    if rank == 0:
        cfg = describe(w)
        used_ws = ws_sp if args.shared_prefix else st.workspace
        chosen = int(used_ws[8:12].view(torch.int32).item())  # plan kernel's choice
        cfg.update({"partition_tokens": (f"auto ({chosen})" if not args.partition_tokens
                                         else args.partition_tokens),
                    "l2": f"inputs larger than L2: {kv_bytes / 1e9:.2f} GB of KV read per step "
                          f"vs 129 MB L2; no flush",
                    "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                    "step_calls": ("copy_blocks (if any pairs) + pkv_decode_step"
                                   + (f" with prefix groups ({args.prefix_kernel} prefix kernel)"
                                      if args.shared_prefix else "")
                                   if fused else
                                   "copy_blocks, compute_slot_mapping, reshape_and_cache, "
                                   "decode as separate calls"),
                    "global_batch": w.S * world})
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": cfg,
            "tokens_per_s": world * w.S / (step_ms * 1e-3),
            "pct_of_hbm_peak": {"of_measured": value / peak, "of_nominal_8000": value / NOMINAL_HBM_GBS},
            "decode_ms": dec_ms,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_kind,
                         "kernel": "pkv paged_attention_decode (plan + decode kernels), events "
                                   "around each call in a second run of the step loop",
                         "algorithmic_bytes_per_launch": dec_bytes,
                         "frac_of_step": dec_bytes / (step_ms * 1e-3) / 1e9 / peak,
                         "clocks_note": "frac uses decode_ms, the decode call alone with an "
                                        "event pair around it; the pair costs the call its "
                                        "launch overlap with the kernel before it, so decode_ms "
                                        "can exceed ms_per_step, which also holds the prologue "
                                        "kernel.  frac_of_step divides the same bytes by the "
                                        "whole timed step (region A's clock): a lower bound "
                                        "on the decode kernel's fraction"},
            "cpu_baseline": cpu,
            "e2e": {"value": weak_value(kv_bytes, world, e2e_ms), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "method": "one CUDA graph per step, then a stream sync; every input and "
                              "the output in pinned host memory: one H2D copy of the block "
                              "tables, context lengths, token positions and copy pairs; the "
                              "kernels read q and the new K/V from pinned host memory and "
                              "write the output into it (NVLink-C2C, no copy node)"},
            "kernels": kernels,
            "gpu_launches": launches_per_step * K,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_swap(args):
    """GPU <-> pinned-host block copies (CPU swap) at the LLaMA-7B layer shape:
    2048 blocks of 16 tokens x 32 heads x 128 fp16 (128 KB of K and 128 KB
    of V each) out to a host pool and back into other GPU blocks."""
    import numpy as np
    import torch
    from paged_kv_cache_162_gb300 import _lib as L
    from paged_kv_cache_162_gb300.engine import swap_blocks

    torch.cuda.set_device(0)
    bs, H, D, NBg, P = 16, 32, 128, 8192, 2048
    rng = np.random.default_rng(1005)
    gk = torch.randn(NBg, bs, H, D, device="cuda").half()
    gv = torch.randn(NBg, bs, H, D, device="cuda").half()
    hk = torch.empty(P, bs, H, D, dtype=torch.float16).pin_memory()
    hv = torch.empty(P, bs, H, D, dtype=torch.float16).pin_memory()
    src = rng.permutation(NBg)[:P]
    out_pairs = torch.from_numpy(np.stack([src, np.arange(P)], 1)).cuda()
    dst = rng.permutation(np.setdiff1d(np.arange(NBg), src))[:P]
    in_pairs = torch.from_numpy(np.stack([np.arange(P), dst], 1)).cuda()
    stream = torch.cuda.Stream()
    nbytes = P * 2 * bs * H * D * 2
    res = {}
    for name, pairs, direction in (("swap_out", out_pairs, L.PKV_SWAP_OUT),
                                   ("swap_in", in_pairs, L.PKV_SWAP_IN)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                swap_blocks(gk, gv, hk, hv, pairs, direction, stream)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(max(1, min(args.steps, 50)))]
            for a, b in evs:
                a.record(stream)
                swap_blocks(gk, gv, hk, hv, pairs, direction, stream)
                b.record(stream)
        stream.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
        res[name] = {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9}
    L.pkv_sync_check(stream)
    assert torch.equal(gk[dst[:4]], hk[:4].cuda()) and torch.equal(gk[src[:4]], gk[dst[:4]])
    print(json.dumps({"metric": "swap_blocks GB/s (K+V block payload per direction)",
                      "unit": "GB/s", "blocks": P, "bytes_per_call": nbytes,
                      "config": {"block_size": bs, "heads": H, "head_dim": D, "dtype": "f16",
                                 "gpu_pool_blocks": NBg, "host": "pinned (cudaHostAlloc)"},
                      **res}), flush=True)


def run_beam(args):
    """Beam search at scale: 16 requests x 4 beams at the LLaMA-7B layer shape,
    every step a fork of all 64 sequences (shared tables), copy-on-write of
    the shared partial blocks, the cache write and decode.  Times whole steps
    (host allocator work, upload of tables, lengths and copy pairs, kernels,
    sync) and the host part alone.  q and new K/V are on the device already,
    as a model running on it would produce them."""
    import numpy as np
    import torch
    import workloads as W
    from paged_kv_cache_162_gb300 import _lib as L
    from paged_kv_cache_162_gb300.engine import DecodeStep

    torch.cuda.set_device(0)
    steps = 64
    bw = W.beam_search(steps=steps)
    w = bw.init
    st = DecodeStep(dtype=w.dtype, S=w.S, H=w.H, D=w.D, bs=w.bs, NB=w.NB, MB=w.MB, scale=w.scale,
                    ctx_before=w.ctx_before, n_new=w.n_new, tables_pre=w.tables_pre,
                    nblocks_pre=w.nblocks_pre, initial_free=w.initial_free, blocks=w.blocks,
                    k_blocks=w.k_blocks, v_blocks=w.v_blocks, q=w.q, new_k=w.new_k,
                    new_v=w.new_v, seq_idx=w.seq_idx, pos=w.pos,
                    fill_bits=int(W.POISON[w.dtype]))
    st.plan()
    if args.shared_prefix:
        # each request's beams as a prefix group over the prompt's full blocks
        plen = w.notes["prompt_len"]
        st.beam_groups = [[r * bw.beams, bw.beams, (p // w.bs) * w.bs] for r, p in enumerate(plen)]
    # each step's q and new K/V on the device, as the model would produce them
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    new_k, new_v, q = dev(bw.new_k), dev(bw.new_v), dev(bw.q)
    # each step's tensors and parents handed over as a model would hand them
    # (views made before the loop: indexing a tensor is not library work)
    per_step = [(np.ascontiguousarray(bw.parents[i], dtype=np.int32), new_k[i], new_v[i], q[i])
                for i in range(steps)]
    stream = torch.cuda.current_stream()
    wall, host, pairs, kv, alloc_s = [], [], [], [], []
    for i in range(steps):
        par, nk, nv, qi = per_step[i]
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        p = st.beam_step(par, nk, nv, qi, stream=stream)
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        t2 = time.perf_counter()
        wall.append(t2 - t0)
        host.append(t1 - t0)
        alloc_s.append(st.last_native_seconds)
        pairs.append(len(p))
        kv.append(int(st.context_lens_host.astype(np.int64).sum()) * w.H * w.D * 4)
    L.pkv_sync_check()
    assert L.pkv_get_device_errors() == 0
    warm = slice(4, None)
    wall_ms = 1e3 * float(np.mean(wall[warm]))
    print(json.dumps({
        "metric": "beam-search steps/s (fork + copy-on-write + cache write + decode, 64 beams)",
        "unit": "steps/s", "value": 1e3 / wall_ms, "ms_per_step": wall_ms,
        "host_ms_per_step": 1e3 * float(np.mean(host[warm])),
        "native_call_us_per_step": 1e6 * float(np.mean(alloc_s[warm])),
        "copy_pairs_per_step": float(np.mean(pairs[warm])),
        "logical_kv_gbs": float(np.mean(kv[warm])) / (wall_ms * 1e-3) / 1e9,
        "config": {"requests": 16, "beams": 4, "heads": w.H, "head_dim": w.D,
                   "step_calls": "pkv_beam_step" + (" with a prefix group per request (its beams,"
                                                    " the prompt's full blocks)"
                                                    if args.shared_prefix else ""),
                   "block_size": w.bs, "prompt_tokens": "U{256..1024}", "steps": steps,
                   "timed_steps": steps - 4,
                   "inputs": "q and new K/V device-resident; tables, context lengths, "
                             "positions and copy pairs uploaded from pinned memory each step"}}),
          flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "ours" and args.measure == "swap_blocks":
        run_swap(args)
        return
    if args.impl == "ours" and args.measure == "beam_search":
        run_beam(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
