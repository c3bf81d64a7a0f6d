"""One decode step, computed by the oracle from a `workloads.Workload`.

Test infrastructure only.  The step, in the order a serving loop does it:
  1. host: rebuild the allocator state (blocks held by several tables are
     held once per table), then for each sequence in order make room for its
     new tokens (copy-on-write of shared blocks, then new blocks);
  2. copy_blocks for the copy-on-write pairs;
  3. slot mapping of the new tokens;
  4. reshape_and_cache of their K/V;
  5. decode attention over every sequence's full context (fp64).

Token data lives in a compact pool holding only the blocks this step can
touch; `row_of_block` maps a physical id to its row (see oracle.c).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import kernels
from .allocator import BlockAllocatorModel, fork_tables


@dataclass
class OracleStep:
    tables: np.ndarray          # [S, MB] int32 after the step (-1 = unused)
    nblocks: np.ndarray         # [S]
    pairs: np.ndarray           # [P, 2] int64 copy-on-write (src, dst)
    slots: np.ndarray           # [T] int64
    pool_ids: np.ndarray        # sorted physical ids held in the compact pool
    row_of_block: np.ndarray    # [NB] int32, -1 for blocks not in the pool
    k_pool: np.ndarray          # [len(pool_ids), bs, H, D] uint16 after the step
    v_pool: np.ndarray
    out: np.ndarray | None      # [S, H, D] float64 (NaN where not computed)
    allocator: BlockAllocatorModel
    k_pre: np.ndarray | None = None   # pool before copy/write (if kept)
    v_pre: np.ndarray | None = None


def rebuild_allocator(w) -> BlockAllocatorModel:
    a = BlockAllocatorModel(w.NB, initial_free=w.initial_free)
    ids, counts = np.unique(w.tables_pre[w.tables_pre >= 0], return_counts=True)
    for b, c in zip(ids.tolist(), counts.tolist()):
        if c > 1:
            a.incref([b] * (c - 1))
    return a


def plan(w):
    """Host part of the step: (allocator, tables [S,MB], nblocks, pairs [P,2])."""
    a = rebuild_allocator(w)
    tables = []
    pairs = []
    for s in range(w.S):
        t = w.tables_pre[s, :w.nblocks_pre[s]].tolist()
        pairs += a.append(t, int(w.ctx_before[s]), int(w.n_new[s]), w.bs)
        tables.append(t)
    nb = np.array([len(t) for t in tables], dtype=np.int32)
    assert nb.max(initial=0) <= w.MB
    out = np.full((w.S, w.MB), -1, dtype=np.int32)
    for s, t in enumerate(tables):
        out[s, :len(t)] = t
    return a, out, nb, np.array(pairs, dtype=np.int64).reshape(-1, 2)


def build_pool(w, tables, pairs, poison):
    ids = np.unique(np.concatenate([w.blocks, tables[tables >= 0].ravel(),
                                    pairs.ravel()]).astype(np.int64)).astype(np.int32)
    row_of_block = np.full(w.NB, -1, dtype=np.int32)
    row_of_block[ids] = np.arange(len(ids), dtype=np.int32)
    shape = (len(ids), w.bs, w.H, w.D)
    k_pool = np.full(shape, poison, dtype=np.uint16)
    v_pool = np.full(shape, poison, dtype=np.uint16)
    if len(w.blocks):
        k_pool[row_of_block[w.blocks]] = w.k_blocks
        v_pool[row_of_block[w.blocks]] = w.v_blocks
    return ids, row_of_block, k_pool, v_pool


def run(w, items=None, nthreads=None, keep_pre=False, attention=True) -> OracleStep:
    from workloads import POISON, BF16
    if nthreads is None:
        nthreads = kernels.default_threads()
    a, tables, nb, pairs = plan(w)
    ids, rob, k_pool, v_pool = build_pool(w, tables, pairs, POISON[w.dtype])
    k_pre = k_pool.copy() if keep_pre else None
    v_pre = v_pool.copy() if keep_pre else None
    kernels.copy_blocks(k_pool, v_pool, pairs, row_of_block=rob)
    slots = kernels.slot_mapping(tables, w.seq_idx, w.pos, w.bs)
    kernels.reshape_and_cache(k_pool, v_pool, w.new_k, w.new_v, slots, row_of_block=rob)
    out = None
    if attention:
        out = kernels.decode(w.q, k_pool, v_pool, tables, w.context_lens, w.scale,
                             w.dtype == BF16, row_of_block=rob, items=items, nthreads=nthreads)
    return OracleStep(tables=tables, nblocks=nb, pairs=pairs, slots=slots, pool_ids=ids,
                      row_of_block=rob, k_pool=k_pool, v_pool=v_pool, out=out, allocator=a,
                      k_pre=k_pre, v_pre=v_pre)


def run_beam(bw, nthreads=None, items=None):
    """Beam search by the oracle: yields, after each step, (tables [S, MB],
    pairs [P, 2], slots [S], k_pool, v_pool, pool_ids, out [S, H, D])."""
    from workloads import POISON, BF16
    w = bw.init
    if nthreads is None:
        nthreads = kernels.default_threads()
    a = rebuild_allocator(w)
    tables = [w.tables_pre[s, :w.nblocks_pre[s]].tolist() for s in range(w.S)]
    ctx = w.ctx_before.astype(np.int64).copy()
    # every block the run can touch lives in the compact pool from the start
    ids = np.arange(w.NB, dtype=np.int32)
    rob = ids.copy()
    k_pool = np.full((w.NB, w.bs, w.H, w.D), POISON[w.dtype], dtype=np.uint16)
    v_pool = k_pool.copy()
    if len(w.blocks):
        k_pool[w.blocks], v_pool[w.blocks] = w.k_blocks, w.v_blocks
    for i in range(bw.steps):
        parents = bw.parents[i]
        tables = fork_tables(a, tables, parents)
        ctx = ctx[parents]
        pairs = []
        for b in range(w.S):
            pairs += a.append(tables[b], int(ctx[b]), 1, w.bs)
        pairs = np.array(pairs, dtype=np.int64).reshape(-1, 2)
        bt = np.full((w.S, w.MB), -1, dtype=np.int32)
        for b, t in enumerate(tables):
            bt[b, :len(t)] = t
        kernels.copy_blocks(k_pool, v_pool, pairs, row_of_block=rob)
        seq_idx = np.arange(w.S, dtype=np.int32)
        slots = kernels.slot_mapping(bt, seq_idx, ctx.astype(np.int32), w.bs)
        kernels.reshape_and_cache(k_pool, v_pool, bw.new_k[i], bw.new_v[i], slots,
                                  row_of_block=rob)
        ctx = ctx + 1
        out = kernels.decode(bw.q[i], k_pool, v_pool, bt, ctx.astype(np.int32), w.scale,
                             w.dtype == BF16, row_of_block=rob, items=items, nthreads=nthreads)
        yield bt, pairs, slots, k_pool, v_pool, ids, out
