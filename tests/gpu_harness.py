"""Runs a `workloads.Workload` through the CUDA library (engine.DecodeStep)
and through the oracle, and compares them.

The bar: bit-exact tables, copy pairs, slots and caches; attention within
|gpu - oracle| <= ATOL + RTOL * |oracle| per element (fp64 oracle, before
its own rounding), ATOL = 2e-3, RTOL = 1e-2.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from oracle import step as OS
from paged_kv_cache_162_gb300.engine import DecodeStep

ATOL = 2e-3
RTOL = 1e-2


def device_step(w: W.Workload, partition_tokens: int = 0) -> DecodeStep:
    return DecodeStep(dtype=w.dtype, S=w.S, H=w.H, D=w.D, bs=w.bs, NB=w.NB, MB=w.MB, scale=w.scale,
                      ctx_before=w.ctx_before, n_new=w.n_new, tables_pre=w.tables_pre,
                      nblocks_pre=w.nblocks_pre, initial_free=w.initial_free, blocks=w.blocks,
                      k_blocks=w.k_blocks, v_blocks=w.v_blocks, q=w.q, new_k=w.new_k,
                      new_v=w.new_v, seq_idx=w.seq_idx, pos=w.pos, fill_bits=int(W.POISON[w.dtype]),
                      partition_tokens=partition_tokens)


def out_to_double(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().double().numpy()


def attention_error(got: np.ndarray, ref: np.ndarray):
    """(max abs error, max rel error over |ref| >= 0.2, worst excess over the bound)."""
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    big = np.abs(ref) >= 0.2
    rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    return float(err.max(initial=0.0)), rel, float((err - bound).max(initial=-1.0))


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mae, mre, excess = attention_error(got, ref)
    assert excess <= 0.0, f"{what}: max abs err {mae:.3g}, max rel {mre:.3g} beyond the bound"
    return mae, mre


def compare_step(w: W.Workload, partition_tokens=0, items=None, check_caches=True,
                 nthreads=None, fused=False):
    """Full comparison of one step; returns a dict of measured errors.
    fused=True runs the device part through pkv_decode_step."""
    ref = OS.run(w, items=items, nthreads=nthreads)
    st = device_step(w, partition_tokens)
    tables, nb, pairs = st.plan()
    assert np.array_equal(tables, ref.tables), "block tables differ"
    assert np.array_equal(nb, ref.nblocks)
    assert np.array_equal(pairs, ref.pairs), "copy-on-write pairs differ"
    st.run(fused=fused)
    torch.cuda.synchronize()
    if w.T:
        slots = st.slot_mapping[:w.T].cpu().numpy()
        assert np.array_equal(slots, ref.slots), "slot mapping differs"
    if check_caches:
        ids = torch.from_numpy(ref.pool_ids.astype(np.int64)).cuda()
        for cache, pool in ((st.k_cache, ref.k_pool), (st.v_cache, ref.v_pool)):
            got = cache.view(torch.int16).index_select(0, ids).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, pool), "cache contents differ"
            rest = torch.ones(w.NB, dtype=torch.bool, device="cuda")
            rest[ids] = False
            poison = int(np.array(W.POISON[w.dtype], dtype=np.uint16).view(np.int16))
            untouched = cache.view(torch.int16)[rest]
            assert bool((untouched == poison).all()), "a block outside the step was written"
    got = out_to_double(st.out)
    if items is None:
        mae, mre = assert_attention_close(got, ref.out, w.name)
    else:
        it = np.asarray(items)
        mae, mre = assert_attention_close(got[it[:, 0], it[:, 1]], ref.out[it[:, 0], it[:, 1]],
                                          w.name)
    return {"max_abs": mae, "max_rel": mre, "pairs": len(pairs), "step": st, "ref": ref}
