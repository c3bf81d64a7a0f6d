"""Pins the fp64 oracle to what the pages and the mathematics fix.

No value here comes from the CUDA path.  Stored values are the pages'
(tests/golden/*.json, each with its citation); the rest are closed forms,
invariants, brute force and an independent library routine (torch fp64
softmax on contiguous K/V).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import kernels as K
from oracle import step as OS
from oracle.allocator import BlockAllocatorModel, OutOfBlocks, fork_tables
from tests.trace_replay import GOLDEN, check_expect, load_traces, replay


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- dtypes
def test_f16_decode_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([K.f16_to_double(b) for b in bits.tolist()])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_bf16_decode_matches_torch_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([K.bf16_to_double(b) for b in bits.tolist()])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# ------------------------------------------------------ address translation
def test_token_to_block_examples():
    g = _golden("address_translation.json")
    for ex in g["token_to_block"]:
        bs = ex["block_size"]
        table = np.arange(10, dtype=np.int32)[None, :]  # identity table
        slot = K.slot_mapping(table, [0], [ex["token"]], bs)[0]
        assert divmod(int(slot), bs) == (ex["logical_block"], ex["offset"])


def test_block_table_example_and_slot_of_token_35():
    g = _golden("address_translation.json")["block_table"]
    bs = g["block_size"]
    table = np.array([g["table"]], dtype=np.int32)
    for logical, physical in g["logical_to_physical"]:
        toks = np.arange(logical * bs, (logical + 1) * bs, dtype=np.int32)
        slots = K.slot_mapping(table, np.zeros_like(toks), toks, bs)
        assert np.all(slots // bs == physical)
        assert np.array_equal(slots % bs, np.arange(bs))
    assert K.slot_mapping(table, [0], [35], bs)[0] == g["token_35_slot"]


def test_tokens_to_blocks_examples():
    g = _golden("address_translation.json")
    for ex in g["tokens_to_blocks"]:
        a = BlockAllocatorModel(1000)
        t = []
        a.append(t, 0, ex["tokens"], ex["block_size"])
        assert len(t) == ex["blocks"]
        if "last_block_tokens" in ex:
            # slots of the tokens that land in the last block
            table = np.array([t], dtype=np.int32)
            toks = np.arange(ex["tokens"], dtype=np.int32)
            slots = K.slot_mapping(table, np.zeros_like(toks), toks, ex["block_size"])
            assert int(np.sum(slots // ex["block_size"] == t[-1])) == ex["last_block_tokens"]


@pytest.mark.parametrize("bs", [1, 2, 3, 7, 8, 16, 32, 64])
def test_slot_mapping_brute_force_walk(bs):
    """Enumerate a sequence by walking its table block by block, slot by slot
    (no division anywhere), and compare with the oracle's translation."""
    rng = np.random.default_rng(bs)
    S, MB, NB = 3, 9, 40
    tables = np.stack([rng.permutation(NB)[:MB] for _ in range(S)]).astype(np.int32)
    seq_idx, pos, want = [], [], []
    for s in range(S):
        p = 0
        for lb in range(MB):
            for off in range(bs):
                seq_idx.append(s)
                pos.append(p)
                want.append(int(tables[s, lb]) * bs + off)
                p += 1
    got = K.slot_mapping(tables, np.array(seq_idx), np.array(pos), bs)
    assert np.array_equal(got, np.array(want, dtype=np.int64))


def test_slot_mapping_negative_position_is_skip():
    assert K.slot_mapping(np.zeros((1, 2), np.int32), [0], [-1], 16)[0] == -1


def test_slot_mapping_unmapped_block_is_skip():
    """A position whose logical block has no physical block (-1 in the
    table) gets no slot, whatever its offset."""
    table = np.array([[7, -1]], np.int32)
    got = K.slot_mapping(table, [0, 0, 0], [3, 16, 31], 16)
    assert got.tolist() == [7 * 16 + 3, -1, -1]


# ----------------------------------------------------------- sizes on pages
def test_kv_bytes_formula_matches_pages():
    g = _golden("kv_sizes.json")
    w = W.uniform_decode("one", 5, W.F16, S=1, H=g["heads"], D=g["head_dim"],
                         bs=g["page_size_tokens"], ctx_lo=1, ctx_hi=1, NB=2, MB=1)
    assert w.kv_bytes() == g["kv_bytes_per_token"]
    assert g["heads"] * g["head_dim"] * g["elem_bytes"] == g["k_bytes_per_token"]
    assert g["page_size_tokens"] * g["kv_bytes_per_token"] == g["page_bytes"]
    c = g["capacity_example"]
    pages = int(c["gpu_gb"] * 1024 ** 3 * c["kv_budget_fraction"] / g["page_bytes"])
    assert pages == c["max_pages"] and pages * g["page_size_tokens"] == c["max_tokens"]


def test_concurrency_example_through_the_allocator_model():
    """The pages' admission example: requests that reserve blocks for their
    maximum length fit 7 at a time in a 1000-block pool; the 8th is refused
    whole and takes nothing (all-or-nothing allocation)."""
    c = _golden("kv_sizes.json")["concurrency_example"]
    per = -(-c["max_seq_len"] // c["block_size"])
    assert per == c["blocks_per_request"]
    a = BlockAllocatorModel(c["pool_blocks"])
    admitted = 0
    while True:
        free_before = a.num_free
        try:
            a.alloc(per)
        except OutOfBlocks:
            assert a.num_free == free_before  # nothing taken
            break
        admitted += 1
    assert admitted == c["max_concurrent"]
    assert a.num_free == c["pool_blocks"] - c["max_concurrent"] * per


# ------------------------------------------------------------- allocator
@pytest.mark.parametrize("trace", load_traces(), ids=lambda t: t["name"])
def test_allocator_model_replays_page_traces(trace):
    a = BlockAllocatorModel(trace["num_blocks"], policy=trace["policy"])
    tables, log = replay(trace, a, OutOfBlocks)
    check_expect(trace, a, tables, log)


def test_allocator_model_invariants_random_ops():
    """Random alloc/share/append/release: every block's refcount equals the
    number of tables holding it; free + held = pool; at most one partial
    block per sequence; no block both free and held."""
    rng = np.random.default_rng(7)
    NB, bs = 200, 16
    a = BlockAllocatorModel(NB)
    tables, ctx = {}, {}
    nxt = 0
    for _ in range(3000):
        op = rng.integers(0, 5)
        try:
            if op == 0:
                t, n = [], int(rng.integers(1, 100))
                a.append(t, 0, n, bs)
                tables[nxt], ctx[nxt] = t, n
                nxt += 1
            elif op == 1 and tables:
                r = list(tables)[rng.integers(len(tables))]
                n = int(rng.integers(1, 20))
                a.append(tables[r], ctx[r], n, bs)
                ctx[r] += n
            elif op == 2 and tables:
                src = list(tables)[rng.integers(len(tables))]
                a.incref(tables[src])
                tables[nxt], ctx[nxt] = list(tables[src]), ctx[src]
                nxt += 1
            elif op == 3 and tables:
                r = list(tables)[rng.integers(len(tables))]
                a.decref(tables.pop(r))
                ctx.pop(r)
        except OutOfBlocks:
            pass
        held = {}
        for t in tables.values():
            for b in t:
                held[b] = held.get(b, 0) + 1
        assert held == a.rc
        assert a.num_free + len(held) == NB
        assert not (set(a.free) & set(held))
        for r, t in tables.items():
            assert len(t) == -(-ctx[r] // bs)  # at most one partial block


def test_append_copies_shared_partial_block_then_allocates():
    a = BlockAllocatorModel(20)
    t1 = []
    a.append(t1, 0, 20, 16)  # 2 blocks, second partial (4 tokens)
    t2 = list(t1)
    a.incref(t2)
    pairs = a.append(t2, 20, 1, 16)  # writes into the shared partial block
    assert pairs == [(t1[1], t2[1])] and t2[0] == t1[0] and t2[1] != t1[1]
    assert a.refcount(t1[1]) == 1 and a.refcount(t2[1]) == 1 and a.refcount(t1[0]) == 2
    # a full shared block is never copied: the next token opens a new block
    t3 = list(t1[:1])
    a.incref(t3)
    assert a.append(t3, 16, 1, 16) == [] and len(t3) == 2


def test_append_is_all_or_nothing():
    a = BlockAllocatorModel(3)
    t = []
    a.append(t, 0, 33, 16)
    state = (list(a.free), dict(a.rc), list(t))
    with pytest.raises(OutOfBlocks):
        a.append(t, 33, 16, 16)
    assert (list(a.free), dict(a.rc), list(t)) == state


def test_decref_of_free_block_is_error():
    a = BlockAllocatorModel(4)
    (b,) = a.alloc(1)
    a.decref([b])
    with pytest.raises(ValueError):
        a.decref([b])


# ------------------------------------------------- cache write and copy
def test_reshape_and_cache_writes_token_35_into_block_12_offset_3():
    H, D, bs, NB = 2, 8, 16, 16
    rng = np.random.default_rng(0)
    k = rng.integers(0, 1 << 15, (NB, bs, H, D)).astype(np.uint16)
    v = rng.integers(0, 1 << 15, (NB, bs, H, D)).astype(np.uint16)
    k0, v0 = k.copy(), v.copy()
    key = rng.integers(0, 1 << 15, (2, H, D)).astype(np.uint16)
    val = rng.integers(0, 1 << 15, (2, H, D)).astype(np.uint16)
    table = np.array([[3, 7, 12]], dtype=np.int32)
    slots = K.slot_mapping(table, [0, 0], [35, -1], bs)
    K.reshape_and_cache(k, v, key, val, slots)
    assert np.array_equal(k[12, 3], key[0]) and np.array_equal(v[12, 3], val[0])
    k0[12, 3], v0[12, 3] = key[0], val[0]
    assert np.array_equal(k, k0) and np.array_equal(v, v0)  # nothing else written


def test_copy_blocks_cow_demo_block_1_to_5():
    """The P2 demo's copy-on-write gives req3 block 5 as a copy of block 1."""
    H, D, bs, NB = 2, 8, 16, 10
    rng = np.random.default_rng(1)
    k = rng.integers(0, 1 << 15, (NB, bs, H, D)).astype(np.uint16)
    v = rng.integers(0, 1 << 15, (NB, bs, H, D)).astype(np.uint16)
    k0, v0 = k.copy(), v.copy()
    K.copy_blocks(k, v, [[1, 5]])
    k0[5], v0[5] = k0[1], v0[1]
    assert np.array_equal(k, k0) and np.array_equal(v, v0)


def test_row_of_block_only_changes_storage():
    w = W.small_case(3, S=3, H=2, D=64, bs=16, ctx_lo=1, ctx_hi=60, NB=30)
    full = OS.run(w, nthreads=1)
    # the same inputs stored densely by physical id: identical results
    k = np.full((w.NB, w.bs, w.H, w.D), W.POISON[w.dtype], np.uint16)
    v = k.copy()
    k[w.blocks], v[w.blocks] = w.k_blocks, w.v_blocks
    slots = K.slot_mapping(full.tables, w.seq_idx, w.pos, w.bs)
    K.reshape_and_cache(k, v, w.new_k, w.new_v, slots)
    out = K.decode(w.q, k, v, full.tables, w.context_lens, w.scale, False)
    assert np.array_equal(out, full.out)
    assert np.array_equal(k[full.pool_ids], full.k_pool)


# ------------------------------------------------------------ attention
def _dense_inputs(rng, ctx, H, D, bs, NB, dtype=W.F16):
    """One sequence with random K/V in random blocks; returns everything."""
    nb = -(-ctx // bs)
    table = np.full((1, max(nb, 1)), -1, np.int32)
    table[0, :nb] = rng.permutation(NB)[:nb]
    k = W.normal_bits(np.random.Generator(np.random.SFC64(int(rng.integers(1 << 30)))),
                      (NB, bs, H, D), dtype)
    v = W.normal_bits(np.random.Generator(np.random.SFC64(int(rng.integers(1 << 30)))),
                      (NB, bs, H, D), dtype)
    q = W.normal_bits(np.random.Generator(np.random.SFC64(int(rng.integers(1 << 30)))),
                      (1, H, D), dtype)
    return q, k, v, table


def _as_double(bits, dtype):
    if dtype == W.F16:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _gather(bits, table, ctx, bs):
    toks = [bits[table[0, j // bs], j % bs] for j in range(ctx)]
    return np.stack(toks) if toks else np.zeros((0,) + bits.shape[2:], bits.dtype)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("ctx,bs", [(1, 16), (15, 16), (16, 16), (17, 16), (100, 16), (33, 32), (70, 8)])
def test_decode_equals_contiguous_softmax_attention(ctx, bs, dtype):
    """Against torch fp64 softmax(q K^T * scale) V on the gathered, contiguous K/V."""
    rng = np.random.default_rng(ctx * 100 + bs)
    H, D, NB = 3, 64, 24
    q, k, v, table = _dense_inputs(rng, ctx, H, D, bs, NB, dtype)
    scale = 0.3
    out = K.decode(q, k, v, table, [ctx], scale, dtype == W.BF16)
    Kc = torch.from_numpy(_as_double(_gather(k, table, ctx, bs), dtype))  # [ctx, H, D]
    Vc = torch.from_numpy(_as_double(_gather(v, table, ctx, bs), dtype))
    Q = torch.from_numpy(_as_double(q, dtype))[0]                          # [H, D]
    logits = torch.einsum("hd,jhd->hj", Q, Kc) * scale
    ref = torch.einsum("hj,jhd->hd", torch.softmax(logits, dim=-1), Vc).numpy()
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-12)


def test_decode_placement_invariance_bit_identical():
    """The same logical K/V under two different physical placements."""
    rng = np.random.default_rng(11)
    H, D, bs, NB, ctx = 2, 64, 16, 20, 75
    q, k, v, table = _dense_inputs(rng, ctx, H, D, bs, NB)
    out1 = K.decode(q, k, v, table, [ctx], 0.125, False)
    perm = rng.permutation(NB)           # block b moves to perm[b]
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm], v2[perm] = k, v
    table2 = perm[table].astype(np.int32)
    out2 = K.decode(q, k2, v2, table2, [ctx], 0.125, False)
    assert np.array_equal(out1, out2)


def test_decode_closed_forms():
    rng = np.random.default_rng(5)
    H, D, bs, NB = 2, 64, 16, 12
    q, k, v, table = _dense_inputs(rng, 40, H, D, bs, NB)
    vd = _as_double(v, W.F16)
    kd = _as_double(k, W.F16)
    qd = _as_double(q, W.F16)
    b0 = table[0, 0]
    # one token: the output is that token's V exactly
    out = K.decode(q, k, v, table, [1], 0.125, False)
    assert np.array_equal(out[0], vd[b0, 0])
    # two tokens: V0 + sigmoid(z1 - z0) (V1 - V0)
    out = K.decode(q, k, v, table, [2], 0.125, False)
    z = [0.125 * np.dot(qd[0, h], kd[b0, j, h]) for j in range(2) for h in range(H)]
    for h in range(H):
        z0, z1 = 0.125 * np.dot(qd[0, h], kd[b0, 0, h]), 0.125 * np.dot(qd[0, h], kd[b0, 1, h])
        sig = 1.0 / (1.0 + math.exp(-(z1 - z0)))
        np.testing.assert_allclose(out[0, h], vd[b0, 0, h] + sig * (vd[b0, 1, h] - vd[b0, 0, h]),
                                   rtol=1e-13, atol=1e-14)
    # q = 0: uniform weights -> mean of V over the context
    qz = np.zeros_like(q)
    out = K.decode(qz, k, v, table, [40], 0.125, False)
    Vc = _as_double(_gather(v, table, 40, bs), W.F16)
    np.testing.assert_allclose(out[0], Vc.mean(axis=0), rtol=1e-13, atol=1e-14)
    # all keys equal -> mean of V
    ke = np.empty_like(k)
    ke[...] = k[b0, 0][None, None]
    out = K.decode(q, ke, v, table, [40], 0.125, False)
    np.testing.assert_allclose(out[0], Vc.mean(axis=0), rtol=1e-13, atol=1e-14)
    # V constant -> that constant
    vc = np.full_like(v, np.float16(0.75).view(np.uint16))
    out = K.decode(q, k, vc, table, [40], 0.125, False)
    np.testing.assert_allclose(out[0], 0.75, rtol=1e-14)
    # empty context -> zeros
    out = K.decode(q, k, v, table, [0], 0.125, False)
    assert np.array_equal(out[0], np.zeros((H, D)))


def test_decode_scale_and_items_and_threads():
    w = W.small_case(9, S=4, H=3, D=64, bs=16, ctx_lo=1, ctx_hi=90)
    a = OS.run(w, nthreads=1)
    b = OS.run(w, nthreads=3)
    assert np.array_equal(a.out, b.out)
    items = np.array([[1, 2], [3, 0]])
    c = OS.run(w, nthreads=2, items=items)
    for s, h in items:
        assert np.array_equal(c.out[s, h], a.out[s, h])
    assert np.isnan(c.out[0, 0]).all()


# ------------------------------------------------------- step workloads
def test_shared_prefix_cow_step_copies_seven_of_eight():
    """First write after a fork into a shared partial block: samples 0-6
    see refcount > 1 and copy, the last sees refcount 1 and writes in place."""
    w = W.shared_prefix(cow=True, prompts=3, samples=8, prefix=64)
    a, tables, nb, pairs = OS.plan(w)
    assert len(pairs) == 3 * 7
    for p in range(3):
        last = (w.ctx_before[p * 8]) // w.bs
        srcs = {int(s) for s, _ in pairs[p * 7:(p + 1) * 7]}
        assert srcs == {int(w.tables_pre[p * 8, last])}
        assert tables[p * 8 + 7, last] == w.tables_pre[p * 8, last]  # in place
        assert len({int(tables[p * 8 + j, last]) for j in range(8)}) == 8


def test_shared_prefix_full_blocks_need_no_copy():
    w = W.shared_prefix(cow=False, prompts=2, samples=8, prefix=64, tail_hi=40)
    _, _, _, pairs = OS.plan(w)
    assert len(pairs) == 0


def test_continuous_batching_step_allocations():
    w = W.continuous_batching_bf16(S=40, NB=3000)
    a, tables, nb, pairs = OS.plan(w)
    fresh = w.notes["fresh"]
    assert len(fresh) == round(0.12 * 40)
    for s in fresh:
        assert nb[s] == 20  # a 320-token prefill takes 20 blocks
    assert len(pairs) == 0
    held = np.unique(tables[tables >= 0])
    assert a.num_free + len(held) == w.NB
    # at most one partial block per sequence
    assert np.all(nb == -(-w.context_lens // w.bs))


def test_swap_blocks_round_trip_and_fancy_indexing():
    """Swap-out then swap-in into other blocks ([P1] 3.3.3): every block
    lands where numpy's fancy indexing puts it, nothing else changes."""
    rng = np.random.default_rng(21)
    H, D, bs, NBg, NBh = 2, 8, 16, 12, 6
    gk = rng.integers(0, 1 << 15, (NBg, bs, H, D)).astype(np.uint16)
    gv = rng.integers(0, 1 << 15, (NBg, bs, H, D)).astype(np.uint16)
    hk = np.zeros((NBh, bs, H, D), np.uint16)
    hv = np.zeros_like(hk)
    out = [[3, 5], [7, 0], [11, 2]]              # gpu block -> host block
    K.swap_blocks(hk, hv, gk, gv, out)
    want_k, want_v = np.zeros_like(hk), np.zeros_like(hv)
    src, dst = np.array(out).T
    want_k[dst], want_v[dst] = gk[src], gv[src]
    assert np.array_equal(hk, want_k) and np.array_equal(hv, want_v)
    back = [[5, 1], [0, 4], [2, 9]]              # host block -> other gpu blocks
    g2k, g2v = gk.copy(), gv.copy()
    K.swap_blocks(g2k, g2v, hk, hv, back)
    for (g0, h), (h2, g1) in zip(out, back):
        assert h == h2
        assert np.array_equal(g2k[g1], gk[g0]) and np.array_equal(g2v[g1], gv[g0])
    untouched = [b for b in range(NBg) if b not in (1, 4, 9)]
    assert np.array_equal(g2k[untouched], gk[untouched])


# ------------------------------------------------------------ beam search
# Values worked out by hand from the pages' rules (share = one more hold per
# block, a block returns to the free list when its count reaches 0, copy on
# write into a block held by more than one table) and the oracle's readings
# (a stack free list: a fresh pool of 12 hands out 11, 10, 9, ...; a fork
# takes the new holds first, then releases the old tables row by row, slot
# by slot).  Sources: "3.3 页面级显存管理" 3.3.2 (share_blocks); notes on
# "vLLM: Easy, Fast, and Cheap LLM Serving with PagedAttention", section
# "Memory Sharing与写时复制" (beams share blocks until they diverge).
def _fork_fixture():
    a = BlockAllocatorModel(12)
    t0 = a.alloc(3)                                  # request 0, beam 0
    a.incref([t0[0]])
    t1 = [t0[0]] + a.alloc(2)                        # request 0, beam 1
    t2 = a.alloc(2)                                  # request 1, beam 0
    a.incref([t2[0]])
    t3 = [t2[0]] + a.alloc(1)                        # request 1, beam 1
    assert [t0, t1, t2, t3] == [[11, 10, 9], [11, 8, 7], [6, 5], [6, 4]]
    assert a.rc == {11: 2, 10: 1, 9: 1, 8: 1, 7: 1, 6: 2, 5: 1, 4: 1}
    return a, [t0, t1, t2, t3]


FORK_PINS = [
    # parents, tables after, refcounts after, free list after (top last),
    # the ids the next allocation hands out
    ([1, 1, 3, 2],
     [[11, 8, 7], [11, 8, 7], [6, 4], [6, 5]],
     {11: 2, 8: 2, 7: 2, 6: 2, 5: 1, 4: 1},
     [0, 1, 2, 3, 10, 9], [9, 10, 3]),
    # two rows lose every child: row 0 frees 10 then 9, row 2 frees 5
    ([1, 1, 3, 3],
     [[11, 8, 7], [11, 8, 7], [6, 4], [6, 4]],
     {11: 2, 8: 2, 7: 2, 6: 2, 4: 2},
     [0, 1, 2, 3, 10, 9, 5], [5, 9, 10, 3]),
]


def _fork_pin_holds(fork):
    for parents, tables, rc, free, nxt in FORK_PINS:
        a, old = _fork_fixture()
        new = fork(a, old, parents)
        if not (new == tables and a.rc == rc and a.free == free and a.alloc(len(nxt)) == nxt):
            return False
    return True


def test_fork_tables_hand_worked():
    assert _fork_pin_holds(fork_tables)


def test_fork_pin_catches_release_in_reverse_row_order():
    """A planted mistake (old tables released last row first) changes which
    blocks the next allocation receives, and the pin sees it."""
    def reversed_rows(alloc, tables, parents):
        new = [list(tables[int(p)]) for p in parents]
        for t in new:
            alloc.incref(t)
        for t in reversed(tables):
            alloc.decref(t)
        return new
    assert not _fork_pin_holds(reversed_rows)


def _beam_fixture():
    """2 requests x 2 beams, 1 head, D = 8, fp16, blocks of 4 tokens, pool of
    10.  Request 0's prompt is 6 tokens in blocks [7, 3]; request 1's is 4
    tokens in block [5]; both beams of a request hold the prompt's blocks.
    Every V row is one constant (prompt token p of request 0: p; of request
    1: 10 + p; new tokens: 16, 20, 24, 28 at step 1 and 32, 40, 48, 56 at
    step 2, by beam) and q = 0, so each output is the plain mean of the V
    values on the sequence's path."""
    f16 = W.F16
    S, H, D, bs, NB, MB = 4, 1, 8, 4, 10, 3
    poison = W.POISON[f16]
    blocks = np.array([3, 5, 7], dtype=np.int32)

    def rows(vals):                                  # one block of V (or K)
        out = np.full((bs, H, D), poison, dtype=np.uint16)
        for off, v in enumerate(vals):
            out[off] = W.to_bits(np.full((H, D), v, np.float32), f16)
        return out
    v_blocks = np.stack([rows([4, 5]), rows([10, 11, 12, 13]), rows([0, 1, 2, 3])])
    k_blocks = np.stack([rows([1, 1]), rows([1, 1, 1, 1]), rows([1, 1, 1, 1])])
    tables = np.array([[7, 3, -1], [7, 3, -1], [5, -1, -1], [5, -1, -1]], dtype=np.int32)
    empty = np.zeros((0, H, D), dtype=np.uint16)
    init = W.Workload(name="beam_pin", dtype=f16, S=S, H=H, D=D, bs=bs, NB=NB, MB=MB,
                      scale=1.0 / math.sqrt(D), ctx_before=np.array([6, 6, 4, 4], np.int32),
                      n_new=np.zeros(S, np.int32), tables_pre=tables,
                      nblocks_pre=np.array([2, 2, 1, 1], np.int32),
                      initial_free=np.array([0, 1, 2, 4, 6, 8, 9], np.int32),
                      blocks=blocks, k_blocks=k_blocks, v_blocks=v_blocks,
                      q=np.zeros((S, H, D), np.uint16), new_k=empty, new_v=empty,
                      seq_idx=np.zeros(0, np.int32), pos=np.zeros(0, np.int32))
    new_v = np.stack([W.to_bits(np.repeat(np.array(v, np.float32)[:, None, None], D, 2), f16)
                      for v in ([16, 20, 24, 28], [32, 40, 48, 56])])
    new_k = W.to_bits(np.ones((2, S, H, D), np.float32), f16)
    return W.BeamWorkload(init=init, beams=2,
                          parents=np.array([[1, 0, 3, 3], [0, 0, 2, 3]], np.int32),
                          new_k=new_k, new_v=new_v, q=np.zeros((2, S, H, D), np.uint16))


# Step 1: the fork changes no count.  Beam 0 writes position 6 into block 3,
# held twice, so it copies 3 to the top of the free list (9); beam 1 then
# holds 3 alone and writes in place; beams 2 and 3 open blocks 8 and 6.
# Step 2: old beam 1 has no child, so its block 3 drops to 0 and goes back
# on top of the free list; beam 0's write into the shared block 9 copies it
# into that same block 3.
BEAM_PINS = [
    ([[7, 9, -1], [7, 3, -1], [5, 8, -1], [5, 6, -1]], [[3, 9]],
     [9 * 4 + 2, 3 * 4 + 2, 8 * 4 + 0, 6 * 4 + 0],
     [(15 + 16) / 7, (15 + 20) / 7, (46 + 24) / 5, (46 + 28) / 5]),
    ([[7, 3, -1], [7, 9, -1], [5, 8, -1], [5, 6, -1]], [[9, 3]],
     [3 * 4 + 3, 9 * 4 + 3, 8 * 4 + 1, 6 * 4 + 1],
     [(15 + 16 + 32) / 8, (15 + 16 + 40) / 8, (46 + 24 + 48) / 6, (46 + 28 + 56) / 6]),
]


def _beam_pin_holds():
    steps = list(OS.run_beam(_beam_fixture(), nthreads=1))
    if len(steps) != len(BEAM_PINS):
        return False
    for (bt, pairs, slots, _k, _v, _ids, out), (t, p, sl, mean) in zip(steps, BEAM_PINS):
        want = np.broadcast_to(np.array(mean)[:, None, None], out.shape)
        if not (np.array_equal(bt, t) and np.array_equal(pairs, np.array(p).reshape(-1, 2))
                and np.array_equal(slots, sl) and np.allclose(out, want, rtol=0, atol=1e-12)):
            return False
    return True


def test_run_beam_hand_worked():
    assert _beam_pin_holds()


def test_beam_pin_catches_slot_one_past_the_context(monkeypatch):
    """A planted mistake (the new token mapped at position ctx + 1 instead of
    ctx) moves the write and the slots, and the pin sees it."""
    real = OS.kernels.slot_mapping
    monkeypatch.setattr(OS.kernels, "slot_mapping",
                        lambda bt, seq, pos, bs: real(bt, seq, np.asarray(pos) + 1, bs))
    assert not _beam_pin_holds()
