"""Host-side tests of libpagedkv.so that need no GPU: every symbol the header
declares is exported, argument checks reject bad calls before any launch,
and the C++ block allocator matches the oracle's allocator model."""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_cache_162_gb300 as P
from paged_kv_cache_162_gb300 import _lib as L
from paged_kv_cache_162_gb300.allocator import BlockAllocator, OutOfBlocks
from oracle.allocator import BlockAllocatorModel, OutOfBlocks as ModelOOM
from tests.trace_replay import check_expect, load_traces, replay

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pkv_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert len(names) >= 20
    lib = L.lib()
    for n in names:
        assert hasattr(lib, n), n
        assert n in L.SIGNATURES, f"binding lacks {n}"


def header_constants():
    """Every PKV_* constant the header gives a value: #defines and enumerators."""
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    consts = {}
    for name, val in re.findall(r"#define\s+(PKV_\w+)\s+(0x[0-9a-fA-F]+|[0-9]+)\b", text):
        consts[name] = int(val, 0)
    for name, val, shift in re.findall(r"#define\s+(PKV_\w+)\s+\(([0-9]+)u\s*<<\s*(\d+)\)", text):
        consts[name] = int(val) << int(shift)
    for name, val in re.findall(r"\b(PKV_\w+)\s*=\s*([0-9]+)", text):
        consts[name] = int(val)
    return consts


def test_binding_constants_equal_the_header():
    """The Python names carry the header's values, device error bits
    included, so a bit read back from the device decodes the same way."""
    consts = header_constants()
    for name in ["PKV_OK", "PKV_ERR_INVALID_ARG", "PKV_ERR_UNSUPPORTED", "PKV_ERR_OOM",
                 "PKV_ERR_WORKSPACE", "PKV_ERR_CUDA", "PKV_ERR_HOST_MEMORY", "PKV_F16", "PKV_BF16",
                 "PKV_DEVERR_BLOCK_ID", "PKV_DEVERR_SLOT", "PKV_DEVERR_CONTEXT",
                 "PKV_DEVERR_POSITION", "PKV_DEVERR_GROUP", "PKV_DEVERR_TIMEOUT",
                 "PKV_NOALLOC_SCRATCH_BYTES", "PKV_SWAP_OUT", "PKV_SWAP_IN"]:
        assert name in consts, f"header lacks {name}"
        assert getattr(L, name) == consts[name], name
    bits = [v for k, v in consts.items() if k.startswith("PKV_DEVERR_")]
    assert len(bits) == 6
    assert all(b and b & (b - 1) == 0 for b in bits) and len(set(bits)) == len(bits)


def test_version_and_workspace_size():
    assert "sm_103a" in P.pkv_version()
    ws = P.pkv_decode_workspace_size(64, 32, 128, 2048, 256)
    # at least the fp32 partials: S*H*parts*(D+2)*4 bytes
    assert ws >= 64 * 32 * 8 * 130 * 4
    assert P.pkv_decode_workspace_size(64, 32, 96, 2048, 256) == 0   # head_dim 96 not built
    assert P.pkv_decode_workspace_size(64, 32, 128, 2048, 24) == 0   # not a multiple of 16
    assert P.pkv_decode_workspace_size(0, 32, 128, 2048, 0) > 0


def _decode_args(**kw):
    a = dict(out=16, q=16, k_cache=16, v_cache=16, block_tables=16, context_lens=16, S=2, H=4,
             D=128, bs=16, NB=8, MB=4, max_context_len=0, scale=0.1, dtype=L.PKV_F16,
             partition_tokens=0, workspace=256, workspace_bytes=1 << 30, stream=0)
    a.update(kw)
    return a


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), L.PKV_ERR_UNSUPPORTED),
    (dict(bs=24), L.PKV_ERR_UNSUPPORTED),
    (dict(dtype=7), L.PKV_ERR_INVALID_ARG),
    (dict(q=0), L.PKV_ERR_INVALID_ARG),
    (dict(out=18), L.PKV_ERR_INVALID_ARG),          # misaligned
    (dict(workspace=272), L.PKV_ERR_INVALID_ARG),   # workspace not 256-aligned
    (dict(workspace_bytes=100), L.PKV_ERR_WORKSPACE),
    (dict(max_context_len=65), L.PKV_ERR_INVALID_ARG),  # > MB*bs
    (dict(partition_tokens=40), L.PKV_ERR_INVALID_ARG),
    (dict(bs=32, partition_tokens=48), L.PKV_ERR_INVALID_ARG),
    (dict(scale=float("nan")), L.PKV_ERR_INVALID_ARG),
    (dict(scale=float("inf")), L.PKV_ERR_INVALID_ARG),
    (dict(H=0), L.PKV_ERR_INVALID_ARG),
    # one past the limits of the packed (sequence << 16 | partition) items
    (dict(S=32768), L.PKV_ERR_INVALID_ARG),
    (dict(S=1, MB=65536, bs=64, max_context_len=65536 * 64, partition_tokens=64),
     L.PKV_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_arguments_before_launch(kw, status):
    a = _decode_args(**kw)
    with pytest.raises(L.PkvError) as e:
        P.pkv_paged_attention_decode(**a)
    assert e.value.status == status
    assert P.pkv_last_error_string()


def test_decode_with_no_sequences_is_a_noop():
    P.pkv_paged_attention_decode(**_decode_args(S=0, out=0, q=0))


def test_cache_ops_reject_bad_arguments():
    with pytest.raises(L.PkvError) as e:
        P.pkv_reshape_and_cache(16, 16, 16, 16, 16, 4, 4, 80, 16, 8, L.PKV_F16, 0)
    assert e.value.status == L.PKV_ERR_UNSUPPORTED
    with pytest.raises(L.PkvError) as e:
        P.pkv_reshape_and_cache(16, 0, 16, 16, 16, 4, 4, 64, 16, 8, L.PKV_F16, 0)
    assert e.value.status == L.PKV_ERR_INVALID_ARG
    with pytest.raises(L.PkvError) as e:
        P.pkv_copy_blocks(16, 24, 16, 3, 4, 64, 16, 8, L.PKV_F16, 0)
    assert e.value.status == L.PKV_ERR_INVALID_ARG
    with pytest.raises(L.PkvError):
        P.pkv_compute_slot_mapping(16, 16, 0, 16, 4, 1, 4, 16, 0)
    # empty work is a no-op that touches nothing
    P.pkv_reshape_and_cache(0, 0, 0, 0, 0, 0, 4, 64, 16, 8, L.PKV_F16, 0)
    P.pkv_copy_blocks(0, 0, 0, 0, 4, 64, 16, 8, L.PKV_F16, 0)
    P.pkv_compute_slot_mapping(0, 0, 0, 0, 0, 1, 4, 16, 0)


# ------------------------------------------------------------- allocator
@pytest.mark.parametrize("trace", [t for t in load_traces() if t["policy"] == "lifo"],
                         ids=lambda t: t["name"])
def test_library_allocator_replays_page_traces(trace):
    a = BlockAllocator(trace["num_blocks"])
    tables, log = replay(trace, a, OutOfBlocks)
    check_expect(trace, a, tables, log)


def test_library_allocator_matches_model_on_random_ops():
    """Random alloc / share / append (with CoW) / release / cow sequences:
    ids, copy pairs, refcounts and the free count agree after every op."""
    rng = np.random.default_rng(123)
    NB, bs = 300, 16
    perm = rng.permutation(NB)
    held0 = perm[:40]
    free0 = perm[40:]
    lib_a = BlockAllocator(NB, initial_free=free0)
    mod_a = BlockAllocatorModel(NB, initial_free=free0)
    tables = {0: [int(b) for b in held0[:20]], 1: [int(b) for b in held0[20:]]}
    ctx = {0: 20 * bs - 3, 1: 20 * bs}
    nxt = 2
    for step in range(4000):
        op = int(rng.integers(0, 6))
        keys = list(tables)
        outcome = []
        for a, oom in ((lib_a, OutOfBlocks), (mod_a, ModelOOM)):
            t2 = {k: list(v) for k, v in tables.items()}
            try:
                if op == 0:
                    n = int(rng.integers(0, 5)) if a is lib_a else n
                    res = a.alloc(n)
                elif op == 1 and keys:
                    r = keys[int(rng.integers(len(keys)))] if a is lib_a else r
                    k = int(rng.integers(1, 40)) if a is lib_a else k
                    res = (a.append(t2[r], ctx[r], k, bs), t2[r])
                elif op == 2 and keys:
                    r = keys[int(rng.integers(len(keys)))] if a is lib_a else r
                    a.incref(t2[r])
                    res = "shared"
                elif op == 3 and keys:
                    r = keys[int(rng.integers(len(keys)))] if a is lib_a else r
                    res = a.decref(t2[r])
                elif op == 4 and keys:
                    r = keys[int(rng.integers(len(keys)))] if a is lib_a else r
                    j = int(rng.integers(len(t2[r]))) if (a is lib_a and t2[r]) else (j if t2[r] else 0)
                    res = a.cow(t2[r][j]) if t2[r] else None
                else:
                    res = None
            except oom:
                res = "oom"
            outcome.append((res, a.num_free, a.num_shared, t2))
        (r1, f1, s1, t1), (r2, f2, s2, _) = outcome
        assert r1 == r2 and f1 == f2 and s1 == s2, (step, op, outcome)
        # apply the op to the harness's view of the tables
        if op == 0 and r1 != "oom":
            tables[nxt] = list(r1)
            ctx[nxt] = len(r1) * bs
            nxt += 1
        elif op == 1 and keys and r1 != "oom":
            tables[r] = t1[r]
            ctx[r] += k
        elif op == 2 and keys:
            tables[nxt] = list(tables[r])
            ctx[nxt] = ctx[r]
            nxt += 1
        elif op == 3 and keys:
            del tables[r]
            del ctx[r]
        elif op == 4 and keys and r1 not in ("oom", None):
            new, copied = r1
            if copied:
                # the writer now holds `new` instead of the shared block
                tables[r][j] = new
        for b in range(0, NB, 7):
            assert lib_a.refcount(b) == mod_a.refcount(b)


def test_library_allocator_errors_change_nothing():
    a = BlockAllocator(8)
    ids = a.alloc(3)
    with pytest.raises(OutOfBlocks):
        a.alloc(6)
    assert a.num_free == 5
    with pytest.raises(L.PkvError):
        a.decref([ids[0], ids[0]])          # held once, released twice
    assert a.refcount(ids[0]) == 1 and a.num_free == 5
    with pytest.raises(L.PkvError):
        a.incref([ids[0], 99])
    assert a.refcount(ids[0]) == 1
    t = list(ids)
    a.incref(t)
    with pytest.raises(OutOfBlocks):
        a.append(t, 40, 100, 16)             # needs 2 CoW copies + 7 blocks, 5 free
    assert t == ids and a.num_free == 5 and a.refcount(ids[2]) == 2
    with pytest.raises(L.PkvError):
        BlockAllocator(4, initial_free=[0, 0])


def test_library_allocator_create_with_order_pops_last_first():
    a = BlockAllocator(10, initial_free=[3, 8, 1])
    assert a.num_free == 3 and a.refcount(0) == 1 and a.refcount(3) == 0
    assert a.alloc(2) == [1, 8]
    assert a.decref([0]) == 1 and a.alloc(1) == [0]


def test_library_beam_fork_matches_model_at_full_size():
    """16 requests x 4 beams, LLaMA-7B-shaped pool, 8 steps of native fork +
    append_batch: the same tables, copies, free and shared counts as the
    model's fork_tables + append."""
    import workloads as W
    from oracle.allocator import fork_tables as model_fork
    from oracle.step import rebuild_allocator

    bw = W.beam_search()
    w = bw.init
    mod = rebuild_allocator(w)
    lib = BlockAllocator(w.NB, w.initial_free)
    ids, counts = np.unique(w.tables_pre[w.tables_pre >= 0], return_counts=True)
    for b, c in zip(ids.tolist(), counts.tolist()):
        if c > 1:
            lib.incref([b] * (c - 1))
    tm = [w.tables_pre[s, :w.nblocks_pre[s]].tolist() for s in range(w.S)]
    tl = np.ascontiguousarray(w.tables_pre.copy())
    nbl = np.ascontiguousarray(w.nblocks_pre.astype(np.int32))
    ctx = w.ctx_before.astype(np.int64)
    total_pairs = 0
    for i in range(bw.steps):
        tm = model_fork(mod, tm, bw.parents[i])
        lib.fork(tl, nbl, bw.parents[i])
        ctx = ctx[bw.parents[i]]
        pm = []
        for b in range(w.S):
            pm += mod.append(tm[b], int(ctx[b]), 1, w.bs)
        pl = lib.append_batch(tl, nbl, ctx, np.ones(w.S), w.bs)
        assert [tuple(p) for p in pl.tolist()] == pm
        total_pairs += len(pm)
        ctx += 1
        for b in range(w.S):
            assert tl[b, :nbl[b]].tolist() == tm[b]
        assert mod.num_free == lib.num_free and mod.num_shared == lib.num_shared
    assert total_pairs > 0


def test_library_fork_and_append_batch_errors():
    a = BlockAllocator(6)
    t = np.full((2, 4), -1, np.int32)
    nb = np.zeros(2, np.int32)
    a.append_batch(t, nb, [0, 0], [20, 10], 16)          # rows: 2 blocks and 1 block
    assert nb.tolist() == [2, 1] and a.num_free == 3
    before = (t.copy(), nb.copy(), a.num_free)
    with pytest.raises(L.PkvError):
        a.fork(t, nb, [0, 2])                              # parent out of range: nothing changes
    assert np.array_equal(t, before[0]) and np.array_equal(nb, before[1]) and a.num_free == 3
    a.fork(t, nb, [0, 0])                                  # both rows share row 0's blocks
    assert nb.tolist() == [2, 2] and a.num_free == 4 and a.num_shared == 2
    # 40 more tokens each: row 0 copies its shared partial block and takes 2
    # new blocks (1 left); row 1 then owns its partial block alone but needs
    # 2 new blocks: out of blocks, row 1 untouched
    with pytest.raises(OutOfBlocks):
        a.append_batch(t, nb, [20, 20], [40, 40], 16)
    assert nb.tolist() == [4, 2] and a.num_free == 1
    assert t[1, :2].tolist() == t[0, :1].tolist() + [t[1, 1]] and t[1, 2] == -1


def test_beam_inputs_layout():
    """pkv_beam_inputs_bytes: tables, lengths, positions and sequence index
    (int32) and room for two copy pairs (2 x 2 int64) per sequence, each
    part on a 256-byte boundary."""
    up = lambda x: (x + 255) // 256 * 256
    for S, MB in [(1, 1), (64, 66), (7, 13), (256, 128)]:
        want = up(4 * S * MB) + 3 * up(4 * S) + up(32 * S)
        assert L.pkv_beam_inputs_bytes(S, MB) == want
    assert L.pkv_beam_inputs_bytes(0, 4) == 0 and L.pkv_beam_inputs_bytes(4, 0) == 0


def test_beam_step_rejects_bad_calls_before_changing_anything():
    """Every argument check of pkv_beam_step runs before the fork: a bad
    call leaves tables, lengths and refcounts as they were (no GPU needed,
    nothing is launched)."""
    S, MB, bs = 4, 4, 16
    a = BlockAllocator(32)
    ids = a.alloc(2)
    a.incref([ids[0], ids[0], ids[0], ids[1], ids[1], ids[1]])
    tables = np.full((S, MB), -1, dtype=np.int32)
    tables[:, 0], tables[:, 1] = ids[0], ids[1]
    nb = np.full(S, 2, dtype=np.int32)
    ctx = np.full(S, 20, dtype=np.int32)
    nbytes = L.pkv_beam_inputs_bytes(S, MB)
    stg = np.zeros(nbytes + 512, dtype=np.uint8)
    base = stg.ctypes.data
    aligned = base + (-base) % 256
    fake_dev = 1 << 20  # 256-byte aligned; never reached by these calls

    def call(parents, staging=aligned, inputs_bytes=nbytes, context=ctx):
        return L.lib().pkv_beam_step(a._h, tables.ctypes.data, nb.ctypes.data, context.ctypes.data,
                                     np.ascontiguousarray(parents, dtype=np.int32).ctypes.data,
                                     S, MB, staging, fake_dev, inputs_bytes, 0, 0, 0, 0, 0, 0, 0,
                                     0, 0, 4, 64, bs, 32, 0.125, L.PKV_F16, 0, 0, 0,
                                     ctypes.addressof(ctypes.c_int32()), 0)

    before = (tables.copy(), nb.copy(), ctx.copy(), [a.refcount(i) for i in ids], a.num_free)
    full = np.full(S, MB * bs, dtype=np.int32)
    for status, kw in [
        (call([0, 1, 2, 4]), "parent out of range"),
        (call([0, -1, 2, 3]), "negative parent"),
        (call([0, 1, 2, 3], staging=aligned + 16), "misaligned staging"),
        (call([0, 1, 2, 3], inputs_bytes=nbytes - 1), "buffers too small"),
        (call([0, 1, 2, 3], context=full), "context would pass the table"),
    ]:
        assert status == L.PKV_ERR_INVALID_ARG, kw
        assert np.array_equal(tables, before[0]) and np.array_equal(nb, before[1]), kw
        assert np.array_equal(ctx, before[2]), kw
        assert [a.refcount(i) for i in ids] == before[3] and a.num_free == before[4], kw


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_library_fork_random_parents_match_model(seed):
    """Forks with parents drawn from every row (rows with no child, one
    child and many, shared and private blocks, ragged lengths) followed by
    appends of 1..20 tokens: tables, copy pairs, every refcount and the free
    list order (seen through the next allocations) equal the model's."""
    from oracle.allocator import fork_tables as model_fork
    rng = np.random.default_rng(seed)
    NB, bs, S, MB = 3000, 8, 12, 200
    lib_a, mod_a = BlockAllocator(NB), BlockAllocatorModel(NB)
    ctx = rng.integers(1, 60, size=S).astype(np.int64)
    tm = [[] for _ in range(S)]
    for s in range(S):
        mod_a.append(tm[s], 0, int(ctx[s]), bs)
    tl = np.full((S, MB), -1, dtype=np.int32)
    nbl = np.zeros(S, dtype=np.int32)
    lib_a.append_batch(tl, nbl, np.zeros(S), ctx, bs)
    for step in range(60):
        parents = rng.integers(0, S, size=S)
        if step % 5 == 0:
            parents[:] = rng.integers(0, S)  # one row takes over every sequence
        tm = model_fork(mod_a, tm, parents)
        lib_a.fork(tl, nbl, parents)
        ctx = ctx[parents]
        n_new = rng.integers(1, 21, size=S)
        pm = []
        for s in range(S):
            pm += mod_a.append(tm[s], int(ctx[s]), int(n_new[s]), bs)
        pl = lib_a.append_batch(tl, nbl, ctx, n_new, bs)
        assert [tuple(p) for p in pl.tolist()] == pm, step
        ctx = ctx + n_new
        for s in range(S):
            assert tl[s, :nbl[s]].tolist() == tm[s], (step, s)
        assert lib_a.num_free == mod_a.num_free and lib_a.num_shared == mod_a.num_shared
        assert all(lib_a.refcount(b) == mod_a.refcount(b) for b in range(NB)), step
    assert ctx.max() <= MB * bs
    assert list(lib_a.alloc(50)) == list(mod_a.alloc(50))  # the free lists agree in order


def test_beam_step_out_of_blocks_after_the_fork():
    """A pool too small for the appends: the fork stands, the sequences
    before the failing one are extended, lengths are unchanged and nothing
    is launched (the error comes before any CUDA call)."""
    S, MB, bs = 2, 4, 16
    a = BlockAllocator(2)
    ids = a.alloc(2)  # pops 1, then 0
    tables = np.full((S, MB), -1, dtype=np.int32)
    tables[0, 0], tables[1, 0] = ids[0], ids[1]
    nb = np.ones(S, dtype=np.int32)
    ctx = np.full(S, bs, dtype=np.int32)  # full blocks: each append needs a new one
    nbytes = L.pkv_beam_inputs_bytes(S, MB)
    stg = np.zeros(nbytes + 512, dtype=np.uint8)
    aligned = stg.ctypes.data + (-stg.ctypes.data) % 256
    npairs = ctypes.c_int32(-1)
    parents = np.zeros(S, dtype=np.int32)  # both continue sequence 0
    status = L.lib().pkv_beam_step(a._h, tables.ctypes.data, nb.ctypes.data, ctx.ctypes.data,
                                   parents.ctypes.data, S, MB, aligned, 1 << 20, nbytes, 0, 0, 0,
                                   0, 0, 0, 0, 0, 0, 4, 64, bs, 2, 0.125, L.PKV_F16, 0, 0, 0,
                                   ctypes.addressof(npairs), 0)
    assert status == L.PKV_ERR_OOM
    # fork: both rows hold sequence 0's block; sequence 1's block was freed
    # and handed to sequence 0's append, then the pool ran dry
    assert tables[0, :2].tolist() == [ids[0], ids[1]] and nb[0] == 2
    assert tables[1, :1].tolist() == [ids[0]] and nb[1] == 1
    assert ctx.tolist() == [bs, bs] and npairs.value == 0
    assert a.refcount(ids[0]) == 2 and a.refcount(ids[1]) == 1 and a.num_free == 0


def test_in_place_arrays_must_be_int32_contiguous():
    """fork / append_batch / append_row write the caller's arrays in place:
    a wrong dtype or a strided view is refused, not silently copied."""
    a = BlockAllocator(16)
    tables = np.full((2, 4), -1, dtype=np.int32)
    nb = np.zeros(2, dtype=np.int32)
    with pytest.raises(L.PkvError):
        a.fork(tables.astype(np.int64), nb, [0, 1])
    with pytest.raises(L.PkvError):
        a.append_batch(tables, nb.astype(np.int64), [0, 0], [1, 1], 16)
    with pytest.raises(L.PkvError):
        a.append_row(np.full(8, -1, dtype=np.int32)[::2], 0, 0, 1, 16)
    assert a.num_free == 16


def test_check_copy_pairs_accepts_allocator_copies_and_names_the_bad_pair():
    """pkv_copy_blocks' precondition, checked on the host: ids in the pool,
    no destination twice, no destination that is also a source."""
    from paged_kv_cache_162_gb300.allocator import check_copy_pairs
    a = BlockAllocator(40)
    t = np.full((8, 4), -1, np.int32)
    nb = np.zeros(8, np.int32)
    a.append_batch(t, nb, np.zeros(8, np.int32), np.full(8, 20, np.int32), 16)
    forked = t.copy()
    fnb = nb.copy()
    a.fork(forked, fnb, np.array([0, 0, 1, 1, 2, 2, 3, 3], np.int32))
    pairs = a.append_batch(forked, fnb, np.full(8, 20, np.int32), np.ones(8, np.int32), 16)
    assert len(pairs) == 4            # first beam of each shared row copies
    check_copy_pairs(pairs, 40)
    check_copy_pairs(np.zeros((0, 2), np.int64), 40)
    cases = {
        "outside": [[1, 2], [3, 40]],
        "same block": [[1, 2], [3, 2]],
        "source of pair 1": [[1, 2], [2, 5]],
        "source of pair 0": [[4, 4]],
    }
    for what, p in cases.items():
        with pytest.raises(L.PkvError) as e:
            check_copy_pairs(np.array(p, np.int64), 40)
        assert e.value.status == L.PKV_ERR_INVALID_ARG and what in str(e.value), (what, e.value)
    assert L.lib().pkv_check_copy_pairs(None, -1, 40) == L.PKV_ERR_INVALID_ARG


def test_nvtx_ranges_only_in_the_traced_build(tmp_path):
    """PKV_NVTX builds an NVTX range into every C-ABI call; the default
    build carries none (the host sources are compiled both ways)."""
    import shutil
    import subprocess
    from paged_kv_cache_162_gb300 import _build
    if shutil.which("g++") is None or shutil.which("nm") is None:
        pytest.skip("needs g++ and nm")
    inc = ["-I", _build.INCLUDE, "-I", _build.CSRC, "-I", os.path.join(_build.cuda_home(), "include")]
    for src in ("allocator.cpp", "beam_step.cpp"):
        for flag, want in ((["-DPKV_NVTX"], True), ([], False)):
            obj = str(tmp_path / (src + ("_nvtx" if flag else "") + ".o"))
            subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", *inc, *flag, "-c",
                            os.path.join(_build.CSRC, src), "-o", obj], check=True)
            syms = subprocess.run(["nm", obj], check=True, capture_output=True, text=True).stdout
            assert ("nvtx" in syms.lower()) == want, (src, flag)


def test_beam_search_create_rejects_bad_arguments_before_any_cuda_call():
    """The beam-search handle checks its arguments on the host first: a
    null handle pointer, a missing allocator, buffers that are too small or
    misaligned are refused (no GPU is needed to see it)."""
    lib = L.lib()
    h = ctypes.c_void_p()
    a = BlockAllocator(64)
    S, MB = 4, 8
    tables = np.zeros((S, MB), np.int32)
    nb = np.zeros(S, np.int32)
    ctx = np.zeros(S, np.int32)
    need = L.pkv_beam_inputs_bytes(S, MB)
    raw = np.zeros(4 * need + 1024, np.uint8)
    base = raw.ctypes.data + (-raw.ctypes.data) % 256
    stg0, stg1, dev = base, base + need + (-need % 256), base + 2 * (need + (-need % 256))
    fake = base  # any non-null address: nothing is dereferenced before the checks fail

    def create(alloc_h, s0, inputs_bytes, out_ptr):
        return lib.pkv_beam_search_create(alloc_h, tables.ctypes.data, nb.ctypes.data,
                                          ctx.ctypes.data, S, MB, s0, stg1, dev, inputs_bytes,
                                          fake, fake, fake, fake, None, 0, 4, 64, 16, 64, 0.125,
                                          L.PKV_F16, 0, fake, 1 << 20, out_ptr)
    assert create(a._h, stg0, need, None) == L.PKV_ERR_INVALID_ARG
    assert create(None, stg0, need, ctypes.addressof(h)) == L.PKV_ERR_INVALID_ARG
    assert create(a._h, stg0, need - 1, ctypes.addressof(h)) == L.PKV_ERR_INVALID_ARG
    assert create(a._h, stg0 + 16, need, ctypes.addressof(h)) == L.PKV_ERR_INVALID_ARG
    assert "aligned" in L.pkv_last_error_string()
    assert h.value is None
    lib.pkv_beam_search_destroy(None)  # a null handle is a no-op
    # a step without a handle, parents or result pointers is refused before
    # it touches a stream or a staging buffer
    n = ctypes.c_int32(-7)
    pairs = ctypes.c_void_p()
    parents = np.zeros(S, np.int32)
    step = lib.pkv_beam_search_step
    assert step(None, parents.ctypes.data, fake, fake, fake, None, ctypes.addressof(n),
                ctypes.addressof(pairs)) == L.PKV_ERR_INVALID_ARG
    assert "beam_search_step" in L.pkv_last_error_string()
    assert n.value == -7 and pairs.value is None
