"""Seeded synthetic inputs for one decode step over a paged KV cache.

This module only *generates inputs*: random q/K/V values, context lengths,
physical block placement, the free-list order and which tokens a step
appends.  It holds none of the method's arithmetic (no slot mapping, no cache
write, no attention, no allocator policy); both the fp64 oracle and the CUDA
path consume what it returns, and neither is imported here.

Recipe (shared by every workload):
  * values ~ N(0, 1) by inverse-transform sampling: 16 random bits from a
    seeded SFC64 stream index a table of the 65,536 mid-point quantiles of
    N(0, 1); each quantile is rounded once (round-to-nearest-even) to the
    storage dtype, so both sides read the same 16-bit patterns;
  * physical placement is a seeded random permutation of the pool, so block
    tables are non-contiguous ("physical blocks may sit anywhere in GPU
    memory": "vLLM三大核心技术分页内存与共享解码", section
    "KV Cache逻辑块物理块映射机制");
  * cache slots that hold no token yet are filled with a NaN pattern, so a
    kernel that lets an unwritten slot reach its output shows NaN;
  * one seed per workload (1000 + index of the workload family).

LLaMA-7B-like layer shape (32 heads x 128 dims, fp16, 16-token blocks) follows
"3.1 PagedAttention的核心原理", section 3.1.2 (page structure: 8 KB of K and
8 KB of V per token per layer, 256 KB per 16-token page).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from statistics import NormalDist

import numpy as np

F16 = "f16"
BF16 = "bf16"
ELEM_BYTES = 2  # both storage dtypes are 16-bit

# NaN bit patterns used to poison unwritten cache slots.
POISON = {F16: np.uint16(0x7E00), BF16: np.uint16(0x7FC0)}

_TABLE_CACHE: dict[str, np.ndarray] = {}


def _round_f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 bit patterns (nearest-even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float array -> uint16 storage bits of `dtype` (round-to-nearest-even)."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        return _round_f32_to_bf16_bits(x)
    raise ValueError(dtype)


def normal_bits_table(dtype: str) -> np.ndarray:
    """65,536 N(0,1) mid-point quantiles, as `dtype` bit patterns."""
    if dtype not in _TABLE_CACHE:
        nd = NormalDist()
        qs = np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)],
                      dtype=np.float32)
        _TABLE_CACHE[dtype] = to_bits(qs, dtype)
    return _TABLE_CACHE[dtype]


def normal_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """Seeded N(0,1) samples of the given shape as `dtype` bit patterns."""
    n = int(np.prod(shape)) if len(shape) else 1
    table = normal_bits_table(dtype)
    out = np.empty(n, dtype=np.uint16)
    chunk = 1 << 22
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        idx = rng.bit_generator.random_raw((m + 3) // 4).view(np.uint16)[:m]
        out[i:i + m] = table[idx]
    return out.reshape(shape)


@dataclass
class Workload:
    """One decode step's inputs.

    Shapes: S sequences, H heads, D head_dim, bs tokens per block, NB physical
    blocks in the pool, MB block-table row length.  All token data is stored
    as uint16 bit patterns of `dtype`.

    Before the step, sequence s holds `ctx_before[s]` tokens in the blocks
    `tables_pre[s, :nblocks_pre[s]]` (unused entries are -1).  The step
    appends `n_new[s]` tokens to each sequence; their K/V are `new_k`,
    `new_v` ([T, H, D], sequence-major) at (seq_idx[t], pos[t]).  Blocks
    the step needs beyond `tables_pre` come from a free list whose order is
    `initial_free` (the last element is popped first); every pool block not
    in `initial_free` is held once per table that references it.

    `blocks` lists (sorted) the physical blocks that hold data before the
    step and `k_blocks`/`v_blocks` their contents [U, bs, H, D]; slots with
    no token yet hold the NaN pattern POISON[dtype], as do all other blocks.
    """
    name: str
    dtype: str
    S: int
    H: int
    D: int
    bs: int
    NB: int
    MB: int
    scale: float
    ctx_before: np.ndarray
    n_new: np.ndarray
    tables_pre: np.ndarray
    nblocks_pre: np.ndarray
    initial_free: np.ndarray
    blocks: np.ndarray
    k_blocks: np.ndarray
    v_blocks: np.ndarray
    q: np.ndarray
    new_k: np.ndarray
    new_v: np.ndarray
    seq_idx: np.ndarray
    pos: np.ndarray
    notes: dict = field(default_factory=dict)

    @property
    def context_lens(self) -> np.ndarray:
        return (self.ctx_before + self.n_new).astype(np.int32)

    @property
    def T(self) -> int:
        return int(self.n_new.sum())

    def kv_bytes(self) -> int:
        """Logical KV bytes one decode pass reads: sum ctx * H * D * 2 * 2 B."""
        return int(self.context_lens.astype(np.int64).sum()) * self.H * self.D * 2 * ELEM_BYTES


def _streams(seed: int, n: int):
    return [np.random.Generator(np.random.SFC64(s))
            for s in np.random.SeedSequence(seed).spawn(n)]


def _cdiv(a, b):
    return -(-np.asarray(a, dtype=np.int64) // b)


def _fill_blocks(rng, blocks, tables_pre, nblocks_pre, ctx_before, bs, H, D, dtype):
    """Random K or V for every pre-step block; slots without a token are NaN.

    The number of filled slots of a block is how many of its owning
    sequence's cached tokens fall into it (tokens fill blocks in order).
    """
    U = len(blocks)
    data = normal_bits(rng, (U, bs, H, D), dtype)
    if U == 0:
        return data
    filled = np.zeros(U, dtype=np.int64)
    for s in range(tables_pre.shape[0]):
        nb = int(nblocks_pre[s])
        if nb == 0:
            continue
        ids = tables_pre[s, :nb]
        cnt = np.clip(int(ctx_before[s]) - np.arange(nb, dtype=np.int64) * bs, 0, bs)
        u = np.searchsorted(blocks, ids)
        filled[u] = np.maximum(filled[u], cnt)
    slot = np.arange(bs)[None, :]
    empty = slot >= filled[:, None]  # [U, bs]
    data[empty] = POISON[dtype]
    return data


def _finish(name, dtype, S, H, D, bs, NB, MB, ctx_before, n_new, tables_pre,
            nblocks_pre, initial_free, rngs, notes=None) -> Workload:
    r_kv, r_q, r_new = rngs
    used = tables_pre[tables_pre >= 0]
    blocks = np.unique(used).astype(np.int32)
    k_blocks = _fill_blocks(r_kv, blocks, tables_pre, nblocks_pre, ctx_before, bs, H, D, dtype)
    v_blocks = _fill_blocks(r_kv, blocks, tables_pre, nblocks_pre, ctx_before, bs, H, D, dtype)
    q = normal_bits(r_q, (S, H, D), dtype)
    T = int(n_new.sum())
    new_k = normal_bits(r_new, (T, H, D), dtype)
    new_v = normal_bits(r_new, (T, H, D), dtype)
    seq_idx = np.repeat(np.arange(S, dtype=np.int32), n_new)
    starts = np.repeat(ctx_before, n_new)
    within = np.arange(T, dtype=np.int64) - np.repeat(np.cumsum(n_new) - n_new, n_new)
    pos = (starts + within).astype(np.int32)
    return Workload(name=name, dtype=dtype, S=S, H=H, D=D, bs=bs, NB=NB, MB=MB,
                    scale=1.0 / math.sqrt(D),
                    ctx_before=ctx_before.astype(np.int32), n_new=n_new.astype(np.int32),
                    tables_pre=tables_pre.astype(np.int32),
                    nblocks_pre=nblocks_pre.astype(np.int32),
                    initial_free=np.asarray(initial_free, dtype=np.int32),
                    blocks=blocks, k_blocks=k_blocks, v_blocks=v_blocks, q=q,
                    new_k=new_k, new_v=new_v, seq_idx=seq_idx, pos=pos,
                    notes=notes or {})


def _placed(ctx_after, ctx_before, bs, NB, MB, perm):
    """Tables that already cover ctx_after, taken in order from `perm`."""
    S = len(ctx_after)
    nb = _cdiv(ctx_after, bs)
    assert nb.sum() <= NB and nb.max() <= MB
    tables = np.full((S, MB), -1, dtype=np.int32)
    k = 0
    for s in range(S):
        tables[s, :nb[s]] = perm[k:k + nb[s]]
        k += nb[s]
    return tables, nb.astype(np.int32), perm[k:]


def uniform_decode(name, seed, dtype, S, H, D, bs, ctx_lo, ctx_hi, NB=None,
                   pool_slack=0.10, MB=None, n_new=1, ctx=None) -> Workload:
    """Every sequence appends `n_new` tokens; context_len ~ U{ctx_lo..ctx_hi}.

    Tables already cover the appended tokens (no allocation in the step).
    NB=None sizes the pool to the total need plus `pool_slack`.
    """
    r_ctx, r_perm, r_kv, r_q, r_new = _streams(seed, 5)
    if ctx is None:
        ctx = r_ctx.integers(ctx_lo, ctx_hi + 1, size=S).astype(np.int64)
    ctx = np.asarray(ctx, dtype=np.int64)
    n_new_arr = np.minimum(np.full(S, n_new, dtype=np.int64), ctx)
    ctx_before = ctx - n_new_arr
    need = int(_cdiv(ctx, bs).sum())
    if NB is None:
        NB = max(1, int(round(need * (1.0 + pool_slack))))
    if MB is None:
        MB = max(1, int(_cdiv(ctx.max(initial=1), bs)))
    perm = r_perm.permutation(NB).astype(np.int32)
    tables, nb, free = _placed(ctx, ctx_before, bs, NB, MB, perm)
    return _finish(name, dtype, S, H, D, bs, NB, MB, ctx_before, n_new_arr, tables, nb,
                   free, (r_kv, r_q, r_new))


def tiny(seed=1000) -> Workload:
    """4 seqs, 4 heads x 64, fp16, bs 16, ctx U{1..100}, 64-block pool."""
    return uniform_decode("tiny", seed, F16, S=4, H=4, D=64, bs=16, ctx_lo=1, ctx_hi=100,
                          NB=64, MB=7)


def llama7b_batch64(seed=1001, S=64, bs=16) -> Workload:
    """LLaMA-7B-shaped layer: 64 seqs, 32 x 128, fp16, bs 16, ctx U{128..2048},
    pool = total need + 10 %, shuffled placement; one new token per seq.
    `bs` changes only the block size (the block-size sweep)."""
    return uniform_decode("llama7b_batch64" if bs == 16 else f"llama7b_batch64_bs{bs}", seed, F16,
                          S=S, H=32, D=128, bs=bs, ctx_lo=128, ctx_hi=2048,
                          MB=-(-2048 // bs))


def long_context(bs=16, seed=1004, S=8, ctx_len=32768, NB=40000) -> Workload:
    """8 seqs of 32,768 tokens, 32 x 128, fp16, random placement in a
    40,000-block pool."""
    return uniform_decode(f"long_context_bs{bs}", seed, F16, S=S, H=32, D=128, bs=bs,
                          ctx_lo=ctx_len, ctx_hi=ctx_len, NB=NB,
                          MB=int(_cdiv(ctx_len, bs)))


def continuous_batching_bf16(seed=1002, S=256, NB=20000, fresh_frac=0.12,
                             prefill=320) -> Workload:
    """Continuous-batching step, bf16: 256 seqs, 32 x 128, bs 16.

    Running sequences: context ~ lognormal(median 512, sigma 1) clamped to
    [16, 4096]; they append one decode token.  round(12 % of 256) = 31 seqs
    are freshly admitted and append a 320-token prefill.  Running sequences'
    existing blocks are randomly placed in a 20,000-block pool; the rest of
    the pool is the free list (seeded shuffle) that the step allocates from.
    """
    r_ctx, r_fresh, r_perm, r_kv, r_q, r_new = _streams(seed, 6)
    bs, H, D = 16, 32, 128
    ctx = np.exp(np.log(512.0) + r_ctx.standard_normal(S))
    ctx = np.clip(np.rint(ctx), 16, 4096).astype(np.int64)
    n_fresh = int(round(fresh_frac * S))
    fresh = np.sort(r_fresh.choice(S, size=n_fresh, replace=False))
    n_new = np.ones(S, dtype=np.int64)
    n_new[fresh] = prefill
    ctx[fresh] = prefill
    ctx_before = ctx - n_new
    MB = int(_cdiv(4096, bs))
    perm = r_perm.permutation(NB).astype(np.int32)
    nb_pre = _cdiv(ctx_before, bs)
    tables = np.full((S, MB), -1, dtype=np.int32)
    k = 0
    for s in range(S):
        tables[s, :nb_pre[s]] = perm[k:k + nb_pre[s]]
        k += nb_pre[s]
    free = perm[k:]
    return _finish("continuous_batching_bf16", BF16, S, H, D, bs, NB, MB, ctx_before, n_new,
                   tables, nb_pre.astype(np.int32), free, (r_kv, r_q, r_new),
                   notes={"fresh": fresh.tolist()})


def shared_prefix(seed=1003, prompts=32, samples=8, prefix=1024, tail_lo=1, tail_hi=256,
                  cow=False, pool_slack=0.10, H=32, D=128, bs=16, dtype=F16) -> Workload:
    """Parallel sampling, fp16: 32 prompts x 8 samples, 32 x 128, bs 16.

    cow=False: every sample shares its prompt's 1024-token prefix (64 full
    blocks, referenced 8 times); each sample's private tail ~ U{1..256}
    tokens ends with the token this step appends.
    cow=True: the prompt is 1024 + r tokens, r ~ U{1..15}, so its last block
    is partial and shared by all 8 samples; the step is the first write after
    the fork (one token per sample), which must copy that block first.
    """
    r_len, r_perm, r_kv, r_q, r_new = _streams(seed + (100 if cow else 0), 5)
    S = prompts * samples
    if cow:
        plen = prefix + r_len.integers(1, min(bs, 16), size=prompts)
        ctx_before = np.repeat(plen, samples).astype(np.int64)
        n_new = np.ones(S, dtype=np.int64)
    else:
        plen = np.full(prompts, prefix, dtype=np.int64)
        tail = r_len.integers(tail_lo, tail_hi + 1, size=S)
        ctx_before = np.repeat(plen, samples) + tail - 1
        n_new = np.ones(S, dtype=np.int64)
    ctx_after = ctx_before + n_new
    pre_blocks = _cdiv(plen, bs)
    MB = int(_cdiv(ctx_after.max(), bs))
    # need: shared prompt blocks once, private blocks per sample (+1 per
    # sample for a copy or a new block)
    priv = _cdiv(ctx_after, bs) - np.repeat(pre_blocks, samples)
    need = int(pre_blocks.sum() + np.maximum(priv, 0).sum() + (S if cow else 0))
    NB = int(round(need * (1.0 + pool_slack)))
    perm = r_perm.permutation(NB).astype(np.int32)
    tables = np.full((S, MB), -1, dtype=np.int32)
    nb_pre = np.zeros(S, dtype=np.int64)
    k = 0
    for p in range(prompts):
        shared = perm[k:k + pre_blocks[p]]
        k += pre_blocks[p]
        for j in range(samples):
            s = p * samples + j
            own = int(_cdiv(ctx_before[s], bs)) - int(pre_blocks[p])
            own = max(own, 0)
            tables[s, :pre_blocks[p]] = shared
            tables[s, pre_blocks[p]:pre_blocks[p] + own] = perm[k:k + own]
            k += own
            nb_pre[s] = pre_blocks[p] + own
    free = perm[k:]
    return _finish("shared_prefix_cow" if cow else "shared_prefix", dtype, S, H, D, bs, NB, MB,
                   ctx_before, n_new, tables, nb_pre.astype(np.int32), free,
                   (r_kv, r_q, r_new), notes={"prompt_len": plen.tolist(), "samples": samples})


WORKLOADS = {
    "tiny": tiny,
    "llama7b_batch64": llama7b_batch64,
    "continuous_batching_bf16": continuous_batching_bf16,
    "shared_prefix": shared_prefix,
    "shared_prefix_cow": lambda **kw: shared_prefix(cow=True, **kw),
    "long_context_bs16": lambda **kw: long_context(bs=16, **kw),
    "long_context_bs32": lambda **kw: long_context(bs=32, **kw),
}


def make(name: str, **kw) -> Workload:
    return WORKLOADS[name](**kw)


def small_case(seed, dtype=F16, S=3, H=2, D=64, bs=16, ctx_lo=1, ctx_hi=80, NB=None,
               n_new=1, ctx=None) -> Workload:
    """Small random case for exhaustive parity (several tiles, ragged tails)."""
    return uniform_decode(f"small_{dtype}_D{D}_bs{bs}", seed, dtype, S=S, H=H, D=D, bs=bs,
                          ctx_lo=ctx_lo, ctx_hi=ctx_hi, NB=NB, n_new=n_new, ctx=ctx)


@dataclass
class BeamWorkload:
    """Beam search over paged KV (fork + copy-on-write every step).

    `init` is the state after the prompts were prefilled: request r's prompt
    blocks are referenced by all `beams` sequences of the request
    (sequences r*beams .. r*beams + beams-1).  Then `steps` decode steps:
    at step i every beam b continues from beam parents[i, b] of its own
    request (it forks the parent's table), then appends one token with K/V
    new_k[i, b] / new_v[i, b] and attends with query q[i, b].
    """
    init: Workload
    beams: int
    parents: np.ndarray   # [steps, S] int32 (sequence index of the parent)
    new_k: np.ndarray     # [steps, S, H, D] uint16
    new_v: np.ndarray
    q: np.ndarray         # [steps, S, H, D] uint16

    @property
    def steps(self) -> int:
        return self.parents.shape[0]


def beam_search(seed=1006, requests=16, beams=4, prompt_lo=256, prompt_hi=1024, steps=8,
                H=32, D=128, bs=16, dtype=F16, pool_slack=1.25) -> BeamWorkload:
    """Beam search, fp16: `requests` prompts x `beams` beams (LLaMA-7B layer
    shape by default); prompts ~ U{prompt_lo..prompt_hi}; parents drawn
    uniformly among the request's beams at every step."""
    r_len, r_perm, r_kv, r_q, r_new, r_par = _streams(seed, 6)
    S = requests * beams
    plen = r_len.integers(prompt_lo, prompt_hi + 1, size=requests).astype(np.int64)
    pre_blocks = _cdiv(plen, bs)
    MB = int(_cdiv(plen.max() + steps, bs))
    # prompts once; every step each beam may need a copy of its last block
    # and at most one new block
    need = int(pre_blocks.sum()) + S * (2 + 2 * _cdiv(steps, bs).item() + steps)
    NB = int(need * pool_slack)
    perm = r_perm.permutation(NB).astype(np.int32)
    tables = np.full((S, MB), -1, dtype=np.int32)
    nb_pre = np.zeros(S, dtype=np.int64)
    k = 0
    for r in range(requests):
        shared = perm[k:k + pre_blocks[r]]
        k += pre_blocks[r]
        for j in range(beams):
            s = r * beams + j
            tables[s, :pre_blocks[r]] = shared
            nb_pre[s] = pre_blocks[r]
    ctx_before = np.repeat(plen, beams)
    init = _finish("beam_search", dtype, S, H, D, bs, NB, MB, ctx_before,
                   np.zeros(S, dtype=np.int64), tables, nb_pre.astype(np.int32), perm[k:],
                   (r_kv, r_q, r_new), notes={"prompt_len": plen.tolist()})
    base = (np.arange(S) // beams) * beams
    parents = (base[None, :] + r_par.integers(0, beams, size=(steps, S))).astype(np.int32)
    new_k = normal_bits(r_new, (steps, S, H, D), dtype)
    new_v = normal_bits(r_new, (steps, S, H, D), dtype)
    q = normal_bits(r_q, (steps, S, H, D), dtype)
    return BeamWorkload(init=init, beams=beams, parents=parents, new_k=new_k, new_v=new_v, q=q)
