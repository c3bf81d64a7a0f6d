"""Twelve steps of a serving loop over one paged pool, through the C ABI,
against the oracle after every step.

Each step, in the order a continuous-batching scheduler works ("3.3
页面级显存管理" 3.3.2 and 3.3.4; "vLLM三大核心技术分页内存与共享解码", continuous
batching and Copy-on-Write sections): finished sequences release their
blocks; new requests are admitted with a prefill; some running sequences
fork (parallel sampling); every running sequence appends one token
(copy-on-write of a shared partial block first).  Then copy_blocks, slot
mapping, reshape_and_cache and decode run on the GPU.  Freed blocks are
reused while they still hold old tokens, so a stale read shows up.

Checked every step: allocator state (free count, shared count, every
table), copy pairs, slots, the whole cache bit for bit, and attention."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import kernels as K
from oracle.allocator import BlockAllocatorModel
from paged_kv_cache_162_gb300 import _lib as L
from paged_kv_cache_162_gb300 import engine as E
from paged_kv_cache_162_gb300.allocator import BlockAllocator
from tests.gpu_harness import assert_attention_close

pytestmark = pytest.mark.gpu


def _bits(rng, shape, dtype):
    return W.normal_bits(np.random.Generator(np.random.SFC64(int(rng.integers(1 << 30)))), shape,
                         dtype)


def _dev(bits, dt):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(dt)


@pytest.mark.parametrize("dtype,bs", [(W.F16, 16), (W.BF16, 8)])
def test_serving_loop_matches_oracle(dtype, bs):
    rng = np.random.default_rng(2024 + bs)
    H, D, NB, MB = 4, 64, 160, 40
    tdt = torch.float16 if dtype == W.F16 else torch.bfloat16
    scale = 1.0 / math.sqrt(D)
    poison = int(W.POISON[dtype])
    pool_k = np.full((NB, bs, H, D), poison, np.uint16)
    pool_v = pool_k.copy()
    gk = _dev(pool_k, tdt)
    gv = _dev(pool_v, tdt)
    lib, mod = BlockAllocator(NB), BlockAllocatorModel(NB)
    seqs = {}        # id -> [table (list), ctx]
    next_id = 0
    for step in range(12):
        # 1. completions
        for sid in [s for s in list(seqs) if rng.random() < 0.15]:
            t = seqs.pop(sid)[0]
            assert lib.decref(t) == mod.decref(t)
        # 2. admissions with a prefill (if the pool allows, all-or-nothing)
        new_tok = {}     # sid -> (positions, K bits, V bits)
        for _ in range(int(rng.integers(0, 3))):
            n = int(rng.integers(1, 120))
            need = -(-n // bs)
            if need > mod.num_free or need > MB:
                continue
            t_lib, t_mod = [], []
            assert lib.append(t_lib, 0, n, bs) == mod.append(t_mod, 0, n, bs) == []
            assert t_lib == t_mod
            seqs[next_id] = [t_mod, n]
            new_tok[next_id] = (np.arange(n), _bits(rng, (n, H, D), dtype), _bits(rng, (n, H, D), dtype))
            next_id += 1
        # 3. forks of running sequences (share every block, same length)
        for sid in [s for s in list(seqs) if s not in new_tok and rng.random() < 0.2]:
            t, c = seqs[sid]
            lib.incref(t)
            mod.incref(t)
            seqs[next_id] = [list(t), c]
            next_id += 1
        # 4. every running (not just admitted) sequence appends one token
        pairs = []
        for sid in sorted(seqs):
            if sid in new_tok:
                continue
            t, c = seqs[sid]
            need = -(-(c + 1) // bs) - len(t)
            shared = c // bs < len(t) and mod.refcount(t[c // bs]) > 1
            if need + shared > mod.num_free or -(-(c + 1) // bs) > MB:
                continue
            t_lib = list(t)
            p_lib = lib.append(t_lib, c, 1, bs)
            p_mod = mod.append(t, c, 1, bs)
            assert p_lib == p_mod and t_lib == t
            pairs += p_mod
            new_tok[sid] = (np.array([c]), _bits(rng, (1, H, D), dtype), _bits(rng, (1, H, D), dtype))
            seqs[sid][1] = c + 1
        assert lib.num_free == mod.num_free and lib.num_shared == mod.num_shared
        if not seqs:
            continue
        # device step
        order = sorted(seqs)
        S = len(order)
        bt = np.full((S, MB), -1, np.int32)
        for i, sid in enumerate(order):
            bt[i, :len(seqs[sid][0])] = seqs[sid][0]
        ctx = np.array([seqs[sid][1] for sid in order], np.int32)
        seq_idx = np.concatenate([np.full(len(new_tok[sid][0]), i, np.int32)
                                  for i, sid in enumerate(order) if sid in new_tok] or [np.zeros(0, np.int32)])
        pos = np.concatenate([new_tok[sid][0] for sid in order if sid in new_tok] or [np.zeros(0)]).astype(np.int32)
        nk = np.concatenate([new_tok[sid][1] for sid in order if sid in new_tok] or [np.zeros((0, H, D), np.uint16)])
        nv = np.concatenate([new_tok[sid][2] for sid in order if sid in new_tok] or [np.zeros((0, H, D), np.uint16)])
        pr = np.array(pairs, np.int64).reshape(-1, 2)
        # oracle
        K.copy_blocks(pool_k, pool_v, pr)
        slots = K.slot_mapping(bt, seq_idx, pos, bs)
        K.reshape_and_cache(pool_k, pool_v, nk, nv, slots)
        q = _bits(rng, (S, H, D), dtype)
        ref = K.decode(q, pool_k, pool_v, bt, ctx, scale, dtype == W.BF16)
        # GPU
        d_bt = torch.from_numpy(bt).cuda()
        if len(pr):
            E.copy_blocks(gk, gv, torch.from_numpy(pr).cuda())
        d_slots = torch.empty(max(len(pos), 1), dtype=torch.int64, device="cuda")
        if len(pos):
            E.compute_slot_mapping(d_slots, d_bt, torch.from_numpy(seq_idx).cuda(),
                                   torch.from_numpy(pos).cuda(), bs)
            E.reshape_and_cache(_dev(nk, tdt), _dev(nv, tdt), gk, gv, d_slots)
        out = torch.empty(S, H, D, dtype=tdt, device="cuda")
        E.paged_attention_decode(out, _dev(q, tdt), gk, gv, d_bt, torch.from_numpy(ctx).cuda(), scale,
                                 partition_tokens=32)
        torch.cuda.synchronize()
        if len(pos):
            assert np.array_equal(d_slots[:len(pos)].cpu().numpy(), slots), f"step {step}: slots"
        assert np.array_equal(gk.view(torch.int16).cpu().numpy().view(np.uint16), pool_k), f"step {step}: K"
        assert np.array_equal(gv.view(torch.int16).cpu().numpy().view(np.uint16), pool_v), f"step {step}: V"
        assert_attention_close(out.float().cpu().double().numpy(), ref, f"serving step {step}")
    assert L.pkv_get_device_errors() == 0
