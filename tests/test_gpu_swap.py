"""CPU swap of KV blocks ("3.3 页面级显存管理" 3.3.3) through the C ABI,
against the oracle: bit-exact block copies both ways, and a swap-out /
reuse / swap-in cycle after which decode attention still matches."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import kernels as K
from oracle.allocator import BlockAllocatorModel
from paged_kv_cache_162_gb300 import _lib as L
from paged_kv_cache_162_gb300 import engine as E
from paged_kv_cache_162_gb300.allocator import BlockAllocator, plan_swap_in, plan_swap_out
from tests.gpu_harness import assert_attention_close

pytestmark = pytest.mark.gpu


def _bits(rng, shape, dtype=W.F16):
    return W.normal_bits(np.random.Generator(np.random.SFC64(int(rng.integers(1 << 30)))), shape,
                         dtype)


def _dev(bits, dtype=torch.float16):
    return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(dtype)


def _host_pool(shape, fill):
    t = torch.empty(shape, dtype=torch.int16).pin_memory()
    t.fill_(int(np.int16(np.uint16(fill))))
    return t.view(torch.float16)


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 32)])
def test_swap_out_and_in_bit_exact(D, bs):
    rng = np.random.default_rng(D + bs)
    H, NBg, NBh = 4, 40, 24
    gk_bits, gv_bits = _bits(rng, (NBg, bs, H, D)), _bits(rng, (NBg, bs, H, D))
    gk, gv = _dev(gk_bits), _dev(gv_bits)
    hk, hv = _host_pool((NBh, bs, H, D), 0x7E00), _host_pool((NBh, bs, H, D), 0x7E00)
    out_pairs = np.stack([rng.permutation(NBg)[:10], rng.permutation(NBh)[:10]], 1)
    E.swap_blocks(gk, gv, hk, hv, torch.from_numpy(out_pairs).cuda(), L.PKV_SWAP_OUT)
    torch.cuda.synchronize()
    want_k = np.full((NBh, bs, H, D), 0x7E00, np.uint16)
    want_v = want_k.copy()
    K.swap_blocks(want_k, want_v, gk_bits, gv_bits, out_pairs)
    assert np.array_equal(hk.view(torch.int16).numpy().view(np.uint16), want_k)
    assert np.array_equal(hv.view(torch.int16).numpy().view(np.uint16), want_v)
    # back into other GPU blocks
    free = np.setdiff1d(np.arange(NBg), out_pairs[:, 0])
    in_pairs = np.stack([out_pairs[:, 1], rng.permutation(free)[:10]], 1)
    E.swap_blocks(gk, gv, hk, hv, torch.from_numpy(in_pairs).cuda(), L.PKV_SWAP_IN)
    torch.cuda.synchronize()
    ref_k, ref_v = gk_bits.copy(), gv_bits.copy()
    K.swap_blocks(ref_k, ref_v, want_k, want_v, in_pairs)
    assert np.array_equal(gk.cpu().view(torch.int16).numpy().view(np.uint16), ref_k)
    assert np.array_equal(gv.cpu().view(torch.int16).numpy().view(np.uint16), ref_v)
    assert L.pkv_get_device_errors() == 0


def test_swap_rejects_pageable_host_memory():
    gk = torch.zeros(4, 16, 4, 64, dtype=torch.float16, device="cuda")
    hk = torch.zeros(4, 16, 4, 64, dtype=torch.float16)  # not page-locked
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    with pytest.raises(L.PkvError) as e:
        E.swap_blocks(gk, gk, hk, hk, pairs, L.PKV_SWAP_OUT)
    assert e.value.status == L.PKV_ERR_INVALID_ARG


def test_swap_cycle_then_decode_matches_oracle():
    """Sequence A is swapped out, its GPU blocks are reused by C (and
    overwritten), then A is swapped back into fresh blocks: A's attention is
    unchanged, C's cache intact."""
    rng = np.random.default_rng(77)
    H, D, bs, NBg, NBh = 8, 128, 16, 60, 64
    ctx = {"A": 300, "B": 200, "C": 320}
    scale = 1.0 / math.sqrt(D)
    pool_k = np.full((NBg, bs, H, D), 0x7E00, np.uint16)   # the oracle's GPU pool
    pool_v = pool_k.copy()
    gk, gv = _dev(pool_k), _dev(pool_v)
    hk, hv = _host_pool((NBh, bs, H, D), 0x7E00), _host_pool((NBh, bs, H, D), 0x7E00)
    host_k = np.full((NBh, bs, H, D), 0x7E00, np.uint16)
    host_v = host_k.copy()
    ga, ha = BlockAllocator(NBg), BlockAllocator(NBh)
    gm, hm = BlockAllocatorModel(NBg), BlockAllocatorModel(NBh)
    tables, tok_k, tok_v = {}, {}, {}

    def prefill(name):
        t, tm = [], []
        ga.append(t, 0, ctx[name], bs)
        gm.append(tm, 0, ctx[name], bs)
        assert t == tm
        tables[name] = t
        tok_k[name], tok_v[name] = _bits(rng, (ctx[name], H, D)), _bits(rng, (ctx[name], H, D))
        table = np.array([t], np.int32)
        pos = np.arange(ctx[name], dtype=np.int32)
        slots = K.slot_mapping(table, np.zeros_like(pos), pos, bs)
        K.reshape_and_cache(pool_k, pool_v, tok_k[name], tok_v[name], slots)
        d_slots = torch.from_numpy(slots).cuda()
        E.reshape_and_cache(_dev(tok_k[name]), _dev(tok_v[name]), gk, gv, d_slots)

    prefill("A")
    prefill("B")
    # swap A out, release its GPU blocks
    host_ids, pairs = plan_swap_out(ga, ha, tables["A"])
    assert host_ids == hm.alloc(len(tables["A"]))
    E.swap_blocks(gk, gv, hk, hv, torch.from_numpy(pairs).cuda(), L.PKV_SWAP_OUT)
    K.swap_blocks(host_k, host_v, pool_k, pool_v, pairs)
    ga.decref(tables["A"])
    gm.decref(tables["A"])
    assert ga.num_free == gm.num_free == NBg - len(tables["B"])
    # C reuses the freed blocks and overwrites them
    prefill("C")
    assert set(tables["C"]) & set(tables["A"])
    # swap A back in, into fresh GPU blocks
    table_a, pairs = plan_swap_in(ga, ha, host_ids)
    assert table_a == gm.alloc(len(host_ids))
    E.swap_blocks(gk, gv, hk, hv, torch.from_numpy(pairs).cuda(), L.PKV_SWAP_IN)
    K.swap_blocks(pool_k, pool_v, host_k, host_v, pairs)
    ha.decref(host_ids)
    hm.decref(host_ids)
    tables["A"] = table_a
    torch.cuda.synchronize()
    assert np.array_equal(gk.cpu().view(torch.int16).numpy().view(np.uint16), pool_k)
    assert np.array_equal(hk.view(torch.int16).numpy().view(np.uint16), host_k)
    # decode all three against the oracle on its own pool
    names = ["A", "B", "C"]
    MB = max(len(tables[n]) for n in names)
    bt = np.full((3, MB), -1, np.int32)
    for i, n in enumerate(names):
        bt[i, :len(tables[n])] = tables[n]
    cl = np.array([ctx[n] for n in names], np.int32)
    q = _bits(rng, (3, H, D))
    ref = K.decode(q, pool_k, pool_v, bt, cl, scale, False)
    out = torch.empty(3, H, D, dtype=torch.float16, device="cuda")
    E.paged_attention_decode(out, _dev(q), gk, gv, torch.from_numpy(bt).cuda(),
                             torch.from_numpy(cl).cuda(), scale)
    assert_attention_close(out.float().cpu().double().numpy(), ref, "swap cycle")
    # A's attention equals attention over A's original tokens
    Kc = torch.from_numpy(tok_k["A"].view(np.float16).astype(np.float64))
    Vc = torch.from_numpy(tok_v["A"].view(np.float16).astype(np.float64))
    Q = torch.from_numpy(q[0].view(np.float16).astype(np.float64))
    w = torch.softmax(torch.einsum("hd,jhd->hj", Q, Kc) * scale, -1)
    np.testing.assert_allclose(ref[0], torch.einsum("hj,jhd->hd", w, Vc).numpy(), atol=1e-10)
    assert L.pkv_get_device_errors() == 0
