"""Beam search over the paged cache (fork + copy-on-write every step)
through the C ABI, step by step against the oracle: tables, copy pairs,
slots and every cache block bit-exact, attention within tolerance."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as OS
from tests.gpu_harness import assert_attention_close, device_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs,device_tokens,groups,pt,prompts,dtype,D", [
    (16, False, False, 32, (20, 70), W.F16, 64), (8, False, False, 32, (20, 70), W.F16, 64),
    (16, True, False, 32, (20, 70), W.F16, 64), (16, True, True, 32, (20, 70), W.F16, 64),
    (8, False, True, 32, (20, 70), W.F16, 64), (16, True, True, 0, (100, 300), W.F16, 64),
    (32, True, False, 0, (100, 300), W.BF16, 128), (32, True, True, 0, (100, 300), W.BF16, 128),
    (64, False, True, 64, (130, 400), W.F16, 128)])
def test_beam_search_steps_match_oracle(bs, device_tokens, groups, pt, prompts, dtype, D):
    """groups: the beams of each request decode as a prefix group over
    their prompt's full blocks, which stay shared for the whole search."""
    bw = W.beam_search(seed=7 + bs, requests=3, beams=4, prompt_lo=prompts[0],
                       prompt_hi=prompts[1], steps=6, H=4, D=D, bs=bs, dtype=dtype)
    st = device_step(bw.init, pt)
    st.plan()
    if groups:
        plen = bw.init.notes["prompt_len"]
        st.beam_groups = [[r * bw.beams, bw.beams, (p // bs) * bs] for r, p in enumerate(plen)]
    if device_tokens:
        # the step's q and new K/V already on the device, as a model makes them
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
        toks = (dev(bw.new_k), dev(bw.new_v), dev(bw.q))
    copies = 0
    for i, (bt, pairs, slots, k_pool, v_pool, ids, out) in enumerate(OS.run_beam(bw, nthreads=2)):
        if device_tokens:
            got_pairs = st.beam_step(bw.parents[i], toks[0][i], toks[1][i], toks[2][i])
        else:
            got_pairs = st.beam_step(bw.parents[i], bw.new_k[i], bw.new_v[i], bw.q[i])
        torch.cuda.synchronize()
        assert np.array_equal(st.tables_host, bt), f"step {i}: tables"
        assert np.array_equal(got_pairs, pairs), f"step {i}: pairs"
        assert np.array_equal(st.slot_mapping[:bw.init.S].cpu().numpy(), slots), f"step {i}"
        for cache, pool in ((st.k_cache, k_pool), (st.v_cache, v_pool)):
            assert np.array_equal(cache.view(torch.int16).cpu().numpy().view(np.uint16), pool)
        assert_attention_close(st.out.float().cpu().double().numpy(), out, f"beam step {i}")
        copies += len(pairs)
    assert copies > 0  # forks made shared partial blocks that had to be copied
