"""GPU parity: the CUDA library against the fp64 oracle, through the C ABI.

Bit-exact: block tables, copy-on-write pairs, slot mapping, both caches
(every block the step may touch, plus a check that no other block changed).
Attention: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| per element.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_harness import compare_step, device_step, out_to_double
from oracle import step as OS

pytestmark = pytest.mark.gpu


def test_tiny_workload():
    r = compare_step(W.tiny())
    assert r["max_abs"] < 2e-3


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("pt", [32, 64, 256])
def test_small_cases_span_tiles_partitions_and_ragged_tails(dtype, D, bs, pt):
    if pt % bs:
        pytest.skip("partition must be a multiple of the block size")
    # 6 heads: the second head group has 2 idle warps
    w = W.small_case(seed=D * 1000 + bs * 10 + pt + (dtype == W.BF16) * 7, dtype=dtype, S=5, H=6, D=D, bs=bs,
                     ctx_lo=1, ctx_hi=300, n_new=3)
    compare_step(w, partition_tokens=pt)


@pytest.mark.parametrize("ctx", [[0, 5, 0], [1, 1, 1], [16, 32, 48], [255, 256, 257], [512, 1, 513]])
def test_edge_context_lengths(ctx):
    w = W.small_case(seed=sum(ctx), S=3, H=4, D=128, bs=16, ctx=ctx, n_new=1, NB=120)
    r = compare_step(w, partition_tokens=256)
    out = out_to_double(r["step"].out)
    for s, c in enumerate(ctx):
        if c == 0:
            assert np.all(out[s] == 0.0)


def test_output_independent_of_partition_size():
    w = W.small_case(seed=77, S=4, H=8, D=128, bs=16, ctx_lo=200, ctx_hi=900)
    outs = []
    for pt in (16, 64, 256, 1024):
        st = device_step(w, pt)
        st.run()
        outs.append(out_to_double(st.out))
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], atol=2e-3, rtol=1e-2)


def test_placement_invariance_bit_identical():
    """Same logical K/V in two different physical placements."""
    w1 = W.small_case(seed=5, S=4, H=4, D=128, bs=16, ctx_lo=50, ctx_hi=600, NB=200)
    w2 = W.small_case(seed=5, S=4, H=4, D=128, bs=16, ctx_lo=50, ctx_hi=600, NB=200)
    rng = np.random.default_rng(9)
    perm = rng.permutation(w2.NB).astype(np.int32)
    w2.tables_pre = np.where(w2.tables_pre >= 0, perm[np.maximum(w2.tables_pre, 0)], -1).astype(np.int32)
    w2.blocks = perm[w1.blocks]
    order = np.argsort(w2.blocks)
    w2.blocks, w2.k_blocks, w2.v_blocks = w2.blocks[order], w1.k_blocks[order], w1.v_blocks[order]
    w2.initial_free = perm[w1.initial_free]
    outs = []
    for w in (w1, w2):
        st = device_step(w, 128)
        st.run()
        outs.append(st.out.cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_repeated_calls_are_deterministic():
    w = W.small_case(seed=3, S=6, H=8, D=128, bs=16, ctx_lo=300, ctx_hi=2000)
    st = device_step(w, 128)
    st.run()
    a = st.out.clone()
    for _ in range(3):
        st.decode()
    assert torch.equal(a.view(torch.int16), st.out.view(torch.int16))


# ------------------------------------------------ full-size workloads
def test_llama7b_batch64_full():
    r = compare_step(W.llama7b_batch64())
    print("llama7b_batch64 max abs", r["max_abs"])


def test_continuous_batching_bf16_full():
    r = compare_step(W.continuous_batching_bf16())
    print("continuous_batching_bf16 max abs", r["max_abs"], "max rel", r["max_rel"])


def test_shared_prefix_full():
    r = compare_step(W.shared_prefix())
    assert r["pairs"] == 0


def test_shared_prefix_cow_full():
    r = compare_step(W.shared_prefix(cow=True))
    assert r["pairs"] == 32 * 7


@pytest.mark.parametrize("bs", [16, 32])
def test_long_context_full(bs):
    r = compare_step(W.long_context(bs=bs))
    print(f"long_context_bs{bs} max abs", r["max_abs"])


def _chosen_partition(st):
    # the plan kernel records its partition size in the workspace header
    return int(st.workspace[8:12].view(torch.int32).item())


def test_automatic_partition_size_on_full_workloads():
    """The automatic choice (largest of 64, 128, ... tokens giving >= 6 items
    per resident CTA and <= 3/4 of the mean context) on GB300's 152 SMs picks
    the sizes measured fastest for these workloads."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip("expected sizes are for a 152-SM GB300")
    for make, want in ((W.llama7b_batch64, 128), (W.continuous_batching_bf16, 512),
                       (W.shared_prefix, 512), (lambda: W.long_context(bs=16), 512)):
        w = make()
        st = device_step(w, 0)
        st.run()
        torch.cuda.synchronize()
        assert _chosen_partition(st) == want, (w.name, _chosen_partition(st))


def _item_list(st):
    # header: n_items at byte 4; the packed (seq << 16 | partition) items
    # start at byte 256
    n = int(st.workspace[4:8].view(torch.int32).item())
    items = st.workspace[256:256 + 4 * n].view(torch.int32).cpu().numpy()
    return items >> 16, items & 0xFFFF


@pytest.mark.parametrize("make,pt", [
    (lambda: W.small_case(81, S=40, H=8, D=128, ctx_lo=0, ctx_hi=700), 0),
    (lambda: W.small_case(82, S=40, H=8, D=128, ctx_lo=1, ctx_hi=700), 64),
    (lambda: W.small_case(83, S=33, H=4, D=64, ctx=[128 * (i % 5) + (i % 3) for i in range(33)]), 128),
    (W.llama7b_batch64, 0),
    (lambda: W.shared_prefix(cow=True), 0),
])
def test_plan_item_list(make, pt):
    """The plan lists every (sequence, partition) once; full partitions in
    sequence order; the partial (last) partitions all before the full ones
    when they average at least 3/8 of a partition, else all after them."""
    w = make()
    st = device_step(w, pt)
    st.run()
    torch.cuda.synchronize()
    PT = _chosen_partition(st)
    seq, part = _item_list(st)
    ctx = np.asarray(w.context_lens, dtype=np.int64)
    want = {(s, k) for s in range(w.S) for k in range(max(1, -(-int(ctx[s]) // PT)))}
    got = list(zip(seq.tolist(), part.tolist()))
    assert len(got) == len(set(got)) and set(got) == want
    is_partial = np.array([(ctx[s] % PT != 0 or ctx[s] == 0) and k == ctx[s] // PT
                           for s, k in got], dtype=bool)
    n_partial = int(is_partial.sum())
    full = [g for g, p in zip(got, is_partial) if not p]
    assert full == sorted(full)
    fill = int((ctx % PT).sum())
    if n_partial:
        first = 8 * fill >= 3 * n_partial * PT
        block = is_partial[:n_partial] if first else is_partial[len(got) - n_partial:]
        assert block.all(), (first, n_partial)
