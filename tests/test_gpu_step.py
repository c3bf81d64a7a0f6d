"""pkv_decode_step (slot mapping, cache write and the decode's plan in one
kernel, then decode) against the oracle, and bit for bit against the
separate calls it replaces."""
import numpy as np
import pytest
import torch

import workloads as W
from paged_kv_cache_162_gb300 import _lib as L
from tests.gpu_harness import compare_step, device_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make,pt", [
    (W.tiny, 0),
    (lambda: W.small_case(61, dtype=W.BF16, S=7, H=6, D=64, bs=8, ctx_lo=0, ctx_hi=300, n_new=3), 64),
    (lambda: W.small_case(62, S=5, H=8, D=128, bs=32, ctx_lo=1, ctx_hi=700, n_new=17), 0),
    (lambda: W.shared_prefix(cow=True, prompts=3, samples=4, prefix=128, tail_lo=1, tail_hi=40), 0),
    (W.continuous_batching_bf16, 0),
])
def test_fused_step_matches_oracle(make, pt):
    compare_step(make(), partition_tokens=pt, fused=True)


@pytest.mark.parametrize("make", [
    lambda: W.small_case(63, S=9, H=4, D=128, bs=16, ctx_lo=0, ctx_hi=500, n_new=2),
    W.llama7b_batch64,
    lambda: W.shared_prefix(cow=True),
])
def test_fused_step_bit_identical_to_separate_calls(make):
    w = make()
    st = device_step(w, 0)
    st.plan()
    k0, v0 = st.k_cache.clone(), st.v_cache.clone()
    st.run()
    torch.cuda.synchronize()
    want = [t.clone() for t in (st.slot_mapping, st.k_cache, st.v_cache, st.out)]
    st.k_cache.copy_(k0)
    st.v_cache.copy_(v0)
    st.out.fill_(float("nan"))
    st.slot_mapping.fill_(-7)
    st.run(fused=True)
    torch.cuda.synchronize()
    got = (st.slot_mapping, st.k_cache, st.v_cache, st.out)
    for name, a, b in zip(("slots", "k_cache", "v_cache", "out"), want, got):
        assert torch.equal(a.view(torch.int16) if a.dtype != torch.int64 else a,
                           b.view(torch.int16) if b.dtype != torch.int64 else b), name


def test_fused_step_flags_bad_positions_like_the_slot_kernel():
    """A position past its table row and one in an unmapped block give slot
    -1 (nothing written) and the same error bits as pkv_compute_slot_mapping."""
    w = W.small_case(64, S=3, H=4, D=64, bs=16, ctx=[40, 70, 20], n_new=2)
    st = device_step(w, 0)
    st.plan()
    L.pkv_get_device_errors()
    pos = st.pos.clone()
    pos[0] = st.MB * st.bs + 3          # past the row
    st.pos = pos
    bt = st.block_tables.clone()
    s2 = int(st.seq_idx[2].item())
    lb = int(pos[2].item()) // st.bs
    bt[s2, lb] = -1                     # the token's block is not mapped
    st.block_tables = bt
    k0 = st.k_cache.clone()
    st.run(fused=True)
    torch.cuda.synchronize()
    flags = L.pkv_get_device_errors()
    assert flags & L.PKV_DEVERR_POSITION and flags & L.PKV_DEVERR_BLOCK_ID
    slots = st.slot_mapping[:st.T].cpu().numpy()
    # expected slots from the modified table, as the address translation
    # gives them
    table, p_h, s_h = bt.cpu().numpy(), pos.cpu().numpy(), st.seq_idx.cpu().numpy()
    want = np.full(st.T, -1, dtype=np.int64)
    for t in range(st.T):
        lb = p_h[t] // st.bs
        if lb < st.MB and table[s_h[t], lb] >= 0:
            want[t] = int(table[s_h[t], lb]) * st.bs + p_h[t] % st.bs
    assert np.array_equal(slots, want)
    assert slots[0] == -1 and slots[2] == -1
    # every token with a slot was written there, and nothing else changed
    rows, rows0 = st.k_cache.view(-1, st.H * st.D), k0.view(-1, st.H * st.D)
    written = set()
    for t in np.nonzero(slots >= 0)[0]:
        assert torch.equal(rows[int(slots[t])].view(torch.int16),
                           st.new_k[t].reshape(-1).view(torch.int16))
        written.add(int(slots[t]))
    keep = torch.ones(rows.shape[0], dtype=torch.bool, device=rows.device)
    keep[list(written)] = False
    assert torch.equal(rows[keep].view(torch.int16), rows0[keep].view(torch.int16))


def test_fused_step_without_new_tokens_is_a_plain_decode():
    w = W.small_case(65, S=4, H=4, D=128, bs=16, ctx_lo=1, ctx_hi=300, n_new=0)
    compare_step(w, fused=True)


@pytest.mark.parametrize("pt", [0, 64])
def test_fused_step_with_prefix_groups(pt):
    """With prefix groups the fused step equals copy_blocks + slot mapping +
    cache write + shared-prefix decode bit for bit, and the oracle."""
    from oracle import step as OS
    from tests.gpu_harness import assert_attention_close, out_to_double
    w = W.shared_prefix(cow=True, prompts=3, samples=4, prefix=128, tail_lo=1, tail_hi=40)
    groups = np.array([[p * 4, 4, 128] for p in range(3)], dtype=np.int32)
    st = device_step(w, pt)
    st.plan()
    k0, v0 = st.k_cache.clone(), st.v_cache.clone()
    st.run(attention=False)
    st.decode_shared_prefix(groups)
    torch.cuda.synchronize()
    want = [t.clone() for t in (st.slot_mapping, st.k_cache, st.v_cache, st.out)]
    st.k_cache.copy_(k0)
    st.v_cache.copy_(v0)
    st.out.fill_(float("nan"))
    st.slot_mapping.fill_(-7)
    st.prefix_groups = torch.from_numpy(groups).cuda()
    st.workspace = torch.empty(L.pkv_decode_shared_prefix_workspace_size(
        w.S, w.H, w.D, len(groups), st.max_context_len, pt), dtype=torch.uint8, device="cuda")
    st.run(fused=True)
    torch.cuda.synchronize()
    got = (st.slot_mapping, st.k_cache, st.v_cache, st.out)
    for name, a, b in zip(("slots", "k_cache", "v_cache", "out"), want, got):
        assert torch.equal(a.view(torch.int16) if a.dtype != torch.int64 else a,
                           b.view(torch.int16) if b.dtype != torch.int64 else b), name
    assert_attention_close(out_to_double(st.out), OS.run(w).out, f"fused shared prefix pt{pt}")
