"""Out-of-range ids are never dereferenced: the kernels skip the access and
set a bit in the device error word, which the host reads.  Every bad id
below is caught by the kernels' own bounds checks.  A bounded in-kernel wait
that runs out reports through the same word and leaves the context usable."""
import numpy as np
import pytest
import torch

import paged_kv_cache_162_gb300 as P
from paged_kv_cache_162_gb300 import _lib as L
from paged_kv_cache_162_gb300 import engine as E

pytestmark = pytest.mark.gpu


def _caches(NB=8, bs=16, H=4, D=64):
    k = torch.randn(NB, bs, H, D, device="cuda").half()
    v = torch.randn(NB, bs, H, D, device="cuda").half()
    return k, v


def test_bad_block_id_in_table_sets_flag_and_is_skipped():
    P.pkv_get_device_errors()  # clear
    k, v = _caches()
    q = torch.randn(2, 4, 64, device="cuda").half()
    out = torch.empty_like(q)
    bt = torch.tensor([[0, 1], [2, 10_000]], dtype=torch.int32, device="cuda")
    ctx = torch.tensor([20, 30], dtype=torch.int32, device="cuda")
    E.paged_attention_decode(out, q, k, v, bt, ctx)
    assert P.pkv_get_device_errors() & L.PKV_DEVERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    assert P.pkv_get_device_errors() == 0  # cleared by the read


def test_bad_context_len_is_clamped_and_flagged():
    P.pkv_get_device_errors()
    k, v = _caches()
    q = torch.randn(1, 4, 64, device="cuda").half()
    out = torch.empty_like(q)
    bt = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
    ctx = torch.tensor([-5], dtype=torch.int32, device="cuda")
    E.paged_attention_decode(out, q, k, v, bt, ctx)
    assert P.pkv_get_device_errors() & L.PKV_DEVERR_CONTEXT
    assert torch.all(out.float() == 0)


def test_bad_slot_and_position_and_copy_pair():
    P.pkv_get_device_errors()
    k, v = _caches()
    k0, v0 = k.clone(), v.clone()
    key = torch.randn(2, 4, 64, device="cuda").half()
    slots = torch.tensor([8 * 16, -1], dtype=torch.int64, device="cuda")  # first is one past the end
    E.reshape_and_cache(key, key, k, v, slots)
    assert P.pkv_get_device_errors() & L.PKV_DEVERR_SLOT
    assert torch.equal(k, k0) and torch.equal(v, v0)
    bt = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
    out = torch.empty(2, dtype=torch.int64, device="cuda")
    E.compute_slot_mapping(out, bt, torch.tensor([0, 3], dtype=torch.int32, device="cuda"),
                           torch.tensor([40, 1], dtype=torch.int32, device="cuda"), 16)
    assert P.pkv_get_device_errors() & L.PKV_DEVERR_POSITION
    assert out.tolist() == [-1, -1]
    # a position in a logical block the table has not mapped (-1)
    bt = torch.tensor([[2, -1]], dtype=torch.int32, device="cuda")
    E.compute_slot_mapping(out, bt, torch.tensor([0, 0], dtype=torch.int32, device="cuda"),
                           torch.tensor([5, 17], dtype=torch.int32, device="cuda"), 16)
    assert P.pkv_get_device_errors() & L.PKV_DEVERR_BLOCK_ID
    assert out.tolist() == [2 * 16 + 5, -1]
    pairs = torch.tensor([[0, 8]], dtype=torch.int64, device="cuda")
    E.copy_blocks(k, v, pairs)
    assert P.pkv_get_device_errors() & L.PKV_DEVERR_BLOCK_ID
    assert torch.equal(k, k0)


def test_bad_prefix_group_is_flagged_and_skipped():
    """A group whose members run past the batch is never used: flagged,
    its sequences decoded as usual."""
    import workloads as W
    from tests.gpu_harness import assert_attention_close, compare_step, out_to_double
    P.pkv_get_device_errors()
    w = W.shared_prefix(seed=3, prompts=2, samples=4, prefix=64, tail_lo=1, tail_hi=40, H=4,
                        D=64)
    r = compare_step(w, partition_tokens=64)
    st = r["step"]
    bad = np.array([[0, 4, 64], [6, 4, 64]], dtype=np.int32)  # the second runs past S = 8
    st.decode_shared_prefix(bad)
    torch.cuda.synchronize()
    assert P.pkv_get_device_errors() & L.PKV_DEVERR_GROUP
    assert_attention_close(out_to_double(st.out), r["ref"].out, "bad group")


@pytest.mark.parametrize("polls", [1, 1 << 12, 1 << 20])
def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable(polls, monkeypatch):
    """A wait that nothing completes runs out after its bounded number of
    polls: the kernel sets PKV_DEVERR_TIMEOUT, frees its tensor memory and
    returns; the host reads the bit, and the next calls -- the tcgen05
    prefix kernel, which takes tensor memory again -- run normally."""
    import time
    import workloads as W
    from tests.gpu_harness import assert_attention_close, compare_step, out_to_double
    P.pkv_get_device_errors()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    L.pkv_selftest_bounded_wait(polls)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert P.pkv_get_device_errors() == L.PKV_DEVERR_TIMEOUT
    print(f"{polls} polls gave up after {dt * 1e3:.2f} ms")
    assert dt < 30.0
    L.pkv_sync_check()
    monkeypatch.setenv("PKV_PREFIX_KERNEL", "tcgen05")
    w = W.shared_prefix(seed=5, prompts=2, samples=4, prefix=256, tail_lo=1, tail_hi=40, H=4,
                        D=128)
    r = compare_step(w, partition_tokens=128)
    st = r["step"]
    st.out.fill_(float("nan"))
    st.decode_shared_prefix(np.array([[0, 4, 256], [4, 4, 256]], dtype=np.int32))
    torch.cuda.synchronize()
    assert_attention_close(out_to_double(st.out), r["ref"].out, "after a timed-out wait")
    assert P.pkv_get_device_errors() == 0


def test_bounded_wait_rejects_out_of_range_polls():
    for bad in (0, -1, (1 << 20) + 1):
        with pytest.raises(L.PkvError):
            L.pkv_selftest_bounded_wait(bad)
