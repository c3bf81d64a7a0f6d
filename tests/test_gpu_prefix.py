"""Shared-prefix decode (one read of each group's prefix, tensor cores)
through the C ABI: against the fp64 oracle and against the plain decode
entry point, for group sizes 1..16, both dtypes, head_dim 64/128 and several
block sizes, with grouped and ungrouped sequences in one batch."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_harness import assert_attention_close, compare_step, device_step, out_to_double

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["mma", "tcgen05"], autouse=True)
def prefix_kernel(request, monkeypatch):
    """Every test runs with the default prefix kernel and with the
    tensor-core one (which serves head_dim 128)."""
    if request.param == "tcgen05":
        monkeypatch.setenv("PKV_PREFIX_KERNEL", "tcgen05")
    else:
        monkeypatch.delenv("PKV_PREFIX_KERNEL", raising=False)
    return request.param


def _groups(w, samples, prefix, every=1):
    prompts = w.S // samples
    return np.array([[p * samples, samples, prefix] for p in range(0, prompts, every)],
                    dtype=np.int32)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("D,bs", [(128, 16), (64, 32), (128, 8)])
@pytest.mark.parametrize("samples", [1, 3, 8, 16])
def test_prefix_groups_small(dtype, D, bs, samples):
    w = W.shared_prefix(seed=samples * 10 + bs + D, prompts=4, samples=samples, prefix=128,
                        tail_lo=1, tail_hi=90, H=6, D=D, bs=bs, dtype=dtype)
    r = compare_step(w, partition_tokens=64)           # plain decode vs the oracle
    st = r["step"]
    ref = r["ref"].out
    plain = out_to_double(st.out)
    st.out.fill_(float("nan"))
    # every other prompt grouped, the rest decoded as usual
    st.decode_shared_prefix(_groups(w, samples, 128, every=2))
    torch.cuda.synchronize()
    got = out_to_double(st.out)
    assert_attention_close(got, ref, f"shared prefix {dtype} D{D} bs{bs} n{samples}")
    np.testing.assert_allclose(got, plain, atol=2e-3, rtol=1e-2)


def test_prefix_shorter_than_a_partition_falls_back():
    w = W.shared_prefix(seed=5, prompts=2, samples=4, prefix=48, tail_lo=1, tail_hi=30, H=4,
                        D=128)
    r = compare_step(w, partition_tokens=64)
    st = r["step"]
    st.decode_shared_prefix(_groups(w, 4, 48))
    torch.cuda.synchronize()
    assert_attention_close(out_to_double(st.out), r["ref"].out, "short prefix")


@pytest.mark.parametrize("cow", [False, True])
def test_shared_prefix_full_workload(cow):
    """32 prompts x 8 samples sharing a 1024-token prefix (64 blocks)."""
    w = W.shared_prefix(cow=cow)
    r = compare_step(w)
    st = r["step"]
    st.out.fill_(float("nan"))
    st.decode_shared_prefix(_groups(w, 8, 1024))
    torch.cuda.synchronize()
    assert_attention_close(out_to_double(st.out), r["ref"].out, "shared prefix full")


def test_many_members_with_long_tails():
    """384 members (48 prompts x 8 samples), so the plan places the partial
    items in two chunks of its threads, with tails up to 256 tokens, so the
    longest-first order is on; each member's tail is one partition and is
    merged with the prefix partial in registers."""
    w = W.shared_prefix(seed=23, prompts=48, samples=8, prefix=1024, tail_lo=1, tail_hi=256, H=8,
                        D=128)
    r = compare_step(w)
    st = r["step"]
    st.out.fill_(float("nan"))
    st.decode_shared_prefix(_groups(w, 8, 1024))
    torch.cuda.synchronize()
    assert_attention_close(out_to_double(st.out), r["ref"].out, "384 members, long tails")


@pytest.mark.parametrize("scale", [0.0, -0.2])
def test_zero_and_negative_scale(scale):
    """The softmax max must be taken after scaling: with a negative scale the
    largest scaled logit comes from the smallest dot product."""
    w = W.shared_prefix(seed=11, prompts=2, samples=4, prefix=128, tail_lo=1, tail_hi=60, H=4,
                        D=128)
    w.scale = scale
    r = compare_step(w, partition_tokens=64)
    st = r["step"]
    st.out.fill_(float("nan"))
    st.decode_shared_prefix(_groups(w, 4, 128))
    torch.cuda.synchronize()
    assert_attention_close(out_to_double(st.out), r["ref"].out, f"scale {scale}")


@pytest.mark.parametrize("bs", [16, 64])
def test_groups_of_one_with_empty_and_short_contexts(bs):
    """Groups of one sequence (a sequence always shares its prefix with
    itself) beside ungrouped sequences, some with empty contexts: the
    ungrouped and tail items run as groups of one with masked ragged tiles."""
    ctx = [0, 300, 5, 0, 170, 64, 17, 129]
    w = W.small_case(seed=bs + 3, S=len(ctx), H=8, D=128, bs=bs, ctx=ctx, n_new=1, NB=80)
    r = compare_step(w, partition_tokens=64)
    st = r["step"]
    st.out.fill_(float("nan"))
    groups = np.array([[1, 1, 256], [4, 1, 128], [5, 1, 64], [7, 1, 128]], dtype=np.int32)
    st.decode_shared_prefix(groups)
    torch.cuda.synchronize()
    got = out_to_double(st.out)
    assert_attention_close(got, r["ref"].out, f"groups of one bs{bs}")
    assert np.all(got[0] == 0.0) and np.all(got[3] == 0.0)


def test_repeated_calls_same_output_and_no_timeout():
    """Hundreds of back-to-back calls on the full shared_prefix_cow shape:
    every output is the first one bit for bit, and no in-kernel wait gives
    up (the device error word stays clear).  The tensor-core kernel hands
    work between its warps through mbarriers; a phase mix-up between them
    shows up here as a wait that runs out (PKV_DEVERR_TIMEOUT) or a
    different output."""
    from paged_kv_cache_162_gb300 import _lib as L
    w = W.shared_prefix(cow=True)
    st = device_step(w, 0)
    st.run()
    torch.cuda.synchronize()
    groups = _groups(w, 8, 1024)
    assert L.pkv_get_device_errors() == 0
    st.decode_shared_prefix(groups)
    first = st.out.clone()
    for i in range(20):
        for _ in range(20):
            st.decode_shared_prefix(groups)
        torch.cuda.synchronize()
        assert L.pkv_get_device_errors() == 0, f"device error after {20 * (i + 1)} calls"
        assert torch.equal(st.out.view(torch.int16), first.view(torch.int16))
