"""The decode entry point that allocates nothing.

Some callers may not allocate device memory (a plugin inside a runtime that
owns all device memory, a latency-critical loop, a plain C host program);
pkv_paged_attention_decode_noalloc serves them with a scratch array built
into the library.  These tests call it through the C ABI and check it
against pkv_paged_attention_decode (with a caller workspace) on two calls in
a row, each with its own inputs, within the attention tolerance the other
tests use.  The file is named to be collected last; it builds all of its
inputs itself, so it passes alone in a fresh process too.
"""
import numpy as np
import pytest
import torch

import workloads as W
from paged_kv_cache_162_gb300 import _lib as L
from tests.gpu_harness import ATOL, RTOL, device_step

pytestmark = pytest.mark.gpu


def _noalloc(st, partition_tokens):
    out = torch.full_like(st.out, float("nan"))
    L.pkv_paged_attention_decode_noalloc(
        out, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, st.S, st.H, st.D,
        st.bs, st.NB, st.MB, st.max_context_len, st.scale, L.PKV_BF16 if st.dtype == torch.bfloat16
        else L.PKV_F16, partition_tokens)
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    # call 1: several split-K partitions per sequence; call 2: other shapes,
    # so the scratch holds the first call's leftovers when the second runs
    cases = [
        (W.small_case(seed=41, dtype=W.F16, S=16, H=32, D=128, bs=16, ctx_lo=300, ctx_hi=2048),
         128),
        (W.small_case(seed=42, dtype=W.BF16, S=5, H=6, D=64, bs=32, ctx_lo=1, ctx_hi=700), 64),
    ]
    need = [L.pkv_decode_workspace_size(w.S, w.H, w.D, int(w.context_lens.max()), pt)
            for w, pt in cases]
    assert all(0 < n <= L.PKV_NOALLOC_SCRATCH_BYTES for n in need)
    for w, pt in cases:
        st = device_step(w, pt)
        st.run()                       # caller-workspace entry point
        torch.cuda.synchronize()
        ref = st.out.float().cpu().double().numpy()
        got = _noalloc(st, pt).float().cpu().double().numpy()
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    assert L.pkv_get_device_errors() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = W.small_case(seed=43, S=2, H=4, D=128, bs=16, ctx_lo=10, ctx_hi=40)
    st = device_step(w, 0)
    st.plan()
    big_S = 4096  # S x 32 heads x 16 partitions of fp32 partials: far above 16 MiB
    assert L.pkv_decode_workspace_size(big_S, 32, 128, 4096, 256) > L.PKV_NOALLOC_SCRATCH_BYTES
    with pytest.raises(L.PkvError) as e:
        L.pkv_paged_attention_decode_noalloc(
            st.out, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, big_S, 32,
            128, 16, st.NB, 256, 4096, st.scale, L.PKV_F16, 256)
    assert e.value.status == L.PKV_ERR_WORKSPACE
    assert "scratch" in L.pkv_last_error_string()
