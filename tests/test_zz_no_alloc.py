"""The decode entry point that allocates nothing.

Some callers may not allocate device memory (a plugin inside a runtime that
owns all device memory, a latency-critical loop, a plain C host program);
pkv_paged_attention_decode_noalloc serves them with a scratch array built
into the library.  These tests call it through the C ABI and check it
against pkv_paged_attention_decode (with a caller workspace) and against
the fp64 oracle on two calls in a row, each with its own inputs, within the
attention tolerance the other tests use.  The file is named to be collected
last; it builds all of its inputs itself, so it passes alone in a fresh
process too.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as OS
from paged_kv_cache_162_gb300 import _lib as L
from tests.gpu_harness import ATOL, RTOL, assert_attention_close, device_step, out_to_double

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
        oracle = OS.run(w).out
        st = device_step(w, pt)
        st.run()                       # caller-workspace entry point
        torch.cuda.synchronize()
        ref = out_to_double(st.out)
        got = out_to_double(_noalloc(st, pt))
        assert np.all(np.isfinite(got))
        # the same partition size runs the same kernels on the same data
        assert np.array_equal(got, ref)
        assert_attention_close(got, oracle, f"noalloc {w.name}")
    assert L.pkv_get_device_errors() == 0


def test_noalloc_automatic_partition_raised_to_fit_the_scratch():
    """With partition_tokens = 0 the smallest automatic partition is raised
    until the partials fit the built-in scratch.  64 sequences x 32 heads
    with one 2048-token context need 33.5 MB of partials at 64-token
    partitions and fit at 256; the call runs there, within the attention
    tolerance of the oracle, twice in a row."""
    ctx = np.r_[np.random.default_rng(44).integers(1, 200, 63), 2048]
    w = W.small_case(seed=44, dtype=W.F16, S=64, H=32, D=128, bs=16, ctx=ctx)
    max_ctx = int(w.context_lens.max())
    assert L.pkv_decode_workspace_size(w.S, w.H, w.D, max_ctx, 64) > L.PKV_NOALLOC_SCRATCH_BYTES
    assert L.pkv_decode_workspace_size(w.S, w.H, w.D, max_ctx, 256) <= L.PKV_NOALLOC_SCRATCH_BYTES
    oracle = OS.run(w).out
    st = device_step(w, 0)
    st.run()
    torch.cuda.synchronize()
    ws_out = out_to_double(st.out)
    for _ in range(2):
        got = out_to_double(_noalloc(st, 0))
        assert_attention_close(got, oracle, "noalloc automatic")
        assert np.all(np.abs(got - ws_out) <= ATOL + RTOL * np.abs(ws_out))
    assert L.pkv_get_device_errors() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """A size whose partials do not fit is refused before any launch.  Every
    buffer passed is as large as the call claims (4096 sequences x 32 heads
    x 128 dims, 256-entry tables of block 0 in a one-block pool), so even a
    call that got past the size check would stay inside its buffers."""
    S, H, D, bs, MB, max_ctx = 4096, 32, 128, 16, 256, 4096
    assert L.pkv_decode_workspace_size(S, H, D, max_ctx, 256) > L.PKV_NOALLOC_SCRATCH_BYTES
    dev = "cuda"
    q = torch.zeros(S, H, D, dtype=torch.float16, device=dev)
    out = torch.zeros_like(q)
    k_cache = torch.zeros(1, bs, H, D, dtype=torch.float16, device=dev)
    v_cache = torch.zeros_like(k_cache)
    block_tables = torch.zeros(S, MB, dtype=torch.int32, device=dev)
    context_lens = torch.full((S,), bs, dtype=torch.int32, device=dev)
    for pt in (256, 0):
        with pytest.raises(L.PkvError) as e:
            L.pkv_paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables,
                                                 context_lens, S, H, D, bs, 1, MB, max_ctx,
                                                 D ** -0.5, L.PKV_F16, pt)
        assert e.value.status == L.PKV_ERR_WORKSPACE
        assert "scratch" in L.pkv_last_error_string()
    torch.cuda.synchronize()
    assert bool((out == 0).all())
