"""One decode step captured in a CUDA graph with its inputs packed into one
buffer: the graph's upload, kernels and download reproduce the eager step."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as OS
from tests.gpu_harness import assert_attention_close, device_step
from paged_kv_cache_162_gb300.engine import StepGraph

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [
    lambda: W.small_case(91, S=7, H=8, D=128, ctx_lo=1, ctx_hi=900, n_new=3),
    lambda: W.shared_prefix(cow=True, prompts=2, samples=4, prefix=256, tail_lo=1, tail_hi=40),
])
def test_packed_inputs_in_a_graph(make):
    w = make()
    st = device_step(w, 0)
    st.run()
    torch.cuda.synchronize()
    ref = st.out.clone()
    dev_in, host_in = st.pack_inputs()
    # every input now lives in the one buffer, at a 256-byte aligned offset
    base = dev_in.data_ptr()
    for name, off in st.input_offsets.items():
        assert off % 256 == 0
        assert getattr(st, name).data_ptr() == base + off
    assert host_in.is_pinned() and host_in.numel() == dev_in.numel()
    stream = torch.cuda.Stream()
    host_out = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    g = StepGraph(st, stream, h2d=[(dev_in, host_in)], d2h=[(host_out, st.out)])
    # wipe the device copy and the output: the replay must bring both back
    with torch.cuda.stream(stream):
        dev_in.zero_()
        st.out.zero_()
    for _ in range(2):
        g.replay()
        stream.synchronize()
        assert torch.equal(host_out.view(torch.int16), ref.cpu().view(torch.int16))
    # the graph's output against the oracle's step, and the cache it wrote
    ref_step = OS.run(w)
    assert_attention_close(host_out.float().double().numpy(), ref_step.out, w.name)
    ids = torch.from_numpy(ref_step.pool_ids.astype(np.int64)).cuda()
    for cache, pool in ((st.k_cache, ref_step.k_pool), (st.v_cache, ref_step.v_pool)):
        got = cache.view(torch.int16).index_select(0, ids).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, pool)
