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
    dev_in, host_in, _ = st.pack_inputs()
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


@pytest.mark.parametrize("make", [
    lambda: W.small_case(92, S=7, H=8, D=128, ctx_lo=1, ctx_hi=900, n_new=3),
    lambda: W.shared_prefix(cow=True, prompts=2, samples=4, prefix=256, tail_lo=1, tail_hi=40),
])
@pytest.mark.parametrize("fused", [False, True])
def test_tokens_and_output_in_pinned_host_memory(make, fused):
    """q and the new K/V read by the kernels from pinned host memory, the
    output written there, one upload of the integer inputs: the graph's
    result is bit-identical to the eager device-resident step, and a new
    value written into the host buffer reaches the next replay."""
    w = make()
    st = device_step(w, 0)
    st.run(fused=fused)
    torch.cuda.synchronize()
    ref = st.out.clone()
    dev_in, host_in, (up_dev, up_host) = st.pack_inputs(on_host=("q", "new_k", "new_v"))
    for n in ("q", "new_k", "new_v"):
        t = getattr(st, n)
        assert not t.is_cuda and t.is_pinned()
        assert t.data_ptr() == host_in.data_ptr() + st.input_offsets[n]
    assert up_host.data_ptr() == host_in.data_ptr() + st.input_offsets["block_tables"]
    host_out = st.pin_output()
    stream = torch.cuda.Stream()
    g = StepGraph(st, stream, h2d=[(up_dev, up_host)], d2h=[], fused=fused)
    with torch.cuda.stream(stream):
        up_dev.zero_()
    host_out.zero_()
    for _ in range(2):
        g.replay()
        stream.synchronize()
        assert torch.equal(host_out.view(torch.int16), ref.cpu().view(torch.int16))
    # a new query for sequence 0, written where the kernels read it
    st.q[0].copy_(-st.q[0])
    g.replay()
    stream.synchronize()
    assert not torch.equal(host_out[0].view(torch.int16), ref[0].cpu().view(torch.int16))
    assert torch.equal(host_out[1:].view(torch.int16), ref[1:].cpu().view(torch.int16))
