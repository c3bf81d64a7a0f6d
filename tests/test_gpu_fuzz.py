"""Seeded random configurations through the whole step (allocation, copies,
slot mapping, cache write, decode; and shared-prefix decode) against the
oracle: sequence counts, head counts (including ones that leave idle warps),
head_dim, block size, dtype, context lengths (including 0), partition size
and group layout all vary."""
import numpy as np
import pytest
import torch

import workloads as W
from paged_kv_cache_162_gb300 import _lib as L
from tests.gpu_harness import assert_attention_close, compare_step, out_to_double

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(12))
def test_random_step(seed):
    rng = np.random.default_rng(4242 + seed)
    dtype = [W.F16, W.BF16][seed % 2]
    D = [64, 128][int(rng.integers(2))]
    bs = [8, 16, 32, 64][int(rng.integers(4))]
    H = int(rng.integers(1, 11))
    S = int(rng.integers(1, 9))
    ctx = rng.integers(0, 700, size=S)
    ctx[rng.random(S) < 0.15] = 0
    n_new = int(rng.integers(1, 4))
    pt = [0, 64, 128, 256][int(rng.integers(4))]
    if pt and pt % bs:
        pt = 0
    w = W.small_case(seed=seed, dtype=dtype, S=S, H=H, D=D, bs=bs, ctx=ctx, n_new=n_new)
    # every third seed runs the device part as pkv_decode_step
    compare_step(w, partition_tokens=pt, fused=seed % 3 == 0)


@pytest.mark.parametrize("seed", range(6))
def test_random_shared_prefix(seed):
    rng = np.random.default_rng(777 + seed)
    dtype = [W.F16, W.BF16][seed % 2]
    D = [64, 128][seed % 2]
    bs = [8, 16, 32][int(rng.integers(3))]
    samples = int(rng.integers(1, 17))
    prompts = int(rng.integers(1, 4))
    prefix = int(rng.integers(2, 12)) * 32
    w = W.shared_prefix(seed=seed, prompts=prompts, samples=samples, prefix=prefix, tail_lo=1,
                        tail_hi=120, H=int(rng.integers(1, 9)), D=D, bs=bs, dtype=dtype,
                        cow=bool(seed % 3 == 0))
    pt = [0, 32, 64][seed % 3]
    r = compare_step(w, partition_tokens=pt)
    st = r["step"]
    groups = np.array([[p * samples, samples, prefix] for p in range(prompts)
                       if rng.random() < 0.8], dtype=np.int32).reshape(-1, 3)
    st.out.fill_(float("nan"))
    st.decode_shared_prefix(groups)
    torch.cuda.synchronize()
    assert_attention_close(out_to_double(st.out), r["ref"].out, f"shared prefix fuzz {seed}")
    # the fused step with the same groups (its cache writes repeat the
    # step's, so the caches do not change) gives the same output bit for bit
    want = st.out.clone()
    st.prefix_groups = torch.from_numpy(groups).cuda()
    st.workspace = torch.empty(L.pkv_decode_shared_prefix_workspace_size(
        w.S, w.H, w.D, len(groups), st.max_context_len, pt), dtype=torch.uint8, device="cuda")
    st.out.fill_(float("nan"))
    st.run(fused=True)
    torch.cuda.synchronize()
    assert torch.equal(st.out.view(torch.int16), want.view(torch.int16))
