"""The library at the edges of its sizes, against the oracle: the most
sequences a call takes (32767: the sequence id is 15 bits of a packed work
item), the most partitions of one sequence (65535: 16 bits), and many
heads (head groups of 4 warps with idle warps in the last one).  One past
each limit is rejected on the host (CPU tests)."""
import numpy as np
import pytest

import workloads as W
from tests.gpu_harness import compare_step

pytestmark = pytest.mark.gpu


def test_most_sequences():
    rng = np.random.default_rng(32767)
    S = 32767
    ctx = rng.integers(0, 49, size=S)
    ctx[rng.random(S) < 0.05] = 0
    w = W.small_case(seed=9001, S=S, H=2, D=64, bs=16, ctx=ctx, n_new=1)
    compare_step(w)


def test_most_partitions_of_one_sequence():
    """65535 partitions of 64 tokens: 4,194,240 tokens of one head, merged
    by one warp through 2048 chunks of 32 partitions."""
    ctx = [65535 * 64]
    w = W.small_case(seed=9002, S=1, H=1, D=64, bs=64, ctx=ctx, n_new=1)
    compare_step(w, partition_tokens=64)


@pytest.mark.parametrize("H,D", [(64, 128), (37, 64)])
def test_many_heads(H, D):
    w = W.small_case(seed=9003 + H, S=5, H=H, D=D, bs=16, ctx_lo=0, ctx_hi=400, n_new=2)
    compare_step(w)
