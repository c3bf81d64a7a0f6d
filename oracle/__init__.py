"""fp64 CPU oracle for the paged decode-attention path.

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the
CPU-baseline leg of `bench.py` may import, call, link or execute anything in
this package.  The library under `paged_kv_cache_162_gb300/` never does, and
this package never imports it: the two share no code.

Contents
  oracle.c      decode attention by definition (double), slot mapping,
                reshape_and_cache, copy_blocks -- built by `build.py`
  kernels.py    ctypes wrappers over oracle.c
  allocator.py  the block allocator written from the pages (free list,
                per-physical-block refcounts, share, copy-on-write)
  step.py       one decode step driven by a `workloads.Workload`

Every function is pinned by `tests/test_oracle_*.py` against what the pages
and the mathematics fix (worked examples, closed forms, invariants, an
independent library routine on contiguous K/V).
"""
