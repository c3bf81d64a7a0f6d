"""Host block allocator (pkv_alloc_* of the C ABI) with a Python face.

A global pool of physical blocks with a free list (a stack: the block freed
last is handed out first) and a refcount per physical block: "3.3 页面级显存管理"
3.3.2 and 3.3.4, "vLLM三大核心技术分页内存与共享解码" (Copy-on-Write section),
"3.1 PagedAttention的核心原理" 3.1.2 and 3.1.5.  Every call is
all-or-nothing; running out of blocks raises OutOfBlocks.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._lib import PKV_ERR_INVALID_ARG, OutOfBlocks, PkvError, check, lib  # noqa: F401


def _need_i32(a: np.ndarray, what: str) -> None:
    """Arrays the library writes in place must already be C-contiguous int32
    (a converted copy would leave the caller's array unchanged)."""
    if not (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous):
        raise PkvError(PKV_ERR_INVALID_ARG, f"{what} must be a C-contiguous int32 numpy array")


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32).ravel())


class BlockAllocator:
    def __init__(self, num_blocks: int, initial_free=None):
        h = ctypes.c_void_p()
        if initial_free is None:
            check(lib().pkv_alloc_create(int(num_blocks), ctypes.addressof(h)), "alloc_create")
        else:
            f = _i32(initial_free)
            check(lib().pkv_alloc_create_with_order(int(num_blocks), f.ctypes.data, len(f),
                                                    ctypes.addressof(h)), "alloc_create_with_order")
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None) and self._h.value:
            lib().pkv_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def alloc(self, n: int) -> list:
        out = np.empty(max(int(n), 1), dtype=np.int32)
        check(lib().pkv_alloc_blocks(self._h, int(n), out.ctypes.data), "alloc_blocks")
        return out[:int(n)].tolist()

    def incref(self, ids) -> None:
        a = _i32(ids)
        check(lib().pkv_alloc_incref(self._h, a.ctypes.data, len(a)), "alloc_incref")

    def decref(self, ids) -> int:
        a = _i32(ids)
        freed = ctypes.c_int32(0)
        check(lib().pkv_alloc_decref(self._h, a.ctypes.data, len(a), ctypes.addressof(freed)),
              "alloc_decref")
        return int(freed.value)

    def cow(self, block: int):
        out, needs = ctypes.c_int32(0), ctypes.c_int32(0)
        check(lib().pkv_alloc_cow(self._h, int(block), ctypes.addressof(out),
                                  ctypes.addressof(needs)), "alloc_cow")
        return int(out.value), bool(needs.value)

    def append_row(self, row: np.ndarray, num_blocks: int, ctx_before: int, n_new: int,
                   block_size: int):
        """In place on `row` (int32, capacity len(row)); returns (num_blocks, pairs)."""
        _need_i32(row, "row")
        nb = ctypes.c_int32(int(num_blocks))
        npairs = ctypes.c_int32(0)
        pairs = np.empty(2 * (int(n_new) // int(block_size) + 2), dtype=np.int64)
        check(lib().pkv_alloc_append(self._h, row.ctypes.data, ctypes.addressof(nb), len(row),
                                     int(ctx_before), int(n_new), int(block_size),
                                     pairs.ctypes.data, ctypes.addressof(npairs)), "alloc_append")
        return int(nb.value), pairs[:2 * npairs.value].reshape(-1, 2)

    def append(self, table: list, ctx_before: int, n_new: int, block_size: int) -> list:
        """Same as append_row on a Python list (grown in place)."""
        need = -(-(int(ctx_before) + int(n_new)) // int(block_size))
        row = np.full(max(need, len(table), 1), -1, dtype=np.int32)
        row[:len(table)] = table
        nb, pairs = self.append_row(row, len(table), ctx_before, n_new, block_size)
        table[:] = row[:nb].tolist()
        return [tuple(int(x) for x in p) for p in pairs]

    def append_batch(self, tables: np.ndarray, nblocks: np.ndarray, ctx_before, n_new,
                     block_size: int):
        """append() for every row of `tables` ([S, MB] int32, in place; nblocks
        [S] int32 in place) in one native call.  Returns the copy pairs
        [P, 2]; raises OutOfBlocks (rows before the failing one are done)."""
        _need_i32(tables, "tables")
        _need_i32(nblocks, "nblocks")
        S, MB = tables.shape
        cb = _i32(ctx_before)
        nn = _i32(n_new)
        cap = int((nn.astype(np.int64) // int(block_size) + 2).sum())
        pairs = np.empty(2 * max(cap, 1), dtype=np.int64)
        npairs, ndone = ctypes.c_int32(0), ctypes.c_int32(0)
        check(lib().pkv_alloc_append_batch(self._h, tables.ctypes.data, nblocks.ctypes.data, S, MB,
                                           cb.ctypes.data, nn.ctypes.data, int(block_size),
                                           pairs.ctypes.data, cap, ctypes.addressof(npairs),
                                           ctypes.addressof(ndone)), "alloc_append_batch")
        return pairs[:2 * npairs.value].reshape(-1, 2)

    def fork(self, tables: np.ndarray, nblocks: np.ndarray, parents) -> None:
        """Row s becomes a copy of row parents[s] (in place), sharing its
        blocks; one native call, all-or-nothing."""
        _need_i32(tables, "tables")
        _need_i32(nblocks, "nblocks")
        S, MB = tables.shape
        par = _i32(parents)
        check(lib().pkv_alloc_fork(self._h, tables.ctypes.data, nblocks.ctypes.data, S, MB,
                                   par.ctypes.data), "alloc_fork")

    def refcount(self, block: int) -> int:
        rc = ctypes.c_int32(0)
        check(lib().pkv_alloc_refcount(self._h, int(block), ctypes.addressof(rc)),
              "alloc_refcount")
        return int(rc.value)

    @property
    def num_blocks(self) -> int:
        return int(lib().pkv_alloc_num_blocks(self._h))

    @property
    def num_free(self) -> int:
        return int(lib().pkv_alloc_num_free(self._h))

    @property
    def num_shared(self) -> int:
        return int(lib().pkv_alloc_num_shared(self._h))


def plan_step(alloc: BlockAllocator, tables_pre: np.ndarray, nblocks_pre: np.ndarray,
              ctx_before: np.ndarray, n_new: np.ndarray, block_size: int):
    """Host part of one decode step: for every sequence in order, make room
    for its new tokens (copy-on-write of shared blocks, then new blocks).

    Returns (tables [S, MB] int32, nblocks [S] int32, pairs [P, 2] int64);
    the pairs have passed pkv_check_copy_pairs (pkv_copy_blocks'
    precondition) before they are returned.
    """
    tables = np.array(tables_pre, dtype=np.int32, copy=True, order="C")
    nb = np.array(nblocks_pre, dtype=np.int32, copy=True)
    pairs = alloc.append_batch(tables, nb, ctx_before, n_new, block_size)
    check_copy_pairs(pairs, alloc.num_blocks)
    return tables, nb, pairs


def check_copy_pairs(pairs: np.ndarray, num_blocks: int) -> None:
    """Raises PkvError unless the (src, dst) copy list meets pkv_copy_blocks'
    precondition: ids in [0, num_blocks), no dst twice, no dst also a src."""
    p = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    check(lib().pkv_check_copy_pairs(p.ctypes.data if len(p) else None, len(p), int(num_blocks)),
          "check_copy_pairs")


def plan_swap_out(gpu: BlockAllocator, host: BlockAllocator, table):
    """CPU swap-out of one sequence ("3.3 页面级显存管理" 3.3.3): a host block
    for each of its GPU blocks.  Returns (host_ids, pairs [P, 2] gpu->host).
    After the copy, call gpu.decref(table) to release the GPU blocks."""
    host_ids = host.alloc(len(table))
    pairs = np.array(list(zip(table, host_ids)), dtype=np.int64).reshape(-1, 2)
    return host_ids, pairs


def plan_swap_in(gpu: BlockAllocator, host: BlockAllocator, host_ids):
    """CPU swap-in: fresh GPU blocks for a swapped-out sequence.  Returns
    (table, pairs [P, 2] host->gpu).  After the copy, call
    host.decref(host_ids) to release the host blocks."""
    table = gpu.alloc(len(host_ids))
    pairs = np.array(list(zip(host_ids, table)), dtype=np.int64).reshape(-1, 2)
    return table, pairs

