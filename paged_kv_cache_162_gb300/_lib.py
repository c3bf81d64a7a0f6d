"""ctypes binding of libpagedkv.so: the C ABI of include/pagedkv.h under the
same names.  Argument marshalling only -- every computation runs in the
library.  A pointer argument may be an int address, a torch.Tensor
(data_ptr()) or a numpy array (host memory); `stream` may be None (the
current torch CUDA stream), an int handle or a torch.cuda.Stream.

Loading fails loudly if the library has not been built: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libpagedkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_UNSUPPORTED = 2
PKV_ERR_OOM = 3
PKV_ERR_WORKSPACE = 4
PKV_ERR_CUDA = 5
PKV_ERR_HOST_MEMORY = 6
PKV_F16 = 0
PKV_BF16 = 1
PKV_DEVERR_BLOCK_ID = 0x1
PKV_DEVERR_SLOT = 0x2
PKV_DEVERR_CONTEXT = 0x4
PKV_DEVERR_POSITION = 0x8
PKV_DEVERR_GROUP = 0x10
PKV_DEVERR_TIMEOUT = 0x20
PKV_NOALLOC_SCRATCH_BYTES = 16 << 20
PKV_SWAP_OUT = 0
PKV_SWAP_IN = 1

_STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
                 3: "PKV_ERR_OOM", 4: "PKV_ERR_WORKSPACE", 5: "PKV_ERR_CUDA",
                 6: "PKV_ERR_HOST_MEMORY"}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class OutOfBlocks(PkvError, MemoryError):
    pass


_P = ctypes.c_void_p
_I = ctypes.c_int
_I32 = ctypes.c_int32
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# name -> (restype, argtypes); the order follows include/pagedkv.h
SIGNATURES = {
    "pkv_last_error_string": (ctypes.c_char_p, []),
    "pkv_version": (ctypes.c_char_p, []),
    "pkv_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "pkv_paged_attention_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                        _I, _P, _SZ, _P]),
    "pkv_decode_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                             _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "pkv_decode_shared_prefix_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "pkv_paged_attention_decode_shared_prefix": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                                      _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "pkv_paged_attention_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                _I, _F, _I, _I, _P]),
    "pkv_compute_slot_mapping": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "pkv_reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pkv_copy_blocks": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pkv_check_copy_pairs": (_I, [_P, _I32, _I32]),
    "pkv_swap_blocks": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "pkv_sync_check": (_I, [_P]),
    "pkv_get_device_errors": (_I, [_P]),
    "pkv_selftest_bounded_wait": (_I, [ctypes.c_int64, _P]),
    "pkv_alloc_create": (_I, [_I32, _P]),
    "pkv_alloc_create_with_order": (_I, [_I32, _P, _I32, _P]),
    "pkv_alloc_destroy": (None, [_P]),
    "pkv_alloc_blocks": (_I, [_P, _I32, _P]),
    "pkv_alloc_incref": (_I, [_P, _P, _I32]),
    "pkv_alloc_decref": (_I, [_P, _P, _I32, _P]),
    "pkv_alloc_cow": (_I, [_P, _I32, _P, _P]),
    "pkv_alloc_append": (_I, [_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P]),
    "pkv_alloc_append_batch": (_I, [_P, _P, _P, _I32, _I32, _P, _P, _I32, _P, _I32, _P, _P]),
    "pkv_alloc_fork": (_I, [_P, _P, _P, _I32, _I32, _P]),
    "pkv_alloc_refcount": (_I, [_P, _I32, _P]),
    "pkv_alloc_num_blocks": (_I32, [_P]),
    "pkv_alloc_num_free": (_I32, [_P]),
    "pkv_alloc_num_shared": (_I32, [_P]),
    "pkv_beam_inputs_bytes": (_SZ, [_I32, _I32]),
    "pkv_beam_step": (_I, [_P, _P, _P, _P, _P, _I32, _I32, _P, _P, _SZ, _P, _P, _P, _P, _P, _P,
                           _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P, _P]),
    "pkv_beam_search_create": (_I, [_P, _P, _P, _P, _I32, _I32, _P, _P, _P, _SZ, _P, _P, _P, _P,
                                    _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "pkv_beam_search_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P]),
    "pkv_beam_search_destroy": (None, [_P]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                f"g.build()\"` (no fallback implementation exists)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def ptr(x) -> int | None:
    """Address of a tensor / numpy array / int (None stays None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(status: int, what: str = "") -> None:
    if status != PKV_OK:
        msg = lib().pkv_last_error_string().decode(errors="replace")
        exc = OutOfBlocks if status == PKV_ERR_OOM else PkvError
        raise exc(status, msg or what)


# ---------------------------------------------------------------- entries
def pkv_last_error_string() -> str:
    return lib().pkv_last_error_string().decode(errors="replace")


def pkv_version() -> str:
    return lib().pkv_version().decode()


def pkv_decode_workspace_size(S, H, D, max_context_len, partition_tokens=0) -> int:
    return int(lib().pkv_decode_workspace_size(S, H, D, max_context_len, partition_tokens))


def pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, S, H, D, bs,
                               NB, MB, max_context_len, scale, dtype, partition_tokens, workspace,
                               workspace_bytes, stream=None) -> None:
    check(lib().pkv_paged_attention_decode(
        ptr(out), ptr(q), ptr(k_cache), ptr(v_cache), ptr(block_tables), ptr(context_lens), S, H,
        D, bs, NB, MB, max_context_len, float(scale), int(dtype), partition_tokens, ptr(workspace),
        int(workspace_bytes), stream_handle(stream)), "paged_attention_decode")


def pkv_decode_step(out, q, key, value, k_cache, v_cache, block_tables, context_lens, seq_idx, pos,
                    slot_mapping, prefix_groups, G, T, S, H, D, bs, NB, MB, max_context_len, scale,
                    dtype, partition_tokens, workspace, workspace_bytes, stream=None) -> None:
    check(lib().pkv_decode_step(
        ptr(out), ptr(q), ptr(key), ptr(value), ptr(k_cache), ptr(v_cache), ptr(block_tables),
        ptr(context_lens), ptr(seq_idx), ptr(pos), ptr(slot_mapping), ptr(prefix_groups), G, T, S,
        H, D, bs, NB, MB, max_context_len, float(scale), int(dtype), partition_tokens,
        ptr(workspace), int(workspace_bytes), stream_handle(stream)), "decode_step")


def pkv_decode_shared_prefix_workspace_size(S, H, D, G, max_context_len, partition_tokens=0):
    return int(lib().pkv_decode_shared_prefix_workspace_size(S, H, D, G, max_context_len,
                                                             partition_tokens))


def pkv_paged_attention_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens,
                                             prefix_groups, G, S, H, D, bs, NB, MB,
                                             max_context_len, scale, dtype, partition_tokens,
                                             workspace, workspace_bytes, stream=None) -> None:
    check(lib().pkv_paged_attention_decode_shared_prefix(
        ptr(out), ptr(q), ptr(k_cache), ptr(v_cache), ptr(block_tables), ptr(context_lens),
        ptr(prefix_groups), G, S, H, D, bs, NB, MB, max_context_len, float(scale), int(dtype),
        partition_tokens, ptr(workspace), int(workspace_bytes), stream_handle(stream)),
        "paged_attention_decode_shared_prefix")


def pkv_paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, S, H,
                                       D, bs, NB, MB, max_context_len, scale, dtype,
                                       partition_tokens, stream=None) -> None:
    """Decode attention with the library's built-in scratch array instead of
    a caller workspace, for callers that may not allocate device memory."""
    check(lib().pkv_paged_attention_decode_noalloc(
        ptr(out), ptr(q), ptr(k_cache), ptr(v_cache), ptr(block_tables), ptr(context_lens), S, H,
        D, bs, NB, MB, max_context_len, float(scale), int(dtype), partition_tokens,
        stream_handle(stream)), "paged_attention_decode_noalloc")


def pkv_compute_slot_mapping(slot_mapping, block_tables, seq_idx, pos, T, S, MB, bs,
                             stream=None) -> None:
    check(lib().pkv_compute_slot_mapping(ptr(slot_mapping), ptr(block_tables), ptr(seq_idx),
                                         ptr(pos), T, S, MB, bs, stream_handle(stream)),
          "compute_slot_mapping")


def pkv_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, T, H, D, bs, NB, dtype,
                          stream=None) -> None:
    check(lib().pkv_reshape_and_cache(ptr(key), ptr(value), ptr(k_cache), ptr(v_cache),
                                      ptr(slot_mapping), T, H, D, bs, NB, int(dtype),
                                      stream_handle(stream)), "reshape_and_cache")


def pkv_copy_blocks(k_cache, v_cache, block_mapping, P, H, D, bs, NB, dtype, stream=None) -> None:
    check(lib().pkv_copy_blocks(ptr(k_cache), ptr(v_cache), ptr(block_mapping), P, H, D, bs, NB,
                                int(dtype), stream_handle(stream)), "copy_blocks")


def pkv_swap_blocks(gpu_k, gpu_v, host_k, host_v, block_mapping, P, H, D, bs, NB_gpu, NB_host,
                    dtype, direction, stream=None) -> None:
    check(lib().pkv_swap_blocks(ptr(gpu_k), ptr(gpu_v), ptr(host_k), ptr(host_v),
                                ptr(block_mapping), P, H, D, bs, NB_gpu, NB_host, int(dtype),
                                int(direction), stream_handle(stream)), "swap_blocks")


def pkv_sync_check(stream=None) -> None:
    check(lib().pkv_sync_check(stream_handle(stream)), "sync_check")


def pkv_get_device_errors() -> int:
    v = ctypes.c_int32(0)
    check(lib().pkv_get_device_errors(ctypes.addressof(v)), "get_device_errors")
    return int(v.value)


def pkv_beam_inputs_bytes(S: int, MB: int) -> int:
    return int(lib().pkv_beam_inputs_bytes(S, MB))


def pkv_beam_step(alloc_handle, tables, num_blocks, context_lens, parents, S, MB, staging,
                  dev_inputs, inputs_bytes, out, q, key, value, k_cache, v_cache, slot_mapping,
                  prefix_groups, G, H, D, bs, NB, scale, dtype, partition_tokens, workspace,
                  workspace_bytes, stream=None) -> int:
    """One beam-search step (fork, append, upload, copy_blocks, decode step);
    returns the number of copy pairs."""
    n = ctypes.c_int32(0)
    check(lib().pkv_beam_step(
        alloc_handle, ptr(tables), ptr(num_blocks), ptr(context_lens), ptr(parents), S, MB,
        ptr(staging), ptr(dev_inputs), inputs_bytes, ptr(out), ptr(q), ptr(key), ptr(value),
        ptr(k_cache), ptr(v_cache), ptr(slot_mapping), ptr(prefix_groups), G, H, D, bs, NB,
        float(scale), int(dtype), partition_tokens, ptr(workspace), workspace_bytes,
        ctypes.addressof(n), stream_handle(stream)), "beam_step")
    return int(n.value)


class BeamSearch:
    """pkv_beam_search_create / _step / _destroy: a beam search whose fixed
    arguments live on the native side, so a step is one short call.  The
    caller keeps every buffer passed here alive as long as this object."""

    def __init__(self, alloc_handle, tables, num_blocks, context_lens, S, MB, staging0, staging1,
                 dev_inputs, inputs_bytes, out, k_cache, v_cache, slot_mapping, prefix_groups, G,
                 H, D, bs, NB, scale, dtype, partition_tokens, workspace, workspace_bytes):
        h = ctypes.c_void_p()
        check(lib().pkv_beam_search_create(
            alloc_handle, ptr(tables), ptr(num_blocks), ptr(context_lens), S, MB, ptr(staging0),
            ptr(staging1), ptr(dev_inputs), int(inputs_bytes), ptr(out), ptr(k_cache),
            ptr(v_cache), ptr(slot_mapping), ptr(prefix_groups), G, H, D, bs, NB, float(scale),
            int(dtype), partition_tokens, ptr(workspace), int(workspace_bytes),
            ctypes.addressof(h)), "beam_search_create")
        self._h = h
        self._n = ctypes.c_int32(0)
        self._pairs = ctypes.c_void_p()  # receives the int64 pairs pointer
        self._n_addr = ctypes.addressof(self._n)
        self._pairs_addr = ctypes.addressof(self._pairs)
        self._step = lib().pkv_beam_search_step

    def step(self, parents_addr: int, q_addr: int, key_addr: int, value_addr: int,
             stream: int):
        """One step (addresses as ints, stream as a handle); returns (number
        of copy pairs, address of the first pair)."""
        st = self._step(self._h, parents_addr, q_addr, key_addr, value_addr, stream, self._n_addr,
                        self._pairs_addr)
        if st != PKV_OK:
            check(st, "beam_search_step")
        return self._n.value, self._pairs.value

    def close(self) -> None:
        if self._h:
            lib().pkv_beam_search_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pkv_selftest_bounded_wait(polls: int, stream=None) -> None:
    check(lib().pkv_selftest_bounded_wait(int(polls), stream_handle(stream)),
          "selftest_bounded_wait")
