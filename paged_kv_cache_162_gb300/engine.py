"""Tensor-level calls and one decode step over a paged KV cache.

PyTorch supplies device memory and streams only; every step of the path
runs in libpagedkv.so through the C ABI (see _lib.py).

The step, in the order a serving loop runs it ("3.3 页面级显存管理" 3.3.2;
"vLLM三大核心技术分页内存与共享解码", Copy-on-Write section):
  host   make room for each sequence's new tokens (copy-on-write of shared
         blocks, new blocks as the token count grows) -- `plan_step`
  device copy_blocks -> compute_slot_mapping -> reshape_and_cache ->
         paged_attention_decode
"""
from __future__ import annotations

import ctypes
import math
import time

import numpy as np
import torch

from . import _lib as L
from .allocator import BlockAllocator, plan_step

_DTYPES = {torch.float16: L.PKV_F16, torch.bfloat16: L.PKV_BF16}
_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}


def dtype_code(t: torch.dtype) -> int:
    if t not in _DTYPES:
        raise L.PkvError(L.PKV_ERR_UNSUPPORTED, f"dtype {t} (fp16 and bf16 only)")
    return _DTYPES[t]


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH[name]


def workspace_size(S, H, D, max_context_len, partition_tokens=0) -> int:
    return L.pkv_decode_workspace_size(S, H, D, max_context_len, partition_tokens)


def new_workspace(S, H, D, max_context_len, partition_tokens=0, device="cuda") -> torch.Tensor:
    n = workspace_size(S, H, D, max_context_len, partition_tokens)
    if n == 0:
        raise L.PkvError(L.PKV_ERR_INVALID_ARG, "bad workspace arguments")
    return torch.empty(n, dtype=torch.uint8, device=device)


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale=None,
                           max_context_len=0, partition_tokens=0, workspace=None, stream=None):
    """out[s,h] = softmax(scale q[s,h] K^T) V over each sequence's paged context.

    q, out: [S, H, D]; caches: [NB, bs, H, D]; block_tables [S, MB] int32;
    context_lens [S] int32 (all on the device).
    """
    S, H, D = q.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    MB = block_tables.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if workspace is None:
        workspace = new_workspace(S, H, D, max_context_len or MB * bs, partition_tokens,
                                  q.device)
    L.pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, S, H, D, bs,
                                 NB, MB, max_context_len, scale, dtype_code(q.dtype),
                                 partition_tokens, workspace, workspace.numel(), stream)
    return out


def decode_step(out, q, key, value, k_cache, v_cache, block_tables, context_lens, seq_idx, pos,
                slot_mapping, prefix_groups=None, scale=None, max_context_len=0,
                partition_tokens=0, workspace=None, stream=None):
    """compute_slot_mapping + reshape_and_cache + paged_attention_decode (or
    its shared-prefix form, with prefix_groups [G, 3] int32 on the device) in
    fewer kernels (see pkv_decode_step): the new tokens (key/value [T, H, D],
    seq_idx/pos [T] int32) are written into the caches, slot_mapping [T]
    int64 receives their slots, then out = attention over every context."""
    S, H, D = q.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    MB = block_tables.shape[1]
    T = int(seq_idx.numel())
    G = 0 if prefix_groups is None else int(prefix_groups.shape[0])
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if workspace is None:
        mc = max_context_len or MB * bs
        n = (L.pkv_decode_shared_prefix_workspace_size(S, H, D, G, mc, partition_tokens) if G
             else workspace_size(S, H, D, mc, partition_tokens))
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    L.pkv_decode_step(out, q, key, value, k_cache, v_cache, block_tables, context_lens, seq_idx,
                      pos, slot_mapping, prefix_groups, G, T, S, H, D, bs, NB, MB,
                      max_context_len, scale, dtype_code(q.dtype), partition_tokens, workspace,
                      workspace.numel(), stream)
    return out


def paged_attention_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens,
                                         prefix_groups, scale=None, max_context_len=0,
                                         partition_tokens=0, workspace=None, stream=None):
    """paged_attention_decode where groups of sequences share a prefix
    (prefix_groups [G, 3] int32 on the device: first sequence, members,
    prefix tokens); the prefix is read once per group (tensor cores)."""
    S, H, D = q.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    MB = block_tables.shape[1]
    G = prefix_groups.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if workspace is None:
        mcl = max_context_len or MB * bs
        need = L.pkv_decode_shared_prefix_workspace_size(S, H, D, G, mcl, partition_tokens)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    L.pkv_paged_attention_decode_shared_prefix(out, q, k_cache, v_cache, block_tables,
                                               context_lens, prefix_groups, G, S, H, D, bs, NB, MB,
                                               max_context_len, scale, dtype_code(q.dtype),
                                               partition_tokens, workspace, workspace.numel(),
                                               stream)
    return out


def compute_slot_mapping(slot_mapping, block_tables, seq_idx, pos, block_size, stream=None):
    L.pkv_compute_slot_mapping(slot_mapping, block_tables, seq_idx, pos, seq_idx.numel(),
                               block_tables.shape[0], block_tables.shape[1], block_size, stream)
    return slot_mapping


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, stream=None):
    T, H, D = key.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    L.pkv_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, T, H, D, bs, NB,
                            dtype_code(key.dtype), stream)


def copy_blocks(k_cache, v_cache, block_mapping, stream=None):
    NB, bs, H, D = k_cache.shape
    P = block_mapping.shape[0] if block_mapping is not None else 0
    L.pkv_copy_blocks(k_cache, v_cache, block_mapping, P, H, D, bs, NB,
                      dtype_code(k_cache.dtype), stream)


def swap_blocks(gpu_k, gpu_v, host_k, host_v, block_mapping, direction, stream=None):
    """GPU <-> pinned-host block copies (CPU swap).  block_mapping [P, 2]
    int64 on the device: (gpu block, host block) pairs for swap-out,
    (host block, gpu block) pairs for swap-in."""
    NBg, bs, H, D = gpu_k.shape
    P = block_mapping.shape[0]
    L.pkv_swap_blocks(gpu_k, gpu_v, host_k, host_v, block_mapping, P, H, D, bs, NBg,
                      host_k.shape[0], dtype_code(gpu_k.dtype), direction, stream)


class DecodeStep:
    """Device-resident state of one decode step and the calls that run it.

    Built from plain arrays (16-bit data as uint16 bit patterns):
      caches: pool [NB, bs, H, D]; `blocks` lists the physical blocks whose
              contents `k_blocks`/`v_blocks` give, every other slot is set
              to `fill_bits`;
      tables_pre/nblocks_pre/ctx_before: the sequences before the step;
      n_new, new_k/new_v [T, H, D], seq_idx/pos [T]: the tokens appended;
      initial_free: the free list (last element handed out first).
    `plan()` runs the host allocator; `run()` launches copy_blocks, slot
    mapping, reshape_and_cache and decode on `stream` (`run(fused=True)`:
    copy_blocks and pkv_decode_step).
    """

    def __init__(self, *, dtype: str, S, H, D, bs, NB, MB, scale, ctx_before, n_new, tables_pre,
                 nblocks_pre, initial_free, blocks, k_blocks, v_blocks, q, new_k, new_v, seq_idx,
                 pos, fill_bits: int, partition_tokens: int = 0, device="cuda"):
        self.dtype = torch_dtype(dtype)
        self.S, self.H, self.D, self.bs, self.NB, self.MB = S, H, D, bs, NB, MB
        self.scale = float(scale)
        self.partition_tokens = partition_tokens
        self.device = torch.device(device)
        self.ctx_before = np.asarray(ctx_before, dtype=np.int32)
        self.n_new = np.asarray(n_new, dtype=np.int32)
        self.context_lens_host = (self.ctx_before + self.n_new).astype(np.int32)
        self.tables_pre = np.asarray(tables_pre, dtype=np.int32)
        self.nblocks_pre = np.asarray(nblocks_pre, dtype=np.int32)
        self.initial_free = np.asarray(initial_free, dtype=np.int32)
        self.max_context_len = max(int(self.context_lens_host.max(initial=0)), 1)
        dev = self.device

        def up16(a):
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
            return t.to(dev).view(self.dtype)

        self.k_cache = torch.empty((NB, bs, H, D), dtype=torch.int16, device=dev)
        self.v_cache = torch.empty((NB, bs, H, D), dtype=torch.int16, device=dev)
        fill = int(np.int16(np.uint16(fill_bits)))
        self.k_cache.fill_(fill)
        self.v_cache.fill_(fill)
        if len(blocks):
            idx = torch.from_numpy(np.asarray(blocks, dtype=np.int64)).to(dev)
            for dst, src in ((self.k_cache, k_blocks), (self.v_cache, v_blocks)):
                chunk = 2048
                for i in range(0, len(blocks), chunk):
                    part = torch.from_numpy(np.ascontiguousarray(src[i:i + chunk]).view(np.int16))
                    dst.index_copy_(0, idx[i:i + chunk], part.to(dev))
        self.k_cache = self.k_cache.view(self.dtype)
        self.v_cache = self.v_cache.view(self.dtype)
        self.q = up16(q)
        self.new_k = up16(new_k)
        self.new_v = up16(new_v)
        self.seq_idx = torch.from_numpy(np.asarray(seq_idx, dtype=np.int32)).to(dev)
        self.pos = torch.from_numpy(np.asarray(pos, dtype=np.int32)).to(dev)
        self.T = int(self.seq_idx.numel())
        self.context_lens = torch.from_numpy(self.context_lens_host).to(dev)
        self.slot_mapping = torch.empty(max(self.T, 1), dtype=torch.int64, device=dev)
        self.out = torch.empty((S, H, D), dtype=self.dtype, device=dev)
        self.workspace = new_workspace(S, H, D, self.max_context_len, partition_tokens, dev)
        self.block_tables = None
        self.pairs = None
        # shared-prefix groups [G, 3] int32 on the device for run(fused=True)
        # (the workspace must then have the shared-prefix size)
        self.prefix_groups = None

    def plan(self):
        """Host allocator: tables and copy-on-write pairs for this step.
        A new plan also starts a new beam search (beam_step)."""
        for name in ("beam_ctx", "_beam_native"):
            old = self.__dict__.pop(name, None)
            if name == "_beam_native" and old is not None:
                torch.cuda.synchronize(self.device)  # its staging buffers may still be in flight
                old.close()
        self.allocator = BlockAllocator(self.NB, self.initial_free)
        ids, counts = np.unique(self.tables_pre[self.tables_pre >= 0], return_counts=True)
        for b, c in zip(ids.tolist(), counts.tolist()):
            if c > 1:
                self.allocator.incref([b] * (c - 1))
        tables, nb, pairs = plan_step(self.allocator, self.tables_pre, self.nblocks_pre,
                                      self.ctx_before, self.n_new, self.bs)
        self.tables_host, self.nblocks_host, self.pairs_host = tables, nb, pairs
        self.block_tables = torch.from_numpy(tables).to(self.device)
        self.pairs = torch.from_numpy(np.ascontiguousarray(pairs)).to(self.device)
        return tables, nb, pairs

    def run(self, stream=None, attention=True, write=True, fused=False):
        """The device part of the step: copy_blocks, slot mapping, cache
        write, decode.  fused=True runs the last three as pkv_decode_step
        (fewer kernels, the same results), with the shared-prefix decode
        when self.prefix_groups is set."""
        if self.block_tables is None:
            self.plan()
        if fused and write and attention:
            if self.pairs.shape[0]:
                copy_blocks(self.k_cache, self.v_cache, self.pairs, stream)
            g = self.prefix_groups
            L.pkv_decode_step(self.out, self.q, self.new_k, self.new_v, self.k_cache, self.v_cache,
                              self.block_tables, self.context_lens, self.seq_idx, self.pos,
                              self.slot_mapping, g, 0 if g is None else int(g.shape[0]), self.T,
                              self.S, self.H, self.D, self.bs, self.NB, self.MB,
                              self.max_context_len, self.scale, dtype_code(self.dtype),
                              self.partition_tokens, self.workspace, self.workspace.numel(),
                              stream)
            return self.out
        if write:
            if self.pairs.shape[0]:
                copy_blocks(self.k_cache, self.v_cache, self.pairs, stream)
            if self.T:
                compute_slot_mapping(self.slot_mapping, self.block_tables, self.seq_idx, self.pos,
                                     self.bs, stream)
                reshape_and_cache(self.new_k, self.new_v, self.k_cache, self.v_cache,
                                  self.slot_mapping, stream)
        if attention:
            self.decode(stream)
        return self.out

    def _beam_buffers(self):
        """Buffers of the native beam step: two pinned staging buffers used
        in turn (an event per buffer keeps one from being rewritten while
        its upload may still be in flight), the device twin they upload to,
        a device buffer for host-given tokens, and a workspace sized for
        the longest context the tables allow."""
        S, MB, H, D = self.S, self.MB, self.H, self.D
        dev = self.device
        nb = L.pkv_beam_inputs_bytes(S, MB)
        self._beam_inputs_bytes = nb
        self._beam_slots = []
        for _ in range(2):
            raw = torch.empty(nb + 256, dtype=torch.uint8).pin_memory()
            off = (-raw.data_ptr()) % 256
            stg = raw[off:off + nb]
            self._beam_slots.append({"stg": stg, "stg_np": stg.numpy(),
                                     "u16": torch.empty(3 * S * H * D, dtype=torch.int16).pin_memory(),
                                     "done": torch.cuda.Event(), "used": False})
        self._beam_dev_inputs = torch.empty(nb, dtype=torch.uint8, device=dev)
        self._beam_dev_u16 = torch.empty(3 * S * H * D, dtype=torch.int16, device=dev)
        self._beam_turn = 0
        # prefix groups ([G, 3]: first sequence, members, prefix tokens) set
        # before the first beam_step as `beam_groups`: the beams of a
        # request keep their prompt's full blocks shared, so each group's
        # prefix is read once per step
        groups = getattr(self, "beam_groups", None)
        if groups is not None and len(groups):
            g = np.ascontiguousarray(groups, dtype=np.int32).reshape(-1, 3)
            self._beam_groups_dev = torch.from_numpy(g).to(dev)
            self._beam_G = int(g.shape[0])
            nws = L.pkv_decode_shared_prefix_workspace_size(S, H, D, self._beam_G, MB * self.bs,
                                                            self.partition_tokens)
            self._beam_ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        else:
            self._beam_groups_dev, self._beam_G = None, 0
            self._beam_ws = new_workspace(S, H, D, MB * self.bs, self.partition_tokens, dev)
        # decode() after beam steps: the tables allow contexts up to MB * bs
        self.max_context_len = MB * self.bs
        if self._beam_G == 0:
            self.workspace = self._beam_ws
        else:
            self.workspace = new_workspace(S, H, D, MB * self.bs, self.partition_tokens, dev)
        if self.slot_mapping.numel() < S:
            self.slot_mapping = torch.empty(S, dtype=torch.int64, device=dev)
        # offsets of the staged inputs (the layout pkv_beam_step documents)
        up = lambda x: (x + 255) // 256 * 256
        o_ctx = up(4 * S * MB)
        o_pos = o_ctx + up(4 * S)
        o_seq = o_pos + up(4 * S)
        self._beam_offsets = {"ctx": o_ctx, "pos": o_pos, "seq": o_seq, "pairs": o_seq + up(4 * S)}
        # the step's device inputs, as views of the uploaded buffer
        d = self._beam_dev_inputs
        self._beam_views = (d[:4 * S * MB].view(torch.int32).view(S, MB),
                            d[o_ctx:o_ctx + 4 * S].view(torch.int32),
                            d[o_pos:o_pos + 4 * S].view(torch.int32),
                            d[o_seq:o_seq + 4 * S].view(torch.int32))
        self._beam_stg_base = [sl["stg"].data_ptr() for sl in self._beam_slots]
        # the native side of the search: every argument of pkv_beam_step
        # that stays the same, and the alternation of the staging buffers
        self._beam_native = L.BeamSearch(
            self.allocator._h, self.tables_host, self.nblocks_host, self.beam_ctx, S, MB,
            self._beam_slots[0]["stg"], self._beam_slots[1]["stg"], self._beam_dev_inputs, nb,
            self.out, self.k_cache, self.v_cache, self.slot_mapping, self._beam_groups_dev,
            self._beam_G, self.H, self.D, self.bs, self.NB, self.scale, dtype_code(self.dtype),
            self.partition_tokens, self._beam_ws, self._beam_ws.numel())

    def beam_step(self, parents, new_k, new_v, q, stream=None):
        """One beam-search step after plan(): every sequence b continues from
        sequence parents[b] (fork: share the parent's blocks), appends one
        token (copy-on-write of its shared partial block first), then the
        device copies, writes and attends -- one native call
        (pkv_beam_step).  new_k/new_v/q: [S, H, D] 16-bit values, either
        host arrays of uint16 bit patterns (uploaded first) or device
        tensors (used in place, as a model on the device would produce
        them).  Returns the (src, dst) copy pairs of the step."""
        S, MB, H, D, bs = self.S, self.MB, self.H, self.D, self.bs
        if not hasattr(self, "beam_ctx"):
            self.beam_ctx = np.ascontiguousarray(self.context_lens_host, dtype=np.int32).copy()
            self.nblocks_host = np.ascontiguousarray(self.nblocks_host, dtype=np.int32)
            self.tables_host = np.ascontiguousarray(self.tables_host, dtype=np.int32)
            self._beam_buffers()
        sh = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
        n = S * H * D
        if (isinstance(q, torch.Tensor) and isinstance(new_k, torch.Tensor)
                and isinstance(new_v, torch.Tensor) and q.is_cuda and new_k.is_cuda and new_v.is_cuda):
            for t in (q, new_k, new_v):
                if t.element_size() != 2 or t.numel() != n or not t.is_contiguous():
                    raise L.PkvError(L.PKV_ERR_INVALID_ARG,
                                     "beam_step: q/new_k/new_v must be contiguous [S, H, D] 16-bit")
            tq, tk, tv = q, new_k, new_v
        else:
            # host arrays: through a pinned buffer (two used in turn, each
            # guarded by an event) into the device token buffer
            slot = self._beam_slots[self._beam_turn]
            self._beam_turn ^= 1
            if slot["used"]:
                slot["done"].synchronize()
            u16 = slot["u16"].numpy().view(np.uint16)
            u16[:n] = np.asarray(q).ravel()
            u16[n:2 * n] = np.asarray(new_k).ravel()
            u16[2 * n:] = np.asarray(new_v).ravel()
            st = stream if stream is not None else torch.cuda.current_stream()
            with torch.cuda.stream(st):
                self._beam_dev_u16.copy_(slot["u16"], non_blocking=True)
            slot["done"].record(st)
            slot["used"] = True
            tok = self._beam_dev_u16.view(self.dtype)
            tq, tk, tv = (tok[:n].view(S, H, D), tok[n:2 * n].view(S, H, D),
                          tok[2 * n:].view(S, H, D))
        par = np.ascontiguousarray(parents, dtype=np.int32)
        t0 = time.perf_counter()
        P, at = self._beam_native.step(par.ctypes.data, tq.data_ptr(), tk.data_ptr(), tv.data_ptr(),
                                       sh)
        self.last_native_seconds = time.perf_counter() - t0
        # the pairs sit in the staging buffer the step used
        k = 0 if 0 <= at - self._beam_stg_base[0] < self._beam_inputs_bytes else 1
        o = at - self._beam_stg_base[k]
        pairs = self._beam_slots[k]["stg_np"][o:o + 16 * P].view(np.int64).reshape(P, 2).copy()
        self.pairs_host = pairs
        self.context_lens_host = self.beam_ctx
        self.T = S
        self.q, self.new_k, self.new_v = tq, tk, tv
        (self.block_tables, self.context_lens, self.pos,
         self.seq_idx) = self._beam_views
        return pairs

    def pack_inputs(self, on_host=()):
        """Move the step's inputs (q, new K/V, block tables, context lengths,
        token positions, copy pairs) into one buffer, at 256-byte aligned
        offsets, so that one copy uploads all of them.

        on_host: names among "q", "new_k", "new_v" that stay in the pinned
        host buffer, where the kernels read them directly (a GPU can address
        pinned host memory; on GB300 the reads cross the coherent NVLink-C2C
        link to the Grace CPU's memory).  They come first in the buffers and
        are not part of the upload.

        Returns (device buffer, pinned host buffer holding the same bytes,
        (device view, host view) of the bytes to upload each step).  The
        step's tensors become views of the device buffer (of the host buffer
        for `on_host`); a caller writes the next step's inputs into the host
        buffer at the same offsets (`input_offsets`) and uploads."""
        if self.block_tables is None:
            self.plan()
        tokens = ["q", "new_k", "new_v"]
        if any(n not in tokens for n in on_host):
            raise L.PkvError(L.PKV_ERR_INVALID_ARG, "pack_inputs: on_host takes q, new_k, new_v")
        names = [n for n in tokens if n in on_host] + [n for n in tokens if n not in on_host]
        names += ["block_tables", "context_lens", "seq_idx", "pos"]
        if self.pairs.numel():
            names.append("pairs")
        offsets, o = {}, 0
        for n in names:
            t = getattr(self, n)
            offsets[n] = o
            o = (o + t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(max(o, 256), dtype=torch.uint8, device=self.device)
        views = {}
        for n in names:
            t = getattr(self, n)
            nbytes = t.numel() * t.element_size()
            views[n] = (t, nbytes)
            view = buf[offsets[n]:offsets[n] + nbytes].view(t.dtype).view(t.shape)
            view.copy_(t)
            setattr(self, n, view)
        host = buf.cpu().pin_memory()
        for n in on_host:
            t, nbytes = views[n]
            setattr(self, n, host[offsets[n]:offsets[n] + nbytes].view(t.dtype).view(t.shape))
        self.input_offsets = offsets
        first = offsets[names[len(on_host)]]  # the first uploaded input
        return buf, host, (buf[first:], host[first:])

    def pin_output(self):
        """The step's output goes to a pinned host tensor (returned), which
        becomes `out`: the kernels write it there directly, so no
        device-to-host copy follows the step."""
        host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.out = host
        return host

    def decode_shared_prefix(self, prefix_groups, stream=None):
        """decode() with the prefix of each group read once (see
        paged_attention_decode_shared_prefix); prefix_groups [G, 3] int32."""
        g = torch.as_tensor(np.asarray(prefix_groups, dtype=np.int32)).to(self.device)
        return paged_attention_decode_shared_prefix(
            self.out, self.q, self.k_cache, self.v_cache, self.block_tables, self.context_lens, g,
            self.scale, self.max_context_len, self.partition_tokens, stream=stream)

    def decode(self, stream=None):
        L.pkv_paged_attention_decode(self.out, self.q, self.k_cache, self.v_cache,
                                     self.block_tables, self.context_lens, self.S, self.H, self.D,
                                     self.bs, self.NB, self.MB, self.max_context_len, self.scale,
                                     dtype_code(self.dtype), self.partition_tokens, self.workspace,
                                     self.workspace.numel(), stream)
        return self.out


_driver = None


def _cu_graph_launch():
    """The driver's cuGraphLaunch(graph_exec, stream) -> CUresult."""
    global _driver
    if _driver is None:
        lib = ctypes.CDLL("libcuda.so.1")
        lib.cuGraphLaunch.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.cuGraphLaunch.restype = ctypes.c_int
        _driver = lib
    return _driver.cuGraphLaunch


class StepGraph:
    """One decode step captured in a CUDA graph, optionally with the copies
    of its inputs from pinned host memory and of its output back to it.

    h2d: [(device_tensor, pinned_host_tensor), ...] copied in first;
    d2h: [(pinned_host_tensor, device_tensor), ...] copied out last;
    fused: run the step through pkv_decode_step (DecodeStep.run).
    The step runs once eagerly before capture so that every per-device
    set-up of the library happens outside the capture.  replay() enqueues
    the whole step on the capture stream with one launch.
    """

    def __init__(self, step: DecodeStep, stream: torch.cuda.Stream, h2d=(), d2h=(), fused=False):
        self.step = step
        self.stream = stream
        with torch.cuda.stream(stream):
            step.run(fused=fused)
        stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            for dev, host in h2d:
                dev.copy_(host, non_blocking=True)
            step.run(fused=fused)
            for host, dev in d2h:
                host.copy_(dev, non_blocking=True)
        self._exec = ctypes.c_void_p(self.graph.raw_cuda_graph_exec())
        self._stream = ctypes.c_void_p(stream.cuda_stream)
        self._launch = _cu_graph_launch()

    def replay(self):
        """Enqueue the captured step on its stream (not torch's current one).

        One driver call: switching torch's current stream around
        CUDAGraph.replay() costs more host time per step than the launch."""
        r = self._launch(self._exec, self._stream)
        if r != 0:
            raise L.PkvError(L.PKV_ERR_CUDA, f"cuGraphLaunch failed (CUresult {r})")
