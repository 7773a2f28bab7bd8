"""Python binding of the C ABI for torch tensors (argument marshalling only).

Every function forwards ``tensor.data_ptr()`` values, sizes and the current
CUDA stream to libpa.so; all computation happens in the library's kernels.
Names and argument order follow include/pa.h.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import CacheDesc, DecodeOpts, PA_KV_BF16, PA_KV_FP8_E4M3

_FP8_DTYPES = (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None, contiguous=True) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    """Descriptor of a [num_blocks, block_size, num_kv_heads, head_dim] cache."""
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, block_size, num_kv_heads, head_dim]")
    if k_cache.dtype == torch.bfloat16:
        dt = PA_KV_BF16
    elif k_cache.dtype in _FP8_DTYPES:
        dt = PA_KV_FP8_E4M3
    else:
        raise ValueError(f"cache dtype must be bfloat16 or float8_e4m3fn/uint8, got {k_cache.dtype}")
    nb, bs, hkv, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d, dt)


def _scales(desc: CacheDesc, k_scale, v_scale):
    if desc.dtype == PA_KV_BF16:
        if k_scale is not None or v_scale is not None:
            raise ValueError("k_scale/v_scale are only for fp8 caches")
        return None, None
    if k_scale is None or v_scale is None:
        raise ValueError("fp8 caches need k_scale and v_scale (device float32 scalars)")
    return (_dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32))


def _same_cache(k_cache, v_cache):
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must have the same shape and dtype")


def _check_meta(desc, q, block_tables, lens, num_seqs, lens_name="context_lens"):
    """Sizes the library cannot check through its raw pointers: one table row
    and one length per sequence, q's head_dim equal to the cache's."""
    if block_tables.dim() != 2 or block_tables.shape[0] != num_seqs:
        raise ValueError(f"block_tables must be [{num_seqs}, max_blocks_per_seq], "
                         f"got {list(block_tables.shape)}")
    if lens.numel() != num_seqs:
        raise ValueError(f"{lens_name} needs {num_seqs} entries, got {lens.numel()}")
    if q.shape[-1] != desc.head_dim:
        raise ValueError(f"q's head_dim {q.shape[-1]} differs from the cache's {desc.head_dim}")


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, k_scale=None,
                      v_scale=None, stream=None) -> None:
    """Write key/value [N, H_kv, d] (bf16) into the caches at ``slot_mapping``."""
    _same_cache(k_cache, v_cache)
    desc = cache_desc(k_cache)
    ks, vs = _scales(desc, k_scale, v_scale)
    n = int(slot_mapping.numel())
    want = (n, desc.num_kv_heads, desc.head_dim)
    if tuple(key.shape) != want or tuple(value.shape) != want:
        raise ValueError(f"key and value must be {list(want)} (one row per slot), "
                         f"got {list(key.shape)} and {list(value.shape)}")
    _lib.check(_lib.lib().pa_reshape_and_cache(
        _dev(key, "key", torch.bfloat16), _dev(value, "value", torch.bfloat16),
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), desc,
        _dev(slot_mapping, "slot_mapping", torch.int32), n, ks, vs, _stream(stream)))


def decode_workspace_size(num_seqs: int, num_heads: int, head_dim: int,
                          max_blocks_per_seq: int, block_size: int,
                          partition_tokens: int = 0) -> int:
    return int(_lib.lib().pa_decode_workspace_size_ex(
        num_seqs, num_heads, head_dim, max_blocks_per_seq, block_size, partition_tokens))


def alloc_workspace(num_seqs, num_heads, head_dim, max_blocks_per_seq, block_size,
                    partition_tokens=0, device=None) -> torch.Tensor:
    """A caller-owned device workspace for ``decode`` (torch allocates it)."""
    n = decode_workspace_size(num_seqs, num_heads, head_dim, max_blocks_per_seq, block_size,
                              partition_tokens)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device or "cuda")


def decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, k_scale=None,
           v_scale=None, workspace=None, partition_tokens=0, kernel=0, stream=None):
    """Paged decode attention; writes ``out`` [B_s, H_q, d] bf16 and returns it."""
    _same_cache(k_cache, v_cache)
    desc = cache_desc(k_cache)
    ks, vs = _scales(desc, k_scale, v_scale)
    if q.dim() != 3 or out.shape != q.shape:
        raise ValueError("q and out must both be [num_seqs, num_heads, head_dim]")
    num_seqs, num_heads, _ = q.shape
    _check_meta(desc, q, block_tables, context_lens, num_seqs)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    opts = DecodeOpts(int(partition_tokens), int(kernel))
    _lib.check(_lib.lib().pa_decode_ex(
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), desc, _dev(block_tables, "block_tables", torch.int32),
        int(block_tables.shape[1]), _dev(context_lens, "context_lens", torch.int32), num_seqs,
        num_heads, ctypes.c_float(scale), ks, vs, ws_ptr, ws_bytes, ctypes.byref(opts),
        _stream(stream)))
    return out


def copy_blocks(k_cache, v_cache, block_pairs, stream=None) -> None:
    """cache[dst] = cache[src] for each (src, dst) row of ``block_pairs`` [n, 2] int32."""
    _same_cache(k_cache, v_cache)
    desc = cache_desc(k_cache)
    n = int(block_pairs.shape[0]) if block_pairs.dim() == 2 else int(block_pairs.numel()) // 2
    ptr = _dev(block_pairs, "block_pairs", torch.int32) if n > 0 else None
    _lib.check(_lib.lib().pa_copy_blocks(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                         desc, ptr, n, _stream(stream)))


def _any_ptr(t: torch.Tensor, name: str) -> int:
    """Pointer of a contiguous CUDA tensor or pinned host tensor."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def varlen_workspace_size(num_tokens: int, num_heads: int, head_dim: int,
                          max_blocks_per_seq: int, block_size: int) -> int:
    return int(_lib.lib().pa_varlen_workspace_size(num_tokens, num_heads, head_dim,
                                                   max_blocks_per_seq, block_size))


def varlen_attention(out, q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale,
                     k_scale=None, v_scale=None, workspace=None, stream=None, method=0):
    """Causal paged attention for a step whose requests add several tokens:
    q/out [num_tokens, H_q, d] (request i's tokens at query_start_loc[i] ..
    query_start_loc[i+1]-1, the last tokens of its seq_lens[i]-token context).
    method: 0 automatic, 1 one decode per new token, 2 tensor-core prefill
    tiles (pa_varlen_attention_ex)."""
    _same_cache(k_cache, v_cache)
    desc = cache_desc(k_cache)
    ks, vs = _scales(desc, k_scale, v_scale)
    if q.dim() != 3 or out.shape != q.shape:
        raise ValueError("q and out must both be [num_tokens, num_heads, head_dim]")
    num_tokens, num_heads, head_dim = q.shape
    num_seqs = int(seq_lens.numel())
    if query_start_loc.numel() != num_seqs + 1:
        raise ValueError("query_start_loc needs num_seqs + 1 entries")
    _check_meta(desc, q, block_tables, seq_lens, num_seqs, "seq_lens")
    max_blocks = int(block_tables.shape[1])
    if workspace is None:
        n = varlen_workspace_size(num_tokens, num_heads, head_dim, max_blocks, desc.block_size)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    _lib.check(_lib.lib().pa_varlen_attention_ex(
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), desc, _dev(block_tables, "block_tables", torch.int32),
        max_blocks, _dev(seq_lens, "seq_lens", torch.int32),
        _dev(query_start_loc, "query_start_loc", torch.int32), num_seqs, int(num_tokens),
        int(num_heads), ctypes.c_float(scale), ks, vs, int(method), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def decode_multi_workspace_size(num_seqs, tokens_per_seq, num_heads, head_dim,
                                max_blocks_per_seq, block_size) -> int:
    return int(_lib.lib().pa_decode_multi_workspace_size(num_seqs, tokens_per_seq, num_heads,
                                                         head_dim, max_blocks_per_seq,
                                                         block_size))


def decode_multi(out, q, k_cache, v_cache, block_tables, context_lens, tokens_per_seq, scale,
                 k_scale=None, v_scale=None, workspace=None, stream=None):
    """Causal attention for ``tokens_per_seq`` new tokens of every sequence:
    q/out [num_seqs * tokens_per_seq, H_q, d], sequence i's tokens at rows
    i * tokens_per_seq + j (the last positions of its context)."""
    _same_cache(k_cache, v_cache)
    desc = cache_desc(k_cache)
    ks, vs = _scales(desc, k_scale, v_scale)
    num_seqs = int(context_lens.numel())
    if q.dim() != 3 or out.shape != q.shape or q.shape[0] != num_seqs * tokens_per_seq:
        raise ValueError("q and out must be [num_seqs * tokens_per_seq, num_heads, head_dim]")
    _, num_heads, head_dim = q.shape
    _check_meta(desc, q, block_tables, context_lens, num_seqs)
    max_blocks = int(block_tables.shape[1])
    if workspace is None:
        n = decode_multi_workspace_size(num_seqs, tokens_per_seq, num_heads, head_dim,
                                        max_blocks, desc.block_size)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    _lib.check(_lib.lib().pa_decode_multi(
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), desc, _dev(block_tables, "block_tables", torch.int32),
        max_blocks, _dev(context_lens, "context_lens", torch.int32), num_seqs,
        int(tokens_per_seq), int(num_heads), ctypes.c_float(scale), ks, vs,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out


def decode_shared_prefix_workspace_size(num_seqs, group_size, num_heads, head_dim,
                                        max_blocks_per_seq, block_size) -> int:
    return int(_lib.lib().pa_decode_shared_prefix_workspace_size(
        num_seqs, group_size, num_heads, head_dim, max_blocks_per_seq, block_size))


def decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens, group_size,
                         scale, k_scale=None, v_scale=None, workspace=None, stream=None):
    """``decode`` for consecutive groups of ``group_size`` sequences forked
    from a common prefix: the shared blocks are read once per group."""
    _same_cache(k_cache, v_cache)
    desc = cache_desc(k_cache)
    ks, vs = _scales(desc, k_scale, v_scale)
    if q.dim() != 3 or out.shape != q.shape:
        raise ValueError("q and out must both be [num_seqs, num_heads, head_dim]")
    num_seqs, num_heads, head_dim = q.shape
    _check_meta(desc, q, block_tables, context_lens, num_seqs)
    max_blocks = int(block_tables.shape[1])
    if workspace is None:
        n = max(decode_shared_prefix_workspace_size(num_seqs, group_size, num_heads, head_dim,
                                                    max_blocks, desc.block_size),
                decode_workspace_size(num_seqs, num_heads, head_dim, max_blocks,
                                      desc.block_size))
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    _lib.check(_lib.lib().pa_decode_shared_prefix(
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), desc, _dev(block_tables, "block_tables", torch.int32),
        max_blocks, _dev(context_lens, "context_lens", torch.int32), num_seqs, int(group_size),
        num_heads, ctypes.c_float(scale), ks, vs, _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def swap_blocks(dst_k, dst_v, src_k, src_v, block_pairs, stream=None) -> None:
    """dst[d] = src[s] for each (s, d) row of ``block_pairs`` [n, 2] int32,
    between two caches of the same block shape (device pool <-> pinned host
    swap space, either direction)."""
    for a, b in ((dst_k, dst_v), (src_k, src_v), (dst_k, src_k)):
        if a.shape[1:] != b.shape[1:] or a.dtype != b.dtype:
            raise ValueError("caches must share block shape and dtype")
    if dst_k.shape != dst_v.shape or src_k.shape != src_v.shape:
        raise ValueError("K and V caches of a side must have the same shape")
    shape = cache_desc(dst_k)
    n = int(block_pairs.shape[0]) if block_pairs.dim() == 2 else int(block_pairs.numel()) // 2
    if n == 0:
        return
    if block_pairs.dtype != torch.int32:
        raise ValueError("block_pairs must be int32")
    _lib.check(_lib.lib().pa_swap_blocks(
        _any_ptr(dst_k, "dst_k"), _any_ptr(dst_v, "dst_v"), int(dst_k.shape[0]),
        _any_ptr(src_k, "src_k"), _any_ptr(src_v, "src_v"), int(src_k.shape[0]), shape,
        _any_ptr(block_pairs, "block_pairs"), n, _stream(stream)))


def step_prepare(block_tables, context_lens, block_size, slot_mapping, updates=None,
                 advance=0, stream=None) -> None:
    """Device-side step metadata: apply ``updates`` ([n, 3] int32 rows of
    (sequence, logical block, physical block)) to ``block_tables``, add
    ``advance`` to every context length, and write each sequence's newest
    token slot into ``slot_mapping`` (-1 where there is none)."""
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    num_seqs, max_blocks = block_tables.shape
    if context_lens.numel() != num_seqs or slot_mapping.numel() != num_seqs:
        raise ValueError("context_lens and slot_mapping need one entry per sequence")
    n_up, up_ptr = 0, None
    if updates is not None and updates.numel() > 0:
        if updates.dim() != 2 or updates.shape[1] != 3:
            raise ValueError("updates must be [n, 3] (sequence, logical block, physical block)")
        n_up, up_ptr = int(updates.shape[0]), _dev(updates, "updates", torch.int32)
    _lib.check(_lib.lib().pa_step_prepare(
        _dev(block_tables, "block_tables", torch.int32), int(num_seqs), int(max_blocks),
        int(block_size), _dev(context_lens, "context_lens", torch.int32), up_ptr, n_up,
        int(advance), _dev(slot_mapping, "slot_mapping", torch.int32), _stream(stream)))


def write_and_decode(key, value, slot_mapping, out, q, k_cache, v_cache, block_tables,
                     context_lens, scale, k_scale=None, v_scale=None, workspace=None,
                     stream=None):
    """One decode step: cache write of the new tokens, then paged decode."""
    _same_cache(k_cache, v_cache)
    desc = cache_desc(k_cache)
    ks, vs = _scales(desc, k_scale, v_scale)
    if q.dim() != 3 or out.shape != q.shape:
        raise ValueError("q and out must both be [num_seqs, num_heads, head_dim]")
    num_seqs, num_heads, _ = q.shape
    _check_meta(desc, q, block_tables, context_lens, num_seqs)
    want = (int(slot_mapping.numel()), desc.num_kv_heads, desc.head_dim)
    if tuple(key.shape) != want or tuple(value.shape) != want:
        raise ValueError(f"key and value must be {list(want)} (one row per slot), "
                         f"got {list(key.shape)} and {list(value.shape)}")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    _lib.check(_lib.lib().pa_write_and_decode(
        _dev(key, "key", torch.bfloat16), _dev(value, "value", torch.bfloat16),
        _dev(slot_mapping, "slot_mapping", torch.int32), int(slot_mapping.numel()),
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), desc, _dev(block_tables, "block_tables", torch.int32),
        int(block_tables.shape[1]), _dev(context_lens, "context_lens", torch.int32), num_seqs,
        num_heads, ctypes.c_float(scale), ks, vs, ws_ptr, ws_bytes, _stream(stream)))
    return out


class StepGraph:
    """One decode step captured once as a CUDA graph over fixed buffers.

    The graph holds, in stream order: the host-to-device copies in ``h2d``
    (pairs ``(device_tensor, pinned_host_tensor)``), ``write_and_decode`` on
    the given tensors (cache write of the new tokens, then paged decode), and
    the device-to-host copies in ``d2h`` (pairs ``(pinned_host_tensor,
    device_tensor)``).  ``replay()`` re-runs all of it on whatever the buffers
    hold, for about one host call's cost; shapes and pointers are fixed at
    capture.  The pages call the per-step host-to-device staging of step
    metadata critical-path work ("4.6 PagedAttention & KV-Cache Memory
    Management", section "From Python bookkeeping to GPU tensors"); a
    captured step issues it with the kernels in one submission.

    The decode kernel's merge counters carry a per-launch tag and are left
    at count zero by every completed launch, so replaying the same captured
    launch is safe; after a launch that reported an error in workspace word 0
    the workspace must be re-zeroed before the next replay."""

    def __init__(self, key, value, slot_mapping, out, q, k_cache, v_cache, block_tables,
                 context_lens, scale, k_scale=None, v_scale=None, workspace=None, h2d=(),
                 d2h=(), device_slots=False):
        self._h2d = list(h2d)
        self._d2h = list(d2h)
        for dev_t, host_t in self._h2d:
            _dev(dev_t, "h2d destination")
            if host_t.is_cuda or not host_t.is_pinned():
                raise ValueError("h2d sources must be pinned host tensors")
        for host_t, dev_t in self._d2h:
            _dev(dev_t, "d2h source")
            if host_t.is_cuda or not host_t.is_pinned():
                raise ValueError("d2h destinations must be pinned host tensors")
        self._args = (key, value, slot_mapping, out, q, k_cache, v_cache, block_tables,
                      context_lens, scale, k_scale, v_scale, workspace)
        # device_slots: the slots of the new tokens are computed in the graph
        # from the tables and lengths (pa_step_prepare) instead of being copied in
        self._device_slots = bool(device_slots)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._body()  # eager run: per-kernel attributes are set before capture
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._body()

    def _body(self):
        for dev_t, host_t in self._h2d:
            dev_t.copy_(host_t, non_blocking=True)
        if self._device_slots:
            key, value, slots, out, q, kc, vc, bt, cl = self._args[:9]
            step_prepare(bt, cl, kc.shape[1], slots)
        write_and_decode(*self._args)
        for host_t, dev_t in self._d2h:
            host_t.copy_(dev_t, non_blocking=True)

    def replay(self):
        """Run the captured step on the current stream (asynchronous)."""
        self.graph.replay()
