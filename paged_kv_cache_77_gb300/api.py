"""Python binding of libpaged_kv.so: argument marshalling only.

Every call forwards raw pointers, sizes and the current CUDA stream to the C ABI of
include/paged_kv.h; all the work happens in the library's kernels (device calls) or
its C++ host generator. PyTorch supplies device memory and streams. There is no
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from ._lib import check, load

PKV_BF16, PKV_F32 = 0, 1


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _np_ptr(a: np.ndarray):
    return C.c_void_p(a.ctypes.data)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _dev_bf16(t, name):
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")


def _dev_i32(t, name):
    if not (t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")


# ------------------------------------------------------------------ host generator
class BlockPool:
    """Handle on the library's BlockPool (FIFO free queue, first popped id = null block)."""

    def __init__(self, num_blocks: int, initial_order: np.ndarray | None = None):
        lib = load()
        self._h = C.c_void_p()
        order = None
        if initial_order is not None:
            order = np.ascontiguousarray(initial_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("initial_order must have num_blocks entries")
        check(lib.pkv_pool_create(num_blocks, None if order is None else _np_ptr(order),
                                  C.byref(self._h)), "pkv_pool_create")
        self.num_blocks = num_blocks

    def __del__(self):
        if getattr(self, "_h", None):
            load().pkv_pool_destroy(self._h)
            self._h = None

    @property
    def null_block(self) -> int:
        return load().pkv_pool_null_block(self._h)

    def num_free(self) -> int:
        return load().pkv_pool_num_free(self._h)

    def alloc(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.int32)
        check(load().pkv_pool_alloc(self._h, n, _np_ptr(out)), "pkv_pool_alloc")
        return out

    def free(self, ids) -> None:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        check(load().pkv_pool_free(self._h, _np_ptr(ids), len(ids)), "pkv_pool_free")

    def build_block_table(self, seq_lens, block_size: int, window: int,
                          max_blocks_per_seq: int) -> np.ndarray:
        lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        table = np.empty((len(lens), max_blocks_per_seq), dtype=np.int32)
        check(load().pkv_build_block_table(self._h, _np_ptr(lens), len(lens), block_size, window,
                                           max_blocks_per_seq, _np_ptr(table)),
              "pkv_build_block_table")
        return table


def build_block_table_arange(batch: int, blocks_per_seq: int) -> np.ndarray:
    table = np.empty((batch, blocks_per_seq), dtype=np.int32)
    check(load().pkv_build_block_table_arange(batch, blocks_per_seq, _np_ptr(table)),
          "pkv_build_block_table_arange")
    return table


def build_slot_mapping(block_table: np.ndarray, start_pos, num_new, block_size: int) -> np.ndarray:
    table = np.ascontiguousarray(block_table, dtype=np.int32)
    sp = np.ascontiguousarray(start_pos, dtype=np.int32)
    nn = np.ascontiguousarray(num_new, dtype=np.int32)
    cap = int(nn.sum())
    out = np.empty(max(cap, 1), dtype=np.int32)
    n = check(load().pkv_build_slot_mapping(_np_ptr(table), table.shape[1], _np_ptr(sp),
                                            _np_ptr(nn), len(nn), block_size, _np_ptr(out), cap),
              "pkv_build_slot_mapping")
    return out[:n]


def num_skipped_tokens(num_computed_tokens: int, window: int) -> int:
    return load().pkv_num_skipped_tokens(num_computed_tokens, window)


def block_num_fixed(max_concurrency, sliding_window, next_n, block_size) -> int:
    return load().pkv_block_num_fixed(max_concurrency, sliding_window, next_n, block_size)


def block_num_full_offline(max_len, block_size, max_concurrency) -> int:
    return load().pkv_block_num_full_offline(max_len, block_size, max_concurrency)


def block_num_full_online(available_bytes, per_token_bytes, block_size) -> int:
    return load().pkv_block_num_full_online(available_bytes, per_token_bytes, block_size)


# ------------------------------------------------------------------ device calls
def kv_cache_write(k_cache, v_cache, k, v, slot_mapping, dev_status=None, stream=None) -> None:
    """Write rows k[t] (and v[t]) at slot_mapping[t] of the paged caches.

    k_cache [nb, bs, H_kv, d_k]; v_cache [nb, bs, H_kv, d_v] or None (with v None)."""
    _dev_bf16(k_cache, "k_cache")
    _dev_bf16(k, "k")
    _dev_i32(slot_mapping, "slot_mapping")
    if v_cache is not None:
        _dev_bf16(v_cache, "v_cache")
        _dev_bf16(v, "v")
    nb, bs, hkv, dk = k_cache.shape
    dv = v_cache.shape[3] if v_cache is not None else 0
    check(load().pkv_kv_cache_write(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v),
                                    _ptr(slot_mapping), slot_mapping.numel(), nb, bs, hkv, dk, dv,
                                    _ptr(dev_status), _stream(stream)), "pkv_kv_cache_write")


KERNEL_AUTO, KERNEL_CUDA_CORE, KERNEL_TENSOR_CORE = 0, 1, 2


def set_decode_kernel(kernel: int) -> None:
    """Select the decode kernel process-wide (KERNEL_AUTO / _CUDA_CORE / _TENSOR_CORE)."""
    check(load().pkv_set_decode_kernel(kernel), "pkv_set_decode_kernel")


def get_decode_kernel() -> int:
    return load().pkv_get_decode_kernel()


def decode_workspace_size(B: int, H: int, H_kv: int, head_dim: int) -> int:
    return load().pkv_decode_workspace_size(B, H, H_kv, head_dim)


def paged_attention_decode(q, k_cache, v_cache, block_table, seq_lens, scale: float, window: int = 0,
                           out=None, lse=None, out_dtype=torch.float32, workspace=None,
                           dev_status=None, stream=None):
    """Decode attention over the paged cache; returns out [B, H, d] (and fills lse)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev_bf16(t, n)
    _dev_i32(block_table, "block_table")
    _dev_i32(seq_lens, "seq_lens")
    B, H, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((B, H, d), dtype=out_dtype, device=q.device)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    if workspace is None:
        need = decode_workspace_size(B, H, hkv, d)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    check(load().pkv_paged_attention_decode(
        _ptr(out), code, _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, H, hkv, d, bs, nb, float(scale), int(window),
        _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream)),
        "pkv_paged_attention_decode")
    return out


def prefill_workspace_size() -> int:
    return load().pkv_prefill_workspace_size()


def paged_attention_prefill(q, cu_seqlens_q, k_cache, v_cache, block_table, seq_lens_kv,
                            scale: float, causal: bool = True, out=None, lse=None,
                            out_dtype=torch.float32, workspace=None, dev_status=None, stream=None):
    """Prefill (TND queries, bottom-right causal) over the paged cache; returns out [T, H, d]."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev_bf16(t, n)
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (block_table, "block_table"),
                 (seq_lens_kv, "seq_lens_kv")):
        _dev_i32(t, n)
    T, H, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    B = cu_seqlens_q.numel()
    if out is None:
        out = torch.empty((T, H, d), dtype=out_dtype, device=q.device)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    if workspace is None:
        workspace = torch.empty(max(prefill_workspace_size(), 256), dtype=torch.uint8,
                                device=q.device)
    check(load().pkv_paged_attention_prefill(
        _ptr(out), code, _ptr(lse), _ptr(q), _ptr(cu_seqlens_q), T, _ptr(k_cache), _ptr(v_cache),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens_kv), B, H, hkv, d, bs, nb,
        float(scale), int(bool(causal)), _ptr(workspace), workspace.numel(), _ptr(dev_status),
        _stream(stream)), "pkv_paged_attention_prefill")
    return out


def mla_decode_workspace_size(B: int, H: int) -> int:
    return load().pkv_mla_decode_workspace_size(B, H)


def mla_paged_decode(q_nope, q_rope, cache_nope, cache_rope, block_table, seq_lens, scale: float,
                     out=None, lse=None, out_dtype=torch.float32, workspace=None, dev_status=None,
                     stream=None):
    """Absorbed MLA decode over the paged latent cache; returns out [B, H, 512]."""
    for t, n in ((q_nope, "q_nope"), (q_rope, "q_rope"), (cache_nope, "cache_nope"),
                 (cache_rope, "cache_rope")):
        _dev_bf16(t, n)
    _dev_i32(block_table, "block_table")
    _dev_i32(seq_lens, "seq_lens")
    B, H, dc = q_nope.shape
    dr = q_rope.shape[2]
    nb, bs, _, _ = cache_nope.shape
    if out is None:
        out = torch.empty((B, H, dc), dtype=out_dtype, device=q_nope.device)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    if workspace is None:
        need = mla_decode_workspace_size(B, H)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q_nope.device)
    check(load().pkv_mla_paged_decode(
        _ptr(out), code, _ptr(lse), _ptr(q_nope), _ptr(q_rope), _ptr(cache_nope), _ptr(cache_rope),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, H, dc, dr, bs, nb, float(scale),
        _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream)),
        "pkv_mla_paged_decode")
    return out


STATIC_SCRATCH_BYTES = 8 * 1024 * 1024  # PKV_DECODE_STATIC_SCRATCH_BYTES


def paged_attention_decode_static(q, k_cache, v_cache, block_table, seq_lens, scale: float,
                                  window: int = 0, out=None, lse=None, out_dtype=torch.float32,
                                  dev_status=None, stream=None):
    """Decode attention without a workspace, for callers that cannot allocate device
    memory: the library keeps the split-KV partials in its own fixed device array
    (STATIC_SCRATCH_BYTES, shared by every call; overlapping calls race). Same result
    as paged_attention_decode. The caller still passes (or lets this wrapper create)
    the output tensor."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev_bf16(t, n)
    _dev_i32(block_table, "block_table")
    _dev_i32(seq_lens, "seq_lens")
    B, H, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty((B, H, d), dtype=out_dtype, device=q.device)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    check(load().pkv_paged_attention_decode_static(
        _ptr(out), code, _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, H, hkv, d, bs, nb, float(scale), int(window),
        _ptr(dev_status), _stream(stream)), "pkv_paged_attention_decode_static")
    return out
