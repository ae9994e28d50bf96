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
    # ctypes turns the int into the c_void_p argument the signature declares.
    return None if t is None else t.data_ptr()


def _np_ptr(a: np.ndarray):
    return a.ctypes.data


# The current stream's raw handle without building a Stream object (the public
# torch.cuda.current_stream() costs ~10 us of host time per call on the machine's cores).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _dev_bf16(t, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16
            and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")


def _dev_i32(t, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32
            and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")


# ---- caller-provided buffers ------------------------------------------------
# The C ABI receives bare pointers and cannot see a tensor's size, so a wrong-shaped
# output would be written out of bounds on the GPU. Every buffer the caller passes
# is checked here, before any pointer crosses the boundary.
def _shape_str(shape) -> str:
    return "[" + ", ".join(str(int(x)) for x in shape) + "]"


def _on_device(t, device, name) -> None:
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def check_same_device(device, **tensors) -> None:
    """Every tensor given lives on `device` (None entries are skipped)."""
    for name, t in tensors.items():
        if t is not None:
            _on_device(t, device, name)


def check_current_device(device) -> None:
    """The library launches on the calling thread's current CUDA device (its SM count,
    the decode-without-workspace scratch array and torch's current stream all belong
    to it), so the tensors must live there."""
    if device.type == "cuda" and device.index != torch.cuda.current_device():
        raise ValueError(f"tensors are on {device} but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}; call under torch.cuda.device(...)")


def check_shape(t, shape, name) -> None:
    if t.shape != tuple(shape):
        raise ValueError(f"{name} has shape {_shape_str(t.shape)}, expected {_shape_str(shape)}")


def out_buffer(out, shape, out_dtype, device, name="out"):
    """The output tensor: a new one when `out` is None, else `out` after checking that
    it is a contiguous bf16 or fp32 tensor of exactly `shape` on `device`."""
    if out is None:
        if out_dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
        return torch.empty(tuple(shape), dtype=out_dtype, device=device)
    if not isinstance(out, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"{name} must be float32 or bfloat16, got {out.dtype}")
    _on_device(out, device, name)
    check_shape(out, shape, name)
    if not out.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return out


def lse_buffer(lse, shape, device, name="lse"):
    """`lse` (nullable): a contiguous fp32 tensor of exactly `shape` on `device`."""
    if lse is None:
        return None
    if not isinstance(lse, torch.Tensor) or lse.dtype != torch.float32:
        raise ValueError(f"{name} must be a float32 tensor")
    _on_device(lse, device, name)
    check_shape(lse, shape, name)
    if not lse.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return lse


def workspace_buffer(ws, need: int, device, name="workspace"):
    """The scratch buffer and its size in bytes: a new uint8 tensor when `ws` is None,
    else `ws` after checking that it is contiguous, on `device` and holds `need` bytes."""
    if ws is None:
        ws = torch.empty(max(int(need), 256), dtype=torch.uint8, device=device)
    if not isinstance(ws, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    _on_device(ws, device, name)
    if not ws.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    nbytes = ws.numel() * ws.element_size()
    if nbytes < need:
        raise ValueError(f"{name} holds {nbytes} bytes, the call needs {need}")
    return ws, nbytes


def status_buffer(st, device, name="dev_status"):
    """`dev_status` (nullable): an int32 tensor of at least one element on `device`."""
    if st is None:
        return None
    if not isinstance(st, torch.Tensor) or st.dtype != torch.int32 or st.numel() < 1:
        raise ValueError(f"{name} must be an int32 tensor with at least one element")
    _on_device(st, device, name)
    return st


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

    def share(self, ids) -> None:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        check(load().pkv_pool_share(self._h, _np_ptr(ids), len(ids)), "pkv_pool_share")

    def ref_count(self, block: int) -> int:
        return load().pkv_pool_ref_count(self._h, block)

    def build_block_table(self, seq_lens, block_size: int, window: int,
                          max_blocks_per_seq: int) -> np.ndarray:
        lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        table = np.empty((len(lens), max_blocks_per_seq), dtype=np.int32)
        check(load().pkv_build_block_table(self._h, _np_ptr(lens), len(lens), block_size, window,
                                           max_blocks_per_seq, _np_ptr(table)),
              "pkv_build_block_table")
        return table


class KVCacheManager:
    """Handle on the library's request-level allocator (pkv_manager_*).

    windows[i] = 0: full attention; > 0: sliding window. One pool per type."""

    def __init__(self, windows, num_blocks, block_size: int, max_model_len: int,
                 prefix_caching: bool = False, initial_orders=None):
        lib = load()
        self.num_types = len(windows)
        w = np.ascontiguousarray(windows, dtype=np.int32)
        n = np.ascontiguousarray(num_blocks, dtype=np.int64)
        self._orders = None
        orders_arg = None
        if initial_orders is not None:
            self._orders = [None if o is None else np.ascontiguousarray(o, dtype=np.int32)
                            for o in initial_orders]
            arr = (C.c_void_p * self.num_types)(*[None if o is None else o.ctypes.data
                                                 for o in self._orders])
            self._orders_arr = arr
            orders_arg = C.cast(arr, C.c_void_p)
        self._h = C.c_void_p()
        check(lib.pkv_manager_create(self.num_types, _np_ptr(w), _np_ptr(n), orders_arg, block_size,
                                     max_model_len, int(prefix_caching), C.byref(self._h)),
              "pkv_manager_create")
        self.block_size = block_size

    def __del__(self):
        if getattr(self, "_h", None):
            load().pkv_manager_destroy(self._h)
            self._h = None

    def allocate_slots(self, request_id: int, computed_tokens: int, num_new_tokens: int,
                       lookahead_tokens: int = 0) -> bool:
        return check(load().pkv_manager_allocate_slots(self._h, request_id, computed_tokens,
                                                       num_new_tokens, lookahead_tokens),
                     "pkv_manager_allocate_slots") == 1

    def get_block_ids(self, request_id: int) -> list[list[int]]:
        out = []
        for t in range(self.num_types):
            n = check(load().pkv_manager_get_block_ids(self._h, request_id, t, None, 0),
                      "pkv_manager_get_block_ids")
            buf = np.empty(max(n, 1), dtype=np.int32)
            load().pkv_manager_get_block_ids(self._h, request_id, t, _np_ptr(buf), n)
            out.append(buf[:n].tolist())
        return out

    def free(self, request_id: int) -> None:
        check(load().pkv_manager_free(self._h, request_id), "pkv_manager_free")

    def num_free(self, type_idx: int = 0) -> int:
        return load().pkv_manager_num_free(self._h, type_idx)

    def null_block(self, type_idx: int = 0) -> int:
        return load().pkv_manager_null_block(self._h, type_idx)

    def ref_count(self, type_idx: int, block: int) -> int:
        return load().pkv_manager_ref_count(self._h, type_idx, block)

    def format_usage(self) -> str:
        n = check(load().pkv_manager_format_usage(self._h, None, 0), "pkv_manager_format_usage")
        buf = C.create_string_buffer(n + 1)
        load().pkv_manager_format_usage(self._h, buf, n + 1)
        return buf.value.decode()

    def block_table(self, type_idx: int, request_ids, max_blocks_per_seq: int) -> np.ndarray:
        ids = np.ascontiguousarray(request_ids, dtype=np.int64)
        table = np.empty((len(ids), max_blocks_per_seq), dtype=np.int32)
        check(load().pkv_manager_block_table(self._h, type_idx, _np_ptr(ids), len(ids),
                                             max_blocks_per_seq, _np_ptr(table)),
              "pkv_manager_block_table")
        return table

    def match_prefix(self, request_id: int, tokens) -> int:
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        return check(load().pkv_manager_match_prefix(self._h, request_id, _np_ptr(toks), len(toks)),
                     "pkv_manager_match_prefix")

    def cache_blocks(self, request_id: int, tokens) -> None:
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        check(load().pkv_manager_cache_blocks(self._h, request_id, _np_ptr(toks), len(toks)),
              "pkv_manager_cache_blocks")

    def fork(self, parent_id: int, child_ids, num_tokens: int, shareable: bool):
        """Returns one list of (src, dst) copies per type."""
        kids = np.ascontiguousarray(child_ids, dtype=np.int64)
        held = max(len(r) for r in self.get_block_ids(parent_id))
        cap = max(1, held * len(kids) * self.num_types)
        src = np.empty(cap, dtype=np.int32)
        dst = np.empty(cap, dtype=np.int32)
        per = np.zeros(self.num_types, dtype=np.int64)
        check(load().pkv_manager_fork(self._h, parent_id, _np_ptr(kids), len(kids), num_tokens,
                                      int(shareable), _np_ptr(src), _np_ptr(dst), cap, _np_ptr(per)),
              "pkv_manager_fork")
        out, k = [], 0
        for t in range(self.num_types):
            out.append([(int(src[i]), int(dst[i])) for i in range(k, k + int(per[t]))])
            k += int(per[t])
        return out


def block_hash(parent, tokens, group_id: int) -> int:
    toks = np.ascontiguousarray(tokens, dtype=np.int32)
    return int(load().pkv_block_hash(0 if parent is None else parent, int(parent is not None),
                                     _np_ptr(toks), len(toks), group_id))


def build_block_table_arange(batch: int, blocks_per_seq: int) -> np.ndarray:
    table = np.empty((batch, blocks_per_seq), dtype=np.int32)
    check(load().pkv_build_block_table_arange(batch, blocks_per_seq, _np_ptr(table)),
          "pkv_build_block_table_arange")
    return table


def build_slot_mapping(block_table: np.ndarray, start_pos, num_new, block_size: int,
                       out: np.ndarray | None = None) -> np.ndarray:
    """slot_mapping of the new rows; `out` (optional): a contiguous int32 array with room
    for them, written in place (a view of its first entries is returned)."""
    table = np.ascontiguousarray(block_table, dtype=np.int32)
    sp = np.ascontiguousarray(start_pos, dtype=np.int32)
    nn = np.ascontiguousarray(num_new, dtype=np.int32)
    if out is None:
        cap = int(nn.sum())
        out = np.empty(max(cap, 1), dtype=np.int32)
    else:
        # Its length is the capacity the library checks the rows against.
        if (not isinstance(out, np.ndarray) or out.dtype != np.int32 or out.ndim != 1
                or not out.flags["C_CONTIGUOUS"]):
            raise ValueError("out must be a contiguous 1-D int32 array")
        cap = len(out)
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
def _cache_dims(cache, name, ndim=4):
    if cache.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions [num_blocks, block_size, H_kv, d]")
    return tuple(cache.shape)


def _table_and_lens(block_table, seq_lens, B, lens_name="seq_lens"):
    _dev_i32(block_table, "block_table")
    _dev_i32(seq_lens, lens_name)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError(f"block_table must be [B={B}, max_blocks_per_seq], "
                         f"got {_shape_str(block_table.shape)}")
    check_shape(seq_lens, (B,), lens_name)


def kv_cache_write(k_cache, v_cache, k, v, slot_mapping, dev_status=None, stream=None) -> None:
    """Write rows k[t] (and v[t]) at slot_mapping[t] of the paged caches.

    k_cache [nb, bs, H_kv, d_k]; v_cache [nb, bs, H_kv, d_v] or None (with v None)."""
    _dev_bf16(k_cache, "k_cache")
    _dev_bf16(k, "k")
    _dev_i32(slot_mapping, "slot_mapping")
    if (v_cache is None) != (v is None):
        raise ValueError("v_cache and v are given together or not at all")
    nb, bs, hkv, dk = _cache_dims(k_cache, "k_cache")
    T = slot_mapping.numel()
    check_shape(k, (T, hkv, dk), "k")
    dv = 0
    if v_cache is not None:
        _dev_bf16(v_cache, "v_cache")
        _dev_bf16(v, "v")
        _, vbs, vhkv, dv = _cache_dims(v_cache, "v_cache")
        check_shape(v_cache, (nb, bs, hkv, dv), "v_cache")
        check_shape(v, (T, hkv, dv), "v")
    dev = k_cache.device
    check_same_device(dev, k=k, v_cache=v_cache, v=v, slot_mapping=slot_mapping)
    check_current_device(dev)
    status_buffer(dev_status, dev)
    check(load().pkv_kv_cache_write(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v),
                                    _ptr(slot_mapping), T, nb, bs, hkv, dk, dv,
                                    _ptr(dev_status), _stream(stream)), "pkv_kv_cache_write")


KERNEL_AUTO, KERNEL_CUDA_CORE, KERNEL_TENSOR_CORE = 0, 1, 2


def copy_blocks(cache, src, dst, dev_status=None, stream=None) -> None:
    """Block dst[i] of `cache` ([num_blocks, ...], contiguous, CUDA) becomes a bit copy
    of block src[i] (the device side of a fork)."""
    if not (isinstance(cache, torch.Tensor) and cache.is_cuda and cache.is_contiguous()):
        raise ValueError("cache must be a contiguous CUDA tensor")
    _dev_i32(src, "src")
    _dev_i32(dst, "dst")
    if src.numel() != dst.numel():
        raise ValueError("src and dst differ in length")
    dev = cache.device
    check_same_device(dev, src=src, dst=dst)
    check_current_device(dev)
    status_buffer(dev_status, dev)
    block_bytes = cache[0].numel() * cache.element_size()
    check(load().pkv_copy_blocks(_ptr(cache), cache.shape[0], block_bytes, _ptr(src), _ptr(dst),
                                 src.numel(), _ptr(dev_status), _stream(stream)),
          "pkv_copy_blocks")


def mla_rmsnorm_rope_write(cache_nope, cache_rope, latent, gamma, cos, sin, slot_mapping,
                           epsilon: float, k_nope_out=None, k_rope_out=None, dev_status=None,
                           stream=None) -> None:
    """Fused RMSNorm (latent 512) + RoPE (rope 64) + paged write of MLA rows.

    latent [T, 512 + 64] bf16 (the latent row followed by the rope row), gamma [512],
    cos / sin [T, 64] fp32; optional k_nope_out [T, 512] / k_rope_out [T, 64] bf16."""
    for t, n in ((cache_nope, "cache_nope"), (cache_rope, "cache_rope"), (latent, "latent"),
                 (gamma, "gamma")):
        _dev_bf16(t, n)
    for t, n in ((cos, "cos"), (sin, "sin")):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32
                and t.is_contiguous()):
            raise ValueError(f"{n} must be a contiguous fp32 CUDA tensor")
    _dev_i32(slot_mapping, "slot_mapping")
    T = slot_mapping.numel()
    nb, bs = cache_nope.shape[0], cache_nope.shape[1]
    dc, dr = cache_nope.shape[-1], cache_rope.shape[-1]
    check_shape(cache_rope, (nb, bs, 1, dr), "cache_rope")
    check_shape(cache_nope, (nb, bs, 1, dc), "cache_nope")
    check_shape(latent, (T, dc + dr), "latent")
    check_shape(gamma, (dc,), "gamma")
    check_shape(cos, (T, dr), "cos")
    check_shape(sin, (T, dr), "sin")
    dev = cache_nope.device
    for t, n, shape in ((k_nope_out, "k_nope_out", (T, dc)), (k_rope_out, "k_rope_out", (T, dr))):
        if t is not None:
            _dev_bf16(t, n)
            check_shape(t, shape, n)
    check_same_device(dev, cache_rope=cache_rope, latent=latent, gamma=gamma, cos=cos, sin=sin,
                      slot_mapping=slot_mapping, k_nope_out=k_nope_out, k_rope_out=k_rope_out)
    check_current_device(dev)
    status_buffer(dev_status, dev)
    check(load().pkv_mla_rmsnorm_rope_write(
        _ptr(cache_nope), _ptr(cache_rope), _ptr(k_nope_out), _ptr(k_rope_out), _ptr(latent),
        _ptr(gamma), _ptr(cos), _ptr(sin), _ptr(slot_mapping), T, nb, bs, dc, dr, epsilon,
        _ptr(dev_status), _stream(stream)), "pkv_mla_rmsnorm_rope_write")


def _fp8_cache(t, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.uint8
            and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous uint8 CUDA tensor")


def _f32_dev(t, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32
            and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")


def kv_cache_write_fp8(k_cache, v_cache, k_scale, v_scale, k, v, slot_mapping, dev_status=None,
                       stream=None) -> None:
    """Quantise new K/V rows to FP8 E4M3 codes + per-row scales and scatter them.

    k_cache / v_cache [nb, bs, H_kv, d] uint8; k_scale / v_scale [nb, H_kv, bs] fp32;
    k / v [T, H_kv, d] bf16."""
    _fp8_cache(k_cache, "k_cache")
    _fp8_cache(v_cache, "v_cache")
    _f32_dev(k_scale, "k_scale")
    _f32_dev(v_scale, "v_scale")
    _dev_bf16(k, "k")
    _dev_bf16(v, "v")
    _dev_i32(slot_mapping, "slot_mapping")
    nb, bs, hkv, d = _cache_dims(k_cache, "k_cache")
    T = slot_mapping.numel()
    check_shape(v_cache, (nb, bs, hkv, d), "v_cache")
    check_shape(k_scale, (nb, hkv, bs), "k_scale")
    check_shape(v_scale, (nb, hkv, bs), "v_scale")
    check_shape(k, (T, hkv, d), "k")
    check_shape(v, (T, hkv, d), "v")
    dev = k_cache.device
    check_same_device(dev, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale, k=k, v=v,
                      slot_mapping=slot_mapping)
    check_current_device(dev)
    status_buffer(dev_status, dev)
    check(load().pkv_kv_cache_write_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                        _ptr(k), _ptr(v), _ptr(slot_mapping), T, nb, bs,
                                        hkv, d, _ptr(dev_status), _stream(stream)),
          "pkv_kv_cache_write_fp8")


def paged_attention_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                               scale: float, window: int = 0, out=None, lse=None,
                               out_dtype=torch.float32, workspace=None, dev_status=None,
                               stream=None):
    """Decode attention over an FP8 cache (codes + per-row scales); returns out [B, H, d]."""
    _dev_bf16(q, "q")
    _fp8_cache(k_cache, "k_cache")
    _fp8_cache(v_cache, "v_cache")
    _f32_dev(k_scale, "k_scale")
    _f32_dev(v_scale, "v_scale")
    B, H, d = q.shape
    nb, bs, hkv, dk = _cache_dims(k_cache, "k_cache")
    if dk != d:
        raise ValueError(f"k_cache head_dim {dk} differs from q's {d}")
    check_shape(v_cache, (nb, bs, hkv, d), "v_cache")
    check_shape(k_scale, (nb, hkv, bs), "k_scale")
    check_shape(v_scale, (nb, hkv, bs), "v_scale")
    _table_and_lens(block_table, seq_lens, B)
    dev = q.device
    check_same_device(dev, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
                      block_table=block_table, seq_lens=seq_lens)
    check_current_device(dev)
    out = out_buffer(out, (B, H, d), out_dtype, dev)
    lse_buffer(lse, (B, H), dev)
    status_buffer(dev_status, dev)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    workspace, ws_bytes = workspace_buffer(workspace, decode_workspace_size(B, H, hkv, d), dev)
    check(load().pkv_paged_attention_decode_fp8(
        _ptr(out), code, _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, H, hkv, d, bs, nb,
        scale, window, _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
        "pkv_paged_attention_decode_fp8")
    return out


def set_decode_kernel(kernel: int) -> None:
    """Select the decode kernel process-wide (KERNEL_AUTO / _CUDA_CORE / _TENSOR_CORE)."""
    check(load().pkv_set_decode_kernel(kernel), "pkv_set_decode_kernel")


def get_decode_kernel() -> int:
    return load().pkv_get_decode_kernel()


def decode_workspace_size(B: int, H: int, H_kv: int, head_dim: int) -> int:
    return load().pkv_decode_workspace_size(B, H, H_kv, head_dim)


def _decode_inputs(q, k_cache, v_cache, block_table, seq_lens, qdims):
    """Checks shared by the bf16-cache decode calls; returns (dims of q, cache dims)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev_bf16(t, n)
    if q.dim() != qdims:
        raise ValueError(f"q must have {qdims} dimensions")
    nb, bs, hkv, dk = _cache_dims(k_cache, "k_cache")
    d = q.shape[-1]
    if dk != d:
        raise ValueError(f"k_cache head_dim {dk} differs from q's {d}")
    check_shape(v_cache, (nb, bs, hkv, d), "v_cache")
    _table_and_lens(block_table, seq_lens, q.shape[0])
    dev = q.device
    check_same_device(dev, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                      seq_lens=seq_lens)
    check_current_device(dev)
    return tuple(int(x) for x in q.shape), (nb, bs, hkv)


def paged_attention_decode(q, k_cache, v_cache, block_table, seq_lens, scale: float, window: int = 0,
                           out=None, lse=None, out_dtype=torch.float32, workspace=None,
                           dev_status=None, stream=None):
    """Decode attention over the paged cache; returns out [B, H, d] (and fills lse [B, H])."""
    (B, H, d), (nb, bs, hkv) = _decode_inputs(q, k_cache, v_cache, block_table, seq_lens, 3)
    dev = q.device
    out = out_buffer(out, (B, H, d), out_dtype, dev)
    lse_buffer(lse, (B, H), dev)
    status_buffer(dev_status, dev)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    workspace, ws_bytes = workspace_buffer(workspace, decode_workspace_size(B, H, hkv, d), dev)
    check(load().pkv_paged_attention_decode(
        _ptr(out), code, _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, H, hkv, d, bs, nb, float(scale), int(window),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
        "pkv_paged_attention_decode")
    return out


def decode_spec_workspace_size(B: int, q_len: int, H: int, H_kv: int, head_dim: int) -> int:
    return load().pkv_decode_spec_workspace_size(B, q_len, H, H_kv, head_dim)


def paged_attention_decode_spec(q, k_cache, v_cache, block_table, seq_lens, scale: float,
                                window: int = 0, out=None, lse=None, out_dtype=torch.float32,
                                workspace=None, dev_status=None, stream=None):
    """Speculative decode: q [B, q_len, H, d], the q_len new rows of each sequence
    already in the cache, bottom-right causal; returns out [B, q_len, H, d] (and fills
    lse [B, q_len, H])."""
    (B, Q, H, d), (nb, bs, hkv) = _decode_inputs(q, k_cache, v_cache, block_table, seq_lens, 4)
    dev = q.device
    out = out_buffer(out, (B, Q, H, d), out_dtype, dev)
    lse_buffer(lse, (B, Q, H), dev)
    status_buffer(dev_status, dev)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    workspace, ws_bytes = workspace_buffer(workspace, decode_spec_workspace_size(B, Q, H, hkv, d),
                                           dev)
    check(load().pkv_paged_attention_decode_spec(
        _ptr(out), code, _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, Q, H, hkv, d, bs, nb, float(scale), int(window),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
        "pkv_paged_attention_decode_spec")
    return out


def prefill_workspace_size() -> int:
    return load().pkv_prefill_workspace_size()


def paged_attention_prefill(q, cu_seqlens_q, k_cache, v_cache, block_table, seq_lens_kv,
                            scale: float, causal: bool = True, out=None, lse=None,
                            out_dtype=torch.float32, workspace=None, dev_status=None, stream=None):
    """Prefill (TND queries, bottom-right causal) over the paged cache; returns out [T, H, d]
    (and fills lse [T, H])."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev_bf16(t, n)
    _dev_i32(cu_seqlens_q, "cu_seqlens_q")
    if q.dim() != 3:
        raise ValueError("q must be TND [T, H, d]")
    T, H, d = (int(x) for x in q.shape)
    nb, bs, hkv, dk = _cache_dims(k_cache, "k_cache")
    if dk != d:
        raise ValueError(f"k_cache head_dim {dk} differs from q's {d}")
    check_shape(v_cache, (nb, bs, hkv, d), "v_cache")
    B = cu_seqlens_q.numel()
    _table_and_lens(block_table, seq_lens_kv, B, "seq_lens_kv")
    dev = q.device
    check_same_device(dev, cu_seqlens_q=cu_seqlens_q, k_cache=k_cache, v_cache=v_cache,
                      block_table=block_table, seq_lens_kv=seq_lens_kv)
    check_current_device(dev)
    out = out_buffer(out, (T, H, d), out_dtype, dev)
    lse_buffer(lse, (T, H), dev)
    status_buffer(dev_status, dev)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    workspace, ws_bytes = workspace_buffer(workspace, prefill_workspace_size(), dev)
    check(load().pkv_paged_attention_prefill(
        _ptr(out), code, _ptr(lse), _ptr(q), _ptr(cu_seqlens_q), T, _ptr(k_cache), _ptr(v_cache),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens_kv), B, H, hkv, d, bs, nb,
        float(scale), int(bool(causal)), _ptr(workspace), ws_bytes, _ptr(dev_status),
        _stream(stream)), "pkv_paged_attention_prefill")
    return out


def mla_decode_workspace_size(B: int, H: int) -> int:
    return load().pkv_mla_decode_workspace_size(B, H)


def _mla_inputs(q_nope, q_rope, cache_nope, cache_rope, block_table, seq_lens, qdims):
    for t, n in ((q_nope, "q_nope"), (q_rope, "q_rope"), (cache_nope, "cache_nope"),
                 (cache_rope, "cache_rope")):
        _dev_bf16(t, n)
    if q_nope.dim() != qdims:
        raise ValueError(f"q_nope must have {qdims} dimensions")
    lead = tuple(int(x) for x in q_nope.shape[:-1])
    dc, dr = int(q_nope.shape[-1]), int(q_rope.shape[-1])
    check_shape(q_rope, lead + (dr,), "q_rope")
    nb, bs = _cache_dims(cache_nope, "cache_nope")[:2]
    check_shape(cache_nope, (nb, bs, 1, dc), "cache_nope")
    check_shape(cache_rope, (nb, bs, 1, dr), "cache_rope")
    _table_and_lens(block_table, seq_lens, lead[0])
    dev = q_nope.device
    check_same_device(dev, q_rope=q_rope, cache_nope=cache_nope, cache_rope=cache_rope,
                      block_table=block_table, seq_lens=seq_lens)
    check_current_device(dev)
    return lead, dc, dr, nb, bs


def mla_paged_decode(q_nope, q_rope, cache_nope, cache_rope, block_table, seq_lens, scale: float,
                     out=None, lse=None, out_dtype=torch.float32, workspace=None, dev_status=None,
                     stream=None):
    """Absorbed MLA decode over the paged latent cache; returns out [B, H, 512] (and
    fills lse [B, H])."""
    (B, H), dc, dr, nb, bs = _mla_inputs(q_nope, q_rope, cache_nope, cache_rope, block_table,
                                         seq_lens, 3)
    dev = q_nope.device
    out = out_buffer(out, (B, H, dc), out_dtype, dev)
    lse_buffer(lse, (B, H), dev)
    status_buffer(dev_status, dev)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    workspace, ws_bytes = workspace_buffer(workspace, mla_decode_workspace_size(B, H), dev)
    check(load().pkv_mla_paged_decode(
        _ptr(out), code, _ptr(lse), _ptr(q_nope), _ptr(q_rope), _ptr(cache_nope), _ptr(cache_rope),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, H, dc, dr, bs, nb, float(scale),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
        "pkv_mla_paged_decode")
    return out


def mla_decode_spec_workspace_size(B: int, q_len: int, H: int) -> int:
    return load().pkv_mla_decode_spec_workspace_size(B, q_len, H)


def mla_paged_decode_spec(q_nope, q_rope, cache_nope, cache_rope, block_table, seq_lens,
                          scale: float, out=None, lse=None, out_dtype=torch.float32, workspace=None,
                          dev_status=None, stream=None):
    """Absorbed MLA decode of q_len new rows per sequence (bottom-right causal);
    q_nope [B, q_len, H, 512], q_rope [B, q_len, H, 64]; returns out [B, q_len, H, 512]
    (and fills lse [B, q_len, H])."""
    (B, Q, H), dc, dr, nb, bs = _mla_inputs(q_nope, q_rope, cache_nope, cache_rope, block_table,
                                            seq_lens, 4)
    dev = q_nope.device
    out = out_buffer(out, (B, Q, H, dc), out_dtype, dev)
    lse_buffer(lse, (B, Q, H), dev)
    status_buffer(dev_status, dev)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    workspace, ws_bytes = workspace_buffer(workspace, mla_decode_spec_workspace_size(B, Q, H), dev)
    check(load().pkv_mla_paged_decode_spec(
        _ptr(out), code, _ptr(lse), _ptr(q_nope), _ptr(q_rope), _ptr(cache_nope), _ptr(cache_rope),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, Q, H, dc, dr, bs, nb,
        float(scale), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)),
        "pkv_mla_paged_decode_spec")
    return out


STATIC_SCRATCH_BYTES = 8 * 1024 * 1024  # PKV_DECODE_STATIC_SCRATCH_BYTES


def paged_attention_decode_static(q, k_cache, v_cache, block_table, seq_lens, scale: float,
                                  window: int = 0, out=None, lse=None, out_dtype=torch.float32,
                                  dev_status=None, stream=None):
    """Decode attention without a workspace, for callers that cannot allocate device
    memory: the library keeps the split-KV partials in its own fixed device array
    (STATIC_SCRATCH_BYTES, shared by every call; overlapping calls race). Same result
    as paged_attention_decode. The caller still passes (or lets this wrapper create)
    the output tensor. The tensors must live on the current CUDA device, whose copy
    of the array the call uses, and `stream` must belong to that device."""
    (B, H, d), (nb, bs, hkv) = _decode_inputs(q, k_cache, v_cache, block_table, seq_lens, 3)
    dev = q.device
    out = out_buffer(out, (B, H, d), out_dtype, dev)
    lse_buffer(lse, (B, H), dev)
    status_buffer(dev_status, dev)
    code = PKV_F32 if out.dtype == torch.float32 else PKV_BF16
    check(load().pkv_paged_attention_decode_static(
        _ptr(out), code, _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, H, hkv, d, bs, nb, float(scale), int(window),
        _ptr(dev_status), _stream(stream)), "pkv_paged_attention_decode_static")
    return out


DEV_TIMEOUT = 8  # PKV_DEV_TIMEOUT: a bounded wait inside a kernel gave up


def selftest_bounded_wait(dev_status, stream=None) -> None:
    """Launch the failure-path self-test: a kernel whose bounded waits on an mbarrier
    that nothing completes run out (about a second) and set DEV_TIMEOUT in
    dev_status (an int32 CUDA tensor of at least one element)."""
    if not (isinstance(dev_status, torch.Tensor) and dev_status.is_cuda):
        raise ValueError("dev_status must be an int32 CUDA tensor")
    status_buffer(dev_status, dev_status.device)
    check_current_device(dev_status.device)
    check(load().pkv_selftest_bounded_wait(_ptr(dev_status), _stream(stream)),
          "pkv_selftest_bounded_wait")
