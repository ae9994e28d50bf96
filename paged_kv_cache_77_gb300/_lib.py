"""ctypes loader for libpaged_kv.so and the C signatures of include/paged_kv.h."""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpaged_kv.so")

i32, i64, f32, vp, sz = C.c_int32, C.c_int64, C.c_float, C.c_void_p, C.c_size_t
P_i32 = C.POINTER(C.c_int32)

# name -> (restype, argtypes); mirrors include/paged_kv.h.
SIGNATURES = {
    "pkv_last_error": (C.c_char_p, []),
    "pkv_version": (C.c_int, []),
    "pkv_pool_create": (C.c_int, [i64, vp, C.POINTER(vp)]),
    "pkv_pool_destroy": (None, [vp]),
    "pkv_pool_null_block": (i32, [vp]),
    "pkv_pool_num_free": (i64, [vp]),
    "pkv_pool_alloc": (C.c_int, [vp, i64, vp]),
    "pkv_pool_free": (C.c_int, [vp, vp, i64]),
    "pkv_pool_share": (C.c_int, [vp, vp, i64]),
    "pkv_pool_ref_count": (i32, [vp, i32]),
    "pkv_manager_create": (C.c_int, [i32, vp, vp, vp, i32, i64, i32, C.POINTER(vp)]),
    "pkv_manager_destroy": (None, [vp]),
    "pkv_manager_allocate_slots": (C.c_int, [vp, i64, i64, i64, i64]),
    "pkv_manager_get_block_ids": (i64, [vp, i64, i32, vp, i64]),
    "pkv_manager_free": (C.c_int, [vp, i64]),
    "pkv_manager_num_free": (i64, [vp, i32]),
    "pkv_manager_null_block": (i32, [vp, i32]),
    "pkv_manager_ref_count": (i32, [vp, i32, i32]),
    "pkv_manager_format_usage": (i64, [vp, C.c_char_p, i64]),
    "pkv_manager_block_table": (C.c_int, [vp, i32, vp, i32, i32, vp]),
    "pkv_block_hash": (C.c_uint64, [C.c_uint64, i32, vp, i32, i32]),
    "pkv_manager_match_prefix": (i64, [vp, i64, vp, i64]),
    "pkv_manager_cache_blocks": (C.c_int, [vp, i64, vp, i64]),
    "pkv_manager_fork": (i64, [vp, i64, vp, i32, i64, i32, vp, vp, i64, vp]),
    "pkv_copy_blocks": (C.c_int, [vp, i64, i64, vp, vp, i64, vp, vp]),
    "pkv_kv_cache_write_fp8": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, vp,
                                         vp]),
    "pkv_paged_attention_decode_fp8": (C.c_int, [vp, i32, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32,
                                                 i32, i32, i32, i32, i64, f32, i32, vp, sz, vp,
                                                 vp]),
    "pkv_mla_rmsnorm_rope_write": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32,
                                             i32, f32, vp, vp]),
    "pkv_num_skipped_tokens": (i64, [i64, i64]),
    "pkv_build_block_table": (C.c_int, [vp, vp, i32, i32, i32, i32, vp]),
    "pkv_build_block_table_arange": (C.c_int, [i32, i32, vp]),
    "pkv_build_slot_mapping": (i64, [vp, i32, vp, vp, i32, i32, vp, i64]),
    "pkv_block_num_fixed": (i64, [i64, i64, i64, i64]),
    "pkv_block_num_full_offline": (i64, [i64, i64, i64]),
    "pkv_block_num_full_online": (i64, [i64, i64, i64]),
    "pkv_kv_cache_write": (C.c_int, [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, i32, vp, vp]),
    "pkv_decode_workspace_size": (sz, [i32, i32, i32, i32]),
    "pkv_set_decode_kernel": (C.c_int, [i32]),
    "pkv_get_decode_kernel": (i32, []),
    "pkv_paged_attention_decode": (C.c_int, [vp, i32, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                             i32, i32, i64, f32, i32, vp, sz, vp, vp]),
    "pkv_decode_spec_workspace_size": (sz, [i32, i32, i32, i32, i32]),
    "pkv_paged_attention_decode_spec": (C.c_int, [vp, i32, vp, vp, vp, vp, vp, i32, vp, i32, i32,
                                                  i32, i32, i32, i32, i64, f32, i32, vp, sz, vp,
                                                  vp]),
    "pkv_prefill_workspace_size": (sz, []),
    "pkv_paged_attention_prefill": (C.c_int, [vp, i32, vp, vp, vp, i32, vp, vp, vp, i32, vp, i32,
                                              i32, i32, i32, i32, i64, f32, i32, vp, sz, vp, vp]),
    "pkv_mla_decode_workspace_size": (sz, [i32, i32]),
    "pkv_mla_paged_decode": (C.c_int, [vp, i32, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                       i32, i64, f32, vp, sz, vp, vp]),
    "pkv_mla_decode_spec_workspace_size": (sz, [i32, i32, i32]),
    "pkv_mla_paged_decode_spec": (C.c_int, [vp, i32, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                            i32, i32, i32, i64, f32, vp, sz, vp, vp]),
    "pkv_paged_attention_decode_static": (C.c_int, [vp, i32, vp, vp, vp, vp, vp, i32, vp, i32, i32,
                                                    i32, i32, i32, i64, f32, i32, vp, vp]),
    "pkv_selftest_bounded_wait": (C.c_int, [vp, vp]),
}

_lib = None


def load() -> C.CDLL:
    """Load the in-tree library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run paged_kv_cache_77_gb300.build.build()")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class PagedKVError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = load().pkv_last_error().decode(errors="replace")
        super().__init__(f"{where} failed with status {code}: {msg}")
        self.code = code


def check(code: int, where: str) -> int:
    if code < 0:
        raise PagedKVError(code, where)
    return code
