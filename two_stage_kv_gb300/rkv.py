"""Thin ctypes binding of the C ABI in include/rkv.h.

Argument marshalling only: every function forwards to the function of the
same name in librkv.so (device pointers from torch tensors, the current CUDA
stream unless one is given) and raises RkvError on a non-OK status.  There is
no fallback: if the library is missing this module raises on first use.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "librkv.so")

RKV_OK = 0
STATUS_NAMES = {0: "RKV_OK", 1: "RKV_ERR_INVALID_ARG", 2: "RKV_ERR_UNSUPPORTED", 3: "RKV_ERR_WORKSPACE",
                4: "RKV_ERR_CUDA", 5: "RKV_ERR_TIMEOUT"}

# Every symbol include/rkv.h declares.
EXPORTED = ["rkv_last_error", "rkv_abi_version", "rkv_budget_split", "rkv_snap_evict_workspace",
            "rkv_snap_evict", "rkv_snap_evict_ragged", "rkv_snap_evict_paged", "rkv_snap_evict_noalloc", "rkv_compact_kt", "rkv_compact_kt_paged", "rkv_build_kt", "rkv_append_kv", "rkv_hsa_decode", "rkv_hsa_decode_mt",
            "rkv_hsa_decode_ragged", "rkv_hsa_decode_paged", "rkv_keep_mask", "rkv_build_kt_masked",
            "rkv_hsa_decode_mt_masked", "rkv_compact_kt_fp8", "rkv_hsa_decode_fp8", "rkv_debug_set_wait",
            "rkv_read_device_flags"]


class RkvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


_lib = None

_i32, _i64, _f32, _f64, _vp, _sz = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double,
                                    ctypes.c_void_p, ctypes.c_size_t)
_SIGS = {
    "rkv_last_error": (ctypes.c_char_p, []),
    "rkv_abi_version": (_i32, []),
    "rkv_budget_split": (_i32, [_i64, _i64, _i32, _i32, _f64, ctypes.POINTER(_f64), ctypes.POINTER(_i64),
                                ctypes.POINTER(_i32)]),
    "rkv_snap_evict_workspace": (_sz, [Dims, _i64, _i32]),
    "rkv_snap_evict": (_i32, [Dims, _vp, _i32, _vp, _vp, _i64, _i64, _i32, _i32, _i64, _f32, _vp, _i64, _vp, _vp,
                              _i64, _vp, _vp, _sz, _vp]),
    "rkv_snap_evict_ragged": (_i32, [Dims, _vp, _i32, _vp, _vp, _i64, _vp, _i64, _i32, _i32, _vp, _i64, _f32, _vp,
                                     _i64, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "rkv_snap_evict_paged": (_i32, [Dims, _vp, _i32, _vp, _vp, _i64, _i32, _vp, _i64, _vp, _i64, _i32, _i32, _vp,
                                    _i64, _f32, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "rkv_snap_evict_noalloc": (_i32, [Dims, _vp, _i32, _vp, _vp, _i64, _i64, _i32, _i32, _i64, _f32, _vp, _i64, _vp,
                                      _vp, _i64, _vp, _vp]),
    "rkv_compact_kt": (_i32, [Dims, _vp, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _i64, _i32, _vp, _i64, _vp]),
    "rkv_compact_kt_paged": (_i32, [Dims, _vp, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _i64, _i32, _vp,
                                    _i64, _vp]),
    "rkv_build_kt": (_i32, [Dims, _vp, _i64, _i64, _vp, _i64, _i32, _vp, _i64, _vp]),
    "rkv_append_kv": (_i32, [Dims, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _i32, _vp]),
    "rkv_hsa_decode": (_i32, [Dims, _vp, _vp, _vp, _i64, _i64, _vp, _i64, _i32, _i32, _i32, _f32, _vp, _vp, _vp,
                              _vp, _vp, _vp]),
    "rkv_hsa_decode_mt": (_i32, [Dims, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _vp, _i64, _i32, _i32, _i32, _f32,
                                 _vp, _vp, _vp, _vp, _vp, _i64, _vp]),
    "rkv_hsa_decode_ragged": (_i32, [Dims, _vp, _vp, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _i32, _i32, _f32, _vp,
                                     _vp, _vp, _vp, _vp, _vp]),
    "rkv_hsa_decode_paged": (_i32, [Dims, _vp, _vp, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _i32, _i32,
                                    _f32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "rkv_keep_mask": (_i32, [Dims, _vp, _i64, _i64, _i64, _vp, _i64, _vp]),
    "rkv_build_kt_masked": (_i32, [Dims, _vp, _i64, _i64, _vp, _i64, _i64, _i32, _vp, _i64, _vp]),
    "rkv_hsa_decode_mt_masked": (_i32, [Dims, _vp, _vp, _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i32, _i32,
                                        _i32, _f32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "rkv_compact_kt_fp8": (_i32, [Dims, _vp, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _i32, _vp, _i64,
                                  _vp]),
    "rkv_hsa_decode_fp8": (_i32, [Dims, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _f32, _vp,
                                  _vp, _vp, _vp, _vp, _vp]),
    "rkv_debug_set_wait": (_i32, [ctypes.c_uint64, ctypes.c_uint32]),
    "rkv_read_device_flags": (_i32, [ctypes.POINTER(ctypes.c_uint32)]),
}


def lib():
    """The loaded librkv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with two_stage_kv_gb300.build.build()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _check(status: int):
    if status != RKV_OK:
        raise RkvError(status, lib().rkv_last_error().decode(errors="replace"))


def _dims(d: Sequence[int]) -> Dims:
    return Dims(*[int(x) for x in d])


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def rkv_abi_version() -> int:
    return lib().rkv_abi_version()


def rkv_budget_split(S: int, t: int, blk: int, W: int = 32, r_override: float = -1.0) -> Tuple[float, int, int]:
    r, B1, k2 = _f64(), _i64(), _i32()
    _check(lib().rkv_budget_split(S, t, blk, W, r_override, ctypes.byref(r), ctypes.byref(B1), ctypes.byref(k2)))
    return r.value, B1.value, k2.value


def rkv_snap_evict_workspace(dims, S: int, W: int) -> int:
    return lib().rkv_snap_evict_workspace(_dims(dims), S, W)


def rkv_snap_evict(dims, q_obs, W, k, v, cap, S, pool_kernel, n_sink, B1, scale, keep_idx, keep_ld, k_out, v_out,
                   out_cap, pooled_out, ws, ws_bytes, stream=None):
    _check(lib().rkv_snap_evict(_dims(dims), _ptr(q_obs), W, _ptr(k), _ptr(v), cap, S, pool_kernel, n_sink, B1,
                                scale, _ptr(keep_idx), keep_ld, _ptr(k_out), _ptr(v_out), out_cap, _ptr(pooled_out),
                                _ptr(ws), ws_bytes, _stream(stream)))


def rkv_snap_evict_ragged(dims, q_obs, W, k, v, cap, S_rows, S_max, pool_kernel, n_sink, B1_rows, B1_max, scale,
                          keep_idx, keep_ld, k_out, v_out, out_cap, pooled_out, ws, ws_bytes, stream=None):
    _check(lib().rkv_snap_evict_ragged(_dims(dims), _ptr(q_obs), W, _ptr(k), _ptr(v), cap, _ptr(S_rows), S_max,
                                       pool_kernel, n_sink, _ptr(B1_rows), B1_max, scale, _ptr(keep_idx), keep_ld,
                                       _ptr(k_out), _ptr(v_out), out_cap, _ptr(pooled_out), _ptr(ws), ws_bytes,
                                       _stream(stream)))


def rkv_snap_evict_paged(dims, q_obs, W, k_pages, v_pages, num_pages, page, block_table, bt_stride, S_rows, S_max,
                         pool_kernel, n_sink, B1_rows, B1_max, scale, keep_idx, keep_ld, k_out, v_out, out_cap,
                         pooled_out, ws, ws_bytes, stream=None):
    _check(lib().rkv_snap_evict_paged(_dims(dims), _ptr(q_obs), W, _ptr(k_pages), _ptr(v_pages), num_pages, page,
                                      _ptr(block_table), bt_stride, _ptr(S_rows), S_max, pool_kernel, n_sink,
                                      _ptr(B1_rows), B1_max, scale, _ptr(keep_idx), keep_ld, _ptr(k_out), _ptr(v_out),
                                      out_cap, _ptr(pooled_out), _ptr(ws), ws_bytes, _stream(stream)))


def rkv_snap_evict_noalloc(dims, q_obs, W, k, v, cap, S, pool_kernel, n_sink, B1, scale, keep_idx, keep_ld, k_out,
                           v_out, out_cap, pooled_out, stream=None):
    """Stage-1 eviction using the library's fixed device scratch (no workspace argument),
    for callers that cannot allocate device memory."""
    _check(lib().rkv_snap_evict_noalloc(_dims(dims), _ptr(q_obs), W, _ptr(k), _ptr(v), cap, S, pool_kernel, n_sink,
                                        B1, scale, _ptr(keep_idx), keep_ld, _ptr(k_out), _ptr(v_out), out_cap,
                                        _ptr(pooled_out), _stream(stream)))


def rkv_compact_kt(dims, k, v, cap, keep_idx, keep_ld, B1, k_out, v_out, out_cap, blk, kt, nblk_cap, stream=None):
    _check(lib().rkv_compact_kt(_dims(dims), _ptr(k), _ptr(v), cap, _ptr(keep_idx), keep_ld, B1, _ptr(k_out),
                                _ptr(v_out), out_cap, blk, _ptr(kt), nblk_cap, _stream(stream)))


def rkv_compact_kt_paged(dims, k, v, cap, keep_idx, keep_ld, B1, k_pages, v_pages, num_pages, block_table, bt_stride,
                         blk, kt, nblk_cap, stream=None):
    _check(lib().rkv_compact_kt_paged(_dims(dims), _ptr(k), _ptr(v), cap, _ptr(keep_idx), keep_ld, B1, _ptr(k_pages),
                                      _ptr(v_pages), num_pages, _ptr(block_table), bt_stride, blk, _ptr(kt), nblk_cap,
                                      _stream(stream)))


def rkv_build_kt(dims, k, cap, n, idx, idx_cap, blk, kt, nblk_cap, stream=None):
    _check(lib().rkv_build_kt(_dims(dims), _ptr(k), cap, n, _ptr(idx), idx_cap, blk, _ptr(kt), nblk_cap,
                              _stream(stream)))


def rkv_append_kv(dims, k_new, v_new, k, v, cap, n, row, idx, idx_cap, kt, nblk_cap, blk, stream=None):
    _check(lib().rkv_append_kv(_dims(dims), _ptr(k_new), _ptr(v_new), _ptr(k), _ptr(v), cap, n, row, _ptr(idx),
                               idx_cap, _ptr(kt), nblk_cap, blk, _stream(stream)))


def rkv_hsa_decode(dims, q, k, v, cap, n, kt, nblk_cap, blk, k1, k2, scale, out, sel_blocks=None,
                   sel_channels=None, k_new=None, v_new=None, stream=None):
    _check(lib().rkv_hsa_decode(_dims(dims), _ptr(q), _ptr(k), _ptr(v), cap, n, _ptr(kt), nblk_cap, blk, k1, k2,
                                scale, _ptr(out), _ptr(sel_blocks), _ptr(sel_channels), _ptr(k_new), _ptr(v_new),
                                _stream(stream)))


def rkv_hsa_decode_mt(dims, q, k, v, cap, idx, idx_cap, n, kt, nblk_cap, blk, k1, k2, scale, out,
                      sel_blocks=None, sel_channels=None, k_new=None, v_new=None, row=0, stream=None):
    _check(lib().rkv_hsa_decode_mt(_dims(dims), _ptr(q), _ptr(k), _ptr(v), cap, _ptr(idx), idx_cap, n, _ptr(kt),
                                   nblk_cap, blk, k1, k2, scale, _ptr(out), _ptr(sel_blocks), _ptr(sel_channels),
                                   _ptr(k_new), _ptr(v_new), row, _stream(stream)))


def rkv_hsa_decode_ragged(dims, q, k, v, cap, n_rows, n_max, kt, nblk_cap, blk, k1, k2, scale, out,
                          sel_blocks=None, sel_channels=None, k_new=None, v_new=None, stream=None):
    """HSA decode with a per-batch-row candidate count n_rows ([B] int32 on the device)."""
    _check(lib().rkv_hsa_decode_ragged(_dims(dims), _ptr(q), _ptr(k), _ptr(v), cap, _ptr(n_rows), n_max, _ptr(kt),
                                       nblk_cap, blk, k1, k2, scale, _ptr(out), _ptr(sel_blocks),
                                       _ptr(sel_channels), _ptr(k_new), _ptr(v_new), _stream(stream)))


def rkv_hsa_decode_paged(dims, q, k_pages, v_pages, num_pages, block_table, bt_stride, n_rows, n_max, kt, nblk_cap,
                         blk, k1, k2, scale, out, sel_blocks=None, sel_channels=None, k_new=None, v_new=None,
                         stream=None):
    """HSA decode over paged K/V pools [num_pages, Hkv, blk, D] addressed by a block table."""
    _check(lib().rkv_hsa_decode_paged(_dims(dims), _ptr(q), _ptr(k_pages), _ptr(v_pages), num_pages,
                                      _ptr(block_table), bt_stride, _ptr(n_rows), n_max, _ptr(kt), nblk_cap, blk, k1,
                                      k2, scale, _ptr(out), _ptr(sel_blocks), _ptr(sel_channels), _ptr(k_new),
                                      _ptr(v_new), _stream(stream)))


def rkv_keep_mask(dims, keep_idx, keep_ld, B1, n_prompt, mask, mask_ld, stream=None):
    """Candidate bits of the prompt rows [0, n_prompt) from a stage-1 keep list."""
    _check(lib().rkv_keep_mask(_dims(dims), _ptr(keep_idx), keep_ld, B1, n_prompt, _ptr(mask), mask_ld,
                               _stream(stream)))


def rkv_build_kt_masked(dims, k, cap, n, mask, mask_ld, n_prompt, blk, kt, nblk_cap, stream=None):
    """KT over fixed blocks of the full cache, candidate rows only."""
    _check(lib().rkv_build_kt_masked(_dims(dims), _ptr(k), cap, n, _ptr(mask), mask_ld, n_prompt, blk, _ptr(kt),
                                     nblk_cap, _stream(stream)))


def rkv_hsa_decode_mt_masked(dims, q, k, v, cap, n, mask, mask_ld, n_prompt, kt, nblk_cap, blk, k1, k2, scale, out,
                             sel_blocks=None, sel_channels=None, k_new=None, v_new=None, stream=None):
    """Multi-turn HSA step over fixed blocks of the full cache (candidate rows from the mask)."""
    _check(lib().rkv_hsa_decode_mt_masked(_dims(dims), _ptr(q), _ptr(k), _ptr(v), cap, n, _ptr(mask), mask_ld,
                                          n_prompt, _ptr(kt), nblk_cap, blk, k1, k2, scale, _ptr(out),
                                          _ptr(sel_blocks), _ptr(sel_channels), _ptr(k_new), _ptr(v_new),
                                          _stream(stream)))


def rkv_compact_kt_fp8(dims, k, v, cap, keep_idx, keep_ld, B1, k_scale, v_scale, k_out, v_out, out_cap, blk, kt,
                       nblk_cap, stream=None):
    """Compaction into e4m3 code caches (uint8) with the KT cache of the key codes."""
    _check(lib().rkv_compact_kt_fp8(_dims(dims), _ptr(k), _ptr(v), cap, _ptr(keep_idx), keep_ld, B1, _ptr(k_scale),
                                    _ptr(v_scale), _ptr(k_out), _ptr(v_out), out_cap, blk, _ptr(kt), nblk_cap,
                                    _stream(stream)))


def rkv_hsa_decode_fp8(dims, q, k, v, cap, n, k_scale, v_scale, kt, nblk_cap, blk, k1, k2, scale, out,
                       sel_blocks=None, sel_channels=None, k_new=None, v_new=None, stream=None):
    """HSA decode step over e4m3 code caches."""
    _check(lib().rkv_hsa_decode_fp8(_dims(dims), _ptr(q), _ptr(k), _ptr(v), cap, n, _ptr(k_scale), _ptr(v_scale),
                                    _ptr(kt), nblk_cap, blk, k1, k2, scale, _ptr(out), _ptr(sel_blocks),
                                    _ptr(sel_channels), _ptr(k_new), _ptr(v_new), _stream(stream)))


def rkv_debug_set_wait(limit_ns: int, extra_bytes: int) -> None:
    _check(lib().rkv_debug_set_wait(limit_ns, extra_bytes))


def rkv_read_device_flags() -> int:
    f = ctypes.c_uint32()
    _check(lib().rkv_read_device_flags(ctypes.byref(f)))
    return f.value
