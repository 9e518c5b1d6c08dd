"""ctypes view of the C ABI declared in include/pg_grouped_attn.h (argument marshalling only)."""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpg_gb300.so")

PG_OK, PG_ERR_INVALID_ARG, PG_ERR_UNSUPPORTED, PG_ERR_CUDA, PG_ERR_TIMEOUT, PG_ERR_DEVICE = range(6)
PG_F32, PG_BF16 = 0, 1
PG_FLAG_SIMT = 1
PG_FLAG_RESPONSES_ONLY = 2
PG_FLAG_DETERMINISTIC = 4
PG_FLAG_KEEP_ROTATED = 8
PG_FLAG_PRE_ROTATED = 16


class PgLayout(C.Structure):
    _fields_ = [
        ("num_groups", C.c_int64),
        ("num_segments", C.c_int64),
        ("total_tokens", C.c_int64),
        ("max_position", C.c_int64),
        ("pairs", C.c_int64),
        ("n_tiles", C.c_int64 * 6),
        ("off_tiles", C.c_int64 * 6),
        ("off_tokens", C.c_int64),
        ("table_bytes", C.c_int64),
        ("position_ids", C.c_void_p),
        ("tables", C.c_void_p),
        ("max_response_rows", C.c_int64),
        ("n_pad_rows", C.c_int64),
        ("off_pad_rows", C.c_int64),
        ("max_depth", C.c_int64),
        ("n_intervals", C.c_int64),
        ("off_intervals", C.c_int64),
    ]


class PgOpts(C.Structure):
    _fields_ = [
        ("softmax_scale", C.c_float),
        ("rope_theta", C.c_float),
        ("flags", C.c_uint32),
        ("debug", C.c_uint32),
    ]


class PgProfile(C.Structure):
    _fields_ = [
        ("kernel", C.c_int32),
        ("reserved", C.c_int32),
        ("ev_begin", C.c_void_p),
        ("ev_end", C.c_void_p),
        ("launches", C.c_int64),
    ]


(PG_KERNEL_NONE, PG_KERNEL_ROPE, PG_KERNEL_ATTN_FWD, PG_KERNEL_BWD_PREPROCESS, PG_KERNEL_BWD_DKDV,
 PG_KERNEL_BWD_DQ, PG_KERNEL_ROPE_BWD, PG_KERNEL_GEMM, PG_KERNEL_LAYER,
 PG_KERNEL_SCORE_COMBINE, PG_KERNEL_PAD_FILL) = range(11)

I32P = C.POINTER(C.c_int32)
I64P = C.POINTER(C.c_int64)
VP = C.c_void_p

# name -> (restype, argtypes); every symbol the header declares.
SIGNATURES = {
    "pg_pack_size": (C.c_int, [C.c_int32, I32P, I32P, I32P, I64P, I64P]),
    "pg_pack_host": (C.c_int, [C.c_int32, I32P, I32P, I32P, I32P, VP, C.c_int64,
                               C.POINTER(PgLayout)]),
    "pg_pack": (C.c_int, [C.c_int32, I32P, I32P, I32P, VP, VP, C.c_int64, C.POINTER(PgLayout),
                          VP]),
    "pg_pack_tree_size": (C.c_int, [C.c_int32, I32P, I32P, I64P, I64P]),
    "pg_pack_tree_host": (C.c_int, [C.c_int32, I32P, I32P, I32P, VP, C.c_int64,
                                    C.POINTER(PgLayout)]),
    "pg_pack_tree": (C.c_int, [C.c_int32, I32P, I32P, VP, VP, C.c_int64, C.POINTER(PgLayout),
                               VP]),
    "pg_pack_padded_size": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, I32P, I64P,
                                      I64P]),
    "pg_pack_padded_host": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, I32P, I32P, VP,
                                      C.c_int64, C.POINTER(PgLayout)]),
    "pg_pack_padded": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, I32P, VP, VP,
                                 C.c_int64, C.POINTER(PgLayout), VP]),
    "pg_workspace_size": (C.c_int, [C.POINTER(PgLayout), C.c_int, C.c_int32, C.c_int32,
                                    C.c_int32, C.POINTER(PgOpts), C.c_int32,
                                    C.POINTER(C.c_size_t)]),
    "pg_grouped_attn_fwd": (C.c_int, [C.POINTER(PgLayout), C.c_int, C.c_int32, C.c_int32,
                                      C.c_int32, VP, VP, VP, VP, VP, C.POINTER(PgOpts), VP,
                                      C.c_size_t, VP]),
    "pg_grouped_attn_bwd": (C.c_int, [C.POINTER(PgLayout), C.c_int, C.c_int32, C.c_int32,
                                      C.c_int32, VP, VP, VP, VP, VP, VP, VP, VP, VP,
                                      C.POINTER(PgOpts), VP, C.c_size_t, VP]),
    "pg_grouped_attn_fwd_noalloc": (C.c_int, [C.POINTER(PgLayout), C.c_int, C.c_int32,
                                              C.c_int32, C.c_int32, VP, VP, VP, VP, VP,
                                              C.POINTER(PgOpts), VP]),
    "pg_rope_table": (C.c_int, [C.POINTER(PgLayout), C.c_int, C.c_int32, C.c_int32, C.c_int32,
                                C.POINTER(PgOpts), VP, C.c_size_t, C.POINTER(VP), VP]),
    "pg_set_profile": (C.c_int, [C.POINTER(PgProfile)]),
    "pg_gemm_bf16": (C.c_int, [C.c_int64, C.c_int64, C.c_int64, VP, C.c_int32, C.c_int64, VP,
                               C.c_int32, C.c_int64, VP, C.c_int, C.c_int64, C.c_int32, VP]),
    "pg_gemm_bf16_rope": (C.c_int, [C.c_int64, C.c_int64, C.c_int64, VP, C.c_int64, VP, C.c_int64,
                                    VP, C.c_int64, C.c_int32, VP, C.c_int64, VP]),
    "pg_rmsnorm_fwd": (C.c_int, [C.c_int64, C.c_int32, VP, VP, VP, C.c_float, VP, VP, VP, VP]),
    "pg_rmsnorm_bwd_workspace": (C.c_size_t, [C.c_int64, C.c_int32]),
    "pg_rmsnorm_bwd": (C.c_int, [C.c_int64, C.c_int32, VP, VP, VP, VP, C.c_int, VP, VP, C.c_int,
                                 VP, VP, C.c_size_t, VP]),
    "pg_swiglu_fwd": (C.c_int, [C.c_int64, C.c_int32, VP, VP, VP]),
    "pg_swiglu_bwd": (C.c_int, [C.c_int64, C.c_int32, VP, VP, VP, VP]),
    "pg_device_status": (C.c_int, [C.c_int32]),
    "pg_status_string": (C.c_char_p, [C.c_int]),
    "pg_last_error_message": (C.c_char_p, []),
}

_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built (there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m shared_prefix_grouped_gb300.build` "
                "(the grouped-attention ops have no non-CUDA implementation)")
        handle = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class PgError(RuntimeError):
    def __init__(self, where: str, status: int):
        L = lib()
        msg = L.pg_last_error_message().decode()
        super().__init__(f"{where}: {L.pg_status_string(status).decode()} ({status}): {msg}")
        self.status = status


def check(where: str, status: int) -> None:
    if status != PG_OK:
        raise PgError(where, status)


def int_array(xs):
    arr = (C.c_int32 * max(len(xs), 1))(*[int(x) for x in xs])
    return arr
