"""ctypes declarations of libpkv.so (include/pkv.h)."""
from __future__ import annotations

import ctypes
import pathlib

LIB_PATH = pathlib.Path(__file__).resolve().parent / "lib" / "libpkv.so"

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_f = ctypes.c_float
_pi32 = ctypes.POINTER(ctypes.c_int32)
_pi64 = ctypes.POINTER(ctypes.c_int64)
_pint = ctypes.POINTER(ctypes.c_int)

# name: (restype, argtypes)
SIGNATURES = {
    "kv_reshape_and_cache": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p]),
    "paged_attention_decode": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p,
                                    _sz, _i, _p]),
    "paged_attention_decode_write": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f,
                                          _i, _p, _sz, _i, _p]),
    "paged_attention_decode_noalloc": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i,
                                            _i, _p]),
    "paged_attention_prefill": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _p, _sz,
                                     _i, _p]),
    "paged_attention_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "paged_attention_workspace_init": (_i, [_p, _sz, _p]),
    "paged_attention_partition_size": (_i, [_i, _i, _i, _i, _i, _i]),
    "copy_blocks": (_i, [_p, _p, _i, _i64, _i, _p]),
    "swap_blocks": (_i, [_p, _p, _p, _i, _i64, _i, _i, _p]),
    "pkv_validate_copy_pairs": (_i, [_p, _i, _i]),
    "pkv_check": (_i, [_p]),
    "pkv_last_error_string": (ctypes.c_char_p, []),
    "pkv_launch_count": (ctypes.c_uint64, []),
    "pkv_version": (_i, []),
    "pkv_selftest_wait_timeout": (_i, [ctypes.c_longlong, _p]),
    "pkv_alloc_create": (_i, [_i, _i, _p, ctypes.POINTER(_p)]),
    "pkv_alloc_destroy": (None, [_p]),
    "pkv_seq_new": (_i, [_p, _i64, _pi32]),
    "pkv_seq_fork": (_i, [_p, ctypes.c_int32, _pi32]),
    "pkv_seq_append": (_i, [_p, ctypes.c_int32, _pi64, _pi32, _pi32]),
    "pkv_seq_append_batch": (_i, [_p, _p, _i, _p, _p, _pint]),
    "pkv_seq_free": (_i, [_p, ctypes.c_int32]),
    "pkv_seq_len": (_i, [_p, ctypes.c_int32, _pi64]),
    "pkv_seq_block_table": (_i, [_p, ctypes.c_int32, _p, _i, _pint]),
    "pkv_build_block_tables": (_i, [_p, _p, _i, _p, _i, _p]),
    "pkv_block_ref": (_i, [_p, ctypes.c_int32]),
    "pkv_num_free": (_i, [_p]),
    "pkv_free_list": (_i, [_p, _p, _i, _pint]),
    "pkv_move_group": (_i, [_p, _p, _p, _i, _p, _p, _i, _pint]),
    "pkv_beam_step": (_i, [_p, _p, _i, _p, _i, _p, _p, _p, _pint]),
    "pkv_blocks_in_use": (_i, [_p]),
}

STATUS = {0: "PKV_OK", 1: "PKV_EINVAL", 2: "PKV_ENOMEM", 3: "PKV_EINDEX", 4: "PKV_ECUDA", 5: "PKV_ETIMEOUT"}

_lib = None


def load() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no
    fallback path."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_cache_139_gb300.build` (there is no fallback)")
        L = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib
