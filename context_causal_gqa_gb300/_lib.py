"""ctypes declarations of the C ABI in include/ccg.h (argument marshalling only)."""

import ctypes
import os

from . import build as _build

c_i32, c_i64, c_f32, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class AttnDesc(ctypes.Structure):
    _fields_ = [("batch", c_i32), ("hq", c_i32), ("hkv", c_i32), ("head_dim", c_i32),
                ("causal", c_i32), ("cp", c_i32), ("head_groups", c_i32), ("head_parts", c_i32),
                ("total_tokens", c_i64), ("softmax_scale", c_f32),
                ("q_pitch", c_i64), ("k_pitch", c_i64), ("v_pitch", c_i64), ("do_pitch", c_i64),
                ("max_seqlen", c_i64)]


# name -> (restype, argtypes)
SIGNATURES = {
    "ccg_workspace_size": (c_sz, [ctypes.POINTER(AttnDesc), ctypes.c_int]),
    "ccg_attn_fwd": (ctypes.c_int, [ctypes.POINTER(AttnDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                    c_vp, c_sz, c_vp, c_vp]),
    "ccg_attn_fwd_fused": (ctypes.c_int, [ctypes.POINTER(AttnDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                          c_vp, c_sz, c_vp, c_vp]),
    "ccg_attn_fwd_step": (ctypes.c_int, [ctypes.POINTER(AttnDesc), c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                                         c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "ccg_attn_bwd": (ctypes.c_int, [ctypes.POINTER(AttnDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                    c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "ccg_attn_bwd_noalloc": (ctypes.c_int, [ctypes.POINTER(AttnDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                            c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "ccg_cp_split": (ctypes.c_int, [c_vp, c_vp, c_i32, c_i64, c_i32, c_vp, c_vp, c_vp]),
    "ccg_cp_lse_merge": (ctypes.c_int, [c_i32, ctypes.POINTER(c_vp), ctypes.POINTER(c_vp), c_i64, c_i32,
                                        c_vp, c_vp, c_vp]),
    "ccg_bwd_dot": (ctypes.c_int, [c_vp, c_vp, c_i64, c_i32, c_vp, c_vp]),
    "ccg_thd_pack": (ctypes.c_int, [c_vp, c_vp, c_i32, c_i64, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "ccg_thd_unpack": (ctypes.c_int, [c_vp, c_vp, c_i32, c_i64, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "ccg_get_status": (ctypes.c_int, [c_vp, c_vp]),
    "ccg_selftest_bounded_wait": (ctypes.c_int, [c_vp, ctypes.c_uint32, c_vp]),
    "ccg_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "ccg_last_launch_count": (c_i32, []),
    "ccg_profile_begin": (ctypes.c_int, [c_i32]),
    "ccg_profile_end": (ctypes.c_int, []),
    "ccg_profile_count": (c_i32, []),
    "ccg_profile_get": (ctypes.c_int, [c_i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(c_f32)]),
}

_LIB = None


def lib_path():
    return _build.LIB


def load(build_if_missing=False):
    """Load libccg.so; raises if it is missing (there is no fallback)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libccg is not built ({path}); run __graft_entry__.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib
