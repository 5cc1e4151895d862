"""Loads libcc.so (built in-tree by ``causal_convolution_gb300.build``) and
declares the C signatures of include/cc.h and include/cc_debug.h.

There is no fallback: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libcc.so")

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_Z = ctypes.c_size_t
_F = ctypes.c_float

# name -> (restype, argtypes); mirrors include/cc.h and include/cc_debug.h
SIGNATURES = {
    "cc_last_error": (ctypes.c_char_p, []),
    "cc_version": (_I, []),
    "cc_check_device": (_I, [_P]),
    "cc_conv3d_prepare": (_I, [_P, _P, _I, _I, _P]),
    "cc_conv3d_causal": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "cc_resample_prepare": (_I, [_P, _P, _I, _I, _P]),
    "cc_resample_workspace_bytes": (_Z, [_I, _I, _I, _I, _I]),
    "cc_resample_phase_conv": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "cc_resample_interleave": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "cc_resample_up2": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "cc_resample_prepare_temporal": (_I, [_P, _P, _I, _I, _P]),
    "cc_resample_up2_fused": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "cc_attn_ld": (_L, [_I]),
    "cc_attn_workspace_bytes": (_Z, [_I, _I]),
    "cc_attn_scores": (_I, [_P, _P, _P, _I, _I, _I, _L, _L, _L, _P]),
    "cc_attn_softmax": (_I, [_P, _P, _I, _I, _L, _L, _F, _P]),
    "cc_attn_pv": (_I, [_P, _P, _P, _I, _I, _I, _L, _L, _L, _P]),
    "cc_attn_frame": (_I, [_P, _P, _P, _P, _I, _I, _I, _L, _L, _L, _L, _F, _P, _Z, _P]),
    "cc_attn_exp_key_tiles": (_I, [_I]),
    "cc_attn_exp_workspace_bytes": (_Z, [_I, _I]),
    "cc_attn_scores_exp": (_I, [_P, _P, _P, _P, _I, _I, _I, _L, _L, _L, _F, _P]),
    "cc_attn_exp_rescale": (_I, [_P, _P, _I, _I, _L, _P]),
    "cc_attn_pv_exp": (_I, [_P, _P, _P, _P, _I, _I, _I, _L, _L, _L, _P]),
    "cc_attn_frame_exp": (_I, [_P, _P, _P, _P, _I, _I, _I, _L, _L, _L, _L, _F, _P, _Z, _P]),
    "cc_attn_scores_stats": (_I, [_P, _P, _P, _I, _I, _I, _L, _L, _F, _P]),
    "cc_attn_fused_workspace_bytes": (_Z, [_I, _I]),
    "cc_attn_frame_fused": (_I, [_P, _P, _P, _P, _I, _I, _I, _L, _L, _L, _L, _F, _P, _Z, _P]),
    "cc_head_prepare": (_I, [_P, _P, _I, _P]),
    "cc_head_workspace_bytes": (_Z, [_I, _I, _I, _I]),
    "cc_head_temporal": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "cc_head_stencil": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "cc_head_out": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "cc_head_out_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "cc_head_out_fused": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "cc_copy_to_host": (_I, [_P, _P, _Z, _I, _P]),
    "cc_debug_im2col_tile": (_I, [_P, _P] + [_I] * 19 + [_P]),
    "cc_debug_wait_timeout": (_I, [_L, _P]),
    "cc_debug_conv_bad_tile_order": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
}

_lib = None


def load() -> ctypes.CDLL:
    """The loaded library with every signature declared (raises if unbuilt)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m causal_convolution_gb300.build` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
