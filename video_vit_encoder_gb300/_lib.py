"""ctypes declarations of the C ABI in include/jepa_gb300.h.

The library is required: importing this module without a built
``libjepa_gb300.so`` raises at first use, and nothing falls back to another
implementation.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libjepa_gb300.so")

OK, ERR_ARG, ERR_BLOB, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_DEVICE_TIMEOUT = range(7)
STATUS_NAMES = {0: "OK", 1: "ERR_ARG", 2: "ERR_BLOB", 3: "ERR_UNSUPPORTED", 4: "ERR_CUDA", 5: "ERR_OOM",
                6: "ERR_DEVICE_TIMEOUT"}
DT_F32, DT_F16, DT_BF16 = 0, 1, 2
CLIP_U8_THWC, CLIP_F32_CTHW = 0, 1
MODALITY_VIDEO, MODALITY_IMAGE, MODALITY_AUTO = 0, 1, 2


class JepaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


ABI_VERSION = 6  # JEPA_ABI_VERSION of include/jepa_gb300.h


class EncoderParams(C.Structure):
    _fields_ = [("embed_dim", C.c_int), ("n_layer", C.c_int), ("n_head", C.c_int), ("ffn_dim", C.c_int),
                ("patch", C.c_int), ("tubelet", C.c_int), ("ln_eps", C.c_float), ("rope_theta", C.c_float),
                ("rope_layout", C.c_int), ("rope_interpolate", C.c_int), ("rope_ref_grid", C.c_int),
                ("n_hier", C.c_int), ("hier_layers", C.c_int * 4), ("has_mod_embed", C.c_int), ("dtype", C.c_int),
                ("has_image_path", C.c_int)]


class PredictorParams(C.Structure):
    _fields_ = [("embed_dim", C.c_int), ("n_layer", C.c_int), ("n_head", C.c_int), ("ffn_dim", C.c_int),
                ("in_dim", C.c_int), ("out_dim", C.c_int), ("n_mask_tokens", C.c_int), ("mask_index", C.c_int),
                ("ln_eps", C.c_float), ("rope_theta", C.c_float), ("rope_layout", C.c_int), ("dtype", C.c_int),
                ("has_mod_embed", C.c_int), ("has_proj_context", C.c_int)]


class HeadParams(C.Structure):
    _fields_ = [("embed_dim", C.c_int), ("n_layer", C.c_int), ("n_head", C.c_int), ("ffn_dim", C.c_int),
                ("n_classes", C.c_int), ("ln_eps", C.c_float), ("dtype", C.c_int)]


VP, I, F, ST, U64 = C.c_void_p, C.c_int, C.c_float, C.c_int, C.c_size_t

# name: (restype, argtypes)
SIGNATURES = {
    "jepa_blob_check": (ST, [VP, U64, C.POINTER(EncoderParams)]),
    "jepa_predictor_blob_check": (ST, [VP, U64, C.POINTER(PredictorParams)]),
    "jepa_encoder_create": (ST, [VP, U64, C.POINTER(EncoderParams), I, C.POINTER(VP)]),
    "jepa_encoder_destroy": (None, [VP]),
    "jepa_encode_workspace_bytes": (U64, [VP, I, I, I, I]),
    "jepa_encode": (ST, [VP, VP, I, I, I, I, I, VP, VP, VP, VP]),
    "jepa_encode_host": (ST, [VP, VP, I, I, I, I, I, VP, VP, VP]),
    "jepa_encode_host_async": (ST, [VP, VP, I, I, I, I, I, VP, VP, VP]),
    "jepa_encoder_embed": (ST, [VP, VP, I, I, I, I, I, VP, VP]),
    "jepa_encoder_blocks": (ST, [VP, VP, I, I, I, I, I, I, VP]),
    "jepa_encoder_sync": (ST, [VP, VP]),
    "jepa_encoder_set_profiling": (ST, [VP, I]),
    "jepa_encoder_profile": (ST, [VP, C.POINTER(C.c_double), C.POINTER(C.c_longlong), I]),
    "jepa_predictor_create": (ST, [VP, U64, C.POINTER(PredictorParams), I, C.POINTER(VP)]),
    "jepa_predictor_destroy": (None, [VP]),
    "jepa_predict": (ST, [VP, VP, I, VP, I, VP, I, I, I, I, VP, VP]),
    "jepa_encode_masked": (ST, [VP, VP, I, I, I, I, I, VP, I, VP, VP, VP, VP]),
    "jepa_encoder_set_graphs": (ST, [VP, I]),
    "jepa_predictor_set_graphs": (ST, [VP, I]),
    "jepa_predict_ex": (ST, [VP, VP, I, VP, I, VP, I, I, I, I, I, VP, VP, VP]),
    "jepa_predictor_sync": (ST, [VP, VP]),
    "jepa_layernorm_f32": (ST, [VP, VP, VP, VP, I, I, F, VP]),
    "jepa_rope3d_f32": (ST, [VP, I, I, I, I, I, I, I, I, I, I, F, VP]),
    "jepa_attention": (ST, [VP, VP, VP, VP, I, I, I, I, I, I, F, VP]),
    "jepa_linear": (ST, [VP, VP, VP, VP, I, I, I, I, I, VP]),
    "jepa_qkv_rope": (ST, [VP, VP, VP, VP, VP, VP, I, I, I, I, I, I, I, I, I, I, I, I, F, VP, VP]),
    "jepa_ops_sync": (ST, [VP]),
    "jepa_selftest_wait_timeout": (ST, [I, VP]),
    "jepa_patch_embed_static": (ST, [VP, VP, VP, VP, VP, I, I, I, I, I, I, VP]),
    "jepa_head_blob_check": (ST, [VP, U64, C.POINTER(HeadParams)]),
    "jepa_head_create": (ST, [VP, U64, C.POINTER(HeadParams), I, C.POINTER(VP)]),
    "jepa_head_destroy": (None, [VP]),
    "jepa_head_forward": (ST, [VP, VP, I, I, VP, VP, VP]),
    "jepa_head_sync": (ST, [VP, VP]),
    "jepa_head_set_graphs": (ST, [VP, I]),
    "jepa_last_error": (C.c_char_p, []),
    "jepa_abi_version": (C.c_int, []),
}

_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> C.CDLL:
    """Loads the library (once) and declares every entry point."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = C.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if lib.jepa_abi_version() != ABI_VERSION:
            raise RuntimeError(f"{p} has ABI version {lib.jepa_abi_version()}, this binding needs {ABI_VERSION}: rebuild it")
        _lib = lib
        return lib


def check(status: int) -> None:
    if status != OK:
        raise JepaError(status, load().jepa_last_error().decode())
