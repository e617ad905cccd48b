"""GB300 (sm_103a) V-JEPA 2 / 2.1 video ViT encoder forward.

The compute lives in ``libjepa_gb300.so`` (hand-written CUDA behind the C ABI
of ``include/jepa_gb300.h``); this package only marshals arguments.
"""
from ._lib import JepaError, LIB_PATH, load  # noqa: F401
from .binding import (  # noqa: F401
    Encoder, Head, Predictor, attention, blob_check, encoder_params, encoder_tensor_order, head_params, head_tensor_order,
    layernorm_f32, linear,
    ops_sync, pack_blob, predictor_params, predictor_tensor_order, qkv_rope, rope3d_f32,
    selftest_wait_timeout,
)
