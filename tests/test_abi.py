"""The C ABI on the host: the library builds, loads and exports every entry
point the header declares; blob and argument validation (no GPU needed)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "jepa_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from video_vit_encoder_gb300 import build
    build.build()
    import video_vit_encoder_gb300 as jg
    return jg.load()


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^JEPA_API [^(]*?\b(jepa_\w+)\(", txt, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 20
    from video_vit_encoder_gb300._lib import SIGNATURES
    for n in names:
        assert hasattr(lib, n), n
        assert n in SIGNATURES, f"binding lacks {n}"
    assert lib.jepa_abi_version() == 6


def _blob(cfg):
    import video_vit_encoder_gb300 as jg
    w = synth.encoder_weights(cfg)
    return jg.pack_blob(jg.encoder_tensor_order(cfg), w, cfg.dtype)


def test_blob_roundtrip_and_faults(lib):
    import video_vit_encoder_gb300 as jg
    from video_vit_encoder_gb300._lib import JepaError, ERR_BLOB, ERR_ARG, ERR_UNSUPPORTED
    cfg = synth.CONFIGS["block-f32-4f128"].with_(n_layer=2, dtype="bf16")
    blob = _blob(cfg)
    jg.blob_check(cfg, blob)                       # valid
    with pytest.raises(JepaError) as e:            # truncated
        jg.blob_check(cfg, blob[: len(blob) - 100])
    assert e.value.status == ERR_BLOB
    bad = bytearray(blob); bad[0] = ord("X")       # wrong magic
    with pytest.raises(JepaError) as e:
        jg.blob_check(cfg, bytes(bad))
    assert e.value.status == ERR_BLOB
    with pytest.raises(JepaError) as e:            # parameters that do not match the blob
        jg.blob_check(cfg.with_(n_layer=3), blob)
    assert e.value.status == ERR_BLOB
    with pytest.raises(JepaError) as e:            # dtype mismatch
        jg.blob_check(cfg.with_(dtype="f16"), blob)
    assert e.value.status == ERR_BLOB
    with pytest.raises(JepaError) as e:            # unsupported head dim
        jg.blob_check(cfg.with_(n_head=6), blob)
    assert e.value.status == ERR_UNSUPPORTED
    with pytest.raises(JepaError) as e:            # bad hierarchical taps
        jg.blob_check(cfg.with_(hier_layers=(1, 1)), blob)
    assert e.value.status == ERR_ARG


def test_blob_with_image_path(lib):
    """The 2.1 image-path tensors follow the hierarchical norms; a blob without
    them does not satisfy params that ask for them, and the other way round."""
    import video_vit_encoder_gb300 as jg
    from video_vit_encoder_gb300._lib import JepaError, ERR_BLOB
    cfg = synth.CONFIGS["img384"].with_(n_layer=2, hier_layers=(1,))
    blob = _blob(cfg)
    jg.blob_check(cfg, blob)
    assert jg.encoder_tensor_order(cfg)[-3:] == [("patch_embed_img.weight", True), ("patch_embed_img.bias", False),
                                                 ("mod_embed_img", False)]
    with pytest.raises(JepaError) as e:
        jg.blob_check(cfg.with_(has_image_path=False), blob)
    assert e.value.status == ERR_BLOB
    with pytest.raises(JepaError) as e:
        jg.blob_check(cfg, _blob(cfg.with_(has_image_path=False)))
    assert e.value.status == ERR_BLOB


def test_blob_layout_is_aligned(lib):
    import struct
    cfg = synth.CONFIGS["block-f32-4f128"].with_(dtype="f16")
    blob = _blob(cfg)
    assert blob[:8] == b"JEPAGB3\0"
    ver, n = struct.unpack_from("<II", blob, 8)
    assert ver == 1 and n == 2 + 12 + 2
    for i in range(n):
        off, nb, dt, nd, d0, d1 = struct.unpack_from("<QQIIII", blob, 24 + 32 * i)
        assert off % 256 == 0 and off + nb <= len(blob)
    # first tensor is the patch embedding in fp16, matching the generator's values
    off, nb, dt, nd, d0, d1 = struct.unpack_from("<QQIIII", blob, 24)
    assert (dt, nd, d0, d1) == (1, 2, 768, 1536)
    w = synth.encoder_weights(cfg)["patch_embed.weight"]
    got = np.frombuffer(blob, np.float16, count=d0 * d1, offset=off).astype(np.float32).reshape(d0, d1)
    np.testing.assert_array_equal(got, w)


def test_argument_errors_without_gpu(lib):
    # Host-side validation happens before any CUDA call.
    from video_vit_encoder_gb300._lib import ERR_ARG, ERR_UNSUPPORTED
    assert lib.jepa_layernorm_f32(None, None, None, None, 4, 128, 1e-6, None) == ERR_ARG
    assert lib.jepa_layernorm_f32(None, None, None, None, 0, 128, 1e-6, None) == 0
    assert lib.jepa_rope3d_f32(C.c_void_p(16), 1, 10, 1, 48, 1, 2, 5, 0, 0, 16, 1e4, None) == ERR_UNSUPPORTED
    assert lib.jepa_rope3d_f32(C.c_void_p(16), 1, 11, 1, 64, 1, 2, 5, 0, 0, 16, 1e4, None) == ERR_ARG
    assert lib.jepa_linear(C.c_void_p(16), C.c_void_p(16), None, C.c_void_p(16), 8, 32, 40, 2, 0, None) == ERR_ARG
    # tensor-core widths are whole 128-column tiles
    assert lib.jepa_linear(C.c_void_p(16), C.c_void_p(16), None, C.c_void_p(16), 8, 96, 64, 2, 0, None) == ERR_ARG
    assert lib.jepa_attention(C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), 2, 1, 1, 100, 64,
                              100, 0.125, None) == ERR_ARG          # ldv not a multiple of 8
    v = C.c_void_p(16)
    # jepa_qkv_rope: head_dim 48 unsupported; a grid that does not hold the
    # tokens without ids; ldv not a multiple of 8; interpolation on a 1-wide grid
    assert lib.jepa_qkv_rope(v, v, None, v, v, v, 2, 1, 64, 384, 8, 64, 1, 8, 8, 0, 0, 16, 1e4, None,
                             None) == ERR_UNSUPPORTED
    assert lib.jepa_qkv_rope(v, v, None, v, v, v, 2, 1, 65, 256, 4, 72, 1, 8, 8, 0, 0, 16, 1e4, None, None) == ERR_ARG
    assert lib.jepa_qkv_rope(v, v, None, v, v, v, 2, 1, 64, 256, 4, 68, 1, 8, 8, 0, 0, 16, 1e4, None, None) == ERR_ARG
    assert lib.jepa_qkv_rope(v, v, None, v, v, v, 2, 1, 64, 256, 4, 64, 4, 16, 1, 0, 1, 16, 1e4, None, None) == ERR_ARG
    assert lib.jepa_qkv_rope(None, v, None, v, v, v, 2, 1, 64, 256, 4, 64, 1, 8, 8, 0, 0, 16, 1e4, None,
                             None) == ERR_ARG
    assert lib.jepa_encoder_sync(None, None) == ERR_ARG
    assert lib.jepa_encode_host_async(None, C.c_void_p(16), 0, 1, 2, 16, 16, C.c_void_p(16), None, None) == ERR_ARG
    assert b"NULL" in lib.jepa_last_error()


def test_predictor21_blob(lib):
    """The 2.1 predictor's modality vectors and context projection follow its
    projection in the blob; params must ask for exactly what the blob holds."""
    import video_vit_encoder_gb300 as jg
    from video_vit_encoder_gb300._lib import ERR_BLOB, check
    import dataclasses
    pc = dataclasses.replace(synth.PREDICTOR_21, n_layer=1)
    cfg = synth.CONFIGS["pred21"].with_(predictor=pc)
    pw = synth.predictor_weights(cfg)
    order = jg.predictor_tensor_order(pc)
    assert order[-4:] == [("mod_embed_video", False), ("mod_embed_img", False), ("proj_context.weight", True),
                          ("proj_context.bias", False)]
    blob = jg.pack_blob(order, pw, cfg.dtype)
    p = jg.predictor_params(pc, cfg.dtype)
    check(lib.jepa_predictor_blob_check(blob, len(blob), C.byref(p)))
    for field in ("has_mod_embed", "has_proj_context"):
        q = jg.predictor_params(pc, cfg.dtype)
        setattr(q, field, 0)
        assert lib.jepa_predictor_blob_check(blob, len(blob), C.byref(q)) == ERR_BLOB


def test_head_blob(lib):
    """The attentive-pool head's blob: the learned query, the pool blocks, the
    cross-attention block and the classifier, in the header's order; params
    must match it, and only head_dim 64 is supported."""
    import video_vit_encoder_gb300 as jg
    from video_vit_encoder_gb300._lib import ERR_BLOB, ERR_UNSUPPORTED, check
    hc = synth.HeadConfig(embed_dim=256, n_layer=2, n_head=4, ffn_dim=512, n_classes=11)
    w = synth.head_weights(hc, 0, "bf16")
    order = jg.head_tensor_order(hc)
    assert [n for n, _ in order] == [n for n, _, _ in synth.tensor_names_head(hc)]
    blob = jg.pack_blob(order, w, "bf16")
    p = jg.head_params(hc, "bf16")
    check(lib.jepa_head_blob_check(blob, len(blob), C.byref(p)))
    p.n_classes = 12
    assert lib.jepa_head_blob_check(blob, len(blob), C.byref(p)) == ERR_BLOB
    p = jg.head_params(hc, "bf16")
    p.n_head = 8   # head_dim 32
    assert lib.jepa_head_blob_check(blob, len(blob), C.byref(p)) == ERR_UNSUPPORTED
