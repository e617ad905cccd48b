"""Pins of the oracle's V-JEPA 2.1 native image path.

"V-JEPA 2 / 2.1 tensor maps and RoPE derivation", §3 (2.1 encoder forward): a
one-frame input is patchified with tubelet 1 by ``patch_embed_img`` (Conv3d
weight ``[D, 3, 1, 16, 16]``), gets ``mod_embed_img``, and runs the same
blocks with the 3-D RoPE (temporal position 0) and the same final norm.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small_image_cfg(**kw):
    base = synth.CONFIGS["img384"].with_(embed_dim=96, n_layer=2, n_head=2, ffn_dim=192, height=64, width=48,
                                         batch=1, hier_layers=(0,))
    return base.with_(**kw)


def test_image_token_count_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "image_tokens.txt")) if l.strip() and not l.startswith("#")]
    assert rows
    for r in rows:
        T, H, W, n = map(int, r[:4])
        cfg = synth.CONFIGS["img384"].with_(n_frames=T, height=H, width=W)
        assert synth.tokens_per_clip(cfg) == n
        assert oracle.encoder_rope(cfg, T, H, W)[0].shape[0] == n


def test_image_patch_embed_is_conv2d():
    """Tubelet 1 is a 2-D convolution with a 16 x 16 kernel and stride 16."""
    rng = np.random.default_rng(0)
    img = rng.integers(0, 256, (1, 64, 48, 3), dtype=np.uint8)
    D = 8
    w = rng.standard_normal((D, 768))
    b = rng.standard_normal(D)
    got = oracle.patch_embed(oracle.normalise_clip(img), w, b, tubelet=1)
    x = torch.from_numpy(oracle.normalise_clip(img)[:, 0])                       # [3, H, W]
    ref = torch.nn.functional.conv2d(x[None], torch.from_numpy(w).reshape(D, 3, 16, 16),
                                     torch.from_numpy(b), stride=16)[0]       # [D, gh, gw]
    ref = ref.permute(1, 2, 0).reshape(-1, D).numpy()                          # tokens h-major, then w
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def _as_video_weights(w):
    """Video weights under which a 2-frame clip repeating the image gives the
    image path's tokens: W_video[:, c, dt, y, x] = W_img[:, c, y, x] / 2 for
    both frames, the image bias and modality vector."""
    v = dict(w)
    D = w["patch_embed_img.weight"].shape[0]
    k = np.asarray(w["patch_embed_img.weight"], np.float64).reshape(D, 3, 1, 16, 16) / 2
    v["patch_embed.weight"] = np.concatenate([k, k], axis=2).reshape(D, 1536)
    v["patch_embed.bias"] = w["patch_embed_img.bias"]
    v["mod_embed_video"] = w["mod_embed_img"]
    return v


def test_image_path_equals_repeated_frame_clip_with_halved_kernel():
    """Summing the two frames of the repeated image with half the kernel each
    is the tubelet-1 embedding, and a 1-tubelet clip has the same RoPE
    positions (t = 0) as the image, so the whole encoder agrees."""
    cfg = _small_image_cfg()
    w = synth.encoder_weights(cfg)
    img = synth.clip_u8(cfg)[0]                                 # [1, H, W, 3]
    a = oracle.encoder_forward(cfg, w, img)
    b = oracle.encoder_forward(cfg, _as_video_weights(w), np.concatenate([img, img], axis=0))
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(a["hier"][0], b["hier"][0], rtol=1e-9, atol=1e-10)


def test_image_path_is_not_the_repeated_frame_video_encoding():
    """The pages call the two encodings valid but not equivalent: with the
    model's own video weights the repeated-frame clip gives other tokens."""
    cfg = _small_image_cfg()
    w = synth.encoder_weights(cfg)
    img = synth.clip_u8(cfg)[0]
    a = oracle.encoder_forward(cfg, w, img)["out"]
    b = oracle.encoder_forward(cfg, w, np.concatenate([img, img], axis=0))["out"]
    assert np.abs(a - b).max() > 0.1


def test_image_modality_vector_is_the_image_one():
    """A change to mod_embed_img moves the image output; one to mod_embed_video
    does not.  (The change is not a constant shift of every feature, which
    the pre-norms would remove.)"""
    cfg = _small_image_cfg()
    w = synth.encoder_weights(cfg)
    img = synth.clip_u8(cfg)[0]
    base = oracle.encoder_forward(cfg, w, img)["out"]
    delta = np.random.default_rng(1).standard_normal(cfg.embed_dim)
    w2 = dict(w, mod_embed_video=np.asarray(w["mod_embed_video"]) + delta)
    np.testing.assert_array_equal(oracle.encoder_forward(cfg, w2, img)["out"], base)
    w3 = dict(w, mod_embed_img=np.asarray(w["mod_embed_img"]) + delta)
    assert np.abs(oracle.encoder_forward(cfg, w3, img)["out"] - base).max() > 1e-3


def test_one_frame_without_image_path_is_not_the_image_path():
    cfg = synth.CONFIGS["vitl16-16f256"]
    assert not oracle.is_image(cfg, 1)
    assert oracle.is_image(synth.CONFIGS["img384"], 1)
    assert not oracle.is_image(synth.CONFIGS["img384"], 2)
