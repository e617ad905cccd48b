"""The allocation-free patch embedding, jepa_patch_embed_static.

It exists for callers that cannot allocate device memory themselves (a host
application or inference server that owns all device memory through its own
pool, or a latency-critical loop that cannot afford cudaMalloc's device-wide
synchronisation or its failure under memory pressure).  Its output must match
what the handle-based jepa_encoder_embed computes from the same clip and
weights, on consecutive calls that reuse the shared static scratch.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import synth
from parity import assert_close_16bit

pytestmark = pytest.mark.gpu


def _call(lib, clip, weight, bias, out, status, embed_dim, dtype_code):
    B, T, H, W, _ = clip.shape
    return lib.jepa_patch_embed_static(C.c_void_p(clip.data_ptr()), C.c_void_p(weight.data_ptr()),
                                       C.c_void_p(bias.data_ptr()), C.c_void_p(out.data_ptr()),
                                       C.c_void_p(status.data_ptr()), B, T, H, W, embed_dim, dtype_code,
                                       C.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_patch_embed_matches_encoder_embed():
    import video_vit_encoder_gb300 as jg
    from video_vit_encoder_gb300._lib import DT_BF16, ERR_ARG, OK
    lib = jg.load()
    cfg = synth.CONFIGS["c3"].with_(n_layer=1)          # ViT-L patch embedding, bf16
    w = synth.encoder_weights(cfg)
    enc = jg.Encoder(cfg, w)
    weight = torch.from_numpy(w["patch_embed.weight"]).to(torch.bfloat16).cuda()
    bias = torch.from_numpy(w["patch_embed.bias"]).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # two calls in a row with different shapes share the static scratch;
    # the first fills it to its 4096-row maximum
    shapes = [(2, 16, 256, 256), (3, 4, 96, 160)]
    for i, (B, T, H, W) in enumerate(shapes):
        c = cfg.with_(batch=B, n_frames=T, height=H, width=W)
        clip = torch.from_numpy(synth.clip_u8(c, first_clip=10 * i)).cuda()
        ref = enc.embed(clip)
        out = torch.full_like(ref, float("nan"))
        assert _call(lib, clip, weight, bias, out, status, cfg.embed_dim, DT_BF16) == OK, lib.jepa_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close_16bit(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64), f"call {i}")
    # a size beyond the static maximum is refused before anything runs
    big = torch.zeros((3, 16, 256, 256, 3), dtype=torch.uint8, device="cuda")
    out = torch.empty((3 * 2048, cfg.embed_dim), dtype=torch.float32, device="cuda")
    assert _call(lib, big, weight, bias, out, status, cfg.embed_dim, DT_BF16) == ERR_ARG
    assert b"4096" in lib.jepa_last_error()
    enc.close()
