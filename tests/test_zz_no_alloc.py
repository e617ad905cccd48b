"""The allocation-free patch embedding, jepa_patch_embed_static.

It exists for callers that cannot allocate device memory themselves (a host
application or inference server that owns all device memory through its own
pool, or a latency-critical loop that cannot afford cudaMalloc's device-wide
synchronisation or its failure under memory pressure).  Its output must match
the oracle's patch embedding of the same clips, and what the handle-based
jepa_encoder_embed computes, on consecutive calls that reuse the shared static
scratch; the optional bias and status arguments may be NULL.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_close_16bit

pytestmark = pytest.mark.gpu

TD = {"bf16": torch.bfloat16, "f16": torch.float16}


def _call(lib, clip, weight, bias, out, status, embed_dim, dtype_code):
    B, T, H, W, _ = clip.shape
    ptr = lambda t: None if t is None else C.c_void_p(t.data_ptr())  # noqa: E731
    return lib.jepa_patch_embed_static(ptr(clip), ptr(weight), ptr(bias), ptr(out), ptr(status), B, T, H, W,
                                       embed_dim, dtype_code, C.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_static_patch_embed_matches_oracle_and_encoder_embed(dtype):
    import video_vit_encoder_gb300 as jg
    from video_vit_encoder_gb300._lib import DT_BF16, DT_F16, ERR_ARG, OK
    code = {"bf16": DT_BF16, "f16": DT_F16}[dtype]
    lib = jg.load()
    cfg = synth.CONFIGS["vitl16-16f256"].with_(n_layer=1, dtype=dtype)     # ViT-L patch embedding
    w = synth.encoder_weights(cfg)
    bias = np.random.default_rng(3).standard_normal(cfg.embed_dim).astype(np.float32) * 0.5
    w_b = dict(w, **{"patch_embed.bias": bias})
    weight = torch.from_numpy(w["patch_embed.weight"]).to(TD[dtype]).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # Two calls in a row share the static scratch: the first fills it to its
    # 4096-row maximum with a bias and a status word, the second (a smaller,
    # ragged shape) passes NULL for both, i.e. no bias and the library's own
    # status word.  Each is checked on every token against the oracle and
    # against jepa_encoder_embed of a handle holding the same bias.
    calls = [((2, 16, 256, 256), bias, w_b), ((3, 4, 96, 160), None, w)]
    for i, ((B, T, H, W), b, wts) in enumerate(calls):
        c = cfg.with_(batch=B, n_frames=T, height=H, width=W)
        clip_np = synth.clip_u8(c, first_clip=10 * i)
        clip = torch.from_numpy(clip_np).cuda()
        n = synth.tokens_per_clip(c)
        out = torch.full((B * n, cfg.embed_dim), float("nan"), dtype=torch.float32, device="cuda")
        st = status if b is not None else None
        db = torch.from_numpy(b).cuda() if b is not None else None
        assert _call(lib, clip, weight, db, out, st, cfg.embed_dim, code) == OK, lib.jepa_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.view(B, n, cfg.embed_dim).cpu().numpy()
        for bb in range(B):
            ref = oracle.encoder_embed(c, wts, clip_np[bb])
            assert_close_16bit(got[bb], ref, f"{dtype} call {i} clip {bb} vs oracle")
        enc = jg.Encoder(c, wts)
        same = enc.embed(clip)
        enc.sync()
        assert_close_16bit(out.cpu().numpy(), same.cpu().numpy().astype(np.float64),
                           f"{dtype} call {i} vs jepa_encoder_embed")
        enc.close()
    # a size beyond the static maximum is refused before anything runs
    big = torch.zeros((3, 16, 256, 256, 3), dtype=torch.uint8, device="cuda")
    out = torch.empty((3 * 2048, cfg.embed_dim), dtype=torch.float32, device="cuda")
    assert _call(lib, big, weight, None, out, status, cfg.embed_dim, code) == ERR_ARG
    assert b"4096" in lib.jepa_last_error()
