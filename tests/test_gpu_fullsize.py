"""Full-size workloads on the GPU against the oracle.

At these sizes the oracle checks what it can compute in seconds to a few minutes:
  * vitl16-16f256 (ViT-L/16, 8 clips of 16x256x256, the benchmark's launch) - every
    clip end to end on every token, clip 7 also block by block on sampled rows;
  * img384 (2.1 native image path, 32 images of 384 px) - two images end to
    end on every token, with the hierarchical taps;
  * vitb16-16f384-f16 (2.1 ViT-B/16, fp16, one 16 x 384 x 384 clip) - end to end on every
    token, and block by block on sampled rows;
  * vitl16-64f256-pred, vitb16-64f384 - block by block on sampled rows (each block recomputed by the
    oracle from the GPU's own input residual), the final norm and the
    hierarchical taps on sampled rows, and the predictor end to end.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_close_16bit, metrics

pytestmark = pytest.mark.gpu

_W = {}


def _weights(name):
    if name not in _W:
        _W[name] = synth.encoder_weights(synth.CONFIGS[name])
    return _W[name]


@pytest.fixture(scope="module")
def jg():
    import video_vit_encoder_gb300 as m
    m.load()
    return m


def _sample_rows(n, k, seed):
    rng = np.random.default_rng(seed)
    rows = np.concatenate([[0, n - 1], rng.choice(np.arange(1, n - 1), size=k - 2, replace=False)])
    return np.sort(rows)


def _check_blocks(enc, cfg, w, clip_t, clip_idx, n_rows, seed, stats):
    """Runs the GPU one block at a time; after each block compares sampled rows
    of clip `clip_idx` with the oracle's block applied to the GPU's input."""
    B, T, H, W, _ = clip_t.shape
    N = synth.tokens_per_clip(cfg)
    D = cfg.embed_dim
    x = enc.embed(clip_t)
    enc.sync()
    COS, SIN = oracle.encoder_rope(cfg, T, H, W)
    ref0 = oracle.encoder_embed(cfg, w, clip_t[clip_idx].cpu().numpy())
    rows = _sample_rows(N, n_rows, seed)
    got0 = x.view(B, N, D)[clip_idx].cpu().numpy().astype(np.float64)
    m = metrics(got0[rows], ref0[rows])
    assert m["rel_max"] <= 1e-2 and m["cos_worst"] >= 0.9999, ("patch embed", m)
    for l in range(cfg.n_layer):
        x_in = x.view(B, N, D)[clip_idx].cpu().numpy().astype(np.float64)
        enc.blocks(x, B, T, H, W, l, l + 1)
        enc.sync()
        got = x.view(B, N, D)[clip_idx].cpu().numpy().astype(np.float64)
        ref = oracle.block_forward_rows(x_in, w, l, cfg.n_head, cfg.ln_eps, COS, SIN, rows)
        assert_close_16bit(got[rows], ref, f"{cfg.name} block {l} output")
        md = metrics(got[rows] - x_in[rows], ref - x_in[rows])   # the block's own contribution
        stats.append((l, md))
        assert md["cos_mean"] >= 0.9999 and md["cos_worst"] >= 0.999 and md["rel_max"] <= 2e-2, (l, md)
    return x, rows


def test_vitl16_16f256_all_clips_end_to_end(jg):
    # the benchmark's launch (8 clips in one encode); the oracle runs each clip
    # on its own, every token of every clip compared
    cfg = synth.CONFIGS["vitl16-16f256"]
    w = _weights("vitl16-16f256")
    clip = synth.clip_u8(cfg)
    enc = jg.Encoder(cfg, w)
    res = enc.encode(torch.from_numpy(clip).cuda(), pooled=True)
    enc.sync()
    out = res["out"].cpu().numpy()
    pooled = res["pooled"].cpu().numpy()
    enc.close()
    for b in range(cfg.batch):
        ref = oracle.encoder_forward(cfg, w, clip[b])
        m = assert_close_16bit(out[b], ref["out"], f"vitl16-16f256 clip {b}")
        print(f"vitl16-16f256 clip {b} end to end:", m)
        np.testing.assert_allclose(pooled[b], ref["pooled"], atol=1e-2 * np.abs(ref["pooled"]).max())


def test_vitl16_16f256_clip7_blocks(jg):
    cfg = synth.CONFIGS["vitl16-16f256"]
    w = _weights("vitl16-16f256")
    clip = torch.from_numpy(synth.clip_u8(cfg)).cuda()
    enc = jg.Encoder(cfg, w)
    stats = []
    x, rows = _check_blocks(enc, cfg, w, clip, 7, 48, 3, stats)
    print("vitl16-16f256 clip 7 per-block delta worst cos:", min(s[1]["cos_worst"] for s in stats),
          "max rel:", max(s[1]["rel_max"] for s in stats))
    enc.close()


def test_vitb16_16f384_f16_blocks_and_final(jg):
    cfg = synth.CONFIGS["vitb16-16f384-f16"]
    w = _weights("vitb16-16f384-f16")
    clip = torch.from_numpy(synth.clip_u8(cfg)).cuda()
    enc = jg.Encoder(cfg, w)
    stats = []
    x, rows = _check_blocks(enc, cfg, w, clip, 0, 48, 5, stats)
    out = enc.encode(clip)["out"]
    enc.sync()
    xr = x.cpu().numpy().astype(np.float64)[rows]
    ref = oracle.layer_norm(xr, w["norm.weight"], w["norm.bias"], cfg.ln_eps)
    assert_close_16bit(out[0].cpu().numpy()[rows], ref, "vitb16-16f384-f16 final norm")
    enc.close()


def test_vitb16_16f384_f16_end_to_end(jg):
    """The 2.1 ViT-B/16 fp16 workload (12 layers, interleaved RoPE
    interpolated to the 16-grid, modality vector, one 16 x 384 x 384 clip of
    4608 tokens) end to end on every token against the oracle, so error that
    grows through the 12 layers is compared too."""
    cfg = synth.CONFIGS["vitb16-16f384-f16"]
    w = _weights("vitb16-16f384-f16")
    clip = synth.clip_u8(cfg)
    enc = jg.Encoder(cfg, w)
    res = enc.encode(torch.from_numpy(clip).cuda(), pooled=True)
    enc.sync()
    ref = oracle.encoder_forward(cfg, w, clip[0])
    m = assert_close_16bit(res["out"][0].cpu().numpy(), ref["out"], "vitb16-16f384-f16 end to end")
    print("vitb16-16f384-f16 end to end:", m)
    np.testing.assert_allclose(res["pooled"][0].cpu().numpy(), ref["pooled"], atol=1e-2 * np.abs(ref["pooled"]).max())
    enc.close()


def test_vitb16_64f384_blocks_taps_final(jg):
    cfg = synth.CONFIGS["vitb16-64f384"]
    w = _weights("vitb16-64f384")
    clip = torch.from_numpy(synth.clip_u8(cfg)).cuda()
    enc = jg.Encoder(cfg, w)
    res = enc.encode(clip, hier=True)
    enc.sync()
    B, T, H, W, _ = clip.shape
    N, D = synth.tokens_per_clip(cfg), cfg.embed_dim
    # taps and output from the GPU's own residual after each tapped block
    stats = []
    x, rows = _check_blocks(enc, cfg, w, clip, 0, 32, 9, stats)
    x_l = enc.embed(clip)
    done = 0
    for k, layer in enumerate(cfg.hier_layers):
        enc.blocks(x_l, B, T, H, W, done, layer + 1)
        done = layer + 1
        enc.sync()
        xr = x_l.view(N, D).cpu().numpy().astype(np.float64)[rows]
        ref = oracle.layer_norm(xr, w[f"hier_norm.{k}.weight"], w[f"hier_norm.{k}.bias"], cfg.ln_eps)
        assert_close_16bit(res["hier"][k, 0].cpu().numpy()[rows], ref, f"vitb16-64f384 tap {k}")
    ref = oracle.layer_norm(x_l.view(N, D).cpu().numpy().astype(np.float64)[rows], w["norm.weight"], w["norm.bias"],
                            cfg.ln_eps)
    assert_close_16bit(res["out"][0].cpu().numpy()[rows], ref, "vitb16-64f384 final norm")
    enc.close()


def test_vitl16_64f256_pred_encoder_blocks_and_predictor(jg):
    cfg = synth.CONFIGS["vitl16-64f256-pred"]
    w = _weights("vitl16-64f256-pred")
    clip = torch.from_numpy(synth.clip_u8(cfg)).cuda()
    enc = jg.Encoder(cfg, w)
    stats = []
    _check_blocks(enc, cfg, w, clip, 0, 32, 11, stats)
    tokens = enc.encode(clip)["out"][0].contiguous()
    enc.sync()
    enc.close()
    pc = cfg.predictor
    pw = synth.predictor_weights(cfg)
    ctx, tgt = synth.context_target_split(cfg)
    pred = jg.Predictor(pc, pw, cfg.dtype)
    out = pred.predict(tokens, torch.from_numpy(ctx).cuda(), torch.from_numpy(tgt).cuda(), cfg.grid())
    pred.sync()
    ref = oracle.predictor_forward(pc, pw, tokens.cpu().numpy().astype(np.float64), ctx, tgt, cfg.grid())
    m = assert_close_16bit(out.cpu().numpy(), ref, "vitl16-64f256-pred predictor")
    print("vitl16-64f256-pred predictor:", m)
    pred.close()


def test_img384_end_to_end(jg):
    """The 2.1 native image path at its workload size (ViT-B/16, 32 images of
    384 x 384, 576 tokens each): images 0 and 31 end to end on every token,
    with the hierarchical taps and the token mean."""
    cfg = synth.CONFIGS["img384"]
    w = _weights("img384")
    clip = synth.clip_u8(cfg)
    enc = jg.Encoder(cfg, w)
    res = enc.encode(torch.from_numpy(clip).cuda(), pooled=True, hier=True)
    enc.sync()
    for b in (0, cfg.batch - 1):
        ref = oracle.encoder_forward(cfg, w, clip[b])
        assert_close_16bit(res["out"][b].cpu().numpy(), ref["out"], f"img384 image {b}")
        for k, tap in enumerate(ref["hier"]):
            assert_close_16bit(res["hier"][k, b].cpu().numpy(), tap, f"img384 tap {k} image {b}")
        np.testing.assert_allclose(res["pooled"][b].cpu().numpy(), ref["pooled"],
                                   atol=1e-2 * np.abs(ref["pooled"]).max())
    enc.close()


def test_pred21_encoder_and_predictor(jg):
    """The 2.1 predictor (D384 L12 hd32, interleaved RoPE on the 8 x 24 x 24
    grid, 8 mask tokens, out 1664, context projection) on the 2.1 ViT-B/16
    encoder's own output for a 16-frame 384 px clip (4608 tokens): target
    predictions and context projections end to end against the oracle run on
    the same encoder tokens, video modality; then the image modality on a
    576-token image encoded by the same model."""
    cfg = synth.CONFIGS["pred21"]
    w = _weights("pred21")
    pc = cfg.predictor
    pw = synth.predictor_weights(cfg)
    enc = jg.Encoder(cfg, w)
    pred = jg.Predictor(pc, pw, cfg.dtype)
    for T, mod in ((cfg.n_frames, "video"), (1, "image")):
        c = cfg.with_(n_frames=T)
        clip = torch.from_numpy(synth.clip_u8(c, batch=1)).cuda()
        tokens = enc.encode(clip)["out"][0].contiguous()
        enc.sync()
        ctx, tgt = synth.context_target_split(c)
        out, octx = pred.predict(tokens, torch.from_numpy(ctx).cuda(), torch.from_numpy(tgt).cuda(), c.grid(),
                                 modality="auto", with_ctx=True)
        pred.sync()
        ref = oracle.predictor_outputs(pc, pw, tokens.cpu().numpy().astype(np.float64), ctx, tgt, c.grid(), mod)
        assert_close_16bit(out.cpu().numpy(), ref["pred"], f"pred21 {mod} targets")
        assert_close_16bit(octx.cpu().numpy(), ref["ctx"], f"pred21 {mod} context projection")
        if mod == "video":   # the plain call is the video modality without the context output
            plain = pred.predict(tokens, torch.from_numpy(ctx).cuda(), torch.from_numpy(tgt).cuda(), c.grid())
            pred.sync()
            assert torch.equal(plain, out)
    pred.close()
    enc.close()


def test_vitl16_16f256_masked_encoder_clip0(jg):
    """Masked encoder forward at the ViT-L/16 16 x 256 x 256 geometry, batch 8,
    each clip keeping its own random half of the 2048 tokens; clip 0 end to end
    against the oracle's masked forward."""
    cfg = synth.CONFIGS["vitl16-16f256"]
    w = _weights("vitl16-16f256")
    clip = synth.clip_u8(cfg)
    n = synth.tokens_per_clip(cfg)
    keep = np.stack([np.random.default_rng(40 + b).choice(n, n // 2, replace=False)
                     for b in range(cfg.batch)]).astype(np.int32)
    enc = jg.Encoder(cfg, w)
    got = enc.encode_masked(torch.from_numpy(clip).cuda(), torch.from_numpy(keep).cuda())["out"]
    enc.sync()
    ref = oracle.encoder_forward(cfg, w, clip[0], keep=keep[0])
    assert_close_16bit(got[0].cpu().numpy(), ref["out"], "vitl16-16f256 masked clip 0")
    enc.close()
