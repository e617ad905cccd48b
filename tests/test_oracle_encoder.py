"""Pins for the oracle's composition (encoder and masked predictor).

A torch float64 forward built from library routines (conv3d, layer_norm,
linear, scaled_dot_product_attention, erf GELU) with the RoPE tables of the
conversion notes §4 must reproduce the oracle; structural cases (zeroed
blocks, row sampling, permutations) pin the rest.
"""
import dataclasses

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle
import synth

BLOCK_F32 = synth.CONFIGS["block-f32-4f128"]
SMALL_21 = synth.CONFIGS["vitb16-16f384-f16"].with_(n_layer=2, n_frames=4, height=128, width=160, hier_layers=(0, 1),
                                     dtype="f32")


def _t(a):
    return torch.from_numpy(np.asarray(a, np.float64))


def _torch_rope(x, pos, layout, theta=10000.0):
    # x [h, N, hd]; tables from §4.1 / §4.2 with torch's repeat / repeat_interleave
    hd = x.shape[-1]
    d = 2 * ((hd // 3) // 2)
    om = 1.0 / theta ** (torch.arange(d // 2, dtype=torch.float64) / (d / 2))
    parts = []
    for a in range(3):
        f = pos[:, a:a + 1] * om[None]
        e = f.repeat(1, 2) if layout == "tiled" else f.repeat_interleave(2, dim=-1)
        parts.append(e)
    ang = torch.cat(parts, dim=-1)                          # [N, 3d]
    xr, xp = x[..., :3 * d], x[..., 3 * d:]
    pairs = xr.unflatten(-1, (-1, 2))
    rot = torch.stack((-pairs[..., 1], pairs[..., 0]), dim=-1).flatten(-2)
    return torch.cat([xr * ang.cos() + rot * ang.sin(), xp], dim=-1)


def _torch_encoder(cfg, w, clip, keep=None):
    T, H, W, _ = clip.shape
    x = torch.from_numpy(clip.astype(np.float64)).permute(3, 0, 1, 2)
    mean = torch.tensor([0.485, 0.456, 0.406], dtype=torch.float64)[:, None, None, None]
    std = torch.tensor([0.229, 0.224, 0.225], dtype=torch.float64)[:, None, None, None]
    x = (x - 255 * mean) / (255 * std)
    D = cfg.embed_dim
    k = _t(w["patch_embed.weight"]).reshape(D, 3, 2, 16, 16)
    tok = Fn.conv3d(x[None], k, _t(w["patch_embed.bias"]), stride=(2, 16, 16))[0]
    tok = tok.flatten(1).T                                   # [N, D], T-major
    if cfg.has_mod_embed:
        tok = tok + _t(w["mod_embed_video"])
    gt, gh, gw = T // 2, H // 16, W // 16
    tt, hh, ww = torch.meshgrid(torch.arange(gt), torch.arange(gh), torch.arange(gw), indexing="ij")
    pos = torch.stack([tt.flatten(), hh.flatten(), ww.flatten()], 1).double()
    if cfg.rope_interpolate:
        pos[:, 1] = pos[:, 1] * (cfg.rope_ref_grid - 1) / (gh - 1)
        pos[:, 2] = pos[:, 2] * (cfg.rope_ref_grid - 1) / (gw - 1)
    if keep is not None:                                     # masked encoder: kept tokens, true positions
        idx = torch.from_numpy(np.asarray(keep)).long()
        tok, pos = tok[idx], pos[idx]
    h = cfg.n_head
    hier = []
    for i in range(cfg.n_layer):
        p = f"blk.{i}."
        y = Fn.layer_norm(tok, (D,), _t(w[p + "ln1.weight"]), _t(w[p + "ln1.bias"]), cfg.ln_eps)
        qkv = Fn.linear(y, _t(w[p + "attn_qkv.weight"]), _t(w[p + "attn_qkv.bias"]))
        q, kk, v = (t.reshape(-1, h, D // h).transpose(0, 1) for t in qkv.split(D, dim=1))
        q, kk = _torch_rope(q, pos, cfg.rope_layout), _torch_rope(kk, pos, cfg.rope_layout)
        o = Fn.scaled_dot_product_attention(q, kk, v).transpose(0, 1).reshape(-1, D)
        tok = tok + Fn.linear(o, _t(w[p + "attn_out.weight"]), _t(w[p + "attn_out.bias"]))
        y = Fn.layer_norm(tok, (D,), _t(w[p + "ln2.weight"]), _t(w[p + "ln2.bias"]), cfg.ln_eps)
        g = Fn.gelu(Fn.linear(y, _t(w[p + "ffn_up.weight"]), _t(w[p + "ffn_up.bias"])))
        tok = tok + Fn.linear(g, _t(w[p + "ffn_down.weight"]), _t(w[p + "ffn_down.bias"]))
        if i in cfg.hier_layers:
            kx = list(cfg.hier_layers).index(i)
            hier.append(Fn.layer_norm(tok, (D,), _t(w[f"hier_norm.{kx}.weight"]),
                                      _t(w[f"hier_norm.{kx}.bias"]), cfg.ln_eps).numpy())
    out = Fn.layer_norm(tok, (D,), _t(w["norm.weight"]), _t(w["norm.bias"]), cfg.ln_eps)
    return out.numpy(), hier


def _perturb_lns(w, seed):
    # LN affines and biases are 1/0 in the workloads; randomise them here so
    # a swapped weight/bias or a dropped bias cannot hide.
    rng = np.random.default_rng(seed)
    w = dict(w)
    for k in list(w):
        if k.endswith(".bias") or "ln" in k or k.startswith("norm") or k.startswith("hier"):
            w[k] = (w[k] + rng.standard_normal(w[k].shape) * 0.1).astype(np.float32)
    return w


@pytest.mark.parametrize("cfg", [BLOCK_F32, SMALL_21], ids=["block-f32-4f128", "vitb21-2layer"])
def test_encoder_matches_torch_composition(cfg):
    w = _perturb_lns(synth.encoder_weights(cfg), 7)
    clip = synth.clip_u8(cfg, batch=1)[0]
    got = oracle.encoder_forward(cfg, w, clip)
    ref, hier = _torch_encoder(cfg, w, clip)
    np.testing.assert_allclose(got["out"], ref, rtol=0, atol=1e-10)
    assert len(got["hier"]) == len(hier) == len(cfg.hier_layers)
    for a, b in zip(got["hier"], hier):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-10)
    np.testing.assert_allclose(got["pooled"], ref.mean(0), atol=1e-10)


def test_zero_blocks_reduce_to_norm_of_patch_embed():
    cfg = BLOCK_F32
    w = synth.encoder_weights(cfg)
    for k in list(w):
        if k.startswith("blk."):
            w[k] = np.zeros_like(w[k])
    clip = synth.clip_u8(cfg, batch=1)[0]
    got = oracle.encoder_forward(cfg, w, clip)["out"]
    x = oracle.patch_embed(oracle.normalise_clip(clip), w["patch_embed.weight"], w["patch_embed.bias"])
    exp = oracle.layer_norm(x, w["norm.weight"], w["norm.bias"], cfg.ln_eps)
    np.testing.assert_array_equal(got, exp)


def test_block_rows_equals_full_block():
    cfg = SMALL_21
    w = _perturb_lns(synth.encoder_weights(cfg), 3)
    clip = synth.clip_u8(cfg, batch=1)[0]
    x = oracle.encoder_embed(cfg, w, clip)
    COS, SIN = oracle.encoder_rope(cfg, *clip.shape[:3])
    full = oracle.block_forward(x, w, 1, cfg.n_head, cfg.ln_eps, COS, SIN)
    rows = np.array([0, 5, 17, x.shape[0] - 1])
    part = oracle.block_forward_rows(x, w, 1, cfg.n_head, cfg.ln_eps, COS, SIN, rows)
    np.testing.assert_allclose(part, full[rows], rtol=0, atol=1e-12)


def test_weight_perturbation_is_visible():
    # The parity gate must see a +1 % error on a single weight matrix.
    cfg = BLOCK_F32
    w = synth.encoder_weights(cfg)
    clip = synth.clip_u8(cfg, batch=1)[0]
    a = oracle.encoder_forward(cfg, w, clip)["out"]
    w2 = dict(w)
    w2["blk.0.attn_out.weight"] = w["blk.0.attn_out.weight"] * 1.01
    b = oracle.encoder_forward(cfg, w2, clip)["out"]
    assert np.max(np.abs(a - b)) / np.max(np.abs(a)) > 1e-4


PRED_CFG = synth.CONFIGS["vitl16-64f256-pred"].with_(
    n_frames=4, height=64, width=64,
    predictor=synth.PredictorConfig(n_layer=2, in_dim=1024))


def _pred_setup(seed=0):
    cfg = PRED_CFG
    pw = _perturb_lns(synth.predictor_weights(cfg), seed)
    gt, gh, gw = cfg.grid()
    n = gt * gh * gw
    enc = np.random.default_rng(seed).standard_normal((n, 1024))
    ctx, tgt = synth.context_target_split(cfg)
    return cfg, pw, enc, ctx, tgt, (gt, gh, gw)


def _torch_predictor(pc, pw, enc, ctx, tgt, grid, modality="video", with_ctx=False):
    D = pc.embed_dim
    z_ctx = Fn.linear(_t(enc)[torch.from_numpy(ctx).long()], _t(pw["embed.weight"]), _t(pw["embed.bias"]))
    m = _t(pw["mask_tokens"])[pc.mask_index % pc.n_mask_tokens]
    z = torch.cat([z_ctx, m.expand(len(tgt), D)], 0)
    if pc.has_mod_embed:
        z = z + _t(pw["mod_embed_img" if modality == "image" else "mod_embed_video"])
    ids = torch.from_numpy(np.concatenate([ctx, tgt])).long()
    gt, gh, gw = grid
    pos = torch.stack([ids // (gh * gw), (ids % (gh * gw)) // gw, ids % gw], 1).double()
    h = pc.n_head
    for i in range(pc.n_layer):
        p = f"blk.{i}."
        y = Fn.layer_norm(z, (D,), _t(pw[p + "ln1.weight"]), _t(pw[p + "ln1.bias"]), pc.ln_eps)
        qkv = Fn.linear(y, _t(pw[p + "attn_qkv.weight"]), _t(pw[p + "attn_qkv.bias"]))
        q, k, v = (t.reshape(-1, h, D // h).transpose(0, 1) for t in qkv.split(D, dim=1))
        q, k = _torch_rope(q, pos, pc.rope_layout), _torch_rope(k, pos, pc.rope_layout)
        o = Fn.scaled_dot_product_attention(q, k, v).transpose(0, 1).reshape(-1, D)
        z = z + Fn.linear(o, _t(pw[p + "attn_out.weight"]), _t(pw[p + "attn_out.bias"]))
        y = Fn.layer_norm(z, (D,), _t(pw[p + "ln2.weight"]), _t(pw[p + "ln2.bias"]), pc.ln_eps)
        z = z + Fn.linear(Fn.gelu(Fn.linear(y, _t(pw[p + "ffn_up.weight"]), _t(pw[p + "ffn_up.bias"]))),
                          _t(pw[p + "ffn_down.weight"]), _t(pw[p + "ffn_down.bias"]))
    z = Fn.layer_norm(z, (D,), _t(pw["norm.weight"]), _t(pw["norm.bias"]), pc.ln_eps)
    pred = Fn.linear(z[len(ctx):], _t(pw["proj.weight"]), _t(pw["proj.bias"])).numpy()
    if not with_ctx:
        return pred
    return pred, Fn.linear(z[:len(ctx)], _t(pw["proj_context.weight"]), _t(pw["proj_context.bias"])).numpy()


def test_predictor_matches_torch_composition():
    cfg, pw, enc, ctx, tgt, grid = _pred_setup()
    got = oracle.predictor_forward(cfg.predictor, pw, enc, ctx, tgt, grid)
    assert got.shape == (len(tgt), 1024)
    ref = _torch_predictor(cfg.predictor, pw, enc, ctx, tgt, grid)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)


def test_predictor_split_and_mask_token():
    cfg, pw, enc, ctx, tgt, grid = _pred_setup(1)
    n = enc.shape[0]
    assert len(ctx) == len(tgt) == n // 2
    assert np.array_equal(np.sort(np.concatenate([ctx, tgt])), np.arange(n))
    z = oracle.predictor_input(cfg.predictor, pw, enc, ctx, tgt)
    np.testing.assert_array_equal(z[len(ctx):], np.broadcast_to(pw["mask_tokens"][1].astype(np.float64),
                                                                 (len(tgt), 384)))


def test_predictor_target_permutation_equivariant():
    # [conversion notes §3]: attention is permutation-equivariant, so the
    # token order fed to the blocks (with positions attached) does not matter.
    cfg, pw, enc, ctx, tgt, grid = _pred_setup(2)
    a = oracle.predictor_forward(cfg.predictor, pw, enc, ctx, tgt, grid)
    perm = np.random.default_rng(0).permutation(len(tgt))
    b = oracle.predictor_forward(cfg.predictor, pw, enc, ctx, tgt[perm], grid)
    np.testing.assert_allclose(a[perm], b, atol=1e-11)


# ----------------------------------------------------------------------------- 2.1 predictor
# [conversion notes §3, 2.1 predictor forward]: the modality vector on every
# row, interleaved RoPE from the ids on the fixed 24-grid with no
# interpolation, pred.norm, pred.proj on the target rows and
# pred.proj_context on the context rows.
PRED21_CFG = synth.CONFIGS["pred21"].with_(
    n_frames=4, height=96, width=96,
    predictor=dataclasses.replace(synth.PREDICTOR_21, n_layer=2))


def _pred21_setup(seed=0, image=False):
    cfg = PRED21_CFG.with_(n_frames=1) if image else PRED21_CFG
    pw = _perturb_lns(synth.predictor_weights(cfg), seed)
    rng = np.random.default_rng(seed)
    for k in ("mod_embed_video", "mod_embed_img"):
        pw[k] = rng.standard_normal(pw[k].shape) * 0.5        # visible against the 0.02-scale weights
    gt, gh, gw = cfg.grid()
    n = gt * gh * gw
    enc = rng.standard_normal((n, 768))
    ctx, tgt = synth.context_target_split(cfg)
    return cfg, pw, enc, ctx, tgt, (gt, gh, gw)


@pytest.mark.parametrize("image", [False, True])
def test_predictor21_matches_torch_composition(image):
    cfg, pw, enc, ctx, tgt, grid = _pred21_setup(3, image)
    mod = "image" if image else "video"
    got = oracle.predictor_outputs(cfg.predictor, pw, enc, ctx, tgt, grid, mod)
    assert got["pred"].shape == (len(tgt), 1664) and got["ctx"].shape == (len(ctx), 1664)
    ref_pred, ref_ctx = _torch_predictor(cfg.predictor, pw, enc, ctx, tgt, grid, mod, with_ctx=True)
    np.testing.assert_allclose(got["pred"], ref_pred, rtol=0, atol=1e-10)
    np.testing.assert_allclose(got["ctx"], ref_ctx, rtol=0, atol=1e-10)


def test_predictor21_zero_blocks_closed_form():
    """With every block zeroed the blocks are the identity, so each target row
    is proj(norm(mask token + modality vector)) and each context row
    proj_context(norm(embed(enc row) + modality vector))."""
    cfg, pw, enc, ctx, tgt, grid = _pred21_setup(4)
    pc = cfg.predictor
    for k in list(pw):
        if k.startswith("blk."):
            pw[k] = np.zeros_like(pw[k])
    got = oracle.predictor_outputs(pc, pw, enc, ctx, tgt, grid, "video")
    mod = pw["mod_embed_video"].astype(np.float64)
    m = pw["mask_tokens"][pc.mask_index % pc.n_mask_tokens].astype(np.float64) + mod
    zt = oracle.layer_norm(m[None], pw["norm.weight"], pw["norm.bias"], pc.ln_eps)
    exp_t = zt @ pw["proj.weight"].astype(np.float64).T + pw["proj.bias"]
    np.testing.assert_allclose(got["pred"], np.broadcast_to(exp_t, got["pred"].shape), rtol=0, atol=1e-12)
    e = enc[ctx] @ pw["embed.weight"].astype(np.float64).T + pw["embed.bias"] + mod
    zc = oracle.layer_norm(e, pw["norm.weight"], pw["norm.bias"], pc.ln_eps)
    exp_c = zc @ pw["proj_context.weight"].astype(np.float64).T + pw["proj_context.bias"]
    np.testing.assert_allclose(got["ctx"], exp_c, rtol=0, atol=1e-12)


def test_predictor21_context_permutation_equivariant():
    """Permuting the context ids permutes the context outputs and leaves the
    target predictions unchanged (attention with positions attached is
    permutation-equivariant)."""
    cfg, pw, enc, ctx, tgt, grid = _pred21_setup(5)
    a = oracle.predictor_outputs(cfg.predictor, pw, enc, ctx, tgt, grid)
    perm = np.random.default_rng(1).permutation(len(ctx))
    b = oracle.predictor_outputs(cfg.predictor, pw, enc, ctx[perm], tgt, grid)
    np.testing.assert_allclose(b["ctx"], a["ctx"][perm], atol=1e-11)
    np.testing.assert_allclose(b["pred"], a["pred"], atol=1e-11)


def test_predictor21_mask_token_and_modality():
    cfg, pw, enc, ctx, tgt, grid = _pred21_setup(6)
    pc = cfg.predictor
    assert pc.n_mask_tokens == 8 and pc.mask_index % pc.n_mask_tokens == 1
    z = oracle.predictor_input(pc, pw, enc, ctx, tgt, "image")
    exp = pw["mask_tokens"][1].astype(np.float64) + pw["mod_embed_img"]
    np.testing.assert_array_equal(z[len(ctx):], np.broadcast_to(exp, (len(tgt), 384)))
    zv = oracle.predictor_input(pc, pw, enc, ctx, tgt, "video")
    np.testing.assert_allclose(z - zv, np.broadcast_to(pw["mod_embed_img"] - pw["mod_embed_video"], z.shape),
                               atol=1e-12)


# ----------------------------------------------------------------------------- masked encoder
# [H] Usage ("Predictor") and Validation: masks given to the encoder drop the
# tokens before the blocks; attention sees only the kept ones and RoPE keeps
# the true positions.
def _keep_ids(cfg, seed, frac=0.4):
    n = synth.tokens_per_clip(cfg)
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(n, int(n * frac), replace=False))


def test_masked_encoder_matches_torch_composition():
    cfg = SMALL_21
    w = _perturb_lns(synth.encoder_weights(cfg), 11)
    clip = synth.clip_u8(cfg, batch=1)[0]
    keep = _keep_ids(cfg, 1)
    got = oracle.encoder_forward(cfg, w, clip, keep=keep)
    ref, hier = _torch_encoder(cfg, w, clip, keep=keep)
    assert got["out"].shape == (len(keep), cfg.embed_dim)
    np.testing.assert_allclose(got["out"], ref, rtol=0, atol=1e-10)
    for a, b in zip(got["hier"], hier):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-10)


def test_masked_encoder_keeping_every_token_is_the_encoder():
    cfg = SMALL_21
    w = synth.encoder_weights(cfg)
    clip = synth.clip_u8(cfg, batch=1)[0]
    n = synth.tokens_per_clip(cfg)
    a = oracle.encoder_forward(cfg, w, clip)["out"]
    b = oracle.encoder_forward(cfg, w, clip, keep=np.arange(n))["out"]
    np.testing.assert_array_equal(a, b)


def test_masked_encoder_is_not_the_gathered_output():
    """The pages' control: dropping tokens before the blocks differs from
    gathering the unmasked encoder's output."""
    cfg = SMALL_21
    w = synth.encoder_weights(cfg)
    clip = synth.clip_u8(cfg, batch=1)[0]
    keep = _keep_ids(cfg, 2)
    masked = oracle.encoder_forward(cfg, w, clip, keep=keep)["out"]
    gathered = oracle.encoder_forward(cfg, w, clip)["out"][keep]
    assert np.abs(masked - gathered).max() > 1e-3


def test_masked_encoder_permutation_equivariant_with_true_positions():
    """Permuting the kept ids permutes the output rows: each token carries its
    own grid position, not its index in the kept list."""
    cfg = SMALL_21
    w = synth.encoder_weights(cfg)
    clip = synth.clip_u8(cfg, batch=1)[0]
    keep = _keep_ids(cfg, 3)
    perm = np.random.default_rng(4).permutation(len(keep))
    a = oracle.encoder_forward(cfg, w, clip, keep=keep)["out"]
    b = oracle.encoder_forward(cfg, w, clip, keep=keep[perm])["out"]
    np.testing.assert_allclose(b, a[perm], atol=1e-11)
