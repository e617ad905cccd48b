"""Plain float64 restatement of the V-JEPA 2 / 2.1 encoder, masked predictor
and attentive-pool classifier head.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Parity of every
function here is pinned by ``tests/test_oracle_*.py`` against library
routines, closed forms and the values the pages print; the composition of
the whole encoder on real-size workloads is "parity unpinned beyond
composition" because no worked example with synthetic weights exists.

Sources (page title, section):
  [N]  "V-JEPA 2 / 2.1 tensor maps and RoPE derivation" (jepa.cpp conversion
       notes): §1 hyper-parameters, §2 HF key map and "Attentive-pool head -
       exact forward", §3 2.1 encoder/predictor forward, §4 3-D RoPE (4.1 tiled, 4.2 interleaved, 4.3 interpolation,
       4.4 predictor ids), §5 preprocessing.
  [P]  "Parity - image ViT encoders ... and video encoders" (jepa.cpp parity
       report): "Preprocessing parity" (fused normalisation form),
       "Parity on a GPU" (LayerNorm is the centred two-pass variance).
  [H]  "V-JEPA 2.1 ViT-B/16 384 - HuggingFace port": Architecture, Usage.

Weights arrive as a dict of float32 arrays with the names of
``synth.tensor_names_encoder``; every computation below promotes them to
float64.  A config object supplies the hyper-parameters (duck typed: any
object with the fields used below).
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

F64 = np.float64

# [N] §1 "pre.mean / std / rescale: ImageNet / 1/255"; [H] Preprocessing
# states the ImageNet statistics explicitly.
IMAGENET_MEAN = (0.485, 0.456, 0.406)
IMAGENET_STD = (0.229, 0.224, 0.225)


# ----------------------------------------------------------------------------- input
def normalise_clip(clip_u8: np.ndarray) -> np.ndarray:
    """THWC uint8 clip -> channel-first ``[3, T, H, W]`` normalised pixels.

    [P] "Preprocessing parity": normalisation is the fused form
    ``(px - 255*mean) / (255*std)``; [N] §5: the model consumes the clip as
    ``[C, T, H, W]``.
    """
    x = np.asarray(clip_u8, dtype=F64)                    # [T, H, W, 3]
    mean = np.asarray(IMAGENET_MEAN, F64)
    std = np.asarray(IMAGENET_STD, F64)
    x = (x - 255.0 * mean) / (255.0 * std)
    return np.transpose(x, (3, 0, 1, 2))                  # [3, T, H, W]


def patch_embed(x: np.ndarray, weight: np.ndarray, bias: np.ndarray,
                tubelet: int = 2, patch: int = 16) -> np.ndarray:
    """Tubelet embedding as the Conv3d it is, stride equal to the kernel.

    [N] §2: the Conv3d weight ``[D, 3, tubelet, patch, patch]`` is stored as
    ``[D, 3*tubelet*patch*patch]`` by a row-major reshape (feature order
    C, T, H, W), so reshaping back recovers the kernel.  The output is one
    token per (t, h, w) tubelet cell, ordered T-major then H then W ([N] §4).

    out[t, i, j, :] = bias + sum_{c, dt, y, x} K[:, c, dt, y, x] *
                      x[c, tubelet*t + dt, patch*i + y, patch*j + x]
    """
    C, T, H, W = x.shape
    D = weight.shape[0]
    K = np.asarray(weight, F64).reshape(D, C, tubelet, patch, patch)
    gt, gh, gw = T // tubelet, H // patch, W // patch
    # x[c, tubelet*t + dt, patch*i + y, patch*j + xx] viewed as [c, t, dt, i, y, j, xx]
    xv = x[:, :gt * tubelet, :gh * patch, :gw * patch].reshape(C, gt, tubelet, gh, patch, gw, patch)
    # the sum over every kernel tap (c, dt, y, xx) at every output cell (t, i, j)
    out = np.einsum("dcpyx,ctpiyjx->tijd", K, xv, optimize=True)
    out = out + np.asarray(bias, F64)
    return out.reshape(gt * gh * gw, D)


# ----------------------------------------------------------------------------- RoPE
def rope_split(head_dim: int) -> int:
    """Per-axis rotated width ``d = 2 * ((head_dim // 3) // 2)`` ([N] §1, §4)."""
    return 2 * ((head_dim // 3) // 2)


def token_positions(gt: int, gh: int, gw: int, interpolate: bool = False,
                    ref_grid: int = 16) -> np.ndarray:
    """Per-token (t, h, w) positions, ``[N, 3]`` float64.

    [N] §4: token i maps T-major to t = i // (gh*gw), h = (i mod gh*gw) // gw,
    w = i mod gw; t counts tubelets.  [N] §4.3: with interpolation the spatial
    positions become h * (ref_grid - 1) / (gh - 1) (same for w), evaluated
    left to right; t is never rescaled; a 1-wide grid is rejected.
    """
    i = np.arange(gt * gh * gw)
    t = (i // (gh * gw)).astype(F64)
    h = ((i % (gh * gw)) // gw).astype(F64)
    w = (i % gw).astype(F64)
    if interpolate:
        if gh <= 1 or gw <= 1:
            raise ValueError("RoPE interpolation needs a grid wider than 1")
        h = h * (ref_grid - 1) / (gh - 1)
        w = w * (ref_grid - 1) / (gw - 1)
    return np.stack([t, h, w], axis=1)


def grid_positions_from_ids(ids: np.ndarray, gt: int, gh: int, gw: int) -> np.ndarray:
    """[N] §4.4: predictor ids index the full encoder grid and decode as in §4."""
    ids = np.asarray(ids, np.int64)
    t = (ids // (gh * gw)).astype(F64)
    h = ((ids % (gh * gw)) // gw).astype(F64)
    w = (ids % gw).astype(F64)
    return np.stack([t, h, w], axis=1)


def rope_tables(pos: np.ndarray, head_dim: int, layout: str, theta: float = 10000.0):
    """Per-token ``COS, SIN`` tables ``[N, head_dim]`` ([N] §4, implementation hint of 4.1).

    omega_k = 1 / theta ** (k / (d/2)), k = 0..d/2-1, and f_k = pos * omega_k
    per axis.  The length-d/2 table is expanded to length d either by tiling
    ([f_0..f_{d/2-1}, f_0..f_{d/2-1}], V-JEPA 2, §4.1) or by repeating each
    entry twice ([f_0, f_0, f_1, f_1, ...], V-JEPA 2.1, §4.2).  Dims
    [0,d) use t, [d,2d) h, [2d,3d) w; the rest pass through (COS 1, SIN 0).
    """
    d = rope_split(head_dim)
    half = d // 2
    omega = 1.0 / theta ** (np.arange(half, dtype=F64) / half)
    N = pos.shape[0]
    COS = np.ones((N, head_dim), F64)
    SIN = np.zeros((N, head_dim), F64)
    for a in range(3):
        f = pos[:, a:a + 1] * omega[None, :]              # [N, d/2]
        if layout == "tiled":
            g = np.concatenate([f, f], axis=1)
        elif layout == "interleaved":
            g = np.repeat(f, 2, axis=1)
        else:
            raise ValueError(f"unknown RoPE layout {layout!r}")
        COS[:, a * d:(a + 1) * d] = np.cos(g)
        SIN[:, a * d:(a + 1) * d] = np.sin(g)
    return COS, SIN


def rot90_pairs(x: np.ndarray) -> np.ndarray:
    """[N] §4: rot90(x)[2k] = -x[2k+1], rot90(x)[2k+1] = x[2k] (last axis)."""
    y = np.empty_like(x)
    y[..., 0::2] = -x[..., 1::2]
    y[..., 1::2] = x[..., 0::2]
    return y


def apply_rope(x: np.ndarray, COS: np.ndarray, SIN: np.ndarray) -> np.ndarray:
    """[N] §4: out = x * COS + rot90(x) * SIN (per head; tables broadcast)."""
    return x * COS + rot90_pairs(x) * SIN


# ----------------------------------------------------------------------------- layers
def layer_norm(x: np.ndarray, weight, bias, eps: float) -> np.ndarray:
    """LayerNorm over the last axis with the biased, centred two-pass variance.

    [N] §1 gives eps 1e-6; [P] "Parity on a GPU" names the CPU reference's
    variance as centred two-pass; eps is added to the variance inside the
    square root (PyTorch LayerNorm semantics the checkpoints were trained with).
    """
    x = np.asarray(x, F64)
    mu = x.mean(axis=-1, keepdims=True)
    xc = x - mu
    var = (xc * xc).mean(axis=-1, keepdims=True)
    return xc / np.sqrt(var + eps) * np.asarray(weight, F64) + np.asarray(bias, F64)


def gelu_erf(z: np.ndarray) -> np.ndarray:
    """[N] §1: the activation is the exact erf GELU, 0.5 z (1 + erf(z / sqrt 2))."""
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def attention_heads(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Unmasked softmax attention per head, ``[h, Nq, hd] x [h, Nk, hd] -> [h, Nq, hd]``.

    Scores are q k^T / sqrt(head_dim) ([N] §4: the scaling comes after RoPE);
    the video encoders use full attention with no mask ([P] "Flash attention
    K/V dtype").  Softmax is max-subtracted, exponentiated and normalised.
    """
    hd = q.shape[-1]
    out = np.empty(q.shape[:-1] + (v.shape[-1],), F64)
    for h in np.ndindex(q.shape[:-2]):        # one head at a time
        s = (q[h] @ k[h].T) / math.sqrt(hd)
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=-1, keepdims=True)
        out[h] = p @ v[h]
    return out


def _linear(x, w, b):
    return x @ np.asarray(w, F64).T + np.asarray(b, F64)


def _split_heads(t: np.ndarray, n_head: int) -> np.ndarray:
    N, D = t.shape
    return t.reshape(N, n_head, D // n_head).transpose(1, 0, 2)   # [h, N, hd]


def _qkv_rope(y, wts, p, n_head, COS, SIN):
    D = y.shape[1]
    qkv = _linear(y, wts[p + "attn_qkv.weight"], wts[p + "attn_qkv.bias"])
    # [N] §2: the fused projection's rows are [Wq; Wk; Wv]
    q, k, v = qkv[:, :D], qkv[:, D:2 * D], qkv[:, 2 * D:]
    q, k, v = (_split_heads(t, n_head) for t in (q, k, v))
    # [N] §4: RoPE on q and k, not v, after the projection bias
    return apply_rope(q, COS, SIN), apply_rope(k, COS, SIN), v


def block_forward(x, wts, layer: int, n_head: int, eps: float, COS, SIN, prefix: str = "blk."):
    """One pre-LN block ([N] §2 block form, §3 2.1 forward):
    x += attn_out(concat_heads(attn(RoPE(qkv(ln1 x))))); x += ffn_down(gelu(ffn_up(ln2 x))).
    """
    p = f"{prefix}{layer}."
    x = np.asarray(x, F64)
    y = layer_norm(x, wts[p + "ln1.weight"], wts[p + "ln1.bias"], eps)
    q, k, v = _qkv_rope(y, wts, p, n_head, COS, SIN)
    o = attention_heads(q, k, v)                              # [h, N, hd]
    o = o.transpose(1, 0, 2).reshape(x.shape[0], -1)          # heads concatenated in order
    x = x + _linear(o, wts[p + "attn_out.weight"], wts[p + "attn_out.bias"])
    y = layer_norm(x, wts[p + "ln2.weight"], wts[p + "ln2.bias"], eps)
    g = gelu_erf(_linear(y, wts[p + "ffn_up.weight"], wts[p + "ffn_up.bias"]))
    return x + _linear(g, wts[p + "ffn_down.weight"], wts[p + "ffn_down.bias"])


def block_forward_rows(x, wts, layer: int, n_head: int, eps: float, COS, SIN, rows,
                       prefix: str = "blk."):
    """``block_forward(...)[rows]`` computing only what those rows depend on.

    Keys and values need every token; queries, the output projection and
    the MLP are row-wise, so they are evaluated for ``rows`` alone.  The
    arithmetic per row is exactly that of ``block_forward``.
    """
    p = f"{prefix}{layer}."
    x = np.asarray(x, F64)
    rows = np.asarray(rows)
    D = x.shape[1]
    y = layer_norm(x, wts[p + "ln1.weight"], wts[p + "ln1.bias"], eps)
    W = np.asarray(wts[p + "attn_qkv.weight"], F64)
    b = np.asarray(wts[p + "attn_qkv.bias"], F64)
    kv = y @ W[D:].T + b[D:]
    k, v = kv[:, :D], kv[:, D:]
    q = y[rows] @ W[:D].T + b[:D]
    q = apply_rope(_split_heads(q, n_head), COS[rows], SIN[rows])
    k = apply_rope(_split_heads(k, n_head), COS, SIN)
    o = attention_heads(q, k, _split_heads(v, n_head))
    o = o.transpose(1, 0, 2).reshape(len(rows), -1)
    xr = x[rows] + _linear(o, wts[p + "attn_out.weight"], wts[p + "attn_out.bias"])
    yr = layer_norm(xr, wts[p + "ln2.weight"], wts[p + "ln2.bias"], eps)
    g = gelu_erf(_linear(yr, wts[p + "ffn_up.weight"], wts[p + "ffn_up.bias"]))
    return xr + _linear(g, wts[p + "ffn_down.weight"], wts[p + "ffn_down.bias"])


# ----------------------------------------------------------------------------- encoder
def is_image(cfg, T: int) -> bool:
    """[N] §3 (2.1 encoder forward): a one-frame input takes the native image
    path (tubelet 1, patch_embed_img, mod_embed_img); Meta's code selects it by
    the frame count.  Models without that path (V-JEPA 2) take clips only."""
    return T == 1 and bool(getattr(cfg, "has_image_path", False))


def encoder_rope(cfg, T: int, H: int, W: int):
    tub = 1 if is_image(cfg, T) else cfg.tubelet
    gt, gh, gw = T // tub, H // cfg.patch, W // cfg.patch
    pos = token_positions(gt, gh, gw, cfg.rope_interpolate, cfg.rope_ref_grid)
    return rope_tables(pos, cfg.embed_dim // cfg.n_head, cfg.rope_layout, cfg.rope_theta)


def encoder_embed(cfg, wts, clip_u8):
    """Patch embedding (+ the 2.1 modality vector, [N] §3) of one clip, or of
    one image ``[1, H, W, 3]`` on the native image path: tubelet 1 with
    ``patch_embed_img`` (Conv3d weight ``[D, 3, 1, 16, 16]``, feature order
    c*256 + y*16 + x) and ``mod_embed_img`` ([N] §2 key map, §3)."""
    T = clip_u8.shape[0]
    if is_image(cfg, T):
        x = patch_embed(normalise_clip(clip_u8), wts["patch_embed_img.weight"], wts["patch_embed_img.bias"],
                        1, cfg.patch)
        if getattr(cfg, "has_mod_embed", False):
            x = x + np.asarray(wts["mod_embed_img"], F64)
        return x
    x = patch_embed(normalise_clip(clip_u8), wts["patch_embed.weight"], wts["patch_embed.bias"],
                    cfg.tubelet, cfg.patch)
    if getattr(cfg, "has_mod_embed", False):
        x = x + np.asarray(wts["mod_embed_video"], F64)
    return x


def encoder_forward(cfg, wts, clip_u8, n_layers: int | None = None, return_residual: bool = False, keep=None):
    """Encoder forward of ONE clip ``[T, H, W, 3]`` uint8.

    Returns dict: ``out`` = enc.norm(x) ``[N, D]`` (last_hidden_state),
    ``hier`` = list of hier_norm.k(x after block hier_layers[k]) ([N] §3,
    [H] Intermediate features), ``pooled`` = token mean of ``out``, and, if
    asked, ``residual`` = x before the final norm.

    ``keep`` (token ids) is the masked encoder forward ([H] Usage, "Predictor";
    Validation, the masked-encoder row): the embedded tokens are gathered at
    ``keep`` before the blocks, so attention sees only them, while RoPE keeps
    each token's true grid position; the rows follow the order of ``keep``.
    """
    T, H, W, _ = clip_u8.shape
    COS, SIN = encoder_rope(cfg, T, H, W)
    x = encoder_embed(cfg, wts, clip_u8)
    if keep is not None:
        keep = np.asarray(keep)
        x, COS, SIN = x[keep], COS[keep], SIN[keep]
    L = cfg.n_layer if n_layers is None else n_layers
    hier = []
    taps = list(getattr(cfg, "hier_layers", ()) or ())
    for i in range(L):
        x = block_forward(x, wts, i, cfg.n_head, cfg.ln_eps, COS, SIN)
        if i in taps:
            kk = taps.index(i)
            hier.append(layer_norm(x, wts[f"hier_norm.{kk}.weight"], wts[f"hier_norm.{kk}.bias"],
                                   cfg.ln_eps))
    out = layer_norm(x, wts["norm.weight"], wts["norm.bias"], cfg.ln_eps)
    res = {"out": out, "hier": hier, "pooled": out.mean(axis=0)}
    if return_residual:
        res["residual"] = x
    return res


# ----------------------------------------------------------------------------- predictor
def predictor_input(pcfg, pwts, enc_out, ids_ctx, ids_tgt, modality: str = "video"):
    """Predictor token sequence before its blocks ([N] §3 predictor forwards, §4.4).

    ctx = enc_out[ids_ctx] W_emb^T + b_emb; every target row is the mask token
    ``mask_tokens[mask_index % n_mask_tokens]``; the sequence is ctx then tgt.
    The 2.1 predictor then adds its own modality vector (``mod_embed_video``,
    or ``mod_embed_img`` for the image path) to every row.
    """
    ctx = _linear(np.asarray(enc_out, F64)[np.asarray(ids_ctx)], pwts["embed.weight"], pwts["embed.bias"])
    m = np.asarray(pwts["mask_tokens"], F64)[pcfg.mask_index % pcfg.n_mask_tokens]
    tgt = np.broadcast_to(m, (len(ids_tgt), m.shape[0]))
    z = np.concatenate([ctx, tgt], axis=0)
    if getattr(pcfg, "has_mod_embed", False):
        z = z + np.asarray(pwts[f"mod_embed_{'img' if modality == 'image' else 'video'}"], F64)
    return z


def predictor_outputs(pcfg, pwts, enc_out, ids_ctx, ids_tgt, grid, modality: str = "video"):
    """Masked predictor ([N] §2 key maps, §3 predictor forwards, §4.4).

    Blocks as the encoder's (head_dim 32, RoPE from the ids on the full
    encoder grid, no interpolation; tiled for V-JEPA 2, interleaved for 2.1),
    then pred.norm.  ``pred`` = pred.proj on the target rows; ``ctx`` =
    pred.proj_context on the context rows where the model has it (2.1), else
    None.  Context and target rows with the same id share a position.
    """
    gt, gh, gw = grid
    z = predictor_input(pcfg, pwts, enc_out, ids_ctx, ids_tgt, modality)
    ids = np.concatenate([np.asarray(ids_ctx), np.asarray(ids_tgt)])
    pos = grid_positions_from_ids(ids, gt, gh, gw)
    COS, SIN = rope_tables(pos, pcfg.embed_dim // pcfg.n_head, pcfg.rope_layout, pcfg.rope_theta)
    for i in range(pcfg.n_layer):
        z = block_forward(z, pwts, i, pcfg.n_head, pcfg.ln_eps, COS, SIN)
    z = layer_norm(z, pwts["norm.weight"], pwts["norm.bias"], pcfg.ln_eps)
    n_ctx = len(ids_ctx)
    out = {"pred": _linear(z[n_ctx:], pwts["proj.weight"], pwts["proj.bias"]), "ctx": None}
    if getattr(pcfg, "has_proj_context", False):
        out["ctx"] = _linear(z[:n_ctx], pwts["proj_context.weight"], pwts["proj_context.bias"])
    return out


def predictor_forward(pcfg, pwts, enc_out, ids_ctx, ids_tgt, grid, modality: str = "video"):
    """The target predictions of :func:`predictor_outputs`."""
    return predictor_outputs(pcfg, pwts, enc_out, ids_ctx, ids_tgt, grid, modality)["pred"]


# ----------------------------------------------------------------------------- attentive-pool head
def attentive_pool_forward(hcfg, hwts, enc_out):
    """Attentive-pool head and classifier of ONE clip ([N] §2, "Attentive-pool
    head - exact forward"; [N] §1 head row: 3 pool layers, 174 classes).

    x = enc_out (after enc.norm); n_layer pre-LN self-attention blocks with NO
    RoPE; then one cross-attention whose single query is the raw learned token
    head.query (not normalised), keys and values from ln_kv(x), separate q/k/v
    projections, softmax(q_h k_h^T / sqrt(head_dim)) v_h concatenated over the
    heads with no output projection; the residual is the raw query; then
    y += ffn_down(gelu(ffn_up(ln2(y)))); logits = y W_cls^T + b_cls with no
    final norm.  Returns ``pooled`` = y (the classifier input) and ``logits``.
    """
    x = np.asarray(enc_out, F64)
    N, D = x.shape
    hd = D // hcfg.n_head
    # no RoPE in the pool blocks: the identity rotation (COS 1, SIN 0)
    ones, zeros = np.ones((N, hd), F64), np.zeros((N, hd), F64)
    for i in range(hcfg.n_layer):
        x = block_forward(x, hwts, i, hcfg.n_head, hcfg.ln_eps, ones, zeros, prefix="head.blk.")
    q0 = np.asarray(hwts["head.query"], F64).reshape(1, D)
    kv = layer_norm(x, hwts["head.xattn.ln_kv.weight"], hwts["head.xattn.ln_kv.bias"], hcfg.ln_eps)
    q = _linear(q0, hwts["head.xattn.q.weight"], hwts["head.xattn.q.bias"])
    k = _linear(kv, hwts["head.xattn.k.weight"], hwts["head.xattn.k.bias"])
    v = _linear(kv, hwts["head.xattn.v.weight"], hwts["head.xattn.v.bias"])
    o = attention_heads(_split_heads(q, hcfg.n_head), _split_heads(k, hcfg.n_head), _split_heads(v, hcfg.n_head))
    o = o.transpose(1, 0, 2).reshape(1, D)             # heads concatenated; no output projection
    y = q0 + o                                         # the residual is the raw query
    yn = layer_norm(y, hwts["head.xattn.ln2.weight"], hwts["head.xattn.ln2.bias"], hcfg.ln_eps)
    y = y + _linear(gelu_erf(_linear(yn, hwts["head.xattn.ffn_up.weight"], hwts["head.xattn.ffn_up.bias"])),
                    hwts["head.xattn.ffn_down.weight"], hwts["head.xattn.ffn_down.bias"])
    logits = _linear(y, hwts["head.cls.weight"], hwts["head.cls.bias"])
    return {"pooled": y[0], "logits": logits[0]}
