"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This module holds no arithmetic of the encoder itself: it only draws numbers.
Both sides of every parity check (the CPU oracle and the CUDA library) receive
exactly the arrays produced here, so a disagreement between them can never
come from the inputs.

Generator (counter based, so any element can be produced independently):

* splitmix64 finaliser ``mix64`` applied to ``key + (i + 1) * GOLDEN`` gives the
  i-th 64-bit draw of a stream; ``key = mix64(seed * GOLDEN ^ stream_id)``.
* Uniform bytes take the top 8 bits of a draw.
* Normals use Box-Muller on two consecutive draws mapped to (0, 1].

Weights follow the workloads' recipe: 2-D matrices, modality and mask-token
vectors ~ N(0, 0.02); biases 0; LayerNorm weight 1 / bias 0.  Matrices are
rounded (round-to-nearest-even) to the storage dtype before either side sees
them, and both sides compute from the rounded values.
"""
from __future__ import annotations

import numpy as np

from .configs import CONFIGS, HEAD_SSV2, PREDICTOR_21, EncoderConfig, HeadConfig, PredictorConfig, tokens_per_clip

__all__ = [
    "GOLDEN", "CONFIGS", "PREDICTOR_21", "HEAD_SSV2", "EncoderConfig", "HeadConfig", "PredictorConfig",
    "tokens_per_clip", "tensor_names_head", "head_weights",
    "mix64", "draws_u64", "uniform_u8", "normal", "round_to_dtype",
    "bf16_bits", "f16_bits", "bits_to_f32",
    "encoder_weights", "predictor_weights", "clip_u8", "context_target_split",
    "tensor_names_encoder", "tensor_names_predictor",
]

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def mix64(z):
    """splitmix64 output function (Steele, Lea, Flood 2014) on uint64 arrays."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.uint64(seed) * GOLDEN
    return mix64(base ^ np.uint64(stream & 0xFFFFFFFFFFFFFFFF))[()]


def _mix64_inplace(z: np.ndarray, tmp: np.ndarray) -> np.ndarray:
    # splitmix64 output function on a uint64 array, in place (same values as mix64)
    np.right_shift(z, np.uint64(30), out=tmp); np.bitwise_xor(z, tmp, out=z); np.multiply(z, _M1, out=z)
    np.right_shift(z, np.uint64(27), out=tmp); np.bitwise_xor(z, tmp, out=z); np.multiply(z, _M2, out=z)
    np.right_shift(z, np.uint64(31), out=tmp); np.bitwise_xor(z, tmp, out=z)
    return z


_CHUNK = 1 << 18


def draws_u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Draws ``start .. start+n-1`` of stream ``stream`` under ``seed``."""
    key = _stream_key(seed, stream)
    out = np.empty(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for c0 in range(0, n, _CHUNK):
            c1 = min(n, c0 + _CHUNK)
            z = out[c0:c1]
            z[:] = np.arange(start + c0 + 1, start + c1 + 1, dtype=np.uint64)
            np.multiply(z, GOLDEN, out=z)
            np.add(z, key, out=z)
            _mix64_inplace(z, np.empty_like(z))
    return out


def uniform_u8(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` bytes uniform on 0..255 inclusive."""
    return (draws_u64(seed, stream, n) >> np.uint64(56)).astype(np.uint8)


def normal(seed: int, stream: int, n: int, std: float) -> np.ndarray:
    """``n`` samples of N(0, std^2) in float64 (Box-Muller on draw pairs)."""
    m = (n + 1) // 2
    d = draws_u64(seed, stream, 2 * m)
    z = np.empty(2 * m, dtype=np.float64)
    half = _CHUNK // 2
    for p0 in range(0, m, half):
        p1 = min(m, p0 + half)
        u = ((d[2 * p0:2 * p1] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        a = 2.0 * np.pi * u[1::2]
        z[2 * p0:2 * p1:2] = r * np.cos(a)
        z[2 * p0 + 1:2 * p1:2] = r * np.sin(a)
    return z[:n] * std


# --------------------------------------------------------------------------- dtype rounding
def bf16_bits(x) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
        return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def f16_bits(x) -> np.ndarray:
    """float32 -> IEEE half bit patterns, round to nearest even."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Stored 16-bit patterns (or float32 values) back to float32 values."""
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    return np.asarray(bits, dtype=np.float32)


def round_to_dtype(x, dtype: str) -> np.ndarray:
    """Round float values to the storage dtype; returns float32 values."""
    x32 = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bits_to_f32(bf16_bits(x32), "bf16").reshape(x32.shape)
    if dtype == "f16":
        return x32.astype(np.float16).astype(np.float32)
    return x32


# --------------------------------------------------------------------------- tensors
def tensor_names_encoder(cfg: EncoderConfig):
    """(name, shape, kind) in the fixed order the weight blob stores them.

    kind: 'mat' (N(0,0.02), storage dtype), 'vec' (N(0,0.02), fp32),
    'zero' (fp32 zeros), 'one' (fp32 ones).
    """
    D, F = cfg.embed_dim, cfg.ffn_dim
    kdim = 3 * cfg.tubelet * cfg.patch * cfg.patch
    out = [("patch_embed.weight", (D, kdim), "mat"), ("patch_embed.bias", (D,), "zero")]
    if cfg.has_mod_embed:
        out.append(("mod_embed_video", (D,), "vec"))
    for i in range(cfg.n_layer):
        p = f"blk.{i}."
        out += [
            (p + "ln1.weight", (D,), "one"), (p + "ln1.bias", (D,), "zero"),
            (p + "attn_qkv.weight", (3 * D, D), "mat"), (p + "attn_qkv.bias", (3 * D,), "zero"),
            (p + "attn_out.weight", (D, D), "mat"), (p + "attn_out.bias", (D,), "zero"),
            (p + "ln2.weight", (D,), "one"), (p + "ln2.bias", (D,), "zero"),
            (p + "ffn_up.weight", (F, D), "mat"), (p + "ffn_up.bias", (F,), "zero"),
            (p + "ffn_down.weight", (D, F), "mat"), (p + "ffn_down.bias", (D,), "zero"),
        ]
    out += [("norm.weight", (D,), "one"), ("norm.bias", (D,), "zero")]
    for k in range(len(cfg.hier_layers)):
        out += [(f"hier_norm.{k}.weight", (D,), "one"), (f"hier_norm.{k}.bias", (D,), "zero")]
    if cfg.has_image_path:      # appended last, so no other tensor's stream moves
        out += [("patch_embed_img.weight", (D, 3 * cfg.patch * cfg.patch), "mat"), ("patch_embed_img.bias", (D,), "zero")]
        if cfg.has_mod_embed:
            out.append(("mod_embed_img", (D,), "vec"))
    return out


def tensor_names_predictor(pc: PredictorConfig):
    D, F = pc.embed_dim, pc.ffn_dim
    out = [("embed.weight", (D, pc.in_dim), "mat"), ("embed.bias", (D,), "zero"),
           ("mask_tokens", (pc.n_mask_tokens, D), "vec")]
    for i in range(pc.n_layer):
        p = f"blk.{i}."
        out += [
            (p + "ln1.weight", (D,), "one"), (p + "ln1.bias", (D,), "zero"),
            (p + "attn_qkv.weight", (3 * D, D), "mat"), (p + "attn_qkv.bias", (3 * D,), "zero"),
            (p + "attn_out.weight", (D, D), "mat"), (p + "attn_out.bias", (D,), "zero"),
            (p + "ln2.weight", (D,), "one"), (p + "ln2.bias", (D,), "zero"),
            (p + "ffn_up.weight", (F, D), "mat"), (p + "ffn_up.bias", (F,), "zero"),
            (p + "ffn_down.weight", (D, F), "mat"), (p + "ffn_down.bias", (D,), "zero"),
        ]
    out += [("norm.weight", (D,), "one"), ("norm.bias", (D,), "zero"),
            ("proj.weight", (pc.out_dim, D), "mat"), ("proj.bias", (pc.out_dim,), "zero")]
    # 2.1 additions, appended last so no other tensor's stream moves
    if pc.has_mod_embed:
        out += [("mod_embed_video", (D,), "vec"), ("mod_embed_img", (D,), "vec")]
    if pc.has_proj_context:
        out += [("proj_context.weight", (pc.out_dim, D), "mat"), ("proj_context.bias", (pc.out_dim,), "zero")]
    return out


def tensor_names_head(hc: HeadConfig):
    """The attentive-pool head's tensors in blob order (conversion notes §2
    head rows): the learned query, the pool blocks (encoder block layout, q/k/v
    fused), the cross-attention block (ln_kv, separate q/k/v projections, ln2,
    MLP) and the classifier."""
    D, F, C = hc.embed_dim, hc.ffn_dim, hc.n_classes
    out = [("head.query", (D,), "vec")]
    for i in range(hc.n_layer):
        p = f"head.blk.{i}."
        out += [
            (p + "ln1.weight", (D,), "one"), (p + "ln1.bias", (D,), "zero"),
            (p + "attn_qkv.weight", (3 * D, D), "mat"), (p + "attn_qkv.bias", (3 * D,), "zero"),
            (p + "attn_out.weight", (D, D), "mat"), (p + "attn_out.bias", (D,), "zero"),
            (p + "ln2.weight", (D,), "one"), (p + "ln2.bias", (D,), "zero"),
            (p + "ffn_up.weight", (F, D), "mat"), (p + "ffn_up.bias", (F,), "zero"),
            (p + "ffn_down.weight", (D, F), "mat"), (p + "ffn_down.bias", (D,), "zero"),
        ]
    x = "head.xattn."
    out += [(x + "ln_kv.weight", (D,), "one"), (x + "ln_kv.bias", (D,), "zero"),
            (x + "q.weight", (D, D), "mat"), (x + "q.bias", (D,), "zero"),
            (x + "k.weight", (D, D), "mat"), (x + "k.bias", (D,), "zero"),
            (x + "v.weight", (D, D), "mat"), (x + "v.bias", (D,), "zero"),
            (x + "ln2.weight", (D,), "one"), (x + "ln2.bias", (D,), "zero"),
            (x + "ffn_up.weight", (F, D), "mat"), (x + "ffn_up.bias", (F,), "zero"),
            (x + "ffn_down.weight", (D, F), "mat"), (x + "ffn_down.bias", (D,), "zero"),
            ("head.cls.weight", (C, D), "mat"), ("head.cls.bias", (C,), "zero")]
    return out


def _one_tensor(args):
    idx, (name, shape, kind), seed, storage, stream_base, std, overrides = args
    for suffix, s in overrides.items():
        if name.endswith(suffix):
            std = s
    n = int(np.prod(shape))
    if kind == "mat":
        v = round_to_dtype(normal(seed, stream_base + idx, n, std), storage)
    elif kind == "vec":
        v = normal(seed, stream_base + idx, n, std).astype(np.float32)
    elif kind == "zero":
        v = np.zeros(n, np.float32)
    else:
        v = np.ones(n, np.float32)
    return name, v.reshape(shape)


def _materialise(names, seed, storage, stream_base, std=0.02, overrides=None):
    # Tensors are independent streams, so they are drawn in parallel threads
    # (numpy releases the GIL); the values do not depend on the schedule.
    import concurrent.futures as cf
    import os
    jobs = [(i, nk, seed, storage, stream_base, std, dict(overrides or {})) for i, nk in enumerate(names)]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        return dict(ex.map(_one_tensor, jobs))


def encoder_weights(cfg: EncoderConfig, std_overrides: dict | None = None) -> dict:
    """Random-init encoder weights (float32 arrays holding storage-dtype values).

    ``std_overrides`` maps a tensor-name suffix (e.g. ``"attn_qkv.weight"``) to
    the standard deviation its normal draws use instead of 0.02; the draws
    come from the same streams, only scaled."""
    return _materialise(tensor_names_encoder(cfg), cfg.seed, cfg.dtype, 1000, overrides=std_overrides)


def predictor_weights(cfg: EncoderConfig) -> dict:
    pc = cfg.predictor
    return _materialise(tensor_names_predictor(pc), cfg.seed, cfg.dtype, 500000)


def head_weights(hc: HeadConfig, seed: int, dtype: str, std_overrides: dict | None = None,
                 kind_overrides: dict | None = None) -> dict:
    """Random-init attentive-pool head weights: matrices and the query
    N(0, 0.02) (matrices rounded to ``dtype``), biases 0, LayerNorm 1 / 0;
    streams of their own (base 700000), so no encoder or predictor tensor
    moves.  ``std_overrides`` maps a name suffix to another standard
    deviation; ``kind_overrides`` a name suffix to another kind ("mat",
    "vec", "zero", "one"), e.g. non-zero biases."""
    names = tensor_names_head(hc)
    if kind_overrides:
        names = [(n, sh, next((k for suf, k in kind_overrides.items() if n.endswith(suf)), kind))
                 for n, sh, kind in names]
    return _materialise(names, seed, dtype, 700000, overrides=std_overrides)


def clip_u8(cfg: EncoderConfig, batch: int | None = None, first_clip: int = 0) -> np.ndarray:
    """Clips ``[B, T, H, W, 3]`` uint8, uniform on 0..255; clip b is its own stream."""
    B = cfg.batch if batch is None else batch
    n = cfg.n_frames * cfg.height * cfg.width * 3
    out = np.empty((B, cfg.n_frames, cfg.height, cfg.width, 3), np.uint8)
    for b in range(B):
        out[b] = uniform_u8(cfg.seed, 7 + first_clip + b, n).reshape(out.shape[1:])
    return out


def context_target_split(cfg: EncoderConfig):
    """Seeded random half/half split of the clip's token ids (each part sorted)."""
    n = tokens_per_clip(cfg)
    keys = draws_u64(cfg.seed, 900001, n)
    perm = np.argsort(keys, kind="stable")
    n_ctx = int(round(n * cfg.predictor.context_fraction))
    ctx = np.sort(perm[:n_ctx]).astype(np.int32)
    tgt = np.sort(perm[n_ctx:]).astype(np.int32)
    return ctx, tgt
