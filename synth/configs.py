"""The five workloads: model geometry, clip shape, dtype and seed.

Geometry follows the hyper-parameter table of the V-JEPA 2 / 2.1 conversion
notes (§1): ViT-L/16 is D 1024, 24 layers, 16 heads, FFN 4096; ViT-B/16 is
D 768, 12 layers, 12 heads, FFN 3072; patch 16, tubelet 2, LN eps 1e-6, RoPE
theta 10000; V-JEPA 2 uses the tiled RoPE layout, V-JEPA 2.1 the interleaved
one with positions interpolated to a 16-wide reference grid; the masked
predictor is D 384, 12 layers, 12 heads, FFN 1536, output 1024, 10 mask
tokens.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional


@dataclass(frozen=True)
class PredictorConfig:
    embed_dim: int = 384
    n_layer: int = 12
    n_head: int = 12
    ffn_dim: int = 1536
    in_dim: int = 1024
    out_dim: int = 1024
    n_mask_tokens: int = 10
    mask_index: int = 1
    context_fraction: float = 0.5
    ln_eps: float = 1e-6
    rope_theta: float = 10000.0
    rope_layout: str = "tiled"
    has_mod_embed: bool = False     # 2.1: pred.mod_embed_video / pred.mod_embed_img on every row
    has_proj_context: bool = False  # 2.1: pred.proj_context on the context rows


# The V-JEPA 2.1 ViT-B/16 384 predictor (conversion notes §1 "pred.*" rows).
PREDICTOR_21 = PredictorConfig(in_dim=768, out_dim=1664, n_mask_tokens=8, rope_layout="interleaved",
                               has_mod_embed=True, has_proj_context=True)


@dataclass(frozen=True)
class HeadConfig:
    """Attentive-pool head + classifier (conversion notes §1 head row and §2
    "Attentive-pool head - exact forward"): the SSv2 ViT-L/16 classifier's
    head, 3 pre-LN self-attention pool blocks (16 heads, head_dim 64, no
    RoPE), one single-query cross-attention block, 174 classes.  The pool
    blocks' FFN width is 4 x D, the encoder's MLP ratio (the pages do not print
    it)."""
    embed_dim: int = 1024
    n_layer: int = 3
    n_head: int = 16
    ffn_dim: int = 4096
    n_classes: int = 174
    ln_eps: float = 1e-6


HEAD_SSV2 = HeadConfig()


@dataclass(frozen=True)
class EncoderConfig:
    name: str
    workload: str
    embed_dim: int
    n_layer: int
    n_head: int
    ffn_dim: int
    n_frames: int
    height: int
    width: int
    batch: int
    dtype: str                  # storage/compute dtype of matrices and activations
    rope_layout: str            # "tiled" | "interleaved"
    rope_interpolate: bool
    seed: int
    rope_ref_grid: int = 16
    hier_layers: tuple = ()
    has_mod_embed: bool = False
    has_image_path: bool = False  # 2.1 native image path: patch_embed_img (+ mod_embed_img) for 1-frame input
    patch: int = 16
    tubelet: int = 2
    ln_eps: float = 1e-6
    rope_theta: float = 10000.0
    predictor: Optional[PredictorConfig] = None

    @property
    def head_dim(self) -> int:
        return self.embed_dim // self.n_head

    def grid(self):
        tub = 1 if (self.n_frames == 1 and self.has_image_path) else self.tubelet
        return (self.n_frames // tub, self.height // self.patch, self.width // self.patch)

    def with_(self, **kw) -> "EncoderConfig":
        return replace(self, **kw)


def tokens_per_clip(cfg: EncoderConfig) -> int:
    gt, gh, gw = cfg.grid()
    return gt * gh * gw


CONFIGS = {
    "block-f32-4f128": EncoderConfig(
        name="block-f32-4f128", workload="single block + patch embed, fp32, D768 h12, 4f 128px (128 tokens), batch 1",
        embed_dim=768, n_layer=1, n_head=12, ffn_dim=3072, n_frames=4, height=128, width=128,
        batch=1, dtype="f32", rope_layout="tiled", rope_interpolate=False, seed=0),
    "vitb16-16f384-f16": EncoderConfig(
        name="vitb16-16f384-f16",
        workload="ViT-B/16 12L, fp16, interleaved interpolated RoPE, 16f 384px (4608 tokens), batch 1",
        embed_dim=768, n_layer=12, n_head=12, ffn_dim=3072, n_frames=16, height=384, width=384,
        batch=1, dtype="f16", rope_layout="interleaved", rope_interpolate=True, seed=1,
        has_mod_embed=True),
    "vitl16-16f256": EncoderConfig(
        name="vitl16-16f256", workload="ViT-L/16 24L, bf16, tiled RoPE, 16f 256px (2048 tokens/clip), batch 8",
        embed_dim=1024, n_layer=24, n_head=16, ffn_dim=4096, n_frames=16, height=256, width=256,
        batch=8, dtype="bf16", rope_layout="tiled", rope_interpolate=False, seed=2),
    "vitl16-64f256-pred": EncoderConfig(
        name="vitl16-64f256-pred", workload="ViT-L/16 24L, bf16, 64f 256px (8192 tokens), batch 1, + masked predictor",
        embed_dim=1024, n_layer=24, n_head=16, ffn_dim=4096, n_frames=64, height=256, width=256,
        batch=1, dtype="bf16", rope_layout="tiled", rope_interpolate=False, seed=3,
        predictor=PredictorConfig()),
    "vitb16-64f384": EncoderConfig(
        name="vitb16-64f384",
        workload="ViT-B/16 12L, bf16, interleaved interpolated RoPE, 64f 384px (18432 tokens), batch 1, hier taps",
        embed_dim=768, n_layer=12, n_head=12, ffn_dim=3072, n_frames=64, height=384, width=384,
        batch=1, dtype="bf16", rope_layout="interleaved", rope_interpolate=True, seed=4,
        hier_layers=(2, 5, 8, 11), has_mod_embed=True),
    # Not a configuration of the measured workload: the 2.1 native image path
    # (one 384 px frame, 576 tokens), the first row after it.
    "img384": EncoderConfig(
        name="img384", workload="ViT-B/16 12L 2.1 native image path, bf16, interleaved interpolated RoPE, "
        "1f 384px (576 tokens), batch 32",
        embed_dim=768, n_layer=12, n_head=12, ffn_dim=3072, n_frames=1, height=384, width=384,
        batch=32, dtype="bf16", rope_layout="interleaved", rope_interpolate=True, seed=5,
        hier_layers=(2, 5, 8, 11), has_mod_embed=True, has_image_path=True),
    # Not a configuration of the measured workload: the 2.1 predictor on the
    # 2.1 ViT-B/16 16f 384 px clip (4608 tokens, grid 8 x 24 x 24), the second
    # row after it.
    "pred21": EncoderConfig(
        name="pred21", workload="ViT-B/16 12L 2.1 encoder + 2.1 masked predictor (D384 L12 hd32, 8 mask tokens, "
        "out 1664, context projection), bf16, 16f 384px (4608 tokens), batch 1",
        embed_dim=768, n_layer=12, n_head=12, ffn_dim=3072, n_frames=16, height=384, width=384,
        batch=1, dtype="bf16", rope_layout="interleaved", rope_interpolate=True, seed=6,
        hier_layers=(2, 5, 8, 11), has_mod_embed=True, has_image_path=True, predictor=PREDICTOR_21),
}
