"""Runs and times one operation of the encoder at the ViT-L/16 batch-8 shapes.

    python -m video_vit_encoder_gb300.opbench OP [--reps R] [--warmup W]

OP is one of attention, qkv (the QKV GEMM with its RoPE epilogue), out_proj, ffn_up, ffn_down, layernorm, and
out_proj_f32 / out_proj_bf16 (the out_proj shape with a plain fp32 or 16-bit
store instead of the residual add), and predictor21: the whole V-JEPA 2.1
masked predictor (D 384, 12 blocks, head_dim 32, FFN 1536, out 1664, context
projection) on a 16-frame 384 px clip's 4608 tokens split 2304 / 2304, random
encoder tokens and weights; head: the SSv2 attentive-pool head and
classifier (3 pool blocks, 174 classes) on 8 x 2048 random encoder tokens;
patch_embed: normalise, unfold and patch-embed GEMM of 8 random 16 x 256 x 256
uint8 clips.  Encoder-op shapes:
8 clips x 2048 tokens = 16384 rows, D 1024, 16 heads (head_dim 64), FFN 4096,
bf16 operands.  Inputs are random (the values do not matter for timing).
Prints the mean time per launch (CUDA events) and the achieved rate.  Used
for single-kernel profiler captures (e.g. under ncu with -k and -c).
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import binding as jb
from ._lib import load

B, N, D, H, F = 8, 2048, 1024, 16, 4096
M = B * N


def _setup(op):
    g = torch.Generator(device="cuda").manual_seed(0)
    bf = torch.bfloat16

    def rnd(*shape, scale=1.0, dtype=bf):
        return (torch.randn(*shape, device="cuda", generator=g) * scale).to(dtype)

    if op == "attention":
        hd = D // H
        q, k = rnd(B * H, N, hd, scale=0.5), rnd(B * H, N, hd, scale=0.5)
        vt = rnd(B * H, hd, N)
        out = torch.empty(B, N, D, dtype=bf, device="cuda")
        return (lambda: jb.attention(q, k, vt, B, H, N, hd, out=out)), 4.0 * B * H * N * N * hd, "TFLOP/s"
    if op == "predictor21":
        import synth
        from . import binding
        pc = synth.PREDICTOR_21
        cfg = synth.CONFIGS["pred21"]
        pw = synth.predictor_weights(cfg)
        grid = cfg.grid()
        n = grid[0] * grid[1] * grid[2]
        ctx, tgt = synth.context_target_split(cfg)
        pred = binding.Predictor(pc, pw, cfg.dtype)
        enc = torch.randn(n, pc.in_dim, device="cuda", generator=g)
        ic, it = torch.from_numpy(ctx).cuda(), torch.from_numpy(tgt).cuda()
        pd, pf, pl = pc.embed_dim, pc.ffn_dim, pc.n_layer
        fl = (2 * len(ctx) * pc.in_dim * pd + pl * (2 * n * (4 * pd * pd + 2 * pd * pf) + 4 * n * n * pd)
              + 2 * n * pd * pc.out_dim)
        return (lambda: pred.predict(enc, ic, it, grid, modality="video", with_ctx=True)), fl, "TFLOP/s"
    if op == "qkv":
        # the fused QKV GEMM with its 3-D RoPE epilogue (tiled, 8 x 16 x 16 grid), head-major q/k and v^T
        A = rnd(M, D)
        W = rnd(3 * D, D, scale=0.02)
        bias = torch.zeros(3 * D, device="cuda")
        hd = D // H
        q = torch.empty(B * H, N, hd, dtype=bf, device="cuda")
        k = torch.empty_like(q)
        vt = torch.zeros(B * H, hd, N, dtype=bf, device="cuda")
        return (lambda: jb.qkv_rope(A, W, bias, B, N, H, (8, 16, 16), "tiled", out=(q, k, vt))), \
            2.0 * M * 3 * D * D, "TFLOP/s"
    if op == "head":
        # the SSv2 attentive-pool head + classifier on 8 clips x 2048 encoder tokens
        import synth
        from . import binding
        hc = synth.HEAD_SSV2
        head = binding.Head(hc, synth.head_weights(hc, 2, "bf16"), "bf16")
        x = torch.randn(B, N, D, device="cuda", generator=g)
        logits = torch.empty(B, hc.n_classes, device="cuda")
        F_ = hc.ffn_dim
        fl = (hc.n_layer * (2 * M * (4 * D * D + 2 * D * F_) + 4 * B * N * N * D)   # pool blocks
              + 4 * M * D * (D // 64) + 2 * B * (2 * D * D + 2 * D * F_ + hc.n_classes * D))
        return (lambda: head.forward(x, out=logits)), fl, "TFLOP/s"
    if op == "patch_embed":
        # normalise + tubelet unfold + patch-embed GEMM of 8 clips of 16 x 256 x 256 (jepa_encoder_embed)
        import synth
        from . import binding
        cfg = synth.CONFIGS["vitl16-16f256"].with_(n_layer=0)
        enc = binding.Encoder(cfg, synth.encoder_weights(cfg))
        clip = torch.randint(0, 256, (B, 16, 256, 256, 3), dtype=torch.uint8, device="cuda", generator=g)
        return (lambda: enc.embed(clip)), 2.0 * M * 1536 * D, "TFLOP/s"
    if op == "layernorm":
        x = rnd(M, D, dtype=torch.float32)
        w, b = torch.ones(D, device="cuda"), torch.zeros(D, device="cuda")
        y = torch.empty_like(x)
        return (lambda: jb.layernorm_f32(x, w, b, 1e-6, out=y)), 8.0 * M * D, "GB/s"
    shapes = {"out_proj": (D, D, 2), "ffn_up": (F, D, 3), "ffn_down": (D, F, 2),
              "out_proj_f32": (D, D, 1), "out_proj_bf16": (D, D, 0)}
    n, kdim, epi = shapes[op]
    A = rnd(M, kdim)
    W = rnd(n, kdim, scale=0.02)
    bias = torch.zeros(n, device="cuda")
    out = torch.empty(M, n, dtype=torch.float32 if epi in (1, 2) else bf, device="cuda").zero_()
    return (lambda: jb.linear(A, W, bias, epi, out=out)), 2.0 * M * n * kdim, "TFLOP/s"


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["attention", "qkv", "out_proj", "ffn_up", "ffn_down", "layernorm", "out_proj_f32",
                                   "out_proj_bf16", "predictor21", "head", "patch_embed"])
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    args = ap.parse_args(argv)
    load()
    fn, work, unit = _setup(args.op)
    for _ in range(args.warmup):
        fn()
    jb.ops_sync()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.reps):
        fn()
    e.record()
    torch.cuda.synchronize()
    jb.ops_sync()
    ms = s.elapsed_time(e) / max(args.reps, 1)
    rate = work / (ms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(f"{args.op}: {ms * 1e3:.1f} us/launch, {rate:.1f} {unit}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
