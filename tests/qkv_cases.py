"""Cases of the fused QKV projection + 3-D RoPE, shared by the GPU parity test
(tests/test_gpu_qkv_rope.py) and the CPU negative controls
(tests/test_qkv_rope_controls.py); and the two small encoders with sharp
attention (SHARP_MODELS) that the end-to-end GPU test and its controls share.

Each case draws seeded inputs (rows A, the fused weight W = [Wq; Wk; Wv], a
non-zero bias, so a RoPE applied before the bias would show) and, where the
rows are a subset of the grid, one id list per clip.  ``reference`` is the
oracle's composition ("V-JEPA 2 / 2.1 tensor maps and RoPE derivation", §2
fused attn_qkv, §4 RoPE after the bias on q and k, §4.1/4.2 layouts, §4.3
interpolation, §4.4 positions from ids) in float64, with switches that plant
the mistakes a RoPE epilogue can make: the other layout, interpolation on or
off, positions taken from the row index instead of the ids, and the h and w
axes swapped.
"""
import numpy as np

import oracle
import synth

# name -> dtype, width D, heads, clips, grid (t, h, w), layout, interpolation,
# ids: None (row r is token r mod n), "unsorted" (each clip keeps `keep`
# random grid cells in random order) or "predictor" (context ids then target
# ids, each half sorted)
CASES = {
    "bf16-hd64-tiled": dict(dtype="bf16", D=256, H=4, batch=2, grid=(2, 16, 16), layout="tiled", interp=False),
    "f16-hd64-interleaved-interp-ragged": dict(dtype="f16", D=384, H=6, batch=2, grid=(3, 20, 7),
                                               layout="interleaved", interp=True),
    "bf16-hd64-interleaved-plain": dict(dtype="bf16", D=256, H=4, batch=2, grid=(2, 12, 10), layout="interleaved",
                                        interp=False),
    "bf16-hd32-tiled-ragged": dict(dtype="bf16", D=256, H=8, batch=3, grid=(3, 5, 9), layout="tiled", interp=False),
    "bf16-hd32-interleaved-interp": dict(dtype="bf16", D=384, H=12, batch=2, grid=(2, 6, 8), layout="interleaved",
                                         interp=True),
    "bf16-hd64-tiled-ids": dict(dtype="bf16", D=256, H=4, batch=2, grid=(4, 16, 16), layout="tiled", interp=False,
                                ids="unsorted", keep=600),
    "bf16-hd64-interleaved-interp-ids": dict(dtype="bf16", D=256, H=4, batch=2, grid=(4, 12, 20),
                                             layout="interleaved", interp=True, ids="unsorted", keep=500),
    "bf16-hd32-tiled-predictor-ids": dict(dtype="bf16", D=384, H=12, batch=1, grid=(8, 6, 8), layout="tiled",
                                          interp=False, ids="predictor"),
    # 15 clips x 1024 tokens: 180 CTA-pair tiles of 256 x 256 for 76 resident
    # pairs, so the last 28 tiles run as half-width units
    "bf16-hd64-tiled-tail-wave": dict(dtype="bf16", D=256, H=4, batch=15, grid=(4, 16, 16), layout="tiled",
                                      interp=False),
    "f32-hd64-tiled": dict(dtype="f32", D=256, H=4, batch=2, grid=(2, 8, 8), layout="tiled", interp=False),
    "f32-hd32-interleaved-interp-ids": dict(dtype="f32", D=256, H=8, batch=2, grid=(2, 6, 10),
                                            layout="interleaved", interp=True, ids="unsorted", keep=70),
}


def n_tokens(case):
    gt, gh, gw = case["grid"]
    kind = case.get("ids")
    return case["keep"] if kind == "unsorted" else gt * gh * gw


def make_inputs(case, seed):
    """A [batch*n, D], W [3D, D] (rounded to the case's dtype), bias [3D] and
    ids (int32 [batch*n] or None)."""
    rng = np.random.default_rng(seed)
    D, B, dt = case["D"], case["batch"], case["dtype"]
    n = n_tokens(case)
    A = synth.round_to_dtype(rng.standard_normal((B * n, D)), dt).astype(np.float64)
    W = synth.round_to_dtype(rng.standard_normal((3 * D, D)) * 0.06, dt).astype(np.float64)
    b = rng.standard_normal(3 * D).astype(np.float32).astype(np.float64) * 0.5
    gt, gh, gw = case["grid"]
    cells = gt * gh * gw
    kind = case.get("ids")
    ids = None
    if kind == "unsorted":
        ids = np.concatenate([rng.choice(cells, n, replace=False) for _ in range(B)]).astype(np.int32)
    elif kind == "predictor":
        perm = rng.permutation(cells)
        ctx, tgt = np.sort(perm[: cells // 2]), np.sort(perm[cells // 2:])
        ids = np.tile(np.concatenate([ctx, tgt]), B).astype(np.int32)
    return A, W, b, ids


def positions(case, ids, interp=None, mode="ids"):
    """Per-row (t, h, w) positions [batch*n, 3] of the case.  mode "ids": the
    row's own id (or r mod n without ids); "row": r mod n even when ids are
    given; "hw_swapped": the h and w grid axes exchanged."""
    gt, gh, gw = case["grid"]
    interp = case["interp"] if interp is None else interp
    n, B = n_tokens(case), case["batch"]
    if mode == "hw_swapped":
        # the grid read as (t, w, h): cell ids decode with the wrong axis sizes
        allpos = oracle.token_positions(gt, gw, gh, interp, 16)
    else:
        allpos = oracle.token_positions(gt, gh, gw, interp, 16)
    rows = np.arange(B * n) % n
    if ids is not None and mode != "row":
        rows = np.minimum(ids, len(allpos) - 1)
    return allpos[rows]


def reference(case, A, W, b, ids, layout=None, interp=None, mode="ids"):
    """q, k, v as [batch*H, n, hd] float64 (q and k rotated, not scaled)."""
    D, H, B = case["D"], case["H"], case["batch"]
    hd, n = D // H, n_tokens(case)
    qkv = A @ W.T + b                                         # [B*n, 3D]: rows q;k;v of the fused weight
    pos = positions(case, ids, interp, mode)
    COS, SIN = oracle.rope_tables(pos, hd, case["layout"] if layout is None else layout)   # [B*n, hd]
    out = []
    for s in range(3):
        t = qkv[:, s * D:(s + 1) * D].reshape(B * n, H, hd)
        if s < 2:
            t = oracle.apply_rope(t, COS[:, None, :], SIN[:, None, :])
        out.append(t.reshape(B, n, H, hd).transpose(0, 2, 1, 3).reshape(B * H, n, hd))
    return out


# Small encoders whose attention is sharp enough for the RoPE to matter end to
# end.  With N(0, 0.02) weights the attention logits have std ~0.1 and the
# output barely depends on the positions; attn_qkv.weight drawn at std
# sqrt(3 / D) (0.108 at D 256) gives logits of std ~3 (LayerNorm'd rows of
# unit variance: q and k elements of variance D std^2 = 3).
SHARP_QKV_STD = 0.108
SHARP_MODELS = {
    # V-JEPA 2 geometry: tiled RoPE, head_dim 32, N = 3*5*9 = 135 (ragged against 128-row tiles)
    "v2-hd32-sharp": synth.CONFIGS["vitl16-16f256"].with_(embed_dim=256, n_head=8, ffn_dim=512, n_layer=2, n_frames=6,
                                               height=80, width=144, batch=2),
    # 2.1 geometry: interleaved RoPE interpolated to the 16-grid, modality vector, taps; N = 2*6*8 = 96
    "b21-hd64-sharp": synth.CONFIGS["vitb16-64f384"].with_(embed_dim=256, n_head=4, ffn_dim=1024, n_layer=3, n_frames=4,
                                                height=96, width=128, batch=2, hier_layers=(0, 2)),
}


def sharp_weights(cfg):
    return synth.encoder_weights(cfg, {"attn_qkv.weight": SHARP_QKV_STD})
