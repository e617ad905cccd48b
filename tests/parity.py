"""Parity metrics shared by the GPU tests.

Tolerances (stated once, used everywhere):
  * token maps of bf16/fp16 compute: per-token cosine mean >= 0.9999, worst
    token >= 0.999, rel_max = max|a-b| / max|b| <= 1e-2;
  * standalone fp32 RoPE and LayerNorm kernels: rel_max <= 1e-5;
  * fp32 compute (CUDA-core path, no TF32): rel_max <= 1e-4 plus the cosine
    bars (derived from fp32 rounding over reductions of length <= 4096:
    ~sqrt(4096) * 6e-8 * growth through the blocks, with margin).
"""
import numpy as np

COS_MEAN, COS_WORST, REL_16BIT = 0.9999, 0.999, 1e-2
REL_F32_KERNEL = 1e-5
REL_F32_PATH = 1e-4


def metrics(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    g = got.reshape(-1, got.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    cos = (g * r).sum(1) / np.maximum(np.linalg.norm(g, axis=1) * np.linalg.norm(r, axis=1), 1e-300)
    rel = float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-300))
    return {"cos_mean": float(cos.mean()), "cos_worst": float(cos.min()), "worst_row": int(cos.argmin()),
            "rel_max": rel}


def assert_close_16bit(got, ref, what=""):
    m = metrics(got, ref)
    assert m["cos_mean"] >= COS_MEAN and m["cos_worst"] >= COS_WORST and m["rel_max"] <= REL_16BIT, (what, m)
    return m


def assert_close_f32(got, ref, rel=REL_F32_PATH, what=""):
    m = metrics(got, ref)
    assert m["cos_mean"] >= COS_MEAN and m["cos_worst"] >= COS_WORST and m["rel_max"] <= rel, (what, m)
    return m
