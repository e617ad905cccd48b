"""Pins for the oracle's layers against library routines, brute force and closed forms."""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_layer_norm_matches_torch_and_brute_force():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((37, 96)) * 3 + 1.5
    w, b = rng.standard_normal(96), rng.standard_normal(96)
    got = oracle.layer_norm(x, w, b, 1e-6)
    ref = Fn.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), torch.from_numpy(b), 1e-6).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # brute force with exactly rounded sums on a tiny case
    xs = rng.standard_normal((3, 8))
    for r in range(3):
        row = [float(v) for v in xs[r]]
        mu = math.fsum(row) / 8
        var = math.fsum((v - mu) ** 2 for v in row) / 8
        exp = [(v - mu) / math.sqrt(var + 1e-6) for v in row]
        np.testing.assert_allclose(oracle.layer_norm(xs[r:r + 1], np.ones(8), np.zeros(8), 1e-6)[0],
                                   exp, rtol=0, atol=1e-14)


def test_layer_norm_large_mean_is_centred():
    # centred two-pass variance: a large common offset must not change the result
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 64))
    a = oracle.layer_norm(x, np.ones(64), np.zeros(64), 1e-6)
    b = oracle.layer_norm(x + 1e4, np.ones(64), np.zeros(64), 1e-6)
    np.testing.assert_allclose(a, b, atol=1e-9)


def test_gelu_is_exact_erf():
    z = np.linspace(-8, 8, 1001)
    exp = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in z])
    np.testing.assert_allclose(oracle.gelu_erf(z), exp, rtol=0, atol=1e-15)
    ref = Fn.gelu(torch.from_numpy(z), approximate="none").numpy()
    np.testing.assert_allclose(oracle.gelu_erf(z), ref, rtol=0, atol=1e-14)
    # not the tanh approximation
    tanh = Fn.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    assert np.max(np.abs(oracle.gelu_erf(z) - tanh)) > 1e-4


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(2)
    q, k, v = (rng.standard_normal((3, 70, 64)) * 2 for _ in range(3))
    got = oracle.attention_heads(q, k, v)
    ref = Fn.scaled_dot_product_attention(*(torch.from_numpy(t) for t in (q, k, v))).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((1, 5, 4)) for _ in range(3))
    got = oracle.attention_heads(q, k, v)[0]
    for i in range(5):
        s = [sum(q[0, i, d] * k[0, j, d] for d in range(4)) / 2.0 for j in range(5)]
        e = [math.exp(t) for t in s]
        z = math.fsum(e)
        for d in range(4):
            assert got[i, d] == pytest.approx(math.fsum(e[j] * v[0, j, d] for j in range(5)) / z, abs=1e-14)


def test_attention_identities():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((2, 9, 8))
    q = rng.standard_normal((2, 6, 8))
    k = np.broadcast_to(rng.standard_normal((2, 1, 8)), (2, 9, 8))
    # all keys equal -> uniform weights -> mean of v
    np.testing.assert_allclose(oracle.attention_heads(q, k, v), np.broadcast_to(v.mean(1, keepdims=True), (2, 6, 8)),
                               atol=1e-14)
    # permuting tokens (keys with their values, queries) permutes the output
    k = rng.standard_normal((2, 9, 8))
    qq = rng.standard_normal((2, 9, 8))
    perm = rng.permutation(9)
    a = oracle.attention_heads(qq, k, v)
    b = oracle.attention_heads(qq[:, perm], k[:, perm], v[:, perm])
    np.testing.assert_allclose(a[:, perm], b, atol=1e-13)


def test_normalisation_constants_and_form():
    rows = []
    with open(os.path.join(GOLDEN, "preprocess.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([float(t) for t in line.split()])
    assert tuple(r[1] for r in rows) == oracle.IMAGENET_MEAN
    assert tuple(r[2] for r in rows) == oracle.IMAGENET_STD
    clip = np.zeros((2, 1, 2, 3), np.uint8)
    clip[1] = 255
    x = oracle.normalise_clip(clip)
    assert x.shape == (3, 2, 1, 2)
    for c, mean, std in rows:
        c = int(c)
        assert x[c, 0, 0, 0] == pytest.approx(-mean / std, rel=1e-15)
        assert x[c, 1, 0, 1] == pytest.approx((1 - mean) / std, rel=1e-14)


def test_patch_embed_equals_conv3d():
    # The stored [D, 1536] matrix is the Conv3d kernel reshaped row-major; the
    # oracle's explicit tap sum must equal torch's Conv3d with stride = kernel.
    rng = np.random.default_rng(5)
    D = 24
    x = rng.standard_normal((3, 4, 32, 48))
    w = rng.standard_normal((D, 1536)) * 0.02
    b = rng.standard_normal(D)
    got = oracle.patch_embed(x, w, b)
    ref = Fn.conv3d(torch.from_numpy(x)[None], torch.from_numpy(w).reshape(D, 3, 2, 16, 16),
                    torch.from_numpy(b), stride=(2, 16, 16))[0]       # [D, 2, 2, 3]
    ref = ref.permute(1, 2, 3, 0).reshape(-1, D).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_patch_embed_equals_unfold_gemm():
    # The same map as a GEMM over rows P[i, c*512 + dt*256 + y*16 + x] built by
    # an index loop (the row layout the GPU path's unfold produces).
    rng = np.random.default_rng(6)
    D = 8
    x = rng.standard_normal((3, 2, 32, 16))
    w = rng.standard_normal((D, 1536))
    b = rng.standard_normal(D)
    gt, gh, gw = 1, 2, 1
    P = np.zeros((gt * gh * gw, 1536))
    for t in range(gt):
        for i in range(gh):
            for j in range(gw):
                row = (t * gh + i) * gw + j
                for c in range(3):
                    for dt in range(2):
                        for y in range(16):
                            for xx in range(16):
                                P[row, c * 512 + dt * 256 + y * 16 + xx] = x[c, 2 * t + dt, 16 * i + y, 16 * j + xx]
    np.testing.assert_allclose(oracle.patch_embed(x, w, b), P @ w.T + b, atol=1e-12)
