"""Pins for the oracle's 3-D RoPE against what the pages fix.

Source: "V-JEPA 2 / 2.1 tensor maps and RoPE derivation", §1 and §4 (4.1 tiled,
4.2 interleaved, 4.3 interpolation, 4.4 predictor ids).
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def test_split_widths_match_pages():
    rows = _rows("rope_widths.txt")
    assert len(rows) == 2
    for hd, d, rot, passthru in (map(int, r[:4]) for r in rows):
        assert oracle.rope_split(hd) == d
        assert 3 * d == rot and hd - 3 * d == passthru
        pos = np.array([[3.0, 5.0, 7.0], [1.0, 2.0, 9.0]])
        for layout in ("tiled", "interleaved"):
            COS, SIN = oracle.rope_tables(pos, hd, layout)
            assert np.all(COS[:, rot:] == 1.0) and np.all(SIN[:, rot:] == 0.0)
            # rotated dims really rotate at these positions
            assert np.all(SIN[:, :rot] != 0.0)


def test_token_counts_match_pages():
    for fr, H, W, n in (map(int, r[:4]) for r in _rows("token_counts.txt")):
        pos = oracle.token_positions(fr // 2, H // 16, W // 16)
        assert pos.shape == (n, 3)


def test_token_order_is_t_major():
    gt, gh, gw = 3, 4, 5
    pos = oracle.token_positions(gt, gh, gw)
    i = 0
    for t in range(gt):
        for h in range(gh):
            for w in range(gw):
                assert tuple(pos[i]) == (t, h, w)
                i += 1


def _elementwise_tiled(x, pos, hd, theta=10000.0):
    """The §4.1 element-wise formula, written per element with the printed
    index rule omega_{j mod (d/2)} for dim j of each axis segment."""
    d = oracle.rope_split(hd)
    half = d // 2
    out = list(x)
    for a in range(3):
        for k in range(half):
            j0, j1 = a * d + 2 * k, a * d + 2 * k + 1
            w0 = 1.0 / theta ** (((2 * k) % half) / half)
            w1 = 1.0 / theta ** (((2 * k + 1) % half) / half)
            out[j0] = x[j0] * math.cos(pos[a] * w0) - x[j1] * math.sin(pos[a] * w0)
            out[j1] = x[j1] * math.cos(pos[a] * w1) + x[j0] * math.sin(pos[a] * w1)
    return np.array(out)


def _elementwise_interleaved(x, pos, hd, theta=10000.0):
    """§4.2: each pair (2k, 2k+1) rotated by the angle pos * omega_k."""
    d = oracle.rope_split(hd)
    half = d // 2
    out = list(x)
    for a in range(3):
        for k in range(half):
            j0, j1 = a * d + 2 * k, a * d + 2 * k + 1
            ang = pos[a] * (1.0 / theta ** (k / half))
            out[j0] = x[j0] * math.cos(ang) - x[j1] * math.sin(ang)
            out[j1] = x[j1] * math.cos(ang) + x[j0] * math.sin(ang)
    return np.array(out)


@pytest.mark.parametrize("hd", [64, 32])
@pytest.mark.parametrize("layout", ["tiled", "interleaved"])
def test_elementwise_formula(hd, layout):
    rng = np.random.default_rng(1)
    ref = _elementwise_tiled if layout == "tiled" else _elementwise_interleaved
    for pos in ([3.0, 5.0, 7.0], [0.0, 15.0, 1.5], [31.0, 0.0, 11.25]):
        x = rng.standard_normal(hd)
        COS, SIN = oracle.rope_tables(np.array([pos]), hd, layout)
        got = oracle.apply_rope(x[None, :], COS, SIN)[0]
        np.testing.assert_allclose(got, ref(x, pos, hd), rtol=0, atol=1e-13)


def test_closed_form_unit_vector_distinguishes_layouts():
    # x = e_0 at t position 1: out[0] = cos(1 * omega_0) = cos 1 in both layouts;
    # out[1] = sin(omega_1) (tiled: dim 1 uses omega_{1 mod 10} = 10000^-0.1)
    # or sin(omega_0) = sin 1 (interleaved: the pair shares omega_0).
    x = np.zeros((1, 64)); x[0, 0] = 1.0
    pos = np.array([[1.0, 0.0, 0.0]])
    t = oracle.apply_rope(x, *oracle.rope_tables(pos, 64, "tiled"))[0]
    i = oracle.apply_rope(x, *oracle.rope_tables(pos, 64, "interleaved"))[0]
    assert t[0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert t[1] == pytest.approx(math.sin(10000.0 ** -0.1), abs=1e-15)
    assert i[0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert i[1] == pytest.approx(math.sin(1.0), abs=1e-15)
    assert np.all(t[2:] == 0.0) and np.all(i[2:] == 0.0)


@pytest.mark.parametrize("hd", [64, 32])
def test_tiled_is_interleaved_permuted(hd):
    # tiled = repeat(f, 2), interleaved = repeat_interleave(f, 2): within each
    # axis segment column j of the tiled table is column 2*(j mod d/2) + j//(d/2)
    # of the interleaved one.
    d = oracle.rope_split(hd)
    half = d // 2
    pos = oracle.token_positions(4, 5, 6).astype(float) * 1.3
    Ct, St = oracle.rope_tables(pos, hd, "tiled")
    Ci, Si = oracle.rope_tables(pos, hd, "interleaved")
    for a in range(3):
        for j in range(d):
            s = 2 * (j % half) + j // half
            np.testing.assert_array_equal(Ct[:, a * d + j], Ci[:, a * d + s])
            np.testing.assert_array_equal(St[:, a * d + j], Si[:, a * d + s])


@pytest.mark.parametrize("hd", [64, 32])
def test_interleaved_is_rotation_tiled_is_not(hd):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((50, hd))
    pos = rng.uniform(0, 20, size=(50, 3))
    xi = oracle.apply_rope(x, *oracle.rope_tables(pos, hd, "interleaved"))
    np.testing.assert_allclose(np.linalg.norm(xi, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    xt = oracle.apply_rope(x, *oracle.rope_tables(pos, hd, "tiled"))
    assert np.max(np.abs(np.linalg.norm(xt, axis=1) / np.linalg.norm(x, axis=1) - 1)) > 1e-3


def test_interleaved_relative_position():
    rng = np.random.default_rng(3)
    hd = 64
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)
    p, pp = np.array([2.0, 3.0, 4.0]), np.array([7.0, 1.0, 9.5])
    delta = np.array([5.0, -2.0, 3.25])

    def dot(a, b):
        ra = oracle.apply_rope(q[None], *oracle.rope_tables(a[None], hd, "interleaved"))[0]
        rb = oracle.apply_rope(k[None], *oracle.rope_tables(b[None], hd, "interleaved"))[0]
        return ra @ rb

    assert dot(p, pp) == pytest.approx(dot(p + delta, pp + delta), rel=1e-12, abs=1e-12)
    # ... and the tiled layout does not have the property
    def dot_t(a, b):
        ra = oracle.apply_rope(q[None], *oracle.rope_tables(a[None], hd, "tiled"))[0]
        rb = oracle.apply_rope(k[None], *oracle.rope_tables(b[None], hd, "tiled"))[0]
        return ra @ rb
    assert abs(dot_t(p, pp) - dot_t(p + delta, pp + delta)) > 1e-6


@pytest.mark.parametrize("layout", ["tiled", "interleaved"])
def test_position_zero_is_identity(layout):
    x = np.random.default_rng(4).standard_normal((3, 64))
    COS, SIN = oracle.rope_tables(np.zeros((3, 3)), 64, layout)
    np.testing.assert_array_equal(oracle.apply_rope(x, COS, SIN), x)


def test_interpolation_factors_match_pages():
    for n, num, den in (map(int, r[:3]) for r in _rows("rope_interp.txt")):
        pos = oracle.token_positions(2, n, n, interpolate=True, ref_grid=16)
        h = pos[:, 1].reshape(2, n, n)[0, :, 0]
        np.testing.assert_allclose(h, np.arange(n) * num / den, rtol=0, atol=1e-13)
        assert h[-1] == pytest.approx(15.0, abs=1e-12)
        # time is never rescaled
        assert np.array_equal(pos[:, 0], np.repeat([0.0, 1.0], n * n))
    # 16-wide grid: identity
    a = oracle.token_positions(3, 16, 16, interpolate=True)
    b = oracle.token_positions(3, 16, 16, interpolate=False)
    np.testing.assert_allclose(a, b, atol=1e-13)
    with pytest.raises(ValueError):
        oracle.token_positions(2, 1, 5, interpolate=True)


def test_predictor_ids_decode_like_encoder_grid():
    ids = np.array([0, 1, 255, 256, 8191])
    pos = oracle.grid_positions_from_ids(ids, 32, 16, 16)
    full = oracle.token_positions(32, 16, 16)
    np.testing.assert_array_equal(pos, full[ids])


def test_wrong_layout_negative_control():
    # Swapping the layout must move RoPE'd queries well beyond rounding noise
    # (the pages' end-to-end control drops the cosine to 0.63 / 0.91).
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2048, 64))
    pos = oracle.token_positions(8, 16, 16)
    a = oracle.apply_rope(q, *oracle.rope_tables(pos, 64, "tiled"))
    b = oracle.apply_rope(q, *oracle.rope_tables(pos, 64, "interleaved"))
    assert np.max(np.abs(a - b)) / np.max(np.abs(a)) > 0.1
