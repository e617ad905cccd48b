"""Single kernels through the C ABI against the oracle, element by element."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import REL_F32_KERNEL, assert_close_16bit, assert_close_f32, metrics

pytestmark = pytest.mark.gpu

TD = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def jg():
    import video_vit_encoder_gb300 as m
    m.load()
    return m


def _dev(a, dtype="f32"):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(TD[dtype]).cuda()


def _rounded(rng, shape, dtype, scale=1.0):
    return synth.round_to_dtype(rng.standard_normal(shape) * scale, dtype).astype(np.float64)


def test_wait_timeout_reports_and_context_survives(jg):
    from video_vit_encoder_gb300._lib import ERR_DEVICE_TIMEOUT
    assert jg.selftest_wait_timeout(200) == ERR_DEVICE_TIMEOUT
    x = torch.randn(8, 128, device="cuda")
    y = jg.layernorm_f32(x, torch.ones(128, device="cuda"), torch.zeros(128, device="cuda"), 1e-6)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    jg.ops_sync()


@pytest.mark.parametrize("rows,dim", [(1000, 768), (37, 1024), (5, 384), (0, 128)])
def test_layernorm_f32(jg, rows, dim):
    rng = np.random.default_rng(rows + dim)
    x = rng.standard_normal((rows, dim)) * 3 + rng.standard_normal((rows, 1)) * 2
    w, b = rng.standard_normal(dim), rng.standard_normal(dim)
    x32, w32, b32 = (np.float32(t) for t in (x, w, b))
    y = jg.layernorm_f32(_dev(x32), _dev(w32), _dev(b32), 1e-6).cpu().numpy()
    if rows == 0:
        return
    ref = oracle.layer_norm(x32.astype(np.float64), w32, b32, 1e-6)
    m = metrics(y, ref)
    assert m["rel_max"] <= REL_F32_KERNEL, m


@pytest.mark.parametrize("hd,layout,interp,grid", [
    (64, "tiled", False, (8, 16, 16)), (64, "interleaved", True, (4, 24, 24)),
    (32, "tiled", False, (32, 4, 4)), (64, "interleaved", True, (3, 20, 7))])
def test_rope3d_f32(jg, hd, layout, interp, grid):
    gt, gh, gw = grid
    N, H, B = gt * gh * gw, 3, 2
    rng = np.random.default_rng(hd + N)
    x = np.float32(rng.standard_normal((B, N, H * hd)))
    t = _dev(x)
    jg.rope3d_f32(t, grid, H, hd, layout, interp)
    got = t.cpu().numpy().reshape(B, N, H, hd)
    pos = oracle.token_positions(gt, gh, gw, interp, 16)
    COS, SIN = oracle.rope_tables(pos, hd, layout)
    ref = oracle.apply_rope(x.astype(np.float64).reshape(B, N, H, hd).transpose(0, 2, 1, 3), COS, SIN)
    m = metrics(got, ref.transpose(0, 2, 1, 3))
    assert m["rel_max"] <= REL_F32_KERNEL, m


def _linear_ref(A, W, b, epi, resid=None):
    acc = A @ W.T + b
    if epi == 2:
        return resid + acc
    if epi == 3:
        return oracle.gelu_erf(acc)
    return acc


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("epi", [0, 1, 2, 3])
@pytest.mark.parametrize("M,N,K", [(300, 256, 1536), (128, 384, 384), (1000, 768, 1024), (64, 1152, 128)])
def test_linear(jg, dtype, epi, M, N, K):
    rng = np.random.default_rng(M + N + K + epi)
    A = _rounded(rng, (M, K), dtype)
    W = _rounded(rng, (N, K), dtype, 0.02)
    b = rng.standard_normal(N).astype(np.float32).astype(np.float64) * 0.1
    resid = rng.standard_normal((M, N)).astype(np.float32).astype(np.float64)
    out = _dev(resid) if epi == 2 else None
    got = jg.linear(_dev(A, dtype), _dev(W, dtype), _dev(b), epi, out=out)
    got = got.float().cpu().numpy()
    ref = _linear_ref(A, W, b, epi, resid)
    if dtype == "f32" or epi in (1, 2):
        m = metrics(got, ref)
        assert m["rel_max"] <= (1e-5 if dtype == "f32" else 1e-4), (dtype, epi, m)
    else:
        assert_close_16bit(got, ref, f"linear {dtype} epi {epi}")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("epi", [0, 1, 2, 3])
@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (3, 384, 64), (129, 128, 192), (300, 640, 128)])
def test_linear_few_rows(jg, dtype, epi, M, N, K):
    """One, three and 129 rows (a row tile of 128 plus one), a single K
    block, a 384-wide output (128-column tiles) and 640 (256 + 256 + 128)."""
    rng = np.random.default_rng(M * 7 + N + K + epi)
    A = _rounded(rng, (M, K), dtype)
    W = _rounded(rng, (N, K), dtype, 0.05)
    b = rng.standard_normal(N).astype(np.float32).astype(np.float64) * 0.1
    resid = rng.standard_normal((M, N)).astype(np.float32).astype(np.float64)
    out = _dev(resid) if epi == 2 else None
    got = jg.linear(_dev(A, dtype), _dev(W, dtype), _dev(b), epi, out=out).float().cpu().numpy()
    ref = _linear_ref(A, W, b, epi, resid)
    if dtype == "f32" or epi in (1, 2):
        m = metrics(got, ref)
        assert m["rel_max"] <= (1e-5 if dtype == "f32" else 1e-4), (dtype, epi, m)
    else:
        assert_close_16bit(got, ref, f"linear {dtype} epi {epi} M{M} N{N}")


@pytest.mark.parametrize("epi", [0, 1, 2, 3])
@pytest.mark.parametrize("N", [32, 96, 160, 224])
def test_linear_f32_ragged_width(jg, epi, N):
    """The fp32 path takes any width that is a multiple of 4 (the tensor-core
    path refuses widths that are not whole 128-column tiles)."""
    M, K, dtype = 70, 48, "f32"
    rng = np.random.default_rng(N + epi)
    A = _rounded(rng, (M, K), dtype)
    W = _rounded(rng, (N, K), dtype, 0.05)
    b = rng.standard_normal(N).astype(np.float32).astype(np.float64) * 0.1
    resid = rng.standard_normal((M, N)).astype(np.float32).astype(np.float64)
    out = _dev(resid) if epi == 2 else None
    got = jg.linear(_dev(A, dtype), _dev(W, dtype), _dev(b), epi, out=out).float().cpu().numpy()
    assert metrics(got, _linear_ref(A, W, b, epi, resid))["rel_max"] <= 1e-5


@pytest.mark.parametrize("epi", [1, 2, 3])
def test_linear_split_tail_wave(jg, epi):
    """16384 x 1024 outputs are 256 tiles of 256 x 256 for 76 resident CTA
    pairs: three full waves, then 28 tiles split into half-width units.  Every
    element is compared with the float64 product (K 256 keeps it quick)."""
    M, N, K = 16384, 1024, 256
    rng = np.random.default_rng(epi + 99)
    A = _rounded(rng, (M, K), "bf16")
    W = _rounded(rng, (N, K), "bf16", 0.05)
    b = rng.standard_normal(N).astype(np.float32).astype(np.float64) * 0.1
    resid = rng.standard_normal((M, N)).astype(np.float32).astype(np.float64)
    out = _dev(resid) if epi == 2 else None
    dA, dW, db = _dev(A, "bf16"), _dev(W, "bf16"), _dev(b)
    got = jg.linear(dA, dW, db, epi, out=out).float().cpu().numpy()
    ref = _linear_ref(A, W, b, epi, resid)
    if epi in (1, 2):
        m = metrics(got, ref)
        assert m["rel_max"] <= 1e-4, (epi, m)
    else:
        assert_close_16bit(got, ref, "linear GELU split tail")
    if epi != 2:
        # one writer per output element: a second run is bit for bit the same
        again = jg.linear(dA, dW, db, epi).float().cpu().numpy()
        np.testing.assert_array_equal(again, got)


def _attn_inputs(rng, B, H, N, hd, dtype, logit_std):
    # q k^T / sqrt(hd) has std ~ sq*sk*sqrt(hd)/sqrt(hd) = sq*sk
    s = math.sqrt(logit_std)
    q = _rounded(rng, (B * H, N, hd), dtype, s)
    k = _rounded(rng, (B * H, N, hd), dtype, s)
    v = _rounded(rng, (B * H, N, hd), dtype)
    return q, k, v


def _plant_lift(q, k, row, key, hd, dtype, lift):
    """k[:, key] = a multiple of q[:, row] whose logit is `lift` above the
    row's largest logit over key tile 0 (keys 0-127), per (clip, head)."""
    scale = 1.0 / math.sqrt(hd)
    m0 = (np.einsum("bd,bkd->bk", q[:, row], k[:, :128]) * scale).max(1)
    qq = (q[:, row] ** 2).sum(1) * scale
    k[:, key] = synth.round_to_dtype(q[:, row] * ((m0 + lift) / qq)[:, None], dtype)


def _run_attn(jg, q, k, v, B, H, N, hd, dtype):
    ldv = (N + 7) // 8 * 8
    vt = np.zeros((B * H, hd, ldv))
    vt[:, :, :N] = v.transpose(0, 2, 1)
    out = jg.attention(_dev(q, dtype), _dev(k, dtype), _dev(vt, dtype), B, H, N, hd)
    jg.ops_sync()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hd", [64, 32])
@pytest.mark.parametrize("N,logit_std", [(200, 1.0), (384, 4.0), (1000, 1.0), (128, 0.3), (1500, 4.0), (2100, 4.0)])
def test_attention_tc(jg, dtype, hd, N, logit_std):
    """Every row against the oracle.  Up to 16 key tiles (2048 tokens; 1500:
    12 key tiles, a ragged last one) run on the persistent kernel, longer
    sequences (2100: 17 key tiles, a ragged last one) on the one-unit-per-CTA
    kernel."""
    B, H = 2, 3
    rng = np.random.default_rng(N + hd)
    q, k, v = _attn_inputs(rng, B, H, N, hd, dtype, logit_std)
    if logit_std > 2:
        # planted large logits: query 3 meets its outlier key in the first key
        # tile; query 130 only in the last one, which moves its running max
        # late and exercises the rescale of the partial output
        k[:, 7] = synth.round_to_dtype(q[:, 3] * 3, dtype)
        k[:, N - 5] = synth.round_to_dtype(q[:, 130] * 3, dtype)
        # moderate ones in key tile 1: query 250's max grows there by ~2^33
        # (in the exponent; within bf16's range, beyond fp16's), query 260's
        # by ~2^11.5 (more than 2^8, within both 16-bit P ranges), so its
        # running max moves only before key tile 2
        k[:, 150] = synth.round_to_dtype(q[:, 250], dtype)
        _plant_lift(q, k, 260, 160, hd, dtype, 8.0)
    got = _run_attn(jg, q, k, v, B, H, N, hd, dtype)
    ref = oracle.attention_heads(q, k, v).reshape(B, H, N, hd).transpose(0, 2, 1, 3).reshape(B, N, H * hd)
    assert_close_16bit(got, ref, f"attention {dtype} hd{hd} N{N}")


@pytest.mark.parametrize("hd", [64, 32])
@pytest.mark.parametrize("N", [1, 2, 7, 127, 129, 255, 257])
def test_attention_tc_tiny_and_tile_edges(jg, hd, N):
    """Every row against the oracle at lengths around the tile sizes: one
    token (the output is v), two, fewer than one 16-byte row of V^T, one
    short of and one past a 128-key tile, one short of and one past a
    256-row query-tile pair."""
    B, H, dtype = 2, 3, "bf16"
    rng = np.random.default_rng(N * 3 + hd)
    q, k, v = _attn_inputs(rng, B, H, N, hd, dtype, 2.0)
    got = _run_attn(jg, q, k, v, B, H, N, hd, dtype)
    ref = oracle.attention_heads(q, k, v).reshape(B, H, N, hd).transpose(0, 2, 1, 3).reshape(B, N, H * hd)
    assert_close_16bit(got, ref, f"attention N{N} hd{hd}")
    if N == 1:
        np.testing.assert_allclose(got.reshape(B, H, hd), v.reshape(B, H, hd), rtol=0, atol=1e-2)


@pytest.mark.parametrize("N", [300, 384])
def test_attention_tc_many_units_per_cta(jg, N):
    """8 clips x 16 heads give 256 units of two query tiles, more than there
    are SMs, so persistent CTAs run two units each; 3 key tiles per unit (an
    odd count, so the CTA-wide barrier parities flip mid-unit) and, at N 300,
    a ragged last key tile and a half-empty second query tile.  Planted large
    logits move the running max in the first and in the last key tile."""
    B, H, hd, dtype = 8, 16, 64, "bf16"
    rng = np.random.default_rng(N + 17)
    q, k, v = _attn_inputs(rng, B, H, N, hd, dtype, 4.0)
    k[:, 7] = synth.round_to_dtype(q[:, 3] * 3, dtype)
    k[:, N - 5] = synth.round_to_dtype(q[:, 130] * 3, dtype)
    k[:, 150] = synth.round_to_dtype(q[:, 250], dtype)
    _plant_lift(q, k, 260, 160, hd, dtype, 8.0)
    got = _run_attn(jg, q, k, v, B, H, N, hd, dtype)
    ref = oracle.attention_heads(q, k, v).reshape(B, H, N, hd).transpose(0, 2, 1, 3).reshape(B, N, H * hd)
    assert_close_16bit(got, ref, f"attention many units N{N}")


@pytest.mark.parametrize("N,hd", [(2048, 64), (8192, 64), (8192, 32), (18432, 64)])
@pytest.mark.parametrize("logit_std", [1.0, 4.0])
def test_attention_tc_long_sampled_rows(jg, N, hd, logit_std):
    """The sequence lengths of the ViT-L 16-frame 256 px clip (2048), the
    64-frame 256 px clip with its hd-32 predictor (8192) and the 64-frame
    384 px clip (18 432), bf16.  Sampled query rows are checked against the
    oracle over all keys.  Planted outliers put one row's largest logit in
    the first key tile and another's in the last key tile; two rows' maxima
    grow in key tile 1, far beyond and a little beyond 2^8 (in the
    exponent)."""
    B, H, dtype = 1, 2, "bf16"
    rng = np.random.default_rng(N * 7 + hd + int(logit_std))
    q, k, v = _attn_inputs(rng, B, H, N, hd, dtype, logit_std)
    k[:, 11] = synth.round_to_dtype(q[:, 5] * 3, dtype)
    k[:, N - 3] = synth.round_to_dtype(q[:, N // 2] * 3, dtype)
    k[:, 200] = synth.round_to_dtype(q[:, N // 3], dtype)
    _plant_lift(q, k, N // 4, 210, hd, dtype, 8.0)
    got = _run_attn(jg, q, k, v, B, H, N, hd, dtype).reshape(N, H, hd)
    rows = np.unique(np.concatenate([[0, 5, N // 4, N // 3, N // 2, N - 1], rng.choice(N, 60, replace=False)]))
    ref = oracle.attention_heads(q[:, rows], k, v)                  # [H, rows, hd]
    assert_close_16bit(got[rows].transpose(1, 0, 2), ref, f"attention N{N} hd{hd} std{logit_std}")


@pytest.mark.parametrize("hd,N", [(64, 130), (32, 77)])
def test_attention_f32(jg, hd, N):
    B, H = 1, 2
    rng = np.random.default_rng(N)
    q, k, v = _attn_inputs(rng, B, H, N, hd, "f32", 2.0)
    got = _run_attn(jg, q, k, v, B, H, N, hd, "f32")
    ref = oracle.attention_heads(q, k, v).reshape(B, H, N, hd).transpose(0, 2, 1, 3).reshape(B, N, H * hd)
    assert_close_f32(got, ref, 1e-5)
