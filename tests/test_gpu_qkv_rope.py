"""The fused QKV projection with 3-D RoPE (jepa_qkv_rope, the epilogue that
jepa_encode runs) against the oracle, element by element.

Every q, k and v^T value of every case is compared with the oracle's float64
product, RoPE'd with its tables ("V-JEPA 2 / 2.1 tensor maps and RoPE
derivation", §4).  The cases cover bf16, fp16 and fp32, head dims 64 and 32,
the tiled and interleaved layouts, interpolation on and off, ragged grids,
several clips, ids in random order (the masked encoder) and context-then-
target ids (the predictor), and the split tail wave of the persistent GEMM.
tests/test_qkv_rope_controls.py shows on the CPU that the same bars fail for
the wrong layout, the wrong interpolation setting and the wrong position
decode.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_close_16bit, assert_close_f32
from qkv_cases import CASES, make_inputs, n_tokens, reference

pytestmark = pytest.mark.gpu

TD = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def jg():
    import video_vit_encoder_gb300 as m
    m.load()
    return m


def _dev(a, dtype="f32"):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(TD[dtype]).cuda()


def _run(jg, case, A, W, b, ids):
    dt = case["dtype"]
    n = n_tokens(case)
    pid = torch.from_numpy(ids).cuda() if ids is not None else None
    q, k, vt = jg.qkv_rope(_dev(A, dt), _dev(W, dt), _dev(b), case["batch"], n, case["H"], case["grid"],
                           case["layout"], case["interp"], pos_ids=pid)
    jg.ops_sync()
    return [t.float().cpu().numpy().astype(np.float64) for t in (q, k, vt)]


@pytest.mark.parametrize("name", list(CASES))
def test_qkv_rope_every_element(jg, name):
    case = CASES[name]
    A, W, b, ids = make_inputs(case, seed=sum(map(ord, name)))
    q, k, vt = _run(jg, case, A, W, b, ids)
    rq, rk, rv = reference(case, A, W, b, ids)
    n = n_tokens(case)
    check = assert_close_f32 if case["dtype"] == "f32" else assert_close_16bit
    kw = {"rel": 1e-5} if case["dtype"] == "f32" else {}
    check(q, rq, what=f"{name} q", **kw)
    check(k, rk, what=f"{name} k", **kw)
    check(vt[:, :, :n], rv.transpose(0, 2, 1), what=f"{name} v^T", **kw)
    # the padding columns of v^T are not written
    assert not np.any(vt[:, :, n:]), name


def test_qkv_rope_vitl_launch_sampled_rows(jg):
    """The ViT-L/16 launch of the benchmark (8 clips x 2048 tokens, D 1024,
    16 heads, tiled RoPE on the 8 x 16 x 16 grid; 768 CTA-pair tiles whose
    last 8 run as half-width units), checked on sampled rows of every clip
    against the oracle's product for those rows."""
    case = dict(dtype="bf16", D=1024, H=16, batch=8, grid=(8, 16, 16), layout="tiled", interp=False)
    rng = np.random.default_rng(7)
    D, H, B, n = 1024, 16, 8, 2048
    A = synth.round_to_dtype(rng.standard_normal((B * n, D)), "bf16").astype(np.float64)
    W = synth.round_to_dtype(rng.standard_normal((3 * D, D)) * 0.03, "bf16").astype(np.float64)
    b = rng.standard_normal(3 * D).astype(np.float32).astype(np.float64) * 0.5
    q, k, vt = _run(jg, case, A, W, b, None)
    toks = np.unique(np.concatenate([[0, 1, 255, 256, n - 1], rng.choice(n, 27, replace=False)]))
    rows = (np.arange(B)[:, None] * n + toks[None, :]).ravel()
    qkv = A[rows] @ W.T + b
    pos = oracle.token_positions(8, 16, 16)[toks]
    COS, SIN = oracle.rope_tables(np.tile(pos, (B, 1)), D // H, "tiled")
    hd = D // H
    for s, got in ((0, q), (1, k)):
        ref = oracle.apply_rope(qkv[:, s * D:(s + 1) * D].reshape(-1, H, hd), COS[:, None], SIN[:, None])
        g = got.reshape(B, H, n, hd)[:, :, toks].transpose(0, 2, 1, 3).reshape(-1, H, hd)
        assert_close_16bit(g, ref, f"vitl {'qk'[s]}")
    g = vt.reshape(B, H, hd, -1)[:, :, :, toks].transpose(0, 3, 1, 2).reshape(-1, H, hd)
    assert_close_16bit(g, qkv[:, 2 * D:].reshape(-1, H, hd), "vitl v")


def test_qkv_rope_bad_ids_reported(jg):
    """Ids outside the grid are clamped (no out-of-range read) and reported."""
    from video_vit_encoder_gb300._lib import ERR_ARG, JepaError
    case = CASES["bf16-hd64-tiled-ids"]
    A, W, b, ids = make_inputs(case, seed=5)
    ids = ids.copy()
    ids[3] = 10 ** 6
    ids[7] = -4
    dt = case["dtype"]
    with pytest.raises(JepaError) as e:
        jg.qkv_rope(_dev(A, dt), _dev(W, dt), _dev(b), case["batch"], n_tokens(case), case["H"], case["grid"],
                    case["layout"], case["interp"], pos_ids=torch.from_numpy(ids).cuda())
        jg.ops_sync()
    assert e.value.status == ERR_ARG
    # the status was cleared and the context works: a valid call passes
    ids[3], ids[7] = 3, 7
    q, k, vt = _run(jg, case, A, W, b, _valid(ids, case))
    rq, _, _ = reference(case, A, W, b, _valid(ids, case))
    assert_close_16bit(q, rq, "after bad ids")


def _valid(ids, case):
    gt, gh, gw = case["grid"]
    return np.clip(ids, 0, gt * gh * gw - 1).astype(np.int32)
