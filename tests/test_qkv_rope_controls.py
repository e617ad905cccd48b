"""Negative controls for the QKV + RoPE parity test (CPU, oracle only).

The GPU test compares q and k with the oracle at the 16-bit bars (per-row
cosine mean 0.9999, worst 0.999, rel_max 1e-2).  These tests show that those
bars fail when the reference is computed with a plausible RoPE mistake, so a
kernel making that mistake cannot pass: the other frequency layout ("V-JEPA 2
/ 2.1 tensor maps and RoPE derivation", §4.1 vs §4.2), interpolation left
out or added (§4.3), positions taken from the row index instead of the ids
(§4.4), and the h and w axes decoded with each other's sizes (§4).
"""
import pytest

from parity import COS_MEAN, COS_WORST, REL_16BIT, metrics
import oracle
import synth
from qkv_cases import CASES, SHARP_MODELS, make_inputs, reference, sharp_weights


def _fails(got, ref):
    m = metrics(got, ref)
    return m["cos_mean"] < COS_MEAN or m["cos_worst"] < COS_WORST or m["rel_max"] > REL_16BIT


CONTROLS = [
    ("bf16-hd64-tiled", dict(layout="interleaved")),
    ("bf16-hd32-tiled-ragged", dict(layout="interleaved")),
    ("f16-hd64-interleaved-interp-ragged", dict(layout="tiled")),
    ("f16-hd64-interleaved-interp-ragged", dict(interp=False)),
    ("bf16-hd32-interleaved-interp", dict(interp=False)),
    ("bf16-hd64-interleaved-plain", dict(interp=True)),
    ("bf16-hd64-tiled-ids", dict(mode="row")),
    ("bf16-hd64-interleaved-interp-ids", dict(mode="row")),
    ("bf16-hd32-tiled-predictor-ids", dict(mode="row")),
    ("bf16-hd64-interleaved-plain", dict(mode="hw_swapped")),
    ("bf16-hd32-tiled-ragged", dict(mode="hw_swapped")),
    ("f16-hd64-interleaved-interp-ragged", dict(mode="hw_swapped")),
]


@pytest.mark.parametrize("name,wrong", CONTROLS, ids=[f"{n}-{'-'.join(map(str, w.items()))}" for n, w in CONTROLS])
def test_wrong_rope_fails_the_bars(name, wrong):
    case = CASES[name]
    A, W, b, ids = make_inputs(case, seed=sum(map(ord, name)))
    rq, rk, rv = reference(case, A, W, b, ids)
    wq, wk, wv = reference(case, A, W, b, ids, **wrong)
    assert _fails(wq, rq) and _fails(wk, rk), (name, wrong, metrics(wq, rq))
    assert metrics(wv, rv)["rel_max"] == 0.0      # v carries no RoPE


def test_right_rope_passes_the_bars():
    """The reference against itself through a 16-bit rounding of its output
    (what the kernel stores) stays inside the bars, so they are not too tight."""
    for name in ("bf16-hd64-tiled", "bf16-hd32-interleaved-interp", "bf16-hd64-tiled-ids"):
        case = CASES[name]
        A, W, b, ids = make_inputs(case, seed=sum(map(ord, name)))
        rq, rk, _ = reference(case, A, W, b, ids)
        assert not _fails(synth.round_to_dtype(rq, "bf16"), rq)
        assert not _fails(synth.round_to_dtype(rk, "bf16"), rk)


def _wrong_settings(cfg):
    out = [("layout", {"rope_layout": "interleaved" if cfg.rope_layout == "tiled" else "tiled"}),
           ("no rotation", {"rope_theta": 1e30})]
    if cfg.rope_interpolate:
        out.append(("no interpolation", {"rope_interpolate": False}))
    return out


@pytest.mark.parametrize("name", list(SHARP_MODELS))
def test_sharp_model_wrong_rope_fails_end_to_end(name):
    """On the sharp-attention encoders of the end-to-end GPU test, the oracle
    run with the wrong layout, without interpolation (2.1 geometry) or with no
    rotation at all fails the end-to-end bars against the right oracle; with
    the default N(0, 0.02) weights the same mistakes pass them."""
    cfg = SHARP_MODELS[name]
    clip = synth.clip_u8(cfg)[0]
    w = sharp_weights(cfg)
    ref = oracle.encoder_forward(cfg, w, clip)["out"]
    w02 = synth.encoder_weights(cfg)
    ref02 = oracle.encoder_forward(cfg, w02, clip)["out"]
    for label, change in _wrong_settings(cfg):
        bad = cfg.with_(**change)
        assert _fails(oracle.encoder_forward(bad, w, clip)["out"], ref), (name, label)
        assert not _fails(oracle.encoder_forward(bad, w02, clip)["out"], ref02), (name, label)
