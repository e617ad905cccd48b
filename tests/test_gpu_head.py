"""The attentive-pool head and classifier (jepa_head_forward) against the
oracle ("V-JEPA 2 / 2.1 tensor maps and RoPE derivation", §2 "Attentive-pool
head - exact forward").

  * a small head (D 256, 4 heads, 2 pool blocks, 11 classes) with non-zero
    biases and LayerNorm affines on random tokens of ragged length, bf16, f16
    and fp32;
  * the same head with sharp attention (the query, its projections and the
    pool blocks' q/k drawn large), so the softmax weights matter;
  * token-permutation invariance (no positions anywhere in the head);
  * the SSv2 ViT-L/16 head (3 pool blocks, 16 heads, 174 classes) on the
    ViT-L/16 encoder's own output for the benchmark's 8 clips of 16 x 256 x 256.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_close_16bit, assert_close_f32

pytestmark = pytest.mark.gpu

HC = synth.HeadConfig(embed_dim=256, n_layer=2, n_head=4, ffn_dim=512, n_classes=11)


@pytest.fixture(scope="module")
def jg():
    import video_vit_encoder_gb300 as m
    m.load()
    return m


def _weights(hc, dtype, sharp=False, seed=1):
    std = {"bias": 0.05, "head.query": 1.0}
    if sharp:
        # cross-attention scores of std ~3 and pool-block logits of std ~3
        std.update({"xattn.q.weight": 0.06, "xattn.k.weight": 0.06,
                    "attn_qkv.weight": float(np.sqrt(3.0 / hc.embed_dim))})
    w = synth.head_weights(hc, seed, dtype, std_overrides=std,
                           kind_overrides={"bias": "vec", "ln1.weight": "vec", "ln2.weight": "vec",
                                           "ln_kv.weight": "vec"})
    for k in list(w):
        if k.endswith(("ln1.weight", "ln2.weight", "ln_kv.weight")):
            w[k] = (1.0 + w[k]).astype(np.float32)
    return w


def _tokens(B, n, D, seed):
    # LayerNorm'd-like encoder tokens: unit scale with a per-token offset
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, n, D)) + rng.standard_normal((B, n, 1)) * 0.3).astype(np.float32)


def _check(jg, hc, w, dtype, x, what):
    head = jg.Head(hc, w, dtype)
    logits, pooled = head.forward(torch.from_numpy(x).cuda(), pooled=True)
    head.sync()
    head.close()
    logits, pooled = logits.cpu().numpy(), pooled.cpu().numpy()
    ref = [oracle.attentive_pool_forward(hc, w, x[b]) for b in range(x.shape[0])]
    rl = np.stack([r["logits"] for r in ref])
    rp = np.stack([r["pooled"] for r in ref])
    if dtype == "f32":
        assert_close_f32(logits, rl, 1e-4, f"{what} logits")
        assert_close_f32(pooled, rp, 1e-4, f"{what} pooled")
    else:
        assert_close_16bit(logits, rl, f"{what} logits")
        assert_close_16bit(pooled, rp, f"{what} pooled")
    return logits


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("sharp", [False, True])
def test_small_head(jg, dtype, sharp):
    w = _weights(HC, dtype, sharp)
    x = _tokens(3, 135, HC.embed_dim, 5)
    _check(jg, HC, w, dtype, x, f"small {dtype} sharp={sharp}")


def test_head_token_permutation(jg):
    w = _weights(HC, "bf16", sharp=True)
    x = _tokens(2, 300, HC.embed_dim, 6)
    perm = np.random.default_rng(8).permutation(300)
    a = _check(jg, HC, w, "bf16", x, "unpermuted")
    b = _check(jg, HC, w, "bf16", np.ascontiguousarray(x[:, perm]), "permuted")
    assert_close_16bit(b, a.astype(np.float64), "permutation")


def test_ssv2_head_on_vitl_encoder_output(jg):
    """The SSv2 classifier head (D 1024, 16 heads, 3 pool blocks, FFN 4096,
    174 classes, bf16) on the ViT-L/16 encoder's own tokens for the
    benchmark's 8 clips of 16 x 256 x 256 (2048 tokens each); clips 0 and 7
    against the oracle run on the same tokens."""
    cfg = synth.CONFIGS["vitl16-16f256"]
    enc = jg.Encoder(cfg, synth.encoder_weights(cfg))
    tokens = enc.encode(torch.from_numpy(synth.clip_u8(cfg)).cuda())["out"]
    enc.sync()
    enc.close()
    hc = synth.HEAD_SSV2
    w = _weights(hc, "bf16", sharp=True, seed=2)
    head = jg.Head(hc, w, "bf16")
    logits, pooled = head.forward(tokens, pooled=True)
    head.sync()
    head.close()
    x = tokens.cpu().numpy()
    for b in (0, 7):
        ref = oracle.attentive_pool_forward(hc, w, x[b])
        assert_close_16bit(logits[b:b + 1].cpu().numpy(), ref["logits"][None], f"ssv2 logits clip {b}")
        assert_close_16bit(pooled[b:b + 1].cpu().numpy(), ref["pooled"][None], f"ssv2 pooled clip {b}")


def test_head_graph_replay_matches_eager(jg):
    """Repeated calls with the same buffers replay one captured graph (the
    first eager, the second captured): bit for bit the eager result, also
    after the tokens' contents change."""
    w = _weights(HC, "bf16", sharp=True)
    x = torch.from_numpy(_tokens(2, 200, HC.embed_dim, 9)).cuda()
    head = jg.Head(HC, w, "bf16")
    logits = torch.empty(2, HC.n_classes, device="cuda")
    runs = []
    for _ in range(3):
        head.forward(x, out=logits)
        head.sync()
        runs.append(logits.clone())
    head.set_graphs(False)
    head.forward(x, out=logits)
    head.sync()
    for r in runs:
        assert torch.equal(r, logits)
    x.copy_(torch.from_numpy(_tokens(2, 200, HC.embed_dim, 10)))
    head.set_graphs(True)
    head.forward(x, out=logits)      # replayed on the new contents
    head.sync()
    replayed = logits.clone()
    head.set_graphs(False)
    head.forward(x, out=logits)
    head.sync()
    assert torch.equal(replayed, logits)
    head.close()
