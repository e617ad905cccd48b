"""Pins of the oracle's attentive-pool head ("V-JEPA 2 / 2.1 tensor maps and
RoPE derivation", §2 "Attentive-pool head - exact forward"; §1 head row).

  * an independent torch float64 composition of the printed steps, with
    non-zero biases and perturbed LayerNorm affines;
  * closed form: pool blocks and the key projection zeroed, so every score is
    equal and the cross-attention returns the mean of the values: pooled =
    query + mean_i(ln_kv(x_i)) W_v^T + b_v (raw query, no output
    projection), and with the MLP zeroed too, logits = pooled W_cls^T + b_cls;
  * closed form: one token, whose value the single query receives whatever
    the scores;
  * no RoPE and no positions anywhere in the head: permuting the encoder
    tokens leaves pooled and logits unchanged;
  * the controls that a normalised query or an output projection would fail
    the first closed form.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

HC = synth.HeadConfig(embed_dim=256, n_layer=2, n_head=4, ffn_dim=512, n_classes=11)


def _weights(hc=HC, seed=0, **kw):
    w = synth.head_weights(hc, seed, "f32", **kw)
    return {k: np.asarray(v, np.float64) for k, v in w.items()}


def _perturbed(hc=HC, seed=1):
    # non-zero biases and LN affines, so a dropped bias or affine shows
    w = _weights(hc, seed, std_overrides={"bias": 0.05, "head.query": 1.0},
                 kind_overrides={"bias": "vec", "ln1.weight": "vec", "ln2.weight": "vec", "ln_kv.weight": "vec"})
    for k in list(w):
        if k.endswith(("ln1.weight", "ln2.weight", "ln_kv.weight")):
            w[k] = 1.0 + w[k]
    return w


def _tokens(n, d, seed):
    return np.random.default_rng(seed).standard_normal((n, d))


def _torch_head(hc, w, x):
    T = {k: torch.from_numpy(v) for k, v in w.items()}
    x = torch.from_numpy(x)
    D, H = hc.embed_dim, hc.n_head
    hd = D // H
    F_ = torch.nn.functional

    def mha(q, k, v):
        q, k, v = (t.reshape(t.shape[0], H, hd).transpose(0, 1) for t in (q, k, v))
        o = F_.scaled_dot_product_attention(q, k, v)
        return o.transpose(0, 1).reshape(-1, D)

    for i in range(hc.n_layer):
        p = f"head.blk.{i}."
        y = F_.layer_norm(x, (D,), T[p + "ln1.weight"], T[p + "ln1.bias"], hc.ln_eps)
        qkv = F_.linear(y, T[p + "attn_qkv.weight"], T[p + "attn_qkv.bias"])
        x = x + F_.linear(mha(qkv[:, :D], qkv[:, D:2 * D], qkv[:, 2 * D:]), T[p + "attn_out.weight"],
                          T[p + "attn_out.bias"])
        y = F_.layer_norm(x, (D,), T[p + "ln2.weight"], T[p + "ln2.bias"], hc.ln_eps)
        x = x + F_.linear(F_.gelu(F_.linear(y, T[p + "ffn_up.weight"], T[p + "ffn_up.bias"])),
                          T[p + "ffn_down.weight"], T[p + "ffn_down.bias"])
    q0 = T["head.query"].reshape(1, D)
    kv = F_.layer_norm(x, (D,), T["head.xattn.ln_kv.weight"], T["head.xattn.ln_kv.bias"], hc.ln_eps)
    o = mha(F_.linear(q0, T["head.xattn.q.weight"], T["head.xattn.q.bias"]),
            F_.linear(kv, T["head.xattn.k.weight"], T["head.xattn.k.bias"]),
            F_.linear(kv, T["head.xattn.v.weight"], T["head.xattn.v.bias"]))
    y = q0 + o
    yn = F_.layer_norm(y, (D,), T["head.xattn.ln2.weight"], T["head.xattn.ln2.bias"], hc.ln_eps)
    y = y + F_.linear(F_.gelu(F_.linear(yn, T["head.xattn.ffn_up.weight"], T["head.xattn.ffn_up.bias"])),
                      T["head.xattn.ffn_down.weight"], T["head.xattn.ffn_down.bias"])
    return y[0].numpy(), F_.linear(y, T["head.cls.weight"], T["head.cls.bias"])[0].numpy()


def test_matches_torch_composition():
    w = _perturbed()
    x = _tokens(37, HC.embed_dim, 3)
    ref = oracle.attentive_pool_forward(HC, w, x)
    pooled, logits = _torch_head(HC, w, x)
    assert ref["logits"].shape == (HC.n_classes,) and ref["pooled"].shape == (HC.embed_dim,)
    np.testing.assert_allclose(ref["pooled"], pooled, rtol=0, atol=1e-10 * np.abs(pooled).max())
    np.testing.assert_allclose(ref["logits"], logits, rtol=0, atol=1e-10 * np.abs(logits).max())


def _ln(x, g, b, eps):
    mu = x.sum(-1, keepdims=True) / x.shape[-1]
    var = ((x - mu) ** 2).sum(-1, keepdims=True) / x.shape[-1]
    return (x - mu) / np.sqrt(var + eps) * g + b


def _uniform_attention_weights():
    w = _perturbed()
    for k in w:
        if k.startswith("head.blk.") and ("attn_out" in k or "ffn_down" in k):
            w[k] = np.zeros_like(w[k])             # the pool blocks add nothing
        if k.startswith(("head.xattn.k.", "head.xattn.ffn_down.")):
            w[k] = np.zeros_like(w[k])             # equal scores; the MLP adds nothing
    return w


def _uniform_closed_form(w, x):
    kv = _ln(x, w["head.xattn.ln_kv.weight"], w["head.xattn.ln_kv.bias"], HC.ln_eps)
    pooled = w["head.query"] + kv.mean(axis=0) @ w["head.xattn.v.weight"].T + w["head.xattn.v.bias"]
    return pooled, pooled @ w["head.cls.weight"].T + w["head.cls.bias"]


def test_closed_form_uniform_attention_gives_mean_of_values():
    w = _uniform_attention_weights()
    x = _tokens(50, HC.embed_dim, 4)
    ref = oracle.attentive_pool_forward(HC, w, x)
    pooled, logits = _uniform_closed_form(w, x)
    np.testing.assert_allclose(ref["pooled"], pooled, rtol=0, atol=1e-12 * np.abs(pooled).max())
    np.testing.assert_allclose(ref["logits"], logits, rtol=0, atol=1e-12 * np.abs(logits).max())


def test_closed_form_fails_for_a_normalised_query_or_an_output_projection():
    """The closed form above separates the pages' head from two plausible
    misreadings: LayerNorm applied to the query, and an output projection
    after the cross-attention."""
    w = _uniform_attention_weights()
    x = _tokens(50, HC.embed_dim, 4)
    pooled, _ = _uniform_closed_form(w, x)
    kv = _ln(x, w["head.xattn.ln_kv.weight"], w["head.xattn.ln_kv.bias"], HC.ln_eps)
    o = kv.mean(axis=0) @ w["head.xattn.v.weight"].T + w["head.xattn.v.bias"]
    q_normed = _ln(w["head.query"], w["head.xattn.ln_kv.weight"], w["head.xattn.ln_kv.bias"], HC.ln_eps)
    wrong_query = q_normed + o
    wrong_proj = w["head.query"] + o @ w["head.xattn.q.weight"].T     # any extra D x D map
    for wrong in (wrong_query, wrong_proj):
        assert np.abs(wrong - pooled).max() > 1e-2 * np.abs(pooled).max()


def test_closed_form_single_token_receives_its_value():
    w = _perturbed()
    for k in w:
        if k.startswith("head.blk.") and ("attn_out" in k or "ffn_down" in k):
            w[k] = np.zeros_like(w[k])
    w["head.xattn.ffn_down.weight"] = np.zeros_like(w["head.xattn.ffn_down.weight"])
    w["head.xattn.ffn_down.bias"] = np.zeros_like(w["head.xattn.ffn_down.bias"])
    x = _tokens(1, HC.embed_dim, 5)
    ref = oracle.attentive_pool_forward(HC, w, x)
    kv = _ln(x, w["head.xattn.ln_kv.weight"], w["head.xattn.ln_kv.bias"], HC.ln_eps)[0]
    pooled = w["head.query"] + kv @ w["head.xattn.v.weight"].T + w["head.xattn.v.bias"]
    np.testing.assert_allclose(ref["pooled"], pooled, rtol=0, atol=1e-12 * np.abs(pooled).max())


def test_no_positions_in_the_head():
    """Permuting the encoder tokens leaves the head's output unchanged: the pool
    blocks carry no RoPE and the cross-attention no positions."""
    w = _perturbed()
    x = _tokens(40, HC.embed_dim, 6)
    a = oracle.attentive_pool_forward(HC, w, x)
    b = oracle.attentive_pool_forward(HC, w, x[np.random.default_rng(7).permutation(40)])
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=0, atol=1e-11 * np.abs(a["logits"]).max())
    np.testing.assert_allclose(a["pooled"], b["pooled"], rtol=0, atol=1e-11 * np.abs(a["pooled"]).max())


def test_head_weights_follow_the_key_map():
    names = [n for n, _, _ in synth.tensor_names_head(synth.HEAD_SSV2)]
    assert names[0] == "head.query" and names[-2:] == ["head.cls.weight", "head.cls.bias"]
    assert sum(n.startswith("head.blk.") for n in names) == 3 * 12     # 3 pool layers ([N] §1)
    shapes = dict((n, s) for n, s, _ in synth.tensor_names_head(synth.HEAD_SSV2))
    assert shapes["head.cls.weight"] == (174, 1024)                     # 174 classes ([N] §1, §2)
