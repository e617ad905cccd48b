"""The whole encoder through the C ABI against the oracle.

Small geometries are compared end to end on every token; the fp32 workload
(single block + patch embed) is compared end to end at its full size.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import REL_F32_PATH, assert_close_16bit, assert_close_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jg():
    import video_vit_encoder_gb300 as m
    m.load()
    return m


SMALL = {
    # 2.1 geometry: interleaved interpolated RoPE, modality vector, hierarchical taps; N = 2*6*8 = 96
    "b21-bf16": synth.CONFIGS["vitb16-64f384"].with_(embed_dim=256, n_head=4, ffn_dim=1024, n_layer=3, n_frames=4,
                                          height=96, width=128, batch=3, hier_layers=(0, 2)),
    "b21-f16": synth.CONFIGS["vitb16-16f384-f16"].with_(embed_dim=256, n_head=4, ffn_dim=1024, n_layer=3, n_frames=4,
                                         height=96, width=128, batch=2, hier_layers=(1,)),
    # V-JEPA 2 geometry, tiled RoPE, head_dim 32, N = 3*5*9 = 135 (ragged against 128-row tiles)
    "v2-hd32": synth.CONFIGS["vitl16-16f256"].with_(embed_dim=256, n_head=8, ffn_dim=512, n_layer=2, n_frames=6,
                                         height=80, width=144, batch=2),
    # 2.1 native image path (one frame, tubelet 1), N = 6*8 = 48 and 11*5 = 55
    "img21-bf16": synth.CONFIGS["img384"].with_(embed_dim=256, n_head=4, ffn_dim=1024, n_layer=3, height=96,
                                                width=128, batch=3, hier_layers=(0, 2)),
    "img21-f16": synth.CONFIGS["img384"].with_(embed_dim=256, n_head=4, ffn_dim=1024, n_layer=2, height=176,
                                               width=80, batch=2, dtype="f16", hier_layers=(1,)),
    # the smallest clips: one token (2 frames of 16 x 16), and two tokens along t
    "v2-1tok": synth.CONFIGS["vitl16-16f256"].with_(embed_dim=256, n_head=4, ffn_dim=512, n_layer=2, n_frames=2,
                                         height=16, width=16, batch=3),
    "v2-2tok": synth.CONFIGS["vitl16-16f256"].with_(embed_dim=256, n_head=4, ffn_dim=512, n_layer=2, n_frames=4,
                                         height=16, width=16, batch=2),
}


def _run(jg, cfg, pooled=True, hier=True):
    w = synth.encoder_weights(cfg)
    clip = synth.clip_u8(cfg)
    enc = jg.Encoder(cfg, w)
    res = enc.encode(torch.from_numpy(clip).cuda(), pooled=pooled, hier=hier)
    enc.sync()
    return enc, w, clip, {k: v.cpu().numpy() for k, v in res.items()}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_end_to_end(jg, name):
    cfg = SMALL[name]
    enc, w, clip, got = _run(jg, cfg)
    for b in range(cfg.batch):
        ref = oracle.encoder_forward(cfg, w, clip[b])
        assert_close_16bit(got["out"][b], ref["out"], f"{name} clip {b}")
        np.testing.assert_allclose(got["pooled"][b], ref["pooled"], atol=1e-2 * np.abs(ref["pooled"]).max())
        for k, tap in enumerate(ref["hier"]):
            assert_close_16bit(got["hier"][k, b], tap, f"{name} tap {k} clip {b}")
    enc.close()


def test_block_f32_4f128_fp32_end_to_end(jg):
    cfg = synth.CONFIGS["block-f32-4f128"]
    enc, w, clip, got = _run(jg, cfg, hier=False)
    ref = oracle.encoder_forward(cfg, w, clip[0])
    m = assert_close_f32(got["out"][0], ref["out"], REL_F32_PATH, "block-f32-4f128")
    print("block-f32-4f128 parity", m)
    enc.close()


def test_embed_then_blocks_equals_encode(jg):
    cfg = SMALL["b21-bf16"]
    w = synth.encoder_weights(cfg)
    clip = torch.from_numpy(synth.clip_u8(cfg)).cuda()
    enc = jg.Encoder(cfg, w)
    out = enc.encode(clip)["out"]
    B, T, H, W, _ = clip.shape
    x = enc.embed(clip)
    enc.blocks(x, B, T, H, W, 0, 1)
    enc.blocks(x, B, T, H, W, 1, cfg.n_layer)
    y = jg.layernorm_f32(x, torch.from_numpy(w["norm.weight"]).cuda(), torch.from_numpy(w["norm.bias"]).cuda(),
                         cfg.ln_eps)
    enc.sync()
    assert torch.equal(y.view_as(out), out)
    enc.close()


def test_encode_host_matches_device(jg):
    cfg = SMALL["v2-hd32"]
    w = synth.encoder_weights(cfg)
    clip = synth.clip_u8(cfg)
    enc = jg.Encoder(cfg, w)
    dev = enc.encode(torch.from_numpy(clip).cuda(), pooled=True)
    enc.sync()
    hclip = torch.from_numpy(clip).pin_memory()
    hout = torch.empty(dev["out"].shape, dtype=torch.float32).pin_memory()
    hpool = torch.empty(dev["pooled"].shape, dtype=torch.float32).pin_memory()
    enc.encode_host(hclip, hout, hpool)
    assert torch.equal(hout, dev["out"].cpu())
    assert torch.equal(hpool, dev["pooled"].cpu())
    enc.close()


def test_encode_host_async_stream_of_clips(jg):
    """Five different clips streamed through jepa_encode_host_async (two
    staging slots used in turn, copies on the handle's own streams) each give
    exactly the device-buffer encode of that clip; a shape change in the middle
    of the stream reallocates a slot only after its earlier work is done."""
    cfg = SMALL["v2-hd32"]
    w = synth.encoder_weights(cfg)
    enc = jg.Encoder(cfg, w)
    rng = np.random.default_rng(11)
    shapes = [(2, 4, 64, 64), (2, 4, 64, 64), (1, 4, 64, 64), (2, 4, 64, 80), (2, 4, 64, 64)]
    clips = [rng.integers(0, 256, (B, T, H, W, 3), dtype=np.uint8) for B, T, H, W in shapes]
    want, hin, hout, hpool = [], [], [], []
    for c in clips:
        d = enc.encode(torch.from_numpy(c).cuda(), pooled=True)
        enc.sync()
        want.append((d["out"].cpu(), d["pooled"].cpu()))
        hin.append(torch.from_numpy(c).pin_memory())
        hout.append(torch.empty(d["out"].shape, dtype=torch.float32).pin_memory())
        hpool.append(torch.empty(d["pooled"].shape, dtype=torch.float32).pin_memory())
    for i in range(len(clips)):
        enc.encode_host_async(hin[i], hout[i], hpool[i])
    enc.sync()
    for i in range(len(clips)):
        assert torch.equal(hout[i], want[i][0]), i
        assert torch.equal(hpool[i], want[i][1]), i
    enc.close()


def test_batch_independence(jg):
    # clips are independent: clip 1 of a batch equals the same clip run alone
    cfg = SMALL["v2-hd32"]
    w = synth.encoder_weights(cfg)
    clip = torch.from_numpy(synth.clip_u8(cfg)).cuda()
    enc = jg.Encoder(cfg, w)
    both = enc.encode(clip)["out"]
    one = enc.encode(clip[1:2].contiguous())["out"]
    enc.sync()
    assert_close_16bit(one[0].cpu().numpy(), both[1].cpu().numpy().astype(np.float64), "batch independence")
    enc.close()


def test_one_handle_encodes_clips_and_images(jg):
    """A model with the image path takes 4-frame clips on the video path and
    single frames on the image path, from the same handle."""
    cfg = SMALL["img21-bf16"]
    w = synth.encoder_weights(cfg)
    enc = jg.Encoder(cfg, w)
    for T in (4, 1, 2):
        c = cfg.with_(n_frames=T)
        clip = synth.clip_u8(c, batch=2, first_clip=T)
        got = enc.encode(torch.from_numpy(clip).cuda())["out"].cpu().numpy()
        enc.sync()
        for b in range(2):
            ref = oracle.encoder_forward(c, w, clip[b])
            assert got.shape[1] == ref["out"].shape[0]
            assert_close_16bit(got[b], ref["out"], f"T={T} clip {b}")
    enc.close()


@pytest.mark.parametrize("name", ["b21-bf16", "img21-bf16"])
def test_normalised_float_input(jg, name):
    """The float [B, 3, T, H, W] input format, already normalised, on the video and image paths."""
    cfg = SMALL[name]
    w = synth.encoder_weights(cfg)
    clip = synth.clip_u8(cfg)
    xf = np.ascontiguousarray(np.stack([oracle.normalise_clip(clip[b]) for b in range(cfg.batch)]), np.float32)
    enc = jg.Encoder(cfg, w)
    got = enc.encode(torch.from_numpy(xf).cuda())["out"].cpu().numpy()
    enc.sync()
    for b in range(cfg.batch):
        assert_close_16bit(got[b], oracle.encoder_forward(cfg, w, clip[b])["out"], f"{name} float input clip {b}")
    enc.close()


@pytest.mark.parametrize("modality", ["video", "image"])
def test_small_pred21(jg, modality):
    """The 2.1 predictor with two blocks on random encoder tokens: both
    modality vectors, the context projection, ragged row counts."""
    import dataclasses
    pc = dataclasses.replace(synth.PREDICTOR_21, n_layer=2)
    cfg = synth.CONFIGS["pred21"].with_(n_frames=4 if modality == "video" else 1, height=96, width=80,
                                        predictor=pc)
    pw = synth.predictor_weights(cfg)
    rng = np.random.default_rng(7)
    for k in ("mod_embed_video", "mod_embed_img"):
        pw[k] = synth.round_to_dtype(rng.standard_normal(pw[k].shape) * 0.5, "f32")
    grid = cfg.grid()
    n = grid[0] * grid[1] * grid[2]
    enc = synth.round_to_dtype(rng.standard_normal((n, 768)), "f32")
    ctx, tgt = synth.context_target_split(cfg)
    pred = jg.Predictor(pc, pw, cfg.dtype)
    out, octx = pred.predict(torch.from_numpy(enc).cuda(), torch.from_numpy(ctx).cuda(), torch.from_numpy(tgt).cuda(),
                             grid, modality=modality, with_ctx=True)
    pred.sync()
    ref = oracle.predictor_outputs(pc, pw, enc.astype(np.float64), ctx, tgt, grid, modality)
    assert_close_16bit(out.cpu().numpy(), ref["pred"], f"small pred21 {modality}")
    assert_close_16bit(octx.cpu().numpy(), ref["ctx"], f"small pred21 {modality} ctx")
    pred.close()


def _keep(cfg, B, frac, seed):
    n = synth.tokens_per_clip(cfg)
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(n, int(n * frac), replace=False) for _ in range(B)]).astype(np.int32)


@pytest.mark.parametrize("name", ["b21-bf16", "v2-hd32"])
def test_masked_encoder(jg, name):
    """Masked encoder forward: each clip keeps its own random 40 % of the
    tokens (unsorted); every kept row, the taps and the mean against the
    oracle's masked forward."""
    cfg = SMALL[name]
    w = synth.encoder_weights(cfg)
    clip = synth.clip_u8(cfg)
    keep = _keep(cfg, cfg.batch, 0.4, 3)
    enc = jg.Encoder(cfg, w)
    got = enc.encode_masked(torch.from_numpy(clip).cuda(), torch.from_numpy(keep).cuda(), pooled=True, hier=True)
    enc.sync()
    for b in range(cfg.batch):
        ref = oracle.encoder_forward(cfg, w, clip[b], keep=keep[b])
        assert_close_16bit(got["out"][b].cpu().numpy(), ref["out"], f"{name} masked clip {b}")
        for k, tap in enumerate(ref["hier"]):
            assert_close_16bit(got["hier"][k, b].cpu().numpy(), tap, f"{name} masked tap {k} clip {b}")
        np.testing.assert_allclose(got["pooled"][b].cpu().numpy(), ref["pooled"],
                                   atol=1e-2 * np.abs(ref["pooled"]).max())
    enc.close()


def test_masked_encoder_all_tokens_is_permuted_encode(jg):
    cfg = SMALL["b21-bf16"]
    w = synth.encoder_weights(cfg)
    clip = torch.from_numpy(synth.clip_u8(cfg)).cuda()
    n = synth.tokens_per_clip(cfg)
    perm = np.stack([np.random.default_rng(b).permutation(n) for b in range(cfg.batch)]).astype(np.int32)
    enc = jg.Encoder(cfg, w)
    full = enc.encode(clip)["out"].cpu().numpy()
    got = enc.encode_masked(clip, torch.from_numpy(perm).cuda())["out"].cpu().numpy()
    enc.sync()
    for b in range(cfg.batch):
        np.testing.assert_allclose(got[b], full[b][perm[b]], rtol=0, atol=5e-3 * np.abs(full).max())
    enc.close()


def test_masked_encoder_bad_ids_are_reported_not_read(jg):
    """Ids outside the grid are clamped by the kernels (no access outside the
    clip or the tables) and the next sync reports JEPA_ERR_ARG; the handle
    then works as before."""
    from video_vit_encoder_gb300._lib import ERR_ARG, JepaError
    cfg = SMALL["v2-hd32"]
    w = synth.encoder_weights(cfg)
    clip = torch.from_numpy(synth.clip_u8(cfg)).cuda()
    n = synth.tokens_per_clip(cfg)
    keep = _keep(cfg, cfg.batch, 0.3, 5)
    bad = keep.copy()
    bad[0, 3] = n + 5
    bad[1, 0] = -3
    enc = jg.Encoder(cfg, w)
    enc.encode_masked(clip, torch.from_numpy(bad).cuda())
    with pytest.raises(JepaError) as e:
        enc.sync()
    assert e.value.status == ERR_ARG
    got = enc.encode_masked(clip, torch.from_numpy(keep).cuda())["out"].cpu().numpy()
    enc.sync()
    ref = oracle.encoder_forward(cfg, w, clip[1].cpu().numpy(), keep=keep[1])
    assert_close_16bit(got[1], ref["out"], "after a bad-id call")
    enc.close()


def test_graph_replay_matches_eager(jg):
    """Repeated calls replay a captured graph: outputs equal the eager run
    bit for bit, through shape changes (the RoPE tables are shared), a
    workspace reallocation, and new contents in the same input buffer."""
    base = SMALL["b21-bf16"]
    w = synth.encoder_weights(base)
    enc = jg.Encoder(base, w)
    shapes = [base, base.with_(n_frames=6, height=64, width=96), base.with_(batch=1)]
    clips = {i: torch.from_numpy(synth.clip_u8(c)).cuda() for i, c in enumerate(shapes)}
    enc.set_graphs(False)
    ref = {i: enc.encode(clips[i], pooled=True)["out"].clone() for i in clips}
    enc.sync()
    enc.set_graphs(True)
    outs = {i: torch.empty_like(ref[i]) for i in clips}
    for i in [0, 0, 1, 0, 1, 1, 2, 0, 2, 1, 0]:
        enc.encode(clips[i], out=outs[i])
        enc.sync()
        assert torch.equal(outs[i], ref[i]), i
    big = base.with_(batch=6)                        # grows the workspace: captured graphs are dropped
    enc.encode(torch.from_numpy(synth.clip_u8(big)).cuda())
    for i in [0, 1, 0, 1]:
        enc.encode(clips[i], out=outs[i])
        enc.sync()
        assert torch.equal(outs[i], ref[i]), ("after growth", i)
    new = torch.from_numpy(synth.clip_u8(base, first_clip=50)).cuda()
    enc.set_graphs(False)
    ref_new = enc.encode(new)["out"].clone()
    enc.set_graphs(True)
    clips[0].copy_(new)                               # same buffer, new contents, replayed graph
    enc.encode(clips[0], out=outs[0])
    enc.sync()
    assert torch.equal(outs[0], ref_new)
    enc.close()


def test_masked_graph_replay_reads_current_ids(jg):
    """A replayed masked call reads the current contents of its id buffer."""
    cfg = SMALL["v2-hd32"]
    w = synth.encoder_weights(cfg)
    clip = torch.from_numpy(synth.clip_u8(cfg)).cuda()
    k1, k2 = _keep(cfg, cfg.batch, 0.5, 8), _keep(cfg, cfg.batch, 0.5, 9)
    enc = jg.Encoder(cfg, w)
    enc.set_graphs(False)
    ref1 = enc.encode_masked(clip, torch.from_numpy(k1).cuda())["out"].clone()
    ref2 = enc.encode_masked(clip, torch.from_numpy(k2).cuda())["out"].clone()
    enc.set_graphs(True)
    ids = torch.from_numpy(k1).cuda()
    got = torch.empty_like(ref1)
    for want, src in [(ref1, k1), (ref1, k1), (ref1, k1), (ref2, k2), (ref1, k1)]:
        ids.copy_(torch.from_numpy(src))
        enc.encode_masked(clip, ids, out=got)   # same buffers every time: eager, capture, replays
        enc.sync()
        assert torch.equal(got, want)
    enc.close()


def test_predictor_graph_replay(jg):
    """Replayed predictor calls equal eager ones and read the current ids."""
    import dataclasses
    pc = dataclasses.replace(synth.PREDICTOR_21, n_layer=2)
    cfg = synth.CONFIGS["pred21"].with_(n_frames=4, height=96, width=80, predictor=pc)
    pw = synth.predictor_weights(cfg)
    grid = cfg.grid()
    n = grid[0] * grid[1] * grid[2]
    enc = torch.from_numpy(synth.round_to_dtype(np.random.default_rng(2).standard_normal((n, 768)), "f32")).cuda()
    splits = []
    for seed in (0, 1):
        perm = np.random.default_rng(seed).permutation(n).astype(np.int32)
        splits.append((np.sort(perm[: n // 2]), np.sort(perm[n // 2:])))
    pred = jg.Predictor(pc, pw, cfg.dtype)
    pred.set_graphs(False)
    refs = []
    for c, t in splits:
        o, oc = pred.predict(enc, torch.from_numpy(c).cuda(), torch.from_numpy(t).cuda(), grid, modality="video",
                             with_ctx=True)
        refs.append((o.clone(), oc.clone()))
    pred.set_graphs(True)
    ic = torch.from_numpy(splits[0][0]).cuda()
    it = torch.from_numpy(splits[0][1]).cuda()
    out, octx = torch.empty_like(refs[0][0]), torch.empty_like(refs[0][1])
    for k in (0, 0, 0, 1, 0, 1):
        ic.copy_(torch.from_numpy(splits[k][0]))
        it.copy_(torch.from_numpy(splits[k][1]))
        pred.predict(enc, ic, it, grid, modality="video", with_ctx=True, out=out, out_ctx=octx)
        pred.sync()
        assert torch.equal(out, refs[k][0]) and torch.equal(octx, refs[k][1]), k
    pred.close()


@pytest.mark.parametrize("name", ["v2-hd32-sharp", "b21-hd64-sharp"])
def test_sharp_attention_end_to_end(jg, name):
    """Encoders whose attn_qkv.weight has std sqrt(3/D), so the attention
    logits have std ~3 and the output depends on the RoPE: every clip, every
    token, the taps and the token mean against the oracle.  The CPU test
    tests/test_qkv_rope_controls.py shows that the oracle with the wrong
    layout, without interpolation or without rotation fails these bars on the
    same models."""
    from qkv_cases import SHARP_MODELS, sharp_weights
    cfg = SHARP_MODELS[name]
    w = sharp_weights(cfg)
    clip = synth.clip_u8(cfg)
    enc = jg.Encoder(cfg, w)
    res = enc.encode(torch.from_numpy(clip).cuda(), pooled=True, hier=True)
    enc.sync()
    got = {k: v.cpu().numpy() for k, v in res.items()}
    for b in range(cfg.batch):
        ref = oracle.encoder_forward(cfg, w, clip[b])
        assert_close_16bit(got["out"][b], ref["out"], f"{name} clip {b}")
        for k, tap in enumerate(ref["hier"]):
            assert_close_16bit(got["hier"][k, b], tap, f"{name} tap {k} clip {b}")
        np.testing.assert_allclose(got["pooled"][b], ref["pooled"], atol=1e-2 * np.abs(ref["pooled"]).max())
    enc.close()


@pytest.mark.parametrize("name", ["v2-hd32-sharp", "b21-hd64-sharp"])
def test_sharp_attention_masked_encoder(jg, name):
    """The masked encoder on the sharp-attention models: each clip keeps its
    own random 45 % of the tokens in random order, so the RoPE positions come
    from the ids; every kept token against the oracle's masked forward."""
    from qkv_cases import SHARP_MODELS, sharp_weights
    cfg = SHARP_MODELS[name]
    w = sharp_weights(cfg)
    clip = synth.clip_u8(cfg)
    n = synth.tokens_per_clip(cfg)
    K = int(n * 0.45)
    keep = np.stack([np.random.default_rng(77 + b).choice(n, K, replace=False)
                     for b in range(cfg.batch)]).astype(np.int32)
    enc = jg.Encoder(cfg, w)
    got = enc.encode_masked(torch.from_numpy(clip).cuda(), torch.from_numpy(keep).cuda())["out"].cpu().numpy()
    enc.sync()
    for b in range(cfg.batch):
        ref = oracle.encoder_forward(cfg, w, clip[b], keep=keep[b])
        assert_close_16bit(got[b], ref["out"], f"{name} masked clip {b}")
    enc.close()


def test_two_handles_two_threads(jg):
    """Two encoder handles on device 0, used from two threads at the same
    time, each on its own stream (the launch set-up kept per device is done
    once under a lock; each handle has its own workspace and graphs).  Each
    thread encodes three times (eager, captured, replayed); every result
    matches the oracle and the three are identical."""
    import threading
    cfgs = [SMALL["b21-bf16"], SMALL["v2-hd32"]]
    results, errors = [None, None], []

    def work(i):
        try:
            cfg = cfgs[i]
            w = synth.encoder_weights(cfg)
            clip = synth.clip_u8(cfg)
            s = torch.cuda.Stream()
            enc = jg.Encoder(cfg, w)
            with torch.cuda.stream(s):
                c = torch.from_numpy(clip).cuda()
                outs = [enc.encode(c, stream=s)["out"] for _ in range(3)]
                enc.sync(s)
                outs = [o.cpu().numpy() for o in outs]
            enc.close()
            results[i] = (cfg, w, clip, outs)
        except Exception as e:  # reported below, in the test's thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for cfg, w, clip, outs in results:
        np.testing.assert_array_equal(outs[1], outs[0])
        np.testing.assert_array_equal(outs[2], outs[0])
        for b in range(cfg.batch):
            assert_close_16bit(outs[0][b], oracle.encoder_forward(cfg, w, clip[b])["out"], f"thread {cfg.name} {b}")
