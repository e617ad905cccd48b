"""Python face of the C ABI: argument marshalling only.

Every computation runs in libjepa_gb300.so; torch supplies device memory and
the current CUDA stream.  Tensors passed in must be contiguous and on the
device the handle was created for.
"""
from __future__ import annotations

import ctypes as C
import struct

import numpy as np
import torch

from . import _lib
from ._lib import EncoderParams, HeadParams, PredictorParams, check, load

DTYPE_CODE = {"f32": _lib.DT_F32, "f16": _lib.DT_F16, "bf16": _lib.DT_BF16}
TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
LAYOUT_CODE = {"tiled": 0, "interleaved": 1}


def _ptr(t) -> C.c_void_p:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream=None) -> C.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


# ----------------------------------------------------------------------------- weight blob
def encoder_tensor_order(cfg):
    """(name, is_matrix) in the blob order of the ABI header."""
    names = [("patch_embed.weight", True), ("patch_embed.bias", False)]
    if cfg.has_mod_embed:
        names.append(("mod_embed_video", False))
    for i in range(cfg.n_layer):
        p = f"blk.{i}."
        names += [(p + "ln1.weight", False), (p + "ln1.bias", False), (p + "attn_qkv.weight", True),
                  (p + "attn_qkv.bias", False), (p + "attn_out.weight", True), (p + "attn_out.bias", False),
                  (p + "ln2.weight", False), (p + "ln2.bias", False), (p + "ffn_up.weight", True),
                  (p + "ffn_up.bias", False), (p + "ffn_down.weight", True), (p + "ffn_down.bias", False)]
    names += [("norm.weight", False), ("norm.bias", False)]
    for k in range(len(cfg.hier_layers)):
        names += [(f"hier_norm.{k}.weight", False), (f"hier_norm.{k}.bias", False)]
    if getattr(cfg, "has_image_path", False):
        names += [("patch_embed_img.weight", True), ("patch_embed_img.bias", False)]
        if cfg.has_mod_embed:
            names.append(("mod_embed_img", False))
    return names


def predictor_tensor_order(pc):
    names = [("embed.weight", True), ("embed.bias", False), ("mask_tokens", False)]
    for i in range(pc.n_layer):
        p = f"blk.{i}."
        names += [(p + "ln1.weight", False), (p + "ln1.bias", False), (p + "attn_qkv.weight", True),
                  (p + "attn_qkv.bias", False), (p + "attn_out.weight", True), (p + "attn_out.bias", False),
                  (p + "ln2.weight", False), (p + "ln2.bias", False), (p + "ffn_up.weight", True),
                  (p + "ffn_up.bias", False), (p + "ffn_down.weight", True), (p + "ffn_down.bias", False)]
    names += [("norm.weight", False), ("norm.bias", False), ("proj.weight", True), ("proj.bias", False)]
    if getattr(pc, "has_mod_embed", False):
        names += [("mod_embed_video", False), ("mod_embed_img", False)]
    if getattr(pc, "has_proj_context", False):
        names += [("proj_context.weight", True), ("proj_context.bias", False)]
    return names


def _as_storage(a: np.ndarray, dtype: str) -> bytes:
    a = np.ascontiguousarray(a, dtype=np.float32)
    if dtype == "f32":
        return a.tobytes()
    t = torch.from_numpy(a).to(TORCH_DTYPE[dtype])
    return t.view(torch.int16).numpy().tobytes()


def pack_blob(order, weights: dict, dtype: str) -> bytes:
    """Serialises tensors into the ABI's blob format (2-D matrices in `dtype`,
    the rest fp32; mask_tokens stays fp32 though it is 2-D)."""
    entries, chunks = [], []
    off = 24 + 32 * len(order)
    off = (off + 255) // 256 * 256
    for name, is_mat in order:
        a = np.asarray(weights[name])
        dt = dtype if is_mat else "f32"
        data = _as_storage(a, dt)
        shape = a.shape if a.ndim == 2 else (a.shape[0], 1)
        entries.append(struct.pack("<QQIIII", off, len(data), DTYPE_CODE[dt], a.ndim, shape[0], shape[1]))
        chunks.append((off, data))
        off = (off + len(data) + 255) // 256 * 256
    buf = bytearray(off)
    buf[0:24] = b"JEPAGB3\0" + struct.pack("<IIQ", 1, len(order), 0)
    buf[24:24 + 32 * len(order)] = b"".join(entries)
    for o, d in chunks:
        buf[o:o + len(d)] = d
    return bytes(buf)


def encoder_params(cfg) -> EncoderParams:
    p = EncoderParams()
    p.embed_dim, p.n_layer, p.n_head, p.ffn_dim = cfg.embed_dim, cfg.n_layer, cfg.n_head, cfg.ffn_dim
    p.patch, p.tubelet = cfg.patch, cfg.tubelet
    p.ln_eps, p.rope_theta = cfg.ln_eps, cfg.rope_theta
    p.rope_layout = LAYOUT_CODE[cfg.rope_layout]
    p.rope_interpolate = int(bool(cfg.rope_interpolate))
    p.rope_ref_grid = cfg.rope_ref_grid
    p.n_hier = len(cfg.hier_layers)
    for i, l in enumerate(cfg.hier_layers):
        p.hier_layers[i] = l
    p.has_mod_embed = int(bool(cfg.has_mod_embed))
    p.has_image_path = int(bool(getattr(cfg, "has_image_path", False)))
    p.dtype = DTYPE_CODE[cfg.dtype]
    return p


def predictor_params(pc, dtype: str) -> PredictorParams:
    p = PredictorParams()
    p.embed_dim, p.n_layer, p.n_head, p.ffn_dim = pc.embed_dim, pc.n_layer, pc.n_head, pc.ffn_dim
    p.in_dim, p.out_dim, p.n_mask_tokens, p.mask_index = pc.in_dim, pc.out_dim, pc.n_mask_tokens, pc.mask_index
    p.ln_eps, p.rope_theta = pc.ln_eps, pc.rope_theta
    p.rope_layout = LAYOUT_CODE[pc.rope_layout]
    p.dtype = DTYPE_CODE[dtype]
    p.has_mod_embed = int(bool(getattr(pc, "has_mod_embed", False)))
    p.has_proj_context = int(bool(getattr(pc, "has_proj_context", False)))
    return p


def blob_check(cfg, blob: bytes) -> None:
    lib = load()
    p = encoder_params(cfg)
    check(lib.jepa_blob_check(blob, len(blob), C.byref(p)))


# ----------------------------------------------------------------------------- encoder
class Encoder:
    """A V-JEPA 2 / 2.1 encoder resident on one GPU."""

    def __init__(self, cfg, weights: dict, device: int = 0, blob: bytes | None = None):
        self.lib = load()
        self.cfg = cfg
        self.device = device
        self.params = encoder_params(cfg)
        blob = blob if blob is not None else pack_blob(encoder_tensor_order(cfg), weights, cfg.dtype)
        h = C.c_void_p()
        with torch.cuda.device(device):
            check(self.lib.jepa_encoder_create(blob, len(blob), C.byref(self.params), device, C.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self.lib.jepa_encoder_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def n_tokens(self, T, H, W):
        # one frame on a model with the 2.1 image path: tubelet 1
        tub = 1 if (T == 1 and getattr(self.cfg, "has_image_path", False)) else self.cfg.tubelet
        return (T // tub) * (H // self.cfg.patch) * (W // self.cfg.patch)

    def encode(self, clip: torch.Tensor, pooled: bool = False, hier: bool = False, out=None, stream=None):
        """clip: uint8 [B,T,H,W,3] (or float [B,3,T,H,W] normalised) on the device."""
        fmt = _lib.CLIP_U8_THWC if clip.dtype == torch.uint8 else _lib.CLIP_F32_CTHW
        if fmt == _lib.CLIP_U8_THWC:
            B, T, H, W, _ = clip.shape
        else:
            B, _, T, H, W = clip.shape
        N, D = self.n_tokens(T, H, W), self.cfg.embed_dim
        dev = clip.device
        out = out if out is not None else torch.empty((B, N, D), dtype=torch.float32, device=dev)
        pool = torch.empty((B, D), dtype=torch.float32, device=dev) if pooled else None
        nh = len(self.cfg.hier_layers)
        taps = torch.empty((nh, B, N, D), dtype=torch.float32, device=dev) if (hier and nh) else None
        check(self.lib.jepa_encode(self.handle, _ptr(clip), fmt, B, T, H, W, _ptr(out), _ptr(pool), _ptr(taps),
                                   _stream(stream)))
        res = {"out": out}
        if pool is not None:
            res["pooled"] = pool
        if taps is not None:
            res["hier"] = taps
        return res

    def encode_masked(self, clip: torch.Tensor, ids_keep: torch.Tensor, pooled: bool = False, hier: bool = False,
                      stream=None, out=None):
        """Masked encoder forward: only the tokens ids_keep [B, K] (int32,
        device) of each clip go through the blocks, at their true positions."""
        fmt = _lib.CLIP_U8_THWC if clip.dtype == torch.uint8 else _lib.CLIP_F32_CTHW
        B, T, H, W = (clip.shape[:4] if fmt == _lib.CLIP_U8_THWC else (clip.shape[0],) + tuple(clip.shape[2:5]))
        K, D = ids_keep.shape[1], self.cfg.embed_dim
        dev = clip.device
        out = out if out is not None else torch.empty((B, K, D), dtype=torch.float32, device=dev)
        pool = torch.empty((B, D), dtype=torch.float32, device=dev) if pooled else None
        nh = len(self.cfg.hier_layers)
        taps = torch.empty((nh, B, K, D), dtype=torch.float32, device=dev) if (hier and nh) else None
        ids = ids_keep.to(dtype=torch.int32).contiguous()
        check(self.lib.jepa_encode_masked(self.handle, _ptr(clip), fmt, B, T, H, W, _ptr(ids), K, _ptr(out),
                                          _ptr(pool), _ptr(taps), _stream(stream)))
        res = {"out": out}
        if pool is not None:
            res["pooled"] = pool
        if taps is not None:
            res["hier"] = taps
        return res

    def encode_host(self, clip: torch.Tensor, out: torch.Tensor, pooled: torch.Tensor | None = None, stream=None):
        """Host (ideally pinned) uint8 clip in, host float out; synchronous."""
        B, T, H, W, _ = clip.shape
        check(self.lib.jepa_encode_host(self.handle, _ptr(clip), _lib.CLIP_U8_THWC, B, T, H, W, _ptr(out),
                                        _ptr(pooled), _stream(stream)))

    def encode_host_async(self, clip: torch.Tensor, out: torch.Tensor, pooled: torch.Tensor | None = None,
                          stream=None):
        """Host (ideally pinned) uint8 clip in, host float out; returns at once.
        Neither buffer may be touched until sync(stream) returns."""
        B, T, H, W, _ = clip.shape
        check(self.lib.jepa_encode_host_async(self.handle, _ptr(clip), _lib.CLIP_U8_THWC, B, T, H, W, _ptr(out),
                                              _ptr(pooled), _stream(stream)))

    def embed(self, clip: torch.Tensor, stream=None) -> torch.Tensor:
        B, T, H, W, _ = clip.shape
        x = torch.empty((B * self.n_tokens(T, H, W), self.cfg.embed_dim), dtype=torch.float32, device=clip.device)
        check(self.lib.jepa_encoder_embed(self.handle, _ptr(clip), _lib.CLIP_U8_THWC, B, T, H, W, _ptr(x),
                                          _stream(stream)))
        return x

    def blocks(self, x: torch.Tensor, batch, T, H, W, l0, l1, stream=None) -> torch.Tensor:
        check(self.lib.jepa_encoder_blocks(self.handle, _ptr(x), batch, T, H, W, l0, l1, _stream(stream)))
        return x

    def sync(self, stream=None):
        check(self.lib.jepa_encoder_sync(self.handle, _stream(stream)))

    def set_graphs(self, on: bool):
        """Replay of repeated encode calls as one CUDA graph (on by default)."""
        check(self.lib.jepa_encoder_set_graphs(self.handle, int(bool(on))))

    def set_profiling(self, on: bool):
        check(self.lib.jepa_encoder_set_profiling(self.handle, int(on)))

    def profile(self, reset: bool = True):
        t = (C.c_double * 8)()
        n = (C.c_longlong * 8)()
        check(self.lib.jepa_encoder_profile(self.handle, t, n, int(reset)))
        names = ["patch_embed", "layernorm", "qkv_gemm", "attention", "out_proj_gemm", "ffn_up_gemm",
                 "ffn_down_gemm", "other"]
        return {k: (t[i], n[i]) for i, k in enumerate(names)}

    def workspace_bytes(self, B, T, H, W) -> int:
        return int(self.lib.jepa_encode_workspace_bytes(self.handle, B, T, H, W))


class Predictor:
    """The V-JEPA 2 / 2.1 masked predictor resident on one GPU."""

    def __init__(self, pcfg, weights: dict, dtype: str, device: int = 0):
        self.lib = load()
        self.pcfg = pcfg
        self.params = predictor_params(pcfg, dtype)
        blob = pack_blob(predictor_tensor_order(pcfg), weights, dtype)
        h = C.c_void_p()
        with torch.cuda.device(device):
            check(self.lib.jepa_predictor_create(blob, len(blob), C.byref(self.params), device, C.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self.lib.jepa_predictor_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_graphs(self, on: bool):
        """Replay of repeated predict calls as one CUDA graph (on by default)."""
        check(self.lib.jepa_predictor_set_graphs(self.handle, int(bool(on))))

    def predict(self, enc_tokens: torch.Tensor, ids_ctx: torch.Tensor, ids_tgt: torch.Tensor, grid, stream=None,
                modality: str | None = None, with_ctx: bool = False, out=None, out_ctx=None):
        """Target predictions [n_tgt, out_dim]; with ``with_ctx`` also the
        context projection [n_ctx, out_dim] (2.1), as ``(pred, ctx)``.
        modality: None (the plain call: video), "video", "image" or "auto"."""
        out = out if out is not None else torch.empty((ids_tgt.numel(), self.pcfg.out_dim), dtype=torch.float32,
                                                      device=enc_tokens.device)
        gt, gh, gw = grid
        if modality is None and not with_ctx:
            check(self.lib.jepa_predict(self.handle, _ptr(enc_tokens), enc_tokens.shape[0], _ptr(ids_ctx),
                                        ids_ctx.numel(), _ptr(ids_tgt), ids_tgt.numel(), gt, gh, gw, _ptr(out),
                                        _stream(stream)))
            return out
        mod = {None: _lib.MODALITY_VIDEO, "video": _lib.MODALITY_VIDEO, "image": _lib.MODALITY_IMAGE,
               "auto": _lib.MODALITY_AUTO}[modality]
        ctx = (out_ctx if out_ctx is not None else
               torch.empty((ids_ctx.numel(), self.pcfg.out_dim), dtype=torch.float32, device=enc_tokens.device)
               ) if with_ctx else None
        check(self.lib.jepa_predict_ex(self.handle, _ptr(enc_tokens), enc_tokens.shape[0], _ptr(ids_ctx),
                                       ids_ctx.numel(), _ptr(ids_tgt), ids_tgt.numel(), gt, gh, gw, mod, _ptr(out),
                                       _ptr(ctx), _stream(stream)))
        return (out, ctx) if with_ctx else out

    def sync(self, stream=None):
        check(self.lib.jepa_predictor_sync(self.handle, _stream(stream)))


# ----------------------------------------------------------------------------- attentive-pool head
def head_tensor_order(hc):
    """(name, is_matrix) in the head blob order of the ABI header."""
    names = [("head.query", False)]
    for i in range(hc.n_layer):
        p = f"head.blk.{i}."
        names += [(p + "ln1.weight", False), (p + "ln1.bias", False), (p + "attn_qkv.weight", True),
                  (p + "attn_qkv.bias", False), (p + "attn_out.weight", True), (p + "attn_out.bias", False),
                  (p + "ln2.weight", False), (p + "ln2.bias", False), (p + "ffn_up.weight", True),
                  (p + "ffn_up.bias", False), (p + "ffn_down.weight", True), (p + "ffn_down.bias", False)]
    x = "head.xattn."
    names += [(x + "ln_kv.weight", False), (x + "ln_kv.bias", False), (x + "q.weight", True), (x + "q.bias", False),
              (x + "k.weight", True), (x + "k.bias", False), (x + "v.weight", True), (x + "v.bias", False),
              (x + "ln2.weight", False), (x + "ln2.bias", False), (x + "ffn_up.weight", True),
              (x + "ffn_up.bias", False), (x + "ffn_down.weight", True), (x + "ffn_down.bias", False),
              ("head.cls.weight", True), ("head.cls.bias", False)]
    return names


def head_params(hc, dtype: str) -> HeadParams:
    p = HeadParams()
    p.embed_dim, p.n_layer, p.n_head, p.ffn_dim = hc.embed_dim, hc.n_layer, hc.n_head, hc.ffn_dim
    p.n_classes, p.ln_eps, p.dtype = hc.n_classes, hc.ln_eps, DTYPE_CODE[dtype]
    return p


class Head:
    """The attentive-pool head and classifier resident on one GPU."""

    def __init__(self, hc, weights: dict, dtype: str, device: int = 0):
        self.lib = load()
        self.hc = hc
        self.params = head_params(hc, dtype)
        blob = pack_blob(head_tensor_order(hc), weights, dtype)
        h = C.c_void_p()
        with torch.cuda.device(device):
            check(self.lib.jepa_head_create(blob, len(blob), C.byref(self.params), device, C.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self.lib.jepa_head_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, tokens: torch.Tensor, pooled: bool = False, stream=None, out=None):
        """tokens: float [B, N, D] on the device.  Returns logits [B, n_classes]
        (and pooled [B, D] when asked, as (logits, pooled))."""
        B, N, _ = tokens.shape
        logits = out if out is not None else torch.empty((B, self.hc.n_classes), dtype=torch.float32,
                                                         device=tokens.device)
        pool = torch.empty((B, self.hc.embed_dim), dtype=torch.float32, device=tokens.device) if pooled else None
        check(self.lib.jepa_head_forward(self.handle, _ptr(tokens), B, N, _ptr(logits), _ptr(pool), _stream(stream)))
        return (logits, pool) if pooled else logits

    def sync(self, stream=None):
        check(self.lib.jepa_head_sync(self.handle, _stream(stream)))

    def set_graphs(self, on: bool):
        """Replay of repeated forward calls as one CUDA graph (on by default)."""
        check(self.lib.jepa_head_set_graphs(self.handle, int(bool(on))))


# ----------------------------------------------------------------------------- single operations
def layernorm_f32(x: torch.Tensor, w: torch.Tensor, b: torch.Tensor, eps: float, out=None) -> torch.Tensor:
    out = out if out is not None else torch.empty_like(x)
    rows, dim = x.shape
    check(load().jepa_layernorm_f32(_ptr(x), _ptr(w), _ptr(b), _ptr(out), rows, dim, eps, _stream()))
    return out


def rope3d_f32(x: torch.Tensor, grid, n_head: int, head_dim: int, layout: str, interpolate: bool = False,
               ref_grid: int = 16, theta: float = 10000.0) -> torch.Tensor:
    """In place on x [B, N, n_head*head_dim] fp32."""
    B, N, _ = x.shape
    gt, gh, gw = grid
    check(load().jepa_rope3d_f32(_ptr(x), B, N, n_head, head_dim, gt, gh, gw, LAYOUT_CODE[layout],
                                 int(interpolate), ref_grid, theta, _stream()))
    return x


def attention(q, k, vt, batch, n_head, n_tokens, head_dim, scale=None, out=None):
    """q, k [B*h, N, hd]; vt [B*h, hd, ldv]; returns [B, N, h*hd] in q's dtype."""
    dt = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[q.dtype]
    out = out if out is not None else torch.empty((batch, n_tokens, n_head * head_dim), dtype=q.dtype,
                                                  device=q.device)
    scale = scale if scale is not None else head_dim ** -0.5
    check(load().jepa_attention(_ptr(q), _ptr(k), _ptr(vt), _ptr(out), DTYPE_CODE[dt], batch, n_head, n_tokens,
                                head_dim, vt.shape[-1], scale, _stream()))
    return out


def linear(A, W, bias, epilogue: int, out=None):
    dt = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[A.dtype]
    M, K = A.shape
    N = W.shape[0]
    if out is None:
        odt = torch.float32 if epilogue in (1, 2) else A.dtype
        out = torch.empty((M, N), dtype=odt, device=A.device)
    check(load().jepa_linear(_ptr(A), _ptr(W), _ptr(bias), _ptr(out), M, N, K, DTYPE_CODE[dt], epilogue, _stream()))
    return out


def qkv_rope(A, W, bias, batch: int, n_tokens: int, n_head: int, grid, layout: str, interpolate: bool = False,
             ref_grid: int = 16, theta: float = 10000.0, pos_ids=None, out=None):
    """Fused QKV projection + 3-D RoPE: A [batch*n_tokens, D], W [3D, D] in one
    dtype, bias float [3D] or None, pos_ids int32 [batch*n_tokens] or None.
    Returns (q, k, vt): q, k [batch*n_head, n_tokens, hd] and vt
    [batch*n_head, hd, ldv] (columns >= n_tokens zeroed here, never written)."""
    dt = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[A.dtype]
    D = A.shape[1]
    hd = D // n_head
    ldv = (n_tokens + 7) // 8 * 8
    if out is None:
        q = torch.empty((batch * n_head, n_tokens, hd), dtype=A.dtype, device=A.device)
        k = torch.empty_like(q)
        vt = torch.zeros((batch * n_head, hd, ldv), dtype=A.dtype, device=A.device)
    else:
        q, k, vt = out
        ldv = vt.shape[-1]
    gt, gh, gw = grid
    ids = pos_ids.to(dtype=torch.int32).contiguous() if pos_ids is not None else None
    check(load().jepa_qkv_rope(_ptr(A), _ptr(W), _ptr(bias), _ptr(q), _ptr(k), _ptr(vt), DTYPE_CODE[dt], batch,
                               n_tokens, D, n_head, ldv, gt, gh, gw, LAYOUT_CODE[layout], int(bool(interpolate)),
                               ref_grid, theta, _ptr(ids), _stream()))
    return q, k, vt


def ops_sync():
    check(load().jepa_ops_sync(_stream()))


def selftest_wait_timeout(timeout_us: int) -> int:
    """Returns the status code (JEPA_ERR_DEVICE_TIMEOUT expected)."""
    return int(load().jepa_selftest_wait_timeout(timeout_us, _stream()))
