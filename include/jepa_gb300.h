/*
 * jepa_gb300.h - C ABI of the GB300 (sm_103a) V-JEPA 2 / 2.1 video ViT encoder.
 *
 * The library computes the forward pass of the V-JEPA 2 / 2.1 video ViT
 * encoder ("V-JEPA 2 / 2.1 tensor maps and RoPE derivation", §2 block form,
 * §3 2.1 encoder forward, §4 3-D RoPE) and of the V-JEPA 2 masked predictor
 * (same page, §2 key map, §3 predictor forward, §4.4 predictor ids), on one
 * GPU, in hand-written CUDA kernels.
 *
 * Conventions for every entry point:
 *   - Buffers documented as device buffers are CUDA device pointers owned by
 *     the caller.  Pointers documented as host pointers are host memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is enqueued asynchronously on it; the call returns
 *     once the work is enqueued unless the entry point says otherwise.
 *   - Every function returns a jepa_status.  Argument errors are found on the
 *     host before anything is launched; nothing is enqueued then.  The
 *     message of the calling thread's last non-OK status is returned by
 *     jepa_last_error().  No C++ exception crosses this boundary.
 *   - Bounded device waits: kernels that wait on an mbarrier give up after a
 *     time limit and set a device status word instead of hanging; the next
 *     jepa_encoder_sync / jepa_predictor_sync reports it as
 *     JEPA_ERR_DEVICE_TIMEOUT.
 *   - Layouts are row-major, innermost dimension last.
 *   - Calls on one handle must not overlap in time, on the host or on the
 *     device (a handle owns one workspace): either every call on a handle
 *     uses the same stream, or the caller synchronises before switching.
 */
#ifndef JEPA_GB300_H
#define JEPA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define JEPA_ABI_VERSION 6  /* 2: jepa_encoder_params.has_image_path; 3: 2.1 predictor fields;
                               4: jepa_encode_host_async; 5: jepa_qkv_rope; 6: attentive-pool head */

#if defined(__GNUC__)
#define JEPA_API __attribute__((visibility("default")))
#else
#define JEPA_API
#endif

typedef enum {
  JEPA_OK = 0,
  JEPA_ERR_ARG = 1,            /* bad argument (null pointer, size, unsupported shape)      */
  JEPA_ERR_BLOB = 2,           /* weight blob truncated, wrong magic, or tensor mismatch    */
  JEPA_ERR_UNSUPPORTED = 3,    /* valid but not implemented (e.g. head_dim not 32 or 64)    */
  JEPA_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed                         */
  JEPA_ERR_OOM = 5,            /* device allocation failed                                  */
  JEPA_ERR_DEVICE_TIMEOUT = 6  /* a kernel gave up waiting on a barrier (reported at sync)  */
} jepa_status;

typedef enum { JEPA_DT_F32 = 0, JEPA_DT_F16 = 1, JEPA_DT_BF16 = 2 } jepa_dtype;
typedef enum { JEPA_ROPE_TILED = 0, JEPA_ROPE_INTERLEAVED = 1 } jepa_rope_layout;
typedef enum { JEPA_CLIP_U8_THWC = 0, JEPA_CLIP_F32_CTHW = 1 } jepa_clip_format;
/* Which 2.1 predictor modality vector joins every row (AUTO: image for a
 * grid of one temporal slice, the grid of the 2.1 image path). */
typedef enum { JEPA_MODALITY_VIDEO = 0, JEPA_MODALITY_IMAGE = 1, JEPA_MODALITY_AUTO = 2 } jepa_modality;

/* Encoder hyper-parameters ("V-JEPA 2 / 2.1 tensor maps and RoPE derivation",
 * §1).  head_dim = embed_dim / n_head must be 32 or 64.  patch must be 16 and
 * tubelet 2 (the Conv3d [D,3,2,16,16] of §2).  rope_layout: tiled (V-JEPA 2,
 * §4.1) or interleaved (V-JEPA 2.1, §4.2).  rope_interpolate rescales spatial
 * positions by (rope_ref_grid-1)/(n-1) (§4.3).  hier_layers (0-based block
 * indices, increasing) select the hierarchical LayerNorm taps (§3).
 * has_mod_embed adds the 2.1 video modality vector after the patch embed (§3).
 * dtype: storage type of the 2-D matrices and of the activations fed to the
 * matrix multiplies (F32 = fp32 CUDA-core path; F16/BF16 = tensor-core path
 * with fp32 accumulation).  The residual stream, LayerNorm statistics,
 * softmax and all outputs are fp32 in every mode.
 * has_image_path: the blob also holds the 2.1 native image path (§2
 * patch_embed_img [D,3,1,16,16] and, with has_mod_embed, img_mod_embed); a
 * one-frame input then takes it (§3, 2.1 encoder forward; Meta's code selects
 * it by the frame count). */
typedef struct jepa_encoder_params {
  int embed_dim, n_layer, n_head, ffn_dim;
  int patch, tubelet;
  float ln_eps, rope_theta;
  int rope_layout, rope_interpolate, rope_ref_grid;
  int n_hier;
  int hier_layers[4];
  int has_mod_embed;
  int dtype;
  int has_image_path;
} jepa_encoder_params;

/* Masked predictor hyper-parameters (same page, §1 "pred.*" rows).
 * in_dim = encoder width; out_dim = projection width; the mask token used for
 * every target row is mask_tokens[mask_index % n_mask_tokens]. */
typedef struct jepa_predictor_params {
  int embed_dim, n_layer, n_head, ffn_dim;
  int in_dim, out_dim, n_mask_tokens, mask_index;
  float ln_eps, rope_theta;
  int rope_layout;
  int dtype;
  int has_mod_embed;     /* 2.1: pred.mod_embed_video / pred.mod_embed_img added to every row (§3) */
  int has_proj_context;  /* 2.1: pred.proj_context [out_dim,D] on the context rows (§2, §3) */
} jepa_predictor_params;

/* ---------------------------------------------------------------- weight blob
 * Little-endian.  Header: char magic[8] = "JEPAGB3\0", uint32 version (1),
 * uint32 n_tensors, uint64 reserved, then n_tensors entries of
 * {uint64 offset, uint64 nbytes, uint32 dtype, uint32 ndim, uint32 dim0,
 *  uint32 dim1} (offset from the blob start, 256-byte aligned).
 * Encoder tensor order (names of §2 of the conversion notes):
 *   patch_embed.weight [D,1536] (feature order C,T,H,W), patch_embed.bias [D],
 *   [mod_embed_video [D] if has_mod_embed],
 *   per block i: ln1.weight, ln1.bias [D], attn_qkv.weight [3D,D] (rows q;k;v),
 *   attn_qkv.bias [3D], attn_out.weight [D,D], attn_out.bias [D],
 *   ln2.weight, ln2.bias [D], ffn_up.weight [F,D], ffn_up.bias [F],
 *   ffn_down.weight [D,F], ffn_down.bias [D];
 *   norm.weight, norm.bias [D]; then hier_norm.k.weight/bias [D] per tap;
 *   then, if has_image_path: patch_embed_img.weight [D,768] (feature order
 *   C,H,W), patch_embed_img.bias [D], [mod_embed_img [D] if has_mod_embed].
 * Predictor order: embed.weight [D,in_dim], embed.bias [D], mask_tokens
 *   [n_mask,D] (fp32), the blocks as above, norm.weight/bias, proj.weight
 *   [out_dim,D], proj.bias [out_dim]; then [mod_embed_video [D],
 *   mod_embed_img [D] if has_mod_embed]; then [proj_context.weight
 *   [out_dim,D], proj_context.bias [out_dim] if has_proj_context].
 * 2-D matrices are stored in params.dtype, everything else in F32. */

/* Host-only validation of a blob against params (no GPU needed). */
JEPA_API jepa_status jepa_blob_check(const void* blob, size_t blob_bytes, const jepa_encoder_params* params);
JEPA_API jepa_status jepa_predictor_blob_check(const void* blob, size_t blob_bytes, const jepa_predictor_params* params);

/* ---------------------------------------------------------------- encoder
 * jepa_encoder_create: validates params and the host blob, makes `device`
 * current, copies the weights to device memory (owned by the handle until
 * jepa_encoder_destroy).  The blob may be freed after the call.  Supported
 * widths (JEPA_ERR_UNSUPPORTED otherwise): embed_dim a multiple of 128 (at
 * most 4096) with head_dim 32 or 64; ffn_dim a multiple of 128 (64 for F32);
 * the same for the predictor and the head, and a predictor out_dim a
 * multiple of 128 (32 for F32). */
typedef struct jepa_encoder jepa_encoder;
JEPA_API jepa_status jepa_encoder_create(const void* blob, size_t blob_bytes, const jepa_encoder_params* params,
                                int device, jepa_encoder** out);
JEPA_API void jepa_encoder_destroy(jepa_encoder* enc);

/* Bytes of device workspace jepa_encode allocates (once, grown on demand)
 * for this clip shape; 0 on invalid arguments. */
JEPA_API size_t jepa_encode_workspace_bytes(const jepa_encoder* enc, int batch, int n_frames, int height, int width);

/* jepa_encode: last_hidden_state of `batch` independent clips.
 *   clip: device buffer, JEPA_CLIP_U8_THWC: uint8 [batch, n_frames, H, W, 3]
 *         raw pixels, normalised inside with the ImageNet mean/std in the
 *         fused form (px - 255*mean)/(255*std) ("Parity ...", Preprocessing
 *         parity); JEPA_CLIP_F32_CTHW: float [batch, 3, n_frames, H, W]
 *         already normalised.
 *   n_frames even, or 1 on a model with has_image_path (the 2.1 native image
 *   path: tubelet 1, patch_embed_img, img_mod_embed, temporal position 0);
 *   H and W multiples of 16 (non-square allowed), H/16 > 1 and W/16 > 1
 *   when interpolating RoPE.  N = (n_frames/tubelet)*(H/16)*(W/16).
 *   out_tokens: device float [batch, N, D] = enc.norm(x) (required).
 *   out_pooled: device float [batch, D] token mean of out_tokens, or NULL.
 *   out_hier:   device float [n_hier, batch, N, D] hierarchical taps, or NULL.
 * The handle allocates its device workspace on the first call with a larger
 * shape (JEPA_ERR_OOM if that fails). */
JEPA_API jepa_status jepa_encode(jepa_encoder* enc, const void* clip, int clip_format, int batch, int n_frames,
                        int height, int width, float* out_tokens, float* out_pooled, float* out_hier,
                        void* stream);

/* jepa_encoder_set_graphs: replay of repeated jepa_encode and
 * jepa_encode_masked calls (on by default).  A call whose shapes and buffers
 * (and, masked, id buffer and count) equal an earlier call's runs as
 * one CUDA graph launch on `stream`: the first such call runs eagerly, the
 * second is captured (on a stream private to the handle) and later ones
 * replay it, so the host issues one launch instead of one per kernel and the
 * kernels follow each other without launch gaps.  The handle keeps graphs
 * for the 8 most recent signatures; a workspace reallocation drops them.
 * Calls made while profiling is on always run eagerly.  on = 0 turns replay
 * off. */
JEPA_API jepa_status jepa_encoder_set_graphs(jepa_encoder* enc, int on);

/* jepa_encode_masked: the masked encoder forward ("V-JEPA 2.1 ViT-B/16 384 -
 * HuggingFace port", Usage / Predictor and Validation): of each clip only the
 * n_keep tokens ids_keep[b*n_keep + r] (device int32 [batch, n_keep], ids in
 * the clip's grid) are embedded and passed through the blocks, so attention
 * sees only them, while RoPE gives each its true grid position.  Not the same
 * as gathering jepa_encode's output.  Outputs as jepa_encode with N = n_keep,
 * rows in the order of ids_keep.  Ids outside the grid are clamped so nothing
 * is read out of range, and the next sync reports JEPA_ERR_ARG. */
JEPA_API jepa_status jepa_encode_masked(jepa_encoder* enc, const void* clip, int clip_format, int batch,
                                        int n_frames, int height, int width, const int32_t* ids_keep, int n_keep,
                                        float* out_tokens, float* out_pooled, float* out_hier, void* stream);

/* Same computation from and to HOST buffers (pinned memory is fastest): copies
 * the clip to the device, encodes, copies out_tokens (and out_pooled if not
 * NULL) back, and synchronises `stream` before returning. */
JEPA_API jepa_status jepa_encode_host(jepa_encoder* enc, const void* host_clip, int clip_format, int batch,
                             int n_frames, int height, int width, float* host_out_tokens,
                             float* host_out_pooled, void* stream);

/* Streaming form of jepa_encode_host for a sequence of clips: enqueues the
 * copy of host_clip to the device, the encode on `stream` and the copy of the
 * result to host_out_tokens (and host_out_pooled if not NULL), and returns
 * without waiting.  Consecutive calls use two device staging slots in turn,
 * and the copies run on two streams of the handle, so one call's copy-in and
 * the previous call's copy-out overlap the encodes.  Events order each slot's
 * reuse: a slot's clip is overwritten only after the encode that read it, and
 * its output only after the copy that read it.
 * The caller keeps host_clip unchanged, and reads neither host output, until
 * jepa_encoder_sync(enc, stream) returns; that call waits for the copies too
 * and reports device-side errors.  Pinned host memory makes the copies truly
 * asynchronous; pageable memory still gives correct results.  Arguments and
 * errors found on the host are those of jepa_encode_host. */
JEPA_API jepa_status jepa_encode_host_async(jepa_encoder* enc, const void* host_clip, int clip_format, int batch,
                                            int n_frames, int height, int width, float* host_out_tokens,
                                            float* host_out_pooled, void* stream);

/* The two halves of jepa_encode, for checking one stage at a time:
 * jepa_encoder_embed writes the patch embedding (+ modality vector) of the
 * clip into x_out, device float [batch*N, D]; jepa_encoder_blocks runs blocks
 * [layer_begin, layer_end) in place on x (device float [batch*N, D]) for the
 * given clip geometry. */
JEPA_API jepa_status jepa_encoder_embed(jepa_encoder* enc, const void* clip, int clip_format, int batch, int n_frames,
                               int height, int width, float* x_out, void* stream);
JEPA_API jepa_status jepa_encoder_blocks(jepa_encoder* enc, float* x, int batch, int n_frames, int height, int width,
                                int layer_begin, int layer_end, void* stream);

/* Synchronises `stream` (and the copy streams of jepa_encode_host_async) and
 * reports a device-side timeout recorded by any earlier call on this handle
 * (then clears it). */
JEPA_API jepa_status jepa_encoder_sync(jepa_encoder* enc, void* stream);

/* Per-kernel-class device time of the calls made while profiling is on,
 * measured with CUDA events recorded on the call's stream around every
 * launch.  Classes: 0 patch embed, 1 LayerNorm, 2 QKV GEMM, 3 attention,
 * 4 out-proj GEMM, 5 FFN-up GEMM, 6 FFN-down GEMM, 7 other.  times_ms[8] and
 * launches[8] are host arrays (either may be NULL); reading synchronises. */
JEPA_API jepa_status jepa_encoder_set_profiling(jepa_encoder* enc, int on);
JEPA_API jepa_status jepa_encoder_profile(jepa_encoder* enc, double* times_ms, long long* launches, int reset);

/* ---------------------------------------------------------------- predictor
 * jepa_predict: V-JEPA 2 masked predictor over one clip's encoder tokens.
 *   enc_tokens: device float [n_tokens, in_dim] (the encoder's output);
 *   ids_ctx [n_ctx], ids_tgt [n_tgt]: device int32 token ids in the encoder
 *   grid grid_t x grid_h x grid_w (T-major), each < n_tokens;
 *   out: device float [n_tgt, out_dim] = pred.proj(pred.norm(z))[n_ctx:]. */
typedef struct jepa_predictor jepa_predictor;
JEPA_API jepa_status jepa_predictor_create(const void* blob, size_t blob_bytes, const jepa_predictor_params* params,
                                  int device, jepa_predictor** out);
JEPA_API void jepa_predictor_destroy(jepa_predictor* pred);
JEPA_API jepa_status jepa_predict(jepa_predictor* pred, const float* enc_tokens, int n_tokens, const int32_t* ids_ctx,
                         int n_ctx, const int32_t* ids_tgt, int n_tgt, int grid_t, int grid_h, int grid_w,
                         float* out, void* stream);
/* jepa_predict_ex: the same, with the 2.1 additions ("V-JEPA 2 / 2.1 tensor
 * maps and RoPE derivation", §3 2.1 predictor forward):
 *   modality: jepa_modality; selects pred.mod_embed_video or _img, added to
 *     every row before the blocks (ignored without has_mod_embed);
 *   out_ctx: device float [n_ctx, out_dim] = pred.proj_context(pred.norm(z))
 *     [:n_ctx], or NULL; non-NULL needs has_proj_context (else JEPA_ERR_ARG).
 * jepa_predict is jepa_predict_ex with JEPA_MODALITY_VIDEO and out_ctx NULL,
 * the default of the pages. */
JEPA_API jepa_status jepa_predict_ex(jepa_predictor* pred, const float* enc_tokens, int n_tokens,
                                     const int32_t* ids_ctx, int n_ctx, const int32_t* ids_tgt, int n_tgt,
                                     int grid_t, int grid_h, int grid_w, int modality, float* out, float* out_ctx,
                                     void* stream);
JEPA_API jepa_status jepa_predictor_sync(jepa_predictor* pred, void* stream);
/* Replay of repeated jepa_predict / jepa_predict_ex calls as one CUDA graph,
 * as jepa_encoder_set_graphs (on by default; the id buffers are read at run
 * time, so a replay sees their current contents). */
JEPA_API jepa_status jepa_predictor_set_graphs(jepa_predictor* pred, int on);

/* ---------------------------------------------------------------- attentive-pool head
 * The attentive-pool head and classifier on top of the encoder ("V-JEPA 2 /
 * 2.1 tensor maps and RoPE derivation", §1 head row: 3 pool layers, 174
 * classes for the SSv2 ViT-L/16 classifier; §2 key map head rows and
 * "Attentive-pool head - exact forward"), per clip:
 *   x = the clip's encoder tokens [N, D] (after enc.norm);
 *   n_layer pre-LN self-attention blocks on x, laid out like the encoder's
 *   blocks (fused q;k;v), with NO RoPE;
 *   q = query Wq^T + bq (the raw learned token, not normalised);
 *   kv = ln_kv(x); k = kv Wk^T + bk; v = kv Wv^T + bv;
 *   o = concat_h softmax(q_h k_h^T / sqrt(64)) v_h (no output projection);
 *   y = query + o; y += ffn_down(gelu(ffn_up(ln2(y))));
 *   pooled = y; logits = y Wcls^T + bcls (no final norm).
 * head_dim (embed_dim / n_head) must be 64 and embed_dim 256, 512, 768 or
 * 1024.  dtype as for the encoder: the storage type of the 2-D matrices and
 * of the pool blocks' matrix-multiply inputs; the cross-attention and the
 * per-clip tail run in fp32.
 * Blob tensor order (the §2 head names): query [D] (fp32); per pool block
 * the encoder block's 12 tensors (ln1, attn_qkv, attn_out, ln2, ffn_up,
 * ffn_down); xattn.ln_kv.weight/bias [D]; xattn.q.weight [D,D], .bias [D];
 * xattn.k.*, xattn.v.* likewise; xattn.ln2.weight/bias [D];
 * xattn.ffn_up.weight [F,D], .bias [F]; xattn.ffn_down.weight [D,F],
 * .bias [D]; cls.weight [n_classes,D], cls.bias [n_classes]. */
typedef struct jepa_head_params {
  int embed_dim, n_layer, n_head, ffn_dim, n_classes;
  float ln_eps;
  int dtype;
} jepa_head_params;
typedef struct jepa_head jepa_head;
JEPA_API jepa_status jepa_head_blob_check(const void* blob, size_t blob_bytes, const jepa_head_params* params);
/* Validates params and the host blob, makes `device` current, copies the
 * weights to device memory (owned by the handle until jepa_head_destroy) and
 * derives the query's projections from them.  The blob may be freed after. */
JEPA_API jepa_status jepa_head_create(const void* blob, size_t blob_bytes, const jepa_head_params* params,
                                      int device, jepa_head** out);
JEPA_API void jepa_head_destroy(jepa_head* head);
/* tokens: device float [batch, n_tokens, D] (jepa_encode's out_tokens; not
 * modified); logits: device float [batch, n_classes]; pooled: device float
 * [batch, D] (the classifier input) or NULL.  Clips are independent.  The
 * handle grows its device workspace on the first call with a larger shape. */
JEPA_API jepa_status jepa_head_forward(jepa_head* head, const float* tokens, int batch, int n_tokens, float* logits,
                                       float* pooled, void* stream);
/* Synchronises `stream` and reports a device-side timeout of an earlier call. */
JEPA_API jepa_status jepa_head_sync(jepa_head* head, void* stream);
/* Replay of repeated jepa_head_forward calls with the same buffers and shapes
 * as one CUDA graph, as jepa_encoder_set_graphs (on by default). */
JEPA_API jepa_status jepa_head_set_graphs(jepa_head* head, int on);

/* ---------------------------------------------------------------- single operations
 * The kernels of the encoder, callable one at a time (the same code runs
 * inside jepa_encode).  All buffers are device buffers. */

/* LayerNorm over the last dimension, biased centred variance, eps inside the
 * square root ("V-JEPA 2 / 2.1 ...", §1 ln_eps; "Parity ...", Parity on a
 * GPU: two-pass variance).  x, y: float [rows, dim]; w, b: float [dim].
 * dim % 128 == 0 and dim <= 4096.  In place (y == x) is allowed. */
JEPA_API jepa_status jepa_layernorm_f32(const float* x, const float* w, const float* b, float* y, int rows, int dim,
                               float eps, void* stream);

/* 3-D RoPE in place on x: float [batch, n_tokens, n_head*head_dim] (q or k,
 * heads concatenated), positions of token i decoded T-major from the grid
 * grid_t x grid_h x grid_w with n_tokens = grid_t*grid_h*grid_w ("V-JEPA 2 /
 * 2.1 ...", §4: split d = 2*((head_dim//3)//2), §4.1 tiled, §4.2 interleaved,
 * §4.3 interpolation).  head_dim 32 or 64. */
JEPA_API jepa_status jepa_rope3d_f32(float* x, int batch, int n_tokens, int n_head, int head_dim, int grid_t, int grid_h,
                            int grid_w, int layout, int interpolate, int ref_grid, float theta, void* stream);

/* Unmasked softmax attention, softmax(scale * q k^T) v per (clip, head)
 * ("V-JEPA 2 / 2.1 ...", §2 concat_heads, §4: scale 1/sqrt(head_dim)).
 *   q, k: dtype [batch*n_head, n_tokens, head_dim];
 *   vt:   dtype [batch*n_head, head_dim, ldv] (V transposed, ldv >= n_tokens,
 *         ldv % 8 == 0, padding columns finite);
 *   out:  dtype [batch, n_tokens, n_head*head_dim] (heads concatenated).
 * head_dim 32 or 64; fp32 softmax statistics and accumulators. */
JEPA_API jepa_status jepa_attention(const void* q, const void* k, const void* vt, void* out, int dtype, int batch,
                           int n_head, int n_tokens, int head_dim, int ldv, float scale, void* stream);

/* Linear layer out = A W^T + bias with a fused epilogue, fp32 accumulation.
 *   A: dtype [M, K]; W: dtype [N, K]; bias: float [N] or NULL.
 *   epilogue 0: out dtype [M, N] = acc + bias
 *            1: out float [M, N] = acc + bias
 *            2: out float [M, N] += acc + bias   (residual add in place)
 *            3: out dtype [M, N] = gelu_erf(acc + bias)
 * F16/BF16 (tensor cores): K % 64 == 0, N % 128 == 0 (whole 128-column
 * output tiles; JEPA_ERR_ARG otherwise).  F32: K % 16 == 0, N % 4 == 0. */
JEPA_API jepa_status jepa_linear(const void* A, const void* W, const float* bias, void* out, int M, int N, int K, int dtype,
                        int epilogue, void* stream);

/* The fused QKV projection with 3-D RoPE, the first half of a block's
 * attention ("V-JEPA 2 / 2.1 tensor maps and RoPE derivation", §2 fused
 * attn_qkv with rows q;k;v and concat_heads; §4 RoPE on q and k after the
 * bias: split d = 2*((head_dim//3)//2) per axis t, h, w, the last
 * head_dim - 3d dims passed through; §4.1 tiled, §4.2 interleaved; §4.3
 * positions p*(ref_grid-1)/(n-1) on the spatial axes; §4.4 positions taken
 * from token ids).  The same kernels and epilogue as inside jepa_encode:
 *   qkv[r, :] = A[r, :] W^T + bias,   r < M = batch*n_tokens;
 *   q[b*n_head + h, i, :] = RoPE(qkv[b*n_tokens + i, h*hd : (h+1)*hd])
 *   k[b*n_head + h, i, :] = RoPE(qkv[b*n_tokens + i, D + h*hd : ...])
 *   vt[b*n_head + h, :, i] = qkv[b*n_tokens + i, 2D + h*hd : ...]
 * with the position of row r the grid cell (t, h, w) of id pos_ids[r]
 * (T-major in grid_t x grid_h x grid_w), or of id i = r mod n_tokens when
 * pos_ids is NULL (then grid_t*grid_h*grid_w must equal n_tokens).  q and k
 * are NOT scaled by 1/sqrt(head_dim): the attention applies the scale.
 *   A: dtype [batch*n_tokens, D]; W: dtype [3D, D]; bias: float [3D] or NULL;
 *   q, k: dtype [batch*n_head, n_tokens, head_dim]; vt: dtype
 *   [batch*n_head, head_dim, ldv], ldv >= n_tokens, ldv % 8 == 0 (columns
 *   >= n_tokens are not written); pos_ids: device int32 [batch*n_tokens] or
 *   NULL; ids outside the grid are clamped and reported by jepa_ops_sync as
 *   JEPA_ERR_ARG.
 * D = embed_dim a multiple of 128 (<= 4096), head_dim = D/n_head 32 or 64;
 * dtype F16/BF16 runs the tensor-core GEMM with the RoPE in its epilogue,
 * F32 the CUDA-core GEMM.  All buffers are caller-owned device buffers. */
JEPA_API jepa_status jepa_qkv_rope(const void* A, const void* W, const float* bias, void* q, void* k, void* vt,
                                   int dtype, int batch, int n_tokens, int embed_dim, int n_head, int ldv,
                                   int grid_t, int grid_h, int grid_w, int layout, int interpolate, int ref_grid,
                                   float theta, const int32_t* pos_ids, void* stream);

/* Synchronises `stream` and reports a device-side timeout recorded by any
 * earlier single-operation call (jepa_attention, jepa_linear, jepa_qkv_rope)
 * of this process (then clears it), or ids outside the grid given to
 * jepa_qkv_rope (JEPA_ERR_ARG). */
JEPA_API jepa_status jepa_ops_sync(void* stream);

/* Failure-detection self test: launches one kernel that waits on a barrier
 * that nothing completes, with a limit of timeout_us microseconds, then
 * synchronises.  Returns JEPA_ERR_DEVICE_TIMEOUT when the kernel reported
 * the expired wait (the expected outcome); the context stays usable. */
JEPA_API jepa_status jepa_selftest_wait_timeout(int timeout_us, void* stream);

/* Patch embedding that allocates no device memory.  The paper has no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc themselves, such as a host application or inference server that
 * owns all device memory through its own pool, or a latency-critical loop that
 * cannot afford cudaMalloc's device-wide synchronisation or its failure under
 * memory pressure.  It computes what jepa_encoder_embed computes, without an
 * encoder handle:
 *   clip:   device uint8 [batch, n_frames, height, width, 3] (THWC);
 *   weight: device dtype [embed_dim, 1536] (the patch-embed matrix, feature
 *           order C,T,H,W); bias: device float [embed_dim] or NULL;
 *   x_out:  device float [batch*N, embed_dim], N = (n_frames/2)(height/16)(width/16);
 *   status: optional device int the kernels OR 1 into if a barrier wait
 *           expired (read it after synchronising); NULL uses a library word
 *           that is not reported;
 *   dtype:  JEPA_DT_BF16 or JEPA_DT_F16.
 * The unfolded patches live in a static device array of 4096 token rows x
 * 1536 16-bit values (12 MiB) that every GPU loading the library holds until
 * the process exits; batch*N above 4096 is rejected with JEPA_ERR_ARG before
 * anything is launched.  All calls on a device share that array: calls whose
 * GPU work overlaps race on it.  The first call on each device (with that
 * device current) looks up the array's device address; make that first call
 * before any stream capture.  Nothing in this call allocates. */
JEPA_API jepa_status jepa_patch_embed_static(const void* clip, const void* weight, const float* bias, float* x_out,
                                             int* status, int batch, int n_frames, int height, int width,
                                             int embed_dim, int dtype, void* stream);

/* Message of the calling thread's last non-OK status ("" if none). */
JEPA_API const char* jepa_last_error(void);
/* JEPA_ABI_VERSION of the built library; a binding checks it before use. */
JEPA_API int jepa_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* JEPA_GB300_H */
