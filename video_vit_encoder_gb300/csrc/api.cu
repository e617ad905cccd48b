// The C ABI: weight blob parsing, encoder / predictor handles and the launch
// sequence of the forward pass on the caller's stream.
//
// Forward pass ("V-JEPA 2 / 2.1 tensor maps and RoPE derivation", §2 block
// form, §3 2.1 encoder forward):
//   x = unfold(normalise(clip)) W_pe^T + b_pe (+ mod_embed)        fp32 residual
//   per block: y = LN1(x); q,k,v^T = RoPE(y W_qkv^T + b_qkv)       fused epilogue
//              o = softmax(q k^T / sqrt(hd)) v;  x += o W_o^T + b_o
//              y = LN2(x); g = gelu(y W_up^T + b_up); x += g W_dn^T + b_dn
//              [hierarchical tap k: out_hier[k] = LN_k(x)]
//   out = LN(x); pooled = mean over tokens of out.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <string>
#include <vector>

#include "internal.h"
#include "jepa_gb300.h"

using namespace jepa;

namespace {

thread_local std::string g_last_error;

jepa_status fail(jepa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define CUDA_TRY(expr)                                                                        \
  do {                                                                                        \
    cudaError_t e_ = (expr);                                                                  \
    if (e_ != cudaSuccess) return fail(JEPA_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

#define JEPA_TRY(expr)              \
  do {                              \
    jepa_status s_ = (expr);        \
    if (s_ != JEPA_OK) return s_;   \
  } while (0)

size_t dtype_size(int dt) { return dt == DTYPE_F32 ? 4 : 2; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ----------------------------------------------------------------------------- blob
struct BlobEntry {
  uint64_t offset, nbytes;
  uint32_t dtype, ndim, dim0, dim1;
};
struct Expect {
  int dtype;
  uint32_t d0, d1;  // d1 = 1 for vectors
  int ndim;
};

jepa_status parse_blob(const void* blob, size_t bytes, const std::vector<Expect>& exp,
                       std::vector<BlobEntry>& entries) {
  if (blob == nullptr) return fail(JEPA_ERR_ARG, "blob is NULL");
  const uint8_t* b = static_cast<const uint8_t*>(blob);
  if (bytes < 24) return fail(JEPA_ERR_BLOB, "blob truncated: %zu bytes, header needs 24", bytes);
  if (memcmp(b, "JEPAGB3\0", 8) != 0) return fail(JEPA_ERR_BLOB, "bad blob magic");
  uint32_t version, n;
  memcpy(&version, b + 8, 4);
  memcpy(&n, b + 12, 4);
  if (version != 1) return fail(JEPA_ERR_BLOB, "unsupported blob version %u", version);
  if (n != exp.size()) return fail(JEPA_ERR_BLOB, "blob holds %u tensors, parameters need %zu", n, exp.size());
  const size_t table_end = 24 + (size_t)n * 32;
  if (bytes < table_end) return fail(JEPA_ERR_BLOB, "blob truncated inside the tensor table");
  entries.resize(n);
  for (uint32_t i = 0; i < n; ++i) {
    BlobEntry& e = entries[i];
    const uint8_t* p = b + 24 + (size_t)i * 32;
    memcpy(&e.offset, p, 8);
    memcpy(&e.nbytes, p + 8, 8);
    memcpy(&e.dtype, p + 16, 4);
    memcpy(&e.ndim, p + 20, 4);
    memcpy(&e.dim0, p + 24, 4);
    memcpy(&e.dim1, p + 28, 4);
    const Expect& x = exp[i];
    if ((int)e.dtype != x.dtype || (int)e.ndim != x.ndim || e.dim0 != x.d0 || e.dim1 != x.d1)
      return fail(JEPA_ERR_BLOB, "tensor %u: got dtype %u ndim %u [%u,%u], expected dtype %d ndim %d [%u,%u]", i,
                  e.dtype, e.ndim, e.dim0, e.dim1, x.dtype, x.ndim, x.d0, x.d1);
    const uint64_t need = (uint64_t)x.d0 * x.d1 * dtype_size(x.dtype);
    if (e.nbytes != need) return fail(JEPA_ERR_BLOB, "tensor %u: %llu bytes, expected %llu", i,
                                      (unsigned long long)e.nbytes, (unsigned long long)need);
    if (e.offset % 256 != 0 || e.offset < table_end)
      return fail(JEPA_ERR_BLOB, "tensor %u: bad offset %llu", i, (unsigned long long)e.offset);
    if (e.offset + e.nbytes > bytes)
      return fail(JEPA_ERR_BLOB, "blob truncated: tensor %u ends at %llu, blob has %zu bytes", i,
                  (unsigned long long)(e.offset + e.nbytes), bytes);
  }
  return JEPA_OK;
}

void push_block(std::vector<Expect>& v, int mat, uint32_t D, uint32_t F) {
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({mat, 3 * D, D, 2});
  v.push_back({DTYPE_F32, 3 * D, 1, 1});
  v.push_back({mat, D, D, 2});
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({mat, F, D, 2});
  v.push_back({DTYPE_F32, F, 1, 1});
  v.push_back({mat, D, F, 2});
  v.push_back({DTYPE_F32, D, 1, 1});
}

std::vector<Expect> expected_encoder(const jepa_encoder_params& p) {
  std::vector<Expect> v;
  const uint32_t D = p.embed_dim, F = p.ffn_dim, kdim = 3u * p.tubelet * p.patch * p.patch;
  v.push_back({p.dtype, D, kdim, 2});
  v.push_back({DTYPE_F32, D, 1, 1});
  if (p.has_mod_embed) v.push_back({DTYPE_F32, D, 1, 1});
  for (int i = 0; i < p.n_layer; ++i) push_block(v, p.dtype, D, F);
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({DTYPE_F32, D, 1, 1});
  for (int k = 0; k < p.n_hier; ++k) {
    v.push_back({DTYPE_F32, D, 1, 1});
    v.push_back({DTYPE_F32, D, 1, 1});
  }
  if (p.has_image_path) {  // 2.1 native image path: tubelet-1 patch embedding (+ image modality vector)
    v.push_back({p.dtype, D, 3u * p.patch * p.patch, 2});
    v.push_back({DTYPE_F32, D, 1, 1});
    if (p.has_mod_embed) v.push_back({DTYPE_F32, D, 1, 1});
  }
  return v;
}

std::vector<Expect> expected_predictor(const jepa_predictor_params& p) {
  std::vector<Expect> v;
  const uint32_t D = p.embed_dim, F = p.ffn_dim;
  v.push_back({p.dtype, D, (uint32_t)p.in_dim, 2});
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({DTYPE_F32, (uint32_t)p.n_mask_tokens, D, 2});
  for (int i = 0; i < p.n_layer; ++i) push_block(v, p.dtype, D, F);
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({p.dtype, (uint32_t)p.out_dim, D, 2});
  v.push_back({DTYPE_F32, (uint32_t)p.out_dim, 1, 1});
  if (p.has_mod_embed) {  // 2.1: pred.mod_embed_video, pred.mod_embed_img
    v.push_back({DTYPE_F32, D, 1, 1});
    v.push_back({DTYPE_F32, D, 1, 1});
  }
  if (p.has_proj_context) {  // 2.1: pred.proj_context
    v.push_back({p.dtype, (uint32_t)p.out_dim, D, 2});
    v.push_back({DTYPE_F32, (uint32_t)p.out_dim, 1, 1});
  }
  return v;
}

jepa_status check_width(int D, int H, int F, int dtype, const char* who) {
  if (D <= 0 || H <= 0 || F <= 0) return fail(JEPA_ERR_ARG, "%s: dimensions must be positive", who);
  if (D % H != 0) return fail(JEPA_ERR_ARG, "%s: embed_dim %d not divisible by n_head %d", who, D, H);
  const int hd = D / H;
  if (hd != 32 && hd != 64) return fail(JEPA_ERR_UNSUPPORTED, "%s: head_dim %d (supported: 32, 64)", who, hd);
  if (D % 128 != 0 || D > 4096) return fail(JEPA_ERR_UNSUPPORTED, "%s: embed_dim %d must be a multiple of 128, <= 4096", who, D);
  if (dtype < 0 || dtype > 2) return fail(JEPA_ERR_ARG, "%s: bad dtype %d", who, dtype);
  // the tensor-core GEMMs take whole 128-column output tiles
  if (F % (dtype == DTYPE_F32 ? 64 : 128) != 0)
    return fail(JEPA_ERR_UNSUPPORTED, "%s: ffn_dim %d must be a multiple of %d", who, F, dtype == DTYPE_F32 ? 64 : 128);
  return JEPA_OK;
}

jepa_status check_encoder_params(const jepa_encoder_params* p) {
  if (p == nullptr) return fail(JEPA_ERR_ARG, "params is NULL");
  JEPA_TRY(check_width(p->embed_dim, p->n_head, p->ffn_dim, p->dtype, "encoder"));
  if (p->patch != 16 || p->tubelet != 2)
    return fail(JEPA_ERR_UNSUPPORTED, "patch %d / tubelet %d (supported: 16 / 2)", p->patch, p->tubelet);
  if (p->n_layer < 0) return fail(JEPA_ERR_ARG, "n_layer %d", p->n_layer);
  if (p->rope_layout != 0 && p->rope_layout != 1) return fail(JEPA_ERR_ARG, "rope_layout %d", p->rope_layout);
  if (p->rope_interpolate && p->rope_ref_grid < 2) return fail(JEPA_ERR_ARG, "rope_ref_grid %d", p->rope_ref_grid);
  if (!(p->ln_eps > 0.f) || !(p->rope_theta > 0.f)) return fail(JEPA_ERR_ARG, "ln_eps and rope_theta must be > 0");
  if (p->n_hier < 0 || p->n_hier > 4) return fail(JEPA_ERR_ARG, "n_hier %d (0..4)", p->n_hier);
  for (int k = 0; k < p->n_hier; ++k) {
    if (p->hier_layers[k] < 0 || p->hier_layers[k] >= p->n_layer || (k > 0 && p->hier_layers[k] <= p->hier_layers[k - 1]))
      return fail(JEPA_ERR_ARG, "hier_layers must be increasing block indices < n_layer");
  }
  return JEPA_OK;
}

jepa_status check_predictor_params(const jepa_predictor_params* p) {
  if (p == nullptr) return fail(JEPA_ERR_ARG, "params is NULL");
  JEPA_TRY(check_width(p->embed_dim, p->n_head, p->ffn_dim, p->dtype, "predictor"));
  if (p->in_dim <= 0 || p->in_dim % 64 != 0) return fail(JEPA_ERR_UNSUPPORTED, "in_dim %d must be a multiple of 64", p->in_dim);
  if (p->out_dim <= 0 || p->out_dim % (p->dtype == DTYPE_F32 ? 32 : 128) != 0)
    return fail(JEPA_ERR_UNSUPPORTED, "out_dim %d must be a multiple of %d", p->out_dim, p->dtype == DTYPE_F32 ? 32 : 128);
  if (p->n_mask_tokens <= 0 || p->mask_index < 0) return fail(JEPA_ERR_ARG, "mask tokens");
  if (p->rope_layout != 0 && p->rope_layout != 1) return fail(JEPA_ERR_ARG, "rope_layout %d", p->rope_layout);
  if (p->n_layer < 0) return fail(JEPA_ERR_ARG, "n_layer %d", p->n_layer);
  return JEPA_OK;
}

// ----------------------------------------------------------------------------- shared device state
struct Block {
  const void *w_qkv, *w_out, *w_up, *w_down;
  const float *ln1_w, *ln1_b, *b_qkv, *b_out, *ln2_w, *ln2_b, *b_up, *b_down;
};

struct RopeCache {
  float* d = nullptr;
  size_t cap = 0;
  int key[7] = {-1, -1, -1, -1, -1, -1, -1};
  RopeParams rp{};
};

// Replay of repeated calls: one captured CUDA graph per call signature (the
// 8 most recently used), with the workspace and table buffers it points at.
struct GraphCache {
  struct Entry {
    uint64_t key[12];
    int eager_runs = 0;
    cudaGraphExec_t exec = nullptr;
    const void* ws = nullptr;
    const void* rope = nullptr;
    uint64_t last_use = 0;
  };
  std::vector<Entry> entries;
  uint64_t calls = 0;
  bool on = true;
  cudaStream_t cap = nullptr;  // capture stream, private to the owning handle
  void release() {
    for (auto& e : entries)
      if (e.exec) cudaGraphExecDestroy(e.exec);
    entries.clear();
    if (cap) cudaStreamDestroy(cap);
    cap = nullptr;
  }
};

// Builds the per-axis cos/sin tables for a grid ("V-JEPA 2 / 2.1 ...", §4:
// omega_k = theta^(-k/(d/2)); §4.3: interpolated spatial positions
// p*(ref-1)/(n-1), evaluated left to right) in double and uploads them.
jepa_status rope_prepare(RopeCache& rc, int head_dim, int layout, float theta, int gt, int gh, int gw, int interp,
                         int ref, cudaStream_t s) {
  const int key[7] = {head_dim, layout, (int)(theta * 16), gt, gh, gw, interp ? ref : 0};
  if (memcmp(key, rc.key, sizeof(key)) == 0 && rc.d != nullptr) return JEPA_OK;
  const int d = 2 * ((head_dim / 3) / 2), half = d / 2;
  const int max_pos = std::max(gt, std::max(gh, gw));
  const size_t n = (size_t)3 * max_pos * half;
  std::vector<float> host(2 * n);
  const int extent[3] = {gt, gh, gw};
  for (int a = 0; a < 3; ++a) {
    for (int p = 0; p < max_pos; ++p) {
      double pos = p;
      if (interp && a > 0 && extent[a] > 1) pos = (double)p * (double)(ref - 1) / (double)(extent[a] - 1);
      for (int k = 0; k < half; ++k) {
        const double omega = 1.0 / pow((double)theta, (double)k / (double)half);
        host[(a * max_pos + p) * half + k] = (float)cos(pos * omega);
        host[n + (a * max_pos + p) * half + k] = (float)sin(pos * omega);
      }
    }
  }
  if (rc.cap < 2 * n) {
    if (rc.d) cudaFree(rc.d);
    rc.d = nullptr;
    if (cudaMalloc(&rc.d, 2 * n * sizeof(float)) != cudaSuccess) return fail(JEPA_ERR_OOM, "RoPE table allocation");
    rc.cap = 2 * n;
  }
  CUDA_TRY(cudaMemcpyAsync(rc.d, host.data(), 2 * n * sizeof(float), cudaMemcpyHostToDevice, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  memcpy(rc.key, key, sizeof(key));
  rc.rp.cos_tab = rc.d;
  rc.rp.sin_tab = rc.d + n;
  rc.rp.max_pos = max_pos;
  rc.rp.d = d;
  rc.rp.layout = layout;
  rc.rp.gt = gt;
  rc.rp.gh = gh;
  rc.rp.gw = gw;
  return JEPA_OK;
}

// Event-based per-class timing of launches.
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  std::vector<std::pair<int, size_t>> marks;  // (class, index of start event)
  double times[8] = {};
  long long launches[8] = {};

  cudaEvent_t next() {
    if (used == pool.size()) {
      cudaEvent_t e;
      cudaEventCreate(&e);
      pool.push_back(e);
    }
    return pool[used++];
  }
  void begin(int cls, cudaStream_t s) {
    if (!on) return;
    const size_t idx = used;
    cudaEventRecord(next(), s);
    marks.push_back({cls, idx});
  }
  void end(cudaStream_t s) {
    if (!on) return;
    cudaEventRecord(next(), s);
  }
  void collect() {
    for (auto& m : marks) {
      float ms = 0.f;
      cudaEventSynchronize(pool[m.second + 1]);
      cudaEventElapsedTime(&ms, pool[m.second], pool[m.second + 1]);
      times[m.first] += ms;
      launches[m.first] += 1;
    }
    marks.clear();
    used = 0;
  }
  ~Profiler() {
    for (auto e : pool) cudaEventDestroy(e);
  }
};

enum { P_EMBED = 0, P_LN = 1, P_QKV = 2, P_ATTN = 3, P_OUT = 4, P_UP = 5, P_DOWN = 6, P_OTHER = 7 };

struct Scope {
  Profiler& p;
  cudaStream_t s;
  Scope(Profiler& pr, int cls, cudaStream_t st) : p(pr), s(st) { p.begin(cls, s); }
  ~Scope() { p.end(s); }
};

jepa_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return JEPA_OK;
  return fail(JEPA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

jepa_status run_linear(int dtype, int epi, const void* A, const void* W, int M, int N, int K, const EpiParams& ep,
                       int* status, cudaStream_t s, int sms) {
  if (M == 0) return JEPA_OK;
  if (dtype == DTYPE_F32)
    return cuda_status(gemm_simt_f32(epi, (const float*)A, (const float*)W, M, N, K, ep, s), "fp32 linear");
  return cuda_status(gemm_tc(dtype, epi, A, W, M, N, K, ep, status, s, sms), "tensor-core linear");
}

jepa_status run_attention(int dtype, const void* q, const void* k, const void* vt, void* out, int batch, int heads,
                          int n, int hd, int ldv, int* status, cudaStream_t s, int sms) {
  const float scale = 1.0f / sqrtf((float)hd);
  if (dtype == DTYPE_F32)
    return cuda_status(attention_simt(dtype, q, k, vt, out, batch, heads, n, hd, ldv, scale, s), "fp32 attention");
  return cuda_status(attention_tc(dtype, q, k, vt, out, batch, heads, n, hd, ldv, scale, status, s, sms),
                     "tensor-core attention");
}

// Workspace of one transformer stack over M rows.
struct Work {
  float* x = nullptr;  // fp32 residual [M, D]
  void* y = nullptr;   // T [M, D]
  void* q = nullptr;   // T [M, D]
  void* k = nullptr;   // T [M, D]
  void* vt = nullptr;  // T [B*h, hd, ldv]
  void* o = nullptr;   // T [M, D]
  void* g = nullptr;   // T [M, F]  (also the unfolded clip [M, 1536])
  int* pos = nullptr;  // predictor positions [M]
  int ldv = 0;
};

size_t work_bytes(int dtype, int clips, int n_tok, int D, int F, int extra_cols, bool with_pos) {
  const size_t M = (size_t)clips * n_tok, e = dtype_size(dtype);
  const size_t ldv = (size_t)((n_tok + 7) / 8) * 8;
  size_t b = align256(M * D * 4) + 4 * align256(M * D * e) + align256((size_t)clips * D * ldv * e) +
             align256(M * std::max(F, extra_cols) * e);
  if (with_pos) b += align256(M * 4);
  return b;
}

Work carve(void* base, int dtype, int clips, int n_tok, int D, int F, int extra_cols, bool with_pos) {
  Work w;
  const size_t M = (size_t)clips * n_tok, e = dtype_size(dtype);
  w.ldv = ((n_tok + 7) / 8) * 8;
  uint8_t* p = static_cast<uint8_t*>(base);
  w.x = reinterpret_cast<float*>(p);  p += align256(M * D * 4);
  w.y = p;                            p += align256(M * D * e);
  w.q = p;                            p += align256(M * D * e);
  w.k = p;                            p += align256(M * D * e);
  w.o = p;                            p += align256(M * D * e);
  w.vt = p;                           p += align256((size_t)clips * D * w.ldv * e);
  w.g = p;                            p += align256(M * std::max(F, extra_cols) * e);
  if (with_pos) w.pos = reinterpret_cast<int*>(p);
  return w;
}

// Runs blocks [l0, l1) of a stack in place on w.x ([clips * n_tok, D] rows).
struct StackDesc {
  int D, H, F, dtype;
  float eps;
  const std::vector<Block>* blocks;
  int n_hier;
  const int* hier_layers;
  const float* const* hier_w;
  const float* const* hier_b;
};

jepa_status run_blocks(const StackDesc& sd, Work& w, int clips, int n_tok, int l0, int l1, const RopeParams& rp,
                       const int* pos_ids, float* out_hier, int* status, Profiler& prof, cudaStream_t s, int sms) {
  const int D = sd.D, F = sd.F, H = sd.H, hd = D / H, dt = sd.dtype;
  const int M = clips * n_tok;
  for (int l = l0; l < l1; ++l) {
    const Block& B = (*sd.blocks)[l];
    {
      Scope sc(prof, P_LN, s);
      JEPA_TRY(cuda_status(layernorm(dt, w.x, B.ln1_w, B.ln1_b, w.y, M, D, sd.eps, s), "layernorm"));
    }
    {
      Scope sc(prof, P_QKV, s);
      EpiParams ep{};
      ep.bias = B.b_qkv;
      ep.q = w.q;
      ep.k = w.k;
      ep.vt = w.vt;
      ep.n_tok = n_tok;
      ep.n_head = H;
      ep.head_dim = hd;
      ep.ldv = w.ldv;
      ep.dmodel = D;
      ep.pos_ids = pos_ids;
      ep.rope = rp;
      JEPA_TRY(run_linear(dt, EPI_QKV, w.y, B.w_qkv, M, 3 * D, D, ep, status, s, sms));
    }
    {
      Scope sc(prof, P_ATTN, s);
      JEPA_TRY(run_attention(dt, w.q, w.k, w.vt, w.o, clips, H, n_tok, hd, w.ldv, status, s, sms));
    }
    {
      Scope sc(prof, P_OUT, s);
      EpiParams ep{};
      ep.bias = B.b_out;
      ep.out = w.x;
      ep.ldo = D;
      JEPA_TRY(run_linear(dt, EPI_RESID, w.o, B.w_out, M, D, D, ep, status, s, sms));
    }
    {
      Scope sc(prof, P_LN, s);
      JEPA_TRY(cuda_status(layernorm(dt, w.x, B.ln2_w, B.ln2_b, w.y, M, D, sd.eps, s), "layernorm"));
    }
    {
      Scope sc(prof, P_UP, s);
      EpiParams ep{};
      ep.bias = B.b_up;
      ep.out = w.g;
      ep.ldo = F;
      JEPA_TRY(run_linear(dt, EPI_GELU, w.y, B.w_up, M, F, D, ep, status, s, sms));
    }
    {
      Scope sc(prof, P_DOWN, s);
      EpiParams ep{};
      ep.bias = B.b_down;
      ep.out = w.x;
      ep.ldo = D;
      JEPA_TRY(run_linear(dt, EPI_RESID, w.g, B.w_down, M, D, F, ep, status, s, sms));
    }
    if (out_hier != nullptr) {
      for (int kk = 0; kk < sd.n_hier; ++kk) {
        if (sd.hier_layers[kk] == l) {
          Scope sc(prof, P_LN, s);
          JEPA_TRY(cuda_status(layernorm(DTYPE_F32, w.x, sd.hier_w[kk], sd.hier_b[kk],
                                         out_hier + (size_t)kk * M * D, M, D, sd.eps, s),
                               "layernorm"));
        }
      }
    }
  }
  return JEPA_OK;
}

// Copies the blob's tensors to one device allocation; returns device
// pointers in blob order.
jepa_status upload_weights(const void* blob, const std::vector<BlobEntry>& ent, void** d_base,
                           std::vector<const void*>& ptrs) {
  size_t total = 0;
  for (auto& e : ent) total += align256(e.nbytes);
  void* base = nullptr;
  if (cudaMalloc(&base, total) != cudaSuccess) return fail(JEPA_ERR_OOM, "weights: cudaMalloc(%zu) failed", total);
  size_t off = 0;
  ptrs.clear();
  for (auto& e : ent) {
    void* dst = static_cast<uint8_t*>(base) + off;
    if (cudaMemcpy(dst, static_cast<const uint8_t*>(blob) + e.offset, e.nbytes, cudaMemcpyHostToDevice) !=
        cudaSuccess) {
      cudaFree(base);
      return fail(JEPA_ERR_CUDA, "weights: copy to device failed");
    }
    ptrs.push_back(dst);
    off += align256(e.nbytes);
  }
  *d_base = base;
  return JEPA_OK;
}

Block take_block(const std::vector<const void*>& P, size_t& i) {
  Block b;
  b.ln1_w = (const float*)P[i++];
  b.ln1_b = (const float*)P[i++];
  b.w_qkv = P[i++];
  b.b_qkv = (const float*)P[i++];
  b.w_out = P[i++];
  b.b_out = (const float*)P[i++];
  b.ln2_w = (const float*)P[i++];
  b.ln2_b = (const float*)P[i++];
  b.w_up = P[i++];
  b.b_up = (const float*)P[i++];
  b.w_down = P[i++];
  b.b_down = (const float*)P[i++];
  return b;
}

__global__ void add_vec_kernel(float* a, const float* b, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) a[i] += b[i];
}

// Device status word of the single operations, one per device (allocated on
// the first single-operation call made with that device current).
DeviceOnce g_ops_once;
int* g_ops_status[kMaxDevices] = {};
jepa_status ops_status(int** out) {
  int dev = 0;
  const cudaError_t e = g_ops_once.run([](int d) -> cudaError_t {
    int* p = nullptr;
    cudaError_t r = cudaMalloc(&p, sizeof(int));
    if (r != cudaSuccess) return r;
    r = cudaMemset(p, 0, sizeof(int));
    if (r != cudaSuccess) {
      cudaFree(p);
      return r;
    }
    g_ops_status[d] = p;
    return cudaSuccess;
  }, &dev);
  if (e != cudaSuccess) return fail(JEPA_ERR_CUDA, "single-operation status word: %s", cudaGetErrorString(e));
  *out = g_ops_status[dev];
  return JEPA_OK;
}

// RoPE tables of the single operations, per calling thread and device.
RopeCache& ops_rope_cache() {
  static thread_local RopeCache rc[kMaxDevices];
  int dev = 0;
  cudaGetDevice(&dev);
  return rc[dev >= 0 && dev < kMaxDevices ? dev : 0];
}

jepa_status read_status(int* d_status, cudaStream_t s) {
  int h = 0;
  CUDA_TRY(cudaStreamSynchronize(s));
  CUDA_TRY(cudaMemcpy(&h, d_status, sizeof(int), cudaMemcpyDeviceToHost));
  if (h != 0) {
    CUDA_TRY(cudaMemset(d_status, 0, sizeof(int)));
    if (h & DEV_TIMEOUT) return fail(JEPA_ERR_DEVICE_TIMEOUT, "a kernel gave up waiting on a barrier (status 0x%x)", h);
    return fail(JEPA_ERR_ARG, "token ids outside the grid (clamped; results invalid) (status 0x%x)", h);
  }
  return JEPA_OK;
}

}  // namespace

namespace jepa {
// Lets other translation units set the message returned by jepa_last_error().
void record_error(const char* msg) { g_last_error = msg; }
}  // namespace jepa

// ============================================================================= encoder
// Staging of jepa_encode_host_async: two slots used in turn, each with its
// device clip / output buffers and the events that order its reuse; the
// copies run on two streams of their own.
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  struct Slot {
    void* clip = nullptr;
    size_t clip_cap = 0;
    void* out = nullptr;
    size_t out_cap = 0;
    void* pool = nullptr;
    size_t pool_cap = 0;
    cudaEvent_t copied_in = nullptr, encoded = nullptr, copied_out = nullptr;
  } slot[2];
  uint64_t calls = 0;
  void release() {
    for (auto& sl : slot) {
      cudaFree(sl.clip);
      cudaFree(sl.out);
      cudaFree(sl.pool);
      if (sl.copied_in) cudaEventDestroy(sl.copied_in);
      if (sl.encoded) cudaEventDestroy(sl.encoded);
      if (sl.copied_out) cudaEventDestroy(sl.copied_out);
      sl = Slot{};
    }
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
    in = out = nullptr;
  }
};

struct jepa_encoder {
  jepa_encoder_params p{};
  int device = 0, sms = 0;
  void* d_weights = nullptr;
  const void* w_pe = nullptr;
  float* b_pe = nullptr;  // patch-embed bias (+ modality vector)
  const void* w_pe_img = nullptr;  // image path (tubelet 1), when present
  float* b_pe_img = nullptr;       // its bias (+ image modality vector)
  std::vector<Block> blocks;
  const float *norm_w = nullptr, *norm_b = nullptr;
  const float* hier_w[4] = {};
  const float* hier_b[4] = {};
  void* ws = nullptr;
  size_t ws_bytes = 0;
  int* d_status = nullptr;
  RopeCache rope;
  Profiler prof;
  void* h_clip_dev = nullptr;
  size_t h_clip_cap = 0;
  float* h_out_dev = nullptr;
  size_t h_out_cap = 0;
  float* h_pool_dev = nullptr;
  size_t h_pool_cap = 0;
  HostPipe pipe;
  GraphCache graphs;
};

namespace {

struct Geom {
  int gt, gh, gw, n_tok;
  int tub;  // tubelet of this input: 2 for clips, 1 on the image path
};

jepa_status check_clip(const jepa_encoder* enc, int batch, int T, int H, int W, Geom& g) {
  if (enc == nullptr) return fail(JEPA_ERR_ARG, "encoder handle is NULL");
  if (batch < 1) return fail(JEPA_ERR_ARG, "batch %d must be >= 1", batch);
  // One frame takes the 2.1 native image path where the model has it (the
  // conversion notes, 2.1 encoder forward: selected by the frame count).
  g.tub = (T == 1 && enc->p.has_image_path) ? 1 : 2;
  if (g.tub == 2 && (T < 2 || T % 2 != 0))
    return fail(JEPA_ERR_ARG, "n_frames %d must be even and >= 2%s", T,
                enc->p.has_image_path ? ", or 1 for an image" : "");
  if (H < 16 || W < 16 || H % 16 != 0 || W % 16 != 0)
    return fail(JEPA_ERR_ARG, "height %d and width %d must be positive multiples of 16", H, W);
  g.gt = T / g.tub;
  g.gh = H / 16;
  g.gw = W / 16;
  if (enc->p.rope_interpolate && (g.gh < 2 || g.gw < 2))
    return fail(JEPA_ERR_ARG, "RoPE interpolation needs at least 2 patches per side (got %dx%d)", g.gh, g.gw);
  const long long n = (long long)g.gt * g.gh * g.gw;
  const long long M = n * batch;
  const long long widest = std::max<long long>(std::max(enc->p.ffn_dim, 3 * enc->p.embed_dim), 1536);
  if (M * widest >= (1ll << 31)) return fail(JEPA_ERR_ARG, "clip too large: %lld rows", M);
  g.n_tok = (int)n;
  return JEPA_OK;
}

jepa_status ensure_ws(jepa_encoder* enc, int batch, const Geom& g) {
  const size_t need = work_bytes(enc->p.dtype, batch, g.n_tok, enc->p.embed_dim, enc->p.ffn_dim, 1536, false);
  if (need <= enc->ws_bytes) return JEPA_OK;
  if (enc->ws) cudaFree(enc->ws);
  enc->ws = nullptr;
  enc->ws_bytes = 0;
  if (cudaMalloc(&enc->ws, need) != cudaSuccess) return fail(JEPA_ERR_OOM, "workspace: cudaMalloc(%zu) failed", need);
  // V^T padding columns must hold finite values (they meet zero weights).
  if (cudaMemset(enc->ws, 0, need) != cudaSuccess) return fail(JEPA_ERR_CUDA, "workspace memset");
  enc->ws_bytes = need;
  return JEPA_OK;
}

StackDesc enc_stack(const jepa_encoder* enc) {
  StackDesc sd;
  sd.D = enc->p.embed_dim;
  sd.H = enc->p.n_head;
  sd.F = enc->p.ffn_dim;
  sd.dtype = enc->p.dtype;
  sd.eps = enc->p.ln_eps;
  sd.blocks = &enc->blocks;
  sd.n_hier = enc->p.n_hier;
  sd.hier_layers = enc->p.hier_layers;
  sd.hier_w = enc->hier_w;
  sd.hier_b = enc->hier_b;
  return sd;
}

// Patch embedding of every token, or (keep != nullptr) of the n_keep tokens
// keep[b * n_keep + r] of each clip b, in that order (the masked encoder).
jepa_status embed_into(jepa_encoder* enc, Work& w, const void* clip, int fmt, int batch, int T, int H, int W,
                       const Geom& g, float* x_out, cudaStream_t s, const int* keep = nullptr, int n_keep = 0) {
  const int D = enc->p.embed_dim, dt = enc->p.dtype;
  const int M = batch * (keep != nullptr ? n_keep : g.n_tok);
  Scope sc(enc->prof, P_EMBED, s);
  if (fmt == JEPA_CLIP_U8_THWC)
    JEPA_TRY(cuda_status(unfold_clip_u8(dt, (const uint8_t*)clip, w.g, batch, T, H, W, g.tub, s, keep, n_keep),
                         "unfold"));
  else
    JEPA_TRY(cuda_status(unfold_clip_f32(dt, (const float*)clip, w.g, batch, T, H, W, g.tub, s, keep, n_keep),
                         "unfold"));
  const bool img = g.tub == 1;
  EpiParams ep{};
  ep.bias = img ? enc->b_pe_img : enc->b_pe;
  ep.out = x_out;
  ep.ldo = D;
  return run_linear(dt, EPI_F32, w.g, img ? enc->w_pe_img : enc->w_pe, M, D, 768 * g.tub, ep, enc->d_status, s,
                    enc->sms);
}

}  // namespace

extern "C" {

const char* jepa_last_error(void) { return g_last_error.c_str(); }
int jepa_abi_version(void) { return JEPA_ABI_VERSION; }

jepa_status jepa_blob_check(const void* blob, size_t blob_bytes, const jepa_encoder_params* params) {
  JEPA_TRY(check_encoder_params(params));
  std::vector<BlobEntry> ent;
  return parse_blob(blob, blob_bytes, expected_encoder(*params), ent);
}

jepa_status jepa_predictor_blob_check(const void* blob, size_t blob_bytes, const jepa_predictor_params* params) {
  JEPA_TRY(check_predictor_params(params));
  std::vector<BlobEntry> ent;
  return parse_blob(blob, blob_bytes, expected_predictor(*params), ent);
}

jepa_status jepa_encoder_create(const void* blob, size_t blob_bytes, const jepa_encoder_params* params, int device,
                                jepa_encoder** out) {
  if (out == nullptr) return fail(JEPA_ERR_ARG, "out is NULL");
  *out = nullptr;
  JEPA_TRY(check_encoder_params(params));
  std::vector<BlobEntry> ent;
  JEPA_TRY(parse_blob(blob, blob_bytes, expected_encoder(*params), ent));
  CUDA_TRY(cudaSetDevice(device));
  jepa_encoder* enc = new jepa_encoder();
  enc->p = *params;
  enc->device = device;
  cudaDeviceGetAttribute(&enc->sms, cudaDevAttrMultiProcessorCount, device);
  std::vector<const void*> P;
  jepa_status st = upload_weights(blob, ent, &enc->d_weights, P);
  if (st != JEPA_OK) {
    delete enc;
    return st;
  }
  const int D = params->embed_dim;
  size_t i = 0;
  enc->w_pe = P[i++];
  const float* b_pe = (const float*)P[i++];
  const float* mod = params->has_mod_embed ? (const float*)P[i++] : nullptr;
  if (cudaMalloc(&enc->b_pe, D * sizeof(float)) != cudaSuccess || cudaMalloc(&enc->d_status, sizeof(int)) != cudaSuccess) {
    jepa_encoder_destroy(enc);
    return fail(JEPA_ERR_OOM, "encoder: small allocations failed");
  }
  cudaMemcpy(enc->b_pe, b_pe, D * sizeof(float), cudaMemcpyDeviceToDevice);
  if (mod) add_vec_kernel<<<(D + 255) / 256, 256>>>(enc->b_pe, mod, D);  // the modality vector joins the bias
  cudaMemset(enc->d_status, 0, sizeof(int));
  for (int l = 0; l < params->n_layer; ++l) enc->blocks.push_back(take_block(P, i));
  enc->norm_w = (const float*)P[i++];
  enc->norm_b = (const float*)P[i++];
  for (int k = 0; k < params->n_hier; ++k) {
    enc->hier_w[k] = (const float*)P[i++];
    enc->hier_b[k] = (const float*)P[i++];
  }
  if (params->has_image_path) {
    enc->w_pe_img = P[i++];
    const float* b_img = (const float*)P[i++];
    const float* mod_img = params->has_mod_embed ? (const float*)P[i++] : nullptr;
    if (cudaMalloc(&enc->b_pe_img, D * sizeof(float)) != cudaSuccess) {
      jepa_encoder_destroy(enc);
      return fail(JEPA_ERR_OOM, "encoder: small allocations failed");
    }
    cudaMemcpy(enc->b_pe_img, b_img, D * sizeof(float), cudaMemcpyDeviceToDevice);
    if (mod_img) add_vec_kernel<<<(D + 255) / 256, 256>>>(enc->b_pe_img, mod_img, D);
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    jepa_encoder_destroy(enc);
    return fail(JEPA_ERR_CUDA, "encoder create: %s", cudaGetErrorString(e));
  }
  *out = enc;
  return JEPA_OK;
}

void jepa_encoder_destroy(jepa_encoder* enc) {
  if (enc == nullptr) return;
  cudaSetDevice(enc->device);
  cudaDeviceSynchronize();
  cudaFree(enc->d_weights);
  cudaFree(enc->b_pe);
  cudaFree(enc->b_pe_img);
  cudaFree(enc->ws);
  cudaFree(enc->d_status);
  cudaFree(enc->rope.d);
  cudaFree(enc->h_clip_dev);
  cudaFree(enc->h_out_dev);
  cudaFree(enc->h_pool_dev);
  enc->pipe.release();
  enc->graphs.release();
  delete enc;
}

size_t jepa_encode_workspace_bytes(const jepa_encoder* enc, int batch, int n_frames, int height, int width) {
  Geom g;
  if (check_clip(enc, batch, n_frames, height, width, g) != JEPA_OK) return 0;
  return work_bytes(enc->p.dtype, batch, g.n_tok, enc->p.embed_dim, enc->p.ffn_dim, 1536, false);
}

jepa_status jepa_encoder_embed(jepa_encoder* enc, const void* clip, int clip_format, int batch, int n_frames,
                               int height, int width, float* x_out, void* stream) {
  Geom g;
  JEPA_TRY(check_clip(enc, batch, n_frames, height, width, g));
  if (clip == nullptr || x_out == nullptr) return fail(JEPA_ERR_ARG, "clip and x_out must be device buffers");
  if (!aligned16(clip) || !aligned16(x_out)) return fail(JEPA_ERR_ARG, "device buffers must be 16-byte aligned");
  if (clip_format != JEPA_CLIP_U8_THWC && clip_format != JEPA_CLIP_F32_CTHW)
    return fail(JEPA_ERR_ARG, "clip_format %d", clip_format);
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_TRY(cudaSetDevice(enc->device));
  JEPA_TRY(ensure_ws(enc, batch, g));
  Work w = carve(enc->ws, enc->p.dtype, batch, g.n_tok, enc->p.embed_dim, enc->p.ffn_dim, 1536, false);
  return embed_into(enc, w, clip, clip_format, batch, n_frames, height, width, g, x_out, s);
}

jepa_status jepa_encoder_blocks(jepa_encoder* enc, float* x, int batch, int n_frames, int height, int width,
                                int layer_begin, int layer_end, void* stream) {
  Geom g;
  JEPA_TRY(check_clip(enc, batch, n_frames, height, width, g));
  if (x == nullptr || !aligned16(x)) return fail(JEPA_ERR_ARG, "x must be a 16-byte aligned device buffer");
  if (layer_begin < 0 || layer_end > enc->p.n_layer || layer_begin > layer_end)
    return fail(JEPA_ERR_ARG, "layer range [%d, %d) outside [0, %d)", layer_begin, layer_end, enc->p.n_layer);
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_TRY(cudaSetDevice(enc->device));
  JEPA_TRY(ensure_ws(enc, batch, g));
  const int hd = enc->p.embed_dim / enc->p.n_head;
  JEPA_TRY(rope_prepare(enc->rope, hd, enc->p.rope_layout, enc->p.rope_theta, g.gt, g.gh, g.gw,
                        enc->p.rope_interpolate, enc->p.rope_ref_grid, s));
  Work w = carve(enc->ws, enc->p.dtype, batch, g.n_tok, enc->p.embed_dim, enc->p.ffn_dim, 1536, false);
  w.x = x;
  return run_blocks(enc_stack(enc), w, batch, g.n_tok, layer_begin, layer_end, enc->rope.rp, nullptr, nullptr,
                    enc->d_status, enc->prof, s, enc->sms);
}

}  // extern "C"

namespace {

// The device work of one jepa_encode call, enqueued on s (arguments checked).
jepa_status encode_body(jepa_encoder* enc, const void* clip, int clip_format, int batch, int n_frames, int height,
                        int width, const Geom& g, float* out_tokens, float* out_pooled, float* out_hier,
                        cudaStream_t s) {
  JEPA_TRY(ensure_ws(enc, batch, g));
  const int hd = enc->p.embed_dim / enc->p.n_head;
  JEPA_TRY(rope_prepare(enc->rope, hd, enc->p.rope_layout, enc->p.rope_theta, g.gt, g.gh, g.gw,
                        enc->p.rope_interpolate, enc->p.rope_ref_grid, s));
  Work w = carve(enc->ws, enc->p.dtype, batch, g.n_tok, enc->p.embed_dim, enc->p.ffn_dim, 1536, false);
  JEPA_TRY(embed_into(enc, w, clip, clip_format, batch, n_frames, height, width, g, w.x, s));
  JEPA_TRY(run_blocks(enc_stack(enc), w, batch, g.n_tok, 0, enc->p.n_layer, enc->rope.rp, nullptr, out_hier,
                      enc->d_status, enc->prof, s, enc->sms));
  const int M = batch * g.n_tok, D = enc->p.embed_dim;
  {
    Scope sc(enc->prof, P_LN, s);
    JEPA_TRY(cuda_status(layernorm(DTYPE_F32, w.x, enc->norm_w, enc->norm_b, out_tokens, M, D, enc->p.ln_eps, s),
                         "final layernorm"));
  }
  if (out_pooled != nullptr) {
    Scope sc(enc->prof, P_OTHER, s);
    JEPA_TRY(cuda_status(mean_pool(out_tokens, out_pooled, batch, g.n_tok, D, s), "mean pool"));
  }
  return JEPA_OK;
}

// Repeated calls with the same signature replay one CUDA graph: the first
// runs eagerly (it sizes the workspace and builds the RoPE tables), the second
// is captured on a private stream (the caller's may be the legacy default
// stream, which cannot be captured) and every later one is a single graph
// launch on the caller's stream.  A graph is dropped when the workspace or
// the table buffer it points at has been reallocated.
// `prep(stream)` readies the workspace and tables outside any capture;
// `ws` and `rope` are the owner's buffer pointers (read after prep);
// `body(stream)` enqueues the call's device work.
template <typename Prep, typename Body>
jepa_status replay(GraphCache& gc, const uint64_t (&key)[12], Prep&& prep, void* const& ws, float* const& rope,
                   Body&& body, cudaStream_t s) {
  using E = GraphCache::Entry;
  E* e = nullptr;
  for (auto& x : gc.entries)
    if (memcmp(x.key, key, sizeof(key)) == 0) e = &x;
  if (e == nullptr) {
    if (gc.entries.size() >= 8) {  // evict the least recently used signature
      auto lru = gc.entries.begin();
      for (auto it = gc.entries.begin(); it != gc.entries.end(); ++it)
        if (it->last_use < lru->last_use) lru = it;
      if (lru->exec) cudaGraphExecDestroy(lru->exec);
      gc.entries.erase(lru);
    }
    gc.entries.push_back(E{});
    e = &gc.entries.back();
    memcpy(e->key, key, sizeof(key));
  }
  e->last_use = ++gc.calls;
  JEPA_TRY(prep(s));
  if (e->exec != nullptr && (e->ws != ws || e->rope != rope)) {
    cudaGraphExecDestroy(e->exec);
    e->exec = nullptr;
  }
  if (e->exec == nullptr) {
    if (e->eager_runs++ == 0) return body(s);
    if (gc.cap == nullptr) CUDA_TRY(cudaStreamCreateWithFlags(&gc.cap, cudaStreamNonBlocking));
    CUDA_TRY(cudaStreamBeginCapture(gc.cap, cudaStreamCaptureModeThreadLocal));
    const jepa_status st = body(gc.cap);
    cudaGraph_t graph = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(gc.cap, &graph);
    if (st != JEPA_OK) {
      if (graph) cudaGraphDestroy(graph);
      return st;
    }
    if (ce != cudaSuccess) return fail(JEPA_ERR_CUDA, "graph capture: %s", cudaGetErrorString(ce));
    const cudaError_t ie = cudaGraphInstantiate(&e->exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) {
      e->exec = nullptr;
      return fail(JEPA_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(ie));
    }
    e->ws = ws;
    e->rope = rope;
  }
  CUDA_TRY(cudaGraphLaunch(e->exec, s));
  return JEPA_OK;
}

// The encoder's replay: workspace for geometry gw, RoPE tables for grid g.
template <typename Body>
jepa_status encode_replayed(jepa_encoder* enc, const uint64_t (&key)[12], int batch, const Geom& gw, const Geom& g,
                            Body&& body, cudaStream_t s) {
  auto prep = [&](cudaStream_t st) -> jepa_status {
    JEPA_TRY(ensure_ws(enc, batch, gw));
    const int hd = enc->p.embed_dim / enc->p.n_head;
    return rope_prepare(enc->rope, hd, enc->p.rope_layout, enc->p.rope_theta, g.gt, g.gh, g.gw,
                        enc->p.rope_interpolate, enc->p.rope_ref_grid, st);
  };
  return replay(enc->graphs, key, prep, enc->ws, enc->rope.d, body, s);
}

}  // namespace

extern "C" {

jepa_status jepa_encode(jepa_encoder* enc, const void* clip, int clip_format, int batch, int n_frames, int height,
                        int width, float* out_tokens, float* out_pooled, float* out_hier, void* stream) {
  Geom g;
  JEPA_TRY(check_clip(enc, batch, n_frames, height, width, g));
  if (clip == nullptr || out_tokens == nullptr) return fail(JEPA_ERR_ARG, "clip and out_tokens are required");
  if (!aligned16(clip) || !aligned16(out_tokens) || !aligned16(out_pooled) || !aligned16(out_hier))
    return fail(JEPA_ERR_ARG, "device buffers must be 16-byte aligned");
  if (clip_format != JEPA_CLIP_U8_THWC && clip_format != JEPA_CLIP_F32_CTHW)
    return fail(JEPA_ERR_ARG, "clip_format %d", clip_format);
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_TRY(cudaSetDevice(enc->device));
  if (enc->prof.on || !enc->graphs.on)  // per-class events need the launches one by one
    return encode_body(enc, clip, clip_format, batch, n_frames, height, width, g, out_tokens, out_pooled, out_hier,
                       s);
  const uint64_t key[12] = {1, (uint64_t)(uintptr_t)clip, (uint64_t)clip_format, (uint64_t)batch,
                            (uint64_t)n_frames, (uint64_t)height, (uint64_t)width, (uint64_t)(uintptr_t)out_tokens,
                            (uint64_t)(uintptr_t)out_pooled, (uint64_t)(uintptr_t)out_hier, 0, 0};
  return encode_replayed(enc, key, batch, g, g, [&](cudaStream_t st) {
    return encode_body(enc, clip, clip_format, batch, n_frames, height, width, g, out_tokens, out_pooled, out_hier, st);
  }, s);
}

jepa_status jepa_encoder_set_graphs(jepa_encoder* enc, int on) {
  if (enc == nullptr) return fail(JEPA_ERR_ARG, "encoder handle is NULL");
  enc->graphs.on = on != 0;
  return JEPA_OK;
}

jepa_status jepa_encode_masked(jepa_encoder* enc, const void* clip, int clip_format, int batch, int n_frames,
                               int height, int width, const int32_t* ids_keep, int n_keep, float* out_tokens,
                               float* out_pooled, float* out_hier, void* stream) {
  Geom g;
  JEPA_TRY(check_clip(enc, batch, n_frames, height, width, g));
  if (clip == nullptr || out_tokens == nullptr || ids_keep == nullptr)
    return fail(JEPA_ERR_ARG, "clip, ids_keep and out_tokens are required");
  if (n_keep < 1 || n_keep > g.n_tok) return fail(JEPA_ERR_ARG, "n_keep %d must be in 1..%d", n_keep, g.n_tok);
  if (!aligned16(clip) || !aligned16(out_tokens) || !aligned16(out_pooled) || !aligned16(out_hier))
    return fail(JEPA_ERR_ARG, "device buffers must be 16-byte aligned");
  if (clip_format != JEPA_CLIP_U8_THWC && clip_format != JEPA_CLIP_F32_CTHW)
    return fail(JEPA_ERR_ARG, "clip_format %d", clip_format);
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_TRY(cudaSetDevice(enc->device));
  Geom gk = g;  // the blocks see n_keep tokens per clip
  gk.n_tok = n_keep;
  auto body = [&](cudaStream_t st) -> jepa_status {
    JEPA_TRY(ensure_ws(enc, batch, gk));
    const int hd = enc->p.embed_dim / enc->p.n_head;
    // RoPE tables for the full grid: each kept token keeps its own grid cell
    JEPA_TRY(rope_prepare(enc->rope, hd, enc->p.rope_layout, enc->p.rope_theta, g.gt, g.gh, g.gw,
                          enc->p.rope_interpolate, enc->p.rope_ref_grid, st));
    Work w = carve(enc->ws, enc->p.dtype, batch, n_keep, enc->p.embed_dim, enc->p.ffn_dim, 1536, false);
    JEPA_TRY(cuda_status(check_ids(ids_keep, (long)batch * n_keep, g.n_tok, enc->d_status, st), "id check"));
    JEPA_TRY(embed_into(enc, w, clip, clip_format, batch, n_frames, height, width, g, w.x, st, ids_keep, n_keep));
    JEPA_TRY(run_blocks(enc_stack(enc), w, batch, n_keep, 0, enc->p.n_layer, enc->rope.rp, ids_keep, out_hier,
                        enc->d_status, enc->prof, st, enc->sms));
    const int M = batch * n_keep, D = enc->p.embed_dim;
    {
      Scope sc(enc->prof, P_LN, st);
      JEPA_TRY(cuda_status(layernorm(DTYPE_F32, w.x, enc->norm_w, enc->norm_b, out_tokens, M, D, enc->p.ln_eps, st),
                           "final layernorm"));
    }
    if (out_pooled != nullptr) {
      Scope sc(enc->prof, P_OTHER, st);
      JEPA_TRY(cuda_status(mean_pool(out_tokens, out_pooled, batch, n_keep, D, st), "mean pool"));
    }
    return JEPA_OK;
  };
  if (enc->prof.on || !enc->graphs.on) return body(s);
  // the ids are read at run time: a replay sees their current contents
  const uint64_t key[12] = {2, (uint64_t)(uintptr_t)clip, (uint64_t)clip_format, (uint64_t)batch,
                            (uint64_t)n_frames, (uint64_t)height, (uint64_t)width, (uint64_t)(uintptr_t)out_tokens,
                            (uint64_t)(uintptr_t)out_pooled, (uint64_t)(uintptr_t)out_hier,
                            (uint64_t)(uintptr_t)ids_keep, (uint64_t)n_keep};
  return encode_replayed(enc, key, batch, gk, g, body, s);
}

jepa_status jepa_encode_host(jepa_encoder* enc, const void* host_clip, int clip_format, int batch, int n_frames,
                             int height, int width, float* host_out_tokens, float* host_out_pooled, void* stream) {
  Geom g;
  JEPA_TRY(check_clip(enc, batch, n_frames, height, width, g));
  if (host_clip == nullptr || host_out_tokens == nullptr) return fail(JEPA_ERR_ARG, "host buffers are required");
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_TRY(cudaSetDevice(enc->device));
  const size_t px = (size_t)batch * n_frames * height * width * 3;
  const size_t clip_bytes = clip_format == JEPA_CLIP_U8_THWC ? px : px * 4;
  const size_t out_bytes = (size_t)batch * g.n_tok * enc->p.embed_dim * 4;
  const size_t pool_bytes = (size_t)batch * enc->p.embed_dim * 4;
  if (enc->h_clip_cap < clip_bytes) {
    cudaFree(enc->h_clip_dev);
    enc->h_clip_dev = nullptr;
    enc->h_clip_cap = 0;
    if (cudaMalloc(&enc->h_clip_dev, clip_bytes) != cudaSuccess) return fail(JEPA_ERR_OOM, "clip staging");
    enc->h_clip_cap = clip_bytes;
  }
  if (enc->h_out_cap < out_bytes) {
    cudaFree(enc->h_out_dev);
    enc->h_out_dev = nullptr;
    enc->h_out_cap = 0;
    if (cudaMalloc(&enc->h_out_dev, out_bytes) != cudaSuccess) return fail(JEPA_ERR_OOM, "output staging");
    enc->h_out_cap = out_bytes;
  }
  if (host_out_pooled != nullptr && enc->h_pool_cap < pool_bytes) {
    cudaFree(enc->h_pool_dev);
    enc->h_pool_dev = nullptr;
    enc->h_pool_cap = 0;
    if (cudaMalloc(&enc->h_pool_dev, pool_bytes) != cudaSuccess) return fail(JEPA_ERR_OOM, "pool staging");
    enc->h_pool_cap = pool_bytes;
  }
  CUDA_TRY(cudaMemcpyAsync(enc->h_clip_dev, host_clip, clip_bytes, cudaMemcpyHostToDevice, s));
  JEPA_TRY(jepa_encode(enc, enc->h_clip_dev, clip_format, batch, n_frames, height, width, enc->h_out_dev,
                       host_out_pooled ? enc->h_pool_dev : nullptr, nullptr, stream));
  CUDA_TRY(cudaMemcpyAsync(host_out_tokens, enc->h_out_dev, out_bytes, cudaMemcpyDeviceToHost, s));
  if (host_out_pooled)
    CUDA_TRY(cudaMemcpyAsync(host_out_pooled, enc->h_pool_dev, pool_bytes, cudaMemcpyDeviceToHost, s));
  return read_status(enc->d_status, s);
}

jepa_status jepa_encode_host_async(jepa_encoder* enc, const void* host_clip, int clip_format, int batch,
                                   int n_frames, int height, int width, float* host_out_tokens,
                                   float* host_out_pooled, void* stream) {
  Geom g;
  JEPA_TRY(check_clip(enc, batch, n_frames, height, width, g));
  if (host_clip == nullptr || host_out_tokens == nullptr) return fail(JEPA_ERR_ARG, "host buffers are required");
  if (clip_format != JEPA_CLIP_U8_THWC && clip_format != JEPA_CLIP_F32_CTHW)
    return fail(JEPA_ERR_ARG, "clip_format %d", clip_format);
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_TRY(cudaSetDevice(enc->device));
  HostPipe& hp = enc->pipe;
  if (hp.in == nullptr) {
    CUDA_TRY(cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking));
    CUDA_TRY(cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking));
    for (auto& sl : hp.slot) {
      CUDA_TRY(cudaEventCreateWithFlags(&sl.copied_in, cudaEventDisableTiming));
      CUDA_TRY(cudaEventCreateWithFlags(&sl.encoded, cudaEventDisableTiming));
      CUDA_TRY(cudaEventCreateWithFlags(&sl.copied_out, cudaEventDisableTiming));
    }
  }
  HostPipe::Slot& sl = hp.slot[hp.calls & 1];
  const size_t px = (size_t)batch * n_frames * height * width * 3;
  const size_t clip_bytes = clip_format == JEPA_CLIP_U8_THWC ? px : px * 4;
  const size_t out_bytes = (size_t)batch * g.n_tok * enc->p.embed_dim * 4;
  const size_t pool_bytes = (size_t)batch * enc->p.embed_dim * 4;
  const size_t need[3] = {clip_bytes, out_bytes, host_out_pooled ? pool_bytes : 0};
  void** buf[3] = {&sl.clip, &sl.out, &sl.pool};
  size_t* cap[3] = {&sl.clip_cap, &sl.out_cap, &sl.pool_cap};
  for (int i = 0; i < 3; ++i) {
    if (*cap[i] >= need[i]) continue;
    // the slot's previous encode and copy-out are done with its buffers
    CUDA_TRY(cudaEventSynchronize(sl.encoded));
    CUDA_TRY(cudaEventSynchronize(sl.copied_out));
    cudaFree(*buf[i]);
    *buf[i] = nullptr;
    *cap[i] = 0;
    if (cudaMalloc(buf[i], need[i]) != cudaSuccess) return fail(JEPA_ERR_OOM, "host staging slot");
    *cap[i] = need[i];
  }
  // in: once the encode that last read this slot's clip is done
  CUDA_TRY(cudaStreamWaitEvent(hp.in, sl.encoded, 0));
  CUDA_TRY(cudaMemcpyAsync(sl.clip, host_clip, clip_bytes, cudaMemcpyHostToDevice, hp.in));
  CUDA_TRY(cudaEventRecord(sl.copied_in, hp.in));
  // encode: once the clip is in and the copy-out that last read this slot's output is done
  CUDA_TRY(cudaStreamWaitEvent(s, sl.copied_in, 0));
  CUDA_TRY(cudaStreamWaitEvent(s, sl.copied_out, 0));
  JEPA_TRY(jepa_encode(enc, sl.clip, clip_format, batch, n_frames, height, width, (float*)sl.out,
                       host_out_pooled ? (float*)sl.pool : nullptr, nullptr, stream));
  CUDA_TRY(cudaEventRecord(sl.encoded, s));
  // out: after the encode
  CUDA_TRY(cudaStreamWaitEvent(hp.out, sl.encoded, 0));
  CUDA_TRY(cudaMemcpyAsync(host_out_tokens, sl.out, out_bytes, cudaMemcpyDeviceToHost, hp.out));
  if (host_out_pooled)
    CUDA_TRY(cudaMemcpyAsync(host_out_pooled, sl.pool, pool_bytes, cudaMemcpyDeviceToHost, hp.out));
  CUDA_TRY(cudaEventRecord(sl.copied_out, hp.out));
  ++hp.calls;
  return JEPA_OK;
}

jepa_status jepa_encoder_sync(jepa_encoder* enc, void* stream) {
  if (enc == nullptr) return fail(JEPA_ERR_ARG, "encoder handle is NULL");
  CUDA_TRY(cudaSetDevice(enc->device));
  if (enc->pipe.out != nullptr) {
    // copies of jepa_encode_host_async (the copy-out follows its encode)
    CUDA_TRY(cudaStreamSynchronize(enc->pipe.in));
    CUDA_TRY(cudaStreamSynchronize(enc->pipe.out));
  }
  return read_status(enc->d_status, (cudaStream_t)stream);
}

jepa_status jepa_encoder_set_profiling(jepa_encoder* enc, int on) {
  if (enc == nullptr) return fail(JEPA_ERR_ARG, "encoder handle is NULL");
  enc->prof.on = on != 0;
  return JEPA_OK;
}

jepa_status jepa_encoder_profile(jepa_encoder* enc, double* times_ms, long long* launches, int reset) {
  if (enc == nullptr) return fail(JEPA_ERR_ARG, "encoder handle is NULL");
  CUDA_TRY(cudaSetDevice(enc->device));
  enc->prof.collect();
  for (int c = 0; c < 8; ++c) {
    if (times_ms) times_ms[c] = enc->prof.times[c];
    if (launches) launches[c] = enc->prof.launches[c];
    if (reset) {
      enc->prof.times[c] = 0;
      enc->prof.launches[c] = 0;
    }
  }
  return JEPA_OK;
}

}  // extern "C"

// ============================================================================= predictor
struct jepa_predictor {
  GraphCache graphs;
  jepa_predictor_params p{};
  int device = 0, sms = 0;
  void* d_weights = nullptr;
  const void* w_emb = nullptr;
  const float* b_emb = nullptr;
  const float* mask_tokens = nullptr;
  std::vector<Block> blocks;
  const float *norm_w = nullptr, *norm_b = nullptr;
  const void* w_proj = nullptr;
  const float* b_proj = nullptr;
  const void* w_projc = nullptr;   // 2.1 context projection, when present
  const float* b_projc = nullptr;
  // Per modality (0 video, 1 image): the embed bias and the mask row with the
  // 2.1 modality vector folded in (the plain ones when the model has none).
  float* b_emb_mod[2] = {nullptr, nullptr};
  float* mask_mod[2] = {nullptr, nullptr};
  void* ws = nullptr;
  size_t ws_bytes = 0;
  int* d_status = nullptr;
  RopeCache rope;
  Profiler prof;
};

extern "C" {

jepa_status jepa_predictor_create(const void* blob, size_t blob_bytes, const jepa_predictor_params* params,
                                  int device, jepa_predictor** out) {
  if (out == nullptr) return fail(JEPA_ERR_ARG, "out is NULL");
  *out = nullptr;
  JEPA_TRY(check_predictor_params(params));
  std::vector<BlobEntry> ent;
  JEPA_TRY(parse_blob(blob, blob_bytes, expected_predictor(*params), ent));
  CUDA_TRY(cudaSetDevice(device));
  jepa_predictor* pr = new jepa_predictor();
  pr->p = *params;
  pr->device = device;
  cudaDeviceGetAttribute(&pr->sms, cudaDevAttrMultiProcessorCount, device);
  std::vector<const void*> P;
  jepa_status st = upload_weights(blob, ent, &pr->d_weights, P);
  if (st != JEPA_OK) {
    delete pr;
    return st;
  }
  size_t i = 0;
  pr->w_emb = P[i++];
  pr->b_emb = (const float*)P[i++];
  pr->mask_tokens = (const float*)P[i++];
  for (int l = 0; l < params->n_layer; ++l) pr->blocks.push_back(take_block(P, i));
  pr->norm_w = (const float*)P[i++];
  pr->norm_b = (const float*)P[i++];
  pr->w_proj = P[i++];
  pr->b_proj = (const float*)P[i++];
  const float* mods[2] = {nullptr, nullptr};
  if (params->has_mod_embed) {
    mods[0] = (const float*)P[i++];
    mods[1] = (const float*)P[i++];
  }
  if (params->has_proj_context) {
    pr->w_projc = P[i++];
    pr->b_projc = (const float*)P[i++];
  }
  const int D = params->embed_dim;
  bool ok = cudaMalloc(&pr->d_status, sizeof(int)) == cudaSuccess;
  for (int m = 0; m < 2 && ok; ++m)
    ok = cudaMalloc(&pr->b_emb_mod[m], D * sizeof(float)) == cudaSuccess &&
         cudaMalloc(&pr->mask_mod[m], D * sizeof(float)) == cudaSuccess;
  if (!ok) {
    jepa_predictor_destroy(pr);
    return fail(JEPA_ERR_OOM, "predictor: small allocations failed");
  }
  cudaMemset(pr->d_status, 0, sizeof(int));
  const float* tok = pr->mask_tokens + (size_t)(params->mask_index % params->n_mask_tokens) * D;
  for (int m = 0; m < 2; ++m) {
    cudaMemcpy(pr->b_emb_mod[m], pr->b_emb, D * sizeof(float), cudaMemcpyDeviceToDevice);
    cudaMemcpy(pr->mask_mod[m], tok, D * sizeof(float), cudaMemcpyDeviceToDevice);
    if (mods[m]) {  // the modality vector joins every row: context rows through the bias, mask rows directly
      add_vec_kernel<<<(D + 255) / 256, 256>>>(pr->b_emb_mod[m], mods[m], D);
      add_vec_kernel<<<(D + 255) / 256, 256>>>(pr->mask_mod[m], mods[m], D);
    }
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    jepa_predictor_destroy(pr);
    return fail(JEPA_ERR_CUDA, "predictor create: %s", cudaGetErrorString(e));
  }
  *out = pr;
  return JEPA_OK;
}

void jepa_predictor_destroy(jepa_predictor* pr) {
  if (pr == nullptr) return;
  cudaSetDevice(pr->device);
  cudaDeviceSynchronize();
  cudaFree(pr->d_weights);
  cudaFree(pr->ws);
  cudaFree(pr->d_status);
  cudaFree(pr->rope.d);
  for (int m = 0; m < 2; ++m) {
    cudaFree(pr->b_emb_mod[m]);
    cudaFree(pr->mask_mod[m]);
  }
  pr->graphs.release();
  delete pr;
}

jepa_status jepa_predict(jepa_predictor* pr, const float* enc_tokens, int n_tokens, const int32_t* ids_ctx, int n_ctx,
                         const int32_t* ids_tgt, int n_tgt, int grid_t, int grid_h, int grid_w, float* out,
                         void* stream) {
  return jepa_predict_ex(pr, enc_tokens, n_tokens, ids_ctx, n_ctx, ids_tgt, n_tgt, grid_t, grid_h, grid_w,
                         JEPA_MODALITY_VIDEO, out, nullptr, stream);
}

jepa_status jepa_predict_ex(jepa_predictor* pr, const float* enc_tokens, int n_tokens, const int32_t* ids_ctx,
                            int n_ctx, const int32_t* ids_tgt, int n_tgt, int grid_t, int grid_h, int grid_w,
                            int modality, float* out, float* out_ctx, void* stream) {
  if (pr == nullptr) return fail(JEPA_ERR_ARG, "predictor handle is NULL");
  if (enc_tokens == nullptr || ids_ctx == nullptr || ids_tgt == nullptr || out == nullptr)
    return fail(JEPA_ERR_ARG, "device buffers are required");
  if (!aligned16(enc_tokens) || !aligned16(out) || (out_ctx != nullptr && !aligned16(out_ctx)))
    return fail(JEPA_ERR_ARG, "buffers must be 16-byte aligned");
  if (modality != JEPA_MODALITY_VIDEO && modality != JEPA_MODALITY_IMAGE && modality != JEPA_MODALITY_AUTO)
    return fail(JEPA_ERR_ARG, "modality %d", modality);
  if (out_ctx != nullptr && !pr->p.has_proj_context)
    return fail(JEPA_ERR_ARG, "out_ctx needs a predictor with a context projection");
  // AUTO: the image vector for a grid of one temporal slice (the image path's grid)
  const int mod = modality == JEPA_MODALITY_AUTO ? (grid_t == 1 ? 1 : 0) : (modality == JEPA_MODALITY_IMAGE ? 1 : 0);
  if (n_ctx < 1 || n_tgt < 1 || n_tokens < 1) return fail(JEPA_ERR_ARG, "n_ctx, n_tgt and n_tokens must be >= 1");
  if (grid_t < 1 || grid_h < 1 || grid_w < 1 || (long long)grid_t * grid_h * grid_w != n_tokens)
    return fail(JEPA_ERR_ARG, "grid %dx%dx%d does not hold %d tokens", grid_t, grid_h, grid_w, n_tokens);
  const int D = pr->p.embed_dim, F = pr->p.ffn_dim, n = n_ctx + n_tgt;
  if ((long long)n * std::max(F, 3 * D) >= (1ll << 31)) return fail(JEPA_ERR_ARG, "too many rows");
  cudaStream_t s0 = (cudaStream_t)stream;
  CUDA_TRY(cudaSetDevice(pr->device));
  const int dt = pr->p.dtype;
  const int hd = D / pr->p.n_head;
  // workspace and RoPE tables (no-ops once sized and built for this grid)
  auto prep = [&](cudaStream_t s) -> jepa_status {
    const size_t need = work_bytes(dt, 1, n, D, F, pr->p.in_dim, true);
    if (need > pr->ws_bytes) {
      cudaFree(pr->ws);
      pr->ws = nullptr;
      pr->ws_bytes = 0;
      if (cudaMalloc(&pr->ws, need) != cudaSuccess) return fail(JEPA_ERR_OOM, "predictor workspace");
      if (cudaMemset(pr->ws, 0, need) != cudaSuccess) return fail(JEPA_ERR_CUDA, "predictor workspace memset");
      pr->ws_bytes = need;
    }
    return rope_prepare(pr->rope, hd, pr->p.rope_layout, pr->p.rope_theta, grid_t, grid_h, grid_w, 0, 0, s);
  };
  auto body = [&](cudaStream_t s) -> jepa_status {
  JEPA_TRY(prep(s));
  Work w = carve(pr->ws, dt, 1, n, D, F, pr->p.in_dim, true);
  // positions of the concatenated sequence: context ids then target ids
  CUDA_TRY(cudaMemcpyAsync(w.pos, ids_ctx, sizeof(int) * n_ctx, cudaMemcpyDeviceToDevice, s));
  CUDA_TRY(cudaMemcpyAsync(w.pos + n_ctx, ids_tgt, sizeof(int) * n_tgt, cudaMemcpyDeviceToDevice, s));
  {
    Scope sc(pr->prof, P_EMBED, s);
    JEPA_TRY(cuda_status(check_ids(ids_ctx, n_ctx, n_tokens, pr->d_status, s), "id check"));
    JEPA_TRY(cuda_status(check_ids(ids_tgt, n_tgt, n_tokens, pr->d_status, s), "id check"));
    JEPA_TRY(cuda_status(gather_rows_cast(dt, enc_tokens, n_tokens, ids_ctx, n_ctx, pr->p.in_dim, w.g, s), "gather"));
    EpiParams ep{};
    ep.bias = pr->b_emb_mod[mod];  // embed bias (+ modality vector)
    ep.out = w.x;
    ep.ldo = D;
    JEPA_TRY(run_linear(dt, EPI_F32, w.g, pr->w_emb, n_ctx, D, pr->p.in_dim, ep, pr->d_status, s, pr->sms));
    JEPA_TRY(cuda_status(fill_rows(w.x + (size_t)n_ctx * D, pr->mask_mod[mod], n_tgt, D, s), "mask tokens"));
  }
  StackDesc sd;
  sd.D = D;
  sd.H = pr->p.n_head;
  sd.F = F;
  sd.dtype = dt;
  sd.eps = pr->p.ln_eps;
  sd.blocks = &pr->blocks;
  sd.n_hier = 0;
  sd.hier_layers = nullptr;
  sd.hier_w = nullptr;
  sd.hier_b = nullptr;
  JEPA_TRY(run_blocks(sd, w, 1, n, 0, pr->p.n_layer, pr->rope.rp, w.pos, nullptr, pr->d_status, pr->prof, s,
                      pr->sms));
  // pred.norm on the target rows (and the context rows when their projection is asked for)
  const int first = out_ctx != nullptr ? 0 : n_ctx;
  {
    Scope sc(pr->prof, P_LN, s);
    JEPA_TRY(cuda_status(layernorm(dt, w.x + (size_t)first * D, pr->norm_w, pr->norm_b, w.y, n - first, D,
                                   pr->p.ln_eps, s),
                         "layernorm"));
  }
  {
    Scope sc(pr->prof, P_OTHER, s);
    const size_t esz = dtype_size(dt);
    EpiParams ep{};
    ep.bias = pr->b_proj;
    ep.out = out;
    ep.ldo = pr->p.out_dim;
    const void* y_tgt = (const char*)w.y + (size_t)(n_ctx - first) * D * esz;
    JEPA_TRY(run_linear(dt, EPI_F32, y_tgt, pr->w_proj, n_tgt, pr->p.out_dim, D, ep, pr->d_status, s, pr->sms));
    if (out_ctx != nullptr) {
      EpiParams ec{};
      ec.bias = pr->b_projc;
      ec.out = out_ctx;
      ec.ldo = pr->p.out_dim;
      JEPA_TRY(run_linear(dt, EPI_F32, w.y, pr->w_projc, n_ctx, pr->p.out_dim, D, ec, pr->d_status, s, pr->sms));
    }
  }
  return JEPA_OK;
  };
  if (pr->prof.on || !pr->graphs.on) return body(s0);
  const uint64_t key[12] = {3, (uint64_t)(uintptr_t)enc_tokens, (uint64_t)n_tokens | ((uint64_t)n_ctx << 32),
                            (uint64_t)(uintptr_t)ids_ctx, (uint64_t)(uintptr_t)ids_tgt, (uint64_t)n_tgt,
                            (uint64_t)grid_t | ((uint64_t)grid_h << 32), (uint64_t)grid_w, (uint64_t)mod,
                            (uint64_t)(uintptr_t)out, (uint64_t)(uintptr_t)out_ctx, 0};
  return replay(pr->graphs, key, prep, pr->ws, pr->rope.d, body, s0);
}

jepa_status jepa_predictor_set_graphs(jepa_predictor* pr, int on) {
  if (pr == nullptr) return fail(JEPA_ERR_ARG, "predictor handle is NULL");
  pr->graphs.on = on != 0;
  return JEPA_OK;
}

jepa_status jepa_predictor_sync(jepa_predictor* pr, void* stream) {
  if (pr == nullptr) return fail(JEPA_ERR_ARG, "predictor handle is NULL");
  CUDA_TRY(cudaSetDevice(pr->device));
  return read_status(pr->d_status, (cudaStream_t)stream);
}

// ============================================================================= single operations
jepa_status jepa_layernorm_f32(const float* x, const float* w, const float* b, float* y, int rows, int dim, float eps,
                               void* stream) {
  if (rows < 0 || dim <= 0 || dim % 128 != 0 || dim > 4096)
    return fail(JEPA_ERR_ARG, "rows %d / dim %d (dim a multiple of 128, <= 4096)", rows, dim);
  if (rows == 0) return JEPA_OK;
  if (!x || !w || !b || !y) return fail(JEPA_ERR_ARG, "NULL buffer");
  if (!aligned16(x) || !aligned16(w) || !aligned16(b) || !aligned16(y)) return fail(JEPA_ERR_ARG, "buffers must be 16-byte aligned");
  if (!(eps > 0.f)) return fail(JEPA_ERR_ARG, "eps must be > 0");
  return cuda_status(layernorm(DTYPE_F32, x, w, b, y, rows, dim, eps, (cudaStream_t)stream), "layernorm");
}

jepa_status jepa_rope3d_f32(float* x, int batch, int n_tokens, int n_head, int head_dim, int grid_t, int grid_h,
                            int grid_w, int layout, int interpolate, int ref_grid, float theta, void* stream) {
  if (!x || !aligned16(x)) return fail(JEPA_ERR_ARG, "x must be a 16-byte aligned buffer");
  if (head_dim != 32 && head_dim != 64) return fail(JEPA_ERR_UNSUPPORTED, "head_dim %d (32 or 64)", head_dim);
  if (batch < 0 || n_head < 1 || grid_t < 1 || grid_h < 1 || grid_w < 1 ||
      (long long)grid_t * grid_h * grid_w != n_tokens)
    return fail(JEPA_ERR_ARG, "grid %dx%dx%d does not hold %d tokens", grid_t, grid_h, grid_w, n_tokens);
  if (layout != 0 && layout != 1) return fail(JEPA_ERR_ARG, "layout %d", layout);
  if (interpolate && (grid_h < 2 || grid_w < 2 || ref_grid < 2))
    return fail(JEPA_ERR_ARG, "interpolation needs a grid and reference wider than 1");
  if (!(theta > 0.f)) return fail(JEPA_ERR_ARG, "theta must be > 0");
  RopeCache& rc = ops_rope_cache();
  cudaStream_t s = (cudaStream_t)stream;
  JEPA_TRY(rope_prepare(rc, head_dim, layout, theta, grid_t, grid_h, grid_w, interpolate, ref_grid, s));
  if (batch == 0) return JEPA_OK;
  return cuda_status(rope_inplace_f32(x, batch, n_tokens, n_head, head_dim, rc.rp, s), "rope");
}

jepa_status jepa_attention(const void* q, const void* k, const void* vt, void* out, int dtype, int batch, int n_head,
                           int n_tokens, int head_dim, int ldv, float scale, void* stream) {
  if (!q || !k || !vt || !out) return fail(JEPA_ERR_ARG, "NULL buffer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(out)) return fail(JEPA_ERR_ARG, "buffers must be 16-byte aligned");
  if (dtype < 0 || dtype > 2) return fail(JEPA_ERR_ARG, "dtype %d", dtype);
  if (head_dim != 32 && head_dim != 64) return fail(JEPA_ERR_UNSUPPORTED, "head_dim %d (32 or 64)", head_dim);
  if (batch < 1 || n_head < 1 || n_tokens < 1) return fail(JEPA_ERR_ARG, "batch, n_head, n_tokens must be >= 1");
  if (ldv < n_tokens || ldv % 8 != 0) return fail(JEPA_ERR_ARG, "ldv %d must be >= n_tokens and a multiple of 8", ldv);
  if ((long long)batch * n_head > 65535) return fail(JEPA_ERR_ARG, "batch * n_head > 65535");
  int* st = nullptr;
  JEPA_TRY(ops_status(&st));
  cudaStream_t s = (cudaStream_t)stream;
  if (dtype == DTYPE_F32)
    return cuda_status(attention_simt(dtype, q, k, vt, out, batch, n_head, n_tokens, head_dim, ldv, scale, s),
                       "attention");
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return cuda_status(attention_tc(dtype, q, k, vt, out, batch, n_head, n_tokens, head_dim, ldv, scale, st, s, sms),
                     "attention");
}

jepa_status jepa_linear(const void* A, const void* W, const float* bias, void* out, int M, int N, int K, int dtype,
                        int epilogue, void* stream) {
  if (!A || !W || !out) return fail(JEPA_ERR_ARG, "NULL buffer");
  if (!aligned16(A) || !aligned16(W) || !aligned16(out) || !aligned16(bias)) return fail(JEPA_ERR_ARG, "buffers must be 16-byte aligned");
  if (dtype < 0 || dtype > 2) return fail(JEPA_ERR_ARG, "dtype %d", dtype);
  if (epilogue < 0 || epilogue > 3) return fail(JEPA_ERR_ARG, "epilogue %d", epilogue);
  if (M < 0 || N <= 0 || K <= 0) return fail(JEPA_ERR_ARG, "M %d N %d K %d", M, N, K);
  if (dtype == DTYPE_F32 && (K % 16 != 0 || N % 4 != 0))
    return fail(JEPA_ERR_ARG, "fp32 linear needs K %% 16 == 0 and N %% 4 == 0");
  if (dtype != DTYPE_F32 && (K % 64 != 0 || N % 128 != 0))
    return fail(JEPA_ERR_ARG, "tensor-core linear needs K %% 64 == 0 and N %% 128 == 0");
  int* st = nullptr;
  JEPA_TRY(ops_status(&st));
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  EpiParams ep{};
  ep.bias = bias;
  ep.out = out;
  ep.ldo = N;
  return run_linear(dtype, epilogue, A, W, M, N, K, ep, st, (cudaStream_t)stream, sms);
}

jepa_status jepa_qkv_rope(const void* A, const void* W, const float* bias, void* q, void* k, void* vt, int dtype,
                          int batch, int n_tokens, int embed_dim, int n_head, int ldv, int grid_t, int grid_h,
                          int grid_w, int layout, int interpolate, int ref_grid, float theta, const int32_t* pos_ids,
                          void* stream) {
  if (!A || !W || !q || !k || !vt) return fail(JEPA_ERR_ARG, "NULL buffer");
  if (!aligned16(A) || !aligned16(W) || !aligned16(bias) || !aligned16(q) || !aligned16(k) || !aligned16(vt))
    return fail(JEPA_ERR_ARG, "buffers must be 16-byte aligned");
  if (dtype < 0 || dtype > 2) return fail(JEPA_ERR_ARG, "dtype %d", dtype);
  JEPA_TRY(check_width(embed_dim, n_head, 128, dtype, "qkv_rope"));   // this call has no FFN: 128 passes its check
  const int hd = embed_dim / n_head;
  if (batch < 1 || n_tokens < 1) return fail(JEPA_ERR_ARG, "batch %d and n_tokens %d must be >= 1", batch, n_tokens);
  if (grid_t < 1 || grid_h < 1 || grid_w < 1) return fail(JEPA_ERR_ARG, "grid %dx%dx%d", grid_t, grid_h, grid_w);
  const long long cells = (long long)grid_t * grid_h * grid_w;
  if (pos_ids == nullptr && cells != n_tokens)
    return fail(JEPA_ERR_ARG, "grid %dx%dx%d does not hold %d tokens (give pos_ids for a subset)", grid_t, grid_h,
                grid_w, n_tokens);
  if (cells >= (1ll << 31)) return fail(JEPA_ERR_ARG, "grid too large");
  if (ldv < n_tokens || ldv % 8 != 0) return fail(JEPA_ERR_ARG, "ldv %d must be >= n_tokens and a multiple of 8", ldv);
  if ((long long)batch * n_tokens * 3 * embed_dim >= (1ll << 31)) return fail(JEPA_ERR_ARG, "too many rows");
  if (layout != 0 && layout != 1) return fail(JEPA_ERR_ARG, "layout %d", layout);
  if (interpolate && (grid_h < 2 || grid_w < 2 || ref_grid < 2))
    return fail(JEPA_ERR_ARG, "interpolation needs a grid and reference wider than 1");
  if (!(theta > 0.f)) return fail(JEPA_ERR_ARG, "theta must be > 0");
  int* st = nullptr;
  JEPA_TRY(ops_status(&st));
  cudaStream_t s = (cudaStream_t)stream;
  RopeCache& rc = ops_rope_cache();
  JEPA_TRY(rope_prepare(rc, hd, layout, theta, grid_t, grid_h, grid_w, interpolate, ref_grid, s));
  const int M = batch * n_tokens;
  if (pos_ids != nullptr) JEPA_TRY(cuda_status(check_ids(pos_ids, M, (int)cells, st, s), "id check"));
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  EpiParams ep{};
  ep.bias = bias;
  ep.q = q;
  ep.k = k;
  ep.vt = vt;
  ep.n_tok = n_tokens;
  ep.n_head = n_head;
  ep.head_dim = hd;
  ep.ldv = ldv;
  ep.dmodel = embed_dim;
  ep.pos_ids = pos_ids;
  ep.rope = rc.rp;
  return run_linear(dtype, EPI_QKV, A, W, M, 3 * embed_dim, embed_dim, ep, st, s, sms);
}

jepa_status jepa_ops_sync(void* stream) {
  int* st = nullptr;
  JEPA_TRY(ops_status(&st));
  return read_status(st, (cudaStream_t)stream);
}

jepa_status jepa_selftest_wait_timeout(int timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 5000000) return fail(JEPA_ERR_ARG, "timeout_us %d (1 .. 5e6)", timeout_us);
  int* st = nullptr;
  JEPA_TRY(ops_status(&st));
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_TRY(wait_timeout_selftest(st, (uint64_t)timeout_us * 1000ull, s));
  return read_status(st, s);
}

}  // extern "C"

// ============================================================================= attentive-pool head
struct jepa_head {
  jepa_head_params p{};
  int device = 0, sms = 0;
  void* d_weights = nullptr;
  const float* query = nullptr;
  std::vector<Block> blocks;
  const float *kv_w = nullptr, *kv_b = nullptr;
  const void *wq = nullptr, *wk = nullptr, *wv = nullptr;
  const float *bq = nullptr, *bk = nullptr, *bv = nullptr;
  const float *ln2_w = nullptr, *ln2_b = nullptr;
  const void *w_up = nullptr, *w_down = nullptr, *w_cls = nullptr;
  const float *b_up = nullptr, *b_down = nullptr, *b_cls = nullptr;
  float* q = nullptr;  // [D]    q0 Wq^T + bq (computed at create)
  float* g = nullptr;  // [H, D] ln_kv's gamma * Wk_h^T q_h / sqrt(hd)
  void* ws = nullptr;
  size_t ws_bytes = 0;
  int* d_status = nullptr;
  RopeCache rope;      // the identity rotation (one grid cell): the pool blocks carry no RoPE
  Profiler prof;
  GraphCache graphs;
};

namespace {

constexpr int kHeadChunk = 256;  // tokens per partial weighted sum

std::vector<Expect> expected_head(const jepa_head_params& p) {
  std::vector<Expect> v;
  const uint32_t D = p.embed_dim, F = p.ffn_dim, C = p.n_classes;
  v.push_back({DTYPE_F32, D, 1, 1});                     // head.query
  for (int i = 0; i < p.n_layer; ++i) push_block(v, p.dtype, D, F);
  v.push_back({DTYPE_F32, D, 1, 1});                     // xattn.ln_kv
  v.push_back({DTYPE_F32, D, 1, 1});
  for (int j = 0; j < 3; ++j) {                          // xattn.q, k, v
    v.push_back({p.dtype, D, D, 2});
    v.push_back({DTYPE_F32, D, 1, 1});
  }
  v.push_back({DTYPE_F32, D, 1, 1});                     // xattn.ln2
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({p.dtype, F, D, 2});                       // xattn.ffn_up
  v.push_back({DTYPE_F32, F, 1, 1});
  v.push_back({p.dtype, D, F, 2});                       // xattn.ffn_down
  v.push_back({DTYPE_F32, D, 1, 1});
  v.push_back({p.dtype, C, D, 2});                       // cls
  v.push_back({DTYPE_F32, C, 1, 1});
  return v;
}

jepa_status check_head_params(const jepa_head_params* p) {
  if (p == nullptr) return fail(JEPA_ERR_ARG, "params is NULL");
  JEPA_TRY(check_width(p->embed_dim, p->n_head, p->ffn_dim, p->dtype, "head"));
  if (p->embed_dim / p->n_head != 64) return fail(JEPA_ERR_UNSUPPORTED, "head: head_dim must be 64");
  if (p->embed_dim > 1024) return fail(JEPA_ERR_UNSUPPORTED, "head: embed_dim %d (at most 1024)", p->embed_dim);
  if (p->n_layer < 0 || p->n_classes < 1) return fail(JEPA_ERR_ARG, "head: n_layer %d, n_classes %d", p->n_layer, p->n_classes);
  if (!(p->ln_eps > 0.f)) return fail(JEPA_ERR_ARG, "head: ln_eps must be > 0");
  return JEPA_OK;
}

// Workspace of one head call: the blocks' Work, then scores [M, H], row
// statistics [M, 2], softmax weights [B, H, n], partial sums [chunks, B, H,
// D], z [B, H, D], y [B, D], ln2(y) [B, D], hidden [B, F], pooled [B, D].
struct HeadWork {
  Work w;
  float *s, *stats, *wts, *part, *z, *y, *yn, *hid, *pooled;
};

size_t head_extra_floats(int B, int n, int D, int F) {
  const size_t H = D / 64, M = (size_t)B * n, chunks = (n + kHeadChunk - 1) / kHeadChunk;
  return align256(M * H * 4) + align256(M * 8) + align256((size_t)B * H * n * 4) +
         align256(chunks * B * H * D * 4) + align256((size_t)B * H * D * 4) + 3 * align256((size_t)B * D * 4) +
         align256((size_t)B * F * 4);
}

HeadWork head_carve(void* base, int dtype, int B, int n, int D, int F) {
  HeadWork hw;
  hw.w = carve(base, dtype, B, n, D, F, 0, false);
  const size_t H = D / 64, M = (size_t)B * n, chunks = (n + kHeadChunk - 1) / kHeadChunk;
  uint8_t* p = static_cast<uint8_t*>(base) + work_bytes(dtype, B, n, D, F, 0, false);
  hw.s = reinterpret_cast<float*>(p);      p += align256(M * H * 4);
  hw.stats = reinterpret_cast<float*>(p);  p += align256(M * 8);
  hw.wts = reinterpret_cast<float*>(p);    p += align256((size_t)B * H * n * 4);
  hw.part = reinterpret_cast<float*>(p);   p += align256(chunks * B * H * D * 4);
  hw.z = reinterpret_cast<float*>(p);      p += align256((size_t)B * H * D * 4);
  hw.y = reinterpret_cast<float*>(p);      p += align256((size_t)B * D * 4);
  hw.yn = reinterpret_cast<float*>(p);     p += align256((size_t)B * D * 4);
  hw.pooled = reinterpret_cast<float*>(p); p += align256((size_t)B * D * 4);
  hw.hid = reinterpret_cast<float*>(p);
  return hw;
}

}  // namespace

extern "C" {

jepa_status jepa_head_blob_check(const void* blob, size_t blob_bytes, const jepa_head_params* params) {
  JEPA_TRY(check_head_params(params));
  std::vector<BlobEntry> ent;
  return parse_blob(blob, blob_bytes, expected_head(*params), ent);
}

jepa_status jepa_head_create(const void* blob, size_t blob_bytes, const jepa_head_params* params, int device,
                             jepa_head** out) {
  if (out == nullptr) return fail(JEPA_ERR_ARG, "out is NULL");
  *out = nullptr;
  JEPA_TRY(check_head_params(params));
  std::vector<BlobEntry> ent;
  JEPA_TRY(parse_blob(blob, blob_bytes, expected_head(*params), ent));
  CUDA_TRY(cudaSetDevice(device));
  jepa_head* hd = new jepa_head();
  hd->p = *params;
  hd->device = device;
  cudaDeviceGetAttribute(&hd->sms, cudaDevAttrMultiProcessorCount, device);
  std::vector<const void*> P;
  jepa_status st = upload_weights(blob, ent, &hd->d_weights, P);
  if (st != JEPA_OK) {
    delete hd;
    return st;
  }
  size_t i = 0;
  hd->query = (const float*)P[i++];
  for (int l = 0; l < params->n_layer; ++l) hd->blocks.push_back(take_block(P, i));
  hd->kv_w = (const float*)P[i++];
  hd->kv_b = (const float*)P[i++];
  hd->wq = P[i++];
  hd->bq = (const float*)P[i++];
  hd->wk = P[i++];
  hd->bk = (const float*)P[i++];
  hd->wv = P[i++];
  hd->bv = (const float*)P[i++];
  hd->ln2_w = (const float*)P[i++];
  hd->ln2_b = (const float*)P[i++];
  hd->w_up = P[i++];
  hd->b_up = (const float*)P[i++];
  hd->w_down = P[i++];
  hd->b_down = (const float*)P[i++];
  hd->w_cls = P[i++];
  hd->b_cls = (const float*)P[i++];
  const int D = params->embed_dim, H = params->n_head;
  if (cudaMalloc(&hd->q, D * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&hd->g, (size_t)H * D * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&hd->d_status, sizeof(int)) != cudaSuccess) {
    jepa_head_destroy(hd);
    return fail(JEPA_ERR_OOM, "head: small allocations failed");
  }
  cudaMemset(hd->d_status, 0, sizeof(int));
  cudaError_t e = head_fold_query(params->dtype, hd->wq, hd->bq, hd->query, hd->wk, hd->kv_w, hd->q, hd->g, D, H, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    jepa_head_destroy(hd);
    return fail(JEPA_ERR_CUDA, "head create: %s", cudaGetErrorString(e));
  }
  // one grid cell: every token at position (0, 0, 0), cos 1 and sin 0 on every pair
  st = rope_prepare(hd->rope, 64, 0, 10000.f, 1, 1, 1, 0, 0, 0);
  if (st != JEPA_OK) {
    jepa_head_destroy(hd);
    return st;
  }
  *out = hd;
  return JEPA_OK;
}

void jepa_head_destroy(jepa_head* hd) {
  if (hd == nullptr) return;
  cudaSetDevice(hd->device);
  cudaDeviceSynchronize();
  cudaFree(hd->d_weights);
  cudaFree(hd->q);
  cudaFree(hd->g);
  cudaFree(hd->ws);
  cudaFree(hd->d_status);
  cudaFree(hd->rope.d);
  hd->graphs.release();
  delete hd;
}

jepa_status jepa_head_forward(jepa_head* hd, const float* tokens, int batch, int n_tokens, float* logits,
                              float* pooled, void* stream) {
  if (hd == nullptr) return fail(JEPA_ERR_ARG, "head handle is NULL");
  if (tokens == nullptr || logits == nullptr) return fail(JEPA_ERR_ARG, "tokens and logits are required");
  if (!aligned16(tokens) || !aligned16(logits) || !aligned16(pooled))
    return fail(JEPA_ERR_ARG, "device buffers must be 16-byte aligned");
  if (batch < 1 || n_tokens < 1) return fail(JEPA_ERR_ARG, "batch %d and n_tokens %d must be >= 1", batch, n_tokens);
  const int D = hd->p.embed_dim, F = hd->p.ffn_dim, H = hd->p.n_head, C = hd->p.n_classes, dt = hd->p.dtype;
  if ((long long)batch * n_tokens * std::max(3 * D, F) >= (1ll << 31)) return fail(JEPA_ERR_ARG, "too many rows");
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_TRY(cudaSetDevice(hd->device));
  // workspace (a no-op once sized for this shape)
  auto prep = [&](cudaStream_t) -> jepa_status {
    const size_t need = work_bytes(dt, batch, n_tokens, D, F, 0, false) + head_extra_floats(batch, n_tokens, D, F);
    if (need <= hd->ws_bytes) return JEPA_OK;
    cudaFree(hd->ws);
    hd->ws = nullptr;
    hd->ws_bytes = 0;
    if (cudaMalloc(&hd->ws, need) != cudaSuccess) return fail(JEPA_ERR_OOM, "head workspace: cudaMalloc(%zu)", need);
    if (cudaMemset(hd->ws, 0, need) != cudaSuccess) return fail(JEPA_ERR_CUDA, "head workspace memset");
    hd->ws_bytes = need;
    return JEPA_OK;
  };
  auto body = [&](cudaStream_t st) -> jepa_status {
    JEPA_TRY(prep(st));
    HeadWork hw = head_carve(hd->ws, dt, batch, n_tokens, D, F);
    const int M = batch * n_tokens;
    // the pool blocks work in place on a copy of the encoder tokens
    CUDA_TRY(cudaMemcpyAsync(hw.w.x, tokens, (size_t)M * D * sizeof(float), cudaMemcpyDeviceToDevice, st));
    StackDesc sd;
    sd.D = D;
    sd.H = H;
    sd.F = F;
    sd.dtype = dt;
    sd.eps = hd->p.ln_eps;
    sd.blocks = &hd->blocks;
    sd.n_hier = 0;
    sd.hier_layers = nullptr;
    sd.hier_w = nullptr;
    sd.hier_b = nullptr;
    JEPA_TRY(run_blocks(sd, hw.w, batch, n_tokens, 0, hd->p.n_layer, hd->rope.rp, nullptr, nullptr, hd->d_status,
                        hd->prof, st, hd->sms));
    // cross-attention of the learned query over ln_kv(x)
    JEPA_TRY(cuda_status(head_xattn_scores(hw.w.x, hd->g, hw.s, hw.stats, M, D, hd->p.ln_eps, hd->sms, st),
                         "head scores"));
    JEPA_TRY(cuda_status(head_xattn_pool(hw.w.x, hw.s, hw.stats, hd->kv_w, hd->kv_b, hw.wts, hw.part, hw.z, batch,
                                         n_tokens, D, kHeadChunk, st),
                         "head pooling"));
    constexpr int kAll = 1 << 30;   // every output column reads the same A row
    float* pool = pooled != nullptr ? pooled : hw.pooled;
    // y = q0 + Wv_h z_h + bv (no output projection; the residual is the raw query)
    JEPA_TRY(cuda_status(head_rowvec(dt, false, hw.z, H * D, 64, D, hd->wv, hd->bv, hd->query, 0, hw.y, D, batch, D,
                                     D, st),
                         "head values"));
    JEPA_TRY(cuda_status(layernorm(DTYPE_F32, hw.y, hd->ln2_w, hd->ln2_b, hw.yn, batch, D, hd->p.ln_eps, st),
                         "head ln2"));
    JEPA_TRY(cuda_status(head_rowvec(dt, true, hw.yn, D, kAll, 0, hd->w_up, hd->b_up, nullptr, 0, hw.hid, F, batch,
                                     F, D, st),
                         "head ffn_up"));
    JEPA_TRY(cuda_status(head_rowvec(dt, false, hw.hid, F, kAll, 0, hd->w_down, hd->b_down, hw.y, D, pool, D, batch,
                                     D, F, st),
                         "head ffn_down"));
    return cuda_status(head_rowvec(dt, false, pool, D, kAll, 0, hd->w_cls, hd->b_cls, nullptr, 0, logits, C, batch,
                                   C, D, st),
                       "head classifier");
  };
  if (!hd->graphs.on) return body(s);
  // repeated calls with the same buffers and shapes replay one captured graph
  const uint64_t key[12] = {4, (uint64_t)(uintptr_t)tokens, (uint64_t)batch, (uint64_t)n_tokens,
                            (uint64_t)(uintptr_t)logits, (uint64_t)(uintptr_t)pooled, 0, 0, 0, 0, 0, 0};
  return replay(hd->graphs, key, prep, hd->ws, hd->rope.d, body, s);
}

jepa_status jepa_head_set_graphs(jepa_head* hd, int on) {
  if (hd == nullptr) return fail(JEPA_ERR_ARG, "head handle is NULL");
  hd->graphs.on = on != 0;
  return JEPA_OK;
}

jepa_status jepa_head_sync(jepa_head* hd, void* stream) {
  if (hd == nullptr) return fail(JEPA_ERR_ARG, "head handle is NULL");
  CUDA_TRY(cudaSetDevice(hd->device));
  return read_status(hd->d_status, (cudaStream_t)stream);
}

}  // extern "C"
