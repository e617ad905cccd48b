// Kernels of the attentive-pool head's cross-attention and of its per-clip
// tail ("V-JEPA 2 / 2.1 tensor maps and RoPE derivation", §2 "Attentive-pool
// head - exact forward"):
//   kv = ln_kv(x); q = q0 Wq^T + bq; k = kv Wk^T + bk; v = kv Wv^T + bv;
//   o_h = softmax(q_h k_h^T / sqrt(hd)) v_h, heads concatenated, no output
//   projection; y = q0 + o; y += ffn_down(gelu(ffn_up(ln2(y)))); logits =
//   y Wcls^T + bcls.
//
// The query is one fixed vector, so the key projection folds into it:
// q_h . k_ih / sqrt(hd) = kv_i . u_h + (q_h . bk_h) / sqrt(hd) with
// u_h = Wk_h^T q_h / sqrt(hd), and the second term, equal for every key,
// drops out of the softmax.  With kv_i = (x_i - mu_i) rstd_i * gamma + beta
// the score of token i for head h is, up to that same kind of constant,
//   s_ih = rstd_i * sum_d (x_id - mu_i) g_hd,   g_h = gamma * u_h,
// and since the weights sum to one the values follow the weighted sum:
//   o_h = Wv_h z_h + bv_h,  z_h = gamma * sum_i w_ih (x_i - mu_i) + beta,
//   w_ih = p_ih rstd_i.
// So the cross-attention reads x twice in fp32 (scores, then the weighted
// sum) instead of projecting every token through Wk and Wv; u, g and q are
// computed once when the head is created.  All of it is fp32 on the CUDA
// cores: a single query row has no tile for the tensor cores to fill.
#include "internal.h"

namespace jepa {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// out[n] = sum_k W[n, k] x[k] + b[n]: one warp per output.
template <typename T>
__global__ void matvec_kernel(const T* __restrict__ W, const float* __restrict__ x, const float* __restrict__ b,
                              float* __restrict__ out, int N, int K) {
  const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  float acc = 0.f;
  for (int k = lane; k < K; k += 32) acc += DT<T>::to(W[(size_t)n * K + k]) * x[k];
  acc = warp_sum(acc);
  if (lane == 0) out[n] = acc + (b != nullptr ? b[n] : 0.f);
}

// Key fold: u[h, d] = scale * sum_r Wk[h*hd + r, d] q[h*hd + r];
// g[h, d] = gamma[d] u[h, d].  One thread per (h, d).
template <typename T>
__global__ void fold_keys_kernel(const T* __restrict__ Wk, const float* __restrict__ q,
                                 const float* __restrict__ gamma, float* __restrict__ g, int D, int H, int hd,
                                 float scale) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= H * D) return;
  const int h = idx / D, d = idx - h * D;
  float acc = 0.f;
  for (int r = 0; r < hd; ++r) acc += DT<T>::to(Wk[(size_t)(h * hd + r) * D + d]) * q[h * hd + r];
  g[idx] = gamma[d] * (acc * scale);
}

// Scores of every token for every head, and its LayerNorm statistics.  One
// warp per token row held in registers (NV float4 per lane, D = 128 NV,
// heads H = 2 NV of width 64); g [H, D] is staged in shared memory by the
// block.  s[r, h] = rstd * sum_d (x_d - mu) g[h, d]; stats[r] = (mu, rstd).
template <int NV>
__global__ void __launch_bounds__(256) xattn_scores_kernel(const float* __restrict__ x,
                                                           const float* __restrict__ g, float* __restrict__ s,
                                                           float2* __restrict__ stats, int rows, float eps) {
  constexpr int D = 128 * NV, H = 2 * NV;
  extern __shared__ float4 g_s[];   // [H][D / 4]
  for (int i = threadIdx.x; i < H * D / 4; i += blockDim.x) g_s[i] = reinterpret_cast<const float4*>(g)[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int n_warps = (gridDim.x * blockDim.x) >> 5;
  for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows; row += n_warps) {
    float4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = reinterpret_cast<const float4*>(x + (size_t)row * D)[lane + 32 * i];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) sum += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    const float mu = warp_sum(sum) * (1.0f / D);
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      v[i].x -= mu; v[i].y -= mu; v[i].z -= mu; v[i].w -= mu;
      q += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
    }
    const float rstd = 1.0f / sqrtf(warp_sum(q) * (1.0f / D) + eps);
    float mine = 0.f;   // lane h keeps head h's score
#pragma unroll 1
    for (int h = 0; h < H; ++h) {
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const float4 gg = g_s[h * (D / 4) + lane + 32 * i];
        a += (v[i].x * gg.x + v[i].y * gg.y) + (v[i].z * gg.z + v[i].w * gg.w);
      }
      a = warp_sum(a);
      if (lane == h) mine = a;
    }
    if (lane < H) s[(size_t)row * H + lane] = mine * rstd;
    if (lane == 0) stats[row] = make_float2(mu, rstd);
  }
}

// Softmax over the n tokens of one (clip, head): block (h, b).
// w[b, h, i] = exp(s_ih - max) / sum * rstd_i.
__global__ void xattn_softmax_kernel(const float* __restrict__ s, const float2* __restrict__ stats,
                                     float* __restrict__ w, int n, int H) {
  const int h = blockIdx.x, b = blockIdx.y;
  __shared__ float red[32];
  const float* sb = s + (size_t)b * n * H + h;
  float mx = -INFINITY;
  for (int i = threadIdx.x; i < n; i += blockDim.x) mx = fmaxf(mx, sb[(size_t)i * H]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    float m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  mx = red[0];
  __syncthreads();
  float l = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) l += expf(sb[(size_t)i * H] - mx);
  l = warp_sum(l);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = l;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = 1.0f / red[0];
  float* wb = w + ((size_t)b * H + h) * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    wb[i] = expf(sb[(size_t)i * H] - mx) * inv * stats[(size_t)b * n + i].y;
}

// Partial weighted sums: part[c, b, h, d] = sum over tokens i of chunk c of
// w[b, h, i] (x[b, i, d] - mu_i).  Block (column group of 128, b, chunk);
// thread = one column; the chunk's weights are staged in shared memory.
template <int H>
__global__ void __launch_bounds__(128) xattn_wsum_kernel(const float* __restrict__ x, const float2* __restrict__ stats,
                                                         const float* __restrict__ w, float* __restrict__ part,
                                                         int n, int D, int chunk) {
  const int d = blockIdx.x * 128 + threadIdx.x;
  const int b = blockIdx.y, c = blockIdx.z;
  const int i0 = c * chunk, i1 = min(n, i0 + chunk);
  __shared__ float ws[64][H];
  __shared__ float mus[64];
  float acc[H];
#pragma unroll
  for (int h = 0; h < H; ++h) acc[h] = 0.f;
  for (int t0 = i0; t0 < i1; t0 += 64) {
    const int cnt = min(64, i1 - t0);
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * H; e += 128) {
      const int h = e >> 6, ii = e & 63;   // consecutive threads read consecutive tokens
      ws[ii][h] = ii < cnt ? w[((size_t)b * H + h) * n + t0 + ii] : 0.f;
    }
    if (threadIdx.x < 64) mus[threadIdx.x] = threadIdx.x < cnt ? stats[(size_t)b * n + t0 + threadIdx.x].x : 0.f;
    __syncthreads();
    if (d < D) {
      const float* xr = x + ((size_t)b * n + t0) * D + d;
      for (int ii = 0; ii < cnt; ++ii) {
        const float xv = xr[(size_t)ii * D] - mus[ii];
#pragma unroll
        for (int h = 0; h < H; ++h) acc[h] += ws[ii][h] * xv;
      }
    }
  }
  if (d < D) {
    const int B = gridDim.y;
#pragma unroll
    for (int h = 0; h < H; ++h) part[(((size_t)c * B + b) * H + h) * D + d] = acc[h];
  }
}

// z[b, h, d] = gamma[d] * sum_c part[c, b, h, d] + beta[d] (the chunks in a fixed order).
__global__ void xattn_finish_kernel(const float* __restrict__ part, const float* __restrict__ gamma,
                                    const float* __restrict__ beta, float* __restrict__ z, int n_chunks, long total,
                                    int D) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  float acc = 0.f;
  for (int c = 0; c < n_chunks; ++c) acc += part[(size_t)c * total + idx];
  const int d = (int)(idx % D);
  z[idx] = gamma[d] * acc + beta[d];
}

// Row-vector products of the per-clip tail, one warp per output column n:
//   out[b, n] = act(sum_k A[b*lda + (n / group)*gstride + k] W[n, k] + bias[n])
//               + (res ? res[b*ldr + n] : 0)
// act: identity, or the exact-erf GELU.  `group` lets the value projection
// read each head's own z row (group = head_dim, gstride = D).
template <typename T, bool GELU>
__global__ void rowvec_kernel(const float* __restrict__ A, int lda, int group, int gstride, const T* __restrict__ W,
                              const float* __restrict__ bias, const float* __restrict__ res, int ldr,
                              float* __restrict__ out, int ldo, int B, int N, int K) {
  const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  const T* wr = W + (size_t)n * K;
  const size_t a_off = (size_t)(n / group) * gstride;
  for (int b = 0; b < B; ++b) {
    const float* ar = A + (size_t)b * lda + a_off;
    float acc = 0.f;
    for (int k = lane; k < K; k += 32) acc += DT<T>::to(wr[k]) * ar[k];
    acc = warp_sum(acc);
    if (lane == 0) {
      float v = acc + (bias != nullptr ? bias[n] : 0.f);
      if (GELU) v = gelu_erf(v);
      if (res != nullptr) v += res[(size_t)b * ldr + n];
      out[(size_t)b * ldo + n] = v;
    }
  }
}

inline unsigned blocks_for(long n, int per) { return (unsigned)((n + per - 1) / per); }

}  // namespace

cudaError_t head_fold_query(int dtype, const void* Wq, const float* bq, const float* q0, const void* Wk,
                            const float* gamma_kv, float* q_out, float* g_out, int D, int H, cudaStream_t s) {
  const int hd = D / H;
  const float scale = 1.0f / sqrtf((float)hd);
  if (dtype == DTYPE_BF16) {
    matvec_kernel<__nv_bfloat16><<<blocks_for(D, 8), 256, 0, s>>>((const __nv_bfloat16*)Wq, q0, bq, q_out, D, D);
    fold_keys_kernel<__nv_bfloat16><<<blocks_for((long)H * D, 256), 256, 0, s>>>(
        (const __nv_bfloat16*)Wk, q_out, gamma_kv, g_out, D, H, hd, scale);
  } else if (dtype == DTYPE_F16) {
    matvec_kernel<__half><<<blocks_for(D, 8), 256, 0, s>>>((const __half*)Wq, q0, bq, q_out, D, D);
    fold_keys_kernel<__half><<<blocks_for((long)H * D, 256), 256, 0, s>>>((const __half*)Wk, q_out, gamma_kv, g_out,
                                                                            D, H, hd, scale);
  } else {
    matvec_kernel<float><<<blocks_for(D, 8), 256, 0, s>>>((const float*)Wq, q0, bq, q_out, D, D);
    fold_keys_kernel<float><<<blocks_for((long)H * D, 256), 256, 0, s>>>((const float*)Wk, q_out, gamma_kv, g_out,
                                                                           D, H, hd, scale);
  }
  return cudaGetLastError();
}

cudaError_t head_xattn_scores(const float* x, const float* g, float* s, float* stats, int rows, int D, float eps,
                              int num_sms, cudaStream_t st) {
  const int nv = D / 128;
  const size_t smem = (size_t)(2 * nv) * D * sizeof(float);
  const int need = (rows + 7) / 8;
  const int blocks = need < 2 * num_sms ? need : 2 * num_sms;
  float2* st2 = reinterpret_cast<float2*>(stats);
#define JEPA_XS(NV)                                                                                              \
  case NV: {                                                                                                     \
    static DeviceOnce setup;                                                                                     \
    cudaError_t e = setup.run([&](int) {                                                                         \
      return cudaFuncSetAttribute(xattn_scores_kernel<NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,          \
                                  (int)(2 * NV * 128 * NV * sizeof(float)));                                     \
    });                                                                                                          \
    if (e != cudaSuccess) return e;                                                                              \
    xattn_scores_kernel<NV><<<blocks, 256, smem, st>>>(x, g, s, st2, rows, eps);                                 \
    break;                                                                                                       \
  }
  switch (nv) {
    JEPA_XS(2)
    JEPA_XS(4)
    JEPA_XS(6)
    JEPA_XS(8)
    default: return cudaErrorInvalidValue;
  }
#undef JEPA_XS
  return cudaGetLastError();
}

cudaError_t head_xattn_pool(const float* x, const float* s, const float* stats, const float* gamma,
                            const float* beta, float* w, float* part, float* z, int B, int n, int D, int chunk,
                            cudaStream_t st) {
  const int H = D / 64;
  const float2* st2 = reinterpret_cast<const float2*>(stats);
  xattn_softmax_kernel<<<dim3(H, B), 256, 0, st>>>(s, st2, w, n, H);
  const int n_chunks = (n + chunk - 1) / chunk;
  dim3 grid((D + 127) / 128, B, n_chunks);
  switch (H) {
    case 4: xattn_wsum_kernel<4><<<grid, 128, 0, st>>>(x, st2, w, part, n, D, chunk); break;
    case 8: xattn_wsum_kernel<8><<<grid, 128, 0, st>>>(x, st2, w, part, n, D, chunk); break;
    case 12: xattn_wsum_kernel<12><<<grid, 128, 0, st>>>(x, st2, w, part, n, D, chunk); break;
    case 16: xattn_wsum_kernel<16><<<grid, 128, 0, st>>>(x, st2, w, part, n, D, chunk); break;
    default: return cudaErrorInvalidValue;
  }
  const long total = (long)B * H * D;
  xattn_finish_kernel<<<blocks_for(total, 256), 256, 0, st>>>(part, gamma, beta, z, n_chunks, total, D);
  return cudaGetLastError();
}

cudaError_t head_rowvec(int dtype, bool gelu, const float* A, int lda, int group, int gstride, const void* W,
                        const float* bias, const float* res, int ldr, float* out, int ldo, int B, int N, int K,
                        cudaStream_t s) {
  const unsigned grid = blocks_for(N, 8);
#define JEPA_RV(T)                                                                                             \
  if (gelu)                                                                                                    \
    rowvec_kernel<T, true><<<grid, 256, 0, s>>>(A, lda, group, gstride, (const T*)W, bias, res, ldr, out, ldo, B, \
                                                N, K);                                                         \
  else                                                                                                         \
    rowvec_kernel<T, false><<<grid, 256, 0, s>>>(A, lda, group, gstride, (const T*)W, bias, res, ldr, out, ldo, \
                                                 B, N, K);
  if (dtype == DTYPE_BF16) {
    JEPA_RV(__nv_bfloat16)
  } else if (dtype == DTYPE_F16) {
    JEPA_RV(__half)
  } else {
    JEPA_RV(float)
  }
#undef JEPA_RV
  return cudaGetLastError();
}

}  // namespace jepa
