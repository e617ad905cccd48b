// Attention on the CUDA cores with fp32 arithmetic: the path of the fp32
// encoder mode.  One thread owns one query row (q and the output accumulator
// in registers); keys and values stream through shared memory in tiles of 64;
// the softmax is the online (running max / running sum) form, exact up to
// rounding.
#include "internal.h"

namespace jepa {

namespace {

constexpr int kQ = 128;   // query rows per block
constexpr int kKT = 64;   // keys per tile

template <typename T, int HD>
__global__ void __launch_bounds__(kQ) attn_simt_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                       const T* __restrict__ vt, T* __restrict__ out, int n_head,
                                                       int n_tok, int ldv, float scale_log2) {
  __shared__ float Ks[kKT][HD];
  __shared__ float Vs[kKT][HD + 1];
  const int bh = blockIdx.y;
  const int b = bh / n_head, head = bh - b * n_head;
  const int row = blockIdx.x * kQ + threadIdx.x;
  const bool valid = row < n_tok;
  float qr[HD], o[HD];
  const T* qp = q + ((size_t)bh * n_tok + (valid ? row : 0)) * HD;
#pragma unroll
  for (int d = 0; d < HD; ++d) {
    qr[d] = DT<T>::to(qp[d]) * scale_log2;
    o[d] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const T* kb = k + (size_t)bh * n_tok * HD;
  const T* vb = vt + (size_t)bh * HD * ldv;
  for (int j0 = 0; j0 < n_tok; j0 += kKT) {
    const int nk = min(kKT, n_tok - j0);
    __syncthreads();
    for (int i = threadIdx.x; i < kKT * HD; i += kQ) {
      const int j = i / HD, d = i - (i / HD) * HD;
      Ks[j][d] = j < nk ? DT<T>::to(kb[(size_t)(j0 + j) * HD + d]) : 0.f;
      const int d2 = i / kKT, j2 = i - (i / kKT) * kKT;
      Vs[j2][d2] = j2 < nk ? DT<T>::to(vb[(size_t)d2 * ldv + j0 + j2]) : 0.f;
    }
    __syncthreads();
    for (int j = 0; j < nk; ++j) {
      float s = 0.f;
#pragma unroll
      for (int d = 0; d < HD; ++d) s = fmaf(qr[d], Ks[j][d], s);
      if (s > m) {
        const float corr = exp2f(m - s);
        l *= corr;
#pragma unroll
        for (int d = 0; d < HD; ++d) o[d] *= corr;
        m = s;
      }
      const float p = exp2f(s - m);
      l += p;
#pragma unroll
      for (int d = 0; d < HD; ++d) o[d] = fmaf(p, Vs[j][d], o[d]);
    }
  }
  if (!valid) return;
  const float inv = 1.0f / l;
  T* op = out + ((size_t)b * n_tok + row) * (size_t)(n_head * HD) + head * HD;
#pragma unroll
  for (int d = 0; d < HD; ++d) op[d] = DT<T>::from(o[d] * inv);
}

template <typename T>
cudaError_t launch_t(const void* q, const void* k, const void* vt, void* out, int batch, int n_head, int n_tok,
                     int hd, int ldv, float scale, cudaStream_t s) {
  dim3 grid((n_tok + kQ - 1) / kQ, batch * n_head);
  const float sl2 = scale * 1.4426950408889634f;
  if (hd == 64)
    attn_simt_kernel<T, 64><<<grid, kQ, 0, s>>>((const T*)q, (const T*)k, (const T*)vt, (T*)out, n_head, n_tok,
                                                ldv, sl2);
  else if (hd == 32)
    attn_simt_kernel<T, 32><<<grid, kQ, 0, s>>>((const T*)q, (const T*)k, (const T*)vt, (T*)out, n_head, n_tok,
                                                ldv, sl2);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace

cudaError_t attention_simt(int dtype, const void* q, const void* k, const void* vt, void* out, int batch, int n_head,
                           int n_tok, int head_dim, int ldv, float scale, cudaStream_t s) {
  if (dtype == DTYPE_F32) return launch_t<float>(q, k, vt, out, batch, n_head, n_tok, head_dim, ldv, scale, s);
  if (dtype == DTYPE_BF16)
    return launch_t<__nv_bfloat16>(q, k, vt, out, batch, n_head, n_tok, head_dim, ldv, scale, s);
  return launch_t<__half>(q, k, vt, out, batch, n_head, n_tok, head_dim, ldv, scale, s);
}

}  // namespace jepa
