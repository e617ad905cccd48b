// The fused GEMM epilogues, shared by the tensor-core and the fp32 CUDA-core
// GEMM.  A thread owns n consecutive columns [col0, col0+n) of one output row.
#pragma once
#include "common.cuh"

namespace jepa {

template <typename T, int n>
__device__ __forceinline__ void store_row_chunk(T* dst, const float (&v)[n]) {
  if constexpr (sizeof(T) == 2 && n % 8 == 0) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < n / 8; ++i) {
      uint4 u;
      u.x = pack2<T>(v[8 * i + 0], v[8 * i + 1]);
      u.y = pack2<T>(v[8 * i + 2], v[8 * i + 3]);
      u.z = pack2<T>(v[8 * i + 4], v[8 * i + 5]);
      u.w = pack2<T>(v[8 * i + 6], v[8 * i + 7]);
      d4[i] = u;
    }
  } else if constexpr (sizeof(T) == 4 && n % 4 == 0) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < n / 4; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < n; ++i) dst[i] = DT<T>::from(v[i]);
  }
}

// Applies epilogue EPI to the accumulator values v of row `row`, columns
// [col0, col0+n), and stores the result.  The caller guarantees row < M and
// col0 + n <= N.
template <typename T, int EPI, int n>
__device__ __forceinline__ void epilogue_apply(const EpiParams& ep, int row, int col0, float (&v)[n]) {
  if (ep.bias != nullptr) {
    const float* b = ep.bias + col0;
    if constexpr (n % 4 == 0) {
#pragma unroll
      for (int i = 0; i < n; i += 4) {
        const float4 bb = __ldg(reinterpret_cast<const float4*>(b + i));
        v[i] += bb.x;
        v[i + 1] += bb.y;
        v[i + 2] += bb.z;
        v[i + 3] += bb.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < n; ++i) v[i] += __ldg(b + i);
    }
  }
  if constexpr (EPI == EPI_STORE) {
    store_row_chunk<T, n>(reinterpret_cast<T*>(ep.out) + (size_t)row * ep.ldo + col0, v);
  } else if constexpr (EPI == EPI_GELU) {
#pragma unroll
    for (int i = 0; i < n; ++i) v[i] = gelu_erf(v[i]);
    store_row_chunk<T, n>(reinterpret_cast<T*>(ep.out) + (size_t)row * ep.ldo + col0, v);
  } else if constexpr (EPI == EPI_F32) {
    store_row_chunk<float, n>(reinterpret_cast<float*>(ep.out) + (size_t)row * ep.ldo + col0, v);
  } else if constexpr (EPI == EPI_RESID) {
    float* dst = reinterpret_cast<float*>(ep.out) + (size_t)row * ep.ldo + col0;
    if constexpr (n % 4 == 0) {
#pragma unroll
      for (int i = 0; i < n; i += 4) {
        const float4 r = *reinterpret_cast<const float4*>(dst + i);
        v[i] += r.x;
        v[i + 1] += r.y;
        v[i + 2] += r.z;
        v[i + 3] += r.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < n; ++i) v[i] += dst[i];
    }
    store_row_chunk<float, n>(dst, v);
  } else if constexpr (EPI == EPI_QKV) {
    const int D = ep.dmodel, hd = ep.head_dim;
    const int which = col0 / D;
    const int cc = col0 - which * D;
    const int head = cc / hd;
    const int d0 = cc - head * hd;
    const int clip = row / ep.n_tok;
    const int tok = row - clip * ep.n_tok;
    const size_t bh = (size_t)clip * ep.n_head + head;
    if (which < 2) {
      const int plane = ep.rope.gh * ep.rope.gw;
      // a caller's id outside the grid is clamped (and reported by the id check)
      const int gid = min(max(ep.pos_ids != nullptr ? __ldg(ep.pos_ids + row) : tok, 0), ep.rope.gt * plane - 1);
      const int t = gid / plane;
      const int rem = gid - t * plane;
      const int h = rem / ep.rope.gw;
      const int w = rem - h * ep.rope.gw;
      rope_apply<n>(v, d0, ep.rope, t, h, w);
      T* dst = reinterpret_cast<T*>(which == 0 ? ep.q : ep.k) + (bh * ep.n_tok + tok) * hd + d0;
      store_row_chunk<T, n>(dst, v);
    } else {
      T* dst = reinterpret_cast<T*>(ep.vt) + (bh * hd + d0) * (size_t)ep.ldv + tok;
#pragma unroll
      for (int i = 0; i < n; ++i) dst[(size_t)i * ep.ldv] = DT<T>::from(v[i]);
    }
  }
}

}  // namespace jepa
