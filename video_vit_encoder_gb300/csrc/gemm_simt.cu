// fp32 linear layer on the CUDA cores (FFMA, no TF32): the path of the fp32
// encoder mode.  64x64 output tile per 256-thread block, K in slices of 16
// staged through shared memory, 4x4 outputs per thread, fused epilogue.
#include "epilogue.cuh"
#include "internal.h"

namespace jepa {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

template <int EPI>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const float* __restrict__ A, const float* __restrict__ W,
                                                        int M, int N, int K, EpiParams ep) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Ws[TK][TN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  // loader mapping: 64 rows x 16 k = 256 float4
  const int lr = tid >> 2;        // 0..63
  const int lk = (tid & 3) * 4;   // 0,4,8,12
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), w = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m0 + lr < M) a = __ldg(reinterpret_cast<const float4*>(A + (size_t)(m0 + lr) * K + k0 + lk));
    if (n0 + lr < N) w = __ldg(reinterpret_cast<const float4*>(W + (size_t)(n0 + lr) * K + k0 + lk));
    __syncthreads();
    As[lk + 0][lr] = a.x; As[lk + 1][lr] = a.y; As[lk + 2][lr] = a.z; As[lk + 3][lr] = a.w;
    Ws[lk + 0][lr] = w.x; Ws[lk + 1][lr] = w.y; Ws[lk + 2][lr] = w.z; Ws[lk + 3][lr] = w.w;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 wv = *reinterpret_cast<const float4*>(&Ws[kk][tx * 4]);
      const float ar[4] = {av.x, av.y, av.z, av.w};
      const float wr[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], wr[j], acc[i][j]);
    }
  }
  const int col0 = n0 + tx * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i;
    if (row < M && col0 < N) {
      float v[4] = {acc[i][0], acc[i][1], acc[i][2], acc[i][3]};
      epilogue_apply<float, EPI, 4>(ep, row, col0, v);
    }
  }
}

}  // namespace

cudaError_t gemm_simt_f32(int epi, const float* A, const float* W, int M, int N, int K, const EpiParams& ep,
                          cudaStream_t s) {
  dim3 grid((N + TN - 1) / TN, (M + TM - 1) / TM);
  switch (epi) {
    case EPI_STORE: gemm_simt_kernel<EPI_STORE><<<grid, 256, 0, s>>>(A, W, M, N, K, ep); break;
    case EPI_F32: gemm_simt_kernel<EPI_F32><<<grid, 256, 0, s>>>(A, W, M, N, K, ep); break;
    case EPI_RESID: gemm_simt_kernel<EPI_RESID><<<grid, 256, 0, s>>>(A, W, M, N, K, ep); break;
    case EPI_GELU: gemm_simt_kernel<EPI_GELU><<<grid, 256, 0, s>>>(A, W, M, N, K, ep); break;
    case EPI_QKV: gemm_simt_kernel<EPI_QKV><<<grid, 256, 0, s>>>(A, W, M, N, K, ep); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace jepa
