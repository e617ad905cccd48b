// Memory-bound kernels: clip normalise + tubelet unfold, LayerNorm, RoPE on
// fp32 rows, token mean pool, predictor row gathers, and the bounded-wait
// self test.  Each is a single pass over HBM with 16-byte accesses.
#include "internal.h"

namespace jepa {

namespace {


// The normalisation is the fused form (px - 255 mean) / (255 std) with the
// ImageNet statistics, as a product with the reciprocal (pix_mean255 and
// pix_rcp255 in common.cuh): a division per value made the kernel bound by
// instruction issue.
//
// One thread per (token, dt, y): reads the 16 pixels x 3 channels of one
// tubelet row (48 contiguous bytes of the THWC clip) and writes the three
// 16-wide runs c*(TUB*256) + dt*256 + y*16 + [0,16) of the token's
// 3*TUB*256-wide row (the row-major C,T,H,W flattening of the Conv3d kernel,
// conversion notes §2).  TUB = 2 for clips, 1 for the 2.1 image path.  With
// `keep` ([batch, n_keep] token ids, the masked encoder) row r of clip b is
// token keep[b * n_keep + r], clamped to the grid.
template <typename T, int TUB>
__global__ void unfold_u8_kernel(const uint8_t* __restrict__ clip, T* __restrict__ out, int batch, int T_, int H,
                                 int W, const int* __restrict__ keep, int n_keep) {
  constexpr int K = 3 * TUB * 256;
  const int gt = T_ / TUB, gh = H >> 4, gw = W >> 4;
  const long n_tok = (long)gt * gh * gw;
  const long rows = keep != nullptr ? n_keep : n_tok;  // rows per clip
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long total = (long)batch * rows * 16 * TUB;
  if (idx >= total) return;
  const int y = idx & 15;
  const int dt = (int)((idx >> 4) % TUB);
  const long row = (idx >> 4) / TUB;
  const long b = row / rows;
  const long tok = keep != nullptr ? min(max(__ldg(keep + row), 0), (int)n_tok - 1) : row - b * rows;
  const int t = tok / (gh * gw);
  const int rem = tok - (long)t * gh * gw;
  const int hh = rem / gw, ww = rem - hh * gw;
  const long frame = (long)b * T_ + TUB * t + dt;
  const uint8_t* src = clip + ((frame * H + 16 * hh + y) * (long)W + 16 * ww) * 3;
  uint4 raw[3];
  raw[0] = __ldg(reinterpret_cast<const uint4*>(src));
  raw[1] = __ldg(reinterpret_cast<const uint4*>(src) + 1);
  raw[2] = __ldg(reinterpret_cast<const uint4*>(src) + 2);
  const uint8_t* px = reinterpret_cast<const uint8_t*>(raw);
  T* dst = out + row * K + dt * 256 + y * 16;
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    float v[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) v[x] = ((float)px[3 * x + c] - pix_mean255(c)) * pix_rcp255(c);
    T* d = dst + c * (TUB * 256);
    if constexpr (sizeof(T) == 2) {
      uint4 u0, u1;
      u0.x = pack2<T>(v[0], v[1]);   u0.y = pack2<T>(v[2], v[3]);
      u0.z = pack2<T>(v[4], v[5]);   u0.w = pack2<T>(v[6], v[7]);
      u1.x = pack2<T>(v[8], v[9]);   u1.y = pack2<T>(v[10], v[11]);
      u1.z = pack2<T>(v[12], v[13]); u1.w = pack2<T>(v[14], v[15]);
      reinterpret_cast<uint4*>(d)[0] = u0;
      reinterpret_cast<uint4*>(d)[1] = u1;
    } else {
#pragma unroll
      for (int x = 0; x < 16; x += 4)
        reinterpret_cast<float4*>(d)[x / 4] = make_float4(v[x], v[x + 1], v[x + 2], v[x + 3]);
    }
  }
}

// Same unfold from an already normalised float clip [batch, 3, T, H, W]:
// one thread per (token, c, dt, y) copies 16 floats.
template <typename T, int TUB>
__global__ void unfold_f32_kernel(const float* __restrict__ clip, T* __restrict__ out, int batch, int T_, int H,
                                  int W, const int* __restrict__ keep, int n_keep) {
  constexpr int K = 3 * TUB * 256;
  const int gt = T_ / TUB, gh = H >> 4, gw = W >> 4;
  const long n_tok = (long)gt * gh * gw;
  const long rows = keep != nullptr ? n_keep : n_tok;  // rows per clip
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long total = (long)batch * rows * 48 * TUB;
  if (idx >= total) return;
  const int y = idx & 15;
  const int dt = (int)((idx >> 4) % TUB);
  const long r2 = (idx >> 4) / TUB;
  const int c = r2 % 3;
  const long row = r2 / 3;
  const long b = row / rows;
  const long tok = keep != nullptr ? min(max(__ldg(keep + row), 0), (int)n_tok - 1) : row - b * rows;
  const int t = tok / (gh * gw);
  const int rem = tok - (long)t * gh * gw;
  const int hh = rem / gw, ww = rem - hh * gw;
  const float* src = clip + ((((b * 3 + c) * T_ + TUB * t + dt) * (long)H + 16 * hh + y) * W + 16 * ww);
  float v[16];
#pragma unroll
  for (int x = 0; x < 16; ++x) v[x] = __ldg(src + x);
  T* d = out + row * K + c * (TUB * 256) + dt * 256 + y * 16;
#pragma unroll
  for (int x = 0; x < 16; ++x) d[x] = DT<T>::from(v[x]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per row; the row stays in registers (NV float4 per lane, dim =
// 128 * NV).  Mean first, then the centred variance, then the affine map.
template <typename T, int NV>
__global__ void layernorm_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                 const float* __restrict__ b, T* __restrict__ y, int rows, float eps) {
  constexpr int dim = 128 * NV;
  const int lane = threadIdx.x & 31;
  const int n_warps = (gridDim.x * blockDim.x) >> 5;
  int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  // Each warp walks rows row, row + n_warps, ...; the next row's loads are
  // issued before the current row is reduced, so two rows are in flight.
  float4 nxt[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) nxt[i] = reinterpret_cast<const float4*>(x + (size_t)row * dim)[lane + 32 * i];
  for (; row < rows; row += n_warps) {
    float4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = nxt[i];
    const int next = row + n_warps;
    if (next < rows) {
#pragma unroll
      for (int i = 0; i < NV; ++i) nxt[i] = reinterpret_cast<const float4*>(x + (size_t)next * dim)[lane + 32 * i];
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    const float mu = warp_sum(s) * (1.0f / dim);
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      v[i].x -= mu; v[i].y -= mu; v[i].z -= mu; v[i].w -= mu;
      q += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
    }
    const float var = warp_sum(q) * (1.0f / dim);
    const float rstd = 1.0f / sqrtf(var + eps);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c = 4 * (lane + 32 * i);
      const float4 ww = __ldg(reinterpret_cast<const float4*>(w + c));
      const float4 bb = __ldg(reinterpret_cast<const float4*>(b + c));
      const float o0 = v[i].x * rstd * ww.x + bb.x;
      const float o1 = v[i].y * rstd * ww.y + bb.y;
      const float o2 = v[i].z * rstd * ww.z + bb.z;
      const float o3 = v[i].w * rstd * ww.w + bb.w;
      T* yr = y + (size_t)row * dim + c;
      if constexpr (sizeof(T) == 2) {
        uint2 u;
        u.x = pack2<T>(o0, o1);
        u.y = pack2<T>(o2, o3);
        *reinterpret_cast<uint2*>(yr) = u;
      } else {
        *reinterpret_cast<float4*>(yr) = make_float4(o0, o1, o2, o3);
      }
    }
  }
}

template <typename T>
cudaError_t layernorm_t(const float* x, const float* w, const float* b, void* y, int rows, int dim, float eps,
                        cudaStream_t s) {
  const int nv = dim / 128;
  // persistent: 2 blocks of 8 warps per SM, each warp striding over ~rows/2432 rows
  static DeviceOnce setup;
  static int sms_on[kMaxDevices];
  int dev = 0;
  cudaError_t e = setup.run([](int d) {
    int n = 0;
    const cudaError_t r = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    sms_on[d] = (r == cudaSuccess && n >= 1) ? n : 1;
    return r;
  }, &dev);
  if (e != cudaSuccess) return e;
  const int sms = sms_on[dev];
  const int need = (rows + 7) / 8;
  const int blocks = need < 2 * sms ? need : 2 * sms;
  T* yy = reinterpret_cast<T*>(y);
  switch (nv) {
    case 1: layernorm_kernel<T, 1><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    case 2: layernorm_kernel<T, 2><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    case 3: layernorm_kernel<T, 3><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    case 4: layernorm_kernel<T, 4><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    case 6: layernorm_kernel<T, 6><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    case 8: layernorm_kernel<T, 8><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    case 12: layernorm_kernel<T, 12><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    case 16: layernorm_kernel<T, 16><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    case 24: layernorm_kernel<T, 24><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    case 32: layernorm_kernel<T, 32><<<blocks, 256, 0, s>>>(x, w, b, yy, rows, eps); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Token mean: block (column chunk of 128, clip, token slice); partial sums are
// combined with atomics into out, which the host zeroes first.
__global__ void mean_pool_kernel(const float* __restrict__ x, float* __restrict__ out, int n_tok, int dim,
                                 int tok_per_block) {
  const int col = blockIdx.x * 128 + threadIdx.x;
  const int b = blockIdx.y;
  const int t0 = blockIdx.z * tok_per_block;
  const int t1 = min(n_tok, t0 + tok_per_block);
  if (col >= dim) return;
  const float* p = x + ((size_t)b * n_tok) * dim + col;
  float s = 0.f;
  for (int t = t0; t < t1; ++t) s += p[(size_t)t * dim];
  atomicAdd(out + (size_t)b * dim + col, s / (float)n_tok);
}

// One thread per (row, head): the head's HD values in registers, rotated in
// place.
template <int HD>
__global__ void rope_f32_kernel(float* __restrict__ x, int rows, int n_tok, int n_head, RopeParams rp) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)rows * n_head) return;
  const long row = idx / n_head;
  const int head = idx - row * n_head;
  const int tok = row % n_tok;
  const int plane = rp.gh * rp.gw;
  const int t = tok / plane, rem = tok - t * plane;
  const int h = rem / rp.gw, w = rem - h * rp.gw;
  float4* p = reinterpret_cast<float4*>(x + (row * n_head + head) * HD);
  float v[HD];
#pragma unroll
  for (int i = 0; i < HD / 4; ++i) {
    const float4 q = p[i];
    v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
  }
  rope_apply<HD>(v, 0, rp, t, h, w);
#pragma unroll
  for (int i = 0; i < HD / 4; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

template <typename T>
__global__ void gather_cast_kernel(const float* __restrict__ src, int n_src, const int* __restrict__ ids, int n,
                                   int dim, T* __restrict__ dst) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const int q = dim >> 2;
  if (idx >= (long)n * q) return;
  const long r = idx / q;
  const int c = (idx - r * q) * 4;
  const int id = min(max(__ldg(ids + r), 0), n_src - 1);  // out-of-range ids are clamped (and reported)
  const float4 v = __ldg(reinterpret_cast<const float4*>(src + (size_t)id * dim + c));
  T* d = dst + r * dim + c;
  d[0] = DT<T>::from(v.x); d[1] = DT<T>::from(v.y); d[2] = DT<T>::from(v.z); d[3] = DT<T>::from(v.w);
}

// Sets DEV_BAD_INDEX when any id lies outside [0, limit).
__global__ void check_ids_kernel(const int* __restrict__ ids, long n, int limit, int* status) {
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const int v = __ldg(ids + i);
    if (v < 0 || v >= limit) atomicOr(status, DEV_BAD_INDEX);
  }
}

__global__ void fill_rows_kernel(float* __restrict__ dst, const float* __restrict__ row, int n, int dim) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)n * dim) return;
  dst[idx] = __ldg(row + idx % dim);
}

// Waits on a barrier that nothing completes; reports the expired wait.
__global__ void wait_timeout_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, limit_ns)) atomicOr(status, DEV_TIMEOUT);
  }
}

inline unsigned grid_for(long n, int block) { return (unsigned)((n + block - 1) / block); }

}  // namespace

template <int TUB>
cudaError_t unfold_u8_t(int dtype, const uint8_t* clip, void* out, int batch, int T, int H, int W, const int* keep,
                        int n_keep, cudaStream_t s) {
  const long rows = keep != nullptr ? n_keep : (long)(T / TUB) * (H / 16) * (W / 16);
  const long total = (long)batch * rows * 16 * TUB;
  if (total == 0) return cudaSuccess;
  if (dtype == DTYPE_BF16)
    unfold_u8_kernel<__nv_bfloat16, TUB><<<grid_for(total, 256), 256, 0, s>>>(clip, (__nv_bfloat16*)out, batch, T, H, W,
                                                                              keep, n_keep);
  else if (dtype == DTYPE_F16)
    unfold_u8_kernel<__half, TUB><<<grid_for(total, 256), 256, 0, s>>>(clip, (__half*)out, batch, T, H, W, keep, n_keep);
  else
    unfold_u8_kernel<float, TUB><<<grid_for(total, 256), 256, 0, s>>>(clip, (float*)out, batch, T, H, W, keep, n_keep);
  return cudaGetLastError();
}

template <int TUB>
cudaError_t unfold_f32_t(int dtype, const float* clip, void* out, int batch, int T, int H, int W, const int* keep,
                         int n_keep, cudaStream_t s) {
  const long rows = keep != nullptr ? n_keep : (long)(T / TUB) * (H / 16) * (W / 16);
  const long total = (long)batch * rows * 48 * TUB;
  if (total == 0) return cudaSuccess;
  if (dtype == DTYPE_BF16)
    unfold_f32_kernel<__nv_bfloat16, TUB><<<grid_for(total, 256), 256, 0, s>>>(clip, (__nv_bfloat16*)out, batch, T, H,
                                                                               W, keep, n_keep);
  else if (dtype == DTYPE_F16)
    unfold_f32_kernel<__half, TUB><<<grid_for(total, 256), 256, 0, s>>>(clip, (__half*)out, batch, T, H, W, keep,
                                                                        n_keep);
  else
    unfold_f32_kernel<float, TUB><<<grid_for(total, 256), 256, 0, s>>>(clip, (float*)out, batch, T, H, W, keep, n_keep);
  return cudaGetLastError();
}

cudaError_t unfold_clip_u8(int dtype, const uint8_t* clip, void* out, int batch, int T, int H, int W, int tubelet,
                           cudaStream_t s, const int* keep, int n_keep) {
  return tubelet == 1 ? unfold_u8_t<1>(dtype, clip, out, batch, T, H, W, keep, n_keep, s)
                      : unfold_u8_t<2>(dtype, clip, out, batch, T, H, W, keep, n_keep, s);
}

cudaError_t unfold_clip_f32(int dtype, const float* clip, void* out, int batch, int T, int H, int W, int tubelet,
                            cudaStream_t s, const int* keep, int n_keep) {
  return tubelet == 1 ? unfold_f32_t<1>(dtype, clip, out, batch, T, H, W, keep, n_keep, s)
                      : unfold_f32_t<2>(dtype, clip, out, batch, T, H, W, keep, n_keep, s);
}

cudaError_t layernorm(int out_dtype, const float* x, const float* w, const float* b, void* y, int rows, int dim,
                      float eps, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (out_dtype == DTYPE_BF16) return layernorm_t<__nv_bfloat16>(x, w, b, y, rows, dim, eps, s);
  if (out_dtype == DTYPE_F16) return layernorm_t<__half>(x, w, b, y, rows, dim, eps, s);
  return layernorm_t<float>(x, w, b, y, rows, dim, eps, s);
}

cudaError_t mean_pool(const float* x, float* out, int batch, int n_tok, int dim, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float) * (size_t)batch * dim, s);
  if (e != cudaSuccess) return e;
  const int tpb = 256;
  dim3 grid((dim + 127) / 128, batch, (n_tok + tpb - 1) / tpb);
  mean_pool_kernel<<<grid, 128, 0, s>>>(x, out, n_tok, dim, tpb);
  return cudaGetLastError();
}

cudaError_t rope_inplace_f32(float* x, int batch, int n_tok, int n_head, int head_dim, const RopeParams& rp,
                             cudaStream_t s) {
  const long rows = (long)batch * n_tok;
  const long n = rows * n_head;
  if (head_dim == 64)
    rope_f32_kernel<64><<<grid_for(n, 128), 128, 0, s>>>(x, (int)rows, n_tok, n_head, rp);
  else if (head_dim == 32)
    rope_f32_kernel<32><<<grid_for(n, 128), 128, 0, s>>>(x, (int)rows, n_tok, n_head, rp);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t gather_rows_cast(int dtype, const float* src, int n_src, const int* ids, int n, int dim, void* dst,
                             cudaStream_t s) {
  const long total = (long)n * (dim / 4);
  if (total == 0) return cudaSuccess;
  if (dtype == DTYPE_BF16)
    gather_cast_kernel<__nv_bfloat16><<<grid_for(total, 256), 256, 0, s>>>(src, n_src, ids, n, dim,
                                                                           (__nv_bfloat16*)dst);
  else if (dtype == DTYPE_F16)
    gather_cast_kernel<__half><<<grid_for(total, 256), 256, 0, s>>>(src, n_src, ids, n, dim, (__half*)dst);
  else
    gather_cast_kernel<float><<<grid_for(total, 256), 256, 0, s>>>(src, n_src, ids, n, dim, (float*)dst);
  return cudaGetLastError();
}

cudaError_t check_ids(const int* ids, long n, int limit, int* status, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  check_ids_kernel<<<grid_for(n, 256), 256, 0, s>>>(ids, n, limit, status);
  return cudaGetLastError();
}

cudaError_t fill_rows(float* dst, const float* row, int n, int dim, cudaStream_t s) {
  const long total = (long)n * dim;
  if (total == 0) return cudaSuccess;
  fill_rows_kernel<<<grid_for(total, 256), 256, 0, s>>>(dst, row, n, dim);
  return cudaGetLastError();
}

cudaError_t wait_timeout_selftest(int* status, uint64_t limit_ns, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace jepa
