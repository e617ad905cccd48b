// Tensor-core attention for sm_103a, softmax(scale q k^T) v per (clip, head).
//
// One CTA owns 128 query rows of one (clip, head).  Keys and values stream
// in tiles of 128 through a TMA ring.  Per tile j:
//   S_j = Q K_j^T   tcgen05.mma into one of two TMEM score buffers (fp32);
//   softmax warps (one thread per query row) read S_j, update the running
//   max m and sum l in fp32, write P_j = exp2(S_j - m) as 16-bit into
//   128B-swizzled shared memory;
//   O += P_j V_j    tcgen05.mma into the TMEM output accumulator.
// The running max is only moved (and O rescaled through TMEM) when it grows
// by more than 2^8, so most tiles skip the rescale; m, l and O stay
// consistent, and the final O / l is exact up to rounding.
// V arrives transposed ([hd, keys], keys contiguous), so every MMA operand is
// K-major.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer and
// tensor-memory owner, warps 2-5 softmax and output (warp w owns TMEM lanes
// and query rows 32*(w%4) .. +31).
#include "internal.h"

namespace jepa {

namespace {

constexpr int kBQ = 128;     // query rows per CTA
constexpr int kBKV = 128;    // keys per tile
constexpr int kStages = 3;   // K/V ring depth
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;  // S0 [0,128), S1 [128,256), O [256, 256+HD)

template <int HD>
struct AttnSmem {
  static constexpr uint32_t kQBytes = kBQ * HD * 2;
  static constexpr uint32_t kKBytes = kBKV * HD * 2;
  static constexpr uint32_t kVBytes = HD * kBKV * 2;    // two 64-key blocks of HD rows x 128 B
  static constexpr uint32_t kVBlock = HD * 128;
  static constexpr uint32_t kPBytes = kBQ * kBKV * 2;   // two 64-key blocks of 128 rows x 128 B
  static constexpr uint32_t kPBlock = kBQ * 128;
  static constexpr uint32_t kOffK = kQBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kKBytes;
  static constexpr uint32_t kOffP = kOffV + kStages * kVBytes;
  static constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;
  static constexpr size_t kBytes = 1024 + kOffBar + 256;
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <typename T, int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, T* __restrict__ out, int n_head, int n_tok,
                   float scale_log2, int* status) {
  using S = AttnSmem<HD>;
  constexpr int kQKRow = HD * 2;  // bytes per Q/K row = swizzle width (128 or 64)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + S::kOffK;
  uint8_t* sV = smem + S::kOffV;
  uint8_t* sP = smem + S::kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;   // [2]
  uint64_t* p_full = s_full + 2;           // [2]
  uint64_t* pv_done = p_full + 2;          // [2]
  uint64_t* mma_done = pv_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int q0 = blockIdx.x * kBQ;
  const int n_kv = (n_tok + kBKV - 1) / kBKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_O = tmem + 256;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, S::kQBytes);
      tma_load_3d(sQ, &tmQ, q_full, 0, q0, bh);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        if (!mbar_wait(&kv_empty[stage], phase ^ 1)) {
          atomicOr(status, DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[stage], S::kKBytes + S::kVBytes);
        tma_load_3d(sK + stage * S::kKBytes, &tmK, &kv_full[stage], 0, j * kBKV, bh);
        tma_load_3d(sV + stage * S::kVBytes, &tmV, &kv_full[stage], j * kBKV, 0, bh);
        tma_load_3d(sV + stage * S::kVBytes + S::kVBlock, &tmV, &kv_full[stage], j * kBKV + 64, 0, bh);
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      mbar_wait(q_full, 0);
      const int pending = issued < kStages ? issued : kStages;
      for (int i = 0; i < pending; ++i) {
        if (--stage < 0) {
          stage = kStages - 1;
          phase ^= 1;
        }
        mbar_wait(&kv_full[stage], phase);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16<T, kBQ, kBKV>();
      constexpr uint32_t idesc_o = idesc_f16<T, kBQ, HD>();
      bool ok = mbar_wait(q_full, 0);
      const uint32_t aq = smem_u32(sQ);
      for (int j = 0; ok && j <= n_kv && !*abort_flag; ++j) {
        if (j < n_kv) {
          const int stage = j % kStages;
          if (!mbar_wait(&kv_full[stage], (j / kStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ak = smem_u32(sK + stage * S::kKBytes);
          const uint32_t d = tmem + (j & 1) * kBKV;
#pragma unroll
          for (int k = 0; k < HD / 16; ++k)
            umma_f16_ss(d, smem_desc_kmajor<kQKRow>(aq + k * 32), smem_desc_kmajor<kQKRow>(ak + k * 32), idesc_s,
                        k != 0);
          umma_commit(&s_full[j & 1]);
        }
        if (j >= 1) {
          const int jp = j - 1;
          if (!mbar_wait(&p_full[jp & 1], (jp >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int stage = jp % kStages;
          const uint32_t ap = smem_u32(sP + (jp & 1) * S::kPBytes);
          const uint32_t av = smem_u32(sV + stage * S::kVBytes);
#pragma unroll
          for (int k = 0; k < kBKV / 16; ++k) {
            const uint32_t off = (k & 3) * 32;
            umma_f16_ss(tmem_O, smem_desc_kmajor<128>(ap + (k >> 2) * S::kPBlock + off),
                        smem_desc_kmajor<128>(av + (k >> 2) * S::kVBlock + off), idesc_o, (jp | k) != 0);
          }
          umma_commit(&kv_empty[stage]);
          umma_commit(&pv_done[jp & 1]);
        }
      }
      if (!ok) {
        atomicOr(status, DEV_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(mma_done);
      mbar_wait(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + output
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;          // row in tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const bool w_ok = mbar_wait(&s_full[j & 1], (j >> 1) & 1);
      // tcgen05.ld/st are warp-collective: every decision that guards them is warp-uniform.
      if (__any_sync(0xffffffffu, !w_ok || *abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kBKV];
#pragma unroll
      for (int c = 0; c < kBKV / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_off + (j & 1) * kBKV + c * 32, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(u[i]) * scale_log2;
      }
      const int kvalid = n_tok - j * kBKV;
      if (kvalid < kBKV) {
#pragma unroll
        for (int i = 0; i < kBKV; ++i)
          if (i >= kvalid) s[i] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int i = 1; i < kBKV; ++i) mx = fmaxf(mx, s[i]);
      if (j == 0) m = mx;
      // Move the running max of the whole warp's rows when any of them grew by
      // more than 2^8: O and l are rescaled by 2^(m_old - m_new) (1 for rows
      // whose max did not grow).
      if (__any_sync(0xffffffffu, j > 0 && mx > m + 8.0f)) {
        const float m_new = fmaxf(m, mx);
        const float corr = exp2f(m - m_new);
        const int jp = j - 1;
        if (!mbar_wait(&pv_done[jp & 1], (jp >> 1) & 1)) ok = false;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(tmem_O + lane_off + c * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * corr);
          tmem_st32(tmem_O + lane_off + c * 32, u);
        }
        tmem_wait_st();
        l *= corr;
        m = m_new;
      }
      // P_j may overwrite its buffer only after PV_{j-2} has read it.
      if (j >= 2) {
        const int jq = j - 2;
        if (!mbar_wait(&pv_done[jq & 1], (jq >> 1) & 1)) ok = false;
      }
      uint8_t* pb = sP + (j & 1) * S::kPBytes + r * 128;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kBKV / 8; ++c) {
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          p[i] = exp2f(s[c * 8 + i] - m);
          rs += p[i];
        }
        uint4 w;
        w.x = pack2<T>(p[0], p[1]);
        w.y = pack2<T>(p[2], p[3]);
        w.z = pack2<T>(p[4], p[5]);
        w.w = pack2<T>(p[6], p[7]);
        const int blk = c >> 3, ch = c & 7;
        *reinterpret_cast<uint4*>(pb + blk * S::kPBlock + ((ch ^ (r & 7)) << 4)) = w;
      }
      l += rs;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
      if (__any_sync(0xffffffffu, !ok)) break;
    }
    if (ok) {
      const int jl = n_kv - 1;
      ok = mbar_wait(&pv_done[jl & 1], (jl >> 1) & 1);
    }
    if (__any_sync(0xffffffffu, !ok)) {
      if (lane == 0) atomicOr(status, DEV_TIMEOUT);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      const int row = q0 + r;
      const float inv = 1.0f / l;
      const int b = bh / n_head, head = bh - (bh / n_head) * n_head;
      T* op = out + ((size_t)b * n_tok + row) * (size_t)(n_head * HD) + head * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem_O + lane_off + c * 32, u);
        tmem_wait_ld();
        if (row < n_tok) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack2<T>(__uint_as_float(u[8 * i + 0]) * inv, __uint_as_float(u[8 * i + 1]) * inv);
            w.y = pack2<T>(__uint_as_float(u[8 * i + 2]) * inv, __uint_as_float(u[8 * i + 3]) * inv);
            w.z = pack2<T>(__uint_as_float(u[8 * i + 4]) * inv, __uint_as_float(u[8 * i + 5]) * inv);
            w.w = pack2<T>(__uint_as_float(u[8 * i + 6]) * inv, __uint_as_float(u[8 * i + 7]) * inv);
            reinterpret_cast<uint4*>(op + c * 32)[i] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T, int HD>
cudaError_t launch_t(const void* q, const void* k, const void* vt, void* out, int batch, int n_head, int n_tok,
                     int ldv, float scale, int* status, cudaStream_t s) {
  using S = AttnSmem<HD>;
  const uint64_t BH = (uint64_t)batch * n_head;
  CUtensorMap tq, tk, tv;
  cudaError_t e = make_tmap_3d(&tq, q, 2, HD, n_tok, BH, (uint64_t)HD * 2, (uint64_t)n_tok * HD * 2, HD, kBQ, 1);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d(&tk, k, 2, HD, n_tok, BH, (uint64_t)HD * 2, (uint64_t)n_tok * HD * 2, HD, kBKV, 1);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d(&tv, vt, 2, n_tok, HD, BH, (uint64_t)ldv * 2, (uint64_t)ldv * HD * 2, 64, HD, 1);
  if (e != cudaSuccess) return e;
  auto kern = attn_tc_kernel<T, HD>;
  static bool configured = false;
  if (!configured) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid((n_tok + kBQ - 1) / kBQ, (unsigned)BH);
  kern<<<grid, kThreads, S::kBytes, s>>>(tq, tk, tv, (T*)out, n_head, n_tok, scale * 1.4426950408889634f, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t attention_tc(int dtype, const void* q, const void* k, const void* vt, void* out, int batch, int n_head,
                         int n_tok, int head_dim, int ldv, float scale, int* status, cudaStream_t s, int num_sms) {
  (void)num_sms;
  if (dtype == DTYPE_BF16) {
    if (head_dim == 64) return launch_t<__nv_bfloat16, 64>(q, k, vt, out, batch, n_head, n_tok, ldv, scale, status, s);
    if (head_dim == 32) return launch_t<__nv_bfloat16, 32>(q, k, vt, out, batch, n_head, n_tok, ldv, scale, status, s);
  } else if (dtype == DTYPE_F16) {
    if (head_dim == 64) return launch_t<__half, 64>(q, k, vt, out, batch, n_head, n_tok, ldv, scale, status, s);
    if (head_dim == 32) return launch_t<__half, 32>(q, k, vt, out, batch, n_head, n_tok, ldv, scale, status, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace jepa
