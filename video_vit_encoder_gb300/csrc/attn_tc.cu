// Tensor-core attention for sm_103a, softmax(scale q k^T) v per (clip, head).
//
// A work unit is two 128-row query tiles (Q0, Q1) of one (clip, head); keys
// and values stream in tiles of 128 through a 4-deep TMA ring shared by both
// query tiles.  Two launch forms: for up to 16 key tiles the CTAs are
// persistent (one per SM, taking units in turn, the ring running on across
// units and Q double-buffered, so one unit's last key tiles overlap the next
// unit's Q load and first score products; a unit's output is staged in its
// own Q buffer and leaves by TMA tile stores, taken at the next unit's first
// key tile); for longer ones each CTA takes one unit on a grid over the
// units.  For query tile t and key tile j:
//   S_t = Q_t K_j^T     tcgen05.mma (both operands in shared memory) into the
//                       tile's TMEM score buffer (fp32, 128 lanes x 128 columns);
//   softmax warpgroup t (one thread per query row) reads its row of S_t into
//   registers in one TMEM round trip and releases the buffer at once, so the
//   scores of key tile j+1 are computed while it works; it takes the row max,
//   writes P_t = 2^((S_t - m) scale log2e) as 16-bit pairs into the tile's
//   TMEM P buffer and accumulates the row sum l in fp32;
//   O_t += P_t V_j      tcgen05.mma with A = P_t read from tensor memory and
//                       B = V_j from shared memory, into the TMEM accumulator.
// P never touches shared memory, whose bandwidth the operand reads of the two
// products and the TMA writes already share.  The running max m is moved (O_t
// and l rescaled through TMEM) only when a row's max grows by more than 2^8 in
// the exponent; m, l and O stay consistent, so O / l is exact up to rounding.
// V arrives transposed ([hd, keys], keys contiguous): both B operands are
// K-major.
//
// Warp roles (384 threads, three warpgroups): warp 0 TMA producer, warp 1
// MMA issuer of Q0 and tensor-memory owner, warp 2 MMA issuer of Q1, warp 3
// idle; warps 4-7 softmax of Q0, warps 8-11 softmax of Q1 (warp w owns TMEM
// lanes / query rows 32*(w%4) .. +31 of its tile).  One issuer per query tile
// keeps each issuer's chain of waits and issues short: every SM
// sub-partition also runs two softmax warps.  The first warpgroup hands
// registers to the softmax warpgroups (setmaxnreg), which hold a whole
// 128-score row each.
#include "internal.h"

namespace jepa {

namespace {

constexpr int kBQ = 128;     // query rows per tile (two tiles per unit)
constexpr int kBKV = 128;    // keys per tile
constexpr int kStages = 4;   // K/V ring depth
constexpr int kThreads = 384;
// Register split after launch (168 per thread at launch): 128 x 72 + 256 x 216
// = 384 x 168, and per SM sub-partition one warp of each warpgroup.
constexpr int kRegsControl = 72;
constexpr int kRegsSoftmax = 216;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * 168, "register split above the launch total");
// TMEM columns: S_t [128 t, 128 t + 128), P_t [256 + 64 t, +64) (128 16-bit
// values per lane), O_t [384 + 64 t, +HD).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColP = 256, kColO = 384;
template <int HD, int QBUF>
struct AttnSmem {
  static constexpr uint32_t kQBytes = kBQ * HD * 2;    // one query tile
  static constexpr uint32_t kKBytes = kBKV * HD * 2;
  static constexpr uint32_t kVBytes = HD * kBKV * 2;   // two 64-key blocks of HD rows x 128 B
  static constexpr uint32_t kVBlock = HD * 128;
  static constexpr uint32_t kOffK = 2 * QBUF * kQBytes;   // QBUF buffers of the two query tiles
  static constexpr uint32_t kOffV = kOffK + kStages * kKBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kVBytes;
  static constexpr size_t kBytes = 1024 + kOffBar + 512;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Two fp32 values in one 64-bit register pair, for the packed f32x2 pipes.
__device__ __forceinline__ uint64_t pk2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Row max of one S tile held in registers (s[c][i] = column 32 c + i);
// columns >= kvalid are ignored when MASK.
template <bool MASK>
__device__ __forceinline__ float row_max(const uint32_t (&s)[kBKV / 32][32], int kvalid) {
  float mxs[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent chains
#pragma unroll
  for (int c = 0; c < kBKV / 32; ++c) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float a = __uint_as_float(s[c][i]), b = __uint_as_float(s[c][i + 1]);
      if (MASK) {
        a = (c * 32 + i < kvalid) ? a : -INFINITY;
        b = (c * 32 + i + 1 < kvalid) ? b : -INFINITY;
      }
      mxs[(i >> 1) & 3] = max3(mxs[(i >> 1) & 3], a, b);
    }
  }
  return fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3]));
}

// P = 2^(S scale_log2 + neg_m) for one S row held in registers, as 16-bit
// pairs (column q holds keys 2q, 2q+1) into the thread's TMEM lane from tP;
// returns the row sum of P (fp32); columns >= kvalid get P = 0 when MASK.
template <typename T, bool MASK>
__device__ __forceinline__ float exp_to_tmem(const uint32_t (&s)[kBKV / 32][32], int kvalid, float scale_log2,
                                             float neg_m, uint32_t tP) {
  const uint64_t sc2 = pk2(__float_as_uint(scale_log2), __float_as_uint(scale_log2));
  const uint64_t nm2 = pk2(__float_as_uint(neg_m), __float_as_uint(neg_m));
  uint64_t rs2[4] = {0, 0, 0, 0};  // four independent (0.f, 0.f) partial sums
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t w[32];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * h + cc;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const uint64_t x2 = fma2(pk2(s[c][i], s[c][i + 1]), sc2, nm2);
        float x0, x1;
        upk2(x2, x0, x1);
        if (MASK) {
          const int col = c * 32 + i;
          x0 = col < kvalid ? x0 : -INFINITY;
          x1 = col + 1 < kvalid ? x1 : -INFINITY;
        }
        const float p0 = ex2(x0), p1 = ex2(x1);
        rs2[(i >> 1) & 3] = add2(rs2[(i >> 1) & 3], pk2(__float_as_uint(p0), __float_as_uint(p1)));
        w[cc * 16 + i / 2] = pack2<T>(p0, p1);
      }
    }
    tmem_st32(tP + h * 32, w);
  }
  float a, b;
  upk2(add2(add2(rs2[0], rs2[1]), add2(rs2[2], rs2[3])), a, b);
  return a + b;
}

// This warp's 32 rows of O_t (HD fp32 columns from tO) scaled by inv and
// rounded to T, into shared memory at stage: 32 rows of 2 HD bytes laid out
// as a TMA tile with the swizzle of that row width (the 16-byte chunk c of
// row r at chunk c ^ (bits 7.. of the byte offset)), for one tile store.
template <typename T, int HD>
__device__ __forceinline__ void stage_o_rows(uint32_t tO, float inv, uint8_t* stage, int lane) {
  constexpr uint32_t kRow = HD * 2;          // bytes per row: 128 or 64
  constexpr uint32_t kMask = kRow / 16 - 1;  // 7 (128-byte swizzle) or 3 (64-byte)
#pragma unroll
  for (int c = 0; c < HD / 8; ++c) {  // 8 columns (one 16-byte chunk) at a time
    uint32_t u[8];
    tmem_ld8(tO + c * 8, u);
    tmem_wait_ld();
    uint4 w;
    w.x = pack2<T>(__uint_as_float(u[0]) * inv, __uint_as_float(u[1]) * inv);
    w.y = pack2<T>(__uint_as_float(u[2]) * inv, __uint_as_float(u[3]) * inv);
    w.z = pack2<T>(__uint_as_float(u[4]) * inv, __uint_as_float(u[5]) * inv);
    w.w = pack2<T>(__uint_as_float(u[6]) * inv, __uint_as_float(u[7]) * inv);
    const uint32_t a = (uint32_t)lane * kRow + (uint32_t)c * 16;
    *reinterpret_cast<uint4*>(stage + (a ^ (((a >> 7) & kMask) << 4))) = w;
  }
}

// Stages this warp's 32 rows of O_t (normalised by 1 / l_fin) at stage and
// has lane 0 store them as one TMA tile: rows row0.., columns head HD.. of
// clip b of the output.
template <typename T, int HD>
__device__ __forceinline__ void store_o_rows(const CUtensorMap* tmO, uint32_t tO, float l_fin, uint8_t* stage,
                                             int lane, int head, int row0, int b) {
  stage_o_rows<T, HD>(tO, 1.0f / l_fin, stage, lane);
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(tmO, stage, head * HD, row0, b);
    bulk_commit_group();
  }
}

// One unit (two query tiles of one (clip, head)) per CTA, on a grid over
// the units: the hardware hands each SM its next CTA as one finishes.
template <typename T, int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, T* __restrict__ out, int n_head, int n_tok,
                   float scale_log2, int* status) {
  using S = AttnSmem<HD, 1>;
  constexpr int kQKRow = HD * 2;  // bytes per Q/K row = swizzle width (128 or 64)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + S::kOffK;
  uint8_t* sV = smem + S::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;  // [2] per query tile: S_t computed
  uint64_t* s_free = s_full + 2;          // [2] S_t read into registers
  uint64_t* p_full = s_free + 2;          // [2] P_t written (and O_t rescaled)
  uint64_t* pv_done = p_full + 2;         // [2] O_t += P_t V done
  uint64_t* mma_done = pv_done + 2;      // [2] per issuer
  uint64_t* exp_tok = mma_done + 2;      // [2][4] exponential phase of tile t done, per TMEM quarter
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(exp_tok + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int q0 = blockIdx.x * (2 * kBQ);
  const int n_kv = (n_tok + kBKV - 1) / kBKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 2);  // both query tiles' issuers
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    for (int i = 0; i < 8; ++i) mbar_init(&exp_tok[i], 32);
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

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, 2 * S::kQBytes);
        tma_load_3d(sQ, &tmQ, q_full, 0, q0, bh);
        tma_load_3d(sQ + S::kQBytes, &tmQ, q_full, 0, q0 + kBQ, bh);
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
        // the CTA does not exit with copies in flight
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
    } else if (warp == 1 || warp == 2) {
      // ------------------------------------------------------------ MMA issuer of query tile t
      // The whole warp walks the schedule (waits are warp-uniform); one
      // elected lane issues each MMA and commit.
      const int t = warp - 1;
      constexpr uint32_t idesc_s = idesc_f16<T, kBQ, kBKV>();
      constexpr uint32_t idesc_o = idesc_f16<T, kBQ, HD>();
      const uint64_t dq = smem_desc_kmajor<kQKRow>(smem_u32(sQ + t * S::kQBytes));
      const uint32_t dS = tmem + kColS + t * kBKV, dP = tmem + kColP + t * 64, dO = tmem + kColO + t * 64;
      bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0));
      // S_t of key tile j into the tile's score buffer, once the tile's
      // softmax has read the previous scores out of it.
      auto issue_s = [&](int j) -> bool {
        const int stage = j % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[stage], (j / kStages) & 1))) return false;
        if (j >= 1 && !__all_sync(0xffffffffu, mbar_wait(&s_free[t], (j - 1) & 1))) return false;
        tc_fence_after();
        const uint64_t dk = smem_desc_kmajor<kQKRow>(smem_u32(sK + stage * S::kKBytes));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)  // +32 bytes along K = +2 in the descriptor's address field
          umma_f16_ss_warp(dS, dq + kk * 2, dk + kk * 2, idesc_s, kk != 0);
        umma_commit_warp(&s_full[t]);
        return true;
      };
      // O_t += P_t V_j, P_t from tensor memory (8 columns per 16 keys).
      auto issue_pv = [&](int j) -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait(&p_full[t], j & 1))) return false;
        tc_fence_after();
        const int stage = j % kStages;
        const uint64_t dv = smem_desc_kmajor<128>(smem_u32(sV + stage * S::kVBytes));
#pragma unroll
        for (int kk = 0; kk < kBKV / 16; ++kk)
          umma_f16_ts_warp(dO, dP + kk * 8, dv + (kk >> 2) * (S::kVBlock >> 4) + (kk & 3) * 2, idesc_o,
                           (j | kk) != 0);
        umma_commit_warp(&pv_done[t]);
        umma_commit_warp(&kv_empty[stage]);  // this tile is done with K_j and V_j
        return true;
      };
      // Order: S_0, then per key tile j: S_{j+1}, PV_j, so the next scores
      // are queued before PV_j waits for the softmax.
      ok = ok && issue_s(0);
      for (int j = 0; ok && j < n_kv; ++j) {
        if (__any_sync(0xffffffffu, *abort_flag)) break;
        if (j + 1 < n_kv) ok = issue_s(j + 1);
        ok = ok && issue_pv(j);
      }
      if (!ok && lane == 0) {
        atomicOr(status, DEV_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit_warp(&mma_done[t]);
      mbar_wait(&mma_done[t], 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax + output (tile t)
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS + t * kBKV;
    const uint32_t tP = tmem + lane_off + kColP + t * 64;
    const uint32_t tO = tmem + lane_off + kColO + t * 64;
    float m = -INFINITY;  // running max of the raw scores
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const bool w_ok = mbar_wait(&s_full[t], j & 1);
      // tcgen05.ld/st are warp-collective: every decision that guards them is warp-uniform.
      if (__any_sync(0xffffffffu, !w_ok || *abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the whole score row into registers in one TMEM round trip; the
      // buffer is released at once so the next scores can be computed into it
      uint32_t sv[kBKV / 32][32];
#pragma unroll
      for (int c = 0; c < kBKV / 32; ++c) tmem_ld32(tS + c * 32, sv[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_free[t]);
      const int kvalid = n_tok - j * kBKV;   // keys of this tile inside the sequence
      const bool full_tile = kvalid >= kBKV;
      const float mx = full_tile ? row_max<false>(sv, kvalid) : row_max<true>(sv, kvalid);
      if (j == 0) m = mx;
      // O_t is stable and P_t's buffer free once PV_t of the previous key tile is done.
      if (j >= 1 && !mbar_wait(&pv_done[t], (j - 1) & 1)) ok = false;
      tc_fence_after();
      // Move the running max of the warp's rows when any grew by more than 2^8
      // (in the exponent): O_t and l are rescaled by 2^((m_old - m_new) scale log2e).
      if (__any_sync(0xffffffffu, j > 0 && (mx - m) * scale_log2 > 8.0f)) {
        const float m_new = fmaxf(m, mx);
        const float corr = ex2((m - m_new) * scale_log2);
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(tO + c * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * corr);
          tmem_st32(tO + c * 32, u);
        }
        l *= corr;
        m = m_new;
      }
      // The two tiles' warps on one SM sub-partition take turns at the
      // exponentials (Q0 of key tile j, Q1 of j, Q0 of j+1, ...), so one
      // tile's TMEM load and row max overlap the other's special-function
      // work instead of both contending for it at once.
      if (t == 1 || j >= 1) {
        const bool tok_ok = mbar_wait(&exp_tok[(1 - t) * 4 + quarter], (t == 0 ? j - 1 : j) & 1);
        if (!tok_ok) ok = false;
      }
      // P = 2^((S - m) scale log2e), 16-bit, into tensor memory
      const float rs = full_tile ? exp_to_tmem<T, false>(sv, kvalid, scale_log2, -m * scale_log2, tP)
                                 : exp_to_tmem<T, true>(sv, kvalid, scale_log2, -m * scale_log2, tP);
      l += rs;
      mbar_arrive(&exp_tok[t * 4 + quarter]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[t]);
      if (__any_sync(0xffffffffu, !ok)) break;
    }
    if (ok) ok = mbar_wait(&pv_done[t], (n_kv - 1) & 1);
    if (__any_sync(0xffffffffu, !ok)) {
      if (lane == 0) atomicOr(status, DEV_TIMEOUT);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      const int row = q0 + t * kBQ + quarter * 32 + lane;
      const float inv = 1.0f / l;
      const int b = bh / n_head, head = bh - (bh / n_head) * n_head;
      T* op = out + ((size_t)b * n_tok + row) * (size_t)(n_head * HD) + head * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tO + c * 32, u);
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

// The same computation with persistent CTAs (described at the top of the
// file): one per SM, taking units in turn.
template <typename T, int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                              int n_head, int n_tok, int n_units, float scale_log2, int* status) {
  using S = AttnSmem<HD, 2>;
  constexpr int kQKRow = HD * 2;  // bytes per Q/K row = swizzle width (128 or 64)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + S::kOffK;
  uint8_t* sV = smem + S::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint64_t* q_full = bars;                 // [2] Q buffer b loaded
  uint64_t* q_empty = bars + 2;            // [2] Q buffer b read by both tiles' score products
  uint64_t* kv_full = bars + 4;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;  // [2] per query tile: S_t computed
  uint64_t* s_free = s_full + 2;          // [2] S_t read into registers
  uint64_t* p_full = s_free + 2;          // [2] P_t written (and O_t rescaled)
  uint64_t* pv_done = p_full + 2;         // [2] O_t += P_t V done
  uint64_t* mma_done = pv_done + 2;      // [2] per issuer
  uint64_t* exp_tok = mma_done + 2;      // [2][4] exponential phase of tile t done, per TMEM quarter
  uint64_t* o_staged = exp_tok + 8;      // [2] Q buffer b's output staging read by its tile stores
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_staged + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work units: (clip x head, pair of query tiles), unit u = bh * n_qp + qp.
  // The CTA is persistent: it takes units blockIdx.x, + gridDim.x, ...; the
  // K/V ring, the score / P / PV barriers and the exponential tokens run on
  // one CTA-wide key-tile counter g (unit k of the CTA, key tile j: g =
  // k n_kv + j), so one unit's last key tiles overlap the next unit's Q load
  // and first score products.
  const int n_kv = (n_tok + kBKV - 1) / kBKV;
  const int n_qp = (n_tok + 2 * kBQ - 1) / (2 * kBQ);
  const int n_my = n_units > (int)blockIdx.x ? (n_units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int n_g = n_my * n_kv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 2);  // both query tiles' issuers
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 2);  // both query tiles' issuers
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    for (int i = 0; i < 8; ++i) mbar_init(&exp_tok[i], 32);
    mbar_init(&o_staged[0], 8);  // lane 0 of each softmax warp
    mbar_init(&o_staged[1], 8);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;    // K/V stage loads
        int q_issued = 0;  // Q loads (one per unit)
        bool ok = true;
        for (int k = 0; ok && k < n_my; ++k) {
          const int u = (int)blockIdx.x + k * (int)gridDim.x;
          const int ubh = u / n_qp, uq0 = (u - ubh * n_qp) * 2 * kBQ;
          const int qb = k & 1;
          // Q buffer qb was last read by the score products of unit k - 2,
          // then held unit k - 2's output on its way to global memory
          if (k >= 2 && (!mbar_wait(&q_empty[qb], ((k >> 1) - 1) & 1) ||
                         !mbar_wait(&o_staged[qb], ((k >> 1) - 1) & 1))) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&q_full[qb], 2 * S::kQBytes);
          tma_load_3d(sQ + qb * 2 * S::kQBytes, &tmQ, &q_full[qb], 0, uq0, ubh);
          tma_load_3d(sQ + qb * 2 * S::kQBytes + S::kQBytes, &tmQ, &q_full[qb], 0, uq0 + kBQ, ubh);
          ++q_issued;
          for (int j = 0; j < n_kv; ++j) {
            if (*abort_flag || !mbar_wait(&kv_empty[stage], phase ^ 1)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&kv_full[stage], S::kKBytes + S::kVBytes);
            tma_load_3d(sK + stage * S::kKBytes, &tmK, &kv_full[stage], 0, j * kBKV, ubh);
            tma_load_3d(sV + stage * S::kVBytes, &tmV, &kv_full[stage], j * kBKV, 0, ubh);
            tma_load_3d(sV + stage * S::kVBytes + S::kVBlock, &tmV, &kv_full[stage], j * kBKV + 64, 0, ubh);
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        if (!ok) {
          atomicOr(status, DEV_TIMEOUT);
          *abort_flag = 1;
        }
        // The CTA does not exit with copies in flight: the last (up to two) Q
        // loads and the last min(issued, kStages) K/V stages have landed.
        for (int kk = q_issued - 1; kk >= 0 && kk >= q_issued - 2; --kk) mbar_wait(&q_full[kk & 1], (kk >> 1) & 1);
        const int pending = issued < kStages ? issued : kStages;
        for (int i = 0; i < pending; ++i) {
          if (--stage < 0) {
            stage = kStages - 1;
            phase ^= 1;
          }
          mbar_wait(&kv_full[stage], phase);
        }
      }
    } else if (warp == 1 || warp == 2) {
      // ------------------------------------------------------------ MMA issuer of query tile t
      // The whole warp walks the schedule (waits are warp-uniform); one
      // elected lane issues each MMA and commit.
      const int t = warp - 1;
      constexpr uint32_t idesc_s = idesc_f16<T, kBQ, kBKV>();
      constexpr uint32_t idesc_o = idesc_f16<T, kBQ, HD>();
      const uint32_t dS = tmem + kColS + t * kBKV, dP = tmem + kColP + t * 64, dO = tmem + kColO + t * 64;
      bool ok = true;
      // S_t of the next CTA key tile (unit ks, key tile js, ring stage
      // st_s) into the tile's score buffer, once the tile's softmax has read
      // the previous scores out of it (and, for a unit's first key tile, once
      // its Q has landed).  Counters advance without divisions.
      int gs = 0, ks = 0, js = 0, st_s = 0;
      uint32_t ph_s = 0;
      auto issue_s = [&]() -> bool {
        if (js == 0 && !__all_sync(0xffffffffu, mbar_wait(&q_full[ks & 1], (ks >> 1) & 1))) return false;
        if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[st_s], ph_s))) return false;
        if (gs >= 1 && !__all_sync(0xffffffffu, mbar_wait(&s_free[t], (gs - 1) & 1))) return false;
        tc_fence_after();
        const uint64_t dq = smem_desc_kmajor<kQKRow>(smem_u32(sQ + (ks & 1) * 2 * S::kQBytes + t * S::kQBytes));
        const uint64_t dk = smem_desc_kmajor<kQKRow>(smem_u32(sK + st_s * S::kKBytes));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)  // +32 bytes along K = +2 in the descriptor's address field
          umma_f16_ss_warp(dS, dq + kk * 2, dk + kk * 2, idesc_s, kk != 0);
        umma_commit_warp(&s_full[t]);
        if (js == n_kv - 1) umma_commit_warp(&q_empty[ks & 1]);  // this tile is done with the unit's Q
        ++gs;
        if (++js == n_kv) {
          js = 0;
          ++ks;
        }
        if (++st_s == kStages) {
          st_s = 0;
          ph_s ^= 1;
        }
        return true;
      };
      // O_t += P_t V of the next CTA key tile, P_t from tensor memory (8
      // columns per 16 keys); a unit's first key tile starts O_t afresh.  The
      // softmax signals P only after it has read the previous unit's O_t.
      int gp = 0, jp = 0, st_p = 0;
      auto issue_pv = [&]() -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait(&p_full[t], gp & 1))) return false;
        tc_fence_after();
        const uint64_t dv = smem_desc_kmajor<128>(smem_u32(sV + st_p * S::kVBytes));
#pragma unroll
        for (int kk = 0; kk < kBKV / 16; ++kk)
          umma_f16_ts_warp(dO, dP + kk * 8, dv + (kk >> 2) * (S::kVBlock >> 4) + (kk & 3) * 2, idesc_o,
                           (jp | kk) != 0);
        umma_commit_warp(&pv_done[t]);
        umma_commit_warp(&kv_empty[st_p]);  // this tile is done with this key tile's K and V
        ++gp;
        if (++jp == n_kv) jp = 0;
        if (++st_p == kStages) st_p = 0;
        return true;
      };
      // Order: S_0, then per key tile g: S_{g+1}, PV_g, so the next scores
      // (possibly the next unit's first) are queued before PV_g waits for the softmax.
      if (n_g > 0) ok = issue_s();
      for (int g = 0; ok && g < n_g; ++g) {
        if (__any_sync(0xffffffffu, *abort_flag)) break;
        if (g + 1 < n_g) ok = issue_s();
        ok = ok && issue_pv();
      }
      if (!ok && lane == 0) {
        atomicOr(status, DEV_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit_warp(&mma_done[t]);
      mbar_wait(&mma_done[t], 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax + output (tile t)
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS + t * kBKV;
    const uint32_t tP = tmem + lane_off + kColP + t * 64;
    const uint32_t tO = tmem + lane_off + kColO + t * 64;
    // A unit's output leaves through its own Q buffer (tile t's half, this
    // warp's 32 rows), no longer read once the unit's last P V is done: the
    // warp stages its rows there and lane 0 stores them with one TMA tile
    // store, so the next unit's first key tile is not held up by global
    // stores.  The previous unit's output is taken at the next unit's first
    // key tile, after that tile's exponentials.
    bool ok = true;
    bool staged = false;  // the previous unit's rows are staged and their store not yet known to have read them
    float l_prev = 0.f;
    int g = 0;  // the CTA's key-tile counter over its units
    for (int k = 0; ok && k < n_my; ++k) {
      float m = -INFINITY;  // running max of the raw scores
      float l = 0.f;
      for (int j = 0; j < n_kv; ++j, ++g) {
        const bool w_ok = mbar_wait(&s_full[t], g & 1);
        // tcgen05.ld/st are warp-collective: every decision that guards them is warp-uniform.
        if (__any_sync(0xffffffffu, !w_ok || *abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the whole score row into registers in one TMEM round trip; the
        // buffer is released at once so the next scores can be computed into it
        uint32_t sv[kBKV / 32][32];
#pragma unroll
        for (int c = 0; c < kBKV / 32; ++c) tmem_ld32(tS + c * 32, sv[c]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&s_free[t]);
        const int kvalid = n_tok - j * kBKV;   // keys of this tile inside the sequence
        const bool full_tile = kvalid >= kBKV;
        const float mx = full_tile ? row_max<false>(sv, kvalid) : row_max<true>(sv, kvalid);
        if (j == 0) m = mx;
        // O_t is stable and P_t's buffer free once PV_t of the previous key
        // tile is done (at a unit's first key tile: the previous unit's last).
        if (g >= 1 && !mbar_wait(&pv_done[t], (g - 1) & 1)) ok = false;
        tc_fence_after();
        // Move the running max of the warp's rows when any grew by more than 2^8
        // (in the exponent): O_t and l are rescaled by 2^((m_old - m_new) scale log2e).
        if (__any_sync(0xffffffffu, j > 0 && (mx - m) * scale_log2 > 8.0f)) {
          const float m_new = fmaxf(m, mx);
          const float corr = ex2((m - m_new) * scale_log2);
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t uo[32];
            tmem_ld32(tO + c * 32, uo);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) uo[i] = __float_as_uint(__uint_as_float(uo[i]) * corr);
            tmem_st32(tO + c * 32, uo);
          }
          l *= corr;
          m = m_new;
        }
        // The two tiles' warps on one SM sub-partition take turns at the
        // exponentials (Q0 of key tile g, Q1 of g, Q0 of g+1, ...), so one
        // tile's TMEM load and row max overlap the other's special-function
        // work instead of both contending for it at once.
        if (t == 1 || g >= 1) {
          const bool tok_ok = mbar_wait(&exp_tok[(1 - t) * 4 + quarter], (t == 0 ? g - 1 : g) & 1);
          if (!tok_ok) ok = false;
        }
        // P = 2^((S - m) scale log2e), 16-bit, into tensor memory
        const float rs = full_tile ? exp_to_tmem<T, false>(sv, kvalid, scale_log2, -m * scale_log2, tP)
                                   : exp_to_tmem<T, true>(sv, kvalid, scale_log2, -m * scale_log2, tP);
        l += rs;
        mbar_arrive(&exp_tok[t * 4 + quarter]);
        // The previous unit's output, read before this unit's first P V
        // replaces O_t (that P V waits for p_full) and after this tile's
        // exponentials, when the score registers are free.
        if (j == 0 && k >= 1) {
          const int pu = (int)blockIdx.x + (k - 1) * (int)gridDim.x;
          const int pbh = pu / n_qp, pq0 = (pu - pbh * n_qp) * 2 * kBQ;
          store_o_rows<T, HD>(&tmO, tO, l_prev,
                              sQ + ((k - 1) & 1) * 2 * S::kQBytes + t * S::kQBytes + quarter * 32 * kQKRow, lane,
                              pbh % n_head, pq0 + t * kBQ + quarter * 32, pbh / n_head);
          staged = true;
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
        // The staging of the previous unit's rows is released to the
        // producer (which reloads that Q buffer two units on) a few key
        // tiles later, when the store has long read it.
        if (staged && (j == 2 || j == n_kv - 1)) {
          if (lane == 0) {
            bulk_wait_read_all();
            mbar_arrive(&o_staged[(k - 1) & 1]);
          }
          staged = false;
        }
        if (__any_sync(0xffffffffu, !ok)) break;
      }
      l_prev = l;
    }
    // the last unit's output, once its last P V is done
    if (ok && n_my > 0) ok = mbar_wait(&pv_done[t], (g - 1) & 1);
    if (__any_sync(0xffffffffu, !ok)) {
      if (lane == 0) atomicOr(status, DEV_TIMEOUT);
      *abort_flag = 1;
    } else if (n_my > 0) {
      tc_fence_after();
      const int pu = (int)blockIdx.x + (n_my - 1) * (int)gridDim.x;
      const int pbh = pu / n_qp, pq0 = (pu - pbh * n_qp) * 2 * kBQ;
      store_o_rows<T, HD>(&tmO, tO, l_prev,
                          sQ + ((n_my - 1) & 1) * 2 * S::kQBytes + t * S::kQBytes + quarter * 32 * kQKRow, lane,
                          pbh % n_head, pq0 + t * kBQ + quarter * 32, pbh / n_head);
    }
    // the CTA does not exit with tile stores in flight
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Sequences of at most this many key tiles run on the persistent kernel:
// there each unit is short, and overlapping its start with the previous
// unit's end pays (576-token images: 1.06 -> 0.84 ms per step; 2048 tokens:
// 152.7 -> 149.9 us per ViT-L launch).  Longer units run one per CTA: the
// hardware's dynamic hand-out of CTAs balances them better than a fixed
// round-robin (8192 and 18432 tokens: 9-10 % faster).
constexpr int kPersistentMaxKeyTiles = 16;

template <typename Kern>
cudaError_t configure(Kern kern, size_t smem_bytes) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc waits until the registers it asks for are free within the
  // block's launch allocation: refuse to launch when the allocation is short.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kThreads < 128 * kRegsControl + 256 * kRegsSoftmax) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

template <typename T, int HD>
cudaError_t launch_t(const void* q, const void* k, const void* vt, void* out, int batch, int n_head, int n_tok,
                     int ldv, float scale, int* status, cudaStream_t s, int num_sms) {
  const uint64_t BH = (uint64_t)batch * n_head;
  CUtensorMap tq, tk, tv;
  cudaError_t e = make_tmap_3d(&tq, q, 2, HD, n_tok, BH, (uint64_t)HD * 2, (uint64_t)n_tok * HD * 2, HD, kBQ, 1);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d(&tk, k, 2, HD, n_tok, BH, (uint64_t)HD * 2, (uint64_t)n_tok * HD * 2, HD, kBKV, 1);
  if (e != cudaSuccess) return e;
  e = make_tmap_3d(&tv, vt, 2, n_tok, HD, BH, (uint64_t)ldv * 2, (uint64_t)ldv * HD * 2, 64, HD, 1);
  if (e != cudaSuccess) return e;
  const float scale_log2 = scale * 1.4426950408889634f;
  const int n_qp = (n_tok + 2 * kBQ - 1) / (2 * kBQ);
  const int n_kv = (n_tok + kBKV - 1) / kBKV;
  if (n_kv > kPersistentMaxKeyTiles) {
    using S = AttnSmem<HD, 1>;
    auto kern = attn_tc_kernel<T, HD>;
    static DeviceOnce setup;   // the shared-memory opt-in is per device
    e = setup.run([&](int) { return configure(kern, S::kBytes); });
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)n_qp, (unsigned)BH);
    kern<<<grid, kThreads, S::kBytes, s>>>(tq, tk, tv, (T*)out, n_head, n_tok, scale_log2, status);
    return cudaGetLastError();
  }
  using S = AttnSmem<HD, 2>;
  auto kern = attn_tc_persistent_kernel<T, HD>;
  static DeviceOnce setup;
  e = setup.run([&](int) { return configure(kern, S::kBytes); });
  if (e != cudaSuccess) return e;
  // output [batch, n_tok, n_head HD] as 32-row tiles of one head (rows past
  // n_tok fall outside the map and are not written)
  CUtensorMap to;
  e = make_tmap_3d(&to, out, 2, (uint64_t)n_head * HD, n_tok, batch, (uint64_t)n_head * HD * 2,
                   (uint64_t)n_tok * n_head * HD * 2, HD, 32, 1);
  if (e != cudaSuccess) return e;
  // persistent grid: one CTA per SM (its shared memory allows no second), each
  // taking every gridDim-th unit
  const int n_units = (int)(n_qp * BH);
  const int slots = num_sms > 0 ? num_sms : 1;
  const int grid = n_units < slots ? n_units : slots;
  kern<<<grid, kThreads, S::kBytes, s>>>(tq, tk, tv, to, n_head, n_tok, n_units, scale_log2, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t attention_tc(int dtype, const void* q, const void* k, const void* vt, void* out, int batch, int n_head,
                         int n_tok, int head_dim, int ldv, float scale, int* status, cudaStream_t s, int num_sms) {
  if (dtype == DTYPE_BF16) {
    if (head_dim == 64) return launch_t<__nv_bfloat16, 64>(q, k, vt, out, batch, n_head, n_tok, ldv, scale, status, s, num_sms);
    if (head_dim == 32) return launch_t<__nv_bfloat16, 32>(q, k, vt, out, batch, n_head, n_tok, ldv, scale, status, s, num_sms);
  } else if (dtype == DTYPE_F16) {
    if (head_dim == 64) return launch_t<__half, 64>(q, k, vt, out, batch, n_head, n_tok, ldv, scale, status, s, num_sms);
    if (head_dim == 32) return launch_t<__half, 32>(q, k, vt, out, batch, n_head, n_tok, ldv, scale, status, s, num_sms);
  }
  return cudaErrorInvalidValue;
}

}  // namespace jepa
