// Tensor-core linear layer for sm_103a: out = epilogue(A W^T + bias).
//
// A [M, K] and W [N, K] (both K contiguous, bf16 or fp16) are streamed by TMA
// into 128B-swizzled shared-memory stages; one thread issues tcgen05.mma
// (M 128 x N BN x K 16, fp32 accumulator in tensor memory); four epilogue
// warps drain the accumulator with tcgen05.ld and apply the fused epilogue.
// The kernel is persistent (one CTA per SM, static tile striding) and keeps
// two accumulators in tensor memory so the epilogue of one tile overlaps the
// main loop of the next.  The tiles of the last, partial wave are split into
// two half-width units run by different CTAs, so that wave takes about half
// a tile's time instead of a whole one.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer and
// tensor-memory owner, warps 2-9 epilogue (warp w reads TMEM lanes
// 32*(w%4) .. 32*(w%4)+31 and column half (w-2)/4 of the tile).
// With more than one row tile, CTAs run as pairs (clusters of two) issuing
// M = 256 x N = BN MMAs over both CTAs' shared memory (cta_group::2): each CTA
// loads its 128 rows of A and half of the W tile, so per SM the bytes moved
// per flop fall by a third against a single-CTA 128 x BN tile.
#include "epilogue.cuh"
#include "internal.h"

namespace jepa {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;  // 64 x 16-bit = one 128-byte swizzle row
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;   // warps 2-9

template <int BN, int STAGES, int CM>
struct GemmSmem {
  static constexpr uint32_t kABytes = kBM * kBK * 2;          // this CTA's 128 rows of A
  static constexpr uint32_t kBBytes = (BN / CM) * kBK * 2;    // this CTA's rows of W
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators; a power of two
  static constexpr uint32_t kEpiStage = 4096;  // per epilogue warp: 32 rows x 128 bytes
  static constexpr uint32_t kEpiOffset = STAGES * kStageBytes;
  static constexpr uint32_t kBarOffset = kEpiOffset + (kEpiThreads / 32) * kEpiStage;
  static constexpr size_t kBytes = 1024 /*alignment slack*/ + kBarOffset + 320;
};

// Writes the staged head rows of one warp (32 rows from row0, head `head` of
// the q (which 0) or k (which 1) section) to the head-major output: HD x 2
// bytes per token, a row's token and clip taken from its own index, so the 32
// rows may span two clips.  Rows at or past M are not written.
template <typename T, int HD>
__device__ __forceinline__ void stage_out_head(const EpiParams& ep, int which, uint8_t* stage, int row0, int head,
                                               int M, int lane) {
  constexpr int kSeg = HD * 2 / 16;        // 16-byte segments per head row
  constexpr int kRowsPer = 32 / kSeg;      // rows per warp instruction
  __syncwarp();
  T* base = reinterpret_cast<T*>(which == 0 ? ep.q : ep.k);
#pragma unroll
  for (int it = 0; it < kSeg; ++it) {
    const int r = it * kRowsPer + lane / kSeg, g = lane % kSeg;
    const int grow = row0 + r;
    const uint4 u = reinterpret_cast<const uint4*>(stage + r * 128)[g ^ (r & 7)];
    if (grow < M) {
      const int clip = grow / ep.n_tok;
      const int tok = grow - clip * ep.n_tok;
      const size_t bh = (size_t)clip * ep.n_head + head;
      reinterpret_cast<uint4*>(base + (bh * ep.n_tok + tok) * HD)[g] = u;
    }
  }
  __syncwarp();   // the buffer is reused for the next head
}

// QKV epilogue of one thread's row of a 128 x BN accumulator tile.  BN
// divides D, so the whole tile lies in the q, the k or the v section.  The
// token's RoPE factors (3 axes x d/2 angles, cos and sin) are loaded once per
// tile and shared by the tile's BN/HD heads; with HD and the layout fixed at
// compile time every axis / angle index below is a constant.
//   out[2k]   = x[2k]   cos(a_f0) - x[2k+1] sin(a_f0)
//   out[2k+1] = x[2k+1] cos(a_f1) + x[2k]   sin(a_f1)
// with f0 = f1 = k' (interleaved) or f0 = 2k' mod d/2, f1 = (2k'+1) mod d/2
// (tiled), k' the pair index within its axis segment.
//
// q and k rows leave through the warp's 4 KB staging buffer: each thread puts
// its head row there (16-byte segments XOR-swizzled by row, so neither side
// has bank conflicts), and the warp then writes whole 128-byte head rows of
// consecutive tokens, one full line per eight lanes, instead of each thread
// writing a half sector of 32 different lines.
//
// n_chunks (<= BN/64) is the number of 32-column chunks this thread covers:
// BN/64 for a whole tile, fewer for a half-width tail tile (whole heads).
template <typename T, int BN, int HD, int LAYOUT>
__device__ __forceinline__ void qkv_tile_epilogue(const EpiParams& ep, uint32_t taddr, int row, bool row_ok,
                                                  int col_base, int col_off, uint8_t* stage, int M, int lane,
                                                  int n_chunks) {
  static_assert(HD == 32 || HD == 64, "head dim");
  static_assert((BN / 2) % HD == 0, "each half tile must hold whole heads");
  constexpr int RD = 2 * ((HD / 3) / 2);
  constexpr int HALF = RD / 2;
  const int D = ep.dmodel;
  const int which = col_base / D;
  const int head0 = (col_base + col_off - which * D) / HD;   // first head of this thread's half tile
  const int clip = row / ep.n_tok;
  const int tok = row - clip * ep.n_tok;
  float cz[3][HALF], sz[3][HALF];
  if (which < 2) {
    int p[3] = {0, 0, 0};
    if (row_ok) {
      const int plane = ep.rope.gh * ep.rope.gw;
      // a caller's id outside the grid is clamped (and reported by the id check)
      const int gid = min(max(ep.pos_ids != nullptr ? __ldg(ep.pos_ids + row) : tok, 0), ep.rope.gt * plane - 1);
      p[0] = gid / plane;
      const int rem = gid - p[0] * plane;
      p[1] = rem / ep.rope.gw;
      p[2] = rem - p[1] * ep.rope.gw;
    }
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      const float* ct = ep.rope.cos_tab + (a * ep.rope.max_pos + p[a]) * HALF;
      const float* st = ep.rope.sin_tab + (a * ep.rope.max_pos + p[a]) * HALF;
      if constexpr (HALF % 2 == 0) {
        // rows of an even number of floats start on 8 bytes: two angles per load
#pragma unroll
        for (int k = 0; k < HALF; k += 2) {
          const float2 cc = __ldg(reinterpret_cast<const float2*>(ct + k));
          const float2 ss = __ldg(reinterpret_cast<const float2*>(st + k));
          cz[a][k] = cc.x;
          cz[a][k + 1] = cc.y;
          sz[a][k] = ss.x;
          sz[a][k + 1] = ss.y;
        }
      } else {
#pragma unroll
        for (int k = 0; k < HALF; ++k) {
          cz[a][k] = __ldg(ct + k);
          sz[a][k] = __ldg(st + k);
        }
      }
    }
  }
  const size_t bh0 = (size_t)clip * ep.n_head + head0;
#pragma unroll
  for (int c = 0; c < BN / 64; ++c) {
    if (c >= n_chunks) break;
    uint32_t r[32];
    tmem_ld32(taddr + c * 32, r);
    tmem_wait_ld();
    const int d0 = (c * 32) % HD;
    const size_t bh = bh0 + (c * 32) / HD;
    if (which < 2 && !row_ok) {
      // the warp still takes part in the staged store of this head
      if (d0 + 32 == HD) stage_out_head<T, HD>(ep, which, stage, row - lane, (int)(bh - bh0) + head0, M, lane);
      continue;
    }
    if (!row_ok) continue;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    if (ep.bias != nullptr) {
      const float* b = ep.bias + col_base + col_off + c * 32;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 bb = __ldg(reinterpret_cast<const float4*>(b + i));
        add2f(v[i], v[i + 1], bb.x, bb.y);
        add2f(v[i + 2], v[i + 3], bb.z, bb.w);
      }
    }
    if (which < 2) {
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int dim = d0 + j;
        if (dim < 3 * RD) {
          const int a = dim / RD;
          const int jj = dim - a * RD;
          const int f0 = LAYOUT == 0 ? jj % HALF : jj / 2;
          const int f1 = LAYOUT == 0 ? (jj + 1) % HALF : jj / 2;
          const float x0 = v[j], x1 = v[j + 1];
          v[j] = x0 * cz[a][f0] - x1 * sz[a][f0];
          v[j + 1] = x1 * cz[a][f1] + x0 * sz[a][f1];
        }
      }
      uint4* srow = reinterpret_cast<uint4*>(stage + lane * 128);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 u;
        u.x = pack2<T>(v[8 * i + 0], v[8 * i + 1]);
        u.y = pack2<T>(v[8 * i + 2], v[8 * i + 3]);
        u.z = pack2<T>(v[8 * i + 4], v[8 * i + 5]);
        u.w = pack2<T>(v[8 * i + 6], v[8 * i + 7]);
        srow[(d0 / 8 + i) ^ (lane & 7)] = u;
      }
      if (d0 + 32 == HD) stage_out_head<T, HD>(ep, which, stage, row - lane, (int)(bh - bh0) + head0, M, lane);
    } else {
      T* dst = reinterpret_cast<T*>(ep.vt) + (bh * HD + d0) * (size_t)ep.ldv + tok;
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[(size_t)i * ep.ldv] = DT<T>::from(v[i]);
    }
  }
}

// Residual epilogue by reduction, for rows row0 .. row0+31 of the tile and
// NCOLS fp32 columns from col0: accumulator (+ bias) -> a 32 x 128-byte
// staging block in the 128B swizzle -> one TMA reduce-add per block into the
// output, which holds the residual: out = residual + (accumulator + bias),
// one fp32 addition per element performed by L2.  The warp's next block waits
// only until the previous reduction has read the buffer, not for its writes.
template <int NCOLS>
__device__ __forceinline__ void reduce_epilogue(const EpiParams& ep, const CUtensorMap* tmC, uint32_t taddr, int row0,
                                                int col0, uint8_t* buf, int lane) {
  constexpr int kCols = 32;  // fp32 columns per 128-byte block
#pragma unroll 1
  for (int c = 0; c < NCOLS / kCols; ++c) {
    float v[kCols];
    {
      uint32_t r[32];
      tmem_ld32(taddr + c * kCols, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    }
    if (ep.bias != nullptr) {
      const float4* b4 = reinterpret_cast<const float4*>(ep.bias + col0 + c * kCols);
#pragma unroll
      for (int i = 0; i < kCols / 4; ++i) {
        const float4 bb = __ldg(b4 + i);
        add2f(v[4 * i], v[4 * i + 1], bb.x, bb.y);
        add2f(v[4 * i + 2], v[4 * i + 3], bb.z, bb.w);
      }
    }
    // the previous block's reduction has read the buffer
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    uint8_t* my_row = buf + lane * 128;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<float4*>(my_row + ((k ^ (lane & 7)) << 4)) =
          make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_reduce_add_2d(tmC, buf, col0 + c * kCols, row0);
      bulk_commit_group();
    }
  }
}

// Epilogue of one warp for rows row0 .. row0+31 of the tile (its TMEM lanes)
// and NCOLS columns from col0: accumulator (+ bias, activation) -> a 32 x
// 128-byte staging buffer in the 128B swizzle -> one TMA tensor store per
// 128-byte column block, so global memory sees whole rows instead of one row
// per lane.  Rows and columns outside the output are clipped by the tensor map.
template <typename T, int EPI, int NCOLS>
__device__ __forceinline__ void staged_epilogue(const EpiParams& ep, const CUtensorMap* tmC, uint32_t taddr, int row0,
                                                int col0, uint8_t* buf, int lane) {
  static_assert(EPI == EPI_STORE || EPI == EPI_F32 || EPI == EPI_GELU, "staged epilogue");
  constexpr bool kF32Out = EPI == EPI_F32;
  constexpr int kCols = kF32Out ? 32 : 64;  // columns per 128-byte block
  uint8_t* my_row = buf + lane * 128;
#pragma unroll 1
  for (int c0 = 0; c0 < NCOLS; c0 += kCols) {
    float v[kCols];
#pragma unroll
    for (int h = 0; h < kCols / 32; ++h) {
      uint32_t r[32];
      tmem_ld32(taddr + c0 + h * 32, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) v[h * 32 + i] = __uint_as_float(r[i]);
    }
    if (ep.bias != nullptr) {
      const float4* b4 = reinterpret_cast<const float4*>(ep.bias + col0 + c0);
#pragma unroll
      for (int i = 0; i < kCols / 4; ++i) {
        const float4 bb = __ldg(b4 + i);
        add2f(v[4 * i], v[4 * i + 1], bb.x, bb.y);
        add2f(v[4 * i + 2], v[4 * i + 3], bb.z, bb.w);
      }
    }
    if constexpr (EPI == EPI_GELU) {
#pragma unroll
      for (int i = 0; i < kCols; i += 2) gelu_as2(v[i], v[i + 1]);
    }
    if (lane == 0) bulk_wait_read_all();  // the previous block's store has left the buffer
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint4 w;
      if constexpr (kF32Out) {
        w = make_uint4(__float_as_uint(v[4 * k]), __float_as_uint(v[4 * k + 1]), __float_as_uint(v[4 * k + 2]),
                       __float_as_uint(v[4 * k + 3]));
      } else {
        w = make_uint4(pack2<T>(v[8 * k], v[8 * k + 1]), pack2<T>(v[8 * k + 2], v[8 * k + 3]),
                       pack2<T>(v[8 * k + 4], v[8 * k + 5]), pack2<T>(v[8 * k + 6], v[8 * k + 7]));
      }
      *reinterpret_cast<uint4*>(my_row + ((k ^ (lane & 7)) << 4)) = w;
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmC, buf, col0 + c0, row0);
      bulk_commit_group();
    }
  }
}

// Tile of work unit u: its row-tile group mp, column tile tn, first output
// column col0 and width (BN, or BN/2 for a half of a split tail tile).
struct UnitTile {
  int mp, tn, col0, width;
};
template <int BN>
__device__ __forceinline__ UnitTile unit_tile(int u, int num_n, int tail_start) {
  UnitTile t;
  const int tile = u < tail_start ? u : tail_start + ((u - tail_start) >> 1);
  t.mp = tile / num_n;
  t.tn = tile - t.mp * num_n;
  t.width = u < tail_start ? BN : BN / 2;
  t.col0 = t.tn * BN + (u < tail_start ? 0 : ((u - tail_start) & 1) * (BN / 2));
  return t;
}

// Whether an instantiation's epilogue can take a half-width (BN/2) tile: each
// epilogue warp then covers BN/4 columns, which must hold whole heads (QKV)
// or whole 128-byte output blocks.
template <int BN, int EPI, int QHD>
__host__ __device__ constexpr bool can_split_tail() {
  if constexpr (EPI == EPI_QKV) return QHD > 0 && (BN / 4) % QHD == 0;
  if constexpr (EPI == EPI_RESID || EPI == EPI_F32) return (BN / 4) % 32 == 0;
  return (BN / 4) % 64 == 0;
}

template <typename T, int BN, int STAGES, int EPI, int QHD = 0, int QLAYOUT = 0, int CM = 1>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, int M, int N, int K, int tail_start, EpiParams ep,
                   int* status) {
  using S = GemmSmem<BN, STAGES, CM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * S::kABytes;
  uint8_t* sEpi = smem + S::kEpiOffset;  // epilogue staging, one 4 KB buffer per epilogue warp
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOffset);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // [2] accumulator ready for the epilogue
  uint64_t* tempty = tfull + 2;      // [2] accumulator drained by the epilogue
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_n = (N + BN - 1) / BN;
  // Work units: CM vertically adjacent 128 x BN tiles (same W rows).  With a
  // CTA pair (CM = 2) the even CTA issues one M = 256 MMA per K step over both
  // CTAs' shared memory; each CTA holds its 128 rows of A and half of the W
  // tile and receives its 128 rows of the accumulator in its tensor memory.
  // Units from tail_start on are the tiles of the last, partial wave, each
  // split into two BN/2-wide halves run by different CTAs (pairs), so that
  // wave takes about half as long; tail_start = the unit count means no split.
  const int num_tiles = ((M + kBM * CM - 1) / (kBM * CM)) * num_n;
  const int num_units = tail_start + 2 * (num_tiles - tail_start);
  const int num_kb = K / kBK;
  const int rank = CM == 2 ? (int)cluster_ctarank() : 0;
  const bool leader = rank == 0;
  const int first_unit = CM == 2 ? (int)cluster_id_x() : (int)blockIdx.x;
  const int unit_stride = CM == 2 ? (int)cluster_count_x() : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);    // the (even) CTA's producer arrives; bytes of both CTAs complete it
      mbar_init(&empty[s], 1);   // released by the MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], CM * (kEpiThreads / 32));   // one arrival per epilogue warp of every CTA
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (EPI != EPI_QKV) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    if constexpr (CM == 2) {
      tmem_alloc_pair(tmem_slot, S::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, S::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (CM == 2) {
    cluster_sync();   // both CTAs' barriers and tensor memory exist before any cross-CTA signal
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (every CTA)
    if (lane == 0) {
      const uint32_t full0 = CM == 2 ? mapa_shared(smem_u32(full), 0) : 0;  // the even CTA's full[0]
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      for (int u = first_unit; u < num_units && !*abort_flag; u += unit_stride) {
        const UnitTile ut = unit_tile<BN>(u, num_n, tail_start);
        const int tm = ut.mp * CM + rank;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            atomicOr(status, DEV_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          if constexpr (CM == 2) {
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * S::kStageBytes);
            tma_load_2d_pair(sA + stage * S::kABytes, &tmA, full0 + 8 * stage, kb * kBK, tm * kBM);
            // each CTA holds width/2 rows of W (a half tile leaves the rest of the box unused)
            tma_load_2d_pair(sB + stage * S::kBBytes, &tmB, full0 + 8 * stage, kb * kBK, ut.col0 + rank * (ut.width / 2));
          } else {
            mbar_arrive_expect_tx(&full[stage], S::kStageBytes);
            tma_load_2d(sA + stage * S::kABytes, &tmA, &full[stage], kb * kBK, tm * kBM);
            tma_load_2d(sB + stage * S::kBBytes, &tmB, &full[stage], kb * kBK, ut.col0);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Every copy issued must land before the CTAs exit: wait (bounded) for the
      // last min(issued, STAGES) stages.  The even CTA's barriers count the
      // bytes of both CTAs of a pair.
      if (leader) {
        const long pending = issued < STAGES ? issued : STAGES;
        for (long i = 0; i < pending; ++i) {
          if (--stage < 0) {
            stage = STAGES - 1;
            phase ^= 1;
          }
          mbar_wait(&full[stage], phase);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the even CTA)
    // The whole warp walks the schedule (waits are warp-uniform); one elected
    // lane issues each MMA and commit.
    if (leader) {
      constexpr uint32_t idesc_full = idesc_f16<T, kBM * CM, BN>();
      constexpr uint32_t idesc_half = idesc_f16<T, kBM * CM, BN / 2>();
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      bool ok = true;
      for (int u = first_unit; u < num_units; u += unit_stride, ++acc) {
        if (__any_sync(0xffffffffu, *abort_flag)) break;
        const int buf = acc & 1;
        const uint32_t acc_phase = (acc >> 1) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&tempty[buf], acc_phase ^ 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        const uint32_t idesc = u < tail_start ? idesc_full : idesc_half;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = smem_desc_kmajor<128>(smem_u32(sA + stage * S::kABytes));
          const uint64_t db = smem_desc_kmajor<128>(smem_u32(sB + stage * S::kBBytes));
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {  // +32 bytes along K = +2 in the descriptor's address field
            if constexpr (CM == 2) {
              umma_f16_ss_pair_warp(d_tmem, da + k * 2, db + k * 2, idesc, (kb | k) != 0);
            } else {
              umma_f16_ss_warp(d_tmem, da + k * 2, db + k * 2, idesc, (kb | k) != 0);
            }
          }
          if constexpr (CM == 2) {
            umma_commit_pair_warp(&empty[stage], (uint16_t)0x3);
          } else {
            umma_commit_warp(&empty[stage]);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (CM == 2) {
          umma_commit_pair_warp(&tfull[buf], (uint16_t)0x3);
        } else {
          umma_commit_warp(&tfull[buf]);
        }
      }
      if (!ok && lane == 0) {
        atomicOr(status, DEV_TIMEOUT);
        *abort_flag = 1;
      }
      // Drain: no MMA may still be running when tensor memory is released.
      if constexpr (CM == 2) {
        umma_commit_pair_warp(mma_done, (uint16_t)0x1);
      } else {
        umma_commit_warp(mma_done);
      }
      mbar_wait(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue (every CTA)
    // Eight warps: warp w drains TMEM lanes 32*(w%4) .. +31 (its rows) and the
    // column half (w-2)/4 of the tile, so two warps per SM sub-partition share
    // the epilogue work and hide each other's latency.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t tempty0 = CM == 2 ? mapa_shared(smem_u32(tempty), 0) : smem_u32(tempty);
    int acc = 0;
    for (int u = first_unit; u < num_units; u += unit_stride, ++acc) {
      const int buf = acc & 1;
      const uint32_t acc_phase = (acc >> 1) & 1;
      const bool ok = mbar_wait(&tfull[buf], acc_phase);
      // tcgen05.ld is warp-collective: the stop decision is warp-uniform.
      if (__any_sync(0xffffffffu, !ok || *abort_flag)) {
        if (lane == 0) atomicOr(status, DEV_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const UnitTile ut = unit_tile<BN>(u, num_n, tail_start);
      const int row = (ut.mp * CM + rank) * kBM + row_in_tile;
      const uint32_t tlane = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * BN;
      uint8_t* stage_buf = sEpi + (warp - 2) * S::kEpiStage;
      if constexpr (EPI == EPI_QKV) {
        // one code path for whole tiles and half-width tail tiles
        const int wcols = ut.width / 2;
        qkv_tile_epilogue<T, BN, QHD, QLAYOUT>(ep, tlane + half * wcols, row, row < M, ut.col0, half * wcols,
                                               stage_buf, M, lane, wcols / 32);
      } else if (ut.width == BN) {
        if constexpr (EPI == EPI_RESID) {
          reduce_epilogue<BN / 2>(ep, &tmC, tlane + half * (BN / 2), row - lane, ut.col0 + half * (BN / 2), stage_buf,
                                  lane);
        } else {
          staged_epilogue<T, EPI, BN / 2>(ep, &tmC, tlane + half * (BN / 2), row - lane, ut.col0 + half * (BN / 2),
                                          stage_buf, lane);
        }
      } else if constexpr (can_split_tail<BN, EPI, QHD>()) {
        // half-width tail tile: each warp drains BN/4 columns
        if constexpr (EPI == EPI_RESID) {
          reduce_epilogue<BN / 4>(ep, &tmC, tlane + half * (BN / 4), row - lane, ut.col0 + half * (BN / 4), stage_buf,
                                  lane);
        } else {
          staged_epilogue<T, EPI, BN / 4>(ep, &tmC, tlane + half * (BN / 4), row - lane, ut.col0 + half * (BN / 4),
                                          stage_buf, lane);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CM == 2) {
          mbar_arrive_cluster(tempty0 + 8 * buf);   // the even CTA's barrier
        } else {
          mbar_arrive(&tempty[buf]);
        }
      }
    }
    if (EPI != EPI_QKV && lane == 0) bulk_wait_all();  // the tile stores have completed
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CM == 2) cluster_sync();   // the pair's MMAs and epilogues are done; no signal targets an exited CTA
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CM == 2) {
      tmem_dealloc_pair(tmem_base, S::kTmemCols);
    } else {
      tmem_dealloc(tmem_base, S::kTmemCols);
    }
  }
}

// First tile of the last wave to split into halves: the tiles beyond the last
// full wave of `slots` resident CTAs (pairs), when twice their count still fits
// in one wave and the epilogue takes half tiles; otherwise `tiles` (no split).
template <int BN, int EPI, int QHD>
int split_tail_start(int tiles, int slots) {
  if constexpr (!can_split_tail<BN, EPI, QHD>()) {
    return tiles;
  } else {
    const int rem = tiles % slots;
    if (rem == 0 || 2 * rem > slots) return tiles;
    return tiles - rem;
  }
}

template <typename T, int BN, int STAGES, int CM, int EPI, int QHD = 0, int QLAYOUT = 0>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, int M, int N, int K,
                       const EpiParams& ep, int* status, cudaStream_t stream, int num_sms) {
  using S = GemmSmem<BN, STAGES, CM>;
  auto kern = gemm_tc_kernel<T, BN, STAGES, EPI, QHD, QLAYOUT, CM>;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = S::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Per device and instantiation: the shared-memory opt-in and, for CTA
  // pairs, how many pairs can be resident at once (the persistent grid's size).
  static DeviceOnce setup;
  static int resident_on[kMaxDevices];
  int dev = 0;
  cudaError_t e = setup.run([&](int d) -> cudaError_t {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kBytes);
    if (r != cudaSuccess) return r;
    int resident = num_sms / 2;
    if constexpr (CM == 2) {
      cudaLaunchConfig_t probe = cfg;
      probe.gridDim = dim3(2 * (num_sms / 2));
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &probe) == cudaSuccess && n >= 1) resident = n;
    }
    resident_on[d] = resident;
    return cudaSuccess;
  }, &dev);
  if (e != cudaSuccess) return e;
  const int num_m = (M + kBM - 1) / kBM, num_n = (N + BN - 1) / BN;
  if constexpr (CM == 2) {
    const int resident = resident_on[dev];
    const int tiles = ((num_m + 1) / 2) * num_n;
    const int tail_start = split_tail_start<BN, EPI, QHD>(tiles, resident);
    const int units = tail_start + 2 * (tiles - tail_start);
    const int clusters = units < resident ? units : resident;
    cfg.gridDim = dim3(2 * clusters);
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, M, N, K, tail_start, ep, status);
  } else {
    const int tiles = num_m * num_n;
    const int tail_start = split_tail_start<BN, EPI, QHD>(tiles, num_sms);
    const int units = tail_start + 2 * (tiles - tail_start);
    const int grid = units < num_sms ? units : num_sms;
    kern<<<grid, kThreads, S::kBytes, stream>>>(ta, tb, tc, M, N, K, tail_start, ep, status);
    return cudaGetLastError();
  }
}

template <typename T, int BN, int STAGES, int CM>
cudaError_t dispatch_epi(int epi, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, int M, int N,
                         int K, const EpiParams& ep, int* status, cudaStream_t s, int sms) {
  switch (epi) {
    case EPI_STORE: return launch_one<T, BN, STAGES, CM, EPI_STORE>(ta, tb, tc, M, N, K, ep, status, s, sms);
    case EPI_F32: return launch_one<T, BN, STAGES, CM, EPI_F32>(ta, tb, tc, M, N, K, ep, status, s, sms);
    case EPI_RESID: return launch_one<T, BN, STAGES, CM, EPI_RESID>(ta, tb, tc, M, N, K, ep, status, s, sms);
    case EPI_GELU: return launch_one<T, BN, STAGES, CM, EPI_GELU>(ta, tb, tc, M, N, K, ep, status, s, sms);
    case EPI_QKV:
      if (ep.head_dim == 64)
        return ep.rope.layout == 0
                   ? launch_one<T, BN, STAGES, CM, EPI_QKV, 64, 0>(ta, tb, tc, M, N, K, ep, status, s, sms)
                   : launch_one<T, BN, STAGES, CM, EPI_QKV, 64, 1>(ta, tb, tc, M, N, K, ep, status, s, sms);
      return ep.rope.layout == 0 ? launch_one<T, BN, STAGES, CM, EPI_QKV, 32, 0>(ta, tb, tc, M, N, K, ep, status, s, sms)
                                 : launch_one<T, BN, STAGES, CM, EPI_QKV, 32, 1>(ta, tb, tc, M, N, K, ep, status, s, sms);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t gemm_tc_typed(int epi, const void* A, const void* W, int M, int N, int K, const EpiParams& ep,
                          int* status, cudaStream_t s, int sms) {
  const int BN = (N % 256 == 0) ? 256 : 128;
  // With at least two row tiles, CTA pairs run M = 256 MMAs.
  const int cm = M > kBM ? 2 : 1;
  CUtensorMap ta, tb;
  cudaError_t e = make_tmap_2d(&ta, A, sizeof(T), K, M, (size_t)K * sizeof(T), kBK, kBM);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&tb, W, sizeof(T), K, N, (size_t)K * sizeof(T), kBK, BN / cm);
  if (e != cudaSuccess) return e;
  // Output map for the staged epilogue: 32-row boxes of one 128-byte column block.
  CUtensorMap tc = ta;
  if (epi != EPI_QKV) {
    const int ob = (epi == EPI_F32 || epi == EPI_RESID) ? 4 : (int)sizeof(T);
    e = make_tmap_2d(&tc, ep.out, ob, N, M, (size_t)ep.ldo * ob, 128 / ob, 32);
    if (e != cudaSuccess) return e;
  }
  if (cm == 2) {
    // a CTA holds 128 rows of A and BN/2 rows of W per stage
    if (BN == 256) return dispatch_epi<T, 256, 6, 2>(epi, ta, tb, tc, M, N, K, ep, status, s, sms);
    return dispatch_epi<T, 128, 8, 2>(epi, ta, tb, tc, M, N, K, ep, status, s, sms);
  }
  if (BN == 256) return dispatch_epi<T, 256, 4, 1>(epi, ta, tb, tc, M, N, K, ep, status, s, sms);
  return dispatch_epi<T, 128, 6, 1>(epi, ta, tb, tc, M, N, K, ep, status, s, sms);
}

}  // namespace

cudaError_t gemm_tc(int dtype, int epi, const void* A, const void* W, int M, int N, int K, const EpiParams& ep,
                    int* status, cudaStream_t s, int num_sms) {
  if (dtype == DTYPE_BF16) return gemm_tc_typed<__nv_bfloat16>(epi, A, W, M, N, K, ep, status, s, num_sms);
  return gemm_tc_typed<__half>(epi, A, W, M, N, K, ep, status, s, num_sms);
}

}  // namespace jepa
