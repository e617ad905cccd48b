// Device-side helpers shared by the kernels: dtype traits, PTX wrappers for
// mbarrier / TMA / tcgen05 (sm_103a), bounded barrier waits, RoPE tables.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace jepa {

// ----------------------------------------------------------------------------- status word
// Bits set by a kernel in the handle's device status word.
// Device status bits: a bounded wait expired; a token id was outside its grid
// (the kernels clamp it so nothing is read out of range).
enum : int { DEV_TIMEOUT = 1, DEV_BAD_INDEX = 2 };
// A wait on a barrier gives up after this many nanoseconds (a correct kernel
// never waits more than microseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ----------------------------------------------------------------------------- dtypes
template <typename T> struct DT;
template <> struct DT<float> {
  static __device__ __forceinline__ float to(float x) { return x; }
  static __device__ __forceinline__ float from(float x) { return x; }
};
template <> struct DT<__nv_bfloat16> {
  static __device__ __forceinline__ float to(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
};
template <> struct DT<__half> {
  static __device__ __forceinline__ float to(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from(float x) { return __float2half_rn(x); }
};

// Packs two floats into one 32-bit word of two 16-bit values (low half = a).
template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
// Exact-erf GELU, 0.5 z (1 + erf(z / sqrt 2)).
__device__ __forceinline__ float gelu_erf(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }

// (a, b) += (x, y) as one packed f32x2 add.
__device__ __forceinline__ void add2f(float& a, float& b, float x, float y) {
  uint64_t p, q;
  asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %2};" : "=l"(q) : "f"(x), "f"(y));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(p) : "l"(q));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(p));
}

// GELU(z) = 0.5 z (1 + erf(z / sqrt 2)) for two values at once, with erf from
// Abramowitz & Stegun, Handbook of Mathematical Functions, eq. 7.1.28
// (Hastings): erf(x) = 1 - (1 + a1 x + ... + a6 x^6)^-16 for x >= 0, absolute
// error <= 3e-7, odd in x.  Uses packed f32x2 arithmetic and one approximate
// reciprocal per value; for the 16-bit outputs of the tensor-core path (the
// fp32 path keeps erff).
__device__ __forceinline__ void gelu_as2(float& z0, float& z1) {
  // u = z / sqrt(2) for both values; |u| by clearing both sign bits at once
  uint64_t z, u, p, ax;
  asm("mov.b64 %0, {%1, %2};" : "=l"(z) : "f"(z0), "f"(z1));
  const float k = 0.70710678118654752f;
  asm("{\n\t.reg .b64 kk;\n\tmov.b64 kk, {%2, %2};\n\tmul.rn.f32x2 %0, %1, kk;\n\t}" : "=l"(u) : "l"(z), "f"(k));
  asm("and.b64 %0, %1, 0x7FFFFFFF7FFFFFFF;" : "=l"(ax) : "l"(u));
#define JEPA_C2(name, v) uint64_t name; asm("mov.b64 %0, {%1, %1};" : "=l"(name) : "f"(v));
  JEPA_C2(a6, 0.0000430638f)
  JEPA_C2(a5, 0.0002765672f)
  JEPA_C2(a4, 0.0001520143f)
  JEPA_C2(a3, 0.0092705272f)
  JEPA_C2(a2, 0.0422820123f)
  JEPA_C2(a1, 0.0705230784f)
  JEPA_C2(one, 1.0f)
  JEPA_C2(half, 0.5f)
#undef JEPA_C2
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(p) : "l"(ax), "l"(a6), "l"(a5));
  asm("fma.rn.f32x2 %0, %1, %0, %2;" : "+l"(p) : "l"(ax), "l"(a4));
  asm("fma.rn.f32x2 %0, %1, %0, %2;" : "+l"(p) : "l"(ax), "l"(a3));
  asm("fma.rn.f32x2 %0, %1, %0, %2;" : "+l"(p) : "l"(ax), "l"(a2));
  asm("fma.rn.f32x2 %0, %1, %0, %2;" : "+l"(p) : "l"(ax), "l"(a1));
  asm("fma.rn.f32x2 %0, %1, %0, %2;" : "+l"(p) : "l"(ax), "l"(one));
  asm("mul.rn.f32x2 %0, %0, %0;" : "+l"(p));  // ^2
  asm("mul.rn.f32x2 %0, %0, %0;" : "+l"(p));  // ^4
  asm("mul.rn.f32x2 %0, %0, %0;" : "+l"(p));  // ^8
  asm("mul.rn.f32x2 %0, %0, %0;" : "+l"(p));  // ^16
  float pa, pb;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(pa), "=f"(pb) : "l"(p));
  float ra, rb;  // r = 1/p^16 = 1 - |erf(u)| (0 once p^16 overflows: erf = +-1 there)
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(ra) : "f"(pa));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rb) : "f"(pb));
  // gelu(z) = z/2 (1 + erf(u)) = z - z r / 2 for z >= 0, z r / 2 for z < 0
  uint64_t r, h;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(ra), "f"(rb));
  asm("{\n\t.reg .b64 zh;\n\tmul.rn.f32x2 zh, %1, %2;\n\tmul.rn.f32x2 %0, zh, %3;\n\t}" : "=l"(h) : "l"(z), "l"(half), "l"(r));
  float ha, hb;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(ha), "=f"(hb) : "l"(h));
  z0 = z0 >= 0.0f ? z0 - ha : ha;
  z1 = z1 >= 0.0f ? z1 - hb : hb;
}

// ----------------------------------------------------------------------------- misc PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// ----------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of parity `parity` to complete.  Returns false if it
// did not within limit_ns (the caller then records a timeout and winds down
// instead of spinning forever).  The limit is counted on the SM clock as
// 2 * limit_ns cycles (about the requested time at this part's 2.07 GHz
// maximum, longer at lower clocks) and checked once every 64 polls, so the
// poll loop itself stays short.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if ((unsigned long long)(clock64() - t0) > 2ull * limit_ns) return false;
  }
}

// ----------------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// TMA tile store from this CTA's shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
// TMA tile reduction from this CTA's shared memory into global memory:
// global += shared, element by element, in the tensor map's element type
// (bulk-group completion).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* m, const void* src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the shared-memory sources of all committed bulk groups have been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until all committed bulk groups have completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// All threads of every CTA in the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier given by its shared::cluster address (possibly in a peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA tile load into this CTA's shared memory whose completion is signalled on
// an mbarrier of either CTA of the CTA pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster_addr, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster_addr), "r"(x), "r"(y)
      : "memory");
}

// ----------------------------------------------------------------------------- tcgen05
// Tensor-memory allocation (the whole warp executes these).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// CTA-pair forms: one warp of each CTA of the pair executes them; the pair's
// allocations sit at the same column in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// MMA issue, warp-wide: every lane of a converged warp calls these with the
// same operands and one elected lane issues.  kind::f16 (bf16 or fp16
// inputs, fp32 accumulator); _ss: A and B from shared memory, _ts: A from
// tensor memory (M rows = TMEM lanes, K 16-bit values packed two per 32-bit
// column, even index in the low half); _pair: over the CTA pair, issued by
// the even CTA (M = 256 rows, A's rows 0-127 and D's lanes in the even CTA,
// rows 128-255 in the odd one, B's rows split the same way).  Keeping
// the whole warp on the issue path lets the operands stay in uniform
// registers; issued from a single divergent lane, each tcgen05.mma costs
// about as many cycles as a 128 x 128 x 16 product takes to execute.
__device__ __forceinline__ void umma_f16_ss_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_f16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void umma_f16_ss_pair_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair_warp(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}\n" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (base lane + i), columns [col, col+32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 8 consecutive 32-bit columns (as tmem_ld32).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// exactly one swizzle atom wide (128-byte rows with the 128B swizzle, or
// 64-byte rows with the 64B swizzle), 8-row atoms stacked contiguously (the
// layout a TMA tile load with that swizzle writes).  Fields: start address
// >> 4 (bits 0-13), leading byte offset >> 4 (bits 16-29; not used by this
// layout, set to 1), stride byte offset >> 4 (bits 32-45: distance between
// 8-row groups), version 1 (bits 46-47), base offset 0 (bits 49-51), layout
// type (bits 61-63: 2 = 128B swizzle, 4 = 64B swizzle).  Advancing along K
// inside the atom is done by adding the byte offset to the start address.
template <int kRowBytes>
__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t saddr) {
  static_assert(kRowBytes == 128 || kRowBytes == 64, "row width must be one swizzle atom");
  constexpr uint64_t layout = kRowBytes == 128 ? 2ull : 4ull;
  constexpr uint64_t sbo = (8ull * kRowBytes) >> 4;
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (sbo << 32) | (1ull << 46) | (layout << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), A and B type (bits 7-9 and 10-12: 0 fp16, 1 bf16), both operands
// K-major (bits 15, 16 = 0), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
template <typename T, int M, int N>
__host__ __device__ constexpr uint32_t idesc_f16() {
  static_assert(M == 64 || M == 128 || M == 256, "M");
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "N");
  constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ----------------------------------------------------------------------------- RoPE
// Per-axis angle tables built on the host in double and rounded to float:
// cos_tab[(a * max_pos + p) * half + k] = cos(pos_a(p) * omega_k) for axis a
// (0 = t, 1 = h, 2 = w), grid index p, k < half = d/2, where pos_a(p) is the
// (possibly interpolated) position of grid index p.
struct RopeParams {
  const float* cos_tab;
  const float* sin_tab;
  int max_pos;      // stride of the position index
  int d;            // rotated width per axis
  int layout;       // 0 tiled, 1 interleaved
  int gt, gh, gw;   // grid for decoding a token id
};

// Rotates the pairs (dim0 + j, dim0 + j + 1), j = 0, 2, .., n-2, of one head
// row held in v (fp32) for the token at grid cell (t, h, w):
// out[2k] = x[2k] c - x[2k+1] s, out[2k+1] = x[2k+1] c' + x[2k] s', where the
// angle index of dim j in axis segment a is (j mod d/2) for the tiled layout
// and (j div 2) for the interleaved one.  dim0 must be even.
template <int n>
__device__ __forceinline__ void rope_apply(float* v, int dim0, const RopeParams& rp, int t, int h, int w) {
  const int d = rp.d, half = d >> 1;
#pragma unroll
  for (int j = 0; j < n; j += 2) {
    const int dim = dim0 + j;
    if (dim < 3 * d) {
      const int a = dim / d;
      const int jj = dim - a * d;
      const int p = a == 0 ? t : (a == 1 ? h : w);
      int f0, f1;
      if (rp.layout == 0) {
        f0 = jj % half;
        f1 = (jj + 1) % half;
      } else {
        f0 = f1 = jj >> 1;
      }
      const float* ct = rp.cos_tab + (a * rp.max_pos + p) * half;
      const float* st = rp.sin_tab + (a * rp.max_pos + p) * half;
      const float c0 = __ldg(ct + f0), s0 = __ldg(st + f0), c1 = __ldg(ct + f1), s1 = __ldg(st + f1);
      const float x0 = v[j], x1 = v[j + 1];
      v[j] = x0 * c0 - x1 * s0;
      v[j + 1] = x1 * c1 + x0 * s1;
    }
  }
}

// ----------------------------------------------------------------------------- GEMM epilogues
enum EpiKind : int { EPI_STORE = 0, EPI_F32 = 1, EPI_RESID = 2, EPI_GELU = 3, EPI_QKV = 4 };

// The fused normalisation (px - 255 mean) / (255 std) of the ImageNet
// statistics ("V-JEPA 2.1 ViT-B/16 384 - HuggingFace port", Preprocessing;
// "Parity ...", Preprocessing parity), evaluated as (px - 255 mean) * r with
// r = 1 / (255 std) rounded once to fp32.
__host__ __device__ constexpr float pix_mean255(int c) {
  return c == 0 ? 255.0f * 0.485f : (c == 1 ? 255.0f * 0.456f : 255.0f * 0.406f);
}
__host__ __device__ constexpr float pix_rcp255(int c) {
  return c == 0 ? 1.0f / (255.0f * 0.229f) : (c == 1 ? 1.0f / (255.0f * 0.224f) : 1.0f / (255.0f * 0.225f));
}

struct EpiParams {
  const float* bias;  // [N] or null
  void* out;          // EPI_STORE/GELU: T [M, ldo]; EPI_F32/RESID: float [M, ldo]
  int ldo;
  // EPI_QKV: columns [0,D) -> q, [D,2D) -> k, [2D,3D) -> v^T, per head.
  void* q;             // T [clips*n_head, n_tok, head_dim]
  void* k;             // T [clips*n_head, n_tok, head_dim]
  void* vt;            // T [clips*n_head, head_dim, ldv]
  int n_tok, n_head, head_dim, ldv, dmodel;
  const int* pos_ids;  // optional: grid cell (token id) of each row; else row % n_tok
  RopeParams rope;
};

}  // namespace jepa
