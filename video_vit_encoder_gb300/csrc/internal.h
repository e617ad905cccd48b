// Host-side declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace jepa {

// Launch set-up that the runtime keeps per device (the opt-in to more than
// 48 KB of dynamic shared memory, occupancy figures, SM counts) is done once
// per device and per call site, under a lock, so handles on different devices
// of one process, and threads launching at the same time, each see it done
// for their own device.  `init(dev)` runs with `dev` current; a failed init
// is retried by the next call.  State it computes goes into arrays indexed by
// the device, written before `done` is released and read after it.
constexpr int kMaxDevices = 64;
class DeviceOnce {
 public:
  template <typename F>
  cudaError_t run(F&& init, int* dev_out = nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (dev_out != nullptr) *dev_out = dev;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = init(dev);
    if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return e;
  }

 private:
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

// dtype codes of the ABI (jepa_dtype)
enum : int { DTYPE_F32 = 0, DTYPE_F16 = 1, DTYPE_BF16 = 2 };

// Tensor maps (TMA descriptors), 16-bit elements, 128B or 64B swizzle chosen
// from the inner box width (128 or 64 bytes).
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                         uint32_t box2);

// Linear layers.
cudaError_t gemm_tc(int dtype, int epi, const void* A, const void* W, int M, int N, int K, const EpiParams& ep,
                    int* status, cudaStream_t s, int num_sms);
cudaError_t gemm_simt_f32(int epi, const float* A, const float* W, int M, int N, int K, const EpiParams& ep,
                          cudaStream_t s);

// Attention: q, k [BH, n, hd]; vt [BH, hd, ldv]; out [B, n, H*hd].
cudaError_t attention_tc(int dtype, const void* q, const void* k, const void* vt, void* out, int batch, int n_head,
                         int n_tok, int head_dim, int ldv, float scale, int* status, cudaStream_t s, int num_sms);
cudaError_t attention_simt(int dtype, const void* q, const void* k, const void* vt, void* out, int batch, int n_head,
                           int n_tok, int head_dim, int ldv, float scale, cudaStream_t s);

// Element-wise / row-wise kernels.
// tubelet 2 (clips) or 1 (the 2.1 image path): rows of 3 * tubelet * 256.
// keep (device [batch, n_keep] token ids, clamped to the grid): only those
// tokens, in that order (the masked encoder); nullptr: every token.
cudaError_t unfold_clip_u8(int dtype, const uint8_t* clip, void* out, int batch, int T, int H, int W, int tubelet,
                           cudaStream_t s, const int* keep = nullptr, int n_keep = 0);
cudaError_t unfold_clip_f32(int dtype, const float* clip, void* out, int batch, int T, int H, int W, int tubelet,
                            cudaStream_t s, const int* keep = nullptr, int n_keep = 0);
cudaError_t layernorm(int out_dtype, const float* x, const float* w, const float* b, void* y, int rows, int dim,
                      float eps, cudaStream_t s);
cudaError_t mean_pool(const float* x, float* out, int batch, int n_tok, int dim, cudaStream_t s);
cudaError_t rope_inplace_f32(float* x, int batch, int n_tok, int n_head, int head_dim, const RopeParams& rp,
                             cudaStream_t s);
// dst row r = src row ids[r] cast to dtype; ids are clamped to [0, n_src).
cudaError_t gather_rows_cast(int dtype, const float* src, int n_src, const int* ids, int n, int dim, void* dst,
                             cudaStream_t s);
// Sets DEV_BAD_INDEX in *status when any of the n ids lies outside [0, limit).
cudaError_t check_ids(const int* ids, long n, int limit, int* status, cudaStream_t s);
cudaError_t fill_rows(float* dst, const float* row, int n, int dim, cudaStream_t s);
cudaError_t wait_timeout_selftest(int* status, uint64_t limit_ns, cudaStream_t s);

// Attentive-pool head (head_dim 64, D = 256, 512, 768 or 1024).
// q_out [D] = Wq q0 + bq; g_out [H, D] = gamma_kv * (Wk_h^T q_h / sqrt(hd)).
cudaError_t head_fold_query(int dtype, const void* Wq, const float* bq, const float* q0, const void* Wk,
                            const float* gamma_kv, float* q_out, float* g_out, int D, int H, cudaStream_t s);
// s [rows, H] scores, stats [rows, 2] = (mean, 1/std) of each row of x [rows, D].
cudaError_t head_xattn_scores(const float* x, const float* g, float* s, float* stats, int rows, int D, float eps,
                              int num_sms, cudaStream_t st);
// z [B, H, D] = gamma * sum_i softmax_i(s[:, h]) rstd_i (x_i - mu_i) + beta per clip;
// w [B, H, n] and part [ceil(n / chunk), B, H, D] are scratch.
cudaError_t head_xattn_pool(const float* x, const float* s, const float* stats, const float* gamma,
                            const float* beta, float* w, float* part, float* z, int B, int n, int D, int chunk,
                            cudaStream_t st);
// out[b, n] = act(A[b*lda + (n/group)*gstride + :K] . W[n, :] + bias[n]) + res[b*ldr + n].
cudaError_t head_rowvec(int dtype, bool gelu, const float* A, int lda, int group, int gstride, const void* W,
                        const float* bias, const float* res, int ldr, float* out, int ldo, int B, int N, int K,
                        cudaStream_t s);

}  // namespace jepa
