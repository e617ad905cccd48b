// Patch embedding without any device allocation.
//
// The ordinary entry points (jepa_encode, jepa_encoder_embed) keep the
// unfolded patch matrix in a workspace the encoder handle allocates with
// cudaMalloc.  Some callers cannot allocate device memory on their own: a host
// application or inference server that owns every byte of device memory
// through its own pool, or a latency-critical loop where cudaMalloc's implicit
// device-wide synchronisation and its chance of failing under memory pressure
// are not acceptable.  jepa_patch_embed_static serves them: the caller passes
// the clip, the weights, the output (and optionally a status word), and the
// only scratch, the unfolded patches, lives in a fixed-size array that is part
// of the library image.
//
// Limits and sharing:
//   * the scratch holds at most kStaticMaxRows token rows of 1536 16-bit
//     values (12 MiB); every GPU that loads the library holds that array
//     until the process exits;
//   * every call on a device shares the one array, so calls whose GPU work
//     overlaps (different streams without ordering) race on it;
//   * the host-side address of the array is looked up once per device, on the
//     first call made with that device current (cudaGetSymbolAddress); make
//     that first call before any stream capture.
#include <mutex>

#include "internal.h"
#include "jepa_gb300.h"

namespace jepa {
void record_error(const char* msg);
}

namespace {

constexpr int kStaticMaxRows = 4096;
constexpr size_t kStaticScratchBytes = (size_t)kStaticMaxRows * 1536 * 2;

// In host code these names are host-side stand-ins, not device addresses:
// kernels receive the addresses returned by cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_patch_scratch[kStaticScratchBytes];
static __device__ int g_patch_status;

using jepa::kMaxDevices;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
int* g_status_addr[kMaxDevices] = {};

jepa_status err(jepa_status st, const char* msg) {
  jepa::record_error(msg);
  return st;
}

// Device addresses of the static arrays for the current device (looked up on
// the first call per device).
jepa_status device_arrays(int dev, void** scratch, int** status) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* s = nullptr;
    void* st = nullptr;
    if (cudaGetSymbolAddress(&s, g_patch_scratch) != cudaSuccess || s == nullptr)
      return err(JEPA_ERR_CUDA, "jepa_patch_embed_static: cudaGetSymbolAddress of the scratch array failed");
    if (cudaGetSymbolAddress(&st, g_patch_status) != cudaSuccess || st == nullptr)
      return err(JEPA_ERR_CUDA, "jepa_patch_embed_static: cudaGetSymbolAddress of the status word failed");
    g_scratch_addr[dev] = s;
    g_status_addr[dev] = static_cast<int*>(st);
  }
  *scratch = g_scratch_addr[dev];
  *status = g_status_addr[dev];
  return JEPA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" jepa_status jepa_patch_embed_static(const void* clip, const void* weight, const float* bias,
                                                        float* x_out, int* status, int batch, int n_frames,
                                                        int height, int width, int embed_dim, int dtype,
                                                        void* stream) {
  using namespace jepa;
  if (clip == nullptr || weight == nullptr || x_out == nullptr)
    return err(JEPA_ERR_ARG, "jepa_patch_embed_static: clip, weight and x_out are required");
  if (!aligned16(clip) || !aligned16(weight) || !aligned16(bias) || !aligned16(x_out))
    return err(JEPA_ERR_ARG, "jepa_patch_embed_static: buffers must be 16-byte aligned");
  if (dtype != DTYPE_BF16 && dtype != DTYPE_F16)
    return err(JEPA_ERR_UNSUPPORTED, "jepa_patch_embed_static: dtype must be F16 or BF16");
  if (embed_dim <= 0 || embed_dim % 128 != 0 || embed_dim > 4096)
    return err(JEPA_ERR_ARG, "jepa_patch_embed_static: embed_dim must be a multiple of 128, at most 4096");
  if (batch < 1 || n_frames < 2 || n_frames % 2 != 0 || height < 16 || width < 16 || height % 16 != 0 ||
      width % 16 != 0)
    return err(JEPA_ERR_ARG,
               "jepa_patch_embed_static: need batch >= 1, even n_frames >= 2, height and width multiples of 16");
  const long long rows = (long long)batch * (n_frames / 2) * (height / 16) * (width / 16);
  if (rows > kStaticMaxRows)
    return err(JEPA_ERR_ARG,
               "jepa_patch_embed_static: batch*(n_frames/2)*(height/16)*(width/16) exceeds the static scratch "
               "maximum of 4096 token rows (12 MiB)");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return err(JEPA_ERR_CUDA, "jepa_patch_embed_static: no usable current device");
  void* scratch = nullptr;
  int* own_status = nullptr;
  jepa_status st = device_arrays(dev, &scratch, &own_status);
  if (st != JEPA_OK) return st;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The unfold overwrites every scratch row the GEMM then reads, so nothing
  // needs clearing between calls.
  if (unfold_clip_u8(dtype, static_cast<const uint8_t*>(clip), scratch, batch, n_frames, height, width, 2, s) !=
      cudaSuccess)
    return err(JEPA_ERR_CUDA, "jepa_patch_embed_static: unfold launch failed");
  EpiParams ep{};
  ep.bias = bias;
  ep.out = x_out;
  ep.ldo = embed_dim;
  if (gemm_tc(dtype, EPI_F32, scratch, weight, (int)rows, embed_dim, 1536, ep,
              status != nullptr ? status : own_status, s, sms) != cudaSuccess)
    return err(JEPA_ERR_CUDA, "jepa_patch_embed_static: GEMM launch failed");
  return JEPA_OK;
}
