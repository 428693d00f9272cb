// Decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: an engine that owns all device memory
// through its own pool and forbids side allocations, a plugin loaded into such a
// host, or a latency-critical loop where an allocation's implicit device
// synchronisation is not acceptable. nc_op_attention_decode_noalloc serves them:
// it runs the same split-KV decode attention as nc_op_attention_decode, but its
// partial softmax states live in a fixed array in the library's device memory
// instead of a caller-provided scratch buffer. It calls no cudaMalloc, cudaFree
// or allocating library routine.
#include <mutex>

#include "common.cuh"
#include "nc_internal.h"

namespace nc {
namespace {

// 8 MiB of split partials: B * H * splits * (head_dim + 2) fp32 values. Every
// GPU that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchBytes / sizeof(float)];

// Device address of g_decode_scratch, looked up once per device. In host code
// the array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress with the device current.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace nc

extern "C" nc_status nc_op_attention_decode_noalloc(const void* q, const void* k, const void* v,
                                                    void* o, int32_t B, int32_t H, int32_t Hkv,
                                                    int32_t len, int32_t t_max, int32_t hd,
                                                    nc_dtype dtype, void* stream) {
  if (!q || !k || !v || !o) {
    nc::set_last_error("NULL pointer");
    return NC_ERR_INVALID_ARG;
  }
  if (B <= 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || len <= 0 || len > t_max || hd <= 0 ||
      hd % 2 != 0 || hd > 128) {
    nc::set_last_error("bad sizes");
    return NC_ERR_INVALID_ARG;
  }
  if (dtype != NC_F32 && dtype != NC_BF16 && dtype != NC_F16) {
    nc::set_last_error("bad dtype");
    return NC_ERR_INVALID_ARG;
  }
  const size_t need = nc::decode_attention_scratch_bytes(B, H, Hkv, len, hd);
  if (need > nc::kNoAllocScratchBytes) {
    nc::set_last_error("needs %zu bytes of scratch; the fixed array holds %zu (B * H * splits * "
                       "(head_dim + 2) * 4, at most 64 splits)",
                       need, nc::kNoAllocScratchBytes);
    return NC_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  const cudaError_t e = nc::scratch_for_current_device(&scratch);
  if (e != cudaSuccess) {
    nc::set_last_error("cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    return NC_ERR_CUDA;
  }
  nc::launch_attention_decode(q, k, v, o, B, H, Hkv, len, t_max, hd, dtype,
                              static_cast<float*>(scratch), static_cast<cudaStream_t>(stream));
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}
