// lora_linear_forward_noalloc: the single LoRA linear's forward (inference) for
// callers that cannot allocate device memory at the point where they run it -- a
// plugin inside a host framework that owns all device memory and hands the plugin
// only its input and output buffers, or a latency-critical loop that must never call
// cudaMalloc (which may synchronise the device).  The caller passes x, the adapter
// and y; every intermediate the forward needs lives in the fixed array below.
#include <cmath>
#include <mutex>

#include "host.cuh"

namespace {

// Scratch shared by every call on a device.  Each GPU that loads this library holds
// these 32 MiB until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device (host code cannot use the array's name as a device address).
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" lora_status_t lora_linear_forward_noalloc(int64_t M, int64_t in, int64_t out, int r, float s,
                                                     const void* x, lora_linear_t lin, void* y,
                                                     cudaStream_t stream) {
  // The same argument rules as lora_linear_forward, checked before anything is enqueued.
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (M < 0 || in <= 0 || out <= 0 || r < 1 || !std::isfinite(s)) return LORA_ERR_INVALID_ARG;
  if ((M > 0 && (x == nullptr || y == nullptr)) || !lin.W || !lin.A || !lin.B) return LORA_ERR_INVALID_ARG;
  if (r > 256 || M > lgb::kMaxExtent || in > lgb::kMaxExtent || out > lgb::kMaxExtent) return LORA_ERR_UNSUPPORTED;
  if (in % 8 || out % 8 || !al(x, 16) || !al(y, 16) || !al(lin.W, 16) || !al(lin.A, 2) || !al(lin.B, 2))
    return LORA_ERR_ALIGNMENT;
  if (lora_linear_workspace_bytes(M, in, out, r) > kNoAllocScratchBytes) return LORA_ERR_WORKSPACE;
  if (M == 0) return LORA_OK;
  void* scratch = scratch_for_current_device();
  if (scratch == nullptr) return LORA_ERR_CUDA;
  // The status word at the front must start at zero for this call; everything else
  // the forward reads, it writes first.
  if (cudaMemsetAsync(scratch, 0, lgb::kWsHeader, stream) != cudaSuccess) return LORA_ERR_CUDA;
  return lora_linear_forward(M, in, out, r, s, x, lin, y, nullptr, scratch, kNoAllocScratchBytes, stream);
}
