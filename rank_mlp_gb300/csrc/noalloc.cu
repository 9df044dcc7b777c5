// lora_linear_forward_noalloc: the single LoRA linear's forward (inference) for
// callers that cannot allocate device memory at the point where they run it -- a
// plugin inside a host framework that owns all device memory and hands the plugin
// only its input and output buffers, or a latency-critical loop that must never call
// cudaMalloc (which may synchronise the device).  The caller passes x, the adapter
// and y; every intermediate the forward needs lives in the fixed array below.
#include <cmath>
#include <mutex>

#include "api_internal.cuh"

namespace {

// Scratch shared by every call on a device.  Each GPU that loads this library holds
// these 32 MiB until the process exits.  Its first 256 bytes are the status word the
// kernels set on an expired wait: zero when the module loads, cleared by
// lora_poll_status(NULL, stream), never by a call.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (ids are never reused within a
// process), or 0 when there is none or the driver does not report one.
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  static const CtxGetIdFn get_id = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetIdFn>(nullptr);
    return reinterpret_cast<CtxGetIdFn>(p);
  }();
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id;
  void* ptr;
};
std::mutex g_setup_mu;
ScratchSlot g_scratch[kMaxDevices] = {};

}  // namespace

namespace lgb {

// Device address of the scratch array in the current device's context.  Host code
// cannot use the array's name as a device address, so it is looked up with
// cudaGetSymbolAddress: once per device, and again whenever the device's context is
// not the one the cached address belongs to (a reset destroys the module and its
// array with the context).  Without a context id from the driver it is looked up on
// every call.
void* noalloc_scratch() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  unsigned long long id = current_context_id();
  ScratchSlot& S = g_scratch[dev];
  if (S.ptr == nullptr || id == 0 || S.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    if (id == 0) id = current_context_id();    // the lookup may have made the context current
    S.ptr = p;
    S.ctx_id = id;
  }
  return S.ptr;
}

}  // namespace lgb

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
  if (lgb::linear_forward_workspace_bytes(M, in, out, r) > kNoAllocScratchBytes) return LORA_ERR_WORKSPACE;
  if (M == 0) return LORA_OK;
  void* scratch = lgb::noalloc_scratch();
  if (scratch == nullptr) return LORA_ERR_CUDA;
  // Everything the forward reads from the scratch it writes first, apart from the
  // status word, which keeps an unpolled error of an earlier call.
  return lgb::linear_forward_whole_tiles(M, in, out, r, s, x, lin, y, scratch, kNoAllocScratchBytes, stream);
}
