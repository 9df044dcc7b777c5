// 128 x 256 tiles: the block's projection GEMMs (forward with K-major weights,
// backward with the weights read MN-major, i.e. untransposed).
#include "host.cuh"

namespace lgb {

template <int BN, int STAGES, bool A_MN, bool B_MN>
static cudaError_t launch_one(const TcParams& p, int grid, cudaStream_t st) {
  auto* k = tc_gemm_kernel<BN, STAGES, A_MN, B_MN>;
  constexpr int smem = TcCfg<BN, STAGES>::kSmemBytes;
  static bool configured = false;   // attribute set once per process (device 0 and peers alike)
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  k<<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tc_big(int variant, const TcParams& p, int grid, cudaStream_t st) {
  switch (variant) {
    case V256_KK: return launch_one<256, 4, false, false>(p, grid, st);
    case V256_KMN: return launch_one<256, 4, false, true>(p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lgb
