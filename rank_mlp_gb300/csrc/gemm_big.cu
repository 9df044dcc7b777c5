// The block's projection GEMMs on CTA pairs, 256 x 256 tiles: forward with K-major
// weights, backward with the weights read MN-major (untransposed).
#include "gemm_pair.cuh"
#include "host.cuh"

namespace lgb {

template <int STAGES, bool B_MN, int EPIW, int ACTB = 0, int ECOLS = 16>
static cudaError_t launch_pair(const TcParams& p, int grid, cudaStream_t st) {
  auto* k = tc_gemm_pair_kernel<STAGES, B_MN, EPIW, ACTB, ECOLS>;
  constexpr int smem = PairCfg<STAGES, EPIW, ACTB >= 2 ? ACTB : 0, ECOLS>::kSmemBytes;
  static std::atomic<unsigned long long> configured{0};
  const cudaError_t e = ensure_smem_limit(k, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(pair_threads(EPIW)), smem, st, p);  // grid: a multiple of 2
}

cudaError_t launch_tc_big(int variant, const TcParams& p, int grid, cudaStream_t st) {
  switch (variant) {
    // forward (gate/up activation, down): 4 epilogue warps, 8 for short K; backward
    // (act', dx): 8
    case VP_KK: return launch_pair<6, false, 4>(p, grid, st);
    case VP_KK8: return launch_pair<6, false, 8>(p, grid, st);
    case VP_KMN: return launch_pair<6, true, 8>(p, grid, st);
    // act': g, u in and dg, du out one row per thread, or through shared memory (short K)
    case VP_KMN_ACT: return launch_pair<6, true, 8, 1>(p, grid, st);
    case VP_KMN_ACT16:
      return launch_pair<kActStagedStages, true, kActStagedWarps, kActStagedSlots, kActStagedCols>(p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lgb
