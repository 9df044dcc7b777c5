// 128 x 64 / 128 x 128 tiles: the rank-r products (token-major projections such as
// x A^T, and the reductions over tokens that give dA and dB).  HBM-bound; deep rings.
#include "gemm_pair.cuh"
#include "host.cuh"
#include "rank_dual_impl.cuh"

namespace lgb {

template <int BN, int STAGES, bool A_MN, bool B_MN>
static cudaError_t launch_one(const TcParams& p, int grid, cudaStream_t st) {
  auto* k = tc_gemm_kernel<BN, STAGES, A_MN, B_MN>;
  constexpr int smem = TcCfg<BN, STAGES>::kSmemBytes;
  static std::atomic<unsigned long long> configured{0};
  const cudaError_t e = ensure_smem_limit(k, smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(kThreads), smem, st, p);
}

cudaError_t launch_tc_skinny(int variant, const TcParams& p, int grid, cudaStream_t st) {
  switch (variant) {
    case V64_KK: return launch_one<64, 8, false, false>(p, grid, st);
    case V64_MNMN: return launch_one<64, 8, true, true>(p, grid, st);
    case V128_KK: return launch_one<128, 6, false, false>(p, grid, st);
    case V128_MNMN: return launch_one<128, 6, true, true>(p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rank_dual(const DualParams& p, int grid, cudaStream_t st) {
  static std::atomic<unsigned long long> configured{0};
  const cudaError_t e = ensure_smem_limit(rank_dual_kernel, kDualSmemBytes, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(rank_dual_kernel, dim3(grid), dim3(kThreads), kDualSmemBytes, st, p);
}

int tc_smem_bytes(int variant) {
  switch (variant) {
    case VP_KK:
    case VP_KK8:
    case VP_KMN: return PairCfg<6>::kSmemBytes;
    case VP_KMN_ACT: return PairCfg<6>::kSmemBytes;
    case VP_KMN_ACT16: return PairCfg<5, 8, 4>::kSmemBytes;
    case V64_KK:
    case V64_MNMN: return TcCfg<64, 8>::kSmemBytes;
    default: return TcCfg<128, 6>::kSmemBytes;
  }
}

}  // namespace lgb
