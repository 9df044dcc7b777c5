// One pass over token-major gradients Q_p (dg and du of the gated MLP; dy_q, dy_k,
// dy_v or dy_o of the attention projections) that makes both of their rank-r products
// ("Model Patches and Kernels", the LoRA backward):
//
//   V[:, slots]  = sum over products p of  Q_p B_p            (a projection: M x NV)
//   dB_p         = s Q_p^T T_p[:, slot_p]                      (a reduction over tokens: F_p x r)
//
// Each 128-token x 128-feature tile of Q is loaded once (TMA, 128-byte swizzle) and
// feeds two tcgen05 MMAs from the same shared memory: the projection reads it K-major
// (rows = tokens), the reduction MN-major (M = features, K = tokens) against the
// transposed rank-r operand T^T (slot rows x tokens, saved by the forward).  A CTA owns
// a range of token tiles and a range of feature blocks: its projection accumulator
// (double-buffered in TMEM) sums its feature blocks for one token tile at a time and
// is written to an f32 slab per feature range; its reduction accumulators (one TMEM
// block of NR columns per feature block of its range) sum its token tiles and are
// written once, to an f32 slab per token range.  The slabs are summed in a fixed order
// by the reduce kernel (deterministic), which also applies s.
#pragma once

#include "gemm_tc.cuh"

namespace lgb {

constexpr int kDualMaxProducts = 3;
constexpr int kDualMaxCtas = 152;
constexpr int kDualStages = 4;
constexpr int kDualNVMax = 32;                         // projection accumulator columns
constexpr int kDualNRMax = 16;                         // reduction accumulator columns
constexpr int kDualTmemCols = 512;
constexpr int kDualVCols = 2 * kDualNVMax;             // the two projection buffers
constexpr int kDualMaxBlocks = (kDualTmemCols - kDualVCols) / kDualNRMax;   // feature blocks per CTA
constexpr int kDualQBytes = 128 * 128 * 2;             // 128 tokens x 128 features
constexpr int kDualBBytes = 2 * kDualNVMax * 128;      // NV rows x 128 features
constexpr int kDualStageBytes = kDualQBytes + kDualBBytes;
constexpr int kDualTBytes = 2 * kDualNRMax * 128;      // one product's T^T: NR rows x 128 tokens
constexpr int kDualSlotBytes = kDualMaxProducts * kDualTBytes;
constexpr int kDualNumBars = 2 * kDualStages + 9;
constexpr int kDualSmemBytes = kDualStages * kDualStageBytes + 2 * kDualSlotBytes + 8 * kDualNumBars + 16 + 1024;
static_assert(kDualStageBytes % 1024 == 0 && kDualSlotBytes % 1024 == 0, "dual alignment");
static_assert(kDualSmemBytes <= 232448, "shared memory per CTA");

struct DualProduct {
  int q_map, b_map, t_map;   // tensor maps: Q [M x F] (box 64 x 128), B^T [NV x F] (box 64 x NV),
                             // T^T [kf x M] (box 64 x NR)
  int nkb;                   // 128-feature blocks of this product
  int t_row;                 // first T^T row of this product's rank slot (rows past the
                             // products' slots may hold anything: they reach only
                             // reduction columns past r, which are never written out)
  float* db_part;            // [gt][nkb * 128][NR] f32 partial dB
};

struct DualParams {
  CUtensorMap maps[3 * kDualMaxProducts];
  DualProduct prod[kDualMaxProducts];
  int nprod;
  int tiles_m;               // 128-token tiles
  int nv, nr;                // projection and reduction accumulator widths (16 or 32; 16)
  int gt, gf;                // token ranges x feature ranges = CTAs
  int kb_total;              // feature blocks of all products
  float* v_part;             // [gf][tiles_m * 128][nv] f32 partial projection
  unsigned int* status;
  unsigned long long timeout_ns;
};

// Defined in gemm_skinny.cu.
cudaError_t launch_rank_dual(const DualParams& p, int grid, cudaStream_t st);

}  // namespace lgb
