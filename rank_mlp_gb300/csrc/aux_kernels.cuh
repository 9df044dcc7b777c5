// Small memory-bound kernels around the tcgen05 GEMM:
//  * pack:   builds the zero-padded rank-r operands of the folded K-segments from the
//            caller's adapters (optionally scaled by s and/or transposed), so that the
//            GEMM's TMA never touches a rank-r tensor with a row stride TMA cannot load.
//  * reduce: sums split-K partial tiles in a fixed order (deterministic), scales, and
//            writes bf16 rows or columns out of the padded f32 slab.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace lgb {

constexpr int kMaxPackJobs = 8;
constexpr int kMaxPackBlocks = 3;

struct PackBlock {
  const __nv_bfloat16* src;
  long long lds;      // row stride of src (elements)
  int ro, co;         // destination row/col of the block's (0, 0)
  int R, C;           // block extent in the destination
  int trans;          // 0: dst(ro+a, co+b) = src[a, b];  1: = src[b, a]
  float scale;
};

struct PackJob {
  __nv_bfloat16* dst;
  int rows, cols;     // dense [rows x cols] destination, row-major
  int nblk;
  PackBlock blk[kMaxPackBlocks];
};

struct PackParams {
  PackJob job[kMaxPackJobs];
  int njob;
};

constexpr int kMaxRedOuts = 3;

struct RedOut {
  const float* part;  // [splits][rows_pad][width] f32 slab
  int rows;           // valid rows of the slab
  long long rows_pad;
  int width;
  __nv_bfloat16* dst;
  int col0, ncols;    // columns [col0, col0 + ncols) of the slab
  long long ld;
  int trans;          // 0: dst[m * ld + c];  1: dst[c * ld + m]
  long long split_stride;  // per-split outputs: elements between consecutive splits' results
};

struct RedParams {
  int splits;
  float scale;
  int per_split;      // 0: out = scale * sum over splits; 1: split k -> dst + k * split_stride
  int nout;
  RedOut out[kMaxRedOuts];
};

// Per-example squared norms: for each example e (one block each), the sum of squares
// of its slice of every listed tensor.  Fixed summation order (deterministic).
constexpr int kMaxNormTensors = 8;

struct NormParams {
  const __nv_bfloat16* src[kMaxNormTensors];
  long long count[kMaxNormTensors];     // elements per example
  int ntensors;
  float* out;                           // [examples]
};

}  // namespace lgb
