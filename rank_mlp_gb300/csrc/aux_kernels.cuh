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

constexpr int kMaxPackJobs = 12;   // the Q/K/V + O forward's six and its backward's six
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

constexpr int kMaxRedOuts = 8;

struct RedOut {
  const float* part;  // [splits][rows_pad][width] f32 slab
  int rows;           // valid rows of the slab
  long long rows_pad;
  int width;
  int splits;
  int per_split;      // 0: out = scale * sum over splits; 1: split k -> dst + k * split_stride
  float scale;
  __nv_bfloat16* dst;
  int col0, ncols;    // columns [col0, col0 + ncols) of the slab
  long long ld;
  int trans;          // 0: dst[m * ld + c];  1: dst[c * ld + m]
  long long split_stride;  // per-split outputs: elements between consecutive splits' results
  int vec4;           // 1: four consecutive columns per thread (16-byte slab loads; host checks the
                      // alignment: col0, ncols multiples of 4, and for trans 0 an 8-byte-aligned
                      // destination row of 4-column groups)
};

struct RedParams {
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

// RoPE helpers ("Model Patches and Kernels", RoPE):
//  * rope_rotate: rotates the heads of up to two bf16 [M x n] tensors pair by pair,
//    (c, c + half) of each head, by sign * the angle of each token's position (sign
//    -1: the transpose rotation, which turns the gradient of rotated q, k into the
//    gradient of the projections' outputs).
//  * rope_table: cos and sin of p * base^(-2i/head_dim), computed in double.
struct RopeParams {
  const __nv_bfloat16* src[2];
  __nv_bfloat16* dst[2];
  long long n[2];          // columns of each tensor (a multiple of 2 * half)
  int ntensors;
  long long M;
  const float* cos;        // [npos x half]
  const float* sin;
  const int* pos;          // [M]
  int half;
  int npos;
  float sign;
  unsigned* status;
};

struct RopeTableParams {
  float* cos;
  float* sin;
  long long npos;
  int half;
  double base;
};

}  // namespace lgb
