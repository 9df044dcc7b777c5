// Kernel bodies of the pack and reduce kernels (parameter structs in aux_kernels.cuh).
// Included by exactly one translation unit, the one that launches them.
#pragma once

#include "aux_kernels.cuh"

namespace lgb {

__global__ void __launch_bounds__(256) pack_kernel(const __grid_constant__ PackParams p) {
  const PackJob& J = p.job[blockIdx.y];
  const long long total = static_cast<long long>(J.rows) * J.cols;
  for (long long idx = blockIdx.x * 256LL + threadIdx.x; idx < total; idx += 256LL * gridDim.x) {
    const int a = static_cast<int>(idx / J.cols);
    const int b = static_cast<int>(idx - static_cast<long long>(a) * J.cols);
    float v = 0.0f;
    for (int k = 0; k < J.nblk; ++k) {
      const PackBlock& B = J.blk[k];
      const int i = a - B.ro, j = b - B.co;
      if (i >= 0 && i < B.R && j >= 0 && j < B.C) {
        const long long s = B.trans ? static_cast<long long>(j) * B.lds + i
                                    : static_cast<long long>(i) * B.lds + j;
        v = B.scale * __bfloat162float(B.src[s]);
      }
    }
    J.dst[idx] = __float2bfloat16_rn(v);
  }
}

__global__ void __launch_bounds__(256) reduce_kernel(const __grid_constant__ RedParams p) {
  const RedOut& O = p.out[blockIdx.y];
  const long long total = static_cast<long long>(O.rows) * O.ncols;
  const long long slab = O.rows_pad * O.width;
  for (long long idx = blockIdx.x * 256LL + threadIdx.x; idx < total; idx += 256LL * gridDim.x) {
    int m, c;
    if (O.trans) {
      c = static_cast<int>(idx / O.rows);
      m = static_cast<int>(idx - static_cast<long long>(c) * O.rows);
    } else {
      m = static_cast<int>(idx / O.ncols);
      c = static_cast<int>(idx - static_cast<long long>(m) * O.ncols);
    }
    const float* src = O.part + static_cast<long long>(m) * O.width + O.col0 + c;
    const long long d = O.trans ? static_cast<long long>(c) * O.ld + m : static_cast<long long>(m) * O.ld + c;
    if (p.per_split) {
      for (int k = 0; k < p.splits; ++k) O.dst[k * O.split_stride + d] = __float2bfloat16_rn(p.scale * src[k * slab]);
    } else {
      float s = 0.0f;
      for (int k = 0; k < p.splits; ++k) s += src[k * slab];
      O.dst[d] = __float2bfloat16_rn(p.scale * s);
    }
  }
}

__global__ void __launch_bounds__(256) norms_kernel(const __grid_constant__ NormParams p) {
  const int e = blockIdx.x;
  float acc = 0.0f;
  for (int t = 0; t < p.ntensors; ++t) {
    const __nv_bfloat16* src = p.src[t] + static_cast<long long>(e) * p.count[t];
    for (long long j = threadIdx.x; j < p.count[t]; j += 256) {
      const float v = __bfloat162float(src[j]);
      acc += v * v;
    }
  }
  __shared__ float red[256];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) p.out[e] = red[0];
}

}  // namespace lgb
