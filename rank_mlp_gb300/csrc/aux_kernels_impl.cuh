// Kernel bodies of the pack, reduce, norms and RoPE kernels (parameter structs in
// aux_kernels.cuh).
// Included by exactly one translation unit, the one that launches them.
#pragma once

#include "aux_kernels.cuh"
#include "gemm_tc.cuh"

namespace lgb {

// Eight consecutive destination elements of one row per thread (destination widths
// are multiples of 8 and rows start 16-byte aligned): each block that overlaps them
// contributes a run of columns read with one stride, the rest stay zero; one 16-byte
// store.  Index arithmetic is 32-bit (the host keeps rows * cols below 2^31).
__global__ void __launch_bounds__(256) pack_kernel(const __grid_constant__ PackParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const PackJob& J = p.job[blockIdx.y];
  const int cols8 = J.cols / 8;
  const int total = J.rows * cols8;
  for (int idx = blockIdx.x * 256 + threadIdx.x; idx < total; idx += 256 * gridDim.x) {
    const int a = idx / cols8;
    const int b0 = (idx - a * cols8) * 8;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.0f;
    for (int k = 0; k < J.nblk; ++k) {
      const PackBlock& B = J.blk[k];
      const int i = a - B.ro, j0 = b0 - B.co;
      if (i < 0 || i >= B.R || j0 + 8 <= 0 || j0 >= B.C) continue;
      const long long step = B.trans ? B.lds : 1;
      const __nv_bfloat16* src = B.src + (B.trans ? static_cast<long long>(i) : static_cast<long long>(i) * B.lds);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = j0 + e;
        if (j >= 0 && j < B.C) v[e] = B.scale * __bfloat162float(src[j * step]);
      }
    }
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
      w[e] = *reinterpret_cast<uint32_t*>(&pr);
    }
    *reinterpret_cast<uint4*>(J.dst + static_cast<long long>(a) * J.cols + b0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void __launch_bounds__(256) reduce_kernel(const __grid_constant__ RedParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const RedOut& O = p.out[blockIdx.y];
  const long long total = static_cast<long long>(O.rows) * O.ncols;
  const long long slab = O.rows_pad * O.width;
  if (O.vec4 && !O.per_split) {
    // Four columns per thread: the same sums, in the same order, as the scalar loop
    // below.  trans 0: threads take consecutive 4-column groups of a row (16-byte loads,
    // 8-byte stores); trans 1: consecutive rows of one group (each column's stores
    // are consecutive in the destination).
    const int groups = O.ncols / 4;
    const int n = O.rows * groups;
    for (int idx = blockIdx.x * 256 + threadIdx.x; idx < n; idx += 256 * gridDim.x) {
      int m, g;
      if (O.trans) {
        g = idx / O.rows;
        m = idx - g * O.rows;
      } else {
        m = idx / groups;
        g = idx - m * groups;
      }
      const float* src = O.part + static_cast<long long>(m) * O.width + O.col0 + 4 * g;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
      for (int k = 0; k < O.splits; ++k) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src + k * slab));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const __nv_bfloat16 b0 = __float2bfloat16_rn(O.scale * acc.x), b1 = __float2bfloat16_rn(O.scale * acc.y);
      const __nv_bfloat16 b2 = __float2bfloat16_rn(O.scale * acc.z), b3 = __float2bfloat16_rn(O.scale * acc.w);
      if (O.trans) {
        __nv_bfloat16* d = O.dst + static_cast<long long>(4 * g) * O.ld + m;
        d[0] = b0;
        d[O.ld] = b1;
        d[2 * O.ld] = b2;
        d[3 * O.ld] = b3;
      } else {
        __nv_bfloat162 lo, hi;
        lo.x = b0;
        lo.y = b1;
        hi.x = b2;
        hi.y = b3;
        uint2 w;
        w.x = *reinterpret_cast<uint32_t*>(&lo);
        w.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(O.dst + static_cast<long long>(m) * O.ld + 4 * g) = w;
      }
    }
    return;
  }
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
    if (O.per_split) {
      for (int k = 0; k < O.splits; ++k) O.dst[k * O.split_stride + d] = __float2bfloat16_rn(O.scale * src[k * slab]);
    } else {
      float s = 0.0f;
      for (int k = 0; k < O.splits; ++k) s += src[k * slab];
      O.dst[d] = __float2bfloat16_rn(O.scale * s);
    }
  }
}

__global__ void __launch_bounds__(256) norms_kernel(const __grid_constant__ NormParams p) {
  pdl_wait();
  pdl_launch_dependents();
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

// One thread per 8 pairs: columns [c, c + 8) and [c + half, c + half + 8) of a head.
__global__ void __launch_bounds__(256) rope_rotate_kernel(const __grid_constant__ RopeParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.y;
  const long long groups_per_row = p.n[t] / 16;       // (n / head_dim) heads x (half / 8)
  const long long total = p.M * groups_per_row;
  const int gph = p.half / 8;
  for (long long it = blockIdx.x * 256ll + threadIdx.x; it < total; it += 256ll * gridDim.x) {
    const long long m = it / groups_per_row;
    const int rem = static_cast<int>(it - m * groups_per_row);
    const int head = rem / gph, g = rem - head * gph;
    const long long ca = static_cast<long long>(head) * 2 * p.half + 8 * g, cb = ca + p.half;
    int pos = __ldg(p.pos + m);
    if (pos < 0 || pos >= p.npos) {
      if (p.status) atomicOr(p.status, kStatusInput);
      pos = 0;
    }
    const uint4 ua = __ldg(reinterpret_cast<const uint4*>(p.src[t] + m * p.n[t] + ca));
    const uint4 ub = __ldg(reinterpret_cast<const uint4*>(p.src[t] + m * p.n[t] + cb));
    const float4* cr = reinterpret_cast<const float4*>(p.cos + static_cast<long long>(pos) * p.half + 8 * g);
    const float4* sr = reinterpret_cast<const float4*>(p.sin + static_cast<long long>(pos) * p.half + 8 * g);
    const float4 c0 = __ldg(cr), c1 = __ldg(cr + 1), s0 = __ldg(sr), s1 = __ldg(sr + 1);
    const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
    uint32_t oa[4], ob[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float ra[2], rb[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float x0 = h ? __uint_as_float(wa[e] & 0xFFFF0000u) : __uint_as_float(wa[e] << 16);
        const float x1 = h ? __uint_as_float(wb[e] & 0xFFFF0000u) : __uint_as_float(wb[e] << 16);
        const float c = cc[2 * e + h], sn = p.sign * ss[2 * e + h];
        ra[h] = x0 * c - x1 * sn;
        rb[h] = x1 * c + x0 * sn;
      }
      __nv_bfloat162 va = __floats2bfloat162_rn(ra[0], ra[1]);
      __nv_bfloat162 vb = __floats2bfloat162_rn(rb[0], rb[1]);
      oa[e] = *reinterpret_cast<uint32_t*>(&va);
      ob[e] = *reinterpret_cast<uint32_t*>(&vb);
    }
    *reinterpret_cast<uint4*>(p.dst[t] + m * p.n[t] + ca) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    *reinterpret_cast<uint4*>(p.dst[t] + m * p.n[t] + cb) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

__global__ void __launch_bounds__(256) rope_table_kernel(const __grid_constant__ RopeTableParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const long long total = p.npos * p.half;
  for (long long it = blockIdx.x * 256ll + threadIdx.x; it < total; it += 256ll * gridDim.x) {
    const long long pos = it / p.half;
    const int i = static_cast<int>(it - pos * p.half);
    const double theta = pow(p.base, -static_cast<double>(i) / p.half);   // base^(-2i/d)
    double sn, cs;
    sincos(static_cast<double>(pos) * theta, &sn, &cs);
    p.cos[it] = static_cast<float>(cs);
    p.sin[it] = static_cast<float>(sn);
  }
}

}  // namespace lgb
