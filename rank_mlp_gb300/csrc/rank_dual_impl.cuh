// Kernel of the one-pass rank-r products (declarations in rank_dual.cuh).  Included by
// exactly one translation unit, the one that launches it.
#pragma once

#include "rank_dual.cuh"

namespace lgb {

// Bounded waits (the GEMM kernels' rule: wall-clock limit, abort flag shared by the CTA).
__device__ __forceinline__ bool dual_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const DualParams& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > p.timeout_ns) {
      *abort_flag = 1;
      if (p.status) atomicOr(p.status, kStatusTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ void dual_wait_drain(uint32_t bar, uint32_t parity, const DualParams& p) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 20000000ull) {
      if (p.status) atomicOr(p.status, kStatusTimeout);
      return;
    }
  }
}

// Feature block kb of the concatenated products: its product and local block.
__device__ __forceinline__ void dual_block(const DualParams& p, int kb, int& prod, int& lb) {
  prod = 0;
  lb = kb;
  while (prod + 1 < p.nprod && lb >= p.prod[prod].nkb) {
    lb -= p.prod[prod].nkb;
    ++prod;
  }
}

__global__ void __launch_bounds__(kThreads, 1) rank_dual_kernel(const __grid_constant__ DualParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t tbase = sbase + kDualStages * kDualStageBytes;          // two T^T slots
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDualStages * kDualStageBytes + 2 * kDualSlotBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kDualNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kDualStages + s); };
  auto vfull_bar = [&](int a) { return bar0 + 8u * (2 * kDualStages + a); };
  auto vempty_bar = [&](int a) { return bar0 + 8u * (2 * kDualStages + 2 + a); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kDualStages + 4 + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kDualStages + 6 + a); };
  const uint32_t dbfull_bar = bar0 + 8u * (2 * kDualStages + 8);
  // (the drain barrier of an aborted MMA lane reuses dbfull: nothing else waits on it then)

  // this CTA's token tiles [t0, t1) and feature blocks [k0, k1)
  const int cta = static_cast<int>(blockIdx.x);
  const int gti = cta / p.gf, gfi = cta - (cta / p.gf) * p.gf;
  const int t0 = static_cast<int>(static_cast<long long>(p.tiles_m) * gti / p.gt);
  const int t1 = static_cast<int>(static_cast<long long>(p.tiles_m) * (gti + 1) / p.gt);
  const int k0 = static_cast<int>(static_cast<long long>(p.kb_total) * gfi / p.gf);
  const int k1 = static_cast<int>(static_cast<long long>(p.kb_total) * (gfi + 1) / p.gf);
  // products with feature blocks in this range (bit p)
  unsigned present = 0;
  {
    int base = 0;
    for (int q = 0; q < p.nprod; ++q) {
      if (k0 < base + p.prod[q].nkb && k1 > base) present |= 1u << q;
      base += p.prod[q].nkb;
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDualStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(vfull_bar(a), 1);
      mbar_init(vempty_bar(a), 4);
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 1);
    }
    mbar_init(dbfull_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < 3 * p.nprod) tma_prefetch_map(&p.maps[lane]);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kDualTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[kDualStages];
      for (int s = 0; s < kDualStages; ++s) armed[s] = -1;
      int tarmed[2] = {-1, -1};
      bool ok = true;
      const uint32_t tbytes = static_cast<uint32_t>(__popc(present)) * 2u * 64u * p.nr * 2u;
      const uint32_t sbytes = static_cast<uint32_t>(kDualQBytes + 2 * 64 * p.nv * 2);
      for (int t = t0; t < t1 && ok; ++t) {
        const int slot = (t - t0) & 1;
        const uint32_t tphase = static_cast<uint32_t>(((t - t0) >> 1) & 1);
        // the transposed rank-r operand of this token tile, once for all its blocks
        if (!dual_wait(tempty_bar(slot), tphase ^ 1u, abort_flag, p)) { ok = false; break; }
        mbar_arrive_expect_tx(tfull_bar(slot), tbytes);
        tarmed[slot] = static_cast<int>(tphase);
        for (int q = 0; q < p.nprod; ++q) {
          if (!((present >> q) & 1u)) continue;
          const uint32_t dst = tbase + slot * kDualSlotBytes + q * kDualTBytes;
          for (int c = 0; c < 2; ++c)
            tma_load_2d(dst + c * (p.nr * 128), &p.maps[p.prod[q].t_map], tfull_bar(slot), t * 128 + 64 * c,
                        p.prod[q].t_row);
        }
        for (int kb = k0; kb < k1; ++kb) {
          int q, lb;
          dual_block(p, kb, q, lb);
          if (!dual_wait(empty_bar(stage), phase ^ 1u, abort_flag, p)) { ok = false; break; }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, sbytes);
          armed[stage] = static_cast<int>(phase);
          const uint32_t sq = sbase + stage * kDualStageBytes;
          const uint32_t sb = sq + kDualQBytes;
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(sq + c * (kDualQBytes / 2), &p.maps[p.prod[q].q_map], fb, lb * 128 + 64 * c, t * 128);
            tma_load_2d(sb + c * (p.nv * 128), &p.maps[p.prod[q].b_map], fb, lb * 128 + 64 * c, 0);
          }
          if (++stage == kDualStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        for (int s = 0; s < kDualStages; ++s)
          if (armed[s] >= 0) dual_wait_drain(full_bar(s), static_cast<uint32_t>(armed[s]), p);
        for (int s = 0; s < 2; ++s)
          if (tarmed[s] >= 0) dual_wait_drain(tfull_bar(s), static_cast<uint32_t>(tarmed[s]), p);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_v = idesc_bf16_f32(128, p.nv, 0, 0);
      const uint32_t idesc_b = idesc_bf16_f32(128, p.nr, 1, 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = t0; t < t1 && ok; ++t) {
        const int slot = (t - t0) & 1;
        const uint32_t tphase = static_cast<uint32_t>(((t - t0) >> 1) & 1);
        const int vb = (t - t0) & 1;
        const uint32_t vphase = static_cast<uint32_t>(((t - t0) >> 1) & 1);
        if (!dual_wait(vempty_bar(vb), vphase ^ 1u, abort_flag, p)) { ok = false; break; }
        if (!dual_wait(tfull_bar(slot), tphase, abort_flag, p)) { ok = false; break; }
        const uint32_t vacc = tmem_base + static_cast<uint32_t>(vb * kDualNVMax);
        for (int kb = k0; kb < k1; ++kb) {
          int q, lb;
          dual_block(p, kb, q, lb);
          if (!dual_wait(full_bar(stage), phase, abort_flag, p)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t sq = sbase + stage * kDualStageBytes;
          const uint32_t sb = sq + kDualQBytes;
          const uint32_t st = tbase + slot * kDualSlotBytes + q * kDualTBytes;
          const uint32_t dacc = tmem_base + static_cast<uint32_t>(kDualVCols + (kb - k0) * p.nr);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            // projection: tokens x features (K-major Q) times B^T rows
            const uint64_t a = smem_desc_sw128(sq + (k >> 2) * (kDualQBytes / 2) + (k & 3) * 32, 16u, 1024u);
            const uint64_t b = smem_desc_sw128(sb + (k >> 2) * (p.nv * 128) + (k & 3) * 32, 16u, 1024u);
            tc_mma_bf16(vacc, a, b, idesc_v, (kb > k0 || k > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            // reduction: features x tokens (Q read MN-major) times T^T rows
            const uint64_t a = smem_desc_sw128(sq + k * 2048, kDualQBytes / 2, 1024u);
            const uint64_t b = smem_desc_sw128(st + (k >> 2) * (p.nr * 128) + (k & 3) * 32, 16u, 1024u);
            tc_mma_bf16(dacc, a, b, idesc_b, (t > t0 || k > 0) ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
          if (++stage == kDualStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(vfull_bar(vb));        // this token tile's projection is complete
        tc_commit(tempty_bar(slot));     // and its T^T slot free
      }
      if (ok) {
        tc_commit(dbfull_bar);           // every reduction block is complete
      } else {
        tc_commit(dbfull_bar);
        dual_wait_drain(dbfull_bar, 0, p);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;             // TMEM lane quarter of this warp
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    bool ok = true;
    for (int t = t0; t < t1; ++t) {
      const int vb = (t - t0) & 1;
      const uint32_t vphase = static_cast<uint32_t>(((t - t0) >> 1) & 1);
      const bool ready = dual_wait(vfull_bar(vb), vphase, abort_flag, p);
      if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
      tc_fence_after_sync();
      const uint32_t vacc = tmem_base + lane_off + static_cast<uint32_t>(vb * kDualNVMax);
      const long long row = static_cast<long long>(t) * 128 + q4 * 32 + lane;
      float* dst = p.v_part + (static_cast<long long>(gfi) * p.tiles_m * 128 + row) * p.nv;
      for (int c = 0; c < p.nv; c += 16) {
        uint32_t v[16];
        __syncwarp();
        tmem_ld16(vacc + c, v);
        tmem_ld_wait();
        st_global_v8(dst + c, v);
        st_global_v8(dst + c + 8, v + 8);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(vempty_bar(vb));
    }
    if (ok) {
      const bool ready = dual_wait(dbfull_bar, 0, abort_flag, p);
      if (__all_sync(0xffffffffu, ready)) {
        tc_fence_after_sync();
        for (int kb = k0; kb < k1; ++kb) {
          int q, lb;
          dual_block(p, kb, q, lb);
          const DualProduct& P = p.prod[q];
          const long long f = static_cast<long long>(lb) * 128 + q4 * 32 + lane;
          float* dst = P.db_part + (static_cast<long long>(gti) * P.nkb * 128 + f) * p.nr;
          uint32_t v[16];
          __syncwarp();
          tmem_ld16(tmem_base + lane_off + static_cast<uint32_t>(kDualVCols + (kb - k0) * p.nr), v);
          tmem_ld_wait();
          st_global_v8(dst, v);
          st_global_v8(dst + 8, v + 8);
        }
      }
    }
  }

  if (*abort_flag) settle_after_abort();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kDualTmemCols);
  }
}

}  // namespace lgb
