// The projection GEMM on a CTA pair (cluster of 2, tcgen05 cta_group::2): one
// 256 x 256 output tile per pair and step.  Each CTA loads its own 128 rows of A and
// one half (128 rows) of the B tile; the even CTA issues 256 x 256 x 16 MMAs that read
// A from both CTAs and B from both halves, so each SM's shared memory moves half of B
// instead of all of it.  Each CTA's TMEM holds its 128 accumulator rows (two
// 256-column buffers) and its own epilogue warps drain them.
//
// Barriers: the even CTA's `full` barrier counts the bytes of both CTAs' copies (it
// alone arms it); the MMA's commits arrive on `empty` and `tfull` of both CTAs
// (multicast); both CTAs' epilogue warps arrive on the even CTA's `tempty`.
// Gate/up tiles put the gate rows in the even CTA's half and the matching up rows in
// the odd CTA's half, so accumulator columns 0-127 are g and 128-255 are u.
#pragma once

#include "gemm_tc.cuh"

namespace lgb {

// Threads of a pair-kernel CTA: producer warp, MMA warp and EPIW epilogue warps.
constexpr int pair_threads(int epiw) { return 64 + 32 * epiw; }

template <int STAGES>
struct PairCfg {
  static constexpr int BN = 256;                       // accumulator columns per tile
  static constexpr int kBLocal = BN / 2;               // B rows held by each CTA
  static constexpr int kABytes = kBM * kBK * 2;        // this CTA's 128 rows of A
  static constexpr int kBBytes = kBLocal * kBK * 2;    // this CTA's half of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTxBytes = 2 * kStageBytes;     // both CTAs, counted on the even CTA
  static constexpr int kTmemCols = 512;
  static constexpr int kBarBytes = 8 * (2 * STAGES + 5) + 16;
  static constexpr int kSmemBytes = STAGES * kStageBytes + kBarBytes + 1024;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
};

// The 32-column accumulator chunks (bit k: columns 32k .. 32k + 31) that epilogue_tile
// reads for the warp with share `part` of `nparts`: the warp's own columns for the
// plain, derivative and partial epilogues; matching gate and up halves for the
// activation epilogue; both chunks of each rotation pair it owns for RoPE.
template <int BN>
__device__ __forceinline__ unsigned epilogue_chunks(const TcParams& p, int epi, int part, int nparts) {
  constexpr int kChunks = BN / 32;
  unsigned m = 0;
  if (epi == EPI_ACT_FWD) {
    const int per = kChunks / 2 / nparts;
    for (int j = 0; j < per; ++j) m |= (1u << (part * per + j)) | (1u << (kChunks / 2 + part * per + j));
  } else if (epi == EPI_ROPE) {
    const int half = p.rope_half, cph = half / 32;
    for (int t = part; t < BN / 64; t += nparts) {
      const int col = (t / cph) * 2 * half + (t % cph) * 32;
      m |= (1u << (col / 32)) | (1u << ((col + half) / 32));
    }
  } else {
    const int per = kChunks / nparts;
    for (int j = 0; j < per; ++j) m |= 1u << (part * per + j);
  }
  return m;
}

// A split-tail piece's epilogue step, for one epilogue warp: its TMEM lane quarter
// (rows `row` of the CTA's 128) and the column chunks its epilogue reads
// (epilogue_chunks).  The warp stores the piece's partial sums for those rows and
// columns, then counts its arrival on the word of (tile, CTA, warp).  Every piece's
// warp with the same role covers the same rows and columns, so each warp's word counts
// its own share of the tile, and a warp that finishes the tile has fixed up everything
// its epilogue then reads.  The last arrival sums the pieces' partials in piece order
// (its own from TMEM, bit-identical to what it stored), writes the total back to TMEM
// and returns true: the caller then runs the epilogue on it.  Earlier arrivals return
// false.
//
// Partial slots: piece s of tail tile t uses slot t * sk_splits + s, which holds
// [2 CTAs][BN/32 column chunks][128 rows][32] f32.  Arrival words hold
// (sk_epoch << 8) + arrivals: a word from another launch counts as zero arrivals, and
// the last arrival resets it, so the same launch replayed (a CUDA graph) counts again
// from zero.
template <int BN>
__device__ __forceinline__ bool sk_piece_arrive(const TcParams& p, const GroupDesc& G, const Unit& U, uint32_t tacc,
                                                int cta, int row, int part, int nparts, int widx) {
  const int lane = threadIdx.x & 31;
  const unsigned mask = epilogue_chunks<BN>(p, G.epi, part, nparts);
  auto chunk = [&](long long slot, int c) -> float* {
    return p.sk_part + (((slot * 2 + cta) * (BN / 32) + c / 32) * kBM + row) * 32;
  };
  const long long slot0 = static_cast<long long>(U.sk_tile) * U.npieces;
  // this piece's partial sums
  const long long mine = slot0 + U.piece;
#pragma unroll 1
  for (int ch = 0; ch < BN / 32; ++ch) {
    if (!((mask >> ch) & 1u)) continue;
    const int c = ch * 32;
    uint32_t v[32];
    __syncwarp();
    tmem_ld32(tacc + c, v);
    tmem_ld_wait();
    float* dst = chunk(mine, c);
#pragma unroll
    for (int j = 0; j < 32; j += 8) st_global_v8(dst + j, v + j);
  }
  __threadfence();
  __syncwarp();
  // count the arrival
  int last = 0;
  if (lane == 0) {
    unsigned long long* w = p.sk_flags + (static_cast<long long>(U.sk_tile) * 2 + cta) * kSkWarps + widx;
    const unsigned long long tag = p.sk_epoch << 8;
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(w);
    for (int n = 0; n < 64; ++n) {     // each failed exchange means another piece arrived
      const unsigned long long base = (cur & ~0xffull) == tag ? cur : tag;
      const unsigned long long seen = atomicCAS(w, cur, base + 1);
      if (seen == cur) {
        last = static_cast<int>((base + 1) & 0xffull) == U.npieces;
        break;
      }
      cur = seen;
    }
    if (last) atomicExch(w, tag);
    __threadfence();
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return false;
  __threadfence();
  // the tile's total, in piece order, 8 columns at a time
#pragma unroll 1
  for (int c = 0; c < BN; c += 8) {
    if (!((mask >> (c / 32)) & 1u)) continue;
    uint32_t v[8];
    __syncwarp();
    tmem_ld8(tacc + c, v);
    tmem_ld_wait();
    float acc[8];
#pragma unroll 1
    for (int j = 0; j < U.npieces; ++j) {
      float x[8];
      if (j == U.piece) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(v[e]);
      } else {
        const float* src = chunk(slot0 + j, c & ~31) + (c & 31);
        const uint4 w0 = ld_global_cg_v4(src), w1 = ld_global_cg_v4(src + 4);
        x[0] = __uint_as_float(w0.x);
        x[1] = __uint_as_float(w0.y);
        x[2] = __uint_as_float(w0.z);
        x[3] = __uint_as_float(w0.w);
        x[4] = __uint_as_float(w1.x);
        x[5] = __uint_as_float(w1.y);
        x[6] = __uint_as_float(w1.z);
        x[7] = __uint_as_float(w1.w);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = j == 0 ? x[e] : acc[e] + x[e];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __float_as_uint(acc[e]);
    tmem_st8(tacc + c, v);
  }
  tmem_st_wait();
  return true;
}

// EPIW = 4 or 8 epilogue warps: with 8, two warps share each TMEM lane quarter and
// take half of the tile's columns each (more loads in flight for epilogues that read
// saved tensors); with 4, fewer warps compete for issue slots with the producer and
// MMA lanes (better for arithmetic-heavy epilogues).
template <int STAGES, bool B_MN, int EPIW>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads(EPIW), 1)
    tc_gemm_pair_kernel(const __grid_constant__ TcParams p) {
  static_assert(EPIW == 4 || EPIW == 8, "epilogue warps");
  using C = PairCfg<STAGES>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int npairs = static_cast<int>(gridDim.x >> 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * EPIW);  // every epilogue warp of both CTAs (even CTA's)
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < p.nmaps) tma_prefetch_map(&p.maps[lane]);
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();                     // both CTAs' barriers exist before any remote arrive
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();                             // the previous kernel's writes are visible from here
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = -1;
      bool ok = true;
      bool first_stage = true;
      WorkIter it(p, pair, npairs);
      Unit U;
      while (ok && it.next(p, U)) {
        const GroupDesc& G = p.grp[U.g];
        // walk the unit's k-range segment by segment; a segment's fields live in registers
        const int nseg = G.nseg;
        int seg_base = 0;
        for (int sg = 0; sg < nseg && ok; ++sg) {
          const int nkb = G.seg[sg].kblocks;
          const int j0 = max(U.kb0 - seg_base, 0), j1 = min(U.kb1 - seg_base, nkb);
          const CUtensorMap* ma = &p.maps[G.seg[sg].a];
          const int b0 = G.seg[sg].b0, b1 = G.seg[sg].b1;
          const CUtensorMap* mb = &p.maps[(rank && b1 >= 0) ? b1 : b0];
          const int a_row = U.tm * (2 * kBM) + static_cast<int>(rank) * kBM;
          const int b_row = (b1 >= 0) ? U.tn * C::kBLocal : U.tn * BN + static_cast<int>(rank) * C::kBLocal;
          seg_base += nkb;
          for (int j = j0; j < j1; ++j) {
            const int kc = j * kBK;
            if (!wait_phase(empty_bar(stage), phase ^ 1u, abort_flag, p)) { ok = false; break; }
            const uint32_t fb = full_bar(stage);
            if (p.inject_stall && first_stage && leader) {   // failure-path tests: never arm it
              first_stage = false;
              if (++stage == STAGES) { stage = 0; phase ^= 1u; }
              continue;
            }
            first_stage = false;
            if (leader) {
              mbar_arrive_expect_tx(fb, C::kTxBytes);
              armed[stage] = static_cast<int>(phase);
            }
            const uint32_t fb_even = mapa_shared(fb, 0);
            const uint32_t sa = sbase + stage * C::kStageBytes;
            const uint32_t sb = sa + C::kABytes;
            tma_load_2d_pair(sa, ma, fb_even, kc, a_row);
            if (!B_MN) {
              tma_load_2d_pair(sb, mb, fb_even, kc, b_row);
            } else {
#pragma unroll
              for (int c = 0; c < C::kBLocal / 64; ++c) tma_load_2d_pair(sb + c * 8192u, mb, fb_even, b_row + c * 64, kc);
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
      if (!ok && leader) {
        for (int s = 0; s < STAGES; ++s)
          if (armed[s] >= 0) wait_phase_drain(full_bar(s), static_cast<uint32_t>(armed[s]), p);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, BN, 0, B_MN ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      WorkIter it(p, pair, npairs);
      Unit U;
      while (ok && it.next(p, U)) {
        const GroupDesc& G = p.grp[U.g];
        if (!wait_phase(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        uint32_t accumulate = 0;
        const int nseg = G.nseg;
        int seg_base = 0;
        for (int sg = 0; sg < nseg && ok; ++sg) {
          const int nkb = G.seg[sg].kblocks, kvalid = G.seg[sg].kvalid;
          const int j0 = max(U.kb0 - seg_base, 0), j1 = min(U.kb1 - seg_base, nkb);
          seg_base += nkb;
          for (int j = j0; j < j1; ++j) {
            const int kc = j * kBK;
            if (!wait_phase(full_bar(stage), phase, abort_flag, p)) { ok = false; break; }
            tc_fence_after_sync();
            const uint32_t sa = sbase + stage * C::kStageBytes;
            const uint32_t sb = sa + C::kABytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              if (kc + 16 * k < kvalid) {
                const uint64_t adesc = smem_desc_sw128(sa + 32u * k, 16u, 1024u);
                const uint64_t bdesc = B_MN ? smem_desc_sw128(sb + 2048u * k, 8192u, 1024u)
                                            : smem_desc_sw128(sb + 32u * k, 16u, 1024u);
                tc_mma_bf16_pair(d_tmem, adesc, bdesc, idesc, accumulate);
                accumulate = 1;
              }
            }
            tc_commit_pair_multicast(empty_bar(stage), 0x3);   // frees this stage in both CTAs
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(tfull_bar(acc), 0x3);       // both halves of the tile ready
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        tc_commit_pair_multicast(drain_bar, 0x1);
        wait_phase_drain(drain_bar, 0, p);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // EPIW / 4 warps per TMEM lane quarter, each taking a share of the tile's columns
    const int q = warp & 3;
    const int part = (warp - 2) >> 2;
    const int row_in_tile = q * 32 + lane;
    const uint32_t tempty_even[2] = {mapa_shared(tempty_bar(0), 0), mapa_shared(tempty_bar(1), 0)};
    int acc = 0;
    uint32_t acc_phase = 0;
    WorkIter it(p, pair, npairs);
    Unit U;
    while (it.next(p, U)) {
      const GroupDesc& G = p.grp[U.g];
      const bool ready = wait_phase(tfull_bar(acc), acc_phase, abort_flag, p);
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after_sync();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      // a split-tail piece: the last piece of its tile to arrive finishes the tile
      const bool finish = U.npieces == 1 ||
                          sk_piece_arrive<BN>(p, G, U, tacc, static_cast<int>(rank), row_in_tile, part, EPIW / 4,
                                              warp - 2);
      if (finish)
        epilogue_tile<BN>(p, G, U, tacc, U.tm * (2 * kBM) + static_cast<int>(rank) * kBM + row_in_tile, part,
                          EPIW / 4);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_even[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  if (*abort_flag) settle_after_abort();
  __syncwarp();
  tc_fence_before_sync();
  cluster_sync_all();                     // no remote arrive or MMA read of either CTA is pending
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

}  // namespace lgb
