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

// Staged epilogue (the activation-derivative GEMM): each epilogue warp owns a ring of
// SLOTS slots in shared memory; a slot holds one chunk (the warp's 32 rows x ECOLS
// columns) of g and of u, loaded by TMA, and then the chunk's dg and du, written in
// place and stored by TMA.
constexpr int epi_tensor_bytes(int ecols) { return 32 * ecols * 2; }   // one tensor's chunk
constexpr int epi_slot_bytes(int ecols) { return 2 * epi_tensor_bytes(ecols); }

// STAGED = 0 (plain epilogues) or the staged epilogue's slots per warp, of ECOLS columns.
template <int STAGES, int EPIW = 4, int STAGED = 0, int ECOLS = 16>
struct PairCfg {
  static constexpr int BN = 256;                       // accumulator columns per tile
  static constexpr int kBLocal = BN / 2;               // B rows held by each CTA
  static constexpr int kABytes = kBM * kBK * 2;        // this CTA's 128 rows of A
  static constexpr int kBBytes = kBLocal * kBK * 2;    // this CTA's half of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTxBytes = 2 * kStageBytes;     // both CTAs, counted on the even CTA
  static constexpr int kTmemCols = 512;
  static constexpr int kEpiBytes = EPIW * STAGED * epi_slot_bytes(ECOLS);
  static constexpr int kNumBars = 2 * STAGES + 5 + EPIW * STAGED;
  static constexpr int kBarBytes = 8 * kNumBars + 16;
  static constexpr int kSmemBytes = STAGES * kStageBytes + kEpiBytes + kBarBytes + 1024;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
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

// dg = dh u act'(g), du = dh act(g) for 16 columns of one row ("Model Patches and
// Kernels", activation table: the derivative of the activation, recomputed from the
// saved g): d the accumulator (dh), gw, uw the saved bf16 pairs; results as bf16 pairs.
template <int ACT>
__device__ __forceinline__ void act_bwd_cols(const uint32_t* d, const uint32_t (&gw)[8], const uint32_t (&uw)[8],
                                             uint32_t (&dg)[8], uint32_t (&du)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float a0, ap0, a1, ap1;
    const float g0 = bf16_lo(gw[e]), g1 = bf16_hi(gw[e]);
    const float u0 = bf16_lo(uw[e]), u1 = bf16_hi(uw[e]);
    act_fwd_bwd<ACT>(g0, a0, ap0);
    act_fwd_bwd<ACT>(g1, a1, ap1);
    const float d0 = __uint_as_float(d[2 * e]), d1 = __uint_as_float(d[2 * e + 1]);
    dg[e] = pack_bf16x2(d0 * u0 * ap0, d1 * u1 * ap1);
    du[e] = pack_bf16x2(d0 * a0, d1 * a1);
  }
}

// The staged activation-derivative epilogue of one epilogue warp (its TMEM lane
// quarter q = warp & 3, its share of the tile's columns), for all its units.  The
// warp walks its chunks of 32 rows x COLS columns in order across tiles; lane 0 keeps
// the TMA loads of g, u SLOTS - 1 chunks ahead (into the slot whose dg, du store has
// finished reading it), so the next tile's first loads fly while the warp waits for
// that tile's accumulator.  Each chunk: wait for its slot, read dh from TMEM (16 columns
// at a time, each read issued before the math of the half before it), compute, write
// dg, du over g, u, make them visible to TMA and store both.  The accumulator is
// released as soon as the tile's last chunk has been read from TMEM.  Rows past M and
// columns past N are zero-filled by the loads and dropped by the stores.  The chunk's
// 64-byte rows sit in the 64-byte swizzle: 16-byte unit j of row r at unit j ^ (r >> 1 & 3).
template <int STAGES, int EPIW, int SLOTS, int COLS>
__device__ __forceinline__ void staged_act_bwd(const TcParams& p, uint32_t epi_smem, uint32_t epi_bar0,
                                               uint32_t tfull0, const uint32_t (&tempty_even)[2], uint32_t tmem_base,
                                               volatile int* abort_flag, uint32_t rank, int pair, int npairs,
                                               int warp) {
  static_assert(SLOTS >= 2 && SLOTS <= 8, "ring slots");
  static_assert(COLS == 32, "chunk columns");
  constexpr int BN = 256;
  constexpr int kParts = EPIW / 4;
  constexpr int kSpan = BN / kParts;                   // columns per warp
  constexpr int kChunks = kSpan / COLS;                // chunks per warp per tile
  constexpr int kTensorBytes = epi_tensor_bytes(COLS);
  constexpr int kSlotBytes = epi_slot_bytes(COLS);
  const int lane = threadIdx.x & 31;
  const int q = warp & 3;
  const int widx = warp - 2;
  const int part = widx >> 2;
  const uint32_t ring = epi_smem + static_cast<uint32_t>(widx) * (SLOTS * kSlotBytes);
  auto slot = [&](uint32_t n) { return ring + (n % SLOTS) * kSlotBytes; };
  auto full = [&](uint32_t n) { return epi_bar0 + 8u * (widx * SLOTS + n % SLOTS); };
  // this lane's row inside a chunk box and where its 16-byte units sit (the swizzle)
  const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
  auto unit_off = [&](int j) { return static_cast<uint32_t>(lane) * (2u * COLS) + ((static_cast<uint32_t>(j) ^ sw) << 4); };

  // the loading cursor: unit and chunk of the next load
  WorkIter ahead(p, pair, npairs);
  Unit UA;
  bool more = ahead.next(p, UA);
  int ca = 0;
  uint32_t issued = 0, used = 0;
  auto issue = [&]() {
    if (lane == 0) {
      const GroupDesc& GA = p.grp[UA.g];
      const int row0 = UA.tm * (2 * kBM) + static_cast<int>(rank) * kBM + q * 32;
      const int col = UA.tn * BN + part * kSpan + ca * COLS;
      const uint32_t b = full(issued), dst = slot(issued);
      mbar_arrive_expect_tx(b, kSlotBytes);
      tma_load_2d(dst, &p.maps[GA.emap[0]], b, col, row0);
      tma_load_2d(dst + kTensorBytes, &p.maps[GA.emap[1]], b, col, row0);
    }
    ++issued;
    if (++ca == kChunks) {
      ca = 0;
      more = ahead.next(p, UA);
    }
  };
  for (int k = 0; k < SLOTS - 1 && more; ++k) issue();

  WorkIter it(p, pair, npairs);
  Unit U;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  while (ok && it.next(p, U)) {
    const GroupDesc& G = p.grp[U.g];
    const bool ready = wait_phase(tfull0 + 8u * acc, acc_phase, abort_flag, p);
    if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
    tc_fence_after_sync();
    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
    const int row0 = U.tm * (2 * kBM) + static_cast<int>(rank) * kBM + q * 32;
    // dh is read from TMEM 16 columns at a time, each read issued one half-chunk ahead of
    // its use, so that its latency overlaps the math of the half before
    uint32_t dlo[16], dhi[16];
    __syncwarp();
    tmem_ld16(tacc + part * kSpan, dlo);
#pragma unroll 1
    for (int c = 0; c < kChunks; ++c) {
      const int col = part * kSpan + c * COLS;
      const bool landed = wait_phase(full(used), (used / SLOTS) & 1u, abort_flag, p);
      tmem_ld_wait();                               // this chunk's first half
      __syncwarp();
      tmem_ld16(tacc + col + 16, dhi);
      if (!__all_sync(0xffffffffu, landed)) {
        tmem_ld_wait();
        ok = false;
        break;
      }
      const uint32_t s0 = slot(used);
      // dg, du of 16 columns (units 2h, 2h + 1 of the lane's row), written over g, u
      auto half = [&](int h, const uint32_t (&d)[16]) {
        const uint32_t off0 = unit_off(2 * h), off1 = unit_off(2 * h + 1);
        const uint4 g0 = ld_shared_v4(s0 + off0), g1 = ld_shared_v4(s0 + off1);
        const uint4 u0 = ld_shared_v4(s0 + kTensorBytes + off0), u1 = ld_shared_v4(s0 + kTensorBytes + off1);
        const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const uint32_t uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        uint32_t dg[8], du[8];
        act_chunk(p.act, [&](auto tag) { act_bwd_cols<decltype(tag)::value>(d, gw, uw, dg, du); });
        st_shared_v4(s0 + off0, make_uint4(dg[0], dg[1], dg[2], dg[3]));
        st_shared_v4(s0 + off1, make_uint4(dg[4], dg[5], dg[6], dg[7]));
        st_shared_v4(s0 + kTensorBytes + off0, make_uint4(du[0], du[1], du[2], du[3]));
        st_shared_v4(s0 + kTensorBytes + off1, make_uint4(du[4], du[5], du[6], du[7]));
      };
      half(0, dlo);
      tmem_ld_wait();                               // this chunk's second half
      if (c + 1 < kChunks) {
        __syncwarp();
        tmem_ld16(tacc + col + COLS, dlo);          // the next chunk's first half
      } else {                                      // the accumulator is no longer needed
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_even[acc]);
      }
      half(1, dhi);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int gcol = U.tn * BN + col;
        tma_store_2d(&p.maps[G.emap[2]], s0, gcol, row0);
        tma_store_2d(&p.maps[G.emap[3]], s0 + kTensorBytes, gcol, row0);
        bulk_commit_group();
      }
      ++used;
      if (more) {
        // the next load goes into the slot of chunk used + SLOTS - 1 - SLOTS = used - 1,
        // whose store must have finished reading it (all stores but the one just
        // committed)
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        issue();
      }
    }
    if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
  }
  if (lane == 0) {
    // loads still in flight (after an abort) land before shared memory is released;
    // every store completes before the kernel ends
    for (uint32_t n = used; n < issued; ++n) wait_phase_drain(full(n), (n / SLOTS) & 1u, p);
    bulk_wait_group_all();
  }
  __syncwarp();
}

// EPIW = 4 or 8 epilogue warps: with 8, two warps share each TMEM lane quarter and
// take half of the tile's columns each (more loads in flight for epilogues that read
// saved tensors); with 4, fewer warps compete for issue slots with the producer and
// MMA lanes (better for arithmetic-heavy epilogues).
//
// ACTB selects the epilogues compiled in: 0 the plain, activation, RoPE and partial
// epilogues (epilogue_tile); the activation-derivative GEMM (every group EPI_ACT_BWD)
// has variants of its own: 1 reads g, u and writes dg, du one row per thread
// (epilogue_act_bwd_rows); 2-8 moves them through the epilogue warps' shared-memory
// rings of that many slots of ECOLS columns (staged_act_bwd; whole tiles only).
template <int STAGES, bool B_MN, int EPIW, int ACTB = 0, int ECOLS = 16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads(EPIW), 1)
    tc_gemm_pair_kernel(const __grid_constant__ TcParams p) {
  static_assert(EPIW == 4 || EPIW == 8, "epilogue warps");
  static_assert(ACTB >= 0 && ACTB <= 8, "epilogue selection");
  constexpr int STAGED = ACTB >= 2 ? ACTB : 0;
  using C = PairCfg<STAGES, EPIW, STAGED, ECOLS>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes + C::kEpiBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
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
    if constexpr (STAGED) {
      for (int k = 0; k < EPIW * STAGED; ++k) mbar_init(bar0 + 8u * (2 * STAGES + 5 + k), 1);
    }
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
  if (p.pdl_seg == 0) {
    pdl_wait();                           // the previous kernel's writes are visible from here
    pdl_launch_dependents();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = -1;
      bool ok = true;
      bool first_stage = true;
      bool waited = p.pdl_seg == 0;
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
          if (!waited && sg >= p.pdl_seg && j0 < j1) {   // the previous kernel's rank-r operand
            pdl_wait();
            // dependents start only after this wait, so that a late-starting one (which
            // reads earlier kernels' outputs at once) finds everything before this
            // kernel complete
            pdl_launch_dependents();
            waited = true;
          }
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
      // This lane's instructions between MMAs are on the tensor pipe's critical path
      // (tcgen05.mma issue keeps only a short queue), so the loop is kept lean: the
      // shared-memory descriptors are those of stage 0 plus constant offsets, and the
      // next stage's data is tested (without blocking) before this stage's last MMA is
      // issued, so the common case needs no wait between stages.
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, BN, 0, B_MN ? 1 : 0);
      const uint64_t adesc0 = smem_desc_sw128(sbase, 16u, 1024u);
      const uint64_t bdesc0 = B_MN ? smem_desc_sw128(sbase + C::kABytes, 8192u, 1024u)
                                   : smem_desc_sw128(sbase + C::kABytes, 16u, 1024u);
      constexpr uint64_t kStageStep = C::kStageBytes >> 4;          // descriptor address units
      constexpr uint64_t kAStep = 32 >> 4;                          // one 16-wide k step
      constexpr uint64_t kBStep = B_MN ? (2048 >> 4) : (32 >> 4);
      int stage = 0;
      uint32_t phase = 0;
      bool landed = false;       // the current stage's copies are known to have landed
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
            if (!landed && !wait_phase(full_bar(stage), phase, abort_flag, p)) { ok = false; break; }
            tc_fence_after_sync();
            const int nstage = stage + 1 == STAGES ? 0 : stage + 1;
            const uint32_t nphase = stage + 1 == STAGES ? phase ^ 1u : phase;
            const uint64_t ad = adesc0 + static_cast<uint64_t>(stage) * kStageStep;
            const uint64_t bd = bdesc0 + static_cast<uint64_t>(stage) * kStageStep;
            if (kc + kBK <= kvalid && accumulate) {
              // a whole k-block after the unit's first: no per-step checks
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k) {
                if (k == kBK / 16 - 1) landed = mbar_test_wait(full_bar(nstage), nphase);
                tc_mma_bf16_pair(d_tmem, ad + k * kAStep, bd + k * kBStep, idesc, 1u);
              }
            } else {
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k) {
                if (k == kBK / 16 - 1) landed = mbar_test_wait(full_bar(nstage), nphase);
                if (kc + 16 * k < kvalid) {
                  tc_mma_bf16_pair(d_tmem, ad + k * kAStep, bd + k * kBStep, idesc, accumulate);
                  accumulate = 1;
                }
              }
            }
            tc_commit_pair_multicast(empty_bar(stage), 0x3);   // frees this stage in both CTAs
            stage = nstage;
            phase = nphase;
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
    if constexpr (STAGED) {
      staged_act_bwd<STAGES, EPIW, STAGED, ECOLS>(p, sbase + STAGES * C::kStageBytes, bar0 + 8u * (2 * STAGES + 5),
                                   tfull_bar(0), tempty_even, tmem_base, abort_flag, rank, pair, npairs, warp);
    } else {
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
      if (finish) {
        const int row = U.tm * (2 * kBM) + static_cast<int>(rank) * kBM + row_in_tile;
        if constexpr (ACTB == 1) {
          epilogue_act_bwd_rows<BN>(p, G, U, tacc, row, part, EPIW / 4);
        } else {
          epilogue_tile<BN>(p, G, U, tacc, row, part, EPIW / 4);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_even[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    }
  }

  if (*abort_flag) settle_after_abort();
  if (p.pdl_seg > 0) pdl_wait();          // complete only after the previous kernel
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
