// Persistent tcgen05 GEMM for sm_103a with the LoRA rank-r term folded in as extra
// K-segments, and the block's epilogues fused in.
//
// C[m, n] = sum over segments s, k in segment:  A_s[m, k] * B_s[n, k]
//
// A LoRA linear y = x W^T + s (x A^T) B^T ("Model Patches and Kernels", section
// "Fused LoRA operations", row opake_lora_w) becomes two segments: [x | T] against
// [W | s B] with T = x A^T computed first; the gated MLP's gate and up projections
// (row opake_lora_mlp) share one tile: the B tile's first half holds gate rows,
// the second half the matching up rows, so the activation epilogue sees both.
//
// Roles (192 threads, one CTA per SM):
//   warp 0     TMA producer (one lane): fills a STAGES-deep ring of A/B tiles.
//   warp 1     TMEM owner + MMA issuer (one lane): 128 x BN x 16 tcgen05.mma per step
//              into one of two TMEM accumulators (the epilogue drains the other).
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter, fused math, stores.
//
// Every wait is bounded in time; on expiry the CTA records a timeout in the status
// word, lets its own copies and MMAs finish (again bounded), frees TMEM and exits.
//
// Launches use programmatic dependent launch: the prologue (barriers, TMEM, descriptor
// prefetch) runs while the previous kernel drains, then griddepcontrol.wait; a launch
// marked pdl_late reads nothing the previous kernel writes and waits only before exit.
// The CTA-pair variant for the projection GEMMs is in gemm_pair.cuh.
#pragma once

#include "ptx.cuh"

namespace lgb {

constexpr int kBM = 128;       // accumulator rows = TMEM lanes
constexpr int kBK = 64;        // one 128-byte swizzle row of bf16 per k-block
constexpr int kThreads = 192;
constexpr int kMaxMaps = 12;   // TMA maps per launch (operand segments and staged epilogue)
constexpr int kMaxGroups = 4;
constexpr int kMaxSegs = 4;
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusInput = 2u;   // a device-side input out of range (a RoPE position)

enum EpiKind : int { EPI_STORE = 0, EPI_ACT_FWD = 1, EPI_ACT_BWD = 2, EPI_PARTIAL = 3, EPI_ROPE = 4 };
enum ActKind : int { ACT_SWIGLU = 0, ACT_GEGLU_TANH = 1, ACT_GEGLU_ERF = 2 };

struct SegDesc {
  int a, b0, b1;   // tensor-map indices; b1 >= 0: B tile = BN/2 rows of b0 + BN/2 rows of b1
  int kblocks;     // number of 64-wide k-blocks in this segment
  int kvalid;      // K columns that may be non-zero; MMA steps at or past it are skipped
};

struct GroupDesc {
  int M, N;                  // logical output extent
  int tiles_m, tiles_n, splits;
  int per_plane;             // 0: the splits share K out (split-K); 1: split s owns plane s of
                             // 3-D maps {x, k, plane} and runs the whole K of that plane
  int unit_begin;            // first work unit of this group
  int nseg, kb_total;
  SegDesc seg[kMaxSegs];
  int epi;
  void* out0;
  void* out1;
  void* out2;
  const void* in0;
  const void* in1;
  long long ldo, ldi;
  float* part;               // EPI_PARTIAL: [splits][tiles_m*128][tiles_n*BN] f32
  long long ldt;             // EPI_STORE with out1: out1 receives columns [0, ntc) of the
  int ntc;                   // tile transposed, [ntc x ldt]
  int emap[4];               // EPI_ACT_BWD on the staged variant: maps of g, u (in) and dg, du (out)
};

struct TcParams {
  CUtensorMap maps[kMaxMaps];
  GroupDesc grp[kMaxGroups];
  int nmaps;
  int ngroups;
  int total_units;
  int band;                  // raster: n-tiles per band, n fastest inside a band
  int act;
  unsigned int* status;
  unsigned long long timeout_ns;
  int inject_stall;          // failure-path tests only: the first stage of the first unit
                             // is never filled, so the waits on it run out
  // EPI_ROPE groups: cos/sin tables [rope_npos x rope_half] f32, token positions [M]
  const float* rope_cos;
  const float* rope_sin;
  const int* rope_pos;
  int rope_half;             // head_dim / 2: 32, 64 or 128
  int rope_npos;
  // 1: the launch reads nothing the previous kernel in the stream writes, and writes
  // nothing it reads, so it starts at once (on SMs the previous kernel has freed) and
  // waits for that kernel only before it exits, keeping the stream's completion order
  int pdl_late;
  // CTA-pair kernel, > 0: only the K-segments from this index on read what the previous
  // kernel writes (a rank-r operand), and nothing else of the launch touches its data:
  // the producers wait for it just before their first load from such a segment (and
  // only then let the next kernel launch), every thread again before it exits, so the
  // earlier segments' copies and MMAs overlap the previous kernel's tail
  int pdl_seg;
  // Split tail (CTA-pair kernel).  Units [0, sk_dp_units) are whole tiles dealt
  // round-robin to the pairs.  The sk_tail tiles after them, which would fill only part
  // of a last wave, are each cut into sk_splits equal k-ranges (of sk_kb k-blocks in
  // all), and these pieces follow, k-range major (every tail tile's first piece, then
  // every second piece, ...), so that pairs working at the same time read the same
  // k-slices of the operands.  Every piece stores its f32 partial sums in sk_part; the
  // last piece of a tile to arrive (an arrival word in sk_flags per tile, CTA and
  // epilogue warp, tagged with sk_epoch) adds the others to its accumulator in piece
  // order and runs the epilogue.  No CTA waits for another.  sk_splits == 0: every unit
  // is a whole tile.
  int sk_dp_units;
  int sk_tail;
  int sk_splits;
  int sk_kb;
  float* sk_part;                 // [sk_tail * sk_splits pieces][2 CTAs][BN/32][128 rows][32] f32
  unsigned long long* sk_flags;   // [sk_tail][2 CTAs][kSkWarps]
  unsigned long long sk_epoch;    // below 2^56
  int sk_cap_pieces;              // pieces / tail tiles the regions are sized for (host)
  int sk_cap_tiles;
};

// Arrival words per tile and CTA (one per epilogue warp, at most 8), and the most
// pieces a tail tile is cut into.
constexpr int kSkWarps = 8;
constexpr int kSkMaxSplits = 4;

template <int BN, int STAGES>
struct TcCfg {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
  static constexpr int kBarBytes = 8 * (2 * STAGES + 5) + 16;
  static constexpr int kSmemBytes = STAGES * kStageBytes + kBarBytes + 1024;
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
};

struct Unit {
  int g, tm, tn, split, kb0, kb1;
  int piece, npieces;   // split tail: piece `piece` of the `npieces` computing this tile
  int sk_tile;          // split tail: the tile's index in the tail
};

__device__ __forceinline__ Unit decode_unit(const TcParams& p, int u) {
  int g = 0;
  while (g + 1 < p.ngroups && u >= p.grp[g + 1].unit_begin) ++g;
  const GroupDesc& G = p.grp[g];
  const int local = u - G.unit_begin;
  const int tiles = G.tiles_m * G.tiles_n;
  const int split = local / tiles;
  const int t = local - split * tiles;
  const int band = p.band;
  const int b = t / (G.tiles_m * band);
  const int rem = t - b * G.tiles_m * band;
  const int nb = min(band, G.tiles_n - b * band);
  Unit U;
  U.g = g;
  U.tm = rem / nb;
  U.tn = b * band + rem % nb;
  U.split = split;
  U.piece = 0;
  U.npieces = 1;
  U.sk_tile = 0;
  if (G.per_plane) {
    U.kb0 = 0;
    U.kb1 = G.kb_total;
  } else {
    U.kb0 = static_cast<int>(static_cast<long long>(G.kb_total) * split / G.splits);
    U.kb1 = static_cast<int>(static_cast<long long>(G.kb_total) * (split + 1) / G.splits);
  }
  return U;
}

// The units of one CTA (or CTA pair) `q` of `nq`, round-robin: whole tiles, then the
// split tail's pieces.  Every role of the CTA walks the same sequence.
struct WorkIter {
  int u, nq, end;
  __device__ __forceinline__ WorkIter(const TcParams& p, int q, int nq_)
      : u(q), nq(nq_), end(p.sk_splits > 0 ? p.sk_dp_units + p.sk_tail * p.sk_splits : p.total_units) {}
  __device__ __forceinline__ bool next(const TcParams& p, Unit& U) {
    if (u >= end) return false;
    if (p.sk_splits == 0 || u < p.sk_dp_units) {
      U = decode_unit(p, u);
    } else {
      const int j = u - p.sk_dp_units;
      const int s = j / p.sk_tail, t = j - s * p.sk_tail;
      U = decode_unit(p, p.sk_dp_units + t);
      U.kb0 = static_cast<int>(static_cast<long long>(p.sk_kb) * s / p.sk_splits);
      U.kb1 = static_cast<int>(static_cast<long long>(p.sk_kb) * (s + 1) / p.sk_splits);
      U.piece = s;
      U.npieces = p.sk_splits;
      U.sk_tile = t;
    }
    u += nq;
    return true;
  }
};

// Bounded wait: true when the phase completed, false on abort (flag set by another
// role, or this wait timed out, which sets the flag and the status word).  The limit
// is wall-clock time (the global nanosecond timer, read after every failed poll from
// the first failed one on), so it holds at any SM clock; a poll sleeps at most the
// suspend-time hint, so the limit is seen at most two hints late.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           const TcParams& p) {
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

// Drain wait after an abort (this CTA's own copies or MMAs, which finish in
// microseconds): bounded by a fixed 20 ms of wall-clock time, whatever timeout_ns is.
__device__ __forceinline__ void wait_phase_drain(uint32_t bar, uint32_t parity, const TcParams& p) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 20000000ull) {
      if (p.status) atomicOr(p.status, kStatusTimeout);
      return;
    }
  }
}

// After an abort: give copies still in flight time to land before shared memory is
// released (200 us).
__device__ __forceinline__ void settle_after_abort() {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < 200000ull) {
  }
}

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kSqrt2OverPi = 0.7978845608028654f;
constexpr float kGeluC = 0.044715f;

constexpr float kSqrtHalf = 0.7071067811865476f;
constexpr float kInvSqrt2Pi = 0.3989422804014327f;

// act(g): silu, tanh-GELU or exact GELU ("Model Patches and Kernels", activation table).
// The activation is a template argument: the act epilogue picks it once per 32-column
// chunk (act_chunk below), so its unrolled per-element loop carries no branch on it.
template <int ACT>
__device__ __forceinline__ float act_fwd(float g) {
  if (ACT == ACT_SWIGLU) return __fdividef(g, 1.0f + __expf(-g));
  if (ACT == ACT_GEGLU_ERF) return 0.5f * g * (1.0f + erff(g * kSqrtHalf));
  const float t = tanh_approx(kSqrt2OverPi * (g + kGeluC * g * g * g));
  return 0.5f * g * (1.0f + t);
}

// act(g) and act'(g) together.
template <int ACT>
__device__ __forceinline__ void act_fwd_bwd(float g, float& a, float& ap) {
  if (ACT == ACT_SWIGLU) {
    const float sg = __fdividef(1.0f, 1.0f + __expf(-g));
    a = g * sg;
    ap = sg * (1.0f + g * (1.0f - sg));
  } else if (ACT == ACT_GEGLU_ERF) {
    const float cdf = 0.5f * (1.0f + erff(g * kSqrtHalf));
    a = g * cdf;
    ap = cdf + g * kInvSqrt2Pi * __expf(-0.5f * g * g);
  } else {
    const float t = tanh_approx(kSqrt2OverPi * (g + kGeluC * g * g * g));
    a = 0.5f * g * (1.0f + t);
    ap = 0.5f * (1.0f + t) + 0.5f * g * (1.0f - t * t) * kSqrt2OverPi * (1.0f + 3.0f * kGeluC * g * g);
  }
}

// The same with the activation chosen at run time, per element.  The act' epilogue
// uses this form: with one compiled copy per activation its 8-warp kernels (at most 168
// registers a thread) spill, and that costs more than the per-element branch.
__device__ __forceinline__ void act_fwd_bwd_rt(float g, int act, float& a, float& ap) {
  if (act == ACT_SWIGLU) {
    act_fwd_bwd<ACT_SWIGLU>(g, a, ap);
  } else if (act == ACT_GEGLU_ERF) {
    act_fwd_bwd<ACT_GEGLU_ERF>(g, a, ap);
  } else {
    act_fwd_bwd<ACT_GEGLU_TANH>(g, a, ap);
  }
}

// Calls f(tag) with tag's `value` the activation, so f is compiled once per activation
// and the branch is taken once per call instead of once per element.
template <int ACT>
struct ActTag {
  static constexpr int value = ACT;
};
template <typename F>
__device__ __forceinline__ void act_chunk(int act, F&& f) {
  if (act == ACT_SWIGLU) {
    f(ActTag<ACT_SWIGLU>{});
  } else if (act == ACT_GEGLU_ERF) {
    f(ActTag<ACT_GEGLU_ERF>{});
  } else {
    f(ActTag<ACT_GEGLU_TANH>{});
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Writes 32 bf16 values (w: 16 packed pairs) of one row at dst, columns col0 ..
// col0+31, keeping the columns below N.  v8 (row start and stride 32-byte aligned):
// two whole-sector stores; otherwise 16-byte pieces.
__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16* dst, const uint32_t (&w)[16], int col0, int N,
                                                 bool v8) {
  if (v8 && col0 + 32 <= N) {
    st_global_v8(dst, w);
    st_global_v8(dst + 16, w + 8);
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (col0 + 8 * j + 8 <= N)
      *reinterpret_cast<uint4*>(dst + 8 * j) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

// store_row32_bf16 with the whole-sector stores under an L2 cache policy.
__device__ __forceinline__ void store_row32_bf16_hint(__nv_bfloat16* dst, const uint32_t (&w)[16], int col0, int N,
                                                      bool v8, uint64_t pol) {
  if (v8 && col0 + 32 <= N) {
    st_global_v8_hint(dst, w, pol);
    st_global_v8_hint(dst + 16, w + 8, pol);
    return;
  }
  store_row32_bf16(dst, w, col0, N, false);
}

__device__ __forceinline__ bool rows_v8_aligned(const void* base, long long ld) {
  return (ld % 16) == 0 && (reinterpret_cast<uintptr_t>(base) & 31) == 0;
}

// Epilogue of one accumulator tile, columns split into `nparts` equal parts of which
// this warp takes part `part`.  The calling thread owns output row `row` and reads its
// TMEM lane at `tacc`.  Warp-collective: every lane of the warp calls it (tcgen05.ld);
// rows past M are computed and dropped.
template <int BN>
__device__ __forceinline__ void epilogue_tile(const TcParams& p, const GroupDesc& G, const Unit& U,
                                              uint32_t tacc, int row, int part, int nparts) {
  const bool row_ok = row < G.M;
  if (G.epi == EPI_STORE) {
    // optional frozen per-column bias (in0, bf16 [N]) added before rounding
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(G.out0);
    const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(G.in0);
    const bool v8 = rows_v8_aligned(out, G.ldo);
    const int span = BN / nparts, c_lo = part * span;
#pragma unroll 1
    for (int c = c_lo; c < c_lo + span; c += 32) {
      uint32_t v[32];
      __syncwarp();
      tmem_ld32(tacc + c, v);
      tmem_ld_wait();
      const int col0 = U.tn * BN + c;
      if (row_ok) {
        uint32_t w[16];
        if (bias != nullptr) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 b = (col0 + 8 * j + 8 <= G.N) ? __ldg(reinterpret_cast<const uint4*>(bias + col0 + 8 * j))
                                                      : make_uint4(0, 0, 0, 0);
            const uint32_t bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[4 * j + e] = pack_bf16x2(__uint_as_float(v[8 * j + 2 * e]) + bf16_lo(bb[e]),
                                         __uint_as_float(v[8 * j + 2 * e + 1]) + bf16_hi(bb[e]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
        }
        store_row32_bf16(out + static_cast<long long>(row) * G.ldo + col0, w, col0, G.N, v8);
        if (G.out1 != nullptr) {
          // the same values, transposed (a warp's 32 rows are consecutive there)
          __nv_bfloat16* ot = static_cast<__nv_bfloat16*>(G.out1) + row;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = col0 + 2 * e;
            if (c < G.ntc) ot[static_cast<long long>(c) * G.ldt] = __ushort_as_bfloat16(static_cast<unsigned short>(w[e]));
            if (c + 1 < G.ntc)
              ot[static_cast<long long>(c + 1) * G.ldt] = __ushort_as_bfloat16(static_cast<unsigned short>(w[e] >> 16));
          }
        }
      }
    }
  } else if (G.epi == EPI_ACT_FWD) {
    // gate in accumulator columns [0, BN/2), up in [BN/2, BN)
    __nv_bfloat16* hout = static_cast<__nv_bfloat16*>(G.out0);
    __nv_bfloat16* gout = static_cast<__nv_bfloat16*>(G.out1);
    __nv_bfloat16* uout = static_cast<__nv_bfloat16*>(G.out2);
    const bool v8 = rows_v8_aligned(hout, G.ldo) && (gout == nullptr || (rows_v8_aligned(gout, G.ldo) &&
                                                                         rows_v8_aligned(uout, G.ldo)));
    const int span = (BN / 2) / nparts, c_lo = part * span;
#pragma unroll 1
    for (int c = c_lo; c < c_lo + span; c += 32) {
      uint32_t vg[32], vu[32];
      __syncwarp();
      tmem_ld32(tacc + c, vg);
      tmem_ld32(tacc + BN / 2 + c, vu);
      tmem_ld_wait();
      const int col0 = U.tn * (BN / 2) + c;
      if (row_ok) {
        const long long off = static_cast<long long>(row) * G.ldo + col0;
        uint32_t w[16];
        act_chunk(p.act, [&](auto tag) {
          constexpr int ACT = decltype(tag)::value;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float h0 = act_fwd<ACT>(__uint_as_float(vg[2 * e])) * __uint_as_float(vu[2 * e]);
            const float h1 = act_fwd<ACT>(__uint_as_float(vg[2 * e + 1])) * __uint_as_float(vu[2 * e + 1]);
            w[e] = pack_bf16x2(h0, h1);
          }
        });
        store_row32_bf16(hout + off, w, col0, G.N, v8);
        if (gout != nullptr) {
          // g, u are saved for the backward: evict-first keeps the weight tiles in L2
          const uint64_t pol = l2_evict_first_policy();
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(__uint_as_float(vg[2 * e]), __uint_as_float(vg[2 * e + 1]));
          store_row32_bf16_hint(gout + off, w, col0, G.N, v8, pol);
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(__uint_as_float(vu[2 * e]), __uint_as_float(vu[2 * e + 1]));
          store_row32_bf16_hint(uout + off, w, col0, G.N, v8, pol);
        }
      }
    }
  } else if (G.epi == EPI_ROPE) {
    // EPI_STORE (bias included) followed by the rotary embedding of every head in the
    // tile ("Model Patches and Kernels", RoPE): the pair (c, c + half) of a head turns
    // by the angle of this token's position.  Heads never straddle a 256-column tile
    // (head_dim divides 256).  The tile row's BN/64 (head, 32-column) chunk pairs are
    // shared out among the `nparts` warps that own this row.
    if constexpr (BN == 256) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(G.out0);
      const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(G.in0);
      const bool v8 = rows_v8_aligned(out, G.ldo);
      const int half = p.rope_half;
      int pos = 0;
      if (row_ok) {
        pos = __ldg(p.rope_pos + row);
        if (pos < 0 || pos >= p.rope_npos) {
          if (p.status) atomicOr(p.status, kStatusInput);
          pos = 0;
        }
      }
      const float* crow = p.rope_cos + static_cast<long long>(pos) * half;
      const float* srow = p.rope_sin + static_cast<long long>(pos) * half;
      const int cph = half / 32;                       // chunk pairs per head
#pragma unroll 1
      for (int t = part; t < BN / 64; t += nparts) {
        const int hb = (t / cph) * 2 * half, c = (t % cph) * 32;
        {
          uint32_t va[32], vb[32];
          __syncwarp();
          tmem_ld32(tacc + hb + c, va);
          tmem_ld32(tacc + hb + half + c, vb);
          tmem_ld_wait();
          const int cola = U.tn * BN + hb + c, colb = cola + half;
          if (row_ok && cola < G.N) {     // N is a multiple of head_dim: colb < N too
            float a[32], b[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              a[e] = __uint_as_float(va[e]);
              b[e] = __uint_as_float(vb[e]);
            }
            if (bias != nullptr) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint4 ba = __ldg(reinterpret_cast<const uint4*>(bias + cola + 8 * j));
                const uint4 bb = __ldg(reinterpret_cast<const uint4*>(bias + colb + 8 * j));
                const uint32_t xa[4] = {ba.x, ba.y, ba.z, ba.w}, xb[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  a[8 * j + 2 * e] += bf16_lo(xa[e]);
                  a[8 * j + 2 * e + 1] += bf16_hi(xa[e]);
                  b[8 * j + 2 * e] += bf16_lo(xb[e]);
                  b[8 * j + 2 * e + 1] += bf16_hi(xb[e]);
                }
              }
            }
            uint32_t wa[16], wb[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 cs = __ldg(reinterpret_cast<const float4*>(crow + c) + j);
              const float4 sn = __ldg(reinterpret_cast<const float4*>(srow + c) + j);
              const float cc[4] = {cs.x, cs.y, cs.z, cs.w}, ss[4] = {sn.x, sn.y, sn.z, sn.w};
              float ra[4], rb[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float x0 = a[4 * j + e], x1 = b[4 * j + e];
                ra[e] = x0 * cc[e] - x1 * ss[e];
                rb[e] = x1 * cc[e] + x0 * ss[e];
              }
              wa[2 * j] = pack_bf16x2(ra[0], ra[1]);
              wa[2 * j + 1] = pack_bf16x2(ra[2], ra[3]);
              wb[2 * j] = pack_bf16x2(rb[0], rb[1]);
              wb[2 * j + 1] = pack_bf16x2(rb[2], rb[3]);
            }
            __nv_bfloat16* orow = out + static_cast<long long>(row) * G.ldo;
            store_row32_bf16(orow + cola, wa, cola, G.N, v8);
            store_row32_bf16(orow + colb, wb, colb, G.N, v8);
          }
        }
      }
    }
  } else {
    // EPI_PARTIAL: f32 tile into the split's slab (rows and columns padded, 32-byte
    // aligned: the slab starts 256-byte aligned and its width is a multiple of 64)
    const long long width = static_cast<long long>(G.tiles_n) * BN;
    float* dst = G.part + (static_cast<long long>(U.split) * G.tiles_m * kBM + row) * width + U.tn * BN;
    const int span = BN / nparts, c_lo = part * span;
#pragma unroll 1
    for (int c = c_lo; c < c_lo + span; c += 32) {
      uint32_t v[32];
      __syncwarp();
      tmem_ld32(tacc + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; j += 8) st_global_v8(dst + c + j, v + j);
    }
  }
}

// The activation-derivative epilogue with one row per thread (the CTA-pair kernel's
// variant for long K, where each tile's MMAs hide it): the accumulator is dh; the saved
// g, u of the row give dg = dh u act'(g), du = dh act(g).  The thread loads the g, u of
// the next 32-column chunk while this one is computed.  Warp-collective like
// epilogue_tile; rows past M are computed and dropped.
template <int BN>
__device__ __forceinline__ void epilogue_act_bwd_rows(const TcParams& p, const GroupDesc& G, const Unit& U,
                                                      uint32_t tacc, int row, int part, int nparts) {
  const bool row_ok = row < G.M;
  const __nv_bfloat16* gin = static_cast<const __nv_bfloat16*>(G.in0);
  const __nv_bfloat16* uin = static_cast<const __nv_bfloat16*>(G.in1);
  __nv_bfloat16* dgo = static_cast<__nv_bfloat16*>(G.out0);
  __nv_bfloat16* duo = static_cast<__nv_bfloat16*>(G.out1);
  const bool v8 = rows_v8_aligned(dgo, G.ldo) && rows_v8_aligned(duo, G.ldo);
  const int span = BN / nparts, c_lo = part * span, c_hi = c_lo + span;
  const long long rbase = static_cast<long long>(row) * G.ldi + U.tn * BN;
  const uint64_t pol = l2_evict_first_policy();   // the saved g, u are read for the last time
  auto load_chunk = [&](int c, uint4 (&gw)[4], uint4 (&uw)[4]) {
    const int col0 = U.tn * BN + c;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (row_ok && col0 + 8 * j + 8 <= G.N) {
        gw[j] = ld_global_nc_v4_hint(gin + rbase + c + 8 * j, pol);
        uw[j] = ld_global_nc_v4_hint(uin + rbase + c + 8 * j, pol);
      } else {
        gw[j] = make_uint4(0, 0, 0, 0);
        uw[j] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  uint4 gw[4], uw[4];
  load_chunk(c_lo, gw, uw);
#pragma unroll 1
  for (int c = c_lo; c < c_hi; c += 32) {
    uint4 gn[4], un[4];
    if (c + 32 < c_hi) load_chunk(c + 32, gn, un);
    const int col0 = U.tn * BN + c;
    uint32_t v[32];
    __syncwarp();
    tmem_ld32(tacc + c, v);
    tmem_ld_wait();
    if (row_ok) {
      const long long ooff = static_cast<long long>(row) * G.ldo + col0;
      uint32_t og[16], ou[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t gg[4] = {gw[j].x, gw[j].y, gw[j].z, gw[j].w};
        const uint32_t uu[4] = {uw[j].x, uw[j].y, uw[j].z, uw[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a0, ap0, a1, ap1;
          const float g0 = bf16_lo(gg[e]), g1 = bf16_hi(gg[e]);
          const float u0 = bf16_lo(uu[e]), u1 = bf16_hi(uu[e]);
          act_fwd_bwd_rt(g0, p.act, a0, ap0);
          act_fwd_bwd_rt(g1, p.act, a1, ap1);
          const float d0 = __uint_as_float(v[8 * j + 2 * e]);
          const float d1 = __uint_as_float(v[8 * j + 2 * e + 1]);
          og[4 * j + e] = pack_bf16x2(d0 * u0 * ap0, d1 * u1 * ap1);
          ou[4 * j + e] = pack_bf16x2(d0 * a0, d1 * a1);
        }
      }
      store_row32_bf16(dgo + ooff, og, col0, G.N, v8);
      store_row32_bf16(duo + ooff, ou, col0, G.N, v8);
    }
    if (c + 32 < c_hi) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        gw[j] = gn[j];
        uw[j] = un[j];
      }
    }
  }
}

template <int BN, int STAGES, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
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
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < p.nmaps) tma_prefetch_map(&p.maps[lane]);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  if (!p.pdl_late) pdl_wait();            // the previous kernel's writes are visible from here
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[STAGES];
      for (int s = 0; s < STAGES; ++s) armed[s] = -1;
      bool ok = true;
      bool first_stage = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
        const Unit U = decode_unit(p, u);
        const GroupDesc& G = p.grp[U.g];
        // walk the unit's k-range segment by segment; a segment's fields live in registers
        const int nseg = G.nseg;
        int seg_base = 0;
        for (int sg = 0; sg < nseg && ok; ++sg) {
          const int nkb = G.seg[sg].kblocks;
          const int j0 = max(U.kb0 - seg_base, 0), j1 = min(U.kb1 - seg_base, nkb);
          const CUtensorMap* ma = &p.maps[G.seg[sg].a];
          const CUtensorMap* mb0 = &p.maps[G.seg[sg].b0];
          const int b1 = G.seg[sg].b1;
          const CUtensorMap* mb1 = &p.maps[b1 >= 0 ? b1 : G.seg[sg].b0];
          seg_base += nkb;
          for (int j = j0; j < j1; ++j) {
            const int kc = j * kBK;
            if (!wait_phase(empty_bar(stage), phase ^ 1u, abort_flag, p)) { ok = false; break; }
            const uint32_t fb = full_bar(stage);
            if (p.inject_stall && first_stage) {   // failure-path tests: leave this stage empty
              first_stage = false;
              if (++stage == STAGES) { stage = 0; phase ^= 1u; }
              continue;
            }
            first_stage = false;
            mbar_arrive_expect_tx(fb, C::kStageBytes);
            armed[stage] = static_cast<int>(phase);
            const uint32_t sa = sbase + stage * C::kStageBytes;
            const uint32_t sb = sa + C::kABytes;
            if (A_MN && B_MN && G.per_plane) {
              // reductions over one plane (one example's tokens) of 3-D maps
              tma_load_3d(sa, ma, fb, U.tm * kBM, kc, U.split);
              tma_load_3d(sa + 8192u, ma, fb, U.tm * kBM + 64, kc, U.split);
#pragma unroll
              for (int c = 0; c < BN / 64; ++c)
                tma_load_3d(sb + c * 8192u, mb0, fb, U.tn * BN + c * 64, kc, U.split);
            } else {
              if (!A_MN) {
                tma_load_2d(sa, ma, fb, kc, U.tm * kBM);
              } else {
                tma_load_2d(sa, ma, fb, U.tm * kBM, kc);
                tma_load_2d(sa + 8192u, ma, fb, U.tm * kBM + 64, kc);
              }
              if (!B_MN) {
                if (b1 >= 0) {
                  tma_load_2d(sb, mb0, fb, kc, U.tn * (BN / 2));
                  tma_load_2d(sb + (BN / 2) * 128u, mb1, fb, kc, U.tn * (BN / 2));
                } else {
                  tma_load_2d(sb, mb0, fb, kc, U.tn * BN);
                }
              } else {
#pragma unroll
                for (int c = 0; c < BN / 64; ++c) tma_load_2d(sb + c * 8192u, mb0, fb, U.tn * BN + c * 64, kc);
              }
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
      if (!ok) {
        // let this CTA's copies land before its shared memory is released
        for (int s = 0; s < STAGES; ++s)
          if (armed[s] >= 0) wait_phase_drain(full_bar(s), static_cast<uint32_t>(armed[s]), p);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // lean MMA loop: see the CTA-pair kernel (descriptors from stage 0 plus offsets;
      // the next stage tested before this stage's last MMA)
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, A_MN ? 1 : 0, B_MN ? 1 : 0);
      const uint64_t adesc0 = A_MN ? smem_desc_sw128(sbase, 8192u, 1024u) : smem_desc_sw128(sbase, 16u, 1024u);
      const uint64_t bdesc0 = B_MN ? smem_desc_sw128(sbase + C::kABytes, 8192u, 1024u)
                                   : smem_desc_sw128(sbase + C::kABytes, 16u, 1024u);
      constexpr uint64_t kStageStep = C::kStageBytes >> 4;
      constexpr uint64_t kAStep = A_MN ? (2048 >> 4) : (32 >> 4);
      constexpr uint64_t kBStep = B_MN ? (2048 >> 4) : (32 >> 4);
      int stage = 0;
      uint32_t phase = 0;
      bool landed = false;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
        const Unit U = decode_unit(p, u);
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
                tc_mma_bf16(d_tmem, ad + k * kAStep, bd + k * kBStep, idesc, 1u);
              }
            } else {
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k) {
                if (k == kBK / 16 - 1) landed = mbar_test_wait(full_bar(nstage), nphase);
                if (kc + 16 * k < kvalid) {
                  tc_mma_bf16(d_tmem, ad + k * kAStep, bd + k * kBStep, idesc, accumulate);
                  accumulate = 1;
                }
              }
            }
            tc_commit(empty_bar(stage));     // frees this smem stage once its MMAs are done
            stage = nstage;
            phase = nphase;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));         // accumulator ready for the epilogue
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        tc_commit(drain_bar);
        wait_phase_drain(drain_bar, 0, p);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
      const Unit U = decode_unit(p, u);
      const GroupDesc& G = p.grp[U.g];
      // tcgen05.ld is warp-collective: the whole warp proceeds or the whole warp stops
      const bool ready = wait_phase(tfull_bar(acc), acc_phase, abort_flag, p);
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after_sync();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      epilogue_tile<BN>(p, G, U, tacc, U.tm * kBM + row_in_tile, 0, 1);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  if (*abort_flag) settle_after_abort();
  if (p.pdl_late) pdl_wait();             // complete only after the previous kernel
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace lgb
