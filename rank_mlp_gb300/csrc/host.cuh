// Host-side plumbing shared by the entry points: tensor-map encoding, the GEMM plan
// builder, workspace carving, launch wrappers (with the launch counter and the
// optional event trace).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "lora_gb300.h"
#include "aux_kernels.cuh"
#include "gemm_tc.cuh"
#include "rank_dual.cuh"

namespace lgb {

// Kernel variants (tile width BN, operand majors) compiled into the library.
enum Variant : int {
  VP_KK = 0,       // projections on a CTA pair, 256 x 256 tiles, K-major B (forward)
  VP_KMN = 1,      // projections on a CTA pair, MN-major B (backward: W read untransposed)
  V64_KK = 2,      // token-major rank-r projections, padded rank <= 64
  V64_MNMN = 3,    // reductions over tokens (dA, dB), padded rank <= 64
  V128_KK = 4,
  V128_MNMN = 5,
  VP_KK8 = 6,      // VP_KK with 8 epilogue warps: short-K launches, where 4 warps' epilogue
                   // outlasts a tile's MMAs
  VP_KMN_ACT = 7,   // VP_KMN for the activation-derivative GEMM: saved g, u in and dg, du out
                    // one row per thread (6 stages)
  VP_KMN_ACT16 = 8, // the same for short K: g, u and dg, du through shared memory by TMA
                    // (kActStaged* below)
  kNumVariants = 9
};

// An activation-derivative launch whose K is at most this many k-blocks runs
// VP_KMN_ACT16: its tiles' MMAs are too short to hide the epilogue's traffic, and the
// staged epilogue keeps more of it in flight.  Longer K needs the sixth stage to keep
// the MMAs fed (measured: the staged variant at 5 stages, or at 6 stages with 8-column
// chunks or with 2-slot rings, was 3-15% slower there than one row per thread).
constexpr int kActShortKBlocks = 32;

// VP_KMN_ACT16's shape: mainloop stages, epilogue warps, ring slots per epilogue warp
// and columns per chunk (a chunk is one warp's 32 rows; 32 columns make 64-byte rows, so
// that each TMA copy moves twice the bytes of a 16-column chunk).  Measured on the
// 0.5B-shaped act' GEMM (15 k-blocks a tile): 5 stages with two 32-column slots 59.3 us
// against 61.6 us for four 16-column slots; 4 or 3 stages with 3 or 4 such slots were no
// faster than the 16-column ring, so the mainloop's fifth stage matters more than depth.
constexpr int kActStagedStages = 5;
constexpr int kActStagedWarps = 8;
constexpr int kActStagedSlots = 2;
constexpr int kActStagedCols = 32;

// A forward pair launch whose longest K is at most this many 64-wide k-blocks runs
// VP_KK8: a tile's MMAs (~0.28 us per k-block) then no longer cover the 4-warp
// epilogue of the previous tile (~8 us for gate/up with SwiGLU).
constexpr int kShortKBlocks = 32;

// Largest token count or feature size: the kernels index rows, columns and tiles with
// 32-bit integers and TMA coordinates are 32-bit.
constexpr int64_t kMaxExtent = 0x7fffffff;

constexpr bool variant_pair(int v) {
  return v == VP_KK || v == VP_KMN || v == VP_KK8 || v == VP_KMN_ACT || v == VP_KMN_ACT16;
}
constexpr int variant_bn(int v) { return variant_pair(v) ? 256 : (v <= V64_MNMN ? 64 : 128); }
constexpr bool variant_a_mn(int v) { return v == V64_MNMN || v == V128_MNMN; }
constexpr bool variant_b_mn(int v) {
  return v == VP_KMN || v == VP_KMN_ACT || v == VP_KMN_ACT16 || v == V64_MNMN || v == V128_MNMN;
}

// The big projection GEMMs run on CTA pairs (256 x 256 tiles).
constexpr int kBigKK = VP_KK;
constexpr int kBigKMN = VP_KMN;

// Programmatic dependent launch for every kernel of the library (on unless the
// environment sets LORA_PDL=0): a kernel may be scheduled while the previous kernel
// in the stream drains, runs its prologue (barriers, tensor memory, descriptor
// prefetch) and then waits in griddepcontrol.wait for that kernel's completion.
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("LORA_PDL");
    return !(e != nullptr && e[0] == '0');
  }();
  return on;
}

// Raster of the GEMM tiles: bands of this many n-tiles, the n-tile fastest inside a band
// (environment LORA_RASTER_BAND overrides the default of 16, for measurements).
inline int raster_band() {
  static const int band = [] {
    const char* e = std::getenv("LORA_RASTER_BAND");
    const int v = e != nullptr ? std::atoi(e) : 0;
    return v >= 1 && v <= 4096 ? v : 16;
  }();
  return band;
}

template <typename Kernel, typename Arg>
inline cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const Arg& arg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

// Raises a kernel's dynamic shared-memory limit to `smem` bytes on the current device,
// once per device (the attribute belongs to the device's context; bit d of `done`
// marks device d).
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel kernel, int smem, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Defined in gemm_big.cu / gemm_skinny.cu.
cudaError_t launch_tc_big(int variant, const TcParams& p, int grid, cudaStream_t st);
cudaError_t launch_tc_skinny(int variant, const TcParams& p, int grid, cudaStream_t st);
int tc_smem_bytes(int variant);

// Defined in lora_api.cu.
int num_sms();
bool encode_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                uint32_t box_inner, uint32_t box_outer, int swizzle_bytes = 128);
bool encode_map_planes(CUtensorMap* m, const void* base, uint64_t inner, uint64_t d1, uint64_t d2, uint64_t ld,
                       uint32_t box_inner, uint32_t box_d1);
lora_status_t launch_gemm(int variant, const TcParams& p, int kind, cudaStream_t st);
lora_status_t launch_norms(const NormParams& p, int examples, cudaStream_t st);
lora_status_t launch_pack(const PackParams& p, cudaStream_t st);
lora_status_t launch_reduce(const RedParams& p, cudaStream_t st);

constexpr int kMaxSplits = 16;        // split-K factors of the rank-r products
constexpr unsigned long long kTimeoutNs = 2000000000ull;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t imax(int64_t a, int64_t b) { return a > b ? a : b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Padded width of the rank-r operands of `nslots` adapters sharing one input.
inline int fold_width(int nslots, int r) { return static_cast<int>(round_up(static_cast<int64_t>(nslots) * r, 64)); }
inline int skinny_bn(int kf) { return kf <= 64 ? 64 : 128; }
inline int skinny_kk(int kf) { return kf <= 64 ? V64_KK : V128_KK; }
inline int skinny_mnmn(int kf) { return kf <= 64 ? V64_MNMN : V128_MNMN; }

// Largest split-K factor for a K of kb_total k-blocks (at least 4 k-blocks per split);
// workspaces are sized for it, so they do not depend on the device.
inline int max_splits(int64_t kb_total) {
  int64_t s = kb_total / 4;
  s = s < 1 ? 1 : (s > kMaxSplits ? kMaxSplits : s);
  return static_cast<int>(s);
}

// Split factor (over tokens) of a reduction over tokens: `tiles` 128-row output tiles
// of kb_total k-blocks each on `sms` SMs.  Minimises the slowest SM's k-blocks,
// ceil(tiles * s / sms) / s * kb_total, plus kSlabKBlocks per split for reading its f32
// partial tile back in the final sums (a 32 KB slab tile against 24 KB a k-block
// streams); ties go to fewer splits.
constexpr int kSlabKBlocks = 2;
inline int choose_splits(int64_t tiles, int64_t kb_total, int sms) {
  if (tiles <= 0 || kb_total <= 0 || sms <= 0) return 1;
  const int smax = max_splits(kb_total);
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= smax; ++s) {
    const double cost = static_cast<double>(ceil_div(tiles * s, sms)) / s * kb_total + kSlabKBlocks * s;
    if (cost < best_cost * (1.0 - 1e-9)) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// Split-K factor of a rank-r projection (`tiles` 128-row tiles of kb_total k-blocks
// each): like choose_splits, but a split pays for the launch that sums its partials,
// worth about kReduceKBlocks k-blocks of one tile (a tile streams 24 KB per k-block:
// ~0.25 us at one SM's share of the bandwidth; the reduce launch ~3 us).  Small
// problems (the Qwen-shaped x A^T: 32 tiles of 14 k-blocks) then run unsplit.
constexpr int kReduceKBlocks = 12;
inline int choose_proj_splits(int64_t tiles, int64_t kb_total, int sms) {
  if (tiles <= 0 || kb_total <= 0 || sms <= 0) return 1;
  const int smax = max_splits(kb_total);
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= smax; ++s) {
    const double cost = static_cast<double>(ceil_div(tiles * s, sms)) / s * kb_total + (s > 1 ? kReduceKBlocks : 0);
    if (cost < best_cost * (1.0 - 1e-9)) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// Bump allocator over a caller-provided buffer (256-byte aligned regions).  Used
// both to size (base == nullptr) and to carve.
struct Carve {
  uint8_t* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off), 256));
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
  template <class T>
  T* take_n(int64_t n) { return static_cast<T*>(take(static_cast<size_t>(n) * sizeof(T))); }
  // Offset (from the base) of a region of `bytes`, carved like take().
  size_t offset_of(size_t bytes) {
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off), 256));
    const size_t at = off;
    off += bytes;
    return at;
  }
};

constexpr size_t kWsHeader = 256;

// Split tail of the pair GEMMs (see TcParams): the partial-sum and arrival-word
// regions are carved from the caller's workspace, sized for the call's largest pair
// GEMM and at most kSkMaxPieces pieces (256 KB of partial sums each), whatever the
// device.  A tail of fewer than 128 tiles is cut into 2 to kSkMaxSplits k-ranges when
// the model in plan_pairs (lora_api.cu) expects the launch to gain at least
// kSkMinGain, and a tile has at least kSkMinKb k-blocks.
constexpr int kSkMaxPieces = 256;
constexpr int kSkMaxTail = 128;
constexpr int kSkMinKb = 8;
constexpr double kSkMinGain = 0.02;

// Tiles of a pair-kernel output [M x N]: 256 x 256, or 256 x (128 + 128) for the
// gate/up interleave (N = i, split_n).
inline int64_t pair_tiles(int64_t M, int64_t N, bool split_n = false) {
  return ceil_div(M, 2 * kBM) * ceil_div(N, split_n ? 128 : 256);
}

// The split-tail regions of one call: partial slots [pieces][2][8][128][32] f32 and
// arrival words [tail tiles][2][kSkWarps].
struct SkRegion {
  float* part = nullptr;
  unsigned long long* flags = nullptr;
  int pieces = 0, tiles = 0;
};
inline SkRegion carve_sk(Carve& c, int64_t max_tiles) {
  SkRegion r;
  r.tiles = static_cast<int>(max_tiles < kSkMaxTail ? max_tiles : kSkMaxTail);
  r.pieces = static_cast<int>(kSkMaxSplits * r.tiles < kSkMaxPieces ? kSkMaxSplits * r.tiles : kSkMaxPieces);
  r.part = c.take_n<float>(static_cast<int64_t>(r.pieces) * 2 * 8 * kBM * 32);
  r.flags = c.take_n<unsigned long long>(static_cast<int64_t>(r.tiles) * 2 * kSkWarps);
  return r;
}

// Builds the TcParams of one GEMM launch.
struct GemmPlan {
  TcParams p;
  int variant;
  int bn;
  bool pair;
  bool ok = true;

  explicit GemmPlan(int v) : variant(v), bn(variant_bn(v)), pair(variant_pair(v)) {
    std::memset(static_cast<void*>(&p), 0, sizeof(p));
    p.band = 8;
    p.timeout_ns = kTimeoutNs;
  }
  // Lets the launch split its tail (pair kernels) with this call's regions.
  void split_tail(const SkRegion& r) {
    p.sk_part = r.part;
    p.sk_flags = r.flags;
    p.sk_cap_pieces = r.pieces;
    p.sk_cap_tiles = r.tiles;
  }

  int add_map(const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t bi, uint32_t bo,
              int swizzle_bytes = 128) {
    if (!ok || p.nmaps >= kMaxMaps) { ok = false; return -1; }
    if (!encode_map(&p.maps[p.nmaps], base, inner, outer, ld, bi, bo, swizzle_bytes)) { ok = false; return -1; }
    return p.nmaps++;
  }
  // An epilogue operand or output [rows x cols] (row stride ld) moved by TMA in boxes of
  // 32 rows x kActStagedCols columns (one warp's rows), in the swizzle of that row width.
  int epi_map(const void* base, int64_t rows, int64_t cols, int64_t ld) {
    return add_map(base, cols, rows, ld, kActStagedCols, 32, 2 * kActStagedCols);
  }
  // A operand, K-major: activation [rows x K] with row stride ld.
  int a_kmajor(const void* base, int64_t rows, int64_t K, int64_t ld) {
    return add_map(base, K, rows, ld, 64, kBM);
  }
  // A operand, MN-major: source [K x rows] (K = tokens, rows = features contiguous).
  int a_mnmajor(const void* base, int64_t rows, int64_t K, int64_t ld) {
    return add_map(base, rows, K, ld, 64, 64);
  }
  // Rows of a whole (not split) K-major B tile held by one CTA.
  int b_rows_full() const { return pair ? bn / 2 : bn; }
  // B operand, K-major: [N x K]; box_rows = b_rows_full(), or BN/2 for a split (gate/up) tile.
  int b_kmajor(const void* base, int64_t N, int64_t K, int64_t ld, int box_rows) {
    return add_map(base, K, N, ld, 64, box_rows);
  }
  // B operand, MN-major: source [K x N] (N contiguous).
  int b_mnmajor(const void* base, int64_t N, int64_t K, int64_t ld) {
    return add_map(base, N, K, ld, 64, 64);
  }
  // MN-major operands read as planes: source [planes * K x rows], plane p = rows
  // [p K, (p+1) K); 3-D view {rows, K, planes} (per-example token reductions).
  int add_map_planes(const void* base, int64_t rows, int64_t K, int64_t planes, int64_t ld) {
    if (!ok || p.nmaps >= kMaxMaps) { ok = false; return -1; }
    if (!encode_map_planes(&p.maps[p.nmaps], base, rows, K, planes, ld, 64, 64)) { ok = false; return -1; }
    return p.nmaps++;
  }
  int a_mnmajor_planes(const void* base, int64_t rows, int64_t K, int64_t planes, int64_t ld) {
    return add_map_planes(base, rows, K, planes, ld);
  }
  int b_mnmajor_planes(const void* base, int64_t N, int64_t K, int64_t planes, int64_t ld) {
    return add_map_planes(base, N, K, planes, ld);
  }

  GroupDesc& group(int M, int N, int epi, bool split_n_tile) {
    GroupDesc& G = p.grp[p.ngroups++];
    G.M = M;
    G.N = N;
    G.epi = epi;
    G.tiles_m = static_cast<int>(ceil_div(M, pair ? 2 * kBM : kBM));
    G.tiles_n = static_cast<int>(ceil_div(N, split_n_tile ? bn / 2 : bn));
    G.splits = 1;
    return G;
  }
  static void seg(GroupDesc& G, int a, int b0, int b1, int64_t K, int64_t kvalid) {
    SegDesc& S = G.seg[G.nseg++];
    S.a = a;
    S.b0 = b0;
    S.b1 = b1;
    // k-blocks wholly past kvalid hold only zero padding: they are not walked, so every
    // k-block of a segment issues at least one MMA
    S.kblocks = static_cast<int>(ceil_div(kvalid < K ? kvalid : K, kBK));
    S.kvalid = static_cast<int>(kvalid);
    G.kb_total += S.kblocks;
  }
  // Total work units; call after every group and segment is in place.
  void finish() {
    int u = 0;
    for (int g = 0; g < p.ngroups; ++g) {
      p.grp[g].unit_begin = u;
      u += p.grp[g].tiles_m * p.grp[g].tiles_n * p.grp[g].splits;
    }
    p.total_units = u;
    p.sk_dp_units = u;
    p.sk_splits = 0;
    int maxtn = 1;
    for (int g = 0; g < p.ngroups; ++g) maxtn = p.grp[g].tiles_n > maxtn ? p.grp[g].tiles_n : maxtn;
    const int band = raster_band();
    p.band = maxtn < band ? maxtn : band;
  }
};

// f32 partial slab size of a split-K group: [splits][tiles_m*128][tiles_n*BN].
inline int64_t partial_elems(int64_t rows, int64_t kf, int bn, int splits) {
  return static_cast<int64_t>(splits) * round_up(rows, kBM) * round_up(kf, bn);
}

}  // namespace lgb
