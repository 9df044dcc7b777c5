// Declarations shared by the entry-point files (lora_linear.cu, lora_mlp.cu,
// lora_qkvo.cu); lora_api.cu defines them.
#pragma once

#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdint>

#include "host.cuh"

namespace lgb {

#define LGB_TRY(expr)                       \
  do {                                      \
    lora_status_t _st = (expr);             \
    if (_st != LORA_OK) return _st;         \
  } while (0)

typedef __nv_bfloat16 bf16;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline bool lin_ok(const lora_linear_t& l) { return l.W && l.A && l.B; }
inline bool lin_aligned(const lora_linear_t& l) { return aligned(l.W, 16) && aligned(l.A, 2) && aligned(l.B, 2); }
inline static void check_size(int64_t v, lora_status_t& st) {
  if (v <= 0) {
    st = LORA_ERR_INVALID_ARG;
  } else if (v > kMaxExtent && st == LORA_OK) {
    st = LORA_ERR_UNSUPPORTED;
  }
}

// M >= 0 (LORA_ERR_UNSUPPORTED above kMaxExtent), r >= 1, s finite.
lora_status_t check_common(int64_t M, int r, float s);

// An NVTX range around each entry point, so that profilers can attribute the launches
// to the call (no cost beyond a pointer test when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Adapter packing: block `src` (row stride lds) lands at (ro, co) of job J's dense
// destination, optionally transposed and scaled.
void pack_block(PackJob& J, const void* src, int64_t lds, int ro, int co, int R, int C, int trans, float scale);
PackJob& pack_job(PackParams& P, void* dst, int64_t rows, int64_t cols);

// C[M x kf] = src[M x K] * P^T with P [kf x K] packed (token-major rank-r
// projection), written as bf16 into dst [M x kf].  `extra` adds more (src, P, K)
// segments summed into the same output.
struct ProjSeg {
  const void* src;
  const void* P;
  int64_t K;
};
// dst_t (optional): columns [0, ntrans) of the result transposed, [ntrans x ldt] (ldt >= M,
// a multiple of 8).
lora_status_t rank_projection(int64_t M, int kf, const ProjSeg* segs, int nseg, void* dst, float* part,
                              unsigned* status, cudaStream_t st, void* dst_t = nullptr, int64_t ldt = 0,
                              int ntrans = 0);
// f32 slab elements of a rank-r projection over ktotal_blocks 64-wide k-blocks.
int64_t rank_projection_part(int64_t M, int kf, int64_t ktotal_blocks);

// Reductions over tokens: for each job j, D_j[f x kf] = Q_j[tokens x f]^T * T_j[tokens x kf],
// then out = s * D_j[:, col0 .. col0+r) written as [f x r] (dB) or transposed [r x f] (dA).
struct GradJob {
  const void* Q;      // [M x f] token-major
  int64_t f;
  int col0;           // rank slot inside T
  void* dst;
  int trans;          // 1: dst is [r x f] (dA), 0: dst is [f x r] (dB)
  const void* T;      // [M x kf] token-major rank-r operand
  int kf = 0;         // T's padded width when it differs from the call's kf (0: the call's)
};
// f32 slab elements of the token reductions of n products (fs[j] features each).
// n_ex > 0: per-example mode, one slab per example.
int64_t token_grad_part(int64_t M, int kf, const int64_t* fs, int n, int64_t n_ex = 0);

// Reductions over tokens whose results no later launch of a call reads (the dA, dB
// outputs): each keeps its own f32 slabs, and one reduce launch at the end of the call
// sums them all.
struct Deferred {
  RedParams rp;
  float* cursor;      // next free slab element
};
void defer_init(Deferred& d, float* slabs);
lora_status_t defer_flush(Deferred& d, cudaStream_t st);
// Reductions over tokens of the jobs in one launch (see lora_api.cu); late: the launch
// reads nothing the previous kernel writes and writes nothing it reads (pdl_late).  kf is
// the widest rank operand of the jobs (it picks the tile width); a job's own kf, when
// set, is its operand's width, with the same tile width (skinny_bn) as kf's.
lora_status_t token_grads(int64_t M, int r, int kf, float s, const GradJob* jobs, int njobs, Deferred& defer,
                          unsigned* status, cudaStream_t st, int64_t n_ex = 0, bool late = false);

// One pass over token-major gradients Q_p that gives both of their rank-r products
// (rank_dual.cuh): V[M x kf] (columns [0, nv), nv = the slots' extent rounded to 16)
// = sum_p Q_p Bt_p^T, and dB_p = s Q_p^T T_p[:, slot_p] written as [F_p x r].  T^T is
// the transposed rank-r operand [kf x ldt].  V is summed from its f32 slab (vslab) at
// once; the dB sums are left to `defer`.  Only where dual_supported.
struct DualJob {
  const void* Q;      // [M x F] token-major
  int64_t F;
  const void* Bt;     // [kf x F] packed: this product's rows of B^T in its V slots, zero elsewhere
  int t_row;          // first row of this product's slot in T^T
  void* dB;           // [F x r]
};
inline bool dual_supported(int r, int kf, int nprod) {
  return nprod >= 1 && nprod <= kDualMaxProducts && r <= kDualNRMax && nprod * r <= kDualNVMax &&
         kf >= static_cast<int>(round_up(nprod * r, 16));
}
// f32 elements of the V slab and of the dB slabs (sum over the jobs) of one pass.
void dual_slab_elems(int64_t M, int r, const int64_t* F, int njobs, int64_t& v_elems, int64_t& db_elems);
lora_status_t rank_dual(int64_t M, int r, int kf, float s, const DualJob* jobs, int njobs, const void* Tt,
                        int64_t ldt, void* V, float* vslab, Deferred& defer, unsigned* status, cudaStream_t st);

lora_status_t launch_rope(const RopeParams& p, cudaStream_t st);

// lora_linear_forward for inference with the projection on whole tiles only (no
// split tail), and the workspace bytes that needs (less than
// lora_linear_workspace_bytes, which also covers the backward and the tail's regions;
// 0 for invalid sizes).  Defined in lora_linear.cu.
lora_status_t linear_forward_whole_tiles(int64_t M, int64_t in, int64_t out, int r, float s, const void* x,
                                         lora_linear_t lin, void* y, void* ws, size_t ws_bytes, cudaStream_t stream);
size_t linear_forward_workspace_bytes(int64_t M, int64_t in, int64_t out, int r);
// Device address of lora_linear_forward_noalloc's fixed scratch on the current device
// (its first 256 bytes are that call's status word), or NULL on a CUDA error.
// Defined in noalloc.cu.
void* noalloc_scratch();

}  // namespace lgb
