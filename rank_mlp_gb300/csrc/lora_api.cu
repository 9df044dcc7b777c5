// C-ABI entry points: argument checks, workspace carving, and the launch sequence of
// each operation on the caller's stream.  See include/lora_gb300.h for the contract.
#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "host.cuh"
#include "aux_kernels_impl.cuh"

namespace lgb {

// ---------------------------------------------------------------- device plumbing

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// 2-D bf16 map with 128-byte swizzle; out-of-bounds elements read as zero.
bool encode_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || inner == 0 || outer == 0) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map {inner, d1, d2} with row stride ld (elements) and plane stride
// ld * d1; box {box_inner, box_d1, 1}.
bool encode_map_planes(CUtensorMap* m, const void* base, uint64_t inner, uint64_t d1, uint64_t d2, uint64_t ld,
                       uint32_t box_inner, uint32_t box_d1) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || inner == 0 || d1 == 0 || d2 == 0) return false;
  const cuuint64_t dims[3] = {inner, d1, d2};
  const cuuint64_t strides[2] = {ld * 2, ld * 2 * d1};
  const cuuint32_t box[3] = {box_inner, box_d1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An NVTX range around each entry point, so that profilers can attribute the launches
// to the call (no cost beyond a pointer test when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---------------------------------------------------------------- counters, trace

static std::atomic<uint64_t> g_launches{0};

struct Trace {
  std::mutex mu;
  int capacity = 0;
  std::vector<cudaEvent_t> ev;     // 2 per entry
  std::vector<int> kind;
  int used = 0;
  unsigned kinds = ~0u;            // bit k: launches of kind k are traced
};
static Trace g_trace;

// Records the start event of a traced launch; returns its slot or -1.
static int trace_begin(int kind, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (g_trace.capacity == 0 || g_trace.used >= g_trace.capacity || !((g_trace.kinds >> kind) & 1u)) return -1;
  const int slot = g_trace.used++;
  g_trace.kind[slot] = kind;
  cudaEventRecord(g_trace.ev[2 * slot], st);
  return slot;
}
static void trace_end(int slot, cudaStream_t st) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_trace.mu);
  cudaEventRecord(g_trace.ev[2 * slot + 1], st);
}

// Wait limit of the GEMM kernels' bounded waits, and the number of coming GEMM
// launches that are told to leave one pipeline stage empty (failure-path tests).
static std::atomic<unsigned long long> g_timeout_ns{kTimeoutNs};
static std::atomic<int> g_expire_next{0};

static int take_expiry() {
  int n = g_expire_next.load();
  while (n > 0 && !g_expire_next.compare_exchange_weak(n, n - 1)) {
  }
  return n > 0 ? 1 : 0;
}

lora_status_t launch_gemm(int variant, const TcParams& plan, int kind, cudaStream_t st) {
  if (plan.total_units <= 0) return LORA_OK;
  if (variant == VP_KK) {
    int kb = 0;
    for (int g = 0; g < plan.ngroups; ++g) kb = plan.grp[g].kb_total > kb ? plan.grp[g].kb_total : kb;
    if (kb <= kShortKBlocks) variant = VP_KK8;
  }
  TcParams p = plan;
  p.timeout_ns = g_timeout_ns.load();
  p.inject_stall = take_expiry();
  int grid;
  if (variant_pair(variant)) {
    const int pairs = num_sms() / 2;
    grid = 2 * (p.total_units < pairs ? p.total_units : pairs);
  } else {
    grid = p.total_units < num_sms() ? p.total_units : num_sms();
  }
  const int slot = trace_begin(kind, st);
  cudaError_t e = variant_pair(variant) ? launch_tc_big(variant, p, grid, st) : launch_tc_skinny(variant, p, grid, st);
  trace_end(slot, st);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return LORA_OK;
}

lora_status_t launch_pack(const PackParams& p, cudaStream_t st) {
  if (p.njob == 0) return LORA_OK;
  int64_t most = 1;
  for (int j = 0; j < p.njob; ++j) {
    const int64_t n = static_cast<int64_t>(p.job[j].rows) * (p.job[j].cols / 8);   // 8 elements per thread
    most = n > most ? n : most;
  }
  int64_t gx = ceil_div(most, 256);
  gx = gx > 1024 ? 1024 : gx;
  const int slot = trace_begin(LORA_KIND_PACK, st);
  cudaError_t e = launch_pdl(pack_kernel, dim3(static_cast<unsigned>(gx), p.njob), dim3(256), 0, st, p);
  trace_end(slot, st);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return LORA_OK;
}

lora_status_t launch_norms(const NormParams& p, int examples, cudaStream_t st) {
  if (examples <= 0) return LORA_OK;
  const int slot = trace_begin(LORA_KIND_REDUCE, st);
  cudaError_t e = launch_pdl(norms_kernel, dim3(examples), dim3(256), 0, st, p);
  trace_end(slot, st);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return LORA_OK;
}

lora_status_t launch_reduce(const RedParams& p, cudaStream_t st) {
  if (p.nout == 0) return LORA_OK;
  int64_t most = 1;
  for (int j = 0; j < p.nout; ++j) {
    const int64_t n = static_cast<int64_t>(p.out[j].rows) * p.out[j].ncols;
    most = n > most ? n : most;
  }
  int64_t gx = ceil_div(most, 256);
  gx = gx > 2048 ? 2048 : gx;
  const int slot = trace_begin(LORA_KIND_REDUCE, st);
  cudaError_t e = launch_pdl(reduce_kernel, dim3(static_cast<unsigned>(gx), p.nout), dim3(256), 0, st, p);
  trace_end(slot, st);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return LORA_OK;
}

lora_status_t launch_rope(const RopeParams& p, cudaStream_t st) {
  if (p.ntensors == 0 || p.M == 0) return LORA_OK;
  long long most = 1;
  for (int t = 0; t < p.ntensors; ++t) most = p.M * (p.n[t] / 16) > most ? p.M * (p.n[t] / 16) : most;
  long long gx = ceil_div(most, 256);
  gx = gx > 4 * num_sms() ? 4 * num_sms() : gx;
  const int slot = trace_begin(LORA_KIND_ROPE, st);
  cudaError_t e = launch_pdl(rope_rotate_kernel, dim3(static_cast<unsigned>(gx), p.ntensors), dim3(256), 0, st, p);
  trace_end(slot, st);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return LORA_OK;
}

// ---------------------------------------------------------------- building blocks

#define LGB_TRY(expr)                       \
  do {                                      \
    lora_status_t _st = (expr);             \
    if (_st != LORA_OK) return _st;         \
  } while (0)

typedef __nv_bfloat16 bf16;

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

static void pack_block(PackJob& J, const void* src, int64_t lds, int ro, int co, int R, int C, int trans,
                       float scale) {
  PackBlock& B = J.blk[J.nblk++];
  B.src = static_cast<const bf16*>(src);
  B.lds = lds;
  B.ro = ro;
  B.co = co;
  B.R = R;
  B.C = C;
  B.trans = trans;
  B.scale = scale;
}
static PackJob& pack_job(PackParams& P, void* dst, int64_t rows, int64_t cols) {
  PackJob& J = P.job[P.njob++];
  J.dst = static_cast<bf16*>(dst);
  J.rows = static_cast<int>(rows);
  J.cols = static_cast<int>(cols);
  J.nblk = 0;
  return J;
}

// C[M x kf] = src[M x K] * P^T with P [kf x K] packed (token-major rank-r
// projection), written as bf16 into dst [M x kf].  `extra` adds more (src, P, K)
// segments summed into the same output.
struct ProjSeg {
  const void* src;
  const void* P;
  int64_t K;
};
static lora_status_t rank_projection(int64_t M, int kf, const ProjSeg* segs, int nseg, void* dst, float* part,
                                     unsigned* status, cudaStream_t st) {
  const int variant = skinny_kk(kf);
  GemmPlan g(variant);
  int64_t kb = 0;
  for (int s = 0; s < nseg; ++s) kb += ceil_div(segs[s].K, kBK);
  const int64_t tiles = ceil_div(M, kBM) * ceil_div(kf, g.bn);
  const int splits = choose_splits(tiles, kb, num_sms());
  GroupDesc& G = g.group(static_cast<int>(M), kf, splits > 1 ? EPI_PARTIAL : EPI_STORE, false);
  G.splits = splits;
  for (int s = 0; s < nseg; ++s) {
    const int a = g.a_kmajor(segs[s].src, M, segs[s].K, segs[s].K);
    const int b = g.b_kmajor(segs[s].P, kf, segs[s].K, segs[s].K, g.bn);
    GemmPlan::seg(G, a, b, -1, segs[s].K, segs[s].K);
  }
  if (splits > 1) {
    G.part = part;
  } else {
    G.out0 = dst;
    G.ldo = kf;
  }
  g.p.status = status;
  g.finish();
  if (!g.ok) return LORA_ERR_CUDA;
  LGB_TRY(launch_gemm(variant, g.p, LORA_KIND_RANK_PROJ, st));
  if (splits > 1) {
    RedParams r;
    std::memset(static_cast<void*>(&r), 0, sizeof(r));
    r.nout = 1;
    RedOut& o = r.out[0];
    o.splits = splits;
    o.scale = 1.0f;
    o.part = part;
    o.rows = static_cast<int>(M);
    o.rows_pad = round_up(M, kBM);
    o.width = static_cast<int>(round_up(kf, g.bn));
    o.dst = static_cast<bf16*>(dst);
    o.col0 = 0;
    o.ncols = kf;
    o.ld = kf;
    o.trans = 0;
    LGB_TRY(launch_reduce(r, st));
  }
  return LORA_OK;
}
static int64_t rank_projection_part(int64_t M, int kf, int64_t ktotal_blocks) {
  const int splits = max_splits(ktotal_blocks);
  return splits > 1 ? partial_elems(M, kf, skinny_bn(kf), splits) : 0;
}

// Reductions over tokens: for each job j, D_j[f x kf] = Q_j[tokens x f]^T * T[tokens x kf],
// then out = s * D_j[:, col0 .. col0+r) written as [f x r] (dB) or transposed [r x f] (dA).
struct GradJob {
  const void* Q;      // [M x f] token-major
  int64_t f;
  int col0;           // rank slot inside T
  void* dst;
  int trans;          // 1: dst is [r x f] (dA), 0: dst is [f x r] (dB)
};
// f32 slab elements of the token reductions of n products (fs[j] features each).
// n_ex > 0: per-example mode, one slab per example.
static int64_t token_grad_part(int64_t M, int kf, const int64_t* fs, int n, int64_t n_ex = 0) {
  const int bn = skinny_bn(kf);
  const int splits = n_ex > 0 ? static_cast<int>(n_ex) : max_splits(ceil_div(M, kBK));
  int64_t tot = 0;
  for (int j = 0; j < n; ++j) tot += round_up(partial_elems(fs[j], kf, bn, splits), 64);
  return tot;
}
// Reductions over tokens whose results no later launch of a call reads (the dA, dB
// outputs): each keeps its own f32 slabs, and one reduce launch at the end of the call
// sums them all.
struct Deferred {
  RedParams rp;
  float* cursor;      // next free slab element
};
static void defer_init(Deferred& d, float* slabs) {
  std::memset(static_cast<void*>(&d.rp), 0, sizeof(d.rp));
  d.cursor = slabs;
}
static lora_status_t defer_flush(Deferred& d, cudaStream_t st) {
  const lora_status_t r = launch_reduce(d.rp, st);
  d.rp.nout = 0;
  return r;
}

// Jobs with the same Q share one slab (several rank slots out of one product).
// n_ex == 0: the sums over all M tokens.  n_ex > 0: one result per example (example e
// = tokens [e seq, (e+1) seq), seq = M / n_ex), each written at dst + e * r * f; the
// products read 3-D views {features, seq, examples} so no k-block straddles two
// examples (rows past seq read as zero).  The slabs start at defer.cursor and the
// sums are left to defer_flush.
// late: the launch follows a kernel whose outputs it does not read (and whose inputs
// it does not write), so it may start on SMs that kernel has freed (pdl_late).
static lora_status_t token_grads(int64_t M, int r, int kf, float s, const void* T, const GradJob* jobs, int njobs,
                                 Deferred& defer, unsigned* status, cudaStream_t st, int64_t n_ex = 0,
                                 bool late = false) {
  const int variant = skinny_mnmn(kf);
  GemmPlan g(variant);
  g.p.pdl_late = late ? 1 : 0;
  const int64_t seq = n_ex > 0 ? M / n_ex : M;
  const int tmap = n_ex > 0 ? g.b_mnmajor_planes(T, kf, seq, n_ex, kf) : g.b_mnmajor(T, kf, M, kf);
  const void* qs[kMaxGroups];
  int nq = 0, group_of[kMaxGroups * 3];
  float* parts[kMaxGroups];
  float* cur = defer.cursor;
  const int slab_splits = n_ex > 0 ? static_cast<int>(n_ex) : max_splits(ceil_div(M, kBK));
  for (int j = 0; j < njobs; ++j) {
    int gi = -1;
    for (int q = 0; q < nq; ++q)
      if (qs[q] == jobs[j].Q) gi = q;
    if (gi < 0) {
      gi = nq++;
      qs[gi] = jobs[j].Q;
      const int64_t tiles = ceil_div(jobs[j].f, kBM) * ceil_div(kf, g.bn);
      GroupDesc& G = g.group(static_cast<int>(jobs[j].f), kf, EPI_PARTIAL, false);
      if (n_ex > 0) {
        G.splits = static_cast<int>(n_ex);
        G.per_plane = 1;
        const int a = g.a_mnmajor_planes(jobs[j].Q, jobs[j].f, seq, n_ex, jobs[j].f);
        GemmPlan::seg(G, a, tmap, -1, seq, seq);
      } else {
        G.splits = choose_splits(tiles, ceil_div(M, kBK), num_sms());
        const int a = g.a_mnmajor(jobs[j].Q, jobs[j].f, M, jobs[j].f);
        GemmPlan::seg(G, a, tmap, -1, M, M);
      }
      G.part = cur;
      parts[gi] = cur;
      cur += round_up(partial_elems(jobs[j].f, kf, g.bn, slab_splits), 64);
    }
    group_of[j] = gi;
  }
  g.p.status = status;
  g.finish();
  if (!g.ok) return LORA_ERR_CUDA;
  LGB_TRY(launch_gemm(variant, g.p, LORA_KIND_RANK_GRAD, st));
  defer.cursor = cur;
  for (int j = 0; j < njobs; ++j) {
    if (defer.rp.nout >= kMaxRedOuts) return LORA_ERR_UNSUPPORTED;   // not reached: <= 8 per call
    RedOut& o = defer.rp.out[defer.rp.nout++];
    o.part = parts[group_of[j]];
    o.rows = static_cast<int>(jobs[j].f);
    o.rows_pad = round_up(jobs[j].f, kBM);
    o.width = static_cast<int>(round_up(kf, g.bn));
    o.splits = g.p.grp[group_of[j]].splits;
    o.per_split = n_ex > 0 ? 1 : 0;
    o.scale = s;
    o.dst = static_cast<bf16*>(jobs[j].dst);
    o.col0 = jobs[j].col0;
    o.ncols = r;
    o.ld = jobs[j].trans ? jobs[j].f : r;
    o.trans = jobs[j].trans;
    o.split_stride = static_cast<long long>(r) * jobs[j].f;
  }
  return LORA_OK;
}

static void check_size(int64_t v, lora_status_t& st) {
  if (v <= 0) st = LORA_ERR_INVALID_ARG;
}

}  // namespace lgb

using namespace lgb;

// ================================================================ single linear

namespace {

struct LinearLayout {
  int kf;
  size_t ws_fwd, ws_bwd, saved;
};

LinearLayout linear_layout(int64_t M, int64_t in, int64_t out, int r) {
  LinearLayout L;
  L.kf = fold_width(1, r);
  const int kf = L.kf;
  {
    Carve c(nullptr);
    c.take(kWsHeader);
    c.take_n<bf16>(kf * in);    // Acat
    c.take_n<bf16>(out * kf);   // BF
    c.take_n<float>(rank_projection_part(M, kf, ceil_div(in, kBK)));
    c.take_n<bf16>(M * kf);     // T when there is no saved blob
    L.ws_fwd = c.off;
  }
  {
    Carve c(nullptr);
    c.take(kWsHeader);
    c.take_n<bf16>(kf * out);   // B^T
    c.take_n<bf16>(kf * in);    // s A
    c.take_n<bf16>(M * kf);     // U
    c.take_n<float>(rank_projection_part(M, kf, ceil_div(out, kBK)));
    c.take_n<float>(token_grad_part(M, kf, &out, 1) + token_grad_part(M, kf, &in, 1));   // dB, dA slabs
    L.ws_bwd = c.off;
  }
  {
    Carve c(nullptr);
    c.take_n<bf16>(M * kf);
    L.saved = c.off;
  }
  return L;
}

lora_status_t check_common(int64_t M, int r, float s) {
  if (M < 0 || r < 1 || !std::isfinite(s)) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

}  // namespace

extern "C" size_t lora_linear_saved_bytes(int64_t M, int64_t in, int64_t out, int r) {
  if (M < 0 || in <= 0 || out <= 0 || r < 1) return 0;
  return linear_layout(M, in, out, r).saved;
}
extern "C" size_t lora_linear_workspace_bytes(int64_t M, int64_t in, int64_t out, int r) {
  if (M < 0 || in <= 0 || out <= 0 || r < 1) return 0;
  const LinearLayout L = linear_layout(M, in, out, r);
  return L.ws_fwd > L.ws_bwd ? L.ws_fwd : L.ws_bwd;
}

extern "C" lora_status_t lora_linear_forward(int64_t M, int64_t in, int64_t out, int r, float s, const void* x,
                                             lora_linear_t lin, void* y, void* saved, void* ws, size_t ws_bytes,
                                             cudaStream_t stream) {
  NvtxRange nvtx_range("lora_linear_forward");
  lora_status_t st = check_common(M, r, s);
  check_size(in, st);
  check_size(out, st);
  if (st != LORA_OK) return st;
  const bool tok = M > 0;   // activations may be NULL when there are no tokens
  if ((tok && (x == nullptr || y == nullptr)) || lin.W == nullptr || lin.A == nullptr || lin.B == nullptr ||
      ws == nullptr)
    return LORA_ERR_INVALID_ARG;
  if (r > 256) return LORA_ERR_UNSUPPORTED;
  if (in % 8 || out % 8 || !aligned(x, 16) || !aligned(y, 16) || !aligned(lin.W, 16) || !aligned(lin.A, 2) ||
      !aligned(lin.B, 2) || !aligned(ws, 256) || (saved && !aligned(saved, 256)))
    return LORA_ERR_ALIGNMENT;
  const LinearLayout L = linear_layout(M, in, out, r);
  if (ws_bytes < L.ws_fwd) return LORA_ERR_WORKSPACE;
  if (M == 0) return LORA_OK;
  const int kf = L.kf;
  Carve c(ws);
  unsigned* status = static_cast<unsigned*>(c.take(kWsHeader));
  bf16* acat = c.take_n<bf16>(kf * in);
  bf16* bf = c.take_n<bf16>(out * kf);
  float* part = c.take_n<float>(rank_projection_part(M, kf, ceil_div(in, kBK)));
  bf16* T = c.take_n<bf16>(M * kf);
  if (saved) T = static_cast<bf16*>(saved);

  PackParams pk;
  std::memset(static_cast<void*>(&pk), 0, sizeof(pk));
  pack_block(pack_job(pk, acat, kf, in), lin.A, in, 0, 0, r, static_cast<int>(in), 0, 1.0f);
  pack_block(pack_job(pk, bf, out, kf), lin.B, r, 0, 0, static_cast<int>(out), r, 0, s);
  LGB_TRY(launch_pack(pk, stream));

  const ProjSeg ps = {x, acat, in};
  LGB_TRY(rank_projection(M, kf, &ps, 1, T, part, status, stream));

  GemmPlan g(kBigKK);
  GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(out), EPI_STORE, false);
  GemmPlan::seg(G, g.a_kmajor(x, M, in, in), g.b_kmajor(lin.W, out, in, in, g.b_rows_full()), -1, in, in);
  GemmPlan::seg(G, g.a_kmajor(T, M, kf, kf), g.b_kmajor(bf, out, kf, kf, g.b_rows_full()), -1, kf, r);
  G.out0 = y;
  G.ldo = out;
  g.p.status = status;
  g.finish();
  if (!g.ok) return LORA_ERR_CUDA;
  return launch_gemm(kBigKK, g.p, LORA_KIND_PROJ, stream);
}

extern "C" lora_status_t lora_linear_backward(int64_t M, int64_t in, int64_t out, int r, float s, const void* x,
                                              lora_linear_t lin, const void* saved, const void* dy, void* dx,
                                              lora_grads_t grads, void* ws, size_t ws_bytes,
                                              cudaStream_t stream) {
  NvtxRange nvtx_range("lora_linear_backward");
  lora_status_t st = check_common(M, r, s);
  check_size(in, st);
  check_size(out, st);
  if (st != LORA_OK) return st;
  const bool tok = M > 0;
  if ((tok && (x == nullptr || dy == nullptr || dx == nullptr)) || saved == nullptr || lin.W == nullptr ||
      lin.A == nullptr || lin.B == nullptr || grads.dA == nullptr || grads.dB == nullptr || ws == nullptr)
    return LORA_ERR_INVALID_ARG;
  if (r > 256) return LORA_ERR_UNSUPPORTED;
  if (in % 8 || out % 8 || !aligned(x, 16) || !aligned(dy, 16) || !aligned(dx, 16) || !aligned(lin.W, 16) ||
      !aligned(lin.A, 2) || !aligned(lin.B, 2) || !aligned(grads.dA, 2) || !aligned(grads.dB, 2) ||
      !aligned(ws, 256) || !aligned(saved, 256))
    return LORA_ERR_ALIGNMENT;
  const LinearLayout L = linear_layout(M, in, out, r);
  if (ws_bytes < L.ws_bwd) return LORA_ERR_WORKSPACE;
  if (M == 0) {
    if (cudaMemsetAsync(grads.dA, 0, sizeof(bf16) * r * in, stream) != cudaSuccess ||
        cudaMemsetAsync(grads.dB, 0, sizeof(bf16) * out * r, stream) != cudaSuccess)
      return LORA_ERR_CUDA;
    return LORA_OK;
  }
  const int kf = L.kf;
  Carve c(ws);
  unsigned* status = static_cast<unsigned*>(c.take(kWsHeader));
  bf16* bt = c.take_n<bf16>(kf * out);
  bf16* af = c.take_n<bf16>(kf * in);
  bf16* U = c.take_n<bf16>(M * kf);
  float* part = c.take_n<float>(rank_projection_part(M, kf, ceil_div(out, kBK)));
  Deferred dr;
  defer_init(dr, c.take_n<float>(token_grad_part(M, kf, &out, 1) + token_grad_part(M, kf, &in, 1)));
  const bf16* T = static_cast<const bf16*>(saved);

  PackParams pk;
  std::memset(static_cast<void*>(&pk), 0, sizeof(pk));
  pack_block(pack_job(pk, bt, kf, out), lin.B, r, 0, 0, r, static_cast<int>(out), 1, 1.0f);
  pack_block(pack_job(pk, af, kf, in), lin.A, in, 0, 0, r, static_cast<int>(in), 0, s);
  LGB_TRY(launch_pack(pk, stream));

  const ProjSeg ps = {dy, bt, out};
  LGB_TRY(rank_projection(M, kf, &ps, 1, U, part, status, stream));

  GemmPlan g(kBigKMN);
  GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(in), EPI_STORE, false);
  GemmPlan::seg(G, g.a_kmajor(dy, M, out, out), g.b_mnmajor(lin.W, in, out, in), -1, out, out);
  GemmPlan::seg(G, g.a_kmajor(U, M, kf, kf), g.b_mnmajor(af, in, kf, in), -1, kf, r);
  G.out0 = dx;
  G.ldo = in;
  g.p.status = status;
  g.finish();
  if (!g.ok) return LORA_ERR_CUDA;
  LGB_TRY(launch_gemm(kBigKMN, g.p, LORA_KIND_DGRAD, stream));

  const GradJob ja = {x, in, 0, grads.dA, 1};
  // dB = s dy^T T and dA = s U^T x read nothing the dx GEMM writes
  const GradJob jb = {dy, out, 0, grads.dB, 0};
  LGB_TRY(token_grads(M, r, kf, s, T, &jb, 1, dr, status, stream, 0, true));
  LGB_TRY(token_grads(M, r, kf, s, U, &ja, 1, dr, status, stream, 0, true));
  return defer_flush(dr, stream);
}

// ================================================================ gated MLP

namespace {

struct MlpLayout {
  int kfg, kfd;    // padded rank widths: gate/up pair, down
  size_t ws_fwd, ws_bwd, saved;
  // saved blob offsets
  size_t off_g, off_u, off_h, off_tgu, off_td;
};

// n_ex > 0: workspace of the per-example backward (one reduction slab per example).
// Backward scratch: the rank-r projections' split-K slabs (reused), then the four token
// reductions' slabs (kept until the call's final reduce).
static int64_t mlp_bwd_rank_part(int64_t M, int64_t h, int64_t i, int kfd, int kfg) {
  return imax(rank_projection_part(M, kfd, ceil_div(h, kBK)), rank_projection_part(M, kfg, 2 * ceil_div(i, kBK)));
}
static int64_t mlp_bwd_slabs(int64_t M, int64_t h, int64_t i, int kfd, int kfg, int64_t n_ex) {
  const int64_t f2[2] = {i, i};
  return token_grad_part(M, kfd, &h, 1, n_ex) + token_grad_part(M, kfd, &i, 1, n_ex) +
         token_grad_part(M, kfg, f2, 2, n_ex) + token_grad_part(M, kfg, &h, 1, n_ex);
}

MlpLayout mlp_layout(int64_t M, int64_t h, int64_t i, int r, int64_t n_ex = 0) {
  MlpLayout L;
  L.kfg = fold_width(2, r);
  L.kfd = fold_width(1, r);
  const int kfg = L.kfg, kfd = L.kfd;
  {
    Carve c(nullptr);
    c.take(kWsHeader);
    c.take_n<bf16>(kfg * h);
    c.take_n<bf16>(i * kfg);
    c.take_n<bf16>(i * kfg);
    c.take_n<bf16>(kfd * i);
    c.take_n<bf16>(h * kfd);
    int64_t p = rank_projection_part(M, kfg, ceil_div(h, kBK));
    const int64_t p2 = rank_projection_part(M, kfd, ceil_div(i, kBK));
    c.take_n<float>(p > p2 ? p : p2);
    c.take_n<bf16>(M * i);       // h, T_gu, T_d when there is no saved blob
    c.take_n<bf16>(M * kfg);
    c.take_n<bf16>(M * kfd);
    L.ws_fwd = c.off;
  }
  {
    Carve c(nullptr);
    c.take(kWsHeader);
    c.take_n<bf16>(kfd * h);     // B_d^T
    c.take_n<bf16>(kfd * i);     // s A_d
    c.take_n<bf16>(kfg * i);     // B_g^T
    c.take_n<bf16>(kfg * i);     // B_u^T
    c.take_n<bf16>(kfg * h);     // s [A_g; A_u]
    c.take_n<bf16>(M * kfd);     // U_d
    c.take_n<bf16>(M * i);       // dg
    c.take_n<bf16>(M * i);       // du
    c.take_n<bf16>(M * kfg);     // V
    c.take_n<float>(mlp_bwd_rank_part(M, h, i, kfd, kfg));
    c.take_n<float>(mlp_bwd_slabs(M, h, i, kfd, kfg, n_ex));
    L.ws_bwd = c.off;
  }
  {
    Carve c(nullptr);
    L.off_g = c.offset_of(sizeof(bf16) * M * i);
    L.off_u = c.offset_of(sizeof(bf16) * M * i);
    L.off_h = c.offset_of(sizeof(bf16) * M * i);
    L.off_tgu = c.offset_of(sizeof(bf16) * M * kfg);
    L.off_td = c.offset_of(sizeof(bf16) * M * kfd);
    L.saved = c.off;
  }
  return L;
}

lora_status_t check_mlp(int64_t M, int64_t h, int64_t i, int r, float s, int act) {
  lora_status_t st = check_common(M, r, s);
  check_size(h, st);
  check_size(i, st);
  if (st != LORA_OK) return st;
  if (act != LORA_ACT_SWIGLU && act != LORA_ACT_GEGLU_TANH && act != LORA_ACT_GEGLU_ERF) return LORA_ERR_INVALID_ARG;
  if (2 * r > 256) return LORA_ERR_UNSUPPORTED;
  if (h % 8 || i % 8) return LORA_ERR_ALIGNMENT;
  return LORA_OK;
}

bool lin_ok(const lora_linear_t& l) { return l.W && l.A && l.B; }
bool lin_aligned(const lora_linear_t& l) { return aligned(l.W, 16) && aligned(l.A, 2) && aligned(l.B, 2); }

}  // namespace

extern "C" size_t lora_mlp_saved_bytes(int64_t M, int64_t h, int64_t i, int r) {
  if (M < 0 || h <= 0 || i <= 0 || r < 1) return 0;
  return mlp_layout(M, h, i, r).saved;
}
extern "C" size_t lora_mlp_workspace_bytes(int64_t M, int64_t h, int64_t i, int r) {
  if (M < 0 || h <= 0 || i <= 0 || r < 1) return 0;
  const MlpLayout L = mlp_layout(M, h, i, r);
  return L.ws_fwd > L.ws_bwd ? L.ws_fwd : L.ws_bwd;
}

extern "C" lora_status_t lora_mlp_forward(int64_t M, int64_t h, int64_t i, int r, float s, lora_act_t act,
                                          const void* x, lora_linear_t gate, lora_linear_t up,
                                          lora_linear_t down, void* y, void* saved, void* ws, size_t ws_bytes,
                                          cudaStream_t stream) {
  NvtxRange nvtx_range("lora_mlp_forward");
  LGB_TRY(check_mlp(M, h, i, r, s, static_cast<int>(act)));
  if ((M > 0 && (!x || !y)) || !ws || !lin_ok(gate) || !lin_ok(up) || !lin_ok(down)) return LORA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !lin_aligned(gate) || !lin_aligned(up) || !lin_aligned(down) ||
      !aligned(ws, 256) || (saved && !aligned(saved, 256)))
    return LORA_ERR_ALIGNMENT;
  const MlpLayout L = mlp_layout(M, h, i, r);
  if (ws_bytes < L.ws_fwd) return LORA_ERR_WORKSPACE;
  if (M == 0) return LORA_OK;
  const int kfg = L.kfg, kfd = L.kfd;
  Carve c(ws);
  unsigned* status = static_cast<unsigned*>(c.take(kWsHeader));
  bf16* acat_gu = c.take_n<bf16>(kfg * h);
  bf16* bf_g = c.take_n<bf16>(i * kfg);
  bf16* bf_u = c.take_n<bf16>(i * kfg);
  bf16* acat_d = c.take_n<bf16>(kfd * i);
  bf16* bf_d = c.take_n<bf16>(h * kfd);
  int64_t pe = rank_projection_part(M, kfg, ceil_div(h, kBK));
  const int64_t pe2 = rank_projection_part(M, kfd, ceil_div(i, kBK));
  float* part = c.take_n<float>(pe > pe2 ? pe : pe2);
  bf16* hbuf = c.take_n<bf16>(M * i);
  bf16* tgu = c.take_n<bf16>(M * kfg);
  bf16* td = c.take_n<bf16>(M * kfd);
  bf16* gbuf = nullptr;
  bf16* ubuf = nullptr;
  if (saved) {
    uint8_t* sv = static_cast<uint8_t*>(saved);
    gbuf = reinterpret_cast<bf16*>(sv + L.off_g);
    ubuf = reinterpret_cast<bf16*>(sv + L.off_u);
    hbuf = reinterpret_cast<bf16*>(sv + L.off_h);
    tgu = reinterpret_cast<bf16*>(sv + L.off_tgu);
    td = reinterpret_cast<bf16*>(sv + L.off_td);
  }

  PackParams pk;
  std::memset(static_cast<void*>(&pk), 0, sizeof(pk));
  {
    PackJob& J = pack_job(pk, acat_gu, kfg, h);
    pack_block(J, gate.A, h, 0, 0, r, static_cast<int>(h), 0, 1.0f);
    pack_block(J, up.A, h, r, 0, r, static_cast<int>(h), 0, 1.0f);
  }
  pack_block(pack_job(pk, bf_g, i, kfg), gate.B, r, 0, 0, static_cast<int>(i), r, 0, s);
  pack_block(pack_job(pk, bf_u, i, kfg), up.B, r, 0, r, static_cast<int>(i), r, 0, s);
  pack_block(pack_job(pk, acat_d, kfd, i), down.A, i, 0, 0, r, static_cast<int>(i), 0, 1.0f);
  pack_block(pack_job(pk, bf_d, h, kfd), down.B, r, 0, 0, static_cast<int>(h), r, 0, s);
  LGB_TRY(launch_pack(pk, stream));

  // T_gu = x [A_g; A_u]^T
  const ProjSeg p1 = {x, acat_gu, h};
  LGB_TRY(rank_projection(M, kfg, &p1, 1, tgu, part, status, stream));

  // [g | u] = [x | T_gu] [W_g | s B_g ; W_u | s B_u]^T, gate and up halves per tile; h = act(g) u
  {
    GemmPlan g(kBigKK);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(i), EPI_ACT_FWD, true);
    GemmPlan::seg(G, g.a_kmajor(x, M, h, h), g.b_kmajor(gate.W, i, h, h, 128), g.b_kmajor(up.W, i, h, h, 128), h,
                  h);
    GemmPlan::seg(G, g.a_kmajor(tgu, M, kfg, kfg), g.b_kmajor(bf_g, i, kfg, kfg, 128),
                  g.b_kmajor(bf_u, i, kfg, kfg, 128), kfg, 2 * r);
    G.out0 = hbuf;
    G.out1 = gbuf;
    G.out2 = ubuf;
    G.ldo = i;
    g.p.act = static_cast<int>(act);
    g.p.status = status;
    g.finish();
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKK, g.p, LORA_KIND_GATE_UP, stream));
  }

  // T_d = h A_d^T
  const ProjSeg p2 = {hbuf, acat_d, i};
  LGB_TRY(rank_projection(M, kfd, &p2, 1, td, part, status, stream));

  // y = [h | T_d] [W_d | s B_d]^T
  GemmPlan g(kBigKK);
  GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(h), EPI_STORE, false);
  GemmPlan::seg(G, g.a_kmajor(hbuf, M, i, i), g.b_kmajor(down.W, h, i, i, g.b_rows_full()), -1, i, i);
  GemmPlan::seg(G, g.a_kmajor(td, M, kfd, kfd), g.b_kmajor(bf_d, h, kfd, kfd, g.b_rows_full()), -1, kfd, r);
  G.out0 = y;
  G.ldo = h;
  g.p.status = status;
  g.finish();
  if (!g.ok) return LORA_ERR_CUDA;
  return launch_gemm(kBigKK, g.p, LORA_KIND_PROJ, stream);
}

// Backward of the gated MLP.  n_ex == 0: dA/dB summed over all tokens.  n_ex > 0:
// dA/dB per example (n_ex examples of M / n_ex consecutive tokens, written at
// example stride), plus their squared norms into sq_norms when it is not NULL.
static lora_status_t mlp_backward_impl(int64_t M, int64_t h, int64_t i, int r, float s, lora_act_t act,
                                       int64_t n_ex, const void* x, lora_linear_t gate, lora_linear_t up,
                                       lora_linear_t down, const void* saved, const void* dy, void* dx,
                                       lora_grads_t d_gate, lora_grads_t d_up, lora_grads_t d_down, float* sq_norms,
                                       void* ws, size_t ws_bytes, cudaStream_t stream) {
  LGB_TRY(check_mlp(M, h, i, r, s, static_cast<int>(act)));
  if ((M > 0 && (!x || !dy || !dx)) || !saved || !ws || !lin_ok(gate) || !lin_ok(up) || !lin_ok(down) || !d_gate.dA ||
      !d_gate.dB || !d_up.dA || !d_up.dB || !d_down.dA || !d_down.dB)
    return LORA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(dy, 16) || !aligned(dx, 16) || !lin_aligned(gate) || !lin_aligned(up) ||
      !lin_aligned(down) || !aligned(ws, 256) || !aligned(saved, 256) || !aligned(d_gate.dA, 2) ||
      !aligned(d_gate.dB, 2) || !aligned(d_up.dA, 2) || !aligned(d_up.dB, 2) || !aligned(d_down.dA, 2) ||
      !aligned(d_down.dB, 2))
    return LORA_ERR_ALIGNMENT;
  if (n_ex < 0 || (n_ex > 0 && M % n_ex != 0)) return LORA_ERR_INVALID_ARG;
  if (sq_norms != nullptr && !aligned(sq_norms, 4)) return LORA_ERR_ALIGNMENT;
  const MlpLayout L = mlp_layout(M, h, i, r, n_ex);
  if (ws_bytes < L.ws_bwd) return LORA_ERR_WORKSPACE;
  if (M == 0) {
    const size_t ne = n_ex > 0 ? static_cast<size_t>(n_ex) : 1;
    const size_t ah = ne * sizeof(bf16) * r * h, ai = ne * sizeof(bf16) * r * i;
    if (n_ex > 0 && sq_norms != nullptr && cudaMemsetAsync(sq_norms, 0, sizeof(float) * n_ex, stream) != cudaSuccess)
      return LORA_ERR_CUDA;
    if (cudaMemsetAsync(d_gate.dA, 0, ah, stream) || cudaMemsetAsync(d_gate.dB, 0, ai, stream) ||
        cudaMemsetAsync(d_up.dA, 0, ah, stream) || cudaMemsetAsync(d_up.dB, 0, ai, stream) ||
        cudaMemsetAsync(d_down.dA, 0, ai, stream) || cudaMemsetAsync(d_down.dB, 0, ah, stream))
      return LORA_ERR_CUDA;
    return LORA_OK;
  }
  const int kfg = L.kfg, kfd = L.kfd;
  const uint8_t* sv = static_cast<const uint8_t*>(saved);
  const bf16* gsv = reinterpret_cast<const bf16*>(sv + L.off_g);
  const bf16* usv = reinterpret_cast<const bf16*>(sv + L.off_u);
  const bf16* hsv = reinterpret_cast<const bf16*>(sv + L.off_h);
  const bf16* tgu = reinterpret_cast<const bf16*>(sv + L.off_tgu);
  const bf16* td = reinterpret_cast<const bf16*>(sv + L.off_td);

  Carve c(ws);
  unsigned* status = static_cast<unsigned*>(c.take(kWsHeader));
  bf16* bt_d = c.take_n<bf16>(kfd * h);
  bf16* af_d = c.take_n<bf16>(kfd * i);
  bf16* bt_g = c.take_n<bf16>(kfg * i);
  bf16* bt_u = c.take_n<bf16>(kfg * i);
  bf16* af_gu = c.take_n<bf16>(kfg * h);
  bf16* ud = c.take_n<bf16>(M * kfd);
  bf16* dg = c.take_n<bf16>(M * i);
  bf16* du = c.take_n<bf16>(M * i);
  bf16* V = c.take_n<bf16>(M * kfg);
  float* part = c.take_n<float>(mlp_bwd_rank_part(M, h, i, kfd, kfg));
  Deferred dr;
  defer_init(dr, c.take_n<float>(mlp_bwd_slabs(M, h, i, kfd, kfg, n_ex)));

  PackParams pk;
  std::memset(static_cast<void*>(&pk), 0, sizeof(pk));
  pack_block(pack_job(pk, bt_d, kfd, h), down.B, r, 0, 0, r, static_cast<int>(h), 1, 1.0f);
  pack_block(pack_job(pk, af_d, kfd, i), down.A, i, 0, 0, r, static_cast<int>(i), 0, s);
  pack_block(pack_job(pk, bt_g, kfg, i), gate.B, r, 0, 0, r, static_cast<int>(i), 1, 1.0f);
  pack_block(pack_job(pk, bt_u, kfg, i), up.B, r, r, 0, r, static_cast<int>(i), 1, 1.0f);
  {
    PackJob& J = pack_job(pk, af_gu, kfg, h);
    pack_block(J, gate.A, h, 0, 0, r, static_cast<int>(h), 0, s);
    pack_block(J, up.A, h, r, 0, r, static_cast<int>(h), 0, s);
  }
  LGB_TRY(launch_pack(pk, stream));

  // U_d = dy B_d
  const ProjSeg p1 = {dy, bt_d, h};
  LGB_TRY(rank_projection(M, kfd, &p1, 1, ud, part, status, stream));

  // dh = [dy | U_d] [W_d ; s A_d];  dg = dh u act'(g), du = dh act(g)
  {
    GemmPlan g(kBigKMN);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(i), EPI_ACT_BWD, false);
    GemmPlan::seg(G, g.a_kmajor(dy, M, h, h), g.b_mnmajor(down.W, i, h, i), -1, h, h);
    GemmPlan::seg(G, g.a_kmajor(ud, M, kfd, kfd), g.b_mnmajor(af_d, i, kfd, i), -1, kfd, r);
    G.in0 = gsv;
    G.in1 = usv;
    G.ldi = i;
    G.out0 = dg;
    G.out1 = du;
    G.ldo = i;
    g.p.act = static_cast<int>(act);
    g.p.status = status;
    g.finish();
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKMN, g.p, LORA_KIND_ACT_BWD, stream));
  }

  // dB_d = s dy^T T_d and dA_d = s U_d^T h read nothing the dh GEMM writes: they start
  // on the SMs its last wave leaves idle
  const GradJob j1 = {dy, h, 0, d_down.dB, 0};
  LGB_TRY(token_grads(M, r, kfd, s, td, &j1, 1, dr, status, stream, n_ex, true));
  const GradJob j2 = {hsv, i, 0, d_down.dA, 1};
  LGB_TRY(token_grads(M, r, kfd, s, ud, &j2, 1, dr, status, stream, n_ex, true));

  // V = [dg B_g | du B_u]
  const ProjSeg p3[2] = {{dg, bt_g, i}, {du, bt_u, i}};
  LGB_TRY(rank_projection(M, kfg, p3, 2, V, part, status, stream));


  // dx = [dg | du | V] [W_g ; W_u ; s A_g ; s A_u]
  {
    GemmPlan g(kBigKMN);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(h), EPI_STORE, false);
    GemmPlan::seg(G, g.a_kmajor(dg, M, i, i), g.b_mnmajor(gate.W, h, i, h), -1, i, i);
    GemmPlan::seg(G, g.a_kmajor(du, M, i, i), g.b_mnmajor(up.W, h, i, h), -1, i, i);
    GemmPlan::seg(G, g.a_kmajor(V, M, kfg, kfg), g.b_mnmajor(af_gu, h, kfg, h), -1, kfg, 2 * r);
    G.out0 = dx;
    G.ldo = h;
    g.p.status = status;
    g.finish();
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKMN, g.p, LORA_KIND_DGRAD, stream));
  }

  // dB_g = s dg^T T_g, dB_u = s du^T T_u and dA_g = s V_g^T x, dA_u = s V_u^T x read
  // nothing the dx GEMM writes: they start on the SMs its last wave leaves idle
  const GradJob j3[2] = {{dg, i, 0, d_gate.dB, 0}, {du, i, r, d_up.dB, 0}};
  LGB_TRY(token_grads(M, r, kfg, s, tgu, j3, 2, dr, status, stream, n_ex, true));
  const GradJob j4[2] = {{x, h, 0, d_gate.dA, 1}, {x, h, r, d_up.dA, 1}};
  LGB_TRY(token_grads(M, r, kfg, s, V, j4, 2, dr, status, stream, n_ex, true));
  LGB_TRY(defer_flush(dr, stream));
  if (n_ex > 0 && sq_norms != nullptr) {
    NormParams np;
    std::memset(static_cast<void*>(&np), 0, sizeof(np));
    const lora_grads_t* gs[3] = {&d_gate, &d_up, &d_down};
    const int64_t fin[3] = {h, h, i}, fout[3] = {i, i, h};
    for (int a = 0; a < 3; ++a) {
      np.src[np.ntensors] = static_cast<const bf16*>(gs[a]->dA);
      np.count[np.ntensors++] = static_cast<long long>(r) * fin[a];
      np.src[np.ntensors] = static_cast<const bf16*>(gs[a]->dB);
      np.count[np.ntensors++] = static_cast<long long>(r) * fout[a];
    }
    np.out = sq_norms;
    LGB_TRY(launch_norms(np, static_cast<int>(n_ex), stream));
  }
  return LORA_OK;
}

extern "C" lora_status_t lora_mlp_backward(int64_t M, int64_t h, int64_t i, int r, float s, lora_act_t act,
                                           const void* x, lora_linear_t gate, lora_linear_t up,
                                           lora_linear_t down, const void* saved, const void* dy, void* dx,
                                           lora_grads_t d_gate, lora_grads_t d_up, lora_grads_t d_down, void* ws,
                                           size_t ws_bytes, cudaStream_t stream) {
  NvtxRange nvtx_range("lora_mlp_backward");
  return mlp_backward_impl(M, h, i, r, s, act, 0, x, gate, up, down, saved, dy, dx, d_gate, d_up, d_down,
                           nullptr, ws, ws_bytes, stream);
}

extern "C" size_t lora_mlp_per_example_workspace_bytes(int64_t M, int64_t h, int64_t i, int r, int64_t n_examples) {
  if (M < 0 || h <= 0 || i <= 0 || r < 1 || n_examples < 1 || M % n_examples != 0) return 0;
  return mlp_layout(M, h, i, r, n_examples).ws_bwd;
}

extern "C" lora_status_t lora_mlp_backward_per_example(int64_t M, int64_t h, int64_t i, int r, float s,
                                                       lora_act_t act, int64_t n_examples, const void* x,
                                                       lora_linear_t gate, lora_linear_t up, lora_linear_t down,
                                                       const void* saved, const void* dy, void* dx,
                                                       lora_grads_t d_gate, lora_grads_t d_up, lora_grads_t d_down,
                                                       float* sq_norms, void* ws, size_t ws_bytes,
                                                       cudaStream_t stream) {
  NvtxRange nvtx_range("lora_mlp_backward_per_example");
  if (n_examples < 1) return LORA_ERR_INVALID_ARG;
  return mlp_backward_impl(M, h, i, r, s, act, n_examples, x, gate, up, down, saved, dy, dx, d_gate, d_up, d_down,
                           sq_norms, ws, ws_bytes, stream);
}

// ================================================================ Q/K/V + O

namespace {

struct QkvoLayout {
  int kfq, kfo;
  size_t ws_fwd, ws_bwd, saved, off_to;
};

// Backward scratch, as for the MLP: rank-r projection slabs, then the token reductions'.
static int64_t qkvo_bwd_rank_part(int64_t M, int64_t h, int64_t nq, int64_t nkv, int kfq, int kfo) {
  return imax(rank_projection_part(M, kfo, ceil_div(h, kBK)),
              rank_projection_part(M, kfq, ceil_div(nq, kBK) + 2 * ceil_div(nkv, kBK)));
}
static int64_t qkvo_bwd_slabs(int64_t M, int64_t h, int64_t nq, int64_t nkv, int kfq, int kfo) {
  const int64_t f3[3] = {nq, nkv, nkv};
  return token_grad_part(M, kfo, &h, 1) + token_grad_part(M, kfo, &nq, 1) + token_grad_part(M, kfq, f3, 3) +
         token_grad_part(M, kfq, &h, 1);
}

QkvoLayout qkvo_layout(int64_t M, int64_t h, int64_t nq, int64_t nkv, int r) {
  QkvoLayout L;
  L.kfq = fold_width(3, r);
  L.kfo = fold_width(1, r);
  const int kfq = L.kfq, kfo = L.kfo;
  {
    Carve c(nullptr);
    c.take(kWsHeader);
    c.take_n<bf16>(kfq * h);
    c.take_n<bf16>(nq * kfq);
    c.take_n<bf16>(nkv * kfq);
    c.take_n<bf16>(nkv * kfq);
    c.take_n<bf16>(kfo * nq);
    c.take_n<bf16>(h * kfo);
    int64_t p = rank_projection_part(M, kfq, ceil_div(h, kBK));
    const int64_t p2 = rank_projection_part(M, kfo, ceil_div(nq, kBK));
    c.take_n<float>(p > p2 ? p : p2);
    c.take_n<bf16>(M * kfq);
    c.take_n<bf16>(M * kfo);
    L.ws_fwd = c.off;
  }
  {
    Carve c(nullptr);
    c.take(kWsHeader);
    c.take_n<bf16>(kfq * nq);
    c.take_n<bf16>(kfq * nkv);
    c.take_n<bf16>(kfq * nkv);
    c.take_n<bf16>(kfq * h);
    c.take_n<bf16>(kfo * h);
    c.take_n<bf16>(kfo * nq);
    c.take_n<bf16>(M * kfo);
    c.take_n<bf16>(M * kfq);
    c.take_n<bf16>(M * nq);     // dy_q, dy_k turned back by the transpose RoPE rotation
    c.take_n<bf16>(M * nkv);
    c.take_n<float>(qkvo_bwd_rank_part(M, h, nq, nkv, kfq, kfo));
    c.take_n<float>(qkvo_bwd_slabs(M, h, nq, nkv, kfq, kfo));
    L.ws_bwd = c.off;
  }
  {
    Carve c(nullptr);
    c.offset_of(sizeof(bf16) * M * kfq);
    L.off_to = c.offset_of(sizeof(bf16) * M * kfo);
    L.saved = c.off;
  }
  return L;
}

// RoPE arguments: NULL is "no RoPE"; otherwise the rules of lora_rope_t.
lora_status_t check_rope(const lora_rope_t* rope, int64_t nq, int64_t nkv) {
  if (rope == nullptr) return LORA_OK;
  if (!rope->cos || !rope->sin || !rope->pos || rope->n_pos < 1 || rope->n_pos > 0x7fffffff)
    return LORA_ERR_INVALID_ARG;
  const int d = rope->head_dim;
  if (d != 64 && d != 128 && d != 256) return LORA_ERR_UNSUPPORTED;
  if (nq % d || nkv % d) return LORA_ERR_INVALID_ARG;
  if (!aligned(rope->cos, 16) || !aligned(rope->sin, 16) || !aligned(rope->pos, 4)) return LORA_ERR_ALIGNMENT;
  return LORA_OK;
}

lora_status_t check_qkvo(int64_t M, int64_t h, int64_t nq, int64_t nkv, int r, float s) {
  lora_status_t st = check_common(M, r, s);
  check_size(h, st);
  check_size(nq, st);
  check_size(nkv, st);
  if (st != LORA_OK) return st;
  if (3 * r > 256) return LORA_ERR_UNSUPPORTED;
  if (h % 8 || nq % 8 || nkv % 8) return LORA_ERR_ALIGNMENT;
  return LORA_OK;
}

}  // namespace

extern "C" size_t lora_qkvo_saved_bytes(int64_t M, int64_t h, int64_t n_q, int64_t n_kv, int r) {
  if (M < 0 || h <= 0 || n_q <= 0 || n_kv <= 0 || r < 1) return 0;
  return qkvo_layout(M, h, n_q, n_kv, r).saved;
}
extern "C" size_t lora_qkvo_workspace_bytes(int64_t M, int64_t h, int64_t n_q, int64_t n_kv, int r) {
  if (M < 0 || h <= 0 || n_q <= 0 || n_kv <= 0 || r < 1) return 0;
  const QkvoLayout L = qkvo_layout(M, h, n_q, n_kv, r);
  return L.ws_fwd > L.ws_bwd ? L.ws_fwd : L.ws_bwd;
}

extern "C" lora_status_t lora_qkvo_forward(int64_t M, int64_t h, int64_t n_q, int64_t n_kv, int r, float s,
                                           const void* x, lora_linear_t q, lora_linear_t k, lora_linear_t v,
                                           void* yq, void* yk, void* yv, const void* o_in, lora_linear_t o,
                                           void* yo, const void* bias_qkv, const lora_rope_t* rope,
                                           void* saved, void* ws, size_t ws_bytes, cudaStream_t stream) {
  NvtxRange nvtx_range("lora_qkvo_forward");
  LGB_TRY(check_qkvo(M, h, n_q, n_kv, r, s));
  if (!ws || (!x && !o_in)) return LORA_ERR_INVALID_ARG;
  if (x) LGB_TRY(check_rope(rope, n_q, n_kv));
  if (bias_qkv != nullptr && !aligned(bias_qkv, 16)) return LORA_ERR_ALIGNMENT;
  if (x && ((M > 0 && (!yq || !yk || !yv)) || !lin_ok(q) || !lin_ok(k) || !lin_ok(v))) return LORA_ERR_INVALID_ARG;
  if (o_in && ((M > 0 && !yo) || !lin_ok(o))) return LORA_ERR_INVALID_ARG;
  if (!aligned(ws, 256) || (saved && !aligned(saved, 256))) return LORA_ERR_ALIGNMENT;
  if (x && (!aligned(x, 16) || !aligned(yq, 16) || !aligned(yk, 16) || !aligned(yv, 16) || !lin_aligned(q) ||
            !lin_aligned(k) || !lin_aligned(v)))
    return LORA_ERR_ALIGNMENT;
  if (o_in && (!aligned(o_in, 16) || !aligned(yo, 16) || !lin_aligned(o))) return LORA_ERR_ALIGNMENT;
  const QkvoLayout L = qkvo_layout(M, h, n_q, n_kv, r);
  if (ws_bytes < L.ws_fwd) return LORA_ERR_WORKSPACE;
  if (M == 0) return LORA_OK;
  const int kfq = L.kfq, kfo = L.kfo;
  Carve c(ws);
  unsigned* status = static_cast<unsigned*>(c.take(kWsHeader));
  bf16* acat = c.take_n<bf16>(kfq * h);
  bf16* bfq = c.take_n<bf16>(n_q * kfq);
  bf16* bfk = c.take_n<bf16>(n_kv * kfq);
  bf16* bfv = c.take_n<bf16>(n_kv * kfq);
  bf16* acat_o = c.take_n<bf16>(kfo * n_q);
  bf16* bf_o = c.take_n<bf16>(h * kfo);
  int64_t pe = rank_projection_part(M, kfq, ceil_div(h, kBK));
  const int64_t pe2 = rank_projection_part(M, kfo, ceil_div(n_q, kBK));
  float* part = c.take_n<float>(pe > pe2 ? pe : pe2);
  bf16* tqkv = c.take_n<bf16>(M * kfq);
  bf16* to = c.take_n<bf16>(M * kfo);
  if (saved) {
    tqkv = static_cast<bf16*>(saved);
    to = reinterpret_cast<bf16*>(static_cast<uint8_t*>(saved) + L.off_to);
  }

  PackParams pk;
  std::memset(static_cast<void*>(&pk), 0, sizeof(pk));
  if (x) {
    PackJob& J = pack_job(pk, acat, kfq, h);
    pack_block(J, q.A, h, 0, 0, r, static_cast<int>(h), 0, 1.0f);
    pack_block(J, k.A, h, r, 0, r, static_cast<int>(h), 0, 1.0f);
    pack_block(J, v.A, h, 2 * r, 0, r, static_cast<int>(h), 0, 1.0f);
    pack_block(pack_job(pk, bfq, n_q, kfq), q.B, r, 0, 0, static_cast<int>(n_q), r, 0, s);
    pack_block(pack_job(pk, bfk, n_kv, kfq), k.B, r, 0, r, static_cast<int>(n_kv), r, 0, s);
    pack_block(pack_job(pk, bfv, n_kv, kfq), v.B, r, 0, 2 * r, static_cast<int>(n_kv), r, 0, s);
  }
  if (o_in) {
    pack_block(pack_job(pk, acat_o, kfo, n_q), o.A, n_q, 0, 0, r, static_cast<int>(n_q), 0, 1.0f);
    pack_block(pack_job(pk, bf_o, h, kfo), o.B, r, 0, 0, static_cast<int>(h), r, 0, s);
  }
  LGB_TRY(launch_pack(pk, stream));

  if (x) {
    const ProjSeg p1 = {x, acat, h};
    LGB_TRY(rank_projection(M, kfq, &p1, 1, tqkv, part, status, stream));
    GemmPlan g(kBigKK);
    const int ax = g.a_kmajor(x, M, h, h);
    const int at = g.a_kmajor(tqkv, M, kfq, kfq);
    const lora_linear_t* lins[3] = {&q, &k, &v};
    bf16* bfs[3] = {bfq, bfk, bfv};
    void* ys[3] = {yq, yk, yv};
    const int64_t ns[3] = {n_q, n_kv, n_kv};
    if (rope != nullptr) {
      g.p.rope_cos = rope->cos;
      g.p.rope_sin = rope->sin;
      g.p.rope_pos = rope->pos;
      g.p.rope_half = rope->head_dim / 2;
      g.p.rope_npos = static_cast<int>(rope->n_pos);
    }
    for (int p = 0; p < 3; ++p) {
      const int epi = (rope != nullptr && p < 2) ? EPI_ROPE : EPI_STORE;
      GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(ns[p]), epi, false);
      GemmPlan::seg(G, ax, g.b_kmajor(lins[p]->W, ns[p], h, h, g.b_rows_full()), -1, h, h);
      GemmPlan::seg(G, at, g.b_kmajor(bfs[p], ns[p], kfq, kfq, g.b_rows_full()), -1, kfq, (p + 1) * r);
      G.out0 = ys[p];
      G.ldo = ns[p];
      if (bias_qkv != nullptr) G.in0 = static_cast<const bf16*>(bias_qkv) + (p == 0 ? 0 : n_q + (p - 1) * n_kv);
    }
    g.p.status = status;
    g.finish();
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKK, g.p, LORA_KIND_PROJ, stream));
  }
  if (o_in) {
    const ProjSeg p2 = {o_in, acat_o, n_q};
    LGB_TRY(rank_projection(M, kfo, &p2, 1, to, part, status, stream));
    GemmPlan g(kBigKK);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(h), EPI_STORE, false);
    GemmPlan::seg(G, g.a_kmajor(o_in, M, n_q, n_q), g.b_kmajor(o.W, h, n_q, n_q, g.b_rows_full()), -1, n_q, n_q);
    GemmPlan::seg(G, g.a_kmajor(to, M, kfo, kfo), g.b_kmajor(bf_o, h, kfo, kfo, g.b_rows_full()), -1, kfo, r);
    G.out0 = yo;
    G.ldo = h;
    g.p.status = status;
    g.finish();
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKK, g.p, LORA_KIND_PROJ, stream));
  }
  return LORA_OK;
}

extern "C" lora_status_t lora_qkvo_backward(int64_t M, int64_t h, int64_t n_q, int64_t n_kv, int r, float s,
                                            const void* x, lora_linear_t q, lora_linear_t k, lora_linear_t v,
                                            const void* o_in, lora_linear_t o, const void* saved,
                                            const lora_rope_t* rope, const void* dyq, const void* dyk,
                                            const void* dyv, void* dx,
                                            const void* dyo, void* do_in, lora_grads_t d_q, lora_grads_t d_k,
                                            lora_grads_t d_v, lora_grads_t d_o, void* ws, size_t ws_bytes,
                                            cudaStream_t stream) {
  NvtxRange nvtx_range("lora_qkvo_backward");
  LGB_TRY(check_qkvo(M, h, n_q, n_kv, r, s));
  if (!ws || !saved || (!x && !o_in)) return LORA_ERR_INVALID_ARG;
  if (x) LGB_TRY(check_rope(rope, n_q, n_kv));
  if (x && ((M > 0 && (!dyq || !dyk || !dyv || !dx)) || !lin_ok(q) || !lin_ok(k) || !lin_ok(v) || !d_q.dA || !d_q.dB ||
            !d_k.dA || !d_k.dB || !d_v.dA || !d_v.dB))
    return LORA_ERR_INVALID_ARG;
  if (o_in && ((M > 0 && (!dyo || !do_in)) || !lin_ok(o) || !d_o.dA || !d_o.dB)) return LORA_ERR_INVALID_ARG;
  if (!aligned(ws, 256) || !aligned(saved, 256)) return LORA_ERR_ALIGNMENT;
  if (x && (!aligned(x, 16) || !aligned(dyq, 16) || !aligned(dyk, 16) || !aligned(dyv, 16) || !aligned(dx, 16) ||
            !lin_aligned(q) || !lin_aligned(k) || !lin_aligned(v) || !aligned(d_q.dA, 2) || !aligned(d_q.dB, 2) ||
            !aligned(d_k.dA, 2) || !aligned(d_k.dB, 2) || !aligned(d_v.dA, 2) || !aligned(d_v.dB, 2)))
    return LORA_ERR_ALIGNMENT;
  if (o_in && (!aligned(o_in, 16) || !aligned(dyo, 16) || !aligned(do_in, 16) || !lin_aligned(o) ||
               !aligned(d_o.dA, 2) || !aligned(d_o.dB, 2)))
    return LORA_ERR_ALIGNMENT;
  const QkvoLayout L = qkvo_layout(M, h, n_q, n_kv, r);
  if (ws_bytes < L.ws_bwd) return LORA_ERR_WORKSPACE;
  if (M == 0) {
    if (x) {
      const size_t ah = sizeof(bf16) * r * h;
      if (cudaMemsetAsync(d_q.dA, 0, ah, stream) || cudaMemsetAsync(d_k.dA, 0, ah, stream) ||
          cudaMemsetAsync(d_v.dA, 0, ah, stream) || cudaMemsetAsync(d_q.dB, 0, sizeof(bf16) * r * n_q, stream) ||
          cudaMemsetAsync(d_k.dB, 0, sizeof(bf16) * r * n_kv, stream) ||
          cudaMemsetAsync(d_v.dB, 0, sizeof(bf16) * r * n_kv, stream))
        return LORA_ERR_CUDA;
    }
    if (o_in) {
      if (cudaMemsetAsync(d_o.dA, 0, sizeof(bf16) * r * n_q, stream) ||
          cudaMemsetAsync(d_o.dB, 0, sizeof(bf16) * r * h, stream))
        return LORA_ERR_CUDA;
    }
    return LORA_OK;
  }
  const int kfq = L.kfq, kfo = L.kfo;
  const bf16* tqkv = static_cast<const bf16*>(saved);
  const bf16* to = reinterpret_cast<const bf16*>(static_cast<const uint8_t*>(saved) + L.off_to);
  Carve c(ws);
  unsigned* status = static_cast<unsigned*>(c.take(kWsHeader));
  bf16* btq = c.take_n<bf16>(kfq * n_q);
  bf16* btk = c.take_n<bf16>(kfq * n_kv);
  bf16* btv = c.take_n<bf16>(kfq * n_kv);
  bf16* af_qkv = c.take_n<bf16>(kfq * h);
  bf16* bt_o = c.take_n<bf16>(kfo * h);
  bf16* af_o = c.take_n<bf16>(kfo * n_q);
  bf16* uo = c.take_n<bf16>(M * kfo);
  bf16* V = c.take_n<bf16>(M * kfq);
  bf16* dyq_r = c.take_n<bf16>(M * n_q);
  bf16* dyk_r = c.take_n<bf16>(M * n_kv);
  float* part = c.take_n<float>(qkvo_bwd_rank_part(M, h, n_q, n_kv, kfq, kfo));
  Deferred dr;
  defer_init(dr, c.take_n<float>(qkvo_bwd_slabs(M, h, n_q, n_kv, kfq, kfo)));

  PackParams pk;
  std::memset(static_cast<void*>(&pk), 0, sizeof(pk));
  if (x) {
    pack_block(pack_job(pk, btq, kfq, n_q), q.B, r, 0, 0, r, static_cast<int>(n_q), 1, 1.0f);
    pack_block(pack_job(pk, btk, kfq, n_kv), k.B, r, r, 0, r, static_cast<int>(n_kv), 1, 1.0f);
    pack_block(pack_job(pk, btv, kfq, n_kv), v.B, r, 2 * r, 0, r, static_cast<int>(n_kv), 1, 1.0f);
    PackJob& J = pack_job(pk, af_qkv, kfq, h);
    pack_block(J, q.A, h, 0, 0, r, static_cast<int>(h), 0, s);
    pack_block(J, k.A, h, r, 0, r, static_cast<int>(h), 0, s);
    pack_block(J, v.A, h, 2 * r, 0, r, static_cast<int>(h), 0, s);
  }
  if (o_in) {
    pack_block(pack_job(pk, bt_o, kfo, h), o.B, r, 0, 0, r, static_cast<int>(h), 1, 1.0f);
    pack_block(pack_job(pk, af_o, kfo, n_q), o.A, n_q, 0, 0, r, static_cast<int>(n_q), 0, s);
  }
  LGB_TRY(launch_pack(pk, stream));

  if (o_in) {
    const ProjSeg p1 = {dyo, bt_o, h};
    LGB_TRY(rank_projection(M, kfo, &p1, 1, uo, part, status, stream));
    GemmPlan g(kBigKMN);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(n_q), EPI_STORE, false);
    GemmPlan::seg(G, g.a_kmajor(dyo, M, h, h), g.b_mnmajor(o.W, n_q, h, n_q), -1, h, h);
    GemmPlan::seg(G, g.a_kmajor(uo, M, kfo, kfo), g.b_mnmajor(af_o, n_q, kfo, n_q), -1, kfo, r);
    G.out0 = do_in;
    G.ldo = n_q;
    g.p.status = status;
    g.finish();
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKMN, g.p, LORA_KIND_DGRAD, stream));
    // dB_o = s dy_o^T T_o and dA_o = s U_o^T o_in read nothing the d o_in GEMM writes
    const GradJob j1 = {dyo, h, 0, d_o.dB, 0};
    LGB_TRY(token_grads(M, r, kfo, s, to, &j1, 1, dr, status, stream, 0, true));
    const GradJob j2 = {o_in, n_q, 0, d_o.dA, 1};
    LGB_TRY(token_grads(M, r, kfo, s, uo, &j2, 1, dr, status, stream, 0, true));
  }
  if (x) {
    if (rope != nullptr) {
      // gradients of the rotated q, k -> gradients of the projections' outputs
      RopeParams rp;
      std::memset(static_cast<void*>(&rp), 0, sizeof(rp));
      rp.src[0] = static_cast<const bf16*>(dyq);
      rp.src[1] = static_cast<const bf16*>(dyk);
      rp.dst[0] = dyq_r;
      rp.dst[1] = dyk_r;
      rp.n[0] = n_q;
      rp.n[1] = n_kv;
      rp.ntensors = 2;
      rp.M = M;
      rp.cos = rope->cos;
      rp.sin = rope->sin;
      rp.pos = rope->pos;
      rp.half = rope->head_dim / 2;
      rp.npos = static_cast<int>(rope->n_pos);
      rp.sign = -1.0f;
      rp.status = status;
      LGB_TRY(launch_rope(rp, stream));
      dyq = dyq_r;
      dyk = dyk_r;
    }
    const ProjSeg p3[3] = {{dyq, btq, n_q}, {dyk, btk, n_kv}, {dyv, btv, n_kv}};
    LGB_TRY(rank_projection(M, kfq, p3, 3, V, part, status, stream));
    GemmPlan g(kBigKMN);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(h), EPI_STORE, false);
    GemmPlan::seg(G, g.a_kmajor(dyq, M, n_q, n_q), g.b_mnmajor(q.W, h, n_q, h), -1, n_q, n_q);
    GemmPlan::seg(G, g.a_kmajor(dyk, M, n_kv, n_kv), g.b_mnmajor(k.W, h, n_kv, h), -1, n_kv, n_kv);
    GemmPlan::seg(G, g.a_kmajor(dyv, M, n_kv, n_kv), g.b_mnmajor(v.W, h, n_kv, h), -1, n_kv, n_kv);
    GemmPlan::seg(G, g.a_kmajor(V, M, kfq, kfq), g.b_mnmajor(af_qkv, h, kfq, h), -1, kfq, 3 * r);
    G.out0 = dx;
    G.ldo = h;
    g.p.status = status;
    g.finish();
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKMN, g.p, LORA_KIND_DGRAD, stream));
    const GradJob j4[3] = {{x, h, 0, d_q.dA, 1}, {x, h, r, d_k.dA, 1}, {x, h, 2 * r, d_v.dA, 1}};
    // the q, k, v dB and dA read nothing the dx GEMM writes
    const GradJob j3[3] = {{dyq, n_q, 0, d_q.dB, 0}, {dyk, n_kv, r, d_k.dB, 0}, {dyv, n_kv, 2 * r, d_v.dB, 0}};
    LGB_TRY(token_grads(M, r, kfq, s, tqkv, j3, 3, dr, status, stream, 0, true));
    LGB_TRY(token_grads(M, r, kfq, s, V, j4, 3, dr, status, stream, 0, true));
  }
  return defer_flush(dr, stream);
}

// ================================================================ status and trace

extern "C" lora_status_t lora_poll_status(void* ws, cudaStream_t stream) {
  if (ws == nullptr || !aligned(ws, 256)) return LORA_ERR_INVALID_ARG;
  unsigned host = 0;
  if (cudaMemcpyAsync(&host, ws, sizeof(unsigned), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return LORA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return LORA_ERR_CUDA;
  if (host != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(unsigned), stream) != cudaSuccess) return LORA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return LORA_ERR_CUDA;
  }
  if (host & kStatusTimeout) return LORA_ERR_TIMEOUT;
  return (host & kStatusInput) ? LORA_ERR_DEVICE_INPUT : LORA_OK;
}

extern "C" lora_status_t lora_rope_table(float* cos, float* sin, int64_t n_pos, int head_dim, double base,
                                         cudaStream_t stream) {
  NvtxRange nvtx_range("lora_rope_table");
  if (!cos || !sin || n_pos < 1 || head_dim < 2 || head_dim % 2 || !(base > 0.0) || !std::isfinite(base))
    return LORA_ERR_INVALID_ARG;
  if (!aligned(cos, 16) || !aligned(sin, 16)) return LORA_ERR_ALIGNMENT;
  RopeTableParams p;
  p.cos = cos;
  p.sin = sin;
  p.npos = n_pos;
  p.half = head_dim / 2;
  p.base = base;
  long long gx = ceil_div(n_pos * p.half, 256);
  gx = gx > 4 * num_sms() ? 4 * num_sms() : gx;
  const int slot = trace_begin(LORA_KIND_ROPE, stream);
  cudaError_t e = launch_pdl(rope_table_kernel, dim3(static_cast<unsigned>(gx)), dim3(256), 0, stream, p);
  trace_end(slot, stream);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return LORA_OK;
}

extern "C" const char* lora_status_string(lora_status_t status) {
  switch (status) {
    case LORA_OK: return "ok";
    case LORA_ERR_INVALID_ARG: return "invalid argument";
    case LORA_ERR_ALIGNMENT: return "alignment: pointers 16-byte (ws/saved 256-byte), feature sizes multiples of 8";
    case LORA_ERR_UNSUPPORTED: return "unsupported: rank too large for the fold";
    case LORA_ERR_WORKSPACE: return "workspace smaller than the size query";
    case LORA_ERR_CUDA: return "CUDA runtime or launch failure";
    case LORA_ERR_TIMEOUT: return "a kernel's bounded wait expired";
    case LORA_ERR_DEVICE_INPUT: return "a device-side input was out of range (RoPE position)";
  }
  return "unknown status";
}

extern "C" lora_status_t lora_set_wait_timeout(uint64_t ns) {
  if (ns == 0) ns = kTimeoutNs;
  if (ns < 1000000ull || ns > 60000000000ull) return LORA_ERR_INVALID_ARG;
  g_timeout_ns.store(ns);
  return LORA_OK;
}

extern "C" uint64_t lora_wait_timeout(void) { return g_timeout_ns.load(); }

extern "C" lora_status_t lora_test_expire_waits(int launches) {
  if (launches < 0 || launches > 64) return LORA_ERR_INVALID_ARG;
  g_expire_next.store(launches);
  return LORA_OK;
}

extern "C" uint64_t lora_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" void lora_trace_kinds(unsigned mask) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  g_trace.kinds = mask;
}

extern "C" lora_status_t lora_trace_enable(int capacity) {
  if (capacity < 0) return LORA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_trace.mu);
  for (cudaEvent_t e : g_trace.ev) cudaEventDestroy(e);
  g_trace.ev.clear();
  g_trace.kind.clear();
  g_trace.used = 0;
  g_trace.capacity = 0;
  if (capacity == 0) return LORA_OK;
  g_trace.ev.resize(2 * static_cast<size_t>(capacity));
  g_trace.kind.resize(static_cast<size_t>(capacity));
  for (auto& e : g_trace.ev)
    if (cudaEventCreate(&e) != cudaSuccess) return LORA_ERR_CUDA;
  g_trace.capacity = capacity;
  return LORA_OK;
}

extern "C" int lora_trace_read(int* kind, float* ms, int max) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  int n = g_trace.used < max ? g_trace.used : max;
  for (int j = 0; j < n; ++j) {
    if (cudaEventSynchronize(g_trace.ev[2 * j + 1]) != cudaSuccess) return -1;
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, g_trace.ev[2 * j], g_trace.ev[2 * j + 1]) != cudaSuccess) return -1;
    kind[j] = g_trace.kind[j];
    ms[j] = t;
  }
  g_trace.used = 0;
  return n;
}
