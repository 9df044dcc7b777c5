// The library's shared host side: device plumbing (tensor maps, launch wrappers, the
// launch counter and event trace, bounded-wait settings), the building blocks the
// operations share (adapter packing, rank-r projections, reductions over tokens), and
// the status, trace and RoPE-table entry points.  The operations' entry points are in
// lora_linear.cu, lora_mlp.cu and lora_qkvo.cu; include/lora_gb300.h is the contract.
#include <unistd.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <mutex>
#include <vector>

#include "api_internal.cuh"
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

// The driver's map encoder needs a current context on the calling thread, which a
// thread that has made no runtime call yet lacks (e.g. the thread autograd runs a
// backward on): the current device's primary context is made current, once per thread
// and device.
static void bind_current_device() {
  thread_local int bound = -1;
  int dev = -1;
  if (cudaGetDevice(&dev) == cudaSuccess && dev != bound && cudaSetDevice(dev) == cudaSuccess) bound = dev;
}

// 2-D bf16 map with a 128-byte, 64-byte, 32-byte or no swizzle (swizzle_bytes 128, 64, 32, 0);
// out-of-bounds elements read as zero.
bool encode_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                uint32_t box_inner, uint32_t box_outer, int swizzle_bytes) {
  bind_current_device();
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || inner == 0 || outer == 0) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
            : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
            : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                  : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map {inner, d1, d2} with row stride ld (elements) and plane stride
// ld * d1; box {box_inner, box_d1, 1}.
bool encode_map_planes(CUtensorMap* m, const void* base, uint64_t inner, uint64_t d1, uint64_t d2, uint64_t ld,
                       uint32_t box_inner, uint32_t box_d1) {
  bind_current_device();
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

// Split-tail mode (lora_set_split_tail): 0 automatic, 1 never, S = 2..kSkMaxSplits
// every tail in S pieces whenever the launch allows it.  The environment variable
// LORA_SPLIT_TAIL sets the initial mode.
static std::atomic<int> g_split_tail{[] {
  const char* e = std::getenv("LORA_SPLIT_TAIL");
  return (e != nullptr && e[0] >= '1' && e[0] <= '0' + kSkMaxSplits && e[1] == 0) ? e[0] - '0' : 0;
}()};

// Launch tags of the split tail's arrival words: distinct for every launch of the
// process, and started from a per-process value so that words left by another process
// in reused memory do not match (56 bits; the low 8 bits of a word count arrivals).
static unsigned long long next_sk_epoch() {
  static std::atomic<unsigned long long> counter{[] {
    unsigned long long z = static_cast<unsigned long long>(
                               std::chrono::steady_clock::now().time_since_epoch().count()) ^
                           (static_cast<unsigned long long>(getpid()) << 32);
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;      // splitmix64 finaliser
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
  }()};
  return counter.fetch_add(1) & ((1ull << 56) - 1);
}

// Chooses the pair launch's schedule and returns the pairs its grid needs.  With T
// tiles on P pairs, round-robin whole tiles take ceil(T / P) tile-times.  The tail
// (T mod P tiles after the full waves, or all T when T < P) may instead be cut into S
// k-ranges: the tail then takes ceil(tail * S / P) / S tile-times, plus the partial
// sums' cost for the piece that finishes a tile, measured at about the time of
// 8 + 24 (S - 1) k-blocks of MMAs (its own partial sums stored, each other piece's read
// back eight columns at a time).  In automatic mode the S in 2..kSkMaxSplits with the
// smallest estimate is used when it saves at least kSkMinGain of the launch; a mode
// S >= 2 uses S pieces whatever the estimate.
static int plan_pairs(TcParams& p, int pairs) {
  const int T = p.total_units;
  p.sk_dp_units = T;
  p.sk_splits = 0;
  const int round_robin = T < pairs ? T : pairs;
  const int mode = g_split_tail.load(std::memory_order_relaxed);
  if (p.sk_part == nullptr || p.sk_flags == nullptr || mode == 1) return round_robin;
  const int kb = p.grp[0].kb_total;
  for (int g = 0; g < p.ngroups; ++g)
    if (p.grp[g].splits != 1 || p.grp[g].per_plane || p.grp[g].kb_total != kb) return round_robin;
  if (kb < kSkMinKb) return round_robin;
  const int W = T / pairs;
  const int tail = W >= 1 ? T - W * pairs : T;
  if (tail == 0 || tail > p.sk_cap_tiles) return round_robin;
  int best_s = 0;
  double best = 1e30;
  for (int S = 2; S <= kSkMaxSplits; ++S) {
    if (tail * S > p.sk_cap_pieces || kb < 2 * S) break;
    const double est = static_cast<double>((tail * S + pairs - 1) / pairs) / S + (8.0 + 24.0 * (S - 1)) / kb;
    if ((mode == 0 && est < best - 1e-12) || mode == S) {
      best = est;
      best_s = S;
    }
  }
  if (best_s == 0 || (mode == 0 && (1.0 - best) / (W + 1) < kSkMinGain)) return round_robin;
  p.sk_dp_units = T - tail;
  p.sk_tail = tail;
  p.sk_splits = best_s;
  p.sk_kb = kb;
  p.sk_epoch = next_sk_epoch();
  const int units = T - tail + tail * best_s;
  return units < pairs ? units : pairs;
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
    grid = 2 * plan_pairs(p, num_sms() / 2);
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
    if (static_cast<int64_t>(p.job[j].rows) * p.job[j].cols >= (int64_t(1) << 31)) return LORA_ERR_UNSUPPORTED;
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

constexpr int kVec4MaxSplits = 8;
lora_status_t launch_reduce(const RedParams& plan, cudaStream_t st) {
  if (plan.nout == 0) return LORA_OK;
  RedParams p = plan;
  int64_t most = 1;
  for (int j = 0; j < p.nout; ++j) {
    RedOut& o = p.out[j];
    const int64_t elems = static_cast<int64_t>(o.rows) * o.ncols;
    // four columns a thread, unless the sums are long (more than kVec4MaxSplits slabs):
    // then a thread per column, four times the threads to hide the loads' latency
    o.vec4 = !o.per_split && o.ncols % 4 == 0 && o.col0 % 4 == 0 && o.width % 4 == 0 && elems < (int64_t(1) << 31) &&
             (o.trans || (o.ld % 4 == 0 && aligned(o.dst, 8))) && o.splits <= kVec4MaxSplits;
    const int64_t n = o.vec4 ? elems / 4 : elems;
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


void pack_block(PackJob& J, const void* src, int64_t lds, int ro, int co, int R, int C, int trans,
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
PackJob& pack_job(PackParams& P, void* dst, int64_t rows, int64_t cols) {
  PackJob& J = P.job[P.njob++];
  J.dst = static_cast<bf16*>(dst);
  J.rows = static_cast<int>(rows);
  J.cols = static_cast<int>(cols);
  J.nblk = 0;
  return J;
}

lora_status_t rank_projection(int64_t M, int kf, const ProjSeg* segs, int nseg, void* dst, float* part,
                                     unsigned* status, cudaStream_t st, void* dst_t, int64_t ldt, int ntrans) {
  const int variant = skinny_kk(kf);
  GemmPlan g(variant);
  int64_t kb = 0;
  for (int s = 0; s < nseg; ++s) kb += ceil_div(segs[s].K, kBK);
  const int64_t tiles = ceil_div(M, kBM) * ceil_div(kf, g.bn);
  const int splits = choose_proj_splits(tiles, kb, num_sms());
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
    G.out1 = dst_t;
    G.ldt = ldt;
    G.ntc = ntrans;
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
    if (dst_t != nullptr) {       // the same sums, transposed
      r.out[1] = o;
      r.out[1].dst = static_cast<bf16*>(dst_t);
      r.out[1].ld = ldt;
      r.out[1].ncols = ntrans;
      r.out[1].trans = 1;
      r.nout = 2;
    }
    LGB_TRY(launch_reduce(r, st));
  }
  return LORA_OK;
}
int64_t rank_projection_part(int64_t M, int kf, int64_t ktotal_blocks) {
  const int splits = max_splits(ktotal_blocks);
  return splits > 1 ? partial_elems(M, kf, skinny_bn(kf), splits) : 0;
}

// f32 slab elements of the token reductions of n products (fs[j] features each).
// n_ex > 0: per-example mode, one slab per example.
int64_t token_grad_part(int64_t M, int kf, const int64_t* fs, int n, int64_t n_ex) {
  const int bn = skinny_bn(kf);
  const int splits = n_ex > 0 ? static_cast<int>(n_ex) : max_splits(ceil_div(M, kBK));
  int64_t tot = 0;
  for (int j = 0; j < n; ++j) tot += round_up(partial_elems(fs[j], kf, bn, splits), 64);
  return tot;
}
void defer_init(Deferred& d, float* slabs) {
  std::memset(static_cast<void*>(&d.rp), 0, sizeof(d.rp));
  d.cursor = slabs;
}
lora_status_t defer_flush(Deferred& d, cudaStream_t st) {
  const lora_status_t r = launch_reduce(d.rp, st);
  d.rp.nout = 0;
  return r;
}

// Jobs with the same Q and T share one group (and one slab: several rank slots out of
// one product).  n_ex == 0: the sums over all M tokens.  n_ex > 0: one result per
// example (example e = tokens [e seq, (e+1) seq), seq = M / n_ex), each written at
// dst + e * r * f; the products read 3-D views {features, seq, examples} so no k-block
// straddles two examples (rows past seq read as zero).  The slabs start at
// defer.cursor and the sums are left to defer_flush.
// late: the launch follows a kernel whose outputs it does not read (and whose inputs
// it does not write), so it may start on SMs that kernel has freed (pdl_late).
lora_status_t token_grads(int64_t M, int r, int kf, float s, const GradJob* jobs, int njobs, Deferred& defer,
                          unsigned* status, cudaStream_t st, int64_t n_ex, bool late) {
  const int variant = skinny_mnmn(kf);
  GemmPlan g(variant);
  g.p.pdl_late = late ? 1 : 0;
  const int64_t seq = n_ex > 0 ? M / n_ex : M;
  const void* qs[kMaxGroups];
  const void* ts[kMaxGroups];
  const void* tmap_src[kMaxGroups];
  int tmap_of[kMaxGroups];
  int nq = 0, nt = 0, group_of[kMaxGroups * 3];
  float* parts[kMaxGroups];
  float* cur = defer.cursor;
  const int slab_splits = n_ex > 0 ? static_cast<int>(n_ex) : max_splits(ceil_div(M, kBK));
  int kfs[kMaxGroups];
  for (int j = 0; j < njobs; ++j) {
    const int kfj = jobs[j].kf > 0 ? jobs[j].kf : kf;
    // not reached: the call's kf is the widest, and the workspace sizes every job's slabs
    // for the tile width of its own kf
    if (kfj > kf || skinny_bn(kfj) != skinny_bn(kf)) return LORA_ERR_UNSUPPORTED;
    int gi = -1;
    for (int q = 0; q < nq; ++q)
      if (qs[q] == jobs[j].Q && ts[q] == jobs[j].T) gi = q;
    if (gi < 0) {
      if (nq >= kMaxGroups) return LORA_ERR_UNSUPPORTED;   // not reached: <= 4 per call site
      // the rank-r operand's map, shared by the groups that read the same T
      int tm = -1;
      for (int k = 0; k < nt; ++k)
        if (tmap_src[k] == jobs[j].T) tm = tmap_of[k];
      if (tm < 0) {
        tm = n_ex > 0 ? g.b_mnmajor_planes(jobs[j].T, kfj, seq, n_ex, kfj) : g.b_mnmajor(jobs[j].T, kfj, M, kfj);
        tmap_src[nt] = jobs[j].T;
        tmap_of[nt++] = tm;
      }
      gi = nq++;
      qs[gi] = jobs[j].Q;
      ts[gi] = jobs[j].T;
      const int64_t tiles = ceil_div(jobs[j].f, kBM) * ceil_div(kfj, g.bn);
      GroupDesc& G = g.group(static_cast<int>(jobs[j].f), kfj, EPI_PARTIAL, false);
      if (n_ex > 0) {
        G.splits = static_cast<int>(n_ex);
        G.per_plane = 1;
        const int a = g.a_mnmajor_planes(jobs[j].Q, jobs[j].f, seq, n_ex, jobs[j].f);
        GemmPlan::seg(G, a, tm, -1, seq, seq);
      } else {
        G.splits = choose_splits(tiles, ceil_div(M, kBK), num_sms());
        const int a = g.a_mnmajor(jobs[j].Q, jobs[j].f, M, jobs[j].f);
        GemmPlan::seg(G, a, tm, -1, M, M);
      }
      G.part = cur;
      parts[gi] = cur;
      kfs[gi] = kfj;
      cur += round_up(partial_elems(jobs[j].f, kfj, g.bn, slab_splits), 64);
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
    o.width = static_cast<int>(round_up(kfs[group_of[j]], g.bn));
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


// ---------------------------------------------------------------- one-pass rank-r products

// The split of a one-pass launch into gt token ranges x gf feature ranges (one CTA
// each): every range non-empty, at most kDualMaxBlocks feature blocks a CTA (its TMEM),
// gt * gf within kDualMaxCtas (the SMs of a GB300; a fixed number, so that workspace
// sizes do not depend on the device).  Cost, in units of one CTA's 128 x 128 tile: the
// busiest CTA's tiles plus the partial sums' bytes (written and read back) spread over
// the CTAs.
struct DualPlan {
  int gt = 0, gf = 0, nv = 0;
};
static DualPlan dual_plan(int64_t M, int r, const int64_t* F, int njobs) {
  DualPlan P;
  int slots = 0;
  for (int j = 0; j < njobs; ++j) slots = r * (j + 1);
  P.nv = static_cast<int>(round_up(slots, 16));
  const int64_t tm = ceil_div(M, 128);
  int64_t kb = 0, frows = 0;
  for (int j = 0; j < njobs; ++j) {
    kb += ceil_div(F[j], 128);
    frows += ceil_div(F[j], 128) * 128;
  }
  constexpr int sms = kDualMaxCtas;
  double best = 1e30;
  for (int64_t gf = ceil_div(kb, kDualMaxBlocks); gf <= kb && gf <= sms; ++gf) {
    const int64_t gt = tm < sms / gf ? tm : sms / gf;
    if (gt < 1) break;
    const double tiles = static_cast<double>(ceil_div(tm, gt) * ceil_div(kb, gf));
    const double bytes = 2.0 * 4.0 * (static_cast<double>(gf) * tm * 128 * P.nv + static_cast<double>(gt) * frows * kDualNRMax);
    const double cost = tiles + bytes / (static_cast<double>(kDualQBytes) * gt * gf);
    if (cost < best) {
      best = cost;
      P.gt = static_cast<int>(gt);
      P.gf = static_cast<int>(gf);
    }
  }
  return P;
}

void dual_slab_elems(int64_t M, int r, const int64_t* F, int njobs, int64_t& v_elems, int64_t& db_elems) {
  const DualPlan P = dual_plan(M, r, F, njobs);
  v_elems = round_up(static_cast<int64_t>(P.gf) * ceil_div(M, 128) * 128 * P.nv, 64);
  db_elems = 0;
  for (int j = 0; j < njobs; ++j) db_elems += round_up(static_cast<int64_t>(P.gt) * ceil_div(F[j], 128) * 128 * kDualNRMax, 64);
}

lora_status_t rank_dual(int64_t M, int r, int kf, float s, const DualJob* jobs, int njobs, const void* Tt,
                        int64_t ldt, void* V, float* vslab, Deferred& defer, unsigned* status, cudaStream_t st) {
  if (M == 0) return LORA_OK;
  if (!dual_supported(r, kf, njobs)) return LORA_ERR_UNSUPPORTED;
  int64_t F[kDualMaxProducts];
  for (int j = 0; j < njobs; ++j) F[j] = jobs[j].F;
  const DualPlan P = dual_plan(M, r, F, njobs);
  if (P.gt < 1 || P.gf < 1 || P.nv > kDualNVMax || P.nv > kf) return LORA_ERR_UNSUPPORTED;
  DualParams d;
  std::memset(static_cast<void*>(&d), 0, sizeof(d));
  d.nprod = njobs;
  d.tiles_m = static_cast<int>(ceil_div(M, 128));
  d.nv = P.nv;
  d.nr = kDualNRMax;
  d.gt = P.gt;
  d.gf = P.gf;
  d.v_part = vslab;
  d.status = status;
  d.timeout_ns = g_timeout_ns.load();
  float* cur = defer.cursor;
  for (int j = 0; j < njobs; ++j) {
    DualProduct& D = d.prod[j];
    D.nkb = static_cast<int>(ceil_div(F[j], 128));
    D.t_row = jobs[j].t_row;
    D.q_map = 3 * j;
    D.b_map = 3 * j + 1;
    D.t_map = 3 * j + 2;
    if (!encode_map(&d.maps[D.q_map], jobs[j].Q, F[j], M, F[j], 64, 128, 128) ||
        !encode_map(&d.maps[D.b_map], jobs[j].Bt, F[j], kf, F[j], 64, P.nv, 128) ||
        !encode_map(&d.maps[D.t_map], Tt, M, kf, ldt, 64, kDualNRMax, 128))
      return LORA_ERR_CUDA;
    D.db_part = cur;
    cur += round_up(static_cast<int64_t>(P.gt) * D.nkb * 128 * kDualNRMax, 64);
    d.kb_total += D.nkb;
  }
  defer.cursor = cur;
  const int slot = trace_begin(LORA_KIND_RANK_GRAD, st);
  cudaError_t e = launch_rank_dual(d, P.gt * P.gf, st);
  trace_end(slot, st);
  if (e != cudaSuccess) return LORA_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  // V now (the next GEMM reads it); the dB sums with the call's other reductions
  RedParams rv;
  std::memset(static_cast<void*>(&rv), 0, sizeof(rv));
  rv.nout = 1;
  RedOut& o = rv.out[0];
  o.part = vslab;
  o.rows = static_cast<int>(M);
  o.rows_pad = d.tiles_m * 128;
  o.width = P.nv;
  o.splits = P.gf;
  o.scale = 1.0f;
  o.dst = static_cast<bf16*>(V);
  o.col0 = 0;
  o.ncols = P.nv;
  o.ld = kf;
  o.trans = 0;
  LGB_TRY(launch_reduce(rv, st));
  for (int j = 0; j < njobs; ++j) {
    if (defer.rp.nout >= kMaxRedOuts) return LORA_ERR_UNSUPPORTED;   // not reached: <= 8 per call
    RedOut& b = defer.rp.out[defer.rp.nout++];
    b.part = d.prod[j].db_part;
    b.rows = static_cast<int>(F[j]);
    b.rows_pad = static_cast<long long>(d.prod[j].nkb) * 128;
    b.width = kDualNRMax;
    b.splits = P.gt;
    b.per_split = 0;
    b.scale = s;
    b.dst = static_cast<bf16*>(jobs[j].dB);
    b.col0 = 0;
    b.ncols = r;
    b.ld = r;
    b.trans = 0;
  }
  return LORA_OK;
}

lora_status_t check_common(int64_t M, int r, float s) {
  if (M < 0 || r < 1 || !std::isfinite(s)) return LORA_ERR_INVALID_ARG;
  if (M > kMaxExtent) return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

}  // namespace lgb

using namespace lgb;

// ================================================================ status and trace

extern "C" lora_status_t lora_poll_status(void* ws, cudaStream_t stream) {
  if (ws == nullptr) {
    ws = noalloc_scratch();     // the no-allocation forward's status word on this device
    if (ws == nullptr) return LORA_ERR_CUDA;
  }
  if (!aligned(ws, 256)) return LORA_ERR_INVALID_ARG;
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

extern "C" lora_status_t lora_set_split_tail(int mode) {
  if (mode < 0 || mode > kSkMaxSplits) return LORA_ERR_INVALID_ARG;
  g_split_tail.store(mode);
  return LORA_OK;
}

extern "C" int lora_split_tail(void) { return g_split_tail.load(); }

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
