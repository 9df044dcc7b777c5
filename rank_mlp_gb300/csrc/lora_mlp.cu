// Entry points of the gated LoRA MLP (lora_mlp_*), including per-example gradients.
#include <cmath>
#include <cstring>

#include "api_internal.cuh"

using namespace lgb;

// ================================================================ gated MLP

namespace {

struct MlpLayout {
  int kfg, kfd;    // padded rank widths: gate/up pair, down
  size_t ws_fwd, ws_bwd, saved;
  // saved blob offsets
  size_t off_g, off_u, off_h, off_tgu, off_td;
  size_t off_tgut;   // T_gu transposed [kfg x ldt] (the backward's one pass over dg, du)
  int64_t ldt;
  // the backward's packed adapter operands, written by the forward's pack launch
  size_t off_bt_d, off_af_d, off_bt_g, off_bt_u, off_af_gu;
};

// The backward's packed operands: B_d^T, s A_d, B_g^T and B_u^T (in their slots), s [A_g; A_u].
struct MlpBwdPack {
  bf16 *bt_d, *af_d, *bt_g, *bt_u, *af_gu;
};
void pack_mlp_bwd(PackParams& pk, const MlpBwdPack& P, lora_linear_t gate, lora_linear_t up, lora_linear_t down,
                  int64_t h, int64_t i, int r, float s, int kfg, int kfd) {
  pack_block(pack_job(pk, P.bt_d, kfd, h), down.B, r, 0, 0, r, static_cast<int>(h), 1, 1.0f);
  pack_block(pack_job(pk, P.af_d, kfd, i), down.A, i, 0, 0, r, static_cast<int>(i), 0, s);
  pack_block(pack_job(pk, P.bt_g, kfg, i), gate.B, r, 0, 0, r, static_cast<int>(i), 1, 1.0f);
  pack_block(pack_job(pk, P.bt_u, kfg, i), up.B, r, r, 0, r, static_cast<int>(i), 1, 1.0f);
  PackJob& J = pack_job(pk, P.af_gu, kfg, h);
  pack_block(J, gate.A, h, 0, 0, r, static_cast<int>(h), 0, s);
  pack_block(J, up.A, h, r, 0, r, static_cast<int>(h), 0, s);
}

// Backward scratch: the rank-r projections' split-K slabs (reused), then the four token
// reductions' slabs (kept until the call's final reduce).
// With one pass over dg, du (dual_supported): the V slab shares the projections' region
// and the dB_g, dB_u slabs join the others.
static bool mlp_dual(int r, int kfg, int64_t n_ex) { return n_ex == 0 && dual_supported(r, kfg, 2); }
static int64_t mlp_bwd_rank_part(int64_t M, int64_t h, int64_t i, int r, int kfd, int kfg, int64_t n_ex) {
  int64_t p = imax(rank_projection_part(M, kfd, ceil_div(h, kBK)), rank_projection_part(M, kfg, 2 * ceil_div(i, kBK)));
  if (mlp_dual(r, kfg, n_ex)) {
    const int64_t F[2] = {i, i};
    int64_t v = 0, db = 0;
    dual_slab_elems(M, r, F, 2, v, db);
    p = imax(p, v);
  }
  return p;
}
static int64_t mlp_bwd_slabs(int64_t M, int64_t h, int64_t i, int r, int kfd, int kfg, int64_t n_ex) {
  const int64_t f2[2] = {i, i};
  int64_t n = token_grad_part(M, kfd, &h, 1, n_ex) + token_grad_part(M, kfd, &i, 1, n_ex) +
              token_grad_part(M, kfg, f2, 2, n_ex) + token_grad_part(M, kfg, &h, 1, n_ex);
  if (mlp_dual(r, kfg, n_ex)) {
    int64_t v = 0, db = 0;
    dual_slab_elems(M, r, f2, 2, v, db);
    n += db;
  }
  return n;
}

// Largest pair-GEMM tile counts of the forward (gate/up, down) and backward (act', dx).
static int64_t mlp_fwd_tiles(int64_t M, int64_t h, int64_t i) {
  return imax(pair_tiles(M, i, true), pair_tiles(M, h));
}
static int64_t mlp_bwd_tiles(int64_t M, int64_t h, int64_t i) { return imax(pair_tiles(M, i), pair_tiles(M, h)); }

// n_ex > 0: workspace of the per-example backward (one reduction slab per example).
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
    carve_sk(c, mlp_fwd_tiles(M, h, i));
    L.ws_fwd = c.off;
  }
  {
    Carve c(nullptr);
    c.take(kWsHeader);
    c.take_n<bf16>(M * kfd);     // U_d
    c.take_n<bf16>(M * i);       // dg
    c.take_n<bf16>(M * i);       // du
    c.take_n<bf16>(M * kfg);     // V
    c.take_n<float>(mlp_bwd_rank_part(M, h, i, r, kfd, kfg, n_ex));
    c.take_n<float>(mlp_bwd_slabs(M, h, i, r, kfd, kfg, n_ex));
    carve_sk(c, mlp_bwd_tiles(M, h, i));
    L.ws_bwd = c.off;
  }
  {
    Carve c(nullptr);
    L.off_g = c.offset_of(sizeof(bf16) * M * i);
    L.off_u = c.offset_of(sizeof(bf16) * M * i);
    L.off_h = c.offset_of(sizeof(bf16) * M * i);
    L.off_tgu = c.offset_of(sizeof(bf16) * M * kfg);
    L.off_td = c.offset_of(sizeof(bf16) * M * kfd);
    L.ldt = round_up(M, 8);
    L.off_tgut = c.offset_of(sizeof(bf16) * kfg * L.ldt);
    L.off_bt_d = c.offset_of(sizeof(bf16) * kfd * h);
    L.off_af_d = c.offset_of(sizeof(bf16) * kfd * i);
    L.off_bt_g = c.offset_of(sizeof(bf16) * kfg * i);
    L.off_bt_u = c.offset_of(sizeof(bf16) * kfg * i);
    L.off_af_gu = c.offset_of(sizeof(bf16) * kfg * h);
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
  const SkRegion sk = carve_sk(c, mlp_fwd_tiles(M, h, i));
  bf16* gbuf = nullptr;
  bf16* ubuf = nullptr;
  bf16* tgut = nullptr;
  if (saved) {
    uint8_t* sv = static_cast<uint8_t*>(saved);
    tgut = reinterpret_cast<bf16*>(sv + L.off_tgut);
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
  if (saved) {
    // the backward's operands too (it reads them from saved, as autograd reads the
    // tensors a forward saved)
    uint8_t* sv = static_cast<uint8_t*>(saved);
    const MlpBwdPack P = {reinterpret_cast<bf16*>(sv + L.off_bt_d), reinterpret_cast<bf16*>(sv + L.off_af_d),
                          reinterpret_cast<bf16*>(sv + L.off_bt_g), reinterpret_cast<bf16*>(sv + L.off_bt_u),
                          reinterpret_cast<bf16*>(sv + L.off_af_gu)};
    pack_mlp_bwd(pk, P, gate, up, down, h, i, r, s, kfg, kfd);
  }
  LGB_TRY(launch_pack(pk, stream));

  // T_gu = x [A_g; A_u]^T (saved also transposed where the backward's pass over dg, du
  // reads it)
  const ProjSeg p1 = {x, acat_gu, h};
  LGB_TRY(rank_projection(M, kfg, &p1, 1, tgu, part, status, stream, mlp_dual(r, kfg, 0) ? tgut : nullptr, L.ldt,
                          2 * r));

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
    g.p.pdl_seg = 1;   // segments from 1 on read the previous kernel's rank-r output
    g.finish();
    g.split_tail(sk);
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
  g.p.pdl_seg = 1;   // segments from 1 on read the previous kernel's rank-r output
  g.finish();
  g.split_tail(sk);
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
  const bf16* tgut = reinterpret_cast<const bf16*>(sv + L.off_tgut);
  const bool dual = mlp_dual(r, kfg, n_ex);

  Carve c(ws);
  unsigned* status = static_cast<unsigned*>(c.take(kWsHeader));
  const bf16* bt_d = reinterpret_cast<const bf16*>(sv + L.off_bt_d);
  const bf16* af_d = reinterpret_cast<const bf16*>(sv + L.off_af_d);
  const bf16* bt_g = reinterpret_cast<const bf16*>(sv + L.off_bt_g);
  const bf16* bt_u = reinterpret_cast<const bf16*>(sv + L.off_bt_u);
  const bf16* af_gu = reinterpret_cast<const bf16*>(sv + L.off_af_gu);
  bf16* ud = c.take_n<bf16>(M * kfd);
  bf16* dg = c.take_n<bf16>(M * i);
  bf16* du = c.take_n<bf16>(M * i);
  bf16* V = c.take_n<bf16>(M * kfg);
  float* part = c.take_n<float>(mlp_bwd_rank_part(M, h, i, r, kfd, kfg, n_ex));
  Deferred dr;
  defer_init(dr, c.take_n<float>(mlp_bwd_slabs(M, h, i, r, kfd, kfg, n_ex)));
  const SkRegion sk = carve_sk(c, mlp_bwd_tiles(M, h, i));

  // the adapter operands come packed from the forward (saved)

  // U_d = dy B_d
  const ProjSeg p1 = {dy, bt_d, h};
  LGB_TRY(rank_projection(M, kfd, &p1, 1, ud, part, status, stream));

  // dh = [dy | U_d] [W_d ; s A_d];  dg = dh u act'(g), du = dh act(g).  Short K: g, u read
  // and dg, du written through shared memory (whole tiles: that variant has no split
  // tail); long K: one row per thread.
  {
    const bool staged = ceil_div(h, kBK) + ceil_div(r, kBK) <= kActShortKBlocks;
    const int variant = staged ? VP_KMN_ACT16 : VP_KMN_ACT;
    GemmPlan g(variant);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(i), EPI_ACT_BWD, false);
    GemmPlan::seg(G, g.a_kmajor(dy, M, h, h), g.b_mnmajor(down.W, i, h, i), -1, h, h);
    GemmPlan::seg(G, g.a_kmajor(ud, M, kfd, kfd), g.b_mnmajor(af_d, i, kfd, i), -1, kfd, r);
    if (staged) {
      G.emap[0] = g.epi_map(gsv, M, i, i);
      G.emap[1] = g.epi_map(usv, M, i, i);
      G.emap[2] = g.epi_map(dg, M, i, i);
      G.emap[3] = g.epi_map(du, M, i, i);
    } else {
      G.in0 = gsv;
      G.in1 = usv;
      G.ldi = i;
      G.out0 = dg;
      G.out1 = du;
      G.ldo = i;
    }
    g.p.act = static_cast<int>(act);
    g.p.status = status;
    g.p.pdl_seg = 1;   // segments from 1 on read the previous kernel's rank-r output
    g.finish();
    if (!staged) g.split_tail(sk);
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(variant, g.p, LORA_KIND_ACT_BWD, stream));
  }

  // dB_d = s dy^T T_d and dA_d = s U_d^T h read nothing the dh GEMM writes.  With the
  // one pass over dg, du below they join the launch after the dx GEMM (one launch
  // fewer; on the 0.5B shape, whose dx GEMM leaves 24 SMs idle throughout, step -1.9%);
  // otherwise they take a launch of their own here, which starts on the SMs the dh
  // GEMM's last wave leaves idle.  (A single pass over dy for U_d and dB_d, as for dg,
  // du below, measured no better: dy is a quarter of dg, du's bytes.)
  const GradJob j1[2] = {{dy, h, 0, d_down.dB, 0, td, kfd}, {hsv, i, 0, d_down.dA, 1, ud, kfd}};
  const bool merge_j1 = dual && skinny_bn(kfd) == skinny_bn(kfg);
  if (!merge_j1) LGB_TRY(token_grads(M, r, kfd, s, j1, 2, dr, status, stream, n_ex, true));

  if (dual) {
    // V = [dg B_g | du B_u], dB_g = s dg^T T_g and dB_u = s du^T T_u in one pass over dg, du
    const DualJob jd[2] = {{dg, i, bt_g, 0, d_gate.dB}, {du, i, bt_u, r, d_up.dB}};
    LGB_TRY(rank_dual(M, r, kfg, s, jd, 2, tgut, L.ldt, V, part, dr, status, stream));
  } else {
    // V = [dg B_g | du B_u]
    const ProjSeg p3[2] = {{dg, bt_g, i}, {du, bt_u, i}};
    LGB_TRY(rank_projection(M, kfg, p3, 2, V, part, status, stream));
  }


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
    g.p.pdl_seg = 2;   // segments from 2 on read the previous kernel's rank-r output
    g.finish();
    g.split_tail(sk);
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKMN, g.p, LORA_KIND_DGRAD, stream));
  }

  // dA_g = s V_g^T x, dA_u = s V_u^T x (and dB_g = s dg^T T_g, dB_u = s du^T T_u when
  // the pass over dg, du has not made them, or dB_d, dA_d when it has) in one launch:
  // they read nothing the dx GEMM writes and start on the SMs its last wave leaves idle
  const GradJob j3[4] = {{dg, i, 0, d_gate.dB, 0, tgu}, {du, i, r, d_up.dB, 0, tgu},
                         {x, h, 0, d_gate.dA, 1, V}, {x, h, r, d_up.dA, 1, V}};
  if (merge_j1) {
    const GradJob jm[4] = {j1[0], j1[1], j3[2], j3[3]};
    LGB_TRY(token_grads(M, r, kfg, s, jm, 4, dr, status, stream, n_ex, true));
  } else {
    LGB_TRY(token_grads(M, r, kfg, s, dual ? j3 + 2 : j3, dual ? 2 : 4, dr, status, stream, n_ex, true));
  }
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
