// Entry points of the Q/K/V + O projections (lora_qkvo_*), with frozen biases and RoPE.
#include <cmath>
#include <cstring>

#include "api_internal.cuh"

using namespace lgb;

// ================================================================ Q/K/V + O

namespace {

struct QkvoLayout {
  int kfq, kfo;
  size_t ws_fwd, ws_bwd, saved, off_to;
  size_t off_tqkvt, off_tot;   // the rank-r projections transposed, [kf x ldt] (single passes
  int64_t ldt;                 // over dy_q, dy_k, dy_v and over dy_o in the backward)
  // the backward's packed adapter operands, written by the forward's pack launch
  size_t off_btq, off_btk, off_btv, off_afqkv, off_bto, off_afo;
};

// Single passes over the backward's gradients (dual_supported): the q/k/v half's three
// products and the o half's one.
static bool qkv_dual(int r, int kfq) { return dual_supported(r, kfq, 3); }
static bool o_dual(int r, int kfo) { return dual_supported(r, kfo, 1); }

// Backward scratch, as for the MLP: rank-r projection slabs (and the single passes' V
// slabs), then the token reductions' (and the single passes' dB slabs).
static int64_t qkvo_bwd_rank_part(int64_t M, int64_t h, int64_t nq, int64_t nkv, int r, int kfq, int kfo) {
  int64_t p = imax(rank_projection_part(M, kfo, ceil_div(h, kBK)),
                   rank_projection_part(M, kfq, ceil_div(nq, kBK) + 2 * ceil_div(nkv, kBK)));
  int64_t v = 0, db = 0;
  if (o_dual(r, kfo)) {
    dual_slab_elems(M, r, &h, 1, v, db);
    p = imax(p, v);
  }
  if (qkv_dual(r, kfq)) {
    const int64_t f3[3] = {nq, nkv, nkv};
    dual_slab_elems(M, r, f3, 3, v, db);
    p = imax(p, v);
  }
  return p;
}
static int64_t qkvo_bwd_slabs(int64_t M, int64_t h, int64_t nq, int64_t nkv, int r, int kfq, int kfo) {
  const int64_t f3[3] = {nq, nkv, nkv};
  int64_t n = token_grad_part(M, kfo, &h, 1) + token_grad_part(M, kfo, &nq, 1) + token_grad_part(M, kfq, f3, 3) +
              token_grad_part(M, kfq, &h, 1);
  int64_t v = 0, db = 0;
  if (o_dual(r, kfo)) {
    dual_slab_elems(M, r, &h, 1, v, db);
    n += db;
  }
  if (qkv_dual(r, kfq)) {
    dual_slab_elems(M, r, f3, 3, v, db);
    n += db;
  }
  return n;
}

// Largest pair-GEMM tile counts of the forward (q/k/v in one launch, o) and the
// backward (d o_in, dx).
static int64_t qkvo_fwd_tiles(int64_t M, int64_t h, int64_t nq, int64_t nkv) {
  return imax(pair_tiles(M, nq) + 2 * pair_tiles(M, nkv), pair_tiles(M, h));
}
static int64_t qkvo_bwd_tiles(int64_t M, int64_t h, int64_t nq) { return imax(pair_tiles(M, nq), pair_tiles(M, h)); }

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
    carve_sk(c, qkvo_fwd_tiles(M, h, nq, nkv));
    L.ws_fwd = c.off;
  }
  {
    Carve c(nullptr);
    c.take(kWsHeader);
    c.take_n<bf16>(M * kfo);
    c.take_n<bf16>(M * kfq);
    c.take_n<bf16>(M * nq);     // dy_q, dy_k turned back by the transpose RoPE rotation
    c.take_n<bf16>(M * nkv);
    c.take_n<float>(qkvo_bwd_rank_part(M, h, nq, nkv, r, kfq, kfo));
    c.take_n<float>(qkvo_bwd_slabs(M, h, nq, nkv, r, kfq, kfo));
    carve_sk(c, qkvo_bwd_tiles(M, h, nq));
    L.ws_bwd = c.off;
  }
  {
    Carve c(nullptr);
    c.offset_of(sizeof(bf16) * M * kfq);
    L.off_to = c.offset_of(sizeof(bf16) * M * kfo);
    L.ldt = round_up(M, 8);
    L.off_tqkvt = c.offset_of(sizeof(bf16) * kfq * L.ldt);
    L.off_tot = c.offset_of(sizeof(bf16) * kfo * L.ldt);
    L.off_btq = c.offset_of(sizeof(bf16) * kfq * nq);
    L.off_btk = c.offset_of(sizeof(bf16) * kfq * nkv);
    L.off_btv = c.offset_of(sizeof(bf16) * kfq * nkv);
    L.off_afqkv = c.offset_of(sizeof(bf16) * kfq * h);
    L.off_bto = c.offset_of(sizeof(bf16) * kfo * h);
    L.off_afo = c.offset_of(sizeof(bf16) * kfo * nq);
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
  const SkRegion sk = carve_sk(c, qkvo_fwd_tiles(M, h, n_q, n_kv));
  bf16* tqkv_t = nullptr;
  bf16* to_t = nullptr;
  if (saved) {
    tqkv = static_cast<bf16*>(saved);
    to = reinterpret_cast<bf16*>(static_cast<uint8_t*>(saved) + L.off_to);
    tqkv_t = reinterpret_cast<bf16*>(static_cast<uint8_t*>(saved) + L.off_tqkvt);
    to_t = reinterpret_cast<bf16*>(static_cast<uint8_t*>(saved) + L.off_tot);
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
  if (saved) {
    // the backward's operands too (it reads them from saved, as autograd reads the
    // tensors a forward saved)
    uint8_t* sv = static_cast<uint8_t*>(saved);
    if (x) {
      pack_block(pack_job(pk, sv + L.off_btq, kfq, n_q), q.B, r, 0, 0, r, static_cast<int>(n_q), 1, 1.0f);
      pack_block(pack_job(pk, sv + L.off_btk, kfq, n_kv), k.B, r, r, 0, r, static_cast<int>(n_kv), 1, 1.0f);
      pack_block(pack_job(pk, sv + L.off_btv, kfq, n_kv), v.B, r, 2 * r, 0, r, static_cast<int>(n_kv), 1, 1.0f);
      PackJob& J = pack_job(pk, sv + L.off_afqkv, kfq, h);
      pack_block(J, q.A, h, 0, 0, r, static_cast<int>(h), 0, s);
      pack_block(J, k.A, h, r, 0, r, static_cast<int>(h), 0, s);
      pack_block(J, v.A, h, 2 * r, 0, r, static_cast<int>(h), 0, s);
    }
    if (o_in) {
      pack_block(pack_job(pk, sv + L.off_bto, kfo, h), o.B, r, 0, 0, r, static_cast<int>(h), 1, 1.0f);
      pack_block(pack_job(pk, sv + L.off_afo, kfo, n_q), o.A, n_q, 0, 0, r, static_cast<int>(n_q), 0, s);
    }
  }
  LGB_TRY(launch_pack(pk, stream));

  if (x) {
    const ProjSeg p1 = {x, acat, h};
    LGB_TRY(rank_projection(M, kfq, &p1, 1, tqkv, part, status, stream, qkv_dual(r, kfq) ? tqkv_t : nullptr, L.ldt,
                            3 * r));
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
    g.p.pdl_seg = 1;   // segments from 1 on read the previous kernel's rank-r output
    g.finish();
    g.split_tail(sk);
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKK, g.p, LORA_KIND_PROJ, stream));
  }
  if (o_in) {
    const ProjSeg p2 = {o_in, acat_o, n_q};
    LGB_TRY(rank_projection(M, kfo, &p2, 1, to, part, status, stream, o_dual(r, kfo) ? to_t : nullptr, L.ldt, r));
    GemmPlan g(kBigKK);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(h), EPI_STORE, false);
    GemmPlan::seg(G, g.a_kmajor(o_in, M, n_q, n_q), g.b_kmajor(o.W, h, n_q, n_q, g.b_rows_full()), -1, n_q, n_q);
    GemmPlan::seg(G, g.a_kmajor(to, M, kfo, kfo), g.b_kmajor(bf_o, h, kfo, kfo, g.b_rows_full()), -1, kfo, r);
    G.out0 = yo;
    G.ldo = h;
    g.p.status = status;
    g.p.pdl_seg = 1;   // segments from 1 on read the previous kernel's rank-r output
    g.finish();
    g.split_tail(sk);
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
  const bf16* tqkv_t = reinterpret_cast<const bf16*>(static_cast<const uint8_t*>(saved) + L.off_tqkvt);
  const bf16* to_t = reinterpret_cast<const bf16*>(static_cast<const uint8_t*>(saved) + L.off_tot);
  Carve c(ws);
  unsigned* status = static_cast<unsigned*>(c.take(kWsHeader));
  // the adapter operands come packed from the forward (saved)
  const uint8_t* svb = static_cast<const uint8_t*>(saved);
  const bf16* btq = reinterpret_cast<const bf16*>(svb + L.off_btq);
  const bf16* btk = reinterpret_cast<const bf16*>(svb + L.off_btk);
  const bf16* btv = reinterpret_cast<const bf16*>(svb + L.off_btv);
  const bf16* af_qkv = reinterpret_cast<const bf16*>(svb + L.off_afqkv);
  const bf16* bt_o = reinterpret_cast<const bf16*>(svb + L.off_bto);
  const bf16* af_o = reinterpret_cast<const bf16*>(svb + L.off_afo);
  bf16* uo = c.take_n<bf16>(M * kfo);
  bf16* V = c.take_n<bf16>(M * kfq);
  bf16* dyq_r = c.take_n<bf16>(M * n_q);
  bf16* dyk_r = c.take_n<bf16>(M * n_kv);
  float* part = c.take_n<float>(qkvo_bwd_rank_part(M, h, n_q, n_kv, r, kfq, kfo));
  Deferred dr;
  defer_init(dr, c.take_n<float>(qkvo_bwd_slabs(M, h, n_q, n_kv, r, kfq, kfo)));
  const SkRegion sk = carve_sk(c, qkvo_bwd_tiles(M, h, n_q));


  // dA_o joins the q, k, v reductions' launch after the dx GEMM when both one-pass
  // kernels run (one launch fewer; GQA 7B-shaped step -0.3%)
  GradJob pend{};
  bool pending = false;
  if (o_in) {
    const bool dual = o_dual(r, kfo);
    if (dual) {
      // U_o = dy_o B_o and dB_o = s dy_o^T T_o in one pass over dy_o
      const DualJob jd = {dyo, h, bt_o, 0, d_o.dB};
      LGB_TRY(rank_dual(M, r, kfo, s, &jd, 1, to_t, L.ldt, uo, part, dr, status, stream));
    } else {
      const ProjSeg p1 = {dyo, bt_o, h};
      LGB_TRY(rank_projection(M, kfo, &p1, 1, uo, part, status, stream));
    }
    GemmPlan g(kBigKMN);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(n_q), EPI_STORE, false);
    GemmPlan::seg(G, g.a_kmajor(dyo, M, h, h), g.b_mnmajor(o.W, n_q, h, n_q), -1, h, h);
    GemmPlan::seg(G, g.a_kmajor(uo, M, kfo, kfo), g.b_mnmajor(af_o, n_q, kfo, n_q), -1, kfo, r);
    G.out0 = do_in;
    G.ldo = n_q;
    g.p.status = status;
    g.p.pdl_seg = 1;   // segments from 1 on read the previous kernel's rank-r output
    g.finish();
    g.split_tail(sk);
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKMN, g.p, LORA_KIND_DGRAD, stream));
    // dA_o = s U_o^T o_in (and dB_o = s dy_o^T T_o when the pass over dy_o has not made
    // it) in one launch: they read nothing the d o_in GEMM writes
    const GradJob j1[2] = {{dyo, h, 0, d_o.dB, 0, to, kfo}, {o_in, n_q, 0, d_o.dA, 1, uo, kfo}};
    if (dual && x != nullptr && qkv_dual(r, kfq) && skinny_bn(kfo) == skinny_bn(kfq)) {
      pend = j1[1];
      pending = true;
    } else {
      LGB_TRY(token_grads(M, r, kfo, s, dual ? j1 + 1 : j1, dual ? 1 : 2, dr, status, stream, 0, true));
    }
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
    const bool dual = qkv_dual(r, kfq);
    if (dual) {
      // V = [dy_q B_q | dy_k B_k | dy_v B_v] and dB_q, dB_k, dB_v in one pass over them
      const DualJob jd[3] = {{dyq, n_q, btq, 0, d_q.dB}, {dyk, n_kv, btk, r, d_k.dB}, {dyv, n_kv, btv, 2 * r, d_v.dB}};
      LGB_TRY(rank_dual(M, r, kfq, s, jd, 3, tqkv_t, L.ldt, V, part, dr, status, stream));
    } else {
      const ProjSeg p3[3] = {{dyq, btq, n_q}, {dyk, btk, n_kv}, {dyv, btv, n_kv}};
      LGB_TRY(rank_projection(M, kfq, p3, 3, V, part, status, stream));
    }
    GemmPlan g(kBigKMN);
    GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(h), EPI_STORE, false);
    GemmPlan::seg(G, g.a_kmajor(dyq, M, n_q, n_q), g.b_mnmajor(q.W, h, n_q, h), -1, n_q, n_q);
    GemmPlan::seg(G, g.a_kmajor(dyk, M, n_kv, n_kv), g.b_mnmajor(k.W, h, n_kv, h), -1, n_kv, n_kv);
    GemmPlan::seg(G, g.a_kmajor(dyv, M, n_kv, n_kv), g.b_mnmajor(v.W, h, n_kv, h), -1, n_kv, n_kv);
    GemmPlan::seg(G, g.a_kmajor(V, M, kfq, kfq), g.b_mnmajor(af_qkv, h, kfq, h), -1, kfq, 3 * r);
    G.out0 = dx;
    G.ldo = h;
    g.p.status = status;
    g.p.pdl_seg = 3;   // segments from 3 on read the previous kernel's rank-r output
    g.finish();
    g.split_tail(sk);
    if (!g.ok) return LORA_ERR_CUDA;
    LGB_TRY(launch_gemm(kBigKMN, g.p, LORA_KIND_DGRAD, stream));
    // the q, k, v dA (and dB when the pass over dy_q, dy_k, dy_v has not made them) in one
    // launch: they read nothing the dx GEMM writes
    const GradJob j3[6] = {{dyq, n_q, 0, d_q.dB, 0, tqkv}, {dyk, n_kv, r, d_k.dB, 0, tqkv},
                           {dyv, n_kv, 2 * r, d_v.dB, 0, tqkv}, {x, h, 0, d_q.dA, 1, V},
                           {x, h, r, d_k.dA, 1, V}, {x, h, 2 * r, d_v.dA, 1, V}};
    if (pending) {
      const GradJob jm[4] = {pend, j3[3], j3[4], j3[5]};
      LGB_TRY(token_grads(M, r, kfq, s, jm, 4, dr, status, stream, 0, true));
    } else {
      LGB_TRY(token_grads(M, r, kfq, s, dual ? j3 + 3 : j3, dual ? 3 : 6, dr, status, stream, 0, true));
    }
  }
  return defer_flush(dr, stream);
}
