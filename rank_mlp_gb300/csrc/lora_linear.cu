// Entry points of the single LoRA linear (lora_linear_*; the no-allocation variant is
// in noalloc.cu).
#include <cmath>
#include <cstring>

#include "api_internal.cuh"

using namespace lgb;

// ================================================================ single linear

namespace {

struct LinearLayout {
  int kf;
  size_t ws_fwd_base;   // the forward without the split-tail regions (last in its layout)
  size_t ws_fwd, ws_bwd, saved;
  size_t off_bt, off_af;   // saved: the backward's packed operands B^T and s A
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
    L.ws_fwd_base = c.off;
    carve_sk(c, pair_tiles(M, out));
    L.ws_fwd = c.off;
  }
  {
    Carve c(nullptr);
    c.take(kWsHeader);
    c.take_n<bf16>(M * kf);     // U
    c.take_n<float>(rank_projection_part(M, kf, ceil_div(out, kBK)));
    c.take_n<float>(token_grad_part(M, kf, &out, 1) + token_grad_part(M, kf, &in, 1));   // dB, dA slabs
    carve_sk(c, pair_tiles(M, in));
    L.ws_bwd = c.off;
  }
  {
    Carve c(nullptr);
    c.take_n<bf16>(M * kf);
    L.off_bt = c.offset_of(sizeof(bf16) * kf * out);
    L.off_af = c.offset_of(sizeof(bf16) * kf * in);
    L.saved = c.off;
  }
  return L;
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

size_t lgb::linear_forward_workspace_bytes(int64_t M, int64_t in, int64_t out, int r) {
  if (M < 0 || in <= 0 || out <= 0 || r < 1) return 0;
  return linear_layout(M, in, out, r).ws_fwd_base;
}

// The forward; with split_tail false the projection runs whole tiles only and ws needs
// only the part of the layout before the split-tail regions
// (linear_forward_workspace_bytes).
static lora_status_t linear_forward_impl(int64_t M, int64_t in, int64_t out, int r, float s, const void* x,
                                         lora_linear_t lin, void* y, void* saved, void* ws, size_t ws_bytes,
                                         cudaStream_t stream, bool split_tail) {
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
  if (ws_bytes < (split_tail ? L.ws_fwd : L.ws_fwd_base)) return LORA_ERR_WORKSPACE;
  if (M == 0) return LORA_OK;
  const int kf = L.kf;
  Carve c(ws);
  unsigned* status = static_cast<unsigned*>(c.take(kWsHeader));
  bf16* acat = c.take_n<bf16>(kf * in);
  bf16* bf = c.take_n<bf16>(out * kf);
  float* part = c.take_n<float>(rank_projection_part(M, kf, ceil_div(in, kBK)));
  bf16* T = c.take_n<bf16>(M * kf);
  if (saved) T = static_cast<bf16*>(saved);
  const SkRegion sk = split_tail ? carve_sk(c, pair_tiles(M, out)) : SkRegion();

  PackParams pk;
  std::memset(static_cast<void*>(&pk), 0, sizeof(pk));
  pack_block(pack_job(pk, acat, kf, in), lin.A, in, 0, 0, r, static_cast<int>(in), 0, 1.0f);
  pack_block(pack_job(pk, bf, out, kf), lin.B, r, 0, 0, static_cast<int>(out), r, 0, s);
  if (saved) {
    // the backward's operands too (it reads them from saved, as autograd reads the
    // tensors a forward saved)
    uint8_t* sv = static_cast<uint8_t*>(saved);
    pack_block(pack_job(pk, sv + L.off_bt, kf, out), lin.B, r, 0, 0, r, static_cast<int>(out), 1, 1.0f);
    pack_block(pack_job(pk, sv + L.off_af, kf, in), lin.A, in, 0, 0, r, static_cast<int>(in), 0, s);
  }
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
  g.p.pdl_seg = 1;   // segments from 1 on read the previous kernel's rank-r output
  g.finish();
  g.split_tail(sk);
  if (!g.ok) return LORA_ERR_CUDA;
  return launch_gemm(kBigKK, g.p, LORA_KIND_PROJ, stream);
}

extern "C" lora_status_t lora_linear_forward(int64_t M, int64_t in, int64_t out, int r, float s, const void* x,
                                             lora_linear_t lin, void* y, void* saved, void* ws, size_t ws_bytes,
                                             cudaStream_t stream) {
  NvtxRange nvtx_range("lora_linear_forward");
  return linear_forward_impl(M, in, out, r, s, x, lin, y, saved, ws, ws_bytes, stream, true);
}

lora_status_t lgb::linear_forward_whole_tiles(int64_t M, int64_t in, int64_t out, int r, float s, const void* x,
                                              lora_linear_t lin, void* y, void* ws, size_t ws_bytes,
                                              cudaStream_t stream) {
  return linear_forward_impl(M, in, out, r, s, x, lin, y, nullptr, ws, ws_bytes, stream, false);
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
  // the adapter operands come packed from the forward (saved)
  const bf16* bt = reinterpret_cast<const bf16*>(static_cast<const uint8_t*>(saved) + L.off_bt);
  const bf16* af = reinterpret_cast<const bf16*>(static_cast<const uint8_t*>(saved) + L.off_af);
  bf16* U = c.take_n<bf16>(M * kf);
  float* part = c.take_n<float>(rank_projection_part(M, kf, ceil_div(out, kBK)));
  Deferred dr;
  defer_init(dr, c.take_n<float>(token_grad_part(M, kf, &out, 1) + token_grad_part(M, kf, &in, 1)));
  const SkRegion sk = carve_sk(c, pair_tiles(M, in));
  const bf16* T = static_cast<const bf16*>(saved);

  const ProjSeg ps = {dy, bt, out};
  LGB_TRY(rank_projection(M, kf, &ps, 1, U, part, status, stream));

  GemmPlan g(kBigKMN);
  GroupDesc& G = g.group(static_cast<int>(M), static_cast<int>(in), EPI_STORE, false);
  GemmPlan::seg(G, g.a_kmajor(dy, M, out, out), g.b_mnmajor(lin.W, in, out, in), -1, out, out);
  GemmPlan::seg(G, g.a_kmajor(U, M, kf, kf), g.b_mnmajor(af, in, kf, in), -1, kf, r);
  G.out0 = dx;
  G.ldo = in;
  g.p.status = status;
  g.p.pdl_seg = 1;   // segments from 1 on read the previous kernel's rank-r output
  g.finish();
  g.split_tail(sk);
  if (!g.ok) return LORA_ERR_CUDA;
  LGB_TRY(launch_gemm(kBigKMN, g.p, LORA_KIND_DGRAD, stream));

  // dB = s dy^T T and dA = s U^T x (one launch) read nothing the dx GEMM writes
  const GradJob jobs[2] = {{dy, out, 0, grads.dB, 0, T}, {x, in, 0, grads.dA, 1, U}};
  LGB_TRY(token_grads(M, r, kf, s, jobs, 2, dr, status, stream, 0, true));
  return defer_flush(dr, stream);
}
