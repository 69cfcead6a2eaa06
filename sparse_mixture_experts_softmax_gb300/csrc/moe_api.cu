// C ABI of the MoE layer: validation, workspace layout and the launch
// sequence of forward, backward and the training step (course "Trainable MoE
// in CUDA", Part 7: host orchestration of the forward pass, the backward pass
// and one training step).  Every step runs in this library's kernels; there is
// no host-side arithmetic on tensors and no fallback path.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "../../include/moe.h"
#include "api_common.h"
#include "kernels.h"

using namespace moe;
using namespace moe::api;

namespace moe {
namespace api {

// Expert MLPs over the row segments of `r` (course Part 5): up-projection
// with bias + activation or the SwiGLU gate, then the down-projection.
moe_status experts_forward(const moe_config& c, const ExpertW& w, const ExpertRows& r,
                           cudaStream_t st) {
  // expert up-projection (+ activation)
  GemmArgs g = rows_gemm(c, r);
  g.ragged_k = false;
  g.a_kcontig = true;
  g.b_kcontig = true;
  g.M = r.M;
  g.N = c.F;
  g.A0 = r.xe;
  g.lda = c.D;
  g.K0 = c.D;
  g.B0 = w.w1;
  g.ldb = c.D;
  g.sBe = (long long)c.F * c.D;
  g.ldc = c.F;
  g.ld_aux = c.F;
  if (c.act == MOE_ACT_SWIGLU && c.dtype == MOE_BF16) {
    // one launch: W1 and W3 tiles side by side in a 2 x 128-column accumulator
    g.epi = EPI_SWIGLU_UP;
    g.B0x = w.w3;
    g.out1 = r.h1;
    g.out2 = r.h3;
    g.C = r.a;
    KL("gemm_up", run_gemm(c, g, st, r.f32x3, r.f32x3_bytes));
  } else if (c.act == MOE_ACT_SWIGLU) {
    g.epi = EPI_STORE;
    g.C = r.h1;
    KL("gemm_up", run_gemm(c, g, st, r.f32x3, r.f32x3_bytes));
    g.B0 = w.w3;
    g.epi = EPI_SWIGLU_FWD;
    g.aux0 = r.h1;
    g.out1 = r.h3;
    g.C = r.a;
    KL("gemm_up_w3", run_gemm(c, g, st, r.f32x3, r.f32x3_bytes));
  } else {
    g.epi = EPI_ACT_FWD;
    g.bias = w.b1;
    g.out1 = r.h1;
    g.C = r.a;
    KL("gemm_up", run_gemm(c, g, st, r.f32x3, r.f32x3_bytes));
  }
  // expert down-projection (+ bias)
  GemmArgs d = rows_gemm(c, r);
  d.ragged_k = false;
  d.a_kcontig = true;
  d.b_kcontig = true;
  d.M = r.M;
  d.N = c.D;
  d.A0 = r.a;
  d.lda = c.F;
  d.K0 = c.F;
  d.B0 = w.w2;
  d.ldb = c.F;
  d.sBe = (long long)c.D * c.F;
  d.ldc = c.D;
  d.epi = EPI_STORE;
  d.bias = w.b2;
  d.C = r.ye;
  KL("gemm_down", run_gemm(c, d, st, r.f32x3, r.f32x3_bytes));

  return MOE_OK;
}

// Backward of the expert MLPs over the row segments of `r` given dYe: dA with
// the activation backward, dW2 (+ SGD), db2, dXe, dW1 / dW3 (+ SGD), db1.
moe_status experts_backward(const moe_config& c, const ExpertW& w, const ExpertRows& r,
                            const moe_grads& gr, const SgdFuse* sgd, cudaStream_t st) {
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  // dA = dYe W2_e with the activation backward in the epilogue
  GemmArgs g = rows_gemm(c, r);
  g.ragged_k = false;
  g.a_kcontig = true;
  g.b_kcontig = false;
  g.M = r.M;
  g.N = c.F;
  g.A0 = r.dye;
  g.lda = c.D;
  g.K0 = c.D;
  g.B0 = w.w2;
  g.ldb = c.F;
  g.sBe = (long long)c.D * c.F;
  g.ldc = c.F;
  g.ld_aux = c.F;
  g.aux0 = r.h1;
  g.C = r.dh1;
  if (swiglu) {
    g.epi = EPI_SWIGLU_BWD;
    g.aux1 = r.h3;
    g.out1 = r.dh3;
  } else {
    g.epi = EPI_ACT_BWD;
  }
  KL("gemm_dA", run_gemm(c, g, st, r.f32x3, r.f32x3_bytes));
  // dW2_e = dYe_e^T A_e  (ragged K)
  GemmArgs w2g = rows_gemm(c, r);
  w2g.ragged_k = true;
  w2g.a_kcontig = false;
  w2g.b_kcontig = false;
  w2g.c_type = MOE_F32;
  w2g.M = c.D;
  w2g.N = c.F;
  w2g.A0 = r.dye;
  w2g.lda = c.D;
  w2g.B0 = r.a;
  w2g.ldb = c.F;
  w2g.K0 = r.M;
  w2g.C = gr.dw2;
  w2g.ldc = c.F;
  w2g.sCe = (long long)c.D * c.F;
  w2g.epi = EPI_STORE;
  if (sgd) {
    w2g.sgd_w = sgd->w2;
    w2g.sgd_wlp = sgd->w2_lp;
    w2g.sgd_lr = sgd->lr;
  }
  KL("gemm_dw2", run_gemm(c, w2g, st, r.f32x3, r.f32x3_bytes));
  if (gr.db2) KL("bias_grad", launch_segment_colsum(c.dtype, r.dye, r.offsets, r.E, c.D, gr.db2, st));
  // dXe = dH1 W1_e (+ dH3 W3_e)
  GemmArgs xg = rows_gemm(c, r);
  xg.ragged_k = false;
  xg.a_kcontig = true;
  xg.b_kcontig = false;
  xg.M = r.M;
  xg.N = c.D;
  xg.A0 = r.dh1;
  xg.lda = c.F;
  xg.K0 = c.F;
  xg.B0 = w.w1;
  xg.ldb = c.D;
  xg.sBe = (long long)c.F * c.D;
  if (swiglu) {
    xg.A1 = r.dh3;
    xg.B1 = w.w3;
    xg.K1 = c.F;
  }
  xg.ldc = c.D;
  xg.epi = EPI_STORE;
  xg.C = r.dxe;
  KL("gemm_dxe", run_gemm(c, xg, st, r.f32x3, r.f32x3_bytes));
  // dW1_e = dH1_e^T Xe_e (dW3 likewise)
  GemmArgs w1g = rows_gemm(c, r);
  w1g.ragged_k = true;
  w1g.a_kcontig = false;
  w1g.b_kcontig = false;
  w1g.c_type = MOE_F32;
  w1g.M = c.F;
  w1g.N = c.D;
  w1g.A0 = r.dh1;
  w1g.lda = c.F;
  w1g.B0 = r.xe;
  w1g.ldb = c.D;
  w1g.K0 = r.M;
  w1g.C = gr.dw1;
  w1g.ldc = c.D;
  w1g.sCe = (long long)c.F * c.D;
  w1g.epi = EPI_STORE;
  if (sgd) {
    w1g.sgd_w = sgd->w1;
    w1g.sgd_wlp = sgd->w1_lp;
    w1g.sgd_lr = sgd->lr;
  }
  KL("gemm_dw1", run_gemm(c, w1g, st, r.f32x3, r.f32x3_bytes));
  if (swiglu) {
    w1g.A0 = r.dh3;
    w1g.C = gr.dw3;
    if (sgd) {
      w1g.sgd_w = sgd->w3;
      w1g.sgd_wlp = sgd->w3_lp;
    }
    KL("gemm_dw3", run_gemm(c, w1g, st, r.f32x3, r.f32x3_bytes));
  }
  if (gr.db1) KL("bias_grad", launch_segment_colsum(c.dtype, r.dh1, r.offsets, r.E, c.F, gr.db1, st));
  return MOE_OK;
}

// Router and dispatch of the T tokens of `x` (course Parts 3 and 4): scores,
// top-k and gates, counts, offsets and slot maps, and the gather into the
// expert-major rows of the workspace.  Also clears the device status word.
moe_status route_tokens(const moe_config& c, const ExpertW& w, const void* x, const Ptrs& P,
                        cudaStream_t st) {
  const Layout& L = *P.L;
  const long long R = (long long)c.T * c.k;
  const RouterArgs ra = router_args(c, w.corr_bias);
  CK(cudaMemsetAsync(P.at<void>(L.status), 0, 16, st));
  if (c.dtype == MOE_BF16) {
    // logits = x W_g^T (+ logit bias) on the tensor cores, then selection
    KL("cast_wg", launch_cast_bf16(w.w_gate, P.at<void>(L.wg_lp), (long long)c.E * c.D, st));
    GemmArgs r{};
    r.a_type = r.b_type = MOE_BF16;
    r.c_type = MOE_F32;
    r.status = P.at<int>(L.status);
    r.ragged_k = false;
    r.b_kcontig = true;
    r.M = c.T;
    r.N = c.E;
    r.K0 = c.D;
    r.A0 = x;
    r.lda = c.D;
    r.B0 = P.at<void>(L.wg_lp);
    r.ldb = c.D;
    r.sBe = (long long)c.E * c.D;
    r.offsets = nullptr;
    r.E = 1;
    r.seg_len = c.T;
    r.C = P.at<void>(L.logits);
    r.ldc = c.E;
    r.bias = w.logit_bias;
    r.epi = EPI_STORE;
    KL("router_logits", launch_gemm_tc(r, st));
    KL("router_select", launch_router_select(P.at<float>(L.logits), ra, P.at<float>(L.scores),
                                             P.at<int>(L.idx), P.at<float>(L.gate),
                                             P.at<float>(L.psum), st));
  } else {
    KL("router_fwd", launch_router_fwd(c.dtype, x, w.w_gate, w.logit_bias, ra, P.at<float>(L.scores),
                                       P.at<int>(L.idx), P.at<float>(L.gate), P.at<float>(L.psum), st));
  }
  int* dbg = P.at<int>(L.status);
  KL("route_count", launch_route_count(P.at<int>(L.idx), R, c.E, P.at<int>(L.chunk), st, dbg));
  // with a capacity factor each expert keeps its first `cap` assignments in
  // token order; dropped ones get slot -1 and are skipped downstream
  const int cap = expert_capacity_rows(c.capacity_factor, c.T, c.k, c.E);
  KL("route_scan", launch_route_scan(P.at<int>(L.chunk), route_chunks(R), c.E, cap,
                                     P.at<int>(L.counts), P.at<int>(L.offsets), st));
  KL("route_scatter", launch_route_scatter(P.at<int>(L.idx), R, c.k, c.E, cap, P.at<int>(L.chunk),
                                           P.at<int>(L.offsets), P.at<int>(L.src_tok),
                                           P.at<int>(L.slot_of), st, dbg));
  KL("gather", launch_gather(c.dtype, x, P.at<int>(L.slot_of), c.T, c.k, c.D, P.at<void>(L.xe), st,
                             dbg));
  return MOE_OK;
}

// Router backward (course Parts 3 and 6): renormalisation and aux gradient
// to the scores, the score backward to dlogits, dW_g = dlogits^T x and
// dX = dlogits W_g + the expert rows of each token scattered back (+ extra_dx,
// a [T, D] block in the layer dtype, or nullptr).  Uses the gate gradients
// and the aux row the combine and the loss finalisation left in the
// workspace.
moe_status router_backward(const moe_config& c, const ExpertW& w, const void* x, float* dw_gate,
                           float* dx, const void* extra_dx, const Ptrs& P, cudaStream_t st) {
  const Layout& L = *P.L;
  // router: renormalisation + aux + score backward
  const RouterArgs ra = router_args(c);
  const bool lp = c.dtype == MOE_BF16;
  KL("router_bwd", launch_router_bwd(P.at<float>(L.scores), P.at<int>(L.idx), P.at<float>(L.gate),
                       P.at<float>(L.dgate), c.aux_alpha != 0.f ? P.at<float>(L.aux_row) : nullptr,
                       ra, P.at<float>(L.dlogits), lp ? P.at<void>(L.dl_lp) : nullptr, st,
                       P.at<int>(L.status)));
  if (lp) {
    // tensor-core router products: dW_g = dlogits^T x (split over token
    // chunks, fixed-order sum) and dX = dlogits W_g + scatter-back of dXe.
    // W_g's bf16 copy is the forward's, still in the workspace: the backward
    // runs with the forward's weights, and a training step updates W_g only
    // after the backward.
    const int S = dwg_splits(c);
    GemmArgs rg{};
    rg.a_type = rg.b_type = MOE_BF16;
    rg.c_type = MOE_F32;
    rg.status = P.at<int>(L.status);
    rg.ragged_k = true;
    rg.M = c.E;
    rg.N = c.D;
    rg.A0 = P.at<void>(L.dl_lp);
    rg.lda = c.E;
    rg.B0 = x;
    rg.ldb = c.D;
    rg.K0 = c.T;
    rg.offsets = nullptr;
    rg.E = S;
    rg.seg_len = (c.T + S - 1) / S;
    rg.C = P.at<void>(L.dwg_part);
    rg.ldc = c.D;
    rg.sCe = (long long)c.E * c.D;
    rg.epi = EPI_STORE;
    KL("gemm_router_dwg", launch_gemm_tc(rg, st));
    KL("router_dwg_sum", launch_sum_partials(P.at<float>(L.dwg_part), S, (long long)c.E * c.D,
                                             dw_gate, st));
    GemmArgs dg{};
    dg.a_type = dg.b_type = MOE_BF16;
    dg.c_type = MOE_F32;
    dg.status = P.at<int>(L.status);
    dg.ragged_k = false;
    dg.b_kcontig = false;
    dg.M = c.T;
    dg.N = c.D;
    dg.K0 = c.E;
    dg.A0 = P.at<void>(L.dl_lp);
    dg.lda = c.E;
    dg.B0 = P.at<void>(L.wg_lp);
    dg.ldb = c.D;
    dg.sBe = (long long)c.E * c.D;
    dg.offsets = nullptr;
    dg.E = 1;
    dg.seg_len = c.T;
    dg.C = dx;
    dg.ldc = c.D;
    dg.epi = EPI_STORE;
    KL("gemm_router_dx", launch_gemm_tc(dg, st));
    KL("scatter_back", launch_scatter_back_add(c.dtype, dx, P.at<void>(L.dxe), P.at<int>(L.slot_of),
                                               c.T, c.D, c.k, extra_dx, st, P.at<int>(L.status)));
    return MOE_OK;
  }
  // dW_g = dlogits^T x (split over token chunks, then a fixed-order sum)
  const int S = dwg_splits(c);
  GemmArgs rg{};
  rg.a_type = MOE_F32;
  rg.b_type = c.dtype;
  rg.c_type = MOE_F32;
  rg.ragged_k = true;
  rg.a_kcontig = false;
  rg.b_kcontig = false;
  rg.M = c.E;
  rg.N = c.D;
  rg.A0 = P.at<void>(L.dlogits);
  rg.lda = c.E;
  rg.B0 = x;
  rg.ldb = c.D;
  rg.K0 = c.T;
  rg.offsets = nullptr;
  rg.E = S;
  rg.seg_len = (c.T + S - 1) / S;
  rg.C = P.at<void>(L.dwg_part);
  rg.ldc = c.D;
  rg.sCe = (long long)c.E * c.D;
  rg.epi = EPI_STORE;
  KL("gemm_router_dwg", launch_gemm_simt(rg, st));
  KL("router_dwg_sum", launch_sum_partials(P.at<float>(L.dwg_part), S, (long long)c.E * c.D, dw_gate, st));
  // dX = dlogits W_g, then each token's expert rows added in j order (the
  // HBM-bound scatter-back pass)
  GemmArgs dg{};
  dg.a_type = MOE_F32;
  dg.b_type = MOE_F32;
  dg.c_type = MOE_F32;
  dg.ragged_k = false;
  dg.a_kcontig = true;
  dg.b_kcontig = false;
  dg.M = c.T;
  dg.N = c.D;
  dg.A0 = P.at<void>(L.dlogits);
  dg.lda = c.E;
  dg.K0 = c.E;
  dg.B0 = w.w_gate;
  dg.ldb = c.D;
  dg.sBe = 0;
  dg.offsets = nullptr;
  dg.E = 1;
  dg.seg_len = c.T;
  dg.C = dx;
  dg.ldc = c.D;
  dg.epi = EPI_STORE;
  dg.status = P.at<int>(L.status);
  KL("gemm_router_dx", launch_gemm_simt(dg, st));
  KL("scatter_back", launch_scatter_back_add(c.dtype, dx, P.at<void>(L.dxe), P.at<int>(L.slot_of),
                                             c.T, c.D, c.k, extra_dx, st, P.at<int>(L.status)));
  return MOE_OK;
}

}  // namespace api
}  // namespace moe

namespace {

// The expert-major row buffers of the single-device step (all E experts).
ExpertRows expert_rows(const moe_config& c, const Ptrs& P) {
  const Layout& L = *P.L;
  ExpertRows r{};
  r.E = c.E;
  r.M = (int)((long long)c.T * c.k);
  r.offsets = P.at<int>(L.offsets);
  r.status = P.at<int>(L.status);
  r.xe = P.at<void>(L.xe);
  r.h1 = P.at<void>(L.h1);
  r.h3 = L.h3 ? P.at<void>(L.h3) : nullptr;
  r.a = P.at<void>(L.a);
  r.ye = P.at<void>(L.ye);
  r.dye = P.at<void>(L.dye);
  r.dh1 = P.at<void>(L.dh1);
  r.dh3 = L.dh3 ? P.at<void>(L.dh3) : nullptr;
  r.dxe = P.at<void>(L.dxe);
  r.f32x3 = L.f32x3_bytes ? P.at<void>(L.f32x3) : nullptr;
  r.f32x3_bytes = L.f32x3_bytes;
  return r;
}

// Forward: router -> dispatch -> experts -> combine.  With a target, combine
// also forms dY and the squared-error partials, and the losses are finalised.
// target_ready: recorded when `target` has landed (its copy may still be in
// flight on another stream while the router and experts run), or nullptr.
moe_status run_forward(const moe_config& c, const ExpertW& w, const void* x, float* y,
                       const float* target, float* d_loss, const Ptrs& P, cudaStream_t st,
                       cudaEvent_t target_ready = nullptr) {
  const Layout& L = *P.L;
  RET_IF(route_tokens(c, w, x, P, st));

  RET_IF(experts_forward(c, w, expert_rows(c, P), st));

  const bool shared = c.n_shared > 0;
  if (shared) {
    // shared experts: one SwiGLU branch over all T tokens (a single segment)
    const int Fs = c.n_shared * c.F;
    GemmArgs su = gemm_base(c, P);
    su.offsets = nullptr;
    su.E = 1;
    su.seg_len = c.T;
    su.ragged_k = false;
    su.a_kcontig = true;
    su.b_kcontig = true;
    su.M = c.T;
    su.N = Fs;
    su.A0 = x;
    su.lda = c.D;
    su.K0 = c.D;
    su.B0 = w.ws1;
    su.B0x = w.ws3;
    su.ldb = c.D;
    su.sBe = (long long)Fs * c.D;
    su.ldc = Fs;
    su.ld_aux = Fs;
    su.epi = EPI_SWIGLU_UP;
    su.out1 = P.at<void>(L.hs1);
    su.out2 = P.at<void>(L.hs3);
    su.C = P.at<void>(L.as);
    KL("gemm_shared_up", run_gemm(c, su, st));
    GemmArgs sd = gemm_base(c, P);
    sd.offsets = nullptr;
    sd.E = 1;
    sd.seg_len = c.T;
    sd.ragged_k = false;
    sd.a_kcontig = true;
    sd.b_kcontig = true;
    sd.M = c.T;
    sd.N = c.D;
    sd.A0 = P.at<void>(L.as);
    sd.lda = Fs;
    sd.K0 = Fs;
    sd.B0 = w.ws2;
    sd.ldb = Fs;
    sd.sBe = (long long)c.D * Fs;
    sd.ldc = c.D;
    sd.epi = EPI_STORE;
    sd.C = P.at<void>(L.ys);
    KL("gemm_shared_down", run_gemm(c, sd, st));
  }
  const void* ys = shared ? P.at<void>(L.ys) : nullptr;

  const bool train = target != nullptr;
  if (target_ready != nullptr) CK(cudaStreamWaitEvent(st, target_ready, 0));
  if (train && y == nullptr && c.k <= 8) {
    // training step: the combine backward runs in the same pass (dYe, dgate)
    KL("combine_fused", launch_combine_train(c.dtype, P.at<void>(L.ye), P.at<float>(L.gate),
                                             P.at<int>(L.slot_of), c.T, c.D, c.k, ys, target,
                                             P.at<double>(L.sq), P.at<void>(L.dye),
                                             P.at<float>(L.dgate),
                                             shared ? P.at<void>(L.dy_lp) : nullptr, st, 0.f,
                                             P.at<int>(L.status)));
  } else {
    KL("combine_loss", launch_combine(c.dtype, P.at<void>(L.ye), P.at<float>(L.gate), P.at<int>(L.slot_of), c.T,
                      c.D, c.k, ys, y, target, train ? P.at<float>(L.dy) : nullptr,
                      train ? P.at<double>(L.sq) : nullptr, st, 0.f, P.at<int>(L.status)));
  }
  if (train)
    KL("finalize_losses", launch_finalize_losses(P.at<double>(L.sq), combine_blocks(c.T), P.at<float>(L.psum),
                              router_fwd_blocks(c.T), P.at<int>(L.counts), c.T, c.D, c.E, c.k,
                              c.aux_alpha, d_loss, P.at<float>(L.aux_row), st));
  return MOE_OK;
}


// Backward of L = L_task + alpha aux given dY (course Parts 4-6).
// dy == nullptr: the forward's fused combine already wrote dYe and dgate.
moe_status run_backward(const moe_config& c, const ExpertW& w, const void* x, const float* dy,
                        const moe_grads& gr, float* dx, bool aux_ready, const Ptrs& P,
                        cudaStream_t st, const SgdFuse* sgd = nullptr) {
  const Layout& L = *P.L;
  if (!aux_ready)
    KL("finalize_losses", launch_finalize_losses(P.at<double>(L.sq), 0, P.at<float>(L.psum), router_fwd_blocks(c.T),
                              P.at<int>(L.counts), c.T, c.D, c.E, c.k, c.aux_alpha, nullptr,
                              P.at<float>(L.aux_row), st));
  if (dy != nullptr)
    KL("combine_bwd", launch_combine_bwd(c.dtype, dy, P.at<void>(L.ye), P.at<float>(L.gate), P.at<int>(L.slot_of),
                          c.T, c.D, c.k, P.at<void>(L.dye), P.at<float>(L.dgate), st,
                          P.at<int>(L.status)));
  RET_IF(experts_backward(c, w, expert_rows(c, P), gr, sgd, st));

  if (c.n_shared > 0) {
    // shared branch: it receives the whole dY (bf16 copy for the tensor cores)
    const int Fs = c.n_shared * c.F;
    void* dyl = P.at<void>(L.dy_lp);
    if (dy != nullptr) KL("cast_dy", launch_cast_bf16(dy, dyl, (long long)c.T * c.D, st));
    auto one_segment = [&](GemmArgs& q) {
      q.offsets = nullptr;
      q.E = 1;
      q.seg_len = c.T;
    };
    // dA_s = dY Ws2 with the SwiGLU backward in the epilogue
    GemmArgs sa = gemm_base(c, P);
    one_segment(sa);
    sa.ragged_k = false;
    sa.a_kcontig = true;
    sa.b_kcontig = false;
    sa.M = c.T;
    sa.N = Fs;
    sa.A0 = dyl;
    sa.lda = c.D;
    sa.K0 = c.D;
    sa.B0 = w.ws2;
    sa.ldb = Fs;
    sa.sBe = (long long)c.D * Fs;
    sa.ldc = Fs;
    sa.ld_aux = Fs;
    sa.aux0 = P.at<void>(L.hs1);
    sa.aux1 = P.at<void>(L.hs3);
    sa.C = P.at<void>(L.dhs1);
    sa.out1 = P.at<void>(L.dhs3);
    sa.epi = EPI_SWIGLU_BWD;
    KL("gemm_shared_dA", run_gemm(c, sa, st));
    // dWs2 = dY^T As over the T rows (SGD fused in a training step)
    GemmArgs s2 = gemm_base(c, P);
    one_segment(s2);
    s2.ragged_k = true;
    s2.a_kcontig = false;
    s2.b_kcontig = false;
    s2.c_type = MOE_F32;
    s2.M = c.D;
    s2.N = Fs;
    s2.A0 = dyl;
    s2.lda = c.D;
    s2.B0 = P.at<void>(L.as);
    s2.ldb = Fs;
    s2.K0 = c.T;
    s2.C = gr.dws2;
    s2.ldc = Fs;
    s2.sCe = (long long)c.D * Fs;
    s2.epi = EPI_STORE;
    if (sgd) {
      s2.sgd_w = sgd->ws2;
      s2.sgd_wlp = sgd->ws2_lp;
      s2.sgd_lr = sgd->lr;
    }
    KL("gemm_shared_dw2", run_gemm(c, s2, st));
    // dXs = dH1s Ws1 + dH3s Ws3 (added to dX by the scatter-back)
    GemmArgs sx = gemm_base(c, P);
    one_segment(sx);
    sx.ragged_k = false;
    sx.a_kcontig = true;
    sx.b_kcontig = false;
    sx.M = c.T;
    sx.N = c.D;
    sx.A0 = P.at<void>(L.dhs1);
    sx.lda = Fs;
    sx.K0 = Fs;
    sx.B0 = w.ws1;
    sx.ldb = c.D;
    sx.sBe = (long long)Fs * c.D;
    sx.A1 = P.at<void>(L.dhs3);
    sx.B1 = w.ws3;
    sx.K1 = Fs;
    sx.ldc = c.D;
    sx.epi = EPI_STORE;
    sx.C = P.at<void>(L.dxs);
    KL("gemm_shared_dx", run_gemm(c, sx, st));
    // dWs1 = dH1s^T x, dWs3 = dH3s^T x (SGD fused in a training step)
    GemmArgs s1 = gemm_base(c, P);
    one_segment(s1);
    s1.ragged_k = true;
    s1.a_kcontig = false;
    s1.b_kcontig = false;
    s1.c_type = MOE_F32;
    s1.M = Fs;
    s1.N = c.D;
    s1.A0 = P.at<void>(L.dhs1);
    s1.lda = Fs;
    s1.B0 = x;
    s1.ldb = c.D;
    s1.K0 = c.T;
    s1.C = gr.dws1;
    s1.ldc = c.D;
    s1.sCe = (long long)Fs * c.D;
    s1.epi = EPI_STORE;
    if (sgd) {
      s1.sgd_w = sgd->ws1;
      s1.sgd_wlp = sgd->ws1_lp;
      s1.sgd_lr = sgd->lr;
    }
    KL("gemm_shared_dw1", run_gemm(c, s1, st));
    s1.A0 = P.at<void>(L.dhs3);
    s1.C = gr.dws3;
    if (sgd) {
      s1.sgd_w = sgd->ws3;
      s1.sgd_wlp = sgd->ws3_lp;
    }
    KL("gemm_shared_dw3", run_gemm(c, s1, st));
  }

  return router_backward(c, w, x, gr.dw_gate, dx, c.n_shared > 0 ? P.at<void>(L.dxs) : nullptr,
                         P, st);
}

moe_status check_ws(const moe_config& c, const void* ws, size_t bytes) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_ALIGNMENT;
  if (bytes < make_layout(c).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

moe_status check_weights(const moe_config& c, const ExpertW& w) {
  if (!w.w_gate || !w.w1 || !w.w2) return MOE_ERR_INVALID_ARG;
  if (c.act == MOE_ACT_SWIGLU && !w.w3) return MOE_ERR_INVALID_ARG;
  if (c.has_bias && (!w.b1 || !w.b2)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (!w.ws1 || !w.ws3 || !w.ws2)) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {w.w_gate, w.w1, w.w3, w.w2, w.b1, w.b2, w.logit_bias, w.corr_bias,
                      w.ws1, w.ws3, w.ws2};
  for (const void* p : ps)
    if (p && !aligned16(p)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

moe_status check_grads(const moe_config& c, const moe_grads& g) {
  if (!g.dw_gate || !g.dw1 || !g.dw2) return MOE_ERR_INVALID_ARG;
  if (c.act == MOE_ACT_SWIGLU && !g.dw3) return MOE_ERR_INVALID_ARG;
  if (c.has_bias && (!g.db1 || !g.db2)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (!g.dws1 || !g.dws3 || !g.dws2)) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {g.dw_gate, g.dw1, g.dw3, g.dw2, g.db1, g.db2, g.dws1, g.dws3, g.dws2};
  for (const void* p : ps)
    if (p && !aligned16(p)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

// Zeroes every gradient buffer that is given (NULL ones are skipped).
moe_status zero_grads(const moe_config& c, const moe_grads& g, cudaStream_t st) {
  const size_t E = c.E, D = c.D, F = c.F;
  const size_t Fs = (size_t)c.n_shared * F;
  struct Z { float* p; size_t bytes; } zs[] = {
      {g.dw_gate, E * D * 4}, {g.dw1, E * F * D * 4}, {g.dw3, E * F * D * 4},
      {g.dw2, E * D * F * 4}, {g.db1, E * F * 4},     {g.db2, E * D * 4},
      {g.dws1, Fs * D * 4},   {g.dws3, Fs * D * 4},   {g.dws2, D * Fs * 4}};
  for (const Z& z : zs)
    if (z.p && z.bytes) CK(launch_fill_zero(z.p, z.bytes, st));
  return MOE_OK;
}

// The gradients a training step works with: the caller's buffers, and for
// each one left NULL a workspace stand-in, except the expert weights of bf16
// layers, whose fused SGD then stores no gradient at all.
moe_grads step_grads(const moe_config& c, const moe_grads& given, const Ptrs& P) {
  moe_grads g = given;
  const Layout& L = *P.L;
  if (!g.dw_gate) g.dw_gate = P.at<float>(L.g_wg);
  if (c.has_bias && !g.db1) g.db1 = P.at<float>(L.g_b1);
  if (c.has_bias && !g.db2) g.db2 = P.at<float>(L.g_b2);
  if (c.dtype != MOE_BF16) {
    if (!g.dw1) g.dw1 = P.at<float>(L.g_w1);
    if (c.act == MOE_ACT_SWIGLU && !g.dw3) g.dw3 = P.at<float>(L.g_w3);
    if (!g.dw2) g.dw2 = P.at<float>(L.g_w2);
  }
  return g;
}

moe_status train_step_impl(const moe_config* cfg, const moe_params* p, const void* x,
                           const float* y_target, float lr, float* d_loss, float* dx,
                           void* workspace, size_t workspace_bytes, cudaStream_t st,
                           cudaEvent_t target_ready = nullptr) {
  RET_IF(validate_config(cfg));
  const moe_config& c = *cfg;
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  RET_IF(check_ws(c, workspace, workspace_bytes));
  if (!p->w_gate || !p->w1 || !p->w2 || (c.act == MOE_ACT_SWIGLU && !p->w3))
    return MOE_ERR_INVALID_ARG;
  if (c.has_bias && (!p->b1 || !p->b2)) return MOE_ERR_INVALID_ARG;
  if (c.dtype == MOE_BF16 && (!p->w1_lp || !p->w2_lp || (c.act == MOE_ACT_SWIGLU && !p->w3_lp)))
    return MOE_ERR_INVALID_ARG;
  if (c.n_shared > 0 && (!p->ws1 || !p->ws3 || !p->ws2 || !p->ws1_lp || !p->ws3_lp || !p->ws2_lp))
    return MOE_ERR_INVALID_ARG;
  // gradient buffers are optional here (NULL: the step still applies that
  // gradient, it just does not hand it out); those given must be aligned
  const moe_grads& gv = p->grads;
  const void* ps[] = {p->w_gate, p->w1, p->w3, p->w2, p->b1, p->b2, p->w1_lp, p->w3_lp, p->w2_lp,
                      p->logit_bias, p->corr_bias, p->ws1, p->ws3, p->ws2, p->ws1_lp,
                      p->ws3_lp, p->ws2_lp, x, y_target, d_loss, dx,
                      gv.dw_gate, gv.dw1, gv.dw3, gv.dw2, gv.db1, gv.db2, gv.dws1, gv.dws3,
                      gv.dws2};
  for (const void* q : ps)
    if (q && !aligned16(q)) return MOE_ERR_ALIGNMENT;
  if (c.T > 0 && (!x || !y_target)) return MOE_ERR_INVALID_ARG;
  if (!d_loss) return MOE_ERR_INVALID_ARG;
  RET_IF(check_device());

  Layout L = make_layout(c);
  Ptrs P{static_cast<char*>(workspace), &L};
  if (c.T == 0) {
    CK(cudaMemsetAsync(d_loss, 0, 2 * sizeof(float), st));
    return zero_grads(c, p->grads, st);
  }
  ExpertW w;
  w.w_gate = p->w_gate;
  w.w1 = c.dtype == MOE_BF16 ? p->w1_lp : p->w1;
  w.w3 = c.dtype == MOE_BF16 ? p->w3_lp : p->w3;
  w.w2 = c.dtype == MOE_BF16 ? p->w2_lp : p->w2;
  w.b1 = p->b1;
  w.b2 = p->b2;
  w.logit_bias = p->logit_bias;
  w.corr_bias = p->corr_bias;
  w.ws1 = p->ws1_lp;   // the shared branch exists only for bf16 layers
  w.ws3 = p->ws3_lp;
  w.ws2 = p->ws2_lp;
  RET_IF(run_forward(c, w, x, nullptr, y_target, d_loss, P, st, target_ready));
  float* dxp = dx ? dx : P.at<float>(L.dx);
  // bf16 layers: the expert weights' SGD runs inside the dW GEMM epilogues
  const bool fused = c.dtype == MOE_BF16;
  const SgdFuse sf{lr, p->w1, p->w3, p->w2, p->w1_lp, p->w3_lp, p->w2_lp,
                   p->ws1, p->ws3, p->ws2, p->ws1_lp, p->ws3_lp, p->ws2_lp};
  const moe_grads g = step_grads(c, p->grads, P);
  // k <= 8: the forward's combine pass already produced dYe and dgate
  RET_IF(run_backward(c, w, x, c.k <= 8 ? nullptr : P.at<float>(L.dy), g, dxp, true, P, st,
                      fused ? &sf : nullptr));
  // SGD on the fp32 masters; bf16 working copies rewritten from the result
  const long long E = c.E, D = c.D, F = c.F;
  // one launch for every tensor the GEMM epilogues did not update
  SgdTensor ts[SGD_MAX_TENSORS];
  int nt = 0;
  ts[nt++] = {p->w_gate, g.dw_gate, E * D, nullptr};
  if (!fused) {
    ts[nt++] = {p->w1, g.dw1, E * F * D, nullptr};
    if (c.act == MOE_ACT_SWIGLU) ts[nt++] = {p->w3, g.dw3, E * F * D, nullptr};
    ts[nt++] = {p->w2, g.dw2, E * D * F, nullptr};
  }
  if (c.has_bias) {
    ts[nt++] = {p->b1, g.db1, E * F, nullptr};
    ts[nt++] = {p->b2, g.db2, E * D, nullptr};
  }
  KL("sgd", launch_sgd(ts, nt, lr, st));
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_size(const moe_config* cfg) {
  if (validate_config(cfg) != MOE_OK) return 0;
  return make_layout(*cfg).total;
}

moe_status moe_forward(const moe_config* cfg, const moe_weights* w, const void* x, float* y,
                       void* workspace, size_t workspace_bytes, void* stream) {
  g_launches = 0;
  RET_IF(validate_config(cfg));
  const moe_config& c = *cfg;
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  ExpertW ew{w->w_gate, w->w1, w->w3, w->w2, w->b1, w->b2, w->logit_bias, w->corr_bias,
             w->ws1, w->ws3, w->ws2};
  RET_IF(check_weights(c, ew));
  RET_IF(check_ws(c, workspace, workspace_bytes));
  if (c.T > 0 && (!x || !y)) return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (y && !aligned16(y))) return MOE_ERR_ALIGNMENT;
  RET_IF(check_device());
  if (c.T == 0) return MOE_OK;
  Layout L = make_layout(c);
  Ptrs P{static_cast<char*>(workspace), &L};
  return run_forward(c, ew, x, y, nullptr, nullptr, P, static_cast<cudaStream_t>(stream));
}

moe_status moe_backward(const moe_config* cfg, const moe_weights* w, const void* x,
                        const float* dy, const moe_grads* g, float* dx, void* workspace,
                        size_t workspace_bytes, void* stream) {
  g_launches = 0;
  RET_IF(validate_config(cfg));
  const moe_config& c = *cfg;
  if (w == nullptr || g == nullptr) return MOE_ERR_INVALID_ARG;
  ExpertW ew{w->w_gate, w->w1, w->w3, w->w2, w->b1, w->b2, w->logit_bias, w->corr_bias,
             w->ws1, w->ws3, w->ws2};
  RET_IF(check_weights(c, ew));
  RET_IF(check_grads(c, *g));
  RET_IF(check_ws(c, workspace, workspace_bytes));
  if (c.T > 0 && (!x || !dy)) return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (dy && !aligned16(dy)) || (dx && !aligned16(dx)))
    return MOE_ERR_ALIGNMENT;
  RET_IF(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) return zero_grads(c, *g, st);
  Layout L = make_layout(c);
  Ptrs P{static_cast<char*>(workspace), &L};
  float* dxp = dx ? dx : P.at<float>(L.dx);
  return run_backward(c, ew, x, dy, *g, dxp, false, P, st);
}

moe_status moe_train_step(const moe_config* cfg, const moe_params* p, const void* x,
                          const float* y_target, float lr, float* d_loss, float* dx,
                          void* workspace, size_t workspace_bytes, void* stream) {
  g_launches = 0;
  return train_step_impl(cfg, p, x, y_target, lr, d_loss, dx, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream));
}

size_t moe_host_staging_size(const moe_config* cfg) {
  if (validate_config(cfg) != MOE_OK) return 0;
  const size_t n = (size_t)cfg->T * cfg->D;
  return align_up(n * esize(cfg->dtype)) + align_up(n * 4) + kAlign;
}

// Per device: a side stream for host-to-device copies and its events (the
// copy may start / the copy is done; per input slot: landed / consumed),
// created on first use.  `busy` serialises the host entry points of one
// device, which share these.
struct HostCopyLane {
  bool ready = false;
  std::mutex busy;
  cudaStream_t side = nullptr;
  cudaEvent_t go = nullptr, done = nullptr;
  cudaEvent_t copied[2] = {nullptr, nullptr};     // inputs of a slot have landed
  cudaEvent_t consumed[2] = {nullptr, nullptr};   // the step using a slot is done
};
moe_status host_copy_lane(HostCopyLane** out) {
  static std::mutex mu;
  static HostCopyLane lanes[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  HostCopyLane& l = lanes[dev];
  if (!l.ready) {
    // create everything, and publish the lane only when all of it exists
    cudaStream_t side = nullptr;
    cudaEvent_t ev[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    bool ok = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; i < 6 && ok; ++i)
      ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      for (cudaEvent_t e : ev)
        if (e) cudaEventDestroy(e);
      if (side) cudaStreamDestroy(side);
      return MOE_ERR_CUDA;
    }
    l.side = side;
    l.go = ev[0];
    l.done = ev[1];
    l.copied[0] = ev[2];
    l.copied[1] = ev[3];
    l.consumed[0] = ev[4];
    l.consumed[1] = ev[5];
    l.ready = true;
  }
  *out = &l;
  return MOE_OK;
}

moe_status moe_train_step_host(const moe_config* cfg, const moe_params* p, const void* x_host,
                               const float* y_target_host, float lr, float* loss_host,
                               void* staging, size_t staging_bytes, void* workspace,
                               size_t workspace_bytes, void* stream) {
  g_launches = 0;
  RET_IF(validate_config(cfg));
  const moe_config& c = *cfg;
  if (!staging || !loss_host || (c.T > 0 && (!x_host || !y_target_host)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(staging)) return MOE_ERR_ALIGNMENT;
  if (staging_bytes < moe_host_staging_size(cfg)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t n = (size_t)c.T * c.D;
  char* sbase = static_cast<char*>(staging);
  void* xd = sbase;
  float* td = reinterpret_cast<float*>(sbase + align_up(n * esize(c.dtype)));
  float* ld = reinterpret_cast<float*>(sbase + align_up(n * esize(c.dtype)) + align_up(n * 4));
  RET_IF(check_device());
  HostCopyLane* lane = nullptr;
  RET_IF(host_copy_lane(&lane));
  std::lock_guard<std::mutex> hold(lane->busy);
  // every return from here on waits for the copies issued so far: the
  // caller's host buffers must outlive them, also on an error
  auto finish = [&](moe_status s) {
    cudaStreamSynchronize(lane->side);
    if (cudaStreamSynchronize(st) != cudaSuccess && s == MOE_OK) s = MOE_ERR_CUDA;
    return s;
  };
  // x goes first on the step's stream; the target (needed only from the
  // combine on) is copied on a side stream while the router and the expert
  // GEMMs run, and the step's stream waits for it just before the combine
  cudaEvent_t target_ready = nullptr;
  if (n > 0) {
    // earlier work on `st` is done with the staging before the side copy starts
    if (cudaEventRecord(lane->go, st) != cudaSuccess ||
        cudaStreamWaitEvent(lane->side, lane->go, 0) != cudaSuccess ||
        cudaMemcpyAsync(xd, x_host, n * esize(c.dtype), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(td, y_target_host, n * 4, cudaMemcpyHostToDevice, lane->side) !=
            cudaSuccess ||
        cudaEventRecord(lane->done, lane->side) != cudaSuccess)
      return finish(MOE_ERR_CUDA);
    target_ready = lane->done;
  }
  moe_status s = train_step_impl(cfg, p, xd, td, lr, ld, nullptr, workspace, workspace_bytes, st,
                                 target_ready);
  if (s != MOE_OK) return finish(s);
  if (cudaMemcpyAsync(loss_host, ld, 2 * sizeof(float), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return finish(MOE_ERR_CUDA);
  return finish(MOE_OK);
}

moe_status moe_train_steps_host(const moe_config* cfg, const moe_params* p, int32_t n_steps,
                                const void* const* x_hosts, const float* const* y_target_hosts,
                                float lr, float* loss_host, void* staging, size_t staging_bytes,
                                void* workspace, size_t workspace_bytes, void* stream) {
  g_launches = 0;
  RET_IF(validate_config(cfg));
  const moe_config& c = *cfg;
  if (n_steps < 0 || !staging || !loss_host || (n_steps > 0 && (!x_hosts || !y_target_hosts)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(staging)) return MOE_ERR_ALIGNMENT;
  const size_t slot_bytes = moe_host_staging_size(cfg);
  if (staging_bytes < 2 * slot_bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const size_t n = (size_t)c.T * c.D;
  for (int i = 0; i < n_steps; ++i)
    if (n > 0 && (!x_hosts[i] || !y_target_hosts[i])) return MOE_ERR_INVALID_ARG;
  if (n_steps == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RET_IF(check_device());
  HostCopyLane* lane = nullptr;
  RET_IF(host_copy_lane(&lane));
  std::lock_guard<std::mutex> hold(lane->busy);
  char* sbase = static_cast<char*>(staging);
  auto slot_x = [&](int q) -> void* { return sbase + q * slot_bytes; };
  auto slot_t = [&](int q) {
    return reinterpret_cast<float*>(sbase + q * slot_bytes + align_up(n * esize(c.dtype)));
  };
  auto slot_l = [&](int q) {
    return reinterpret_cast<float*>(sbase + q * slot_bytes + align_up(n * esize(c.dtype)) +
                                    align_up(n * 4));
  };
  auto upload = [&](int i) -> moe_status {   // step i's batch into slot i % 2 (side stream)
    const int q = i & 1;
    CK(cudaStreamWaitEvent(lane->side, lane->consumed[q], 0));
    if (n > 0) {
      CK(cudaMemcpyAsync(slot_x(q), x_hosts[i], n * esize(c.dtype), cudaMemcpyHostToDevice,
                         lane->side));
      CK(cudaMemcpyAsync(slot_t(q), y_target_hosts[i], n * 4, cudaMemcpyHostToDevice,
                         lane->side));
    }
    CK(cudaEventRecord(lane->copied[q], lane->side));
    return MOE_OK;
  };
  // both slots are free once the work already queued on `stream` is done
  CK(cudaEventRecord(lane->consumed[0], st));
  CK(cudaEventRecord(lane->consumed[1], st));
  moe_status s = upload(0);
  for (int i = 0; i < n_steps && s == MOE_OK; ++i) {
    const int q = i & 1;
    if (i + 1 < n_steps) s = upload(i + 1);     // overlaps step i below
    if (s != MOE_OK) break;
    if (cudaStreamWaitEvent(st, lane->copied[q], 0) != cudaSuccess) { s = MOE_ERR_CUDA; break; }
    s = train_step_impl(cfg, p, slot_x(q), slot_t(q), lr, slot_l(q), nullptr, workspace,
                        workspace_bytes, st);   // launches accumulate over the steps
    if (s != MOE_OK) break;
    if (cudaMemcpyAsync(loss_host + 2 * (size_t)i, slot_l(q), 2 * sizeof(float),
                        cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaEventRecord(lane->consumed[q], st) != cudaSuccess)
      s = MOE_ERR_CUDA;
  }
  // the caller's host batches must outlive every copy, also on an early return
  cudaStreamSynchronize(lane->side);
  if (cudaStreamSynchronize(st) != cudaSuccess && s == MOE_OK) s = MOE_ERR_CUDA;
  return s;
}

moe_status moe_get_routing(const moe_config* cfg, const void* workspace, size_t workspace_bytes,
                           float* scores, int32_t* idx, float* gate, int32_t* counts,
                           int32_t* offsets, int32_t* src_tok, int32_t* slot_of, void* stream) {
  RET_IF(validate_config(cfg));
  const moe_config& c = *cfg;
  RET_IF(check_ws(c, workspace, workspace_bytes));
  Layout L = make_layout(c);
  const char* b = static_cast<const char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t T = c.T, E = c.E, R = (size_t)c.T * c.k;
  struct Cp { void* dst; size_t off; size_t bytes; } cps[] = {
      {scores, L.scores, T * E * 4}, {idx, L.idx, R * 4},       {gate, L.gate, R * 4},
      {counts, L.counts, E * 4},     {offsets, L.offsets, (E + 1) * 4},
      {src_tok, L.src_tok, R * 4},   {slot_of, L.slot_of, R * 4}};
  for (const Cp& cp : cps)
    if (cp.dst && cp.bytes)
      if (cudaMemcpyAsync(cp.dst, b + cp.off, cp.bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_get_intermediates(const moe_config* cfg, const void* workspace,
                                 size_t workspace_bytes, void* ye, void* dxe, float* dlogits,
                                 void* stream) {
  RET_IF(validate_config(cfg));
  const moe_config& c = *cfg;
  RET_IF(check_ws(c, workspace, workspace_bytes));
  Layout L = make_layout(c);
  const char* b = static_cast<const char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t R = (size_t)c.T * c.k, es = esize(c.dtype);
  struct Cp { void* dst; size_t off; size_t bytes; } cps[] = {
      {ye, L.ye, R * c.D * es}, {dxe, L.dxe, R * c.D * es}, {dlogits, L.dlogits, (size_t)c.T * c.E * 4}};
  for (const Cp& cp : cps)
    if (cp.dst && cp.bytes)
      if (cudaMemcpyAsync(cp.dst, b + cp.off, cp.bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_get_hidden(const moe_config* cfg, const void* workspace, size_t workspace_bytes,
                          void* h1, void* h3, void* stream) {
  RET_IF(validate_config(cfg));
  const moe_config& c = *cfg;
  RET_IF(check_ws(c, workspace, workspace_bytes));
  if (h3 != nullptr && c.act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  Layout L = make_layout(c);
  const char* b = static_cast<const char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)c.T * c.k * c.F * esize(c.dtype);
  if (h1 != nullptr && bytes > 0)
    CK(cudaMemcpyAsync(h1, b + L.h1, bytes, cudaMemcpyDeviceToDevice, st));
  if (h3 != nullptr && bytes > 0)
    CK(cudaMemcpyAsync(h3, b + L.h3, bytes, cudaMemcpyDeviceToDevice, st));
  return MOE_OK;
}

moe_status moe_device_status(const moe_config* cfg, const void* workspace, size_t workspace_bytes,
                             int32_t* status_host, void* stream) {
  RET_IF(validate_config(cfg));
  RET_IF(check_ws(*cfg, workspace, workspace_bytes));
  if (!status_host) return MOE_ERR_INVALID_ARG;
  Layout L = make_layout(*cfg);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CK(cudaMemcpyAsync(status_host, static_cast<const char*>(workspace) + L.status, 4,
                     cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  return MOE_OK;
}

static moe_status grouped_gemm_impl(int32_t form, int32_t M, int32_t N, int32_t K, int32_t E,
                                    const int32_t* offsets, const void* A, const void* B, void* C,
                                    int32_t* dev_status, long long wait_ns, int stall,
                                    void* stream);

moe_status moe_grouped_gemm(int32_t form, int32_t M, int32_t N, int32_t K, int32_t E,
                            const int32_t* offsets, const void* A, const void* B, void* C,
                            int32_t* dev_status, void* stream) {
  return grouped_gemm_impl(form, M, N, K, E, offsets, A, B, C, dev_status, 0, 0, stream);
}

moe_status moe_selftest_wait_timeout(int32_t form, int32_t M, int32_t N, int32_t K, int32_t E,
                                     const int32_t* offsets, const void* A, const void* B, void* C,
                                     int32_t* dev_status, int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 2000000000ll) return MOE_ERR_INVALID_ARG;
  return grouped_gemm_impl(form, M, N, K, E, offsets, A, B, C, dev_status, limit_ns, 1, stream);
}

static moe_status grouped_gemm_impl(int32_t form, int32_t M, int32_t N, int32_t K, int32_t E,
                                    const int32_t* offsets, const void* A, const void* B, void* C,
                                    int32_t* dev_status, long long wait_ns, int stall,
                                    void* stream) {
  g_launches = 0;
  if (form < 0 || form > 2 || M < 0 || N <= 0 || K < 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  // inner (contiguous) dimensions must be multiples of 8 elements; form 2's K
  // counts rows and has no alignment requirement
  if (E > 256 || N % 8 != 0 || (form != 2 && K % 8 != 0) || (form == 2 && M % 8 != 0))
    return MOE_ERR_UNSUPPORTED;
  if (!offsets || !A || !B || !C || !dev_status) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {offsets, A, B, C, dev_status};
  for (const void* q : ps)
    if (!aligned16(q)) return MOE_ERR_ALIGNMENT;
  RET_IF(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GemmArgs g{};
  g.a_type = g.b_type = MOE_BF16;
  g.offsets = offsets;
  g.E = E;
  g.status = dev_status;
  g.epi = EPI_STORE;
  g.A0 = A;
  g.B0 = B;
  g.C = C;
  g.wait_ns = wait_ns;
  g.stall = stall;
  if (form == 2) {
    // C[e][m][n] = sum over rows r of segment e of A[r, m] B[r, n]; K = total rows
    g.ragged_k = true;
    g.c_type = MOE_F32;
    g.M = M;
    g.N = N;
    g.K0 = K;
    g.lda = M;
    g.ldb = N;
    g.ldc = N;
    g.sCe = (long long)M * N;
  } else {
    // C[r, n] = sum_k A[r, k] B_e(k, n); M = total rows, B [E, N, K] or [E, K, N]
    g.ragged_k = false;
    g.c_type = MOE_BF16;
    g.b_kcontig = form == 0;
    g.M = M;
    g.N = N;
    g.K0 = K;
    g.lda = K;
    g.ldb = form == 0 ? K : N;
    g.sBe = (long long)N * K;
    g.ldc = N;
  }
  KL("grouped_gemm", launch_gemm_tc(g, st));
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration, dtype or device";
    case MOE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "bounded device wait expired";
  }
  return "unknown status";
}

int32_t moe_last_launch_count(void) { return g_launches; }

int32_t moe_expert_gemm_path(const moe_config* cfg) {
  const moe_status v = validate_config(cfg);
  if (v != MOE_OK) return -(int32_t)v;
  if (cfg->dtype == MOE_BF16) return MOE_GEMM_TENSOR_BF16;
  return make_layout(*cfg).f32x3_bytes > 0 ? MOE_GEMM_TENSOR_F32X3 : MOE_GEMM_CUDA_CORES;
}

int32_t moe_build_flags(void) {
#ifdef MOE_DEBUG
  return MOE_BUILD_DEBUG_CHECKS;
#else
  return 0;
#endif
}

moe_status moe_debug_poke_routing(const moe_config* cfg, void* workspace, size_t workspace_bytes,
                                  int32_t field, int64_t index, int32_t value, void* stream) {
#ifndef MOE_DEBUG
  (void)cfg; (void)workspace; (void)workspace_bytes; (void)field; (void)index; (void)value;
  (void)stream;
  return MOE_ERR_UNSUPPORTED;   // a release build never corrupts its own state
#else
  RET_IF(validate_config(cfg));
  const moe_config& c = *cfg;
  RET_IF(check_ws(c, workspace, workspace_bytes));
  if (field != 0 && field != 1) return MOE_ERR_INVALID_ARG;
  if (index < 0 || index >= (int64_t)c.T * c.k) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(c);
  char* at = static_cast<char*>(workspace) + (field == 0 ? L.idx : L.slot_of) + (size_t)index * 4;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CK(cudaMemcpyAsync(at, &value, sizeof(value), cudaMemcpyHostToDevice, st));
  CK(cudaStreamSynchronize(st));
  return MOE_OK;
#endif
}

void moe_profile_enable(int32_t on) {
  g_prof = on != 0;
  g_prof_n = 0;
}

int32_t moe_profile_count(void) { return g_prof_n; }

const char* moe_profile_name(int32_t i) {
  return (i >= 0 && i < g_prof_n) ? g_prof_recs[i].name : "";
}

float moe_profile_ms(int32_t i) {
  if (i < 0 || i >= g_prof_n) return -1.f;
  float ms = -1.f;
  if (cudaEventSynchronize(g_prof_recs[i].b) != cudaSuccess) return -1.f;
  if (cudaEventElapsedTime(&ms, g_prof_recs[i].a, g_prof_recs[i].b) != cudaSuccess) return -1.f;
  return ms;
}

}  // extern "C"
