// Expert-parallel training step: the rank-local phases of one step ("AI Infra
// Kernel Lab", "Project status": expert parallelism over a variable
// All-to-All; "Numerical contracts": unweighted rows are dispatched, the
// routing weights are applied after the outputs return to their source
// rank, uneven and empty token shards are supported, and the backward runs
// through both exchanges).  The phases run the same kernels, with the same
// launch arguments, as the single-device step; only the rows' location
// differs: a rank's own tokens live in its workspace (routing, x_e, y_e,
// dy_e, dx_e over all E experts), the rows it receives for its local experts
// in caller buffers (moe_ep_rows).  The caller moves rows between ranks and
// sums the per-rank statistics; nothing here waits on another rank.
#include <cuda_runtime.h>

#include <initializer_list>

#include "../../include/moe_ep.h"
#include "api_common.h"
#include "kernels.h"

using namespace moe;
using namespace moe::api;

namespace {

moe_status ep_check(const moe_config* cfg, const moe_ep_config* ep) {
  RET_IF(validate_config(cfg));
  if (ep == nullptr) return MOE_ERR_INVALID_ARG;
  if (ep->n_ranks <= 0 || ep->rank < 0 || ep->rank >= ep->n_ranks) return MOE_ERR_INVALID_ARG;
  if (ep->T_total < cfg->T) return MOE_ERR_INVALID_ARG;
  if (cfg->E % ep->n_ranks != 0) return MOE_ERR_UNSUPPORTED;
  // an expert capacity ranks a token among all ranks' tokens, and shared
  // experts are a data-parallel branch: neither is part of this step
  if (cfg->capacity_factor != 0.f || cfg->n_shared != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// The source-side workspace: routing and the rank's own expert-major rows.
Layout ep_layout(const moe_config& c) { return make_layout(c, /*expert_buffers=*/false); }

moe_status ep_ws(const moe_config& c, const void* ws, size_t bytes) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_ALIGNMENT;
  if (bytes < ep_layout(c).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

moe_status all_aligned(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p && !aligned16(p)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

// The received rows of the local experts as expert segments.
moe_status rows_of(const moe_config& c, const moe_ep_config& ep, const moe_ep_rows* rows,
                   bool backward, ExpertRows* out) {
  if (rows == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_ep_rows& r = *rows;
  if (r.rows < 0) return MOE_ERR_INVALID_ARG;
  if ((long long)r.rows > (long long)ep.T_total * c.k) return MOE_ERR_INVALID_ARG;
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  if (!r.offsets || !r.status) return MOE_ERR_INVALID_ARG;
  if (r.rows > 0) {
    if (!r.x || !r.h1 || !r.a || (swiglu && !r.h3)) return MOE_ERR_INVALID_ARG;
    if (!backward && !r.y) return MOE_ERR_INVALID_ARG;
    if (backward && (!r.dy || !r.dh1 || !r.dx || (swiglu && !r.dh3))) return MOE_ERR_INVALID_ARG;
  }
  RET_IF(all_aligned({r.offsets, r.x, r.h1, r.h3, r.a, r.y, r.dy, r.dh1, r.dh3, r.dx, r.status}));
  ExpertRows e{};
  e.E = c.E / ep.n_ranks;
  e.M = r.rows;
  e.offsets = r.offsets;
  e.status = r.status;
  e.xe = const_cast<void*>(r.x);
  e.h1 = r.h1;
  e.h3 = r.h3;
  e.a = r.a;
  e.ye = r.y;
  e.dye = const_cast<void*>(r.dy);
  e.dh1 = r.dh1;
  e.dh3 = r.dh3;
  e.dxe = r.dx;
  if (c.dtype == MOE_F32 && r.f32_scratch != nullptr && r.f32_scratch_bytes > 0) {
    if (!aligned16(r.f32_scratch)) return MOE_ERR_ALIGNMENT;
    e.f32x3 = r.f32_scratch;
    e.f32x3_bytes = r.f32_scratch_bytes;
  }
  *out = e;
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_ep_workspace_size(const moe_config* cfg, const moe_ep_config* ep) {
  if (ep_check(cfg, ep) != MOE_OK) return 0;
  return ep_layout(*cfg).total;
}

size_t moe_ep_f32_scratch_size(const moe_config* cfg, const moe_ep_config* ep, int32_t rows) {
  if (ep_check(cfg, ep) != MOE_OK || rows < 0 || (long long)rows > (long long)ep->T_total * cfg->k)
    return 0;
  return f32x3_scratch(*cfg, (size_t)rows, (size_t)(cfg->E / ep->n_ranks));
}

moe_status moe_ep_buffer_offsets(const moe_config* cfg, const moe_ep_config* ep, size_t* out4) {
  RET_IF(ep_check(cfg, ep));
  if (out4 == nullptr) return MOE_ERR_INVALID_ARG;
  const Layout L = ep_layout(*cfg);
  out4[0] = L.xe;
  out4[1] = L.ye;
  out4[2] = L.dye;
  out4[3] = L.dxe;
  return MOE_OK;
}

moe_status moe_ep_get_routing(const moe_config* cfg, const moe_ep_config* ep,
                              const void* workspace, size_t workspace_bytes, float* scores,
                              int32_t* idx, float* gate, int32_t* counts, int32_t* offsets,
                              int32_t* src_tok, int32_t* slot_of, void* stream) {
  RET_IF(ep_check(cfg, ep));
  const moe_config& c = *cfg;
  RET_IF(ep_ws(c, workspace, workspace_bytes));
  const Layout L = ep_layout(c);
  const char* b = static_cast<const char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t T = c.T, E = c.E, R = (size_t)c.T * c.k;
  struct Cp { void* dst; size_t off; size_t bytes; } cps[] = {
      {scores, L.scores, T * E * 4}, {idx, L.idx, R * 4},       {gate, L.gate, R * 4},
      {counts, L.counts, E * 4},     {offsets, L.offsets, (E + 1) * 4},
      {src_tok, L.src_tok, R * 4},   {slot_of, L.slot_of, R * 4}};
  for (const Cp& cp : cps)
    if (cp.dst && cp.bytes)
      CK(cudaMemcpyAsync(cp.dst, b + cp.off, cp.bytes, cudaMemcpyDeviceToDevice, st));
  return MOE_OK;
}

moe_status moe_ep_route(const moe_config* cfg, const moe_ep_config* ep, const moe_weights* w,
                        const void* x, float* score_sum, void* workspace, size_t workspace_bytes,
                        void* stream) {
  g_launches = 0;
  RET_IF(ep_check(cfg, ep));
  const moe_config& c = *cfg;
  if (w == nullptr || w->w_gate == nullptr || score_sum == nullptr) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && x == nullptr) return MOE_ERR_INVALID_ARG;
  RET_IF(all_aligned({w->w_gate, w->logit_bias, w->corr_bias, x, score_sum}));
  RET_IF(ep_ws(c, workspace, workspace_bytes));
  RET_IF(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = ep_layout(c);
  Ptrs P{static_cast<char*>(workspace), &L};
  if (c.T == 0) {
    // an empty shard routes nothing: zero counts, offsets and score sums
    CK(cudaMemsetAsync(P.at<void>(L.status), 0, 16, st));
    CK(cudaMemsetAsync(P.at<void>(L.counts), 0, (size_t)c.E * 4, st));
    CK(cudaMemsetAsync(P.at<void>(L.offsets), 0, (size_t)(c.E + 1) * 4, st));
    CK(cudaMemsetAsync(score_sum, 0, (size_t)c.E * 4, st));
    return MOE_OK;
  }
  ExpertW ew{};
  ew.w_gate = w->w_gate;
  ew.logit_bias = w->logit_bias;
  ew.corr_bias = w->corr_bias;
  RET_IF(route_tokens(c, ew, x, P, st));
  // this rank's score column sums: the per-block partials of the router,
  // added in block order
  KL("score_colsum", launch_sum_partials(P.at<float>(L.psum), router_fwd_blocks(c.T), c.E,
                                         score_sum, st));
  return MOE_OK;
}

moe_status moe_ep_expert_forward(const moe_config* cfg, const moe_ep_config* ep,
                                 const moe_weights* w, const moe_ep_rows* rows, void* stream) {
  g_launches = 0;
  RET_IF(ep_check(cfg, ep));
  const moe_config& c = *cfg;
  if (w == nullptr || !w->w1 || !w->w2 || (c.act == MOE_ACT_SWIGLU && !w->w3))
    return MOE_ERR_INVALID_ARG;
  if (c.has_bias && (!w->b1 || !w->b2)) return MOE_ERR_INVALID_ARG;
  RET_IF(all_aligned({w->w1, w->w3, w->w2, w->b1, w->b2}));
  ExpertRows r{};
  RET_IF(rows_of(c, *ep, rows, false, &r));
  RET_IF(check_device());
  if (r.M == 0) return MOE_OK;
  ExpertW ew{};
  ew.w1 = w->w1;
  ew.w3 = w->w3;
  ew.w2 = w->w2;
  ew.b1 = w->b1;
  ew.b2 = w->b2;
  return experts_forward(c, ew, r, static_cast<cudaStream_t>(stream));
}

moe_status moe_ep_combine(const moe_config* cfg, const moe_ep_config* ep,
                          const int32_t* counts_total, const float* score_sum_total,
                          const float* y_target, float* d_loss, void* workspace,
                          size_t workspace_bytes, void* stream) {
  g_launches = 0;
  RET_IF(ep_check(cfg, ep));
  const moe_config& c = *cfg;
  if (!counts_total || !score_sum_total || !d_loss || (c.T > 0 && !y_target))
    return MOE_ERR_INVALID_ARG;
  RET_IF(all_aligned({counts_total, score_sum_total, y_target, d_loss}));
  RET_IF(ep_ws(c, workspace, workspace_bytes));
  RET_IF(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = ep_layout(c);
  Ptrs P{static_cast<char*>(workspace), &L};
  if (ep->T_total == 0) {
    CK(cudaMemsetAsync(d_loss, 0, 2 * sizeof(float), st));
    return MOE_OK;
  }
  // the MSE seed is normalised by every rank's tokens: 1 / (T_total D)
  const float inv_n = 1.0f / ((float)ep->T_total * (float)c.D);
  if (c.T > 0) {
    if (c.k <= 8) {
      KL("combine_fused", launch_combine_train(c.dtype, P.at<void>(L.ye), P.at<float>(L.gate),
                                               P.at<int>(L.slot_of), c.T, c.D, c.k, nullptr,
                                               y_target, P.at<double>(L.sq), P.at<void>(L.dye),
                                               P.at<float>(L.dgate), nullptr, st, inv_n,
                                               P.at<int>(L.status)));
    } else {
      KL("combine_loss", launch_combine(c.dtype, P.at<void>(L.ye), P.at<float>(L.gate),
                                        P.at<int>(L.slot_of), c.T, c.D, c.k, nullptr, nullptr,
                                        y_target, P.at<float>(L.dy), P.at<double>(L.sq), st,
                                        inv_n, P.at<int>(L.status)));
      KL("combine_bwd", launch_combine_bwd(c.dtype, P.at<float>(L.dy), P.at<void>(L.ye),
                                           P.at<float>(L.gate), P.at<int>(L.slot_of), c.T, c.D,
                                           c.k, P.at<void>(L.dye), P.at<float>(L.dgate), st,
                                           P.at<int>(L.status)));
    }
  }
  // losses from the statistics of all ranks: this rank's squared errors over
  // T_total D, and the aux loss (and its score gradient row) from the summed
  // counts and score sums, one "partial" row of each
  KL("finalize_losses",
     launch_finalize_losses(P.at<double>(L.sq), c.T > 0 ? combine_blocks(c.T) : 0,
                            score_sum_total, 1, counts_total, ep->T_total, c.D, c.E, c.k,
                            c.aux_alpha, d_loss, P.at<float>(L.aux_row), st));
  return MOE_OK;
}

moe_status moe_ep_expert_backward(const moe_config* cfg, const moe_ep_config* ep,
                                  const moe_params* p, const moe_ep_rows* rows, float lr,
                                  void* stream) {
  g_launches = 0;
  RET_IF(ep_check(cfg, ep));
  const moe_config& c = *cfg;
  const bool lp = c.dtype == MOE_BF16;
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  if (p == nullptr || !p->w1 || !p->w2 || (swiglu && !p->w3)) return MOE_ERR_INVALID_ARG;
  if (lp && (!p->w1_lp || !p->w2_lp || (swiglu && !p->w3_lp))) return MOE_ERR_INVALID_ARG;
  if (c.has_bias && (!p->b1 || !p->b2 || !p->grads.db1 || !p->grads.db2))
    return MOE_ERR_INVALID_ARG;
  // fp32 layers apply SGD after the GEMMs and need the gradients stored
  if (!lp && (!p->grads.dw1 || !p->grads.dw2 || (swiglu && !p->grads.dw3)))
    return MOE_ERR_INVALID_ARG;
  const moe_grads& g = p->grads;
  RET_IF(all_aligned({p->w1, p->w3, p->w2, p->b1, p->b2, p->w1_lp, p->w3_lp, p->w2_lp, g.dw1,
                      g.dw3, g.dw2, g.db1, g.db2}));
  ExpertRows r{};
  RET_IF(rows_of(c, *ep, rows, true, &r));
  RET_IF(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long Lx = c.E / ep->n_ranks, D = c.D, F = c.F;
  if (r.M == 0) {
    // no rows for the local experts: zero gradients; the SGD step leaves the
    // masters as they are
    struct Z { float* p; long long n; } zs[] = {
        {g.dw1, Lx * F * D}, {g.dw3, Lx * F * D}, {g.dw2, Lx * D * F}, {g.db1, Lx * F},
        {g.db2, Lx * D}};
    for (const Z& z : zs)
      if (z.p) CK(launch_fill_zero(z.p, (size_t)z.n * 4, st));
    return MOE_OK;
  }
  ExpertW ew{};
  ew.w1 = lp ? p->w1_lp : p->w1;
  ew.w3 = lp ? p->w3_lp : p->w3;
  ew.w2 = lp ? p->w2_lp : p->w2;
  ew.b1 = p->b1;
  ew.b2 = p->b2;
  SgdFuse sf{};
  sf.lr = lr;
  sf.w1 = p->w1;
  sf.w3 = p->w3;
  sf.w2 = p->w2;
  sf.w1_lp = p->w1_lp;
  sf.w3_lp = p->w3_lp;
  sf.w2_lp = p->w2_lp;
  RET_IF(experts_backward(c, ew, r, g, lp ? &sf : nullptr, st));
  // SGD of what the GEMM epilogues did not update
  SgdTensor ts[SGD_MAX_TENSORS];
  int nt = 0;
  if (!lp) {
    ts[nt++] = {p->w1, g.dw1, Lx * F * D, nullptr};
    if (swiglu) ts[nt++] = {p->w3, g.dw3, Lx * F * D, nullptr};
    ts[nt++] = {p->w2, g.dw2, Lx * D * F, nullptr};
  }
  if (c.has_bias) {
    ts[nt++] = {p->b1, g.db1, Lx * F, nullptr};
    ts[nt++] = {p->b2, g.db2, Lx * D, nullptr};
  }
  if (nt > 0) KL("sgd", launch_sgd(ts, nt, lr, st));
  return MOE_OK;
}

moe_status moe_ep_router_backward(const moe_config* cfg, const moe_ep_config* ep,
                                  const float* w_gate, const void* x, float* dw_gate_part,
                                  float* dx, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  g_launches = 0;
  RET_IF(ep_check(cfg, ep));
  const moe_config& c = *cfg;
  if (!w_gate || !dw_gate_part || (c.T > 0 && !x)) return MOE_ERR_INVALID_ARG;
  RET_IF(all_aligned({w_gate, x, dw_gate_part, dx}));
  RET_IF(ep_ws(c, workspace, workspace_bytes));
  RET_IF(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c.T == 0) {
    CK(launch_fill_zero(dw_gate_part, (size_t)c.E * c.D * 4, st));
    return MOE_OK;
  }
  const Layout L = ep_layout(c);
  Ptrs P{static_cast<char*>(workspace), &L};
  ExpertW ew{};
  ew.w_gate = w_gate;
  float* dxp = dx ? dx : P.at<float>(L.dx);
  return router_backward(c, ew, x, dw_gate_part, dxp, nullptr, P, st);
}

moe_status moe_ep_router_update(const moe_config* cfg, float* w_gate, const float* dw_gate,
                                float lr, void* stream) {
  g_launches = 0;
  RET_IF(validate_config(cfg));
  if (!w_gate || !dw_gate) return MOE_ERR_INVALID_ARG;
  RET_IF(all_aligned({w_gate, dw_gate}));
  RET_IF(check_device());
  SgdTensor t{w_gate, dw_gate, (long long)cfg->E * cfg->D, nullptr};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  KL("sgd", launch_sgd(&t, 1, lr, st));
  return MOE_OK;
}

}  // extern "C"
