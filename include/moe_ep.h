/*
 * moe_ep.h -- expert-parallel training step of the MoE layer: the rank-local
 * phases, C ABI.
 *
 * "AI Infra Kernel Lab", "Project status" (expert parallelism with a variable
 * All-to-All) and "Numerical contracts": the E experts are split over
 * n_ranks ranks, rank r owning the L = E / n_ranks experts
 * [r L, (r + 1) L).  Every rank routes its own tokens with the replicated
 * router; the dispatch exchange sends UNWEIGHTED expert-major rows to the
 * experts' owners; the outputs come back to their source rank, where the
 * routing weights are applied in the combine; the backward runs through both
 * exchanges in reverse.  Token shards may be uneven or empty.
 *
 * The library runs the phases; the caller moves rows between ranks (NCCL
 * grouped send / receive, gloo, or plain copies when one process drives
 * every rank) and sums the small per-rank statistics over the ranks.  One
 * training step is, on every rank r, in this order:
 *
 *   1. moe_ep_route          router, dispatch and gather of this rank's T_r
 *                            tokens over all E experts; writes this rank's
 *                            score column sums.  The caller reads the
 *                            per-expert counts (moe_ep_get_routing), shares
 *                            them with every rank (an all-gather).
 *   2. exchange              rows [offsets[e], offsets[e] + counts[e]) of the
 *                            x_e buffer (moe_ep_buffer_offsets) go to the
 *                            owner of expert e, which stores the rows of its
 *                            local expert l from source ranks 0, 1, ... one
 *                            after the other (source order), experts in
 *                            order: moe_ep_rows.x.
 *   3. moe_ep_expert_forward the local experts' MLPs on the received rows.
 *   4. exchange back         moe_ep_rows.y blocks to their sources' y_e
 *                            buffer (the same blocks, reversed).
 *   5. moe_ep_combine        gate-weighted combine, MSE seed, combine
 *                            backward, and both losses from the counts and
 *                            score sums summed over all ranks.
 *   6. exchange              dy_e blocks to the owners: moe_ep_rows.dy.
 *   7. moe_ep_expert_backward the experts' backward and their SGD step.
 *   8. exchange back         moe_ep_rows.dx blocks to their sources' dx_e.
 *   9. moe_ep_router_backward router backward of this rank's tokens: its
 *                            share of dW_g and dL/dx of its tokens.
 *  10. moe_ep_router_update  after the caller sums dW_g over the ranks: the
 *                            router's SGD step (identical on every rank).
 * With the rows of each expert in source-rank order, an owner's rows are
 * those a single device would hold for the concatenation of the ranks'
 * tokens, in the same order.
 *
 * Conventions are those of moe.h (device pointers, caller-owned memory,
 * stream-ordered, host-side validation first, deterministic).  cfg->T is the
 * token count of THIS rank (0 allowed) and cfg->E the number of experts of
 * the whole layer.  Not supported here (MOE_ERR_UNSUPPORTED): an expert
 * capacity and shared experts.
 */
#ifndef MOE_GB300_EP_H
#define MOE_GB300_EP_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Which rank this is and the token count of the whole layer. */
typedef struct {
  int32_t n_ranks;   /* ranks the experts are split over; divides E          */
  int32_t rank;      /* 0 <= rank < n_ranks: owns experts [rank L, rank L + L) */
  int32_t T_total;   /* tokens over all ranks: the normaliser of both losses  */
} moe_ep_config;

/* Rows a rank received for its L local experts, expert-major (all rows of
 * local expert 0 first, each expert's rows in source-rank order), and the
 * buffers the local experts' forward and backward use.  Caller-owned device
 * memory, in cfg->dtype unless stated. */
typedef struct {
  int32_t rows;            /* received rows (0 allowed)                      */
  const int32_t* offsets;  /* [L + 1] int32: local expert l owns rows
                              [offsets[l], offsets[l + 1]); offsets[L] = rows */
  const void* x;           /* [rows, D] received unweighted activations      */
  void* h1;                /* [rows, F] saved pre-activations (H or H1)      */
  void* h3;                /* [rows, F] SwiGLU H3, else NULL                 */
  void* a;                 /* [rows, F] activations                          */
  void* y;                 /* [rows, D] expert outputs, to be sent back      */
  const void* dy;          /* [rows, D] received output gradients            */
  void* dh1;               /* [rows, F]                                      */
  void* dh3;               /* [rows, F] SwiGLU only, else NULL               */
  void* dx;                /* [rows, D] input gradients, to be sent back     */
  int32_t* status;         /* device int32: 0, or MOE_ERR_TIMEOUT if a
                              bounded device wait expired (caller zeroes it) */
  void* f32_scratch;       /* fp32 layers: moe_ep_f32_scratch_size bytes of
                              device scratch (16-byte aligned) for the expert
                              GEMMs on the tensor cores, or NULL (CUDA-core
                              GEMMs); ignored by bf16 layers                 */
  size_t f32_scratch_bytes;
} moe_ep_rows;

/* Scratch bytes that let the expert GEMMs of an fp32 layer over `rows`
 * received rows run on the tensor cores (each fp32 operand split into three
 * bf16 terms, the six leading term products summed in fp32): the same
 * arithmetic as the single-device step, which takes its scratch from its
 * workspace; without it (or when the answer is 0) they run on the CUDA cores
 * and results may differ from the single-device step's in the last bits.
 * 0 for bf16 layers and on an invalid request. */
MOE_API size_t moe_ep_f32_scratch_size(const moe_config* cfg, const moe_ep_config* ep,
                                       int32_t rows);

/* Workspace bytes of one rank's source-side state (routing, its tokens'
 * expert-major rows x_e / y_e / dy_e / dx_e, router buffers); 0 on an
 * invalid request. */
MOE_API size_t moe_ep_workspace_size(const moe_config* cfg, const moe_ep_config* ep);

/* Byte offsets, inside that workspace, of the expert-major row buffers the
 * exchanges read and write, each [T k, D] in cfg->dtype with the rows of
 * expert e at [offsets[e], offsets[e] + counts[e]) of moe_get_routing:
 * out[0] x_e (sent), out[1] y_e (received back), out[2] dy_e (sent),
 * out[3] dx_e (received back).  Host call, no device work. */
MOE_API moe_status moe_ep_buffer_offsets(const moe_config* cfg, const moe_ep_config* ep,
                                         size_t* out4);

/* moe_get_routing for an expert-parallel rank's workspace: the routing of
 * its tokens over all E experts (device copies on `stream`; any output may
 * be NULL): scores [T,E], idx [T,k], gate [T,k], counts [E], offsets [E+1],
 * src_tok [T k], slot_of [T,k]. */
MOE_API moe_status moe_ep_get_routing(const moe_config* cfg, const moe_ep_config* ep,
                                      const void* workspace, size_t workspace_bytes,
                                      float* scores, int32_t* idx, float* gate, int32_t* counts,
                                      int32_t* offsets, int32_t* src_tok, int32_t* slot_of,
                                      void* stream);

/* Step 1 (course Parts 3 and 4 on this rank's tokens): router scores,
 * top-k and gates, per-expert counts, offsets and slot maps, the gather of
 * x [T, D] into x_e; score_sum [E] fp32 receives the column sums over this
 * rank's tokens of the router scores (summed over ranks, they give the aux
 * loss's mean score P_e).  Reads w->w_gate, w->logit_bias, w->corr_bias
 * only. */
MOE_API moe_status moe_ep_route(const moe_config* cfg, const moe_ep_config* ep,
                                const moe_weights* w, const void* x, float* score_sum,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Step 3 (course Part 5): the local experts' up- and down-projections on the
 * received rows.  w->w1, w3, w2 (and b1, b2) hold the L local experts:
 * [L, F, D], [L, D, F], [L, F], [L, D]. */
MOE_API moe_status moe_ep_expert_forward(const moe_config* cfg, const moe_ep_config* ep,
                                         const moe_weights* w, const moe_ep_rows* rows,
                                         void* stream);

/* Step 5 (course Parts 4, 6 and 7): Y = sum_j g_tj y_e[slot(t, j)] for this
 * rank's tokens, dY = 2 (Y - y_target) / (T_total D), the combine backward
 * (dy_e rows, gate gradients), and the losses: d_loss[0] = this rank's share
 * sum_t |Y - y_target|^2 / (T_total D) of L_mse (the sum over ranks is
 * L_mse), d_loss[1] = aux = E sum_e f_e P_e with f_e = counts_total[e] /
 * (T_total k) and P_e = score_sum_total[e] / T_total (the same on every
 * rank).  counts_total [E] int32 and score_sum_total [E] fp32 are the
 * per-expert counts and score sums summed over all ranks. */
MOE_API moe_status moe_ep_combine(const moe_config* cfg, const moe_ep_config* ep,
                                  const int32_t* counts_total, const float* score_sum_total,
                                  const float* y_target, float* d_loss, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Step 7 (course Parts 5 and 7): the local experts' backward on the received
 * output gradients (dA with the activation backward, dW2, db2, dX_e, dW1,
 * dW3, db1) and SGD on their fp32 masters (p->w1, w3, w2, b1, b2 hold the L
 * local experts; bf16 layers also rewrite the bf16 copies p->w1_lp ...).
 * p->grads receives the local experts' gradients; for bf16 layers dw1 / dw3
 * / dw2 may be NULL (applied, not stored); fp32 layers and biases need their
 * buffers.  p->w_gate and the router fields are not used. */
MOE_API moe_status moe_ep_expert_backward(const moe_config* cfg, const moe_ep_config* ep,
                                          const moe_params* p, const moe_ep_rows* rows,
                                          float lr, void* stream);

/* Step 9 (course Parts 3, 4 and 6): router backward of this rank's tokens
 * from the gate gradients of step 5 and the aux gradient alpha E f_e /
 * T_total: dlogits, this rank's share dw_gate_part [E, D] fp32 of dL/dW_g
 * (the sum over ranks is dL/dW_g), and, when dx is not NULL, dx [T, D] fp32
 * = the router term plus the returned dx_e rows of each token (j order). */
MOE_API moe_status moe_ep_router_backward(const moe_config* cfg, const moe_ep_config* ep,
                                          const float* w_gate, const void* x,
                                          float* dw_gate_part, float* dx, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* Step 10 (course Part 7): w_gate -= lr * dw_gate (fp32 [E, D]; dw_gate the
 * gradient summed over all ranks). */
MOE_API moe_status moe_ep_router_update(const moe_config* cfg, float* w_gate,
                                        const float* dw_gate, float lr, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_EP_H */
