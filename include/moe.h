/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse top-k mixture-of-experts layer.
 *
 * One training step of a sparse top-k MoE layer, as the course "Trainable MoE
 * in CUDA" lays it out (Parts 1-7): router gate matmul -> scores (softmax, or
 * the sigmoid group-limited variant of "AI Infra Kernel Lab", "Project status")
 * -> per-token top-k and renormalisation -> dispatch (per-expert histogram,
 * exclusive-scan slot offsets, gather into expert-major rows) -> each expert's
 * two-layer MLP (ReLU / GELU-tanh with biases, or SwiGLU W2(SiLU(W1 x) * W3 x),
 * "AI Infra Kernel Lab", "Numerical contracts") -> gate-weighted combine ->
 * MSE task loss + load-balancing aux loss -> the full backward -> SGD.
 * Optional, per moe_config / moe_weights: a selection-only correction bias
 * (the DeepSeek gate of "AI Infra Kernel Lab"), a shared-expert SwiGLU branch
 * on every token, and an expert capacity that drops assignments beyond it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Shapes: T tokens, D model width, F expert hidden width, E experts, k
 *   experts per token, R = T*k routed rows.  All tensors are dense, row-major
 *   and contiguous.  x is [T,D]; the router weight W_g is [E,D]; expert
 *   weights use the [out,in] layout: W1, W3 [E,F,D], W2 [E,D,F], b1 [E,F],
 *   b2 [E,D].  Index tensors are int32.
 * - Memory: every pointer is a DEVICE pointer unless its comment says "host".
 *   The caller owns all memory, including the workspace; the library never
 *   allocates or frees.  Pointers must be 16-byte aligned (MOE_ERR_ALIGNMENT).
 * - Streams: all work is enqueued on `stream` (a cudaStream_t; NULL = the
 *   legacy default stream).  No entry point synchronises the host except
 *   moe_train_step_host / moe_train_steps_host, which wait for their own loss
 *   read-back (and use one internal side stream per device for uploads).
 *   Those two run one call at a time per device when called from several
 *   host threads, and every return, an error included, comes after their
 *   copies from the caller's host buffers have finished.
 *   After its first call on a device, moe_train_step neither synchronises
 *   nor allocates, so it can be captured into a CUDA graph.
 * - Validation: every call checks its arguments on the host before the first
 *   launch and returns a status; an unsupported request fails, it never falls
 *   back to another code path.
 * - Determinism: no floating-point atomics anywhere; the same inputs give the
 *   same bits on every call.  Routing ties go to the smaller expert id (and
 *   the smaller group id), as the grouped gate of "AI Infra Kernel Lab"
 *   specifies; rows of one expert keep ascending token order.
 * - Inputs are not modified, except the parameters moe_train_step updates.
 *   Repeated calls are independent (course lesson "Define Expert Mlp Forward
 *   And Backward", "Prove it works").
 * - Precision: MOE_F32 computes in fp32 on CUDA cores.  MOE_BF16 feeds the
 *   expert and router GEMMs bf16 operands with fp32 accumulation (tcgen05
 *   tensor cores; the router multiplies with a bf16 copy of its fp32 master);
 *   scores, gates, Y, dY, losses and every gradient of a parameter are fp32.
 *
 * Limits (MOE_ERR_UNSUPPORTED beyond them): 1 <= E <= 256, 1 <= k <= 32,
 * k <= E; n_groups divides E and is <= 32; D and F are multiples of 8;
 * for MOE_BF16 also E; T*k < 2^31.  SwiGLU experts carry no biases; shared
 * experts need SwiGLU and MOE_BF16.  T = 0 is accepted and does no work
 * (train step losses read 0).  The device must be sm_103.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* NULL pointer, negative size, inconsistent shape     */
  MOE_ERR_UNSUPPORTED = 2,          /* dtype / activation / limits / device arch           */
  MOE_ERR_ALIGNMENT = 3,            /* a pointer is not 16-byte aligned                    */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace smaller than moe_workspace_size()         */
  MOE_ERR_CUDA = 5,                 /* a CUDA runtime/driver call failed                   */
  MOE_ERR_TIMEOUT = 6               /* a bounded device-side wait expired                  */
} moe_status;

enum { MOE_ACT_RELU = 0, MOE_ACT_GELU_TANH = 1, MOE_ACT_SWIGLU = 2 };
enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
/* Group score of the group-limited router: the pages do not define it; the
 * default sums the two largest scores of a group, the alternative takes the
 * group maximum. */
enum { MOE_GROUP_TOP2_SUM = 0, MOE_GROUP_MAX = 1 };
enum { MOE_F32 = 0, MOE_BF16 = 1 };

/* Layer configuration.  n_groups = topk_groups = 1 selects plain top-k. */
typedef struct {
  int32_t T, D, F, E, k;
  int32_t n_groups, topk_groups, group_score;
  int32_t act;        /* MOE_ACT_*                                           */
  int32_t score;      /* MOE_SCORE_*                                         */
  int32_t dtype;      /* MOE_F32 | MOE_BF16: element type of x and expert W  */
  int32_t has_bias;   /* expert biases b1, b2 (not with SwiGLU)              */
  float aux_alpha;    /* L = L_mse + aux_alpha * aux                         */
  int32_t n_shared;   /* shared experts: 0 = none; n > 0 adds one SwiGLU
                         branch of hidden width n * F that every token passes
                         through, added to the output without a gate ("AI
                         Infra Kernel Lab").  Requires SwiGLU and MOE_BF16.  */
  float capacity_factor; /* 0: no expert capacity.  cf > 0: each expert keeps
                         its first C = ceil(cf * T * k / E) assignments in token
                         order and drops the rest (no output, zero gate
                         gradient, gates not renormalised); moe_get_routing then
                         reports slot_of = -1 for a dropped assignment, counts
                         before the drop (they also feed the aux loss) and
                         offsets over the kept rows.                          */
} moe_config;

/* Read-only weights for moe_forward / moe_backward. */
typedef struct {
  const float* w_gate;      /* [E,D] fp32 router weight (the router has no bias)   */
  const void* w1;           /* [E,F,D] in cfg.dtype                                */
  const void* w3;           /* [E,F,D] in cfg.dtype, SwiGLU only, else NULL         */
  const void* w2;           /* [E,D,F] in cfg.dtype                                */
  const float* b1;          /* [E,F] fp32 or NULL (has_bias = 0)                   */
  const float* b2;          /* [E,D] fp32 or NULL                                  */
  const float* logit_bias;  /* [E] fixed, non-trainable bias added to the logits
                               before the score, or NULL; -INFINITY never routes  */
  const float* corr_bias;   /* [E] selection-only correction bias, or NULL: the
                               experts are chosen by score + corr_bias (fp32 sum;
                               grouped routing ranks groups on these keys too),
                               while the gates, the aux loss and every gradient
                               use the unbiased scores ("AI Infra Kernel Lab",
                               grouped Top-K gate with correction bias).  Not
                               updated by the library.                            */
  const void* ws1;          /* shared branch (n_shared > 0, bf16), else NULL:
                               [n_shared*F, D]                                    */
  const void* ws3;          /* [n_shared*F, D]                                    */
  const void* ws2;          /* [D, n_shared*F]                                    */
} moe_weights;

/* fp32 gradient buffers, overwritten (never accumulated into) by each call:
 * zeroing them beforehand is not needed.  Experts that receive no rows get
 * exact zeros. */
typedef struct {
  float* dw_gate;   /* [E,D]              */
  float* dw1;       /* [E,F,D]            */
  float* dw3;       /* [E,F,D] or NULL    */
  float* dw2;       /* [E,D,F]            */
  float* db1;       /* [E,F] or NULL      */
  float* db2;       /* [E,D] or NULL      */
  float* dws1;      /* shared branch [n_shared*F, D] or NULL (n_shared = 0) */
  float* dws3;      /* [n_shared*F, D] or NULL                              */
  float* dws2;      /* [D, n_shared*F] or NULL                              */
} moe_grads;

/* Trainable parameters for moe_train_step.  The fp32 masters are updated in
 * place by SGD; for MOE_BF16 the bf16 working copies (used by the expert GEMMs)
 * are rewritten from the updated masters with round-to-nearest-even.  The
 * router reads its fp32 master (MOE_BF16 casts it to bf16 for its GEMMs). */
typedef struct {
  float* w_gate;            /* [E,D] fp32 master                         */
  float* w1;                /* [E,F,D] fp32 master                       */
  float* w3;                /* [E,F,D] fp32 master or NULL               */
  float* w2;                /* [E,D,F] fp32 master                       */
  float* b1;                /* [E,F] or NULL                             */
  float* b2;                /* [E,D] or NULL                             */
  void* w1_lp;              /* [E,F,D] bf16 copy (MOE_BF16) or NULL      */
  void* w3_lp;              /* [E,F,D] bf16 copy or NULL                 */
  void* w2_lp;              /* [E,D,F] bf16 copy or NULL                 */
  const float* logit_bias;  /* [E] or NULL                               */
  const float* corr_bias;   /* [E] selection-only correction bias or NULL
                               (as in moe_weights; never updated)         */
  float* ws1;               /* shared branch fp32 masters (n_shared > 0)
                               [n_shared*F, D], or NULL                   */
  float* ws3;               /* [n_shared*F, D]                            */
  float* ws2;               /* [D, n_shared*F]                            */
  void* ws1_lp;             /* their bf16 copies, rewritten by the step   */
  void* ws3_lp;
  void* ws2_lp;
  moe_grads grads;          /* gradient buffers, written by the step.
                               Any member may be NULL: the step still
                               computes that gradient and applies it to
                               its parameter, but does not hand it out.
                               For MOE_BF16 layers a NULL dw1 / dw3 / dw2
                               (dws1 / dws3 / dws2) also saves the HBM
                               traffic of storing it: the SGD update runs
                               inside the weight-gradient GEMM, which then
                               writes only the updated master and its
                               bf16 copy.  The updated parameters are
                               bit-identical either way.                */
} moe_params;

/* Bytes of device workspace the forward / backward / train step need for one
 * configuration: routing state, expert-major activations saved for the
 * backward, and reduction partials.  0 on an invalid configuration.  The size
 * is not monotone in T (the router's tokens per block and whether an fp32
 * layer's GEMMs take the tensor-core scratch both depend on it), so a
 * workspace is sized for the configuration of each call that uses it; a call
 * given fewer bytes returns MOE_ERR_WORKSPACE_TOO_SMALL. */
MOE_API size_t moe_workspace_size(const moe_config* cfg);

/* Forward (course Parts 3, 4 and 5): router, dispatch, expert MLPs, combine.
 * x [T,D] in cfg.dtype; y [T,D] fp32 output.  The routing and the activations
 * the backward needs stay in `workspace`, which must then be passed unchanged
 * to moe_backward. */
MOE_API moe_status moe_forward(const moe_config* cfg, const moe_weights* w, const void* x, float* y,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Backward of L = L_task + aux_alpha * aux given dy = dL_task/dy [T,D] fp32,
 * using the state moe_forward left in `workspace` (same cfg, w and x).  Writes
 * every gradient in `g` and, when dx is not NULL, dx [T,D] fp32 (expert path
 * scattered back plus the router term).  The aux gradient to the router
 * scores is aux_alpha * E * f_e / T with f_e = count_e / (T k) held constant
 * (course Part 6, "Load Balancing Auxiliary Loss"). */
MOE_API moe_status moe_backward(const moe_config* cfg, const moe_weights* w, const void* x,
                        const float* dy, const moe_grads* g, float* dx,
                        void* workspace, size_t workspace_bytes, void* stream);

/* One training step (course Part 7, "Loss, Optimizer, and Training Loop"):
 * forward, L_mse = mean over T*D of (y - y_target)^2, aux = E sum_e f_e P_e
 * with P_e the mean router score of expert e, the full backward of
 * L = L_mse + aux_alpha * aux (dx included), then theta <- theta - lr * grad
 * for W_g, W1, W3, W2, b1, b2.  x is in cfg.dtype (it must equal the bf16
 * rounding the expert weights' copies use for MOE_BF16); y_target [T,D] fp32.
 * d_loss: device float[2] receiving (L_mse, aux) of the forward, before the
 * update.  dx, when not NULL, receives dL/dx [T,D] fp32.  p->grads members
 * may be NULL (see moe_params). */
MOE_API moe_status moe_train_step(const moe_config* cfg, const moe_params* p, const void* x,
                          const float* y_target, float lr, float* d_loss, float* dx,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device staging moe_train_step_host needs for x and y_target. */
MOE_API size_t moe_host_staging_size(const moe_config* cfg);

/* moe_train_step from HOST buffers: copies x_host [T,D] (cfg.dtype) and
 * y_target_host [T,D] fp32 into `staging` (device, moe_host_staging_size
 * bytes), runs the step on `stream`, copies the two losses back into
 * loss_host[2] and waits for that copy.  Host buffers should be pinned for
 * full copy bandwidth; pageable memory works but is slower. */
MOE_API moe_status moe_train_step_host(const moe_config* cfg, const moe_params* p, const void* x_host,
                               const float* y_target_host, float lr, float* loss_host,
                               void* staging, size_t staging_bytes,
                               void* workspace, size_t workspace_bytes, void* stream);

/* n_steps training steps from HOST batches, pipelined for a data loader:
 * while step i runs on `stream`, the inputs of step i+1 are copied on an
 * internal side stream into the other half of `staging` (two input slots:
 * 2 * moe_host_staging_size(cfg) bytes).  x_hosts[i] -> [T,D] in cfg.dtype and
 * y_target_hosts[i] -> [T,D] fp32 are step i's batch (the same pointer may
 * repeat); the losses of step i land in loss_host[2 i], loss_host[2 i + 1].
 * Every step is exactly moe_train_step on its batch, in order.  Returns after
 * the last step's losses have been copied back.  Host batches should be
 * pinned and must stay valid until the call returns. */
MOE_API moe_status moe_train_steps_host(const moe_config* cfg, const moe_params* p,
                                        int32_t n_steps, const void* const* x_hosts,
                                        const float* const* y_target_hosts, float lr,
                                        float* loss_host, void* staging, size_t staging_bytes,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* Copies the routing the last forward left in `workspace` into caller buffers
 * (device, any may be NULL): scores [T,E] fp32, idx [T,k], gate [T,k] fp32,
 * counts [E], offsets [E+1], src_tok [R] (slot -> token), slot_of [T,k]
 * (token, j -> slot).  Device-to-device copies on `stream`. */
MOE_API moe_status moe_get_routing(const moe_config* cfg, const void* workspace, size_t workspace_bytes,
                           float* scores, int32_t* idx, float* gate, int32_t* counts,
                           int32_t* offsets, int32_t* src_tok, int32_t* slot_of, void* stream);

/* Copies expert-major intermediates of the last forward/backward out of the
 * workspace for inspection (device, any may be NULL): ye [R,D] and dxe [R,D]
 * in cfg.dtype, dlogits [T,E] fp32. */
MOE_API moe_status moe_get_intermediates(const moe_config* cfg, const void* workspace,
                                 size_t workspace_bytes, void* ye, void* dxe, float* dlogits,
                                 void* stream);

/* Copies the expert pre-activations of the last forward out of `workspace`
 * for inspection (device, either may be NULL), [R,F] each in cfg.dtype with
 * rows in the expert-major slot order of moe_get_routing: h1 = X_e W1^T (+ b1)
 * for ReLU / GELU experts (the backward's activation derivative reads it) or
 * H1 = X_e W1^T for SwiGLU; h3 = X_e W3^T (SwiGLU only, else
 * MOE_ERR_INVALID_ARG).  Rows past the last kept row of an expert capacity
 * are unspecified.  Device-to-device copies on `stream`. */
MOE_API moe_status moe_get_hidden(const moe_config* cfg, const void* workspace,
                                  size_t workspace_bytes, void* h1, void* h3, void* stream);

/* Reads the device status word of the last call that used `workspace`: 0, or
 * MOE_ERR_TIMEOUT when a bounded device-side wait of a tensor-core kernel
 * expired (that kernel then stopped early and its outputs are invalid), or,
 * in the MOE_DEBUG variant only, MOE_ERR_INVALID_ARG when a routing index was
 * out of range (see moe_build_flags).  A forward clears it.  Synchronises
 * `stream`. */
MOE_API moe_status moe_device_status(const moe_config* cfg, const void* workspace,
                                     size_t workspace_bytes, int32_t* status_host, void* stream);

/* Grouped GEMM over contiguous expert row segments on the tcgen05 tensor
 * cores, bf16 operands, fp32 accumulation (course "Trainable MoE in CUDA",
 * Part 1 matmul variants, applied per expert as in Part 5).  Segment e holds
 * rows [offsets[e], offsets[e+1]) of the row-indexed operands (offsets [E+1],
 * device, non-decreasing, offsets[E] = total rows).
 *   form 0: C[r,n] = sum_k A[r,k] B[e,n,k]    A [M,K], B [E,N,K], C [M,N] bf16
 *   form 1: C[r,n] = sum_k A[r,k] B[e,k,n]    A [M,K], B [E,K,N], C [M,N] bf16
 *   form 2: C[e,m,n] = sum_{r in e} A[r,m] B[r,n]
 *                                            A [K,M], B [K,N], C [E,M,N] fp32
 * (forms 0/1: M = total rows; form 2: K = total rows).  Offsets that break
 * these rules are clamped on the device to a non-decreasing sequence within
 * [0, total rows] (each entry raised to its predecessor, then capped), so no
 * access leaves A, B or C; rows outside the clamped segments are not
 * written.  The contiguous
 * dimensions must be multiples of 8: N always, K for forms 0/1, M for form 2.  dev_status: device int32, set to
 * MOE_ERR_TIMEOUT if a bounded wait expired (the caller zeroes it). */
MOE_API moe_status moe_grouped_gemm(int32_t form, int32_t M, int32_t N, int32_t K, int32_t E,
                                    const int32_t* offsets, const void* A, const void* B,
                                    void* C, int32_t* dev_status, void* stream);

/* Self-test of the bounded device waits: runs moe_grouped_gemm with every
 * load withheld, so the tensor-core kernel's waits run out after limit_ns
 * (0 < limit_ns <= 2e9).  The kernel then stops cleanly (drains, frees tensor
 * memory) and writes MOE_ERR_TIMEOUT to *dev_status; C is left unwritten.
 * The context stays usable.  Diagnostic only; the pages have no counterpart. */
MOE_API moe_status moe_selftest_wait_timeout(int32_t form, int32_t M, int32_t N, int32_t K,
                                             int32_t E, const int32_t* offsets, const void* A,
                                             const void* B, void* C, int32_t* dev_status,
                                             int64_t limit_ns, void* stream);

/* Build options of the loaded library: MOE_BUILD_DEBUG_CHECKS is set in the
 * MOE_DEBUG variant (libmoe_gb300_debug.so), whose gather, combine, combine
 * backward, scatter-back, route count / scatter and router backward kernels
 * check every routing index (expert ids against [0, E), expert-major slots
 * against [-1, T k)) before dereferencing it; an index out of range is
 * skipped and MOE_ERR_INVALID_ARG is recorded in the workspace status word
 * (read by moe_device_status).  The release library trusts the dispatch that
 * wrote the indices. */
#define MOE_BUILD_DEBUG_CHECKS 1
MOE_API int32_t moe_build_flags(void);

/* Which units run the expert GEMMs of a layer (host call, no device work):
 * MOE_GEMM_TENSOR_BF16 for bf16 layers (tcgen05 with bf16 operands);
 * MOE_GEMM_TENSOR_F32X3 for fp32 layers whose workspace holds the scratch
 * of the tensor-core path, where each fp32 operand is split into three bf16
 * terms and the six leading term products are summed in fp32 (the GEMMs with
 * a bias, ReLU / GELU or no epilogue; SwiGLU's activation GEMMs stay on the
 * CUDA cores); MOE_GEMM_CUDA_CORES for the other fp32 layers (D F below
 * 65536, or a scratch past 1 GiB); a negative moe_status on an invalid
 * configuration. */
#define MOE_GEMM_CUDA_CORES 0
#define MOE_GEMM_TENSOR_BF16 1
#define MOE_GEMM_TENSOR_F32X3 2
MOE_API int32_t moe_expert_gemm_path(const moe_config* cfg);

/* Fault injection for the MOE_DEBUG variant's tests, on the host side: writes
 * `value` into entry `index` (0 <= index < T k) of the routing state the last
 * forward left in `workspace`: field 0 the expert ids idx [T,k], field 1 the
 * slot map slot_of [T,k].  Synchronises `stream`.  The release library
 * returns MOE_ERR_UNSUPPORTED and writes nothing.  Diagnostic only; the pages
 * have no counterpart. */
MOE_API moe_status moe_debug_poke_routing(const moe_config* cfg, void* workspace,
                                          size_t workspace_bytes, int32_t field, int64_t index,
                                          int32_t value, void* stream);

/* Static text for a status code. */
MOE_API const char* moe_status_string(moe_status s);

/* Launch statistics of the last forward/backward/train-step call on this host
 * thread: the number of kernels it enqueued.  Host-side bookkeeping only. */
MOE_API int32_t moe_last_launch_count(void);

/* Kernel timing for measurement tools.  While enabled, every kernel launch of
 * the calling host thread is bracketed by two CUDA events on the launch
 * stream.  Records accumulate over calls from the moe_profile_enable(1) that
 * started them (at most 4096 kernels are kept); moe_profile_ms waits for the
 * i-th recorded kernel to finish and returns its duration in milliseconds (-1
 * for an invalid index). */
MOE_API void moe_profile_enable(int32_t on);
MOE_API int32_t moe_profile_count(void);
MOE_API const char* moe_profile_name(int32_t i);
MOE_API float moe_profile_ms(int32_t i);

/* Dispatch without a workspace, for callers that may not allocate device
 * memory when they route (for example while a stream is being captured into a
 * CUDA graph, inside a runtime whose memory pool forbids outside allocations,
 * or in a loop where an allocation could synchronise the device).  The pages
 * have no counterpart of this entry point: it is a deployment convenience.
 *
 * Given idx [T,k] (each entry in [0,E)), writes counts [E], offsets [E+1],
 * src_tok [T*k] and slot_of [T,k] exactly as moe_forward's dispatch does,
 * including the expert capacity of cfg->capacity_factor (a NaN or negative
 * factor is MOE_ERR_INVALID_ARG, as for moe_forward).  An idx entry outside
 * [0,E) is not counted and gets slot_of = -1.  The
 * per-chunk scratch counts live in one fixed device array inside the library
 * (1 MiB on every GPU that loads it, held until the process exits), so T*k
 * must not exceed MOE_NOALLOC_MAX_ROUTED (MOE_ERR_UNSUPPORTED otherwise).  It
 * calls no allocating routine.  The first call on a device looks up that
 * array's device address (with the device current); make that first call
 * before any stream capture.  All calls share the array: calls whose work
 * overlaps on the GPU (different streams, or different host threads) race
 * and must be serialised by the caller. */
#define MOE_NOALLOC_MAX_ROUTED (1024 * 1024)
MOE_API moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* idx,
                                        int32_t* counts, int32_t* offsets, int32_t* src_tok,
                                        int32_t* slot_of, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
