// Host-side launchers of the MoE kernels (internal to the library).
#pragma once

#include <atomic>
#include <cmath>
#include <utility>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Raises a kernel's dynamic shared-memory limit once per device: the
// attribute belongs to the current device's context, so a process that drives
// several devices sets it on each.  `done` holds one bit per device ordinal
// (ordinals from 64 on set it on every call).  Safe to call from several host
// threads: a race only repeats the idempotent setting.
template <typename Kernel>
inline cudaError_t ensure_dynamic_smem(Kernel* kernel, int bytes,
                                       std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

#ifndef MOE_PDL
#define MOE_PDL 1
#endif
// Launches `kernel` on `st` with programmatic stream serialization allowed:
// it may start while the previous kernel of the stream finishes, and waits
// for it (pdl_begin in common.cuh) before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = MOE_PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Returns the launch's error from the enclosing launcher, if any.
#define MOE_LAUNCH(expr)                          \
  do {                                            \
    cudaError_t _le = (expr);                     \
    if (_le != cudaSuccess) return _le;           \
  } while (0)

struct RouterArgs {
  int T, D, E, k;
  int score;         // 0 softmax, 1 sigmoid
  int n_groups, topk_groups, group_score;
  const float* corr_bias;   // [E] selection-only correction bias, or nullptr
};

// ---- router (router.cu)
int router_fwd_blocks(int T);
cudaError_t launch_router_fwd(int dtype, const void* x, const float* wg, const float* logit_bias,
                              const RouterArgs& a, float* scores, int* idx, float* gate,
                              float* psum_partial, cudaStream_t st);
cudaError_t launch_router_bwd(const float* scores, const int* idx, const float* gate,
                              const float* dgate, const float* aux_row, const RouterArgs& a,
                              float* dlogits, void* dlogits_lp, cudaStream_t st,
                              int* dbg = nullptr);
// selection from precomputed logits (bias already added) and the bf16 weight cast
cudaError_t launch_router_select(const float* logits, const RouterArgs& a, float* scores, int* idx,
                                 float* gate, float* psum_partial, cudaStream_t st);
cudaError_t launch_cast_bf16(const float* src, void* dst, long long n, cudaStream_t st);

// ---- dispatch, combine, losses, optimizer (dispatch.cu)
// Routed assignments per dispatch chunk (one warp walks a chunk in the
// scatter): about ROUTE_TARGET_CHUNKS chunks, a multiple of 32 assignments
// between ROUTE_CHUNK_MIN and ROUTE_CHUNK_MAX.  Any chunking gives the same
// result; so at most max(ROUTE_TARGET_CHUNKS, ceil(R / ROUTE_CHUNK_MAX)) chunks.
constexpr int ROUTE_CHUNK_MIN = 256;
constexpr int ROUTE_CHUNK_MAX = 1024;
constexpr int ROUTE_TARGET_CHUNKS = 608;   // four per SM
int route_chunk(long long R);
int route_chunks(long long R);
// dbg: the status word a MOE_DEBUG build records an out-of-range routing
// index in (unused by release builds), or nullptr; see common.cuh.
cudaError_t launch_route_count(const int* idx, long long R, int E, int* chunk_counts,
                               cudaStream_t st, int* dbg = nullptr);
// Rows an expert may keep under a capacity factor cf > 0: ceil(cf * T * k / E)
// (computed in double), else INT_MAX (no limit).
inline int expert_capacity_rows(float cf, int T, int k, int E) {
  if (!(cf > 0.f)) return 0x7fffffff;
  const double c = std::ceil((double)cf * (double)T * (double)k / (double)E);
  return c >= 2147483647.0 ? 0x7fffffff : (int)c;
}
// cap: rows an expert may keep (an expert capacity), INT_MAX for no limit;
// counts stay the routed (pre-drop) counts, offsets scan the kept counts and a
// dropped assignment gets slot_of = -1.
cudaError_t launch_route_scan(int* chunk_counts, int nchunks, int E, int cap, int* counts,
                              int* offsets, cudaStream_t st);
cudaError_t launch_route_scatter(const int* idx, long long R, int k, int E, int cap,
                                 const int* chunk_base, const int* offsets, int* src_tok,
                                 int* slot_of, cudaStream_t st, int* dbg = nullptr);
cudaError_t launch_gather(int dtype, const void* x, const int* slot_of, int T, int k, int D,
                          void* xe, cudaStream_t st, int* dbg = nullptr);
int combine_blocks(int T);
// ys: the shared-expert branch's output [T, D] added to Y, or nullptr.
// inv_n: the MSE normaliser 1 / (tokens D); 0 takes 1 / (T D) (a single
// device; an expert-parallel rank passes the one over all ranks' tokens).
cudaError_t launch_combine(int dtype, const void* ye, const float* gate, const int* slot_of,
                           int T, int D, int k, const void* ys, float* y, const float* target,
                           float* dy, double* sq_partial, cudaStream_t st, float inv_n = 0.f,
                           int* dbg = nullptr);
cudaError_t launch_finalize_losses(const double* sq_partial, int n_sq, const float* psum_partial,
                                   int n_ps, const int* counts, int T, int D, int E, int k,
                                   float alpha, float* d_loss, float* aux_row, cudaStream_t st);
// Training-step combine + MSE seed + combine backward in one pass (k <= 8).
// ys as in launch_combine; dy_lp (bf16 layers): also store dY in bf16, or nullptr.
cudaError_t launch_combine_train(int dtype, const void* ye, const float* gate, const int* slot_of,
                                 int T, int D, int k, const void* ys, const float* target,
                                 double* sq_partial, void* dye, float* dgate, void* dy_lp,
                                 cudaStream_t st, float inv_n = 0.f, int* dbg = nullptr);
cudaError_t launch_combine_bwd(int dtype, const float* dy, const void* ye, const float* gate,
                               const int* slot_of, int T, int D, int k, void* dye, float* dgate,
                               cudaStream_t st, int* dbg = nullptr);
// extra: a [T, D] row block (cfg dtype) added to dX after the expert rows, or nullptr.
cudaError_t launch_scatter_back_add(int dtype, float* dx, const void* dxe, const int* slot_of,
                                    int T, int D, int k, const void* extra, cudaStream_t st,
                                    int* dbg = nullptr);
cudaError_t launch_segment_colsum(int dtype, const void* src, const int* offsets, int E, int N,
                                  float* out, cudaStream_t st);
cudaError_t launch_sum_partials(const float* partials, int nparts, long long n, float* out,
                                cudaStream_t st);
// SGD on up to SGD_MAX_TENSORS fp32 tensors in one launch: w -= lr * g over
// n elements (a multiple of 4) of each, and w_lp (bf16 copy, or null)
// rewritten from the result with round-to-nearest-even.
constexpr int SGD_MAX_TENSORS = 6;
struct SgdTensor {
  float* w;
  const float* g;
  long long n;
  void* w_lp;
};
cudaError_t launch_sgd(const SgdTensor* tensors, int count, float lr, cudaStream_t st);
cudaError_t launch_fill_zero(void* p, size_t bytes, cudaStream_t st);

// ---- grouped GEMMs (gemm_simt_f32.cu for fp32; gemm_tc.cu for bf16 on tcgen05)
enum Epi {
  EPI_STORE = 0,        // C = acc (+ bias[e, n])
  EPI_ACT_FWD = 1,      // out1 = H = acc + bias;  C = act(H)
  EPI_SWIGLU_FWD = 2,   // acc = H3; H1 read from aux0;  out1 = H3;  C = SiLU(H1) * H3
  EPI_ACT_BWD = 3,      // acc = dA; H from aux0;  C = dA * act'(H)
  EPI_SWIGLU_BWD = 4,   // acc = dA; H1 aux0, H3 aux1;  C = dH1;  out1 = dH3
  EPI_SWIGLU_UP = 6     // tcgen05 only: B0 = W1, B0x = W3 in one N = 2 x 128 tile;
                        //   out1 = H1, out2 = H3, C = SiLU(H1) * H3
};

// One grouped GEMM.  Ragged-M form (ragged_k = 0): rows [off_e, off_{e+1}) of
// A use expert e's B;  C[r, n] = sum_k A(r, k) B_e(k, n).  Ragged-K form
// (ragged_k = 1): C_e[m, n] = sum_{r in segment e} A(r, m) B(r, n).
// Operand element (row, col) addresses: a_kcontig ? A[m*lda + k] : A[k*lda + m],
// b_kcontig ? B_e[n*ldb + k] : B_e[k*ldb + n].  A second operand pair
// (A1, B1, K1) extends the reduction (ragged-M only).  offsets == nullptr
// means segments of seg_len rows.
struct GemmArgs {
  int a_type, b_type, c_type;   // 0 fp32, 1 bf16
  const void* A0;
  const void* B0;
  int K0;
  const void* A1;
  const void* B1;
  int K1;
  long long lda, ldb, sBe;
  bool a_kcontig, b_kcontig;
  bool ragged_k;
  int M, N;                     // ragged-M: M = total rows R; ragged-K: per-expert output M
  const int* offsets;
  int E;
  int seg_len;
  void* C;
  long long ldc, sCe;
  int epi;
  int act;                      // 0 relu, 1 gelu_tanh
  const float* bias;            // [E, N] or nullptr
  const void* aux0;
  const void* aux1;
  void* out1;
  long long ld_aux;
  const void* B0x;              // second B operand of EPI_SWIGLU_UP (W3)
  void* out2;                   // second extra output (H3 of EPI_SWIGLU_UP)
  int* status;                  // device status word (bounded-wait timeouts), tcgen05 only
  long long wait_ns;            // bound of each device wait (0: the default, ~2 s)
  int stall;                    // self-test of the timeout path: withhold every load
  // ragged-K weight gradients only: with sgd_w set, the epilogue also applies
  // SGD, sgd_w -= sgd_lr * dW, and rewrites the bf16 copy sgd_wlp (same layout as C)
  float* sgd_w;
  void* sgd_wlp;
  float sgd_lr;
};

// CUDA-core GEMMs serve fp32 layers only; bf16 operands go to the tensor cores.
cudaError_t launch_gemm_simt_f32(const GemmArgs& g, cudaStream_t st);
inline cudaError_t launch_gemm_simt(const GemmArgs& g, cudaStream_t st) {
  if (g.M == 0 || g.N == 0 || g.E == 0) return cudaSuccess;
  if (g.a_type != 0 || g.b_type != 0) return cudaErrorInvalidValue;
  return launch_gemm_simt_f32(g, st);
}

// tcgen05 / TMA grouped GEMM for bf16 operands (gemm_tc.cu).
cudaError_t launch_gemm_tc(const GemmArgs& g, cudaStream_t st);

// fp32 operands on the bf16 tensor cores through a three-term bf16 split of
// each operand (gemm_f32x3.cu): scratch for the expanded operands, and the
// launch; cudaErrorNotSupported (before any launch) for forms, epilogues or
// strides it does not take, and when the scratch is missing or too small.
// `kernels` (optional) receives the number of kernels launched.
size_t gemm_f32x3_scratch_bytes(const GemmArgs& g);
cudaError_t launch_gemm_f32x3(const GemmArgs& g, void* scratch, size_t scratch_bytes,
                              cudaStream_t st, int* kernels = nullptr);
// Device status word values written by kernels (0 = ok).
constexpr int DEV_STATUS_TIMEOUT = 6;

}  // namespace moe
