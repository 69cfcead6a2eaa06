// Host-side helpers shared by the translation units of the C ABI
// (moe_api.cu: the layer's entry points; ep_api.cu: the expert-parallel
// phases): workspace layout, argument validation, launch bookkeeping.
// Internal to the library.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {
namespace api {

inline thread_local int g_launches = 0;

// Optional per-kernel timing: CUDA events recorded around every kernel launch
// of the calling thread's last entry-point call.
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
inline thread_local bool g_prof = false;
inline thread_local std::vector<ProfRec> g_prof_recs;
inline thread_local int g_prof_n = 0;

// Every kernel launch is also an NVTX range named after the step it runs
// ("gemm_dw1", "combine_fused", ...), so that profilers can select kernels
// by step (ncu --nvtx --nvtx-include "gemm_dw1/").  NVTX v3 is header-only:
// with no tool attached a range costs a check of a function pointer.
inline void prof_begin(const char* name, cudaStream_t st) {
  nvtxRangePushA(name);
  if (!g_prof || g_prof_n >= 4096) return;
  if (g_prof_n == (int)g_prof_recs.size()) {
    ProfRec r{name, nullptr, nullptr};
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return;
    g_prof_recs.push_back(r);
  }
  g_prof_recs[g_prof_n].name = name;
  cudaEventRecord(g_prof_recs[g_prof_n].a, st);
}
inline void prof_end(cudaStream_t st) {
  nvtxRangePop();
  if (!g_prof || g_prof_n >= 4096 || g_prof_n >= (int)g_prof_recs.size()) return;
  cudaEventRecord(g_prof_recs[g_prof_n].b, st);
  ++g_prof_n;
}

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline size_t esize(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// split-K factor of the router weight gradient dW_g = dlogits^T x
// Token chunks of the router weight gradient dW_g = dlogits^T x: each chunk
// is one ragged-K segment of the grouped GEMM and a fixed-order sum adds the
// partial products.  Enough chunks that chunks x output tiles fill two waves
// of 152 SMs (output tiles of 128 x 256 on the tensor-core path, 128 x 128 on
// the CUDA-core one), at least one per 2048 tokens, each at least 64
// tokens, at most 64 chunks.
inline int dwg_splits(const moe_config& c) {
  const bool tc = c.dtype == MOE_BF16;
  const long long bn = tc ? 256 : 128;
  const long long tiles = (((long long)c.E + 127) / 128) * (((long long)c.D + bn - 1) / bn);
  long long s = (2 * 152 + tiles - 1) / tiles;
  if (s < c.T / 2048) s = c.T / 2048;
  if (s > c.T / 64) s = c.T / 64;
  if (s > 64) s = 64;
  return s < 1 ? 1 : (int)s;
}

struct Layout {
  size_t status, scores, idx, gate, counts, offsets, chunk, src_tok, slot_of, psum, sq, aux_row;
  size_t xe, h1, h3, a, ye, dy, dye, dgate, dh1, dh3, dxe, dlogits, dwg_part, dx;
  size_t logits, wg_lp, dl_lp;   // bf16 layers: router logits, bf16 W_g, bf16 dlogits
  // shared-expert branch (n_shared > 0): H1s, H3s, As [T, Fs]; Ys [T, D]; bf16
  // dY [T, D]; dH1s, dH3s [T, Fs]; dXs [T, D] (all bf16)
  size_t hs1, hs3, as, ys, dy_lp, dhs1, dhs3, dxs;
  // stand-ins for gradients a training step's caller leaves NULL: the router
  // gradient and biases always; the expert weights' of fp32 layers (their SGD
  // runs after the GEMMs; bf16 layers apply it inside the GEMM epilogues and
  // store nothing)
  size_t g_wg, g_b1, g_b2, g_w1, g_w3, g_w2;
  // fp32 layers: expanded operands of the expert GEMMs on the tensor cores
  size_t f32x3, f32x3_bytes;
  size_t total;
};

// Scratch of the fp32 expert GEMMs on the tensor cores (gemm_f32x3.cu) for R
// expert rows over E experts: the largest pair of expanded operands among
// the layer's expert GEMMs (six bf16 terms, 12 bytes, per fp32 value).  0,
// and the CUDA-core GEMMs serve, for bf16 layers, for layers with D F below
// F32X3_MIN_DF (their few-microsecond GEMMs would pay more for the operand
// expansion launches than they gain) and past F32X3_MAX_BYTES.  The choice
// depends on the layer alone, so an expert-parallel rank makes the one the
// single-device step makes.
constexpr size_t F32X3_MAX_BYTES = (size_t)1 << 30;
constexpr size_t F32X3_MIN_DF = (size_t)1 << 16;
inline size_t f32x3_scratch(const moe_config& c, size_t R, size_t E) {
  if (c.dtype != MOE_F32 || (size_t)c.D * (size_t)c.F < F32X3_MIN_DF) return 0;
  const size_t D = (size_t)c.D, F = (size_t)c.F, u = 12;
  auto r = [](size_t b) { return (b + 255) & ~(size_t)255; };
  size_t m = r(R * D * u) + r(E * F * D * u);                          // up (K = D)
  m = std::max(m, r(R * F * u) + r(E * D * F * u));                   // down, dXe (K = F)
  if (c.act == MOE_ACT_SWIGLU) m = std::max(m, 2 * (r(R * F * u) + r(E * D * F * u)));   // dXe, 2 pairs
  m = std::max(m, r(R * D * u) + r(R * F * u) + r((E + 1) * 4));      // dW (6R rows)
  return m > F32X3_MAX_BYTES ? 0 : m;
}

// expert_buffers = false: the source-side workspace of an expert-parallel
// rank, without the buffers of the expert MLPs (H, A, dH and the fp32
// gradient stand-ins), which live with the rows a rank receives.
inline Layout make_layout(const moe_config& c, bool expert_buffers = true) {
  Layout L{};
  const size_t T = (size_t)c.T, D = (size_t)c.D, F = (size_t)c.F, E = (size_t)c.E;
  const size_t R = T * (size_t)c.k;
  const size_t es = esize(c.dtype);
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o += align_up(bytes > 0 ? bytes : 1);
    return at;
  };
  L.status = take(16);
  L.scores = take(T * E * 4);
  L.idx = take(R * 4);
  L.gate = take(R * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.chunk = take((size_t)route_chunks((long long)R) * E * 4);
  L.src_tok = take(R * 4);
  L.slot_of = take(R * 4);
  L.psum = take((size_t)router_fwd_blocks(c.T) * E * 4);
  L.sq = take((size_t)combine_blocks(c.T) * 8);
  L.aux_row = take(E * 4);
  L.xe = take(R * D * es);
  L.h1 = expert_buffers ? take(R * F * es) : 0;
  L.h3 = expert_buffers && swiglu ? take(R * F * es) : 0;
  L.a = expert_buffers ? take(R * F * es) : 0;
  L.ye = take(R * D * es);
  L.dy = take(T * D * 4);
  L.dye = take(R * D * es);
  L.dgate = take(R * 4);
  L.dh1 = expert_buffers ? take(R * F * es) : 0;
  L.dh3 = expert_buffers && swiglu ? take(R * F * es) : 0;
  L.dxe = take(R * D * es);
  L.dlogits = take(T * E * 4);
  L.dwg_part = take((size_t)dwg_splits(c) * E * D * 4);
  L.dx = take(T * D * 4);
  const bool lp = c.dtype == MOE_BF16;
  L.logits = lp ? take(T * E * 4) : 0;
  L.wg_lp = lp ? take(E * D * 2) : 0;
  L.dl_lp = lp ? take(T * E * 2) : 0;
  if (c.n_shared > 0) {
    const size_t Fs = (size_t)c.n_shared * F;
    L.hs1 = take(T * Fs * 2);
    L.hs3 = take(T * Fs * 2);
    L.as = take(T * Fs * 2);
    L.ys = take(T * D * 2);
    L.dy_lp = take(T * D * 2);
    L.dhs1 = take(T * Fs * 2);
    L.dhs3 = take(T * Fs * 2);
    L.dxs = take(T * D * 2);
  }
  L.g_wg = take(E * D * 4);
  L.g_b1 = c.has_bias ? take(E * F * 4) : 0;
  L.g_b2 = c.has_bias ? take(E * D * 4) : 0;
  if (!lp && expert_buffers) {
    L.g_w1 = take(E * F * D * 4);
    L.g_w3 = swiglu ? take(E * F * D * 4) : 0;
    L.g_w2 = take(E * D * F * 4);
  }
  L.f32x3_bytes = expert_buffers ? f32x3_scratch(c, R, E) : 0;
  L.f32x3 = L.f32x3_bytes ? take(L.f32x3_bytes) : 0;
  L.total = o;
  return L;
}

inline moe_status validate_config(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->D <= 0 || c->F <= 0 || c->E <= 0 || c->k <= 0) return MOE_ERR_INVALID_ARG;
  if (c->act < 0 || c->act > 2 || c->score < 0 || c->score > 1 || c->dtype < 0 || c->dtype > 1 ||
      c->group_score < 0 || c->group_score > 1)
    return MOE_ERR_INVALID_ARG;
  if (c->n_groups <= 0 || c->topk_groups <= 0 || c->topk_groups > c->n_groups)
    return MOE_ERR_INVALID_ARG;
  if (c->E > 256 || c->k > 32 || c->k > c->E) return MOE_ERR_UNSUPPORTED;
  if (c->E % c->n_groups != 0 || c->n_groups > 32) return MOE_ERR_UNSUPPORTED;
  if ((long long)c->k > (long long)c->topk_groups * (c->E / c->n_groups)) return MOE_ERR_UNSUPPORTED;
  if (c->D % 8 != 0 || c->F % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->act == MOE_ACT_SWIGLU && c->has_bias) return MOE_ERR_UNSUPPORTED;
  if (c->dtype == MOE_BF16 && c->E % 8 != 0) return MOE_ERR_UNSUPPORTED;   // TMA row alignment
  if ((long long)c->T * c->k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if ((long long)c->T * c->D >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  if (c->n_shared < 0) return MOE_ERR_INVALID_ARG;
  if (!(c->capacity_factor >= 0.f) || c->capacity_factor > 1e6f) return MOE_ERR_INVALID_ARG;
  if (c->n_shared > 0 && (c->act != MOE_ACT_SWIGLU || c->dtype != MOE_BF16 ||
                          (long long)c->n_shared * c->F > (1LL << 20)))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Device check, once per device: sm_103 only.
inline moe_status check_device() {
  static std::mutex mu;
  static int checked[64] = {0};   // 0 unknown, 1 ok, 2 bad
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (checked[dev] == 0) {
    int maj = 0, min = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    checked[dev] = (maj == 10 && min == 3) ? 1 : 2;
  }
  return checked[dev] == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

// KL: a named kernel launch on stream `st` (counted, optionally timed);
// CK: any other CUDA call.
#define KL(name, expr)                           \
  do {                                           \
    prof_begin(name, st);                        \
    cudaError_t _e = (expr);                     \
    prof_end(st);                                \
    ++g_launches;                                \
    if (_e != cudaSuccess) return MOE_ERR_CUDA;  \
  } while (0)
#define CK(expr)                                 \
  do {                                           \
    cudaError_t _e = (expr);                     \
    if (_e != cudaSuccess) return MOE_ERR_CUDA;  \
  } while (0)

struct Ptrs {
  char* base;
  const Layout* L;
  template <typename T> T* at(size_t off) const { return reinterpret_cast<T*>(base + off); }
};

struct ExpertW {
  const float* w_gate;
  const void* w1;
  const void* w3;
  const void* w2;
  const float* b1;
  const float* b2;
  const float* logit_bias;
  const float* corr_bias;   // selection-only correction bias [E] or nullptr
  const void* ws1;          // shared branch (bf16), or nullptr
  const void* ws3;
  const void* ws2;
};

inline RouterArgs router_args(const moe_config& c, const float* corr_bias = nullptr) {
  RouterArgs a;
  a.T = c.T; a.D = c.D; a.E = c.E; a.k = c.k; a.score = c.score;
  a.n_groups = c.n_groups; a.topk_groups = c.topk_groups; a.group_score = c.group_score;
  a.corr_bias = corr_bias;
  return a;
}

inline GemmArgs gemm_base(const moe_config& c, const Ptrs& P) {
  GemmArgs g{};
  g.status = P.at<int>(P.L->status);
  g.a_type = g.b_type = g.c_type = c.dtype;
  g.offsets = P.at<int>(P.L->offsets);
  g.E = c.E;
  g.act = c.act == MOE_ACT_GELU_TANH ? 1 : 0;
  return g;
}


// Expert GEMMs: tcgen05 tensor cores for bf16 layers; for fp32 layers the
// tensor cores through the three-term split where the rows carry scratch for
// it and the GEMM is of a form it takes, else the CUDA cores.
inline cudaError_t run_gemm(const moe_config& c, const GemmArgs& g, cudaStream_t st,
                            void* f32x3 = nullptr, size_t f32x3_bytes = 0) {
  if (c.dtype == MOE_BF16) return launch_gemm_tc(g, st);
  if (f32x3 != nullptr) {
    int kernels = 0;
    const cudaError_t e = launch_gemm_f32x3(g, f32x3, f32x3_bytes, st, &kernels);
    if (e != cudaErrorNotSupported) {
      g_launches += kernels > 0 ? kernels - 1 : 0;   // the caller counts one
      return e;
    }
  }
  return launch_gemm_simt(g, st);
}

#define RET_IF(expr)                \
  do {                              \
    moe_status _s = (expr);         \
    if (_s != MOE_OK) return _s;    \
  } while (0)


// Row segments of expert-major activations, one segment per expert: the
// single-device step's (all E experts, rows of the workspace) or, in an
// expert-parallel step, the rows a rank received for its local experts.
struct ExpertRows {
  int E;                 // segments (experts)
  int M;                 // rows of the buffers (GEMM M, ragged-K length)
  const int* offsets;    // [E + 1] device: segment e = rows [offsets[e], offsets[e + 1])
  int* status;           // device status word of the bounded waits
  void *xe, *h1, *h3, *a, *ye, *dye, *dh1, *dh3, *dxe;
  void* f32x3;           // fp32 layers: scratch of the tensor-core GEMMs, or nullptr
  size_t f32x3_bytes;
};

inline GemmArgs rows_gemm(const moe_config& c, const ExpertRows& r) {
  GemmArgs g{};
  g.status = r.status;
  g.a_type = g.b_type = g.c_type = c.dtype;
  g.offsets = r.offsets;
  g.E = r.E;
  g.act = c.act == MOE_ACT_GELU_TANH ? 1 : 0;
  return g;
}

// SGD folded into the weight-gradient GEMMs of a bf16 training step: each
// expert weight is updated, and its bf16 copy rewritten, as soon as its
// gradient tile exists (every GEMM reading that copy has run by then).
struct SgdFuse {
  float lr;
  float *w1, *w3, *w2;
  void *w1_lp, *w3_lp, *w2_lp;
  float *ws1, *ws3, *ws2;        // shared branch
  void *ws1_lp, *ws3_lp, *ws2_lp;
};


moe_status experts_forward(const moe_config& c, const ExpertW& w, const ExpertRows& r,
                           cudaStream_t st);
moe_status experts_backward(const moe_config& c, const ExpertW& w, const ExpertRows& r,
                            const moe_grads& gr, const SgdFuse* sgd, cudaStream_t st);
moe_status route_tokens(const moe_config& c, const ExpertW& w, const void* x, const Ptrs& P,
                        cudaStream_t st);
moe_status router_backward(const moe_config& c, const ExpertW& w, const void* x, float* dw_gate,
                           float* dx, const void* extra_dx, const Ptrs& P, cudaStream_t st);

}  // namespace api
}  // namespace moe
