// Router kernels: gate matmul -> scores -> top-k -> renormalised gates, and
// the router backward (course "Trainable MoE in CUDA", Parts 2, 3 and 6;
// group-limited sigmoid selection and its tie rule from "AI Infra Kernel Lab",
// "Project status").
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Tokens per block: 64, or 16 when 64-token blocks would not fill two
// blocks per SM (152 SMs), so that short batches still spread over the GPU.
constexpr int RT_TOK = 64;
constexpr int RT_TOK_SMALL = 16;
constexpr int RT_BK = 32;     // D chunk staged in shared memory
constexpr int RT_THREADS = 256;

__host__ __device__ constexpr int router_tok_per_block(int T) {
  return T >= RT_TOK * 2 * 152 ? RT_TOK : RT_TOK_SMALL;
}

template <int NJ, int TB>
struct RouterSmem {
  static constexpr int EP = 16 * NJ;
  static constexpr int stage_floats = RT_BK * (TB + 1) + RT_BK * (EP + 1);
  static constexpr int logit_floats = TB * (EP + 1);
  static constexpr int main_floats = stage_floats > logit_floats ? stage_floats : logit_floats;
  static constexpr size_t bytes = sizeof(float) * (size_t)(main_floats + (RT_THREADS / 32) * EP);
};

struct Cand {
  float v;
  int id;
};

// (v, id) beats (v', id'): larger score, equal score -> smaller id.
__device__ __forceinline__ bool better(float v, int id, float v2, int id2) {
  return v > v2 || (v == v2 && id < id2);
}

// Selection keys: the scores, plus the correction bias when there is one
// ("AI Infra Kernel Lab": the bias chooses experts only; gates and their
// gradients use the unbiased scores).  Without a bias the keys are the scores.
template <int NC>
__device__ __forceinline__ void selection_keys(const float (&s)[NC], const float* cb, int lane,
                                               int E, float (&key)[NC]) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int e = lane + 32 * c;
    key[c] = (cb != nullptr && e < E) ? s[c] + cb[e] : s[c];
  }
}
// v[c] held by lane (id % 32) for id = lane + 32 c, broadcast to the warp.
template <int NC>
__device__ __forceinline__ float lane_value(const float (&v)[NC], int lane, int id) {
  float mine = 0.f;
#pragma unroll
  for (int c = 0; c < NC; ++c)
    if (lane + 32 * c == id) mine = v[c];
  return __shfl_sync(0xffffffffu, mine, id & 31);
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, c.v, o);
    int id2 = __shfl_xor_sync(0xffffffffu, c.id, o);
    if (better(v2, id2, c.v, c.id)) { c.v = v2; c.id = id2; }
  }
  return c;
}

// Logits for TB tokens x E_pad experts (E_pad = 16*NJ), then one warp per
// token for score, selection and renormalisation.  Each logit is one fp32
// accumulation over d in ascending order, whatever TB is.
template <typename XT, int NJ, int TB>
__global__ void __launch_bounds__(RT_THREADS)
router_fwd_kernel(const XT* __restrict__ x, const float* __restrict__ wg,
                  const float* __restrict__ logit_bias, RouterArgs a,
                  float* __restrict__ scores, int* __restrict__ idx, float* __restrict__ gate,
                  float* __restrict__ psum_partial) {
  pdl_begin();
  constexpr int EP = 16 * NJ;
  constexpr int NC = (EP + 31) / 32;   // scores per lane
  constexpr int TI = TB / 16;          // tokens per thread in the logits tile
  constexpr int XPT = TB * RT_BK / RT_THREADS, WPT = EP * RT_BK / RT_THREADS;
  static_assert(TB % 16 == 0 && XPT * RT_THREADS == TB * RT_BK && WPT * RT_THREADS == EP * RT_BK,
                "staging splits evenly over the threads");
  // dynamic shared memory: the logits tile ls aliases the staging tiles xs/ws
  extern __shared__ __align__(16) float rsm[];
  float(*xs)[TB + 1] = reinterpret_cast<float(*)[TB + 1]>(rsm);
  float(*ws)[EP + 1] = reinterpret_cast<float(*)[EP + 1]>(rsm + RT_BK * (TB + 1));
  float(*ls)[EP + 1] = reinterpret_cast<float(*)[EP + 1]>(rsm);
  float(*wsum)[EP] = reinterpret_cast<float(*)[EP]>(rsm + RouterSmem<NJ, TB>::main_floats);

  const int T = a.T, D = a.D, E = a.E;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.x * TB;

  float acc[TI][NJ];
#pragma unroll
  for (int i = 0; i < TI; ++i)
#pragma unroll
    for (int j = 0; j < NJ; ++j) acc[i][j] = 0.f;

  // the next D chunk is read into registers while the current one is used
  float xr[XPT], wr[WPT];
  auto fetch = [&](int d0) {
#pragma unroll
    for (int u = 0; u < XPT; ++u) {
      const int l = tid + u * RT_THREADS, tk = l / RT_BK, d = d0 + l % RT_BK, t = t0 + tk;
      xr[u] = (t < T && d < D) ? to_f(x[(size_t)t * D + d]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < WPT; ++u) {
      const int l = tid + u * RT_THREADS, e = l / RT_BK, d = d0 + l % RT_BK;
      wr[u] = (e < E && d < D) ? wg[(size_t)e * D + d] : 0.f;
    }
  };
  fetch(0);
  for (int d0 = 0; d0 < D; d0 += RT_BK) {
#pragma unroll
    for (int u = 0; u < XPT; ++u) {
      const int l = tid + u * RT_THREADS;
      xs[l % RT_BK][l / RT_BK] = xr[u];
    }
#pragma unroll
    for (int u = 0; u < WPT; ++u) {
      const int l = tid + u * RT_THREADS;
      ws[l % RT_BK][l / RT_BK] = wr[u];
    }
    __syncthreads();
    if (d0 + RT_BK < D) fetch(d0 + RT_BK);
#pragma unroll 8
    for (int kk = 0; kk < RT_BK; ++kk) {
      float av[TI], bv[NJ];
#pragma unroll
      for (int i = 0; i < TI; ++i) av[i] = xs[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < NJ; ++j) bv[j] = ws[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < TI; ++i)
#pragma unroll
        for (int j = 0; j < NJ; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < TI; ++i)
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      int e = tx + 16 * j;
      float bias = (logit_bias != nullptr && e < E) ? logit_bias[e] : 0.f;
      ls[ty + 16 * i][e] = acc[i][j] + bias;
    }
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31;
  constexpr int TOK_PER_WARP = TB / (RT_THREADS / 32);
  float colsum[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) colsum[c] = 0.f;

  const int per = E / a.n_groups;
  for (int tt = 0; tt < TOK_PER_WARP; ++tt) {
    const int tk = warp * TOK_PER_WARP + tt;
    const int t = t0 + tk;
    if (t >= T) break;
    float s[NC];
    // score: softmax with max subtraction, or sigmoid
    if (a.score == 0) {
      float m = -FLT_MAX;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        s[c] = (e < E) ? ls[tk][e] : -INFINITY;
        m = fmaxf(m, s[c]);
      }
      m = warp_max(m);
      float z = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        s[c] = (e < E) ? expf(s[c] - m) : 0.f;
        z += s[c];
      }
      z = warp_sum(z);
      float inv = 1.0f / z;
#pragma unroll
      for (int c = 0; c < NC; ++c) s[c] *= inv;
    } else {
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        s[c] = (e < E) ? sigmoidf_(ls[tk][e]) : 0.f;
      }
    }
    float key[NC];
    selection_keys(s, a.corr_bias, lane, E, key);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      int e = lane + 32 * c;
      if (e < E) {
        scores[(size_t)t * E + e] = s[c];
        ls[tk][e] = key[c];   // the warp's own row now holds the selection keys
        colsum[c] += s[c];
      }
    }
    __syncwarp();

    // candidate mask: plain top-k = every expert; grouped = kept groups only
    bool allowed[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) allowed[c] = (lane + 32 * c) < E;
    if (a.n_groups > 1) {
      float gs = -INFINITY;
      if (lane < a.n_groups) {
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int e = lane * per; e < (lane + 1) * per; ++e) {
          float v = ls[tk][e];
          if (v > m1) { m2 = m1; m1 = v; } else if (v > m2) { m2 = v; }
        }
        gs = (per == 1 || a.group_score == 1) ? m1 : m1 + m2;
      }
      bool taken = false;
      unsigned keep = 0u;
      for (int r = 0; r < a.topk_groups; ++r) {
        Cand c;
        c.v = (lane < a.n_groups && !taken) ? gs : -INFINITY;
        c.id = (lane < a.n_groups && !taken) ? lane : 0x7fffffff;
        c = warp_best(c);
        int gsel = c.id;
        if (gsel >= a.n_groups) {   // only reachable with NaN scores
          gsel = __ffs(~keep & ((a.n_groups >= 32) ? 0xffffffffu : ((1u << a.n_groups) - 1u))) - 1;
        }
        keep |= 1u << gsel;
        if (lane == gsel) taken = true;
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        allowed[c] = allowed[c] && ((keep >> (e / per)) & 1u);
      }
    }
    // k rounds of a warp-wide arg-max; ties -> smaller id
    float selv = 0.f, ssum = 0.f;
    int selid = 0;
    for (int j = 0; j < a.k; ++j) {
      Cand best;
      best.v = -INFINITY;
      best.id = 0x7fffffff;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        if (allowed[c] && better(key[c], e, best.v, best.id)) { best.v = key[c]; best.id = e; }
      }
      best = warp_best(best);
      if (best.id >= E) {
        // no comparable candidate left (NaN scores): take the smallest allowed id
        int cand = 0x7fffffff;
#pragma unroll
        for (int c = 0; c < NC; ++c)
          if (allowed[c]) cand = min(cand, lane + 32 * c);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
        best.id = (cand < E) ? cand : 0;
      }
      const float sv = lane_value(s, lane, best.id);   // unbiased score of the pick
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (lane + 32 * c == best.id) allowed[c] = false;
      if (lane == j) { selv = sv; selid = best.id; }
      ssum += sv;   // j order, identical on every lane
    }
    if (lane < a.k) {
      idx[(size_t)t * a.k + lane] = selid;
      gate[(size_t)t * a.k + lane] = selv / ssum;
    }
  }
  // deterministic per-block column sums of the scores (for the aux loss)
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    int e = lane + 32 * c;
    if (e < EP) wsum[warp][e] = colsum[c];
  }
  __syncthreads();
  for (int e = tid; e < E; e += RT_THREADS) {
    float sacc = 0.f;
#pragma unroll
    for (int w = 0; w < RT_THREADS / 32; ++w) sacc += wsum[w][e];
    psum_partial[(size_t)blockIdx.x * E + e] = sacc;
  }
}

// Score, selection and renormalisation from precomputed logits (the bf16
// layers compute logits = x W_g^T + logit_bias on the tensor cores).  One warp
// per token; a warp-private shared row serves the group-limited selection.
// Per-block column sums of the scores feed the aux loss.
template <int NC, int TB>
__global__ void __launch_bounds__(256)
router_select_kernel(const float* __restrict__ logits, RouterArgs a, float* __restrict__ scores,
                     int* __restrict__ idx, float* __restrict__ gate,
                     float* __restrict__ psum_partial) {
  pdl_begin();
  constexpr int EP = 32 * NC;
  __shared__ float rows[8][EP];
  __shared__ float wsum[8][EP];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, T = a.T;
  const int per = E / a.n_groups;
  float colsum[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) colsum[c] = 0.f;
  for (int tt = 0; tt < TB / 8; ++tt) {
    const int t = blockIdx.x * TB + warp * (TB / 8) + tt;
    if (t >= T) break;
    float s[NC];
    if (a.score == 0) {
      float m = -FLT_MAX;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        s[c] = (e < E) ? logits[(size_t)t * E + e] : -INFINITY;
        m = fmaxf(m, s[c]);
      }
      m = warp_max(m);
      float z = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        s[c] = (e < E) ? expf(s[c] - m) : 0.f;
        z += s[c];
      }
      z = warp_sum(z);
      float inv = 1.0f / z;
#pragma unroll
      for (int c = 0; c < NC; ++c) s[c] *= inv;
    } else {
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        s[c] = (e < E) ? sigmoidf_(logits[(size_t)t * E + e]) : 0.f;
      }
    }
    float key[NC];
    selection_keys(s, a.corr_bias, lane, E, key);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      int e = lane + 32 * c;
      if (e < E) {
        scores[(size_t)t * E + e] = s[c];
        rows[warp][e] = key[c];
        colsum[c] += s[c];
      }
    }
    __syncwarp();
    bool allowed[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) allowed[c] = (lane + 32 * c) < E;
    if (a.n_groups > 1) {
      float gs = -INFINITY;
      if (lane < a.n_groups) {
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int e = lane * per; e < (lane + 1) * per; ++e) {
          float v = rows[warp][e];
          if (v > m1) { m2 = m1; m1 = v; } else if (v > m2) { m2 = v; }
        }
        gs = (per == 1 || a.group_score == 1) ? m1 : m1 + m2;
      }
      bool taken = false;
      unsigned keep = 0u;
      for (int r = 0; r < a.topk_groups; ++r) {
        Cand c;
        c.v = (lane < a.n_groups && !taken) ? gs : -INFINITY;
        c.id = (lane < a.n_groups && !taken) ? lane : 0x7fffffff;
        c = warp_best(c);
        int gsel = c.id;
        if (gsel >= a.n_groups)
          gsel = __ffs(~keep & ((a.n_groups >= 32) ? 0xffffffffu : ((1u << a.n_groups) - 1u))) - 1;
        keep |= 1u << gsel;
        if (lane == gsel) taken = true;
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        allowed[c] = allowed[c] && ((keep >> (e / per)) & 1u);
      }
    }
    float selv = 0.f, ssum = 0.f;
    int selid = 0;
    for (int j = 0; j < a.k; ++j) {
      Cand best;
      best.v = -INFINITY;
      best.id = 0x7fffffff;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        int e = lane + 32 * c;
        if (allowed[c] && better(key[c], e, best.v, best.id)) { best.v = key[c]; best.id = e; }
      }
      best = warp_best(best);
      if (best.id >= E) {
        int cand = 0x7fffffff;
#pragma unroll
        for (int c = 0; c < NC; ++c)
          if (allowed[c]) cand = min(cand, lane + 32 * c);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
        best.id = (cand < E) ? cand : 0;
      }
      const float sv = lane_value(s, lane, best.id);   // unbiased score of the pick
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (lane + 32 * c == best.id) allowed[c] = false;
      if (lane == j) { selv = sv; selid = best.id; }
      ssum += sv;
    }
    if (lane < a.k) {
      idx[(size_t)t * a.k + lane] = selid;
      gate[(size_t)t * a.k + lane] = selv / ssum;
    }
    __syncwarp();
  }
#pragma unroll
  for (int c = 0; c < NC; ++c) wsum[warp][lane + 32 * c] = colsum[c];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 256) {
    float sacc = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sacc += wsum[w][e];
    psum_partial[(size_t)blockIdx.x * E + e] = sacc;
  }
}

// Round-to-nearest-even bf16 copy of an fp32 tensor (the router weight).
__global__ void __launch_bounds__(256)
cast_bf16_kernel(const float* __restrict__ src, bf16* __restrict__ dst, long long n) {
  pdl_begin();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

// Router backward, one warp per token:
//   dsel_j = (dg_j - sum_i dg_i g_i) / S,  S = sum_j s_{idx_j}
//   ds_e   = aux_row_e + [e selected] dsel
//   softmax: dl = s (ds - <ds, s>);  sigmoid: dl = ds s (1 - s)
template <int NC>
__global__ void __launch_bounds__(256)
router_bwd_kernel(const float* __restrict__ scores, const int* __restrict__ idx,
                  const float* __restrict__ gate, const float* __restrict__ dgate,
                  const float* __restrict__ aux_row, RouterArgs a,
                  float* __restrict__ dlogits, bf16* __restrict__ dlogits_lp, int* dbg) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int E = a.E, k = a.k;
  float s[NC], ds[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    int e = lane + 32 * c;
    s[c] = (e < E) ? scores[(size_t)t * E + e] : 0.f;
    ds[c] = (e < E && aux_row != nullptr) ? aux_row[e] : 0.f;
  }
  // gather S and <dg, g> in j order (identical on every lane)
  float S = 0.f, inner = 0.f;
  for (int j = 0; j < k; ++j) {
    int e = idx[(size_t)t * k + j];
    // an expert id only selects a lane and a register here (never an
    // address); a MOE_DEBUG build still reports and skips one out of range
    if (kDebugChecks && !valid_expert(e, E, dbg)) continue;
    float sv = __shfl_sync(0xffffffffu, s[0], e & 31);
#pragma unroll
    for (int c = 1; c < NC; ++c) {
      float v = __shfl_sync(0xffffffffu, s[c], e & 31);
      if ((e >> 5) == c) sv = v;
    }
    S += sv;
    inner += dgate[(size_t)t * k + j] * gate[(size_t)t * k + j];
  }
  for (int j = 0; j < k; ++j) {
    int e = idx[(size_t)t * k + j];
    if (kDebugChecks && !valid_expert(e, E, dbg)) continue;
    float dsel = (dgate[(size_t)t * k + j] - inner) / S;
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if (lane + 32 * c == e) ds[c] += dsel;
  }
  if (a.score == 0) {
    float dot = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) dot += ds[c] * s[c];
    dot = warp_sum(dot);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      int e = lane + 32 * c;
      if (e < E) {
        const float v = s[c] * (ds[c] - dot);
        dlogits[(size_t)t * E + e] = v;
        if (dlogits_lp) dlogits_lp[(size_t)t * E + e] = __float2bfloat16_rn(v);
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      int e = lane + 32 * c;
      if (e < E) {
        const float v = ds[c] * s[c] * (1.0f - s[c]);
        dlogits[(size_t)t * E + e] = v;
        if (dlogits_lp) dlogits_lp[(size_t)t * E + e] = __float2bfloat16_rn(v);
      }
    }
  }
}

}  // namespace

int router_fwd_blocks(int T) {
  const int tb = router_tok_per_block(T);
  return (T + tb - 1) / tb;
}

template <typename XT, int NJ, int TB>
static cudaError_t launch_fwd_tb(const void* x, const float* wg, const float* lb,
                                 const RouterArgs& a, float* scores, int* idx, float* gate,
                                 float* psum, cudaStream_t st) {
  dim3 grid((a.T + TB - 1) / TB);
  const size_t smem = RouterSmem<NJ, TB>::bytes;
  static std::atomic<unsigned long long> attr_done{0};   // per instantiation and device
  cudaError_t e = ensure_dynamic_smem(router_fwd_kernel<XT, NJ, TB>, (int)smem, attr_done);
  if (e != cudaSuccess) return e;
  MOE_LAUNCH(launch_pdl(router_fwd_kernel<XT, NJ, TB>, dim3(grid), dim3(RT_THREADS), smem, st,
      static_cast<const XT*>(x), wg, lb, a, scores, idx, gate, psum));
  return cudaGetLastError();
}

template <typename XT, int NJ>
static cudaError_t launch_fwd_nj(const void* x, const float* wg, const float* lb,
                                 const RouterArgs& a, float* scores, int* idx, float* gate,
                                 float* psum, cudaStream_t st) {
  if (router_tok_per_block(a.T) == RT_TOK)
    return launch_fwd_tb<XT, NJ, RT_TOK>(x, wg, lb, a, scores, idx, gate, psum, st);
  return launch_fwd_tb<XT, NJ, RT_TOK_SMALL>(x, wg, lb, a, scores, idx, gate, psum, st);
}

template <typename XT>
static cudaError_t launch_fwd_t(const void* x, const float* wg, const float* lb,
                                const RouterArgs& a, float* scores, int* idx, float* gate,
                                float* psum, cudaStream_t st) {
  if (a.E <= 16) return launch_fwd_nj<XT, 1>(x, wg, lb, a, scores, idx, gate, psum, st);
  if (a.E <= 32) return launch_fwd_nj<XT, 2>(x, wg, lb, a, scores, idx, gate, psum, st);
  if (a.E <= 64) return launch_fwd_nj<XT, 4>(x, wg, lb, a, scores, idx, gate, psum, st);
  if (a.E <= 128) return launch_fwd_nj<XT, 8>(x, wg, lb, a, scores, idx, gate, psum, st);
  return launch_fwd_nj<XT, 16>(x, wg, lb, a, scores, idx, gate, psum, st);
}

// fp32 layers: logits on CUDA cores inside the fused router kernel.
cudaError_t launch_router_fwd(int dtype, const void* x, const float* wg, const float* logit_bias,
                              const RouterArgs& a, float* scores, int* idx, float* gate,
                              float* psum_partial, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (dtype != 0) return cudaErrorInvalidValue;
  return launch_fwd_t<float>(x, wg, logit_bias, a, scores, idx, gate, psum_partial, st);
}

cudaError_t launch_router_bwd(const float* scores, const int* idx, const float* gate,
                              const float* dgate, const float* aux_row, const RouterArgs& a,
                              float* dlogits, void* dlogits_lp, cudaStream_t st, int* dbg) {
  if (a.T == 0) return cudaSuccess;
  dim3 grid((a.T + 7) / 8);
  bf16* lp = static_cast<bf16*>(dlogits_lp);
  if (a.E <= 32) MOE_LAUNCH(launch_pdl(router_bwd_kernel<1>, dim3(grid), dim3(256), 0, st, scores, idx, gate, dgate, aux_row, a, dlogits, lp, dbg));
  else if (a.E <= 64) MOE_LAUNCH(launch_pdl(router_bwd_kernel<2>, dim3(grid), dim3(256), 0, st, scores, idx, gate, dgate, aux_row, a, dlogits, lp, dbg));
  else if (a.E <= 128) MOE_LAUNCH(launch_pdl(router_bwd_kernel<4>, dim3(grid), dim3(256), 0, st, scores, idx, gate, dgate, aux_row, a, dlogits, lp, dbg));
  else MOE_LAUNCH(launch_pdl(router_bwd_kernel<8>, dim3(grid), dim3(256), 0, st, scores, idx, gate, dgate, aux_row, a, dlogits, lp, dbg));
  return cudaGetLastError();
}

template <int TB>
static cudaError_t launch_select_tb(const float* logits, const RouterArgs& a, float* scores, int* idx,
                                   float* gate, float* psum_partial, cudaStream_t st) {
  dim3 grid((a.T + TB - 1) / TB);
  if (a.E <= 32) MOE_LAUNCH(launch_pdl(router_select_kernel<1, TB>, dim3(grid), dim3(256), 0, st, logits, a, scores, idx, gate, psum_partial));
  else if (a.E <= 64) MOE_LAUNCH(launch_pdl(router_select_kernel<2, TB>, dim3(grid), dim3(256), 0, st, logits, a, scores, idx, gate, psum_partial));
  else if (a.E <= 128) MOE_LAUNCH(launch_pdl(router_select_kernel<4, TB>, dim3(grid), dim3(256), 0, st, logits, a, scores, idx, gate, psum_partial));
  else MOE_LAUNCH(launch_pdl(router_select_kernel<8, TB>, dim3(grid), dim3(256), 0, st, logits, a, scores, idx, gate, psum_partial));
  return cudaGetLastError();
}

cudaError_t launch_router_select(const float* logits, const RouterArgs& a, float* scores, int* idx,
                                 float* gate, float* psum_partial, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  if (router_tok_per_block(a.T) == RT_TOK)
    return launch_select_tb<RT_TOK>(logits, a, scores, idx, gate, psum_partial, st);
  return launch_select_tb<RT_TOK_SMALL>(logits, a, scores, idx, gate, psum_partial, st);
}

cudaError_t launch_cast_bf16(const float* src, void* dst, long long n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  MOE_LAUNCH(launch_pdl(cast_bf16_kernel, dim3((int)blocks), dim3(256), 0, st, src, static_cast<bf16*>(dst), n));
  return cudaGetLastError();
}

}  // namespace moe
