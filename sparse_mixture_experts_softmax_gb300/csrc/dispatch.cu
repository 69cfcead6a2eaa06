// Token dispatch and combine (course "Trainable MoE in CUDA", Part 4), the
// losses (Parts 6 and 7) and the SGD update (Part 7).  No floating-point
// atomics: every reduction has a fixed order, so results are bit-reproducible.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// ---------------------------------------------------------------- dispatch --

// Per-chunk expert histogram of the routed assignments (t, j) in token order.
__global__ void __launch_bounds__(256)
route_count_kernel(const int* __restrict__ idx, long long R, int chunk, int E,
                   int* __restrict__ chunk_counts, int* dbg) {
  pdl_begin();
  __shared__ int hist[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const long long lo = (long long)blockIdx.x * chunk;
  const long long hi = min(lo + chunk, R);
  for (long long f = lo + threadIdx.x; f < hi; f += blockDim.x) {
    int e = idx[f];
    if (valid_expert(e, E, dbg)) atomicAdd(&hist[e], 1);   // integer: order-independent
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// counts[e] = sum over chunks (the routed assignments); with an expert
// capacity `cap` an expert keeps min(counts[e], cap) rows; offsets = exclusive
// scan of the kept counts; chunk_counts[c][e] becomes the rank of chunk c's
// first assignment to expert e among all of e's assignments (token order).
// G = SCAN_THREADS / E groups of E threads: group g owns a contiguous range of
// chunks, sums it, and after the ranges' bases are known (a scan over the
// groups, in order) writes the running ranks of its range.  Integer sums:
// exact in any grouping.
constexpr int SCAN_THREADS = 1024;
__global__ void __launch_bounds__(SCAN_THREADS)
route_scan_kernel(int* __restrict__ cc, int nchunks, int E, int cap, int* __restrict__ counts,
                  int* __restrict__ offsets) {
  pdl_begin();
  __shared__ int part[SCAN_THREADS];   // (group, expert): the range's sum, then its base
  __shared__ int tot[256];
  __shared__ int scan[257];
  const int G = SCAN_THREADS / E;      // E <= 256, so G >= 4
  const int g = threadIdx.x / E, e = threadIdx.x - g * E;
  const bool active = g < G;
  const int per = (nchunks + G - 1) / G;
  const int c0 = active ? min(g * per, nchunks) : 0;
  const int c1 = active ? min(c0 + per, nchunks) : 0;
  int sum = 0;
#pragma unroll 8
  for (int c = c0; c < c1; ++c) sum += cc[(size_t)c * E + e];
  part[threadIdx.x] = sum;
  __syncthreads();
  if (threadIdx.x < E) {
    int run = 0;
    for (int q = 0; q < G; ++q) {
      const int v = part[q * E + threadIdx.x];
      part[q * E + threadIdx.x] = run;
      run += v;
    }
    tot[threadIdx.x] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < E; ++i) {
      scan[i] = run;
      run += min(tot[i], cap);
    }
    scan[E] = run;
  }
  __syncthreads();
  if (threadIdx.x < E) {
    counts[threadIdx.x] = tot[threadIdx.x];
    offsets[threadIdx.x] = scan[threadIdx.x];
  }
  if (threadIdx.x == 0) offsets[E] = scan[E];
  if (active) {
    int run = part[threadIdx.x];
#pragma unroll 8
    for (int c = c0; c < c1; ++c) {
      const int v = cc[(size_t)c * E + e];
      cc[(size_t)c * E + e] = run;
      run += v;
    }
  }
}

// Stable scatter: one warp walks its chunk in token order; lanes holding the
// same expert are ranked by lane id (match_any), so slots keep token order.
// An assignment of rank >= cap within its expert is dropped (slot -1), and so
// is one whose expert id lies outside [0, E) (the count skipped it too).
__global__ void __launch_bounds__(32)
route_scatter_kernel(const int* __restrict__ idx, long long R, int chunk, int k, int E, int cap,
                     const int* __restrict__ chunk_base, const int* __restrict__ offsets,
                     int* __restrict__ src_tok, int* __restrict__ slot_of, int* dbg) {
  pdl_begin();
  __shared__ int cursor[256];
  __shared__ int off[256];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) {
    cursor[e] = chunk_base[(size_t)blockIdx.x * E + e];
    off[e] = offsets[e];
  }
  __syncwarp();
  const long long lo = (long long)blockIdx.x * chunk;
  const long long hi = min(lo + chunk, R);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (long long base = lo; base < hi; base += 32) {
    const long long f = base + lane;
    const bool valid = f < hi;
    int e = valid ? idx[f] : -1;
    if (valid && !valid_expert(e, E, dbg)) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0) {
      const int r = cursor[e] + rank;
      int slot = -1;
      if (r < cap) {
        slot = off[e] + r;
        src_tok[slot] = (int)(f / k);
      }
      slot_of[f] = slot;
    } else if (valid) {
      slot_of[f] = -1;   // an expert id outside [0, E): no slot
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) cursor[e] += __popc(peers);
    __syncwarp();
  }
}

// Xe[slot(t, j), :] = X[t, :] for j < k: one warp per token reads its row
// once (16-byte vectors, 4 in flight per lane) and writes it to its k slots.
template <typename T>
__global__ void __launch_bounds__(256)
gather_kernel(const T* __restrict__ x, const int* __restrict__ slot_of, int Tn, int k, int D,
              T* __restrict__ xe, int* dbg) {
  pdl_begin();
  constexpr int VN = 16 / sizeof(T);
  const long long R = (long long)Tn * k;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int nv = D / VN;
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < Tn; t += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * D);
    const int* so = slot_of + (size_t)t * k;
    int v = lane;
    for (; v + 96 < nv; v += 128) {
      const uint4 a0 = src[v], a1 = src[v + 32], a2 = src[v + 64], a3 = src[v + 96];
      for (int j = 0; j < k; ++j) {
        if (!use_slot(so[j], R, dbg)) continue;   // dropped by the expert capacity
        uint4* dst = reinterpret_cast<uint4*>(xe + (size_t)so[j] * D);
        dst[v] = a0; dst[v + 32] = a1; dst[v + 64] = a2; dst[v + 96] = a3;
      }
    }
    for (; v < nv; v += 32) {
      const uint4 a = src[v];
      for (int j = 0; j < k; ++j)
        if (use_slot(so[j], R, dbg)) reinterpret_cast<uint4*>(xe + (size_t)so[j] * D)[v] = a;
    }
  }
}

// ------------------------------------------------------------------ combine --

constexpr int CB_TOK = 8;    // tokens per block (one per warp)

// Y[t] = sum_j g_tj Ye[slot(t, j)] in j order (fp32), + Ys[t] (the shared-
// expert branch) when given.  With a target it also forms dY = 2 (Y - target)
// / (T D) and a per-block sum of squared errors.
template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ ye, const float* __restrict__ gate,
               const int* __restrict__ slot_of, int Tn, int D, int k, const T* __restrict__ ys,
               float* __restrict__ y,
               const float* __restrict__ target, float* __restrict__ dy, float inv_n,
               double* __restrict__ sq_partial, int* dbg) {
  pdl_begin();
  constexpr int VN = Vec<T>::N;
  const long long R = (long long)Tn * k;
  __shared__ float wpart[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float sq = 0.f;
  for (int tt = 0; tt < CB_TOK / 8; ++tt) {
    const int t = blockIdx.x * CB_TOK + warp * (CB_TOK / 8) + tt;
    if (t >= Tn) break;
    for (int d = lane * VN; d < D; d += 32 * VN) {
      float acc[VN];
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = 0.f;
      for (int j = 0; j < k; ++j) {
        const int s = slot_of[(size_t)t * k + j];
        if (!use_slot(s, R, dbg)) continue;   // dropped by the expert capacity: no output
        const float g = gate[(size_t)t * k + j];
        Vec<T> v;
        v.load(ye + (size_t)s * D + d);
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] = fmaf(g, v.get(i), acc[i]);
      }
      if (ys != nullptr) {   // shared-expert branch, added after the routed sum
        Vec<T> v;
        v.load(ys + (size_t)t * D + d);
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] += v.get(i);
      }
      if (y != nullptr) {
#pragma unroll
        for (int i = 0; i < VN; i += 4)
          *reinterpret_cast<float4*>(y + (size_t)t * D + d + i) =
              make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
      }
      if (target != nullptr) {
#pragma unroll
        for (int i = 0; i < VN; i += 4) {
          float4 tg = *reinterpret_cast<const float4*>(target + (size_t)t * D + d + i);
          float d0 = acc[i] - tg.x, d1 = acc[i + 1] - tg.y, d2 = acc[i + 2] - tg.z,
                d3 = acc[i + 3] - tg.w;
          sq += d0 * d0 + d1 * d1 + d2 * d2 + d3 * d3;
          *reinterpret_cast<float4*>(dy + (size_t)t * D + d + i) =
              make_float4(2.f * d0 * inv_n, 2.f * d1 * inv_n, 2.f * d2 * inv_n, 2.f * d3 * inv_n);
        }
      }
    }
  }
  if (sq_partial != nullptr) {
    sq = warp_sum(sq);
    if (lane == 0) wpart[warp] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
      double s = 0.0;
      for (int w = 0; w < 8; ++w) s += (double)wpart[w];
      sq_partial[blockIdx.x] = s;
    }
  }
}

// Training-step combine with its backward fused (k <= 8): for each token,
// with its k expert rows held in registers,
//   Y[t]  = sum_j g_tj Ye[slot(t, j)] (+ Ys[t])  (j order, as combine_kernel)
//   dY[t] = 2 (Y[t] - target[t]) / (T D)          (MSE seed, never stored)
//   dYe[slot(t, j)] = g_tj dY[t],  dg_tj = <dY[t], Ye[slot(t, j)]>
// with the same arithmetic and order as combine_kernel followed by
// combine_bwd_kernel, so dYe and dg are bit-identical to that pair; one pass
// moves Ye and the target in and dYe out (dY never goes to HBM).  Two tokens
// per warp and one squared-error partial per block of CB_TOK tokens (the
// partial groups its warps' sums differently from combine_kernel, so the MSE
// value may differ from that path in the last bits).
// 128-thread blocks: with the k rows held in registers (~150 per thread), four
// warps per block let three blocks share an SM.
// SHARED: the layer has a shared-expert branch (Ys added, bf16 dY written);
// a separate instantiation keeps the plain kernel's registers down.
constexpr int CT_WARPS = 4;
template <typename T, bool SHARED>
__global__ void __launch_bounds__(32 * CT_WARPS)
combine_train_kernel(const T* __restrict__ ye, const float* __restrict__ gate,
                     const int* __restrict__ slot_of, int Tn, int D, int k,
                     const T* __restrict__ ys, const float* __restrict__ target, float inv_n,
                     double* __restrict__ sq_partial, T* __restrict__ dye,
                     float* __restrict__ dgate, bf16* __restrict__ dy_lp, int* dbg) {
  pdl_begin();
  constexpr int VN = Vec<T>::N;
  constexpr int MAXK = 8;
  const long long R = (long long)Tn * k;
  __shared__ float wpart[CT_WARPS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float sq = 0.f;
  for (int tt = 0; tt < CB_TOK / CT_WARPS; ++tt) {
    const int t = blockIdx.x * CB_TOK + warp * (CB_TOK / CT_WARPS) + tt;
    if (t >= Tn) break;
    int slot[MAXK];
    bool use[MAXK];
    float g[MAXK], dot[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      slot[j] = (j < k) ? slot_of[(size_t)t * k + j] : 0;
      use[j] = j < k && use_slot(slot[j], R, dbg);
      g[j] = (j < k) ? gate[(size_t)t * k + j] : 0.f;
      dot[j] = 0.f;
    }
    for (int d = lane * VN; d < D; d += 32 * VN) {
      Vec<T> v[MAXK];
#pragma unroll
      for (int j = 0; j < MAXK; ++j)
        if (use[j]) v[j].load(ye + (size_t)slot[j] * D + d);
      float acc[VN];
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < MAXK; ++j)
        if (use[j]) {
#pragma unroll
          for (int i = 0; i < VN; ++i) acc[i] = fmaf(g[j], v[j].get(i), acc[i]);
        }
      if constexpr (SHARED) {   // shared-expert branch, added after the routed sum
        Vec<T> u;
        u.load(ys + (size_t)t * D + d);
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] += u.get(i);
      }
      float dv[VN];
#pragma unroll
      for (int i = 0; i < VN; i += 4) {
        const float4 tg = *reinterpret_cast<const float4*>(target + (size_t)t * D + d + i);
        const float d0 = acc[i] - tg.x, d1 = acc[i + 1] - tg.y, d2 = acc[i + 2] - tg.z,
                    d3 = acc[i + 3] - tg.w;
        sq += d0 * d0 + d1 * d1 + d2 * d2 + d3 * d3;
        dv[i] = 2.f * d0 * inv_n;
        dv[i + 1] = 2.f * d1 * inv_n;
        dv[i + 2] = 2.f * d2 * inv_n;
        dv[i + 3] = 2.f * d3 * inv_n;
      }
      if constexpr (SHARED && VN == 8) {   // bf16 dY for the shared branch's GEMMs
        Vec<bf16> q;
#pragma unroll
        for (int i = 0; i < 8; ++i) q.set(i, dv[i]);
        q.store(dy_lp + (size_t)t * D + d);
      }
#pragma unroll
      for (int j = 0; j < MAXK; ++j)
        if (use[j]) {   // a dropped assignment keeps dg = 0
          Vec<T> o;
#pragma unroll
          for (int i = 0; i < VN; ++i) {
            dot[j] = fmaf(dv[i], v[j].get(i), dot[j]);
            o.set(i, g[j] * dv[i]);
          }
          o.store(dye + (size_t)slot[j] * D + d);
        }
    }
#pragma unroll
    for (int j = 0; j < MAXK; ++j)
      if (j < k) {
        const float s2 = warp_sum(dot[j]);
        if (lane == 0) dgate[(size_t)t * k + j] = s2;
      }
  }
  sq = warp_sum(sq);
  if (lane == 0) wpart[warp] = sq;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < CT_WARPS; ++w) s += (double)wpart[w];
    sq_partial[blockIdx.x] = s;
  }
}

// L_mse = sum(sq_partial) / (T D);  P_e = sum_b psum[b][e] / T;  f_e = c_e / (T k);
// aux = E sum_e f_e P_e;  aux_row[e] = alpha E f_e / T (d aux / d s_te, f constant).
// One block, every sum in a fixed order (deterministic).  This GPU's fp64 rate
// is a small fraction of its fp32 rate, so double is kept only for the sum of
// the squared-error partials (which are double already): the score column sums
// use G = FL_THREADS / E groups of E threads (group g takes partial rows g,
// g + G, ... into four fp32 accumulators), folded pairwise over the groups;
// the per-expert terms and their sum are fp32 as well.
constexpr int FL_THREADS = 1024;
__global__ void __launch_bounds__(FL_THREADS)
finalize_losses_kernel(const double* __restrict__ sq_partial, int n_sq,
                       const float* __restrict__ psum, int n_ps, const int* __restrict__ counts,
                       int T, int D, int E, int k, float alpha, float* __restrict__ d_loss,
                       float* __restrict__ aux_row) {
  pdl_begin();
  __shared__ double sq_warp[FL_THREADS / 32];
  __shared__ float col[FL_THREADS];
  __shared__ float term_warp[FL_THREADS / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // squared error: a double per thread, a shuffle tree per warp, warps in order
  double s = 0.0;
  for (int i = tid; i < n_sq; i += FL_THREADS) s += sq_partial[i];
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
  if (lane == 0) sq_warp[warp] = s;
  // score column sums
  const int G = FL_THREADS / E;   // E <= 256, so G >= 4
  const int g = tid / E, e = tid - g * E;
  float P = 0.f;
  if (g < G) {
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
    int b = g;
    for (; b + 3 * G < n_ps; b += 4 * G) {
      p0 += psum[(size_t)b * E + e];
      p1 += psum[(size_t)(b + G) * E + e];
      p2 += psum[(size_t)(b + 2 * G) * E + e];
      p3 += psum[(size_t)(b + 3 * G) * E + e];
    }
    for (; b < n_ps; b += G) p0 += psum[(size_t)b * E + e];
    P = (p0 + p1) + (p2 + p3);
  }
  col[tid] = P;
  __syncthreads();
  // fold the groups: those from Gp on (Gp = largest power of two <= G) onto
  // the first ones, then halve Gp until group 0 holds the column sums
  int Gp = 1;
  while (2 * Gp <= G) Gp *= 2;
  if (g >= Gp && g < G) col[tid - Gp * E] += col[tid];
  __syncthreads();
  for (int w = Gp / 2; w > 0; w >>= 1) {
    if (g < w) col[tid] += col[tid + w * E];
    __syncthreads();
  }
  float term = 0.f;
  if (tid < E) {
    const float f = (float)counts[tid] / ((float)T * (float)k);
    term = f * (col[tid] / (float)T);
    if (aux_row != nullptr) aux_row[tid] = alpha * (float)E * f / (float)T;
  }
  for (int o = 16; o > 0; o >>= 1) term += __shfl_down_sync(0xffffffffu, term, o);
  if (lane == 0) term_warp[warp] = term;
  __syncthreads();
  if (tid == 0 && d_loss != nullptr) {
    double sq = 0.0;
    float aux = 0.f;
    for (int w = 0; w < FL_THREADS / 32; ++w) {
      sq += sq_warp[w];
      aux += term_warp[w];
    }
    d_loss[0] = (float)(sq / ((double)T * (double)D));
    d_loss[1] = (float)E * aux;
  }
}

// dYe[slot(t,j)] = g_tj dY[t];  dg_tj = <dY[t], Ye[slot(t,j)]>; one warp per token.
template <typename T, int MAXK>
__global__ void __launch_bounds__(256)
combine_bwd_kernel(const float* __restrict__ dy, const T* __restrict__ ye,
                   const float* __restrict__ gate, const int* __restrict__ slot_of, int Tn, int D,
                   int k, T* __restrict__ dye, float* __restrict__ dgate, int* dbg) {
  pdl_begin();
  constexpr int VN = Vec<T>::N;
  const long long R = (long long)Tn * k;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= Tn) return;
  int slot[MAXK];
  bool use[MAXK];
  float g[MAXK], dot[MAXK];
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    slot[j] = (j < k) ? slot_of[(size_t)t * k + j] : 0;
    use[j] = j < k && use_slot(slot[j], R, dbg);
    g[j] = (j < k) ? gate[(size_t)t * k + j] : 0.f;
    dot[j] = 0.f;
  }
  for (int d = lane * VN; d < D; d += 32 * VN) {
    float dv[VN];
#pragma unroll
    for (int i = 0; i < VN; i += 4) {
      float4 q = *reinterpret_cast<const float4*>(dy + (size_t)t * D + d + i);
      dv[i] = q.x; dv[i + 1] = q.y; dv[i + 2] = q.z; dv[i + 3] = q.w;
    }
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (use[j]) {   // dropped by the expert capacity: dg = 0
        Vec<T> v, o;
        v.load(ye + (size_t)slot[j] * D + d);
#pragma unroll
        for (int i = 0; i < VN; ++i) {
          dot[j] = fmaf(dv[i], v.get(i), dot[j]);
          o.set(i, g[j] * dv[i]);
        }
        o.store(dye + (size_t)slot[j] * D + d);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    if (j < k) {
      float s = warp_sum(dot[j]);
      if (lane == 0) dgate[(size_t)t * k + j] = s;
    }
  }
}

// dX[t] += sum_j dXe[slot(t, j)] in j order (scatter-back of the expert rows
// onto the router's dX term), then + extra[t] (the shared-expert branch's dX)
// when given; one warp per token, 16-byte vectors along D.
template <typename T>
__global__ void __launch_bounds__(256)
scatter_back_add_kernel(float* __restrict__ dx, const T* __restrict__ dxe,
                        const int* __restrict__ slot_of, int Tn, int D, int k,
                        const T* __restrict__ extra, int* dbg) {
  pdl_begin();
  constexpr int VN = Vec<T>::N;
  const long long R = (long long)Tn * k;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= Tn) return;
  for (int d = lane * VN; d < D; d += 32 * VN) {
    float acc[VN];
#pragma unroll
    for (int i = 0; i < VN; i += 4) {
      const float4 q = *reinterpret_cast<const float4*>(dx + (size_t)t * D + d + i);
      acc[i] = q.x; acc[i + 1] = q.y; acc[i + 2] = q.z; acc[i + 3] = q.w;
    }
    for (int j = 0; j < k; ++j) {
      const int s = slot_of[(size_t)t * k + j];
      if (!use_slot(s, R, dbg)) continue;   // dropped by the expert capacity
      Vec<T> v;
      v.load(dxe + (size_t)s * D + d);
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] += v.get(i);
    }
    if (extra != nullptr) {   // the shared branch's dX row, added last
      Vec<T> v;
      v.load(extra + (size_t)t * D + d);
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] += v.get(i);
    }
#pragma unroll
    for (int i = 0; i < VN; i += 4)
      *reinterpret_cast<float4*>(dx + (size_t)t * D + d + i) =
          make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
  }
}

// out[e, n] = sum over rows of segment e of src[r, n], for db.  A cluster of
// CS_SPLIT CTAs shares one column block of one segment: CTA z sums rows
// [lo + n z / S, lo + n (z+1) / S) (8 warps, rows w, w+8, ... with four
// accumulators per thread), the warps' sums are added in warp order, and CTA
// 0 adds the CTAs' sums in rank order through distributed shared memory.
// The order depends on the segment's rows alone, so a segment gives the same
// bits wherever it sits.  VEC: one 16-byte load per row for the thread's
// V = 16 / sizeof(T) columns (N a multiple of V, src 16-byte aligned).
constexpr int CS_SPLIT = 8;
template <typename T, bool VEC>
__global__ void __cluster_dims__(1, 1, CS_SPLIT) __launch_bounds__(256)
segment_colsum_kernel(const T* __restrict__ src, const int* __restrict__ offsets, int N,
                      float* __restrict__ out) {
  pdl_begin();
  namespace cg = cooperative_groups;
  constexpr int V = 16 / (int)sizeof(T), COLS = 32 * V;
  __shared__ float part[8][COLS];
  __shared__ float csum[COLS];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e = blockIdx.y;
  const int z = (int)blockIdx.z;   // the cluster spans z: z is the CTA's rank in it
  const int c0 = blockIdx.x * COLS + lane * V;
  const int lo = offsets[e], n = offsets[e + 1] - lo;
  const int r0 = lo + (int)((long long)n * z / CS_SPLIT);
  const int r1 = lo + (int)((long long)n * (z + 1) / CS_SPLIT);

  float acc[4][V];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[j][v] = 0.f;
  auto add_row = [&](float (&a)[V], int r) {
    const T* p = src + (size_t)r * N + c0;
    if (VEC) {
      const uint4 q = *reinterpret_cast<const uint4*>(p);
      const T* h = reinterpret_cast<const T*>(&q);
#pragma unroll
      for (int v = 0; v < V; ++v) a[v] += to_f(h[v]);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (c0 + v < N) a[v] += to_f(p[v]);
    }
  };
  if (c0 < N) {
    int r = r0 + w;
    for (; r + 24 < r1; r += 32) {
      add_row(acc[0], r);
      add_row(acc[1], r + 8);
      add_row(acc[2], r + 16);
      add_row(acc[3], r + 24);
    }
    for (; r < r1; r += 8) add_row(acc[0], r);
  }
#pragma unroll
  for (int v = 0; v < V; ++v) part[w][lane * V + v] = (acc[0][v] + acc[1][v]) + (acc[2][v] + acc[3][v]);
  __syncthreads();
  for (int c = threadIdx.x; c < COLS; c += blockDim.x) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += part[i][c];
    csum[c] = s;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();   // every CTA's csum is complete
  if (z == 0) {
    for (int c = threadIdx.x; c < COLS; c += blockDim.x) {
      const int col = blockIdx.x * COLS + c;
      if (col >= N) continue;
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < CS_SPLIT; ++q) s += cluster.map_shared_rank(csum, q)[c];
      out[(size_t)e * N + col] = s;
    }
  }
  cluster.sync();   // the other CTAs keep their shared memory until CTA 0 has read it
}

__global__ void __launch_bounds__(256)
sum_partials_kernel(const float* __restrict__ p, int nparts, long long n, float* __restrict__ out) {
  pdl_begin();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int q = 0; q < nparts; ++q) s += p[(size_t)q * n + i];
    out[i] = s;
  }
}

// theta <- theta - lr * grad (fp32 master); optional bf16 working copy (RNE).
// Several tensors per launch: element i of the concatenated float4 index
// space belongs to the first tensor whose running end4 exceeds i.
struct SgdList {
  float* w[SGD_MAX_TENSORS];
  const float* g[SGD_MAX_TENSORS];
  bf16* lp[SGD_MAX_TENSORS];
  long long end4[SGD_MAX_TENSORS];   // running sums of n / 4
  int count;
};
__global__ void __launch_bounds__(256) sgd_kernel(const SgdList L, float lr) {
  pdl_begin();
  const long long total = L.end4[L.count - 1];
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    int t = 0;
    while (i >= L.end4[t]) ++t;
    const long long j = i - (t > 0 ? L.end4[t - 1] : 0);
    float4 wv = reinterpret_cast<float4*>(L.w[t])[j];
    const float4 gv = reinterpret_cast<const float4*>(L.g[t])[j];
    wv.x = fmaf(-lr, gv.x, wv.x);
    wv.y = fmaf(-lr, gv.y, wv.y);
    wv.z = fmaf(-lr, gv.z, wv.z);
    wv.w = fmaf(-lr, gv.w, wv.w);
    reinterpret_cast<float4*>(L.w[t])[j] = wv;
    if (L.lp[t] != nullptr) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(wv.x, wv.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(wv.z, wv.w);
      uint2 q;
      q.x = *reinterpret_cast<uint32_t*>(&lo);
      q.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(L.lp[t])[j] = q;
    }
  }
}

inline int grid_for(long long n, int per_block, int cap) {
  long long b = (n + per_block - 1) / per_block;
  if (b < 1) b = 1;
  return (int)(b < cap ? b : cap);
}

}  // namespace

int route_chunk(long long R) {
  long long c = (R + ROUTE_TARGET_CHUNKS - 1) / ROUTE_TARGET_CHUNKS;
  c = (c + 31) / 32 * 32;
  return (int)(c < ROUTE_CHUNK_MIN ? ROUTE_CHUNK_MIN : c > ROUTE_CHUNK_MAX ? ROUTE_CHUNK_MAX : c);
}
int route_chunks(long long R) {
  const int c = route_chunk(R);
  return (int)((R + c - 1) / c);
}

cudaError_t launch_route_count(const int* idx, long long R, int E, int* chunk_counts,
                               cudaStream_t st, int* dbg) {
  int nc = route_chunks(R);
  if (nc == 0) return cudaSuccess;
  MOE_LAUNCH(launch_pdl(route_count_kernel, dim3(nc), dim3(256), 0, st, idx, R, route_chunk(R), E, chunk_counts, dbg));
  return cudaGetLastError();
}

cudaError_t launch_route_scan(int* chunk_counts, int nchunks, int E, int cap, int* counts,
                              int* offsets, cudaStream_t st) {
  MOE_LAUNCH(launch_pdl(route_scan_kernel, dim3(1), dim3(SCAN_THREADS), 0, st, chunk_counts, nchunks, E, cap, counts, offsets));
  return cudaGetLastError();
}

cudaError_t launch_route_scatter(const int* idx, long long R, int k, int E, int cap,
                                 const int* chunk_base, const int* offsets, int* src_tok,
                                 int* slot_of, cudaStream_t st, int* dbg) {
  int nc = route_chunks(R);
  if (nc == 0) return cudaSuccess;
  MOE_LAUNCH(launch_pdl(route_scatter_kernel, dim3(nc), dim3(32), 0, st, idx, R, route_chunk(R), k, E, cap, chunk_base, offsets,
                                          src_tok, slot_of, dbg));
  return cudaGetLastError();
}

cudaError_t launch_gather(int dtype, const void* x, const int* slot_of, int T, int k, int D,
                          void* xe, cudaStream_t st, int* dbg) {
  if (T == 0) return cudaSuccess;
  int grid = grid_for(T, 8, 152 * 16);
  if (dtype == 1)
    MOE_LAUNCH(launch_pdl(gather_kernel<bf16>, dim3(grid), dim3(256), 0, st, static_cast<const bf16*>(x), slot_of, T, k, D,
                                              static_cast<bf16*>(xe), dbg));
  else
    MOE_LAUNCH(launch_pdl(gather_kernel<float>, dim3(grid), dim3(256), 0, st, static_cast<const float*>(x), slot_of, T, k, D,
                                               static_cast<float*>(xe), dbg));
  return cudaGetLastError();
}

int combine_blocks(int T) { return (T + CB_TOK - 1) / CB_TOK; }

cudaError_t launch_combine(int dtype, const void* ye, const float* gate, const int* slot_of, int T,
                           int D, int k, const void* ys, float* y, const float* target, float* dy,
                           double* sq_partial, cudaStream_t st, float inv_n, int* dbg) {
  if (T == 0) return cudaSuccess;
  if (inv_n == 0.f) inv_n = 1.0f / ((float)T * (float)D);
  int grid = combine_blocks(T);
  if (dtype == 1)
    MOE_LAUNCH(launch_pdl(combine_kernel<bf16>, dim3(grid), dim3(256), 0, st, static_cast<const bf16*>(ye), gate, slot_of, T, D, k,
                                               static_cast<const bf16*>(ys), y, target, dy, inv_n,
                                               sq_partial, dbg));
  else
    MOE_LAUNCH(launch_pdl(combine_kernel<float>, dim3(grid), dim3(256), 0, st, static_cast<const float*>(ye), gate, slot_of, T, D,
                                                k, static_cast<const float*>(ys), y, target, dy,
                                                inv_n, sq_partial, dbg));
  return cudaGetLastError();
}

cudaError_t launch_combine_train(int dtype, const void* ye, const float* gate, const int* slot_of,
                                 int T, int D, int k, const void* ys, const float* target,
                                 double* sq_partial, void* dye, float* dgate, void* dy_lp,
                                 cudaStream_t st, float inv_n, int* dbg) {
  // the shared branch exists only for bf16 layers and comes with both Ys and dY
  const bool shared = ys != nullptr;
  if (k > 8 || (shared && (dy_lp == nullptr || dtype != 1))) return cudaErrorInvalidValue;
  if (T == 0) return cudaSuccess;
  if (inv_n == 0.f) inv_n = 1.0f / ((float)T * (float)D);
  const int grid = combine_blocks(T);
  if (dtype == 1 && shared)
    MOE_LAUNCH(launch_pdl(combine_train_kernel<bf16, true>, dim3(grid), dim3(32 * CT_WARPS), 0, st,
        static_cast<const bf16*>(ye), gate, slot_of, T, D, k, static_cast<const bf16*>(ys), target,
        inv_n, sq_partial, static_cast<bf16*>(dye), dgate, static_cast<bf16*>(dy_lp), dbg));
  else if (dtype == 1)
    MOE_LAUNCH(launch_pdl(combine_train_kernel<bf16, false>, dim3(grid), dim3(32 * CT_WARPS), 0, st,
        static_cast<const bf16*>(ye), gate, slot_of, T, D, k, nullptr, target, inv_n, sq_partial,
        static_cast<bf16*>(dye), dgate, nullptr, dbg));
  else
    MOE_LAUNCH(launch_pdl(combine_train_kernel<float, false>, dim3(grid), dim3(32 * CT_WARPS), 0, st,
        static_cast<const float*>(ye), gate, slot_of, T, D, k, nullptr, target, inv_n,
        sq_partial, static_cast<float*>(dye), dgate, nullptr, dbg));
  return cudaGetLastError();
}

cudaError_t launch_finalize_losses(const double* sq_partial, int n_sq, const float* psum_partial,
                                   int n_ps, const int* counts, int T, int D, int E, int k,
                                   float alpha, float* d_loss, float* aux_row, cudaStream_t st) {
  MOE_LAUNCH(launch_pdl(finalize_losses_kernel, dim3(1), dim3(FL_THREADS), 0, st, sq_partial, n_sq, psum_partial, n_ps, counts, T,
                                                   D, E, k, alpha, d_loss, aux_row));
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(int dtype, const float* dy, const void* ye, const float* gate,
                               const int* slot_of, int T, int D, int k, void* dye, float* dgate,
                               cudaStream_t st, int* dbg) {
  if (T == 0) return cudaSuccess;
  int grid = (T + 7) / 8;
  if (dtype == 1) {
    if (k <= 8)
      MOE_LAUNCH(launch_pdl(combine_bwd_kernel<bf16, 8>, dim3(grid), dim3(256), 0, st, dy, static_cast<const bf16*>(ye), gate,
                                                        slot_of, T, D, k, static_cast<bf16*>(dye),
                                                        dgate, dbg));
    else
      MOE_LAUNCH(launch_pdl(combine_bwd_kernel<bf16, 32>, dim3(grid), dim3(256), 0, st, dy, static_cast<const bf16*>(ye), gate,
                                                         slot_of, T, D, k, static_cast<bf16*>(dye),
                                                         dgate, dbg));
  } else {
    if (k <= 8)
      MOE_LAUNCH(launch_pdl(combine_bwd_kernel<float, 8>, dim3(grid), dim3(256), 0, st, dy, static_cast<const float*>(ye), gate,
                                                         slot_of, T, D, k,
                                                         static_cast<float*>(dye), dgate, dbg));
    else
      MOE_LAUNCH(launch_pdl(combine_bwd_kernel<float, 32>, dim3(grid), dim3(256), 0, st, dy, static_cast<const float*>(ye), gate,
                                                          slot_of, T, D, k,
                                                          static_cast<float*>(dye), dgate, dbg));
  }
  return cudaGetLastError();
}

cudaError_t launch_scatter_back_add(int dtype, float* dx, const void* dxe, const int* slot_of,
                                    int T, int D, int k, const void* extra, cudaStream_t st,
                                    int* dbg) {
  if (T == 0) return cudaSuccess;
  const int grid = (T + 7) / 8;
  if (dtype == 1)
    MOE_LAUNCH(launch_pdl(scatter_back_add_kernel<bf16>, dim3(grid), dim3(256), 0, st, dx, static_cast<const bf16*>(dxe), slot_of,
                                                         T, D, k, static_cast<const bf16*>(extra),
                                                         dbg));
  else
    MOE_LAUNCH(launch_pdl(scatter_back_add_kernel<float>, dim3(grid), dim3(256), 0, st, dx, static_cast<const float*>(dxe),
                                                          slot_of, T, D, k,
                                                          static_cast<const float*>(extra), dbg));
  return cudaGetLastError();
}

cudaError_t launch_segment_colsum(int dtype, const void* src, const int* offsets, int E, int N,
                                  float* out, cudaStream_t st) {
  if (E == 0 || N == 0) return cudaSuccess;
  const bool aligned = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  if (dtype == 1) {
    const dim3 grid((N + 255) / 256, E, CS_SPLIT);
    const bf16* s = static_cast<const bf16*>(src);
    if (aligned && N % 8 == 0)
      MOE_LAUNCH(launch_pdl(segment_colsum_kernel<bf16, true>, grid, dim3(256), 0, st, s, offsets, N, out));
    else
      MOE_LAUNCH(launch_pdl(segment_colsum_kernel<bf16, false>, grid, dim3(256), 0, st, s, offsets, N, out));
  } else {
    const dim3 grid((N + 127) / 128, E, CS_SPLIT);
    const float* s = static_cast<const float*>(src);
    if (aligned && N % 4 == 0)
      MOE_LAUNCH(launch_pdl(segment_colsum_kernel<float, true>, grid, dim3(256), 0, st, s, offsets, N, out));
    else
      MOE_LAUNCH(launch_pdl(segment_colsum_kernel<float, false>, grid, dim3(256), 0, st, s, offsets, N, out));
  }
  return cudaGetLastError();
}

cudaError_t launch_sum_partials(const float* partials, int nparts, long long n, float* out,
                                cudaStream_t st) {
  MOE_LAUNCH(launch_pdl(sum_partials_kernel, dim3(grid_for(n, 256, 152 * 8)), dim3(256), 0, st, partials, nparts, n, out));
  return cudaGetLastError();
}

cudaError_t launch_sgd(const SgdTensor* tensors, int count, float lr, cudaStream_t st) {
  if (count < 1 || count > SGD_MAX_TENSORS) return cudaErrorInvalidValue;
  SgdList L{};
  long long total = 0;
  int n = 0;
  for (int i = 0; i < count; ++i) {
    if (tensors[i].n == 0) continue;
    total += tensors[i].n / 4;   // every parameter tensor holds a multiple of 8 elements
    L.w[n] = tensors[i].w;
    L.g[n] = tensors[i].g;
    L.lp[n] = static_cast<bf16*>(tensors[i].w_lp);
    L.end4[n] = total;
    ++n;
  }
  if (n == 0) return cudaSuccess;
  L.count = n;
  MOE_LAUNCH(launch_pdl(sgd_kernel, dim3(grid_for(total, 256, 152 * 16)), dim3(256), 0, st, L, lr));
  return cudaGetLastError();
}

cudaError_t launch_fill_zero(void* p, size_t bytes, cudaStream_t st) {
  return cudaMemsetAsync(p, 0, bytes, st);
}

}  // namespace moe
