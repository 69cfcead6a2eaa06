// Grouped GEMMs on CUDA cores (fp32 FFMA), used where the operands are fp32:
// the expert MLPs of fp32 layers and the router's dW_g / dX products.  Course
// "Trainable MoE in CUDA", Part 1 (matmul variants, bias add) and Part 5
// (expert MLP forward and backward over each expert's slice of rows).
//
// Tile 128x128x16, 256 threads (two blocks per SM), 8x8 outputs per thread,
// register-prefetched double buffering.  Each operand tile is fetched with
// 128-bit loads along its contiguous dimension (K for x W^T / dY W operands,
// M or N for the ragged-K weight gradients) wherever the leading dimension
// keeps them 16-byte aligned, and written to shared memory k-major (a
// transpose in registers for the K-contiguous ones).  Three operand forms
// (see GemmArgs in kernels.h):
//   FORM 0  C[r,n] = sum_k A[r,k] B_e[n,k]   ragged M (x W^T)
//   FORM 1  C[r,n] = sum_k A[r,k] B_e[k,n]   ragged M (x W)
//   FORM 2  C_e[m,n] = sum_{r in e} A[r,m] B[r,n]   ragged K (weight gradients)
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace simt {

constexpr int BM = 128, BN = 128, BK = 16, NT = 256;

template <typename T>
__device__ __forceinline__ float ld_f(const void* p, size_t i) {
  return to_f(static_cast<const T*>(p)[i]);
}
__device__ __forceinline__ float ld_rt(const void* p, size_t i, int type) {
  return type == 1 ? ld_f<bf16>(p, i) : ld_f<float>(p, i);
}
__device__ __forceinline__ void st_rt(void* p, size_t i, float v, int type) {
  if (type == 1) static_cast<bf16*>(p)[i] = __float2bfloat16_rn(v);
  else static_cast<float*>(p)[i] = v;
}

// Four consecutive elements of row `row` of a row-major matrix (leading
// dimension ld), columns col0 .. col0 + 3; entries with row >= row_lim or
// column >= col_lim read as zero.  One 128-bit load when `vec` (fp32, 16-byte
// aligned rows and col0) and the four are in range.
template <typename T>
__device__ __forceinline__ float4 load4(const T* p, long long ld, int row, int row_lim, int col0,
                                        int col_lim, bool vec) {
  if (row >= row_lim) return make_float4(0.f, 0.f, 0.f, 0.f);
  const T* q = p + (size_t)row * ld + col0;
  if constexpr (sizeof(T) == 4) {
    if (vec && col0 + 3 < col_lim) return *reinterpret_cast<const float4*>(q);
  }
  float v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = (col0 + i < col_lim) ? to_f(q[i]) : 0.f;
  return make_float4(v[0], v[1], v[2], v[3]);
}

__device__ __forceinline__ int seg_lo(const GemmArgs& g, int e, int total) {
  if (g.offsets) return g.offsets[e];
  long long v = (long long)e * g.seg_len;
  return (int)(v < total ? v : total);
}
__device__ __forceinline__ int seg_hi(const GemmArgs& g, int e, int total) {
  if (g.offsets) return g.offsets[e + 1];
  long long v = (long long)(e + 1) * g.seg_len;
  return (int)(v < total ? v : total);
}

template <typename TA, typename TB, int FORM, int EPI>
__global__ void __launch_bounds__(NT, 2) gemm_simt_kernel(const GemmArgs g) {
  pdl_begin();
  constexpr bool AK = FORM != 2;   // A element (m, k) has k contiguous
  constexpr bool BKC = FORM == 0;  // B element (k, n) has k contiguous
  constexpr bool RAGK = FORM == 2;
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Bs[2][BK][BN + 4];
  __shared__ int tile_start[258];
  __shared__ int sel[3];

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int n0 = blockIdx.y * BN;
  int e, m0, lo, hi;   // ragged-M: rows [lo, hi) of expert e; ragged-K: reduction rows
  if (!RAGK) {
    // map the linear tile index onto (expert, m-tile)
    const int E = g.E;
    for (int i = tid; i < E; i += NT) {
      int l = seg_lo(g, i, g.M), h = seg_hi(g, i, g.M);
      tile_start[i + 1] = (h - l + BM - 1) / BM;
    }
    if (tid == 0) { tile_start[0] = 0; sel[0] = -1; }
    __syncthreads();
    if (tid == 0)
      for (int i = 1; i <= E; ++i) tile_start[i] += tile_start[i - 1];
    __syncthreads();
    const int tile = blockIdx.x;
    for (int i = tid; i < E; i += NT)
      if (tile >= tile_start[i] && tile < tile_start[i + 1]) {
        sel[0] = i;
        sel[1] = tile - tile_start[i];
      }
    __syncthreads();
    e = sel[0];
    if (e < 0) return;
    lo = seg_lo(g, e, g.M);
    hi = seg_hi(g, e, g.M);
    m0 = lo + sel[1] * BM;
  } else {
    e = blockIdx.z;
    m0 = blockIdx.x * BM;
    lo = seg_lo(g, e, g.K0);
    hi = seg_hi(g, e, g.K0);
  }

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  // one or two (A, B, K) pairs; ragged-K has a single pair over rows [lo, hi)
  const int npairs = (!RAGK && g.A1 != nullptr && g.K1 > 0) ? 2 : 1;
  for (int pair = 0; pair < npairs; ++pair) {
    const TA* A = static_cast<const TA*>(pair == 0 ? g.A0 : g.A1);
    const TB* B = static_cast<const TB*>(pair == 0 ? g.B0 : g.B1);
    if (!RAGK) B += (size_t)e * g.sBe;
    const int kbeg = RAGK ? lo : 0;
    const int kend = RAGK ? hi : (pair == 0 ? g.K0 : g.K1);
    const int mlim = RAGK ? g.M : hi;
    if (kend <= kbeg) continue;

    // 512 four-element vectors per operand tile, two per thread
    const bool vec_a = (g.lda % 4) == 0 && (AK ? (kbeg % 4) == 0 : true);
    const bool vec_b = (g.ldb % 4) == 0 && (BKC ? (kbeg % 4) == 0 : true);
    float4 ra[2], rb[2];
    auto load_tiles = [&](int k0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = tid + h * NT;
        if (AK) ra[h] = load4(A, g.lda, m0 + (q >> 2), mlim, k0 + (q & 3) * 4, kend, vec_a);
        else ra[h] = load4(A, g.lda, k0 + (q >> 5), kend, m0 + (q & 31) * 4, mlim, vec_a);
        if (BKC) rb[h] = load4(B, g.ldb, n0 + (q >> 2), g.N, k0 + (q & 3) * 4, kend, vec_b);
        else rb[h] = load4(B, g.ldb, k0 + (q >> 5), kend, n0 + (q & 31) * 4, g.N, vec_b);
      }
    };
    auto store_tiles = [&](int buf) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = tid + h * NT;
        if (AK) {
          const int m = q >> 2, kq = (q & 3) * 4;
          As[buf][kq][m] = ra[h].x;
          As[buf][kq + 1][m] = ra[h].y;
          As[buf][kq + 2][m] = ra[h].z;
          As[buf][kq + 3][m] = ra[h].w;
        } else {
          *reinterpret_cast<float4*>(&As[buf][q >> 5][(q & 31) * 4]) = ra[h];
        }
        if (BKC) {
          const int n = q >> 2, kq = (q & 3) * 4;
          Bs[buf][kq][n] = rb[h].x;
          Bs[buf][kq + 1][n] = rb[h].y;
          Bs[buf][kq + 2][n] = rb[h].z;
          Bs[buf][kq + 3][n] = rb[h].w;
        } else {
          *reinterpret_cast<float4*>(&Bs[buf][q >> 5][(q & 31) * 4]) = rb[h];
        }
      }
    };

    __syncthreads();
    load_tiles(kbeg);
    store_tiles(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = kbeg; k0 < kend; k0 += BK) {
      const bool more = k0 + BK < kend;
      if (more) load_tiles(k0 + BK);
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        float a[8], b[8];
        const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
        const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
        const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
        const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
        a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
        a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
        b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
        b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      if (more) {
        store_tiles(buf ^ 1);
        __syncthreads();
        buf ^= 1;
      }
    }
  }

  // epilogue
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    const bool rok = RAGK ? (r < g.M) : (r < hi);
    if (!rok) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (c >= g.N) continue;
      float v = acc[i][j];
      const size_t ci = RAGK ? (size_t)e * g.sCe + (size_t)r * g.ldc + c : (size_t)r * g.ldc + c;
      const size_t ai = (size_t)r * g.ld_aux + c;
      switch (EPI) {
        case EPI_STORE:
          if (g.bias) v += g.bias[(size_t)e * g.N + c];
          st_rt(g.C, ci, v, g.c_type);
          break;
        case EPI_ACT_FWD: {
          float h = v + (g.bias ? g.bias[(size_t)e * g.N + c] : 0.f);
          st_rt(g.out1, ci, h, g.c_type);
          st_rt(g.C, ci, g.act == 0 ? fmaxf(h, 0.f) : gelu_tanh_f(h), g.c_type);
          break;
        }
        case EPI_SWIGLU_FWD: {
          float h1 = ld_rt(g.aux0, ai, g.c_type);
          st_rt(g.out1, ci, v, g.c_type);
          st_rt(g.C, ci, silu_f(h1) * v, g.c_type);
          break;
        }
        case EPI_ACT_BWD: {
          float h = ld_rt(g.aux0, ai, g.c_type);
          float dh = g.act == 0 ? (h > 0.f ? v : 0.f) : v * gelu_tanh_grad_f(h);
          st_rt(g.C, ci, dh, g.c_type);
          break;
        }
        case EPI_SWIGLU_BWD: {
          float h1 = ld_rt(g.aux0, ai, g.c_type);
          float h3 = ld_rt(g.aux1, ai, g.c_type);
          st_rt(g.C, ci, v * h3 * silu_grad_f(h1), g.c_type);
          st_rt(g.out1, ci, v * silu_f(h1), g.c_type);
          break;
        }
      }
    }
  }
}

// FORM 0 / 1 are ragged-M (B k-contiguous / n-contiguous), FORM 2 ragged-K.
template <typename TA, typename TB, int FORM, int EPI>
cudaError_t launch_form(const GemmArgs& g, cudaStream_t st) {
  if constexpr (FORM != 2) {
    dim3 grid((g.M + BM - 1) / BM + g.E, (g.N + BN - 1) / BN);
    MOE_LAUNCH(launch_pdl(gemm_simt_kernel<TA, TB, FORM, EPI>, dim3(grid), dim3(NT), 0, st, g));
  } else {
    dim3 grid((g.M + BM - 1) / BM, (g.N + BN - 1) / BN, g.E);
    MOE_LAUNCH(launch_pdl(gemm_simt_kernel<TA, TB, 2, EPI>, dim3(grid), dim3(NT), 0, st, g));
  }
  return cudaGetLastError();
}

// Only the (form, epilogue) pairs the layer uses are instantiated.
template <typename TA, typename TB>
cudaError_t launch_expert_forms(const GemmArgs& g, cudaStream_t st) {
  const int form = g.ragged_k ? 2 : (g.b_kcontig ? 0 : 1);
  if (form == 0) {
    if (g.epi == EPI_STORE) return launch_form<TA, TB, 0, EPI_STORE>(g, st);
    if (g.epi == EPI_ACT_FWD) return launch_form<TA, TB, 0, EPI_ACT_FWD>(g, st);
    if (g.epi == EPI_SWIGLU_FWD) return launch_form<TA, TB, 0, EPI_SWIGLU_FWD>(g, st);
  } else if (form == 1) {
    if (g.epi == EPI_STORE) return launch_form<TA, TB, 1, EPI_STORE>(g, st);
    if (g.epi == EPI_ACT_BWD) return launch_form<TA, TB, 1, EPI_ACT_BWD>(g, st);
    if (g.epi == EPI_SWIGLU_BWD) return launch_form<TA, TB, 1, EPI_SWIGLU_BWD>(g, st);
  } else {
    if (g.epi == EPI_STORE) return launch_form<TA, TB, 2, EPI_STORE>(g, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace simt
}  // namespace moe
