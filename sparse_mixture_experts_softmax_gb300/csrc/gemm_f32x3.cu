// fp32 expert GEMMs on the bf16 tensor cores.  Course "Trainable MoE in
// CUDA", Part 1 (matmul variants) and Part 5 (expert MLP forward and
// backward); the fp32 layers keep their fp32 tolerance.
//
// Each fp32 operand value is split into three bf16 terms,
//   x1 = RN(x),  x2 = RN(x - x1),  x3 = RN(x - x1 - x2),
// (both differences are exact in fp32), which together hold x to about
// 2^-24 of |x|.  A product a b is then the fp32-accumulated sum of the six
// term products of order up to a2 b2:
//   a1 b1 + a1 b2 + a2 b1 + a1 b3 + a2 b2 + a3 b1,
// each exact in fp32 (8 x 8 significant bits); the three left out are below
// 2^-26 of |a b|.  The six products of a dot product over K become one bf16
// GEMM over 6 K: the A side lays its terms out along the reduction as
// [a3 a2 a1 a2 a1 a1], the B side as [b1 b2 b3 b1 b2 b1], the smallest
// products first: the tensor cores' fp32 accumulation rounds more coarsely
// than IEEE additions, and with a1 b1 last the partial sums stay small while
// the other five blocks are added.  So the
// tensor-core grouped GEMM (gemm_tc.cu) runs unchanged on operands expanded
// here:
//   ragged M, A [M, K] K-major          -> A' [M, 6K]
//   ragged M, B [E, N, K] K-major (NT)  -> B' [E, N, 6K]
//   ragged M, B [E, K, N] N-major (NN)  -> B' [E, 6K, N]
//   ragged K, A [R, M] and B [R, N]     -> [6R, M] and [6R, N]: expert e's
//            rows [o_e, o_e+1) become six blocks of its rows at 6 o_e
//            (offsets scaled by 6).
// The GEMM stores fp32 (+ bias); the activation and its backward, which the
// CUDA-core GEMM applies in its epilogue, run as elementwise passes over that
// output with the same functions.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

// a launch counted in n_k (kernels launched by this call)
#define MOE_LAUNCH_N(expr) \
  do {                     \
    MOE_LAUNCH(expr);      \
    ++n_k;                 \
  } while (0)

namespace moe {
namespace {

// The three bf16 terms of x.
__device__ __forceinline__ void split3(float x, bf16 (&t)[3]) {
  t[0] = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(t[0]);
  t[1] = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(t[1]);
  t[2] = __float2bfloat16_rn(r2);
}

// Term index of reduction block b (0..5) on side A (0) or B (1); constant
// once the block loop is unrolled, so the terms stay in registers.
template <int SIDE>
__device__ __forceinline__ constexpr int term_of(int b) {
  // A: 3 2 1 2 1 1    B: 1 2 3 1 2 1   (0-based below, nibble b)
  return ((SIDE == 0 ? 0x001012 : 0x010210) >> (4 * b)) & 0xF;
}

// Eight consecutive values -> their term `which` as eight packed bf16.
__device__ __forceinline__ uint4 pack_term(const bf16 (&t)[8][3], int which) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h;
    h.x = t[2 * i][which];
    h.y = t[2 * i + 1][which];
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The terms of eight consecutive fp32 values at p (16-byte aligned).
__device__ __forceinline__ void split8(const float* p, bf16 (&t)[8][3]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  split3(a.x, t[0]);
  split3(a.y, t[1]);
  split3(a.z, t[2]);
  split3(a.w, t[3]);
  split3(b.x, t[4]);
  split3(b.y, t[5]);
  split3(b.z, t[6]);
  split3(b.w, t[7]);
}

// One operand's expansion.  kind 0: rows of K values (row stride ldx) ->
// rows of 6K, the blocks side by side.  kind 1: [E][K][N] (row stride N) ->
// [E][6K][N], the six K blocks one below the other.  kind 2: row segments
// [R][M] (row stride ldx, segment e = rows [o_e, o_e+1)) -> [6R][M], segment
// e's six blocks of its rows starting at row 6 o_e; rows past o_E belong to
// no segment and are not written.  Eight values per work item.
struct ExpandJob {
  const float* X;
  long long ldx;
  long long rows;        // kind 0: rows; kind 1: E; kind 2: R
  int K;                 // kind 0 and 1: reduction length; kind 2: M (row length)
  int N;                 // kind 1: row length
  const int* offsets;    // kind 2: [E + 1]
  int E;
  bf16* Y;
  int kind;
  long long items;       // eight-value work items
  int blocks;            // blocks of the launch given to this job
};

template <int SIDE>
__device__ __forceinline__ void run_job(const ExpandJob& j, long long first, long long stride) {
  const int end = j.kind == 2 ? j.offsets[j.E] : 0;
  for (long long i = first; i < j.items; i += stride) {
    bf16 t[8][3];
    if (j.kind == 0) {
      const int kq = j.K / 8;
      const long long r = i / kq;
      const int k = (int)(i - r * kq) * 8;
      split8(j.X + r * j.ldx + k, t);
      bf16* y = j.Y + r * 6LL * j.K + k;
#pragma unroll
      for (int b = 0; b < 6; ++b)
        *reinterpret_cast<uint4*>(y + (long long)b * j.K) = pack_term(t, term_of<SIDE>(b));
    } else if (j.kind == 1) {
      const int nq = j.N / 8;
      const long long row = i / nq;          // e * K + k
      const int c = (int)(i - row * nq) * 8;
      const long long e = row / j.K;
      const int k = (int)(row - e * j.K);
      split8(j.X + row * j.N + c, t);
#pragma unroll
      for (int b = 0; b < 6; ++b)
        *reinterpret_cast<uint4*>(j.Y + ((e * 6 + b) * j.K + k) * j.N + c) =
            pack_term(t, term_of<SIDE>(b));
    } else {
      const int M = j.K, mq = M / 8;
      const long long r = i / mq;
      if (r >= end) continue;
      const int c = (int)(i - r * mq) * 8;
      int lo = 0, hi = j.E;   // the segment holding r: largest e with offsets[e] <= r
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (j.offsets[mid] <= r) lo = mid; else hi = mid;
      }
      const long long o = j.offsets[lo], rows = j.offsets[lo + 1] - o, jr = r - o;
      split8(j.X + r * j.ldx + c, t);
#pragma unroll
      for (int b = 0; b < 6; ++b)
        *reinterpret_cast<uint4*>(j.Y + (6 * o + b * rows + jr) * M + c) =
            pack_term(t, term_of<SIDE>(b));
    }
  }
}

// A GEMM's two operand expansions in one launch: blocks [0, a.blocks) take
// job a (side A), the rest job b (side B).
__global__ void expand_pair_kernel(const ExpandJob a, const ExpandJob b) {
  pdl_begin();
  if ((int)blockIdx.x < a.blocks)
    run_job<0>(a, (long long)blockIdx.x * blockDim.x + threadIdx.x, (long long)a.blocks * blockDim.x);
  else
    run_job<1>(b, (long long)(blockIdx.x - a.blocks) * blockDim.x + threadIdx.x,
            (long long)b.blocks * blockDim.x);
}

__global__ void scale_offsets_kernel(const int* __restrict__ in, int n, int* __restrict__ out) {
  pdl_begin();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = 6 * in[i];
}

// A = act(H) over the expert rows of the GEMM output (rows [0, *end) of
// N values, row stride ld).
__global__ void act_fwd_kernel(const float* __restrict__ H, float* __restrict__ A,
                               const int* __restrict__ end, int N, long long ld, int act) {
  pdl_begin();
  const long long n = (long long)*end * N;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / N, o = r * ld + (i - r * N);
    const float h = H[o];
    A[o] = act == 0 ? fmaxf(h, 0.f) : gelu_tanh_f(h);
  }
}

// dH = dA * act'(H), in place over dA (expert rows only).
__global__ void act_bwd_kernel(float* __restrict__ dA, const float* __restrict__ H,
                               const int* __restrict__ end, int N, long long ld, long long ld_h,
                               int act) {
  pdl_begin();
  const long long n = (long long)*end * N;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / N, c = i - r * N, o = r * ld + c;
    const float v = dA[o], h = H[r * ld_h + c];
    dA[o] = act == 0 ? (h > 0.f ? v : 0.f) : v * gelu_tanh_grad_f(h);
  }
}

int grid_of(long long n) {
  const long long b = (n + 255) / 256;
  return (int)(b < 152 * 16 ? (b < 1 ? 1 : b) : 152 * 16);
}

ExpandJob job(int kind, const void* X, long long ldx, long long rows, int K, int N,
              const int* offsets, int E, bf16* Y) {
  ExpandJob j{static_cast<const float*>(X), ldx, rows, K, N, offsets, E, Y, kind, 0, 0};
  j.items = kind == 0 ? rows * (K / 8) : kind == 1 ? rows * K * (long long)(N / 8) : rows * (K / 8);
  j.blocks = grid_of(j.items);
  return j;
}

size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

size_t gemm_f32x3_scratch_bytes(const GemmArgs& g) {
  if (g.ragged_k)
    return up256((size_t)6 * g.K0 * g.M * 2) + up256((size_t)6 * g.K0 * g.N * 2) +
           up256((size_t)(g.E + 1) * 4);
  const size_t per = up256((size_t)g.M * 6 * g.K0 * 2) + up256((size_t)g.E * g.N * 6 * g.K0 * 2);
  const size_t pair = (g.A1 != nullptr && g.K1 > 0)
                          ? up256((size_t)g.M * 6 * g.K1 * 2) + up256((size_t)g.E * g.N * 6 * g.K1 * 2)
                          : 0;
  return per + pair;
}

cudaError_t launch_gemm_f32x3(const GemmArgs& g, void* scratch, size_t scratch_bytes, cudaStream_t st,
                              int* kernels) {
  int n_k = 0;
  if (kernels) *kernels = 0;
  if (g.M == 0 || g.N == 0 || g.E == 0) return cudaSuccess;
  if (g.a_type != 0 || g.b_type != 0 || g.c_type != 0 || g.offsets == nullptr || g.sgd_w != nullptr)
    return cudaErrorNotSupported;
  const bool fwd = g.epi == EPI_ACT_FWD, bwd = g.epi == EPI_ACT_BWD;
  if (g.epi != EPI_STORE && !fwd && !bwd) return cudaErrorNotSupported;
  if (g.ragged_k && g.epi != EPI_STORE) return cudaErrorNotSupported;
  if (scratch == nullptr || scratch_bytes < gemm_f32x3_scratch_bytes(g)) return cudaErrorNotSupported;
  char* s = static_cast<char*>(scratch);
  auto take = [&](size_t bytes) {
    char* p = s;
    s += up256(bytes);
    return p;
  };
  GemmArgs t = g;
  t.a_type = t.b_type = 1;
  t.bias = (g.epi == EPI_ACT_BWD) ? nullptr : g.bias;
  t.epi = EPI_STORE;
  if (g.ragged_k) {
    // weight gradient: A [R, M], B [R, N], segments of rows
    if (g.lda % 4 || g.ldb % 4 || g.M % 8 || g.N % 8) return cudaErrorNotSupported;
    const long long R = g.K0;
    bf16* A = reinterpret_cast<bf16*>(take((size_t)6 * R * g.M * 2));
    bf16* B = reinterpret_cast<bf16*>(take((size_t)6 * R * g.N * 2));
    int* off6 = reinterpret_cast<int*>(take((size_t)(g.E + 1) * 4));
    MOE_LAUNCH_N(launch_pdl(scale_offsets_kernel, dim3(1), dim3(256), 0, st, g.offsets, g.E + 1, off6));
    const ExpandJob ja = job(2, g.A0, g.lda, R, g.M, 0, g.offsets, g.E, A);
    const ExpandJob jb = job(2, g.B0, g.ldb, R, g.N, 0, g.offsets, g.E, B);
    MOE_LAUNCH_N(launch_pdl(expand_pair_kernel, dim3(ja.blocks + jb.blocks), dim3(256), 0, st, ja, jb));
    t.A0 = A;
    t.lda = g.M;
    t.B0 = B;
    t.ldb = g.N;
    t.K0 = (int)(6 * R);
    t.offsets = off6;
    const cudaError_t e = launch_gemm_tc(t, st);
    if (kernels) *kernels = n_k + 1;
    return e;
  }
  // ragged M: A [M, K] K-major; B per expert K-major (NT) or N-major (NN),
  // its rows packed (row stride K or N, expert stride N K)
  if (!g.a_kcontig) return cudaErrorNotSupported;
  const int pairs = (g.A1 != nullptr && g.K1 > 0) ? 2 : 1;
  if (pairs == 2 && g.K0 != g.K1) return cudaErrorNotSupported;   // one row stride for both
  for (int q = 0; q < pairs; ++q) {
    const int K = q == 0 ? g.K0 : g.K1;
    const float* Aq = static_cast<const float*>(q == 0 ? g.A0 : g.A1);
    const float* Bq = static_cast<const float*>(q == 0 ? g.B0 : g.B1);
    const long long ldb_want = g.b_kcontig ? K : g.N;
    if (K % 8 || g.lda % 4 || g.N % 8 || g.ldb != ldb_want || g.sBe != (long long)g.N * K)
      return cudaErrorNotSupported;
    bf16* A = reinterpret_cast<bf16*>(take((size_t)g.M * 6 * K * 2));
    bf16* B = reinterpret_cast<bf16*>(take((size_t)g.E * g.N * 6 * K * 2));
    const ExpandJob ja = job(0, Aq, g.lda, g.M, K, 0, nullptr, 0, A);
    const ExpandJob jb = g.b_kcontig ? job(0, Bq, K, (long long)g.E * g.N, K, 0, nullptr, 0, B)
                                     : job(1, Bq, g.N, g.E, K, g.N, nullptr, 0, B);
    MOE_LAUNCH_N(launch_pdl(expand_pair_kernel, dim3(ja.blocks + jb.blocks), dim3(256), 0, st, ja, jb));
    if (q == 0) {
      t.A0 = A;
      t.B0 = B;
      t.K0 = 6 * K;
    } else {
      t.A1 = A;
      t.B1 = B;
      t.K1 = 6 * K;
    }
    t.lda = 6LL * K;   // both pairs have the same K in every caller (F for dXe)
    t.ldb = g.b_kcontig ? 6LL * K : g.N;
    t.sBe = (long long)g.N * 6 * K;
  }
  if (fwd) t.C = g.out1;   // H = acc + bias, then A = act(H)
  cudaError_t e = launch_gemm_tc(t, st);
  if (e != cudaSuccess) return e;
  ++n_k;
  if (fwd)
    MOE_LAUNCH_N(launch_pdl(act_fwd_kernel, dim3(grid_of((long long)g.M * g.N)), dim3(256), 0, st,
                          static_cast<const float*>(g.out1), static_cast<float*>(g.C),
                          g.offsets + g.E, g.N, g.ldc, g.act));
  if (bwd)
    MOE_LAUNCH_N(launch_pdl(act_bwd_kernel, dim3(grid_of((long long)g.M * g.N)), dim3(256), 0, st,
                          static_cast<float*>(g.C), static_cast<const float*>(g.aux0),
                          g.offsets + g.E, g.N, g.ldc, g.ld_aux, g.act));
  if (kernels) *kernels = n_k;
  return cudaGetLastError();
}

}  // namespace moe
