// Grouped expert GEMMs on the 5th-generation tensor cores (sm_103a), bf16
// operands with fp32 accumulation in tensor memory.  Course "Trainable MoE in
// CUDA", Part 5 ("Expert MLP Forward and Backward": up/down projections,
// biases, activation, and the backward for inputs, weights and biases over
// each expert's slice of rows); the SwiGLU form W2(SiLU(W1 x) * W3 x) is the
// one of "AI Infra Kernel Lab", "Numerical contracts".
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: 2-D / 3-D tiled bulk-tensor loads, 128-byte
//               swizzle, into a 4-stage shared-memory ring (mbarrier tx count);
//   warp 1      allocates 512 TMEM columns, issues tcgen05.mma (M=128, N=256,
//               K=16) from one lane, frees ring stages with tcgen05.commit;
//   warps 2..9  epilogue, two warps per TMEM lane quarter (each takes half of
//               the tile's columns): tcgen05.ld of the fp32 accumulator, a
//               swizzled shared-memory transpose per 16-column chunk so that
//               every global access is coalesced, bias / activation / SwiGLU
//               (and their backward, and the fused SGD update of weight
//               gradients) applied in registers.
// Two 256-column accumulators let the epilogue of one tile overlap the main
// loop of the next.
//
// Forms (tile = 128 rows x 256 columns of the output):
//   NT  C[r, n]   = sum_k A[r, k] W_e[n, k]        A, W both K-major   (x W^T)
//   NN  C[r, n]   = sum_k A[r, k] W_e[k, n]        W N-major           (dY W)
//   TN  C_e[m, n] = sum_{r in e} A[r, m] B[r, n]   both M/N-major, ragged K (dW)
// Rows of expert e are [off_e, off_{e+1}) of the expert-major buffers.  A
// 128-row tile that runs past its expert's last row computes junk rows that are
// never stored; a ragged-K tail block has the rows past the expert zeroed in
// shared memory before its MMAs.  Experts without rows get exact-zero dW.
//
// Every wait is bounded (about 2 s of %globaltimer); on expiry the CTA sets
// an abort flag and the device status word, drains its own copies and MMAs
// in flight, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;                  // one 128-byte swizzle row of bf16
constexpr int UK = 16;                  // K of one tcgen05.mma kind::f16
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int B_BYTES = BN * BK * 2;    // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
// Epilogue warps: EPI_PARTS per TMEM lane quarter, each draining an equal
// share of the tile's columns.
#ifndef MOE_EPI_PARTS
#define MOE_EPI_PARTS 2
#endif
constexpr int EPI_PARTS = MOE_EPI_PARTS;
constexpr int NUM_EPI_WARPS = 4 * EPI_PARTS;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int TMEM_COLS = 512;
constexpr int MAX_E = 256;
constexpr int CHUNK = 16;                // accumulator columns per epilogue step
constexpr int STG_BYTES = 32 * CHUNK * 4; // epilogue staging buffer of one warp
constexpr long long WAIT_LIMIT_NS = 2000000000ll;   // default bound of every wait

enum Form { FORM_NT = 0, FORM_NN = 1, FORM_TN = 2 };
constexpr int EPI_STORE_F32_TAG = 100;   // TN: fp32 weight-gradient tile store
constexpr int EPI_ROWS_F32_TAG = 101;    // fp32 row store (+ bias[n]): router logits, router dX
constexpr int EPI_SGD_F32_TAG = 102;     // TN: fp32 weight-gradient store + fused SGD step

// The activation backward's side inputs (H, or H1 and H3) can come by TMA
// into a ring of SIDE_SLOTS buffers per epilogue warp, each one 16-column
// chunk of the warp's 32 rows (2 KB: bf16 H1 then H3), so that the data in
// flight costs no registers.  Such an instantiation (SIDE = true) runs the
// operand ring with 3 stages to make room, which pays only at short reduction
// lengths: the host picks it for K <= SIDE_TMA_MAX_K.  Other instantiations
// keep 4 stages and fetch side inputs into registers (a ring of PF + 1
// register buffers).
constexpr int SIDE_SLOTS = 4;
constexpr int SIDE_SLOT_BYTES = 2048;
constexpr int SIDE_TMA_MAX_K = 2048;
// 1: weight-gradient tiles in size order and snake order over the grid when
// the largest expert has more than SNAKE_SKEW times the mean rows (see
// sched_tile).  0 (the default): always round-robin in expert order.  The
// skewed schedule shortens the weight-gradient launches of a skewed layer by
// a fifth, but the run-time choice slows those of balanced layers by 2-4%,
// the layers the default build is tuned for.
#ifndef MOE_TC_SNAKE
#define MOE_TC_SNAKE 0
#endif
constexpr int SNAKE_SKEW = 2;
// The MMAs of a tile whose columns run past N use a smaller N (see the
// MMA issuer); 0 keeps N = 256 on every tile.
#ifndef MOE_TC_TRIM_N
#define MOE_TC_TRIM_N 1
#endif
template <bool SIDE>
__host__ __device__ constexpr int stages_of() { return SIDE ? 3 : STAGES; }

// Dynamic shared memory: the stage ring, the epilogue staging buffers and the
// side-input rings.  The stage ring needs 1024-byte alignment (128-byte
// swizzle): the declaration asks for it, and the static shared memory
// (barriers, segment tables) is padded in front of it to 3 KB.  All of it
// must fit the 227 KB a block may opt into.
template <bool SIDE>
__host__ __device__ constexpr size_t smem_bytes() {
  return (size_t)stages_of<SIDE>() * STAGE_BYTES + NUM_EPI_WARPS * STG_BYTES +
         (SIDE ? (size_t)NUM_EPI_WARPS * SIDE_SLOTS * SIDE_SLOT_BYTES : 0);
}
static_assert(smem_bytes<false>() + 3072 <= 232448, "shared memory of one block");
static_assert(smem_bytes<true>() + 3072 <= 232448, "shared memory of one block");

struct TcParams {
  int M, N, E;          // ragged-M: M = total rows; TN: output rows per expert
  int K0, K1;           // reduction lengths of pair 0 / pair 1 (ragged-M)
  int nM, nN;           // tiles along M (TN) and N
  int m_fast;           // TN: tiles of an expert ordered M-fastest (else N-fastest)
  int ntile_n;          // columns of one N tile in output space (128 for SwiGLU up)
  const int* offsets;   // [E+1]
  void* C;
  long long ldc, sCe;
  const float* bias;
  const bf16* aux0;
  const bf16* aux1;
  void* out1;
  void* out2;
  long long ld_aux;
  int act;              // 0 relu, 1 gelu_tanh
  int* status;
  int seg_len;          // offsets == nullptr: segment e = [e*seg_len, min((e+1)*seg_len, rows))
  int seg_rows;         // total rows of the implicit segments
  float* sgd_w;         // EPI_SGD_F32_TAG: fp32 master weights, indexed like C
  bf16* sgd_wlp;        //   and their bf16 copy (may be null)
  float sgd_lr;
  long long wait_ns;    // bound of every mbarrier wait
  int stall;            // self-test: the producer withholds every load
};

// ------------------------------------------------------------ PTX helpers --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: false once the CTA has aborted or the limit expired (which
// aborts the CTA and records a timeout in the device status word).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* status, long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((long long)(global_ns() - t0) > limit_ns) {
      *abort_flag = 1;
      if (status) atomicExch(status, DEV_STATUS_TIMEOUT);
      return false;
    }
  }
}
// Bounded wait used while draining (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long limit_ns) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if ((long long)(global_ns() - t0) > limit_ns) return;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 layout type 2,
// descriptor version 1): start address, leading / stride byte offsets.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 D, bf16 A and B, K- or MN-major
// operands, N >> 3 at bit 17, M >> 4 at bit 24.
template <int FORM>
__host__ __device__ constexpr uint32_t instr_desc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((FORM == FORM_TN ? 1u : 0u) << 15) |
         ((FORM == FORM_NT ? 0u : 1u) << 16) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  uint4 q;
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 c = __floats2bfloat162_rn(v[4], v[5]);
  __nv_bfloat162 d = __floats2bfloat162_rn(v[6], v[7]);
  q.x = *reinterpret_cast<uint32_t*>(&a);
  q.y = *reinterpret_cast<uint32_t*>(&b);
  q.z = *reinterpret_cast<uint32_t*>(&c);
  q.w = *reinterpret_cast<uint32_t*>(&d);
  return q;
}
__device__ __forceinline__ uint2 pack4_bf16(const float* v) {
  uint2 q;
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  q.x = *reinterpret_cast<uint32_t*>(&a);
  q.y = *reinterpret_cast<uint32_t*>(&b);
  return q;
}
__device__ __forceinline__ void unpack4_bf16(uint2 q, float* v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
  v[0] = __low2float(h[0]);
  v[1] = __high2float(h[0]);
  v[2] = __low2float(h[1]);
  v[3] = __high2float(h[1]);
}

// Activations of the epilogues.  Every value they produce is stored in bf16
// (8 significant bits), so the sigmoid uses the hardware's approximate
// exponential and division (__expf, __fdividef: relative errors of a few fp32
// ulps, far below the bf16 rounding that follows) and is evaluated once per
// element; tanh is 2 sigmoid(2u) - 1.  The CUDA-core GEMMs of fp32 layers keep
// the IEEE-accurate functions of common.cuh.
__device__ __forceinline__ float sigmoid_epi(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float gelu_epi(float h) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  const float t = 2.0f * sigmoid_epi(2.0f * c * (h + a * h * h * h)) - 1.0f;
  return 0.5f * h * (1.0f + t);
}
__device__ __forceinline__ float gelu_grad_epi(float h) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  const float t = 2.0f * sigmoid_epi(2.0f * c * (h + a * h * h * h)) - 1.0f;
  return 0.5f * (1.0f + t) + 0.5f * h * (1.0f - t * t) * c * (1.0f + 3.0f * a * h * h);
}

// Side inputs of one epilogue chunk in the coalesced layout (four rows per
// lane): H or H1 / H3 for the backward epilogues, fp32 master weights for the
// fused SGD.  Members an epilogue does not use are never touched.
struct Side {
  uint2 h1[4], h3[4];
  float4 w[4];
};


// Epilogue outputs are stored with an L2 evict-first policy: no later launch
// re-reads them soon, and the operand tiles that neighbouring CTAs and the
// next wave re-read then stay in L2 (fewer DRAM re-reads of the weights).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void st_ef(void* ptr, uint2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.b32 [%0], {%1, %2}, %3;" ::"l"(ptr), "r"(v.x),
               "r"(v.y), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_ef(void* ptr, float4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "l"(pol)
               : "memory");
}

// Four bf16 at column n of rows row0 + 8 j (j = 0..3) of a row-major matrix
// with leading dimension ld; zeros for rows >= row_hi or n >= N.
__device__ __forceinline__ void load_bf16x4_rows(const bf16* base, long long ld, int row0,
                                                 int row_hi, int n, int N, uint2 (&d)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int g = row0 + 8 * j;
    d[j] = (g < row_hi && n < N) ? __ldg(reinterpret_cast<const uint2*>(base + (size_t)g * ld + n))
                                 : make_uint2(0u, 0u);
  }
}
// The same for fp32 (plain loads: the SGD epilogue rewrites these weights).
__device__ __forceinline__ void load_f32x4_rows(const float* base, long long ld, int row0,
                                                int row_hi, int n, int N, float4 (&d)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int g = row0 + 8 * j;
    d[j] = (g < row_hi && n < N) ? *reinterpret_cast<const float4*>(base + (size_t)g * ld + n)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// 16 accumulator columns from TMEM (row = this lane's TMEM lane) through a
// 32 x 16 fp32 shared buffer of the warp; 16-byte pieces are XOR-swizzled by
// row pairs so that the row-wise writes and the column-wise reads are both
// free of bank conflicts.  out[j] = columns 4 (lane % 4) .. +3 of row
// lane / 4 + 8 j.
__device__ __forceinline__ void stage_chunk(float* stg, int lane, uint32_t taddr, float4 (&out)[4]) {
  float v[16];
  tmem_ld16(taddr, v);
  tmem_ld_wait();
  __syncwarp();   // the previous chunk's readers are done with the buffer
  float4* mine = reinterpret_cast<float4*>(stg + lane * CHUNK);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    mine[q ^ ((lane >> 1) & 3)] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  __syncwarp();
  const int cq = lane & 3, cr = lane >> 2;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int rr = cr + 8 * j;
    out[j] = reinterpret_cast<const float4*>(stg + rr * CHUNK)[cq ^ ((rr >> 1) & 3)];
  }
}

struct Tile {
  int e, m0, n0, row_hi, kbeg, kend, nkb, nkb0;
};

// How many 16-column chunks ahead an epilogue loads its side inputs: the
// fp32 master weights of the fused SGD step come from DRAM under a heavy
// write stream, so they are fetched further ahead than the activation
// backward's H1 / H3.
#ifndef MOE_SGD_PREFETCH
#define MOE_SGD_PREFETCH 3
#endif
#ifndef MOE_BWD_PREFETCH
#define MOE_BWD_PREFETCH 3
#endif
template <int EPI>
__host__ __device__ constexpr int side_prefetch() {
  return EPI == EPI_SGD_F32_TAG ? MOE_SGD_PREFETCH
         : (EPI == EPI_ACT_BWD || EPI == EPI_SWIGLU_BWD) ? MOE_BWD_PREFETCH : 1;
}

template <int FORM>
__device__ __forceinline__ Tile map_tile(int t, const TcParams& p, const int* offs,
                                         const int* tpre) {
  Tile T;
  if (FORM != FORM_TN) {
    const int mt = t / p.nN, nt = t % p.nN;
    int lo = 0, hi = p.E;   // largest lo with tpre[lo] <= mt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tpre[mid] <= mt) lo = mid; else hi = mid;
    }
    T.e = lo;
    T.m0 = offs[lo] + (mt - tpre[lo]) * BM;
    T.row_hi = offs[lo + 1];
    T.n0 = nt * p.ntile_n;
    T.kbeg = 0;
    T.kend = 0;
    T.nkb0 = (p.K0 + BK - 1) / BK;
    T.nkb = T.nkb0 + (p.K1 > 0 ? (p.K1 + BK - 1) / BK : 0);
  } else {
    // ragged K: experts in order of decreasing row count (tpre holds that
    // order for this form)
    const int per = p.nM * p.nN;
    T.e = tpre[t / per];
    const int rem = t % per;
    if (p.m_fast) {
      T.m0 = (rem % p.nM) * BM;
      T.n0 = (rem / p.nM) * BN;
    } else {
      T.m0 = (rem / p.nN) * BM;
      T.n0 = (rem % p.nN) * BN;
    }
    T.row_hi = p.M;
    T.kbeg = offs[T.e];
    T.kend = offs[T.e + 1];
    T.nkb = (T.kend - T.kbeg + BK - 1) / BK;
    T.nkb0 = T.nkb;
  }
  return T;
}

// The i-th tile of this CTA's persistent schedule, or -1 past its last.
// Tiles are dealt round by round over the grid.  A weight-gradient tile
// (ragged K) costs in proportion to its expert's rows: when those are
// skewed (`snake`), the tiles come largest expert first and are dealt in
// alternating direction, so that the sums of tile costs of the CTAs stay
// close to their mean.
template <int FORM>
__device__ __forceinline__ int sched_tile(int i, int total, bool snake) {
  const int base = i * (int)gridDim.x;
  if (base >= total) return -1;
  const int pos = (FORM == FORM_TN && snake && (i & 1)) ? (int)gridDim.x - 1 - (int)blockIdx.x
                                                       : (int)blockIdx.x;
  const int t = base + pos;
  return t < total ? t : -1;
}

template <int FORM, int EPI, bool SIDE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB0x, const __grid_constant__ CUtensorMap tmA1,
               const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmS0,
               const __grid_constant__ CUtensorMap tmS1, const TcParams p) {
  static_assert(!SIDE || EPI == EPI_ACT_BWD || EPI == EPI_SWIGLU_BWD, "side ring: activation backward");
  constexpr int NST = stages_of<SIDE>();   // operand ring stages of this instantiation
  // stage ring in dynamic shared memory (1024-byte aligned for the 128-byte
  // swizzle); barriers, the TMEM address slot and the segment tables static
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_mb[STAGES], empty_mb[STAGES], tfull_mb[2], tempty_mb[2], drain_mb;
  __shared__ __align__(8) uint64_t side_mb[NUM_EPI_WARPS * SIDE_SLOTS];   // side-input ring
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_word;
  __shared__ int offs[MAX_E + 1];
  __shared__ int tpre[MAX_E + 1];
  __shared__ int snake_word;
  volatile int* abort_flag = &abort_word;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t drain_bar = smem_u32(&drain_mb);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&full_mb[s]), 1);
      mbar_init(smem_u32(&empty_mb[s]), 1);
    }
    if (SIDE)
      for (int s = 0; s < NUM_EPI_WARPS * SIDE_SLOTS; ++s) mbar_init(smem_u32(&side_mb[s]), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull_mb[b]), 1);
      mbar_init(smem_u32(&tempty_mb[b]), NUM_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    abort_word = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), TMEM_COLS);
  pdl_wait();   // the previous kernel's outputs (segment offsets, operands) are visible from here
  for (int i = tid; i <= p.E; i += NUM_THREADS)
    offs[i] = p.offsets ? p.offsets[i] : min(i * p.seg_len, p.seg_rows);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    // Offsets given by a caller are clamped to a non-decreasing sequence
    // within [0, total rows]: no tile then reads or stores past the row
    // operands or C, whatever the table holds (the routing path's own
    // offsets already satisfy this and are unchanged by it).
    int prev = 0;
    for (int e = 0; e <= p.E; ++e) {
      const int v = min(max(offs[e], prev), p.seg_rows);
      offs[e] = v;
      prev = v;
    }
    if (FORM != FORM_TN) {
      tpre[0] = 0;
      for (int e = 0; e < p.E; ++e) tpre[e + 1] = tpre[e] + (offs[e + 1] - offs[e] + BM - 1) / BM;
    }
    int mx = 0;
    for (int e = 0; e < p.E; ++e) mx = max(mx, offs[e + 1] - offs[e]);
    snake_word = (FORM == FORM_TN && MOE_TC_SNAKE &&
                  (long long)mx * p.E > (long long)SNAKE_SKEW * offs[p.E]) ? 1 : 0;
  }
  __syncthreads();
  const bool snake = snake_word != 0;
  if (FORM == FORM_TN) {
    // tpre[rank] = expert: by decreasing row count, ties by id, when the
    // loads are skewed; else in id order
    for (int e = tid; e < p.E; e += NUM_THREADS) {
      int rank = e;
      if (snake) {
        const int re = offs[e + 1] - offs[e];
        rank = 0;
        for (int j = 0; j < p.E; ++j) {
          const int rj = offs[j + 1] - offs[j];
          rank += (rj > re || (rj == re && j < e)) ? 1 : 0;
        }
      }
      tpre[rank] = e;
    }
    __syncthreads();
  }
  const uint32_t tmem_base = tmem_slot;
  const int total = (FORM != FORM_TN) ? tpre[p.E] * p.nN : p.E * p.nM * p.nN;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 issues the operand loads and nothing else.
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      uint32_t last_par = 0;
      bool ok = p.stall == 0;   // a stalled self-test issues nothing: the MMA waits run out
      for (int it = 0, t; ok && (t = sched_tile<FORM>(it, total, snake)) >= 0; ++it) {
        const Tile T = map_tile<FORM>(t, p, offs, tpre);
        for (int kb = 0; kb < T.nkb; ++kb) {
          if (!wait_bar(smem_u32(&empty_mb[s]), ph ^ 1u, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full_mb[s]);
          const uint32_t a_dst = sbase + s * STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          if (FORM == FORM_NT) {
            const int k0 = kb * BK;
            tma_load_2d(a_dst, &tmA0, fb, k0, T.m0);
            if (EPI == EPI_SWIGLU_UP) {
              // 64-row boxes of W1 and W3 for the same output columns side
              // by side: accumulator columns 128 h + [0, 64) hold W1 x and
              // 128 h + [64, 128) W3 x of output columns 64 h + [0, 64)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                tma_load_3d(b_dst + (2 * h) * (64 * BK * 2), &tmB0, fb, k0, T.n0 + 64 * h, T.e);
                tma_load_3d(b_dst + (2 * h + 1) * (64 * BK * 2), &tmB0x, fb, k0, T.n0 + 64 * h, T.e);
              }
            } else {
              tma_load_3d(b_dst, &tmB0, fb, k0, T.n0, T.e);
              tma_load_3d(b_dst + BM * BK * 2, &tmB0, fb, k0, T.n0 + 128, T.e);
            }
          } else if (FORM == FORM_NN) {
            const bool second = kb >= T.nkb0;
            const int k0 = (second ? kb - T.nkb0 : kb) * BK;
            tma_load_2d(a_dst, second ? &tmA1 : &tmA0, fb, k0, T.m0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_3d(b_dst + j * (64 * BK * 2), second ? &tmB1 : &tmB0, fb, T.n0 + 64 * j, k0,
                          T.e);
          } else {
            const int r0 = T.kbeg + kb * BK;
#pragma unroll
            for (int j = 0; j < 2; ++j) tma_load_2d(a_dst + j * (64 * BK * 2), &tmA0, fb, T.m0 + 64 * j, r0);
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_2d(b_dst + j * (64 * BK * 2), &tmB0, fb, T.n0 + 64 * j, r0);
          }
          issued |= 1 << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
          if (++s == NST) { s = 0; ph ^= 1u; }
        }
      }
      // drain: every stage's last load must have landed before the CTA exits
      for (int q = 0; q < NST; ++q)
          if (issued & (1 << q)) drain_wait(smem_u32(&full_mb[q]), (last_par >> q) & 1u, p.wait_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = instr_desc<FORM>();
    int s = 0;
    uint32_t ph = 0;
    int buf = 0;
    uint32_t aph = 0;
    bool ok = true, any_mma = false;
    for (int it = 0, t; ok && (t = sched_tile<FORM>(it, total, snake)) >= 0; ++it) {
      const Tile T = map_tile<FORM>(t, p, offs, tpre);
      if (T.nkb == 0) continue;
      if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&tempty_mb[buf]), aph ^ 1u, abort_flag, p.status, p.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
      // A tile whose columns run past N multiplies only the B rows it needs:
      // N of the MMA rounded up to 16 (a SwiGLU tile keeps its W1 / W3
      // halves at columns 0 and 64 of each 128).  The accumulator columns
      // past it keep stale values that the epilogue never stores.
      uint32_t id_t = idesc;
      if (MOE_TC_TRIM_N) {
        const int v = min(EPI == EPI_SWIGLU_UP ? 128 : BN, p.N - T.n0);
        const int nv = EPI != EPI_SWIGLU_UP ? (v + 15) & ~15
                       : v <= 64 ? 64 + ((v + 15) & ~15) : 192 + ((v - 64 + 15) & ~15);
        id_t = (idesc & ~(0x3Fu << 17)) | ((uint32_t)(nv >> 3) << 17);
      }
      for (int kb = 0; kb < T.nkb; ++kb) {
        if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&full_mb[s]), ph, abort_flag, p.status, p.wait_ns))) {
          ok = false;
          break;
        }
        const uint32_t a_base = sbase + s * STAGE_BYTES;
        const uint32_t b_base = a_base + A_BYTES;
        if (FORM == FORM_TN && kb == T.nkb - 1) {
          const int valid = T.kend - (T.kbeg + kb * BK);
          if (valid < BK) {
            // rows past the expert's last row: zero them in both operands
            // (the two A and four B boxes, each BK rows of 128 bytes; whole
            // rows are invariant under the 128-byte swizzle).  Zeroing A
            // alone is not enough: rows past the last kept row of an
            // expert capacity are never written, and 0 * NaN is NaN.
            const int nchunk = (BK - valid) * 8;   // 16-byte chunks per box
            for (int j = 0; j < 6; ++j) {
              uint4* dst = reinterpret_cast<uint4*>(smem + s * STAGE_BYTES + j * (64 * BK * 2) + valid * 128);
              for (int c = lane; c < nchunk; c += 32) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            uint64_t adesc, bdesc;
            if (FORM == FORM_TN) adesc = smem_desc(a_base + kk * 2048, 64 * BK * 2, 1024);
            else adesc = smem_desc(a_base + kk * 32, 16, 1024);
            if (FORM == FORM_NT) bdesc = smem_desc(b_base + kk * 32, 16, 1024);
            else bdesc = smem_desc(b_base + kk * 2048, 64 * BK * 2, 1024);
            mma_bf16(d_tmem, adesc, bdesc, id_t, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&empty_mb[s]));
        }
        any_mma = true;
        __syncwarp();
        if (++s == NST) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(smem_u32(&tfull_mb[buf]));
      __syncwarp();
      if (++buf == 2) { buf = 0; aph ^= 1u; }
    }
    if (any_mma && lane == 0) {
      mma_commit(drain_bar);
      drain_wait(drain_bar, 0, p.wait_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    float* stg = reinterpret_cast<float*>(smem + NST * STAGE_BYTES + (warp - 2) * STG_BYTES);
    // TMEM lane quarter of this warp (a warp may only read lanes
    // 32 (warp % 4) .. +31) and which share of the tile's columns it takes
    const int lane_base = (warp & 3) * 32;
    const int part = (warp - 2) >> 2;
    const int row = lane_base + lane;
    const uint64_t pol = policy_evict_first();
    int buf = 0;
    uint32_t aph = 0;
    // Side-input ring (SIDE): this warp's chunks form one sequence
    // over its tiles (NCH chunks of 16 columns per tile); chunk g goes to slot
    // g % SIDE_SLOTS, loaded by TMA SIDE_SLOTS chunks ahead of its use, the
    // next tile's first chunks while this tile's last ones are processed.
    constexpr int NCH = (BN / EPI_PARTS) / CHUNK;
    const size_t side_off = (size_t)NST * STAGE_BYTES + NUM_EPI_WARPS * STG_BYTES +
                            (size_t)(warp - 2) * SIDE_SLOTS * SIDE_SLOT_BYTES;
    const uint32_t side_bar0 = smem_u32(&side_mb[(warp - 2) * SIDE_SLOTS]);
    int side_it = 0, side_i = 0;           // issue cursor: schedule position, chunk
    int side_t = sched_tile<FORM>(0, total, snake);   // its tile (-1: none left)
    long long side_iss = 0, side_con = 0;  // chunks issued / consumed
    auto side_skip_empty = [&]() {
      while (side_t >= 0 && map_tile<FORM>(side_t, p, offs, tpre).nkb == 0)
        side_t = sched_tile<FORM>(++side_it, total, snake);
    };
    auto side_issue = [&](int slot) {
      const Tile Ti = map_tile<FORM>(side_t, p, offs, tpre);
      const int n = Ti.n0 + part * (BN / EPI_PARTS) + side_i * CHUNK;   // a multiple of 16
      if (lane == 0) {
        const uint32_t bar = side_bar0 + 8u * (uint32_t)slot;
        const uint32_t dst = smem_u32(smem + side_off + (size_t)slot * SIDE_SLOT_BYTES);
        // the lanes' reads of this slot's previous contents come first
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(bar, EPI == EPI_SWIGLU_BWD ? 2048u : 1024u);
        tma_load_2d(dst, &tmS0, bar, n, Ti.m0 + lane_base);
        if (EPI == EPI_SWIGLU_BWD) tma_load_2d(dst + 1024, &tmS1, bar, n, Ti.m0 + lane_base);
      }
      ++side_iss;
      if (++side_i == NCH) {
        side_i = 0;
        side_t = sched_tile<FORM>(++side_it, total, snake);
        side_skip_empty();
      }
    };
    // the slot's rows in the coalesced layout: lane l takes columns
    // 4 (l % 4) .. +3 of rows l / 4 + 8 j (box rows of 16 bf16 values)
    auto side_read = [&](int slot, Side& d) {
      const uint8_t* sp = smem + side_off + (size_t)slot * SIDE_SLOT_BYTES;
      const int rr = lane >> 2, cq4 = lane & 3;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        d.h1[j] = *reinterpret_cast<const uint2*>(sp + (rr + 8 * j) * 32 + cq4 * 8);
        if (EPI == EPI_SWIGLU_BWD)
          d.h3[j] = *reinterpret_cast<const uint2*>(sp + 1024 + (rr + 8 * j) * 32 + cq4 * 8);
      }
    };
    bool side_fail = false;
    if (SIDE) {
      side_skip_empty();
      for (int q = 0; q < SIDE_SLOTS && side_t >= 0; ++q) side_issue(q);
    }
    for (int it = 0, t; (t = sched_tile<FORM>(it, total, snake)) >= 0; ++it) {
      const Tile T = map_tile<FORM>(t, p, offs, tpre);
      const int r = T.m0 + row;
      const bool rok = r < T.row_hi;
      if (T.nkb == 0) {
        // ragged K with an empty expert: dW tile is exactly zero (and the SGD
        // step leaves W as it is; its bf16 copy is still rewritten from W)
        if (FORM == FORM_TN && rok) {
          const size_t o = (size_t)T.e * p.sCe + (size_t)r * p.ldc;
          const int nb = T.n0 + part * (BN / EPI_PARTS), ne = min(nb + BN / EPI_PARTS, p.N);
          if (p.C != nullptr) {
            float* c = static_cast<float*>(p.C) + o;
            for (int n = nb; n < ne; n += 4)
              *reinterpret_cast<float4*>(c + n) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          if (EPI == EPI_SGD_F32_TAG && p.sgd_wlp) {
            for (int n = nb; n < ne; n += 8) {
              float w[8];
              *reinterpret_cast<float4*>(w) = *reinterpret_cast<const float4*>(p.sgd_w + o + n);
              *reinterpret_cast<float4*>(w + 4) = *reinterpret_cast<const float4*>(p.sgd_w + o + n + 4);
              *reinterpret_cast<uint4*>(p.sgd_wlp + o + n) = pack8_bf16(w);
            }
          }
        }
        continue;
      }
      // Each 16-column chunk of the accumulator goes TMEM -> registers (one
      // row per lane) -> this warp's swizzled shared buffer -> registers in a
      // coalesced layout: lane l then owns columns 4 (l % 4) .. +3 of rows
      // l / 4 + 8 j, j = 0..3, so four lanes cover 64 contiguous bytes of a
      // fp32 row and every global load and store below is coalesced.
      const int cq = lane & 3;
      const int row0 = T.m0 + lane_base + (lane >> 2);
      const int ncols = EPI == EPI_SWIGLU_UP ? 128 : BN;
      const int c_begin = part * (ncols / EPI_PARTS), c_end = c_begin + ncols / EPI_PARTS;
      const size_t wbase = (size_t)T.e * p.sCe;
      // side inputs are fetched PF chunks ahead into a ring of PF + 1
      // register buffers (the first PF while the accumulator is still being
      // produced)
      constexpr int PF = side_prefetch<EPI>();
      constexpr int NB = PF + 1;
      auto load_side = [&](int n, Side& d) {
        if (EPI == EPI_ACT_BWD || EPI == EPI_SWIGLU_BWD) {
          load_bf16x4_rows(p.aux0, p.ld_aux, row0, T.row_hi, n, p.N, d.h1);
          if (EPI == EPI_SWIGLU_BWD) load_bf16x4_rows(p.aux1, p.ld_aux, row0, T.row_hi, n, p.N, d.h3);
        }
        if (EPI == EPI_SGD_F32_TAG) load_f32x4_rows(p.sgd_w + wbase, p.ldc, row0, T.row_hi, n, p.N, d.w);
      };
      Side sd[NB];
      if (!SIDE) {
#pragma unroll
        for (int q = 0; q < PF; ++q)
          if (c_begin + q * CHUNK < c_end) load_side(T.n0 + c_begin + q * CHUNK + 4 * cq, sd[q]);
      }
      // warp-uniform: the tcgen05.ld below is a warp-collective instruction
      if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&tfull_mb[buf]), aph, abort_flag, p.status, p.wait_ns))) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(buf * BN);
      auto chunk = [&](int cc, const Side& use, Side& fill) {
        const int n = T.n0 + cc + 4 * cq;
        if (!SIDE && cc + PF * CHUNK < c_end) load_side(n + PF * CHUNK, fill);
        float4 acc[4], acc3[4];
        if (EPI == EPI_SWIGLU_UP) {
          // output columns 64 h + c: W1 x at accumulator column 128 h + c,
          // W3 x at 128 h + 64 + c
          const int c1 = cc + (cc & ~63);
          stage_chunk(stg, lane, t_row + c1, acc);
          stage_chunk(stg, lane, t_row + c1 + 64, acc3);
        } else {
          stage_chunk(stg, lane, t_row + cc, acc);
        }
        constexpr bool BIAS_EPI = EPI == EPI_STORE || EPI == EPI_ROWS_F32_TAG || EPI == EPI_ACT_FWD;
        const bool add_bias = BIAS_EPI && p.bias != nullptr && n < p.N;
        float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (add_bias) b4 = *reinterpret_cast<const float4*>(p.bias + (size_t)T.e * p.N + n);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int g = row0 + 8 * j;
          if (g >= T.row_hi || n >= p.N) continue;
          float x[4] = {acc[j].x, acc[j].y, acc[j].z, acc[j].w};
          if (add_bias) {
            x[0] += b4.x;
            x[1] += b4.y;
            x[2] += b4.z;
            x[3] += b4.w;
          }
          const size_t o = (size_t)g * p.ldc + n;
          if (EPI == EPI_STORE) {
            st_ef(static_cast<bf16*>(p.C) + o, pack4_bf16(x), pol);
          } else if (EPI == EPI_ROWS_F32_TAG) {
            st_ef(static_cast<float*>(p.C) + o, make_float4(x[0], x[1], x[2], x[3]), pol);
          } else if (EPI == EPI_STORE_F32_TAG) {
            st_ef(static_cast<float*>(p.C) + wbase + o, acc[j], pol);
          } else if (EPI == EPI_SGD_F32_TAG) {
            // dW stored as is (unless the caller asked for no gradient); the
            // update uses the same fused multiply-add and round-to-nearest
            // bf16 conversion as the stand-alone SGD kernel
            if (p.C != nullptr) st_ef(static_cast<float*>(p.C) + wbase + o, acc[j], pol);
            float w[4] = {use.w[j].x, use.w[j].y, use.w[j].z, use.w[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = fmaf(-p.sgd_lr, x[i], w[i]);
            st_ef(p.sgd_w + wbase + o, make_float4(w[0], w[1], w[2], w[3]), pol);
            if (p.sgd_wlp) st_ef(p.sgd_wlp + wbase + o, pack4_bf16(w), pol);
          } else if (EPI == EPI_ACT_FWD) {
            float a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = p.act == 0 ? fmaxf(x[i], 0.f) : gelu_epi(x[i]);
            st_ef(static_cast<bf16*>(p.out1) + o, pack4_bf16(x), pol);
            st_ef(static_cast<bf16*>(p.C) + o, pack4_bf16(a), pol);
          } else if (EPI == EPI_ACT_BWD) {
            float h[4], dh[4];
            unpack4_bf16(use.h1[j], h);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dh[i] = p.act == 0 ? (h[i] > 0.f ? x[i] : 0.f) : x[i] * gelu_grad_epi(h[i]);
            st_ef(static_cast<bf16*>(p.C) + o, pack4_bf16(dh), pol);
          } else if (EPI == EPI_SWIGLU_BWD) {
            float h1[4], h3[4], d1[4], d3[4];
            unpack4_bf16(use.h1[j], h1);
            unpack4_bf16(use.h3[j], h3);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              // SiLU(h) = h s, SiLU'(h) = s (1 + h (1 - s)), s = sigmoid(h)
              const float sg = sigmoid_epi(h1[i]);
              d1[i] = x[i] * h3[i] * (sg * (1.0f + h1[i] * (1.0f - sg)));
              d3[i] = x[i] * (h1[i] * sg);
            }
            st_ef(static_cast<bf16*>(p.C) + o, pack4_bf16(d1), pol);
            st_ef(static_cast<bf16*>(p.out1) + o, pack4_bf16(d3), pol);
          } else if (EPI == EPI_SWIGLU_UP) {
            const float h3[4] = {acc3[j].x, acc3[j].y, acc3[j].z, acc3[j].w};
            float a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = (x[i] * sigmoid_epi(x[i])) * h3[i];
            st_ef(static_cast<bf16*>(p.out1) + o, pack4_bf16(x), pol);
            st_ef(static_cast<bf16*>(p.out2) + o, pack4_bf16(h3), pol);
            st_ef(static_cast<bf16*>(p.C) + o, pack4_bf16(a), pol);
          }
        }
      };
      // chunks per warp: 8 (SwiGLU-up tiles: 4), a multiple of NB; chunk i
      // reads buffer i % NB and fills buffer (i + PF) % NB with chunk i + PF
      static_assert(((EPI == EPI_SWIGLU_UP ? 128 : BN) / EPI_PARTS / CHUNK) % NB == 0, "whole rings");
      if (SIDE) {
        // side inputs from the TMA ring; each consumed slot is refilled with
        // the chunk SIDE_SLOTS further on
#pragma unroll 1
        for (int i = 0; i < NCH; ++i) {
          const int slot = (int)(side_con % SIDE_SLOTS);
          const uint32_t par = (uint32_t)((side_con / SIDE_SLOTS) & 1);
          if (!__all_sync(0xffffffffu, wait_bar(side_bar0 + 8u * (uint32_t)slot, par, abort_flag,
                                                p.status, p.wait_ns))) {
            side_fail = true;
            break;
          }
          Side cur;
          side_read(slot, cur);
          chunk(c_begin + i * CHUNK, cur, cur);
          __syncwarp();
          ++side_con;
          if (side_t >= 0) side_issue(slot);
        }
        if (side_fail) break;
      } else {
#pragma unroll 1
        for (int cc = c_begin; cc < c_end; cc += NB * CHUNK) {
#pragma unroll
          for (int q = 0; q < NB; ++q) chunk(cc + q * CHUNK, sd[q], sd[(q + PF) % NB]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty_mb[buf]));
      if (++buf == 2) { buf = 0; aph ^= 1u; }
    }
    // side loads still in flight (an aborted CTA) land before the CTA exits
    for (long long g = side_con; g < side_iss; ++g)
      drain_wait(side_bar0 + 8u * (uint32_t)(g % SIDE_SLOTS), (uint32_t)((g / SIDE_SLOTS) & 1),
                 p.wait_ns);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------- host --

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// bf16 tensor map, 128-byte swizzle, zero fill out of bounds.  dims[0] is
// the contiguous dimension; strides are in bytes for dims 1..rank-1.
bool make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  cuuint64_t d[3], s[2];
  cuuint32_t b[3];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides[i];
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), d, s,
                  b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D tensor map without swizzle for the epilogues' side inputs: [rows, cols]
// row-major, `ld` elements between rows, fp32 (elem 4) or bf16 (elem 2), box
// of 16 columns x 32 rows (out-of-range parts read as zeros).
bool make_side_map(CUtensorMap* m, const void* ptr, int elem, uint64_t cols, uint64_t rows,
                   uint64_t ld) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t d[2] = {cols, rows};
  const cuuint64_t st[1] = {ld * (uint64_t)elem};
  const cuuint32_t b[2] = {16, 32};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, elem == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  2, const_cast<void*>(ptr), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// SMs of the current device (cached per device ordinal): the persistent grid.
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const bool slot = dev >= 0 && dev < 64;
  if (slot) {
    const int n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  int n = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0)
    return 152;   // any grid is correct (tiles are strided over the grid); this one fits a GB300
  if (slot) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int FORM, int EPI, bool SIDE = false>
cudaError_t launch_inst(const CUtensorMap* maps, const TcParams& p, int tiles_upper,
                        cudaStream_t st) {
  static std::atomic<unsigned long long> attr_done{0};
  constexpr size_t SMEM = smem_bytes<SIDE>();
  cudaError_t e = ensure_dynamic_smem(tc_gemm_kernel<FORM, EPI, SIDE>, (int)SMEM, attr_done);
  if (e != cudaSuccess) return e;
  int grid = sm_count();
  if (tiles_upper < grid) grid = tiles_upper;
  if (grid < 1) return cudaSuccess;
  MOE_LAUNCH(launch_pdl(tc_gemm_kernel<FORM, EPI, SIDE>, dim3(grid), dim3(NUM_THREADS), SMEM, st,
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], p));
  return cudaGetLastError();
}

}  // namespace tc

cudaError_t launch_gemm_tc(const GemmArgs& g, cudaStream_t st) {
  using namespace tc;
  if (g.M == 0 || g.N == 0 || g.E == 0) return cudaSuccess;
  if (g.a_type != 1 || g.b_type != 1 || g.E > MAX_E) return cudaErrorInvalidValue;
  if (g.offsets == nullptr && g.seg_len <= 0) return cudaErrorInvalidValue;
  // every pointer the chosen epilogue dereferences must be set; a weight
  // gradient with the SGD step fused may go unstored (C == nullptr)
  const bool sgd_only = g.ragged_k && g.sgd_w != nullptr;
  if (g.A0 == nullptr || g.B0 == nullptr || (g.C == nullptr && !sgd_only)) return cudaErrorInvalidValue;
  if ((g.epi == EPI_SWIGLU_UP && (g.B0x == nullptr || g.out1 == nullptr || g.out2 == nullptr)) ||
      (g.epi == EPI_ACT_FWD && g.out1 == nullptr) || (g.epi == EPI_ACT_BWD && g.aux0 == nullptr) ||
      (g.epi == EPI_SWIGLU_BWD && (g.aux0 == nullptr || g.aux1 == nullptr || g.out1 == nullptr)) ||
      (g.A1 != nullptr && (g.B1 == nullptr || g.K1 <= 0)))
    return cudaErrorInvalidValue;
  CUtensorMap maps[7];   // operands (5), then the epilogue's side inputs (2)
  TcParams p{};
  p.M = g.M;
  p.N = g.N;
  p.E = g.E;
  p.K0 = g.K0;
  p.K1 = (g.A1 != nullptr) ? g.K1 : 0;
  p.offsets = g.offsets;
  p.C = g.C;
  p.ldc = g.ldc;
  p.sCe = g.sCe;
  p.bias = g.bias;
  p.aux0 = static_cast<const bf16*>(g.aux0);
  p.aux1 = static_cast<const bf16*>(g.aux1);
  p.out1 = g.out1;
  p.out2 = g.out2;
  p.ld_aux = g.ld_aux;
  p.act = g.act;
  p.status = g.status;
  p.seg_len = g.seg_len;
  p.seg_rows = g.ragged_k ? g.K0 : g.M;
  p.sgd_w = g.sgd_w;
  p.sgd_wlp = static_cast<bf16*>(g.sgd_wlp);
  p.sgd_lr = g.sgd_lr;
  p.wait_ns = g.wait_ns > 0 ? g.wait_ns : WAIT_LIMIT_NS;
  p.stall = g.stall;
  int tiles_upper = 0;
  const uint64_t R = (uint64_t)g.M;
  if (!g.ragged_k && g.b_kcontig) {
    // NT: A [R, K0] K-major; W [E, N, K0] K-major (3-D so tiles never cross experts)
    const uint64_t ad[2] = {(uint64_t)g.K0, R}, as[1] = {(uint64_t)g.lda * 2};
    const uint32_t ab[2] = {BK, BM};
    const uint64_t bd[3] = {(uint64_t)g.K0, (uint64_t)g.N, (uint64_t)g.E};
    const uint64_t bs[2] = {(uint64_t)g.ldb * 2, (uint64_t)g.sBe * 2};
    const bool swiglu = g.epi == EPI_SWIGLU_UP;
    const uint32_t bb[3] = {BK, swiglu ? 64u : 128u, 1};
    if (!make_map(&maps[0], g.A0, 2, ad, as, ab) || !make_map(&maps[1], g.B0, 3, bd, bs, bb))
      return cudaErrorInvalidValue;
    if (swiglu) {
      if (!make_map(&maps[2], g.B0x, 3, bd, bs, bb)) return cudaErrorInvalidValue;
    } else {
      maps[2] = maps[1];
    }
    maps[3] = maps[0];
    maps[4] = maps[1];
    maps[5] = maps[6] = maps[0];
    p.ntile_n = swiglu ? 128 : BN;
    p.nN = (g.N + p.ntile_n - 1) / p.ntile_n;
    p.nM = 0;
    p.K1 = 0;
    tiles_upper = (int)(((R + BM - 1) / BM + g.E) * p.nN);
    switch (g.epi) {
      case EPI_SWIGLU_UP: return launch_inst<FORM_NT, EPI_SWIGLU_UP>(maps, p, tiles_upper, st);
      case EPI_ACT_FWD: return launch_inst<FORM_NT, EPI_ACT_FWD>(maps, p, tiles_upper, st);
      case EPI_STORE:
        if (g.c_type == 0) return launch_inst<FORM_NT, EPI_ROWS_F32_TAG>(maps, p, tiles_upper, st);
        return launch_inst<FORM_NT, EPI_STORE>(maps, p, tiles_upper, st);
    }
    return cudaErrorInvalidValue;
  }
  if (!g.ragged_k) {
    // NN: A [R, K] K-major; W [E, K, N] N-major
    const uint64_t ad[2] = {(uint64_t)g.K0, R}, as[1] = {(uint64_t)g.lda * 2};
    const uint32_t ab[2] = {BK, BM};
    const uint64_t bd[3] = {(uint64_t)g.N, (uint64_t)g.K0, (uint64_t)g.E};
    const uint64_t bs[2] = {(uint64_t)g.ldb * 2, (uint64_t)g.sBe * 2};
    const uint32_t bb[3] = {64, BK, 1};
    if (!make_map(&maps[0], g.A0, 2, ad, as, ab) || !make_map(&maps[1], g.B0, 3, bd, bs, bb))
      return cudaErrorInvalidValue;
    maps[2] = maps[1];
    if (p.K1 > 0) {
      const uint64_t ad1[2] = {(uint64_t)g.K1, R};
      const uint64_t bd1[3] = {(uint64_t)g.N, (uint64_t)g.K1, (uint64_t)g.E};
      if (!make_map(&maps[3], g.A1, 2, ad1, as, ab) || !make_map(&maps[4], g.B1, 3, bd1, bs, bb))
        return cudaErrorInvalidValue;
    } else {
      maps[3] = maps[0];
      maps[4] = maps[1];
    }
    p.ntile_n = BN;
    p.nN = (g.N + BN - 1) / BN;
    maps[5] = maps[6] = maps[0];
    // the activation backward at a short reduction length: side inputs by TMA
    const bool side = (g.epi == EPI_SWIGLU_BWD || g.epi == EPI_ACT_BWD) &&
                      g.K0 + (p.K1 > 0 ? g.K1 : 0) <= SIDE_TMA_MAX_K;
    tiles_upper = (int)(((R + BM - 1) / BM + g.E) * p.nN);
    if (side) {
      // H (H1) and H3 [R, N] bf16, leading dimension ld_aux
      if (!make_side_map(&maps[5], g.aux0, 2, (uint64_t)g.N, R, (uint64_t)g.ld_aux) ||
          (g.epi == EPI_SWIGLU_BWD &&
           !make_side_map(&maps[6], g.aux1, 2, (uint64_t)g.N, R, (uint64_t)g.ld_aux)))
        return cudaErrorInvalidValue;
    }
    switch (g.epi) {
      case EPI_SWIGLU_BWD:
        if (side) return launch_inst<FORM_NN, EPI_SWIGLU_BWD, true>(maps, p, tiles_upper, st);
        return launch_inst<FORM_NN, EPI_SWIGLU_BWD>(maps, p, tiles_upper, st);
      case EPI_ACT_BWD:
        if (side) return launch_inst<FORM_NN, EPI_ACT_BWD, true>(maps, p, tiles_upper, st);
        return launch_inst<FORM_NN, EPI_ACT_BWD>(maps, p, tiles_upper, st);
      case EPI_STORE:
        if (g.c_type == 0) return launch_inst<FORM_NN, EPI_ROWS_F32_TAG>(maps, p, tiles_upper, st);
        return launch_inst<FORM_NN, EPI_STORE>(maps, p, tiles_upper, st);
    }
    return cudaErrorInvalidValue;
  }
  // TN (ragged K): A [Rk, M] M-major, B [Rk, N] N-major; Rk = K0 rows in total
  if (g.c_type != 0 || g.epi != EPI_STORE) return cudaErrorInvalidValue;
  const uint64_t Rk = (uint64_t)g.K0;
  if (Rk == 0) {
    // no rows at all: every expert's gradient is zero (callers with no rows
    // skip the SGD step, so a fused update has nothing to do here)
    if (g.sgd_w != nullptr) return cudaErrorInvalidValue;
    return cudaMemsetAsync(g.C, 0, (size_t)g.E * g.sCe * sizeof(float), st);
  }
  const uint64_t ad[2] = {(uint64_t)g.M, Rk}, as[1] = {(uint64_t)g.lda * 2};
  const uint64_t bd[2] = {(uint64_t)g.N, Rk}, bs[1] = {(uint64_t)g.ldb * 2};
  const uint32_t box[2] = {64, BK};
  if (!make_map(&maps[0], g.A0, 2, ad, as, box) || !make_map(&maps[1], g.B0, 2, bd, bs, box))
    return cudaErrorInvalidValue;
  maps[2] = maps[3] = maps[0];
  maps[4] = maps[1];
  maps[5] = maps[6] = maps[0];
  p.ntile_n = BN;
  p.nM = (g.M + BM - 1) / BM;
  p.nN = (g.N + BN - 1) / BN;
  p.K1 = 0;
  // An expert's tiles span more than one wave of CTAs, and the operand indexed
  // by the slower tile coordinate is re-read from DRAM by every wave that
  // touches it; step fastest along the smaller operand's dimension (M: the
  // A operand [rows, M]; N: B [rows, N]) so that the larger one is read once.
  p.m_fast = g.M < g.N ? 1 : 0;
  tiles_upper = g.E * p.nM * p.nN;
  if (g.sgd_w != nullptr) return launch_inst<FORM_TN, EPI_SGD_F32_TAG>(maps, p, tiles_upper, st);
  return launch_inst<FORM_TN, EPI_STORE_F32_TAG>(maps, p, tiles_upper, st);
}

}  // namespace moe
