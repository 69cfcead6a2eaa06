// Token dispatch for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocating routine) at the
// point where they need routing: code running while a stream is being
// captured into a CUDA graph (an allocation there breaks or invalidates the
// capture), code inside another runtime's memory pool that forbids outside
// allocations, and latency-critical loops where an allocation could
// synchronise the device.  moe_dispatch_noalloc gives them the histogram /
// exclusive-scan / stable-scatter dispatch with its per-chunk scratch counts
// held in a fixed, file-scope device array instead of a caller workspace.
//
// The array is sized for MOE_NOALLOC_MAX_ROUTED routed assignments (T*k) and
// up to 256 experts: at most max(ROUTE_TARGET_CHUNKS, R / ROUTE_CHUNK_MAX) =
// 1024 chunks x 256 experts x 4 bytes = 1 MiB, which every GPU that loads this
// library keeps until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace {

constexpr int kMaxChunks = MOE_NOALLOC_MAX_ROUTED / moe::ROUTE_CHUNK_MAX > moe::ROUTE_TARGET_CHUNKS
                               ? MOE_NOALLOC_MAX_ROUTED / moe::ROUTE_CHUNK_MAX
                               : moe::ROUTE_TARGET_CHUNKS;
static_assert(MOE_NOALLOC_MAX_ROUTED % moe::ROUTE_CHUNK_MAX == 0, "whole chunks");

// Per-chunk expert counts, then per-chunk first slots.  Shared by every call:
// each call overwrites the entries it reads before reading them, so nothing
// needs clearing, but two calls that overlap on the GPU race on it.
static __device__ __align__(256) int g_dispatch_scratch[kMaxChunks * 256];

// Host code may not use the array's name as an address; its device address
// is looked up once per device, with that device current.
int* scratch_address(moe_status* st) {
  static std::mutex mu;
  static int* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *st = MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) {
      *st = MOE_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = static_cast<int*>(p);
  }
  *st = MOE_OK;
  return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* idx,
                                           int32_t* counts, int32_t* offsets, int32_t* src_tok,
                                           int32_t* slot_of, void* stream) {
  if (cfg == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cfg;
  if (c.T < 0 || c.k <= 0 || c.E <= 0) return MOE_ERR_INVALID_ARG;
  // the routing fields are checked exactly as moe_forward checks them
  if (!(c.capacity_factor >= 0.f) || c.capacity_factor > 1e6f) return MOE_ERR_INVALID_ARG;
  if (c.E > 256 || c.k > 32 || c.k > c.E) return MOE_ERR_UNSUPPORTED;
  const long long R = (long long)c.T * c.k;
  if (R > MOE_NOALLOC_MAX_ROUTED) return MOE_ERR_UNSUPPORTED;   // beyond the fixed scratch
  if (!counts || !offsets || (R > 0 && (!idx || !src_tok || !slot_of))) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {idx, counts, offsets, src_tok, slot_of};
  for (const void* p : ps)
    if (p && !aligned16(p)) return MOE_ERR_ALIGNMENT;
  int dev = 0, maj = 0, min = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (maj != 10 || min != 3) return MOE_ERR_UNSUPPORTED;
  moe_status st = MOE_OK;
  int* scratch = scratch_address(&st);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nchunks = moe::route_chunks(R);
  if (nchunks > kMaxChunks) return MOE_ERR_UNSUPPORTED;   // cannot happen within the limit
  if (moe::launch_route_count(idx, R, c.E, scratch, s) != cudaSuccess) return MOE_ERR_CUDA;
  const int cap = moe::expert_capacity_rows(c.capacity_factor, c.T, c.k, c.E);
  if (moe::launch_route_scan(scratch, nchunks, c.E, cap, counts, offsets, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_route_scatter(idx, R, c.k, c.E, cap, scratch, offsets, src_tok, slot_of, s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
