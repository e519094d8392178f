// common.cuh -- shared definitions of the CUDA path: status codes, the
// work-plan layout produced by the planning kernel, the CP chunk arithmetic
// and THD (head-grouped) addressing.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/ccg.h"

namespace ccg {

constexpr int kMaxCP = 16;
constexpr int kPlanHeaderBytes = 256;

// Work plan written by the planning kernel into the head of the workspace.
struct PlanHeader {
  int32_t n_fwd[kMaxCP];   // forward items per ring step
  int32_t n_dq;            // dQ-pass items
  int32_t n_kv;            // dK/dV-pass items
  int32_t valid;           // 1 when the sequence promise held
  int32_t n_fwd_all;       // forward items of all planned steps (one combined list)
  int32_t pad[64 - kMaxCP - 4];
};
static_assert(sizeof(PlanHeader) == kPlanHeaderBytes, "plan header size");

// One unit of work: sequence b, chunk c, tile index inside the chunk; for
// forward items `step` is the ring step, for dK/dV items the kv head (0 in
// the dQ list).
struct WorkItem {
  int32_t b, c, tile, step;
};

// Arguments of the K-way LSE merge (a4).  CP-aware mode when cu_pad is
// non-null: partial presence follows the chunk structure and padding rows
// get O = 0 / LSE = -inf; otherwise a partial is absent where its LSE is -inf.
struct MergeArgs {
  const void* o_parts[kMaxCP];    // bf16 [rows][D]
  const float* lse_parts[kMaxCP]; // float [rows]
  int nparts;
  const int32_t* cu;
  const int32_t* cu_pad;
  int B, cp, hpg;
  int64_t T;
  void* o;                        // bf16 [rows][D], or strided (out_heads > 0)
  float* lse;
  int64_t rows;
  int D;
  const int32_t* status;          // may be null
  // out_heads > 0: the partials hold hpg heads per token and row r (token
  // r / hpg, head r % hpg) is written to output row (r / hpg) * out_heads +
  // out_h0 + r % hpg (a head subset of a [T][out_heads] tensor); 0: row r
  int out_heads, out_h0;
};

// Sizes shared by host and device.
struct Problem {
  int32_t B, hq, hkv, D, cp, C, head_groups;
  int64_t T;
  float scale_log2;      // softmax scale * log2(e)
  float scale;           // softmax scale
};

// Chunk c's owner under the load-balanced split: ranks hold c and 2CP-1-c.
__host__ __device__ __forceinline__ int chunk_owner(int c, int cp) {
  return c < cp ? c : 2 * cp - 1 - c;
}
__host__ __device__ __forceinline__ int ring_source(int r, int s, int cp) {
  return ((r - s) % cp + cp) % cp;
}

// KV chunks of rank `src` that query chunk `cq` sees; returns the count
// (0..2) and writes them ascending.
__host__ __device__ __forceinline__ int visible_kv_chunks(int cq, int src, int cp, int* out) {
  int n = 0;
  const int a = src, b = 2 * cp - 1 - src;
  if (a <= cq) out[n++] = a;
  if (b <= cq) out[n++] = b;
  return n;
}

// The same into two scalars (v1 only meaningful when two are visible): the
// kernels' tile iterators keep no indexed arrays.
__host__ __device__ __forceinline__ int visible_kv_chunks2(int cq, int src, int cp, int& v0, int& v1) {
  const int a = src, b = 2 * cp - 1 - src;
  v0 = a <= cq ? a : b;
  v1 = b;
  return (a <= cq ? 1 : 0) + (b <= cq ? 1 : 0);
}

// Row offset in a head-grouped THD tensor: element (t, h, d) lives at
// ((h / hpg) * T + t) * hpg * D + (h % hpg) * D + d.
__host__ __device__ __forceinline__ int64_t thd_row(int64_t t, int h, int hpg, int64_t T) {
  return (static_cast<int64_t>(h / hpg) * T + t) * hpg + (h % hpg);
}

// Sequence containing physical row t (cu_pad ascending, cu_pad[0] = 0).
__device__ __forceinline__ int find_sequence(const int32_t* __restrict__ cu_pad, int B, int64_t t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(__ldg(cu_pad + mid)) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Runs `set` (a per-device function attribute call) once for every device
// it is used on; concurrent first calls may both run it, which is harmless.
template <class F>
inline cudaError_t once_per_device(std::atomic<uint64_t>& done, F set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = set();
  if (e != cudaSuccess) return e;
  done.fetch_or(bit, std::memory_order_release);
  return cudaSuccess;
}

// Launch timing hooks (defined in api.cu): no-ops unless a profile is open
// on the calling host thread.
void prof_begin(const char* kernel_name, cudaStream_t stream);
void prof_end(cudaStream_t stream);

__device__ __forceinline__ bool status_bad(const int32_t* status) {
  return *reinterpret_cast<const volatile int32_t*>(status) != 0;
}

__device__ __forceinline__ void raise_status(int32_t* status, int32_t code) {
  atomicCAS(status, 0, code);
}

}  // namespace ccg
