// plan.cu -- the CP split (a1): validates the sequence promise on device
// and writes the work plan every later kernel reads: forward items per ring
// step, dQ-pass items and dK/dV-pass items.
//
// TransformerEngine PR "Optimize context parallel attention layouts and
// gradient accumulation", Changes: the device re-validates the promised
// sequence lengths and physical offsets at every call.  Here a broken
// promise writes CCG_ERR_SEQLENS into the status word (no trap) and an
// empty plan, so that every later kernel returns without writing.
#include "common.cuh"
#include "ptx.cuh"

namespace ccg {

namespace {

constexpr int kPlanThreads = 1024;

// Inclusive block-wide prefix sum of one int per thread; returns the
// inclusive value and the block total through *total.
__device__ int block_inclusive_scan(int v, int* total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int prefix = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return x + prefix;
}

// Emits, for i = 0..n-1 in order, count(i) consecutive items written by
// write(i, first_slot, count).  Returns the running slot after the last.
template <class CountF, class WriteF>
__device__ int block_emit(int n, int base, CountF count, WriteF write) {
  int carry = base;
  for (int start = 0; start < n; start += blockDim.x) {
    const int i = start + threadIdx.x;
    const int c = i < n ? count(i) : 0;
    int total;
    const int incl = block_inclusive_scan(c, &total);
    if (i < n && c > 0) write(i, carry + incl - c, c);
    carry += total;
  }
  return carry;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_pad, int B, int64_t T,
            int cp, int hkv, int bm, int bn, int cap_q, int cap_kv, int want, int step_only, PlanHeader* hdr,
            WorkItem* fwd_items, WorkItem* dq_items, WorkItem* kv_items, int64_t max_pad, int64_t* ds_base,
            int32_t* status) {
  __shared__ int bad;
  const int C = 2 * cp;
  if (threadIdx.x == 0) {
    bad = 0;
    if (__ldg(cu) != 0 || __ldg(cu_pad) != 0 || static_cast<int64_t>(__ldg(cu_pad + B)) != T) bad = 1;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int S = __ldg(cu + b + 1) - __ldg(cu + b);
    const int P = __ldg(cu_pad + b + 1) - __ldg(cu_pad + b);
    if (S < 0 || P < S || P % C != 0) atomicExch(&bad, 1);
    if (ds_base != nullptr && P > max_pad) atomicExch(&bad, 1);    // the padded-length bound of the dS backward
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      raise_status(status, CCG_ERR_SEQLENS);
      for (int s = 0; s < kMaxCP; ++s) hdr->n_fwd[s] = 0;
      hdr->n_fwd_all = 0;
      hdr->n_dq = 0;
      hdr->n_kv = 0;
      hdr->valid = 0;
    }
    return;
  }
  const int npairs = B * C;
  auto seq_len = [&](int b) { return __ldg(cu + b + 1) - __ldg(cu + b); };
  auto chunk_len = [&](int b) { return (__ldg(cu_pad + b + 1) - __ldg(cu_pad + b)) / C; };
  // tiles of `rows` rows covering the real tokens of chunk c of sequence b
  auto valid_tiles = [&](int b, int c, int rows) {
    const int L = chunk_len(b);
    const int real = min(L, max(0, seq_len(b) - c * L));
    return (real + rows - 1) / rows;
  };
  auto all_tiles = [&](int b, int rows) { return (chunk_len(b) + rows - 1) / rows; };

  int overflow = 0;
  if (want & 1) {
    // one combined list over the planned ring steps (all, or only `step_only`),
    // heavy items first: two visible KV chunks, then one full chunk, then the
    // diagonal chunk alone; inside a class by step, sequence, chunk, tile
    int slot = 0;
    const int cap_all = cp * cap_q;
    for (int cls = 0; cls < 3; ++cls) {
      for (int s = 0; s < cp; ++s) {
        if (step_only >= 0 && s != step_only) continue;
        auto count = [&](int i) {
          const int b = i / C, c = i % C;
          int vis[2];
          const int nv = visible_kv_chunks(c, ring_source(chunk_owner(c, cp), s, cp), cp, vis);
          int k = nv == 2 ? 0 : (nv == 1 ? (vis[0] == c ? 2 : 1) : -1);
          return k == cls ? valid_tiles(b, c, bm) : 0;
        };
        auto write = [&](int i, int first, int n) {
          const int b = i / C, c = i % C;
          for (int t = 0; t < n && first + t < cap_all; ++t) fwd_items[first + t] = WorkItem{b, c, t, s};
        };
        slot = block_emit(npairs, slot, count, write);
      }
    }
    if (slot > cap_all) overflow = 1;
    if (threadIdx.x == 0) {
      hdr->n_fwd_all = min(slot, cap_all);
      for (int s = 0; s < kMaxCP; ++s) hdr->n_fwd[s] = 0;
    }
  }
  if (want & 4) {
    // fused forward: one item per query tile with real rows, all ring steps of
    // its rank; later query chunks see more keys, so they go first
    int slot = 0;
    const int cap_all = cp * cap_q;
    for (int c = C - 1; c >= 0; --c) {
      auto count = [&](int b) { return valid_tiles(b, c, bm); };
      auto write = [&](int b, int first, int n) {
        for (int t = 0; t < n && first + t < cap_all; ++t) fwd_items[first + t] = WorkItem{b, c, t, -1};
      };
      slot = block_emit(B, slot, count, write);
    }
    if (slot > cap_all) overflow = 1;
    if (threadIdx.x == 0) {
      hdr->n_fwd_all = min(slot, cap_all);
      for (int s = 0; s < kMaxCP; ++s) hdr->n_fwd[s] = 0;
    }
  }
  if (want & 2) {
    // dQ pass: sequence-major; later query chunks see more keys, so they go first
    int slot = 0;
    {
      auto count = [&](int i) { return all_tiles(i / C, bm); };
      auto write = [&](int i, int first, int n) {
        const int b = i / C, c = C - 1 - i % C;
        for (int t = 0; t < n && first + t < cap_q; ++t) dq_items[first + t] = WorkItem{b, c, t, 0};
      };
      slot = block_emit(B * C, 0, count, write);
    }
    if (slot > cap_q) overflow = 1;
    if (threadIdx.x == 0) hdr->n_dq = min(slot, cap_q);
    // dK/dV pass: one item per (KV tile, kv head), (sequence, kv head)-major,
    // so that the CTAs in flight stream the Q/dO of few kv heads' groups;
    // earlier KV chunks are seen by more queries, so they go first.  The dS
    // backward (CTA pairs, one launch per kv head) instead takes one item per
    // pair of KV tiles (2i, 2i+1) of a chunk, kv-head-major, so that a kv
    // head's items are one contiguous n_kv / hkv range.
    if (ds_base != nullptr) {
      auto count = [&](int i) { return (all_tiles((i / C) % B, bn) + 1) / 2; };
      auto write = [&](int i, int first, int n) {
        const int g = i / (B * C), b = (i / C) % B, j = i % C;
        for (int t = 0; t < n && first + t < cap_kv; ++t) kv_items[first + t] = WorkItem{b, j, t, g};
      };
      slot = block_emit(hkv * B * C, 0, count, write);
    } else {
      auto count = [&](int i) { return all_tiles(i / (hkv * C), bn); };
      auto write = [&](int i, int first, int n) {
        const int b = i / (hkv * C), g = (i / C) % hkv, j = i % C;
        for (int t = 0; t < n && first + t < cap_kv; ++t) kv_items[first + t] = WorkItem{b, j, t, g};
      };
      slot = block_emit(B * hkv * C, 0, count, write);
    }
    if (slot > cap_kv) overflow = 1;
    if (threadIdx.x == 0) hdr->n_kv = min(slot, cap_kv);
  }
  // dS backward: each sequence's first tile in a q head's dS region (t^2 *
  // 2CP(2CP+1)/2 tiles for t 128-row tiles a chunk; the host sized the region
  // from the padded-length bound checked above)
  if (ds_base != nullptr && threadIdx.x == 0) {
    int64_t run = 0;
    for (int b = 0; b < B; ++b) {
      const int64_t t = (chunk_len(b) + 127) / 128;
      ds_base[b] = run;
      run += t * t * (C * (C + 1) / 2);
    }
    ds_base[B] = run;
  }
  if (threadIdx.x == 0) {
    hdr->valid = 1;
    if (overflow) raise_status(status, CCG_ERR_SEQLENS);
  }
}

__global__ void chunk_table_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_pad,
                                   int B, int64_t T, int cp, int32_t* table, int32_t* status) {
  const int C = 2 * cp;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * C) return;
  const int b = i / C, c = i % C;
  const int S = __ldg(cu + b + 1) - __ldg(cu + b);
  const int P = __ldg(cu_pad + b + 1) - __ldg(cu_pad + b);
  bool ok = S >= 0 && P >= S && P % C == 0;
  if (i == 0) ok = ok && __ldg(cu) == 0 && __ldg(cu_pad) == 0 && static_cast<int64_t>(__ldg(cu_pad + B)) == T;
  if (!ok) raise_status(status, CCG_ERR_SEQLENS);
  const int L = ok ? P / C : 0;
  table[2 * i + 0] = __ldg(cu_pad + b) + c * L;
  table[2 * i + 1] = L;
}

// A bounded wait on a barrier nothing arrives at: gives up after limit_ns and
// records the timeout, like every wait in the attention kernels.
__global__ void bounded_wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int never = 0;
    if (!mbar_wait(&bar, 0, &never, limit_ns)) raise_status(status, CCG_ERR_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int32_t* status, uint32_t limit_us, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(status, static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError();
}

cudaError_t launch_plan(const int32_t* cu, const int32_t* cu_pad, int B, int64_t T, int cp, int hkv, int bm,
                        int bn, int cap_q, int cap_kv, int want, int step_only, PlanHeader* hdr,
                        WorkItem* fwd_items, WorkItem* dq_items, WorkItem* kv_items,
                        int32_t* status, cudaStream_t stream, int64_t max_pad, int64_t* ds_base) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(cu, cu_pad, B, T, cp, hkv, bm, bn, cap_q, cap_kv, want, step_only,
                                               hdr, fwd_items, dq_items, kv_items, max_pad, ds_base, status);
  return cudaGetLastError();
}

cudaError_t launch_chunk_table(const int32_t* cu, const int32_t* cu_pad, int B, int64_t T, int cp,
                               int32_t* table, int32_t* status, cudaStream_t stream) {
  const int n = B * 2 * cp;
  chunk_table_kernel<<<(n + 255) / 256, 256, 0, stream>>>(cu, cu_pad, B, T, cp, table, status);
  return cudaGetLastError();
}

}  // namespace ccg
