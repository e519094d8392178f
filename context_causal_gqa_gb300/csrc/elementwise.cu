// elementwise.cu -- the HBM-bound steps of the path:
//   a4  K-way LSE merge of the per-step partial outputs,
//   a5  Delta = rowsum(O * dO) for the backward,
//   a2/a8  A2A head-split pack / unpack copies.
// All use 16-byte vector loads/stores and 64-bit row arithmetic.
#include <cuda_bf16.h>

#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace ccg {


namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Cached lookup of the sequence holding physical row t: rows handled by one
// thread are ascending, so the binary search runs only when t leaves the
// cached sequence.
struct SeqCache {
  int64_t lo = 1, hi = 0;   // empty
  int b = 0;
  __device__ __forceinline__ int get(const int32_t* cu_pad, int B, int64_t t) {
    if (t < lo || t >= hi) {
      b = find_sequence(cu_pad, B, t);
      lo = __ldg(cu_pad + b);
      hi = __ldg(cu_pad + b + 1);
    }
    return b;
  }
};

// Each block merges a contiguous range of rows (better DRAM locality and a
// cached sequence lookup); TPR threads per row, 16 bytes each.  NP bounds the
// number of partials (registers for NP 16-byte slices per thread).  Four
// blocks an SM (64 registers a thread): rows of early query chunks have few
// partials, so a thread has few loads in flight there, and the bytes in
// flight come from more resident threads instead (12.3 -> 10.9 ms on the
// large step against three blocks).  The grid has up to 64 blocks an SM
// (16 waves): rows of different query chunks carry 1 to CP partials, so
// short blocks let the waves even out that imbalance (11.0 -> 10.3 ms
// against 16 blocks an SM).
template <int TPR, int NP>
__global__ void __launch_bounds__(256, 4) lse_merge_kernel(MergeArgs a, int64_t rows_per_block) {
  if (a.status != nullptr && status_bad(a.status)) return;
  const int sub = threadIdx.x % TPR;
  constexpr int kRowsPerPass = 256 / TPR;
  const int64_t r_begin = blockIdx.x * rows_per_block;
  const int64_t r_end = min(a.rows, r_begin + rows_per_block);
  SeqCache sc;
  for (int64_t r = r_begin + threadIdx.x / TPR; r < r_end; r += kRowsPerPass) {
    int K = a.nparts;
    bool valid = true;
    if (a.cu_pad != nullptr) {
      const int64_t t = (r / a.hpg) % a.T;
      const int b = sc.get(a.cu_pad, a.B, t);
      const int start = static_cast<int>(sc.lo);
      const int pos = static_cast<int>(t - start);
      const int L = (static_cast<int>(sc.hi) - start) / (2 * a.cp);
      const int S = __ldg(a.cu + b + 1) - __ldg(a.cu + b);
      valid = pos < S;
      const int c = L > 0 ? pos / L : 0;
      K = c >= a.cp ? a.cp : c + 1;
    }
    // every partial's LSE and O slice is requested before any is used: the
    // loads depend only on the row's partial count, not on each other
    const int64_t off = r * a.D + sub * 8;
    float l[NP];
    uint4 u[NP];
#pragma unroll
    for (int s = 0; s < NP; ++s) {
      if (s < K) {
        l[s] = __ldg(a.lse_parts[s] + r);
        u[s] = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.o_parts[s]) + off));
      } else {
        l[s] = -INFINITY;
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int s = 0; s < NP; ++s) m = fmaxf(m, l[s]);
    uint4 outv;
    float lse_out;
    if (!valid || m == -INFINITY) {
      outv = make_uint4(0, 0, 0, 0);
      lse_out = -INFINITY;
    } else {
      float sigma = 0.f;
#pragma unroll
      for (int s = 0; s < NP; ++s)
        if (s < K) sigma += ex2_approx((l[s] - m) * kLog2e);
      lse_out = m + __logf(sigma);
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
      for (int s = 0; s < NP; ++s) {
        if (s < K && l[s] != -INFINITY) {
          const float w = ex2_approx((l[s] - lse_out) * kLog2e);
          float f[8];
          bf16x8_to_f32(u[s], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, f[i], acc[i]);
        }
      }
      outv.x = pack_bf16x2(acc[0], acc[1]);
      outv.y = pack_bf16x2(acc[2], acc[3]);
      outv.z = pack_bf16x2(acc[4], acc[5]);
      outv.w = pack_bf16x2(acc[6], acc[7]);
    }
    const int64_t ro = a.out_heads > 0 ? (r / a.hpg) * a.out_heads + a.out_h0 + r % a.hpg : r;
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) + ro * a.D + sub * 8) = outv;
    if (sub == 0) a.lse[ro] = lse_out;
  }
}

template <int TPR>
__global__ void __launch_bounds__(256)
bwd_dot_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
               int64_t rows, int D, int dout_heads, int64_t dout_pitch, float* __restrict__ delta,
               const int32_t* status) {
  if (status != nullptr && status_bad(status)) return;
  const int sub = threadIdx.x % TPR;
  const int64_t rows_per_block = 256 / TPR;
  const int64_t row0 = blockIdx.x * rows_per_block + threadIdx.x / TPR;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * rows_per_block;
  for (int64_t r = row0; r < rows; r += stride) {
    const int64_t off = r * D + sub * 8;
    // dO row r = (token r / H, head r % H), rows dout_pitch elements apart
    const int64_t off_do = (r / dout_heads) * dout_pitch + (r % dout_heads) * D + sub * 8;
    float a[8], b[8];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(o + off)), a);
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(dout + off_do)), b);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(a[i], b[i], acc);
#pragma unroll
    for (int w = TPR / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w, TPR);
    if (sub == 0) delta[r] = acc;
  }
}

// One warp per (head group g, sequence row t), each warp walking a contiguous
// range of such rows: copies hpg*D contiguous 16-bit elements between the
// rank-major row and the head-split row.  Rank-major row of sequence row t:
// rank r = owner of t's chunk; r*T/CP + start_b/CP + (chunk is r ? 0 : L_b) + i.
// Every lane keeps four 16-byte loads in flight: rows of 128 vectors or more
// are copied one at a time, shorter rows (one head of 256 or 128 columns)
// several per warp iteration, each lane loading from its own row.
template <bool kPack>
__global__ void __launch_bounds__(256)
thd_permute_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                   const int32_t* __restrict__ cu_pad, int B, int64_t T, int H, int D, int cp,
                   int64_t rows_per_warp, int32_t* status) {
  if (status_bad(status)) return;
  const int lane = threadIdx.x & 31;
  const int C = 2 * cp;
  const int hpg = H / cp;
  const int w16 = hpg * D / 8;                               // uint4 per head-split row
  const int64_t row_w16 = static_cast<int64_t>(H) * D / 8;  // uint4 per rank-major row
  const int64_t nrows = static_cast<int64_t>(cp) * T;
  const int64_t warp_id = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t w_begin = warp_id * rows_per_warp;
  const int64_t w_end = min(nrows, w_begin + rows_per_warp);
  SeqCache sc;                    // rows are visited in ascending order by every lane
  // source and destination of head-split row w, and the number of rows from
  // w on that stay in w's chunk (their rank-major rows are consecutive too);
  // false if w's sequence breaks the promise
  auto row_ptrs = [&](int64_t w, const uint4*& s, uint4*& d, int& run) -> bool {
    const int g = static_cast<int>(w / T);
    const int64_t t = w - static_cast<int64_t>(g) * T;
    sc.get(cu_pad, B, t);
    const int start = static_cast<int>(sc.lo);
    const int P = static_cast<int>(sc.hi) - start;
    if (P % C != 0 || P <= 0) return false;
    const int L = P / C;
    const int pos = static_cast<int>(t - start);
    const int c = pos / L, i = pos - c * L;
    const int r = chunk_owner(c, cp);
    const int64_t pr = static_cast<int64_t>(r) * (T / cp) + start / cp + (c == r ? 0 : L) + i;
    run = L - i;
    if (kPack) {
      s = src + pr * row_w16 + static_cast<int64_t>(g) * w16;
      d = dst + w * w16;
    } else {
      s = src + w * w16;
      d = dst + pr * row_w16 + static_cast<int64_t>(g) * w16;
    }
    return true;
  };
  if (w16 >= 128) {
    for (int64_t w = w_begin; w < w_end; ++w) {
      const uint4* s;
      uint4* d;
      int run;
      if (!row_ptrs(w, s, d, run)) {
        if (lane == 0) raise_status(status, CCG_ERR_SEQLENS);
        return;
      }
      int u = lane;
      for (; u + 96 < w16; u += 128) {
        const uint4 x0 = __ldg(s + u), x1 = __ldg(s + u + 32), x2 = __ldg(s + u + 64), x3 = __ldg(s + u + 96);
        d[u] = x0;
        d[u + 32] = x1;
        d[u + 64] = x2;
        d[u + 96] = x3;
      }
      for (; u < w16; u += 32) d[u] = __ldg(s + u);
    }
    return;
  }
  const int nb = 128 / w16;                                  // rows per warp iteration
  const int span = nb * w16;                                 // vectors per warp iteration (<= 128)
  // strides between consecutive rows of one chunk on the source / destination side
  const int64_t s_step = kPack ? row_w16 : w16, d_step = kPack ? w16 : row_w16;
  for (int64_t w = w_begin; w < w_end; w += nb) {
    const uint4* s0;
    uint4* d0;
    int run;
    if (!row_ptrs(w, s0, d0, run)) {                          // the same for every lane
      if (lane == 0) raise_status(status, CCG_ERR_SEQLENS);
      return;
    }
    uint4 x[4];
    uint4* dp[4];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int f = lane + 32 * j;
      const int k = f / w16, u = f - k * w16;
      dp[j] = nullptr;
      if (f < span && w + k < w_end) {
        const uint4* s = s0 + k * s_step;
        uint4* d = d0 + k * d_step;
        int run2;
        if (k >= run && !row_ptrs(w + k, s, d, run2)) {      // the batch crosses a chunk end
          bad = true;
        } else {
          x[j] = __ldg(s + u);
          dp[j] = d + u;
        }
      }
    }
    if (__any_sync(0xffffffffu, bad)) {
      if (lane == 0) raise_status(status, CCG_ERR_SEQLENS);
      return;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (dp[j] != nullptr) *dp[j] = x[j];
  }
}

// O = 0 and LSE = -inf on padding rows (positions >= S_b of their sequence):
// one warp per token, walking a contiguous range of tokens.
__global__ void __launch_bounds__(256)
pad_rows_kernel(uint4* __restrict__ o, float* __restrict__ lse, const int32_t* __restrict__ cu,
                const int32_t* __restrict__ cu_pad, int B, int64_t T, int H, int hpg, int D,
                int64_t tokens_per_warp, const int32_t* status) {
  if (status_bad(status)) return;
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t t_begin = warp_id * tokens_per_warp, t_end = min(T, t_begin + tokens_per_warp);
  const int w16 = D / 8;
  SeqCache sc;
  for (int64_t t = t_begin; t < t_end; ++t) {
    const int b = sc.get(cu_pad, B, t);
    const int S = __ldg(cu + b + 1) - __ldg(cu + b);
    if (t - sc.lo < S) continue;                     // a real token: written by the attention kernel
    for (int h = 0; h < H; ++h) {
      const int64_t row = thd_row(t, h, hpg, T);
      for (int u = lane; u < w16; u += 32) o[row * w16 + u] = make_uint4(0, 0, 0, 0);
      if (lane == 0) lse[row] = -INFINITY;
    }
  }
}

int grid_for(int64_t units, int per_block, int max_blocks) {
  int64_t g = (units + per_block - 1) / per_block;
  if (g > max_blocks) g = max_blocks;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_lse_merge(const MergeArgs& a, int num_sms, cudaStream_t stream) {
  const int tpr = a.D / 8;
  const int grid = grid_for(a.rows, 256 / tpr, num_sms * 64);
  const int64_t rpb = (a.rows + grid - 1) / grid;
  auto go = [&](auto np) -> cudaError_t {
    constexpr int NP = decltype(np)::value;
    if (tpr == 16) lse_merge_kernel<16, NP><<<grid, 256, 0, stream>>>(a, rpb);
    else if (tpr == 32) lse_merge_kernel<32, NP><<<grid, 256, 0, stream>>>(a, rpb);
    else return cudaErrorInvalidValue;
    return cudaSuccess;
  };
  cudaError_t e;
  if (a.nparts <= 2) e = go(std::integral_constant<int, 2>{});
  else if (a.nparts <= 4) e = go(std::integral_constant<int, 4>{});
  else if (a.nparts <= 8) e = go(std::integral_constant<int, 8>{});
  else e = go(std::integral_constant<int, kMaxCP>{});
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_pad_rows(void* o, float* lse, const int32_t* cu, const int32_t* cu_pad, int B, int64_t T,
                            int H, int hpg, int D, const int32_t* status, int num_sms, cudaStream_t stream) {
  const int grid = grid_for(T, 8, num_sms * 16);
  const int64_t warps = static_cast<int64_t>(grid) * 8;
  const int64_t tpw = (T + warps - 1) / warps;
  pad_rows_kernel<<<grid, 256, 0, stream>>>(static_cast<uint4*>(o), lse, cu, cu_pad, B, T, H, hpg, D, tpw, status);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dot(const void* o, const void* dout, int64_t rows, int D, int dout_heads,
                           int64_t dout_pitch, float* delta, const int32_t* status, int num_sms,
                           cudaStream_t stream) {
  const int tpr = D / 8;
  const int grid = grid_for(rows, 256 / tpr, num_sms * 16);
  auto* po = static_cast<const __nv_bfloat16*>(o);
  auto* pd = static_cast<const __nv_bfloat16*>(dout);
  if (tpr == 16) bwd_dot_kernel<16><<<grid, 256, 0, stream>>>(po, pd, rows, D, dout_heads, dout_pitch, delta, status);
  else if (tpr == 32) bwd_dot_kernel<32><<<grid, 256, 0, stream>>>(po, pd, rows, D, dout_heads, dout_pitch, delta, status);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_thd_permute(bool pack, const void* src, void* dst, const int32_t* cu_pad, int B,
                               int64_t T, int H, int D, int cp, int32_t* status, int num_sms,
                               cudaStream_t stream) {
  const int64_t nrows = static_cast<int64_t>(cp) * T;
  // up to 64 blocks an SM: shorter row ranges a warp (1.73 -> 1.67 ms a
  // launch at D=256 against 16 blocks an SM)
  const int grid = grid_for(nrows, 8, num_sms * 64);
  const int64_t warps = static_cast<int64_t>(grid) * 8;
  const int64_t rpw = (nrows + warps - 1) / warps;
  auto* s = static_cast<const uint4*>(src);
  auto* d = static_cast<uint4*>(dst);
  if (pack) thd_permute_kernel<true><<<grid, 256, 0, stream>>>(s, d, cu_pad, B, T, H, D, cp, rpw, status);
  else thd_permute_kernel<false><<<grid, 256, 0, stream>>>(s, d, cu_pad, B, T, H, D, cp, rpw, status);
  return cudaGetLastError();
}

}  // namespace ccg
