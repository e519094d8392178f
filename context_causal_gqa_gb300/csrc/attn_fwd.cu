// attn_fwd.cu -- a3: one ring step of the CP-emulated causal GQA forward on
// the 5th-generation tensor cores (sm_103a).
//
// TransformerEngine PR "Optimize context parallel attention layouts and
// gradient accumulation", Independent-node complete-CP evidence: each CP
// rank attends its two query chunks against the KV it holds at a ring
// step and keeps the partial output with its LSE ("Stats") for the merge.
//
// One CTA = one 128-row query tile of NH q heads that share one kv head
// (GQA K/V reuse: every K/V tile is loaded once for the NH heads), looping
// over the visible KV tiles of the step (causal block skipping: KV tiles past
// the tile's last row are never loaded).  Roles:
//   warp 0     TMA producer: Q once, then K/V tiles through an NSTAGE ring
//   warp 1     MMA issuer (one thread): S = Q K^T (SMEM x SMEM -> TMEM),
//              O += P V (P from TMEM, V from SMEM -> TMEM)
//   warp 2     TMEM allocator
//   warps 4..  one 128-thread softmax warpgroup per head, one row per thread:
//              online softmax in registers, P written back to TMEM as BF16,
//              lazy O rescaling, epilogue O / l and LSE.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ccg {

namespace {

constexpr int kBM = 128;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale only past 2^8 growth

template <int D, int NH>
struct FwdCfg {
  static constexpr int BN = D == 128 ? 128 : 64;
  static constexpr int SBUF = NH == 1 ? 2 : 1;
  static constexpr int NSTAGE = 2;
  static constexpr int KCH = D / 64;                       // 64-wide (128-byte) column chunks
  static constexpr int Q_BYTES = kBM * D * 2;              // one head
  static constexpr int KV_BYTES = BN * D * 2;              // one K (or V) tile
  static constexpr int SMEM_Q = 0;
  static constexpr int SMEM_K = SMEM_Q + NH * Q_BYTES;
  static constexpr int SMEM_V = SMEM_K + NSTAGE * KV_BYTES;
  static constexpr int SMEM_BAR = SMEM_V + NSTAGE * KV_BYTES;
  static constexpr int SMEM_TOTAL = SMEM_BAR + 256;
  static constexpr int TMEM_HEAD = SBUF * BN + D;
  static constexpr int TMEM_USED = NH * TMEM_HEAD;
  static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : (TMEM_USED <= 256 ? 256 : 512);
  static constexpr int THREADS = 128 + 128 * NH;
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(SMEM_TOTAL + 1024 <= 232448, "SMEM budget");
};

struct FwdParams {
  const WorkItem* items;        // this step's items
  const PlanHeader* hdr;
  const int32_t* cu;
  const int32_t* cu_pad;
  __nv_bfloat16* o;             // partial O of this step, head-grouped THD
  float* lse;                   // partial LSE of this step
  int32_t* status;
  int step, cp, hq, hkv, hpg_q, hpg_kv;
  int64_t T;
  float scale_log2;
};

// KV tiles of one work item: up to two segments (KV chunks of the source
// rank), each [lo, hi) in sequence positions; `diag` marks the causal chunk.
struct TilePlan {
  int q_lo, q_hi;               // rows [q_lo, q_hi) are written
  int nseg;
  int seg_lo[2], seg_hi[2], seg_tiles[2];
  bool seg_diag[2];
  int ntiles;
  int seq_start;
};

template <int BN>
__device__ __forceinline__ TilePlan make_tile_plan(const FwdParams& p, const WorkItem& it) {
  TilePlan tp;
  const int C = 2 * p.cp;
  const int start = __ldg(p.cu_pad + it.b);
  const int S = __ldg(p.cu + it.b + 1) - __ldg(p.cu + it.b);
  const int L = (__ldg(p.cu_pad + it.b + 1) - start) / C;
  tp.seq_start = start;
  tp.q_lo = it.c * L + it.tile * kBM;
  tp.q_hi = min(min(tp.q_lo + kBM, (it.c + 1) * L), S);
  int vis[2];
  const int src = ring_source(chunk_owner(it.c, p.cp), p.step, p.cp);
  tp.nseg = visible_kv_chunks(it.c, src, p.cp, vis);
  tp.ntiles = 0;
  for (int i = 0; i < 2; ++i) {
    if (i < tp.nseg) {
      const int j = vis[i];
      tp.seg_diag[i] = (j == it.c);
      tp.seg_lo[i] = j * L;
      int hi = min((j + 1) * L, S);
      if (tp.seg_diag[i]) hi = min(hi, tp.q_hi);   // keys past the last row are invisible
      tp.seg_hi[i] = hi;
      tp.seg_tiles[i] = hi > tp.seg_lo[i] ? (hi - tp.seg_lo[i] + BN - 1) / BN : 0;
    } else {
      tp.seg_diag[i] = false;
      tp.seg_lo[i] = tp.seg_hi[i] = 0;
      tp.seg_tiles[i] = 0;
    }
    tp.ntiles += tp.seg_tiles[i];
  }
  return tp;
}

// Sequence position of the first key of tile j, its segment end and kind.
template <int BN>
__device__ __forceinline__ void tile_of(const TilePlan& tp, int j, int* k0, int* khi, bool* diag) {
  if (j < tp.seg_tiles[0]) {
    *k0 = tp.seg_lo[0] + j * BN;
    *khi = tp.seg_hi[0];
    *diag = tp.seg_diag[0];
  } else {
    j -= tp.seg_tiles[0];
    *k0 = tp.seg_lo[1] + j * BN;
    *khi = tp.seg_hi[1];
    *diag = tp.seg_diag[1];
  }
}

template <int D, int NH>
__global__ void __launch_bounds__(FwdCfg<D, NH>::THREADS, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Cfg = FwdCfg<D, NH>;
  constexpr int BN = Cfg::BN, SBUF = Cfg::SBUF, NSTAGE = Cfg::NSTAGE, KCH = Cfg::KCH;

  const int nhg = p.hq / NH;                           // head groups per item
  const int item_idx = blockIdx.x / nhg;
  if (item_idx >= p.hdr->n_fwd[p.step]) return;
  if (status_bad(p.status)) return;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;                        // [NSTAGE]
  uint64_t* kv_empty = kv_full + NSTAGE;               // [NSTAGE]
  uint64_t* s_full = kv_empty + NSTAGE;                // [NH][SBUF]
  uint64_t* p_full = s_full + NH * SBUF;               // [NH][SBUF]
  uint64_t* o_done = p_full + NH * SBUF;               // [NH]
  uint64_t* mma_done = o_done + NH;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[item_idx];
  const TilePlan tp = make_tile_plan<BN>(p, it);
  const int h0 = (blockIdx.x % nhg) * NH;              // first q head of this CTA
  const int g = h0 / (p.hq / p.hkv);                   // shared kv head

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(kv_full + s, 1);
      mbar_init(kv_empty + s, 1);
    }
    for (int i = 0; i < NH * SBUF; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 128);
    }
    for (int h = 0; h < NH; ++h) mbar_init(o_done + h, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n = tp.ntiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int qrow_base = tp.seq_start + tp.q_lo;
      mbar_arrive_expect_tx(q_full, NH * Cfg::Q_BYTES);
      for (int h = 0; h < NH; ++h) {
        const int hq = h0 + h;
        const int row = static_cast<int>((hq / p.hpg_q) * p.T) + qrow_base;
        for (int kc = 0; kc < KCH; ++kc)
          tma_load_3d(smem + Cfg::SMEM_Q + h * Cfg::Q_BYTES + kc * kBM * 128, &tm_q, kc * 64,
                      hq % p.hpg_q, row, q_full);
      }
      const int kv_group_row = static_cast<int>((g / p.hpg_kv) * p.T) + tp.seq_start;
      int issued[NSTAGE] = {};
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        const int st = j % NSTAGE;
        if (j >= NSTAGE) ok = mbar_wait(kv_empty + st, ((j / NSTAGE) - 1) & 1, abort_flag);
        if (!ok) break;
        int k0, khi;
        bool diag;
        tile_of<BN>(tp, j, &k0, &khi, &diag);
        mbar_arrive_expect_tx(kv_full + st, 2 * Cfg::KV_BYTES);
        for (int kc = 0; kc < KCH; ++kc) {
          tma_load_3d(smem + Cfg::SMEM_K + st * Cfg::KV_BYTES + kc * BN * 128, &tm_k, kc * 64,
                      g % p.hpg_kv, kv_group_row + k0, kv_full + st);
          tma_load_3d(smem + Cfg::SMEM_V + st * Cfg::KV_BYTES + kc * BN * 128, &tm_v, kc * 64,
                      g % p.hpg_kv, kv_group_row + k0, kv_full + st);
        }
        issued[st]++;
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // never leave a copy in flight into shared memory we are about to release
      mbar_wait(q_full, 0, abort_flag, 200000000ull);
      for (int s = 0; s < NSTAGE; ++s)
        if (issued[s] > 0) {
          volatile int never = 0;
          mbar_wait(kv_full + s, (issued[s] - 1) & 1, &never, 200000000ull);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, BN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, false, true);
      const uint32_t q_base = smem_u32(smem + Cfg::SMEM_Q);
      const uint32_t k_base = smem_u32(smem + Cfg::SMEM_K);
      const uint32_t v_base = smem_u32(smem + Cfg::SMEM_V);
      uint64_t q_desc[NH], k_desc[NSTAGE], v_desc[NSTAGE];
#pragma unroll
      for (int h = 0; h < NH; ++h) q_desc[h] = smem_desc_sw128(q_base + h * Cfg::Q_BYTES, 16, 1024);
#pragma unroll
      for (int st = 0; st < NSTAGE; ++st) {
        k_desc[st] = smem_desc_sw128(k_base + st * Cfg::KV_BYTES, 16, 1024);
        v_desc[st] = smem_desc_sw128(v_base + st * Cfg::KV_BYTES, BN * 128, 1024);
      }
      bool ok = mbar_wait(q_full, 0, abort_flag);
      tc_fence_after();
      auto issue_s = [&](int h, int j) {
        const int st = j % NSTAGE, buf = j % SBUF;
        const uint32_t d_tmem = tmem + h * Cfg::TMEM_HEAD + buf * BN;
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss(d_tmem, q_desc[h] + kmajor_step(kBM, k), k_desc[st] + kmajor_step(BN, k), idesc_s,
                  k > 0 ? 1u : 0u);
        umma_commit(s_full + h * SBUF + buf);
      };
      auto issue_pv = [&](int h, int j) {
        const int st = j % NSTAGE, buf = j % SBUF;
        const uint32_t d_tmem = tmem + h * Cfg::TMEM_HEAD + SBUF * BN;
        const uint32_t p_tmem = tmem + h * Cfg::TMEM_HEAD + buf * BN;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          umma_ts(d_tmem, p_tmem + k * 8, v_desc[st] + mnmajor_step(k), idesc_o, (j > 0 || k > 0) ? 1u : 0u);
        umma_commit(o_done + h);
      };
      if (ok && n > 0) {
        ok = mbar_wait(kv_full + 0, 0, abort_flag);
        tc_fence_after();
        if (ok)
          for (int h = 0; h < NH; ++h) issue_s(h, 0);
      }
      for (int j = 0; j < n && ok; ++j) {
        const int st = j % NSTAGE;
        const bool has_next = j + 1 < n;
        bool next_ready = false;
        if (SBUF == 2 && has_next) {
          ok = mbar_wait(kv_full + (j + 1) % NSTAGE, ((j + 1) / NSTAGE) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          next_ready = true;
          issue_s(0, j + 1);
        }
        for (int h = 0; h < NH && ok; ++h) {
          const int buf = j % SBUF;
          ok = mbar_wait(p_full + h * SBUF + buf, (j / SBUF) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          issue_pv(h, j);
          if (SBUF == 1 && has_next) {
            if (!next_ready) {
              ok = mbar_wait(kv_full + (j + 1) % NSTAGE, ((j + 1) / NSTAGE) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
              next_ready = true;
            }
            issue_s(h, j + 1);
          }
        }
        umma_commit(kv_empty + st);
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(mma_done);
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, 200000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int h = (warp - 4) >> 2;
    const int row = ((warp & 3) << 5) + lane;         // TMEM lane == tile row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_head = tmem + lane_base + h * Cfg::TMEM_HEAD;
    const uint32_t t_o = t_head + SBUF * BN;
    const int q_pos = tp.q_lo + row;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int buf = j % SBUF;
      ok = __all_sync(0xffffffffu, mbar_wait(s_full + h * SBUF + buf, (j / SBUF) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      int k0, khi;
      bool diag;
      tile_of<BN>(tp, j, &k0, &khi, &diag);
      // keys visible to this row: k < kend (segment end, and k <= q_pos on the diagonal chunk)
      const int kend = diag ? min(khi, q_pos + 1) : khi;
      const int nvalid = kend - k0;                     // may be <= 0 or >= BN
      const uint32_t t_s = t_head + buf * BN;
      uint32_t r[32];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        tmem_ld32(t_s + c * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const float sv = __uint_as_float(r[x]) * p.scale_log2;
          mx = (c * 32 + x < nvalid) ? fmaxf(mx, sv) : mx;
        }
      }
      float alpha = 1.f;
      if (mx > m) {
        if (m == -INFINITY) {
          m = mx;
        } else if (mx > m + kRescaleThreshold) {
          alpha = ex2_approx(m - mx);
          m = mx;
        }
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        tmem_ld32(t_s + c * 32, r);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const int c0 = c * 32 + 2 * x;
          const float p0 = (c0 < nvalid) ? ex2_approx(__uint_as_float(r[2 * x]) * p.scale_log2 - m_use) : 0.f;
          const float p1 = (c0 + 1 < nvalid) ? ex2_approx(__uint_as_float(r[2 * x + 1]) * p.scale_log2 - m_use) : 0.f;
          psum += p0 + p1;
          pk[x] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + c * 16, pk);
      }
      tmem_wait_st();
      l = l * alpha + psum;
      // consume the previous P V product's completion (every phase, in order,
      // so that parity waits stay unambiguous); it is needed before O may be
      // rescaled and costs nothing when it has already landed
      if (j > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(o_done + h, (j - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          tmem_ld32(t_o + c * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
          tmem_st32(t_o + c * 32, r);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(p_full + h * SBUF + buf);
    }
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_done + h, (n - 1) & 1, abort_flag));
    if (!ok) {
      raise_status(p.status, CCG_ERR_TIMEOUT);
      *abort_flag = 1;
    } else if (n > 0) {
      tc_fence_after();
      const bool valid = q_pos < tp.q_hi;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const int hq = h0 + h;
      const int64_t orow = thd_row(tp.seq_start + q_pos, hq, p.hpg_q, p.T);
      uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D);
      uint32_t r[32];
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(t_o + c * 32, r);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(r[8 * v4 + 0]) * inv_l, __uint_as_float(r[8 * v4 + 1]) * inv_l);
            u.y = pack_bf16x2(__uint_as_float(r[8 * v4 + 2]) * inv_l, __uint_as_float(r[8 * v4 + 3]) * inv_l);
            u.z = pack_bf16x2(__uint_as_float(r[8 * v4 + 4]) * inv_l, __uint_as_float(r[8 * v4 + 5]) * inv_l);
            u.w = pack_bf16x2(__uint_as_float(r[8 * v4 + 6]) * inv_l, __uint_as_float(r[8 * v4 + 7]) * inv_l);
            dst[c * 4 + v4] = u;
          }
        }
      }
      if (valid) p.lse[orow] = (m + __log2f(l)) * kLn2;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

template <int D, int NH>
cudaError_t launch_fwd_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, int grid_x, cudaStream_t stream) {
  using Cfg = FwdCfg<D, NH>;
  auto kern = attn_fwd_kernel<D, NH>;
  static bool attr_set = false;
  const int smem = Cfg::SMEM_TOTAL + 1024;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // consecutive CTAs share one item (same K/V tiles, different heads): the
  // K/V tiles they read stay hot in L2
  const int64_t grid = static_cast<int64_t>(grid_x) * (p.hq / NH);
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(grid), Cfg::THREADS, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

int fwd_kv_tile_rows(int D) { return D == 128 ? FwdCfg<128, 2>::BN : FwdCfg<256, 1>::BN; }
int fwd_heads_per_cta(int D, int group) { return (D == 128 && group % 2 == 0) ? 2 : 1; }

cudaError_t launch_attn_fwd_step(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const WorkItem* items, const PlanHeader* hdr, const int32_t* cu,
                                 const int32_t* cu_pad, void* o, float* lse, int32_t* status,
                                 int step, int cp, int hq, int hkv, int head_groups, int64_t T,
                                 int D, float scale, int grid_x, cudaStream_t stream) {
  FwdParams p;
  p.items = items;
  p.hdr = hdr;
  p.cu = cu;
  p.cu_pad = cu_pad;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.status = status;
  p.step = step;
  p.cp = cp;
  p.hq = hq;
  p.hkv = hkv;
  p.hpg_q = hq / head_groups;
  p.hpg_kv = hkv / head_groups;
  p.T = T;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int nh = fwd_heads_per_cta(D, hq / hkv);
  if (D == 128 && nh == 2) return launch_fwd_impl<128, 2>(tq, tk, tv, p, grid_x, stream);
  if (D == 128) return launch_fwd_impl<128, 1>(tq, tk, tv, p, grid_x, stream);
  if (D == 256) return launch_fwd_impl<256, 1>(tq, tk, tv, p, grid_x, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ccg
