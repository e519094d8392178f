// attn_bwd.cu -- a6 (dQ pass) and a7 (dK/dV pass) of the CP-emulated causal
// GQA backward on the 5th-generation tensor cores (sm_103a).
//
// TransformerEngine PR "Optimize context parallel attention layouts and
// gradient accumulation", Changes and CP8 first-gradient accumulator reuse:
// dK/dV contributions are accumulated in a fixed order and the first
// contribution is used as the accumulator (no zero-filled buffer, no first
// add into zero).  Here every output tile is owned by exactly one CTA that
// walks its contributions in the canonical ring order, and the first MMA of
// every accumulator runs with accumulation disabled; there are no atomics,
// so results are bitwise repeatable.
//
// dQ pass: one CTA per (128-row query tile, q head).  Q and dO tiles stay in
//   SMEM; K/V tiles stream through the slots.  Per KV tile:
//   S = Q K^T, dP = dO V^T (TMEM), then dS = P (dP - Delta) * scale in
//   registers (P = exp(S*scale - LSE) from the merged LSE), written back to
//   TMEM as BF16, and dQ += dS K (TMEM accumulator).
// dK/dV pass: one CTA per (128-row KV tile, kv head).  K and V stay in SMEM;
//   Q_i / dO_i tiles of every contributing (query chunk, tile, q head)
//   stream through the slots.  Per contribution: S^T = K Q^T, dP^T = V dO^T,
//   P^T and dS^T in registers -> TMEM (BF16), dV += P^T dO, dK += dS^T Q.
// At D = 256 the two 256-column FP32 accumulators alone fill TMEM, so the
// recomputing dK/dV pass runs as two kernels (dV, then dK), and every D = 256
// kernel streams its 128-row tiles as two 128-column halves, so that every
// product runs at full width next to the resident tiles in shared memory.
//
// The backward that keeps dS (a padded-length bound in the descriptor) takes
// one kv head's GQA group at a time: its dQ pass also stores every unit's
// BF16 dS tile (and at D = 256 its P tile) in the workspace, and the dK/dV
// passes read them back instead of recomputing dP^T (and at D = 256 S^T):
// D = 256 one product per unit each for dK and dV, on CTA pairs
// (attn_bwd_dkv_pair_kernel); D = 128 one pass recomputing only P^T
// (attn_bwd_dkdv_ds128_kernel).
#include <cuda_bf16.h>

#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace ccg {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  const WorkItem* items;
  const PlanHeader* hdr;
  const int32_t* cu;
  const int32_t* cu_pad;
  const float* lse;       // merged LSE, natural log, head-grouped [G_h][T][Hq/G_h]
  const float* delta;     // rowsum(O * dO), same layout as lse
  __nv_bfloat16* out0;    // dQ (dQ pass) or dV (dK/dV pass)
  __nv_bfloat16* out1;    // dK (dK/dV pass)
  int32_t* status;
  int cp, hq, hkv, hpg_q, hpg_kv;
  int64_t T;
  float scale, scale_log2;
  // q heads of the dQ pass: head0 .. head0 + nheads - 1 (the grid is items x nheads)
  int head0, nheads;
  // dS backward (ds != null): the dQ pass also writes every unit's dS tile
  // and the dK pass of kv head kv_head reads them.  Tile of (sequence b, q
  // tile (cq, tq), KV tile j of the sequence, q head h of the kv head's
  // group): ds + ((h % G) * ds_cap + ds_base[b] + t^2 cq(cq+1)/2 +
  // tq (cq+1) t + j) * 128 * 128, t = 128-row tiles a chunk.  A tile holds,
  // for each 8-column (16-byte) piece of the KV columns, the piece of all 128
  // query rows: element (q row r, KV column c) at ((c / 8) * 128 + r) * 8 + c % 8.
  // The unit's BF16 P tile follows in the same layout G * ds_cap tiles later,
  // for the dV pass (dV += P^T dO).
  __nv_bfloat16* ds;
  const int64_t* ds_base;
  int64_t ds_cap;
  int kv_head;
};

__device__ __forceinline__ int64_t ds_tile_index(const BwdParams& p, int b, int L, int cq, int tq, int kv_tile,
                                                 int head_in_group) {
  const int64_t t = (L + 127) / 128;
  return head_in_group * p.ds_cap + __ldg(p.ds_base + b) + t * t * cq * (cq + 1) / 2 +
         static_cast<int64_t>(tq) * (cq + 1) * t + kv_tile;
}

// ---------------------------------------------------------------------------
// tile configurations
//
// Both passes keep two S/dP tile buffers in TMEM and run two softmax
// warpgroups: tile (or contribution) j is formed by warpgroup j % 2 in
// buffer j % 2 while the tensor core computes the neighbouring tile, since
// with the final LSE every tile's P is independent of the others.
// warp 0 TMA, 1 MMA, 2 TMEM alloc, 3 idle, 4-11 two softmax warpgroups (the
// D = 128 dQ and dK/dV passes of the dS backward: warps 1-3 issue products)
constexpr int kThreads = 384;

// dQ pass (D = 128).  TMEM: S of tile j in buffer j % 2 at (j % 2) * BN,
// with dS packed over each softmax warpgroup's own S columns; dP at 2 BN,
// released by the softmax as soon as it has loaded dP of tile j; the dQ
// accumulator at 3 BN.  dP of tile j+1 is computed while the softmax forms
// dS of tile j, S of tile j+2 once dQ of tile j has read dS(j).  The slots
// form two rings, NK for K (held from S(j) to dQ(j)) and NV for V (held for
// dP(j) only), so that each ring's slots are released in the order they are
// loaded.  The three products are issued by three warps (1, 2, 3), each
// waiting only for its own inputs: dP(j+1) does not queue behind the wait
// for dS(j), nor S(j+2) behind dP(j+1).
template <int D, int BN_, int NSLOT_>
struct DqCfg {
  static constexpr int BM = 128;                 // query rows (MMA M)
  static constexpr int BN = BN_;                 // key rows per tile (MMA N of S, K of dQ)
  static constexpr int NSLOT = NSLOT_;           // single-tile slots for K_j / V_j
  static constexpr int NV = 2;
  static constexpr int NK = NSLOT - NV;
  static constexpr int RES_BYTES = BM * D * 2;   // Q or dO
  static constexpr int SLOT_BYTES = BN * D * 2;
  static constexpr int SMEM_RES = 0;
  static constexpr int SMEM_SLOT = 2 * RES_BYTES;
  static constexpr int SMEM_BAR = SMEM_SLOT + NSLOT * SLOT_BYTES;
  static constexpr int SMEM_TOTAL = SMEM_BAR + 256;
  static constexpr int T_DP = 2 * BN;
  static constexpr int T_ACC = 3 * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(T_ACC + D <= TMEM_COLS, "TMEM");
  static_assert(BN == 128, "two 32-column chunks of every tile per softmax warpgroup");
  static_assert(NK >= 2, "K ring");
  static_assert(SMEM_TOTAL + 1024 <= 232448, "SMEM");
};

template <int D, int BN_, int NSLOT_, int NBUF_>
struct KvCfg {
  static constexpr int BM = 128;                 // key rows (MMA M)
  static constexpr int BN = BN_;                 // query rows per contribution tile
  static constexpr int NBUF = NBUF_;             // as in DqCfg
  static constexpr bool SPLIT = NBUF == 1;
  static constexpr int NRES = 2;                 // K and V resident
  static constexpr int NSLOT = NSLOT_;
  static constexpr int RES_BYTES = BM * D * 2;
  static constexpr int SLOT_BYTES = BN * D * 2;
  static constexpr int SMEM_RES = 0;
  static constexpr int SMEM_SLOT = NRES * RES_BYTES;
  static constexpr int SMEM_VEC = SMEM_SLOT + NSLOT * SLOT_BYTES;   // [WG][-lse2 BN | -delta*scale BN]
  static constexpr int SMEM_BAR = SMEM_VEC + 2 * 2 * BN * 4;
  static constexpr int SMEM_TOTAL = SMEM_BAR + 256;
  // TMEM: buffer b holds S^T at b*T_BUF and dP^T at b*T_BUF + BN
  static constexpr int T_BUF = 2 * BN;
  static constexpr int T_DV = NBUF * T_BUF;
  static constexpr int T_DK = NBUF * T_BUF + D;
  static constexpr int ACC_END = NBUF * T_BUF + 2 * D;
  // P^T / dS^T (BF16 A operands) are packed in place over S^T / dP^T: over
  // the tile's first BN/2 columns when one warpgroup owns the tile, over the
  // first half of each warpgroup's own columns when the columns are split
  // (a warpgroup never writes columns the other one still reads)
  static constexpr int TMEM_COLS = 512;
  static_assert(ACC_END <= 512, "TMEM");
  static_assert((SPLIT ? BN / 2 : BN) % 32 == 0, "softmax chunking");
  static_assert(SMEM_TOTAL + 1024 <= 232448, "SMEM");
};

// ---------------------------------------------------------------------------
// iteration orders (identical in every role of a CTA)

// KV tiles feeding one query tile's dQ, in ring-step order: steps s ascending,
// the source rank's visible KV chunks ascending, tiles ascending.
template <int BN>
struct DqIter {
  int cp, r, cq, L, S, q_valid_hi;
  int s, nv, vi, vis0, vis1, t, ntile, kv_lo, kv_hi;   // vis0/vis1: no indexed array (stays in registers)
  bool diag, done;

  __device__ void load_vis() {
    nv = visible_kv_chunks2(cq, ring_source(r, s, cp), cp, vis0, vis1);
  }
  __device__ void load_segment() {
    const int j = vi == 0 ? vis0 : vis1;
    diag = (j == cq);
    kv_lo = j * L;
    kv_hi = min((j + 1) * L, S);
    if (diag) kv_hi = min(kv_hi, q_valid_hi);
    ntile = kv_hi > kv_lo ? (kv_hi - kv_lo + BN - 1) / BN : 0;
    t = 0;
  }
  __device__ void settle() {
    // advance to the next non-empty tile from the current (s, vi, t)
    while (!done) {
      if (vi < nv && t < ntile) return;
      if (vi < nv) {
        ++vi;
        if (vi < nv) { load_segment(); continue; }
      }
      ++s;
      if (s >= cp) { done = true; return; }
      load_vis();
      vi = 0;
      if (nv > 0) load_segment();
    }
  }
  __device__ void init(int cp_, int cq_, int L_, int S_, int q_lo, int q_valid_hi_) {
    cp = cp_; cq = cq_; r = chunk_owner(cq_, cp_); L = L_; S = S_; q_valid_hi = q_valid_hi_;
    done = q_valid_hi <= q_lo;       // no real query row in this tile
    s = 0;
    vis0 = vis1 = 0;
    load_vis();
    vi = 0;
    ntile = 0;
    t = 0;
    if (!done && nv > 0) load_segment();
    settle();
  }
  __device__ int k0() const { return kv_lo + t * BN; }
  __device__ void next() { ++t; settle(); }
};

// Contributions feeding one KV tile's dK/dV, in the canonical order: ring
// steps s = 0..CP-1 (rank src+s), query chunk r before 2CP-1-r, query tile
// ascending, q head of the GQA group ascending.
template <int BN>
struct KvIter {
  int cp, C, j, src, L, S, k_lo, G, g;
  int s, which, cq, tq, ntq, h, q_valid_hi;
  bool done;

  __device__ bool load_chunk() {
    // sets up query tiles of chunk cq; false if none contribute
    const int r = (src + s) % cp;
    cq = which == 0 ? r : C - 1 - r;
    if (j > cq) return false;
    const int qa = cq * L;
    q_valid_hi = min((cq + 1) * L, S);
    if (q_valid_hi <= qa) return false;
    ntq = (q_valid_hi - qa + BN - 1) / BN;
    tq = 0;
    if (cq == j) tq = max(0, (k_lo - qa) / BN);   // diagonal: tiles ending before the KV tile see nothing
    h = 0;
    return tq < ntq;
  }
  __device__ void settle_chunk() {
    while (!done) {
      if (load_chunk()) return;
      if (++which == 2) {
        which = 0;
        if (++s >= cp) { done = true; return; }
      }
    }
  }
  __device__ void init(int cp_, int j_, int L_, int S_, int k_lo_, int G_, int g_) {
    cp = cp_; C = 2 * cp_; j = j_; src = chunk_owner(j_, cp_); L = L_; S = S_; k_lo = k_lo_;
    G = G_; g = g_;
    s = 0; which = 0;
    done = k_lo >= S;               // no real key row in this tile
    settle_chunk();
  }
  __device__ int q0() const { return cq * L + tq * BN; }
  __device__ int head() const { return g * G + h; }
  __device__ void next() {
    if (++h < G) return;
    h = 0;
    if (++tq < ntq) return;
    if (++which == 2) {
      which = 0;
      if (++s >= cp) { done = true; return; }
    }
    settle_chunk();
  }
};

struct SeqInfo {
  int start, S, L;
};

__device__ __forceinline__ SeqInfo seq_info(const BwdParams& p, int b) {
  SeqInfo si;
  si.start = __ldg(p.cu_pad + b);
  si.S = __ldg(p.cu + b + 1) - __ldg(p.cu + b);
  si.L = (__ldg(p.cu_pad + b + 1) - si.start) / (2 * p.cp);
  return si;
}

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&r)[32], float mul,
                                               bool zero) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v4 = 0; v4 < 4; ++v4) {
    uint4 u;
    if (zero) {
      u = make_uint4(0, 0, 0, 0);
    } else {
      u.x = pack_bf16x2(__uint_as_float(r[8 * v4 + 0]) * mul, __uint_as_float(r[8 * v4 + 1]) * mul);
      u.y = pack_bf16x2(__uint_as_float(r[8 * v4 + 2]) * mul, __uint_as_float(r[8 * v4 + 3]) * mul);
      u.z = pack_bf16x2(__uint_as_float(r[8 * v4 + 4]) * mul, __uint_as_float(r[8 * v4 + 5]) * mul);
      u.w = pack_bf16x2(__uint_as_float(r[8 * v4 + 6]) * mul, __uint_as_float(r[8 * v4 + 7]) * mul);
    }
    d[v4] = u;
  }
}

// Writes one warp's 32 rows of 128 BF16 columns (four 32-column TMEM chunks
// from t_col on, scaled by `mul`; zeros where `zero`) to global memory
// through a 8 KB staging block in shared memory: each thread converts its own
// row into its 256-byte staging row (16-byte slot k at k ^ (lane & 15), so
// that the warp's accesses hit every bank), then the warp stores whole rows,
// sixteen lanes per row (coalesced).  row_ptr(r) gives the destination of
// the warp's row r, or nullptr for a row the tile does not own.
template <class RowPtr>
__device__ __forceinline__ void store_rows_staged(uint4* stage, uint32_t t_col, bool load, bool zero, float mul,
                                                  int lane, RowPtr row_ptr) {
  uint4* srow = stage + lane * 16;
  const int swz = lane & 15;
  uint32_t r[32];
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    if (load) {                       // warp-uniform
      tmem_ld32(t_col + c * 32, r);
      tmem_wait_ld();
    }
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4) {
      uint4 u = make_uint4(0, 0, 0, 0);
      if (!zero) {
        u.x = pack_bf16x2(__uint_as_float(r[8 * v4 + 0]) * mul, __uint_as_float(r[8 * v4 + 1]) * mul);
        u.y = pack_bf16x2(__uint_as_float(r[8 * v4 + 2]) * mul, __uint_as_float(r[8 * v4 + 3]) * mul);
        u.z = pack_bf16x2(__uint_as_float(r[8 * v4 + 4]) * mul, __uint_as_float(r[8 * v4 + 5]) * mul);
        u.w = pack_bf16x2(__uint_as_float(r[8 * v4 + 6]) * mul, __uint_as_float(r[8 * v4 + 7]) * mul);
      }
      srow[(c * 4 + v4) ^ swz] = u;
    }
  }
  __syncwarp();
  const int u = lane & 15;
#pragma unroll 2
  for (int k = 0; k < 16; ++k) {
    const int rr = 2 * k + (lane >> 4);
    uint4* d = row_ptr(rr);
    if (d != nullptr) d[u] = stage[rr * 16 + (u ^ (rr & 15))];
  }
  __syncwarp();
}

// Issue the K-major (x) K-major product D[tmem] = A[smem tile, M rows] * B[smem tile, N rows]^T
// over a contraction of length KD (both tiles TMA SW128 layout, 64-column chunks);
// a_desc / b_desc are the tiles' base descriptors.
template <int MROWS, int NROWS, int KD>
__device__ __forceinline__ void mma_kk(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(MROWS, NROWS, false, false);
#pragma unroll
  for (int k = 0; k < KD / 16; ++k)
    umma_ss(d_tmem, a_desc + kmajor_step(MROWS, k), b_desc + kmajor_step(NROWS, k), idesc, k > 0 ? 1u : 0u);
}

// As mma_tn, with A packed per warpgroup when the columns are split: the
// first KROWS/2 rows of A at a_tmem, the second half KROWS/2 columns later.
template <int KROWS, int D, bool SPLIT_A>
__device__ __forceinline__ void mma_tn_split(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, false, true);
  constexpr int KPW = SPLIT_A ? KROWS / 32 : KROWS / 16;   // k-steps per packed run
#pragma unroll
  for (int k = 0; k < KROWS / 16; ++k)
    umma_ts(d_tmem, a_tmem + (k / KPW) * (KROWS / 2) + (k % KPW) * 8, b_desc + mnmajor_step(k), idesc,
            (accumulate || k > 0) ? 1u : 0u);
}

// As mma_tn_split, with A packed by NWG warpgroups that split the KROWS
// columns: warpgroup w's KROWS/NWG keys at a_tmem + w * KROWS/NWG, packed.
template <int KROWS, int N, int NWG>
__device__ __forceinline__ void mma_tn_wg(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, N, false, true);
  constexpr int KPW = KROWS / (16 * NWG);          // k-steps per warpgroup's packed run
  static_assert(KPW >= 1, "a warpgroup owns at least one 16-key step");
#pragma unroll
  for (int k = 0; k < KROWS / 16; ++k)
    umma_ts(d_tmem, a_tmem + (k / KPW) * (KROWS / NWG) + (k % KPW) * 8, b_desc + mnmajor_step(k), idesc,
            (accumulate || k > 0) ? 1u : 0u);
}

// D[tmem, M=128 x N=D] (+)= A[tmem bf16, 128 x KROWS] * B[smem tile KROWS rows x D, MN-major];
// b_desc is the base descriptor of B built with LBO = KROWS*128.
template <int KROWS, int D>
__device__ __forceinline__ void mma_tn(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, false, true);
#pragma unroll
  for (int k = 0; k < KROWS / 16; ++k)
    umma_ts(d_tmem, a_tmem + k * 8, b_desc + mnmajor_step(k), idesc, (accumulate || k > 0) ? 1u : 0u);
}

// ---------------------------------------------------------------------------
// dQ pass
template <class Cfg, int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const BwdParams p) {
  constexpr int BM = Cfg::BM, BN = Cfg::BN, NSLOT = Cfg::NSLOT, NK = Cfg::NK, NV = Cfg::NV, KCH = D / 64;
  const int item_idx = blockIdx.x / p.nheads;
  if (item_idx >= p.hdr->n_dq) return;
  if (status_bad(p.status)) return;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // Barriers indexed [2] are per S buffer: phase k of barrier b belongs to
  // tile 2k + b, so that no waiter can see a phase complete twice.
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_BAR);
  uint64_t* res_full = bars;
  uint64_t* full = bars + 1;              // [NSLOT]
  uint64_t* empty = full + NSLOT;         // [NSLOT]
  uint64_t* s_full = empty + NSLOT;       // [2] S(j) complete
  uint64_t* ds_full = s_full + 2;         // [2] dS(j) packed (both warpgroups)
  uint64_t* dq_done = ds_full + 2;        // [2] dQ(j) complete: S buffer j % 2 is free
  uint64_t* dp_full = dq_done + 2;        // dP(j) complete
  uint64_t* dp_free = dp_full + 1;        // the softmax has loaded dP(j)
  uint64_t* acc_done = dp_free + 1;
  uint64_t* drained = acc_done + 1;       // [2] warps 1 and 3: their products are complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drained + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[item_idx];
  const int h = p.head0 + blockIdx.x % p.nheads;   // q head
  const int G = p.hq / p.hkv;
  const int g = h / G;
  const SeqInfo si = seq_info(p, it.b);
  const int q_lo = it.c * si.L + it.tile * BM;                    // first row (sequence position)
  const int q_hi = min(q_lo + BM, (it.c + 1) * si.L);              // rows owned by this tile
  const int q_valid_hi = min(q_hi, si.S);

  if (threadIdx.x == 0) {
    mbar_init(res_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(ds_full + b, 256);
      mbar_init(dq_done + b, 1);
    }
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 256);
    mbar_init(acc_done, 1);
    mbar_init(drained + 0, 1);
    mbar_init(drained + 1, 1);
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
  const int kv_group_row = static_cast<int>((g / p.hpg_kv) * p.T) + si.start;

  if (warp == 0) {
    if (lane == 0) {
      DqIter<BN> itr;
      itr.init(p.cp, it.c, si.L, si.S, q_lo, q_valid_hi);
      int64_t n_loads = 0;                       // copies issued: K_j then V_j per tile
      bool ok = true;
      if (!itr.done) {
        const int row = static_cast<int>((h / p.hpg_q) * p.T) + si.start + q_lo;
        mbar_arrive_expect_tx(res_full, 2 * Cfg::RES_BYTES);
        for (int kc = 0; kc < KCH; ++kc) {
          tma_load_3d(smem + Cfg::SMEM_RES + kc * BM * 128, &tm_q, kc * 64, h % p.hpg_q, row, res_full);
          tma_load_3d(smem + Cfg::SMEM_RES + Cfg::RES_BYTES + kc * BM * 128, &tm_do, kc * 64, h % p.hpg_q, row,
                      res_full);
        }
        // K_j through the K ring (slots 0 .. NK-1), V_j through the V ring
        for (int t = 0; !itr.done && ok; ++t) {
          const bool is_v = (t & 1) == 1;
          const int pos = t >> 1;                                  // tile j = position in its ring
          const int ring = is_v ? NV : NK;
          const int slot = (is_v ? NK : 0) + pos % ring;
          if (pos >= ring) ok = mbar_wait(empty + slot, ((pos / ring) - 1) & 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(full + slot, Cfg::SLOT_BYTES);
          uint8_t* dst = smem + Cfg::SMEM_SLOT + slot * Cfg::SLOT_BYTES;
          for (int kc = 0; kc < KCH; ++kc)
            tma_load_3d(dst + kc * BN * 128, is_v ? &tm_v : &tm_k, kc * 64, g % p.hpg_kv, kv_group_row + itr.k0(),
                        full + slot);
          ++n_loads;
          if (is_v) itr.next();
        }
        if (!ok) {
          raise_status(p.status, CCG_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        volatile int never = 0;
        mbar_wait(res_full, 0, &never, 200000000ull);
        wait_last_copies(full, NK, (n_loads + 1) / 2);
        wait_last_copies(full + NK, NV, n_loads / 2);
      }
    }
  } else if (warp <= 3) {
    // ------------------------------------------------------------ MMA issuers
    // warp 1: S(j) = Q K_j^T into S buffer j % 2, S(j+2) once dQ(j) is done;
    // warp 3: dP(j) = dO V_j^T, dP(j+1) once the softmax has loaded dP(j);
    // warp 2: dQ += dS(j) K_j once dS(j) is packed
    // (each a whole warp, one elected lane issuing)
    {
      DqIter<BN> cnt;
      cnt.init(p.cp, it.c, si.L, si.S, q_lo, q_valid_hi);
      int n = 0;
      for (; !cnt.done; cnt.next()) ++n;
      bool ok = true;
      if (n > 0) {
        const uint32_t q_base = smem_u32(smem + Cfg::SMEM_RES);
        const uint32_t slot_base = smem_u32(smem + Cfg::SMEM_SLOT);
        constexpr uint32_t kSlotStep = Cfg::SLOT_BYTES >> 4;
        if (warp == 2) {
          // slot s: MN-major descriptor of K_j (the B operand of dQ += dS K_j)
          const uint64_t slot_mn0 = smem_desc_sw128(slot_base, BN * 128, 1024);
          for (int j = 0; ok && j < n; ++j) {
            ok = mbar_wait_warp(ds_full + (j & 1), (j >> 1) & 1, abort_flag);
            if (!ok) break;
            // K_j has landed (warp 1 saw it; its slot is released only below)
            const int sk = j % NK;
            ok = mbar_wait_warp(full + sk, (j / NK) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            mma_tn_split<BN, D, true>(tmem + Cfg::T_ACC, tmem + (j & 1) * BN, slot_mn0 + sk * kSlotStep, j > 0);
            umma_commit(empty + sk);                  // K_j done
            umma_commit(dq_done + (j & 1));
          }
        } else {
          ok = mbar_wait_warp(res_full, 0, abort_flag);
          const uint64_t r_desc = smem_desc_sw128(q_base + (warp == 1 ? 0 : Cfg::RES_BYTES), 16, 1024);
          const uint64_t slot_k0 = smem_desc_sw128(slot_base, 16, 1024);
          for (int j = 0; ok && j < n; ++j) {
            int sl;
            uint32_t ph;
            if (warp == 1) {
              if (j >= 2) {
                ok = mbar_wait_warp(dq_done + (j & 1), ((j - 2) >> 1) & 1, abort_flag);
                if (!ok) break;
              }
              sl = j % NK;
              ph = (j / NK) & 1;
            } else {
              if (j >= 1) {
                ok = mbar_wait_warp(dp_free, (j - 1) & 1, abort_flag);
                if (!ok) break;
              }
              sl = NK + j % NV;
              ph = (j / NV) & 1;
            }
            ok = mbar_wait_warp(full + sl, ph, abort_flag);
            if (!ok) break;
            tc_fence_after();
            if (warp == 1) {
              mma_kk<BM, BN, D>(tmem + (j & 1) * BN, r_desc, slot_k0 + sl * kSlotStep);
              umma_commit(s_full + (j & 1));
            } else {
              mma_kk<BM, BN, D>(tmem + Cfg::T_DP, r_desc, slot_k0 + sl * kSlotStep);
              umma_commit(empty + sl);                // V_j done
              umma_commit(dp_full);
            }
          }
        }
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // a commit tracks only its own thread's products: each issuer waits for
      // its own before the CTA may free TMEM (on the normal path the S and dP
      // products are long complete: the softmax of tile n-1 read them)
      uint64_t* own = warp == 2 ? acc_done : drained + (warp == 1 ? 0 : 1);
      umma_commit(own);
      volatile int never = 0;
      mbar_wait(own, 0, &never, 200000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // two warpgroups, each 64 of every tile's 128 columns
    const int wg = (warp - 4) >> 2;
    const int row = ((warp & 3) << 5) + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t0 = tmem + lane_base;
    const int c_first = 2 * wg;                       // its two 32-column chunks
    const int q_pos = q_lo + row;
    const bool row_valid = q_pos < q_valid_hi;
    const int64_t grow = thd_row(si.start + q_pos, h, p.hpg_q, p.T);
    const float lse2 = row_valid ? __ldg(p.lse + grow) * kLog2e : 0.f;
    const float dlt = row_valid ? __ldg(p.delta + grow) : 0.f;
    const uint64_t scale2 = f32x2(p.scale_log2, p.scale_log2), neg_lse2 = f32x2(-lse2, -lse2);
    const uint64_t sc2 = f32x2(p.scale, p.scale), neg_dlt_s = f32x2(-dlt * p.scale, -dlt * p.scale);
    DqIter<BN> itr;
    itr.init(p.cp, it.c, si.L, si.S, q_lo, q_valid_hi);
    const bool any = !itr.done;
    bool ok = true;
    for (int j = 0; !itr.done; ++j, itr.next()) {
      const uint32_t ts = t0 + (j & 1) * BN;
      const uint32_t tdp = t0 + Cfg::T_DP;
      ok = __all_sync(0xffffffffu, mbar_wait(s_full + (j & 1), (j >> 1) & 1, abort_flag) &&
                                       mbar_wait(dp_full, j & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int k0 = itr.k0();
      const int kend = itr.diag ? min(itr.kv_hi, q_pos + 1) : itr.kv_hi;
      const int nvalid = row_valid ? kend - k0 : 0;
      // dS backward: this unit's dS tile (the dK/dV pass reads it back)
      uint4* ds_tile = nullptr;
      if (p.ds != nullptr) {
        const int tpc = (si.L + 127) / 128;
        const int kv_tile = (k0 / si.L) * tpc + (k0 % si.L) / 128;
        ds_tile = reinterpret_cast<uint4*>(p.ds) + ds_tile_index(p, it.b, si.L, it.c, it.tile, kv_tile, h % G) * (128 * 128 / 8);
      }
      // hidden keys only on tiles that cross a row's last visible key: their
      // scores become -inf in registers, so P (and dS) come out exactly 0
      const bool masked = __any_sync(0xffffffffu, nvalid < BN);
      // dP of both chunks (and S of the first) first, then release the dP
      // buffer for the next tile's dP product
      uint32_t rs[32], rp[32], rp2[32];
      tmem_ld32(tdp + c_first * 32, rp);
      tmem_ld32(tdp + (c_first + 1) * 32, rp2);
      tmem_ld32(ts + c_first * 32, rs);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(dp_free);
#pragma unroll
      for (int c = c_first; c < c_first + 2; ++c) {
        if (c != c_first) {
          tmem_ld32(ts + c * 32, rs);
#pragma unroll
          for (int x = 0; x < 32; ++x) rp[x] = rp2[x];
          tmem_wait_ld();
        }
        if (masked) {
#pragma unroll
          for (int x = 0; x < 32; ++x) rs[x] = (c * 32 + x < nvalid) ? rs[x] : 0xff800000u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          // P = 2^(s * scale_log2 - lse2); dS = P * (dP * scale - Delta * scale)
          float a0, a1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(rs[2 * x]), __uint_as_float(rs[2 * x + 1])), scale2, neg_lse2),
                      a0, a1);
          const uint64_t pv = f32x2(ex2_approx(a0), ex2_approx(a1));
          const uint64_t t =
              fma_f32x2(f32x2(__uint_as_float(rp[2 * x]), __uint_as_float(rp[2 * x + 1])), sc2, neg_dlt_s);
          float d0, d1;
          f32x2_split(mul_f32x2(pv, t), d0, d1);
          pk[x] = pack_bf16x2(d0, d1);
        }
        tmem_st16(ts + c_first * 32 + (c - c_first) * 16, pk);     // over the warpgroup's own S columns
        if (ds_tile != nullptr) {
          // 16-byte pieces 4c .. 4c+3 of this row: a warp's store covers 32
          // consecutive rows of one piece (512 bytes)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            ds_tile[(4 * c + i) * 128 + row] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_full + (j & 1));
    }
    if (ok && any) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag));
    if (!ok) {
      raise_status(p.status, CCG_ERR_TIMEOUT);
      *abort_flag = 1;
    } else {
      // each warpgroup writes half of the columns of the tile's rows in this
      // chunk: real rows get dQ, padding rows 0
      tc_fence_after();
      const bool own = q_pos < q_hi;
      __nv_bfloat16* dst = p.out0 + grow * D;
      uint32_t r[32];
#pragma unroll 1
      for (int c = wg * (D / 64); c < (wg + 1) * (D / 64); ++c) {
        if (any) {                        // CTA-uniform: every lane loads
          tmem_ld32(t0 + Cfg::T_ACC + c * 32, r);
          tmem_wait_ld();
        }
        if (own) store_row_bf16(dst + c * 32, r, 1.f, !any || !row_valid);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// dK/dV pass
template <class Cfg, int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const BwdParams p) {
  constexpr int BM = Cfg::BM, BN = Cfg::BN, NSLOT = Cfg::NSLOT, KCH = D / 64;
  const int item_idx = blockIdx.x;            // items carry their kv head
  if (item_idx >= p.hdr->n_kv) return;
  if (status_bad(p.status)) return;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_BAR);
  uint64_t* res_full = bars;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + NSLOT;
  uint64_t* s_full = empty + NSLOT;       // [2]
  uint64_t* p_full = s_full + 2;          // [2]
  uint64_t* acc_done = p_full + 2;
  uint64_t* vec_ready = acc_done + 1;     // [2 WG]: LSE/Delta of the next contribution staged
  uint64_t* vec_free = vec_ready + 2;     // [2 WG]: every thread finished reading them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(vec_free + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* vec = reinterpret_cast<float*>(smem + Cfg::SMEM_VEC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[item_idx];
  const int g = it.step;                      // kv head of the item
  const int G = p.hq / p.hkv;
  const SeqInfo si = seq_info(p, it.b);
  const int k_lo = it.c * si.L + it.tile * BM;
  const int k_hi = min(k_lo + BM, (it.c + 1) * si.L);
  const int k_valid_hi = min(k_hi, si.S);

  if (threadIdx.x == 0) {
    mbar_init(res_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, Cfg::SPLIT ? 256 : 128);
    }
    mbar_init(acc_done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(vec_ready + b, 128);
      mbar_init(vec_free + b, 128);
    }
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

  // streamed tiles per contribution: dO_i, then Q_i

  if (warp == 0) {
    if (lane == 0) {
      KvIter<BN> itr;
      itr.init(p.cp, it.c, si.L, si.S, k_lo, G, g);
      int64_t n_loads = 0;                       // copies issued (slot = position % NSLOT)
      bool ok = true;
      if (!itr.done) {
        const int krow = static_cast<int>((g / p.hpg_kv) * p.T) + si.start + k_lo;
        mbar_arrive_expect_tx(res_full, Cfg::NRES * Cfg::RES_BYTES);
        for (int kc = 0; kc < KCH; ++kc) {
          tma_load_3d(smem + Cfg::SMEM_RES + kc * BM * 128, &tm_k, kc * 64, g % p.hpg_kv, krow, res_full);
          tma_load_3d(smem + Cfg::SMEM_RES + Cfg::RES_BYTES + kc * BM * 128, &tm_v, kc * 64, g % p.hpg_kv,
                      krow, res_full);
        }
        for (int t = 0; !itr.done && ok; ++t) {
          const int slot = t % NSLOT;
          if (t >= NSLOT) ok = mbar_wait(empty + slot, ((t / NSLOT) - 1) & 1, abort_flag);
          if (!ok) break;
          const bool first = (t & 1) == 0;
          const bool is_q = !first;
          const int hq = itr.head();
          const int qrow = static_cast<int>((hq / p.hpg_q) * p.T) + si.start + itr.q0();
          mbar_arrive_expect_tx(full + slot, Cfg::SLOT_BYTES);
          uint8_t* dst = smem + Cfg::SMEM_SLOT + slot * Cfg::SLOT_BYTES;
          for (int kc = 0; kc < KCH; ++kc)
            tma_load_3d(dst + kc * BN * 128, is_q ? &tm_q : &tm_do, kc * 64, hq % p.hpg_q, qrow, full + slot);
          ++n_loads;
          if (!first) itr.next();
        }
        if (!ok) {
          raise_status(p.status, CCG_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        volatile int never = 0;
        mbar_wait(res_full, 0, &never, 200000000ull);
        wait_last_copies(full, NSLOT, n_loads);
      }
    }
  } else if (warp == 1) {
    {   // the whole warp; one elected lane issues
      KvIter<BN> ahead;
      ahead.init(p.cp, it.c, si.L, si.S, k_lo, G, g);
      bool ok = true;
      if (!ahead.done) {
        const uint32_t k_base = smem_u32(smem + Cfg::SMEM_RES);
        const uint64_t k_desc = smem_desc_sw128(k_base, 16, 1024);
        const uint64_t v_desc = smem_desc_sw128(k_base + Cfg::RES_BYTES, 16, 1024);
        const uint32_t slot_base = smem_u32(smem + Cfg::SMEM_SLOT);
        const uint64_t slot_k0 = smem_desc_sw128(slot_base, 16, 1024);
        const uint64_t slot_mn0 = smem_desc_sw128(slot_base, BN * 128, 1024);
        constexpr uint32_t kSlotStep = Cfg::SLOT_BYTES >> 4;
        auto slot_k = [&](int s2) { return slot_k0 + s2 * kSlotStep; };
        auto slot_mn = [&](int s2) { return slot_mn0 + s2 * kSlotStep; };
        ok = mbar_wait_warp(res_full, 0, abort_flag);
        tc_fence_after();
        auto slot_q = [&](int j) { return 2 * j + 1; };
        auto slot_do = [&](int j) { return 2 * j; };
        // S^T (and dP^T) of contribution j into buffer j % 2
        auto issue_sp = [&](int j) -> bool {
          const int tq = slot_q(j), tdo = slot_do(j);
          const int sq = tq % NSLOT, sdo = tdo % NSLOT;
          const int b = j % Cfg::NBUF;
          const uint32_t buf = tmem + b * Cfg::T_BUF;
          // dP^T first (dO_i arrives first)
          if (!mbar_wait_warp(full + sdo, (tdo / NSLOT) & 1, abort_flag)) return false;
          tc_fence_after();
          mma_kk<BM, BN, D>(buf + BN, v_desc, slot_k(sdo));
          if (!mbar_wait_warp(full + sq, (tq / NSLOT) & 1, abort_flag)) return false;
          tc_fence_after();
          mma_kk<BM, BN, D>(buf, k_desc, slot_k(sq));
          umma_commit(s_full + b);
          return true;
        };
        int j_sp = 0;
        while (ok && !ahead.done && j_sp < Cfg::NBUF) {
          ok = issue_sp(j_sp++);
          ahead.next();
        }
        for (int j = 0; ok && j < j_sp; ++j) {
          const int tq = slot_q(j), tdo = slot_do(j);
          const int sq = tq % NSLOT, sdo = tdo % NSLOT;
          const int b = j % Cfg::NBUF;
          const uint32_t buf = tmem + b * Cfg::T_BUF;
          ok = mbar_wait_warp(p_full + b, (j / Cfg::NBUF) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          mma_tn_split<BN, D, Cfg::SPLIT>(tmem + Cfg::T_DV, buf, slot_mn(sdo), j > 0);
          mma_tn_split<BN, D, Cfg::SPLIT>(tmem + Cfg::T_DK, buf + BN, slot_mn(sq), j > 0);
          umma_commit(empty + sdo);
          umma_commit(empty + sq);
          if (!ahead.done) {
            ok = issue_sp(j_sp++);
            ahead.next();
          }
        }
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(acc_done);
      volatile int never = 0;
      mbar_wait(acc_done, 0, &never, 200000000ull);
    }
  } else if (warp >= 4) {
    const int wg = (warp - 4) >> 2;   // contributions j % 2 == wg, or half the columns (SPLIT)
    const int row = ((warp & 3) << 5) + lane;        // key row of the tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t0 = tmem + lane_base;
    constexpr int NC = Cfg::SPLIT ? BN / 64 : BN / 32;
    const int c_first = Cfg::SPLIT ? wg * NC : 0;
    constexpr int VEC_N = Cfg::SPLIT ? BN / 2 : BN;  // query rows whose LSE/Delta this warpgroup stages
    const int k_pos = k_lo + row;
    const bool k_valid = k_pos < k_valid_hi;
    KvIter<BN> itr;
    itr.init(p.cp, it.c, si.L, si.S, k_lo, G, g);
    const bool any = !itr.done;
    bool ok = true;
    int k = 0;                                       // this warpgroup's contribution count
    for (int j = 0; !itr.done; ++j, itr.next()) {
      if (!Cfg::SPLIT && (j & 1) != wg) continue;
      const int b = j % Cfg::NBUF;
      const uint32_t tb = t0 + b * Cfg::T_BUF;
      // LSE (log2 units) and Delta of this contribution's query rows -> SMEM
      float* vb = vec + wg * 2 * BN;
      if (k > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(vec_free + wg, (k - 1) & 1, abort_flag));
        if (!ok) break;
      }
      if (row < VEC_N) {
        const int col = c_first * 32 + row;
        const int qp = itr.q0() + col;
        const bool qv = qp < itr.q_valid_hi;
        const int64_t gr = thd_row(si.start + qp, itr.head(), p.hpg_q, p.T);
        vb[col] = qv ? -__ldg(p.lse + gr) * kLog2e : 0.f;                 // -LSE in log2 units
        vb[BN + col] = qv ? -__ldg(p.delta + gr) * p.scale : 0.f;  // -Delta * scale
      }
      mbar_arrive(vec_ready + wg);
      ok = __all_sync(0xffffffffu, mbar_wait(vec_ready + wg, k & 1, abort_flag));
      if (!ok) break;
      ++k;
      ok = __all_sync(0xffffffffu, mbar_wait(s_full + b, (j / Cfg::NBUF) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int q0 = itr.q0();
      // query column c is visible to this key row iff q0+c >= k_pos and q0+c < q_valid_hi
      const int c_lo = k_valid ? max(0, k_pos - q0) : BN;
      const int c_hi = k_valid ? itr.q_valid_hi - q0 : 0;
      // only contributions that cross the causal diagonal or a ragged end
      // need a mask: hidden scores become -inf, so P and dS come out 0
      const bool masked = __any_sync(0xffffffffu, c_lo > 0 || c_hi < BN);
      const uint64_t scale2 = f32x2(p.scale_log2, p.scale_log2), sc2 = f32x2(p.scale, p.scale);
      uint32_t rs[32], rp[32];
#pragma unroll
      for (int c = c_first; c < c_first + NC; ++c) {
        tmem_ld32(tb + c * 32, rs);
        tmem_ld32(tb + BN + c * 32, rp);
        tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int col = c * 32 + x;
            rs[x] = (col >= c_lo && col < c_hi) ? rs[x] : 0xff800000u;
          }
        }
        // the columns' -LSE2 and -Delta*scale, four columns per 16-byte load
        const ulonglong2* nl4 = reinterpret_cast<const ulonglong2*>(vb + c * 32);
        const ulonglong2* nd4 = reinterpret_cast<const ulonglong2*>(vb + BN + c * 32);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int x2 = 0; x2 < 8; ++x2) {
          const ulonglong2 lv = nl4[x2], dv = nd4[x2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int x = 2 * x2 + e;
            // P = 2^(s * scale_log2 - lse2); dS = P * (dP * scale - Delta * scale)
            float a0, a1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(rs[2 * x]), __uint_as_float(rs[2 * x + 1])), scale2,
                                  e ? lv.y : lv.x),
                        a0, a1);
            const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            pk[x] = pack_bf16x2(p0, p1);
            const uint64_t t = fma_f32x2(f32x2(__uint_as_float(rp[2 * x]), __uint_as_float(rp[2 * x + 1])), sc2,
                                         e ? dv.y : dv.x);
            float d0, d1;
            f32x2_split(mul_f32x2(f32x2(p0, p1), t), d0, d1);
            dk[x] = pack_bf16x2(d0, d1);
          }
        }
        const int packed = c_first * 32 + (c - c_first) * 16;   // in place, own columns
        tmem_st16(tb + packed, pk);
        tmem_st16(tb + BN + packed, dk);
      }
      mbar_arrive(vec_free + wg);          // done reading this contribution's LSE/Delta
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full + b);
    }
    if (ok && any) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag));
    if (!ok) {
      raise_status(p.status, CCG_ERR_TIMEOUT);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      const bool own = k_pos < k_hi;     // rows of this tile inside the chunk
      const int64_t grow = thd_row(si.start + k_pos, g, p.hpg_kv, p.T);
      uint32_t r[32];
      // warpgroup 0 writes dV, warpgroup 1 dK
      const bool write_dv = wg == 0;
      const bool write_dk = wg == 1;
      const int c_begin = 0;
      const int c_end = D / 32;
      if (write_dv) {
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
          if (any) {
            tmem_ld32(t0 + Cfg::T_DV + c * 32, r);
            tmem_wait_ld();
          }
          if (own) store_row_bf16(p.out0 + grow * D + c * 32, r, 1.f, !any || !k_valid);
        }
      }
      if (write_dk) {
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
          if (any) {
            tmem_ld32(t0 + Cfg::T_DK + c * 32, r);
            tmem_wait_ld();
          }
          if (own) store_row_bf16(p.out1 + grow * D + c * 32, r, 1.f, !any || !k_valid);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// D = 256 dQ pass and dK pass with full-width products.
//
// At D = 256 the two resident 128-row tiles (Q and dO, or K and V) take 128 KB
// of shared memory, which leaves no room for a whole streamed 128-row tile
// (64 KB) next to a second one.  Here every streamed tile is loaded as its
// two 128-column halves (32 KB each) through three half-tile slots, so that
// the products of S (S^T), dP (dP^T) and the gradient all run at N = 128 or
// wider (full tensor-core rate) instead of N = 64:
//   S  = sum_h R0[:, h] Y_h^T,  dP = sum_h R1[:, h] X_h^T   (K = 128 per half)
//   G[:, h] += dS Y_h                                         (N = 128 per half)
// with, for the dQ role, R0 = Q, R1 = dO, X = V_j, Y = K_j, G = dQ (one CTA per
// 128-row query tile and q head, KV tiles in ring-step order), and for the dK
// role R0 = K, R1 = V, X = dO_i, Y = Q_i, G = dK (one CTA per 128-row KV tile
// and kv head, contributions in the canonical order, the first MMA of the
// accumulator without accumulation).  TMEM: S at columns [0,128), dP at
// [128,256), G at [256,512); the two softmax warpgroups split the 128 columns
// of every unit and pack their BF16 dS over the first half of their own dP
// columns (the A operand of the gradient product).  Half-tiles stream in the
// order X0 X1 Y0 Y1 per unit; X_h is released after its dP product, Y_h after
// its gradient product.
enum class HalfRole { kDq = 0, kDk = 1 };

template <int NWG_>
struct HalfCfg {
  static constexpr int NWG = NWG_;               // softmax warpgroups (they split every unit's columns)
  static constexpr int THREADS = 128 + 128 * NWG;
  static constexpr int D = 256;
  static constexpr int BM = 128;                 // stationary rows (MMA M)
  static constexpr int BN = 128;                 // streamed rows per unit
  static constexpr int DH = 128;                 // columns of a half-tile
  static constexpr int NSLOT = 3;
  static constexpr int RES_BYTES = BM * D * 2;   // 64 KB
  static constexpr int HALF_BYTES = BN * DH * 2; // 32 KB
  static constexpr int SMEM_SLOT = 2 * RES_BYTES;
  static constexpr int WCOLS = BN / NWG;         // columns of a unit per warpgroup
  static constexpr int SMEM_BAR = SMEM_SLOT + NSLOT * HALF_BYTES;
  static constexpr int SMEM_TOTAL = SMEM_BAR + 256;
  static constexpr int T_S = 0, T_P = BN, T_ACC = 2 * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(T_ACC + D <= TMEM_COLS, "TMEM");
  static_assert(SMEM_TOTAL + 1024 <= 232448, "SMEM");
  static_assert(WCOLS == 64, "a lane holds two of its warpgroup's columns (dK role)");
};

// D[tmem] (+)= A[smem, 128 rows, K-major] * B[smem, 128 rows, K-major]^T over
// one 128-column half (8 K steps); a_desc already points at the half.
__device__ __forceinline__ void mma_kk_half(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    umma_ss(d_tmem, a_desc + kmajor_step(128, k), b_desc + kmajor_step(128, k), idesc,
            (accumulate || k > 0) ? 1u : 0u);
}

template <HalfRole ROLE, int NWG>
__global__ void __launch_bounds__(HalfCfg<NWG>::THREADS, 1)
attn_bwd_half_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
  using Cfg = HalfCfg<NWG>;
  constexpr bool DQ = ROLE == HalfRole::kDq;
  constexpr int BM = Cfg::BM, BN = Cfg::BN, NSLOT = Cfg::NSLOT, D = Cfg::D;
  using Iter = typename std::conditional<DQ, DqIter<BN>, KvIter<BN>>::type;
  // dQ role: one CTA per (item, q head); dK role: the items carry their kv head
  const int item_idx = DQ ? blockIdx.x / p.nheads : blockIdx.x;
  if (item_idx >= (DQ ? p.hdr->n_dq : p.hdr->n_kv)) return;
  if (status_bad(p.status)) return;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_BAR);
  uint64_t* res_full = bars;
  uint64_t* full = bars + 1;              // [NSLOT]
  uint64_t* empty = full + NSLOT;         // [NSLOT]
  uint64_t* s_full = empty + NSLOT;       // S and dP of the unit complete
  uint64_t* ds_full = s_full + 1;         // dS of the unit packed (every warpgroup)
  uint64_t* acc_done = ds_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[item_idx];
  const int head = DQ ? p.head0 + blockIdx.x % p.nheads : it.step;   // q head (dQ role) or kv head (dK role)
  const int G = p.hq / p.hkv;
  const int g = DQ ? head / G : head;          // kv head
  const SeqInfo si = seq_info(p, it.b);
  const int r_lo = it.c * si.L + it.tile * BM;               // first stationary row (sequence position)
  const int r_hi = min(r_lo + BM, (it.c + 1) * si.L);        // rows owned by this tile
  const int r_valid_hi = min(r_hi, si.S);

  auto iter_init = [&](Iter& itr) {
    if constexpr (DQ) itr.init(p.cp, it.c, si.L, si.S, r_lo, r_valid_hi);
    else itr.init(p.cp, it.c, si.L, si.S, r_lo, G, g);
  };

  if (threadIdx.x == 0) {
    mbar_init(res_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(ds_full, 128 * NWG);
    mbar_init(acc_done, 1);
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
  const int kv_group_row = static_cast<int>((g / p.hpg_kv) * p.T) + si.start;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Iter itr;
      iter_init(itr);
      int64_t n_loads = 0;                       // copies issued (slot = position % NSLOT)
      bool ok = true;
      if (!itr.done) {
        // resident tiles: Q and dO of (tile, q head), or K and V of (tile, kv head)
        const CUtensorMap* r0 = DQ ? &tm_q : &tm_k;
        const CUtensorMap* r1 = DQ ? &tm_do : &tm_v;
        const int rhead = DQ ? head % p.hpg_q : g % p.hpg_kv;
        const int rrow = DQ ? static_cast<int>((head / p.hpg_q) * p.T) + si.start + r_lo : kv_group_row + r_lo;
        mbar_arrive_expect_tx(res_full, 2 * Cfg::RES_BYTES);
        for (int kc = 0; kc < D / 64; ++kc) {
          tma_load_3d(smem + kc * BM * 128, r0, kc * 64, rhead, rrow, res_full);
          tma_load_3d(smem + Cfg::RES_BYTES + kc * BM * 128, r1, kc * 64, rhead, rrow, res_full);
        }
        // half-tiles X0 X1 Y0 Y1 of every unit, in the order the MMA warp uses them
        for (int t = 0; !itr.done && ok; ++t) {
          const int slot = t % NSLOT;
          if (t >= NSLOT) ok = mbar_wait(empty + slot, ((t / NSLOT) - 1) & 1, abort_flag);
          if (!ok) break;
          const int part = t & 3, half = part & 1;
          const bool is_x = part < 2;
          const CUtensorMap* map;
          int hc, row;
          if constexpr (DQ) {
            map = is_x ? &tm_v : &tm_k;
            hc = g % p.hpg_kv;
            row = kv_group_row + itr.k0();
          } else {
            const int hq = itr.head();
            map = is_x ? &tm_do : &tm_q;
            hc = hq % p.hpg_q;
            row = static_cast<int>((hq / p.hpg_q) * p.T) + si.start + itr.q0();
          }
          mbar_arrive_expect_tx(full + slot, Cfg::HALF_BYTES);
          uint8_t* dst = smem + Cfg::SMEM_SLOT + slot * Cfg::HALF_BYTES;
          for (int kc = 0; kc < 2; ++kc)
            tma_load_3d(dst + kc * BN * 128, map, (2 * half + kc) * 64, hc, row, full + slot);
          ++n_loads;
          if (part == 3) itr.next();
        }
        if (!ok) {
          raise_status(p.status, CCG_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        volatile int never = 0;
        mbar_wait(res_full, 0, &never, 200000000ull);
        wait_last_copies(full, NSLOT, n_loads);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    {   // the whole warp; one elected lane issues
      Iter ahead;
      iter_init(ahead);
      bool ok = true;
      if (!ahead.done) {
        const uint32_t base = smem_u32(smem);
        const uint64_t r0_desc = smem_desc_sw128(base, 16, 1024);
        const uint64_t r1_desc = smem_desc_sw128(base + Cfg::RES_BYTES, 16, 1024);
        const uint32_t slot_base = smem_u32(smem + Cfg::SMEM_SLOT);
        const uint64_t slot_k0 = smem_desc_sw128(slot_base, 16, 1024);
        const uint64_t slot_mn0 = smem_desc_sw128(slot_base, BN * 128, 1024);
        constexpr uint32_t kSlotStep = Cfg::HALF_BYTES >> 4;
        auto slot_k = [&](int s2) { return slot_k0 + s2 * kSlotStep; };
        auto slot_mn = [&](int s2) { return slot_mn0 + s2 * kSlotStep; };
        ok = mbar_wait_warp(res_full, 0, abort_flag);
        tc_fence_after();
        // dP (from X0, X1) then S (from Y0, Y1) of unit j
        auto issue_sp = [&](int j) -> bool {
          for (int h = 0; h < 2; ++h) {
            const int t = 4 * j + h, sl = t % NSLOT;
            if (!mbar_wait_warp(full + sl, (t / NSLOT) & 1, abort_flag)) return false;
            tc_fence_after();
            mma_kk_half(tmem + Cfg::T_P, r1_desc + kmajor_step(128, 8 * h), slot_k(sl), h > 0);
            umma_commit(empty + sl);                  // X_h done
          }
          for (int h = 0; h < 2; ++h) {
            const int t = 4 * j + 2 + h, sl = t % NSLOT;
            if (!mbar_wait_warp(full + sl, (t / NSLOT) & 1, abort_flag)) return false;
            tc_fence_after();
            mma_kk_half(tmem + Cfg::T_S, r0_desc + kmajor_step(128, 8 * h), slot_k(sl), h > 0);
          }
          umma_commit(s_full);
          return true;
        };
        int j_sp = 0;
        if (ok) {
          ok = issue_sp(j_sp++);
          ahead.next();
        }
        for (int j = 0; ok && j < j_sp; ++j) {
          ok = mbar_wait_warp(ds_full, j & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          for (int h = 0; h < 2; ++h) {
            const int sl = (4 * j + 2 + h) % NSLOT;
            mma_tn_wg<BN, Cfg::DH, NWG>(tmem + Cfg::T_ACC + h * Cfg::DH, tmem + Cfg::T_P, slot_mn(sl), j > 0);
            umma_commit(empty + sl);                  // Y_h done
          }
          if (!ahead.done) {
            ok = issue_sp(j_sp++);
            ahead.next();
          }
        }
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(acc_done);
      volatile int never = 0;
      mbar_wait(acc_done, 0, &never, 200000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int wg = (warp - 4) >> 2;                  // the warpgroup's share of every unit's columns
    const int row = ((warp & 3) << 5) + lane;        // stationary row of the tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t0 = tmem + lane_base;
    constexpr int NC = Cfg::WCOLS / 32;               // 32-column chunks per warpgroup
    const int c_first = wg * NC;
    const int r_pos = r_lo + row;
    const bool r_valid = r_pos < r_valid_hi;
    const int64_t grow = DQ ? thd_row(si.start + r_pos, head, p.hpg_q, p.T)
                            : thd_row(si.start + r_pos, g, p.hpg_kv, p.T);
    // dQ role: this row's LSE (log2 units) and Delta
    float lse2 = 0.f, dlt = 0.f;
    if (DQ && r_valid) {
      lse2 = __ldg(p.lse + grow) * kLog2e;
      dlt = __ldg(p.delta + grow);
    }
    const uint64_t scale2 = f32x2(p.scale_log2, p.scale_log2), sc2 = f32x2(p.scale, p.scale);
    const uint64_t row_nl2 = f32x2(-lse2, -lse2), row_nds = f32x2(-dlt * p.scale, -dlt * p.scale);
    Iter itr;
    iter_init(itr);
    const bool any = !itr.done;
    bool ok = true;
    uint64_t col_l = 0, col_d = 0;
    for (int j = 0; !itr.done; ++j, itr.next()) {
      int c_lo = 0, c_hi = BN;                        // visible streamed columns of this row
      uint4* ds_tile = nullptr;                      // dS backward: this unit's dS tile
      auto store_ds_p = [&](uint4* tile, int c, const uint32_t (&dsv)[16], const uint32_t (&pv)[16]) {
        uint4* p_tile = tile + static_cast<int64_t>(G) * p.ds_cap * (128 * 128 / 8);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tile[(4 * c + i) * 128 + row] = make_uint4(dsv[4 * i], dsv[4 * i + 1], dsv[4 * i + 2], dsv[4 * i + 3]);
          p_tile[(4 * c + i) * 128 + row] = make_uint4(pv[4 * i], pv[4 * i + 1], pv[4 * i + 2], pv[4 * i + 3]);
        }
      };
      if constexpr (DQ) {
        const int k0 = itr.k0();
        const int kend = itr.diag ? min(itr.kv_hi, r_pos + 1) : itr.kv_hi;
        c_hi = r_valid ? kend - k0 : 0;
        if (p.ds != nullptr) {
          const int tpc = (si.L + 127) / 128;
          const int kv_tile = (k0 / si.L) * tpc + (k0 % si.L) / 128;
          ds_tile = reinterpret_cast<uint4*>(p.ds) +
                    ds_tile_index(p, it.b, si.L, it.c, it.tile, kv_tile, head % G) * (128 * 128 / 8);
        }
      } else {
        // -LSE (log2 units) and -Delta * scale of this contribution's query
        // columns: every lane holds two of its warpgroup's 64 columns (2*lane
        // and 2*lane + 1) and hands them to the other lanes by shuffles, so
        // that the softmax reads no shared memory (which the products keep busy)
        {
          const int qp0 = itr.q0() + c_first * 32 + 2 * lane;
          float l0 = 0.f, l1 = 0.f, e0 = 0.f, e1 = 0.f;
          if (qp0 < itr.q_valid_hi) {
            const int64_t gr = thd_row(si.start + qp0, itr.head(), p.hpg_q, p.T);
            l0 = -__ldg(p.lse + gr) * kLog2e;
            e0 = -__ldg(p.delta + gr) * p.scale;
          }
          if (qp0 + 1 < itr.q_valid_hi) {
            const int64_t gr = thd_row(si.start + qp0 + 1, itr.head(), p.hpg_q, p.T);
            l1 = -__ldg(p.lse + gr) * kLog2e;
            e1 = -__ldg(p.delta + gr) * p.scale;
          }
          col_l = f32x2(l0, l1);
          col_d = f32x2(e0, e1);
        }
        const int q0 = itr.q0();
        // query column c is visible to this key row iff q0+c >= r_pos and q0+c < q_valid_hi
        c_lo = r_valid ? max(0, r_pos - q0) : BN;
        c_hi = r_valid ? itr.q_valid_hi - q0 : 0;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, j & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      // hidden columns only on units that cross the causal diagonal or a
      // ragged end: their scores become -inf, so P and dS come out 0
      const bool masked = __any_sync(0xffffffffu, c_lo > 0 || c_hi < BN);
      uint32_t rs[32], rp[32];
#pragma unroll
      for (int c = c_first; c < c_first + NC; ++c) {
        tmem_ld32(t0 + Cfg::T_S + c * 32, rs);
        tmem_ld32(t0 + Cfg::T_P + c * 32, rp);
        tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int col = c * 32 + x;
            rs[x] = (col >= c_lo && col < c_hi) ? rs[x] : 0xff800000u;
          }
        }
        // dK role: the columns' -LSE2 and -Delta*scale, from the lanes that hold them
        uint32_t pk[16];
        uint32_t pp[16];                             // dQ role, dS backward: BF16 P
#pragma unroll
        for (int x2 = 0; x2 < 8; ++x2) {
          ulonglong2 lv, dv;
          if constexpr (DQ) {
            lv = make_ulonglong2(row_nl2, row_nl2);
            dv = make_ulonglong2(row_nds, row_nds);
          } else {
            const int src = (c - c_first) * 16 + 2 * x2;
            lv.x = __shfl_sync(0xffffffffu, col_l, src);
            lv.y = __shfl_sync(0xffffffffu, col_l, src + 1);
            dv.x = __shfl_sync(0xffffffffu, col_d, src);
            dv.y = __shfl_sync(0xffffffffu, col_d, src + 1);
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int x = 2 * x2 + e;
            // P = 2^(s * scale_log2 - lse2); dS = P * (dP * scale - Delta * scale)
            float a0, a1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(rs[2 * x]), __uint_as_float(rs[2 * x + 1])), scale2,
                                  e ? lv.y : lv.x),
                        a0, a1);
            const uint64_t pv = f32x2(ex2_approx(a0), ex2_approx(a1));
            const uint64_t t = fma_f32x2(f32x2(__uint_as_float(rp[2 * x]), __uint_as_float(rp[2 * x + 1])), sc2,
                                         e ? dv.y : dv.x);
            float d0, d1;
            f32x2_split(mul_f32x2(pv, t), d0, d1);
            pk[x] = pack_bf16x2(d0, d1);
            if constexpr (DQ) {
              float q0, q1;
              f32x2_split(pv, q0, q1);
              pp[x] = pack_bf16x2(q0, q1);
            }
          }
        }
        tmem_st16(t0 + Cfg::T_P + c_first * 32 + (c - c_first) * 16, pk);   // in place, own columns
        if constexpr (DQ) {
          // 16-byte pieces 4c .. 4c+3 (8 columns each) of this row, of dS and
          // of P: a warp's store covers 32 consecutive rows of one piece (512
          // bytes).  The last chunk's go out after the hand-over below, while
          // the gradient product runs.
          if (ds_tile != nullptr) {
            store_ds_p(ds_tile, c, pk, pp);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    if (ok && any) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag));
    if (!ok) {
      raise_status(p.status, CCG_ERR_TIMEOUT);
      *abort_flag = 1;
    } else {
      // each warpgroup writes its share of the columns of the tile's rows
      // (real rows get the gradient, padding rows 0), through a staging
      // block in the slot area, idle now that every product is done
      tc_fence_after();
      static_assert(D / NWG == 128, "a warpgroup writes 128 columns");
      __nv_bfloat16* outp = (DQ ? p.out0 : p.out1) + wg * (D / NWG);
      uint4* stage = reinterpret_cast<uint4*>(smem + Cfg::SMEM_SLOT) + (warp - 4) * 32 * 16;
      const int wrow0 = r_lo + (warp & 3) * 32;
      const int rhead = DQ ? head : g, rhpg = DQ ? p.hpg_q : p.hpg_kv;
      store_rows_staged(stage, t0 + Cfg::T_ACC + wg * (D / NWG), any, !any || !r_valid, 1.f, lane,
                        [&](int rr) -> uint4* {
                          const int pos = wrow0 + rr;
                          if (pos >= r_hi) return nullptr;
                          return reinterpret_cast<uint4*>(outp + thd_row(si.start + pos, rhead, rhpg, p.T) * D);
                        });
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// D = 256 dK pass of the dS backward: dK = sum over the contributions of
// dS^T Q, with the dS tiles the dQ pass wrote (the dV pass: dV = sum of
// P^T dO, with the P tiles).  Per contribution (canonical order) a stage
// receives the KV tile's dS tile and the contribution's Q tile, and one
// product accumulates dK in TMEM (the first one with accumulation off).
// dS^T is read from the unswizzled tile as an MN-major A operand: its
// 8-column pieces hold the 128 query rows contiguously, so a core matrix (8
// query rows x 8 KV columns) is 128 contiguous bytes, core matrices 128
// bytes apart along K (query rows: the descriptor's leading offset) and 2048
// along M (KV columns: its stride offset).
//
// CTA pairs: a (2,1,1) cluster takes KV tiles 2i and 2i+1 of a chunk and
// computes both with one M = 256, N = 256, K = 128 tcgen05 product per
// contribution, issued by rank 0.  Each CTA loads its
// own tile's dS^T (P^T) rows (A, 32 KB) and half of the contribution's Q
// (dO) tile, its 128 of the 256 columns (B, 32 KB): 64 KB a CTA a
// contribution instead of 96 KB (dS and P tiles loaded with an evict-first
// L2 policy, the Q and dO halves with evict-last: 3.5 -> 3.1 ms a launch).
// Both CTAs follow tile 2i's contributions;
// tile 2i+1 sees all of them but the diagonal query tile 2i (a tile-level
// causal rule), where its CTA loads a zero tile instead (a load past the
// tile map's start, which TMA fills with zeros), so that it adds exactly 0
// in the canonical order.  Without a tile 2i+1 (odd tiles in the chunk)
// rank 1 computes zeros and writes nothing.  The items are pairs, kv head
// p.kv_head's at [kv_head * n, (kv_head + 1) * n), n = n_kv / hkv.
struct DkvPairCfg {
  static constexpr int THREADS = 384;           // 0 TMA, 1 MMA (rank 0), 2 TMEM, 4..11 epilogue
  static constexpr int D = 256;
  static constexpr int BM = 128, BN = 128;
  static constexpr int A_BYTES = 128 * 128 * 2;
  static constexpr int B_BYTES = BN * (D / 2) * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int NST = 3;
  static constexpr int SMEM_BAR = NST * STAGE;
  static constexpr int SMEM_TOTAL = SMEM_BAR + 256;
  static constexpr int T_ACC = 0, TMEM_COLS = 256;
  static_assert(SMEM_TOTAL + 1024 <= 232448, "SMEM");
  static_assert(NST * STAGE >= 8 * 32 * 256, "epilogue staging fits the stages");
};

template <bool DV>
__global__ void __launch_bounds__(DkvPairCfg::THREADS, 1)
attn_bwd_dkv_pair_kernel(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_t,
                         const BwdParams p) {
  using Cfg = DkvPairCfg;
  constexpr int BM = Cfg::BM, BN = Cfg::BN, D = Cfg::D, NST = Cfg::NST;
  const int n_head = p.hdr->n_kv / p.hkv;
  const int pair = blockIdx.x >> 1;
  if (pair >= n_head) return;                       // both CTAs of the cluster, or neither
  // (a pair never returns on the status word: its two reads could differ)
  const uint32_t rank = cluster_ctarank();
  const WorkItem it = p.items[static_cast<int64_t>(p.kv_head) * n_head + pair];

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_BAR);
  uint64_t* full = bars;                  // [NST] rank 0's count both CTAs' copies
  uint64_t* empty = full + NST;           // [NST] both CTAs (multicast commits)
  uint64_t* acc_done = empty + NST;       // both CTAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = it.step;
  const int G = p.hq / p.hkv;
  const SeqInfo si = seq_info(p, it.b);
  const int tpc = (si.L + 127) / 128;
  const int tile = 2 * it.tile + static_cast<int>(rank);   // this CTA's KV tile of the chunk
  const bool has_tile = tile < tpc;
  const int r_lo = it.c * si.L + tile * BM;
  const int r_hi = min(r_lo + BM, (it.c + 1) * si.L);
  const int r_valid_hi = min(r_hi, si.S);
  const int kv_tile = it.c * tpc + tile;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(acc_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();                     // both CTAs' barriers initialised
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the contributions of tile 2i (those of tile 2i+1 are among them)
  KvIter<BN> itr0;
  itr0.init(p.cp, it.c, si.L, si.S, it.c * si.L + 2 * it.tile * BM, G, g);
  const bool any = !itr0.done;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      KvIter<BN> itr = itr0;
      int64_t n_loads = 0;
      bool ok = true;
      const int64_t plane = DV ? static_cast<int64_t>(G) * p.ds_cap : 0;
      // L2: a dS (P) tile is read once; a Q (dO) tile again by every KV tile pair that sees it
      const uint64_t pol_once = l2_evict_first(), pol_reuse = l2_evict_last();
      for (int j = 0; !itr.done && ok; ++j, itr.next()) {
        const int st = j % NST;
        if (j >= NST) ok = mbar_wait(empty + st, ((j / NST) - 1) & 1, abort_flag);
        if (!ok) break;
        const uint32_t bar = mapa_u32(full + st, 0);
        if (rank == 0) mbar_arrive_expect_tx(full + st, 2 * Cfg::STAGE);
        uint8_t* dst = smem + st * Cfg::STAGE;
        // this CTA's unit of the contribution exists unless its tile lies
        // past the sequence or above the diagonal query tile
        const int q0 = itr.q0();
        const bool unit = has_tile && r_lo < si.S && (itr.cq != it.c || r_lo < min(q0 + BN, itr.q_valid_hi));
        const int32_t t_idx =
            unit ? static_cast<int32_t>(plane + ds_tile_index(p, it.b, si.L, itr.cq, itr.tq, kv_tile, itr.h)) : -1;
        tma_load_3d_pair_hint(dst, &tm_t, 0, 0, t_idx, bar, pol_once);
        const int hq = itr.head();
        const int row = static_cast<int>((hq / p.hpg_q) * p.T) + si.start + q0;
        for (int kc = 0; kc < 2; ++kc)
          tma_load_3d_pair_hint(dst + Cfg::A_BYTES + kc * BN * 128, &tm_b, (2 * static_cast<int>(rank) + kc) * 64,
                                hq % p.hpg_q, row, bar, pol_reuse);
        ++n_loads;
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // rank 0's barriers count both CTAs' copies; the CTAs leave together
      if (rank == 0) wait_last_copies(full, NST, n_loads);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0's
    // whole warp; one elected lane issues)
    if (rank == 0) {
      KvIter<BN> itr = itr0;
      bool ok = true;
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, D, true, true);
      for (int j = 0; !itr.done && ok; ++j, itr.next()) {
        const int st = j % NST;
        ok = mbar_wait_warp(full + st, (j / NST) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t base = smem_u32(smem + st * Cfg::STAGE);
        const uint64_t a_desc = smem_desc_noswz(base, 128, 2048);           // dS^T (P^T), MN-major
        const uint64_t b_desc = smem_desc_sw128(base + Cfg::A_BYTES, BN * 128, 1024);   // Q (dO) half, MN-major
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          umma_ss_pair(tmem + Cfg::T_ACC, a_desc + static_cast<uint64_t>(k * 16 * 16 >> 4),
                       b_desc + mnmajor_step(k), idesc, (j > 0 || k > 0) ? 1u : 0u);
        umma_commit_pair_both(empty + st);
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit_pair_both(acc_done);
      volatile int never = 0;
      mbar_wait(acc_done, 0, &never, 200000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int wg = (warp - 4) >> 2;
    const int row = ((warp & 3) << 5) + lane;
    const uint32_t t0 = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool r_valid = r_lo + row < r_valid_hi;
    bool ok = true;
    if (any) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag));
    if (!ok) {
      raise_status(p.status, CCG_ERR_TIMEOUT);
      *abort_flag = 1;
    } else if (has_tile) {
      // each warpgroup writes 128 columns of the tile's rows (real rows the
      // gradient, padding rows 0), staged in the idle stage area
      tc_fence_after();
      __nv_bfloat16* outp = (DV ? p.out0 : p.out1) + wg * (D / 2);
      uint4* stage = reinterpret_cast<uint4*>(smem) + (warp - 4) * 32 * 16;
      const int wrow0 = r_lo + (warp & 3) * 32;
      store_rows_staged(stage, t0 + Cfg::T_ACC + wg * (D / 2), any, !any || !r_valid, 1.f, lane,
                        [&](int rr) -> uint4* {
                          const int pos = wrow0 + rr;
                          if (pos >= r_hi) return nullptr;
                          return reinterpret_cast<uint4*>(outp + thd_row(si.start + pos, g, p.hpg_kv, p.T) * D);
                        });
    }
  }
  // neither CTA leaves (nor frees TMEM) while the other may still use its
  // shared memory or TMEM: rank 0's MMA thread has seen every product
  // complete, its producer every copy land
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 2) tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// D = 128 dK/dV pass of the dS backward: dV = sum of P^T dO with P^T
// recomputed from S^T = K Q^T, and dK = sum of dS^T Q with the dS tiles the
// dQ pass stored, so dP^T is never formed.  One CTA per 128-row KV tile of
// kv head p.kv_head (the items are the dS backward's KV tile pairs; CTA 2i+s
// takes tile s of pair i).  K is resident (32 KB); per contribution (the
// canonical order) the Q tile and the dS tile arrive together in one of two
// 64 KB stages, the dO tile in one of two 32 KB stages.  TMEM: two S^T
// buffers (128 columns each) next to the dV and dK accumulators, so the
// softmax warpgroup of contribution j (j % 2) forms P^T while the tensor
// core runs dV(j-1), dK(j) and S^T(j+1) (both warpgroups splitting every
// contribution's columns instead measured 5.4 against 5.2 ms a launch).  The
// three products are issued by three warps, each waiting only for its own
// inputs: warp 1 S^T(j) (S^T(j+2) once dV(j) has read P^T(j) from buffer
// j % 2), warp 2 dK(j) (as soon as its stage has landed), warp 3 dV(j) (once
// P^T(j) is packed).  A Q/dS stage is released
// when both its S^T and dK products are done, a dO stage by its dV.  The Q
// tile is read as the K-major B operand of
// S^T and as the MN-major B operand of dK; dS^T is read MN-major from the
// unswizzled stored tile (core matrices 128 B apart along K, 2048 B along M).
struct DkvDs128Cfg {
  static constexpr int THREADS = 384;           // 0 TMA, 1 MMA, 2 TMEM, 4..11 two softmax warpgroups
  static constexpr int D = 128;
  static constexpr int BM = 128, BN = 128;
  static constexpr int K_BYTES = BM * D * 2;    // resident K
  static constexpr int Q_BYTES = BN * D * 2;
  static constexpr int DS_BYTES = 128 * 128 * 2;
  static constexpr int QS_BYTES = Q_BYTES + DS_BYTES;
  static constexpr int DO_BYTES = BN * D * 2;
  static constexpr int SMEM_QS = K_BYTES;
  static constexpr int SMEM_DO = SMEM_QS + 2 * QS_BYTES;
  static constexpr int SMEM_BAR = SMEM_DO + 2 * DO_BYTES;
  static constexpr int SMEM_TOTAL = SMEM_BAR + 256;
  static constexpr int T_DV = 2 * BN, T_DK = 2 * BN + D, TMEM_COLS = 512;
  static_assert(T_DK + D <= TMEM_COLS, "TMEM");
  static_assert(SMEM_TOTAL + 1024 <= 232448, "SMEM");
  static_assert(2 * QS_BYTES >= 8 * 32 * 256, "epilogue staging fits the Q/dS stages");
};

__global__ void __launch_bounds__(DkvDs128Cfg::THREADS, 1)
attn_bwd_dkdv_ds128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using Cfg = DkvDs128Cfg;
  constexpr int BM = Cfg::BM, BN = Cfg::BN, D = Cfg::D, KCH = D / 64;
  const int n_head = p.hdr->n_kv / p.hkv;
  const int pair = blockIdx.x >> 1;
  if (pair >= n_head) return;
  if (status_bad(p.status)) return;
  const WorkItem it = p.items[static_cast<int64_t>(p.kv_head) * n_head + pair];
  const SeqInfo si = seq_info(p, it.b);
  const int tpc = (si.L + 127) / 128;
  const int tile = 2 * it.tile + static_cast<int>(blockIdx.x & 1);
  if (tile >= tpc) return;                          // a chunk with an odd number of tiles

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_BAR);
  uint64_t* res_full = bars;
  uint64_t* qs_full = res_full + 1;       // [2] Q and dS of a contribution
  uint64_t* qs_empty = qs_full + 2;       // [2]
  uint64_t* do_full = qs_empty + 2;       // [2] dO of a contribution
  uint64_t* do_empty = do_full + 2;       // [2]
  uint64_t* s_full = do_empty + 2;        // [2] S^T in buffer b
  uint64_t* p_full = s_full + 2;          // [2] P^T packed over buffer b
  uint64_t* dv_done = p_full + 2;         // [2] dV(j) complete: buffer j % 2 is free
  uint64_t* acc_done = dv_done + 2;       // every issuer's products complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = it.step;
  const int G = p.hq / p.hkv;
  const int k_lo = it.c * si.L + tile * BM;
  const int k_hi = min(k_lo + BM, (it.c + 1) * si.L);
  const int k_valid_hi = min(k_hi, si.S);
  const int kv_tile = it.c * tpc + tile;

  if (threadIdx.x == 0) {
    mbar_init(res_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(qs_full + b, 1);
      mbar_init(qs_empty + b, 2);                  // S^T and dK
      mbar_init(do_full + b, 1);
      mbar_init(do_empty + b, 1);
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, 128);
      mbar_init(dv_done + b, 1);
    }
    mbar_init(acc_done, 3);
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
  KvIter<BN> itr0;
  itr0.init(p.cp, it.c, si.L, si.S, k_lo, G, g);
  const bool any = !itr0.done;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      KvIter<BN> itr = itr0;
      int64_t n = 0;                                 // contributions
      int64_t n_qs = 0, n_do = 0;                    // Q/dS and dO copies issued
      bool ok = true;
      // L2: a dS tile is read once; a Q (dO) tile again by every KV tile that sees it
      const uint64_t pol_once = l2_evict_first(), pol_reuse = l2_evict_last();
      if (!itr.done) {
        const int krow = static_cast<int>((g / p.hpg_kv) * p.T) + si.start + k_lo;
        mbar_arrive_expect_tx(res_full, Cfg::K_BYTES);
        for (int kc = 0; kc < KCH; ++kc)
          tma_load_3d(smem + kc * BM * 128, &tm_k, kc * 64, g % p.hpg_kv, krow, res_full);
        for (; !itr.done && ok; ++n, itr.next()) {
          const int st = static_cast<int>(n & 1);
          const uint32_t ph = static_cast<uint32_t>(((n >> 1) - 1) & 1);
          const int hq = itr.head();
          const int qrow = static_cast<int>((hq / p.hpg_q) * p.T) + si.start + itr.q0();
          // Q and dS
          if (n >= 2) ok = mbar_wait(qs_empty + st, ph, abort_flag);
          if (!ok) break;
          uint8_t* qs = smem + Cfg::SMEM_QS + st * Cfg::QS_BYTES;
          mbar_arrive_expect_tx(qs_full + st, Cfg::QS_BYTES);
          for (int kc = 0; kc < KCH; ++kc)
            tma_load_3d_hint(qs + kc * BN * 128, &tm_q, kc * 64, hq % p.hpg_q, qrow, qs_full + st, pol_reuse);
          const __nv_bfloat16* ds = p.ds + ds_tile_index(p, it.b, si.L, itr.cq, itr.tq, kv_tile, itr.h) * (128 * 128);
          bulk_load_hint(qs + Cfg::Q_BYTES, ds, Cfg::DS_BYTES, qs_full + st, pol_once);
          ++n_qs;
          // dO
          if (n >= 2) ok = mbar_wait(do_empty + st, ph, abort_flag);
          if (!ok) break;
          uint8_t* dst = smem + Cfg::SMEM_DO + st * Cfg::DO_BYTES;
          mbar_arrive_expect_tx(do_full + st, Cfg::DO_BYTES);
          for (int kc = 0; kc < KCH; ++kc)
            tma_load_3d_hint(dst + kc * BN * 128, &tm_do, kc * 64, hq % p.hpg_q, qrow, do_full + st, pol_reuse);
          ++n_do;
        }
        if (!ok) {
          raise_status(p.status, CCG_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        volatile int never = 0;
        mbar_wait(res_full, 0, &never, 200000000ull);
        wait_last_copies(qs_full, 2, n_qs);
        wait_last_copies(do_full, 2, n_do);
      }
    }
  } else if (warp <= 3) {
    // ------------------------------------------------------------ MMA issuers
    // (each a whole warp; one elected lane issues)
    {
      KvIter<BN> cnt = itr0;
      int n = 0;
      for (; !cnt.done; cnt.next()) ++n;
      bool ok = true;
      if (n > 0) {
        const uint32_t qs0 = smem_u32(smem + Cfg::SMEM_QS), do0 = smem_u32(smem + Cfg::SMEM_DO);
        if (warp == 1) {
          // S^T(j) = K Q_j^T into buffer j % 2
          const uint64_t k_desc = smem_desc_sw128(smem_u32(smem), 16, 1024);
          ok = mbar_wait_warp(res_full, 0, abort_flag);
          for (int j = 0; ok && j < n; ++j) {
            const int st = j & 1;
            if (j >= 2) {
              ok = mbar_wait_warp(dv_done + st, ((j - 2) >> 1) & 1, abort_flag);
              if (!ok) break;
            }
            ok = mbar_wait_warp(qs_full + st, (j >> 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            mma_kk<BM, BN, D>(tmem + st * BN, k_desc, smem_desc_sw128(qs0 + st * Cfg::QS_BYTES, 16, 1024));
            umma_commit(s_full + st);
            umma_commit(qs_empty + st);
          }
        } else if (warp == 2) {
          // dK += dS_j^T Q_j
          constexpr uint32_t idesc_dk = idesc_bf16_f32(BM, D, true, true);
          for (int j = 0; ok && j < n; ++j) {
            const int st = j & 1;
            ok = mbar_wait_warp(qs_full + st, (j >> 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            const uint32_t base = qs0 + st * Cfg::QS_BYTES;
            const uint64_t a_desc = smem_desc_noswz(base + Cfg::Q_BYTES, 128, 2048);
            const uint64_t b_desc = smem_desc_sw128(base, BN * 128, 1024);
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
              umma_ss(tmem + Cfg::T_DK, a_desc + static_cast<uint64_t>(k * 16 * 16 >> 4), b_desc + mnmajor_step(k),
                      idesc_dk, (j > 0 || k > 0) ? 1u : 0u);
            umma_commit(qs_empty + st);
          }
        } else {
          // dV += P_j^T dO_j
          for (int j = 0; ok && j < n; ++j) {
            const int b = j & 1;
            ok = mbar_wait_warp(p_full + b, (j >> 1) & 1, abort_flag);
            if (!ok) break;
            ok = mbar_wait_warp(do_full + b, (j >> 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            mma_tn<BN, D>(tmem + Cfg::T_DV, tmem + b * BN, smem_desc_sw128(do0 + b * Cfg::DO_BYTES, BN * 128, 1024),
                          j > 0);
            umma_commit(do_empty + b);
            umma_commit(dv_done + b);
          }
        }
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // a commit tracks only its own thread's products: all three arrive
      umma_commit(acc_done);
      volatile int never = 0;
      mbar_wait(acc_done, 0, &never, 200000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax: P^T of contributions j % 2 == wg
    const int wg = (warp - 4) >> 2;
    const int row = ((warp & 3) << 5) + lane;        // key row of the tile
    const uint32_t t0 = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int k_pos = k_lo + row;
    const bool k_valid = k_pos < k_valid_hi;
    const uint64_t scale2 = f32x2(p.scale_log2, p.scale_log2);
    KvIter<BN> itr = itr0;
    bool ok = true;
    for (int j = 0; !itr.done; ++j, itr.next()) {
      if ((j & 1) != wg) continue;
      const uint32_t tb = t0 + wg * BN;
      // -LSE (log2 units) of the contribution's query columns: lane l holds
      // columns 2l, 2l+1 (lo) and 64+2l, 64+2l+1 (hi), handed out by shuffles
      uint64_t lse_lo, lse_hi;
      {
        const int q0 = itr.q0();
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = (e >> 1) * 64 + 2 * lane + (e & 1);
          v[e] = 0.f;
          if (q0 + col < itr.q_valid_hi)
            v[e] = -__ldg(p.lse + thd_row(si.start + q0 + col, itr.head(), p.hpg_q, p.T)) * kLog2e;
        }
        lse_lo = f32x2(v[0], v[1]);
        lse_hi = f32x2(v[2], v[3]);
      }
      const int q0 = itr.q0();
      // query column c is visible to this key row iff q0+c >= k_pos and q0+c < q_valid_hi
      const int c_lo = k_valid ? max(0, k_pos - q0) : BN;
      const int c_hi = k_valid ? itr.q_valid_hi - q0 : 0;
      const bool masked = __any_sync(0xffffffffu, c_lo > 0 || c_hi < BN);
      ok = __all_sync(0xffffffffu, mbar_wait(s_full + wg, (j >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t rs[32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        tmem_ld32(tb + c * 32, rs);
        tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int col = c * 32 + x;
            rs[x] = (col >= c_lo && col < c_hi) ? rs[x] : 0xff800000u;
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          // columns c*32 + 2x, +1: held by lane (16c + x) % 32, in lo (c < 2) or hi
          const uint64_t nl = __shfl_sync(0xffffffffu, c < 2 ? lse_lo : lse_hi, (16 * c + x) & 31);
          float a0, a1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(rs[2 * x]), __uint_as_float(rs[2 * x + 1])), scale2, nl),
                      a0, a1);
          pk[x] = pack_bf16x2(ex2_approx(a0), ex2_approx(a1));
        }
        tmem_st16(tb + c * 16, pk);                 // P^T packed over the buffer's first 64 columns
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full + wg);
    }
    if (ok && any) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag));
    if (!ok) {
      raise_status(p.status, CCG_ERR_TIMEOUT);
      *abort_flag = 1;
    } else {
      // warpgroup 0 writes dV, warpgroup 1 dK (real rows the gradient,
      // padding rows 0), staged in the idle Q/dS stages
      tc_fence_after();
      __nv_bfloat16* outp = wg == 0 ? p.out0 : p.out1;
      uint4* stage = reinterpret_cast<uint4*>(smem + Cfg::SMEM_QS) + (warp - 4) * 32 * 16;
      const int wrow0 = k_lo + (warp & 3) * 32;
      store_rows_staged(stage, t0 + (wg == 0 ? Cfg::T_DV : Cfg::T_DK), any, !any || !k_valid, 1.f, lane,
                        [&](int rr) -> uint4* {
                          const int pos = wrow0 + rr;
                          if (pos >= k_hi) return nullptr;
                          return reinterpret_cast<uint4*>(outp + thd_row(si.start + pos, g, p.hpg_kv, p.T) * D);
                        });
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// D = 256 dV pass: one CTA per (128-row KV tile, kv head) with only K
// resident (64 KB), so five half-tile slots stream the 128-column halves of
// Q_i (for S^T = sum_h K[:, h] Q_i,h^T) and dO_i (for dV[:, h] += P^T dO_i,h)
// of every contribution in the canonical order, and TMEM holds two S^T
// buffers next to the 256-column dV accumulator: S^T of contribution i+1 is
// computed while the softmax warpgroups form P^T of contribution i (they
// split its 128 columns and pack P^T in place, over the first half of their
// own columns).  Stream order: Q_0, then Q_{i+1}, dO_i for i = 0, 1, ...
// (two halves each), which is the order the MMA warp uses them in.
struct DvCfg {
  static constexpr int D = 256;
  static constexpr int BM = 128;                 // key rows (MMA M)
  static constexpr int BN = 128;                 // query rows per contribution
  static constexpr int DH = 128;
  static constexpr int NSLOT = 5;
  static constexpr int RES_BYTES = BM * D * 2;   // K
  static constexpr int HALF_BYTES = BN * DH * 2;
  static constexpr int SMEM_SLOT = RES_BYTES;
  static constexpr int SMEM_VEC = SMEM_SLOT + NSLOT * HALF_BYTES;  // [WG][-lse2 x 64]
  static constexpr int VEC_BYTES = 2 * (BN / 2) * 4;
  static constexpr int SMEM_BAR = SMEM_VEC + VEC_BYTES;
  static constexpr int SMEM_TOTAL = SMEM_BAR + 256;
  static constexpr int T_BUF = BN;               // S^T buffer b at b * T_BUF
  static constexpr int T_ACC = 2 * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(T_ACC + D <= TMEM_COLS, "TMEM");
  static_assert(SMEM_TOTAL + 1024 <= 232448, "SMEM");
};

__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dv256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const BwdParams p) {
  using Cfg = DvCfg;
  constexpr int BM = Cfg::BM, BN = Cfg::BN, NSLOT = Cfg::NSLOT, D = Cfg::D;
  const int item_idx = blockIdx.x;              // items carry their kv head
  if (item_idx >= p.hdr->n_kv) return;
  if (status_bad(p.status)) return;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_BAR);
  uint64_t* res_full = bars;
  uint64_t* full = bars + 1;              // [NSLOT]
  uint64_t* empty = full + NSLOT;         // [NSLOT]
  uint64_t* s_full = empty + NSLOT;       // [2]: S^T of the contribution in buffer b complete
  uint64_t* p_full = s_full + 2;          // [2]: P^T packed in buffer b (both warpgroups)
  uint64_t* acc_done = p_full + 2;
  uint64_t* vec_ready = acc_done + 1;     // [2 WG]
  uint64_t* vec_free = vec_ready + 2;     // [2 WG]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(vec_free + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* vec = reinterpret_cast<float*>(smem + Cfg::SMEM_VEC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[item_idx];
  const int g = it.step;                       // kv head of the item
  const int G = p.hq / p.hkv;
  const SeqInfo si = seq_info(p, it.b);
  const int k_lo = it.c * si.L + it.tile * BM;
  const int k_hi = min(k_lo + BM, (it.c + 1) * si.L);
  const int k_valid_hi = min(k_hi, si.S);

  if (threadIdx.x == 0) {
    mbar_init(res_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, 256);
    }
    mbar_init(acc_done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(vec_ready + b, 128);
      mbar_init(vec_free + b, 128);
    }
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
  const int kv_group_row = static_cast<int>((g / p.hpg_kv) * p.T) + si.start;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      KvIter<BN> qi, di;                         // Q runs one contribution ahead of dO
      qi.init(p.cp, it.c, si.L, si.S, k_lo, G, g);
      di.init(p.cp, it.c, si.L, si.S, k_lo, G, g);
      int64_t n_loads = 0;                       // copies issued (slot = position % NSLOT)
      bool ok = true;
      int t = 0;                                 // stream position
      auto load = [&](const KvIter<BN>& itr, const CUtensorMap* map) -> bool {
        const int hq = itr.head();
        const int row = static_cast<int>((hq / p.hpg_q) * p.T) + si.start + itr.q0();
        for (int hf = 0; hf < 2; ++hf, ++t) {
          const int slot = t % NSLOT;
          if (t >= NSLOT && !mbar_wait(empty + slot, ((t / NSLOT) - 1) & 1, abort_flag)) return false;
          mbar_arrive_expect_tx(full + slot, Cfg::HALF_BYTES);
          uint8_t* dst = smem + Cfg::SMEM_SLOT + slot * Cfg::HALF_BYTES;
          for (int kc = 0; kc < 2; ++kc)
            tma_load_3d(dst + kc * BN * 128, map, (2 * hf + kc) * 64, hq % p.hpg_q, row, full + slot);
          ++n_loads;
        }
        return true;
      };
      if (!qi.done) {
        mbar_arrive_expect_tx(res_full, Cfg::RES_BYTES);
        for (int kc = 0; kc < D / 64; ++kc)
          tma_load_3d(smem + kc * BM * 128, &tm_k, kc * 64, g % p.hpg_kv, kv_group_row + k_lo, res_full);
        ok = load(qi, &tm_q);
        qi.next();
        while (ok && !di.done) {
          if (!qi.done) {
            ok = load(qi, &tm_q);
            qi.next();
            if (!ok) break;
          }
          ok = load(di, &tm_do);
          di.next();
        }
        if (!ok) {
          raise_status(p.status, CCG_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        volatile int never = 0;
        mbar_wait(res_full, 0, &never, 200000000ull);
        wait_last_copies(full, NSLOT, n_loads);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp; one elected lane issues)
    {
      KvIter<BN> ahead;
      ahead.init(p.cp, it.c, si.L, si.S, k_lo, G, g);
      bool ok = true;
      if (!ahead.done) {
        const uint64_t k_desc = smem_desc_sw128(smem_u32(smem), 16, 1024);
        const uint32_t slot_base = smem_u32(smem + Cfg::SMEM_SLOT);
        const uint64_t slot_k0 = smem_desc_sw128(slot_base, 16, 1024);
        const uint64_t slot_mn0 = smem_desc_sw128(slot_base, BN * 128, 1024);
        constexpr uint32_t kSlotStep = Cfg::HALF_BYTES >> 4;
        int u = 0;                                // stream position consumed
        ok = mbar_wait_warp(res_full, 0, abort_flag);
        tc_fence_after();
        auto issue_st = [&](int j) -> bool {      // S^T of contribution j -> buffer j % 2
          const uint32_t buf = tmem + (j & 1) * Cfg::T_BUF;
          for (int hf = 0; hf < 2; ++hf, ++u) {
            const int sl = u % NSLOT;
            if (!mbar_wait_warp(full + sl, (u / NSLOT) & 1, abort_flag)) return false;
            tc_fence_after();
            mma_kk_half(buf, k_desc + kmajor_step(128, 8 * hf), slot_k0 + sl * kSlotStep, hf > 0);
            umma_commit(empty + sl);              // Q half done
          }
          umma_commit(s_full + (j & 1));
          return true;
        };
        int j_st = 0;
        while (ok && !ahead.done && j_st < 2) {
          ok = issue_st(j_st++);
          ahead.next();
        }
        for (int j = 0; ok && j < j_st; ++j) {
          const int b = j & 1;
          ok = mbar_wait_warp(p_full + b, (j >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          for (int hf = 0; hf < 2 && ok; ++hf, ++u) {
            const int sl = u % NSLOT;
            ok = mbar_wait_warp(full + sl, (u / NSLOT) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            mma_tn_split<BN, Cfg::DH, true>(tmem + Cfg::T_ACC + hf * Cfg::DH, tmem + b * Cfg::T_BUF,
                                            slot_mn0 + sl * kSlotStep, j > 0);
            umma_commit(empty + sl);              // dO half done
          }
          if (ok && !ahead.done) {
            ok = issue_st(j_st++);
            ahead.next();
          }
        }
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(acc_done);
      volatile int never = 0;
      mbar_wait(acc_done, 0, &never, 200000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax: P^T
    const int wg = (warp - 4) >> 2;
    const int row = ((warp & 3) << 5) + lane;        // key row of the tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t0 = tmem + lane_base;
    constexpr int NC = BN / 64;
    const int c_first = wg * NC;
    const int k_pos = k_lo + row;
    const bool k_valid = k_pos < k_valid_hi;
    float* vb = vec + wg * (BN / 2);                 // -LSE (log2 units) of this warpgroup's columns
    const uint64_t scale2 = f32x2(p.scale_log2, p.scale_log2);
    KvIter<BN> itr;
    itr.init(p.cp, it.c, si.L, si.S, k_lo, G, g);
    const bool any = !itr.done;
    bool ok = true;
    for (int j = 0; !itr.done; ++j, itr.next()) {
      const int b = j & 1;
      const uint32_t tb = t0 + b * Cfg::T_BUF;
      if (j > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(vec_free + wg, (j - 1) & 1, abort_flag));
        if (!ok) break;
      }
      if (row < BN / 2) {
        const int qp = itr.q0() + c_first * 32 + row;
        const bool qv = qp < itr.q_valid_hi;
        const int64_t gr = thd_row(si.start + qp, itr.head(), p.hpg_q, p.T);
        vb[row] = qv ? -__ldg(p.lse + gr) * kLog2e : 0.f;
      }
      mbar_arrive(vec_ready + wg);
      ok = __all_sync(0xffffffffu, mbar_wait(vec_ready + wg, j & 1, abort_flag));
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(s_full + b, (j >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int q0 = itr.q0();
      const int c_lo = k_valid ? max(0, k_pos - q0) : BN;
      const int c_hi = k_valid ? itr.q_valid_hi - q0 : 0;
      const bool masked = __any_sync(0xffffffffu, c_lo > 0 || c_hi < BN);
      uint32_t rs[32];
#pragma unroll
      for (int c = c_first; c < c_first + NC; ++c) {
        tmem_ld32(tb + c * 32, rs);
        tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int col = c * 32 + x;
            rs[x] = (col >= c_lo && col < c_hi) ? rs[x] : 0xff800000u;
          }
        }
        const ulonglong2* nl4 = reinterpret_cast<const ulonglong2*>(vb + (c - c_first) * 32);
        uint32_t pk[16];
#pragma unroll
        for (int x2 = 0; x2 < 8; ++x2) {
          const ulonglong2 lv = nl4[x2];                   // four columns' -LSE2 per 16-byte load
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int x = 2 * x2 + e;
            float a0, a1;   // P = 2^(s * scale_log2 - lse2)
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(rs[2 * x]), __uint_as_float(rs[2 * x + 1])), scale2,
                                  e ? lv.y : lv.x),
                        a0, a1);
            pk[x] = pack_bf16x2(ex2_approx(a0), ex2_approx(a1));
          }
        }
        tmem_st16(tb + c_first * 32 + (c - c_first) * 16, pk);   // in place, own columns
      }
      mbar_arrive(vec_free + wg);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full + b);
    }
    if (ok && any) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag));
    if (!ok) {
      raise_status(p.status, CCG_ERR_TIMEOUT);
      *abort_flag = 1;
    } else {
      // each warpgroup writes 128 of the tile rows' dV columns (padding rows
      // 0) through a staging block in the idle slot area
      tc_fence_after();
      __nv_bfloat16* outp = p.out0 + wg * (D / 2);
      uint4* stage = reinterpret_cast<uint4*>(smem + Cfg::SMEM_SLOT) + (warp - 4) * 32 * 16;
      const int wrow0 = k_lo + (warp & 3) * 32;
      store_rows_staged(stage, t0 + Cfg::T_ACC + wg * (D / 2), any, !any || !k_valid, 1.f, lane,
                        [&](int rr) -> uint4* {
                          const int pos = wrow0 + rr;
                          if (pos >= k_hi) return nullptr;
                          return reinterpret_cast<uint4*>(outp + thd_row(si.start + pos, g, p.hpg_kv, p.T) * D);
                        });
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

template <class K>
cudaError_t set_smem(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <class Cfg, int D>
cudaError_t launch_dq(const CUtensorMap* m, const BwdParams& p, int grid_items, cudaStream_t s) {
  const int smem = Cfg::SMEM_TOTAL + 1024;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [&] { return set_smem(attn_bwd_dq_kernel<Cfg, D>, smem); });
  if (e != cudaSuccess) return e;
  const int64_t grid = static_cast<int64_t>(grid_items) * p.nheads;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  attn_bwd_dq_kernel<Cfg, D><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(m[0], m[1], m[2], m[3], p);
  return cudaGetLastError();
}

template <class Cfg, int D>
cudaError_t launch_kv(const CUtensorMap* m, const BwdParams& p, int grid_items, cudaStream_t s) {
  const int smem = Cfg::SMEM_TOTAL + 1024;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [&] { return set_smem(attn_bwd_kv_kernel<Cfg, D>, smem); });
  if (e != cudaSuccess) return e;
  const int64_t grid = static_cast<int64_t>(grid_items) * p.hkv;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  attn_bwd_kv_kernel<Cfg, D><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(m[0], m[1], m[2], m[3], p);
  return cudaGetLastError();
}

// Softmax warpgroups of the D = 256 dQ and dK passes: two, each thread
// forming 64 of every unit's 128 columns (four warpgroups, at 96 registers a
// thread, measured 3-6% slower).
constexpr int kHalfWarpgroups = 2;

template <HalfRole ROLE>
cudaError_t launch_half(const CUtensorMap* m, const BwdParams& p, int grid_items, cudaStream_t s) {
  using Cfg = HalfCfg<kHalfWarpgroups>;
  const int smem = Cfg::SMEM_TOTAL + 1024;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(
      attr_done, [&] { return set_smem(attn_bwd_half_kernel<ROLE, kHalfWarpgroups>, smem); });
  if (e != cudaSuccess) return e;
  const int64_t grid = static_cast<int64_t>(grid_items) * (ROLE == HalfRole::kDq ? p.nheads : p.hkv);
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  attn_bwd_half_kernel<ROLE, kHalfWarpgroups>
      <<<static_cast<unsigned>(grid), Cfg::THREADS, smem, s>>>(m[0], m[1], m[2], m[3], p);
  return cudaGetLastError();
}

template <bool DV>
cudaError_t launch_dkv_pair(const CUtensorMap& tb, const CUtensorMap& tt, const BwdParams& p, int pairs,
                            cudaStream_t s) {
  auto kern = attn_bwd_dkv_pair_kernel<DV>;
  const int smem = DkvPairCfg::SMEM_TOTAL + 1024;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [&] { return set_smem(kern, smem); });
  if (e != cudaSuccess) return e;
  if (pairs < 1 || pairs > 0x3fffffff) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(DkvPairCfg::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tb, tt, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_dkdv_ds128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tdo,
                              const BwdParams& p, int pairs, cudaStream_t s) {
  const int smem = DkvDs128Cfg::SMEM_TOTAL + 1024;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [&] { return set_smem(attn_bwd_dkdv_ds128_kernel, smem); });
  if (e != cudaSuccess) return e;
  if (pairs < 1 || pairs > 0x3fffffff) return cudaErrorInvalidValue;
  attn_bwd_dkdv_ds128_kernel<<<static_cast<unsigned>(2 * pairs), DkvDs128Cfg::THREADS, smem, s>>>(tq, tk, tdo, p);
  return cudaGetLastError();
}

cudaError_t launch_dv256(const CUtensorMap* m, const BwdParams& p, int grid_items, cudaStream_t s) {
  const int smem = DvCfg::SMEM_TOTAL + 1024;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [&] { return set_smem(attn_bwd_dv256_kernel, smem); });
  if (e != cudaSuccess) return e;
  const int64_t grid = static_cast<int64_t>(grid_items) * p.hkv;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  attn_bwd_dv256_kernel<<<static_cast<unsigned>(grid), kThreads, smem, s>>>(m[0], m[1], m[2], m[3], p);
  return cudaGetLastError();
}

// Tile shapes.  D = 128: whole streamed tiles, dK and dV in one kernel.
// D = 256: the dQ and dK passes (attn_bwd_half_kernel) and the dV pass
// (attn_bwd_dv256_kernel) stream 128-column halves of 128-row tiles.
using Dq128 = DqCfg<128, 128, 5>;
using Kv128 = KvCfg<128, 128, 4, 1>;

}  // namespace

int bwd_q_tile_rows(int) { return 128; }
int bwd_kv_tile_rows(int) { return 128; }
// Box rows of the twelve tensor maps: 0..3 = q, k, v, dO for the dQ pass,
// 4..7 = the same for the first dK/dV kernel, 8..11 for the second (D = 256).
// Every pass moves 128-row boxes.
int bwd_map_rows(int, int) { return 128; }

cudaError_t launch_attn_bwd(const CUtensorMap* maps, const WorkItem* dq_items, const WorkItem* kv_items,
                            const PlanHeader* hdr, const int32_t* cu, const int32_t* cu_pad, const float* lse,
                            const float* delta, void* dq, void* dk, void* dv, int32_t* status, int cp, int hq,
                            int hkv, int head_groups, int64_t T, int D, float scale, int grid_q, int grid_kv,
                            int* launches, cudaStream_t stream, void* ds, const int64_t* ds_base, int64_t ds_cap,
                            const CUtensorMap* ds_map, int kv_pairs) {
  BwdParams p;
  p.hdr = hdr;
  p.cu = cu;
  p.cu_pad = cu_pad;
  p.lse = lse;
  p.delta = delta;
  p.status = status;
  p.cp = cp;
  p.hq = hq;
  p.hkv = hkv;
  p.hpg_q = hq / head_groups;
  p.hpg_kv = hkv / head_groups;
  p.T = T;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.head0 = 0;
  p.nheads = hq;
  p.ds = nullptr;
  p.ds_base = ds_base;
  p.ds_cap = ds_cap;
  p.kv_head = 0;
  cudaError_t e;
  if (D == 128 && ds != nullptr) {
    // dS backward at D = 128: per kv head, the dQ pass over its q heads
    // writes their dS tiles, then one dK/dV pass recomputes P^T and reads them
    const int G = hq / hkv;
    for (int g = 0; g < hkv; ++g) {
      p.items = dq_items;
      p.out0 = static_cast<__nv_bfloat16*>(dq);
      p.out1 = nullptr;
      p.head0 = g * G;
      p.nheads = G;
      p.ds = static_cast<__nv_bfloat16*>(ds);
      prof_begin("attn_bwd_dq", stream);
      e = launch_dq<Dq128, 128>(maps, p, grid_q, stream);
      prof_end(stream);
      if (e != cudaSuccess) return e;
      ++*launches;
      p.items = kv_items;
      p.out0 = static_cast<__nv_bfloat16*>(dv);
      p.out1 = static_cast<__nv_bfloat16*>(dk);
      p.kv_head = g;
      prof_begin("attn_bwd_dkdv", stream);
      e = launch_dkdv_ds128(maps[4], maps[5], maps[7], p, kv_pairs, stream);
      prof_end(stream);
      if (e != cudaSuccess) return e;
      ++*launches;
    }
    return cudaSuccess;
  }
  if (D == 256 && ds != nullptr) {
    // dS backward: per kv head, the dQ pass over its q heads writes their dS
    // and P tiles, then its dK pass and its dV pass read them
    const int G = hq / hkv;
    for (int g = 0; g < hkv; ++g) {
      p.items = dq_items;
      p.out0 = static_cast<__nv_bfloat16*>(dq);
      p.out1 = nullptr;
      p.head0 = g * G;
      p.nheads = G;
      p.ds = static_cast<__nv_bfloat16*>(ds);
      prof_begin("attn_bwd_dq", stream);
      e = launch_half<HalfRole::kDq>(maps, p, grid_q, stream);
      prof_end(stream);
      if (e != cudaSuccess) return e;
      ++*launches;
      p.items = kv_items;
      p.out0 = static_cast<__nv_bfloat16*>(dv);
      p.out1 = static_cast<__nv_bfloat16*>(dk);
      p.kv_head = g;
      prof_begin("attn_bwd_dk", stream);
      e = launch_dkv_pair<false>(maps[8], *ds_map, p, kv_pairs, stream);
      prof_end(stream);
      if (e != cudaSuccess) return e;
      ++*launches;
      prof_begin("attn_bwd_dv", stream);
      e = launch_dkv_pair<true>(maps[11], *ds_map, p, kv_pairs, stream);
      prof_end(stream);
      if (e != cudaSuccess) return e;
      ++*launches;
    }
    return cudaSuccess;
  }
  // dQ pass
  p.items = dq_items;
  p.out0 = static_cast<__nv_bfloat16*>(dq);
  p.out1 = nullptr;
  prof_begin("attn_bwd_dq", stream);
  e = D == 128 ? launch_dq<Dq128, 128>(maps, p, grid_q, stream) : launch_half<HalfRole::kDq>(maps, p, grid_q, stream);
  prof_end(stream);
  if (e != cudaSuccess) return e;
  ++*launches;
  // dK/dV pass
  p.items = kv_items;
  p.out0 = static_cast<__nv_bfloat16*>(dv);
  p.out1 = static_cast<__nv_bfloat16*>(dk);
  if (D == 128) {
    prof_begin("attn_bwd_dkdv", stream);
    e = launch_kv<Kv128, 128>(maps + 4, p, grid_kv, stream);
    prof_end(stream);
    if (e != cudaSuccess) return e;
    ++*launches;
  } else {
    prof_begin("attn_bwd_dv", stream);
    e = launch_dv256(maps + 4, p, grid_kv, stream);
    prof_end(stream);
    if (e != cudaSuccess) return e;
    ++*launches;
    prof_begin("attn_bwd_dk", stream);
    e = launch_half<HalfRole::kDk>(maps + 8, p, grid_kv, stream);
    prof_end(stream);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  return cudaSuccess;
}

}  // namespace ccg
