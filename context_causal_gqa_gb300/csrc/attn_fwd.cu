// attn_fwd.cu -- a3: the ring-step partials of the CP-emulated causal GQA
// forward on the 5th-generation tensor cores (sm_103a).
//
// TransformerEngine PR "Optimize context parallel attention layouts and
// gradient accumulation", Independent-node complete-CP evidence: each CP
// rank attends its two query chunks against the KV it holds at a ring step
// and keeps the partial output with its LSE ("Stats") for the merge.
//
// One persistent launch covers every ring step: the work list holds one item
// per (query chunk, 128-row query tile), heaviest first, and each item is
// computed for NH q heads that share one kv head (GQA K/V reuse: every K/V
// tile is loaded once for the NH heads).  An item walks the ring steps of its
// chunk's rank in order; at each step it attends the source rank's KV chunks
// that it can see (causal block skipping: KV tiles past the tile's last row
// are never loaded) with a fresh online softmax and writes that step's
// partial (O_s, LSE_s).  Q is loaded once per item and the K/V stream, the S
// lookahead and the tensor core run on across the step boundaries; only the
// O read-out of a finished step waits on its last P V product.  CTAs stride
// through the list, so the next item's Q load and first S = Q K^T products
// overlap the current item's last P V product and its epilogue.  The same
// kernel computes one ring step alone (one item per tile of that step), or
// every step in one online softmax (the fused forward, no partials).
// Roles:
//   warp 0     TMA producer: Q per item, K and V tiles through single-tile slots
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

template <int D, int NH, bool PAIR = false>
struct FwdCfg {
  // 128-key tiles: the S = Q K^T products run at N = 128 (full tensor rate;
  // N = 64 issues at two thirds of it) and the MMA warp's per-tile
  // synchronisation is spread over twice the keys.
  static constexpr int BN = 128;
  // TMEM per head: SBUF S buffers (BN columns each) + O (D columns).
  //   D=128, one head:  3 S buffers, S of tile t+2 issued before P of tile t (LA = 2)
  //   D=256, one head:  2 S buffers, LA = 1
  //   D=128, two heads: 1 S buffer per head, the heads interleave (LA = 1)
  static constexpr int SBUF = NH == 2 ? 1 : (D == 128 ? 3 : 2);
  static constexpr int LA = SBUF == 3 ? 2 : 1;
  static constexpr int KCH = D / 64;                       // 64-wide (128-byte) column chunks
  static constexpr int Q_BYTES = kBM * D * 2;              // one head
  static constexpr int KV_BYTES = BN * D * 2;              // one K (or V) tile
  // A CTA pair (2 NH q heads of one kv group, NH per CTA; head slot h of
  // both CTAs in one M = 256 product) holds half of every K tile in each CTA
  // (BN/2 keys, all D columns: the N half of S = Q K^T) and half of every V
  // tile (all BN keys, D/2 columns: the N half of O += P V).
  static constexpr int SLOT_BYTES = PAIR ? KV_BYTES / 2 : KV_BYTES;
  static constexpr int K_ROWS = PAIR ? BN / 2 : BN;        // key rows of a K slot
  static constexpr int V_CH = PAIR ? KCH / 2 : KCH;        // 64-column chunks of a V slot
  // D=256: shared memory beside the K/V slots stages half of a finished
  // segment's O rows (128 columns, 256 B a row), so that O can be released
  // to the next segment's first P V product before the global stores of
  // the partial are issued
  // D=128, two heads: each head's finished O leaves through its own 16 KB
  // box (64 columns x 128 rows, TMA stores), one K/V slot fewer
  static constexpr bool STAGE = (D == 256 && NH == 1) || (D == 128 && NH == 2);
  static constexpr int BOX_BYTES = kBM * 128;
  static constexpr int STAGE_BYTES = (D == 256 && NH == 1) ? kBM * (D / 2) * 2 : (STAGE ? NH * BOX_BYTES : 0);
  // K and V tiles stream through NSLOT slots in the order the MMA warp
  // consumes them (per item: K_0..K_{LA-1}, then K_{j+LA} and V_j for
  // j = 0, 1, ...); a slot is released when its S or P V product is done.
  // At D=256 one CTA holds only two whole-tile slots: K_{t+1} reloads while
  // softmax(t) runs and V_{t+1} while S(t+2) and softmax(t+1) run.  A pair
  // holds four half-tile slots in each CTA: V_t loads as soon as P V of tile
  // t-2 is done, K_{t+1} as soon as S(t-1) is.
  static constexpr int NSLOT =
      (227 * 1024 - 2048 - NH * Q_BYTES - ((D == 256 && NH == 1 && !PAIR) ? 0 : STAGE_BYTES)) / SLOT_BYTES;
  static constexpr int SMEM_Q = 0;
  static constexpr int SMEM_KV = SMEM_Q + NH * Q_BYTES;
  static constexpr int SMEM_STAGE = SMEM_KV + NSLOT * SLOT_BYTES;
  static constexpr int SMEM_BAR = SMEM_STAGE + STAGE_BYTES;
  static constexpr int BAR_WORDS = 3 + 2 * NSLOT + 2 * NH * SBUF + 5 * NH;  // mbarriers (8 bytes each)
  static constexpr int SMEM_TOTAL = SMEM_BAR + 512;
  static constexpr int TMEM_HEAD = SBUF * BN + D;  // S buffers, then O
  static constexpr int TMEM_USED = NH * TMEM_HEAD;
  static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : (TMEM_USED <= 256 ? 256 : 512);
  static constexpr int THREADS = 128 + 128 * NH;
  static_assert(NSLOT >= 2, "K and V slots");
  static_assert(!PAIR || (D == 256 && NH == 1) || (D == 128 && NH == 2), "CTA pairs: D = 256 x 1 or D = 128 x 2 heads");
  static_assert(BAR_WORDS * 8 + 8 + 4 * NH * SBUF <= 512, "barrier region");
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(SMEM_TOTAL + 1024 <= 232448, "SMEM budget");
};

struct FwdParams {
  const WorkItem* items;        // combined work list (all planned steps)
  const PlanHeader* hdr;
  const int32_t* cu;
  const int32_t* cu_pad;
  __nv_bfloat16* o;             // partial O of step s at o + s * o_slab (head-grouped THD)
  float* lse;                   // partial LSE of step s at lse + s * lse_slab
  int64_t o_slab, lse_slab;     // elements between consecutive steps' partials (0: one step)
  int32_t* status;
  int cp, hq, hkv, hpg_q, hpg_kv;
  int64_t T;
  float scale_log2;
  // 0: an item is one ring step of a query tile, written as that step's partial;
  // 1: an item is every ring step of a query tile's rank, a fresh online
  //    softmax per step and one partial (O_s, LSE_s) written per step;
  // 2: an item is every ring step in ONE online softmax (final O and LSE).
  int mode;
};

// The query rows of one work item.
struct ItemRows {
  int q_lo, q_hi;               // rows [q_lo, q_hi) are written (real tokens of the tile)
  int seq_start;
};

__device__ __forceinline__ ItemRows item_rows(const FwdParams& p, const WorkItem& it) {
  ItemRows ir;
  const int start = __ldg(p.cu_pad + it.b);
  const int S = __ldg(p.cu + it.b + 1) - __ldg(p.cu + it.b);
  const int L = (__ldg(p.cu_pad + it.b + 1) - start) / (2 * p.cp);
  ir.seq_start = start;
  ir.q_lo = it.c * L + it.tile * kBM;
  ir.q_hi = min(min(ir.q_lo + kBM, (it.c + 1) * L), S);
  return ir;
}

// KV tiles one work item attends, in ring order: for each ring step of the
// item (its own step, or every step of its rank in modes 1 and 2), the source
// rank's KV chunks the query chunk can see, ascending; tiles ascending.  On
// the diagonal chunk, keys past the item's last real row are skipped.
template <int BN>
struct KvTileIter {
  int cp, cq, r, L, S, q_hi, s, s_end, nv, vi, vis0, vis1, t, ntile, lo, hi;
  bool diag, done;

  __device__ void load_vis() {
    nv = visible_kv_chunks2(cq, ring_source(r, s, cp), cp, vis0, vis1);
  }
  __device__ void load_segment() {
    const int j = vi == 0 ? vis0 : vis1;
    diag = (j == cq);
    lo = j * L;
    hi = min((j + 1) * L, S);
    if (diag) hi = min(hi, q_hi);
    ntile = hi > lo ? (hi - lo + BN - 1) / BN : 0;
    t = 0;
  }
  __device__ void settle() {
    while (!done) {
      if (vi < nv && t < ntile) return;
      if (vi < nv) {
        ++vi;
        if (vi < nv) { load_segment(); continue; }
      }
      if (++s > s_end) { done = true; return; }
      load_vis();
      vi = 0;
      if (nv > 0) load_segment();
    }
  }
  __device__ void init(const FwdParams& p, const WorkItem& it, const ItemRows& ir) {
    cp = p.cp;
    cq = it.c;
    r = chunk_owner(cq, cp);
    const int start = ir.seq_start;
    S = __ldg(p.cu + it.b + 1) - __ldg(p.cu + it.b);
    L = (__ldg(p.cu_pad + it.b + 1) - start) / (2 * cp);
    q_hi = ir.q_hi;
    s = p.mode != 0 ? 0 : it.step;
    s_end = p.mode != 0 ? cp - 1 : it.step;
    done = q_hi <= ir.q_lo;
    vi = 0;
    t = 0;
    ntile = 0;
    load_vis();
    if (!done && nv > 0) load_segment();
    settle();
  }
  __device__ int k0() const { return lo + t * BN; }
  __device__ void next() {
    ++t;
    settle();
  }
};

// Tile j of an item opens a new online-softmax segment (fresh max, sum and
// O accumulator): the item's first tile, and with one partial per ring step
// the first tile of each later step.
__device__ __forceinline__ bool new_segment(int mode, int j, int step, int prev_step) {
  return j == 0 || (mode == 1 && step != prev_step);
}

template <int BN>
__device__ __forceinline__ int count_tiles(const FwdParams& p, const WorkItem& it, const ItemRows& ir) {
  KvTileIter<BN> c;
  c.init(p, it, ir);
  int n = 0;
  for (; !c.done; c.next()) ++n;
  return n;
}

// PAIR: launched as (2,1,1) clusters; the two CTAs of a cluster take 2 NH q
// heads of one kv group (heads 2 NH i + NH rank + h) of the same work item and
// run every product as one M = 256 tcgen05 product issued by rank 0 (head
// slot h of both CTAs), each CTA loading its half of every K and V tile
// (tm_k2: boxes of BN/2 key rows).
// tm_o (D = 256): the output (partials) as (D, heads of a group, rows, step
// slab), boxes of 64 columns x 128 rows, for the TMA stores of O.
template <int D, int NH, bool PAIR>
__global__ void __launch_bounds__(FwdCfg<D, NH, PAIR>::THREADS, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using Cfg = FwdCfg<D, NH, PAIR>;
  constexpr int BN = Cfg::BN, SBUF = Cfg::SBUF, NSLOT = Cfg::NSLOT, KCH = Cfg::KCH;

  // PAIR: work unit w = (item, 2 NH heads); this CTA's heads are
  // 2 NH (w % nhg) + NH rank + h
  const int nhg = p.hq / (PAIR ? 2 * NH : NH);         // work units per item
  const int64_t n_work = static_cast<int64_t>(p.hdr->n_fwd_all) * nhg;
  const int64_t w_first = PAIR ? blockIdx.x / 2 : blockIdx.x;
  const int64_t w_step = PAIR ? gridDim.x / 2 : gridDim.x;
  if (w_first >= n_work) return;                       // both CTAs of a pair, or neither
  // (a pair never returns on the status word: its two reads could differ)
  if (!PAIR && status_bad(p.status)) return;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  auto head_of = [&](int64_t w) {
    return PAIR ? static_cast<int>(w % nhg) * 2 * NH + static_cast<int>(rank) * NH : static_cast<int>(w % nhg) * NH;
  };

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::SMEM_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_free = bars + 1;                         // last S of the item done: Q may be reloaded
  uint64_t* kv_full = bars + 2;                        // [NSLOT]
  uint64_t* kv_empty = kv_full + NSLOT;                // [NSLOT]
  uint64_t* s_full = kv_empty + NSLOT;                 // [NH][SBUF]
  uint64_t* p_full = s_full + NH * SBUF;               // [NH][SBUF]
  // [NH][4]: P V product of tile t completes on o_done[h][t % 4].  A wait for
  // PV(t) is then unambiguous without consuming every phase: when S(t) is
  // complete, PV(t-3) is too (S is issued at most two tiles ahead of P V), so
  // the barrier's previous phase (PV(t-4)) has completed and PV(t+4) cannot
  // have been issued.  The softmax waits only when it must rescale O, and
  // once per segment before reading O out.
  uint64_t* o_done = p_full + NH * SBUF;
  uint64_t* o_free = o_done + NH * 4;                  // [NH]: a segment's O has been read out
  uint64_t* mma_done = o_free + NH;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // [NH][SBUF]: 1 when the P in that S buffer opens a softmax segment (its
  // P V starts a fresh O); written by the softmax before it arrives on
  // p_full, read by the MMA issuer after its wait on p_full.
  volatile int* seg_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(kv_full + s, 1);
      mbar_init(kv_empty + s, 1);
    }
    // P ready / O read out: every softmax thread of the CTA, or (pair) one
    // lane of each of the four softmax warps of both CTAs, on rank 0's barrier
    const uint32_t n_soft = PAIR ? 8 : 128;
    for (int i = 0; i < NH * SBUF; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, n_soft);
    }
    for (int h = 0; h < NH; ++h) {
      for (int i = 0; i < 4; ++i) mbar_init(o_done + h * 4 + i, 1);
      mbar_init(o_free + h, n_soft);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncwarp();
  // a pair: the other CTA's barriers are initialised before anything arrives on them
  if constexpr (PAIR) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(PAIR ? &tm_k2 : &tm_k);
      tma_prefetch_desc(&tm_v);
      int64_t n_loads = 0;                       // copies issued (slot = position % NSLOT)
      int q_loads = 0;
      bool ok = true;
      int64_t u = 0;                                   // K/V tile positions streamed by this CTA
      int item_k = 0;
      // a pair counts both CTAs' copies on rank 0's q_full / kv_full, which
      // rank 0 alone arms with the bytes of both halves
      const bool arm = !PAIR || rank == 0;
      constexpr uint32_t kArmQ = (PAIR ? 2 * NH : NH) * Cfg::Q_BYTES;
      constexpr uint32_t kArmKV = PAIR ? 2 * Cfg::SLOT_BYTES : Cfg::SLOT_BYTES;
      for (int64_t w = w_first; w < n_work && ok; w += w_step, ++item_k) {
        const WorkItem it = p.items[w / nhg];
        const int h0 = head_of(w);
        const int g = h0 / (p.hq / p.hkv);
        const ItemRows ir = item_rows(p, it);
        if (item_k > 0) ok = mbar_wait(q_free, (item_k - 1) & 1, abort_flag);
        if (!ok) break;
        const int qrow_base = ir.seq_start + ir.q_lo;
        if (arm) mbar_arrive_expect_tx(q_full, kArmQ);
        for (int h = 0; h < NH; ++h) {
          const int hq = h0 + h;
          const int row = static_cast<int>((hq / p.hpg_q) * p.T) + qrow_base;
          for (int kc = 0; kc < KCH; ++kc) {
            uint8_t* dst = smem + Cfg::SMEM_Q + h * Cfg::Q_BYTES + kc * kBM * 128;
            if constexpr (PAIR) tma_load_3d_pair(dst, &tm_q, kc * 64, hq % p.hpg_q, row, mapa_u32(q_full, 0));
            else tma_load_3d(dst, &tm_q, kc * 64, hq % p.hpg_q, row, q_full);
          }
        }
        ++q_loads;
        const int kv_group_row = static_cast<int>((g / p.hpg_kv) * p.T) + ir.seq_start;
        auto load = [&](int which, int k0) -> bool {         // which: 0 = K tile, 1 = V tile
          const int sl = static_cast<int>(u % NSLOT);
          if (u >= NSLOT && !mbar_wait(kv_empty + sl, static_cast<uint32_t>((u / NSLOT) - 1) & 1, abort_flag))
            return false;
          if (arm) mbar_arrive_expect_tx(kv_full + sl, kArmKV);
          uint8_t* dst = smem + Cfg::SMEM_KV + sl * Cfg::SLOT_BYTES;
          if constexpr (PAIR) {
            const uint32_t bar = mapa_u32(kv_full + sl, 0);
            if (which == 0) {
              // K: this CTA's BN/2 keys, every column
              for (int kc = 0; kc < KCH; ++kc)
                tma_load_3d_pair(dst + kc * Cfg::K_ROWS * 128, &tm_k2, kc * 64, g % p.hpg_kv,
                                 kv_group_row + k0 + static_cast<int>(rank) * Cfg::K_ROWS, bar);
            } else {
              // V: every key, this CTA's D/2 columns
              for (int kc = 0; kc < Cfg::V_CH; ++kc)
                tma_load_3d_pair(dst + kc * BN * 128, &tm_v, (static_cast<int>(rank) * Cfg::V_CH + kc) * 64,
                                 g % p.hpg_kv, kv_group_row + k0, bar);
            }
          } else {
            for (int kc = 0; kc < KCH; ++kc)
              tma_load_3d(dst + kc * BN * 128, which == 0 ? &tm_k : &tm_v, kc * 64, g % p.hpg_kv,
                          kv_group_row + k0, kv_full + sl);
          }
          ++n_loads;
          ++u;
          return true;
        };
        const int n = count_tiles<BN>(p, it, ir);
        KvTileIter<BN> ahead, cur;                      // K runs LA tiles ahead of V
        ahead.init(p, it, ir);
        cur.init(p, it, ir);
        for (int j = 0; j < min(Cfg::LA, n) && ok; ++j, ahead.next()) ok = load(0, ahead.k0());
        for (int j = 0; j < n && ok; ++j, cur.next()) {
          if (j + Cfg::LA < n) {
            ok = load(0, ahead.k0());
            ahead.next();
          }
          if (ok) ok = load(1, cur.k0());
        }
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // never leave a copy in flight into shared memory we are about to
      // release (a pair: rank 0's barriers count both CTAs' copies, and the
      // CTAs leave together)
      volatile int never = 0;
      if (arm) {
        if (q_loads > 0) mbar_wait(q_full, (q_loads - 1) & 1, &never, 200000000ull);
        wait_last_copies(kv_full, NSLOT, n_loads);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (a pair: rank 0 issues for both CTAs; M = 256, each CTA's TMEM gets its
    // 128 rows, and every completion is signalled in both CTAs).  The whole
    // warp runs this; one elected lane issues.
    if (rank == 0) {
      constexpr int MM = PAIR ? 2 * kBM : kBM;
      constexpr uint32_t idesc_s = idesc_bf16_f32(MM, BN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(MM, D, false, true);
      auto mma_ss = [](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (PAIR) umma_ss_pair(d, a, b, id, acc);
        else umma_ss(d, a, b, id, acc);
      };
      auto mma_ts = [](uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (PAIR) umma_ts_pair(d, a, b, id, acc);
        else umma_ts(d, a, b, id, acc);
      };
      auto commit = [](uint64_t* bar) {
        if constexpr (PAIR) umma_commit_pair_both(bar);
        else umma_commit(bar);
      };
      const uint32_t q_base = smem_u32(smem + Cfg::SMEM_Q);
      const uint32_t kv_base = smem_u32(smem + Cfg::SMEM_KV);
      // base descriptors in registers; head h / slot sl are constant offsets
      const uint64_t q_desc0 = smem_desc_sw128(q_base, 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(kv_base, 16, 1024);
      const uint64_t v_desc0 = smem_desc_sw128(kv_base, BN * 128, 1024);
      constexpr uint32_t kQStep = Cfg::Q_BYTES >> 4, kKVStep = Cfg::SLOT_BYTES >> 4;
      int64_t u = 0;     // K/V stream positions consumed (same order as the producer's)
      int64_t gs = 0;    // S tiles computed (S buffers, P and O barriers)
      bool ok = true;
      auto wait_pos = [&](int64_t pos) -> bool {
        const bool r = mbar_wait_warp(kv_full + (pos % NSLOT), static_cast<uint32_t>(pos / NSLOT) & 1, abort_flag);
        tc_fence_after();
        return r;
      };
      // S_h of the tile with global index t (K in slot sl) -> buffer t % SBUF
      auto issue_s = [&](int h, int64_t t, int sl) {
        const int buf = static_cast<int>(t % SBUF);
        const uint32_t d_tmem = tmem + h * Cfg::TMEM_HEAD + buf * BN;
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(d_tmem, q_desc0 + h * kQStep + kmajor_step(kBM, k),
                 k_desc0 + sl * kKVStep + kmajor_step(Cfg::K_ROWS, k), idesc_s, k > 0 ? 1u : 0u);
        commit(s_full + h * SBUF + buf);
      };
      auto issue_pv = [&](int h, int64_t t, int sl, bool first) {
        const int buf = static_cast<int>(t % SBUF);
        const uint32_t d_tmem = tmem + h * Cfg::TMEM_HEAD + SBUF * BN;
        const uint32_t p_tmem = tmem + h * Cfg::TMEM_HEAD + buf * BN;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ts(d_tmem, p_tmem + k * 8, v_desc0 + sl * kKVStep + mnmajor_step(k), idesc_o,
                 (!first || k > 0) ? 1u : 0u);
        commit(o_done + h * 4 + static_cast<int>(t % 4));
      };
      // all NH heads' S of tile t, K at the next stream position; then K is free
      auto issue_s_all = [&](int64_t t) -> bool {
        if (!wait_pos(u)) return false;
        const int sl = static_cast<int>(u % NSLOT);
        for (int h = 0; h < NH; ++h) issue_s(h, t, sl);
        commit(kv_empty + sl);
        ++u;
        return true;
      };
      int item_k = 0;
      int64_t segs = 0;  // softmax segments opened by this CTA (one O read-out each)
      for (int64_t w = w_first; w < n_work && ok; w += w_step, ++item_k) {
        const WorkItem it = p.items[w / nhg];
        const int n = count_tiles<BN>(p, it, item_rows(p, it));
        ok = mbar_wait_warp(q_full, item_k & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const int a = min(Cfg::LA, n);
        for (int j = 0; j < a && ok; ++j) ok = issue_s_all(gs + j);
        if (!ok) break;
        if (n <= Cfg::LA) commit(q_free);               // every S of the item issued
        for (int j = 0; j < n && ok; ++j) {
          const int64_t t = gs + j;
          const bool ahead = j + Cfg::LA < n;
          if (SBUF > 1 && ahead) {
            ok = issue_s_all(t + Cfg::LA);               // S LA tiles ahead of this P V
            if (!ok) break;
            if (j + Cfg::LA == n - 1) commit(q_free);
          }
          int64_t k_next = -1;                           // NH = 2: K of the next tile
          if (SBUF == 1 && ahead) {
            k_next = u++;
            ok = wait_pos(k_next);
            if (!ok) break;
          }
          const int64_t vpos = u++;                      // V_j
          ok = wait_pos(vpos);
          if (!ok) break;
          const int vsl = static_cast<int>(vpos % NSLOT);
          for (int h = 0; h < NH && ok; ++h) {
            const int buf = static_cast<int>(t % SBUF);
            ok = mbar_wait_warp(p_full + h * SBUF + buf, static_cast<uint32_t>(t / SBUF) & 1, abort_flag);
            if (!ok) break;
            const bool seg_start = p.mode == 1 ? seg_flag[h * SBUF + buf] != 0 : j == 0;
            if (h == 0 && seg_start) ++segs;
            if (seg_start && segs > 1) {
              // the previous segment's O must have been read out before it is overwritten
              ok = mbar_wait_warp(o_free + h, static_cast<uint32_t>(segs - 2) & 1, abort_flag);
              if (!ok) break;
            }
            tc_fence_after();
            issue_pv(h, t, vsl, seg_start);
            // one buffer per head: this head's next S goes right behind its P V,
            // while the other head's softmax keeps the tensor core busy
            if (SBUF == 1 && ahead) issue_s(h, t + 1, static_cast<int>(k_next % NSLOT));
          }
          if (!ok) break;
          commit(kv_empty + vsl);
          if (SBUF == 1 && ahead) {
            commit(kv_empty + static_cast<int>(k_next % NSLOT));
            if (j + 2 == n) commit(q_free);
          }
        }
        gs += n;
      }
      if (!ok) {
        raise_status(p.status, CCG_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      if constexpr (PAIR) umma_commit_pair_own(mma_done);
      else umma_commit(mma_done);
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
    int64_t gs = 0;
    bool ok = true;
    // P ready / O read out, to the MMA issuer (a pair: on rank 0's barrier,
    // one lane per warp once the whole warp's TMEM accesses are done)
    auto arrive_mma = [&](uint64_t* bar) {
      if constexpr (PAIR) {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_u32(bar, 0));
      } else {
        mbar_arrive(bar);
      }
    };
    for (int64_t w = w_first; w < n_work && ok; w += w_step) {
      const WorkItem it = p.items[w / nhg];
      const int h0 = head_of(w);
      const ItemRows ir = item_rows(p, it);
      KvTileIter<BN> kt_it;
      kt_it.init(p, it, ir);
      const int q_pos = ir.q_lo + row;
      const bool valid = q_pos < ir.q_hi;
      const int64_t orow = thd_row(ir.seq_start + q_pos, h0 + h, p.hpg_q, p.T);
      float m = -INFINITY, l = 0.f;
      int seg_step = -1;                                // ring step of the open segment
      // Closes a segment (running max mseg, sum lseg) once its last P V
      // product (tile t_last) has landed: reads O out of TMEM, releases it for
      // the next segment's first P V, and writes O / l and the LSE -- the
      // partial of ring step `step` (modes 0, 1) or the final output (mode 2).
      auto flush = [&](int64_t t_last, int step, float mseg, float lseg) -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait(o_done + h * 4 + static_cast<int>(t_last % 4),
                                               static_cast<uint32_t>(t_last / 4) & 1, abort_flag)))
          return false;
        tc_fence_after();
        const float inv_l = lseg > 0.f ? 1.f / lseg : 0.f;
        const int64_t slab = p.mode == 2 ? 0 : step;
        uint4* dst = reinterpret_cast<uint4*>(p.o + slab * p.o_slab + orow * D);
        if constexpr (Cfg::STAGE) {
          if (ir.q_hi - ir.q_lo == kBM) {
            // A whole tile: each 64-column quarter of O goes from TMEM through
            // this thread's row of a 16 KB box (128-byte swizzle: a warp's
            // 16-byte writes to 32 rows hit every bank) and leaves by one TMA
            // store issued by one thread; the two boxes alternate, so the
            // softmax threads never wait on global stores, only (rarely) on a
            // box's previous store having read it.
            const bool issuer = warp == 4 + 4 * h && lane == 0;
            uint8_t* sbox = smem + Cfg::SMEM_STAGE;
            const int grow = static_cast<int>(((h0 + h) / p.hpg_q) * p.T) + ir.seq_start + ir.q_lo;
            const int hc = (h0 + h) % p.hpg_q;
            const int slab_c = p.o_slab > 0 ? static_cast<int>(slab) : 0;   // one-slab outputs: slab 0
            const int swz = row & 7;
            // D=128: the row's whole O (128 columns) is loaded first and O
            // released at once, before the conversions and box writes
            uint32_t ro[D == 128 ? 4 : 1][32];
            if constexpr (D == 128) {
#pragma unroll
              for (int c = 0; c < 4; ++c) tmem_ld32(t_o + c * 32, ro[c]);
              tmem_wait_ld();
              tc_fence_before();
              arrive_mma(o_free + h);                   // O is free for the next segment's first P V
            }
#pragma unroll (D == 128 ? 2 : 1)
            for (int qq = 0; qq < D / 64; ++qq) {
              // D=256: two boxes, alternating; D=128: the head's own box
              uint8_t* box = sbox + (NH == 2 ? h : (qq & 1)) * Cfg::BOX_BYTES;
              if (issuer) {                             // the box's previous store has read it
                if constexpr (NH == 2) bulk_wait_group_read<0>();
                else bulk_wait_group_read<1>();
              }
              named_bar_sync(1 + h, 128);
              uint32_t r0[32], r1[32];
              if constexpr (D == 128) {
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                  r0[x] = ro[2 * qq][x];
                  r1[x] = ro[2 * qq + 1][x];
                }
              } else {
                tmem_ld32(t_o + qq * 64, r0);
                tmem_ld32(t_o + qq * 64 + 32, r1);
                tmem_wait_ld();
                if (qq == D / 64 - 1) {
                  tc_fence_before();
                  arrive_mma(o_free + h);               // O is free for the next segment's first P V
                }
              }
              uint4* brow = reinterpret_cast<uint4*>(box + row * 128);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const uint32_t* r = j < 4 ? r0 + 8 * j : r1 + 8 * (j - 4);
                uint4 w4;
                w4.x = pack_bf16x2(__uint_as_float(r[0]) * inv_l, __uint_as_float(r[1]) * inv_l);
                w4.y = pack_bf16x2(__uint_as_float(r[2]) * inv_l, __uint_as_float(r[3]) * inv_l);
                w4.z = pack_bf16x2(__uint_as_float(r[4]) * inv_l, __uint_as_float(r[5]) * inv_l);
                w4.w = pack_bf16x2(__uint_as_float(r[6]) * inv_l, __uint_as_float(r[7]) * inv_l);
                brow[j ^ swz] = w4;
              }
              fence_proxy_async_smem();
              named_bar_sync(1 + h, 128);
              if (issuer) {
                tma_store_4d(&tm_o, box, qq * 64, hc, grow, slab_c);
                bulk_commit_group();
              }
            }
            if (valid) p.lse[slab * p.lse_slab + orow] = (mseg + __log2f(lseg)) * kLn2;
            return true;
          }
          // (a partial tile, D=256) the staging area is free once the TMA
          // stores of earlier whole tiles have read it; D=128 partial tiles
          // take the plain row stores below
          if constexpr (D == 256) {
          if (warp == 4 && lane == 0) bulk_wait_group_read<0>();
          named_bar_sync(1, 128);
          // Each half of the row (128 columns) goes from TMEM to this thread's
          // own 256-byte staging row (16-byte slot k at k ^ (row & 15), so that
          // a warp's accesses hit every bank); each warp then stores its 32
          // rows from the staging area two whole 256-byte row halves per
          // instruction (coalesced).  O is free after the second half's TMEM
          // loads.
          uint4* stage = reinterpret_cast<uint4*>(smem + Cfg::SMEM_STAGE);
          uint4* srow = stage + row * 16;
          const int swz = row & 15;
          const int wrow0 = (warp & 3) * 32;
          const int u = lane & 15;
          __nv_bfloat16* obase = p.o + slab * p.o_slab;
          auto stage_half = [&](int c0) {
#pragma unroll
            for (int c = c0; c < c0 + D / 64; ++c) {
              uint32_t r[32];
              tmem_ld32(t_o + c * 32, r);
              tmem_wait_ld();
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                uint4 w4;
                w4.x = pack_bf16x2(__uint_as_float(r[8 * v4 + 0]) * inv_l, __uint_as_float(r[8 * v4 + 1]) * inv_l);
                w4.y = pack_bf16x2(__uint_as_float(r[8 * v4 + 2]) * inv_l, __uint_as_float(r[8 * v4 + 3]) * inv_l);
                w4.z = pack_bf16x2(__uint_as_float(r[8 * v4 + 4]) * inv_l, __uint_as_float(r[8 * v4 + 5]) * inv_l);
                w4.w = pack_bf16x2(__uint_as_float(r[8 * v4 + 6]) * inv_l, __uint_as_float(r[8 * v4 + 7]) * inv_l);
                srow[((c - c0) * 4 + v4) ^ swz] = w4;
              }
            }
            __syncwarp();
          };
          // lane l stores slot (l & 15) of row 2k + (l >> 4) of this warp's rows
          auto store_half = [&](int col0) {
#pragma unroll 2
            for (int k = 0; k < 16; ++k) {
              const int r = 2 * k + (lane >> 4);
              const int qp = ir.q_lo + wrow0 + r;
              const uint4 v = stage[(wrow0 + r) * 16 + (u ^ ((wrow0 + r) & 15))];
              if (qp < ir.q_hi) {
                const int64_t orr = thd_row(ir.seq_start + qp, h0 + h, p.hpg_q, p.T);
                reinterpret_cast<uint4*>(obase + orr * D + col0)[u] = v;
              }
            }
            __syncwarp();
          };
          stage_half(0);
          store_half(0);
          stage_half(D / 64);
          tc_fence_before();
          arrive_mma(o_free + h);
          store_half(D / 2);
          if (valid) p.lse[slab * p.lse_slab + orow] = (mseg + __log2f(lseg)) * kLn2;
          return true;
          }
        }
        uint32_t r[32];
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          tmem_ld32(t_o + c * 32, r);
          tmem_wait_ld();
          if (c == D / 32 - 1) {
            tc_fence_before();
            arrive_mma(o_free + h);
          }
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
        if (valid) p.lse[slab * p.lse_slab + orow] = (mseg + __log2f(lseg)) * kLn2;
        return true;
      };
      int n = 0;                                        // tiles of this item (counted as they go)
      // A segment that ends inside the item (its ring step is over) is read
      // out after the next segment's first P has been handed to the MMA warp,
      // so that the tensor core finishes the last P V meanwhile.
      bool pend = false;
      float pm = 0.f, pl = 0.f;
      int pstep = -1;
      for (int j = 0;; ++j) {
        const int64_t t = gs + j;
        const bool end = kt_it.done;
        if (end) {
          if (j > 0) {                                  // the item's last segment
            pend = true;
            pm = m;
            pl = l;
            pstep = seg_step;
          }
        } else {
          const bool seg_open = new_segment(p.mode, j, kt_it.s, seg_step);
          if (seg_open) {
            pend = j > 0;
            pm = m;
            pl = l;
            pstep = seg_step;
            m = -INFINITY;
            l = 0.f;
            seg_step = kt_it.s;
          }
          const int buf = static_cast<int>(t % SBUF);
          ok = __all_sync(0xffffffffu,
                          mbar_wait(s_full + h * SBUF + buf, static_cast<uint32_t>(t / SBUF) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          const int k0 = kt_it.k0();
          // keys visible to this row: k < kend (segment end, and k <= q_pos on the diagonal chunk)
          const int kend = kt_it.diag ? min(kt_it.hi, q_pos + 1) : kt_it.hi;
          const int nvalid = kend - k0;                     // may be <= 0 or >= BN
          const uint32_t t_s = t_head + buf * BN;
          // S row columns held in registers at once: the whole row when the
          // register budget allows (one TMEM round trip), else halves
          constexpr int HOLD = (NH == 1) ? BN : 64;
          uint32_t sr[HOLD];
          // Only tiles that cross a row's last visible key need a mask; there
          // the hidden scores are set to -inf in registers, so that the max
          // ignores them and their probabilities come out exactly 0.
          const bool masked = __any_sync(0xffffffffu, nvalid < BN);
          auto load_s = [&](int g0) {
#pragma unroll
            for (int c = 0; c < HOLD / 32; ++c)
              tmem_ld32(t_s + g0 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + c * 32));
            tmem_wait_ld();
            if (masked) {
#pragma unroll
              for (int x = 0; x < HOLD; ++x) sr[x] = (g0 + x < nvalid) ? sr[x] : 0xff800000u;
            }
          };
          // max of the raw scores, scaled once (the scale is positive, and a
          // correctly rounded product preserves order)
          // four independent running maxima: a single chain of dependent
          // max instructions would be latency-bound with one or two warps
          // per SM sub-partition
          float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int g0 = 0; g0 < BN; g0 += HOLD) {
            load_s(g0);
#pragma unroll
            for (int x = 0; x < HOLD; x += 2)
              mq[(x >> 1) & 3] = fmax3(mq[(x >> 1) & 3], __uint_as_float(sr[x]), __uint_as_float(sr[x + 1]));
          }
          const float mxr = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
          const float mx = mxr * p.scale_log2;
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
          // p = 2^(s * scale_log2 - m), two columns per packed FMA
          const uint64_t scale2 = f32x2(p.scale_log2, p.scale_log2);
          const uint64_t negm2 = f32x2(-m_use, -m_use);
          uint64_t psum2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};   // two independent sum chains
#pragma unroll
          for (int g0 = 0; g0 < BN; g0 += HOLD) {
            if (HOLD < BN) load_s(g0);
#pragma unroll
            for (int c = 0; c < HOLD / 32; ++c) {
              uint32_t pk[16];
#pragma unroll
              for (int x = 0; x < 16; ++x) {
                const int cl = c * 32 + 2 * x;
                float a0, a1;
                f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[cl]), __uint_as_float(sr[cl + 1])), scale2, negm2), a0,
                            a1);
                const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
                psum2[x & 1] = add_f32x2(psum2[x & 1], f32x2(p0, p1));
                pk[x] = pack_bf16x2(p0, p1);
              }
              tmem_st16(t_s + (g0 + c * 32) / 2, pk);
            }
          }
          tmem_wait_st();
          float ps0, ps1;
          f32x2_split(add_f32x2(psum2[0], psum2[1]), ps0, ps1);
          l = l * alpha + (ps0 + ps1);
          // rescale the running O (rare: the reference max grew past the
          // threshold) once the previous P V product has landed
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            const int64_t tp1 = t - 1;                     // alpha != 1: not a segment's first tile
            ok = __all_sync(0xffffffffu, mbar_wait(o_done + h * 4 + static_cast<int>(tp1 % 4),
                                                   static_cast<uint32_t>(tp1 / 4) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            uint32_t r[32];
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
          if (row == 0) seg_flag[h * SBUF + buf] = seg_open ? 1 : 0;
          tc_fence_before();
          arrive_mma(p_full + h * SBUF + buf);
        }
        if (pend) {
          pend = false;
          ok = flush(t - 1, pstep, pm, pl);              // the segment ended with tile t - 1
          if (!ok) break;
        }
        if (end) {
          n = j;
          break;
        }
        kt_it.next();
      }
      if (!ok) break;
      gs += n;
    }
    if (!ok) {
      raise_status(p.status, CCG_ERR_TIMEOUT);
      *abort_flag = 1;
    }
    // the TMA stores of O have read their boxes and written global memory
    if (Cfg::STAGE && (warp & 3) == 0 && lane == 0) bulk_wait_group<0>();
  }
  tc_fence_before();
  __syncwarp();
  // a pair: neither CTA leaves (nor frees TMEM) while the other may still
  // touch its shared memory or TMEM; rank 0's MMA thread has seen every
  // product complete before it arrives
  if constexpr (PAIR) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  if (warp == 2) {
    if constexpr (PAIR) tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
    else tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

template <int D, int NH, bool PAIR>
cudaError_t launch_fwd_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tk2,
                            const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& p, int grid,
                            cudaStream_t stream) {
  using Cfg = FwdCfg<D, NH, PAIR>;
  auto kern = attn_fwd_kernel<D, NH, PAIR>;
  static std::atomic<uint64_t> attr_done{0};
  const int smem = Cfg::SMEM_TOTAL + 1024;
  cudaError_t e = once_per_device(
      attr_done, [&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
  if (e != cudaSuccess) return e;
  if constexpr (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // persistent: as many pairs as can be resident at once (not every SM
    // need belong to a usable pair)
    static std::atomic<uint64_t> pairs_done{0};
    static int max_pairs[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = once_per_device(pairs_done, [&] {
      cfg.gridDim = dim3(static_cast<unsigned>(grid / 2 * 2));
      int n = 0;
      const cudaError_t r = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (dev < 64) max_pairs[dev] = n;
      return r;
    });
    if (e != cudaSuccess) return e;
    const int pairs = min(grid / 2, dev < 64 && max_pairs[dev] > 0 ? max_pairs[dev] : grid / 2);
    if (pairs < 1) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tk2, tv, to, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  } else {
    kern<<<grid, Cfg::THREADS, smem, stream>>>(tq, tk, tk2, tv, to, p);
    return cudaGetLastError();
  }
}

}  // namespace

int fwd_heads_per_cta(int D, int group) { return (D == 128 && group % 2 == 0) ? 2 : 1; }

// CTA pairs sharing every K/V tile load (each CTA loads half of it): D = 256
// with an even q-head group (two heads a pair), D = 128 with a group of a
// multiple of 4 (four heads a pair, two a CTA)
bool fwd_uses_pairs(int D, int group) { return (D == 256 && group % 2 == 0) || (D == 128 && group % 4 == 0); }

// Persistent launch over the combined work list: one CTA per SM (the work
// count is only known on the device; CTAs with nothing to do exit at once).
cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tk2,
                            const CUtensorMap& tv, const CUtensorMap& to, const WorkItem* items, const PlanHeader* hdr, const int32_t* cu,
                            const int32_t* cu_pad, void* o, float* lse, int64_t o_slab, int64_t lse_slab,
                            int32_t* status, int cp, int hq, int hkv, int head_groups, int64_t T, int D,
                            float scale, int mode, int num_sms, cudaStream_t stream) {
  FwdParams p;
  p.mode = mode;
  p.items = items;
  p.hdr = hdr;
  p.cu = cu;
  p.cu_pad = cu_pad;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.o_slab = o_slab;
  p.lse_slab = lse_slab;
  p.status = status;
  p.cp = cp;
  p.hq = hq;
  p.hkv = hkv;
  p.hpg_q = hq / head_groups;
  p.hpg_kv = hkv / head_groups;
  p.T = T;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int nh = fwd_heads_per_cta(D, hq / hkv);
  if (D == 128 && nh == 2 && fwd_uses_pairs(D, hq / hkv))
    return launch_fwd_impl<128, 2, true>(tq, tk, tk2, tv, to, p, num_sms, stream);
  if (D == 128 && nh == 2) return launch_fwd_impl<128, 2, false>(tq, tk, tk, tv, to, p, num_sms, stream);
  if (D == 128) return launch_fwd_impl<128, 1, false>(tq, tk, tk, tv, to, p, num_sms, stream);
  if (D == 256 && fwd_uses_pairs(D, hq / hkv))
    return launch_fwd_impl<256, 1, true>(tq, tk, tk2, tv, to, p, num_sms, stream);
  if (D == 256) return launch_fwd_impl<256, 1, false>(tq, tk, tk, tv, to, p, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ccg
