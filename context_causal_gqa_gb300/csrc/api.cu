// api.cu -- host side of the C ABI declared in include/ccg.h: argument
// validation (fail-closed), workspace layout, TMA tensor maps and the
// launch sequence of each entry point.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace ccg {


cudaError_t launch_plan(const int32_t* cu, const int32_t* cu_pad, int B, int64_t T, int cp, int hkv, int bm,
                        int bn, int cap_q, int cap_kv, int want, int step_only, PlanHeader* hdr,
                        WorkItem* fwd_items, WorkItem* dq_items, WorkItem* kv_items,
                        int32_t* status, cudaStream_t stream, int64_t max_pad = 0, int64_t* ds_base = nullptr);
cudaError_t launch_chunk_table(const int32_t* cu, const int32_t* cu_pad, int B, int64_t T, int cp,
                               int32_t* table, int32_t* status, cudaStream_t stream);
cudaError_t launch_bwd_dot(const void* o, const void* dout, int64_t rows, int D, int dout_heads,
                           int64_t dout_pitch, float* delta,
                           const int32_t* status, int num_sms, cudaStream_t stream);
cudaError_t launch_thd_permute(bool pack, const void* src, void* dst, const int32_t* cu_pad, int B,
                               int64_t T, int H, int D, int cp, int32_t* status, int num_sms,
                               cudaStream_t stream);
cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tk2,
                            const CUtensorMap& tv, const CUtensorMap& to, const WorkItem* items, const PlanHeader* hdr, const int32_t* cu,
                            const int32_t* cu_pad, void* o, float* lse, int64_t o_slab, int64_t lse_slab,
                            int32_t* status, int cp, int hq, int hkv, int head_groups, int64_t T, int D,
                            float scale, int mode, int num_sms, cudaStream_t stream);
cudaError_t launch_pad_rows(void* o, float* lse, const int32_t* cu, const int32_t* cu_pad, int B, int64_t T,
                            int H, int hpg, int D, const int32_t* status, int num_sms, cudaStream_t stream);
cudaError_t launch_attn_bwd(const CUtensorMap* maps, const WorkItem* dq_items,
                            const WorkItem* kv_items, const PlanHeader* hdr, const int32_t* cu,
                            const int32_t* cu_pad, const float* lse, const float* delta, void* dq,
                            void* dk, void* dv, int32_t* status, int cp, int hq, int hkv,
                            int head_groups, int64_t T, int D, float scale, int grid_q,
                            int grid_kv, int* launches, cudaStream_t stream, void* ds = nullptr,
                            const int64_t* ds_base = nullptr, int64_t ds_cap = 0,
                            const CUtensorMap* ds_map = nullptr, int kv_pairs = 0);
int bwd_kv_tile_rows(int D);
int bwd_q_tile_rows(int D);
int bwd_map_rows(int which, int D);

cudaError_t launch_lse_merge(const MergeArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_bounded_wait_selftest(int32_t* status, uint32_t limit_us, cudaStream_t stream);

}  // namespace ccg

namespace {

struct ProfState {
  bool on = false;
  std::vector<cudaEvent_t> ev;       // 2 per launch
  std::vector<const char*> names;
  int n = 0;
};
thread_local ProfState g_prof;

}  // namespace

namespace ccg {

void prof_begin(const char* kernel_name, cudaStream_t stream) {
  ProfState& p = g_prof;
  if (!p.on || 2 * (p.n + 1) > static_cast<int>(p.ev.size())) return;
  p.names[p.n] = kernel_name;
  cudaEventRecord(p.ev[2 * p.n], stream);
}

void prof_end(cudaStream_t stream) {
  ProfState& p = g_prof;
  if (!p.on || 2 * (p.n + 1) > static_cast<int>(p.ev.size())) return;
  cudaEventRecord(p.ev[2 * p.n + 1], stream);
  ++p.n;
}

}  // namespace ccg

namespace {

using namespace ccg;

thread_local int32_t g_last_launches = 0;

constexpr int kQTile = 128;          // query-tile rows of the forward and dQ pass
constexpr int kMinKvTile = 64;       // smallest KV-tile rows of any pass (plan capacity)

int num_sms_cached() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t ds_cap_tiles(const ccg_attn_desc* d);

ccg_status check_desc(const ccg_attn_desc* d) {
  if (d == nullptr) return CCG_ERR_INVALID_ARG;
  if (d->batch < 1 || d->hq < 1 || d->hkv < 1 || d->total_tokens < 0 || d->head_parts < 0 || d->max_seqlen < 0)
    return CCG_ERR_INVALID_ARG;
  if (d->causal != 1) return CCG_ERR_UNSUPPORTED;
  if (d->head_dim != 128 && d->head_dim != 256) return CCG_ERR_UNSUPPORTED;
  if (d->hq % d->hkv != 0) return CCG_ERR_UNSUPPORTED;
  if (d->cp < 1 || d->cp > kMaxCP) return CCG_ERR_UNSUPPORTED;
  if (d->head_groups < 1) return CCG_ERR_INVALID_ARG;
  if (d->hq % d->head_groups != 0 || d->hkv % d->head_groups != 0) return CCG_ERR_UNSUPPORTED;
  // head partitioning: whole GQA groups per part, and in the head-split
  // layout whole head groups (a part is then one contiguous sub-tensor)
  if (d->head_parts > 1) {
    if (d->hkv % d->head_parts != 0) return CCG_ERR_UNSUPPORTED;
    if (d->head_groups > 1 && d->head_groups % d->head_parts != 0) return CCG_ERR_UNSUPPORTED;
  }
  if (d->total_tokens % (2 * d->cp) != 0) return CCG_ERR_UNSUPPORTED;
  // 32-bit coordinates inside the kernels and TMA maps
  if (d->total_tokens * d->head_groups >= (int64_t(1) << 31)) return CCG_ERR_UNSUPPORTED;
  if (d->batch > (1 << 20)) return CCG_ERR_UNSUPPORTED;
  // dK/dV work items (one per KV tile and kv head) are indexed with 32 bits
  if ((d->total_tokens / 64 + int64_t(d->batch) * 2 * d->cp + 1) * d->hkv >= (int64_t(1) << 31))
    return CCG_ERR_UNSUPPORTED;
  const int64_t pitches[4] = {d->q_pitch, d->k_pitch, d->v_pitch, d->do_pitch};
  const int64_t dense[4] = {int64_t(d->hq) * d->head_dim, int64_t(d->hkv) * d->head_dim,
                            int64_t(d->hkv) * d->head_dim, int64_t(d->hq) * d->head_dim};
  for (int i = 0; i < 4; ++i) {
    if (pitches[i] == 0) continue;
    if (pitches[i] < dense[i]) return CCG_ERR_INVALID_ARG;
    if (pitches[i] % 8 != 0) return CCG_ERR_ALIGNMENT;     // TMA row strides are multiples of 16 bytes
    if (d->head_groups != 1) return CCG_ERR_UNSUPPORTED;
    if (pitches[i] >= (int64_t(1) << 36)) return CCG_ERR_UNSUPPORTED;
  }
  // the dS backward addresses its dS and P tiles with 32-bit TMA coordinates
  if (2 * ds_cap_tiles(d) * (d->hq / d->hkv) >= (int64_t(1) << 31)) return CCG_ERR_UNSUPPORTED;
  return CCG_OK;
}

// Row pitch (elements) of input `which` (0 q, 1 k, 2 v, 3 dO) in its
// head-grouped layout: the caller's pitch, or dense H/G_h * D.
int64_t input_pitch(const ccg_attn_desc* d, int which) {
  const int64_t p[4] = {d->q_pitch, d->k_pitch, d->v_pitch, d->do_pitch};
  const int h = (which == 1 || which == 2) ? d->hkv : d->hq;
  return p[which] != 0 ? p[which] : int64_t(h / d->head_groups) * d->head_dim;
}

float softmax_scale(const ccg_attn_desc* d) {
  return d->softmax_scale > 0.f ? d->softmax_scale : 1.0f / std::sqrt(static_cast<float>(d->head_dim));
}

int head_parts_of(const ccg_attn_desc* d) { return d->head_parts > 1 ? d->head_parts : 1; }

struct Layout {
  size_t hdr, fwd_items, dq_items, kv_items, o_parts, lse_parts, delta, ds_base, ds, total;
  int cap_q, cap_kv;
  int64_t ds_cap_tiles;     // dS tiles of one q head the dS region holds (0: no dS backward)
};

// The backward that keeps dS (a padded-length bound in the descriptor): one
// 128 x 128 BF16 dS tile per (query tile, visible KV tile) of each q head of
// one GQA group (and at D = 256 a P tile each as well).  Per sequence and head the tiles number
// t^2 * 2CP(2CP+1)/2 (t = 128-row tiles of a chunk), and
// sum_b t_b^2 <= t_max * sum_b t_b <= t_max * (T / (128 * 2CP) + B).
bool bwd_keeps_ds(const ccg_attn_desc* d) { return d->max_seqlen > 0; }
// dS tiles, then (D = 256) P tiles
int64_t ds_planes(const ccg_attn_desc* d) { return d->head_dim == 256 ? 2 : 1; }
int64_t ds_cap_tiles(const ccg_attn_desc* d) {
  if (!bwd_keeps_ds(d)) return 0;
  const int64_t C = 2 * d->cp;
  const int64_t t_max = (d->max_seqlen / C + 127) / 128;
  const int64_t sum_t = d->total_tokens / (128 * C) + d->batch;
  return t_max * sum_t * (C * (C + 1) / 2);
}
constexpr int64_t kDsTileBytes = 128 * 128 * 2;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// kind: 0 forward (plan + CP partials), 1 backward (plan + Delta), 2 fused
// forward (plan only).
Layout workspace_layout(const ccg_attn_desc* d, int kind) {
  const int is_bwd = kind == 1;
  const bool partials = kind == 0;
  Layout L{};
  const int64_t C = 2 * d->cp;
  L.cap_q = static_cast<int>(d->total_tokens / kQTile + d->batch * C + 1);
  L.cap_kv = static_cast<int>(d->total_tokens / kMinKvTile + d->batch * C + 1);
  size_t off = 0;
  L.hdr = off;
  off += kPlanHeaderBytes;
  L.fwd_items = off;
  off = align_up(off + (is_bwd ? 0 : size_t(d->cp) * L.cap_q * sizeof(WorkItem)), 256);
  L.dq_items = off;
  off = align_up(off + (is_bwd ? size_t(L.cap_q) * sizeof(WorkItem) : 0), 256);
  L.kv_items = off;
  off = align_up(off + (is_bwd ? size_t(L.cap_kv) * d->hkv * sizeof(WorkItem) : 0), 256);
  // dS backward: per-sequence first tile of the dS region, then the region
  // (one GQA group's q heads)
  L.ds_cap_tiles = is_bwd ? ds_cap_tiles(d) : 0;
  L.ds_base = off;
  off = align_up(off + (L.ds_cap_tiles > 0 ? size_t(d->batch + 1) * sizeof(int64_t) : 0), 256);
  L.ds = off;
  off = align_up(off + ds_planes(d) * size_t(L.ds_cap_tiles) * (d->hq / d->hkv) * kDsTileBytes, 256);
  // the partial slabs hold one head part (all heads without partitioning)
  const size_t rows = size_t(d->total_tokens) * d->hq / head_parts_of(d);
  L.o_parts = off;
  off = align_up(off + (partials ? size_t(d->cp) * rows * d->head_dim * 2 : 0), 256);
  L.lse_parts = off;
  off = align_up(off + (partials ? size_t(d->cp) * rows * 4 : 0), 256);
  L.delta = off;
  off = align_up(off + (is_bwd ? size_t(d->total_tokens) * d->hq * 4 : 0), 256);
  L.total = off;
  return L;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so that
// the library has no link-time dependency on the driver library.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over a head-grouped THD tensor: dims (D, H/G_h, G_h*T), heads D
// elements apart, rows `pitch` elements apart (dense: H/G_h * D), 128-byte
// swizzled boxes of 64 columns x 1 head x `box_rows` rows.
bool make_thd_map(CUtensorMap* m, const void* base, int D, int hpg, int64_t rows, int box_rows, int64_t pitch) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(hpg),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(pitch) * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over an output in the head-grouped THD layout, `nslab` copies of it
// `slab` elements apart (the ring steps' partials): dims (D, H/G_h, G_h*T,
// nslab), rows H/G_h * D elements apart, 128-byte swizzled boxes of 64
// columns x 1 head x 128 rows x 1 slab, for TMA stores.
bool make_out_map(CUtensorMap* m, void* base, int D, int hpg, int64_t rows, int nslab, int64_t slab) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const int64_t pitch = static_cast<int64_t>(hpg) * D;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(hpg), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(nslab)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(pitch) * 2,
                           static_cast<cuuint64_t>(nslab > 1 ? slab : rows * pitch) * 2};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the dS and P tiles of the dS backward: dims (128 columns,
// 128 rows, ntiles), unswizzled boxes of one whole 32 KB tile (its bytes in
// order).  A load at tile -1 lies wholly outside and reads zeros.
bool make_tile_map(CUtensorMap* m, void* base, int64_t ntiles) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {128, 128, static_cast<cuuint64_t>(ntiles)};
  cuuint64_t strides[2] = {128 * 2, 128 * 128 * 2};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#define CCG_LAUNCH(name, stream, expr)       \
  do {                                       \
    prof_begin(name, stream);                \
    const cudaError_t e_ = (expr);           \
    prof_end(stream);                        \
    if (e_ != cudaSuccess) return CCG_ERR_CUDA; \
    ++launches;                              \
  } while (0)

ccg_status fwd_prepare(const ccg_attn_desc* d, const void* q, const void* k, const void* v,
                       const int32_t* cu, const int32_t* cu_pad, void* workspace, size_t ws_bytes,
                       int32_t* status, Layout* L, int kind = 0) {
  ccg_status st = check_desc(d);
  if (st != CCG_OK) return st;
  if (!q || !k || !v || !cu || !cu_pad || !status) return CCG_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return CCG_ERR_ALIGNMENT;
  *L = workspace_layout(d, kind);
  if (workspace == nullptr || ws_bytes < L->total) return CCG_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CCG_ERR_ALIGNMENT;
  return CCG_OK;
}

}  // namespace

extern "C" {

size_t ccg_workspace_size(const ccg_attn_desc* desc, int kind) {
  if (check_desc(desc) != CCG_OK) return 0;
  if (kind < 0 || kind > 2) return 0;
  return workspace_layout(desc, kind).total;
}

const char* ccg_status_str(ccg_status s) {
  switch (s) {
    case CCG_OK: return "ok";
    case CCG_ERR_INVALID_ARG: return "invalid argument";
    case CCG_ERR_UNSUPPORTED: return "unsupported problem (shape, head dim, CP size or layout)";
    case CCG_ERR_ALIGNMENT: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case CCG_ERR_WORKSPACE: return "workspace missing or too small";
    case CCG_ERR_SEQLENS: return "sequence lengths / padded offsets break the promise";
    case CCG_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case CCG_ERR_CUDA: return "CUDA runtime or driver call failed";
  }
  return "unknown status";
}

int32_t ccg_last_launch_count(void) { return g_last_launches; }

ccg_status ccg_profile_begin(int32_t capacity) {
  ProfState& p = g_prof;
  if (capacity < 1) return CCG_ERR_INVALID_ARG;
  for (cudaEvent_t e : p.ev) cudaEventDestroy(e);
  p.ev.assign(2 * static_cast<size_t>(capacity), nullptr);
  p.names.assign(capacity, nullptr);
  for (auto& e : p.ev)
    if (cudaEventCreate(&e) != cudaSuccess) {
      p.ev.clear();
      p.on = false;
      return CCG_ERR_CUDA;
    }
  p.n = 0;
  p.on = true;
  return CCG_OK;
}

ccg_status ccg_profile_end(void) {
  g_prof.on = false;
  return CCG_OK;
}

int32_t ccg_profile_count(void) { return g_prof.n; }

ccg_status ccg_profile_get(int32_t i, const char** kernel_name, float* ms) {
  ProfState& p = g_prof;
  if (i < 0 || i >= p.n || !kernel_name || !ms) return CCG_ERR_INVALID_ARG;
  if (cudaEventSynchronize(p.ev[2 * i + 1]) != cudaSuccess) return CCG_ERR_CUDA;
  if (cudaEventElapsedTime(ms, p.ev[2 * i], p.ev[2 * i + 1]) != cudaSuccess) return CCG_ERR_CUDA;
  *kernel_name = p.names[i];
  return CCG_OK;
}

ccg_status ccg_selftest_bounded_wait(int32_t* d_status, uint32_t limit_us, ccg_stream_t stream) {
  int launches = 0;
  g_last_launches = 0;
  if (d_status == nullptr) return CCG_ERR_INVALID_ARG;
  if (limit_us < 1 || limit_us > 1000000) return CCG_ERR_INVALID_ARG;
  CCG_LAUNCH("selftest_bounded_wait", reinterpret_cast<cudaStream_t>(stream),
             launch_bounded_wait_selftest(d_status, limit_us, reinterpret_cast<cudaStream_t>(stream)));
  g_last_launches = launches;
  return CCG_OK;
}

ccg_status ccg_get_status(const int32_t* d_status, ccg_stream_t stream) {
  if (d_status == nullptr) return CCG_ERR_INVALID_ARG;
  int32_t h = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&h, d_status, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CCG_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CCG_ERR_CUDA;
  return static_cast<ccg_status>(h);
}

ccg_status ccg_cp_split(const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, int32_t batch,
                        int64_t total_tokens, int32_t cp, int32_t* chunk_table, int32_t* d_status,
                        ccg_stream_t stream) {
  int launches = 0;
  g_last_launches = 0;
  if (!cu_seqlens || !cu_seqlens_padded || !chunk_table || !d_status) return CCG_ERR_INVALID_ARG;
  if (batch < 1 || total_tokens < 0) return CCG_ERR_INVALID_ARG;
  if (cp < 1 || cp > kMaxCP) return CCG_ERR_UNSUPPORTED;
  CCG_LAUNCH("cp_split", reinterpret_cast<cudaStream_t>(stream),
             launch_chunk_table(cu_seqlens, cu_seqlens_padded, batch, total_tokens, cp, chunk_table, d_status,
                                reinterpret_cast<cudaStream_t>(stream)));
  g_last_launches = launches;
  return CCG_OK;
}

ccg_status ccg_cp_lse_merge(int32_t nparts, const void* const* o_parts, const float* const* lse_parts,
                            int64_t rows, int32_t head_dim, void* o, float* lse, ccg_stream_t stream) {
  int launches = 0;
  g_last_launches = 0;
  if (nparts < 1 || nparts > kMaxCP || rows < 0 || !o_parts || !lse_parts || !o || !lse)
    return CCG_ERR_INVALID_ARG;
  if (head_dim != 128 && head_dim != 256) return CCG_ERR_UNSUPPORTED;
  MergeArgs a{};
  for (int s = 0; s < nparts; ++s) {
    if (!o_parts[s] || !lse_parts[s]) return CCG_ERR_INVALID_ARG;
    if (!aligned16(o_parts[s])) return CCG_ERR_ALIGNMENT;
    a.o_parts[s] = o_parts[s];
    a.lse_parts[s] = lse_parts[s];
  }
  if (!aligned16(o)) return CCG_ERR_ALIGNMENT;
  if (rows == 0) return CCG_OK;
  a.nparts = nparts;
  a.o = o;
  a.lse = lse;
  a.rows = rows;
  a.D = head_dim;
  a.status = nullptr;
  CCG_LAUNCH("lse_merge", reinterpret_cast<cudaStream_t>(stream),
             launch_lse_merge(a, num_sms_cached(), reinterpret_cast<cudaStream_t>(stream)));
  g_last_launches = launches;
  return CCG_OK;
}

ccg_status ccg_bwd_dot(const void* o, const void* dout, int64_t rows, int32_t head_dim, float* delta,
                       ccg_stream_t stream) {
  int launches = 0;
  g_last_launches = 0;
  if (!o || !dout || !delta || rows < 0) return CCG_ERR_INVALID_ARG;
  if (head_dim != 128 && head_dim != 256) return CCG_ERR_UNSUPPORTED;
  if (!aligned16(o) || !aligned16(dout)) return CCG_ERR_ALIGNMENT;
  if (rows == 0) return CCG_OK;
  CCG_LAUNCH("bwd_dot", reinterpret_cast<cudaStream_t>(stream),
             launch_bwd_dot(o, dout, rows, head_dim, 1, head_dim, delta, nullptr, num_sms_cached(),
                            reinterpret_cast<cudaStream_t>(stream)));
  g_last_launches = launches;
  return CCG_OK;
}

static ccg_status thd_permute(bool pack, const void* src, const int32_t* cu_pad, int32_t batch,
                              int64_t T, int32_t heads, int32_t head_dim, int32_t cp, void* dst,
                              int32_t* d_status, ccg_stream_t stream) {
  int launches = 0;
  g_last_launches = 0;
  if (!src || !dst || !cu_pad || !d_status || batch < 1 || T < 0 || heads < 1 || head_dim < 1)
    return CCG_ERR_INVALID_ARG;
  if (cp < 1 || cp > kMaxCP || heads % cp != 0 || T % (2 * cp) != 0) return CCG_ERR_UNSUPPORTED;
  if ((static_cast<int64_t>(heads / cp) * head_dim) % 8 != 0) return CCG_ERR_UNSUPPORTED;
  if (!aligned16(src) || !aligned16(dst)) return CCG_ERR_ALIGNMENT;
  if (T == 0) return CCG_OK;
  CCG_LAUNCH(pack ? "thd_pack" : "thd_unpack", reinterpret_cast<cudaStream_t>(stream),
             launch_thd_permute(pack, src, dst, cu_pad, batch, T, heads, head_dim, cp, d_status,
                                num_sms_cached(), reinterpret_cast<cudaStream_t>(stream)));
  g_last_launches = launches;
  return CCG_OK;
}

ccg_status ccg_thd_pack(const void* x_rank_major, const int32_t* cu_seqlens_padded, int32_t batch,
                        int64_t total_tokens, int32_t heads, int32_t head_dim, int32_t cp,
                        void* out_head_split, int32_t* d_status, ccg_stream_t stream) {
  return thd_permute(true, x_rank_major, cu_seqlens_padded, batch, total_tokens, heads, head_dim, cp,
                     out_head_split, d_status, stream);
}

ccg_status ccg_thd_unpack(const void* in_head_split, const int32_t* cu_seqlens_padded, int32_t batch,
                          int64_t total_tokens, int32_t heads, int32_t head_dim, int32_t cp,
                          void* x_rank_major, int32_t* d_status, ccg_stream_t stream) {
  return thd_permute(false, in_head_split, cu_seqlens_padded, batch, total_tokens, heads, head_dim, cp,
                     x_rank_major, d_status, stream);
}

// Plans and launches the forward attention kernel.  mode 0: the partial of
// ring step `step_only` into o_part / lse_part; mode 1: the partials of every
// ring step into consecutive slabs of o_part / lse_part (one item per query
// tile walks all steps of its rank); mode 2: every ring step in one online
// softmax, the final O and LSE into o_part / lse_part.
// Tensor maps and the launch of the forward attention kernel over the plan
// already in the workspace.  mode 0: the partial of one ring step into
// o_part / lse_part; mode 1: the partials of every ring step into
// consecutive slabs of o_part / lse_part (one item per query tile walks all
// steps of its rank); mode 2: every ring step in one online softmax, the
// final O and LSE into o_part / lse_part.
static ccg_status fwd_attention(const ccg_attn_desc* d, const void* q, const void* k, const void* v,
                                const int32_t* cu, const int32_t* cu_pad, void* o_part, int64_t o_slab,
                                float* lse_part, int64_t lse_slab, void* workspace, const Layout& L,
                                int32_t* status, cudaStream_t s, int* launches_out, int mode) {
  int launches = *launches_out;
  auto* base = static_cast<uint8_t*>(workspace);
  auto* hdr = reinterpret_cast<PlanHeader*>(base + L.hdr);
  auto* items = reinterpret_cast<WorkItem*>(base + L.fwd_items);
  const int hg = d->head_groups;
  const int64_t rows = d->total_tokens * hg;
  const int bn = 128;                                   // forward K/V tile rows
  CUtensorMap tq, tk, tk2, tv, to;
  // tk2: half-tile boxes (bn/2 key rows), for the CTA pairs of the D = 256
  // kernel; to: the output (the steps' partials, o_slab apart), for its TMA
  // stores of O (mode 0 and 2: one slab)
  const int nslab = o_slab > 0 ? d->cp : 1;
  if (!make_thd_map(&tq, q, d->head_dim, d->hq / hg, rows, kQTile, input_pitch(d, 0)) ||
      !make_thd_map(&tk, k, d->head_dim, d->hkv / hg, rows, bn, input_pitch(d, 1)) ||
      !make_thd_map(&tk2, k, d->head_dim, d->hkv / hg, rows, bn / 2, input_pitch(d, 1)) ||
      !make_thd_map(&tv, v, d->head_dim, d->hkv / hg, rows, bn, input_pitch(d, 2)) ||
      !make_out_map(&to, o_part, d->head_dim, d->hq / hg, rows, nslab, o_slab))
    return CCG_ERR_CUDA;
  CCG_LAUNCH("attn_fwd", s,
             launch_attn_fwd(tq, tk, tk2, tv, to, items, hdr, cu, cu_pad, o_part, lse_part, o_slab, lse_slab, status, d->cp,
                             d->hq, d->hkv, hg, d->total_tokens, d->head_dim, softmax_scale(d), mode,
                             num_sms_cached(), s));
  *launches_out = launches;
  return CCG_OK;
}

// The work plan (all ring steps, or step `step_only` in mode 0), then the
// forward attention kernel.
static ccg_status fwd_partials(const ccg_attn_desc* d, int step_only, const void* q, const void* k,
                               const void* v, const int32_t* cu, const int32_t* cu_pad, void* o_part,
                               int64_t o_slab, float* lse_part, int64_t lse_slab, void* workspace,
                               const Layout& L, int32_t* status, cudaStream_t s, int* launches_out, int mode) {
  int launches = *launches_out;
  auto* base = static_cast<uint8_t*>(workspace);
  CCG_LAUNCH("plan", s,
             launch_plan(cu, cu_pad, d->batch, d->total_tokens, d->cp, d->hkv, kQTile, kMinKvTile, L.cap_q,
                         L.cap_kv * d->hkv, mode == 0 ? 1 : 4, step_only, reinterpret_cast<PlanHeader*>(base + L.hdr),
                         reinterpret_cast<WorkItem*>(base + L.fwd_items), nullptr, nullptr, status, s));
  *launches_out = launches;
  return fwd_attention(d, q, k, v, cu, cu_pad, o_part, o_slab, lse_part, lse_slab, workspace, L, status, s,
                       launches_out, mode);
}

ccg_status ccg_attn_fwd_step(const ccg_attn_desc* desc, int32_t step, const void* q, const void* k,
                             const void* v, const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded,
                             void* o_part, float* lse_part, void* workspace, size_t workspace_bytes,
                             int32_t* d_status, ccg_stream_t stream) {
  g_last_launches = 0;
  Layout L;
  ccg_status st = fwd_prepare(desc, q, k, v, cu_seqlens, cu_seqlens_padded, workspace, workspace_bytes,
                              d_status, &L);
  if (st != CCG_OK) return st;
  if (step < 0 || step >= desc->cp) return CCG_ERR_INVALID_ARG;
  if (!o_part || !lse_part) return CCG_ERR_INVALID_ARG;
  if (!aligned16(o_part)) return CCG_ERR_ALIGNMENT;
  if (desc->total_tokens == 0) return CCG_OK;
  int launches = 0;
  st = fwd_partials(desc, step, q, k, v, cu_seqlens, cu_seqlens_padded, o_part, 0, lse_part, 0, workspace, L,
                    d_status, reinterpret_cast<cudaStream_t>(stream), &launches, 0);
  g_last_launches = launches;
  return st;
}

ccg_status ccg_attn_fwd(const ccg_attn_desc* desc, const void* q, const void* k, const void* v,
                        const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, void* o, float* lse,
                        void* workspace, size_t workspace_bytes, int32_t* d_status, ccg_stream_t stream) {
  g_last_launches = 0;
  Layout L;
  ccg_status st = fwd_prepare(desc, q, k, v, cu_seqlens, cu_seqlens_padded, workspace, workspace_bytes,
                              d_status, &L);
  if (st != CCG_OK) return st;
  if (!o || !lse) return CCG_ERR_INVALID_ARG;
  if (!aligned16(o)) return CCG_ERR_ALIGNMENT;
  if (desc->total_tokens == 0) return CCG_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto* base = static_cast<uint8_t*>(workspace);
  const int parts = head_parts_of(desc);
  const int D = desc->head_dim;
  const int64_t T = desc->total_tokens;
  const size_t rows = size_t(T) * desc->hq / parts;          // partial rows of one head part
  const size_t o_stride = rows * D * 2, l_stride = rows * 4;
  int launches = 0;
  // Head partitioning (TransformerEngine PR, native head partitioning): the
  // ring forward and its merge run over one head part at a time, reusing the
  // one set of partial slabs.  Each output row's partials and merge order
  // are those of the unpartitioned run, so the results are bitwise equal.
  for (int part = 0; part < parts; ++part) {
    ccg_attn_desc pd = *desc;
    const void *qp = q, *kp = k, *vp = v;
    void* op = o;
    float* lp = lse;
    int out_heads = 0, out_h0 = 0;
    if (parts > 1) {
      pd.hq = desc->hq / parts;
      pd.hkv = desc->hkv / parts;
      pd.head_parts = 0;
      if (desc->head_groups > 1) {
        // whole head groups: the part is a contiguous [G_h/parts][T][H/G_h][D] sub-tensor
        const int gpp = desc->head_groups / parts;
        pd.head_groups = gpp;
        const int64_t q_grp = T * (desc->hq / desc->head_groups), kv_grp = T * (desc->hkv / desc->head_groups);
        qp = static_cast<const uint16_t*>(q) + int64_t(part) * gpp * q_grp * D;
        kp = static_cast<const uint16_t*>(k) + int64_t(part) * gpp * kv_grp * D;
        vp = static_cast<const uint16_t*>(v) + int64_t(part) * gpp * kv_grp * D;
        op = static_cast<uint16_t*>(o) + int64_t(part) * gpp * q_grp * D;
        lp = lse + int64_t(part) * gpp * q_grp;
      } else {
        // a head slice of every token row: the inputs keep their row pitch,
        // the merge writes the part's heads of each output row
        pd.q_pitch = input_pitch(desc, 0);
        pd.k_pitch = input_pitch(desc, 1);
        pd.v_pitch = input_pitch(desc, 2);
        qp = static_cast<const uint16_t*>(q) + int64_t(part) * pd.hq * D;
        kp = static_cast<const uint16_t*>(k) + int64_t(part) * pd.hkv * D;
        vp = static_cast<const uint16_t*>(v) + int64_t(part) * pd.hkv * D;
        out_heads = desc->hq;
        out_h0 = part * pd.hq;
      }
    }
    if (part == 0) {
      CCG_LAUNCH("plan", s,
                 launch_plan(cu_seqlens, cu_seqlens_padded, desc->batch, T, desc->cp, desc->hkv, kQTile,
                             kMinKvTile, L.cap_q, L.cap_kv * desc->hkv, 4, -1,
                             reinterpret_cast<PlanHeader*>(base + L.hdr),
                             reinterpret_cast<WorkItem*>(base + L.fwd_items), nullptr, nullptr, d_status, s));
    }
    st = fwd_attention(&pd, qp, kp, vp, cu_seqlens, cu_seqlens_padded, base + L.o_parts,
                       static_cast<int64_t>(rows * D), reinterpret_cast<float*>(base + L.lse_parts),
                       static_cast<int64_t>(rows), workspace, L, d_status, s, &launches, 1);
    if (st != CCG_OK) return st;
    MergeArgs a{};
    for (int p = 0; p < desc->cp; ++p) {
      a.o_parts[p] = base + L.o_parts + p * o_stride;
      a.lse_parts[p] = reinterpret_cast<const float*>(base + L.lse_parts + p * l_stride);
    }
    a.nparts = desc->cp;
    a.cu = cu_seqlens;
    a.cu_pad = cu_seqlens_padded;
    a.B = desc->batch;
    a.cp = desc->cp;
    a.hpg = pd.hq / pd.head_groups;
    a.T = T;
    a.o = op;
    a.lse = lp;
    a.rows = static_cast<int64_t>(rows);
    a.D = D;
    a.status = d_status;
    a.out_heads = out_heads;
    a.out_h0 = out_h0;
    CCG_LAUNCH("lse_merge", s, launch_lse_merge(a, num_sms_cached(), s));
  }
  g_last_launches = launches;
  return CCG_OK;
}

ccg_status ccg_attn_fwd_fused(const ccg_attn_desc* desc, const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, void* o, float* lse,
                              void* workspace, size_t workspace_bytes, int32_t* d_status, ccg_stream_t stream) {
  g_last_launches = 0;
  Layout L;
  ccg_status st = fwd_prepare(desc, q, k, v, cu_seqlens, cu_seqlens_padded, workspace, workspace_bytes,
                              d_status, &L, 2);
  if (st != CCG_OK) return st;
  if (!o || !lse) return CCG_ERR_INVALID_ARG;
  if (!aligned16(o)) return CCG_ERR_ALIGNMENT;
  if (desc->total_tokens == 0) return CCG_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int launches = 0;
  st = fwd_partials(desc, -1, q, k, v, cu_seqlens, cu_seqlens_padded, o, 0, lse, 0, workspace, L, d_status, s,
                    &launches, 2);
  if (st != CCG_OK) return st;
  CCG_LAUNCH("pad_rows", s,
             launch_pad_rows(o, lse, cu_seqlens, cu_seqlens_padded, desc->batch, desc->total_tokens, desc->hq,
                             desc->hq / desc->head_groups, desc->head_dim, d_status, num_sms_cached(), s));
  g_last_launches = launches;
  return CCG_OK;
}

ccg_status ccg_attn_bwd(const ccg_attn_desc* desc, const void* q, const void* k, const void* v,
                        const void* o, const void* dout, const float* lse, const int32_t* cu_seqlens,
                        const int32_t* cu_seqlens_padded, void* dq, void* dk, void* dv, void* workspace,
                        size_t workspace_bytes, int32_t* d_status, ccg_stream_t stream) {
  g_last_launches = 0;
  ccg_status st = check_desc(desc);
  if (st != CCG_OK) return st;
  if (!q || !k || !v || !o || !dout || !lse || !cu_seqlens || !cu_seqlens_padded || !dq || !dk || !dv ||
      !d_status)
    return CCG_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, o, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    if (!aligned16(p)) return CCG_ERR_ALIGNMENT;
  const Layout L = workspace_layout(desc, 1);
  if (workspace == nullptr || workspace_bytes < L.total) return CCG_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CCG_ERR_ALIGNMENT;
  if (desc->total_tokens == 0) return CCG_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto* base = static_cast<uint8_t*>(workspace);
  auto* hdr = reinterpret_cast<PlanHeader*>(base + L.hdr);
  auto* dq_items = reinterpret_cast<WorkItem*>(base + L.dq_items);
  auto* kv_items = reinterpret_cast<WorkItem*>(base + L.kv_items);
  auto* delta = reinterpret_cast<float*>(base + L.delta);
  const int D = desc->head_dim;
  const int hg = desc->head_groups;
  const int64_t rows = desc->total_tokens * hg;
  int launches = 0;
  CCG_LAUNCH("plan", s,
             launch_plan(cu_seqlens, cu_seqlens_padded, desc->batch, desc->total_tokens, desc->cp, desc->hkv,
                         bwd_q_tile_rows(D), bwd_kv_tile_rows(D), L.cap_q, L.cap_kv * desc->hkv, 2, -1, hdr, nullptr, dq_items,
                         kv_items, d_status, s, desc->max_seqlen,
                         L.ds_cap_tiles > 0 ? reinterpret_cast<int64_t*>(base + L.ds_base) : nullptr));
  CCG_LAUNCH("bwd_dot", s,
             launch_bwd_dot(o, dout, desc->total_tokens * desc->hq, D, desc->hq / desc->head_groups,
                            input_pitch(desc, 3), delta,
                            d_status, num_sms_cached(), s));
  // maps: q, k, v, dO for each of the three backward kernels (row boxes differ)
  CUtensorMap maps[12];
  const int hq_g = desc->hq / hg, hkv_g = desc->hkv / hg;
  const void* bases[4] = {q, k, v, dout};
  const int hpgs[4] = {hq_g, hkv_g, hkv_g, hq_g};
  for (int i = 0; i < 12; ++i)
    if (!make_thd_map(&maps[i], bases[i % 4], D, hpgs[i % 4], rows, bwd_map_rows(i, D), input_pitch(desc, i % 4)))
      return CCG_ERR_CUDA;
  // dS backward: the tile map of its dS and P tiles, and a bound on the KV
  // tile pairs of one kv head (sum over sequences and chunks of ceil(t / 2))
  CUtensorMap ds_map;
  int kv_pairs = 0;
  if (L.ds_cap_tiles > 0) {
    if (D == 256 && !make_tile_map(&ds_map, base + L.ds, 2 * L.ds_cap_tiles * (desc->hq / desc->hkv)))
      return CCG_ERR_CUDA;
    kv_pairs = static_cast<int>(desc->total_tokens / 256 + int64_t(desc->batch) * 2 * desc->cp + 1);
  }
  int kl = 0;
  if (launch_attn_bwd(maps, dq_items, kv_items, hdr, cu_seqlens, cu_seqlens_padded, lse, delta, dq, dk, dv,
                      d_status, desc->cp, desc->hq, desc->hkv, hg, desc->total_tokens, D,
                      softmax_scale(desc), L.cap_q, L.cap_kv, &kl, s, L.ds_cap_tiles > 0 ? base + L.ds : nullptr,
                      reinterpret_cast<const int64_t*>(base + L.ds_base), L.ds_cap_tiles,
                      L.ds_cap_tiles > 0 ? &ds_map : nullptr, kv_pairs) != cudaSuccess)
    return CCG_ERR_CUDA;
  launches += kl;
  g_last_launches = launches;
  return CCG_OK;
}

}  // extern "C"
