/*
 * ccg.h -- C ABI of libccg: context-parallel causal grouped-query attention
 * over packed THD BF16 sequences, computed the way a context-parallel (CP)
 * rank computes it, with every CP rank emulated as a partition of one GPU.
 *
 * The operation is the one described by the TransformerEngine pull request
 * "Optimize context parallel attention layouts and gradient accumulation"
 * (sections Description, Changes, CP8 first-gradient accumulator reuse,
 * Independent-node complete-CP evidence): BF16 causal THD attention, GQA
 * (Hq query heads sharing Hkv key/value heads), D = 128 or 256, each
 * sequence cut into 2*CP load-balanced chunks (rank r holds chunks r and
 * 2CP-1-r), per-rank partial outputs carrying log-sum-exp (LSE) stats that
 * are merged by LSE rescaling, dK/dV accumulated in a fixed order with the
 * first contribution used as the accumulator, and the A2A head-split
 * pack/unpack layout copies.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - All tensor pointers are DEVICE pointers unless stated otherwise, 16-byte
 *    aligned, contiguous.  The caller owns every buffer; the library
 *    allocates no device memory and keeps no per-call state.
 *  - Every call is asynchronous on the caller's `stream`; none synchronises
 *    except ccg_get_status.
 *  - Errors are fail-closed: an unsupported shape, dtype, head dimension, CP
 *    size or alignment returns an error code and launches nothing.  There is
 *    no fallback route.
 *  - Device-detected errors (broken sequence-length promises, a bounded wait
 *    that ran out) are written into the caller's int32 status word
 *    `d_status` (device memory, zeroed by the caller before first use).  A
 *    status word is sticky: kernels only ever write a non-zero code into it,
 *    and every kernel of this library that is given a non-zero status word
 *    returns without writing its outputs.  Read it with ccg_get_status.
 *  - Tensor layout "THD with head groups": a tensor with H heads of width D
 *    and `head_groups` = G_h (1 or CP) is stored as [G_h][T][H/G_h][D]; head
 *    h of token t lives at row (h / (H/G_h)) * T + t, slot h % (H/G_h).
 *    G_h = 1 is the plain packed THD layout [T][H][D].  G_h = the A2A size is
 *    the head-split layout produced by ccg_thd_pack.  LSE tensors use the same
 *    grouping with D = 1: [G_h][T][Hq/G_h] float.
 *  - Sequences: cu_seqlens[B+1] (logical lengths S_b) and
 *    cu_seqlens_padded[B+1] (physical offsets, padded lengths P_b), int32,
 *    device memory.  Sequence b occupies physical rows
 *    [cu_seqlens_padded[b], cu_seqlens_padded[b+1]); its first S_b rows are
 *    tokens, the rest padding.  cu_seqlens_padded may equal cu_seqlens.
 *    Every P_b must be a multiple of 2*CP (the chunks are cut on P_b) and
 *    cu_seqlens_padded[B] must equal T.  Padding rows neither attend nor are
 *    attended: their O, dQ, dK, dV are written as 0 and their LSE as -inf.
 */
#ifndef CCG_H_
#define CCG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ccg_stream_t;   /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  CCG_OK = 0,
  CCG_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shapes      */
  CCG_ERR_UNSUPPORTED = 2,   /* D not in {128,256}, Hq % Hkv, CP out of range, ...     */
  CCG_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned                       */
  CCG_ERR_WORKSPACE = 4,     /* workspace missing or smaller than ccg_workspace_size   */
  CCG_ERR_SEQLENS = 5,       /* device-detected: cu_seqlens / cu_seqlens_padded break
                                the promise (not monotone, S_b > P_b, P_b % 2CP != 0,
                                cu_seqlens_padded[B] != T)                              */
  CCG_ERR_TIMEOUT = 6,       /* device-detected: a bounded wait inside a kernel ran out */
  CCG_ERR_CUDA = 7           /* a CUDA runtime/driver call failed (launch, tensor map)  */
} ccg_status;

/* Problem description shared by ccg_attn_fwd / ccg_attn_bwd. */
typedef struct {
  int32_t batch;          /* B, number of packed sequences (>= 1)                     */
  int32_t hq;             /* query heads                                               */
  int32_t hkv;            /* key/value heads; hq % hkv == 0; q head h uses kv head
                             h / (hq/hkv) (contiguous GQA groups)                       */
  int32_t head_dim;       /* D: 128 or 256                                             */
  int32_t causal;         /* must be 1 (the path is causal attention)                  */
  int32_t cp;             /* emulated context-parallel ranks, 1..16                    */
  int32_t head_groups;    /* G_h >= 1: 1 = plain THD, >1 = head-split layout (e.g. the
                             A2A layout of ccg_thd_pack); hq, hkv divisible by it    */
  int32_t head_parts;     /* 0 or 1: no head partitioning; P > 1: ccg_attn_fwd runs the
                             ring forward and merge over P head parts in turn (the
                             PR's native head partitioning, Description and Native
                             head partitioning: bounded workspace), reusing one set
                             of partial slabs sized for hq/P heads; results are
                             bitwise equal to P = 1.  hkv % P == 0, and with
                             head_groups > 1, head_groups % P == 0.  The other
                             entry points ignore it.                                  */
  int64_t total_tokens;   /* T = cu_seqlens_padded[B]                                  */
  float softmax_scale;    /* <= 0 selects 1/sqrt(D)                                    */
  /* Physical row pitch of the THD inputs: elements from one token's row to the
   * next in q, k, v and dO (e.g. q, k, v sliced out of one fused [T][Hq+2Hkv][D]
   * projection output).  0 = dense (H*D).  A nonzero pitch is at least H*D,
   * a multiple of 8 (16 bytes), and needs head_groups == 1; the heads of a row
   * stay contiguous (stride D).  Outputs (o, lse, dq, dk, dv) are always dense.
   * This is the page's physical-pitch (strided) THD input (PR, CP8 AllGather:
   * composition with first-gradient reuse). */
  int64_t q_pitch, k_pitch, v_pitch, do_pitch;
  /* 0, or an upper bound on every sequence's padded length
   * (cu_seqlens_padded[b+1] - cu_seqlens_padded[b] <= max_seqlen, checked on
   * the device: CCG_ERR_SEQLENS).  A bound selects the backward that keeps
   * dS: the dQ pass also writes each unit's BF16 dS tile to the workspace
   * and the dK pass reads it back (dK += dS^T Q, instead of recomputing dP^T
   * and dS^T).  With D = 256 it keeps P as well (dV += P^T dO from the stored
   * P: one product per unit each for dK and dV); with D = 128 one dK/dV pass
   * recomputes only P^T.  The kv heads are then taken one at a time (the dQ
   * pass over the kv head's q heads, then its dK/dV passes), so the tiles
   * the workspace holds are those of one GQA group:
   * ccg_workspace_size(desc, 1) grows by about
   * K (hq/hkv) * ceil(max_seqlen / (256 cp)) * (T / (256 cp) + B) * cp (2 cp + 1) * 32 KiB,
   * K = 2 at D = 256 (dS and P), 1 at D = 128 (dS).
   * 0 keeps the backward that recomputes them. */
  int64_t max_seqlen;
} ccg_attn_desc;

/* Bytes of device workspace needed for `desc` by ccg_attn_fwd (kind = 0),
 * ccg_attn_bwd (kind = 1) or ccg_attn_fwd_fused (kind = 2); 0 if `desc` or
 * `kind` is invalid.  The forward workspace holds the work plan plus CP
 * per-step partial outputs (CP x T x Hq/P x D BF16, P = head_parts or 1) and
 * their LSE (CP x T x Hq/P float); the backward workspace holds the work plans
 * and Delta (T x Hq float); the fused forward workspace holds only the work
 * plan. */
size_t ccg_workspace_size(const ccg_attn_desc* desc, int kind);

/* Forward: O = softmax(scale Q K^T + causal mask) V and its row LSE, computed
 * as CP emulated ranks do it (TransformerEngine PR, Independent-node
 * complete-CP evidence; ring exchange as in Related optimization work, P2P):
 * for ring step s = 0..CP-1 every rank r attends its two query chunks over
 * the KV chunks of rank (r - s) mod CP, producing a partial (O_s, LSE_s);
 * the partials are then merged by LSE rescaling in ascending step order.
 *   q: [G_h][T][Hq/G_h][D] bf16;  k, v: [G_h][T][Hkv/G_h][D] bf16
 *   o: same layout as q (bf16, written);  lse: [G_h][T][Hq/G_h] float (written,
 *      natural log)
 *   workspace: >= ccg_workspace_size(desc, 0) bytes, 256-byte aligned.
 * Every element of o and lse is written (padding rows 0 / -inf). */
ccg_status ccg_attn_fwd(const ccg_attn_desc* desc, const void* q, const void* k, const void* v,
                        const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded,
                        void* o, float* lse, void* workspace, size_t workspace_bytes,
                        int32_t* d_status, ccg_stream_t stream);

/* Forward with the merge folded into the attention (the next step after the
 * ring-partials path; TransformerEngine PR, Description: the partials exist
 * only to be combined by LSE rescaling): each query tile runs ONE online
 * softmax over the KV chunks of every ring step of its rank, in ring order,
 * instead of one softmax per step followed by the K-way merge.  Same result
 * up to rounding order, same arguments and layouts as ccg_attn_fwd; the
 * workspace is ccg_workspace_size(desc, 2) bytes (the plan only: no partials
 * are materialised). */
ccg_status ccg_attn_fwd_fused(const ccg_attn_desc* desc, const void* q, const void* k,
                              const void* v, const int32_t* cu_seqlens,
                              const int32_t* cu_seqlens_padded, void* o, float* lse,
                              void* workspace, size_t workspace_bytes, int32_t* d_status,
                              ccg_stream_t stream);

/* One ring step of the forward, exposed for inspection: the partial
 * (O_s, LSE_s) of step `step` for all emulated ranks.  Rows that have no
 * partial at this step (an early chunk whose source rank only holds later
 * KV, and padding rows) are NOT written.  Same layouts and workspace as
 * ccg_attn_fwd (the partial buffers inside the workspace are not used). */
ccg_status ccg_attn_fwd_step(const ccg_attn_desc* desc, int32_t step, const void* q,
                             const void* k, const void* v, const int32_t* cu_seqlens,
                             const int32_t* cu_seqlens_padded, void* o_part, float* lse_part,
                             void* workspace, size_t workspace_bytes, int32_t* d_status,
                             ccg_stream_t stream);

/* Backward (TransformerEngine PR, Changes and CP8 first-gradient accumulator
 * reuse): dQ, dK, dV of the forward above given dO, the merged O and LSE.
 * Delta = rowsum(O * dO) is computed first; dQ of each query chunk sums its
 * KV contributions in ring-step order; dK/dV of each KV chunk sum the
 * contributions of ranks src, src+1, ... (ring steps 0..CP-1), query chunk r
 * before 2CP-1-r, query tile ascending, q head ascending, the FIRST
 * contribution initialising the accumulator (no zero fill).  The order is
 * fixed, so results are bitwise repeatable run to run.
 *   o, dout: layout of q (bf16);  lse: as written by ccg_attn_fwd
 *   dq: layout of q; dk, dv: layout of k (bf16, all written, padding rows 0)
 *   workspace: >= ccg_workspace_size(desc, 1) bytes, 256-byte aligned. */
ccg_status ccg_attn_bwd(const ccg_attn_desc* desc, const void* q, const void* k, const void* v,
                        const void* o, const void* dout, const float* lse,
                        const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded,
                        void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        int32_t* d_status, ccg_stream_t stream);

/* Allocation-free variant of ccg_attn_bwd, for callers that cannot allocate
 * device memory (for example a plugin whose host framework owns all device
 * memory and hands it only input and output pointers, or code that must not
 * call cudaMalloc once it is running).  It computes exactly what
 * ccg_attn_bwd computes, with the same arguments minus the workspace: its
 * scratch (work plan and Delta) is a fixed 16 MiB array in the library's
 * device image, held by every GPU that loads the library until the process
 * exits.  This entry point has no counterpart in the TransformerEngine pull
 * request the rest of this header follows.
 *   Limit: ccg_workspace_size(desc, 1) must be at most 16,776,960 bytes
 *   (16 MiB - 256); larger problems return CCG_ERR_WORKSPACE and launch
 *   nothing.  A padded-length bound (max_seqlen > 0) adds the dS tiles to
 *   the workspace and exceeds the scratch for all but the smallest
 *   problems: pass max_seqlen = 0 (the backward that recomputes dS) here.  The library itself allocates nothing here (no cudaMalloc,
 *   no cudaFree).
 *   d_status: the caller's status word, as in ccg_attn_bwd; NULL selects a
 *   status word inside the fixed scratch that is cleared at the start of
 *   every call and cannot be read back.  With d_status NULL, a failure the
 *   device detects (a broken sequence-length promise, CCG_ERR_SEQLENS, or
 *   a bounded wait that ran out, CCG_ERR_TIMEOUT) is NOT reported: the call
 *   still returns CCG_OK and dq, dk, dv are left unwritten (they keep
 *   whatever the caller had there).  Pass a status word unless the
 *   sequence offsets are already known to be valid.
 *   The first call on a device looks up the array's device address on that
 *   device (cudaGetSymbolAddress, with the device current), and so does the
 *   first call after the device's CUDA context changed (cudaDeviceReset);
 *   make that first call before any stream capture.  All calls on a device share the one
 *   array, which keeps the previous call's contents (every call rewrites
 *   the plan and Delta before reading them): calls whose execution overlaps
 *   on the GPU race on it and must not be issued. */
ccg_status ccg_attn_bwd_noalloc(const ccg_attn_desc* desc, const void* q, const void* k,
                                const void* v, const void* o, const void* dout, const float* lse,
                                const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded,
                                void* dq, void* dk, void* dv, int32_t* d_status,
                                ccg_stream_t stream);

/* Load-balanced CP split (TransformerEngine PR, Independent-node complete-CP
 * evidence: CP8 over packed THD; the 2*CP chunk "reorder"): writes
 * chunk_table[b][c] = {first physical row, length} for c = 0..2CP-1, with
 * length P_b / (2CP); chunk c is held by rank c < CP ? c : 2CP-1-c.
 * Validates the sequence promise on device (status word as above).
 *   cu_seqlens, cu_seqlens_padded: device int32 [batch+1]
 *   chunk_table: device int32 [batch][2cp][2], written. */
ccg_status ccg_cp_split(const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded,
                        int32_t batch, int64_t total_tokens, int32_t cp, int32_t* chunk_table,
                        int32_t* d_status, ccg_stream_t stream);

/* K-way LSE merge of partial attention outputs (the CP "LSE correction";
 * TransformerEngine PR, Description: partial outputs with their Stats):
 *   M = max_s LSE_s, LSE = M + ln sum_s exp(LSE_s - M),
 *   O = sum_s exp(LSE_s - LSE) O_s, summed in the given order s = 0..K-1.
 * A partial whose LSE is -inf is absent for that row (its O is not read).
 * Rows whose partials are all absent get O = 0, LSE = -inf.
 *   o_parts, lse_parts: HOST arrays of `nparts` (1..16) DEVICE pointers to
 *      bf16 [rows][head_dim] and float [rows]
 *   o: bf16 [rows][head_dim], lse: float [rows], written. */
ccg_status ccg_cp_lse_merge(int32_t nparts, const void* const* o_parts,
                            const float* const* lse_parts, int64_t rows, int32_t head_dim,
                            void* o, float* lse, ccg_stream_t stream);

/* Delta[row] = sum_d O[row][d] * dO[row][d] in float (TransformerEngine PR,
 * CP8 AllGather composition: the backward's row dot of O and dO over pitched rows).
 *   o, dout: bf16 [rows][head_dim];  delta: float [rows], written. */
ccg_status ccg_bwd_dot(const void* o, const void* dout, int64_t rows, int32_t head_dim,
                       float* delta, ccg_stream_t stream);

/* A2A head-split pack (TransformerEngine PR, Changes: "vectorized A2A layout
 * copies"): from the rank-major local layout (for rank r, for sequence b:
 * chunk r then chunk 2CP-1-r; [T][H][D]) to the head-split layout
 * [CP][T][H/CP][D] in sequence order:
 *   out[g][t][h'][:] = x[pi(t)][g*H/CP + h'][:],  pi = sequence row -> rank-major row.
 * Bit-exact copy of 16-bit elements.  H % cp == 0; P_b % 2cp == 0. */
ccg_status ccg_thd_pack(const void* x_rank_major, const int32_t* cu_seqlens_padded,
                        int32_t batch, int64_t total_tokens, int32_t heads, int32_t head_dim,
                        int32_t cp, void* out_head_split, int32_t* d_status, ccg_stream_t stream);

/* Inverse of ccg_thd_pack: head-split [CP][T][H/CP][D] -> rank-major [T][H][D]. */
ccg_status ccg_thd_unpack(const void* in_head_split, const int32_t* cu_seqlens_padded,
                          int32_t batch, int64_t total_tokens, int32_t heads, int32_t head_dim,
                          int32_t cp, void* x_rank_major, int32_t* d_status, ccg_stream_t stream);

/* Self-test of the device failure path; no fault is involved.  Launches one
 * CTA whose thread waits, bounded by `limit_us` microseconds (1..1000000), on
 * a shared-memory barrier that nothing arrives at: the wait gives up, the
 * kernel writes CCG_ERR_TIMEOUT into d_status and returns normally, exactly
 * as the attention kernels do when one of their bounded waits runs out.  Lets
 * a caller check that device-detected errors reach the host and that the
 * CUDA context stays usable afterwards. */
ccg_status ccg_selftest_bounded_wait(int32_t* d_status, uint32_t limit_us, ccg_stream_t stream);

/* Synchronises `stream`, reads the device status word and returns it
 * (CCG_OK, CCG_ERR_SEQLENS or CCG_ERR_TIMEOUT), or CCG_ERR_CUDA if the
 * synchronisation itself failed. */
ccg_status ccg_get_status(const int32_t* d_status, ccg_stream_t stream);

/* Static description of a status code. */
const char* ccg_status_str(ccg_status s);

/* Number of kernel launches the most recent successful ccg_* call on this
 * host thread issued (for launch accounting by callers). */
int32_t ccg_last_launch_count(void);

/* Launch timing for callers that measure the library.  Between
 * ccg_profile_begin and ccg_profile_end, every kernel the library launches
 * from the calling host thread is bracketed by two CUDA events recorded on
 * the stream it is launched on.  `capacity` event pairs are created by
 * ccg_profile_begin (host-side CUDA events; no device memory is allocated);
 * launches beyond the capacity are not timed.  Returns CCG_ERR_CUDA if the
 * events cannot be created. */
ccg_status ccg_profile_begin(int32_t capacity);
ccg_status ccg_profile_end(void);
/* Number of launches timed by the last profile. */
int32_t ccg_profile_count(void);
/* Kernel name (static string) and elapsed milliseconds of the i-th timed
 * launch; waits for that launch's end event. */
ccg_status ccg_profile_get(int32_t i, const char** kernel_name, float* ms);

#ifdef __cplusplus
}
#endif

#endif /* CCG_H_ */
