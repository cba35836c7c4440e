/*
 * df_attn.h -- C ABI of the exact DeBERTa-v2/v3 disentangled attention for
 * NVIDIA GB300 (sm_103a): the fused forward pass, its backward pass, the
 * forward from host buffers, and the steps on either side of the attention
 * (padded <-> packed conversion, projections, LayerNorm).
 *
 * The operation (DisentangledFlash 0.2.0 README, section "Status":
 * "DeBERTa-v2/v3-style C2P/P2C disentangled attention", "factorized 2-D padding
 * masks", "packed, unpadded inference with cu_seqlens"; kernels-community
 * discussion "DisentangledFlash", section "Motivation": content-to-position and
 * position-to-content terms, evaluated exactly without materialising the
 * [B, H, L, L] matrix):
 *
 *   score(i,j) = ( Q_i.K_j + Q_i.PK[idx(i-j)] + K_j.PQ[idx(i-j)] ) / sqrt(3 d)
 *   idx(r)     = clamp(bucket(r) + span, 0, 2 span - 1)
 *   bucket(r)  = r                                   for |r| <= buckets/2,
 *              = sign(r) (mid + ceil(ln(|r|/mid) / ln((max_rel-1)/mid) (mid-1)))
 *                                                    otherwise (mid = buckets/2);
 *              = r for every r when buckets <= 0.
 *   O_i        = sum_j softmax_j(score(i, .)) V_j  over valid keys j;
 *   O_i        = 0 for a query row whose own mask bit is 0.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     allocates nothing, never synchronises (except df_attn_get_device_status)
 *     and enqueues all work on `stream` (NULL = legacy default stream).
 *   - Layouts are dense row-major.  Padded mode: q, k, v, out are [B, L, H, d]
 *     and key_mask is uint8 [B, L] (nonzero = valid; applied to keys and, as
 *     the factorized mask, to query rows).  Packed mode: q, k, v, out are
 *     [T, H, d] with int32 cu_seqlens [B + 1] (cu_seqlens[0] = 0,
 *     cu_seqlens[B] = T, non-decreasing, every length <= L).  pos_key (PK) and
 *     pos_query (PQ) are [2 span, H, d].  All of q, k, v, pos_key, pos_query,
 *     out share `dtype`.
 *   - Positions restart at 0 in every sequence (padded: index inside the batch
 *     row; packed: offset from cu_seqlens[s]).
 *   - Pointers must be 16-byte aligned (tensor-memory-access copies).
 *   - Argument checks run on the host before any launch; a failing check
 *     returns a status and enqueues nothing.  There is no fallback path.
 */
#ifndef DF_ATTN_H
#define DF_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / cudaEvent_t; declared here so that this header
 * needs no CUDA include. */
typedef struct CUstream_st* df_stream_t;
typedef struct CUevent_st* df_event_t;

typedef enum {
  DF_OK = 0,
  DF_ERR_INVALID_ARG = 1,     /* a pointer, size or parameter is out of contract */
  DF_ERR_UNSUPPORTED = 2,     /* valid request this build does not implement (e.g. d = 48) */
  DF_ERR_ALIGNMENT = 3,       /* a pointer is not 16-byte aligned */
  DF_ERR_WORKSPACE = 4,       /* workspace NULL or smaller than df_attn_workspace_size() */
  DF_ERR_CUDA = 5,            /* a CUDA runtime call failed (launch, tensor-map encode) */
  DF_ERR_DEVICE_TIMEOUT = 6   /* a kernel's bounded wait ran out (read back by
                                 df_attn_get_device_status) */
} df_status;

typedef enum { DF_BF16 = 0, DF_FP16 = 1, DF_FP32 = 2 } df_dtype;

/*
 * Fused forward pass.
 *
 *   q, k, v            [B, L, H, d] (padded) or [T, H, d] (packed), `dtype`
 *   pos_key, pos_query [2 span, H, d], `dtype` (the projected relative embeddings)
 *   key_mask           uint8 [B, L] in padded mode, NULL in packed mode
 *   cu_seqlens         int32 [B + 1] in packed mode, NULL in padded mode
 *   B                  batch rows (padded) or number of sequences (packed), >= 0
 *   H, d               heads and head size; d in {32, 64, 128} (bf16 / fp16 run on
 *                      the tensor cores, d = 32 as d = 64 on zero-widened copies
 *                      in the workspace; every fp32 call on the CUDA-core kernel)
 *   L                  padded length, or an upper bound of every packed length
 *                      (max_seqlen); 1 <= L <= 65536
 *   total_tokens       rows of q/k/v/out: B*L in padded mode, cu_seqlens[B] in
 *                      packed mode (the host cannot read cu_seqlens)
 *   buckets, max_rel   DeBERTa position_buckets and max_relative_positions; with
 *                      buckets > 0 it must hold 2 <= buckets/2 < max_rel - 1
 *   span               attention span: PK/PQ have 2*span rows; span >= 1
 *   dtype              DF_BF16 / DF_FP16 (tensor-core path) or DF_FP32 (strict
 *                      fp32: FFMA on CUDA cores, no TF32)
 *   out                same layout and dtype as q; every row is written (padded
 *                      query rows and rows of empty sequences get zeros)
 *   workspace          device scratch of at least df_attn_workspace_size() bytes,
 *                      256-byte aligned; its contents need not be initialised
 *                      and are overwritten by every call (calls that share a
 *                      workspace must not overlap in time)
 *   stream             CUDA stream for every launch
 *
 * Precision (bf16 / fp16): Q.K^T and both position terms are accumulated and
 * added in fp32 on every tile; P is rounded to the I/O type for P.V; the output
 * is rounded from fp32.  Magnitude limit: a masked key inside a tile whose
 * position terms are saturated (padded mode with holes in the mask) is removed
 * by adding -131008 to its raw score (a finite stand-in for -inf), so the
 * result is exact while the raw scores |Q_i.K_j + Q_i.PK + K_j.PQ| of a row stay
 * well below 131008; keys past a sequence's last valid token are removed
 * exactly.  NaN / Inf inputs are out of contract.
 *
 * Returns DF_OK once the work is enqueued; errors raised on the device are
 * reported by df_attn_get_device_status().
 */
df_status df_attn_fwd(const void* q, const void* k, const void* v,
                      const void* pos_key, const void* pos_query,
                      const uint8_t* key_mask, const int32_t* cu_seqlens,
                      int B, int H, int L, int total_tokens, int d,
                      int buckets, int max_rel, int span, df_dtype dtype,
                      void* out, void* workspace, size_t workspace_bytes,
                      df_stream_t stream);

/* Bytes of workspace df_attn_fwd / df_attn_plan need for these sizes (an upper
 * bound over both layouts and every dtype; T is bounded by B*L).  Returns 0 for
 * arguments df_attn_supported() rejects. */
size_t df_attn_workspace_size(int B, int H, int L, int d, int buckets, int max_rel, int span);

/*
 * Fast fp32 mode (DisentangledFlash 0.2.0 README, "Status": the optional fast
 * FP32/TF32 mode).  The same forward as df_attn_fwd for fp32 q, k, v, pos_key,
 * pos_query and out (arguments, layouts and the padded / packed modes as
 * there, without `dtype`), computed on the fp16 tensor-core path: every input
 * is rounded to fp16 (RNE; an 11-bit significand, as TF32 keeps), the scores
 * and P.V accumulate in fp32 as for fp16 I/O, and the output is rounded to
 * fp16 and widened back to fp32.  Not the strict-fp32 result: expect the fp16
 * path's error plus the rounding of the inputs.  Range: every input value must
 * satisfy |x| <= 65504 (fp16's largest finite value); a value outside it (or
 * not finite) makes the call record DF_ERR_INVALID_ARG in the device status
 * word (df_attn_get_device_status on this workspace), and the output is then
 * undefined.  workspace: at least df_attn_fwd_fp32_fast_workspace_size() bytes,
 * 256-byte aligned; it holds df_attn_fwd's workspace at offset 0 and fp16
 * copies of the inputs and the output after it.  Host-side errors as for
 * df_attn_fwd (checked before anything is enqueued).  Two kernel launches
 * more than df_attn_fwd's (the conversions) and one 4-byte memset.
 */
df_status df_attn_fwd_fp32_fast(const void* q, const void* k, const void* v,
                                const void* pos_key, const void* pos_query,
                                const uint8_t* key_mask, const int32_t* cu_seqlens,
                                int B, int H, int L, int total_tokens, int d,
                                int buckets, int max_rel, int span,
                                void* out, void* workspace, size_t workspace_bytes,
                                df_stream_t stream);

/* Bytes of workspace df_attn_fwd_fp32_fast needs (T bounded by B*L); 0 for
 * arguments df_attn_supported() rejects. */
size_t df_attn_fwd_fp32_fast_workspace_size(int B, int H, int L, int d, int buckets, int max_rel,
                                            int span);

/*
 * Backward pass: gradients of sum(out * dout) with respect to q, k, v, pos_key
 * and pos_query, for the forward defined above.  The pages have no backward
 * (DisentangledFlash 0.2.0 README, "Status": training keeps the stock path);
 * this one differentiates the same score exactly.  With p the softmax row,
 * dP_ij = dout_i.V_j, D_i = dout_i.O_i and dS_ij = p_ij (dP_ij - D_i)/sqrt(3 d):
 *   dv_j      = sum_i p_ij dout_i
 *   dq_i      = sum_j dS_ij (K_j + PK[idx(i-j)])
 *   dk_j      = sum_i dS_ij (Q_i + PQ[idx(i-j)])
 *   dpos_key[r]   = sum over (i, j) with idx(i-j) = r of dS_ij Q_i
 *   dpos_query[r] = sum over (i, j) with idx(i-j) = r of dS_ij K_j
 * A masked query row (its output is the constant 0) and a masked key pass no
 * gradient: their rows of dq, dk, dv are 0, as are rows outside every sequence.
 *
 *   q, k, v, pos_key, pos_query, key_mask, cu_seqlens, B, H, L, total_tokens,
 *   d, buckets, max_rel, span, dtype: as for df_attn_fwd (every dtype and
 *                      d in {32, 64, 128})
 *   dout               gradient of the output, layout and dtype of q
 *   dq, dk, dv         float32, layout of q: written in full (overwritten)
 *   dpos_key, dpos_query  float32 [2 span, H, d]: written in full, summed over
 *                      every sequence of the call
 *   workspace          at least df_attn_bwd_workspace_size() bytes, 256-byte
 *                      aligned, contents need not be initialised
 *
 * Everything is computed in fp32 on CUDA cores: the forward is recomputed per
 * query block (row log-sum-exp and O, so `out` is not an input), the score
 * tiles are recomputed on the key side, the sums of dS by relative index are
 * accumulated in the workspace with atomic adds (so the last bits may differ
 * from run to run), and the position gradients are then reduced over fixed
 * token ranges.  Returns once the work is enqueued.
 */
df_status df_attn_bwd(const void* q, const void* k, const void* v,
                      const void* pos_key, const void* pos_query, const void* dout,
                      const uint8_t* key_mask, const int32_t* cu_seqlens,
                      int B, int H, int L, int total_tokens, int d,
                      int buckets, int max_rel, int span, df_dtype dtype,
                      float* dq, float* dk, float* dv, float* dpos_key, float* dpos_query,
                      void* workspace, size_t workspace_bytes, df_stream_t stream);

/* Bytes of workspace df_attn_bwd needs for these sizes (T bounded by B*L);
 * about 16 * B*L*H*span bytes for the two bucket-sum tables.  0 for arguments
 * that df_attn_bwd rejects. */
size_t df_attn_bwd_workspace_size(int B, int H, int L, int d, int buckets, int max_rel, int span);

/*
 * Forward from HOST buffers with the copies overlapped: q, k, v, pos_key,
 * pos_query, out, and key_mask / cu_seqlens are HOST pointers (page-locked
 * memory lets the copies run asynchronously; pageable memory works but
 * serialises them).  Sequences are independent (padded: batch rows), so the
 * batch is cut into groups of whole sequences of at most
 * max(group_tokens, L) tokens (group_tokens = 0: max(B*L/4, L)), the first
 * groups ramping up from L tokens by doubling, and each group runs as one
 * df_attn_fwd call, with results identical to a single call on the whole
 * batch.  Library-owned streams (two for copies, two for the forwards of
 * alternate groups, created once per device) pipeline the copy-in of group
 * g + 1 and the copy-out of group g - 1 around the forward of group g, and let
 * the next group's kernels fill the SMs the previous group leaves idle; all
 * of it starts after the work already on `stream`, which waits for the last
 * copy-out, so `out` is complete once `stream` is.  In packed mode cu_seqlens is validated
 * on the host (cu_seqlens[0] = 0, cu_seqlens[B] = total_tokens, every length
 * in [0, L]).
 *
 *   scratch   device memory of df_attn_fwd_host_scratch_size() bytes, 256-byte
 *             aligned: two slots of q, k, v, out for one group, the relative
 *             embeddings and two forward workspaces of
 *             df_attn_workspace_size(B, H, L, d, ...) bytes each, the first at
 *             offset 0 and the second at that size rounded up to 256
 *             (df_attn_get_device_status reads each one's status)
 *
 * Calls are serialised by a mutex while they enqueue; calls that share a
 * scratch buffer must be ordered by their streams.  Returns DF_ERR_CUDA if a
 * copy or event call fails (work may then be partly enqueued).
 */
df_status df_attn_fwd_host(const void* q, const void* k, const void* v,
                           const void* pos_key, const void* pos_query,
                           const uint8_t* key_mask, const int32_t* cu_seqlens,
                           int B, int H, int L, int total_tokens, int d,
                           int buckets, int max_rel, int span, df_dtype dtype,
                           void* out, long long group_tokens,
                           void* scratch, size_t scratch_bytes, df_stream_t stream);

/* Bytes of device scratch df_attn_fwd_host needs (0 for rejected arguments). */
size_t df_attn_fwd_host_scratch_size(int B, int H, int L, int d, int buckets, int max_rel, int span,
                                     df_dtype dtype, long long group_tokens);

/* DF_OK if (H, L, d, dtype, buckets, max_rel, span) is implemented; otherwise
 * DF_ERR_INVALID_ARG or DF_ERR_UNSUPPORTED.  Host only, no CUDA call. */
df_status df_attn_supported(int H, int L, int d, df_dtype dtype, int buckets, int max_rel,
                            int span);

/* Static, NUL-terminated description of a status code. */
const char* df_attn_status_string(df_status s);

/* Synchronises `stream`, reads the device status word in `workspace` (written by
 * the kernels of earlier calls on that workspace), clears it and returns it:
 * DF_OK, or DF_ERR_DEVICE_TIMEOUT when a bounded wait ran out.  DF_ERR_CUDA if
 * the copy itself fails. */
df_status df_attn_get_device_status(void* workspace, df_stream_t stream);

/*
 * Relative-position index table (the first step of df_attn_fwd, exposed for
 * testing): idx[r + max_len - 1] = clamp(bucket(r) + span, 0, 2 span - 1) for
 * every r in [-(max_len-1), max_len-1].  `idx` is a device int32 array of
 * 2*max_len - 1 entries.  The logarithm is evaluated in double precision.
 */
df_status df_rel_index_table(int buckets, int max_rel, int span, int max_len, int32_t* idx,
                             df_stream_t stream);

/* Where df_attn_fwd keeps its planning data inside the workspace (byte offsets
 * from the workspace base, all 256-byte aligned).  Filled by
 * df_attn_workspace_layout for the same sizes as df_attn_workspace_size. */
typedef struct {
  size_t header;     /* df_ws_header                                        */
  size_t idx_table;  /* int32 [2 table_half - 1], idx of r at r + table_half - 1 */
  size_t items;      /* int32x4 [max_items] work items {start, n, head, qblk} */
  size_t scalars;    /* float [H][4][Tpad]: log2-scaled Q.PK[0], Q.PK[2span-1],
                        K.PQ[0], K.PQ[2span-1] of every token (-inf for masked keys) */
  size_t keybias;    /* float [Tpad]: 0 for a valid key, -inf otherwise       */
  size_t partial;    /* float [T][H][d + 2] un-normalised partial output, max, sum */
  size_t total;      /* == df_attn_workspace_size()                           */
  int max_items;     /* capacity of the work-item list                        */
  int t_pad;         /* Tpad = round_up(B*L + 128, 128)                       */
  int table_half;    /* round_up(L, 128) + 128: the table covers |r| < table_half */
  /* Diagonal position tables (d = 64 and 128; 0 bytes otherwise), 128 (n_diag + 1)
   * rows each: row r holds PK[idx(128 diag_m0 - 127 + r)] (diag_pk) and
   * PQ[idx(128 diag_m0 - 127 + r)] (diag_pq), [rows][H][d] in the I/O type of
   * PK / PQ.  For a tile offset m in [diag_m0, diag_m0 + n_diag) -- query block
   * minus key block of a near tile -- diagonal t in [0, 256) is row
   * 128 (m - diag_m0) + t. */
  size_t diag_pk;
  size_t diag_pq;
  int n_diag;
  int diag_m0;
  /* Key-term block of far tiles (16-bit I/O types): [Tpad][H][16] in the I/O
   * type, per key the raw p2c products K.PQ[0] and K.PQ[2span-1], each as a
   * high and a low part (hi + lo), then zeros; masked keys hold -65504 in each
   * part (the score MMA adds hi + lo = -131008).  Below
   * it, kaug_sel: [256][16] selector rows (1, 1, 0, ...) and (0, 0, 1, 1, ...). */
  size_t kaug;
  size_t kaug_sel;
  /* Position rows of the far-tile terms per head (16-bit I/O types, d = 64):
   * [H][16][64] in the I/O type, rows PK[0], PK[2span-1], PQ[0], PQ[2span-1],
   * then zeros.  With them the d = 64 near-tile kernel forms the far tiles'
   * scalars and key-term blocks from the Q and K tiles it already holds. */
  size_t absel;
} df_ws_layout;

/* Header at workspace offset 0, written on the device by every call. */
typedef struct {
  int32_t status;        /* df_status of the first device-side error, else 0 */
  int32_t status_where;  /* kernel / wait site that raised it                */
  int32_t n_items;       /* work items planned (query blocks of 128 rows)    */
  int32_t r_sat_pos;     /* smallest r with idx(r) = 2 span - 1 (>= L if none) */
  int32_t r_sat_neg;     /* largest r with idx(r) = 0 (<= -L if none)          */
  int32_t n_seqs;        /* sequences seen                                    */
  int32_t next_item;     /* near-tile kernel: next work item to hand out (its
                            CTAs take items from the list in order, longest
                            first, as each one finishes its previous item)   */
  int32_t next_far_item; /* the same for the far-tile kernel                 */
  int32_t reserved[8];
} df_ws_header;

df_status df_attn_workspace_layout(int B, int H, int L, int d, int buckets, int max_rel, int span,
                                   df_ws_layout* layout);

/* Planning step of df_attn_fwd alone (same arguments and checks): writes the
 * index table, the saturation points, the work list (query blocks of 128 rows,
 * longest sequences first) and the per-token position scalars into the
 * workspace, and zeros the output rows of padded / masked query tokens.  Used
 * by tests of the scheduler; df_attn_fwd runs it itself. */
df_status df_attn_plan(const void* q, const void* k, const void* pos_key, const void* pos_query,
                       const uint8_t* key_mask, const int32_t* cu_seqlens,
                       int B, int H, int L, int total_tokens, int d,
                       int buckets, int max_rel, int span, df_dtype dtype,
                       void* out, void* workspace, size_t workspace_bytes, df_stream_t stream);

/* Profiling hook (process-wide, not thread-safe): while set, df_attn_fwd
 * records events[0] before and events[1] after its dominant attention kernel on
 * `stream`.  Pass NULL to clear.  The events are created and owned by the
 * caller. */
void df_attn_set_profile_events(df_event_t start, df_event_t stop);

/* Profiling hook (process-wide, not thread-safe), used with the one above: while
 * set, the tensor-core path also records `mid` between its near-tile and
 * far-tile kernels, so that each can be timed alone; the strict-fp32 path (one
 * fused kernel) records it right after `start`.  Pass NULL to clear.  Owned by
 * the caller.  No counterpart in the pages: a measurement aid. */
void df_attn_set_profile_split(df_event_t mid);

/* Upper bound, in SM clock cycles, of every spin-wait on an mbarrier inside the
 * kernels (process-wide; 0 restores the default of about 2^31 cycles, ~1 s).
 * When a wait runs out the kernel records DF_ERR_DEVICE_TIMEOUT in the
 * workspace header, drains its own copies in flight, frees its tensor memory
 * and returns. */
void df_attn_set_wait_budget(unsigned long long cycles);

/* Number of kernel launches the last successful df_attn_fwd enqueued. */
int df_attn_last_launch_count(void);

/*
 * df_attn_fwd without a workspace argument, for callers that cannot allocate
 * device memory (a plug-in inside a host application that owns all device
 * memory and offers no allocator, a service that forbids cudaMalloc / cudaFree
 * after start-up).  No counterpart exists in the pages: this is a packaging
 * variant of df_attn_fwd, with identical arguments, results and errors except:
 *   - the scratch is a fixed DF_ATTN_NOALLOC_SCRATCH_BYTES array compiled into
 *     the library; every GPU that loads the library holds it until the process
 *     exits;
 *   - a problem whose df_attn_workspace_size() exceeds that size is rejected
 *     with DF_ERR_WORKSPACE and nothing is enqueued;
 *   - every call looks the array's device address up with the caller's device
 *     current; the first call on a device loads the library's module there, so
 *     make it before any stream capture;
 *   - every call on a device shares the one array, which keeps the previous
 *     call's contents: calls that overlap on the GPU (other streams, other host
 *     threads) race on it and must be serialised by the caller;
 *   - errors raised on the device (a bounded wait that ran out, bad
 *     cu_seqlens) are recorded in the status word at the start of the shared
 *     array, where each call's planning kernel resets it; read them with
 *     df_attn_noalloc_get_device_status.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define DF_ATTN_NOALLOC_SCRATCH_BYTES (64u << 20)
df_status df_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                              const void* pos_key, const void* pos_query,
                              const uint8_t* key_mask, const int32_t* cu_seqlens,
                              int B, int H, int L, int total_tokens, int d,
                              int buckets, int max_rel, int span, df_dtype dtype,
                              void* out, df_stream_t stream);

/* Device-side status of the latest df_attn_fwd_noalloc call on the current
 * device: synchronises `stream`, reads the status word from the shared scratch
 * array and clears it (the df_attn_get_device_status of that array).  Returns
 * DF_OK, DF_ERR_DEVICE_TIMEOUT or DF_ERR_INVALID_ARG as the kernels recorded
 * them, or DF_ERR_CUDA if the synchronisation or the copy fails.  Allocates
 * nothing.  No counterpart in the pages, like df_attn_fwd_noalloc. */
df_status df_attn_noalloc_get_device_status(df_stream_t stream);

/* ---------------------------------------------------------------------------
 * Packing between the padded and the packed layout (DisentangledFlash 0.2.0
 * README, "Packed unpadded inference": right-padded [B, L, hidden] input is
 * converted to FlashAttention-style [total_tokens, hidden] rows with
 * cu_seqlens, and the conversion's metadata is reused for every encoder layer
 * and for unpacking the output).  The valid positions of a uint8 mask [B, L]
 * (nonzero = valid; holes allowed) are taken in row-major order: packed row k
 * is padded row indices[k] = b L + i, sequence b owns packed rows
 * cu_seqlens[b] .. cu_seqlens[b + 1] - 1, and inverse[b L + i] is the packed
 * row of a valid position or -1.  Rows are moved as bytes, so any element type
 * works: a row is `row_bytes` bytes (a multiple of 16) and every data pointer
 * is 16-byte aligned.
 */

/* Metadata of a mask.  Device outputs, all caller-owned:
 *   cu_seqlens int32 [B + 1]; indices int32 [B L] (entries 0 .. T - 1 are
 *   written); inverse int32 [B L]; stats int32 [2] = { T, max_seqlen }.
 * T is left on the device (reading it back is the caller's synchronisation).
 * Errors: DF_ERR_INVALID_ARG for a NULL pointer, B < 1, L < 1 or B L > 2^30;
 * DF_ERR_CUDA if a launch fails.  Three kernel launches. */
df_status df_pack_info(const uint8_t* mask, int B, int L, int32_t* cu_seqlens,
                       int32_t* indices, int32_t* inverse, int32_t* stats,
                       df_stream_t stream);

/* tokens[k] = x[indices[k]] for k < stats[0]; x is [B L] rows, tokens holds at
 * least stats[0] rows.  Reads T from stats on the device.  Errors:
 * DF_ERR_INVALID_ARG (NULL pointer, rows < 1, row_bytes = 0 or not a multiple
 * of 16), DF_ERR_ALIGNMENT (x or tokens not 16-byte aligned), DF_ERR_CUDA. */
df_status df_pack_rows(const void* x, const int32_t* indices, const int32_t* stats,
                       int rows, size_t row_bytes, void* tokens, df_stream_t stream);

/* out[r] = tokens[inverse[r]] for inverse[r] >= 0, else zero bytes, for the
 * `rows` = B L padded rows.  Errors as df_pack_rows. */
df_status df_unpack_rows(const void* tokens, const int32_t* inverse, int rows,
                         size_t row_bytes, void* out, df_stream_t stream);

/* ---------------------------------------------------------------------------
 * Projections that feed the attention (DisentangledFlash 0.2.0 README,
 * "Status": the fused QKV projection; and the relative-position projections PK
 * and PQ of the relative embeddings), also the encoder's output and
 * feed-forward projections: for i < n_out (1..3),
 *     out[i][m][n] = act( sum_k x[m][k] w[i][n][k] + bias[i][n] )
 * in fp32 on the tensor cores, rounded to `dtype` (bf16 or fp16); act is the
 * identity (activation 0) or GELU x (1 + erf(x / sqrt 2)) / 2 (activation 1).  x is
 * [M, K], every w[i] is [N, K] (the nn.Linear weight layout), bias[i] is [N]
 * (a NULL `bias` array or NULL entry means no bias) and out[i] is [M, N], all
 * row-major device buffers of `dtype`.  `w`, `bias` and `out` are HOST arrays of
 * n_out device pointers.  With the stacked QKV weight [3 N, K] pass its three
 * row blocks as w[0..2]; out[0..2] are then Q, K, V in the [M, H, d] layout.
 * Constraints: K a multiple of 64, N a multiple of 256, every pointer 16-byte
 * aligned.  `status` (a device int32, may be NULL) receives
 * DF_ERR_DEVICE_TIMEOUT if a bounded wait of the kernel runs out; the caller
 * zeroes it.  Errors: DF_ERR_INVALID_ARG (NULL pointer, sizes < 1, n_out out of
 * 1..3, activation not 0 or 1), DF_ERR_UNSUPPORTED (dtype, K or N),
 * DF_ERR_ALIGNMENT, DF_ERR_CUDA. */
df_status df_linear(const void* x, int M, int K, int n_out, const void* const* w,
                    const void* const* bias, int N, void* const* out, int activation,
                    df_dtype dtype, int32_t* status, df_stream_t stream);

/* Residual add + LayerNorm, the normalisation of a DeBERTa encoder layer (after
 * the attention output and after the feed-forward block) and of its relative
 * embeddings: for every row m of [M, N],
 *     y = x[m] + residual[m]   (residual may be NULL)
 *     out[m] = (y - mean(y)) / sqrt(var(y) + eps) * gamma + beta
 * with fp32 statistics (population variance), rounded to `dtype` (bf16 or
 * fp16).  gamma, beta are [N] in `dtype`; every buffer is a row-major device
 * buffer, 16-byte aligned.  N must be 256 v with v in {1, 2, 3, 4, 6, 8}.
 * Errors: DF_ERR_INVALID_ARG (NULL pointer, M < 1, eps <= 0),
 * DF_ERR_UNSUPPORTED (dtype or N), DF_ERR_ALIGNMENT, DF_ERR_CUDA. */
df_status df_layernorm(const void* x, const void* residual, const void* gamma, const void* beta,
                       int M, int N, float eps, void* out, df_dtype dtype, df_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DF_ATTN_H */
