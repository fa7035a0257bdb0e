/*
 * lcsa.h -- C ABI of the hybrid compressed attention library (CSA / HCA), sm_103a.
 *
 * The operations follow the description of DeepSeek-V4's hybrid attention on the page
 * m.x-techcon.com/article/133366, section "2. 核心技术创新：混合压缩注意力":
 *   CSA step 1  compress every m raw KV rows into one entry (learned per-token score plus a
 *               positional bias, softmax-normalised weights, weighted sum; adjacent blocks
 *               overlap)                                          -> csa_compress
 *   CSA step 2  a low-rank lightning indexer scores every entry; each query keeps its top-k
 *                                                                 -> csa_index_topk
 *   CSA step 3  shared-KV multi-query attention over the selected entries together with the
 *               most recent 128 uncompressed tokens               -> csa_attend
 *   HCA         m' = 128 compression, no selection, dense attention over every entry plus the
 *               same window                                      -> hca_compress, hca_attend
 * and, on the same page, the efficiency paragraph (RoPE dims BF16, the rest FP8; indexer QK
 * path FP4) and section 4 (state cache for the window and the uncompressed tail; compressed
 * cache allocated in blocks of LCM(4,128) = 128 raw tokens).
 *
 * Conventions for every entry point
 *  - Pointers marked "device" are CUDA device pointers; "host" are host pointers.  Every
 *    buffer is owned by the caller.  The library allocates nothing, frees nothing, never
 *    synchronises and keeps no pointer after a call returns.  It is reentrant and keeps no state
 *    between calls apart from the bound of its device waits (lcs_set_wait_polls).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Calls
 *    enqueue kernels and return; results are ready once the stream reaches them.
 *  - Argument errors are reported synchronously by the return value (nothing is launched).
 *    Errors found on the device (a block id or an index outside its buffer) are written to
 *    `*dev_status` (device int32, may be NULL) with atomicCAS(status, 0, code): the first code
 *    wins, the offending row is skipped, the kernel never traps.  Read it after the stream.
 *  - Launch failures return LCS_ERR_CUDA.
 *  - Results are deterministic: identical inputs give identical bits, independent of the
 *    other sequences in the batch.
 *
 * Row format.  A KV row has D dims in the order [rope(64) | nope(D-64)].
 *  LCS_ROW_FP8_SPLIT: rope dims BF16 (64 x 2 bytes), nope dims FP8 E4M3 (D-64 bytes) with one
 *    fp32 scale per row: value = code * scale; scale = fp32(amax)/448 over the nope dims (1 for
 *    an all-zero row); codes round to nearest even and saturate at +-448.  580 bytes at D=512.
 *  LCS_ROW_BF16: all D dims BF16.
 *  A row set (lcs_rows) stores row i at nope + i*(D-64) (FP8) or nope + i*D*2 (BF16),
 *  rope + i*128, scale + i.
 */
#ifndef LCSA_H_
#define LCSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LCSA_ABI_VERSION 3
#define LCSA_WINDOW 128      /* sliding-window rows (x-techcon section 2, CSA step 3)      */
#define LCSA_ROPE_DIMS 64    /* BF16 RoPE slice (chenxutan.com/d/4230, section 4.5)         */
#define LCSA_BLOCK_TOKENS 128 /* raw tokens per cache block, LCM(4,128) (x-techcon sec. 4) */
#define LCSA_DEFAULT_WAIT_POLLS (1u << 20) /* polls of a bounded device wait (~1 us each)  */

typedef enum {
  LCS_OK = 0,
  LCS_ERR_INVALID_ARG = 1,  /* NULL where a buffer is required, negative size, bad flag    */
  LCS_ERR_SHAPE = 2,        /* inconsistent sizes                                         */
  LCS_ERR_ALIGNMENT = 3,    /* a buffer is not 16-byte aligned                             */
  LCS_ERR_UNSUPPORTED = 4,  /* a size outside the supported set (see each call)            */
  LCS_ERR_CUDA = 5,         /* a CUDA launch or device query failed                        */
  LCS_ERR_DEVICE_GUARD = 6, /* (device status) a block id / index / row outside its buffer */
  LCS_ERR_TIMEOUT = 7,      /* (device status) a bounded wait gave up                      */
  LCS_ERR_WORKSPACE = 8     /* workspace NULL or smaller than the *_workspace() size       */
} lcs_status;

enum { LCS_ROW_BF16 = 0, LCS_ROW_FP8_SPLIT = 1 };
/* flags of csa_index_topk: phi = ReLU instead of identity; run only the scoring or only the
 * selection phase; leave n SMs (0..255) free for work the caller runs next to the call (see
 * csa_index_topk) */
enum { LCS_INDEX_RELU = 1, LCS_INDEX_SCORE_ONLY = 2, LCS_INDEX_SELECT_ONLY = 4 };
#define LCS_INDEX_SPARE_SMS(n) ((int32_t)(((n) & 0xFF) << 8))

/* A batch: num_seqs sequences that each receive new tokens in this call (a prefill chunk,
 * one decode token, or several speculative tokens).  Sequence b holds seq_len[b] raw tokens
 * after the call; its new tokens are the last q_b = cu_new[b+1]-cu_new[b] of them, at
 * absolute positions seq_len[b]-q_b .. seq_len[b]-1, and they are also the queries.  Global
 * token / query index of new token i of sequence b: cu_new[b] + i.
 * The host fields are used for grid sizing and validation and must be upper bounds. */
typedef struct {
  int32_t num_seqs;          /* host                                                        */
  const int32_t* cu_new;     /* device int32[num_seqs+1], cu_new[0] = 0, non-decreasing      */
  const int32_t* seq_len;    /* device int32[num_seqs], seq_len[b] >= q_b                     */
  int32_t total_new;         /* host: cu_new[num_seqs]                                        */
  int32_t max_new;           /* host: >= every q_b                                            */
  int32_t max_seq_len;       /* host: >= every seq_len[b]                                     */
} lcs_batch;

/* A set of rows in the row format (see the file comment). */
typedef struct {
  int32_t format;            /* LCS_ROW_BF16 | LCS_ROW_FP8_SPLIT                             */
  int32_t dim;               /* D: 128 or 512                                                */
  int64_t num_rows;          /* rows the arrays hold (device-side bounds check)             */
  void* nope;                /* device; FP8: uint8[num_rows][D-64]; BF16: bf16[num_rows][D]  */
  void* rope;                /* device; FP8: bf16[num_rows][64]; BF16: NULL                  */
  float* scale;              /* device; FP8: f32[num_rows]; BF16: NULL                        */
} lcs_rows;

/* Paging of a per-sequence array of entries: entry j of sequence b lives in physical block
 * block_table[b*max_blocks_per_seq + j/entries_per_block], slot j % entries_per_block, i.e. at
 * row block*entries_per_block + slot.  entries_per_block = 128/m (32 for CSA, 1 for HCA). */
typedef struct {
  int32_t entries_per_block;
  int32_t max_blocks_per_seq;
  const int32_t* block_table;  /* device int32[num_seqs][max_blocks_per_seq]; < 0 = unmapped */
} lcs_paging;

/* Per-sequence state cache (x-techcon section 4: window rows and the uncompressed tail).
 *  window:   ring of the last 128 raw rows in the row format; token p of sequence b is row
 *            b*128 + p%128.  num_rows >= num_seqs*128.
 *  pending:  ring of raw BF16 rows not yet folded into a complete entry, plus (overlapping
 *            compressors) the previous block: token p of sequence b is row
 *            b*pending_slots + p%pending_slots of a bf16[num_seqs][pending_slots][D] array.
 *            pending_slots = 2m (overlap) or m.
 *  new_rows: rows of this call's new tokens in the row format (row = global token index), so
 *            that attention can read window rows of a multi-token chunk before they enter
 *            the ring.  If new_rows.nope is NULL, compress writes the ring itself: use it when
 *            the call is not followed by attention over the same tokens, or when every sequence
 *            has at most one new token (decode).  Token p then replaces token p-128, which is
 *            outside p's window, so attention can read the whole window from the ring and no
 *            lcs_window_commit is needed. */
typedef struct {
  lcs_rows window;
  void* pending;
  int32_t pending_slots;
  lcs_rows new_rows;
  void* pending_scores;      /* per-channel compressors only: bf16[num_seqs][pending_slots][D], the
                                score rows of the pending tokens (same ring as `pending`); else NULL */
} lcs_state;

/* Separate value rows (chenxutan.com/d/4230, section 4.5: the hybrid cache keeps K and V apart;
 * the other pages describe shared-KV attention, where the row is key and value).  Each set holds
 * the value row of the key row with the same number in its counterpart: entries <-> the entry
 * cache (same paging), window <-> state->window (same ring), new_rows <-> state->new_rows.  Each
 * set has its counterpart's format, dim and num_rows; new_rows.nope is NULL exactly when
 * state->new_rows.nope is.  Value entries are produced like key entries (csa_compress /
 * hca_compress over the raw value rows). */
typedef struct {
  lcs_rows entries;
  lcs_rows window;
  lcs_rows new_rows;
} lcs_values;

/* Compressor parameters.  Entry j uses tokens [(j-1)m, (j+1)m) with overlap, [jm, (j+1)m)
 * without; o = offset of token t in the entry's window (0 .. 2m-1 with overlap, 0 .. m-1
 * without); tokens before 0 are left out of the softmax.
 *  scalar weights (scores NULL; x-techcon section 2, CSA step 1):
 *    z_t = w . k_t + bias[o]; alpha = softmax over the window's rows; c = sum_t alpha_t k_t.
 *  per-channel weights (scores set; the compressor sketch of chenxutan.com/d/4230, section 4.2,
 *  with a per-offset bias): every raw token t comes with a score row s_t (D values, the output of
 *  the compressor's own score projection, computed by the caller like the raw KV rows);
 *    z[t,d] = s_t[d] + bias[o][d]; alpha[.,d] = softmax over the window's rows, channel by
 *    channel; c[d] = sum_t alpha[t,d] k_t[d].  Requires m <= 4 and state->pending_scores. */
typedef struct {
  const float* w;            /* device f32[D] (scalar weights; unused with scores)           */
  const float* bias;         /* device f32[2m] or f32[m]; with scores f32[2m][D] or f32[m][D] */
  int32_t m;                 /* ratio; a power of two dividing 128                            */
  int32_t overlap;           /* 1: overlapping windows of 2m rows                             */
  const void* scores;        /* device bf16[total_new][D]: score rows of this call's new tokens
                                (row = global token index), or NULL for scalar weights          */
} lcs_compressor;

/* Indexer keys: one per compressed entry, paged like the entries. */
typedef struct {
  const uint8_t* fp4;        /* device uint8[num_rows][rank/2]: E2M1 codes, element 2i in the low nibble */
  const uint8_t* scale;      /* device uint8[num_rows][rank/32]: UE8M0 per-32 block scales    */
  int32_t rank;              /* r: 64 or 128                                                  */
  int64_t num_rows;
} lcs_index_keys;

/* --- compression (x-techcon section 2, CSA step 1 and the HCA paragraph) ---------------------
 * Consumes the new raw rows raw[cu_new[b]+i] (device bf16[total_new][D], tokens at positions
 * seq_len[b]-q_b+i) and, for every sequence, writes the entries completed by them:
 * j in [floor(n0/m), floor(n1/m)) with n0 = seq_len-q_b, n1 = seq_len, quantised into
 * `entries` through `paging`.  Updates state->pending and writes state->new_rows (or, when
 * new_rows.nope is NULL, the window ring).  csa_compress accepts any ratio with overlap = 1 or 0;
 * hca_compress requires overlap = 0.  Supported: D in {128, 512}, m a power of two <= 128. */
lcs_status csa_compress(const lcs_batch* batch, const void* raw, const lcs_compressor* comp,
                        const lcs_state* state, const lcs_rows* entries, const lcs_paging* paging,
                        int32_t* dev_status, void* stream);
lcs_status hca_compress(const lcs_batch* batch, const void* raw, const lcs_compressor* comp,
                        const lcs_state* state, const lcs_rows* entries, const lcs_paging* paging,
                        int32_t* dev_status, void* stream);

/* Moves the window rows of this call's new tokens from state->new_rows into the window ring
 * (the last min(q_b, 128) of each sequence).  Call it after the attention of the same tokens. */
lcs_status lcs_window_commit(const lcs_batch* batch, const lcs_state* state, int32_t* dev_status,
                             void* stream);

/* --- lightning indexer + top-k (x-techcon section 2, CSA step 2; section 4, FP4 QK path) -----
 * For query i at position t and every visible entry j < N(t) = floor((t+1)/m):
 *   score(i,j) = sum_h w[i,h] * phi( sum_c qhat[i,h,c] * khat[j,c] ),
 * qhat/khat = E2M1 value * 2^(ue8m0-127) of its 32-element block, phi = identity or ReLU
 * (flags & LCS_INDEX_RELU).  Scores are computed exactly (fp32, every partial sum exact) when
 * block exponents of q and k stay within [-8, 8] of 0 and head weights are powers of two times
 * at most 2 significant bits; outside that range they round like fp32 sums.
 * out_idx[i][0..k) receives the min(k, N(t)) entries with the largest scores (ties: lower j),
 * in ascending j, padded with -1; out_cnt[i] = min(k, N(t)).
 *   q_fp4   device uint8[total_new][heads][rank/2]    q_scale device uint8[total_new][heads][rank/32]
 *   head_w  device f32[total_new][heads] or NULL (all 1)
 *   heads in {1, 2, 4, 8}; rank in {64, 128}; 1 <= k <= 4096.
 * Workspace: device, >= lcs_index_topk_workspace(batch, heads, keys, paging, m, k) bytes (the
 * same arguments as the call), 256-byte aligned.  Its first lcs_index_topk_workspace_zeroed()
 * bytes must hold zeros before the first call on it (e.g. cudaMemset once after allocation): they
 * are per-sequence counters and per-query thresholds that every completed call leaves at zero
 * again.  After a call whose device status is LCS_ERR_TIMEOUT, zero them again before reusing the
 * workspace.
 * How the work is split: at rank 128 with 1, 2, 4 or 8 heads, 9k/8 + 256 <= 4096 and up to 16
 * queries per sequence, the scoring runs on the tensor cores with the top-k fused into it -- a CTA
 * scores a run of the cache for a group of up to 4 queries of a sequence and keeps each query's
 * best entries, the runs of a query share the best threshold any of them has reached, and the
 * group's last CTA merges the runs' lists -- and the workspace holds only those lists (at most
 * about 8 k bytes per query and run); otherwise (longer query runs, rank 64) every score's
 * order-preserving key is written to the workspace (4 bytes per query and visible entry) and a
 * selection pass reads them back.
 * Phases: a call runs the scoring phase and the selection phase.  With LCS_INDEX_SCORE_ONLY it
 * runs only the first (the scores, or the runs' lists, into the workspace), with
 * LCS_INDEX_SELECT_ONLY only the second (the selection from the workspace into out_idx,
 * out_cnt), which reads what an earlier scoring call with the same batch, heads, keys, paging, m,
 * k and workspace left there (it must be ordered after it: same stream or an event); the pair gives
 * exactly the result of one call.  Both flags at once: LCS_ERR_INVALID_ARG.
 * Sharing the GPU: with LCS_INDEX_SPARE_SMS(n) the scoring kernel sizes its grid for n SMs fewer
 * than the GPU has (at least 16 remain), so that kernels the caller runs next to it on another
 * stream -- e.g. the window part of attention, one CTA of about 208 KB of shared memory per query
 * and 64-head group -- find whole SMs free instead of waiting for the scorer's CTAs to drain.  The
 * result is the same; the workspace size above covers every n. */
size_t lcs_index_topk_workspace(const lcs_batch* batch, int32_t heads, const lcs_index_keys* keys,
                                const lcs_paging* paging, int32_t m, int32_t k);
/* Leading bytes of that workspace that must be zero before its first use (see above). */
size_t lcs_index_topk_workspace_zeroed(const lcs_batch* batch);
lcs_status csa_index_topk(const lcs_batch* batch, const uint8_t* q_fp4, const uint8_t* q_scale,
                          const float* head_w, int32_t heads, const lcs_index_keys* keys,
                          const lcs_paging* paging, int32_t m, int32_t k, int32_t flags,
                          int32_t* out_idx, int32_t* out_cnt, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, void* stream);
/* The exact fp32 scores themselves: out_scores[i*ld + j] for j < N(t); other slots untouched.
 * ld >= floor(max_seq_len/m).  For verification and analysis. */
lcs_status csa_index_scores(const lcs_batch* batch, const uint8_t* q_fp4, const uint8_t* q_scale,
                            const float* head_w, int32_t heads, const lcs_index_keys* keys,
                            const lcs_paging* paging, int32_t m, int32_t flags, float* out_scores,
                            int64_t ld, int32_t* dev_status, void* stream);

/* Same as csa_index_topk for callers that cannot allocate device memory (for example code
 * running while another framework captures a CUDA graph, or a runtime that hands out all device
 * memory from its own pool at start-up): no workspace argument; the scratch is a fixed array of
 * LCSA_NOALLOC_SCRATCH_BYTES in the library's device image, reserved on every GPU that loads the
 * library until the process exits.  Not a step of the method: the pages have no counterpart.
 *  - Requests needing more scratch than that (lcs_index_topk_workspace(batch, heads, keys, paging,
 *    m, k) > LCSA_NOALLOC_SCRATCH_BYTES) return LCS_ERR_WORKSPACE and launch nothing.
 *  - The array starts as zeros when the library is loaded and every completed call leaves its
 *    leading counters at zero (see csa_index_topk); a call whose device status is LCS_ERR_TIMEOUT
 *    may leave them non-zero, and later calls then report LCS_ERR_DEVICE_GUARD.
 *  - A call with LCS_INDEX_SELECT_ONLY reads what the last LCS_INDEX_SCORE_ONLY call left in the
 *    array: same batch, heads, keys, paging, m and k, ordered after it, with no other call to this
 *    entry point in between.
 *  - Runs on the current device.  Its first call on a device looks up the array's device
 *    address (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Calls no allocator.  All calls share the array: calls whose kernels overlap on the GPU
 *    race and must be ordered by the caller. */
#define LCSA_NOALLOC_SCRATCH_BYTES (8u << 20)
lcs_status csa_index_topk_noalloc(const lcs_batch* batch, const uint8_t* q_fp4, const uint8_t* q_scale,
                                  const float* head_w, int32_t heads, const lcs_index_keys* keys,
                                  const lcs_paging* paging, int32_t m, int32_t k, int32_t flags,
                                  int32_t* out_idx, int32_t* out_cnt, int32_t* dev_status, void* stream);

/* --- attention (x-techcon section 2, CSA step 3 and the HCA paragraph) -----------------------
 * For query i (position t of sequence b) and every head h: one softmax over the rows
 *   CSA: the entries topk_idx[i][0..cnt) (cnt = topk_cnt[i], or the count of non-negative
 *        values when topk_cnt is NULL; every index must be below N(t) = floor((t+1)/m)),
 *        then window tokens max(0,t-127) .. t;
 *   HCA: the entries 0 .. N(t)-1, N(t) = floor((t+1)/m), then the same window tokens;
 * logits = softmax_scale * q[i,h,:] . row, o[i,h,:] = sum p * row (shared KV: the row is key
 * and value), or, with `values` set, o[i,h,:] = sum p * value row (the row with the same number in
 * the matching set of *values; values NULL = shared KV).  With values set the calls run the
 * warp-MMA kernel (csa_attend_window then launches nothing and csa_attend_topk computes
 * everything); value rows obey the row bounds below and a value row outside them is left out of
 * the softmax with LCS_ERR_DEVICE_GUARD.
 * sink: device f32[heads] or NULL: a per-head logit (natural log, not scaled by softmax_scale)
 * that joins every softmax denominator and carries no value, o = sum_r p_r v_r / (sum_r p_r +
 * e^sink), out_lse = log(sum_r e^logit_r + e^sink) (the csdn attention-details table names an
 * attention sink; this is the common learned-sink reading); finite values; the same result as
 * lcs_attention_sink applied to the call's outputs, rounded once.  csa_attend_window takes none.  Window token p is read from state->new_rows when p is one of this call's new
 * tokens (p >= seq_len-q_b) and from the window ring otherwise; with new_rows.nope NULL every
 * window row comes from the ring, which requires batch->max_new <= 1 (LCS_ERR_SHAPE otherwise).
 *   q       device bf16[total_new][heads][D]    out device bf16[total_new][heads][D]
 *   out_lse device f32[total_new][heads] (natural log of the softmax denominator) or NULL
 *   heads in {8, 16, 64, 128} (multiples of 16 up to 128, or 8); D in {128, 512}.
 * FP8-split rows: query values of the FP8 dims must lie within the f16 range; a row's scale s_r
 * must stay below 256 (|x| < 114688 before quantisation) and, at D = 512, its RoPE values within
 * 65504 * s_r (the kernels compute in f16 on the rows divided by s_r).  A row outside these bounds
 * is left out of the softmax and LCS_ERR_DEVICE_GUARD is reported.
 * Workspace: device, >= lcs_attend_workspace(batch, heads, D, max_rows) bytes, where max_rows
 * bounds the rows of one query (CSA: k + 128; HCA: floor(max_seq_len/m) + 128); the size covers
 * calls with and without values.
 * Errors (nothing launched): LCS_ERR_SHAPE for value sets whose format, dim or num_rows differ
 * from their key counterparts. */
size_t lcs_attend_workspace(const lcs_batch* batch, int32_t heads, int32_t dim, int32_t max_rows);
lcs_status csa_attend(const lcs_batch* batch, const void* q, int32_t heads, const int32_t* topk_idx,
                      const int32_t* topk_cnt, int32_t k, int32_t m, const lcs_rows* entries,
                      const lcs_paging* paging, const lcs_state* state, const lcs_values* values,
                      const float* sink, float softmax_scale, void* out, float* out_lse, void* workspace,
                      size_t workspace_bytes, int32_t* dev_status, void* stream);
/* csa_attend in two calls, so that the sliding-window part, which does not depend on the top-k
 * selection, can run while the indexer does (CSA step 3 of x-techcon section 2 attends the window
 * rows and the selected entries in one softmax; splitting the rows and merging the per-part
 * (max, sum, weighted sum) partials is exact up to rounding).
 *  csa_attend_window: the window rows of every query into the workspace (no output yet).
 *  csa_attend_topk:   the selected entries, then the merge with the window part into out/out_lse.
 * Arguments as for csa_attend (the window call needs no top-k list).  Both calls must get the same
 * batch, heads, k, m, row sets and workspace, and the window call must complete before the top-k
 * call's merge starts (same stream, or an event).  csa_attend_window + csa_attend_topk give
 * exactly the bits of csa_attend.  The library computes the window part apart only for D = 512
 * FP8-split rows, up to 128 heads, k <= 2048 and at most half as many (query, 64-head group)
 * pairs as the GPU has SMs; otherwise (other shapes, or runs of queries that fill the GPU by
 * themselves, or calls with values) csa_attend_window launches nothing and csa_attend_topk
 * computes everything. */
lcs_status csa_attend_window(const lcs_batch* batch, const void* q, int32_t heads, int32_t k, int32_t m,
                             const lcs_rows* entries, const lcs_paging* paging, const lcs_state* state,
                             const lcs_values* values, float softmax_scale, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, void* stream);
lcs_status csa_attend_topk(const lcs_batch* batch, const void* q, int32_t heads, const int32_t* topk_idx,
                           const int32_t* topk_cnt, int32_t k, int32_t m, const lcs_rows* entries,
                           const lcs_paging* paging, const lcs_state* state, const lcs_values* values,
                           const float* sink, float softmax_scale, void* out, float* out_lse, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, void* stream);
lcs_status hca_attend(const lcs_batch* batch, const void* q, int32_t heads, int32_t m,
                      const lcs_rows* entries, const lcs_paging* paging, const lcs_state* state,
                      const lcs_values* values, const float* sink, float softmax_scale, void* out, float* out_lse,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/* --- indexer key / query production: block-scaled FP4 (x-techcon section 4) -------------------
 * Quantises BF16 rows x[rows][r] (r a multiple of 32, at most 4096) to E2M1 codes
 * codes[rows][r/2] (two per byte, even element in the low nibble) and UE8M0 scale bytes
 * scales[rows][r/32], the layout csa_index_topk reads for keys and queries.  Per 32-element
 * block: the scale is the smallest power of two 2^e with amax <= 6 * 2^e (so nothing saturates),
 * e clamped to [-127, 127] (all-zero blocks: e = -127, byte 0); each element is x / 2^e rounded to
 * the nearest E2M1 value, ties to the code with mantissa bit 0, zero stored as +0.  (The pages fix
 * the format, not the scale choice: this is the reading taken.)  x: device, 16-byte aligned;
 * codes: device, 8-byte aligned; scales: device.  NaN / infinite inputs are not supported.  Errors: LCS_ERR_UNSUPPORTED
 * for r outside the range, LCS_ERR_INVALID_ARG for NULL buffers; nothing is launched then. */
lcs_status lcs_quantize_e2m1(const void* x, int64_t rows, int32_t r, uint8_t* codes, uint8_t* scales, void* stream);

/* --- attention sink (a per-head logit in every softmax denominator, carrying no value) ----------
 * The standalone form, for outputs of calls made without `sink` (the attention calls fold the
 * same term into their own normalisation).
 * Applied after csa_attend / csa_attend_topk / hca_attend from their outputs and log-sum-exp:
 *   out[i,h,:] *= 1 / (1 + exp(sink[h] - lse[i,h])),  lse[i,h] = log(exp(lse[i,h]) + exp(sink[h])),
 * which equals attention whose softmax has one more term exp(sink[h]) per head.  (The pages name
 * an attention sink without defining it; this is the common learned-sink definition.)
 *   out device bf16[total_new][heads][dim] (16-byte aligned, updated in place),
 *   out_lse device f32[total_new][heads] (natural log, updated in place), sink device f32[heads]
 *   in the logits' units (softmax_scale * q . row).  dim a multiple of 8.
 * Errors: LCS_ERR_UNSUPPORTED for sizes out of range, LCS_ERR_INVALID_ARG for NULL buffers. */
lcs_status lcs_attention_sink(void* out, float* out_lse, const float* sink, int64_t total_new, int32_t heads,
                              int32_t dim, void* stream);

/* --- staging copies (serving input/output; not a step of the method) --------------------------
 * Copies n <= 8 buffers, bytes[i] bytes from src[i] to dst[i], with one kernel on `stream` whose
 * threads load and store the bytes themselves.  Each pointer may be device memory or pinned host
 * memory (cudaHostAlloc / cudaHostRegister; it is used through its device alias), so a step's
 * inputs can be read straight from pinned host pages: for MB-sized inputs this is several times
 * faster than the copy engine on B300.  Buffers must not overlap.  16-byte aligned pairs move in
 * 16-byte pieces.  Errors: LCS_ERR_UNSUPPORTED for n > 8, LCS_ERR_INVALID_ARG for a NULL or
 * pageable pointer of a non-empty copy; nothing is launched then.  Capturable in a CUDA graph
 * (the pointer lookups happen on the host at call time). */
lcs_status lcs_stage_copy(int32_t n, void* const* dst, const void* const* src, const size_t* bytes, void* stream);

/* --- bounded waits --------------------------------------------------------------------------
 * Every wait of a kernel on one of its own pipeline stages (tensor-core completion, TMA arrival)
 * gives up after a bounded number of polls of up to about a microsecond each, records
 * LCS_ERR_TIMEOUT in the call's device status word and lets the kernel finish without its
 * results (it waits for its own copies still in flight first).  The bound applies to the calls
 * made after this one on any host thread; default LCSA_DEFAULT_WAIT_POLLS (about a second).  0 makes
 * every such wait give up at once: for testing the error path only.  Returns the previous bound. */
uint32_t lcs_set_wait_polls(uint32_t polls);

/* --- tensor-pipe throughput probe (measurement; not a step of the method) ---------------------
 * Launches `ctas` CTAs (one per SM is the intended use) that each issue mmas_per_cta tcgen05 MMAs of
 * M = 128 back to back from shared memory into tensor memory: kind 0 = kind::f8f6f4 with E2M1
 * operands, N = 256, K = 32 (the indexer's MMA); kind 1 = kind::f16 with F16 operands, N = 256,
 * K = 16 (the attention's MMA); kind 2 = kind::mxf4, block-scaled E2M1 operands packed two codes a
 * byte with a UE8M0 scale per 32 codes, N = 240, K = 64.  The caller times the launch and divides
 * 2 * 128 * N * K * mmas_per_cta * ctas by the time.  mmas_per_cta >= 64.  Errors:
 * LCS_ERR_UNSUPPORTED for other kinds or sizes. */
lcs_status lcs_mma_probe(int32_t kind, int32_t mmas_per_cta, int32_t ctas, int32_t* dev_status, void* stream);

/* --- library information -------------------------------------------------------------------- */
int32_t lcs_abi_version(void);
const char* lcs_status_string(int32_t status);
/* LCS_OK when the current device can run the library's kernels (compute capability 10.3). */
lcs_status lcs_device_check(void);

#ifdef __cplusplus
}
#endif
#endif /* LCSA_H_ */
