/*
 * dsa.h -- C ABI of the DeepSeek Sparse Attention (DSA) decode hot path for
 * NVIDIA GB300 (sm_103a).
 *
 * The path (Eq. (1) and Eq. (2) of "Feature Request: DeepSeek V3.2-Exp
 * support", llama.cpp issue 16331, section "1. Architecture"):
 *
 *   1. lightning-indexer logits over a paged FP8 key cache  dsa_indexer_logits
 *   2. exact per-row top-k of the logits                    dsa_topk
 *   3. sparse MLA attention over the selected latents       dsa_sparse_mla_decode
 *
 * and the two-level candidate-block indexer of the vLLM "sparse_indexer"
 * backend page (consumer layers score only the candidate blocks):
 *
 *   a. candidate expansion, once per step                   dsa_candidate_expand
 *   b. candidate (sparse MQA) logits over MXFP4 keys        dsa_candidate_logits
 *   c. top-k over the candidate columns, mapped to tokens   dsa_topk (col_blocks)
 *   (b and c also with bf16 logits:  dsa_candidate_logits_bf16, dsa_topk_bf16)
 *
 * and a multi-layer decode step with the IndexCache / Multi-layer Indexer
 * selection schedules (JEV Paper Radar efficiency digest) dsa_decode_layers
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Pointers documented as "device" point to GPU memory of the current
 *   device; the caller allocates, owns and frees every buffer.  The library
 *   allocates no memory per call: scratch comes from a caller-provided
 *   workspace whose size the matching *_size query returns.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *   only enqueues work and returns; nothing is synchronised.
 * - The indexer, top-k and sparse-attention kernels are launched with
 *   programmatic stream serialization: one of them may be placed on the GPU
 *   while the kernel before it in the stream finishes, but it waits for that
 *   kernel to complete (and for its writes to be visible) before it reads or
 *   writes any memory.  Stream order is kept exactly as for plain launches.
 * - Every argument is validated on the host before anything is enqueued; an
 *   unsupported shape or a bad argument returns an error and enqueues nothing.
 *   There is no fallback path.  dsa_last_error() gives a message.
 * - Device-side checks (block-table entries outside the cache, selected
 *   indices outside a row, a wait that ran out) never trap: the kernel skips
 *   the access, records a bit in a per-device error word and finishes.
 *   dsa_get_device_error() reads (and optionally clears) that word.
 * - Query rows are flattened per request: row r = b * next_n + j (j = 0 ..
 *   next_n-1) is the j-th of the next_n consecutive query positions of
 *   request b.  It sees L_r = ctx_len[b] - (next_n - 1 - j) cached tokens
 *   (the cache already holds all next_n positions; a query sees itself).
 * - Caches are paged with 64-token pages: token t of request b lives in page
 *   block_table[b * bt_stride + t / 64], slot t % 64.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned buffer, ... */
  DSA_ERR_UNSUPPORTED = 2, /* a shape or device this library does not implement */
  DSA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the query said */
  DSA_ERR_CUDA = 4,        /* a CUDA runtime call failed (message has the code) */
  DSA_ERR_DEVICE = 5       /* the device error word is set (dsa_get_device_error) */
} dsa_status;

/* Bits of the device error word. */
#define DSA_DEVERR_TIMEOUT 0x1u   /* a bounded wait inside a kernel ran out */
#define DSA_DEVERR_BAD_PAGE 0x2u  /* block-table entry outside [0, num_pages) */
#define DSA_DEVERR_BAD_INDEX 0x4u /* selected index outside [0, L_r), or row_len > ld */
#define DSA_DEVERR_CAPACITY 0x8u  /* cutoff estimate missed; the exact full-row path ran */

/* Fixed problem sizes of the path (the indexer of Eq. (1) and the MLA of
 * Eq. (2) as the DeepSeek V3.2 pages size them). */
#define DSA_PAGE_TOKENS 64
#define DSA_INDEX_HEADS 64 /* H^I */
#define DSA_INDEX_DIM 128  /* d^I */
#define DSA_MLA_HEADS 128
#define DSA_MLA_DQK 576 /* 512 latent + 64 rope */
#define DSA_MLA_DV 512
#define DSA_MAX_TOPK 8192
#define DSA_HIST_BINS 4096 /* bins of a row's score histogram (dsa_indexer_logits_hist) */

/* Version of this ABI (major*100 + minor). */
int dsa_version(void);

/* Message of the last failing call made by this host thread ("" if none). */
const char* dsa_last_error(void);

/* Reads the device error word of the current device after synchronising
 * `stream`; clears it when `clear` != 0.  Returns DSA_OK (and *bits) or
 * DSA_ERR_CUDA. */
dsa_status dsa_get_device_error(void* stream, uint32_t* bits, int clear);

/* ------------------------------------------------------------------------
 * dsa_indexer_logits -- lightning-indexer logits, Eq. (1):
 *
 *   logits[r, t] = s_t * sum_h w[r,h] * sq[r,h] * ReLU(q'[r,h] . k'_t),  t < L_r
 *
 * which is I_{t,s} of Eq. (1) with q = sq * q' (per-head FP8 scale) and
 * k = s_t * k' (per-token FP8 scale; both scales are positive, so they leave
 * the ReLU).  FP8 is e4m3 ("fn": no inf; 0x7F/0xFF are NaN and unsupported).
 *
 *   q_fp8      device [R, 64, 128] e4m3 codes, R = num_req * next_n.
 *   q_scale    device [R, 64] f32, > 0.
 *   weights    device [R, 64] f32 (w of Eq. (1); any sign).
 *   k_cache    device; page p's 64 keys (128 e4m3 bytes each, slot-major) start
 *              at k_cache + p * k_page_stride bytes.  16-byte aligned, stride % 16 == 0.
 *   k_scale    device; page p's 64 f32 per-token scales start at
 *              k_scale + p * s_page_stride bytes.  16-byte aligned, stride % 16 == 0.
 *              (The canonical page is 8448 bytes: keys, then scales.)
 *   num_pages  pages in the cache (block-table entries must be < num_pages).
 *   block_table device [num_req, bt_stride] int32; only the first ceil(L/64)
 *              entries of a request are read.
 *   ctx_len    device [num_req] int32 (>= 0).  num_req <= 4096.
 *   next_n     query rows per request (1 = plain decode, 2 = MTP; a prefill
 *              chunk of n queries is next_n = n).  1 <= next_n <= 65536.
 *   logits     device [R, ld] f32; for each row only t < L_r is written.
 *              ld >= max L_r, ld % 4 == 0, 16-byte aligned.
 * Work: one TMA-fed tcgen05 (kind::f8f6f4) contraction per 128-token tile with
 * the ReLU, head weighting and key scale fused into the TMEM epilogue.
 * ---------------------------------------------------------------------- */
dsa_status dsa_indexer_logits(const uint8_t* q_fp8, const float* q_scale, const float* weights,
                              const uint8_t* k_cache, int64_t k_page_stride,
                              const uint8_t* k_scale, int64_t s_page_stride, int num_pages,
                              const int32_t* block_table, int64_t bt_stride,
                              const int32_t* ctx_len, int num_req, int next_n, float* logits,
                              int64_t ld, void* stream);

/* ------------------------------------------------------------------------
 * dsa_topk -- exact fine-grained token selection (the Top-k of Eq. (2)).
 *
 * For each row r: the k largest logits[r, c], c < row_len[r], as column
 * indices in any order; a row with row_len <= k returns all its columns
 * followed by -1.  Ties are broken towards the lower column, so the selected
 * set equals the first k of a stable sort by score descending.  -0.0 == +0.0.
 * NaN logits are unsupported.
 *
 * Long rows (row_len >= 8k, or longer than 40960) take the cutoff path
 * described for vLLM's persistent top-k: estimate a cutoff from a sample,
 * compact the survivors into shared memory in one pass over the row, finish
 * with an exact selection on them (redoing the row with the full-row radix if
 * the estimate missed).  Shorter rows take the full-row radix select over
 * their keys staged in shared memory.  `force_path`: 0 = that rule, 1 = always full-row, 2 = always
 * cutoff (for tests; the selected set is the same).
 *
 *   logits     device [R, ld] f32; ld % 4 == 0, 16-byte aligned.
 *   row_len    device [R] int32 (0 <= row_len <= ld).
 *   col_blocks NULL, or device [R, nb] int32: then column c is reported as token
 *              col_blocks[r, c / block_size] * block_size + c % block_size
 *              (the candidate path's sparse column -> token map).
 *   out_idx    device [R, k] int32.
 *   1 <= k <= DSA_MAX_TOPK.
 * ---------------------------------------------------------------------- */
dsa_status dsa_topk(const float* logits, int64_t ld, const int32_t* row_len, int R, int k,
                    const int32_t* col_blocks, int nb, int block_size, int32_t* out_idx,
                    int force_path, void* stream);

/* ------------------------------------------------------------------------
 * dsa_indexer_logits_hist + dsa_topk_hist -- the indexer and the top-k with
 * the top-k's first pass fused into the indexer's epilogue.
 *
 * dsa_indexer_logits_hist is dsa_indexer_logits that also counts every logit
 * it writes into a per-row histogram: hist[r, b] += #{t < L_r : the top 12
 * bits of key(logits[r, t]) == b}, where key is the order-preserving u32 of
 * the f32 (sign bit flipped for positives, all bits for negatives; -0.0 as
 * +0.0), so bin b holds the scores of one sign, exponent and 3 leading
 * mantissa bits, and the bins are ordered like the scores.  Decode only:
 * next_n <= 2, else DSA_ERR_UNSUPPORTED.
 * dsa_topk_hist is dsa_topk (no column map) that reads row r's histogram to
 * place its cutoff at once (the lower edge of the bin holding the k-th
 * largest score) instead of estimating it from a sample, and clears every
 * row's histogram to zero before it returns.
 *
 *   hist   device [R, DSA_HIST_BINS] uint32 (dsa_score_hist_size(R) bytes),
 *          16-byte aligned.  Zero-fill it once after allocating it; each
 *          dsa_indexer_logits_hist adds its counts and the dsa_topk_hist that
 *          follows leaves it zero again.  The result never depends on the
 *          histogram: one that does not count exactly row_len[r] scores is
 *          ignored (the sample estimate is used), and a cutoff that keeps
 *          fewer than k scores or more than fit is redone exactly.
 * ---------------------------------------------------------------------- */
size_t dsa_score_hist_size(int R);

dsa_status dsa_indexer_logits_hist(const uint8_t* q_fp8, const float* q_scale,
                                   const float* weights, const uint8_t* k_cache,
                                   int64_t k_page_stride, const uint8_t* k_scale,
                                   int64_t s_page_stride, int num_pages,
                                   const int32_t* block_table, int64_t bt_stride,
                                   const int32_t* ctx_len, int num_req, int next_n, float* logits,
                                   int64_t ld, uint32_t* hist, void* stream);

dsa_status dsa_topk_hist(const float* logits, int64_t ld, const int32_t* row_len, int R, int k,
                         uint32_t* hist, int32_t* out_idx, int force_path, void* stream);

/* dsa_topk over bf16 scores (the vLLM sparse_indexer page's pairing: bf16
 * sparse logits selected by a bf16 top-k).  Same arguments and result; each
 * score is widened to f32 exactly, so the selected set is the f32 one of the
 * same values (bf16 rounding makes ties frequent; they go to the lower
 * column).  logits: device [R, ld] bf16, ld % 4 == 0, 16-byte aligned. */
dsa_status dsa_topk_bf16(const uint16_t* logits, int64_t ld, const int32_t* row_len, int R, int k,
                         const int32_t* col_blocks, int nb, int block_size, int32_t* out_idx,
                         int force_path, void* stream);

/* ------------------------------------------------------------------------
 * dsa_sparse_mla_decode -- sparse MLA attention, Eq. (2):
 *
 *   for head g of row r:  z_j = sm_scale * q[r,g,:] . c_{idx[r,j]}   (576-d)
 *                         out[r,g,:] = sum_j softmax(z)_j c_{idx[r,j]}[0:512]
 *                         lse[r,g]   = log sum_j exp(z_j)           (natural log)
 *
 * over the valid selected tokens only (idx = -1 is skipped; a row with none
 * gives out = 0, lse = -inf).  An index whose page is outside the request's
 * block-table row (idx / 64 >= bt_stride) or whose block-table entry is
 * outside [0, num_pages) is skipped the same way and sets
 * DSA_DEVERR_BAD_INDEX.  Token positions are logical positions of the
 * row's request (row r belongs to request r / next_n) and go through the block
 * table.  bf16 inputs, f32 accumulation and softmax, bf16 output.
 *
 *   q         device [R, 128, 576] bf16.
 *   kv_cache  device; page p = [64, 576] bf16 at kv_cache + p * kv_page_stride
 *             bytes; the pages must be contiguous (kv_page_stride == 73728) and
 *             kv_cache 16-byte aligned (the gathers use one TMA map over the cache).
 *   idx       device [R, k] int32, 1 <= k <= DSA_MAX_TOPK.
 *   out       device [R, 128, 512] bf16.   lse  device [R, 128] f32 (may be NULL).
 *   workspace device, dsa_sparse_mla_workspace_size(R, k) bytes (split-K
 *             partial results; may be NULL when that size is 0).
 *
 * The rows' selections are split (split-K) only while the CTA pairs of all
 * rows and splits still fit the device's SMs in one wave, so the workspace
 * size depends on the SM count of the device current when it is asked for
 * (152 on GB300; 152 is also assumed when no device can be queried): ask on
 * the device that will run the call.
 * ---------------------------------------------------------------------- */
size_t dsa_sparse_mla_workspace_size(int R, int k);

dsa_status dsa_sparse_mla_decode(const uint16_t* q, const uint16_t* kv_cache,
                                 int64_t kv_page_stride, int num_pages,
                                 const int32_t* block_table, int64_t bt_stride, int num_req,
                                 int next_n, const int32_t* idx, int k, float sm_scale,
                                 uint16_t* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dsa_sparse_mla_decode_static -- dsa_sparse_mla_decode for callers that
 * cannot allocate device memory.  (No counterpart in the paper: this is an
 * interface convenience of this library, not part of the method.)
 *
 * Who needs it: code that is not allowed to call cudaMalloc -- for example a
 * plug-in running inside a host program that owns all device memory and
 * hands out no allocator, or a latency-critical loop that cannot afford the
 * implicit device synchronisation a cudaMalloc may cause -- and so cannot
 * provide the workspace of dsa_sparse_mla_decode.
 *
 * Same arguments and results as dsa_sparse_mla_decode, without the workspace:
 * the split-K partial results go to a scratch array compiled into the library
 * (dsa_sparse_mla_static_scratch_bytes() = 24 MiB, held on every GPU that
 * loads the library until the process exits).  The work split is the same as
 * dsa_sparse_mla_decode's, so the outputs are the same.  A batch whose
 * partials would not fit returns DSA_ERR_UNSUPPORTED with the size it needs
 * (use dsa_sparse_mla_decode then).  Nothing is allocated, by this call or by
 * the library.
 *
 * The first call on a device, whatever its batch, looks up that device's
 * scratch address (cudaGetSymbolAddress, once per device, with the device
 * current); make that first call before any stream capture.  All calls on a device share the one
 * scratch array and it keeps the previous call's contents (no part of it has
 * to start at zero: each call writes every value it reads back); calls that
 * overlap on the GPU -- on two streams, or from two host threads -- race on
 * it, so serialise them.
 * ---------------------------------------------------------------------- */
size_t dsa_sparse_mla_static_scratch_bytes(void);

dsa_status dsa_sparse_mla_decode_static(const uint16_t* q, const uint16_t* kv_cache,
                                        int64_t kv_page_stride, int num_pages,
                                        const int32_t* block_table, int64_t bt_stride,
                                        int num_req, int next_n, const int32_t* idx, int k,
                                        float sm_scale, uint16_t* out, float* lse, void* stream);

/* ------------------------------------------------------------------------
 * dsa_candidate_expand -- the once-per-step candidate expansion shared by all
 * consumer indexer layers (vLLM sparse_indexer: sparse_indices, end and the
 * kernel schedule are filled by the first consumer layer and reused).
 *
 *   cand           device [R, nb] int32 candidate block ids (blocks of
 *                  block_size tokens) published by the source layer
 *                  (distinct; ids >= ceil(L/block_size) mark padding).
 *   block_size     candidate_block_size: m * 64 tokens, 1 <= m <= 64.  The
 *                  sparse blocks are 64-token pages (sparse_block_kv = 64): a
 *                  candidate block b is the m sparse blocks b*m .. b*m+m-1, so
 *                  a row has ns = nb * m sparse blocks (the page's
 *                  num_sparse_blocks = candidate_topk_blocks *
 *                  (candidate_block_size // sparse_block_kv)); ns <= 4096.
 *   sparse_indices device [R, ns] int32 out: the sparse block ids sorted
 *                  ascending.
 *   end            device [R] int32 out: valid sparse columns of the row, i.e.
 *                  #{c < ns*64 : 0 <= tok(c) < L_r}, tok(c) =
 *                  sparse_indices[r, c/64]*64 + c%64.  (Sorted ascending, the
 *                  valid columns are a prefix.)
 *   schedule       device, dsa_candidate_schedule_size(R) bytes out: the work
 *                  schedule dsa_candidate_logits reads.
 * The later calls take nb = ns and block_size = 64 (dsa_candidate_logits and
 * dsa_topk's col_blocks).
 * ---------------------------------------------------------------------- */
size_t dsa_candidate_schedule_size(int R);

dsa_status dsa_candidate_expand(const int32_t* cand, int R, int nb, int block_size,
                                const int32_t* ctx_len, int next_n, int32_t* sparse_indices,
                                int32_t* end, void* schedule, size_t schedule_bytes,
                                void* stream);

/* ------------------------------------------------------------------------
 * dsa_candidate_logits -- candidate (sparse MQA) logits over MXFP4 keys:
 *
 *   logits[r, c] = sum_h w[r,h] * sq[r,h] * ReLU(q'[r,h] . k_tok(c)),  c < end[r]
 *
 * with k the MXFP4-dequantised key: e2m1 elements (element 2i in the low
 * nibble of byte i) times a UE8M0 scale 2^(e-127) per 32 elements.
 *
 *   k_fp4     device, 32-byte aligned; page p's 64 keys (64 packed bytes
 *             each) at k_fp4 + p * k_page_stride bytes (k_page_stride >= 4096,
 *             a multiple of 32).
 *   k_sf      device; page p's 64 x 4 UE8M0 bytes (byte g of slot i scales
 *             elements 32g..32g+31) at k_sf + p * sf_page_stride bytes.
 *             (The canonical page is 4352 bytes: packed keys, then scales.)
 *   sparse_indices, end, schedule: as written by dsa_candidate_expand.
 *   logits    device [R, ld] f32, ld >= nb * block_size, ld % 4 == 0; only
 *             c < end[r] is written.
 * ---------------------------------------------------------------------- */
dsa_status dsa_candidate_logits(const uint8_t* q_fp8, const float* q_scale, const float* weights,
                                const uint8_t* k_fp4, int64_t k_page_stride, const uint8_t* k_sf,
                                int64_t sf_page_stride, int num_pages,
                                const int32_t* block_table, int64_t bt_stride, int num_req,
                                int next_n, const int32_t* sparse_indices, int nb,
                                int block_size, const int32_t* end, const void* schedule,
                                size_t schedule_bytes, float* logits, int64_t ld, void* stream);

/* dsa_candidate_logits writing bf16 logits (each the f32 result rounded to
 * nearest even), as the vLLM sparse_indexer page's kernels do: half the bytes
 * written here and read by dsa_topk_bf16.  logits: device [R, ld] bf16. */
dsa_status dsa_candidate_logits_bf16(const uint8_t* q_fp8, const float* q_scale,
                                     const float* weights, const uint8_t* k_fp4,
                                     int64_t k_page_stride, const uint8_t* k_sf,
                                     int64_t sf_page_stride, int num_pages,
                                     const int32_t* block_table, int64_t bt_stride, int num_req,
                                     int next_n, const int32_t* sparse_indices, int nb,
                                     int block_size, const int32_t* end, const void* schedule,
                                     size_t schedule_bytes, uint16_t* logits, int64_t ld,
                                     void* stream);

/* ------------------------------------------------------------------------
 * Prefill in chunks (the vLLM sparse_indexer page: "the prefill chunker
 * (which budgets fp32 [rows, seq_len])", chunks of rows with per-row K
 * ranges that may come from several requests).
 *
 * dsa_prefill_chunk_plan (host) -- splits a batch's query rows into chunks.
 * Rows are taken request by request, position by position; a row of request
 * b needs a logits row of max(ctx_len[b], min_cols) columns (min_cols is the
 * page's min_split_seq_len), rounded up to a multiple of 4; a chunk's f32
 * scratch is rows x (its widest row) x 4 bytes, and rows join the current
 * chunk while that stays within budget_bytes (a row alone above it is a chunk
 * by itself).  Writes *num_pieces records pieces[4 i .. 4 i + 3] = (chunk,
 * request, row_begin, row_end): each chunk is a run of consecutive pieces,
 * each piece rows [row_begin, row_end) of one request.  q_len, ctx_len: host
 * [num_req].  DSA_ERR_WORKSPACE if more than max_pieces pieces are needed.
 *
 * A chunk is run as entries, one per piece: entry e = (request b, rows
 * [j0, j1)) has j1 - j0 rows, the last of which sees ctx_len[b] - (q_len[b] -
 * j1) tokens, and reads block-table row b.
 *
 * dsa_indexer_logits_varlen -- dsa_indexer_logits over entries of different
 * row counts: entry e's rows are [cu_rows[e], cu_rows[e+1]) (device
 * [num_entries + 1], total_rows = cu_rows[num_entries], every entry at most
 * max_rows rows), row cu_rows[e] + j of n_e sees ctx_len[e] - (n_e - 1 - j)
 * tokens of block-table row bt_rows[e] (device [num_entries]; NULL = row e),
 * and the block table has bt_num_rows rows.  q_fp8 / q_scale / weights /
 * logits have total_rows rows.  Entries whose row range is reversed or past
 * total_rows, and block-table rows outside [0, bt_num_rows), are skipped and
 * set DSA_DEVERR_BAD_INDEX / DSA_DEVERR_BAD_PAGE.
 *
 * dsa_varlen_row_lengths -- row_len[cu_rows[e] + j] = that row's token count
 * (device [total_rows]), the row_len dsa_topk takes.
 *
 * dsa_sparse_mla_decode_varlen -- dsa_sparse_mla_decode for R query rows whose
 * block-table rows are row_bt[r] (device [R]; rows outside [0, bt_num_rows)
 * read nothing and set DSA_DEVERR_BAD_PAGE); workspace as
 * dsa_sparse_mla_workspace_size(R, k).
 * ---------------------------------------------------------------------- */
dsa_status dsa_prefill_chunk_plan(const int32_t* q_len, const int32_t* ctx_len, int num_req,
                                  int64_t budget_bytes, int64_t min_cols, int32_t* pieces,
                                  int max_pieces, int* num_pieces);

dsa_status dsa_indexer_logits_varlen(const uint8_t* q_fp8, const float* q_scale,
                                     const float* weights, const uint8_t* k_cache,
                                     int64_t k_page_stride, const uint8_t* k_scale,
                                     int64_t s_page_stride, int num_pages,
                                     const int32_t* block_table, int64_t bt_stride,
                                     int bt_num_rows, const int32_t* bt_rows,
                                     const int32_t* ctx_len, const int32_t* cu_rows,
                                     int num_entries, int max_rows, int total_rows,
                                     float* logits, int64_t ld, void* stream);

dsa_status dsa_varlen_row_lengths(const int32_t* ctx_len, const int32_t* cu_rows, int num_entries,
                                  int total_rows, int32_t* row_len, void* stream);

dsa_status dsa_sparse_mla_decode_varlen(const uint16_t* q, const uint16_t* kv_cache,
                                        int64_t kv_page_stride, int num_pages,
                                        const int32_t* block_table, int64_t bt_stride,
                                        int bt_num_rows, const int32_t* row_bt, int R,
                                        const int32_t* idx, int k, float sm_scale, uint16_t* out,
                                        float* lse, void* workspace, size_t workspace_bytes,
                                        void* stream);

/* ------------------------------------------------------------------------
 * dsa_decode_layers -- one decode step over several DSA layers with the
 * cross-layer selection schedules of the Multi-layer Indexer (MLI) abstract
 * ("JEV Paper Radar" efficiency digest, 2026-11-04):
 *
 *   IndexCache  only the layers with keep_indexer[l] != 0 run an indexer
 *               (dsa_indexer_logits + dsa_topk); the others attend an earlier
 *               layer's selection;
 *   MLI         (mli != 0) every layer attends the selection of the previous
 *               indexer layer instead of its own, which removes the dependency
 *               of its attention on its own indexer: that indexer and its
 *               top-k run on side_stream, concurrently with the attention.
 *
 * Layer l attends the selection of layer dsa_layer_sources(...)[l]: the
 * latest indexer layer j <= l (mli = 0) or j < l (mli != 0; layer 0, which
 * must keep its indexer, attends its own).  Each attention is one
 * dsa_sparse_mla_decode of that layer's q and latent cache with that
 * selection, so a layer's out / lse equal those of the three single calls
 * made in the schedule's order.
 *
 *   layers[l]      host array of num_layers records (below); the indexer
 *                  fields are read only for layers that keep an indexer.
 *   keep_indexer   host [num_layers]; keep_indexer[0] must be set.
 *   shared geometry: as dsa_indexer_logits (k_page_stride, s_page_stride,
 *                  num_pages, block_table, bt_stride, ctx_len, num_req,
 *                  next_n) and dsa_sparse_mla_decode (kv_page_stride,
 *                  sm_scale); every layer's caches use the same block table.
 *   row_len        device [R] int32: L_r of every query row (dsa_topk's row_len).
 *   k              selected tokens per row (1 <= k <= DSA_MAX_TOPK).
 *   ld             row stride of the logits scratch (>= max L_r, % 4 == 0).
 *   workspace      device, dsa_decode_layers_workspace_size(R, ld, k) bytes:
 *                  the logits, two selection buffers, the MLA split partials.
 *   stream         the step's stream: the attentions (and layer 0's indexer)
 *                  run on it, and it waits at the end for everything the call
 *                  put on side_stream.
 *   side_stream    a second stream for MLI's indexers, or NULL (then they run
 *                  on `stream`, with the same results and no overlap).
 * The call records and waits on CUDA events it creates once per host thread
 * and device.  All arguments are checked before anything is enqueued.
 * ---------------------------------------------------------------------- */
typedef struct dsa_layer {
  const uint8_t* q_fp8;     /* [R, 64, 128] e4m3 indexer query            */
  const float* q_scale;     /* [R, 64]                                    */
  const float* weights;     /* [R, 64]                                    */
  const uint8_t* k_cache;   /* the layer's FP8 key pages                  */
  const uint8_t* k_scale;   /* the layer's per-token key scales           */
  const uint16_t* q;        /* [R, 128, 576] bf16 attention query          */
  const uint16_t* kv_cache; /* the layer's latent pages                    */
  uint16_t* out;            /* [R, 128, 512] bf16                          */
  float* lse;               /* [R, 128] f32, or NULL                       */
} dsa_layer;

/* Host-only: src[l] = the layer whose selection layer l attends under the
 * schedule above.  DSA_ERR_INVALID_ARG if keep_indexer[0] == 0. */
dsa_status dsa_layer_sources(const uint8_t* keep_indexer, int num_layers, int mli, int32_t* src);

size_t dsa_decode_layers_workspace_size(int R, int64_t ld, int k);

dsa_status dsa_decode_layers(const dsa_layer* layers, int num_layers,
                             const uint8_t* keep_indexer, int mli, int64_t k_page_stride,
                             int64_t s_page_stride, int64_t kv_page_stride, int num_pages,
                             const int32_t* block_table, int64_t bt_stride,
                             const int32_t* ctx_len, const int32_t* row_len, int num_req,
                             int next_n, int k, float sm_scale, int64_t ld, void* workspace,
                             size_t workspace_bytes, void* stream, void* side_stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
