/*
 * locks.h - C ABI of the LOCKS page-local key-summary sparse decode library
 * (liblocks.so, sm_103a).
 *
 * The method: "LOCKS: Page-Local Compact Key Summaries for Efficient
 * Long-Context Decoding", as restated in the LOCKS reading notes
 * (zhongzhuzhou.org, 2026-07-29) and the gist.science technical summary.
 * Every entry point below names the passage that defines its operation.
 *
 * Conventions for every call
 *  - All array pointers are CUDA device pointers owned by the caller unless a
 *    comment says "host".  The library allocates no device memory, never
 *    synchronises the stream (except locks_read_status and
 *    locks_decoder_step_host, which say so) and launches its kernels on
 *    `stream` (NULL = the legacy default stream).
 *  - Shapes: page size B = 16 tokens, head dim d = 128, summary rank r = 8.
 *    K/V caches are bf16, laid out [num_phys_pages][h_kv][16][128] so that
 *    each (page, KV head) is one contiguous 4 KB run.
 *    page_table is int32 [batch][max_pages] (logical page -> physical page).
 *    Queries are bf16 [batch][h_q][128]; query head hq belongs to KV head
 *    hq / G with G = h_q / h_kv (1 <= G <= 16).
 *  - Host-detectable argument errors return a locks_status_t before anything
 *    is launched.  Data errors found on the device (a page id outside the
 *    cache, a selected index outside the sequence, a length above
 *    16*max_pages) never trap: the kernel skips the offending access and ORs
 *    a LOCKS_DEV_* bit into a device status word (first int32 of the
 *    workspace, or the explicit `status` pointer), which the caller reads
 *    with locks_read_status and clears with locks_clear_status.
 *  - Numerics: scoring feeds the tensor cores fp16 operands (summary codes
 *    exact; the query converted from bf16 after a power-of-two prescale per
 *    (sequence, KV head) that keeps it below 2^14, undone in fp32) with
 *    fp32 accumulation; any finite query is accepted.
 *
 * Summary record (one per (sequence, KV head, logical page)), 832 bytes,
 * 16-byte aligned, laid out so that the scoring kernel's tensor-core
 * fragments load with one 16-byte read per lane:
 *   [  0, 512)  V4  int4 basis codes, two's complement, in [-7, 7].
 *               128 little-endian u32 words.  The code of V[d][n] (d < 128,
 *               component n < 8) sits in word (4n + c)*4 + w at bit
 *               16e + 8sp + 4h, where c = (d%8)/2, e = d%2, h = (d%16)/8,
 *               s = d/16, w = s/2, sp = s%2.
 *   [512, 640)  C8  int8 coefficient codes C[i][n] (token i < 16), in
 *               [-127, 127], stored excess-128 (byte value = code + 128),
 *               at byte 512 + 4*(4*(i%8) + n/2) + 2*(i/8) + n%2.
 *   [640, 768)  MU8 int8 centroid codes mu[d], stored excess-128, at byte
 *               640 + 32*((d%8)/2) + 4*(d/16) + (d%2) + 2*((d%16)/8).
 *   [768, 832)  fp16 scales, four 16-byte groups: group t (0..3) at
 *               768 + 16t holds sV[2t], sV[2t+1] (per-column basis
 *               scales), sC[2t], sC[2t+1], sC[8+2t], sC[9+2t] (per-row
 *               coefficient scales), then the centroid scale sMU in group 0
 *               (byte 780) and zero padding elsewhere: each scoring lane
 *               reads all its scales with one 16-byte load.  25 scales =
 *               50 payload bytes; 14 bytes are padding.
 * Dequantised: mu = sMU*MU8, V[:,n] = sV[n]*V4[:,n], c_i = sC[i]*C8[i,:].
 * The summary store is [batch][h_kv][max_pages] records in logical page
 * order, so one (sequence, KV head) is a contiguous stream.
 */
#ifndef LOCKS_H
#define LOCKS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *locks_stream_t; /* same type as cudaStream_t */

typedef enum {
  LOCKS_OK = 0,
  LOCKS_ERR_INVALID_ARG = 1, /* null pointer, bad size, k < 2, ...      */
  LOCKS_ERR_UNSUPPORTED = 2, /* G outside 1..16, size above a limit:
                                batch above 1594 for the scoring and
                                selection calls (their per-sequence tables
                                sit on chip beside the summary ring),
                                above 41712 for sparse decode           */
  LOCKS_ERR_WORKSPACE = 3,   /* workspace smaller than locks_workspace_size */
  LOCKS_ERR_CUDA = 4         /* a CUDA call failed: locks_last_cuda_error */
} locks_status_t;

/* device status bits (OR-ed into the status word) */
#define LOCKS_DEV_BAD_PAGE_ID 0x1 /* page_table entry outside the cache   */
#define LOCKS_DEV_BAD_INDEX 0x2   /* selected page outside the sequence   */
#define LOCKS_DEV_BAD_SEQ_LEN 0x4 /* seq_len < 0 or > 16*max_pages        */
#define LOCKS_DEV_BAD_PAIR 0x8    /* build pair outside batch/max_pages   */
#define LOCKS_DEV_TIMEOUT 0x10    /* an on-chip copy wait gave up         */

/* GQA merge rules of the selection (LOCKS reading notes §4.2 design
 * discussion and the §6 ablation).  The shipped rule is the share-average
 * of Eq.(5); group-max ranks pages by the largest mass fraction any head of
 * the group gives them; group-mass by the group's pooled unnormalised page
 * mass sum_g exp(s_hat[g][j]).  Per-head selection (each query head its own
 * page set) needs no rule: call locks_select_pages with h_kv = h_q. */
/* Build flags (locks_build_summaries_ex, locks_append_kv_ex,
 * locks_pack_summaries_ex).  0 = one basis scale per column, as the reading
 * notes' Algorithm 1 stores it (the default).  LOCKS_BUILD_VSCALE_PER_PAGE
 * is the alternative reading of the basis scale: one fp16 scale
 * sV = fp16(max over all 128 x 8 entries of |V| / 7) for the whole page,
 * written into all eight column slots, so the record layout and every
 * scoring call are unchanged. */
#define LOCKS_BUILD_VSCALE_PER_PAGE 0x1

#define LOCKS_MERGE_SHARE_AVERAGE 0
#define LOCKS_MERGE_GROUP_MAX 1
#define LOCKS_MERGE_GROUP_MASS 2

#define LOCKS_PAGE_TOKENS 16
#define LOCKS_HEAD_DIM 128
#define LOCKS_RANK 8
#define LOCKS_RECORD_BYTES 832
#define LOCKS_RECORD_PAYLOAD_BYTES 818
#define LOCKS_UNQUANTISED_FLOATS 1296 /* 16 + 128 + 128*8 + 16*8 */

/* Human-readable name of a status code (static string). */
const char *locks_status_string(locks_status_t s);

/* cudaError_t of the last failing CUDA call in this thread (0 if none). */
int locks_last_cuda_error(void);

/* Kernels this process has launched through the library: every kernel
 * launch call (including one recorded into a stream capture) plus, for
 * every replay of a decoder's graph (locks_decoder_step_host), the kernels
 * the graph holds.  Monotone; read it before and after a region to count
 * the region's launches. */
long long locks_kernel_launches(void);

/* Bytes per summary record (832: 818 B payload + 14 B padding). */
size_t locks_summary_record_bytes(void);

/* Workspace bytes needed by locks_score_select, locks_select_pages and
 * locks_sparse_decode for these sizes (k = max_pages covers dense decode).
 * One workspace may serve those calls in stream order.  Its first int32 is
 * the device status word: clear it once (locks_clear_status) before use. */
locks_status_t locks_workspace_size(int batch, int h_q, int h_kv,
                                    int max_pages, int k, size_t *bytes);

/* Page summary build, LOCKS reading notes §4.1 Eq.(2)-(3), storage
 * paragraph, and §4.3 Algorithm 1: for each listed (seq_ids[i], page_ids[i])
 * pair and every KV head, centre the page's 16 keys on their mean, take the
 * top r = 8 eigenpairs of the 16x16 Gram matrix D D^T (descending; each
 * eigenvector signed so its largest-magnitude entry is positive), form
 * V = D^T U_r Sigma_r^{-1} and C = U_r Sigma_r, quantise (int4 V with a
 * per-column fp16 scale, int8 C with a per-row scale, int8 mean with one
 * scale; scale = fp16(absmax/qmax), code = round-half-even(x/scale)) and
 * write the record at summaries[seq][h][page].  Components with eigenvalue
 * <= 1e-6 * lambda_1 are stored as zero.  Only full pages should be listed
 * (the pages build a summary when a page fills).
 *   k_cache       bf16 [num_phys_pages][h_kv][16][128]
 *   page_table    int32 [batch][max_pages]
 *   seq_ids, page_ids  int32 [n_pairs]
 *   summaries     records [batch][h_kv][max_pages] (written for the pairs)
 *   tau_out       optional float [n_pairs][h_kv]: spectral tail
 *                 sum_{k>8} sigma_k^2 (the diagnostic of Algorithm 1)
 *   unquantised_out  optional float [n_pairs][h_kv][1296]: the fp32 values
 *                 before quantisation, per page-head in this order:
 *                 eigenvalues [16] (descending, clipped at 0), centroid
 *                 [128], basis V [128][8], coefficients C [16][8]
 *   status        optional int32 device status word (LOCKS_DEV_* bits) */
locks_status_t locks_build_summaries(
    const void *k_cache, int64_t num_phys_pages, int h_kv,
    const int32_t *page_table, int batch, int max_pages,
    const int32_t *seq_ids, const int32_t *page_ids, int n_pairs,
    void *summaries, float *tau_out, float *unquantised_out, int32_t *status,
    locks_stream_t stream);

/* locks_build_summaries with build flags (LOCKS_BUILD_*); flags = 0 is
 * locks_build_summaries.  Unknown flag bits return LOCKS_ERR_INVALID_ARG. */
locks_status_t locks_build_summaries_ex(
    const void *k_cache, int64_t num_phys_pages, int h_kv,
    const int32_t *page_table, int batch, int max_pages,
    const int32_t *seq_ids, const int32_t *page_ids, int n_pairs,
    void *summaries, float *tau_out, float *unquantised_out, int flags,
    int32_t *status, locks_stream_t stream);

/* Rank / precision variants of the page summary (LOCKS reading notes §6
 * ablation "rank and quantisation precision": int8, int4 and int2 bases at
 * several ranks).  A variant record of rank r in {4, 8, 12, 15} with a
 * basis of vbits in {2, 4, 8} bits is laid out, like the shipped record, so
 * that each scoring lane finds its tensor-core fragments in aligned words;
 * the (r = 8, 4-bit) variant record is the shipped 832-byte record, byte
 * for byte.  With t = (d%8)/2, e = d%2, h = (d%16)/8, s = d/16 for head dim
 * d, g = i%8 for token i, and C_OFF = 16 r vbits:
 *   [0, C_OFF)  basis codes V[d][k]: the 32 codes of component k with the
 *               same t form slot 4k + t (4*vbits bytes at 4*vbits*(4k + t));
 *               inside the slot, as little-endian u32 words,
 *                 vbits 4: word s/2, bit 16e + 8(s%2) + 4h, two's complement
 *                 vbits 2: word s/4, bit 16e + 2(2(s%4) + h), two's complement
 *                 vbits 8: byte 4s + 2h + e, excess-128 (byte = code + 128)
 *   C_OFF       int8 C[i][k], excess-128, at C_OFF plus
 *                 r <= 8: 4(g r/2 + k/2) + 2(i/8) + k%2            (16 r B)
 *                 r = 15: 32g + 8t' + 4(i/8) + 2(k/8) + k%2       (256 B)
 *                 r = 12: 24g + 8t' + 4(i/8) + 2(k/8) + k%2, but
 *                         24g + 16 + 4(t'-2) + 2(i/8) + k%2 when t' >= 2
 *                                                                 (192 B)
 *               with t' = (k%8)/2; unused bytes hold code 0 (byte 128)
 *   MU_OFF      int8 mu[128], excess-128, in the shipped record's order
 *               (MU_OFF = C_OFF + coefficient bytes)
 *   S_OFF       64-byte fp16 scale block (S_OFF = MU_OFF + 128): group t
 *               (16 bytes at S_OFF + 16t) holds sV[2t], sV[2t+1], sC[2t],
 *               sC[2t+1], sC[8+2t], sC[9+2t], then for r <= 8 sMU (group 0,
 *               byte 12) and zeros, for r > 8 sV[8+2t], sV[9+2t] (sMU in the
 *               sV[15] slot, byte 62); scales of absent components are 0
 * Record stride S_OFF + 64: 384, 512, 768 (r 4); 576, 832, 1344 (r 8);
 * 768, 1152, 1920 (r 12); 928, 1408, 2368 (r 15) bytes for 2-, 4-, 8-bit
 * bases.  Quantiser as the shipped record (symmetric, fp16 scale =
 * fp16_rn(absmax / qmax), qmax = 2^(vbits-1) - 1, codes rint(x / s)
 * clamped).
 * locks_variant_record_bytes: the stride (0 for an unsupported pair). */
size_t locks_variant_record_bytes(int rank, int vbits);

/* Algorithm 1 at rank `rank` with a `vbits`-bit basis for the listed
 * (seq_ids[i], page_ids[i]) pairs and every KV head, written to
 *   records  [batch][h_kv][max_pages] variant records of
 *            locks_variant_record_bytes(rank, vbits) bytes.
 * Other arguments, status bits and errors as locks_build_summaries. */
locks_status_t locks_build_variant(
    const void *k_cache, int64_t num_phys_pages, int h_kv,
    const int32_t *page_table, int batch, int max_pages,
    const int32_t *seq_ids, const int32_t *page_ids, int n_pairs, int rank,
    int vbits, void *records, float *tau_out, int32_t *status,
    locks_stream_t stream);

/* Eq.(4) page scores of every full page from variant records, in the
 * layout of locks_score_pages (scores_out float [batch][h_kv][G][max_pages];
 * entries of pages that are not full are left untouched).  Feed them to
 * locks_select_pages for the variant's selection.  `records` must be
 * 16-byte aligned (LOCKS_ERR_INVALID_ARG otherwise); batch is limited by
 * the per-sequence tables kept on chip beside the record ring (about 1600
 * sequences, LOCKS_ERR_UNSUPPORTED above). */
locks_status_t locks_score_variant(const void *q, const void *records,
                                   int rank, int vbits,
                                   const int32_t *seq_lens, int batch,
                                   int h_q, int h_kv, int max_pages,
                                   float *scores_out, int32_t *status,
                                   locks_stream_t stream);

/* Quantise and pack n given fp32 summaries into records with the same rule
 * as locks_build_summaries (the storage paragraph of §4.1).
 *   mu [n][128], basis [n][128][8] (V), coeffs [n][16][8] (C): float32
 *   records [n][832] */
locks_status_t locks_pack_summaries(const float *mu, const float *basis,
                                    const float *coeffs, int n,
                                    void *records, locks_stream_t stream);

/* locks_pack_summaries with build flags (LOCKS_BUILD_*). */
locks_status_t locks_pack_summaries_ex(const float *mu, const float *basis,
                                       const float *coeffs, int n,
                                       void *records, int flags,
                                       locks_stream_t stream);

/* Score and select, LOCKS reading notes §4.2 Eq.(4)-(5) and §4.4
 * Algorithm 2, one decode step: for every full page j of every (sequence b,
 * KV head h) and each query head g of its group,
 *   s_hat[g][j] = log sum_i exp((q_g.mu_j + (V_j^T q_g).c_i) / sqrt(128)),
 * from the summary records alone; then mass fractions
 * m_g(j) = exp(s_hat[g][j]) / sum_{j' full} exp(s_hat[g][j']), their group
 * average m_bar_j (Eq.(5)), and the selection: the sink page 0, the recent
 * page ceil(L/16)-1 and the k-2 other pages of largest m_bar (ties to the
 * lower page); all pages when ceil(L/16) <= k.
 *   q          bf16 [batch][h_q][128]
 *   summaries  records [batch][h_kv][max_pages], built for every full page
 *   seq_lens   int32 [batch] (tokens; a partial last page has no summary)
 *   idx_out    int32 [batch][h_kv][k]: selected logical pages, ascending,
 *              -1 padded when a sequence has fewer than k pages
 *   workspace  >= locks_workspace_size bytes; after the call, bytes
 *              [256, 256 + 4*batch*h_kv*G*max_pages) hold the scores s_hat
 *              as float [batch][h_kv][G][max_pages] (full pages only) */
locks_status_t locks_score_select(const void *q, const void *summaries,
                                  const int32_t *seq_lens, int batch, int h_q,
                                  int h_kv, int max_pages, int k,
                                  int32_t *idx_out, void *workspace,
                                  size_t workspace_bytes,
                                  locks_stream_t stream);

/* Scoring alone (§4.2 Eq.(4)): writes the natural-log page scores
 * s_hat[g][j] of every full page to scores_out, float
 * [batch][h_kv][G][max_pages] (entries of pages that are not full are left
 * untouched).  locks_score_select = locks_score_pages + locks_select_pages.
 *   status  optional int32 device status word */
locks_status_t locks_score_pages(const void *q, const void *summaries,
                                 const int32_t *seq_lens, int batch, int h_q,
                                 int h_kv, int max_pages, float *scores_out,
                                 int32_t *status, locks_stream_t stream);

/* Exact page scores (LOCKS reading notes §4.2 Eq.(4), the quantity the
 * summaries estimate; ranking by it is the exact-mass selector of §6
 * Fig. 1(b) and Fig. 2, which reads every key): for every full page j of
 * every (b, KV head) and query head g,
 *   scores_out[b][h][g][j] = ln sum_{i < 16} exp(q_g . k_i / sqrt(128))
 * in the layout of locks_score_pages (entries of pages that are not full
 * are left untouched; a page whose physical id is out of range gets -inf
 * and sets LOCKS_DEV_BAD_PAGE_ID).  Feeding these scores to
 * locks_select_pages gives the exact-mass selection.
 *   q           bf16 [batch][h_q][128]
 *   k_cache     bf16 [num_phys_pages][h_kv][16][128]
 *   page_table  int32 [batch][max_pages];  seq_lens int32 [batch]
 *   scores_out  float [batch][h_kv][h_q/h_kv][max_pages] (device)
 *   status      optional int32 device status word
 * Returns LOCKS_ERR_UNSUPPORTED when batch * h_kv * max_pages exceeds
 * 2^31 - 1 or the per-sequence table does not fit in shared memory
 * (batch above about 48,000). */
locks_status_t locks_exact_page_scores(
    const void *q, const void *k_cache, int64_t num_phys_pages,
    const int32_t *page_table, const int32_t *seq_lens, int batch, int h_q,
    int h_kv, int max_pages, float *scores_out, int32_t *status,
    locks_stream_t stream);

/* Score and select without any caller workspace, for callers that may not
 * allocate device memory on the decode path (an engine whose memory plan is
 * frozen after start-up, or a plugin handed only its input and output
 * buffers).  The pages describe no such call; it exists for deployment.
 * Computes exactly what locks_score_select computes, with the page scores
 * and selection keys kept in a 16 MiB array built into the library (every
 * GPU that loads the library holds it until the process exits).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - Limit: 256-byte-rounded 4*batch*h_kv*G*max_pages (scores) plus
 *     4*batch*h_kv*max_pages (keys) must fit in 16 MiB, else
 *     LOCKS_ERR_UNSUPPORTED and nothing is launched.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: do not call this entry point on a device after
 *     cudaDeviceReset has been called for it (the array may then sit at
 *     another address).
 *   - Every call shares the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls that overlap on the GPU
 *     (on different streams) race on it.
 *   - status: optional int32 device status word (LOCKS_DEV_* bits).
 *   - On LOCKS_ERR_CUDA the CUDA error is not kept for
 *     locks_last_cuda_error.
 * Other arguments as locks_score_select. */
locks_status_t locks_score_select_static(const void *q, const void *summaries,
                                         const int32_t *seq_lens, int batch,
                                         int h_q, int h_kv, int max_pages,
                                         int k, int32_t *idx_out,
                                         int32_t *status,
                                         locks_stream_t stream);

/* Selection alone (Eq.(5) and the sink/recent rule of §4.2) from given
 * natural-log page scores scores[batch][h_kv][G][max_pages] (entries of
 * full pages are read; a score of exact LSE turns this into the exact-mass
 * selector).  Arguments as locks_score_select. */
locks_status_t locks_select_pages(const float *scores, const int32_t *seq_lens,
                                  int batch, int h_q, int h_kv, int max_pages,
                                  int k, int32_t *idx_out, void *workspace,
                                  size_t workspace_bytes,
                                  locks_stream_t stream);

/* locks_select_pages with the candidates ranked by another GQA merge rule
 * (LOCKS_MERGE_*; LOCKS_MERGE_SHARE_AVERAGE is locks_select_pages itself).
 * Same arguments, layouts and workspace; the sink and recent pages and the
 * tie rule are unchanged.  Returns LOCKS_ERR_INVALID_ARG for an unknown
 * rule. */
locks_status_t locks_select_pages_merge(const float *scores,
                                        const int32_t *seq_lens, int batch,
                                        int h_q, int h_kv, int max_pages,
                                        int k, int rule, int32_t *idx_out,
                                        void *workspace,
                                        size_t workspace_bytes,
                                        locks_stream_t stream);

/* Attention over the selected pages, LOCKS reading notes §2 (fetch full
 * K/V only for the selected pages, then standard softmax attention for all
 * G heads of the group) and §4.4 Algorithm 2: for each (b, query head),
 *   o = sum_t softmax_t(q.k_t / sqrt(128)) v_t,  lse = log sum_t exp(...)
 * over the tokens t = 16p + s (p in idx[b][h], s < 16, t < seq_lens[b]).
 *   idx      int32 [batch][h_kv][k] (-1 entries skipped); NULL means every
 *            page of the sequence (dense decode, used as a baseline)
 *   o_out    bf16 [batch][h_q][128];  lse_out float [batch][h_q] (natural
 *            log; -inf and o = 0 for a sequence with no tokens) */
locks_status_t locks_sparse_decode(
    const void *q, const void *k_cache, const void *v_cache,
    int64_t num_phys_pages, const int32_t *page_table,
    const int32_t *seq_lens, const int32_t *idx, int k, int batch, int h_q,
    int h_kv, int max_pages, void *o_out, float *lse_out, void *workspace,
    size_t workspace_bytes, locks_stream_t stream);

/* Append one generated token per sequence and build the summary of every
 * page this append fills (the build runs "when a page fills", LOCKS reading
 * notes §2, Fig. 1): token position L = seq_lens[b] is written to page
 * L/16 slot L%16 for every KV head, then, if (L+1) % 16 == 0, the record of
 * that page is built as in locks_build_summaries; seq_lens[b] becomes L+1.
 *   k_new, v_new  bf16 [batch][h_kv][128]
 *   seq_lens      int32 [batch], updated in place on the device
 *   tau_out       optional float [batch][h_kv] (written for built pages) */
locks_status_t locks_append_kv(const void *k_new, const void *v_new,
                               void *k_cache, void *v_cache,
                               int64_t num_phys_pages, int h_kv,
                               const int32_t *page_table, int batch,
                               int max_pages, int32_t *seq_lens,
                               void *summaries, float *tau_out,
                               int32_t *status, locks_stream_t stream);

/* locks_append_kv with build flags (LOCKS_BUILD_*) for the pages it
 * builds; use the flags the store was built with. */
locks_status_t locks_append_kv_ex(const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache,
                                  int64_t num_phys_pages, int h_kv,
                                  const int32_t *page_table, int batch,
                                  int max_pages, int32_t *seq_lens,
                                  void *summaries, float *tau_out, int flags,
                                  int32_t *status, locks_stream_t stream);

/* Decoder object: one layer's decode step driven from host buffers (the
 * decode path of LOCKS reading notes §2 Fig. 1: score every page summary,
 * select k pages, attend over them; the same computation as
 * locks_score_select followed by locks_sparse_decode).  The pages describe
 * the computation only; this object is the deployment form of it.
 *
 * locks_decoder_create binds the caller's device buffers and sizes:
 *   k_cache, v_cache, num_phys_pages, page_table, summaries, seq_lens,
 *   batch, h_q, h_kv, max_pages, k   as in locks_score_select /
 *                  locks_sparse_decode (seq_lens is read on the device at
 *                  every step, so appends between steps take effect)
 *   q_dev         bf16 [batch][h_q][128] device staging buffer for the query
 *   idx           int32 [batch][h_kv][k] device buffer for the selection
 *   workspace     >= locks_workspace_size(batch, h_q, h_kv, max_pages, k)
 * It checks the arguments, creates a private non-blocking capture stream
 * and a 4-byte mapped page-locked host word, and allocates no device
 * memory.  All
 * bound buffers stay owned by the caller and must outlive the decoder.
 * Errors: LOCKS_ERR_INVALID_ARG / _UNSUPPORTED / _WORKSPACE as the step
 * calls would return them; LOCKS_ERR_CUDA if the stream or the host word
 * cannot be created.  *out is NULL on any error. */
typedef struct locks_decoder locks_decoder_t;
locks_status_t locks_decoder_create(
    const void *k_cache, const void *v_cache, int64_t num_phys_pages,
    const int32_t *page_table, const void *summaries, const int32_t *seq_lens,
    int batch, int h_q, int h_kv, int max_pages, int k, void *q_dev,
    int32_t *idx, void *workspace, size_t workspace_bytes,
    locks_decoder_t **out);

/* One decode step from host buffers, synchronous:
 *   q_host    host bf16 [batch][h_q][128] query (page-locked)
 *   o_host    host bf16 [batch][h_q][128] attention output (page-locked)
 *   lse_host  host float [batch][h_q] natural-log LSE (page-locked)
 *   status_out  optional plain host int32: the device status word
 *             (LOCKS_DEV_* bits, sticky until locks_clear_status) as read
 *             back at the end of this step
 *   stream    the step is ordered after earlier work on `stream` (NULL =
 *             the legacy default stream) and the call returns when it is
 *             done (the stream is synchronised).
 * The first call records the whole step (a kernel that reads the query
 * from host memory into q_dev, the four kernels, the attention kernels
 * writing o and lse straight into the host buffers and the merge kernel
 * copying the status word out) as one CUDA graph on the decoder's capture
 * stream, after one plain run of the same step that completes first; every
 * call then launches that graph once.  The host buffers are reached through
 * their mapped device addresses, so they must be page-locked
 * (cudaHostAlloc, or cudaHostRegister with mapping) with a 16-byte aligned
 * device address; anything else returns LOCKS_ERR_INVALID_ARG before
 * anything runs.  Another query buffer than the previous call's is patched
 * into the graph; other output buffers make the call record the graph
 * again (keep them fixed for the fast path).  The decoder remembers the
 * mapped addresses of the buffers it last used: a buffer must stay
 * page-locked for as long as the decoder may still be given it.
 * On LOCKS_ERR_CUDA, locks_decoder_last_cuda_error gives the cudaError_t.
 * Calls on one decoder must not overlap (one host thread at a time). */
locks_status_t locks_decoder_step_host(locks_decoder_t *decoder,
                                       const void *q_host, void *o_host,
                                       float *lse_host, int32_t *status_out,
                                       locks_stream_t stream);

/* cudaError_t of the decoder's last failing CUDA call (0 if none). */
int locks_decoder_last_cuda_error(const locks_decoder_t *decoder);

/* Release the decoder's graph, stream and host word (NULL is a no-op).
 * The caller's buffers are untouched. */
void locks_decoder_destroy(locks_decoder_t *decoder);

/* Zero the device status word (the first int32 of `status_word`). */
locks_status_t locks_clear_status(void *status_word, locks_stream_t stream);

/* Copy the device status word to *host_out; synchronises `stream`. */
locks_status_t locks_read_status(const void *status_word, int32_t *host_out,
                                 locks_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LOCKS_H */
