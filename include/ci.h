/*
 * ci.h -- C ABI of the GB300 two-level candidate indexer (libci.so).
 *
 * The DeepSeek-V4.1 indexer picks, for every query row t, the compressed
 * positions s < L_t that sparse attention will read.  It works in two levels
 * (sglang PR #40352 "Score prefill consumer index layers on candidate blocks
 * with DeepGEMM", Motivation and Design; sglang PR #39671 "dsv4.1: candidate
 * indexer library", Summary):
 *
 *   level one, once per step, on the source index layer:
 *     ci_score_dense_amax8   logit[t,s] = sum_h w[t,h] * ReLU(q[t,h] . k[s])
 *                            for every s < L_t, reduced on chip to one key per
 *                            block of 8 positions (the block maximum), the
 *                            row's newest block forced to +inf;
 *     ci_publish_blocks      each row's top topk_blocks block ids by key,
 *                            ascending, INT32_MAX padded;
 *     ci_publish_blocks2     the same for two block counts at once (the
 *                            consumers' K and the source's own P + 1),
 *                            reading the keys once;
 *     ci_prefill_tail        the published table of the last rows of each
 *                            request of a multi-request chunk;
 *   context sharding (one device emulating W shards):
 *     ci_dcp_merge_keys      shards' local block maxima -> global keys;
 *     ci_dcp_merge_topk      shards' local top-k -> global top-k;
 *   before level one, once per layer:
 *     ci_q_rope_quant        the query producer: RoPE, quantization to the
 *                            indexer's query format, head-weight scaling;
 *   level two, once per layer (the source itself and each consumer):
 *     ci_select_sparse       scores only the positions inside a row's
 *                            published blocks and returns its top-k positions,
 *                            ascending, -1 padded;
 *     ci_select_sparse_layers  the same for several layers in one launch.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - H = 64 heads, D = 128 dims, blocks of 8 positions, pages of 64 positions.
 *  - All array arguments are DEVICE pointers owned by the caller.  The library
 *    allocates nothing, never synchronizes the device or the stream, records
 *    no events, and enqueues its kernels on `stream` (a cudaStream_t; NULL =
 *    the legacy default stream).
 *  - Query (MXFP4): q_fp4 uint8 [rows][64][64], two e2m1 codes per byte,
 *    element 2i in the low nibble; q_sf uint8 [rows][64][4], one ue8m0 scale
 *    per 32 elements (vLLM sparse_attn_indexer.py, "MXFP4 layout" comment).
 *  - Head weights: w float [rows][64].
 *  - Index-K pool, in one of two page formats (`kv_format`):
 *      CI_KV_FP8    k_pool uint8 [num_pages][8448].  Page p holds 64
 *                   positions: bytes [0, 8192) are their FP8 e4m3 vectors
 *                   (128 bytes each), bytes [8192, 8448) their fp32 scales
 *                   (little endian).  The scale multiplies the decoded vector.
 *      CI_KV_MXFP4  k_pool uint8 [num_pages][4352].  Bytes [0, 4096) are the
 *                   64 positions' MXFP4 vectors (64 bytes each, two e2m1
 *                   codes per byte, element 2i in the low nibble), bytes
 *                   [4096, 4352) one 32-bit word per position whose byte j is
 *                   the ue8m0 scale of elements 32j .. 32j + 31 (vLLM
 *                   sparse_attn_indexer.py, _gather_workspace_shapes and
 *                   kv_cache_as_quant_view, the use_fp4_cache path: head_dim/2
 *                   packed bytes and head_dim/32 ue8m0 scales per position).
 *    k_pool, q_sf and w must be 16-byte aligned, q_fp4 8-byte aligned.
 *  - Page table: page_table int32 [num_req][max_pages]; logical page j of a
 *    request lives in physical page page_table[req][j].  Position s of a row
 *    is slot s % 64 of logical page s / 64.
 *  - Row layout (`layout`):
 *      CI_LAYOUT_DECODE  row t is request t (num_req == rows);
 *      CI_LAYOUT_PREFILL all rows belong to request 0 (num_req == 1) and share
 *                        its pages; row t reaches its first L_t positions.
 *      CI_LAYOUT_VARLEN  a prefill chunk of several requests: rows
 *                        req_row_start[r] .. req_row_start[r+1]-1 belong to
 *                        request r and read its pages (sglang PR #40352,
 *                        Design: the chunk's inputs carry request starts and
 *                        rows per request).  req_row_start: device int32
 *                        [num_req + 1], 0 = req_row_start[0] <= ... <=
 *                        req_row_start[num_req] = rows, 1 <= num_req <= 4096;
 *                        ignored (may be NULL) for the other layouts.  A
 *                        violation found on the device sets CI_DEVERR_REQ.
 *    Output positions are request-relative in every layout.
 *  - seq_len int32 [rows]: L_t, with 0 <= L_t <= max_len <= 64 * max_pages.
 *    max_len is the caller's host-side bound; the kernels check every L_t
 *    against it on the device.
 *  - dev_err: optional (may be NULL) device int32.  Kernels OR CI_DEVERR_*
 *    bits into it when they meet data that breaks the contract (a length above
 *    max_len, a page id outside [0, num_pages), a block id out of range); the
 *    offending row or tile is skipped and its outputs are undefined.  The
 *    caller clears it and reads it back when convenient.
 *  - Return value: CI_OK or a negative CI_ERR_* code from the host-side
 *    argument checks (nothing is launched then), or CI_ERR_CUDA if a launch
 *    failed.  ci_strerror() names the code.
 *  - Ties are broken toward the lower index, for blocks and for positions.
 */
#ifndef CI_H_
#define CI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CI_API __attribute__((visibility("default")))
#else
#define CI_API
#endif

#define CI_HEADS 64
#define CI_DIM 128
#define CI_BLOCK 8
#define CI_PAGE 64
#define CI_PAGE_BYTES (CI_PAGE * CI_DIM + CI_PAGE * 4)
#define CI_PAGE_BYTES_MXFP4 (CI_PAGE * CI_DIM / 2 + CI_PAGE * 4)

enum ci_status {
  CI_OK = 0,
  CI_ERR_NULL = -1,        /* a required pointer is NULL */
  CI_ERR_SHAPE = -2,       /* inconsistent sizes or strides */
  CI_ERR_ALIGN = -3,       /* a pointer or stride breaks an alignment rule */
  CI_ERR_RANGE = -4,       /* a size is out of its supported range */
  CI_ERR_UNSUPPORTED = -5, /* a valid request this library does not implement */
  CI_ERR_CUDA = -6         /* a CUDA call failed (launch or attribute) */
};

enum ci_layout { CI_LAYOUT_DECODE = 0, CI_LAYOUT_PREFILL = 1, CI_LAYOUT_VARLEN = 2 };
enum ci_kv_format { CI_KV_FP8 = 0, CI_KV_MXFP4 = 1 };
enum ci_q_format { CI_Q_MXFP4 = 0, CI_Q_FP8 = 1 };

/* Bits OR-ed into *dev_err by the kernels. */
#define CI_DEVERR_LEN 1u     /* seq_len[t] < 0 or > max_len */
#define CI_DEVERR_PAGE 2u    /* page id outside [0, num_pages) */
#define CI_DEVERR_BLOCK 4u   /* candidate block id outside [0, ceil(L_t/8)) or nvalid out of range */
#define CI_DEVERR_TIMEOUT 8u /* an on-chip pipeline wait gave up (should never happen) */
#define CI_DEVERR_REQ 16u    /* req_row_start is not a partition of the rows (CI_LAYOUT_VARLEN) */
#define CI_DEVERR_POS 32u    /* a RoPE position outside [0, max_pos) (ci_q_rope_quant) */

/*
 * Level one, scoring: block keys of the source layer.
 *
 * For every row t with nb_t = ceil(L_t / 8) > skip_le_blocks and every block
 * b < nb_t writes
 *     keys[t * keys_stride + b] = max_{8b <= s < min(8b + 8, L_t)} logit[t, s]
 * with logit[t, s] = kscale[s] * sum_h w[t,h] * ReLU(q[t,h] . k[s]) computed in
 * fp32 (products exact, fp32 accumulation; kscale = 1 for CI_KV_MXFP4, whose
 * scales are part of k), and keys[t*keys_stride + nb_t - 1]
 * = +inf.  Precondition: every FP8 position scale kscale[s] is finite and
 * positive.  The method's score is sum_h w * ReLU(q . (kscale * k)); only for
 * kscale > 0 may the scale leave the ReLU, so for a zero, negative or
 * non-finite scale the result is this formula, not the method's score (the
 * kernels do not check it).  Rows with nb_t <= skip_le_blocks are not scored and their keys are
 * left untouched (sglang PR #40352, Design, "Level one"; the block_amax.cuh
 * listing in the same PR's review: max of 8, last key +inf, rows with at most
 * topk blocks skipped).  The [rows, L] score matrix is never written.
 *
 * keys: float [rows][keys_stride], 16-byte aligned, keys_stride % 8 == 0 and
 * keys_stride >= ceil(max_len / block_positions).
 *
 * block_positions is 8 for the method's blocks.  A shard of a context-sharded
 * indexer (vLLM sparse_attn_indexer.py, two-level candidate filtering under
 * DCP: W shards, interleave 1, position s on shard s % W at local position
 * s / W) passes its local pool and lengths with block_positions = 8 / W (4, 2
 * or 1; FP8 pages): key b is then the maximum over local positions
 * [b * block_positions, (b + 1) * block_positions), its part of global block b,
 * and no key is pinned to +inf (ci_dcp_merge_keys pins the global newest block).
 */
CI_API int ci_score_dense_amax8(const uint8_t* q_fp4, const uint8_t* q_sf, const float* w, const uint8_t* k_pool,
                         int64_t num_pages, int32_t kv_format, const int32_t* page_table, int32_t num_req, int32_t max_pages,
                         int32_t layout, const int32_t* req_row_start, const int32_t* seq_len, int32_t rows,
                         int32_t max_len,
                         int32_t skip_le_blocks, int32_t block_positions, float* keys, int64_t keys_stride,
                         int32_t* dev_err, void* stream);

/*
 * Level one, publishing: each row's candidate blocks.
 *
 * For every row t: if nb_t <= topk_blocks, blocks[t][0..nb_t) = 0..nb_t-1
 * (keep everything, keys not read); otherwise the topk_blocks block ids with
 * the largest keys (ties: lower id first).  The ids are written ascending into
 * blocks[t * blocks_stride + i], i < topk_blocks, the rest of the first
 * topk_blocks slots INT32_MAX; nvalid[t] = min(nb_t, topk_blocks)
 * (sglang PR #40352, Design: ragged top-k over the keys, rows with at most
 * 2048 blocks keep everything, ids sorted ascending and INT32_MAX padded).
 *
 * keys as written by ci_score_dense_amax8 (same stride rules);
 * blocks: int32 [rows][blocks_stride], blocks_stride >= topk_blocks;
 * nvalid: int32 [rows].  1 <= topk_blocks <= 16384; max_len <= 393216.
 */
CI_API int ci_publish_blocks(const int32_t* seq_len, int32_t rows, int32_t max_len, const float* keys,
                      int64_t keys_stride, int32_t topk_blocks, int32_t* blocks, int64_t blocks_stride,
                      int32_t* nvalid, int32_t* dev_err, void* stream);

/*
 * Two selections from the same keys in one pass: exactly the results of
 * ci_publish_blocks(..., topk_blocks, blocks, blocks_stride, nvalid, ...) and
 * ci_publish_blocks(..., topk_blocks2, blocks2, blocks2_stride, nvalid2, ...),
 * with each row's keys read once.  The step of the two-level method needs
 * both: the consumers select within the top K blocks, the source within its
 * top P + 1 (sglang PR #40352, Design, "Level one").  blocks2 == NULL makes it
 * ci_publish_blocks (topk_blocks2, blocks2_stride and nvalid2 are then
 * ignored); otherwise nvalid2 must not be NULL, 1 <= topk_blocks2 <= 16384 and
 * blocks2_stride >= topk_blocks2.  The two tables must not overlap: the
 * narrower selection is read back from the wider one's table while it is
 * written, so the int32 ranges [blocks, blocks + (rows - 1) * blocks_stride +
 * topk_blocks) and the same for blocks2 must be disjoint (CI_ERR_SHAPE
 * otherwise).  Same errors as ci_publish_blocks.
 */
CI_API int ci_publish_blocks2(const int32_t* seq_len, int32_t rows, int32_t max_len, const float* keys,
                       int64_t keys_stride, int32_t topk_blocks, int32_t* blocks, int64_t blocks_stride,
                       int32_t* nvalid, int32_t topk_blocks2, int32_t* blocks2, int64_t blocks2_stride,
                       int32_t* nvalid2, int32_t* dev_err, void* stream);

/*
 * The published table restricted to the tail rows of each request (sglang
 * PR #40352, Design: prefill_tail restricts what was published to the last
 * rows of each request, for the late layers that run on the tail only).
 *
 * Request r owns rows req_row_start[r] .. req_row_start[r+1]-1 (the
 * CI_LAYOUT_VARLEN partition) and keeps its last m_r = min(max(tail_len[r],
 * 0), its row count) rows.  The kept rows, in order, become output rows
 * 0 .. M-1 (M = sum of m_r, written to *out_count): for each output row o,
 * out_row[o] = its source row, out_blocks[o * out_blocks_stride + i] =
 * blocks[out_row[o] * blocks_stride + i] for i < topk_blocks, out_nvalid[o] =
 * nvalid[out_row[o]].  Output rows M .. out_cap-1 get out_row -1, nvalid 0
 * and INT32_MAX ids.  If M > out_cap only the first out_cap are written and
 * CI_DEVERR_REQ is set, as it is for row starts that are not a partition.
 * req_row_start: int32 [num_req + 1], 1 <= num_req <= 4096; tail_len: int32
 * [num_req]; all device memory.
 */
CI_API int ci_prefill_tail(const int32_t* req_row_start, int32_t num_req, const int32_t* tail_len, int32_t rows,
                    const int32_t* blocks, int64_t blocks_stride, const int32_t* nvalid, int32_t topk_blocks,
                    int32_t* out_row, int32_t* out_blocks, int64_t out_blocks_stride, int32_t* out_nvalid,
                    int32_t* out_count, int32_t out_cap, int32_t* dev_err, void* stream);

/*
 * Level two: a layer's top-k positions inside the candidate blocks.
 *
 * For every row t the candidate positions are s = 8 * blocks[t][i] + j,
 * i < nvalid[t], j < 8, s < L_t, in ascending order (blocks must be ascending,
 * as ci_publish_blocks writes them).  Each is scored with this layer's q, w
 * and k_pool exactly as in ci_score_dense_amax8, and the topk best (ties:
 * lower position first) are written ascending to out_pos[t * out_stride + i],
 * i < topk, with -1 past min(topk, number of candidate positions)
 * (sglang PR #40352, Design, "Level two": top-512 of the first valid_len
 * columns, page transform to request-relative positions, -1 past
 * min(512, valid_len)).  If out_score is not NULL, out_score[t*out_stride+i]
 * receives the fp32 score of out_pos[...] (-inf where out_pos is -1).
 *
 * The source layer's own top-512 is this call on the source layer with the
 * top max(topk_blocks, 513) blocks: every position of the dense top-512 lies
 * in those blocks.
 *
 * blocks: int32 [rows][blocks_stride]; nvalid: int32 [rows], each
 * 0 <= nvalid[t] <= max_blocks <= min(blocks_stride, 2176).
 * 1 <= topk <= 2048, topk <= out_stride; num_pages <= 2^21.
 *
 * block_positions is 8 for the method's blocks; a shard of a context-sharded
 * indexer (see ci_score_dense_amax8) passes 8 / W: block id b then names its
 * local positions [b * block_positions, (b + 1) * block_positions), and the
 * output positions are local.
 */
CI_API int ci_select_sparse(const uint8_t* q_fp4, const uint8_t* q_sf, const float* w, const uint8_t* k_pool,
                     int64_t num_pages, int32_t kv_format, const int32_t* page_table, int32_t num_req, int32_t max_pages,
                     int32_t layout, const int32_t* req_row_start, const int32_t* seq_len, int32_t rows,
                     int32_t max_len,
                     const int32_t* blocks, int64_t blocks_stride, const int32_t* nvalid, int32_t max_blocks,
                     int32_t block_positions, int32_t topk, int32_t* out_pos, float* out_score, int64_t out_stride,
                     int32_t* dev_err, void* stream);

/*
 * Level two for several layers in one launch: layer l (0 <= l < num_layers
 * <= 8) is exactly ci_select_sparse with q_fp4[l], q_sf[l], w[l], k_pool[l],
 * blocks[l], blocks_stride[l], nvalid[l], max_blocks[l], out_pos[l] and
 * out_score[l] (out_score itself may be NULL: no scores for any layer; or
 * out_score[l] NULL: none for layer l).  The page table, layout, lengths,
 * pool format and size, block_positions, topk and out_stride are shared:
 * the layers of one step (the source with its own top-(P+1) blocks and every
 * consumer with the published ones; PR #40352, Design, "Level two") read
 * their own pools through the same pages.  The per-layer arguments are HOST
 * arrays of num_layers entries, each entry a device pointer (or, for
 * blocks_stride and max_blocks, a value).  One persistent grid works through
 * the (layer, row) pairs layer by layer, so a layer's last rows overlap the
 * next layer's first and small batches fill every SM.  Each layer's checks
 * are ci_select_sparse's; CI_ERR_RANGE if num_layers is outside 1..8.
 */
CI_API int ci_select_sparse_layers(int32_t num_layers, const uint8_t* const* q_fp4, const uint8_t* const* q_sf,
                                   const float* const* w, const uint8_t* const* k_pool, int64_t num_pages,
                                   int32_t kv_format, const int32_t* page_table, int32_t num_req, int32_t max_pages,
                                   int32_t layout, const int32_t* req_row_start, const int32_t* seq_len, int32_t rows,
                                   int32_t max_len, const int32_t* const* blocks, const int64_t* blocks_stride,
                                   const int32_t* const* nvalid, const int32_t* max_blocks, int32_t block_positions,
                                   int32_t topk, int32_t* const* out_pos, float* const* out_score, int64_t out_stride,
                                   int32_t* dev_err, void* stream);

/*
 * The exchange steps of a context-sharded indexer with W = world shards
 * (2, 4 or 8; interleave 1), run on one device over all shards' buffers
 * (vLLM sparse_attn_indexer.py: the producer MAX-reduces block scores across
 * ranks and pins the global newest block; _merge_dcp_topk_global merges each
 * rank's local top-K exactly).
 *
 * ci_dcp_merge_keys: keys_local[r * rank_stride + t * local_stride + b] are
 * shard r's local block maxima (ci_score_dense_amax8 with block_positions =
 * 8 / W and skip_le_blocks = 0).  For every row t with nb_t = ceil(L_t / 8) >
 * skip_le_blocks (seq_len = the global lengths) writes keys[t * keys_stride +
 * b], b < nb_t: the maximum over the shards that hold a position of global
 * block b, and +inf for b = nb_t - 1 -- exactly the keys ci_score_dense_amax8
 * writes for the unsharded row.  keys_stride, local_stride >= ceil(max_len/8).
 *
 * ci_dcp_merge_topk: pos_local / score_local[r * rank_stride + t *
 * local_stride + i], i < topk, are shard r's ci_select_sparse outputs (local
 * positions ascending, -1 padded, with their scores).  Writes out_pos[t *
 * out_stride + i], i < topk: the topk best of all shards' candidates (global
 * position = local * W + r; ties toward the lower position), ascending, -1
 * padded, and their scores to out_score if it is not NULL.  world * topk <=
 * 4096.
 */
CI_API int ci_dcp_merge_keys(const float* keys_local, int32_t world, int64_t rank_stride, int64_t local_stride,
                             const int32_t* seq_len, int32_t rows, int32_t max_len, int32_t skip_le_blocks,
                             float* keys, int64_t keys_stride, int32_t* dev_err, void* stream);
CI_API int ci_dcp_merge_topk(const int32_t* pos_local, const float* score_local, int32_t world, int64_t rank_stride,
                             int64_t local_stride, int32_t rows, int32_t topk, int32_t* out_pos, float* out_score,
                             int64_t out_stride, void* stream);

/*
 * The query producer (vLLM indexer.py page, rope_quant_q; the
 * fused_indexer_q_rope_quant kernel of sparse_attn_indexer.py).
 *
 * For every token t and head h of q (bf16 bit patterns, [tokens][64][128]):
 * the pairs (x0, x1) of dims (i, 32 + i) (is_neox != 0) or (2i, 2i + 1)
 * (is_neox == 0), i < 32, become r0 = x0 c - x1 s and r1 = x1 c + x0 s with
 * c = cos_sin[p][i], s = cos_sin[p][32 + i], p = positions[t], computed in
 * fp32 with one rounding per operation and then rounded to bf16; dims 64..127
 * pass unrotated.  With e(v, m) = ceil(log2(max(v, 1e-10) * (1/m))) taken
 * exactly from the bits of the fp32 product:
 *   CI_Q_MXFP4  per block of 32 dims, e = e(amax of the block, 6): q_out
 *               [tokens][64][64] holds the e2m1 codes of x * 2^-e (nearest,
 *               ties to even, saturating at 6; element 2i in the low nibble),
 *               q_sf [tokens][64][4] the codes e + 127, and w_out[t][h] =
 *               (w[t][h] * softmax_scale) * head_scale: the indexer's inputs.
 *   CI_Q_FP8    one e = e(amax of the head, 448) per head: q_out
 *               [tokens][64][128] holds e4m3(clamp(x * 2^-e, -448, 448))
 *               (nearest even), q_sf is unused (may be NULL), and w_out =
 *               ((w * 2^e) * softmax_scale) * head_scale, the scale folded into
 *               the weight as the pages print it.
 * A position outside [0, max_pos) sets CI_DEVERR_POS and the token's heads are
 * produced from zeros.  positions int32 [tokens]; cos_sin float [max_pos][64];
 * w, w_out float [tokens][64]; all device memory; q 8-byte, cos_sin 16-byte,
 * q_out and q_sf 4-byte aligned.
 */
CI_API int ci_q_rope_quant(const int32_t* positions, const uint16_t* q, const float* cos_sin, int32_t max_pos,
                           const float* w, float softmax_scale, float head_scale, int32_t is_neox, int32_t tokens,
                           int32_t out_format, uint8_t* q_out, uint8_t* q_sf, float* w_out, int32_t* dev_err,
                           void* stream);

/* Human-readable name of a ci_status code (static storage). */
CI_API const char* ci_strerror(int status);

/* ABI version of this header (major * 100 + minor). */
CI_API int ci_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CI_H_ */
