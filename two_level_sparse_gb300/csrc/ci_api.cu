// The C ABI declared in include/ci.h: host-side argument checks, then one
// kernel launch per call.  No allocation, no synchronization.
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/ci.h"
#include "ci_internal.h"

namespace ci {

int device_sm_count() {
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (counts[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    counts[dev] = n > 0 ? n : 1;
  }
  return counts[dev];
}

int64_t device_l2_bytes() {
  static int64_t sizes[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (sizes[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev);
    sizes[dev] = n > 0 ? n : 1;
  }
  return sizes[dev];
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

cudaError_t make_pool_tmap(CUtensorMap* map, const uint8_t* k_pool, int64_t num_pages, int kv_format, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  // [pages][64 positions][row bytes]: 128-byte e4m3 rows (128-byte swizzle) or
  // 64-byte packed e2m1 rows (64-byte swizzle)
  const bool fp4 = kv_format == CI_KV_MXFP4;
  const cuuint64_t row = fp4 ? CI_DIM / 2 : CI_DIM;
  const cuuint64_t dims[3] = {row, static_cast<cuuint64_t>(CI_PAGE), static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[2] = {row, static_cast<cuuint64_t>(fp4 ? CI_PAGE_BYTES_MXFP4 : CI_PAGE_BYTES)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(row), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(k_pool), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace ci

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks shared by the two scoring entry points.
int check_pool(const uint8_t* q_fp4, const uint8_t* q_sf, const float* w, const uint8_t* k_pool, int64_t num_pages,
               int32_t kv_format, const int32_t* page_table, int32_t num_req, int32_t max_pages, int32_t layout,
               const int32_t* req_row_start, const int32_t* seq_len, int32_t rows, int32_t max_len) {
  if (rows < 0 || max_len < 0 || num_pages < 0 || num_req < 0 || max_pages < 0) return CI_ERR_SHAPE;
  if (layout != CI_LAYOUT_DECODE && layout != CI_LAYOUT_PREFILL && layout != CI_LAYOUT_VARLEN)
    return CI_ERR_UNSUPPORTED;
  if (kv_format != CI_KV_FP8 && kv_format != CI_KV_MXFP4) return CI_ERR_UNSUPPORTED;
  if (rows == 0) return CI_OK;
  if (!q_fp4 || !q_sf || !w || !k_pool || !page_table || !seq_len) return CI_ERR_NULL;
  if (layout == CI_LAYOUT_DECODE && num_req != rows) return CI_ERR_SHAPE;
  if (layout == CI_LAYOUT_PREFILL && num_req != 1) return CI_ERR_SHAPE;
  if (layout == CI_LAYOUT_VARLEN) {
    if (!req_row_start) return CI_ERR_NULL;
    if (num_req < 1 || num_req > ci::kMaxReq) return CI_ERR_RANGE;
  }
  if (static_cast<int64_t>(max_len) > static_cast<int64_t>(max_pages) * CI_PAGE) return CI_ERR_SHAPE;
  if (num_pages < 1 || num_pages > INT32_MAX) return CI_ERR_RANGE;
  if (!aligned(k_pool, 16) || !aligned(q_fp4, 8) || !aligned(q_sf, 16) || !aligned(w, 16)) return CI_ERR_ALIGN;
  return CI_OK;
}

int launched(cudaError_t e) { return e == cudaSuccess ? CI_OK : CI_ERR_CUDA; }

// log2 of 8, 4, 2 or 1 positions per block; -1 otherwise.
int block_shift_of(int32_t block_positions) {
  switch (block_positions) {
    case 8: return 3;
    case 4: return 2;
    case 2: return 1;
    case 1: return 0;
    default: return -1;
  }
}

}  // namespace

extern "C" {

int ci_version(void) { return 301; }

const char* ci_strerror(int status) {
  switch (status) {
    case CI_OK: return "ok";
    case CI_ERR_NULL: return "a required pointer is NULL";
    case CI_ERR_SHAPE: return "inconsistent sizes or strides";
    case CI_ERR_ALIGN: return "a pointer or stride breaks an alignment rule";
    case CI_ERR_RANGE: return "a size is out of its supported range";
    case CI_ERR_UNSUPPORTED: return "a valid request this library does not implement";
    case CI_ERR_CUDA: return "a CUDA call failed";
    default: return "unknown status";
  }
}

int ci_score_dense_amax8(const uint8_t* q_fp4, const uint8_t* q_sf, const float* w, const uint8_t* k_pool,
                         int64_t num_pages, int32_t kv_format, const int32_t* page_table, int32_t num_req, int32_t max_pages,
                         int32_t layout, const int32_t* req_row_start, const int32_t* seq_len, int32_t rows,
                         int32_t max_len, int32_t skip_le_blocks, int32_t block_positions, float* keys,
                         int64_t keys_stride, int32_t* dev_err, void* stream) {
  int st = check_pool(q_fp4, q_sf, w, k_pool, num_pages, kv_format, page_table, num_req, max_pages, layout,
                      req_row_start, seq_len, rows, max_len);
  if (st != CI_OK) return st;
  if (skip_le_blocks < 0) return CI_ERR_RANGE;
  const int shift = block_shift_of(block_positions);
  if (shift < 0) return CI_ERR_RANGE;
  if (shift != 3 && kv_format != CI_KV_FP8) return CI_ERR_UNSUPPORTED;
  if (rows == 0) return CI_OK;
  if (!keys) return CI_ERR_NULL;
  if (keys_stride % 8 != 0 || keys_stride < (static_cast<int64_t>(max_len) + block_positions - 1) >> shift)
    return CI_ERR_SHAPE;
  if (!aligned(keys, 16)) return CI_ERR_ALIGN;
  ci::DenseArgs a{{q_fp4, q_sf, w, k_pool, num_pages, kv_format, page_table, max_pages, layout, req_row_start, num_req, seq_len,
                   rows, max_len, dev_err},
                  shift,
                  skip_le_blocks,
                  keys,
                  keys_stride};
  return launched(ci::launch_dense_amax8(a, static_cast<cudaStream_t>(stream)));
}

int ci_publish_blocks2(const int32_t* seq_len, int32_t rows, int32_t max_len, const float* keys, int64_t keys_stride,
                       int32_t topk_blocks, int32_t* blocks, int64_t blocks_stride, int32_t* nvalid,
                       int32_t topk_blocks2, int32_t* blocks2, int64_t blocks2_stride, int32_t* nvalid2,
                       int32_t* dev_err, void* stream) {
  if (rows < 0 || max_len < 0) return CI_ERR_SHAPE;
  if (topk_blocks < 1 || topk_blocks > 16384) return CI_ERR_RANGE;
  if (blocks2 != nullptr && (topk_blocks2 < 1 || topk_blocks2 > 16384)) return CI_ERR_RANGE;
  if (max_len > 393216) return CI_ERR_RANGE;
  if (rows == 0) return CI_OK;
  if (!seq_len || !keys || !blocks || !nvalid) return CI_ERR_NULL;
  if (blocks2 != nullptr && !nvalid2) return CI_ERR_NULL;
  if (blocks_stride < topk_blocks) return CI_ERR_SHAPE;
  if (blocks2 != nullptr && blocks2_stride < topk_blocks2) return CI_ERR_SHAPE;
  if (blocks2 != nullptr) {
    // the K' selection reads the K selection's winners back while it writes:
    // the two tables must not share a byte
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(blocks), b0 = reinterpret_cast<uintptr_t>(blocks2);
    const uintptr_t a1 = a0 + (static_cast<uint64_t>(rows - 1) * blocks_stride + topk_blocks) * sizeof(int32_t);
    const uintptr_t b1 = b0 + (static_cast<uint64_t>(rows - 1) * blocks2_stride + topk_blocks2) * sizeof(int32_t);
    if (a0 < b1 && b0 < a1) return CI_ERR_SHAPE;
  }
  if (keys_stride % 8 != 0 || keys_stride < (static_cast<int64_t>(max_len) + 7) / 8) return CI_ERR_SHAPE;
  if (!aligned(keys, 16)) return CI_ERR_ALIGN;
  ci::PublishArgs a{seq_len, rows,   max_len, keys, keys_stride, topk_blocks,
                    blocks,  blocks_stride, nvalid, blocks2 ? topk_blocks2 : 0, blocks2, blocks2_stride,
                    nvalid2, dev_err};
  return launched(ci::launch_publish(a, static_cast<cudaStream_t>(stream)));
}

int ci_publish_blocks(const int32_t* seq_len, int32_t rows, int32_t max_len, const float* keys, int64_t keys_stride,
                      int32_t topk_blocks, int32_t* blocks, int64_t blocks_stride, int32_t* nvalid, int32_t* dev_err,
                      void* stream) {
  return ci_publish_blocks2(seq_len, rows, max_len, keys, keys_stride, topk_blocks, blocks, blocks_stride, nvalid, 0,
                            nullptr, 0, nullptr, dev_err, stream);
}

int ci_prefill_tail(const int32_t* req_row_start, int32_t num_req, const int32_t* tail_len, int32_t rows,
                    const int32_t* blocks, int64_t blocks_stride, const int32_t* nvalid, int32_t topk_blocks,
                    int32_t* out_row, int32_t* out_blocks, int64_t out_blocks_stride, int32_t* out_nvalid,
                    int32_t* out_count, int32_t out_cap, int32_t* dev_err, void* stream) {
  if (rows < 0 || out_cap < 0) return CI_ERR_SHAPE;
  if (num_req < 1 || num_req > ci::kMaxReq) return CI_ERR_RANGE;
  if (topk_blocks < 1 || topk_blocks > 16384) return CI_ERR_RANGE;
  if (!req_row_start || !tail_len || !out_count) return CI_ERR_NULL;
  if (out_cap > 0 && (!blocks || !nvalid || !out_row || !out_blocks || !out_nvalid)) return CI_ERR_NULL;
  if (blocks_stride < topk_blocks || out_blocks_stride < topk_blocks) return CI_ERR_SHAPE;
  ci::TailArgs a{req_row_start, num_req, tail_len,   rows,    blocks,    blocks_stride, nvalid, topk_blocks,
                 out_row,       out_blocks, out_blocks_stride, out_nvalid, out_count, out_cap, dev_err};
  return launched(ci::launch_tail(a, static_cast<cudaStream_t>(stream)));
}

int ci_q_rope_quant(const int32_t* positions, const uint16_t* q, const float* cos_sin, int32_t max_pos,
                    const float* w, float softmax_scale, float head_scale, int32_t is_neox, int32_t tokens,
                    int32_t out_format, uint8_t* q_out, uint8_t* q_sf, float* w_out, int32_t* dev_err, void* stream) {
  if (tokens < 0 || max_pos < 0) return CI_ERR_SHAPE;
  if (out_format != CI_Q_MXFP4 && out_format != CI_Q_FP8) return CI_ERR_UNSUPPORTED;
  if (tokens == 0) return CI_OK;
  if (!positions || !q || !cos_sin || !w || !q_out || !w_out) return CI_ERR_NULL;
  if (out_format == CI_Q_MXFP4 && !q_sf) return CI_ERR_NULL;
  if ((q_sf != nullptr && !aligned(q_sf, 4)) || !aligned(q, 8) || !aligned(cos_sin, 16) || !aligned(q_out, 4))
    return CI_ERR_ALIGN;
  ci::QProdArgs a{positions, q,      cos_sin, max_pos, w,    softmax_scale, head_scale, tokens,
                  is_neox != 0, out_format == CI_Q_FP8, q_out, q_sf, w_out, dev_err};
  return launched(ci::launch_qprod(a, static_cast<cudaStream_t>(stream)));
}

int ci_dcp_merge_keys(const float* keys_local, int32_t world, int64_t rank_stride, int64_t local_stride,
                      const int32_t* seq_len, int32_t rows, int32_t max_len, int32_t skip_le_blocks, float* keys,
                      int64_t keys_stride, int32_t* dev_err, void* stream) {
  if (rows < 0 || max_len < 0) return CI_ERR_SHAPE;
  if (world != 2 && world != 4 && world != 8) return CI_ERR_RANGE;
  if (skip_le_blocks < 0) return CI_ERR_RANGE;
  if (rows == 0) return CI_OK;
  if (!keys_local || !seq_len || !keys) return CI_ERR_NULL;
  const int64_t nb = (static_cast<int64_t>(max_len) + 7) / 8;
  if (keys_stride < nb || local_stride < nb || rank_stride < local_stride * rows) return CI_ERR_SHAPE;
  ci::DcpKeysArgs a{keys_local, world, rank_stride, local_stride, seq_len, rows, max_len, skip_le_blocks,
                    keys,       keys_stride, dev_err};
  return launched(ci::launch_dcp_merge_keys(a, static_cast<cudaStream_t>(stream)));
}

int ci_dcp_merge_topk(const int32_t* pos_local, const float* score_local, int32_t world, int64_t rank_stride,
                      int64_t local_stride, int32_t rows, int32_t topk, int32_t* out_pos, float* out_score,
                      int64_t out_stride, void* stream) {
  if (rows < 0) return CI_ERR_SHAPE;
  if (world != 2 && world != 4 && world != 8) return CI_ERR_RANGE;
  if (topk < 1 || static_cast<int64_t>(topk) * world > 4096) return CI_ERR_RANGE;
  if (rows == 0) return CI_OK;
  if (!pos_local || !score_local || !out_pos) return CI_ERR_NULL;
  if (local_stride < topk || out_stride < topk || rank_stride < local_stride * rows) return CI_ERR_SHAPE;
  ci::DcpTopkArgs a{pos_local, score_local, world, rank_stride, local_stride, rows, topk, out_pos, out_score, out_stride};
  return launched(ci::launch_dcp_merge_topk(a, static_cast<cudaStream_t>(stream)));
}

int ci_select_sparse_layers(int32_t num_layers, const uint8_t* const* q_fp4, const uint8_t* const* q_sf,
                            const float* const* w, const uint8_t* const* k_pool, int64_t num_pages, int32_t kv_format,
                            const int32_t* page_table, int32_t num_req, int32_t max_pages, int32_t layout,
                            const int32_t* req_row_start, const int32_t* seq_len, int32_t rows, int32_t max_len,
                            const int32_t* const* blocks, const int64_t* blocks_stride,
                            const int32_t* const* nvalid, const int32_t* max_blocks, int32_t block_positions,
                            int32_t topk, int32_t* const* out_pos, float* const* out_score, int64_t out_stride,
                            int32_t* dev_err, void* stream) {
  if (num_layers < 1 || num_layers > ci::kMaxSelectLayers) return CI_ERR_RANGE;
  if (!q_fp4 || !q_sf || !w || !k_pool || !blocks || !blocks_stride || !nvalid || !max_blocks || !out_pos)
    return CI_ERR_NULL;
  ci::SelectArgs a{};
  for (int l = 0; l < num_layers; ++l) {
    int st = check_pool(q_fp4[l], q_sf[l], w[l], k_pool[l], num_pages, kv_format, page_table, num_req, max_pages,
                        layout, req_row_start, seq_len, rows, max_len);
    if (st != CI_OK) return st;
    if (max_blocks[l] < 0 || max_blocks[l] > 2176) return CI_ERR_RANGE;
    if (rows == 0) continue;
    if (!blocks[l] || !nvalid[l] || !out_pos[l]) return CI_ERR_NULL;
    if (blocks_stride[l] < max_blocks[l]) return CI_ERR_SHAPE;
    a.layer[l] = ci::SelectLayer{q_fp4[l], q_sf[l], w[l], k_pool[l], blocks[l], blocks_stride[l], nvalid[l],
                                 max_blocks[l], out_pos[l], out_score != nullptr ? out_score[l] : nullptr};
  }
  if (topk < 1 || topk > 2048) return CI_ERR_RANGE;
  const int shift = block_shift_of(block_positions);
  if (shift < 0) return CI_ERR_RANGE;
  if (num_pages > (int64_t{1} << 21)) return CI_ERR_RANGE;  // page ids are packed into 21 bits
  if (rows == 0) return CI_OK;
  if (out_stride < topk) return CI_ERR_SHAPE;
  a.p = ci::PoolArgs{nullptr, nullptr, nullptr, nullptr, num_pages, kv_format, page_table, max_pages, layout,
                     req_row_start, num_req, seq_len, rows, max_len, dev_err};
  a.block_shift = shift;
  a.topk = topk;
  a.out_stride = out_stride;
  a.num_layers = num_layers;
  return launched(ci::launch_select(a, static_cast<cudaStream_t>(stream)));
}

int ci_select_sparse(const uint8_t* q_fp4, const uint8_t* q_sf, const float* w, const uint8_t* k_pool,
                     int64_t num_pages, int32_t kv_format, const int32_t* page_table, int32_t num_req, int32_t max_pages, int32_t layout,
                     const int32_t* req_row_start, const int32_t* seq_len, int32_t rows, int32_t max_len,
                     const int32_t* blocks, int64_t blocks_stride, const int32_t* nvalid, int32_t max_blocks,
                     int32_t block_positions, int32_t topk, int32_t* out_pos, float* out_score, int64_t out_stride,
                     int32_t* dev_err, void* stream) {
  return ci_select_sparse_layers(1, &q_fp4, &q_sf, &w, &k_pool, num_pages, kv_format, page_table, num_req, max_pages,
                                 layout, req_row_start, seq_len, rows, max_len, &blocks, &blocks_stride, &nvalid,
                                 &max_blocks, block_positions, topk, &out_pos, &out_score, out_stride, dev_err, stream);
}

}  // extern "C"
