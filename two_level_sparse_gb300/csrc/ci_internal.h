// Host-side interface between the C ABI (ci_api.cu) and the kernel launchers.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ci {

constexpr int kMaxReq = 4096;  // requests of one multi-request chunk (layout 2)

struct PoolArgs {
  const uint8_t* q_fp4;
  const uint8_t* q_sf;
  const float* w;
  const uint8_t* k_pool;
  int64_t num_pages;
  int32_t kv_format;  // 0 FP8 pages, 1 MXFP4 pages
  const int32_t* page_table;
  int32_t max_pages;
  int32_t layout;  // 0 decode (row t = request t), 1 prefill (one request), 2 several requests
  const int32_t* req_start;  // layout 2: rows of request r are [req_start[r], req_start[r + 1])
  int32_t num_req;
  const int32_t* seq_len;
  int32_t rows;
  int32_t max_len;
  int32_t* dev_err;
};

struct DenseArgs {
  PoolArgs p;
  int32_t block_shift;  // log2 of the positions per key: 3, or 2/1/0 for a context shard (no +inf pin)
  int32_t skip_le_blocks;
  float* keys;
  int64_t keys_stride;
};

struct PublishArgs {
  const int32_t* seq_len;
  int32_t rows;
  int32_t max_len;
  const float* keys;
  int64_t keys_stride;
  int32_t topk_blocks;
  int32_t* blocks;
  int64_t blocks_stride;
  int32_t* nvalid;
  int32_t topk_blocks2;  // second selection from the same keys (0: none)
  int32_t* blocks2;
  int64_t blocks2_stride;
  int32_t* nvalid2;
  int32_t* dev_err;
};

// One layer of a select launch: its query, weights, index-K pool, candidate
// blocks and outputs.  The page table, layout and lengths are shared.
constexpr int kMaxSelectLayers = 8;
struct SelectLayer {
  const uint8_t* q_fp4;
  const uint8_t* q_sf;
  const float* w;
  const uint8_t* k_pool;
  const int32_t* blocks;
  int64_t blocks_stride;
  const int32_t* nvalid;
  int32_t max_blocks;
  int32_t* out_pos;
  float* out_score;
};

struct SelectArgs {
  PoolArgs p;  // the shared page table, layout, lengths and pool format (its q / w / k_pool fields unused)
  int32_t block_shift;  // log2 of the positions per candidate block: 3, or 2/1/0 for a context shard
  int32_t topk;
  int64_t out_stride;
  int32_t num_layers;  // 1 .. kMaxSelectLayers; work units are (layer, row), layer-major
  SelectLayer layer[kMaxSelectLayers];
};

// Each returns a cudaError_t from the launch (cudaSuccess when enqueued).
cudaError_t launch_dense_amax8(const DenseArgs& a, cudaStream_t stream);
struct TailArgs {
  const int32_t* req_start;
  int32_t num_req;
  const int32_t* tail_len;
  int32_t rows;
  const int32_t* blocks;
  int64_t blocks_stride;
  const int32_t* nvalid;
  int32_t topk_blocks;
  int32_t* out_row;
  int32_t* out_blocks;
  int64_t out_blocks_stride;
  int32_t* out_nvalid;
  int32_t* out_count;
  int32_t out_cap;
  int32_t* dev_err;
};

struct QProdArgs {
  const int32_t* positions;
  const uint16_t* q;  // bf16 [tokens][64][128]
  const float* cos_sin;  // [max_pos][64]: 32 cos, then 32 sin
  int32_t max_pos;
  const float* w;
  float softmax_scale, head_scale;
  int32_t tokens;
  bool neox, fp8;
  uint8_t* q_out;
  uint8_t* q_sf;
  float* w_out;
  int32_t* dev_err;
};

struct DcpKeysArgs {
  const float* keys_local;  // [world][rows][local_stride]
  int32_t world;
  int64_t rank_stride, local_stride;
  const int32_t* seq_len;  // global lengths
  int32_t rows, max_len, skip_le_blocks;
  float* keys;
  int64_t keys_stride;
  int32_t* dev_err;
};

struct DcpTopkArgs {
  const int32_t* pos_local;  // [world][rows][local_stride]
  const float* score_local;
  int32_t world;
  int64_t rank_stride, local_stride;
  int32_t rows, topk;
  int32_t* out_pos;
  float* out_score;
  int64_t out_stride;
};

cudaError_t launch_publish(const PublishArgs& a, cudaStream_t stream);
cudaError_t launch_publish_rows(const PublishArgs& a, cudaStream_t stream);  // few rows: one per CTA at a time
cudaError_t launch_dcp_merge_keys(const DcpKeysArgs& a, cudaStream_t stream);
cudaError_t launch_dcp_merge_topk(const DcpTopkArgs& a, cudaStream_t stream);
cudaError_t launch_qprod(const QProdArgs& a, cudaStream_t stream);
cudaError_t launch_tail(const TailArgs& a, cudaStream_t stream);
cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream);

// Shared host helpers (ci_api.cu).
int device_sm_count();
int64_t device_l2_bytes();  // L2 cache size of the current device
// Tensor map over the value bytes of a paged index-K pool viewed as
// [num_pages][64 positions][128 bytes], 128-byte swizzle, box of `box_rows`
// positions of one page.
cudaError_t make_pool_tmap(CUtensorMap* map, const uint8_t* k_pool, int64_t num_pages, int kv_format, int box_rows);

}  // namespace ci
