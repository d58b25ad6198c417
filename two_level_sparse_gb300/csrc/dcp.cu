// The two exchange steps of a context-sharded indexer (vLLM
// sparse_attn_indexer.py: _merge_dcp_topk_global and the two-level candidate
// filtering under DCP), for W shards with interleave 1: global position s
// lives on shard s % W at local position s / W, so a shard's local block b
// (8 / W positions) is exactly its part of global block b.
//
//   merge_keys  key[t][b] = max over shards of their local block maxima, the
//               row's newest global block then pinned to +inf (a shard's own
//               newest local block is not the global newest in general);
//   merge_topk  the global top-k of the union of the shards' local top-k,
//               candidates (score, global id = local * W + shard), ties toward
//               the lower id, written ascending with -1 padding: a position
//               of the global top-k has at most k - 1 positions above it, so
//               it is in its own shard's local top-k, and the union holds it.
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMaxCand = 4096;  // shards x topk per row

__global__ void __launch_bounds__(kMergeThreads) merge_keys_kernel(const DcpKeysArgs a) {
  const int t = blockIdx.x;
  const int L = a.seq_len[t];
  if (L < 0 || L > a.max_len) {
    if (threadIdx.x == 0) report(a.dev_err, kDevErrLen);
    return;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  if (nb <= a.skip_le_blocks) return;  // kept whole by the publish step: keys not read
  const int W = a.world, bs = kBlock / W;
  float* out = a.keys + static_cast<int64_t>(t) * a.keys_stride;
  for (int b = threadIdx.x; b < nb; b += kMergeThreads) {
    float k = -__int_as_float(0x7f800000);
    for (int r = 0; r < W; ++r) {
      const int lr = L > r ? (L - r + W - 1) / W : 0;  // positions of the row on shard r
      if (b * bs < lr) k = fmaxf(k, a.keys_local[r * a.rank_stride + static_cast<int64_t>(t) * a.local_stride + b]);
    }
    out[b] = b == nb - 1 ? __int_as_float(0x7f800000) : k;
  }
}

// 64-bit candidate key: larger = better (score, then lower id); 0 = none.
__device__ __forceinline__ unsigned long long cand_key(float score, int id) {
  return (static_cast<unsigned long long>(order_key(score)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(id));
}

// In-place bitonic sort of n (a power of two) keys in shared memory, descending.
__device__ void bitonic_desc(unsigned long long* v, int n) {
  for (int k = 2; k <= n; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kMergeThreads) {
        const int p = i ^ j;
        if (p > i) {
          const bool desc = (i & k) == 0;
          const unsigned long long x = v[i], y = v[p];
          if (desc ? x < y : x > y) {
            v[i] = y;
            v[p] = x;
          }
        }
      }
      __syncthreads();
    }
}

__global__ void __launch_bounds__(kMergeThreads) merge_topk_kernel(const DcpTopkArgs a) {
  __shared__ unsigned long long cand[kMaxCand];
  const int t = blockIdx.x, W = a.world, k = a.topk;
  int n = 1;
  while (n < W * k) n <<= 1;
  for (int i = threadIdx.x; i < n; i += kMergeThreads) {
    unsigned long long key = 0;
    if (i < W * k) {
      const int r = i / k, j = i % k;
      const int64_t off = r * a.rank_stride + static_cast<int64_t>(t) * a.local_stride + j;
      const int lp = a.pos_local[off];
      if (lp >= 0) key = cand_key(a.score_local[off], lp * W + r);
    }
    cand[i] = key;
  }
  __syncthreads();
  bitonic_desc(cand, n);
  // the first k live candidates are the global top-k; order their ids ascending
  // (a descending sort of the complemented ids)
  int m = 1;
  while (m < k) m <<= 1;
  for (int i = threadIdx.x; i < m; i += kMergeThreads) {
    const unsigned long long key = i < k ? cand[i] : 0;
    // ids as keys: larger key = lower id; scores ride in the low word for output
    cand[kMaxCand / 2 + i] =
        key == 0 ? 0 : (static_cast<unsigned long long>(static_cast<uint32_t>(key)) << 32) | static_cast<uint32_t>(key >> 32);
  }
  __syncthreads();
  bitonic_desc(cand + kMaxCand / 2, m);
  int32_t* op = a.out_pos + static_cast<int64_t>(t) * a.out_stride;
  float* os = a.out_score != nullptr ? a.out_score + static_cast<int64_t>(t) * a.out_stride : nullptr;
  for (int i = threadIdx.x; i < k; i += kMergeThreads) {
    const unsigned long long key = cand[kMaxCand / 2 + i];
    op[i] = key == 0 ? -1 : static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key >> 32));
    if (os) os[i] = key == 0 ? -__int_as_float(0x7f800000) : order_key_inv(static_cast<uint32_t>(key));
  }
}

}  // namespace

cudaError_t launch_dcp_merge_keys(const DcpKeysArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return cudaSuccess;
  merge_keys_kernel<<<a.rows, kMergeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dcp_merge_topk(const DcpTopkArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return cudaSuccess;
  merge_topk_kernel<<<a.rows, kMergeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ci
