// Level one, publishing: each row's candidate blocks from its block keys.
//
// Rows with nb_t = ceil(L_t / 8) <= topk_blocks keep every block; the others
// keep the topk_blocks largest keys (ties toward the lower block id).  The ids
// come out ascending and INT32_MAX padded (sglang PR #40352 "Score prefill
// consumer index layers on candidate blocks with DeepGEMM", Design, "Level
// one": ragged top-k over the keys, trivial path for rows with at most 2048
// blocks, sort_candidate_blocks ascending with INT32_MAX padding).
//
// One CTA per row.  The row's keys are staged once in shared memory as
// order-preserving uint32 codes; a radix select finds the threshold and an
// ordered compaction writes the winners in ascending id order, so no sort is
// needed.
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kThreads = 512;

__global__ void __launch_bounds__(kThreads) publish_kernel(const PublishArgs a) {
  extern __shared__ uint32_t sk[];
  __shared__ TopkShared sh;
  const int row = blockIdx.x, tid = threadIdx.x;
  int L = a.seq_len[row];
  if (L < 0 || L > a.max_len) {
    if (tid == 0) report(a.dev_err, kDevErrLen);
    L = 0;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  const int K = a.topk_blocks;
  int32_t* out = a.blocks + static_cast<int64_t>(row) * a.blocks_stride;
  if (tid == 0) a.nvalid[row] = min(nb, K);
  if (nb <= K) {
    for (int i = tid; i < K; i += kThreads) out[i] = i < nb ? i : 0x7FFFFFFF;
    return;
  }
  const float* keys = a.keys + static_cast<int64_t>(row) * a.keys_stride;
  const int nb4 = nb & ~3;
  for (int i = tid * 4; i < nb4; i += kThreads * 4) {
    const float4 v = *reinterpret_cast<const float4*>(keys + i);
    *reinterpret_cast<uint4*>(sk + i) = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
  }
  for (int i = nb4 + tid; i < nb; i += kThreads) sk[i] = order_key(keys[i]);
  __syncthreads();
  block_topk(sk, nb, K, sh, tid, kThreads, 1, [&](int rank, int idx, uint32_t) { out[rank] = idx; });
}

}  // namespace

cudaError_t launch_publish(const PublishArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return cudaSuccess;
  const int nb_max = (a.max_len + kBlock - 1) / kBlock;
  const int smem = ((max(nb_max, 4) + 3) & ~3) * 4;
  cudaError_t e = cudaFuncSetAttribute(publish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  publish_kernel<<<a.rows, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ci
