// Level one, publishing: each row's candidate blocks from its block keys,
// for one or two block counts at once (the consumers' K and the source's own
// K' = P + 1 are selected from the same keys).
//
// Rows with nb_t = ceil(L_t / 8) <= K keep every block; the others keep the K
// largest keys (ties toward the lower block id).  The ids come out ascending
// and INT32_MAX padded (sglang PR #40352 "Score prefill consumer index layers
// on candidate blocks with DeepGEMM", Design, "Level one": ragged top-k over
// the keys, trivial path for rows with at most 2048 blocks,
// sort_candidate_blocks ascending with INT32_MAX padding).
//
// One CTA per row.  The row's keys are read once, converted to
// order-preserving uint32 codes in shared memory, and histogrammed on their
// top 12 bits (sign, exponent, 3 mantissa bits) on the way in: keys of one
// row concentrate on few exponents, so a wide first digit spreads the
// histogram's atomics where an 8-bit one would pile them onto a handful of
// bins.  That histogram serves both selections; two 10-bit passes over the
// keys sharing the chosen prefix finish each threshold (skipped as soon as
// the threshold bucket is taken whole).  An ordered compaction per selection
// writes the winners in ascending id order, so no sort is needed; the
// narrower selection compacts only the wider one's winners (its top K' lie
// inside the top K >= K' under the same order).
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins1 = 4096;  // key bits 31..20
constexpr int kBins2 = 1024;  // key bits 19..10, then 9..0

struct PublishShared {
  uint32_t h1[kBins1];
  uint32_t h2[2][kBins2];
  uint32_t part[2][kWarps];
  uint32_t warp_gt[kWarps], warp_eq[kWarps];
  uint32_t digit[2], rem[2], match[2];
};

// For each selection s with want[s] > 0: the bin d (bins numbered upward) such
// that the keys in bins above d number fewer than want[s] and those in bins
// >= d at least want[s]; rem[s] = want[s] minus the keys above d, match[s] =
// the keys in bin d.  Thread t owns bins [t * per, (t + 1) * per).
__device__ __forceinline__ void find_digit(const uint32_t* hist, int nbins, const uint32_t (&want)[2],
                                           PublishShared& sh, int tid) {
  const int per = nbins / kThreads, lane = tid & 31, wid = tid >> 5;
  uint32_t c[4] = {0, 0, 0, 0}, lsum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < per) {
      c[j] = hist[tid * per + j];
      lsum += c[j];
    }
  uint32_t suffix = lsum;  // over lanes >= lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, suffix, o);
    if (lane + o < 32) suffix += v;
  }
  if (lane == 0) sh.part[0][wid] = suffix;
  __syncthreads();
  uint32_t above = suffix - lsum;
  for (int w = wid + 1; w < kWarps; ++w) above += sh.part[0][w];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const uint32_t k = want[s];
    if (k == 0 || !(above < k && k <= above + lsum)) continue;
    uint32_t acc = above;
    for (int j = per - 1; j >= 0; --j) {
      if (acc + c[j] >= k) {
        sh.digit[s] = tid * per + j;
        sh.rem[s] = k - acc;
        sh.match[s] = c[j];
        break;
      }
      acc += c[j];
    }
  }
  __syncthreads();
}

// Ordered compaction of the keys above the threshold (prefix under mask) and
// the first need_eq at it, in index order: warps own contiguous segments.
// Candidates are the block ids 0 .. n - 1, or, with ids, the n ascending ids
// ids[0 .. n - 1] (a wider selection's winners).
__device__ __forceinline__ void emit_selected(const uint32_t* sk, int n, uint32_t prefix, uint32_t mask,
                                              uint32_t need_eq, int32_t* out, PublishShared& sh, int tid,
                                              const int32_t* ids = nullptr) {
  const int wid = tid >> 5, lane = tid & 31;
  const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int begin = min(n, wid * seg), end = min(n, begin + seg);
  uint32_t gt = 0, eq = 0;
  for (int i = begin + lane; i < end; i += 32) {
    const uint32_t m = sk[ids != nullptr ? ids[i] : i] & mask;
    gt += m > prefix;
    eq += m == prefix;
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (lane == 0) {
    sh.warp_gt[wid] = gt;
    sh.warp_eq[wid] = eq;
  }
  __syncthreads();
  uint32_t gt_before = 0, eq_before = 0;
  for (int w = 0; w < wid; ++w) {
    gt_before += sh.warp_gt[w];
    eq_before += sh.warp_eq[w];
  }
  const uint32_t lt = lanemask_lt();
  for (int base = begin; base < end; base += 32) {
    const int i = base + lane;
    const bool valid = i < end;
    const int id = valid ? (ids != nullptr ? ids[i] : i) : 0;
    const uint32_t m = valid ? sk[id] & mask : 0u;
    const bool is_gt = valid && m > prefix;
    const bool is_eq = valid && m == prefix;
    const uint32_t bg = __ballot_sync(0xffffffffu, is_gt);
    const uint32_t be = __ballot_sync(0xffffffffu, is_eq);
    const uint32_t eq_rank = eq_before + __popc(be & lt);
    if (is_gt || (is_eq && eq_rank < need_eq)) out[gt_before + __popc(bg & lt) + min(eq_rank, need_eq)] = id;
    gt_before += __popc(bg);
    eq_before += __popc(be);
  }
  __syncthreads();  // the shared counts are reused by the next selection
}

__global__ void __launch_bounds__(kThreads, 1) publish_kernel(const PublishArgs a) {
  extern __shared__ uint32_t sk[];
  __shared__ PublishShared sh;
  const int row = blockIdx.x, tid = threadIdx.x;
  int L = a.seq_len[row];
  if (L < 0 || L > a.max_len) {
    if (tid == 0) report(a.dev_err, kDevErrLen);
    L = 0;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  const int K[2] = {a.topk_blocks, a.topk_blocks2};
  int32_t* out[2] = {a.blocks + static_cast<int64_t>(row) * a.blocks_stride,
                     a.blocks2 != nullptr ? a.blocks2 + static_cast<int64_t>(row) * a.blocks2_stride : nullptr};
  int32_t* nvalid[2] = {a.nvalid, a.nvalid2};
  uint32_t want[2] = {0, 0};
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    if (K[s] <= 0 || out[s] == nullptr) continue;
    if (tid == 0) nvalid[s][row] = min(nb, K[s]);
    if (nb <= K[s]) {
      for (int i = tid; i < K[s]; i += kThreads) out[s][i] = i < nb ? i : 0x7FFFFFFF;
    } else {
      want[s] = static_cast<uint32_t>(K[s]);
    }
  }
  if (want[0] == 0 && want[1] == 0) return;

  // keys -> order codes in shared memory, histogram of their top 12 bits
  for (int i = tid; i < kBins1; i += kThreads) sh.h1[i] = 0;
  __syncthreads();
  const float* keys = a.keys + static_cast<int64_t>(row) * a.keys_stride;
  const int nb4 = nb & ~3;
  // kBatch 16-byte loads in flight per thread before their codes are counted
  constexpr int kBatch = 8;
  for (int i0 = tid * 4; i0 < nb4; i0 += kThreads * 4 * kBatch) {
    float4 v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j * kThreads * 4;
      v[j] = i < nb4 ? *reinterpret_cast<const float4*>(keys + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j * kThreads * 4;
      if (i >= nb4) break;
      const uint4 u = make_uint4(order_key(v[j].x), order_key(v[j].y), order_key(v[j].z), order_key(v[j].w));
      *reinterpret_cast<uint4*>(sk + i) = u;
      atomicAdd(&sh.h1[u.x >> 20], 1u);
      atomicAdd(&sh.h1[u.y >> 20], 1u);
      atomicAdd(&sh.h1[u.z >> 20], 1u);
      atomicAdd(&sh.h1[u.w >> 20], 1u);
    }
  }
  for (int i = nb4 + tid; i < nb; i += kThreads) {
    const uint32_t u = order_key(keys[i]);
    sk[i] = u;
    atomicAdd(&sh.h1[u >> 20], 1u);
  }
  __syncthreads();
  find_digit(sh.h1, kBins1, want, sh, tid);
  uint32_t prefix[2], mask[2] = {0xFFF00000u, 0xFFF00000u}, need[2];
  bool open[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    prefix[s] = want[s] ? sh.digit[s] << 20 : 0u;
    need[s] = want[s] ? sh.rem[s] : 0u;
    open[s] = want[s] && sh.match[s] != sh.rem[s];  // the bucket is not taken whole
  }
  // two 10-bit passes over the keys sharing the chosen prefix
  for (int shift = 10; shift >= 0 && (open[0] || open[1]); shift -= 10) {
    for (int i = tid; i < 2 * kBins2; i += kThreads) sh.h2[i / kBins2][i % kBins2] = 0;
    __syncthreads();
    for (int i = tid; i < nb; i += kThreads) {
      const uint32_t u = sk[i];
#pragma unroll
      for (int s = 0; s < 2; ++s)
        if (open[s] && (u & mask[s]) == prefix[s]) atomicAdd(&sh.h2[s][(u >> shift) & (kBins2 - 1)], 1u);
    }
    __syncthreads();
    uint32_t w2[2] = {open[0] ? need[0] : 0u, open[1] ? need[1] : 0u};
    for (int s = 0; s < 2; ++s) {
      if (!open[s]) continue;
      const uint32_t ws[2] = {s == 0 ? w2[0] : 0u, s == 1 ? w2[1] : 0u};
      find_digit(sh.h2[s], kBins2, ws, sh, tid);
      prefix[s] |= sh.digit[s] << shift;
      mask[s] |= static_cast<uint32_t>(kBins2 - 1) << shift;
      need[s] = sh.rem[s];
      open[s] = sh.match[s] != sh.rem[s];
    }
  }
  if (want[0]) emit_selected(sk, nb, prefix[0], mask[0], need[0], out[0], sh, tid);
  if (want[1]) {
    // The top K' (ties toward the lower id) lie inside the top K >= K': pick
    // them from the first selection's K ascending winners (visible to the
    // whole CTA after emit_selected's closing barrier) instead of all keys.
    if (want[0] && want[1] <= want[0])
      emit_selected(sk, static_cast<int>(want[0]), prefix[1], mask[1], need[1], out[1], sh, tid, out[0]);
    else
      emit_selected(sk, nb, prefix[1], mask[1], need[1], out[1], sh, tid);
  }
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
