// The published table restricted to the tail rows of each request (sglang
// PR #40352, Design: prefill_tail restricts what was published to the last
// rows of each request, for the late layers that run on the tail only).
//
// Request r owns rows req_start[r] .. req_start[r+1]-1 and keeps its last
// m_r = min(max(tail_len[r], 0), n_r) of them.  Output rows are the kept rows
// in order: request r's start at the exclusive prefix sum of m.  One launch:
// every CTA rebuilds the per-request prefix in shared memory (at most 4096
// requests), then copies its share of the output rows (their block ids and
// count) and names each one's source row.
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kThreads = 256;  // a 2048-id row is two 16-byte copies per thread
constexpr int kPer = kMaxReq / kThreads;

__global__ void __launch_bounds__(kThreads) tail_kernel(const TailArgs a) {
  __shared__ int32_t tstart[kMaxReq + 1];  // output row of each request's first tail row
  __shared__ int32_t wsum[kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int m[kPer], local = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int r = tid * kPer + j;
    m[j] = 0;
    if (r < a.num_req) {
      const int s0 = a.req_start[r], s1 = a.req_start[r + 1];
      const bool ok = 0 <= s0 && s0 <= s1 && s1 <= a.rows && (r > 0 || s0 == 0) && (r < a.num_req - 1 || s1 == a.rows);
      if (!ok && blockIdx.x == 0) report(a.dev_err, kDevErrReq);
      m[j] = ok ? min(max(a.tail_len[r], 0), s1 - s0) : 0;
    }
    local += m[j];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) before += wsum[w];
    total += wsum[w];
  }
  int run = before + incl - local;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int r = tid * kPer + j;
    if (r < a.num_req) tstart[r] = run;
    run += m[j];
  }
  if (tid == 0) tstart[a.num_req] = total;
  __syncthreads();
  if (blockIdx.x == 0 && tid == 0) {
    *a.out_count = total;
    if (total > a.out_cap) report(a.dev_err, kDevErrReq);
  }
  const int n = min(total, a.out_cap);
  // 16-byte copies when every row of both tables starts on a 16-byte boundary
  const bool vec = ((a.topk_blocks | a.blocks_stride | a.out_blocks_stride) & 3) == 0 &&
                   ((reinterpret_cast<uintptr_t>(a.blocks) | reinterpret_cast<uintptr_t>(a.out_blocks)) & 15) == 0;
  const int nvec = vec ? a.topk_blocks / 4 : 0;
  for (int o = blockIdx.x; o < a.out_cap; o += gridDim.x) {
    int src = -1;
    if (o < n) {
      int lo = 0, hi = a.num_req;  // the request r with tstart[r] <= o < tstart[r + 1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tstart[mid] <= o)
          lo = mid;
        else
          hi = mid;
      }
      src = a.req_start[lo + 1] - (tstart[lo + 1] - tstart[lo]) + (o - tstart[lo]);
    }
    int32_t* ob = a.out_blocks + static_cast<int64_t>(o) * a.out_blocks_stride;
    if (src >= 0) {
      const int32_t* ib = a.blocks + static_cast<int64_t>(src) * a.blocks_stride;
      for (int i = tid; i < nvec; i += kThreads) reinterpret_cast<int4*>(ob)[i] = reinterpret_cast<const int4*>(ib)[i];
      for (int i = 4 * nvec + tid; i < a.topk_blocks; i += kThreads) ob[i] = ib[i];
    } else {
      const int4 pad = make_int4(0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF);
      for (int i = tid; i < nvec; i += kThreads) reinterpret_cast<int4*>(ob)[i] = pad;
      for (int i = 4 * nvec + tid; i < a.topk_blocks; i += kThreads) ob[i] = 0x7FFFFFFF;
    }
    if (tid == 0) {
      a.out_row[o] = src;
      a.out_nvalid[o] = src >= 0 ? a.nvalid[src] : 0;
    }
  }
}

}  // namespace

cudaError_t launch_tail(const TailArgs& a, cudaStream_t stream) {
  // one output row per CTA (several rounds only past 64 K rows): the rows'
  // copies all start at once instead of one after another in each CTA
  const int grid = max(1, min(a.out_cap, 65536));
  tail_kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ci
