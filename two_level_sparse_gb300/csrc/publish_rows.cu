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
// This file serves launches with few rows (fewer than two per SM; publish.cu
// takes the others, several rows per SM at a time).  Persistent CTAs of 1024
// threads, one row at a time, the next row's keys prefetched into L2 while the
// current one is selected.  A row's keys are
// read once and kept in shared memory as order-preserving uint32 codes.  Two
// ways to the threshold:
//
//  * bracketed (long rows, K <= 2560): a strided sample of 1 key in 16 (at
//    most 2048) gives a lower bound for the K-th largest key, an order
//    statistic of the sample four standard deviations of the sampling noise
//    below its expected rank; one counting pass checks it (at least K keys
//    at or above it, no more than the list holds) and an ordered compaction
//    copies those keys -- about 1.4 K of them, in ascending id order -- into
//    a list.  Every winner is in the list, so the exact threshold is a radix
//    selection on the list and the winners a compaction of it.  Every key is
//    touched by three cheap passes (load, count, compact) and no atomic: the
//    selection's histograms see only the sample and the list;
//  * radix (short rows, wide K, or a bound the sample missed): a 4096-bin
//    histogram of the codes' top 12 bits, then 10-bit passes over the keys
//    sharing the chosen prefix, then an ordered compaction of all keys.
//
// Either way the narrower selection is taken from the wider one's winners
// (its top K' lie inside the top K >= K' under the same order), ascending.
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins1 = 4096;  // key bits 31..20
constexpr int kBins2 = 1024;  // key bits 19..10, then 9..0
// bracketed selection
constexpr int kSamples = 2048;
constexpr int kListCap = 4096;        // keys at or above the lower bound (at most 4 per thread)
constexpr int kFastMaxK = 2560;       // widest selection it serves
constexpr int kFastMinBlocks = 4096;  // shorter rows take the radix path

struct PublishShared {
  uint32_t h1[kBins1];
  uint32_t h2[2][kBins2];
  uint32_t part[2][kWarps];
  uint32_t warp_gt[kWarps], warp_eq[kWarps];
  unsigned long long wtot[kWarps];
  uint32_t digit[2], rem[2], match[2];
  int overflow;
};

// Dynamic shared memory after the row's codes, when it fits (see launch_publish).
// The list has one region of kRegion slots per warp (warp w's keys, ascending).
constexpr int kRegion = kListCap / kWarps;  // 128: four slots per lane
struct FastArea {
  uint32_t samp[kSamples];
  uint32_t lcode[kListCap];
  int32_t lid[kListCap];
  uint32_t rcount[kWarps];
};
constexpr size_t kFastAreaBytes = sizeof(FastArea);

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
  // bins of the warps above this one: a suffix sum over the 32 warp totals
  uint32_t wsuf = sh.part[0][lane];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, wsuf, o);
    if (lane + o < 32) wsuf += v;
  }
  const uint32_t warps_above = __shfl_sync(0xffffffffu, wsuf, (wid + 1) & 31);
  uint32_t above = suffix - lsum + (wid + 1 < kWarps ? warps_above : 0u);
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

// A threshold: entries whose code under `mask` exceeds `prefix` are taken,
// and the first `need` (in order) whose code under `mask` equals it.
struct Sel {
  uint32_t prefix, mask, need;
};

// Radix selection of the `k` largest of n <= 4096 codes held in shared memory
// (11, 11 and 10-bit digits; stops as soon as the threshold bucket is taken
// whole).  k must be in [1, n].
__device__ Sel list_select(const uint32_t* codes, int n, uint32_t k, PublishShared& sh, int tid) {
  Sel s{0u, 0u, k};
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  for (int p = 0; p < 3; ++p) {
    const int nbins = 1 << widths[p], shift = shifts[p];
    const uint32_t dmask = static_cast<uint32_t>(nbins - 1);
    for (int i = tid; i < nbins; i += kThreads) sh.h1[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t c = codes[i];
      if ((c & s.mask) == s.prefix) atomicAdd(&sh.h1[(c >> shift) & dmask], 1u);
    }
    __syncthreads();
    const uint32_t want[2] = {s.need, 0u};
    find_digit(sh.h1, nbins, want, sh, tid);
    s.prefix |= sh.digit[0] << shift;
    s.mask |= dmask << shift;
    s.need = sh.rem[0];
    if (sh.match[0] == sh.rem[0]) break;
  }
  return s;
}

// The four list slots of thread t: 4 t .. 4 t + 3, all in its warp's region
// (slot 4 lane + j of region wid, live below the region's count).
struct Slots {
  uint32_t c[4];
  bool live[4];
};
__device__ __forceinline__ Slots load_slots(const FastArea& fa, int tid) {
  Slots r;
  const int n = static_cast<int>(fa.rcount[tid >> 5]), l4 = 4 * (tid & 31);
  const uint4 v = *reinterpret_cast<const uint4*>(&fa.lcode[4 * tid]);
  r.c[0] = v.x;
  r.c[1] = v.y;
  r.c[2] = v.z;
  r.c[3] = v.w;
#pragma unroll
  for (int j = 0; j < 4; ++j) r.live[j] = l4 + j < n;
  return r;
}

// Radix selection of the want[s] largest live slots of the list, for both
// selections at once (want[1] may be 0): a shared first digit, then a
// histogram per open selection.
__device__ void regions_select(const Slots& sl, const uint32_t (&want)[2], Sel (&out)[2], PublishShared& sh,
                               int tid) {
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  bool open[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    out[s] = Sel{0u, 0u, want[s]};
    open[s] = want[s] > 0;
  }
  for (int p = 0; p < 3 && (open[0] || open[1]); ++p) {
    const int nbins = 1 << widths[p], shift = shifts[p];
    const uint32_t dmask = static_cast<uint32_t>(nbins - 1);
    const bool shared_digit = p == 0;  // both prefixes are still empty
    for (int i = tid; i < 2 * nbins; i += kThreads) sh.h1[i] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!sl.live[j]) continue;
      const uint32_t c = sl.c[j], d = (c >> shift) & dmask;
      if (shared_digit) {
        atomicAdd(&sh.h1[d], 1u);
      } else {
#pragma unroll
        for (int s = 0; s < 2; ++s)
          if (open[s] && (c & out[s].mask) == out[s].prefix) atomicAdd(&sh.h1[s * nbins + d], 1u);
      }
    }
    __syncthreads();
    if (shared_digit) {
      const uint32_t w2[2] = {out[0].need, out[1].need};
      find_digit(sh.h1, nbins, w2, sh, tid);
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      if (!open[s]) continue;
      if (!shared_digit) {
        const uint32_t ws[2] = {s == 0 ? out[0].need : 0u, s == 1 ? out[1].need : 0u};
        find_digit(sh.h1 + s * nbins, nbins, ws, sh, tid);
      }
      out[s].prefix |= sh.digit[s] << shift;
      out[s].mask |= dmask << shift;
      out[s].need = sh.rem[s];
      open[s] = sh.match[s] != sh.rem[s];
    }
  }
}

// Ordered compaction of the list's live slots under both thresholds at once:
// out_s[rank] = id of each selected slot, in list (= id) order.  The counts
// ride packed in 64 bits: per selection, above-threshold count in bits 0-15
// and at-threshold count in bits 16-31 (at most 4096 each).
__device__ void regions_emit(const Slots& sl, const FastArea& fa, const Sel (&sel)[2], int32_t* out0, int32_t* out1,
                             PublishShared& sh, int tid) {
  const int lane = tid & 31, wid = tid >> 5;
  bool gt[2][4], eq[2][4];
  unsigned long long cnt = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t m = sl.c[j] & sel[s].mask;
      gt[s][j] = sl.live[j] && m > sel[s].prefix;
      eq[s][j] = sl.live[j] && m == sel[s].prefix;
      cnt += static_cast<unsigned long long>((gt[s][j] ? 1u : 0u) + (eq[s][j] ? 0x10000u : 0u)) << (32 * s);
    }
  unsigned long long incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) sh.wtot[wid] = incl;
  __syncthreads();
  unsigned long long wx = sh.wtot[lane], wincl = wx;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long x = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += x;
  }
  const unsigned long long warps_before = __shfl_sync(0xffffffffu, wincl - wx, wid);
  unsigned long long before = warps_before + incl - cnt;
  int32_t* outs[2] = {out0, out1};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t b = static_cast<uint32_t>(before >> (32 * s));
      const uint32_t gb = b & 0xFFFFu, eb = b >> 16;
      if (outs[s] != nullptr && (gt[s][j] || (eq[s][j] && eb < sel[s].need)))
        outs[s][gb + min(eb, sel[s].need)] = fa.lid[4 * tid + j];
      before += static_cast<unsigned long long>((gt[s][j] ? 1u : 0u) + (eq[s][j] ? 0x10000u : 0u)) << (32 * s);
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

// Radix path: thresholds for one or two selections over all nb codes.
__device__ void radix_thresholds(const uint32_t* sk, int nb, const uint32_t (&want)[2], uint32_t (&prefix)[2],
                                 uint32_t (&mask)[2], uint32_t (&need)[2], PublishShared& sh, int tid) {
  for (int i = tid; i < kBins1; i += kThreads) sh.h1[i] = 0;
  __syncthreads();
  for (int i = tid; i < nb; i += kThreads) atomicAdd(&sh.h1[sk[i] >> 20], 1u);
  __syncthreads();
  find_digit(sh.h1, kBins1, want, sh, tid);
  bool open[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    prefix[s] = want[s] ? sh.digit[s] << 20 : 0u;
    mask[s] = 0xFFF00000u;
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
}

// The bracketed selection of the want[s] largest codes for both selections
// at once (max <= kFastMaxK; want[s] = 0: none).  Returns false, having
// written nothing, when fewer than the wider selection's count reach the
// sample's bound or a warp's list region would overflow; the caller then
// takes the radix path.
__device__ bool bracketed_select(const uint32_t* sk, int nb, const uint32_t (&want)[2], int32_t* out0, int32_t* out1,
                                 FastArea& fa, PublishShared& sh, int tid) {
  const int wid = tid >> 5, lane = tid & 31;
  const uint32_t kb = max(want[0], want[1]);
  // the sample: about every stride-th code, at most kSamples of them (offset
  // by m % 16 so that the reads spread over the banks)
  const int stride = max(16, (nb + kSamples - 1) / kSamples);
  const int S = (nb + stride - 1) / stride;
  for (int m = tid; m < S; m += kThreads) fa.samp[m] = sk[min(m * stride + (m & 15), nb - 1)];
  if (tid == 0) sh.overflow = 0;
  __syncthreads();
  // the rank the K-th largest key has in the sample, plus a margin of four
  // standard deviations of its binomial spread and a little; the bound is the
  // bottom of the bucket holding the sample of that rank (code 0 is no key)
  const float est = static_cast<float>(kb) * static_cast<float>(S) / static_cast<float>(nb);
  const int r_lo = static_cast<int>(ceilf(est + 4.0f * sqrtf(est) + 4.0f));
  uint32_t t_lo = 1u;
  if (r_lo <= S) t_lo = max(list_select(fa.samp, S, static_cast<uint32_t>(r_lo), sh, tid).prefix, 1u);
  // the keys at or above t_lo, each warp's contiguous share of the ids into
  // its own region of the list, in ascending order
  const int seg = ((nb + kWarps - 1) / kWarps + 31) & ~31;
  const int begin = min(nb, wid * seg), end = min(nb, begin + seg);
  const uint32_t lt = lanemask_lt();
  uint32_t n = 0;
  for (int b0 = begin; b0 < end; b0 += 32) {
    const int i = b0 + lane;
    const uint32_t c = i < end ? sk[i] : 0u;
    const bool f = i < end && c >= t_lo;
    const uint32_t bal = __ballot_sync(0xffffffffu, f);
    const uint32_t r = n + __popc(bal & lt);
    if (f && r < static_cast<uint32_t>(kRegion)) {
      fa.lcode[wid * kRegion + r] = c;
      fa.lid[wid * kRegion + r] = i;
    }
    n += __popc(bal);
  }
  if (lane == 0) {
    fa.rcount[wid] = min(n, static_cast<uint32_t>(kRegion));
    sh.warp_eq[wid] = n;
    if (n > static_cast<uint32_t>(kRegion)) sh.overflow = 1;
  }
  __syncthreads();
  uint32_t total = sh.warp_eq[lane];
  total = __reduce_add_sync(0xffffffffu, total);
  // every winner is at or above t_lo when at least kb keys are
  if (sh.overflow || total < kb) return false;
  const Slots sl = load_slots(fa, tid);
  Sel sel[2];
  regions_select(sl, want, sel, sh, tid);
  regions_emit(sl, fa, sel, want[0] ? out0 : nullptr, want[1] ? out1 : nullptr, sh, tid);
  return true;
}

__global__ void __launch_bounds__(kThreads, 1) publish_row_kernel(const PublishArgs a, int fast) {
  extern __shared__ __align__(16) uint32_t sk[];
  __shared__ PublishShared sh;
  const int tid = threadIdx.x;
  const int nb_pad = (((a.max_len + kBlock - 1) / kBlock) + 3) & ~3;
  FastArea& fa = *reinterpret_cast<FastArea*>(sk + nb_pad);
  for (int row = blockIdx.x; row < a.rows; row += gridDim.x) {
    int L = a.seq_len[row];
    if (L < 0 || L > a.max_len) {
      if (tid == 0) report(a.dev_err, kDevErrLen);
      L = 0;
    }
    const int nb = (L + kBlock - 1) / kBlock;
    // the next row of this CTA: its keys into L2 while this one is selected
    const int next = row + gridDim.x;
    if (tid < 8 && next < a.rows) {
      const int Ln = a.seq_len[next];
      const int nbn = (min(max(Ln, 0), a.max_len) + kBlock - 1) / kBlock;
      if (nbn > min(a.topk_blocks, a.blocks2 != nullptr ? a.topk_blocks2 : a.topk_blocks)) {
        const uint32_t bytes = static_cast<uint32_t>((nbn * 4 + 15) & ~15);
        const uint32_t chunk = ((bytes / 8) + 15) & ~15u;
        const uint32_t off = chunk * tid;
        if (off < bytes)
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                           reinterpret_cast<const uint8_t*>(a.keys + static_cast<int64_t>(next) * a.keys_stride) + off),
                       "r"(min(chunk, bytes - off))
                       : "memory");
      }
    }
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
    if (want[0] == 0 && want[1] == 0) continue;  // CTA-uniform

    // keys -> order codes in shared memory (16-byte loads, a batch in flight)
    const float* keys = a.keys + static_cast<int64_t>(row) * a.keys_stride;
    const int nb4 = nb & ~3;
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
        *reinterpret_cast<uint4*>(sk + i) =
            make_uint4(order_key(v[j].x), order_key(v[j].y), order_key(v[j].z), order_key(v[j].w));
      }
    }
    for (int i = nb4 + tid; i < nb; i += kThreads) sk[i] = order_key(keys[i]);
    __syncthreads();

    const int big = want[0] >= want[1] ? 0 : 1, small = 1 - big;
    const uint32_t kb = want[big], ks = want[small];
    bool done = false;
    if (fast && nb >= kFastMinBlocks && kb <= static_cast<uint32_t>(kFastMaxK))
      done = bracketed_select(sk, nb, want, out[0], out[1], fa, sh, tid);
    if (!done) {
      // the wider selection over every key, the narrower from its winners
      uint32_t prefix[2], mask[2], need[2];
      radix_thresholds(sk, nb, want, prefix, mask, need, sh, tid);
      emit_selected(sk, nb, prefix[big], mask[big], need[big], out[big], sh, tid);
      if (ks) {
        // visible to the whole CTA after emit_selected's closing barrier
        emit_selected(sk, static_cast<int>(kb), prefix[small], mask[small], need[small], out[small], sh, tid,
                      out[big]);
      }
    }
    __syncthreads();  // shared memory is reused by the next row
  }
}

}  // namespace

cudaError_t launch_publish_rows(const PublishArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return cudaSuccess;
  const int nb_max = (a.max_len + kBlock - 1) / kBlock;
  const size_t codes = static_cast<size_t>((max(nb_max, 4) + 3) & ~3) * 4;
  // the bracketed path's scratch follows the codes when both fit
  const size_t limit = 232448 - sizeof(PublishShared) - 1024;
  const int fast = codes + kFastAreaBytes <= limit ? 1 : 0;
  const int smem = static_cast<int>(codes + (fast ? kFastAreaBytes : 0));
  cudaError_t e = cudaFuncSetAttribute(publish_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = a.rows < device_sm_count() ? a.rows : device_sm_count();
  publish_row_kernel<<<grid, kThreads, smem, stream>>>(a, fast);
  return cudaGetLastError();
}

}  // namespace ci
