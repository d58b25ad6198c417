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
// This file serves launches with at least two rows per SM (publish_rows.cu,
// one row per CTA at a time with the row's codes in shared memory, the
// others).  A row is handled by a group of G = 256 threads with a named
// barrier of its own, four rows in flight per SM.  The group streams its
// row's keys (from HBM, then L2) as order-preserving uint32 codes and selects
// with 8-bit radix digits.  (Prefetching each group's next row into L2 as well
// made the launch slower, 1.30 against 1.01 ms on 16384 rows: four rows in
// flight per SM and their successors outgrow L2.)  Two ways to the
// threshold:
//
//  * bracketed (long rows, K <= 2560): a strided sample of 1 key in 16 (at
//    most 2048) gives a lower bound for the K-th largest key, an order
//    statistic of the sample four standard deviations of the sampling noise
//    below its expected rank; one pass over the keys copies those at or above
//    it into a list (each warp its contiguous share of the ids into its own
//    region, in ascending order) and counts them.  When at least K reach the
//    bound and no region overflows, every winner is in the list, so the exact
//    thresholds are radix selections on the list and the winners an ordered
//    compaction of it;
//  * radix (short rows, wide K, or a bound the sample missed): digit passes
//    over all keys, then an ordered compaction of them.
//
// The narrower selection is taken from the same candidates as the wider one
// (its top K' lie inside the top K >= K' under the same order), ascending.
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kCtaThreads = 1024;
constexpr int kBins = 256;  // 8-bit digits
constexpr int kSamples = 2048;
constexpr int kListCap = 4096;        // keys at or above the lower bound
constexpr int kFastMaxK = 2560;       // widest selection the bracketed path serves
constexpr int kFastMinBlocks = 4096;  // shorter rows take the radix path

// One group's shared memory.
struct GroupShared {
  uint32_t hist[2][kBins];
  uint32_t part[kBins / 32];
  unsigned long long wtot[32];
  uint32_t wgt[32], weq[32];  // per-warp counts of an ordered compaction
  uint32_t rcount[32];        // live entries of each warp's list region
  uint32_t wn[32];            // keys each warp found at or above the bound
  uint32_t digit[2], rem[2], match[2];
  int overflow;
  uint32_t samp[kSamples];
  uint32_t lcode[kListCap];
  int32_t lid[kListCap];
};

// A threshold: codes whose bits under `mask` exceed `prefix` are taken, and
// the first `need` (in id order) whose bits under `mask` equal it.
struct Sel {
  uint32_t prefix, mask, need;
};

template <int G>
struct Group {
  static constexpr int kWarps = G / 32;
  GroupShared& sh;
  int t;    // thread index in the group
  int bar;  // the group's named barrier
  __device__ __forceinline__ void sync() const { named_sync(bar, G); }
};

// For each selection s with want[s] > 0: the bin d (bins numbered upward) such
// that the codes in bins above d number fewer than want[s] and those in bins
// >= d at least want[s]; rem[s] = want[s] minus the codes above d, match[s] =
// the codes in bin d.  Threads 0..255 own one bin each.
template <int G>
__device__ void find_digit(const Group<G>& g, const uint32_t* hist, uint32_t want0, uint32_t want1) {
  const int lane = g.t & 31, wid = g.t >> 5;
  uint32_t c = 0, suffix = 0;
  if (g.t < kBins) {
    c = hist[g.t];
    suffix = c;  // over this warp's bins >= mine
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_down_sync(0xffffffffu, suffix, o);
      if (lane + o < 32) suffix += v;
    }
    if (lane == 0) g.sh.part[wid] = suffix;
  }
  g.sync();
  if (g.t < kBins) {
    uint32_t above = suffix - c;
    for (int w = wid + 1; w < kBins / 32; ++w) above += g.sh.part[w];
    const uint32_t want[2] = {want0, want1};
#pragma unroll
    for (int s = 0; s < 2; ++s)
      if (want[s] != 0 && above < want[s] && want[s] <= above + c) {
        g.sh.digit[s] = static_cast<uint32_t>(g.t);
        g.sh.rem[s] = want[s] - above;
        g.sh.match[s] = c;
      }
  }
  g.sync();
}

// Radix selection of the want[s] largest codes for up to two selections at
// once (want[s] = 0: none; each want[s] at most the number of codes), over
// the codes that each(f) hands to this thread (it calls f(code) for each):
// 8-bit digits, most significant first, one shared histogram while both
// prefixes are empty; a selection stops once its threshold bucket is taken
// whole.
//
// Every code handed over may share its bits above `top` with `prefix` (their
// common prefix, under `mask`): the digits then start at bit `top`.
template <int G, class Each>
__device__ void radix_select(const Group<G>& g, Each each, const uint32_t (&want)[2], Sel (&out)[2],
                             uint32_t prefix = 0u, uint32_t mask = 0u, int top = 31) {
  bool open[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    out[s] = Sel{prefix, mask, want[s]};
    open[s] = want[s] != 0;
  }
  for (int p = 0; top >= 0 && (open[0] || open[1]); ++p) {
    const int shift = max(top - 7, 0), width = top - shift + 1;
    const uint32_t dmask = (1u << width) - 1u;
    top = shift - 1;
    const bool shared = p == 0;
    for (int i = g.t; i < 2 * kBins; i += G) (&g.sh.hist[0][0])[i] = 0;
    g.sync();
    each([&](uint32_t c) {
      const uint32_t d = (c >> shift) & dmask;
      if (shared) {
        atomicAdd(&g.sh.hist[0][d], 1u);
      } else {
#pragma unroll
        for (int s = 0; s < 2; ++s)
          if (open[s] && (c & out[s].mask) == out[s].prefix) atomicAdd(&g.sh.hist[s][d], 1u);
      }
    });
    g.sync();
    if (shared) {
      find_digit(g, g.sh.hist[0], out[0].need, out[1].need);
    } else {
      if (open[0]) find_digit(g, g.sh.hist[0], out[0].need, 0u);
      if (open[1]) find_digit(g, g.sh.hist[1], 0u, out[1].need);
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      if (!open[s]) continue;
      out[s].prefix |= g.sh.digit[s] << shift;
      out[s].mask |= dmask << shift;
      out[s].need = g.sh.rem[s];
      open[s] = g.sh.match[s] != g.sh.rem[s];
    }
  }
}

// Four consecutive keys as codes (0 past `end`); i is a multiple of 4 and the
// row 16-byte aligned.
__device__ __forceinline__ void load4(const float* keys, int i, int end, uint32_t (&c)[4]) {
  if (i + 3 < end) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(keys + i));
    c[0] = order_key(v.x);
    c[1] = order_key(v.y);
    c[2] = order_key(v.z);
    c[3] = order_key(v.w);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = i + j < end ? order_key(__ldg(keys + i + j)) : 0u;
  }
}

// Ordered compaction of the list's live slots under both thresholds at once:
// out_s[rank] = id of each selected slot, in list (= id) order.  Warp w's
// region holds its entries in slots 32 j + lane (conflict-free); a first walk
// counts each warp's winners, a second writes them by ballot ranks.
template <int G>
__device__ void emit_list(const Group<G>& g, const Sel (&sel)[2], int32_t* out0, int32_t* out1) {
  constexpr int W = Group<G>::kWarps, kRegion = kListCap / W;
  const int lane = g.t & 31, wid = g.t >> 5;
  const int n = static_cast<int>(g.sh.rcount[wid]);
  const uint32_t* rcode = g.sh.lcode + wid * kRegion;
  const int32_t* rid = g.sh.lid + wid * kRegion;
  const uint32_t lt = lanemask_lt();
  uint32_t cgt[2] = {0, 0}, ceq[2] = {0, 0};
  for (int base = 0; base < n; base += 32) {
    const int r = base + lane;
    const uint32_t c = r < n ? rcode[r] : 0u;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t m = c & sel[s].mask;
      cgt[s] += __popc(__ballot_sync(0xffffffffu, r < n && m > sel[s].prefix));
      ceq[s] += __popc(__ballot_sync(0xffffffffu, r < n && m == sel[s].prefix));
    }
  }
  if (lane == 0) {
    g.sh.wgt[wid] = cgt[0] | (cgt[1] << 16);
    g.sh.weq[wid] = ceq[0] | (ceq[1] << 16);
  }
  g.sync();
  uint32_t gb[2] = {0, 0}, eb[2] = {0, 0};
  for (int w = 0; w < wid; ++w) {
    const uint32_t x = g.sh.wgt[w], y = g.sh.weq[w];
    gb[0] += x & 0xFFFFu;
    gb[1] += x >> 16;
    eb[0] += y & 0xFFFFu;
    eb[1] += y >> 16;
  }
  int32_t* outs[2] = {out0, out1};
  for (int base = 0; base < n; base += 32) {
    const int r = base + lane;
    const uint32_t c = r < n ? rcode[r] : 0u;
    const int32_t id = r < n ? rid[r] : 0;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t m = c & sel[s].mask;
      const bool is_gt = r < n && m > sel[s].prefix, is_eq = r < n && m == sel[s].prefix;
      const uint32_t bg = __ballot_sync(0xffffffffu, is_gt), be = __ballot_sync(0xffffffffu, is_eq);
      const uint32_t er = eb[s] + __popc(be & lt);
      if (outs[s] != nullptr && (is_gt || (is_eq && er < sel[s].need)))
        outs[s][gb[s] + __popc(bg & lt) + min(er, sel[s].need)] = id;
      gb[s] += __popc(bg);
      eb[s] += __popc(be);
    }
  }
  g.sync();
}

// The bracketed selection (see the top of the file) of the want[s] largest
// codes for both selections at once.  Returns false, having written nothing,
// when fewer than the wider selection's count reach the sample's bound or a
// warp's list region would overflow; the caller then takes the radix path.
template <int G>
__device__ bool bracketed_select(const Group<G>& g, const float* keys, int nb, const uint32_t (&want)[2],
                                 int32_t* out0, int32_t* out1) {
  constexpr int W = Group<G>::kWarps, kRegion = kListCap / W;
  const int lane = g.t & 31, wid = g.t >> 5;
  const uint32_t kb = max(want[0], want[1]);
  // the sample: about every stride-th code, at most kSamples of them
  const int stride = max(16, (nb + kSamples - 1) / kSamples);
  const int S = (nb + stride - 1) / stride;
  {
    constexpr int kPer = (kSamples + G - 1) / G;  // loads in flight together
    uint32_t v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int m = g.t + k * G;
      v[k] = m < S ? order_key(__ldg(keys + min(m * stride + (m & 15), nb - 1))) : 0u;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (g.t + k * G < S) g.sh.samp[g.t + k * G] = v[k];
  }
  if (g.t == 0) g.sh.overflow = 0;
  g.sync();
  // the rank the K-th largest key has in the sample, plus a margin of four
  // standard deviations of its binomial spread and a little; the bound is the
  // bottom of the bucket holding the sample of that rank (code 0 is no key)
  const float est = static_cast<float>(kb) * static_cast<float>(S) / static_cast<float>(nb);
  const int r_lo = static_cast<int>(ceilf(est + 4.0f * sqrtf(est) + 4.0f));
  uint32_t t_lo = 1u;
  if (r_lo <= S) {
    const uint32_t w[2] = {static_cast<uint32_t>(r_lo), 0u};
    Sel sb[2];
    radix_select(
        g,
        [&](auto f) {
          for (int m = g.t; m < S; m += G) f(g.sh.samp[m]);
        },
        w, sb);
    t_lo = max(sb[0].prefix, 1u);
  }
  // the keys at or above t_lo, each warp's contiguous share of the ids into
  // its own region of the list, in ascending order (four keys per lane per
  // step: id order is lane-major within a step)
  const int seg = ((nb + W - 1) / W + 127) & ~127;
  const int begin = min(nb, wid * seg), end = min(nb, begin + seg);
  const uint32_t lt = lanemask_lt();
  uint32_t* rcode = g.sh.lcode + wid * kRegion;
  int32_t* rid = g.sh.lid + wid * kRegion;
  uint32_t n = 0, cmax = 0;
  constexpr int kSteps = 4;  // steps whose loads are in flight together
  for (int b0 = begin; b0 < end; b0 += 128 * kSteps) {
    uint32_t c[kSteps][4];
#pragma unroll
    for (int u = 0; u < kSteps; ++u) load4(keys, b0 + 128 * u + 4 * lane, end, c[u]);
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      const int i0 = b0 + 128 * u + 4 * lane;
      uint32_t bal[4], below = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bal[j] = __ballot_sync(0xffffffffu, c[u][j] >= t_lo);
        below += __popc(bal[j] & lt);
      }
      uint32_t r = n + below;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (c[u][j] >= t_lo) {
          cmax = max(cmax, c[u][j]);
          if (r < static_cast<uint32_t>(kRegion)) {
            rcode[r] = c[u][j];
            rid[r] = i0 + j;
          }
          ++r;
        }
        n += __popc(bal[j]);
      }
    }
  }
  cmax = __reduce_max_sync(0xffffffffu, cmax);
  if (lane == 0) {
    g.sh.rcount[wid] = min(n, static_cast<uint32_t>(kRegion));
    g.sh.wn[wid] = n;
    g.sh.wgt[wid] = cmax;
    if (n > static_cast<uint32_t>(kRegion)) g.sh.overflow = 1;
  }
  g.sync();
  uint32_t total = lane < W ? g.sh.wn[lane] : 0u;
  total = __reduce_add_sync(0xffffffffu, total);
  // every list code lies in [t_lo, lmax]: their common leading bits are fixed
  const uint32_t lmax = __reduce_max_sync(0xffffffffu, lane < W ? g.sh.wgt[lane] : 0u);
  // every winner is at or above t_lo when at least kb keys are
  if (g.sh.overflow || total < kb) return false;
  Sel sel[2];
  const int live_n = static_cast<int>(g.sh.rcount[wid]);
  const uint32_t diff = t_lo ^ lmax;
  const int top = diff == 0 ? 0 : 31 - __clz(diff);
  const uint32_t cmask = top >= 31 ? 0u : ~((2u << top) - 1u);
  radix_select(
      g,
      [&](auto f) {
        for (int r = lane; r < live_n; r += 32) f(g.sh.lcode[wid * kRegion + r]);
      },
      want, sel, t_lo & cmask, cmask, top);
  emit_list(g, sel, want[0] ? out0 : nullptr, want[1] ? out1 : nullptr);
  return true;
}

// Ordered compaction of the keys above the threshold and the first sel.need
// at it, in id order: warps own contiguous segments.  Candidates are the
// block ids 0 .. n - 1, or, with ids, the n ascending ids ids[0 .. n - 1] (a
// wider selection's winners, written by this group before its last barrier).
template <int G>
__device__ void emit_stream(const Group<G>& g, const float* keys, int n, const Sel& sel, int32_t* out,
                            const int32_t* ids) {
  constexpr int W = Group<G>::kWarps;
  const int lane = g.t & 31, wid = g.t >> 5;
  const int seg = ((n + W - 1) / W + 31) & ~31;
  const int begin = min(n, wid * seg), end = min(n, begin + seg);
  auto code_of = [&](int i, int& id) -> uint32_t {
    id = ids != nullptr ? ids[i] : i;
    return order_key(__ldg(keys + id)) & sel.mask;
  };
  uint32_t gt = 0, eq = 0;
  for (int i = begin + lane; i < end; i += 32) {
    int id;
    const uint32_t m = code_of(i, id);
    gt += m > sel.prefix;
    eq += m == sel.prefix;
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (lane == 0) {
    g.sh.wgt[wid] = gt;
    g.sh.weq[wid] = eq;
  }
  g.sync();
  uint32_t gt_before = 0, eq_before = 0;
  for (int w = 0; w < wid; ++w) {
    gt_before += g.sh.wgt[w];
    eq_before += g.sh.weq[w];
  }
  const uint32_t lt = lanemask_lt();
  for (int base = begin; base < end; base += 32) {
    const int i = base + lane;
    const bool valid = i < end;
    int id = 0;
    const uint32_t m = valid ? code_of(i, id) : 0u;
    const bool is_gt = valid && m > sel.prefix;
    const bool is_eq = valid && m == sel.prefix;
    const uint32_t bg = __ballot_sync(0xffffffffu, is_gt);
    const uint32_t be = __ballot_sync(0xffffffffu, is_eq);
    const uint32_t eq_rank = eq_before + __popc(be & lt);
    if (is_gt || (is_eq && eq_rank < sel.need)) out[gt_before + __popc(bg & lt) + min(eq_rank, sel.need)] = id;
    gt_before += __popc(bg);
    eq_before += __popc(be);
  }
  g.sync();  // the winners are visible to the group; the shared counts are reused
}

template <int G>
__global__ void __launch_bounds__(kCtaThreads, 1) publish_kernel(const PublishArgs a) {
  constexpr int kGroups = kCtaThreads / G;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GroupShared* groups = reinterpret_cast<GroupShared*>(smem_raw);
  const int gi = static_cast<int>(threadIdx.x) / G;
  const Group<G> g{groups[gi], static_cast<int>(threadIdx.x) % G, 1 + gi};
  const int slots = static_cast<int>(gridDim.x) * kGroups;
  for (int row = static_cast<int>(blockIdx.x) * kGroups + gi; row < a.rows; row += slots) {
    int L = a.seq_len[row];
    if (L < 0 || L > a.max_len) {
      if (g.t == 0) report(a.dev_err, kDevErrLen);
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
      if (g.t == 0) nvalid[s][row] = min(nb, K[s]);
      if (nb <= K[s]) {
        for (int i = g.t; i < K[s]; i += G) out[s][i] = i < nb ? i : 0x7FFFFFFF;
      } else {
        want[s] = static_cast<uint32_t>(K[s]);
      }
    }
    if (want[0] == 0 && want[1] == 0) continue;  // group-uniform

    const float* keys = a.keys + static_cast<int64_t>(row) * a.keys_stride;
    const int big = want[0] >= want[1] ? 0 : 1, small = 1 - big;
    const uint32_t kb = want[big];
    bool done = false;
    if (nb >= kFastMinBlocks && kb <= static_cast<uint32_t>(kFastMaxK))
      done = bracketed_select(g, keys, nb, want, out[0], out[1]);
    if (!done) {
      // the thresholds over every key; the wider selection over every key,
      // the narrower from its winners
      Sel sel[2];
      radix_select(
          g,
          [&](auto f) {
            for (int i = 4 * g.t; i < nb; i += 16 * G) {
              uint32_t c[4][4];
#pragma unroll
              for (int u = 0; u < 4; ++u) load4(keys, i + 4 * G * u, nb, c[u]);
#pragma unroll
              for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  if (i + 4 * G * u + j < nb) f(c[u][j]);
            }
          },
          want, sel);
      emit_stream(g, keys, nb, sel[big], out[big], nullptr);
      if (want[small]) emit_stream(g, keys, static_cast<int>(kb), sel[small], out[small], out[big]);
    }
    g.sync();  // the group's shared memory is reused by its next row
  }
}

}  // namespace

cudaError_t launch_publish(const PublishArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return cudaSuccess;
  const int sms = device_sm_count();
  if (a.rows < 2 * sms) return launch_publish_rows(a, stream);
  constexpr int kG = 256, kGroups = kCtaThreads / kG;
  const int smem = static_cast<int>(kGroups * sizeof(GroupShared));
  const int want_grid = (a.rows + kGroups - 1) / kGroups;
  const int grid = want_grid < sms ? want_grid : sms;
  cudaError_t e = cudaFuncSetAttribute(publish_kernel<kG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  publish_kernel<kG><<<grid, kCtaThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ci
