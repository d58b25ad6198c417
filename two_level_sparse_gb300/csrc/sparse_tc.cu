// Level two of the two-level indexer: a layer scores only the positions inside
// each row's candidate blocks and keeps its top-k.
//
// For row t the candidate positions are s = 8 * blocks[t][i] + j (i < nvalid,
// j < 8, s < L_t), scored exactly like the dense pass
//   logit[t, s] = kscale[s] * sum_h w[t, h] * ReLU(q[t, h] . k[s]),
// and the top-k (ties toward the lower position) are written ascending, -1
// padded (sglang PR #40352 "Score prefill consumer index layers on candidate
// blocks with DeepGEMM", Design, "Level two": sparse logits over the published
// blocks read from the paged index-K pool, top-512 of the first valid_len
// columns, page transform to request-relative positions).
//
// One launch scores up to eight layers that share a page table (the source
// with its own top-(P+1) blocks, the consumers with the published ones): the
// work units are (layer, row) pairs, layer-major, so that one layer's pool is
// live in L2 at a time.  One persistent CTA per SM works through its units;
// consecutive units overlap (a unit is called a row below):
//   warp 0      MMA issuer: per row, tcgen05.cp of the row's query scale
//               factors into tensor memory, then per 128-position tile four
//               tcgen05.mma kind::mxf8f6f4 block_scale (M = 128 gathered
//               positions, N = 64 heads, K = 32 each) into one of three
//               accumulator stages -- or, for MXFP4 K, a tcgen05.cp of the
//               tile's K scale factors and two kind::mxf4 steps of K = 64;
//   warps 1-3   gather a tile's 16 candidate blocks (each contiguous K in its
//               page: 1 KB FP8, 512 B MXFP4) into a swizzled MMA tile of a
//               9-deep ring: tiles go round-robin to the three warps, and
//               lanes 0-15 of the tile's warp each issue one tensor-map load
//               of an 8-row box (128- or 64-byte swizzle) in a single
//               instruction, the tile's barrier counting the bytes; for MXFP4
//               the same warp stages the 128 positions' scale words for the
//               MMA warp's tcgen05.cp with 4-byte cp.async;
//   warps 4-7   top-k of the previous row, read back from tensor memory, and
//               around it the prep of the row two ahead in the buffers it
//               frees: the page of every candidate block, the query (widened
//               from e2m1 to e4m3 against FP8 K, packed against MXFP4 K) and
//               its scale factors staged;
//   warps 8-15  two scoring warpgroups, tiles alternating: each thread loads
//               its position's FP8 K scale from the pool (straight when the
//               pool fits in L2, a few tiles ahead through a ring otherwise), then the
//               same epilogue arithmetic as the dense pass and one
//               order-preserving key per candidate stored as one
//               tensor-memory column per tile.
// Scores never leave the chip, and the shared memory they would need goes to
// the gather ring instead.
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kThreads = 512;
constexpr int kStages = 9;       // gathered K tiles in flight
constexpr int kNumAcc = 3;
constexpr int kSfaCol = 192;      // 4 columns of A scale factors (all 1.0)
constexpr int kSfbCol = 196;      // two buffers of 4 columns of B scale factors
constexpr int kScoreCol = 208;    // two buffers of kMaxTiles score columns
constexpr int kSfa4Col = 480;     // MXFP4 K: 4 columns of A scale factors per accumulator stage
constexpr int kBlocksPerTile = kTileM / kBlock;  // 16
constexpr int kMaxBlocks = 2176;                 // >= topk + 1 for every supported topk
constexpr int kMaxTiles = kMaxBlocks / kBlocksPerTile;  // 136
constexpr int kGatherWarp0 = 1, kGatherWarps = 3;  // cp.async gatherers
constexpr int kTopkWarp0 = 4, kTopkThreads = 128, kTopkBar = 2;  // also the next-row prep
constexpr int kPrepThreads = kTopkThreads;
constexpr int kScoreWarp0 = 8;
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;
static_assert(kScoreCol + 2 * kMaxTiles + 32 <= 512, "score columns must fit in tensor memory");

// Top-k working set: radix digits of up to kDigitBits bits.
constexpr int kDigitBits = 11;
struct TopkShared {
  uint32_t hist[1 << kDigitBits];
  uint32_t part[kTopkThreads / 32];
  uint32_t sel_digit, sel_remaining, sel_match;
};

struct __align__(1024) Smem {
  // gathered A tiles (1024-aligned); MXFP4 tiles take the first 8 KB of a slot
  // and stage their scale factors for tcgen05.cp at byte 8192 of it
  uint8_t kv[kStages][kTileM * kDim];
  uint8_t q[2][kHeads * kDim];         // widened queries, double-buffered (1024-aligned: swizzled B tiles)
  uint8_t sf[2][512];                  // query scale factors staged for tcgen05.cp
  // per candidate: (page << 10) | (8-position group in the page << 7) |
  // (first position in the group << 4) | positions below L (1..8), or -1
  int32_t info[2][kMaxBlocks];
  int32_t bid[2][kMaxBlocks];  // the candidate block ids, for the top-k's output positions
  uint4 mgt[kMaxTiles], meq[kMaxTiles];  // top-k compaction ballots, one word per warp
  int gbase[kMaxTiles], ebase[kMaxTiles];  // top-k: entries above / at the threshold before each tile
  int scan_part[2][kTopkThreads / 32];
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t t_full[kNumAcc], t_empty[kNumAcc];
  uint64_t q_full[2], q_empty[2];
  uint64_t info_full[2], info_empty[2];
  uint64_t sc_full[2], sc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int vcount[2];
  int topk_go;
  int prep_ok[4];
  uint32_t kmin, kmax;
  float kring[8][3][32];  // FP8 K scales fetched ahead, per scoring warp: 3 tiles x 32 positions
  TopkShared topk;
};
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory per block");
static_assert(offsetof(Smem, q) % 1024 == 0 && offsetof(Smem, kv) % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(offsetof(Smem, sf) % 16 == 0, "tcgen05.cp needs 16-byte alignment");

__device__ __forceinline__ void set_abort(Smem& sm, int32_t* dev_err) {
  sm.abort_flag = 1;
  report(dev_err, kDevErrTimeout);
}

// The request whose pages row `row` reads (several requests: the last r
// with req_start[r] <= row).
__device__ __forceinline__ int row_request(const SelectArgs& a, int row) {
  if (a.p.layout == kLayoutDecode) return row;
  if (a.p.layout == kLayoutPrefill) return 0;
  int lo = 0, hi = a.p.num_req;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a.p.req_start + mid) <= row)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

struct RowInfo {
  int layer, row, L, nv, nb, ntiles;
};

// kMulti: the launch scores several layers and a unit's per-layer pointers
// come from a dynamically indexed kernel parameter; pinned in a register once
// per unit, they are not re-read from the constant bank at every use inside
// the tile loops.  A one-layer launch (kMulti false) reads layer 0's fields
// as constant-bank operands, as a fixed parameter.
template <bool kMulti, class T>
__device__ __forceinline__ void pin(T*& p) {
  if (kMulti) asm volatile("" : "+l"(p));
}
template <bool kMulti>
__device__ __forceinline__ const SelectLayer& layer_of(const SelectArgs& a, int l) {
  return a.layer[kMulti ? l : 0];
}
// The i-th unit of this CTA.  One layer: round robin.  Several layers (their
// order set by the launcher, the largest candidate lists first): a snake,
// CTA c taking units c, 2G - 1 - c, 2G + c, ... of a grid of G, so that the
// CTAs that took the last of the large units in one pass take the first of
// the next pass's (smaller) ones.  Increasing in i for every CTA.
template <bool kMulti>
__device__ __forceinline__ int unit_of(int i) {
  const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return i * g + (kMulti && (i & 1) ? g - 1 - c : c);
}

// Work unit u: layer u / rows, row u % rows.
template <bool kMulti>
__device__ __forceinline__ RowInfo row_info(const SelectArgs& a, int u, bool report_errors) {
  RowInfo r;
  r.layer = kMulti ? u / a.p.rows : 0;
  r.row = kMulti ? u - r.layer * a.p.rows : u;
  const int row = r.row;
  const SelectLayer& ly = layer_of<kMulti>(a, r.layer);
  r.L = a.p.seq_len[row];
  r.nv = ly.nvalid[row];
  bool bad = false;
  if (r.L < 0 || r.L > a.p.max_len) {
    if (report_errors) report(a.p.dev_err, kDevErrLen);
    bad = true;
  }
  if (r.nv < 0 || r.nv > ly.max_blocks) {
    if (report_errors) report(a.p.dev_err, kDevErrBlock);
    bad = true;
  }
  if (bad) r.L = r.nv = 0;
  r.nb = (r.L + (1 << a.block_shift) - 1) >> a.block_shift;
  r.ntiles = (r.nv + kBlocksPerTile - 1) / kBlocksPerTile;
  return r;
}

// Ring position: slot index and phase parity, advanced one tile at a time.
struct Ring {
  uint32_t idx = 0, phase = 0;
  __device__ __forceinline__ void next(uint32_t n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1;
    }
  }
};

// Prep of a row (by the four top-k warps, two rows ahead, in that row's
// buffers): the query widened from e2m1 to e4m3 into the swizzled B tile, its
// scale factors staged for tcgen05.cp, and for every candidate block its
// physical page, its slot in the page and how many of its positions lie below
// L.  Three steps, so that the global reads overlap the top-k of the row that
// last used the buffers: prep_issue puts the row's reads in flight (query,
// scale words, the first 2048 candidate block ids); prep_query stages the
// query once the MMAs of that row are done and looks up the candidates'
// pages; prep_table writes the candidate table once that row's top-k output
// (which reads the table) is done.
constexpr int kPrepBatch = 16;  // candidate blocks per prep thread per batch
struct PrepRegs {
  uint2 qv[4];  // the query's 4 KB: 32 bytes per thread
  uint32_t sf0, sf1;
  int blk[kPrepBatch], pid[kPrepBatch];
};
static_assert(kHeads * 64 == kPrepThreads * 32, "four query words per prep thread");

template <int KV, bool kMulti>
__device__ __forceinline__ void prep_issue(const SelectArgs& a, const RowInfo& r, int pid_t, PrepRegs& pr) {
  const SelectLayer& ly = layer_of<kMulti>(a, r.layer);
  const uint8_t* q_fp4 = ly.q_fp4 + static_cast<int64_t>(r.row) * kHeads * 64;
  const uint8_t* q_sf = ly.q_sf + static_cast<int64_t>(r.row) * kHeads * 4;
  const int32_t* brow = ly.blocks + static_cast<int64_t>(r.row) * ly.blocks_stride;
  pin<kMulti>(q_fp4);
  pin<kMulti>(q_sf);
  pin<kMulti>(brow);
  if (KV == kKvMxfp4) {
    // thread slots idx = pid_t + 128 j, j < 2: head idx >> 2, 16-byte chunk idx & 3
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = pid_t + kPrepThreads * j;
      const uint2* src = reinterpret_cast<const uint2*>(q_fp4 + (idx >> 2) * 64 + (idx & 3) * 16);
      pr.qv[2 * j] = src[0];
      pr.qv[2 * j + 1] = src[1];
    }
  } else {
    // thread slots idx = pid_t + 128 j, j < 4: head idx >> 3, 8-byte chunk idx & 7
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int idx = pid_t + kPrepThreads * j;
      pr.qv[j] = *reinterpret_cast<const uint2*>(q_fp4 + (idx >> 3) * 64 + (idx & 7) * 8);
    }
  }
  pr.sf0 = pr.sf1 = 0;
  if (pid_t < 32) {
    const uint32_t* sfp = reinterpret_cast<const uint32_t*>(q_sf);
    pr.sf0 = sfp[pid_t];
    pr.sf1 = sfp[32 + pid_t];
  }
#pragma unroll
  for (int j = 0; j < kPrepBatch; ++j) {
    const int i = j * kPrepThreads + pid_t;
    pr.blk[j] = i < r.nv ? brow[i] : -1;
  }
}

// Page of candidate block blk (covering positions blk << shift ..
// + (1 << shift) - 1: 8 positions, or a context shard's 4, 2 or 1, inside one
// 8-position group), or -1 when it has none.
__device__ __forceinline__ int prep_page(const int32_t* pt, const RowInfo& r, int blk, int sh) {
  return (blk >= 0 && blk < r.nb) ? pt[(blk << sh) >> 6] : -1;
}

template <int KV, bool kMulti>
__device__ __forceinline__ bool prep_query(Smem& sm, const SelectArgs& a, const RowInfo& r, int ri, int pid_t,
                                           volatile int* abort_flag, PrepRegs& pr) {
  const int b = ri & 1;
  const uint32_t ph = (ri >> 1) & 1;
  const bool ok = warp_wait(&sm.q_empty[b], ph ^ 1, abort_flag);  // MMAs of row ri - 2 done
  if (ok) {
    if (KV == kKvMxfp4) {
      // packed e2m1 rows of 64 bytes, 64-byte swizzle
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int idx = pid_t + kPrepThreads * j;
        *reinterpret_cast<uint4*>(sm.q[b] + sw64_offset(idx >> 2, (idx & 3) * 16)) =
            make_uint4(pr.qv[2 * j].x, pr.qv[2 * j].y, pr.qv[2 * j + 1].x, pr.qv[2 * j + 1].y);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int idx = pid_t + kPrepThreads * j;
        *reinterpret_cast<uint4*>(sm.q[b] + sw128_offset(idx >> 3, (idx & 7) * 16)) = widen_fp4x16(pr.qv[j]);
      }
    }
    // lane l of the scale-factor columns: heads l and 32 + l, byte j = K block j
    if (pid_t < 32)
      *reinterpret_cast<uint4*>(sm.sf[b] + 16 * pid_t) = make_uint4(pr.sf0, pr.sf1, kUnitScales, kUnitScales);
  }
  fence_proxy_async_smem();
  mbar_arrive(&sm.q_full[b]);
  const int32_t* pt = a.p.page_table + static_cast<int64_t>(row_request(a, r.row)) * a.p.max_pages;
#pragma unroll
  for (int j = 0; j < kPrepBatch; ++j) pr.pid[j] = prep_page(pt, r, pr.blk[j], a.block_shift);
  return ok;
}

template <int KV, bool kMulti>
__device__ __forceinline__ bool prep_table(Smem& sm, const SelectArgs& a, const RowInfo& r, int ri, int pid_t,
                                           volatile int* abort_flag, bool ok, PrepRegs& pr) {
  const int b = ri & 1;
  const uint32_t ph = (ri >> 1) & 1;
  const SelectLayer& ly = layer_of<kMulti>(a, r.layer);
  const int32_t* brow = ly.blocks + static_cast<int64_t>(r.row) * ly.blocks_stride;
  pin<kMulti>(brow);
  const int sh = a.block_shift;
  ok = ok && warp_wait(&sm.info_empty[b], ph ^ 1, abort_flag);  // row ri - 2 gathered and scored
  for (int i0 = 0; ok && i0 < r.nv; i0 += kPrepThreads * kPrepBatch) {
    if (i0 > 0) {  // rows of more than 2048 candidates: the rest in further batches
      const int32_t* pt = a.p.page_table + static_cast<int64_t>(row_request(a, r.row)) * a.p.max_pages;
#pragma unroll
      for (int j = 0; j < kPrepBatch; ++j) {
        const int i = i0 + j * kPrepThreads + pid_t;
        pr.blk[j] = i < r.nv ? brow[i] : -1;
      }
#pragma unroll
      for (int j = 0; j < kPrepBatch; ++j) pr.pid[j] = prep_page(pt, r, pr.blk[j], sh);
    }
#pragma unroll
    for (int j = 0; j < kPrepBatch; ++j) {
      const int i = i0 + j * kPrepThreads + pid_t;
      if (i >= r.nv) continue;
      const int blk = pr.blk[j], pid = pr.pid[j];
      int v = -1;
      if (blk < 0 || (blk >= r.nb && sh == 3))
        report(a.p.dev_err, kDevErrBlock);
      else if (blk >= r.nb)
        ;  // a context shard holds no position of this (global) block: empty
      else if (pid < 0 || pid >= a.p.num_pages)
        report(a.p.dev_err, kDevErrPage);
      else
        v = (pid << 10) | ((((blk << sh) >> 3) & 7) << 7) | (((blk << sh) & 7) << 4) | min(1 << sh, r.L - (blk << sh));
      sm.info[b][i] = v;
      sm.bid[b][i] = blk;
    }
  }
  mbar_arrive(&sm.info_full[b]);
  return ok;
}

// Top-k of one row whose order keys sit in tensor memory: column t of the
// buffer holds tile t, lane p the tile's position p (key 0 = no candidate).
// Run by the 128 threads of warps 4-7, thread kt owning lane kt.
// after_first() is called by every thread once the first pass over the keys
// (their range) is done: other work of the same threads goes there.
template <class EmitPos, class EmitScore, class AfterFirst>
__device__ __forceinline__ void tmem_topk(Smem& sm, uint32_t lane_col0, int nt, int k, int kt, EmitPos emit_pos,
                                          bool want_scores, EmitScore emit_score, AfterFirst after_first) {
  TopkShared& sh = sm.topk;
  const int q = kt >> 5, l = kt & 31;
  uint32_t x[32];
  // live range: the bits below the common prefix of the smallest and largest live key
  if (kt == 0) {
    sm.kmin = 0xFFFFFFFFu;
    sm.kmax = 0;
  }
  named_sync(kTopkBar, kTopkThreads);
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  for (int c0 = 0; c0 < nt; c0 += 32) {
    tmem_ld32(lane_col0 + c0, x);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (c0 + j < nt && x[j] != 0) {
        mn = min(mn, x[j]);
        mx = max(mx, x[j]);
      }
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (l == 0) {
    atomicMin(&sm.kmin, mn);
    atomicMax(&sm.kmax, mx);
  }
  named_sync(kTopkBar, kTopkThreads);
  mn = sm.kmin;
  mx = sm.kmax;
  after_first();
  int hi = mn == mx ? 0 : 32 - __clz(mn ^ mx);  // low bits not shared by every live key
  uint32_t mask = hi == 32 ? 0u : ~((1u << hi) - 1u);
  uint32_t prefix = mn & mask;
  int remaining = k;
  while (hi > 0) {
    const int width = min(kDigitBits, hi), shift = hi - width;
    const uint32_t dmask = (1u << width) - 1u;
    const int nbins = 1 << width;
    for (int i = kt; i < nbins; i += kTopkThreads) sh.hist[i] = 0;
    named_sync(kTopkBar, kTopkThreads);
    for (int c0 = 0; c0 < nt; c0 += 32) {
      tmem_ld32(lane_col0 + c0, x);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < nt && (x[j] & mask) == prefix) atomicAdd(&sh.hist[(x[j] >> shift) & dmask], 1u);
    }
    named_sync(kTopkBar, kTopkThreads);
    // the threshold digit: thread kt owns bins [16 kt, 16 kt + 16)
    constexpr int kPer = (1 << kDigitBits) / kTopkThreads;
    uint32_t c[kPer], lsum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int bin = kt * kPer + j;
      c[j] = bin < nbins ? sh.hist[bin] : 0u;
      lsum += c[j];
    }
    uint32_t suffix = lsum;  // over lanes >= l
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_down_sync(0xffffffffu, suffix, o);
      if (l + o < 32) suffix += v;
    }
    if (l == 0) sh.part[q] = suffix;
    named_sync(kTopkBar, kTopkThreads);
    uint32_t above = suffix - lsum;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w)
      if (w > q) above += sh.part[w];
    const uint32_t want = static_cast<uint32_t>(remaining);
    if (above < want && want <= above + lsum) {
      uint32_t acc = above;
#pragma unroll
      for (int j = kPer - 1; j >= 0; --j) {
        if (acc + c[j] >= want) {
          sh.sel_digit = kt * kPer + j;
          sh.sel_remaining = want - acc;
          sh.sel_match = c[j];
          break;
        }
        acc += c[j];
      }
    }
    named_sync(kTopkBar, kTopkThreads);
    const uint32_t d = sh.sel_digit, match = sh.sel_match;
    remaining = static_cast<int>(sh.sel_remaining);
    prefix |= d << shift;
    mask |= dmask << shift;
    hi = shift;
    if (match == static_cast<uint32_t>(remaining)) break;
  }
  const uint32_t need_eq = static_cast<uint32_t>(remaining);
  // ordered compaction: ballots per (tile, warp), then ranks in index order
  for (int c0 = 0; c0 < nt; c0 += 32) {
    tmem_ld32(lane_col0 + c0, x);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (c0 + j >= nt) break;
      const uint32_t m = x[j] & mask;
      const uint32_t bg = __ballot_sync(0xffffffffu, m > prefix);
      const uint32_t be = __ballot_sync(0xffffffffu, m == prefix);
      if (l == 0) {
        reinterpret_cast<uint32_t*>(&sm.mgt[c0 + j])[q] = bg;
        reinterpret_cast<uint32_t*>(&sm.meq[c0 + j])[q] = be;
      }
    }
  }
  named_sync(kTopkBar, kTopkThreads);
  // Entries above / at the threshold in the tiles before each tile: thread kt
  // counts tiles kt and kt + 128, then a block-wide exclusive scan.
  {
    int g0 = 0, e0 = 0, g1 = 0, e1 = 0;
    if (kt < nt) {
      const uint4 g4 = sm.mgt[kt], e4 = sm.meq[kt];
      g0 = __popc(g4.x) + __popc(g4.y) + __popc(g4.z) + __popc(g4.w);
      e0 = __popc(e4.x) + __popc(e4.y) + __popc(e4.z) + __popc(e4.w);
    }
    if (kt + kTopkThreads < nt) {
      const uint4 g4 = sm.mgt[kt + kTopkThreads], e4 = sm.meq[kt + kTopkThreads];
      g1 = __popc(g4.x) + __popc(g4.y) + __popc(g4.z) + __popc(g4.w);
      e1 = __popc(e4.x) + __popc(e4.y) + __popc(e4.z) + __popc(e4.w);
    }
    // first 128 tiles, then the rest, each scanned across the block
    int gi = g0, ei = e0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int gv = __shfl_up_sync(0xffffffffu, gi, o), ev = __shfl_up_sync(0xffffffffu, ei, o);
      if (l >= o) {
        gi += gv;
        ei += ev;
      }
    }
    if (l == 31) {
      sm.scan_part[0][q] = gi;
      sm.scan_part[1][q] = ei;
    }
    int gj = g1, ej = e1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int gv = __shfl_up_sync(0xffffffffu, gj, o), ev = __shfl_up_sync(0xffffffffu, ej, o);
      if (l >= o) {
        gj += gv;
        ej += ev;
      }
    }
    named_sync(kTopkBar, kTopkThreads);
    int gw_before = 0, ew_before = 0, gtot = 0, etot = 0;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
      const int gs = sm.scan_part[0][w], es = sm.scan_part[1][w];
      if (w < q) {
        gw_before += gs;
        ew_before += es;
      }
      gtot += gs;
      etot += es;
    }
    named_sync(kTopkBar, kTopkThreads);
    if (l == 31) {
      sm.scan_part[0][q] = gj;
      sm.scan_part[1][q] = ej;
    }
    named_sync(kTopkBar, kTopkThreads);
    int gw2 = 0, ew2 = 0;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w)
      if (w < q) {
        gw2 += sm.scan_part[0][w];
        ew2 += sm.scan_part[1][w];
      }
    if (kt < nt) {
      sm.gbase[kt] = gw_before + gi - g0;
      sm.ebase[kt] = ew_before + ei - e0;
    }
    if (kt + kTopkThreads < nt) {
      sm.gbase[kt + kTopkThreads] = gtot + gw2 + gj - g1;
      sm.ebase[kt + kTopkThreads] = etot + ew2 + ej - e1;
    }
  }
  named_sync(kTopkBar, kTopkThreads);
  // Positions, word-parallel: thread kt walks the selected entries of ballot
  // words kt, kt + 128, ... (word w of tile t: positions 32 w .. 32 w + 31) in
  // position order.  Rank = entries above the threshold before it + entries
  // at it before it (capped at need_eq), in (tile, position) order.
  for (int it = kt; it < 4 * nt; it += kTopkThreads) {
    const int t = it >> 2, w = it & 3;
    const uint4 g4 = sm.mgt[t], e4 = sm.meq[t];
    uint32_t gtb = static_cast<uint32_t>(sm.gbase[t]), eqb = static_cast<uint32_t>(sm.ebase[t]);
    if (w > 0) {
      gtb += __popc(g4.x);
      eqb += __popc(e4.x);
    }
    if (w > 1) {
      gtb += __popc(g4.y);
      eqb += __popc(e4.y);
    }
    if (w > 2) {
      gtb += __popc(g4.z);
      eqb += __popc(e4.z);
    }
    const uint32_t gw = w == 0 ? g4.x : w == 1 ? g4.y : w == 2 ? g4.z : g4.w;
    const uint32_t ew = w == 0 ? e4.x : w == 1 ? e4.y : w == 2 ? e4.z : e4.w;
    uint32_t bits = gw | ew;
    while (bits) {
      const int lb = __ffs(bits) - 1;
      bits &= bits - 1;
      const uint32_t below = (1u << lb) - 1u;
      const uint32_t gt_before = gtb + __popc(gw & below), eq_before = eqb + __popc(ew & below);
      if (((gw >> lb) & 1u) || eq_before < need_eq) emit_pos(static_cast<int>(gt_before + min(eq_before, need_eq)), t, 32 * w + lb);
    }
  }
  if (!want_scores) return;
  // Scores, lane-parallel (only this lane can read its keys): the same ranks.
  const uint32_t lt = lanemask_lt();
  for (int c0 = 0; c0 < nt; c0 += 32) {
    tmem_ld32(lane_col0 + c0, x);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int t = c0 + j;
      if (t >= nt) break;
      const uint32_t m = x[j] & mask;
      const bool is_gt = m > prefix, is_eq = m == prefix;
      if (!(is_gt || is_eq)) continue;
      const uint4 g4 = sm.mgt[t], e4 = sm.meq[t];
      const uint32_t g[4] = {g4.x, g4.y, g4.z, g4.w}, e[4] = {e4.x, e4.y, e4.z, e4.w};
      uint32_t gtb = static_cast<uint32_t>(sm.gbase[t]) + __popc(g[q] & lt);
      uint32_t eqb = static_cast<uint32_t>(sm.ebase[t]) + __popc(e[q] & lt);
#pragma unroll
      for (int w = 0; w < 4; ++w)
        if (w < q) {
          gtb += __popc(g[w]);
          eqb += __popc(e[w]);
        }
      if (is_gt || eqb < need_eq) emit_score(static_cast<int>(gtb + min(eqb, need_eq)), x[j]);
    }
  }
}

// The layers' tensor maps over their pools (8-row boxes, one candidate block).
struct SelectMaps {
  CUtensorMap m[kMaxSelectLayers];
};
// A tensor-map load issued by every active lane (each lane its own box).
__device__ __forceinline__ void tma_load_3d_lane(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                 uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// kRing: FP8 K scales fetched tiles ahead (pools too large to stay in L2).
template <int KV, bool kMulti, bool kRing>
__global__ void __launch_bounds__(kThreads, 1)
    select_kernel(const __grid_constant__ SelectMaps maps, const SelectArgs a) {
  constexpr bool kFp4 = KV == kKvMxfp4;
  constexpr bool kAbsAdd = scorer_relu_abs_add<KV>();  // ReLU form: identical to the dense scorer's
  constexpr int kBlockBytes = kBlock * row_bytes<KV>();  // one candidate block's values: 1 KB or 512 B
  constexpr int kPVB = page_value_bytes<KV>(), kPB = page_bytes<KV>();
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      // the tile's tensor-map loads (one expect_tx arrival), and for MXFP4
      // every lane of the issuing warp once its scale-word copies landed
      mbar_init(&sm.k_full[s], kFp4 ? 1 + 32 : 1);
      mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < kNumAcc; ++s) {
      mbar_init(&sm.t_full[s], 1);
      mbar_init(&sm.t_empty[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_full[b], kPrepThreads);
      mbar_init(&sm.q_empty[b], 1);
      mbar_init(&sm.info_full[b], kPrepThreads);
      mbar_init(&sm.info_empty[b], 32 * kGatherWarps + 8);  // gather lanes + scoring warps
      mbar_init(&sm.sc_full[b], 8);
      mbar_init(&sm.sc_empty[b], 1);
      sm.vcount[b] = 0;
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  if (warp >= kTopkWarp0 && warp < kTopkWarp0 + 4) {
    // A scale factors: all ones, in every lane quadrant
    tmem_st4(tmem_addr(tbase, 32 * (warp & 3), kSfaCol), kUnitScales, kUnitScales, kUnitScales, kUnitScales);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int rows = a.num_layers * a.p.rows;  // work units
  if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer (whole warp, one lane issues)
    Ring kr, ar;
    int ri = 0;
    bool ok = true;
    for (int u = unit_of<kMulti>(ri); u < rows && ok; u = unit_of<kMulti>(++ri)) {
      const RowInfo r = row_info<kMulti>(a, u, lane == 0);
      const int b = ri & 1;
      if (!warp_wait_fast(&sm.q_full[b], (ri >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sfb = tbase + kSfbCol + 4 * b;
      tmem_cp_32x128b_x4_elect(sfb, sdesc_rows16(smem_u32(sm.sf[b])));
      uint64_t bdesc[4];
      uint32_t idesc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bdesc[k] = kFp4 ? sdesc_k64_sw64(smem_u32(sm.q[b]) + 32 * (k & 1)) : sdesc_k128_sw128(smem_u32(sm.q[b]) + 32 * k);
        idesc[k] = kFp4 ? idesc_mxf4(kTileM, kHeads, 2 * (k & 1), 2 * (k & 1)) : idesc_mxf8f6f4_e4m3(kTileM, kHeads, k, k);
      }
      // One tile: its MMAs into accumulator stage acc, then the commits that
      // free the K slot and hand the stage to the scoring warps.
      auto issue = [&](const Ring& k, const Ring& acc) {
        const uint32_t d = tbase + acc.idx * kHeads;
        const uint32_t a0 = smem_u32(sm.kv[k.idx]);
        const uint32_t ke = smem_u32(&sm.k_empty[k.idx]), tf = smem_u32(&sm.t_full[acc.idx]);
        if (kFp4)
          // the tile's A scale factors (staged transposed by the gather warp),
          // one slot per accumulator stage: the MMAs that read a slot finished
          // before t_empty let this stage be reused
          mma_tile_mxf4_commit2_elect(d, sdesc_k64_sw64(a0), bdesc, idesc, sdesc_rows16(a0 + 8192),
                                      tbase + kSfa4Col + 4 * acc.idx, sfb, ke, tf);
        else
          mma_tile_mxf8f6f4_commit2_elect(d, sdesc_k128_sw128(a0), bdesc, idesc, tbase + kSfaCol, sfb, ke, tf);
      };
      // Two tiles per pass where the row has them: lane 0 probes all their
      // barriers before acting on any probe, so the probes' latencies overlap
      // (this warp's loop sets the pace of the whole pipeline); the first
      // tile goes as soon as its own two have passed, and bounded waits run
      // only where a probe found a phase incomplete.
      auto go = [&](bool probed, const Ring& k, const Ring& acc) -> bool {
        bool ready = true;
        if (lane == 0 && !probed)
          ready = mbar_wait(&sm.k_full[k.idx], k.phase, abort_flag) &&
                  mbar_wait(&sm.t_empty[acc.idx], acc.phase ^ 1, abort_flag);
        ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
        __syncwarp();
        if (!ready) return false;
        if (kFp4) fence_proxy_async_smem();  // MXFP4 scale words are written through the generic proxy (cp.async)
        tc_fence_after();
        issue(k, acc);
        return true;
      };
      for (int t = 0; t < r.ntiles; t += 2) {
        const bool two = t + 1 < r.ntiles;
        Ring k2 = kr, a2 = ar;
        k2.next(kStages);
        a2.next(kNumAcc);
        bool pa = true, pb = true;  // lane 0: both barriers of tile a / b seen complete
        if (lane == 0) {
          const bool p0 = mbar_try_wait(&sm.k_full[kr.idx], kr.phase);
          const bool p1 = mbar_try_wait(&sm.t_empty[ar.idx], ar.phase ^ 1);
          bool p2 = true, p3 = true;
          if (two) {
            p2 = mbar_try_wait(&sm.k_full[k2.idx], k2.phase);
            p3 = mbar_try_wait(&sm.t_empty[a2.idx], a2.phase ^ 1);
          }
          pa = p0 && p1;
          pb = p2 && p3;
        }
        if (!go(pa, kr, ar) || (two && !go(pb, k2, a2))) {
          ok = false;
          break;
        }
        kr = k2;
        ar = a2;
        if (two) {
          kr.next(kStages);
          ar.next(kNumAcc);
        }
      }
      if (ok) mma_commit_elect(&sm.q_empty[b]);  // the query buffer is free once these MMAs complete
    }
    if (!ok && lane == 0) set_abort(sm, a.p.dev_err);
  } else if (warp >= kGatherWarp0 && warp < kGatherWarp0 + kGatherWarps) {
    // ------------------------------------------------------------------ gather
    // Random 1 KB blocks from L2 or HBM: copies issued by many lanes at once
    // reach several times the rate of one lane issuing them in turn, and one
    // tensor-map load per block (a lane each) costs a single instruction per
    // tile where 16-byte cp.async from every lane costs two per block plus an
    // arrival per lane.  Block blk is contiguous in its page and lands on its
    // own 8-row swizzle atom.
    const int gw = warp - kGatherWarp0;
    Ring kr;  // slot of the next tile to issue
    int ri = 0;
    bool ok = true;
    uint32_t nt = 0;           // tiles so far (all warps): FP8 tile n is issued by warp n % 3
    uint32_t last_issued = 0;  // FP8: 1 + sequence number of this warp's last issued tile
    if (lane < a.num_layers) prefetch_tmap(&maps.m[lane]);
    for (int u = unit_of<kMulti>(ri); u < rows && ok; u = unit_of<kMulti>(++ri)) {
      const RowInfo r = row_info<kMulti>(a, u, false);
      const int b = ri & 1;
      const uint8_t* k_pool = layer_of<kMulti>(a, r.layer).k_pool;
      pin<kMulti>(k_pool);
      const CUtensorMap* tmap = &maps.m[kMulti ? r.layer : 0];
      ok = warp_wait_lane0(&sm.info_full[b], (ri >> 1) & 1, abort_flag);
      const int32_t* info = sm.info[b];
      for (int t = 0; t < r.ntiles && ok; ++t, ++nt) {
        // the tile's 16 blocks: one 8-row box each (landing swizzled on its
        // own atom), issued by lanes 0-15 at once
        if (nt % kGatherWarps == static_cast<uint32_t>(gw)) {
          if (!warp_wait_lane0(&sm.k_empty[kr.idx], kr.phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* dst = sm.kv[kr.idx];
          const int row_base = t * kBlocksPerTile;
          const int v = lane < kBlocksPerTile && row_base + lane < r.nv ? info[row_base + lane] : -1;
          const uint32_t live = __ballot_sync(0xffffffffu, v >= 0);
          if (lane == 0) mbar_arrive_expect_tx(&sm.k_full[kr.idx], __popc(live) * kBlockBytes);
          __syncwarp();
          if (v >= 0)
            tma_load_3d_lane(dst + lane * kBlockBytes, tmap, 0, ((v >> 7) & 7) * kBlock, v >> 10, &sm.k_full[kr.idx]);
          if (kFp4) {
            // the scale words of all 128 positions, staged for tcgen05.cp:
            // position p = 32 c + l goes to byte 16 l + 4 c; every lane
            // arrives once its four copies have landed
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int p = 32 * c + lane;
              const int vb = __shfl_sync(0xffffffffu, v, p >> 3);
              if (vb >= 0)
                cp_async4(dst + 8192 + 16 * lane + 4 * c,
                          k_pool + static_cast<int64_t>(vb >> 10) * kPB + kPVB + 4 * (((vb >> 7) & 7) * kBlock + (p & 7)));
            }
            cp_async_arrive_noinc(&sm.k_full[kr.idx]);
          }
          last_issued = nt + 1;
        }
        kr.next(kStages);
      }
      __syncwarp();
      if (ok) mbar_arrive(&sm.info_empty[b]);
    }
    cp_async_wait<0>();
    if (!ok && lane == 0) {
      // no tensor-map load of this warp may still be writing when the CTA exits
      for (uint32_t i = last_issued > kStages ? last_issued - kStages : 0; i < last_issued; ++i)
        if (i % kGatherWarps == static_cast<uint32_t>(gw))
          mbar_wait(&sm.k_full[i % kStages], (i / kStages) & 1, nullptr, 1000000000ull);
    }
    if (!ok && lane == 0) set_abort(sm, a.p.dev_err);
  } else if (warp >= kTopkWarp0 && warp < kTopkWarp0 + 4) {
    // ------------------------------------------------------------------ top-k of finished rows + next-row prep
    const int kt = tid - kTopkWarp0 * 32;
    const uint32_t lane_base = tmem_addr(tbase, 32 * (warp & 3), 0);
    // the prep verdict (mine: this thread's steps succeeded) made uniform across
    // the four warps before anyone acts on it
    auto all_ok = [&](bool mine) -> bool {
      if (lane == 0) sm.prep_ok[warp & 3] = mine ? 1 : 0;
      named_sync(kTopkBar, kTopkThreads);
      const bool all = sm.prep_ok[0] && sm.prep_ok[1] && sm.prep_ok[2] && sm.prep_ok[3];
      named_sync(kTopkBar, kTopkThreads);
      return all;
    };
    // the prep of row index pi (the pi-th row of this CTA), all steps at once
    auto prep = [&](int pi) -> bool {
      const int pu = unit_of<kMulti>(pi);
      bool mine = true;
      if (pu < rows) {
        const RowInfo rp = row_info<kMulti>(a, pu, false);
        PrepRegs pr;
        prep_issue<KV, kMulti>(a, rp, kt, pr);
        mine = prep_query<KV, kMulti>(sm, a, rp, pi, kt, abort_flag, pr);
        mine = prep_table<KV, kMulti>(sm, a, rp, pi, kt, abort_flag, mine, pr);
      }
      return all_ok(mine);
    };
    bool ok = prep(0) && prep(1);
    int ri = 0;
    for (int u = unit_of<kMulti>(ri); u < rows && ok; u = unit_of<kMulti>(++ri)) {
      const RowInfo r = row_info<kMulti>(a, u, false);
      const SelectLayer& ly = layer_of<kMulti>(a, r.layer);
      const int b = ri & 1;
      // row ri + 2 is prepared in this row's buffers around its top-k: reads
      // issued now, the query staged after the top-k's first pass, the table
      // written after the top-k's output
      const int u2 = unit_of<kMulti>(ri + 2);
      const bool has2 = u2 < rows;
      RowInfo r2 = {};
      PrepRegs pr;
      if (has2) {
        r2 = row_info<kMulti>(a, u2, false);
        prep_issue<KV, kMulti>(a, r2, kt, pr);
      }
      bool mine = true;
      auto stage_query = [&]() {
        if (has2) mine = prep_query<KV, kMulti>(sm, a, r2, ri + 2, kt, abort_flag, pr);
      };
      if (kt == 0) sm.topk_go = mbar_wait(&sm.sc_full[b], (ri >> 1) & 1, abort_flag) ? 1 : 0;
      named_sync(kTopkBar, kTopkThreads);
      if (!sm.topk_go) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int k = min(a.topk, sm.vcount[b]);
      int32_t* out = ly.out_pos + static_cast<int64_t>(r.row) * a.out_stride;
      float* osc = ly.out_score != nullptr ? ly.out_score + static_cast<int64_t>(r.row) * a.out_stride : nullptr;
      pin<kMulti>(out);
      pin<kMulti>(osc);
      if (k > 0) {
        tmem_topk(
            sm, lane_base + kScoreCol + b * kMaxTiles, r.ntiles, k, kt,
            [&](int rank, int t, int p) {
              const int i = t * kBlocksPerTile + (p >> 3);
              out[rank] = (sm.bid[b][i] << a.block_shift) + (p & 7) - ((sm.info[b][i] >> 4) & 7);
            },
            osc != nullptr, [&](int rank, uint32_t u) { osc[rank] = order_key_inv(u); }, stage_query);
      } else {
        stage_query();
      }
      for (int i = max(k, 0) + kt; i < a.topk; i += kTopkThreads) {
        out[i] = -1;
        if (osc) osc[i] = -__int_as_float(0x7f800000);
      }
      tc_fence_before();
      named_sync(kTopkBar, kTopkThreads);
      if (kt == 0) {
        sm.vcount[b] = 0;
        mbar_arrive(&sm.sc_empty[b]);
      }
      if (has2) mine = prep_table<KV, kMulti>(sm, a, r2, ri + 2, kt, abort_flag, mine, pr);
      ok = all_ok(mine);
    }
    if (!ok && kt == 0) set_abort(sm, a.p.dev_err);
  } else if (warp >= kScoreWarp0) {
    // ------------------------------------------------------------------ scoring epilogue
    const int e = (warp - kScoreWarp0) >> 2;  // scoring warpgroup 0 / 1
    const int quad = warp & 3;
    const int p = 32 * quad + lane;
    uint32_t tseq = 0;
    int ri = 0;
    unsigned long long w2[32];  // head weights, packed pairs
    bool ok = true;
    for (int u = unit_of<kMulti>(ri); u < rows && ok; u = unit_of<kMulti>(++ri)) {
      const RowInfo r = row_info<kMulti>(a, u, false);
      const int b = ri & 1;
      const uint8_t* k_pool = layer_of<kMulti>(a, r.layer).k_pool;
      pin<kMulti>(k_pool);
      load_head_weights(w2, layer_of<kMulti>(a, r.layer).w + static_cast<int64_t>(r.row) * kHeads);
      // the candidate page lookups (prepared with the row) tell which positions are live
      if (!warp_wait(&sm.info_full[b], (ri >> 1) & 1, abort_flag) ||
          (ri >= 2 && !warp_wait(&sm.sc_empty[b], ((ri >> 1) & 1) ^ 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t score_col = tmem_addr(tbase, 32 * quad, kScoreCol + b * kMaxTiles);
      uint32_t nvalid_seen = 0;
      // FP8 K scales.  From a pool in L2: each lane loads its position's
      // scale as the tile starts.  From a pool in HBM (kRing): this warp's
      // tiles alternate with the other warpgroup's, and each lane copies its
      // position's scale two of the warp's tiles ahead (cp.async, one group
      // per tile) into a 3-slot ring of its own, so that the load has four
      // tiles of time to land.  (MXFP4: the scales are inside the MMA.)
      constexpr bool ks_ring = !kFp4 && kRing;
      float* kring = &sm.kring[warp - kScoreWarp0][0][0];
      auto ks_issue = [&](int tt, int slot) {
        if (!ks_ring) return;
        const int s2 = tt * kBlocksPerTile + (p >> 3);
        const int v = tt < r.ntiles && s2 < r.nv ? sm.info[b][s2] : -1;
        const int off = (v >> 4) & 7;
        if (v >= 0 && (p & 7) >= off && (p & 7) < off + (v & 15))
          cp_async4(kring + 32 * slot + lane,
                    k_pool + static_cast<int64_t>(v >> 10) * kPB + kPVB + 4 * (((v >> 7) & 7) * kBlock + (p & 7)));
        cp_async_commit();
      };
      const int t_first = static_cast<int>((static_cast<uint32_t>(e) - tseq) & 1u);  // this warp's first tile
      int own = 0;  // this warp's tiles of the row so far
      ks_issue(t_first, 0);
      ks_issue(t_first + 2, 1);
      // this warp's tiles of the row: every other one, from t_first; their
      // accumulator stages follow the tile sequence (stage q % 3, phase q / 3)
      const uint32_t q0 = tseq + static_cast<uint32_t>(t_first);
      uint32_t aidx = q0 % kNumAcc, aph = (q0 / kNumAcc) & 1u;
      for (int t = t_first; t < r.ntiles; t += 2) {
        {
          const int slot = t * kBlocksPerTile + (p >> 3);
          const int v = slot < r.nv ? sm.info[b][slot] : -1;
          const int off = (v >> 4) & 7;
          const bool valid = v >= 0 && (p & 7) >= off && (p & 7) < off + (v & 15);
          ks_issue(t + 4, (own + 2) % 3);
          float kscale = 1.0f;
          if (ks_ring) {
            cp_async_wait<2>();  // this tile's group (the two newest may still be in flight)
            if (valid) kscale = kring[32 * (own % 3) + lane];
          } else if (!kFp4 && valid) {
            kscale = __ldg(reinterpret_cast<const float*>(k_pool + static_cast<int64_t>(v >> 10) * kPB + kPVB) +
                           ((v >> 7) & 7) * kBlock + (p & 7));
          }
          ++own;
          if (!warp_wait_fast(&sm.t_full[aidx], aph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          HeadAcc acc = {{0, 0, 0, 0}};
          uint32_t x[32];
          const uint32_t taddr = tmem_addr(tbase, 32 * quad, aidx * kHeads);
          tmem_ld32(taddr, x);
          tmem_ld_wait();
          head_reduce_half<kAbsAdd>(acc, x, w2);
          tmem_ld32(taddr + 32, x);
          tmem_ld_wait();
          head_reduce_half<kAbsAdd>(acc, x, w2 + 16);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.t_empty[aidx]);
          const float score = head_reduce_finish<kAbsAdd>(acc);
          tmem_st1(score_col + t, valid ? order_key(score * kscale) : 0u);
          nvalid_seen += __popc(__ballot_sync(0xffffffffu, valid));
        }
        static_assert(kNumAcc >= 2, "the stage steps by two with one wrap at most");
        aidx += 2;
        if (aidx >= kNumAcc) {
          aidx -= kNumAcc;
          aph ^= 1u;
        }
      }
      tseq += static_cast<uint32_t>(r.ntiles);
      if (!ok) break;
      tmem_st_wait();
      tc_fence_before();
      if (lane == 0 && nvalid_seen) atomicAdd(&sm.vcount[b], static_cast<int>(nvalid_seen));
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.sc_full[b]);
        mbar_arrive(&sm.info_empty[b]);  // done reading this row's candidate lookups
      }
    }
    if (!ok && lane == 0) set_abort(sm, a.p.dev_err);
  }

  // ------------------------------------------------------------------ tear-down
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, nullptr, 1000000000ull);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

}  // namespace

size_t select_smem_bytes(int) { return sizeof(Smem) + 1024; }

template <int KV, bool kMulti, bool kRing>
cudaError_t launch_select_kv(const SelectArgs& a, cudaStream_t stream) {
  const int smem = static_cast<int>(select_smem_bytes(0));
  cudaError_t e = cudaFuncSetAttribute(select_kernel<KV, kMulti, kRing>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t units = static_cast<int64_t>(a.num_layers) * a.p.rows;
  const int grid = units < device_sm_count() ? static_cast<int>(units) : device_sm_count();
  SelectMaps maps;
  for (int l = 0; l < a.num_layers; ++l) {
    e = make_pool_tmap(&maps.m[l], a.layer[l].k_pool, a.p.num_pages, KV, kBlock);
    if (e != cudaSuccess) return e;
  }
  select_kernel<KV, kMulti, kRing><<<grid, kThreads, smem, stream>>>(maps, a);
  return cudaGetLastError();
}

// FP8 pools: scales fetched ahead when a layer's pool (the layers run one
// after another) cannot stay in L2.
template <bool kMulti>
cudaError_t launch_select_fmt(const SelectArgs& a, cudaStream_t stream) {
  if (a.p.kv_format == kKvMxfp4) return launch_select_kv<kKvMxfp4, kMulti, false>(a, stream);
  const bool ring = a.p.num_pages * static_cast<int64_t>(page_bytes<kKvFp8>()) > device_l2_bytes() / 2;
  return ring ? launch_select_kv<kKvFp8, kMulti, true>(a, stream) : launch_select_kv<kKvFp8, kMulti, false>(a, stream);
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream) {
  if (a.p.rows == 0 || a.num_layers == 0) return cudaSuccess;
  if (a.num_layers > 1) {
    // layers with the most candidate blocks first (stable), for the snake order
    SelectArgs s = a;
    for (int i = 1; i < s.num_layers; ++i)
      for (int j = i; j > 0 && s.layer[j].max_blocks > s.layer[j - 1].max_blocks; --j) {
        const SelectLayer t = s.layer[j];
        s.layer[j] = s.layer[j - 1];
        s.layer[j - 1] = t;
      }
    return launch_select_fmt<true>(s, stream);
  }
  return launch_select_fmt<false>(a, stream);
}

}  // namespace ci
