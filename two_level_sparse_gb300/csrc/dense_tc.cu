// Level one of the two-level indexer: dense MQA indexer scores of the source
// layer, reduced on chip to one key per block of 8 positions.
//
//   logit[t, s] = kscale[s] * sum_h w[t, h] * ReLU(q[t, h] . k[s]),  s < L_t
//   key[t, b]   = max_{s in block b} logit[t, s];  key[t, nb_t - 1] = +inf
//
// (sglang PR #40352 "Score prefill consumer index layers on candidate blocks
// with DeepGEMM", Motivation/Design and the block_amax.cuh contract in its
// review; vLLM sparse_attn_indexer.py, fp8_fp4_mqa_logits and the paged
// variant.)  The [rows, L] score matrix is never written.
//
// Design (one persistent CTA per SM, 16 warps):
//   warps 0, 2  TMA producers (warp 0 the even tiles of the sequence, warp 2
//               the odd ones, so that the producer work sits on two
//               sub-partitions beside the epilogue warps, not one): two
//               64-position pages of FP8 K per
//               128-position tile (one tensor-map load each, 128-byte
//               swizzle) into an 8-stage ring, their fp32 scales (bulk
//               copies) into a separate 16-slot ring, both completing on
//               the K stage's barrier;
//   warp 1      MMA issuer: tcgen05.mma kind::mxf8f6f4 block_scale, M = 128
//               positions, N = 64 R columns (R rows x 64 heads), K = 128 in
//               four K = 32 steps; A = K tile (scale 1), B = the rows' queries
//               widened from e2m1 to e4m3 (exact) with their ue8m0 scales in
//               tensor memory; fp32 accumulators in tensor memory;
//   warp 3      set-up only;
//   warps 4-15  epilogue, three warpgroups: tcgen05.ld of one row's 64 head
//               columns per position, ReLU + head weights, K scale, length
//               mask, max over 8 lanes by shuffles, key store.
// MXFP4 index-K (the use_fp4_cache variant of vLLM sparse_attn_indexer.py):
// 64-byte packed rows with 64-byte swizzle, the query kept packed, two
// kind::mxf4 steps of K = 64 per tile; the MMA warp transposes each tile's
// 128 scale words into shared memory and copies them into tensor memory as
// the A scale factors (row 32 c + l at column c, lane l); no per-position K
// scale in the epilogue.
// Prefill rows share one request's pages, so R = 3 rows ride one MMA
// (N = 192, two accumulator stages); decode rows each have their own pages,
// R = 1 (N = 64, four stages) and the three epilogue warpgroups take tiles
// round-robin.  Work is the list of (row group, 128-position tile) pairs,
// split evenly across the CTAs.
#include <type_traits>

#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kThreads = 512;
constexpr int kStages = 8;       // K ring (power of two: slot and phase come from the tile counter)
constexpr int kScaleSlots = 16;  // scale ring (power of two)
constexpr int kEpiWarp0 = 4;
constexpr int kTmemCols = 512;
constexpr int kSfaCol = 384;  // 4 columns: A scale factors (all 1.0)
constexpr int kSfbCol = 388;  // 8 columns: B scale factors
constexpr int kSfa4Col = 400;  // MXFP4 K: 4 columns of A scale factors per K stage (32 columns)
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;

struct __align__(1024) Smem {
  // A tiles, 1024-aligned.  MXFP4 tiles take the first 8 KB of a slot and
  // stage their scale factors for tcgen05.cp at byte 8192 of it.
  uint8_t kv[kStages][kTileM * kDim];
  uint8_t q[3 * kHeads * kDim];        // B tile (up to 192 rows of 128 B)
  float ks[kScaleSlots][kTileM];       // per-position K scales
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t s_empty[kScaleSlots];  // scale slot read by every epilogue warp (one-row groups only)
  uint64_t t_full[4], t_empty[4];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int g_begin, o_begin;
  long long t_begin, t_end;
  long long warp_sum[kThreads / 32];
  int32_t gpre[kMaxReq + 1];  // several requests: groups of requests < r
};

// Length that row `row` is scored over: L if it has more than skip_le_blocks
// blocks, 0 if skipped, -1 if its length breaks the contract.
__device__ __forceinline__ int scored_len(const DenseArgs& a, int row) {
  const int L = a.p.seq_len[row];
  if (L < 0 || L > a.p.max_len) return -1;
  return ((L + kBlock - 1) / kBlock) > a.skip_le_blocks ? L : 0;
}

// Group g: up to R consecutive rows of one request, sharing its pages.
struct RowGroup {
  int req, first, count;
};
template <int R>
__device__ __forceinline__ RowGroup row_group(const DenseArgs& a, const int32_t* gpre, int g) {
  if (a.p.layout == kLayoutVarlen) {
    int lo = 0, hi = a.p.num_req;  // the request r with gpre[r] <= g < gpre[r + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (gpre[mid] <= g)
        lo = mid;
      else
        hi = mid;
    }
    const int first = __ldg(a.p.req_start + lo) + R * (g - gpre[lo]);
    return {lo, first, min(R, __ldg(a.p.req_start + lo + 1) - first)};
  }
  const int first = g * R;
  return {a.p.layout == kLayoutPrefill ? 0 : g, first, min(R, a.p.rows - first)};
}

template <int R>
__device__ __forceinline__ int group_len(const DenseArgs& a, const RowGroup& grp) {
  int m = 0;
#pragma unroll
  for (int i = 0; i < R; ++i)
    if (i < grp.count) m = max(m, scored_len(a, grp.first + i));
  return m;
}

__device__ __forceinline__ void set_abort(Smem& sm, int32_t* dev_err) {
  sm.abort_flag = 1;
  report(dev_err, kDevErrTimeout);
}

template <int R, int KV, bool kLocal>
__global__ void __launch_bounds__(kThreads, 1)
    dense_amax8_kernel(const __grid_constant__ CUtensorMap tmap, const DenseArgs a) {
  constexpr int N = 64 * R;                    // MMA N
  constexpr int kNumAcc = R == 3 ? 2 : 4;      // accumulator stages (power of two)
  constexpr int kEpiPerTile = R == 3 ? 3 : 1;  // epilogue warpgroups consuming each tile
  constexpr bool kFp4 = KV == kKvMxfp4;
  constexpr int kPVB = page_value_bytes<KV>(), kPB = page_bytes<KV>();
  // With R = 3 every epilogue warp reads every tile's K scales in order, and
  // the copy into scale slot u + 16 waits for MMA u + 8, which needs all of
  // them past tile u + 6: the slot is free without a barrier of its own.
  // Round-robin warpgroups (R = 1) give no such order, so they release slots.
  // MXFP4 scales are read by the MMA warp, in order, before it issues tile u,
  // so they never need a release either.
  constexpr bool kScaleRelease = R != 3 && !kFp4;
  constexpr bool kAbsAdd = scorer_relu_abs_add<KV>();  // ReLU form: identical to the sparse scorer's
  // FP8: every lane of an epilogue warp releases the accumulator itself (one
  // arrive instruction, no warp barrier before it): the chunk's dense pass
  // 31.4 -> 30.7 ms.  MXFP4's epilogue is faster with one arrive per warp
  // after a warp barrier (29.9 against 31.1 ms).
  constexpr bool kLaneArrive = !kFp4;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sm.abort_flag;

  // ---------------------------------------------------------------- set-up
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < kScaleSlots; ++s) {
      mbar_init(&sm.s_empty[s], 32 * 4 * kEpiPerTile);  // FP8 one-row groups: every lane releases
    }
    for (int s = 0; s < kNumAcc; ++s) {
      mbar_init(&sm.t_full[s], 1);
      mbar_init(&sm.t_empty[s], (kLaneArrive ? 32 : 1) * 4 * kEpiPerTile);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Several requests: groups per request (checked row starts), their prefix.
  int num_groups = (a.p.rows + R - 1) / R;
  if (a.p.layout == kLayoutVarlen) {
    constexpr int kPer = (kMaxReq + kThreads - 1) / kThreads;
    int cnt[kPer], local = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int r = tid * kPer + j;
      cnt[j] = 0;
      if (r < a.p.num_req) {
        const int s0 = a.p.req_start[r], s1 = a.p.req_start[r + 1];
        const bool ok = 0 <= s0 && s0 <= s1 && s1 <= a.p.rows && (r > 0 || s0 == 0) &&
                        (r < a.p.num_req - 1 || s1 == a.p.rows);
        if (!ok && blockIdx.x == 0) report(a.p.dev_err, kDevErrReq);
        cnt[j] = ok ? (s1 - s0 + R - 1) / R : 0;
      }
      local += cnt[j];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sm.warp_sum[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      if (w < warp) before += static_cast<int>(sm.warp_sum[w]);
      total += static_cast<int>(sm.warp_sum[w]);
    }
    int run = before + incl - local;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int r = tid * kPer + j;
      if (r < a.p.num_req) sm.gpre[r] = run;
      run += cnt[j];
    }
    if (tid == 0) sm.gpre[a.p.num_req] = total;
    num_groups = total;
    __syncthreads();
  }
  // Work split: this CTA's share of the (group, tile) list.
  {
    const int per = (num_groups + kThreads - 1) / kThreads;
    const int g0 = min(num_groups, tid * per), g1 = min(num_groups, g0 + per);
    long long mine = 0;
    for (int g = g0; g < g1; ++g) {
      const RowGroup grp = row_group<R>(a, sm.gpre, g);
      if (blockIdx.x == 0)
        for (int i = 0; i < grp.count; ++i)
          if (scored_len(a, grp.first + i) < 0) report(a.p.dev_err, kDevErrLen);
      mine += (group_len<R>(a, grp) + kTileM - 1) / kTileM;
    }
    long long incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) sm.warp_sum[warp] = incl;
    __syncthreads();
    long long before = 0, total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      if (w < warp) before += sm.warp_sum[w];
      total += sm.warp_sum[w];
    }
    const long long excl = before + incl - mine;
    const long long tb = total * blockIdx.x / gridDim.x, te = total * (blockIdx.x + 1) / gridDim.x;
    if (tid == 0) {
      sm.t_begin = tb;
      sm.t_end = te;
      sm.g_begin = num_groups;
      sm.o_begin = 0;
    }
    __syncthreads();
    if (tb < te && excl <= tb && tb < excl + mine) {
      long long acc = excl;
      for (int g = g0; g < g1; ++g) {
        const int n = (group_len<R>(a, row_group<R>(a, sm.gpre, g)) + kTileM - 1) / kTileM;
        if (tb < acc + n) {
          sm.g_begin = g;
          sm.o_begin = static_cast<int>(tb - acc);
          break;
        }
        acc += n;
      }
    }
  }
  // A scale factors: all ones, written once into every lane quadrant.
  if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    tmem_st4(tmem_addr(sm.tmem_base, 32 * (warp & 3), kSfaCol), kUnitScales, kUnitScales, kUnitScales, kUnitScales);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tbase = sm.tmem_base;
  long long remaining = sm.t_end - sm.t_begin;
  int g = sm.g_begin, off = sm.o_begin;
  uint32_t tseq = 0;    // tiles so far: every ring slot and phase derives from it
  uint32_t issued = 0;  // producer warps: one past the sequence number of the last tile this warp issued
  const int epi = warp >= kEpiWarp0 ? (warp - kEpiWarp0) >> 2 : -1;  // epilogue warpgroup
  const int quad = warp & 3;
  unsigned long long w2[32];  // head weights, packed pairs

  while (remaining > 0 && g < num_groups) {
    const RowGroup grp = row_group<R>(a, sm.gpre, g);
    const int glen = group_len<R>(a, grp);
    const int ntiles = (glen + kTileM - 1) / kTileM;
    const int take = static_cast<int>(min(static_cast<long long>(ntiles - off), remaining));
    if (take <= 0) {
      ++g;
      off = 0;
      continue;
    }
    __syncthreads();  // the previous group is fully consumed
    if (*abort_flag) break;
    // ---- group set-up: the B tile, queries widened to e4m3 (128-byte
    // swizzled rows) against FP8 K, or kept packed (64-byte swizzled rows)
    // against MXFP4 K
    if (kFp4) {
      for (int idx = tid; idx < N * 4; idx += kThreads) {
        const int n = idx >> 2, c = idx & 3;
        const int row = grp.first + n / kHeads, head = n % kHeads;
        uint2 lo = make_uint2(0, 0), hi = make_uint2(0, 0);
        if (n / kHeads < grp.count) {
          const uint2* src =
              reinterpret_cast<const uint2*>(a.p.q_fp4 + (static_cast<int64_t>(row) * kHeads + head) * 64 + c * 16);
          lo = src[0];
          hi = src[1];
        }
        *reinterpret_cast<uint4*>(sm.q + sw64_offset(n, c * 16)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
      }
    } else {
      for (int idx = tid; idx < N * 8; idx += kThreads) {
        const int n = idx >> 3, c = idx & 7;
        const int row = grp.first + n / kHeads, head = n % kHeads;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (n / kHeads < grp.count) {
          const uint2 packed =
              *reinterpret_cast<const uint2*>(a.p.q_fp4 + (static_cast<int64_t>(row) * kHeads + head) * 64 + c * 8);
          v = widen_fp4x16(packed);
        }
        *reinterpret_cast<uint4*>(sm.q + sw128_offset(n, c * 16)) = v;
      }
    }
    fence_proxy_async_smem();
    if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
      // B scale factors: column c, lane l <-> B row n = 32 c + l, byte j = K block j
      uint32_t sf[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int n = 32 * c + lane;
        const int row = grp.first + n / kHeads, head = n % kHeads;
        sf[c] = (n < N && n / kHeads < grp.count)
                    ? *reinterpret_cast<const uint32_t*>(a.p.q_sf + (static_cast<int64_t>(row) * kHeads + head) * 4)
                    : kUnitScales;
      }
      tmem_st4(tmem_addr(tbase, 32 * quad, kSfbCol), sf[0], sf[1], sf[2], sf[3]);
      tmem_st4(tmem_addr(tbase, 32 * quad, kSfbCol + 4), sf[4], sf[5], sf[6], sf[7]);
      tmem_st_wait();
    }
    // epilogue: this warpgroup's row and its head weights
    int row = -1, rlen = 0;
    if (epi >= 0) {
      const int i = R == 3 ? epi : 0;
      row = i < grp.count ? grp.first + i : a.p.rows;
      if (row < a.p.rows) {
        rlen = max(scored_len(a, row), 0);  // 0 when the row is skipped: nothing is stored
        load_head_weights(w2, a.p.w + static_cast<int64_t>(row) * kHeads);
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0 || warp == 2) {
      // ---------------------------------------------------------------- TMA producers
      // warp 0 the even tiles of the sequence, warp 2 the odd ones, so that
      // the producer work sits on two sub-partitions, not one
      const uint32_t par = static_cast<uint32_t>(warp >> 1);
      const int req = grp.req;
      const int32_t* pt = a.p.page_table + static_cast<int64_t>(req) * a.p.max_pages;
      const int end = off + take;
      uint32_t ts = tseq;
      bool ok = true;
      TilePages nxt{-1, -1};
      if (off + lane < end) nxt = load_tile_pages(pt, off + lane, glen, a.p.num_pages, a.p.dev_err);
      for (int c0 = off; c0 < end && ok; c0 += 32) {
        const TilePages cur = nxt;
        if (c0 + 32 + lane < end) nxt = load_tile_pages(pt, c0 + 32 + lane, glen, a.p.num_pages, a.p.dev_err);
        const int n = min(32, end - c0);
        for (int i = 0; i < n; ++i, ++ts) {
          if ((ts & 1u) != par) continue;
          const int pid[2] = {__shfl_sync(0xffffffffu, cur.lo, i), __shfl_sync(0xffffffffu, cur.hi, i)};
          const uint32_t ki = ts & (kStages - 1), kp = (ts / kStages) & 1;
          const uint32_t si = ts & (kScaleSlots - 1), sp = (ts / kScaleSlots) & 1;
          if (!warp_wait_fast(&sm.k_empty[ki], kp ^ 1, abort_flag) ||
              (kScaleRelease && !warp_wait_fast(&sm.s_empty[si], sp ^ 1, abort_flag))) {
            if (lane == 0) set_abort(sm, a.p.dev_err);
            ok = false;
            break;
          }
          const uint32_t nvalid = (pid[0] >= 0) + (pid[1] >= 0);
          // the tile's scale words complete on its K barrier: the MMA warp
          // waits on it before the MMAs (MXFP4 stages the words from there),
          // and the epilogue reads the scales once the accumulator is full,
          // which follows that wait
          mbar_arrive_expect_tx_elect(&sm.k_full[ki], nvalid * (kPVB + kPage * 4));
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (pid[j] < 0) continue;
            tma_load_3d_elect(sm.kv[ki] + j * kPVB, &tmap, 0, 0, pid[j], &sm.k_full[ki]);
            bulk_load_elect(&sm.ks[si][j * kPage], a.p.k_pool + static_cast<int64_t>(pid[j]) * kPB + kPVB, kPage * 4,
                            &sm.k_full[ki]);
          }
          issued = ts + 1;
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer (whole warp, one lane issues)
      // FP8 K: four kind::mxf8f6f4 steps of K = 32 (A scale factors 1);
      // MXFP4 K: two kind::mxf4 steps of K = 64, A scale factors from the
      // tile's scale words, staged transposed and copied into tensor memory.
      uint64_t bdesc[4];
      uint32_t idesc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bdesc[k] = kFp4 ? sdesc_k64_sw64(smem_u32(sm.q) + 32 * (k & 1)) : sdesc_k128_sw128(smem_u32(sm.q) + 32 * k);
        idesc[k] = kFp4 ? idesc_mxf4(kTileM, N, 2 * (k & 1), 2 * (k & 1)) : idesc_mxf8f6f4_e4m3(kTileM, N, k, k);
      }
      uint32_t ts = tseq;
      for (int t = off; t < off + take; ++t, ++ts) {
        const uint32_t ki = ts & (kStages - 1), kp = (ts / kStages) & 1;
        const uint32_t ai = ts & (kNumAcc - 1), ap = (ts / kNumAcc) & 1;
        const uint32_t si = ts & (kScaleSlots - 1);
        if (!warp_wait_fast(&sm.k_full[ki], kp, abort_flag) ||
            !warp_wait_fast(&sm.t_empty[ai], ap ^ 1, abort_flag)) {
          if (lane == 0) set_abort(sm, a.p.dev_err);
          break;
        }
        tc_fence_after();
        const uint32_t d = tbase + ai * N;
        const uint32_t a0 = smem_u32(sm.kv[ki]);
        if (kFp4) {
          // lane l's 16 bytes: the scale words of positions l, 32 + l, 64 + l,
          // 96 + l (A row 32 c + l <-> column c, lane l, every lane quadrant)
          const uint32_t* ksw = reinterpret_cast<const uint32_t*>(sm.ks[si]);
          uint8_t* stage = sm.kv[ki] + 8192;
          *reinterpret_cast<uint4*>(stage + 16 * lane) =
              make_uint4(ksw[lane], ksw[32 + lane], ksw[64 + lane], ksw[96 + lane]);
          fence_proxy_async_smem();
          __syncwarp();
          const uint32_t sfa = tbase + kSfa4Col + 4 * ki;
          tmem_cp_32x128b_x4_elect(sfa, sdesc_rows16(smem_u32(stage)));
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_mxf4_elect(d, sdesc_k64_sw64(a0 + 32 * kk), bdesc[kk], idesc[kk], sfa, tbase + kSfbCol, kk);
        } else {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_mxf8f6f4_elect(d, sdesc_k128_sw128(a0 + 32 * kk), bdesc[kk], idesc[kk], tbase + kSfaCol,
                               tbase + kSfbCol, kk);
        }
        mma_commit_elect(&sm.k_empty[ki]);
        mma_commit_elect(&sm.t_full[ai]);
      }
    } else if (epi >= 0) {
      // ---------------------------------------------------------------- epilogue
      const int p = 32 * quad + lane;
      const int nb = (rlen + kBlock - 1) / kBlock;
      float* keys_row = row >= 0 && row < a.p.rows ? a.keys + static_cast<int64_t>(row) * a.keys_stride : nullptr;
      const uint32_t col0 = R == 3 ? epi * kHeads : 0;
      const uint32_t ts0 = tseq;
      float* kp_row = keys_row != nullptr ? keys_row + (p >> 3) : nullptr;  // + 16 t per tile
      // per-warp bases: this warp's tensor-memory lanes and columns, its scale
      // word in slot 0 of the scale ring
      const uint32_t tq = tmem_addr(tbase, 32 * quad, col0);
      const uint32_t ks0 = smem_u32(&sm.ks[0][p]);
      // One tile: accumulator stage ai (a compile-time constant where the
      // caller knows it), phases from the tile's sequence number ts.
      // kIn (a compile-time flag): every position of the tile is below the
      // row's length and its last block is not the newest, so neither the
      // mask nor the +inf pin applies.
      auto tile = [&](int t, uint32_t ts, uint32_t ai, auto interior) -> bool {
        constexpr bool kIn = decltype(interior)::value;
        const uint32_t ap = (ts / kNumAcc) & 1;
        const uint32_t si = ts & (kScaleSlots - 1);
        if (!warp_wait_fast(&sm.t_full[ai], ap, abort_flag)) {
          if (lane == 0) set_abort(sm, a.p.dev_err);
          return false;
        }
        tc_fence_after();
        HeadAcc part = {{0, 0, 0, 0}};
        uint32_t x[32];
        const uint32_t taddr = tq + ai * N;
        tmem_ld32(taddr, x);
        tmem_ld_wait();
        head_reduce_half<kAbsAdd>(part, x, w2);
        tmem_ld32(taddr + 32, x);
        tmem_ld_wait();
        head_reduce_half<kAbsAdd>(part, x, w2 + 16);
        tc_fence_before();
        if (kLaneArrive) {
          mbar_arrive(&sm.t_empty[ai]);  // every lane, once its own loads are done
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.t_empty[ai]);
        }
        const float score = head_reduce_finish<kAbsAdd>(part);
        float kscale = 1.0f;  // MXFP4: the scales are inside the MMA
        if (!kFp4) {
          kscale = lds_f32(ks0 + si * (kTileM * 4));
        }
        if (kScaleRelease) mbar_arrive(&sm.s_empty[si]);  // every lane, after its scale read (FP8 only)
        const int pos = t * kTileM + p;
        float v = (kIn || pos < rlen) ? score * kscale : -__int_as_float(0x7f800000);
        if (kLocal) {
          // a context shard's blocks of 1 << shift positions, no +inf pin (the
          // merge across shards pins the global newest block)
          const int bs = 1 << a.block_shift;
          for (int o = 1; o < bs; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          if ((lane & (bs - 1)) == 0 && pos < rlen) keys_row[pos >> a.block_shift] = v;
        } else {
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          if (kIn) {
            // every lane of a block's 8 holds its maximum: all store (one
            // 16-byte segment per warp), no predicate
            kp_row[t * (kTileM / kBlock)] = v;
          } else if ((lane & 7) == 0 && pos < rlen) {
            kp_row[t * (kTileM / kBlock)] = (pos >> 3) == nb - 1 ? __int_as_float(0x7f800000) : v;
          }
        }
        return true;
      };
      using kYes = std::true_type;
      using kNo = std::false_type;
      const int end = off + take;
      if (R == 3) {
        // two accumulator stages: tiles in pairs, stage 0 then stage 1, so
        // that every stage-dependent address is a constant of its copy
        int t = off;
        bool ok = true;
        if ((ts0 & 1) && t < end) {
          ok = tile(t, ts0, 1, kNo{});
          ++t;
        }
        for (; ok && t + 1 < end; t += 2) {
          const uint32_t ts = ts0 + (t - off);
          if ((t + 2) * kTileM < rlen)  // both tiles interior
            ok = tile(t, ts, 0, kYes{}) && tile(t + 1, ts + 1, 1, kYes{});
          else
            ok = tile(t, ts, 0, kNo{}) && tile(t + 1, ts + 1, 1, kNo{});
        }
        if (ok && t < end) ok = tile(t, ts0 + (t - off), 0, kNo{});
      } else {
        for (int t = off; t < end; ++t) {
          const uint32_t ts = ts0 + (t - off);
          if (static_cast<int>(ts % 3) != epi) continue;  // round-robin warpgroups
          if (!tile(t, ts, ts & (kNumAcc - 1), kNo{})) break;
        }
      }
    }
    tseq += take;
    remaining -= take;
    ++g;
    off = 0;
  }

  // ---------------------------------------------------------------- tear-down
  __syncthreads();
  if (*abort_flag) {
    // make sure no copy or MMA is still writing before the CTA exits
    if (warp == 1 && lane == 0) {
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, nullptr, 1000000000ull);
    }
    if ((warp == 0 || warp == 2) && lane == 0) {
      // this producer's tiles (its parity) among the last kStages issued
      const uint32_t par = static_cast<uint32_t>(warp >> 1);
      for (uint32_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
        if ((i & 1u) != par) continue;
        mbar_wait(&sm.k_full[i % kStages], (i / kStages) & 1, nullptr, 1000000000ull);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

template <int R, int KV, bool kLocal = false>
cudaError_t launch_one(const CUtensorMap& tmap, const DenseArgs& a, int smem, cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(dense_amax8_kernel<R, KV, kLocal>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dense_amax8_kernel<R, KV, kLocal><<<device_sm_count(), kThreads, smem, stream>>>(tmap, a);
  return cudaGetLastError();
}

cudaError_t launch_dense_amax8(const DenseArgs& a, cudaStream_t stream) {
  CUtensorMap tmap;
  cudaError_t e = make_pool_tmap(&tmap, a.p.k_pool, a.p.num_pages, a.p.kv_format, kPage);
  if (e != cudaSuccess) return e;
  const int smem = static_cast<int>(sizeof(Smem)) + 1024;
  const bool prefill = a.p.layout != kLayoutDecode;
  if (a.block_shift != 3)  // a context shard's blocks (FP8 pages)
    return prefill ? launch_one<3, kKvFp8, true>(tmap, a, smem, stream) : launch_one<1, kKvFp8, true>(tmap, a, smem, stream);
  if (a.p.kv_format == kKvMxfp4)
    return prefill ? launch_one<3, kKvMxfp4>(tmap, a, smem, stream) : launch_one<1, kKvMxfp4>(tmap, a, smem, stream);
  return prefill ? launch_one<3, kKvFp8>(tmap, a, smem, stream) : launch_one<1, kKvFp8>(tmap, a, smem, stream);
}

}  // namespace ci
