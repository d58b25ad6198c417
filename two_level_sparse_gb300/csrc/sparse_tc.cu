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
// One persistent CTA per SM works through its rows; every stage is
// double-buffered so consecutive rows overlap:
//   warp 0      MMA issuer: per row, tcgen05.cp of the row's query scale
//               factors into tensor memory, then per 128-position tile four
//               tcgen05.mma kind::mxf8f6f4 block_scale (M = 128 gathered
//               positions, N = 64 heads, K = 32 each);
//   warps 1-3   top-k of the previous row from its score buffer (radix select
//               + ordered compaction), concurrent with the next row's scoring;
//   warps 4-5   gather: 16-byte cp.async copies of the 16 candidate blocks of
//               a tile (each block is 1 KB of contiguous K in its page) into
//               the 128-byte-swizzled MMA tile, plus their fp32 scales; and,
//               one row ahead, the next row's page lookups, its query widened
//               from e2m1 to e4m3 and its scale-factor staging;
//   warps 8-15  two scoring warpgroups, tiles alternating: the same epilogue
//               arithmetic as the dense pass, one order-preserving key per
//               candidate into the row's score buffer in shared memory.
// Scores never leave the chip.
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kThreads = 512;
constexpr int kStages = 3;
constexpr int kLag = 1;  // cp.async groups a gather thread keeps in flight before signalling
constexpr int kNumAcc = 6;
constexpr int kSfaCol = 384;  // 4 columns of A scale factors (all 1.0)
constexpr int kSfbCol = 392;  // two buffers of 4 columns of B scale factors
constexpr int kBlocksPerTile = kTileM / kBlock;  // 16
constexpr int kMaxBlocks = 2176;  // >= topk + 1 for every supported topk
constexpr int kTopkWarp0 = 1, kTopkThreads = 96, kTopkBar = 2;
constexpr int kGatherWarp0 = 4, kGatherThreads = 64;
constexpr int kScoreWarp0 = 8;
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;

struct __align__(1024) Smem {
  uint8_t kv[kStages][kTileM * kDim];  // gathered A tiles (1024-aligned)
  uint8_t q[2][kHeads * kDim];         // widened queries, double-buffered
  uint8_t sf[2][512];                  // query scale factors staged for tcgen05.cp
  float ks[kStages][kTileM];           // K scales of each stage
  int32_t info[2][kMaxBlocks];         // per candidate: (page << 3) | (block & 7), or -1
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
  TopkShared topk;
  // followed by the score keys: 2 x round_up(max_blocks, 16) * 8 uint32
};

__device__ __forceinline__ void set_abort(Smem& sm, int32_t* dev_err) {
  sm.abort_flag = 1;
  report(dev_err, kDevErrTimeout);
}

struct RowInfo {
  int row, L, nv, nb, ntiles;
};

__device__ __forceinline__ RowInfo row_info(const SelectArgs& a, int row, bool report_errors) {
  RowInfo r;
  r.row = row;
  r.L = a.p.seq_len[row];
  r.nv = a.nvalid[row];
  bool bad = false;
  if (r.L < 0 || r.L > a.p.max_len) {
    if (report_errors) report(a.p.dev_err, kDevErrLen);
    bad = true;
  }
  if (r.nv < 0 || r.nv > a.max_blocks) {
    if (report_errors) report(a.p.dev_err, kDevErrBlock);
    bad = true;
  }
  if (bad) r.L = r.nv = 0;
  r.nb = (r.L + kBlock - 1) / kBlock;
  r.ntiles = (r.nv + kBlocksPerTile - 1) / kBlocksPerTile;
  return r;
}

// Ring position: stage index and phase parity, advanced one tile at a time.
struct Ring {
  uint32_t idx = 0, phase = 0;
  __device__ __forceinline__ void next(uint32_t n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1;
    }
  }
};

// Gather threads: the next row's query (e2m1 -> e4m3, swizzled), its scale
// factors staged for tcgen05.cp, and its candidates' page lookups.
__device__ __forceinline__ void prep_row(Smem& sm, const SelectArgs& a, const RowInfo& r, int ri, int gt,
                                         volatile int* abort_flag) {
  const int b = ri & 1;
  const uint32_t ph = (ri >> 1) & 1;
  // the query buffer is free once the MMAs of row ri - 2 completed
  bool ok = warp_wait(&sm.q_empty[b], ph ^ 1, abort_flag);
  for (int idx = gt; ok && idx < kHeads * 8; idx += kGatherThreads) {
    const int head = idx >> 3, c = idx & 7;
    const uint2 packed =
        *reinterpret_cast<const uint2*>(a.p.q_fp4 + (static_cast<int64_t>(r.row) * kHeads + head) * 64 + c * 8);
    *reinterpret_cast<uint4*>(sm.q[b] + sw128_offset(head, c * 16)) = widen_fp4x16(packed);
  }
  if (ok && gt < 32) {
    // lane l of the scale-factor columns: heads l and 32 + l, byte j = K block j
    const uint32_t* sfp = reinterpret_cast<const uint32_t*>(a.p.q_sf + static_cast<int64_t>(r.row) * kHeads * 4);
    *reinterpret_cast<uint4*>(sm.sf[b] + 16 * gt) = make_uint4(sfp[gt], sfp[32 + gt], kUnitScales, kUnitScales);
  }
  fence_proxy_async_smem();
  mbar_arrive(&sm.q_full[b]);
  // page lookups of the candidates, once the previous user of the buffer is done
  ok = ok && warp_wait(&sm.info_empty[b], ph ^ 1, abort_flag);
  const int req = a.p.layout == 1 ? 0 : r.row;
  const int32_t* pt = a.p.page_table + static_cast<int64_t>(req) * a.p.max_pages;
  const int32_t* brow = a.blocks + static_cast<int64_t>(r.row) * a.blocks_stride;
  for (int i = gt; ok && i < r.nv; i += kGatherThreads) {
    const int blk = brow[i];
    int v = -1;
    if (blk < 0 || blk >= r.nb) {
      report(a.p.dev_err, kDevErrBlock);
    } else {
      const int pid = pt[blk >> 3];
      if (pid < 0 || pid >= a.p.num_pages)
        report(a.p.dev_err, kDevErrPage);
      else
        v = (pid << 3) | (blk & 7);
    }
    sm.info[b][i] = v;
  }
  mbar_arrive(&sm.info_full[b]);
}

__global__ void __launch_bounds__(kThreads, 1)
    select_kernel(const SelectArgs a, const int score_cap) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* scores = reinterpret_cast<uint32_t*>(&sm + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], kGatherThreads);
      mbar_init(&sm.k_empty[s], 1 + 4);
    }
    for (int s = 0; s < kNumAcc; ++s) {
      mbar_init(&sm.t_full[s], 1);
      mbar_init(&sm.t_empty[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_full[b], kGatherThreads);
      mbar_init(&sm.q_empty[b], 1);
      mbar_init(&sm.info_full[b], kGatherThreads);
      mbar_init(&sm.info_empty[b], kGatherThreads);
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
  if (warp >= kScoreWarp0 && warp < kScoreWarp0 + 4) {
    // A scale factors: all ones, in every lane quadrant
    tmem_st4(tmem_addr(tbase, 32 * (warp & 3), kSfaCol), kUnitScales, kUnitScales, kUnitScales, kUnitScales);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int rows = a.p.rows;
  if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Ring kr, ar;
      int ri = 0;
      for (int row = blockIdx.x; row < rows; row += gridDim.x, ++ri) {
        const RowInfo r = row_info(a, row, true);
        const int b = ri & 1;
        if (!mbar_wait(&sm.q_full[b], (ri >> 1) & 1, abort_flag)) {
          set_abort(sm, a.p.dev_err);
          break;
        }
        tc_fence_after();
        const uint32_t sfb = tbase + kSfbCol + 4 * b;
        tmem_cp_32x128b_x4(sfb, sdesc_rows16(smem_u32(sm.sf[b])));
        uint64_t bdesc[4];
        uint32_t idesc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          bdesc[k] = sdesc_k128_sw128(smem_u32(sm.q[b]) + 32 * k);
          idesc[k] = idesc_mxf8f6f4_e4m3(kTileM, kHeads, k, k);
        }
        bool ok = true;
        for (int t = 0; t < r.ntiles && ok; ++t) {
          ok = mbar_wait(&sm.k_full[kr.idx], kr.phase, abort_flag) &&
               mbar_wait(&sm.t_empty[ar.idx], ar.phase ^ 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tbase + ar.idx * kHeads;
          const uint32_t a0 = smem_u32(sm.kv[kr.idx]);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_mxf8f6f4(d, sdesc_k128_sw128(a0 + 32 * k), bdesc[k], idesc[k], tbase + kSfaCol, sfb, k);
          mma_commit(&sm.k_empty[kr.idx]);
          mma_commit(&sm.t_full[ar.idx]);
          kr.next(kStages);
          ar.next(kNumAcc);
        }
        if (!ok) {
          set_abort(sm, a.p.dev_err);
          break;
        }
        mma_commit(&sm.q_empty[b]);  // the query buffer is free once these MMAs complete
      }
    }
    __syncwarp();
  } else if (warp >= kTopkWarp0 && warp < kTopkWarp0 + 3) {
    // ------------------------------------------------------------------ top-k of finished rows
    const int kt = tid - kTopkWarp0 * 32;
    int ri = 0;
    for (int row = blockIdx.x; row < rows; row += gridDim.x, ++ri) {
      const RowInfo r = row_info(a, row, false);
      const int b = ri & 1;
      if (kt == 0) sm.topk_go = mbar_wait(&sm.sc_full[b], (ri >> 1) & 1, abort_flag) ? 1 : 0;
      named_sync(kTopkBar, kTopkThreads);
      const int go = sm.topk_go;
      if (!go) {
        if (kt == 0) set_abort(sm, a.p.dev_err);
        break;
      }
      // every scoring warp arrived on sc_full after its stores; the barrier
      // above gives the other top-k threads the same view
      const int k = min(a.topk, sm.vcount[b]);
      const int32_t* brow = a.blocks + static_cast<int64_t>(row) * a.blocks_stride;
      int32_t* out = a.out_pos + static_cast<int64_t>(row) * a.out_stride;
      float* osc = a.out_score != nullptr ? a.out_score + static_cast<int64_t>(row) * a.out_stride : nullptr;
      const uint32_t* sc = scores + b * score_cap;
      if (k > 0) {
        block_topk(sc, r.nv * kBlock, k, sm.topk, kt, kTopkThreads, kTopkBar, [&](int rank, int idx, uint32_t u) {
          out[rank] = brow[idx >> 3] * kBlock + (idx & 7);
          if (osc) osc[rank] = order_key_inv(u);
        });
      }
      for (int i = max(k, 0) + kt; i < a.topk; i += kTopkThreads) {
        out[i] = -1;
        if (osc) osc[i] = -__int_as_float(0x7f800000);
      }
      named_sync(kTopkBar, kTopkThreads);
      if (kt == 0) {
        sm.vcount[b] = 0;
        mbar_arrive(&sm.sc_empty[b]);
      }
    }
  } else if (warp >= kGatherWarp0 && warp < kGatherWarp0 + 2) {
    // ------------------------------------------------------------------ gather + next-row prep
    const int gt = tid - kGatherWarp0 * 32;  // 0..63
    const int g = gt >> 5;                   // this warp's half of each tile: blocks 8g .. 8g+7
    Ring kr;
    uint32_t issued = 0, signalled = 0;
    int ri = 0;
    bool ok = true;
    int row = blockIdx.x;
    RowInfo r{};
    if (row < rows) {
      r = row_info(a, row, false);
      prep_row(sm, a, r, 0, gt, abort_flag);
    }
    for (; row < rows && ok; row += gridDim.x, ++ri) {
      const int b = ri & 1;
      const int next_row = row + gridDim.x;
      const RowInfo rn = next_row < rows ? row_info(a, next_row, false) : RowInfo{};
      const int prep_at = min(kStages, r.ntiles);
      const uint32_t row_start = issued;
      bool prepped = next_row >= rows;
      // the next row's prep waits for the MMAs of the previous row: every one of
      // its tiles must have been signalled first
      auto flush_previous = [&]() {
        if (signalled < row_start) {
          cp_async_wait<0>();
          fence_proxy_async_smem();
          while (signalled < issued) {
            mbar_arrive(&sm.k_full[signalled % kStages]);
            ++signalled;
          }
        }
      };
      ok = warp_wait(&sm.info_full[b], (ri >> 1) & 1, abort_flag);
      const int32_t* info = sm.info[b];
      for (int t = 0; t < r.ntiles && ok; ++t) {
        if (t == prep_at && !prepped) {
          flush_previous();
          prep_row(sm, a, rn, ri + 1, gt, abort_flag);
          prepped = true;
        }
        if (!warp_wait(&sm.k_empty[kr.idx], kr.phase ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* dst = sm.kv[kr.idx];
#pragma unroll 4
        for (int j = 0; j < 16; ++j) {
          const int blk = 8 * g + (j >> 1);
          const int slot = t * kBlocksPerTile + blk;
          const int v = slot < r.nv ? info[slot] : -1;
          if (v >= 0) {
            const int o = (j & 1) * 32 + lane;  // 16-byte chunk of the block's 1 KB
            const uint8_t* src =
                a.p.k_pool + static_cast<int64_t>(v >> 3) * kPageBytes + (v & 7) * (kBlock * kDim) + o * 16;
            cp_async16(dst + sw128_offset(blk * kBlock + (o >> 3), (o & 7) * 16), src);
          }
        }
        if (lane < 16) {
          const int blk = 8 * g + (lane >> 1), half = lane & 1;
          const int slot = t * kBlocksPerTile + blk;
          const int v = slot < r.nv ? info[slot] : -1;
          if (v >= 0)
            cp_async16(&sm.ks[kr.idx][blk * kBlock + half * 4],
                       a.p.k_pool + static_cast<int64_t>(v >> 3) * kPageBytes + kPageValueBytes +
                           ((v & 7) * kBlock + half * 4) * 4);
        }
        cp_async_commit();
        ++issued;
        if (issued - signalled > kLag) {
          cp_async_wait<kLag>();
          fence_proxy_async_smem();
          mbar_arrive(&sm.k_full[signalled % kStages]);
          ++signalled;
        }
        kr.next(kStages);
      }
      if (!ok) break;
      if (!prepped) {
        flush_previous();
        prep_row(sm, a, rn, ri + 1, gt, abort_flag);
        prepped = true;
      }
      mbar_arrive(&sm.info_empty[b]);
      r = rn;
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    while (signalled < issued) {
      mbar_arrive(&sm.k_full[signalled % kStages]);
      ++signalled;
    }
    if (!ok && lane == 0) set_abort(sm, a.p.dev_err);
  } else if (warp >= kScoreWarp0) {
    // ------------------------------------------------------------------ scoring epilogue
    const int e = (warp - kScoreWarp0) >> 2;  // scoring warpgroup 0 / 1
    const int quad = warp & 3;
    const int p = 32 * quad + lane;
    Ring kr, ar;
    uint32_t tseq = 0;
    int ri = 0;
    float w[kHeads];
    bool ok = true;
    for (int row = blockIdx.x; row < rows && ok; row += gridDim.x, ++ri) {
      const RowInfo r = row_info(a, row, false);
      const int b = ri & 1;
      uint32_t* sc = scores + b * score_cap;
      const float4* wp = reinterpret_cast<const float4*>(a.p.w + static_cast<int64_t>(row) * kHeads);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 v = wp[j];
        w[4 * j] = v.x;
        w[4 * j + 1] = v.y;
        w[4 * j + 2] = v.z;
        w[4 * j + 3] = v.w;
      }
      const int32_t* brow = a.blocks + static_cast<int64_t>(row) * a.blocks_stride;
      // the score buffer must have been read by the top-k of row ri - 2
      if (ri >= 2 && !warp_wait(&sm.sc_empty[b], ((ri >> 1) & 1) ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      uint32_t nvalid_seen = 0;
      for (int t = 0; t < r.ntiles; ++t, ++tseq) {
        const bool mine = (tseq & 1) == static_cast<uint32_t>(e);
        if (mine) {
          if (!warp_wait(&sm.t_full[ar.idx], ar.phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          uint32_t x[32];
          const uint32_t taddr = tmem_addr(tbase, 32 * quad, ar.idx * kHeads);
          tmem_ld32(taddr, x);
          tmem_ld_wait();
          head_reduce_half(acc, x, w);
          tmem_ld32(taddr + 32, x);
          tmem_ld_wait();
          head_reduce_half(acc, x, w + 32);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.t_empty[ar.idx]);
          const float score = head_reduce_finish(acc);
          if (!warp_wait(&sm.k_full[kr.idx], kr.phase, abort_flag)) {
            ok = false;
            break;
          }
          const float kscale = sm.ks[kr.idx][p];
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.k_empty[kr.idx]);
          const int slot = t * kBlocksPerTile + (p >> 3);
          bool valid = false;
          if (slot < r.nv) {
            const int blk = brow[slot];
            valid = blk >= 0 && blk < r.nb && blk * kBlock + (p & 7) < r.L;
          }
          sc[t * kTileM + p] = valid ? order_key(score * kscale) : 0u;
          nvalid_seen += __popc(__ballot_sync(0xffffffffu, valid));
        }
        kr.next(kStages);
        ar.next(kNumAcc);
      }
      if (!ok) break;
      if (lane == 0 && nvalid_seen) atomicAdd(&sm.vcount[b], static_cast<int>(nvalid_seen));
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sc_full[b]);
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

size_t select_smem_bytes(int max_blocks) {
  const size_t cap = static_cast<size_t>((max_blocks + kBlocksPerTile - 1) / kBlocksPerTile) * kTileM;
  return sizeof(Smem) + 2 * cap * 4 + 1024;
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream) {
  if (a.p.rows == 0) return cudaSuccess;
  const int cap = ((a.max_blocks + kBlocksPerTile - 1) / kBlocksPerTile) * kTileM;
  const int smem = static_cast<int>(select_smem_bytes(a.max_blocks));
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = min(device_sm_count(), a.p.rows);
  select_kernel<<<grid, kThreads, smem, stream>>>(a, cap);
  return cudaGetLastError();
}

}  // namespace ci
