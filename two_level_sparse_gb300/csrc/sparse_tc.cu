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
// One persistent CTA per SM, 16 warps:
//   warp 0      gathers one 128-position tile = 16 candidate blocks: each lane
//               of half the warp issues one tensor-map load of a block's eight
//               128-byte K vectors (1 KB, 128-byte swizzle, landing on its own
//               8-row atom of the MMA tile), the other half bulk-copies the
//               block's eight fp32 scales;
//   warp 1      tcgen05.mma kind::mxf8f6f4 block_scale, M = 128 gathered
//               positions, N = 64 heads, K = 128;
//   warps 4-15  three epilogue warpgroups take tiles round-robin: ReLU + head
//               weights + K scale (the same arithmetic as the dense pass), and
//               store an order-preserving key per candidate in shared memory;
//               after the row's last tile they run the radix top-k together.
// Scores never leave the chip.
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kThreads = 512;
constexpr int kStages = 6;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiThreads = 384;
constexpr int kTmemCols = 512;
constexpr int kNumAcc = 6;  // 6 x 64 accumulator columns
constexpr int kSfaCol = 384;
constexpr int kSfbCol = 388;
constexpr int kBlocksPerTile = kTileM / kBlock;  // 16
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;

struct __align__(1024) Smem {
  uint8_t kv[kStages][kTileM * kDim];
  uint8_t q[kHeads * kDim];
  float ks[kStages][kTileM];
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t t_full[kNumAcc], t_empty[kNumAcc];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int valid_count;
  int row_abort;
  TopkShared topk;
  // followed by the score keys: round_up(max_blocks, 16) * 8 uint32
};

__device__ __forceinline__ void set_abort(Smem& sm, int32_t* dev_err) {
  sm.abort_flag = 1;
  report(dev_err, kDevErrTimeout);
}

__global__ void __launch_bounds__(kThreads, 1)
    select_kernel(const __grid_constant__ CUtensorMap tmap, const SelectArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* sc = reinterpret_cast<uint32_t*>(&sm + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1 + 4);
    }
    for (int s = 0; s < kNumAcc; ++s) {
      mbar_init(&sm.t_full[s], 1);
      mbar_init(&sm.t_empty[s], 4);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    tmem_st4(tmem_addr(tbase, 32 * (warp & 3), kSfaCol), kUnitScales, kUnitScales, kUnitScales, kUnitScales);
    tmem_st_wait();
  }

  uint32_t kcount = 0, issued = 0;
  const int epi = warp >= kEpiWarp0 ? (warp - kEpiWarp0) >> 2 : -1;
  const int quad = warp & 3;
  uint64_t w2[32];

  for (int row = blockIdx.x; row < a.p.rows; row += gridDim.x) {
    int L = a.p.seq_len[row];
    int nv = a.nvalid[row];
    bool bad = false;
    if (L < 0 || L > a.p.max_len) {
      if (tid == 0) report(a.p.dev_err, kDevErrLen);
      bad = true;
    }
    if (nv < 0 || nv > a.max_blocks) {
      if (tid == 0) report(a.p.dev_err, kDevErrBlock);
      bad = true;
    }
    if (bad) {
      L = 0;
      nv = 0;
    }
    const int nb = (L + kBlock - 1) / kBlock;
    const int ntiles = (nv + kBlocksPerTile - 1) / kBlocksPerTile;
    const int32_t* brow = a.blocks + static_cast<int64_t>(row) * a.blocks_stride;
    const int req = a.p.layout == 1 ? 0 : row;
    const int32_t* pt = a.p.page_table + static_cast<int64_t>(req) * a.p.max_pages;

    tc_fence_before();
    __syncthreads();  // the previous row is fully consumed (scores, Q, scale factors)
    tc_fence_after();
    if (*abort_flag) break;
    for (int idx = tid; idx < kHeads * 8; idx += kThreads) {
      const int head = idx >> 3, c = idx & 7;
      const uint2 packed =
          *reinterpret_cast<const uint2*>(a.p.q_fp4 + (static_cast<int64_t>(row) * kHeads + head) * 64 + c * 8);
      *reinterpret_cast<uint4*>(sm.q + sw128_offset(head, c * 16)) = widen_fp4x16(packed);
    }
    fence_proxy_async_smem();
    if (tid == 0) sm.valid_count = 0;
    if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
      uint32_t sf[2];
#pragma unroll
      for (int c = 0; c < 2; ++c)
        sf[c] = *reinterpret_cast<const uint32_t*>(a.p.q_sf + (static_cast<int64_t>(row) * kHeads + 32 * c + lane) * 4);
      tmem_st4(tmem_addr(tbase, 32 * quad, kSfbCol), sf[0], sf[1], kUnitScales, kUnitScales);
      tmem_st_wait();
    }
    if (epi >= 0) {
      const float2* wp = reinterpret_cast<const float2*>(a.p.w + static_cast<int64_t>(row) * kHeads);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float2 v = wp[j];
        w2[j] = pack2(v.x, v.y);
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0) {
      // ---------------------------------------------------------------- gather
      for (int t = 0; t < ntiles; ++t) {
        const uint32_t i = kcount + t, s = i % kStages, ph = (i / kStages) & 1;
        if (!warp_wait(&sm.k_empty[s], ph ^ 1, abort_flag)) {
          if (lane == 0) set_abort(sm, a.p.dev_err);
          break;
        }
        const int j = lane & 15;
        const int slot = t * kBlocksPerTile + j;
        int pid = -1, b = -1;
        if (slot < nv) {
          b = brow[slot];
          if (b < 0 || b >= nb) {
            if (lane < 16) report(a.p.dev_err, kDevErrBlock);
          } else {
            pid = pt[b >> 3];
            if (pid < 0 || pid >= a.p.num_pages) {
              if (lane < 16) report(a.p.dev_err, kDevErrPage);
              pid = -1;
            }
          }
        }
        const uint32_t nload = __popc(__ballot_sync(0xffffffffu, pid >= 0 && lane < 16));
        if (lane == 0) mbar_arrive_expect_tx(&sm.k_full[s], nload * (kBlock * kDim + kBlock * 4));
        __syncwarp();
        if (pid >= 0) {
          const int off = (b & 7) * kBlock;
          if (lane < 16)
            tma_load_3d(sm.kv[s] + j * (kBlock * kDim), &tmap, 0, off, pid, &sm.k_full[s]);
          else
            bulk_load(&sm.ks[s][j * kBlock],
                      a.p.k_pool + static_cast<int64_t>(pid) * kPageBytes + kPageValueBytes + off * 4, kBlock * 4,
                      &sm.k_full[s]);
        }
        ++issued;
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA
      if (lane == 0) {
        uint64_t bdesc[4];
        uint32_t idesc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          bdesc[k] = sdesc_k128_sw128(smem_u32(sm.q) + 32 * k);
          idesc[k] = idesc_mxf8f6f4_e4m3(kTileM, kHeads, k, k);
        }
        for (int t = 0; t < ntiles; ++t) {
          const uint32_t i = kcount + t, s = i % kStages, ph = (i / kStages) & 1;
          const uint32_t acc = i % kNumAcc, aph = (i / kNumAcc) & 1;
          if (!mbar_wait(&sm.k_full[s], ph, abort_flag) || !mbar_wait(&sm.t_empty[acc], aph ^ 1, abort_flag)) {
            set_abort(sm, a.p.dev_err);
            break;
          }
          tc_fence_after();
          const uint32_t d = tbase + acc * kHeads;
          const uint32_t a0 = smem_u32(sm.kv[s]);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_mxf8f6f4(d, sdesc_k128_sw128(a0 + 32 * k), bdesc[k], idesc[k], tbase + kSfaCol, tbase + kSfbCol, k);
          mma_commit(&sm.k_empty[s]);
          mma_commit(&sm.t_full[acc]);
        }
      }
      __syncwarp();
    } else if (epi >= 0) {
      // ---------------------------------------------------------------- score epilogue
      const int p = 32 * quad + lane;
      for (int t = epi; t < ntiles; t += 3) {
        const uint32_t i = kcount + t, s = i % kStages, ph = (i / kStages) & 1;
        const uint32_t acc = i % kNumAcc, aph = (i / kNumAcc) & 1;
        if (!warp_wait(&sm.t_full[acc], aph, abort_flag)) {
          if (lane == 0) set_abort(sm, a.p.dev_err);
          break;
        }
        tc_fence_after();
        uint64_t part[4] = {0, 0, 0, 0};
        uint32_t x[32];
        const uint32_t taddr = tmem_addr(tbase, 32 * quad, acc * kHeads);
        tmem_ld32(taddr, x);
        tmem_ld_wait();
        head_reduce_half(part, x, w2);
        tmem_ld32(taddr + 32, x);
        tmem_ld_wait();
        head_reduce_half(part, x, w2 + 16);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.t_empty[acc]);
        const float score = head_reduce_finish(part);
        if (!warp_wait(&sm.k_full[s], ph, abort_flag)) {
          if (lane == 0) set_abort(sm, a.p.dev_err);
          break;
        }
        const float kscale = sm.ks[s][p];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.k_empty[s]);
        const int slot = t * kBlocksPerTile + (p >> 3);
        bool valid = false;
        if (slot < nv) {
          const int b = brow[slot];
          const int pos = b * kBlock + (p & 7);
          valid = b >= 0 && b < nb && pos < L;
        }
        sc[t * kTileM + p] = valid ? order_key(score * kscale) : 0u;
        const uint32_t vb = __ballot_sync(0xffffffffu, valid);
        if (lane == 0 && vb) atomicAdd(&sm.valid_count, __popc(vb));
      }
      // ---------------------------------------------------------------- top-k of the row
      const int etid = tid - kEpiWarp0 * 32;
      named_sync(1, kEpiThreads);
      if (etid == 0) sm.row_abort = *abort_flag;
      named_sync(1, kEpiThreads);
      const int n = nv * kBlock;
      const int k = min(a.topk, sm.valid_count);
      int32_t* out = a.out_pos + static_cast<int64_t>(row) * a.out_stride;
      float* osc = a.out_score != nullptr ? a.out_score + static_cast<int64_t>(row) * a.out_stride : nullptr;
      if (k > 0 && !sm.row_abort) {
        block_topk(sc, n, k, sm.topk, etid, kEpiThreads, 1, [&](int rank, int idx, uint32_t u) {
          out[rank] = brow[idx >> 3] * kBlock + (idx & 7);
          if (osc) osc[rank] = order_key_inv(u);
        });
      }
      for (int r = max(k, 0) + etid; r < a.topk; r += kEpiThreads) {
        out[r] = -1;
        if (osc) osc[r] = -__int_as_float(0x7f800000);
      }
    }
    kcount += ntiles;
  }

  __syncthreads();
  if (*abort_flag) {
    if (warp == 1 && lane == 0) {
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, nullptr, 1000000000ull);
    }
    if (warp == 0 && lane == 0) {
      for (uint32_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        mbar_wait(&sm.k_full[i % kStages], (i / kStages) & 1, nullptr, 1000000000ull);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

size_t select_smem_bytes(int max_blocks) {
  const size_t nsc = static_cast<size_t>((max_blocks + kBlocksPerTile - 1) / kBlocksPerTile) * kTileM;
  return sizeof(Smem) + nsc * 4 + 1024;
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream) {
  if (a.p.rows == 0) return cudaSuccess;
  CUtensorMap tmap;
  cudaError_t e = make_pool_tmap(&tmap, a.p.k_pool, a.p.num_pages, kBlock);
  if (e != cudaSuccess) return e;
  const int smem = static_cast<int>(select_smem_bytes(a.max_blocks));
  e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = min(device_sm_count(), a.p.rows);
  select_kernel<<<grid, kThreads, smem, stream>>>(tmap, a);
  return cudaGetLastError();
}

}  // namespace ci
