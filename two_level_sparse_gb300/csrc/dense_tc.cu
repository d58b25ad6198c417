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
//   warp 0      TMA producer: two 64-position pages of FP8 K per 128-position
//               tile (one tensor-map load each, 128-byte swizzle) plus their
//               fp32 scales (bulk copy), into an 8-stage ring;
//   warp 1      MMA issuer: tcgen05.mma kind::mxf8f6f4 block_scale, M = 128
//               positions, N = 64 * R columns (R rows x 64 heads), K = 128 in
//               four K=32 steps; A = K tile (scale 1), B = the rows' queries
//               widened from e2m1 to e4m3 (exact) with their ue8m0 scales in
//               tensor memory; fp32 accumulators in tensor memory;
//   warps 4-15  epilogue, three warpgroups: tcgen05.ld of one row's 64 head
//               columns per position, ReLU + head weights (packed fp32x2 FMA),
//               K scale, length mask, max over 8 lanes, key store.
// Prefill rows share one request's pages, so R = 3 rows ride one MMA
// (N = 192); decode rows each have their own pages, R = 1 (N = 64) and the
// three epilogue warpgroups take tiles round-robin.  Work is the list of
// (row group, 128-position tile) pairs, split evenly across the CTAs.
#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kThreads = 512;
constexpr int kStages = 8;
constexpr int kEpiWarp0 = 4;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 384;  // accumulator columns (2 x 192 or 6 x 64)
constexpr int kSfaCol = 384;   // 4 columns: A scale factors (all 1.0)
constexpr int kSfbCol = 388;   // 8 columns: B scale factors
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;

struct __align__(1024) Smem {
  uint8_t kv[kStages][kTileM * kDim];  // A tiles, 1024-aligned
  uint8_t q[3 * kHeads * kDim];        // B tile (up to 192 rows of 128 B)
  float ks[kStages][kTileM];           // per-position K scales of each stage
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t t_full[6], t_empty[6];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int g_begin, o_begin;
  long long t_begin, t_end;
  long long warp_sum[kThreads / 32];
};

struct Geometry {
  int R;       // rows per group
  int N;       // MMA N = 64 R
  int n_acc;   // accumulator stages
  int epi_per_tile;  // epilogue warpgroups consuming each tile
};

__device__ __forceinline__ Geometry geometry(int layout) {
  Geometry g;
  g.R = layout == 1 ? 3 : 1;
  g.N = 64 * g.R;
  g.n_acc = kAccCols / g.N;
  g.epi_per_tile = g.R == 3 ? 3 : 1;
  return g;
}

// Length that row `row` is scored over: L if it has more than skip_le_blocks
// blocks, 0 if skipped, -1 if its length breaks the contract.
__device__ __forceinline__ int scored_len(const DenseArgs& a, int row) {
  const int L = a.p.seq_len[row];
  if (L < 0 || L > a.p.max_len) return -1;
  return ((L + kBlock - 1) / kBlock) > a.skip_le_blocks ? L : 0;
}

__device__ __forceinline__ int group_len(const DenseArgs& a, int g, int R) {
  int m = 0;
  for (int r = g * R; r < min(a.p.rows, g * R + R); ++r) m = max(m, scored_len(a, r));
  return m;
}

__device__ __forceinline__ int group_tiles(const DenseArgs& a, int g, int R) {
  return (group_len(a, g, R) + kTileM - 1) / kTileM;
}

__device__ __forceinline__ void set_abort(Smem& sm, int32_t* dev_err) {
  sm.abort_flag = 1;
  report(dev_err, kDevErrTimeout);
}

__global__ void __launch_bounds__(kThreads, 1)
    dense_amax8_kernel(const __grid_constant__ CUtensorMap tmap, const DenseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Geometry geo = geometry(a.p.layout);
  const int num_groups = (a.p.rows + geo.R - 1) / geo.R;
  volatile int* abort_flag = &sm.abort_flag;

  // ---------------------------------------------------------------- set-up
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1 + 4 * geo.epi_per_tile);
    }
    for (int s = 0; s < 6; ++s) {
      mbar_init(&sm.t_full[s], 1);
      mbar_init(&sm.t_empty[s], 4 * geo.epi_per_tile);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Work split: this CTA's share of the (group, tile) list.
  {
    const int per = (num_groups + kThreads - 1) / kThreads;
    const int g0 = min(num_groups, tid * per), g1 = min(num_groups, g0 + per);
    long long mine = 0;
    for (int g = g0; g < g1; ++g) {
      for (int r = g * geo.R; r < min(a.p.rows, g * geo.R + geo.R); ++r)
        if (scored_len(a, r) < 0 && blockIdx.x == 0) report(a.p.dev_err, kDevErrLen);
      mine += group_tiles(a, g, geo.R);
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
        const int n = group_tiles(a, g, geo.R);
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
  uint32_t kcount = 0, acount = 0;  // tiles issued so far through the rings (same on every role)
  uint32_t issued = 0;              // TMA thread: tiles whose loads were issued
  const int epi = warp >= kEpiWarp0 ? (warp - kEpiWarp0) >> 2 : -1;  // epilogue warpgroup
  const int quad = warp & 3;
  float w[kHeads];

  while (remaining > 0 && g < num_groups) {
    const int glen = group_len(a, g, geo.R);
    const int ntiles = (glen + kTileM - 1) / kTileM;
    const int take = static_cast<int>(min(static_cast<long long>(ntiles - off), remaining));
    if (take <= 0) {
      ++g;
      off = 0;
      continue;
    }
    __syncthreads();  // the previous group is fully consumed
    if (*abort_flag) break;
    // ---- group set-up: queries widened to e4m3 in the swizzled B tile
    for (int idx = tid; idx < geo.N * 8; idx += kThreads) {
      const int n = idx >> 3, c = idx & 7;
      const int row = g * geo.R + n / kHeads, head = n % kHeads;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < a.p.rows) {
        const uint2 packed = *reinterpret_cast<const uint2*>(a.p.q_fp4 + (static_cast<int64_t>(row) * kHeads + head) * 64 + c * 8);
        v = widen_fp4x16(packed);
      }
      *reinterpret_cast<uint4*>(sm.q + sw128_offset(n, c * 16)) = v;
    }
    fence_proxy_async_smem();
    if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
      // B scale factors: column c, lane l <-> B row n = 32 c + l, byte j = K block j
      uint32_t sf[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int n = 32 * c + lane;
        const int row = g * geo.R + n / kHeads, head = n % kHeads;
        sf[c] = (n < geo.N && row < a.p.rows)
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
      row = geo.R == 3 ? g * 3 + epi : g;
      if (row < a.p.rows) {
        rlen = max(scored_len(a, row), 0);
        const float4* wp = reinterpret_cast<const float4*>(a.p.w + static_cast<int64_t>(row) * kHeads);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float4 v = wp[j];
          w[4 * j] = v.x;
          w[4 * j + 1] = v.y;
          w[4 * j + 2] = v.z;
          w[4 * j + 3] = v.w;
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0) {
      // ---------------------------------------------------------------- TMA producer
      if (lane == 0) {
        const int req = a.p.layout == 1 ? 0 : g;
        const int32_t* pt = a.p.page_table + static_cast<int64_t>(req) * a.p.max_pages;
        for (int t = off; t < off + take; ++t) {
          const uint32_t i = kcount + (t - off), s = i % kStages, ph = (i / kStages) & 1;
          if (!mbar_wait(&sm.k_empty[s], ph ^ 1, abort_flag)) {
            set_abort(sm, a.p.dev_err);
            break;
          }
          const int npos = min(kTileM, glen - t * kTileM);
          const int npages = (npos + kPage - 1) / kPage;
          int pid[2] = {-1, -1};
          uint32_t bytes = 0;
          for (int j = 0; j < npages; ++j) {
            const int p = pt[t * 2 + j];
            if (p < 0 || p >= a.p.num_pages) {
              report(a.p.dev_err, kDevErrPage);
            } else {
              pid[j] = p;
              bytes += kPageValueBytes + kPage * 4;
            }
          }
          mbar_arrive_expect_tx(&sm.k_full[s], bytes);
          for (int j = 0; j < npages; ++j) {
            if (pid[j] < 0) continue;
            tma_load_3d(sm.kv[s] + j * kPageValueBytes, &tmap, 0, 0, pid[j], &sm.k_full[s]);
            bulk_load(&sm.ks[s][j * kPage], a.p.k_pool + static_cast<int64_t>(pid[j]) * kPageBytes + kPageValueBytes,
                      kPage * 4, &sm.k_full[s]);
          }
          ++issued;
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        uint64_t bdesc[4];
        uint32_t idesc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          bdesc[k] = sdesc_k128_sw128(smem_u32(sm.q) + 32 * k);
          idesc[k] = idesc_mxf8f6f4_e4m3(kTileM, geo.N, k, k);
        }
        for (int t = off; t < off + take; ++t) {
          const uint32_t i = kcount + (t - off), s = i % kStages, ph = (i / kStages) & 1;
          const uint32_t ai = acount + (t - off), acc = ai % geo.n_acc, aph = (ai / geo.n_acc) & 1;
          if (!mbar_wait(&sm.k_full[s], ph, abort_flag) || !mbar_wait(&sm.t_empty[acc], aph ^ 1, abort_flag)) {
            set_abort(sm, a.p.dev_err);
            break;
          }
          tc_fence_after();
          const uint32_t d = tbase + acc * geo.N;
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
      // ---------------------------------------------------------------- epilogue
      const int p = 32 * quad + lane;
      const int nb = (rlen + kBlock - 1) / kBlock;
      float* keys_row = row >= 0 && row < a.p.rows ? a.keys + static_cast<int64_t>(row) * a.keys_stride : nullptr;
      const uint32_t col0 = geo.R == 3 ? epi * kHeads : 0;
      for (int t = off; t < off + take; ++t) {
        const uint32_t ai = acount + (t - off);
        if (geo.R == 1 && static_cast<int>(ai % 3) != epi) continue;
        const uint32_t acc = ai % geo.n_acc, aph = (ai / geo.n_acc) & 1;
        const uint32_t i = kcount + (t - off), s = i % kStages, ph = (i / kStages) & 1;
        if (!warp_wait(&sm.t_full[acc], aph, abort_flag)) {
          if (lane == 0) set_abort(sm, a.p.dev_err);
          break;
        }
        tc_fence_after();
        float part[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        uint32_t x[32];
        const uint32_t taddr = tmem_addr(tbase, 32 * quad, acc * geo.N + col0);
        tmem_ld32(taddr, x);
        tmem_ld_wait();
        head_reduce_half(part, x, w);
        tmem_ld32(taddr + 32, x);
        tmem_ld_wait();
        head_reduce_half(part, x, w + 32);
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
        const int pos = t * kTileM + p;
        const bool valid = keys_row != nullptr && pos < rlen;
        float v = valid ? score * kscale : -__int_as_float(0x7f800000);
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        if ((lane & 7) == 0 && valid) {
          const int b = pos >> 3;
          keys_row[b] = b == nb - 1 ? __int_as_float(0x7f800000) : v;
        }
      }
    }
    kcount += take;
    acount += take;
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

cudaError_t launch_dense_amax8(const DenseArgs& a, cudaStream_t stream) {
  CUtensorMap tmap;
  cudaError_t e = make_pool_tmap(&tmap, a.p.k_pool, a.p.num_pages, kPage);
  if (e != cudaSuccess) return e;
  const int smem = static_cast<int>(sizeof(Smem)) + 1024;
  e = cudaFuncSetAttribute(dense_amax8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dense_amax8_kernel<<<device_sm_count(), kThreads, smem, stream>>>(tmap, a);
  return cudaGetLastError();
}

}  // namespace ci
