// The indexer's query producer: RoPE on the first 64 dims of every head,
// quantization, head-weight scaling (vLLM indexer.py page, rope_quant_q, and
// the fused_indexer_q_rope_quant kernel of sparse_attn_indexer.py).
//
// Per (token, head), from bf16 q[128]:
//   (x0, x1) pairs -- dims (i, 32 + i) in the NeoX layout, (2i, 2i + 1) in
//   the interleaved one, i < 32 -- become r0 = x0 cos - x1 sin and
//   r1 = x1 cos + x0 sin in fp32 (one rounding per operation, no contraction),
//   each rounded to bf16 and back; dims 64..127 pass unrotated.
//   MXFP4 output (the indexer's query format): per block of 32 dims the scale
//   2^ceil(log2(max(amax, 1e-10) * (1/6))) stored as its ue8m0 code, the
//   values x / scale rounded to e2m1 (nearest even, saturating), element 2i in
//   the low nibble; w_out = w * softmax_scale * head_scale.
//   FP8 output (as the pages print it): one scale per head with 448 in place
//   of 6, the values clamped to +-448 and rounded to e4m3, and the scale folded
//   into the weight: w_out = w * scale * softmax_scale * head_scale.
// ceil(log2(v)) is taken exactly from the bits of v.
//
// One warp per eight heads of a token, lane l holding dims 4l .. 4l + 3 of each.
// Memory-bound: 256 bytes in, 68 (MXFP4) or 128 (FP8) out per head.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kHeadsPerWarp = 8;  // loads of eight heads in flight per warp before any is processed

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Exact ceil(log2(max(amax, 1e-10) * (1 / vmax))).
__device__ __forceinline__ int scale_exp(float amax, float inv_vmax) {
  const uint32_t u = __float_as_uint(__fmul_rn(fmaxf(amax, 1e-10f), inv_vmax));
  return static_cast<int>((u >> 23) & 0xFFu) - 127 + ((u & 0x7FFFFFu) != 0u);
}
// 2^k from its bits, for -126 <= k <= 127 (the scale exponents here lie in
// [-33, 126]: amax is at least 1e-10 and at most the largest bf16).
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float(static_cast<uint32_t>(k + 127) << 23); }
// x * 2^-e, exact (a power-of-two scaling).
__device__ __forceinline__ float unscale(float x, int e) { return __fmul_rn(x, pow2i(-e)); }
// Two fp32 values -> one byte of e2m1 codes, `lo` in the low nibble.
__device__ __forceinline__ uint8_t e2m1_pair(float lo, float hi) {
  return static_cast<uint8_t>(__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest));
}
__device__ __forceinline__ uint8_t e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// Lane l loads dims 4l .. 4l + 3 of the head (one 8-byte load per lane, the
// head's 256 bytes per warp instruction).  Lanes 0-15 hold the rotated half:
// in the NeoX layout lane l < 8 holds x0 of pairs 4l .. 4l + 3 and lane l + 8
// their x1 (exchanged by one shuffle); in the interleaved layout lane l holds
// both elements of pairs 2l and 2l + 1.  Lanes 16-31 hold dims 64..127.  The
// 32-dim blocks are the lane octets 0-7, 8-15, 16-23, 24-31.
template <bool kFp8, bool kNeox>
__device__ __forceinline__ void qprod_head(const QProdArgs& a, int64_t gw, int lane, uint2 raw, const float (&cc)[4],
                                           const float (&ss)[4]) {
  float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u), __uint_as_float(raw.y << 16),
                __uint_as_float(raw.y & 0xFFFF0000u)};
  float v[4];  // this lane's four output dims, in order
  {
    // the partner values of the other half of each NeoX pair
    float pr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) pr[j] = __shfl_xor_sync(0xffffffffu, x[j], 8);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = x[j];
    if (lane < 16) {
      if (kNeox) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float x0 = lane < 8 ? x[j] : pr[j], x1 = lane < 8 ? pr[j] : x[j];
          v[j] = lane < 8 ? bf16_round(__fsub_rn(__fmul_rn(x0, cc[j]), __fmul_rn(x1, ss[j])))
                          : bf16_round(__fadd_rn(__fmul_rn(x1, cc[j]), __fmul_rn(x0, ss[j])));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float x0 = x[2 * j], x1 = x[2 * j + 1];
          v[2 * j] = bf16_round(__fsub_rn(__fmul_rn(x0, cc[j]), __fmul_rn(x1, ss[j])));
          v[2 * j + 1] = bf16_round(__fadd_rn(__fmul_rn(x1, cc[j]), __fmul_rn(x0, ss[j])));
        }
      }
    }
  }
  const float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  const float w = a.w[gw];
  if (kFp8) {
    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
    const int e = scale_exp(amax, 1.0f / 448.0f);
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      packed |= static_cast<uint32_t>(e4m3(fminf(fmaxf(unscale(v[j], e), -448.0f), 448.0f))) << (8 * j);
    *reinterpret_cast<uint32_t*>(a.q_out + gw * kDim + 4 * lane) = packed;
    if (lane == 0) a.w_out[gw] = __fmul_rn(__fmul_rn(__fmul_rn(w, pow2i(e)), a.softmax_scale), a.head_scale);
  } else {
    float bm = m;  // block maximum over this lane's octet
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
    const int e = scale_exp(bm, 1.0f / 6.0f);
    const uint32_t lo = e2m1_pair(unscale(v[0], e), unscale(v[1], e));
    const uint32_t hi = e2m1_pair(unscale(v[2], e), unscale(v[3], e));
    *reinterpret_cast<uint16_t*>(a.q_out + gw * (kDim / 2) + 2 * lane) = static_cast<uint16_t>(lo | (hi << 8));
    const int e1 = __shfl_sync(0xffffffffu, e, 8), e2 = __shfl_sync(0xffffffffu, e, 16),
              e3 = __shfl_sync(0xffffffffu, e, 24);
    if (lane == 0) {
      *reinterpret_cast<uint32_t*>(a.q_sf + gw * 4) =
          static_cast<uint32_t>(e + 127) | (static_cast<uint32_t>(e1 + 127) << 8) |
          (static_cast<uint32_t>(e2 + 127) << 16) | (static_cast<uint32_t>(e3 + 127) << 24);
      a.w_out[gw] = __fmul_rn(__fmul_rn(w, a.softmax_scale), a.head_scale);
    }
  }
}

// Each warp takes kHeadsPerWarp consecutive heads of one token (64 is a
// multiple), their loads issued before any is processed.
template <bool kFp8, bool kNeox>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) qprod_kernel(const QProdArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t g0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) * kHeadsPerWarp;
  if (g0 >= static_cast<int64_t>(a.tokens) * kHeads) return;
  const int t = static_cast<int>(g0 / kHeads);
  const int pos = a.positions[t];
  const bool ok = pos >= 0 && pos < a.max_pos;
  if (!ok && lane == 0 && (g0 % kHeads) == 0) report(a.dev_err, kDevErrPos);
  uint2 raw[kHeadsPerWarp];
#pragma unroll
  for (int k = 0; k < kHeadsPerWarp; ++k)
    raw[k] = ok ? *reinterpret_cast<const uint2*>(a.q + (g0 + k) * kDim + 4 * lane) : make_uint2(0, 0);
  // cos / sin of this lane's pairs (NeoX lanes 0-15: pairs 4 (l % 8) ..; interleaved
  // lanes 0-15: pairs 2l, 2l + 1), zeros for a bad position
  float cc[4] = {0.f, 0.f, 0.f, 0.f}, ss[4] = {0.f, 0.f, 0.f, 0.f};
  if (ok && lane < 16) {
    const float* cs = a.cos_sin + static_cast<int64_t>(pos) * 64;
    if (kNeox) {
      const int i0 = 4 * (lane & 7);
      const float4 c = *reinterpret_cast<const float4*>(cs + i0), sn = *reinterpret_cast<const float4*>(cs + 32 + i0);
      cc[0] = c.x, cc[1] = c.y, cc[2] = c.z, cc[3] = c.w;
      ss[0] = sn.x, ss[1] = sn.y, ss[2] = sn.z, ss[3] = sn.w;
    } else {
      const int i0 = 2 * lane;
      const float2 c = *reinterpret_cast<const float2*>(cs + i0), sn = *reinterpret_cast<const float2*>(cs + 32 + i0);
      cc[0] = c.x, cc[1] = c.y;
      ss[0] = sn.x, ss[1] = sn.y;
    }
  }
#pragma unroll
  for (int k = 0; k < kHeadsPerWarp; ++k) qprod_head<kFp8, kNeox>(a, g0 + k, lane, raw[k], cc, ss);
}

}  // namespace

cudaError_t launch_qprod(const QProdArgs& a, cudaStream_t stream) {
  if (a.tokens == 0) return cudaSuccess;
  const int64_t warps = static_cast<int64_t>(a.tokens) * kHeads / kHeadsPerWarp;
  const unsigned grid = static_cast<unsigned>((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
  const int threads = 32 * kWarpsPerBlock;
  if (a.fp8) {
    if (a.neox)
      qprod_kernel<true, true><<<grid, threads, 0, stream>>>(a);
    else
      qprod_kernel<true, false><<<grid, threads, 0, stream>>>(a);
  } else {
    if (a.neox)
      qprod_kernel<false, true><<<grid, threads, 0, stream>>>(a);
    else
      qprod_kernel<false, false><<<grid, threads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace ci
