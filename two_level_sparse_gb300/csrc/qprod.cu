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
// One warp per (token, head): lane l holds the rotated pair i = l and dims
// 64 + l, 96 + l.  Memory-bound: 256 bytes in, 68 (MXFP4) or 128 (FP8) out
// per head.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ float warp_absmax(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
}
__device__ __forceinline__ float half_absmax(float v) {  // over the 16 lanes of this half-warp
  float m = fabsf(v);
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}
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

template <bool kFp8, bool kNeox>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) qprod_kernel(const QProdArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (gw >= static_cast<int64_t>(a.tokens) * kHeads) return;
  const int t = static_cast<int>(gw / kHeads);
  const int pos = a.positions[t];
  const bool ok = pos >= 0 && pos < a.max_pos;
  if (!ok && lane == 0 && (gw % kHeads) == 0) report(a.dev_err, kDevErrPos);
  const uint16_t* q = a.q + gw * kDim;
  auto ld = [&](int d) { return ok ? __uint_as_float(static_cast<uint32_t>(q[d]) << 16) : 0.0f; };
  const float c = ok ? a.cos_sin[static_cast<int64_t>(pos) * 64 + lane] : 0.0f;
  const float s = ok ? a.cos_sin[static_cast<int64_t>(pos) * 64 + 32 + lane] : 0.0f;
  const float x0 = kNeox ? ld(lane) : ld(2 * lane), x1 = kNeox ? ld(32 + lane) : ld(2 * lane + 1);
  const float r0 = bf16_round(__fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s)));
  const float r1 = bf16_round(__fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s)));
  const float n0 = ld(64 + lane), n1 = ld(96 + lane);
  const float w = a.w[gw];
  if (kFp8) {
    const float amax = warp_absmax(fmaxf(fmaxf(fabsf(r0), fabsf(r1)), fmaxf(fabsf(n0), fabsf(n1))));
    const int e = scale_exp(amax, 1.0f / 448.0f);
    auto q8 = [&](float x) { return e4m3(fminf(fmaxf(unscale(x, e), -448.0f), 448.0f)); };
    uint8_t* o = a.q_out + gw * kDim;
    o[kNeox ? lane : 2 * lane] = q8(r0);
    o[kNeox ? 32 + lane : 2 * lane + 1] = q8(r1);
    o[64 + lane] = q8(n0);
    o[96 + lane] = q8(n1);
    if (lane == 0)
      a.w_out[gw] = __fmul_rn(__fmul_rn(__fmul_rn(w, pow2i(e)), a.softmax_scale), a.head_scale);
  } else {
    // blocks of 32 dims: NeoX r0 | r1 | n0 | n1 across the lanes; interleaved
    // (r0, r1) of lanes 0-15 | of lanes 16-31 | n0 | n1
    float m01a, m01b;
    if (kNeox) {
      m01a = warp_absmax(r0);
      m01b = warp_absmax(r1);
    } else {
      const float m = half_absmax(fmaxf(fabsf(r0), fabsf(r1)));
      m01a = __shfl_sync(0xffffffffu, m, 0);
      m01b = __shfl_sync(0xffffffffu, m, 16);
    }
    const int e0 = scale_exp(m01a, 1.0f / 6.0f), e1 = scale_exp(m01b, 1.0f / 6.0f);
    const int e2 = scale_exp(warp_absmax(n0), 1.0f / 6.0f), e3 = scale_exp(warp_absmax(n1), 1.0f / 6.0f);
    uint8_t* o = a.q_out + gw * (kDim / 2);
    // a byte holds dims (2m, 2m + 1): the pair of neighbouring lanes, written by the even lane
    auto put_pair = [&](float v, int e, int byte0) {
      const float y = unscale(v, e);
      const float yn = __shfl_xor_sync(0xffffffffu, y, 1);
      if ((lane & 1) == 0) o[byte0 + (lane >> 1)] = e2m1_pair(y, yn);
    };
    if (kNeox) {
      put_pair(r0, e0, 0);
      put_pair(r1, e1, 16);
    } else {
      const int e = lane < 16 ? e0 : e1;
      o[lane] = e2m1_pair(unscale(r0, e), unscale(r1, e));
    }
    put_pair(n0, e2, 32);
    put_pair(n1, e3, 48);
    if (lane == 0) {
      *reinterpret_cast<uint32_t*>(a.q_sf + gw * 4) =
          static_cast<uint32_t>(e0 + 127) | (static_cast<uint32_t>(e1 + 127) << 8) |
          (static_cast<uint32_t>(e2 + 127) << 16) | (static_cast<uint32_t>(e3 + 127) << 24);
      a.w_out[gw] = __fmul_rn(__fmul_rn(w, a.softmax_scale), a.head_scale);
    }
  }
}

}  // namespace

cudaError_t launch_qprod(const QProdArgs& a, cudaStream_t stream) {
  if (a.tokens == 0) return cudaSuccess;
  const int64_t warps = static_cast<int64_t>(a.tokens) * kHeads;
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
