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
// One warp per eight heads of a token, two heads at a time: half-warp hh
// takes one, and its lane m (0..15) holds dims 4m .. 4m + 3 (the rotated
// half) and 64 + 4m .. 64 + 4m + 3 (the unrotated half), so that every lane
// does the same RoPE work.  Memory-bound: 256 bytes in, 68 (MXFP4) or 128
// (FP8) out per head.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "ci_common.cuh"
#include "ci_internal.h"

namespace ci {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kHeadsPerWarp = 8;  // loads of eight heads in flight per warp before any is processed

// The biased scale exponent 127 + ceil(log2(max(amax, 1e-10) * (1 / vmax))),
// which is also the ue8m0 code of the scale.  For a positive normal float,
// adding 0x7FFFFF to its bits carries into the exponent field exactly when
// the mantissa is nonzero, so the field of the sum is the ceiling.  (The
// product lies in [2^-43, 2^126]: amax is at least 1e-10 and at most the
// largest bf16.)
__device__ __forceinline__ uint32_t scale_code(float amax, float inv_vmax) {
  return (__float_as_uint(__fmul_rn(fmaxf(amax, 1e-10f), inv_vmax)) + 0x7FFFFFu) >> 23;
}
// The scale 2^(code - 127) and its inverse, from bits (both exact).
__device__ __forceinline__ float scale_of(uint32_t code) { return __uint_as_float(code << 23); }
__device__ __forceinline__ float inv_scale_of(uint32_t code) { return __uint_as_float((254u - code) << 23); }
// Two fp32 values -> one byte of e2m1 codes, `lo` in the low nibble.
__device__ __forceinline__ uint8_t e2m1_pair(float lo, float hi) {
  return static_cast<uint8_t>(__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest));
}
__device__ __forceinline__ uint8_t e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// x c + o s with one IEEE round-to-nearest rounding per multiply and per add
// (the _rn intrinsics are never contracted into an fma).
__device__ __forceinline__ float rope1(float x, float c, float o, float sn) {
  return __fadd_rn(__fmul_rn(x, c), __fmul_rn(o, sn));
}
// Both values rounded to bf16 and back to fp32.
__device__ __forceinline__ void bf16_round2(float& a, float& b) {
  const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);  // .x <- a (low half)
  const uint32_t u = *reinterpret_cast<const uint32_t*>(&r);
  a = __uint_as_float(u << 16);
  b = __uint_as_float(u & 0xFFFF0000u);
}
__device__ __forceinline__ void unpack_bf16x4(uint2 raw, float (&x)[4]) {
  x[0] = __uint_as_float(raw.x << 16);
  x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  x[2] = __uint_as_float(raw.y << 16);
  x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
}
__device__ __forceinline__ float absmax4(const float (&v)[4]) {
  return fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
}

// One head (gw = token * 64 + head) in half-warp lane m: lo = dims 4m .. 4m + 3,
// hi = dims 64 + 4m .. 64 + 4m + 3 (bf16).  C, S: this lane's cos and signed
// sin, so that rotated value j is x[j] C[j] + partner[j] S[j] (S = -sin where
// the value is the pair's first element); the partner is the pair's other
// element: in the NeoX layout lane m ^ 8's value j, in the interleaved one
// value j ^ 1 of this lane.  The 32-dim blocks: lanes m < 8 hold blocks 0
// (lo) and 2 (hi), lanes m >= 8 blocks 1 and 3.
template <bool kFp8, bool kNeox>
__device__ __forceinline__ void qprod_head(const QProdArgs& a, int64_t gw, int m, uint2 lo, uint2 hi, float w,
                                           const float (&C)[4], const float (&S)[4]) {
  float x[4], o[4], v[4], y[4];
  unpack_bf16x4(lo, x);
  if (kNeox) {
    const uint2 pr = make_uint2(__shfl_xor_sync(0xffffffffu, lo.x, 8), __shfl_xor_sync(0xffffffffu, lo.y, 8));
    unpack_bf16x4(pr, o);
  } else {
    o[0] = x[1], o[1] = x[0], o[2] = x[3], o[3] = x[2];
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = rope1(x[j], C[j], o[j], S[j]);
  bf16_round2(v[0], v[1]);
  bf16_round2(v[2], v[3]);
  unpack_bf16x4(hi, y);
  const float ma = absmax4(v), mb = absmax4(y);
  if (kFp8) {
    float amax = fmaxf(ma, mb);  // over the head's 16 lanes
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const uint32_t code = scale_code(amax, 1.0f / 448.0f);
    const float inv = inv_scale_of(code);
    uint32_t pa = 0, pb = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      pa |= static_cast<uint32_t>(e4m3(fminf(fmaxf(__fmul_rn(v[j], inv), -448.0f), 448.0f))) << (8 * j);
      pb |= static_cast<uint32_t>(e4m3(fminf(fmaxf(__fmul_rn(y[j], inv), -448.0f), 448.0f))) << (8 * j);
    }
    *reinterpret_cast<uint32_t*>(a.q_out + gw * kDim + 4 * m) = pa;
    *reinterpret_cast<uint32_t*>(a.q_out + gw * kDim + 64 + 4 * m) = pb;
    if (m == 0) a.w_out[gw] = __fmul_rn(__fmul_rn(__fmul_rn(w, scale_of(code)), a.softmax_scale), a.head_scale);
  } else {
    // block maxima over lane octets, both blocks in one word: every value is
    // a bf16, so |max| is the upper half of its fp32 bits, and for
    // non-negative floats the bit patterns order like the values
    uint32_t pm = __byte_perm(__float_as_uint(ma), __float_as_uint(mb), 0x7632);
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) pm = __vmaxu2(pm, __shfl_xor_sync(0xffffffffu, pm, off));
    const uint32_t ka = scale_code(__uint_as_float(pm << 16), 1.0f / 6.0f);
    const uint32_t kb = scale_code(__uint_as_float(pm & 0xFFFF0000u), 1.0f / 6.0f);
    const float sa = inv_scale_of(ka), sb = inv_scale_of(kb);
    const uint32_t ca = e2m1_pair(__fmul_rn(v[0], sa), __fmul_rn(v[1], sa)) |
                        (static_cast<uint32_t>(e2m1_pair(__fmul_rn(v[2], sa), __fmul_rn(v[3], sa))) << 8);
    const uint32_t cb = e2m1_pair(__fmul_rn(y[0], sb), __fmul_rn(y[1], sb)) |
                        (static_cast<uint32_t>(e2m1_pair(__fmul_rn(y[2], sb), __fmul_rn(y[3], sb))) << 8);
    *reinterpret_cast<uint16_t*>(a.q_out + gw * (kDim / 2) + 2 * m) = static_cast<uint16_t>(ca);
    *reinterpret_cast<uint16_t*>(a.q_out + gw * (kDim / 2) + 32 + 2 * m) = static_cast<uint16_t>(cb);
    // ue8m0 codes: byte j of the head's word = block j
    const uint32_t cw = ka | (kb << 16);
    const uint32_t other = __shfl_xor_sync(0xffffffffu, cw, 8);  // blocks 1 and 3 (lane 8 of the half)
    if (m == 0) {
      *reinterpret_cast<uint32_t*>(a.q_sf + gw * 4) = cw | (other << 8);
      a.w_out[gw] = __fmul_rn(__fmul_rn(w, a.softmax_scale), a.head_scale);
    }
  }
}

// One block per token: warp wi takes heads 8 wi .. 8 wi + 7, two per step.
// Every load that does not need the token's position (the heads' values and
// weights) is issued together with the position's, before any head is
// processed; only the cos / sin loads wait for the position.
template <bool kFp8, bool kNeox>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) qprod_kernel(const QProdArgs a) {
  const int lane = threadIdx.x & 31, m = lane & 15, hh = lane >> 4;
  const int64_t g0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5)) * kHeadsPerWarp;
  if (g0 >= static_cast<int64_t>(a.tokens) * kHeads) return;
  const int t = static_cast<int>(g0 / kHeads);
  const int pos = a.positions[t];
  constexpr int kSteps = kHeadsPerWarp / 2;
  uint2 lo[kSteps], hi[kSteps];
#pragma unroll
  for (int k = 0; k < kSteps; ++k) {
    const uint16_t* src = a.q + (g0 + 2 * k + hh) * kDim + 4 * m;
    lo[k] = *reinterpret_cast<const uint2*>(src);
    hi[k] = *reinterpret_cast<const uint2*>(src + 64);
  }
  const float wl = lane < kHeadsPerWarp ? a.w[g0 + lane] : 0.f;  // lane k: the weight of head g0 + k
  const bool ok = pos >= 0 && pos < a.max_pos;
  if (!ok) {
    if (lane == 0 && (g0 % kHeads) == 0) report(a.dev_err, kDevErrPos);
#pragma unroll
    for (int k = 0; k < kSteps; ++k) lo[k] = hi[k] = make_uint2(0, 0);
  }
  // cos and signed sin of this lane's four rotated values (zeros for a bad position)
  float C[4] = {0.f, 0.f, 0.f, 0.f}, S[4] = {0.f, 0.f, 0.f, 0.f};
  if (ok) {
    const float* cs = a.cos_sin + static_cast<int64_t>(pos) * 64;
    if (kNeox) {
      // lane m < 8: first elements of pairs 4m .. 4m + 3; lane m >= 8: second elements of pairs 4(m - 8) ..
      const int i0 = 4 * (m & 7);
      const float4 c = *reinterpret_cast<const float4*>(cs + i0), sn = *reinterpret_cast<const float4*>(cs + 32 + i0);
      const float sg = m < 8 ? -1.0f : 1.0f;
      C[0] = c.x, C[1] = c.y, C[2] = c.z, C[3] = c.w;
      S[0] = sg * sn.x, S[1] = sg * sn.y, S[2] = sg * sn.z, S[3] = sg * sn.w;
    } else {
      // dims 4m .. 4m + 3 are pairs 2m and 2m + 1, first element at even dims
      const float2 c = *reinterpret_cast<const float2*>(cs + 2 * m), sn = *reinterpret_cast<const float2*>(cs + 32 + 2 * m);
      C[0] = C[1] = c.x;
      C[2] = C[3] = c.y;
      S[0] = -sn.x, S[1] = sn.x, S[2] = -sn.y, S[3] = sn.y;
    }
  }
#pragma unroll
  for (int k = 0; k < kSteps; ++k)
    qprod_head<kFp8, kNeox>(a, g0 + 2 * k + hh, m, lo[k], hi[k], __shfl_sync(0xffffffffu, wl, 2 * k + hh), C, S);
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
