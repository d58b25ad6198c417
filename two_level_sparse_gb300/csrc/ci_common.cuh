// Device helpers shared by the scoring, publishing and selection kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace ci {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kBlock = 8;
constexpr int kPage = 64;
constexpr int kPageValueBytes = kPage * kDim;          // 8192
constexpr int kPageBytes = kPageValueBytes + kPage * 4;  // 8448
constexpr int kTileM = 128;                            // positions per MMA tile
// Index-K formats.  FP8: a page is 64 x 128 e4m3 bytes, then 64 fp32 scales.
// MXFP4: a page is 64 x 64 bytes of packed e2m1 (element 2i in the low
// nibble), then one 32-bit word per position whose byte j is the ue8m0 scale
// of elements 32j .. 32j + 31.
constexpr int kKvFp8 = 0, kKvMxfp4 = 1;
template <int KV>
__host__ __device__ constexpr int row_bytes() {  // bytes of one position's values
  return KV == kKvMxfp4 ? kDim / 2 : kDim;
}
template <int KV>
__host__ __device__ constexpr int page_value_bytes() {
  return kPage * row_bytes<KV>();
}
template <int KV>
__host__ __device__ constexpr int page_bytes() {
  return page_value_bytes<KV>() + kPage * 4;
}
constexpr uint32_t kDevErrLen = 1u, kDevErrPage = 2u, kDevErrBlock = 4u, kDevErrTimeout = 8u, kDevErrReq = 16u,
                   kDevErrPos = 32u;
constexpr int kLayoutDecode = 0, kLayoutPrefill = 1, kLayoutVarlen = 2;

__device__ __forceinline__ void report(int32_t* dev_err, uint32_t bits) {
  if (dev_err != nullptr) atomicOr(reinterpret_cast<unsigned int*>(dev_err), bits);
}

// Byte offset of (row r, byte kb) inside a K-major tile of 64-byte rows in the
// 64-byte swizzle layout (8-row atoms of 512 B; the 16-byte chunk index is
// XOR-ed with (r / 2) mod 4).
__device__ __forceinline__ uint32_t sw64_offset(uint32_t r, uint32_t kb) {
  return (r >> 3) * 512u + (r & 7u) * 64u + ((((kb >> 4) ^ ((r >> 1) & 3u)) << 4) | (kb & 15u));
}

// Byte offset of (row r, byte kb) inside a K-major tile of 128-byte rows in the
// 128-byte swizzle layout (8-row atoms of 1024 B; the 16-byte chunk index is
// XOR-ed with the row index inside the atom).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t kb) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((((kb >> 4) ^ (r & 7u)) << 4) | (kb & 15u));
}

// e2m1 code (sign bit 3) -> e4m3 byte of the same value.  Every e2m1 value
// {0, 0.5, 1, 1.5, 2, 3, 4, 6} is exact in e4m3.
__device__ __forceinline__ uint32_t e2m1_to_e4m3(uint32_t code) {
  constexpr uint64_t kMag = 0x4C4844403C383000ull;  // bytes for magnitudes 0..7
  return static_cast<uint32_t>((kMag >> ((code & 7u) * 8u)) & 0xFFu) | ((code & 8u) << 4);
}

// 8 packed MXFP4 bytes (16 codes, element 2i in the low nibble) -> 16 e4m3 bytes.
__device__ __forceinline__ uint4 widen_fp4x16(uint2 in) {
  uint32_t o[4];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t v = half ? in.y : in.x;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t b = v >> (16 * q);  // two bytes -> four codes
      o[half * 2 + q] = e2m1_to_e4m3(b & 0xF) | (e2m1_to_e4m3((b >> 4) & 0xF) << 8) |
                        (e2m1_to_e4m3((b >> 8) & 0xF) << 16) | (e2m1_to_e4m3((b >> 12) & 0xF) << 24);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Warp-uniform bounded wait: lane 0 waits (giving up on abort or timeout), the
// verdict is broadcast, and on success every lane observes the completed phase
// itself (an immediate try_wait) so that each has acquire ordering.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok) mbar_wait(bar, parity, nullptr);
  return ok;
}

// Bounded wait by lane 0 alone, the verdict broadcast and the warp
// synchronized after it (its memory ordering carries lane 0's acquire to the
// other lanes): for warps whose lanes then only write shared memory or whose
// work is issued by one elected lane, one probe per wait instead of 32.
__device__ __forceinline__ bool warp_wait_lane0(uint64_t* bar, uint32_t parity, volatile int* abort) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

// The common case first: every lane probes once and the warp votes; only when
// the phase is not complete yet does it fall back to the bounded wait.
__device__ __forceinline__ bool warp_wait_fast(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  return warp_wait(bar, parity, abort);
}

// ---------------------------------------------------------------- score epilogue
// Head-weighted ReLU reduction of one (row, position) pair from its 64 fp32
// accumulator columns, delivered in two halves of 32: eight partial sums
// (head h feeds partial h % 8), combined in a fixed tree.  Every kernel that
// scores a position uses these functions, so identical K vectors give
// bit-identical scores wherever they are scored.
//
// The partial sums live as four packed pairs (2m, 2m + 1) and the head
// weights as 32 packed pairs (w[2m], w[2m + 1]), low word first; heads 2m and
// 2m + 1 go through two ReLUs and one fma.rn.f32x2 (two IEEE round-to-nearest
// FMAs, the same results as two fmaf calls) without leaving the pair registers.
struct HeadAcc {
  unsigned long long p[4];
};
// (The ReLU is taken in place: x0, x1 are consumed.)
__device__ __forceinline__ void relu_fma_pair(unsigned long long& acc, unsigned long long w2, uint32_t& x0,
                                              uint32_t& x1) {
  asm("{\n\t.reg .b64 c;\n\t"
      "max.f32 %1, %1, 0f00000000;\n\tmax.f32 %2, %2, 0f00000000;\n\t"
      "mov.b64 c, {%1, %2};\n\tfma.rn.f32x2 %0, %3, c, %0;\n\t}"
      : "+l"(acc), "+r"(x0), "+r"(x1)
      : "l"(w2));
}
// The same with the ReLU on the FMA pipe: x + |x| = 2 ReLU(x) exactly, so
// the partial sums carry twice the values of the max form, each rounding
// scaled by two as well, and the finish halves them exactly -- the same bits
// wherever no partial sum is subnormal (|sum| < 2^-126).  Every kernel scoring
// one K format uses one form (scorer_relu_abs_add below), which keeps the
// dense keys and the sparse rescoring bit-identical in every case.
__device__ __forceinline__ void relu2_fma_pair(unsigned long long& acc, unsigned long long w2, uint32_t& x0,
                                               uint32_t& x1) {
  asm("{\n\t.reg .b64 c;\n\t.reg .f32 a0, a1;\n\t"
      "abs.f32 a0, %1;\n\tabs.f32 a1, %2;\n\t"
      "add.rn.f32 %1, %1, a0;\n\tadd.rn.f32 %2, %2, a1;\n\t"
      "mov.b64 c, {%1, %2};\n\tfma.rn.f32x2 %0, %3, c, %0;\n\t}"
      : "+l"(acc), "+r"(x0), "+r"(x1)
      : "l"(w2));
}
// ReLU form per K format: max.f32 (ALU pipe) for FP8 pools, x + |x| (FMA
// pipe) for MXFP4 pools, whose scorers are shorter of FMA work and longer of
// ALU work (the faster choice of each, by measurement).
template <int KV>
__host__ __device__ constexpr bool scorer_relu_abs_add() {
  return KV == kKvMxfp4;
}
// x: heads 32 half .. 32 half + 31 of the position; w2: their 16 weight pairs.
template <bool kAbsAdd>
__device__ __forceinline__ void head_reduce_half(HeadAcc& acc, uint32_t (&x)[32], const unsigned long long* w2) {
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    if (kAbsAdd)
      relu2_fma_pair(acc.p[m & 3], w2[m], x[2 * m], x[2 * m + 1]);
    else
      relu_fma_pair(acc.p[m & 3], w2[m], x[2 * m], x[2 * m + 1]);
  }
}
template <bool kAbsAdd>
__device__ __forceinline__ float head_reduce_finish(const HeadAcc& acc) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] = __uint_as_float(static_cast<uint32_t>(acc.p[i]));
    a[2 * i + 1] = __uint_as_float(static_cast<uint32_t>(acc.p[i] >> 32));
  }
  const float s = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
  return kAbsAdd ? 0.5f * s : s;
}
// The 64 head weights of a row (16-byte aligned) as 32 packed pairs.
__device__ __forceinline__ void load_head_weights(unsigned long long (&w2)[32], const float* w) {
  const ulonglong2* wp = reinterpret_cast<const ulonglong2*>(w);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const ulonglong2 v = wp[j];
    w2[2 * j] = v.x;
    w2[2 * j + 1] = v.y;
  }
}

// ---------------------------------------------------------------- page ids of K tiles
// The two pages (64 positions each) behind 128-position tile t of a request
// whose page table is pt, for a scan over the first len positions: -1 where
// the tile has no such position or where the id is out of range (reported).
// A producer warp loads 32 tiles' ids at once (one tile per lane) one chunk
// ahead of the tiles it issues, so no tile waits on a dependent global load.
struct TilePages {
  int lo, hi;
};
__device__ __forceinline__ TilePages load_tile_pages(const int32_t* pt, int t, int len, int64_t num_pages,
                                                     int32_t* dev_err) {
  TilePages r{-1, -1};
  const int p0 = t * kTileM;
  if (p0 < len) {
    const int a = pt[2 * t];
    const int b = p0 + kPage < len ? pt[2 * t + 1] : -1;
    if (a < 0 || a >= num_pages)
      report(dev_err, kDevErrPage);
    else
      r.lo = a;
    if (p0 + kPage < len) {
      if (b < 0 || b >= num_pages)
        report(dev_err, kDevErrPage);
      else
        r.hi = b;
    }
  }
  return r;
}

// ---------------------------------------------------------------- ordering keys
// Order-preserving map fp32 -> uint32 (larger float -> larger key); -0 maps
// like +0.  Every finite score and -inf map above 0, which marks "no entry".
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_inv(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace ci
