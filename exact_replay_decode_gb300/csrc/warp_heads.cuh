// Warp-per-head building blocks of the bandwidth-shaped decode and verify kernels (CUDA-core
// engine, dstate N = 128).  A warp owns one head; lane j holds elements [4j, 4j+4) of every state
// row, the lane split of Dot<128> (ers_common.cuh), so every row dot product is a per-lane fmaf
// chain over 4 elements followed by the xor-16,8,4,2,1 butterfly, evaluated here as a
// reduce-scatter that keeps each row's pairings (and therefore its bits).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "ers_common.cuh"
#include "tc_common.cuh"

namespace ers {
namespace wh {

constexpr int kHeadsPerCta = kThreads / 32;

// Read-once state streams: 16 (fp32) or 8 (bf16) bytes per lane, through the read-only path
// without L1 allocation and with a 256-byte L2 fetch (a warp's row is 512 or 256 contiguous
// bytes).  Only for memory that no thread writes during the kernel before reading it this way.
template <typename HT> struct Quad;
template <> struct Quad<float> {
  using raw = float4;
  __device__ __forceinline__ static raw ld_stream(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
  }
  __device__ __forceinline__ static void unpack(raw u, float (&v)[4]) {
    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
  }
};
template <> struct Quad<uint8_t> {   // FP8 e4m3 read copy: a lane's 4 codes (dequantised with the row scale)
  using raw = uint32_t;
  __device__ __forceinline__ static raw ld_stream(const uint8_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
  }
};
template <> struct Quad<__nv_bfloat16> {
  using raw = uint2;
  __device__ __forceinline__ static raw ld_stream(const __nv_bfloat16* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
  }
  __device__ __forceinline__ static void unpack(raw u, float (&v)[4]) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
    v[0] = __low2float(a); v[1] = __high2float(a); v[2] = __low2float(b); v[3] = __high2float(b);
  }
};

// four consecutive io elements from shared memory, widened
__device__ __forceinline__ void lds4(const float* p, float (&v)[4]) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
}
__device__ __forceinline__ void lds4(const __nv_bfloat16* p, float (&v)[4]) {
  Quad<__nv_bfloat16>::unpack(*reinterpret_cast<const uint2*>(p), v);
}

// Paired fp32 arithmetic (one instruction for two IEEE round-to-nearest operations; per element the
// result is that of the scalar operation).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void up2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ void fma2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// A 4-row x 4-column block of fold accumulators (lane j: columns 4j..4j+3), rows paired:
// add(w, b) is acc[r][e] = fma(w[r], b[e], acc[r][e]) for every r, e, as 8 paired fmas.
struct Fold4 {
  uint64_t a[2][4];   // a[p][e] = (acc[2p][e], acc[2p + 1][e])
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int e = 0; e < 4; ++e) a[p][e] = 0ull;
  }
  __device__ __forceinline__ void add(float4 w, const float (&b)[4]) {
    const uint64_t w01 = pk2(w.x, w.y), w23 = pk2(w.z, w.w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint64_t b2 = pk2(b[e], b[e]);
      fma2(a[0][e], w01, b2);
      fma2(a[1][e], w23, b2);
    }
  }
  __device__ __forceinline__ float get(int r, int e) const {
    float lo, hi;
    up2(a[r >> 1][e], lo, hi);
    return (r & 1) ? hi : lo;
  }
};

// Reduce-scatter of 32 partials v[0..31] (row r of the 32 in v[r]) with the pairings of
// Dot<128>'s butterfly: each stage keeps the half of the rows whose index bit matches the lane's,
// so lane j returns row j's reduction, bit-identical to Dot<128>::reduce of that row (same tree;
// fp32 addition is commutative) at one shuffle per row instead of five.
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int j) {
#pragma unroll
  for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
    const bool up = (j & o) != 0;
#pragma unroll
    for (int r = 0; r < n / 2; ++r) {
      const float keep = up ? v[r + n / 2] : v[r];
      const float send = up ? v[r] : v[r + n / 2];
      v[r] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, o));
    }
  }
  return v[0];
}

// Reduce-scatter of 16 rows' lane partials v[0..15] with the pairings of Dot<128>'s butterfly
// (xor 16, 8, 4, 2, then 1 on the single remaining row): lane j returns row (j >> 1)'s reduction,
// bit-identical to Dot<128>::reduce of that row (same tree; fp32 addition is commutative).
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int j) {
#pragma unroll
  for (int o = 16, n = 16; o >= 2; o >>= 1, n >>= 1) {
    const bool up = (j & o) != 0;
#pragma unroll
    for (int r = 0; r < n / 2; ++r) {
      const float keep = up ? v[r + n / 2] : v[r];
      const float send = up ? v[r] : v[r + n / 2];
      v[r] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, o));
    }
  }
  return __fadd_rn(v[0], __shfl_xor_sync(kFull, v[0], 1));
}

using tc::cp_async16;
using tc::cp_async_wait_all;


// Inclusive double-float prefix over the lanes (lane s holds row s): the warp form of chunk_scan.
// For rows < 32 the strides >= 32 of chunk_scan leave every value unchanged, so the bits are
// chunk_scan's.
__device__ __forceinline__ df warp_scan_df(df v, int j) {
#pragma unroll
  for (int st = 1; st < 32; st <<= 1) {
    const float ph = __shfl_up_sync(kFull, v.hi, st), pl = __shfl_up_sync(kFull, v.lo, st);
    if (j >= st) v = df_add(df{ph, pl}, v);
  }
  return v;
}

// ---- FP8 e4m3 read copy with one power-of-two scale per state row --------------------------------
// Row d of a head is held by the warp, lane j owning elements [4j, 4j+4).  The row scale is s = 2^k,
// k the smallest integer with amax_n |S[d][n]| <= 448 * 2^k (no code saturates), at least -127;
// q[n] = RNE(S[d][n] / s) in e4m3 (an exact scaling, then one rounding); the value is q[n] * s.
// Lane j's 4 codes form one 32-bit word, element 4j in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {   // two codes, lo in the low byte
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantises the warp's row (lane quad v); returns lane j's 4 codes, the row scale in *scale.
__device__ __forceinline__ uint32_t fp8_quant_row(const float (&v)[4], float* scale) {
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  // m = (1 + f) 2^(E - 127) for a normal m; 448 = 1.75 * 2^8, so k = E - 135 + (f > 0.75), i.e. the
  // mantissa field above 0x600000; zero and subnormal maxima take k = -127
  const uint32_t b = __float_as_uint(m);
  const int E = (int)(b >> 23);
  const int k = E == 0 ? -127 : max(E - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0), -127);
  *scale = k == -127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(k + 127) << 23);
  const float inv = __uint_as_float((uint32_t)(127 - k) << 23);   // 2^-k, a normal float for k >= -127
  return e4m3x2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)) |
         (e4m3x2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)) << 16);
}

// Lane quad of an FP8 row as code values q (exact in fp32).  Output streams apply the row scale to
// the row's dot product instead of to each element: (sum_n q[n] C[n]) * s.
__device__ __forceinline__ void fp8_codes(uint32_t w, float (&v)[4]) {
  uint32_t h01, h23;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((uint16_t)(w & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((uint16_t)(w >> 16)));
  const __half2 a = *reinterpret_cast<const __half2*>(&h01);
  const __half2 b = *reinterpret_cast<const __half2*>(&h23);
  v[0] = __low2float(a);
  v[1] = __high2float(a);
  v[2] = __low2float(b);
  v[3] = __high2float(b);
}

// Writes row d (lane quad v) of an FP8 copy: codes to R8 + d*N + 4j, scale to Rs[d].
template <int N>
__device__ __forceinline__ void fp8_store_row(const float (&v)[4], uint8_t* R8, float* Rs, int d, int j) {
  float s;
  const uint32_t w = fp8_quant_row(v, &s);
  *reinterpret_cast<uint32_t*>(R8 + (size_t)d * N + 4 * j) = w;
  if (j == 0) Rs[d] = s;
}

// ---- NVFP4 read copy: e2m1 codes, an e4m3 scale per 16 values, a power-of-two scale per row -------
// Row d of a head: codes at C4 + d*N/2 (lane j's 4 codes in the 16 bits at byte 2j, element 4j+e in
// bits 4e..4e+3), block scales at Bs + d*N/16 (block b = values [16b, 16b+16), lanes 4b..4b+3),
// row scale Rs[d] = 2^k, k the smallest integer with amax <= 2688 * 2^k (448 * 6: no block scale
// saturates), at least -127.  With u = v / 2^k (exact): beta = e4m3(amax_b(|u|) / 6) (fp32 division),
// q = e2m1(u * rcp(beta)) (fp32 reciprocal and product; q = 0 where beta = 0); value q * beta * 2^k.
struct Nvfp4 {};   // tag type of the NVFP4 read copy

// A lane's view of one NVFP4 row: its 16 code bits and its block's scale byte in bits 16..23.
__device__ __forceinline__ uint32_t nvfp4_ld(const uint8_t* C4row, const uint8_t* Bsrow, int j) {
  uint16_t c;
  uint16_t b;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(c) : "l"(C4row + 2 * j));
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(b) : "l"(Bsrow + (j >> 2)));
  return (uint32_t)c | ((uint32_t)(b & 0xFFu) << 16);
}

// e2m1 values of the 4 codes of w (exact in fp32) and the block scale beta.
__device__ __forceinline__ void nvfp4_codes(uint32_t w, float (&v)[4], float* beta) {
  uint32_t h01, h23, hb;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h01) : "r"(w & 0xFFu));
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h23) : "r"((w >> 8) & 0xFFu));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hb) : "h"((uint16_t)((w >> 16) & 0xFFu)));
  const __half2 a = *reinterpret_cast<const __half2*>(&h01);
  const __half2 b = *reinterpret_cast<const __half2*>(&h23);
  v[0] = __low2float(a);
  v[1] = __high2float(a);
  v[2] = __low2float(b);
  v[3] = __high2float(b);
  *beta = __low2float(*reinterpret_cast<const __half2*>(&hb));
}

__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {   // two codes, lo in the low nibble
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Stochastic rounding of x to the e2m1 grid with the random word r: with lo the largest e2m1
// magnitude <= |x| and step the spacing above it (0.5 below 2, 1 below 4, 2 below 6), |x| goes up to
// lo + step iff r < 2^32 (|x| - lo) / step, else down to lo; |x| >= 6 gives 6; the sign is kept.
// From the fp32 fields of |x| (m its bits without the sign): at or above 1 the step is the top
// mantissa bit, so frac * 2^32 = (m & 0x3FFFFF) * 2^10 and r < that iff (r >> 10) < (m & 0x3FFFFF);
// in [0.5, 1) lo = 0.5 and frac * 2^32 = (m & 0x7FFFFF) * 2^9; below 0.5 lo = 0 and frac * 2^32 =
// |x| * 2^33 (exact, below 2^32), which r must be below the ceiling of.
__device__ __forceinline__ float sr_e2m1(float x, uint32_t r) {
  const uint32_t b = __float_as_uint(x), sign = b & 0x80000000u, m = b & 0x7FFFFFFFu;
  uint32_t q;
  if (m >= 0x40C00000u) {                 // |x| >= 6 (and NaN): 6
    q = 0x40C00000u;
  } else if (m >= 0x3F800000u) {          // [1, 6): lo has the top mantissa bit; the sum is a grid value
    q = (m & ~0x3FFFFFu) + ((r >> 10) < (m & 0x3FFFFFu) ? 0x400000u : 0u);
  } else if (m >= 0x3F000000u) {          // [0.5, 1): 0.5 or 1
    q = (r >> 9) < (m & 0x7FFFFFu) ? 0x3F800000u : 0x3F000000u;
  } else {                                // [0, 0.5): 0 or 0.5
    q = r < __float2uint_ru(__fmul_rn(__uint_as_float(m), 8589934592.f)) ? 0x3F000000u : 0u;
  }
  return __uint_as_float(sign | q);
}

// Quantises the warp's row (lane quad v): returns lane j's 16 code bits; the block scale byte, its
// value and the row scale in *bs, *beta, *scale.  kSR: the codes round stochastically (sr_e2m1 with
// the words of rw, word e for value 4j + e) instead of to nearest; the scales are the same.
template <bool kSR = false>
__device__ __forceinline__ uint32_t nvfp4_quant_row(const float (&v)[4], int j, uint32_t* bs, float* beta,
                                                    float* scale, uint4 rw = make_uint4(0u, 0u, 0u, 0u)) {
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  float mb = m;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  // 2688 = 1.3125 * 2^11: k = E - 138 + (mantissa field > 0x280000) for a normal maximum
  const uint32_t b = __float_as_uint(m);
  const int E = (int)(b >> 23);
  const int k = E == 0 ? -127 : max(E - 138 + ((b & 0x7FFFFFu) > 0x280000u ? 1 : 0), -127);
  *scale = k == -127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(k + 127) << 23);
  const float inv = __uint_as_float((uint32_t)(127 - k) << 23);
  float u[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) u[e] = __fmul_rn(v[e], inv);
  mb = __fmul_rn(mb, inv);   // |u| max of the lane (a power-of-two scaling commutes with max)
  mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 1));
  mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 2));
  const uint32_t bcode = e4m3x2(__fdiv_rn(mb, 6.f), 0.f) & 0xFFu;
  uint32_t hb;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hb) : "h"((uint16_t)bcode));
  const float bv = __low2float(*reinterpret_cast<const __half2*>(&hb));
  *bs = bcode;
  *beta = bv;
  if (bv == 0.f) return 0u;
  const float rho = __frcp_rn(bv);
  float x[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = __fmul_rn(u[e], rho);
  if constexpr (kSR) {
    x[0] = sr_e2m1(x[0], rw.x);
    x[1] = sr_e2m1(x[1], rw.y);
    x[2] = sr_e2m1(x[2], rw.z);
    x[3] = sr_e2m1(x[3], rw.w);
  }
  return e2m1x2(x[0], x[1]) | (e2m1x2(x[2], x[3]) << 8);
}

// Writes row d (lane quad v) of an NVFP4 copy; returns the code values (rv) and the block scale
// (*beta) that a dot product reads, and the row scale in *scale.
template <int N, bool kSR = false>
__device__ __forceinline__ void nvfp4_store_row(const float (&v)[4], uint8_t* C4, uint8_t* Bs, float* Rs, int d,
                                                int j, float (&rv)[4], float* beta, float* scale,
                                                uint4 rw = make_uint4(0u, 0u, 0u, 0u)) {
  uint32_t bs;
  const uint32_t c = nvfp4_quant_row<kSR>(v, j, &bs, beta, scale, rw);
  *reinterpret_cast<uint16_t*>(C4 + (size_t)d * (N / 2) + 2 * j) = (uint16_t)c;
  if ((j & 3) == 0) Bs[(size_t)d * (N / 16) + (j >> 2)] = (uint8_t)bs;
  if (j == 0) Rs[d] = *scale;
  float bb;
  nvfp4_codes(c | (bs << 16), rv, &bb);
}

// ---- fp16 anchors written by stochastic rounding (ReplaySSM "FP16+SR" recurrence) --------------------
// Random words: Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC 2011)
// at counter (nonce, slot, h * P + d, j) with the caller's 64-bit key; word e serves value 4j + e of
// row d.  Rounding: |v| goes up to the next fp16 value iff r < 2^32 (|v| - lo) / ulp, lo = |v|
// rounded toward zero on the fp16 grid, ulp its spacing (2^-24 below 2^-14); the sign is kept;
// magnitudes >= 65504 give 65504.
struct SrCtr {
  uint32_t k0, k1, nonce, slot;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int rnd = 0; rnd < 10; ++rnd) {
    if (rnd) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

__device__ __forceinline__ uint16_t sr_fp16_bits(float v, uint32_t r) {
  const uint32_t b = __float_as_uint(v);
  const uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
  const uint32_t m = b & 0x7FFFFFFFu;
  if (m >= 0x38800000u && m < 0x477FE000u) {
    // fp16 normal range [2^-14, 65504): the step is 2^13 fp32 mantissa units, so frac * 2^32 =
    // (m & 0x1FFF) * 2^19 and r < frac * 2^32 iff (r >> 19) < (m & 0x1FFF); the result is exact in fp16
    const uint32_t q = (m & ~0x1FFFu) + ((r >> 19) < (m & 0x1FFFu) ? 0x2000u : 0u);
    return sign | __half_as_ushort(__float2half_rn(__uint_as_float(q)));
  }
  const float a = __uint_as_float(m);
  if (!(a < 65504.f)) return sign | 0x7BFFu;   // saturate (65504)
  if (a == 0.f) return sign;
  const int e = (int)((b >> 23) & 0xFFu) - 127;   // floor(log2 a) for a normal a; fp32-subnormal a: -127
  const int ue = max(e, -14) - 10;                // log2 of the fp16 spacing at a
  const float t = __fmul_rn(a, __uint_as_float((uint32_t)(127 - ue) << 23));   // a / 2^ue, exact
  const float fl = floorf(t);
  const float x = __fmul_rn(__fsub_rn(t, fl), 4294967296.f);                   // frac * 2^32, exact
  const bool up = (unsigned long long)r < (unsigned long long)ceilf(x);
  const float q = __fmul_rn(__fadd_rn(fl, up ? 1.f : 0.f), __uint_as_float((uint32_t)(127 + ue) << 23));
  return sign | __half_as_ushort(__float2half_rn(q));   // q is on the fp16 grid: the conversion is exact
}

// ---- a shared NVFP4 state (ReplaySSM "Paper-reported results": the shared-FP4 recurrence mode) ------
// The NVFP4 read copy is the only state: a refresh folds from its values (code * (beta * s) in fp32)
// and writes it back with the NVFP4 cast, its codes rounded by sr_e2m1 with the words of counter
// (nonce, slot, h * P + d, j).  The rows are read with coherent loads: the same launch rewrites them.
struct Nvfp4Shared {};   // anchor tag: the anchor is the NVFP4 read copy itself

template <int N>
__device__ __forceinline__ float4 nvfp4_shared_ld(const uint8_t* C4, const uint8_t* Bs, const float* Rs, int d, int j) {
  const uint32_t c = *reinterpret_cast<const uint16_t*>(C4 + (size_t)d * (N / 2) + 2 * j);
  const uint32_t b = Bs[(size_t)d * (N / 16) + (j >> 2)];
  float q[4], beta;
  nvfp4_codes(c | (b << 16), q, &beta);
  const float bs = __fmul_rn(beta, Rs[d]);
  return make_float4(__fmul_rn(q[0], bs), __fmul_rn(q[1], bs), __fmul_rn(q[2], bs), __fmul_rn(q[3], bs));
}

// One lane's 4 anchor values of row d (offset o = d * N + 4j): fp32, or fp16 read exactly.
template <typename AT>
__device__ __forceinline__ float4 anchor_ld(const AT* H, size_t o) {
  if constexpr (std::is_same<AT, __half>::value) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(H + o));
    const __half2 a = *reinterpret_cast<const __half2*>(&u.x), b = *reinterpret_cast<const __half2*>(&u.y);
    return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
  } else {
    return __ldcs(reinterpret_cast<const float4*>(H + o));
  }
}

// Stores them: fp32 as is, fp16 by stochastic rounding with the words of counter (row, j).
template <typename AT>
__device__ __forceinline__ void anchor_st(AT* H, size_t o, const float (&v)[4], const SrCtr& sr, uint32_t row, int j) {
  if constexpr (std::is_same<AT, Nvfp4Shared>::value) {
    // nothing: the state is written by the copy's cast
  } else if constexpr (std::is_same<AT, __half>::value) {
    const uint4 r = philox4x32_10(make_uint4(sr.nonce, sr.slot, row, (uint32_t)j), sr.k0, sr.k1);
    uint2 u;
    u.x = (uint32_t)sr_fp16_bits(v[0], r.x) | ((uint32_t)sr_fp16_bits(v[1], r.y) << 16);
    u.y = (uint32_t)sr_fp16_bits(v[2], r.z) | ((uint32_t)sr_fp16_bits(v[3], r.w) << 16);
    *reinterpret_cast<uint2*>(H + o) = u;
  } else {
    *reinterpret_cast<float4*>(H + o) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// Row d of the anchor as the fold reads it: fp32, fp16, or the shared NVFP4 state (R, Rb, Rs).
template <typename AT, int N>
__device__ __forceinline__ float4 anchor_row(const AT* Hd, const void* R, const uint8_t* Rb, const float* Rs, int d,
                                             int j) {
  if constexpr (std::is_same<AT, Nvfp4Shared>::value) {
    return nvfp4_shared_ld<N>((const uint8_t*)R, Rb, Rs, d, j);
  } else {
    return anchor_ld<AT>(Hd, (size_t)d * N + 4 * j);
  }
}

// The random words of a shared NVFP4 row write (zeros for the other anchors, which do not use them).
template <typename AT>
__device__ __forceinline__ uint4 copy_words(const SrCtr& sr, uint32_t row, int j) {
  if constexpr (std::is_same<AT, Nvfp4Shared>::value) {
    return philox4x32_10(make_uint4(sr.nonce, sr.slot, row, (uint32_t)j), sr.k0, sr.k1);
  } else {
    return make_uint4(0u, 0u, 0u, 0u);
  }
}

// A head's anchor rows at element offset soff of the state (none for the shared NVFP4 state).
template <typename AT>
__device__ __forceinline__ AT* anchor_ptr(const LaunchArgs& a, size_t soff) {
  if constexpr (std::is_same<AT, Nvfp4Shared>::value) {
    return nullptr;
  } else {
    return reinterpret_cast<AT*>(a.state) + soff;
  }
}

// ---- how the output streams read one row of their source -------------------------------------------
// fp32 checkpoint, bf16 or FP8 read copy (lane j: elements [4j, 4j+4) of row d), or NVFP4 read copy.
template <typename HT> struct RawOf { using type = typename Quad<HT>::raw; };
template <> struct RawOf<Nvfp4> { using type = uint32_t; };

template <typename HT> constexpr bool kRowScale = std::is_same<HT, uint8_t>::value || std::is_same<HT, Nvfp4>::value;
template <typename HT> constexpr bool kLaneScale = std::is_same<HT, Nvfp4>::value;

template <typename HT, int N> struct RowSrc {
  const HT* p;
  __device__ __forceinline__ typename RawOf<HT>::type ld(int d, int j) const {
    return Quad<HT>::ld_stream(p + (size_t)d * N + 4 * j);
  }
};
template <int N> struct RowSrc<Nvfp4, N> {
  const uint8_t* c4;
  const uint8_t* bs;
  __device__ __forceinline__ uint32_t ld(int d, int j) const {
    return nvfp4_ld(c4 + (size_t)d * (N / 2), bs + (size_t)d * (N / 16), j);
  }
};

// The 4 values a lane multiplies with C (fp32 or bf16 values, FP8 or e2m1 codes) and, for NVFP4,
// the factor of the lane's partial dot product (its block scale).  Row scales apply after the
// row's reduction.
template <typename HT>
__device__ __forceinline__ void row_values(typename RawOf<HT>::type r, float (&h)[4], float* lane_scale) {
  if constexpr (std::is_same<HT, Nvfp4>::value) {
    nvfp4_codes(r, h, lane_scale);
  } else if constexpr (std::is_same<HT, uint8_t>::value) {
    fp8_codes(r, h);
  } else {
    Quad<HT>::unpack(r, h);
  }
}

// A head's NVFP4 copy staged in shared memory (P N / 2 code bytes, then P N / 16 block-scale bytes),
// read row by row with the global reader's word layout (RowSrc<Nvfp4, N>::ld).
template <int P, int N>
constexpr size_t staged_bytes() { return (size_t)P * N / 2 + (size_t)P * N / 16; }

template <typename HT, int N> struct RowSmem;
template <int N> struct RowSmem<Nvfp4, N> {     // e2m1 codes (row d at c4 + d N / 2), block scales after them
  const uint8_t* c4;
  const uint8_t* bs;
  __device__ __forceinline__ uint32_t ld(int d, int j) const {
    const uint32_t c = *reinterpret_cast<const uint16_t*>(c4 + (size_t)d * (N / 2) + 2 * j);
    return c | ((uint32_t)bs[(size_t)d * (N / 16) + (j >> 2)] << 16);
  }
};

template <typename K>
cudaError_t prep(K kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// Programmatic dependent launch, device side: the first launch of a split call lets its dependent
// start once every CTA has read its position; the dependent's last CTA waits for the first launch.
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ bool last_cta_of_grid() {
  return blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 && blockIdx.z == gridDim.z - 1;
}

// A split call (kPartFlushes, then kPartPlain as its programmatic dependent) of kernel(LaunchArgs).
template <typename K>
cudaError_t launch_parts(K kernel, dim3 grid, int threads, size_t smem, cudaStream_t s, LaunchArgs a) {
  a.part = kPartFlushes;
  kernel<<<grid, threads, smem, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  a.part = kPartPlain;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace wh
}  // namespace ers
