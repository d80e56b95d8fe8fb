// Tensor-core (tcgen05) chunk engine for bf16 io with headdim P = 64 and dstate N = 128.
//
// The chunked SSD scan (exact-replay RFC, vLLM issue 55524, section 1), per chunk of Q tokens
// from boundary state H ([P x N] fp32), with Acum the within-chunk prefix of delta*A:
//   G^T[t,s] = C_t . B_s                                       (Gram, K = N)
//   M^T[t,s] = G^T[t,s] delta_s exp(Acum_t - Acum_s) [s<=t]    (masked, decayed)
//   Ydiag^T[t,d] = sum_s M^T[t,s] x_s[d]                        (K = s)
//   Yoff^T[t,d] = sum_n C_t[n] H[d,n]                           (K = N)
//   y[t,d] = fma(D, x_t[d], exp(Acum_t) Yoff^T[t,d] + Ydiag^T[t,d])
//   S^T[n,d] = sum_s B_s[n] (delta_s exp(Acum_last - Acum_s) x_s[d]),  H' = fma(exp(Acum_last), H, S)
//
// Every contraction runs on the tensor cores as M = 128 MMAs with bf16 operands and fp32
// accumulation.  Operands that are fp32 are split into bf16 terms: M^T as hi + lo (a single bf16
// term costs ~0.05% of output accuracy), each with its own accumulator, summed once in fp32; H as
// hi and lo stacked along N of one MMA (columns [0, 64) hi, [64, 128) lo), summed once in fp32; the
// state input as hi + mid + lo accumulated in that order (the fp32 state must match the fp64
// recurrence to 1e-5).  An MMA costs about the same for any N up to 256, so the off-diagonal
// contraction puts the tokens on M and the headdim rows (of one or two heads) on N.
//
// Bitwise identity.  Prefill, chunked prefill, replay decode, refresh and verify all build the
// same operand VALUES for a token and issue the same instruction sequence (shapes, K order, split
// order) for the tile containing it: a 128-row "t-tile" [t0, t0+TT) of a chunk, with s running over
// [0, S_ext = t0 + TT).  Rows and columns that a path does not need may hold anything finite: on
// this hardware a row's (A side) or column's (B side) MMA result does not depend on other rows or
// columns, and a product with an exact zero contributes nothing.
#pragma once

#include "ers_common.cuh"
#include "tc_common.cuh"

namespace ers {
namespace tc {

constexpr int P = 64;
constexpr int N = 128;
constexpr uint32_t kHTile = 128u * 256u;  // [H_hi; H_lo] tile: 128 rows x 128 n (two atoms of 16 KB)

struct Geom {
  int t0, TT, S_ext, nblk;
};
// t-tile tau of a chunk of size Q (Q a multiple of 16, <= 256)
__host__ __device__ __forceinline__ Geom geom(int Q, int tau) {
  Geom g;
  g.t0 = 128 * tau;
  g.TT = Q - g.t0 < 128 ? Q - g.t0 : 128;
  g.S_ext = g.t0 + g.TT;
  g.nblk = (g.S_ext + 127) / 128;
  return g;
}

// TMEM columns: [0, RG) Gram, reused for the diagonal (hi [0, 64), lo [64, 128)) and the chunk
// state; [RG, RG + 128) the off-diagonal (hi [RG, RG + 64), lo [RG + 64, RG + 128)).
__host__ __device__ __forceinline__ int tmem_rg(int S_ext) { return S_ext < 128 ? 128 : S_ext; }
__host__ __device__ __forceinline__ uint32_t tmem_cols(int Q) {
  const Geom g = geom(Q, (Q - 1) / 128);
  const int need = tmem_rg(g.S_ext) + 128;
  uint32_t c = 32;
  while ((int)c < need) c <<= 1;
  return c;
}

// ---- MMA issue sequences (one thread) -------------------------------------------------------------
// Gram: G^T[t, s] into columns [tG, tG + S_ext).  A = C tile (rows t; atoms cR rows apart, SBO cS),
// B = B tile (rows s; atoms bR rows apart).
__device__ __forceinline__ void issue_gram(uint32_t tG, uint32_t cT, uint32_t cR, uint32_t cS, uint32_t bT,
                                           uint32_t bR, int S_ext) {
  const uint32_t id = idesc_bf16(128, S_ext, false, false);
#pragma unroll
  for (int k = 0; k < N / 16; ++k) {
    const uint32_t ao = (k >> 2) * cR * 128u + (k & 3) * 32u, bo = (k >> 2) * bR * 128u + (k & 3) * 32u;
    mma(tG, sdesc(cT + ao, 16, cS), sdesc(bT + bo, 16, 1024), id, k > 0);
  }
}

// Off-diagonal: Yoff^T[t, j] into columns [tY, tY + hR), A = C tile (rows t; atoms cR rows apart,
// SBO cS), B = hR rows of [H_hi; H_lo] tiles (one head: hR = 128; two heads packed: 256), K = N.
__device__ __forceinline__ void issue_yoff(uint32_t tY, uint32_t cT, uint32_t cR, uint32_t cS, uint32_t hT,
                                           uint32_t hR) {
  const uint32_t id = idesc_bf16(128, (int)hR, false, false);
#pragma unroll
  for (int k = 0; k < N / 16; ++k) {
    const uint32_t ao = (k >> 2) * cR * 128u + (k & 3) * 32u, bo = (k >> 2) * hR * 128u + (k & 3) * 32u;
    mma(tY, sdesc(cT + ao, 16, cS), sdesc(hT + bo, 16, 1024), id, k > 0);
  }
}

// Diagonal block blk (s in [128 blk, min(S_ext, 128 blk + 128))) of ONE bf16 term: Ydiag^T[t, d] +=
// Mterm X into columns [tD, tD + 64).  The M tile holds s - 128 blk as its inner index (rows t,
// atoms mR rows apart, SBO mS); the X tile holds rows s (MN-major B, N = 64).  The hi and lo terms
// run as two such chains into two accumulators (decode may hold both in one 8-row aliased tile,
// hi at row t % 8 and lo at row (t + 4) % 8, and run a single chain).
__device__ __forceinline__ void issue_ydiag(uint32_t tD, uint32_t mT, uint32_t mR, uint32_t mS, uint32_t xT, int blk,
                                            int S_ext) {
  const uint32_t id = idesc_bf16(128, P, false, true);
  const int s0 = 128 * blk;
  const int nk = ((S_ext - s0 < 128 ? S_ext - s0 : 128)) / 16;
  for (int k = 0; k < nk; ++k) {
    const uint32_t ao = (k >> 2) * mR * 128u + (k & 3) * 32u;
    const uint32_t bo = (uint32_t)(s0 + 16 * k) * 128u;
    mma(tD, sdesc(mT + ao, 16, mS), sdesc(xT + bo, 1024, 1024), id, (blk > 0 || k > 0) ? 1u : 0u);
  }
}

// Chunk state, one K block: S^T[n, d] (+)= sum_term B^T U_term into columns [tS, tS + 64) for
// rows s in [s0, s0 + 16 nk).  A = B tile read MN-major (rows s; the two 64-wide n atoms bR rows
// apart), B = U tiles holding rows s - s0.  Canonical order for every path: K blocks of 128 rows in
// order, and within a block the hi, mid, lo terms, each over its k steps.
__device__ __forceinline__ void issue_state_block(uint32_t tS, uint32_t bT, uint32_t bR, uint32_t u0, uint32_t u1,
                                                  uint32_t u2, int s0, int nk) {
  const uint32_t id = idesc_bf16(128, P, true, true);
  for (int term = 0; term < 3; ++term) {
    const uint32_t uT = term == 0 ? u0 : (term == 1 ? u1 : u2);
    for (int k = 0; k < nk; ++k)
      mma(tS, sdesc(bT + (uint32_t)(s0 + 16 * k) * 128u, bR * 128u, 1024), sdesc(uT + (uint32_t)k * 2048u, 1024, 1024),
          id, (s0 > 0 || term > 0 || k > 0) ? 1u : 0u);
  }
}

// ---- operand builders (generic proxy writes; the caller fences before issuing) ---------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 8 fp32 values -> hi and lo bf16 chunks
__device__ __forceinline__ void split8(const float (&v)[8], uint4& hi, uint4& lo) {
  float h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
    l[i] = __fsub_rn(v[i], h[i]);
  }
  hi = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]), pack_bf16x2(h[6], h[7]));
  lo = make_uint4(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]), pack_bf16x2(l[4], l[5]), pack_bf16x2(l[6], l[7]));
}

// 4 fp32 values -> hi and lo bf16 (8 bytes each), the same operations as split8
__device__ __forceinline__ void split4(const float (&v)[4], uint2& hi, uint2& lo) {
  float h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
    l[i] = __fsub_rn(v[i], h[i]);
  }
  hi = make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
  lo = make_uint2(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]));
}

// fp32 state [64][128] -> [H_hi; H_lo] tile.  Called by all kThreads threads (blockDim.x ==
// kThreads); every thread's loads are issued before any of its splits.
__device__ __forceinline__ void state_to_tile(const float* __restrict__ H, uint8_t* tile) {
  constexpr int IT = P * (N / 8) / kThreads;
  static_assert(P * (N / 8) % kThreads == 0, "whole iterations");
  float4 a[IT], b[IT];
#pragma unroll
  for (int k = 0; k < IT; ++k) {
    const int id = threadIdx.x + k * kThreads;
    const int d = id / (N / 8), c = id % (N / 8);
    a[k] = *reinterpret_cast<const float4*>(H + d * N + 8 * c);
    b[k] = *reinterpret_cast<const float4*>(H + d * N + 8 * c + 4);
  }
#pragma unroll
  for (int k = 0; k < IT; ++k) {
    const int id = threadIdx.x + k * kThreads;
    const int d = id / (N / 8), c = id % (N / 8);
    const float v[8] = {a[k].x, a[k].y, a[k].z, a[k].w, b[k].x, b[k].y, b[k].z, b[k].w};
    uint4 hi, lo;
    split8(v, hi, lo);
    *reinterpret_cast<uint4*>(tile + sw128(128, d, 8 * c)) = hi;
    *reinterpret_cast<uint4*>(tile + sw128(128, P + d, 8 * c)) = lo;
  }
}

// bf16 read copy [64][128] -> [R; 0] tile (a single term); asynchronous (cp.async), complete after
// cp_async_wait_all (publish() waits)
__device__ __forceinline__ void readcopy_to_tile(const __nv_bfloat16* __restrict__ R, uint8_t* tile) {
  for (int id = threadIdx.x; id < P * (N / 8); id += blockDim.x) {
    const int d = id / (N / 8), c = id % (N / 8);
    cp_async16(tile + sw128(128, d, 8 * c), R + d * N + 8 * c);
    *reinterpret_cast<uint4*>(tile + sw128(128, P + d, 8 * c)) = make_uint4(0, 0, 0, 0);
  }
}

// 16-byte chunk of one token row into tile row r (atoms R rows apart); asynchronous (cp.async),
// complete after cp_async_wait_all (publish() waits)
__device__ __forceinline__ void row_to_tile(const __nv_bfloat16* __restrict__ src, uint8_t* tile, uint32_t R,
                                            uint32_t r, int chunk) {
  cp_async16(tile + sw128(R, r, 8 * chunk), src + 8 * chunk);
}
__device__ __forceinline__ void zero_tile_chunk(uint8_t* tile, uint32_t R, uint32_t r, int chunk) {
  *reinterpret_cast<uint4*>(tile + sw128(R, r, 8 * chunk)) = make_uint4(0, 0, 0, 0);
}

// U_term rows [0, nk16) for chunk rows s = s0 + r: u = w_s x_s[d]; hi = bf16(u),
// mid = bf16(u - hi), lo = bf16(u - hi - mid).  xT holds rows s (MN-major, 64 wide); rows with
// s >= nrows are written as zeros.  Threads [0, nthreads) of the block take part (default: all).
__device__ __forceinline__ void build_u_tiles(const uint8_t* xT, const float* w, int nrows, int s0, int nr,
                                              uint8_t* u0, uint8_t* u1, uint8_t* u2, int nthreads = 0) {
  const int stride = nthreads > 0 ? nthreads : (int)blockDim.x;
  for (int id = threadIdx.x; id < nr * (P / 8); id += stride) {
    const int r = id / (P / 8), c = id % (P / 8);
    const int s = s0 + r;
    uint4 h4 = make_uint4(0, 0, 0, 0), m4 = h4, l4 = h4;
    if (s < nrows) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xT + sw128(1, s, 8 * c));
      const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&xv);
      const float ws = w[s];
      float hh[8], mm[8], ll[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float u = __fmul_rn(ws, __bfloat162float(xb[i]));
        hh[i] = __bfloat162float(__float2bfloat16_rn(u));
        const float r1 = __fsub_rn(u, hh[i]);
        mm[i] = __bfloat162float(__float2bfloat16_rn(r1));
        ll[i] = __fsub_rn(r1, mm[i]);
      }
      h4 = make_uint4(pack_bf16x2(hh[0], hh[1]), pack_bf16x2(hh[2], hh[3]), pack_bf16x2(hh[4], hh[5]),
                      pack_bf16x2(hh[6], hh[7]));
      m4 = make_uint4(pack_bf16x2(mm[0], mm[1]), pack_bf16x2(mm[2], mm[3]), pack_bf16x2(mm[4], mm[5]),
                      pack_bf16x2(mm[6], mm[7]));
      l4 = make_uint4(pack_bf16x2(ll[0], ll[1]), pack_bf16x2(ll[2], ll[3]), pack_bf16x2(ll[4], ll[5]),
                      pack_bf16x2(ll[6], ll[7]));
    }
    const uint32_t off = sw128(1, r, 8 * c);
    *reinterpret_cast<uint4*>(u0 + off) = h4;
    *reinterpret_cast<uint4*>(u1 + off) = m4;
    *reinterpret_cast<uint4*>(u2 + off) = l4;
  }
}

// Row `row` (chunk row t = t0 + row) of the masked decayed Gram for block blk, NC columns
// [col0, col0 + NC) of the block, from NC Gram values g[] (TMEM columns of the same range).
// The segment decay uses the hardware exponential (__expf): its relative error (a few 1e-7 for the
// O(1) segment sums that matter, growing with |Acum_t - Acum_s| only where the decay is already
// negligible) is far below the 2^-16 resolution of the hi + lo bf16 split it feeds.
// Writes hi and lo bf16 to the M tiles at tile row `trow` (atoms mR rows apart).  Entries with
// s > t, s >= S_ext or t >= tmax are zero.  Called by every lane of a warp together (the warp's
// lanes agree on blk, col0 and S_ext): an 8-column group that is zero on every lane is stored
// without arithmetic, and one that is live on every lane skips the per-entry mask; the value of
// every entry is the same in all three cases.  delta / ahi / alo are 16-byte aligned.
template <int NC>
__device__ __forceinline__ void m_row(const float (&g)[NC], int t, int tmax, int blk, int col0, int S_ext,
                                      const float* delta, const float* ahi, const float* alo, uint8_t* mhi,
                                      uint8_t* mlo, uint32_t mR, uint32_t trow) {
  static_assert(NC % 8 == 0, "whole 16-byte chunks");
  const df at = {ahi[t], alo[t]};
  const bool row_ok = t < tmax;
#pragma unroll
  for (int c = 0; c < NC / 8; ++c) {
    const int s0 = 128 * blk + col0 + 8 * c;   // first s of the group, a multiple of 8
    uint4 hi = make_uint4(0, 0, 0, 0), lo = hi;
    if (!__all_sync(0xffffffffu, !row_ok || s0 > t || s0 >= S_ext)) {
      const bool full = __all_sync(0xffffffffu, row_ok && s0 + 7 <= t && s0 + 7 < S_ext);
      const float4 d0 = *reinterpret_cast<const float4*>(delta + s0), d1 = *reinterpret_cast<const float4*>(delta + s0 + 4);
      const float4 h0 = *reinterpret_cast<const float4*>(ahi + s0), h1 = *reinterpret_cast<const float4*>(ahi + s0 + 4);
      const float4 l0 = *reinterpret_cast<const float4*>(alo + s0), l1 = *reinterpret_cast<const float4*>(alo + s0 + 4);
      const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
      const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float m = __fmul_rn(__fmul_rn(g[8 * c + i], dv[i]), __expf(df_diff(at, df{hv[i], lv[i]})));
        v[i] = (full || (row_ok && s0 + i <= t && s0 + i < S_ext)) ? m : 0.f;
      }
      split8(v, hi, lo);
    }
    const uint32_t off = sw128(mR, trow, col0 + 8 * c);
    *reinterpret_cast<uint4*>(mhi + off) = hi;
    *reinterpret_cast<uint4*>(mlo + off) = lo;
  }
}

}  // namespace tc
}  // namespace ers
