// Output-only speculative verify, refresh and commit for a gated-delta-rule (GDN) layer (ReplaySSM
// notes, "Core equations": the GDN residuals u_j solve the triangular system
//     u_j + sum_{i<j} beta_j gamma_{i+1:j} (k_i . k_j) u_i = beta_j (v_j - gamma_j S_ckpt k_j),
// the state after h committed records is S_h = gamma_h S_ckpt + sum_j gamma_{j+1:h} u_j k_j^T, and a
// draft's output is o_s = S_{h+s} q_s written in the same terms; "Data protocol and entry point": an empty
// committed history leaves the anchor unchanged and never runs an empty solve).
//
// Per (sequence, value head) the cache keeps an fp32 anchor S [dv, dk], a bf16 read copy cast from
// it, and the committed records since the last refresh: k (per key group), v, the log-gate g and
// beta, and the residual u_j that the verify that first saw the record computed from the read copy.
// With those cached, a verify streams the read copy once, computing for each of its T drafts
// S_read k_s and S_read q_s (bf16 io: one tensor-core MMA chain per head; fp32 io: CUDA-core
// reduce-scatters); the residuals and outputs then need only scalars per row.  A flush
// (h + T > L) folds the committed records into the anchor: one pass over the anchor rows computes
// S k_i, solves the residuals and folds them, row by row, and casts the read copy from the same
// fp32 values.  Fixed orders everywhere: gates are summed from the checkpoint in row order
// (Gc[t] = g_0 + ... + g_t), gamma_{a..b} = exp(Gc[b] - Gc[a-1]), dot products are Dot<128>, the
// residual and output sums run in row order.  The same rows give the same bits whether they are
// drafts of one verify or tokens of T = 1 verifies, and a refresh gives the bits of the flush that
// a verify would run.
#include <stddef.h>
#include <stdint.h>

#include "ers_common.cuh"
#include "ers_internal.h"
#include "warp_heads.cuh"

namespace ers {
namespace {

using namespace wh;
using tc::bulk_g2s;
using tc::sw128;
using tc::fence_mbar_init;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;

constexpr int kGD = 128;                       // dk = dv
constexpr int kGWarps = kThreads / 32;         // 8
constexpr int kGRows = kGD / kGWarps;          // state rows per warp
constexpr int kGL = 32;                        // max window L
constexpr int kGT = 8;                         // max drafts T
constexpr int kYS = kGD + 8;                   // padded row of the y / z tables (8 banks apart)

// What only a flushing CTA uses; a CTA without a flush keeps a head's read copy in the same bytes.
// LM is the largest window the layout holds.
template <int LM>
struct GdnFlushT {
  static constexpr int kHead = LM * kGD + LM * LM + kGWarps * kGRows * (LM + 1);
  static constexpr int kPad = kGD * kGD / 2 - kHead;   // floats up to the read copy's bytes
  float vc[LM][kGD];         // committed v (per head)
  float cf[LM][LM];          // beta_r gamma_{i+1..r} (k_i . k_r), i < r (per head)
  float yu[kGWarps][kGRows][LM + 1];   // per warp and row, S k_i then the residual u_i (per head)
  float pad[kPad > 0 ? kPad : 4];
  float kkf[LM][LM];         // k_i . k_r, committed rows (per group: past the read-copy tile's bytes)
};

// Every row array starts on a 16-byte boundary (lane quads are read as 16-byte vectors).  LM and TM
// are the largest window and draft count the layout holds: 32 and 8 in general, 16 and 4 in a
// layout small enough for three CTAs per SM.
template <int LM, int TM>
struct GdnSmemT {
  static constexpr int kL = LM;
  static constexpr int kZ0 = TM * kYS + 4;   // z table: 4 banks after y's
  union alignas(1024) {
    GdnFlushT<LM> f;
    // without a flush, or after a flush's fold: the head's read copy; fp32 io keeps it row-major
    // (one bulk copy), bf16 io in the 128-byte-swizzled K-major operand layout of the tensor core
    __nv_bfloat16 cb[kGD * kGD];
  } x;
  // bf16 io: the drafts' key rows (operand rows 0..7) and query rows (8..15), swizzled, K = dk
  alignas(1024) uint8_t bq[16 * kGD * 2];
  alignas(16) float k[LM + TM][kGD];   // committed rows 0..hc-1, drafts at LM + s
  float q[TM][kGD];
  float v[TM][kGD];          // drafts' v
  float u[LM + TM][kGD];     // residuals: committed (cached), drafts at LM + s
  // S_read k_s (row s at s * kYS) and S_read q_s (row s at kZ0 + s * kYS): rows padded so that the
  // 32 lanes of a reduce-scatter (4 rows x 4 drafts x {k, q}) store to 32 different banks
  float yz[kZ0 + TM * kYS];
  float gc[LM + TM];         // cumulative log-gates of the output rows
  float bt[LM + TM];         // beta of the output rows
  float gf[LM];              // cumulative log-gates of the committed rows (flush)
  float bf[LM];
  float kk[LM + TM][TM];     // k_row . k_draft
  float kq[LM + TM][TM];     // k_row . q_draft
  // per-head coefficients, computed once per head (same expressions, so the same bits, as inline)
  float gamf[LM];            // flush: gamma_{1..r}
  float wf[LM];              // flush: gamma_{r+1..hc}
  float cc[LM + TM][TM];     // drafts: beta_t gamma_{r+1..t} (k_r . k_s), r < t = h0 + s
  float wq[LM + TM][TM];     // drafts: gamma_{r+1..t} (k_r . q_s), r <= t
  float gam[TM];             // drafts: gamma_{1..t}
  float gd[TM];              // drafts' own log-gates (for the buffer)
  uint64_t bar;
  uint64_t mbar;             // bf16 io: completion of the drafts' MMAs, one phase per head
  uint32_t tmem;             // bf16 io: the CTA's tensor-memory columns (32)
};
using GdnSmemWide = GdnSmemT<kGL, kGT>;   // any window and draft count (two CTAs per SM)
using GdnSmemSmall = GdnSmemT<16, 4>;     // L <= 16, T <= 4 (three CTAs per SM)

template <class SM, int kCtas>
constexpr bool gdn_layout_ok() {
  using F = decltype(SM::x.f);
  return sizeof(F) >= kGD * kGD * 2 && offsetof(F, kkf) >= kGD * kGD * 2 && offsetof(F, kkf) % 16 == 0 &&
         sizeof(SM) + 1024 + 1024 <= 228 * 1024 / kCtas && offsetof(SM, k) % 16 == 0 && offsetof(SM, q) % 16 == 0 &&
         offsetof(SM, u) % 16 == 0 && offsetof(SM, v) % 16 == 0 && offsetof(SM, x) % 16 == 0 &&
         offsetof(SM, bar) % 8 == 0;
}
// the read copy fits the flush arrays' bytes; reloading a head's copy keeps the group's key products;
// the CTAs per SM fit (1 KB reserved per CTA); 16-byte rows, an 8-byte mbarrier
static_assert(gdn_layout_ok<GdnSmemWide, 2>() && gdn_layout_ok<GdnSmemSmall, 3>(), "shared-memory layout");

// Rows r = w, w + kGWarps, ... < n of warp w: 128-vectors src(r) -> dst(r), every load issued before
// any store, so that a warp's rows cost one round trip rather than one each (kMax rows per warp).
template <typename T, int kMax, typename Src, typename Dst>
__device__ __forceinline__ void load_rows(int n, Src src, Dst dst) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  typename Quad<T>::raw v[kMax];
#pragma unroll
  for (int q = 0; q < kMax; ++q) {
    const int r = w + q * kGWarps;
    if (r < n) v[q] = *reinterpret_cast<const typename Quad<T>::raw*>(src(r) + 4 * l);
  }
#pragma unroll
  for (int q = 0; q < kMax; ++q) {
    const int r = w + q * kGWarps;
    if (r < n) {
      float f[4];
      Quad<T>::unpack(v[q], f);
      *reinterpret_cast<float4*>(dst(r) + 4 * l) = make_float4(f[0], f[1], f[2], f[3]);
    }
  }
}

template <typename T>
__device__ __forceinline__ void store_vec(const float* src, T* __restrict__ p) {   // exact: src holds T values
  const int l = threadIdx.x & 31;
  const float4 f = *reinterpret_cast<const float4*>(src + 4 * l);
  p[4 * l] = from_f<T>(f.x);
  p[4 * l + 1] = from_f<T>(f.y);
  p[4 * l + 2] = from_f<T>(f.z);
  p[4 * l + 3] = from_f<T>(f.w);
}

// Warp-per-dot products of two smem vectors (Dot<128> order); lane 0 stores.
__device__ __forceinline__ float sdot(const float* a, const float* b, int j) {
  float qa[4], qb[4];
  lds4(a + 4 * j, qa);
  lds4(b + 4 * j, qb);
  return Dot<kGD>::reduce(Dot<kGD>::partial(qa, qb));
}

// bf16 io, the drafts' dot products on the tensor core: D[d][n] = sum_e S_read[d][e] Bq[n][e] for the
// 16 operand rows n (k_s at n = s, q_s at n = 8 + s, zero rows for absent drafts): one
// tcgen05.mma kind::f16 chain (M = 128 state rows, N = 16, K = dk in 8 steps of 16) into 16 TMEM
// columns.  A column's result does not depend on the other columns, so a draft gets the same bits
// whether it is one of several drafts or alone.
constexpr int kBq = 16;   // operand rows of the drafts' tile

__device__ __forceinline__ void copy_tile_async(uint8_t* tile, const __nv_bfloat16* __restrict__ src) {
  for (int id = threadIdx.x; id < kGD * (kGD / 8); id += kThreads) {   // 16-byte chunks, swizzled
    const int d = id >> 4, c = id & 15;
    tc::cp_async16(tile + sw128(kGD, d, 8 * c), src + (size_t)d * kGD + 8 * c);
  }
}

__device__ __forceinline__ void issue_draft_mma(uint32_t tmem_d, uint32_t aT, uint32_t bT) {
  const uint32_t id = tc::idesc_bf16(128, kBq, false, false);
#pragma unroll
  for (int k = 0; k < kGD / 16; ++k) {
    const uint32_t ao = (k >> 2) * (uint32_t)kGD * 128u + (k & 3) * 32u, bo = (k >> 2) * (uint32_t)kBq * 128u + (k & 3) * 32u;
    tc::mma(tmem_d, tc::sdesc(aT + ao, 16, 1024), tc::sdesc(bT + bo, 16, 1024), id, k > 0);
  }
}

template <class SM>
__device__ __forceinline__ SM& gdn_smem(unsigned char* raw) {   // 1024-byte aligned (swizzled tiles)
  return *reinterpret_cast<SM*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// S_src k_s and S_src q_s for the drafts (at most TM of them), RPG = 32 / (2 TM) rows per
// reduce-scatter: lane l gets the sum of partial l = 2 TM * (row of the group) + (s for k, TM + s
// for q); the pairings are Dot<128>'s, so each value has the bits of a Dot<128> reduction.
template <int TM, class SM>
__device__ __forceinline__ void draft_dots(SM& sm, const float (&rv)[32 / (2 * TM)][4], int d0, int Td, int j) {
  constexpr int RPG = 32 / (2 * TM);
  float part[32];
#pragma unroll
  for (int s = 0; s < TM; ++s) {
    float ka[4], qb[4];
    lds4(sm.k[SM::kL + s] + 4 * j, ka);
    lds4(sm.q[s] + 4 * j, qb);
#pragma unroll
    for (int g = 0; g < RPG; ++g) {
      part[2 * TM * g + s] = Dot<kGD>::partial(ka, rv[g]);
      part[2 * TM * g + TM + s] = Dot<kGD>::partial(qb, rv[g]);
    }
  }
  const float v = reduce_scatter32(part, j);
  const int d = d0 + j / (2 * TM), idx = j % (2 * TM);
  if (idx < TM) {
    if (idx < Td) sm.yz[idx * kYS + d] = v;
  } else if (idx - TM < Td) {
    sm.yz[SM::kZ0 + (idx - TM) * kYS + d] = v;
  }
}

// The flush of warp w's anchor rows, in three passes:
//  A. S k_i for the hc committed records, by reduce-scatter: with hc <= 16 two rows per reduce-scatter
//     (lane i: row rr's S k_i, lane 16 + i: row rr + 1's), else one row (lane i: S k_i);
//  B. the triangular solve, one row per lane (lanes 0..15), in row order, in place of S k_i;
//  C. the fold S'[d][n] = gamma_{1..hc} S[d][n] + sum_i gamma_{i+1..hc} u_i[d] k_i[n] (fma chain in
//     row order), two rows per pass sharing the key loads, stored to the anchor and cast to the bf16
//     read copy; with drafts, S' k_s and S' q_s from the cast values (draft_dots).
// Passes A and C keep the next pair of anchor rows in flight.  Each S k_i is a Dot<128> reduction
// whichever lane and row pairing carries it, so the bits do not depend on hc's branch.
template <int TM, class SM>
__device__ __forceinline__ void gdn_fold_rows(SM& sm, float* __restrict__ S, __nv_bfloat16* __restrict__ R,
                                              int hc, int ndraft, int w, int j) {
  constexpr int RPG = 32 / (2 * TM);
  static_assert(kGRows % 2 == 0 && RPG % 2 == 0 || RPG == 2, "row pairs fill the draft groups");
  float (*YU)[SM::kL + 1] = sm.x.f.yu[w];   // [row of the warp][record]: S k_i, then u_i
  const float* Sw = S + (size_t)(w * kGRows) * kGD + 4 * j;
  auto ldrow = [&](int rr) { return *reinterpret_cast<const float4*>(Sw + (size_t)rr * kGD); };
  if (SM::kL <= 16 || hc <= 16) {
    float4 c0 = ldrow(0), c1 = ldrow(1);
    for (int rr = 0; rr < kGRows; rr += 2) {
      float4 n0 = c0, n1 = c1;
      if (rr + 2 < kGRows) {
        n0 = ldrow(rr + 2);
        n1 = ldrow(rr + 3);
      }
      float h0[4], h1[4];
      Quad<float>::unpack(c0, h0);
      Quad<float>::unpack(c1, h1);
      float part[32];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float kq4[4];
        lds4(sm.k[r] + 4 * j, kq4);
        part[r] = r < hc ? Dot<kGD>::partial(kq4, h0) : 0.f;
        part[16 + r] = r < hc ? Dot<kGD>::partial(kq4, h1) : 0.f;
      }
      YU[rr + (j >> 4)][j & 15] = reduce_scatter32(part, j);
      c0 = n0;
      c1 = n1;
    }
  } else if constexpr (SM::kL > 16) {
    float4 c0 = ldrow(0);
    for (int rr = 0; rr < kGRows; ++rr) {
      const float4 n0 = rr + 1 < kGRows ? ldrow(rr + 1) : c0;
      float hq[4];
      Quad<float>::unpack(c0, hq);
      float part[32];
#pragma unroll
      for (int r = 0; r < SM::kL; ++r) {
        float kq4[4];
        lds4(sm.k[r] + 4 * j, kq4);
        part[r] = r < hc ? Dot<kGD>::partial(kq4, hq) : 0.f;
      }
      YU[rr][j] = reduce_scatter32(part, j);
      c0 = n0;
    }
  }
  __syncwarp();
  if (j < kGRows) {
    const int d = w * kGRows + j;
    for (int r = 0; r < hc; ++r) {
      float acc = __fmul_rn(sm.bf[r], __fmaf_rn(-sm.gamf[r], YU[j][r], sm.x.f.vc[r][d]));
      for (int i = 0; i < r; ++i) acc = __fmaf_rn(-sm.x.f.cf[i][r], YU[j][i], acc);
      YU[j][r] = acc;
    }
  }
  __syncwarp();
  const float gall = sm.gamf[hc - 1];
  float rvg[RPG][4];
  float4 c0 = ldrow(0), c1 = ldrow(1);
  for (int rr = 0; rr < kGRows; rr += 2) {
    float4 n0 = c0, n1 = c1;
    if (rr + 2 < kGRows) {
      n0 = ldrow(rr + 2);
      n1 = ldrow(rr + 3);
    }
    float h0[4], h1[4], v0[4], v1[4];
    Quad<float>::unpack(c0, h0);
    Quad<float>::unpack(c1, h1);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v0[e] = __fmul_rn(gall, h0[e]);
      v1[e] = __fmul_rn(gall, h1[e]);
    }
    for (int r = 0; r < hc; ++r) {
      float kq4[4];
      lds4(sm.k[r] + 4 * j, kq4);
      const float wf = sm.wf[r];
      const float wu0 = __fmul_rn(wf, YU[rr][r]), wu1 = __fmul_rn(wf, YU[rr + 1][r]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v0[e] = __fmaf_rn(wu0, kq4[e], v0[e]);
        v1[e] = __fmaf_rn(wu1, kq4[e], v1[e]);
      }
    }
    auto emit = [&](const float (&v)[4], int row) {
      const int d = w * kGRows + row;
      *reinterpret_cast<float4*>(S + (size_t)d * kGD + 4 * j) = make_float4(v[0], v[1], v[2], v[3]);
      const __nv_bfloat162 lo2 = __floats2bfloat162_rn(v[0], v[1]), hi2 = __floats2bfloat162_rn(v[2], v[3]);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&lo2);
      pk.y = *reinterpret_cast<const uint32_t*>(&hi2);
      *reinterpret_cast<uint2*>(R + (size_t)d * kGD + 4 * j) = pk;
      if (ndraft > 0) {
        float rv[4];
        Quad<__nv_bfloat16>::unpack(pk, rv);
#pragma unroll
        for (int g = 0; g < RPG; ++g)
          if (row % RPG == g)
#pragma unroll
            for (int e = 0; e < 4; ++e) rvg[g][e] = rv[e];
        if (row % RPG == RPG - 1) draft_dots<TM>(sm, rvg, d - (RPG - 1), ndraft, j);
      }
    };
    emit(v0, rr);
    emit(v1, rr + 1);
    c0 = n0;
    c1 = n1;
  }
}

// Committed records' key rows (the group's; shared by its heads) and per-head rows.
template <typename T, class SM>
__device__ __forceinline__ void load_committed_k(SM& sm, const GdnArgs& a, int slot, int g, int hc) {
  load_rows<T, (SM::kL + kGWarps - 1) / kGWarps>(
      hc, [&](int r) { return (const T*)a.bk + (((size_t)slot * a.L + r) * a.G + g) * kGD; },
      [&](int r) { return sm.k[r]; });
}

template <typename T, class SM>
__device__ __forceinline__ void load_committed_head(SM& sm, const GdnArgs& a, int slot, int h, int hc, bool flush) {
  constexpr int kMax = (SM::kL + kGWarps - 1) / kGWarps;
  if (flush)
    load_rows<T, kMax>(
        hc, [&](int r) { return (const T*)a.bv + (((size_t)slot * a.L + r) * a.H + h) * kGD; },
        [&](int r) { return sm.x.f.vc[r]; });
  else
    load_rows<float, kMax>(
        hc, [&](int r) { return a.bu + (((size_t)slot * a.L + r) * a.H + h) * kGD; }, [&](int r) { return sm.u[r]; });
}

// Lane r of a warp gets v_0 + v_1 + ... + v_r (n <= 32 values, lane q holding v_q), added one at a
// time from 0 in row order: the bits of a serial running sum.
__device__ __forceinline__ float ordered_prefix(float v, int n, int r) {
  float acc = 0.f;
  for (int q = 0; q < n; ++q) {
    const float vq = __shfl_sync(kFull, v, q);
    if (q <= r) acc = __fadd_rn(acc, vq);
  }
  return acc;
}

// Gates of the committed records summed in row order, and their betas (warp 0).
// (Warp 0: the lanes load one row each, then lane 0 sums in row order.)
template <class SM>
__device__ __forceinline__ void flush_scalars(SM& sm, const GdnArgs& a, int slot, int h, int hc) {
  if (threadIdx.x < 32) {
    const int r = threadIdx.x;
    float gr = 0.f;
    if (r < hc) {
      const size_t row = (size_t)slot * a.L + r;
      gr = a.bg[row * a.H + h];
      sm.bf[r] = a.bbeta[row * a.H + h];
    }
    const float acc = ordered_prefix(gr, hc, r);
    if (r < hc) sm.gf[r] = acc;
  }
}

template <class SM>
__device__ __forceinline__ void flush_gram(SM& sm, int hc) {
  const int w = threadIdx.x >> 5, j = threadIdx.x & 31;
  for (int p = w; p < hc * hc; p += kGWarps) {
    const int i = p / hc, r = p % hc;
    if (i < r) {
      const float v = sdot(sm.k[i], sm.k[r], j);
      if (j == 0) sm.x.f.kkf[i][r] = v;
    }
  }
}

// Per-head flush coefficients from gf, bf and kkf (all threads; call after both are in smem).
template <class SM>
__device__ __forceinline__ void flush_coeffs(SM& sm, int hc) {
  for (int p = threadIdx.x; p < hc * hc; p += kThreads) {
    const int i = p / hc, r = p % hc;
    if (i < r)
      sm.x.f.cf[i][r] = __fmul_rn(__fmul_rn(sm.bf[r], expf(__fsub_rn(sm.gf[r], sm.gf[i]))), sm.x.f.kkf[i][r]);
  }
  for (int r = threadIdx.x; r < hc; r += kThreads) {
    sm.gamf[r] = expf(sm.gf[r]);
    sm.wf[r] = expf(__fsub_rn(sm.gf[hc - 1], sm.gf[r]));
  }
}

// Per-head draft coefficients from gc, bt, kk and kq.
template <class SM>
__device__ __forceinline__ void draft_coeffs(SM& sm, int h0, int Td) {
  for (int p = threadIdx.x; p < (h0 + Td) * Td; p += kThreads) {
    const int r = p / Td, s = p % Td, t = h0 + s;
    if (r <= t) {
      const float e = expf(__fsub_rn(sm.gc[t], sm.gc[r]));
      sm.wq[r][s] = __fmul_rn(e, sm.kq[r][s]);
      if (r < t) sm.cc[r][s] = __fmul_rn(__fmul_rn(sm.bt[t], e), sm.kk[r][s]);
    }
  }
  for (int s = threadIdx.x; s < Td; s += kThreads) sm.gam[s] = expf(sm.gc[h0 + s]);
}

__device__ __forceinline__ bool gdn_slot(const GdnArgs& a, int i, int* slot) {
  const int s = a.slot != nullptr ? a.slot[i] : i;
  if (s < 0 || s >= a.nslots) {
    if (threadIdx.x == 0) report(a.status, ERS_ESLOT);
    return false;
  }
  *slot = s;
  return true;
}

// One CTA per (sequence, key group); its value heads run one after another, so the group's key rows
// are read once and the drafts' key rows are written after every head of the group has read the
// committed ones (a flush reuses buffer rows from 0).
// LM and TM bound the window and the drafts the shared-memory layout holds.  With L <= 16 and up to
// 4 drafts the layout takes 69.6 KB and three CTAs fit on an SM (80 registers); other windows with up
// to 4 drafts run two per SM (111.6 KB, 128 registers); the 8-draft variant needs more registers
// than two CTAs leave.
template <typename T, int TM, int LM>
__global__ void __launch_bounds__(kThreads, TM == 8 ? 1 : (LM == 16 ? 3 : 2)) k_gdn_verify(GdnArgs a) {
  using SM = GdnSmemT<LM, TM>;
  constexpr int RPG = 32 / (2 * TM);
  constexpr bool kTc = std::is_same<T, __nv_bfloat16>::value;   // bf16 io: drafts' dots on the tensor core
  extern __shared__ __align__(16) unsigned char gsm_raw[];
  SM& sm = gdn_smem<SM>(gsm_raw);
  const int g = blockIdx.x, i = blockIdx.y, tid = threadIdx.x, w = tid >> 5, j = tid & 31;
  const int hpg = a.H / a.G;
  const int Td = a.T;
  int slot;
  if (!gdn_slot(a, i, &slot)) return;
  const int hc = a.pos[slot];
  if (hc < 0 || hc > a.L) {
    if (tid == 0) report(a.status, ERS_EALIGN);
    return;
  }
  const bool flush = hc + Td > a.L;
  if (flush && !(a.flags & ERS_FLAG_AUTO_FLUSH)) {
    if (tid == 0) report(a.status, ERS_EOVERFLOW);
    return;
  }
  const int h0 = flush ? 0 : hc;   // committed rows that precede the drafts
  constexpr uint32_t kCopyBytes = kGD * kGD * 2;
  const __nv_bfloat16* Rg = (const __nv_bfloat16*)a.copy + (size_t)slot * a.H * kGD * kGD;   // the slot's copy
  if constexpr (kTc) {
    if (w == 0) tc::tmem_alloc(&sm.tmem, 32);
    if (tid == 0) {
      mbar_init(&sm.mbar, 1);
      fence_mbar_init();
    }
    if (!flush) copy_tile_async((uint8_t*)sm.x.cb, Rg + (size_t)(g * hpg) * kGD * kGD);   // first head's copy
  } else if (!flush && tid == 0) {   // the first head's read copy, in flight through the prologue
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&sm.bar, kCopyBytes);
    bulk_g2s(sm.x.cb, Rg + (size_t)(g * hpg) * kGD * kGD, kCopyBytes, &sm.bar);
  }
  load_committed_k<T>(sm, a, slot, g, hc);
  // the drafts' k rows (r < Td) and q rows (r >= Td), one batch
  load_rows<T, (2 * TM + kGWarps - 1) / kGWarps>(
      2 * Td,
      [&](int r) { return (const T*)(r < Td ? a.k : a.q) + (((size_t)i * Td + (r < Td ? r : r - Td)) * a.G + g) * kGD; },
      [&](int r) { return r < Td ? sm.k[LM + r] : sm.q[r - Td]; });
  __syncthreads();
  if constexpr (kTc) {   // the drafts' operand tile: row n = k_n (n < 8) or q_{n-8}; zeros past the drafts
    const int n = tid >> 4, c = tid & 15, s = n & 7;
    uint32_t pk[4] = {0u, 0u, 0u, 0u};
    if (s < Td) {
      const float* src = (n < 8 ? sm.k[LM + s] : sm.q[s]) + 8 * c;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(src[2 * e], src[2 * e + 1]);   // bf16 values: exact
        pk[e] = *reinterpret_cast<const uint32_t*>(&b2);
      }
    }
    *reinterpret_cast<uint4*>(sm.bq + sw128(kBq, n, 8 * c)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  if (flush && hc > 0) flush_gram(sm, hc);
  // k_row . k_s (rows before draft s) and k_row . q_s (rows up to draft s), row r of the output rows
  for (int p = w; p < (h0 + Td) * Td; p += kGWarps) {
    const int r = p / Td, s = p % Td;
    const float* kr = r < h0 ? sm.k[r] : sm.k[LM + r - h0];
    if (r <= h0 + s) {
      const float vq = sdot(kr, sm.q[s], j);
      const float vk = r < h0 + s ? sdot(kr, sm.k[LM + s], j) : 0.f;
      if (j == 0) {
        sm.kq[r][s] = vq;
        sm.kk[r][s] = vk;
      }
    }
  }
  for (int hh = 0; hh < hpg; ++hh) {
    const int h = g * hpg + hh;
    const size_t soff = ((size_t)slot * a.H + h) * kGD * kGD;
    load_committed_head<T>(sm, a, slot, h, hc, flush);
    load_rows<T, (TM + kGWarps - 1) / kGWarps>(
        Td, [&](int s) { return (const T*)a.v + (((size_t)i * Td + s) * a.H + h) * kGD; }, [&](int s) { return sm.v[s]; });
    if (flush && hc > 0) flush_scalars(sm, a, slot, h, hc);
    if (w == 1) {   // output rows: committed rows 0..h0-1, then the drafts (h0 + Td <= 32); gates in row order
      const int r = j, n = h0 + Td;
      float gr = 0.f;
      if (r < n) {
        const size_t br = ((size_t)slot * a.L + r) * a.H + h, tr = ((size_t)i * Td + (r - h0)) * a.H + h;
        gr = r < h0 ? a.bg[br] : a.g[tr];
        sm.bt[r] = r < h0 ? a.bbeta[br] : a.beta[tr];
        if (r >= h0) sm.gd[r - h0] = gr;
      }
      const float acc = ordered_prefix(gr, n, r);
      if (r < n) sm.gc[r] = acc;
    }
    if constexpr (kTc) {
      tc::publish();   // the head's copy (without a flush) and the drafts' tile, visible to the tensor core
      if (flush && hc > 0) flush_coeffs(sm, hc);
      draft_coeffs(sm, h0, Td);
      if (flush) {
        __syncthreads();
        if (hc > 0) gdn_fold_rows<TM>(sm, a.anchor + soff, (__nv_bfloat16*)a.copy + soff, hc, 0, w, j);
        __syncthreads();   // the new copy is written; the fold's arrays are free
        copy_tile_async((uint8_t*)sm.x.cb, (const __nv_bfloat16*)a.copy + soff);
        tc::publish();
      }
      if (tid == 0) {
        issue_draft_mma(sm.tmem, tc::smem_u32(sm.x.cb), tc::smem_u32(sm.bq));
        tc::commit(&sm.mbar);
      }
      mbar_wait(&sm.mbar, hh & 1, a.status);   // bounded; a wait that gave up has reported ERS_ETIMEOUT
      tc::after_sync();
      if (w < 4) {   // warp w reads TMEM lanes 32w..32w+31 = state rows d = tid
        float dv[kBq];
        tc::tmem_ld16(tc::taddr(sm.tmem, 32 * w, 0), dv);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          if (s < Td) {
            sm.yz[s * kYS + tid] = dv[s];
            sm.yz[SM::kZ0 + s * kYS + tid] = dv[8 + s];
          }
        }
      }
      tc::before_sync();
      __syncthreads();   // y, z ready; the MMA has read the copy tile
      if (!flush && hh + 1 < hpg) copy_tile_async((uint8_t*)sm.x.cb, Rg + (size_t)(h + 1) * kGD * kGD);
    } else {
    // the head's read copy has landed (without a flush); a wait that gave up ends the CTA
    const bool late = !flush && !mbar_wait(&sm.bar, hh & 1, a.status);
    if (__syncthreads_or(late)) {
      if (tid == 0) mbar_wait(&sm.bar, hh & 1, nullptr);   // bounded: no copy left in flight on exit
      return;
    }
    if (flush && hc > 0) flush_coeffs(sm, hc);
    draft_coeffs(sm, h0, Td);
    if (flush) __syncthreads();   // the fold reads the flush coefficients; the plain stream needs none
    if (flush && hc > 0) {
      gdn_fold_rows<TM>(sm, a.anchor + soff, (__nv_bfloat16*)a.copy + soff, hc, Td, w, j);
    } else {
      // S_read k_s and S_read q_s for every draft from the head's copy in shared memory
#pragma unroll
      for (int rr = 0; rr < kGRows; rr += RPG) {
        float rvg[RPG][4];
#pragma unroll
        for (int g = 0; g < RPG; ++g) {
          const uint2 raw = *reinterpret_cast<const uint2*>(sm.x.cb + (size_t)(w * kGRows + rr + g) * kGD + 4 * j);
          Quad<__nv_bfloat16>::unpack(raw, rvg[g]);
        }
        draft_dots<TM>(sm, rvg, w * kGRows + rr, Td, j);
      }
    }
    __syncthreads();
    if (!flush && tid == 0 && hh + 1 < hpg) {   // every warp is done with this head's copy
      mbar_arrive_expect_tx(&sm.bar, kCopyBytes);
      bulk_g2s(sm.x.cb, Rg + (size_t)(h + 1) * kGD * kGD, kCopyBytes, &sm.bar);
    }
    }
    // residuals, one state row d per thread, drafts in order (draft s needs the residuals before it)
    if (tid < kGD) {
      const int d = tid;
      for (int s = 0; s < Td; ++s) {
        const int t = h0 + s;
        float acc = __fmul_rn(sm.bt[t], __fmaf_rn(-sm.gam[s], sm.yz[s * kYS + d], sm.v[s][d]));
#pragma unroll 4
        for (int r = 0; r < h0; ++r) acc = __fmaf_rn(-sm.cc[r][s], sm.u[r][d], acc);
        for (int r = h0; r < t; ++r) acc = __fmaf_rn(-sm.cc[r][s], sm.u[LM + r - h0][d], acc);
        sm.u[LM + s][d] = acc;
      }
    }
    __syncthreads();
    // outputs, (row d, draft s) over all threads, each sum in row order
    for (int p = tid; p < Td * kGD; p += kThreads) {
      const int d = p % kGD, s = p / kGD, t = h0 + s;
      float out = __fmul_rn(sm.gam[s], sm.yz[SM::kZ0 + s * kYS + d]);
#pragma unroll 4
      for (int r = 0; r < h0; ++r) out = __fmaf_rn(sm.wq[r][s], sm.u[r][d], out);
      for (int r = h0; r <= t; ++r) out = __fmaf_rn(sm.wq[r][s], sm.u[LM + r - h0][d], out);
      ((T*)a.o)[(((size_t)i * Td + s) * a.H + h) * kGD + d] = from_f<T>(out);
    }
    // this head's draft rows (v, residual, gate, beta) go to buffer rows h0..h0+T-1
    for (int s = w; s < Td; s += kGWarps) {
      const size_t row = (size_t)slot * a.L + h0 + s;
      store_vec<T>(sm.v[s], (T*)a.bv + (row * a.H + h) * kGD);
      store_vec<float>(sm.u[LM + s], a.bu + (row * a.H + h) * kGD);
      if (j == 0) {
        a.bg[row * a.H + h] = sm.gd[s];
        a.bbeta[row * a.H + h] = sm.bt[h0 + s];
      }
    }
    __syncthreads();   // the next head's loads overwrite the committed residuals the outputs read
  }
  // the group's draft key rows, after every head has read the committed ones
  for (int s = w; s < Td; s += kGWarps) {
    const size_t row = (size_t)slot * a.L + h0 + s;
    store_vec<T>(sm.k[LM + s], (T*)a.bk + (row * a.G + g) * kGD);
  }
  if constexpr (kTc) {   // every TMEM read finished before the last head's barriers: free the columns
    tc::after_sync();
    if (w == 0) tc::tmem_dealloc(sm.tmem, 32);
  }
}

// Standalone refresh: slots with h + T > L (T = drafts_T) and h > 0 fold their records exactly as a
// verify's flush does.  Positions are reset by k_gdn_setpos afterwards.
template <typename T>
__global__ void __launch_bounds__(kThreads, 2) k_gdn_refresh(GdnArgs a) {
  extern __shared__ __align__(16) unsigned char gsm_raw[];
  GdnSmemWide& sm = gdn_smem<GdnSmemWide>(gsm_raw);
  const int g = blockIdx.x, i = blockIdx.y, w = threadIdx.x >> 5, j = threadIdx.x & 31;
  const int hpg = a.H / a.G;
  int slot;
  if (!gdn_slot(a, i, &slot)) return;
  const int hc = a.pos[slot];
  if (hc < 0 || hc > a.L) {
    if (threadIdx.x == 0) report(a.status, ERS_EALIGN);
    return;
  }
  if (!(hc + a.T > a.L) || hc == 0) return;
  load_committed_k<T>(sm, a, slot, g, hc);
  __syncthreads();
  flush_gram(sm, hc);
  for (int hh = 0; hh < hpg; ++hh) {
    const int h = g * hpg + hh;
    load_committed_head<T>(sm, a, slot, h, hc, true);
    flush_scalars(sm, a, slot, h, hc);
    __syncthreads();
    flush_coeffs(sm, hc);
    __syncthreads();
    const size_t soff = ((size_t)slot * a.H + h) * kGD * kGD;
    gdn_fold_rows<4>(sm, a.anchor + soff, (__nv_bfloat16*)a.copy + soff, hc, 0, w, j);
    __syncthreads();
  }
}

__global__ void k_gdn_setpos(GdnArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.nseq) return;
  const int s = a.slot != nullptr ? a.slot[i] : i;
  if (s < 0 || s >= a.nslots) return;
  const int hc = a.pos[s];
  if (hc >= 0 && hc <= a.L && hc + a.T > a.L) a.pos[s] = 0;
}

// Commit: h = (flushed ? 0 : h) + accepted, flushed = AUTO_FLUSH && h + T > L.
__global__ void k_gdn_commit(GdnArgs a, const int32_t* accepted) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.nseq) return;
  const int s = a.slot != nullptr ? a.slot[i] : i;
  if (s < 0 || s >= a.nslots) {
    report(a.status, ERS_ESLOT);
    return;
  }
  const int acc = accepted[i];
  if (acc < 0 || acc > a.T) {
    report(a.status, ERS_ECOMMIT);
    return;
  }
  const int hc = a.pos[s];
  const bool flushed = (a.flags & ERS_FLAG_AUTO_FLUSH) && hc + a.T > a.L;
  a.pos[s] = (flushed ? 0 : hc) + acc;
}

}  // namespace

bool gdn_supported(int dk, int dv, int L, int T) {
  return dk == kGD && dv == kGD && L >= 1 && L <= kGL && T >= 0 && T <= kGT;
}

cudaError_t gdn_launch(const GdnArgs& a, int kind, const int32_t* accepted, cudaStream_t s) {
  cudaError_t e;
  if (kind == 2) {
    k_gdn_commit<<<(a.nseq + 255) / 256, 256, 0, s>>>(a, accepted);
    return cudaGetLastError();
  }
  const dim3 grid(a.G, a.nseq);
  // + room to align the tiles to 1024 bytes; the shared-memory carveout at its maximum, so that the
  // small layout's three CTAs fit on an SM
  auto run = [&](auto kernel, size_t sm) {
    cudaError_t err = prep(kernel, sm);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    kernel<<<grid, kThreads, sm, s>>>(a);
    return cudaGetLastError();
  };
  const size_t wide = sizeof(GdnSmemWide) + 1024, narrow = sizeof(GdnSmemSmall) + 1024;
  const bool small = a.T <= 4;   // drafts' dot products 4 wide (4 rows per reduce-scatter), else 8
  const bool short_window = small && a.L <= 16;   // the small layout, three CTAs per SM
  if (a.io == ERS_DTYPE_BF16) {
    e = kind == 1        ? run(k_gdn_refresh<__nv_bfloat16>, wide)
        : short_window ? run(k_gdn_verify<__nv_bfloat16, 4, 16>, narrow)
        : small        ? run(k_gdn_verify<__nv_bfloat16, 4, kGL>, wide)
                       : run(k_gdn_verify<__nv_bfloat16, 8, kGL>, wide);
  } else {
    e = kind == 1        ? run(k_gdn_refresh<float>, wide)
        : short_window ? run(k_gdn_verify<float, 4, 16>, narrow)
        : small        ? run(k_gdn_verify<float, 4, kGL>, wide)
                       : run(k_gdn_verify<float, 8, kGL>, wide);
  }
  if (e != cudaSuccess) return e;
  if (kind == 1) {
    k_gdn_setpos<<<(a.nseq + 255) / 256, 256, 0, s>>>(a);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace ers
