// ReplaySSM decode and speculative verify for small refresh periods (L <= 16) with bf16 io, a bf16
// read copy, P = 64, N = 128 and at most 8 heads per B/C group: the read copy's products on the
// tensor core.
//
// ReplaySSM notes ("Motivation and method", "Core equations"): the output of a token at buffer row t
// is the off-diagonal term (S_read C_t), decayed by exp(Acum_t), plus the replay of the committed
// records and earlier drafts, (C_t . B_s) w_s x_s, plus D x_t.  A slot whose records would overflow
// the buffer (h + T > L) first folds its h records into the anchor and recasts the copy from the same
// unrounded values; the drafts then start at row 0.  Decode is the T = 1 case of the same kernel (the
// fused flush of a full buffer is the same rule with T = 1), so verify outputs equal non-speculative
// decode bit for bit.
//
// The drafts' products S_read C_k (M = state rows, N = drafts, K = dstate) are one dense contraction
// per head: tcgen05.mma kind::f16 with the bf16 copy as the A operand and the drafts' C rows as the
// B operand (row k = draft k, zero rows past the drafts), fp32 accumulators in tensor memory.  A column's result depends only on its own B row, so a draft gets
// the same bits in column k of a verify as in column 0 of a decode step.
//
// Layout: one CTA per (sequence, group), one warp per head (8 warps).  The A operand is a ring of two
// 32 KB chain buffers of 128 rows x K 128; round r in {0, 1} holds state rows [32r, 32r + 32) of
// heads 4c..4c+3 in buffer c, so warp w reads its head's results from the TMEM lane quarter w % 4 of
// chain (r, w / 4): lane j gets row 32r + j, the lane layout of the outputs.  A plain step streams
// the copy through the ring as TMA boxes {64, 32, 1, 4} (a 4-D map over the copy, this GPU's memory
// only); a flushing slot's warps fold their anchor rows and store the freshly cast values into the
// ring.  Every wait is bounded.  FP8 and NVFP4 copies keep the CUDA-core kernels for decode and
// verify alike: their tiles would have to be converted by the warps between the rounds, which cost
// more than the products it saves.
#include <cuda.h>
#include <string.h>

#include <type_traits>

#include "ers_common.cuh"
#include "ers_internal.h"
#include "tma_host.h"
#include "warp_heads.cuh"

namespace ers {
namespace {

using namespace wh;
using tc::mbar_wait;
using tc::sw128;

constexpr int kRP = 64, kRN = 128;         // headdim, dstate
constexpr int kRWarps = 8;                 // math warps: one head each
constexpr int kRIssuer = kRWarps;          // the warp that allocates TMEM, loads with TMA and issues the MMAs
constexpr int kRMath = 32 * kRWarps;
constexpr int kRThreads = kRMath + 32;
constexpr int kRQM = 16;                   // largest refresh period L
constexpr int kRTM = 16;                   // most drafts: N of the MMA, rows of the C tile
constexpr int kRRows = kRQM + kRTM;        // B / x rows: committed records, then the drafts at kRQM
constexpr uint32_t kChainBytes = 128u * kRN * 2u;   // 128 rows x K 128, bf16 (two 16 KB K halves)
constexpr uint32_t kCTileBytes = kRTM * kRN * 2u;
constexpr uint32_t kRTmemCols = 64;        // 2 rounds x 2 chains x 16 columns
constexpr uint32_t kBoxBytes = 4u * 32u * 64u * 2u;   // one TMA box: 4 heads x 32 rows x 64 values
constexpr uint32_t kHalfBytes = 128u * 128u;           // one K half of a chain (a ring slot)

struct RsmSmem {
  uint8_t ring[2][kChainBytes];            // A operand: slot 2c + kh = K half kh of chain c (1024-byte aligned)
  uint8_t ct[kCTileBytes];                 // B operand: the drafts' C rows
  __nv_bfloat16 b[kRRows * kRN];           // the group's B rows: committed, then drafts
  __nv_bfloat16 x[kRWarps][kRRows * kRP];  // each head's x rows, same row order
  float g[kRTM * kRRows];                  // Gram rows: g[k][s] = C of draft k . B of output row s
  uint64_t full[4];                        // a slot's TMA unit landed (phase 0: round 0, phase 1: round 1)
  uint64_t empty[4];                       // round 0's MMAs on a slot done: the slot may be refilled
  uint64_t ready[2];                       // a round's rows written by the math warps (one arrival each)
  uint64_t done[2];                        // a round's MMAs done: its TMEM columns readable, the ring free
  uint32_t tmem;
};

constexpr size_t rsm_smem_bytes() { return sizeof(RsmSmem) + 1024; }

__device__ __forceinline__ RsmSmem& rsm_smem(unsigned char* raw) {
  return *reinterpret_cast<RsmSmem*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// A operand address of state row d (round d / 32) of head w, K element 4j (lane j's 4 values).
__device__ __forceinline__ uint8_t* ring_at(RsmSmem& sm, int w, int d, int j) {
  return sm.ring[w >> 2] + sw128(128, (uint32_t)((w & 3) * 32 + (d & 31)), (uint32_t)(4 * j));
}

// K steps [k0, k1) of chain (r, c): D[row][n] (+)= sum over the step's 16 values of A[row][.] Ct[n][.],
// into the 16 TMEM columns of chain (r, c).  Every chain issues steps 0..7 in order, whichever way its
// operand arrived, so a row's result has one definition.
__device__ __forceinline__ void issue_chain(const RsmSmem& sm, int r, int c, int k0, int k1) {
  constexpr uint32_t id = tc::idesc_bf16(128, kRTM, false, false);
  const uint32_t at = tc::smem_u32(sm.ring[c]), bt = tc::smem_u32(sm.ct);
  const uint32_t d = sm.tmem + (uint32_t)(16 * (2 * r + c));
  for (int k = k0; k < k1; ++k) {
    const uint32_t ao = (uint32_t)(k >> 2) * kHalfBytes + (k & 3) * 32u, bo = (k >> 2) * (uint32_t)kRTM * 128u + (k & 3) * 32u;
    tc::mma(d, tc::sdesc(at + ao, 16, 1024), tc::sdesc(bt + bo, 16, 1024), id, k > 0);
  }
}

// 4-D TMA load (x innermost, in elements) into shared memory, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* map, int x, int y, int z, int v, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(tc::smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(v), "r"(tc::smem_u32(bar))
      : "memory");
}

// TMA unit (round r, chain c, K half kh) of a bf16 copy: rows [32r, 32r + 32) of heads 4c..4c+3 of the
// CTA, values [64 kh, 64 kh + 64), into slot 2c + kh.
__device__ __forceinline__ void load_unit(RsmSmem& sm, const CUtensorMap* map, int r, int c, int kh, int head0) {
  uint64_t* bar = &sm.full[2 * c + kh];
  tc::mbar_arrive_expect_tx(bar, kBoxBytes);
  tma_load_4d(sm.ring[c] + (uint32_t)kh * kHalfBytes, map, 64 * kh, 0, r, head0 + 4 * c, bar);
}

// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void st_ring_raw(RsmSmem& sm, int w, int d, int j, uint2 u) {
  *reinterpret_cast<uint2*>(ring_at(sm, w, d, j)) = u;
}

// Position advance inside a decode launch: every CTA of a slot adds 1 << 16 to pos[slot] once all of
// its threads have read the position (the low 16 bits); the CTA that completes the count (ncta CTAs
// per slot) stores the new position, which also clears the count.
constexpr int32_t kRPosMask = 0xFFFF;

__device__ __forceinline__ void count_and_advance(int32_t* pos, int ncta, int32_t newp) {
  const int32_t old = atomicAdd(pos, 1 << 16);
  if ((old >> 16) == ncta - 1) atomicExch(pos, newp);
}

// Flush, rows [32r, 32r + 32) of head w: each anchor row is folded with the hc committed records in
// chunk_state / fold_state order (acc = fma(w_s x_s[d], B_s[n], acc) over s < hc, w_s x_s[d] one fp32
// product, then fma(decay, H, acc)), written back (fp32, or fp16 by stochastic rounding), cast into
// the bf16 read copy, and the cast values stored into the ring.  Lane s holds w_s in wl.  Every value
// gets the operations of the standalone refresh, so anchors and copies get its bits; 4 rows share each
// record's loads, and the products and sums run as paired instructions.
template <typename AT>
__device__ __forceinline__ void flush_round(RsmSmem& sm, AT* __restrict__ Hd, __nv_bfloat16* __restrict__ R, int w,
                                            int j, int r, int hc, float wl, float decay, SrCtr sr, uint32_t row0) {
  const __nv_bfloat16* sx = sm.x[w];
#pragma unroll 1
  for (int blk = 0; blk < 8; ++blk) {
    const int d0 = 32 * r + 4 * blk;
    float4 cur[4];   // the block's anchor rows (in L2 by then), landing while the records are summed
#pragma unroll
    for (int q = 0; q < 4; ++q) cur[q] = anchor_ld<AT>(Hd, (size_t)(d0 + q) * kRN + 4 * j);
    uint64_t acc[2][4];   // acc[p][e] = rows (d0 + 2p, d0 + 2p + 1), column 4j + e
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[p][e] = 0ull;
#pragma unroll 4
    for (int s = 0; s < hc; ++s) {
      float bs[4];
      lds4(sm.b + s * kRN + 4 * j, bs);
      const uint2 xw = *reinterpret_cast<const uint2*>(sx + s * kRP + d0);   // x_s[d0 .. d0 + 4), bf16
      const float ws = __shfl_sync(kFull, wl, s);
      const uint64_t w2 = pk2(ws, ws);
      const uint32_t xv[2] = {xw.x, xw.y};
      uint64_t wx[2];
#pragma unroll
      for (int p = 0; p < 2; ++p)
        wx[p] = mul2(w2, pk2(__uint_as_float(xv[p] << 16), __uint_as_float(xv[p] & 0xFFFF0000u)));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint64_t b2 = pk2(bs[e], bs[e]);
#pragma unroll
        for (int p = 0; p < 2; ++p) fma2(acc[p][e], wx[p], b2);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int d = d0 + q;
      float h[4], v[4];
      Quad<float>::unpack(cur[q], h);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float lo, hi;
        up2(acc[q >> 1][e], lo, hi);
        v[e] = hc > 0 ? __fmaf_rn(decay, h[e], (q & 1) ? hi : lo) : h[e];
      }
      const size_t o = (size_t)d * kRN + 4 * j;
      if (hc > 0) anchor_st<AT>(Hd, o, v, sr, row0 + d, j);
      const __nv_bfloat162 lo2 = __floats2bfloat162_rn(v[0], v[1]), hi2 = __floats2bfloat162_rn(v[2], v[3]);
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&lo2);
      u.y = *reinterpret_cast<const uint32_t*>(&hi2);
      *reinterpret_cast<uint2*>(R + o) = u;
      st_ring_raw(sm, w, d, j, u);
    }
  }
}

// Outputs of every draft for state row d = 32r + j of head w (lane j): the product from TMEM, the
// replay over output rows s <= t = h0 + k in order, and combine_out.  Lane s holds output row s's decay term dl and log-decay prefix v.
__device__ __forceinline__ void out_round(const RsmSmem& sm, const float (&dv)[kRTM], int w, int j, int r,
                                          int h0, int Td, float dl, df v, float Dh, __nv_bfloat16* __restrict__ y,
                                          size_t ystride) {
  const __nv_bfloat16* sx = sm.x[w];
  const int d = 32 * r + j;
#pragma unroll
  for (int k = 0; k < kRTM; ++k) {
    if (k >= Td) break;
    const int t = h0 + k;
    const df at = {__shfl_sync(kFull, v.hi, t), __shfl_sync(kFull, v.lo, t)};
    const float M = j <= t ? __fmul_rn(__fmul_rn(sm.g[k * kRRows + j], dl), expf(df_diff(at, v))) : 0.f;
    float acc = 0.f;
    for (int s = 0; s <= t; ++s)
      acc = __fmaf_rn(__shfl_sync(kFull, M, s), to_f(sx[(s < h0 ? s : kRQM + s - h0) * kRP + d]), acc);
    y[(size_t)k * ystride + d] = from_f<__nv_bfloat16>(combine_out(expf(at.hi), dv[k], acc, Dh, to_f(sx[(kRQM + k) * kRP + d])));
  }
}

// The issuer warp's lane 0: TMEM is allocated by the whole warp beforehand.  A plain step with a bf16
// copy streams its units through the four slots (at most 64 KB in flight): round 0's units are issued
// as they land and each slot is refilled with its round-1 unit once the MMAs reading it are done.  A
// flushing slot or a narrow copy waits for the math warps' rows of each round.
__device__ __forceinline__ void issuer(RsmSmem& sm, const CUtensorMap* map, bool tma, int nchains, int head0,
                                       int32_t* st, uint64_t lim) {
  if (tma) {
    const int nu = 2 * nchains;   // units (slots) per round
    for (int u = 0; u < nu; ++u) {
      mbar_wait(&sm.full[u], 0, st, lim);
      issue_chain(sm, 0, u >> 1, 4 * (u & 1), 4 * (u & 1) + 4);
      tc::commit(&sm.empty[u]);
      if (u > 0) {   // the previous slot's MMAs have had a unit's time to finish
        mbar_wait(&sm.empty[u - 1], 0, st, lim);
        load_unit(sm, map, 1, (u - 1) >> 1, (u - 1) & 1, head0);
      }
    }
    tc::commit(&sm.done[0]);
    mbar_wait(&sm.empty[nu - 1], 0, st, lim);
    load_unit(sm, map, 1, (nu - 1) >> 1, (nu - 1) & 1, head0);
    for (int u = 0; u < nu; ++u) {
      mbar_wait(&sm.full[u], 1, st, lim);
      issue_chain(sm, 1, u >> 1, 4 * (u & 1), 4 * (u & 1) + 4);
    }
    tc::commit(&sm.done[1]);
    for (int u = 0; u < nu; ++u) mbar_wait(&sm.full[u], 1, nullptr, lim);   // none in flight at exit
  } else {
    for (int r = 0; r < 2; ++r) {
      mbar_wait(&sm.ready[r], 0, st, lim);
      for (int c = 0; c < nchains; ++c) issue_chain(sm, r, c, 0, kRN / 16);
      tc::commit(&sm.done[r]);
    }
  }
  mbar_wait(&sm.done[1], 0, nullptr, lim);   // no MMA in flight when the columns are freed
}

// A math warp's rows of round r are in the ring: visible to the tensor core, counted on ready[r].
__device__ __forceinline__ void rows_ready(RsmSmem& sm, int r, int j) {
  tc::fence_async_smem();
  __syncwarp();
  if (j == 0) tc::mbar_arrive(&sm.ready[r]);
}

// decode != 0: one token per sequence (Td = 1) with the position advance (and, with
// ERS_FLAG_FUSE_REFRESH, the flush of a full buffer); else a verify of Td drafts (pointers unchanged;
// ERS_FLAG_AUTO_FLUSH allows flushes).
// part: kPartAll, or one of the two launches of a call that may flush (kPartFlushes, then kPartPlain
// as its programmatic dependent; ers_internal.h), so that the long flushing CTAs run alongside the
// plain ones instead of after them.

template <typename AT>
__global__ void __maxnreg__(96)
    k_rssm_tc(const __grid_constant__ LaunchArgs a, const __grid_constant__ CUtensorMap map, int Td, int decode,
              int part) {
  using T = __nv_bfloat16;
  extern __shared__ __align__(16) unsigned char rsm_raw[];
  RsmSmem& sm = rsm_smem(rsm_raw);
  const int tid = threadIdx.x, w = tid >> 5, j = tid & 31;
  const int i = blockIdx.y, g = blockIdx.x;
  const int hpg = a.H / a.G;
  const bool active = w < hpg;   // a math warp with a head
  const int h = g * hpg + (active ? w : 0);
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const int32_t praw = a.pos[slot];
  const int hc = decode ? (praw & kRPosMask) : praw;   // decode: other CTAs of the slot may have counted
  bool flush;
  if (decode) {
    flush = (a.flags & ERS_FLAG_FUSE_REFRESH) != 0 && hc == a.Q;
    if (hc > a.Q || (hc == a.Q && !flush)) {   // the same in every CTA of the slot: none counts
      if (tid == 0) report(a.status, ERS_EALIGN);
      return;
    }
  } else {
    if (hc < 0 || hc > a.Q) {
      if (tid == 0) report(a.status, ERS_EALIGN);
      return;
    }
    flush = hc + Td > a.Q;
    if (flush && !(a.flags & ERS_FLAG_AUTO_FLUSH)) {
      if (tid == 0) report(a.status, ERS_EOVERFLOW);
      return;
    }
  }
  if (part == kPartFlushes) {
    allow_dependents();   // this CTA has read its position
    if (!flush) return;
  } else if (part == kPartPlain) {
    if (last_cta_of_grid()) wait_primary();   // completes only after the flushing launch
    if (flush) {   // done by the first launch; a decode still counts the slot's CTAs here
      __syncthreads();   // every thread of the CTA has read the position
      if (decode && tid == 0) count_and_advance(&a.pos[slot], a.G, 1);
      return;
    }
  }
  const int h0 = flush ? 0 : hc;   // committed rows that precede the drafts
  const int nchains = hpg > 4 ? 2 : 1;
  const bool tma = !flush;
  const int head0 = slot * a.H + g * hpg;   // the CTA's first head in the copy's head index
  const uint64_t lim = a.wait_ns ? a.wait_ns : tc::kWaitLimitNs;
  const size_t HP = (size_t)a.H * kRP, GN = (size_t)a.G * kRN;
  if (w == kRIssuer) {
    if (j == 0) {
      for (int u = 0; u < 4; ++u) {
        tc::mbar_init(&sm.full[u], 1);
        tc::mbar_init(&sm.empty[u], 1);
      }
      for (int r = 0; r < 2; ++r) {
        tc::mbar_init(&sm.ready[r], kRWarps);
        tc::mbar_init(&sm.done[r], 1);
      }
      tc::fence_mbar_init();
      if (tma)
        for (int u = 0; u < 2 * nchains; ++u) load_unit(sm, &map, 0, u >> 1, u & 1, head0);
    }
    tc::tmem_alloc(&sm.tmem, kRTmemCols);
  }
  const size_t soff = ((size_t)slot * a.H + h) * kRP * kRN;
  if (flush && active && j == 0)   // the head's anchor rows stream into L2 while the prologue runs
    l2_prefetch(reinterpret_cast<const AT*>(a.state) + soff, kRP * kRN * sizeof(AT));
  // committed rows 0..hc-1 at smem rows 0..hc-1, drafts at rows kRQM..kRQM+Td-1
  const T* bB = (const T*)a.bB + (size_t)g * kRN;
  constexpr int kBChunks = kRN * 2 / 16, kXChunks = kRP * 2 / 16;
  for (int k = tid; k < (hc + Td) * kBChunks; k += kRThreads) {
    const int r = k / kBChunks, e = k % kBChunks;
    const T* s = r < hc ? bB + buf_row(a, slot, r) * GN : (const T*)a.B + ((size_t)i * Td + (r - hc)) * GN + (size_t)g * kRN;
    cp_async16(reinterpret_cast<char*>(sm.b + (r < hc ? r : kRQM + r - hc) * kRN) + 16 * e,
               reinterpret_cast<const char*>(s) + 16 * e);
  }
  T* sx = sm.x[w < kRWarps ? w : 0];
  if (active) {
    const T* bx = (const T*)a.bx + (size_t)h * kRP;
    for (int k = j; k < (hc + Td) * kXChunks; k += 32) {
      const int r = k / kXChunks, e = k % kXChunks;
      const T* s = r < hc ? bx + buf_row(a, slot, r) * HP : (const T*)a.x + ((size_t)i * Td + (r - hc)) * HP + (size_t)h * kRP;
      cp_async16(reinterpret_cast<char*>(sx + (r < hc ? r : kRQM + r - hc) * kRP) + 16 * e,
                 reinterpret_cast<const char*>(s) + 16 * e);
    }
  }
  if (tid < kRMath) {   // the drafts' C rows: the B operand (row n = draft n, zero rows past the drafts)
    const int n = tid >> 4, c = tid & 15;
    uint8_t* dst = sm.ct + sw128(kRTM, n, 8 * c);
    if (n < Td)
      cp_async16(dst, (const T*)a.C + ((size_t)i * Td + n) * GN + (size_t)g * kRN + 8 * c);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
  // per-head scalars, in flight with the rows
  const float dt_c = j < hc ? a.bdt[buf_row(a, slot, j) * a.H + h] : 0.f;
  const float dt_d = j < Td ? a.dt[((size_t)i * Td + j) * a.H + h] : 0.f;
  const float Ah = a.A[h], bias = a.dt_bias[h], Dh = a.D[h];
  tc::publish();   // rows, C tile, barriers and the TMEM address visible (to the tensor core too)
  if (w == kRIssuer) {
    if (j == 0) issuer(sm, &map, tma, nchains, head0, a.status, lim);
    __syncwarp();
  } else {
    if (decode && part != kPartFlushes && tid == 0) count_and_advance(&a.pos[slot], a.G, h0 + 1);   // pos read by all
    // output rows s < h0 + Td: committed rows, then the drafts; lane s holds row s
    const int nout = h0 + Td;
    const float dt_o_d = __shfl_sync(kFull, dt_d, max(j - h0, 0) & 31);
    float dl = 0.f;
    df v = {0.f, 0.f};
    if (j < nout) {
      dl = delta_of(j < h0 ? dt_c : dt_o_d, bias);
      v.hi = __fmul_rn(dl, Ah);
    }
    v = warp_scan_df(v, j);
    // Gram rows of the drafts: g[k][s] = C_{h0+k} . B_s for s <= h0 + k (Dot<128> order)
    for (int k = 0; k < Td; ++k) {
      float ck[4];
      Quad<T>::unpack(*reinterpret_cast<const uint2*>(sm.ct + sw128(kRTM, k, 4 * j)), ck);
      for (int s = w; s <= h0 + k; s += kRWarps) {
        float bs[4];
        lds4(sm.b + (s < h0 ? s : kRQM + s - h0) * kRN + 4 * j, bs);
        const float gv = Dot<kRN>::reduce(Dot<kRN>::partial(ck, bs));
        if (j == 0) sm.g[k * kRRows + s] = gv;
      }
    }
    tc::named_sync(1, kRMath);   // Gram rows complete (math warps only)
    T* y = (T*)a.y + (size_t)i * Td * HP + (size_t)h * kRP;
    auto out = [&](int r) {
      mbar_wait(&sm.done[r], 0, a.status, lim);   // bounded; a wait that gave up has reported ERS_ETIMEOUT
      tc::after_sync();
      if (active) {
        float dv[kRTM];
        tc::tmem_ld16(tc::taddr(sm.tmem, 32 * (w & 3), 16 * (2 * r + (w >> 2))), dv);
        out_round(sm, dv, w, j, r, h0, Td, dl, v, Dh, y, HP);
      }
    };
    if (tma) {
      out(0);
      out(1);
    } else {   // a flushing slot: fold, write back and recast each round's anchor rows into the ring
      float dc = 0.f;
      df vc = {0.f, 0.f};
      if (j < hc) {
        dc = delta_of(dt_c, bias);
        vc.hi = __fmul_rn(dc, Ah);
      }
      vc = warp_scan_df(vc, j);
      const df last = {__shfl_sync(kFull, vc.hi, hc - 1), __shfl_sync(kFull, vc.lo, hc - 1)};
      const float wl = j < hc ? __fmul_rn(dc, expf(df_diff(last, vc))) : 0.f;   // state_weights
      const float decay = expf(last.hi);
      AT* Hd = reinterpret_cast<AT*>(a.state) + soff;
      T* R = (T*)a.read_copy + soff;
      const SrCtr sr{a.sr_key0, a.sr_key1, a.sr_nonce, (uint32_t)slot};
      if (active) flush_round<AT>(sm, Hd, R, w, j, 0, hc, wl, decay, sr, (uint32_t)(h * kRP));
      rows_ready(sm, 0, j);
      mbar_wait(&sm.done[0], 0, a.status, lim);   // round 0's MMAs have read the ring
      if (active) flush_round<AT>(sm, Hd, R, w, j, 1, hc, wl, decay, sr, (uint32_t)(h * kRP));
      rows_ready(sm, 1, j);
      out(0);
      out(1);
    }
    if (active) {   // the drafts go to buffer rows h0..h0+Td-1 (B/C once per group)
      for (int k = 0; k < Td; ++k) {
        T* dx = (T*)a.bx + buf_row(a, slot, h0 + k) * HP + (size_t)h * kRP;
        for (int d = j; d < kRP; d += 32) dx[d] = sx[(kRQM + k) * kRP + d];
      }
      if (j < Td) a.bdt[buf_row(a, slot, h0 + j) * a.H + h] = dt_d;
    }
    for (int k = w; k < Td; k += kRWarps) {   // the group's B and C rows from shared memory, 4 values a lane
      const size_t dst = buf_row(a, slot, h0 + k) * GN + (size_t)g * kRN + 4 * j;
      *reinterpret_cast<uint2*>((T*)a.bB + dst) = *reinterpret_cast<const uint2*>(sm.b + (kRQM + k) * kRN + 4 * j);
      *reinterpret_cast<uint2*>((T*)a.bC + dst) = *reinterpret_cast<const uint2*>(sm.ct + sw128(kRTM, k, 4 * j));
    }
  }
  tc::before_sync();
  __syncthreads();   // every TMEM read is done; no MMA or copy in flight
  if (w == kRIssuer) {
    tc::after_sync();
    tc::tmem_dealloc(sm.tmem, kRTmemCols);
  }
}

// ---- host side ---------------------------------------------------------------------------------------
// 4-D map over a bf16 read copy [heads, P = 64, N = 128] (heads = slots x H): dims {N, 32, 2, heads}
// (a head's rows as two halves of 32), box {64, 32, 1, 4}: one K half of 32 rows of 4 heads.
bool encode_copy_map(CUtensorMap* m, const void* base, long long heads) {
  EncodeTiledFn fn = tma_encode_fn();
  if (fn == nullptr || heads <= 0) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kRN, 32, 2, (cuuint64_t)heads};
  const cuuint64_t strides[3] = {(cuuint64_t)kRN * 2, 32ull * kRN * 2, 64ull * kRN * 2};
  const cuuint32_t box[4] = {64, 32, 1, 4};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// split: the call may flush (a fused decode flush, or a verify with ERS_FLAG_AUTO_FLUSH): two launches.
template <typename AT>
cudaError_t launch_rssm(const LaunchArgs& a, const CUtensorMap& map, int T, bool decode, bool split, cudaStream_t s) {
  constexpr size_t sm = rsm_smem_bytes();
  auto k = k_rssm_tc<AT>;
  cudaError_t e = prep(k, sm);
  if (e != cudaSuccess) return e;
  // the largest shared-memory carveout: two CTAs per SM (the default follows the occupancy rule for
  // kernels that allocate tensor memory, one CTA per SM, and leaves room for one)
  e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.G, a.nseq);
  const int dec = decode ? 1 : 0;
  if (!split) {
    k<<<grid, kRThreads, sm, s>>>(a, map, T, dec, (int)kPartAll);
    return cudaGetLastError();
  }
  k<<<grid, kRThreads, sm, s>>>(a, map, T, dec, (int)kPartFlushes);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a, map, T, dec, (int)kPartPlain);
}

}  // namespace

bool rssm_tc_supported(int io, int P, int N, int Q, int H, int G, int read_dtype, int anchor_dtype) {
  return io == ERS_DTYPE_BF16 && read_dtype == ERS_READ_BF16 && anchor_dtype != ERS_ANCHOR_NVFP4_SHARED_SR &&
         P == kRP && N == kRN && Q >= 1 && Q <= kRQM && G > 0 && H % G == 0 && H / G <= kRWarps;
}

cudaError_t rssm_tc(const LaunchArgs& a, int T, bool decode, cudaStream_t s) {
  if (a.read_copy == nullptr || T < 1 || T > a.Q || (decode && T != 1)) return cudaErrorInvalidValue;
  if (a.nseq == 0) return cudaSuccess;
  const bool split = decode ? (a.flags & ERS_FLAG_FUSE_REFRESH) != 0 : (a.flags & ERS_FLAG_AUTO_FLUSH) != 0;
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  if (!encode_copy_map(&map, a.read_copy, (long long)a.nslots * a.H)) return cudaErrorNotSupported;
  if (a.read_fp8 || a.read_nvfp4 || a.anchor_shared) return cudaErrorNotSupported;
  if (a.anchor_f16) return launch_rssm<__half>(a, map, T, decode, split, s);
  return launch_rssm<float>(a, map, T, decode, split, s);
}

}  // namespace ers
