// Single-pass tensor-core SSD scan (prefill and chunked prefill) for bf16 io, P = 64, N = 128,
// chunk Q a multiple of 16 in [64, 256].
//
// The chunked scan of the exact-replay RFC (vLLM issue 55524), section 1, with the inter-chunk
// state passing of Evidence item 4 (fp32 inside one call, rounded only on store), in ONE launch:
// a CTA per (chunk c, sequence i, head h) unit
//   1. loads the chunk's x, B and C rows once (TMA, 128-byte swizzled tiles) and scans its decays,
//   2. issues the Gram MMAs of both 128-row t-tiles, builds the state operand and runs the chunk
//      state MMAs S_c = sum_s B_s (w_s x_s),
//   3. publishes S_c and its decay factor e_c = exp(Acum_last) for later chunks of (i, h),
//   4. builds the first t-tile's masked decayed Gram and issues its diagonal MMAs,
//   5. looks back over the earlier chunks of (i, h) for the start state H_c: from the nearest
//      chunk that has published its end state H_{k+1}, H <- fma(e_j, H, S_j) for j = k+1 .. c-1,
//      and publishes its own end state H_{c+1} = fma(e_c, H_c, S_c),
//   6. splits H_c into the [H_hi; H_lo] operand tile and finishes both t-tiles (off-diagonal MMAs,
//      remaining diagonal blocks, epilogue).
// The chain is evaluated in the canonical order (one fma per chunk, chunks in order) whichever
// chunk the look-back stops at, and every MMA shape, operand value and K order is the one the
// tensor-core decode, refresh and verify kernels issue (tc_engine.cuh), so every path keeps the
// bits of this scan.  Waits on other CTAs are bounded (ERS_ETIMEOUT); units are numbered chunk-major
// so that every chunk a CTA waits for belongs to a CTA launched before it.
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "ers_common.cuh"
#include "ers_internal.h"
#include "tc_engine.cuh"

namespace ers {

struct ScanMaps {
  CUtensorMap x;   // [T, H, P] bf16 as a 3-D map {P, H, T}, box {64, 1, Q}, 128-byte swizzle
  CUtensorMap B;   // [T, G, N] bf16 as {N, G, T}, box {64, 1, Q}
  CUtensorMap C;
};

namespace {

using bf16 = __nv_bfloat16;
using namespace tc;

constexpr int kScanWarps = 32;
constexpr int kScanThreads = kScanWarps * 32;
constexpr int kSlices = kScanWarps / 4;   // column slices per TMEM lane quarter
constexpr int kMC = 128 / kSlices;        // M-tile columns per warp
constexpr int kOC = 64 / kSlices;         // output columns / state rows per thread
constexpr uint32_t kScanTmemCols = 512;
// TMEM columns: [0, 128) Gram of t-tile 0, then its diagonal sums (hi [0, 64), lo [64, 128));
// [128, 384) Gram of t-tile 1, then its diagonal sums in [128, 256) and its off-diagonal sums in
// [256, 384); [384, 448) the chunk state S^T, then [384, 512) t-tile 0's off-diagonal sums.
constexpr uint32_t kColG1 = 128, kColState = 384, kColOff = 384, kColOff1 = 256;

struct ScanHdr {
  uint64_t bar_tma, bar_c, bar_gram, bar_state, bar_diag[2], bar_off;
  uint32_t tmem;
  int32_t lb_stop;   // look-back: the chunk whose published end state starts the chain
  int32_t lb_ok;
  alignas(16) float delta[kQMax];
  alignas(16) float ahi[kQMax];
  alignas(16) float alo[kQMax];
  alignas(16) float w[kQMax];
};

extern __shared__ __align__(1024) unsigned char scan_smem[];

constexpr size_t kScanHdrBytes = (sizeof(ScanHdr) + 1023) & ~size_t(1023);
constexpr uint32_t kUTile = 128u * 128u;   // one bf16 U term: 128 rows x 64 d

// Shared-memory arena: header | X [Q x 64] | B region max(Q x 128, M tile) | C region max(Q x 128,
// M tile) | U (3 terms).  Once the Gram MMAs are done the C region holds the second K block's state
// operand, then M tiles (hi, lo: 2 x 128 x 128 bf16) alternate between the B and C regions, and the
// C tile is reloaded for the off-diagonal MMAs; the [H_hi; H_lo] tile reuses the U region.
struct ScanArena {
  ScanHdr* hd;
  uint8_t* X;
  uint8_t* B;
  uint8_t* C;
  uint8_t* U;
};
__host__ __device__ __forceinline__ size_t scan_b_bytes(int Q) {
  const size_t b = (size_t)Q * 256;
  return b > 65536 ? b : 65536;
}
__host__ __device__ __forceinline__ size_t scan_smem_bytes(int Q) {
  return 1024 + kScanHdrBytes + (size_t)Q * 128 + 2 * scan_b_bytes(Q) + 3 * kUTile;
}
__device__ __forceinline__ ScanArena scan_arena(int Q) {
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(scan_smem) + 1023) & ~uintptr_t(1023));
  ScanArena ar;
  ar.hd = reinterpret_cast<ScanHdr*>(base);
  ar.X = base + kScanHdrBytes;
  ar.B = ar.X + (size_t)Q * 128;
  ar.C = ar.B + scan_b_bytes(Q);
  ar.U = ar.C + scan_b_bytes(Q);
  return ar;
}

__device__ __forceinline__ size_t unit_index(const LaunchArgs& a, int i, int c, int h) {
  return ((size_t)i * a.max_chunks + c) * a.H + h;
}

// Waits for an MMA group's completion on all threads; false on timeout (reported).
__device__ __forceinline__ bool mma_done(uint64_t* bar, uint32_t parity, const LaunchArgs& a) {
  const bool ok = __syncthreads_and(mbar_wait(bar, parity, a.status, a.wait_ns));
  after_sync();
  return ok;
}

// Rows [r0, Q) of the X, B and C tiles as zeros (generic-proxy stores; the caller fences).
__device__ __forceinline__ void zero_rows(const ScanArena& ar, int Q, int r0) {
  for (int id = threadIdx.x; id < (Q - r0) * 40; id += kScanThreads) {
    const int r = r0 + id / 40, k = id % 40;
    uint8_t* dst = k < 8 ? ar.X + sw128(1, r, 8 * k)
                         : (k < 24 ? ar.B + sw128(Q, r, 8 * (k - 8)) : ar.C + sw128(Q, r, 8 * (k - 24)));
    *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
}

// X, B and C rows by cp.async from `rows` (buffer rows and/or tokens), zeros from row nrows on.
__device__ __forceinline__ void load_rows_async(const ScanArena& ar, const Rows<bf16>& rows, int Q, int nrows) {
  for (int id = threadIdx.x; id < Q * 40; id += kScanThreads) {
    const int r = id / 40, k = id % 40;
    uint8_t* dst = k < 8 ? ar.X + sw128(1, r, 8 * k)
                         : (k < 24 ? ar.B + sw128(Q, r, 8 * (k - 8)) : ar.C + sw128(Q, r, 8 * (k - 24)));
    if (r < nrows) {
      const bf16* src = k < 8 ? rows.x(r) + 8 * k : (k < 24 ? rows.B(r) + 8 * (k - 8) : rows.C(r) + 8 * (k - 24));
      cp_async16(dst, src);
    } else {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
}

// Masked decayed Gram block `blk` of t-tile tau into the M tile at `mt` (hi, then lo 32 KB on),
// from Gram columns [gcol, gcol + 128): every warp handles one TMEM lane quarter (rows) and a
// kMC-column slice.
__device__ __forceinline__ void build_m(const ScanArena& ar, uint8_t* mt, uint32_t tb, uint32_t gcol, int Q, int tau,
                                       int blk, int nrows) {
  const Geom ge = geom(Q, tau);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3, sl = warp >> 2;
  const int row = 32 * q + lane;
  const int width = ge.S_ext - 128 * blk < 128 ? ge.S_ext - 128 * blk : 128;
  const int tlim = nrows < ge.t0 + ge.TT ? nrows : ge.t0 + ge.TT;
  if (kMC * sl < width) {
    float g[kMC];
    tmem_ld16(taddr(tb, 32 * q, gcol + kMC * sl), g);
    m_row<kMC>(g, ge.t0 + row, tlim, blk, kMC * sl, ge.S_ext, ar.hd->delta, ar.hd->ahi, ar.hd->alo, mt, mt + 32768,
               128, row);
  }
}

// Outputs of t-tile tau, rows [out_lo, out_hi): y = fma(D, x, exp(Acum_t) (Yoff_hi + Yoff_lo) +
// (Ydiag_hi + Ydiag_lo)), kOC consecutive d per thread.
__device__ __forceinline__ void epilogue(const ScanArena& ar, uint32_t tb, uint32_t dcol, uint32_t ocol, int Q, int tau,
                                         int out_lo, int out_hi, float Dh, bf16* y, long long tok0, int H, int h) {
  const Geom ge = geom(Q, tau);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3, sl = warp >> 2;
  const int row = 32 * q + lane;
  const int t = ge.t0 + row;
  float oh[kOC], ol[kOC], dh[kOC], dl[kOC];
  tmem_ld8(taddr(tb, 32 * q, ocol + kOC * sl), oh);
  tmem_ld8(taddr(tb, 32 * q, ocol + 64 + kOC * sl), ol);
  tmem_ld8(taddr(tb, 32 * q, dcol + kOC * sl), dh);
  tmem_ld8(taddr(tb, 32 * q, dcol + 64 + kOC * sl), dl);
  if (t < out_lo || t >= out_hi || row >= ge.TT) return;
  const float et = expf(ar.hd->ahi[t]);
  const uint4 xr = *reinterpret_cast<const uint4*>(ar.X + sw128(1, t, kOC * sl));
  const bf16* xv = reinterpret_cast<const bf16*>(&xr);
  uint32_t packed[kOC / 2];
#pragma unroll
  for (int e = 0; e < kOC; e += 2) {
    const float o0 = combine_out(et, __fadd_rn(oh[e], ol[e]), __fadd_rn(dh[e], dl[e]), Dh, __bfloat162float(xv[e]));
    const float o1 =
        combine_out(et, __fadd_rn(oh[e + 1], ol[e + 1]), __fadd_rn(dh[e + 1], dl[e + 1]), Dh, __bfloat162float(xv[e + 1]));
    packed[e / 2] = pack_bf16x2(o0, o1);
  }
  *reinterpret_cast<uint4*>(y + ((tok0 + t) * H + h) * P + kOC * sl) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

// Publishes `value` in a unit's flag after every thread's stores before this call (one fence).
__device__ __forceinline__ void publish_flag(int32_t* flag, int32_t value) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    st_release(flag, value);
  }
}

// The C tile again (its region held operands in between): TMA, or cp.async from `rows`.
__device__ __forceinline__ void reload_c(const ScanArena& ar, const ScanMaps& maps, const Rows<bf16>& rows, bool tma,
                                         int Q, int nrows, int g, int z, uint64_t* bar) {
  if (tma) {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(bar, (uint32_t)Q * 256u);
      tma_load_3d(ar.C, &maps.C, 0, g, z, bar);
      tma_load_3d(ar.C + Q * 128, &maps.C, 64, g, z, bar);
    }
  } else {
    for (int id = threadIdx.x; id < Q * 16; id += kScanThreads) {
      const int r = id / 16, k = id % 16;
      uint8_t* dst = ar.C + sw128(Q, r, 8 * k);
      if (r < nrows) cp_async16(dst, rows.C(r) + 8 * k);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
}

template <bool CHUNKED>
__global__ void __launch_bounds__(kScanThreads, 1)
    k_tc_scan(const __grid_constant__ LaunchArgs a, const __grid_constant__ ScanMaps maps, int use_tma) {
  const int per_chunk = a.nseq * a.H;
  const int c = (int)(blockIdx.x / per_chunk);
  const int rem = (int)(blockIdx.x - (unsigned)c * per_chunk);
  const int i = rem / a.H, h = rem - (rem / a.H) * a.H;
  SeqGrid sg;
  if (!seq_grid(a, CHUNKED, i, &sg)) return;
  const int tid = threadIdx.x;
  const size_t hs = (size_t)P * N;
  const int warp = tid / 32, lane = tid % 32;
  const int q = warp & 3, sl = warp >> 2;
  const int n = 32 * q + lane;   // state column owned by this thread
  const int d0 = kOC * sl;       // and its kOC state rows d0 ..
  if (sg.nch == 0) {             // empty sequence: the final state is the initial one
    if (!CHUNKED && c == 0) {
      const float* init = a.init_state ? a.init_state + ((size_t)i * a.H + h) * hs : nullptr;
      float* fs = a.final_state + ((size_t)i * a.H + h) * hs;
      for (int e = tid; e < (int)hs; e += kScanThreads) fs[e] = init ? init[e] : 0.f;
    }
    return;
  }
  if (c >= sg.nch) return;
  const int Q = a.Q;
  const int nrows = min(Q, sg.total - c * Q);
  const int nbuf = max(0, sg.p - c * Q);
  if (nbuf >= nrows) return;   // a resumed slot's partial chunk with no new token: nothing changes
  const long long tok0 = (long long)a.cu[i] + (long long)c * Q - sg.p;
  const int g = h / (a.H / a.G);
  const size_t unit = unit_index(a, i, c, h);
  const ScanArena ar = scan_arena(Q);
  ScanHdr& hd = *ar.hd;
  const bool tma = use_tma != 0 && nbuf == 0;
  const int ntiles = (Q + 127) / 128;
  const int K = (nrows + 15) & ~15;
  const bool two_state_blocks = K > 128;
  if (tid == 0) {
    mbar_init(&hd.bar_tma, 1);
    mbar_init(&hd.bar_c, 1);
    mbar_init(&hd.bar_gram, 1);
    mbar_init(&hd.bar_state, 1);
    mbar_init(&hd.bar_diag[0], 1);
    mbar_init(&hd.bar_diag[1], 1);
    mbar_init(&hd.bar_off, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&hd.tmem, kScanTmemCols);
  before_sync();
  __syncthreads();
  after_sync();
  const uint32_t tb = hd.tmem;
  // ---- 1. token tiles and decays -------------------------------------------------------------------
  if (tma) {
    if (tid == 0) {
      const int z = (int)tok0;
      mbar_arrive_expect_tx(&hd.bar_tma, (uint32_t)Q * 640u);
      tma_load_3d(ar.X, &maps.x, 0, h, z, &hd.bar_tma);
      tma_load_3d(ar.B, &maps.B, 0, g, z, &hd.bar_tma);
      tma_load_3d(ar.B + Q * 128, &maps.B, 64, g, z, &hd.bar_tma);
      tma_load_3d(ar.C, &maps.C, 0, g, z, &hd.bar_tma);
      tma_load_3d(ar.C + Q * 128, &maps.C, 64, g, z, &hd.bar_tma);
    }
  } else {
    load_rows_async(ar, make_rows<bf16>(a, sg.slot, h, nbuf, tok0), Q, nrows);
  }
  if (tid < kQMax) {
    float dl = 0.f, da = 0.f;
    if (tid < nrows) {
      dl = delta_of(make_rows<bf16>(a, sg.slot, h, nbuf, tok0).dt(tid), a.dt_bias[h]);
      da = __fmul_rn(dl, a.A[h]);
    }
    hd.delta[tid] = dl;
    hd.ahi[tid] = da;
    hd.alo[tid] = 0.f;
  }
  __syncthreads();
  chunk_scan(hd.ahi, hd.alo);
  bool ok = true;
  if (tma) {
    ok = mbar_wait(&hd.bar_tma, 0, a.status, a.wait_ns);
    if (nrows < Q) zero_rows(ar, Q, nrows);   // the box reads the next tokens (or zeros) there
  }
  if (tid < nrows) {   // chunk-state weights w_s = delta_s exp(Acum_last - Acum_s)
    const df last = {hd.ahi[nrows - 1], hd.alo[nrows - 1]};
    hd.w[tid] = __fmul_rn(hd.delta[tid], expf(df_diff(last, df{hd.ahi[tid], hd.alo[tid]})));
  }
  publish();
  ok = __syncthreads_and(ok);
  // ---- 2. Gram MMAs of every t-tile; chunk state (its second K block's operand in the C region) ------
  if (ok && tid == 0) {
    issue_gram(tb, smem_u32(ar.C), Q, 1024, smem_u32(ar.B), Q, geom(Q, 0).S_ext);
    if (ntiles > 1) issue_gram(tb + kColG1, smem_u32(ar.C + 128 * 128), Q, 1024, smem_u32(ar.B), Q, geom(Q, 1).S_ext);
    commit(&hd.bar_gram);
  }
  if (ok) {
    build_u_tiles(ar.X, hd.w, nrows, 0, K < 128 ? K : 128, ar.U, ar.U + kUTile, ar.U + 2 * kUTile);
    publish();
    if (tid == 0)
      issue_state_block(tb + kColState, smem_u32(ar.B), Q, smem_u32(ar.U), smem_u32(ar.U + kUTile),
                        smem_u32(ar.U + 2 * kUTile), 0, (K < 128 ? K : 128) / 16);
    ok = mma_done(&hd.bar_gram, 0, a);   // the C tile is free from here until it is reloaded
  }
  if (ok && two_state_blocks) {
    build_u_tiles(ar.X, hd.w, nrows, 128, K - 128, ar.C, ar.C + kUTile, ar.C + 2 * kUTile);
    publish();
    if (tid == 0)
      issue_state_block(tb + kColState, smem_u32(ar.B), Q, smem_u32(ar.C), smem_u32(ar.C + kUTile),
                        smem_u32(ar.C + 2 * kUTile), 128, (K - 128) / 16);
  }
  if (ok && tid == 0) commit(&hd.bar_state);
  if (ok) ok = mma_done(&hd.bar_state, 0, a);
  // ---- 3. publish: chunk 0 its end state H_1 at once (H_0 is known), later chunks their S_c and e_c --
  // Published states are laid out [n][d] (each thread's kOC values contiguous); the public outputs
  // (chunk states, final state, checkpoint) keep the [d][n] layout.  S_c stays in TMEM until the
  // off-diagonal MMAs, so no register holds it across the diagonal work.
  const bool has_next = c + 1 < sg.nch;
  auto store_end_state = [&](const float (&Hn)[kOC]) {
    if (has_next) {
      float4* wi = reinterpret_cast<float4*>(a.ws_incl + unit * hs + (size_t)n * P + d0);
      wi[0] = make_float4(Hn[0], Hn[1], Hn[2], Hn[3]);
      wi[1] = make_float4(Hn[4], Hn[5], Hn[6], Hn[7]);
    }
    float* out = nullptr;
    if (!CHUNKED && a.chunk_states != nullptr) out = a.chunk_states + unit * hs;
    if (!CHUNKED && c == sg.nch - 1) {
      float* fs = a.final_state + ((size_t)i * a.H + h) * hs;
#pragma unroll
      for (int j = 0; j < kOC; ++j) fs[(d0 + j) * N + n] = Hn[j];
    }
    if (CHUNKED && c + 1 == sg.total / Q) out = a.state + ((size_t)sg.slot * a.H + h) * hs;   // new checkpoint
    if (out != nullptr) {
#pragma unroll
      for (int j = 0; j < kOC; ++j) out[(d0 + j) * N + n] = Hn[j];
    }
  };
  // the [H_hi; H_lo] operand tile of the start state (U region: the state MMAs are done)
  auto store_h_tile = [&](const float (&Hc)[kOC]) {
#pragma unroll
    for (int j = 0; j < kOC; ++j) {
      const bf16 hi = __float2bfloat16_rn(Hc[j]);
      const bf16 lo = __float2bfloat16_rn(__fsub_rn(Hc[j], __bfloat162float(hi)));
      *reinterpret_cast<bf16*>(ar.U + sw128(128, d0 + j, n)) = hi;
      *reinterpret_cast<bf16*>(ar.U + sw128(128, P + d0 + j, n)) = lo;
    }
  };
  if (ok && c == 0) {
    float S[kOC], Hc[kOC], Hn[kOC];
    tmem_ld8(taddr(tb, 32 * q, kColState + d0), S);
    const float e_c = expf(hd.ahi[nrows - 1]);
    const float* init = CHUNKED ? a.state + ((size_t)sg.slot * a.H + h) * hs
                                : (a.init_state ? a.init_state + ((size_t)i * a.H + h) * hs : nullptr);
#pragma unroll
    for (int j = 0; j < kOC; ++j) Hc[j] = init ? init[(d0 + j) * N + n] : 0.f;
#pragma unroll
    for (int j = 0; j < kOC; ++j) Hn[j] = __fmaf_rn(e_c, Hc[j], S[j]);
    store_end_state(Hn);
    store_h_tile(Hc);
    if (has_next) publish_flag(a.ws_flags + unit, 2);
  }
  if (ok && c > 0 && has_next) {
    float S[kOC];
    tmem_ld8(taddr(tb, 32 * q, kColState + d0), S);
    const float e_c = expf(hd.ahi[nrows - 1]);
    float4* ws = reinterpret_cast<float4*>(a.ws_states + unit * hs + (size_t)n * P + d0);
    ws[0] = make_float4(S[0], S[1], S[2], S[3]);
    ws[1] = make_float4(S[4], S[5], S[6], S[7]);
    if (tid == 0) a.ws_tot[unit] = e_c;
    publish_flag(a.ws_flags + unit, 1);
  }
  // ---- 4. every diagonal block (needs no start state), M tiles alternating between the B and C ------
  // regions; accumulators: t-tile 0 in [0, 128), t-tile 1 in [128, 256) over the Gram block each uses.
  uint32_t ph_diag[2] = {0, 0};
  bool pend[2] = {false, false};
  int jb = 0;
  for (int tau = 0; tau < ntiles && ok; ++tau) {
    const Geom ge = geom(Q, tau);
    const uint32_t dcol = tau == 0 ? 0u : kColG1;
    for (int blk = 0; blk < ge.nblk && ok; ++blk, ++jb) {
      const int bi = jb & 1;
      uint8_t* mt = bi == 0 ? ar.B : ar.C;
      if (pend[bi]) {   // the diagonal MMAs two blocks back still read this M tile
        ok = mma_done(&hd.bar_diag[bi], ph_diag[bi], a);
        ph_diag[bi] ^= 1;
        pend[bi] = false;
        if (!ok) break;
      }
      build_m(ar, mt, tb, dcol + 128 * blk, Q, tau, blk, nrows);
      publish();
      if (tid == 0) {
        issue_ydiag(tb + dcol, smem_u32(mt), 128, 1024, smem_u32(ar.X), blk, ge.S_ext);
        issue_ydiag(tb + dcol + 64, smem_u32(mt + 32768), 128, 1024, smem_u32(ar.X), blk, ge.S_ext);
        commit(&hd.bar_diag[bi]);
      }
      pend[bi] = true;
    }
  }
  // the C tile comes back once nothing reads its region (state operand, M tile)
  const bool c_used = two_state_blocks || jb > 1;
  bool c_pending = false;   // a TMA reload of the C tile is in flight
  if (ok && c_used) {
    if (pend[1]) {
      ok = mma_done(&hd.bar_diag[1], ph_diag[1], a);
      ph_diag[1] ^= 1;
      pend[1] = false;
    }
    if (ok) {
      reload_c(ar, maps, make_rows<bf16>(a, sg.slot, h, nbuf, tok0), tma, Q, nrows, g, (int)tok0, &hd.bar_c);
      c_pending = tma;
    }
  }
  // ---- 5. start state H_c of a later chunk: look back over the earlier chunks, publish H_{c+1} --------
  if (ok && c > 0) {
    // warp 0: lane l watches chunk top - l, 32 chunks per window, from c - 1 down; the chain starts
    // at the nearest chunk that has published its end state, once every chunk above it has
    // published its chunk state (chunk 0 publishes its end state, never its chunk state)
    if (warp == 0) {
      int top = c - 1, k0 = -1, good = 1;
      while (good && k0 < 0) {
        const int k = top - lane;
        int32_t f = 2;
        if (k >= 0) f = flag_wait(a.ws_flags + unit_index(a, i, k, h), a.status, a.wait_ns);
        if (!__all_sync(kFull, f != 0)) {
          good = 0;
          break;
        }
        const unsigned inc = __ballot_sync(kFull, k >= 0 && f == 2);
        if (inc != 0) k0 = top - (__ffs(inc) - 1);
        else if (top < 32) good = 0;
        top -= 32;
      }
      if (lane == 0) {
        hd.lb_stop = k0;
        hd.lb_ok = good;
      }
    }
    __syncthreads();
    ok = hd.lb_ok != 0;
    if (ok) {
      float Hc[kOC];
      const int k0 = hd.lb_stop;
      const float4* Hk = reinterpret_cast<const float4*>(a.ws_incl + unit_index(a, i, k0, h) * hs + (size_t)n * P + d0);
      const float4 v0 = __ldcg(Hk), v1 = __ldcg(Hk + 1);
      Hc[0] = v0.x; Hc[1] = v0.y; Hc[2] = v0.z; Hc[3] = v0.w;
      Hc[4] = v1.x; Hc[5] = v1.y; Hc[6] = v1.z; Hc[7] = v1.w;
      for (int kk = k0 + 1; kk < c; kk += 2) {   // two chunks' loads in flight
        float4 sv[2][2];
        float ev[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          ev[u] = 0.f;
          if (kk + u < c) {
            const size_t uk = unit_index(a, i, kk + u, h);
            ev[u] = __ldcg(a.ws_tot + uk);
            const float4* Sk = reinterpret_cast<const float4*>(a.ws_states + uk * hs + (size_t)n * P + d0);
            sv[u][0] = __ldcg(Sk);
            sv[u][1] = __ldcg(Sk + 1);
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (kk + u < c) {
            const float sx[kOC] = {sv[u][0].x, sv[u][0].y, sv[u][0].z, sv[u][0].w,
                                   sv[u][1].x, sv[u][1].y, sv[u][1].z, sv[u][1].w};
#pragma unroll
            for (int j = 0; j < kOC; ++j) Hc[j] = __fmaf_rn(ev[u], Hc[j], sx[j]);
          }
        }
      }
      float S[kOC], Hn[kOC];
      tmem_ld8(taddr(tb, 32 * q, kColState + d0), S);
      const float e_c = expf(hd.ahi[nrows - 1]);
#pragma unroll
      for (int j = 0; j < kOC; ++j) Hn[j] = __fmaf_rn(e_c, Hc[j], S[j]);
      store_end_state(Hn);
      store_h_tile(Hc);
      if (has_next) publish_flag(a.ws_flags + unit, 2);
    }
  }
  // ---- 6. off-diagonal MMAs ------------------------------------------------------------------------------
  if (c_pending) {   // waited for even after an error: no copy may land in a finished CTA's memory
    ok = mbar_wait(&hd.bar_c, 0, a.status, a.wait_ns) && ok;
    c_pending = false;
  }
  publish();   // also completes a cp.async reload of the C tile
  ok = __syncthreads_and(ok);
  // t-tile 0 into [384, 512) (the chunk state's columns, read above), t-tile 1 into [256, 384) (its
  // second Gram block, consumed by its M tile).
  if (ok && tid == 0) {
    for (int tau = 0; tau < ntiles; ++tau)
      issue_yoff(tb + (tau == 0 ? kColOff : kColOff1), smem_u32(ar.C + 128 * 128 * tau), Q, 1024, smem_u32(ar.U), 128);
    commit(&hd.bar_off);
  }
  for (int bi = 0; bi < 2 && ok; ++bi) {
    if (pend[bi]) {
      ok = mma_done(&hd.bar_diag[bi], ph_diag[bi], a);
      ph_diag[bi] ^= 1;
      pend[bi] = false;
    }
  }
  if (ok) ok = mma_done(&hd.bar_off, 0, a);
  // ---- 7. epilogues ---------------------------------------------------------------------------------
  const float Dh = a.D[h];
  for (int tau = 0; tau < ntiles && ok; ++tau) {
    const Geom ge = geom(Q, tau);
    epilogue(ar, tb, tau == 0 ? 0u : kColG1, tau == 0 ? kColOff : kColOff1, Q, tau, max(nbuf, ge.t0),
             min(nrows, ge.t0 + ge.TT), Dh, (bf16*)a.y, tok0, a.H, h);
  }
  for (int bi = 0; bi < 2; ++bi)   // no MMA may outlive the TMEM allocation
    if (pend[bi]) mma_done(&hd.bar_diag[bi], ph_diag[bi], a);
  before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, kScanTmemCols);
}

// ---- host side ---------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool looked = false;
  if (!looked) {
    looked = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    cudaGetLastError();
  }
  return fn;
}

// 3-D map over a token-major bf16 tensor [T, R, W] (W contiguous): dims {W, R, T}, box {64, 1, Q}.
bool encode_rows(CUtensorMap* m, const void* base, long long T, int R, int W, int Q) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || T <= 0) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)W, (cuuint64_t)R, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)W * 2, (cuuint64_t)W * R * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)Q};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The kernels' dynamic shared-memory limit, raised to the largest size once per device (a call made
// under stream capture after the first one on its device sets nothing).
cudaError_t smem_attr(bool chunked, size_t bytes) {
  static std::mutex mu;
  static bool done[2][64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[chunked][dev]) return cudaSuccess;
  (void)bytes;
  const int most = (int)scan_smem_bytes(kQMaxHost);
  e = chunked ? cudaFuncSetAttribute(k_tc_scan<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, most)
              : cudaFuncSetAttribute(k_tc_scan<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
  if (e == cudaSuccess) done[chunked][dev] = true;
  return e;
}

}  // namespace

size_t tc_scan_workspace(int nseq, int max_chunks, int H) {
  const size_t units = (size_t)(nseq > 0 ? nseq : 0) * (size_t)(max_chunks > 1 ? max_chunks : 1) * (size_t)H;
  const size_t st = align256(units * (size_t)P * N * sizeof(float));
  return 2 * st + align256(units * sizeof(float)) + align256(units * sizeof(int32_t));
}

void tc_scan_carve(LaunchArgs& a, void* ws) {
  const size_t units = (size_t)a.nseq * (size_t)(a.max_chunks > 1 ? a.max_chunks : 1) * (size_t)a.H;
  const size_t st = align256(units * (size_t)P * N * sizeof(float));
  char* p = (char*)ws;
  a.ws_states = (float*)p;
  a.ws_incl = (float*)(p + st);
  a.ws_tot = (float*)(p + 2 * st);
  a.ws_flags = (int32_t*)(p + 2 * st + align256(units * sizeof(float)));
}

cudaError_t tc_prefill(const LaunchArgs& a0, Op op, cudaStream_t s) {
  const bool chunked = op == Op::kChunkedPrefill;
  LaunchArgs a = a0;
  if (a.max_chunks < 1) a.max_chunks = 1;   // empty sequences still get their final state
  if (a.wait_ns == 0) a.wait_ns = kWaitLimitNs;
  cudaError_t e;
  if (a.nseq > 0) {
    const size_t units = (size_t)a.nseq * a.max_chunks * a.H;
    if (units > 0x7fffffffu) return cudaErrorInvalidValue;
    if ((e = cudaMemsetAsync(a.ws_flags, 0, units * sizeof(int32_t), s)) != cudaSuccess) return e;
    ScanMaps maps;
    memset(&maps, 0, sizeof(maps));
    int use_tma = encode_rows(&maps.x, a.x, a.ntokens, a.H, P, a.Q) && encode_rows(&maps.B, a.B, a.ntokens, a.G, N, a.Q) &&
                  encode_rows(&maps.C, a.C, a.ntokens, a.G, N, a.Q);
    const size_t sm = scan_smem_bytes(a.Q);
    if ((e = smem_attr(chunked, sm)) != cudaSuccess) return e;
    if (chunked)
      k_tc_scan<true><<<(unsigned)units, kScanThreads, sm, s>>>(a, maps, use_tma);
    else
      k_tc_scan<false><<<(unsigned)units, kScanThreads, sm, s>>>(a, maps, use_tma);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (chunked) return launch_tail(a0, s);
  return cudaGetLastError();
}

}  // namespace ers

// ---- bounded waits that run out ---------------------------------------------------------------------
namespace ers {
namespace {

__device__ int32_t never_set_flag;   // zero for the life of the module: nothing writes it

// Block 0 waits on an mbarrier phase that nothing completes, block 1 on a device flag that nothing
// sets; both give up after limit_ns, report ERS_ETIMEOUT through `status` and return.
__global__ void k_wait_selftest(unsigned long long limit_ns, int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  if (blockIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    tc::mbar_wait(&bar, 0, status, limit_ns);
  } else {
    tc::flag_wait(&never_set_flag, status, limit_ns);
  }
}

}  // namespace

cudaError_t wait_selftest(unsigned long long limit_ns, int32_t* status, cudaStream_t s) {
  k_wait_selftest<<<2, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace ers
