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

constexpr int kScanWarps = 16;
constexpr int kScanThreads = kScanWarps * 32;
constexpr uint32_t kScanTmemCols = 512;
// TMEM columns: [0, 128) Gram of t-tile 0, then its diagonal sums (hi [0, 64), lo [64, 128));
// [128, 384) Gram of t-tile 1, then its diagonal sums in [128, 256) and its off-diagonal sums in
// [256, 384); [384, 448) the chunk state S^T, then [384, 512) t-tile 0's off-diagonal sums.
constexpr uint32_t kColG1 = 128, kColState = 384, kColOff = 384, kColOff1 = 256;

struct ScanHdr {
  uint64_t bar_tma, bar_gram, bar_state, bar_diag, bar_off;
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

// Shared-memory arena: header | X [Q x 64] | B region max(Q x 128, M tile) | C [Q x 128] | U (3 terms).
// The M tile (hi, lo: 2 x 128 x 128 bf16) reuses the B region once the Gram and state MMAs are
// done; the [H_hi; H_lo] tile reuses the U region once the state MMAs are done.
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
  return 1024 + kScanHdrBytes + (size_t)Q * 128 + scan_b_bytes(Q) + (size_t)Q * 256 + 3 * kUTile;
}
__device__ __forceinline__ ScanArena scan_arena(int Q) {
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(scan_smem) + 1023) & ~uintptr_t(1023));
  ScanArena ar;
  ar.hd = reinterpret_cast<ScanHdr*>(base);
  ar.X = base + kScanHdrBytes;
  ar.B = ar.X + (size_t)Q * 128;
  ar.C = ar.B + scan_b_bytes(Q);
  ar.U = ar.C + (size_t)Q * 256;
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

// Masked decayed Gram block `blk` of t-tile tau into the M tile (hi, lo), from Gram columns
// [gcol, gcol + 128): every warp handles one TMEM lane quarter (rows) and a 32-column slice.
__device__ __forceinline__ void build_m(const ScanArena& ar, uint32_t tb, uint32_t gcol, int Q, int tau, int blk,
                                       int nrows) {
  const Geom ge = geom(Q, tau);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3, sl = warp >> 2;
  const int row = 32 * q + lane;
  const int width = ge.S_ext - 128 * blk < 128 ? ge.S_ext - 128 * blk : 128;
  const int tlim = nrows < ge.t0 + ge.TT ? nrows : ge.t0 + ge.TT;
  if (32 * sl < width) {
    float g[32];
    tmem_ld32(taddr(tb, 32 * q, gcol + 32 * sl), g);
    m_row<32>(g, ge.t0 + row, tlim, blk, 32 * sl, ge.S_ext, ar.hd->delta, ar.hd->ahi, ar.hd->alo, ar.B,
              ar.B + 32768, 128, row);
  }
}

// Outputs of t-tile tau, rows [out_lo, out_hi): y = fma(D, x, exp(Acum_t) (Yoff_hi + Yoff_lo) +
// (Ydiag_hi + Ydiag_lo)), 16 consecutive d per thread.
__device__ __forceinline__ void epilogue(const ScanArena& ar, uint32_t tb, uint32_t dcol, uint32_t ocol, int Q, int tau,
                                         int out_lo, int out_hi, float Dh, bf16* y, long long tok0, int H, int h) {
  const Geom ge = geom(Q, tau);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3, sl = warp >> 2;
  const int row = 32 * q + lane;
  const int t = ge.t0 + row;
  float oh[16], ol[16], dh[16], dl[16];
  tmem_ld16(taddr(tb, 32 * q, ocol + 16 * sl), oh);
  tmem_ld16(taddr(tb, 32 * q, ocol + 64 + 16 * sl), ol);
  tmem_ld16(taddr(tb, 32 * q, dcol + 16 * sl), dh);
  tmem_ld16(taddr(tb, 32 * q, dcol + 64 + 16 * sl), dl);
  if (t < out_lo || t >= out_hi || row >= ge.TT) return;
  const float et = expf(ar.hd->ahi[t]);
  const uint4 x0 = *reinterpret_cast<const uint4*>(ar.X + sw128(1, t, 16 * sl));
  const uint4 x1 = *reinterpret_cast<const uint4*>(ar.X + sw128(1, t, 16 * sl + 8));
  const bf16* xa = reinterpret_cast<const bf16*>(&x0);
  const bf16* xb = reinterpret_cast<const bf16*>(&x1);
  uint32_t packed[8];
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    float o[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = j + u;
      const float xv = __bfloat162float(e < 8 ? xa[e] : xb[e - 8]);
      o[u] = combine_out(et, __fadd_rn(oh[e], ol[e]), __fadd_rn(dh[e], dl[e]), Dh, xv);
    }
    packed[j / 2] = pack_bf16x2(o[0], o[1]);
  }
  uint4* dst = reinterpret_cast<uint4*>(y + ((tok0 + t) * H + h) * P + 16 * sl);
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
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
  const int d0 = 16 * sl;        // and its 16 state rows d0 .. d0 + 15
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
  const Rows<bf16> rows = make_rows<bf16>(a, sg.slot, h, nbuf, tok0);
  const int g = h / (a.H / a.G);
  const size_t unit = unit_index(a, i, c, h);
  const ScanArena ar = scan_arena(Q);
  ScanHdr& hd = *ar.hd;
  const bool tma = use_tma != 0 && nbuf == 0;
  if (tid == 0) {
    mbar_init(&hd.bar_tma, 1);
    mbar_init(&hd.bar_gram, 1);
    mbar_init(&hd.bar_state, 1);
    mbar_init(&hd.bar_diag, 1);
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
    load_rows_async(ar, rows, Q, nrows);
  }
  if (tid < kQMax) {
    float dl = 0.f, da = 0.f;
    if (tid < nrows) {
      dl = delta_of(rows.dt(tid), a.dt_bias[h]);
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
  const int ntiles = (Q + 127) / 128;
  // ---- 2. Gram MMAs of every t-tile, then the chunk state --------------------------------------------
  if (ok && tid == 0) {
    issue_gram(tb, smem_u32(ar.C), Q, 1024, smem_u32(ar.B), Q, geom(Q, 0).S_ext);
    if (ntiles > 1) issue_gram(tb + kColG1, smem_u32(ar.C + 128 * 128), Q, 1024, smem_u32(ar.B), Q, geom(Q, 1).S_ext);
    commit(&hd.bar_gram);
  }
  uint8_t* u0 = ar.U;
  uint8_t* u1 = ar.U + kUTile;
  uint8_t* u2 = ar.U + 2 * kUTile;
  const int K = (nrows + 15) & ~15;
  uint32_t ph_state = 0;
  for (int s0 = 0; s0 < K && ok; s0 += 128) {
    const int nr = K - s0 < 128 ? K - s0 : 128;
    build_u_tiles(ar.X, hd.w, nrows, s0, nr, u0, u1, u2);
    publish();
    if (tid == 0) {
      issue_state_block(tb + kColState, smem_u32(ar.B), Q, smem_u32(u0), smem_u32(u1), smem_u32(u2), s0, nr / 16);
      commit(&hd.bar_state);
    }
    ok = mma_done(&hd.bar_state, ph_state, a);
    ph_state ^= 1;
  }
  float S[16];
  const float e_c = expf(hd.ahi[nrows - 1]);
  if (ok) tmem_ld16(taddr(tb, 32 * q, kColState + d0), S);
  // ---- 3. publish S_c (and e_c) for the later chunks of (i, h) ----------------------------------------
  // Published states are laid out [n][d] (each thread's 16 values contiguous); the public outputs
  // (chunk states, final state, checkpoint) keep the [d][n] layout.
  const bool has_next = c + 1 < sg.nch;
  if (ok && c > 0 && has_next) {
    float4* ws = reinterpret_cast<float4*>(a.ws_states + unit * hs + (size_t)n * P + d0);
#pragma unroll
    for (int j = 0; j < 4; ++j) ws[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
    if (tid == 0) a.ws_tot[unit] = e_c;
    __threadfence();
  }
  __syncthreads();
  if (ok && c > 0 && has_next && tid == 0) st_release(a.ws_flags + unit, 1);
  // ---- 4. every diagonal block (needs no start state) ------------------------------------------------
  // Accumulators: t-tile 0 in [0, 128), t-tile 1 in [128, 256) over the Gram block each consumes.
  uint32_t ph_diag = 0;
  bool diag_pending = false;
  if (ok) ok = mma_done(&hd.bar_gram, 0, a);
  for (int tau = 0; tau < ntiles && ok; ++tau) {
    const Geom ge = geom(Q, tau);
    const uint32_t dcol = tau == 0 ? 0u : kColG1;
    for (int blk = 0; blk < ge.nblk && ok; ++blk) {
      if (diag_pending) {   // the previous diagonal MMAs still read the M tile
        ok = mma_done(&hd.bar_diag, ph_diag, a);
        ph_diag ^= 1;
        diag_pending = false;
        if (!ok) break;
      }
      build_m(ar, tb, dcol + 128 * blk, Q, tau, blk, nrows);
      publish();
      if (tid == 0) {
        issue_ydiag(tb + dcol, smem_u32(ar.B), 128, 1024, smem_u32(ar.X), blk, ge.S_ext);
        issue_ydiag(tb + dcol + 64, smem_u32(ar.B + 32768), 128, 1024, smem_u32(ar.X), blk, ge.S_ext);
        commit(&hd.bar_diag);
      }
      diag_pending = true;
    }
  }
  // ---- 5. start state H_c: look back over the earlier chunks, then publish H_{c+1} -----------------------
  float Hc[16];
  if (ok) {
    if (c == 0) {
      const float* init = CHUNKED ? a.state + ((size_t)sg.slot * a.H + h) * hs
                                  : (a.init_state ? a.init_state + ((size_t)i * a.H + h) * hs : nullptr);
#pragma unroll
      for (int j = 0; j < 16; ++j) Hc[j] = init ? init[(d0 + j) * N + n] : 0.f;
    } else {
      // warp 0: lane l watches chunk top - l, 32 chunks per window, from c - 1 down; the chain
      // starts at the nearest chunk that has published its end state, once every chunk above it has
      // published its chunk state (chunk 0 publishes only its end state)
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
          else if (top < 32) good = 0;   // no end state at all: cannot happen (chunk 0 publishes one)
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
        const int k0 = hd.lb_stop;
        const float4* Hk = reinterpret_cast<const float4*>(a.ws_incl + unit_index(a, i, k0, h) * hs + (size_t)n * P + d0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 v = __ldcg(Hk + j);
          Hc[4 * j] = v.x; Hc[4 * j + 1] = v.y; Hc[4 * j + 2] = v.z; Hc[4 * j + 3] = v.w;
        }
        for (int kk = k0 + 1; kk < c; kk += 2) {   // two chunks' loads in flight
          float4 sv[2][4];
          float ev[2] = {0.f, 0.f};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (kk + u < c) {
              const size_t uk = unit_index(a, i, kk + u, h);
              ev[u] = __ldcg(a.ws_tot + uk);
              const float4* Sk = reinterpret_cast<const float4*>(a.ws_states + uk * hs + (size_t)n * P + d0);
#pragma unroll
              for (int j = 0; j < 4; ++j) sv[u][j] = __ldcg(Sk + j);
            }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (kk + u < c) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                Hc[4 * j] = __fmaf_rn(ev[u], Hc[4 * j], sv[u][j].x);
                Hc[4 * j + 1] = __fmaf_rn(ev[u], Hc[4 * j + 1], sv[u][j].y);
                Hc[4 * j + 2] = __fmaf_rn(ev[u], Hc[4 * j + 2], sv[u][j].z);
                Hc[4 * j + 3] = __fmaf_rn(ev[u], Hc[4 * j + 3], sv[u][j].w);
              }
            }
          }
        }
      }
    }
  }
  if (ok) {
    float Hn[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) Hn[j] = __fmaf_rn(e_c, Hc[j], S[j]);
    if (has_next) {
      float4* wi = reinterpret_cast<float4*>(a.ws_incl + unit * hs + (size_t)n * P + d0);
#pragma unroll
      for (int j = 0; j < 4; ++j) wi[j] = make_float4(Hn[4 * j], Hn[4 * j + 1], Hn[4 * j + 2], Hn[4 * j + 3]);
      __threadfence();
    }
    float* out = nullptr;
    if (!CHUNKED && a.chunk_states != nullptr) out = a.chunk_states + unit * hs;
    if (!CHUNKED && c == sg.nch - 1) {
      float* fs = a.final_state + ((size_t)i * a.H + h) * hs;
#pragma unroll
      for (int j = 0; j < 16; ++j) fs[(d0 + j) * N + n] = Hn[j];
    }
    if (CHUNKED && c + 1 == sg.total / Q) out = a.state + ((size_t)sg.slot * a.H + h) * hs;   // new checkpoint
    if (out != nullptr) {
#pragma unroll
      for (int j = 0; j < 16; ++j) out[(d0 + j) * N + n] = Hn[j];
    }
    // the [H_hi; H_lo] operand tile (U region: the state MMAs are done)
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const bf16 hi = __float2bfloat16_rn(Hc[j]);
      const bf16 lo = __float2bfloat16_rn(__fsub_rn(Hc[j], __bfloat162float(hi)));
      *reinterpret_cast<bf16*>(ar.U + sw128(128, d0 + j, n)) = hi;
      *reinterpret_cast<bf16*>(ar.U + sw128(128, P + d0 + j, n)) = lo;
    }
  }
  publish();
  if (ok && has_next && tid == 0) st_release(a.ws_flags + unit, 2);
  // ---- 6. off-diagonal sums of every t-tile, then the epilogues ----------------------------------------
  // t-tile 0 into [384, 512) (the chunk state's columns, read above), t-tile 1 into [256, 384) (its
  // second Gram block, consumed by its M tile).
  if (ok && tid == 0) {
    for (int tau = 0; tau < ntiles; ++tau)
      issue_yoff(tb + (tau == 0 ? kColOff : kColOff1), smem_u32(ar.C + 128 * 128 * tau), Q, 1024, smem_u32(ar.U), 128);
    commit(&hd.bar_off);
  }
  if (ok && diag_pending) {
    ok = mma_done(&hd.bar_diag, ph_diag, a);
    ph_diag ^= 1;
    diag_pending = false;
  }
  if (ok) ok = mma_done(&hd.bar_off, 0, a);
  const float Dh = a.D[h];
  for (int tau = 0; tau < ntiles && ok; ++tau) {
    const Geom ge = geom(Q, tau);
    epilogue(ar, tb, tau == 0 ? 0u : kColG1, tau == 0 ? kColOff : kColOff1, Q, tau, max(nbuf, ge.t0),
             min(nrows, ge.t0 + ge.TT), Dh, (bf16*)a.y, tok0, a.H, h);
  }
  if (diag_pending) mma_done(&hd.bar_diag, ph_diag, a);   // no MMA may outlive the TMEM allocation
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
