// Single-pass tensor-core SSD scan (prefill and chunked prefill) for bf16 io, P = 64, N = 128,
// chunk Q a multiple of 16 in [64, 256].
//
// The chunked scan of the exact-replay RFC (vLLM issue 55524), section 1, with the inter-chunk
// state passing of Evidence item 4 (fp32 inside one call, rounded only on store), in ONE launch
// with a CTA per (chunk c, sequence i, head h) unit.  Warp roles:
//   * 16 math warps build every operand tile (state input U, masked decayed Gram M, the start-state
//     tile [H_hi; H_lo]), fold the inter-chunk chain and write the outputs;
//   * the issuer warp loads the token tiles with TMA and issues every tcgen05 MMA as soon as the
//     math warps hand it an operand (a barrier among the math warps, then one mbarrier arrival), so
//     that no math warp waits behind the tensor pipe's queue;
//   * the publisher warp releases this unit's results to later chunks (one device-scope fence each)
//     and polls their flags for the look-back while the math warps build the diagonal tiles.
// Per unit: the token tiles and decays; the Gram MMAs of both 128-row t-tiles; the chunk state
// S_c = sum_s B_s (w_s x_s), published with its decay factor e_c = exp(Acum_last); every diagonal
// block (M tiles alternating between two regions); then the start state H_c from the nearest
// earlier chunk that has published its end state H_{k+1}: H <- fma(e_j, H, S_j) for j = k+1 .. c-1,
// its own end state H_{c+1} = fma(e_c, H_c, S_c) published in turn; the off-diagonal MMAs; the
// epilogue.  Chunk 0 knows H_0 and publishes H_1 right after its chunk state.
// The chain is evaluated in the canonical order (one fma per chunk, chunks in order) whichever
// chunk the look-back stops at, and every MMA shape, operand value and K order is the one the
// tensor-core decode, refresh and verify kernels issue (tc_engine.cuh), so every path keeps the
// bits of this scan.  Every wait is bounded (ERS_ETIMEOUT); units are numbered chunk-major so that
// every chunk a CTA waits for belongs to a CTA launched before it.
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "ers_common.cuh"
#include "ers_internal.h"
#include "tc_engine.cuh"
#include "tma_host.h"

namespace ers {

struct ScanMaps {
  CUtensorMap x;   // [T, H, P] bf16 as a 3-D map {P, H, T}, box {64, 1, Q}, 128-byte swizzle
  CUtensorMap B;   // [T, G, N] bf16 as {N, G, T}, box {64, 1, Q}
  CUtensorMap C;
};

namespace {

using bf16 = __nv_bfloat16;
using namespace tc;

constexpr int kMathWarps = 16;
constexpr int kMath = kMathWarps * 32;               // math threads (named barrier 1)
constexpr int kIssuerWarp = kMathWarps;              // TMA + MMA issue (lane 0)
constexpr int kPubWarp = kMathWarps + 1;             // flag releases and look-back polling
constexpr int kScanThreads = (kMathWarps + 2) * 32;
constexpr int kSlices = kMathWarps / 4;              // column slices per TMEM lane quarter
constexpr int kMC = 128 / kSlices;                   // M-tile columns per math warp
constexpr int kOC = 64 / kSlices;                    // output columns / state rows per math thread
constexpr uint32_t kBarMath = 1;
// Operand hand-offs per unit: token tiles, up to two state operands, up to three M tiles, the
// start-state tile.  Each has its own single-use mbarrier, so that the math warps may run any
// number of hand-offs ahead of the issuer.
constexpr int kMaxHandoffs = 8;
constexpr uint32_t kScanTmemCols = 512;
// TMEM columns: [0, 128) Gram of t-tile 0, then its diagonal sums (hi [0, 64), lo [64, 128));
// [128, 384) Gram of t-tile 1, then its diagonal sums in [128, 256) and its off-diagonal sums in
// [256, 384); [384, 448) the chunk state S^T, then [384, 512) t-tile 0's off-diagonal sums.
constexpr uint32_t kColG1 = 128, kColState = 384, kColOff = 384, kColOff1 = 256;

struct ScanHdr {
  uint64_t bar_tma, bar_c, bar_gram, bar_state, bar_diag[2], bar_off;
  uint64_t bar_ready[kMaxHandoffs];   // math -> issuer: hand-off k's operand is in shared memory
  uint64_t bar_sdone;   // math -> publisher: S_c and e_c are stored
  uint64_t bar_hdone;   // math -> publisher: H_{c+1} is stored
  uint64_t bar_lb;      // publisher -> math: the look-back result is in lb_stop / lb_ok
  uint32_t tmem;
  int32_t lb_stop;      // the chunk whose published end state starts the chain
  int32_t lb_ok;
  alignas(16) float delta[kQMax];
  alignas(16) float ahi[kQMax];
  alignas(16) float alo[kQMax];
  alignas(16) float w[kQMax];
  alignas(16) float shi[kQMax];   // second buffer of the decay scan
  alignas(16) float slo[kQMax];
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

__device__ __forceinline__ void math_sync() { named_sync(kBarMath, kMath); }

// Math threads: their shared-memory writes (generic proxy, cp.async) are complete and visible to
// the tensor core and their TMEM loads are done; after a barrier among them, one arrival on the
// hand-off's own barrier.
__device__ __forceinline__ void hand_off(ScanHdr& hd, int& k) {
  cp_async_wait_all();
  fence_async_smem();
  before_sync();
  math_sync();
  if (threadIdx.x == 0) mbar_arrive(&hd.bar_ready[k]);
  ++k;
}

// Math threads: wait for an MMA group; true unless the wait gave up (reported).
__device__ __forceinline__ bool mma_wait(uint64_t* bar, uint32_t parity, const LaunchArgs& a) {
  const bool ok = mbar_wait(bar, parity, a.status, a.wait_ns);
  after_sync();
  return ok;
}

// Inclusive double-float prefix scan of rows [0, kQMax) among the math threads: the Kogge-Stone
// tree of chunk_scan (strides 1, 2, 4, ..., the same operand order in every df_add), with the
// values of consecutive strides alternating between two buffers so that one barrier per stride
// suffices; the result lands in (hi, lo) and is identical to chunk_scan's.
__device__ __forceinline__ void scan_decays(ScanHdr& hd) {
  const int t = threadIdx.x;
  df v = {0.f, 0.f};
  if (t < kQMax) v = df{hd.ahi[t], hd.alo[t]};
  int k = 0;
#pragma unroll 1
  for (int stride = 1; stride < kQMax; stride <<= 1, ++k) {
    float* bh = (k & 1) ? hd.shi : hd.ahi;
    float* bl = (k & 1) ? hd.slo : hd.alo;
    if (k > 0 && t < kQMax) {
      bh[t] = v.hi;
      bl[t] = v.lo;
    }
    math_sync();
    if (t < kQMax && t >= stride) v = df_add(df{bh[t - stride], bl[t - stride]}, v);
  }
  if (t < kQMax) {   // buffer 0 was last read two strides ago: every math thread is past that
    hd.ahi[t] = v.hi;
    hd.alo[t] = v.lo;
  }
  math_sync();
}

// Rows [r0, Q) of the X and B tiles as zeros (math threads; generic-proxy stores).
__device__ __forceinline__ void zero_rows(const ScanArena& ar, int Q, int r0) {
  for (int id = threadIdx.x; id < (Q - r0) * 24; id += kMath) {
    const int r = r0 + id / 24, k = id % 24;
    uint8_t* dst = k < 8 ? ar.X + sw128(1, r, 8 * k) : ar.B + sw128(Q, r, 8 * (k - 8));
    *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
}

// X, B and C rows by cp.async from `rows` (buffer rows and/or tokens), zeros from row nrows on.
__device__ __forceinline__ void load_rows_async(const ScanArena& ar, const Rows<bf16>& rows, int Q, int nrows,
                                                bool only_c) {
  for (int id = threadIdx.x; id < Q * 40; id += kMath) {
    const int r = id / 40, k = id % 40;
    if (only_c && k < 24) continue;
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
// from Gram columns [gcol, gcol + 128): every math warp handles one TMEM lane quarter (rows) and a
// kMC-column slice.
__device__ __forceinline__ void build_m(const ScanArena& ar, uint8_t* mt, uint32_t tb, uint32_t gcol, int Q, int tau,
                                       int blk, int nrows) {
  const Geom ge = geom(Q, tau);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3, sl = warp >> 2;
  const int row = 32 * q + lane;
  const int width = ge.S_ext - 128 * blk < 128 ? ge.S_ext - 128 * blk : 128;
  const int tlim = nrows < ge.t0 + ge.TT ? nrows : ge.t0 + ge.TT;
#pragma unroll 1
  for (int half = 0; half < kMC / 16; ++half) {   // 16 columns at a time
    const int col0 = kMC * sl + 16 * half;
    if (col0 < width) {
      float g[16];
      tmem_ld16(taddr(tb, 32 * q, gcol + col0), g);
      m_row<16>(g, ge.t0 + row, tlim, blk, col0, ge.S_ext, ar.hd->delta, ar.hd->ahi, ar.hd->alo, mt, mt + 32768, 128,
                row);
    }
  }
}

// Outputs of t-tile tau, rows [out_lo, out_hi): y = fma(D, x, exp(Acum_t) (Yoff_hi + Yoff_lo) +
// (Ydiag_hi + Ydiag_lo)), kOC consecutive d per math thread.
__device__ __forceinline__ void epilogue(const ScanArena& ar, uint32_t tb, uint32_t dcol, uint32_t ocol, int Q, int tau,
                                         int out_lo, int out_hi, float Dh, bf16* y, long long tok0, int H, int h) {
  const Geom ge = geom(Q, tau);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3, sl = warp >> 2;
  const int row = 32 * q + lane;
  const int t = ge.t0 + row;
  float oh[kOC], ol[kOC], dh[kOC], dl[kOC];
  tmem_ld16(taddr(tb, 32 * q, ocol + kOC * sl), oh);
  tmem_ld16(taddr(tb, 32 * q, ocol + 64 + kOC * sl), ol);
  tmem_ld16(taddr(tb, 32 * q, dcol + kOC * sl), dh);
  tmem_ld16(taddr(tb, 32 * q, dcol + 64 + kOC * sl), dl);
  if (t < out_lo || t >= out_hi || row >= ge.TT) return;
  const float et = expf(ar.hd->ahi[t]);
  uint32_t packed[kOC / 2];
#pragma unroll
  for (int e8 = 0; e8 < kOC; e8 += 8) {
    const uint4 xr = *reinterpret_cast<const uint4*>(ar.X + sw128(1, t, kOC * sl + e8));
    const bf16* xv = reinterpret_cast<const bf16*>(&xr);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const int j = e8 + e;
      const float o0 = combine_out(et, __fadd_rn(oh[j], ol[j]), __fadd_rn(dh[j], dl[j]), Dh, __bfloat162float(xv[e]));
      const float o1 = combine_out(et, __fadd_rn(oh[j + 1], ol[j + 1]), __fadd_rn(dh[j + 1], dl[j + 1]), Dh,
                                   __bfloat162float(xv[e + 1]));
      packed[j / 2] = pack_bf16x2(o0, o1);
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(y + ((tok0 + t) * H + h) * P + kOC * sl);
#pragma unroll
  for (int k = 0; k < kOC / 8; ++k) dst[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
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
  if (sg.nch == 0) {   // empty sequence: the final state is the initial one
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
  int nblocks = 0;   // diagonal blocks of all t-tiles
  for (int tau = 0; tau < ntiles; ++tau) nblocks += geom(Q, tau).nblk;
  const bool c_used = two_state_blocks || nblocks > 1;   // the C region holds operands in between
  const bool has_next = c + 1 < sg.nch;
  if (tid == 0) {
    mbar_init(&hd.bar_tma, 1);
    mbar_init(&hd.bar_c, 1);
    mbar_init(&hd.bar_gram, 1);
    mbar_init(&hd.bar_state, 1);
    mbar_init(&hd.bar_diag[0], 1);
    mbar_init(&hd.bar_diag[1], 1);
    mbar_init(&hd.bar_off, 1);
    for (int k = 0; k < kMaxHandoffs; ++k) mbar_init(&hd.bar_ready[k], 1);
    mbar_init(&hd.bar_sdone, kMath);
    mbar_init(&hd.bar_hdone, kMath);
    mbar_init(&hd.bar_lb, 1);
    fence_mbar_init();
  }
  if (warp == kIssuerWarp) tmem_alloc(&hd.tmem, kScanTmemCols);
  before_sync();
  __syncthreads();
  after_sync();
  const uint32_t tb = hd.tmem;

  if (warp == kIssuerWarp) {
    // ================================ issuer: TMA and every MMA =====================================
    if (lane == 0) {
      const int z = (int)tok0;
      if (tma) {
        mbar_arrive_expect_tx(&hd.bar_tma, (uint32_t)Q * 640u);
        tma_load_3d(ar.X, &maps.x, 0, h, z, &hd.bar_tma);
        tma_load_3d(ar.B, &maps.B, 0, g, z, &hd.bar_tma);
        tma_load_3d(ar.B + Q * 128, &maps.B, 64, g, z, &hd.bar_tma);
        tma_load_3d(ar.C, &maps.C, 0, g, z, &hd.bar_tma);
        tma_load_3d(ar.C + Q * 128, &maps.C, 64, g, z, &hd.bar_tma);
      }
      int hk = 0;
      auto ready = [&]() {   // the next operand hand-off of the math threads
        mbar_wait(&hd.bar_ready[hk++], 0, a.status, a.wait_ns);
        after_sync();
      };
      ready();   // token tiles in place (tail rows zeroed)
      issue_gram(tb, smem_u32(ar.C), Q, 1024, smem_u32(ar.B), Q, geom(Q, 0).S_ext);
      if (ntiles > 1) issue_gram(tb + kColG1, smem_u32(ar.C + 128 * 128), Q, 1024, smem_u32(ar.B), Q, geom(Q, 1).S_ext);
      commit(&hd.bar_gram);
      ready();   // first state operand
      issue_state_block(tb + kColState, smem_u32(ar.B), Q, smem_u32(ar.U), smem_u32(ar.U + kUTile),
                        smem_u32(ar.U + 2 * kUTile), 0, (K < 128 ? K : 128) / 16);
      if (two_state_blocks) {
        ready();   // second state operand, in the C region
        issue_state_block(tb + kColState, smem_u32(ar.B), Q, smem_u32(ar.C), smem_u32(ar.C + kUTile),
                          smem_u32(ar.C + 2 * kUTile), 128, (K - 128) / 16);
      }
      commit(&hd.bar_state);
      int jb = 0;
      for (int tau = 0; tau < ntiles; ++tau) {
        const Geom ge = geom(Q, tau);
        const uint32_t dcol = tau == 0 ? 0u : kColG1;
        for (int blk = 0; blk < ge.nblk; ++blk, ++jb) {
          uint8_t* mt = (jb & 1) == 0 ? ar.B : ar.C;
          ready();   // M tile of this block
          issue_ydiag(tb + dcol, smem_u32(mt), 128, 1024, smem_u32(ar.X), blk, ge.S_ext);
          issue_ydiag(tb + dcol + 64, smem_u32(mt + 32768), 128, 1024, smem_u32(ar.X), blk, ge.S_ext);
          commit(&hd.bar_diag[jb & 1]);
        }
      }
      if (c_used && tma) {   // the C tile again, once nothing reads its region
        if (nblocks > 1) mbar_wait(&hd.bar_diag[1], 0, a.status, a.wait_ns);
        else mbar_wait(&hd.bar_state, 0, a.status, a.wait_ns);
        mbar_arrive_expect_tx(&hd.bar_c, (uint32_t)Q * 256u);
        tma_load_3d(ar.C, &maps.C, 0, g, z, &hd.bar_c);
        tma_load_3d(ar.C + Q * 128, &maps.C, 64, g, z, &hd.bar_c);
      }
      ready();   // start-state tile (and, without TMA, the C tile again)
      if (c_used && tma) mbar_wait(&hd.bar_c, 0, a.status, a.wait_ns);
      for (int tau = 0; tau < ntiles; ++tau)
        issue_yoff(tb + (tau == 0 ? kColOff : kColOff1), smem_u32(ar.C + 128 * 128 * tau), Q, 1024, smem_u32(ar.U),
                   128);
      commit(&hd.bar_off);
    }
  } else if (warp == kPubWarp) {
    // ================ publisher: flag releases and the look-back over earlier chunks ================
    if (c > 0 && has_next) {   // S_c and e_c for later chunks
      mbar_wait(&hd.bar_sdone, 0, a.status, a.wait_ns);
      if (lane == 0) {
        __threadfence();
        st_release(a.ws_flags + unit, 1);
      }
    }
    if (c > 0) {
      // lane l watches chunk top - l, 32 chunks per window, from c - 1 down; the chain starts at the
      // nearest chunk that has published its end state, once every chunk above it has published
      // its chunk state (chunk 0 publishes its end state, never its chunk state)
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
        hd.lb_stop = k0 < 0 ? 0 : k0;
        hd.lb_ok = good;
        mbar_arrive(&hd.bar_lb);
      }
    }
    if (has_next) {   // H_{c+1}
      mbar_wait(&hd.bar_hdone, 0, a.status, a.wait_ns);
      if (lane == 0) {
        __threadfence();
        st_release(a.ws_flags + unit, 2);
      }
    }
  } else {
    // ============================================ math warps ============================================
    const int q = warp & 3, sl = warp >> 2;
    const int n = 32 * q + lane;   // state column owned by this thread
    const int d0 = kOC * sl;       // and its kOC state rows d0 ..
    int hk = 0;                    // hand-offs so far
    if (!tma) load_rows_async(ar, make_rows<bf16>(a, sg.slot, h, nbuf, tok0), Q, nrows, false);
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
    math_sync();
    scan_decays(hd);
    if (tma) {
      mbar_wait(&hd.bar_tma, 0, a.status, a.wait_ns);
      if (nrows < Q) zero_rows(ar, Q, nrows);   // the boxes read the next tokens (or zeros) there
    }
    if (tid < nrows) {   // chunk-state weights w_s = delta_s exp(Acum_last - Acum_s)
      const df last = {hd.ahi[nrows - 1], hd.alo[nrows - 1]};
      hd.w[tid] = __fmul_rn(hd.delta[tid], expf(df_diff(last, df{hd.ahi[tid], hd.alo[tid]})));
    }
    hand_off(hd, hk);   // token tiles (and the weights, for every math thread)
    // ---- chunk state: U operands (the second K block's in the C region, once the Gram MMAs are done) ----
    build_u_tiles(ar.X, hd.w, nrows, 0, K < 128 ? K : 128, ar.U, ar.U + kUTile, ar.U + 2 * kUTile, kMath);
    hand_off(hd, hk);
    mma_wait(&hd.bar_gram, 0, a);
    if (two_state_blocks) {
      build_u_tiles(ar.X, hd.w, nrows, 128, K - 128, ar.C, ar.C + kUTile, ar.C + 2 * kUTile, kMath);
      hand_off(hd, hk);
    }
    mma_wait(&hd.bar_state, 0, a);
    // ---- publish: chunk 0 its end state H_1 (H_0 is known), later chunks S_c and e_c ------------------
    // Published states are laid out [n][d] (each thread's kOC values contiguous); the public outputs
    // (chunk states, final state, checkpoint) keep the [d][n] layout.  S_c stays in TMEM until the
    // off-diagonal MMAs.
    auto store_end_state = [&](const float (&Hn)[kOC]) {
      if (has_next) {
        float4* wi = reinterpret_cast<float4*>(a.ws_incl + unit * hs + (size_t)n * P + d0);
#pragma unroll
        for (int j = 0; j < kOC / 4; ++j) wi[j] = make_float4(Hn[4 * j], Hn[4 * j + 1], Hn[4 * j + 2], Hn[4 * j + 3]);
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
      if (has_next) mbar_arrive(&hd.bar_hdone);
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
    if (c == 0) {
      float S[kOC], Hc[kOC], Hn[kOC];
      tmem_ld16(taddr(tb, 32 * q, kColState + d0), S);
      const float e_c = expf(hd.ahi[nrows - 1]);
      const float* init = CHUNKED ? a.state + ((size_t)sg.slot * a.H + h) * hs
                                  : (a.init_state ? a.init_state + ((size_t)i * a.H + h) * hs : nullptr);
#pragma unroll
      for (int j = 0; j < kOC; ++j) Hc[j] = init ? init[(d0 + j) * N + n] : 0.f;
#pragma unroll
      for (int j = 0; j < kOC; ++j) Hn[j] = __fmaf_rn(e_c, Hc[j], S[j]);
      store_end_state(Hn);
      store_h_tile(Hc);
    } else if (has_next) {
      float S[kOC];
      tmem_ld16(taddr(tb, 32 * q, kColState + d0), S);
      float4* ws = reinterpret_cast<float4*>(a.ws_states + unit * hs + (size_t)n * P + d0);
#pragma unroll
      for (int j = 0; j < kOC / 4; ++j) ws[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
      if (tid == 0) a.ws_tot[unit] = expf(hd.ahi[nrows - 1]);
      mbar_arrive(&hd.bar_sdone);
    }
    // ---- every diagonal block (needs no start state); M tiles alternate between the B and C regions ----
    // accumulators: t-tile 0 in [0, 128), t-tile 1 in [128, 256) over the Gram block each uses
    uint32_t ph_diag[2] = {0, 0};
    bool pend[2] = {false, false};
    int jb = 0;
    for (int tau = 0; tau < ntiles; ++tau) {
      const Geom ge = geom(Q, tau);
      const uint32_t dcol = tau == 0 ? 0u : kColG1;
      for (int blk = 0; blk < ge.nblk; ++blk, ++jb) {
        const int bi = jb & 1;
        uint8_t* mt = bi == 0 ? ar.B : ar.C;
        if (pend[bi]) {   // the diagonal MMAs two blocks back still read this M tile
          mma_wait(&hd.bar_diag[bi], ph_diag[bi], a);
          ph_diag[bi] ^= 1;
          pend[bi] = false;
          math_sync();   // ... for every math thread before any overwrites it
        }
        build_m(ar, mt, tb, dcol + 128 * blk, Q, tau, blk, nrows);
        hand_off(hd, hk);
        pend[bi] = true;
      }
    }
    if (c_used && !tma) {   // the C tile again by cp.async, once nothing reads its region
      if (pend[1]) {
        mma_wait(&hd.bar_diag[1], ph_diag[1], a);
        ph_diag[1] ^= 1;
        pend[1] = false;
      }
      math_sync();
      load_rows_async(ar, make_rows<bf16>(a, sg.slot, h, nbuf, tok0), Q, nrows, true);
    }
    // ---- start state of a later chunk: the chain from the look-back's chunk, then H_{c+1} ---------------
    if (c > 0) {
      mbar_wait(&hd.bar_lb, 0, a.status, a.wait_ns);
      float Hc[kOC];
      const int k0 = hd.lb_stop;
      const bool good = hd.lb_ok != 0;
      const float4* Hk = reinterpret_cast<const float4*>(a.ws_incl + unit_index(a, i, k0, h) * hs + (size_t)n * P + d0);
#pragma unroll
      for (int j = 0; j < kOC / 4; ++j) {
        const float4 v = good ? __ldcg(Hk + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        Hc[4 * j] = v.x; Hc[4 * j + 1] = v.y; Hc[4 * j + 2] = v.z; Hc[4 * j + 3] = v.w;
      }
      for (int kk = k0 + 1; good && kk < c; kk += 2) {   // two chunks' loads in flight
        float4 sv[2][kOC / 4];
        float ev[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          ev[u] = 0.f;
          if (kk + u < c) {
            const size_t uk = unit_index(a, i, kk + u, h);
            ev[u] = __ldcg(a.ws_tot + uk);
            const float4* Sk = reinterpret_cast<const float4*>(a.ws_states + uk * hs + (size_t)n * P + d0);
#pragma unroll
            for (int j = 0; j < kOC / 4; ++j) sv[u][j] = __ldcg(Sk + j);
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (kk + u < c) {
#pragma unroll
            for (int j = 0; j < kOC / 4; ++j) {
              Hc[4 * j] = __fmaf_rn(ev[u], Hc[4 * j], sv[u][j].x);
              Hc[4 * j + 1] = __fmaf_rn(ev[u], Hc[4 * j + 1], sv[u][j].y);
              Hc[4 * j + 2] = __fmaf_rn(ev[u], Hc[4 * j + 2], sv[u][j].z);
              Hc[4 * j + 3] = __fmaf_rn(ev[u], Hc[4 * j + 3], sv[u][j].w);
            }
          }
        }
      }
      float S[kOC], Hn[kOC];
      tmem_ld16(taddr(tb, 32 * q, kColState + d0), S);
      const float e_c = expf(hd.ahi[nrows - 1]);
#pragma unroll
      for (int j = 0; j < kOC; ++j) Hn[j] = __fmaf_rn(e_c, Hc[j], S[j]);
      store_end_state(Hn);
      store_h_tile(Hc);
    }
    hand_off(hd, hk);   // start-state tile (the off-diagonal MMAs overwrite the state's TMEM columns)
    for (int bi = 0; bi < 2; ++bi)
      if (pend[bi]) {
        mma_wait(&hd.bar_diag[bi], ph_diag[bi], a);
        ph_diag[bi] ^= 1;
        pend[bi] = false;
      }
    mma_wait(&hd.bar_off, 0, a);
    // ---- epilogues ------------------------------------------------------------------------------------
    const float Dh = a.D[h];
    for (int tau = 0; tau < ntiles; ++tau) {
      const Geom ge = geom(Q, tau);
      epilogue(ar, tb, tau == 0 ? 0u : kColG1, tau == 0 ? kColOff : kColOff1, Q, tau, max(nbuf, ge.t0),
               min(nrows, ge.t0 + ge.TT), Dh, (bf16*)a.y, tok0, a.H, h);
    }
  }
  before_sync();
  __syncthreads();
  if (warp == kIssuerWarp) tmem_dealloc(tb, kScanTmemCols);
}

// ---- host side ---------------------------------------------------------------------------------------
// 3-D map over a token-major bf16 tensor [T, R, W] (W contiguous): dims {W, R, T}, box {64, 1, Q}.
bool encode_rows(CUtensorMap* m, const void* base, long long T, int R, int W, int Q) {
  EncodeTiledFn fn = tma_encode_fn();
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

EncodeTiledFn tma_encode_fn() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult qr;
    EncodeTiledFn r = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      r = reinterpret_cast<EncodeTiledFn>(f);
    cudaGetLastError();
    return r;
  }();
  return fn;
}

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
