// Tensor-core (tcgen05) kernels for bf16 io, P = 64, N = 128: exact-replay decode with fused
// refresh, refresh, and output-only speculative verify (the SSD prefill is ers_tc_scan.cu).  Every
// output row and chunk state goes through tc_outputs() / tc_state() below, which issue the same MMA
// sequences and build the same operand values as the prefill, so all paths agree bit for bit
// (exact-replay RFC, vLLM issue 55524, section 3; ReplaySSM notes, "Core equations").
#include "ers_common.cuh"
#include "ers_internal.h"
#include "tc_engine.cuh"

namespace ers {
namespace {

using bf16 = __nv_bfloat16;
using namespace tc;

// Shared-memory header at the start of dynamic shared memory.
struct TcHdr {
  uint64_t bar;          // MMA completion
  uint32_t tmem;         // TMEM base written by tcgen05.alloc
  uint32_t pad;
  alignas(16) float delta[kQMax];
  alignas(16) float ahi[kQMax];      // Acum (double-float); dA before the scan
  alignas(16) float alo[kQMax];
  alignas(16) float w[kQMax];        // chunk-state weights
  float ydiag_row[P];    // decode: Ydiag of the output row
};

extern __shared__ __align__(1024) unsigned char tc_smem[];

// 1024-byte aligned base (the launch reserves 1 KB of slack for this)
__device__ __forceinline__ unsigned char* smem_base() {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tc_smem) + 1023) & ~uintptr_t(1023));
}
constexpr size_t kHdrBytes = (sizeof(TcHdr) + 1023) & ~size_t(1023);
__device__ __forceinline__ TcHdr& hdr() { return *reinterpret_cast<TcHdr*>(smem_base()); }
__device__ __forceinline__ uint8_t* tiles() { return smem_base() + kHdrBytes; }

__host__ __device__ __forceinline__ int round16(int v) { return (v + 15) & ~15; }

// Tile arena of the output/decode/verify kernels: [C 32K | H 32K | B (BR x 256) | X (BR x 128)];
// M^T (hi, lo) reuse C and H once the Gram and off-diagonal MMAs have completed; the transposed
// off-diagonal sums reuse them again after the diagonal MMAs.  BR = B/X tile rows.
struct Arena {
  uint8_t* C;
  uint8_t* Hs;
  uint8_t* B;
  uint8_t* X;
  uint32_t BR;
};
__host__ __device__ __forceinline__ size_t arena_bytes(int BR) {
  return 32768 + kHTile + (size_t)BR * 256 + (size_t)BR * 128;
}
__device__ __forceinline__ Arena arena(int BR) {
  Arena ar;
  ar.C = tiles();
  ar.Hs = ar.C + 32768;
  ar.B = ar.Hs + kHTile;
  ar.X = ar.B + (size_t)BR * 256;
  ar.BR = BR;
  return ar;
}

__device__ __forceinline__ void setup_tmem(uint32_t ncols) {
  TcHdr& hd = hdr();
  if (threadIdx.x == 0) {
    mbar_init(&hd.bar, 1);
    fence_mbar_init();
  }
  if (threadIdx.x / 32 == 0) tmem_alloc(&hd.tmem, ncols);
  before_sync();
  __syncthreads();
  after_sync();
}

__device__ __forceinline__ void teardown_tmem(uint32_t ncols) {
  before_sync();
  __syncthreads();
  if (threadIdx.x / 32 == 0) tmem_dealloc(hdr().tmem, ncols);
}


// delta / dA for rows [0, nrows) (zeros beyond), then the chunk scan
__device__ __forceinline__ void load_decays(const Rows<bf16>& rows, int nrows, float A, float bias) {
  TcHdr& hd = hdr();
  const int t = threadIdx.x;
  if (t < kQMax) {
    float d = 0.f, da = 0.f;
    if (t < nrows) {
      d = delta_of(rows.dt(t), bias);
      da = __fmul_rn(d, A);
    }
    hd.delta[t] = d;
    hd.ahi[t] = da;
    hd.alo[t] = 0.f;
  }
  __syncthreads();
  chunk_scan(hd.ahi, hd.alo);
}

// X and B tile rows [0, BR): valid rows [0, nrows) from `rows`, zeros beyond
__device__ __forceinline__ void load_xb(const Rows<bf16>& rows, int nrows, const Arena& ar) {
  for (int id = threadIdx.x; id < (int)ar.BR * 24; id += blockDim.x) {
    const int r = id / 24, c = id % 24;
    if (c < 8) {
      if (r < nrows) row_to_tile(rows.x(r), ar.X, 1, r, c);
      else zero_tile_chunk(ar.X, 1, r, c);
    } else {
      if (r < nrows) row_to_tile(rows.B(r), ar.B, ar.BR, r, c - 8);
      else zero_tile_chunk(ar.B, ar.BR, r, c - 8);
    }
  }
}

// C tile (128 rows): tile row j holds chunk row t0 + j for j in [lo - t0, hi - t0), zeros elsewhere
__device__ __forceinline__ void load_c(const Rows<bf16>& rows, int t0, int lo, int hi, const Arena& ar) {
  for (int id = threadIdx.x; id < 128 * 16; id += blockDim.x) {
    const int j = id / 16, c = id % 16;
    const int t = t0 + j;
    if (t >= lo && t < hi) row_to_tile(rows.C(t), ar.C, 128, j, c);
    else zero_tile_chunk(ar.C, 128, j, c);
  }
}

// ---------------------------------------------------------------------------------------------
// Outputs of chunk rows [out_lo, out_hi) inside t-tile tau, by all NW warps of the CTA (NW = 8 or
// 16; warp w reads TMEM lane quarter w % 4 and a 1/(NW/4) slice of the columns).  Tiles (C, H, B,
// X) and the scanned decays must be in place.  Rows >= tmax are invalid (their M^T rows are zero).
// Row t's output goes to ybase + (t - out_lo) * yrs.  Returns false if a wait timed out.  The MMA
// sequence and every value are independent of NW.
template <int NW>
__device__ bool tc_outputs(const Arena& ar, int Q, int tau, int tmax, int out_lo, int out_hi, float Dh,
                           bf16* ybase, long long yrs, int32_t* status) {
  static_assert(NW == 8 || NW == 16, "4 TMEM lane quarters x 2 or 4 column slices");
  constexpr int NS = NW / 4;          // column slices
  constexpr int MC = 128 / NS;        // M columns per warp and block
  constexpr int OC = 64 / NS;         // output columns per warp
  TcHdr& hd = hdr();
  const Geom ge = geom(Q, tau);
  const uint32_t tb = hd.tmem;
  const int RG = tmem_rg(ge.S_ext);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3, sl = warp >> 2;
  const int row = 32 * q + lane;
  const int t = ge.t0 + row;
  uint32_t phase = 0;
  bool ok = true;
  if (threadIdx.x == 0) {
    issue_gram(tb, smem_u32(ar.C), 128, 1024, smem_u32(ar.B), ar.BR, ge.S_ext);
    issue_yoff(tb + RG, smem_u32(ar.C), 128, 1024, smem_u32(ar.Hs), 128);
    commit(&hd.bar);
  }
  ok = __syncthreads_and(mbar_wait(&hd.bar, phase, status));
  phase ^= 1;
  after_sync();
  const int tlim = tmax < ge.t0 + ge.TT ? tmax : ge.t0 + ge.TT;
  // M tiles (hi over the C tile, lo over the H tile) once the Gram and off-diagonal MMAs are done
  for (int blk = 0; blk < ge.nblk && ok; ++blk) {
    const int width = ge.S_ext - 128 * blk < 128 ? ge.S_ext - 128 * blk : 128;
    if (MC * sl < width) {
      float g[MC];
      if constexpr (MC == 64) tmem_ld64(taddr(tb, 32 * q, 128 * blk + MC * sl), g);
      else tmem_ld32(taddr(tb, 32 * q, 128 * blk + MC * sl), g);
      m_row<MC>(g, t, tlim, blk, MC * sl, ge.S_ext, hd.delta, hd.ahi, hd.alo, ar.C, ar.Hs, 128, row);
    }
    publish();
    if (threadIdx.x == 0) {
      issue_ydiag(tb, smem_u32(ar.C), 128, 1024, smem_u32(ar.X), blk, ge.S_ext);
      issue_ydiag(tb + 64, smem_u32(ar.Hs), 128, 1024, smem_u32(ar.X), blk, ge.S_ext);
      commit(&hd.bar);
    }
    ok = __syncthreads_and(mbar_wait(&hd.bar, phase, status));
    phase ^= 1;
    after_sync();
  }
  if (!ok) return false;
  // combine: thread (row, slice) writes d in [OC sl, OC sl + OC)
  float oh[OC], ol[OC], dh[OC], dl[OC];
  if constexpr (OC == 32) {
    tmem_ld32(taddr(tb, 32 * q, RG + OC * sl), oh);
    tmem_ld32(taddr(tb, 32 * q, RG + 64 + OC * sl), ol);
    tmem_ld32(taddr(tb, 32 * q, OC * sl), dh);
    tmem_ld32(taddr(tb, 32 * q, 64 + OC * sl), dl);
  } else {
    tmem_ld16(taddr(tb, 32 * q, RG + OC * sl), oh);
    tmem_ld16(taddr(tb, 32 * q, RG + 64 + OC * sl), ol);
    tmem_ld16(taddr(tb, 32 * q, OC * sl), dh);
    tmem_ld16(taddr(tb, 32 * q, 64 + OC * sl), dl);
  }
  if (t >= out_lo && t < out_hi && row < ge.TT) {
    const float et = expf(hd.ahi[t]);
    uint32_t packed[OC / 2];
#pragma unroll
    for (int j = 0; j < OC; j += 2) {
      float o[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int d = OC * sl + j + u;
        const float xv = __bfloat162float(*reinterpret_cast<const bf16*>(ar.X + sw128(1, t, d)));
        o[u] = combine_out(et, __fadd_rn(oh[j + u], ol[j + u]), __fadd_rn(dh[j + u], dl[j + u]), Dh, xv);
      }
      packed[j / 2] = pack_bf16x2(o[0], o[1]);
    }
    uint4* dst = reinterpret_cast<uint4*>(ybase + (long long)(t - out_lo) * yrs + OC * sl);
#pragma unroll
    for (int k = 0; k < OC / 8; ++k) dst[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
  }
  return true;
}

// Chunk state over rows [0, nrows) (K = round16(nrows)) from the B and X tiles, in K blocks of
// 128 rows; each block's U tiles are built in `u` (3 x 16 KB).  The result S^T[n][d] is left in
// TMEM columns [0, 64).
constexpr uint32_t kUBytes = 3u * 128u * 128u;
__device__ bool tc_state(const Arena& ar, int nrows, uint8_t* u, int32_t* status, uint32_t* phase) {
  TcHdr& hd = hdr();
  const int K = round16(nrows);
  if (threadIdx.x < nrows) {
    const df last = {hd.ahi[nrows - 1], hd.alo[nrows - 1]};
    hd.w[threadIdx.x] =
        __fmul_rn(hd.delta[threadIdx.x], expf(df_diff(last, df{hd.ahi[threadIdx.x], hd.alo[threadIdx.x]})));
  }
  __syncthreads();
  uint8_t* u0 = u;
  uint8_t* u1 = u + 128 * 128;
  uint8_t* u2 = u + 2 * 128 * 128;
  bool ok = true;
  for (int s0 = 0; s0 < K && ok; s0 += 128) {
    const int nr = K - s0 < 128 ? K - s0 : 128;
    build_u_tiles(ar.X, hd.w, nrows, s0, nr, u0, u1, u2);
    publish();
    if (threadIdx.x == 0) {
      issue_state_block(hd.tmem, smem_u32(ar.B), ar.BR, smem_u32(u0), smem_u32(u1), smem_u32(u2), s0, nr / 16);
      commit(&hd.bar);
    }
    ok = __syncthreads_and(mbar_wait(&hd.bar, *phase, status));
    *phase ^= 1;
    after_sync();
  }
  return ok;
}

// H' = fma(exp(Acum_last), H, S) from TMEM S^T, written over H (and the read copy, if any)
__device__ __forceinline__ void fold_from_tmem(float* Hd, bf16* Rd, float decay) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3, half = warp >> 2;
  const int n = 32 * q + lane;
  float s[32];
  tmem_ld32(taddr(hdr().tmem, 32 * q, 32 * half), s);
#pragma unroll 4
  for (int j = 0; j < 32; ++j) {
    const int d = 32 * half + j;
    const float v = __fmaf_rn(decay, Hd[d * N + n], s[j]);
    Hd[d * N + n] = v;
    if (Rd != nullptr) Rd[d * N + n] = __float2bfloat16_rn(v);
  }
}

// ---- replay decode (one CTA per sequence and head) ---------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) k_tc_decode(LaunchArgs a, uint32_t tcols) {
  const int i = blockIdx.x, h = blockIdx.y;
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const bool rssm = (a.flags & ERS_FLAG_REPLAYSSM) != 0;
  const int p = a.pos[slot];
  if (p < 0 || p >= a.Q) {
    if (threadIdx.x == 0) report(a.status, ERS_EALIGN);
    return;
  }
  const int tau = p / 128;
  const Geom ge = geom(a.Q, tau);
  const bool refresh = !rssm && (a.flags & ERS_FLAG_FUSE_REFRESH) && p + 1 == a.Q;
  const Rows<bf16> rows = make_rows<bf16>(a, slot, h, p, (long long)i - p);
  setup_tmem(tcols);
  const Arena ar = arena(a.Q);
  const size_t hs = (size_t)P * N;
  float* Hd = a.state + ((size_t)slot * a.H + h) * hs;
  bf16* Rd = a.read_copy ? (bf16*)a.read_copy + ((size_t)slot * a.H + h) * hs : nullptr;
  load_decays(rows, p + 1, a.A[h], a.dt_bias[h]);
  load_xb(rows, p + 1, ar);
  load_c(rows, ge.t0, p, p + 1, ar);
  if (rssm) readcopy_to_tile(Rd, ar.Hs);
  else state_to_tile(Hd, ar.Hs);
  publish();
  bool ok = tc_outputs<8>(ar, a.Q, tau, p + 1, p, p + 1, a.D[h], (bf16*)a.y + ((size_t)i * a.H + h) * P, 0, a.status);
  // append the new token to the buffer (B/C once per group)
  const int g = h / (a.H / a.G);
  const bf16* nx = (const bf16*)a.x + ((size_t)i * a.H + h) * P;
  bf16* bx = (bf16*)a.bx + (buf_row(a, slot, p) * a.H + h) * P;
  for (int d = threadIdx.x; d < P; d += kThreads) bx[d] = nx[d];
  if (threadIdx.x == 0) a.bdt[buf_row(a, slot, p) * a.H + h] = a.dt[(size_t)i * a.H + h];
  if (h % (a.H / a.G) == 0) {
    const size_t dst = (buf_row(a, slot, p) * a.G + g) * N, src = ((size_t)i * a.G + g) * N;
    for (int n = threadIdx.x; n < N; n += kThreads) {
      ((bf16*)a.bB)[dst + n] = ((const bf16*)a.B)[src + n];
      ((bf16*)a.bC)[dst + n] = ((const bf16*)a.C)[src + n];
    }
  }
  if (ok && refresh) {
    __syncthreads();
    uint32_t phase = 1 + ge.nblk;  // completions so far: Gram+Yoff, then one per diagonal block
    phase &= 1;
    // U tiles over the dead C/H tiles
    if (tc_state(ar, a.Q, ar.C, a.status, &phase)) fold_from_tmem(Hd, Rd, expf(hdr().ahi[a.Q - 1]));
  }
  teardown_tmem(tcols);
}

// ---- refresh: exact (pos == Q) or ReplaySSM flush rule (pos + T > L) ---------------------------------
__global__ void __launch_bounds__(kThreads, 1) k_tc_refresh(LaunchArgs a, bool verify_flush) {
  const int i = blockIdx.x, h = blockIdx.y;
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const bool rssm = verify_flush || (a.flags & ERS_FLAG_REPLAYSSM) != 0;
  const int p = a.pos[slot];
  if (p < 0 || p > a.Q) {
    if (threadIdx.x == 0) report(a.status, ERS_EALIGN);
    return;
  }
  const bool go = rssm ? (p + a.T > a.Q) : (p == a.Q);
  if (!go) return;
  if (verify_flush && !(a.flags & ERS_FLAG_AUTO_FLUSH)) {
    if (threadIdx.x == 0) report(a.status, ERS_EOVERFLOW);
    return;
  }
  const size_t hs = (size_t)P * N;
  float* Hd = a.state + ((size_t)slot * a.H + h) * hs;
  bf16* Rd = a.read_copy ? (bf16*)a.read_copy + ((size_t)slot * a.H + h) * hs : nullptr;
  if (p == 0) {  // empty committed history: anchor bits unchanged, read copy recast from them
    if (Rd != nullptr)
      for (int idx = threadIdx.x; idx < P * N; idx += kThreads) Rd[idx] = __float2bfloat16_rn(Hd[idx]);
    return;
  }
  const Rows<bf16> rows = make_rows<bf16>(a, slot, h, p, 0);
  const int K = round16(p);
  setup_tmem(64);
  Arena ar;
  ar.BR = K;
  ar.B = tiles();
  ar.X = ar.B + (size_t)K * 256;
  ar.C = nullptr;
  ar.Hs = nullptr;
  load_decays(rows, p, a.A[h], a.dt_bias[h]);
  load_xb(rows, p, ar);
  cp_async_wait_all();
  __syncthreads();
  uint32_t phase = 0;
  if (tc_state(ar, p, ar.X + (size_t)K * 128, a.status, &phase)) fold_from_tmem(Hd, Rd, expf(hdr().ahi[p - 1]));
  teardown_tmem(64);
}

// ---- speculative verify: drafts to buffer rows [h', h'+T), outputs from the read copy -----------
__global__ void __launch_bounds__(kThreads, 1) k_tc_verify(LaunchArgs a, uint32_t tcols) {
  const int i = blockIdx.x, h = blockIdx.y;
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const int hc = a.pos[slot];
  if (hc < 0 || hc > a.Q) return;  // reported by the flush launch
  int h0 = hc;
  if (hc + a.T > a.Q) {
    if (!(a.flags & ERS_FLAG_AUTO_FLUSH)) return;
    h0 = 0;
  }
  const int nrows = h0 + a.T;
  const Rows<bf16> rows = make_rows<bf16>(a, slot, h, h0, (long long)i * a.T - h0);
  setup_tmem(tcols);
  const Arena ar = arena(a.Q);
  const size_t hs = (size_t)P * N;
  const bf16* Rd = (const bf16*)a.read_copy + ((size_t)slot * a.H + h) * hs;
  load_decays(rows, nrows, a.A[h], a.dt_bias[h]);
  load_xb(rows, nrows, ar);
  // all output rows lie in t-tile 0 when Q <= 128; otherwise process each tile they touch
  bool ok = true;
  for (int tau = h0 / 128; tau <= (nrows - 1) / 128 && ok; ++tau) {
    const Geom ge = geom(a.Q, tau);
    const int lo = max(h0, ge.t0), hi = min(nrows, ge.t0 + ge.TT);
    load_c(rows, ge.t0, lo, hi, ar);
    readcopy_to_tile(Rd, ar.Hs);
    publish();
    bf16* ybase = (bf16*)a.y + (((size_t)i * a.T + (lo - h0)) * a.H + h) * P;
    // a fresh barrier phase sequence per tile: re-initialise between tiles
    ok = tc_outputs<8>(ar, a.Q, tau, nrows, lo, hi, a.D[h], ybase, (long long)a.H * P, a.status);
    if (tau < (nrows - 1) / 128) {
      __syncthreads();
      if (threadIdx.x == 0) {
        mbar_init(&hdr().bar, 1);
        fence_mbar_init();
      }
      __syncthreads();
    }
  }
  // drafts into the buffer
  const int g = h / (a.H / a.G);
  for (int idx = threadIdx.x; idx < a.T * P; idx += kThreads) {
    const int j = idx / P, d = idx % P;
    ((bf16*)a.bx)[(buf_row(a, slot, h0 + j) * a.H + h) * P + d] =
        ((const bf16*)a.x)[(((size_t)i * a.T + j) * a.H + h) * P + d];
  }
  for (int j = threadIdx.x; j < a.T; j += kThreads)
    a.bdt[buf_row(a, slot, h0 + j) * a.H + h] = a.dt[((size_t)i * a.T + j) * a.H + h];
  if (h % (a.H / a.G) == 0) {
    for (int idx = threadIdx.x; idx < a.T * N; idx += kThreads) {
      const int j = idx / N, n = idx % N;
      const size_t dst = (buf_row(a, slot, h0 + j) * a.G + g) * N + n;
      const size_t src = (((size_t)i * a.T + j) * a.G + g) * N + n;
      ((bf16*)a.bB)[dst] = ((const bf16*)a.B)[src];
      ((bf16*)a.bC)[dst] = ((const bf16*)a.C)[src];
    }
  }
  teardown_tmem(tcols);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

size_t out_smem(int BR) { return kHdrBytes + arena_bytes(BR) + 1024; }
size_t state_smem(int K) { return kHdrBytes + (size_t)K * (256 + 128) + kUBytes + 1024; }

}  // namespace

bool tc_supported(int io, int P_, int N_, int Q) {
  return io == ERS_DTYPE_BF16 && P_ == P && N_ == N && Q % 16 == 0 && Q >= kTcMinChunk && Q <= kQMax;
}

cudaError_t tc_decode(const LaunchArgs& a, cudaStream_t s) {
  const size_t so = out_smem(a.Q);
  cudaError_t e = set_smem(k_tc_decode, so);
  if (e != cudaSuccess) return e;
  k_tc_decode<<<dim3(a.nseq, a.H), kThreads, so, s>>>(a, tmem_cols(a.Q));
  return launch_setpos(a, 0, s);
}

cudaError_t tc_refresh(const LaunchArgs& a, cudaStream_t s) {
  const size_t ss = state_smem(a.Q);
  cudaError_t e = set_smem(k_tc_refresh, ss);
  if (e != cudaSuccess) return e;
  k_tc_refresh<<<dim3(a.nseq, a.H), kThreads, ss, s>>>(a, false);
  return launch_setpos(a, 1, s);
}

cudaError_t tc_verify(const LaunchArgs& a, cudaStream_t s) {
  const size_t ss = state_smem(a.Q), so = out_smem(a.Q);
  cudaError_t e;
  if ((e = set_smem(k_tc_refresh, ss)) != cudaSuccess) return e;
  if ((e = set_smem(k_tc_verify, so)) != cudaSuccess) return e;
  k_tc_refresh<<<dim3(a.nseq, a.H), kThreads, ss, s>>>(a, true);
  k_tc_verify<<<dim3(a.nseq, a.H), kThreads, so, s>>>(a, tmem_cols(a.Q));
  return cudaGetLastError();
}

}  // namespace ers
