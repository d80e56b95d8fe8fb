// Replay decode for small chunks (chunk <= 32, P a multiple of 32, N = 128): the bandwidth-shaped
// decode kernel of the CUDA-core engine.
//
// A decode step at a small chunk is, per head, a matrix-vector product with the fp32 boundary
// checkpoint plus a replay of at most 31 buffered rows (exact-replay RFC, section 3), so its cost is
// streaming the checkpoint from HBM.  The arithmetic is the engine's, operation for operation
// (row_output, state_weights, chunk_state, fold_state in ers_fma.cu; Dot<128> and chunk_scan in
// ers_common.cuh), so decode equals single-shot and chunked prefill bit for bit.
#include <type_traits>

#include "ers_common.cuh"
#include "ers_internal.h"
#include "warp_heads.cuh"

namespace ers {
namespace {

using namespace wh;

// ---- replay decode for small chunks, shaped for HBM bandwidth -------------------------------------
// Same arithmetic as k_decode (row_output, state_weights, chunk_state and fold_state, operation for
// operation), organised so that a step costs little more than streaming the boundary state once.
//  * One CTA per (sequence, block of up to 8 heads of one B/C group), one warp per head.  The warp
//    streams its head's [P x N] state through registers, 8 rows at a time, two blocks in flight;
//    lane j holds elements [4j, 4j+4) of each row, the lane split of Dot<128>.
//  * The lane partials of 16 rows are combined by reduce_scatter16 (warp_heads.cuh), which keeps
//    the pairings of Dot<128>'s butterfly and so each row's bits, at about one shuffle per row.
//  * The group's Gram row C_p . B_s is computed once per CTA; buffer rows arrive by cp.async while
//    the state streams; the log-decay scan runs per warp with shuffles (for rows < 32 the strides
//    >= 32 of chunk_scan change nothing, so the bits are chunk_scan's).
//  * When the step fills the chunk, the state is streamed after the chunk's weights are known and
//    each row is folded (fold_state) and written back in the same pass.

// B and x rows: up to QM buffered rows plus the new token (a ReplaySSM flush holds L = Q committed
// rows and the new token).
template <int QM>
constexpr int heads_rows() { return QM + 1; }

// The last region serves a step that fills or flushes the chunk as the per-warp w_s x_s[d] table and a
// plain step with an NVFP4 copy as the heads' staged copy (P N / 2 code bytes + P N / 16 block-scale
// bytes per warp), so it takes the larger of the two.
template <int P, int N, int QM>
constexpr size_t heads_table_bytes() {
  return (size_t)kHeadsPerCta * ((size_t)QM * P * sizeof(float) > staged_bytes<P, N>() ? (size_t)QM * P * sizeof(float)
                                                                                       : staged_bytes<P, N>());
}

template <typename T, int P, int N, int QM>
constexpr size_t heads_smem_bytes() {
  return (size_t)heads_rows<QM>() * N * sizeof(T) + (size_t)kHeadsPerCta * heads_rows<QM>() * P * sizeof(T) +
         QM * sizeof(float) + (size_t)kHeadsPerCta * P * sizeof(float) + heads_table_bytes<P, N, QM>();
}

// A plain ReplaySSM step with an NVFP4 copy stages each head's whole copy (4 KB of codes + 512 B of
// block scales) in shared memory with one burst of 16-byte copies, so that every byte of the CTA is
// in flight at once (32 rows of 3 bytes per lane in registers kept too few bytes in flight), and
// streams the rows from there.  (Staging the 8 KB FP8 copies measured slower: 83 against 72 us.)
template <typename HT> constexpr bool kStaged = std::is_same<HT, Nvfp4>::value;


// Streams one head's state: lane j of row d reads elements [4j, 4j+4), 8 rows per block, with
// rows_in_flight rows in flight (q holds the first of them on entry).  yo[d] ends with the
// off-diagonal term (H C_p)[d] (per-warp shared memory).  FP8 and NVFP4 copies are read as codes:
// an NVFP4 lane partial is scaled by its block scale, and each row's dot product by the row scale,
// which lane d % 32 holds in sc[d / 32].

// Rows of the stream in flight per warp: 16 fp32 rows, 32 rows of a read copy (measured: more FP8
// rows than 32 spill registers and run slower).
template <typename HT>
constexpr int rows_in_flight() { return sizeof(typename RawOf<HT>::type) == 16 ? 16 : 32; }

template <typename HT, int P, int N, typename Src>
__device__ __forceinline__ void stream_state(const Src& src,
                                             typename RawOf<HT>::type (&q)[rows_in_flight<HT>()],
                                             const float (&c)[4], float* yo, int j, const float (&sc)[2]) {
  constexpr int NBLK = P / 8, RIF = rows_in_flight<HT>();
  static_assert(RIF % 16 == 0 && RIF <= P, "whole 16-row reduction groups in flight");
  float part[16];
#pragma unroll
  for (int blk = 0; blk < NBLK; ++blk) {
    const int sl = (blk & 1) * 8;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int d = blk * 8 + r;
      float h[4], ls;
      row_values<HT>(q[d % RIF], h, &ls);
      float pp = Dot<N>::partial(c, h);
      if constexpr (kLaneScale<HT>) pp = __fmul_rn(pp, ls);
      part[sl + r] = pp;
      if (d + RIF < P) q[d % RIF] = src.ld(d + RIF, j);
    }
    if (blk & 1) {
      float v = reduce_scatter16(part, j);   // row (blk - 1) * 8 + j / 2 on even lanes
      if constexpr (kRowScale<HT>)
        v = __fmul_rn(v, __shfl_sync(kFull, sc[((blk - 1) * 8) >> 5], ((blk - 1) * 8 + (j >> 1)) & 31));
      if ((j & 1) == 0) yo[(blk - 1) * 8 + (j >> 1)] = v;
    }
  }
  __syncwarp();
}

// The same stream for a step that fills the chunk: each row is also folded with the chunk state and
// written back, in chunk_state / fold_state order,
//   H'[d][n] = fma(decay, H[d][n], acc),  acc = fma(wx[s][d], B_s[n], acc) over s = 0..p,
// where wx[s][d] = w_s x_s[d] is a per-warp shared-memory table.  Rows are read (coherently: this
// loop writes the rows it has consumed) 8 at a time with the next 8 in flight, and each 4 rows'
// fold accumulates over the chunk with 16 independent chains.
template <typename T, int P, int N>
__device__ __noinline__ void stream_state_refresh(float* __restrict__ Hd, __nv_bfloat16* __restrict__ Rd,
                                                  uint8_t* __restrict__ R8, float* __restrict__ Rs, float c0,
                                                  float c1, float c2, float c3, float* yo, int j, int p,
                                                  const float* wx, float decay, const T* sB) {
  constexpr int NBLK = P / 8;
  const float c[4] = {c0, c1, c2, c3};
  float4 cur[8], nxt[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) cur[r] = __ldcs(reinterpret_cast<const float4*>(Hd + (size_t)r * N + 4 * j));
  float part[16];
#pragma unroll 1
  for (int blk = 0; blk < NBLK; ++blk) {
    if (blk + 1 < NBLK) {
#pragma unroll
      for (int r = 0; r < 8; ++r)
        nxt[r] = __ldcs(reinterpret_cast<const float4*>(Hd + (size_t)((blk + 1) * 8 + r) * N + 4 * j));
    }
    float pb[8];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      Fold4 acc;
      acc.zero();
      for (int s = 0; s <= p; ++s) {
        float bs[4];
        lds4(sB + s * N + 4 * j, bs);
        acc.add(*reinterpret_cast<const float4*>(wx + s * P + blk * 8 + 4 * hf), bs);
      }
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        const int r = 4 * hf + r4;
        float h[4];
        Quad<float>::unpack(cur[r], h);
        pb[r] = Dot<N>::partial(c, h);
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __fmaf_rn(decay, h[e], acc.get(r4, e));
        const size_t o = (size_t)(blk * 8 + r) * N + 4 * j;
        *reinterpret_cast<float4*>(Hd + o) = make_float4(v[0], v[1], v[2], v[3]);
        if (Rd != nullptr) {
          __nv_bfloat162 lo2 = __floats2bfloat162_rn(v[0], v[1]), hi2 = __floats2bfloat162_rn(v[2], v[3]);
          uint2 u;
          u.x = *reinterpret_cast<uint32_t*>(&lo2);
          u.y = *reinterpret_cast<uint32_t*>(&hi2);
          *reinterpret_cast<uint2*>(Rd + o) = u;
        }
        if (R8 != nullptr) fp8_store_row<N>(v, R8, Rs, blk * 8 + r, j);   // warp-uniform branch
      }
    }
    if ((blk & 1) == 0) {
#pragma unroll
      for (int r = 0; r < 8; ++r) part[r] = pb[r];
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r) part[8 + r] = pb[r];
      const float v = reduce_scatter16(part, j);
      if ((j & 1) == 0) yo[(blk - 1) * 8 + (j >> 1)] = v;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) cur[r] = nxt[r];
  }
  __syncwarp();
}

// ReplaySSM flush inside decode: each anchor row is folded with the h committed records in the same
// order as stream_state_refresh (and the refresh kernels), written back, and cast into the read
// copy (bf16, FP8 or NVFP4); the new token's dot product reads the cast values, exactly as a decode
// after a separate refresh reads them from the copy.  FP8 / NVFP4 rows' dot products are scaled
// after the reduction (srow: lane j keeps the scale of the 16-row group's row j / 2).
// kOut = false (the standalone refresh): no output, and HT = NoCopy when the cache keeps no copy; an
// empty history (hc = 0) leaves the anchor's bits as they are and only recasts the copy.
struct NoCopy {};

template <typename HT>
__host__ __device__ constexpr size_t sizeof_copy() {   // bytes per value of a bf16 / FP8 copy
  return std::is_same<HT, __nv_bfloat16>::value ? 2 : 1;
}

template <typename T, typename HT, int P, int N, bool kOut = true, typename AT = float>
__device__ __noinline__ void stream_flush_copy(AT* __restrict__ Hd, void* __restrict__ R, uint8_t* __restrict__ Rb,
                                               float* __restrict__ Rs, float c0, float c1, float c2, float c3,
                                               float* yo, int j, int hc, const float* wx, float decay,
                                               const T* sB, SrCtr sr, uint32_t row0) {
  constexpr int NBLK = P / 8;
  constexpr bool kF8 = std::is_same<HT, uint8_t>::value;
  constexpr bool kNv = std::is_same<HT, Nvfp4>::value;
  constexpr bool kBf = std::is_same<HT, __nv_bfloat16>::value;
  constexpr bool kSh = std::is_same<AT, Nvfp4Shared>::value;   // the NVFP4 copy is the state
  static_assert(!kSh || kNv, "a shared state is an NVFP4 copy");
  const float c[4] = {c0, c1, c2, c3};
  float4 cur[8], nxt[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) cur[r] = anchor_row<AT, N>(Hd, R, Rb, Rs, r, j);
  float part[16];
  float srow = 0.f;
#pragma unroll 1
  for (int blk = 0; blk < NBLK; ++blk) {
    if (blk + 1 < NBLK) {
#pragma unroll
      for (int r = 0; r < 8; ++r)
        nxt[r] = anchor_row<AT, N>(Hd, R, Rb, Rs, (blk + 1) * 8 + r, j);
    }
    float pb[8];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      Fold4 acc;
      acc.zero();
      for (int s = 0; s < hc; ++s) {
        float bs[4];
        lds4(sB + s * N + 4 * j, bs);
        acc.add(*reinterpret_cast<const float4*>(wx + s * P + blk * 8 + 4 * hf), bs);
      }
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        const int r = 4 * hf + r4;
        float h[4], v[4], rv[4];
        Quad<float>::unpack(cur[r], h);
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = hc > 0 ? __fmaf_rn(decay, h[e], acc.get(r4, e)) : h[e];
        const size_t o = (size_t)(blk * 8 + r) * N + 4 * j;
        if (hc > 0) anchor_st<AT>(Hd, o, v, sr, row0 + blk * 8 + r, j);
        float ls = 1.f;
        if constexpr (kNv) {
          float rsc;
          nvfp4_store_row<N, kSh>(v, (uint8_t*)R, Rb, Rs, blk * 8 + r, j, rv, &ls, &rsc,
                                  copy_words<AT>(sr, row0 + blk * 8 + r, j));
          if ((j >> 1) == (blk & 1) * 8 + r) srow = rsc;
        } else if constexpr (kF8) {
          float sr;
          const uint32_t wq = fp8_quant_row(v, &sr);
          *reinterpret_cast<uint32_t*>((uint8_t*)R + o) = wq;
          if (j == 0) Rs[blk * 8 + r] = sr;
          if ((j >> 1) == (blk & 1) * 8 + r) srow = sr;
          fp8_codes(wq, rv);
        } else if constexpr (kBf) {
          __nv_bfloat162 lo2 = __floats2bfloat162_rn(v[0], v[1]), hi2 = __floats2bfloat162_rn(v[2], v[3]);
          uint2 u;
          u.x = *reinterpret_cast<uint32_t*>(&lo2);
          u.y = *reinterpret_cast<uint32_t*>(&hi2);
          *reinterpret_cast<uint2*>((__nv_bfloat16*)R + o) = u;
          Quad<__nv_bfloat16>::unpack(u, rv);
        }
        if constexpr (kOut) {
          pb[r] = Dot<N>::partial(c, rv);
          if constexpr (kNv) pb[r] = __fmul_rn(pb[r], ls);
        }
      }
    }
    if constexpr (kOut) {
      if ((blk & 1) == 0) {
#pragma unroll
        for (int r = 0; r < 8; ++r) part[r] = pb[r];
      } else {
#pragma unroll
        for (int r = 0; r < 8; ++r) part[8 + r] = pb[r];
        float v = reduce_scatter16(part, j);
        if constexpr (kF8 || kNv) v = __fmul_rn(v, srow);
        if ((j & 1) == 0) yo[(blk - 1) * 8 + (j >> 1)] = v;
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) cur[r] = nxt[r];
  }
  __syncwarp();
}

// Position advance inside the decode launch.  Every CTA of a slot adds 1 << 16 to pos[slot] once
// all of its threads have read the position (the low 16 bits); the CTA that completes the count
// (ncta CTAs per slot) stores the new position, which also clears the count.  No CTA of the slot can
// read pos after that store, and pos holds a plain position again when the launch ends.  A position
// outside [0, Q) reads as out of range in every CTA of the slot, so none counts and it is left as
// it was (reported as ERS_EALIGN).
constexpr int kPosBits = 16;
constexpr int32_t kPosMask = (1 << kPosBits) - 1;

// Counts the calling CTA in the upper bits of a slot's position; the last of the slot's ncta CTAs
// stores the new position and gets true.
__device__ __forceinline__ bool advance_pos(int32_t* pos, int ncta, int32_t newp) {
  const int32_t old = atomicAdd(pos, 1 << kPosBits);
  if ((old >> kPosBits) != ncta - 1) return false;
  atomicExch(pos, newp);
  return true;
}

// HT: what the output stream reads (fp32 checkpoint, bf16 or FP8 read copy); W8: the read copy a
// fused refresh writes is FP8 (else bf16, or none when read_copy is null).
// AT: the ReplaySSM anchor (fp32; fp16 written by stochastic rounding; or Nvfp4Shared: the NVFP4 read
// copy is the state itself).
template <typename T, typename HT, bool W8, int P, int N, int QM, typename AT = float>
__global__ void __launch_bounds__(kThreads, 2) k_decode_heads(LaunchArgs a) {
  static_assert(N == 128 && P % 32 == 0, "lane split of Dot<128>; 32-row reduction blocks");
  static_assert(QM <= 32, "one warp scans the chunk");
  extern __shared__ __align__(16) unsigned char hsm[];
  constexpr int QR = heads_rows<QM>();
  T* sB = reinterpret_cast<T*>(hsm);                                  // [QR][N] group B rows 0..p
  T* sxa = sB + QR * N;                                               // [warp][QR][P] x rows 0..p
  float* sg = reinterpret_cast<float*>(sxa + kHeadsPerCta * QR * P);  // [QM] Gram row
  float* syo = sg + QM;                                               // [warp][P] off-diagonal terms
  float* swa = syo + kHeadsPerCta * P;                                // [warp][QM][P] w_s x_s[d] (refresh)
  const int tid = threadIdx.x, w = tid >> 5, j = tid & 31;
  const int i = blockIdx.y;
  const int hpg = a.H / a.G, nbl = (hpg + kHeadsPerCta - 1) / kHeadsPerCta;
  const int g = blockIdx.x / nbl, hb = blockIdx.x % nbl;
  const int hl = hb * kHeadsPerCta + w;  // head within the group
  const bool active = hl < hpg;
  const int h = g * hpg + (active ? hl : 0);
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const bool rssm = (a.flags & ERS_FLAG_REPLAYSSM) != 0;
  const size_t HP = (size_t)a.H * P, GN = (size_t)a.G * N;
  const size_t soff = ((size_t)slot * a.H + h) * P * N;
  RowSrc<HT, N> src;
  if constexpr (std::is_same<HT, Nvfp4>::value) {
    src.c4 = (const uint8_t*)a.read_copy + soff / 2;
    src.bs = a.read_bscale + soff / 16;
  } else {
    src.p = rssm ? (const HT*)a.read_copy + soff : (const HT*)(a.state + soff);
  }
  float sc[2] = {0.f, 0.f};   // FP8 / NVFP4 read copy: scales of rows j and 32 + j
  if constexpr (kRowScale<HT>) {
    const float* Rs = a.read_scale + ((size_t)slot * a.H + h) * P;
    sc[0] = Rs[j];
    sc[1] = Rs[32 + j];
  }
  const int p = a.pos[slot] & kPosMask;
  const int ncta = a.G * nbl;   // CTAs that read this slot's position
  float c[4];
  load_k<T, 4>((const T*)a.C + (size_t)i * GN + (size_t)g * N + 4 * j, c);
  typename RawOf<HT>::type q[rows_in_flight<HT>()];
  if (!kStaged<HT> && active && a.part != kPartFlushes) {   // the first launch of a split call streams anchors only
#pragma unroll
    for (int r = 0; r < rows_in_flight<HT>(); ++r) q[r] = src.ld(r, j);
  }
  const bool fuse = (a.flags & ERS_FLAG_FUSE_REFRESH) != 0;
  // ReplaySSM with a fused flush: a slot holding h = L committed records (h + 1 > L) first folds
  // them into the anchor and recasts its read copy, then decodes the new token as record 0
  const bool flush = !std::is_same<HT, float>::value && rssm && fuse && p == a.Q;
  if (p > a.Q || (p == a.Q && !flush)) {   // the same for every CTA of the slot: none counts, pos stays
    if (tid == 0) report(a.status, ERS_EALIGN);
    return;
  }
  // exact mode (which streams the fp32 checkpoint) refreshes when the new token fills the chunk
  const bool refresh = std::is_same<HT, float>::value && !rssm && fuse && p + 1 == a.Q;
  // a split call (a fused refresh or flush, one CTA per group): the first launch does the slots
  // whose step fills the chunk (exact mode) or flushes (ReplaySSM), the second the others
  const bool heavy = flush || refresh;
  if (a.part == kPartFlushes) {
    allow_dependents();
    if (!heavy) return;
  } else if (a.part == kPartPlain) {
    if (last_cta_of_grid()) wait_primary();
    if (heavy) {   // done by the first launch; its position advances here
      __syncthreads();   // every thread of the CTA has read the position
      if (tid == 0) advance_pos(&a.pos[slot], ncta, refresh ? 0 : 1);
      return;
    }
  }
  uint8_t* stage = reinterpret_cast<uint8_t*>(swa) + (size_t)w * (heads_table_bytes<P, N, QM>() / kHeadsPerCta);
  if constexpr (kStaged<HT>) {   // a plain step: the head's copy into shared memory, all at once
    if (!flush && active) {
      constexpr int kCodeBytes = P * N / 2;
      const uint8_t* cg = (const uint8_t*)a.read_copy + soff / 2;
      for (int k = j; k < kCodeBytes / 16; k += 32) cp_async16(stage + 16 * k, cg + 16 * k);
      for (int k = j; k < P * N / 16 / 16; k += 32) cp_async16(stage + kCodeBytes + 16 * k, a.read_bscale + soff / 16 + 16 * k);
    }
  }
  const int o0 = flush ? p : 0, pn = p - o0;   // output rows s = 0..pn are smem rows o0 + s
  // buffer rows 0..p-1 and the new token as row p: the group's B rows, this head's x rows
  const T* bB = (const T*)a.bB + (size_t)g * N;   // buffer row r at buf_row(a, slot, r)
  const T* nB = (const T*)a.B + (size_t)i * GN + (size_t)g * N;
  constexpr int kBChunks = N * sizeof(T) / 16, kXChunks = P * sizeof(T) / 16;
  for (int k = tid; k < (p + 1) * kBChunks; k += kThreads) {
    const int s = k / kBChunks, e = k % kBChunks;
    cp_async16(reinterpret_cast<char*>(sB + s * N) + 16 * e,
               reinterpret_cast<const char*>(s < p ? bB + buf_row(a, slot, s) * GN : nB) + 16 * e);
  }
  T* sx = sxa + w * QR * P;
  const T* bx = (const T*)a.bx + (size_t)h * P;
  const T* nx = (const T*)a.x + (size_t)i * HP + (size_t)h * P;
  if (active)
    for (int k = j; k < (p + 1) * kXChunks; k += 32) {
      const int s = k / kXChunks, e = k % kXChunks;
      cp_async16(reinterpret_cast<char*>(sx + s * P) + 16 * e,
                 reinterpret_cast<const char*>(s < p ? bx + buf_row(a, slot, s) * HP : nx) + 16 * e);
    }
  const float dt_buf = j < p ? a.bdt[buf_row(a, slot, j) * a.H + h] : 0.f;
  const float dt_raw = j <= pn ? (o0 + j < p ? dt_buf : a.dt[(size_t)i * a.H + h]) : 0.f;
  float dl = 0.f;
  df v = {0.f, 0.f};
  if (j <= pn) {
    dl = delta_of(dt_raw, a.dt_bias[h]);
    v.hi = __fmul_rn(dl, a.A[h]);
  }
  // this head's log-decay prefix (lane s holds row s) and the group's Gram row, while the first
  // state rows are in flight
  v = warp_scan_df(v, j);
  const df at = {__shfl_sync(kFull, v.hi, pn), __shfl_sync(kFull, v.lo, pn)};
  cp_async_wait_all();
  __syncthreads();
  // A fused flush stores the new token as buffer row 0, which is a committed record that every CTA
  // of the slot folds.  With one CTA per group (nbl == 1) each group's rows are read and written by
  // that CTA alone; with several, the group's B/C rows are written only by the slot's last CTA to
  // count itself, after every CTA of the slot has finished reading its rows (fences on both sides
  // of the count order those reads before the writes).
  const bool shared_rows = flush && nbl > 1;
  __shared__ int last_cta;
  if (tid == 0) {
    if (shared_rows) __threadfence();
    last_cta = a.part == kPartFlushes ? 0 : advance_pos(&a.pos[slot], ncta, refresh ? 0 : pn + 1);
    if (shared_rows) __threadfence();
  }
  for (int s = w; s <= pn; s += kHeadsPerCta) {
    float bs[4];
    lds4(sB + (o0 + s) * N + 4 * j, bs);
    const float gv = Dot<N>::reduce(Dot<N>::partial(c, bs));
    if (j == 0) sg[s] = gv;
  }
  __syncthreads();
  if (!active) return;
  float M = 0.f;
  if (j <= pn) M = __fmul_rn(__fmul_rn(sg[j], dl), expf(df_diff(at, v)));
  float* yo = syo + w * P;
  if (refresh) {
    float* wx = swa + w * QM * P;
    const float wl = j <= p ? __fmul_rn(dl, expf(df_diff(at, v))) : 0.f;   // state_weights
    for (int s = 0; s <= p; ++s) {                                          // chunk_state's w_s x_s[d]
      const float ws = __shfl_sync(kFull, wl, s);
#pragma unroll
      for (int m = 0; m < P / 32; ++m) wx[s * P + 32 * m + j] = __fmul_rn(ws, to_f(sx[s * P + 32 * m + j]));
    }
    __syncwarp();
    if constexpr (W8) {   // the copy pointers are compile-time nulls in the other variants (fewer live registers)
      stream_state_refresh<T, P, N>(a.state + soff, nullptr, (uint8_t*)a.read_copy + soff,
                                    a.read_scale + ((size_t)slot * a.H + h) * P, c[0], c[1], c[2], c[3], yo, j, p,
                                    wx, expf(at.hi), sB);
    } else {
      __nv_bfloat16* Rd = a.read_copy ? (__nv_bfloat16*)a.read_copy + soff : nullptr;
      stream_state_refresh<T, P, N>(a.state + soff, Rd, nullptr, nullptr, c[0], c[1], c[2], c[3], yo, j, p, wx,
                                    expf(at.hi), sB);
    }
  } else if (flush) {
    // the committed records' weights (chunk_state's state_weights over rows 0..p-1) and decay
    float* wx = swa + w * QM * P;
    float dc = 0.f;
    df vc = {0.f, 0.f};
    if (j < p) {
      dc = delta_of(dt_buf, a.dt_bias[h]);
      vc.hi = __fmul_rn(dc, a.A[h]);
    }
    vc = warp_scan_df(vc, j);
    const df last = {__shfl_sync(kFull, vc.hi, p - 1), __shfl_sync(kFull, vc.lo, p - 1)};
    const float wl = j < p ? __fmul_rn(dc, expf(df_diff(last, vc))) : 0.f;
    for (int s = 0; s < p; ++s) {
      const float ws = __shfl_sync(kFull, wl, s);
#pragma unroll
      for (int m = 0; m < P / 32; ++m) wx[s * P + 32 * m + j] = __fmul_rn(ws, to_f(sx[s * P + 32 * m + j]));
    }
    __syncwarp();
    if constexpr (!std::is_same<HT, float>::value)
      stream_flush_copy<T, HT, P, N, true, AT>(anchor_ptr<AT>(a, soff),
                                     std::is_same<HT, Nvfp4>::value ? (void*)((uint8_t*)a.read_copy + soff / 2)
                                                                    : (void*)((HT*)a.read_copy + soff),
                                     a.read_bscale + soff / 16, a.read_scale + ((size_t)slot * a.H + h) * P, c[0],
                                     c[1], c[2], c[3], yo, j, p, wx, expf(last.hi), sB,
                                     SrCtr{a.sr_key0, a.sr_key1, a.sr_nonce, (uint32_t)slot}, (uint32_t)(h * P));
  } else if constexpr (kStaged<HT>) {   // rows from the staged copy (landed before the last barrier)
    RowSmem<HT, N> ss;
    ss.c4 = stage;
    ss.bs = stage + P * N / 2;
#pragma unroll
    for (int r = 0; r < rows_in_flight<HT>(); ++r) q[r] = ss.ld(r, j);
    stream_state<HT, P, N>(ss, q, c, yo, j, sc);
  } else {
    stream_state<HT, P, N>(src, q, c, yo, j, sc);
  }
  // outputs d = 32k + j
  const float et = expf(at.hi), Dh = a.D[h];
  T* y = (T*)a.y + (size_t)i * HP + (size_t)h * P;
#pragma unroll
  for (int k = 0; k < P / 32; ++k) {
    const int d = 32 * k + j;
    float acc = 0.f;
    for (int s = 0; s <= pn; ++s) acc = __fmaf_rn(__shfl_sync(kFull, M, s), to_f(sx[(o0 + s) * P + d]), acc);
    y[d] = from_f<T>(combine_out(et, yo[d], acc, Dh, to_f(sx[p * P + d])));
  }
  // append the new token to the buffer (B/C once per group)
  const long long brow = buf_row(a, slot, pn);
  T* dx = (T*)a.bx + brow * HP + (size_t)h * P;
  for (int d = j; d < P; d += 32) dx[d] = sx[p * P + d];
  if (j == 0) a.bdt[brow * a.H + h] = a.dt[(size_t)i * a.H + h];
  if (shared_rows) {
    if (last_cta && w == 0) {   // every group's rows of the slot, from the new token's inputs
      for (int e = j; e < a.G * N; e += 32) {
        ((T*)a.bB)[brow * GN + e] = ((const T*)a.B)[(size_t)i * GN + e];
        ((T*)a.bC)[brow * GN + e] = ((const T*)a.C)[(size_t)i * GN + e];
      }
    }
  } else if (hl == 0) {   // lane j's 4 values of the group's rows: B from shared memory, C from its registers
    const size_t dst = brow * GN + (size_t)g * N + 4 * j;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      ((T*)a.bB)[dst + e] = sB[p * N + 4 * j + e];
      ((T*)a.bC)[dst + e] = from_f<T>(c[e]);   // exact: c holds io values
    }
  }
}

template <typename T, int P, int N, int QM>
cudaError_t launch_decode_heads(const LaunchArgs& a, cudaStream_t s) {
  const int hpg = a.H / a.G, nbl = (hpg + kHeadsPerCta - 1) / kHeadsPerCta;
  const dim3 grid(a.G * nbl, a.nseq);
  constexpr size_t sm = heads_smem_bytes<T, P, N, QM>();
  const bool rssm = (a.flags & ERS_FLAG_REPLAYSSM) != 0;
  // a fused refresh (exact mode) or flush (ReplaySSM) with one CTA per group: two launches
  // (launch_parts), the slots whose step refreshes or flushes first
  const bool split = (a.flags & ERS_FLAG_FUSE_REFRESH) && nbl == 1;
  auto run = [&](auto kernel) {
    cudaError_t e = prep(kernel, sm);
    if (e != cudaSuccess) return e;
    if (split) return launch_parts(kernel, grid, kThreads, sm, s, a);
    kernel<<<grid, kThreads, sm, s>>>(a);
    return cudaGetLastError();   // the kernel advances the positions itself
  };
  if constexpr (QM <= 16 && std::is_same<T, __nv_bfloat16>::value) {   // fp16 anchors: ReplaySSM only
    if (a.anchor_shared && rssm && a.read_nvfp4) return run(k_decode_heads<T, Nvfp4, false, P, N, QM, Nvfp4Shared>);
    if (a.anchor_f16 && rssm) {
      if (a.read_nvfp4) return run(k_decode_heads<T, Nvfp4, false, P, N, QM, __half>);
      if (a.read_fp8) return run(k_decode_heads<T, uint8_t, true, P, N, QM, __half>);
      return run(k_decode_heads<T, __nv_bfloat16, false, P, N, QM, __half>);
    }
  }
  if (a.anchor_f16 || a.anchor_shared) return cudaErrorNotSupported;
  if constexpr (QM <= 16) {   // FP8 read copies: chunk <= 16 only (checked by the API)
    if (a.read_fp8)
      return rssm ? run(k_decode_heads<T, uint8_t, true, P, N, QM>) : run(k_decode_heads<T, float, true, P, N, QM>);
  }
  if constexpr (QM <= 16) {   // NVFP4 read copies: ReplaySSM mode, chunk <= 16 (checked by the API)
    if (a.read_nvfp4 && rssm) return run(k_decode_heads<T, Nvfp4, false, P, N, QM>);
  }
  if (a.read_fp8 || a.read_nvfp4) return cudaErrorNotSupported;
  return rssm ? run(k_decode_heads<T, __nv_bfloat16, false, P, N, QM>) : run(k_decode_heads<T, float, false, P, N, QM>);
}

// ---- standalone refresh (ers_refresh) on the warp-per-head layout ---------------------------------------
// Exact mode: slots with pos == Q fold their Q buffered rows; ReplaySSM: slots with pos + T > L fold
// their pos committed records (pos = 0: the anchor keeps its bits, the copy is recast).  The same
// arithmetic as k_refresh and the fused flushes (state_weights, chunk_state, fold_state order), one
// CTA per (sequence, 8 heads of a group), so a launch has 8x fewer CTAs than one per (sequence,
// head), and the read copy (bf16, FP8 or NVFP4) is cast in the same pass from the fp32 values.
// Positions are reset by k_setpos afterwards.
template <typename T, typename HT, int P, int N, int QM, typename AT = float>
__global__ void __launch_bounds__(kThreads, 2) k_refresh_heads(LaunchArgs a) {
  extern __shared__ __align__(16) unsigned char rsm[];
  T* sB = reinterpret_cast<T*>(rsm);                          // [QM][N] group B rows
  T* sxa = sB + QM * N;                                       // [warp][QM][P] x rows
  float* swa = reinterpret_cast<float*>(sxa + kHeadsPerCta * QM * P);   // [warp][QM][P] w_s x_s[d]
  const int tid = threadIdx.x, w = tid >> 5, j = tid & 31;
  const int i = blockIdx.y;
  const int hpg = a.H / a.G, nbl = (hpg + kHeadsPerCta - 1) / kHeadsPerCta;
  const int g = blockIdx.x / nbl, hb = blockIdx.x % nbl;
  const int hl = hb * kHeadsPerCta + w;
  const bool active = hl < hpg;
  const int h = g * hpg + (active ? hl : 0);
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const int p = a.pos[slot];
  if (p < 0 || p > a.Q) {
    if (tid == 0) report(a.status, ERS_EALIGN);
    return;
  }
  const bool rssm = (a.flags & ERS_FLAG_REPLAYSSM) != 0;
  if (!(rssm ? (p + a.T > a.Q) : (p == a.Q))) return;
  if (std::is_same<AT, Nvfp4Shared>::value && p == 0) return;   // an empty history leaves the state as it is
  const size_t HP = (size_t)a.H * P, GN = (size_t)a.G * N;
  const T* bB = (const T*)a.bB + (size_t)g * N;
  constexpr int kBChunks = N * sizeof(T) / 16, kXChunks = P * sizeof(T) / 16;
  for (int k = tid; k < p * kBChunks; k += kThreads) {
    const int s = k / kBChunks, e = k % kBChunks;
    cp_async16(reinterpret_cast<char*>(sB + s * N) + 16 * e,
               reinterpret_cast<const char*>(bB + buf_row(a, slot, s) * GN) + 16 * e);
  }
  T* sx = sxa + w * QM * P;
  const T* bx = (const T*)a.bx + (size_t)h * P;
  if (active)
    for (int k = j; k < p * kXChunks; k += 32) {
      const int s = k / kXChunks, e = k % kXChunks;
      cp_async16(reinterpret_cast<char*>(sx + s * P) + 16 * e,
                 reinterpret_cast<const char*>(bx + buf_row(a, slot, s) * HP) + 16 * e);
    }
  float dc = 0.f;
  df vc = {0.f, 0.f};
  if (j < p) {
    dc = delta_of(a.bdt[buf_row(a, slot, j) * a.H + h], a.dt_bias[h]);
    vc.hi = __fmul_rn(dc, a.A[h]);
  }
  vc = warp_scan_df(vc, j);
  cp_async_wait_all();
  __syncthreads();
  if (!active) return;
  float* wx = swa + w * QM * P;
  float decay = 1.f;
  if (p > 0) {
    const df last = {__shfl_sync(kFull, vc.hi, p - 1), __shfl_sync(kFull, vc.lo, p - 1)};
    const float wl = j < p ? __fmul_rn(dc, expf(df_diff(last, vc))) : 0.f;   // state_weights
    for (int s = 0; s < p; ++s) {
      const float ws = __shfl_sync(kFull, wl, s);
#pragma unroll
      for (int m = 0; m < P / 32; ++m) wx[s * P + 32 * m + j] = __fmul_rn(ws, to_f(sx[s * P + 32 * m + j]));
    }
    __syncwarp();
    decay = expf(last.hi);
  }
  const size_t soff = ((size_t)slot * a.H + h) * P * N;
  void* R = std::is_same<HT, Nvfp4>::value ? (void*)((uint8_t*)a.read_copy + soff / 2)
                                           : (void*)((uint8_t*)a.read_copy + soff * sizeof_copy<HT>());
  stream_flush_copy<T, HT, P, N, false, AT>(anchor_ptr<AT>(a, soff), R, a.read_bscale + soff / 16,
                                            a.read_scale + ((size_t)slot * a.H + h) * P, 0.f, 0.f, 0.f, 0.f, nullptr,
                                            j, p, wx, decay, sB,
                                            SrCtr{a.sr_key0, a.sr_key1, a.sr_nonce, (uint32_t)slot},
                                            (uint32_t)(h * P));
}

template <typename T, int P, int N, int QM>
constexpr size_t refresh_heads_smem_bytes() {
  return (size_t)QM * N * sizeof(T) + (size_t)kHeadsPerCta * QM * P * sizeof(T) +
         (size_t)kHeadsPerCta * QM * P * sizeof(float);
}

template <typename T, int P, int N, int QM>
cudaError_t launch_refresh_heads(const LaunchArgs& a, cudaStream_t s) {
  const int hpg = a.H / a.G, nbl = (hpg + kHeadsPerCta - 1) / kHeadsPerCta;
  const dim3 grid(a.G * nbl, a.nseq);
  constexpr size_t sm = refresh_heads_smem_bytes<T, P, N, QM>();
  auto run = [&](auto kernel) {
    cudaError_t e = prep(kernel, sm);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, sm, s>>>(a);
    return cudaGetLastError();
  };
  if constexpr (QM <= 16 && std::is_same<T, __nv_bfloat16>::value) {   // fp16 anchors (checked by the API)
    if (a.anchor_shared && a.read_nvfp4) return run(k_refresh_heads<T, Nvfp4, P, N, QM, Nvfp4Shared>);
    if (a.anchor_f16) {
      if (a.read_nvfp4) return run(k_refresh_heads<T, Nvfp4, P, N, QM, __half>);
      if (a.read_fp8) return run(k_refresh_heads<T, uint8_t, P, N, QM, __half>);
      return run(k_refresh_heads<T, __nv_bfloat16, P, N, QM, __half>);
    }
  }
  if (a.anchor_f16 || a.anchor_shared) return cudaErrorNotSupported;
  if (a.read_copy == nullptr) return run(k_refresh_heads<T, NoCopy, P, N, QM>);
  if constexpr (QM <= 16) {
    if (a.read_nvfp4) return run(k_refresh_heads<T, Nvfp4, P, N, QM>);
    if (a.read_fp8) return run(k_refresh_heads<T, uint8_t, P, N, QM>);
  }
  if (a.read_fp8 || a.read_nvfp4) return cudaErrorNotSupported;
  return run(k_refresh_heads<T, __nv_bfloat16, P, N, QM>);
}

}  // namespace

bool heads_decode_supported(int P, int N, int Q) { return N == 128 && (P == 64) && Q >= 1 && Q <= 32; }

cudaError_t heads_refresh(const LaunchArgs& a, cudaStream_t s) {
  constexpr int P = 64, N = 128;
  if (a.io == ERS_DTYPE_BF16) {
    if (a.Q <= 16) return launch_refresh_heads<__nv_bfloat16, P, N, 16>(a, s);
    return launch_refresh_heads<__nv_bfloat16, P, N, 32>(a, s);
  }
  if (a.Q <= 16) return launch_refresh_heads<float, P, N, 16>(a, s);
  return launch_refresh_heads<float, P, N, 32>(a, s);
}

cudaError_t heads_decode(const LaunchArgs& a, cudaStream_t s) {
  constexpr int P = 64, N = 128;
  if (a.io == ERS_DTYPE_BF16) {
    if (a.Q <= 16) return launch_decode_heads<__nv_bfloat16, P, N, 16>(a, s);
    return launch_decode_heads<__nv_bfloat16, P, N, 32>(a, s);
  }
  if (a.Q <= 16) return launch_decode_heads<float, P, N, 16>(a, s);
  return launch_decode_heads<float, P, N, 32>(a, s);
}

}  // namespace ers

