// Output-only speculative verify for small chunks (chunk <= 32, P = 64, N = 128, up to 4 drafts,
// at most 8 heads per B/C group): the bandwidth-shaped verify kernel of the CUDA-core engine.
//
// ReplaySSM ("Motivation and method", "Core equations"): outputs of the T draft tokens are computed
// causally from the low-precision read copy over the committed records plus drafts 1..s; the
// commit moves only the pointer.  A slot whose committed pointer h would overflow (h + T > L)
// first folds its h records into the fp32 anchor and recasts the read copy from the same unrounded
// values.  The arithmetic is the engine's, operation for operation (k_verify_flush and k_verify in
// ers_fma.cu: load_rows, state_weights, chunk_state, fold_state, row_output), so verify equals
// ReplaySSM-mode replay decode bit for bit.
//
// One CTA per (sequence, B/C group), one warp per head.  A warp streams its head's state once:
// the bf16 read copy, or, for a flushing slot, the fp32 anchor, which it folds, writes back and
// recasts row by row, feeding the freshly cast bf16 values (the values the read copy now holds)
// to the drafts' dot products.  The T drafts' lane partials of 8 rows are reduce-scattered
// together (32 values, one shuffle each).  The flush and the outputs are one launch because each
// warp reads only its own head's state and the CTA's own group rows, which it has staged in shared
// memory before any draft is written into the buffer.
#include <type_traits>

#include "ers_common.cuh"
#include "ers_internal.h"
#include "warp_heads.cuh"

namespace ers {
namespace {

using namespace wh;

constexpr int kDraftsMax = 4;
constexpr int kVerifyRowsInFlight = 8;

template <typename T, int P, int N, int QM>
constexpr size_t verify_smem_bytes() {
  constexpr int QR = QM + kDraftsMax;
  return (size_t)QR * N * sizeof(T)                                  // B rows: committed, then drafts
         + (size_t)kHeadsPerCta * QR * P * sizeof(T)                 // x rows, per warp
         + (size_t)kDraftsMax * QR * sizeof(float)                   // Gram rows, per draft
         + (size_t)kHeadsPerCta * kDraftsMax * P * sizeof(float)     // off-diagonal terms, per warp
         + (size_t)kHeadsPerCta *                                    // flush w_s x_s[d], or a plain
               ((size_t)QM * P * sizeof(float) > staged_bytes<P, N>()     // step's staged NVFP4 copy, per warp
                    ? (size_t)QM * P * sizeof(float)
                    : staged_bytes<P, N>());
}

// Read-copy stream: yo[k * P + d] = Dot<128>(C of draft k, R[d]) for all rows d.  q holds rows
// [0, kVerifyRowsInFlight) on entry.  FP8 and NVFP4 copies are read as codes: NVFP4 lane partials
// are scaled by their block scale and each row's dot products by the row scale (lane d % 32 holds
// it in sc[d / 32]), as in the decode stream.
template <typename HT, int P, int N, typename Src>
__device__ __forceinline__ void stream_read_copy(const Src& src,
                                                 typename RawOf<HT>::type (&q)[kVerifyRowsInFlight],
                                                 const float (&c)[kDraftsMax][4], float* yo, int j,
                                                 const float (&sc)[2]) {
  constexpr int NBLK = P / 8, QB = kVerifyRowsInFlight / 8;
#pragma unroll
  for (int blk = 0; blk < NBLK; ++blk) {
    float part[32];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int qs = (blk % QB) * 8 + r;
      float hv[4], ls;
      row_values<HT>(q[qs], hv, &ls);
#pragma unroll
      for (int k = 0; k < kDraftsMax; ++k) {
        part[k * 8 + r] = Dot<N>::partial(c[k], hv);
        if constexpr (kLaneScale<HT>) part[k * 8 + r] = __fmul_rn(part[k * 8 + r], ls);
      }
      if (blk + QB < NBLK) q[qs] = src.ld(blk * 8 + r + kVerifyRowsInFlight, j);
    }
    float v = reduce_scatter32(part, j);   // draft j / 8, row blk * 8 + j % 8
    if constexpr (kRowScale<HT>)
      v = __fmul_rn(v, __shfl_sync(kFull, sc[(blk * 8) >> 5], (blk * 8 + (j & 7)) & 31));
    yo[(j >> 3) * P + blk * 8 + (j & 7)] = v;
  }
  __syncwarp();
}

// Flush stream: each anchor row is folded with the committed records (chunk_state / fold_state
// order: acc = fma(w_s x_s[d], B_s[n], acc) over s < hc, then fma(decay, H, acc)), written back to
// the anchor, cast into the read copy (CT: bf16, FP8 or NVFP4), and the cast values feed the
// drafts' dot products (yo as above).  wx[s * P + d] = w_s x_s[d] is precomputed per warp; 8 rows
// per pass.
template <typename T, typename CT, int P, int N, typename AT>
__device__ __noinline__ void stream_anchor_flush(AT* __restrict__ Hd, void* __restrict__ R,
                                                 uint8_t* __restrict__ Rb, float* __restrict__ Rs,
                                                 const float (&c)[kDraftsMax][4], float* yo, int j, int hc,
                                                 const float* wx, float decay, const T* sB, SrCtr sr, uint32_t row0) {
  constexpr bool kF8 = std::is_same<CT, uint8_t>::value, kNv = std::is_same<CT, Nvfp4>::value;
  constexpr bool kSh = std::is_same<AT, Nvfp4Shared>::value;   // the NVFP4 copy is the state
  static_assert(!kSh || kNv, "a shared state is an NVFP4 copy");
#pragma unroll 1
  for (int d0 = 0; d0 < P; d0 += 8) {
    float h[8][4];
    Fold4 acc[2];   // rows d0..d0+3, d0+4..d0+7
#pragma unroll
    for (int r = 0; r < 8; ++r) Quad<float>::unpack(anchor_row<AT, N>(Hd, R, Rb, Rs, d0 + r, j), h[r]);
    acc[0].zero();
    acc[1].zero();
    for (int s = 0; s < hc; ++s) {
      float bs[4];
      lds4(sB + s * N + 4 * j, bs);
      acc[0].add(*reinterpret_cast<const float4*>(wx + s * P + d0), bs);
      acc[1].add(*reinterpret_cast<const float4*>(wx + s * P + d0 + 4), bs);
    }
    float part[32];
    float srow = 0.f;   // FP8: scale of row d0 + j % 8
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = __fmaf_rn(decay, h[r][e], acc[r >> 2].get(r & 3, e));
      const size_t o = (size_t)(d0 + r) * N + 4 * j;
      anchor_st<AT>(Hd, o, v, sr, row0 + d0 + r, j);
      float rv[4];   // what the read copy now holds (FP8 / NVFP4: the codes, scaled as they are read)
      float ls = 1.f;
      if constexpr (kNv) {
        float s;
        nvfp4_store_row<N, kSh>(v, (uint8_t*)R, Rb, Rs, d0 + r, j, rv, &ls, &s, copy_words<AT>(sr, row0 + d0 + r, j));
        if ((j & 7) == r) srow = s;
      } else if constexpr (kF8) {
        float s;
        const uint32_t wq = fp8_quant_row(v, &s);
        *reinterpret_cast<uint32_t*>((uint8_t*)R + o) = wq;
        if (j == 0) Rs[d0 + r] = s;
        if ((j & 7) == r) srow = s;
        fp8_codes(wq, rv);
      } else {
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(v[0], v[1]), hi2 = __floats2bfloat162_rn(v[2], v[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo2);
        u.y = *reinterpret_cast<uint32_t*>(&hi2);
        *reinterpret_cast<uint2*>((__nv_bfloat16*)R + o) = u;
        Quad<__nv_bfloat16>::unpack(u, rv);
      }
#pragma unroll
      for (int k = 0; k < kDraftsMax; ++k) {
        part[k * 8 + r] = Dot<N>::partial(c[k], rv);
        if constexpr (kNv) part[k * 8 + r] = __fmul_rn(part[k * 8 + r], ls);
      }
    }
    float v = reduce_scatter32(part, j);
    if constexpr (kF8 || kNv) v = __fmul_rn(v, srow);
    yo[(j >> 3) * P + d0 + (j & 7)] = v;
  }
  __syncwarp();
}

template <typename T, typename HT, int P, int N, int QM, typename AT = float>
__global__ void __launch_bounds__(kThreads, 2) k_verify_heads(LaunchArgs a) {
  static_assert(N == 128 && P % 8 == 0 && QM <= 32 - kDraftsMax, "lane split of Dot<128>; one warp scans");
  constexpr int QR = QM + kDraftsMax;
  extern __shared__ __align__(16) unsigned char vsm[];
  T* sB = reinterpret_cast<T*>(vsm);
  T* sxa = sB + QR * N;
  float* sg = reinterpret_cast<float*>(sxa + kHeadsPerCta * QR * P);
  float* syo = sg + kDraftsMax * QR;
  float* swa = syo + kHeadsPerCta * kDraftsMax * P;
  const int tid = threadIdx.x, w = tid >> 5, j = tid & 31;
  const int i = blockIdx.y, g = blockIdx.x;
  const int hpg = a.H / a.G;
  const bool active = w < hpg;
  const int h = g * hpg + (active ? w : 0);
  const int Td = a.T;
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const int hc = a.pos[slot];
  if (hc < 0 || hc > a.Q) {
    if (tid == 0) report(a.status, ERS_EALIGN);
    return;
  }
  const bool flush = hc + Td > a.Q;
  if (flush && !(a.flags & ERS_FLAG_AUTO_FLUSH)) {
    if (tid == 0) report(a.status, ERS_EOVERFLOW);
    return;
  }
  if (a.part == kPartFlushes) {   // a split call: the flushing slots only
    allow_dependents();
    if (!flush) return;
  } else if (a.part == kPartPlain) {
    if (last_cta_of_grid()) wait_primary();
    if (flush) return;   // done by the first launch
  }
  const int h0 = flush ? 0 : hc;   // committed rows that precede the drafts
  const size_t HP = (size_t)a.H * P, GN = (size_t)a.G * N;
  const size_t soff = ((size_t)slot * a.H + h) * P * N;
  RowSrc<HT, N> src;   // bf16 values, FP8 codes or NVFP4 codes + block scales
  if constexpr (std::is_same<HT, Nvfp4>::value) {
    src.c4 = (const uint8_t*)a.read_copy + soff / 2;
    src.bs = a.read_bscale + soff / 16;
  } else {
    src.p = (const HT*)a.read_copy + soff;
  }
  float sc[2] = {0.f, 0.f};   // FP8 / NVFP4: scales of rows j and 32 + j
  if constexpr (kRowScale<HT>) {
    if (!flush && active) {
      const float* Rs = a.read_scale + ((size_t)slot * a.H + h) * P;
      sc[0] = Rs[j];
      sc[1] = Rs[32 + j];
    }
  }
  // the drafts' C rows (lane quads); drafts >= T contribute nothing
  float c[kDraftsMax][4];
#pragma unroll
  for (int k = 0; k < kDraftsMax; ++k) {
    if (k < Td) {
      load_k<T, 4>((const T*)a.C + ((size_t)i * Td + k) * GN + (size_t)g * N + 4 * j, c[k]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) c[k][e] = 0.f;
    }
  }
  // a plain step with an NVFP4 copy stages the head's copy in shared memory in one burst and streams
  // the rows from there: read from global memory, 8 rows of 3 bytes per lane in flight are too few
  constexpr bool kStaged = std::is_same<HT, Nvfp4>::value;
  constexpr int kCodeBytes = P * N / 2;
  uint8_t* stage = reinterpret_cast<uint8_t*>(swa) + (size_t)w * staged_bytes<P, N>();
  typename RawOf<HT>::type q[kVerifyRowsInFlight];
  if (!kStaged && !flush && active) {
#pragma unroll
    for (int r = 0; r < kVerifyRowsInFlight; ++r) q[r] = src.ld(r, j);
  }
  if constexpr (kStaged) {
    if (!flush && active) {
      const uint8_t* cg = (const uint8_t*)a.read_copy + soff / 2;
      for (int k = j; k < kCodeBytes / 16; k += 32) cp_async16(stage + 16 * k, cg + 16 * k);
      for (int k = j; k < P * N / 16 / 16; k += 32) cp_async16(stage + kCodeBytes + 16 * k, a.read_bscale + soff / 16 + 16 * k);
    }
  }
  // committed rows 0..hc-1 at smem rows 0..hc-1, drafts at rows QM..QM+T-1
  const T* bB = (const T*)a.bB + (size_t)g * N;   // buffer row r at buf_row(a, slot, r)
  constexpr int kBChunks = N * sizeof(T) / 16, kXChunks = P * sizeof(T) / 16;
  for (int k = tid; k < (hc + Td) * kBChunks; k += kThreads) {
    const int r = k / kBChunks, e = k % kBChunks;
    const T* src = r < hc ? bB + buf_row(a, slot, r) * GN : (const T*)a.B + ((size_t)i * Td + (r - hc)) * GN + (size_t)g * N;
    cp_async16(reinterpret_cast<char*>(sB + (r < hc ? r : QM + r - hc) * N) + 16 * e,
               reinterpret_cast<const char*>(src) + 16 * e);
  }
  T* sx = sxa + w * QR * P;
  if (active) {
    const T* bx = (const T*)a.bx + (size_t)h * P;
    for (int k = j; k < (hc + Td) * kXChunks; k += 32) {
      const int r = k / kXChunks, e = k % kXChunks;
      const T* src = r < hc ? bx + buf_row(a, slot, r) * HP : (const T*)a.x + ((size_t)i * Td + (r - hc)) * HP + (size_t)h * P;
      cp_async16(reinterpret_cast<char*>(sx + (r < hc ? r : QM + r - hc) * P) + 16 * e,
                 reinterpret_cast<const char*>(src) + 16 * e);
    }
  }
  const float dt_c = j < hc ? a.bdt[buf_row(a, slot, j) * a.H + h] : 0.f;
  const float dt_d = j < Td ? a.dt[((size_t)i * Td + j) * a.H + h] : 0.f;
  const float Ah = a.A[h], bias = a.dt_bias[h];
  float* yo = syo + w * kDraftsMax * P;
  if (!kStaged && !flush && active) stream_read_copy<HT, P, N>(src, q, c, yo, j, sc);
  // output rows s < h0 + T: committed rows then drafts
  const int nout = h0 + Td;
  const float dt_o_d = __shfl_sync(kFull, dt_d, max(j - h0, 0) & 31);
  float dl = 0.f;
  df v = {0.f, 0.f};
  if (j < nout) {
    dl = delta_of(j < h0 ? dt_c : dt_o_d, bias);
    v.hi = __fmul_rn(dl, Ah);
  }
  v = warp_scan_df(v, j);
  cp_async_wait_all();
  __syncthreads();
  if constexpr (kStaged) {
    if (!flush && active) {
      const RowSmem<Nvfp4, N> ss{stage, stage + kCodeBytes};
#pragma unroll
      for (int r = 0; r < kVerifyRowsInFlight; ++r) q[r] = ss.ld(r, j);
      stream_read_copy<HT, P, N>(ss, q, c, yo, j, sc);
    }
  }
  // Gram rows of the drafts: G[k][s] = C_{h0+k} . B_s for s <= h0 + k
  for (int k = 0; k < Td; ++k)
    for (int s = w; s <= h0 + k; s += kHeadsPerCta) {
      float bs[4];
      lds4(sB + (s < h0 ? s : QM + s - h0) * N + 4 * j, bs);
      const float gv = Dot<N>::reduce(Dot<N>::partial(c[k], bs));
      if (j == 0) sg[k * QR + s] = gv;
    }
  // a flushing slot folds its committed records (rows 0..hc-1) into the anchor
  float* sw = swa + w * QM * P;
  float decay = 0.f;
  if (flush) {
    float dc = 0.f;
    df vc = {0.f, 0.f};
    if (j < hc) {
      dc = delta_of(dt_c, bias);
      vc.hi = __fmul_rn(dc, Ah);
    }
    vc = warp_scan_df(vc, j);
    const df last = {__shfl_sync(kFull, vc.hi, hc - 1), __shfl_sync(kFull, vc.lo, hc - 1)};
    const float wl = j < hc ? __fmul_rn(dc, expf(df_diff(last, vc))) : 0.f;   // state_weights
    decay = expf(last.hi);
    for (int s = 0; s < hc; ++s) {   // chunk_state's w_s x_s[d], once per (s, d)
      const float ws = __shfl_sync(kFull, wl, s);
#pragma unroll
      for (int m = 0; m < P / 32; ++m) sw[s * P + 32 * m + j] = __fmul_rn(ws, to_f(sx[s * P + 32 * m + j]));
    }
    __syncwarp();
  }
  __syncthreads();
  if (!active) return;
  if (flush)
    stream_anchor_flush<T, HT, P, N, AT>(anchor_ptr<AT>(a, soff),
                                     std::is_same<HT, Nvfp4>::value ? (void*)((uint8_t*)a.read_copy + soff / 2)
                                                                    : (void*)((HT*)a.read_copy + soff),
                                     a.read_bscale + soff / 16, a.read_scale + ((size_t)slot * a.H + h) * P, c, yo,
                                     j, hc, sw, decay, sB, SrCtr{a.sr_key0, a.sr_key1, a.sr_nonce, (uint32_t)slot},
                                         (uint32_t)(h * P));
  // outputs of draft k (row t_k = h0 + k), d = j + 32 m: one pass over the rows s serves every draft
  // (each draft's sum still runs over s = 0..t_k in order)
  const float Dh = a.D[h];
  float Mk[kDraftsMax], et[kDraftsMax];
#pragma unroll
  for (int k = 0; k < kDraftsMax; ++k) {
    Mk[k] = 0.f;
    et[k] = 0.f;
    if (k < Td) {
      const int t = h0 + k;
      const df at = {__shfl_sync(kFull, v.hi, t), __shfl_sync(kFull, v.lo, t)};
      if (j <= t) Mk[k] = __fmul_rn(__fmul_rn(sg[k * QR + j], dl), expf(df_diff(at, v)));
      et[k] = expf(at.hi);
    }
  }
  constexpr int DPL = P / 32;   // outputs per lane and draft
  float acc[kDraftsMax][DPL];
#pragma unroll
  for (int k = 0; k < kDraftsMax; ++k)
#pragma unroll
    for (int m = 0; m < DPL; ++m) acc[k][m] = 0.f;
  const int tlast = h0 + Td - 1;
  for (int s = 0; s <= tlast; ++s) {
    float xs[DPL];
    const T* xr = sx + (s < h0 ? s : QM + s - h0) * P;
#pragma unroll
    for (int m = 0; m < DPL; ++m) xs[m] = to_f(xr[32 * m + j]);
#pragma unroll
    for (int k = 0; k < kDraftsMax; ++k) {
      const float Ms = __shfl_sync(kFull, Mk[k], s);
      if (k < Td && s <= h0 + k) {
#pragma unroll
        for (int m = 0; m < DPL; ++m) acc[k][m] = __fmaf_rn(Ms, xs[m], acc[k][m]);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kDraftsMax; ++k) {
    if (k >= Td) break;
    T* y = (T*)a.y + ((size_t)i * Td + k) * HP + (size_t)h * P;
#pragma unroll
    for (int m = 0; m < DPL; ++m) {
      const int d = 32 * m + j;
      y[d] = from_f<T>(combine_out(et[k], yo[k * P + d], acc[k][m], Dh, to_f(sx[(QM + k) * P + d])));
    }
  }
  // the drafts go to buffer rows h0..h0+T-1 (B/C once per group)
  for (int k = 0; k < Td; ++k) {
    T* dx = (T*)a.bx + buf_row(a, slot, h0 + k) * HP + (size_t)h * P;
    for (int d = j; d < P; d += 32) dx[d] = sx[(QM + k) * P + d];
  }
  if (j < Td) a.bdt[buf_row(a, slot, h0 + j) * a.H + h] = dt_d;
  if (w == 0) {   // lane j's 4 values of each draft's group rows: B from shared memory, C from registers
#pragma unroll
    for (int k = 0; k < kDraftsMax; ++k) {
      if (k < Td) {
        const size_t dst = buf_row(a, slot, h0 + k) * GN + (size_t)g * N + 4 * j;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ((T*)a.bB)[dst + e] = sB[(QM + k) * N + 4 * j + e];
          ((T*)a.bC)[dst + e] = from_f<T>(c[k][e]);   // exact: c holds io values
        }
      }
    }
  }
}

template <typename T, typename HT, int QM, typename AT = float>
cudaError_t launch_verify_heads(const LaunchArgs& a, cudaStream_t s) {
  constexpr int P = 64, N = 128;
  constexpr size_t sm = verify_smem_bytes<T, P, N, QM>();
  cudaError_t e = prep(k_verify_heads<T, HT, P, N, QM, AT>, sm);
  if (e != cudaSuccess) return e;
  if (a.flags & ERS_FLAG_AUTO_FLUSH) return launch_parts(k_verify_heads<T, HT, P, N, QM, AT>, dim3(a.G, a.nseq), kThreads, sm, s, a);
  k_verify_heads<T, HT, P, N, QM, AT><<<dim3(a.G, a.nseq), kThreads, sm, s>>>(a);
  return cudaGetLastError();
}

// ---- exact-mode speculative verify in one pass (exact-replay RFC, sections 3 and 6) ----------------
// Drafts at chunk positions hc + k.  A draft before the chunk end takes its output from the fp32
// checkpoint H and the replay of the chunk's rows up to it, exactly as an exact-mode decode step at
// that position does.  When the drafts run past the chunk end (hc + T > Q), the first kb = Q - hc of
// them complete the chunk, and a later draft takes its output from the checkpoint H' that the chunk
// fold of exact decode would write (fold_state over the Q rows: the committed records and the
// completing drafts), with the replay restarting at the new chunk.  H' is formed row by row from H as
// the rows stream and feeds the later drafts' dot products; nothing is written, so the cache keeps
// its state.  Every operation is exact decode's (scans, Gram rows, the Dot<128> pairings, the fold
// order, combine_out), so each output has the bits of the decode step it stands for.

// The fold stream: H rows and, per 8 rows, the chunk fold H' = fma(decay, H, sum_s w_s x_s[d] B_s) over
// the Q rows; draft k < kb dots H, draft k >= kb dots H' (yo as in stream_read_copy).
// The chunk's row s (committed rows s < hc, then the completing drafts) is smem row s or QM + s - hc.
template <typename T, int P, int N, int QM>
__device__ __noinline__ void stream_exact_fold(const float* __restrict__ Hd, const float (&c)[kDraftsMax][4],
                                               float* yo, int j, int hc, int kb, const float* wx, float decay,
                                               const T* sB) {
  const int q = hc + kb;
#pragma unroll 1
  for (int d0 = 0; d0 < P; d0 += 8) {
    float h[8][4];
    Fold4 acc[2];   // rows d0..d0+3, d0+4..d0+7
#pragma unroll
    for (int r = 0; r < 8; ++r) Quad<float>::unpack(Quad<float>::ld_stream(Hd + (size_t)(d0 + r) * N + 4 * j), h[r]);
    acc[0].zero();
    acc[1].zero();
    for (int s = 0; s < q; ++s) {
      float bs[4];
      lds4(sB + (s < hc ? s : QM + s - hc) * N + 4 * j, bs);
      acc[0].add(*reinterpret_cast<const float4*>(wx + s * P + d0), bs);
      acc[1].add(*reinterpret_cast<const float4*>(wx + s * P + d0 + 4), bs);
    }
    float part[32];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = __fmaf_rn(decay, h[r][e], acc[r >> 2].get(r & 3, e));
#pragma unroll
      for (int k = 0; k < kDraftsMax; ++k) part[k * 8 + r] = Dot<N>::partial(c[k], k < kb ? h[r] : v);
    }
    yo[(j >> 3) * P + d0 + (j & 7)] = reduce_scatter32(part, j);
  }
  __syncwarp();
}

template <typename T, int P, int N, int QM>
__global__ void __launch_bounds__(kThreads, 2) k_verify_exact_heads(LaunchArgs a) {
  static_assert(N == 128 && P % 8 == 0 && QM <= 32 - kDraftsMax, "lane split of Dot<128>; one warp scans");
  constexpr int QR = QM + kDraftsMax;
  extern __shared__ __align__(16) unsigned char vsm[];
  T* sB = reinterpret_cast<T*>(vsm);                                   // [QR] rows: committed, then drafts at QM
  T* sxa = sB + QR * N;                                                // [warp][QR][P]
  float* sg = reinterpret_cast<float*>(sxa + kHeadsPerCta * QR * P);   // [draft][QR] Gram rows
  float* syo = sg + kDraftsMax * QR;                                   // [warp][draft][P]
  float* swa = syo + kHeadsPerCta * kDraftsMax * P;                    // [warp][QM][P] w_s x_s[d]
  const int tid = threadIdx.x, w = tid >> 5, j = tid & 31;
  const int i = blockIdx.y, g = blockIdx.x;
  const int hpg = a.H / a.G;
  const bool active = w < hpg;
  const int h = g * hpg + (active ? w : 0);
  const int Td = a.T;
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const int hc = a.pos[slot];
  if (hc < 0 || hc >= a.Q) {   // an exact-mode position is in [0, Q)
    if (tid == 0) report(a.status, ERS_EALIGN);
    return;
  }
  const int kb = min(Td, a.Q - hc);   // drafts up to the chunk end
  const bool cross = kb < Td;         // later drafts see the folded checkpoint
  const size_t HP = (size_t)a.H * P, GN = (size_t)a.G * N;
  const size_t soff = ((size_t)slot * a.H + h) * P * N;
  RowSrc<float, N> src;
  src.p = a.state + soff;
  float c[kDraftsMax][4];
#pragma unroll
  for (int k = 0; k < kDraftsMax; ++k) {
    if (k < Td) {
      load_k<T, 4>((const T*)a.C + ((size_t)i * Td + k) * GN + (size_t)g * N + 4 * j, c[k]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) c[k][e] = 0.f;
    }
  }
  typename RawOf<float>::type qr[kVerifyRowsInFlight];
  if (!cross && active) {
#pragma unroll
    for (int r = 0; r < kVerifyRowsInFlight; ++r) qr[r] = src.ld(r, j);
  }
  // committed rows 0..hc-1 at smem rows 0..hc-1, drafts at rows QM..QM+T-1
  const T* bB = (const T*)a.bB + (size_t)g * N;
  constexpr int kBChunks = N * sizeof(T) / 16, kXChunks = P * sizeof(T) / 16;
  for (int k = tid; k < (hc + Td) * kBChunks; k += kThreads) {
    const int r = k / kBChunks, e = k % kBChunks;
    const T* s = r < hc ? bB + buf_row(a, slot, r) * GN : (const T*)a.B + ((size_t)i * Td + (r - hc)) * GN + (size_t)g * N;
    cp_async16(reinterpret_cast<char*>(sB + (r < hc ? r : QM + r - hc) * N) + 16 * e, reinterpret_cast<const char*>(s) + 16 * e);
  }
  T* sx = sxa + w * QR * P;
  if (active) {
    const T* bx = (const T*)a.bx + (size_t)h * P;
    for (int k = j; k < (hc + Td) * kXChunks; k += 32) {
      const int r = k / kXChunks, e = k % kXChunks;
      const T* s = r < hc ? bx + buf_row(a, slot, r) * HP : (const T*)a.x + ((size_t)i * Td + (r - hc)) * HP + (size_t)h * P;
      cp_async16(reinterpret_cast<char*>(sx + (r < hc ? r : QM + r - hc) * P) + 16 * e, reinterpret_cast<const char*>(s) + 16 * e);
    }
  }
  const float dt_c = j < hc ? a.bdt[buf_row(a, slot, j) * a.H + h] : 0.f;
  const float dt_d = j < Td ? a.dt[((size_t)i * Td + j) * a.H + h] : 0.f;
  const float Ah = a.A[h], bias = a.dt_bias[h];
  // the old chunk's rows (lane s: committed s < hc, then the completing drafts) and the new chunk's
  // (lane s: draft kb + s); their decay terms and prefix scans, as exact decode builds them
  const float dt_sh = __shfl_sync(kFull, dt_d, max(j - hc, 0) & 31);   // every lane shuffles
  const float dt_new = __shfl_sync(kFull, dt_d, (kb + j) & 31);
  const float dt_old = j < hc ? dt_c : dt_sh;
  float dlo = 0.f, dln = 0.f;
  df vo = {0.f, 0.f}, vn = {0.f, 0.f};
  if (j < hc + kb) {
    dlo = delta_of(dt_old, bias);
    vo.hi = __fmul_rn(dlo, Ah);
  }
  if (j < Td - kb) {
    dln = delta_of(dt_new, bias);
    vn.hi = __fmul_rn(dln, Ah);
  }
  vo = warp_scan_df(vo, j);
  vn = warp_scan_df(vn, j);
  cp_async_wait_all();
  __syncthreads();
  // Gram rows: a draft before the chunk end against the old chunk's rows s <= hc + k, a later one
  // against the new chunk's rows s <= k - kb (smem row of new-chunk row s: QM + kb + s)
  for (int k = 0; k < Td; ++k) {
    const int last = k < kb ? hc + k : k - kb;
    for (int s = w; s <= last; s += kHeadsPerCta) {
      const int row = k < kb ? (s < hc ? s : QM + s - hc) : QM + kb + s;
      float bs[4];
      lds4(sB + row * N + 4 * j, bs);
      const float gv = Dot<N>::reduce(Dot<N>::partial(c[k], bs));
      if (j == 0) sg[k * QR + s] = gv;
    }
  }
  // the chunk fold's w_s x_s[d] over the Q rows (state_weights with the old chunk's last prefix)
  float* sw = swa + w * QM * P;
  float decay = 0.f;
  if (cross) {
    const int q = hc + kb;   // = Q
    const df last = {__shfl_sync(kFull, vo.hi, q - 1), __shfl_sync(kFull, vo.lo, q - 1)};
    const float wl = j < q ? __fmul_rn(dlo, expf(df_diff(last, vo))) : 0.f;
    decay = expf(last.hi);
    for (int s = 0; s < q; ++s) {
      const float ws = __shfl_sync(kFull, wl, s);
      const T* xr = sx + (s < hc ? s : QM + s - hc) * P;
#pragma unroll
      for (int m = 0; m < P / 32; ++m) sw[s * P + 32 * m + j] = __fmul_rn(ws, to_f(xr[32 * m + j]));
    }
    __syncwarp();
  }
  __syncthreads();
  if (!active) return;
  float* yo = syo + w * kDraftsMax * P;
  if (cross) {
    stream_exact_fold<T, P, N, QM>(a.state + soff, c, yo, j, hc, kb, sw, decay, sB);
  } else {
    const float sc[2] = {1.f, 1.f};
    stream_read_copy<float, P, N>(src, qr, c, yo, j, sc);
  }
  // outputs of draft k at d = j + 32 m
  const float Dh = a.D[h];
  constexpr int DPL = P / 32;
  for (int k = 0; k < Td; ++k) {
    const bool pre = k < kb;
    const int t = pre ? hc + k : k - kb;
    const df vv = pre ? vo : vn;
    const float dl = pre ? dlo : dln;
    const df at = {__shfl_sync(kFull, vv.hi, t), __shfl_sync(kFull, vv.lo, t)};
    const float M = j <= t ? __fmul_rn(__fmul_rn(sg[k * QR + j], dl), expf(df_diff(at, vv))) : 0.f;
    float acc[DPL];
#pragma unroll
    for (int m = 0; m < DPL; ++m) acc[m] = 0.f;
    for (int s = 0; s <= t; ++s) {
      const float Ms = __shfl_sync(kFull, M, s);
      const T* xr = sx + (pre ? (s < hc ? s : QM + s - hc) : QM + kb + s) * P;
#pragma unroll
      for (int m = 0; m < DPL; ++m) acc[m] = __fmaf_rn(Ms, to_f(xr[32 * m + j]), acc[m]);
    }
    const float et = expf(at.hi);
    T* y = (T*)a.y + ((size_t)i * Td + k) * HP + (size_t)h * P;
#pragma unroll
    for (int m = 0; m < DPL; ++m) {
      const int d = 32 * m + j;
      y[d] = from_f<T>(combine_out(et, yo[k * P + d], acc[m], Dh, to_f(sx[(QM + k) * P + d])));
    }
  }
}

template <typename T, int QM>
cudaError_t launch_verify_exact_heads(const LaunchArgs& a, cudaStream_t s) {
  constexpr int P = 64, N = 128;
  constexpr size_t sm = verify_smem_bytes<T, P, N, QM>();
  cudaError_t e = prep(k_verify_exact_heads<T, P, N, QM>, sm);
  if (e != cudaSuccess) return e;
  k_verify_exact_heads<T, P, N, QM><<<dim3(a.G, a.nseq), kThreads, sm, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool heads_verify_supported(int P, int N, int Q, int T, int H, int G) {
  return P == 64 && N == 128 && Q >= 1 && Q <= 16 && T >= 1 && T <= kDraftsMax && G > 0 && H % G == 0 &&
         H / G <= kHeadsPerCta;
}

bool exact_verify_supported(int io, int P, int N, int Q, int T, int H, int G) {
  return (io == ERS_DTYPE_BF16 || io == ERS_DTYPE_F32) && P == 64 && N == 128 && Q >= 1 && Q <= 16 && T >= 1 &&
         T <= kDraftsMax && G > 0 && H % G == 0 && H / G <= kHeadsPerCta;
}

cudaError_t exact_verify(const LaunchArgs& a, cudaStream_t s) {
  if (a.io == ERS_DTYPE_BF16) return launch_verify_exact_heads<__nv_bfloat16, 16>(a, s);
  return launch_verify_exact_heads<float, 16>(a, s);
}

cudaError_t heads_verify(const LaunchArgs& a, cudaStream_t s) {
  if (a.anchor_shared) {   // the shared NVFP4 state: bf16 io, an NVFP4 copy (checked by the API)
    if (a.io != ERS_DTYPE_BF16 || !a.read_nvfp4) return cudaErrorNotSupported;
    return launch_verify_heads<__nv_bfloat16, Nvfp4, 16, Nvfp4Shared>(a, s);
  }
  if (a.anchor_f16) {   // fp16 anchors: bf16 io only (checked by the API)
    if (a.io != ERS_DTYPE_BF16) return cudaErrorNotSupported;
    if (a.read_nvfp4) return launch_verify_heads<__nv_bfloat16, Nvfp4, 16, __half>(a, s);
    if (a.read_fp8) return launch_verify_heads<__nv_bfloat16, uint8_t, 16, __half>(a, s);
    return launch_verify_heads<__nv_bfloat16, __nv_bfloat16, 16, __half>(a, s);
  }
  if (a.read_fp8) {
    if (a.io == ERS_DTYPE_BF16) return launch_verify_heads<__nv_bfloat16, uint8_t, 16>(a, s);
    return launch_verify_heads<float, uint8_t, 16>(a, s);
  }
  if (a.read_nvfp4) {
    if (a.io == ERS_DTYPE_BF16) return launch_verify_heads<__nv_bfloat16, Nvfp4, 16>(a, s);
    return launch_verify_heads<float, Nvfp4, 16>(a, s);
  }
  if (a.io == ERS_DTYPE_BF16) return launch_verify_heads<__nv_bfloat16, __nv_bfloat16, 16>(a, s);
  return launch_verify_heads<float, __nv_bfloat16, 16>(a, s);
}

}  // namespace ers
