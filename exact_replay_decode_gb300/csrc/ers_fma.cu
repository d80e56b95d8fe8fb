// CUDA-core ("FMA") chunk engine: every path of the library built on one set of fixed-order
// device functions.
//
// The chunked SSD scan (exact-replay RFC, vLLM issue 55524, section 1) computes, for a chunk of Q
// tokens starting from boundary state H (per head, [P x N]):
//   Acum_t      = sum_{r<=t} delta_r A                           (prefix of log-decays)
//   y_t         = exp(Acum_t) (H C_t) + sum_{s<=t} (C_t . B_s) delta_s exp(Acum_t - Acum_s) x_s + D x_t
//   H'          = exp(Acum_last) H + sum_s delta_s exp(Acum_last - Acum_s) x_s B_s^T
// Exact replay (RFC section 3) recomputes the outputs of a partial chunk from its boundary state
// and buffered inputs.  Here each output element and each chunk state is produced by the same
// device function in every path (row_output / chunk_state below), so prefill, chunked prefill,
// decode, refresh and verify agree bit for bit by construction.
//
// This engine serves fp32 io (all paths) and is the first, simple implementation for bf16 io.
#include <stdio.h>

#include "ers_common.cuh"
#include "ers_internal.h"
#include "tc_common.cuh"

namespace ers {
namespace {

struct FmaSmem {
  float hi[kQMax];     // Acum (double-float, hi part); holds dA before the scan
  float lo[kQMax];
  float delta[kQMax];  // softplus(dt + dt_bias)
  float w[kQMax];      // chunk-state weights delta_s exp(Acum_last - Acum_s)
  float M[kQMax];      // one output row's masked, decayed Gram column
  const void* rowB[kQMax];
  const void* rowC[kQMax];
  float yoff[64];
};
// followed in dynamic shared memory by xs[Q][P] (x rows as fp32)

__host__ __device__ constexpr size_t fma_smem_bytes(int Q, int P) {
  return ((sizeof(FmaSmem) + 15) & ~size_t(15)) + (size_t)Q * P * sizeof(float);
}

// Loads rows [0, nrows) (x as fp32, delta, dA, B/C row pointers), zeroes the rest, and scans the
// log-decays.  All kThreads threads must call it.
template <typename T, int P>
__device__ void load_rows(FmaSmem& sm, float* xs, int nrows, const Rows<T>& rows, float A, float bias) {
  const int tid = threadIdx.x;
  if (tid < kQMax) {
    if (tid < nrows) {
      const float d = delta_of(rows.dt(tid), bias);
      sm.delta[tid] = d;
      sm.hi[tid] = __fmul_rn(d, A);
      sm.rowB[tid] = rows.B(tid);
      sm.rowC[tid] = rows.C(tid);
    } else {
      sm.delta[tid] = 0.f;
      sm.hi[tid] = 0.f;
      sm.rowB[tid] = nullptr;
      sm.rowC[tid] = nullptr;
    }
    sm.lo[tid] = 0.f;
  }
  for (int idx = tid; idx < nrows * P; idx += kThreads) {
    const int r = idx / P, d = idx % P;
    xs[idx] = to_f(rows.x(r)[d]);
  }
  __syncthreads();
  chunk_scan(sm.hi, sm.lo);
}

// y for chunk row t (all kThreads threads call it).  Hd points at the [P x N] boundary state (fp32
// checkpoint/anchor, or the bf16 read copy).  out points at the row's P outputs.
template <typename T, int P, int N, typename HT>
__device__ void row_output(FmaSmem& sm, const float* xs, int t, const HT* __restrict__ Hd, float Dh, T* out) {
  using Dt = Dot<N>;
  constexpr int NG = kThreads / Dt::W;
  const int tid = threadIdx.x;
  const int gid = tid / Dt::W, j = tid % Dt::W;
  float c[Dt::K];
  load_k<T, Dt::K>((const T*)sm.rowC[t] + j * Dt::K, c);
  const df at = {sm.hi[t], sm.lo[t]};
  // masked, decayed Gram column M[s] = (C_t . B_s) delta_s exp(Acum_t - Acum_s), s <= t
  for (int s0 = 0; s0 <= t; s0 += NG) {
    const int s = s0 + gid;
    float b[Dt::K];
    if (s <= t) {
      load_k<T, Dt::K>((const T*)sm.rowB[s] + j * Dt::K, b);
    } else {
#pragma unroll
      for (int k = 0; k < Dt::K; ++k) b[k] = 0.f;
    }
    const float g = Dt::reduce(Dt::partial(c, b));
    if (s <= t && j == 0)
      sm.M[s] = __fmul_rn(__fmul_rn(g, sm.delta[s]), expf(df_diff(at, df{sm.hi[s], sm.lo[s]})));
  }
  // off-diagonal term H C_t, one dot product per headdim row
  for (int d0 = 0; d0 < P; d0 += NG) {
    const int d = d0 + gid;
    float hv[Dt::K];
    if (d < P) {
      load_k<HT, Dt::K>(Hd + (size_t)d * N + j * Dt::K, hv);
    } else {
#pragma unroll
      for (int k = 0; k < Dt::K; ++k) hv[k] = 0.f;
    }
    const float v = Dt::reduce(Dt::partial(c, hv));
    if (d < P && j == 0) sm.yoff[d] = v;
  }
  __syncthreads();
  if (tid < P) {
    float acc = 0.f;
    for (int s = 0; s <= t; ++s) acc = __fmaf_rn(sm.M[s], xs[s * P + tid], acc);
    out[tid] = from_f<T>(combine_out(expf(at.hi), sm.yoff[tid], acc, Dh, xs[t * P + tid]));
  }
  __syncthreads();
}

// Chunk-state weights w_s = delta_s exp(Acum_last - Acum_s) for s < nrows.
__device__ __forceinline__ void state_weights(FmaSmem& sm, int nrows) {
  const int tid = threadIdx.x;
  if (tid < nrows) {
    const df last = {sm.hi[nrows - 1], sm.lo[nrows - 1]};
    sm.w[tid] = __fmul_rn(sm.delta[tid], expf(df_diff(last, df{sm.hi[tid], sm.lo[tid]})));
  }
  __syncthreads();
}

// S[d][n] = sum_{s < nrows} (w_s x_s[d]) B_s[n], in s order.  Thread tid owns elements
// tid + e*kThreads (row-major [P][N]).
template <typename T, int P, int N>
__device__ __forceinline__ void chunk_state(const FmaSmem& sm, const float* xs, int nrows,
                                            float (&acc)[P * N / kThreads]) {
  constexpr int EPT = P * N / kThreads;
  const int tid = threadIdx.x;
#pragma unroll
  for (int e = 0; e < EPT; ++e) acc[e] = 0.f;
  for (int s = 0; s < nrows; ++s) {
    const T* b = (const T*)sm.rowB[s];
    const float ws = sm.w[s];
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int idx = tid + e * kThreads;
      const int d = idx / N, n = idx % N;
      acc[e] = __fmaf_rn(__fmul_rn(ws, xs[s * P + d]), to_f(b[n]), acc[e]);
    }
  }
}

// H' = exp(Acum_last) H + S written over H (fp32) and, if present, the bf16 read copy cast from the
// same fp32 value (ReplaySSM "Core equations": both copies cast independently from one state).
template <int P, int N>
__device__ __forceinline__ void fold_state(float* Hd, __nv_bfloat16* Rd, float decay, const float (&S)[P * N / kThreads]) {
  constexpr int EPT = P * N / kThreads;
  const int tid = threadIdx.x;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int idx = tid + e * kThreads;
    const float v = __fmaf_rn(decay, Hd[idx], S[e]);
    Hd[idx] = v;
    if (Rd != nullptr) Rd[idx] = __float2bfloat16_rn(v);
  }
}

extern __shared__ __align__(16) unsigned char dyn_smem[];

__device__ __forceinline__ FmaSmem& smem_hdr() { return *reinterpret_cast<FmaSmem*>(dyn_smem); }
__device__ __forceinline__ float* smem_xs() {
  return reinterpret_cast<float*>(dyn_smem + ((sizeof(FmaSmem) + 15) & ~size_t(15)));
}

// ---- prefill: chunk states -------------------------------------------------------------------
template <typename T, int P, int N>
__global__ void __launch_bounds__(kThreads) k_prefill_state(LaunchArgs a, bool chunked) {
  const int c = blockIdx.x, i = blockIdx.y, h = blockIdx.z;
  SeqGrid sg;
  if (!seq_grid(a, chunked, i, &sg) || c >= sg.nch) return;
  FmaSmem& sm = smem_hdr();
  float* xs = smem_xs();
  const int nrows = min(a.Q, sg.total - c * a.Q);
  const int nbuf = max(0, sg.p - c * a.Q);
  const Rows<T> rows = make_rows<T>(a, sg.slot, h, nbuf, (long long)a.cu[i] + (long long)c * a.Q - sg.p);
  load_rows<T, P>(sm, xs, nrows, rows, a.A[h], a.dt_bias[h]);
  state_weights(sm, nrows);
  float S[P * N / kThreads];
  chunk_state<T, P, N>(sm, xs, nrows, S);
  const size_t base = (((size_t)i * a.max_chunks + c) * a.H + h);
  float* out = a.ws_states + base * P * N;
#pragma unroll
  for (int e = 0; e < P * N / kThreads; ++e) out[threadIdx.x + e * kThreads] = S[e];
  if (threadIdx.x == 0) a.ws_tot[base] = sm.hi[nrows - 1];
}

// ---- prefill: inter-chunk state passing in fp32 (RFC Evidence 4: the state stays fp32 inside one
// call and is rounded only on store; here it is never rounded) ----------------------------------
template <int P, int N>
__global__ void __launch_bounds__(kThreads) k_prefill_chain(LaunchArgs a, bool chunked) {
  const int i = blockIdx.x, h = blockIdx.y;
  SeqGrid sg;
  if (!seq_grid(a, chunked, i, &sg)) return;
  constexpr int EPT = P * N / kThreads;
  const size_t hs = (size_t)P * N;
  float* ckpt = chunked ? a.state + ((size_t)sg.slot * a.H + h) * hs : nullptr;
  const float* init = chunked ? ckpt : (a.init_state ? a.init_state + ((size_t)i * a.H + h) * hs : nullptr);
  float Hr[EPT], keep[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    Hr[e] = init ? init[threadIdx.x + e * kThreads] : 0.f;
    keep[e] = Hr[e];
  }
  const bool aligned_end = (sg.total % a.Q) == 0;
  for (int c = 0; c < sg.nch; ++c) {
    const size_t base = ((size_t)i * a.max_chunks + c) * a.H + h;
    float* S = a.ws_states + base * hs;
    const float decay = expf(a.ws_tot[base]);
    if (c == sg.nch - 1 && !aligned_end) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) keep[e] = Hr[e];
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int idx = threadIdx.x + e * kThreads;
      const float s = S[idx];
      S[idx] = Hr[e];  // the state at the start of chunk c, read by the output kernel
      Hr[e] = __fmaf_rn(decay, Hr[e], s);
    }
    if (a.chunk_states != nullptr) {
      float* cs = a.chunk_states + base * hs;
#pragma unroll
      for (int e = 0; e < EPT; ++e) cs[threadIdx.x + e * kThreads] = Hr[e];
    }
  }
  if (!chunked) {
    float* fin = a.final_state + ((size_t)i * a.H + h) * hs;
#pragma unroll
    for (int e = 0; e < EPT; ++e) fin[threadIdx.x + e * kThreads] = Hr[e];
  } else if (sg.nch > 0) {
#pragma unroll
    for (int e = 0; e < EPT; ++e) ckpt[threadIdx.x + e * kThreads] = aligned_end ? Hr[e] : keep[e];
  }
}

// ---- prefill: outputs ---------------------------------------------------------------------------
template <typename T, int P, int N>
__global__ void __launch_bounds__(kThreads) k_prefill_out(LaunchArgs a, bool chunked) {
  const int c = blockIdx.x, i = blockIdx.y, h = blockIdx.z;
  SeqGrid sg;
  if (!seq_grid(a, chunked, i, &sg) || c >= sg.nch) return;
  FmaSmem& sm = smem_hdr();
  float* xs = smem_xs();
  const int nrows = min(a.Q, sg.total - c * a.Q);
  const int nbuf = max(0, sg.p - c * a.Q);
  const long long tok0 = (long long)a.cu[i] + (long long)c * a.Q - sg.p;
  const Rows<T> rows = make_rows<T>(a, sg.slot, h, nbuf, tok0);
  load_rows<T, P>(sm, xs, nrows, rows, a.A[h], a.dt_bias[h]);
  const float* Hc = a.ws_states + (((size_t)i * a.max_chunks + c) * a.H + h) * P * N;
  const float Dh = a.D[h];
  T* y = (T*)a.y;
  for (int t = nbuf; t < nrows; ++t)
    row_output<T, P, N, float>(sm, xs, t, Hc, Dh, y + ((tok0 + t) * a.H + h) * P);
}

// ---- replay decode --------------------------------------------------------------------------------
template <typename T, int P, int N>
__global__ void __launch_bounds__(kThreads) k_decode(LaunchArgs a) {
  const int i = blockIdx.x, h = blockIdx.y;
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const bool rssm = (a.flags & ERS_FLAG_REPLAYSSM) != 0;
  const int p = a.pos[slot];
  if (p < 0 || p >= a.Q) {
    if (threadIdx.x == 0) report(a.status, ERS_EALIGN);
    return;
  }
  FmaSmem& sm = smem_hdr();
  float* xs = smem_xs();
  // rows 0..p-1 from the buffer, row p is the new token (input index i == tok0 + p)
  const Rows<T> rows = make_rows<T>(a, slot, h, p, (long long)i - p);
  load_rows<T, P>(sm, xs, p + 1, rows, a.A[h], a.dt_bias[h]);
  const size_t hs = (size_t)P * N;
  float* Hd = a.state + ((size_t)slot * a.H + h) * hs;
  T* y = (T*)a.y + ((size_t)i * a.H + h) * P;
  if (rssm)
    row_output<T, P, N, __nv_bfloat16>(sm, xs, p, (const __nv_bfloat16*)a.read_copy + ((size_t)slot * a.H + h) * hs,
                                       a.D[h], y);
  else
    row_output<T, P, N, float>(sm, xs, p, Hd, a.D[h], y);
  // append the new token to the buffer (B/C once per group)
  const int g = h / (a.H / a.G);
  T* bx = (T*)a.bx + (((size_t)slot * a.Q + p) * a.H + h) * P;
  const T* nx = (const T*)a.x + ((size_t)i * a.H + h) * P;
  for (int d = threadIdx.x; d < P; d += kThreads) bx[d] = nx[d];
  if (threadIdx.x == 0) a.bdt[((size_t)slot * a.Q + p) * a.H + h] = a.dt[(size_t)i * a.H + h];
  if (h % (a.H / a.G) == 0) {
    T* bB = (T*)a.bB + (((size_t)slot * a.Q + p) * a.G + g) * N;
    T* bC = (T*)a.bC + (((size_t)slot * a.Q + p) * a.G + g) * N;
    const T* nB = (const T*)a.B + ((size_t)i * a.G + g) * N;
    const T* nC = (const T*)a.C + ((size_t)i * a.G + g) * N;
    for (int n = threadIdx.x; n < N; n += kThreads) {
      bB[n] = nB[n];
      bC[n] = nC[n];
    }
  }
  // the chunk filled: its final state becomes the new boundary state
  if (!rssm && (a.flags & ERS_FLAG_FUSE_REFRESH) && p + 1 == a.Q) {
    state_weights(sm, a.Q);
    float S[P * N / kThreads];
    chunk_state<T, P, N>(sm, xs, a.Q, S);
    __nv_bfloat16* Rd = a.read_copy ? (__nv_bfloat16*)a.read_copy + ((size_t)slot * a.H + h) * hs : nullptr;
    fold_state<P, N>(Hd, Rd, expf(sm.hi[a.Q - 1]), S);
  }
}

template <typename K>
cudaError_t prep(K kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// ---- replay decode for small chunks, shaped for HBM bandwidth -------------------------------------
// Same arithmetic as k_decode (row_output, state_weights, chunk_state and fold_state, operation for
// operation), organised so that a step costs little more than streaming the boundary state once.
//  * One CTA per (sequence, block of up to 8 heads of one B/C group), one warp per head.  The warp
//    streams its head's [P x N] state through registers, 8 rows at a time, two blocks in flight;
//    lane j holds elements [4j, 4j+4) of each row, the lane split of Dot<128>.
//  * The 32 lane partials of 32 rows are combined by a reduce-scatter whose pairings are those of
//    Dot<128>'s butterfly (xor 16, 8, 4, 2, 1): each stage halves the rows a lane keeps, and lane j
//    ends with row j's dot product, bit-identical to the butterfly (same tree; fp32 addition is
//    commutative) at about one shuffle per row instead of five.
//  * The group's Gram row C_p . B_s is computed once per CTA; buffer rows arrive by cp.async while
//    the state streams; the log-decay scan runs per warp with shuffles (for rows < 32 the strides
//    >= 32 of chunk_scan change nothing, so the bits are chunk_scan's).
//  * When the step fills the chunk, the state is streamed after the chunk's weights are known and
//    each row is folded (fold_state) and written back in the same pass.
constexpr int kHeadsPerCta = kThreads / 32;

template <typename HT> struct Quad;
template <> struct Quad<float> {
  using raw = float4;
  __device__ __forceinline__ static raw ld_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
  __device__ __forceinline__ static void unpack(raw u, float (&v)[4]) {
    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
  }
};
template <> struct Quad<__nv_bfloat16> {
  using raw = uint2;
  __device__ __forceinline__ static raw ld_stream(const __nv_bfloat16* p) {
    return __ldcs(reinterpret_cast<const uint2*>(p));
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

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

template <typename T, int P, int N, int QM>
constexpr size_t heads_smem_bytes() {
  return (size_t)QM * N * sizeof(T) + (size_t)kHeadsPerCta * QM * P * sizeof(T) + QM * sizeof(float) +
         (size_t)kHeadsPerCta * (P + QM) * sizeof(float);
}

// Streams one head's state: lane j of row d reads elements [4j, 4j+4), 8 rows per block, two
// blocks in flight (q holds rows 0..15 on entry).  yo[d] ends with the off-diagonal term (H C_p)[d]
// (per-warp shared memory).
template <typename HT, int P, int N>
__device__ __forceinline__ void stream_state(const HT* __restrict__ Hsrc, typename Quad<HT>::raw (&q)[16],
                                             const float (&c)[4], float* yo, int j) {
  constexpr int NBLK = P / 8;
  float part[16];
#pragma unroll
  for (int blk = 0; blk < NBLK; ++blk) {
    const int sl = (blk & 1) * 8;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int d = blk * 8 + r;
      float h[4];
      Quad<HT>::unpack(q[sl + r], h);
      part[sl + r] = Dot<N>::partial(c, h);
      if (blk + 2 < NBLK) q[sl + r] = Quad<HT>::ld_stream(Hsrc + (size_t)(d + 16) * N + 4 * j);
    }
    if (blk & 1) {
      const float v = reduce_scatter16(part, j);
      if ((j & 1) == 0) yo[(blk - 1) * 8 + (j >> 1)] = v;
    }
  }
  __syncwarp();
}

// The same stream for a step that fills the chunk: each row is also folded with the chunk state,
// H'[d] = exp(Acum_last) H[d] + sum_s (w_s x_s[d]) B_s (chunk_state / fold_state order; weights
// sw[s] in shared memory), and written to Hd and, if present, the bf16 copy Rd.  Rows go 8 at a
// time so that 32 independent accumulation chains hide the FMA latency.
template <typename T, int P, int N>
__device__ __noinline__ void stream_state_refresh(const float* __restrict__ Hsrc, const float (&c)[4], float* yo,
                                                  int j, int p, const float* sw, float decay, const T* sB,
                                                  const T* sx, float* Hd, __nv_bfloat16* Rd) {
#pragma unroll 1
  for (int d0 = 0; d0 < P; d0 += 16) {
    float part[16];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int db = d0 + 8 * half;
      float h[8][4], acc[8][4];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        Quad<float>::unpack(__ldcs(reinterpret_cast<const float4*>(Hsrc + (size_t)(db + r) * N + 4 * j)), h[r]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][e] = 0.f;
      }
      for (int s = 0; s <= p; ++s) {
        float bs[4];
        lds4(sB + s * N + 4 * j, bs);
        const float ws = sw[s];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float wx = __fmul_rn(ws, to_f(sx[s * P + db + r]));
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[r][e] = __fmaf_rn(wx, bs[e], acc[r][e]);
        }
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        part[8 * half + r] = Dot<N>::partial(c, h[r]);
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __fmaf_rn(decay, h[r][e], acc[r][e]);
        const size_t o = (size_t)(db + r) * N + 4 * j;
        *reinterpret_cast<float4*>(Hd + o) = make_float4(v[0], v[1], v[2], v[3]);
        if (Rd != nullptr) {
          __nv_bfloat162 lo2 = __floats2bfloat162_rn(v[0], v[1]), hi2 = __floats2bfloat162_rn(v[2], v[3]);
          uint2 u;
          u.x = *reinterpret_cast<uint32_t*>(&lo2);
          u.y = *reinterpret_cast<uint32_t*>(&hi2);
          *reinterpret_cast<uint2*>(Rd + o) = u;
        }
      }
    }
    const float v = reduce_scatter16(part, j);
    if ((j & 1) == 0) yo[d0 + (j >> 1)] = v;
  }
  __syncwarp();
}

template <typename T, typename HT, int P, int N, int QM>
__global__ void __launch_bounds__(kThreads, 2) k_decode_heads(LaunchArgs a) {
  static_assert(N == 128 && P % 32 == 0, "lane split of Dot<128>; 32-row reduction blocks");
  static_assert(QM <= 32, "one warp scans the chunk");
  extern __shared__ __align__(16) unsigned char hsm[];
  T* sB = reinterpret_cast<T*>(hsm);                                  // [QM][N] group B rows 0..p
  T* sxa = sB + QM * N;                                               // [warp][QM][P] x rows 0..p
  float* sg = reinterpret_cast<float*>(sxa + kHeadsPerCta * QM * P);  // [QM] Gram row
  float* syo = sg + QM;                                               // [warp][P] off-diagonal terms
  float* swa = syo + kHeadsPerCta * P;                                // [warp][QM] chunk-state weights
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
  const HT* Hsrc = rssm ? (const HT*)((const __nv_bfloat16*)a.read_copy + soff) : (const HT*)(a.state + soff);
  const int p = a.pos[slot];
  float c[4];
  load_k<T, 4>((const T*)a.C + (size_t)i * GN + (size_t)g * N + 4 * j, c);
  typename Quad<HT>::raw q[16];
  if (active) {
#pragma unroll
    for (int r = 0; r < 16; ++r) q[r] = Quad<HT>::ld_stream(Hsrc + (size_t)r * N + 4 * j);
  }
  if (p < 0 || p >= a.Q) {
    if (tid == 0) report(a.status, ERS_EALIGN);
    return;
  }
  const bool refresh = !rssm && (a.flags & ERS_FLAG_FUSE_REFRESH) && p + 1 == a.Q;
  // buffer rows 0..p-1 and the new token as row p: the group's B rows, this head's x rows
  const T* bB = (const T*)a.bB + (size_t)slot * a.Q * GN + (size_t)g * N;
  const T* nB = (const T*)a.B + (size_t)i * GN + (size_t)g * N;
  constexpr int kBChunks = N * sizeof(T) / 16, kXChunks = P * sizeof(T) / 16;
  for (int k = tid; k < (p + 1) * kBChunks; k += kThreads) {
    const int s = k / kBChunks, e = k % kBChunks;
    cp_async16(reinterpret_cast<char*>(sB + s * N) + 16 * e,
               reinterpret_cast<const char*>(s < p ? bB + s * GN : nB) + 16 * e);
  }
  T* sx = sxa + w * QM * P;
  const T* bx = (const T*)a.bx + (size_t)slot * a.Q * HP + (size_t)h * P;
  const T* nx = (const T*)a.x + (size_t)i * HP + (size_t)h * P;
  if (active)
    for (int k = j; k < (p + 1) * kXChunks; k += 32) {
      const int s = k / kXChunks, e = k % kXChunks;
      cp_async16(reinterpret_cast<char*>(sx + s * P) + 16 * e,
                 reinterpret_cast<const char*>(s < p ? bx + s * HP : nx) + 16 * e);
    }
  const float dt_raw = j <= p ? (j < p ? a.bdt[((size_t)slot * a.Q + j) * a.H + h] : a.dt[(size_t)i * a.H + h]) : 0.f;
  const float Ah = a.A[h], bias = a.dt_bias[h];
  float* yo = syo + w * P;
  if (!refresh && active)
    stream_state<HT, P, N>(Hsrc, q, c, yo, j);
  float dl = 0.f;
  df v = {0.f, 0.f};
  if (j <= p) {
    dl = delta_of(dt_raw, bias);
    v.hi = __fmul_rn(dl, Ah);
  }
  cp_async_wait_all();
  __syncthreads();
  // the group's Gram row, split over the warps
  for (int s = w; s <= p; s += kHeadsPerCta) {
    float bs[4];
    lds4(sB + s * N + 4 * j, bs);
    const float gv = Dot<N>::reduce(Dot<N>::partial(c, bs));
    if (j == 0) sg[s] = gv;
  }
  // this head's log-decay prefix (lane s holds row s)
#pragma unroll
  for (int st = 1; st < 32; st <<= 1) {
    const float ph = __shfl_up_sync(kFull, v.hi, st), pl = __shfl_up_sync(kFull, v.lo, st);
    if (j >= st) v = df_add(df{ph, pl}, v);
  }
  const df at = {__shfl_sync(kFull, v.hi, p), __shfl_sync(kFull, v.lo, p)};
  __syncthreads();
  if (!active) return;
  float M = 0.f;
  if (j <= p) M = __fmul_rn(__fmul_rn(sg[j], dl), expf(df_diff(at, v)));
  if (refresh) {
    float* sw = swa + w * QM;
    if (j <= p) sw[j] = __fmul_rn(dl, expf(df_diff(at, v)));
    __syncwarp();
    __nv_bfloat16* Rd = a.read_copy ? (__nv_bfloat16*)a.read_copy + soff : nullptr;
    stream_state_refresh<T, P, N>(a.state + soff, c, yo, j, p, sw, expf(at.hi), sB, sx, a.state + soff, Rd);
  }
  // outputs d = 32k + j
  const float et = expf(at.hi), Dh = a.D[h];
  T* y = (T*)a.y + (size_t)i * HP + (size_t)h * P;
#pragma unroll
  for (int k = 0; k < P / 32; ++k) {
    const int d = 32 * k + j;
    float acc = 0.f;
    for (int s = 0; s <= p; ++s) acc = __fmaf_rn(__shfl_sync(kFull, M, s), to_f(sx[s * P + d]), acc);
    y[d] = from_f<T>(combine_out(et, yo[d], acc, Dh, to_f(sx[p * P + d])));
  }
  // append the new token to the buffer (B/C once per group)
  T* dx = (T*)a.bx + ((size_t)slot * a.Q + p) * HP + (size_t)h * P;
  for (int d = j; d < P; d += 32) dx[d] = sx[p * P + d];
  if (j == 0) a.bdt[((size_t)slot * a.Q + p) * a.H + h] = a.dt[(size_t)i * a.H + h];
  if (hl == 0) {
    const size_t dst = ((size_t)slot * a.Q + p) * GN + (size_t)g * N, src = (size_t)i * GN + (size_t)g * N;
    for (int n = j; n < N; n += 32) {
      ((T*)a.bB)[dst + n] = sB[p * N + n];
      ((T*)a.bC)[dst + n] = ((const T*)a.C)[src + n];
    }
  }
}

template <typename T, int P, int N, int QM>
cudaError_t launch_decode_heads(const LaunchArgs& a, cudaStream_t s) {
  const int hpg = a.H / a.G, nbl = (hpg + kHeadsPerCta - 1) / kHeadsPerCta;
  const dim3 grid(a.G * nbl, a.nseq);
  constexpr size_t sm = heads_smem_bytes<T, P, N, QM>();
  cudaError_t e;
  if (a.flags & ERS_FLAG_REPLAYSSM) {
    if ((e = prep(k_decode_heads<T, __nv_bfloat16, P, N, QM>, sm)) != cudaSuccess) return e;
    k_decode_heads<T, __nv_bfloat16, P, N, QM><<<grid, kThreads, sm, s>>>(a);
  } else {
    if ((e = prep(k_decode_heads<T, float, P, N, QM>, sm)) != cudaSuccess) return e;
    k_decode_heads<T, float, P, N, QM><<<grid, kThreads, sm, s>>>(a);
  }
  return launch_setpos(a, 0, s);
}

// ---- refresh (exact: pos == Q; ReplaySSM: pos + T > L) ---------------------------------------------
template <typename T, int P, int N>
__global__ void __launch_bounds__(kThreads) k_refresh(LaunchArgs a) {
  const int i = blockIdx.x, h = blockIdx.y;
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const bool rssm = (a.flags & ERS_FLAG_REPLAYSSM) != 0;
  const int p = a.pos[slot];
  if (p < 0 || p > a.Q) {
    if (threadIdx.x == 0) report(a.status, ERS_EALIGN);
    return;
  }
  const bool go = rssm ? (p + a.T > a.Q) : (p == a.Q);
  if (!go) return;
  const size_t hs = (size_t)P * N;
  float* Hd = a.state + ((size_t)slot * a.H + h) * hs;
  __nv_bfloat16* Rd = a.read_copy ? (__nv_bfloat16*)a.read_copy + ((size_t)slot * a.H + h) * hs : nullptr;
  if (p == 0) {  // empty committed history: anchor unchanged, read copy recast from it
    if (Rd != nullptr)
      for (int idx = threadIdx.x; idx < P * N; idx += kThreads) Rd[idx] = __float2bfloat16_rn(Hd[idx]);
    return;
  }
  FmaSmem& sm = smem_hdr();
  float* xs = smem_xs();
  const Rows<T> rows = make_rows<T>(a, slot, h, p, 0);
  load_rows<T, P>(sm, xs, p, rows, a.A[h], a.dt_bias[h]);
  state_weights(sm, p);
  float S[P * N / kThreads];
  chunk_state<T, P, N>(sm, xs, p, S);
  fold_state<P, N>(Hd, Rd, expf(sm.hi[p - 1]), S);
}

// ---- speculative verify --------------------------------------------------------------------------
// Launch 1: slots whose committed pointer would overflow fold their committed records first.
template <typename T, int P, int N>
__global__ void __launch_bounds__(kThreads) k_verify_flush(LaunchArgs a) {
  const int i = blockIdx.x, h = blockIdx.y;
  int slot;
  if (!resolve_slot(a, i, &slot)) return;
  const int hc = a.pos[slot];
  if (hc < 0 || hc > a.Q) {
    if (threadIdx.x == 0) report(a.status, ERS_EALIGN);
    return;
  }
  if (hc + a.T <= a.Q) return;
  if (!(a.flags & ERS_FLAG_AUTO_FLUSH)) {
    if (threadIdx.x == 0) report(a.status, ERS_EOVERFLOW);
    return;
  }
  const size_t hs = (size_t)P * N;
  float* Hd = a.state + ((size_t)slot * a.H + h) * hs;
  __nv_bfloat16* Rd = (__nv_bfloat16*)a.read_copy + ((size_t)slot * a.H + h) * hs;
  FmaSmem& sm = smem_hdr();
  float* xs = smem_xs();
  const Rows<T> rows = make_rows<T>(a, slot, h, hc, 0);
  load_rows<T, P>(sm, xs, hc, rows, a.A[h], a.dt_bias[h]);
  state_weights(sm, hc);
  float S[P * N / kThreads];
  chunk_state<T, P, N>(sm, xs, hc, S);
  fold_state<P, N>(Hd, Rd, expf(sm.hi[hc - 1]), S);
}

// Launch 2: drafts go to buffer rows [h', h'+T); outputs for each draft from the read copy.
template <typename T, int P, int N>
__global__ void __launch_bounds__(kThreads) k_verify(LaunchArgs a) {
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
  FmaSmem& sm = smem_hdr();
  float* xs = smem_xs();
  // rows [0, h0) committed (buffer), rows [h0, h0+T) the drafts: input token i*T + (r - h0)
  const Rows<T> rows = make_rows<T>(a, slot, h, h0, (long long)i * a.T - h0);
  const int nrows = h0 + a.T;
  load_rows<T, P>(sm, xs, nrows, rows, a.A[h], a.dt_bias[h]);
  const size_t hs = (size_t)P * N;
  const __nv_bfloat16* Rd = (const __nv_bfloat16*)a.read_copy + ((size_t)slot * a.H + h) * hs;
  T* y = (T*)a.y;
  for (int j = 0; j < a.T; ++j)
    row_output<T, P, N, __nv_bfloat16>(sm, xs, h0 + j, Rd, a.D[h], y + (((size_t)i * a.T + j) * a.H + h) * P);
  // write the drafts into the buffer
  const int g = h / (a.H / a.G);
  for (int idx = threadIdx.x; idx < a.T * P; idx += kThreads) {
    const int j = idx / P, d = idx % P;
    ((T*)a.bx)[(((size_t)slot * a.Q + h0 + j) * a.H + h) * P + d] =
        ((const T*)a.x)[(((size_t)i * a.T + j) * a.H + h) * P + d];
  }
  for (int j = threadIdx.x; j < a.T; j += kThreads)
    a.bdt[((size_t)slot * a.Q + h0 + j) * a.H + h] = a.dt[((size_t)i * a.T + j) * a.H + h];
  if (h % (a.H / a.G) == 0) {
    for (int idx = threadIdx.x; idx < a.T * N; idx += kThreads) {
      const int j = idx / N, n = idx % N;
      const size_t dst = (((size_t)slot * a.Q + h0 + j) * a.G + g) * N + n;
      const size_t src = (((size_t)i * a.T + j) * a.G + g) * N + n;
      ((T*)a.bB)[dst] = ((const T*)a.B)[src];
      ((T*)a.bC)[dst] = ((const T*)a.C)[src];
    }
  }
}

// ---- pointer-only kernels ---------------------------------------------------------------------------
// Runs after the compute launch of the same call, so every head of a slot has read the old pos.
__global__ void k_setpos(LaunchArgs a, int kind) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.nseq) return;
  const int slot = a.slot != nullptr ? a.slot[i] : i;
  if (slot < 0 || slot >= a.nslots) return;
  const int p = a.pos[slot];
  const bool rssm = (a.flags & ERS_FLAG_REPLAYSSM) != 0;
  if (kind == 0) {  // after a decode step
    if (p < 0 || p >= a.Q) return;
    a.pos[slot] = (!rssm && (a.flags & ERS_FLAG_FUSE_REFRESH) && p + 1 == a.Q) ? 0 : p + 1;
  } else {  // after a refresh
    if (p < 0 || p > a.Q) return;
    const bool go = rssm ? (p + a.T > a.Q) : (p == a.Q);
    if (go) a.pos[slot] = 0;
  }
}

__global__ void k_commit(LaunchArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.nseq) return;
  const int slot = a.slot != nullptr ? a.slot[i] : i;
  if (slot < 0 || slot >= a.nslots) {
    report(a.status, ERS_ESLOT);
    return;
  }
  const int hc = a.pos[slot];
  const int acc = a.accepted[i];
  if (acc < 0 || acc > a.T) {
    report(a.status, ERS_ECOMMIT);
    return;
  }
  if (hc < 0 || hc > a.Q) {
    report(a.status, ERS_EALIGN);
    return;
  }
  const bool overflow = hc + a.T > a.Q;
  if (overflow && !(a.flags & ERS_FLAG_AUTO_FLUSH)) {
    report(a.status, ERS_EOVERFLOW);
    return;
  }
  a.pos[slot] = (overflow ? 0 : hc) + acc;
}

// Chunked prefill epilogue: the trailing partial chunk's inputs go to the buffer and pos advances.
template <typename T>
__global__ void k_tail(LaunchArgs a) {
  const int i = blockIdx.x;
  SeqGrid sg;
  if (!seq_grid(a, true, i, &sg)) return;
  const int nfull = sg.total / a.Q;
  const int rem = sg.total - nfull * a.Q;
  const int HP = a.H * a.P, GN = a.G * a.N;
  for (int r = 0; r < rem; ++r) {
    const int rs = nfull * a.Q + r;  // stream position
    if (rs < sg.p) continue;          // already buffered at row r (only when nfull == 0)
    const size_t tok = (size_t)a.cu[i] + (rs - sg.p);
    const size_t brow = (size_t)sg.slot * a.Q + r;
    for (int k = threadIdx.x; k < HP; k += blockDim.x) ((T*)a.bx)[brow * HP + k] = ((const T*)a.x)[tok * HP + k];
    for (int k = threadIdx.x; k < a.H; k += blockDim.x) a.bdt[brow * a.H + k] = a.dt[tok * a.H + k];
    for (int k = threadIdx.x; k < GN; k += blockDim.x) {
      ((T*)a.bB)[brow * GN + k] = ((const T*)a.B)[tok * GN + k];
      ((T*)a.bC)[brow * GN + k] = ((const T*)a.C)[tok * GN + k];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) a.pos[sg.slot] = rem;
}

// ---- host dispatch -------------------------------------------------------------------------------

template <typename T, int P, int N>
cudaError_t prefill_impl(const LaunchArgs& a, Op op, cudaStream_t s) {
  const bool chunked = op == Op::kChunkedPrefill;
  const size_t sm = fma_smem_bytes(a.Q, P);
  cudaError_t e;
  if ((e = prep(k_prefill_state<T, P, N>, sm)) != cudaSuccess) return e;
  if ((e = prep(k_prefill_out<T, P, N>, sm)) != cudaSuccess) return e;
  if (a.max_chunks > 0 && a.nseq > 0) {
    dim3 grid(a.max_chunks, a.nseq, a.H);
    k_prefill_state<T, P, N><<<grid, kThreads, sm, s>>>(a, chunked);
    k_prefill_chain<P, N><<<dim3(a.nseq, a.H), kThreads, 0, s>>>(a, chunked);
    k_prefill_out<T, P, N><<<grid, kThreads, sm, s>>>(a, chunked);
  }
  if (chunked && a.nseq > 0) k_tail<T><<<a.nseq, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int P, int N>
cudaError_t decode_impl(const LaunchArgs& a, cudaStream_t s) {
  if constexpr (N == 128 && P % 32 == 0) {
    if (a.Q <= 16) return launch_decode_heads<T, P, N, 16>(a, s);
    if (a.Q <= 32) return launch_decode_heads<T, P, N, 32>(a, s);
  }
  const size_t sm = fma_smem_bytes(a.Q, P);
  cudaError_t e = prep(k_decode<T, P, N>, sm);
  if (e != cudaSuccess) return e;
  k_decode<T, P, N><<<dim3(a.nseq, a.H), kThreads, sm, s>>>(a);
  return launch_setpos(a, 0, s);
}

template <typename T, int P, int N>
cudaError_t refresh_impl(const LaunchArgs& a, cudaStream_t s) {
  const size_t sm = fma_smem_bytes(a.Q, P);
  cudaError_t e = prep(k_refresh<T, P, N>, sm);
  if (e != cudaSuccess) return e;
  k_refresh<T, P, N><<<dim3(a.nseq, a.H), kThreads, sm, s>>>(a);
  return launch_setpos(a, 1, s);
}

template <typename T, int P, int N>
cudaError_t verify_impl(const LaunchArgs& a, cudaStream_t s) {
  const size_t sm = fma_smem_bytes(a.Q, P);
  cudaError_t e;
  if ((e = prep(k_verify_flush<T, P, N>, sm)) != cudaSuccess) return e;
  if ((e = prep(k_verify<T, P, N>, sm)) != cudaSuccess) return e;
  k_verify_flush<T, P, N><<<dim3(a.nseq, a.H), kThreads, sm, s>>>(a);
  k_verify<T, P, N><<<dim3(a.nseq, a.H), kThreads, sm, s>>>(a);
  return cudaGetLastError();
}

// Supported (P, N) pairs of this engine.
#define ERS_FMA_SHAPES(X) X(16, 16) X(32, 32) X(64, 64) X(64, 128)

#define ERS_DISPATCH()                                                                               \
  do {                                                                                               \
    if (a.io == ERS_DTYPE_BF16) {                                                                    \
      ERS_FMA_SHAPES(ERS_CASE_BF16)                                                                  \
    } else {                                                                                         \
      ERS_FMA_SHAPES(ERS_CASE_F32)                                                                   \
    }                                                                                                \
    return cudaErrorInvalidValue;                                                                    \
  } while (0)

}  // namespace

bool fma_supported(int P, int N) {
#define ERS_SUP(p_, n_) if (P == p_ && N == n_) return true;
  ERS_FMA_SHAPES(ERS_SUP)
#undef ERS_SUP
  return false;
}

#define ERS_CASE_BF16(p_, n_) if (a.P == p_ && a.N == n_) return IMPL<__nv_bfloat16, p_, n_>(ERS_ARGS);
#define ERS_CASE_F32(p_, n_) if (a.P == p_ && a.N == n_) return IMPL<float, p_, n_>(ERS_ARGS);

cudaError_t fma_prefill(const LaunchArgs& a, Op op, cudaStream_t s) {
#define IMPL prefill_impl
#define ERS_ARGS a, op, s
  ERS_DISPATCH();
#undef IMPL
#undef ERS_ARGS
}

cudaError_t fma_decode(const LaunchArgs& a, cudaStream_t s) {
#define IMPL decode_impl
#define ERS_ARGS a, s
  ERS_DISPATCH();
#undef IMPL
#undef ERS_ARGS
}

cudaError_t fma_refresh(const LaunchArgs& a, cudaStream_t s) {
#define IMPL refresh_impl
#define ERS_ARGS a, s
  ERS_DISPATCH();
#undef IMPL
#undef ERS_ARGS
}

cudaError_t fma_verify(const LaunchArgs& a, cudaStream_t s) {
#define IMPL verify_impl
#define ERS_ARGS a, s
  ERS_DISPATCH();
#undef IMPL
#undef ERS_ARGS
}

cudaError_t launch_setpos(const LaunchArgs& a, int kind, cudaStream_t s) {
  if (a.nseq > 0) k_setpos<<<(a.nseq + 255) / 256, 256, 0, s>>>(a, kind);
  return cudaGetLastError();
}

cudaError_t launch_commit(const LaunchArgs& a, cudaStream_t s) {
  if (a.nseq > 0) k_commit<<<(a.nseq + 255) / 256, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_chain(const LaunchArgs& a, bool chunked, cudaStream_t s) {
  if (a.nseq <= 0 || a.max_chunks <= 0) return cudaSuccess;
#define ERS_CH(p_, n_) if (a.P == p_ && a.N == n_) { k_prefill_chain<p_, n_><<<dim3(a.nseq, a.H), kThreads, 0, s>>>(a, chunked); return cudaGetLastError(); }
  ERS_FMA_SHAPES(ERS_CH)
#undef ERS_CH
  return cudaErrorInvalidValue;
}

cudaError_t launch_tail(const LaunchArgs& a, cudaStream_t s) {
  if (a.nseq <= 0) return cudaSuccess;
  if (a.io == ERS_DTYPE_BF16)
    k_tail<__nv_bfloat16><<<a.nseq, kThreads, 0, s>>>(a);
  else
    k_tail<float><<<a.nseq, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ers
