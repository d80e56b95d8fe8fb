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
// H_{c+1} = fma(exp(Acum_last,c), H_c, S_c) is elementwise, so each (sequence, head) state is split
// over kChainSlices CTAs of kThreads threads x 4 consecutive elements (one 16-byte access each).
// The chunk states and log-decays are inputs of the chain, not results of it, so a thread loads
// them for kChainBatch chunks at once and only the fma chain itself runs in chunk order.
constexpr int kChainElems = 4;
constexpr int kChainBatch = 8;

__host__ __device__ constexpr int chain_slices(int P, int N) {
  return (P * N + kThreads * kChainElems - 1) / (kThreads * kChainElems);
}

template <int P, int N>
__global__ void __launch_bounds__(kThreads) k_prefill_chain(LaunchArgs a, bool chunked) {
  static_assert((P * N) % kChainElems == 0, "whole 16-byte groups");
  const int i = blockIdx.x, h = blockIdx.y;
  SeqGrid sg;
  if (!seq_grid(a, chunked, i, &sg)) return;
  const int idx = (blockIdx.z * kThreads + threadIdx.x) * kChainElems;
  if (idx >= P * N) return;
  const size_t hs = (size_t)P * N;
  float* ckpt = chunked ? a.state + ((size_t)sg.slot * a.H + h) * hs : nullptr;
  const float* init = chunked ? ckpt : (a.init_state ? a.init_state + ((size_t)i * a.H + h) * hs : nullptr);
  float Hr[kChainElems], keep[kChainElems];
  if (init != nullptr) {
    const float4 v = *reinterpret_cast<const float4*>(init + idx);
    Hr[0] = v.x; Hr[1] = v.y; Hr[2] = v.z; Hr[3] = v.w;
  } else {
#pragma unroll
    for (int e = 0; e < kChainElems; ++e) Hr[e] = 0.f;
  }
#pragma unroll
  for (int e = 0; e < kChainElems; ++e) keep[e] = Hr[e];
  const bool aligned_end = (sg.total % a.Q) == 0;
  for (int c0 = 0; c0 < sg.nch; c0 += kChainBatch) {
    float4 sv[kChainBatch];
    float tot[kChainBatch];
#pragma unroll
    for (int k = 0; k < kChainBatch; ++k) {
      if (c0 + k < sg.nch) {
        const size_t base = ((size_t)i * a.max_chunks + c0 + k) * a.H + h;
        sv[k] = *reinterpret_cast<const float4*>(a.ws_states + base * hs + idx);
        tot[k] = a.ws_tot[base];
      }
    }
#pragma unroll
    for (int k = 0; k < kChainBatch; ++k) {
      const int c = c0 + k;
      if (c >= sg.nch) break;
      const size_t base = ((size_t)i * a.max_chunks + c) * a.H + h;
      const float decay = expf(tot[k]);
      if (c == sg.nch - 1 && !aligned_end) {
#pragma unroll
        for (int e = 0; e < kChainElems; ++e) keep[e] = Hr[e];
      }
      const float sc[kChainElems] = {sv[k].x, sv[k].y, sv[k].z, sv[k].w};
      // the state at the start of chunk c, read by the output kernel (each thread overwrites the
      // 16 bytes it read above)
      *reinterpret_cast<float4*>(a.ws_states + base * hs + idx) = make_float4(Hr[0], Hr[1], Hr[2], Hr[3]);
#pragma unroll
      for (int e = 0; e < kChainElems; ++e) Hr[e] = __fmaf_rn(decay, Hr[e], sc[e]);
      if (a.chunk_states != nullptr)
        *reinterpret_cast<float4*>(a.chunk_states + base * hs + idx) = make_float4(Hr[0], Hr[1], Hr[2], Hr[3]);
    }
  }
  if (!chunked) {
    *reinterpret_cast<float4*>(a.final_state + ((size_t)i * a.H + h) * hs + idx) = make_float4(Hr[0], Hr[1], Hr[2], Hr[3]);
  } else if (sg.nch > 0) {
    const float* v = aligned_end ? Hr : keep;
    *reinterpret_cast<float4*>(ckpt + idx) = make_float4(v[0], v[1], v[2], v[3]);
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
  T* bx = (T*)a.bx + (buf_row(a, slot, p) * a.H + h) * P;
  const T* nx = (const T*)a.x + ((size_t)i * a.H + h) * P;
  for (int d = threadIdx.x; d < P; d += kThreads) bx[d] = nx[d];
  if (threadIdx.x == 0) a.bdt[buf_row(a, slot, p) * a.H + h] = a.dt[(size_t)i * a.H + h];
  if (h % (a.H / a.G) == 0) {
    T* bB = (T*)a.bB + (buf_row(a, slot, p) * a.G + g) * N;
    T* bC = (T*)a.bC + (buf_row(a, slot, p) * a.G + g) * N;
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
    ((T*)a.bx)[(buf_row(a, slot, h0 + j) * a.H + h) * P + d] =
        ((const T*)a.x)[(((size_t)i * a.T + j) * a.H + h) * P + d];
  }
  for (int j = threadIdx.x; j < a.T; j += kThreads)
    a.bdt[buf_row(a, slot, h0 + j) * a.H + h] = a.dt[((size_t)i * a.T + j) * a.H + h];
  if (h % (a.H / a.G) == 0) {
    for (int idx = threadIdx.x; idx < a.T * N; idx += kThreads) {
      const int j = idx / N, n = idx % N;
      const size_t dst = (buf_row(a, slot, h0 + j) * a.G + g) * N + n;
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
    const size_t brow = buf_row(a, sg.slot, r);
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
    k_prefill_chain<P, N><<<dim3(a.nseq, a.H, chain_slices(P, N)), kThreads, 0, s>>>(a, chunked);
    k_prefill_out<T, P, N><<<grid, kThreads, sm, s>>>(a, chunked);
  }
  if (chunked && a.nseq > 0) k_tail<T><<<a.nseq, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int P, int N>
cudaError_t decode_impl(const LaunchArgs& a, cudaStream_t s) {
  if (heads_decode_supported(a.P, a.N, a.Q)) return heads_decode(a, s);
  const size_t sm = fma_smem_bytes(a.Q, P);
  cudaError_t e = prep(k_decode<T, P, N>, sm);
  if (e != cudaSuccess) return e;
  k_decode<T, P, N><<<dim3(a.nseq, a.H), kThreads, sm, s>>>(a);
  return launch_setpos(a, 0, s);
}

template <typename T, int P, int N>
cudaError_t refresh_impl(const LaunchArgs& a, cudaStream_t s) {
  cudaError_t e;
  if (heads_decode_supported(a.P, a.N, a.Q)) {   // warp-per-head kernel (bf16 / FP8 / NVFP4 copies)
    if ((e = heads_refresh(a, s)) != cudaSuccess) return e;
    return launch_setpos(a, 1, s);
  }
  const size_t sm = fma_smem_bytes(a.Q, P);
  if ((e = prep(k_refresh<T, P, N>, sm)) != cudaSuccess) return e;
  k_refresh<T, P, N><<<dim3(a.nseq, a.H), kThreads, sm, s>>>(a);
  return launch_setpos(a, 1, s);
}

template <typename T, int P, int N>
cudaError_t verify_impl(const LaunchArgs& a, cudaStream_t s) {
  if (heads_verify_supported(a.P, a.N, a.Q, a.T, a.H, a.G)) return heads_verify(a, s);
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

// ---- exact-mode speculative decode: shadow copies and draft rows ------------------------------
// Copies a row of `n` io elements; bf16 and fp32 rows are moved as 16-bit / 32-bit words.
__device__ __forceinline__ void copy_elems(void* dst, const void* src, int n, int es, int lane, int nl) {
  if (es == 2) {
    for (int k = lane; k < n; k += nl) ((uint16_t*)dst)[k] = ((const uint16_t*)src)[k];
  } else {
    for (int k = lane; k < n; k += nl) ((uint32_t*)dst)[k] = ((const uint32_t*)src)[k];
  }
}

// Draft rows j0 .. j0+n-1 of sequence i (token rows i T + j of x, B, C; dt as floats) into buffer rows
// r0 .. r0+n-1 of its slot.  The x, B and C rows move as 16-byte words (their sizes are multiples of
// 16 bytes: P = 64 or N = 128 io elements per head or group), each thread loading all of its words
// before storing any, so that a CTA's copies overlap instead of waiting one round trip each; dt
// (H floats a row) moves as floats.
__device__ __forceinline__ void copy_draft_rows(const LaunchArgs& a, int i, int slot, int j0, int n, int r0) {
  const int es = a.io == ERS_DTYPE_BF16 ? 2 : 4;
  const long long HP = (long long)a.H * a.P, GN = (long long)a.G * a.N;
  const int xw = (int)(HP * es / 16), gw = (int)(GN * es / 16), per = xw + 2 * gw, W = n * per;
  constexpr int kBatch = 8;
  for (int base = threadIdx.x; base < W; base += kBatch * blockDim.x) {
    uint4 v[kBatch];
    uint4* dst[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int wi = base + u * blockDim.x;
      dst[u] = nullptr;
      if (wi < W) {
        const int r = wi / per, o = wi % per;
        const long long tok = (long long)i * a.T + j0 + r, br = buf_row(a, slot, r0 + r);
        const uint4* src;
        if (o < xw) {
          src = (const uint4*)((const char*)a.x + tok * HP * es) + o;
          dst[u] = (uint4*)((char*)a.bx + br * HP * es) + o;
        } else if (o < xw + gw) {
          src = (const uint4*)((const char*)a.B + tok * GN * es) + (o - xw);
          dst[u] = (uint4*)((char*)a.bB + br * GN * es) + (o - xw);
        } else {
          src = (const uint4*)((const char*)a.C + tok * GN * es) + (o - xw - gw);
          dst[u] = (uint4*)((char*)a.bC + br * GN * es) + (o - xw - gw);
        }
        v[u] = __ldg(src);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (dst[u] != nullptr) *dst[u] = v[u];
  }
  for (int e = threadIdx.x; e < n * a.H; e += blockDim.x) {
    const int r = e / a.H, k = e % a.H;
    a.bdt[buf_row(a, slot, r0 + r) * a.H + k] = a.dt[((long long)i * a.T + j0 + r) * a.H + k];
  }
}

// Shadow of sequence i's slot (blockIdx.y = i, blockIdx.x = head): its fp32 checkpoint head, its
// buffered rows [0, pos) (x, dt of the head; B, C of group h when h < G) in the contiguous layout,
// its position.  `a` describes the real cache; sh_* the shadow (slot i, Q rows per slot).
__global__ void k_spec_snapshot(LaunchArgs a, float* sh_state, void* sh_bx, float* sh_bdt, void* sh_bB, void* sh_bC,
                                int32_t* sh_pos) {
  const int i = blockIdx.y, h = blockIdx.x;
  const int slot = a.slot != nullptr ? a.slot[i] : i;
  if (slot < 0 || slot >= a.nslots) {
    if (threadIdx.x == 0 && h == 0) {
      report(a.status, ERS_ESLOT);
      sh_pos[i] = -1;   // the shadow decode reports it again and touches nothing
    }
    return;
  }
  const int p = a.pos[slot];
  if (p < 0 || p >= a.Q) {
    if (threadIdx.x == 0 && h == 0) {
      report(a.status, ERS_EALIGN);
      sh_pos[i] = -1;
    }
    return;
  }
  const size_t hs = (size_t)a.P * a.N;
  const float4* src = reinterpret_cast<const float4*>(a.state + ((size_t)slot * a.H + h) * hs);
  float4* dst = reinterpret_cast<float4*>(sh_state + ((size_t)i * a.H + h) * hs);
  for (size_t k = threadIdx.x; k < hs / 4; k += blockDim.x) dst[k] = src[k];
  const int es = a.io == ERS_DTYPE_BF16 ? 2 : 4;
  const long long HP = (long long)a.H * a.P, GN = (long long)a.G * a.N;
  for (int r = 0; r < p; ++r) {
    const long long br = buf_row(a, slot, r), sr = (long long)i * a.Q + r;
    copy_elems((char*)sh_bx + (sr * HP + (long long)h * a.P) * es, (const char*)a.bx + (br * HP + (long long)h * a.P) * es,
               a.P, es, threadIdx.x, blockDim.x);
    if (threadIdx.x == 0) sh_bdt[sr * a.H + h] = a.bdt[br * a.H + h];
    if (h < a.G) {
      copy_elems((char*)sh_bB + (sr * GN + (long long)h * a.N) * es, (const char*)a.bB + (br * GN + (long long)h * a.N) * es,
                 a.N, es, threadIdx.x, blockDim.x);
      copy_elems((char*)sh_bC + (sr * GN + (long long)h * a.N) * es, (const char*)a.bC + (br * GN + (long long)h * a.N) * es,
                 a.N, es, threadIdx.x, blockDim.x);
    }
  }
  if (threadIdx.x == 0 && h == 0) sh_pos[i] = p;
}

// Draft j of every sequence into contiguous one-token inputs (dir = 0), or a one-token output back
// into draft j's output row (dir = 1).  blockIdx.x = sequence.
__global__ void k_spec_draft_rows(LaunchArgs a, int j, int dir, const void* x, const float* dt, const void* B,
                                  const void* C, void* x1, float* dt1, void* B1, void* C1, void* y, const void* y1) {
  const int i = blockIdx.x;
  const int es = a.io == ERS_DTYPE_BF16 ? 2 : 4;
  const long long HP = (long long)a.H * a.P, GN = (long long)a.G * a.N;
  const long long row = (long long)i * a.T + j;
  if (dir == 0) {
    copy_elems((char*)x1 + i * HP * es, (const char*)x + row * HP * es, (int)HP, es, threadIdx.x, blockDim.x);
    for (int k = threadIdx.x; k < a.H; k += blockDim.x) dt1[(long long)i * a.H + k] = dt[row * a.H + k];
    copy_elems((char*)B1 + i * GN * es, (const char*)B + row * GN * es, (int)GN, es, threadIdx.x, blockDim.x);
    copy_elems((char*)C1 + i * GN * es, (const char*)C + row * GN * es, (int)GN, es, threadIdx.x, blockDim.x);
  } else {
    copy_elems((char*)y + row * HP * es, (const char*)y1 + i * HP * es, (int)HP, es, threadIdx.x, blockDim.x);
  }
}

// Commit, part 1: sequence i (blockIdx.x) appends its accepted drafts [0, a) that fit the chunk
// to buffer rows [p, min(Q, p + a)) and keeps p in `old_pos`; a chunk that fills is marked for the
// refresh with pos = Q, otherwise pos = p + a.
__global__ void k_commit_exact_fill(LaunchArgs a, int32_t* old_pos) {
  const int i = blockIdx.x;
  const int slot = a.slot != nullptr ? a.slot[i] : i;
  old_pos[i] = -1;
  if (slot < 0 || slot >= a.nslots) {
    if (threadIdx.x == 0) report(a.status, ERS_ESLOT);
    return;
  }
  const int p = a.pos[slot], acc = a.accepted[i];
  if (p < 0 || p >= a.Q) {
    if (threadIdx.x == 0) report(a.status, ERS_EALIGN);
    return;
  }
  if (acc < 0 || acc > a.T) {
    if (threadIdx.x == 0) report(a.status, ERS_ECOMMIT);
    return;
  }
  const int end = p + acc < a.Q ? p + acc : a.Q;
  copy_draft_rows(a, i, slot, 0, end - p, p);   // drafts 0 .. end-p-1 into rows p .. end-1
  __syncthreads();
  if (threadIdx.x == 0) {
    old_pos[i] = p;
    a.pos[slot] = p + acc >= a.Q ? a.Q : p + acc;
  }
}

// Commit, part 3 (after the refresh of the filled chunks): the accepted drafts past the chunk
// boundary become buffer rows [0, p + a - Q) and pos = p + a - Q.
__global__ void k_commit_exact_tail(LaunchArgs a, const int32_t* old_pos) {
  const int i = blockIdx.x;
  const int p = old_pos[i];
  if (p < 0) return;
  const int slot = a.slot != nullptr ? a.slot[i] : i;
  const int acc = a.accepted[i];
  if (p + acc < a.Q) return;
  const int n2 = p + acc - a.Q;
  copy_draft_rows(a, i, slot, a.Q - p, n2, 0);   // drafts Q-p .. into rows 0 .. n2-1
  __syncthreads();
  if (threadIdx.x == 0) a.pos[slot] = n2;
}

cudaError_t launch_spec_snapshot(const LaunchArgs& a, float* st, void* bx, float* bdt, void* bB, void* bC, int32_t* pos,
                                 cudaStream_t s) {
  if (a.nseq > 0) k_spec_snapshot<<<dim3(a.H, a.nseq), kThreads, 0, s>>>(a, st, bx, bdt, bB, bC, pos);
  return cudaGetLastError();
}

cudaError_t launch_spec_rows(const LaunchArgs& a, int j, int dir, const void* x, const float* dt, const void* B,
                             const void* C, void* x1, float* dt1, void* B1, void* C1, void* y, const void* y1,
                             cudaStream_t s) {
  if (a.nseq > 0) k_spec_draft_rows<<<a.nseq, kThreads, 0, s>>>(a, j, dir, x, dt, B, C, x1, dt1, B1, C1, y, y1);
  return cudaGetLastError();
}

cudaError_t launch_commit_exact(const LaunchArgs& a, int part, int32_t* old_pos, cudaStream_t s) {
  if (a.nseq <= 0) return cudaSuccess;
  if (part == 0) k_commit_exact_fill<<<a.nseq, kThreads, 0, s>>>(a, old_pos);
  else k_commit_exact_tail<<<a.nseq, kThreads, 0, s>>>(a, old_pos);
  return cudaGetLastError();
}

cudaError_t launch_setpos(const LaunchArgs& a, int kind, cudaStream_t s) {
  if (a.nseq > 0) k_setpos<<<(a.nseq + 255) / 256, 256, 0, s>>>(a, kind);
  return cudaGetLastError();
}

cudaError_t launch_commit(const LaunchArgs& a, cudaStream_t s) {
  if (a.nseq > 0) k_commit<<<(a.nseq + 255) / 256, 256, 0, s>>>(a);
  return cudaGetLastError();
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
