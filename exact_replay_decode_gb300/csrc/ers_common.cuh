// Device helpers shared by every kernel of the library.
//
// Bitwise identity across prefill, chunked prefill, replay decode, refresh and
// speculative verify (exact-replay RFC, vLLM issue 55524, section 3) rests on
// every path evaluating each output element and each chunk state with the SAME
// sequence of fp32 operations.  Everything that feeds an output or a state is
// therefore written once, here or in the engine headers, with explicit
// round-to-nearest intrinsics (__fadd_rn / __fmul_rn / __fmaf_rn) so the
// compiler can neither contract nor reorder it, and with reduction orders fixed
// by element index rather than by thread count.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ers.h"
#include "ers_internal.h"

namespace ers {

constexpr int kQMax = 256;       // largest chunk / refresh period supported
constexpr int kThreads = 256;    // block size of every engine kernel
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void report(int32_t* st, int32_t code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

// ---- io element conversions ---------------------------------------------------------------
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// ---- dt -> delta ------------------------------------------------------------------------------
// delta = softplus(dt_raw + dt_bias) (RFC section 3: the buffers keep the raw dt and the kernels
// apply softplus with the bias).  Above 20 softplus(z) equals z to within fp32 rounding, so the
// argument passes through.
__device__ __forceinline__ float delta_of(float dt_raw, float bias) {
  const float z = __fadd_rn(dt_raw, bias);
  return z > 20.f ? z : log1pf(expf(z));
}

// ---- double-float prefix sums of log-decays -------------------------------------------------
// A chunk's cumulative log-decay can reach a few hundred while the segment sums that matter are
// O(1); keeping the prefix as an unevaluated pair (hi, lo) makes Acum_t - Acum_s accurate to a few
// ulp of the SEGMENT, not of the prefix.
struct df {
  float hi, lo;
};

__device__ __forceinline__ df df_add(df a, df b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bb = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));  // TwoSum error
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  const float h = __fadd_rn(s, e);  // Fast2Sum renormalisation
  const float l = __fsub_rn(e, __fsub_rn(h, s));
  return {h, l};
}

// (a - b) for two prefix pairs, rounded once at the end.
__device__ __forceinline__ float df_diff(df a, df b) {
  return __fadd_rn(__fsub_rn(a.hi, b.hi), __fsub_rn(a.lo, b.lo));
}

// Inclusive prefix scan of rows [0, nrows) of (hi, lo) in shared memory, Kogge-Stone with
// strides 1, 2, 4, ... < kQMax.  Row t's result depends only on rows <= t and is computed by the
// same operations whatever nrows is, so a chunk scanned with later rows present (prefill) and the
// same chunk scanned with only rows 0..t present (decode) agree bit for bit.  Rows >= nrows must
// hold (0, 0).  Must be called by all kThreads threads.
__device__ __forceinline__ void chunk_scan(float* hi, float* lo) {
  const int t = threadIdx.x;
#pragma unroll 1
  for (int stride = 1; stride < kQMax; stride <<= 1) {
    df v = {0.f, 0.f};
    if (t < kQMax) {
      v = df{hi[t], lo[t]};
      if (t >= stride) v = df_add(df{hi[t - stride], lo[t - stride]}, v);
    }
    __syncthreads();
    if (t < kQMax) {
      hi[t] = v.hi;
      lo[t] = v.lo;
    }
    __syncthreads();
  }
}

// ---- fixed-order dot products over dstate ------------------------------------------------------
// A length-N dot product is computed by a group of W = min(32, N) consecutive lanes: lane j of the
// group accumulates elements [j*K, j*K+K) (K = N/W) in index order with fmaf starting from 0, then
// the group combines its lanes with a butterfly (xor W/2, ..., 1).  Every lane of the group ends
// with the same value, and the value does not depend on which warp or which group computes it.
template <int N>
struct Dot {
  static constexpr int W = N < 32 ? N : 32;
  static constexpr int K = N / W;
  static_assert(N % W == 0, "dstate must be a multiple of the group width");

  __device__ __forceinline__ static float reduce(float acc) {
#pragma unroll
    for (int off = W / 2; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, off));
    return acc;
  }
  __device__ __forceinline__ static float partial(const float (&a)[K], const float (&b)[K]) {
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) acc = __fmaf_rn(a[k], b[k], acc);
    return acc;
  }
};

template <typename T, int K>
__device__ __forceinline__ void load_k(const T* __restrict__ p, float (&v)[K]) {
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = to_f(p[k]);
}

// Output combine for one element: y = fma(D, x, exp(Acum_t) * Y_off + Y_diag), one rounding to
// the io dtype at the end.
__device__ __forceinline__ float combine_out(float decay_t, float yoff, float ydiag, float Dh, float xt) {
  return __fmaf_rn(Dh, xt, __fadd_rn(__fmul_rn(decay_t, yoff), ydiag));
}

// Buffer row of row r (0 <= r < Q) of a slot's partial-chunk buffer: slot * Q + r when the buffers are
// contiguous, else the page table's page for r.  A page index outside [0, npages) is reported
// (ERS_ESLOT) and clamped, so a bad table cannot address outside the buffers.
struct BufMap {
  const int32_t* pages;
  int Q, pr, npages;
  int32_t* status;
  __device__ __forceinline__ long long row(int slot, int r) const {
    if (pages == nullptr) return (long long)slot * Q + r;
    int pg = pages[(long long)slot * (Q / pr) + r / pr];
    if (pg < 0 || pg >= npages) {
      report(status, ERS_ESLOT);
      pg = pg < 0 ? 0 : npages - 1;
    }
    return (long long)pg * pr + r % pr;
  }
};

__device__ __forceinline__ BufMap buf_map(const LaunchArgs& a) {
  return BufMap{a.buf_pages, a.Q, a.page_rows, a.npages, a.status};
}

__device__ __forceinline__ long long buf_row(const LaunchArgs& a, int slot, int r) { return buf_map(a).row(slot, r); }

// Row source of a chunk: rows [0, nbuf) come from a slot's partial-chunk buffer, rows >= nbuf from
// packed token inputs (row r is token tok0 + r).  Row strides are the token strides H*P, H, G*N.
template <typename T>
struct Rows {
  int nbuf, slot;
  BufMap map;
  const T* bx;
  const float* bdt;
  const T* bB;
  const T* bC;
  const T* x0;
  const float* dt0;
  const T* B0;
  const T* C0;
  long long tok0;
  int sx, sdt, sB;
  __device__ __forceinline__ const T* x(int r) const {
    return r < nbuf ? bx + map.row(slot, r) * sx : x0 + (tok0 + r) * sx;
  }
  __device__ __forceinline__ float dt(int r) const {
    return r < nbuf ? bdt[map.row(slot, r) * sdt] : dt0[(tok0 + r) * sdt];
  }
  __device__ __forceinline__ const T* B(int r) const {
    return r < nbuf ? bB + map.row(slot, r) * sB : B0 + (tok0 + r) * sB;
  }
  __device__ __forceinline__ const T* C(int r) const {
    return r < nbuf ? bC + map.row(slot, r) * sB : C0 + (tok0 + r) * sB;
  }
};

template <typename T>
__device__ __forceinline__ Rows<T> make_rows(const LaunchArgs& a, int slot, int h, int nbuf, long long tok0) {
  const int g = h / (a.H / a.G);
  Rows<T> r;
  r.nbuf = nbuf;
  r.slot = slot;
  r.map = buf_map(a);
  r.sx = a.H * a.P;
  r.sdt = a.H;
  r.sB = a.G * a.N;
  if (slot >= 0 && a.bx != nullptr) {
    r.bx = (const T*)a.bx + (size_t)h * a.P;
    r.bdt = a.bdt + h;
    r.bB = (const T*)a.bB + (size_t)g * a.N;
    r.bC = (const T*)a.bC + (size_t)g * a.N;
  } else {
    r.bx = nullptr; r.bdt = nullptr; r.bB = nullptr; r.bC = nullptr;
  }
  r.x0 = (const T*)a.x + (size_t)h * a.P;
  r.dt0 = a.dt + h;
  r.B0 = (const T*)a.B + (size_t)g * a.N;
  r.C0 = (const T*)a.C + (size_t)g * a.N;
  r.tok0 = tok0;
  return r;
}

__device__ __forceinline__ bool resolve_slot(const LaunchArgs& a, int i, int* slot) {
  const int s = a.slot != nullptr ? a.slot[i] : i;
  if (s < 0 || s >= a.nslots) {
    if (threadIdx.x == 0) report(a.status, ERS_ESLOT);
    return false;
  }
  *slot = s;
  return true;
}

// Boundary-anchored chunk grid of sequence i: buffered p rows then the new tokens.
struct SeqGrid {
  int slot, p, len, total, nch;
};

__device__ __forceinline__ bool seq_grid(const LaunchArgs& a, bool chunked, int i, SeqGrid* g) {
  g->slot = -1;
  g->p = 0;
  if (chunked) {
    if (!resolve_slot(a, i, &g->slot)) return false;
    g->p = a.pos[g->slot];
    if (g->p < 0 || g->p >= a.Q) {
      if (threadIdx.x == 0) report(a.status, ERS_EALIGN);
      return false;
    }
  }
  g->len = a.cu[i + 1] - a.cu[i];
  g->total = g->p + g->len;
  g->nch = (g->total + a.Q - 1) / a.Q;
  return true;
}

}  // namespace ers
