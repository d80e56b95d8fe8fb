// Causal depthwise conv1d with a conv state: the step upstream of the SSM in a Mamba2 layer, whose
// prefill and decode-update paths must agree bit for bit (exact-replay RFC, §2 Evidence item 6; the
// bf16 operands are promoted to fp32 before accumulation, as the RFC's referenced fix does).
//
// Per channel c, with u the sequence's inputs preceded by its W - 1 earlier inputs (the conv state,
// oldest first):
//     y[t, c] = act(fma(w[c][W-1], u[t+W-1], ... fma(w[c][1], u[t+1], fma(w[c][0], u[t], bias[c]))))
// i.e. the bias first, then the taps from the oldest input to the newest, each one fmaf; act is SiLU
// a / (1 + exp(-a)) (IEEE division) or the identity.  Both kernels evaluate exactly this, so a
// prefill, a prefill resumed from a conv state, and token-by-token updates give the same bits.
//
// Both kernels are HBM-bound streams: a thread owns 8 adjacent channels (one 16-byte access per token
// for bf16, two for fp32, so a warp moves 512 or 1024 contiguous bytes per token) and keeps the
// inputs it needs in registers.
#include <stdint.h>

#include "ers_common.cuh"
#include "ers_internal.h"

namespace ers {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvVec = 8;    // channels per thread: one 16-byte access per token for bf16
constexpr int kConvRun = 8;   // tokens per CTA in the prefill kernel, all loaded before the math

// 8 consecutive channels of one token: bf16 as one uint4, fp32 as two float4.
template <typename T> struct Row8;
template <> struct Row8<__nv_bfloat16> {
  uint4 r;
  __device__ __forceinline__ void ld(const __nv_bfloat16* p) { r = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void st(__nv_bfloat16* p) const { *reinterpret_cast<uint4*>(p) = r; }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ void put(const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
      w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    r = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ __forceinline__ void zero() { r = make_uint4(0, 0, 0, 0); }
};
template <> struct Row8<float> {
  float4 a, b;
  __device__ __forceinline__ void ld(const float* p) {
    a = *reinterpret_cast<const float4*>(p);
    b = *reinterpret_cast<const float4*>(p + 4);
  }
  __device__ __forceinline__ void st(float* p) const {
    *reinterpret_cast<float4*>(p) = a;
    *reinterpret_cast<float4*>(p + 4) = b;
  }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  __device__ __forceinline__ void put(const float (&v)[8]) {
    a = make_float4(v[0], v[1], v[2], v[3]);
    b = make_float4(v[4], v[5], v[6], v[7]);
  }
  __device__ __forceinline__ void zero() {
    a = make_float4(0.f, 0.f, 0.f, 0.f);
    b = a;
  }
};

__device__ __forceinline__ float conv_act(float a, bool silu) {
  return silu ? __fdiv_rn(a, __fadd_rn(1.f, expf(-a))) : a;
}

// One output from the window u[0..W-1] (oldest first): bias, then the taps oldest to newest.
template <int W>
__device__ __forceinline__ float conv_out(float bias, const float (&w)[W], const float (&u)[W], bool silu) {
  float acc = bias;
#pragma unroll
  for (int k = 0; k < W; ++k) acc = __fmaf_rn(w[k], u[k], acc);
  return conv_act(acc, silu);
}

// Outputs of 8 channels from a window of W rows (row k = input k positions after the oldest).
template <typename T, int W>
__device__ __forceinline__ void conv_row(const Row8<T> (&win)[W], const float (&w)[kConvVec][W],
                                         const float (&b)[kConvVec], bool silu, Row8<T>* out) {
  float u[W][kConvVec], y[kConvVec];
#pragma unroll
  for (int k = 0; k < W; ++k) win[k].get(u[k]);
#pragma unroll
  for (int e = 0; e < kConvVec; ++e) {
    float ue[W];
#pragma unroll
    for (int k = 0; k < W; ++k) ue[k] = u[k][e];
    y[e] = conv_out<W>(b[e], w[e], ue, silu);
  }
  out->put(y);
}

struct ConvArgs {
  int C, nseq, nslots, read_state, silu;
  const int32_t* cu;
  const int32_t* slot;
  const void* x;
  const void* w;
  const void* bias;
  void* state;   // [nslots, W-1, C] or nullptr
  void* y;
  int32_t* status;
};

__device__ __forceinline__ bool conv_slot(const ConvArgs& a, int i, int* slot) {
  const int s = a.slot != nullptr ? a.slot[i] : i;
  if (s < 0 || s >= a.nslots) {
    if (threadIdx.x == 0) report(a.status, ERS_ESLOT);
    return false;
  }
  *slot = s;
  return true;
}

// The thread's 8 channels' taps are 8 W consecutive values of weight [C, W] (16-byte aligned since c
// is a multiple of 8): W (bf16) or 2 W (fp32) 16-byte loads.
template <typename T, int W>
__device__ __forceinline__ void load_weights(const ConvArgs& a, int c, float (&w)[kConvVec][W], float (&b)[kConvVec]) {
  const T* wp = (const T*)a.w + (size_t)c * W;
  float flat[kConvVec * W];
#pragma unroll
  for (int q = 0; q < W; ++q) {   // 8 values per Row8
    Row8<T> r;
    r.ld(wp + 8 * q);
    float v[8];
    r.get(v);
#pragma unroll
    for (int e = 0; e < 8; ++e) flat[8 * q + e] = v[e];
  }
#pragma unroll
  for (int e = 0; e < kConvVec; ++e)
#pragma unroll
    for (int k = 0; k < W; ++k) w[e][k] = flat[e * W + k];
  if (a.bias != nullptr) {
    Row8<T> r;
    r.ld((const T*)a.bias + c);
    r.get(b);
  } else {
#pragma unroll
    for (int e = 0; e < kConvVec; ++e) b[e] = 0.f;
  }
}

// Prefill over packed sequences: CTA (channel block, run of kConvRun tokens, sequence).  A thread
// loads its W - 1 halo rows and the run's rows first, then computes.  The CTA of run 0 also writes
// the final conv state (the last W - 1 entries of u), so the only CTA that writes a slot's state is
// the one that read it.
template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads) k_conv1d_fwd(ConvArgs a) {
  const int c = kConvVec * (blockIdx.x * kConvThreads + threadIdx.x);
  const int i = blockIdx.z, run = blockIdx.y;
  const int t0 = a.cu[i], n = a.cu[i + 1] - t0;
  const int r0 = run * kConvRun;
  if (r0 >= n && run != 0) return;
  int slot = -1;
  if (a.state != nullptr && !conv_slot(a, i, &slot)) return;
  if (c >= a.C) return;
  const T* __restrict__ x = (const T*)a.x;
  T* __restrict__ y = (T*)a.y;
  T* st = a.state != nullptr ? (T*)a.state + (size_t)slot * (W - 1) * a.C : nullptr;
  // u[k] = input at position r0 - (W - 1) + k, k < W - 1 + kConvRun
  Row8<T> u[W - 1 + kConvRun];
#pragma unroll
  for (int k = 0; k < W - 1 + kConvRun; ++k) {
    const int p = r0 - (W - 1) + k;
    if (p >= 0 && p < n) {
      u[k].ld(x + (size_t)(t0 + p) * a.C + c);
    } else if (p < 0 && st != nullptr && a.read_state) {
      u[k].ld(st + (size_t)(W - 1 + p) * a.C + c);
    } else {
      u[k].zero();
    }
  }
  float w[kConvVec][W], b[kConvVec];
  load_weights<T, W>(a, c, w, b);
#pragma unroll
  for (int t = 0; t < kConvRun; ++t) {
    if (r0 + t < n) {
      Row8<T> win[W], o;
#pragma unroll
      for (int k = 0; k < W; ++k) win[k] = u[t + k];
      conv_row<T, W>(win, w, b, a.silu, &o);
      o.st(y + (size_t)(t0 + r0 + t) * a.C + c);
    }
  }
  if (run == 0 && st != nullptr) {
    // final state: the W - 1 entries of u ending at position n - 1 (some may come from the old state)
    Row8<T> fin[W - 1];
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
      const int p = n - (W - 1) + k;
      if (p >= 0) {
        fin[k].ld(x + (size_t)(t0 + p) * a.C + c);
      } else if (a.read_state) {
        fin[k].ld(st + (size_t)(W - 1 + p) * a.C + c);
      } else {
        fin[k].zero();
      }
    }
#pragma unroll
    for (int k = 0; k < W - 1; ++k) fin[k].st(st + (size_t)k * a.C + c);
  }
}

// One decode step per sequence: y = conv(state, x_new), state <- (state[1:], x_new).  A thread
// serves its 8 channels of kConvSeqs sequences (the taps load once; all rows load before the math).
constexpr int kConvSeqs = 4;

template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads) k_conv1d_update(ConvArgs a) {
  const int c = kConvVec * (blockIdx.x * kConvThreads + threadIdx.x);
  const int i0 = blockIdx.y * kConvSeqs;
  int slots[kConvSeqs];
  bool ok[kConvSeqs];
#pragma unroll
  for (int q = 0; q < kConvSeqs; ++q) {
    ok[q] = i0 + q < a.nseq && conv_slot(a, i0 + q, &slots[q]);
  }
  if (c >= a.C) return;
  Row8<T> win[kConvSeqs][W];
#pragma unroll
  for (int q = 0; q < kConvSeqs; ++q) {
    if (!ok[q]) continue;
    const T* st = (const T*)a.state + (size_t)slots[q] * (W - 1) * a.C;
#pragma unroll
    for (int k = 0; k < W - 1; ++k) win[q][k].ld(st + (size_t)k * a.C + c);
    win[q][W - 1].ld((const T*)a.x + (size_t)(i0 + q) * a.C + c);
  }
  float w[kConvVec][W], b[kConvVec];
  load_weights<T, W>(a, c, w, b);
#pragma unroll
  for (int q = 0; q < kConvSeqs; ++q) {
    if (!ok[q]) continue;
    Row8<T> o;
    conv_row<T, W>(win[q], w, b, a.silu, &o);
    o.st((T*)a.y + (size_t)(i0 + q) * a.C + c);
    T* st = (T*)a.state + (size_t)slots[q] * (W - 1) * a.C;
#pragma unroll
    for (int k = 0; k < W - 1; ++k) win[q][k + 1].st(st + (size_t)k * a.C + c);
  }
}

template <typename T>
cudaError_t conv_dispatch(const ConvArgs& a, int W, bool update, int max_seqlen, cudaStream_t s) {
  const int cblocks = (a.C / kConvVec + kConvThreads - 1) / kConvThreads;
  const dim3 gu(cblocks, (a.nseq + kConvSeqs - 1) / kConvSeqs);
  const dim3 gf(cblocks, max(1, (max_seqlen + kConvRun - 1) / kConvRun), a.nseq);
#define ERS_CONV_W(w_)                                                     \
  if (W == w_) {                                                           \
    if (update)                                                            \
      k_conv1d_update<T, w_><<<gu, kConvThreads, 0, s>>>(a);               \
    else                                                                   \
      k_conv1d_fwd<T, w_><<<gf, kConvThreads, 0, s>>>(a);                  \
    return cudaGetLastError();                                             \
  }
  ERS_CONV_W(2)
  ERS_CONV_W(3)
  ERS_CONV_W(4)
#undef ERS_CONV_W
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t conv1d(const ConvLaunch& l, cudaStream_t s) {
  ConvArgs a;
  a.C = l.C;
  a.nseq = l.nseq;
  a.nslots = l.nslots;
  a.read_state = l.read_state;
  a.silu = l.silu;
  a.cu = l.cu;
  a.slot = l.slot;
  a.x = l.x;
  a.w = l.w;
  a.bias = l.bias;
  a.state = l.state;
  a.y = l.y;
  a.status = l.status;
  if (l.io == ERS_DTYPE_BF16) return conv_dispatch<__nv_bfloat16>(a, l.W, l.update, l.max_seqlen, s);
  return conv_dispatch<float>(a, l.W, l.update, l.max_seqlen, s);
}

}  // namespace ers
