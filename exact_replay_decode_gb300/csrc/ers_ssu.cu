// Per-token state-writeback update ("selective state update"): the recurrent decode kernel the
// exact-replay RFC (vLLM issue 55524, section 1) contrasts with the chunked scan, built here as the
// comparison point for replay decode.  Each step reads and writes the whole fp32 state:
//   S <- exp(delta A) S + (delta x) B^T ;  y = S C + D x
// One CTA per (sequence, head); a group of min(32, N) lanes owns one headdim row at a time, loads
// it with vector loads, updates it, and reduces S C over dstate with warp shuffles.
#include "ers_common.cuh"
#include "ers_internal.h"

namespace ers {
namespace {

template <typename T, int P, int N>
__global__ void __launch_bounds__(kThreads) k_ssu(LaunchArgs a) {
  using Dt = Dot<N>;
  constexpr int NG = kThreads / Dt::W;
  const int i = blockIdx.x, h = blockIdx.y;
  const int slot = a.slot != nullptr ? a.slot[i] : i;
  if (slot < 0 || slot >= a.nslots) {
    if (threadIdx.x == 0) report(a.status, ERS_ESLOT);
    return;
  }
  const int g = h / (a.H / a.G);
  const int gid = threadIdx.x / Dt::W, j = threadIdx.x % Dt::W;
  const float delta = delta_of(a.dt[(size_t)i * a.H + h], a.dt_bias[h]);
  const float decay = expf(__fmul_rn(delta, a.A[h]));
  const float Dh = a.D[h];
  const T* xr = (const T*)a.x + ((size_t)i * a.H + h) * P;
  float b[Dt::K], c[Dt::K];
  load_k<T, Dt::K>((const T*)a.B + ((size_t)i * a.G + g) * N + j * Dt::K, b);
  load_k<T, Dt::K>((const T*)a.C + ((size_t)i * a.G + g) * N + j * Dt::K, c);
  float* S = a.state + ((size_t)slot * a.H + h) * P * N;
  T* y = (T*)a.y + ((size_t)i * a.H + h) * P;
#pragma unroll 2
  for (int d0 = 0; d0 < P; d0 += NG) {
    const int d = d0 + gid;  // P is a multiple of NG for every supported shape
    float* row = S + (size_t)d * N + j * Dt::K;
    float sv[Dt::K];
    if constexpr (Dt::K == 4) {
      const float4 v = *reinterpret_cast<const float4*>(row);
      sv[0] = v.x; sv[1] = v.y; sv[2] = v.z; sv[3] = v.w;
    } else {
#pragma unroll
      for (int k = 0; k < Dt::K; ++k) sv[k] = row[k];
    }
    const float xd = to_f(xr[d]);
    const float u = __fmul_rn(delta, xd);
#pragma unroll
    for (int k = 0; k < Dt::K; ++k) sv[k] = __fmaf_rn(decay, sv[k], __fmul_rn(u, b[k]));
    if constexpr (Dt::K == 4) {
      *reinterpret_cast<float4*>(row) = make_float4(sv[0], sv[1], sv[2], sv[3]);
    } else {
#pragma unroll
      for (int k = 0; k < Dt::K; ++k) row[k] = sv[k];
    }
    const float dot = Dt::reduce(Dt::partial(sv, c));
    if (j == 0) y[d] = from_f<T>(__fmaf_rn(Dh, xd, dot));
  }
}

template <typename T, int P, int N>
cudaError_t ssu_impl(const LaunchArgs& a, cudaStream_t s) {
  static_assert(P % (kThreads / Dot<N>::W) == 0, "headdim must be a multiple of the row groups");
  if (a.nseq > 0) k_ssu<T, P, N><<<dim3(a.nseq, a.H), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

#define ERS_SSU_SHAPES(X) X(16, 16) X(32, 32) X(64, 64) X(64, 128)

}  // namespace

bool ssu_supported(int P, int N) {
#define ERS_SUP(p_, n_) if (P == p_ && N == n_) return true;
  ERS_SSU_SHAPES(ERS_SUP)
#undef ERS_SUP
  return false;
}

cudaError_t ssu_update(const LaunchArgs& a, cudaStream_t s) {
#define ERS_C(p_, n_)                                                   \
  if (a.P == p_ && a.N == n_) {                                         \
    if (a.io == ERS_DTYPE_BF16) return ssu_impl<__nv_bfloat16, p_, n_>(a, s); \
    return ssu_impl<float, p_, n_>(a, s);                               \
  }
  ERS_SSU_SHAPES(ERS_C)
#undef ERS_C
  return cudaErrorInvalidValue;
}

}  // namespace ers
