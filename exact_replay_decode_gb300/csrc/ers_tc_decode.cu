// Persistent replay-decode kernel (tensor-core engine, bf16 io, P = 64, N = 128, chunk Q <= 32):
// the exact-replay RFC's decode step (vLLM issue 55524, section 3) for a batch of sequences.
//
// Each CTA is one warpgroup (128 threads, one thread per tensor-memory lane) and walks (sequence,
// head) items; four CTAs share an SM so that while one waits on its tensor-core MMAs or loads,
// the others stream their checkpoints.  Per item:
//   * the fp32 boundary checkpoint (32 KiB) is loaded with 16-byte loads issued before anything
//     else and converted to the [H_hi; H_lo] operand tile;
//   * the buffered rows 0..p-1 and the new token are staged into the operand tiles (the new
//     token's C row in an 8-row aliased tile), and its inputs are appended to the buffer;
//   * the Gram (C_p . B_s), off-diagonal ([H_hi; H_lo] . C_p) and diagonal (M_p . X) MMAs are the
//     exact instruction sequences the prefill kernels issue for the same t-tile (tc_engine.cuh), so
//     y_p equals single-shot prefill bit for bit;
//   * when the chunk fills (p = Q - 1) the chunk state is contracted on the tensor cores and folded
//     into the checkpoint in the same launch.
// Tensor memory: 64 columns, used in turn by the Gram [0, Q), the off-diagonal [32, 32 + Q), the
// diagonal [0, 64) and the chunk state [0, 64).  ReplaySSM mode reads the bf16 read copy instead
// and never refreshes.
#include "ers_common.cuh"
#include "ers_internal.h"
#include "tc_engine.cuh"

namespace ers {
namespace {

using bf16 = __nv_bfloat16;
using namespace tc;

constexpr int kDecThreads = 128;
constexpr int kDecQMax = 32;
constexpr int kMetaBatch = 256;
constexpr uint32_t kDecCols = 64;
constexpr uint32_t kYoffCol = 32;

struct DecHdr {
  uint64_t mma_bar;
  uint32_t tmem;
  uint32_t pad;
  int32_t meta_slot[kMetaBatch];
  int32_t meta_p[kMetaBatch];
  float delta[kDecQMax];
  float ahi[kDecQMax];
  float alo[kDecQMax];
  float w[kDecQMax];
  float yh[P];
  float yl[P];
  float grow[64];   // Gram row p
  float ydg[P];     // diagonal row p
};
constexpr size_t kDecHdr = (sizeof(DecHdr) + 1023) & ~size_t(1023);

struct DecLayout {
  size_t Ht, Ca, Bt, Xt, Mhi, Mlo, total;
};
__host__ __device__ __forceinline__ DecLayout dec_layout(int Q) {
  DecLayout L;
  size_t o = kDecHdr;
  L.Ht = o; o += kHTile;                 // [H_hi; H_lo]; the refresh's U tiles reuse it
  L.Ca = o; o += 2048;                   // C alias tile: 8 rows x 2 atoms
  L.Mhi = o; o += 2048;                  // M alias tiles: 8 rows x 2 atoms
  L.Mlo = o; o += 2048;
  L.Bt = o; o += (size_t)Q * 256;
  L.Xt = o; o += (size_t)Q * 128;
  L.total = (o + 1023) & ~size_t(1023);
  return L;
}

extern __shared__ __align__(1024) unsigned char dec_smem[];

__device__ __forceinline__ unsigned char* dbase() {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dec_smem) + 1023) & ~uintptr_t(1023));
}

// warp-level Kogge-Stone scan of rows 0..31 (strides 1..16): per row, the same operations as the
// block scan the prefill kernels run (its strides >= 32 leave rows < 32 unchanged).
__device__ __forceinline__ void warp_scan32(float* hi, float* lo) {
  const int t = threadIdx.x;
  if (t < 32) {
    df v = {hi[t], lo[t]};
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const float oh = __shfl_up_sync(kFull, v.hi, s), ol = __shfl_up_sync(kFull, v.lo, s);
      if (t >= s) v = df_add(df{oh, ol}, v);
    }
    hi[t] = v.hi;
    lo[t] = v.lo;
  }
}

// slot and position of this CTA's items kb .. kb + kMetaBatch - 1 (p = -1 marks a skipped item)
__device__ __forceinline__ void load_meta(const LaunchArgs& a, int first, int stride, int kb, int nitems,
                                          DecHdr& hd) {
  for (int m = threadIdx.x; m < kMetaBatch; m += kDecThreads) {
    const int j = first + (kb + m) * stride;
    int slot = -1, p = -1;
    if (j < nitems) {
      const int i = j / a.H;
      const int s = a.slot != nullptr ? a.slot[i] : i;
      if (s < 0 || s >= a.nslots) {
        report(a.status, ERS_ESLOT);
      } else {
        const int pp = a.pos[s];
        if (pp < 0 || pp >= a.Q) report(a.status, ERS_EALIGN);
        else { slot = s; p = pp; }
      }
    }
    hd.meta_slot[m] = slot;
    hd.meta_p[m] = p;
  }
}

// issues the 16-byte loads of an item's checkpoint (fp32) or read copy (bf16) into registers
template <bool RSSM>
__device__ __forceinline__ void load_state(const LaunchArgs& a, int slot, int h, float4 (&sv)[RSSM ? 1 : 16],
                                           uint4 (&rv)[RSSM ? 8 : 1]) {
  const int tid = threadIdx.x;
  const size_t hs = (size_t)P * N;
  if (RSSM) {
    const uint4* R = reinterpret_cast<const uint4*>((const bf16*)a.read_copy + ((size_t)slot * a.H + h) * hs);
#pragma unroll
    for (int c = 0; c < 8; ++c) rv[c] = R[tid + c * kDecThreads];
  } else {
    const float4* S4 = reinterpret_cast<const float4*>(a.state + ((size_t)slot * a.H + h) * hs);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      sv[2 * c] = S4[2 * (tid + c * kDecThreads)];
      sv[2 * c + 1] = S4[2 * (tid + c * kDecThreads) + 1];
    }
  }
}

template <bool RSSM>
__global__ void __launch_bounds__(kDecThreads, 4) k_tc_decode_persistent(LaunchArgs a, int nitems) {
  const int first = blockIdx.x, stride = gridDim.x;
  if (first >= nitems) return;
  unsigned char* base = dbase();
  const int Q = a.Q;
  const DecLayout L = dec_layout(Q);
  DecHdr& hd = *reinterpret_cast<DecHdr*>(base);
  uint8_t* Ht = base + L.Ht;
  uint8_t* Ca = base + L.Ca;
  uint8_t* Bt = base + L.Bt;
  uint8_t* Xt = base + L.Xt;
  uint8_t* Mhi = base + L.Mhi;
  uint8_t* Mlo = base + L.Mlo;
  const Geom ge = geom(Q, 0);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tid = threadIdx.x;

  // one-time setup: zeroed operand tiles (every stale row stays finite), barrier, tensor memory
  for (size_t o = L.Ht + tid * 16; o < L.total; o += kDecThreads * 16)
    *reinterpret_cast<uint4*>(base + o) = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    mbar_init(&hd.mma_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&hd.tmem, kDecCols);
  before_sync();
  __syncthreads();
  after_sync();
  const uint32_t tb = hd.tmem;
  uint32_t mma_phase = 0;
  bool ok = true;
  const int nmine = (nitems - first + stride - 1) / stride;
  float4 sv[RSSM ? 1 : 16];
  uint4 rv[RSSM ? 8 : 1];
  bool have_next = false;
  int next_j = -1;

  for (int k = 0; k < nmine && ok; ++k) {
    if ((k % kMetaBatch) == 0) {
      __syncthreads();
      load_meta(a, first, stride, k, nitems, hd);
      __syncthreads();
    }
    const int j = first + k * stride;
    const int slot = hd.meta_slot[k % kMetaBatch], p = hd.meta_p[k % kMetaBatch];
    if (p < 0) continue;  // block-uniform
    const int i = j / a.H, h = j % a.H;
    const int g = h / (a.H / a.G);
    const size_t hs = (size_t)P * N;
    const bool refresh = !RSSM && (a.flags & ERS_FLAG_FUSE_REFRESH) && p + 1 == Q;

    // ---- the checkpoint (prefetched at the end of the previous item when possible)
    if (!have_next || next_j != j) load_state<RSSM>(a, slot, h, sv, rv);
    // ---- rows 0..p (buffer + new token), C_p, decays; append the new token to the buffer
    const Rows<bf16> rows = make_rows<bf16>(a, slot, h, p, (long long)i - p);
    for (int id = tid; id < (p + 1) * 24 + 16; id += kDecThreads) {
      if (id < (p + 1) * 24) {
        const int r = id / 24, c = id % 24;
        if (c < 8) row_to_tile(rows.x(r), Xt, 1, r, c);
        else row_to_tile(rows.B(r), Bt, Q, r, c - 8);
      } else {
        row_to_tile(rows.C(p), Ca, 8, p & 7, id - (p + 1) * 24);
      }
    }
    if (tid < kDecQMax) {
      float d = 0.f, da = 0.f;
      if (tid <= p) {
        d = delta_of(rows.dt(tid), a.dt_bias[h]);
        da = __fmul_rn(d, a.A[h]);
      }
      hd.delta[tid] = d;
      hd.ahi[tid] = da;
      hd.alo[tid] = 0.f;
    }
    {
      bf16* bx = (bf16*)a.bx + (((size_t)slot * Q + p) * a.H + h) * P;
      const bf16* nx = (const bf16*)a.x + ((size_t)i * a.H + h) * P;
      if (tid < 8) reinterpret_cast<uint4*>(bx)[tid] = reinterpret_cast<const uint4*>(nx)[tid];
      if (tid == 8) a.bdt[((size_t)slot * Q + p) * a.H + h] = a.dt[(size_t)i * a.H + h];
      if (h % (a.H / a.G) == 0 && tid >= 32 && tid < 64) {
        const int c = tid - 32;  // 16 chunks of B, then 16 of C
        const size_t dst = (((size_t)slot * Q + p) * a.G + g) * N, src = ((size_t)i * a.G + g) * N;
        if (c < 16)
          reinterpret_cast<uint4*>((bf16*)a.bB + dst)[c] = reinterpret_cast<const uint4*>((const bf16*)a.B + src)[c];
        else
          reinterpret_cast<uint4*>((bf16*)a.bC + dst)[c - 16] =
              reinterpret_cast<const uint4*>((const bf16*)a.C + src)[c - 16];
      }
    }
    __syncthreads();
    warp_scan32(hd.ahi, hd.alo);
    // ---- checkpoint -> [H_hi; H_lo] tile (or the read copy -> [R; 0]; the zero half is never written)
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int id = tid + c * kDecThreads;
      const int d = id / (N / 8), cc = id % (N / 8);
      if (RSSM) {
        *reinterpret_cast<uint4*>(Ht + sw128(128, d, 8 * cc)) = rv[c];
      } else {
        const float v[8] = {sv[2 * c].x, sv[2 * c].y, sv[2 * c].z, sv[2 * c].w,
                            sv[2 * c + 1].x, sv[2 * c + 1].y, sv[2 * c + 1].z, sv[2 * c + 1].w};
        uint4 hi, lo;
        split8(v, hi, lo);
        *reinterpret_cast<uint4*>(Ht + sw128(128, d, 8 * cc)) = hi;
        *reinterpret_cast<uint4*>(Ht + sw128(128, P + d, 8 * cc)) = lo;
      }
    }
    // the registers are free again: start the next item's checkpoint load now
    have_next = false;
    if (k + 1 < nmine && ((k + 1) % kMetaBatch) != 0) {
      const int pn = hd.meta_p[(k + 1) % kMetaBatch];
      if (pn >= 0) {
        next_j = first + (k + 1) * stride;
        load_state<RSSM>(a, hd.meta_slot[(k + 1) % kMetaBatch], next_j % a.H, sv, rv);
        have_next = true;
      }
    }
    publish();
    if (tid == 0) {
      issue_gram(tb, smem_u32(Ca), 8, 0, smem_u32(Bt), Q, ge.S_ext);
      issue_yoff(tb + kYoffCol, smem_u32(Ht), smem_u32(Ca), 8, 0, ge.TT);
      commit(&hd.mma_bar);
    }
    ok = __syncthreads_and(mbar_wait(&hd.mma_bar, mma_phase, a.status));
    mma_phase ^= 1;
    after_sync();
    if (!ok) break;
    // ---- off-diagonal column p -> yh / yl (all lanes); masked decayed Gram row p -> M alias tiles
    {
      float v[16];
      tmem_ld16(taddr(tb, 32 * warp, kYoffCol + 16 * (p / 16)), v);
      float val = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (e == (p & 15)) val = v[e];
      if (tid < P) hd.yh[tid] = val;
      else hd.yl[tid - P] = val;
    }
    if (warp == p / 32) {
      float gv[64];
      tmem_ld64(taddr(tb, 32 * warp, 0), gv);
      if (lane == (p & 31)) {
#pragma unroll
        for (int c = 0; c < kDecQMax / 4; ++c)
          *reinterpret_cast<float4*>(&hd.grow[4 * c]) = make_float4(gv[4 * c], gv[4 * c + 1], gv[4 * c + 2], gv[4 * c + 3]);
      }
    }
    __syncthreads();
    if (tid < kDecQMax) {  // M[p][s] = (G[p][s] delta_s) exp(Acum_p - Acum_s), s <= p; split hi + lo
      const int sidx = tid;
      float m = 0.f;
      if (sidx <= p)
        m = __fmul_rn(__fmul_rn(hd.grow[sidx], hd.delta[sidx]),
                      expf(df_diff(df{hd.ahi[p], hd.alo[p]}, df{hd.ahi[sidx], hd.alo[sidx]})));
      const bf16 mh = __float2bfloat16_rn(m);
      const bf16 ml = __float2bfloat16_rn(__fsub_rn(m, __bfloat162float(mh)));
      const uint32_t off = sw128(8, p & 7, sidx);
      *reinterpret_cast<bf16*>(Mhi + off) = mh;
      *reinterpret_cast<bf16*>(Mlo + off) = ml;
    }
    publish();
    if (tid == 0) {
      issue_ydiag(tb, smem_u32(Mhi), smem_u32(Mlo), 8, 0, smem_u32(Xt), 0, ge.S_ext);
      commit(&hd.mma_bar);
    }
    ok = __syncthreads_and(mbar_wait(&hd.mma_bar, mma_phase, a.status));
    mma_phase ^= 1;
    after_sync();
    if (!ok) break;
    // ---- combine row p: the diagonal row goes through shared memory, one thread per headdim column
    if (warp == p / 32) {
      float yd[64];
      tmem_ld64(taddr(tb, 32 * warp, 0), yd);
      if (lane == (p & 31)) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<float4*>(&hd.ydg[4 * c]) = make_float4(yd[4 * c], yd[4 * c + 1], yd[4 * c + 2], yd[4 * c + 3]);
      }
    }
    __syncthreads();
    if (tid < P) {
      const int d = tid;
      const float xv = __bfloat162float(*reinterpret_cast<const bf16*>(Xt + sw128(1, p, d)));
      const float o = combine_out(expf(hd.ahi[p]), __fadd_rn(hd.yh[d], hd.yl[d]), hd.ydg[d], a.D[h], xv);
      ((bf16*)a.y)[((size_t)i * a.H + h) * P + d] = __float2bfloat16_rn(o);
    }
    // ---- the chunk filled: contract its state and fold it into the checkpoint
    if (refresh) {
      if (tid < Q) {
        const df last = {hd.ahi[Q - 1], hd.alo[Q - 1]};
        hd.w[tid] = __fmul_rn(hd.delta[tid], expf(df_diff(last, df{hd.ahi[tid], hd.alo[tid]})));
      }
      __syncthreads();
      uint8_t* u0 = Ht;
      uint8_t* u1 = Ht + (size_t)Q * 128;
      uint8_t* u2 = Ht + (size_t)2 * Q * 128;
      build_u_tiles(Xt, hd.w, Q, 0, Q, u0, u1, u2);
      publish();
      if (tid == 0) {
        issue_state_block(tb, smem_u32(Bt), Q, smem_u32(u0), smem_u32(u1), smem_u32(u2), 0, Q / 16);
        commit(&hd.mma_bar);
      }
      ok = __syncthreads_and(mbar_wait(&hd.mma_bar, mma_phase, a.status));
      mma_phase ^= 1;
      after_sync();
      if (!ok) break;
      const float decay = expf(hd.ahi[Q - 1]);
      float* Hd = a.state + ((size_t)slot * a.H + h) * hs;
      bf16* Rd = a.read_copy ? (bf16*)a.read_copy + ((size_t)slot * a.H + h) * hs : nullptr;
      float s[64];
      tmem_ld64(taddr(tb, 32 * warp, 0), s);
      const int n = tid;
#pragma unroll 8
      for (int d = 0; d < P; ++d) {
        const float v = __fmaf_rn(decay, Hd[d * N + n], s[d]);
        Hd[d * N + n] = v;
        if (Rd != nullptr) Rd[d * N + n] = __float2bfloat16_rn(v);
      }
    }
    // every thread is done with this item's tiles and tensor memory before the next item writes them
    before_sync();
    __syncthreads();
    after_sync();
  }
  before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, kDecCols);
}

}  // namespace

bool tc_decode_persistent_supported(int Q) { return Q <= kDecQMax; }

cudaError_t tc_decode_persistent(const LaunchArgs& a, cudaStream_t s) {
  const DecLayout L = dec_layout(a.Q);
  const size_t smem = L.total + 1024;
  const int nitems = a.nseq * a.H;
  int dev = 0, nsm = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int grid = nitems < 4 * nsm ? nitems : 4 * nsm;
  cudaError_t e;
  if (a.flags & ERS_FLAG_REPLAYSSM) {
    if ((e = cudaFuncSetAttribute(k_tc_decode_persistent<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    if (grid > 0) k_tc_decode_persistent<true><<<grid, kDecThreads, smem, s>>>(a, nitems);
  } else {
    if ((e = cudaFuncSetAttribute(k_tc_decode_persistent<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    if (grid > 0) k_tc_decode_persistent<false><<<grid, kDecThreads, smem, s>>>(a, nitems);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_setpos(a, 0, s);
}

}  // namespace ers
