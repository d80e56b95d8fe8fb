// Warp-specialized persistent replay-decode kernel (tensor-core engine, bf16 io, P = 64, N = 128,
// chunk Q = 16).  One item is a sequence and a block of up to 8 heads sharing one B/C group.
//
// Exact-replay decode (vLLM issue 55524, section 3) per head: replay the buffered rows 0..p-1 and
// the new token from the fp32 boundary checkpoint, output y_p, append the token, and fold the
// chunk into the checkpoint when it fills.  Heads of one group read the same B and C rows, so an
// item stages those rows once and computes the Gram C_p . B_s once.
//
// A tcgen05 MMA costs about the same for any N up to 256, so the off-diagonal contraction
// (tokens on M, headdim rows on N) takes two heads per instruction: their checkpoints land by bulk
// asynchronous copy in one 64 KB ring stage, which the workers rewrite in place as the 256-row
// operand [H_hi(a); H_lo(a); H_hi(b); H_lo(b)].  The diagonal term holds M_hi and M_lo in two rows
// of one 8-row aliased tile and runs one MMA chain per head.
//
// Roles (one CTA per SM, 9 warps):
//   warp 8 (lane 0) — producer and MMA issuer: keeps the two ring stages filled and issues each
//     head pair's off-diagonal MMAs once its stage is rewritten;
//   warps 0-7 — stage the rows, rewrite the ring stages, read the results, and run the item's
//     epilogue (Gram, M rows, diagonal MMAs, outputs, refresh), synchronising among themselves
//     with a named barrier.
// Every per-head result is bit-identical to the prefill kernels' for the same t-tile (a row's or
// column's MMA result depends only on that row/column, whatever N or the column position).
//
// Tensor memory (512 columns): off-diagonal of head pair g at [256 (g % 2), +256) (per head: hi 64
// columns then lo 64); epilogue: Gram [0, 16), then the diagonal of head hh at [64 hh, +64), then
// chunk states of up to four heads at [64 u, +64).
#include "ers_common.cuh"
#include "ers_internal.h"
#include "tc_engine.cuh"

namespace ers {
namespace {

using bf16 = __nv_bfloat16;
using namespace tc;

constexpr int kWorkers = 256;     // warps 0-7
constexpr int kGThreads = kWorkers + 32;
constexpr int kGQ = 16;           // the chunk size this kernel handles
constexpr int kGHeads = 8;        // heads per item (at most)
constexpr int kGMeta = 256;
constexpr uint32_t kGCols = 512;
constexpr int kGStage = 6;        // 16-byte chunks staged per worker: ceil((16*16 + 16 + 8*16*8) / 256)
constexpr uint32_t kPairBytes = 65536;
constexpr uint32_t kWorkBar = 1;  // named barrier id of the workers

struct GHdr {
  uint64_t stage_full[2];   // bulk copies landed (tx)
  uint64_t tile_full[2];    // stage rewritten as an operand (8 worker warps)
  uint64_t stage_empty[2];  // the pair's MMAs completed (commit)
  uint64_t pair_done[2];    // per TMEM region: the pair's MMAs completed (commit)
  uint64_t tmem_free[2];    // per TMEM region: the pair's row was read (worker)
  uint64_t bar_mma;         // worker-issued epilogue MMAs
  uint32_t tmem;
  uint32_t abort;
  int32_t meta_slot[kGMeta];
  int32_t meta_p[kGMeta];
  float delta[kGHeads][32];
  float ahi[kGHeads][32];
  float alo[kGHeads][32];
  float w[kGHeads][kGQ];
  float yo[kGHeads][2 * P];  // off-diagonal row p: hi then lo
  float yd[kGHeads][2 * P];  // diagonal row p: hi then lo
  float grow[kGQ];
};
constexpr size_t kGHdr = (sizeof(GHdr) + 1023) & ~size_t(1023);

struct GLayout {
  size_t St, Ca, Ma, Bt, Xt, U, total;
};
__host__ __device__ __forceinline__ GLayout g_layout() {
  GLayout L;
  size_t o = kGHdr;
  L.St = o; o += 2 * (size_t)kPairBytes;        // two pair stages
  L.Ca = o; o += 2048;                          // C alias tile (8 rows x 2 atoms)
  L.Ma = o; o += (size_t)kGHeads * 1024;        // per head: M alias tile (hi row p%8, lo row (p+4)%8)
  L.Bt = o; o += (size_t)kGQ * 256;
  L.Xt = o; o += (size_t)kGHeads * kGQ * 128;
  L.U = o; o += (size_t)4 * 3 * kGQ * 128;      // refresh U tiles for four heads
  L.total = (o + 1023) & ~size_t(1023);
  return L;
}

extern __shared__ __align__(1024) unsigned char g_smem[];

__device__ __forceinline__ unsigned char* gbase() {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(g_smem) + 1023) & ~uintptr_t(1023));
}

// warp-level Kogge-Stone scan of rows 0..31: per row the same operations as the prefill block scan
__device__ __forceinline__ void warp_scan_rows(float* hi, float* lo, int lane) {
  df v = {hi[lane], lo[lane]};
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const float oh = __shfl_up_sync(kFull, v.hi, s), ol = __shfl_up_sync(kFull, v.lo, s);
    if (lane >= s) v = df_add(df{oh, ol}, v);
  }
  if (lane < kGQ) {  // rows >= kGQ stay zero
    hi[lane] = v.hi;
    lo[lane] = v.lo;
  }
}

// Rewrites a pair stage in place: fp32 checkpoints of heads a (bytes [0, 32K)) and b ([32K, 64K)),
// or bf16 read copies (a at [0, 16K), b at [16K, 32K)), become the 256-row swizzled operand
// [H_hi(a); H_lo(a); H_hi(b); H_lo(b)] (read copies: lo rows zero).  Workers only.
template <bool RSSM>
__device__ __forceinline__ void g_rewrite(unsigned char* stage) {
  const int tid = threadIdx.x;
  if (RSSM) {
    uint4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = reinterpret_cast<const uint4*>(stage)[tid + c * kWorkers];
    named_sync(kWorkBar, kWorkers);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int id = tid + c * kWorkers;          // (head, d, 8-column chunk)
      const int hb = id / (P * 16), d = (id / 16) % P, cc = id % 16;
      const uint32_t r = 128 * hb + d;
      *reinterpret_cast<uint4*>(stage + sw128(256, r, 8 * cc)) = v[c];
      *reinterpret_cast<uint4*>(stage + sw128(256, r + P, 8 * cc)) = make_uint4(0, 0, 0, 0);
    }
  } else {
    float4 v[16];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      v[2 * c] = reinterpret_cast<const float4*>(stage)[2 * (tid + c * kWorkers)];
      v[2 * c + 1] = reinterpret_cast<const float4*>(stage)[2 * (tid + c * kWorkers) + 1];
    }
    named_sync(kWorkBar, kWorkers);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int id = tid + c * kWorkers;
      const int hb = id / (P * 16), d = (id / 16) % P, cc = id % 16;
      const uint32_t r = 128 * hb + d;
      const float f[8] = {v[2 * c].x, v[2 * c].y, v[2 * c].z, v[2 * c].w,
                          v[2 * c + 1].x, v[2 * c + 1].y, v[2 * c + 1].z, v[2 * c + 1].w};
      uint4 hi, lo;
      split8(f, hi, lo);
      *reinterpret_cast<uint4*>(stage + sw128(256, r, 8 * cc)) = hi;
      *reinterpret_cast<uint4*>(stage + sw128(256, r + P, 8 * cc)) = lo;
    }
  }
}

// Producer cursor over the CTA's head pairs of the current metadata batch.
struct GCursor {
  int item, pair;
};

template <bool RSSM>
__device__ __forceinline__ bool g_issue_pair(const LaunchArgs& a, const GHdr& hd, GCursor& cur, int nbatch,
                                             int nblk, int HB, int first, int stride, int kb, unsigned char* stage,
                                             uint64_t* bar) {
  while (cur.item < nbatch && hd.meta_p[cur.item] < 0) { ++cur.item; cur.pair = 0; }
  if (cur.item >= nbatch) return false;
  const int j = first + (kb + cur.item) * stride;
  const int slot = hd.meta_slot[cur.item];
  const int ha = (j % nblk) * HB + 2 * cur.pair;
  const int nh = (2 * cur.pair + 1 < HB) ? 2 : 1;
  const size_t hs = (size_t)P * N;
  const uint32_t hb = RSSM ? (uint32_t)(hs * 2) : (uint32_t)(hs * 4);
  mbar_arrive_expect_tx(bar, hb * nh);
  for (int u = 0; u < nh; ++u) {
    if (RSSM) bulk_g2s(stage + u * hb, (const bf16*)a.read_copy + ((size_t)slot * a.H + ha + u) * hs, hb, bar);
    else bulk_g2s(stage + u * hb, a.state + ((size_t)slot * a.H + ha + u) * hs, hb, bar);
  }
  if (++cur.pair == (HB + 1) / 2) { cur.pair = 0; ++cur.item; }
  return true;
}

template <bool RSSM>
__global__ void __launch_bounds__(kGThreads, 1) k_tc_decode_group(LaunchArgs a, int HB, int nitems) {
  const int first = blockIdx.x, stride = gridDim.x;
  if (first >= nitems) return;
  unsigned char* base = gbase();
  const int Q = kGQ;
  const GLayout L = g_layout();
  GHdr& hd = *reinterpret_cast<GHdr*>(base);
  uint8_t* Ca = base + L.Ca;
  uint8_t* Ma0 = base + L.Ma;
  uint8_t* Bt = base + L.Bt;
  uint8_t* Xt0 = base + L.Xt;
  uint8_t* U0 = base + L.U;
  const Geom ge = geom(Q, 0);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3, half = (warp >> 2) & 1;
  const int tid = threadIdx.x;
  const bool worker = warp < 8;
  const int nblk = a.H / HB;
  const int npairs = (HB + 1) / 2;
  const size_t hs = (size_t)P * N;

  for (size_t o = L.St + tid * 16; o < L.total; o += kGThreads * 16)
    *reinterpret_cast<uint4*>(base + o) = make_uint4(0, 0, 0, 0);
  for (int e = tid; e < kGHeads * 32; e += kGThreads) {
    hd.delta[e / 32][e % 32] = 0.f;
    hd.ahi[e / 32][e % 32] = 0.f;
    hd.alo[e / 32][e % 32] = 0.f;
  }
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&hd.stage_full[s], 1);
      mbar_init(&hd.tile_full[s], 8);
      mbar_init(&hd.stage_empty[s], 1);
      mbar_init(&hd.pair_done[s], 1);
      mbar_init(&hd.tmem_free[s], 1);
    }
    mbar_init(&hd.bar_mma, 1);
    hd.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&hd.tmem, kGCols);
  before_sync();
  __syncthreads();
  after_sync();
  const uint32_t tb = hd.tmem;
  const int nmine = (nitems - first + stride - 1) / stride;
  uint32_t gp = 0;          // head pairs processed so far (both roles count identically)
  uint32_t mma_phase = 0;   // worker-issued epilogue MMAs

  for (int kb = 0; kb < nmine; kb += kGMeta) {
    const int nbatch = nmine - kb < kGMeta ? nmine - kb : kGMeta;
    __syncthreads();
    for (int m = tid; m < kGMeta; m += kGThreads) {
      int slot = -1, p = -1;
      if (m < nbatch) {
        const int jj = first + (kb + m) * stride;
        const int i = jj / nblk;
        const int sl = a.slot != nullptr ? a.slot[i] : i;
        if (sl < 0 || sl >= a.nslots) {
          if ((jj % nblk) == 0) report(a.status, ERS_ESLOT);
        } else {
          const int pp = a.pos[sl];
          if (pp < 0 || pp >= Q) {
            if ((jj % nblk) == 0) report(a.status, ERS_EALIGN);
          } else {
            slot = sl;
            p = pp;
          }
        }
      }
      hd.meta_slot[m] = slot;
      hd.meta_p[m] = p;
    }
    __syncthreads();
    if (hd.abort) break;

    if (!worker) {
      // ======================= producer / MMA issuer (one thread) =======================
      if (lane == 0) {
        GCursor cur = {0, 0};
        uint32_t g = gp;
        bool have = g_issue_pair<RSSM>(a, hd, cur, nbatch, nblk, HB, first, stride, kb,
                                       base + L.St + (size_t)(g % 2) * kPairBytes, &hd.stage_full[g % 2]);
        bool ok = true;
        while (have && ok) {
          // refill the other stage with the next pair once its previous pair's MMAs are done
          const uint32_t gn = g + 1;
          if (gn >= 2) ok = mbar_wait(&hd.stage_empty[gn % 2], ((gn - 2) / 2) & 1u, a.status);
          if (!ok) break;
          const bool have_next = g_issue_pair<RSSM>(a, hd, cur, nbatch, nblk, HB, first, stride, kb,
                                                    base + L.St + (size_t)(gn % 2) * kPairBytes,
                                                    &hd.stage_full[gn % 2]);
          // this pair: operand ready, TMEM region read by the workers
          ok = mbar_wait(&hd.tile_full[g % 2], (g / 2) & 1u, a.status);
          if (ok && g >= 2) ok = mbar_wait(&hd.tmem_free[g % 2], ((g - 2) / 2) & 1u, a.status);
          if (!ok) break;
          after_sync();
          issue_yoff(tb + 256 * (g % 2), smem_u32(Ca), 8, 0, smem_u32(base + L.St + (size_t)(g % 2) * kPairBytes), 256);
          commit(&hd.stage_empty[g % 2]);
          commit(&hd.pair_done[g % 2]);
          g = gn;
          have = have_next;
        }
        // the last pair's stage must be free before the next batch (or the end)
        if (ok && g >= 1) ok = mbar_wait(&hd.stage_empty[(g - 1) % 2], ((g - 1) / 2) & 1u, a.status);
        if (!ok) atomicExch(&hd.abort, 1u);
      }
    } else {
      // ============================ workers (warps 0-7) ============================
      bool ok = true;
      for (int kk = 0; kk < nbatch && ok; ++kk) {
        const int slot = hd.meta_slot[kk], p = hd.meta_p[kk];
        if (p < 0) continue;
        const int j = first + (kb + kk) * stride;
        const int i = j / nblk, h0 = (j % nblk) * HB;
        const int grp = h0 / (a.H / a.G);
        const bool refresh = !RSSM && (a.flags & ERS_FLAG_FUSE_REFRESH) && p + 1 == Q;
        // ---- stage B rows 0..p, C_p, x rows 0..p of every head; the new token also goes to the buffer
        {
          const int nB = (p + 1) * 16, nX = (p + 1) * 8;
          const int total = nB + 16 + HB * nX;
          uint4 buf[kGStage];
#pragma unroll
          for (int u = 0; u < kGStage; ++u) {
            const int id = tid + u * kWorkers;
            if (id < total) {
              const bf16* src;
              if (id < nB) {
                const int r = id / 16;
                src = (r < p ? (const bf16*)a.bB + (((size_t)slot * Q + r) * a.G + grp) * N
                             : (const bf16*)a.B + ((size_t)i * a.G + grp) * N) + 8 * (id % 16);
              } else if (id < nB + 16) {
                src = (const bf16*)a.C + ((size_t)i * a.G + grp) * N + 8 * (id - nB);
              } else {
                const int id2 = id - nB - 16, hh = id2 / nX, r = (id2 % nX) / 8, c = id2 % 8;
                const int h = h0 + hh;
                src = (r < p ? (const bf16*)a.bx + (((size_t)slot * Q + r) * a.H + h) * P
                             : (const bf16*)a.x + ((size_t)i * a.H + h) * P) + 8 * c;
              }
              buf[u] = *reinterpret_cast<const uint4*>(src);
            }
          }
          if (tid < HB * kGQ) {
            const int hh = tid / kGQ, r = tid % kGQ, h = h0 + hh;
            float d = 0.f, da = 0.f;
            if (r <= p) {
              const float dtr = r < p ? a.bdt[((size_t)slot * Q + r) * a.H + h] : a.dt[(size_t)i * a.H + h];
              d = delta_of(dtr, a.dt_bias[h]);
              da = __fmul_rn(d, a.A[h]);
              if (r == p) a.bdt[((size_t)slot * Q + p) * a.H + h] = dtr;
            }
            hd.delta[hh][r] = d;
            hd.ahi[hh][r] = da;
            hd.alo[hh][r] = 0.f;
          }
#pragma unroll
          for (int u = 0; u < kGStage; ++u) {
            const int id = tid + u * kWorkers;
            if (id < total) {
              if (id < nB) {
                const int r = id / 16, c = id % 16;
                *reinterpret_cast<uint4*>(Bt + sw128(Q, r, 8 * c)) = buf[u];
                if (r == p && h0 % (a.H / a.G) == 0)
                  *reinterpret_cast<uint4*>((bf16*)a.bB + (((size_t)slot * Q + p) * a.G + grp) * N + 8 * c) = buf[u];
              } else if (id < nB + 16) {
                const int c = id - nB;
                *reinterpret_cast<uint4*>(Ca + sw128(8, p & 7, 8 * c)) = buf[u];
                if (h0 % (a.H / a.G) == 0)
                  *reinterpret_cast<uint4*>((bf16*)a.bC + (((size_t)slot * Q + p) * a.G + grp) * N + 8 * c) = buf[u];
              } else {
                const int id2 = id - nB - 16, hh = id2 / nX, r = (id2 % nX) / 8, c = id2 % 8;
                *reinterpret_cast<uint4*>(Xt0 + (size_t)hh * Q * 128 + sw128(1, r, 8 * c)) = buf[u];
                if (r == p)
                  *reinterpret_cast<uint4*>((bf16*)a.bx + (((size_t)slot * Q + p) * a.H + h0 + hh) * P + 8 * c) =
                      buf[u];
              }
            }
          }
        }
        fence_async_smem();
        named_sync(kWorkBar, kWorkers);
        if (warp < HB) warp_scan_rows(hd.ahi[warp], hd.alo[warp], lane);
        // ---- head pairs: rewrite each stage as an operand; read the previous pair's row p
        for (int pp = 0; pp <= npairs && ok; ++pp) {
          if (pp < npairs) {
            const uint32_t g = gp + pp;
            ok = named_sync_and(kWorkBar, kWorkers,
                                mbar_wait(&hd.stage_full[g % 2], (g / 2) & 1u, a.status) && !hd.abort);
            if (!ok) break;
            g_rewrite<RSSM>(base + L.St + (size_t)(g % 2) * kPairBytes);
            fence_async_smem();
            before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&hd.tile_full[g % 2]);
          }
          if (pp >= 1 && warp == 0) {  // row p of pair pp - 1 (lane p holds it)
            const uint32_t g = gp + pp - 1;
            const bool w = mbar_wait(&hd.pair_done[g % 2], (g / 2) & 1u, a.status);
            if (__all_sync(kFull, w)) {
              after_sync();
              const int nh = (2 * (pp - 1) + 1 < HB) ? 2 : 1;
              for (int u = 0; u < nh; ++u) {
                float v[64];
                tmem_ld64(taddr(tb, 0, 256 * (g % 2) + 128 * u), v);
                if (lane == p) {
#pragma unroll
                  for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<float4*>(&hd.yo[2 * (pp - 1) + u][4 * c]) =
                        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                }
                tmem_ld64(taddr(tb, 0, 256 * (g % 2) + 128 * u + 64), v);
                if (lane == p) {
#pragma unroll
                  for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<float4*>(&hd.yo[2 * (pp - 1) + u][P + 4 * c]) =
                        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                }
              }
              before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(&hd.tmem_free[g % 2]);
            } else if (lane == 0) {
              atomicExch(&hd.abort, 1u);
            }
          }
        }
        gp += npairs;
        ok = named_sync_and(kWorkBar, kWorkers, ok && !hd.abort);
        if (!ok) break;
        after_sync();
        // ---- epilogue: Gram, M rows, diagonal (TMEM regions are free: every pair was read)
        if (tid == 0) {
          issue_gram(tb, smem_u32(Ca), 8, 0, smem_u32(Bt), Q, ge.S_ext);
          commit(&hd.bar_mma);
        }
        ok = named_sync_and(kWorkBar, kWorkers, mbar_wait(&hd.bar_mma, mma_phase, a.status));
        mma_phase ^= 1;
        if (!ok) break;
        after_sync();
        if (warp == 0) {
          float gv[16];
          tmem_ld16(taddr(tb, 0, 0), gv);
          if (lane == p) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<float4*>(&hd.grow[4 * c]) = make_float4(gv[4 * c], gv[4 * c + 1], gv[4 * c + 2], gv[4 * c + 3]);
          }
        }
        before_sync();
        named_sync(kWorkBar, kWorkers);
        after_sync();
        // M[p][s] = (G[p][s] delta_s) exp(Acum_p - Acum_s) for s <= p: hi at row p % 8, lo at row (p + 4) % 8
        if (tid < HB * kGQ) {
          const int hh = tid / kGQ, s2 = tid % kGQ;
          float m = 0.f;
          if (s2 <= p)
            m = __fmul_rn(__fmul_rn(hd.grow[s2], hd.delta[hh][s2]),
                          expf(df_diff(df{hd.ahi[hh][p], hd.alo[hh][p]}, df{hd.ahi[hh][s2], hd.alo[hh][s2]})));
          const bf16 mh = __float2bfloat16_rn(m);
          const bf16 ml = __float2bfloat16_rn(__fsub_rn(m, __bfloat162float(mh)));
          uint8_t* mt = Ma0 + (size_t)hh * 1024;
          *reinterpret_cast<bf16*>(mt + sw128(8, p & 7, s2)) = mh;
          *reinterpret_cast<bf16*>(mt + sw128(8, (p + 4) & 7, s2)) = ml;
        }
        fence_async_smem();
        before_sync();
        named_sync(kWorkBar, kWorkers);
        after_sync();
        if (tid == 0) {
          for (int hh = 0; hh < HB; ++hh)
            issue_ydiag(tb + 64 * hh, smem_u32(Ma0 + hh * 1024), 8, 0, smem_u32(Xt0 + (size_t)hh * Q * 128), 0,
                        ge.S_ext);
          commit(&hd.bar_mma);
        }
        ok = named_sync_and(kWorkBar, kWorkers, mbar_wait(&hd.bar_mma, mma_phase, a.status));
        mma_phase ^= 1;
        if (!ok) break;
        after_sync();
        if (q == 0) {  // warps 0 and 4 split the heads; lane p holds the hi row, lane p + 4 the lo row
          for (int hh = half; hh < HB; hh += 2) {
            float v[64];
            tmem_ld64(taddr(tb, 0, 64 * hh), v);
            if (lane == p || lane == p + 4) {
              float* dst = &hd.yd[hh][lane == p ? 0 : P];
#pragma unroll
              for (int c = 0; c < 16; ++c)
                *reinterpret_cast<float4*>(dst + 4 * c) = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            }
          }
        }
        before_sync();
        named_sync(kWorkBar, kWorkers);
        after_sync();
        // ---- outputs: one worker per (head, headdim column)
        for (int o = tid; o < HB * P; o += kWorkers) {
          const int hh = o / P, d = o % P, h = h0 + hh;
          const float xv =
              __bfloat162float(*reinterpret_cast<const bf16*>(Xt0 + (size_t)hh * Q * 128 + sw128(1, p, d)));
          const float y = combine_out(expf(hd.ahi[hh][p]), __fadd_rn(hd.yo[hh][d], hd.yo[hh][P + d]),
                                      __fadd_rn(hd.yd[hh][d], hd.yd[hh][P + d]), a.D[h], xv);
          ((bf16*)a.y)[((size_t)i * a.H + h) * P + d] = __float2bfloat16_rn(y);
        }
        // ---- the chunk filled: contract every head's chunk state and fold it into its checkpoint
        if (refresh) {
          if (tid < HB * kGQ) {
            const int hh = tid / kGQ, s2 = tid % kGQ;
            const df last = {hd.ahi[hh][Q - 1], hd.alo[hh][Q - 1]};
            hd.w[hh][s2] = __fmul_rn(hd.delta[hh][s2], expf(df_diff(last, df{hd.ahi[hh][s2], hd.alo[hh][s2]})));
          }
          named_sync(kWorkBar, kWorkers);
          const size_t usz = (size_t)Q * 128;
          for (int b0 = 0; b0 < HB && ok; b0 += 4) {
            const int nb = HB - b0 < 4 ? HB - b0 : 4;
            for (int u = 0; u < nb; ++u) {
              uint8_t* ub = U0 + (size_t)u * 3 * usz;
              build_u_tiles(Xt0 + (size_t)(b0 + u) * Q * 128, hd.w[b0 + u], Q, 0, Q, ub, ub + usz, ub + 2 * usz);
            }
            fence_async_smem();
            before_sync();
            named_sync(kWorkBar, kWorkers);
            after_sync();
            if (tid == 0) {
              for (int u = 0; u < nb; ++u) {
                const uint8_t* ub = U0 + (size_t)u * 3 * usz;
                issue_state_block(tb + 64 * u, smem_u32(Bt), Q, smem_u32(ub), smem_u32(ub + usz),
                                  smem_u32(ub + 2 * usz), 0, Q / 16);
              }
              commit(&hd.bar_mma);
            }
            ok = named_sync_and(kWorkBar, kWorkers, mbar_wait(&hd.bar_mma, mma_phase, a.status));
            mma_phase ^= 1;
            if (!ok) break;
            after_sync();
            for (int u = 0; u < nb; ++u) {  // warp (q, half): lanes n = 32 q + lane, columns [32 half, +32)
              const int h = h0 + b0 + u;
              const float decay = expf(hd.ahi[b0 + u][Q - 1]);
              float* Hd = a.state + ((size_t)slot * a.H + h) * hs;
              bf16* Rd = a.read_copy ? (bf16*)a.read_copy + ((size_t)slot * a.H + h) * hs : nullptr;
              const int n = 32 * q + lane;
              float sv2[32];
              tmem_ld32(taddr(tb, 32 * q, 64 * u + 32 * half), sv2);
              float old[32];
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) old[jj] = Hd[(32 * half + jj) * N + n];
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int d = 32 * half + jj;
                const float v = __fmaf_rn(decay, old[jj], sv2[jj]);
                Hd[d * N + n] = v;
                if (Rd != nullptr) Rd[d * N + n] = __float2bfloat16_rn(v);
              }
            }
            before_sync();
            named_sync(kWorkBar, kWorkers);
            after_sync();
          }
        }
        before_sync();
        named_sync(kWorkBar, kWorkers);
        after_sync();
      }
      if (!ok && tid == 0) atomicExch(&hd.abort, 1u);
    }
    __syncthreads();
    if (hd.abort) break;
  }
  // a timed-out wait may leave ring copies in flight: give them a bounded time to land
  if (hd.abort && tid == 0) {
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 50000000ull) {
    }
  }
  before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, kGCols);
}

}  // namespace

// heads per item: the largest divisor of the group size that is at most 8
int tc_decode_group_heads(int H, int G) {
  const int HG = H / G;
  for (int hb = kGHeads; hb >= 1; --hb)
    if (HG % hb == 0) return hb;
  return 1;
}

bool tc_decode_group_supported(int Q) { return Q == kGQ; }

cudaError_t tc_decode_group(const LaunchArgs& a, cudaStream_t s) {
  const GLayout L = g_layout();
  const size_t smem = L.total + 1024;
  const int HB = tc_decode_group_heads(a.H, a.G);
  const int nitems = a.nseq * (a.H / HB);
  int dev = 0, nsm = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int grid = nitems < nsm ? nitems : nsm;
  cudaError_t e;
  if (a.flags & ERS_FLAG_REPLAYSSM) {
    if ((e = cudaFuncSetAttribute(k_tc_decode_group<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    if (grid > 0) k_tc_decode_group<true><<<grid, kGThreads, smem, s>>>(a, HB, nitems);
  } else {
    if ((e = cudaFuncSetAttribute(k_tc_decode_group<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    if (grid > 0) k_tc_decode_group<false><<<grid, kGThreads, smem, s>>>(a, HB, nitems);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_setpos(a, 0, s);
}

}  // namespace ers
