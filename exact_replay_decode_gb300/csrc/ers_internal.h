// Internal launch interface between the C-ABI layer (ers_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ers.h"

namespace ers {

constexpr int kQMaxHost = 256;  // largest chunk / refresh period (matches kQMax in ers_common.cuh)

// Everything one launch needs; unused pointers are NULL.
struct LaunchArgs {
  // dims
  int H, G, P, N, Q;
  int io;  // ERS_DTYPE_*
  // per-head parameters
  const float* A;
  const float* D;
  const float* dt_bias;
  // packed token inputs (prefill: [ntokens, ...]; decode: [nseq, ...]; verify: [nseq, T, ...])
  const void* x;
  const float* dt;
  const void* B;
  const void* C;
  const int32_t* cu;  // prefill: [nseq+1]
  int nseq;
  int max_chunks;     // prefill grid bound
  int T;              // verify: drafts per sequence; refresh: flush-rule T
  uint32_t flags;
  // cache
  float* state;
  void* read_copy;
  int read_fp8;        // read copy is FP8 e4m3 with per-row scales (read_scale [nslots, H, P])
  int read_nvfp4;      // read copy is NVFP4: e2m1 codes, e4m3 block scales (read_bscale), row scales
  float* read_scale;
  uint8_t* read_bscale;   // NVFP4 block scales [nslots, H, P, N / 16]
  int anchor_f16;         // ReplaySSM anchor stored as fp16 (state points to __half), written by SR
  int anchor_shared;      // ReplaySSM: the NVFP4 read copy is the only state (state unused), written by SR
  uint32_t sr_key0, sr_key1, sr_nonce;   // counter-based random words for the SR writes
  void* bx;
  float* bdt;
  void* bB;
  void* bC;
  int32_t* pos;
  const int32_t* slot;
  int nslots;
  // paged partial-chunk buffers: row r of slot s is buffer row buf_pages[s][r / page_rows] *
  // page_rows + r % page_rows (buffers hold npages * page_rows rows); contiguous when null
  const int32_t* buf_pages;
  int page_rows, npages;
  // outputs / plain-scan state
  void* y;
  const float* init_state;
  float* final_state;
  float* chunk_states;
  long long ntokens;  // prefill: rows of the packed token tensors
  // workspace
  float* ws_states;  // [nseq, max_chunks, H, P, N]: chunk states (CUDA cores: the start states after the chain)
  float* ws_tot;     // [nseq, max_chunks, H]: chunk log-decay (CUDA cores) or decay factor (tensor cores)
  float* ws_incl;    // tensor cores: [nseq, max_chunks, H, P, N] end state of each chunk, for the look-back
  int32_t* ws_flags; // tensor cores: [nseq, max_chunks, H] 0 / 1 (chunk state published) / 2 (end state too)
  unsigned long long wait_ns;   // limit of every bounded device wait (0: the default, 1 s)
  int part;                     // a ReplaySSM call that may flush, split in two launches: kPart*
  const int32_t* accepted;
  int32_t* status;
};

enum class Op { kScan, kChunkedPrefill };

// A ReplaySSM decode or verify that may flush runs as two launches so that the long flushing CTAs
// overlap the others instead of trailing them: kPartFlushes (the flushing slots; every CTA reads its
// position, then lets the dependent launch start; no position is written) and kPartPlain (launched as
// its programmatic dependent: the other slots and every position advance; its last CTA waits for the
// first launch, so the pair completes together).  kPartAll: one launch does everything.
enum : int { kPartAll = 0, kPartFlushes = 1, kPartPlain = 2 };

// FMA (CUDA-core) engine, ers_fma.cu
cudaError_t fma_prefill(const LaunchArgs& a, Op op, cudaStream_t s);
cudaError_t fma_decode(const LaunchArgs& a, cudaStream_t s);
cudaError_t fma_refresh(const LaunchArgs& a, cudaStream_t s);
cudaError_t fma_verify(const LaunchArgs& a, cudaStream_t s);
bool fma_supported(int P, int N);

// warp-per-head replay decode of the CUDA-core engine (chunk <= 32, P = 64, N = 128), ers_decode.cu
bool heads_decode_supported(int P, int N, int Q);
cudaError_t heads_decode(const LaunchArgs& a, cudaStream_t s);
// FP8 read-copy recast after a refresh (P = 64, N = 128), ers_decode.cu
// standalone refresh on the warp-per-head layout (P = 64, N = 128, chunk <= 32), ers_decode.cu
cudaError_t heads_refresh(const LaunchArgs& a, cudaStream_t s);
// warp-per-head speculative verify (chunk <= 16, P = 64, N = 128, T <= 4, H/G <= 8), ers_verify.cu
bool heads_verify_supported(int P, int N, int Q, int T, int H, int G);
// exact-mode speculative verify in one pass over the checkpoints (chunk <= 16, P = 64, N = 128,
// T <= 4, H/G <= 8; the chunk fold of drafts past the boundary formed row by row), ers_verify.cu
bool exact_verify_supported(int io, int P, int N, int Q, int T, int H, int G);
cudaError_t exact_verify(const LaunchArgs& a, cudaStream_t s);
cudaError_t heads_verify(const LaunchArgs& a, cudaStream_t s);

// ReplaySSM decode (T = 1, position advance, fused flush) and verify of T <= L drafts with the read
// copy's products on the tensor core (bf16 io and read copy, fp32 or fp16 anchors, P = 64, N = 128,
// L <= 16, H/G <= 8), ers_rssm_tc.cu.  Both calls run the same kernel, so verify outputs keep
// decode's bits; every other configuration runs decode and verify on the CUDA-core kernels.
bool rssm_tc_supported(int io, int P, int N, int Q, int H, int G, int read_dtype, int anchor_dtype);
cudaError_t rssm_tc(const LaunchArgs& a, int T, bool decode, cudaStream_t s);

// pointer-only kernels, ers_fma.cu
cudaError_t launch_setpos(const LaunchArgs& a, int kind, cudaStream_t s);  // kind: 0 decode, 1 refresh
cudaError_t launch_commit(const LaunchArgs& a, cudaStream_t s);
cudaError_t launch_tail(const LaunchArgs& a, cudaStream_t s);
// exact-mode speculative decode: shadow snapshot of slots, draft rows in / outputs out, commit parts
cudaError_t launch_spec_snapshot(const LaunchArgs& a, float* st, void* bx, float* bdt, void* bB, void* bC, int32_t* pos,
                                 cudaStream_t s);
cudaError_t launch_spec_rows(const LaunchArgs& a, int j, int dir, const void* x, const float* dt, const void* B,
                             const void* C, void* x1, float* dt1, void* B1, void* C1, void* y, const void* y1,
                             cudaStream_t s);
cudaError_t launch_commit_exact(const LaunchArgs& a, int part, int32_t* old_pos, cudaStream_t s);

// tensor-core engine (bf16 io, P = 64, N = 128, Q % 16 == 0, Q >= kTcMinChunk), ers_tc.cu.  Each
// configuration runs every path on ONE engine (bitwise identity needs identical arithmetic):
// chunks of at least kTcMinChunk tokens make the intra-chunk products dense enough for the tensor
// cores; below that a decode step is a bandwidth-bound matrix-vector product and the CUDA-core
// engine defines the arithmetic.
constexpr int kTcMinChunk = 64;
bool tc_supported(int io, int P, int N, int Q);
cudaError_t tc_prefill(const LaunchArgs& a, Op op, cudaStream_t s);   // single-pass scan, ers_tc_scan.cu
size_t tc_scan_workspace(int nseq, int max_chunks, int H);               // its workspace bytes
void tc_scan_carve(LaunchArgs& a, void* workspace);                      // and layout
// a 2-CTA launch whose bounded waits (an mbarrier, a flag) are never satisfied, ers_tc_scan.cu
cudaError_t wait_selftest(unsigned long long limit_ns, int32_t* status, cudaStream_t s);
cudaError_t tc_decode(const LaunchArgs& a, cudaStream_t s);
cudaError_t tc_refresh(const LaunchArgs& a, cudaStream_t s);
cudaError_t tc_verify(const LaunchArgs& a, cudaStream_t s);

// SSU baseline, ers_ssu.cu
cudaError_t ssu_update(const LaunchArgs& a, cudaStream_t s);
bool ssu_supported(int P, int N);

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// gated delta rule (GDN) verify / refresh / commit, ers_gdn.cu
struct GdnArgs {
  int H, G, L, io, T, nseq, nslots;
  uint32_t flags;
  const int32_t* slot;
  float* anchor;   // [nslots, H, dv, dk]
  void* copy;      // bf16, same shape
  void* bk;        // [nslots, L, G, dk] io
  void* bv;        // [nslots, L, H, dv] io
  float* bg;       // [nslots, L, H]
  float* bbeta;    // [nslots, L, H]
  float* bu;       // [nslots, L, H, dv] fp32 residuals
  int32_t* pos;
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  void* o;
  int32_t* status;
};
bool gdn_supported(int dk, int dv, int L, int T);
cudaError_t gdn_launch(const GdnArgs& a, int kind, const int32_t* accepted, cudaStream_t s);   // 0 verify, 1 refresh, 2 commit

// causal depthwise conv1d with a conv state, ers_conv.cu
struct ConvLaunch {
  int C, W, io, silu, nseq, nslots, read_state, update, max_seqlen;
  const int32_t* cu;
  const int32_t* slot;
  const void* x;
  const void* w;
  const void* bias;
  void* state;
  void* y;
  int32_t* status;
};
cudaError_t conv1d(const ConvLaunch& l, cudaStream_t s);

}  // namespace ers
