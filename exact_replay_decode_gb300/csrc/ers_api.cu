// C ABI of the library (declared in include/ers.h): host-side validation, workspace carving and
// dispatch to the kernels.  A call that fails validation launches nothing.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "ers.h"
#include "ers_internal.h"

using ers::LaunchArgs;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ers_status check_ptr(const void* p, bool required) {
  if (p == nullptr) return required ? ERS_EINVAL : ERS_OK;
  return aligned16(p) ? ERS_OK : ERS_EPTR;
}

#define ERS_TRY(expr)                  \
  do {                                 \
    const ers_status st_ = (expr);     \
    if (st_ != ERS_OK) return st_;     \
  } while (0)

ers_status check_dims(const ers_dims* d) {
  if (d == nullptr) return ERS_EINVAL;
  if (d->io_dtype != ERS_DTYPE_F32 && d->io_dtype != ERS_DTYPE_BF16) return ERS_EDTYPE;
  if (d->nheads <= 0 || d->ngroups <= 0 || d->nheads % d->ngroups != 0) return ERS_ESHAPE;
  if (d->chunk < 1 || d->chunk > ers::kQMaxHost) return ERS_ESHAPE;
  if (!ers::fma_supported(d->headdim, d->dstate)) return ERS_ESHAPE;
  return ERS_OK;
}

ers_status check_params(const ers_params* p) {
  if (p == nullptr) return ERS_EINVAL;
  ERS_TRY(check_ptr(p->A, true));
  ERS_TRY(check_ptr(p->D, true));
  ERS_TRY(check_ptr(p->dt_bias, true));
  return ERS_OK;
}

// The shared NVFP4 state keeps no separate anchor: state is unused (may be NULL).
ers_status check_state_ptrs(const ers_cache* c) {
  return check_ptr(c->state, c->anchor_dtype != ERS_ANCHOR_NVFP4_SHARED_SR);
}

// FP8 and NVFP4 read copies are implemented by the CUDA-core warp-per-head kernels only.
bool narrow_read_shape(const ers_dims* d) {
  return d->headdim == 64 && d->dstate == 128 && d->chunk >= 1 && d->chunk <= 16;
}
bool has_narrow_copy(const ers_cache* c) { return c->read_copy != nullptr && c->read_dtype != ERS_READ_BF16; }
bool has_nvfp4_copy(const ers_cache* c) { return c->read_copy != nullptr && c->read_dtype == ERS_READ_NVFP4; }
bool f16_anchor(const ers_cache* c) {   // an anchor other than fp32: fp16 SR or the shared NVFP4 state
  return c->anchor_dtype == ERS_ANCHOR_F16_SR || c->anchor_dtype == ERS_ANCHOR_NVFP4_SHARED_SR;
}

// fp16 anchors and the shared NVFP4 state: ReplaySSM calls only, bf16 io, a read copy (NVFP4 for the
// shared state), the warp-per-head shapes.
ers_status check_f16_anchor(const ers_dims* d, const ers_cache* c, bool rssm) {
  if (!f16_anchor(c)) return ERS_OK;
  if (!rssm || d->io_dtype != ERS_DTYPE_BF16 || c->read_copy == nullptr || !narrow_read_shape(d))
    return ERS_EUNSUPPORTED;
  if (c->anchor_dtype == ERS_ANCHOR_NVFP4_SHARED_SR && c->read_dtype != ERS_READ_NVFP4) return ERS_EUNSUPPORTED;
  return ERS_OK;
}

ers_status check_pages(const ers_dims* d, const ers_cache* c) {
  if (c->buf_pages != nullptr && d->chunk % c->page_rows != 0) return ERS_ESHAPE;
  return ERS_OK;
}

ers_status check_cache(const ers_cache* c, bool need_read_copy) {
  if (c == nullptr || c->nslots < 0) return ERS_EINVAL;
  if (c->read_dtype != ERS_READ_BF16 && c->read_dtype != ERS_READ_FP8_E4M3 && c->read_dtype != ERS_READ_NVFP4)
    return ERS_EDTYPE;
  if (c->anchor_dtype != ERS_ANCHOR_F32 && c->anchor_dtype != ERS_ANCHOR_F16_SR &&
      c->anchor_dtype != ERS_ANCHOR_NVFP4_SHARED_SR)
    return ERS_EDTYPE;
  ERS_TRY(check_ptr(c->buf_pages, false));
  if (c->buf_pages != nullptr && (c->page_rows < 1 || c->npages < 1)) return ERS_EINVAL;
  ERS_TRY(check_state_ptrs(c));
  ERS_TRY(check_ptr(c->read_copy, need_read_copy));
  if (c->read_dtype != ERS_READ_BF16 && c->read_copy != nullptr) ERS_TRY(check_ptr(c->read_scale, true));
  if (c->read_dtype == ERS_READ_NVFP4 && c->read_copy != nullptr) ERS_TRY(check_ptr(c->read_block_scale, true));
  ERS_TRY(check_ptr(c->buf_x, true));
  ERS_TRY(check_ptr(c->buf_dt, true));
  ERS_TRY(check_ptr(c->buf_B, true));
  ERS_TRY(check_ptr(c->buf_C, true));
  ERS_TRY(check_ptr(c->pos, true));
  return ERS_OK;
}

LaunchArgs base_args(const ers_dims* d, const ers_params* p) {
  LaunchArgs a;
  memset(&a, 0, sizeof(a));
  a.H = d->nheads;
  a.G = d->ngroups;
  a.P = d->headdim;
  a.N = d->dstate;
  a.Q = d->chunk;
  a.io = d->io_dtype;
  if (p != nullptr) {
    a.A = p->A;
    a.D = p->D;
    a.dt_bias = p->dt_bias;
  }
  return a;
}

void set_cache(LaunchArgs& a, const ers_cache* c) {
  a.state = (float*)c->state;   // fp16 data when anchor_f16
  a.read_copy = c->read_copy;
  a.read_fp8 = c->read_copy != nullptr && c->read_dtype == ERS_READ_FP8_E4M3;
  a.read_nvfp4 = c->read_copy != nullptr && c->read_dtype == ERS_READ_NVFP4;
  a.read_scale = c->read_scale;
  a.read_bscale = c->read_block_scale;
  a.buf_pages = c->buf_pages;
  a.page_rows = c->buf_pages != nullptr ? c->page_rows : 1;
  a.npages = c->npages;
  a.anchor_f16 = c->anchor_dtype == ERS_ANCHOR_F16_SR;
  a.anchor_shared = c->anchor_dtype == ERS_ANCHOR_NVFP4_SHARED_SR;
  a.sr_key0 = c->sr_key[0];
  a.sr_key1 = c->sr_key[1];
  a.sr_nonce = c->sr_nonce;
  a.bx = c->buf_x;
  a.bdt = c->buf_dt;
  a.bB = c->buf_B;
  a.bC = c->buf_C;
  a.pos = c->pos;
  a.nslots = c->nslots;
}

// Prefill scratch.  CUDA-core engine: per (sequence, chunk, head) the chunk state (later the state
// at the chunk's start) and the chunk's total log-decay.  Tensor-core engine: the single-pass scan's
// chunk states, chunk end states, decay factors and look-back flags (tc_scan_workspace).
size_t prefill_workspace(const ers_dims* d, int32_t nseq, int32_t max_chunks) {
  if (ers::tc_supported(d->io_dtype, d->headdim, d->dstate, d->chunk))
    return ers::tc_scan_workspace(nseq, max_chunks, d->nheads);
  const size_t units = (size_t)(nseq > 0 ? nseq : 0) * (size_t)(max_chunks > 0 ? max_chunks : 0) * d->nheads;
  return ers::align256(units * d->headdim * d->dstate * sizeof(float)) + ers::align256(units * sizeof(float));
}

void carve_workspace(LaunchArgs& a, void* workspace) {
  if (ers::tc_supported(a.io, a.P, a.N, a.Q)) {
    ers::tc_scan_carve(a, workspace);
    return;
  }
  const size_t units = (size_t)a.nseq * (size_t)a.max_chunks * a.H;
  a.ws_states = (float*)workspace;
  a.ws_tot = (float*)((char*)workspace + ers::align256(units * a.P * a.N * sizeof(float)));
}

int32_t scan_chunks(int32_t max_seqlen, int32_t Q) { return (max_seqlen + Q - 1) / Q; }
int32_t resume_chunks(int32_t max_seqlen, int32_t Q) { return (max_seqlen + Q - 1 + Q - 1) / Q; }

ers_status finish(cudaError_t e) { return e == cudaSuccess ? ERS_OK : ERS_ECUDA; }

ers_status check_tokens(const void* x, const float* dt, const void* B, const void* C, bool required) {
  ERS_TRY(check_ptr(x, required));
  ERS_TRY(check_ptr(dt, required));
  ERS_TRY(check_ptr(B, required));
  ERS_TRY(check_ptr(C, required));
  return ERS_OK;
}

}  // namespace

extern "C" {

const char* ers_status_str(ers_status s) {
  switch (s) {
    case ERS_OK: return "ok";
    case ERS_EINVAL: return "invalid argument";
    case ERS_ESHAPE: return "unsupported dimensions";
    case ERS_EDTYPE: return "unsupported dtype";
    case ERS_EPTR: return "pointer not 16-byte aligned";
    case ERS_EALIGN: return "slot position outside its legal range";
    case ERS_EOVERFLOW: return "committed pointer plus drafts exceeds the refresh period";
    case ERS_ECOMMIT: return "accepted count outside [0, T]";
    case ERS_ESLOT: return "slot index out of range";
    case ERS_ETIMEOUT: return "bounded device wait gave up";
    case ERS_EWORKSPACE: return "workspace missing or too small";
    case ERS_ECUDA: return "CUDA launch error";
    case ERS_EUNSUPPORTED: return "unsupported request";
    default: return "unknown status";
  }
}

int32_t ers_version(void) { return 200; }

ers_status ers_selftest_bounded_wait(uint64_t limit_ns, ers_stream_t stream, int32_t* dev_status) {
  if (dev_status == nullptr || limit_ns == 0 || limit_ns > 10000000000ull) return ERS_EINVAL;
  ERS_TRY(check_ptr(dev_status, true));
  return finish(ers::wait_selftest(limit_ns, dev_status, (cudaStream_t)stream));
}

size_t ers_ssd_scan_fwd_workspace_size(const ers_dims* dims, int32_t nseq, int32_t max_seqlen) {
  if (check_dims(dims) != ERS_OK || nseq < 0 || max_seqlen < 0) return 0;
  return prefill_workspace(dims, nseq, scan_chunks(max_seqlen, dims->chunk));
}

size_t ers_chunked_prefill_workspace_size(const ers_dims* dims, int32_t nseq, int32_t max_seqlen) {
  if (check_dims(dims) != ERS_OK || nseq < 0 || max_seqlen < 0) return 0;
  return prefill_workspace(dims, nseq, resume_chunks(max_seqlen, dims->chunk));
}

ers_status ers_ssd_scan_fwd(const ers_dims* dims, const ers_params* prm, int32_t nseq, int64_t ntokens,
                            int32_t max_seqlen, const int32_t* cu_seqlens, const void* x, const float* dt,
                            const void* B, const void* C, const float* init_state, void* y,
                            float* final_state, float* chunk_states, void* workspace, size_t workspace_bytes,
                            ers_stream_t stream, int32_t* dev_status) {
  ERS_TRY(check_dims(dims));
  ERS_TRY(check_params(prm));
  if (nseq < 0 || ntokens < 0 || max_seqlen < 0) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  ERS_TRY(check_ptr(cu_seqlens, true));
  ERS_TRY(check_tokens(x, dt, B, C, ntokens > 0));
  ERS_TRY(check_ptr(y, ntokens > 0));
  ERS_TRY(check_ptr(final_state, true));
  ERS_TRY(check_ptr(init_state, false));
  ERS_TRY(check_ptr(chunk_states, false));
  ERS_TRY(check_ptr(dev_status, false));
  const int32_t mc = scan_chunks(max_seqlen, dims->chunk);
  const size_t wsz = prefill_workspace(dims, nseq, mc);
  if (wsz > 0 && (workspace == nullptr || workspace_bytes < wsz)) return ERS_EWORKSPACE;
  ERS_TRY(check_ptr(workspace, false));
  LaunchArgs a = base_args(dims, prm);
  a.x = x; a.dt = dt; a.B = B; a.C = C;
  a.cu = cu_seqlens;
  a.nseq = nseq;
  a.ntokens = ntokens;
  a.max_chunks = mc;
  a.y = y;
  a.init_state = init_state;
  a.final_state = final_state;
  a.chunk_states = chunk_states;
  carve_workspace(a, workspace);
  a.status = dev_status;
  if (ers::tc_supported(a.io, a.P, a.N, a.Q)) return finish(ers::tc_prefill(a, ers::Op::kScan, (cudaStream_t)stream));
  return finish(ers::fma_prefill(a, ers::Op::kScan, (cudaStream_t)stream));
}

ers_status ers_chunked_prefill(const ers_dims* dims, const ers_params* prm, const ers_cache* cache,
                               int32_t nseq, int64_t ntokens, int32_t max_seqlen, const int32_t* cu_seqlens,
                               const int32_t* slot, const void* x, const float* dt, const void* B,
                               const void* C, void* y, void* workspace, size_t workspace_bytes,
                               ers_stream_t stream, int32_t* dev_status) {
  ERS_TRY(check_dims(dims));
  ERS_TRY(check_params(prm));
  ERS_TRY(check_cache(cache, false));
  ERS_TRY(check_pages(dims, cache));
  if (f16_anchor(cache)) return ERS_EUNSUPPORTED;   // chunked prefill writes fp32 checkpoints
  if (nseq < 0 || ntokens < 0 || max_seqlen < 0) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  if (slot == nullptr && nseq > cache->nslots) return ERS_EINVAL;
  ERS_TRY(check_ptr(cu_seqlens, true));
  ERS_TRY(check_ptr(slot, false));
  ERS_TRY(check_tokens(x, dt, B, C, ntokens > 0));
  ERS_TRY(check_ptr(y, ntokens > 0));
  ERS_TRY(check_ptr(dev_status, false));
  const int32_t mc = resume_chunks(max_seqlen, dims->chunk);
  const size_t wsz = prefill_workspace(dims, nseq, mc);
  if (wsz > 0 && (workspace == nullptr || workspace_bytes < wsz)) return ERS_EWORKSPACE;
  ERS_TRY(check_ptr(workspace, false));
  LaunchArgs a = base_args(dims, prm);
  set_cache(a, cache);
  a.x = x; a.dt = dt; a.B = B; a.C = C;
  a.cu = cu_seqlens;
  a.slot = slot;
  a.nseq = nseq;
  a.ntokens = ntokens;
  a.max_chunks = mc;
  a.y = y;
  carve_workspace(a, workspace);
  a.status = dev_status;
  if (ers::tc_supported(a.io, a.P, a.N, a.Q))
    return finish(ers::tc_prefill(a, ers::Op::kChunkedPrefill, (cudaStream_t)stream));
  return finish(ers::fma_prefill(a, ers::Op::kChunkedPrefill, (cudaStream_t)stream));
}

ers_status ers_replay_decode(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                             const int32_t* slot, const void* x, const float* dt, const void* B, const void* C,
                             uint32_t flags, void* y, ers_stream_t stream, int32_t* dev_status) {
  ERS_TRY(check_dims(dims));
  ERS_TRY(check_params(prm));
  const bool rssm = (flags & ERS_FLAG_REPLAYSSM) != 0;
  if ((flags & ~(ERS_FLAG_FUSE_REFRESH | ERS_FLAG_REPLAYSSM)) != 0) return ERS_EINVAL;
  ERS_TRY(check_cache(cache, rssm));
  ERS_TRY(check_pages(dims, cache));
  if (nseq < 0) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  if (slot == nullptr && nseq > cache->nslots) return ERS_EINVAL;
  ERS_TRY(check_ptr(slot, false));
  ERS_TRY(check_tokens(x, dt, B, C, true));
  ERS_TRY(check_ptr(y, true));
  ERS_TRY(check_ptr(dev_status, false));
  if (has_narrow_copy(cache) && !narrow_read_shape(dims)) return ERS_EUNSUPPORTED;
  if (has_nvfp4_copy(cache) && !rssm) return ERS_EUNSUPPORTED;   // NVFP4 copies: ReplaySSM mode only
  ERS_TRY(check_f16_anchor(dims, cache, rssm));
  LaunchArgs a = base_args(dims, prm);
  set_cache(a, cache);
  a.x = x; a.dt = dt; a.B = B; a.C = C;
  a.slot = slot;
  a.nseq = nseq;
  a.flags = flags;
  a.y = y;
  a.status = dev_status;
  if (rssm && ers::rssm_tc_supported(a.io, a.P, a.N, a.Q, a.H, a.G, cache->read_dtype, cache->anchor_dtype))
    return finish(ers::rssm_tc(a, 1, true, (cudaStream_t)stream));
  const bool tc = ers::tc_supported(a.io, a.P, a.N, a.Q);
  if (rssm && (flags & ERS_FLAG_FUSE_REFRESH) && (tc || !ers::heads_decode_supported(a.P, a.N, a.Q))) {
    // engines without the fused flush: the flush rule for one token (ers_refresh with T = 1), then
    // the plain ReplaySSM decode; the warp-per-head kernel does both in one launch, same bits
    LaunchArgs r = a;
    r.flags = ERS_FLAG_REPLAYSSM;
    r.T = 1;
    const cudaError_t e = tc ? ers::tc_refresh(r, (cudaStream_t)stream) : ers::fma_refresh(r, (cudaStream_t)stream);
    if (e != cudaSuccess) return finish(e);
    a.flags = ERS_FLAG_REPLAYSSM;
  }
  if (tc) return finish(ers::tc_decode(a, (cudaStream_t)stream));
  return finish(ers::fma_decode(a, (cudaStream_t)stream));
}

ers_status ers_refresh(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                       const int32_t* slot, uint32_t flags, int32_t drafts_T, ers_stream_t stream,
                       int32_t* dev_status) {
  ERS_TRY(check_dims(dims));
  ERS_TRY(check_params(prm));
  if ((flags & ~ERS_FLAG_REPLAYSSM) != 0) return ERS_EINVAL;
  ERS_TRY(check_cache(cache, false));
  ERS_TRY(check_pages(dims, cache));
  if (nseq < 0 || drafts_T < 0) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  if (slot == nullptr && nseq > cache->nslots) return ERS_EINVAL;
  ERS_TRY(check_ptr(slot, false));
  ERS_TRY(check_ptr(dev_status, false));
  if (has_narrow_copy(cache) && !narrow_read_shape(dims)) return ERS_EUNSUPPORTED;
  if (has_nvfp4_copy(cache) && !(flags & ERS_FLAG_REPLAYSSM)) return ERS_EUNSUPPORTED;
  ERS_TRY(check_f16_anchor(dims, cache, (flags & ERS_FLAG_REPLAYSSM) != 0));
  LaunchArgs a = base_args(dims, prm);
  set_cache(a, cache);
  a.slot = slot;
  a.nseq = nseq;
  a.flags = flags;
  a.T = drafts_T;
  a.status = dev_status;
  if (ers::tc_supported(a.io, a.P, a.N, a.Q)) return finish(ers::tc_refresh(a, (cudaStream_t)stream));
  return finish(ers::fma_refresh(a, (cudaStream_t)stream));
}

ers_status ers_spec_verify(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                           const int32_t* slot, int32_t T, const void* x, const float* dt, const void* B,
                           const void* C, uint32_t flags, void* y, ers_stream_t stream, int32_t* dev_status) {
  ERS_TRY(check_dims(dims));
  ERS_TRY(check_params(prm));
  if ((flags & ~ERS_FLAG_AUTO_FLUSH) != 0) return ERS_EINVAL;
  ERS_TRY(check_cache(cache, true));
  ERS_TRY(check_pages(dims, cache));
  if (nseq < 0 || T < 1 || T > dims->chunk) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  if (slot == nullptr && nseq > cache->nslots) return ERS_EINVAL;
  ERS_TRY(check_ptr(slot, false));
  ERS_TRY(check_tokens(x, dt, B, C, true));
  ERS_TRY(check_ptr(y, true));
  ERS_TRY(check_ptr(dev_status, false));
  const bool rssm_tc = ers::rssm_tc_supported(dims->io_dtype, dims->headdim, dims->dstate, dims->chunk, dims->nheads,
                                              dims->ngroups, cache->read_dtype, cache->anchor_dtype);
  if ((has_narrow_copy(cache) || f16_anchor(cache)) && !rssm_tc &&
      !(narrow_read_shape(dims) && ers::heads_verify_supported(dims->headdim, dims->dstate, dims->chunk, T,
                                                               dims->nheads, dims->ngroups)))
    return ERS_EUNSUPPORTED;
  ERS_TRY(check_f16_anchor(dims, cache, true));
  LaunchArgs a = base_args(dims, prm);
  set_cache(a, cache);
  a.x = x; a.dt = dt; a.B = B; a.C = C;
  a.slot = slot;
  a.nseq = nseq;
  a.T = T;
  a.flags = flags;
  a.y = y;
  a.status = dev_status;
  if (rssm_tc) return finish(ers::rssm_tc(a, T, false, (cudaStream_t)stream));
  if (ers::tc_supported(a.io, a.P, a.N, a.Q)) return finish(ers::tc_verify(a, (cudaStream_t)stream));
  return finish(ers::fma_verify(a, (cudaStream_t)stream));
}

ers_status ers_commit(const ers_dims* dims, const ers_cache* cache, int32_t nseq, const int32_t* slot,
                      const int32_t* accepted, int32_t T, uint32_t flags, ers_stream_t stream,
                      int32_t* dev_status) {
  ERS_TRY(check_dims(dims));
  if ((flags & ~ERS_FLAG_AUTO_FLUSH) != 0) return ERS_EINVAL;
  if (cache == nullptr || cache->nslots < 0) return ERS_EINVAL;
  ERS_TRY(check_ptr(cache->pos, true));
  if (nseq < 0 || T < 1 || T > dims->chunk) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  if (slot == nullptr && nseq > cache->nslots) return ERS_EINVAL;
  ERS_TRY(check_ptr(slot, false));
  ERS_TRY(check_ptr(accepted, true));
  ERS_TRY(check_ptr(dev_status, false));
  LaunchArgs a = base_args(dims, nullptr);
  a.pos = cache->pos;
  a.nslots = cache->nslots;
  a.slot = slot;
  a.nseq = nseq;
  a.accepted = accepted;
  a.T = T;
  a.flags = flags;
  a.status = dev_status;
  return finish(ers::launch_commit(a, (cudaStream_t)stream));
}

}  // extern "C"

// ---- exact-mode speculative decode -----------------------------------------------------------
namespace {
struct ExactSpecWs {
  size_t st, bx, bdt, bB, bC, pos, x1, dt1, B1, C1, y1, total;
};
ExactSpecWs exact_spec_ws(const ers_dims* d, int32_t nseq) {
  ExactSpecWs w;
  const size_t S = (size_t)(nseq > 0 ? nseq : 0), es = d->io_dtype == ERS_DTYPE_BF16 ? 2 : 4;
  const size_t HP = (size_t)d->nheads * d->headdim, GN = (size_t)d->ngroups * d->dstate, Q = (size_t)d->chunk;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += ers::align256(bytes);
    return o;
  };
  w.st = take(S * HP * d->dstate * sizeof(float));
  w.bx = take(S * Q * HP * es);
  w.bdt = take(S * Q * d->nheads * sizeof(float));
  w.bB = take(S * Q * GN * es);
  w.bC = take(S * Q * GN * es);
  w.pos = take(S * sizeof(int32_t));
  w.x1 = take(S * HP * es);
  w.dt1 = take(S * d->nheads * sizeof(float));
  w.B1 = take(S * GN * es);
  w.C1 = take(S * GN * es);
  w.y1 = take(S * HP * es);
  w.total = off;
  return w;
}

ers_status check_exact_spec(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                            const int32_t* slot, int32_t T, const void* x, const float* dt, const void* B,
                            const void* C, int32_t* dev_status) {
  ERS_TRY(check_dims(dims));
  ERS_TRY(check_params(prm));
  ERS_TRY(check_cache(cache, false));
  ERS_TRY(check_pages(dims, cache));
  if (cache->anchor_dtype != ERS_ANCHOR_F32 || cache->state == nullptr) return ERS_EUNSUPPORTED;
  if (has_nvfp4_copy(cache)) return ERS_EUNSUPPORTED;   // NVFP4 copies are kept in ReplaySSM mode only
  if (has_narrow_copy(cache) && !narrow_read_shape(dims)) return ERS_EUNSUPPORTED;
  if (nseq < 0 || T < 1 || T > dims->chunk) return ERS_EINVAL;
  if (nseq > 0 && slot == nullptr && nseq > cache->nslots) return ERS_EINVAL;
  ERS_TRY(check_ptr(slot, false));
  ERS_TRY(check_tokens(x, dt, B, C, nseq > 0));
  ERS_TRY(check_ptr(dev_status, false));
  return ERS_OK;
}
}  // namespace

extern "C" {

size_t ers_spec_verify_exact_workspace_size(const ers_dims* dims, int32_t nseq) {
  if (check_dims(dims) != ERS_OK || nseq < 0) return 0;
  return exact_spec_ws(dims, nseq).total;
}

ers_status ers_spec_verify_exact(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                                 const int32_t* slot, int32_t T, const void* x, const float* dt, const void* B,
                                 const void* C, void* y, void* workspace, size_t workspace_bytes, ers_stream_t stream,
                                 int32_t* dev_status) {
  ERS_TRY(check_exact_spec(dims, prm, cache, nseq, slot, T, x, dt, B, C, dev_status));
  if (nseq == 0) return ERS_OK;
  ERS_TRY(check_ptr(y, true));
  const ExactSpecWs w = exact_spec_ws(dims, nseq);
  if (workspace == nullptr || workspace_bytes < w.total) return ERS_EWORKSPACE;
  ERS_TRY(check_ptr(workspace, true));
  const cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  LaunchArgs a = base_args(dims, prm);
  set_cache(a, cache);
  a.slot = slot;
  a.nseq = nseq;
  a.T = T;
  a.status = dev_status;
  if (ers::exact_verify_supported(a.io, a.P, a.N, a.Q, T, a.H, a.G) && !ers::tc_supported(a.io, a.P, a.N, a.Q)) {
    // one pass over the checkpoints (the workspace is not used)
    a.x = x; a.dt = dt; a.B = B; a.C = C;
    a.y = y;
    return finish(ers::exact_verify(a, s));
  }
  cudaError_t e = ers::launch_spec_snapshot(a, (float*)(ws + w.st), ws + w.bx, (float*)(ws + w.bdt), ws + w.bB,
                                            ws + w.bC, (int32_t*)(ws + w.pos), s);
  if (e != cudaSuccess) return finish(e);
  // the shadow cache: slot i of the workspace, contiguous buffers, exact-mode decode with refresh
  LaunchArgs d = base_args(dims, prm);
  d.state = (float*)(ws + w.st);
  d.bx = ws + w.bx;
  d.bdt = (float*)(ws + w.bdt);
  d.bB = ws + w.bB;
  d.bC = ws + w.bC;
  d.pos = (int32_t*)(ws + w.pos);
  d.nslots = nseq;
  d.page_rows = 1;
  d.nseq = nseq;
  d.flags = ERS_FLAG_FUSE_REFRESH;
  d.x = ws + w.x1;
  d.dt = (float*)(ws + w.dt1);
  d.B = ws + w.B1;
  d.C = ws + w.C1;
  d.y = ws + w.y1;
  d.status = dev_status;
  const bool tc = ers::tc_supported(d.io, d.P, d.N, d.Q);
  for (int j = 0; j < T; ++j) {
    if ((e = ers::launch_spec_rows(a, j, 0, x, dt, B, C, (void*)d.x, (float*)d.dt, (void*)d.B, (void*)d.C, nullptr,
                                   nullptr, s)) != cudaSuccess)
      return finish(e);
    if ((e = tc ? ers::tc_decode(d, s) : ers::fma_decode(d, s)) != cudaSuccess) return finish(e);
    if ((e = ers::launch_spec_rows(a, j, 1, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, y,
                                   d.y, s)) != cudaSuccess)
      return finish(e);
  }
  return ERS_OK;
}

ers_status ers_commit_exact(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                            const int32_t* slot, const int32_t* accepted, int32_t T, const void* x, const float* dt,
                            const void* B, const void* C, void* workspace, size_t workspace_bytes, ers_stream_t stream,
                            int32_t* dev_status) {
  ERS_TRY(check_exact_spec(dims, prm, cache, nseq, slot, T, x, dt, B, C, dev_status));
  if (nseq == 0) return ERS_OK;
  ERS_TRY(check_ptr(accepted, true));
  if (workspace == nullptr || workspace_bytes < ers::align256((size_t)nseq * sizeof(int32_t))) return ERS_EWORKSPACE;
  ERS_TRY(check_ptr(workspace, true));
  const cudaStream_t s = (cudaStream_t)stream;
  LaunchArgs a = base_args(dims, prm);
  set_cache(a, cache);
  a.slot = slot;
  a.nseq = nseq;
  a.T = T;
  a.accepted = accepted;
  a.x = x; a.dt = dt; a.B = B; a.C = C;
  a.status = dev_status;
  int32_t* old_pos = (int32_t*)workspace;
  cudaError_t e = ers::launch_commit_exact(a, 0, old_pos, s);
  if (e != cudaSuccess) return finish(e);
  LaunchArgs r = a;   // the chunks the accepted drafts filled: the exact-mode refresh (pos == Q)
  r.flags = 0;
  r.x = r.dt = nullptr;
  r.B = r.C = nullptr;
  if ((e = ers::tc_supported(r.io, r.P, r.N, r.Q) ? ers::tc_refresh(r, s) : ers::fma_refresh(r, s)) != cudaSuccess)
    return finish(e);
  return finish(ers::launch_commit_exact(a, 1, old_pos, s));
}

}  // extern "C"

extern "C" {

ers_status ers_ssu_update(const ers_dims* dims, const ers_params* prm, float* state, int32_t nslots,
                          int32_t nseq, const int32_t* slot, const void* x, const float* dt, const void* B,
                          const void* C, void* y, ers_stream_t stream, int32_t* dev_status) {
  ERS_TRY(check_dims(dims));
  ERS_TRY(check_params(prm));
  if (!ers::ssu_supported(dims->headdim, dims->dstate)) return ERS_ESHAPE;
  if (nseq < 0 || nslots < 0) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  if (slot == nullptr && nseq > nslots) return ERS_EINVAL;
  ERS_TRY(check_ptr(state, true));
  ERS_TRY(check_ptr(slot, false));
  ERS_TRY(check_tokens(x, dt, B, C, true));
  ERS_TRY(check_ptr(y, true));
  ERS_TRY(check_ptr(dev_status, false));
  LaunchArgs a = base_args(dims, prm);
  a.state = state;
  a.nslots = nslots;
  a.slot = slot;
  a.nseq = nseq;
  a.x = x; a.dt = dt; a.B = B; a.C = C;
  a.y = y;
  a.status = dev_status;
  return finish(ers::ssu_update(a, (cudaStream_t)stream));
}

namespace {
ers_status check_gdn(const ers_gdn_dims* d, const ers_gdn_cache* c, int32_t nseq, const int32_t* slot, int32_t T) {
  if (d == nullptr || c == nullptr) return ERS_EINVAL;
  if (d->io_dtype != ERS_DTYPE_F32 && d->io_dtype != ERS_DTYPE_BF16) return ERS_EDTYPE;
  if (d->nheads <= 0 || d->ngroups <= 0 || d->nheads % d->ngroups != 0) return ERS_ESHAPE;
  if (!ers::gdn_supported(d->dk, d->dv, d->window, T)) return ERS_ESHAPE;
  if (nseq < 0 || c->nslots < 0) return ERS_EINVAL;
  if (slot == nullptr && nseq > c->nslots) return ERS_EINVAL;
  ERS_TRY(check_ptr(c->anchor, true));
  ERS_TRY(check_ptr(c->read_copy, true));
  ERS_TRY(check_ptr(c->buf_k, true));
  ERS_TRY(check_ptr(c->buf_v, true));
  ERS_TRY(check_ptr(c->buf_g, true));
  ERS_TRY(check_ptr(c->buf_beta, true));
  ERS_TRY(check_ptr(c->buf_u, true));
  ERS_TRY(check_ptr(c->pos, true));
  ERS_TRY(check_ptr(slot, false));
  return ERS_OK;
}

ers::GdnArgs gdn_args(const ers_gdn_dims* d, const ers_gdn_cache* c, int32_t nseq, const int32_t* slot, int32_t T,
                      uint32_t flags, int32_t* st) {
  ers::GdnArgs a;
  memset(&a, 0, sizeof(a));
  a.H = d->nheads;
  a.G = d->ngroups;
  a.L = d->window;
  a.io = d->io_dtype;
  a.T = T;
  a.nseq = nseq;
  a.nslots = c->nslots;
  a.flags = flags;
  a.slot = slot;
  a.anchor = c->anchor;
  a.copy = c->read_copy;
  a.bk = c->buf_k;
  a.bv = c->buf_v;
  a.bg = c->buf_g;
  a.bbeta = c->buf_beta;
  a.bu = c->buf_u;
  a.pos = c->pos;
  a.status = st;
  return a;
}

ers_status check_conv(const ers_conv_dims* d) {
  if (d == nullptr) return ERS_EINVAL;
  if (d->io_dtype != ERS_DTYPE_F32 && d->io_dtype != ERS_DTYPE_BF16) return ERS_EDTYPE;
  if (d->channels <= 0 || d->channels % 8 != 0 || d->width < 2 || d->width > 4) return ERS_ESHAPE;
  if ((d->flags & ~ERS_CONV_SILU) != 0) return ERS_EINVAL;
  return ERS_OK;
}

ers::ConvLaunch conv_launch(const ers_conv_dims* d) {
  ers::ConvLaunch l;
  memset(&l, 0, sizeof(l));
  l.C = d->channels;
  l.W = d->width;
  l.io = d->io_dtype;
  l.silu = (d->flags & ERS_CONV_SILU) != 0;
  return l;
}
}  // namespace

ers_status ers_gdn_verify(const ers_gdn_dims* dims, const ers_gdn_cache* cache, int32_t nseq, const int32_t* slot,
                          int32_t T, const void* q, const void* k, const void* v, const float* g, const float* beta,
                          uint32_t flags, void* o, ers_stream_t stream, int32_t* dev_status) {
  if (T < 1) return ERS_EINVAL;
  ERS_TRY(check_gdn(dims, cache, nseq, slot, T));
  if (T > dims->window) return ERS_EINVAL;   // the drafts must fit the buffer after a flush
  if ((flags & ~ERS_FLAG_AUTO_FLUSH) != 0) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  ERS_TRY(check_ptr(q, true));
  ERS_TRY(check_ptr(k, true));
  ERS_TRY(check_ptr(v, true));
  ERS_TRY(check_ptr(g, true));
  ERS_TRY(check_ptr(beta, true));
  ERS_TRY(check_ptr(o, true));
  ERS_TRY(check_ptr(dev_status, false));
  ers::GdnArgs a = gdn_args(dims, cache, nseq, slot, T, flags, dev_status);
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.o = o;
  return finish(ers::gdn_launch(a, 0, nullptr, (cudaStream_t)stream));
}

ers_status ers_gdn_commit(const ers_gdn_dims* dims, const ers_gdn_cache* cache, int32_t nseq, const int32_t* slot,
                          const int32_t* accepted, int32_t T, uint32_t flags, ers_stream_t stream,
                          int32_t* dev_status) {
  if (T < 1) return ERS_EINVAL;
  ERS_TRY(check_gdn(dims, cache, nseq, slot, T));
  if (T > dims->window) return ERS_EINVAL;
  if ((flags & ~ERS_FLAG_AUTO_FLUSH) != 0) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  ERS_TRY(check_ptr(accepted, true));
  ERS_TRY(check_ptr(dev_status, false));
  ers::GdnArgs a = gdn_args(dims, cache, nseq, slot, T, flags, dev_status);
  return finish(ers::gdn_launch(a, 2, accepted, (cudaStream_t)stream));
}

ers_status ers_gdn_refresh(const ers_gdn_dims* dims, const ers_gdn_cache* cache, int32_t nseq, const int32_t* slot,
                           int32_t drafts_T, ers_stream_t stream, int32_t* dev_status) {
  if (drafts_T < 0) return ERS_EINVAL;
  ERS_TRY(check_gdn(dims, cache, nseq, slot, 0));
  if (nseq == 0) return ERS_OK;
  ERS_TRY(check_ptr(dev_status, false));
  ers::GdnArgs a = gdn_args(dims, cache, nseq, slot, drafts_T, 0, dev_status);
  return finish(ers::gdn_launch(a, 1, nullptr, (cudaStream_t)stream));
}

ers_status ers_conv1d_fwd(const ers_conv_dims* dims, int32_t nseq, int64_t ntokens, int32_t max_seqlen,
                          const int32_t* cu_seqlens, const void* x, const void* weight, const void* bias,
                          void* conv_state, int32_t nslots, const int32_t* slot, int32_t read_state, void* y,
                          ers_stream_t stream, int32_t* dev_status) {
  ERS_TRY(check_conv(dims));
  if (nseq < 0 || ntokens < 0 || max_seqlen < 0 || nslots < 0) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  ERS_TRY(check_ptr(cu_seqlens, true));
  ERS_TRY(check_ptr(x, ntokens > 0));
  ERS_TRY(check_ptr(y, ntokens > 0));
  ERS_TRY(check_ptr(weight, true));
  ERS_TRY(check_ptr(bias, false));
  ERS_TRY(check_ptr(conv_state, read_state != 0));
  ERS_TRY(check_ptr(slot, false));
  ERS_TRY(check_ptr(dev_status, false));
  if (conv_state != nullptr && slot == nullptr && nseq > nslots) return ERS_EINVAL;
  ers::ConvLaunch l = conv_launch(dims);
  l.nseq = nseq;
  l.nslots = conv_state != nullptr ? nslots : 0;
  l.read_state = read_state != 0;
  l.update = 0;
  l.max_seqlen = max_seqlen;
  l.cu = cu_seqlens;
  l.slot = slot;
  l.x = x;
  l.w = weight;
  l.bias = bias;
  l.state = conv_state;
  l.y = y;
  l.status = dev_status;
  return finish(ers::conv1d(l, (cudaStream_t)stream));
}

ers_status ers_conv1d_update(const ers_conv_dims* dims, int32_t nseq, const void* x, const void* weight,
                             const void* bias, void* conv_state, int32_t nslots, const int32_t* slot, void* y,
                             ers_stream_t stream, int32_t* dev_status) {
  ERS_TRY(check_conv(dims));
  if (nseq < 0 || nslots < 0) return ERS_EINVAL;
  if (nseq == 0) return ERS_OK;
  ERS_TRY(check_ptr(x, true));
  ERS_TRY(check_ptr(y, true));
  ERS_TRY(check_ptr(weight, true));
  ERS_TRY(check_ptr(bias, false));
  ERS_TRY(check_ptr(conv_state, true));
  ERS_TRY(check_ptr(slot, false));
  ERS_TRY(check_ptr(dev_status, false));
  if (slot == nullptr && nseq > nslots) return ERS_EINVAL;
  ers::ConvLaunch l = conv_launch(dims);
  l.nseq = nseq;
  l.nslots = nslots;
  l.update = 1;
  l.slot = slot;
  l.x = x;
  l.w = weight;
  l.bias = bias;
  l.state = conv_state;
  l.y = y;
  l.status = dev_status;
  return finish(ers::conv1d(l, (cudaStream_t)stream));
}

}  // extern "C"

// ---- scan with library-owned scratch ------------------------------------------------------------
// Scratch of ers_ssd_scan_fwd_static, for callers that cannot pass a workspace (see include/ers.h).
// A file-scope device array: it exists once per device context, sized at build time, and no byte
// of it needs an initial value.
static __device__ __align__(256) unsigned char ers_scan_scratch[ERS_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxScratchDevices = 64;
std::mutex scratch_mu;
struct ScratchEntry {
  unsigned long long ctx_id;   // cuCtxGetId of the context the address belongs to (0: none yet)
  void* addr;
};
ScratchEntry scratch_cache[kMaxScratchDevices];

typedef int (*CtxGetCurrentFn)(void**);
typedef int (*CtxGetIdFn)(void*, unsigned long long*);

// Process-unique id of the calling thread's current context (cuCtxGetCurrent + cuCtxGetId, reached
// through the runtime's driver entry points so that the library needs no link against the driver),
// or 0 when there is none or the driver cannot say.
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    looked_up = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
    cudaGetLastError();
  }
  if (get_current == nullptr || get_id == nullptr) return 0;
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != 0 || ctx == nullptr || get_id(ctx, &id) != 0) return 0;
  return id;
}

// Address of ers_scan_scratch in the current device's current context.  The address is looked up
// with that device current (cudaGetSymbolAddress) and cached together with the context's id; a
// different context on the same device (after cudaDeviceReset, or a context the caller made
// current) has its own copy of the array, so a changed id triggers a fresh lookup.
ers_status static_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ERS_ECUDA;
  }
  if (dev < 0 || dev >= kMaxScratchDevices) return ERS_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(scratch_mu);
  ScratchEntry& e = scratch_cache[dev];
  const unsigned long long id = current_ctx_id();
  if (e.addr == nullptr || id == 0 || e.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, ers_scan_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ERS_ECUDA;
    }
    e.addr = p;
    e.ctx_id = current_ctx_id();   // the lookup may have created the primary context
  }
  *out = e.addr;
  return ERS_OK;
}
}  // namespace

extern "C" {

ers_status ers_ssd_scan_fwd_static(const ers_dims* dims, const ers_params* prm, int32_t nseq, int64_t ntokens,
                                   int32_t max_seqlen, const int32_t* cu_seqlens, const void* x, const float* dt,
                                   const void* B, const void* C, const float* init_state, void* y,
                                   float* final_state, float* chunk_states, ers_stream_t stream,
                                   int32_t* dev_status) {
  void* scratch = nullptr;
  if (nseq > 0) ERS_TRY(static_scratch(&scratch));   // an empty or invalid count needs no scratch
  return ers_ssd_scan_fwd(dims, prm, nseq, ntokens, max_seqlen, cu_seqlens, x, dt, B, C, init_state, y,
                          final_state, chunk_states, scratch, ERS_STATIC_SCRATCH_BYTES, stream, dev_status);
}

}  // extern "C"
