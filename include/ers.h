/*
 * ers.h — C ABI of the exact-replay SSD library (Mamba2 selective state space,
 * hand-written CUDA for sm_103a / GB300).
 *
 * The operations follow two sources:
 *  - "[RFC] Mamba2: exact-replay decode so that prefill, chunked prefill and
 *    decode produce identical bits" (vLLM issue 55524), section 3 "Proposal":
 *    per sequence an fp32 boundary state at the last multiple of the chunk size
 *    plus a partial-chunk buffer of (x, raw dt, B, C); decode replays the buffer
 *    from the boundary state; any prefill/chunked prefill starts at the boundary.
 *  - The ReplaySSM reproduction notes (arXiv 2610.13778), "Motivation and
 *    method" and "Core equations": periodic refresh of a checkpoint from
 *    buffered inputs, output-only speculative verification, commit that moves
 *    only the committed-input pointer, and a fp32 recurrence anchor with a
 *    separately cast low-precision read copy.
 *
 * Per head h (group g = h / (H/G)), with delta = softplus(dt + dt_bias):
 *     S_t = exp(delta_t A[h]) S_{t-1} + delta_t x_t B_t^T      (S is [P x N])
 *     y_t = S_t C_t + D[h] x_t
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers to caller-owned, densely packed
 *    row-major memory with the shapes given below.  The library takes no strides
 *    (there are no stride descriptors and no stride status code): a caller holding
 *    a strided view copies it to a dense buffer first.  The library keeps no pointer
 *    after a call returns and allocates no device or host memory.  Scratch
 *    memory, where needed, is a caller buffer sized by the matching
 *    *_workspace_size query.
 *  - Dtypes: x, B, C, y and the partial-chunk buffers x/B/C use dims->io_dtype
 *    (ERS_DTYPE_BF16 or ERS_DTYPE_F32, the same for all of them); dt, A, D,
 *    dt_bias and every recurrence state are fp32 (a ReplaySSM anchor may be
 *    fp16, see ers_cache); the read copy is bf16, FP8 or NVFP4; index arrays are
 *    int32.  Every pointer must be 16-byte aligned.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream).  Host
 *    validation runs first; a call that returns an error has launched nothing.
 *  - Errors the host cannot see (slot positions, slot indices, accepted counts,
 *    a bounded device wait that gave up) are reported through `dev_status`, a
 *    device int32 that the caller zeroes and reads back after synchronising; the
 *    first error wins.  It may be NULL, in which case such errors are dropped
 *    (the affected sequence's outputs are left unwritten).  No kernel traps.
 *  - Within one call, distinct sequences must name distinct slots.
 *  - An empty batch (nseq == 0) is valid everywhere: after the descriptor
 *    checks (dims, params, cache) the call returns ERS_OK, launches nothing and
 *    reads none of its per-call pointers, which may then be NULL.  A negative
 *    nseq is ERS_EINVAL.
 */
#ifndef ERS_H
#define ERS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ERS_API __attribute__((visibility("default")))
#else
#define ERS_API
#endif

typedef struct CUstream_st* ers_stream_t; /* a cudaStream_t */

typedef int32_t ers_status;
#define ERS_OK 0
#define ERS_EINVAL 1        /* NULL pointer, bad count or bad flag combination */
#define ERS_ESHAPE 2        /* unsupported dimensions (see ers_dims) */
#define ERS_EDTYPE 3        /* unsupported io dtype or read-copy dtype */
#define ERS_EPTR 4          /* pointer not 16-byte aligned */
#define ERS_EALIGN 5        /* device: a slot's buffered position is outside its legal range, i.e. the
                               state's physical offset would differ from the offset the caller tracks */
#define ERS_EOVERFLOW 6     /* device: h + T > L in a verify without ERS_FLAG_AUTO_FLUSH */
#define ERS_ECOMMIT 7       /* device: accepted count outside [0, T] */
#define ERS_ESLOT 8         /* device: slot index outside [0, nslots) */
#define ERS_ETIMEOUT 9      /* device: a bounded wait gave up */
#define ERS_EWORKSPACE 10   /* workspace NULL or smaller than the size query returns */
#define ERS_ECUDA 11        /* the CUDA runtime rejected a launch */
#define ERS_EUNSUPPORTED 12 /* a valid request this build does not implement */

#define ERS_DTYPE_F32 0
#define ERS_DTYPE_BF16 1

/* Flags */
#define ERS_FLAG_FUSE_REFRESH 1u /* replay_decode: refresh (exact mode) or flush (ReplaySSM) in the same call */
#define ERS_FLAG_REPLAYSSM 2u    /* replay_decode / refresh: ReplaySSM mode (read copy, flush rule) */
#define ERS_FLAG_AUTO_FLUSH 4u   /* spec_verify / commit: flush when h + T > L instead of failing */

/* Problem dimensions.  Supported: headdim P in {16, 32, 64}, dstate N in {16, 32, 64, 128},
 * nheads % ngroups == 0, chunk Q in [1, 256].  In ReplaySSM mode `chunk` is the refresh
 * period L (the buffer capacity). */
typedef struct ers_dims {
  int32_t nheads;   /* H */
  int32_t ngroups;  /* G; head h reads B/C group h / (H/G) */
  int32_t headdim;  /* P */
  int32_t dstate;   /* N */
  int32_t chunk;    /* Q (exact mode) or L (ReplaySSM mode) */
  int32_t io_dtype; /* ERS_DTYPE_BF16 or ERS_DTYPE_F32 */
} ers_dims;

/* Per-head layer parameters, fp32 [H] each.  A < 0; dt_bias is added to the raw dt before softplus. */
typedef struct ers_params {
  const float* A;
  const float* D;
  const float* dt_bias;
} ers_params;

/* Per-slot replay cache (exact-replay RFC section 3; ReplaySSM "Motivation and method").
 *   state     [nslots, H, P, N] fp32 (or fp16, or unused, see anchor_dtype): the boundary checkpoint
 *             (exact mode) or recurrence anchor (ReplaySSM)
 *   read_copy [nslots, H, P, N] or NULL: low-precision copy cast from the same fp32 values as `state`,
 *             bf16 (read_dtype ERS_READ_BF16) or FP8 e4m3 bytes (ERS_READ_FP8_E4M3)
 *   buf_x     [nslots, Q, H, P] io dtype;  buf_dt [nslots, Q, H] fp32 raw dt
 *   buf_B, buf_C [nslots, Q, G, N] io dtype: token-major partial-chunk input buffers
 *   pos       [nslots] int32: buffered tokens p (exact mode, 0 <= p < Q between calls) or the
 *             committed pointer h (ReplaySSM mode, 0 <= h <= L).
 *   read_dtype ERS_READ_BF16 (0), ERS_READ_FP8_E4M3 (1) or ERS_READ_NVFP4 (2).
 *   read_scale [nslots, H, P] fp32, FP8 and NVFP4 read copies only (else NULL): one power-of-two
 *             scale per state row.
 *   read_block_scale [nslots, H, P, N / 16] e4m3 bytes, NVFP4 only (else NULL).
 *   buf_pages [nslots, Q / page_rows] int32 or NULL: paged partial-chunk buffers (RFC section 6,
 *             "contiguous and paged buffer layouts": slot and position indexed separately).  With a
 *             table, buf_x / buf_dt / buf_B / buf_C hold npages * page_rows rows ([npages,
 *             page_rows, H, P] and so on) and row r of slot s is row buf_pages[s][r / page_rows] *
 *             page_rows + r % page_rows; page_rows divides Q.  A page index outside [0, npages) is
 *             reported as ERS_ESLOT and clamped.  NULL: the contiguous [nslots, Q, ...] layout.
 *
 * FP8 read copy (ReplaySSM "Paper-reported results", the FP8-read / FP32-recurrence mode; the page
 * names the mode without its quantisation, so this library defines it): each state row (one d of
 * one head) has a power-of-two scale s = 2^k, k the smallest integer with amax_n |S[d][n]| <= 448 * 2^k
 * (no code saturates) and at least -127 (all-zero rows read as zeros); the row is stored as e4m3
 * bytes q[n] = RNE(S[d][n] / s) and read as q[n] * s, both scalings exact.  Outputs apply s to the
 * row's dot product with C.  read_copy is [nslots, H, P, N] bytes.
 * NVFP4 read copy ("Paper-reported results": FP32 recurrence + NVFP4 read; the format's per-tensor
 * fp32 scale is taken per state row): s = 2^k, k the smallest integer with amax <= 2688 * 2^k and at
 * least -127; with u = S / s (exact), each block of 16 consecutive values n has the e4m3 scale
 * beta = RNE_e4m3(amax_block |u| / 6) (fp32 division) and codes q = RNE_e2m1_satfinite(u * (1 / beta))
 * (fp32 reciprocal, fp32 product; q = 0 where beta = 0); the value is q * beta * s (exact).  read_copy
 * is [nslots, H, P, N / 2] bytes, value n of a row in bits 4 (n % 2)..4 (n % 2) + 3 of byte n / 2.
 * Outputs apply beta to each lane's 4-value partial dot product and s to the row's.  NVFP4 copies
 * are kept in ReplaySSM mode only.
 * Both are supported where the CUDA-core warp-per-head kernels run (headdim 64, dstate 128,
 * chunk <= 16; verify with at most 4 drafts and 8 heads per group); elsewhere calls that read or
 * write the copy return ERS_EUNSUPPORTED. */
#define ERS_READ_BF16 0
#define ERS_READ_FP8_E4M3 1
#define ERS_READ_NVFP4 2

/* Anchor (state) storage.  ERS_ANCHOR_F32: state is fp32 (every mode).  ERS_ANCHOR_F16_SR (ReplaySSM
 * "Paper-reported results", the NVFP4-read / FP16+SR-recurrence mode; the rounding is this library's
 * reading): state is IEEE fp16 [nslots, H, P, N]; a refresh folds in fp32 from the fp16 values, casts
 * the read copy from the fp32 result and stores the anchor by stochastic rounding: value n of row d
 * of head h in slot s goes up to the next fp16 value iff r < 2^32 (|v| - lo) / ulp (lo = |v| rounded
 * toward zero on the fp16 grid, ulp its spacing, 2^-24 below 2^-14; sign kept; >= 65504 gives 65504),
 * r = word n % 4 of Philox4x32-10(counter = (sr_nonce, s, h * P + d, n / 4), key = sr_key).  The
 * caller gives every call that may write anchors a fresh sr_nonce.  ReplaySSM mode only, bf16 io,
 * with a read copy, where the warp-per-head kernels run (headdim 64, dstate 128, chunk <= 16). */
/* ERS_ANCHOR_NVFP4_SHARED_SR (ReplaySSM "Paper-reported results", the shared-FP4 recurrence mode; the
 * rounding is this library's reading): the NVFP4 read copy is the only state and `state` is unused
 * (may be NULL).  A refresh folds from the copy's values (code * (beta * s), fp32), then writes the
 * copy with the NVFP4 cast above except that each code rounds stochastically: with x = u * (1 / beta)
 * (as above), lo the largest e2m1 magnitude <= |x| and step the spacing above it (0.5 below 2, 1
 * below 4, 2 below 6), |x| goes up to lo + step iff r < 2^32 (|x| - lo) / step, else down to lo;
 * |x| >= 6 gives 6; the sign is kept; r as for fp16 anchors (word n % 4 of Philox4x32-10 at counter
 * (sr_nonce, s, h * P + d, n / 4), key sr_key).  The scales are those of the round-to-nearest cast.
 * A slot with pos == 0 is never rewritten (an empty history leaves the state as it is).  To start
 * from an fp32 state, cast it with ers_refresh (ReplaySSM, pos = 0) on a cache with ERS_ANCHOR_F32,
 * that state and the same NVFP4 copy, then use the copy with this mode.  ReplaySSM mode only, bf16
 * io, an NVFP4 read copy, the warp-per-head shapes. */
#define ERS_ANCHOR_F32 0
#define ERS_ANCHOR_F16_SR 1
#define ERS_ANCHOR_NVFP4_SHARED_SR 2

typedef struct ers_cache {
  void* state;
  void* read_copy;
  void* buf_x;
  float* buf_dt;
  void* buf_B;
  void* buf_C;
  int32_t* pos;
  int32_t nslots;
  int32_t read_dtype;
  float* read_scale;
  uint8_t* read_block_scale;
  int32_t anchor_dtype;
  uint32_t sr_key[2];
  uint32_t sr_nonce;
  const int32_t* buf_pages;
  int32_t page_rows;
  int32_t npages;
} ers_cache;

/* Human-readable name of a status code (static storage, never NULL). */
ERS_API const char* ers_status_str(ers_status s);

/* Library version as major*10000 + minor*100 + patch. */
ERS_API int32_t ers_version(void);

/* Check of the library's bounded device waits (no counterpart on the pages; every wait in the
 * library gives up after a limit instead of spinning forever, and reports ERS_ETIMEOUT).  Launches
 * two blocks on `stream`: one waits on an mbarrier phase that nothing completes, the other on a
 * device flag that nothing sets, each with the library's own wait routine and the given limit
 * (1 ns .. 10 s).  Both give up after limit_ns, write ERS_ETIMEOUT to *dev_status (device int32,
 * required, zeroed by the caller) and return; the context stays usable.  ERS_EINVAL for a NULL
 * status or a limit outside that range. */
ERS_API ers_status ers_selftest_bounded_wait(uint64_t limit_ns, ers_stream_t stream, int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Chunked SSD scan (prefill).  RFC section 1 (the chunked scan used for prefill), Evidence 3
 * (prefix- and packing-invariant outputs) and Evidence 4 (fp32 inter-chunk state passing inside
 * one call, rounded only on store).
 *
 * nseq sequences are packed along the token axis: sequence i owns tokens
 * [cu_seqlens[i], cu_seqlens[i+1]) (cu_seqlens: device int32 [nseq+1], cu_seqlens[0] = 0,
 * non-decreasing, cu_seqlens[nseq] = ntokens); max_seqlen >= every sequence length.  Each
 * sequence's chunk grid starts at its own first token; no chunk spans two sequences.
 *   x [ntokens, H, P], dt [ntokens, H] raw, B/C [ntokens, G, N]
 *   init_state [nseq, H, P, N] fp32 or NULL (zero)
 *   y [ntokens, H, P] (out), final_state [nseq, H, P, N] fp32 (out)
 *   chunk_states [nseq, ceil(max_seqlen/Q), H, P, N] fp32 or NULL (out): the state at the end of
 *     each chunk of each sequence ("return_intermediate_states"); entries past a sequence's last
 *     chunk are left unwritten.
 * Workspace: ers_ssd_scan_fwd_workspace_size(dims, nseq, max_seqlen) bytes. */
ERS_API size_t ers_ssd_scan_fwd_workspace_size(const ers_dims* dims, int32_t nseq, int32_t max_seqlen);
ERS_API ers_status ers_ssd_scan_fwd(const ers_dims* dims, const ers_params* prm, int32_t nseq, int64_t ntokens,
                            int32_t max_seqlen, const int32_t* cu_seqlens, const void* x, const float* dt,
                            const void* B, const void* C, const float* init_state, void* y,
                            float* final_state, float* chunk_states, void* workspace, size_t workspace_bytes,
                            ers_stream_t stream, int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Boundary-anchored prefill / chunked prefill / recompute.  RFC section 3, second bullet: the
 * call starts at each sequence's boundary, the buffered tokens are prepended and their outputs
 * discarded, the trailing partial chunk's inputs go to the buffer, and the boundary state becomes
 * the state at the last full chunk.
 *
 * Sequence i resumes slot slot[i] (slot: device int32 [nseq], or NULL for slot = i), whose pos p
 * must satisfy 0 <= p < Q, and appends its new tokens (packed as in ers_ssd_scan_fwd; max_seqlen
 * bounds the NEW token counts).  y receives the outputs of the new tokens only.  On return
 * (stream order) cache->state holds the state at the last chunk boundary, the buffer holds the
 * (p + len) mod Q trailing inputs, and pos = (p + len) mod Q.
 * Workspace: ers_chunked_prefill_workspace_size(dims, nseq, max_seqlen) bytes. */
ERS_API size_t ers_chunked_prefill_workspace_size(const ers_dims* dims, int32_t nseq, int32_t max_seqlen);
ERS_API ers_status ers_chunked_prefill(const ers_dims* dims, const ers_params* prm, const ers_cache* cache,
                               int32_t nseq, int64_t ntokens, int32_t max_seqlen, const int32_t* cu_seqlens,
                               const int32_t* slot, const void* x, const float* dt, const void* B,
                               const void* C, void* y, void* workspace, size_t workspace_bytes,
                               ers_stream_t stream, int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Exact-replay decode step.  RFC section 3, first bullet: each sequence's buffered partial chunk
 * plus its new token is replayed from the boundary state; the last token's output is the layer
 * output; the new token's inputs are appended to the buffer; when the chunk fills, the chunk's
 * final state becomes the new boundary state and the buffer empties.
 *
 *   x [nseq, H, P], dt [nseq, H], B/C [nseq, G, N]: one new token per sequence; y [nseq, H, P] (out)
 * Exact mode (flags without ERS_FLAG_REPLAYSSM): requires 0 <= pos < Q, reads cache->state (fp32).
 *   With ERS_FLAG_FUSE_REFRESH a slot that fills its chunk is refreshed in the same call (pos -> 0);
 *   without it pos reaches Q and ers_refresh(EXACT) must run before the next decode.  Both give
 *   identical bits.
 * ReplaySSM mode (ERS_FLAG_REPLAYSSM): requires a read copy; outputs read the read copy.  Without
 *   ERS_FLAG_FUSE_REFRESH it requires 0 <= pos < L and never refreshes (ers_refresh applies the flush
 *   rule).  With ERS_FLAG_FUSE_REFRESH it accepts 0 <= pos <= L and applies the flush rule for one
 *   token first (pos + 1 > L: fold the L committed records into the anchor, recast the read copy,
 *   pos = 0), so the new token always fits; identical bits to ers_refresh(ERS_FLAG_REPLAYSSM,
 *   drafts_T = 1) followed by the decode without the flag.
 * pos advances by one per call (or returns to 0, or 1 after a ReplaySSM flush); while the call runs, the
 * upper 16 bits of a slot's pos entry may hold a count of the kernel's own, cleared before it ends,
 * so no other work may read or write pos concurrently with the call.
 * Launches (all on `stream`): with ERS_FLAG_FUSE_REFRESH and at most 8 heads per group (chunk <= 32)
 * the call is two launches, the slots whose step refreshes or flushes first and the others as its
 * programmatic dependent, which completes after it.  ReplaySSM with bf16 io and a bf16 read copy
 * (chunk <= 16, P = 64, N = 128, at most 8 heads per group) computes the read copy's products on the
 * tensor core, in the kernel ers_spec_verify runs for the same cache, so the two keep each other's
 * bits; FP8 and NVFP4 copies use the CUDA-core kernels for both calls.
 * Device errors: ERS_EALIGN (pos out of range), ERS_ESLOT. */
ERS_API ers_status ers_replay_decode(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                             const int32_t* slot, const void* x, const float* dt, const void* B, const void* C,
                             uint32_t flags, void* y, ers_stream_t stream, int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Checkpoint refresh.  RFC section 3 (the chunk's final state becomes the new boundary state) and
 * ReplaySSM "Core equations" (refresh forms S from the committed raw records, then casts the
 * high- and low-precision copies independently from the same unrounded state).
 *
 * Exact mode (flags = 0): slots with pos == Q fold their Q buffered tokens into cache->state and
 *   get pos = 0; other slots are untouched.
 * ReplaySSM mode (ERS_FLAG_REPLAYSSM): slots with pos + T > L (T = drafts_T, the flush rule; pass
 *   drafts_T > L to refresh every slot) fold their pos committed records into the anchor, write the
 *   read copy (if present) from the same fp32 values, and get pos = 0.  A slot with pos == 0 keeps
 *   its anchor bits unchanged (its read copy is rewritten from them).
 * Device errors: ERS_EALIGN (pos outside [0, Q] / [0, L]), ERS_ESLOT. */
ERS_API ers_status ers_refresh(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                       const int32_t* slot, uint32_t flags, int32_t drafts_T, ers_stream_t stream,
                       int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Output-only speculative verification.  ReplaySSM "Motivation and method" (outputs replay the
 * checkpoint and buffered inputs; verification uses an output-only form rather than a per-draft
 * state) and "Core equations" (O = S_ckpt Q D + V (W . K^T Q); flush when h + T > L).
 *
 *   x [nseq, T, H, P], dt [nseq, T, H], B/C [nseq, T, G, N]: T draft tokens per sequence
 *   y [nseq, T, H, P] (out): draft s's output given committed records and drafts 1..s, computed
 *     from the bf16 read copy (required).
 * The drafts are written to buffer rows [h', h'+T) where h' = 0 if the slot flushed, else h = pos.
 * pos is NOT changed: ers_commit must follow before the next verify on the same slots.
 * With ERS_FLAG_AUTO_FLUSH a slot with h + T > L first refreshes its h committed records (as
 * ers_refresh in ReplaySSM mode); without it such a slot reports ERS_EOVERFLOW.
 * Requires 1 <= T <= L.  Supported read copies: bf16 for any T (bf16 io, L <= 16, P = 64, N = 128,
 * at most 8 heads per group: the drafts' products on the tensor core, the kernel ReplaySSM decode of
 * the same cache runs); FP8, NVFP4 and fp16 / shared anchors otherwise need T <= 4, L <= 16, P = 64,
 * N = 128 and at most 8 heads per group (ERS_EUNSUPPORTED).  With ERS_FLAG_AUTO_FLUSH the call is two
 * launches on `stream` (the flushing slots first, the others as its programmatic dependent). */
ERS_API ers_status ers_spec_verify(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                           const int32_t* slot, int32_t T, const void* x, const float* dt, const void* B,
                           const void* C, uint32_t flags, void* y, ers_stream_t stream, int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Commit.  ReplaySSM "Motivation and method": the acceptance length advances only the
 * committed-input pointer; rejected drafts never enter the recurrence and may be overwritten.
 *
 * accepted: device int32 [nseq] with 0 <= accepted[i] <= T.  For each sequence,
 *   pos[slot] = (flushed ? 0 : pos[slot]) + accepted[i], flushed = (flags & AUTO_FLUSH) && pos + T > L,
 * i.e. the same decision the preceding ers_spec_verify (same T, L and flags) took.  Nothing but
 * pos is touched.  Device errors: ERS_ECOMMIT, ERS_ESLOT. */
ERS_API ers_status ers_commit(const ers_dims* dims, const ers_cache* cache, int32_t nseq, const int32_t* slot,
                      const int32_t* accepted, int32_t T, uint32_t flags, ers_stream_t stream,
                      int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Exact-mode speculative verify and commit: speculation that keeps the chunk grid.  RFC section 6
 * (the phase-1 prototype's speculative decoding on the exact-replay path) with ReplaySSM "Motivation
 * and method" (outputs of drafts from the checkpoint and the buffered inputs; rejected drafts never
 * enter the state).  In exact mode the checkpoint sits on the chunk grid, so a draft past the end of
 * the current chunk gets the output exact-replay decode would give it: from the boundary state that
 * the full chunk (buffered rows, then the drafts before the boundary) folds into.
 *
 * ers_spec_verify_exact: T drafts per sequence, 1 <= T <= Q: x [nseq, T, H, P], dt [nseq, T, H] raw,
 *   B/C [nseq, T, G, N]; y [nseq, T, H, P] (out).  Draft j's output is, bit for bit, the output
 *   ers_replay_decode (exact mode, ERS_FLAG_FUSE_REFRESH) gives draft j after drafts 0 .. j-1 were
 *   decoded, crossing the chunk boundary where they reach it.  The cache is not changed.  With
 *   Q <= 16, T <= 4, P = 64, N = 128 and at most 8 heads per group the call is one launch that
 *   streams each checkpoint once and forms the folded boundary state row by row for the drafts past
 *   it (`workspace` is not touched); otherwise it copies the slots' checkpoints, buffered rows and
 *   positions into `workspace` (ers_spec_verify_exact_workspace_size(dims, nseq) bytes, about an
 *   fp32 state and a buffer per sequence) and decodes the drafts there one at a time (T decode
 *   launches and their row copies).  The workspace is required in both cases.
 *   Requires an fp32 checkpoint (ERS_ANCHOR_F32; read copies, if any, are neither read nor written)
 *   and 0 <= pos < Q.
 * ers_commit_exact: after a verify, the first accepted[i] (0 <= accepted[i] <= T, device int32 [nseq])
 *   drafts of sequence i, passed again as the same x, dt, B, C, enter the cache: those that fit the
 *   current chunk are appended to the buffer; if they fill it, the chunk folds into the checkpoint by
 *   the exact-mode refresh (the arithmetic of decode's fused refresh; a read copy is recast with it)
 *   and the drafts past the boundary become the new buffer; pos = (pos + accepted) mod Q.  The state
 *   afterwards is bit for bit the one decoding the accepted drafts would leave.  workspace: at least
 *   nseq * 4 bytes rounded up to 256 (the verify's workspace serves).
 * Device errors: ERS_EALIGN (pos outside [0, Q)), ERS_ECOMMIT, ERS_ESLOT. */
ERS_API size_t ers_spec_verify_exact_workspace_size(const ers_dims* dims, int32_t nseq);
ERS_API ers_status ers_spec_verify_exact(const ers_dims* dims, const ers_params* prm, const ers_cache* cache,
                                         int32_t nseq, const int32_t* slot, int32_t T, const void* x, const float* dt,
                                         const void* B, const void* C, void* y, void* workspace,
                                         size_t workspace_bytes, ers_stream_t stream, int32_t* dev_status);
ERS_API ers_status ers_commit_exact(const ers_dims* dims, const ers_params* prm, const ers_cache* cache, int32_t nseq,
                                    const int32_t* slot, const int32_t* accepted, int32_t T, const void* x,
                                    const float* dt, const void* B, const void* C, void* workspace,
                                    size_t workspace_bytes, ers_stream_t stream, int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Per-token state-writeback update (the recurrent "selective state update" the RFC's section 1
 * contrasts with the chunked scan; the comparison point for replay decode).
 *   state [nslots, H, P, N] fp32, updated in place for slot[i] (slot NULL = identity)
 *   x [nseq, H, P], dt [nseq, H], B/C [nseq, G, N]; y [nseq, H, P] (out)
 * Device errors: ERS_ESLOT. */
ERS_API ers_status ers_ssu_update(const ers_dims* dims, const ers_params* prm, float* state, int32_t nslots,
                          int32_t nseq, const int32_t* slot, const void* x, const float* dt, const void* B,
                          const void* C, void* y, ers_stream_t stream, int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Gated delta rule (GDN) layer: output-only speculative verify, refresh and commit (ReplaySSM notes,
 * "Core equations": GDN residuals solve u_j + sum_{i<j} beta_j gamma_{i+1:j} (k_i . k_j) u_i =
 * beta_j (v_j - gamma_j S_ckpt k_j); "Data protocol and entry point": an empty history leaves the anchor unchanged).
 * Per value head h (key group h / (H/G)), token t: a_t = exp(g_t), u_t = beta_t (v_t - a_t S k_t),
 * S <- a_t S + u_t k_t^T, o_t = S q_t; S is [dv, dk] (maps keys to values).
 *
 *   dims: H, G (G divides H), dk = dv = 128, window L in [1, 32], io_dtype for q, k, v, o and the
 *         k / v buffers.
 *   cache: anchor [nslots, H, dv, dk] fp32; read_copy [nslots, H, dv, dk] bf16 (cast from the same
 *         fp32 values at every refresh); buf_k [nslots, L, G, dk], buf_v [nslots, L, H, dv] (io);
 *         buf_g, buf_beta [nslots, L, H] fp32; buf_u [nslots, L, H, dv] fp32 (each committed record's
 *         residual as computed from the read copy by the verify that produced it); pos [nslots] =
 *         committed records h (0 <= h <= L).
 * ers_gdn_verify: T drafts per sequence (1 <= T <= min(8, L)): q, k [nseq, T, G, dk], v [nseq, T, H, dv] (io),
 *   g, beta [nseq, T, H] fp32 (g = log of the gate, beta in (0, 1)); o [nseq, T, H, dv] (out).  With
 *   ERS_FLAG_AUTO_FLUSH a slot with h + T > L first folds its h records into the anchor (h > 0) and
 *   recasts the read copy; without it such a slot reports ERS_EOVERFLOW.  Outputs read the read copy;
 *   drafts are written to buffer rows h.. (0.. after a flush); pos is not moved.
 * ers_gdn_commit: h = (flushed ? 0 : h) + accepted[i], flushed = AUTO_FLUSH && h + T > L.
 * ers_gdn_refresh: slots with h + T > L (T = drafts_T) fold their records (h > 0) and get h = 0.
 * The same committed stream and refresh points give the same bits whether tokens arrive as drafts
 * of one verify or as T = 1 verifies.  Device errors: ERS_EALIGN, ERS_EOVERFLOW, ERS_ECOMMIT, ERS_ESLOT. */
typedef struct ers_gdn_dims {
  int32_t nheads;
  int32_t ngroups;
  int32_t dk;
  int32_t dv;
  int32_t window;
  int32_t io_dtype;
} ers_gdn_dims;

typedef struct ers_gdn_cache {
  float* anchor;
  void* read_copy;
  void* buf_k;
  void* buf_v;
  float* buf_g;
  float* buf_beta;
  float* buf_u;
  int32_t* pos;
  int32_t nslots;
} ers_gdn_cache;

ERS_API ers_status ers_gdn_verify(const ers_gdn_dims* dims, const ers_gdn_cache* cache, int32_t nseq,
                                  const int32_t* slot, int32_t T, const void* q, const void* k, const void* v,
                                  const float* g, const float* beta, uint32_t flags, void* o, ers_stream_t stream,
                                  int32_t* dev_status);

ERS_API ers_status ers_gdn_commit(const ers_gdn_dims* dims, const ers_gdn_cache* cache, int32_t nseq,
                                  const int32_t* slot, const int32_t* accepted, int32_t T, uint32_t flags,
                                  ers_stream_t stream, int32_t* dev_status);

ERS_API ers_status ers_gdn_refresh(const ers_gdn_dims* dims, const ers_gdn_cache* cache, int32_t nseq,
                                   const int32_t* slot, int32_t drafts_T, ers_stream_t stream, int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * Causal depthwise conv1d with a conv state: the step upstream of the SSM, whose prefill and
 * decode-update paths must give identical bits (exact-replay RFC, section 2 Evidence item 6; bf16
 * operands promoted to fp32 before accumulation).  Per channel c, with u the inputs preceded by
 * the W - 1 earlier inputs held in the conv state (oldest first; zeros when not read):
 *     acc = bias[c];  acc = fmaf(w[c][k], u[t + k], acc) for k = 0 .. W-1;  y[t][c] = act(acc)
 * with act(a) = a / (1 + exp(-a)) (SiLU, IEEE division) when ERS_CONV_SILU is set, else a.
 *
 *   dims->channels C (a multiple of 8), dims->width W in {2, 3, 4}, dims->io_dtype for x, weight, bias, y and
 *   the state; x, y [T, C] (prefill, packed by cu_seqlens [nseq+1]) or [nseq, C] (update); weight
 *   [C, W]; bias [C] or NULL; conv_state [nslots, W-1, C], row 0 the oldest input; slot [nseq] or
 *   NULL (sequence i uses slot i).
 * ers_conv1d_fwd: reads the initial state when read_state != 0 (else zeros) and writes the final
 *   state (the last W - 1 entries of u) when conv_state is not NULL.  max_seqlen bounds the longest
 *   sequence.
 * ers_conv1d_update: one token per sequence; shifts the state by one and stores the new input.
 * Device errors: ERS_ESLOT. */
#define ERS_CONV_SILU 1u

typedef struct ers_conv_dims {
  int32_t channels;
  int32_t width;
  int32_t io_dtype;
  uint32_t flags;
} ers_conv_dims;

ERS_API ers_status ers_conv1d_fwd(const ers_conv_dims* dims, int32_t nseq, int64_t ntokens, int32_t max_seqlen,
                                  const int32_t* cu_seqlens, const void* x, const void* weight, const void* bias,
                                  void* conv_state, int32_t nslots, const int32_t* slot, int32_t read_state,
                                  void* y, ers_stream_t stream, int32_t* dev_status);

ERS_API ers_status ers_conv1d_update(const ers_conv_dims* dims, int32_t nseq, const void* x, const void* weight,
                                     const void* bias, void* conv_state, int32_t nslots, const int32_t* slot,
                                     void* y, ers_stream_t stream, int32_t* dev_status);

/* ---------------------------------------------------------------------------------------------
 * ers_ssd_scan_fwd with library-owned scratch.  The pages have no counterpart to this call; it
 * exists for callers that cannot hand the scan a workspace: a host program that owns no device
 * allocator (plain C over the runtime, no tensor library), and serving loops that must not
 * allocate per call because cudaMalloc/cudaFree synchronise the device.
 *
 * Same arguments, semantics and outputs as ers_ssd_scan_fwd minus the workspace.  The scratch is a
 * fixed device array of ERS_STATIC_SCRATCH_BYTES inside this library (one per device context); a
 * call whose ers_ssd_scan_fwd_workspace_size exceeds it returns ERS_EWORKSPACE and launches
 * nothing (32 MiB holds, e.g., 2048 tokens x 32 heads x headdim 64 x dstate 128 at chunk 256,
 * which needs 16.8 MB).  Nothing in the scratch needs to start at zero: a call clears what it
 * reads before writing it (the look-back flags, by an asynchronous memset on `stream`) or reads
 * only bytes it wrote earlier in the same call.  The first call in a context looks up the scratch address with
 * that context current (cudaGetSymbolAddress) and caches it with the context's id; a call made
 * in another context of the same device (after cudaDeviceReset, or with a context the caller
 * created made current) has its own copy of the array and looks it up again.  Make one call in
 * each context before any stream capture.  Allocates nothing.  The scratch is shared: two calls
 * on the same device that can run at the same time (different streams, or different host
 * threads) race on it and must be serialised by the caller. */
#define ERS_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
ERS_API ers_status ers_ssd_scan_fwd_static(const ers_dims* dims, const ers_params* prm, int32_t nseq,
                                   int64_t ntokens, int32_t max_seqlen, const int32_t* cu_seqlens,
                                   const void* x, const float* dt, const void* B, const void* C,
                                   const float* init_state, void* y, float* final_state, float* chunk_states,
                                   ers_stream_t stream, int32_t* dev_status);

#ifdef __cplusplus
}
#endif

#endif /* ERS_H */
