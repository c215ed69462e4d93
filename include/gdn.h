/*
 * gdn.h -- C ABI of the GB300 (sm_103a) chunked Gated DeltaNet prefill library.
 *
 * The operation.  The pages name a "chunked Gated DeltaNet prefill" as one of the
 * fused operations of their native Qwen3.5 prefill workers and test it against
 * float64 references ("Cua-S1 4B 0.2 native text worker", kernel-test paragraph;
 * "Open-Jev-27B-v1.1 native text worker", section "Validation and optimization
 * scope").  They print no equations; the library computes the gated delta rule
 * per (sequence, value head):
 *
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   alpha_t = exp(g_t)
 *     o_t = S_t q_t / sqrt(dk)
 *
 * with S a dv x dk fp32 state (S_0 = init_state, or zeros) and the last S
 * returned as the final state.  q and k are expected to be L2-normalised per
 * token by the caller (the pages do this in a separate fused norm operation).
 * Internally the tokens of each sequence are processed in chunks of 64 with
 * the WY / UT-transform form of the recurrence.
 *
 * Versioning.  Like the pages' library ("ABI 4", later "CUDA ABI is 5"), the
 * ABI carries a version number; callers built against another version must be
 * rebuilt together with the library.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 5

/* Status codes (0 = success, negative = error). */
#define GDN_OK 0
#define GDN_ERR_ARG (-1)    /* null required pointer, bad size, Hv % Hk != 0, unsupported dk/dv */
#define GDN_ERR_ALIGN (-2)  /* a pointer is not 16-byte aligned */
#define GDN_ERR_ALLOC (-3)  /* the library's device workspace could not be grown */
#define GDN_ERR_LAUNCH (-4) /* a CUDA call or kernel launch failed (see gdn_last_cuda_error) */
#define GDN_ERR_SCRATCH (-5) /* the problem needs more scratch than the fixed or caller-given workspace */

/* Flags of gdn_prefill_ex. */
#define GDN_FLAG_L2NORM_QK 1u /* normalise q and k per token inside the kernels: x / max(||x||, 1e-6) */
#define GDN_FLAG_TWO_LEVEL 2u /* use the two-level chunk scan (dense batches only) */
#define GDN_FLAG_ONE_LEVEL 4u /* never use the two-level chunk scan */
/* Segments per sequence for GDN_FLAG_TWO_LEVEL (2..255; 0 or absent = chosen by the library). */
#define GDN_FLAG_SEGMENTS(n) ((((unsigned)(n)) & 0xffu) << 8)
#define GDN_FLAG_SLICE32 0x10000u /* state carry: 32 state rows per CTA */
#define GDN_FLAG_SLICE16 0x40000u /* state carry: 16 state rows per CTA */
#define GDN_FLAG_SLICE64 0x20000u /* state carry: 64 state rows per CTA (dv a multiple of 64) */
#define GDN_FLAG_WIDE_RANGE 0x80000u /* state carry on bf16 hi + lo operand pairs (fp32 range; slower) */

/* Size of the fixed device scratch array behind gdn_prefill_static (64 MiB per device). */
#define GDN_STATIC_SCRATCH_BYTES (128u << 20)

/* Returns GDN_ABI_VERSION of the loaded library. */
int gdn_abi_version(void);

/* Human-readable text for a status code (static storage, never NULL). */
const char *gdn_strerror(int status);

/* The cudaError_t of the most recent GDN_ERR_LAUNCH / GDN_ERR_ALLOC on this thread (0 if none). */
int gdn_last_cuda_error(void);

/*
 * gdn_prefill -- chunked Gated DeltaNet prefill on the GPU, asynchronous on `stream`.
 *
 * Pointers (all DEVICE memory, owned by the caller, not retained after return,
 * each 16-byte aligned):
 *   q, k        bf16 [Ttot, Hk, dk]   queries and keys (L2-normalised per token)
 *   v           bf16 [Ttot, Hv, dv]   values
 *   g           fp32 [Ttot, Hv]       log decay, g <= 0 (alpha = exp(g))
 *   beta        fp32 [Ttot, Hv]       write strength in (0, 1)
 *   cu_seqlens  int32 [B + 1] or NULL packed sequence boundaries (see below)
 *   init_state  fp32 [B, Hv, dv, dk] or NULL (NULL = zero initial states)
 *   out         bf16 [Ttot, Hv, dv]   outputs o_t (written; must not alias any input)
 *   final_state fp32 [B, Hv, dv, dk] or NULL (NULL = not written); may alias init_state
 *
 * Sizes.  With cu_seqlens == NULL there are B sequences of T tokens each and
 * Ttot = B * T.  Otherwise B is the number of packed sequences, sequence b covers
 * tokens [cu_seqlens[b], cu_seqlens[b + 1]), cu_seqlens[0] = 0, cu_seqlens[B] =
 * T = Ttot, entries non-decreasing; zero-length sequences are allowed and return
 * their initial state.  The contents of cu_seqlens are not checked on the host
 * (that would need a synchronisation); out-of-range entries are clamped to
 * [0, T] on the device so no access leaves the buffers, and a malformed array sets
 * GDN_STATUS_BAD_CU_SEQLENS (see gdn_device_status).  Value head h reads key head
 * h / (Hv / Hk).  dk and dv must each be 32, 64 or 128.
 *
 * Precision and range.  The chunk products run on the tensor cores with fp32
 * accumulation and fp16 operands: k and q (converted from bf16, exact for
 * magnitudes 2^-17 .. 65504), the chunk's UT transform and score product, and the
 * state-side operands rounded from the fp32 state (2^-11 relative).  The state
 * itself is carried in fp32.  Operands beyond fp16's range (about 65504: values of
 * that size, or a state that grows to it) make the state non-finite, which sets
 * GDN_STATUS_NONFINITE_STATE.  Below it, fp16 keeps full precision only down to 2^-14:
 * with values of order 1e-5 and less the operands lose accuracy, and a single-level
 * call whose final state for some (sequence, head, row block) is nonzero but below
 * 2^-12 sets GDN_STATUS_SMALL_STATE.  gdn_prefill_ex with GDN_FLAG_WIDE_RANGE carries
 * the state-side operands as bf16 hi + lo pairs instead (fp32 range, 2^-16, slower).
 *
 * Memory.  The library keeps a per-device, grow-only workspace (allocated on the
 * first call that needs more; about 16 KB per 64-token chunk and value head, plus
 * 32 KB per chunk and key head for dk = 128, 16 KB for dk <= 64).
 * After a call at the largest size, later calls allocate nothing.  gdn_prefill,
 * gdn_prefill_ex and gdn_prefill_host calls on one device share that workspace
 * (and gdn_prefill_host's staging area): calls whose GPU work could overlap
 * (different streams, or host threads without ordering) must be ordered by the
 * caller, or use gdn_prefill_ws with a workspace each.
 *
 * Long prompts with few heads.  The chunks of a sequence are processed in order,
 * so a dense batch (cu_seqlens == NULL) whose B * Hv * dv / 32 state-carry blocks
 * leave most SMs idle is cut into P segments on 64-token boundaries and run as a
 * two-level scan instead: every segment's state transition and zero-start end
 * state at once, a short fp32 combine of the segment start states, then every
 * segment again from its true start state.  This applies when at least three
 * segments of four or more chunks fit one wave of B * P * Hv * (dv + dk) / 32
 * blocks (for example one 16,384-token prompt with 4 value heads of 128).  It
 * uses a second library-owned buffer (two bf16 [Ttot, Hv, dk] tensors and a few
 * fp32 state sets, also grow-only) and a library-owned second stream joined back
 * into `stream` by events.  Its results agree with the single-level path to the
 * stated tolerances, not bit for bit.  gdn_prefill_ex can force or forbid it.
 *
 * Returns GDN_OK, or an error code before anything is launched (argument and
 * alignment errors), or GDN_ERR_LAUNCH / GDN_ERR_ALLOC.  B == 0 returns GDN_OK
 * and does nothing.  The call does not synchronise the stream.
 */
int gdn_prefill(const void *q, const void *k, const void *v,
                const float *g, const float *beta,
                const int32_t *cu_seqlens, const float *init_state,
                void *out, float *final_state,
                int B, int T, int Hk, int Hv, int dk, int dv,
                void *stream /* cudaStream_t; NULL = legacy default stream */);

/*
 * gdn_prefill_host -- the same operation on HOST buffers (same layouts; any
 * alignment).  Copies the inputs to the library's device staging area, runs
 * gdn_prefill on `stream`, copies out and final_state back and synchronises
 * `stream` before returning.  Page-locked host buffers give the fastest copies.
 * cu_seqlens, init_state and final_state may be NULL as above.  For problems of
 * 8 MB or more (q, k and v together) the copies overlap the kernels, on
 * library-owned streams that are joined back into `stream`:
 *   - equal-length batches: 2 to 8 windows of whole 64-token chunks (about 16
 *     chunks each, the last one half as many).  The copies of one window overlap the kernels of the previous
 *     one and the copy-back of earlier ones; each window's state carry starts from
 *     the state the previous window left (kept on the device in fp32);
 *   - packed batches: up to four groups of whole key heads, whose state carries
 *     run side by side.
 * Either way the results are bit for bit those of gdn_prefill.
 */
int gdn_prefill_host(const void *q, const void *k, const void *v,
                     const float *g, const float *beta,
                     const int32_t *cu_seqlens, const float *init_state,
                     void *out, float *final_state,
                     int B, int T, int Hk, int Hv, int dk, int dv,
                     void *stream);

/*
 * gdn_prefill_ex -- gdn_prefill with option flags.
 *
 * GDN_FLAG_L2NORM_QK: q and k are taken as they come out of the projections and
 * L2-normalised per token inside the kernels (the pages run this normalisation
 * as a separate fused "norm ... QK" operation before the prefill; "Open-Jev-27B-v1.1
 * native text worker", "Validation and optimization scope").  The norms are summed
 * in fp32 from the bf16 inputs and applied as row scalings of the fp32 products, so
 * no normalised copy of q or k is written.
 *
 * GDN_FLAG_TWO_LEVEL: use the two-level chunk scan described under gdn_prefill
 * whenever the batch is dense and has at least two chunks per sequence, with
 * GDN_FLAG_SEGMENTS(n) segments per sequence (capped at the chunk count) or, without
 * it, the library's choice (at least 3).  GDN_FLAG_ONE_LEVEL: never use it.  Both
 * together, or unknown flag bits, are GDN_ERR_ARG.
 *
 * GDN_FLAG_SLICE16 / GDN_FLAG_SLICE32 / GDN_FLAG_SLICE64: each state-carry CTA owns
 * 16, 32 or 64 rows of the dv x dk state.  Without one, the library takes 64 when dv is
 * a multiple of 64 and 1.5 x the waves (of one CTA per SM) of 64-row CTAs are fewer
 * than those of 32-row CTAs (many sequences or heads), 16 when twice as many 32-row
 * CTAs would still fit one wave (few heads), else 32.  More than one of them, or
 * GDN_FLAG_SLICE64 with dv = 32, is GDN_ERR_ARG.
 * The results are the same for every width.
 *
 * GDN_FLAG_WIDE_RANGE: the state carry takes its state-side tensor-core operands as
 * bf16 hi + lo pairs (fp32 range, ~2^-16 relative) and the chunk's UT transform and
 * score product as bf16, instead of fp16 throughout.  For inputs or states beyond
 * fp16's range (see "Precision and range" under gdn_prefill); slower.  Everything
 * else as gdn_prefill.
 */
int gdn_prefill_ex(const void *q, const void *k, const void *v,
                   const float *g, const float *beta,
                   const int32_t *cu_seqlens, const float *init_state,
                   void *out, float *final_state,
                   int B, int T, int Hk, int Hv, int dk, int dv,
                   unsigned flags, void *stream);

/*
 * gdn_prefill_ws -- gdn_prefill with a caller-owned workspace.
 *
 * Same arguments, layouts, alignment rules and status codes as gdn_prefill, plus
 * `workspace` (device memory, 256-byte aligned, at least gdn_workspace_bytes(B, T,
 * Hk, Hv, dk, dv, cu_seqlens != NULL) bytes, not shared with concurrent calls) and
 * its size.  The call allocates nothing and never synchronises the host, so a
 * caller can record it into a CUDA graph and replay it with new input values in
 * the same buffers -- the calling convention behind the pages' per-prompt-length
 * CUDA Graph replay ("Cua-S1 4B 0.2 native text worker", CUDA Graph paragraph).
 * Returns GDN_ERR_SCRATCH when the workspace is too small, GDN_ERR_ALIGN when it
 * is not 256-byte aligned.  Always the single-level path (no second stream, no
 * library buffers).
 */
int gdn_prefill_ws(const void *q, const void *k, const void *v,
                   const float *g, const float *beta,
                   const int32_t *cu_seqlens, const float *init_state,
                   void *out, float *final_state,
                   int B, int T, int Hk, int Hv, int dk, int dv,
                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_decode -- one token per sequence on a carried state, the state updated in place.
 *
 *   q, k   bf16 [B, Hk, dk];  v bf16 [B, Hv, dv];  g, beta fp32 [B, Hv]
 *   state  fp32 [B, Hv, dv, dk]  read as S_{t-1}, overwritten with S_t
 *   out    bf16 [B, Hv, dv]      o_t = S_t q_t / sqrt(dk)
 *
 * The same recurrence as gdn_prefill applied to a single token, so a prefill of
 * T tokens followed by gdn_decode of token T+1 matches a prefill of T+1 tokens.
 * All pointers device memory, 16-byte aligned; out must not alias the inputs.
 * Asynchronous on `stream`; allocates nothing.  Returns GDN_OK or an argument /
 * alignment / launch error.
 */
int gdn_decode(const void *q, const void *k, const void *v, const float *g, const float *beta,
               float *state, void *out, int B, int Hk, int Hv, int dk, int dv, void *stream);

/*
 * gdn_set_phase_events -- timing hook for the NEXT gdn_prefill call on this host
 * thread.  ev_begin, ev_mid and ev_end are cudaEvent_t handles created by the
 * caller; they are recorded on the call's stream before the chunk-preparation
 * kernel, between it and the state-carry kernel, and after the state-carry
 * kernel.  The hook is consumed by that one call (pass NULLs to clear it).
 */
void gdn_set_phase_events(void *ev_begin, void *ev_mid, void *ev_end);

/*
 * gdn_prefill_static -- gdn_prefill for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point.  It exists for callers that
 * are not allowed to call cudaMalloc: a plugin whose host engine owns all device
 * memory, a service with a memory budget fixed at start-up, or code that must not
 * take the implicit device synchronisation of cudaMalloc / cudaFree.  Same
 * arguments, layouts, alignment rules and status codes as gdn_prefill; the caller
 * still passes the inputs and outputs.  Instead of the grow-only workspace it uses
 * a fixed array of GDN_STATIC_SCRATCH_BYTES in device memory that every GPU
 * loading the library holds until the process exits; it calls no allocator.
 *   - Returns GDN_ERR_SCRATCH, before launching anything, when the problem needs
 *     more scratch than that.  gdn_workspace_bytes gives the need: 16 KiB per
 *     (64-token chunk, value head) pair, 32.5 KiB per (chunk, key head) pair for
 *     dk = 128 (16.5 KiB for dk <= 64) and a small table -- for example 64.5 MiB for
 *     one 4,096-token sequence with 32 value heads over 16 key heads.
 *   - All calls on a device share the array and it keeps the last call's contents.
 *     Calls whose GPU work overlaps (other streams, other host threads) race on it:
 *     the caller must order them.
 *   - The first call on each device looks the array's address up (with that device
 *     current); make that first call before capturing the stream into a CUDA graph.
 *   - Always the single-level path (no two-level scan).
 *   - Status bits of its kernels go to the array's first word; gdn_device_status reads
 *     and clears them with the workspace's.  gdn_set_phase_events applies as to
 *     gdn_prefill, and gdn_last_cuda_error reports its launch errors.
 */
int gdn_prefill_static(const void *q, const void *k, const void *v,
                       const float *g, const float *beta,
                       const int32_t *cu_seqlens, const float *init_state,
                       void *out, float *final_state,
                       int B, int T, int Hk, int Hv, int dk, int dv,
                       void *stream);

/*
 * Device status bits.  Every wait inside the kernels (on an MMA completion or a
 * TMA load) is bounded; a wait that runs out sets one of these bits in the first
 * word of the workspace, lets its copies and MMAs in flight land (bounded again),
 * frees its tensor memory and returns, so the context stays usable.  With
 * gdn_prefill_ws the word is the first 4 bytes of the caller's workspace; with
 * gdn_prefill_static it is the first word of the fixed array.
 */
#define GDN_STATUS_MMA_TIMEOUT 1       /* the state-carry kernel gave up waiting for an MMA phase */
#define GDN_STATUS_LOAD_TIMEOUT 2      /* the state-carry kernel gave up waiting for a tile load */
#define GDN_STATUS_PREP_LOAD_TIMEOUT 4 /* the preparation kernel gave up waiting (tile load or Gram product) */
#define GDN_STATUS_BAD_CU_SEQLENS 8    /* cu_seqlens was not 0 = cu[0] <= ... <= cu[B] = T (entries clamped) */
#define GDN_STATUS_NONFINITE_STATE 16  /* a final state of the fp16 state carry was not finite (see gdn_prefill) */
#define GDN_STATUS_SMALL_STATE 32      /* a final state of the fp16 state carry stayed below 2^-12 (see gdn_prefill) */

/*
 * gdn_device_status -- synchronise the current device, return the status bits
 * accumulated since the last call (in *status: the OR of the library workspace's
 * word and, once gdn_prefill_static has run on the device, the fixed array's) and
 * clear them.  Returns GDN_OK or GDN_ERR_LAUNCH.
 */
int gdn_device_status(int *status);

/*
 * gdn_selftest_wait_timeout -- run the bounded-wait path on purpose: one CTA
 * waits on an mbarrier that nothing completes, gives up after `max_polls` polls,
 * and records GDN_STATUS_MMA_TIMEOUT, exactly as the kernels do.  *status gets
 * the recorded bits (synchronous).  Used to test failure detection without a GPU
 * fault.
 */
int gdn_selftest_wait_timeout(int max_polls, int *status);

/*
 * gdn_selftest_static_wait_timeout -- the same bounded wait, but recording its bit in
 * the status word of gdn_prefill_static's fixed array, where a wait that runs out
 * inside that entry point would; gdn_device_status then reports it.  Synchronous;
 * allocates nothing.  Returns GDN_OK, GDN_ERR_ARG (max_polls < 1) or GDN_ERR_LAUNCH.
 */
int gdn_selftest_static_wait_timeout(int max_polls);

/*
 * gdn_debug_fail_allocations -- test hook for failure handling: the next `count`
 * device allocations the library would make (workspace, staging or scan buffers)
 * fail as if cudaMalloc had run out of memory, so the call returns GDN_ERR_ALLOC
 * before launching anything and keeps its previous buffers.  0 switches it off.
 * Returns the count that was pending.  Needs no GPU.
 */
int gdn_debug_fail_allocations(int count);

/* Segments per sequence that gdn_prefill_ex with these flags (gdn_prefill: flags = 0)
 * would use on the current device: 1 for the single-level path, P >= 2 for the
 * two-level chunk scan.  0 on bad arguments or unknown flags. */
int gdn_scan_segments(int B, int T, int Hk, int Hv, int dk, int dv, int packed, unsigned flags);

/* Bytes of device workspace gdn_prefill needs for these sizes (0 on bad arguments). */
size_t gdn_workspace_bytes(int B, int T, int Hk, int Hv, int dk, int dv, int packed);

/* Release the calling device's workspace and staging buffers (synchronises the device). */
void gdn_release_workspace(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
