/*
 * kda.h -- C ABI of the KDA (Kimi Delta Attention) forward-prefill library for
 * GB300 (sm_103a).
 *
 * The operation (per sequence n, head h, token t = 1..L_n):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * with a fp32 state S in R^{128 x 128} per (sequence, head), S_0 = the initial
 * state (zero when none is given) and final state = S_{L_n}.  It is computed
 * chunkwise with CHUNK = 16 and D = 128, forward only: a K1 stage prepares the
 * decayed q/k, applies beta and forms the WY inverse by a 16x16 unit-lower
 * triangular solve; a K2 stage runs the inter-chunk state recurrence and the
 * intra-chunk output.  Long sequences may instead run segment-parallel:
 * K1 -> pre_scan (per-segment summaries) -> merge (carries) -> segment-K2.
 * Sources: cuLA PR #103 "feat(kda/sm90): FlashKDA prefill port + intracard-CP
 * prefill" (commit notes: the K1/K2 split, CHUNK=16, D=128, forward only; the
 * segment pipeline; both states optional), flashinfer PR #4351 "fix(cake_kda):
 * support non-aligned recurrent prefill head counts" (any positive head count,
 * H=12 packed varlen, in-place state, atol = rtol = 1e-2 against a reference).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layouts (row-major, contiguous, C order), H = num_heads (equal head counts; see
 * kda_shape for grouped heads, where q, k and out have their own head counts):
 *   q, k, v, out : bf16 [T_total][H][128]   (dense input [B][T][H][128] is the same memory)
 *   g            : fp32 [T_total][H][128]   per-token log-decay (not cumulative)
 *   beta         : bf16 [T_total][H]
 *   states       : fp32 [N][H][128][128], indexed [n][h][i_k][j_v]
 *   cu_seqlens   : int32 [N + 1], cu[0] = 0, non-decreasing, cu[N] = T_total
 * bf16 tensors are passed as uint16_t pointers holding IEEE bfloat16 bits.
 * Base pointers of q, k, v, g, out, initial_state and final_state must be
 * 16-byte aligned; beta 2-byte aligned; cu_seqlens 4-byte aligned.
 *
 * Ownership: the caller owns every tensor.  The library owns only its
 * workspaces (device scratch, per device and stream, bounded in number) and
 * releases them in kda_release_workspaces().  No caller pointer is retained
 * after a call returns.
 *
 * Errors: every entry point returns a kda_status; nothing throws across the
 * ABI.  Argument validation runs on the host before any launch and has no side
 * effects when it fails; kda_last_error_message() then says why.  Device-side
 * conditions (malformed cu_seqlens contents, a bounded wait that ran out) are
 * recorded in a per-device status word read by kda_get_device_status().
 *
 * Asynchrony: kda_prefill, kda_prefill_ex and kda_decode enqueue work on `stream` and
 * return without synchronising.  `stream` is a cudaStream_t passed as void* (NULL =
 * the legacy default stream).  The current CUDA device must own all pointers.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1,     /* bad shape, null/misaligned pointer, bad option */
    KDA_ERR_ALIASING = 2,             /* out overlaps an input; partial state overlap (exact
                                         alias allowed: flashinfer PR #4351, review of
                                         CheckNoPartialOverlapOrExactAlias) */
    KDA_ERR_UNSUPPORTED_DEVICE = 3,   /* current device is not compute capability 10.3 */
    KDA_ERR_OUT_OF_MEMORY = 4,        /* a workspace allocation failed */
    KDA_ERR_CUDA = 5,                 /* a CUDA runtime call or launch failed */
    KDA_ERR_CAPTURE_NEEDS_WARMUP = 6, /* a workspace would be allocated during stream capture
                                         (flashinfer PR #4313, review of EncodeTmaPointers:
                                         warm the workspace before capture) */
    KDA_ERR_DEVICE_TIMEOUT = 7        /* a device-side bounded wait ran out (status word) */
} kda_status;

/* Problem shape.  Dense: cu_seqlens == NULL, `batch` sequences of `seq_len`
 * tokens each (T_total = batch * seq_len, N = batch).  Packed varlen:
 * cu_seqlens != NULL, batch == 1, seq_len = T_total, num_seqs = N >= 1.
 *
 * Grouped heads (the pages name GVA, unequal head counts, as a follow-up: cuLA PR #103,
 * intracard-CP planner notes).  H = num_heads counts the heads of v, g, beta and the
 * states; Hq = num_q_heads (0 means H) the heads of q; one must divide the other.  k has
 * min(Hq, H) heads and out max(Hq, H):
 *   Hq <= H  grouped value heads: state head h reads q and k head h / (H / Hq); the
 *            output has a row per state head;
 *   Hq >  H  grouped query heads: query head j reads k, v, g, beta and state head
 *            j / (Hq / H); the output has a row per query head, and the state of a group
 *            is written once.
 * Every mode takes grouped shapes; segment summaries run once per state head. */
typedef struct kda_shape {
    int32_t batch;
    int64_t seq_len;
    int32_t num_seqs;     /* varlen only; ignored for dense input */
    int32_t num_heads;    /* H >= 1; need not be a multiple of 8 */
    int32_t head_dim;     /* must be 128 (Dk = Dv = 128) */
    int32_t num_q_heads;  /* heads of q; 0 = num_heads */
} kda_shape;

/* Execution modes of kda_prefill_ex. */
#define KDA_MODE_SERIAL 0   /* one fused K1+K2 chain per (sequence, head) */
#define KDA_MODE_SEGMENT 1  /* segment-parallel: pre_scan -> merge -> segment-K2 (dense or packed varlen) */
#define KDA_MODE_AUTO 2     /* library picks serial or segment from the shape */

/* State storage types (kda_options.state_dtype, kda_decode).  A bf16 final state is
 * what the reference facade returns (flashinfer PR #4313 "feat(cake_kda): share recurrent
 * prefill kernels across SM100 family", review of kda_prefill.py).  The arithmetic stays
 * fp32 either way: a bf16 initial state is widened exactly on load, a bf16 final state
 * rounded to nearest even on store, and the prefill's own carries between segments or
 * host token blocks stay fp32. */
#define KDA_STATE_F32 0   /* fp32 [N][H][128][128] */
#define KDA_STATE_BF16 1  /* bf16 [N][H][128][128] */

typedef struct kda_options {
    int32_t mode;         /* KDA_MODE_* (default serial) */
    int32_t segment_len;  /* segment mode: tokens per segment, multiple of 16; 0 = 8192 */
    int64_t wait_limit;   /* rounds of each device barrier wait (a round sleeps at most
                             ~1 us); 0 = library default (2^22, about 4 s) */
    int32_t debug_flags;  /* 0 in normal use; KDA_DEBUG_* bits for failure-path tests */
    int32_t host_pieces;  /* kda_prefill_host: pieces the call is streamed in, 0..64;
                             0 = the library's choice, 1 = one piece; ignored by the
                             device entry points */
    int32_t state_dtype;  /* KDA_STATE_F32 (0, the default) or KDA_STATE_BF16: the type of
                             both initial_state and final_state of kda_prefill_ex and
                             kda_prefill_host */
} kda_options;

/* debug_flags bit: the kernel's first state-pipeline wait is on a barrier that nothing
 * signals, so its bounded wait runs out; the call then records KDA_ERR_DEVICE_TIMEOUT in
 * the device status word, drains its in-flight copies and returns with garbage outputs.
 * Exists to test the timeout path without faulting or hanging the GPU. */
#define KDA_DEBUG_STALL_WAIT 1

/* kda_prefill -- the forward prefill in serial mode.
 *   shape          problem shape (host pointer, read during the call only)
 *   q, k, v, g     device inputs, layouts above; may be NULL only when T_total == 0
 *   beta           device bf16 [T_total][H]
 *   scale          output scale (finite), typically 1/sqrt(128)
 *   initial_state  device fp32 [N][H][128][128] or NULL (= zero state)
 *   cu_seqlens     device int32 [N + 1] or NULL (dense input)
 *   out            device bf16 [T_total][H][128]; must not overlap any other argument
 *   final_state    device fp32 [N][H][128][128] or NULL (not written); may be the
 *                  very same pointer as initial_state (in-place update) but must not
 *                  otherwise overlap it or any input
 *   stream         cudaStream_t (as void*)
 * A sequence of length 0 writes no output and its final state equals its
 * initial state.  T_total == 0 with no final state is a no-op returning KDA_OK. */
kda_status kda_prefill(const kda_shape* shape, const uint16_t* q, const uint16_t* k,
                       const uint16_t* v, const float* g, const uint16_t* beta, float scale,
                       const float* initial_state, const int32_t* cu_seqlens, uint16_t* out,
                       float* final_state, void* stream);

/* kda_prefill_ex -- kda_prefill with options (mode, segment length, wait limit, state
 * type).  opts == NULL behaves as kda_prefill.  Segment mode takes dense or packed varlen
 * input; segment_len must be a positive multiple of 16.  initial_state and final_state
 * point at states of opts->state_dtype (fp32 by default; [N][H][128][128] either way),
 * with the aliasing rule of kda_prefill. */
kda_status kda_prefill_ex(const kda_shape* shape, const uint16_t* q, const uint16_t* k,
                          const uint16_t* v, const float* g, const uint16_t* beta, float scale,
                          const void* initial_state, const int32_t* cu_seqlens, uint16_t* out,
                          void* final_state, void* stream, const kda_options* opts);

/* kda_prefill_host -- the same computation on HOST buffers, end to end.
 * Every tensor pointer (including cu_seqlens) is a host pointer with the
 * layouts above, the states of opts->state_dtype as in kda_prefill_ex; page-locked
 * memory gives full copy bandwidth.  The call
 * copies the inputs into a library-owned device arena, runs the prefill on
 * `stream`, copies out (and final_state when non-NULL) back, and synchronises
 * `stream` before returning.
 *   Streaming: in serial mode (chosen, or picked by KDA_MODE_AUTO) a call whose
 *   inputs reach 32 MiB runs in pieces (8 by default, opts->host_pieces to set):
 *   each piece's inputs copy in on a library stream while earlier pieces compute
 *   on `stream` and their outputs copy out on a second library stream, so input
 *   copies, output copies and kernels overlap.  Several sequences split into
 *   ranges of whole sequences, balanced by tokens: the results are bit-identical
 *   to one kda_prefill_ex call.  One sequence splits into token blocks of whole
 *   16-token chunks, the fp32 state carried from block to block in the arena:
 *   the results equal one call up to rounding (each block restarts the chunk
 *   pipeline from the stored state).  Segment mode runs in one piece.
 *   Both copy streams, their events and the arena are kept per (device, stream)
 *   and reused; kda_release_workspaces() frees them.  Concurrent calls with the
 *   same stream from several threads are not supported. */
kda_status kda_prefill_host(const kda_shape* shape, const uint16_t* q, const uint16_t* k,
                            const uint16_t* v, const float* g, const uint16_t* beta,
                            float scale, const void* initial_state,
                            const int32_t* cu_seqlens, uint16_t* out, void* final_state,
                            void* stream, const kda_options* opts);

/* kda_prefill_segment_noalloc -- segment-parallel prefill that allocates no device
 * memory.  The pages have no counterpart.  Some callers of a prefill cannot call
 * cudaMalloc: applications whose caching allocator owns all of device memory and
 * forbids side allocations, real-time services that must not risk an allocation failure
 * or the device synchronisation a cudaMalloc can imply in the middle of a request, and
 * plugin hosts that give a library no allocation rights.  This entry point is segment
 * mode (kda_prefill_ex with KDA_MODE_SEGMENT, the same kernels on the same plan) with its
 * scratch in one fixed 32 MiB device array inside the library instead of a workspace.
 *   Arguments as kda_prefill for dense input (no cu_seqlens); segment_len is the
 *   segment length in tokens, a positive multiple of 16.
 *   Limit: B * H * (3 * nseg - 2) <= 512, nseg = ceil(seq_len / segment_len) (each
 *   term a 64 KiB fp32 state); larger shapes return KDA_ERR_INVALID_ARGUMENT before any
 *   device work.  A single segment needs no scratch.
 *   The array is shared by every call in the process and keeps the last call's
 *   contents; no part of it needs to start at zero (each call writes every byte it
 *   reads before reading it).  Calls that overlap on the GPU (other streams, other
 *   threads) race on it: serialise them.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current, once.  Every GPU that loads the
 *   library holds the 32 MiB until exit. */
kda_status kda_prefill_segment_noalloc(const kda_shape* shape, const uint16_t* q,
                                       const uint16_t* k, const uint16_t* v, const float* g,
                                       const uint16_t* beta, float scale,
                                       const float* initial_state, uint16_t* out,
                                       float* final_state, int32_t segment_len, void* stream);

/* (kda_decode with KDA_STATE_BF16 rounds the state to bf16 after every token.) */

/* kda_decode -- the recurrent step for a few tokens (typically one) of each sequence,
 * the inner step of autoregressive decoding: per (sequence, head) and token, the
 * recurrence at the top of this header (Kimi Delta Attention: the gated delta rule
 * with a per-channel decay, the method cuLA PR #103 "feat(kda/sm90): FlashKDA prefill
 * port + intracard-CP prefill" computes chunkwise), applied token by token to
 * a state that stays resident on the device.  The pages mention a decode registration
 * beside the prefill (flashinfer PR #4313 "feat(cake_kda): share recurrent prefill
 * kernels across SM100 family", publication notes) and a bf16 final state in the
 * reference facade (flashinfer PR #4313, review of kda_prefill.py); neither gives the
 * kernel, so this one is the recurrence itself, HBM-bound on the state.
 *   shape          dense only: batch = N sequences, seq_len = T tokens of each
 *                  (T >= 0; the cost grows linearly in T, use kda_prefill for long
 *                  inputs), num_seqs ignored, head_dim 128, num_heads >= 1
 *   q, k, v, g     device, layouts as kda_prefill ([N][T][H][128]); may be NULL only
 *                  when N * T == 0
 *   beta           device bf16 [N][T][H]
 *   scale          output scale (finite)
 *   initial_state  device [N][H][128][128] of state_dtype, or NULL (zero state)
 *   final_state    device, same layout and type, or NULL (not written); may be the very
 *                  same pointer as initial_state (the usual in-place update of a state
 *                  cache) but must not otherwise overlap it or any input
 *   state_dtype    KDA_STATE_F32 or KDA_STATE_BF16, for both state pointers
 *   out            device bf16 [N][T][H][128]; must not overlap any other argument
 * Alignment as kda_prefill (16 bytes for every tensor but beta).  Asynchronous on
 * `stream`; no workspace, no device status word.  T == 0 copies (or zero-fills, with
 * no initial state) the state; with T == 0 and no final state it is a no-op.
 * Errors: KDA_ERR_INVALID_ARGUMENT (shape, pointer, state_dtype), KDA_ERR_ALIASING,
 * KDA_ERR_UNSUPPORTED_DEVICE, KDA_ERR_CUDA (launch). */
kda_status kda_decode(const kda_shape* shape, const uint16_t* q, const uint16_t* k,
                      const uint16_t* v, const float* g, const uint16_t* beta, float scale,
                      const void* initial_state, void* final_state, int32_t state_dtype,
                      uint16_t* out, void* stream);

/* Bytes of device workspace a call with this shape and these options uses
 * (0 for serial mode).  The segment pipeline's scratch (per-segment summaries,
 * transitions and carries: cuLA PR #103, review of the CP driver's _get_scratch, which
 * sizes b_seg, m_seg, carries and seg_final per shape) is reported here so a caller can
 * budget it before the first call.  A shape with num_seqs > 0 is taken as packed varlen
 * input (segment mode then sizes for at most num_seqs + seq_len / segment_len segments).
 * kda_prefill_host holds, besides, an arena the size of its tensors.  No device work,
 * except that KDA_MODE_AUTO reads the current device's resident cluster count to
 * resolve the plan; *bytes is written on success. */
kda_status kda_workspace_bytes(const kda_shape* shape, const kda_options* opts, size_t* bytes);

/* The execution plan KDA_MODE_AUTO picks for this shape on a device that holds
 * `resident_clusters` co-resident clusters of the fused kernel (kda_prefill_ex uses
 * the current device's count): KDA_MODE_SERIAL (*segment_len = 0) or
 * KDA_MODE_SEGMENT with *segment_len tokens per segment.  Packed varlen input
 * (`varlen` != 0) is always serial.  The cost model counts chunk periods of one
 * state chain: every pass of the fused kernel costs about the same per chunk,
 * clusters beyond the resident count run in further waves, and the merge walks a
 * chain's segments in order (segment-parallel prefill, cuLA PR #103 "intracard-CP
 * prefill", planner notes).  Candidates: for every segment count, the shortest
 * multiple of 16 tokens (at least 512) that covers the sequence in that many
 * segments, under a 4 GiB workspace cap; segment mode is chosen only when it beats
 * serial by 20%.  Host only, no device work.  Errors:
 * KDA_ERR_INVALID_ARGUMENT for a bad shape, NULL outputs or resident_clusters < 1. */
kda_status kda_plan(const kda_shape* shape, int32_t varlen, int32_t resident_clusters, int32_t* mode,
                    int32_t* segment_len);

/* kda_plan_varlen -- the plan for packed varlen input whose offsets the caller holds on
 * the host (`host_cu_seqlens`, int32 [N + 1], host memory): what kda_prefill_host with
 * KDA_MODE_AUTO runs for such input (the device entry points cannot see device-resident
 * lengths and keep varlen input serial).  Same units as kda_plan: serial costs the longer
 * of the longest chain and all chains over the resident clusters; a segment plan of
 * length L gives sequence n max(1, ceil(len_n / L)) segment rows (segment-parallel
 * prefill for packed batches, cuLA PR #103 "intracard-CP prefill", planner notes), its two
 * summary passes run every row but each sequence's last, and segment mode is chosen only
 * when it beats serial by 20%.  Host only.  Errors: KDA_ERR_INVALID_ARGUMENT for a bad
 * shape (varlen rules), NULL pointers, malformed offsets or resident_clusters < 1. */
kda_status kda_plan_varlen(const kda_shape* shape, const int32_t* host_cu_seqlens, int32_t resident_clusters,
                           int32_t* mode, int32_t* segment_len);

/* Reads and clears the device status word of the current device after
 * synchronising `stream`.  *code receives KDA_OK, KDA_ERR_INVALID_ARGUMENT
 * (malformed cu_seqlens contents seen by a kernel) or KDA_ERR_DEVICE_TIMEOUT.
 * The pages validate on the host and abort the call with a message (flashinfer PR
 * #4313, review of flashkda_binding_common.cuh: the TVM_FFI_ICHECK target, shape and
 * capacity checks) and record a device-side hazard only in review (flashinfer PR #4351,
 * review of the beta packing: a kernel that reads uninitialised workspace); conditions
 * that only a kernel can see (cu_seqlens contents, a bounded wait that ran out) are
 * therefore kept in a per-device word the kernels write and this call reads. */
kda_status kda_get_device_status(void* stream, int32_t* code);

/* Frees every workspace the library holds on `device` (-1 = all devices).
 * The caller must ensure no call using them is still running.  Workspaces are keyed by
 * (device, stream, kind), at most 8 of them, least recently used evicted first: the
 * pages' scratch cache raced across streams because its key lacked the stream (cuLA PR
 * #103, review of _get_scratch) and their per-stream workspace maps grew without bound
 * (flashinfer PR #4313, review of kda_prefill.py, which asks for a bound or an eviction
 * path); this call is the explicit release. */
kda_status kda_release_workspaces(int32_t device);

/* Static description of a status code.  The pages' bindings fail with a message per
 * check (flashinfer PR #4313, review of flashkda_binding_common.cuh; flashinfer PR #4351,
 * review of CheckNoPartialOverlapOrExactAlias for KDA_ERR_ALIASING; the capture guard
 * of EncodeTmaPointers, "prepare_descriptors must be 0 during CUDA graph capture", for
 * KDA_ERR_CAPTURE_NEEDS_WARMUP); across a C ABI that becomes a code plus this text. */
const char* kda_status_string(kda_status status);

/* Message of the last failing call on this host thread ("" if none): the specific
 * reason (which argument, which size), as the pages' per-check messages give it
 * (flashinfer PR #4313, review of flashkda_binding_common.cuh). */
const char* kda_last_error_message(void);

/* Library version, e.g. "0.1.0". */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
