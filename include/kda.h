/*
 * kda.h -- C ABI of the KDA (Kimi Delta Attention) recurrence library for
 * NVIDIA GB300 (sm_103a).  libkda.so exports exactly the functions below.
 *
 * The operation (source: "[논문 리뷰] Kimi K3 Technical Report",
 * jw9603.github.io, section 3.2 "KDA의 핵심 상태 업데이트"; delta form in
 * section 3.3; alpha = exp(g) in section 3.5).  Per sequence and head, with a
 * state S in R^{d_k x d_v} whose rows are key channels:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t                  (read after token t's write)
 *     alpha_t = exp(log_alpha_t)       (per key channel), beta_t a scalar.
 *
 * Conventions shared by every call:
 *  - All pointers are DEVICE pointers unless stated otherwise (only
 *    kda_prefill_host takes host buffers); the caller owns every buffer.  The
 *    library allocates nothing and keeps no state between calls other than
 *    cached device attributes.
 *  - Work is enqueued on `stream`; no call synchronises the host.  Argument
 *    errors are returned synchronously before anything is launched; a launch
 *    failure returns KDA_ERR_CUDA.  Nothing is thrown across the ABI.
 *  - Tensors are dense, row-major, with the last index fastest:
 *      q, k, log_alpha : [T_tot, H, d_k]
 *      v, o            : [T_tot, H, d_v]
 *      beta            : [T_tot, H]
 *      states          : [N, H, d_k, d_v]   fp32
 *    q, k, v share one dtype and o has the output dtype (kda_dtype_t);
 *    log_alpha, beta and states are always fp32.  Base pointers must be
 *    16-byte aligned.
 *  - Preconditions that are documented, not checked on the device:
 *    -5 <= log_alpha <= 0 (the lower-bounded decay of section 3.5); k is
 *    L2-normalised and q pre-scaled by the caller (the op uses them as given);
 *    beta is any finite value (beta up to 2 gives a reflection, "Kimi 모델
 *    분석", rlaope.github.io, section "반사가 계층을 바꿈"); inputs finite.
 *    On the tensor-core path (bf16 q/k/v with d_k = d_v = 128, see
 *    kda_prefill's Paths) v, the states (S0 and every state the recurrence
 *    passes through) and the chunk products formed from them enter the
 *    tensor cores as fp16, so |v| and every state entry must stay below
 *    65504, the largest finite fp16 value; beyond it the results are not
 *    finite.  The fp32 CUDA-core path has no such limit: a caller whose
 *    values may exceed it passes fp32 inputs (KDA_FP32).
 *  - Supported shapes: every dtype code with d_k = d_v in {16, 32, 64, 128}.
 *    Anything else returns KDA_ERR_UNSUPPORTED.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null required pointer, bad count, misalignment */
    KDA_ERR_UNSUPPORTED = 2,   /* dtype / head size not implemented */
    KDA_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small */
    KDA_ERR_CUDA = 4           /* a kernel launch failed (cudaGetLastError) */
} kda_status_t;

typedef enum {
    KDA_BF16 = 0,              /* q, k, v, o are bfloat16 */
    KDA_FP32 = 1,              /* q, k, v, o are float32  */
    KDA_BF16_F32OUT = 2        /* q, k, v are bfloat16, o is float32 */
} kda_dtype_t;

/* Bytes of device workspace kda_prefill needs for num_seqs sequences of H
 * heads.  The workspace always holds the varlen work list (sequences ordered
 * longest first, counters, an error word).  When d_k = d_v = 128 and the
 * num_seqs x H (sequence, head) units fill at most half of the current
 * device's SMs (and num_seqs <= 128), the value also covers the operand ring
 * of the producer / consumer prefill kernel (tens of MB at most; the size
 * depends on the SM count).  Returns 0 when num_seqs < 1. */
size_t kda_prefill_workspace_bytes(int32_t num_seqs, int32_t H, int32_t d_k,
                                   int32_t d_v);

/* Chunked prefill over packed variable-length sequences.
 *
 * Computes o_t for every token of every sequence and, optionally, the state
 * after each sequence's last token.  The chunkwise-parallel form used on the
 * GPU ("Kimi 모델 분석", section "순환을 GPU에 올리기": chunks of 64 tokens,
 * intra-chunk matrix products, inter-chunk state carry) gives the same result
 * as the token-by-token recurrence up to rounding.
 *
 *   q, k, v       [T_tot, H, d] in the input dtype of `dtype`
 *   log_alpha     [T_tot, H, d_k] fp32, g = ln(alpha)
 *   beta          [T_tot, H] fp32
 *   S0            [N, H, d_k, d_v] fp32 initial states, or NULL for zeros
 *   cu_seqlens    device int32 [N+1]: cu[0] = 0, non-decreasing,
 *                 cu[N] = total_tokens; sequence n owns tokens
 *                 cu[n] .. cu[n+1]-1.  NULL means one sequence (N must be 1).
 *                 Empty sequences are allowed (their S_final = S0).
 *   num_seqs      N >= 1;  total_tokens >= 0;  H >= 1
 *   o             [T_tot, H, d_v] in the output dtype of `dtype` (written)
 *   S_final       [N, H, d_k, d_v] fp32, or NULL when not wanted.  May alias
 *                 S0 exactly (in-place resume); any other overlap is an error
 *                 the library cannot detect.
 *   workspace     device buffer of at least 256 + 256 * ceil(N / 64) bytes
 *                 (the work list), 256-byte aligned; its contents on entry do
 *                 not matter and are overwritten.  It must not be shared by
 *                 calls that may run concurrently.  A workspace of
 *                 kda_prefill_workspace_bytes(...) bytes lets the call use the
 *                 producer / consumer kernel where it applies (see Paths); a
 *                 smaller one selects the single-CTA kernel, with the same
 *                 results.
 *
 * If cu_seqlens violates its contract the kernels write nothing and set the
 * 32-bit word at byte offset 4 of the workspace to a nonzero value (it is
 * cleared to zero by every call that finds cu_seqlens valid).  The 32-bit word
 * at byte offset 8 gets bit 1 set if a wait inside the tensor-core kernel gave
 * up after two seconds (which means a library fault; the kernel then stops
 * early and its outputs are incomplete); the library never clears it, so a
 * caller who wants to watch it zeroes it first.  Both are device-side flags:
 * reading them needs a synchronisation by the caller.
 *
 * Paths: bf16 inputs with d_k = d_v = 128 run on the tensor cores (tcgen05,
 * chunks of 64 tokens).  With few (sequence, head) units (at most half the
 * SM count) and a full-size workspace, one cooperative launch of one CTA per
 * SM splits each chunk's work: producer CTAs compute the parts that do not
 * depend on the state and hand them, through the workspace, to one consumer
 * CTA per unit that carries the state; otherwise one CTA per unit does both.
 * Every other supported shape, and every call made while the environment
 * variable KDA_FORCE_SIMT is set, runs the fp32 CUDA-core path (chunks of 16
 * tokens).  All paths compute the same result up to rounding (the two
 * tensor-core kernels bit for bit).
 */
kda_status_t kda_prefill(const void *q, const void *k, const void *v,
                         const float *log_alpha, const float *beta,
                         const float *S0, const int32_t *cu_seqlens,
                         int32_t num_seqs, int64_t total_tokens, int32_t H,
                         int32_t d_k, int32_t d_v, kda_dtype_t dtype, void *o,
                         float *S_final, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/* kda_prefill that also records prefix states ("snapshots") for a prefix
 * cache: the state of each sequence after every `interval` tokens, which a
 * serving stack stores and later restores with S0 to resume from that prefix
 * ("[논문 리뷰] Kimi K3 Technical Report", section 13, the KDA-aware prefix
 * cache; "Kimi 모델 분석", section "요약본 저장 위치").
 *
 * Arguments, layouts and results are those of kda_prefill, plus:
 *   interval      a positive multiple of 64 (so that every snapshot falls on
 *                 a chunk boundary of every path); else KDA_ERR_INVALID_ARG.
 *   snap_offsets  device int32 [N+1] with snap_offsets[0] = 0 and
 *                 snap_offsets[n+1] - snap_offsets[n] = floor(len_n / interval);
 *                 required when cu_seqlens is given, ignored (offset 0)
 *                 otherwise.  Checked on the device: a mismatch is reported
 *                 like an invalid cu_seqlens (workspace word at byte 4, nothing
 *                 written).
 *   snapshots     device fp32 [snap_offsets[N], H, d_k, d_v] (written).
 *                 Snapshot j of sequence n, at snap_offsets[n] + j, is the
 *                 state after that sequence's first (j + 1) * interval tokens;
 *                 when interval divides the length, the last one equals the
 *                 sequence's S_final.  Must not overlap the other buffers.
 * The outputs o and S_final are those kda_prefill computes, bit for bit. */
kda_status_t kda_prefill_snapshots(const void *q, const void *k, const void *v,
                                   const float *log_alpha, const float *beta,
                                   const float *S0, const int32_t *cu_seqlens,
                                   int32_t num_seqs, int64_t total_tokens,
                                   int32_t H, int32_t d_k, int32_t d_v,
                                   kda_dtype_t dtype, void *o, float *S_final,
                                   int32_t interval, const int32_t *snap_offsets,
                                   float *snapshots, void *workspace,
                                   size_t workspace_bytes, cudaStream_t stream);

/* kda_prefill with the steps in front of the recurrence fused into the
 * kernels ("Kimi 모델 분석", section "커널 최적화": one kernel for the KDA
 * layer): the lower-bounded decay of "[논문 리뷰] Kimi K3 Technical Report",
 * section 3.5,
 *     g = -5 Sigmoid(e^A z),   alpha = exp(g) in (e^-5, 1),
 * and the L2 normalisation of q and k over the key channels (q then
 * multiplied by q_scale, typically d_k^-1/2).
 *
 * Arguments and results are those of kda_prefill, except:
 *   q, k   raw (not normalised) in the input dtype; each row of d_k values
 *          must be nonzero
 *   z      [T_tot, H, d_k] fp32, the gate pre-activation (in place of
 *          log_alpha)
 *   A      [H, d_k] fp32, 16-byte aligned (a per-head A is its value repeated
 *          over the channels); NULL is KDA_ERR_INVALID_ARG
 *   q_scale  the factor applied to the normalised q
 * Normalised q and k enter the products in fp32 before any rounding to the
 * operand precision, so the result is at least as accurate as calling
 * kda_prefill on q, k normalised and rounded by the caller. */
kda_status_t kda_prefill_fused(const void *q, const void *k, const void *v,
                               const float *z, const float *A, const float *beta,
                               const float *S0, const int32_t *cu_seqlens,
                               int32_t num_seqs, int64_t total_tokens, int32_t H,
                               int32_t d_k, int32_t d_v, kda_dtype_t dtype,
                               float q_scale, void *o, float *S_final,
                               void *workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/* Bytes of device workspace kda_prefill_segmented needs for one sequence of
 * total_tokens tokens and H heads cut into `segments` segments (<= 0: the
 * number the call would choose).  When the call would not cut the sequence
 * (see below) this is kda_prefill_workspace_bytes(1, H, d_k, d_v).  The
 * workspace holds, besides kda_prefill's, two fp32 copies of the outputs
 * (8 * total_tokens * H * d_v bytes) and 3 * segments states per head. */
size_t kda_prefill_segmented_workspace_bytes(int64_t total_tokens, int32_t H,
                                             int32_t d_k, int32_t d_v,
                                             int32_t segments);

/* kda_prefill of ONE sequence with its chunks cut into `segments` groups
 * that run at once (chunk-group parallel prefill): the form for a short
 * prompt whose chunk chain, not the amount of work, sets the time.
 *
 * The recurrence carries only the state from chunk to chunk ("Kimi 모델
 * 분석", section "순환을 GPU에 올리기") and is linear in (S, v), so each
 * segment g >= 1 runs twice on the same chunk operands: from S = 0 (its local
 * outputs and final state L_g) and, with v = 0, from S = I (the product
 * Phi_g of its token transitions and, per token, Phi_t^T q_t).  A scan then
 * gives the state entering each segment, S_1 = L_0, S_{g+1} = Phi_g S_g +
 * L_g, and a fix-up adds S_g^T Phi_t^T q_t to the local outputs.  This is the
 * one-GPU form of what "[논문 리뷰] Kimi K3 Technical Report", section 13,
 * calls KDA context parallelism.  The result equals kda_prefill's up to
 * rounding.
 *
 * Arguments and layouts are those of kda_prefill with N = 1 (no cu_seqlens),
 * plus:
 *   segments   the number of segments, >= 2 (used when every segment has a
 *              chunk and the 2 * segments - 1 chains of each head fill at
 *              most half of the SMs), or <= 0 to let the library choose: the
 *              most segments for which those chains fill about a third of
 *              the SMs and every segment has at least 32 chunks (one GB300:
 *              2 at H = 16, 3 at H = 8, 6 at H = 4; none at H >= 24 or below
 *              4,096 tokens, where cutting does not pay).
 *   workspace  kda_prefill_segmented_workspace_bytes(...) bytes, 256-byte
 *              aligned, not shared with concurrent calls.
 * When the shape cannot be cut (not bf16 inputs with d_k = d_v = 128, too
 * many heads for two segments, a single chunk) or the workspace is smaller
 * than that size, the call is kda_prefill, with the same results.  The
 * device-side status words are those of kda_prefill (workspace bytes 4 and
 * 8).  Launches: the work list, the cut prefill, the scan and the fix-up. */
kda_status_t kda_prefill_segmented(const void *q, const void *k, const void *v,
                                   const float *log_alpha, const float *beta,
                                   const float *S0, int64_t total_tokens,
                                   int32_t H, int32_t d_k, int32_t d_v,
                                   kda_dtype_t dtype, void *o, float *S_final,
                                   int32_t segments, void *workspace,
                                   size_t workspace_bytes, cudaStream_t stream);

/* Device staging bytes kda_prefill_host needs for segments of
 * segment_tokens tokens (a multiple of 64): two input and two output segment
 * buffers, two state buffers and a prefill workspace.  0 for bad arguments. */
size_t kda_prefill_host_staging_bytes(int32_t H, int32_t d_k, int32_t d_v,
                                      kda_dtype_t dtype, int64_t segment_tokens);

/* kda_prefill of ONE sequence whose token inputs and output live in HOST
 * memory (a long prompt that arrives from the host).  The sequence is cut into
 * segments of segment_tokens tokens (a positive multiple of 64) that flow
 * through a pipeline: copies in on `h2d`, kda_prefill on `compute` (the state
 * carried from segment to segment, "Kimi 모델 분석", section "순환을 GPU에
 * 올리기": only the state passes between chunks), copies out on `d2h`, so that
 * the three overlap.  The result equals kda_prefill over the whole sequence
 * bit for bit.
 *
 *   q, k, v, log_alpha, beta, o   HOST pointers, layouts of kda_prefill with
 *                 N = 1 (page-locked memory for full copy bandwidth; pageable
 *                 memory works, with slower copies).  Page-locked pages that
 *                 the CPU has never written are mapped for the GPU on first
 *                 access, and the first passes over them copy at a fraction of
 *                 the link rate; buffers the host filled run at full rate.
 *   S0, S_final   DEVICE [H, d_k, d_v] fp32 or NULL, as in kda_prefill
 *   staging       DEVICE buffer of kda_prefill_host_staging_bytes(...) bytes,
 *                 256-byte aligned, not shared with concurrent calls
 *   compute, h2d, d2h  three streams (distinct for overlap).  When `compute`
 *                 is complete, so is everything the call enqueued.  The first
 *                 copy in waits for the work already on `compute` (a previous
 *                 call on the same staging area, the producer of S0).
 * The pipeline fills and drains over one segment, so shorter segments bound
 * the overhead; 16384 tokens keep each segment's launches well above their
 * fixed cost.
 * The call creates six CUDA events and releases them before it returns; it
 * allocates no memory and does not synchronise the host.  Argument errors are
 * returned before anything is enqueued. */
kda_status_t kda_prefill_host(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta,
                              const float *S0, int64_t total_tokens, int32_t H,
                              int32_t d_k, int32_t d_v, kda_dtype_t dtype,
                              void *o, float *S_final, void *staging,
                              size_t staging_bytes, int64_t segment_tokens,
                              cudaStream_t compute, cudaStream_t h2d,
                              cudaStream_t d2h);

/* One decode step for N independent sequences (one new token each): the
 * recurrence above applied once per (sequence, head), state updated in place.
 * Decode reads and writes a fixed 2 * 4 * d_k * d_v bytes of fp32 state per
 * (sequence, head) whatever the context length ("Kimi 모델 분석", section
 * "Decoding이 왜 느린가"); it is memory-bound.
 *
 *   q, k          [N, H, d_k], v: [N, H, d_v], in the input dtype of `dtype`
 *   log_alpha     [N, H, d_k] fp32;  beta: [N, H] fp32
 *   S_inout       [N, H, d_k, d_v] fp32, read and overwritten with S_t
 *   o             [N, H, d_v] in the output dtype of `dtype` (written); must
 *                 not overlap S_inout
 */
kda_status_t kda_decode_step(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta,
                             float *S_inout, int32_t N, int32_t H, int32_t d_k,
                             int32_t d_v, kda_dtype_t dtype, void *o,
                             cudaStream_t stream);

/* kda_decode_step with the gate prologue fused (see kda_prefill_fused): z
 * [N, H, d_k] fp32 in place of log_alpha, A [H, d_k] fp32, raw q and k
 * (nonzero rows), q_scale. */
kda_status_t kda_decode_step_fused(const void *q, const void *k, const void *v,
                                   const float *z, const float *A,
                                   const float *beta, float *S_inout, int32_t N,
                                   int32_t H, int32_t d_k, int32_t d_v,
                                   kda_dtype_t dtype, float q_scale, void *o,
                                   cudaStream_t stream);

/* Several decode tokens per sequence, keeping the state after every token:
 * the verification step of speculative decoding, which must be able to
 * return to the state after any accepted prefix of the draft, since the state
 * is overwritten in place and cannot be truncated ("[논문 리뷰] Kimi K3
 * Technical Report", section 13, speculative decoding replay; "Kimi 모델
 * 분석", section "Dspark 투기적 디코딩").  Token t of each sequence is one
 * decode step (the recurrence above) from the state after token t - 1.
 *
 *   q, k, log_alpha [N, Ts, H, d_k]; v [N, Ts, H, d_v]; beta [N, Ts, H]
 *                   in the dtypes of kda_decode_step
 *   S_in            [N, H, d_k, d_v] fp32, the state before the first token
 *                   (read only)
 *   o               [N, Ts, H, d_v] in the output dtype (written)
 *   states          [N, Ts, H, d_k, d_v] fp32: states[n, t] is the state after
 *                   token t of sequence n (written)
 * No two of S_in, o and states may overlap.  The launch reads S_in once and
 * writes Ts states: 4 (1 + Ts) d_k d_v bytes per (sequence, head). */
kda_status_t kda_decode_multi(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta,
                              const float *S_in, int32_t N, int32_t Ts,
                              int32_t H, int32_t d_k, int32_t d_v,
                              kda_dtype_t dtype, void *o, float *states,
                              cudaStream_t stream);

/* After verification: the state of each sequence after its accepted prefix.
 * S_out[n] = states[n, accept[n] - 1] when accept[n] > 0, else S_in[n]
 * (all heads).  accept: device int32 [N] in [0, Ts] (values outside are
 * clamped).  S_out may be S_in itself (in-place update of the cache) and must
 * not overlap `states`. */
kda_status_t kda_state_gather(const float *states, const float *S_in,
                              const int32_t *accept, int32_t N, int32_t Ts,
                              int32_t H, int32_t d_k, int32_t d_v, float *S_out,
                              cudaStream_t stream);

/* kda_prefill for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point: it exists for callers
 * that cannot call cudaMalloc, such as an inference engine that plans all of
 * its device memory once at start-up and forbids allocation afterwards, or a
 * plugin host that passes a library only the operation's inputs and outputs.
 *
 * Same arguments, layouts and results as kda_prefill, without the workspace:
 * the work list lives in a fixed scratch array inside the library's device
 * image (about 16 KiB, room for at most 4096 sequences; every GPU that loads
 * the library keeps it until the process exits).  num_seqs above 4096
 * returns KDA_ERR_WORKSPACE.  The first call on each device, with that device
 * current, looks the array's device address up (cudaGetSymbolAddress, which
 * may load the library's device code), so make that first call before any
 * stream capture; the address is looked up again only when the device's
 * current context changes (after cudaDeviceReset, for example).  All calls on
 * a device share the array: calls that may overlap on the GPU race on it and
 * must be ordered by the caller.  Nothing is allocated and nothing in the
 * array needs clearing between calls.  KDA_ERR_CUDA is returned if the
 * device or the array's address cannot be determined.
 *
 * What differs from kda_prefill:
 *  - The device-side status words (invalid cu_seqlens, a wait that gave up)
 *    live in the private array and cannot be read by the caller.  An invalid
 *    cu_seqlens therefore still returns KDA_OK, with o and S_final not
 *    written; a caller that cannot vouch for its cu_seqlens validates it
 *    before the call, or calls kda_prefill.
 *  - The array has room for the work list only, never for the operand ring
 *    of the producer / consumer kernel, so every call takes the one-CTA-per-
 *    (sequence, head) kernel.  The results are the same, but a batch with few
 *    units (one long sequence of 32 heads, say) keeps only that many SMs
 *    busy: several times slower than kda_prefill with a full workspace. */
kda_status_t kda_prefill_noalloc(const void *q, const void *k, const void *v,
                                 const float *log_alpha, const float *beta,
                                 const float *S0, const int32_t *cu_seqlens,
                                 int32_t num_seqs, int64_t total_tokens,
                                 int32_t H, int32_t d_k, int32_t d_v,
                                 kda_dtype_t dtype, void *o, float *S_final,
                                 cudaStream_t stream);

/* A static, human-readable name for a status code (never NULL). */
const char *kda_status_string(kda_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
