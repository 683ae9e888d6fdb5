// kda_internal.cuh -- declarations shared by the library's translation units.
// Nothing here is part of the public ABI (include/kda.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "kda.h"

namespace kda {

// Workspace layout used by kda_prefill (see kda_prefill_workspace_bytes):
//   byte 0   : int32 work counter (persistent kernels take items from it)
//   byte 4   : int32 error word (nonzero => cu_seqlens violated its contract)
//   byte 8   : int32 timeout word (bit 1 set => a device-side wait gave up)
//   byte 12  : int32 longest sequence length (written by the work-list kernel)
//   byte 16  : int64 job counter of the split kernel's producers
//   byte 24  : int32 abort word of the split kernel (nonzero => a CTA gave up
//              and the others stop); cleared by the work-list kernel
//   byte 256 : int32 order[N], sequence indices, longest first
// and, when the split kernel is used (split_plan below), after order[]:
//   flags    : int32 full[U][R], int32 consumed[U]   (U = N H units, R = ring depth)
//   ring     : [U][R][2 steps][kSplitStepBytes] chunk operands, 1024-aligned
constexpr size_t kWsHeaderBytes = 256;
constexpr int kWsCounterWord = 0;
constexpr int kWsErrorWord = 1;
constexpr int kWsTimeoutWord = 2;
constexpr int kWsMaxLenWord = 3;
constexpr int kWsJobWord = 4;          // 64-bit, words 4 and 5
constexpr int kWsAbortWord = 6;
// Sequences are ordered longest-first when N <= this; above it the order is
// the input order (the rank sort is O(N^2) on one CTA).
constexpr int kMaxSortedSeqs = 2048;

inline size_t workspace_bytes(int32_t num_seqs) {
    if (num_seqs < 1) return 0;
    size_t order = ((size_t)num_seqs * sizeof(int32_t) + 255) / 256 * 256;
    return kWsHeaderBytes + order;
}

// The split (producer / consumer) tensor-core prefill: one consumer CTA per
// (sequence, head) unit and `producers` CTAs on the other SMs, handing chunk
// operands over through a ring of `ring` chunk slots per unit in the
// workspace.  Used when the units fill at most half of the SMs.
constexpr size_t kSplitStepBytes = 66560;       // one step's operand block (65 KB)
constexpr int kSplitMaxRing = 32;

struct SplitPlan {
    int32_t units, producers, ring;
    int32_t groups;       // ring groups (one per unit, or per segment and head)
    size_t flags_off, ring_off, bytes;
};

// The producers keep each sequence's token range in shared memory.
constexpr int kSplitMaxSeqs = 128;

inline bool split_plan(int32_t num_seqs, int32_t H, int sms, SplitPlan* plan) {
    if (num_seqs > kSplitMaxSeqs) return false;
    if (num_seqs < 1 || H < 1 || sms < 3) return false;
    const long long units = (long long)num_seqs * H;
    if (units > sms / 2) return false;
    SplitPlan p;
    p.units = (int32_t)units;
    p.producers = sms - p.units;
    // Producers claim chunks in chunk-major order, so about producers / units
    // chunks of each unit are being computed; each producer may also hold its
    // next claim and a finished job not yet published.  The ring holds three
    // times producers / units plus the consumer's own pipeline: with fewer
    // slots, producers block on full slots while holding jobs other consumers
    // wait for, and the launch slows down by about half.
    const int ahead = (p.producers + p.units - 1) / p.units;
    p.ring = 3 * ahead + 4;
    if (p.ring < 4) p.ring = 4;
    if (p.ring > kSplitMaxRing) p.ring = kSplitMaxRing;
    p.groups = p.units;
    p.flags_off = workspace_bytes(num_seqs);
    const size_t nflags = (size_t)p.units * (p.ring + 1);
    p.ring_off = (p.flags_off + nflags * sizeof(int32_t) + 1023) / 1024 * 1024;
    p.bytes = p.ring_off + (size_t)p.units * p.ring * 2 * kSplitStepBytes;
    *plan = p;
    return true;
}

// Chunk-group parallel prefill of one sequence (kda_prefill_segmented): the
// sequence is cut into G segments of seg_chunks chunks.  Segment 0 runs from
// the caller's S0 and writes the final outputs.  Every later segment g runs
// twice on the producers' shared operands: a local run from S = 0 (outputs
// o_loc, final state L_g) and an identity run with v = 0 from S = I (outputs
// qt = Phi_t^T q_t, final state M_g = Phi_g, the segment's transition).  By
// linearity the true state entering segment g is S_g = M_{g-1} S_{g-1} +
// L_{g-1} (S_1 = L_0) and the true output is o_t = o_loc,t + S_g^T qt_t.
struct SegArgs {
    int32_t G;            // segments (1 or less: not segmented)
    int32_t seg_chunks;   // chunks per segment (even: segments are whole 128-token tiles)
    __half* o_aux;        // [2][T][H][d_v] fp16: o_loc, qt (segments >= 1)
    float* st_aux;        // [2][G][H][d_k][d_v] fp32: L_g, M_g (L_0: segment 0's state)
};

// Consumer units of a segmented launch: H units of segment 0 (mode 0), then
// per later segment H local units (mode 1) and H identity units (mode 2).
struct SegUnit {
    int g, mode, h;
};

__host__ __device__ __forceinline__ int seg_units(int H, int G) { return H * (2 * G - 1); }

__host__ __device__ __forceinline__ SegUnit seg_unit(int u, int H)
{
    SegUnit r;
    if (u < H) {
        r.g = 0;
        r.mode = 0;
        r.h = u;
        return r;
    }
    const int v = u - H;
    r.g = 1 + v / (2 * H);
    r.mode = 1 + (v % (2 * H)) / H;
    r.h = v % H;
    return r;
}

// The consumer units that read ring group (g, h): one for segment 0, two after.
__host__ __device__ __forceinline__ int seg_group_consumers(int g, int h, int H, int (&u)[2])
{
    if (g == 0) {
        u[0] = h;
        return 1;
    }
    u[0] = H + (g - 1) * 2 * H + h;
    u[1] = u[0] + H;
    return 2;
}

// Workspace of kda_prefill_segmented: the work list, the split kernel's flags
// (full[groups][ring], consumed[units]) and ring, then o_aux, st_aux and the
// segment entry states S_g, transposed to fp16 in the 128-byte swizzled
// K-major layout of an MMA operand ([G][H] blocks of 32 KB), written by the
// scan for the fix-up's tensor-core product.
struct SegPlan {
    SplitPlan split;
    int32_t G, seg_chunks;
    size_t o_aux_off, st_aux_off, sstart_off, bytes;
};

inline bool seg_plan(int64_t T, int32_t H, int32_t G, int sms, SegPlan* plan)
{
    if (T < 1 || H < 1 || G < 2 || sms < 3) return false;
    const long long nch = (T + 63) / 64;
    SegPlan p;
    p.G = G;
    p.seg_chunks = (int32_t)((nch + G - 1) / G);
    p.seg_chunks += p.seg_chunks & 1;              // whole 128-token tiles
    if ((long long)(G - 1) * p.seg_chunks >= nch) return false;   // every segment has a chunk
    const long long units = (long long)seg_units(H, G);
    if (units > sms / 2) return false;
    SplitPlan& s = p.split;
    s.units = (int32_t)units;
    s.groups = G * H;
    s.producers = sms - s.units;
    const int ahead = (s.producers + s.groups - 1) / s.groups;
    s.ring = 3 * ahead + 4;
    if (s.ring > kSplitMaxRing) s.ring = kSplitMaxRing;
    s.flags_off = workspace_bytes(1);
    const size_t nflags = (size_t)s.groups * s.ring + s.units;
    s.ring_off = (s.flags_off + nflags * sizeof(int32_t) + 1023) / 1024 * 1024;
    s.bytes = s.ring_off + (size_t)s.groups * s.ring * 2 * kSplitStepBytes;
    const size_t state = (size_t)H * 128 * 128 * sizeof(float);
    p.o_aux_off = (s.bytes + 255) / 256 * 256;
    p.st_aux_off = p.o_aux_off + 2 * (size_t)T * H * 128 * sizeof(__half);
    p.st_aux_off = (p.st_aux_off + 255) / 256 * 256;
    p.sstart_off = p.st_aux_off + 2 * (size_t)G * state;
    p.bytes = p.sstart_off + (size_t)G * state / 2;
    *plan = p;
    return true;
}

// Number of SMs of the current device (cached per device; 0 on failure).
int device_sm_count();

// The gate prologue fused into the kernels ("[논문 리뷰] Kimi K3 Technical
// Report", section 3.5), when A is not null: the log_alpha input then holds
// the gate pre-activation z, g = -5 sigmoid(e^A z) with A [H, d_k] fp32, and
// q and k are L2-normalised over the key channels inside the kernel, q also
// multiplied by q_scale.  A null A: log_alpha is g and q, k are used as given.
struct GateArgs {
    const float* A;
    float q_scale;
};

__device__ __forceinline__ float gate_from_z(float z, float eA)
{
    // -5 sigmoid(e^A z) = -5 / (1 + e^{-e^A z}); the limits -5 and 0 are exact
    return __fdividef(-5.f, 1.f + __expf(-eA * z));
}

// 1 / ||x|| of a row whose sum of squares is ss (a zero row stays zero).
__device__ __forceinline__ float inv_norm(float ss) { return rsqrtf(fmaxf(ss, 1e-30f)); }

// Prefix-state snapshots requested from a prefill (interval 0: none).
// Snapshot j of sequence n, the state after its first (j + 1) * interval
// tokens, goes to out + ((offsets[n] + j) * H + h) * d_k * d_v; offsets is
// null for a single sequence (offset 0).  interval is a multiple of 64, so
// every snapshot falls on a chunk boundary of every path.
struct SnapArgs {
    int32_t interval;
    const int32_t* offsets;
    float* out;
};

// KDA_DEBUG set in the environment: failing host-side steps are reported on
// stderr (the status codes stay the same).
inline bool debug_enabled() { return getenv("KDA_DEBUG") != nullptr; }

// Scalar load / store helpers for the two I/O dtypes.
__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Launchers (return cudaGetLastError() after enqueueing).
// Validates cu_seqlens (when given) and the snapshot offsets (when snapshots
// are requested with cu_seqlens), writes order[], the error word and the
// longest length, resets the counters and zeroes `nflags` words at `flags`.
cudaError_t launch_worklist(const int32_t* cu_seqlens, int32_t num_seqs,
                            int64_t total_tokens, int32_t* ws, int32_t* flags,
                            int32_t nflags, const SnapArgs& snap, cudaStream_t stream);

cudaError_t launch_decode(const void* q, const void* k, const void* v,
                          const float* log_alpha, const float* beta, float* S,
                          int32_t N, int32_t H, int32_t d, kda_dtype_t dtype,
                          void* o, const GateArgs& gate, cudaStream_t stream);

// Ts tokens per sequence from S_in, the state after each token to `states`
// ([N, Ts, H, d, d]); the one-token decode above is the case Ts = 1 in place.
cudaError_t launch_decode_multi(const void* q, const void* k, const void* v,
                                const float* log_alpha, const float* beta, const float* S_in,
                                float* states, int32_t N, int32_t Ts, int32_t H, int32_t d,
                                kda_dtype_t dtype, void* o, const GateArgs& gate,
                                cudaStream_t stream);

cudaError_t launch_state_gather(const float* states, const float* S_in, const int32_t* accept,
                                int32_t N, int32_t Ts, int32_t H, int32_t d_k, int32_t d_v,
                                float* S_out, cudaStream_t stream);

cudaError_t launch_prefill_simt(const void* q, const void* k, const void* v,
                                const float* log_alpha, const float* beta,
                                const float* S0, const int32_t* cu_seqlens,
                                int32_t num_seqs, int64_t total_tokens, int32_t H,
                                int32_t d, kda_dtype_t dtype, void* o,
                                float* S_final, const int32_t* ws, const SnapArgs& snap,
                                const GateArgs& gate, cudaStream_t stream);

// Tensor-core prefill (bf16 q/k/v, d = 128).  Returns false when the call
// must take the CUDA-core path instead (other dtypes or head sizes, no tokens,
// or KDA_FORCE_SIMT set in the environment).
bool prefill_tc_supported(kda_dtype_t dtype, int32_t d, int64_t total_tokens);

cudaError_t launch_prefill_tc(const void* q, const void* k, const void* v,
                              const float* log_alpha, const float* beta, const float* S0,
                              const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                              int32_t H, kda_dtype_t dtype, void* o, float* S_final,
                              int32_t* ws, const SnapArgs& snap, const GateArgs& gate,
                              cudaStream_t stream);

cudaError_t launch_prefill_split(const void* q, const void* k, const void* v,
                                 const float* log_alpha, const float* beta, const float* S0,
                                 const int32_t* cu_seqlens, int32_t num_seqs,
                                 int64_t total_tokens, int32_t H, kda_dtype_t dtype, void* o,
                                 float* S_final, int32_t* ws, const SplitPlan& plan,
                                 const SnapArgs& snap, const GateArgs& gate, const SegArgs& seg,
                                 cudaStream_t stream);

// The segmented prefill's second pass: the scan over segments (S_g, and the
// caller's S_final) and the output fix-up o_t += S_g^T qt_t for segments >= 1.
cudaError_t launch_segment_fixup(const SegArgs& seg, int64_t total_tokens, int32_t H,
                                 kda_dtype_t dtype, void* o, float* S_final, __half* sstart,
                                 int32_t* timeout_word, cudaStream_t stream);

}  // namespace kda
