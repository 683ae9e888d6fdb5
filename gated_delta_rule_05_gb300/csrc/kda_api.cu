// kda_api.cu -- the C ABI declared in include/kda.h: argument validation,
// dispatch to the kernels, status mapping.  No allocation, no host sync.
#include <stdint.h>

#include <mutex>

#include "kda_internal.cuh"

namespace kda {

int device_sm_count()
{
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static int cached[kMaxDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace kda

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_d(int32_t d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// True when [a, a+na) and [b, b+nb) overlap.
bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool valid_dtype(kda_dtype_t t) { return t == KDA_BF16 || t == KDA_FP32 || t == KDA_BF16_F32OUT; }

// Bytes of one element of o.
size_t out_bytes(kda_dtype_t t) { return t == KDA_BF16 ? 2 : 4; }

}  // namespace

extern "C" {

size_t kda_prefill_workspace_bytes(int32_t num_seqs, int32_t H, int32_t d_k,
                                   int32_t d_v)
{
    kda::SplitPlan plan;
    if (d_k == 128 && d_v == 128 && kda::split_plan(num_seqs, H, kda::device_sm_count(), &plan))
        return plan.bytes;
    return kda::workspace_bytes(num_seqs);
}

}  // extern "C"

namespace {

kda_status_t prefill_impl(const void* q, const void* k, const void* v, const float* log_alpha,
                          const float* beta, const float* S0, const int32_t* cu_seqlens,
                          int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                          int32_t d_v, kda_dtype_t dtype, void* o, float* S_final,
                          const kda::SnapArgs& snap, const kda::GateArgs& gate, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream)
{
    if (!valid_dtype(dtype)) return KDA_ERR_UNSUPPORTED;
    if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 1 || H < 1 || total_tokens < 0) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && num_seqs != 1) return KDA_ERR_INVALID_ARG;
    // Token offsets are 32-bit in cu_seqlens.
    if (total_tokens > INT32_MAX) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !o))
        return KDA_ERR_INVALID_ARG;
    if (gate.A && !aligned(gate.A, 16)) return KDA_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, log_alpha, o, S0, S_final, snap.out};
    for (const void* p : ptrs16)
        if (p && !aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (beta && !aligned(beta, 4)) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned(cu_seqlens, 4)) return KDA_ERR_INVALID_ARG;
    const size_t state_bytes = (size_t)num_seqs * H * d_k * d_v * sizeof(float);
    if (S0 && S_final && S0 != S_final && overlaps(S0, state_bytes, S_final, state_bytes))
        return KDA_ERR_INVALID_ARG;
    if (o && S_final &&
        overlaps(o, (size_t)total_tokens * H * d_v * out_bytes(dtype), S_final, state_bytes))
        return KDA_ERR_INVALID_ARG;
    const size_t need = kda::workspace_bytes(num_seqs);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return KDA_ERR_WORKSPACE;

    int32_t* ws = static_cast<int32_t*>(workspace);
    cudaError_t err = cudaSuccess;
    const bool tc = kda::prefill_tc_supported(dtype, d_k, total_tokens);
    // Few (sequence, head) units and a workspace with room for the ring: the
    // producer / consumer kernel.
    kda::SplitPlan plan;
    const bool split = tc && kda::split_plan(num_seqs, H, kda::device_sm_count(), &plan) &&
                       workspace_bytes >= plan.bytes;
    if (cu_seqlens || split) {
        int32_t* flags =
            split ? reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + plan.flags_off)
                  : nullptr;
        const int32_t nflags = split ? plan.units * (plan.ring + 1) : 0;
        err = kda::launch_worklist(cu_seqlens, num_seqs, total_tokens, ws, flags, nflags, snap,
                                   stream);
        if (err != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (split) {
        const kda::SegArgs no_seg{0, 0, nullptr, nullptr};
        err = kda::launch_prefill_split(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs,
                                        total_tokens, H, dtype, o, S_final, ws, plan, snap, gate,
                                        no_seg, stream);
        if (err == cudaSuccess) return KDA_OK;
        // The launch was refused (a configuration error, nothing ran): the
        // single-CTA kernel computes the same result.
        (void)cudaGetLastError();
    }
    if (tc)
        err = kda::launch_prefill_tc(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs,
                                     total_tokens, H, dtype, o, S_final, ws, snap, gate, stream);
    else
        err = kda::launch_prefill_simt(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs,
                                       total_tokens, H, d_k, dtype, o, S_final, ws, snap, gate,
                                       stream);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

extern "C" {

kda_status_t kda_prefill(const void* q, const void* k, const void* v,
                         const float* log_alpha, const float* beta,
                         const float* S0, const int32_t* cu_seqlens,
                         int32_t num_seqs, int64_t total_tokens, int32_t H,
                         int32_t d_k, int32_t d_v, kda_dtype_t dtype, void* o,
                         float* S_final, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream)
{
    const kda::SnapArgs none{0, nullptr, nullptr};
    const kda::GateArgs given{nullptr, 1.f};
    return prefill_impl(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, d_k,
                        d_v, dtype, o, S_final, none, given, workspace, workspace_bytes, stream);
}

namespace {

// The number of segments kda_prefill_segmented uses for `requested` (<= 0:
// automatic); 1 means the sequence is not cut.  An explicit request is used
// when it is possible: every segment non-empty, the consumer units (H (2G - 1))
// at most half of the SMs.  The automatic choice keeps the units to about a
// third of the SMs and the segments to at least 32 chunks: more units leave
// too few producers, shorter segments too little chain to save.  Measured on
// one GB300 (152 SMs), one sequence, L2 flushed, the launches' kernel
// times summed, against kda_prefill: H = 16 (2 segments) 1.19x at 4,096
// tokens (118 against 140 us) and 1.39x at 16,384; H = 8 (3 segments) 2.2x
// at 65,536; H = 4 (6 segments) 3.4x at 32,768; H = 24 slower, so not cut.
int32_t resolve_segments(int64_t T, int32_t H, int32_t requested, int sms, kda::SegPlan* plan)
{
    const long long nch = (T + 63) / 64;
    if (requested > 0) {
        if (requested >= 2 && kda::seg_plan(T, H, requested, sms, plan)) return requested;
        return 1;
    }
    const int units_budget = sms * 8 / 25;
    int32_t G = 1;
    while (kda::seg_units(H, G + 1) <= units_budget && nch / (G + 1) >= 32) ++G;
    for (; G >= 2; --G)
        if (kda::seg_plan(T, H, G, sms, plan)) return G;
    return 1;
}

}  // namespace

size_t kda_prefill_segmented_workspace_bytes(int64_t total_tokens, int32_t H, int32_t d_k,
                                             int32_t d_v, int32_t segments)
{
    kda::SegPlan plan;
    if (d_k == 128 && d_v == 128 && H >= 1 && total_tokens >= 1 &&
        resolve_segments(total_tokens, H, segments, kda::device_sm_count(), &plan) >= 2)
        return plan.bytes;
    return kda_prefill_workspace_bytes(1, H, d_k, d_v);
}

kda_status_t kda_prefill_segmented(const void* q, const void* k, const void* v,
                                   const float* log_alpha, const float* beta, const float* S0,
                                   int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                   kda_dtype_t dtype, void* o, float* S_final, int32_t segments,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    kda::SegPlan plan;
    const bool tc = (dtype == KDA_BF16 || dtype == KDA_BF16_F32OUT) && d_k == 128 && d_v == 128 &&
                    kda::prefill_tc_supported(dtype, d_k, total_tokens);
    const int32_t G = (tc && H >= 1 && total_tokens >= 1)
                          ? resolve_segments(total_tokens, H, segments, kda::device_sm_count(), &plan)
                          : 1;
    if (G < 2 || workspace_bytes < plan.bytes)
        // Not worth (or not possible) to cut: the plain prefill, same results.
        return kda_prefill(q, k, v, log_alpha, beta, S0, nullptr, 1, total_tokens, H, d_k, d_v,
                           dtype, o, S_final, workspace, workspace_bytes, stream);
    // Argument checks of kda_prefill (one sequence).
    if (total_tokens > INT32_MAX) return KDA_ERR_INVALID_ARG;
    if (!q || !k || !v || !log_alpha || !beta || !o) return KDA_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, log_alpha, o, S0, S_final};
    for (const void* p : ptrs16)
        if (p && !aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (!aligned(beta, 4)) return KDA_ERR_INVALID_ARG;
    const size_t state_bytes = (size_t)H * d_k * d_v * sizeof(float);
    if (S0 && S_final && S0 != S_final && overlaps(S0, state_bytes, S_final, state_bytes))
        return KDA_ERR_INVALID_ARG;
    if (S_final && overlaps(o, (size_t)total_tokens * H * d_v * out_bytes(dtype), S_final, state_bytes))
        return KDA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256)) return KDA_ERR_WORKSPACE;

    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    int32_t* ws = reinterpret_cast<int32_t*>(wsb);
    const kda::SplitPlan& sp = plan.split;
    const kda::SnapArgs none{0, nullptr, nullptr};
    const kda::GateArgs given{nullptr, 1.f};
    const kda::SegArgs seg{G, plan.seg_chunks, reinterpret_cast<__half*>(wsb + plan.o_aux_off),
                           reinterpret_cast<float*>(wsb + plan.st_aux_off)};
    int32_t* flags = reinterpret_cast<int32_t*>(wsb + sp.flags_off);
    const int32_t nflags = sp.groups * sp.ring + sp.units;
    cudaError_t err = kda::launch_worklist(nullptr, 1, total_tokens, ws, flags, nflags, none, stream);
    if (err != cudaSuccess) return KDA_ERR_CUDA;
    // S_final may alias S0: segment 0 has read S0 before the scan writes it.
    err = kda::launch_prefill_split(q, k, v, log_alpha, beta, S0, nullptr, 1, total_tokens, H, dtype,
                                    o, nullptr, ws, sp, none, given, seg, stream);
    if (err != cudaSuccess) return KDA_ERR_CUDA;
    err = kda::launch_segment_fixup(seg, total_tokens, H, dtype, o, S_final,
                                    reinterpret_cast<__half*>(wsb + plan.sstart_off),
                                    ws + kda::kWsTimeoutWord, stream);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_prefill_snapshots(const void* q, const void* k, const void* v,
                                   const float* log_alpha, const float* beta, const float* S0,
                                   const int32_t* cu_seqlens, int32_t num_seqs,
                                   int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                   kda_dtype_t dtype, void* o, float* S_final, int32_t interval,
                                   const int32_t* snap_offsets, float* snapshots, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream)
{
    if (interval <= 0 || interval % 64 != 0) return KDA_ERR_INVALID_ARG;
    if (snapshots == nullptr) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens != nullptr && (snap_offsets == nullptr || !aligned(snap_offsets, 4)))
        return KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && total_tokens > 0) {
        // one sequence: its floor(T / interval) snapshots must not overlap o or S_final
        const size_t snap_bytes = (size_t)(total_tokens / interval) * H * d_k * d_v * sizeof(float);
        const size_t state_bytes = (size_t)H * d_k * d_v * sizeof(float);
        if (o && overlaps(snapshots, snap_bytes, o,
                          (size_t)total_tokens * H * d_v * out_bytes(dtype)))
            return KDA_ERR_INVALID_ARG;
        if (S_final && overlaps(snapshots, snap_bytes, S_final, state_bytes))
            return KDA_ERR_INVALID_ARG;
    }
    const kda::SnapArgs snap{interval, cu_seqlens ? snap_offsets : nullptr, snapshots};
    const kda::GateArgs given{nullptr, 1.f};
    return prefill_impl(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, d_k,
                        d_v, dtype, o, S_final, snap, given, workspace, workspace_bytes, stream);
}

kda_status_t kda_prefill_fused(const void* q, const void* k, const void* v, const float* z,
                               const float* A, const float* beta, const float* S0,
                               const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                               int32_t H, int32_t d_k, int32_t d_v, kda_dtype_t dtype,
                               float q_scale, void* o, float* S_final, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream)
{
    if (A == nullptr) return KDA_ERR_INVALID_ARG;
    const kda::SnapArgs none{0, nullptr, nullptr};
    const kda::GateArgs gate{A, q_scale};
    return prefill_impl(q, k, v, z, beta, S0, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v,
                        dtype, o, S_final, none, gate, workspace, workspace_bytes, stream);
}

kda_status_t kda_decode_step(const void* q, const void* k, const void* v,
                             const float* log_alpha, const float* beta,
                             float* S_inout, int32_t N, int32_t H, int32_t d_k,
                             int32_t d_v, kda_dtype_t dtype, void* o,
                             cudaStream_t stream)
{
    if (!valid_dtype(dtype)) return KDA_ERR_UNSUPPORTED;
    if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
    if (N < 1 || H < 1) return KDA_ERR_INVALID_ARG;
    if (!q || !k || !v || !log_alpha || !beta || !S_inout || !o) return KDA_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, log_alpha, o, S_inout};
    for (const void* p : ptrs16)
        if (!aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (!aligned(beta, 4)) return KDA_ERR_INVALID_ARG;
    const size_t state_bytes = (size_t)N * H * d_k * d_v * sizeof(float);
    if (overlaps(o, (size_t)N * H * d_v * out_bytes(dtype), S_inout, state_bytes))
        return KDA_ERR_INVALID_ARG;
    cudaError_t err = kda::launch_decode(q, k, v, log_alpha, beta, S_inout, N, H, d_k,
                                         dtype, o, kda::GateArgs{nullptr, 1.f}, stream);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_step_fused(const void* q, const void* k, const void* v, const float* z,
                                   const float* A, const float* beta, float* S_inout, int32_t N,
                                   int32_t H, int32_t d_k, int32_t d_v, kda_dtype_t dtype,
                                   float q_scale, void* o, cudaStream_t stream)
{
    if (!valid_dtype(dtype)) return KDA_ERR_UNSUPPORTED;
    if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
    if (N < 1 || H < 1) return KDA_ERR_INVALID_ARG;
    if (!q || !k || !v || !z || !A || !beta || !S_inout || !o) return KDA_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, z, A, o, S_inout};
    for (const void* p : ptrs16)
        if (!aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (!aligned(beta, 4)) return KDA_ERR_INVALID_ARG;
    const size_t state_bytes = (size_t)N * H * d_k * d_v * sizeof(float);
    if (overlaps(o, (size_t)N * H * d_v * out_bytes(dtype), S_inout, state_bytes))
        return KDA_ERR_INVALID_ARG;
    cudaError_t err = kda::launch_decode(q, k, v, z, beta, S_inout, N, H, d_k, dtype, o,
                                         kda::GateArgs{A, q_scale}, stream);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_multi(const void* q, const void* k, const void* v,
                              const float* log_alpha, const float* beta, const float* S_in,
                              int32_t N, int32_t Ts, int32_t H, int32_t d_k, int32_t d_v,
                              kda_dtype_t dtype, void* o, float* states, cudaStream_t stream)
{
    if (!valid_dtype(dtype)) return KDA_ERR_UNSUPPORTED;
    if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
    if (N < 1 || Ts < 1 || H < 1) return KDA_ERR_INVALID_ARG;
    if (!q || !k || !v || !log_alpha || !beta || !S_in || !o || !states) return KDA_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, log_alpha, o, S_in, states};
    for (const void* p : ptrs16)
        if (!aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (!aligned(beta, 4)) return KDA_ERR_INVALID_ARG;
    const size_t state_bytes = (size_t)N * H * d_k * d_v * sizeof(float);
    const size_t states_bytes = state_bytes * Ts;
    const size_t o_bytes = (size_t)N * Ts * H * d_v * out_bytes(dtype);
    if (overlaps(states, states_bytes, S_in, state_bytes) || overlaps(states, states_bytes, o, o_bytes) ||
        overlaps(o, o_bytes, S_in, state_bytes))
        return KDA_ERR_INVALID_ARG;
    cudaError_t err = kda::launch_decode_multi(q, k, v, log_alpha, beta, S_in, states, N, Ts, H,
                                               d_k, dtype, o, kda::GateArgs{nullptr, 1.f}, stream);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_state_gather(const float* states, const float* S_in, const int32_t* accept,
                              int32_t N, int32_t Ts, int32_t H, int32_t d_k, int32_t d_v,
                              float* S_out, cudaStream_t stream)
{
    if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
    if (N < 1 || Ts < 1 || H < 1) return KDA_ERR_INVALID_ARG;
    if (!states || !S_in || !accept || !S_out) return KDA_ERR_INVALID_ARG;
    const void* ptrs16[] = {states, S_in, S_out};
    for (const void* p : ptrs16)
        if (!aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (!aligned(accept, 4)) return KDA_ERR_INVALID_ARG;
    const size_t state_bytes = (size_t)N * H * d_k * d_v * sizeof(float);
    if (overlaps(S_out, state_bytes, states, state_bytes * Ts)) return KDA_ERR_INVALID_ARG;
    if (S_out != S_in && overlaps(S_out, state_bytes, S_in, state_bytes)) return KDA_ERR_INVALID_ARG;
    cudaError_t err = kda::launch_state_gather(states, S_in, accept, N, Ts, H, d_k, d_v, S_out, stream);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

const char* kda_status_string(kda_status_t status)
{
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: dtype or head size not supported";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA launch failed";
        default: return "KDA_ERR_UNKNOWN: unknown status code";
    }
}

}  // extern "C"
