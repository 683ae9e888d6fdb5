// kda_host.cu -- kda_prefill_host: the prefill of one sequence whose inputs
// and outputs live in host memory.
//
// A long prompt arrives from the host: a 1M-token prompt at H = 32 is 43 GB
// of q, k, v, log-decay and beta.  Copied in, computed and copied back one
// after the other, the copies dominate.  Here the sequence is cut into
// segments of `segment_tokens` tokens (a multiple of 64, a chunk boundary of
// every path) that flow through a pipeline on three caller streams:
//   h2d stream      segment i's inputs -> staging slot i % 2
//   compute stream  kda_prefill on the slot, the state carried from segment
//                   i - 1 (its S_final) as segment i's S0
//   d2h stream      segment i's o -> host
// so that copies in, compute and copies out of different segments overlap.
// The state only passes between segments at a chunk boundary, in fp32, so the
// result equals one kda_prefill over the whole sequence bit for bit.
//
// The library still allocates nothing: the caller passes the device staging
// area (kda_prefill_host_staging_bytes).  The call creates six events to order
// the streams and releases them before it returns (the release completes once
// the work that waits on them is done).  Nothing is synchronised with the
// host: the work is enqueued and `compute` waits for the last copy out.
#include <stdint.h>

#include "kda_internal.cuh"

namespace {

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct HostPlan {
    size_t in_bytes_per_token, out_bytes_per_token;
    size_t in_slot, out_slot, state, ws, total;
};

size_t isize(kda_dtype_t t) { return t == KDA_FP32 ? 4 : 2; }
size_t osize(kda_dtype_t t) { return t == KDA_BF16 ? 2 : 4; }

HostPlan host_plan(int32_t H, int32_t d, kda_dtype_t dtype, int64_t seg)
{
    HostPlan p;
    // q, k, v in the input dtype, log_alpha fp32 [d], beta fp32 [1] per token-head
    p.in_bytes_per_token = (size_t)H * (3 * d * isize(dtype) + 4 * d + 4);
    p.out_bytes_per_token = (size_t)H * d * osize(dtype);
    // each tensor of a slot starts on a 256-byte boundary
    p.in_slot = 5 * 256 + (size_t)seg * p.in_bytes_per_token;
    p.out_slot = align256((size_t)seg * p.out_bytes_per_token);
    p.state = align256((size_t)H * d * d * sizeof(float));
    p.ws = align256(kda_prefill_workspace_bytes(1, H, d, d));
    p.total = 2 * align256(p.in_slot) + 2 * p.out_slot + 2 * p.state + p.ws;
    return p;
}

}  // namespace

extern "C" {

size_t kda_prefill_host_staging_bytes(int32_t H, int32_t d_k, int32_t d_v, kda_dtype_t dtype,
                                      int64_t segment_tokens)
{
    if (H < 1 || d_k != d_v || segment_tokens < 64 || segment_tokens % 64 != 0) return 0;
    return host_plan(H, d_k, dtype, segment_tokens).total;
}

kda_status_t kda_prefill_host(const void* q, const void* k, const void* v, const float* log_alpha,
                              const float* beta, const float* S0, int64_t total_tokens, int32_t H,
                              int32_t d_k, int32_t d_v, kda_dtype_t dtype, void* o,
                              float* S_final, void* staging, size_t staging_bytes,
                              int64_t segment_tokens, cudaStream_t compute, cudaStream_t h2d,
                              cudaStream_t d2h)
{
    if (dtype != KDA_BF16 && dtype != KDA_FP32 && dtype != KDA_BF16_F32OUT)
        return KDA_ERR_UNSUPPORTED;
    if (d_k != d_v || (d_k != 16 && d_k != 32 && d_k != 64 && d_k != 128))
        return KDA_ERR_UNSUPPORTED;
    if (H < 1 || total_tokens < 0 || total_tokens > INT32_MAX) return KDA_ERR_INVALID_ARG;
    if (segment_tokens < 64 || segment_tokens % 64 != 0) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !o))
        return KDA_ERR_INVALID_ARG;
    if (!staging || reinterpret_cast<uintptr_t>(staging) % 256 != 0) return KDA_ERR_WORKSPACE;
    const int32_t d = d_k;
    const int64_t seg = segment_tokens < total_tokens ? segment_tokens
                                                      : (total_tokens + 63) / 64 * 64;
    const HostPlan p = host_plan(H, d, dtype, seg > 0 ? seg : 64);
    if (staging_bytes < p.total) return KDA_ERR_WORKSPACE;

    uint8_t* base = static_cast<uint8_t*>(staging);
    uint8_t* in_slot[2] = {base, base + align256(p.in_slot)};
    uint8_t* out_slot[2] = {base + 2 * align256(p.in_slot),
                            base + 2 * align256(p.in_slot) + p.out_slot};
    float* state[2] = {reinterpret_cast<float*>(out_slot[1] + p.out_slot),
                       reinterpret_cast<float*>(out_slot[1] + p.out_slot + p.state)};
    void* ws = out_slot[1] + p.out_slot + 2 * p.state;

    const size_t qk_tok = (size_t)H * d * isize(dtype);      // bytes of q (k, v) per token
    const size_t g_tok = (size_t)H * d * 4, b_tok = (size_t)H * 4;
    const size_t o_tok = p.out_bytes_per_token;
    // slot layout: q | k | v | log_alpha | beta, each on a 256-byte boundary
    auto slot_ptr = [&](int s, int which) {
        const size_t sizes[5] = {qk_tok, qk_tok, qk_tok, g_tok, b_tok};
        uint8_t* ptr = in_slot[s];
        for (int i = 0; i < which; ++i) ptr += align256(sizes[i] * seg);
        return ptr;
    };

    if (total_tokens == 0) {
        if (S_final && S_final != S0) {
            const size_t sb = (size_t)H * d * d * sizeof(float);
            cudaError_t e = S0 ? cudaMemcpyAsync(S_final, S0, sb, cudaMemcpyDeviceToDevice, compute)
                               : cudaMemsetAsync(S_final, 0, sb, compute);
            return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
        }
        return KDA_OK;
    }

    cudaEvent_t ev[6] = {};
    for (int i = 0; i < 6; ++i) {
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            return KDA_ERR_CUDA;
        }
    }
    cudaEvent_t* ev_in = ev;           // [2]: a slot's inputs are in
    cudaEvent_t* ev_comp = ev + 2;     // [2]: a slot's compute is done
    cudaEvent_t* ev_out = ev + 4;      // [2]: a slot's output has left
    kda_status_t st = KDA_OK;
    // Work already on `compute` (a previous call still reading the staging
    // slots, or the caller's producers of S0) precedes the first copy in.
    cudaError_t err = cudaEventRecord(ev_comp[1], compute);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(h2d, ev_comp[1], 0);
    const int64_t nseg = (total_tokens + seg - 1) / seg;
    for (int64_t i = 0; i < nseg && st == KDA_OK && err == cudaSuccess; ++i) {
        const int s = (int)(i & 1);
        const int64_t t0 = i * seg;
        const int64_t n = (total_tokens - t0 < seg) ? total_tokens - t0 : seg;
        // 1. inputs of segment i into slot s, once segment i - 2's compute has read it
        if (i >= 2) err = cudaStreamWaitEvent(h2d, ev_comp[s], 0);
        const void* src[5] = {static_cast<const uint8_t*>(q) + t0 * qk_tok,
                              static_cast<const uint8_t*>(k) + t0 * qk_tok,
                              static_cast<const uint8_t*>(v) + t0 * qk_tok,
                              reinterpret_cast<const uint8_t*>(log_alpha) + t0 * g_tok,
                              reinterpret_cast<const uint8_t*>(beta) + t0 * b_tok};
        const size_t bytes[5] = {qk_tok * n, qk_tok * n, qk_tok * n, g_tok * n, b_tok * n};
        for (int w = 0; w < 5 && err == cudaSuccess; ++w)
            err = cudaMemcpyAsync(slot_ptr(s, w), src[w], bytes[w], cudaMemcpyHostToDevice, h2d);
        if (err == cudaSuccess) err = cudaEventRecord(ev_in[s], h2d);
        // 2. compute, once the inputs are in and segment i - 2's o has left slot s
        if (err == cudaSuccess) err = cudaStreamWaitEvent(compute, ev_in[s], 0);
        if (err == cudaSuccess && i >= 2) err = cudaStreamWaitEvent(compute, ev_out[s], 0);
        if (err != cudaSuccess) break;
        const float* s_in = (i == 0) ? S0 : state[(i - 1) & 1];
        float* s_out = (i == nseg - 1 && S_final) ? S_final : state[i & 1];
        st = kda_prefill(slot_ptr(s, 0), slot_ptr(s, 1), slot_ptr(s, 2),
                         reinterpret_cast<const float*>(slot_ptr(s, 3)),
                         reinterpret_cast<const float*>(slot_ptr(s, 4)), s_in, nullptr, 1, n, H, d,
                         d, dtype, out_slot[s], s_out, ws, p.ws, compute);
        if (st != KDA_OK) break;
        err = cudaEventRecord(ev_comp[s], compute);
        // 3. o of segment i back to the host
        if (err == cudaSuccess) err = cudaStreamWaitEvent(d2h, ev_comp[s], 0);
        if (err == cudaSuccess)
            err = cudaMemcpyAsync(static_cast<uint8_t*>(o) + t0 * o_tok, out_slot[s], o_tok * n,
                                  cudaMemcpyDeviceToHost, d2h);
        if (err == cudaSuccess) err = cudaEventRecord(ev_out[s], d2h);
    }
    // The compute stream completes only after the last copy out.
    if (st == KDA_OK && err == cudaSuccess)
        err = cudaStreamWaitEvent(compute, ev_out[(nseg - 1) & 1], 0);
    for (int i = 0; i < 6; ++i) cudaEventDestroy(ev[i]);
    if (st != KDA_OK) return st;
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
