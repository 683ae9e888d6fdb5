// kda_worklist.cu -- varlen scheduling for prefill: validate cu_seqlens and
// order the sequences longest-first on the device.
//
// Serving stacks hand a packed batch to the attention kernels together with
// per-request extents ("attention metadata"); building that metadata with many
// small host-driven ops was itself a measurable cost ("Kimi 모델 분석",
// rlaope.github.io, section "커널 최적화", the metadata-builder bullet).  Here
// the whole step is one single-CTA kernel on the caller's stream, with no host
// round trip:
//   * checks cu[0] = 0, cu[n] <= cu[n+1], cu[N] = total_tokens;
//   * writes the error word (0 = valid) and the longest sequence length, and
//     resets the work counters;
//   * writes order[] = sequence indices sorted by length, longest first (ties
//     by index), so that work items handed out in order approximate the
//     longest-processing-time-first schedule;
//   * checks the prefix-snapshot offsets when snapshots are requested
//     (offsets[0] = 0, sequence n owning floor(len_n / interval) of them);
//   * zeroes the hand-over flags of the split prefill kernel when it runs.
// Without cu_seqlens (one sequence) only the counters, the length word and
// the flags are written.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads)
worklist_kernel(const int32_t* __restrict__ cu, int32_t N, int64_t total_tokens,
                int32_t* __restrict__ ws, int32_t* __restrict__ flags, int32_t nflags,
                int32_t snap_interval, const int32_t* __restrict__ snap_off)
{
    __shared__ int bad;
    __shared__ int32_t maxlen;
    __shared__ int32_t len[kMaxSortedSeqs];
    const int tid = threadIdx.x;
    for (int i = tid; i < nflags; i += kThreads) flags[i] = 0;
    if (cu == nullptr) {                       // one sequence of total_tokens
        if (tid == 0) {
            ws[kWsCounterWord] = 0;
            ws[kWsErrorWord] = 0;
            ws[kWsMaxLenWord] = (int32_t)total_tokens;
            *reinterpret_cast<unsigned long long*>(ws + kWsJobWord) = 0ull;
            ws[kWsAbortWord] = 0;
            ws[kWsHeaderBytes / sizeof(int32_t)] = 0;
        }
        return;
    }
    if (tid == 0) {
        bad = (cu[0] != 0 || (int64_t)cu[N] != total_tokens) ? 1 : 0;
        if (snap_off != nullptr && snap_off[0] != 0) bad = 1;
        maxlen = 0;
    }
    __syncthreads();
    for (int n = tid; n < N; n += kThreads) {
        const int32_t l = cu[n + 1] - cu[n];
        if (l < 0) atomicOr(&bad, 1);
        // snapshot offsets: sequence n owns floor(len / interval) of them
        if (snap_off != nullptr && l >= 0 && snap_off[n + 1] - snap_off[n] != l / snap_interval)
            atomicOr(&bad, 1);
        atomicMax(&maxlen, l);
        if (N <= kMaxSortedSeqs) len[n] = l;
    }
    __syncthreads();
    int32_t* order = ws + kWsHeaderBytes / sizeof(int32_t);
    if (N <= kMaxSortedSeqs) {
        for (int n = tid; n < N; n += kThreads) {
            const int32_t ln = len[n];
            int rank = 0;
            for (int m = 0; m < N; ++m) {
                const int32_t lm = len[m];
                rank += (lm > ln) || (lm == ln && m < n);
            }
            order[rank] = n;
        }
    } else {
        for (int n = tid; n < N; n += kThreads) order[n] = n;
    }
    if (tid == 0) {
        ws[kWsCounterWord] = 0;
        ws[kWsErrorWord] = bad;
        ws[kWsMaxLenWord] = maxlen;
        *reinterpret_cast<unsigned long long*>(ws + kWsJobWord) = 0ull;
        ws[kWsAbortWord] = 0;
    }
}

}  // namespace

cudaError_t launch_worklist(const int32_t* cu_seqlens, int32_t num_seqs,
                            int64_t total_tokens, int32_t* ws, int32_t* flags,
                            int32_t nflags, const SnapArgs& snap, cudaStream_t stream)
{
    const int32_t* off = (cu_seqlens != nullptr && snap.interval > 0) ? snap.offsets : nullptr;
    worklist_kernel<<<1, kThreads, 0, stream>>>(cu_seqlens, num_seqs, total_tokens, ws, flags,
                                                nflags, snap.interval, off);
    return cudaGetLastError();
}

}  // namespace kda
