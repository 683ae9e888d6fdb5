// kda_prefill_simt.cu -- chunked KDA prefill on the fp32 CUDA cores.
//
// This is the exact-precision path: every head size in {16, 32, 64, 128},
// fp32 or bf16 I/O, all arithmetic in fp32.  It computes the chunkwise form of
// the recurrence ("Kimi 모델 분석", rlaope.github.io, section "순환을 GPU에
// 올리기": intra-chunk work as dense products, only the state carried from
// chunk to chunk) with chunks of C = 16 tokens.
//
// Chunk algebra (derived from the update of "[논문 리뷰] Kimi K3 Technical
// Report", jw9603.github.io, sections 3.2-3.3).  Inside a chunk with entry
// state S0, let G_r = sum_{i<=r} g_i (per key channel, relative to the chunk
// start) and gamma_r = exp(G_r).  Unrolling the update gives
//     S_r = Diag(gamma_r) S0 + sum_{i<=r} Diag(gamma_r / gamma_i) k_i u_i^T,
//     u_r = beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r),
// hence, with A_ri = beta_r sum_c k_rc k_ic exp(G_rc - G_ic) for i < r and
// P_ri = sum_c q_rc k_ic exp(G_rc - G_ic) for i <= r:
//     (I + A) U = Diag(beta) (V - (gamma .* K) S0)         (forward substitution)
//     O         = (gamma .* Q) S0 + P U
//     S_C       = Diag(gamma_last) S0 + sum_i ((gamma_last / gamma_i) .* k_i) u_i^T
// With the gate prologue (see GateArgs) phase 0 forms each chunk row's q and k
// norms and phase 1 turns z into g = -5 sigmoid(e^A z) and scales q and k.
//
// The decay is normalised to the chunk start, as the pages require for long
// chunks.  exp(G_rc - G_ic) is factored as exp(G_rc) * exp(-G_ic); with
// g >= -5 (the lower bound of section 3.5) and 16 tokens per chunk the larger
// factor is at most exp(80), inside the fp32 range.
//
// Mapping: one CTA per (sequence, head, 32-column value slab); the slab's
// state lives in shared memory for the whole sequence.  Rows past the end of
// a sequence in its last chunk enter as exact identity steps (g = 0, k = 0,
// beta = 0) and produce no output.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kC = 16;          // chunk length of this path
constexpr int kThreads = 256;

template <int DK, int DVS>
struct SimtSmem {
    static constexpr int LD = DK + 1;      // padded row stride of the chunk tiles
    static constexpr int LDS = DVS + 1;
    static constexpr int kQg = 0;
    static constexpr int kKg = kQg + kC * LD;
    static constexpr int kKi = kKg + kC * LD;
    static constexpr int kKt = kKi + kC * LD;
    static constexpr int kS = kKt + kC * LD;
    static constexpr int kV = kS + DK * LDS;
    static constexpr int kU = kV + kC * DVS;
    static constexpr int kO = kU + kC * LDS;
    static constexpr int kA = kO + kC * DVS;
    static constexpr int kP = kA + kC * (kC + 1);
    static constexpr int kB = kP + kC * (kC + 1);
    static constexpr int kGl = kB + kC;
    static constexpr int kInv = kGl + DK;    // gate prologue: 1/||q_r|| (x q_scale), 1/||k_r||
    static constexpr int kFloats = kInv + 2 * kC;
    static constexpr size_t kBytes = kFloats * sizeof(float);
};

template <typename TI, typename TO, int DK, int DVS>
__global__ void __launch_bounds__(kThreads)
prefill_simt_kernel(const TI* __restrict__ q, const TI* __restrict__ k,
                    const TI* __restrict__ v, const float* __restrict__ g,
                    const float* __restrict__ beta, const float* S0,
                    const int32_t* __restrict__ cu, const int32_t* __restrict__ ws,
                    long long total_tokens, int H, TO* __restrict__ o,
                    float* S_final,   // may alias S0: no __restrict__ on either
                    const SnapArgs snap, const GateArgs gate)
{
    using L = SimtSmem<DK, DVS>;
    constexpr int LD = L::LD, LDS = L::LDS;
    constexpr int DV = DK;
    constexpr int NSLAB = DV / DVS;
    extern __shared__ float sm[];
    float* sQg = sm + L::kQg;
    float* sKg = sm + L::kKg;
    float* sKi = sm + L::kKi;
    float* sKt = sm + L::kKt;
    float* sS = sm + L::kS;
    float* sV = sm + L::kV;
    float* sU = sm + L::kU;
    float* sO = sm + L::kO;
    float* sA = sm + L::kA;
    float* sP = sm + L::kP;
    float* sB = sm + L::kB;
    float* sGl = sm + L::kGl;
    float* sInv = sm + L::kInv;
    const bool fused = gate.A != nullptr;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int item = blockIdx.x;
    const int rank = item / (H * NSLAB);
    const int h = (item / NSLAB) % H;
    const int slab = item % NSLAB;
    const int col0 = slab * DVS;

    long long bos = 0, eos = total_tokens;
    int n = 0;
    if (cu != nullptr) {
        if (ws[kWsErrorWord] != 0) return;
        n = ws[kWsHeaderBytes / sizeof(int32_t) + rank];
        bos = cu[n];
        eos = cu[n + 1];
    }
    const long long sbase = ((long long)n * H + h) * DK * DV;
    const int seq_off = (cu != nullptr && snap.interval > 0) ? snap.offsets[n] : 0;
    // e^A of this thread's key channel (gate prologue)
    const float eA = (fused && tid < DK) ? expf(gate.A[h * DK + tid]) : 0.f;

    for (int e = tid; e < DK * DVS; e += kThreads) {
        const int c = e / DVS, j = e % DVS;
        sS[c * LDS + j] = S0 ? S0[sbase + (long long)c * DV + col0 + j] : 0.f;
    }

    for (long long t0 = bos; t0 < eos; t0 += kC) {
        __syncthreads();
        // Phase 0 (gate prologue only): the inverse norms of the chunk's q
        // and k rows, one warp per (row, tensor) pair.
        if (fused) {
            for (int pr = warp; pr < 2 * kC; pr += kThreads / 32) {
                const int r = pr >> 1;
                const long long t = t0 + r;
                float ss = 0.f;
                if (t < eos) {
                    const TI* row = ((pr & 1) ? k : q) + (t * H + h) * DK;
                    for (int c = lane; c < DK; c += 32) {
                        const float x = ld_f(row + c);
                        ss = fmaf(x, x, ss);
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (lane == 0) sInv[pr] = (pr & 1) ? inv_norm(ss) : gate.q_scale * inv_norm(ss);
            }
            __syncthreads();
        }
        // Phase 1: gates, decayed operands; v slab and beta.
        if (tid < DK) {
            const int c = tid;
            float G = 0.f;
            float Gr[kC], kr[kC];
#pragma unroll
            for (int r = 0; r < kC; ++r) {
                const long long t = t0 + r;
                float gg = 0.f, kk = 0.f, qq = 0.f;
                if (t < eos) {
                    const long long off = (t * H + h) * DK + c;
                    gg = g[off];
                    kk = ld_f(k + off);
                    qq = ld_f(q + off);
                    if (fused) {
                        gg = gate_from_z(gg, eA);
                        qq *= sInv[2 * r];
                        kk *= sInv[2 * r + 1];
                    }
                }
                G += gg;
                const float gam = expf(G);
                const float gin = expf(-G);
                sQg[r * LD + c] = qq * gam;
                sKg[r * LD + c] = kk * gam;
                sKi[r * LD + c] = kk * gin;
                Gr[r] = G;
                kr[r] = kk;
            }
#pragma unroll
            for (int r = 0; r < kC; ++r) sKt[r * LD + c] = kr[r] * expf(G - Gr[r]);
            sGl[c] = expf(G);
        } else {
            for (int e = tid - DK; e < kC * DVS; e += kThreads - DK) {
                const int r = e / DVS, j = e % DVS;
                const long long t = t0 + r;
                sV[r * DVS + j] = t < eos ? ld_f(v + (t * H + h) * DV + col0 + j) : 0.f;
            }
            for (int r = tid - DK; r < kC; r += kThreads - DK) {
                const long long t = t0 + r;
                sB[r] = t < eos ? beta[t * H + h] : 0.f;
            }
        }
        __syncthreads();

        // Phase 2: A (strictly lower, times beta_r), P (lower incl. diagonal),
        // the right-hand side beta_r (v_r - (gamma_r .* k_r) S0) and
        // (gamma_r .* q_r) S0.
        for (int e = tid; e < kC * kC; e += kThreads) {
            const int r = e / kC, i = e % kC;
            float a = 0.f, p = 0.f;
#pragma unroll 8
            for (int c = 0; c < DK; ++c) {
                const float ki = sKi[i * LD + c];
                a = fmaf(sKg[r * LD + c], ki, a);
                p = fmaf(sQg[r * LD + c], ki, p);
            }
            sA[r * (kC + 1) + i] = i < r ? sB[r] * a : 0.f;
            sP[r * (kC + 1) + i] = i <= r ? p : 0.f;
        }
        for (int e = tid; e < kC * DVS; e += kThreads) {
            const int r = e / DVS, j = e % DVS;
            float w = 0.f, os = 0.f;
#pragma unroll 8
            for (int c = 0; c < DK; ++c) {
                const float s = sS[c * LDS + j];
                w = fmaf(sKg[r * LD + c], s, w);
                os = fmaf(sQg[r * LD + c], s, os);
            }
            sU[r * LDS + j] = sB[r] * (sV[r * DVS + j] - w);
            sO[r * DVS + j] = os;
        }
        __syncthreads();

        // Phase 3: forward substitution (I + A) U = RHS, one value column per
        // thread.
        if (tid < DVS) {
            const int j = tid;
#pragma unroll
            for (int r = 1; r < kC; ++r) {
                float u = sU[r * LDS + j];
                for (int i = 0; i < r; ++i) u = fmaf(-sA[r * (kC + 1) + i], sU[i * LDS + j], u);
                sU[r * LDS + j] = u;
            }
        }
        __syncthreads();

        // Phase 4: outputs and the state carry (and a prefix snapshot when a
        // full chunk ends on a multiple of the snapshot interval).
        for (int e = tid; e < kC * DVS; e += kThreads) {
            const int r = e / DVS, j = e % DVS;
            const long long t = t0 + r;
            if (t >= eos) continue;
            float acc = sO[r * DVS + j];
            for (int i = 0; i <= r; ++i) acc = fmaf(sP[r * (kC + 1) + i], sU[i * LDS + j], acc);
            st_f(o + (t * H + h) * DV + col0 + j, acc);
        }
        float* snp = nullptr;
        if (snap.interval > 0 && t0 + kC <= eos && (t0 + kC - bos) % snap.interval == 0)
            snp = snap.out + ((long long)(seq_off + (t0 + kC - bos) / snap.interval - 1) * H + h) *
                                 DK * DV;
        for (int e = tid; e < DK * DVS; e += kThreads) {
            const int c = e / DVS, j = e % DVS;
            float s = sGl[c] * sS[c * LDS + j];
#pragma unroll
            for (int r = 0; r < kC; ++r) s = fmaf(sKt[r * LD + c], sU[r * LDS + j], s);
            sS[c * LDS + j] = s;
            if (snp) snp[(long long)c * DV + col0 + j] = s;
        }
    }
    __syncthreads();
    if (S_final) {
        for (int e = tid; e < DK * DVS; e += kThreads) {
            const int c = e / DVS, j = e % DVS;
            S_final[sbase + (long long)c * DV + col0 + j] = sS[c * LDS + j];
        }
    }
}

template <typename TI, typename TO, int D>
cudaError_t launch_typed(const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* S0,
                         const int32_t* cu, int32_t N, int64_t T_tot, int32_t H,
                         void* o, float* S_final, const int32_t* ws, const SnapArgs& snap,
                         const GateArgs& gate, cudaStream_t stream)
{
    constexpr int DVS = D < 32 ? D : 32;
    using L = SimtSmem<D, DVS>;
    auto kern = prefill_simt_kernel<TI, TO, D, DVS>;
    static bool attr_set = false;   // benign race: every writer stores the same value
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const long long blocks = (long long)N * H * (D / DVS);
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)blocks, kThreads, L::kBytes, stream>>>(
        static_cast<const TI*>(q), static_cast<const TI*>(k), static_cast<const TI*>(v),
        g, beta, S0, cu, ws, (long long)T_tot, H, static_cast<TO*>(o), S_final, snap, gate);
    return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_d(int32_t d, const void* q, const void* k, const void* v,
                     const float* g, const float* beta, const float* S0,
                     const int32_t* cu, int32_t N, int64_t T_tot, int32_t H,
                     void* o, float* S_final, const int32_t* ws, const SnapArgs& snap,
                     const GateArgs& gate, cudaStream_t stream)
{
    switch (d) {
        case 16: return launch_typed<TI, TO, 16>(q, k, v, g, beta, S0, cu, N, T_tot, H, o, S_final, ws, snap, gate, stream);
        case 32: return launch_typed<TI, TO, 32>(q, k, v, g, beta, S0, cu, N, T_tot, H, o, S_final, ws, snap, gate, stream);
        case 64: return launch_typed<TI, TO, 64>(q, k, v, g, beta, S0, cu, N, T_tot, H, o, S_final, ws, snap, gate, stream);
        case 128: return launch_typed<TI, TO, 128>(q, k, v, g, beta, S0, cu, N, T_tot, H, o, S_final, ws, snap, gate, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prefill_simt(const void* q, const void* k, const void* v,
                                const float* log_alpha, const float* beta,
                                const float* S0, const int32_t* cu_seqlens,
                                int32_t num_seqs, int64_t total_tokens, int32_t H,
                                int32_t d, kda_dtype_t dtype, void* o,
                                float* S_final, const int32_t* ws, const SnapArgs& snap,
                                const GateArgs& gate, cudaStream_t stream)
{
    switch (dtype) {
        case KDA_BF16:
            return launch_d<__nv_bfloat16, __nv_bfloat16>(d, q, k, v, log_alpha, beta, S0, cu_seqlens,
                                                          num_seqs, total_tokens, H, o, S_final, ws, snap, gate, stream);
        case KDA_BF16_F32OUT:
            return launch_d<__nv_bfloat16, float>(d, q, k, v, log_alpha, beta, S0, cu_seqlens,
                                                  num_seqs, total_tokens, H, o, S_final, ws, snap, gate, stream);
        default:
            return launch_d<float, float>(d, q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs,
                                          total_tokens, H, o, S_final, ws, snap, gate, stream);
    }
}

}  // namespace kda
