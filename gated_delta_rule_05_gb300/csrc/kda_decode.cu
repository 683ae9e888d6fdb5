// kda_decode.cu -- one KDA decode step: a fused, bandwidth-bound
// read-modify-write of the fp32 state.
//
// Method: "[논문 리뷰] Kimi K3 Technical Report" (jw9603.github.io), sections
// 3.2-3.3.  For one (sequence, head) with state S (rows = key channels):
//     Sbar = Diag(alpha) S,          alpha = exp(log_alpha)
//     w    = Sbar^T k = S^T (alpha .* k)
//     p    = Sbar^T q = S^T (alpha .* q)
//     u    = beta (v - w)
//     S'   = Sbar + k u^T
//     o    = S'^T q = p + (k . q) u
// Decode is bound by the state bytes it streams ("Kimi 모델 분석",
// rlaope.github.io, section "Decoding이 왜 느린가"): each state element is read
// once and written once, so one launch moves 8 * d_k * d_v bytes per
// (sequence, head) plus a few hundred bytes of token inputs.
//
// Several tokens per sequence (the verification step of speculative decoding,
// "[논문 리뷰] Kimi K3 Technical Report", section 13; "Kimi 모델 분석", section
// "Dspark 투기적 디코딩"): the state is overwritten in place and cannot be
// truncated, so the kernel keeps the state after every token.  It reads the
// state once, applies Ts steps to it in registers and writes each step's state
// to its own slot; the one-token decode is the case Ts = 1 written in place.
//
// With the gate prologue (A not null; "[논문 리뷰] Kimi K3 Technical Report",
// section 3.5) the log_alpha input is the gate pre-activation z,
// g = -5 sigmoid(e^A z), and q, k are L2-normalised in the kernel: the sums
// of squares are reduced across the block with k.q, and the norms scale k and
// q where they are used (a factor of exactly 1 without the prologue).
//
// Mapping: one CTA per (sequence, head, value-column slab).  Value columns of
// S never mix (column j is updated with v_j alone), so a slab is independent.
// Each thread holds R float4 of its slab in registers between the read and the
// write; rows are spread over threads so that every warp reads whole 16-byte
// aligned row segments (fully coalesced 128-bit accesses).  The state is read
// with the streaming (evict-first) hint and written with streaming stores: it
// is touched once per step and must not evict the token inputs.
#include "kda_internal.cuh"

namespace kda {
namespace {

template <int DK, int DVS, int THREADS>
struct DecodeShape {
    static constexpr int kLanesPerRow = DVS / 4;              // float4 per slab row
    static constexpr int kRowsPerPass = THREADS / kLanesPerRow;
    static constexpr int kR = DK / kRowsPerPass;              // float4 per thread
    static constexpr int kWarps = THREADS / 32;
    static_assert(DVS % 4 == 0 && kLanesPerRow <= 32, "slab width");
    static_assert(THREADS % kLanesPerRow == 0, "thread count");
    static_assert(DK % kRowsPerPass == 0, "rows per pass must divide d_k");
    static_assert(DVS <= THREADS && DK <= THREADS, "one thread per column / row");
};

// Token inputs are [N, Ts, H, .]; S_in is [N, H, d_k, d_v] and the state
// after token t of (n, h) goes to S_out + ((n Ts + t) H + h) d_k d_v (for
// Ts = 1 this is S_in's own layout, so the one-token decode passes
// S_out = S_in).
template <typename TI, typename TO, int DK, int DVS, int THREADS>
__global__ void __launch_bounds__(THREADS)
decode_kernel(const TI* __restrict__ q, const TI* __restrict__ k,
              const TI* __restrict__ v, const float* __restrict__ log_alpha,
              const float* __restrict__ beta, const float* S_in, float* S_out,
              TO* __restrict__ o, int dv, int Ts, int H, const float* __restrict__ gateA,
              float q_scale)
{
    using Sh = DecodeShape<DK, DVS, THREADS>;
    constexpr int LPR = Sh::kLanesPerRow;
    constexpr int RPP = Sh::kRowsPerPass;
    constexpr int R = Sh::kR;

    const int nslab = dv / DVS;
    const int slab = blockIdx.x % nslab;
    const long long nh = blockIdx.x / nslab;     // sequence * H + head
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int c4 = tid % LPR;                     // float4 column within the slab
    const int rg = tid / LPR;                     // first row of this thread
    const int col = slab * DVS + c4 * 4;
    const long long n = nh / H, h = nh % H;

    const float* Sp = S_in + nh * (long long)DK * dv;

    // 1. Issue every state load first so that they are all in flight.
    float4 s[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int i = rg + r * RPP;
        s[r] = __ldcs(reinterpret_cast<const float4*>(Sp + (long long)i * dv + col));
    }

    __shared__ float sh_a[DK], sh_k[DK], sh_ak[DK], sh_aq[DK];
    __shared__ float sh_red_w[Sh::kWarps][DVS];
    __shared__ float sh_red_p[Sh::kWarps][DVS];
    __shared__ float sh_kq[Sh::kWarps], sh_kk[Sh::kWarps], sh_qq[Sh::kWarps];
    __shared__ float sh_u[DVS];
    const bool fused = gateA != nullptr;
    const float eA = (fused && tid < DK) ? expf(gateA[h * DK + tid]) : 0.f;

    for (int t = 0; t < Ts; ++t) {
        const long long tok = (n * Ts + t) * H + h;       // token row of this (n, t, h)
        float* Sq = S_out + tok * (long long)DK * dv;
        if (t > 0) __syncthreads();                        // the previous token's reads are done

        // 2. Token inputs: alpha, k, alpha.*k, alpha.*q and the partial k.q.
        float kq = 0.f, kk2 = 0.f, qq2 = 0.f;
        if (tid < DK) {
            const long long off = tok * DK + tid;
            const float gg = fused ? gate_from_z(log_alpha[off], eA) : log_alpha[off];
            const float a = expf(gg);
            const float kk = ld_f(k + off);
            const float qq = ld_f(q + off);
            sh_a[tid] = a;
            sh_k[tid] = kk;
            sh_ak[tid] = a * kk;
            sh_aq[tid] = a * qq;
            kq = kk * qq;
            kk2 = kk * kk;
            qq2 = qq * qq;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
            if (fused) {
                kk2 += __shfl_xor_sync(0xffffffffu, kk2, off);
                qq2 += __shfl_xor_sync(0xffffffffu, qq2, off);
            }
        }
        if (lane == 0) {
            sh_kq[warp] = kq;
            sh_kk[warp] = kk2;
            sh_qq[warp] = qq2;
        }
        __syncthreads();
        // 1 / ||k|| and q_scale / ||q|| (exactly 1 without the prologue)
        float ik = 1.f, iq = 1.f;
        if (fused) {
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int i = 0; i < Sh::kWarps; ++i) {
                sk += sh_kk[i];
                sq += sh_qq[i];
            }
            ik = inv_norm(sk);
            iq = q_scale * inv_norm(sq);
        }

        // 3. Partial column sums of S^T(alpha.*k) and S^T(alpha.*q) over this
        //    thread's rows, then across lanes that share the same columns.
        float4 w = make_float4(0.f, 0.f, 0.f, 0.f), p = w;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = rg + r * RPP;
            const float ak = sh_ak[i] * ik, aq = sh_aq[i] * iq;
            w.x = fmaf(ak, s[r].x, w.x); w.y = fmaf(ak, s[r].y, w.y);
            w.z = fmaf(ak, s[r].z, w.z); w.w = fmaf(ak, s[r].w, w.w);
            p.x = fmaf(aq, s[r].x, p.x); p.y = fmaf(aq, s[r].y, p.y);
            p.z = fmaf(aq, s[r].z, p.z); p.w = fmaf(aq, s[r].w, p.w);
        }
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
            w.x += __shfl_xor_sync(0xffffffffu, w.x, off);
            w.y += __shfl_xor_sync(0xffffffffu, w.y, off);
            w.z += __shfl_xor_sync(0xffffffffu, w.z, off);
            w.w += __shfl_xor_sync(0xffffffffu, w.w, off);
            p.x += __shfl_xor_sync(0xffffffffu, p.x, off);
            p.y += __shfl_xor_sync(0xffffffffu, p.y, off);
            p.z += __shfl_xor_sync(0xffffffffu, p.z, off);
            p.w += __shfl_xor_sync(0xffffffffu, p.w, off);
        }
        if (lane < LPR) {
            sh_red_w[warp][c4 * 4 + 0] = w.x; sh_red_w[warp][c4 * 4 + 1] = w.y;
            sh_red_w[warp][c4 * 4 + 2] = w.z; sh_red_w[warp][c4 * 4 + 3] = w.w;
            sh_red_p[warp][c4 * 4 + 0] = p.x; sh_red_p[warp][c4 * 4 + 1] = p.y;
            sh_red_p[warp][c4 * 4 + 2] = p.z; sh_red_p[warp][c4 * 4 + 3] = p.w;
        }
        __syncthreads();

        // 4. Per value column: u = beta (v - w), o = p + (k.q) u.
        if (tid < DVS) {
            float ws = 0.f, ps = 0.f, kqs = 0.f;
#pragma unroll
            for (int i = 0; i < Sh::kWarps; ++i) {
                ws += sh_red_w[i][tid];
                ps += sh_red_p[i][tid];
                kqs += sh_kq[i];
            }
            const int j = slab * DVS + tid;
            const long long vo = tok * dv + j;
            const float u = beta[tok] * (ld_f(v + vo) - ws);
            st_f(o + vo, fmaf(kqs * ik * iq, u, ps));
            sh_u[tid] = u;
        }
        __syncthreads();

        // 5. S' = Diag(alpha) S + k u^T, streamed out; kept for the next token.
        const float4 u4 = make_float4(sh_u[c4 * 4 + 0], sh_u[c4 * 4 + 1],
                                      sh_u[c4 * 4 + 2], sh_u[c4 * 4 + 3]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = rg + r * RPP;
            const float a = sh_a[i], kk = sh_k[i] * ik;
            float4 x;
            x.x = fmaf(a, s[r].x, kk * u4.x);
            x.y = fmaf(a, s[r].y, kk * u4.y);
            x.z = fmaf(a, s[r].z, kk * u4.z);
            x.w = fmaf(a, s[r].w, kk * u4.w);
            __stcs(reinterpret_cast<float4*>(Sq + (long long)i * dv + col), x);
            s[r] = x;
        }
    }
}

// The state after the accepted prefix of a multi-token step: for each
// (sequence, head), states[n, accept[n] - 1] when accept[n] > 0, else S_in[n]
// (accept values are clamped to [0, Ts]).  One CTA per (sequence, head).
__global__ void __launch_bounds__(256)
state_gather_kernel(const float* __restrict__ states, const float* S_in,
                    const int32_t* __restrict__ accept, float* S_out, int Ts, int H,
                    long long elems)
{
    const long long nh = blockIdx.x;
    const long long n = nh / H, h = nh % H;
    int a = accept[n];
    a = a < 0 ? 0 : (a > Ts ? Ts : a);
    const float4* src = reinterpret_cast<const float4*>(
        a > 0 ? states + ((n * Ts + (a - 1)) * H + h) * elems : S_in + nh * elems);
    float4* dst = reinterpret_cast<float4*>(S_out + nh * elems);
    if (reinterpret_cast<const void*>(src) == reinterpret_cast<const void*>(dst)) return;
    for (long long i = threadIdx.x; i < elems / 4; i += blockDim.x) dst[i] = __ldcs(src + i);
}

template <typename TI, typename TO, int D>
cudaError_t launch_typed(const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* S_in, float* S_out,
                         int32_t N, int32_t Ts, int32_t H, void* o, const GateArgs& gate,
                         cudaStream_t stream)
{
    // Slab widths and thread counts: 32 KiB of state per CTA at d = 128
    // (8 float4 per thread), one warp-row pattern per smaller head size.
    constexpr int DVS = D >= 64 ? 64 : D;
    constexpr int THREADS = D == 128 ? 256 : (D == 64 ? 128 : (D == 32 ? 64 : 32));
    const long long blocks = (long long)N * H * (D / DVS);
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    decode_kernel<TI, TO, D, DVS, THREADS><<<(unsigned)blocks, THREADS, 0, stream>>>(
        static_cast<const TI*>(q), static_cast<const TI*>(k), static_cast<const TI*>(v),
        g, beta, S_in, S_out, static_cast<TO*>(o), D, Ts, H, gate.A, gate.q_scale);
    return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_d(int32_t d, const void* q, const void* k, const void* v,
                     const float* g, const float* beta, const float* S_in, float* S_out,
                     int32_t N, int32_t Ts, int32_t H, void* o, const GateArgs& gate,
                     cudaStream_t stream)
{
    switch (d) {
        case 16: return launch_typed<TI, TO, 16>(q, k, v, g, beta, S_in, S_out, N, Ts, H, o, gate, stream);
        case 32: return launch_typed<TI, TO, 32>(q, k, v, g, beta, S_in, S_out, N, Ts, H, o, gate, stream);
        case 64: return launch_typed<TI, TO, 64>(q, k, v, g, beta, S_in, S_out, N, Ts, H, o, gate, stream);
        case 128: return launch_typed<TI, TO, 128>(q, k, v, g, beta, S_in, S_out, N, Ts, H, o, gate, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_multi(const void* q, const void* k, const void* v, const float* log_alpha,
                         const float* beta, const float* S_in, float* S_out, int32_t N,
                         int32_t Ts, int32_t H, int32_t d, kda_dtype_t dtype, void* o,
                         const GateArgs& gate, cudaStream_t stream)
{
    switch (dtype) {
        case KDA_BF16:
            return launch_d<__nv_bfloat16, __nv_bfloat16>(d, q, k, v, log_alpha, beta, S_in, S_out,
                                                          N, Ts, H, o, gate, stream);
        case KDA_BF16_F32OUT:
            return launch_d<__nv_bfloat16, float>(d, q, k, v, log_alpha, beta, S_in, S_out, N, Ts,
                                                  H, o, gate, stream);
        default:
            return launch_d<float, float>(d, q, k, v, log_alpha, beta, S_in, S_out, N, Ts, H, o,
                                          gate, stream);
    }
}

}  // namespace

cudaError_t launch_decode(const void* q, const void* k, const void* v,
                          const float* log_alpha, const float* beta, float* S,
                          int32_t N, int32_t H, int32_t d, kda_dtype_t dtype,
                          void* o, const GateArgs& gate, cudaStream_t stream)
{
    return launch_multi(q, k, v, log_alpha, beta, S, S, N, 1, H, d, dtype, o, gate, stream);
}

cudaError_t launch_decode_multi(const void* q, const void* k, const void* v,
                                const float* log_alpha, const float* beta, const float* S_in,
                                float* states, int32_t N, int32_t Ts, int32_t H, int32_t d,
                                kda_dtype_t dtype, void* o, const GateArgs& gate,
                                cudaStream_t stream)
{
    return launch_multi(q, k, v, log_alpha, beta, S_in, states, N, Ts, H, d, dtype, o, gate,
                        stream);
}

cudaError_t launch_state_gather(const float* states, const float* S_in, const int32_t* accept,
                                int32_t N, int32_t Ts, int32_t H, int32_t d_k, int32_t d_v,
                                float* S_out, cudaStream_t stream)
{
    const long long blocks = (long long)N * H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    state_gather_kernel<<<(unsigned)blocks, 256, 0, stream>>>(states, S_in, accept, S_out, Ts, H,
                                                              (long long)d_k * d_v);
    return cudaGetLastError();
}

}  // namespace kda
