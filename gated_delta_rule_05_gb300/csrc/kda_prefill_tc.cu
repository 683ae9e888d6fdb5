// kda_prefill_tc.cu -- chunked KDA prefill on the Blackwell tensor cores
// (tcgen05.mma, TMEM accumulators, TMA-staged tiles), bf16 q/k/v, d_k = d_v =
// 128, chunks of C = 64 tokens, fp32 state carried in tensor memory: the
// single-CTA kernel, one CTA per (sequence, head) running every phase of
// every chunk.  It is the path for batches with many (sequence, head) units;
// batches with few units take the producer / consumer kernel of
// kda_prefill_split.cu.
//
// Method.  The recurrence of "[논문 리뷰] Kimi K3 Technical Report"
// (jw9603.github.io) section 3.2, S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T,
// o_t = S_t^T q_t, evaluated in the chunkwise-parallel form of "Kimi 모델 분석"
// (rlaope.github.io) section "순환을 GPU에 올리기": within a chunk the token
// updates are folded into dense products (the WY/UT form, with the triangular
// inverse built from small block products) and only the state passes from one
// chunk to the next; the decay is normalised to the chunk start.  The chunk
// algebra, the Gram factorisation, the operand precisions and the UT solve
// are described with the phases in kda_tc_chunk.cuh.
//
// CTA roles (320 threads):
//   warp 0      TMA: q, k, g tiles (64 x 128) and the v tile, beta by plain
//               loads one chunk ahead, the next chunk's tiles prefetched to L2
//   warp 1      issues every tcgen05.mma and commit (warp-wide, one elected lane)
//   warps 2..9  the compute group (256 threads) runs every CUDA-core phase of a
//               chunk together: gate prep, state decay, Gram readout, the UT
//               solve's diagonal blocks, and every TMEM readout.  The chunk's
//               steps form one dependency chain, so the group moves through it
//               as a whole; the state decay overlaps the Gram product on the
//               tensor cores.
//
// Every wait is bounded in time; a timeout sets a flag in the workspace,
// drains the CTA and frees its tensor memory.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>

#include "kda_internal.cuh"
#include "kda_tc_chunk.cuh"

namespace kda {

// ------------------------------------------------------------ host side
// The driver's tensor-map encoder (looked up once through the runtime).  Also
// used by the split kernel's launcher.
PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A 2-D map over a [T, H * 128] row-major tensor with boxes of box_x columns
// by 64 rows (one chunk).
bool tc_make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int H,
                 long long T, int box_x, CUtensorMapSwizzle swz)
{
    using tc::kC;
    using tc::kD;
    auto fn = tc_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H * kD, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * kD * elem};
    const cuuint32_t box[2] = {(cuuint32_t)box_x, (cuuint32_t)kC};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && debug_enabled())
        fprintf(stderr, "kda: cuTensorMapEncodeTiled failed (CUresult %d, box %d x %d)\n", (int)r,
                box_x, kC);
    return r == CUDA_SUCCESS;
}

namespace {

using namespace tc;

constexpr int kThreads = 320;

// ------------------------------------------------------------- the kernel
// FUSED: the gate prologue runs in the kernel (gate.A not null).
template <typename TO, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_o,
                  const float* __restrict__ beta, const float* S0,
                  const int32_t* __restrict__ cu, int32_t* ws, long long total_tokens, int H,
                  TO* __restrict__ o, float* S_final, const SnapArgs snap,
                  const GateArgs gate)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Ctx X;
    X.sm = sm;
    X.bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    X.desc = reinterpret_cast<StepDesc*>(sm + OFF_DESC);
    X.misc = reinterpret_cast<Misc*>(sm + OFF_MISC);
    X.ws_err = ws + kWsTimeoutWord;
    X.ws_abort = nullptr;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = blockIdx.x / H, h = blockIdx.x % H;

    long long bos = 0, eos = total_tokens;
    int n = 0;
    if (cu != nullptr) {
        if (ws[kWsErrorWord] != 0) return;     // uniform: every thread returns
        n = ws[kWsHeaderBytes / sizeof(int32_t) + rank];
        bos = cu[n];
        eos = cu[n + 1];
    }
    const int nch = (int)((eos - bos + kC - 1) / kC);
    const long long sbase = ((long long)n * H + h) * kD * kD;

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) mbar_init(&X.bar[b], 1);
        X.misc->abort = 0;
        X.misc->wide = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&X.misc->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = X.misc->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_g);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_o);
        }
        float* sBin = reinterpret_cast<float*>(sm + OFF_BIN);
        int issued_qkg = 0, issued_v = 0;
        // Each lane's two beta values are loaded one chunk ahead, so that
        // their latency passes while the tiles are still in use; the next
        // chunk's tiles are prefetched into L2 for the same reason.  Both keep
        // plain global latency off the step between one chunk's W product and
        // the next chunk's gate prep.
        float b_next[2];
        auto load_beta = [&](int ch, float* b) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const long long t = bos + (long long)ch * kC + lane * 2 + j;
                b[j] = (t < eos) ? beta[t * H + h] : 0.f;
            }
        };
        if (nch > 0) load_beta(0, b_next);
        for (int ch = 0; ch < nch; ++ch) {
            const long long t0 = bos + (long long)ch * kC;
            int ok = 1;
            if (lane == 0 && ch > 0) ok = wait_bar(X, B_QKG_EMPTY, ch - 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            sBin[lane * 2] = b_next[0];
            sBin[lane * 2 + 1] = b_next[1];
            __syncwarp();
            if (ch + 1 < nch) load_beta(ch + 1, b_next);
            if (lane == 0) {
                mbar_arrive_expect_tx(&X.bar[B_QKG_FULL], 2 * 16384 + 32768);
                tma_load_2d(sm + OFF_Q, &tm_q, h * kD, (int32_t)t0, &X.bar[B_QKG_FULL]);
                tma_load_2d(sm + OFF_K, &tm_k, h * kD, (int32_t)t0, &X.bar[B_QKG_FULL]);
                tma_load_2d(sm + OFF_G, &tm_g, h * kD, (int32_t)t0, &X.bar[B_QKG_FULL]);
                ++issued_qkg;
                ok = (ch == 0) ? 1 : wait_bar(X, B_V_EMPTY, ch - 1);
                if (ok) {
                    mbar_arrive_expect_tx(&X.bar[B_V_FULL], 16384);
                    tma_load_2d(sm + OFF_V, &tm_v, h * kD, (int32_t)t0, &X.bar[B_V_FULL]);
                    tma_load_2d(sm + OFF_V + 8192, &tm_v, h * kD + 64, (int32_t)t0,
                                &X.bar[B_V_FULL]);
                    ++issued_v;
                }
                if (ok && ch + 1 < nch) {
                    const int32_t tn = (int32_t)(t0 + kC);
                    tma_prefetch_l2_2d(&tm_q, h * kD, tn);
                    tma_prefetch_l2_2d(&tm_k, h * kD, tn);
                    tma_prefetch_l2_2d(&tm_g, h * kD, tn);
                    tma_prefetch_l2_2d(&tm_v, h * kD, tn);
                    tma_prefetch_l2_2d(&tm_v, h * kD + 64, tn);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
        }
        // On abort, let the copies already issued land before the CTA exits.
        if (lane == 0 && X.misc->abort) {
            if (issued_qkg) mbar_wait(&X.bar[B_QKG_FULL], (issued_qkg - 1) & 1, 1ll << 28);
            if (issued_v) mbar_wait(&X.bar[B_V_FULL], (issued_v - 1) & 1, 1ll << 28);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        // The whole warp runs this loop; the issue helpers elect one lane.
        if (nch > 0) {
            const FrontDescs D = make_front_descs(sm, OFF_G);
            for (int step = 0;; ++step) {
                if (!warp_wait(X, B_OPS, step)) break;
                tc_fence_after();
                const StepDesc d = X.desc[step & 1];
                if (!mma_front(X, tmem, D, step)) break;
                if (!warp_wait(X, B_CV, step)) break;   // -W^T, S^T copy, v tile ready
                tc_fence_after();
                // The U^T P^T term of O^T follows once U^T is ready.
                mma_back_c(tmem, smem_u32(sm + OFF_WT), smem_u32(sm + OFF_T16), smem_u32(sm + OFF_V));
                mma_commit(&X.bar[B_MMA_C]);
                if (d.last_pass) mma_commit(&X.bar[B_V_EMPTY]);
                if (!warp_wait(X, B_U, step)) break;
                tc_fence_after();
                mma_back_os(tmem, smem_u32(sm + OFF_P));
                mma_commit(&X.bar[B_MMA_OS]);
                if (d.last_step) break;
            }
        }
    } else {
        // -------------------------------------------------- compute group
        const Lane t = make_lane(tid - 64, warp, lane);
        const int ct = t.ct;
        const int seq_off = (cu != nullptr && snap.interval > 0) ? snap.offsets[n] : 0;
        const float* Ah = FUSED ? gate.A + (long long)h * kD : nullptr;
        state_load(t, tmem, S0, sbase);

        int step = 0, chunk_v = 0;
        bool alive = true;
        for (int ch = 0; ch < nch && alive; ++ch) {
            const long long t0 = bos + (long long)ch * kC;
            const int len = (eos - t0 < kC) ? (int)(eos - t0) : kC;
            if (!group_wait(X, B_QKG_FULL, ch)) break;
            float2 Gq[16];
            PassParams pp;
            if (FUSED) qk_norms(X, t, gate.q_scale);
            const float* sG = reinterpret_cast<const float*>(sm + OFF_G);
            const int npass = gate_prep<FUSED>(X, t, len, sG, Ah, Gq, pp);
            for (int p = 0; p < npass; ++p) {
                const Pass ps = select_pass(pp, p, npass, len);
                pass_factors(X, t, ps, reinterpret_cast<float*>(sm + OFF_GL));
                if (ct == 0) {
                    StepDesc d;
                    d.t0 = (int32_t)t0;
                    d.len = len;
                    d.lo = ps.lo;
                    d.hi = ps.hi;
                    d.first_pass = (p == 0);
                    d.last_pass = (p == npass - 1);
                    d.last_step = (ch == nch - 1) && (p == npass - 1);
                    d.chunk = ch;
                    X.desc[step & 1] = d;
                }
                // The previous chunk's O store has read its staging area and
                // everyone has read the decay stats: both lie in the Gram
                // operand region.  The (e^G K)^T tile takes the g tile's place.
                if (ct == 0) bulk_wait_group_read0();
                group_sync();
                gram_operands<FUSED, sizeof(TO) == 4>(X, t, ps, Gq, sm + OFF_QG, sm + OFF_KT, sm + OFF_G);
                fence_proxy_async_smem();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_OPS]);

                // ---- while the Gram runs: the state decay with its fp16 copy.
                // (The v tile is converted to fp16 during the UT solve, by the
                // warps that run no chain: during the Gram its shared-memory
                // traffic competes with the product's operand reads.)
                const StepDesc d = X.desc[step & 1];
                const uint32_t v_phase = (uint32_t)chunk_v;
                if (d.last_pass) ++chunk_v;
                tc_fence_after();
                state_decay(t, tmem, reinterpret_cast<const float*>(sm + OFF_GL),
                            d.first_pass ? snapshot_at(snap, ch, eos - bos, seq_off, H, h) : nullptr);
                tc_fence_before();

                if (!gram_readout(X, t, tmem, ps.lo, ps.hi, step, sm + OFF_P)) { alive = false; break; }
                ut_solve_mma(X, t, sm + OFF_T16, d.first_pass ? sm + OFF_V : nullptr, v_phase);
                if (!w_readout(X, t, tmem, step, sm + OFF_WT)) { alive = false; break; }
                if (ct == 0) {
                    // The W product has read the (e^G K)^T tile: after the
                    // chunk's last pass the next q / k / g may load.
                    if (d.last_pass) mbar_arrive(&X.bar[B_QKG_EMPTY]);
                    mbar_arrive(&X.bar[B_CV]);
                }

                // ---- U^T -> fp16 A operand
                if (!group_wait(X, B_MMA_C, step)) { alive = false; break; }
                tc_fence_after();
                u_to_f16(t, tmem);
                tc_fence_before();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_U]);

                // ---- O^T readout (the staging area is the A / X region, idle
                // until the next chunk's Gram operands).
                if (!group_wait(X, B_MMA_OS, step)) { alive = false; break; }
                tc_fence_after();
                {
                    uint32_t dd[32];
                    o_load(t, tmem, dd);
                    const bool tma_out = (sizeof(TO) == 2) && d.lo == 0 && d.hi == kC;
                    if (tma_out) tc_fence_before();
                    o_store<TO>(t, dd, tma_out, &tm_o, sm + OFF_OST, o, (long long)d.t0, d.lo,
                                d.hi, h, H);
                    if (!tma_out) tc_fence_before();
                }
                ++step;
            }
        }
        if (ct == 0) bulk_wait_group0();                   // the last O store has landed
        if (!*reinterpret_cast<volatile int32_t*>(&X.misc->abort)) {
            if (S_final) state_store(t, tmem, S_final, sbase);
            float* last = snapshot_at(snap, nch, eos - bos, seq_off, H, h);
            if (last) state_store(t, tmem, last, 0);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <typename TO, bool FUSED>
cudaError_t launch_typed(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* S0, const int32_t* cu, int32_t N,
                         int64_t T, int32_t H, void* o, float* S_final, int32_t* ws,
                         const SnapArgs& snap, const GateArgs& gate, cudaStream_t stream)
{
    CUtensorMap mq, mk, mg, mv, mo;
    // The output map is used for bf16 output only (fp32 output is stored by
    // the threads); for fp32 a copy of the q map fills the slot.
    const bool bf16_out = sizeof(TO) == 2;
    if (!tc_make_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        (bf16_out && !tc_make_map(&mo, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD,
                               CU_TENSOR_MAP_SWIZZLE_NONE)) ||
        !tc_make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tc_make_map(&mg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, T, kD, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tc_make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    auto kern = prefill_tc_kernel<TO, FUSED>;
    static bool attr_set = false;   // benign race: every writer stores the same value
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) {
            if (debug_enabled())
                fprintf(stderr, "kda: cudaFuncSetAttribute(%u B smem) failed: %s\n",
                        kSmemBytes, cudaGetErrorString(e));
            return e;
        }
        attr_set = true;
    }
    const long long blocks = (long long)N * H;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (!bf16_out) mo = mq;
    kern<<<(unsigned)blocks, kThreads, kSmemBytes, stream>>>(mq, mk, mg, mv, mo, beta, S0, cu, ws,
                                                            (long long)T, H,
                                                            static_cast<TO*>(o), S_final, snap,
                                                            gate);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess && debug_enabled())
        fprintf(stderr, "kda: prefill_tc launch failed: %s\n", cudaGetErrorString(e));
    return e;
}

}  // namespace

bool prefill_tc_supported(kda_dtype_t dtype, int32_t d, int64_t total_tokens)
{
    if (getenv("KDA_FORCE_SIMT") != nullptr) return false;
    return (dtype == KDA_BF16 || dtype == KDA_BF16_F32OUT) && d == kD && total_tokens > 0 &&
           tc_encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const void* q, const void* k, const void* v,
                              const float* log_alpha, const float* beta, const float* S0,
                              const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                              int32_t H, kda_dtype_t dtype, void* o, float* S_final,
                              int32_t* ws, const SnapArgs& snap, const GateArgs& gate,
                              cudaStream_t stream)
{
    const bool fused = gate.A != nullptr;
    if (dtype == KDA_BF16_F32OUT)
        return fused ? launch_typed<float, true>(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs,
                                                 total_tokens, H, o, S_final, ws, snap, gate, stream)
                     : launch_typed<float, false>(q, k, v, log_alpha, beta, S0, cu_seqlens,
                                                  num_seqs, total_tokens, H, o, S_final, ws, snap,
                                                  gate, stream);
    return fused ? launch_typed<__nv_bfloat16, true>(q, k, v, log_alpha, beta, S0, cu_seqlens,
                                                     num_seqs, total_tokens, H, o, S_final, ws, snap,
                                                     gate, stream)
                 : launch_typed<__nv_bfloat16, false>(q, k, v, log_alpha, beta, S0, cu_seqlens,
                                                      num_seqs, total_tokens, H, o, S_final, ws,
                                                      snap, gate, stream);
}

}  // namespace kda
