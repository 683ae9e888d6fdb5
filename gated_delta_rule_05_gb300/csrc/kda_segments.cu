// kda_segments.cu -- the second pass of the chunk-group parallel prefill of
// one sequence (kda_prefill_segmented).
//
// The first pass (the producer / consumer kernel, kda_prefill_split.cu, with
// SegArgs) cuts the sequence into G segments and runs every segment's chain at
// once: segment 0 from the caller's S0 into o; every later segment g twice on
// the same producer operands, from S = 0 (outputs o_loc, final state L_g) and,
// with v = 0, from S = I (outputs qt_t = Phi_t^T q_t, final state M_g = Phi_g,
// where Phi_t is the product of the transitions (I - b k k^T) Diag(a) from the
// segment start to token t).  The recurrence of "[논문 리뷰] Kimi K3 Technical
// Report" section 3.2 is linear in (S, v), so with S_g the true state at the
// start of segment g,
//     S_t = Phi_t S_g + S_loc,t        o_t = S_t^T q_t = o_loc,t + S_g^T qt_t,
//     S_1 = L_0,   S_{g+1} = M_g S_g + L_g,   S_final = S_G.
// Only the state passes from chunk to chunk, and here from segment to segment
// ("Kimi 모델 분석", section "순환을 GPU에 올리기"; the K3 review's section 13
// describes the multi-GPU form, KDA context parallelism).
//
//   segment_scan_kernel   the scan over segments, fp32 on the CUDA cores.
//                         Column block j of S_{g+1} depends only on column
//                         block j of S_g, so each CTA runs the whole scan for
//                         16 state columns of one head.  M_{g+1} is copied in
//                         (asynchronously, 16 bytes per copy) while step g
//                         computes.  It writes S_g^T in fp16, in the swizzled
//                         layout of an MMA operand.
//   segment_fixup_kernel  o_t = o_loc,t + S_g^T qt_t for every token of
//                         segments 1 .. G-1: one tcgen05 product per tile of
//                         128 tokens (D = QT S_g, M = N = K = 128, fp16
//                         operands, fp32 accumulator in tensor memory), the
//                         qt tile loaded by TMA; each thread then adds its
//                         token's o_loc row, loaded while the product runs,
//                         and stores its o row.
#include <cudaTypedefs.h>
#include <stdio.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {

bool tc_make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int H,
                 long long T, int box_x, CUtensorMapSwizzle swz);

namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr int kScanCols = 16;             // state columns per scan CTA
constexpr int kLdM = 132;                 // row stride (floats) of M_g in shared memory: 16-byte
                                          //   aligned rows, at most 2-way conflicts on column reads
constexpr int kTile = 128;                // tokens per fix-up CTA (even chunks per segment)
constexpr int kFixThreads = 128;          // four warps: one TMEM lane quarter each
constexpr uint32_t FX_A = 0;              // qt tile: 2 K blocks x [128 tok][64 k] fp16 (32 KB)
constexpr uint32_t FX_B = 32768;          // S_g^T: 2 K blocks x [128 v][64 k] fp16 (32 KB)
constexpr uint32_t FX_BAR = 65536;        // 2 mbarriers
constexpr uint32_t FX_TM = FX_BAR + 16;   // TMEM base address
constexpr uint32_t kFixSmem = FX_BAR + 64 + 1024;   // + alignment slack
constexpr uint32_t kStateHalfs = kD * kD;           // one S_g^T operand block (32 KB)

// Index (in halfs) of element (row r, column c) of a [128][128] fp16 operand
// in the K-major layout with the 128-byte swizzle: two 64-column blocks of
// 16 KB, 8-row groups 1024 bytes apart, the 16-byte chunk j of row r stored at
// position j ^ (r % 8).
__device__ __forceinline__ uint32_t swz_index(int r, int c)
{
    return ((uint32_t)(c >> 6) << 13) + ((uint32_t)(r >> 3) << 9) + ((uint32_t)(r & 7) << 6) +
           ((((uint32_t)(c & 63) >> 3) ^ (uint32_t)(r & 7)) << 3) + (uint32_t)(c & 7);
}

// Asynchronous 16-byte global -> shared copies (completion tracked per
// thread in groups).
__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// grid (H, d_v / 16).  st_aux: L_g = st_aux[g], M_g = st_aux[G + g] ([H][d][d]
// each).  Writes S_g^T (g >= 1) as fp16 operand blocks to sstart[g][h] and
// S_G to S_final (if not null).  Shared memory: M in two buffers (the next
// one copied in while a step computes) and this CTA's 16 columns of S_g.
__global__ void __launch_bounds__(kThreads)
segment_scan_kernel(const float* __restrict__ st_aux, int G, int H, __half* __restrict__ sstart,
                    float* __restrict__ S_final)
{
    extern __shared__ __align__(16) float smem[];
    float* sS = smem + 2 * kD * kLdM;           // S_g [k][16]
    const int h = blockIdx.x, j0 = blockIdx.y * kScanCols, tid = threadIdx.x;
    const size_t state = (size_t)kD * kD;
    // M_g into buffer (g - 1) % 2: 4096 copies of 16 bytes, 16 per thread.
    auto load_M = [&](int g) {
        const float* Mg = st_aux + ((size_t)(G + g) * H + h) * state;
        float* dst = smem + ((g - 1) & 1) * kD * kLdM;
        for (int e = tid; e < kD * kD / 4; e += kThreads) {
            const int r = e >> 5, c4 = e & 31;
            cp_async16(dst + r * kLdM + 4 * c4, Mg + (size_t)r * kD + 4 * c4);
        }
        cp_async_commit();
    };
    if (G > 1) load_M(1);
    const float* L0 = st_aux + (size_t)h * state;
    // S_1 = L_0 (columns j0 .. j0+15)
    for (int e = tid; e < kD * kScanCols; e += kThreads) {
        const int r = e / kScanCols, c = e % kScanCols;
        sS[e] = L0[(size_t)r * kD + j0 + c];
    }
    __syncthreads();
    const int i = tid >> 1, c0 = (tid & 1) * 8;   // this thread: row i, columns c0 .. c0+7
    for (int g = 1; g < G; ++g) {
        const float* Lg = st_aux + ((size_t)g * H + h) * state;
        __half* Sg = sstart + ((size_t)g * H + h) * kStateHalfs;
        {
            // S_g^T out: row v = j0 + c of the operand, 16-byte chunk q (k = 8q .. 8q+7)
            const int c = tid & 15, q = tid >> 4;
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pk[e] = pack_f16x2(sS[(8 * q + 2 * e) * kScanCols + c], sS[(8 * q + 2 * e + 1) * kScanCols + c]);
            *reinterpret_cast<uint4*>(Sg + swz_index(j0 + c, 8 * q)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = Lg[(size_t)i * kD + j0 + c0 + c];
        if (g + 1 < G) {
            load_M(g + 1);                        // its buffer was last read in step g - 1
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();                          // M_g has landed for every thread
        const float* sM = smem + ((g - 1) & 1) * kD * kLdM + i * kLdM;
#pragma unroll 2
        for (int k4 = 0; k4 < kD / 4; ++k4) {
            const float4 m4 = *reinterpret_cast<const float4*>(sM + 4 * k4);
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int k = 4 * k4 + kk;
                const float4 s0 = *reinterpret_cast<const float4*>(sS + k * kScanCols + c0);
                const float4 s1 = *reinterpret_cast<const float4*>(sS + k * kScanCols + c0 + 4);
                acc[0] = fmaf(mv[kk], s0.x, acc[0]);
                acc[1] = fmaf(mv[kk], s0.y, acc[1]);
                acc[2] = fmaf(mv[kk], s0.z, acc[2]);
                acc[3] = fmaf(mv[kk], s0.w, acc[3]);
                acc[4] = fmaf(mv[kk], s1.x, acc[4]);
                acc[5] = fmaf(mv[kk], s1.y, acc[5]);
                acc[6] = fmaf(mv[kk], s1.z, acc[6]);
                acc[7] = fmaf(mv[kk], s1.w, acc[7]);
            }
        }
        __syncthreads();                              // everyone has read S_g and M_g
#pragma unroll
        for (int c = 0; c < 8; ++c) sS[i * kScanCols + c0 + c] = acc[c];
        __syncthreads();
    }
    if (S_final != nullptr) {
        for (int e = tid; e < kD * kScanCols; e += kThreads) {
            const int r = e / kScanCols, c = e % kScanCols;
            S_final[(size_t)h * state + (size_t)r * kD + j0 + c] = sS[e];
        }
    }
}

__device__ __forceinline__ void store4(float* p, float a, float b, float c, float d)
{
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

__device__ __forceinline__ void store4(__nv_bfloat16* p, float a, float b, float c, float d)
{
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

// The two fp16 values of a packed pair, as floats.
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w)
{
    return make_float2(__half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))),
                       __half2float(__ushort_as_half((unsigned short)(w >> 16))));
}

// grid (tiles of 128 tokens after segment 0, H).  o_loc: [T][H][d] fp16; the
// qt map covers [T][H d] fp16.  A tile never straddles a segment (segments
// are whole tiles).  A wait that gives up sets bit 1 of *timeout_word.
template <typename TO>
__global__ void __launch_bounds__(kFixThreads, 3)
segment_fixup_kernel(const __grid_constant__ CUtensorMap tm_qt, const __half* __restrict__ o_loc,
                     const __half* __restrict__ sstart, long long T, int H, long long seg_tokens,
                     TO* __restrict__ o, int32_t* timeout_word)
{
    extern __shared__ __align__(1024) uint8_t fx_raw[];
    uint8_t* sm = fx_raw + ((1024u - (smem_u32(fx_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + FX_BAR);
    const int h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long t0 = seg_tokens + (long long)blockIdx.x * kTile;
    if (t0 >= T) return;                               // uniform
    const int g = (int)(t0 / seg_tokens);
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(reinterpret_cast<uint32_t*>(sm + FX_TM), kD);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + FX_TM);
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], 2 * 32768);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
            for (int rh = 0; rh < 2; ++rh)
                tma_load_2d(sm + FX_A + kb * 16384 + rh * 8192, &tm_qt, h * kD + kb * 64,
                            (int32_t)(t0 + rh * 64), &bar[0]);
        bulk_load(sm + FX_B, sstart + ((size_t)g * H + h) * kStateHalfs, 32768, &bar[0]);
    }
    // This thread's token: TMEM lane r of the product.  Its o_loc row (256
    // bytes) is loaded while the operand tiles land and the product runs.
    const int r = warp * 32 + lane;
    const long long t = t0 + r;
    const size_t row = ((size_t)t * H + h) * kD;
    uint4 lv[16];
    if (t < T) {
#pragma unroll
        for (int q = 0; q < 16; ++q) lv[q] = reinterpret_cast<const uint4*>(o_loc + row)[q];
    }
    bool ok = mbar_wait(&bar[0], 0);
    if (warp == 0) {
        ok = __all_sync(0xffffffffu, ok) != 0;
        if (ok) {
            tc_fence_after();
            const uint32_t id = make_idesc_f16(128, 128, false, false);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int kb = s >> 2;
                const uint64_t da = make_sdesc(smem_u32(sm + FX_A + kb * 16384), 16, 1024, kSwizzle128B);
                const uint64_t db = make_sdesc(smem_u32(sm + FX_B + kb * 16384), 16, 1024, kSwizzle128B);
                mma_ss(tmem, da + 2 * (s & 3), db + 2 * (s & 3), id, s > 0);
            }
            mma_commit(&bar[1]);
        } else if (lane == 0) {
            mbar_wait(&bar[0], 0, 1ll << 28);         // let the copies land before exiting
        }
    }
    ok = ok && mbar_wait(&bar[1], 0);
    if (!ok && lane == 0) atomicOr(timeout_word, 2);
    // o = o_loc + D, 32 columns at a time, straight from TMEM to global.
    if (ok) {
        tc_fence_after();
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            uint32_t d[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + cb * 32, d);
            tmem_ld_wait();
            if (t < T) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 l = lv[4 * cb + q];
                    const uint32_t lw[4] = {l.x, l.y, l.z, l.w};
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = f16x2_to_float2(lw[e]);
                        x[2 * e] = f.x + __uint_as_float(d[8 * q + 2 * e]);
                        x[2 * e + 1] = f.y + __uint_as_float(d[8 * q + 2 * e + 1]);
                    }
                    TO* op = o + row + 32 * cb + 8 * q;
                    store4(op, x[0], x[1], x[2], x[3]);
                    store4(op + 4, x[4], x[5], x[6], x[7]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kD);
    }
}

template <typename TO>
cudaError_t launch_fixup(const CUtensorMap& map, const __half* o_loc, const __half* sstart,
                         long long T, int H, long long seg_tokens, void* o, int32_t* timeout_word,
                         cudaStream_t stream)
{
    auto kern = segment_fixup_kernel<TO>;
    static bool attr = false;   // benign race: every writer stores the same value
    if (!attr) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFixSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const long long rest = T - seg_tokens;
    const dim3 grid((unsigned)((rest + kTile - 1) / kTile), (unsigned)H);
    kern<<<grid, kFixThreads, kFixSmem, stream>>>(map, o_loc, sstart, T, H, seg_tokens,
                                                  static_cast<TO*>(o), timeout_word);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_segment_fixup(const SegArgs& seg, int64_t total_tokens, int32_t H,
                                 kda_dtype_t dtype, void* o, float* S_final, __half* sstart,
                                 int32_t* timeout_word, cudaStream_t stream)
{
    const int scan_smem = (2 * kD * kLdM + kD * kScanCols) * (int)sizeof(float);
    static bool scan_attr = false;   // benign race: every writer stores the same value
    if (!scan_attr) {
        const cudaError_t e = cudaFuncSetAttribute(segment_scan_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   scan_smem);
        if (e != cudaSuccess) return e;
        scan_attr = true;
    }
    segment_scan_kernel<<<dim3((unsigned)H, kD / kScanCols), kThreads, scan_smem, stream>>>(
        seg.st_aux, seg.G, H, sstart, S_final);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long seg_tokens = (long long)seg.seg_chunks * 64;
    if (total_tokens - seg_tokens <= 0) return cudaSuccess;
    const __half* o_loc = seg.o_aux;
    const __half* qt = seg.o_aux + (size_t)total_tokens * H * kD;
    CUtensorMap map;
    if (!tc_make_map(&map, qt, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, H, total_tokens, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    e = (dtype == KDA_BF16)
            ? launch_fixup<__nv_bfloat16>(map, o_loc, sstart, total_tokens, H, seg_tokens, o,
                                          timeout_word, stream)
            : launch_fixup<float>(map, o_loc, sstart, total_tokens, H, seg_tokens, o,
                                  timeout_word, stream);
    if (e != cudaSuccess && debug_enabled())
        fprintf(stderr, "kda: segment fix-up launch failed: %s\n", cudaGetErrorString(e));
    return e;
}

}  // namespace kda
