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
//                         16 state columns of one head.  It writes S_g^T in
//                         fp16, in the swizzled layout of an MMA operand.
//   segment_fixup_kernel  o_t = o_loc,t + S_g^T qt_t for every token of
//                         segments 1 .. G-1: one tcgen05 product per tile of
//                         128 tokens (D = QT S_g, M = N = K = 128, fp16
//                         operands, fp32 accumulator in tensor memory), the
//                         qt tile loaded by TMA, o_loc added in the epilogue.
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
constexpr int kLdM = 129;                 // row stride (floats) of M_g in shared memory
constexpr int kTile = 128;                // tokens per fix-up CTA (even chunks per segment)
constexpr int kFixThreads = 128;          // four warps: one TMEM lane quarter each
constexpr uint32_t FX_A = 0;              // qt tile: 2 K blocks x [128 tok][64 k] fp16 (32 KB)
constexpr uint32_t FX_B = 32768;          // S_g^T: 2 K blocks x [128 v][64 k] fp16 (32 KB)
constexpr int kLdStage = 129;             // after the product: D staged [tok][v] fp32 (66 KB)
constexpr uint32_t FX_BAR = 66560;        // 2 mbarriers
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

// grid (H, d_v / 16).  st_aux: L_g = st_aux[g], M_g = st_aux[G + g] ([H][d][d]
// each).  Writes S_g^T (g >= 1) as fp16 operand blocks to sstart[g][h] and
// S_G to S_final (if not null).
__global__ void __launch_bounds__(kThreads)
segment_scan_kernel(const float* __restrict__ st_aux, int G, int H, __half* __restrict__ sstart,
                    float* __restrict__ S_final)
{
    extern __shared__ __align__(16) float smem[];
    float* sM = smem;                           // M_g [i][k], row stride kLdM
    float* sS = smem + kD * kLdM;               // S_g [k][16]
    const int h = blockIdx.x, j0 = blockIdx.y * kScanCols, tid = threadIdx.x;
    const size_t state = (size_t)kD * kD;
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
        const float* Mg = st_aux + ((size_t)(G + g) * H + h) * state;
        __half* Sg = sstart + ((size_t)g * H + h) * kStateHalfs;
        // S_g^T out (row v = j0 + c, column k), M_g in (the odd row stride
        // keeps both the copy and the column reads below free of conflicts)
        for (int e = tid; e < kD * kScanCols; e += kThreads) {
            const int k = e / kScanCols, c = e % kScanCols;
            Sg[swz_index(j0 + c, k)] = __float2half_rn(sS[e]);
        }
        for (int e = tid; e < kD * kD; e += kThreads) {
            const int r = e / kD, k = e % kD;
            sM[r * kLdM + k] = Mg[e];
        }
        __syncthreads();
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = Lg[(size_t)i * kD + j0 + c0 + c];
#pragma unroll 4
        for (int k = 0; k < kD; ++k) {
            const float m = sM[i * kLdM + k];
            const float4 s0 = *reinterpret_cast<const float4*>(sS + k * kScanCols + c0);
            const float4 s1 = *reinterpret_cast<const float4*>(sS + k * kScanCols + c0 + 4);
            acc[0] = fmaf(m, s0.x, acc[0]);
            acc[1] = fmaf(m, s0.y, acc[1]);
            acc[2] = fmaf(m, s0.z, acc[2]);
            acc[3] = fmaf(m, s0.w, acc[3]);
            acc[4] = fmaf(m, s1.x, acc[4]);
            acc[5] = fmaf(m, s1.y, acc[5]);
            acc[6] = fmaf(m, s1.z, acc[6]);
            acc[7] = fmaf(m, s1.w, acc[7]);
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
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

// grid (tiles of 128 tokens after segment 0, H).  o_loc: [T][H][d] fp16; the
// qt map covers [T][H d] fp16.  A tile never straddles a segment (segments
// are whole tiles).  A wait that gives up sets bit 1 of *timeout_word.
template <typename TO>
__global__ void __launch_bounds__(kFixThreads)
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
    // The product to shared memory, one token row per thread (the operand
    // tiles are no longer read), then o = o_loc + D row by row, each warp
    // covering a row with coalesced 8- or 16-byte accesses.
    float* stage = reinterpret_cast<float*>(sm);
    if (ok) {
        tc_fence_after();
        const int r = warp * 32 + lane;               // this thread's TMEM lane
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            uint32_t d[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + cb * 32, d);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) stage[r * kLdStage + cb * 32 + i] = __uint_as_float(d[i]);
        }
    }
    __syncthreads();
    if (ok) {
        for (int r = warp; r < kTile; r += kFixThreads / 32) {
            const long long t = t0 + r;
            if (t >= T) break;
            const size_t row = ((size_t)t * H + h) * kD + 4 * lane;
            const uint2 lv = *reinterpret_cast<const uint2*>(o_loc + row);
            const float2 l01 = __half22float2(*reinterpret_cast<const __half2*>(&lv.x));
            const float2 l23 = __half22float2(*reinterpret_cast<const __half2*>(&lv.y));
            const float* sr = stage + r * kLdStage + 4 * lane;
            store4(o + row, l01.x + sr[0], l01.y + sr[1], l23.x + sr[2], l23.y + sr[3]);
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
    const int scan_smem = (kD * kLdM + kD * kScanCols) * (int)sizeof(float);
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
