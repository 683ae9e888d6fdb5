// kda_prefill_tc.cu -- chunked KDA prefill on the Blackwell tensor cores
// (tcgen05.mma, TMEM accumulators, TMA-staged tiles), bf16 q/k/v, d_k = d_v =
// 128, chunks of C = 64 tokens, fp32 state carried in tensor memory.
//
// Method.  The recurrence of "[논문 리뷰] Kimi K3 Technical Report"
// (jw9603.github.io) section 3.2, S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T,
// o_t = S_t^T q_t, evaluated in the chunkwise-parallel form of "Kimi 모델 분석"
// (rlaope.github.io) section "순환을 GPU에 올리기": within a chunk the token
// updates are folded into dense products (the WY/UT form, with the triangular
// inverse built from small block products) and only the state passes from one
// chunk to the next; the decay is normalised to the chunk start.
//
// Chunk algebra (entry state S, rows r = tokens of the chunk, G_r = running
// sum of log-decay since the chunk start, per key channel):
//   A_ri = b_r sum_c k_rc k_ic e^{G_rc - G_ic}  (i < r)      P_ri = sum_c q_rc k_ic e^{G_rc - G_ic}  (i <= r)
//   T    = (I + A)^{-1} Diag(b)
//   W    = T (e^{G} .* K)              U = T V - W S
//   O    = (e^{G} .* Q) S + P U        S' = Diag(e^{G_last}) S + (e^{G_last - G} .* K)^T U
// The value-side products are evaluated transposed so that every MMA has
// M = 128 (value columns, or key channels): U^T = V^T T^T - S^T W^T,
// O^T = S^T (e^G Q)^T + U^T P^T, S'^T = S^T Diag(e^{G_last}) + U^T Ktil.
//
// The Gram products need e^{G_r - G_i} split into a row factor and a column
// factor.  A per-channel reference R (the middle of the chunk's range of G)
// keeps both factors below 2^126 when the chunk's decay span is at most 250
// (log2 units); with g >= -5 (the lower bound of section 3.5 of the K3
// review) a 32-token window always satisfies this, and a 64-token chunk whose
// span is larger is processed as two masked passes of 32 rows.  Entries above
// the diagonal may overflow; they are discarded by selection.
//
// Operand precision.  The Gram operands carry the exponent factors (up to
// 2^125) and so need bf16's range; each is stored as a bf16 hi/lo pair and the
// Gram is the sum of three products (hi.hi + lo.hi + hi.lo), which brings the
// factor rounding down to about 2^-16.  Every other operand (T, P, U, S, V, W,
// e^G Q, Ktil) is bounded by O(1) and is fed to the tensor cores as fp16,
// which keeps 3 more mantissa bits than bf16.  Accumulation is fp32
// throughout and the state carry is fp32.  This path therefore also assumes
// |v| and the entries of S stay inside the fp16 range (|x| < 65504).
//
// CTA roles (320 threads, one CTA per (sequence, head)):
//   warp 0      TMA: q, k, g tiles (64 x 128) and the v tile, beta by plain loads
//   warp 1      one thread issues every tcgen05.mma and commit
//   warps 2..9  the compute group (256 threads) runs every CUDA-core phase of a
//               chunk together: gate prep, state decay, Gram readout, the UT
//               solve's diagonal blocks, and every TMEM readout.  The chunk's steps form one
//               dependency chain, so the group moves through it as a whole;
//               the state decay overlaps the Gram product on the tensor cores.
// UT solve.  With D the inverse of the 16 x 16 diagonal blocks of L = I + A
// (forward substitution on CUDA cores) and N = D A_off (A_off = the blocks
// below the diagonal), N is nilpotent of order 4, so
//     (I + A)^{-1} = (I + N)^{-1} D = (I - N)(I + N^2) D,
// and T = (I + A)^{-1} Diag(b) = (I - N)(I + N^2) D'  with D' = D Diag(b).
// The four 64 x 64 products N = D A_off, N^2, Y = D' + N^2 D' and
// T = Y - N Y run on the tensor cores with fp16 operands (the small
// triangular inverse becomes dense products, as the UT transform intends).
// They use tensor memory and shared memory that are idle at that point of
// the chunk; the MMA has M = 128 and only rows 0..63 are read back.
//
// Every wait is bounded in time; a timeout sets a flag in the workspace,
// drains the CTA and frees its tensor memory.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 320;
constexpr int kGroup = 256;            // compute group: warps 2..9
constexpr int kGroupBar = 1;           // its named barrier
constexpr float kLog2e = 1.4426950408889634f;
// Largest decay span (in log2 units) handled in one pass: both Gram factors
// stay below 2^125.
constexpr float kSpanMax = 250.f;

// ---- shared memory map (bytes from a 1024-aligned base) -------------------
constexpr uint32_t OFF_Q = 0;          // q tile  [64 tok][128 ch] bf16, plain rows
constexpr uint32_t OFF_K = 16384;      // k tile  [64][128] bf16
constexpr uint32_t OFF_G = 32768;      // g tile  [64][128] fp32; after the decay scan:
constexpr uint32_t OFF_ADLO = OFF_G;   //   Gram A lo parts [ch][Kr lo | Qr lo] bf16
constexpr uint32_t OFF_V = 65536;      // v tile  2 x [64 tok][64 v], 128B swizzle (bf16 -> fp16)
constexpr uint32_t OFF_AD = 81920;     // Gram A hi parts [ch][Kr | Qr] bf16, 2 x 16 KB
constexpr uint32_t OFF_BD = 114688;    // Gram B hi part  [ch][Kc] bf16
constexpr uint32_t OFF_T = 131072;     // T       [r][i] bf16 (W product)
constexpr uint32_t OFF_WT = 139264;    // -W^T    [ch][r] fp16
constexpr uint32_t OFF_QG = 155648;    // (e^G Q)^T [ch][r] fp16
constexpr uint32_t OFF_P = 172032;     // P       [r][i] fp16
constexpr uint32_t OFF_KT = 180224;    // Ktil^T  [ch][i] fp16
constexpr uint32_t OFF_A32 = 196608;   // A, then X = (I+A)^-1: fp32 [64][68]; before the
constexpr uint32_t OFF_BDLO = OFF_A32; //   Gram readout: Gram B lo part [ch][Kc lo] bf16
constexpr uint32_t OFF_T16 = 214016;   // T       [r][i] fp16 (V product); during gate prep:
constexpr uint32_t OFF_STAT = OFF_T16; //   per row-quarter decay stats, fp32 [3][4][128]
constexpr uint32_t OFF_Y = 222208;     // (spare)
// Solve tiles, all fp16, in regions idle during the solve (the g tile's and
// the Gram B tile's space; the next q/k/g load waits for them):
constexpr uint32_t OFF_DM = OFF_G;            // D  as MN-major A [k][r]
constexpr uint32_t OFF_AO = OFF_G + 8192;     // A_off as MN-major B [k][c]
constexpr uint32_t OFF_NB = OFF_G + 16384;    // N  as MN-major B [m][c]
constexpr uint32_t OFF_DPK = OFF_G + 24576;   // D' as K-major B [c][m] (column c of D')
constexpr uint32_t OFF_YB = OFF_BD;           // Y  as MN-major B [m][c]
// O tile staging for the TMA store, [64 tok][128 v] bf16 plain rows (the A / X
// region, idle from the end of the solve until the next chunk's Gram operands):
constexpr uint32_t OFF_OST = OFF_A32;
constexpr uint32_t OFF_GL = 225280;    // e^{G_last} per channel
constexpr uint32_t OFF_R = 225792;     // 2^R per channel
constexpr uint32_t OFF_BIN = 226304;   // beta of the loaded chunk
constexpr uint32_t OFF_BST = 226560;   // beta of the current pass (masked)
constexpr uint32_t OFF_DESC = 226816;  // 2 step descriptors
constexpr uint32_t OFF_BAR = 226880;   // mbarriers (20 x 8 B)
constexpr uint32_t OFF_MISC = 227040;  // tmem base, flags
constexpr uint32_t kSmemUsed = 227072;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;   // + alignment slack
constexpr int LDA = 68;                // row stride (floats) of A / X: 16-byte aligned rows

enum Bar {
    B_QKG_FULL = 0, B_QKG_EMPTY, B_V_FULL, B_V_EMPTY, B_OPS, B_MMA_G, B_T, B_MMA_W,
    B_CV, B_MMA_C, B_U, B_MMA_OS,
    B_S1, B_R1, B_S2, B_R2, B_S3, B_R3, B_S4, B_R4,   // UT solve rounds
    kNumBars
};

// TMEM columns (512 allocated).  C|O and O|S are adjacent so that one MMA
// can write both of a pair.
constexpr uint32_t TM_G = 0;      // Gram [Kr rows; Qr rows] x [Kc hi | Kc lo]   128 cols
constexpr uint32_t TM_W = 0;      // W^T (unscaled) [ch][r], after the solve      64 cols
constexpr uint32_t TM_SB = 128;   // S^T fp16 A operand                           64 cols
constexpr uint32_t TM_C = 192;    // U^T fp32 [v][r]                              64 cols
constexpr uint32_t TM_O = 256;    // O^T fp32 [v][r]                              64 cols
constexpr uint32_t TM_S = 320;    // S^T fp32 [v][ch]                            128 cols
constexpr uint32_t TM_UB = 448;   // U^T fp16 A operand                           32 cols
constexpr uint32_t kTmemCols = 512;
// During the UT solve (rows 0..63 used), in columns otherwise idle then:
constexpr uint32_t TM_N = 0;      // N = D A_off, fp32
constexpr uint32_t TM_N2A = 64;   // N^2 as fp16 A operand
constexpr uint32_t TM_IA = 96;    // identity rows as fp16 A operand
constexpr uint32_t TM_NA = TM_UB; // N as fp16 A operand
constexpr uint32_t TM_N2 = TM_C;  // N^2, fp32; then Y, then T

struct StepDesc {
    int32_t t0, len, lo, hi, first_pass, last_pass, last_step, chunk;
};

struct Misc {
    uint32_t tmem_base;
    int32_t abort;
    int32_t wide;      // vote: this chunk needs two passes
    int32_t pad;
};

__device__ __forceinline__ void st_chunk(uint8_t* tile, int row, int chunk, uint4 val)
{
    const uint32_t off = (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4);
    *reinterpret_cast<uint4*>(tile + off) = val;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lo_bf16(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ void out_store(float* p, float x) { *p = x; }
__device__ __forceinline__ void out_store(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

struct Ctx {
    uint8_t* sm;
    uint64_t* bar;
    StepDesc* desc;
    Misc* misc;
    int32_t* ws_err;
};

// A bounded wait that records a timeout.
__device__ __forceinline__ bool wait_bar(const Ctx& X, int b, uint32_t phase)
{
    if (mbar_wait(&X.bar[b], phase & 1u)) return true;
    atomicExch(&X.misc->abort, 1);
    atomicOr(X.ws_err, 2);
    return false;
}

// The compute group waits, then agrees on abort at its named barrier (every
// thread passes the barrier, so no thread is left waiting on it).
__device__ __forceinline__ bool group_wait(const Ctx& X, int b, uint32_t phase)
{
    wait_bar(X, b, phase);
    named_bar_sync(kGroupBar, kGroup);
    return *reinterpret_cast<volatile int32_t*>(&X.misc->abort) == 0;
}

__device__ __forceinline__ void group_sync() { named_bar_sync(kGroupBar, kGroup); }

// 16 x 16 unit-lower diagonal block inverse, column j (j < 16) of block b by
// forward substitution; x[r] for r < j is 0 and x[j] is 1.
__device__ __forceinline__ void diag_block_column(const float* sA, int b, int j, float (&x)[16])
{
    const float* L = sA + (b * 16) * LDA + b * 16;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) {
            if (i & 1) a1 = fmaf(L[r * LDA + i], x[i], a1);
            else a0 = fmaf(L[r * LDA + i], x[i], a0);
        }
        x[r] = (r == j) ? 1.f : ((r < j) ? 0.f : -(a0 + a1));
    }
}

// Reads 32 fp32 columns of a TMEM row, converts them to 16 packed fp16 pairs.
__device__ __forceinline__ void tmem_row_f16(uint32_t taddr, uint32_t (&out)[16])
{
    uint32_t d[32];
    tmem_ld32(taddr, d);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i)
        out[i] = pack_f16x2(__uint_as_float(d[2 * i]), __uint_as_float(d[2 * i + 1]));
}

// ------------------------------------------------------------- the kernel
template <typename TO>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_o,
                  const float* __restrict__ beta, const float* S0,
                  const int32_t* __restrict__ cu, int32_t* ws, long long total_tokens, int H,
                  TO* __restrict__ o, float* S_final)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Ctx X;
    X.sm = sm;
    X.bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    X.desc = reinterpret_cast<StepDesc*>(sm + OFF_DESC);
    X.misc = reinterpret_cast<Misc*>(sm + OFF_MISC);
    X.ws_err = ws + kWsTimeoutWord;

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
        for (int ch = 0; ch < nch; ++ch) {
            const long long t0 = bos + (long long)ch * kC;
            int ok = 1;
            if (lane == 0 && ch > 0) ok = wait_bar(X, B_QKG_EMPTY, ch - 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = lane * 2 + j;
                const long long t = t0 + r;
                sBin[r] = (t < eos) ? beta[t * H + h] : 0.f;
            }
            __syncwarp();
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
        if (lane == 0 && nch > 0) {
            const uint32_t id_g = make_idesc_bf16(128, 128, true, true);    // Gram
            const uint32_t id_w = make_idesc_bf16(128, 64, false, false);   // W
            const uint32_t id_cv = make_idesc_f16(128, 64, true, false);    // V^T T^T
            const uint32_t id_mn = make_idesc_f16(128, 64, false, true);    // S^T x MN-major B
            const uint32_t id_k64 = make_idesc_f16(128, 64, false, false);  // U^T P^T
            const uint32_t id_os = make_idesc_f16(128, 192, false, false);  // U^T [P | Ktil]^T
            const uint32_t id_mn128 = make_idesc_f16(128, 128, false, true); // S^T [-W^T | (e^G Q)^T]
            // Base descriptors; a K step advances the start address field
            // (16-byte units) by 128 for MN-major tiles, by 2 for K-major ones.
            const uint64_t dAD = make_sdesc(smem_u32(sm + OFF_AD), 16384, 1024, kSwizzle128B);
            const uint64_t dADLO = make_sdesc(smem_u32(sm + OFF_ADLO), 16384, 1024, kSwizzle128B);
            const uint64_t dBDHL = make_sdesc(smem_u32(sm + OFF_BD), OFF_BDLO - OFF_BD, 1024, kSwizzle128B);
            const uint64_t dADK = make_sdesc(smem_u32(sm + OFF_AD), 16, 1024, kSwizzle128B);
            const uint64_t dT = make_sdesc(smem_u32(sm + OFF_T), 16, 1024, kSwizzle128B);
            const uint64_t dT16 = make_sdesc(smem_u32(sm + OFF_T16), 16, 1024, kSwizzle128B);
            const uint64_t dV = make_sdesc(smem_u32(sm + OFF_V), 8192, 1024, kSwizzle128B);
            const uint64_t dWQ = make_sdesc(smem_u32(sm + OFF_WT), OFF_QG - OFF_WT, 1024, kSwizzle128B);
            const uint64_t dPK = make_sdesc(smem_u32(sm + OFF_P), 16, 1024, kSwizzle128B);
            // D as the A operand of N = D A_off: M = 128 with the second 64-row
            // block pointed at the next tile (finite data; its rows are unused).
            const uint64_t dDM = make_sdesc(smem_u32(sm + OFF_DM), 8192, 1024, kSwizzle128B);
            const uint64_t dAO = make_sdesc(smem_u32(sm + OFF_AO), 8192, 1024, kSwizzle128B);
            const uint64_t dNB = make_sdesc(smem_u32(sm + OFF_NB), 8192, 1024, kSwizzle128B);
            const uint64_t dDPK = make_sdesc(smem_u32(sm + OFF_DPK), 16, 1024, kSwizzle128B);
            const uint64_t dYB = make_sdesc(smem_u32(sm + OFF_YB), 8192, 1024, kSwizzle128B);
            const uint32_t id_r1 = make_idesc_f16(128, 64, true, true);
            const uint32_t id_mn_neg = make_idesc_f16(128, 64, false, true, true);
            for (int step = 0;; ++step) {
                if (!wait_bar(X, B_OPS, step)) break;
                tc_fence_after();
                const StepDesc d = X.desc[step & 1];
                // Gram: [Kr; Qr] (MN-major A) x [Kc hi | Kc lo] (MN-major B, N = 128),
                // K = 128 channels, hi and lo A parts: the readout adds the halves.
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_ss(tmem + TM_G, dAD + 128 * s, dBDHL + 128 * s, id_g, s > 0);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_ss(tmem + TM_G, dADLO + 128 * s, dBDHL + 128 * s, id_g, 1);
                mma_commit(&X.bar[B_MMA_G]);
                // UT solve: N = D A_off ; N^2 = N N ; Y = I D' + N^2 D' ; T = Y - N Y.
                if (!wait_bar(X, B_S1, step)) break;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ss(tmem + TM_N, dDM + 128 * s, dAO + 128 * s, id_r1, s > 0);
                mma_commit(&X.bar[B_R1]);
                if (!wait_bar(X, B_S2, step)) break;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ts(tmem + TM_N2, tmem + TM_NA + 8 * s, dNB + 128 * s, id_mn, s > 0);
                mma_commit(&X.bar[B_R2]);
                if (!wait_bar(X, B_S3, step)) break;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ts(tmem + TM_N2, tmem + TM_IA + 8 * s, dDPK + 2 * s, id_k64, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ts(tmem + TM_N2, tmem + TM_N2A + 8 * s, dDPK + 2 * s, id_k64, 1);
                mma_commit(&X.bar[B_R3]);
                if (!wait_bar(X, B_S4, step)) break;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ts(tmem + TM_N2, tmem + TM_NA + 8 * s, dYB + 128 * s, id_mn_neg, 1);
                mma_commit(&X.bar[B_R4]);
                if (!wait_bar(X, B_T, step)) break;
                tc_fence_after();
                // W^T (unscaled) = Kr^T T^T: A = Kr hi as K-major [ch][tok], B = T [r][i].
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_ss(tmem + TM_W, dADK + 2 * s, dT + 2 * s, id_w, s > 0);
                mma_commit(&X.bar[B_MMA_W]);
                if (!wait_bar(X, B_CV, step)) break;   // -W^T, S^T copy, v tile ready
                tc_fence_after();
                // [U^T | O^T] = S^T [-W^T | (e^G Q)^T] ;  U^T += V^T T^T
                // (the U^T P^T term of O^T follows once U^T is ready)
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_ts(tmem + TM_C, tmem + TM_SB + s * 8, dWQ + 128 * s, id_mn128, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ss(tmem + TM_C, dV + 128 * s, dT16 + 2 * s, id_cv, 1);
                mma_commit(&X.bar[B_MMA_C]);
                if (d.last_pass) mma_commit(&X.bar[B_V_EMPTY]);
                if (!wait_bar(X, B_U, step)) break;
                tc_fence_after();
                // [O^T | S^T] += U^T [P | Ktil^T]^T   (N = 64 + 128)
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ts(tmem + TM_O, tmem + TM_UB + s * 8, dPK + 2 * s, id_os, 1);
                mma_commit(&X.bar[B_MMA_OS]);
                if (d.last_step) break;
            }
        }
    } else {
        // -------------------------------------------------- compute group
        const int ct = tid - 64;                           // 0..255
        const int half = ct >> 7;                          // which half of a TMEM row
        const int L = ((warp & 3) << 5) | lane;            // this thread's TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
        // gate-prep mapping: channels 2cp, 2cp+1; rows 16rq .. 16rq+15
        const int cp = ct & 63, rq = ct >> 6;
        const uint8_t* sQ = sm + OFF_Q;
        const uint8_t* sK = sm + OFF_K;
        const float* sG = reinterpret_cast<const float*>(sm + OFF_G);
        const float* sBin = reinterpret_cast<const float*>(sm + OFF_BIN);
        float* sStat = reinterpret_cast<float*>(sm + OFF_STAT);   // [3][4][128]
        float* sBst = reinterpret_cast<float*>(sm + OFF_BST);
        float* sGl = reinterpret_cast<float*>(sm + OFF_GL);
        float* sR = reinterpret_cast<float*>(sm + OFF_R);
        float* sA = reinterpret_cast<float*>(sm + OFF_A32);

        // S^T <- S0^T (row v of S^T is column v of S0); this thread: 64 channels.
#pragma unroll
        for (int jb = 0; jb < 2; ++jb) {
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = 64 * half + 32 * jb + i;
                r[i] = __float_as_uint(S0 ? S0[sbase + (long long)c * kD + L] : 0.f);
            }
            tmem_st32(tmem + lane_base + TM_S + 64 * half + 32 * jb, r);
        }
        tmem_st_wait();

        int step = 0, chunk_v = 0;
        bool alive = true;
        for (int ch = 0; ch < nch && alive; ++ch) {
            const long long t0 = bos + (long long)ch * kC;
            const int len = (eos - t0 < kC) ? (int)(eos - t0) : kC;
            if (!group_wait(X, B_QKG_FULL, ch)) break;
            // ---- decay scan of this thread's 16 rows x 2 channels (log2 units,
            // relative to the start of its row quarter); kept in registers.
            float2 Gq[16];
            {
                float2 G = make_float2(0.f, 0.f), mx = G, mn = G;
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    const int r = 16 * rq + rr;
                    const float2 g = (r < len) ? *reinterpret_cast<const float2*>(sG + r * kD + 2 * cp)
                                               : make_float2(0.f, 0.f);
                    G.x = fmaf(g.x, kLog2e, G.x);
                    G.y = fmaf(g.y, kLog2e, G.y);
                    Gq[rr] = G;
                    mx.x = fmaxf(mx.x, G.x); mx.y = fmaxf(mx.y, G.y);
                    mn.x = fminf(mn.x, G.x); mn.y = fminf(mn.y, G.y);
                }
                *reinterpret_cast<float2*>(sStat + (0 * 4 + rq) * kD + 2 * cp) = G;
                *reinterpret_cast<float2*>(sStat + (1 * 4 + rq) * kD + 2 * cp) = mx;
                *reinterpret_cast<float2*>(sStat + (2 * 4 + rq) * kD + 2 * cp) = mn;
            }
            group_sync();
            // Per channel: the four per-quarter (total, max, min) triples, read once.
            // They give the span over the whole chunk (the two-pass vote) and, for
            // either pass layout, R, 2^R, 2^{G_last - R}, e^{G_last} and the decay
            // at the start of this thread's row quarter.
            float st[3][4][2];
#pragma unroll
            for (int k = 0; k < 3; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 x = *reinterpret_cast<const float2*>(sStat + (k * 4 + q) * kD + 2 * cp);
                    st[k][q][0] = x.x;
                    st[k][q][1] = x.y;
                }
            auto range = [&](int u, int qa, int qb, float& pmax, float& pmin, float& tot) {
                float off = 0.f;
                pmax = 0.f;
                pmin = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (q < qa || q > qb) continue;
                    pmax = fmaxf(pmax, off + st[1][q][u]);
                    pmin = fminf(pmin, off + st[2][q][u]);
                    off += st[0][q][u];
                }
                tot = off;
            };
            bool wide_me = false;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float a, b, t;
                range(u, 0, 3, a, b, t);
                wide_me = wide_me || (a - b > kSpanMax);
            }
            const int npass = named_bar_red_or(kGroupBar, kGroup, wide_me) ? 2 : 1;
            float R[2][2], pR[2][2], pL[2][2], gl[2][2], base[2][2];
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const int qa = (npass == 1) ? 0 : 2 * p, qb = (npass == 1) ? 3 : 2 * p + 1;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float pmax, pmin, tot;
                    range(u, qa, qb, pmax, pmin, tot);
                    R[p][u] = 0.5f * (pmax + pmin);
                    pR[p][u] = ex2(R[p][u]);
                    pL[p][u] = ex2(tot - R[p][u]);
                    gl[p][u] = ex2(tot);
                    float b = 0.f;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q >= qa && q < rq) b += st[0][q][u];
                    base[p][u] = b;
                }
            }
            for (int p = 0; p < npass; ++p) {
                const int lo = (npass == 1) ? 0 : (p == 0 ? 0 : 32);
                const int hi = (npass == 1) ? len : (p == 0 ? min(32, len) : len);
                // this pass's parameters (selected, so the arrays stay in registers)
                float Rc[2], pRc[2], pLc[2], glc[2], basec[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    Rc[u] = p ? R[1][u] : R[0][u];
                    pRc[u] = p ? pR[1][u] : pR[0][u];
                    pLc[u] = p ? pL[1][u] : pL[0][u];
                    glc[u] = p ? gl[1][u] : gl[0][u];
                    basec[u] = p ? base[1][u] : base[0][u];
                }
                if (rq == 0) {
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        sGl[2 * cp + u] = glc[u];
                        sR[2 * cp + u] = pRc[u];
                    }
                }
                if (ct < kC) sBst[ct] = (ct >= lo && ct < hi) ? sBin[ct] : 0.f;
                if (ct == 0) {
                    StepDesc d;
                    d.t0 = (int32_t)t0;
                    d.len = len;
                    d.lo = lo;
                    d.hi = hi;
                    d.first_pass = (p == 0);
                    d.last_pass = (p == npass - 1);
                    d.last_step = (ch == nch - 1) && (p == npass - 1);
                    d.chunk = ch;
                    X.desc[step & 1] = d;
                }
                // The previous chunk's O store has read its staging area (the
                // Gram B lo part goes there), and everyone has read the decay
                // stats before the lo parts overwrite the g tile.
                if (ct == 0) bulk_wait_group_read0();
                group_sync();
                // ---- Gram operands (bf16 hi/lo), e^G Q and Ktil (fp16); this
                // thread writes 2 channels x 2 chunks of 8 rows of each.
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    uint32_t kp[8], qp[8];             // bf16 pairs (channels 2cp, 2cp+1)
#pragma unroll
                    for (int w8 = 0; w8 < 8; ++w8) {
                        const int r = 16 * rq + 8 * jj + w8;
                        kp[w8] = *reinterpret_cast<const uint32_t*>(sK + r * 256 + 4 * cp);
                        qp[w8] = *reinterpret_cast<const uint32_t*>(sQ + r * 256 + 4 * cp);
                    }
                    const int chunk = 2 * rq + jj;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        uint32_t krh[4], krl[4], qrh[4], qrl[4], kch[4], kcl[4], gq[4], kt[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float vk[2], vq[2], vc[2];
#pragma unroll
                            for (int w = 0; w < 2; ++w) {
                                const int w8 = 2 * e + w, rr = 8 * jj + w8, r = 16 * rq + rr;
                                const bool act = (r >= lo && r < hi);
                                const float kk = u ? hi_bf16(kp[w8]) : lo_bf16(kp[w8]);
                                const float qq = u ? hi_bf16(qp[w8]) : lo_bf16(qp[w8]);
                                const float gv = u ? Gq[rr].y : Gq[rr].x;
                                const float x = basec[u] + gv - Rc[u];
                                const float e1 = act ? ex2(x) : 0.f;
                                const float e2 = act ? ex2(-x) : 0.f;
                                vk[w] = kk * e1;
                                vq[w] = qq * e1;
                                vc[w] = kk * e2;
                            }
                            krh[e] = pack_bf16x2(vk[0], vk[1]);
                            qrh[e] = pack_bf16x2(vq[0], vq[1]);
                            kch[e] = pack_bf16x2(vc[0], vc[1]);
                            krl[e] = pack_bf16x2(vk[0] - lo_bf16(krh[e]), vk[1] - hi_bf16(krh[e]));
                            qrl[e] = pack_bf16x2(vq[0] - lo_bf16(qrh[e]), vq[1] - hi_bf16(qrh[e]));
                            kcl[e] = pack_bf16x2(vc[0] - lo_bf16(kch[e]), vc[1] - hi_bf16(kch[e]));
                            gq[e] = pack_f16x2(vq[0] * pRc[u], vq[1] * pRc[u]);
                            kt[e] = pack_f16x2(vc[0] * pLc[u], vc[1] * pLc[u]);
                        }
                        const int c = 2 * cp + u;
                        st_chunk(sm + OFF_AD, c, chunk, make_uint4(krh[0], krh[1], krh[2], krh[3]));
                        st_chunk(sm + OFF_AD + 16384, c, chunk, make_uint4(qrh[0], qrh[1], qrh[2], qrh[3]));
                        st_chunk(sm + OFF_ADLO, c, chunk, make_uint4(krl[0], krl[1], krl[2], krl[3]));
                        st_chunk(sm + OFF_ADLO + 16384, c, chunk, make_uint4(qrl[0], qrl[1], qrl[2], qrl[3]));
                        st_chunk(sm + OFF_BD, c, chunk, make_uint4(kch[0], kch[1], kch[2], kch[3]));
                        st_chunk(sm + OFF_BDLO, c, chunk, make_uint4(kcl[0], kcl[1], kcl[2], kcl[3]));
                        st_chunk(sm + OFF_QG, c, chunk, make_uint4(gq[0], gq[1], gq[2], gq[3]));
                        st_chunk(sm + OFF_KT, c, chunk, make_uint4(kt[0], kt[1], kt[2], kt[3]));
                    }
                }
                fence_proxy_async_smem();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_OPS]);

                // ---- while the Gram runs: the v tile to fp16 (first pass of a
                // chunk) and the state decay with its fp16 copy.
                const StepDesc d = X.desc[step & 1];
                if (d.first_pass) {
                    if (!group_wait(X, B_V_FULL, chunk_v)) { alive = false; break; }
                    uint4* vt = reinterpret_cast<uint4*>(sm + OFF_V);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint4 x = vt[ct + 256 * u];
                        x.x = bf16x2_to_f16x2(x.x);
                        x.y = bf16x2_to_f16x2(x.y);
                        x.z = bf16x2_to_f16x2(x.z);
                        x.w = bf16x2_to_f16x2(x.w);
                        vt[ct + 256 * u] = x;
                    }
                }
                if (d.last_pass) ++chunk_v;
                tc_fence_after();
#pragma unroll
                for (int jb = 0; jb < 2; ++jb) {
                    const int c0 = 64 * half + 32 * jb;
                    uint32_t r[32], b[16];
                    tmem_ld32(tmem + lane_base + TM_S + c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        b[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    tmem_st16(tmem + lane_base + TM_SB + (c0 >> 1), b);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        r[i] = __float_as_uint(__uint_as_float(r[i]) * sGl[c0 + i]);
                    tmem_st32(tmem + lane_base + TM_S + c0, r);
                }
                tmem_st_wait();
                fence_proxy_async_smem();                  // the converted v tile
                tc_fence_before();

                // ---- Gram readout: rows 0..63 -> A (times beta, strictly lower,
                // fp32), rows 64..127 -> P (lower including the diagonal, fp16).
                if (!group_wait(X, B_MMA_G, step)) { alive = false; break; }
                tc_fence_after();
                {
                    uint32_t dg[32], dl[32];
                    tmem_ld32(tmem + lane_base + TM_G + 32 * half, dg);
                    tmem_ld32(tmem + lane_base + TM_G + 64 + 32 * half, dl);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        dg[i] = __float_as_uint(__uint_as_float(dg[i]) + __uint_as_float(dl[i]));
                    if (L < kC) {
                        const int r = L;
                        const bool act_r = (r >= lo && r < hi);
                        const float b = sBst[r];
#pragma unroll
                        for (int i4 = 0; i4 < 8; ++i4) {
                            float v4[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int i = 32 * half + 4 * i4 + u;
                                const bool keep = act_r && i < r && i >= lo;
                                v4[u] = keep ? b * __uint_as_float(dg[4 * i4 + u]) : 0.f;
                            }
                            *reinterpret_cast<float4*>(sA + r * LDA + 32 * half + 4 * i4) =
                                make_float4(v4[0], v4[1], v4[2], v4[3]);
                        }
                    } else {
                        const int r = L - kC;
                        const bool act_r = (r >= lo && r < hi);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t pk[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float pv[2];
#pragma unroll
                                for (int u = 0; u < 2; ++u) {
                                    const int i = 32 * half + 8 * j + 2 * e + u;
                                    const bool keep = act_r && i <= r && i >= lo;
                                    pv[u] = keep ? __uint_as_float(dg[8 * j + 2 * e + u]) : 0.f;
                                }
                                pk[e] = pack_f16x2(pv[0], pv[1]);
                            }
                            st_chunk(sm + OFF_P, r, 4 * half + j, make_uint4(pk[0], pk[1], pk[2], pk[3]));
                        }
                    }
                }
                tc_fence_before();
                group_sync();
                // ---- UT solve, S1: diagonal-block inverses D (warps of ct < 128),
                // A_off as fp16 and identity rows in TMEM (the other warps).
                if (ct < 128) {
                    const int b = ct >> 5, j = ct & 31;
                    float x[16];
                    diag_block_column(sA, b, j, x);
                    if (j < 16) {
                        const int k = 16 * b + j;        // column k of D = row k of the tiles
                        const float bk = sBst[k];
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) {
                            uint32_t pd[4], pp[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float dv[2];
#pragma unroll
                                for (int u = 0; u < 2; ++u) {
                                    const int r = 8 * c8 + 2 * e + u;
                                    dv[u] = ((r >> 4) == b) ? x[r & 15] : 0.f;
                                }
                                pd[e] = pack_f16x2(dv[0], dv[1]);
                                pp[e] = pack_f16x2(dv[0] * bk, dv[1] * bk);
                            }
                            st_chunk(sm + OFF_DM, k, c8, make_uint4(pd[0], pd[1], pd[2], pd[3]));
                            st_chunk(sm + OFF_DPK, k, c8, make_uint4(pp[0], pp[1], pp[2], pp[3]));
                        }
                    }
                } else {
                    const int k = (ct - 128) >> 1, hh = ct & 1;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c0 = 32 * hh + 8 * j + 2 * e;
                            const float a0 = ((c0 >> 4) < (k >> 4)) ? sA[k * LDA + c0] : 0.f;
                            const float a1 = (((c0 + 1) >> 4) < (k >> 4)) ? sA[k * LDA + c0 + 1] : 0.f;
                            pk[e] = pack_f16x2(a0, a1);
                        }
                        st_chunk(sm + OFF_AO, k, 4 * hh + j, make_uint4(pk[0], pk[1], pk[2], pk[3]));
                    }
                    if ((warp & 3) < 2) {                // lanes 0..63: identity rows
                        uint32_t id[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            id[i] = ((2 * i == L) ? 0x3C00u : 0u) | ((2 * i + 1 == L) ? 0x3C000000u : 0u);
                        tmem_st32(tmem + lane_base + TM_IA, id);
                        tmem_st_wait();
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_S1]);
                const bool top = (warp & 3) < 2;         // this warp holds rows 0..63
                // S2: N -> fp16 A operand (TMEM) and MN-major B tile
                if (!group_wait(X, B_R1, step)) { alive = false; break; }
                tc_fence_after();
                if (top) {
                    uint32_t nb[16];
                    tmem_row_f16(tmem + lane_base + TM_N + 32 * half, nb);
                    tmem_st16(tmem + lane_base + TM_NA + 16 * half, nb);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        st_chunk(sm + OFF_NB, L, 4 * half + j,
                                 make_uint4(nb[4 * j], nb[4 * j + 1], nb[4 * j + 2], nb[4 * j + 3]));
                    tmem_st_wait();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_S2]);
                // S3: N^2 -> fp16 A operand
                if (!group_wait(X, B_R2, step)) { alive = false; break; }
                tc_fence_after();
                if (top) {
                    uint32_t nb[16];
                    tmem_row_f16(tmem + lane_base + TM_N2 + 32 * half, nb);
                    tmem_st16(tmem + lane_base + TM_N2A + 16 * half, nb);
                    tmem_st_wait();
                }
                tc_fence_before();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_S3]);
                // S4: Y -> fp16 MN-major B tile (Y stays in TMEM as the accumulator)
                if (!group_wait(X, B_R3, step)) { alive = false; break; }
                // The g tile's space is no longer read: the next chunk may load.
                if (ct == 0 && d.last_pass) mbar_arrive(&X.bar[B_QKG_EMPTY]);
                tc_fence_after();
                if (top) {
                    uint32_t yb[16];
                    tmem_row_f16(tmem + lane_base + TM_N2 + 32 * half, yb);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        st_chunk(sm + OFF_YB, L, 4 * half + j,
                                 make_uint4(yb[4 * j], yb[4 * j + 1], yb[4 * j + 2], yb[4 * j + 3]));
                }
                fence_proxy_async_smem();
                tc_fence_before();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_S4]);
                // S5: T -> bf16 (W product) and fp16 (V product) rows
                if (!group_wait(X, B_R4, step)) { alive = false; break; }
                tc_fence_after();
                if (top) {
                    uint32_t d[32];
                    tmem_ld32(tmem + lane_base + TM_N2 + 32 * half, d);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t pb[4], ph[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float t0v = __uint_as_float(d[8 * j + 2 * e]);
                            const float t1v = __uint_as_float(d[8 * j + 2 * e + 1]);
                            pb[e] = pack_bf16x2(t0v, t1v);
                            ph[e] = pack_f16x2(t0v, t1v);
                        }
                        st_chunk(sm + OFF_T, L, 4 * half + j, make_uint4(pb[0], pb[1], pb[2], pb[3]));
                        st_chunk(sm + OFF_T16, L, 4 * half + j, make_uint4(ph[0], ph[1], ph[2], ph[3]));
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_T]);

                // ---- W readout: -W^T row c = -2^R_c x (Kr^T T^T) row c, fp16
                if (!group_wait(X, B_MMA_W, step)) { alive = false; break; }
                tc_fence_after();
                {
                    uint32_t dw[32];
                    tmem_ld32(tmem + lane_base + TM_W + 32 * half, dw);
                    tmem_ld_wait();
                    const float sc = -sR[L];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            pk[e] = pack_f16x2(sc * __uint_as_float(dw[8 * j + 2 * e]),
                                               sc * __uint_as_float(dw[8 * j + 2 * e + 1]));
                        st_chunk(sm + OFF_WT, L, 4 * half + j, make_uint4(pk[0], pk[1], pk[2], pk[3]));
                    }
                }
                tc_fence_before();
                fence_proxy_async_smem();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_CV]);

                // ---- U^T -> fp16 A operand
                if (!group_wait(X, B_MMA_C, step)) { alive = false; break; }
                tc_fence_after();
                {
                    uint32_t du[32], b[16];
                    tmem_ld32(tmem + lane_base + TM_C + 32 * half, du);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        b[i] = pack_f16x2(__uint_as_float(du[2 * i]), __uint_as_float(du[2 * i + 1]));
                    tmem_st16(tmem + lane_base + TM_UB + 16 * half, b);
                    tmem_st_wait();
                }
                tc_fence_before();
                group_sync();
                if (ct == 0) mbar_arrive(&X.bar[B_U]);

                // ---- O^T readout.  A full single-pass chunk with bf16 output is
                // staged in shared memory (the A/X region, idle until the next
                // chunk's Gram operands) and written by one TMA tensor store; other
                // chunks (a ragged tail, the two passes of a wide chunk, fp32
                // output) are stored by the threads.
                if (!group_wait(X, B_MMA_OS, step)) { alive = false; break; }
                tc_fence_after();
                {
                    uint32_t dd[32];
                    tmem_ld32(tmem + lane_base + TM_O + 32 * half, dd);
                    tmem_ld_wait();
                    const bool tma_out = (sizeof(TO) == 2) && d.lo == 0 && d.hi == kC;
                    if (tma_out) {
                        uint8_t* stg = sm + OFF_OST;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int r = 32 * half + i;
                            *reinterpret_cast<__nv_bfloat16*>(stg + r * 256 + 2 * L) =
                                __float2bfloat16_rn(__uint_as_float(dd[i]));
                        }
                        fence_proxy_async_smem();
                        tc_fence_before();
                        group_sync();
                        if (ct == 0) {
                            tma_store_2d(&tm_o, h * kD, d.t0, stg);
                            bulk_commit_group();
                        }
                    } else {
                        TO* op = o + ((long long)d.t0 * H + h) * kD + L;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int r = 32 * half + i;
                            if (r >= d.lo && r < d.hi)
                                out_store(op + (long long)r * H * kD, __uint_as_float(dd[i]));
                        }
                        tc_fence_before();
                    }
                }
                ++step;
            }
        }
        if (ct == 0) bulk_wait_group0();                   // the last O store has landed
        if (S_final && !*reinterpret_cast<volatile int32_t*>(&X.misc->abort)) {
            tc_fence_after();
#pragma unroll
            for (int jb = 0; jb < 2; ++jb) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + TM_S + 64 * half + 32 * jb, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    S_final[sbase + (long long)(64 * half + 32 * jb + i) * kD + L] = __uint_as_float(r[i]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
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

bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int H,
              long long T, int box_x, CUtensorMapSwizzle swz)
{
    auto fn = encode_fn();
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

template <typename TO>
cudaError_t launch_typed(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* S0, const int32_t* cu, int32_t N,
                         int64_t T, int32_t H, void* o, float* S_final, int32_t* ws,
                         cudaStream_t stream)
{
    CUtensorMap mq, mk, mg, mv, mo;
    // The output map is used for bf16 output only (fp32 output is stored by
    // the threads); for fp32 a copy of the q map fills the slot.
    const bool bf16_out = sizeof(TO) == 2;
    if (!make_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        (bf16_out && !make_map(&mo, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD,
                               CU_TENSOR_MAP_SWIZZLE_NONE)) ||
        !make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, T, kD, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    auto kern = prefill_tc_kernel<TO>;
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
                                                            static_cast<TO*>(o), S_final);
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
           encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const void* q, const void* k, const void* v,
                              const float* log_alpha, const float* beta, const float* S0,
                              const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                              int32_t H, kda_dtype_t dtype, void* o, float* S_final,
                              int32_t* ws, cudaStream_t stream)
{
    if (dtype == KDA_BF16_F32OUT)
        return launch_typed<float>(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs,
                                   total_tokens, H, o, S_final, ws, stream);
    return launch_typed<__nv_bfloat16>(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs,
                                       total_tokens, H, o, S_final, ws, stream);
}

}  // namespace kda
