// kda_tc_chunk.cuh -- the phases of one chunk step of the tensor-core prefill
// (bf16 q/k/v, d_k = d_v = 128, chunks of C = 64 tokens), shared by the
// single-CTA kernel (kda_prefill_tc.cu) and the producer / consumer kernel
// (kda_prefill_split.cu).
//
// Chunk algebra (entry state S, rows r = tokens of the chunk, G_r = running
// sum of log-decay since the chunk start, per key channel), the chunkwise form
// of "Kimi 모델 분석" (rlaope.github.io), section "순환을 GPU에 올리기", applied
// to the recurrence of "[논문 리뷰] Kimi K3 Technical Report" section 3.2:
//   A_ri = b_r sum_c k_rc k_ic e^{G_rc - G_ic}  (i < r)      P_ri = sum_c q_rc k_ic e^{G_rc - G_ic}  (i <= r)
//   T    = (I + A)^{-1} Diag(b)
//   W    = T (e^{G} .* K)              U = T V - W S
//   O    = (e^{G} .* Q) S + P U        S' = Diag(e^{G_last}) S + (e^{G_last - G} .* K)^T U
// The value-side products are evaluated transposed so that every MMA has
// M = 128: U^T = V^T T^T - S^T W^T, O^T = S^T (e^G Q)^T + U^T P^T,
// S'^T = S^T Diag(e^{G_last}) + U^T Ktil.
//
// Everything up to W (gate prep, the Gram products, the UT solve, W) does not
// involve the state: these are the "front" phases.  The "back" phases (state
// decay, U, O, the state update) form the chain that carries S from chunk to
// chunk.  The single-CTA kernel runs both on one CTA; the split kernel runs
// the front phases on producer CTAs that hand T, -W^T, (e^G Q)^T, P, Ktil^T
// and e^{G_last} to the CTA that owns the state.
//
// Gram factorisation.  e^{G_r - G_i} is split into a row factor and a column
// factor around a per-channel reference R (the middle of the chunk's range of
// G, log2 units); both stay below 2^125 when the chunk's decay span is at most
// 250.  With g >= -5 (section 3.5 of the K3 review) a 32-token window always
// satisfies this, and a 64-token chunk with a larger span is processed as two
// masked passes of 32 rows (two steps).  Entries above the diagonal may
// overflow; they are discarded by selection.
//
// Operand precision.  The Gram operands carry the exponent factors and need
// bf16's range: each is a bf16 hi/lo pair and the Gram sums hi.hi, lo.hi and
// hi.lo, bringing the factor rounding to about 2^-16.  T, P, U, S, V, W, e^G Q
// and Ktil are O(1) and enter the tensor cores as fp16 (3 more mantissa bits
// than bf16).  Accumulation and the state carry are fp32.  |v| and the state
// entries are assumed to stay inside the fp16 range (|x| < 65504).
//
// UT solve.  With D the inverse of the 16 x 16 diagonal blocks of L = I + A
// and N = D A_off (A_off = the blocks below the diagonal), N is nilpotent of
// order 4, so
//     (I + A)^{-1} = (I + N)^{-1} D = (I + N^2)(I - N) D,
// and T = (I + N^2) Z with Z = (I - N) D', D' = D Diag(b).  D (forward
// substitution) and N (six 16 x 16 block products) are formed on CUDA cores;
// N^2 and Z are one round of tensor-core products, T = (I + N^2) Z a second
// (fp16 operands, in tensor memory and shared memory idle at that point of
// the chunk).
#pragma once

#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace tc {

using namespace sm100;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kGroup = 256;            // compute group: 8 warps
constexpr int kGroupBar = 1;           // its named barrier
constexpr float kLog2e = 1.4426950408889634f;
// Largest decay span (log2 units) handled in one pass.
constexpr float kSpanMax = 250.f;

// ---- shared memory map of the front phases (bytes from a 1024-aligned base)
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
constexpr uint32_t OFF_Y = 222208;     // 3 KB: the first 1 KB not used by the phases, then
constexpr uint32_t OFF_NRM = OFF_Y + 1024;    // gate prologue: q_scale/||q_r|| [64], 1/||k_r|| [64]
constexpr uint32_t OFF_AH = OFF_Y + 1536;     // gate prologue: the head's A row [128] (split producer)
// Solve tiles, in regions idle during the solve (the g tile's and the Gram
// B tile's space; the next q/k/g load waits for the first three):
constexpr uint32_t OFF_DF = OFF_G;            // D blocks, fp32 [4][16][17] (padded rows)
constexpr uint32_t OFF_IMN = OFF_G + 8192;    // I - N as K-major fp16 A [r][k]
constexpr uint32_t OFF_NB = OFF_G + 16384;    // N  as MN-major fp16 B [m][c] = K-major A [r][k]
constexpr uint32_t OFF_DPK = OFF_G + 24576;   // D' as K-major fp16 B [c][m] (column c of D')
constexpr uint32_t OFF_ZB = OFF_BD;           // Z  as MN-major fp16 B [m][c]
constexpr uint32_t OFF_OST = OFF_A32;  // O tile staging of the single-CTA kernel
constexpr uint32_t OFF_GL = 225280;    // e^{G_last} per channel
constexpr uint32_t OFF_R = 225792;     // 2^R per channel
constexpr uint32_t OFF_BIN = 226304;   // beta of the loaded chunk
constexpr uint32_t OFF_BST = 226560;   // beta of the current pass (masked)
constexpr uint32_t OFF_DESC = 226816;  // 2 step descriptors
constexpr uint32_t OFF_BAR = 226880;   // mbarriers (kNumBars x 8 B)
constexpr uint32_t OFF_MISC = 227152;  // tmem base, flags
constexpr uint32_t kSmemUsed = 227168;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;   // + alignment slack
constexpr int LDA = 68;                // row stride (floats) of A / X: 16-byte aligned rows

// Byte offsets of the back-phase operands inside one step's block (the same
// block layout is used in shared memory and in the split kernel's ring):
// -W^T, (e^G Q)^T, P, Ktil^T, T (fp16) and e^{G_last}.
constexpr uint32_t BLK_WT = 0;
constexpr uint32_t BLK_QG = 16384;
constexpr uint32_t BLK_P = 32768;
constexpr uint32_t BLK_KT = 40960;
constexpr uint32_t BLK_T16 = 57344;
constexpr uint32_t BLK_GL = 65536;
constexpr uint32_t kBlkBytes = 66048;

enum Bar {
    B_QKG_FULL = 0, B_QKG_EMPTY, B_V_FULL, B_V_EMPTY, B_OPS, B_MMA_G, B_T, B_MMA_W,
    B_CV, B_MMA_C, B_U, B_MMA_OS,
    B_S1, B_R1, B_S2, B_R2,                            // UT solve rounds
    B_JOB_DONE,                                        // split producer: operands written
    B_SV_FULL0, B_SV_FULL1, B_SV_FULL2, B_SV_FULL3,    // split consumer: v tile buffers
    B_SV_EMPTY0, B_SV_EMPTY1, B_SV_EMPTY2, B_SV_EMPTY3,
    B_ST_FULL0, B_ST_FULL1, B_ST_EMPTY0, B_ST_EMPTY1,  // split consumer: operand stages
    kNumBars
};
static_assert(OFF_BAR + kNumBars * 8 <= OFF_MISC, "barrier area overflows");

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
constexpr uint32_t TM_Z = 0;      // Z = (I - N) D', fp32                         64 cols
constexpr uint32_t TM_N2 = 64;    // N^2, fp32                                    64 cols
constexpr uint32_t TM_T = TM_C;   // T = (I + N^2) Z, fp32                        64 cols
constexpr uint32_t TM_IPN = TM_UB;  // I + N^2 as fp16 A operand                  32 cols

struct StepDesc {
    int32_t t0, len, lo, hi, first_pass, last_pass, last_step, chunk;
};

struct Misc {
    uint32_t tmem_base;
    int32_t abort;
    int32_t wide;      // vote: this chunk needs two passes
    int32_t pad;
};

// 16-byte chunk `chunk` (8 fp16 / bf16 values) of row `row` of a tile stored
// in the 128-byte swizzled K-major / MN-major layout of the MMA descriptors.
// `tile` may point to shared or global memory.
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
    int32_t* ws_err;     // the caller-visible timeout word (bit 1 set on a timeout)
    int32_t* ws_abort;   // split kernel: the abort word its CTAs watch (else null)
};

// A bounded wait that records a timeout.
__device__ __forceinline__ bool wait_bar(const Ctx& X, int b, uint32_t phase)
{
    if (mbar_wait(&X.bar[b], phase & 1u)) return true;
    atomicExch(&X.misc->abort, 1);
    atomicOr(X.ws_err, 2);
    if (X.ws_abort) atomicExch(X.ws_abort, 1);
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

// The MMA warp runs its loop with all 32 lanes (the issue helpers elect one
// lane).  Every lane waits on the barrier itself and the lanes then agree on
// the outcome, so the warp never diverges: a warp whose lane 0 polls while
// the other lanes wait for it at a warp-synchronous instruction was measured
// to slow the whole kernel down by half.
__device__ __forceinline__ bool warp_wait(const Ctx& X, int b, uint32_t phase)
{
    const bool ok = wait_bar(X, b, phase);
    return __all_sync(0xffffffffu, ok) != 0;
}

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

// Per-thread coordinates inside the compute group (ct = 0..255 in the group).
struct Lane {
    int ct;            // thread index in the group
    int half;          // which half of a TMEM row this thread reads
    int L;             // this thread's TMEM lane
    uint32_t lane_base;
    int cp, rq;        // gate prep: channels 2cp, 2cp+1; rows 16rq .. 16rq+15
};

__device__ __forceinline__ Lane make_lane(int ct, int warp, int lane)
{
    Lane t;
    t.ct = ct;
    t.half = ct >> 7;
    t.L = ((warp & 3) << 5) | lane;
    t.lane_base = (uint32_t)((warp & 3) << 5) << 16;
    t.cp = ct & 63;
    t.rq = ct >> 6;
    return t;
}

// The two pass layouts' factors for this thread's two channels.
struct PassParams {
    float R[2][2], pR[2][2], pL[2][2], gl[2][2], base[2][2];
};

// One pass's factors, selected (not indexed) so that the arrays stay in
// registers.
struct Pass {
    int lo, hi;
    float Rc[2], pRc[2], pLc[2], glc[2], basec[2];
};

// ---------------------------------------------------------------------------
// Front phase 0 (gate prologue only): the inverse L2 norms of the chunk's q
// and k rows, from the bf16 tiles in shared memory, to OFF_NRM.  Thread ct
// sums 32 channels of row ct / 4 (16-byte loads rotated by the row, so that a
// warp's loads hit distinct banks); four threads combine.  Ends with a group
// barrier.
__device__ __forceinline__ void qk_norms(const Ctx& X, const Lane& t, float q_scale)
{
    const int r = t.ct >> 2, qq = t.ct & 3;
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int jj = (j + r) & 3;
        const uint32_t off = r * 256 + 64 * qq + 16 * jj;
        const uint4 a = *reinterpret_cast<const uint4*>(X.sm + OFF_Q + off);
        const uint4 b = *reinterpret_cast<const uint4*>(X.sm + OFF_K + off);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float q0 = lo_bf16(av[e]), q1 = hi_bf16(av[e]);
            const float k0 = lo_bf16(bv[e]), k1 = hi_bf16(bv[e]);
            sq = fmaf(q0, q0, fmaf(q1, q1, sq));
            sk = fmaf(k0, k0, fmaf(k1, k1, sk));
        }
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
    }
    float* nrm = reinterpret_cast<float*>(X.sm + OFF_NRM);
    if (qq == 0) {
        nrm[r] = q_scale * inv_norm(sq);
        nrm[64 + r] = inv_norm(sk);
    }
    group_sync();
}

// ---------------------------------------------------------------------------
// Front phase 1: decay scan of this thread's 16 rows x 2 channels of the g
// tile sG ([64][128] fp32; log2 units, relative to the start of its row
// quarter, kept in Gq), the two-pass vote and both pass layouts' factors.
// With the gate prologue (FUSED) the tile holds z and g = -5 sigmoid(e^A z),
// Ah = the head's A row (d_k values).  Returns the number of passes (1, 2).
template <bool FUSED>
__device__ __forceinline__ int gate_prep(const Ctx& X, const Lane& t, int len, const float* sG,
                                         const float* Ah, float2 (&Gq)[16], PassParams& pp)
{
    const int cp = t.cp, rq = t.rq;
    const float2 eA = FUSED ? make_float2(expf(Ah[2 * cp]), expf(Ah[2 * cp + 1]))
                            : make_float2(0.f, 0.f);
    float* sStat = reinterpret_cast<float*>(X.sm + OFF_STAT);   // [3][4][128]
    {
        float2 G = make_float2(0.f, 0.f), mx = G, mn = G;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            const int r = 16 * rq + rr;
            float2 g = (r < len) ? *reinterpret_cast<const float2*>(sG + r * kD + 2 * cp)
                                 : make_float2(0.f, 0.f);
            if (FUSED && r < len) {
                g.x = gate_from_z(g.x, eA.x);
                g.y = gate_from_z(g.y, eA.y);
            }
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
        float a, b, tt;
        range(u, 0, 3, a, b, tt);
        wide_me = wide_me || (a - b > kSpanMax);
    }
    const int npass = named_bar_red_or(kGroupBar, kGroup, wide_me) ? 2 : 1;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int qa = (npass == 1) ? 0 : 2 * p, qb = (npass == 1) ? 3 : 2 * p + 1;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float pmax, pmin, tot;
            range(u, qa, qb, pmax, pmin, tot);
            pp.R[p][u] = 0.5f * (pmax + pmin);
            pp.pR[p][u] = ex2(pp.R[p][u]);
            pp.pL[p][u] = ex2(tot - pp.R[p][u]);
            pp.gl[p][u] = ex2(tot);
            float b = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (q >= qa && q < rq) b += st[0][q][u];
            pp.base[p][u] = b;
        }
    }
    return npass;
}

__device__ __forceinline__ Pass select_pass(const PassParams& pp, int p, int npass, int len)
{
    Pass s;
    s.lo = (npass == 1) ? 0 : (p == 0 ? 0 : 32);
    s.hi = (npass == 1) ? len : (p == 0 ? min(32, len) : len);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        s.Rc[u] = p ? pp.R[1][u] : pp.R[0][u];
        s.pRc[u] = p ? pp.pR[1][u] : pp.pR[0][u];
        s.pLc[u] = p ? pp.pL[1][u] : pp.pL[0][u];
        s.glc[u] = p ? pp.gl[1][u] : pp.gl[0][u];
        s.basec[u] = p ? pp.base[1][u] : pp.base[0][u];
    }
    return s;
}

// Front phase 2: this pass's per-channel factors (e^{G_last} to gl_dst, 2^R)
// and the masked beta.  No barrier.
__device__ __forceinline__ void pass_factors(const Ctx& X, const Lane& t, const Pass& ps,
                                             float* gl_dst)
{
    const float* sBin = reinterpret_cast<const float*>(X.sm + OFF_BIN);
    float* sBst = reinterpret_cast<float*>(X.sm + OFF_BST);
    float* sR = reinterpret_cast<float*>(X.sm + OFF_R);
    if (t.rq == 0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            gl_dst[2 * t.cp + u] = ps.glc[u];
            sR[2 * t.cp + u] = ps.pRc[u];
        }
    }
    if (t.ct < kC) sBst[t.ct] = (t.ct >= ps.lo && t.ct < ps.hi) ? sBin[t.ct] : 0.f;
}

// Front phase 3: the Gram operands (bf16 hi/lo) in shared memory, and
// (e^G Q)^T and Ktil^T (fp16) to qg_dst / kt_dst; this thread writes
// 2 channels x 2 chunks of 8 rows of each.  With the gate prologue (FUSED)
// q and k are scaled by their rows' inverse norms (OFF_NRM).  No barrier.
template <bool FUSED>
__device__ __forceinline__ void gram_operands(const Ctx& X, const Lane& t, const Pass& ps,
                                              const float2 (&Gq)[16], uint8_t* qg_dst,
                                              uint8_t* kt_dst)
{
    const float* nrm = reinterpret_cast<const float*>(X.sm + OFF_NRM);
    const int cp = t.cp, rq = t.rq, lo = ps.lo, hi = ps.hi;
    const uint8_t* sQ = X.sm + OFF_Q;
    const uint8_t* sK = X.sm + OFF_K;
    uint8_t* sm = X.sm;
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
                    float kk = u ? hi_bf16(kp[w8]) : lo_bf16(kp[w8]);
                    float qq = u ? hi_bf16(qp[w8]) : lo_bf16(qp[w8]);
                    if (FUSED) {
                        kk *= nrm[64 + r];
                        qq *= nrm[r];
                    }
                    const float gv = u ? Gq[rr].y : Gq[rr].x;
                    const float x = ps.basec[u] + gv - ps.Rc[u];
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
                gq[e] = pack_f16x2(vq[0] * ps.pRc[u], vq[1] * ps.pRc[u]);
                kt[e] = pack_f16x2(vc[0] * ps.pLc[u], vc[1] * ps.pLc[u]);
            }
            const int c = 2 * cp + u;
            st_chunk(sm + OFF_AD, c, chunk, make_uint4(krh[0], krh[1], krh[2], krh[3]));
            st_chunk(sm + OFF_AD + 16384, c, chunk, make_uint4(qrh[0], qrh[1], qrh[2], qrh[3]));
            st_chunk(sm + OFF_ADLO, c, chunk, make_uint4(krl[0], krl[1], krl[2], krl[3]));
            st_chunk(sm + OFF_ADLO + 16384, c, chunk, make_uint4(qrl[0], qrl[1], qrl[2], qrl[3]));
            st_chunk(sm + OFF_BD, c, chunk, make_uint4(kch[0], kch[1], kch[2], kch[3]));
            st_chunk(sm + OFF_BDLO, c, chunk, make_uint4(kcl[0], kcl[1], kcl[2], kcl[3]));
            st_chunk(qg_dst, c, chunk, make_uint4(gq[0], gq[1], gq[2], gq[3]));
            st_chunk(kt_dst, c, chunk, make_uint4(kt[0], kt[1], kt[2], kt[3]));
        }
    }
}

// Front phase 4: Gram readout.  Rows 0..63 -> A (times beta, strictly lower,
// fp32, shared memory), rows 64..127 -> P (lower including the diagonal,
// fp16, to p_dst).  Waits for the Gram product; ends with a group barrier.
__device__ __forceinline__ bool gram_readout(const Ctx& X, const Lane& t, uint32_t tmem, int lo,
                                             int hi, int step, uint8_t* p_dst)
{
    if (!group_wait(X, B_MMA_G, step)) return false;
    tc_fence_after();
    const float* sBst = reinterpret_cast<const float*>(X.sm + OFF_BST);
    float* sA = reinterpret_cast<float*>(X.sm + OFF_A32);
    const int L = t.L, half = t.half;
    {
        uint32_t dg[32], dl[32];
        tmem_ld32(tmem + t.lane_base + TM_G + 32 * half, dg);
        tmem_ld32(tmem + t.lane_base + TM_G + 64 + 32 * half, dl);
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
                st_chunk(p_dst, r, 4 * half + j, make_uint4(pk[0], pk[1], pk[2], pk[3]));
            }
        }
    }
    fence_proxy_async_smem();      // P may be copied out by the async proxy
    tc_fence_before();
    group_sync();
    return true;
}

// Front phase 5: the UT solve (CUDA-core part; the MMA warp runs the two
// product rounds, mma_front below).  Leaves T as bf16 in shared memory (the
// W product) and as fp16 at t16_dst.  Arrives B_QKG_EMPTY after the first
// round when `release_qkg` (the g tile's space is no longer read) and B_T at
// the end.
__device__ __forceinline__ bool ut_solve(const Ctx& X, const Lane& t, uint32_t tmem, int warp,
                                         int step, bool release_qkg, uint8_t* t16_dst)
{
    uint8_t* sm = X.sm;
    const float* sBst = reinterpret_cast<const float*>(sm + OFF_BST);
    const float* sA = reinterpret_cast<const float*>(sm + OFF_A32);
    float* sD = reinterpret_cast<float*>(sm + OFF_DF);
    const int ct = t.ct, L = t.L, half = t.half;
    const uint32_t lane_base = t.lane_base;
    const bool top = (warp & 3) < 2;         // this warp holds rows 0..63
    // S1a: diagonal-block inverses (warps of ct < 128, one column each): D
    // in fp32 and D' = D Diag(b) as the K-major fp16 B tile.  Meanwhile the
    // other warps fill the chunks of the N and I - N tiles that lie in
    // diagonal or upper blocks (zero in N; identity or zero in I - N).
    if (ct < 128) {
        const int b = ct >> 5, j = ct & 31;
        float x[16];
        diag_block_column(sA, b, j, x);
        if (j < 16) {
            const int k = 16 * b + j;        // column k of D = row k of the D' tile
            const float bk = sBst[k];
#pragma unroll
            for (int r = 0; r < 16; ++r) sD[(16 * b + r) * 17 + j] = x[r];
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint32_t pq[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float dv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int r = 8 * c8 + 2 * e + u;
                        dv[u] = ((r >> 4) == b) ? x[r & 15] : 0.f;
                    }
                    pq[e] = pack_f16x2(dv[0] * bk, dv[1] * bk);
                }
                st_chunk(sm + OFF_DPK, k, c8, make_uint4(pq[0], pq[1], pq[2], pq[3]));
            }
        }
    } else {
        // row R, column blocks 2 jb .. 2 jb + 1 of 16 (chunks 4 jb .. 4 jb + 3)
        const int R = (ct - 128) >> 1, jb = (ct - 128) & 1;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            const int blk16 = 2 * jb + cb;
            if (blk16 >= (R >> 4)) {
#pragma unroll
                for (int h8 = 0; h8 < 2; ++h8) {
                    const int chunk = 2 * blk16 + h8;
                    st_chunk(sm + OFF_NB, R, chunk, make_uint4(0, 0, 0, 0));
                    // the 1 of I - N: column R, in chunk R / 8 at position R % 8
                    uint32_t w[4] = {0, 0, 0, 0};
                    if (chunk == (R >> 3)) w[(R & 7) >> 1] = (R & 1) ? 0x3C000000u : 0x3C00u;
                    st_chunk(sm + OFF_IMN, R, chunk, make_uint4(w[0], w[1], w[2], w[3]));
                }
            }
        }
    }
    group_sync();
    // S1b: N = D A_off, whose non-zero blocks are N_ij = D_ii A_ij for
    // (i, j) = (1,0) (2,0) (2,1) (3,0) (3,1) (3,2): 6 x 16 rows x 8 column
    // pairs = 768 segments, three per thread (computed together), written
    // (fp16) to the N tile and, negated, to the I - N tile.  Both tiles serve
    // as K-major A operands of the first product round (the N tile also as
    // its MN-major B operand).
    {
        const float* drow[3];
        const float* acol[3];
        uint32_t off[3];
#pragma unroll
        for (int rep = 0; rep < 3; ++rep) {
            const int sgi = ct + 256 * rep;
            const int b6 = sgi >> 7, rr = (sgi >> 3) & 15, cpair = sgi & 7;
            const int bi = (b6 == 0) ? 1 : ((b6 < 3) ? 2 : 3);
            const int bj = (b6 == 0) ? 0 : ((b6 < 3) ? b6 - 1 : b6 - 3);
            drow[rep] = sD + (16 * bi + rr) * 17;
            acol[rep] = sA + (16 * bi) * LDA + 16 * bj + 2 * cpair;
            const int R = 16 * bi + rr, col = 16 * bj + 2 * cpair, chunk = col >> 3;
            off[rep] = (R >> 3) * 1024 + (R & 7) * 128 + ((chunk ^ (R & 7)) << 4) + (col & 7) * 2;
        }
        float n[3][2];
#pragma unroll
        for (int rep = 0; rep < 3; ++rep) n[rep][0] = n[rep][1] = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
#pragma unroll
            for (int rep = 0; rep < 3; ++rep) {
                const float d = drow[rep][m];
                const float2 a = *reinterpret_cast<const float2*>(acol[rep] + m * LDA);
                n[rep][0] = fmaf(d, a.x, n[rep][0]);
                n[rep][1] = fmaf(d, a.y, n[rep][1]);
            }
        }
#pragma unroll
        for (int rep = 0; rep < 3; ++rep) {
            *reinterpret_cast<uint32_t*>(sm + OFF_NB + off[rep]) = pack_f16x2(n[rep][0], n[rep][1]);
            *reinterpret_cast<uint32_t*>(sm + OFF_IMN + off[rep]) = pack_f16x2(-n[rep][0], -n[rep][1]);
        }
    }
    fence_proxy_async_smem();
    group_sync();
    if (ct == 0) mbar_arrive(&X.bar[B_S1]);
    // S2: Z -> fp16 MN-major B tile; I + N^2 -> fp16 A operand.
    if (!group_wait(X, B_R1, step)) return false;
    // The g tile's space (D, N, D' tiles) is no longer read: the next chunk may load.
    if (ct == 0 && release_qkg) mbar_arrive(&X.bar[B_QKG_EMPTY]);
    tc_fence_after();
    if (top) {
        uint32_t zb[16], d[32], ip[16];
        tmem_row_f16(tmem + lane_base + TM_Z + 32 * half, zb);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            st_chunk(sm + OFF_ZB, L, 4 * half + j,
                     make_uint4(zb[4 * j], zb[4 * j + 1], zb[4 * j + 2], zb[4 * j + 3]));
        tmem_ld32(tmem + lane_base + TM_N2 + 32 * half, d);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int k = 32 * half + 2 * i;
            const float a0 = __uint_as_float(d[2 * i]) + ((k == L) ? 1.f : 0.f);
            const float a1 = __uint_as_float(d[2 * i + 1]) + ((k + 1 == L) ? 1.f : 0.f);
            ip[i] = pack_f16x2(a0, a1);
        }
        tmem_st16(tmem + lane_base + TM_IPN + 16 * half, ip);
        tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    group_sync();
    if (ct == 0) mbar_arrive(&X.bar[B_S2]);
    // S3: T -> bf16 (W product) and fp16 (V product) rows
    if (!group_wait(X, B_R2, step)) return false;
    tc_fence_after();
    if (top) {
        uint32_t d[32];
        tmem_ld32(tmem + lane_base + TM_T + 32 * half, d);
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
            st_chunk(t16_dst, L, 4 * half + j, make_uint4(ph[0], ph[1], ph[2], ph[3]));
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    group_sync();
    if (ct == 0) mbar_arrive(&X.bar[B_T]);
    return true;
}

// Front phase 6: W readout, -W^T row c = -2^R_c x (Kr^T T^T) row c, fp16 to
// wt_dst.  Ends with a group barrier.
__device__ __forceinline__ bool w_readout(const Ctx& X, const Lane& t, uint32_t tmem, int step,
                                          uint8_t* wt_dst)
{
    if (!group_wait(X, B_MMA_W, step)) return false;
    tc_fence_after();
    const float* sR = reinterpret_cast<const float*>(X.sm + OFF_R);
    {
        uint32_t dw[32];
        tmem_ld32(tmem + t.lane_base + TM_W + 32 * t.half, dw);
        tmem_ld_wait();
        const float sc = -sR[t.L];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pk[e] = pack_f16x2(sc * __uint_as_float(dw[8 * j + 2 * e]),
                                   sc * __uint_as_float(dw[8 * j + 2 * e + 1]));
            st_chunk(wt_dst, t.L, 4 * t.half + j, make_uint4(pk[0], pk[1], pk[2], pk[3]));
        }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    group_sync();
    return true;
}

// ---------------------------------------------------------------------------
// Back phases (the state chain).

// The v tile (two 64-column halves, 128-byte swizzle) from bf16 to fp16 in
// place.  No barrier.
__device__ __forceinline__ void v_tile_to_f16(uint8_t* vtile, int ct)
{
    uint4* vt = reinterpret_cast<uint4*>(vtile);
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

// State decay with its fp16 copy: S^T fp16 (the A operand of this step's
// products) <- S^T, then S^T <- S^T Diag(e^{G_last}).  When `snap` is not
// null the state before the decay (the state at this chunk's start) is also
// stored there ([d_k][d_v] fp32).  This thread: 64 channels of its TMEM lane.
// No barrier.
__device__ __forceinline__ void state_decay(const Lane& t, uint32_t tmem, const float* gl,
                                            float* snap = nullptr)
{
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
        const int c0 = 64 * t.half + 32 * jb;
        uint32_t r[32], b[16];
        tmem_ld32(tmem + t.lane_base + TM_S + c0, r);
        tmem_ld_wait();
        if (snap != nullptr) {
#pragma unroll
            for (int i = 0; i < 32; ++i) snap[(long long)(c0 + i) * kD + t.L] = __uint_as_float(r[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
            b[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        tmem_st16(tmem + t.lane_base + TM_SB + (c0 >> 1), b);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            r[i] = __float_as_uint(__uint_as_float(r[i]) * gl[c0 + i]);
        tmem_st32(tmem + t.lane_base + TM_S + c0, r);
    }
    tmem_st_wait();
}

// U^T (fp32, TMEM) -> the fp16 A operand of the second product.  No barrier.
__device__ __forceinline__ void u_to_f16(const Lane& t, uint32_t tmem)
{
    uint32_t du[32], b[16];
    tmem_ld32(tmem + t.lane_base + TM_C + 32 * t.half, du);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i)
        b[i] = pack_f16x2(__uint_as_float(du[2 * i]), __uint_as_float(du[2 * i + 1]));
    tmem_st16(tmem + t.lane_base + TM_UB + 16 * t.half, b);
    tmem_st_wait();
}

// This thread's 32 rows of O^T (its lane = value column L).
__device__ __forceinline__ void o_load(const Lane& t, uint32_t tmem, uint32_t (&dd)[32])
{
    tmem_ld32(tmem + t.lane_base + TM_O + 32 * t.half, dd);
    tmem_ld_wait();
}

// Stores rows [lo, hi) of a chunk's O (token t0 + r).  A full chunk with bf16
// output is staged in shared memory (stg, [64 tok][128 v] bf16 plain rows) and
// written by one TMA tensor store issued by ct 0 (committed to its bulk
// group; the caller waits for the staging to be read before reusing it);
// other chunks (a ragged tail, the passes of a wide chunk, fp32 output) are
// stored by the threads.  `use_tma` must be uniform over the group.
template <typename TO>
__device__ __forceinline__ void o_store(const Lane& t, const uint32_t (&dd)[32], bool use_tma,
                                        const CUtensorMap* tm_o, uint8_t* stg, TO* o, long long t0,
                                        int lo, int hi, int h, int H)
{
    if (use_tma) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int r = 32 * t.half + i;
            *reinterpret_cast<__nv_bfloat16*>(stg + r * 256 + 2 * t.L) =
                __float2bfloat16_rn(__uint_as_float(dd[i]));
        }
        fence_proxy_async_smem();
        group_sync();
        if (t.ct == 0) {
            tma_store_2d(tm_o, h * kD, (int32_t)t0, stg);
            bulk_commit_group();
        }
    } else {
        TO* op = o + (t0 * H + h) * kD + t.L;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int r = 32 * t.half + i;
            if (r >= lo && r < hi) out_store(op + (long long)r * H * kD, __uint_as_float(dd[i]));
        }
    }
}

// S^T <- S0^T (row v of S^T is column v of S0), or zeros.  This thread: 64
// channels of its TMEM lane.
__device__ __forceinline__ void state_load(const Lane& t, uint32_t tmem, const float* S0,
                                           long long sbase)
{
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int c = 64 * t.half + 32 * jb + i;
            r[i] = __float_as_uint(S0 ? S0[sbase + (long long)c * kD + t.L] : 0.f);
        }
        tmem_st32(tmem + t.lane_base + TM_S + 64 * t.half + 32 * jb, r);
    }
    tmem_st_wait();
}

// Where the prefix snapshot taken at the start of chunk `ch` (the state after
// the sequence's first 64 ch tokens) goes, or null when none is due there.
// ch = the sequence's chunk count gives the end-of-sequence snapshot, due only
// when 64 ch is the sequence's length `len`.
__device__ __forceinline__ float* snapshot_at(const SnapArgs& sn, int ch, long long len, int seq_off,
                                              int H, int h)
{
    if (sn.interval <= 0 || ch <= 0) return nullptr;
    const long long tok = (long long)ch * kC;
    if (tok > len || tok % sn.interval != 0) return nullptr;
    const long long j = tok / sn.interval - 1;
    return sn.out + ((long long)(seq_off + j) * H + h) * kD * kD;
}

__device__ __forceinline__ void state_store(const Lane& t, uint32_t tmem, float* S_final,
                                            long long sbase)
{
    tc_fence_after();
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
        uint32_t r[32];
        tmem_ld32(tmem + t.lane_base + TM_S + 64 * t.half + 32 * jb, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
            S_final[sbase + (long long)(64 * t.half + 32 * jb + i) * kD + t.L] = __uint_as_float(r[i]);
    }
}

// ---------------------------------------------------------------------------
// MMA warp (one thread).

struct FrontDescs {
    uint64_t AD, ADLO, BDHL, ADK, T, NA, IMN, NB, DPK, ZB;
    uint32_t id_g, id_w, id_mn, id_k64;
};

// Base descriptors; a K step advances the start address field (16-byte
// units) by 128 for MN-major tiles, by 2 for K-major ones.
__device__ __forceinline__ FrontDescs make_front_descs(uint8_t* sm)
{
    FrontDescs D;
    D.id_g = make_idesc_bf16(128, 128, true, true);     // Gram
    D.id_w = make_idesc_bf16(128, 64, false, false);    // W
    D.id_mn = make_idesc_f16(128, 64, false, true);     // K-major A x MN-major B
    D.id_k64 = make_idesc_f16(128, 64, false, false);   // K-major A x K-major B
    D.AD = make_sdesc(smem_u32(sm + OFF_AD), 16384, 1024, kSwizzle128B);
    D.ADLO = make_sdesc(smem_u32(sm + OFF_ADLO), 16384, 1024, kSwizzle128B);
    D.BDHL = make_sdesc(smem_u32(sm + OFF_BD), OFF_BDLO - OFF_BD, 1024, kSwizzle128B);
    D.ADK = make_sdesc(smem_u32(sm + OFF_AD), 16, 1024, kSwizzle128B);
    D.T = make_sdesc(smem_u32(sm + OFF_T), 16, 1024, kSwizzle128B);
    D.NA = make_sdesc(smem_u32(sm + OFF_NB), 16, 1024, kSwizzle128B);   // N as K-major A
    D.IMN = make_sdesc(smem_u32(sm + OFF_IMN), 16, 1024, kSwizzle128B);
    D.NB = make_sdesc(smem_u32(sm + OFF_NB), 8192, 1024, kSwizzle128B);
    D.DPK = make_sdesc(smem_u32(sm + OFF_DPK), 16, 1024, kSwizzle128B);
    D.ZB = make_sdesc(smem_u32(sm + OFF_ZB), 8192, 1024, kSwizzle128B);
    return D;
}

// The front products of one step, after B_OPS: the Gram, the two solve
// rounds and W^T.  Called by the whole MMA warp.  Returns false if a wait
// gave up.
__device__ __forceinline__ bool mma_front(const Ctx& X, uint32_t tmem, const FrontDescs& D,
                                          int step)
{
    // Gram: [Kr; Qr] (MN-major A) x [Kc hi | Kc lo] (MN-major B, N = 128),
    // K = 128 channels, hi and lo A parts: the readout adds the halves.
#pragma unroll
    for (int s = 0; s < 8; ++s) mma_ss(tmem + TM_G, D.AD + 128 * s, D.BDHL + 128 * s, D.id_g, s > 0);
#pragma unroll
    for (int s = 0; s < 8; ++s) mma_ss(tmem + TM_G, D.ADLO + 128 * s, D.BDHL + 128 * s, D.id_g, 1);
    mma_commit(&X.bar[B_MMA_G]);
    // UT solve, round 1: N^2 = N N and Z = (I - N) D'; round 2: T = (I + N^2) Z.
    if (!warp_wait(X, B_S1, step)) return false;
    tc_fence_after();
    // (M = 128 with A rows 64..127 read from the next tile: finite data,
    // rows unused.)
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_ss(tmem + TM_N2, D.NA + 2 * s, D.NB + 128 * s, D.id_mn, s > 0);
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_ss(tmem + TM_Z, D.IMN + 2 * s, D.DPK + 2 * s, D.id_k64, s > 0);
    mma_commit(&X.bar[B_R1]);
    if (!warp_wait(X, B_S2, step)) return false;
    tc_fence_after();
#pragma unroll
    for (int s = 0; s < 4; ++s)
        mma_ts(tmem + TM_T, tmem + TM_IPN + 8 * s, D.ZB + 128 * s, D.id_mn, s > 0);
    mma_commit(&X.bar[B_R2]);
    if (!warp_wait(X, B_T, step)) return false;
    tc_fence_after();
    // W^T (unscaled) = Kr^T T^T: A = Kr hi as K-major [ch][tok], B = T [r][i].
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_ss(tmem + TM_W, D.ADK + 2 * s, D.T + 2 * s, D.id_w, s > 0);
    mma_commit(&X.bar[B_MMA_W]);
    return true;
}

// [U^T | O^T] = S^T [-W^T | (e^G Q)^T] ;  U^T += V^T T^T.  Shared-memory
// addresses: wt = -W^T with (e^G Q)^T 16 KB after it, t16 = T (fp16),
// vtile = the fp16 v tile.
__device__ __forceinline__ void mma_back_c(uint32_t tmem, uint32_t wt, uint32_t t16, uint32_t vtile)
{
    const uint32_t id_cv = make_idesc_f16(128, 64, true, false);     // V^T T^T
    const uint32_t id_mn128 = make_idesc_f16(128, 128, false, true); // S^T x [-W^T | (e^G Q)^T]
    const uint64_t dWQ = make_sdesc(wt, BLK_QG - BLK_WT, 1024, kSwizzle128B);
    const uint64_t dV = make_sdesc(vtile, 8192, 1024, kSwizzle128B);
    const uint64_t dT16 = make_sdesc(t16, 16, 1024, kSwizzle128B);
#pragma unroll
    for (int s = 0; s < 8; ++s) mma_ts(tmem + TM_C, tmem + TM_SB + s * 8, dWQ + 128 * s, id_mn128, s > 0);
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_ss(tmem + TM_C, dV + 128 * s, dT16 + 2 * s, id_cv, 1);
}

// [O^T | S^T] += U^T [P | Ktil^T]^T   (N = 64 + 128).  p = the shared-memory
// address of P, with Ktil^T 8 KB after it.
__device__ __forceinline__ void mma_back_os(uint32_t tmem, uint32_t p)
{
    const uint32_t id_os = make_idesc_f16(128, 192, false, false);
    const uint64_t dPK = make_sdesc(p, 16, 1024, kSwizzle128B);
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_ts(tmem + TM_O, tmem + TM_UB + s * 8, dPK + 2 * s, id_os, 1);
}

}  // namespace tc
}  // namespace kda
