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
// Operand precision.  The Gram operands carry the exponent factors and need an
// 8-bit exponent: they are fp32 values multiplied as tf32 (10-bit mantissa)
// with fp32 accumulation.  With fp32 output they are rounded to nearest
// first; with bf16 output the tensor cores' truncation is left in place (its
// bias stays well below the output's own rounding, and the rounding costs
// several percent of the launch).  T, P, U, S, V, W, e^G Q, e^G K and Ktil
// are O(1) and enter the tensor cores as fp16 (3 more mantissa bits than
// bf16).  The UT solve keeps about 22 significant bits (fp32 diagonal blocks,
// two-term fp16 operands in its block products) and the state is carried in
// fp32.  |v| and the state entries are assumed to stay inside the fp16 range
// (|x| < 65504).
//
// UT solve.  X = (I + A)^{-1} by block forward substitution on 16 x 16 blocks:
// the diagonal blocks' inverses X_bb in fp32 on the CUDA cores by column-wise
// substitution, then X_ij = -X_ii sum_{j <= k < i} A_ik X_kj for i > j as six
// warp chains of 16 x 16 products on the warp tensor cores, each operand split
// into two fp16 terms (about 22 significant bits, see ut_solve_mma).
// T = X Diag(b).  W = T (e^G K) is then one tensor-core product with the fp16
// T and (e^G K)^T tiles.

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
// Named barriers of the UT solve's warp chains (ids 2 .. 4), see ut_solve_mma.
constexpr int kBarSolve0 = 2;
constexpr float kLog2e = 1.4426950408889634f;
// Largest decay span (log2 units) handled in one pass.
constexpr float kSpanMax = 250.f;

// ---- shared memory map of the front phases (bytes from a 1024-aligned base)
constexpr uint32_t OFF_Q = 0;          // q tile  [64 tok][128 ch] bf16, plain rows
constexpr uint32_t OFF_K = 16384;      // k tile  [64][128] bf16
constexpr uint32_t OFF_G = 32768;      // g tile  [64][128] fp32 (after gate prep, in the
                                       //   single-CTA kernel: the (e^G K)^T tile, 16 KB)
constexpr uint32_t OFF_V = 65536;      // v tile  2 x [64 tok][64 v], 128B swizzle (bf16 -> fp16);
                                       //   split producer: the (e^G K)^T tile
constexpr uint32_t OFF_A = 81920;      // Gram A operand [Kr; Qr] tf32, K-major [128][128] (64 KB)
constexpr uint32_t OFF_KC = 147456;    // Gram B operand Kc tf32, K-major [64][128] (32 KB)
// After the Gram product, in the operand region [OFF_A, OFF_QG):
constexpr uint32_t OFF_A32 = OFF_A;           // A fp32 [64][LDA]
constexpr uint32_t OFF_X = OFF_A + 17408;     // X = (I + A)^-1 fp32 [64][LDA]
constexpr uint32_t OFF_ZS = OFF_X + 17408;    // solve scratch, 6 x [16][LDZ] (or [16][LDT]) fp32;
constexpr uint32_t OFF_STAT = OFF_ZS;         //   before it, the gate prep's decay stats [3][4][128]
constexpr uint32_t OFF_T16 = 126976;   // T       [r][i] fp16 (W and V products)
constexpr uint32_t OFF_WT = 163840;    // -W^T    [ch][r] fp16 (directly before (e^G Q)^T)
constexpr uint32_t OFF_QG = 180224;    // (e^G Q)^T [ch][r] fp16
constexpr uint32_t OFF_P = 196608;     // P       [r][i] fp16 (directly before Ktil^T)
constexpr uint32_t OFF_KT = 204800;    // Ktil^T  [ch][i] fp16
constexpr uint32_t OFF_OST = OFF_A32;  // O tile staging of the single-CTA kernel
constexpr uint32_t OFF_Y = 221184;     // 2 KB: the first 1 KB not used by the phases, then
constexpr uint32_t OFF_NRM = OFF_Y + 1024;    // gate prologue: q_scale/||q_r|| [64], 1/||k_r|| [64]
constexpr uint32_t OFF_AH = OFF_Y + 1536;     // gate prologue: the head's A row [128] (split producer)
constexpr uint32_t OFF_GL = 223232;    // e^{G_last} per channel
constexpr uint32_t OFF_BIN = 223744;   // beta of the loaded chunk
constexpr uint32_t OFF_BST = 224000;   // beta of the current pass (masked)
constexpr uint32_t OFF_DESC = 224256;  // 2 step descriptors
constexpr uint32_t OFF_BAR = 224320;   // mbarriers (kNumBars x 8 B)
constexpr uint32_t OFF_MISC = 224544;  // tmem base, flags
constexpr uint32_t kSmemUsed = 224560;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;   // + alignment slack
constexpr int LDA = 68;                // row stride (floats) of A / X: 16-byte aligned rows
constexpr int LDZ = 20;                // row stride (floats) of a chain's scratch block
static_assert(OFF_STAT + 6144 <= OFF_T16 && OFF_ZS + 6 * 16 * LDZ * 4 <= OFF_T16 &&
              OFF_ZS + 6 * 16 * 24 * 4 <= OFF_T16 &&
              OFF_T16 + 8192 <= OFF_WT, "post-Gram tiles overlap");
static_assert(OFF_KC + 32768 == OFF_QG && OFF_A + 65536 == OFF_KC, "operand region");
static_assert(OFF_QG - OFF_WT == 16384 && OFF_KT - OFF_P == 8192,
              "the back products read -W^T | (e^G Q)^T and P | Ktil^T as one tile each");

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
    B_JOB_DONE,                                        // split producer: operands written
    B_SV_FULL0, B_SV_FULL1, B_SV_FULL2, B_SV_FULL3,    // split consumer: v tile buffers
    B_SV_EMPTY0, B_SV_EMPTY1, B_SV_EMPTY2, B_SV_EMPTY3,
    B_ST_FULL0, B_ST_FULL1, B_ST_EMPTY0, B_ST_EMPTY1,  // split consumer: operand stages
    kNumBars
};
static_assert(OFF_BAR + kNumBars * 8 <= OFF_MISC, "barrier area overflows");

// TMEM columns (512 allocated).  C|O and O|S are adjacent so that one MMA
// can write both of a pair.
constexpr uint32_t TM_G = 0;      // Gram [Kr rows; Qr rows] x Kc                 64 cols
constexpr uint32_t TM_W = 0;      // W^T [ch][r], after the Gram readout          64 cols
constexpr uint32_t TM_SB = 128;   // S^T fp16 A operand                           64 cols
constexpr uint32_t TM_C = 192;    // U^T fp32 [v][r]                              64 cols
constexpr uint32_t TM_O = 256;    // O^T fp32 [v][r]                              64 cols
constexpr uint32_t TM_S = 320;    // S^T fp32 [v][ch]                            128 cols
constexpr uint32_t TM_UB = 448;   // U^T fp16 A operand                           32 cols
constexpr uint32_t kTmemCols = 512;

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

// x as a tf32 operand rounded to nearest: the tensor cores read only the top
// 19 bits (sign, exponent, 10 mantissa bits) and would otherwise truncate,
// a bias of the same sign on every operand.  Adding half a unit of the 10th
// mantissa bit to the bit pattern rounds the magnitude to nearest (a carry
// into the exponent is the correct result); the low 13 bits are ignored.
__device__ __forceinline__ float tf32_round(float x)
{
    return __uint_as_float(__float_as_uint(x) + 0x1000u);
}

__device__ __forceinline__ float lo_bf16(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ void out_store(float* p, float x) { *p = x; }
__device__ __forceinline__ void out_store(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void out_store(__half* p, float x) { *p = __float2half_rn(x); }

// Limit of a bounded wait: 2^32 SM cycles, about two seconds.  (A compile-
// time constant: a limit held in a register measured 5 % slower at 1M tokens.)
constexpr long long kWaitLimit = 1ll << 32;

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
    if (mbar_wait(&X.bar[b], phase & 1u, kWaitLimit)) return true;
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

// A chunk of two passes: the threads whose rows fall in the second pass
// (rq >= 2) keep their running sums in the g tile, in place of the g values
// they were computed from (each thread writes only what it read), so that
// they need not stay in registers through the first pass.  The second half
// of the g tile is not overwritten before the second pass.
__device__ __forceinline__ void stash_running_sums(const Lane& t, float* sG, const float2 (&Gq)[16])
{
    if (t.rq < 2) return;
#pragma unroll
    for (int rr = 0; rr < 16; ++rr)
        *reinterpret_cast<float2*>(sG + (16 * t.rq + rr) * kD + 2 * t.cp) = Gq[rr];
}

__device__ __forceinline__ void load_running_sums(const Lane& t, const float* sG, float2 (&Gq)[16])
{
    const int rq = t.rq < 2 ? t.rq + 2 : t.rq;      // rows of the first pass: unused values
#pragma unroll
    for (int rr = 0; rr < 16; ++rr)
        Gq[rr] = *reinterpret_cast<const float2*>(sG + (16 * rq + rr) * kD + 2 * t.cp);
}

// Front phase 2: this pass's per-channel e^{G_last} (to gl_dst) and the
// masked beta.  No barrier.
__device__ __forceinline__ void pass_factors(const Ctx& X, const Lane& t, const Pass& ps,
                                             float* gl_dst)
{
    const float* sBin = reinterpret_cast<const float*>(X.sm + OFF_BIN);
    float* sBst = reinterpret_cast<float*>(X.sm + OFF_BST);
    if (t.rq == 0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) gl_dst[2 * t.cp + u] = ps.glc[u];
    }
    if (t.ct < kC) sBst[t.ct] = (t.ct >= ps.lo && t.ct < ps.hi) ? sBin[t.ct] : 0.f;
}

// Byte offset of element (row, channel ch) in a K-major tf32 tile with the
// 128-byte swizzle: 32 channels per 128-byte row, 8-row groups 1024 bytes
// apart, channel groups of 32 `kstride` bytes apart.
__device__ __forceinline__ uint32_t tf32_kmajor(int row, int ch, uint32_t kstride)
{
    return (uint32_t)(ch >> 5) * kstride + (uint32_t)(row >> 3) * 1024 + (uint32_t)(row & 7) * 128 +
           ((((uint32_t)(ch & 31) >> 2) ^ (uint32_t)(row & 7)) << 4) + (uint32_t)(ch & 3) * 4;
}

// Front phase 3: the operands of the Gram product, Kr = k e^{G-R} and
// Qr = q e^{G-R} (rows 0..63 and 64..127 of the A tile) and Kc = k e^{R-G}
// (the B tile), fp32 in the K-major tf32 layout; and the fp16 [channel][token]
// tiles (e^G Q)^T, Ktil^T = (k e^{G_last-G})^T and (e^G K)^T to qg_dst, kt_dst
// and gk_dst.  This thread: channels 2cp, 2cp+1 of rows 16rq .. 16rq+15.  Each
// tf32 row store covers both channels (8 bytes; a warp's 32 stores fill two
// 128-byte rows); the fp16 chunks of the two channels are stored in an order
// that alternates between lane groups, so that a warp's 16-byte stores spread
// over all eight swizzle positions.  With the gate prologue (FUSED) q and k
// are scaled by their rows' inverse norms (OFF_NRM).  ROUND: the tf32
// operands are rounded to nearest (see the precision note above).  No barrier.
template <bool FUSED, bool ROUND>
__device__ __forceinline__ void gram_operands(const Ctx& X, const Lane& t, const Pass& ps,
                                              const float2 (&Gq)[16], uint8_t* qg_dst,
                                              uint8_t* kt_dst, uint8_t* gk_dst)
{
    const float* nrm = reinterpret_cast<const float*>(X.sm + OFF_NRM);
    const int cp = t.cp, rq = t.rq, lo = ps.lo, hi = ps.hi;
    const uint8_t* sQ = X.sm + OFF_Q;
    const uint8_t* sK = X.sm + OFF_K;
    uint8_t* sA = X.sm + OFF_A;
    uint8_t* sKc = X.sm + OFF_KC;
    const bool swap = ((cp >> 2) & 1) != 0;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        uint32_t kp[8], qp[8];             // bf16 pairs (channels 2cp, 2cp+1)
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8) {
            const int r = 16 * rq + 8 * jj + w8;
            kp[w8] = *reinterpret_cast<const uint32_t*>(sK + r * 256 + 4 * cp);
            qp[w8] = *reinterpret_cast<const uint32_t*>(sQ + r * 256 + 4 * cp);
        }
        uint32_t gq[2][4], kt[2][4], gk[2][4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float vk[2][2], vq[2][2], vc[2][2];      // [channel u][row w]
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const int w8 = 2 * e + w, rr = 8 * jj + w8, r = 16 * rq + rr;
                const bool act = (r >= lo && r < hi);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
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
                    vk[u][w] = kk * e1;
                    vq[u][w] = qq * e1;
                    vc[u][w] = kk * e2;
                }
                auto rnd = [](float x) { return ROUND ? tf32_round(x) : x; };
                *reinterpret_cast<float2*>(sA + tf32_kmajor(r, 2 * cp, 16384)) =
                    make_float2(rnd(vk[0][w]), rnd(vk[1][w]));
                *reinterpret_cast<float2*>(sA + tf32_kmajor(64 + r, 2 * cp, 16384)) =
                    make_float2(rnd(vq[0][w]), rnd(vq[1][w]));
                *reinterpret_cast<float2*>(sKc + tf32_kmajor(r, 2 * cp, 8192)) =
                    make_float2(rnd(vc[0][w]), rnd(vc[1][w]));
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                gq[u][e] = pack_f16x2(vq[u][0] * ps.pRc[u], vq[u][1] * ps.pRc[u]);
                kt[u][e] = pack_f16x2(vc[u][0] * ps.pLc[u], vc[u][1] * ps.pLc[u]);
                gk[u][e] = pack_f16x2(vk[u][0] * ps.pRc[u], vk[u][1] * ps.pRc[u]);
            }
        }
        const int chunk = 2 * rq + jj;
#pragma unroll
        for (int o = 0; o < 2; ++o) {
            const bool u1 = (o == 1) != swap;
            const int c = 2 * cp + (u1 ? 1 : 0);
            st_chunk(qg_dst, c, chunk, u1 ? make_uint4(gq[1][0], gq[1][1], gq[1][2], gq[1][3])
                                          : make_uint4(gq[0][0], gq[0][1], gq[0][2], gq[0][3]));
            st_chunk(kt_dst, c, chunk, u1 ? make_uint4(kt[1][0], kt[1][1], kt[1][2], kt[1][3])
                                          : make_uint4(kt[0][0], kt[0][1], kt[0][2], kt[0][3]));
            st_chunk(gk_dst, c, chunk, u1 ? make_uint4(gk[1][0], gk[1][1], gk[1][2], gk[1][3])
                                          : make_uint4(gk[0][0], gk[0][1], gk[0][2], gk[0][3]));
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
        uint32_t dg[32];
        tmem_ld32(tmem + t.lane_base + TM_G + 32 * half, dg);
        tmem_ld_wait();
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

// ---- the UT solve's 16 x 16 block products on the warp tensor cores.
// Operands are fp32 values split into fp16 pairs x = hi + lo (hi = x rounded
// to fp16, lo = the rest rounded to fp16); a product takes the three terms
// hi hi + hi lo + lo hi with fp32 accumulation: about 22 significant bits
// (entries below 2^-3 keep an absolute accuracy of about 2^-25, from lo's
// subnormals).  X's entries must stay below 65504 (T = X Diag(beta) is fp16
// anyway).  A bf16 split (16 bits, fp32's range) lost too much where the
// chain products cancel: beta = 2 with no decay moved o by 4 % of its RMS.

// Splits (x0, x1) into packed fp16 pairs: hi and lo.
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    hi = pack_f16x2(x0, x1);
    const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    lo = pack_f16x2(x0 - h.x, x1 - h.y);
}

// d += a b for one m16n8k16 tile (a: 4 registers, b: 2, d: 4).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// c[nh] += L R for a 16 x 16 output in two 16 x 8 halves, three terms each.
// The A fragment is given split (ah, al); the B fragment of half nh is read
// from row-major fp32 storage where element (k, n) of B sits at
// bsrc[n * ldb + k] (so B^T is stored row-major), for the lane's rows g and
// g + 8 of each half and columns 2 tq, 2 tq + 1 and 2 tq + 8, 2 tq + 9.
__device__ __forceinline__ void blk_mma(float (&c)[2][4], const uint32_t (&ah)[4],
                                        const uint32_t (&al)[4], const float* bsrc, int ldb,
                                        int g, int tq)
{
#pragma unroll
    for (int nh = 0; nh < 2; ++nh) {
        const float* br = bsrc + (8 * nh + g) * ldb + 2 * tq;
        const float2 x0 = *reinterpret_cast<const float2*>(br);
        const float2 x1 = *reinterpret_cast<const float2*>(br + 8);
        uint32_t bh0, bl0, bh1, bl1;
        split_f16x2(x0.x, x0.y, bh0, bl0);
        split_f16x2(x1.x, x1.y, bh1, bl1);
        mma_f16_16816(c[nh], ah, bh0, bh1);
        mma_f16_16816(c[nh], ah, bl0, bl1);
        mma_f16_16816(c[nh], al, bh0, bh1);
    }
}

// Transposed copies of the blocks that later chains read as A operands:
// X00, X11, X22 and Y10, Y20, Y21, [16][LDT] fp32 each, at OFF_ZS.
constexpr int LDT = 24;                // row stride (floats): conflict-free 8-byte fragment loads
__device__ __forceinline__ int xt_slot(int k, int j)
{
    return (k == j) ? k : (k == 1 ? 3 : (j == 0 ? 4 : 5));
}

// Front phase 5: the UT solve with its block products on the warp tensor
// cores.  With a v tile given, the two warps that run no chain convert it to
// fp16 meanwhile (see the end of the chain phase).  From A (OFF_A32) builds X = (I + A)^{-1}
// (OFF_X) block by block and writes T = X Diag(b) as the fp16 tile t16_dst
// ([r][i], zero above the diagonal; b = the masked beta of the pass, so T is
// zero outside the pass).  Arrives B_T at the end.
//
// The diagonal blocks' inverses X_bb come first (64 threads, one column of
// one block each, by forward substitution, in fp32).  Then X_ij = -X_ii
// sum_{j<=k<i} A_ik X_kj for the six blocks below the diagonal, one warp per
// block, as chains of 16 x 16 products on the warp tensor cores (blk_mma):
//   (1,0) (2,0) (3,0) (2,1) (3,1) (3,2)
// Each chain works on transposes, Z^T = sum X_kj^T A_ik^T and X_ij^T =
// -Z^T X_ii^T, so that the first product's accumulators are already the A
// fragment of the second.  A chain needs the blocks X_kj (j < k < i) of the
// chains before it: Y10 for (2,0) and (3,0), Y20 for (3,0), Y21 for (3,1);
// the chain that stores such a block arrives on its named barrier and the
// chains that read it wait there.  (With fp32 FMAs on the CUDA cores, the
// chains' critical path of six products took about 3.3K cycles per chunk.)
__device__ __forceinline__ void ut_solve_mma(const Ctx& X, const Lane& t, uint8_t* t16_dst,
                                             uint8_t* vtile = nullptr, uint32_t v_phase = 0)
{
    uint8_t* sm = X.sm;
    const float* sBst = reinterpret_cast<const float*>(sm + OFF_BST);
    const float* sA = reinterpret_cast<const float*>(sm + OFF_A32);
    float* sX = reinterpret_cast<float*>(sm + OFF_X);
    float* sXt = reinterpret_cast<float*>(sm + OFF_ZS);
    const int ct = t.ct;
    if (ct < 64) {
        // Column j of the unit-lower diagonal block b, by forward substitution.
        const int b = ct >> 4, j = ct & 15;
        const float* L = sA + (16 * b) * LDA + 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < 15; ++i)
#pragma unroll
            for (int r = i + 1; r < 16; ++r) x[r] = fmaf(-L[r * LDA + i], x[i], x[r]);
        float* xo = sX + (16 * b) * LDA + 16 * b + j;
#pragma unroll
        for (int r = 0; r < 16; ++r) xo[r * LDA] = x[r];
        if (b < 3) {   // the transposed copy: column j of X_bb is row j of X_bb^T
            float4* xt = reinterpret_cast<float4*>(sXt + xt_slot(b, b) * 16 * LDT + j * LDT);
#pragma unroll
            for (int r4 = 0; r4 < 4; ++r4)
                xt[r4] = make_float4(x[4 * r4], x[4 * r4 + 1], x[4 * r4 + 2], x[4 * r4 + 3]);
        }
    }
    group_sync();
    const int wc = ct >> 5, lane = ct & 31;
    if (wc < 6) {
        // chain wc computes block (bi, bj); barrier ids: (1,0) +0, (2,0) +1, (2,1) +2
        const int bi = (wc < 3) ? wc + 1 : (wc < 5 ? wc - 1 : 3);
        const int bj = (wc < 3) ? 0 : (wc < 5 ? 1 : 2);
        const int g = lane >> 2, tq = lane & 3;
        float c[2][4];
#pragma unroll
        for (int nh = 0; nh < 2; ++nh)
#pragma unroll
            for (int e = 0; e < 4; ++e) c[nh][e] = 0.f;
#pragma unroll 1
        for (int k = bj; k < bi; ++k) {
            if (k > bj) {
                // block (k, bj) is another chain's result: (1,0), (2,0) or (2,1)
                const int id = (bj == 0) ? k - 1 : 2;
                named_bar_sync(kBarSolve0 + id, id == 0 ? 96 : 64);
            }
            // A fragment: X_kj^T (rows of the transposed copy).
            const float* xt = sXt + xt_slot(k, bj) * 16 * LDT + 2 * tq;
            const float2 a0 = *reinterpret_cast<const float2*>(xt + g * LDT);
            const float2 a1 = *reinterpret_cast<const float2*>(xt + (g + 8) * LDT);
            const float2 a2 = *reinterpret_cast<const float2*>(xt + g * LDT + 8);
            const float2 a3 = *reinterpret_cast<const float2*>(xt + (g + 8) * LDT + 8);
            uint32_t ah[4], al[4];
            split_f16x2(a0.x, a0.y, ah[0], al[0]);
            split_f16x2(a1.x, a1.y, ah[1], al[1]);
            split_f16x2(a2.x, a2.y, ah[2], al[2]);
            split_f16x2(a3.x, a3.y, ah[3], al[3]);
            // B = A_ik^T: element (k', n) = A_ik[n][k'], rows of A.
            blk_mma(c, ah, al, sA + (16 * bi) * LDA + 16 * k, LDA, g, tq);
        }
        // Y^T = Z^T X_ii^T: the accumulators are the A fragment; B = X_ii^T,
        // element (k', n) = X_ii[n][k'], rows of X_ii.
        uint32_t ah[4], al[4];
        split_f16x2(c[0][0], c[0][1], ah[0], al[0]);
        split_f16x2(c[0][2], c[0][3], ah[1], al[1]);
        split_f16x2(c[1][0], c[1][1], ah[2], al[2]);
        split_f16x2(c[1][2], c[1][3], ah[3], al[3]);
        float y[2][4];
#pragma unroll
        for (int nh = 0; nh < 2; ++nh)
#pragma unroll
            for (int e = 0; e < 4; ++e) y[nh][e] = 0.f;
        blk_mma(y, ah, al, sX + (16 * bi) * LDA + 16 * bi, LDA, g, tq);
        // X_ij = -Y: element (m, n) of Y^T is X_ij[n][m] with m = g, g + 8 and
        // n = 8 nh + 2 tq, 8 nh + 2 tq + 1.
        float* xo = sX + (16 * bi) * LDA + 16 * bj;
#pragma unroll
        for (int nh = 0; nh < 2; ++nh)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = g + 8 * (e >> 1), n = 8 * nh + 2 * tq + (e & 1);
                xo[n * LDA + m] = -y[nh][e];
            }
        if (wc == 0 || wc == 1 || wc == 3) {
            // (1,0) is read by chains 1 and 2, (2,0) by chain 2, (2,1) by chain 4
            float* xt = sXt + xt_slot(bi, bj) * 16 * LDT + 2 * tq;
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
                *reinterpret_cast<float2*>(xt + g * LDT + 8 * nh) = make_float2(-y[nh][0], -y[nh][1]);
                *reinterpret_cast<float2*>(xt + (g + 8) * LDT + 8 * nh) =
                    make_float2(-y[nh][2], -y[nh][3]);
            }
            named_bar_arrive(kBarSolve0 + (wc == 3 ? 2 : wc), wc == 0 ? 96 : 64);
        }
    } else if (vtile != nullptr) {
        // The two warps without a chain: the chunk's v tile (its TMA load,
        // phase v_phase of B_V_FULL) from bf16 to fp16 in place, off the
        // Gram product's shared-memory reads.
        if (wait_bar(X, B_V_FULL, v_phase)) {
            uint4* vt = reinterpret_cast<uint4*>(vtile);
            for (int i = ct - 192; i < 1024; i += 64) {
                uint4 x = vt[i];
                x.x = bf16x2_to_f16x2(x.x);
                x.y = bf16x2_to_f16x2(x.y);
                x.z = bf16x2_to_f16x2(x.z);
                x.w = bf16x2_to_f16x2(x.w);
                vt[i] = x;
            }
            fence_proxy_async_smem();
        }
    }
    group_sync();
    // T = X Diag(b), fp16, zero above the diagonal: 512 chunks of 8, two per thread.
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int q = ct + 256 * e, rr = q >> 3, j = q & 7;
        const float4* xr = reinterpret_cast<const float4*>(sX + rr * LDA + 8 * j);
        const float4* bb = reinterpret_cast<const float4*>(sBst + 8 * j);
        const float4 x0 = xr[0], x1 = xr[1], b0 = bb[0], b1 = bb[1];
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        uint32_t pk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i0 = 8 * j + 2 * k;
            pk[k] = pack_f16x2(i0 <= rr ? xv[2 * k] * bv[2 * k] : 0.f,
                               i0 + 1 <= rr ? xv[2 * k + 1] * bv[2 * k + 1] : 0.f);
        }
        st_chunk(t16_dst, rr, j, make_uint4(pk[0], pk[1], pk[2], pk[3]));
    }
    fence_proxy_async_smem();      // T is read by the W product (and copied out)
    group_sync();
    if (ct == 0) mbar_arrive(&X.bar[B_T]);
}

// Front phase 6: W readout, -W^T (fp16 [ch][r]) to wt_dst.  Ends with a group
// barrier.
__device__ __forceinline__ bool w_readout(const Ctx& X, const Lane& t, uint32_t tmem, int step,
                                          uint8_t* wt_dst)
{
    if (!group_wait(X, B_MMA_W, step)) return false;
    tc_fence_after();
    {
        uint32_t dw[32];
        tmem_ld32(tmem + t.lane_base + TM_W + 32 * t.half, dw);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pk[e] = pack_f16x2(-__uint_as_float(dw[8 * j + 2 * e]),
                                   -__uint_as_float(dw[8 * j + 2 * e + 1]));
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
    // 16 columns at a time: this phase runs while many other values are live,
    // and wider pieces spilled registers.
#pragma unroll 1
    for (int jb = 0; jb < 4; ++jb) {
        const int c0 = 64 * t.half + 16 * jb;
        uint32_t r[16], b[8];
        tmem_ld16(tmem + t.lane_base + TM_S + c0, r);
        tmem_ld_wait();
        if (snap != nullptr) {
#pragma unroll
            for (int i = 0; i < 16; ++i) snap[(long long)(c0 + i) * kD + t.L] = __uint_as_float(r[i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            b[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        tmem_st8(tmem + t.lane_base + TM_SB + (c0 >> 1), b);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            r[i] = __float_as_uint(__uint_as_float(r[i]) * gl[c0 + i]);
        tmem_st16(tmem + t.lane_base + TM_S + c0, r);
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
// output is staged in shared memory (stg, [64 tok][128 v] plain rows of the
// 16-bit output type) and written by one TMA tensor store issued by ct 0
// (committed to its bulk group; the caller waits for the staging to be read
// before reusing it); other chunks (a ragged tail, the passes of a wide chunk,
// fp32 output) are stored by the threads.  `use_tma` must be uniform over the
// group, and false for fp32 output.
__device__ __forceinline__ void stage16(uint8_t* p, float x, const __nv_bfloat16*)
{
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(x);
}
__device__ __forceinline__ void stage16(uint8_t* p, float x, const __half*)
{
    *reinterpret_cast<__half*>(p) = __float2half_rn(x);
}
__device__ __forceinline__ void stage16(uint8_t*, float, const float*) {}

template <typename TO>
__device__ __forceinline__ void o_store(const Lane& t, const uint32_t (&dd)[32], bool use_tma,
                                        const CUtensorMap* tm_o, uint8_t* stg, TO* o, long long t0,
                                        int lo, int hi, int h, int H)
{
    if (use_tma) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int r = 32 * t.half + i;
            stage16(stg + r * 256 + 2 * t.L, __uint_as_float(dd[i]), static_cast<const TO*>(nullptr));
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

// S^T <- S0^T (row v of S^T is column v of S0), zeros, or (identity) the
// unit matrix.  This thread: 64 channels of its TMEM lane.
__device__ __forceinline__ void state_load(const Lane& t, uint32_t tmem, const float* S0,
                                           long long sbase, bool identity = false)
{
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int c = 64 * t.half + 32 * jb + i;
            const float x = identity ? (c == t.L ? 1.f : 0.f)
                                     : (S0 ? S0[sbase + (long long)c * kD + t.L] : 0.f);
            r[i] = __float_as_uint(x);
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
// MMA warp.

struct FrontDescs {
    uint64_t GA, GB, WA, WB;
    uint32_t id_g, id_w;
};

// Base descriptors (K-major, 128-byte swizzle); a K step of 32 bytes advances
// the start address field (16-byte units) by 2 inside a swizzle row, and the
// tf32 tiles move to the next 32-channel group every four steps.  gk_off is
// where the (e^G K)^T tile lives.
__device__ __forceinline__ FrontDescs make_front_descs(uint8_t* sm, uint32_t gk_off)
{
    FrontDescs D;
    D.id_g = make_idesc_tf32(128, 64);                  // [Kr; Qr] Kc^T
    D.id_w = make_idesc_f16(128, 64, false, false);     // (e^G K)^T T^T
    D.GA = make_sdesc(smem_u32(sm + OFF_A), 16, 1024, kSwizzle128B);
    D.GB = make_sdesc(smem_u32(sm + OFF_KC), 16, 1024, kSwizzle128B);
    D.WA = make_sdesc(smem_u32(sm + gk_off), 16, 1024, kSwizzle128B);
    D.WB = make_sdesc(smem_u32(sm + OFF_T16), 16, 1024, kSwizzle128B);
    return D;
}

// The front products of one step, after B_OPS: the Gram, then (after the
// solve) W^T.  Called by the whole MMA warp.  Returns false if a wait gave up.
__device__ __forceinline__ bool mma_front(const Ctx& X, uint32_t tmem, const FrontDescs& D,
                                          int step)
{
    // Gram: [Kr; Qr] (M = 128) x Kc^T (N = 64), K = 128 channels in 16 tf32 steps.
#pragma unroll
    for (int s = 0; s < 16; ++s)
        mma_ss_tf32(tmem + TM_G, D.GA + (s >> 2) * (16384 >> 4) + (s & 3) * 2,
                    D.GB + (s >> 2) * (8192 >> 4) + (s & 3) * 2, D.id_g, s > 0);
    mma_commit(&X.bar[B_MMA_G]);
    if (!warp_wait(X, B_T, step)) return false;
    tc_fence_after();
    // W^T = (e^G K)^T T^T: A = (e^G K)^T [ch][i], B = T [r][i], K = 64 tokens.
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_ss(tmem + TM_W, D.WA + 2 * s, D.WB + 2 * s, D.id_w, s > 0);
    mma_commit(&X.bar[B_MMA_W]);
    return true;
}

// [U^T | O^T] = S^T [-W^T | (e^G Q)^T] ;  U^T += V^T T^T.  Shared-memory
// addresses: wt = -W^T with (e^G Q)^T 16 KB after it, t16 = T (fp16),
// vtile = the fp16 v tile.
__device__ __forceinline__ void mma_back_c(uint32_t tmem, uint32_t wt, uint32_t t16, uint32_t vtile,
                                           bool with_v = true)
{
    const uint32_t id_cv = make_idesc_f16(128, 64, true, false);     // V^T T^T
    const uint32_t id_mn128 = make_idesc_f16(128, 128, false, true); // S^T x [-W^T | (e^G Q)^T]
    const uint64_t dWQ = make_sdesc(wt, BLK_QG - BLK_WT, 1024, kSwizzle128B);
    const uint64_t dV = make_sdesc(vtile, 8192, 1024, kSwizzle128B);
    const uint64_t dT16 = make_sdesc(t16, 16, 1024, kSwizzle128B);
#pragma unroll
    for (int s = 0; s < 8; ++s) mma_ts(tmem + TM_C, tmem + TM_SB + s * 8, dWQ + 128 * s, id_mn128, s > 0);
    if (!with_v) return;      // v = 0: U^T = -S^T W^T
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

// ---------------------------------------------------------------------------
// The split consumer's form of the state decay, in two halves: the fp16 copy
// (the A operand of the step's first product, on the chain) and the decay of
// the fp32 state in place (during the first product, which does not read it).

// S^T fp16 copy into columns sb; when `snap` is not null the state (the state
// at the chunk start) is also stored there ([d_k][d_v] fp32).  This thread: 64
// channels of its TMEM lane.  No barrier.
__device__ __forceinline__ void state_copy_f16(const Lane& t, uint32_t tmem, uint32_t sb, float* snap)
{
    const int c0 = 64 * t.half;
    uint32_t r0[32], r1[32], b[16];
    tmem_ld32(tmem + t.lane_base + TM_S + c0, r0);
    tmem_ld32(tmem + t.lane_base + TM_S + c0 + 32, r1);
    tmem_ld_wait();
    if (snap != nullptr) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            snap[(long long)(c0 + i) * kD + t.L] = __uint_as_float(r0[i]);
            snap[(long long)(c0 + 32 + i) * kD + t.L] = __uint_as_float(r1[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
        b[i] = pack_f16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
    tmem_st16(tmem + t.lane_base + sb + (c0 >> 1), b);
#pragma unroll
    for (int i = 0; i < 16; ++i)
        b[i] = pack_f16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
    tmem_st16(tmem + t.lane_base + sb + (c0 >> 1) + 16, b);
    tmem_st_wait();
}

// S^T <- S^T Diag(e^{G_last}) in place.  No barrier.
__device__ __forceinline__ void state_scale(const Lane& t, uint32_t tmem, const float* gl)
{
#pragma unroll 1
    for (int jb = 0; jb < 4; ++jb) {
        const int c0 = 64 * t.half + 16 * jb;
        uint32_t r[16];
        tmem_ld16(tmem + t.lane_base + TM_S + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * gl[c0 + i]);
        tmem_st16(tmem + t.lane_base + TM_S + c0, r);
    }
    tmem_st_wait();
}

}  // namespace tc
}  // namespace kda
