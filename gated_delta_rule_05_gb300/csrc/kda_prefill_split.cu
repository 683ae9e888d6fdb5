// kda_prefill_split.cu -- the producer / consumer tensor-core prefill for
// batches with few (sequence, head) units (bf16 q/k/v, d_k = d_v = 128).
//
// Why.  A chunk step of the chunkwise form ("Kimi 모델 분석", rlaope.github.io,
// section "순환을 GPU에 올리기") is a chain of dependent phases, and only the
// state carries from one chunk to the next.  Most of the chain (gate prep, the
// Gram products, the UT solve, W: the front phases of kda_tc_chunk.cuh) does
// not involve the state at all, so with one CTA per unit a batch of a few long
// sequences keeps only a few SMs busy, each waiting on its own chain.  Here the
// front phases of every chunk run on producer CTAs spread over the rest of the
// GPU, and the CTA that owns a unit's state (its consumer) runs only the back
// phases: state decay, U, O and the state update, about a fifth of the chain.
//
// Grid: one cooperative launch of exactly one CTA per SM (every CTA resident,
// so CTAs may wait on one another).  CTA b < U is the consumer of unit b (the
// b-th (sequence, head) pair, sequences longest first); the others are
// producers.  All CTAs have the same 320 threads: warp 0 moves data, warp 1
// issues the tensor-core products, warps 2..9 are the compute group.
//
// Hand-over.  Producers claim jobs (chunk c of unit u) from a 64-bit counter
// in chunk-major order (job j = c U + u) and write the chunk's back-phase
// operands (-W^T, (e^G Q)^T, P, Ktil^T, T as fp16 tiles in the 128-byte
// swizzled layout of the MMA descriptors, and e^{G_last}), staged in shared
// memory, into slot c mod R of the unit's ring in the workspace with bulk
// copies; a chunk whose decay span needs two passes fills two step blocks.
// The producer's data-movement warp then publishes the slot with a release
// store of full[u][slot] = 2 (c + 1) + (passes - 1).  The consumer's loader
// polls that word with relaxed loads and, once it shows the chunk, issues an
// acquire fence (the relaxed load and the fence form an acquire pattern that
// synchronises with the release store) and a proxy fence, then copies each
// step block into one of two shared-memory stages with one bulk copy.  The
// consumer raises consumed[u] to c + 1 with a relaxed reduction once the copy
// has landed (see the MMA warp for why not a release); a producer writes a
// slot only after an acquire of consumed[u] shows that the chunk R places
// earlier has left it.
//
// Progress.  Jobs are claimed in order and every job depends only on jobs of
// earlier chunks, and a producer publishes a job before it waits for the slot
// of its next one; the earliest unfinished job therefore always runs, so the
// launch cannot deadlock while every CTA is resident.  Every wait is bounded
// in time (about two seconds): one that gives up sets bit 1 of the workspace's
// timeout word and the kernel's abort word (which the work-list kernel clears
// before the launch), every other CTA polling a global flag sees the abort and
// stops, and each CTA waits for its own copies in flight and frees its tensor
// memory before it exits.
//
// Test hook.  With KDA_TEST_STARVE_CONSUMERS set in the environment, the
// launch runs the abort path on purpose: the producers exit at once without
// publishing anything.  The consumers' waits then run out after their usual
// limit (about two seconds), the timeout bit and the abort word are set,
// every CTA drains and exits, and o and S_final are not written.  It exists
// for the test of that path only.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>

#include "kda_internal.cuh"
#include "kda_tc_chunk.cuh"

namespace kda {

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn();
bool tc_make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int H,
                 long long T, int box_x, CUtensorMapSwizzle swz);

namespace {

using namespace tc;

constexpr int kThreads = 320;

// Consumer shared memory (from the same 1024-aligned base; the descriptor,
// barrier and misc areas are those of the front map).
constexpr uint32_t kStage = (uint32_t)kSplitStepBytes;   // one step block, 65 KB
constexpr uint32_t C_V0 = 2 * kStage;                    // four v tiles, 16 KB each
constexpr int kVBufs = 4;
constexpr int kVAhead = 2;                               // v tiles are loaded 2 chunks ahead
constexpr uint32_t C_OST = C_V0 + kVBufs * 16384;        // O staging [64][128] bf16
constexpr uint32_t kConsumerEnd = C_OST + 16384;
static_assert(kBlkBytes <= kStage && kStage % 1024 == 0, "step block layout");
static_assert(kConsumerEnd <= OFF_DESC, "consumer map overlaps the bookkeeping area");

// A producer's job, written by its data-movement warp.
struct JobDesc {
    long long bos, eos;
    int32_t u, c, h, npass;
    int32_t terminate, pad;
};
constexpr uint32_t OFF_JOB = OFF_Y;        // 2 JobDesc (unused by the front phases)
static_assert(OFF_JOB + 2 * sizeof(JobDesc) <= OFF_GL, "job area overflows");
// The producer's operand tiles are staged in the front map's tiles (-W^T,
// (e^G Q)^T, P, Ktil^T, T) and sent to the ring with bulk copies (e^{G_last}
// from OFF_GL): written straight from registers, each warp store of the
// swizzled tiles would touch 32 different lines.  The (e^G K)^T tile takes
// the v tile's place (a producer has no v), so the q / k / g tiles are free
// for the next job's load as soon as pass B is done.
constexpr uint32_t P_GK = OFF_V;
// The token range (cu[n], cu[n + 1]) of each sequence, by rank, read once
// from cu and order so that a claim costs one atomic.
constexpr uint32_t P_SEQ = kSmemUsed;
constexpr uint32_t kSplitSmemBytes = kSmemBytes + kSplitMaxSeqs * 8;
static_assert(P_SEQ % 8 == 0, "sequence table alignment");

// Polls a global flag until pred(value) holds.  Returns false after about
// kWaitLimit cycles (recording the timeout for the caller and the abort for
// the other CTAs), or at once when another CTA has already given up.
// ACQ = false polls with relaxed loads: an acquire load also waits for the
// polling warp's own bulk copies still in flight, which the consumer's loader
// must not do (see there).
template <bool ACQ = true, typename Pred>
__device__ __forceinline__ bool poll_flag(const Ctx& X, const int32_t* flag, Pred pred,
                                          int32_t* seen)
{
    const long long t0 = clock64();
    for (int i = 0;; ++i) {
        const int32_t v = ACQ ? ld_acquire_gpu(flag) : ld_relaxed_gpu(flag);
        if (pred(v)) {
            *seen = v;
            return true;
        }
        if ((i & 31) == 31) {
            if (ld_relaxed_gpu(X.ws_abort) != 0) return false;
            if (clock64() - t0 > kWaitLimit) {
                atomicOr(X.ws_err, 2);
                atomicExch(X.ws_abort, 1);
                return false;
            }
        }
        __nanosleep(40);
    }
}

__device__ __forceinline__ bool global_abort(const Ctx& X)
{
    return ld_relaxed_gpu(X.ws_abort) != 0;
}

// ------------------------------------------------------------- consumer
// SEG: a segmented launch (kda_prefill_segmented); the plain instantiations
// carry none of its bookkeeping.
template <typename TO, bool SEG>
__device__ __forceinline__ void consumer(const Ctx& X, uint32_t tmem, int warp, int lane,
                                         const CUtensorMap* tm_v, const CUtensorMap* tm_o,
                                         const float* S0, const int32_t* cu, const int32_t* ws,
                                         long long total_tokens, int H, TO* o, float* S_final,
                                         int U, int R, int32_t* flags, const uint8_t* ring,
                                         const SnapArgs& snap, const SegArgs& seg,
                                         const CUtensorMap* tm_aux0, const CUtensorMap* tm_aux1)
{
    uint8_t* sm = X.sm;
    const int u = blockIdx.x;
    int rank = u / H, h = u % H;
    long long bos = 0, eos = total_tokens;
    int n = 0;
    if (cu != nullptr) {
        n = ws[kWsHeaderBytes / sizeof(int32_t) + rank];
        bos = cu[n];
        eos = cu[n + 1];
    }
    // Segmented launch (one sequence): this unit's segment, its mode (0: the
    // first segment, from S0 into o; 1: a later segment from S = 0 into the
    // local outputs; 2: its identity run, v = 0 from S = I) and its ring group
    // (segment, head), which the local and identity units share.
    int mode = 0, group = u, groups = U;
    __half* o_aux = nullptr;
    float* s_dst = S_final;
    long long sdst_base = 0;
    if (SEG) {
        const SegUnit su = seg_unit(u, H);
        h = su.h;
        mode = su.mode;
        group = su.g * H + su.h;
        groups = seg.G * H;
        bos = (long long)su.g * seg.seg_chunks * kC;
        eos = bos + (long long)seg.seg_chunks * kC;
        if (eos > total_tokens) eos = total_tokens;
        if (mode > 0) o_aux = seg.o_aux + (size_t)(mode - 1) * total_tokens * H * kD;
        s_dst = seg.st_aux + (size_t)(mode == 2 ? seg.G : 0) * H * kD * kD;
        sdst_base = ((long long)su.g * H + h) * kD * kD;
    }
    const int nch = (int)((eos - bos + kC - 1) / kC);
    const long long sbase = ((long long)n * H + h) * kD * kD;
    if (!SEG) sdst_base = sbase;
    const bool with_v = !SEG || mode != 2;
    const int32_t* full = flags + (size_t)group * R;
    int32_t* consumed = flags + (size_t)groups * R + u;
    const uint8_t* uring = ring + (size_t)group * R * 2 * kStage;

    if (warp == 0) {
        // ------------------------------------------------------ loader
        if (lane != 0) return;
        tma_prefetch_desc(tm_v);
        int step = 0, issued_st[2] = {0, 0}, issued_v[kVBufs] = {0, 0, 0, 0};
        bool ok = true;
        // v tile of chunk cv into buffer cv % 4, once chunk cv - 4 has left it.
        auto issue_v = [&](int cv) -> bool {
            const int vb = cv & (kVBufs - 1);
            if (cv >= kVBufs && !wait_bar(X, B_SV_EMPTY0 + vb, (cv - kVBufs) / kVBufs)) return false;
            const long long tv = bos + (long long)cv * kC;
            mbar_arrive_expect_tx(&X.bar[B_SV_FULL0 + vb], 16384);
            tma_load_2d(sm + C_V0 + vb * 16384, tm_v, h * kD, (int32_t)tv, &X.bar[B_SV_FULL0 + vb]);
            tma_load_2d(sm + C_V0 + vb * 16384 + 8192, tm_v, h * kD + 64, (int32_t)tv,
                        &X.bar[B_SV_FULL0 + vb]);
            ++issued_v[vb];
            return true;
        };
        for (int cv = 0; cv < kVAhead && cv < nch && with_v; ++cv) issue_v(cv);
        for (int c = 0; c < nch && ok; ++c) {
            if (with_v && c + kVAhead < nch && !issue_v(c + kVAhead)) { ok = false; break; }
            const int slot = c % R;
            int32_t val = 0;
            // Relaxed polls: an acquire load would also wait for this warp's
            // copy of the previous chunk, still in flight, and so run the two
            // stages one after the other; where copies are slow every step
            // then took a whole copy.  The slot was complete before its flag
            // was stored (the producer's bulk stores had completed and been
            // fenced before the release store).  The acquire fence after the
            // poll that saw the flag makes the poll an acquire: the
            // producer's writes happen before this thread's later accesses,
            // and the proxy fence extends that order to the bulk copies below.
            ok = poll_flag<false>(X, full + slot, [&](int32_t v) { return (v >> 1) == c + 1; }, &val);
            if (!ok) break;
            fence_acquire_gpu();
            fence_proxy_async_global();        // the bulk copies below read what the producer wrote
            const int npass = (val & 1) + 1;
            const long long t0 = bos + (long long)c * kC;
            const int len = (eos - t0 < kC) ? (int)(eos - t0) : kC;
            for (int p = 0; p < npass; ++p) {
                const int s = step & 1;
                if (step >= 2 && !wait_bar(X, B_ST_EMPTY0 + s, (step - 2) >> 1)) { ok = false; break; }
                StepDesc d;
                d.t0 = (int32_t)t0;
                d.len = len;
                d.lo = (npass == 1) ? 0 : (p == 0 ? 0 : 32);
                d.hi = (npass == 1) ? len : (p == 0 ? min(32, len) : len);
                d.first_pass = (p == 0);
                d.last_pass = (p == npass - 1);
                d.last_step = (c == nch - 1) && (p == npass - 1);
                d.chunk = c;
                X.desc[s] = d;
                mbar_arrive_expect_tx(&X.bar[B_ST_FULL0 + s], kBlkBytes);
                // Four copies of a quarter each: one copy of the whole block
                // streamed at about 24 bytes per cycle.
                static_assert(kBlkBytes % 64 == 0, "quarters of 16-byte multiples");
#pragma unroll
                for (int qb = 0; qb < 4; ++qb)
                    bulk_load(sm + s * kStage + qb * (kBlkBytes / 4),
                              uring + ((size_t)slot * 2 + p) * kStage + qb * (kBlkBytes / 4),
                              kBlkBytes / 4, &X.bar[B_ST_FULL0 + s]);
                ++issued_st[s];
                ++step;
            }
        }
        if (!ok) {
            // Stop the other warps and let the copies already issued land.
            atomicExch(&X.misc->abort, 1);
            for (int s = 0; s < 2; ++s)
                if (issued_st[s]) mbar_wait(&X.bar[B_ST_FULL0 + s], (issued_st[s] - 1) & 1, 1ll << 28);
            for (int vb = 0; vb < kVBufs; ++vb)
                if (issued_v[vb]) mbar_wait(&X.bar[B_SV_FULL0 + vb], (issued_v[vb] - 1) & 1, 1ll << 28);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        // The whole warp runs this loop; the issue helpers elect one lane.
        if (nch == 0) return;
        for (int step = 0;; ++step) {
            if (!warp_wait(X, B_OPS, step)) break;
            tc_fence_after();
            const StepDesc d = X.desc[step & 1];
            const uint32_t blk = smem_u32(sm + (step & 1) * kStage);
            const int vb = d.chunk & (kVBufs - 1);
            // The compute group saw this block land: the ring slot is free
            // once the chunk's last block is here.  (A reduction rather than
            // a store: it is performed at L2 at once, so waiting producers
            // see the free slot promptly.  Relaxed: the bulk copies that read
            // the slot have completed before this point, so nothing the
            // producer writes afterwards can reach them.  A release form,
            // which the PTX memory model would also order formally, measured
            // slower at 1M tokens x 32 heads: 27 % here, where it waits for
            // the warp's products in flight; 46 % from a compute thread; 6 %
            // from an eleventh warp that did nothing else.)
            if (d.last_pass && lane == 0) red_max_relaxed_gpu(consumed, d.chunk + 1);
            mma_back_c(tmem, blk + BLK_WT, blk + BLK_T16, smem_u32(sm + C_V0 + vb * 16384), with_v);
            mma_commit(&X.bar[B_MMA_C]);
            if (d.last_pass && with_v) mma_commit(&X.bar[B_SV_EMPTY0 + vb]);
            if (!warp_wait(X, B_U, step)) break;
            tc_fence_after();
            mma_back_os(tmem, blk + BLK_P);
            mma_commit(&X.bar[B_MMA_OS]);
            mma_commit(&X.bar[B_ST_EMPTY0 + (step & 1)]);
            if (d.last_step) break;
        }
    } else {
        // ------------------------------------------------ compute group
        // Per step, on the chain: the previous step's O^T and the state read
        // from tensor memory, the fp16 copy of the state (then the first
        // product may start), U^T to fp16 (then the second).  While the first
        // product runs: the previous O to o (staged, one TMA store) and the
        // decay of the state in place; while the second runs, the next
        // chunk's v tile to fp16.
        const Lane t = make_lane(threadIdx.x - 64, warp, lane);
        const int seq_off = (cu != nullptr && snap.interval > 0) ? snap.offsets[n] : 0;
        state_load(t, tmem, mode == 0 ? S0 : nullptr, sbase, mode == 2);
        bool alive = nch > 0;
        StepDesc prev;
        prev.t0 = 0;
        prev.lo = prev.hi = 0;
        int step = 0;
        auto store_prev_o = [&](const uint32_t (&dd)[32]) {
            if (SEG && o_aux != nullptr) {   // a later segment's run: fp16, through its own map
                const bool tma_aux = prev.lo == 0 && prev.hi == kC;
                o_store<__half>(t, dd, tma_aux, mode == 1 ? tm_aux0 : tm_aux1, sm + C_OST, o_aux,
                                (long long)prev.t0, prev.lo, prev.hi, h, H);
                return;
            }
            const bool tma_out = (sizeof(TO) == 2) && prev.lo == 0 && prev.hi == kC;
            o_store<TO>(t, dd, tma_out, tm_o, sm + C_OST, o, (long long)prev.t0, prev.lo, prev.hi,
                        h, H);
        };
        // The v tile of chunk cv to fp16, once it has landed.
        auto convert_v = [&](int cv) -> bool {
            const int vb = cv & (kVBufs - 1);
            if (!group_wait(X, B_SV_FULL0 + vb, cv / kVBufs)) return false;
            v_tile_to_f16(sm + C_V0 + vb * 16384, t.ct);
            fence_proxy_async_smem();
            return true;
        };
        if (alive && with_v) alive = convert_v(0);
        while (alive) {
            const int s = step & 1;
            if (!group_wait(X, B_ST_FULL0 + s, step >> 1)) { alive = false; break; }
            const StepDesc d = X.desc[s];
            uint32_t dd[32];
            if (step > 0 && !group_wait(X, B_MMA_OS, step - 1)) { alive = false; break; }
            tc_fence_after();
            if (step > 0) o_load(t, tmem, dd);
            state_copy_f16(t, tmem, TM_SB,
                           d.first_pass ? snapshot_at(snap, d.chunk, eos - bos, seq_off, H, h)
                                        : nullptr);
            tc_fence_before();
            if (t.ct == 0) bulk_wait_group_read0();   // the O staging is free again
            group_sync();
            if (t.ct == 0) mbar_arrive(&X.bar[B_OPS]);
            if (step > 0) store_prev_o(dd);
            prev = d;
            state_scale(t, tmem, reinterpret_cast<const float*>(sm + s * kStage + BLK_GL));
            if (!group_wait(X, B_MMA_C, step)) { alive = false; break; }
            tc_fence_after();
            u_to_f16(t, tmem);
            tc_fence_before();
            group_sync();
            if (t.ct == 0) mbar_arrive(&X.bar[B_U]);
            if (with_v && d.last_pass && d.chunk + 1 < nch && !convert_v(d.chunk + 1)) { alive = false; break; }
            ++step;
            if (d.last_step) break;
        }
        if (alive && step > 0 && group_wait(X, B_MMA_OS, step - 1)) {
            tc_fence_after();
            uint32_t dd[32];
            o_load(t, tmem, dd);
            tc_fence_before();
            if (t.ct == 0) bulk_wait_group_read0();
            group_sync();
            store_prev_o(dd);
        }
        if (t.ct == 0) bulk_wait_group0();               // the last O store has landed
        // (A wait that gave up has set the abort flag; a unit without chunks
        // stores its S0.)
        if (!*reinterpret_cast<volatile int32_t*>(&X.misc->abort)) {
            if (s_dst) state_store(t, tmem, s_dst, sdst_base);
            float* last = snapshot_at(snap, nch, eos - bos, seq_off, H, h);
            if (last) state_store(t, tmem, last, 0);
        }
    }
}

// ------------------------------------------------------------- producer
template <typename TO, bool FUSED, bool SEG>
__device__ __forceinline__ void producer(const Ctx& X, uint32_t tmem, int warp, int lane,
                                         const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                         const CUtensorMap* tm_g, const float* beta,
                                         const int32_t* cu, int32_t* ws, long long total_tokens,
                                         int H, int U, int R, int32_t* flags, uint8_t* ring,
                                         const GateArgs& gate, const SegArgs& seg)
{
    // Ring groups: one per consumer unit, or (segmented) one per segment and
    // head, read by that segment's one or two consumer units.
    const int groups = SEG ? seg.G * H : U;
    uint8_t* sm = X.sm;
    JobDesc* jd = reinterpret_cast<JobDesc*>(sm + OFF_JOB);
    if (warp == 0) {
        // ---------------------------------------------- data movement
        if (lane == 0) {
            tma_prefetch_desc(tm_q);
            tma_prefetch_desc(tm_k);
            tma_prefetch_desc(tm_g);
        }
        float* sBin = reinterpret_cast<float*>(sm + OFF_BIN);
        const long long maxlen = (cu != nullptr) ? ws[kWsMaxLenWord] : total_tokens;
        // Segmented: jobs in order of the chunk index within the segment, so
        // that every segment's chain starts at once.
        const long long total_jobs = SEG ? (long long)seg.G * H * seg.seg_chunks
                                         : (long long)U * ((maxlen + kC - 1) / kC);
        unsigned long long* counter = reinterpret_cast<unsigned long long*>(ws + kWsJobWord);
        const int32_t* order = ws + kWsHeaderBytes / sizeof(int32_t);
        int2* seq_tab = reinterpret_cast<int2*>(sm + P_SEQ);
        if (cu != nullptr) {
            for (int r = lane; r < U / H; r += 32) {
                const int n = order[r];
                seq_tab[r] = make_int2(cu[n], cu[n + 1]);
            }
            __syncwarp();
        }
        // Publishes job jc's slot once the compute group has written it.
        auto publish = [&](int jc) -> bool {
            if (!wait_bar(X, B_JOB_DONE, jc)) return false;
            const JobDesc& j = jd[jc & 1];
            // The release store orders the slot's contents before the flag:
            // the compute group's bulk stores completed and were fenced to
            // the generic proxy before its CTA-scope hand-over (JOB_DONE).
            st_release_gpu(flags + (size_t)j.u * R + j.c % R, 2 * (j.c + 1) + (j.npass - 1));
            return true;
        };
        int jc = 0, issued = 0;
        bool ok = true;
        for (;; ++jc) {
            if (jc > 0) {
                if (lane == 0) ok = wait_bar(X, B_QKG_EMPTY, jc - 1);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            long long bos = 0, eos = 0;
            int uu = -1, c = 0, hh = 0;
            if (lane == 0) {
                for (;;) {
                    const long long j = (long long)atomicAdd(counter, 1ull);
                    if (j >= total_jobs || global_abort(X)) {
                        uu = -1;
                        break;
                    }
                    if (SEG) {
                        c = (int)(j / ((long long)seg.G * H));
                        uu = (int)(j % ((long long)seg.G * H));     // the group: segment, head
                        hh = uu % H;
                        bos = (long long)(uu / H) * seg.seg_chunks * kC;
                        eos = bos + (long long)seg.seg_chunks * kC;
                        if (eos > total_tokens) eos = total_tokens;
                    } else {
                        c = (int)(j / U);
                        uu = (int)(j % U);
                        hh = uu % H;
                        if (cu != nullptr) {
                            const int2 se = seq_tab[uu / H];
                            bos = se.x;
                            eos = se.y;
                        } else {
                            bos = 0;
                            eos = total_tokens;
                        }
                    }
                    if ((long long)c * kC < eos - bos) break;   // else: this unit has no chunk c
                }
            }
            uu = __shfl_sync(0xffffffffu, uu, 0);
            if (uu < 0) {
                if (lane == 0) {
                    jd[jc & 1].terminate = 1;
                    mbar_arrive(&X.bar[B_QKG_FULL]);       // wakes the compute group
                }
                break;
            }
            c = __shfl_sync(0xffffffffu, c, 0);
            hh = __shfl_sync(0xffffffffu, hh, 0);
            bos = __shfl_sync(0xffffffffu, bos, 0);
            eos = __shfl_sync(0xffffffffu, eos, 0);
            const long long t0 = bos + (long long)c * kC;
            // The tiles are requested first; the barrier's single arrival
            // follows once beta (and A) are in shared memory, so the phase
            // completes only when both have landed.
            if (lane == 0) {
                mbar_expect_tx(&X.bar[B_QKG_FULL], 2 * 16384 + 32768);
                tma_load_2d(sm + OFF_Q, tm_q, hh * kD, (int32_t)t0, &X.bar[B_QKG_FULL]);
                tma_load_2d(sm + OFF_K, tm_k, hh * kD, (int32_t)t0, &X.bar[B_QKG_FULL]);
                tma_load_2d(sm + OFF_G, tm_g, hh * kD, (int32_t)t0, &X.bar[B_QKG_FULL]);
                ++issued;
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = lane * 2 + j;
                const long long tt = t0 + r;
                sBin[r] = (tt < eos) ? beta[tt * H + hh] : 0.f;
            }
            if (FUSED)   // the head's A row, read by gate prep (like beta)
                reinterpret_cast<float4*>(sm + OFF_AH)[lane] =
                    reinterpret_cast<const float4*>(gate.A + (long long)hh * kD)[lane];
            __syncwarp();
            if (lane == 0) {
                JobDesc& j = jd[jc & 1];
                j.bos = bos;
                j.eos = eos;
                j.u = uu;
                j.c = c;
                j.h = hh;
                j.npass = 1;
                j.terminate = 0;
                mbar_arrive(&X.bar[B_QKG_FULL]);
                if (jc > 0) ok = publish(jc - 1);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
        }
        if (lane == 0) {
            if (ok && jc > 0) ok = publish(jc - 1);
            // On abort, let the copies already issued land before the CTA exits.
            if (!ok || X.misc->abort) {
                atomicExch(&X.misc->abort, 1);
                if (issued) mbar_wait(&X.bar[B_QKG_FULL], (issued - 1) & 1, 1ll << 28);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        // The whole warp runs this loop; the issue helpers elect one lane.
        const FrontDescs D = make_front_descs(sm, P_GK);
        for (int step = 0;; ++step) {
            if (!warp_wait(X, B_OPS, step)) break;
            tc_fence_after();
            if (X.desc[step & 1].last_step) break;     // no more jobs
            if (!mma_front(X, tmem, D, step)) break;
        }
    } else {
        // ------------------------------------------------ compute group
        const Lane t = make_lane(threadIdx.x - 64, warp, lane);
        const int ct = t.ct;
        const int32_t* consumed = flags + (size_t)groups * R;
        int step = 0;
        // A job's operand tiles go to its ring slot with bulk copies issued by
        // four threads in four warps, one per staging point: ct 0 the
        // (e^G Q)^T, Ktil^T and e^{G_last} tiles after pass B, ct 32 P after
        // the Gram readout, ct 64 T after the solve, ct 96 -W^T after the W
        // readout.  (Issued by one thread, a copy could hold that thread, and
        // with it the whole group at its next barrier, while the copies
        // before it drained.)  Each issuer waits for its own copies: for
        // their reads of a staging tile just before the tile is written
        // again, and for their completion before job jc - 1 is handed to
        // the data-movement warp (JOB_DONE, four arrivals) during job jc,
        // once pass B is done.  It is always handed over before job jc
        // writes its own ring slot (a later chunk of the same unit may need
        // job jc - 1).
        const bool issuer = ct == 0 || ct == 32 || ct == 64 || ct == 96;
        auto job_done = [&](int jc_done, int npass_done) {
            bulk_wait_group0();
            fence_proxy_async_global();
            if (ct == 0) jd[jc_done & 1].npass = npass_done;
            mbar_arrive(&X.bar[B_JOB_DONE]);
        };
        int prev_npass = 0;
        for (int jc = 0;; ++jc) {
            if (!group_wait(X, B_QKG_FULL, jc)) break;
            const JobDesc job = jd[jc & 1];
            if (job.terminate) {
                if (issuer && jc > 0) job_done(jc - 1, prev_npass);
                if (ct == 0) {
                    X.desc[step & 1].last_step = 1;
                    mbar_arrive(&X.bar[B_OPS]);        // lets the MMA warp finish
                }
                break;
            }
            const long long t0 = job.bos + (long long)job.c * kC;
            const int len = (job.eos - t0 < kC) ? (int)(job.eos - t0) : kC;
            uint8_t* slot = ring + ((size_t)job.u * R + job.c % R) * 2 * kStage;
            // The slot is free once the consumer has copied out chunk c - R.
            // A first look is issued now and checked after pass B.
            const int32_t want = job.c - R + 1;
            // The group's consumer units (two in a later segment of a
            // segmented launch: the slot is free once both have copied it).
            int cons[2] = {job.u, job.u};
            int ncons = 1;
            if (SEG) ncons = seg_group_consumers(job.u / H, job.u % H, H, cons);
            int32_t seen = want;
            if (ct == 0 && job.c >= R) {
                seen = ld_relaxed_gpu(consumed + cons[0]);
                if (ncons > 1) seen = min(seen, ld_relaxed_gpu(consumed + cons[1]));
            }
            float2 Gq[16];
            PassParams pp;
            if (FUSED) qk_norms(X, t, gate.q_scale);
            const float* sG = reinterpret_cast<const float*>(sm + OFF_G);
            const float* Ah = reinterpret_cast<const float*>(sm + OFF_AH);
            const int npass = gate_prep<FUSED>(X, t, len, sG, Ah, Gq, pp);
            // One pass of the job's front phases into step block p of the
            // slot.  (Two call sites rather than a loop over the passes, so
            // that the running sums are not live through the first pass's
            // solve: a second pass reloads them from the g tile.)
            auto run_pass = [&](int p, const Pass& ps, const float2 (&Gp)[16]) -> bool {
                uint8_t* blk = slot + (size_t)p * kStage;
                if (ct == 0) {
                    X.desc[step & 1].last_step = 0;
                    bulk_wait_group_read0();       // its staging tiles free again
                }
                group_sync();
                pass_factors(X, t, ps, reinterpret_cast<float*>(sm + OFF_GL));
                gram_operands<FUSED, sizeof(TO) == 4>(X, t, ps, Gp, sm + OFF_QG, sm + OFF_KT, sm + P_GK);
                fence_proxy_async_smem();
                group_sync();
                if (p == 0 && jc > 0 && issuer && ct != 0) job_done(jc - 1, prev_npass);
                if (ct == 0) {
                    mbar_arrive(&X.bar[B_OPS]);
                    bool free_slot = true;
                    if (p == 0) {
                        if (jc > 0) job_done(jc - 1, prev_npass);
                        // The consumer raises consumed[u] only after its
                        // copy of chunk c - R has landed in its shared
                        // memory.  The acquire fence turns the relaxed first
                        // look into an acquire (the poll's loads already
                        // are), and the proxy fence orders the bulk stores
                        // below after it.
                        for (int ci = 0; ci < ncons && free_slot && seen < want; ++ci) {
                            int32_t sc = 0;
                            free_slot = poll_flag(X, consumed + cons[ci],
                                                  [&](int32_t v) { return v >= want; }, &sc);
                        }
                        fence_acquire_gpu();
                        fence_proxy_async_global();
                    }
                    // q, k, g and beta are read: the next job may be claimed
                    // and loaded.  (Only now: a producer that waits for a
                    // slot holds no further claim that a consumer may need.)
                    if (p == npass - 1) mbar_arrive(&X.bar[B_QKG_EMPTY]);
                    if (free_slot) {
                        bulk_store(blk + BLK_QG, sm + OFF_QG, 16384);
                        bulk_store(blk + BLK_KT, sm + OFF_KT, 16384);
                        bulk_store(blk + BLK_GL, sm + OFF_GL, 512);
                        bulk_commit_group();
                    } else {
                        atomicExch(&X.misc->abort, 1);   // the group stops at its next wait
                    }
                }
                // Each later issuer orders its copies after ct 0's look at
                // the slot (the group barriers in between) with a proxy
                // fence, and lets its previous copy finish reading the
                // staging tile before the tile is written again.
                if (ct == 32) bulk_wait_group_read0();
                if (!gram_readout(X, t, tmem, ps.lo, ps.hi, step, sm + OFF_P)) return false;
                if (ct == 32) {
                    fence_proxy_async_global();
                    bulk_store(blk + BLK_P, sm + OFF_P, 8192);
                    bulk_commit_group();
                }
                if (ct == 64) bulk_wait_group_read0();
                ut_solve_mma(X, t, sm + OFF_T16);
                if (ct == 64) {
                    fence_proxy_async_global();
                    bulk_store(blk + BLK_T16, sm + OFF_T16, 8192);
                    bulk_commit_group();
                }
                if (ct == 96) bulk_wait_group_read0();
                if (!w_readout(X, t, tmem, step, sm + OFF_WT)) return false;
                if (ct == 96) {
                    fence_proxy_async_global();
                    bulk_store(blk + BLK_WT, sm + OFF_WT, 16384);
                    bulk_commit_group();
                }
                ++step;
                return true;
            };
            const Pass ps0 = select_pass(pp, 0, npass, len);
            const Pass ps1 = select_pass(pp, 1, npass, len);
            if (npass == 2) stash_running_sums(t, const_cast<float*>(sG), Gq);
            bool alive = run_pass(0, ps0, Gq);
            if (alive && npass == 2) {
                float2 G2[16];
                load_running_sums(t, sG, G2);
                alive = run_pass(1, ps1, G2);
            }
            if (!alive) break;
            prev_npass = npass;
        }
        // (After an abort: the copies still reading shared memory land
        // before the CTA exits.)
        if (issuer) bulk_wait_group0();
    }
}

// ------------------------------------------------------------- the kernel
// FUSED: the gate prologue runs in the producers (gate.A not null).  SEG: a
// segmented launch (seg.G > 1).
template <typename TO, bool FUSED, bool SEG>
__global__ void __launch_bounds__(kThreads, 1)
prefill_split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o,
                     const __grid_constant__ CUtensorMap tm_aux0,
                     const __grid_constant__ CUtensorMap tm_aux1, const float* __restrict__ beta,
                     const float* S0, const int32_t* __restrict__ cu, int32_t* ws,
                     long long total_tokens, int H, TO* __restrict__ o, float* S_final, int U, int R,
                     int32_t* flags, uint8_t* ring, const SnapArgs snap, const GateArgs gate,
                     const SegArgs seg, int test_starve)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Ctx X;
    X.sm = sm;
    X.bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    X.desc = reinterpret_cast<StepDesc*>(sm + OFF_DESC);
    X.misc = reinterpret_cast<Misc*>(sm + OFF_MISC);
    X.ws_err = ws + kWsTimeoutWord;
    X.ws_abort = ws + kWsAbortWord;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (cu != nullptr && ws[kWsErrorWord] != 0) return;   // uniform: every thread returns

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) mbar_init(&X.bar[b], b == B_JOB_DONE ? 4 : 1);
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

    if ((int)blockIdx.x < U)
        consumer<TO, SEG>(X, tmem, warp, lane, &tm_v, &tm_o, S0, cu, ws, total_tokens, H, o, S_final, U,
                     R, flags, ring, snap, seg, &tm_aux0, &tm_aux1);
    else if (!test_starve)
        producer<TO, FUSED, SEG>(X, tmem, warp, lane, &tm_q, &tm_k, &tm_g, beta, cu, ws, total_tokens, H, U,
                        R, flags, ring, gate, seg);

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <typename TO, bool FUSED, bool SEG>
cudaError_t launch_typed(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* S0, const int32_t* cu, int64_t T,
                         int32_t H, void* o, float* S_final, int32_t* ws, const SplitPlan& plan,
                         const SnapArgs& snap, const GateArgs& gate, const SegArgs& seg,
                         cudaStream_t stream)
{
    CUtensorMap mq, mk, mg, mv, mo;
    const bool bf16_out = sizeof(TO) == 2;
    if (!tc_make_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        (bf16_out && !tc_make_map(&mo, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD,
                                  CU_TENSOR_MAP_SWIZZLE_NONE)) ||
        !tc_make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, kD, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tc_make_map(&mg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, T, kD, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tc_make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!bf16_out) mo = mq;
    // A segmented launch's fp16 outputs of the later segments' two runs.
    CUtensorMap ma0 = mq, ma1 = mq;
    if (seg.G > 1 &&
        (!tc_make_map(&ma0, seg.o_aux, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, H, T, kD,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
         !tc_make_map(&ma1, seg.o_aux + (size_t)T * H * kD, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, H,
                      T, kD, CU_TENSOR_MAP_SWIZZLE_NONE)))
        return cudaErrorInvalidValue;
    auto kern = prefill_split_kernel<TO, FUSED, SEG>;
    static bool attr_set = false;   // benign race: every writer stores the same value
    if (!attr_set) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)kSplitSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSplitSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = plan.units + plan.producers;
    if (per_sm < 1 || grid > per_sm * device_sm_count()) return cudaErrorCooperativeLaunchTooLarge;

    int32_t* flags = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(ws) + plan.flags_off);
    uint8_t* ring = reinterpret_cast<uint8_t*>(ws) + plan.ring_off;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSplitSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int test_starve = getenv("KDA_TEST_STARVE_CONSUMERS") != nullptr ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mg, mv, mo, ma0, ma1, beta, S0, cu, ws, (long long)T, (int)H,
                           static_cast<TO*>(o), S_final, (int)plan.units, (int)plan.ring, flags,
                           ring, snap, gate, seg, test_starve);
    if (e != cudaSuccess && debug_enabled())
        fprintf(stderr, "kda: prefill_split launch failed: %s\n", cudaGetErrorString(e));
    return e;
}

}  // namespace

cudaError_t launch_prefill_split(const void* q, const void* k, const void* v,
                                 const float* log_alpha, const float* beta, const float* S0,
                                 const int32_t* cu_seqlens, int32_t num_seqs,
                                 int64_t total_tokens, int32_t H, kda_dtype_t dtype, void* o,
                                 float* S_final, int32_t* ws, const SplitPlan& plan,
                                 const SnapArgs& snap, const GateArgs& gate, const SegArgs& seg,
                                 cudaStream_t stream)
{
    (void)num_seqs;
    const bool fused = gate.A != nullptr;
    if (seg.G > 1) {   // segmented launches take no gate prologue
        if (fused) return cudaErrorInvalidValue;
        if (dtype == KDA_BF16_F32OUT)
            return launch_typed<float, false, true>(q, k, v, log_alpha, beta, S0, cu_seqlens,
                                                    total_tokens, H, o, S_final, ws, plan, snap,
                                                    gate, seg, stream);
        return launch_typed<__nv_bfloat16, false, true>(q, k, v, log_alpha, beta, S0, cu_seqlens,
                                                        total_tokens, H, o, S_final, ws, plan,
                                                        snap, gate, seg, stream);
    }
    if (dtype == KDA_BF16_F32OUT)
        return fused ? launch_typed<float, true, false>(q, k, v, log_alpha, beta, S0, cu_seqlens,
                                                        total_tokens, H, o, S_final, ws, plan, snap,
                                                        gate, seg, stream)
                     : launch_typed<float, false, false>(q, k, v, log_alpha, beta, S0, cu_seqlens,
                                                         total_tokens, H, o, S_final, ws, plan,
                                                         snap, gate, seg, stream);
    return fused ? launch_typed<__nv_bfloat16, true, false>(q, k, v, log_alpha, beta, S0,
                                                            cu_seqlens, total_tokens, H, o, S_final,
                                                            ws, plan, snap, gate, seg, stream)
                 : launch_typed<__nv_bfloat16, false, false>(q, k, v, log_alpha, beta, S0,
                                                             cu_seqlens, total_tokens, H, o,
                                                             S_final, ws, plan, snap, gate, seg,
                                                             stream);
}

}  // namespace kda
