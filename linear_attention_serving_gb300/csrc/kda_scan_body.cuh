// kda_scan_body.cuh -- the sequential chunk scan on tcgen05 tensor cores (the
// device code; kda_scan_tc.cu and kda_fused_tc.cu launch it).
//
// With the record of the prep kernel (G = K_restore^T W, H = K_restore^T U0,
// a_C), one chunk of the scan is
//   S <- Diag(a_C) S + H - G S          (one M = 128 MMA per chunk)
// which is "Kimi K3: the Manos, the Mythos ..." (SemiAnalysis), "FlashKDA 算法"
// K2 (U = INV Diag(beta)(V - K_decay S), S = Diag(a[-1]) S + K_restore^T U)
// with its products regrouped so that only one tensor-core round trip sits on
// the sequential path.  The output O = O0 + Q' S of every chunk is off the
// path: either this kernel stores each chunk's entering state S (bf16) into
// the record and the output kernel (kda_out_tc.cu) forms all outputs in
// parallel afterwards, or (EMIT_O) the block forms its columns' outputs itself
// on warps of their own.
//
// A block owns N = 16, 64 or 128 state columns (columns evolve independently).
// With 256 state columns the extra 128 start from the identity with H = 0:
// they carry the transition M of "Kimi K3 模型结构（7）" eq. (17) for the
// segment pairs.
//
// Chain warps (4 per TPR): thread t of a row group owns state row t (TMEM lane
//   t) and N / TPR of its columns; the fp32 state master lives in registers,
//   its bf16 copy (double buffered) in shared memory is the B operand
//   (MN-major) of the next chunk's MMA; a_C and H are read while the MMA runs.
//   After writing their rows of that operand the chain warps arrive at a named
//   barrier and go on.
// MMA warp: waits at that barrier (a hardware barrier wakes it at once),
//   checks the chunk's stage and issues the chain's MMA (the whole warp runs
//   the issue code, one elected lane issuing, as the output-MMA warp does).
// Output-MMA warp (EMIT_O): once a chunk's chain MMA is issued, issues its
//   output MMA O = Q' S_enter (M = 64) into one of two TMEM accumulators, so
//   that the chain never waits for the output path.
// Producer warp: waits for a chunk's record (its ready flag, when another part
//   of the launch writes it), then streams G, a_C and the block's H slices
//   through a bulk-copy pipeline.
// Q' producer warp (EMIT_O): the same for Q' and the block's O0 slices, through
//   a ring of their own, so that the chain's stages never wait for the output
//   path.
// Output warps (EMIT_O): read O0 from that ring, read an output accumulator,
//   add, store bf16 o.
// Every wait is bounded; on a timeout the block records KDA_DEVERR_TIMEOUT,
// leaves its loops, and frees its TMEM.
#pragma once

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

using namespace tc;

// Block layout for N state columns with TPR threads per state row: warps
// 0 .. 4 TPR - 1 run the chain (warp w: rows 32 (w % 4) .., columns
// (w / 4) N / TPR ..), then the MMA warp, the producer warp and, when the
// block forms the outputs itself (EMIT_O), the output-MMA warp, the Q'
// producer warp and four output warps.
template <int N, int TPR, bool EMIT_O = false>
struct ScanCfg {
    static constexpr int NT = N / TPR;  // state columns per chain thread
    static constexpr int CHAIN_WARPS = 4 * TPR;
    static constexpr int MMA_WARP = CHAIN_WARPS;
    static constexpr int PRODUCER_WARP = CHAIN_WARPS + 1;
    static constexpr int OMMA_WARP = CHAIN_WARPS + 2;
    static constexpr int QPROD_WARP = CHAIN_WARPS + 3;
    static constexpr int OUT_WARP0 = CHAIN_WARPS + 4;
    static constexpr int OUT_WARPS = EMIT_O ? 4 : 0;
    static constexpr int THREADS = 32 * (CHAIN_WARPS + 2 + (EMIT_O ? 2 + OUT_WARPS : 0));
    static constexpr int OPERAND_BAR_THREADS = 32 * (CHAIN_WARPS + 1);  // chain warps + MMA warp
    static_assert(NT % 16 == 0, "a chain thread owns whole 16-column blocks");
};
// Named barrier at which the chain warps hand the next S operand to the MMA
// warp: they arrive without waiting, the MMA warp waits.
constexpr int OPERAND_BAR = 1;
__device__ __forceinline__ void bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// A pipeline stage holds one chunk's G (32 KB, the MMA operand) and its a_C
// and the block's H slices.  With EMIT_O, Q' (the output MMA's A operand) and
// the block's O0 slices ride a ring of their own, freed once that MMA and the
// output warps have read them, so that the stages the chain waits on stay
// small.  Shared memory, from a 1024-byte-aligned base:
//   [G of every stage | Q' + O0 ring slots | 2 S operands | a_C + H of every stage]
// (the operands 1024-byte aligned; the a_C + H areas need 16 bytes).
template <int N, bool EMIT_O = false>
struct Stage {
    static constexpr int NS = N / 16;
    static constexpr int G_BYTES = 32768;                                        // G of one stage
    static constexpr int AC = 0;                                                 // in a stage's a_C + H area
    static constexpr int H = (int)(REC_BF16_SHARED - REC_BF16_AC);               // H slices after a_C
    static constexpr int AH_BYTES = H + NS * (int)REC_BF16_HSLICE;               // a_C + H of one stage
    static constexpr int QO0 = 16384;                                            // O0 slices after Q' in a slot
    static constexpr int QUSED = EMIT_O ? QO0 + NS * (int)REC_BF16_OSLICE : 0;   // bytes copied per slot
    static constexpr int QBYTES = (QUSED + 1023) / 1024 * 1024;                  // one ring slot (1024-aligned)
    static constexpr int QSTAGES = 2;
    static constexpr int SOP = 2 * N * 128;  // one bf16 S operand: 128 rows x N columns
    static constexpr int OCOL = N;           // TMEM: output accumulators at N and 2 N
    static constexpr int NCOLS = EMIT_O ? 256 : (N < 32 ? 32 : N);
    static_assert(H % 16 == 0 && AH_BYTES % 16 == 0, "stage areas keep bulk-copy alignment");
};

template <int N, int STAGES, bool EMIT_O = false>
constexpr size_t scan_tc_smem_bytes() {
    using ST = Stage<N, EMIT_O>;
    return (size_t)STAGES * (ST::G_BYTES + ST::AH_BYTES) + (size_t)ST::QSTAGES * ST::QBYTES + 2 * ST::SOP + 1024;
}

__device__ __forceinline__ float state_init(const ScanArgs &a, int unit, int h, int r, int g) {
    if (a.mode == SCAN_DOCS) {
        if (g >= D) return 0.f;
        return a.init_state ? a.init_state[(((size_t)unit * a.H + h) * D + r) * D + g] : 0.f;
    }
    if (a.phase == 1) return (g >= D && r == g - D) ? 1.f : 0.f;
    return a.s_enter[(((size_t)h * a.n_seg + unit) * D + r) * D + g];
}

__device__ __forceinline__ float state_reset(const ScanArgs &a, int doc, int h, int r, int g) {
    if (g >= D) return 0.f;
    return a.init_state ? a.init_state[(((size_t)doc * a.H + h) * D + r) * D + g] : 0.f;
}

__device__ __forceinline__ uint4 pack8f(const float *f) {
    uint4 u;
    __nv_bfloat162 *b = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    return u;
}

// The bf16 S operand is MN-major (k = state row, the block's N columns
// contiguous): 16 columns with the 32-byte swizzle, 64 with the 128-byte one,
// 128 as two 64-column blocks BLOCK bytes apart.
template <int N>
struct SOp {
    static_assert(N == 16 || N == 64 || N == 128, "S operand layouts exist for 16, 64 and 128 columns");
    static constexpr uint32_t ROW = N == 16 ? 32 : 128;  // bytes per state row of one block
    static constexpr uint32_t SBO = 8 * ROW;              // 8-row group
    static constexpr uint32_t KSTEP = 16 * ROW;           // one K = 16 MMA step
    static constexpr uint32_t BLOCK = 128 * ROW;          // one block of columns (128 state rows)
    static constexpr uint32_t MODE = N == 16 ? SWZ_32B : SWZ_128B;
};

// bf16 pairs of this thread's state row
template <int N>
__device__ __forceinline__ void pack_row(const float *s, uint4 *pk) {
#pragma unroll
    for (int c = 0; c < N / 8; ++c) pk[c] = pack8f(s + 8 * c);
}

// NT packed columns [c16 * 16, c16 * 16 + NT) of row t into the S operand
template <int N, int NT>
__device__ __forceinline__ void write_sop(uint8_t *sop, int t, int c16, const uint4 *pk) {
#pragma unroll
    for (int c = 0; c < NT / 8; ++c) {
        const int cg = 2 * c16 + c;  // 16-byte chunk of the state row, over all N columns
        const int blk = N == 128 ? (cg >> 3) : 0, cb = N == 128 ? (cg & 7) : cg;
        const int sc = N == 16 ? (cb ^ ((t >> 2) & 1)) : (cb ^ (t & 7));
        *reinterpret_cast<uint4 *>(sop + blk * SOp<N>::BLOCK + t * SOp<N>::ROW + sc * 16) = pk[c];
    }
}

// the same columns of row t into the record's S field (32-byte swizzled
// 16-column blocks, block = global 16-column index)
template <int NT>
__device__ __forceinline__ void store_s(char *rec, int blk0, int t, const uint4 *pk) {
#pragma unroll
    for (int blk = 0; blk < NT / 16; ++blk) {
        char *row = rec + REC_BF16_S + (size_t)(blk0 + blk) * REC_BF16_SBLOCK + t * 32;
#pragma unroll
        for (int c = 0; c < 2; ++c) *reinterpret_cast<uint4 *>(row + ((c ^ ((t >> 2) & 1)) << 4)) = pk[2 * blk + c];
    }
}

template <int N>
__device__ __forceinline__ uint64_t sop_desc(const uint8_t *sop) {
    return sdesc_mn(smem_u32(sop), N == 128 ? SOp<N>::BLOCK : SOp<N>::SBO, SOp<N>::SBO, SOp<N>::MODE);
}

// The two 16-byte halves of row r of a 16-column slice (32-byte rows), in
// the order a thread reads them: rows r with (r >> 2) odd read the upper half
// first, so that the eight rows a quarter-warp reads at once cover all 32
// banks instead of half of them twice.  lo = columns 0-7, hi = 8-15.
__device__ __forceinline__ void slice_row_halves(const uint8_t *row, int r, uint4 &lo, uint4 &hi) {
    const int sw = (r & 4) << 2;  // 0 or 16
    const uint4 a = *reinterpret_cast<const uint4 *>(row + sw);
    const uint4 b = *reinterpret_cast<const uint4 *>(row + (sw ^ 16));
    lo = sw ? b : a;
    hi = sw ? a : b;
}

// N bf16 values of row r from consecutive 16-column slices of `rows` rows each
template <int N>
__device__ __forceinline__ void load_slices(const uint8_t *base, int r, int rows, float *out) {
#pragma unroll
    for (int j = 0; j < N; j += 16) {
        uint4 u[2];
        slice_row_halves(base + slice_offset(r, j, rows), r, u[0], u[1]);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u[hf]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(p[e]);
                out[j + 8 * hf + 2 * e] = f.x;
                out[j + 8 * hf + 2 * e + 1] = f.y;
            }
        }
    }
}

// Wait until *flag is set by another block of the same launch, giving up
// after `budget` clock cycles (the launch's budget for waits on other blocks)
// or as soon as the block's abort flag rises; the acquire and the proxy fence
// order the bulk copies that follow after the writes the flag publishes.
__device__ __forceinline__ bool wait_flag(const int *flag, long long budget, const volatile int *abort) {
    const long long t0 = clock64();
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v != 0) break;
        if (*abort || clock64() - t0 > budget) return false;
        __nanosleep(64);
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

template <int N>
__device__ __forceinline__ void tmem_row(uint32_t taddr, float *out) {
#pragma unroll
    for (int j = 0; j < N; j += 16) tmem_ld16(taddr + j, out + j);
    tmem_ld_wait();
}

// One scan block: state columns [16 zc16, 16 zc16 + N) of head h over unit
// `unit` (document or segment).  With `ready` non-null the producer waits,
// before copying chunk c's record, until ready[c * H + h] is set (the record
// is written by other blocks of the same launch).
// CKPT compiles the state checkpoints in (output blocks have them only in
// their own instantiation, so that the default launch keeps its registers).
template <int N, int STAGES, int TPR, bool EMIT_O = false, bool CKPT = !EMIT_O>
__device__ __forceinline__ void scan_block(const ScanArgs &a, int unit, int h, int zc16, uint8_t *smraw,
                                           const int *ready) {
    using ST = Stage<N, EMIT_O>;
    using CF = ScanCfg<N, TPR, EMIT_O>;
    constexpr int NT = CF::NT;
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES], g_bar, sop_bar[2], o_bar[2], oempty_bar[2], drain_bar,
        odrain_bar;
    __shared__ uint64_t qfull_bar[ST::QSTAGES], qfree_bar[ST::QSTAGES];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int col0 = zc16 * 16;
    const bool value_cols = col0 < D;
    // the output kernel needs S, unless this block forms the outputs itself
    const bool emit_s = !EMIT_O && value_cols && a.o && a.phase != 1;
    const Plan &p = a.plan;
    if (plan_failed(p)) return;
    int c0, c1;
    if (a.mode == SCAN_DOCS) {
        if (unit >= p.n_seqs) return;
        plan_doc_range(p, unit, c0, c1);
    } else {
        segment_range(plan_n_chunks(p), a.n_seg, unit, c0, c1);
    }
    const int nchunks = c1 - c0;

    uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    uint8_t *qring = sm + STAGES * ST::G_BYTES;
    uint8_t *sop0 = qring + ST::QSTAGES * ST::QBYTES;
    uint8_t *aharea = sop0 + 2 * ST::SOP;  // a_C + H of every stage
    char *records = (char *)a.records;
    const size_t rec_stride = (size_t)a.H * REC_BF16_BYTES;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], CF::CHAIN_WARPS);  // released by the chain warps once they read it
        }
        mbar_init(&g_bar, 1);
        mbar_init(&drain_bar, 1);
        mbar_init(&odrain_bar, 1);
        // chunk i's chain MMA issued, so its S operand is complete (for the output
        // MMA); two of them alternate, so that a waiter one chunk behind never
        // mistakes a later phase for the one it waits for
        mbar_init(&sop_bar[0], 1);
        mbar_init(&sop_bar[1], 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&o_bar[b], 1);                // output accumulator b written
            mbar_init(&oempty_bar[b], CF::OUT_WARPS > 0 ? CF::OUT_WARPS : 1);  // and read back
        }
        for (int s = 0; s < ST::QSTAGES; ++s) {
            mbar_init(&qfull_bar[s], 1);
            mbar_init(&qfree_bar[s], 1 + CF::OUT_WARPS);  // the output MMA's commit and the output warps
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, ST::NCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_g = tmem_slot;
    const volatile int *abort = &abort_flag;
    const long long flag_budget = p.wait_budget;

    if (warp == CF::PRODUCER_WARP) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            bool timed_out = false;
            const uint32_t bytes = (uint32_t)REC_BF16_SHARED + (value_cols ? (uint32_t)(ST::NS * REC_BF16_HSLICE) : 0u);
            int stage = 0;
            uint32_t ph = 0;
            for (int i = 0; i < nchunks; ++i) {
                // the record first: its flag is read while the stage drains
                if (ready && !wait_flag(ready + (size_t)(c0 + i) * a.H + h, flag_budget, abort)) { timed_out = true; break; }
                if (!mbar_wait_ab(&empty_bar[stage], ph ^ 1u, abort)) { timed_out = true; break; }
                if (*abort) break;
                const char *rec = records + (size_t)(c0 + i) * rec_stride + (size_t)h * REC_BF16_BYTES;
                uint8_t *ah = aharea + stage * ST::AH_BYTES;
                mbar_expect_tx(&full_bar[stage], bytes);
                bulk_g2s(sm + stage * ST::G_BYTES, rec + REC_BF16_G, (uint32_t)ST::G_BYTES, &full_bar[stage]);
                bulk_g2s(ah + ST::AC, rec + REC_BF16_AC, (uint32_t)ST::H, &full_bar[stage]);
                if (value_cols)
                    bulk_g2s(ah + ST::H, rec + REC_BF16_H + (size_t)(col0 / 16) * REC_BF16_HSLICE,
                             (uint32_t)(ST::NS * REC_BF16_HSLICE), &full_bar[stage]);
                issued = i + 1;
                if (++stage == STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            if (timed_out) abort_flag = 1;  // the other warps stop at their next wait
            if (timed_out || *abort) {
                // let the copies this thread started land before the block exits
                for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
                    mbar_wait(&full_bar[i % STAGES], (uint32_t)((i / STAGES) & 1));
                if (timed_out) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            }
        }
    } else if (EMIT_O && warp == CF::QPROD_WARP) {
        // ------------------------------------------------------------ Q' producer
        if (lane == 0) {
            int q_issued = 0;
            bool timed_out = false;
            for (int i = 0; i < nchunks; ++i) {
                if (ready && !wait_flag(ready + (size_t)(c0 + i) * a.H + h, flag_budget, abort)) { timed_out = true; break; }
                const int qs = i % ST::QSTAGES;
                if (!mbar_wait_ab(&qfree_bar[qs], (uint32_t)(((i / ST::QSTAGES) & 1) ^ 1), abort)) { timed_out = true; break; }
                if (*abort) break;
                const char *rec = records + (size_t)(c0 + i) * rec_stride + (size_t)h * REC_BF16_BYTES;
                mbar_expect_tx(&qfull_bar[qs], (uint32_t)ST::QUSED);
                bulk_g2s(qring + qs * ST::QBYTES, rec + REC_BF16_QP, 16384u, &qfull_bar[qs]);
                bulk_g2s(qring + qs * ST::QBYTES + ST::QO0, rec + REC_BF16_O0 + (size_t)(col0 / 16) * REC_BF16_OSLICE,
                         (uint32_t)(ST::NS * REC_BF16_OSLICE), &qfull_bar[qs]);
                q_issued = i + 1;
            }
            if (timed_out) abort_flag = 1;
            if (timed_out || *abort) {
                for (int i = (q_issued > ST::QSTAGES ? q_issued - ST::QSTAGES : 0); i < q_issued; ++i)
                    mbar_wait(&qfull_bar[i % ST::QSTAGES], (uint32_t)((i / ST::QSTAGES) & 1));
                if (timed_out) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            }
        }
    } else if (warp == CF::MMA_WARP) {
        // ------------------------------------------------------------ chain MMAs
        // Chunk i: wait for the chunk's stage (G), then at the operand barrier
        // until every chain warp has written its rows of S_i (or given up), then
        // issue S_i -> G S_i.  The stage wait comes first so that it overlaps the
        // chain's update of the previous chunk.  The chain warps arrive once per
        // chunk, also when they stop, so this warp never waits at a barrier
        // nobody reaches.
        const uint64_t gd0 = sdesc_sw128(smem_u32(sm));
        const uint64_t sd0 = sop_desc<N>(sop0);
        int stage = 0;
        uint32_t ph = 0;
        bool issued_any = false;
        for (int i = 0; i < nchunks; ++i) {
            bool go = true;
            if (lane == 0 && !mbar_wait_ab(&full_bar[stage], ph, abort)) {
                abort_flag = 1;
                go = false;
            }
            bar_sync(OPERAND_BAR, CF::OPERAND_BAR_THREADS);
            if (__shfl_sync(0xffffffffu, (int)(*abort) || !go, 0)) break;
            {
                // the whole warp runs the issue code (one elected lane issues)
                tc_fence_after();
                constexpr uint32_t IDESC = idesc_bf16_f32_bmn(128, N);
                const uint64_t gd = gd0 + (uint64_t)((stage * ST::G_BYTES) >> 4);
                const uint64_t sd = sd0 + (uint64_t)(((i & 1) * ST::SOP) >> 4);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_w(tmem_g, gd + (uint64_t)(((k >> 2) * 16384 + (k & 3) * 32) >> 4),
                               sd + (uint64_t)((k * SOp<N>::KSTEP) >> 4), IDESC, k > 0);
                mma_commit_w(&g_bar);
                __syncwarp();
                if (EMIT_O && lane == 0) mbar_arrive(&sop_bar[i & 1]);
                issued_any = true;
            }
            if (++stage == STAGES) {
                stage = 0;
                ph ^= 1u;
            }
        }
        if (issued_any) {
            // every chain MMA has completed before TMEM is freed, also when the
            // block stopped early
            mma_commit_w(&drain_bar);
            mbar_wait(&drain_bar, 0);
        }
    } else if (EMIT_O && warp == CF::OMMA_WARP) {
        // ------------------------------------------------------------ output MMAs
        // (the whole warp: one elected lane issues)
        const uint64_t sd0 = sop_desc<N>(sop0);
        for (int i = 0; i < nchunks; ++i) {
            const int b = i & 1, qs = i % ST::QSTAGES;
            // chunk i's chain MMA is issued (so its S operand is complete), the
            // output warps have read what chunk i - 2 left in accumulator b, and
            // chunk i's Q' has landed
            const bool fail = !mbar_wait_ab(&sop_bar[b], (uint32_t)((i >> 1) & 1), abort) ||
                              (i >= 2 && !mbar_wait_ab(&oempty_bar[b], (uint32_t)(((i - 2) >> 1) & 1), abort)) ||
                              !mbar_wait_ab(&qfull_bar[qs], (uint32_t)((i / ST::QSTAGES) & 1), abort);
            if (__any_sync(0xffffffffu, fail)) {
                if (lane == 0) abort_flag = 1;
                break;
            }
            tc_fence_after();
            constexpr uint32_t IDO = idesc_bf16_f32_bmn(64, N);
            const uint64_t qd = sdesc_sw128(smem_u32(qring + qs * ST::QBYTES));
            const uint64_t sd = sd0 + (uint64_t)((b * ST::SOP) >> 4);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_bf16_w(tmem_g + ST::OCOL + b * N, qd + (uint64_t)(((k >> 2) * 8192 + (k & 3) * 32) >> 4),
                           sd + (uint64_t)((k * SOp<N>::KSTEP) >> 4), IDO, k > 0);
            mma_commit_w(&o_bar[b]);
            mma_commit_w(&qfree_bar[qs]);  // Q' read
        }
        // every output MMA has completed before TMEM is freed, also when the
        // block stopped early
        if (nchunks > 0) {
            mma_commit_w(&odrain_bar);
            mbar_wait(&odrain_bar, 0);
        }
    } else if (warp < CF::CHAIN_WARPS) {
        // ------------------------------------------------------------ chain warps
        const int t = (warp & 3) * 32 + lane;  // state row == TMEM lane
        const int part = warp >> 2;            // columns [part NT, part NT + NT) of the block
        const int pc = col0 + part * NT;       // first state column of this thread
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const bool segs = a.mode == SCAN_SEGMENTS;
        float s[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) s[j] = state_init(a, unit, h, t, pc + j);
        if (a.mode == SCAN_DOCS && nchunks == 0 && value_cols && a.final_state) {
            float *f = a.final_state + (((size_t)unit * a.H + h) * D + t) * D + pc;
#pragma unroll
            for (int j = 0; j < NT; j += 4) *reinterpret_cast<float4 *>(f + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
        }
        ChunkInfo ci_next;
        if (segs && nchunks > 0) {
            ci_next = plan_chunk(p, c0);
            if (ci_next.flags & CHUNK_FIRST) {
                // a document starts at the segment's first chunk
#pragma unroll
                for (int j = 0; j < NT; ++j) s[j] = state_reset(a, ci_next.doc, h, t, pc + j);
            }
        }
        uint4 pk[NT / 8];  // bf16 copy of this thread's part of the state row entering the chunk
        pack_row<NT>(s, pk);
        write_sop<N, NT>(sop0, t, part * NT / 16, pk);
        fence_async_smem();
        tc_fence_before();
        if (nchunks > 0) bar_arrive(OPERAND_BAR, CF::OPERAND_BAR_THREADS);  // S_0 is written
        const bool write_final = value_cols && a.final_state && a.phase != 1;
        const bool write_ckpt = CKPT && value_cols && a.ckpt && a.phase != 1;
        // one document per chain (SCAN_DOCS): its checkpoints are counted down
        // instead of derived from the chunk table at every chunk
        int ck_left = a.ckpt_ic, ck_j = 0;
        bool ok = true;
        int stage = 0;
        uint32_t ph = 0;
        for (int i = 0; i < nchunks; ++i) {
            const int b = i & 1;
            int doc = unit;
            bool last = i == nchunks - 1;
            bool next_first = false;
            if (segs) {
                const ChunkInfo ci = ci_next;
                if (i + 1 < nchunks) {
                    ci_next = plan_chunk(p, c0 + i + 1);
                    next_first = (ci_next.flags & CHUNK_FIRST) != 0;
                }
                doc = ci.doc;
                last = (ci.flags & CHUNK_LAST) != 0;
            }
            ok = mbar_wait_ab(&full_bar[stage], ph, abort);
            // the entering state of this chunk, for the output kernel
            if (emit_s && ok) store_s<NT>(records + (size_t)(c0 + i) * rec_stride + (size_t)h * REC_BF16_BYTES, pc / 16, t, pk);
            // ---- S <- Diag(a_C) S + H - G S: Diag(a_C) S + H is formed while the
            // chunk's MMA runs (it does not depend on G S)
            const uint8_t *stg = aharea + stage * ST::AH_BYTES;
            float hv[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) hv[j] = 0.f;
            if (ok) {
                const float ac = reinterpret_cast<const float *>(stg + ST::AC)[t];
                if (value_cols) load_slices<NT>(stg + ST::H + slice_offset(0, part * NT, 128), t, 128, hv);
#pragma unroll
                for (int j = 0; j < NT; j += 2) {
                    const float2 r2 = __ffma2_rn(make_float2(ac, ac), make_float2(s[j], s[j + 1]),
                                                 make_float2(hv[j], hv[j + 1]));
                    hv[j] = r2.x;
                    hv[j + 1] = r2.y;
                }
            }
            // operand buffer b ^ 1 (rewritten below) was also read by chunk i - 1's
            // output MMA, which the tensor pipe ran before this chunk's MMA: checked
            // here, while this chunk's MMA runs
            if (EMIT_O && ok && i >= 1 && i + 1 < nchunks)
                ok = mbar_wait_ab(&o_bar[b ^ 1], (uint32_t)(((i - 1) >> 1) & 1), abort);
            ok = ok && mbar_wait_ab(&g_bar, (uint32_t)(i & 1), abort);
            // a warp that gave up skips the update, raises the abort flag, and still
            // arrives at the operand barrier before it stops
            bool good = __all_sync(0xffffffffu, ok) && !*abort;
            if (good) {
                tc_fence_after();
                float d[NT];
                tmem_row<NT>(tmem_g + lane_off + part * NT, d);
#pragma unroll
                for (int j = 0; j < NT; ++j) s[j] = hv[j] - d[j];
                if (write_final && last) {
                    float *f = a.final_state + (((size_t)doc * a.H + h) * D + t) * D + pc;
#pragma unroll
                    for (int j = 0; j < NT; j += 4) *reinterpret_cast<float4 *>(f + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
                }
                if (CKPT && write_ckpt) {
                    // the state after this chunk, when it ends on a checkpoint position
                    // (only a full chunk does; a document's last chunk may be partial)
                    float *f = nullptr;
                    if (!segs) {
                        if (--ck_left == 0) {
                            ck_left = a.ckpt_ic;
                            if (ck_j < a.ckpt_per_seq && (i + 1 < nchunks || plan_chunk(p, c0 + i).len == C)) {
                                const int slot = a.ckpt_slot[(size_t)unit * a.ckpt_per_seq + ck_j];
                                if (slot >= 0 && slot < a.ckpt_n_slots)
                                    f = a.ckpt + (((size_t)slot * a.H + h) * D + t) * D;
                            }
                            ++ck_j;
                        }
                    } else {
                        const ChunkInfo cik = plan_chunk(p, c0 + i);
                        f = ckpt_row(a, cik, c0 + i, h, t);
                    }
                    if (f) {
                        f += pc;
#pragma unroll
                        for (int j = 0; j < NT; j += 4)
                            *reinterpret_cast<float4 *>(f + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
                    }
                }
                if (next_first) {
                    // a document starts at the next chunk: the state restarts there
#pragma unroll
                    for (int j = 0; j < NT; ++j) s[j] = state_reset(a, ci_next.doc, h, t, pc + j);
                }
                pack_row<NT>(s, pk);
                if (i + 1 < nchunks) {
                    write_sop<N, NT>(sop0 + (b ^ 1) * ST::SOP, t, part * NT / 16, pk);
                    fence_async_smem();
                }
            }
            tc_fence_before();
            if (!good && lane == 0) abort_flag = 1;
            __syncwarp();
            if (i + 1 < nchunks) bar_arrive(OPERAND_BAR, CF::OPERAND_BAR_THREADS);  // S_{i+1} (or the stop)
            if (!good) {
                ok = false;
                break;
            }
            // stage i is read (a_C, H here, G by chunk i's MMA, which has completed)
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
            if (++stage == STAGES) {
                stage = 0;
                ph ^= 1u;
            }
        }
        if (!ok) {
            if (lane == 0) {
                abort_flag = 1;
                atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            }
        } else if (a.mode == SCAN_SEGMENTS && a.phase == 1) {
            const int which = value_cols ? 1 : 0;
            const int pc0 = value_cols ? pc : pc - D;
            float *dst = a.pairs + ((((size_t)which * a.H + h) * a.n_seg + unit) * D + t) * D + pc0;
#pragma unroll
            for (int j = 0; j < NT; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
        }
    }
    if (EMIT_O && warp >= CF::OUT_WARP0 && warp < CF::OUT_WARP0 + CF::OUT_WARPS) {
        // ------------------------------------------------------------ output warps
        // M = 64 accumulator: token r sits in lane 32 (r / 16) + r % 16, so the
        // warp of lane quadrant q4 drains tokens 16 q4 .. 16 q4 + 15
        const int q4 = warp & 3, r = 16 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        for (int i = 0; i < nchunks; ++i) {
            const int b = i & 1;
            const int c = c0 + i;
            const ChunkInfo ci = plan_chunk(p, c);
            const bool mine = a.o && lane < 16 && r < ci.len;
            // O0 of this thread's token and the block's columns, from the ring slot
            // the producer filled with the chunk's Q' and O0 slices (ST::NS slices of
            // 64 tokens x 32 bytes); the slot is released once every output warp has
            // its rows
            const int qs = i % ST::QSTAGES;
            bool okw = mbar_wait_ab(&qfull_bar[qs], (uint32_t)((i / ST::QSTAGES) & 1), abort);
            uint4 o0v[2 * ST::NS];
            if (okw && mine) {
                const uint8_t *o0 = qring + qs * ST::QBYTES + ST::QO0 + r * 32;
#pragma unroll
                for (int sl = 0; sl < ST::NS; ++sl) slice_row_halves(o0 + sl * REC_BF16_OSLICE, r, o0v[2 * sl], o0v[2 * sl + 1]);
            }
            __syncwarp();
            if (okw && lane == 0) mbar_arrive(&qfree_bar[qs]);
            okw = okw && mbar_wait_ab(&o_bar[b], (uint32_t)((i >> 1) & 1), abort);
            if (!__all_sync(0xffffffffu, okw) || *(volatile int *)&abort_flag) {
                if (lane == 0) {
                    abort_flag = 1;
                    atomicOr(p.err, KDA_DEVERR_TIMEOUT);
                }
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < N / 32; ++half) {
                float d[32];
                tmem_ld16(tmem_g + lane_off + ST::OCOL + b * N + 32 * half, d);
                tmem_ld16(tmem_g + lane_off + ST::OCOL + b * N + 32 * half + 16, d + 16);
                tmem_ld_wait();
                if (mine) {
                    __nv_bfloat16 *orow =
                        reinterpret_cast<__nv_bfloat16 *>(a.o) + ((size_t)(ci.tok + r) * a.H + h) * D + col0 + 32 * half;
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&o0v[(32 * half + j) / 8]);
                        uint4 w;
                        __nv_bfloat162 *wp = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(x[e]);
                            wp[e] = __floats2bfloat162_rn(f.x + d[j + 2 * e], f.y + d[j + 2 * e + 1]);
                        }
                        *reinterpret_cast<uint4 *>(orow + j) = w;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&oempty_bar[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_g, ST::NCOLS);
}

}  // namespace

}  // namespace kda
