// kda_scan_tc.cu -- the sequential chunk scan on tcgen05 tensor cores.
//
// Per chunk ("Kimi K3: the Manos, the Mythos ..." (SemiAnalysis),
// "FlashKDA 算法", the K2 recurrence, with the state-independent products
// folded by the prep kernel into W, U0, Q', O0):
//   D1 = [W ; Q'] S          (one M = 128 MMA: rows 0..63 W S, rows 64..127 Q' S)
//   U  = U0 - D1[0:64],  O = O0 + D1[64:128]
//   D2 = K_restore^T U       (one M = 128 MMA over the chunk's 64 tokens)
//   S <- Diag(a_C) S + D2
// The fp32 state master lives in registers (thread t owns state row t); its
// bf16 copy in shared memory is the B operand of the next chunk's first MMA,
// and U's bf16 copy is the B operand of the second.  Accumulators live in
// TMEM.  The chunk operands (A1 = [W ; Q'] and K_restore^T, 48 KB per chunk,
// stored by the prep kernel as ready-swizzled images) stream in through a
// multi-stage bulk-copy pipeline driven by a producer warp.
//
// A block owns N state columns (they evolve independently); with 256 state
// columns the extra 128 start from the identity and see V = 0, which carries
// the transition M of "Kimi K3 模型结构（7）" eq. (17) for the segment pairs.
//
// Warps 0-3: epilogue (TMEM lane = warp * 32 + lane), thread 0 issues the MMAs.
// Warp 4: producer.  Every wait is bounded; on a timeout the block records
// KDA_DEVERR_TIMEOUT, leaves its loop, and frees its TMEM.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int CONSUMERS = 128;
constexpr int THREADS = CONSUMERS + 32;

// One pipeline stage: the shared part of a record (A1, K_restore^T, a_C) and
// this block's U0 / O0 column slices.
template <int N>
struct TcSmem {
    static constexpr int NS = N / 16;                          // 16-column slices
    static constexpr int U0 = (int)REC_BF16_SHARED;            // stage offset of the U0 slices
    static constexpr int O0 = U0 + NS * (int)REC_BF16_SLICE;   // stage offset of the O0 slices
    static constexpr int STAGE = ((O0 + NS * (int)REC_BF16_SLICE) + 1023) / 1024 * 1024;
    static constexpr int SOP = 2 * N * 128;  // S^T operand: 2 k-blocks x N rows x 128 B
    static constexpr int UOP = N * 128;      // U^T operand: 1 k-block x N rows x 128 B
    // TMEM: D1 in P1 partial accumulators, D2 in P2 (independent MMA chains overlap)
    static constexpr int P1 = 4, P2 = 2;
    static constexpr int COLS = (P1 + P2) * N;
    static constexpr int NCOLS = COLS <= 32 ? 32 : (COLS <= 64 ? 64 : (COLS <= 128 ? 128 : (COLS <= 256 ? 256 : 512)));
};

template <int N, int STAGES>
constexpr size_t scan_tc_smem_bytes() {
    return (size_t)STAGES * TcSmem<N>::STAGE + TcSmem<N>::SOP + TcSmem<N>::UOP + 1024;
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

// bf16 copy of this thread's state row into the K-major S^T operand (row n = column, k = state row t)
template <int N>
__device__ __forceinline__ void write_sop(uint8_t *sop, int t, const float *s) {
#pragma unroll
    for (int n = 0; n < N; ++n)
        *reinterpret_cast<__nv_bfloat16 *>(sop + sw128_offset(n, t, N)) = __float2bfloat16_rn(s[n]);
}

// Sum of P partial accumulators (N columns each, N apart) of this thread's TMEM lane.
template <int N, int P>
__device__ __forceinline__ void tmem_sum(uint32_t taddr, float *out) {
#pragma unroll
    for (int j = 0; j < N; j += 16) {
        float part[P][16];
#pragma unroll
        for (int pp = 0; pp < P; ++pp) tmem_ld16(taddr + pp * N + j, part[pp]);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            float acc = part[0][e];
#pragma unroll
            for (int pp = 1; pp < P; ++pp) acc += part[pp][e];
            out[j + e] = acc;
        }
    }
}

// N bf16 values of token row r from consecutive 16-column slices (2 KB apart)
template <int N>
__device__ __forceinline__ void load_row_slices(const uint8_t *base, int r, float *out) {
#pragma unroll
    for (int j = 0; j < N; j += 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(base + slice_offset(r, j));
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(p[e]);
            out[j + 2 * e] = f.x;
            out[j + 2 * e + 1] = f.y;
        }
    }
}

template <int N, int STAGES>
__global__ void __launch_bounds__(THREADS, 1) scan_tc_kernel(ScanArgs a) {
    extern __shared__ uint8_t smraw[];
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES], mma1_bar, mma2_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int unit = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int col0 = blockIdx.z * N;
    const bool value_cols = col0 < D;
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

    constexpr int STAGE_BYTES = TcSmem<N>::STAGE;
    uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    uint8_t *sop = sm + STAGES * STAGE_BYTES;
    uint8_t *uop = sop + TcSmem<N>::SOP;
    const char *records = (const char *)a.records;
    const size_t rec_stride = (size_t)a.H * REC_BF16_BYTES;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(&mma1_bar, 1);
        mbar_init(&mma2_bar, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, TcSmem<N>::NCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    constexpr int P1 = TcSmem<N>::P1, P2 = TcSmem<N>::P2;
    const uint32_t tmem_d1 = tmem, tmem_d2 = tmem + P1 * N;

    if (warp == CONSUMERS / 32) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            bool timed_out = false;
            for (int i = 0; i < nchunks; ++i) {
                const int stage = i % STAGES;
                const uint32_t ph = (uint32_t)((i / STAGES) & 1);
                if (!mbar_wait(&empty_bar[stage], ph ^ 1u)) { timed_out = true; break; }
                if (*(volatile int *)&abort_flag) break;
                const char *rec = records + (size_t)(c0 + i) * rec_stride + (size_t)h * REC_BF16_BYTES;
                uint8_t *st = sm + stage * STAGE_BYTES;
                const uint32_t slices = value_cols ? (uint32_t)(TcSmem<N>::NS * REC_BF16_SLICE) : 0u;
                mbar_expect_tx(&full_bar[stage], (uint32_t)REC_BF16_SHARED + 2u * slices);
                bulk_g2s(st, rec, (uint32_t)REC_BF16_SHARED, &full_bar[stage]);
                if (value_cols) {
                    const size_t so = (size_t)(col0 / 16) * REC_BF16_SLICE;
                    bulk_g2s(st + TcSmem<N>::U0, rec + REC_BF16_U0 + so, slices, &full_bar[stage]);
                    bulk_g2s(st + TcSmem<N>::O0, rec + REC_BF16_O0 + so, slices, &full_bar[stage]);
                }
                issued = i + 1;
            }
            if (timed_out || *(volatile int *)&abort_flag) {
                // let the copies this thread started land before the block exits
                for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
                    mbar_wait(&full_bar[i % STAGES], (uint32_t)((i / STAGES) & 1));
                if (timed_out) atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue + MMA issue
        const int t = tid;  // TMEM lane == state row (D2) == token row (D1)
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        float s[N];
#pragma unroll
        for (int j = 0; j < N; ++j) s[j] = state_init(a, unit, h, t, col0 + j);
        if (a.mode == SCAN_DOCS && nchunks == 0) {
            if (value_cols && a.final_state) {
                float *f = a.final_state + (((size_t)unit * a.H + h) * D + t) * D + col0;
#pragma unroll
                for (int j = 0; j < N; j += 4) *reinterpret_cast<float4 *>(f + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
            }
        }
        write_sop<N>(sop, t, s);
        fence_async_smem();
        bool aborted = bar_or(1, CONSUMERS, false);

        ChunkInfo ci_next;
        if (nchunks > 0) ci_next = plan_chunk(p, c0);

        constexpr uint32_t IDESC = idesc_bf16_f32(128, N);
        for (int i = 0; i < nchunks && !aborted; ++i) {
            const int stage = i % STAGES;
            const uint32_t ph = (uint32_t)((i / STAGES) & 1);
            const ChunkInfo ci = ci_next;
            if (i + 1 < nchunks) ci_next = plan_chunk(p, c0 + i + 1);
            if (a.mode == SCAN_SEGMENTS && (ci.flags & CHUNK_FIRST)) {
                // a document starts here: the state restarts (uniform branch)
#pragma unroll
                for (int j = 0; j < N; ++j) s[j] = state_reset(a, ci.doc, h, t, col0 + j);
                write_sop<N>(sop, t, s);
                fence_async_smem();
                bar_or(1, CONSUMERS, false);
            }
            bool bad = false;
            if (t == 0) {
                if (mbar_wait(&full_bar[stage], ph)) {
                    tc_fence_after();
                    uint8_t *st = sm + stage * STAGE_BYTES;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t ad = sdesc_sw128(smem_u32(st + (k >> 2) * 16384 + (k & 3) * 32));
                        const uint64_t bd = sdesc_sw128(smem_u32(sop + (k >> 2) * (N * 128) + (k & 3) * 32));
                        mma_bf16(tmem_d1 + (k % P1) * N, ad, bd, IDESC, k >= P1);
                    }
                    mma_commit(&mma1_bar);
                } else {
                    bad = true;
                }
            }
            // ---- D1 -> U (rows 0..63), O (rows 64..127)
            const bool ok1 = !bad && mbar_wait(&mma1_bar, (uint32_t)(i & 1)) && mbar_wait(&full_bar[stage], ph);
            __syncwarp();
            tc_fence_after();
            // everything this thread needs from the stage, read before the stage is released
            const uint8_t *stg = sm + stage * STAGE_BYTES;
            const float ac = reinterpret_cast<const float *>(stg + REC_BF16_AC)[t];
            float x[N];
            if (value_cols)
                load_row_slices<N>(stg + (t < C ? TcSmem<N>::U0 : TcSmem<N>::O0), t < C ? t : t - C, x);
            else
#pragma unroll
                for (int j = 0; j < N; ++j) x[j] = 0.f;
            float d[N];
            tmem_sum<N, P1>(tmem_d1 + lane_off, d);
            if (t < C) {
#pragma unroll
                for (int n = 0; n < N; ++n)
                    *reinterpret_cast<__nv_bfloat16 *>(uop + sw128_offset(n, t, N)) = __float2bfloat16_rn(x[n] - d[n]);
            } else if (value_cols && a.o && a.phase != 1 && (t - C) < ci.len) {
                __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(a.o) + ((size_t)(ci.tok + t - C) * a.H + h) * D + col0;
#pragma unroll
                for (int j = 0; j < N; j += 8) {
                    __align__(16) __nv_bfloat16 ob[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) ob[e] = __float2bfloat16_rn(x[j + e] + d[j + e]);
                    *reinterpret_cast<uint4 *>(orow + j) = *reinterpret_cast<const uint4 *>(ob);
                }
            }
            fence_async_smem();
            tc_fence_before();
            aborted = bar_or(1, CONSUMERS, !ok1);
            if (aborted) break;
            // ---- D2 = K_restore^T U
            if (t == 0) {
                tc_fence_after();
                uint8_t *kr = sm + stage * STAGE_BYTES + REC_BF16_KRT;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t ad = sdesc_sw128(smem_u32(kr + k * 32));
                    const uint64_t bd = sdesc_sw128(smem_u32(uop + k * 32));
                    mma_bf16(tmem_d2 + (k % P2) * N, ad, bd, IDESC, k >= P2);
                }
                mma_commit(&mma2_bar);
                mma_commit(&empty_bar[stage]);
            }
            const bool ok2 = mbar_wait(&mma2_bar, (uint32_t)(i & 1));
            __syncwarp();
            tc_fence_after();
            tmem_sum<N, P2>(tmem_d2 + lane_off, d);
#pragma unroll
            for (int j = 0; j < N; ++j) s[j] = fmaf(ac, s[j], d[j]);
            write_sop<N>(sop, t, s);
            if (value_cols && a.final_state && a.phase != 1 && (ci.flags & CHUNK_LAST)) {
                float *f = a.final_state + (((size_t)ci.doc * a.H + h) * D + t) * D + col0;
#pragma unroll
                for (int j = 0; j < N; j += 4) *reinterpret_cast<float4 *>(f + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
            }
            fence_async_smem();
            tc_fence_before();
            aborted = bar_or(1, CONSUMERS, !ok2);
        }
        if (aborted) {
            if (t == 0) {
                abort_flag = 1;
                atomicOr(p.err, KDA_DEVERR_TIMEOUT);
            }
        } else if (a.mode == SCAN_SEGMENTS && a.phase == 1) {
            const int which = value_cols ? 1 : 0;
            const int pc0 = value_cols ? col0 : col0 - D;
            float *dst = a.pairs + ((((size_t)which * a.H + h) * a.n_seg + unit) * D + t) * D + pc0;
#pragma unroll
            for (int j = 0; j < N; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TcSmem<N>::NCOLS);
}

template <int N, int STAGES>
int launch_n(const ScanArgs &a, cudaStream_t s) {
    auto kern = scan_tc_kernel<N, STAGES>;
    const size_t smem = scan_tc_smem_bytes<N, STAGES>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return KDA_ERR_CUDA;
    dim3 grid(a.n_units, a.H, a.ncols / N);
    kern<<<grid, THREADS, smem, s>>>(a);
    note_launch("scan_tc", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

int launch_scan_tc(const ScanArgs &a, int n_sm, cudaStream_t s) {
    if (a.n_units == 0) return KDA_OK;
    // Few independent column slices: narrow blocks spread the chain over more
    // SMs.  Many: wider blocks, two per SM, amortise the per-chunk latency.
    const long long slices16 = (long long)a.n_units * a.H * (a.ncols / 16);
    if (slices16 <= 2LL * n_sm) return launch_n<16, 3>(a, s);
    return launch_n<64, 2>(a, s);
}

}  // namespace kda
