// kda_scan_tc.cu -- the sequential chunk scan on tcgen05 tensor cores.
//
// With the record of the prep kernel (G = K_restore^T W, H = K_restore^T U0,
// Q' = Q_decay - M_qk W, O0 = M_qk U0, a_C), one chunk of the scan is
//   S <- Diag(a_C) S + H - G S          (the chain: one M = 128 MMA per chunk)
//   O  = O0 + Q' S                      (off the chain)
// which is "Kimi K3: the Manos, the Mythos ..." (SemiAnalysis), "FlashKDA 算法"
// K2 (U = INV Diag(beta)(V - K_decay S), O = Q_decay S + M_qk U,
// S = Diag(a[-1]) S + K_restore^T U) with its products regrouped so that only
// one tensor-core round trip sits on the sequential path.
//
// A block owns N state columns (columns evolve independently).  With 256
// state columns the extra 128 start from the identity with H = 0: they carry
// the transition M of "Kimi K3 模型结构（7）" eq. (17) for the segment pairs.
//
// Warps 0-3 (chain): thread t owns state row t (TMEM lane t); the fp32 state
//   master lives in registers, its bf16 copy (double buffered) in shared
//   memory is the B operand of the next chunk's MMAs; thread 0 issues them.
// Warps 4-5 (output): one of their threads issues O = Q' S into a
//   double-buffered TMEM accumulator as soon as the chain has published S,
//   and the two warps drain O0 + Q' S while the chain moves on.
// Warp 6 (producer): streams each chunk's record (G, a_C, Q', the block's H
//   and O0 column slices) through a bulk-copy pipeline.
// Every wait is bounded; on a timeout the block records KDA_DEVERR_TIMEOUT,
// leaves its loops, and frees its TMEM.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int CHAIN = 128;          // warps 0-3
constexpr int PRODUCER_WARP = 6;
constexpr int THREADS = 224;

// pipeline stage: G (32 KB) | a_C | Q' (16 KB) | H slices | O0 slices
template <int N>
struct Stage {
    static constexpr int NS = N / 16;
    static constexpr int G = 0;
    static constexpr int AC = (int)REC_BF16_AC;
    static constexpr int QP = (int)REC_BF16_QP;
    static constexpr int H = (int)REC_BF16_H;
    static constexpr int O0 = H + NS * (int)REC_BF16_HSLICE;
    static constexpr int BYTES = ((O0 + NS * (int)REC_BF16_OSLICE) + 1023) / 1024 * 1024;
    static constexpr int SOP = 2 * N * 128;  // one bf16 S operand: 2 k-blocks x N rows x 128 B
    static constexpr int COLS = 3 * N;       // TMEM: chain accumulator + two output accumulators
    static constexpr int NCOLS = COLS <= 32 ? 32 : (COLS <= 64 ? 64 : (COLS <= 128 ? 128 : 256));
};

template <int N, int STAGES>
constexpr size_t scan_tc_smem_bytes() {
    return (size_t)STAGES * Stage<N>::BYTES + 2 * Stage<N>::SOP + 1024;
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

// bf16 copy of this thread's state row into the K-major S operand (row n = column, k = state row t)
template <int N>
__device__ __forceinline__ void write_sop(uint8_t *sop, int t, const float *s) {
#pragma unroll
    for (int n = 0; n < N; ++n)
        *reinterpret_cast<__nv_bfloat16 *>(sop + sw128_offset(n, t, N)) = __float2bfloat16_rn(s[n]);
}

// N bf16 values of row r from consecutive 16-column slices of `rows` rows each
template <int N>
__device__ __forceinline__ void load_slices(const uint8_t *base, int r, int rows, float *out) {
#pragma unroll
    for (int j = 0; j < N; j += 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(base + slice_offset(r, j, rows));
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(p[e]);
            out[j + 2 * e] = f.x;
            out[j + 2 * e + 1] = f.y;
        }
    }
}

template <int N>
__device__ __forceinline__ void tmem_row(uint32_t taddr, float *out) {
#pragma unroll
    for (int j = 0; j < N; j += 16) tmem_ld16(taddr + j, out + j);
    tmem_ld_wait();
}

template <int N, int STAGES>
__global__ void __launch_bounds__(THREADS, 1) scan_tc_kernel(ScanArgs a) {
    using ST = Stage<N>;
    extern __shared__ uint8_t smraw[];
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES], g_bar, o_bar[2], sready_bar[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int unit = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int col0 = blockIdx.z * N;
    const bool value_cols = col0 < D;
    const bool emit_o = value_cols && a.o && a.phase != 1;
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
    uint8_t *sop0 = sm + STAGES * ST::BYTES;
    const char *records = (const char *)a.records;
    const size_t rec_stride = (size_t)a.H * REC_BF16_BYTES;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            // released by: the chain MMA (commit), the chain warps, and when the
            // output is emitted the output MMA (commit) and the output warps
            mbar_init(&empty_bar[s], emit_o ? 4 : 2);
        }
        mbar_init(&g_bar, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&o_bar[b], 1);
            mbar_init(&sready_bar[b], 1);  // the S operand of buffer b holds the entering state
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, ST::NCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t tmem_g = tmem, tmem_o = tmem + N;  // output accumulators at tmem_o + b * N

    if (warp == PRODUCER_WARP) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            bool timed_out = false;
            const uint32_t bytes = (uint32_t)REC_BF16_SHARED +
                                   (value_cols ? (uint32_t)(16384 + ST::NS * (REC_BF16_HSLICE + REC_BF16_OSLICE)) : 0u);
            for (int i = 0; i < nchunks; ++i) {
                const int stage = i % STAGES;
                const uint32_t ph = (uint32_t)((i / STAGES) & 1);
                if (!mbar_wait(&empty_bar[stage], ph ^ 1u)) { timed_out = true; break; }
                if (*(volatile int *)&abort_flag) break;
                const char *rec = records + (size_t)(c0 + i) * rec_stride + (size_t)h * REC_BF16_BYTES;
                uint8_t *st = sm + stage * ST::BYTES;
                mbar_expect_tx(&full_bar[stage], bytes);
                bulk_g2s(st, rec, (uint32_t)REC_BF16_SHARED, &full_bar[stage]);
                if (value_cols) {
                    const int s0 = col0 / 16;
                    bulk_g2s(st + ST::QP, rec + REC_BF16_QP, 16384, &full_bar[stage]);
                    bulk_g2s(st + ST::H, rec + REC_BF16_H + (size_t)s0 * REC_BF16_HSLICE,
                             (uint32_t)(ST::NS * REC_BF16_HSLICE), &full_bar[stage]);
                    bulk_g2s(st + ST::O0, rec + REC_BF16_O0 + (size_t)s0 * REC_BF16_OSLICE,
                             (uint32_t)(ST::NS * REC_BF16_OSLICE), &full_bar[stage]);
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
    } else if (warp >= 4) {
        // ------------------------------------------------------------ output warps
        if (emit_o) {
            const int r = tid - CHAIN;  // token row of the chunk = TMEM lane
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            constexpr uint32_t IDESC = idesc_bf16_f32(128, N);
            for (int i = 0; i < nchunks; ++i) {
                const int stage = i % STAGES, b = i & 1;
                const uint32_t ph = (uint32_t)((i / STAGES) & 1);
                const ChunkInfo ci = plan_chunk(p, c0 + i);
                bool ok = true;
                if (r == 0) {
                    // O = Q' S of this chunk, once its stage has landed and the chain has
                    // published the entering state in S operand buffer b
                    ok = mbar_wait(&full_bar[stage], ph) && mbar_wait(&sready_bar[b], (uint32_t)((i >> 1) & 1));
                    if (ok) {
                        tc_fence_after();
                        const uint8_t *st = sm + stage * ST::BYTES;
                        const uint8_t *sop = sop0 + b * ST::SOP;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint64_t ad = sdesc_sw128(smem_u32(st + ST::QP + (k >> 2) * 8192 + (k & 3) * 32));
                            const uint64_t bd = sdesc_sw128(smem_u32(sop + (k >> 2) * (N * 128) + (k & 3) * 32));
                            mma_bf16(tmem_o + b * N, ad, bd, IDESC, k > 0);
                        }
                        mma_commit(&o_bar[b]);
                        mma_commit(&empty_bar[stage]);
                    }
                }
                ok = ok && mbar_wait(&o_bar[b], (uint32_t)((i >> 1) & 1)) && mbar_wait(&full_bar[stage], ph);
                __syncwarp();
                tc_fence_after();
                float d[N], x[N];
                tmem_row<N>(tmem_o + b * N + lane_off, d);
                load_slices<N>(sm + stage * ST::BYTES + ST::O0, r, 64, x);
                tc_fence_before();
                // both output warps are done with this accumulator and stage (or both give up)
                if (bar_or(2, 64, !ok || *(volatile int *)&abort_flag)) break;
                if (r == 0) mbar_arrive(&empty_bar[stage]);
                if (r < ci.len) {
                    __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(a.o) + ((size_t)(ci.tok + r) * a.H + h) * D + col0;
#pragma unroll
                    for (int j = 0; j < N; j += 8) {
                        __align__(16) __nv_bfloat16 ob[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) ob[e] = __float2bfloat16_rn(x[j + e] + d[j + e]);
                        *reinterpret_cast<uint4 *>(orow + j) = *reinterpret_cast<const uint4 *>(ob);
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ chain warps
        const int t = tid;  // state row == TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        float s[N];
#pragma unroll
        for (int j = 0; j < N; ++j) s[j] = state_init(a, unit, h, t, col0 + j);
        if (a.mode == SCAN_DOCS && nchunks == 0 && value_cols && a.final_state) {
            float *f = a.final_state + (((size_t)unit * a.H + h) * D + t) * D + col0;
#pragma unroll
            for (int j = 0; j < N; j += 4) *reinterpret_cast<float4 *>(f + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
        }
        write_sop<N>(sop0, t, s);
        fence_async_smem();
        bool aborted = bar_or(1, CHAIN, false);
        ChunkInfo ci_next;
        if (nchunks > 0) ci_next = plan_chunk(p, c0);
        constexpr uint32_t IDESC = idesc_bf16_f32(128, N);
        for (int i = 0; i < nchunks && !aborted; ++i) {
            const int stage = i % STAGES;
            const uint32_t ph = (uint32_t)((i / STAGES) & 1);
            const ChunkInfo ci = ci_next;
            if (i + 1 < nchunks) ci_next = plan_chunk(p, c0 + i + 1);
            uint8_t *sop = sop0 + (i & 1) * ST::SOP;
            if (a.mode == SCAN_SEGMENTS && (ci.flags & CHUNK_FIRST)) {
                // a document starts here: the state restarts (uniform branch)
#pragma unroll
                for (int j = 0; j < N; ++j) s[j] = state_reset(a, ci.doc, h, t, col0 + j);
                write_sop<N>(sop, t, s);
                fence_async_smem();
                bar_or(1, CHAIN, false);
            }
            bool bad = false;
            if (t == 0) {
                if (mbar_wait(&full_bar[stage], ph)) {
                    tc_fence_after();
                    uint8_t *st = sm + stage * ST::BYTES;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t ad = sdesc_sw128(smem_u32(st + ST::G + (k >> 2) * 16384 + (k & 3) * 32));
                        const uint64_t bd = sdesc_sw128(smem_u32(sop + (k >> 2) * (N * 128) + (k & 3) * 32));
                        mma_bf16(tmem_g, ad, bd, IDESC, k > 0);
                    }
                    mma_commit(&g_bar);
                    mma_commit(&empty_bar[stage]);
                    // the S operand of this chunk is final: the output MMA may read it
                    if (emit_o) mbar_arrive(&sready_bar[i & 1]);
                } else {
                    bad = true;
                }
            }
            // ---- S <- Diag(a_C) S + H - G S
            const bool ok = !bad && mbar_wait(&g_bar, (uint32_t)(i & 1)) && mbar_wait(&full_bar[stage], ph);
            __syncwarp();
            tc_fence_after();
            const uint8_t *stg = sm + stage * ST::BYTES;
            const float ac = reinterpret_cast<const float *>(stg + ST::AC)[t];
            float d[N], hv[N];
            tmem_row<N>(tmem_g + lane_off, d);
            if (value_cols) load_slices<N>(stg + ST::H, t, 128, hv);
            else
#pragma unroll
                for (int j = 0; j < N; ++j) hv[j] = 0.f;
#pragma unroll
            for (int j = 0; j < N; ++j) s[j] = fmaf(ac, s[j], hv[j] - d[j]);
            // buffer (i+1)&1 was last read by chunk i-1's output MMA, which must be done
            const bool ok_o = !emit_o || i < 1 || mbar_wait(&o_bar[(i + 1) & 1], (uint32_t)(((i - 1) >> 1) & 1));
            write_sop<N>(sop0 + ((i + 1) & 1) * ST::SOP, t, s);
            if (value_cols && a.final_state && a.phase != 1 && (ci.flags & CHUNK_LAST)) {
                float *f = a.final_state + (((size_t)ci.doc * a.H + h) * D + t) * D + col0;
#pragma unroll
                for (int j = 0; j < N; j += 4) *reinterpret_cast<float4 *>(f + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
            }
            fence_async_smem();
            tc_fence_before();
            aborted = bar_or(1, CHAIN, !ok || !ok_o);
            if (t == 0 && !aborted) mbar_arrive(&empty_bar[stage]);
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
    if (warp == 0) tmem_dealloc(tmem, ST::NCOLS);
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
    // Few independent column slices: narrow blocks spread the chains over more
    // SMs.  Many: wider blocks amortise the per-chunk latency.
    const long long slices16 = (long long)a.n_units * a.H * (a.ncols / 16);
    if (slices16 <= 2LL * n_sm) return launch_n<16, 3>(a, s);
    return launch_n<64, 2>(a, s);
}

}  // namespace kda
