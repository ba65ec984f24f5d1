// kda_scan_simt.cu -- the sequential chunk scan in fp32 CUDA cores.
//
// Per chunk, with the record written by the prep kernel ("Kimi K3: the
// Manos, the Mythos ..." (SemiAnalysis), "FlashKDA 算法", the K2 recurrence
// U = INV Diag(beta)(V - K_decay S), O = Q_decay S + M_qk U,
// S = Diag(a[-1]) S + K_restore^T U, with the state-independent products
// folded into W, U0, Q', O0):
//   U = U0 - W S,   O = O0 + Q' S,   S <- Diag(a_C) S + K_restore^T U.
// The columns of S evolve independently (every update acts on the left), so a
// block owns 16 state columns (more blocks on the SMs, two per SM in shared
// memory), a thread one row and 8 of them.  With 256 state columns the extra 128 columns
// start from the identity and see V = 0: they carry the transition M of
// "Kimi K3 模型结构（7）" eq. (17) (M I = M), giving the segment pair (M, S~).
// Document starts reset the state ("文档边界").
//
// This is the exact-fp32 scan used for fp32 inputs (fp32 records).
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int SCAN_THREADS = 256;
constexpr int NC = 16;       // state columns per block
constexpr int PER = NC / 2;  // state columns per thread (two threads per row)
constexpr int LDA = 132;     // padded row stride of 128-wide fp32 tiles
constexpr int LDS = NC + 1;  // padded row stride of NC-wide tiles

struct ScanSmem {
    static constexpr int a1 = 0;                // [128][LDA]  rows 0..63 W, 64..127 Q'
    static constexpr int kr = a1 + 128 * LDA;   // [64][LDA]   K_restore (token-major)
    static constexpr int s = kr + 64 * LDA;     // [128][LDS]  state slice
    static constexpr int u = s + 128 * LDS;     // [64][LDS]
    static constexpr int ac = u + 64 * LDS;     // [128]
    static constexpr int total = ac + 128;
};
constexpr size_t SCAN_SMEM_BYTES = sizeof(float) * ScanSmem::total;

__device__ __forceinline__ void load_record(const char *rec, float *a1, float *kr, float *ac, int tid) {
    const float *W = reinterpret_cast<const float *>(rec + REC_F32_W);
    const float *Q = reinterpret_cast<const float *>(rec + REC_F32_Q);
    const float *K = reinterpret_cast<const float *>(rec + REC_F32_KR);
    for (int idx = tid; idx < 64 * 32; idx += SCAN_THREADS) {
        const int r = idx >> 5, c4 = (idx & 31) * 4;
        *reinterpret_cast<float4 *>(a1 + r * LDA + c4) = *reinterpret_cast<const float4 *>(W + r * 128 + c4);
        *reinterpret_cast<float4 *>(a1 + (64 + r) * LDA + c4) = *reinterpret_cast<const float4 *>(Q + r * 128 + c4);
        *reinterpret_cast<float4 *>(kr + r * LDA + c4) = *reinterpret_cast<const float4 *>(K + r * 128 + c4);
    }
    if (tid < 128) ac[tid] = reinterpret_cast<const float *>(rec + REC_F32_AC)[tid];
}

__device__ __forceinline__ float rec_u0(const char *rec, int r, int col) {
    return reinterpret_cast<const float *>(rec + REC_F32_U0)[r * 128 + col];
}
__device__ __forceinline__ float rec_o0(const char *rec, int r, int col) {
    return reinterpret_cast<const float *>(rec + REC_F32_O0)[r * 128 + col];
}

// Initial / reset value of state column `gcol` (0..ncols-1), row r.
__device__ __forceinline__ float state_reset(const ScanArgs &a, int doc, int h, int r, int gcol) {
    if (gcol >= D) return 0.f;  // transition columns restart from zero at a document start
    return a.init_state ? a.init_state[(((size_t)doc * a.H + h) * D + r) * D + gcol] : 0.f;
}

__global__ void __launch_bounds__(SCAN_THREADS) scan_simt_kernel(ScanArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int unit = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int col0 = blockIdx.z * NC;  // global state column of this block
    const bool value_cols = col0 < D;
    const Plan &p = a.plan;
    float *a1 = sm + ScanSmem::a1, *kr = sm + ScanSmem::kr, *S = sm + ScanSmem::s;
    float *U = sm + ScanSmem::u, *ac = sm + ScanSmem::ac;

    if (plan_failed(p)) return;
    int c0, c1;
    if (a.mode == SCAN_DOCS) {
        if (unit >= p.n_seqs) return;
        plan_doc_range(p, unit, c0, c1);
    } else {
        segment_range(plan_n_chunks(p), a.n_seg, unit, c0, c1);
    }

    // initial state of the unit
    for (int idx = tid; idx < 128 * NC; idx += SCAN_THREADS) {
        const int r = idx / NC, j = idx % NC, g = col0 + j;
        float x;
        if (a.mode == SCAN_DOCS) x = state_reset(a, unit, h, r, g);
        else if (a.phase == 1) x = (g >= D && r == g - D) ? 1.f : 0.f;
        else x = a.s_enter[(((size_t)h * a.n_seg + unit) * D + r) * D + g];
        S[r * LDS + j] = x;
    }
    if (a.mode == SCAN_DOCS && c1 <= c0) {
        // empty document: its final state is its initial state
        __syncthreads();
        if (a.final_state)
            for (int idx = tid; idx < 128 * NC; idx += SCAN_THREADS) {
                const int r = idx / NC, j = idx % NC;
                a.final_state[(((size_t)unit * a.H + h) * D + r) * D + col0 + j] = S[r * LDS + j];
            }
        return;
    }

    const int row = tid >> 1, cc = (tid & 1) * PER;  // this thread's PER outputs
    for (int c = c0; c < c1; ++c) {
        const ChunkInfo ci = plan_chunk(p, c);
        const char *rec = (const char *)a.records +
                          ((size_t)c * a.H + h) * REC_F32_BYTES;
        __syncthreads();  // previous chunk finished with a1 / kr / S
        if (a.mode == SCAN_SEGMENTS && (ci.flags & CHUNK_FIRST)) {
            for (int idx = tid; idx < 128 * NC; idx += SCAN_THREADS) {
                const int r = idx / NC, j = idx % NC;
                S[r * LDS + j] = state_reset(a, ci.doc, h, r, col0 + j);
            }
        }
        load_record(rec, a1, kr, ac, tid);
        __syncthreads();

        // D1 = [W ; Q'] S   (row < 64: W S, row >= 64: Q' S)
        float acc[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) acc[j] = 0.f;
        for (int kk = 0; kk < D; ++kk) {
            const float w = a1[row * LDA + kk];
#pragma unroll
            for (int j = 0; j < PER; ++j) acc[j] = fmaf(w, S[kk * LDS + cc + j], acc[j]);
        }
        if (row < C) {
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int g = col0 + cc + j;
                const float u0 = (g < D) ? rec_u0(rec, row, g) : 0.f;
                U[row * LDS + cc + j] = u0 - acc[j];
            }
        } else if (value_cols && a.o && a.phase != 1 && row - C < ci.len) {
            const int r = row - C;
            float *orow = reinterpret_cast<float *>(a.o) + ((size_t)(ci.tok + r) * a.H + h) * D + col0 + cc;
#pragma unroll
            for (int j = 0; j < PER; ++j)
                orow[j] = rec_o0(rec, r, col0 + cc + j) + acc[j];
        }
        __syncthreads();

        // S <- Diag(a_C) S + K_restore^T U
        float nacc[PER];
        const float dec = ac[row];
#pragma unroll
        for (int j = 0; j < PER; ++j) nacc[j] = dec * S[row * LDS + cc + j];
        for (int t = 0; t < C; ++t) {
            const float kv = kr[t * LDA + row];
#pragma unroll
            for (int j = 0; j < PER; ++j) nacc[j] = fmaf(kv, U[t * LDS + cc + j], nacc[j]);
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < PER; ++j) S[row * LDS + cc + j] = nacc[j];

        if (value_cols && a.final_state && a.phase != 1 && (ci.flags & CHUNK_LAST)) {
            float *f = a.final_state + (((size_t)ci.doc * a.H + h) * D + row) * D + col0 + cc;
#pragma unroll
            for (int j = 0; j < PER; ++j) f[j] = nacc[j];
        }
        if (value_cols && a.ckpt && a.phase != 1) {
            // the state after this chunk, when it ends on a checkpoint position
            float *f = ckpt_row(a, ci, c, h, row);
            if (f) {
#pragma unroll
                for (int j = 0; j < PER; ++j) f[col0 + cc + j] = nacc[j];
            }
        }
    }

    if (a.mode == SCAN_SEGMENTS && a.phase == 1) {
        __syncthreads();
        // pairs: [0] = M (columns D..2D-1), [1] = S~ (columns 0..D-1)
        const int which = value_cols ? 1 : 0;
        const int pc0 = value_cols ? col0 : col0 - D;
        float *dst = a.pairs + ((((size_t)which * a.H + h) * a.n_seg + unit) * D) * D;
        for (int idx = tid; idx < 128 * NC; idx += SCAN_THREADS) {
            const int r = idx / NC, j = idx % NC;
            dst[(size_t)r * D + pc0 + j] = S[r * LDS + j];
        }
    }
}

}  // namespace

int launch_scan_simt(const ScanArgs &a, int dtype, cudaStream_t s) {
    if (a.n_units == 0) return KDA_OK;
    if (dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
    dim3 grid(a.n_units, a.H, a.ncols / NC);
    if (cudaFuncSetAttribute(scan_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SCAN_SMEM_BYTES) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    scan_simt_kernel<<<grid, SCAN_THREADS, SCAN_SMEM_BYTES, s>>>(a);
    note_launch("scan_simt", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
