// kda_plan.cu -- chunk plan of packed documents, and empty-document states.
//
// Documents are cut into 64-token chunks that never straddle a document
// boundary, because the state restarts at every document start
// ("Kimi K3 模型结构（7）：结构决定系统", section "文档边界").  One block
// validates cu_seqlens, numbers the chunks of every document with an
// exclusive scan, and writes one ChunkInfo per chunk.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int PLAN_THREADS = 1024;

__global__ void __launch_bounds__(PLAN_THREADS) plan_kernel(const int32_t *__restrict__ cu,
                                                            int n_seqs, int T_total,
                                                            ChunkInfo *__restrict__ table,
                                                            int32_t *__restrict__ doc_off,
                                                            int32_t *__restrict__ header,
                                                            int max_chunks) {
    __shared__ int s_scan[PLAN_THREADS];
    __shared__ int s_run, s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_run = 0;
        s_bad = (cu[0] != 0 || cu[n_seqs] != T_total) ? 1 : 0;
    }
    __syncthreads();
    for (int base = 0; base < n_seqs; base += PLAN_THREADS) {
        const int d = base + tid;
        int nc = 0;
        if (d < n_seqs) {
            const int a = cu[d], b = cu[d + 1];
            if (b < a || a < 0 || b > T_total) atomicOr(&s_bad, 1);
            else nc = (b - a + C - 1) / C;
        }
        s_scan[tid] = nc;
        __syncthreads();
        for (int o = 1; o < PLAN_THREADS; o <<= 1) {
            const int x = tid >= o ? s_scan[tid - o] : 0;
            __syncthreads();
            s_scan[tid] += x;
            __syncthreads();
        }
        if (d < n_seqs) doc_off[d] = s_run + s_scan[tid] - nc;
        __syncthreads();
        if (tid == PLAN_THREADS - 1) s_run += s_scan[tid];
        __syncthreads();
    }
    const int n_chunks = s_run;
    if (s_bad || n_chunks > max_chunks) {
        if (tid == 0) {
            atomicOr(&header[0], KDA_DEVERR_CU_SEQLENS);
            header[1] = 0;
        }
        // an empty plan: every document range is empty, nothing downstream runs
        for (int d = tid; d <= n_seqs; d += PLAN_THREADS) doc_off[d] = 0;
        return;
    }
    if (tid == 0) {
        doc_off[n_seqs] = n_chunks;
        header[1] = n_chunks;
    }
    __syncthreads();
    for (int c = tid; c < n_chunks; c += PLAN_THREADS) {
        // last document d with doc_off[d] <= c (empty documents share offsets)
        int lo = 0, hi = n_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (doc_off[mid] <= c) lo = mid;
            else hi = mid - 1;
        }
        const int d = lo;
        const int i = c - doc_off[d];
        const int nd = doc_off[d + 1] - doc_off[d];
        ChunkInfo ci;
        ci.doc = d;
        ci.tok = cu[d] + i * C;
        const int rem = cu[d + 1] - ci.tok;
        ci.len = rem < C ? rem : C;
        ci.flags = (i == 0 ? CHUNK_FIRST : 0) | (i == nd - 1 ? CHUNK_LAST : 0);
        table[c] = ci;
    }
}

// final_state[d] = init_state[d] (or zeros) for documents without tokens.
__global__ void empty_docs_kernel(Plan p, int H, const float *__restrict__ init,
                                  float *__restrict__ fin) {
    const int d = blockIdx.x, h = blockIdx.y;
    if (plan_failed(p)) return;
    int c0, c1;
    plan_doc_range(p, d, c0, c1);
    if (c1 > c0) return;
    const size_t base = ((size_t)d * H + h) * D * D;
    for (int i = threadIdx.x; i < D * D; i += blockDim.x)
        fin[base + i] = init ? init[base + i] : 0.0f;
}

}  // namespace

int launch_plan(const int32_t *cu, int n_seqs, int64_t T_total, void *ws, const Workspace &w,
                cudaStream_t s) {
    char *base = (char *)ws;
    plan_kernel<<<1, PLAN_THREADS, 0, s>>>(cu, n_seqs, (int)T_total,
                                           (ChunkInfo *)(base + w.off_table),
                                           (int32_t *)(base + w.off_doc), (int32_t *)base,
                                           w.max_chunks);
    note_launch("plan", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int launch_empty_docs(const Plan &p, int H, const float *init_state, float *final_state,
                      cudaStream_t s) {
    if (!final_state) return KDA_OK;
    dim3 grid(p.n_seqs, H);
    empty_docs_kernel<<<grid, 256, 0, s>>>(p, H, init_state, final_state);
    note_launch("empty_docs", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
