// kda_scan_tc.cu -- the scan kernel for bf16 records (device code in
// kda_scan_body.cuh): one block per (document or segment, head, column block).
// Few chains: 16-column blocks that store each chunk's entering state for the
// output kernel.  Many chains: 64-column blocks that form the outputs of their
// columns themselves (as the fused launch's chain blocks do), and 128-column
// blocks for the segment pairs.  Packed documents
// of unequal length start longest first (the document is the grid's slowest
// dimension, ranked by chunk count), so that the last blocks to start hold
// the shortest chains.
#include "kda_scan_body.cuh"

namespace kda {

namespace {

constexpr int LPT_MAX_DOCS = 64;  // documents ranked by length (more keep the index order)

// The document of rank r when the n documents are ordered by chunk count, the
// longest first (ties by index).  Every thread of the block gets the answer.
__device__ __forceinline__ int doc_of_rank(const Plan &p, int n, int r) {
    __shared__ int s_nc[LPT_MAX_DOCS];
    __shared__ int s_doc;
    const int t = threadIdx.x;
    if (t == 0) s_doc = r;
    if (t < n) s_nc[t] = p.doc_off[t + 1] - p.doc_off[t];
    __syncthreads();
    if (t < n) {
        const int mine = s_nc[t];
        int rank = 0;
        for (int e = 0; e < n; ++e) rank += (s_nc[e] > mine) || (s_nc[e] == mine && e < t);
        if (rank == r) s_doc = t;
    }
    __syncthreads();
    return s_doc;
}

template <int N, int STAGES, int TPR, bool EMIT_O, bool CKPT>
__global__ void __launch_bounds__(ScanCfg<N, TPR, EMIT_O>::THREADS, 1) scan_tc_kernel(ScanArgs a, int lpt) {
    extern __shared__ uint8_t smraw[];
    int unit = blockIdx.x, h = blockIdx.y, cb = blockIdx.z;
    if (lpt) {
        unit = doc_of_rank(a.plan, a.n_units, blockIdx.z);
        h = blockIdx.x;
        cb = blockIdx.y;
    }
    scan_block<N, STAGES, TPR, EMIT_O, CKPT>(a, unit, h, cb * (N / 16), smraw, nullptr);
}

template <int N, int STAGES, int TPR, bool EMIT_O = false, bool CKPT = !EMIT_O>
int launch_n(const ScanArgs &a, cudaStream_t s) {
    auto kern = scan_tc_kernel<N, STAGES, TPR, EMIT_O, CKPT>;
    const size_t smem = scan_tc_smem_bytes<N, STAGES, EMIT_O>();
    if (prepare_kernel((const void *)kern, (int)smem, ScanCfg<N, TPR, EMIT_O>::THREADS, nullptr) != KDA_OK)
        return KDA_ERR_CUDA;
    const int lpt = a.mode == SCAN_DOCS && !a.plan.uniform && a.n_units > 1 && a.n_units <= LPT_MAX_DOCS;
    const dim3 grid = lpt ? dim3(a.H, a.ncols / N, a.n_units) : dim3(a.n_units, a.H, a.ncols / N);
    kern<<<grid, ScanCfg<N, TPR, EMIT_O>::THREADS, smem, s>>>(a, lpt);
    note_launch("scan_tc", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

int launch_scan_tc(const ScanArgs &a, int n_sm, cudaStream_t s) {
    if (a.n_units == 0) return KDA_OK;
    // Few independent column slices: narrow blocks spread the chains over more
    // SMs.  Many: wider blocks amortise the per-chunk latency.
    const long long slices16 = (long long)a.n_units * a.H * (a.ncols / 16);
    if (slices16 <= 2LL * n_sm) {
        const int rc = launch_n<16, 3, 1>(a, s);
        // the outputs of every chunk, from the entering states the scan stored
        return (rc || !a.o || a.phase == 1) ? rc : launch_out_tc(a.plan, a.H, a.records, a.o, n_sm, s);
    }
    // many chains: 64-column blocks that also form the outputs of their columns
    // (checkpoints in an instantiation of their own)
    if (a.o && a.phase != 1 && a.ncols == D)
        return a.ckpt ? launch_n<64, 3, 2, true, true>(a, s) : launch_n<64, 3, 2, true, false>(a, s);
    // the segment pairs (256 columns: values and transition): 128-column blocks,
    // so that each chunk's G is read twice per (segment, head), not four times
    if (a.phase == 1 && a.ncols == 2 * D) return launch_n<128, 2, 4>(a, s);
    const int rc = launch_n<64, 2, 2>(a, s);
    return (rc || !a.o || a.phase == 1) ? rc : launch_out_tc(a.plan, a.H, a.records, a.o, n_sm, s);
}

}  // namespace kda
