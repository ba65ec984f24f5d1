// kda_noalloc.cu -- kda_chunk_fwd for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device workspace at call time: an
// engine that reserved the whole device for its own memory pool before this
// library was loaded, or host code on a latency-critical path where a
// cudaMalloc (which may synchronise the device) is not acceptable.  For them
// kda_chunk_fwd_noalloc runs the same kernels as kda_chunk_fwd with the
// workspace taken from a fixed array in device global memory that the library
// module itself owns.  The array is KDA_NOALLOC_SCRATCH_BYTES long and every
// GPU that loads the library holds it until the process exits.
//
// Nothing here allocates: the device address of the array is looked up once
// per device (the first call on that device, with that device current) and
// cached together with the CUDA context it belongs to; a call under another
// context (after a device reset, say) looks it up again.  Every other call
// only launches kernels and issues one cudaMemsetAsync of the workspace
// header.  All calls share the one array, so calls whose executions overlap on
// the GPU race on it; the caller must order them (for example by issuing them
// on one stream).  The array's first word is the device error word of the
// last call (kda_noalloc_read_device_error reads it).
#include <cuda.h>  // CUcontext / CUresult types only: the driver function comes through the runtime

#include <cstring>
#include <mutex>

#include "kda_internal.cuh"

using namespace kda;

namespace {

// The scratch array.  In host code this name is only a stand-in for the
// device symbol; kernels must be given the address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
void *g_scratch_addr[MAX_DEVICES] = {nullptr};
CUcontext g_scratch_ctx[MAX_DEVICES] = {nullptr};
std::mutex g_scratch_mu;

// cuCtxGetCurrent, fetched through the runtime so that the library keeps no
// link-time dependency on the driver library.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return (CtxGetCurrentFn)f;
    }();
    return fn;
}

// Device address of the scratch array on the current device, looked up on the
// first call under the current context of that device.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KDA_ERR_CUDA;
    CtxGetCurrentFn get_ctx = ctx_get_current();
    if (!get_ctx) return KDA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
        // the lookup also makes the device's primary context current when no
        // runtime call has done so yet
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
        if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return KDA_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" int kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *z,
                                     const float *A, const float *beta, const int32_t *cu_seqlens,
                                     int n_seqs, int64_t T_total, int H, int Dm, int dtype, float g_min,
                                     const float *init_state, void *o, float *final_state,
                                     int flags, kda_stream_t stream) {
    // the same argument checks as kda_chunk_fwd
    int rc = check_prefill(q, k, v, z, A, beta, cu_seqlens, n_seqs, T_total, H, Dm, dtype, g_min, o, flags);
    if (rc) return rc;
    // the call must fit the fixed scratch array: this path runs the prep and
    // scan kernels one after the other (no fused launch, no segments), whose
    // workspace is the layout without segment buffers
    const Workspace w = workspace_layout(T_total, H, n_seqs, 0, dtype);
    if (w.total > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;

    void *ws = nullptr;
    rc = scratch_address(&ws);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    note_begin(s);

    // chunk plan; the header (error word, chunk count) is cleared because the
    // array keeps whatever the previous call left in it
    Plan p;
    memset(&p, 0, sizeof(p));
    char *base = (char *)ws;
    p.n_seqs = n_seqs;
    p.err = (int32_t *)base;
    p.table = (const ChunkInfo *)(base + w.off_table);
    p.doc_off = (const int32_t *)(base + w.off_doc);
    p.n_chunks = (const int32_t *)(base + 4);
    p.flags = flags;
    p.wait_budget = wait_budget();
    if (cudaMemsetAsync(base, 0, 8, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (!cu_seqlens) {
        p.uniform = 1;
        p.seq_len = (int)(T_total / n_seqs);
        p.chunks_per_seq = (p.seq_len + C - 1) / C;
        p.max_chunks = n_seqs * p.chunks_per_seq;
    } else {
        p.max_chunks = w.max_chunks;
        if ((rc = launch_plan(cu_seqlens, n_seqs, T_total, ws, w, s))) return rc;
    }

    void *records = base + w.off_rec;
    if (dtype == KDA_BF16)
        rc = launch_prep_tc(q, k, v, z, A, beta, T_total, H, g_min, p, records, device_sm_count(), s);
    else
        rc = launch_prep_simt(q, k, v, z, A, beta, H, dtype, g_min, p, records, s);
    if (rc) return rc;
    ScanArgs a;
    memset(&a, 0, sizeof(a));
    a.plan = p;
    a.H = H;
    a.records = records;
    a.mode = SCAN_DOCS;
    a.n_units = n_seqs;
    a.ncols = D;
    a.phase = 0;
    a.init_state = init_state;
    a.o = o;
    a.final_state = final_state;
    return dtype == KDA_BF16 ? launch_scan_tc(a, device_sm_count(), s) : launch_scan_simt(a, dtype, s);
}

extern "C" int kda_noalloc_read_device_error(int32_t *code, kda_stream_t stream) {
    if (!code) return KDA_ERR_INVALID_ARG;
    void *ws = nullptr;
    const int rc = scratch_address(&ws);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    *code = h;
    return KDA_OK;
}
