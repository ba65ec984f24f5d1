// kda_fused_tc.cu -- bf16 prefill as one cooperative launch: the prep and the
// state chain run at the same time on different SMs.
//
// The chain of a head is sequential in the chunks ("Kimi K3 模型结构（2）",
// "块间递推与块内输出") and keeps only a few SMs busy, while the per-(chunk, head)
// prep is parallel work for the whole GPU.  Run one after the other, the chain
// adds its full latency to the prep's time.  Here the first blocks of the grid
// run the chains (64 state columns each, kda_scan_body.cuh) and the others the
// prep (kda_prep_body.cuh), in chunk-major unit order; a prep block publishes
// each finished record with a release flag, and a chain's producer waits for
// the flag (acquire, bounded) before copying the record.  The chain blocks
// start with one prep unit each, since their first records take a unit's
// time to appear anyway.  The launch is cooperative, so every block is
// resident and a waiting chain cannot starve the prep it waits for; the prep
// never waits for a chain.  The chain blocks also form the outputs
// O = O0 + Q' S of their columns (an M = 64 MMA issued right after the chain's
// own, drained by four output warps): a chain keeps pace with the prep, so
// the outputs cost no extra pass.
#include "kda_prep_body.cuh"
#include "kda_scan_body.cuh"

namespace kda {

namespace {

constexpr int FUSED_N = 64, FUSED_STAGES = 3, FUSED_TPR = 2;
constexpr int FUSED_SLICES = D / FUSED_N;  // chain blocks per (document, head)

// OPTS: input options; CKPT: state checkpoints (separate instantiations, so
// that the default launch keeps its registers).
template <bool OPTS, bool CKPT>
__global__ void __launch_bounds__(PT_THREADS, 1)
fused_tc_kernel(const __grid_constant__ InputMaps maps, const float *__restrict__ A, const float *__restrict__ beta,
                int H, float g_min, Plan plan, char *__restrict__ records, ScanArgs sa, int n_chain, int *ready) {
    extern __shared__ uint8_t smraw[];
    // A chain would only wait for its first records at the start, so each chain
    // block first prepares one unit (units 0 .. n_chain - 1); prep block j takes
    // units n_chain + j, n_chain + j + n_prep, ...  (One call site: the prep
    // code is inlined once.)
    const bool chain = (int)blockIdx.x < n_chain;
    prep_blocks<OPTS>(&maps, A, beta, H, g_min, plan, records, smraw, blockIdx.x,
                      chain ? (1 << 30) : (int)gridDim.x - n_chain, ready);
    if (chain) {
        fence_async_smem();
        __syncthreads();
        const int per_doc = H * FUSED_SLICES;
        const int doc = blockIdx.x / per_doc, rem = blockIdx.x - doc * per_doc;
        const int h = rem / FUSED_SLICES, zc = rem - h * FUSED_SLICES;
        scan_block<FUSED_N, FUSED_STAGES, FUSED_TPR, true, CKPT>(sa, doc, h, zc * (FUSED_N / 16), smraw, ready);
    }
}

}  // namespace

int launch_fused_tc(const void *q, const void *k, const void *v, const float *z, const float *A,
                    const float *beta, int64_t T_total, int H, float g_min, const ScanArgs &sa, int *ready, int n_sm,
                    cudaStream_t s, bool *used) {
    *used = false;
    const Plan &p = sa.plan;
    const long long n_chain = (long long)sa.n_units * H * FUSED_SLICES;
    // the chains may take at most a quarter of the SMs, and there must be units to prepare
    if (sa.mode != SCAN_DOCS || n_chain < 1 || n_chain > n_sm / 4 || (long long)p.max_chunks * H < 1) return KDA_OK;
    int dev = 0, coop = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
        return KDA_OK;
    constexpr size_t chain_smem = scan_tc_smem_bytes<FUSED_N, FUSED_STAGES, true>();
    static_assert(ScanCfg<FUSED_N, FUSED_TPR, true>::THREADS <= PT_THREADS, "chain block fits the prep's block");
    const size_t smem = PREP_TC_SMEM > chain_smem ? PREP_TC_SMEM : chain_smem;
    auto kern = p.flags ? (sa.ckpt ? fused_tc_kernel<true, true> : fused_tc_kernel<true, false>)
                        : (sa.ckpt ? fused_tc_kernel<false, true> : fused_tc_kernel<false, false>);
    if (prepare_kernel((const void *)kern, (int)smem, PT_THREADS, &per_sm) != KDA_OK) return KDA_ERR_CUDA;
    if (per_sm < 1) return KDA_OK;
    InputMaps maps;
    const int rc = make_input_maps(q, k, v, z, T_total, H, &maps);
    if (rc) return rc;
    char *records = (char *)sa.records;
    Plan plan = p;
    ScanArgs a = sa;
    int nc = (int)n_chain;
    void *args[] = {&maps, &A, &beta, &H, &g_min, &plan, &records, &a, &nc, &ready};
    const cudaError_t e = cudaLaunchCooperativeKernel((const void *)kern, dim3(n_sm), dim3(PT_THREADS),
                                                      args, smem, s);
    if (e != cudaSuccess) {
        cudaGetLastError();  // a cooperative launch that does not fit leaves the three-kernel path
        return e == cudaErrorCooperativeLaunchTooLarge ? KDA_OK : KDA_ERR_CUDA;
    }
    note_launch("fused_tc", s);
    *used = true;
    return KDA_OK;
}

}  // namespace kda
