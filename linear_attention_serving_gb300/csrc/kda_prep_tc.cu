// kda_prep_tc.cu -- the prep kernel for bf16 inputs (device code in
// kda_prep_body.cuh): persistent blocks, one per SM, over all (chunk, head)
// units; the input tiles come in through the tensor maps of kda_tma.cu.
#include "kda_prep_body.cuh"

namespace kda {

namespace {

template <bool OPTS>
__global__ void __launch_bounds__(PT_THREADS, 1)
prep_tc_kernel(const __grid_constant__ InputMaps maps, const float *__restrict__ A, const float *__restrict__ beta,
               int H, float g_min, Plan plan, char *__restrict__ records) {
    extern __shared__ uint8_t smraw[];
    prep_blocks<OPTS>(&maps, A, beta, H, g_min, plan, records, smraw, blockIdx.x, gridDim.x, nullptr);
}

}  // namespace

int launch_prep_tc(const void *q, const void *k, const void *v, const float *z, const float *A,
                   const float *beta, int64_t T_total, int H, float g_min, const Plan &p, void *records, int n_sm,
                   cudaStream_t s) {
    const long long units = (long long)p.max_chunks * H;
    if (units == 0 || T_total == 0) return KDA_OK;
    InputMaps maps;
    int rc = make_input_maps(q, k, v, z, T_total, H, &maps);
    if (rc) return rc;
    auto kern = p.flags ? prep_tc_kernel<true> : prep_tc_kernel<false>;
    if (prepare_kernel((const void *)kern, (int)PREP_TC_SMEM, PT_THREADS, nullptr) != KDA_OK) return KDA_ERR_CUDA;
    const int grid = (int)(units < n_sm ? units : n_sm);
    kern<<<grid, PT_THREADS, PREP_TC_SMEM, s>>>(maps, A, beta, H, g_min, p, (char *)records);
    note_launch("prep_tc", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
