// kda_compose.cu -- sequential composition of segment pairs (phase 2 of the
// intra-device segment scan).
//
// "Kimi K3 模型结构（7）：结构决定系统", sections "公式 (17) 的推导" (steps 2-4):
// a segment maps an entering state S to M S + S~, so the entering state of
// segment i+1 is S_in[i+1] = M_i S_in[i] + S~_i, evaluated in order from
// S_in[0] = 0 (the first segment always opens a document, where its pair
// already has M = 0, section "文档边界").  The page runs this as a sequential
// prefix scan because each step costs about one chunk; here a block owns 16
// state columns of one head (columns are independent), so all heads and column
// slices run in parallel while the segment chain stays sequential.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int CMP_THREADS = 256;
constexpr int CMP_NC = 16;
constexpr int KSLAB = 32;

__global__ void __launch_bounds__(CMP_THREADS)
compose_kernel(int H, int n_seg, const float *__restrict__ pairs, float *__restrict__ s_enter) {
    __shared__ __align__(16) float S[D][CMP_NC + 1];
    __shared__ __align__(16) float Ms[D][KSLAB + 4];
    const int h = blockIdx.x, col0 = blockIdx.y * CMP_NC, tid = threadIdx.x;
    const int row = tid >> 1, cc = (tid & 1) * 8;
    for (int idx = tid; idx < D * CMP_NC; idx += CMP_THREADS) S[idx / CMP_NC][idx % CMP_NC] = 0.f;
    __syncthreads();
    const size_t mat = (size_t)D * D;
    for (int i = 0; i < n_seg; ++i) {
        float *dst = s_enter + ((size_t)h * n_seg + i) * mat;
        for (int idx = tid; idx < D * CMP_NC; idx += CMP_THREADS) {
            const int r = idx / CMP_NC, j = idx % CMP_NC;
            dst[(size_t)r * D + col0 + j] = S[r][j];
        }
        if (i == n_seg - 1) break;
        const float *M = pairs + ((size_t)(0 * H + h) * n_seg + i) * mat;
        const float *St = pairs + ((size_t)(1 * H + h) * n_seg + i) * mat;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = St[(size_t)row * D + col0 + cc + j];
        for (int k0 = 0; k0 < D; k0 += KSLAB) {
            __syncthreads();
            for (int idx = tid; idx < D * (KSLAB / 4); idx += CMP_THREADS) {
                const int r = idx / (KSLAB / 4), c4 = (idx % (KSLAB / 4)) * 4;
                *reinterpret_cast<float4 *>(&Ms[r][c4]) =
                    *reinterpret_cast<const float4 *>(M + (size_t)r * D + k0 + c4);
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < KSLAB; ++kk) {
                const float m = Ms[row][kk];
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(m, S[k0 + kk][cc + j], acc[j]);
            }
        }
        __syncthreads();  // everyone finished reading S
#pragma unroll
        for (int j = 0; j < 8; ++j) S[row][cc + j] = acc[j];
        __syncthreads();
    }
}

}  // namespace

int launch_compose(const Plan &p, int H, int n_seg, const float *pairs, float *s_enter,
                   cudaStream_t s) {
    (void)p;
    if (n_seg <= 0) return KDA_OK;
    dim3 grid(H, D / CMP_NC);
    compose_kernel<<<grid, CMP_THREADS, 0, s>>>(H, n_seg, pairs, s_enter);
    note_launch("compose", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
