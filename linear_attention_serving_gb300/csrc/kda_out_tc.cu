// kda_out_tc.cu -- the chunk outputs O = O0 + Q' S on tcgen05 tensor cores.
//
// "Kimi K3: the Manos, the Mythos ..." (SemiAnalysis), "FlashKDA 算法": the
// output of a chunk is O = Q_decay S + M_qk U with U = INV Diag(beta)(V -
// K_decay S); with the prep kernel's Q' = Q_decay - M_qk W and O0 = M_qk U0
// this is O = O0 + Q' S, S the state entering the chunk.  Once the scan has
// stored every chunk's entering state, the outputs of all (chunk, head) units
// are independent: one M = 64, N = 128, K = 128 MMA each.
//
// Persistent blocks of 288 threads walk the units with a two-stage pipeline:
// warp 8 (one thread) bulk-copies a unit's Q', O0 and S into shared memory and
// issues its MMA into one of two TMEM accumulators; warps 0-7 read the
// accumulator (lane quadrant = warp % 4, column half = warp / 4), add O0 and
// store the bf16 rows of o.  Every wait is bounded; a timeout records
// KDA_DEVERR_TIMEOUT and ends the block.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int OT_THREADS = 288;
constexpr int OT_EPI = 256;          // warps 0-7
constexpr int OT_STAGE = 65536;      // Q' (16 KB) | O0 (16 KB) | S (32 KB)
constexpr int OS_QP = 0, OS_O0 = 16384, OS_S = 32768;
constexpr size_t OT_SMEM = 2 * OT_STAGE + 1024;
static_assert(REC_BF16_S == REC_BF16_O0 + 16384, "O0 and S are copied together");

__global__ void __launch_bounds__(OT_THREADS, 1)
out_tc_kernel(Plan plan, int H, const char *__restrict__ records, __nv_bfloat16 *__restrict__ o) {
    extern __shared__ uint8_t smraw[];
    __shared__ uint64_t full_bar[2], empty_bar[2], mma_bar[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    if (plan_failed(plan)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
            mbar_init(&mma_bar[s], 1);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int n_units = plan_n_chunks(plan) * H;
    const int n_mine = blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (warp == 8) {
        // ------------------------------------------------------------ loads + MMA issue
        if (lane == 0) {
            bool timed_out = false;
            int loaded = 0;
            auto load = [&](int j) -> bool {
                const int st = j & 1;
                if (!mbar_wait(&empty_bar[st], (uint32_t)(((j >> 1) & 1) ^ 1))) return false;
                const int u = blockIdx.x + j * gridDim.x;
                const char *rec = records + (size_t)u * REC_BF16_BYTES;  // unit u = chunk * H + head
                uint8_t *stage = sm + st * OT_STAGE;
                mbar_expect_tx(&full_bar[st], 16384 + 49152);
                bulk_g2s(stage + OS_QP, rec + REC_BF16_QP, 16384, &full_bar[st]);
                bulk_g2s(stage + OS_O0, rec + REC_BF16_O0, 49152, &full_bar[st]);
                loaded = j + 1;
                return true;
            };
            constexpr uint32_t IDESC = idesc_bf16_f32_bmn(64, 128);
            if (n_mine > 0 && !load(0)) timed_out = true;
            for (int j = 0; j < n_mine && !timed_out; ++j) {
                if (j + 1 < n_mine && !load(j + 1)) { timed_out = true; break; }
                const int st = j & 1;
                if (!mbar_wait(&full_bar[st], (uint32_t)((j >> 1) & 1))) { timed_out = true; break; }
                if (*(volatile int *)&abort_flag) break;
                tc_fence_after();
                const uint8_t *stage = sm + st * OT_STAGE;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t ad = sdesc_sw128(smem_u32(stage + OS_QP + (k >> 2) * 8192 + (k & 3) * 32));
                    const uint64_t bd = sdesc_mn(smem_u32(stage + OS_S + k * 512), 4096, 256, SWZ_32B);
                    mma_bf16(tmem + st * 128, ad, bd, IDESC, k > 0);
                }
                mma_commit(&mma_bar[st]);
            }
            if (timed_out) {
                abort_flag = 1;
                atomicOr(plan.err, KDA_DEVERR_TIMEOUT);
            }
            // let the copies this thread started land before the block exits
            for (int j = loaded > 2 ? loaded - 2 : 0; j < loaded; ++j) mbar_wait(&full_bar[j & 1], (uint32_t)((j >> 1) & 1));
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int q4 = warp & 3, hf = warp >> 2;
        const int m = 16 * q4 + lane;  // token row of the chunk (lanes < 16)
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        for (int j = 0; j < n_mine; ++j) {
            const int st = j & 1;
            const int u = blockIdx.x + j * gridDim.x;
            const int c = u / H, h = u - c * H;
            bool ok = mbar_wait(&mma_bar[st], (uint32_t)((j >> 1) & 1)) && mbar_wait(&full_bar[st], (uint32_t)((j >> 1) & 1));
            __syncwarp();
            tc_fence_after();
            float d[64];
#pragma unroll
            for (int c16 = 0; c16 < 4; ++c16) tmem_ld16(tmem + lane_off + st * 128 + 64 * hf + 16 * c16, d + 16 * c16);
            tmem_ld_wait();
            uint4 o0[8];
            const uint8_t *stage = sm + st * OT_STAGE;
            if (lane < 16) {
#pragma unroll
                for (int h8 = 0; h8 < 8; ++h8)
                    o0[h8] = *reinterpret_cast<const uint4 *>(stage + OS_O0 + slice_offset(m, 64 * hf + 8 * h8, 64));
            }
            tc_fence_before();
            // every epilogue thread is done with this stage and accumulator (or all give up)
            if (bar_or(1, OT_EPI, !ok || *(volatile int *)&abort_flag)) {
                if (tid == 0) {
                    abort_flag = 1;
                    atomicOr(plan.err, KDA_DEVERR_TIMEOUT);
                }
                break;
            }
            if (tid == 0) mbar_arrive(&empty_bar[st]);
            const ChunkInfo ci = plan_chunk(plan, c);
            if (lane < 16 && m < ci.len) {
                __nv_bfloat16 *orow = o + ((size_t)(ci.tok + m) * H + h) * D + 64 * hf;
#pragma unroll
                for (int h8 = 0; h8 < 8; ++h8) {
                    const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&o0[h8]);
                    uint4 w;
                    __nv_bfloat162 *wp = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(x[e]);
                        wp[e] = __floats2bfloat162_rn(f.x + d[8 * h8 + 2 * e], f.y + d[8 * h8 + 2 * e + 1]);
                    }
                    *reinterpret_cast<uint4 *>(orow + 8 * h8) = w;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

int launch_out_tc(const Plan &p, int H, const void *records, void *o, int n_sm, cudaStream_t s) {
    const long long units = (long long)p.max_chunks * H;
    if (units == 0) return KDA_OK;
    if (cudaFuncSetAttribute(out_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)OT_SMEM) != cudaSuccess)
        return KDA_ERR_CUDA;
    const int grid = (int)(units < n_sm ? units : n_sm);
    out_tc_kernel<<<grid, OT_THREADS, OT_SMEM, s>>>(p, H, (const char *)records, (__nv_bfloat16 *)o);
    note_launch("out_tc", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
