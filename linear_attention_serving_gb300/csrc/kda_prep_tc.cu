// kda_prep_tc.cu -- per-(chunk, head) preparation for bf16 inputs, with the
// contractions on tcgen05 tensor cores.
//
// For one 64-token chunk of one head this computes everything of the chunk
// form that does not depend on the entering state ("Kimi K3: the Manos, the
// Mythos ..." (SemiAnalysis), "FlashKDA 算法": a = exp(cumsum g), K_decay,
// Q_decay, K_inv, K_restore, L, INV = (I+L)^-1, M_qk), folded into the record
// the scan consumes:  W = INV Diag(beta) K_decay,  U0 = INV Diag(beta) V,
// Q' = Q_decay - M_qk W,  O0 = M_qk U0,  K_restore^T,  a_C.
//
// Steps (one block per SM, walking (chunk, head) units):
//  1. each thread owns one channel c and 32 consecutive tokens: it reads z, q,
//     k, v straight from global memory, applies the gate of "Kimi K3 模型结构
//     （2）" eq. (5), takes the cumulative log decay inside each 16-token tile
//     ("数值问题：1/Γ 会溢出") and e_i = exp(G_i - G_{tile start}) in (e^-80, 1];
//  2. it writes the factored MMA operands (bf16, K-major, 128-byte swizzle):
//     for key tile q the query-side rows x_i e_i F_pq (x = q and x = k, rows of
//     tiles p >= q only) and the key-side rows k_j exp(Delta_q) / e_j, where
//     F_pp = exp(-Delta_p) <= e^80 and F_pq = prod_{q<t<p} exp(Delta_t) <= 1;
//     and the operands Diag(beta) K_decay, Diag(beta) V, K_restore^T, Q_decay;
//  3. four M = 128, N = 16 MMAs give M_qk and A_kk block column by block
//     column (TMEM), from which L = StrictTril(Diag(beta) A_kk) and M_qk;
//  4. INV = (I + L)^-1 and Z = M_qk INV in fp32 CUDA cores ("UT 变换");
//  5. one M = 128, N = 256, K = 64 MMA: [INV ; Z] [Diag(beta) K_decay | Diag(beta) V]
//     = [W | U0 ; M_qk W | O0];
//  6. epilogue: Q' = Q_decay - M_qk W; the record is staged in shared memory
//     and written with bulk copies that overlap the next unit.
// Every wait is bounded; a timeout records KDA_DEVERR_TIMEOUT and ends the block.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tri.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int PT_THREADS = 256;

// shared-memory map (bytes from a 1024-aligned base)
constexpr int SM_AREG = 0;           // A_q images (2 k-blocks x 384 rows x 128 B); later fp32
                                     // L | M_qk | INV | Z | tmp; later the output staging
constexpr int SM_AREG_KB = 49152;    // offset of the second k-block of the A_q images
constexpr int SM_BQ = 98304;         // key-side images, 4 x (2 k-blocks x 16 rows x 128 B)
constexpr int SM_B2 = 114688;        // [Diag(beta) K_decay | Diag(beta) V]^T: 256 rows x 64 tokens
constexpr int SM_A2 = 147456;        // [INV ; Z]: 128 rows x 64
constexpr int SM_KRT = 163840;       // K_restore^T: 128 channels x 64 tokens
constexpr int SM_QD = 180224;        // Q_decay bf16 [64][128] row-major
constexpr int SM_MISC = 196608;      // beta [64] | Delta [4][128] | a_C [128]
constexpr int SM_BYTES = 200704;
constexpr size_t PREP_TC_SMEM = SM_BYTES + 1024;

// staging of the output record inside SM_AREG
constexpr int ST_A1 = 0;
constexpr int ST_U0 = 32768;
constexpr int ST_O0 = 49152;

// fp32 matrices inside SM_AREG (row stride TRI_LD floats)
constexpr int MAT_BYTES = 64 * TRI_LD * 4;
constexpr int SM_L = 0;
constexpr int SM_MQK = MAT_BYTES;
constexpr int SM_INV = 2 * MAT_BYTES;
constexpr int SM_Z = 3 * MAT_BYTES;
constexpr int SM_TMP = 4 * MAT_BYTES;

__device__ __forceinline__ int arow_base(int q) { return q == 0 ? 0 : (q == 1 ? 128 : (q == 2 ? 224 : 288)); }

__device__ __forceinline__ uint32_t swz(int row, int cc) {  // cc: column within a 64-column k-block
    return (uint32_t)(row * 128 + ((((cc >> 3) ^ (row & 7)) & 7) << 4) + (cc & 7) * 2);
}

__global__ void __launch_bounds__(PT_THREADS, 1)
prep_tc_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
               const __nv_bfloat16 *__restrict__ v, const float *__restrict__ z, const float *__restrict__ A,
               const float *__restrict__ beta, int H, float g_min, Plan plan, char *__restrict__ records) {
    extern __shared__ uint8_t smraw[];
    __shared__ uint64_t mbar_p, mbar_e;
    __shared__ uint32_t tmem_slot;

    if (plan_failed(plan)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = tid & 127, half = tid >> 7;
    uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    float *sbeta = reinterpret_cast<float *>(sm + SM_MISC);
    float *sDelta = sbeta + 64;           // [4][128]
    float *sAC = sDelta + 4 * 128;        // [128]

    if (tid == 0) {
        mbar_init(&mbar_p, 1);
        mbar_init(&mbar_e, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;

    const int n_units = plan_n_chunks(plan) * H;
    bool timed_out = false;
    int it = 0;
    for (int u = blockIdx.x; u < n_units && !timed_out; u += gridDim.x, ++it) {
        const int cidx = u / H, h = u - cidx * H;
        const ChunkInfo ci = plan_chunk(plan, cidx);
        const int t0 = ci.tok, len = ci.len;
        const float eA = expf(A[h]);
        const int r0 = half * 32;  // first token of this thread

        // ---- 1. inputs of channel c, tokens r0 .. r0+31 (rows past the end are k = q = v = 0, g = 0)
        float g[32];
        __nv_bfloat162 qp[16], kp[16], vp[16];
#pragma unroll
        for (int r = 0; r < 32; r += 2) {
            const int i = r0 + r;
            const size_t a0 = ((size_t)(t0 + i) * H + h) * D + c;
            const size_t a1 = a0 + (size_t)H * D;
            const bool ok0 = i < len, ok1 = i + 1 < len;
            const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
            qp[r / 2] = __halves2bfloat162(ok0 ? q[a0] : zero, ok1 ? q[a1] : zero);
            kp[r / 2] = __halves2bfloat162(ok0 ? k[a0] : zero, ok1 ? k[a1] : zero);
            vp[r / 2] = __halves2bfloat162(ok0 ? v[a0] : zero, ok1 ? v[a1] : zero);
            g[r] = ok0 ? z[a0] : 0.f;
            g[r + 1] = ok1 ? z[a1] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) g[r] = (r0 + r < len) ? kda_gate(g_min, eA, g[r]) : 0.f;
        // within-tile cumulative log decay r_i, tile totals Delta_p
        float e[32];
        float dl0 = 0.f, dl1 = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) { dl0 += g[r]; e[r] = dl0; }
#pragma unroll
        for (int r = 16; r < 32; ++r) { dl1 += g[r]; e[r] = dl1; }
        // the previous unit's bulk stores must have read the staging area before it is reused
        if (tid == 0) bulk_wait_read_all();
        sDelta[(2 * half) * 128 + c] = dl0;
        sDelta[(2 * half + 1) * 128 + c] = dl1;
        if (tid < 64) sbeta[tid] = tid < len ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
        __syncthreads();
        float Dl[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) Dl[t] = sDelta[t * 128 + c];
        float eD[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) eD[t] = expf(Dl[t]);
#pragma unroll
        for (int r = 0; r < 32; ++r) e[r] = expf(e[r]);
        if (half == 1 && tid - 128 == c) sAC[c] = eD[0] * eD[1] * eD[2] * eD[3];

        // ---- 2. operands
#pragma unroll
        for (int pl = 0; pl < 2; ++pl) {
            const int p = 2 * half + pl;  // this thread's tile
            const float eDinv = expf(-Dl[p]);
            float ePfx = 1.f, eSfx = 1.f;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (t < p) ePfx *= eD[t];
                if (t > p) eSfx *= eD[t];
            }
            float F[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                float f = 1.f;
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    if (t > qq && t < p) f *= eD[t];
                F[qq] = (qq == p) ? eDinv : f;
            }
            const int kb = c >> 6, cc = c & 63;
            __align__(16) __nv_bfloat16 bkd[16], bv[16], bkr[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const int r = pl * 16 + rr, i = r0 + r;
                const float2 qf = __bfloat1622float2(qp[r / 2]);
                const float2 kf2 = __bfloat1622float2(kp[r / 2]);
                const float2 vf = __bfloat1622float2(vp[r / 2]);
                const float qv = (r & 1) ? qf.y : qf.x, kv = (r & 1) ? kf2.y : kf2.x, vv = (r & 1) ? vf.y : vf.x;
                const float ei = e[r];
                const float qe = qv * ei, ke = kv * ei;
                // query-side rows for key tiles q <= p
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    if (qq > p) continue;
                    const int nq = 16 * (4 - qq);
                    const int rowQ = arow_base(qq) + (i - 16 * qq);
                    const int rowK = rowQ + nq;
                    uint8_t *base = sm + SM_AREG + kb * SM_AREG_KB;
                    *reinterpret_cast<__nv_bfloat16 *>(base + swz(rowQ, cc)) = __float2bfloat16_rn(qe * F[qq]);
                    *reinterpret_cast<__nv_bfloat16 *>(base + swz(rowK, cc)) = __float2bfloat16_rn(ke * F[qq]);
                }
                // key side of tile p: k_j exp(Delta_p) / e_j  (<= 1)
                const float kfac = kv * (eD[p] / ei);
                *reinterpret_cast<__nv_bfloat16 *>(sm + SM_BQ + p * 4096 + kb * 2048 + swz(i - 16 * p, cc)) =
                    __float2bfloat16_rn(kfac);
                const float b = sbeta[i];
                bkd[rr] = __float2bfloat16_rn(b * ePfx * ke);   // Diag(beta) K_decay
                bv[rr] = __float2bfloat16_rn(b * vv);           // Diag(beta) V
                bkr[rr] = __float2bfloat16_rn(eSfx * kfac);     // K_restore = exp(G_last - G_j) k_j
                *reinterpret_cast<__nv_bfloat16 *>(sm + SM_QD + (i * D + c) * 2) = __float2bfloat16_rn(ePfx * qe);
            }
            // transposed rows (row = channel, column = token), 8 tokens per 16-byte store
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
                const int i0 = r0 + pl * 16 + g8 * 8;
                *reinterpret_cast<uint4 *>(sm + SM_B2 + c * 128 + ((((i0 >> 3) ^ (c & 7)) & 7) << 4)) =
                    *reinterpret_cast<const uint4 *>(bkd + g8 * 8);
                *reinterpret_cast<uint4 *>(sm + SM_B2 + (128 + c) * 128 + ((((i0 >> 3) ^ ((128 + c) & 7)) & 7) << 4)) =
                    *reinterpret_cast<const uint4 *>(bv + g8 * 8);
                *reinterpret_cast<uint4 *>(sm + SM_KRT + c * 128 + ((((i0 >> 3) ^ (c & 7)) & 7) << 4)) =
                    *reinterpret_cast<const uint4 *>(bkr + g8 * 8);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 3. A_qk / A_kk block columns on the tensor cores
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t ID16 = idesc_bf16_f32(128, 16);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const int kb = s >> 2, w = s & 3;
                    const uint64_t ad = sdesc_sw128(smem_u32(sm + SM_AREG + kb * SM_AREG_KB + arow_base(qq) * 128 + w * 32));
                    const uint64_t bd = sdesc_sw128(smem_u32(sm + SM_BQ + qq * 4096 + kb * 2048 + w * 32));
                    mma_bf16(tmem + 16 * qq, ad, bd, ID16, s > 0);
                }
            }
            mma_commit(&mbar_p);
        }
        bool ok = mbar_wait(&mbar_p, (uint32_t)(it & 1));
        __syncwarp();
        tc_fence_after();
        float *Lm = reinterpret_cast<float *>(sm + SM_AREG + SM_L);
        float *Mq = reinterpret_cast<float *>(sm + SM_AREG + SM_MQK);
        float *INV = reinterpret_cast<float *>(sm + SM_AREG + SM_INV);
        float *Zm = reinterpret_cast<float *>(sm + SM_AREG + SM_Z);
        float *tmp = reinterpret_cast<float *>(sm + SM_AREG + SM_TMP);
        {
            // warps 0-3 read key tiles 0, 1; warps 4-7 key tiles 2, 3 (all 128 TMEM lanes each)
            const int r = (warp & 3) * 32 + lane;
#pragma unroll
            for (int qi = 0; qi < 2; ++qi) {
                const int qq = half * 2 + qi;
                float d[16];
                tmem_ld16(tmem + lane_off + 16 * qq, d);
                tmem_ld_wait();
                const int nq = 16 * (4 - qq);
                if (r < nq) {
                    const int i = 16 * qq + r;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) Mq[i * TRI_LD + 16 * qq + jj] = (16 * qq + jj <= i) ? d[jj] : 0.f;
                } else if (r < 2 * nq) {
                    const int i = 16 * qq + (r - nq);
                    const float b = sbeta[i];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) Lm[i * TRI_LD + 16 * qq + jj] = (16 * qq + jj < i) ? b * d[jj] : 0.f;
                }
            }
        }
        // blocks above the block diagonal are zero in L, M_qk and INV
        for (int idx = tid; idx < 64 * 64; idx += PT_THREADS) {
            const int i = idx >> 6, j = idx & 63;
            if ((j >> 4) > (i >> 4)) {
                Lm[i * TRI_LD + j] = 0.f;
                Mq[i * TRI_LD + j] = 0.f;
            }
            INV[i * TRI_LD + j] = 0.f;
        }
        tc_fence_before();
        ok = !__syncthreads_or(!ok);
        if (!ok) { timed_out = true; break; }

        // ---- 4. INV = (I + L)^-1 and Z = M_qk INV (fp32)
        tri_inverse(Lm, INV, tmp, tid, PT_THREADS);
        for (int idx = tid; idx < 64 * 64; idx += PT_THREADS) {
            const int i = idx >> 6, j = idx & 63;
            float acc = 0.f;
            for (int s = j; s <= i; ++s) acc = fmaf(Mq[i * TRI_LD + s], INV[s * TRI_LD + j], acc);
            Zm[i * TRI_LD + j] = acc;  // zero above the diagonal (empty sum)
        }
        __syncthreads();
        // A2 = [INV ; Z] as a bf16 K-major image (128 rows x 64)
        for (int idx = tid; idx < 128 * 8; idx += PT_THREADS) {
            const int row = idx >> 3, g8 = idx & 7;
            const float *src = (row < 64 ? INV + row * TRI_LD : Zm + (row - 64) * TRI_LD) + g8 * 8;
            __align__(16) __nv_bfloat16 b8[8];
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) b8[e8] = __float2bfloat16_rn(src[e8]);
            *reinterpret_cast<uint4 *>(sm + SM_A2 + row * 128 + (((g8 ^ (row & 7)) & 7) << 4)) =
                *reinterpret_cast<const uint4 *>(b8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 5. [INV ; Z] [Diag(beta) K_decay | Diag(beta) V]  (M = 128, N = 256, K = 64)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t ID256 = idesc_bf16_f32(128, 256);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t ad = sdesc_sw128(smem_u32(sm + SM_A2 + s * 32));
                const uint64_t bd = sdesc_sw128(smem_u32(sm + SM_B2 + s * 32));
                mma_bf16(tmem, ad, bd, ID256, s > 0);
            }
            mma_commit(&mbar_e);
        }
        ok = mbar_wait(&mbar_e, (uint32_t)(it & 1));
        __syncwarp();
        tc_fence_after();

        // ---- 6. epilogue into the staging area
        {
            const int r = (warp & 3) * 32 + lane;  // TMEM lane = row of [W | U0 ; M_qk W | O0]
            const int col_base = half * 128;       // warps 0-3: W | M_qk W, warps 4-7: U0 | O0
#pragma unroll 1
            for (int cb = 0; cb < 8; ++cb) {
                float d[16];
                tmem_ld16(tmem + lane_off + col_base + 16 * cb, d);
                tmem_ld_wait();
                __align__(16) __nv_bfloat16 o16[16];
                if (half == 0) {
                    if (r < 64) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) o16[j] = __float2bfloat16_rn(d[j]);
                    } else {
                        const __nv_bfloat16 *qd = reinterpret_cast<const __nv_bfloat16 *>(sm + SM_QD) + (r - 64) * D + 16 * cb;
#pragma unroll
                        for (int j = 0; j < 16; ++j) o16[j] = __float2bfloat16_rn(__bfloat162float(qd[j]) - d[j]);
                    }
                    const int col = 16 * cb;
                    *reinterpret_cast<uint4 *>(sm + SM_AREG + ST_A1 + sw128_offset(r, col, 128)) =
                        *reinterpret_cast<const uint4 *>(o16);
                    *reinterpret_cast<uint4 *>(sm + SM_AREG + ST_A1 + sw128_offset(r, col + 8, 128)) =
                        *reinterpret_cast<const uint4 *>(o16 + 8);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) o16[j] = __float2bfloat16_rn(d[j]);
                    uint8_t *dst = sm + SM_AREG + (r < 64 ? ST_U0 : ST_O0) + slice_offset(r & 63, 16 * cb);
                    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(o16);
                    *reinterpret_cast<uint4 *>(dst + 16) = *reinterpret_cast<const uint4 *>(o16 + 8);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = !__syncthreads_or(!ok);
        if (!ok) { timed_out = true; break; }
        if (tid == 0) {
            char *rec = records + ((size_t)cidx * H + h) * REC_BF16_BYTES;
            bulk_s2g(rec + REC_BF16_A1, sm + SM_AREG + ST_A1, 32768);
            bulk_s2g(rec + REC_BF16_KRT, sm + SM_KRT, 16384);
            bulk_s2g(rec + REC_BF16_AC, sAC, 512);
            bulk_s2g(rec + REC_BF16_U0, sm + SM_AREG + ST_U0, 16384);
            bulk_s2g(rec + REC_BF16_O0, sm + SM_AREG + ST_O0, 16384);
            bulk_commit();
        }
    }
    if (tid == 0) {
        bulk_wait_all();
        if (timed_out) atomicOr(plan.err, KDA_DEVERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

int launch_prep_tc(const void *q, const void *k, const void *v, const float *z, const float *A,
                   const float *beta, int H, float g_min, const Plan &p, void *records, int n_sm,
                   cudaStream_t s) {
    const long long units = (long long)p.max_chunks * H;
    if (units == 0) return KDA_OK;
    if (cudaFuncSetAttribute(prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PREP_TC_SMEM) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    const int grid = (int)(units < n_sm ? units : n_sm);
    prep_tc_kernel<<<grid, PT_THREADS, PREP_TC_SMEM, s>>>((const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                                                          (const __nv_bfloat16 *)v, z, A, beta, H, g_min, p,
                                                          (char *)records);
    note_launch("prep_tc", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
