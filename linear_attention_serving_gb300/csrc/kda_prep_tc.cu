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
// One block per SM walks (chunk, head) units with 512 threads:
//  1. column phase, thread = (channel c, 16-token sub-tile p): read z, k, v of
//     its tile and channel (the next unit's are prefetched while the current
//     one computes); gate of "Kimi K3 模型结构（2）" eq. (5); cumulative log
//     decay inside the tile ("数值问题：1/Γ 会溢出"), e_i = exp(G_i - G_{tile
//     start}) in (e^-80, 1], per-(tile, channel) factors; write the transposed
//     operands Diag(beta) K_decay, Diag(beta) V, K_restore^T (token-contiguous);
//  2. row phase, thread = (token i, 8 channels): the factored MMA operands
//     (bf16, K-major, 128-byte swizzle, 16-byte stores): for key tile q the
//     query-side rows x_i e_i F_pq (x = q and x = k, rows of tiles p >= q) and
//     the key side k_j exp(Delta_q) / e_j, with F_pp = exp(-Delta_p) <= e^80
//     and F_pq = prod_{q<t<p} exp(Delta_t) <= 1; and Q_decay;
//  3. four M = 128, N = 16 MMAs give M_qk and A_kk block column by block
//     column, from which L = StrictTril(Diag(beta) A_kk) and M_qk;
//  4. INV = (I + L)^-1 in fp32 CUDA cores ("UT 变换"); one MMA
//     [I ; M_qk] INV = [INV ; Z] gives Z = M_qk INV;
//  5. one M = 128, N = 256, K = 64 MMA:
//     [INV ; Z] [Diag(beta) K_decay | Diag(beta) V] = [W | U0 ; M_qk W | O0];
//  6. epilogue: Q' = Q_decay - M_qk W; the record is staged in shared memory
//     and written with bulk copies that overlap the next unit.
// Every wait is bounded; a timeout records KDA_DEVERR_TIMEOUT and ends the block.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tri.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int PT_THREADS = 512;

// shared-memory map (bytes from a 1024-aligned base)
constexpr int SM_AREG = 0;           // A_q images (2 k-blocks x 320 rows x 128 B); later fp32
                                     // L | M_qk | INV | tmp; later the output staging.  An
                                     // M = 128 read of the last image runs past its 32 valid
                                     // rows into the following bytes; those rows are ignored.
constexpr int SM_AREG_KB = 40960;    // offset of the second k-block of the A_q images
constexpr int SM_BQ = 81920;         // key-side images, 4 x (2 k-blocks x 16 rows x 128 B);
                                     // later [I ; M_qk] (128 rows x 64)
constexpr int SM_B2 = 98304;         // [Diag(beta) K_decay | Diag(beta) V]^T: 256 rows x 64 tokens
constexpr int SM_A2 = 131072;        // INV^T (64 rows x 64), then [INV ; Z] (128 rows x 64)
constexpr int SM_KRT = 147456;       // K_restore^T: 128 channels x 64 tokens
constexpr int SM_QD = 163840;        // Q_decay bf16 [64][128] row-major
constexpr int SM_MISC = 180224;      // beta [64] | Delta [4][128] | a_C [128]
constexpr int SM_E = 184320;         // e_i [64][128] fp32 (column phase -> row phase)
constexpr int SM_TAB = 217088;       // F [10][128] | exp(Delta) [4][128] | ePfx [4][128] fp32
constexpr int SM_BYTES = 226304;
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
constexpr int SM_TMP = 3 * MAT_BYTES;

__device__ __forceinline__ int arow_base(int q) { return q == 0 ? 0 : (q == 1 ? 128 : (q == 2 ? 224 : 288)); }

// byte offset of (row, cc) in a 128-byte-swizzled k-block; cc < 64
__device__ __forceinline__ uint32_t swz(int row, int cc) {
    return (uint32_t)(row * 128 + ((((cc >> 3) ^ (row & 7)) & 7) << 4) + (cc & 7) * 2);
}

// column phase inputs: z, k, v of tokens 16p .. 16p+15, channel c (rows past the end: zero)
__device__ __forceinline__ void load_col(const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                                         const float *__restrict__ z, int H, int h, int t0, int len, int p, int c,
                                         __nv_bfloat162 *kp, __nv_bfloat162 *vp, float *zf) {
    const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
#pragma unroll
    for (int rr = 0; rr < 16; rr += 2) {
        const int i = 16 * p + rr;
        const size_t a0 = ((size_t)(t0 + i) * H + h) * D + c;
        const size_t a1 = a0 + (size_t)H * D;
        const bool ok0 = i < len, ok1 = i + 1 < len;
        kp[rr / 2] = __halves2bfloat162(ok0 ? k[a0] : zero, ok1 ? k[a1] : zero);
        vp[rr / 2] = __halves2bfloat162(ok0 ? v[a0] : zero, ok1 ? v[a1] : zero);
        zf[rr] = ok0 ? z[a0] : 0.f;
        zf[rr + 1] = ok1 ? z[a1] : 0.f;
    }
}

// row phase inputs: 8 channels [8 g, 8 g + 8) of token i of q and k (zero past the end)
__device__ __forceinline__ void load_row(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                                         int H, int h, int t0, int len, int i, int g, uint4 &qr, uint4 &kr) {
    if (i < len) {
        const size_t a = ((size_t)(t0 + i) * H + h) * D + 8 * g;
        qr = *reinterpret_cast<const uint4 *>(q + a);
        kr = *reinterpret_cast<const uint4 *>(k + a);
    } else {
        qr = make_uint4(0, 0, 0, 0);
        kr = make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
    const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 t = __bfloat1622float2(b[j]);
        f[2 * j] = t.x;
        f[2 * j + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float *f) {
    uint4 u;
    __nv_bfloat162 *b = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    return u;
}

__device__ __forceinline__ int fpq(int p, int q) { return p * (p + 1) / 2 + q; }

__global__ void __launch_bounds__(PT_THREADS, 1)
prep_tc_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
               const __nv_bfloat16 *__restrict__ v, const float *__restrict__ z, const float *__restrict__ A,
               const float *__restrict__ beta, int H, float g_min, Plan plan, char *__restrict__ records) {
    extern __shared__ uint8_t smraw[];
    __shared__ uint64_t mbar_p, mbar_z, mbar_e;
    __shared__ uint32_t tmem_slot;

    if (plan_failed(plan)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = tid & 127, p = tid >> 7;  // channel, sub-tile
    uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    float *sbeta = reinterpret_cast<float *>(sm + SM_MISC);
    float *sDelta = sbeta + 64;     // [4][128]
    float *sAC = sDelta + 4 * 128;  // [128]

    if (tid == 0) {
        mbar_init(&mbar_p, 1);
        mbar_init(&mbar_z, 1);
        mbar_init(&mbar_e, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int lg = warp & 3;                       // TMEM lane group of this warp
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int r_lane = lg * 32 + lane;             // TMEM lane (row) this thread reads

    const int n_units = plan_n_chunks(plan) * H;
    // row-phase items of this thread: (token i, channel group g) for idx = tid, tid + 512
    const int ri0 = tid >> 4, rg0 = tid & 15, ri1 = ri0 + 32;
    __nv_bfloat162 kp[8], vp[8];
    float e[16];
    uint4 qr0, kr0, qr1, kr1;
    int u = blockIdx.x;
    ChunkInfo ci;
    if (u < n_units) {
        ci = plan_chunk(plan, u / H);
        load_col(k, v, z, H, u % H, ci.tok, ci.len, p, c, kp, vp, e);
        load_row(q, k, H, u % H, ci.tok, ci.len, ri0, rg0, qr0, kr0);
        load_row(q, k, H, u % H, ci.tok, ci.len, ri1, rg0, qr1, kr1);
    }
    bool timed_out = false;
    for (int it = 0; u < n_units && !timed_out; u += gridDim.x, ++it) {
        const int cidx = u / H, h = u - cidx * H;
        const int len = ci.len;
        const float eA = __expf(A[h]);

        // ---- 1. gate, within-tile cumulative log decay, tile total
        float dl = 0.f;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            const float gv = (16 * p + rr < len) ? __fdividef(g_min, 1.f + __expf(-eA * e[rr])) : 0.f;
            dl += gv;
            e[rr] = dl;
        }
        // the previous unit's bulk stores must have read the staging area first
        if (tid == 0) bulk_wait_read_all();
        sDelta[p * 128 + c] = dl;
        if (tid < 64) sbeta[tid] = tid < len ? beta[(size_t)(ci.tok + tid) * H + h] : 0.f;
        __syncthreads();
        float eD[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) eD[t] = __expf(sDelta[t * 128 + c]);
        float *sE = reinterpret_cast<float *>(sm + SM_E);
        float *sF = reinterpret_cast<float *>(sm + SM_TAB);
        float *sED = sF + 10 * 128;
        float *sPF = sED + 4 * 128;
        {
            // column phase: e_i, factors, transposed operands
            const float eDinv = __expf(-dl);
            float ePfx = 1.f, eSfx = 1.f;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (t < p) ePfx *= eD[t];
                if (t > p) eSfx *= eD[t];
            }
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                if (qq > p) continue;
                float f = 1.f;
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    if (t > qq && t < p) f *= eD[t];
                sF[fpq(p, qq) * 128 + c] = (qq == p) ? eDinv : f;
            }
            sED[p * 128 + c] = eD[p];
            sPF[p * 128 + c] = ePfx;
            if (p == 0) sAC[c] = eD[0] * eD[1] * eD[2] * eD[3];
            __align__(16) __nv_bfloat16 bkd[16], bv[16], bkr[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const int i = 16 * p + rr;
                const float ei = __expf(e[rr]);
                sE[i * 128 + c] = ei;
                const float2 kf2 = __bfloat1622float2(kp[rr / 2]);
                const float2 vf = __bfloat1622float2(vp[rr / 2]);
                const float kv = (rr & 1) ? kf2.y : kf2.x, vv = (rr & 1) ? vf.y : vf.x;
                const float b = sbeta[i];
                const float kfac = kv * __fdividef(eD[p], ei);  // k_j exp(Delta_p) / e_j, <= |k_j|
                bkd[rr] = __float2bfloat16_rn(b * ePfx * ei * kv);  // Diag(beta) K_decay
                bv[rr] = __float2bfloat16_rn(b * vv);               // Diag(beta) V
                bkr[rr] = __float2bfloat16_rn(eSfx * kfac);         // K_restore = exp(G_last - G_j) k_j
            }
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
                const int grp = 2 * p + g8;  // 8-token group
                *reinterpret_cast<uint4 *>(sm + SM_B2 + c * 128 + (((grp ^ (c & 7)) & 7) << 4)) =
                    *reinterpret_cast<const uint4 *>(bkd + g8 * 8);
                *reinterpret_cast<uint4 *>(sm + SM_B2 + (128 + c) * 128 + (((grp ^ (c & 7)) & 7) << 4)) =
                    *reinterpret_cast<const uint4 *>(bv + g8 * 8);
                *reinterpret_cast<uint4 *>(sm + SM_KRT + c * 128 + (((grp ^ (c & 7)) & 7) << 4)) =
                    *reinterpret_cast<const uint4 *>(bkr + g8 * 8);
            }
        }
        __syncthreads();
        // row phase: factored A_q rows, key-side rows, Q_decay, 8 channels per 16-byte store
#pragma unroll
        for (int item = 0; item < 2; ++item) {
            const int i = item ? ri1 : ri0, g = rg0;
            const int pi = i >> 4, kb = g >> 3, cc = (g & 7) * 8;
            float qv[8], kv[8], ev[8];
            unpack8(item ? qr1 : qr0, qv);
            unpack8(item ? kr1 : kr0, kv);
            const float4 e0 = *reinterpret_cast<const float4 *>(sE + i * 128 + 8 * g);
            const float4 e1 = *reinterpret_cast<const float4 *>(sE + i * 128 + 8 * g + 4);
            ev[0] = e0.x; ev[1] = e0.y; ev[2] = e0.z; ev[3] = e0.w;
            ev[4] = e1.x; ev[5] = e1.y; ev[6] = e1.z; ev[7] = e1.w;
            float qe[8], ke[8], t8[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) { qe[j] = qv[j] * ev[j]; ke[j] = kv[j] * ev[j]; }
            uint8_t *abase = sm + SM_AREG + kb * SM_AREG_KB;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                if (qq > pi) continue;
                const float *Fr = sF + fpq(pi, qq) * 128 + 8 * g;
                const int rowQ = arow_base(qq) + (i - 16 * qq);
                const int rowK = rowQ + 16 * (4 - qq);
#pragma unroll
                for (int j = 0; j < 8; ++j) t8[j] = qe[j] * Fr[j];
                *reinterpret_cast<uint4 *>(abase + swz(rowQ, cc)) = pack8(t8);
#pragma unroll
                for (int j = 0; j < 8; ++j) t8[j] = ke[j] * Fr[j];
                *reinterpret_cast<uint4 *>(abase + swz(rowK, cc)) = pack8(t8);
            }
            const float *Er = sED + pi * 128 + 8 * g;
#pragma unroll
            for (int j = 0; j < 8; ++j) t8[j] = kv[j] * __fdividef(Er[j], ev[j]);
            *reinterpret_cast<uint4 *>(sm + SM_BQ + pi * 4096 + kb * 2048 + swz(i - 16 * pi, cc)) = pack8(t8);
            const float *Pr = sPF + pi * 128 + 8 * g;
#pragma unroll
            for (int j = 0; j < 8; ++j) t8[j] = Pr[j] * qe[j];
            *reinterpret_cast<uint4 *>(sm + SM_QD + (i * D + 8 * g) * 2) = pack8(t8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 3. A_qk / A_kk block columns on the tensor cores
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t ID16 = idesc_bf16_f32(128, 16);
            // k-step major: the four block columns accumulate independently, so their
            // MMAs overlap in the tensor pipe instead of waiting on one accumulator
#pragma unroll
            for (int s = 0; s < 8; ++s) {
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const int kb = s >> 2, w = s & 3;
                    const uint64_t ad = sdesc_sw128(smem_u32(sm + SM_AREG + kb * SM_AREG_KB + arow_base(qq) * 128 + w * 32));
                    const uint64_t bd = sdesc_sw128(smem_u32(sm + SM_BQ + qq * 4096 + kb * 2048 + w * 32));
                    mma_bf16(tmem + 16 * qq, ad, bd, ID16, s > 0);
                }
            }
            mma_commit(&mbar_p);
        }
        // prefetch the next unit's inputs while this one computes
        const int u_next = u + gridDim.x;
        ChunkInfo ci_next = ci;
        if (u_next < n_units) {
            ci_next = plan_chunk(plan, u_next / H);
            load_col(k, v, z, H, u_next % H, ci_next.tok, ci_next.len, p, c, kp, vp, e);
            load_row(q, k, H, u_next % H, ci_next.tok, ci_next.len, ri0, rg0, qr0, kr0);
            load_row(q, k, H, u_next % H, ci_next.tok, ci_next.len, ri1, rg0, qr1, kr1);
        }
        bool ok = mbar_wait(&mbar_p, (uint32_t)(it & 1));
        __syncwarp();
        tc_fence_after();
        float *Lm = reinterpret_cast<float *>(sm + SM_AREG + SM_L);
        float *Mq = reinterpret_cast<float *>(sm + SM_AREG + SM_MQK);
        float *INV = reinterpret_cast<float *>(sm + SM_AREG + SM_INV);
        float *tmp = reinterpret_cast<float *>(sm + SM_AREG + SM_TMP);
        {
            const int qq = warp >> 2;  // key tile read by this warp
            float d[16];
            tmem_ld16(tmem + lane_off + 16 * qq, d);
            tmem_ld_wait();
            const int nq = 16 * (4 - qq), r = r_lane;
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

        // ---- 4. INV = (I + L)^-1; then [I ; M_qk] INV on the tensor cores
        tri_inverse(Lm, INV, tmp, tid, PT_THREADS);
        for (int idx = tid; idx < 128 * 8; idx += PT_THREADS) {
            // A operand [I ; M_qk]: row m (0..127), 8 k-columns per store
            const int row = idx >> 3, g8 = idx & 7;
            __align__(16) __nv_bfloat16 b8[8];
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) {
                const int s = g8 * 8 + e8;
                b8[e8] = __float2bfloat16_rn(row < 64 ? (s == row ? 1.f : 0.f) : Mq[(row - 64) * TRI_LD + s]);
            }
            *reinterpret_cast<uint4 *>(sm + SM_BQ + row * 128 + (((g8 ^ (row & 7)) & 7) << 4)) =
                *reinterpret_cast<const uint4 *>(b8);
        }
        {
            // B operand INV^T: row j, k = s  (element INV[s][j])
            const int j = tid & 63, g8 = tid >> 6;  // 512 threads = 64 rows x 8 groups
            __align__(16) __nv_bfloat16 b8[8];
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) b8[e8] = __float2bfloat16_rn(INV[(g8 * 8 + e8) * TRI_LD + j]);
            *reinterpret_cast<uint4 *>(sm + SM_A2 + j * 128 + (((g8 ^ (j & 7)) & 7) << 4)) =
                *reinterpret_cast<const uint4 *>(b8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t ID64 = idesc_bf16_f32(128, 64);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t ad = sdesc_sw128(smem_u32(sm + SM_BQ + s * 32));
                const uint64_t bd = sdesc_sw128(smem_u32(sm + SM_A2 + s * 32));
                mma_bf16(tmem, ad, bd, ID64, s > 0);
            }
            mma_commit(&mbar_z);
        }
        ok = mbar_wait(&mbar_z, (uint32_t)(it & 1));
        __syncwarp();
        tc_fence_after();
        {
            // [INV ; Z] rows -> A2 image (overwrites INV^T: the MMA that read it has completed)
            const int cb = warp >> 2;  // 16-column block of the 64 columns
            float d[16];
            tmem_ld16(tmem + lane_off + 16 * cb, d);
            tmem_ld_wait();
            __align__(16) __nv_bfloat16 b16[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) b16[jj] = __float2bfloat16_rn(d[jj]);
            const int row = r_lane;
            *reinterpret_cast<uint4 *>(sm + SM_A2 + row * 128 + ((((2 * cb) ^ (row & 7)) & 7) << 4)) =
                *reinterpret_cast<const uint4 *>(b16);
            *reinterpret_cast<uint4 *>(sm + SM_A2 + row * 128 + ((((2 * cb + 1) ^ (row & 7)) & 7) << 4)) =
                *reinterpret_cast<const uint4 *>(b16 + 8);
        }
        fence_async_smem();
        tc_fence_before();
        ok = !__syncthreads_or(!ok);
        if (!ok) { timed_out = true; break; }

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
            const int qt = warp >> 2;  // column quarter: 0,1 = W | M_qk W, 2,3 = U0 | O0
            const int r = r_lane;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                const int col = 64 * qt + 16 * cb;  // TMEM column
                float d[16];
                tmem_ld16(tmem + lane_off + col, d);
                tmem_ld_wait();
                __align__(16) __nv_bfloat16 o16[16];
                if (qt < 2) {
                    if (r < 64) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) o16[j] = __float2bfloat16_rn(d[j]);
                    } else {
                        const __nv_bfloat16 *qd = reinterpret_cast<const __nv_bfloat16 *>(sm + SM_QD) + (r - 64) * D + col;
#pragma unroll
                        for (int j = 0; j < 16; ++j) o16[j] = __float2bfloat16_rn(__bfloat162float(qd[j]) - d[j]);
                    }
                    *reinterpret_cast<uint4 *>(sm + SM_AREG + ST_A1 + sw128_offset(r, col, 128)) =
                        *reinterpret_cast<const uint4 *>(o16);
                    *reinterpret_cast<uint4 *>(sm + SM_AREG + ST_A1 + sw128_offset(r, col + 8, 128)) =
                        *reinterpret_cast<const uint4 *>(o16 + 8);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) o16[j] = __float2bfloat16_rn(d[j]);
                    uint8_t *dst = sm + SM_AREG + (r < 64 ? ST_U0 : ST_O0) + slice_offset(r & 63, col - 128);
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
        ci = ci_next;
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
