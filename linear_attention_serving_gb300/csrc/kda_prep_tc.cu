// kda_prep_tc.cu -- per-(chunk, head) preparation for bf16 inputs, with the
// contractions on tcgen05 tensor cores.
//
// For one 64-token chunk of one head this computes everything of the chunk
// form that does not depend on the entering state ("Kimi K3: the Manos, the
// Mythos ..." (SemiAnalysis), "FlashKDA 算法": a = exp(cumsum g), K_decay,
// Q_decay, K_inv, K_restore, L, INV = (I+L)^-1, M_qk), and folds it into the
// record the scan consumes:
//   W = INV Diag(beta) K_decay,  U0 = INV Diag(beta) V,  Q' = Q_decay - M_qk W,
//   O0 = M_qk U0,  G = K_restore^T W,  H = K_restore^T U0,  a_C,
// so that a chunk of the scan is S <- Diag(a_C) S + H - G S and O = O0 + Q' S,
// which is the pages' U = INV Diag(beta)(V - K_decay S), O = Q_decay S + M_qk U,
// S <- Diag(a[-1]) S + K_restore^T U with the products regrouped.
//
// One block per SM walks (chunk, head) units with 512 threads:
//  1. column phase, thread = (2 channels, 8 tokens): z, k, v of its channels
//     and tokens (the next unit's are prefetched while the current one
//     computes); gate of "Kimi K3 模型结构（2）" eq. (5); cumulative log decay
//     inside each 16-token sub-tile ("数值问题：1/Γ 会溢出"); e_i = exp(G_i -
//     G_{tile start}) in (e^-80, 1]; per-(tile, channel) factors; the
//     token-contiguous operands Diag(beta) K_decay, Diag(beta) V, K_restore^T;
//  2. row phase, thread = (token, 8 channels): the factored MMA operands (bf16,
//     K-major, 128-byte swizzle, 16-byte stores): for key tile q the
//     query-side rows x_i e_i F_pq (x = q and x = k, rows of tiles p >= q) and
//     the key side k_j exp(Delta_q) / e_j, with F_pp = exp(-Delta_p) <= e^80 and
//     F_pq = prod_{q<t<p} exp(Delta_t) <= 1; and Q_decay;
//  3. four M = 128, N = 16 MMAs give M_qk and A_kk block column by block
//     column, from which L = StrictTril(Diag(beta) A_kk) and M_qk;
//  4. INV = (I + L)^-1 in fp32 CUDA cores ("UT 变换"), then one MMA
//     [I ; M_qk] INV = [INV ; Z] for Z = M_qk INV;
//  5. one M = 128, N = 256, K = 64 MMA:
//     [INV ; Z] [Diag(beta) K_decay | Diag(beta) V] = [W | U0 ; M_qk W | O0];
//  6. Q' = Q_decay - M_qk W and O0 go to the record; W and U0 become the
//     operand of one more M = 128, N = 256, K = 64 MMA,
//     K_restore^T [W | U0] = [G | H], which goes to the record.
// The record is staged in shared memory and written with bulk copies that
// overlap the next unit.  Every wait is bounded; a timeout records
// KDA_DEVERR_TIMEOUT and ends the block.
#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tri.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int PT_THREADS = 512;

// shared-memory map (bytes from a 1024-aligned base)
constexpr int SM_AREG = 0;           // A_q images (2 k-blocks x 320 rows x 128 B); later fp32
                                     // L | M_qk | INV | tmp.  An M = 128 read of the last
                                     // image runs past its 32 valid rows into the following
                                     // bytes; those rows are ignored.
constexpr int SM_AREG_KB = 40960;    // offset of the second k-block of the A_q images
constexpr int SM_BQ = 81920;         // key-side images, 4 x (2 k-blocks x 16 rows x 128 B);
                                     // later [I ; M_qk] (128 rows x 64)
constexpr int SM_B2 = 98304;         // [Diag(beta) K_decay | Diag(beta) V]^T (256 rows x 64 tokens);
                                     // later [W | U0]^T (256 rows x 64 tokens)
constexpr int SM_A2 = 131072;        // INV^T (64 rows x 64), then [INV ; Z] (128 rows x 64)
constexpr int SM_KRT = 147456;       // K_restore^T: 128 channels x 64 tokens
constexpr int SM_QD = 163840;        // Q_decay bf16 [64][128] row-major
constexpr int SM_MISC = 180224;      // beta [64] | partial log-decay sums [8][128]
constexpr int SM_E = 184576;         // e_i [64][128] fp32 (column phase -> row phase)
constexpr int SM_TAB = 217344;       // F [10][128] | exp(Delta) [4][128] | ePfx [4][128] fp32
constexpr int SM_BYTES = 226560;
constexpr size_t PREP_TC_SMEM = SM_BYTES + 1024;

// staging of the output record (after the last MMA has read its operands)
constexpr int ST_G = SM_AREG;               // 32 KB
constexpr int ST_H = SM_AREG + 32768;       // 32 KB
constexpr int ST_QP = SM_AREG + 65536;      // 16 KB
constexpr int ST_O0 = SM_E;                 // 16 KB

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

__device__ __forceinline__ int fpq(int p, int q) { return p * (p + 1) / 2 + q; }

// column phase inputs: channels 2 cp, 2 cp + 1 of tokens 8 rg .. 8 rg + 7
struct ColIn {
    __nv_bfloat162 k[8], v[8];
    float2 z[8];
};
__device__ __forceinline__ void load_col(const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                                         const float *__restrict__ z, int H, int h, int t0, int len, int rg, int cp,
                                         ColIn &in) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = 8 * rg + r;
        if (i < len) {
            const size_t a = ((size_t)(t0 + i) * H + h) * D + 2 * cp;
            in.k[r] = *reinterpret_cast<const __nv_bfloat162 *>(k + a);
            in.v[r] = *reinterpret_cast<const __nv_bfloat162 *>(v + a);
            in.z[r] = *reinterpret_cast<const float2 *>(z + a);
        } else {
            in.k[r] = __float2bfloat162_rn(0.f);
            in.v[r] = __float2bfloat162_rn(0.f);
            in.z[r] = make_float2(0.f, 0.f);
        }
    }
}

// row phase inputs: 8 channels [8 g, 8 g + 8) of token i of q and k
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

__global__ void __launch_bounds__(PT_THREADS, 1)
prep_tc_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
               const __nv_bfloat16 *__restrict__ v, const float *__restrict__ z, const float *__restrict__ A,
               const float *__restrict__ beta, int H, float g_min, Plan plan, char *__restrict__ records) {
    extern __shared__ uint8_t smraw[];
    __shared__ uint64_t mbar_p, mbar_z, mbar_e, mbar_g;
    __shared__ uint32_t tmem_slot;

    if (plan_failed(plan)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cp = tid & 63, rg = tid >> 6;  // column phase: channel pair, 8-token group
    const int tile = rg >> 1;                // the 16-token sub-tile of the column phase rows
    uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    float *sbeta = reinterpret_cast<float *>(sm + SM_MISC);
    float *sHalf = sbeta + 64;  // [8][128] partial log-decay sums of each 8-token group
    float *sE = reinterpret_cast<float *>(sm + SM_E);
    float *sF = reinterpret_cast<float *>(sm + SM_TAB);
    float *sED = sF + 10 * 128;
    float *sPF = sED + 4 * 128;

    if (tid == 0) {
        mbar_init(&mbar_p, 1);
        mbar_init(&mbar_z, 1);
        mbar_init(&mbar_e, 1);
        mbar_init(&mbar_g, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int lg = warp & 3;  // TMEM lane group of this warp
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int r_lane = lg * 32 + lane;  // TMEM lane (row) this thread reads
    const int qt = warp >> 2;           // column quarter / block read by this warp

    const int n_units = plan_n_chunks(plan) * H;
    // row phase items: (token i, channel group g), tokens paired from both ends
    const int ri0 = tid >> 4, rg0 = tid & 15, ri1 = 63 - ri0;
    ColIn cin;
    uint4 qr0, kr0, qr1, kr1;
    int u = blockIdx.x;
    ChunkInfo ci;
    if (u < n_units) {
        ci = plan_chunk(plan, u / H);
        load_col(k, v, z, H, u % H, ci.tok, ci.len, rg, cp, cin);
        load_row(q, k, H, u % H, ci.tok, ci.len, ri0, rg0, qr0, kr0);
        load_row(q, k, H, u % H, ci.tok, ci.len, ri1, rg0, qr1, kr1);
    }
    bool timed_out = false;
    for (int it = 0; u < n_units && !timed_out; u += gridDim.x, ++it) {
        const int cidx = u / H, h = u - cidx * H;
        const int len = ci.len;
        char *rec = records + ((size_t)cidx * H + h) * REC_BF16_BYTES;
        const float eA = __expf(A[h]);

        // ---- 1. column phase: gate, partial cumulative log decay of 8 tokens
        float rl[8][2];
        float h0 = 0.f, h1 = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const bool ok = 8 * rg + r < len;
            const float g0 = ok ? __fdividef(g_min, 1.f + __expf(-eA * cin.z[r].x)) : 0.f;
            const float g1 = ok ? __fdividef(g_min, 1.f + __expf(-eA * cin.z[r].y)) : 0.f;
            h0 += g0;
            h1 += g1;
            rl[r][0] = h0;
            rl[r][1] = h1;
        }
        if (tid == 0) bulk_wait_read_all();  // the previous unit's record has left the staging area
        __syncthreads();                      // the previous unit is done with every shared buffer
        *reinterpret_cast<float2 *>(sHalf + rg * 128 + 2 * cp) = make_float2(h0, h1);
        if (tid < 64) sbeta[tid] = tid < len ? beta[(size_t)(ci.tok + tid) * H + h] : 0.f;
        __syncthreads();
        {
            float eD[4][2], carry[2] = {0.f, 0.f};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 a0 = *reinterpret_cast<const float2 *>(sHalf + (2 * t) * 128 + 2 * cp);
                const float2 a1 = *reinterpret_cast<const float2 *>(sHalf + (2 * t + 1) * 128 + 2 * cp);
                eD[t][0] = __expf(a0.x + a1.x);
                eD[t][1] = __expf(a0.y + a1.y);
                if (t == tile && (rg & 1)) {
                    carry[0] = a0.x;
                    carry[1] = a0.y;
                }
            }
            float ePfx[2] = {1.f, 1.f}, eSfx[2] = {1.f, 1.f};
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (t < tile) ePfx[j] *= eD[t][j];
                    if (t > tile) eSfx[j] *= eD[t][j];
                }
            if ((rg & 1) == 0) {
                // per-(tile, channel) factors, written once per tile
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    if (qq > tile) continue;
                    float f[2] = {1.f, 1.f};
#pragma unroll
                    for (int t = 0; t < 4; ++t)
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            if (t > qq && t < tile) f[j] *= eD[t][j];
                    if (qq == tile) {
                        f[0] = __fdividef(1.f, eD[tile][0]);
                        f[1] = __fdividef(1.f, eD[tile][1]);
                    }
                    *reinterpret_cast<float2 *>(sF + fpq(tile, qq) * 128 + 2 * cp) = make_float2(f[0], f[1]);
                }
                *reinterpret_cast<float2 *>(sED + tile * 128 + 2 * cp) = make_float2(eD[tile][0], eD[tile][1]);
                *reinterpret_cast<float2 *>(sPF + tile * 128 + 2 * cp) = make_float2(ePfx[0], ePfx[1]);
                if (tile == 0)
                    *reinterpret_cast<float2 *>(rec + REC_BF16_AC + 8 * cp) =
                        make_float2(eD[0][0] * eD[1][0] * eD[2][0] * eD[3][0], eD[0][1] * eD[1][1] * eD[2][1] * eD[3][1]);
            }
            // e_i, and the token-contiguous operands: 8 tokens per 16-byte store
            float bkd[2][8], bv[2][8], bkr[2][8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = 8 * rg + r;
                const float2 kf = __bfloat1622float2(cin.k[r]);
                const float2 vf = __bfloat1622float2(cin.v[r]);
                const float e0 = __expf(carry[0] + rl[r][0]), e1 = __expf(carry[1] + rl[r][1]);
                *reinterpret_cast<float2 *>(sE + i * 128 + 2 * cp) = make_float2(e0, e1);
                const float b = sbeta[i];
                const float kf0 = kf.x * __fdividef(eD[tile][0], e0), kf1 = kf.y * __fdividef(eD[tile][1], e1);
                bkd[0][r] = b * ePfx[0] * e0 * kf.x;  // Diag(beta) K_decay
                bkd[1][r] = b * ePfx[1] * e1 * kf.y;
                bv[0][r] = b * vf.x;                  // Diag(beta) V
                bv[1][r] = b * vf.y;
                bkr[0][r] = eSfx[0] * kf0;            // K_restore = exp(G_last - G_j) k_j
                bkr[1][r] = eSfx[1] * kf1;
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = 2 * cp + j;
                const uint32_t sw = (uint32_t)(((rg ^ (c & 7)) & 7) << 4);
                *reinterpret_cast<uint4 *>(sm + SM_B2 + c * 128 + sw) = pack8(bkd[j]);
                *reinterpret_cast<uint4 *>(sm + SM_B2 + (128 + c) * 128 + sw) = pack8(bv[j]);
                *reinterpret_cast<uint4 *>(sm + SM_KRT + c * 128 + sw) = pack8(bkr[j]);
            }
        }
        __syncthreads();

        // ---- 2. row phase: factored A_q rows, key-side rows, Q_decay
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
                const float4 f0 = *reinterpret_cast<const float4 *>(sF + fpq(pi, qq) * 128 + 8 * g);
                const float4 f1 = *reinterpret_cast<const float4 *>(sF + fpq(pi, qq) * 128 + 8 * g + 4);
                const float Fr[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
                const int rowQ = arow_base(qq) + (i - 16 * qq);
                const int rowK = rowQ + 16 * (4 - qq);
#pragma unroll
                for (int j = 0; j < 8; ++j) t8[j] = qe[j] * Fr[j];
                *reinterpret_cast<uint4 *>(abase + swz(rowQ, cc)) = pack8(t8);
#pragma unroll
                for (int j = 0; j < 8; ++j) t8[j] = ke[j] * Fr[j];
                *reinterpret_cast<uint4 *>(abase + swz(rowK, cc)) = pack8(t8);
            }
            const float4 d0 = *reinterpret_cast<const float4 *>(sED + pi * 128 + 8 * g);
            const float4 d1 = *reinterpret_cast<const float4 *>(sED + pi * 128 + 8 * g + 4);
            const float Er[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) t8[j] = kv[j] * __fdividef(Er[j], ev[j]);
            *reinterpret_cast<uint4 *>(sm + SM_BQ + pi * 4096 + kb * 2048 + swz(i - 16 * pi, cc)) = pack8(t8);
            const float4 p0 = *reinterpret_cast<const float4 *>(sPF + pi * 128 + 8 * g);
            const float4 p1 = *reinterpret_cast<const float4 *>(sPF + pi * 128 + 8 * g + 4);
            const float Pr[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
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
            load_col(k, v, z, H, u_next % H, ci_next.tok, ci_next.len, rg, cp, cin);
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
            const int qq = qt;  // key tile read by this warp
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
        tri_inverse<PT_THREADS>(Lm, INV, tmp, tid);
        for (int idx = tid; idx < 128 * 8; idx += PT_THREADS) {
            // A operand [I ; M_qk]: row m (0..127), 8 k-columns per store
            const int row = idx >> 3, g8 = idx & 7;
            float f8[8];
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) {
                const int s = g8 * 8 + e8;
                f8[e8] = row < 64 ? (s == row ? 1.f : 0.f) : Mq[(row - 64) * TRI_LD + s];
            }
            *reinterpret_cast<uint4 *>(sm + SM_BQ + row * 128 + (((g8 ^ (row & 7)) & 7) << 4)) = pack8(f8);
        }
        {
            // B operand INV^T: row j, k = s  (element INV[s][j]); 512 threads = 64 rows x 8 groups
            const int j = tid & 63, g8 = tid >> 6;
            float f8[8];
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) f8[e8] = INV[(g8 * 8 + e8) * TRI_LD + j];
            *reinterpret_cast<uint4 *>(sm + SM_A2 + j * 128 + (((g8 ^ (j & 7)) & 7) << 4)) = pack8(f8);
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
            const int cb = qt;  // 16-column block of the 64 columns
            float d[16];
            tmem_ld16(tmem + lane_off + 16 * cb, d);
            tmem_ld_wait();
            const int row = r_lane;
            *reinterpret_cast<uint4 *>(sm + SM_A2 + row * 128 + ((((2 * cb) ^ (row & 7)) & 7) << 4)) = pack8(d);
            *reinterpret_cast<uint4 *>(sm + SM_A2 + row * 128 + ((((2 * cb + 1) ^ (row & 7)) & 7) << 4)) = pack8(d + 8);
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

        // ---- 6a. rows 0..63 -> [W | U0]^T operand; rows 64..127 -> Q', O0 in the record
        {
            const int r = r_lane;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                const int col = 64 * qt + 16 * cb;  // TMEM column
                float d[16];
                tmem_ld16(tmem + lane_off + col, d);
                tmem_ld_wait();
                if (r < 64) {
                    // transposed: row n = col + j of [W | U0]^T, column (token) r
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = col + j;
                        *reinterpret_cast<__nv_bfloat16 *>(sm + SM_B2 + n * 128 + ((((r >> 3) ^ (n & 7)) & 7) << 4) + (r & 7) * 2) =
                            __float2bfloat16_rn(d[j]);
                    }
                } else if (qt < 2) {
                    const int i = r - 64;
                    const __nv_bfloat16 *qd = reinterpret_cast<const __nv_bfloat16 *>(sm + SM_QD) + i * D + col;
                    float t16[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) t16[j] = __bfloat162float(qd[j]) - d[j];
                    *reinterpret_cast<uint4 *>(sm + ST_QP + sw128_offset(i, col, 64)) = pack8(t16);
                    *reinterpret_cast<uint4 *>(sm + ST_QP + sw128_offset(i, col + 8, 64)) = pack8(t16 + 8);
                } else {
                    uint8_t *dst = sm + ST_O0 + slice_offset(r - 64, col - 128, 64);
                    *reinterpret_cast<uint4 *>(dst) = pack8(d);
                    *reinterpret_cast<uint4 *>(dst + 16) = pack8(d + 8);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = !__syncthreads_or(!ok);
        if (!ok) { timed_out = true; break; }

        // ---- 6b. K_restore^T [W | U0] = [G | H]  (M = 128, N = 256, K = 64)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t ID256 = idesc_bf16_f32(128, 256);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t ad = sdesc_sw128(smem_u32(sm + SM_KRT + s * 32));
                const uint64_t bd = sdesc_sw128(smem_u32(sm + SM_B2 + s * 32));
                mma_bf16(tmem, ad, bd, ID256, s > 0);
            }
            mma_commit(&mbar_g);
        }
        ok = mbar_wait(&mbar_g, (uint32_t)(it & 1));
        __syncwarp();
        tc_fence_after();
        {
            const int c = r_lane;  // state row (channel)
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                const int col = 64 * qt + 16 * cb;
                float d[16];
                tmem_ld16(tmem + lane_off + col, d);
                tmem_ld_wait();
                if (qt < 2) {
                    *reinterpret_cast<uint4 *>(sm + ST_G + sw128_offset(c, col, 128)) = pack8(d);
                    *reinterpret_cast<uint4 *>(sm + ST_G + sw128_offset(c, col + 8, 128)) = pack8(d + 8);
                } else {
                    uint8_t *dst = sm + ST_H + slice_offset(c, col - 128, 128);
                    *reinterpret_cast<uint4 *>(dst) = pack8(d);
                    *reinterpret_cast<uint4 *>(dst + 16) = pack8(d + 8);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = !__syncthreads_or(!ok);
        if (!ok) { timed_out = true; break; }
        if (tid == 0) {
            bulk_s2g(rec + REC_BF16_G, sm + ST_G, 32768);
            bulk_s2g(rec + REC_BF16_QP, sm + ST_QP, 16384);
            bulk_s2g(rec + REC_BF16_H, sm + ST_H, 32768);
            bulk_s2g(rec + REC_BF16_O0, sm + ST_O0, 16384);
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
