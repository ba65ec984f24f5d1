// kda_prep_body.cuh -- per-(chunk, head) preparation for bf16 inputs, with the
// contractions on tcgen05 tensor cores (the device code; kda_prep_tc.cu and
// kda_fused_tc.cu launch it).
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
//  1. operand build, thread = (2 channels, 8 tokens): q, k, v, z of its
//     channels and tokens, read from the unit's input tiles, which the tensor
//     memory accelerator (TMA) loaded into shared memory while the previous
//     unit computed; gate of "Kimi K3 模型结构（2）" eq. (5) in base-2 log space;
//     cumulative log decay inside each 16-token sub-tile ("数值问题：1/Γ 会溢出");
//     e_i = exp(G_i - G_{tile start}) in (e^-80, 1]; and every MMA operand of
//     the chunk, in bf16 with the 128-byte swizzle: for key tile q the
//     query-side rows x_i e_i F_pq (x = q and x = k, rows of tiles p >= q) and
//     the key side k_j exp(Delta_q) / e_j, with F_pp = exp(-Delta_p) <= e^80 and
//     F_pq = prod_{q<t<p} exp(Delta_t) <= 1; Q_decay; and the token-contiguous
//     Diag(beta) K_decay, Diag(beta) V, K_restore^T;
//  2. block-column MMAs, M = 128: per k-step one N = 16 product for key tile 0,
//     one for key tile 1, and one N = 32 product over the adjacent images of
//     tiles 2 and 3, give M_qk and A_kk, from which
//     L = StrictTril(Diag(beta) A_kk) (fp32) and the bf16 operand M_qk;
//  3. INV = (I + L)^-1 ("UT 变换"): the 16 x 16 diagonal blocks by forward
//     substitution in fp32, the block products as split-tf32 mma.sync tiles
//     (kda_tri.cuh), written as a bf16 operand;
//  4. two M = 128, N = 64, K = 64 MMAs: [Diag(beta) K_decay | Diag(beta) V]^T
//     INV^T = [W | U0]^T (a channel per TMEM lane);
//  5. [W | U0]^T becomes the K-major B operand of the MMAs issued together:
//     K_restore^T [W | U0] = [G | H] (M = 128) and, with M = 64,
//     Q' = I Q_decay + (-M_qk) W and O0 = M_qk U0; G, H, Q', O0 go to the record.
// Warp 0 runs the tcgen05 issue code as a whole warp, one elected lane issuing.
// The record is staged in shared memory, in the operand areas the last
// products have finished reading, and written with bulk copies that overlap
// the next unit's first phases.  Where chain blocks consume the records as
// they appear, the thread that issued the copies waits for them to complete
// while the next unit's inverse runs on the other threads, then raises the
// unit's ready flag.  Every wait is bounded; a timeout records
// KDA_DEVERR_TIMEOUT and ends the block.
#pragma once

#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_tri.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int PT_THREADS = 512;
constexpr int PT_TMEM_COLS = 512;
constexpr int PT_STORE_TID = 384;  // issues the bulk stores of a record and publishes it
constexpr float LOG2E = 1.4426950408889634f;

// shared-memory map (bytes from a 1024-aligned base)
constexpr int SM_AREG = 0;           // the unit's input tiles (TMA), read into registers at its
                                     // start; then the A_q images (2 k-blocks x 320 rows x 128 B);
                                     // after their MMA, fp32 L | INV | scratch; then free for the
                                     // next unit's input tiles.  A read of an image past its valid
                                     // rows runs into the following bytes; those rows are ignored.
constexpr int SM_AREG_KB = 40960;    // offset of the second k-block of the A_q images
constexpr int SM_BQ = 81920;         // key-side images, 2 k-blocks x (4 tiles x 16 rows x 128 B)
constexpr int SM_B2 = 98304;         // [Diag(beta) K_decay | Diag(beta) V]^T (256 rows x 64 tokens);
                                     // later [W | U0]^T in the same K-major layout
constexpr int SM_A2 = 131072;        // INV (64 rows x 64), then O0 staging
constexpr int SM_KRT = 147456;       // K_restore^T: 128 channels x 64 tokens
constexpr int SM_QD = 163840;        // Q_decay, MN-major (2 blocks of 64 channels x 64 tokens)
constexpr int SM_MQ = 180224;        // M_qk (64 rows x 64)
constexpr int SM_ID = 188416;        // identity (64 rows x 64), written once
constexpr int SM_MISC = 196608;      // beta [64] | partial log2-decay sums [8][128] |
                                     // squared norms of q, k per token and warp half [64][4]
constexpr int SM_BYTES = SM_MISC + 256 + 4096 + 1024;
constexpr size_t PREP_TC_SMEM = SM_BYTES + 1024;

// staging of the output record, in operand areas that the unit's last products
// have read: written by the last epilogue, read by the bulk stores until the
// next unit's operand build (which waits for that before writing B2, KRT,
// BQ, QD; A2 is rewritten only after the next inverse)
constexpr int ST_G = SM_B2;   // 32 KB
constexpr int ST_H = SM_KRT;  // 32 KB (KRT and QD)
constexpr int ST_QP = SM_BQ;  // 16 KB
constexpr int ST_O0 = SM_A2;  // 16 KB
static_assert(SM_QD == SM_KRT + 16384 && SM_MQ == SM_QD + 16384, "H staging spans KRT and QD");

// the unit's input tiles inside SM_AREG: [64 tokens][128 channels] each
constexpr int IN_Q = 0, IN_K = 16384, IN_V = 32768, IN_Z = 49152;  // q, k, v bf16; z fp32
constexpr uint32_t IN_BYTES = 81920;
static_assert(IN_BYTES <= SM_BQ - SM_AREG, "input tiles fit the image area");

// fp32 matrices inside SM_AREG (row stride TRI_LD floats)
constexpr int MAT_BYTES = 64 * TRI_LD * 4;
constexpr int SM_L = 0;
constexpr int SM_INV = MAT_BYTES;
constexpr int SM_TMP = 2 * MAT_BYTES;
static_assert(3 * MAT_BYTES <= SM_BQ - SM_AREG, "fp32 work matrices fit the image area");

__device__ __forceinline__ int arow_base(int q) { return q == 0 ? 0 : (q == 1 ? 128 : (q == 2 ? 224 : 288)); }

// byte offset of (row, cc) in a 128-byte-swizzled k-block; cc < 64
__device__ __forceinline__ uint32_t swz(int row, int cc) {
    return (uint32_t)(row * 128 + ((((cc >> 3) ^ (row & 7)) & 7) << 4) + (cc & 7) * 2);
}
// byte offset of 16-byte chunk g8 of row `row` in a 128-byte-swizzled k-block
__device__ __forceinline__ uint32_t swz_chunk(int row, int g8) {
    return (uint32_t)(row * 128 + (((g8 ^ (row & 7)) & 7) << 4));
}

// inputs of the operand build: channels 2 cp, 2 cp + 1 of tokens 8 rg .. 8 rg + 7
struct BuildIn {
    __nv_bfloat162 q[8], k[8], v[8];
    float2 z[8];
};
// This thread's inputs from the unit's tiles in shared memory; rows at or past
// the chunk's length (another document, or zeros past the tensor) read as 0.
__device__ __forceinline__ void read_inputs(const uint8_t *tiles, int len, int rg, int cp, BuildIn &in) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = 8 * rg + r;
        const bool ok = i < len;
        const int e = i * D + 2 * cp;
        in.z[r] = ok ? *reinterpret_cast<const float2 *>(tiles + IN_Z + 4 * e) : make_float2(0.f, 0.f);
        in.q[r] = ok ? *reinterpret_cast<const __nv_bfloat162 *>(tiles + IN_Q + 2 * e) : __float2bfloat162_rn(0.f);
        in.k[r] = ok ? *reinterpret_cast<const __nv_bfloat162 *>(tiles + IN_K + 2 * e) : __float2bfloat162_rn(0.f);
        in.v[r] = ok ? *reinterpret_cast<const __nv_bfloat162 *>(tiles + IN_V + 2 * e) : __float2bfloat162_rn(0.f);
    }
}
// One thread: the TMA loads of a unit's four input tiles (head h, the chunk
// starting at token t0) into the tile area, counted on `bar`.
__device__ __forceinline__ void load_tiles(const InputMaps *maps, uint8_t *tiles, int h, int t0, uint64_t *bar) {
    mbar_expect_tx(bar, IN_BYTES);
    tma_load_3d(tiles + IN_Q, &maps->q, 0, h, t0, bar);
    tma_load_3d(tiles + IN_K, &maps->k, 0, h, t0, bar);
    tma_load_3d(tiles + IN_V, &maps->v, 0, h, t0, bar);
    tma_load_3d(tiles + IN_Z, &maps->z, 0, h, t0, bar);
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 ex2x2(float2 a) { return make_float2(ex2(a.x), ex2(a.y)); }
// Gate of "Kimi K3 模型结构（2）" eq. (5) in base-2 log space, g log2(e) =
// g_min log2(e) sigmoid(e^{A_h} z), and its running sums over this thread's tokens.
__device__ __forceinline__ void gate_sums(const BuildIn &in, float A_h, float gm2, int first, int len, float2 *rl) {
    const float c1 = -ex2(A_h * 1.4426950408889634f) * 1.4426950408889634f;  // exp(-e^{A_h} z) = 2^(c1 z)
    float2 hs = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const float2 uu = make_float2(ex2(in.z[r].x * c1), ex2(in.z[r].y * c1));
        const float2 den = __fadd2_rn(uu, make_float2(1.f, 1.f));
        const float2 g2 = first + r < len ? make_float2(__fdividef(gm2, den.x), __fdividef(gm2, den.y)) : make_float2(0.f, 0.f);
        hs = __fadd2_rn(hs, g2);
        rl[r] = hs;
    }
}

__device__ __forceinline__ uint32_t bf2(float2 a) {
    const __nv_bfloat162 b = __float22bfloat162_rn(a);
    return *reinterpret_cast<const uint32_t *>(&b);
}
// Release *flag = 1 after this block's earlier writes, including the
// completed bulk stores (async proxy) and the stores of the other threads
// that reached the last block barrier.
__device__ __forceinline__ void publish(int *flag) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}

__device__ __forceinline__ uint4 pack8(const float *f) {
    uint4 u;
    u.x = bf2(make_float2(f[0], f[1]));
    u.y = bf2(make_float2(f[2], f[3]));
    u.z = bf2(make_float2(f[4], f[5]));
    u.w = bf2(make_float2(f[6], f[7]));
    return u;
}

// The units first, first + stride, ... of the launch, on one block of
// PT_THREADS threads.  OPTS compiles the input options (KDA_FLAG_*, read from
// the plan) in: a separate instantiation, so that the default path keeps its
// registers.  With `ready` non-null, ready[u] is set (release, after
// the record's bulk stores have completed) once unit u's record is in memory.
template <bool OPTS>
__device__ __forceinline__ void prep_blocks(const InputMaps *maps, const float *__restrict__ A,
                                            const float *__restrict__ beta, int H, float g_min, const Plan &plan,
                                            char *__restrict__ records, uint8_t *smraw, int first, int stride,
                                            int *ready) {
    __shared__ uint64_t mbar_p, mbar_w, mbar_g, mbar_q, mbar_in, mbar_dr;
    __shared__ uint32_t tmem_slot;

    if (plan_failed(plan)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cp = tid & 63, rg = tid >> 6;      // build phase: channel pair, 8-token group
    const int tile = rg >> 1;                    // the 16-token sub-tile of this thread's tokens
    const int kb = cp >> 5, cc = (2 * cp) & 63;  // k-block and column of the channel pair in K-major images
    uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
    float *sbeta = reinterpret_cast<float *>(sm + SM_MISC);
    float *sHalf = sbeta + 64;  // [8][128] log2-decay sums of each 8-token group
    float *snorm = sHalf + 8 * 128;  // [64 tokens][q half 0, q half 1, k half 0, k half 1]
    const bool l2norm = OPTS && (plan.flags & KDA_FLAG_QK_L2NORM) != 0;
    const bool bsig = OPTS && (plan.flags & KDA_FLAG_BETA_SIGMOID) != 0;
    const bool qscale = OPTS && (plan.flags & KDA_FLAG_Q_SCALE) != 0;
    const float gm2 = g_min * LOG2E;

    if (tid == 0) {
        mbar_init(&mbar_p, 1);
        mbar_init(&mbar_w, 1);
        mbar_init(&mbar_g, 1);
        mbar_init(&mbar_q, 1);
        mbar_init(&mbar_in, 1);
        mbar_init(&mbar_dr, 1);
        mbar_fence_init();
    }
    // a block that publishes its records may run a chain afterwards, which
    // allocates TMEM again: it keeps its permit to allocate
    if (warp == 0) tmem_alloc(&tmem_slot, PT_TMEM_COLS, ready == nullptr);
    {
        // identity operand: row m has its 1 at k = m
        const int m = tid >> 3, g8 = tid & 7;
        uint4 w = make_uint4(0, 0, 0, 0);
        if ((m >> 3) == g8) {
            uint32_t *wp = reinterpret_cast<uint32_t *>(&w);
            wp[(m & 7) >> 1] = (m & 1) ? 0x3F800000u : 0x00003F80u;
        }
        *reinterpret_cast<uint4 *>(sm + SM_ID + swz_chunk(m, g8)) = w;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int lg = warp & 3;  // TMEM lane quadrant of this warp
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int qt = warp >> 2;  // column quarter / block read by this warp

    const int n_units = plan_n_chunks(plan) * H;
    BuildIn cin;
    float b_next = 0.f, a_next = 0.f;
    int u = first;
    int u_prev = -1;  // unit whose record was written last (its flag is raised during the next inverse)
    int tiles_issued = 0, tiles_landed = 0;  // TMA tile loads into the tile area (one per unit)
    ChunkInfo ci;
    if (u < n_units) {
        ci = plan_chunk(plan, u / H);
        if (tid == 0) load_tiles(maps, sm + SM_AREG, u % H, ci.tok, &mbar_in);
        tiles_issued = 1;
        if (tid < 64 && tid < ci.len) {
            b_next = beta[(size_t)(ci.tok + tid) * H + u % H];
            if (bsig) b_next = 1.f / (1.f + __expf(-b_next));  // input option: beta logit
        }
        a_next = A[u % H];
    }
    bool timed_out = false;
    for (int it = 0; u < n_units && !timed_out; u += stride, ++it) {
        const int cidx = u / H, h = u - cidx * H;
        char *rec = records + ((size_t)cidx * H + h) * REC_BF16_BYTES;

        // ---- 0. the unit's input tiles have landed: this thread's part into registers
        if (!__syncthreads_and(mbar_wait(&mbar_in, (uint32_t)(it & 1)))) { timed_out = true; break; }
        tiles_landed = it + 1;
        read_inputs(sm + SM_AREG, ci.len, rg, cp, cin);

        // ---- 1. gate, partial log2-decay sums of each 8-token group, and beta
        float2 rl[8];
        gate_sums(cin, a_next, gm2, 8 * rg, ci.len, rl);
        *reinterpret_cast<float2 *>(sHalf + rg * 128 + 2 * cp) = rl[7];
        // input option: squared norms of q and k over this warp's 64 channels (the
        // token's other 64 sit in the neighbouring warp)
        if (tid < 64) sbeta[tid] = b_next;
        if (l2norm) {
            // transpose reduction: eight token sums over the warp's 32 lanes in 9
            // shuffles per tensor; lane l ends with token ((l >> 2) & 7)'s total
            float pq[8], pk[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float2 qf = __bfloat1622float2(cin.q[r]), kf = __bfloat1622float2(cin.k[r]);
                pq[r] = qf.x * qf.x + qf.y * qf.y;
                pk[r] = kf.x * kf.x + kf.y * kf.y;
            }
            const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
            float q4[4], k4[4], q2[2], k2[2];
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // keep tokens 4 b4 + j, send the other half
                q4[j] = (b4 ? pq[j + 4] : pq[j]) + __shfl_xor_sync(0xffffffffu, b4 ? pq[j] : pq[j + 4], 16);
                k4[j] = (b4 ? pk[j + 4] : pk[j]) + __shfl_xor_sync(0xffffffffu, b4 ? pk[j] : pk[j + 4], 16);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {  // tokens 4 b4 + 2 b3 + j
                q2[j] = (b3 ? q4[j + 2] : q4[j]) + __shfl_xor_sync(0xffffffffu, b3 ? q4[j] : q4[j + 2], 8);
                k2[j] = (b3 ? k4[j + 2] : k4[j]) + __shfl_xor_sync(0xffffffffu, b3 ? k4[j] : k4[j + 2], 8);
            }
            float sq = (b2 ? q2[1] : q2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? q2[0] : q2[1], 4);
            float sk = (b2 ? k2[1] : k2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? k2[0] : k2[1], 4);
            sq += __shfl_xor_sync(0xffffffffu, sq, 2);
            sk += __shfl_xor_sync(0xffffffffu, sk, 2);
            sq += __shfl_xor_sync(0xffffffffu, sq, 1);
            sk += __shfl_xor_sync(0xffffffffu, sk, 1);
            if ((lane & 3) == 0) {
                const int r = (lane >> 2) & 7;
                snorm[4 * (8 * rg + r) + (warp & 1)] = sq;
                snorm[4 * (8 * rg + r) + 2 + (warp & 1)] = sk;
            }
        }
        // the previous unit's record has left the staging areas the build rewrites
        if (tid == PT_STORE_TID) bulk_wait_read_all();
        __syncthreads();

        // tile sums Delta_t (log2), exp(Delta_t), and this thread's carry into its tile
        float2 Dl = make_float2(0.f, 0.f), carry = make_float2(0.f, 0.f), eD[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 a0 = *reinterpret_cast<const float2 *>(sHalf + (2 * t) * 128 + 2 * cp);
            const float2 a1 = *reinterpret_cast<const float2 *>(sHalf + (2 * t + 1) * 128 + 2 * cp);
            const float2 st = add2(a0, a1);
            eD[t] = ex2x2(st);
            if (t == tile) {
                Dl = st;
                if (rg & 1) carry = a0;
            }
        }
        float2 ePfx = make_float2(1.f, 1.f), eSfx = make_float2(1.f, 1.f);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (t < tile) ePfx = mul2(ePfx, eD[t]);
            if (t > tile) eSfx = mul2(eSfx, eD[t]);
        }
        if (rg == 0)
            *reinterpret_cast<float2 *>(rec + REC_BF16_AC + 8 * cp) = mul2(mul2(eD[0], eD[1]), mul2(eD[2], eD[3]));

        // ---- 1b. per-token factors, the key sides and the query-side rows of the
        // A_q images (what the first products read)
        if (l2norm) {
            // input option: this thread's q and k divided by their tokens' norms
            // (rounded back to bf16, as the operands they feed are)
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float4 nn = *reinterpret_cast<const float4 *>(snorm + 4 * (8 * rg + r));
                const float iq = rsqrtf(nn.x + nn.y + L2NORM_EPS), ik = rsqrtf(nn.z + nn.w + L2NORM_EPS);
                cin.q[r] = __float22bfloat162_rn(mul2(__bfloat1622float2(cin.q[r]), make_float2(iq, iq)));
                cin.k[r] = __float22bfloat162_rn(mul2(__bfloat1622float2(cin.k[r]), make_float2(ik, ik)));
            }
        }
        float2 qe[8], ke[8], kx[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int i = 8 * rg + r;
            float2 qf = __bfloat1622float2(cin.q[r]);
            if (qscale) qf = mul2(qf, make_float2(Q_SCALE, Q_SCALE));  // input option: q d_k^-1/2
            const float2 kf = __bfloat1622float2(cin.k[r]);
            const float2 c2 = add2(carry, rl[r]);
            const float2 e = ex2x2(c2);
            const float2 x = ex2x2(add2(Dl, make_float2(-c2.x, -c2.y)));  // exp(Delta_p) / e_i
            qe[r] = mul2(qf, e);
            ke[r] = mul2(kf, e);
            kx[r] = mul2(kf, x);
            // key side of key tile p
            *reinterpret_cast<uint32_t *>(sm + SM_BQ + kb * 8192 + tile * 2048 + swz(i - 16 * tile, cc)) = bf2(kx[r]);
        }
        {
            uint8_t *abase = sm + SM_AREG + kb * SM_AREG_KB;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                if (qq > tile) continue;
                float2 F = make_float2(1.f, 1.f);
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    if (t > qq && t < tile) F = mul2(F, eD[t]);
                if (qq == tile) F = make_float2(__fdividef(1.f, eD[tile].x), __fdividef(1.f, eD[tile].y));
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int i = 8 * rg + r;
                    const int rowQ = arow_base(qq) + (i - 16 * qq);
                    const int rowK = rowQ + 16 * (4 - qq);
                    *reinterpret_cast<uint32_t *>(abase + swz(rowQ, cc)) = bf2(mul2(qe[r], F));
                    *reinterpret_cast<uint32_t *>(abase + swz(rowK, cc)) = bf2(mul2(ke[r], F));
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 2. A_qk / A_kk block columns on the tensor cores.  Key tiles 0 and 1
        // take one M = 128 MMA each (N = 16); the images of tiles 2 and 3 (64 and
        // 32 rows) are adjacent, so one M = 128, N = 32 MMA over both key tiles
        // serves them: the blocks it forms across the two (tile 2's rows against
        // tile 3's keys and the reverse) are never read.
        if (warp == 0) {  // the whole warp: one elected lane issues
            tc_fence_after();
            constexpr uint32_t ID16 = idesc_bf16_f32(128, 16), ID32 = idesc_bf16_f32(128, 32);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
#pragma unroll
                for (int qq = 0; qq < 3; ++qq) {
                    const int kbs = s >> 2, w = s & 3;
                    const uint64_t ad = sdesc_sw128(smem_u32(sm + SM_AREG + kbs * SM_AREG_KB + arow_base(qq) * 128 + w * 32));
                    const uint64_t bd = sdesc_sw128(smem_u32(sm + SM_BQ + kbs * 8192 + qq * 2048 + w * 32));
                    mma_bf16_w(tmem + 16 * qq, ad, bd, qq < 2 ? ID16 : ID32, s > 0);
                }
            }
            mma_commit_w(&mbar_p);
        }

        // ---- 1c. while those products run: the token-contiguous operands of the
        // later products, Diag(beta) K_decay, Diag(beta) V, K_restore^T, and Q_decay
        {
            // two tokens per packed word: [channel][token pair]
            uint32_t bkd[2][4], bv[2][4], bkr[2][4];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = 8 * rg + r;
                const float2 vf = __bfloat1622float2(cin.v[r]);
                const float b = sbeta[i];
                const float2 vbkd = mul2(mul2(ePfx, make_float2(b, b)), ke[r]);  // Diag(beta) K_decay
                const float2 vbv = mul2(vf, make_float2(b, b));                  // Diag(beta) V
                const float2 vbkr = mul2(eSfx, kx[r]);                           // K_restore = exp(G_last - G_i) k_i
                // channel j of this token -> low (even token) or high (odd token) half of a word
                const uint32_t w0 = bf2(make_float2(vbkd.x, vbkd.y)), w1 = bf2(make_float2(vbv.x, vbv.y)),
                               w2 = bf2(make_float2(vbkr.x, vbkr.y));
                const int pr = r >> 1;
                if ((r & 1) == 0) {
                    bkd[0][pr] = w0 & 0xFFFFu;
                    bkd[1][pr] = w0 >> 16;
                    bv[0][pr] = w1 & 0xFFFFu;
                    bv[1][pr] = w1 >> 16;
                    bkr[0][pr] = w2 & 0xFFFFu;
                    bkr[1][pr] = w2 >> 16;
                } else {
                    bkd[0][pr] |= w0 << 16;
                    bkd[1][pr] |= w0 & 0xFFFF0000u;
                    bv[0][pr] |= w1 << 16;
                    bv[1][pr] |= w1 & 0xFFFF0000u;
                    bkr[0][pr] |= w2 << 16;
                    bkr[1][pr] |= w2 & 0xFFFF0000u;
                }
                *reinterpret_cast<uint32_t *>(sm + SM_QD + kb * 8192 + swz(i, cc)) = bf2(mul2(ePfx, qe[r]));
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = 2 * cp + j;
                const uint32_t sw = (uint32_t)(((rg ^ (c & 7)) & 7) << 4);
                *reinterpret_cast<uint4 *>(sm + SM_B2 + c * 128 + sw) = make_uint4(bkd[j][0], bkd[j][1], bkd[j][2], bkd[j][3]);
                *reinterpret_cast<uint4 *>(sm + SM_B2 + (128 + c) * 128 + sw) = make_uint4(bv[j][0], bv[j][1], bv[j][2], bv[j][3]);
                *reinterpret_cast<uint4 *>(sm + SM_KRT + c * 128 + sw) = make_uint4(bkr[j][0], bkr[j][1], bkr[j][2], bkr[j][3]);
            }
        }
        fence_async_smem();  // read by the later products, issued after the next barriers
        // next unit: its betas now, its input tiles once the image area is free
        const int u_next = u + stride;
        const bool has_next = u_next < n_units;
        ChunkInfo ci_next = ci;
        if (has_next) {
            ci_next = plan_chunk(plan, u_next / H);
            if (tid < 64) {
                b_next = tid < ci_next.len ? beta[(size_t)(ci_next.tok + tid) * H + u_next % H] : 0.f;
                if (bsig && tid < ci_next.len) b_next = 1.f / (1.f + __expf(-b_next));
            }
            a_next = A[u_next % H];
        }
        bool ok = mbar_wait(&mbar_p, (uint32_t)(it & 1));
        __syncwarp();
        tc_fence_after();
        float *Lm = reinterpret_cast<float *>(sm + SM_AREG + SM_L);
        float *INV = reinterpret_cast<float *>(sm + SM_AREG + SM_INV);
        float *tmp = reinterpret_cast<float *>(sm + SM_AREG + SM_TMP);
        {
            // block column qq: image rows < nq are M_qk rows, rows nq .. 2 nq - 1 are
            // A_kk rows.  Image row r sits in TMEM lane r (tiles 0-2) or 64 + r (tile 3)
            const int qq = qt;
            float d[16];
            tmem_ld16(tmem + lane_off + 16 * qq, d);
            tmem_ld_wait();
            const int nq = 16 * (4 - qq);
            const int r = qq < 3 ? lg * 32 + lane : (lg == 2 ? lane : 1 << 20);
            if (r < nq) {
                const int i = 16 * qq + r;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) d[jj] = (16 * qq + jj <= i) ? d[jj] : 0.f;
                *reinterpret_cast<uint4 *>(sm + SM_MQ + swz_chunk(i, 2 * qq)) = pack8(d);
                *reinterpret_cast<uint4 *>(sm + SM_MQ + swz_chunk(i, 2 * qq + 1)) = pack8(d + 8);
            } else if (r < 2 * nq) {
                const int i = 16 * qq + (r - nq);
                const float b = sbeta[i];
                float *dst = Lm + i * TRI_LD + 16 * qq;
#pragma unroll
                for (int j4 = 0; j4 < 16; j4 += 4) {
                    float4 t;
                    t.x = (16 * qq + j4 < i) ? b * d[j4] : 0.f;
                    t.y = (16 * qq + j4 + 1 < i) ? b * d[j4 + 1] : 0.f;
                    t.z = (16 * qq + j4 + 2 < i) ? b * d[j4 + 2] : 0.f;
                    t.w = (16 * qq + j4 + 3 < i) ? b * d[j4 + 3] : 0.f;
                    *reinterpret_cast<float4 *>(dst + j4) = t;
                }
            }
        }
        if (tid < 256) {
            // M_qk is zero above its block diagonal: row i, 16-column block t > tile(i)
            const int i = tid >> 2, t = tid & 3;
            if (t > (i >> 4)) {
                const uint4 zz = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(sm + SM_MQ + swz_chunk(i, 2 * t)) = zz;
                *reinterpret_cast<uint4 *>(sm + SM_MQ + swz_chunk(i, 2 * t + 1)) = zz;
            }
        }
        tc_fence_before();
        ok = !__syncthreads_or(!ok);
        if (!ok) { timed_out = true; break; }

        // ---- 3. INV = (I + L)^-1, written as its bf16 image (row i, k = s).
        // The storing thread idles during the inverse's block products: it
        // waits there for the previous unit's record to be complete in memory
        // and publishes it
        tri_inverse<PT_THREADS>(Lm, INV, tmp, sm + SM_A2, tid, [&] {
            if (tid == PT_STORE_TID && ready && u_prev >= 0) {
                bulk_wait_all();
                publish(ready + u_prev);
            }
        });

        // ---- 4. [W | U0]^T = [Diag(beta) K_decay | Diag(beta) V]^T INV^T: two M = 128,
        //         N = 64, K = 64 products (the channels of K_decay, then of V, against
        //         the INV image as a K-major B operand); every TMEM lane holds a
        //         channel, so the epilogue below keeps all 128 lanes busy
        if (warp == 0) {
            if (lane == 0 && has_next) {
                // the image area is free until the next unit's build: its input tiles
                fence_async_smem();
                load_tiles(maps, sm + SM_AREG, u_next % H, ci_next.tok, &mbar_in);
            }
            __syncwarp();
            tc_fence_after();
            constexpr uint32_t IDT = idesc_bf16_f32(128, 64);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ad = sdesc_sw128(smem_u32(sm + SM_B2 + hf * 16384 + s * 32));
                    const uint64_t bd = sdesc_sw128(smem_u32(sm + SM_A2 + s * 32));
                    mma_bf16_w(tmem + 64 * hf, ad, bd, IDT, s > 0);
                }
            }
            mma_commit_w(&mbar_w);
        }
        if (has_next) ++tiles_issued;
        ok = mbar_wait(&mbar_w, (uint32_t)(it & 1));
        __syncwarp();
        tc_fence_after();
        {
            // channel c = TMEM lane, tokens 32 qt .. 32 qt + 31 of the 128 columns
            // [W^T | U0^T] -> row n of [W | U0]^T (K-major, the B2 layout): n = c for
            // W, 128 + c for U0
            const int c = lg * 32 + lane, n = (qt < 2 ? 0 : 128) + c, g0 = 4 * (qt & 1);
            float d[32];
            tmem_ld16(tmem + lane_off + 32 * qt, d);
            tmem_ld16(tmem + lane_off + 32 * qt + 16, d + 16);
            tmem_ld_wait();
#pragma unroll
            for (int h8 = 0; h8 < 4; ++h8)
                *reinterpret_cast<uint4 *>(sm + SM_B2 + swz_chunk(n, g0 + h8)) = pack8(d + 8 * h8);
        }
        fence_async_smem();
        tc_fence_before();
        ok = !__syncthreads_or(!ok);
        if (!ok) { timed_out = true; break; }

        // ---- 5. K_restore^T [W | U0] = [G | H] (M = 128), and with M = 64
        //         (-M_qk) [W | U0] = [-M_qk W | -O0] (one N = 256 product), to which
        //         I Q_decay is added on the left half: Q' = Q_decay - M_qk W.  The
        //         epilogue flips the sign of the right half back to O0.  The M = 64
        //         group goes first, with a commit of its own: its epilogue stages Q'
        //         and O0 in areas the [G | H] products do not read, while they run.
        if (warp == 0) {
            tc_fence_after();
            constexpr uint32_t IDG = idesc_bf16_f32(128, 256), IDM = idesc_bf16_f32_bmn(64, 128);
            constexpr uint32_t IDW = idesc_bf16_f32(64, 256);
            constexpr uint32_t NEG_A = 1u << 13;
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_w(tmem + 256, sdesc_sw128(smem_u32(sm + SM_MQ + s * 32)),
                           sdesc_sw128(smem_u32(sm + SM_B2 + s * 32)), IDW | NEG_A, s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_w(tmem + 256, sdesc_sw128(smem_u32(sm + SM_ID + s * 32)),
                           sdesc_mn(smem_u32(sm + SM_QD + s * 2048), 8192, 1024, SWZ_128B), IDM, true);
            mma_commit_w(&mbar_q);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_w(tmem, sdesc_sw128(smem_u32(sm + SM_KRT + s * 32)),
                           sdesc_sw128(smem_u32(sm + SM_B2 + s * 32)), IDG, s > 0);
            mma_commit_w(&mbar_g);
        }
        ok = mbar_wait(&mbar_q, (uint32_t)(it & 1));
        __syncwarp();
        tc_fence_after();
        {
            const int m = 16 * lg + lane;  // token of [M_qk W | O0] (lanes < 16)
#pragma unroll
            for (int cb = 0; cb < 4; cb += 2) {
                const int col = 64 * qt + 16 * cb;
                float d[32];
                tmem_ld16(tmem + lane_off + 256 + col, d);
                tmem_ld16(tmem + lane_off + 256 + col + 16, d + 16);
                tmem_ld_wait();
                if (lane < 16) {
                    if (qt < 2) {
#pragma unroll
                        for (int h8 = 0; h8 < 4; ++h8)
                            *reinterpret_cast<uint4 *>(sm + ST_QP + sw128_offset(m, col + 8 * h8, 64)) = pack8(d + 8 * h8);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) d[j] = -d[j];  // -O0 -> O0
#pragma unroll
                        for (int h16 = 0; h16 < 2; ++h16) {
                            uint8_t *dst = sm + ST_O0 + slice_offset(m, col + 16 * h16 - 128, 64);
                            *reinterpret_cast<uint4 *>(dst) = pack8(d + 16 * h16);
                            *reinterpret_cast<uint4 *>(dst + 16) = pack8(d + 16 * h16 + 8);
                        }
                    }
                }
            }
        }
        ok = mbar_wait(&mbar_g, (uint32_t)(it & 1)) && ok;
        __syncwarp();
        tc_fence_after();
        {
            const int c = lg * 32 + lane;  // state row (channel) of [G | H]
#pragma unroll
            for (int cb = 0; cb < 4; cb += 2) {
                const int col = 64 * qt + 16 * cb;
                float d[32];
                tmem_ld16(tmem + lane_off + col, d);
                tmem_ld16(tmem + lane_off + col + 16, d + 16);
                tmem_ld_wait();
                if (qt < 2) {
#pragma unroll
                    for (int h8 = 0; h8 < 4; ++h8)
                        *reinterpret_cast<uint4 *>(sm + ST_G + sw128_offset(c, col + 8 * h8, 128)) = pack8(d + 8 * h8);
                } else {
#pragma unroll
                    for (int h16 = 0; h16 < 2; ++h16) {
                        uint8_t *dst = sm + ST_H + slice_offset(c, col + 16 * h16 - 128, 128);
                        *reinterpret_cast<uint4 *>(dst) = pack8(d + 16 * h16);
                        *reinterpret_cast<uint4 *>(dst + 16) = pack8(d + 16 * h16 + 8);
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = !__syncthreads_or(!ok);
        if (!ok) { timed_out = true; break; }
        if (tid == PT_STORE_TID) {
            bulk_s2g(rec + REC_BF16_G, sm + ST_G, 32768);
            bulk_s2g(rec + REC_BF16_QP, sm + ST_QP, 16384);
            bulk_s2g(rec + REC_BF16_H, sm + ST_H, 32768);
            bulk_s2g(rec + REC_BF16_O0, sm + ST_O0, 16384);
            bulk_commit();
        }
        u_prev = u;
        ci = ci_next;
    }
    if (tid == PT_STORE_TID) {
        bulk_wait_all();
        if (ready && u_prev >= 0 && !timed_out) publish(ready + u_prev);
    }
    if (warp == 0) {
        if (lane == 0) {
            if (timed_out) atomicOr(plan.err, KDA_DEVERR_TIMEOUT);
            // tile loads and tensor-core work this block started have finished
            // before the block leaves or frees its TMEM (no-ops after a full run)
            if (tiles_issued > tiles_landed) mbar_wait(&mbar_in, (uint32_t)((tiles_issued - 1) & 1));
        }
        __syncwarp();
        mma_commit_w(&mbar_dr);
        mbar_wait(&mbar_dr, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, PT_TMEM_COLS);
}

}  // namespace

}  // namespace kda
