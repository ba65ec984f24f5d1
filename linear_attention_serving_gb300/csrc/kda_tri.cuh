// kda_tri.cuh -- the UT-transform inverse of one chunk, in fp32 CUDA cores.
//
// "Kimi K3 模型结构（2）：序列维度（下），chunkwise 并行与下界衰减", section
// "UT 变换": I + L is unit lower triangular, so its inverse is unique.  The
// 64 x 64 matrix is split twice by the block rule
//   [[P, 0], [R, Q]]^-1 = [[P^-1, 0], [-Q^-1 R P^-1, Q^-1]]:
//   D.  the four 16 x 16 diagonal blocks by forward substitution;
//   1.  the two 32 x 32 diagonal blocks: X_10 = -X_11 (L_10 X_00) and
//       X_32 = -X_33 (L_32 X_22);
//   2.  the lower-left 32 x 32 block: -X_B (L_BA X_A), X_A and X_B the inverses
//       of the two 32 x 32 diagonal blocks.
// Phases 1 and 2 are products of small dense blocks; each thread forms four
// adjacent outputs of a row, so one 16-byte shared load of the right operand
// serves four multiply-adds (two paired fp32 FMAs).
#pragma once

namespace kda {

constexpr int TRI_LD = 68;  // row stride (floats) of the 64 x 64 fp32 matrices; 16-byte rows

// L: strictly lower with beta folded in.  Only its lower blocks are read: the
// strictly lower part of the diagonal blocks and the whole of the blocks below
// them.  INV is written in full (zeros above the block diagonal).  T is scratch
// of at least 32 x TRI_LD floats.  All NT >= 512 threads of the block call
// this; it synchronises internally and ends with a block barrier.  Phases 1
// and 2 run on threads 0-255 only (named barrier 1); threads 256 and up call
// `idle()` meanwhile and meet the others at the final barrier.
template <int NT, typename Idle>
__device__ __forceinline__ void tri_inverse(const float *__restrict__ L, float *__restrict__ INV,
                                            float *__restrict__ T, int tid, Idle &&idle) {
    static_assert(NT >= 512, "tri_inverse wants at least 512 threads");
    const int warp = tid >> 5, lane = tid & 31;
    // ---- D: warp p inverts diagonal block p, one column per lane; the other
    // warps clear the six blocks above the block diagonal
    if (warp < 4) {
        if (lane < 16) {
            const int p = warp, col = lane;
            const float *Lp = L + (16 * p) * TRI_LD + 16 * p;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float a0 = (i == col) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                for (int s = 0; s < i; s += 4) {
                    a0 = fmaf(-Lp[i * TRI_LD + s], x[s], a0);
                    if (s + 1 < i) a1 = fmaf(-Lp[i * TRI_LD + s + 1], x[s + 1], a1);
                    if (s + 2 < i) a2 = fmaf(-Lp[i * TRI_LD + s + 2], x[s + 2], a2);
                    if (s + 3 < i) a3 = fmaf(-Lp[i * TRI_LD + s + 3], x[s + 3], a3);
                }
                x[i] = (a0 + a1) + (a2 + a3);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) INV[(16 * p + i) * TRI_LD + 16 * p + col] = x[i];
        }
    } else {
        for (int idx = tid - 128; idx < 6 * 64; idx += NT - 128) {
            const int blk = idx >> 6, w = idx & 63;
            const int p = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int q = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            *reinterpret_cast<float4 *>(INV + (16 * p + (w >> 2)) * TRI_LD + 16 * q + 4 * (w & 3)) =
                make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();

    if (tid >= 256) {
        idle();
    } else {
        // ---- 1a: T_b = L_pq X_qq for (p, q) = (1, 0), (3, 2)
        if (tid < 128) {
            const int b = tid >> 6, row = (tid >> 2) & 15, c4 = 4 * (tid & 3);
            const int p = 2 * b + 1, q = 2 * b;
            const float *Lr = L + (16 * p + row) * TRI_LD + 16 * q;
            const float *X = INV + (16 * q) * TRI_LD + 16 * q + c4;
            float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
    #pragma unroll
            for (int s = 0; s < 16; ++s) {
                const float l = Lr[s];
                const float4 x = *reinterpret_cast<const float4 *>(X + s * TRI_LD);
                acc01 = __ffma2_rn(make_float2(l, l), make_float2(x.x, x.y), acc01);
                acc23 = __ffma2_rn(make_float2(l, l), make_float2(x.z, x.w), acc23);
            }
            *reinterpret_cast<float4 *>(T + (16 * b + row) * TRI_LD + c4) = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        // ---- 1b: X_pq = -X_pp T_b
        if (tid < 128) {
            const int b = tid >> 6, row = (tid >> 2) & 15, c4 = 4 * (tid & 3);
            const int p = 2 * b + 1, q = 2 * b;
            const float *Xr = INV + (16 * p + row) * TRI_LD + 16 * p;
            const float *Tb = T + (16 * b) * TRI_LD + c4;
            float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
    #pragma unroll
            for (int s = 0; s < 16; ++s) {
                const float l = Xr[s];
                const float4 t = *reinterpret_cast<const float4 *>(Tb + s * TRI_LD);
                acc01 = __ffma2_rn(make_float2(l, l), make_float2(t.x, t.y), acc01);
                acc23 = __ffma2_rn(make_float2(l, l), make_float2(t.z, t.w), acc23);
            }
            *reinterpret_cast<float4 *>(INV + (16 * p + row) * TRI_LD + 16 * q + c4) =
                make_float4(-acc01.x, -acc01.y, -acc23.x, -acc23.y);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");

        // ---- 2a: P = L[32:64, 0:32] X_A  (X_A lower triangular, zeros above)
        if (tid < 256) {
            const int row = tid >> 3, c4 = 4 * (tid & 7);
            const float *Lr = L + (32 + row) * TRI_LD;
            const float *X = INV + c4;
            float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
    #pragma unroll 8
            for (int s = 0; s < 32; ++s) {
                const float l = Lr[s];
                const float4 x = *reinterpret_cast<const float4 *>(X + s * TRI_LD);
                acc01 = __ffma2_rn(make_float2(l, l), make_float2(x.x, x.y), acc01);
                acc23 = __ffma2_rn(make_float2(l, l), make_float2(x.z, x.w), acc23);
            }
            *reinterpret_cast<float4 *>(T + row * TRI_LD + c4) = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        // ---- 2b: INV[32:64, 0:32] = -X_B P; row r of X_B is zero beyond column r,
        // and a warp's rows end at 4 (warp + 1), so that bounds its loop
        if (tid < 256) {
            const int row = tid >> 3, c4 = 4 * (tid & 7);
            const int smax = 4 * ((tid >> 5) + 1);
            const float *Xr = INV + (32 + row) * TRI_LD + 32;
            const float *P = T + c4;
            float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
    #pragma unroll 4
            for (int s = 0; s < smax; ++s) {
                const float l = Xr[s];
                const float4 t = *reinterpret_cast<const float4 *>(P + s * TRI_LD);
                acc01 = __ffma2_rn(make_float2(l, l), make_float2(t.x, t.y), acc01);
                acc23 = __ffma2_rn(make_float2(l, l), make_float2(t.z, t.w), acc23);
            }
            *reinterpret_cast<float4 *>(INV + (32 + row) * TRI_LD + c4) = make_float4(-acc01.x, -acc01.y, -acc23.x, -acc23.y);
        }
    }
    __syncthreads();
}

}  // namespace kda
