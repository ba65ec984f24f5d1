// kda_tri.cuh -- the UT-transform inverse of one chunk, in fp32 CUDA cores.
//
// "Kimi K3 模型结构（2）：序列维度（下），chunkwise 并行与下界衰减", section
// "UT 变换": I + L is unit lower triangular, so its inverse is unique and is
// obtained by forward substitution.  Here the 64 x 64 matrix is handled as
// 4 x 4 blocks of 16: the diagonal blocks by forward substitution, then
// X_pq = -X_pp sum_{q<=r<p} L_pr X_rq one block diagonal at a time.  Every
// loop bound is a compile-time constant so the shared-memory loads are issued
// ahead of the FMA chains, which use two partial sums.
#pragma once

namespace kda {

constexpr int TRI_LD = 65;  // row stride of the 64 x 64 fp32 matrices

// INV (zeroed above its diagonal blocks by the caller), L strictly lower with
// beta folded in, tmp [3][16][17].  All NT threads of the block call this; it
// synchronises internally and ends with a barrier.
template <int NT>
__device__ __forceinline__ void tri_inverse(const float *__restrict__ L, float *__restrict__ INV,
                                            float *__restrict__ tmp, int tid) {
    if (tid < 64) {
        const int p = tid >> 4, col = tid & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float v0 = (i == col) ? 1.f : 0.f, v1 = 0.f;
#pragma unroll
            for (int s = 0; s < i; s += 2) {
                v0 = fmaf(-L[(p * 16 + i) * TRI_LD + p * 16 + s], x[s], v0);
                if (s + 1 < i) v1 = fmaf(-L[(p * 16 + i) * TRI_LD + p * 16 + s + 1], x[s + 1], v1);
            }
            x[i] = v0 + v1;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) INV[(p * 16 + i) * TRI_LD + p * 16 + col] = x[i];
    }
    __syncthreads();
#pragma unroll
    for (int lvl = 1; lvl < 4; ++lvl) {
        const int nblk = 4 - lvl;
        for (int e = tid; e < nblk * 256; e += NT) {
            const int b = e >> 8, i = (e >> 4) & 15, jj = e & 15;
            const int p = lvl + b, qb = b;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int rr = 0; rr < lvl; ++rr) {
                const int r = qb + rr;
#pragma unroll
                for (int s = 0; s < 16; s += 2) {
                    a0 = fmaf(L[(p * 16 + i) * TRI_LD + r * 16 + s], INV[(r * 16 + s) * TRI_LD + qb * 16 + jj], a0);
                    a1 = fmaf(L[(p * 16 + i) * TRI_LD + r * 16 + s + 1], INV[(r * 16 + s + 1) * TRI_LD + qb * 16 + jj], a1);
                }
            }
            tmp[(b * 16 + i) * 17 + jj] = a0 + a1;
        }
        __syncthreads();
        for (int e = tid; e < nblk * 256; e += NT) {
            const int b = e >> 8, i = (e >> 4) & 15, jj = e & 15;
            const int p = lvl + b, qb = b;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int s = 0; s < 16; s += 2) {
                a0 = fmaf(INV[(p * 16 + i) * TRI_LD + p * 16 + s], tmp[(b * 16 + s) * 17 + jj], a0);
                a1 = fmaf(INV[(p * 16 + i) * TRI_LD + p * 16 + s + 1], tmp[(b * 16 + s + 1) * 17 + jj], a1);
            }
            INV[(p * 16 + i) * TRI_LD + qb * 16 + jj] = -(a0 + a1);
        }
        __syncthreads();
    }
}

}  // namespace kda
