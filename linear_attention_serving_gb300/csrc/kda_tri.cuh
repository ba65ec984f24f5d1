// kda_tri.cuh -- the UT-transform inverse of one chunk at fp32 accuracy,
// written straight into the bf16 operand image of the product that uses it.
//
// "Kimi K3 模型结构（2）：序列维度（下），chunkwise 并行与下界衰减", section
// "UT 变换": I + L is unit lower triangular, so its inverse is unique.  With
// X_pq the 16 x 16 blocks of the inverse and L_pq those of L, the block rule
//   [[P, 0], [R, Q]]^-1 = [[P^-1, 0], [-Q^-1 R P^-1, Q^-1]]
// applied to the 16-row and then to the 32-row halves gives:
//   D.  X_pp = (I + L_pp)^-1, p = 0..3, by forward substitution;
//   1.  T0 = L_10 X_00,  T1 = L_32 X_22,
//       Q0 = L_[2:4],0 X_00,  Q1 = L_[2:4],1 X_11   (32 rows: block rows 2, 3);
//   2.  X_10 = -X_11 T0,  X_32 = -X_33 T1,  P0 = Q0 - Q1 T0;
//   3.  [[X_20, X_21], [X_30, X_31]] = -[[X_22, 0], [X_32, X_33]] [P0 | Q1].
// (Step 3 is -X_B (L_BA X_A) of the 32-row split: its left half
// L_[2:4],0 X_00 + L_[2:4],1 X_10 equals P0 because X_10 = -X_11 T0.)
//
// Steps 1-3 are 16 x 8 output tiles, one per warp, on the mma.sync tensor-core
// path in split tf32 (fp32 accuracy): a 64 x 64 inverse is too small for the
// asynchronous tensor-core round trip, and fp32 dot products on the CUDA cores
// spend their time in shared-memory broadcasts.
#pragma once

#include <cuda_bf16.h>

namespace kda {

constexpr int TRI_LD = 68;  // row stride (floats) of the 64 x 64 fp32 matrices; 16-byte rows

// element (row i, column c) of a 64-column bf16 operand image with the
// 128-byte swizzle (128-byte rows; 16-byte chunks permuted by i % 8)
__device__ __forceinline__ void tri_img_put(uint8_t *img, int i, int c, float v) {
    *reinterpret_cast<__nv_bfloat16 *>(img + i * 128 + ((((c >> 3) ^ (i & 7)) & 7) << 4) + (c & 7) * 2) =
        __float2bfloat16_rn(v);
}

// Warp-level 16 x 8 tiles of the block products on the mma.sync tensor-core
// path with tf32 operands.  Each fp32 operand is split into two tf32 parts,
// hi = v with its 13 low mantissa bits cleared and lo = (v - hi) cleared the
// same way (v - hi is exact), and three products (hi hi, hi lo, lo hi) are
// accumulated, which keeps the products at fp32 accuracy: what is dropped is
// below 2^-20 of each term.  Fragment layout of m16n8k8 (g = lane / 4,
// t = lane % 4):
//   A (16 x 8): (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4)
//   B (8 x 8):  (t, g), (t + 4, g)
//   C (16 x 8): (g, 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1)
__device__ __forceinline__ void tri_split(float v, uint32_t &hi, uint32_t &lo) {
    hi = __float_as_uint(v) & 0xffffe000u;
    lo = __float_as_uint(v - __uint_as_float(hi)) & 0xffffe000u;
}
__device__ __forceinline__ void tri_mma(float *c, const uint32_t *a, const uint32_t *b) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// c += sign * A B for A 16 x K (rows at stride lda) and B K x 8 (row-major,
// stride ldb), both fp32 in shared memory; c a C fragment of the calling warp
template <int K>
__device__ __forceinline__ void tri_tile(float *c, const float *A, int lda, const float *B, int ldb, float sign,
                                         int lane) {
    const int g = lane >> 2, t = lane & 3;
    float e1[4] = {0.f, 0.f, 0.f, 0.f}, e2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t ah[4], al[4], bh[2], bl[2];
        tri_split(sign * A[g * lda + k0 + t], ah[0], al[0]);
        tri_split(sign * A[(g + 8) * lda + k0 + t], ah[1], al[1]);
        tri_split(sign * A[g * lda + k0 + t + 4], ah[2], al[2]);
        tri_split(sign * A[(g + 8) * lda + k0 + t + 4], ah[3], al[3]);
        tri_split(B[(k0 + t) * ldb + g], bh[0], bl[0]);
        tri_split(B[(k0 + t + 4) * ldb + g], bh[1], bl[1]);
        tri_mma(e1, al, bh);
        tri_mma(e2, ah, bl);
        tri_mma(c, ah, bh);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] += e1[j] + e2[j];
}
// C fragment -> fp32 matrix (row-major, stride ld)
__device__ __forceinline__ void tri_put_f32(float *M, int ld, const float *c, int lane) {
    const int g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2 *>(M + g * ld + 2 * t) = make_float2(c[0], c[1]);
    *reinterpret_cast<float2 *>(M + (g + 8) * ld + 2 * t) = make_float2(c[2], c[3]);
}
// C fragment -> bf16 image, tile origin (row r0, column c0)
__device__ __forceinline__ void tri_put_img(uint8_t *img, int r0, int c0, const float *c, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = r0 + g + 8 * h, col = c0 + 2 * t;
        const __nv_bfloat162 v = __floats2bfloat162_rn(c[2 * h], c[2 * h + 1]);
        *reinterpret_cast<__nv_bfloat162 *>(img + i * 128 + ((((col >> 3) ^ (i & 7)) & 7) << 4) + (col & 7) * 2) = v;
    }
}

// L: strictly lower with beta folded in; only its blocks on and below the
// block diagonal are read (the diagonal blocks zero on and above their
// diagonal).  X: fp32 scratch for the blocks the later steps read (64 rows of
// TRI_LD floats); T: fp32 scratch of 48 rows.  img: the bf16 image of the
// whole inverse (row i, k = s), written in full, zeros above the block
// diagonal.  All 512 threads of the block call this; it ends with a block
// barrier after a proxy fence, so that the tensor cores may read the image.
// Steps 1-3 run on warps 0-11 (named barrier 1); warps 12-15 call `idle()`
// meanwhile and meet the others at the final barrier.
template <int NT, typename Idle>
__device__ __forceinline__ void tri_inverse(const float *__restrict__ L, float *__restrict__ X, float *__restrict__ T,
                                            uint8_t *__restrict__ img, int tid, Idle &&idle) {
    static_assert(NT == 512, "tri_inverse is laid out for 512 threads");
    const int warp = tid >> 5, lane = tid & 31;
    // ---- D: warp p inverts diagonal block p, lane c forming column c (each
    // solved row updates the rows below it); warps 4.. clear the image above
    // the block diagonal
    if (warp < 4) {
        if (lane < 16) {
            const int o = 16 * warp, c = lane;
            float a[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) a[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < 15; ++i) {
#pragma unroll
                for (int r = i + 1; r < 16; ++r) a[r] = fmaf(-L[(o + r) * TRI_LD + o + i], a[i], a[r]);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                X[(o + r) * TRI_LD + o + c] = a[r];
                tri_img_put(img, o + r, o + c, a[r]);
            }
        }
    } else if (tid < 128 + 192) {
        // six blocks x 16 rows x two 16-byte chunks
        const int idx = tid - 128, blk = idx >> 5, w = idx & 31;
        const int p = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int q = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        const int row = 16 * p + (w >> 1), g8 = 2 * q + (w & 1);
        *reinterpret_cast<uint4 *>(img + row * 128 + (((g8 ^ (row & 7)) & 7) << 4)) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();

    if (warp >= 12) {
        idle();
    } else {
        // ---- 1: T rows 0-15 = [T0 | T1], rows 16-47 = [Q0 | Q1]; one 16 x 8 tile per warp
        {
            const int n = warp & 1;
            const float *A, *B;
            float *out;
            if (warp < 2) {  // T0 = L_10 X_00
                A = L + 16 * TRI_LD; B = X; out = T;
            } else if (warp < 6) {  // Q0 = L_[2:4],0 X_00
                const int m = (warp - 2) >> 1;
                A = L + (32 + 16 * m) * TRI_LD; B = X; out = T + (16 + 16 * m) * TRI_LD;
            } else if (warp < 8) {  // T1 = L_32 X_22
                A = L + 48 * TRI_LD + 32; B = X + 32 * TRI_LD + 32; out = T + 16;
            } else {  // Q1 = L_[2:4],1 X_11
                const int m = (warp - 8) >> 1;
                A = L + (32 + 16 * m) * TRI_LD + 16; B = X + 16 * TRI_LD + 16; out = T + (16 + 16 * m) * TRI_LD + 16;
            }
            float c4[4] = {0.f, 0.f, 0.f, 0.f};
            tri_tile<16>(c4, A, TRI_LD, B + 8 * n, TRI_LD, 1.f, lane);
            tri_put_f32(out + 8 * n, TRI_LD, c4, lane);
        }
        asm volatile("bar.sync 1, 384;" ::: "memory");
        // ---- 2: X_10 = -X_11 T0 (image), P0 = Q0 - Q1 T0 (over Q0), X_32 = -X_33 T1
        if (warp < 8) {
            const int n = warp & 1;
            float c4[4] = {0.f, 0.f, 0.f, 0.f};
            if (warp < 2) {
                tri_tile<16>(c4, X + 16 * TRI_LD + 16, TRI_LD, T + 8 * n, TRI_LD, -1.f, lane);
                tri_put_img(img, 16, 8 * n, c4, lane);
            } else if (warp < 6) {
                const int m = (warp - 2) >> 1;
                float *q0 = T + (16 + 16 * m) * TRI_LD + 8 * n;
                const int g = lane >> 2, t = lane & 3;
                const float2 u = *reinterpret_cast<const float2 *>(q0 + g * TRI_LD + 2 * t);
                const float2 w = *reinterpret_cast<const float2 *>(q0 + (g + 8) * TRI_LD + 2 * t);
                c4[0] = u.x; c4[1] = u.y; c4[2] = w.x; c4[3] = w.y;
                tri_tile<16>(c4, T + (16 + 16 * m) * TRI_LD + 16, TRI_LD, T + 8 * n, TRI_LD, -1.f, lane);
                tri_put_f32(q0, TRI_LD, c4, lane);
            } else {
                tri_tile<16>(c4, X + 48 * TRI_LD + 48, TRI_LD, T + 16 + 8 * n, TRI_LD, -1.f, lane);
                tri_put_f32(X + 48 * TRI_LD + 32 + 8 * n, TRI_LD, c4, lane);
                tri_put_img(img, 48, 32 + 8 * n, c4, lane);
            }
        }
        asm volatile("bar.sync 1, 384;" ::: "memory");
        // ---- 3: rows 32..63, columns 0..31 of the inverse = -X_B [P0 | Q1]
        if (warp < 8) {
            const int n = warp & 3;
            float c4[4] = {0.f, 0.f, 0.f, 0.f};
            if (warp < 4) {
                tri_tile<16>(c4, X + 32 * TRI_LD + 32, TRI_LD, T + 16 * TRI_LD + 8 * n, TRI_LD, -1.f, lane);
                tri_put_img(img, 32, 8 * n, c4, lane);
            } else {
                tri_tile<32>(c4, X + 48 * TRI_LD + 32, TRI_LD, T + 16 * TRI_LD + 8 * n, TRI_LD, -1.f, lane);
                tri_put_img(img, 48, 8 * n, c4, lane);
            }
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
}

}  // namespace kda
