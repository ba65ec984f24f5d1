// kda_decode.cu -- decode step with MTP draft replay.
//
// "Kimi K3 模型结构（7）：结构决定系统", section "KDA：三种执行形态，三种内核"
// (decode): the state after any accepted draft prefix is fixed by the drafts'
// projected inputs, so only those are cached; the accepted prefix is replayed
// on chip, the bonus token is applied and the state is written back in place,
// and the next draft window runs in the same recurrence loop.  Per token the
// delta form of "Kimi K3: the Manos, the Mythos ..." (SemiAnalysis),
// "FlashKDA 算法":  S <- D_t S;  u = beta (v - S^T k);  S <- S + k u^T;  o = S^T q.
//
// Mapping: one block per (sequence b, head h); thread (column j, part p) keeps
// rows [p*R, p*R + R) of state column j in registers, so the d_k reductions
// are a register sum plus one shuffle, and the fp32 state is read and written
// exactly once per step with coalesced 64-byte row segments.
//
// The per-channel decay is applied lazily: with s_t = prod_{tau<=t} alpha_tau
// (per row, over this step's tokens) the kernel keeps S = Diag(s_t) S^ and
// updates S^ only:
//   u = beta (v - S^^T (s_t . k)),  S^ += (k / s_t) u^T,  o = S^^T (s_t . q),
// which removes the Diag(alpha) pass over the state for every token.  At most
// 2W - 1 <= 15 tokens run per step, so s_t >= e^{5 * 15} = e^-75 stays a
// normal fp32 number (bounded gate, "Kimi K3 模型结构（2）", "后果一").
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int MAX_W = 8;
constexpr int MAX_TOK = 2 * MAX_W - 1;
constexpr int DEC_TPC = 2;                  // threads per state column
constexpr int DEC_R = D / DEC_TPC;          // rows per thread
constexpr int DEC_THREADS = D * DEC_TPC;    // 256
constexpr int VPAD = D + 4;                 // padded vector stride (second half shifted by 4)

__device__ __forceinline__ int vidx(int r) { return r + (r >= DEC_R ? 4 : 0); }

template <typename InT>
__global__ void __launch_bounds__(DEC_THREADS, 2)
decode_kernel(float *__restrict__ state, const InT *__restrict__ q, const InT *__restrict__ k,
              const InT *__restrict__ v, const float *__restrict__ z, const float *__restrict__ beta,
              const float *__restrict__ A, InT *__restrict__ cq, InT *__restrict__ ck,
              InT *__restrict__ cv, float *__restrict__ cz, float *__restrict__ cb,
              const int32_t *__restrict__ nacc_p, int H, int W, float g_min, InT *__restrict__ o,
              int32_t *__restrict__ err) {
    __shared__ __align__(16) float kt[MAX_TOK][VPAD];  // s_t . k
    __shared__ __align__(16) float kh[MAX_TOK][VPAD];  // k / s_t
    __shared__ __align__(16) float qt[MAX_TOK][VPAD];  // s_t . q
    __shared__ float vt[MAX_TOK][D];
    __shared__ float bt[MAX_TOK];
    __shared__ float scommit[VPAD];

    const int bh = blockIdx.x;
    const int b = bh / H, h = bh - b * H;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int col = warp * (32 / DEC_TPC) + (lane & (32 / DEC_TPC - 1));
    const int part = lane / (32 / DEC_TPC);
    const int rbase = part * DEC_R;

    const int nacc = nacc_p ? nacc_p[b] : 0;
    if (nacc < 0 || nacc > W - 1) {
        if (tid == 0 && err) atomicOr(err, KDA_DEVERR_NUM_ACCEPTED);
        return;
    }
    const int ntok = nacc + W;

    // 1. issue the state loads first; they are in flight during the prologue
    float *Sg = state + (size_t)bh * D * D;
    float s[DEC_R];
#pragma unroll
    for (int i = 0; i < DEC_R; ++i) s[i] = Sg[(size_t)(rbase + i) * D + col];

    // 2. token inputs: replayed drafts from the cache, then the window
    const float eA = expf(A[h]);
    for (int idx = tid; idx < ntok * D; idx += DEC_THREADS) {
        const int t = idx >> 7, c = idx & 127;
        size_t row;
        float kk, qq, vv, zz;
        if (t < nacc) {
            row = ((size_t)b * (W - 1) + t) * H + h;
            kk = to_f32(ck[row * D + c]);
            qq = 0.f;
            vv = to_f32(cv[row * D + c]);
            zz = cz[row * D + c];
        } else {
            row = ((size_t)b * W + (t - nacc)) * H + h;
            kk = to_f32(k[row * D + c]);
            qq = to_f32(q[row * D + c]);
            vv = to_f32(v[row * D + c]);
            zz = z[row * D + c];
        }
        kt[t][vidx(c)] = kk;
        qt[t][vidx(c)] = qq;
        kh[t][vidx(c)] = expf(kda_gate(g_min, eA, zz));  // alpha, scaled below
        vt[t][c] = vv;
    }
    if (tid < ntok) {
        const int t = tid;
        bt[t] = t < nacc ? cb[((size_t)b * (W - 1) + t) * H + h] : beta[((size_t)b * W + (t - nacc)) * H + h];
    }
    __syncthreads();
    if (tid < D) {
        const int c = vidx(tid);
        float sc = 1.f;
        for (int t = 0; t < ntok; ++t) {
            sc *= kh[t][c];
            const float kk = kt[t][c];
            kt[t][c] = kk * sc;
            kh[t][c] = kk / sc;
            qt[t][c] *= sc;
            if (t == nacc) scommit[c] = sc;
        }
    }
    __syncthreads();

    // 3. the recurrence over replay + bonus + drafts
    for (int t = 0; t < ntok; ++t) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < DEC_R; i += 4) {
            const float4 kv = *reinterpret_cast<const float4 *>(&kt[t][vidx(rbase + i)]);
            acc = fmaf(s[i], kv.x, acc);
            acc = fmaf(s[i + 1], kv.y, acc);
            acc = fmaf(s[i + 2], kv.z, acc);
            acc = fmaf(s[i + 3], kv.w, acc);
        }
#pragma unroll
        for (int m = 32 / DEC_TPC; m < 32; m <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        const float u = bt[t] * (vt[t][col] - acc);
#pragma unroll
        for (int i = 0; i < DEC_R; i += 4) {
            const float4 kv = *reinterpret_cast<const float4 *>(&kh[t][vidx(rbase + i)]);
            s[i] = fmaf(kv.x, u, s[i]);
            s[i + 1] = fmaf(kv.y, u, s[i + 1]);
            s[i + 2] = fmaf(kv.z, u, s[i + 2]);
            s[i + 3] = fmaf(kv.w, u, s[i + 3]);
        }
        if (t >= nacc) {
            float ao = 0.f;
#pragma unroll
            for (int i = 0; i < DEC_R; i += 4) {
                const float4 qv = *reinterpret_cast<const float4 *>(&qt[t][vidx(rbase + i)]);
                ao = fmaf(s[i], qv.x, ao);
                ao = fmaf(s[i + 1], qv.y, ao);
                ao = fmaf(s[i + 2], qv.z, ao);
                ao = fmaf(s[i + 3], qv.w, ao);
            }
#pragma unroll
            for (int m = 32 / DEC_TPC; m < 32; m <<= 1) ao += __shfl_xor_sync(0xffffffffu, ao, m);
            if (part == 0) o[(((size_t)b * W + (t - nacc)) * H + h) * D + col] = from_f32<InT>(ao);
        }
        if (t == nacc) {
            // commit: S = Diag(s_t) S^, written back in place
#pragma unroll
            for (int i = 0; i < DEC_R; ++i)
                Sg[(size_t)(rbase + i) * D + col] = s[i] * scommit[vidx(rbase + i)];
        }
    }

    // 4. the new drafts' projected inputs replace the cache (all cache reads are done)
    for (int idx = tid; idx < (W - 1) * D; idx += DEC_THREADS) {
        const int j = idx >> 7, c = idx & 127;
        const size_t src = (((size_t)b * W + (j + 1)) * H + h) * D + c;
        const size_t dst = (((size_t)b * (W - 1) + j) * H + h) * D + c;
        cq[dst] = q[src];
        ck[dst] = k[src];
        cv[dst] = v[src];
        cz[dst] = z[src];
    }
    if (tid < W - 1) cb[((size_t)b * (W - 1) + tid) * H + h] = beta[((size_t)b * W + tid + 1) * H + h];
}

}  // namespace

int launch_decode(float *state, const void *q, const void *k, const void *v, const float *z,
                  const float *beta, const float *A, void *cq, void *ck, void *cv, float *cz,
                  float *cb, const int32_t *nacc, int N, int H, int W, int dtype, float g_min,
                  void *o, int32_t *err, cudaStream_t s) {
    const int64_t blocks = (int64_t)N * H;
    if (blocks <= 0) return KDA_OK;
    if (W > MAX_W) return KDA_ERR_UNSUPPORTED;
    if (dtype == KDA_BF16) {
        decode_kernel<__nv_bfloat16><<<(unsigned)blocks, DEC_THREADS, 0, s>>>(
            state, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, z, beta,
            A, (__nv_bfloat16 *)cq, (__nv_bfloat16 *)ck, (__nv_bfloat16 *)cv, cz, cb, nacc, H, W, g_min,
            (__nv_bfloat16 *)o, err);
    } else {
        decode_kernel<float><<<(unsigned)blocks, DEC_THREADS, 0, s>>>(
            state, (const float *)q, (const float *)k, (const float *)v, z, beta, A, (float *)cq,
            (float *)ck, (float *)cv, cz, cb, nacc, H, W, g_min, (float *)o, err);
    }
    note_launch("decode", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
