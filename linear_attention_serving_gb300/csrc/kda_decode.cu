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
// Mapping: persistent blocks walk the (sequence b, head h) items; thread
// (column pair j, part p) keeps rows [32 p, 32 p + 32) of state columns 2j and
// 2j + 1 in registers, so the d_k reductions are a register sum plus two
// shuffles, and every per-token vector element read from shared memory
// serves two columns.  The fp32 state
// is read and written exactly once per step.  While an item computes, one
// thread has already started bulk copies (cp.async.bulk + mbarrier) of the
// next item's state and token rows into shared memory, so the HBM stream
// never waits for the arithmetic.
//
// The per-channel decay is applied lazily: with s_t = prod_{tau<=t} alpha_tau
// (per row, over this step's tokens) the kernel keeps S = Diag(s_t) S^ and
// updates S^ only:
//   u = beta (v - S^^T (s_t . k)),  S^ += (k / s_t) u^T,  o = S^^T (s_t . q),
// which removes the Diag(alpha) pass over the state for every token.  At most
// 2W - 1 <= 15 tokens run per step, so s_t >= e^{5 * 15} = e^-75 stays a
// normal fp32 number (bounded gate, "Kimi K3 模型结构（2）", "后果一").
//
// The fused instantiation (FUSE) adds what the same decode paragraph puts in
// the kernel around the recurrence, with the module of "Kimi K3: the Manos,
// the Mythos ..." section "Kimi Linear": a causal depthwise short convolution
// (width 4) of the projected q, k and v over the committed stream (the cache
// and the convolution state hold pre-convolution inputs, so a replay runs the
// convolution again), and a per-head RMS norm of the outputs scaled by a
// sigmoid output gate.  Per item it adds the convolution state to the rows'
// bulk copy, reads the convolution weights of the head, and keeps the window's
// raw outputs and gate factors in shared memory for a final pass.
//
// Token prep.  The plain step prepares the step's tokens in one pass over the
// 128 channels.  With input options or the fusion it runs in two phases: all
// 256 threads take a token half each (convolution sliding in registers, gate
// factor, squared norms per warp), then the channel threads form the
// cumulative decay and the scaled vectors while the others write the
// convolution state and the output-gate factors.  Input options (beta's
// sigmoid included) are applied once per item and token, never in the
// recurrence loop.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

using namespace tc;

constexpr int MAX_W = 8;
constexpr int DEC_RP = 4;                     // row parts: threads sharing a pair of state columns
constexpr int DEC_R = D / DEC_RP;             // rows per thread (32)
constexpr int DEC_THREADS = D / 2 * DEC_RP;   // 256
constexpr int VPAD = D + 4 * DEC_RP;          // padded vector stride: row part p shifted by 4 p floats
constexpr int ROW_SLOT = 4 * 512;             // raw bytes per token: q | k | v | z rows, 512 B each

// Row part p of a vector starts 4 p floats further on, in its own 16-byte bank
// group.  A warp holds 8 column pairs x 4 row parts with the row part in the
// high lane bits, so each 8-lane phase of a 128-bit load reads one address.
__device__ __forceinline__ int vidx(int r) { return r + 4 * (r / DEC_R); }

__device__ __forceinline__ void store_pair(float *p, float a, float b) { *reinterpret_cast<float2 *>(p) = make_float2(a, b); }
__device__ __forceinline__ void store_pair(__nv_bfloat16 *p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}

constexpr int CONV_TAPS = 4;                  // short convolution width
constexpr int CONV_HIST = CONV_TAPS - 1;      // inputs kept per channel between steps
constexpr uint32_t CONV_STATE_BYTES = 3 * CONV_HIST * D * 4;  // q, k, v x 3 inputs x 128 channels

struct DecSmem {
    int ntok_max;
    size_t state, raw, kt, kh, qt, vt, cs, sg, ot, total;
    __host__ __device__ DecSmem(int W, bool fuse) {
        ntok_max = 2 * W - 1;
        state = 0;                                        // [128][128] fp32
        raw = state + (size_t)D * D * 4;                  // [ntok][q | k | v | z]
        kt = raw + (size_t)ntok_max * ROW_SLOT;           // s_t . k    [ntok][VPAD]
        kh = kt + (size_t)ntok_max * VPAD * 4;            // k / s_t    [ntok][VPAD]
        qt = kh + (size_t)ntok_max * VPAD * 4;            // s_t . q    [ntok][VPAD]
        vt = qt + (size_t)ntok_max * VPAD * 4;            // v          [ntok][D]
        cs = vt + (size_t)ntok_max * D * 4;               // FUSE: convolution state [3][3][D]
        sg = cs + (fuse ? CONV_STATE_BYTES : 0);          // FUSE: norm weight x sigmoid(gate) [W][D]
        ot = sg + (fuse ? (size_t)W * D * 4 : 0);         // FUSE: the window's raw outputs [W][D]
        total = ot + (fuse ? (size_t)W * D * 4 : 0);
    }
};


// One thread starts the bulk copies of item `item` (its state and token rows)
// into shared memory; completion is counted on `bar`, in two parts so that the
// state copy can start as soon as the state buffer is free and the rows copy
// as soon as the row buffer is.  `nacc` was read ahead of time; when it is out
// of range nothing is copied and the barrier completes without data.
template <bool FUSE>
__device__ __forceinline__ uint32_t item_bytes(int nacc, int W, uint32_t rowb) {
    // replayed rows carry no q unless the convolution needs it
    const uint32_t replay_row = (FUSE ? 3 : 2) * rowb + 512;
    return (uint32_t)(D * D * 4) + (uint32_t)nacc * replay_row + (uint32_t)W * (3 * rowb + 512) +
           (FUSE ? CONV_STATE_BYTES : 0u);
}
template <bool FUSE>
__device__ __forceinline__ void issue_state(int item, int nacc, int W, uint32_t rowb, const float *__restrict__ state,
                                            uint8_t *sm, const DecSmem &L, uint64_t *bar) {
    if (nacc < 0 || nacc > W - 1) {
        mbar_arrive(bar);
        return;
    }
    mbar_expect_tx(bar, item_bytes<FUSE>(nacc, W, rowb));
    bulk_g2s(sm + L.state, state + (size_t)item * D * D, D * D * 4, bar);
}
template <typename InT, bool FUSE>
__device__ __forceinline__ void issue_rows(int item, int nacc, int H, int W, const InT *__restrict__ q,
                                           const InT *__restrict__ k, const InT *__restrict__ v,
                                           const float *__restrict__ z, const InT *__restrict__ cq,
                                           const InT *__restrict__ ck, const InT *__restrict__ cv,
                                           const float *__restrict__ cz, const float *__restrict__ conv_state,
                                           uint8_t *sm, const DecSmem &L, uint64_t *bar) {
    if (nacc < 0 || nacc > W - 1) return;
    if (FUSE) bulk_g2s(sm + L.cs, conv_state + (size_t)item * (3 * CONV_HIST * D), CONV_STATE_BYTES, bar);
    const int b = item / H, h = item - b * H;
    const int ntok = nacc + W;
    const uint32_t rowb = (uint32_t)(D * sizeof(InT));
    for (int t = 0; t < ntok; ++t) {
        uint8_t *slot = sm + L.raw + (size_t)t * ROW_SLOT;
        if (t < nacc) {
            const size_t row = ((size_t)b * (W - 1) + t) * H + h;
            if (FUSE) bulk_g2s(slot, cq + row * D, rowb, bar);
            bulk_g2s(slot + 512, ck + row * D, rowb, bar);
            bulk_g2s(slot + 1024, cv + row * D, rowb, bar);
            bulk_g2s(slot + 1536, cz + row * D, 512, bar);
        } else {
            const size_t row = ((size_t)b * W + (t - nacc)) * H + h;
            bulk_g2s(slot, q + row * D, rowb, bar);
            bulk_g2s(slot + 512, k + row * D, rowb, bar);
            bulk_g2s(slot + 1024, v + row * D, rowb, bar);
            bulk_g2s(slot + 1536, z + row * D, 512, bar);
        }
    }
}

// Decay factor exp(g) of one channel, g = g_min sigmoid(e^{A_h} z) (the gate of
// "Kimi K3 模型结构（2）" eq. (5)), with the hardware base-2 exponential and a
// fast reciprocal; relative error a few fp32 ulp.
__device__ __forceinline__ float dec_decay(float g_min, float eA, float z) {
    const float e = ex2(-eA * z * 1.4426950408889634f);
    return ex2(__fdividef(g_min, 1.f + e) * 1.4426950408889634f);
}

// beta of token slot t of item `item` for either accepted count: thread t < W-1
// holds the cached draft's beta in `bc`, thread t < W the window's in `bw`.
__device__ __forceinline__ void load_betas(int item, int H, int W, int tid, const float *__restrict__ beta,
                                           const float *__restrict__ cb, float &bc, float &bw) {
    const int b = item / H, h = item - b * H;
    bc = (tid < W - 1) ? cb[((size_t)b * (W - 1) + tid) * H + h] : 0.f;
    bw = (tid < W) ? beta[((size_t)b * W + tid) * H + h] : 0.f;
}

// OPTS compiles the input options (KDA_FLAG_*) in: a separate instantiation,
// so that the default path keeps its registers.  FUSE adds the short
// convolution and the gated output norm (the fused step).
template <typename InT, bool OPTS, bool FUSE>
__global__ void __launch_bounds__(DEC_THREADS, 2)
decode_kernel(float *__restrict__ state, const InT *__restrict__ q, const InT *__restrict__ k,
              const InT *__restrict__ v, const float *__restrict__ z, const float *__restrict__ beta,
              const float *__restrict__ A, InT *__restrict__ cq, InT *__restrict__ ck,
              InT *__restrict__ cv, float *__restrict__ cz, float *__restrict__ cb,
              const int32_t *__restrict__ nacc_p, int N, int H, int W, float g_min, InT *__restrict__ o,
              int32_t *__restrict__ err, int flags, DecFuse fz, long long wait_budget) {
    extern __shared__ __align__(128) uint8_t smdyn[];
    __shared__ uint64_t full_bar;
    __shared__ float sbeta[2][2 * MAX_W];
    __shared__ float sbeff[OPTS ? 2 : 1][2 * MAX_W];  // OPTS: the betas the recurrence uses (after the sigmoid option)
    __shared__ __align__(16) float scommit[VPAD];
    __shared__ float snorm[2 * MAX_W][4][2];  // KDA_FLAG_QK_L2NORM: squared norms per token and warp
    __shared__ __align__(16) float sqo[MAX_W][DEC_THREADS / 32];  // FUSE: squared output sums per window token and warp
    const bool l2norm = OPTS && (flags & KDA_FLAG_QK_L2NORM) != 0;
    const bool bsig = OPTS && (flags & KDA_FLAG_BETA_SIGMOID) != 0;
    const bool qscale = OPTS && (flags & KDA_FLAG_Q_SCALE) != 0;
    const bool silu = FUSE && OPTS && (flags & KDA_FLAG_CONV_SILU) != 0;

    const DecSmem L(W, FUSE);
    uint8_t *sm = smdyn;
    float *sS = reinterpret_cast<float *>(sm + L.state);
    float(*kt)[VPAD] = reinterpret_cast<float(*)[VPAD]>(sm + L.kt);
    float(*kh)[VPAD] = reinterpret_cast<float(*)[VPAD]>(sm + L.kh);
    float(*qt)[VPAD] = reinterpret_cast<float(*)[VPAD]>(sm + L.qt);
    float(*vt)[D] = reinterpret_cast<float(*)[D]>(sm + L.vt);
    const float(*cst)[CONV_HIST][D] = reinterpret_cast<const float(*)[CONV_HIST][D]>(sm + L.cs);
    float(*sg)[D] = reinterpret_cast<float(*)[D]>(sm + L.sg);
    float(*ot)[D] = reinterpret_cast<float(*)[D]>(sm + L.ot);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int part = lane >> 3;                                 // row part: lanes 8 p .. 8 p + 7
    const int col = 2 * (warp * (32 / DEC_RP) + (lane & 7));  // first of this thread's two columns
    const int rbase = part * DEC_R;
    const int n_items = N * H;
    const uint32_t rowb = (uint32_t)(D * sizeof(InT));

    if (tid == 0) {
        mbar_init(&full_bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    int item = blockIdx.x;
    // per-item scalars (accepted count and betas) are read two items ahead, so
    // their global-load latency never sits in front of a bulk-copy issue
    int nacc_cur = 0, nacc_nx = 0;
    float bc_cur = 0.f, bw_cur = 0.f, bc_nx = 0.f, bw_nx = 0.f;
    if (item < n_items) {
        nacc_cur = nacc_p ? nacc_p[item / H] : 0;
        load_betas(item, H, W, tid, beta, cb, bc_cur, bw_cur);
        if (item + (int)gridDim.x < n_items) {
            nacc_nx = nacc_p ? nacc_p[(item + gridDim.x) / H] : 0;
            load_betas(item + gridDim.x, H, W, tid, beta, cb, bc_nx, bw_nx);
        }
        if (tid == 0) {
            issue_state<FUSE>(item, nacc_cur, W, rowb, state, sm, L, &full_bar);
            issue_rows<InT, FUSE>(item, nacc_cur, H, W, q, k, v, z, cq, ck, cv, cz, fz.conv_state, sm, L,
                                  &full_bar);
        }
    }
    bool timed_out = false;
    for (int it = 0; item < n_items; item += gridDim.x, ++it) {
        const int b = item / H, h = item - b * H;
        const float A_h = __ldg(A + h);  // loaded before the wait for the item's copies
        // FUSE: the head's convolution taps of this thread's channel, loaded before
        // the wait for the item's copies so that their latency hides behind it
        float4 wq, wk, wv;
        if (FUSE) {
            const int c = tid & (D - 1);
            wq = __ldg(reinterpret_cast<const float4 *>(fz.conv_w) + ((size_t)0 * H + h) * D + c);
            wk = __ldg(reinterpret_cast<const float4 *>(fz.conv_w) + ((size_t)1 * H + h) * D + c);
            wv = __ldg(reinterpret_cast<const float4 *>(fz.conv_w) + ((size_t)2 * H + h) * D + c);
        }
        const int next = item + gridDim.x, next2 = next + gridDim.x;
        const int nacc_next = nacc_nx;
        int nacc_nn = 0;
        float bc_nn = 0.f, bw_nn = 0.f;
        if (next2 < n_items) {
            nacc_nn = nacc_p ? nacc_p[next2 / H] : 0;
            load_betas(next2, H, W, tid, beta, cb, bc_nn, bw_nn);
        }
        const int nacc = nacc_cur;
        if (!mbar_wait_for(&full_bar, (uint32_t)(it & 1), wait_budget)) timed_out = true;
        if (__syncthreads_or(timed_out)) {
            if (tid == 0) {
                if (err) atomicOr(err, KDA_DEVERR_TIMEOUT);
                // the item's copies are still landing in shared memory: let them
                // finish (fixed budget) before the block leaves
                mbar_wait(&full_bar, (uint32_t)(it & 1));
            }
            break;
        }
        if (nacc < 0 || nacc > W - 1) {
            // out-of-range accepted count: this sequence is left untouched
            if (tid == 0) {
                if (err) atomicOr(err, KDA_DEVERR_NUM_ACCEPTED);
                if (next < n_items) {
                    issue_state<FUSE>(next, nacc_next, W, rowb, state, sm, L, &full_bar);
                    issue_rows<InT, FUSE>(next, nacc_next, H, W, q, k, v, z, cq, ck, cv, cz, fz.conv_state, sm,
                                          L, &full_bar);
                }
            }
            nacc_cur = nacc_nx;
            bc_cur = bc_nx;
            bw_cur = bw_nx;
            nacc_nx = nacc_nn;
            bc_nx = bc_nn;
            bw_nx = bw_nn;
            continue;
        }
        const int ntok = nacc + W;
        float *Sg = state + (size_t)item * D * D;
        float *sbt = sbeta[it & 1];
        float *sbe = OPTS ? sbeff[it & 1] : sbt;
        if (tid < nacc) sbt[tid] = bc_cur;
        if (tid < W) sbt[nacc + tid] = bw_cur;
        if (OPTS) {
            // input option: beta logits through the sigmoid, once per item and token
            if (tid < nacc) sbe[tid] = bsig ? 1.f / (1.f + expf(-bc_cur)) : bc_cur;
            if (tid < W) sbe[nacc + tid] = bsig ? 1.f / (1.f + expf(-bw_cur)) : bw_cur;
        }

        const float eA = expf(A_h);
        if (tid == D) {
            // the new drafts' projected inputs replace this sequence's cache slots
            // (the prep reads the raw rows but never writes them)
            for (int t = nacc + 1; t < ntok; ++t) {
                const uint8_t *slot = sm + L.raw + (size_t)t * ROW_SLOT;
                const size_t row = ((size_t)b * (W - 1) + (t - nacc - 1)) * H + h;
                bulk_s2g(cq + row * D, slot, rowb);
                bulk_s2g(ck + row * D, slot + 512, rowb);
                bulk_s2g(cv + row * D, slot + 1024, rowb);
                bulk_s2g(cz + row * D, slot + 1536, 512);
            }
            bulk_commit();
        }
        // FUSE: the window's output-gate logits, loaded here and used after phase A
        float gl[MAX_W];
        if (FUSE && tid >= D) {
#pragma unroll
            for (int j = 0; j < MAX_W; ++j)
                gl[j] = j < W ? __ldg(fz.o_gate + (((size_t)b * W + j) * H + h) * D + (tid - D)) : 0.f;
        }
        if (!FUSE && !OPTS) {
            // plain step: channel c of every token in one pass (inputs, the
            // cumulative decay s_t over the step's tokens, s_t k, k / s_t, s_t q)
            if (tid < D) {
                const int c = tid, vc = vidx(c);
                float sc = 1.f;
#pragma unroll 2
                for (int t = 0; t < ntok; ++t) {
                    const uint8_t *slot = sm + L.raw + (size_t)t * ROW_SLOT;
                    float qq = t < nacc ? 0.f : to_f32(reinterpret_cast<const InT *>(slot)[c]);
                    float kk = to_f32(reinterpret_cast<const InT *>(slot + 512)[c]);
                    const float zz = reinterpret_cast<const float *>(slot + 1536)[c];
                    sc *= dec_decay(g_min, eA, zz);
                    kt[t][vc] = kk * sc;
                    kh[t][vc] = __fdividef(kk, sc);
                    qt[t][vc] = qq * sc;
                    vt[t][c] = to_f32(reinterpret_cast<const InT *>(slot + 1024)[c]);
                    if (t == nacc) scommit[vc] = sc;
                }
            }
        } else {
            {
                // phase A, token-parallel: warps 0-3 take the first half of the step's
                // tokens and warps 4-7 the second, a warp = 32 channels of one token.
                // The (convolved) inputs go to qt, kt, vt, the decay factor exp(g_t)
                // to kh, and the squared norms of q and k to snorm.
                const int c = tid & (D - 1), vc = vidx(c), quarter = warp & 3;
                const int tmid = (ntok + 1) >> 1;
                const int t_begin = tid < D ? 0 : tmid, t_end = tid < D ? tmid : ntok;
                float hq0, hq1, hq2, hk0, hk1, hk2, hv0, hv1, hv2;  // FUSE: x_{t-3}, x_{t-2}, x_{t-1}
                if (FUSE) {
                    // the three inputs before t_begin: token rows, or the convolution state
                    // for stream positions before the first token
                    auto hist = [&](int x, int ps) {
                        return ps >= 0 ? to_f32(reinterpret_cast<const InT *>(sm + L.raw + (size_t)ps * ROW_SLOT + x * 512)[c])
                                       : cst[x][CONV_HIST + ps][c];
                    };
                    hq0 = hist(0, t_begin - 3), hq1 = hist(0, t_begin - 2), hq2 = hist(0, t_begin - 1);
                    hk0 = hist(1, t_begin - 3), hk1 = hist(1, t_begin - 2), hk2 = hist(1, t_begin - 1);
                    hv0 = hist(2, t_begin - 3), hv1 = hist(2, t_begin - 2), hv2 = hist(2, t_begin - 1);
                }
#pragma unroll 2
                for (int t = t_begin; t < t_end; ++t) {
                    const uint8_t *slot = sm + L.raw + (size_t)t * ROW_SLOT;
                    // replayed tokens of the plain step carry no q (never read below)
                    float xq = to_f32(reinterpret_cast<const InT *>(slot)[c]);
                    float xk = to_f32(reinterpret_cast<const InT *>(slot + 512)[c]);
                    float xv = to_f32(reinterpret_cast<const InT *>(slot + 1024)[c]);
                    if (FUSE) {
                        // short convolution over [state, replayed drafts, window]:
                        // y_t = sum_j w_j x_{t-3+j}, tap 3 on the current token
                        float yq = fmaf(wq.w, xq, fmaf(wq.z, hq2, fmaf(wq.y, hq1, wq.x * hq0)));
                        float yk = fmaf(wk.w, xk, fmaf(wk.z, hk2, fmaf(wk.y, hk1, wk.x * hk0)));
                        float yv = fmaf(wv.w, xv, fmaf(wv.z, hv2, fmaf(wv.y, hv1, wv.x * hv0)));
                        hq0 = hq1, hq1 = hq2, hq2 = xq;
                        hk0 = hk1, hk1 = hk2, hk2 = xk;
                        hv0 = hv1, hv1 = hv2, hv2 = xv;
                        if (silu) {
                            yq = __fdividef(yq, 1.f + __expf(-yq));
                            yk = __fdividef(yk, 1.f + __expf(-yk));
                            yv = __fdividef(yv, 1.f + __expf(-yv));
                        }
                        xq = yq;
                        xk = yk;
                        xv = yv;
                    }
                    qt[t][vc] = xq;
                    kt[t][vc] = xk;
                    vt[t][c] = xv;
                    kh[t][vc] = dec_decay(g_min, eA, reinterpret_cast<const float *>(slot + 1536)[c]);
                    if (l2norm) {
                        // input option: squared norms over the 128 channels (no q for replays)
                        float pq = t < nacc ? 0.f : xq * xq, pk = xk * xk;
#pragma unroll
                        for (int m = 16; m > 0; m >>= 1) {
                            pq += __shfl_xor_sync(0xffffffffu, pq, m);
                            pk += __shfl_xor_sync(0xffffffffu, pk, m);
                        }
                        if (lane == 0) {
                            snorm[t][quarter][0] = pq;
                            snorm[t][quarter][1] = pk;
                        }
                    }
                }
            }
            __syncthreads();
            if (tid < D) {
                // phase B, channel c: the cumulative decay s_t over the step's tokens
                // and the scaled vectors s_t k, k / s_t, s_t q
                const int c = tid, vc = vidx(c);
                float sc = 1.f;
#pragma unroll 2
                for (int t = 0; t < ntok; ++t) {
                    sc *= kh[t][vc];
                    float qq = t < nacc ? 0.f : qt[t][vc];
                    float kk = kt[t][vc];
                    if (l2norm) {
                        qq *= rsqrtf(snorm[t][0][0] + snorm[t][1][0] + snorm[t][2][0] + snorm[t][3][0] + L2NORM_EPS);
                        kk *= rsqrtf(snorm[t][0][1] + snorm[t][1][1] + snorm[t][2][1] + snorm[t][3][1] + L2NORM_EPS);
                    }
                    if (qscale) qq *= Q_SCALE;  // input option: q d_k^-1/2, after the norm
                    kt[t][vc] = kk * sc;
                    kh[t][vc] = __fdividef(kk, sc);
                    qt[t][vc] = qq * sc;
                    if (t == nacc) scommit[vc] = sc;
                }
            } else if (FUSE) {
                const int c = tid - D;
                // the convolution state becomes the three inputs ending at t0 (stream
                // positions nacc - 2 .. nacc; negative ones are still in the old state)
                float *cs_out = fz.conv_state + (size_t)item * (3 * CONV_HIST * D) + c;
#pragma unroll
                for (int x = 0; x < 3; ++x)
#pragma unroll
                    for (int j = 0; j < CONV_HIST; ++j) {
                        const int ps = nacc - (CONV_HIST - 1) + j;
                        cs_out[(x * CONV_HIST + j) * D] =
                            ps >= 0 ? to_f32(reinterpret_cast<const InT *>(sm + L.raw + (size_t)ps * ROW_SLOT + x * 512)[c])
                                    : cst[x][CONV_HIST + ps][c];
                    }
                // output gate: norm weight x sigmoid(gate logit) per window token and channel
                const float wn = __ldg(fz.o_norm_w + c);
#pragma unroll
                for (int j = 0; j < MAX_W; ++j)
                    if (j < W) sg[j][c] = __fdividef(wn, 1.f + __expf(-gl[j]));
            }
        }
        if (tid < W - 1) cb[((size_t)b * (W - 1) + tid) * H + h] = sbt[nacc + 1 + tid];
        // state of this item: shared memory -> registers, after the token prep (which
        // so runs with the registers the state takes); past the barrier the state
        // buffer takes the next item's state
        // (row r: columns col, col + 1 as one pair, updated by paired fp32 FMAs)
        float2 sp[DEC_R];
#pragma unroll
        for (int i = 0; i < DEC_R; ++i) sp[i] = *reinterpret_cast<const float2 *>(&sS[(rbase + i) * D + col]);
        __syncthreads();
        if (tid == 0 && next < n_items) issue_state<FUSE>(next, nacc_next, W, rowb, state, sm, L, &full_bar);
        // the row buffers are free once the cache copies have read them: the next item's token rows
        if (tid == D) bulk_wait_read_all();
        if (tid == D && next < n_items)
            issue_rows<InT, FUSE>(next, nacc_next, H, W, q, k, v, z, cq, ck, cv, cz, fz.conv_state, sm, L,
                                  &full_bar);

        // the recurrence over replay + bonus + drafts
        const float *bt = sbe;
        for (int t = 0; t < ntok; ++t) {
            // two partial sums per column keep the FMA chains short: pa (rows i, i + 2)
            // and pb (rows i + 1, i + 3), each holding both columns
            float2 pa = make_float2(0.f, 0.f), pb = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < DEC_R; i += 4) {
                const float4 kv = *reinterpret_cast<const float4 *>(&kt[t][vidx(rbase + i)]);
                pa = __ffma2_rn(sp[i], make_float2(kv.x, kv.x), pa);
                pb = __ffma2_rn(sp[i + 1], make_float2(kv.y, kv.y), pb);
                pa = __ffma2_rn(sp[i + 2], make_float2(kv.z, kv.z), pa);
                pb = __ffma2_rn(sp[i + 3], make_float2(kv.w, kv.w), pb);
            }
            float acc0 = pa.x + pb.x, acc1 = pa.y + pb.y;
#pragma unroll
            for (int m = 8; m < 32; m <<= 1) {  // the four row parts
                acc0 += __shfl_xor_sync(0xffffffffu, acc0, m);
                acc1 += __shfl_xor_sync(0xffffffffu, acc1, m);
            }
            const float2 vv = *reinterpret_cast<const float2 *>(&vt[t][col]);
            const float bb = bt[t];
            const float2 uu = make_float2(bb * (vv.x - acc0), bb * (vv.y - acc1));
#pragma unroll
            for (int i = 0; i < DEC_R; i += 4) {
                const float4 kv = *reinterpret_cast<const float4 *>(&kh[t][vidx(rbase + i)]);
                sp[i] = __ffma2_rn(make_float2(kv.x, kv.x), uu, sp[i]);
                sp[i + 1] = __ffma2_rn(make_float2(kv.y, kv.y), uu, sp[i + 1]);
                sp[i + 2] = __ffma2_rn(make_float2(kv.z, kv.z), uu, sp[i + 2]);
                sp[i + 3] = __ffma2_rn(make_float2(kv.w, kv.w), uu, sp[i + 3]);
            }
            if (t >= nacc) {
                float2 qa = make_float2(0.f, 0.f), qb = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < DEC_R; i += 4) {
                    const float4 qv = *reinterpret_cast<const float4 *>(&qt[t][vidx(rbase + i)]);
                    qa = __ffma2_rn(sp[i], make_float2(qv.x, qv.x), qa);
                    qb = __ffma2_rn(sp[i + 1], make_float2(qv.y, qv.y), qb);
                    qa = __ffma2_rn(sp[i + 2], make_float2(qv.z, qv.z), qa);
                    qb = __ffma2_rn(sp[i + 3], make_float2(qv.w, qv.w), qb);
                }
                float ao0 = qa.x + qb.x, ao1 = qa.y + qb.y;
#pragma unroll
                for (int m = 8; m < 32; m <<= 1) {  // the four row parts
                    ao0 += __shfl_xor_sync(0xffffffffu, ao0, m);
                    ao1 += __shfl_xor_sync(0xffffffffu, ao1, m);
                }
                if (FUSE) {
                    // the window's raw outputs wait for their norm; squared sums per warp
                    // (fixed order later: the result does not depend on warp timing)
                    float pp = ao0 * ao0 + ao1 * ao1;
                    pp += __shfl_xor_sync(0xffffffffu, pp, 1);
                    pp += __shfl_xor_sync(0xffffffffu, pp, 2);
                    pp += __shfl_xor_sync(0xffffffffu, pp, 4);
                    if (part == 0) *reinterpret_cast<float2 *>(&ot[t - nacc][col]) = make_float2(ao0, ao1);
                    if (lane == 0) sqo[t - nacc][warp] = pp;
                } else if (part == 0) {
                    store_pair(o + (((size_t)b * W + (t - nacc)) * H + h) * D + col, ao0, ao1);
                }
            }
            if (t == nacc) {
                // commit: S = Diag(s_t) S^, written back in place
#pragma unroll
                for (int i = 0; i < DEC_R; i += 4) {
                    const float4 sc4 = *reinterpret_cast<const float4 *>(&scommit[vidx(rbase + i)]);
                    __stcs(reinterpret_cast<float2 *>(&Sg[(size_t)(rbase + i) * D + col]), __fmul2_rn(sp[i], make_float2(sc4.x, sc4.x)));
                    __stcs(reinterpret_cast<float2 *>(&Sg[(size_t)(rbase + i + 1) * D + col]), __fmul2_rn(sp[i + 1], make_float2(sc4.y, sc4.y)));
                    __stcs(reinterpret_cast<float2 *>(&Sg[(size_t)(rbase + i + 2) * D + col]), __fmul2_rn(sp[i + 2], make_float2(sc4.z, sc4.z)));
                    __stcs(reinterpret_cast<float2 *>(&Sg[(size_t)(rbase + i + 3) * D + col]), __fmul2_rn(sp[i + 3], make_float2(sc4.w, sc4.w)));
                }
            }
        }

        nacc_cur = nacc_nx;
        bc_cur = bc_nx;
        bw_cur = bw_nx;
        nacc_nx = nacc_nn;
        bc_nx = bc_nn;
        bw_nx = bw_nn;
        __syncthreads();  // vectors are rewritten by the next item
        if (FUSE) {
            // gated RMS norm over the 128 value channels of each window token; the
            // next item's shared-memory writes come after its first barrier
            for (int i = tid; i < W * (D / 4); i += DEC_THREADS) {
                const int j = i / (D / 4), cc = 4 * (i % (D / 4));
                const float4 s0 = *reinterpret_cast<const float4 *>(&sqo[j][0]);
                const float4 s1 = *reinterpret_cast<const float4 *>(&sqo[j][4]);
                const float ss = ((s0.x + s0.y) + (s0.z + s0.w)) + ((s1.x + s1.y) + (s1.z + s1.w));
                const float r = rsqrtf(ss * (1.f / D) + fz.o_norm_eps);
                const float4 ov = *reinterpret_cast<const float4 *>(&ot[j][cc]);
                const float4 gv = *reinterpret_cast<const float4 *>(&sg[j][cc]);
                InT *op = o + (((size_t)b * W + j) * H + h) * D + cc;
                store_pair(op, ov.x * r * gv.x, ov.y * r * gv.y);
                store_pair(op + 2, ov.z * r * gv.z, ov.w * r * gv.w);
            }
        }
    }
    if (tid == D) bulk_wait_all();  // the cache copies have landed before the block exits
}

}  // namespace

namespace {

template <typename InT, bool FUSE>
int launch_decode_t(float *state, const void *q, const void *k, const void *v, const float *z,
                    const float *beta, const float *A, void *cq, void *ck, void *cv, float *cz, float *cb,
                    const int32_t *nacc, int N, int H, int W, float g_min, void *o, int32_t *err, int flags,
                    const DecFuse &fz, cudaStream_t s) {
    const long long items = (long long)N * H;
    const DecSmem L(W, FUSE);
    const int smem = (int)L.total;
    auto kern = flags ? decode_kernel<InT, true, FUSE> : decode_kernel<InT, false, FUSE>;
    int per_sm = 1;
    if (prepare_kernel((const void *)kern, smem, DEC_THREADS, &per_sm) != KDA_OK) return KDA_ERR_CUDA;
    const long long slots = (long long)device_sm_count() * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(items < slots ? items : slots);
    kern<<<grid, DEC_THREADS, smem, s>>>(state, (const InT *)q, (const InT *)k, (const InT *)v, z, beta, A,
                                         (InT *)cq, (InT *)ck, (InT *)cv, cz, cb, nacc, N, H, W, g_min,
                                         (InT *)o, err, flags, fz, wait_budget());
    return KDA_OK;
}

}  // namespace

// fz == nullptr: the plain step; otherwise the fused step with those operands.
int launch_decode(float *state, const void *q, const void *k, const void *v, const float *z,
                  const float *beta, const float *A, void *cq, void *ck, void *cv, float *cz,
                  float *cb, const int32_t *nacc, int N, int H, int W, int dtype, float g_min,
                  void *o, int32_t *err, int flags, const DecFuse *fz, cudaStream_t s) {
    if ((long long)N * H <= 0) return KDA_OK;
    if (W > MAX_W) return KDA_ERR_UNSUPPORTED;
    const DecFuse none{};
    int rc;
    if (dtype == KDA_BF16)
        rc = fz ? launch_decode_t<__nv_bfloat16, true>(state, q, k, v, z, beta, A, cq, ck, cv, cz, cb, nacc, N, H,
                                                        W, g_min, o, err, flags, *fz, s)
                : launch_decode_t<__nv_bfloat16, false>(state, q, k, v, z, beta, A, cq, ck, cv, cz, cb, nacc, N,
                                                         H, W, g_min, o, err, flags, none, s);
    else
        rc = fz ? launch_decode_t<float, true>(state, q, k, v, z, beta, A, cq, ck, cv, cz, cb, nacc, N, H, W,
                                                g_min, o, err, flags, *fz, s)
                : launch_decode_t<float, false>(state, q, k, v, z, beta, A, cq, ck, cv, cz, cb, nacc, N, H, W,
                                                 g_min, o, err, flags, none, s);
    if (rc != KDA_OK) return rc;
    note_launch(fz ? "decode_fused" : "decode", s);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
