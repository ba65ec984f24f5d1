// kda_internal.cuh -- shared definitions of the KDA forward kernels (sm_103a).
//
// Sources cited in this library (page title, section):
//   [K3-7] "Kimi K3 模型结构（7）：结构决定系统"
//   [K3-2] "Kimi K3 模型结构（2）：序列维度（下），chunkwise 并行与下界衰减"
//   [SA]   "Kimi K3: the Manos, the Mythos ..." (SemiAnalysis), "FlashKDA 算法"
//
// Chunk algebra used by every prefill kernel ([SA] "算法", [K3-2] "UT 变换",
// "块间递推与块内输出"), per chunk of C = 64 tokens with inclusive cumulative
// log decay G_r = sum_{s<=r} g_s and a_r = exp(G_r):
//   L    = StrictTril(Diag(beta) K_decay K_inv^T),  INV = (I + L)^-1
//   M_qk = Tril(Q_decay K_inv^T)
// The prep kernel folds everything that does not depend on the entering state
// into five per-chunk operands:
//   W  = INV Diag(beta) K_decay            U0 = INV Diag(beta) V
//   Q' = Q_decay - M_qk W                  O0 = M_qk U0
//   K_restore^T,  a_C = exp(G_last)
// so that the sequential scan over chunks is
//   U = U0 - W S,   O = O0 + Q' S,   S <- Diag(a_C) S + K_restore^T U,
// which is the same U = INV Diag(beta)(V - K_decay S), O = Q_decay S + M_qk U
// as the pages, with the state-independent products moved off the chain.
#pragma once

#include <cuda.h>  // CUtensorMap (a type only; the driver functions come through the runtime)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int D = 128;       // d_k = d_v
constexpr int C = 64;        // chunk length
constexpr int SUB = 16;      // sub-tile length ([K3-2] "数值问题：1/Γ 会溢出")
constexpr int NSUB = C / SUB;

// ---------------------------------------------------------------- chunk plan
struct ChunkInfo {
    int32_t tok;    // first token (global index)
    int32_t len;    // 1..64 valid tokens
    int32_t doc;    // document index
    int32_t flags;  // bit 0: first chunk of its document, bit 1: last chunk
};
constexpr int32_t CHUNK_FIRST = 1;
constexpr int32_t CHUNK_LAST = 2;

// Chunks are cut per document ([K3-7] "文档边界": the state restarts at every
// document start), so no chunk straddles two documents.  With cu_seqlens NULL
// the documents have equal length and the plan is arithmetic ("uniform").
struct Plan {
    int uniform;             // 1: equal-length documents, no table
    int n_seqs;
    int seq_len;             // uniform mode
    int chunks_per_seq;      // uniform mode
    int max_chunks;          // grid bound
    const ChunkInfo *table;  // table mode: [max_chunks]
    const int32_t *doc_off;  // table mode: [n_seqs + 1] first chunk of each document
    const int32_t *n_chunks; // table mode: device count
    int32_t *err;            // device error word (bit flags kda_device_error)
    int flags;               // input options (KDA_FLAG_*) for the preparation kernels
    long long wait_budget;   // clock cycles a wait on another block's flag may take
};

constexpr float L2NORM_EPS = 1e-6f;  // KDA_FLAG_QK_L2NORM: x / sqrt(sum(x^2) + eps)
constexpr float Q_SCALE = 0.08838834764831845f;  // KDA_FLAG_Q_SCALE: d_k^-1/2 = 1 / sqrt(128)
// every input option of the prefill and the plain decode step
constexpr int PREFILL_FLAGS = KDA_FLAG_QK_L2NORM | KDA_FLAG_BETA_SIGMOID | KDA_FLAG_Q_SCALE;

__device__ __forceinline__ int plan_n_chunks(const Plan &p) {
    return p.uniform ? p.n_seqs * p.chunks_per_seq : *p.n_chunks;
}

__device__ __forceinline__ ChunkInfo plan_chunk(const Plan &p, int c) {
    if (!p.uniform) return p.table[c];
    ChunkInfo ci;
    const int d = c / p.chunks_per_seq;
    const int i = c - d * p.chunks_per_seq;
    ci.doc = d;
    ci.tok = d * p.seq_len + i * C;
    const int rem = p.seq_len - i * C;
    ci.len = rem < C ? rem : C;
    ci.flags = (i == 0 ? CHUNK_FIRST : 0) | (i == p.chunks_per_seq - 1 ? CHUNK_LAST : 0);
    return ci;
}

// True when the device planner rejected cu_seqlens; kernels then write nothing.
__device__ __forceinline__ bool plan_failed(const Plan &p) {
    return !p.uniform && (*(volatile const int32_t *)p.err & KDA_DEVERR_CU_SEQLENS);
}

__device__ __forceinline__ void plan_doc_range(const Plan &p, int d, int &c0, int &c1) {
    if (p.uniform) {
        c0 = d * p.chunks_per_seq;
        c1 = c0 + p.chunks_per_seq;
    } else {
        c0 = p.doc_off[d];
        c1 = p.doc_off[d + 1];
    }
}

// Balanced chunk-aligned split of n chunks into nseg segments; earlier
// segments take one more chunk when the split is not exact.
__host__ __device__ __forceinline__ void segment_range(int n, int nseg, int i, int &c0, int &c1) {
    const int base = n / nseg, extra = n % nseg;
    c0 = i * base + (i < extra ? i : extra);
    c1 = c0 + base + (i < extra ? 1 : 0);
}

// ---------------------------------------------------------------- records
// bf16 record of one (chunk, head), written by the tcgen05 prep kernel, read
// by the tcgen05 scan (the state chain) and by the output kernel.  With
// G = K_restore^T W and H = K_restore^T U0 the state update of a chunk is one
// product, S <- Diag(a_C) S + H - G S; the output O = O0 + Q' S needs the
// entering state S, which the scan stores into the record.
//   [0, 32768)       G: 128 x 128 bf16 image, K-major, 128-byte swizzle, two
//                    64-column k-blocks of 128 rows x 128 B
//   [32768, 33280)   a_C [128] fp32
//   [33792, 50176)   Q': 64 x 128 bf16 image, two k-blocks of 64 rows x 128 B
//   [50176, 82944)   H in 16-column slices: [8][128 rows][16] bf16
//   [82944, 99328)   O0 in 16-column slices: [8][64 rows][16] bf16
//   [99328, 132096)  S entering the chunk, bf16, MN-major with the 32-byte
//                    swizzle: [8 column blocks][128 rows][16], the two 16-byte
//                    halves of row r swapped when (r >> 2) is odd
// A scan block that owns state columns [16 s, 16 (s + n)) copies [0, 33280)
// and n adjacent H slices, and writes n adjacent S blocks.
constexpr size_t REC_BF16_G = 0;
constexpr size_t REC_BF16_AC = 32768;
constexpr size_t REC_BF16_SHARED = 33280;
constexpr size_t REC_BF16_QP = 33792;
constexpr size_t REC_BF16_H = 50176;
constexpr size_t REC_BF16_HSLICE = 4096;
constexpr size_t REC_BF16_O0 = 82944;
constexpr size_t REC_BF16_OSLICE = 2048;
constexpr size_t REC_BF16_S = 99328;
constexpr size_t REC_BF16_SBLOCK = 4096;
constexpr size_t REC_BF16_BYTES = 132096;

// Byte offset of element (row r, column col) inside a 16-column slice region
// whose slices hold `rows` rows.
__host__ __device__ __forceinline__ uint32_t slice_offset(int r, int col, int rows) {
    return (uint32_t)((col >> 4) * rows * 32 + r * 32 + (col & 15) * 2);
}

// fp32 record of one (chunk, head), plain row-major, for the exact path.
//   W, Q', K_restore, U0, O0: [64][128] fp32 each;  a_C [128] fp32
constexpr size_t REC_F32_W = 0;
constexpr size_t REC_F32_Q = 32768;
constexpr size_t REC_F32_KR = 65536;
constexpr size_t REC_F32_U0 = 98304;
constexpr size_t REC_F32_O0 = 131072;
constexpr size_t REC_F32_AC = 163840;
constexpr size_t REC_F32_BYTES = 164352;

// Byte offset of element (row, col) of a bf16 K-major operand image with the
// 128-byte swizzle: 64 columns per k-block, rows of 128 B, the 16-byte group
// index XOR-ed with (row mod 8).  `rows` is the number of rows per k-block.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int row, int col, int rows) {
    const int kb = col >> 6, cc = col & 63;
    return (uint32_t)(kb * rows * 128 + row * 128 + ((((cc >> 3) ^ (row & 7)) & 7) << 4) + (cc & 7) * 2);
}

// ---------------------------------------------------------------- workspace
// [0, 256)                   header: int32 err, int32 n_chunks
// table                      ChunkInfo[max_chunks]
// doc_off                    int32[n_seqs + 1]
// records                    max_chunks * H * record bytes
// (segment scan) pairs       fp32 [2][H][n_seg][D][D]  (M then S~)
// (segment scan) s_enter     fp32 [H][n_seg][D][D]
struct Workspace {
    size_t off_table, off_doc, off_rec, off_ready, off_pairs, off_enter, total;
    int max_chunks;
    size_t rec_bytes;
};

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static inline Workspace workspace_layout(int64_t T_total, int H, int n_seqs, int n_seg, int dtype) {
    Workspace w;
    w.max_chunks = (int)(T_total / C + n_seqs);
    w.rec_bytes = dtype == KDA_BF16 ? REC_BF16_BYTES : REC_F32_BYTES;
    size_t off = 256;
    w.off_ready = off;  // one record-ready flag per (chunk, head) for the fused prefill, right after
                        // the header so that one memset clears both
    off = align_up(off + sizeof(int) * (size_t)w.max_chunks * (size_t)H, 256);
    w.off_table = off;
    off = align_up(off + sizeof(ChunkInfo) * (size_t)w.max_chunks, 256);
    w.off_doc = off;
    off = align_up(off + sizeof(int32_t) * (size_t)(n_seqs + 1), 1024);
    w.off_rec = off;
    off = align_up(off + w.rec_bytes * (size_t)w.max_chunks * (size_t)H, 1024);
    w.off_pairs = off;
    if (n_seg > 0) off = align_up(off + sizeof(float) * 2 * (size_t)H * n_seg * D * D, 1024);
    w.off_enter = off;
    if (n_seg > 0) off = align_up(off + sizeof(float) * (size_t)H * n_seg * D * D, 1024);
    w.total = off;
    return w;
}

// ---------------------------------------------------------------- helpers
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Gate, [K3-2] eq. (5): g = g_min * sigmoid(exp(A_h) * z), natural log.
__device__ __forceinline__ float kda_gate(float g_min, float eA, float z) {
    return g_min / (1.0f + expf(-eA * z));
}

// Clock-cycle budget of the waits on flags that other blocks raise and of the
// decode's waits on its own copies (kda_set_wait_budget; about one second by
// default).
long long wait_budget();

// Argument checks of kda_chunk_fwd, shared by its variants (kda_host.cu).
int check_prefill(const void *q, const void *k, const void *v, const float *z, const float *A,
                  const float *beta, const int32_t *cu, int n_seqs, int64_t T_total, int H, int Dm,
                  int dtype, float g_min, const void *o, int flags);

// Sets a kernel's dynamic shared-memory limit to smem_bytes and returns (in
// *blocks_per_sm, when non-null) how many blocks of `threads` threads fit on an
// SM; the driver is asked once per (kernel, size, device) and the answer is
// cached, so repeated calls cost no driver round trips (kda_host.cu).
int prepare_kernel(const void *func, int smem_bytes, int threads, int *blocks_per_sm);

// Per-launch bookkeeping (kda_host.cu): counts every launch and, when
// profiling is enabled, records an event after it on stream `s`.
void note_launch(const char *name, cudaStream_t s);
void note_begin(cudaStream_t s);

// Launch helpers implemented in the kernel translation units.
int launch_plan(const int32_t *cu, int n_seqs, int64_t T_total, void *ws, const Workspace &w,
                cudaStream_t s);
int launch_empty_docs(const Plan &p, int H, const float *init_state, float *final_state,
                      cudaStream_t s);
int launch_prep_simt(const void *q, const void *k, const void *v, const float *z, const float *A,
                     const float *beta, int H, int dtype, float g_min, const Plan &p, void *records,
                     cudaStream_t s);

// Scan work description shared by the scan kernels.
struct ScanArgs {
    Plan plan;
    int H;
    const void *records;       // per-(chunk, head) records
    int mode;                  // SCAN_DOCS or SCAN_SEGMENTS
    int n_units;               // documents or segments
    int n_seg;                 // segments (SCAN_SEGMENTS)
    int ncols;                 // total state columns: 128 (values) or 256 (values | M)
    int phase;                 // 1: pairs from zero / identity, 3: emit from s_enter
    const float *init_state;   // [n_seqs, H, D, D] or null
    const float *s_enter;      // [H, n_seg, D, D] (phase 3)
    float *pairs;              // [2][H][n_seg][D][D] (phase 1)
    void *o;                   // [T, H, D] dtype (null: no output)
    float *final_state;        // [n_seqs, H, D, D] or null
    // state checkpoints (null ckpt: none): the state after every ckpt_ic chunks
    // of a document goes to ckpt[slot], slot = ckpt_slot[doc * ckpt_per_seq + j]
    float *ckpt;               // [n_slots, H, D, D]
    const int32_t *ckpt_slot;  // [n_seqs, ckpt_per_seq], -1 = skip
    int ckpt_per_seq;
    int ckpt_n_slots;          // slots outside 0 .. n_slots - 1 are skipped
    int ckpt_ic;               // checkpoint interval in chunks
};

// Index j of the checkpoint chunk c completes (the state after (j + 1) x
// interval tokens of its document), or -1.  Only a full chunk ends on an
// interval boundary: chunks are cut from each document's start.
__device__ __forceinline__ int ckpt_index(const Plan &p, int c, const ChunkInfo &ci, int ic) {
    if (ci.len != C) return -1;
    const int first = p.uniform ? ci.doc * p.chunks_per_seq : p.doc_off[ci.doc];
    const int k = c - first + 1;  // chunks of the document up to and including c
    return k % ic == 0 ? k / ic - 1 : -1;
}
__device__ __forceinline__ float *ckpt_row(const ScanArgs &a, const ChunkInfo &ci, int c, int h, int row) {
    const int j = ckpt_index(a.plan, c, ci, a.ckpt_ic);
    if (j < 0 || j >= a.ckpt_per_seq) return nullptr;
    const int slot = a.ckpt_slot[(size_t)ci.doc * a.ckpt_per_seq + j];
    return (slot < 0 || slot >= a.ckpt_n_slots) ? nullptr : a.ckpt + (((size_t)slot * a.H + h) * D + row) * D;
}
constexpr int SCAN_DOCS = 0;
constexpr int SCAN_SEGMENTS = 1;

// Tensor maps of the bf16 prep's input tiles (kda_tma.cu): q, k, v, z as 3-D
// tensors {D, H, T}, box {D, 1, C} (one head over one 64-token chunk).
struct InputMaps {
    CUtensorMap q, k, v, z;
};
int make_input_maps(const void *q, const void *k, const void *v, const float *z, int64_t T, int H, InputMaps *out);

int launch_prep_tc(const void *q, const void *k, const void *v, const float *z, const float *A,
                   const float *beta, int64_t T_total, int H, float g_min, const Plan &p, void *records, int n_sm,
                   cudaStream_t s);
int launch_scan_simt(const ScanArgs &a, int dtype, cudaStream_t s);
int launch_scan_tc(const ScanArgs &a, int n_sm, cudaStream_t s);
int launch_out_tc(const Plan &p, int H, const void *records, void *o, int n_sm, cudaStream_t s);
// `ready` holds plan max_chunks x H flags that the caller has zeroed on stream s.
int launch_fused_tc(const void *q, const void *k, const void *v, const float *z, const float *A,
                    const float *beta, int64_t T_total, int H, float g_min, const ScanArgs &sa, int *ready, int n_sm,
                    cudaStream_t s, bool *used);
int device_sm_count();
int launch_compose(const Plan &p, int H, int n_seg, const float *pairs, float *s_enter,
                   cudaStream_t s);
// Extra operands of the fused decode step.
struct DecFuse {
    const float *conv_w;      // [3][H][D][4]: q, k, v taps, tap 3 on the current token
    float *conv_state;        // [N][H][3][3][D]: q, k, v x the last three inputs, oldest first
    const float *o_gate;      // [N][W][H][D] output-gate logits
    const float *o_norm_w;    // [D]
    float o_norm_eps;
};
// fz == nullptr runs the plain decode step.
int launch_decode(float *state, const void *q, const void *k, const void *v, const float *z,
                  const float *beta, const float *A, void *cq, void *ck, void *cv, float *cz,
                  float *cb, const int32_t *nacc, int N, int H, int W, int dtype, float g_min,
                  void *o, int32_t *err, int flags, const DecFuse *fz, cudaStream_t s);

}  // namespace kda
