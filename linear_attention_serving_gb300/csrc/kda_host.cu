// kda_host.cu -- the C ABI (include/kda.h): argument checks, workspace layout,
// chunk planning and the launch sequence of every entry point.
#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "kda_internal.cuh"

using namespace kda;

// ---------------------------------------------------------------- diagnostics
namespace {
constexpr int PROF_MAX = 256;
bool g_prof = false;
bool g_prof_ready = false;
cudaEvent_t g_ev[PROF_MAX];
const char *g_name[PROF_MAX];
int g_nmarks = 0;
unsigned long long g_launches = 0;

void prof_mark(const char *name, cudaStream_t s) {
    if (!g_prof || !g_prof_ready || g_nmarks >= PROF_MAX) return;
    if (cudaEventRecord(g_ev[g_nmarks], s) == cudaSuccess) g_name[g_nmarks++] = name;
}
}  // namespace

namespace kda {
// SM count of the current device, queried once per device.
int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {
constexpr long long DEFAULT_WAIT_BUDGET = 2000000000ll;  // about one second at GB300 clocks
long long g_wait_budget = DEFAULT_WAIT_BUDGET;
}  // namespace
long long wait_budget() { return __atomic_load_n(&g_wait_budget, __ATOMIC_RELAXED); }

namespace {
struct KernelSetup {
    const void *func;
    int smem, threads, dev, per_sm;
};
constexpr int SETUP_MAX = 128;
KernelSetup g_setup[SETUP_MAX];
int g_nsetup = 0;
std::mutex g_setup_mu;
}  // namespace

int prepare_kernel(const void *func, int smem_bytes, int threads, int *blocks_per_sm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    for (int i = 0; i < g_nsetup; ++i) {
        const KernelSetup &k = g_setup[i];
        if (k.func == func && k.smem == smem_bytes && k.threads == threads && k.dev == dev) {
            if (blocks_per_sm) *blocks_per_sm = k.per_sm;
            return KDA_OK;
        }
    }
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
        return KDA_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, threads, (size_t)smem_bytes) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (g_nsetup < SETUP_MAX) g_setup[g_nsetup++] = KernelSetup{func, smem_bytes, threads, dev, per_sm};
    if (blocks_per_sm) *blocks_per_sm = per_sm;
    return KDA_OK;
}

void note_launch(const char *name, cudaStream_t s) {
    __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);
    prof_mark(name, s);
}
void note_begin(cudaStream_t s) { prof_mark("begin", s); }
}  // namespace kda

namespace {

bool aligned16(const void *p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

}  // namespace

// Validation shared by kda_chunk_fwd, its variants and kda_segment_scan.
int kda::check_prefill(const void *q, const void *k, const void *v, const float *z, const float *A,
                  const float *beta, const int32_t *cu, int n_seqs, int64_t T_total, int H, int Dm,
                  int dtype, float g_min, const void *o, int flags) {
    if (Dm != D) return KDA_ERR_UNSUPPORTED;
    if (flags & ~PREFILL_FLAGS) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (H < 1 || n_seqs < 1 || T_total < 0 || T_total >= (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
    if (!(g_min >= -5.0f && g_min < 0.0f)) return KDA_ERR_INVALID_ARG;
    if (T_total > 0 && (!q || !k || !v || !z || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!A) return KDA_ERR_INVALID_ARG;
    if (!cu && (T_total % n_seqs) != 0) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(z) || !aligned16(o))
        return KDA_ERR_INVALID_ARG;
    // the largest element offset of a [T, H, 128] tensor must fit the kernels' 64-bit math;
    // the chunk count must fit an int
    if ((int64_t)(T_total / C + n_seqs) >= (int64_t)INT32_MAX / 2) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

namespace {

// Prep launch by input type: tcgen05 tensor cores for bf16 inputs, exact fp32
// CUDA cores for fp32 inputs.
int launch_prep(const void *q, const void *k, const void *v, const float *z, const float *A,
                const float *beta, int64_t T_total, int H, int dtype, float g_min, const Plan &p, void *records,
                cudaStream_t s) {
    if (dtype == KDA_BF16)
        return launch_prep_tc(q, k, v, z, A, beta, T_total, H, g_min, p, records, device_sm_count(), s);
    return launch_prep_simt(q, k, v, z, A, beta, H, dtype, g_min, p, records, s);
}

// Scan launch by input type: tcgen05 tensor cores for bf16 operands, exact
// fp32 CUDA cores for fp32 inputs.
int launch_scan(const ScanArgs &a, int dtype, cudaStream_t s) {
    if (dtype == KDA_BF16) return launch_scan_tc(a, device_sm_count(), s);
    return launch_scan_simt(a, dtype, s);
}

// Chunk plan: arithmetic for equal-length documents, a device table otherwise.
// Clears the workspace's first `zero_bytes` (at least the 8-byte header: error
// word and chunk count) and fills in the chunk plan.
int make_plan(const int32_t *cu, int n_seqs, int64_t T_total, void *ws, const Workspace &w,
              cudaStream_t s, Plan &p, int flags, size_t zero_bytes = 8) {
    memset(&p, 0, sizeof(p));
    p.flags = flags;
    char *base = (char *)ws;
    p.n_seqs = n_seqs;
    p.err = (int32_t *)base;
    p.table = (const ChunkInfo *)(base + w.off_table);
    p.doc_off = (const int32_t *)(base + w.off_doc);
    p.n_chunks = (const int32_t *)(base + 4);
    p.wait_budget = wait_budget();
    int rc = cuda_status(cudaMemsetAsync(base, 0, zero_bytes, s));
    if (rc) return rc;
    if (!cu) {
        p.uniform = 1;
        p.seq_len = (int)(T_total / n_seqs);
        p.chunks_per_seq = (p.seq_len + C - 1) / C;
        p.max_chunks = n_seqs * p.chunks_per_seq;
        return KDA_OK;
    }
    p.uniform = 0;
    p.max_chunks = w.max_chunks;
    return launch_plan(cu, n_seqs, T_total, ws, w, s);
}

// Automatic segment count for kda_chunk_fwd ("Kimi K3 模型结构（7）", section
// "KDA：三种执行形态" (SM-level CP): with few (document, head) chains over a
// long document the sequential chain, not the parallel preparation, sets the
// time; cutting the chunk list into segments that run side by side and are
// then composed shortens it).  bf16 only.  Equal-length batches plan from
// their length; packed batches from their longest document.  The model,
// measured on GB300 (kda_planner_model returns it; a GPU test checks it
// against the kernels):
//   one chain        about 1.3 us per chunk (64 state columns per block);
//   preparation      about 8.6 us per (chunk, head) unit on one SM, on the SMs
//                    the chains leave free (all SMs without the fused launch);
//   segments         pay a second pass over the chain and the composition
//                    (about 25 us per segment), so they win only when the
//                    chain is over 1.5x the preparation; their count is set
//                    by the scan's waves (below).
// Segment count, measured on GB300: the scan blocks run one per SM, so whole
// waves decide the time.  Take the most segments whose phase 3 (two 64-column
// blocks per (segment, head)) fits in one wave of the SMs, and phase 1 (four
// per pair) in two; more segments or an extra partial wave cost more than the
// shorter chains save.  At most sqrt(chunks / 6), where the composition (about
// 25 us per segment) outweighs the shorter chains (about 4 us per chunk over
// the three phases); at most 64 and half the chunks; at least 1.
int wave_segments(int64_t total_chunks, int H, int n_sm) {
    int64_t n = n_sm / (2LL * H);
    const int64_t cap = llround(sqrt((double)total_chunks / 6.0));
    if (n > cap) n = cap;
    if (n > 64) n = 64;
    if (n > total_chunks / 2) n = total_chunks / 2;
    return n >= 1 ? (int)n : 1;
}

constexpr double PLAN_PREP_US_PER_UNIT = 8.6;
constexpr double PLAN_CHAIN_US_PER_CHUNK = 1.3;

// Segment count for a batch of n_seqs documents with `total` chunks in all,
// the longest `longest` chunks; 0 for one chain per (document, head).
int plan_from_chunks(int64_t longest, int64_t total, int H, int n_seqs, int dtype, int n_sm) {
    if (dtype != KDA_BF16 || longest <= 0 || total <= 0 || n_seqs < 1 || H < 1) return 0;
    const double units = (double)total * H;
    const int64_t chains = 2LL * n_seqs * H;
    const int prep_sms = chains <= n_sm / 4 ? n_sm - (int)chains : n_sm;
    const double prep_us = PLAN_PREP_US_PER_UNIT * units / (double)(prep_sms > 0 ? prep_sms : 1);
    const double chain_us = PLAN_CHAIN_US_PER_CHUNK * (double)longest;
    if (chain_us <= 1.5 * prep_us) return 0;
    const int n = wave_segments(total, H, n_sm);
    return n >= 2 ? n : 0;
}

// Equal-length batches (varlen = false) plan from their length.  Packed
// batches (varlen) get the count for the longest document they can hold (one
// of T_total tokens): an upper bound, since a call plans again from its actual
// longest document.
int plan_segments(int64_t T_total, int H, int n_seqs, bool varlen, int dtype, int n_sm) {
    if (T_total <= 0 || n_seqs < 1 || H < 1) return 0;
    if (varlen) {
        const int64_t longest = (T_total + C - 1) / C;
        return plan_from_chunks(longest, T_total / C + n_seqs, H, n_seqs, dtype, n_sm);
    }
    const int64_t chunks = (T_total / n_seqs + C - 1) / C;  // per document
    return plan_from_chunks(chunks, chunks * n_seqs, H, n_seqs, dtype, n_sm);
}

// A packed call's own count: its longest document, read from cu_seqlens (the
// call waits for the stream once).  Only asked when the bound above says
// segments could pay, never while the stream is being captured into a graph.
int plan_packed(const int32_t *cu_seqlens, int64_t T_total, int H, int n_seqs, int dtype, int n_sm,
                cudaStream_t s) {
    if (plan_segments(T_total, H, n_seqs, true, dtype, n_sm) == 0) return 0;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return 0;
    std::vector<int32_t> cu((size_t)n_seqs + 1);
    if (cudaMemcpyAsync(cu.data(), cu_seqlens, cu.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return 0;
    int64_t longest = 0, total = 0;
    for (int n = 0; n < n_seqs; ++n) {
        const int64_t len = (int64_t)cu[n + 1] - cu[n];
        if (len < 0) return 0;  // the plan kernel reports the bad offsets
        const int64_t ch = (len + C - 1) / C;
        longest = ch > longest ? ch : longest;
        total += ch;
    }
    return plan_from_chunks(longest, total, H, n_seqs, dtype, n_sm);
}

// kda_segment_scan's n_segments, with 0 meaning the wave rule's count.
int resolve_segments(int n_segments, int64_t T_total, int H, int n_seqs) {
    if (n_segments != 0) return n_segments;
    if (T_total < 0 || H < 1 || n_seqs < 1) return 0;
    return wave_segments(T_total / C + n_seqs, H, device_sm_count());
}

// The three phases of the segment scan over a workspace laid out for n_segments.
int run_segment_scan(const void *q, const void *k, const void *v, const float *z, const float *A,
                     const float *beta, const int32_t *cu_seqlens, int n_seqs, int64_t T_total, int H,
                     int dtype, float g_min, const float *init_state, int n_segments, float *pairs_M,
                     float *pairs_S, void *o, float *final_state, void *workspace, const Workspace &w,
                     int flags, cudaStream_t s, const ScanArgs *ckpt = nullptr) {
    int rc;
    Plan p;
    if ((rc = make_plan(cu_seqlens, n_seqs, T_total, workspace, w, s, p, flags))) return rc;
    char *base = (char *)workspace;
    void *records = base + w.off_rec;
    float *pairs = (float *)(base + w.off_pairs);
    float *s_enter = (float *)(base + w.off_enter);
    if ((rc = launch_prep(q, k, v, z, A, beta, T_total, H, dtype, g_min, p, records, s))) return rc;

    ScanArgs a;
    memset(&a, 0, sizeof(a));
    a.plan = p;
    a.H = H;
    a.records = records;
    a.mode = SCAN_SEGMENTS;
    a.n_units = n_segments;
    a.n_seg = n_segments;
    a.init_state = init_state;
    a.s_enter = s_enter;
    a.pairs = pairs;
    // phase 1: pairs (M, S~) of every (head, segment) from zero / identity
    a.ncols = 2 * D;
    a.phase = 1;
    if ((rc = launch_scan(a, dtype, s))) return rc;
    // phase 2: entering states by sequential composition
    if ((rc = launch_compose(p, H, n_segments, pairs, s_enter, s))) return rc;
    // phase 3: every segment from its exact entering state
    a.ncols = D;
    a.phase = 3;
    a.o = o;
    a.final_state = final_state;
    if (ckpt) {
        a.ckpt = ckpt->ckpt;
        a.ckpt_slot = ckpt->ckpt_slot;
        a.ckpt_per_seq = ckpt->ckpt_per_seq;
        a.ckpt_n_slots = ckpt->ckpt_n_slots;
        a.ckpt_ic = ckpt->ckpt_ic;
    }
    if ((rc = launch_scan(a, dtype, s))) return rc;
    if ((rc = launch_empty_docs(p, H, init_state, final_state, s))) return rc;
    const size_t mat = sizeof(float) * (size_t)H * n_segments * D * D;
    if (pairs_M && (rc = cuda_status(cudaMemcpyAsync(pairs_M, pairs, mat, cudaMemcpyDeviceToDevice, s))))
        return rc;
    if (pairs_S &&
        (rc = cuda_status(cudaMemcpyAsync(pairs_S, (char *)pairs + mat, mat, cudaMemcpyDeviceToDevice, s))))
        return rc;
    return KDA_OK;
}

}  // namespace

extern "C" {

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_DEVICE_CHECK: return "KDA_ERR_DEVICE_CHECK";
        default: return "KDA_ERR_UNKNOWN";
    }
}

int kda_version(void) { return 100; }

int kda_profile_enable(int on) {
    if (on && !g_prof_ready) {
        for (int i = 0; i < PROF_MAX; ++i)
            if (cudaEventCreate(&g_ev[i]) != cudaSuccess) return KDA_ERR_CUDA;
        g_prof_ready = true;
    }
    g_prof = on != 0;
    g_nmarks = 0;
    return KDA_OK;
}

int kda_profile_collect(const char **names, float *ms, int max) {
    if (!g_prof_ready || g_nmarks == 0) {
        g_nmarks = 0;
        return 0;
    }
    if (cudaEventSynchronize(g_ev[g_nmarks - 1]) != cudaSuccess) return -KDA_ERR_CUDA;
    int n = 0;
    for (int i = 1; i < g_nmarks && n < max; ++i) {
        if (strcmp(g_name[i], "begin") == 0) continue;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, g_ev[i - 1], g_ev[i]) != cudaSuccess) return -KDA_ERR_CUDA;
        if (names) names[n] = g_name[i];
        if (ms) ms[n] = t;
        ++n;
    }
    g_nmarks = 0;
    return n;
}

long long kda_launch_count(void) { return (long long)__atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

long long kda_set_wait_budget(long long cycles) {
    const long long v = cycles > 0 ? cycles : DEFAULT_WAIT_BUDGET;
    return __atomic_exchange_n(&g_wait_budget, v, __ATOMIC_RELAXED);
}

size_t kda_chunk_fwd_workspace_size(int64_t T_total, int H, int n_seqs, int dtype) {
    if (T_total < 0 || H < 1 || n_seqs < 1) return 0;
    // room for the segmented path whenever a batch of this shape can take it:
    // equal lengths, or packed with a long document
    const int n_sm = device_sm_count();
    const int a = plan_segments(T_total, H, n_seqs, false, dtype, n_sm);
    const int b = plan_segments(T_total, H, n_seqs, true, dtype, n_sm);
    const size_t wa = workspace_layout(T_total, H, n_seqs, a, dtype).total;
    const size_t wb = workspace_layout(T_total, H, n_seqs, b, dtype).total;
    return wa > wb ? wa : wb;
}

int kda_chunk_fwd_plan_segments(int64_t T_total, int H, int n_seqs, int dtype, int varlen) {
    if (T_total < 0 || H < 1 || n_seqs < 1) return 0;
    return plan_segments(T_total, H, n_seqs, varlen != 0, dtype, device_sm_count());
}

void kda_planner_model(double *prep_us_per_unit, double *chain_us_per_chunk) {
    if (prep_us_per_unit) *prep_us_per_unit = PLAN_PREP_US_PER_UNIT;
    if (chain_us_per_chunk) *chain_us_per_chunk = PLAN_CHAIN_US_PER_CHUNK;
}

size_t kda_segment_scan_workspace_size(int64_t T_total, int H, int n_seqs, int n_segments,
                                       int dtype) {
    n_segments = resolve_segments(n_segments, T_total, H, n_seqs);
    if (T_total < 0 || H < 1 || n_seqs < 1 || n_segments < 1) return 0;
    return workspace_layout(T_total, H, n_seqs, n_segments, dtype).total;
}

int kda_segment_scan_auto_segments(int64_t T_total, int H, int n_seqs) {
    return resolve_segments(0, T_total, H, n_seqs);
}

}  // extern "C"

namespace {

// kda_chunk_fwd with an optional checkpoint description (ckpt fields of a ScanArgs).
int chunk_fwd_impl(const void *q, const void *k, const void *v, const float *z, const float *A,
                   const float *beta, const int32_t *cu_seqlens, int n_seqs, int64_t T_total, int H,
                   int Dm, int dtype, float g_min, const float *init_state, void *o,
                   float *final_state, void *workspace, size_t workspace_bytes, int flags,
                   kda_stream_t stream, const ScanArgs *ckpt) {
    int rc = check_prefill(q, k, v, z, A, beta, cu_seqlens, n_seqs, T_total, H, Dm, dtype, g_min, o, flags);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    int n_seg = cu_seqlens ? plan_packed(cu_seqlens, T_total, H, n_seqs, dtype, device_sm_count(), s)
                           : plan_segments(T_total, H, n_seqs, false, dtype, device_sm_count());
    // a workspace sized for the single-chain path keeps that path (same results)
    if (n_seg > 0 && workspace_bytes < workspace_layout(T_total, H, n_seqs, n_seg, dtype).total) n_seg = 0;
    const Workspace w = workspace_layout(T_total, H, n_seqs, n_seg, dtype);
    if (!workspace || workspace_bytes < w.total || ((uintptr_t)workspace & 255u)) return KDA_ERR_WORKSPACE;
    note_begin(s);
    if (n_seg > 0)
        return run_segment_scan(q, k, v, z, A, beta, cu_seqlens, n_seqs, T_total, H, dtype, g_min, init_state,
                                n_seg, nullptr, nullptr, o, final_state, workspace, w, flags, s, ckpt);
    Plan p;
    // bf16: the header and the fused launch's ready flags, in one memset
    const size_t zero = dtype == KDA_BF16 ? w.off_ready + sizeof(int) * (size_t)w.max_chunks * H : 8;
    if ((rc = make_plan(cu_seqlens, n_seqs, T_total, workspace, w, s, p, flags, zero))) return rc;
    void *records = (char *)workspace + w.off_rec;
    ScanArgs a;
    memset(&a, 0, sizeof(a));
    a.plan = p;
    a.H = H;
    a.records = records;
    a.mode = SCAN_DOCS;
    a.n_units = n_seqs;
    a.ncols = D;
    a.phase = 0;
    a.init_state = init_state;
    a.o = o;
    a.final_state = final_state;
    if (ckpt) {
        a.ckpt = ckpt->ckpt;
        a.ckpt_slot = ckpt->ckpt_slot;
        a.ckpt_per_seq = ckpt->ckpt_per_seq;
        a.ckpt_n_slots = ckpt->ckpt_n_slots;
        a.ckpt_ic = ckpt->ckpt_ic;
    }
    if (dtype == KDA_BF16) {
        // few (document, head) chains: prep, chains and outputs in one launch
        bool used = false;
        if ((rc = launch_fused_tc(q, k, v, z, A, beta, T_total, H, g_min, a,
                                  (int *)((char *)workspace + w.off_ready), device_sm_count(), s, &used)))
            return rc;
        if (used) return KDA_OK;
    }
    if ((rc = launch_prep(q, k, v, z, A, beta, T_total, H, dtype, g_min, p, records, s))) return rc;
    return launch_scan(a, dtype, s);
}

}  // namespace

extern "C" {

int kda_chunk_fwd(const void *q, const void *k, const void *v, const float *z, const float *A,
                  const float *beta, const int32_t *cu_seqlens, int n_seqs, int64_t T_total, int H,
                  int Dm, int dtype, float g_min, const float *init_state, void *o,
                  float *final_state, void *workspace, size_t workspace_bytes, int flags,
                  kda_stream_t stream) {
    return chunk_fwd_impl(q, k, v, z, A, beta, cu_seqlens, n_seqs, T_total, H, Dm, dtype, g_min, init_state, o,
                          final_state, workspace, workspace_bytes, flags, stream, nullptr);
}

int kda_chunk_fwd_ckpt(const void *q, const void *k, const void *v, const float *z, const float *A,
                       const float *beta, const int32_t *cu_seqlens, int n_seqs, int64_t T_total, int H,
                       int Dm, int dtype, float g_min, const float *init_state, void *o,
                       float *final_state, int ckpt_interval, const int32_t *ckpt_slot, int ckpt_per_seq,
                       float *ckpt, int n_slots, void *workspace, size_t workspace_bytes, int flags,
                       kda_stream_t stream) {
    if (ckpt_interval < C || ckpt_interval % C != 0 || ckpt_per_seq < 1 || n_slots < 1 || !ckpt_slot || !ckpt ||
        !aligned16(ckpt))
        return KDA_ERR_INVALID_ARG;
    ScanArgs c;
    memset(&c, 0, sizeof(c));
    c.ckpt = ckpt;
    c.ckpt_slot = ckpt_slot;
    c.ckpt_per_seq = ckpt_per_seq;
    c.ckpt_n_slots = n_slots;
    c.ckpt_ic = ckpt_interval / C;
    return chunk_fwd_impl(q, k, v, z, A, beta, cu_seqlens, n_seqs, T_total, H, Dm, dtype, g_min, init_state, o,
                          final_state, workspace, workspace_bytes, flags, stream, &c);
}

int kda_segment_scan(const void *q, const void *k, const void *v, const float *z, const float *A,
                     const float *beta, const int32_t *cu_seqlens, int n_seqs, int64_t T_total,
                     int H, int Dm, int dtype, float g_min, const float *init_state, int n_segments,
                     float *pairs_M, float *pairs_S, void *o, float *final_state, void *workspace,
                     size_t workspace_bytes, int flags, kda_stream_t stream) {
    int rc = check_prefill(q, k, v, z, A, beta, cu_seqlens, n_seqs, T_total, H, Dm, dtype, g_min, o, flags);
    if (rc) return rc;
    n_segments = resolve_segments(n_segments, T_total, H, n_seqs);
    if (n_segments < 1 || n_segments > (1 << 20)) return KDA_ERR_INVALID_ARG;
    const Workspace w = workspace_layout(T_total, H, n_seqs, n_segments, dtype);
    if (!workspace || workspace_bytes < w.total || ((uintptr_t)workspace & 255u)) return KDA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    note_begin(s);
    return run_segment_scan(q, k, v, z, A, beta, cu_seqlens, n_seqs, T_total, H, dtype, g_min, init_state,
                            n_segments, pairs_M, pairs_S, o, final_state, workspace, w, flags, s);
}

int kda_decode_step(float *state, const void *q, const void *k, const void *v, const float *z,
                    const float *beta, const float *A, void *cache_q, void *cache_k, void *cache_v,
                    float *cache_z, float *cache_beta, const int32_t *num_accepted, int N, int H,
                    int Dm, int W, int dtype, float g_min, void *o, int32_t *error_word, int flags,
                    kda_stream_t stream) {
    if (Dm != D) return KDA_ERR_UNSUPPORTED;
    if (flags & ~PREFILL_FLAGS) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (N < 1 || H < 1 || W < 1 || W > 8) return KDA_ERR_INVALID_ARG;
    if ((int64_t)N * H >= (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
    if (!(g_min >= -5.0f && g_min < 0.0f)) return KDA_ERR_INVALID_ARG;
    if (!state || !q || !k || !v || !z || !beta || !A || !o) return KDA_ERR_INVALID_ARG;
    if (W > 1 && (!cache_q || !cache_k || !cache_v || !cache_z || !cache_beta)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(z) ||
        !aligned16(o) || !aligned16(cache_q) || !aligned16(cache_k) || !aligned16(cache_v) ||
        !aligned16(cache_z))
        return KDA_ERR_INVALID_ARG;
    note_begin((cudaStream_t)stream);
    return launch_decode(state, q, k, v, z, beta, A, cache_q, cache_k, cache_v, cache_z, cache_beta,
                         num_accepted, N, H, W, dtype, g_min, o, error_word, flags, nullptr,
                         (cudaStream_t)stream);
}

int kda_decode_step_fused(float *state, const void *q, const void *k, const void *v, const float *z,
                          const float *beta, const float *A, const float *conv_w, float *conv_state,
                          const float *o_gate, const float *o_norm_w, float o_norm_eps, void *cache_q,
                          void *cache_k, void *cache_v, float *cache_z, float *cache_beta,
                          const int32_t *num_accepted, int N, int H, int Dm, int W, int dtype, float g_min,
                          void *o, int32_t *error_word, int flags, kda_stream_t stream) {
    if (Dm != D) return KDA_ERR_UNSUPPORTED;
    if (flags & ~(PREFILL_FLAGS | KDA_FLAG_CONV_SILU)) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
    if (N < 1 || H < 1 || W < 1 || W > 8) return KDA_ERR_INVALID_ARG;
    if ((int64_t)N * H >= (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
    if (!(g_min >= -5.0f && g_min < 0.0f)) return KDA_ERR_INVALID_ARG;
    if (!(o_norm_eps >= 0.0f) || o_norm_eps > 1e30f) return KDA_ERR_INVALID_ARG;
    if (!state || !q || !k || !v || !z || !beta || !A || !o) return KDA_ERR_INVALID_ARG;
    if (!conv_w || !conv_state || !o_gate || !o_norm_w) return KDA_ERR_INVALID_ARG;
    if (W > 1 && (!cache_q || !cache_k || !cache_v || !cache_z || !cache_beta)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(z) ||
        !aligned16(o) || !aligned16(cache_q) || !aligned16(cache_k) || !aligned16(cache_v) ||
        !aligned16(cache_z) || !aligned16(conv_w) || !aligned16(conv_state))
        return KDA_ERR_INVALID_ARG;
    note_begin((cudaStream_t)stream);
    const DecFuse fz{conv_w, conv_state, o_gate, o_norm_w, o_norm_eps};
    return launch_decode(state, q, k, v, z, beta, A, cache_q, cache_k, cache_v, cache_z, cache_beta,
                         num_accepted, N, H, W, dtype, g_min, o, error_word, flags, &fz,
                         (cudaStream_t)stream);
}

int kda_read_device_error(const void *workspace, int32_t *code, kda_stream_t stream) {
    if (!workspace || !code) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    *code = h;
    return KDA_OK;
}

}  // extern "C"
