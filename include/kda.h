/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library.
 *
 * The operation (K3 convention, state S in R^{d_k x d_v}):
 *   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *   o_t = S_t^T q_t,
 *   alpha_t = exp(g_t),  g_t = g_min * sigmoid(exp(A_h) * z_t)   (per channel)
 * ("Kimi K3 模型结构（7）：结构决定系统", section "KDA 上下文并行", eq. (1);
 *  "Kimi K3 模型结构（2）：序列维度（下），chunkwise 并行与下界衰减", section
 *  "K3 的改动：下界衰减", eq. (5); "Kimi K3: the Manos, the Mythos ..."
 *  (SemiAnalysis), section "FlashKDA 算法", delta form).
 * No query scaling is applied; beta is taken after its sigmoid and q, k are
 * taken already L2-normalised.
 *
 * Conventions shared by every entry point
 *   - Pointers marked (device) are device memory owned by the caller; the
 *     library never allocates or frees them and keeps no reference after the
 *     call returns.  Pointers marked (host) are read during the call only.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Results are ready when the stream reaches that point.
 *   - d_k = d_v = D must be 128 (KDA_ERR_UNSUPPORTED otherwise).
 *   - Layouts are row-major, innermost dimension last, no padding:
 *       q, k, z : [T_total, H, D]      v, o : [T_total, H, D]
 *       beta    : [T_total, H]         A    : [H]
 *       states  : [n_seqs, H, D(d_k), D(d_v)]  (fp32)
 *   - dtype selects the element type of q, k, v and o: KDA_BF16 or KDA_F32.
 *     z, A, beta and all states are always fp32.
 *   - Return value: KDA_OK or one of the KDA_ERR_* codes below.  Argument
 *     errors are detected on the host before anything is launched.  Checks
 *     that need device data (cu_seqlens, num_accepted) record a device error
 *     code that kda_read_device_error() / the decode error word returns.
 *   - Every device-side wait in the library is bounded; a wait that gives up
 *     records KDA_DEVERR_TIMEOUT instead of hanging.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same ABI as cudaStream_t. */
typedef struct CUstream_st *kda_stream_t;

enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer   */
    KDA_ERR_UNSUPPORTED = 2,   /* D != 128, or a mode the library does not implement */
    KDA_ERR_CUDA = 3,          /* a CUDA runtime/driver call or launch failed   */
    KDA_ERR_TIMEOUT = 4,       /* a bounded device wait gave up                 */
    KDA_ERR_WORKSPACE = 5,     /* workspace missing or smaller than required    */
    KDA_ERR_DEVICE_CHECK = 6   /* device-side validation failed (see code)      */
};

enum kda_dtype { KDA_BF16 = 0, KDA_F32 = 1 };

/* Input options (bit flags), the kernel-side options of the pages' chunk_kda /
 * fused_recurrent_kda ("Kimi K3 模型结构（2）", section "训练、prefill、decode
 * 各用哪种形式": use_qk_l2norm_in_kernel, use_beta_sigmoid_in_kernel):
 *   KDA_FLAG_QK_L2NORM     q and k are divided by their L2 norm over the 128 key
 *                          channels, x / sqrt(sum(x^2) + 1e-6), per (token, head)
 *   KDA_FLAG_BETA_SIGMOID  beta holds logits; the kernels use 1 / (1 + exp(-beta))
 *   KDA_FLAG_CONV_SILU     kda_decode_step_fused only: SiLU, y / (1 + exp(-y)), after
 *                          the short convolution (the pages name no activation)
 *   KDA_FLAG_Q_SCALE       q is multiplied by d_k^-1/2 = 1 / sqrt(128) (after the L2
 *                          norm when both are set), the usual attention scale of the
 *                          chunk_kda interface; the pages give no scale, so it is off
 *                          by default (o = S^T q)
 * The decode cache keeps the projected inputs as given (unnormalised, logits). */
enum kda_flags {
    KDA_FLAG_QK_L2NORM = 1,
    KDA_FLAG_BETA_SIGMOID = 2,
    KDA_FLAG_CONV_SILU = 4,
    KDA_FLAG_Q_SCALE = 8
};

/* Device error codes (bit flags) written into the workspace / error word. */
enum kda_device_error {
    KDA_DEVERR_NONE = 0,
    KDA_DEVERR_CU_SEQLENS = 1,     /* cu_seqlens not 0 .. T_total, non-decreasing */
    KDA_DEVERR_NUM_ACCEPTED = 2,   /* num_accepted[b] outside 0 .. W-1            */
    KDA_DEVERR_TIMEOUT = 4         /* a bounded wait gave up                       */
};

/* Human-readable name of a kda_status. Never NULL. */
const char *kda_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int kda_version(void);

/* --------------------------------------------------------------------------
 * kda_chunk_fwd -- chunkwise prefill (chunk C = 64, 16-token sub-tiles).
 *
 * Defined by "Kimi K3 模型结构（2）", sections "UT 变换" and "块间递推与块内
 * 输出" (eqs. (4), (8)), computed in the matrix form of "Kimi K3: the Manos,
 * the Mythos ..." section "FlashKDA 算法":
 *   per chunk: U = (I+L)^{-1} Diag(beta) (V - K_decay S),
 *              O = Q_decay S + M_qk U,  S <- Diag(a_C) S + K_restore^T U,
 * with the 16-token sub-tile factorisation of "数值问题：1/Γ 会溢出" that the
 * bounded gate makes safe in bf16.  Packed documents restart the state at
 * every start given by cu_seqlens ("Kimi K3 模型结构（7）", section "文档边界").
 *
 *   q, k, v      (device) [T_total, H, D]  dtype
 *   z            (device) [T_total, H, D]  fp32 gate logits
 *   A            (device) [H]              fp32 per-head log scale A_h
 *   beta         (device) [T_total, H]     fp32, after sigmoid (logits with
 *                KDA_FLAG_BETA_SIGMOID)
 *   cu_seqlens   (device) int32 [n_seqs+1]: document offsets, cu[0] = 0,
 *                non-decreasing, cu[n_seqs] = T_total (empty documents allowed).
 *                NULL: n_seqs equal-length sequences (T_total % n_seqs == 0).
 *                Validated on the device: a bad array records
 *                KDA_DEVERR_CU_SEQLENS in the workspace and leaves o / final
 *                state unwritten.
 *   n_seqs       number of documents (>= 1)
 *   T_total      total tokens (>= 0, < 2^31)
 *   H            heads (>= 1);  D: must be 128
 *   dtype        KDA_BF16 or KDA_F32
 *   g_min        gate lower bound (the pages fix -5); must be in [-5, 0)
 *   flags        0 or an OR of KDA_FLAG_* (others: KDA_ERR_INVALID_ARG)
 *   init_state   (device) fp32 [n_seqs, H, D, D] or NULL (zeros)
 *   o            (device) [T_total, H, D] dtype, written
 *   final_state  (device) fp32 [n_seqs, H, D, D] or NULL (not written)
 *   workspace    (device) scratch of at least kda_chunk_fwd_workspace_size()
 *                bytes, 256-byte aligned; contents need no initialisation and
 *                are overwritten; must not be shared by calls in flight.
 * Pointers q, k, v, z, o must be 16-byte aligned.
 * ------------------------------------------------------------------------ */
size_t kda_chunk_fwd_workspace_size(int64_t T_total, int H, int n_seqs, int dtype);

/* --------------------------------------------------------------------------
 * kda_chunk_fwd_ckpt -- kda_chunk_fwd that also writes the state at
 * interval-aligned positions of every document ("Kimi K3 模型结构（7）",
 * section "混合架构的前缀缓存": a cached prefix is usable only where the KDA
 * state was persisted, so after each forward the kernel saves the state at
 * the last hash-aligned position, into a fresh slot).
 * Same arguments, checks and results as kda_chunk_fwd, plus
 *   ckpt_interval  tokens between checkpoints: a positive multiple of 64 (C)
 *   ckpt_slot      (device) int32 [n_seqs, ckpt_per_seq]: ckpt_slot[n][j] is
 *                  the page that receives the state of document n after its
 *                  first (j + 1) * ckpt_interval tokens; -1 (or any value
 *                  outside 0 .. n_slots - 1) skips it.  Positions past a
 *                  document's end are never written, so a caller that wants
 *                  only the last aligned state of each document marks only
 *                  that entry.
 *   ckpt_per_seq   columns of ckpt_slot (>= 1)
 *   ckpt           (device) fp32 [n_slots, H, D, D], 16-byte aligned: pages
 *   n_slots        pages in ckpt (>= 1)
 * Invalid checkpoint arguments return KDA_ERR_INVALID_ARG before any launch.
 * A call with checkpoints runs the same path as kda_chunk_fwd (fused launch,
 * three kernels or segments), in instantiations that carry the checkpoint
 * stores.
 * ------------------------------------------------------------------------ */
int kda_chunk_fwd_ckpt(const void *q, const void *k, const void *v,
                       const float *z, const float *A, const float *beta,
                       const int32_t *cu_seqlens, int n_seqs,
                       int64_t T_total, int H, int D, int dtype, float g_min,
                       const float *init_state, void *o, float *final_state,
                       int ckpt_interval, const int32_t *ckpt_slot, int ckpt_per_seq,
                       float *ckpt, int n_slots,
                       void *workspace, size_t workspace_bytes, int flags, kda_stream_t stream);

/* --------------------------------------------------------------------------
 * kda_chunk_fwd_plan_segments -- the segment count kda_chunk_fwd picks by
 * itself ("Kimi K3 模型结构（7）", section "KDA：三种执行形态" (SM-level CP):
 * when a few (document, head) chains over long documents would leave the
 * chain, not the parallel preparation, setting the time, kda_chunk_fwd runs
 * the kda_segment_scan decomposition with this many segments instead; its
 * results equal the single-chain run up to rounding).
 *   varlen  nonzero when the call passes cu_seqlens: the count for the
 *           longest document such a batch can hold (one of T_total tokens).
 *           The call itself plans from its actual longest document: when
 *           this bound is nonzero it reads cu_seqlens back to the host (it
 *           waits once for the stream; not while the stream is captured into
 *           a graph, which keeps the single-chain path).
 * Returns 0 for the single-chain path, else the segment count (2 .. 64).  The
 * choice depends on the shape, the dtype (bf16 only) and the current device's
 * SM count; kda_chunk_fwd_workspace_size already includes the room it needs
 * (a call given less keeps the single-chain path, with the same results).
 * No device work; never fails (invalid shapes return 0).
 * ------------------------------------------------------------------------ */
int kda_chunk_fwd_plan_segments(int64_t T_total, int H, int n_seqs, int dtype, int varlen);

/* The timing model behind that choice, measured on GB300: microseconds per
 * (chunk, head) preparation unit on one SM, and per chunk of one chain.  A
 * chain over L chunks is split when 1.3 us x L exceeds 1.5 times the
 * preparation time of the batch on the SMs the chains leave free.  NULL
 * arguments are skipped. */
void kda_planner_model(double *prep_us_per_unit, double *chain_us_per_chunk);

int kda_chunk_fwd(const void *q, const void *k, const void *v,
                  const float *z, const float *A, const float *beta,
                  const int32_t *cu_seqlens, int n_seqs,
                  int64_t T_total, int H, int D, int dtype, float g_min,
                  const float *init_state, void *o, float *final_state,
                  void *workspace, size_t workspace_bytes, int flags, kda_stream_t stream);

/* --------------------------------------------------------------------------
 * kda_chunk_fwd_noalloc -- kda_chunk_fwd without a caller-provided workspace.
 * The pages have no counterpart: this is an interface for callers that cannot
 * allocate device memory at call time (an engine that reserved the whole
 * device for its own pool, or a latency-critical path that cannot afford the
 * device synchronisation a cudaMalloc may imply).
 *
 * Same arguments, checks and results as kda_chunk_fwd, without workspace and
 * workspace_bytes.  It always runs the preparation and scan kernels one after
 * the other (never the single fused launch or the automatic segments), so its
 * results equal kda_chunk_fwd's up to rounding.  The workspace is a fixed array
 * of KDA_NOALLOC_SCRATCH_BYTES bytes in device global memory owned by the
 * library (every GPU that loads the library holds it until exit); the call
 * allocates nothing and calls no allocating routine.
 *   - The call needs the workspace of that sequential path: a header, the
 *     chunk table and one record per (chunk, head), with chunks =
 *     T_total / 64 + n_seqs (132,096 bytes per record in bf16, 164,352 in
 *     fp32).  A call needing more than KDA_NOALLOC_SCRATCH_BYTES returns
 *     KDA_ERR_WORKSPACE before any launch (about 500 (chunk, head) records in
 *     bf16, 400 in fp32).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it with the device's CUDA context; a
 *     call under a new context (after a device reset) looks it up again.
 *     Make the first call on each device before any stream capture.
 *   - Every call uses the same array: calls whose executions overlap on the
 *     GPU race.  Order them, e.g. by issuing them on one stream.
 *   - Device-side errors (bad cu_seqlens, a timed-out wait) are recorded in
 *     the array's first word, which the next call clears;
 *     kda_noalloc_read_device_error() reads it.
 * ------------------------------------------------------------------------ */
#define KDA_NOALLOC_SCRATCH_BYTES (64ull << 20)

int kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                          const float *z, const float *A, const float *beta,
                          const int32_t *cu_seqlens, int n_seqs,
                          int64_t T_total, int H, int D, int dtype, float g_min,
                          const float *init_state, void *o, float *final_state,
                          int flags, kda_stream_t stream);

/* kda_noalloc_read_device_error -- synchronise `stream` and read the device
 * error code (bit flags of kda_device_error) that the last
 * kda_chunk_fwd_noalloc on the current device recorded in the library's
 * array.  Allocates nothing.  Returns KDA_OK, KDA_ERR_INVALID_ARG (code NULL)
 * or KDA_ERR_CUDA. */
int kda_noalloc_read_device_error(int32_t *code, kda_stream_t stream);

/* --------------------------------------------------------------------------
 * kda_segment_scan -- intra-device context parallelism over one long packed
 * token stream ("Kimi K3 模型结构（7）", section "KDA：三种执行形态" (SM-level
 * CP of long prefill), eq. (17) and "公式 (17) 的推导": segments are affine
 * maps S -> M S + S~; pairs compose as (M2,S~2) o (M1,S~1) = (M2 M1, M2 S~1 + S~2);
 * section "文档边界": only pairs of the same document are composed).
 *
 * The chunk list (documents cut into 64-token chunks, as in kda_chunk_fwd) is
 * split into n_segments contiguous, chunk-aligned ranges of balanced length
 * (earlier segments one chunk longer when the split is not exact).
 *   phase 1: every (head, segment) computes its pair (M, S~) from a zero state
 *            on its own SMs; a document start inside a segment resets the
 *            pair to (0, init_state[doc]) at that point;
 *   phase 2: entering states S_in[0] = 0, S_in[i+1] = M_i S_in[i] + S~_i;
 *   phase 3: every segment reruns from its exact entering state, writing o and
 *            the final state of every document that ends inside it.
 * Results equal kda_chunk_fwd on the same inputs up to rounding.
 *
 * Arguments as kda_chunk_fwd, plus
 *   n_segments   >= 1 (more segments than chunks leaves some empty), or 0 for
 *                the automatic count kda_segment_scan_auto_segments() returns
 *   pairs_M      (device) fp32 [H, n, D, D] or NULL: M of each segment
 *   pairs_S      (device) fp32 [H, n, D, D] or NULL: S~ of each segment
 *                (n = n_segments, or the automatic count)
 *   workspace    at least kda_segment_scan_workspace_size() bytes (same
 *                n_segments, 0 included).
 * ------------------------------------------------------------------------ */
size_t kda_segment_scan_workspace_size(int64_t T_total, int H, int n_seqs, int n_segments,
                                       int dtype);

/* The segment count kda_segment_scan takes for n_segments = 0: the most
 * segments whose rerun (two blocks per (segment, head)) fits in one wave of
 * the current device's SMs, at most sqrt(chunks / 6) (beyond it the
 * sequential composition costs more than the shorter chains save), at most 64
 * and half the chunks, at least 1; chunks = T_total / 64 + n_seqs.  No device
 * work; 0 for invalid shapes. */
int kda_segment_scan_auto_segments(int64_t T_total, int H, int n_seqs);

int kda_segment_scan(const void *q, const void *k, const void *v,
                     const float *z, const float *A, const float *beta,
                     const int32_t *cu_seqlens, int n_seqs,
                     int64_t T_total, int H, int D, int dtype, float g_min,
                     const float *init_state, int n_segments,
                     float *pairs_M, float *pairs_S,
                     void *o, float *final_state,
                     void *workspace, size_t workspace_bytes, int flags, kda_stream_t stream);

/* --------------------------------------------------------------------------
 * kda_decode_step -- one decode step with MTP draft replay ("Kimi K3 模型结构
 * （7）", section "KDA：三种执行形态，三种内核", decode paragraph: only the
 * projected inputs of draft tokens are cached; the accepted prefix is replayed
 * on chip, the bonus token is applied and the state is written back in place;
 * the next draft window runs speculatively in the same recurrence loop).
 * Per token the delta form of "Kimi K3: the Manos, the Mythos ..." section
 * "FlashKDA 算法": S <- D_t S; u = beta (v - S^T k); S <- S + k u^T; o = S^T q.
 *
 * A window holds W = 1 + n_draft tokens [t0, d1 .. d_{W-1}].  For each b:
 *   1. replay cache[b, 0 .. n_b - 1] (the drafts of the previous window that
 *      were accepted, n_b = num_accepted[b], 0 when num_accepted is NULL);
 *   2. apply t0 (bonus / next token), write o[b, 0], store the state in place;
 *   3. run d1 .. d_{W-1} from that state without storing it, write o[b, j];
 *   4. copy the projected inputs of d1 .. d_{W-1} into cache[b, 0 .. W-2].
 *
 *   state        (device) fp32 [N, H, D, D], read and written in place
 *   q, k, v      (device) [N, W, H, D] dtype;  z (device) fp32 [N, W, H, D]
 *   beta         (device) fp32 [N, W, H] (logits with KDA_FLAG_BETA_SIGMOID);
 *                A (device) fp32 [H]
 *   cache_q, cache_k, cache_v (device) [N, W-1, H, D] dtype, read and written
 *   cache_z      (device) fp32 [N, W-1, H, D]; cache_beta (device) fp32 [N, W-1, H]
 *                (the cache pointers may be NULL only when W == 1)
 *   num_accepted (device) int32 [N] with values in 0 .. W-1, or NULL
 *   N >= 1, H >= 1, D == 128, 1 <= W <= 8
 *   o            (device) [N, W, H, D] dtype, written
 *   error_word   (device) int32 or NULL: KDA_DEVERR_NUM_ACCEPTED is OR-ed in
 *                when a num_accepted value is out of range; that sequence's
 *                state, cache and outputs are then left untouched.
 *   flags        0 or an OR of KDA_FLAG_*, the same for every step of a
 *                sequence (the cache holds inputs as given)
 * state, q, k, v, z, o and the caches must be 16-byte aligned.
 * ------------------------------------------------------------------------ */
int kda_decode_step(float *state,
                    const void *q, const void *k, const void *v,
                    const float *z, const float *beta, const float *A,
                    void *cache_q, void *cache_k, void *cache_v,
                    float *cache_z, float *cache_beta,
                    const int32_t *num_accepted,
                    int N, int H, int D, int W, int dtype, float g_min,
                    void *o, int32_t *error_word, int flags, kda_stream_t stream);

/* --------------------------------------------------------------------------
 * kda_decode_step_fused -- the decode step with what the same paragraph puts
 * in the fused kernel around the recurrence ("Kimi K3 模型结构（7）", section
 * "KDA：三种执行形态，三种内核", decode: short convolution, input normalisation,
 * gate, KDA recurrence and output normalisation in one loop over the replayed
 * drafts, the bonus token and the next draft window).  The module around the
 * recurrence is the one of "Kimi K3: the Manos, the Mythos ..." section "Kimi
 * Linear": q, k, v pass a causal short convolution (left padding; width 4, as
 * in "Kimi K3 模型结构（7）", section "KDA 上下文并行", short-conv note) after
 * their projection; q and k are L2-normalised; the output is normalised per
 * head and scaled by an output gate.
 *
 * Per sequence b the committed stream continues the convolution state:
 * [conv_state (3 inputs), replayed drafts 0 .. n_b - 1, t0], and the window's
 * drafts follow t0.  Per token, in order:
 *   1. y_t = sum_{j<4} conv_w[., c, j] x_{t-3+j} per channel for each of q, k, v
 *      (pre-convolution inputs x come from the window or the cache), then SiLU
 *      with KDA_FLAG_CONV_SILU;
 *   2. the input options (KDA_FLAG_QK_L2NORM on the convolved q, k;
 *      KDA_FLAG_BETA_SIGMOID on beta);
 *   3. the recurrence exactly as kda_decode_step (replay, t0 committed in place,
 *      drafts speculative);
 *   4. o = o_raw / sqrt(mean_c(o_raw^2) + o_norm_eps) * o_norm_w[c] * sigmoid(o_gate)
 *      for the window's tokens, the mean over the 128 value channels of one
 *      (token, head).
 * The convolution state becomes the last three pre-convolution inputs of the
 * committed stream (ending at t0); the cache takes the window's drafts as given.
 *
 * Arguments as kda_decode_step, plus
 *   conv_w       (device) fp32 [3, H, D, 4]: taps of q, k, v per channel, tap 3
 *                on the current token (16-byte aligned)
 *   conv_state   (device) fp32 [N, H, 3, 3, D], read and written in place:
 *                q, k, v x the three latest committed inputs, oldest first
 *   o_gate       (device) fp32 [N, W, H, D]: output-gate logits
 *   o_norm_w     (device) fp32 [D]: output-norm weight (one vector for all heads)
 *   o_norm_eps   >= 0, added under the root
 *   flags        0 or an OR of KDA_FLAG_QK_L2NORM, KDA_FLAG_BETA_SIGMOID,
 *                KDA_FLAG_CONV_SILU
 * A sequence with an out-of-range num_accepted keeps its convolution state too.
 * ------------------------------------------------------------------------ */
int kda_decode_step_fused(float *state,
                          const void *q, const void *k, const void *v,
                          const float *z, const float *beta, const float *A,
                          const float *conv_w, float *conv_state,
                          const float *o_gate, const float *o_norm_w, float o_norm_eps,
                          void *cache_q, void *cache_k, void *cache_v,
                          float *cache_z, float *cache_beta,
                          const int32_t *num_accepted,
                          int N, int H, int D, int W, int dtype, float g_min,
                          void *o, int32_t *error_word, int flags, kda_stream_t stream);

/* --------------------------------------------------------------------------
 * kda_read_device_error -- synchronise `stream` and read the device error
 * code that the last kda_chunk_fwd / kda_segment_scan on `workspace`
 * recorded (bit flags of kda_device_error; 0 = none).
 * Returns KDA_OK, KDA_ERR_INVALID_ARG or KDA_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int kda_read_device_error(const void *workspace, int32_t *code, kda_stream_t stream);

/* --------------------------------------------------------------------------
 * Diagnostics (no counterpart in the pages): per-launch timing and counting.
 *
 * kda_profile_enable(1) makes every following entry point record a CUDA event
 * on its stream before its first launch and after each of its kernel launches
 * (at most 256 marks are kept).  kda_profile_collect() synchronises on the
 * last mark, returns up to `max` (kernel name, milliseconds since the previous
 * mark) pairs in launch order, and clears the marks.  Names are static strings
 * owned by the library.  Returns the number of pairs, or -KDA_ERR_CUDA.
 * kda_launch_count() is the number of kernels the library has launched since
 * it was loaded (always counted, profiling or not).
 * ------------------------------------------------------------------------ */
int kda_profile_enable(int on);
int kda_profile_collect(const char **names, float *ms, int max);
long long kda_launch_count(void);

/* kda_set_wait_budget -- the clock-cycle limit of the library's waits on
 * flags that other blocks of the same launch raise (the fused prefill's
 * record-ready flags) and of the decode's waits on its own copies, for every
 * call made afterwards in this process (not thread-safe against calls in
 * flight on other host threads).  A wait that runs out records
 * KDA_DEVERR_TIMEOUT (workspace error word, decode error word), its block
 * stops, lets its own copies and tensor-core work finish and frees its TMEM,
 * and the call's outputs are then undefined.  cycles <= 0 restores the
 * default (2e9 cycles, about one second).  Returns the previous limit.  Meant
 * for tests of the timeout path; the other waits keep the default. */
long long kda_set_wait_budget(long long cycles);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
