/*
 * kda.h: C ABI of the GB300 (sm_103a) KDA recurrence library (libkda.so).
 *
 * The operation.  Per (sequence, head), with key dimension dk and value
 * dimension dv (both 128 here), a matrix state S in R^{dk x dv} evolves token
 * by token as
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * ("Kimi K3" study notes, dimensionstp, section 3-2 "2) Kimi Delta Attention":
 * state-update and read-out equations).  alpha_t = exp(log_alpha_t) is a decay
 * per key channel ("Kimi K3: 架构、训练与系统全景解析", section 4.2.2, first of
 * the three parts of the update), beta_t is the scalar write strength, and the
 * read-out uses the post-update state with no scale factor (same section, last
 * paragraph).  K3 bounds the log-decay below by -5 (same page, sections 2.1 and
 * 4.2.5), so over any 16-token tile the cumulative log-decay lies in [-80, 0]
 * and its inverse exponential stays within the bf16/fp32 range.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are caller-owned DEVICE memory unless stated
 *     otherwise and C-contiguous.  Alignment: see each entry point (beta is
 *     always only element-aligned).  The library never allocates or frees
 *     device memory, reads no environment variables and keeps no global state
 *     (the one exception, kda_chunk_fwd_noalloc's fixed device array, is
 *     described there).
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = legacy default stream).  Inputs must stay alive and unmodified
 *     until the stream has passed the call.
 *   - Every function returns a kda_status code; nothing is launched when the
 *     return value is not KDA_OK.  No exceptions cross the ABI.
 *   - Preconditions that are NOT checked (accuracy is only guaranteed inside
 *     them): log_alpha in [-5, 0], beta in [0, 1], q and k finite with
 *     ||k||_2 <= 1 (the KDA layer L2-normalises q and k).
 *   - Only dk = dv = 128 is supported (KDA head dimension of K3); any other
 *     positive value returns KDA_ERR_UNSUPPORTED.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
enum kda_status_code {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null / misaligned / overlapping / inconsistent args */
  KDA_ERR_UNSUPPORTED = 2, /* dk, dv or dtype outside what the kernels implement  */
  KDA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required          */
  KDA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed         */
  KDA_ERR_TIMEOUT = 5      /* a bounded in-kernel wait gave up (device status)     */
};

/* Element type of q, k, v and out.  log_alpha, beta and states are always fp32. */
enum kda_dtype_code {
  KDA_F32 = 0,
  KDA_BF16 = 1
};

/* Static description of a status code.  Never returns NULL. */
const char *kda_status_string(int status);

/* Library version as major * 10000 + minor * 100 + patch. */
int kda_version(void);

/*
 * Bytes of device workspace kda_chunk_fwd needs for this problem size on the
 * current device, written to *bytes.  The workspace holds:
 *   - the device status word (bounded waits that give up record
 *     KDA_ERR_TIMEOUT there; a device-resident cu_seqlens that is not a valid
 *     prefix sum records KDA_ERR_INVALID_ARG);
 *   - when cu_seqlens is a host pointer, a device copy of it;
 *   - for a bf16 call with few enough (sequence, head) chains that each
 *     sequence can be cut into K >= 2 segments with 2 K x chains <= SMs (or
 *     (2 K - 1) x chains <= SMs for a call without an initial state, whose
 *     first segments need no transition run; the size covers the larger K), the
 *     scratch of the in-device split (segment bounds, three fp32 states per
 *     segment and head, and one bf16 value per token, head and channel): the
 *     segments run side by side and their states are stitched together exactly
 *     ("Kimi K3: 架构、训练与系统全景解析", section 7.1: segments compose as
 *     affine maps of the state);
 *   - otherwise, for a bf16 call whose chains leave at least four times as
 *     many of the device's SMs idle as there are chains, the ring of the
 *     helper CTAs.
 *     These run on the idle SMs and compute the state-independent half of
 *     later chunks (operand build, Gram matrix, triangular solve); about
 *     455 KiB per chain.
 * The size covers every schedule kda_chunk_fwd_sched may be asked for.
 * kda_chunk_fwd runs without the split or the helpers when the workspace it
 * gets has room for neither.  Helpers leave the results bitwise unchanged; the
 * split changes the rounding (its results meet the same tolerances).  Because
 * the schedule follows the device's SM count, kda_chunk_fwd's results can
 * differ in rounding between GPUs with different SM counts; a caller that
 * needs the same bits everywhere passes max_split = 0 to kda_chunk_fwd_sched.
 * Errors: KDA_ERR_INVALID_ARG for a NULL `bytes` or negative sizes,
 * KDA_ERR_UNSUPPORTED for dk/dv/dtype outside the supported set.
 */
int kda_chunk_fwd_workspace_size(int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk,
                                 int32_t dv, int dtype, size_t *bytes);

/*
 * Chunkwise-parallel prefill over packed variable-length sequences.
 *
 * The sequences are cut into chunks of 64 tokens (never straddling a sequence
 * boundary; the last chunk of a sequence may be partial).  Inside a chunk the
 * causal token-token interactions are dense lower-triangular matrix products;
 * across chunks the fp32 state is carried serially ("Kimi K3: 架构、训练与系统
 * 全景解析", section 4.2.4: state passed between chunks, lower-triangular
 * matrix work within a chunk, output = a term reading the pre-chunk state plus
 * an intra-chunk causal term; the UT-transform form of the intra-chunk solve).
 * The result equals the token-by-token recurrence above up to rounding.
 *
 * Arguments (N = n_tokens, S = n_seqs):
 *   q, k       [N, H, dk]  dtype       queries / keys
 *   v          [N, H, dv]  dtype       values
 *   log_alpha  [N, H, dk]  fp32        per-channel log-decay (<= 0, >= -5)
 *   beta       [N, H]      fp32        write strength
 *   init_state [S, H, dk, dv] fp32 or NULL (zero state).  READ ONLY: a cached
 *              state snapshot is never modified (prefix-cache snapshots are
 *              copied, not advanced in place: same page, section 7.4).
 *   cu_seqlens [S + 1] int32, cu_seqlens[0] = 0, non-decreasing,
 *              cu_seqlens[S] = N.  May be host or device memory: a host array
 *              is validated here (KDA_ERR_INVALID_ARG on failure) and copied
 *              into the workspace; a device array is validated by the kernel,
 *              which then writes nothing and records KDA_ERR_INVALID_ARG in
 *              the device status.
 *   dtype      KDA_F32 (fp32 CUDA-core path) or KDA_BF16 (tcgen05 tensor-core
 *              path; fp32 state and accumulation).
 *   out        [N, H, dv]  dtype       o_t for every token
 *   final_state [S, H, dk, dv] fp32 or NULL.  Must not overlap init_state.
 *   workspace  device memory of at least kda_chunk_fwd_workspace_size() bytes,
 *              16-byte aligned; its device status word is cleared at the start
 *              of every call (stream-ordered).
 * Alignment: q, k, v, log_alpha, out, init_state, final_state 16 bytes (tiles
 * are fetched by TMA); beta 4 bytes.
 * A zero-length sequence writes final_state = init_state (or zeros).
 * Errors (returned before any launch): KDA_ERR_INVALID_ARG (NULL required
 * pointer, H <= 0, negative sizes, misalignment, init/final overlap, bad host
 * cu_seqlens), KDA_ERR_UNSUPPORTED (dk or dv != 128, unknown dtype),
 * KDA_ERR_WORKSPACE (NULL or too small), KDA_ERR_CUDA (launch failure).
 */
int kda_chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  const float *beta, const float *init_state, const int32_t *cu_seqlens,
                  int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv,
                  int dtype, void *out, float *final_state, void *workspace,
                  size_t workspace_bytes, void *stream);

/*
 * The gradient of kda_chunk_fwd (the backward pass for training: "Kimi K3:
 * 架构、训练与系统全景解析", section 7.1, the chunked KDA kernel serves training
 * as well as prefill; the pages print no gradient, so this is the chain rule
 * through the update and read-out above, in reverse token order).  For a loss
 * whose gradients with respect to every output o_t (d_out) and every final
 * state (d_final_state) are given, it returns the gradients with respect to
 * every input:
 *   d_out        [N, H, dv]  dtype           gradient of the outputs
 *   d_final_state [S, H, dk, dv] fp32 or NULL (zero)
 *   dq, dk       [N, H, dk]  dtype;  dv [N, H, dv] dtype
 *   d_log_alpha  [N, H, dk]  fp32;   d_beta [N, H] fp32
 *   d_init_state [S, H, dk, dv] fp32 or NULL (not written); the gradient with
 *                respect to init_state (also when init_state is NULL: the
 *                gradient at the zero state)
 * The other arguments are those of kda_chunk_fwd (same inputs, same
 * cu_seqlens rules: host arrays are validated here, device arrays in the
 * kernels, which record KDA_ERR_INVALID_ARG in the workspace's status word; the
 * gradients are then undefined).  A forward
 * sweep stores states in the workspace and a reverse sweep recomputes what it
 * needs from them.  Two passes:
 *  - bf16 (when the states fit in 16 GiB): the chunked pass.  States every 16
 *    tokens, as bf16 (32 KiB per head for every 16 tokens and per sequence),
 *    from a chunked forward sweep with the same bf16 operands; the reverse
 *    sweep takes 16-token chunks in the chunk form of the recurrence, every
 *    product on the tensor cores with bf16 operands and fp32 accumulation (the
 *    gradient of the state as an operand in a pair of bf16 terms), fp32 state
 *    gradient.  Every result element is written once: results do not vary
 *    between calls.
 *  - otherwise, and for fp32: the token-loop pass.  States every E tokens, E
 *    the smallest power of two >= 4 whose stored states fit in 16 GiB, or 1024
 *    (kda_chunk_bwd_sched takes E from the caller, and with it this pass, for
 *    bf16 too); the reverse sweep recomputes the states in between in groups
 *    of four tokens.  fp32 arithmetic on CUDA cores; dq, dk, d_log_alpha and
 *    d_beta are sums over the value channels, added in fp32 in an order that
 *    may vary between calls (last bits only).
 * Alignment: q, k, v, log_alpha and d_out 16 bytes (their rows are fetched by
 * 16-byte asynchronous copies); element alignment for every other tensor.  No
 * output may overlap an input or another output.
 * Errors: as kda_chunk_fwd, with the workspace of kda_chunk_bwd_workspace_size.
 */
int kda_chunk_bwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  const float *beta, const float *init_state, const int32_t *cu_seqlens,
                  int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv, int dtype,
                  const void *d_out, const float *d_final_state, void *dq, void *dk_, void *dv_,
                  float *d_log_alpha, float *d_beta, float *d_init_state, void *workspace,
                  size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace kda_chunk_bwd needs: the status block, a device
 * copy of a host cu_seqlens, the stored states (32 KiB per head for every 16
 * tokens, or 64 KiB for every E, and per sequence, as in kda_chunk_bwd) and,
 * for the token-loop pass, fp32 accumulators of dq and dk.
 * Errors: as kda_chunk_fwd_workspace_size.
 */
int kda_chunk_bwd_workspace_size(int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk,
                                 int32_t dv, int dtype, size_t *bytes);

/*
 * kda_chunk_bwd with the checkpoint interval E chosen by the caller:
 * ckpt_every = 0 is the library's choice (as kda_chunk_bwd), otherwise a power
 * of two in [4, 1024], which selects the token-loop pass with that interval
 * for either dtype.  E = 4 recomputes nothing twice and stores the most
 * states; each doubling halves the stored states and adds about (E / 4 - 1) / 2
 * recomputed forward steps per token.  Every E gives the same results: the
 * states replayed from a stored one are the forward sweep's own, bit for bit
 * (the token-loop pass; the chunked pass rounds differently, within the same
 * tolerance).
 * Arguments, results and errors otherwise those of kda_chunk_bwd; another
 * ckpt_every is KDA_ERR_INVALID_ARG.  The workspace must hold
 * kda_chunk_bwd_workspace_size_sched bytes for the same ckpt_every.
 */
int kda_chunk_bwd_sched(const void *q, const void *k, const void *v, const float *log_alpha,
                        const float *beta, const float *init_state, const int32_t *cu_seqlens,
                        int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv,
                        int dtype, const void *d_out, const float *d_final_state, void *dq,
                        void *dk_, void *dv_, float *d_log_alpha, float *d_beta,
                        float *d_init_state, int32_t ckpt_every, void *workspace,
                        size_t workspace_bytes, void *stream);

/* Workspace bytes of kda_chunk_bwd_sched for ckpt_every (0: the library's choice). */
int kda_chunk_bwd_workspace_size_sched(int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk,
                                       int32_t dv, int dtype, int32_t ckpt_every, size_t *bytes);

/*
 * kda_chunk_fwd with the schedule capped by the caller.  Arguments, results
 * and errors are those of kda_chunk_fwd, plus:
 *   max_split    upper bound on the segments per sequence of the in-device
 *                split (-1: the library's choice, as in kda_chunk_fwd;
 *                0 or 1: never split);
 *   max_helpers  upper bound on the helper CTAs (-1: the library's choice;
 *                0: no helpers).
 * kda_chunk_fwd(...) is kda_chunk_fwd_sched(..., -1, -1, ...).  The caps only
 * lower what the library would pick for the device (they never force a
 * schedule that does not fit), so every call stays within the workspace size
 * kda_chunk_fwd_workspace_size reports.
 */
int kda_chunk_fwd_sched(const void *q, const void *k, const void *v, const float *log_alpha,
                        const float *beta, const float *init_state, const int32_t *cu_seqlens,
                        int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv,
                        int dtype, void *out, float *final_state, int32_t max_split,
                        int32_t max_helpers, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * kda_chunk_fwd without a workspace argument, for callers that cannot provide
 * or allocate device memory for the library: for instance a serving engine
 * whose framework allocator owns all device memory and forbids cudaMalloc or
 * extra buffers outside its pool.  (Library-level entry point: the pages have
 * no counterpart.)
 *
 * Arguments and errors are those of kda_chunk_fwd minus the workspace.  The
 * scratch kda_chunk_fwd keeps in its workspace (device status block, device
 * copy of a host cu_seqlens) lives instead in one fixed-size device array
 * inside libkda, which every GPU that loads the library holds until process
 * exit.  Nothing is allocated or freed by the call.
 *   - At most 4095 sequences per call; more returns KDA_ERR_WORKSPACE and
 *     launches nothing.
 *   - The array is shared by every call on a device and keeps the last call's
 *     contents (the status block is cleared, stream-ordered, by each call).
 *     Calls that overlap on the GPU race on it: issue them on one stream or
 *     serialise them.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, once per device); make that first call before
 *     any stream capture begins.
 *   - The array has no room for the in-device split, the helper ring or the
 *     longest-first order, so the call always takes the plain schedule (one
 *     CTA per sequence and head).  Results equal kda_chunk_fwd's bitwise where
 *     kda_chunk_fwd takes the plain or helper schedule, and meet the same
 *     tolerance where it splits; few-chain shapes run slower than there.
 *   - Kernel-recorded errors (a malformed device cu_seqlens, a bounded wait
 *     that gave up) go to the array's status block: the call itself returns
 *     KDA_OK; read them with kda_noalloc_read_status.
 */
int kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, const float *init_state, const int32_t *cu_seqlens,
                          int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv,
                          int dtype, void *out, float *final_state, void *stream);

/*
 * The device status of the last kda_chunk_fwd_noalloc calls on the current
 * device, read from the library's fixed array exactly as
 * kda_read_device_status reads a workspace (synchronises `stream` first;
 * `clear` non-zero resets it).  Allocates nothing.  No counterpart on the pages.
 * Errors: KDA_ERR_INVALID_ARG (NULL device_status), KDA_ERR_CUDA.
 */
int kda_noalloc_read_status(void *stream, int clear, int32_t *device_status);

/*
 * Reads (and, if `clear` is non-zero, resets) the device status word of a
 * kda_chunk_fwd or kda_chunk_bwd workspace (both start with it).  Synchronises `stream` first, so it reports the
 * status of every call issued on that stream before it.  *device_status gets
 * KDA_OK or the kda_status code a kernel recorded.
 * Errors: KDA_ERR_INVALID_ARG (NULL workspace or device_status), KDA_ERR_CUDA.
 */
int kda_read_device_status(void *workspace, void *stream, int clear, int32_t *device_status);

/*
 * As kda_read_device_status, with where the status was recorded:
 * detail4[0] = code, detail4[1] = a kernel-specific tag of the failing step,
 * detail4[2] = the chain (sequence * H + head), detail4[3] = the chunk index.
 */
int kda_read_device_status_detail(void *workspace, void *stream, int clear, int32_t *detail4);

/*
 * TEST CONTROL of the bounded waits (fault-handling tests only; the pages have
 * no counterpart).  Arms `workspace` so that, in the next bf16 kda_chunk_fwd
 * call that takes the plain schedule with it, the CTA of chain `chain`
 * (sequence * H + head) bounds each of its waits by `wait_us` microseconds and
 * one of its warps withholds its arrival on the barrier that releases chunk
 * `chunk`'s Gram products.  The wait that then never completes gives up:
 * the kernel records KDA_ERR_TIMEOUT with that chain and chunk in the device
 * status, drains its copies and MMAs, frees its tensor memory and returns,
 * leaving that chain's outputs from the chunk before on, and its final
 * state, unwritten.  Nothing traps or waits without bound.  The control is
 * consumed by the CTA that acts on it; chain < 0 disarms it.  Synchronises
 * `stream`.  Errors: KDA_ERR_INVALID_ARG (NULL or misaligned workspace,
 * chunk < 0 or wait_us outside [1, 2000000] when arming), KDA_ERR_CUDA.
 */
int kda_test_arm_timeout(void *workspace, int32_t chain, int32_t chunk, uint32_t wait_us,
                         void *stream);

/*
 * The affine state map of every packed sequence, for context parallelism
 * ("Kimi K3: 架构、训练与系统全景解析", section 7.1: a sequence segment maps the
 * state it starts from to the one it ends with as S_end = M S_start + B, its
 * "affine pair"; pairs of consecutive segments compose, so devices holding
 * different segments of one sequence exchange their pairs once and each then
 * runs its segment from its true start state).  For sequence s and head h:
 *   state_b[s, h] = B = the final state of kda_chunk_fwd from a zero state,
 *   state_m[s, h] = M = the product of the sequence's transitions
 *                       (I - beta_t k_t k_t^T) Diag(alpha_t), latest on the left,
 * computed in one launch (the chunk kernel run from 0, and from I with v = 0)
 * that writes no outputs.
 * Arguments as for kda_chunk_fwd; state_b, state_m [S, H, 128, 128] fp32,
 * 16-byte aligned, not overlapping.
 * Errors: as kda_chunk_fwd; KDA_ERR_UNSUPPORTED for fp32 inputs (bf16 only).
 */
int kda_chunk_fwd_transitions(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta,
                              const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens,
                              int32_t H, int32_t dk, int32_t dv, int dtype, float *state_b,
                              float *state_m, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * Composition of affine state maps (same section).  For every sequence s, head
 * h, with the sequence's n_segments pairs (B_j, M_j) at index s * n_segments + j:
 *   S_0 = init_state[s, h] (zeros if init_state is NULL),
 *   S_{j+1} = M_j S_j + B_j          (fp32, DEVICE memory throughout)
 *   start_states[s * n_segments + j, h] = S_j  (j < n_segments; if non-NULL)
 *   end_state[s, h] = S_{n_segments}           (if non-NULL)
 * State tensors are [., H, 128, 128] fp32, 16-byte aligned; outputs may not
 * overlap inputs or each other.
 * Errors: KDA_ERR_INVALID_ARG (NULL state_b/state_m, n_segments < 1, H <= 0,
 * misalignment, overlap), KDA_ERR_UNSUPPORTED (dk or dv != 128), KDA_ERR_CUDA.
 */
int kda_state_combine(const float *init_state, const float *state_b, const float *state_m,
                      int32_t n_seqs, int32_t n_segments, int32_t H, int32_t dk, int32_t dv,
                      float *start_states, float *end_state, void *stream);

/*
 * Helper activity of the last kda_chunk_fwd call that used `workspace`:
 * *help_published = chunk packages the helper CTAs wrote, *help_consumed = the
 * ones a chain CTA used instead of computing the chunk itself (both 0 when no
 * helpers ran).  Synchronises `stream` first.
 * Errors: KDA_ERR_INVALID_ARG (NULL pointer), KDA_ERR_CUDA.
 */
int kda_read_chunk_stats(void *workspace, void *stream, int32_t *help_published,
                         int32_t *help_consumed);

/*
 * One recurrent decode step for B sequences x H heads, one new token each,
 * state advanced IN PLACE (the decode state is advanced in place:
 * "Kimi K3: 架构、训练与系统全景解析", section 4.2.7).
 *
 *   state      [B, H, dk, dv] fp32   read, then overwritten with S_t
 *   q, k       [B, H, dk]  dtype
 *   v          [B, H, dv]  dtype
 *   log_alpha  [B, H, dk]  fp32
 *   beta       [B, H]      fp32
 *   out        [B, H, dv]  dtype     o_t = S_t^T q_t
 * One HBM pass: each state is read once and written once.
 * Alignment: state 16 bytes; v and out 4 elements; q, k 1 element;
 * log_alpha and beta 4 bytes.
 * Errors (before any launch): KDA_ERR_INVALID_ARG (NULL pointer, B < 0,
 * H <= 0, misalignment, `out` overlapping `state`), KDA_ERR_UNSUPPORTED
 * (dk or dv != 128, unknown dtype), KDA_ERR_CUDA (launch failure).
 */
int kda_decode_step(float *state, const void *q, const void *k, const void *v,
                    const float *log_alpha, const float *beta, int32_t B, int32_t H,
                    int32_t dk, int32_t dv, int dtype, void *out, void *stream);

/*
 * Replay of accepted draft tokens after speculative-decode verification ("Kimi
 * K3: 架构、训练与系统全景解析", KDA state replay under speculative decoding: the
 * per-token projected inputs of the draft tokens are cached instead of a state
 * per draft position; after verification only the accepted prefix is replayed
 * in an on-chip recurrence and only the final state is written back).
 *
 * For every sequence b and head h, applies the decode step of kda_decode_step
 * to tokens t = 0 .. n_b - 1 in order, n_b = n_accept[b] clamped to [0, T]:
 *
 *   state      [B, H, dk, dv] fp32   read once, overwritten once with the state
 *                                    after token n_b - 1 (untouched if n_b = 0)
 *   q, k       [B, T, H, dk]  dtype  cached inputs of the T draft positions
 *   v          [B, T, H, dv]  dtype
 *   log_alpha  [B, T, H, dk]  fp32
 *   beta       [B, T, H]      fp32
 *   n_accept   [B]            int32, DEVICE memory: accepted tokens per sequence
 *   out        [B, T, H, dv]  dtype  o_t of every replayed token, or NULL; rows
 *                                    t >= n_b are not written
 * Alignment: state, q, k, v and log_alpha 16 bytes (their rows are fetched by
 * bulk copies); out 4 elements; beta and n_accept 4 bytes.
 * Errors (before any launch): KDA_ERR_INVALID_ARG (NULL pointer other than
 * out, B < 0, T <= 0, H <= 0, misalignment, `out` overlapping `state`),
 * KDA_ERR_UNSUPPORTED (dk or dv != 128, unknown dtype), KDA_ERR_CUDA.
 * No counterpart on the pages' interface (they give none); the layout is this
 * library's.
 */
int kda_decode_replay(float *state, const void *q, const void *k, const void *v,
                      const float *log_alpha, const float *beta, const int32_t *n_accept,
                      int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, int dtype,
                      void *out, void *stream);

/*
 * The per-token steps before the recurrence, in one pass ("Kimi K3: 架构、训练与
 * 系统全景解析", section 4.2.3: short convolution of kernel size 4, Swish,
 * L2Norm(q, k), the write strength beta and the decay alpha; sections 2.1 and
 * 4.2.5: the decay is a lower-bounded scaled sigmoid with bound -5).  The pages
 * print no formulas for these steps; this library computes, per packed
 * sequence, token t, head h and channel c:
 *   conv(x)[t]  = sum_{j<4} conv_w[., h, c, j] x[t - 3 + j]   (0 before the
 *                 sequence start; no state carried across calls)
 *   q = l2norm(swish(conv(q_raw))),  k = l2norm(swish(conv(k_raw))),
 *   v = swish(conv(v_raw)),  swish(x) = x sigmoid(x),
 *   l2norm(x) = x / sqrt(sum_c x^2 + 1e-6)  (over the 128 channels of a head),
 *   log_alpha = -5 sigmoid(a_logit),  beta = sigmoid(b_logit).
 *
 *   q_raw, k_raw, v_raw, q, k, v  [N, H, 128] dtype
 *   conv_w      [3, H, 128, 4] fp32   (q, k, v weights; taps oldest first)
 *   a_logit, log_alpha            [N, H, 128] fp32
 *   b_logit, beta                 [N, H] fp32
 *   cu_seqlens  [n_seqs + 1] int32, DEVICE memory, prefix sums from 0 to N
 * Alignment: the dtype tensors 4 elements; conv_w, a_logit, log_alpha 16
 * bytes; b_logit, beta, cu_seqlens 4 bytes.  No output may overlap an input.
 * Errors: KDA_ERR_INVALID_ARG (NULL pointer, n_seqs < 1, n_tokens < 0 or above
 * INT32_MAX (cu_seqlens is int32), H <= 0, misalignment, overlap),
 * KDA_ERR_UNSUPPORTED (dk or dv != 128, unknown dtype), KDA_ERR_CUDA.  A
 * malformed device cu_seqlens gives wrong values, never an out-of-range access.
 */
int kda_prep_fwd(const void *q_raw, const void *k_raw, const void *v_raw, const float *conv_w,
                 const float *a_logit, const float *b_logit, const int32_t *cu_seqlens,
                 int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv, int dtype,
                 void *q, void *k, void *v, float *log_alpha, float *beta, void *stream);

/*
 * kda_prep_fwd continuing every packed sequence across calls: the short
 * convolution reads the three raw rows before each sequence's first token in
 * this call from a carried window instead of zeros, so a prefill may be split
 * into several calls, and decode steps (every sequence of length 1) continue
 * the same window ("Kimi K3: 架构、训练与系统全景解析", section 4.2.3: the short
 * convolution of kernel size 4 before the recurrence; section 7.4: decode
 * carries a fixed-size per-sequence state).  Arguments as kda_prep_fwd, plus:
 *   conv_state_in  [n_seqs, 3, 3, H, 128] dtype or NULL (zeros): per sequence,
 *                  for q, k and v, the three raw (unconvolved) rows before
 *                  its first token here, oldest first;
 *   conv_state_out [n_seqs, 3, 3, H, 128] dtype or NULL (not written): the
 *                  same three rows before the token after this call: the
 *                  sequence's last three raw rows, or, for a sequence shorter
 *                  than three tokens, the newest rows of conv_state_in
 *                  followed by all of its rows.
 * conv_state_out may be conv_state_in itself (updated in place, after every
 * read of it); otherwise neither may overlap the other or any tensor argument.
 * The results equal kda_prep_fwd over the concatenated tokens of all calls.
 * Alignment: the windows 4 elements.  Errors: as kda_prep_fwd.
 */
int kda_prep_fwd_state(const void *q_raw, const void *k_raw, const void *v_raw,
                       const float *conv_w, const float *a_logit, const float *b_logit,
                       const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t H,
                       int32_t dk, int32_t dv, int dtype, const void *conv_state_in,
                       void *conv_state_out, void *q, void *k, void *v, float *log_alpha,
                       float *beta, void *stream);

/*
 * The whole KDA layer between its projections, replayed over the accepted
 * draft tokens of a speculative decode step in one kernel ("Kimi K3: 架构、训练
 * 与系统全景解析", KDA state replay under speculative decoding: the short
 * convolution, norms, gating, the KDA recurrence and the output norm are fused
 * and replayed on chip over the accepted prefix; the recurrent state and the
 * convolution window are written back once).  For every sequence b and head h,
 * with n_b = n_accept[b] clamped to [0, T], tokens t = 0 .. n_b - 1 in order:
 *   q, k, v, log_alpha, beta = kda_prep_fwd_state of the cached raw rows from
 *       the sequence's window (so q, k are L2-normalised Swish(conv(.)) and v
 *       is Swish(conv(.)), in fp32 inside the kernel);
 *   the decode step of kda_decode_step on the state;
 *   out = the kda_post_fwd of that step's output o with gate logits g.
 *   state      [B, H, 128, 128] fp32, IN PLACE (untouched if n_b = 0)
 *   conv_state [B, 3, 3, H, 128] dtype, IN PLACE: (q, k, v) x three raw rows,
 *              oldest first, before the next token (untouched if n_b = 0)
 *   q_raw, k_raw, v_raw, g  [B, T, H, 128] dtype  cached projections / gate logits
 *   a_logit    [B, T, H, 128] fp32;  b_logit [B, T, H] fp32
 *   conv_w     [3, H, 128, 4] fp32;  gamma [128] fp32
 *   n_accept   [B] int32, DEVICE memory
 *   out        [B, T, H, 128] dtype or NULL; rows t >= n_b are not written
 * The library's layout, not the pages' (they give none).
 * Alignment: state, conv_state, q_raw, k_raw, v_raw, g, a_logit, conv_w and
 * gamma 16 bytes (rows are fetched by bulk copies); out 4 elements; b_logit
 * and n_accept 4 bytes.
 * Errors (before any launch): KDA_ERR_INVALID_ARG (NULL pointer other than
 * out, B < 0, T <= 0, H <= 0, misalignment, out overlapping state or the
 * window, the window overlapping the state), KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA.
 */
int kda_layer_replay(float *state, void *conv_state, const void *q_raw, const void *k_raw,
                     const void *v_raw, const float *a_logit, const float *b_logit, const void *g,
                     const float *conv_w, const float *gamma, const int32_t *n_accept, int32_t B,
                     int32_t T, int32_t H, int32_t dk, int32_t dv, int dtype, void *out,
                     void *stream);

/*
 * The step after the recurrence ("Kimi K3: 架构、训练与系统全景解析", section
 * 4.2.6): head-wise RMSNorm of the recurrent output, then the sigmoid output
 * gate whose logits g come from the input-dependent full-rank projection
 * (computed outside this library):
 *   out = o / sqrt(mean_c o^2 + 1e-5) * gamma[c] * sigmoid(g)
 *   o, g, out  [N, H, 128] dtype;  gamma [128] fp32 (shared by all heads)
 * out may alias o (in place).  Alignment: o, g, out 4 elements; gamma 16 bytes.
 * Errors: KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED (dv != 128, unknown dtype),
 * KDA_ERR_CUDA.
 */
int kda_post_fwd(const void *o, const void *g, const float *gamma, int64_t n_tokens, int32_t H,
                 int32_t dv, int dtype, void *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
