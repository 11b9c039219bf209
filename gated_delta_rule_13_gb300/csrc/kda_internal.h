// Internal host-side declarations shared by the translation units of libkda.
// Not part of the public ABI (include/kda.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int kHeadDim = 128;    // dk = dv = 128 (KDA head dimension of K3)
constexpr int kChunk = 64;       // tokens per chunk of the tensor-core prefill
constexpr int kChunkF32 = 32;    // tokens per chunk of the fp32 CUDA-core prefill
constexpr size_t kStatusBytes = 256;  // device status block at the start of the workspace
constexpr int kNoAllocMaxSeqs = 4095;  // sequence limit of kda_chunk_fwd_noalloc

// Device status block, first bytes of the kda_chunk_fwd workspace.
struct DeviceStatus {
  int32_t code;     // KDA_OK or the first recorded kda_status code
  int32_t detail;   // where it happened (kernel-specific tag)
  int32_t chain;    // chain (seq * H + head) that recorded it
  int32_t chunk;    // chunk index inside the chain
  int32_t help_published;  // chunk packages the helper CTAs wrote (bf16 prefill)
  int32_t help_consumed;   // of those, the ones a chain CTA used
};

// Test control of the bf16 prefill, at kTestControlOffset inside the status
// block (not cleared by a call).  When both magic words are set, the chain CTA
// `chain` of the next plain launch waits at most `wait_us` microseconds on any
// barrier, one of its compute warps withholds its arrival on the "Gram operands
// built" barrier of chunk `chunk`, and the CTA clears the magic words (one
// shot).  The wait that can then never complete gives up and records
// KDA_ERR_TIMEOUT, which is how the tests exercise the timeout path without
// faulting or hanging anything.
constexpr size_t kTestControlOffset = 128;
constexpr uint64_t kTestMagic0 = 0x4b44412d74657374ull, kTestMagic1 = 0x74696d656f75742eull;
struct TestControl {
  uint64_t magic0, magic1;
  int32_t chain, chunk;
  uint32_t wait_us;
  int32_t pad;
};
static_assert(sizeof(DeviceStatus) <= kTestControlOffset, "status block layout");
static_assert(kTestControlOffset + sizeof(TestControl) <= kStatusBytes, "status block layout");

// Helper CTAs of the tensor-core prefill.  When a call has fewer chains than the
// GPU has SMs, the idle SMs run "helpers" that compute the state-independent
// half of chunks ahead of the chain CTAs: the operand build, the Gram matrix,
// P and the triangular solve.  Each result ("package": the shared-memory images
// of [Qt; Kt], Kdec, T', P and Gamma) goes to a per-chain ring of slots in the
// workspace.  A chain CTA that finds a chunk's package ready copies it in and
// skips that work; otherwise it computes the chunk itself.  It never waits for a
// helper.
constexpr int kHelpLead = 4;    // helpers claim chunks >= (chain's current chunk) + kHelpLead
constexpr int kHelpSlots = 7;   // ring slots per chain (> kHelpLead + 1)
constexpr size_t kHelpPackageBytes = 66048;   // 32768 + 16384 + 8192 + 8192 + 512
constexpr size_t kHelpSlotStride = 66560;     // 1024-byte aligned slots
struct HelpRing {
  int32_t *cons_pos;    // [chains] chunk each chain CTA has started (n_chunks when done)
  int32_t *next_claim;  // [chains] lowest chunk no helper has claimed yet
  int32_t *flag;        // [chains * kHelpSlots] chunk + 1 of the package a slot holds, 0: none
  int32_t *busy;        // [chains * kHelpSlots] chunk + 1 of the helper writing a slot, 0: free
  int32_t *finished;    // chain CTAs that have finished
  unsigned char *ring;  // [chains * kHelpSlots] package slots
  int32_t n_chains;     // chain CTAs; blocks beyond them are helpers
};
// Bytes of the helper header (cons_pos, next_claim, flag, busy, counter), 1024-aligned.
inline size_t help_header_bytes(int64_t chains) {
  const size_t words = (size_t)chains * (2 + 2 * kHelpSlots) + 1;
  return (words * sizeof(int32_t) + 1023) / 1024 * 1024;
}

// Arguments common to the prefill launchers.
struct ChunkArgs {
  const void *q, *k, *v;
  const float *log_alpha, *beta, *init_state;
  const int32_t *cu_seqlens;  // device pointer (validated in-kernel)
  int32_t n_seqs;
  int64_t n_tokens;
  int32_t H;
  void *out;
  float *final_state;
  DeviceStatus *status;
  // Helper workspace (header then ring) for the bf16 prefill, or nullptr; its
  // header must be zeroed before each launch.
  unsigned char *help_ws;
  int32_t n_help;  // helper CTAs to launch beside the chains (0: none)
  // kTransitions (bf16 only): first pass of an in-device split.  Every chain runs
  // twice without writing outputs: from a zero state (final state -> final_state,
  // the segment's B) and from the identity with v = 0 (final state ->
  // final_state_m, the segment's transition M).  init_state is ignored.
  enum Mode { kPlain = 0, kTransitions = 2 };
  int32_t mode = kPlain;
  float *final_state_m = nullptr;
  // Scratch of n_seqs int32 (or nullptr): the bf16 prefill then runs the
  // sequences longest first.
  int32_t *seq_order = nullptr;
  // kTransitions: the zero-start runs write their outputs to out and the
  // transition runs theirs (M_t^T q_t) to out_m ([N, H, 128] bf16); with
  // out_m NULL the transition runs write to out as well.  With write_out false
  // no output is written at all (out is then only a valid tensor-map base).
  void *out_m = nullptr;
  bool write_out = true;
  // kTransitions: with K >= 2, the chains are sequences of K segments each whose
  // first segment starts from a zero state, so it gets no transition run (its
  // M_0 and out_m rows are not written).  0: every chain gets one.
  int32_t split_skip_k = 0;
  // Test control in the status block (kPlain launches of the bf16 kernel), or nullptr.
  TestControl *test_control = nullptr;
};

cudaError_t launch_decode_step(float *state, const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, int32_t B, int32_t H,
                               bool bf16, void *out, cudaStream_t stream);

cudaError_t launch_decode_replay(float *state, const void *q, const void *k, const void *v,
                                 const float *log_alpha, const float *beta,
                                 const int32_t *n_accept, int32_t B, int32_t T, int32_t H,
                                 bool bf16, void *out, cudaStream_t stream);

cudaError_t launch_prep(const void *q_raw, const void *k_raw, const void *v_raw,
                        const float *conv_w, const float *a_logit, const float *b_logit,
                        const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t H,
                        bool bf16, void *q, void *k, void *v, float *log_alpha, float *beta,
                        cudaStream_t stream);

// kda_prep_fwd with a carried convolution window (win_in may be NULL: zeros;
// win_out may be NULL: not written; both [n_seqs, 3, 3, H, 128] dtype, and may
// be the same array).
cudaError_t launch_prep_window(const void *q_raw, const void *k_raw, const void *v_raw,
                               const float *conv_w, const float *a_logit, const float *b_logit,
                               const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens,
                               int32_t H, bool bf16, const void *win_in, void *win_out, void *q,
                               void *k, void *v, float *log_alpha, float *beta,
                               cudaStream_t stream);

cudaError_t launch_layer_replay(float *state, void *win, const void *q_raw, const void *k_raw,
                                const void *v_raw, const float *a_logit, const float *b_logit,
                                const void *g, const float *conv_w, const float *gamma,
                                const int32_t *n_accept, int32_t B, int32_t T, int32_t H,
                                bool bf16, void *out, cudaStream_t stream);

// Backward pass (kda_chunk_bwd).  Workspace pieces are device pointers.
struct BwdArgs {
  const void *q, *k, *v;
  const float *log_alpha, *beta, *init_state;
  const int32_t *cu_seqlens;  // device
  int32_t n_seqs;
  int64_t n_tokens;
  int32_t H;
  bool bf16;
  const void *d_out;
  const float *d_final;       // or nullptr
  void *dq, *dk, *dv;
  float *d_log_alpha, *d_beta, *d_init;  // d_init may be nullptr
  int32_t ckpt_every;         // tokens between stored states: a power of two in [4, 1024]
  bool chunked;               // bf16 only: the chunked tensor-core pass (ckpt_every == kBwdChunk)
  // workspace
  float *ckpt;                // [bwd_ckpt_slots][H][128][128] fp32 (chunked pass: bf16)
  float *dq_acc, *dk_acc;     // [n_tokens][H][128], zeroed
  DeviceStatus *status;
};
// Tokens per chunk of the chunked (tensor-core) backward pass, which takes its
// states every kBwdChunk tokens, stored as bf16 (bytes per element).
constexpr int32_t kBwdChunk = 16;
constexpr size_t kBwdChunkStateBytes = 2;
// Checkpoint slot of the first state of sequence s (states every `every`
// tokens from its start): floor(cu[s] / every) + s.  Consecutive sequences never
// share slots, since floor(b / c) - floor(a / c) + 1 >= ceil((b - a) / c).
__host__ __device__ inline int64_t bwd_ckpt_slot_base(int64_t cu_s, int64_t s, int32_t every) {
  return cu_s / every + s;
}
// Checkpoint interval bounds of the backward pass, and the budget its default
// interval keeps the stored states within.
constexpr int32_t kMaxCkptEvery = 1024;
constexpr size_t kCkptBudgetBytes = (size_t)16 << 30;
// Checkpoint slots the backward pass needs with states stored every `every` tokens.
size_t bwd_ckpt_slots(int32_t n_seqs, int64_t n_tokens, int32_t every);
// The default interval: the smallest power of two >= 4 whose checkpoints fit
// kCkptBudgetBytes (kMaxCkptEvery if none does).
int32_t bwd_ckpt_every(int32_t n_seqs, int64_t n_tokens, int32_t H);
cudaError_t launch_chunk_bwd(const BwdArgs &a, cudaStream_t stream);
// The chunked pass proper (after the checkpoints), and its shared memory.
cudaError_t launch_bwd_chunk(const BwdArgs &a, cudaStream_t stream);
size_t bwd_chunk_smem_bytes();

cudaError_t launch_post(const void *o, const void *g, const float *gamma, int64_t n_tokens,
                        int32_t H, bool bf16, void *out, cudaStream_t stream);

cudaError_t launch_chunk_fwd_f32(const ChunkArgs &a, cudaStream_t stream);

// Returns cudaErrorNotSupported if the tensor-map entry point is unavailable.
cudaError_t launch_chunk_fwd_bf16_tc(const ChunkArgs &a, cudaStream_t stream);

// In-device split of every sequence into K segments (K >= 2; bf16): scratch of
// split_workspace_bytes() at `ws` (1024-byte aligned); a.help_ws is ignored.
size_t split_workspace_bytes(int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t K);
// Composition of affine state maps: for each (sequence s, head), S_0 = init
// (zeros if NULL), S_{j+1} = M[s K + j] S_j + B[s K + j]; start[s K + j] = S_j
// for j < K and end[s] = S_K, each when non-null.  States [., H, 128, 128] fp32.
cudaError_t launch_state_combine(const float *init, const float *B, const float *M,
                                 int32_t n_seqs, int32_t K, int32_t H, float *start, float *end,
                                 cudaStream_t stream);
cudaError_t launch_chunk_fwd_split(const ChunkArgs &a, int32_t K, unsigned char *ws,
                                   cudaStream_t stream);

}  // namespace kda
