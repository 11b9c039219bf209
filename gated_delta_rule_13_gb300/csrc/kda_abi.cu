// C ABI of libkda: argument validation (the error boundary), workspace layout,
// and dispatch to the kernels.  See include/kda.h for the contract.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

using kda::kHeadDim;
using kda::kStatusBytes;

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool aligned16(const void *p) { return aligned(p, 16); }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int check_dims(int32_t dk, int32_t dv, int dtype) {
  if (dk <= 0 || dv <= 0) return KDA_ERR_INVALID_ARG;
  if (dk != kHeadDim || dv != kHeadDim) return KDA_ERR_UNSUPPORTED;
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

// Status block and the device copy of a host cu_seqlens array.
size_t base_workspace_bytes(int32_t n_seqs) {
  return kStatusBytes + round_up(sizeof(int32_t) * ((size_t)n_seqs + 1), 256);
}

// Helper CTAs for a bf16 prefill of `chains` chains on the current device: the
// SMs the chains leave idle, when they are at least four times as many as the
// chains.  With fewer, the helpers cover too few chunks to repay what the
// protocol costs the chain CTAs (measured on a GB300 with 152 SMs: 8 chains
// 1.22x faster, 24 chains 1.06x, 32 chains 0.97x, 96 chains 0.78x).  A
// non-negative `cap` (the caller's max_helpers) caps the count; 0 turns helpers off.
int32_t help_ctas(int64_t chains, int dtype, int32_t cap = -1) {
  if (dtype != KDA_BF16 || chains <= 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int64_t n = sms - chains < 4 * chains ? 0 : sms - chains;
  if (cap >= 0 && cap < n) n = cap;
  return n > 0 ? (int32_t)n : 0;
}

// Segments per sequence for the in-device split of a bf16 prefill (0: no
// split).  Its pass runs 2 K CTAs per chain, or 2 K - 1 for a call without an
// initial state (the first segment then needs no transition run), and takes
// about T / K chunk-steps (plus a combine and an output correction), so it needs
// (2 K or 2 K - 1) x chains <= SMs and pays off from K = 2 on; segments are kept
// at two chunks or more on average.  A non-negative `cap` (the caller's
// max_split) caps K; 0 turns the split off.
int32_t split_factor(int32_t n_seqs, int64_t n_tokens, int32_t H, int dtype, bool zero_init,
                     int32_t cap = -1) {
  const int64_t chains = (int64_t)n_seqs * H;
  if (dtype != KDA_BF16 || chains <= 0 || n_tokens <= 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  // 2 K C blocks in the first pass, or (2 K - 1) C without an initial state
  int64_t k = zero_init ? (sms + chains) / (2 * chains) : sms / (2 * chains);
  const int64_t by_length = n_tokens / ((int64_t)n_seqs * 2 * kda::kChunk);
  if (by_length < k) k = by_length;
  if (cap >= 0 && cap < k) k = cap;
  return k >= 2 ? (int32_t)k : 0;
}

size_t help_workspace_bytes(int64_t chains) {
  return kda::help_header_bytes(chains) + (size_t)chains * kda::kHelpSlots * kda::kHelpSlotStride;
}

// The sequence order of a bf16 prefill of several sequences (longest first).
size_t order_bytes(int32_t n_seqs, int dtype) {
  return (dtype == KDA_BF16 && n_seqs > 1) ? round_up(sizeof(int32_t) * (size_t)n_seqs, 1024) : 0;
}

// Full workspace: the base part, the sequence order, then the larger of the
// scratch of the in-device split (without an initial state: the most segments)
// and the helper header and ring, so that any schedule a caller picks fits.
size_t workspace_bytes_for(int32_t n_seqs, int64_t n_tokens, int32_t H, int dtype) {
  const int64_t chains = (int64_t)n_seqs * H;
  size_t b = base_workspace_bytes(n_seqs) + order_bytes(n_seqs, dtype);
  const int32_t k_zero = split_factor(n_seqs, n_tokens, H, dtype, true);
  size_t extra = k_zero > 0 ? kda::split_workspace_bytes(n_seqs, n_tokens, H, k_zero) : 0;
  if (help_ctas(chains, dtype) > 0 && help_workspace_bytes(chains) > extra)
    extra = help_workspace_bytes(chains);
  return b + extra;
}

// True when `p` is memory the device can read directly as a device array.
bool is_device_pointer(const void *p, bool *ok) {
  cudaPointerAttributes attr;
  memset(&attr, 0, sizeof(attr));
  const cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *ok = false;
    return false;
  }
  *ok = true;
  return attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged;
}

// The backward pass's schedule: its checkpoint interval and which pass runs.
// The caller's interval (a power of two in [4, kda::kMaxCkptEvery]) selects the
// token-loop pass with that interval.  0 leaves the choice to the library: for
// bf16 the chunked tensor-core pass (states every kda::kBwdChunk tokens) when
// those states fit kda::kCkptBudgetBytes, else, and for fp32, the token-loop
// pass with kda::bwd_ckpt_every's interval.  every < 0: invalid.
struct BwdPlan {
  int32_t every;
  bool chunked;
};
BwdPlan bwd_plan(int32_t want, int32_t n_seqs, int64_t n_tokens, int32_t H, int dtype) {
  if (want != 0) {
    if (want < 4 || want > kda::kMaxCkptEvery || (want & (want - 1)) != 0) return {-1, false};
    return {want, false};
  }
  if (dtype == KDA_BF16 &&
      kda::bwd_ckpt_slots(n_seqs, n_tokens, kda::kBwdChunk) * (size_t)H * kHeadDim * kHeadDim *
              kda::kBwdChunkStateBytes <= kda::kCkptBudgetBytes)
    return {kda::kBwdChunk, true};
  return {kda::bwd_ckpt_every(n_seqs, n_tokens, H), false};
}

// Backward-pass workspace: status block, device copy of a host cu_seqlens, the
// state checkpoints (fp32, or bf16 for the chunked pass), and (token-loop pass
// only) the fp32 accumulators of dq and dk.
struct BwdLayout {
  size_t cu, ckpt, dq, dk, total;
};
BwdLayout bwd_layout(int32_t n_seqs, int64_t n_tokens, int32_t H, BwdPlan plan) {
  BwdLayout l;
  l.cu = kStatusBytes;
  l.ckpt = l.cu + round_up(sizeof(int32_t) * ((size_t)n_seqs + 1), 256);
  const size_t state_elem = plan.chunked ? kda::kBwdChunkStateBytes : sizeof(float);
  l.dq = l.ckpt + round_up(kda::bwd_ckpt_slots(n_seqs, n_tokens, plan.every) * H * kHeadDim *
                               kHeadDim * state_elem,
                           256);
  const size_t acc = plan.chunked ? 0 : round_up((size_t)n_tokens * H * kHeadDim * 4, 256);
  l.dk = l.dq + acc;
  l.total = l.dk + acc;
  return l;
}

}  // namespace

extern "C" {

int kda_chunk_bwd_workspace_size_sched(int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk,
                                       int32_t dv, int dtype, int32_t ckpt_every, size_t *bytes) {
  if (!bytes || n_seqs < 0 || n_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  const BwdPlan plan = bwd_plan(ckpt_every, n_seqs, n_tokens, H, dtype);
  if (plan.every < 0) return KDA_ERR_INVALID_ARG;
  *bytes = bwd_layout(n_seqs, n_tokens, H, plan).total;
  return KDA_OK;
}

int kda_chunk_bwd_workspace_size(int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk,
                                 int32_t dv, int dtype, size_t *bytes) {
  return kda_chunk_bwd_workspace_size_sched(n_seqs, n_tokens, H, dk, dv, dtype, 0, bytes);
}

int kda_chunk_bwd_sched(const void *q, const void *k, const void *v, const float *log_alpha,
                        const float *beta, const float *init_state, const int32_t *cu_seqlens,
                        int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv,
                        int dtype, const void *d_out, const float *d_final_state, void *dq,
                        void *dk_, void *dv_, float *d_log_alpha, float *d_beta,
                        float *d_init_state, int32_t ckpt_every, void *workspace,
                        size_t workspace_bytes, void *stream) {
  if (n_seqs < 0 || n_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  const BwdPlan plan = bwd_plan(ckpt_every, n_seqs, n_tokens, H, dtype);
  if (plan.every < 0) return KDA_ERR_INVALID_ARG;
  if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !d_out || !dq || !dk_ || !dv_ ||
                       !d_log_alpha || !d_beta))
    return KDA_ERR_INVALID_ARG;
  if ((int64_t)n_seqs * H * 4 > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  const size_t esz = dtype == KDA_BF16 ? 2 : 4;
  // q, k, v, log_alpha and d_out rows are fetched by 16-byte asynchronous copies
  const void *rows[] = {q, k, v, log_alpha, d_out};
  for (const void *p : rows)
    if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
  const void *elem[] = {dq, dk_, dv_};
  for (const void *p : elem)
    if (p && !aligned(p, esz)) return KDA_ERR_INVALID_ARG;
  const void *f32[] = {beta, init_state, d_final_state, d_log_alpha, d_beta, d_init_state};
  for (const void *p : f32)
    if (p && !aligned(p, 4)) return KDA_ERR_INVALID_ARG;
  // no output may overlap an input or another output
  const size_t nt = (size_t)n_tokens * H;
  const size_t sb = (size_t)n_seqs * H * dk * dv * 4;
  const void *outs[] = {dq, dk_, dv_, d_log_alpha, d_beta, d_init_state};
  const size_t out_b[] = {nt * dk * esz, nt * dk * esz, nt * dv * esz, nt * dk * 4, nt * 4, sb};
  const void *ins[] = {q, k, v, log_alpha, beta, init_state, d_out, d_final_state};
  const size_t in_b[] = {nt * dk * esz, nt * dk * esz, nt * dv * esz, nt * dk * 4, nt * 4, sb,
                         nt * dv * esz, sb};
  for (int i = 0; i < 6; ++i) {
    if (!outs[i] || out_b[i] == 0) continue;
    for (int j = 0; j < 8; ++j)
      if (ins[j] && in_b[j] > 0 && ranges_overlap(outs[i], out_b[i], ins[j], in_b[j]))
        return KDA_ERR_INVALID_ARG;
    for (int j = i + 1; j < 6; ++j)
      if (outs[j] && out_b[j] > 0 && ranges_overlap(outs[i], out_b[i], outs[j], out_b[j]))
        return KDA_ERR_INVALID_ARG;
  }
  const BwdLayout lay = bwd_layout(n_seqs, n_tokens, H, plan);
  if (!workspace || workspace_bytes < lay.total || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  bool attr_ok = false;
  const bool cu_on_device = is_device_pointer(cu_seqlens, &attr_ok);
  if (!attr_ok) return KDA_ERR_CUDA;
  const int32_t *cu_dev = cu_seqlens;
  if (!cu_on_device) {
    if (cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != n_tokens) return KDA_ERR_INVALID_ARG;
    for (int32_t s = 0; s < n_seqs; ++s)
      if (cu_seqlens[s + 1] < cu_seqlens[s]) return KDA_ERR_INVALID_ARG;
    int32_t *dst = reinterpret_cast<int32_t *>(ws + lay.cu);
    if (cudaMemcpyAsync(dst, cu_seqlens, sizeof(int32_t) * ((size_t)n_seqs + 1),
                        cudaMemcpyHostToDevice, st) != cudaSuccess) {
      cudaGetLastError();
      return KDA_ERR_CUDA;
    }
    cu_dev = dst;
  }
  kda::DeviceStatus *status = reinterpret_cast<kda::DeviceStatus *>(ws);
  // the token-loop pass adds into its accumulators and into d_log_alpha and
  // d_beta; the chunked pass writes every element once
  const bool ok = cudaMemsetAsync(status, 0, sizeof(kda::DeviceStatus), st) == cudaSuccess &&
                  (nt == 0 || plan.chunked ||
                   (cudaMemsetAsync(ws + lay.dq, 0, lay.total - lay.dq, st) == cudaSuccess &&
                    cudaMemsetAsync(d_log_alpha, 0, nt * dk * 4, st) == cudaSuccess &&
                    cudaMemsetAsync(d_beta, 0, nt * 4, st) == cudaSuccess));
  if (!ok) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  if (n_seqs == 0) return KDA_OK;
  kda::BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.init_state = init_state;
  a.cu_seqlens = cu_dev; a.n_seqs = n_seqs; a.n_tokens = n_tokens; a.H = H;
  a.bf16 = dtype == KDA_BF16;
  a.d_out = d_out; a.d_final = d_final_state;
  a.dq = dq; a.dk = dk_; a.dv = dv_; a.d_log_alpha = d_log_alpha; a.d_beta = d_beta;
  a.d_init = d_init_state;
  a.ckpt_every = plan.every;
  a.chunked = plan.chunked;
  a.ckpt = reinterpret_cast<float *>(ws + lay.ckpt);
  a.dq_acc = reinterpret_cast<float *>(ws + lay.dq);
  a.dk_acc = reinterpret_cast<float *>(ws + lay.dk);
  a.status = status;
  const cudaError_t e = kda::launch_chunk_bwd(a, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

int kda_chunk_bwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  const float *beta, const float *init_state, const int32_t *cu_seqlens,
                  int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv, int dtype,
                  const void *d_out, const float *d_final_state, void *dq, void *dk_, void *dv_,
                  float *d_log_alpha, float *d_beta, float *d_init_state, void *workspace,
                  size_t workspace_bytes, void *stream) {
  return kda_chunk_bwd_sched(q, k, v, log_alpha, beta, init_state, cu_seqlens, n_seqs, n_tokens,
                             H, dk, dv, dtype, d_out, d_final_state, dq, dk_, dv_, d_log_alpha,
                             d_beta, d_init_state, 0, workspace, workspace_bytes, stream);
}

const char *kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported head size or dtype";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing or too small";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime or launch failure";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded in-kernel wait gave up";
    default: return "KDA: unknown status";
  }
}

int kda_version(void) { return kVersion; }

int kda_chunk_fwd_workspace_size(int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk,
                                 int32_t dv, int dtype, size_t *bytes) {
  if (!bytes || n_seqs < 0 || n_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  *bytes = workspace_bytes_for(n_seqs, n_tokens, H, dtype);
  return KDA_OK;
}

int kda_chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  const float *beta, const float *init_state, const int32_t *cu_seqlens,
                  int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv,
                  int dtype, void *out, float *final_state, void *workspace,
                  size_t workspace_bytes, void *stream) {
  return kda_chunk_fwd_sched(q, k, v, log_alpha, beta, init_state, cu_seqlens, n_seqs, n_tokens,
                             H, dk, dv, dtype, out, final_state, -1, -1, workspace,
                             workspace_bytes, stream);
}

int kda_chunk_fwd_sched(const void *q, const void *k, const void *v, const float *log_alpha,
                        const float *beta, const float *init_state, const int32_t *cu_seqlens,
                        int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv,
                        int dtype, void *out, float *final_state, int32_t max_split,
                        int32_t max_helpers, void *workspace, size_t workspace_bytes,
                        void *stream) {
  // ---- host-side validation: nothing is launched unless all of it passes
  if (n_seqs < 0 || n_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !out)) return KDA_ERR_INVALID_ARG;
  if ((int64_t)n_seqs * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  // TMA-read tensors and states: 16 bytes; beta is read element-wise.
  const void *tensors[] = {q, k, v, log_alpha, init_state, out, final_state};
  for (const void *p : tensors)
    if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
  if (beta && !aligned(beta, 4)) return KDA_ERR_INVALID_ARG;
  const size_t state_bytes = (size_t)n_seqs * H * dk * dv * sizeof(float);
  if (init_state && final_state && state_bytes > 0 &&
      ranges_overlap(init_state, state_bytes, final_state, state_bytes))
    return KDA_ERR_INVALID_ARG;
  size_t need = base_workspace_bytes(n_seqs);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KDA_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool attr_ok = false;
  const bool cu_on_device = is_device_pointer(cu_seqlens, &attr_ok);
  if (!attr_ok) return KDA_ERR_CUDA;
  const int32_t *cu_dev = cu_seqlens;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  if (!cu_on_device) {
    // Host array: validate it here, then stage a device copy in the workspace.
    if (cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != n_tokens) return KDA_ERR_INVALID_ARG;
    for (int32_t s = 0; s < n_seqs; ++s)
      if (cu_seqlens[s + 1] < cu_seqlens[s]) return KDA_ERR_INVALID_ARG;
    int32_t *dst = reinterpret_cast<int32_t *>(ws + kStatusBytes);
    if (cudaMemcpyAsync(dst, cu_seqlens, sizeof(int32_t) * ((size_t)n_seqs + 1),
                        cudaMemcpyHostToDevice, st) != cudaSuccess) {
      cudaGetLastError();
      return KDA_ERR_CUDA;
    }
    cu_dev = dst;
  }
  kda::DeviceStatus *status = reinterpret_cast<kda::DeviceStatus *>(ws);
  if (cudaMemsetAsync(status, 0, sizeof(kda::DeviceStatus), st) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  if (n_seqs == 0) return KDA_OK;

  kda::ChunkArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta;
  a.init_state = init_state; a.cu_seqlens = cu_dev; a.n_seqs = n_seqs; a.n_tokens = n_tokens;
  a.H = H; a.out = out; a.final_state = final_state; a.status = status;
  a.help_ws = nullptr;
  a.n_help = 0;
  a.test_control = reinterpret_cast<kda::TestControl *>(ws + kda::kTestControlOffset);
  const int64_t chains = (int64_t)n_seqs * H;
  // Longest sequences first, when the workspace has room for their order.
  const size_t ob = order_bytes(n_seqs, dtype);
  if (ob > 0 && workspace_bytes >= need + ob) {
    a.seq_order = reinterpret_cast<int32_t *>(ws + need);
    need += ob;
  }
  // The in-device split, when it applies and the workspace has its scratch.
  const int32_t n_split =
      split_factor(n_seqs, n_tokens, H, dtype, init_state == nullptr, max_split);
  if (n_split > 0 && workspace_bytes >= need + kda::split_workspace_bytes(n_seqs, n_tokens, H, n_split)) {
    const cudaError_t e = kda::launch_chunk_fwd_split(a, n_split, ws + need, st);
    if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  }
  // Helpers run when the workspace has room for their ring (a workspace sized by
  // kda_chunk_fwd_workspace_size on this device does); their header starts zeroed.
  const int32_t n_help = help_ctas(chains, dtype, max_helpers);
  if (n_help > 0 && n_tokens > 0 && workspace_bytes >= need + help_workspace_bytes(chains)) {
    a.help_ws = ws + need;
    a.n_help = n_help;
    if (cudaMemsetAsync(a.help_ws, 0, kda::help_header_bytes(chains), st) != cudaSuccess) {
      cudaGetLastError();
      return KDA_ERR_CUDA;
    }
  }
  const cudaError_t e = dtype == KDA_BF16 ? kda::launch_chunk_fwd_bf16_tc(a, st)
                                          : kda::launch_chunk_fwd_f32(a, st);
  if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_read_device_status(void *workspace, void *stream, int clear, int32_t *device_status) {
  if (!workspace || !device_status) return KDA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  kda::DeviceStatus host;
  if (cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemcpy(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  if (clear && cudaMemset(workspace, 0, sizeof(host)) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  *device_status = host.code;
  return KDA_OK;
}

int kda_read_device_status_detail(void *workspace, void *stream, int clear,
                                  int32_t *detail4) {
  if (!workspace || !detail4) return KDA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  kda::DeviceStatus host;
  if (cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemcpy(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  if (clear && cudaMemset(workspace, 0, sizeof(host)) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  detail4[0] = host.code;
  detail4[1] = host.detail;
  detail4[2] = host.chain;
  detail4[3] = host.chunk;
  return KDA_OK;
}

int kda_test_arm_timeout(void *workspace, int32_t chain, int32_t chunk, uint32_t wait_us,
                         void *stream) {
  if (!workspace || !aligned16(workspace)) return KDA_ERR_INVALID_ARG;
  kda::TestControl c;
  memset(&c, 0, sizeof(c));
  if (chain >= 0) {
    if (chunk < 0 || wait_us < 1 || wait_us > 2000000) return KDA_ERR_INVALID_ARG;
    c.magic0 = kda::kTestMagic0;
    c.magic1 = kda::kTestMagic1;
    c.chain = chain;
    c.chunk = chunk;
    c.wait_us = wait_us;
  }
  unsigned char *dst = static_cast<unsigned char *>(workspace) + kda::kTestControlOffset;
  if (cudaMemcpyAsync(dst, &c, sizeof(c), cudaMemcpyHostToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

int kda_chunk_fwd_transitions(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta,
                              const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens,
                              int32_t H, int32_t dk, int32_t dv, int dtype, float *state_b,
                              float *state_m, void *workspace, size_t workspace_bytes,
                              void *stream) {
  if (n_seqs < 0 || n_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  if (dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
  if (!cu_seqlens || !state_b || !state_m) return KDA_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!q || !k || !v || !log_alpha || !beta)) return KDA_ERR_INVALID_ARG;
  if ((int64_t)n_seqs * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  const void *tensors[] = {q, k, v, log_alpha, state_b, state_m};
  for (const void *p : tensors)
    if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
  if (beta && !aligned(beta, 4)) return KDA_ERR_INVALID_ARG;
  const size_t state_bytes = (size_t)n_seqs * H * dk * dv * sizeof(float);
  if (state_bytes > 0 && ranges_overlap(state_b, state_bytes, state_m, state_bytes))
    return KDA_ERR_INVALID_ARG;
  const size_t need = base_workspace_bytes(n_seqs);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool attr_ok = false;
  const bool cu_on_device = is_device_pointer(cu_seqlens, &attr_ok);
  if (!attr_ok) return KDA_ERR_CUDA;
  const int32_t *cu_dev = cu_seqlens;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  if (!cu_on_device) {
    if (cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != n_tokens) return KDA_ERR_INVALID_ARG;
    for (int32_t s = 0; s < n_seqs; ++s)
      if (cu_seqlens[s + 1] < cu_seqlens[s]) return KDA_ERR_INVALID_ARG;
    int32_t *dst = reinterpret_cast<int32_t *>(ws + kStatusBytes);
    if (cudaMemcpyAsync(dst, cu_seqlens, sizeof(int32_t) * ((size_t)n_seqs + 1),
                        cudaMemcpyHostToDevice, st) != cudaSuccess) {
      cudaGetLastError();
      return KDA_ERR_CUDA;
    }
    cu_dev = dst;
  }
  kda::DeviceStatus *status = reinterpret_cast<kda::DeviceStatus *>(ws);
  if (cudaMemsetAsync(status, 0, sizeof(kda::DeviceStatus), st) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  if (n_seqs == 0) return KDA_OK;
  kda::ChunkArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta;
  a.init_state = nullptr; a.cu_seqlens = cu_dev; a.n_seqs = n_seqs; a.n_tokens = n_tokens;
  a.H = H;
  a.out = const_cast<void *>(q);  // a valid tensor map base; this pass writes no outputs
  a.final_state = state_b; a.status = status;
  a.help_ws = nullptr; a.n_help = 0;
  a.mode = kda::ChunkArgs::kTransitions;
  a.final_state_m = state_m;
  a.write_out = false;
  const cudaError_t e = kda::launch_chunk_fwd_bf16_tc(a, st);
  if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_state_combine(const float *init_state, const float *state_b, const float *state_m,
                      int32_t n_seqs, int32_t n_segments, int32_t H, int32_t dk, int32_t dv,
                      float *start_states, float *end_state, void *stream) {
  if (n_seqs < 0 || n_segments < 1 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, KDA_F32);
  if (d != KDA_OK) return d;
  if (!state_b || !state_m) return KDA_ERR_INVALID_ARG;
  if ((int64_t)n_seqs * n_segments * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  const void *tensors[] = {init_state, state_b, state_m, start_states, end_state};
  for (const void *p : tensors)
    if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
  const size_t one = (size_t)H * dk * dv * sizeof(float);
  const size_t seg = one * n_seqs * n_segments, seqs = one * n_seqs;
  // the outputs may not overlap any input, nor each other
  const void *ins[] = {init_state, state_b, state_m};
  const size_t in_bytes[] = {seqs, seg, seg};
  for (int i = 0; i < 3; ++i) {
    if (!ins[i] || seqs == 0) continue;
    if (start_states && ranges_overlap(start_states, seg, ins[i], in_bytes[i]))
      return KDA_ERR_INVALID_ARG;
    if (end_state && ranges_overlap(end_state, seqs, ins[i], in_bytes[i]))
      return KDA_ERR_INVALID_ARG;
  }
  if (start_states && end_state && seqs > 0 && ranges_overlap(start_states, seg, end_state, seqs))
    return KDA_ERR_INVALID_ARG;
  const cudaError_t e = kda::launch_state_combine(init_state, state_b, state_m, n_seqs,
                                                  n_segments, H, start_states, end_state,
                                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_read_chunk_stats(void *workspace, void *stream, int32_t *help_published,
                         int32_t *help_consumed) {
  if (!workspace || !help_published || !help_consumed) return KDA_ERR_INVALID_ARG;
  kda::DeviceStatus host;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaMemcpy(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  *help_published = host.help_published;
  *help_consumed = host.help_consumed;
  return KDA_OK;
}

int kda_decode_step(float *state, const void *q, const void *k, const void *v,
                    const float *log_alpha, const float *beta, int32_t B, int32_t H,
                    int32_t dk, int32_t dv, int dtype, void *out, void *stream) {
  if (B < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  if (!state || !q || !k || !v || !log_alpha || !beta || !out) return KDA_ERR_INVALID_ARG;
  const size_t units = (size_t)B * H;
  const size_t esz = dtype == KDA_BF16 ? 2 : 4;
  // state: float4 accesses; v and out: 4-element vectors; the rest element-wise.
  if (!aligned16(state) || !aligned(v, 4 * esz) || !aligned(out, 4 * esz) || !aligned(q, esz) ||
      !aligned(k, esz) || !aligned(log_alpha, 4) || !aligned(beta, 4))
    return KDA_ERR_INVALID_ARG;
  if (units > 0 && ranges_overlap(state, units * dk * dv * sizeof(float), out, units * dv * esz))
    return KDA_ERR_INVALID_ARG;
  const cudaError_t e = kda::launch_decode_step(state, q, k, v, log_alpha, beta, B, H,
                                                dtype == KDA_BF16, out,
                                                static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

int kda_decode_replay(float *state, const void *q, const void *k, const void *v,
                      const float *log_alpha, const float *beta, const int32_t *n_accept,
                      int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, int dtype,
                      void *out, void *stream) {
  if (B < 0 || T <= 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  if (!state || !q || !k || !v || !log_alpha || !beta || !n_accept) return KDA_ERR_INVALID_ARG;
  const size_t esz = dtype == KDA_BF16 ? 2 : 4;
  // q, k, v and log_alpha rows are fetched by bulk copies: 16-byte aligned bases
  if (!aligned16(state) || !aligned16(v) || (out && !aligned(out, 4 * esz)) || !aligned16(q) ||
      !aligned16(k) || !aligned16(log_alpha) || !aligned(beta, 4) || !aligned(n_accept, 4))
    return KDA_ERR_INVALID_ARG;
  const size_t units = (size_t)B * H;
  if (out && units > 0 &&
      ranges_overlap(state, units * dk * dv * sizeof(float), out, units * (size_t)T * dv * esz))
    return KDA_ERR_INVALID_ARG;
  const cudaError_t e = kda::launch_decode_replay(state, q, k, v, log_alpha, beta, n_accept, B, T,
                                                  H, dtype == KDA_BF16, out,
                                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

int kda_prep_fwd(const void *q_raw, const void *k_raw, const void *v_raw, const float *conv_w,
                 const float *a_logit, const float *b_logit, const int32_t *cu_seqlens,
                 int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk, int32_t dv, int dtype,
                 void *q, void *k, void *v, float *log_alpha, float *beta, void *stream) {
  if (n_seqs < 1 || n_tokens < 0 || n_tokens > 0x7fffffffLL || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  if (!q_raw || !k_raw || !v_raw || !conv_w || !a_logit || !b_logit || !cu_seqlens || !q || !k ||
      !v || !log_alpha || !beta)
    return KDA_ERR_INVALID_ARG;
  const size_t esz = dtype == KDA_BF16 ? 2 : 4;
  const void *vec[] = {q_raw, k_raw, v_raw, q, k, v};
  for (const void *p : vec)
    if (!aligned(p, 4 * esz)) return KDA_ERR_INVALID_ARG;
  if (!aligned16(conv_w) || !aligned16(a_logit) || !aligned16(log_alpha) || !aligned(b_logit, 4) ||
      !aligned(beta, 4) || !aligned(cu_seqlens, 4))
    return KDA_ERR_INVALID_ARG;
  // The convolution reads neighbouring tokens: no output may overlap an input.
  const size_t n = (size_t)n_tokens * H * dk;
  const void *outs[] = {q, k, v};
  const void *ins[] = {q_raw, k_raw, v_raw};
  for (const void *o : outs)
    for (const void *i : ins)
      if (n > 0 && ranges_overlap(o, n * esz, i, n * esz)) return KDA_ERR_INVALID_ARG;
  if (n > 0 && (ranges_overlap(log_alpha, n * 4, a_logit, n * 4) ||
                ranges_overlap(beta, (size_t)n_tokens * H * 4, b_logit, (size_t)n_tokens * H * 4)))
    return KDA_ERR_INVALID_ARG;
  const cudaError_t e = kda::launch_prep(q_raw, k_raw, v_raw, conv_w, a_logit, b_logit,
                                         cu_seqlens, n_seqs, n_tokens, H, dtype == KDA_BF16, q, k,
                                         v, log_alpha, beta, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

int kda_prep_fwd_state(const void *q_raw, const void *k_raw, const void *v_raw,
                       const float *conv_w, const float *a_logit, const float *b_logit,
                       const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t H,
                       int32_t dk, int32_t dv, int dtype, const void *conv_state_in,
                       void *conv_state_out, void *q, void *k, void *v, float *log_alpha,
                       float *beta, void *stream) {
  if (n_seqs < 1 || n_tokens < 0 || n_tokens > 0x7fffffffLL || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  if (!q_raw || !k_raw || !v_raw || !conv_w || !a_logit || !b_logit || !cu_seqlens || !q || !k ||
      !v || !log_alpha || !beta)
    return KDA_ERR_INVALID_ARG;
  const size_t esz = dtype == KDA_BF16 ? 2 : 4;
  const void *vec[] = {q_raw, k_raw, v_raw, q, k, v, conv_state_in, conv_state_out};
  for (const void *p : vec)
    if (p && !aligned(p, 4 * esz)) return KDA_ERR_INVALID_ARG;
  if (!aligned16(conv_w) || !aligned16(a_logit) || !aligned16(log_alpha) || !aligned(b_logit, 4) ||
      !aligned(beta, 4) || !aligned(cu_seqlens, 4))
    return KDA_ERR_INVALID_ARG;
  const size_t n = (size_t)n_tokens * H * dk;
  const void *outs[] = {q, k, v};
  const void *ins[] = {q_raw, k_raw, v_raw};
  for (const void *o : outs)
    for (const void *i : ins)
      if (n > 0 && ranges_overlap(o, n * esz, i, n * esz)) return KDA_ERR_INVALID_ARG;
  if (n > 0 && (ranges_overlap(log_alpha, n * 4, a_logit, n * 4) ||
                ranges_overlap(beta, (size_t)n_tokens * H * 4, b_logit, (size_t)n_tokens * H * 4)))
    return KDA_ERR_INVALID_ARG;
  // the window: 3 tensors x 3 rows x [H, 128] per sequence; in and out may be
  // the same array (updated in place) but may not overlap otherwise, nor touch
  // any input or output tensor
  const size_t wb = (size_t)n_seqs * 9 * H * dk * esz;
  if (conv_state_in && conv_state_out && conv_state_in != conv_state_out &&
      ranges_overlap(conv_state_in, wb, conv_state_out, wb))
    return KDA_ERR_INVALID_ARG;
  const void *wins[] = {conv_state_in, conv_state_out};
  const void *tens[] = {q_raw, k_raw, v_raw, q, k, v};
  for (const void *w : wins) {
    if (!w) continue;
    for (const void *t : tens)
      if (n > 0 && ranges_overlap(w, wb, t, n * esz)) return KDA_ERR_INVALID_ARG;
  }
  const cudaError_t e = kda::launch_prep_window(q_raw, k_raw, v_raw, conv_w, a_logit, b_logit,
                                                cu_seqlens, n_seqs, n_tokens, H, dtype == KDA_BF16,
                                                conv_state_in, conv_state_out, q, k, v, log_alpha,
                                                beta, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

int kda_layer_replay(float *state, void *conv_state, const void *q_raw, const void *k_raw,
                     const void *v_raw, const float *a_logit, const float *b_logit, const void *g,
                     const float *conv_w, const float *gamma, const int32_t *n_accept, int32_t B,
                     int32_t T, int32_t H, int32_t dk, int32_t dv, int dtype, void *out,
                     void *stream) {
  if (B < 0 || T <= 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dk, dv, dtype);
  if (d != KDA_OK) return d;
  if (!state || !conv_state || !q_raw || !k_raw || !v_raw || !a_logit || !b_logit || !g ||
      !conv_w || !gamma || !n_accept)
    return KDA_ERR_INVALID_ARG;
  const size_t esz = dtype == KDA_BF16 ? 2 : 4;
  // the window, taps and raw input rows are fetched by bulk copies: 16-byte aligned bases
  if (!aligned16(state) || !aligned16(conv_state) || !aligned16(q_raw) || !aligned16(k_raw) ||
      !aligned16(v_raw) || !aligned16(g) || !aligned16(a_logit) || !aligned(b_logit, 4) ||
      !aligned16(conv_w) || !aligned16(gamma) || !aligned(n_accept, 4) ||
      (out && !aligned(out, 4 * esz)))
    return KDA_ERR_INVALID_ARG;
  const size_t units = (size_t)B * H;
  const size_t sb = units * dk * dv * sizeof(float), wb = (size_t)B * 9 * H * dk * esz;
  if (units > 0 && ranges_overlap(state, sb, conv_state, wb)) return KDA_ERR_INVALID_ARG;
  if (out && units > 0) {
    const size_t ob = units * (size_t)T * dv * esz;
    if (ranges_overlap(out, ob, state, sb) || ranges_overlap(out, ob, conv_state, wb))
      return KDA_ERR_INVALID_ARG;
  }
  const cudaError_t e = kda::launch_layer_replay(state, conv_state, q_raw, k_raw, v_raw, a_logit,
                                                 b_logit, g, conv_w, gamma, n_accept, B, T, H,
                                                 dtype == KDA_BF16, out,
                                                 static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

int kda_post_fwd(const void *o, const void *g, const float *gamma, int64_t n_tokens, int32_t H,
                 int32_t dv, int dtype, void *out, void *stream) {
  if (n_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  const int d = check_dims(dv, dv, dtype);
  if (d != KDA_OK) return d;
  if (!o || !g || !gamma || !out) return KDA_ERR_INVALID_ARG;
  const size_t esz = dtype == KDA_BF16 ? 2 : 4;
  if (!aligned(o, 4 * esz) || !aligned(g, 4 * esz) || !aligned(out, 4 * esz) || !aligned16(gamma))
    return KDA_ERR_INVALID_ARG;
  const cudaError_t e = kda::launch_post(o, g, gamma, n_tokens, H, dtype == KDA_BF16, out,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

}  // extern "C"
