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
};

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

cudaError_t launch_post(const void *o, const void *g, const float *gamma, int64_t n_tokens,
                        int32_t H, bool bf16, void *out, cudaStream_t stream);

cudaError_t launch_chunk_fwd_f32(const ChunkArgs &a, cudaStream_t stream);

// Returns cudaErrorNotSupported if the tensor-map entry point is unavailable.
cudaError_t launch_chunk_fwd_bf16_tc(const ChunkArgs &a, cudaStream_t stream);

}  // namespace kda
