// In-device sequence parallelism for the bf16 prefill: when a call has so few
// (sequence, head) chains that most SMs would sit idle, every sequence is cut
// into K segments that run side by side, and their states are stitched
// together exactly ("Kimi K3: 架构、训练与系统全景解析", section 7.1: a segment
// maps the state it starts from to the one it ends with affinely,
// S_end = M S_start + B, and such maps compose; the pages use this for context
// parallelism across devices, and within one device to fill its SMs).
//
//   pass 1  one launch, 2 K chains per original chain, no outputs written:
//           segment j from S = 0          -> B_j (final state)
//           segment j from S = I, v = 0   -> M_j (final state = the product of
//                                            the segment's transitions)
//   combine S_0 = init,  S_{j+1} = M_j S_j + B_j            (fp32, per head)
//   pass 2  the plain kernel over all segments from S_j: outputs and final
//           states; the last segment's final state is the sequence's.
//
// Pass 1 runs 2 K x chains CTAs in one wave, pass 2 K x chains, so the wall
// time is about 2 T / K chunk-steps instead of T.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int D = kHeadDim;
constexpr int C = kChunk;

// seg_cu[s K + j] = start of segment j of sequence s: the sequence cut into K
// pieces of equal whole-chunk length (the last one shorter, trailing ones
// possibly empty); seg_cu[n_seqs K] = cu[n_seqs].  A malformed cu_seqlens gives
// a malformed seg_cu, which the prefill kernel then reports.
__global__ void kda_split_bounds_kernel(const int32_t *__restrict__ cu, int32_t n_seqs, int32_t K,
                                      int32_t *__restrict__ seg_cu) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n = (int64_t)n_seqs * K;
  if (i > n) return;
  if (i == n) {
    seg_cu[n] = cu[n_seqs];
    return;
  }
  const int s = (int)(i / K), j = (int)(i % K);
  const int64_t a = cu[s], len = (int64_t)cu[s + 1] - a;
  const int64_t chunks = len > 0 ? (len + C - 1) / C : 0;
  const int64_t per = (chunks + K - 1) / K * C;  // tokens per segment, whole chunks
  int64_t off = per * j;
  if (off > len) off = len > 0 ? len : 0;
  seg_cu[i] = (int32_t)(a + off);
}

// One CTA per (sequence, head, 32-column block of the state): the columns of
// S evolve independently under S <- M S + B.  start[s K + j] receives S_j
// (j < K) and end[s] the composed S_K, each when non-null.
constexpr int kCols = 32;
__global__ void __launch_bounds__(256, 1)
kda_split_combine_kernel(const float *__restrict__ init, const float *__restrict__ B,
               const float *__restrict__ M, int32_t n_seqs, int32_t K, int32_t H,
               float *__restrict__ start, float *__restrict__ end) {
  __shared__ float4 sbuf[2][D][kCols / 4];
  const int sh = blockIdx.x, s = sh / H, h = sh % H;
  const int col0 = kCols * blockIdx.y;
  const int t = threadIdx.x;
  const int row = t >> 1, c4 = (t & 1) * 4;  // row of S, first of this thread's 4 float4 columns
  auto blk = [=](int64_t seg) {  // offset of the [seg][h] 128 x 128 block
    return ((seg * H + h) * (int64_t)D) * D;
  };
  // S_0
  for (int i = t; i < D * kCols / 4; i += 256) {
    const int r = i / (kCols / 4), c = i % (kCols / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (init)
      v = *reinterpret_cast<const float4 *>(init + blk(s) + (int64_t)r * D + col0 + 4 * c);
    sbuf[0][r][c] = v;
  }
  __syncthreads();
  for (int j = 0;; ++j) {
    const int64_t seg = (int64_t)s * K + j;
    const int cur = j & 1;
    float *dst = j < K ? (start ? start + blk(seg) : nullptr) : (end ? end + blk(s) : nullptr);
    if (dst) {
      float4 *out = reinterpret_cast<float4 *>(dst + (int64_t)row * D + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) out[c4 + q] = sbuf[cur][row][c4 + q];
    }
    if (j == K || (j + 1 == K && !end)) break;
    // S_{j+1}[row][cols] = B_j[row][cols] + sum_k M_j[row][k] S_j[k][cols]
    const float *m = M + blk(seg) + (int64_t)row * D;
    const float4 *b = reinterpret_cast<const float4 *>(B + blk(seg) + (int64_t)row * D + col0);
    float4 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = b[c4 + q];
    for (int k = 0; k < D; k += 4) {
      const float4 mk = *reinterpret_cast<const float4 *>(m + k);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float mv = kk == 0 ? mk.x : kk == 1 ? mk.y : kk == 2 ? mk.z : mk.w;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 sv = sbuf[cur][k + kk][c4 + q];
          acc[q].x = fmaf(mv, sv.x, acc[q].x);
          acc[q].y = fmaf(mv, sv.y, acc[q].y);
          acc[q].z = fmaf(mv, sv.z, acc[q].z);
          acc[q].w = fmaf(mv, sv.w, acc[q].w);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) sbuf[cur ^ 1][row][c4 + q] = acc[q];
    __syncthreads();
  }
}

}  // namespace

size_t split_workspace_bytes(int32_t n_seqs, int32_t H, int32_t K) {
  const size_t nseg = (size_t)n_seqs * K;
  const size_t cu_bytes = ((nseg + 1) * sizeof(int32_t) + 1023) / 1024 * 1024;
  return cu_bytes + 3 * nseg * H * (size_t)D * D * sizeof(float);
}

cudaError_t launch_chunk_fwd_split(const ChunkArgs &a, int32_t K, unsigned char *ws,
                                   cudaStream_t stream) {
  const int64_t nseg = (int64_t)a.n_seqs * K;
  if (K < 2 || nseg > 0x7fffffffLL) return cudaErrorInvalidValue;
  const size_t cu_bytes = ((size_t)(nseg + 1) * sizeof(int32_t) + 1023) / 1024 * 1024;
  const size_t states = (size_t)nseg * a.H * D * D;
  int32_t *seg_cu = reinterpret_cast<int32_t *>(ws);
  float *B = reinterpret_cast<float *>(ws + cu_bytes), *M = B + states, *S = M + states;

  kda_split_bounds_kernel<<<(unsigned)((nseg + 1 + 255) / 256), 256, 0, stream>>>(
      a.cu_seqlens, a.n_seqs, K, seg_cu);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  ChunkArgs p = a;  // pass 1: every segment's B and M
  p.seq_order = nullptr;  // sized for the sequences, not the segments
  p.cu_seqlens = seg_cu;
  p.n_seqs = (int32_t)nseg;
  p.init_state = nullptr;
  p.final_state = B;
  p.final_state_m = M;
  p.mode = ChunkArgs::kTransitions;
  p.help_ws = nullptr;
  p.n_help = 0;
  e = launch_chunk_fwd_bf16_tc(p, stream);
  if (e != cudaSuccess) return e;

  kda_split_combine_kernel<<<dim3((unsigned)(a.n_seqs * a.H), D / kCols), 256, 0, stream>>>(
      a.init_state, B, M, a.n_seqs, K, a.H, S, nullptr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  p.init_state = S;  // pass 2: the outputs, from each segment's true start state
  p.final_state = B;
  p.final_state_m = nullptr;
  p.mode = ChunkArgs::kPlain;
  e = launch_chunk_fwd_bf16_tc(p, stream);
  if (e != cudaSuccess) return e;

  if (a.final_state) {  // the last segment's final state is the sequence's
    const size_t bytes = (size_t)a.H * D * D * sizeof(float);
    for (int32_t s = 0; s < a.n_seqs; ++s) {
      e = cudaMemcpyAsync(a.final_state + (size_t)s * a.H * D * D,
                          B + ((size_t)s * K + K - 1) * a.H * D * D, bytes,
                          cudaMemcpyDeviceToDevice, stream);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

cudaError_t launch_state_combine(const float *init, const float *B, const float *M,
                                 int32_t n_seqs, int32_t K, int32_t H, float *start, float *end,
                                 cudaStream_t stream) {
  if (n_seqs == 0 || H == 0) return cudaSuccess;
  if ((int64_t)n_seqs * H > 0x7fffffffLL) return cudaErrorInvalidValue;
  kda_split_combine_kernel<<<dim3((unsigned)(n_seqs * H), D / kCols), 256, 0, stream>>>(
      init, B, M, n_seqs, K, H, start, end);
  return cudaGetLastError();
}

}  // namespace kda
