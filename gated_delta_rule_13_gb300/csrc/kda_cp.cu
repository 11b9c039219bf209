// In-device sequence parallelism for the bf16 prefill: when a call has so few
// (sequence, head) chains that most SMs would sit idle, every sequence is cut
// into K segments that run side by side, and their states are stitched
// together exactly ("Kimi K3: 架构、训练与系统全景解析", section 7.1: a segment
// maps the state it starts from to the one it ends with affinely,
// S_end = M S_start + B, and such maps compose; the pages use this for context
// parallelism across devices, and within one device to fill its SMs).
//
//   pass 1  one launch, 2 K chains per original chain:
//           segment j from S = 0          -> B_j (final state), o0_t (outputs)
//           segment j from S = I, v = 0   -> M_j (final state = the product of
//                                            the segment's transitions) and
//                                            q_eff_t = M_t^T q_t (outputs)
//   combine S_0 = init,  S_{j+1} = M_j S_j + B_j            (fp32, per head);
//           S_K is the sequence's final state
//   correct o_t = o0_t + S_j^T q_eff_t   (S_t = M_t S_j + B_t, so
//           o_t = S_t^T q_t = o0_t + S_j^T M_t^T q_t)
//
// Pass 1 runs 2 K x chains CTAs in one wave (2 K - 1 per chain for a call without
// an initial state: the first segment needs no transition run), so the wall time
// is about T / K chunk-steps instead of T, plus the combine and the correction.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;
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

// One CTA per (sequence, head, 16-column block of the state): the columns of
// S evolve independently under S <- M S + B.  start[s K + j] receives S_j
// (j < K) and end[s] the composed S_K, each when non-null.
constexpr int kCols = 16;          // columns of S per CTA (columns evolve independently)
constexpr int kColQ = kCols / 8;   // float4 per thread: 2 threads per row
__global__ void __launch_bounds__(256, 1)
kda_split_combine_kernel(const float *__restrict__ init, const float *__restrict__ B,
               const float *__restrict__ M, int32_t n_seqs, int32_t K, int32_t H,
               float *__restrict__ start, float *__restrict__ end) {
  __shared__ float4 sbuf[2][D][kCols / 4];
  const int sh = blockIdx.x, s = sh / H, h = sh % H;
  const int col0 = kCols * blockIdx.y;
  const int t = threadIdx.x;
  const int row = t >> 1, c4 = (t & 1) * kColQ;  // row of S, first of this thread's float4 columns
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
      for (int q = 0; q < kColQ; ++q) out[c4 + q] = sbuf[cur][row][c4 + q];
    }
    if (j == K || (j + 1 == K && !end)) break;
    // S_{j+1}[row][cols] = B_j[row][cols] + sum_k M_j[row][k] S_j[k][cols]; with
    // no initial state S_0 = 0, and M_0 is not read (it may not have been made)
    const float *m = M + blk(seg) + (int64_t)row * D;
    const float4 *b = reinterpret_cast<const float4 *>(B + blk(seg) + (int64_t)row * D + col0);
    float4 acc[kColQ];
#pragma unroll
    for (int q = 0; q < kColQ; ++q) acc[q] = b[c4 + q];
    for (int k = 0; (j > 0 || init) && k < D; k += 4) {
      const float4 mk = *reinterpret_cast<const float4 *>(m + k);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float mv = kk == 0 ? mk.x : kk == 1 ? mk.y : kk == 2 ? mk.z : mk.w;
#pragma unroll
        for (int q = 0; q < kColQ; ++q) {
          const float4 sv = sbuf[cur][k + kk][c4 + q];
          acc[q].x = fmaf(mv, sv.x, acc[q].x);
          acc[q].y = fmaf(mv, sv.y, acc[q].y);
          acc[q].z = fmaf(mv, sv.z, acc[q].z);
          acc[q].w = fmaf(mv, sv.w, acc[q].w);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kColQ; ++q) sbuf[cur ^ 1][row][c4 + q] = acc[q];
    __syncthreads();
  }
}

// out[t, h] += S_jᵀ q_eff[t, h] for the tokens t of segment j: the correction
// that turns the zero-start outputs o⁰_t into the true ones,
// o_t = o⁰_t + (M_t S_j)ᵀ q_t with q_eff = M_tᵀ q_t.  One CTA per (segment,
// kCorrTilesPerCta consecutive 64-token tiles, head), which converts S_j once:
// block x = j * ctas_per_seg + c (ctas_per_seg: a bound on any segment's tile
// count over kCorrTilesPerCta; CTAs and tiles past their segment's end stop).  Warp MMAs with
// bf16 operands (S_j rounded like the state operands of the prefill), fp32
// accumulation; `skip_first` leaves segment 0 of every sequence alone (its
// start state is zero).
constexpr int kCorrTile = 64;
constexpr int kCorrTilesPerCta = 8;  // tiles of one segment and head per CTA (one S_j load)
constexpr int kSbPitch = D + 8;   // u32 per row of the bf16 pairs of S_j: bank-conflict free
constexpr int kQsPitch = D + 8;   // bf16 per row of the q_eff tile
__global__ void __launch_bounds__(256, 2)
kda_split_correct_kernel(__nv_bfloat16 *__restrict__ out, const __nv_bfloat16 *__restrict__ qe,
                         const float *__restrict__ start, const int32_t *__restrict__ seg_cu,
                         int64_t n_tokens, int32_t K, int32_t H, int32_t ctas_per_seg,
                         int skip_first) {
  extern __shared__ __align__(16) uint32_t corr_smem[];
  uint32_t *sb = corr_smem;                                              // [64 k-pairs][kSbPitch]
  __nv_bfloat16 *qs = reinterpret_cast<__nv_bfloat16 *>(corr_smem + (D / 2) * kSbPitch);  // [64][kQsPitch]
  const int seg = blockIdx.x / ctas_per_seg, h = blockIdx.y;
  if (skip_first && seg % K == 0) return;
  const int64_t s0 = seg_cu[seg], s1 = seg_cu[seg + 1];
  // this CTA's tiles: kCorrTilesPerCta consecutive ones from tb0
  const int64_t tb0 = s0 + (int64_t)kCorrTile * kCorrTilesPerCta * (blockIdx.x % ctas_per_seg);
  if (s0 < 0 || s1 > n_tokens || tb0 >= s1) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  // S_j as bf16 pairs along k: sb[kp][n] = (S[2 kp][n], S[2 kp + 1][n])
  const float *S = start + ((int64_t)seg * H + h) * D * D;
  for (int i = tid; i < (D / 2) * D; i += 256) {
    const int kp = i / D, n = i % D;
    const __nv_bfloat162 v = __floats2bfloat162_rn(S[(2 * kp) * D + n], S[(2 * kp + 1) * D + n]);
    sb[kp * kSbPitch + n] = *reinterpret_cast<const uint32_t *>(&v);
  }
  const int mt = warp & 3, nh = warp >> 2;  // 16 tokens x 64 columns per warp
  for (int ti = 0; ti < kCorrTilesPerCta; ++ti) {
    const int64_t tb = tb0 + (int64_t)kCorrTile * ti;
    if (tb >= s1) break;  // uniform
    if (ti > 0) __syncthreads();  // the previous tile's products have read qs
    const int rows = (int)(s1 - tb < kCorrTile ? s1 - tb : kCorrTile);
    for (int i = tid; i < kCorrTile * (D / 8); i += 256) {
      const int r = i / (D / 8), c8 = i % (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) v = *reinterpret_cast<const uint4 *>(qe + ((tb + r) * H + h) * D + 8 * c8);
      *reinterpret_cast<uint4 *>(qs + r * kQsPitch + 8 * c8) = v;
    }
    __syncthreads();
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
#pragma unroll
    for (int kt = 0; kt < D / 16; ++kt) {
      const __nv_bfloat16 *qa = qs + (16 * mt + g) * kQsPitch + 16 * kt + 2 * t4;
      const uint32_t a0 = *reinterpret_cast<const uint32_t *>(qa);
      const uint32_t a1 = *reinterpret_cast<const uint32_t *>(qa + 8 * kQsPitch);
      const uint32_t a2 = *reinterpret_cast<const uint32_t *>(qa + 8);
      const uint32_t a3 = *reinterpret_cast<const uint32_t *>(qa + 8 * kQsPitch + 8);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int n = 64 * nh + 8 * nt + g;
        mma_bf16_16x8x16(acc[nt], a0, a1, a2, a3, sb[(8 * kt + t4) * kSbPitch + n],
                         sb[(8 * kt + 4 + t4) * kSbPitch + n]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int n = 64 * nh + 8 * nt + 2 * t4;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = 16 * mt + g + 8 * half;
        if (r >= rows) continue;
        __nv_bfloat162 *o = reinterpret_cast<__nv_bfloat162 *>(out + ((tb + r) * H + h) * D + n);
        const float2 v = __bfloat1622float2(*o);
        *o = __floats2bfloat162_rn(v.x + acc[nt][2 * half], v.y + acc[nt][2 * half + 1]);
      }
    }
  }
}
constexpr size_t kCorrSmem = (size_t)(D / 2) * kSbPitch * 4 + (size_t)kCorrTile * kQsPitch * 2;

}  // namespace

size_t split_workspace_bytes(int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t K) {
  const size_t nseg = (size_t)n_seqs * K;
  const size_t cu_bytes = ((nseg + 1) * sizeof(int32_t) + 1023) / 1024 * 1024;
  return cu_bytes + 3 * nseg * H * (size_t)D * D * sizeof(float) +
         (size_t)n_tokens * H * D * sizeof(__nv_bfloat16);
}

cudaError_t launch_chunk_fwd_split(const ChunkArgs &a, int32_t K, unsigned char *ws,
                                   cudaStream_t stream) {
  const int64_t nseg = (int64_t)a.n_seqs * K;
  if (K < 2 || nseg > 0x7fffffffLL || nseg * a.H > 0x7fffffffLL) return cudaErrorInvalidValue;
  const size_t cu_bytes = ((size_t)(nseg + 1) * sizeof(int32_t) + 1023) / 1024 * 1024;
  const size_t states = (size_t)nseg * a.H * D * D;
  int32_t *seg_cu = reinterpret_cast<int32_t *>(ws);
  float *B = reinterpret_cast<float *>(ws + cu_bytes), *M = B + states, *S = M + states;
  __nv_bfloat16 *qe = reinterpret_cast<__nv_bfloat16 *>(S + states);  // [N, H, 128]

  kda_split_bounds_kernel<<<(unsigned)((nseg + 1 + 255) / 256), 256, 0, stream>>>(
      a.cu_seqlens, a.n_seqs, K, seg_cu);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // pass 1: per segment, B and the outputs o0 from a zero state (into out), M and
  // q_eff = M_t^T q_t from the identity with v = 0 (into qe)
  ChunkArgs p = a;
  p.cu_seqlens = seg_cu;
  p.n_seqs = (int32_t)nseg;
  p.init_state = nullptr;
  p.final_state = B;
  p.final_state_m = M;
  p.out_m = qe;
  p.write_out = true;
  p.mode = ChunkArgs::kTransitions;
  p.help_ws = nullptr;
  p.n_help = 0;
  p.seq_order = nullptr;  // sized for the sequences, not the segments
  p.split_skip_k = a.init_state == nullptr ? K : 0;  // S_0 = 0: M_0 is never needed
  e = launch_chunk_fwd_bf16_tc(p, stream);
  if (e != cudaSuccess) return e;

  // the start state of every segment, and every sequence's final state
  kda_split_combine_kernel<<<dim3((unsigned)(a.n_seqs * a.H), D / kCols), 256, 0, stream>>>(
      a.init_state, B, M, a.n_seqs, K, a.H, S, a.final_state);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // o_t = o0_t + S_j^T q_eff_t (segment 0 of a sequence without init state starts from 0)
  e = cudaFuncSetAttribute(kda_split_correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kCorrSmem);
  if (e != cudaSuccess) return e;
  // no segment is longer than ceil(ceil(N / 64) / K) chunks of 64 tokens
  const int64_t tiles = ((a.n_tokens + kChunk - 1) / kChunk + K - 1) / K;
  if (tiles == 0) return cudaSuccess;
  const int64_t cps = (tiles + kCorrTilesPerCta - 1) / kCorrTilesPerCta;
  if (nseg * cps > 0x7fffffffLL || a.H > 65535) return cudaErrorInvalidValue;
  kda_split_correct_kernel<<<dim3((unsigned)(nseg * cps), (unsigned)a.H), 256, kCorrSmem,
                             stream>>>(static_cast<__nv_bfloat16 *>(a.out), qe, S, seg_cu,
                                       a.n_tokens, K, a.H, (int32_t)cps,
                                       a.init_state == nullptr ? 1 : 0);
  return cudaGetLastError();
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
