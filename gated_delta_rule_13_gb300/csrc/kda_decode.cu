// KDA recurrent decode step: one token per (sequence, head), state in place.
//
// Per unit (b, h) with state S in R^{128 x 128} (dk rows, dv contiguous):
//   X   = Diag(alpha) S                       (alpha = exp(log_alpha), per key row)
//   u   = beta (v - X^T k)                    (delta-rule correction)
//   S'  = X + k u^T                           (= (I - beta k k^T) X + beta k v^T)
//   o   = S'^T q = X^T q + (k . q) u
// ("Kimi K3" study notes, section 3-2 "2) Kimi Delta Attention": update and
// read-out equations; the decode state advances in place: "Kimi K3: 架构、训练
// 与系统全景解析", section 4.2.7).
//
// HBM-bound: a unit reads and writes its 64 KiB state exactly once.  One CTA
// of 8 warps per unit; warp w owns value columns [16w, 16w+16) for all 128 key
// rows, lane l owns 4 consecutive columns (one float4) of rows l/4 + 8j,
// j = 0..15.  Both column reductions over the key dimension (X^T k, X^T q)
// then stay inside a warp (three xor-shuffles), so the only block-wide barrier
// is the one that publishes alpha, k and q.  The 16 float4 state loads are
// issued before that barrier so their HBM latency overlaps it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;
constexpr int D = kHeadDim;
constexpr int kThreads = 256;

template <bool BF16>
__device__ __forceinline__ float load_elem(const void *p, int64_t i) {
  if constexpr (BF16) {
    return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
  } else {
    return static_cast<const float *>(p)[i];
  }
}

template <bool BF16>
__device__ __forceinline__ float4 load4(const void *p, int64_t i) {
  if constexpr (BF16) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p) + i);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
  } else {
    return *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
  }
}

template <bool BF16>
__device__ __forceinline__ void store4(void *p, int64_t i, float4 x) {
  if constexpr (BF16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
    uint2 raw;
    raw.x = *reinterpret_cast<uint32_t *>(&lo);
    raw.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p) + i) = raw;
  } else {
    *reinterpret_cast<float4 *>(static_cast<float *>(p) + i) = x;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 2)
kda_decode_step_kernel(float *__restrict__ state, const void *__restrict__ q,
                       const void *__restrict__ k, const void *__restrict__ v,
                       const float *__restrict__ log_alpha, const float *__restrict__ beta,
                       void *__restrict__ out) {
  __shared__ float s_alpha[D], s_k[D], s_q[D];
  const int64_t unit = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int col = 16 * warp + 4 * (lane & 3);
  const int row0 = lane >> 2;
  float *S = state + unit * (int64_t)(D * D);

  float4 s[16];
#pragma unroll
  for (int j = 0; j < 16; ++j)
    s[j] = __ldcs(reinterpret_cast<const float4 *>(S + (row0 + 8 * j) * D + col));

  if (tid < D) {
    s_alpha[tid] = expf(log_alpha[unit * D + tid]);
    s_k[tid] = load_elem<BF16>(k, unit * D + tid);
    s_q[tid] = load_elem<BF16>(q, unit * D + tid);
  }
  const float4 vv = load4<BF16>(v, unit * D + col);
  const float b = beta[unit];
  __syncthreads();

  // X = Diag(alpha) S; partial sums of X^T k and X^T q over this lane's rows.
  float pk0 = 0.f, pk1 = 0.f, pk2 = 0.f, pk3 = 0.f;
  float pq0 = 0.f, pq1 = 0.f, pq2 = 0.f, pq3 = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int r = row0 + 8 * j;
    const float a = s_alpha[r], kr = s_k[r], qr = s_q[r];
    s[j].x *= a; s[j].y *= a; s[j].z *= a; s[j].w *= a;
    pk0 = fmaf(kr, s[j].x, pk0); pk1 = fmaf(kr, s[j].y, pk1);
    pk2 = fmaf(kr, s[j].z, pk2); pk3 = fmaf(kr, s[j].w, pk3);
    pq0 = fmaf(qr, s[j].x, pq0); pq1 = fmaf(qr, s[j].y, pq1);
    pq2 = fmaf(qr, s[j].z, pq2); pq3 = fmaf(qr, s[j].w, pq3);
  }
  // Lanes with equal (lane & 3) hold the same columns: reduce over lane bits 2..4.
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    pk0 += __shfl_xor_sync(0xffffffffu, pk0, off);
    pk1 += __shfl_xor_sync(0xffffffffu, pk1, off);
    pk2 += __shfl_xor_sync(0xffffffffu, pk2, off);
    pk3 += __shfl_xor_sync(0xffffffffu, pk3, off);
    pq0 += __shfl_xor_sync(0xffffffffu, pq0, off);
    pq1 += __shfl_xor_sync(0xffffffffu, pq1, off);
    pq2 += __shfl_xor_sync(0xffffffffu, pq2, off);
    pq3 += __shfl_xor_sync(0xffffffffu, pq3, off);
  }
  // k . q over the 128 key channels (every warp computes it).
  float kq = 0.f;
#pragma unroll
  for (int j = 0; j < D / 32; ++j) kq = fmaf(s_k[lane + 32 * j], s_q[lane + 32 * j], kq);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);

  const float u0 = b * (vv.x - pk0), u1 = b * (vv.y - pk1);
  const float u2 = b * (vv.z - pk2), u3 = b * (vv.w - pk3);
  if (row0 == 0) {
    store4<BF16>(out, unit * D + col,
                 make_float4(fmaf(kq, u0, pq0), fmaf(kq, u1, pq1), fmaf(kq, u2, pq2),
                             fmaf(kq, u3, pq3)));
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float kr = s_k[row0 + 8 * j];
    float4 x = s[j];
    x.x = fmaf(kr, u0, x.x); x.y = fmaf(kr, u1, x.y);
    x.z = fmaf(kr, u2, x.z); x.w = fmaf(kr, u3, x.w);
    __stcs(reinterpret_cast<float4 *>(S + (row0 + 8 * j) * D + col), x);
  }
}

// Replay of the accepted draft tokens of a speculative decode step ("Kimi K3:
// 架构、训练与系统全景解析", section on KDA state replay under speculative decoding:
// the small per-token projected inputs are cached instead of per-position
// states; after verification only the accepted prefix is replayed in an
// on-chip recurrence and only the final state is written back).
//
// Unit (b, h) applies the decode step above to tokens t = 0 .. n_b - 1 of its
// cached inputs in order, n_b = n_accept[b] clamped to [0, T], keeping the
// state in registers: one HBM read and one write of the state for all n_b
// tokens (none at all when n_b = 0).  The inputs of up to kReplayGroup tokens
// are fetched into shared memory in one cooperative pass.
//
// The CTAs are persistent (two per SM), each walking units with a stride of the
// grid, and while one unit's tokens run from registers the next unit's state and
// the cached inputs of its first kReplayGroup tokens are already being copied
// into shared memory by bulk copies (its beta values by 4-byte asynchronous
// copies): the memory system has the next unit in flight throughout the
// compute, and a unit starts without a round trip to HBM.  The issuing thread
// waits on no load either: the accepted count of the unit after next is copied
// the same way one unit ahead of its use (a synchronous load of the count
// stalled that thread's warp, and with it the whole CTA at its next barrier, by
// a memory round trip per unit).
constexpr int kReplayGroup = 8;
// Staged inputs of one token: log_alpha (fp32), then k, q, v in the input type.
template <bool BF16>
constexpr int replay_raw_token_bytes() { return D * 4 + 3 * D * (BF16 ? 2 : 4); }
template <bool BF16>
constexpr size_t replay_smem_bytes() {
  return (size_t)D * D * sizeof(float) + (size_t)kReplayGroup * replay_raw_token_bytes<BF16>();
}
constexpr uint64_t kReplayWaitNs = 2000000000ull;  // bound on the state copy wait

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 2)
kda_decode_replay_kernel(float *__restrict__ state, const void *__restrict__ q,
                         const void *__restrict__ k, const void *__restrict__ v,
                         const float *__restrict__ log_alpha, const float *__restrict__ beta,
                         const int32_t *__restrict__ n_accept, int32_t T, int32_t H,
                         int64_t units, void *__restrict__ out) {
  // the next unit's state [D][D], then the staged inputs of its first tokens
  extern __shared__ __align__(128) float stage[];
  constexpr int kEsz = BF16 ? 2 : 4, kRawTok = replay_raw_token_bytes<BF16>();
  uint8_t *const raw = reinterpret_cast<uint8_t *>(stage + D * D);
  __shared__ __align__(16) float s_alpha[kReplayGroup][D], s_k[kReplayGroup][D],
      s_q[kReplayGroup][D], s_v[kReplayGroup][D];
  __shared__ float s_beta[kReplayGroup];
  __shared__ float s_nbeta[2][kReplayGroup];  // staged betas of the first tokens, by unit parity
  __shared__ int64_t s_cand;                  // the next unit to look at (thread 0)
  __shared__ int32_t s_cand_n;                // its accepted count, unclamped
  __shared__ __align__(8) uint64_t bar;
  __shared__ int64_t s_next;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int col = 16 * warp + 4 * (lane & 3);
  const int row0 = lane >> 2;
  auto accepted = [&](int64_t u) {
    const int n = n_accept[u / H];
    return n < 0 ? 0 : (n > T ? T : n);
  };
  // thread 0: the next unit with accepted tokens from s_cand on (stride
  // gridDim.x), its state and first tokens' inputs copied into the stage, its
  // betas into s_nbeta[slot]; then the count of the candidate after it
  auto prefetch_next = [&](int slot) {
    int64_t u = s_cand;
    int n_u = u < units ? (s_cand_n < 0 ? 0 : (s_cand_n > T ? T : s_cand_n)) : 0;
    while (u < units && n_u == 0) {
      u += gridDim.x;
      n_u = u < units ? accepted(u) : 0;
    }
    s_next = u;
    s_cand = u + gridDim.x;
    if (u + gridDim.x < units) cp_async4(&s_cand_n, n_accept + (u + gridDim.x) / H);
    if (u < units) {
      const int cnt = n_u < kReplayGroup ? n_u : kReplayGroup;
      const int64_t b = u / H, h = u % H;
      mbar_arrive_expect_tx(&bar, D * D * sizeof(float) + (uint32_t)(cnt * kRawTok));
      bulk_load(smem_u32(stage), state + u * (int64_t)(D * D), D * D * sizeof(float), &bar);
#pragma unroll
      for (int t = 0; t < kReplayGroup; ++t) {
        if (t < cnt) {
          const int64_t iu = (b * T + t) * H + h;  // (sequence, token, head)
          const uint32_t dst = smem_u32(raw + t * kRawTok);
          bulk_load(dst, log_alpha + iu * D, D * 4, &bar);
          bulk_load(dst + D * 4, static_cast<const uint8_t *>(k) + iu * D * kEsz, D * kEsz, &bar);
          bulk_load(dst + D * 4 + D * kEsz, static_cast<const uint8_t *>(q) + iu * D * kEsz,
                    D * kEsz, &bar);
          bulk_load(dst + D * 4 + 2 * D * kEsz, static_cast<const uint8_t *>(v) + iu * D * kEsz,
                    D * kEsz, &bar);
          cp_async4(&s_nbeta[slot][t], beta + iu);
        }
      }
    }
    cp_async_commit();
  };
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    s_cand = blockIdx.x;
    s_cand_n = (int64_t)blockIdx.x < units ? n_accept[blockIdx.x / H] : 0;
    prefetch_next(0);
  }
  __syncthreads();
  int64_t u = s_next;
  uint32_t phase = 0;
  while (u < units) {
    const bool landed = mbar_wait(&bar, phase, kReplayWaitNs);
    if (tid == 0) cp_async_wait_all();  // the betas and the next candidate's count
    if (__syncthreads_or(!landed)) {  // a copy that never lands: leave, every thread alike
      if (tid == 0) mbar_wait(&bar, phase, kReplayWaitNs);  // (bounded) no copy outlives the CTA
      return;
    }
    const int slot = (int)phase;  // this unit's parity
    phase ^= 1u;
    float4 s[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      s[j] = *reinterpret_cast<const float4 *>(stage + (row0 + 8 * j) * D + col);
    const int64_t b = u / H, h = u % H;
    const int n = accepted(u);
    {  // the first tokens' staged inputs, converted
      const int cnt = n < kReplayGroup ? n : kReplayGroup;
      for (int e = tid; e < cnt * D; e += kThreads) {
        const int t = e / D, c = e % D;
        const uint8_t *rt = raw + t * kRawTok;
        s_alpha[t][c] = expf(reinterpret_cast<const float *>(rt)[c]);
        s_k[t][c] = load_elem<BF16>(rt + D * 4, c);
        s_q[t][c] = load_elem<BF16>(rt + D * 4 + D * kEsz, c);
        s_v[t][c] = load_elem<BF16>(rt + D * 4 + 2 * D * kEsz, c);
      }
      if (tid < cnt) s_beta[tid] = s_nbeta[slot][tid];
    }
    __syncthreads();  // the stage is free for the next unit; the first inputs are in place
    if (tid == 0) prefetch_next(slot ^ 1);

    float *S = state + u * (int64_t)(D * D);
    for (int t0 = 0; t0 < n; t0 += kReplayGroup) {
      const int cnt = n - t0 < kReplayGroup ? n - t0 : kReplayGroup;
      if (t0 > 0) __syncthreads();  // the previous group's inputs are consumed
      for (int e = tid; t0 > 0 && e < cnt * D; e += kThreads) {
        const int t = e / D, c = e % D;
        const int64_t iu = (b * T + t0 + t) * H + h;  // (sequence, token, head)
        s_alpha[t][c] = expf(log_alpha[iu * D + c]);
        s_k[t][c] = load_elem<BF16>(k, iu * D + c);
        s_q[t][c] = load_elem<BF16>(q, iu * D + c);
        s_v[t][c] = load_elem<BF16>(v, iu * D + c);
      }
      if (t0 > 0 && tid < cnt) s_beta[tid] = beta[(b * T + t0 + tid) * H + h];
      if (t0 > 0) __syncthreads();

      for (int t = 0; t < cnt; ++t) {
        const float *sa = s_alpha[t], *sk = s_k[t], *sq = s_q[t];
        const float4 vv = *reinterpret_cast<const float4 *>(&s_v[t][col]);
        const float bt = s_beta[t];
        float pk0 = 0.f, pk1 = 0.f, pk2 = 0.f, pk3 = 0.f;
        float pq0 = 0.f, pq1 = 0.f, pq2 = 0.f, pq3 = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = row0 + 8 * j;
          const float a = sa[r], kr = sk[r], qr = sq[r];
          s[j].x *= a; s[j].y *= a; s[j].z *= a; s[j].w *= a;
          pk0 = fmaf(kr, s[j].x, pk0); pk1 = fmaf(kr, s[j].y, pk1);
          pk2 = fmaf(kr, s[j].z, pk2); pk3 = fmaf(kr, s[j].w, pk3);
          pq0 = fmaf(qr, s[j].x, pq0); pq1 = fmaf(qr, s[j].y, pq1);
          pq2 = fmaf(qr, s[j].z, pq2); pq3 = fmaf(qr, s[j].w, pq3);
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          pk0 += __shfl_xor_sync(0xffffffffu, pk0, off);
          pk1 += __shfl_xor_sync(0xffffffffu, pk1, off);
          pk2 += __shfl_xor_sync(0xffffffffu, pk2, off);
          pk3 += __shfl_xor_sync(0xffffffffu, pk3, off);
          pq0 += __shfl_xor_sync(0xffffffffu, pq0, off);
          pq1 += __shfl_xor_sync(0xffffffffu, pq1, off);
          pq2 += __shfl_xor_sync(0xffffffffu, pq2, off);
          pq3 += __shfl_xor_sync(0xffffffffu, pq3, off);
        }
        float kq = 0.f;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) kq = fmaf(sk[lane + 32 * j], sq[lane + 32 * j], kq);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);

        const float u0 = bt * (vv.x - pk0), u1 = bt * (vv.y - pk1);
        const float u2 = bt * (vv.z - pk2), u3 = bt * (vv.w - pk3);
        if (out != nullptr && row0 == 0) {
          const int64_t iu = (b * T + t0 + t) * H + h;
          store4<BF16>(out, iu * D + col,
                       make_float4(fmaf(kq, u0, pq0), fmaf(kq, u1, pq1), fmaf(kq, u2, pq2),
                                   fmaf(kq, u3, pq3)));
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float kr = sk[row0 + 8 * j];
          s[j].x = fmaf(kr, u0, s[j].x); s[j].y = fmaf(kr, u1, s[j].y);
          s[j].z = fmaf(kr, u2, s[j].z); s[j].w = fmaf(kr, u3, s[j].w);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      __stcs(reinterpret_cast<float4 *>(S + (row0 + 8 * j) * D + col), s[j]);
    __syncthreads();  // s_next is set; the input buffers may be refilled
    u = s_next;
  }
}

}  // namespace

cudaError_t launch_decode_step(float *state, const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, int32_t B, int32_t H,
                               bool bf16, void *out, cudaStream_t stream) {
  const int64_t units = (int64_t)B * H;
  if (units == 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)units), block(kThreads);
  if (bf16) {
    kda_decode_step_kernel<true><<<grid, block, 0, stream>>>(state, q, k, v, log_alpha, beta, out);
  } else {
    kda_decode_step_kernel<false><<<grid, block, 0, stream>>>(state, q, k, v, log_alpha, beta, out);
  }
  return cudaGetLastError();
}


cudaError_t launch_decode_replay(float *state, const void *q, const void *k, const void *v,
                                 const float *log_alpha, const float *beta,
                                 const int32_t *n_accept, int32_t B, int32_t T, int32_t H,
                                 bool bf16, void *out, cudaStream_t stream) {
  const int64_t units = (int64_t)B * H;
  if (units == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t ctas = units < 2 * (int64_t)sms ? units : 2 * (int64_t)sms;
  const size_t stage = bf16 ? replay_smem_bytes<true>() : replay_smem_bytes<false>();
  auto kern = bf16 ? kda_decode_replay_kernel<true> : kda_decode_replay_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stage);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)ctas, kThreads, stage, stream>>>(state, q, k, v, log_alpha, beta, n_accept, T,
                                                    H, units, out);
  return cudaGetLastError();
}

}  // namespace kda
