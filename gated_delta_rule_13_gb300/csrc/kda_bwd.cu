// Gradient of the KDA recurrence (the backward pass of kda_chunk_fwd).
//
// The pages give no gradient ("Kimi K3: 架构、训练与系统全景解析", section 7.1:
// the chunked KDA kernel serves training as well as prefill).  This is the chain
// rule through the token form of the update and read-out ("Kimi K3" study
// notes, section 3-2 "2) Kimi Delta Attention"):
//   X = Diag(alpha) S_{t-1},  p = X^T k,  d = beta (v - p),  S_t = X + k d^T,
//   o_t = S_t^T q
// taken in reverse, token by token, from the last token of each sequence:
//   dS += q do^T;  dq = S_t do;  dd = dS^T k;  dk = dS d;  dv = beta dd;
//   dbeta = dd . (v - p);  dp = -beta dd;  dX = dS + k dp^T;  dk += X dp;
//   dlog_alpha = rowsum(dX o X);  dS_{t-1} = Diag(alpha) dX.
//
// Work split.  The columns of S (value channels) evolve independently, so a
// chain is cut into four blocks of 32 value columns, one CTA each (8 warps:
// lane = value column, warp w = key rows 16w .. 16w + 15, 16 state values per
// thread).  dv and the initial-state gradient belong to one block; dq, dk,
// dlog_alpha and dbeta are sums over all value columns, reduced inside the
// warp (a transposing butterfly) and added across the four blocks with fp32
// atomics (so their last bits depend on the order of those four additions).
//
// States.  A forward pass stores the state before every `every`-th token (a
// power of two >= kGroup, chosen by the caller of launch_chunk_bwd); the
// backward pass recomputes, for each group of kGroup tokens, the decayed states
// X of those tokens from the nearest checkpoint into shared memory, then runs
// them in reverse.  With every == kGroup nothing is recomputed twice; a wider
// interval trades (every / kGroup - 1) / 2 extra forward steps per token for
// less checkpoint memory.  CUDA cores, fp32 arithmetic, fp32 state and
// gradients.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int D = kHeadDim;       // 128
constexpr int kCols = 32;         // value columns per CTA
constexpr int kBlocks = D / kCols;
constexpr int kThreads = 256;
constexpr int kRows = 16;         // key rows per thread
constexpr int kGroup = 4;         // tokens whose X a CTA keeps at a time

// Checkpoint slot of sequence s: floor(cu[s] / every) + s.  Consecutive
// sequences never share slots, since floor(b / c) - floor(a / c) + 1 >=
// ceil((b - a) / c).
__device__ __forceinline__ int64_t ckpt_base(int64_t cu_s, int64_t s, int every) {
  return cu_s / every + s;
}

template <bool BF16>
__device__ __forceinline__ float ld(const void *p, int64_t i) {
  if constexpr (BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
  else return static_cast<const float *>(p)[i];
}

// Inputs of up to kGroup consecutive tokens of one (sequence, head), staged.
struct Stage {
  float q[kGroup][D], k[kGroup][D], alpha[kGroup][D];
  float v[kGroup][kCols], dout[kGroup][kCols], beta[kGroup];
};

template <bool BF16>
__device__ void stage_tokens(Stage &st, int64_t tb, int n, int h, int H, int cb, const void *q,
                             const void *k, const void *v, const float *la, const float *beta,
                             const void *dout) {
  for (int e = threadIdx.x; e < n * D; e += kThreads) {
    const int i = e / D, c = e % D;
    const int64_t row = ((tb + i) * H + h) * D + c;
    st.q[i][c] = q ? ld<BF16>(q, row) : 0.f;
    st.k[i][c] = ld<BF16>(k, row);
    st.alpha[i][c] = expf(la[row]);
  }
  for (int e = threadIdx.x; e < n * kCols; e += kThreads) {
    const int i = e / kCols, c = e % kCols;
    const int64_t row = ((tb + i) * H + h) * D + cb * kCols + c;
    st.v[i][c] = ld<BF16>(v, row);
    st.dout[i][c] = dout ? ld<BF16>(dout, row) : 0.f;
  }
  if (threadIdx.x < n) st.beta[threadIdx.x] = beta[(tb + threadIdx.x) * H + h];
}

// One forward token on this thread's 16 state values (rows r0 + j, column
// lane); the decayed state X and the per-column p, d are returned.  Uses red.
__device__ __forceinline__ void fwd_token(float (&s)[kRows], float (&x)[kRows], float &p, float &d,
                                          const Stage &st, int i, int r0, int lane, int warp,
                                          float (*red)[kCols]) {
  float part = 0.f;
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    x[j] = st.alpha[i][r0 + j] * s[j];
    part = fmaf(x[j], st.k[i][r0 + j], part);
  }
  red[warp][lane] = part;
  __syncthreads();
  p = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) p += red[w][lane];
  d = st.beta[i] * (st.v[i][lane] - p);
#pragma unroll
  for (int j = 0; j < kRows; ++j) s[j] = fmaf(st.k[i][r0 + j], d, x[j]);
  __syncthreads();  // red is free again
}

// Sum of v[j] over the 32 lanes, for each of the 16 rows j: after four
// halving exchanges lane L holds one row, row_of(L), summed over 16 lanes,
// and the last exchange completes it (lanes 2m and 2m + 1 hold the same row).
__device__ __forceinline__ float row_sum(float (&v)[kRows], int lane) {
  float a[8];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float mine = hi ? v[8 + j] : v[j], give = hi ? v[j] : v[8 + j];
      a[j] = mine + __shfl_xor_sync(0xffffffffu, give, 16);
    }
  }
  float b[4];
  {
    const bool hi = lane & 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float mine = hi ? a[4 + j] : a[j], give = hi ? a[j] : a[4 + j];
      b[j] = mine + __shfl_xor_sync(0xffffffffu, give, 8);
    }
  }
  float c[2];
  {
    const bool hi = lane & 4;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float mine = hi ? b[2 + j] : b[j], give = hi ? b[j] : b[2 + j];
      c[j] = mine + __shfl_xor_sync(0xffffffffu, give, 4);
    }
  }
  const bool hi = lane & 2;
  float e = (hi ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, hi ? c[0] : c[1], 2);
  return e + __shfl_xor_sync(0xffffffffu, e, 1);
}
__device__ __forceinline__ int row_of(int lane) {
  return 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
}

struct Chain {
  int seq, h, cb;
  int64_t t0, t1;
  bool ok;
};
__device__ __forceinline__ Chain chain_of(const int32_t *cu, int32_t n_seqs, int64_t n_tokens,
                                          int H) {
  Chain c;
  const int64_t u = blockIdx.x / kBlocks;
  c.cb = (int)(blockIdx.x % kBlocks);
  c.seq = (int)(u / H);
  c.h = (int)(u % H);
  c.t0 = cu[c.seq];
  c.t1 = cu[c.seq + 1];
  c.ok = c.t0 >= 0 && c.t1 >= c.t0 && c.t1 <= n_tokens &&
         (c.seq != 0 || (cu[0] == 0 && cu[n_seqs] == n_tokens));
  return c;
}

// Forward pass: the state before every kCkpt-th token, per block of columns.
template <bool BF16>
__global__ void __launch_bounds__(kThreads, 2)
kda_bwd_ckpt_kernel(const void *__restrict__ k, const void *__restrict__ v,
                    const float *__restrict__ la, const float *__restrict__ beta,
                    const float *__restrict__ init_state, const int32_t *__restrict__ cu,
                    int32_t n_seqs, int64_t n_tokens, int32_t H, int every,
                    float *__restrict__ ckpt, DeviceStatus *status) {
  __shared__ Stage st;
  __shared__ float red[kThreads / 32][kCols];
  const Chain c = chain_of(cu, n_seqs, n_tokens, H);
  if (!c.ok) {
    if (threadIdx.x == 0) atomicCAS(&status->code, 0, 1 /* KDA_ERR_INVALID_ARG */);
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, r0 = kRows * warp;
  const int col = c.cb * kCols + lane;
  const int64_t sbase = ((int64_t)c.seq * H + c.h) * D * D;
  float s[kRows], x[kRows];
#pragma unroll
  for (int j = 0; j < kRows; ++j) s[j] = init_state ? init_state[sbase + (r0 + j) * D + col] : 0.f;
  const int64_t base = ckpt_base(c.t0, c.seq, every);
  for (int64_t tb = c.t0; tb < c.t1; tb += kGroup) {
    const int n = (int)(c.t1 - tb < kGroup ? c.t1 - tb : kGroup);
    __syncthreads();  // the previous group's stage is consumed
    stage_tokens<BF16>(st, tb, n, c.h, H, c.cb, nullptr, k, v, la, beta, nullptr);
    __syncthreads();
    for (int i = 0; i < n; ++i) {
      const int64_t t = tb + i;
      if ((t - c.t0) % every == 0) {
        float *dst = ckpt + ((base + (t - c.t0) / every) * H + c.h) * D * D;
#pragma unroll
        for (int j = 0; j < kRows; ++j) dst[(r0 + j) * D + col] = s[j];
      }
      float p, d;
      fwd_token(s, x, p, d, st, i, r0, lane, warp, red);
    }
  }
}

// Backward pass.
template <bool BF16>
__global__ void __launch_bounds__(kThreads, 2)
kda_bwd_kernel(const void *__restrict__ q, const void *__restrict__ k, const void *__restrict__ v,
               const float *__restrict__ la, const float *__restrict__ beta,
               const int32_t *__restrict__ cu, int32_t n_seqs, int64_t n_tokens, int32_t H,
               int every, const float *__restrict__ ckpt, const void *__restrict__ dout,
               const float *__restrict__ d_final, float *__restrict__ dq_acc,
               float *__restrict__ dk_acc, void *__restrict__ dv_out, float *__restrict__ dla,
               float *__restrict__ dbeta, float *__restrict__ d_init) {
  extern __shared__ __align__(16) float xs[];  // [kGroup][D][kCols] decayed states
  __shared__ Stage st;
  __shared__ float red[kThreads / 32][kCols];
  __shared__ float s_p[kGroup][kCols], s_d[kGroup][kCols];
  const Chain c = chain_of(cu, n_seqs, n_tokens, H);
  if (!c.ok) return;  // recorded by the forward pass
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, r0 = kRows * warp;
  const int col = c.cb * kCols + lane;
  const int64_t sbase = ((int64_t)c.seq * H + c.h) * D * D;
  float ds[kRows];
#pragma unroll
  for (int j = 0; j < kRows; ++j) ds[j] = d_final ? d_final[sbase + (r0 + j) * D + col] : 0.f;
  const int64_t base = ckpt_base(c.t0, c.seq, every);
  const int64_t len = c.t1 - c.t0;
  const int64_t n_ck = (len + every - 1) / every;
  for (int64_t blk = n_ck - 1; blk >= 0; --blk) {
    const int64_t a = c.t0 + blk * every;
    const int64_t e = a + every < c.t1 ? a + every : c.t1;
    const int n_groups = (int)((e - a + kGroup - 1) / kGroup);
    for (int g = n_groups - 1; g >= 0; --g) {
      // state before token a, then forward to the group's first token
      float s[kRows], x[kRows];
      const float *src = ckpt + ((base + blk) * H + c.h) * D * D;
#pragma unroll
      for (int j = 0; j < kRows; ++j) s[j] = src[(r0 + j) * D + col];
      for (int64_t tb = a; tb < a + (int64_t)g * kGroup; tb += kGroup) {
        __syncthreads();
        stage_tokens<BF16>(st, tb, kGroup, c.h, H, c.cb, nullptr, k, v, la, beta, nullptr);
        __syncthreads();
        for (int i = 0; i < kGroup; ++i) {
          float p, d;
          fwd_token(s, x, p, d, st, i, r0, lane, warp, red);
        }
      }
      // the group's tokens: X, p and d kept
      const int64_t gb = a + (int64_t)g * kGroup;
      const int n = (int)(e - gb < kGroup ? e - gb : kGroup);
      __syncthreads();
      stage_tokens<BF16>(st, gb, n, c.h, H, c.cb, q, k, v, la, beta, dout);
      __syncthreads();
      for (int i = 0; i < n; ++i) {
        float p, d;
        fwd_token(s, x, p, d, st, i, r0, lane, warp, red);
#pragma unroll
        for (int j = 0; j < kRows; ++j) xs[(i * D + r0 + j) * kCols + lane] = x[j];
        if (warp == 0) {
          s_p[i][lane] = p;
          s_d[i][lane] = d;
        }
      }
      __syncthreads();
      // ... in reverse
      for (int i = n - 1; i >= 0; --i) {
        const int64_t t = gb + i;
        const int64_t trow = (t * H + c.h) * D;
        const float p = s_p[i][lane], d = s_d[i][lane], b = st.beta[i];
        const float dov = st.dout[i][lane];
        float cq[kRows], ck[kRows], cl[kRows];
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const int r = r0 + j;
          const float xv = xs[(i * D + r) * kCols + lane];
          const float kr = st.k[i][r];
          cq[j] = fmaf(kr, d, xv) * dov;                // S_t do (row sums: dq)
          ds[j] = fmaf(st.q[i][r], dov, ds[j]);          // dS += q do^T
          part = fmaf(ds[j], kr, part);                  // dd = dS^T k (column sums)
          cl[j] = xv;                                    // X, kept for the next pass
        }
        red[warp][lane] = part;
        __syncthreads();
        float dd = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) dd += red[w][lane];
        const float dp = -b * dd;
        if (warp == 0) {
          const float dvv = b * dd;
          if constexpr (BF16)
            static_cast<__nv_bfloat16 *>(dv_out)[trow + col] = __float2bfloat16_rn(dvv);
          else
            static_cast<float *>(dv_out)[trow + col] = dvv;
          float db = dd * (st.v[i][lane] - p);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) db += __shfl_xor_sync(0xffffffffu, db, off);
          if (lane == 0) atomicAdd(dbeta + t * H + c.h, db);
        }
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const int r = r0 + j;
          const float xv = cl[j];
          const float dx = fmaf(st.k[i][r], dp, ds[j]);  // dX = dS + k dp^T
          ck[j] = fmaf(ds[j], d, xv * dp);               // dk: dS d + X dp
          cl[j] = dx * xv;                               // dlog_alpha: dX o X
          ds[j] = st.alpha[i][r] * dx;                   // dS_{t-1} = Diag(alpha) dX
        }
        const float sq = row_sum(cq, lane), sk = row_sum(ck, lane), sl = row_sum(cl, lane);
        if ((lane & 1) == 0) {
          const int r = r0 + row_of(lane);
          atomicAdd(dq_acc + trow + r, sq);
          atomicAdd(dk_acc + trow + r, sk);
          atomicAdd(dla + trow + r, sl);
        }
        __syncthreads();  // red is free again
      }
    }
  }
  if (d_init) {
#pragma unroll
    for (int j = 0; j < kRows; ++j) d_init[sbase + (r0 + j) * D + col] = ds[j];
  }
}

// dq, dk in the input type from their fp32 accumulators.
template <bool BF16>
__global__ void kda_bwd_finish_kernel(const float *__restrict__ dq_acc,
                                      const float *__restrict__ dk_acc, void *__restrict__ dq,
                                      void *__restrict__ dk, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    if constexpr (BF16) {
      static_cast<__nv_bfloat16 *>(dq)[i] = __float2bfloat16_rn(dq_acc[i]);
      static_cast<__nv_bfloat16 *>(dk)[i] = __float2bfloat16_rn(dk_acc[i]);
    } else {
      static_cast<float *>(dq)[i] = dq_acc[i];
      static_cast<float *>(dk)[i] = dk_acc[i];
    }
  }
}

}  // namespace

size_t bwd_ckpt_slots(int32_t n_seqs, int64_t n_tokens, int32_t every) {
  return (size_t)(n_tokens / every) + (size_t)n_seqs + 1;
}

int32_t bwd_ckpt_every(int32_t n_seqs, int64_t n_tokens, int32_t H) {
  int32_t every = kGroup;
  while (every < kMaxCkptEvery &&
         bwd_ckpt_slots(n_seqs, n_tokens, every) * (size_t)H * D * D * sizeof(float) >
             kCkptBudgetBytes)
    every *= 2;
  return every;
}

cudaError_t launch_chunk_bwd(const BwdArgs &a, cudaStream_t stream) {
  const int64_t chains = (int64_t)a.n_seqs * a.H;
  if (chains == 0) return cudaSuccess;
  if (chains * kBlocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (a.ckpt_every < kGroup || a.ckpt_every > kMaxCkptEvery ||
      (a.ckpt_every & (a.ckpt_every - 1)) != 0)
    return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)(chains * kBlocks);
  const size_t xs_bytes = (size_t)kGroup * D * kCols * sizeof(float);
  auto bwd = a.bf16 ? kda_bwd_kernel<true> : kda_bwd_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(bwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)xs_bytes);
  if (e != cudaSuccess) return e;
  if (a.bf16)
    kda_bwd_ckpt_kernel<true><<<grid, kThreads, 0, stream>>>(a.k, a.v, a.log_alpha, a.beta,
                                                            a.init_state, a.cu_seqlens, a.n_seqs,
                                                            a.n_tokens, a.H, a.ckpt_every, a.ckpt,
                                                            a.status);
  else
    kda_bwd_ckpt_kernel<false><<<grid, kThreads, 0, stream>>>(a.k, a.v, a.log_alpha, a.beta,
                                                             a.init_state, a.cu_seqlens, a.n_seqs,
                                                             a.n_tokens, a.H, a.ckpt_every, a.ckpt,
                                                             a.status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd<<<grid, kThreads, xs_bytes, stream>>>(a.q, a.k, a.v, a.log_alpha, a.beta, a.cu_seqlens,
                                            a.n_seqs, a.n_tokens, a.H, a.ckpt_every, a.ckpt, a.d_out,
                                            a.d_final, a.dq_acc, a.dk_acc, a.dv, a.d_log_alpha,
                                            a.d_beta, a.d_init);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n = a.n_tokens * a.H * D;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
  if (a.bf16)
    kda_bwd_finish_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(a.dq_acc, a.dk_acc, a.dq,
                                                                     a.dk, n);
  else
    kda_bwd_finish_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(a.dq_acc, a.dk_acc, a.dq,
                                                                      a.dk, n);
  return cudaGetLastError();
}

}  // namespace kda
