// fp32 chunkwise KDA prefill on CUDA cores (fp32 inputs, fp32 arithmetic).
//
// This is the plain chunk algebra with no tile factorisation of the decay: every
// decay ratio exp(g_r - g_i) is evaluated directly, so it serves fp32 callers
// that need ~1e-4 agreement with the exact recurrence.  One CTA carries one
// (sequence, head) chain through chunks of C = 32 tokens.
//
// Chunk algebra (plainest reading of "Kimi K3: 架构、训练与系统全景解析",
// section 4.2.4: state passed across chunks, lower-triangular matrix products
// inside, output = pre-chunk-state term + intra-chunk causal term), with g_r the
// within-chunk cumulative log-decay per key channel (g_0 = 0), S the incoming
// state, D_r = Diag(alpha_r):
//   S_r = D_r S_{r-1} + k_r d_r^T,  d_r = beta_r (v_r - (D_r S_{r-1})^T k_r).
// Unrolling,
//   A_ri = beta_r sum_c k_rc k_ic e^{g_rc - g_ic}  (i < r),  T = (I + A)^{-1}
//   W = T Diag(beta) (K o e^{g}),  U = T Diag(beta) V,  Delta = U - W S
//   P_ri = sum_c q_rc k_ic e^{g_rc - g_ic}          (i <= r)
//   O = (Q o e^{g}) S + P Delta
//   S <- Diag(e^{g_C}) S + (K o e^{g_C - g})^T Delta.
// Rows past the end of a sequence get beta = 0 and log_alpha = 0, which makes
// their Delta rows zero and leaves g constant, so a partial chunk needs no
// other special case.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int D = kHeadDim;
constexpr int C = kChunkF32;
constexpr int P = D + 1;  // padded pitch: column walks over rows are conflict-free
constexpr int kThreads = 256;

struct F32Smem {
  float S[D][D];   // state [key c][value n]
  float q[C][P];   // q, then q o e^{g}
  float k[C][P];   // k, then k o e^{g}
  float v[C][P];
  float g[C][P];   // log_alpha, then cumulative log-decay, then O
  float w[C][P];   // W
  float u[C][P];   // U, then Delta
  float kd[C][P];  // k o e^{g_C - g}
  float A[C][C + 1];
  float Pm[C][C + 1];
  float T[C][C + 1];  // T Diag(beta)
  float beta[C];
  float gC[D];
};

__device__ void record_error(DeviceStatus *st, int code, int detail, int chain, int chunk) {
  if (atomicCAS(&st->code, 0, code) == 0) {
    st->detail = detail;
    st->chain = chain;
    st->chunk = chunk;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
kda_chunk_fwd_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                         const float *__restrict__ v, const float *__restrict__ log_alpha,
                         const float *__restrict__ beta, const float *__restrict__ init_state,
                         const int32_t *__restrict__ cu_seqlens, int32_t n_seqs,
                         int64_t n_tokens, int32_t H, float *__restrict__ out,
                         float *__restrict__ final_state, DeviceStatus *status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  F32Smem &sm = *reinterpret_cast<F32Smem *>(smem_raw);
  const int tid = threadIdx.x;
  const int chain = blockIdx.x;
  const int seq = chain / H, h = chain % H;

  const int64_t t0 = cu_seqlens[seq], t1 = cu_seqlens[seq + 1];
  const bool bad = t0 < 0 || t1 < t0 || t1 > n_tokens ||
                   (chain == 0 && (cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != n_tokens));
  if (bad) {
    if (tid == 0) record_error(status, KDA_ERR_INVALID_ARG, 1, chain, -1);
    return;
  }

  const int64_t sbase = ((int64_t)seq * H + h) * D * D;
  for (int e = tid; e < D * D; e += kThreads)
    (&sm.S[0][0])[e] = init_state ? init_state[sbase + e] : 0.f;

  const int64_t len = t1 - t0;
  for (int64_t c0 = 0; c0 < len; c0 += C) {
    const int64_t rem = len - c0;
    const int nv = rem < C ? (int)rem : C;
    // ---- load the chunk (rows >= nv: zero, beta = 0, log_alpha = 0)
    for (int e = tid; e < C * D; e += kThreads) {
      const int r = e / D, c = e % D;
      const bool ok = r < nv;
      const int64_t off = ((t0 + c0 + r) * H + h) * D + c;
      sm.q[r][c] = ok ? q[off] : 0.f;
      sm.k[r][c] = ok ? k[off] : 0.f;
      sm.v[r][c] = ok ? v[off] : 0.f;
      sm.g[r][c] = ok ? log_alpha[off] : 0.f;
    }
    if (tid < C) sm.beta[tid] = tid < nv ? beta[(t0 + c0 + tid) * H + h] : 0.f;
    __syncthreads();
    // ---- within-chunk cumulative log-decay per key channel
    if (tid < D) {
      float acc = 0.f;
      for (int r = 0; r < C; ++r) {
        acc += sm.g[r][tid];
        sm.g[r][tid] = acc;
      }
      sm.gC[tid] = acc;
    }
    __syncthreads();
    // ---- A (strictly lower, beta-scaled) and P (lower incl. diagonal)
    for (int e = tid; e < C * C; e += kThreads) {
      const int r = e / C, i = e % C;
      float a = 0.f, p = 0.f;
      if (i <= r) {
        for (int c = 0; c < D; ++c) {
          const float ki = sm.k[i][c] * expf(sm.g[r][c] - sm.g[i][c]);
          a = fmaf(sm.k[r][c], ki, a);
          p = fmaf(sm.q[r][c], ki, p);
        }
      }
      sm.A[r][i] = i < r ? sm.beta[r] * a : 0.f;
      sm.Pm[r][i] = p;
    }
    __syncthreads();
    // ---- T = (I + A)^{-1} by forward substitution; lane j owns column j.
    if (tid < 32) {
      const int j = tid;
      float tcol[C];
#pragma unroll
      for (int r = 0; r < C; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < r; ++m) acc = fmaf(sm.A[r][m], tcol[m], acc);
        tcol[r] = (j == r) ? 1.f : (j < r ? -acc : 0.f);
      }
      const float bj = sm.beta[j];
#pragma unroll
      for (int r = 0; r < C; ++r) sm.T[r][j] = tcol[r] * bj;
    }
    // ---- decay-weighted operands (P already used the raw q, k)
    for (int e = tid; e < C * D; e += kThreads) {
      const int r = e / D, c = e % D;
      const float g = sm.g[r][c];
      const float kr = sm.k[r][c];
      sm.kd[r][c] = kr * expf(sm.gC[c] - g);
      sm.k[r][c] = kr * expf(g);
      sm.q[r][c] *= expf(g);
    }
    __syncthreads();
    // ---- W = T' (K o e^g), U = T' V
    for (int e = tid; e < C * D; e += kThreads) {
      const int r = e / D, c = e % D;
      float w = 0.f, u = 0.f;
      for (int i = 0; i <= r; ++i) {
        const float t = sm.T[r][i];
        w = fmaf(t, sm.k[i][c], w);
        u = fmaf(t, sm.v[i][c], u);
      }
      sm.w[r][c] = w;
      sm.u[r][c] = u;
    }
    __syncthreads();
    // ---- Delta = U - W S and O_inter = (Q o e^g) S
    for (int e = tid; e < C * D; e += kThreads) {
      const int r = e / D, n = e % D;
      float ws = 0.f, qs = 0.f;
      for (int c = 0; c < D; ++c) {
        const float s = sm.S[c][n];
        ws = fmaf(sm.w[r][c], s, ws);
        qs = fmaf(sm.q[r][c], s, qs);
      }
      sm.u[r][n] -= ws;
      sm.g[r][n] = qs;
    }
    __syncthreads();
    // ---- O = O_inter + P Delta (valid rows only)
    for (int e = tid; e < C * D; e += kThreads) {
      const int r = e / D, n = e % D;
      if (r < nv) {
        float o = sm.g[r][n];
        for (int i = 0; i <= r; ++i) o = fmaf(sm.Pm[r][i], sm.u[i][n], o);
        out[((t0 + c0 + r) * H + h) * D + n] = o;
      }
    }
    // ---- S <- Diag(e^{g_C}) S + Kdec^T Delta
    for (int e = tid; e < D * D; e += kThreads) {
      const int c = e / D, n = e % D;
      float s = sm.S[c][n] * expf(sm.gC[c]);
      for (int i = 0; i < C; ++i) s = fmaf(sm.kd[i][c], sm.u[i][n], s);
      sm.S[c][n] = s;
    }
    __syncthreads();
  }
  if (final_state) {
    for (int e = tid; e < D * D; e += kThreads) final_state[sbase + e] = (&sm.S[0][0])[e];
  }
}

}  // namespace

cudaError_t launch_chunk_fwd_f32(const ChunkArgs &a, cudaStream_t stream) {
  const int64_t chains = (int64_t)a.n_seqs * a.H;
  if (chains == 0) return cudaSuccess;
  if (chains > 0x7fffffffLL) return cudaErrorInvalidValue;
  const size_t smem = sizeof(F32Smem);
  cudaError_t e = cudaFuncSetAttribute(kda_chunk_fwd_f32_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kda_chunk_fwd_f32_kernel<<<(unsigned)chains, kThreads, smem, stream>>>(
      static_cast<const float *>(a.q), static_cast<const float *>(a.k),
      static_cast<const float *>(a.v), a.log_alpha, a.beta, a.init_state, a.cu_seqlens,
      a.n_seqs, a.n_tokens, a.H, static_cast<float *>(a.out), a.final_state, a.status);
  return cudaGetLastError();
}

}  // namespace kda
