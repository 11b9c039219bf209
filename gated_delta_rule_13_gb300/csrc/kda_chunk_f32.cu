// fp32 chunkwise KDA prefill on CUDA cores (fp32 inputs, fp32 arithmetic).
//
// One CTA carries one (sequence, head) chain through chunks of C = 32 tokens,
// fp32 throughout, so it serves fp32 callers that need ~1e-4 agreement with the
// exact recurrence.
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
//
// Decay ratios.  e^{g_r - g_i} is split at the chunk's middle row m:
// E_r = e^{g_r - g_m} and Ei_i = e^{g_m - g_i}, each one accurate expf, and
// e^{g_r - g_i} = E_r Ei_i.  With log_alpha >= -5 (the K3 bound; "Kimi K3:
// 架构、训练与系统全景解析", section 4.2.5) each factor lies within e^{+-80}, far
// inside fp32, and for i <= r their product is the ratio itself (<= 1); the
// arguments are clamped at 80 so that inputs outside the bound stay finite.
// The products are register-tiled: every thread owns a small output tile and
// streams the shared contraction dimension.
//
// The value columns of S evolve independently (every key-side quantity above is
// shared by all of them), so a chain may be split over P = 128 / NVS CTAs, each
// carrying NVS value columns of S, U, Delta and O and repeating the key-side
// work; they exchange nothing.  With few chains (a single long sequence) this
// runs P CTAs side by side instead of one.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int D = kHeadDim;
constexpr int C = kChunkF32;
constexpr int kThreads = 256;
constexpr int PR = D + 4;   // pitch of row-streamed [C][D] arrays (16-byte aligned rows)
constexpr int PC = D + 1;   // pitch of column-walked [C][D] arrays (conflict-free columns)
constexpr int PT = C + 4;   // pitch of the C x C matrices (16-byte aligned rows)
constexpr float kMaxArg = 80.f;
static_assert(C == 32 && kThreads == 256, "the tilings below assume C = 32 and 256 threads");

template <int NVS>
struct F32Smem {
  static constexpr int PV = NVS + 4;  // pitch of the value-column arrays
  float S[D][NVS];   // the CTA's value columns of the state [key c][value n]
  float qe[C][PR];   // q, then q o E
  float ke[C][PR];   // k o E
  float kei[C][PC];  // k, then k o Ei
  float kd[C][PR];   // Kdec = K o e^{g_C - g}
  float v[C][PV];    // v (the CTA's columns)
  float g[C][PR];    // log_alpha, then the cumulative log-decay
  float w[C][PR];    // W = T' (K o e^g)
  float u[C][PV];    // U = T' V, then Delta (the CTA's columns)
  float At[C][PT];   // A^T (beta-scaled, strictly lower A)
  float Pm[C][PT];   // P (lower incl. diagonal)
  float Tp[C][PT];   // T' = T Diag(beta)
  float beta[C];
  float egm[D];      // e^{g_m}
  float egc[D];      // e^{g_C}
  float egcm[D];     // e^{g_C - g_m}
  float gm[D];       // g_m
};

// With a split chain (NVS < 128) the next chunk's raw inputs also fit: copied
// by asynchronous 16-byte copies while the current chunk computes.
template <int NVS>
struct F32Ahead {
  float q[C][D], k[C][D], la[C][D];
  float v[C][NVS];
  float beta[C];
};
template <int NVS> constexpr bool kF32Ahead = NVS < D;
template <int NVS>
constexpr size_t f32_smem_bytes() {
  return sizeof(F32Smem<NVS>) + (kF32Ahead<NVS> ? sizeof(F32Ahead<NVS>) : 0);
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ void record_error(DeviceStatus *st, int code, int detail, int chain, int chunk) {
  if (atomicCAS(&st->code, 0, code) == 0) {
    st->detail = detail;
    st->chain = chain;
    st->chunk = chunk;
  }
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 x) { *reinterpret_cast<float4 *>(p) = x; }

template <int NVS>
__global__ void __launch_bounds__(kThreads, 1)
kda_chunk_fwd_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                         const float *__restrict__ v, const float *__restrict__ log_alpha,
                         const float *__restrict__ beta, const float *__restrict__ init_state,
                         const int32_t *__restrict__ cu_seqlens, int32_t n_seqs,
                         int64_t n_tokens, int32_t H, float *__restrict__ out,
                         float *__restrict__ final_state, DeviceStatus *status) {
  static_assert(NVS == 32 || NVS == 64 || NVS == 128, "value columns per CTA");
  constexpr int P = D / NVS;        // CTAs per chain
  constexpr int RT = NVS / 32;      // rows of a thread's C x NVS output tile (4 columns)
  constexpr int KT = NVS / 8;       // key rows of a thread's D x NVS state tile (4 columns)
  constexpr int NG = NVS / 4;       // 4-column groups of the CTA's value columns
  extern __shared__ __align__(16) unsigned char smem_raw[];
  F32Smem<NVS> &sm = *reinterpret_cast<F32Smem<NVS> *>(smem_raw);
  F32Ahead<NVS> &ah = *reinterpret_cast<F32Ahead<NVS> *>(smem_raw + sizeof(F32Smem<NVS>));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chain = blockIdx.x / P, nb = NVS * (blockIdx.x % P);  // chain, first value column
  const int seq = chain / H, h = chain % H;

  const int64_t t0 = cu_seqlens[seq], t1 = cu_seqlens[seq + 1];
  const bool bad = t0 < 0 || t1 < t0 || t1 > n_tokens ||
                   (chain == 0 && (cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != n_tokens));
  if (bad) {
    if (tid == 0) record_error(status, KDA_ERR_INVALID_ARG, 1, chain, -1);
    return;
  }

  const int64_t sbase = ((int64_t)seq * H + h) * D * D;
  for (int e = tid; e < D * NVS; e += kThreads)
    sm.S[e / NVS][e % NVS] = init_state ? init_state[sbase + (e / NVS) * D + nb + e % NVS] : 0.f;

  const int64_t len = t1 - t0;
  // the raw inputs of the valid rows of the chunk at c0, copied ahead
  auto issue_ahead = [&](int64_t c0) {
    const int64_t rem = len - c0;
    const int nv = rem < C ? (int)rem : C;
    for (int e = tid; e < C * (D / 4); e += kThreads) {
      const int r = e / (D / 4), c = 4 * (e % (D / 4));
      if (r < nv) {
        const int64_t off = ((t0 + c0 + r) * H + h) * D + c;
        cp_async16(&ah.q[r][c], q + off);
        cp_async16(&ah.k[r][c], k + off);
        cp_async16(&ah.la[r][c], log_alpha + off);
      }
    }
    for (int e = tid; e < C * (NVS / 4); e += kThreads) {
      const int r = e / (NVS / 4), n = 4 * (e % (NVS / 4));
      if (r < nv) cp_async16(&ah.v[r][n], v + ((t0 + c0 + r) * H + h) * D + nb + n);
    }
    if (tid < nv) cp_async4(&ah.beta[tid], beta + (t0 + c0 + tid) * H + h);
    cp_async_commit();
  };
  if constexpr (kF32Ahead<NVS>) {
    if (len > 0) issue_ahead(0);
  }
  for (int64_t c0 = 0; c0 < len; c0 += C) {
    const int64_t rem = len - c0;
    const int nv = rem < C ? (int)rem : C;
    // ---- load the chunk (rows >= nv: zero, beta = 0, log_alpha = 0)
    if constexpr (kF32Ahead<NVS>) {
      cp_async_commit_wait_all();  // this thread's copies of the chunk
      __syncthreads();             // everyone's
      for (int e = tid; e < C * D; e += kThreads) {
        const int r = e / D, c = e % D;
        const bool ok = r < nv;
        sm.qe[r][c] = ok ? ah.q[r][c] : 0.f;
        sm.kei[r][c] = ok ? ah.k[r][c] : 0.f;
        sm.g[r][c] = ok ? ah.la[r][c] : 0.f;
      }
      for (int e = tid; e < C * NVS; e += kThreads) {
        const int r = e / NVS, n = e % NVS;
        sm.v[r][n] = r < nv ? ah.v[r][n] : 0.f;
      }
      if (tid < C) sm.beta[tid] = tid < nv ? ah.beta[tid] : 0.f;
      __syncthreads();             // the ahead buffers are free
      if (c0 + C < len) issue_ahead(c0 + C);
    } else {
      for (int e = tid; e < C * D; e += kThreads) {
        const int r = e / D, c = e % D;
        const bool ok = r < nv;
        const int64_t off = ((t0 + c0 + r) * H + h) * D + c;
        sm.qe[r][c] = ok ? q[off] : 0.f;
        sm.kei[r][c] = ok ? k[off] : 0.f;
        sm.g[r][c] = ok ? log_alpha[off] : 0.f;
      }
      for (int e = tid; e < C * NVS; e += kThreads) {
        const int r = e / NVS, n = e % NVS;
        sm.v[r][n] = r < nv ? v[((t0 + c0 + r) * H + h) * D + nb + n] : 0.f;
      }
      if (tid < C) sm.beta[tid] = tid < nv ? beta[(t0 + c0 + tid) * H + h] : 0.f;
    }
    __syncthreads();
    // ---- within-chunk cumulative log-decay per key channel, its middle and end
    if (tid < D) {
      float acc = 0.f, mid = 0.f;
      for (int r = 0; r < C; ++r) {
        acc += sm.g[r][tid];
        sm.g[r][tid] = acc;
        if (r == C / 2 - 1) mid = acc;
      }
      sm.gm[tid] = mid;
      sm.egm[tid] = expf(mid);
      sm.egc[tid] = expf(acc);
      sm.egcm[tid] = expf(acc - mid);
    }
    __syncthreads();
    // ---- the split decay factors: K o E, Q o E, K o Ei
    for (int e = tid; e < C * D; e += kThreads) {
      const int r = e / D, c = e % D;
      const float x = sm.g[r][c] - sm.gm[c];
      const float E = expf(fminf(x, kMaxArg)), Ei = expf(fminf(-x, kMaxArg));
      const float kr = sm.kei[r][c];
      sm.ke[r][c] = kr * E;
      sm.qe[r][c] *= E;
      sm.kei[r][c] = kr * Ei;
      sm.kd[r][c] = kr * Ei * sm.egcm[c];
    }
    __syncthreads();
    // ---- A (strictly lower, beta-scaled; stored transposed) and P (lower incl.):
    // thread tile rows r0, r0 + 1 x columns i0, i0 + 1
    {
      const int r0 = 2 * (tid >> 4), i0 = 2 * (tid & 15);
      float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
      float p00 = 0.f, p01 = 0.f, p10 = 0.f, p11 = 0.f;
      if (i0 <= r0 + 1) {
#pragma unroll 8
        for (int c = 0; c < D; ++c) {
          const float k0 = sm.ke[r0][c], k1 = sm.ke[r0 + 1][c];
          const float q0 = sm.qe[r0][c], q1 = sm.qe[r0 + 1][c];
          const float x0 = sm.kei[i0][c], x1 = sm.kei[i0 + 1][c];
          a00 = fmaf(k0, x0, a00); a01 = fmaf(k0, x1, a01);
          a10 = fmaf(k1, x0, a10); a11 = fmaf(k1, x1, a11);
          p00 = fmaf(q0, x0, p00); p01 = fmaf(q0, x1, p01);
          p10 = fmaf(q1, x0, p10); p11 = fmaf(q1, x1, p11);
        }
      }
      const float b0 = sm.beta[r0], b1 = sm.beta[r0 + 1];
      sm.At[i0][r0] = i0 < r0 ? b0 * a00 : 0.f;
      sm.At[i0 + 1][r0] = i0 + 1 < r0 ? b0 * a01 : 0.f;
      sm.At[i0][r0 + 1] = i0 < r0 + 1 ? b1 * a10 : 0.f;
      sm.At[i0 + 1][r0 + 1] = i0 + 1 < r0 + 1 ? b1 * a11 : 0.f;
      sm.Pm[r0][i0] = i0 <= r0 ? p00 : 0.f;
      sm.Pm[r0][i0 + 1] = i0 + 1 <= r0 ? p01 : 0.f;
      sm.Pm[r0 + 1][i0] = i0 <= r0 + 1 ? p10 : 0.f;
      sm.Pm[r0 + 1][i0 + 1] = i0 + 1 <= r0 + 1 ? p11 : 0.f;
    }
    __syncthreads();
    // ---- T = (I + A)^{-1} by column-oriented forward substitution (warp 0,
    // lane j owns column j: once t[m] is final it is eliminated from every later
    // row), then T' = T Diag(beta)
    if (warp == 0) {
      const int j = lane;
      float t[C];
#pragma unroll
      for (int r = 0; r < C; ++r) t[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < C - 1; ++m) {
        const float tm = t[m];
#pragma unroll
        for (int r4 = 0; r4 < C / 4; ++r4) {
          if (4 * r4 + 3 <= m) continue;
          const float4 a = ld4(&sm.At[m][4 * r4]);
          const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int z = 0; z < 4; ++z)
            if (4 * r4 + z > m) t[4 * r4 + z] = fmaf(-av[z], tm, t[4 * r4 + z]);
        }
      }
      const float bj = sm.beta[j];
#pragma unroll
      for (int r = 0; r < C; ++r) sm.Tp[r][j] = t[r] * bj;
    }
    __syncthreads();
    // ---- W = T' (K o e^g): thread tile rows r0..r0+3 x key columns k0..k0+3;
    // U = T' V: rows ru..ru+RT-1 x the CTA's value columns nu..nu+3
    {
      const int r0 = 4 * warp, k0 = 4 * lane;
      const float4 em = ld4(&sm.egm[k0]);
      float4 w[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) w[a] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i <= r0 + 3; ++i) {
        float4 kt = ld4(&sm.ke[i][k0]);
        kt.x *= em.x; kt.y *= em.y; kt.z *= em.z; kt.w *= em.w;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float tp = sm.Tp[r0 + a][i];
          w[a].x = fmaf(tp, kt.x, w[a].x); w[a].y = fmaf(tp, kt.y, w[a].y);
          w[a].z = fmaf(tp, kt.z, w[a].z); w[a].w = fmaf(tp, kt.w, w[a].w);
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) st4(&sm.w[r0 + a][k0], w[a]);
      const int ru = RT * (tid / NG), nu = 4 * (tid % NG);
      float4 u[RT];
#pragma unroll
      for (int a = 0; a < RT; ++a) u[a] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i <= ru + RT - 1; ++i) {
        const float4 vv = ld4(&sm.v[i][nu]);
#pragma unroll
        for (int a = 0; a < RT; ++a) {
          const float tp = sm.Tp[ru + a][i];
          u[a].x = fmaf(tp, vv.x, u[a].x); u[a].y = fmaf(tp, vv.y, u[a].y);
          u[a].z = fmaf(tp, vv.z, u[a].z); u[a].w = fmaf(tp, vv.w, u[a].w);
        }
      }
#pragma unroll
      for (int a = 0; a < RT; ++a) st4(&sm.u[ru + a][nu], u[a]);
    }
    __syncthreads();
    // ---- Delta = U - W S and O_inter = (Q o e^g) S: thread tile rows
    // r0..r0+RT-1 x the CTA's value columns n0..n0+3; then O = O_inter + P Delta
    {
      const int r0 = RT * (tid / NG), n0 = 4 * (tid % NG);
      float4 dl[RT], oi[RT];
#pragma unroll
      for (int a = 0; a < RT; ++a) dl[a] = oi[a] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int c = 0; c < D; ++c) {
        const float4 s4 = ld4(&sm.S[c][n0]);
        const float em = sm.egm[c];
#pragma unroll
        for (int a = 0; a < RT; ++a) {
          const float wv = sm.w[r0 + a][c], qv = sm.qe[r0 + a][c] * em;
          dl[a].x = fmaf(wv, s4.x, dl[a].x); dl[a].y = fmaf(wv, s4.y, dl[a].y);
          dl[a].z = fmaf(wv, s4.z, dl[a].z); dl[a].w = fmaf(wv, s4.w, dl[a].w);
          oi[a].x = fmaf(qv, s4.x, oi[a].x); oi[a].y = fmaf(qv, s4.y, oi[a].y);
          oi[a].z = fmaf(qv, s4.z, oi[a].z); oi[a].w = fmaf(qv, s4.w, oi[a].w);
        }
      }
      __syncthreads();  // every thread has read W and U's rows it needs
#pragma unroll
      for (int a = 0; a < RT; ++a) {
        float4 uu = ld4(&sm.u[r0 + a][n0]);
        uu.x -= dl[a].x; uu.y -= dl[a].y; uu.z -= dl[a].z; uu.w -= dl[a].w;
        st4(&sm.u[r0 + a][n0], uu);
      }
      __syncthreads();  // Delta complete
      for (int i = 0; i <= r0 + RT - 1; ++i) {
        const float4 d4 = ld4(&sm.u[i][n0]);
#pragma unroll
        for (int a = 0; a < RT; ++a) {
          const float pv = sm.Pm[r0 + a][i];
          oi[a].x = fmaf(pv, d4.x, oi[a].x); oi[a].y = fmaf(pv, d4.y, oi[a].y);
          oi[a].z = fmaf(pv, d4.z, oi[a].z); oi[a].w = fmaf(pv, d4.w, oi[a].w);
        }
      }
#pragma unroll
      for (int a = 0; a < RT; ++a)
        if (r0 + a < nv) st4(out + ((t0 + c0 + r0 + a) * H + h) * D + nb + n0, oi[a]);
    }
    // ---- S <- Diag(e^{g_C}) S + Kdec^T Delta: thread tile key rows
    // k0..k0+KT-1 x the CTA's value columns n0..n0+3
    {
      const int k0 = KT * (tid / NG), n0 = 4 * (tid % NG);
      float4 acc[KT];
#pragma unroll
      for (int j = 0; j < KT; ++j) {
        const float4 s4 = ld4(&sm.S[k0 + j][n0]);
        const float gc = sm.egc[k0 + j];
        acc[j] = make_float4(s4.x * gc, s4.y * gc, s4.z * gc, s4.w * gc);
      }
      for (int i = 0; i < C; ++i) {
        const float4 d4 = ld4(&sm.u[i][n0]);
#pragma unroll
        for (int j = 0; j < KT; ++j) {
          const float kd = sm.kd[i][k0 + j];
          acc[j].x = fmaf(kd, d4.x, acc[j].x); acc[j].y = fmaf(kd, d4.y, acc[j].y);
          acc[j].z = fmaf(kd, d4.z, acc[j].z); acc[j].w = fmaf(kd, d4.w, acc[j].w);
        }
      }
#pragma unroll
      for (int j = 0; j < KT; ++j) st4(&sm.S[k0 + j][n0], acc[j]);
    }
    __syncthreads();
  }
  if (final_state) {
    for (int e = tid; e < D * NVS; e += kThreads)
      final_state[sbase + (e / NVS) * D + nb + e % NVS] = sm.S[e / NVS][e % NVS];
  }
}

template <int NVS>
cudaError_t launch_f32(const ChunkArgs &a, int64_t chains, cudaStream_t stream) {
  const int64_t ctas = chains * (D / NVS);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  const size_t smem = f32_smem_bytes<NVS>();
  cudaError_t e = cudaFuncSetAttribute(kda_chunk_fwd_f32_kernel<NVS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kda_chunk_fwd_f32_kernel<NVS><<<(unsigned)ctas, kThreads, smem, stream>>>(
      static_cast<const float *>(a.q), static_cast<const float *>(a.k),
      static_cast<const float *>(a.v), a.log_alpha, a.beta, a.init_state, a.cu_seqlens,
      a.n_seqs, a.n_tokens, a.H, static_cast<float *>(a.out), a.final_state, a.status);
  return cudaGetLastError();
}

}  // namespace

// CTAs per chain: as many as fit the device's SMs beside the other chains (4,
// 2 or 1; each CTA repeats the chain's key-side work).
cudaError_t launch_chunk_fwd_f32(const ChunkArgs &a, cudaStream_t stream) {
  const int64_t chains = (int64_t)a.n_seqs * a.H;
  if (chains == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 0;
  }
  if (4 * chains <= sms) return launch_f32<32>(a, chains, stream);
  if (2 * chains <= sms) return launch_f32<64>(a, chains, stream);
  return launch_f32<128>(a, chains, stream);
}

}  // namespace kda
