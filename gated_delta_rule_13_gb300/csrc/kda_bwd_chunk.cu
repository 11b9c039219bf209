// Chunked backward pass of the KDA recurrence for bf16 inputs: 16-token chunks,
// every product on the tensor cores (warp-level bf16 MMAs, fp32 accumulation).
//
// The pages give no gradient ("Kimi K3: 架构、训练与系统全景解析", section 7.1:
// the chunked KDA kernel serves training as well as prefill).  This is the
// chain rule through the chunk form of the update and read-out ("Kimi K3" study
// notes, section 3-2 "2) Kimi Delta Attention"; 全景解析 sections 4.2.4-4.2.5 for
// the chunk form).  Per chunk of n <= 16 tokens (rows r, i), padded to 16 with
// k = q = v = dO = 0, log_alpha = 0, beta = 0, with g_r the cumulative
// log_alpha through row r, the middle row m = 7 as the decay reference and
// l = 15 the last row (padding leaves g_l = g_{n-1}):
//   Kt = K e^{g - g_m}, Qt = Q e^{g - g_m}, Kh = K e^{g_m - g}, Kd = K e^{g_l - g}
//   Ks = K e^{g}, Qs = Q e^{g}            (each factor within e^{+-40} or <= 1)
//   G = Kt Kh^T, A = tril(Diag(beta) G, -1), P = tril(Qt Kh^T), T = (I + A)^{-1}
//   R = V - Ks S, U = Diag(beta) R, delta = T U
//   S' = Diag(e^{g_l}) S + Kd^T delta,   O = Qs S + P delta
// and in reverse, from dS' (the gradient of S') and dO:
//   d delta = P^T dO + Kd dS',  dU = T^T d delta,  dR = Diag(beta) dU = dv
//   dA = tril(-dU delta^T, -1),  dP = tril(dO delta^T),  dG = Diag(beta) dA
//   dbeta = rowsum(R o dU) + rowsum(dA o G)
//   dKt = -e^{g_m} o (dR S^T) + dG Kh,   dQt = e^{g_m} o (dO S^T) + dP Kh
//   dKh = dG^T Kt + dP^T Qt,   dKd = delta dS'^T
//   X = Qs^T dO - Ks^T dR,   dS = Diag(e^{g_l}) dS' + X
//   dq = dQt e^{g - g_m},  dk = dKt e^{g - g_m} + dKh e^{g_m - g} + dKd e^{g_l - g}
//   dg = dKt o Kt + dQt o Qt - dKh o Kh - dKd o Kd,  then at row m
//        - colsum(dKt o Kt + dQt o Qt) + colsum(dKh o Kh) + rowsum_v(S o X)
//   and at row l  colsum(dKd o Kd) + e^{g_l} rowsum_v(S o dS'),
//   dlog_alpha_j = sum_{r >= j} dg_r (within the chunk).
// (Written out from the token form by hand and checked in fp64 against the
// gradient oracle on ragged lengths.)
//
// Work split: a chain (sequence, head) is one CTA of 8 warps, or, when the
// chains leave half the SMs idle, a cluster of two CTAs that take 64 value
// columns each (the columns of S evolve independently).  A CTA walks the
// chain's chunks from the last.  dS lives in registers as MMA accumulators
// (warp w: key rows 16 w .. 16 w + 15 of the CTA's value columns); the chunk's
// operands are bf16 tiles in shared memory, read by ldmatrix.  Value-side
// products give warp w an eighth of the CTA's value columns, key-side ones the
// keys 16 w .. 16 w + 15; the 16 x 16 products (G, P, dA, dP) run on warps 0-1
// and T = (I + A)^{-1} (forward substitution) on warp 0.  The key-side
// gradients (dq, dk, dlog_alpha, dbeta) are sums over the value columns: in a
// cluster each CTA computes its part for every key and sends the other CTA's
// key half through distributed shared memory, and each finishes its own half
// (own part + received part, in that order).  The state at every chunk start
// comes from the checkpoint pass (states every 16 tokens).  Every gradient
// element is written once: no atomics, results independent of scheduling.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"


namespace kda {
namespace {

using namespace sm100;

constexpr int D = kHeadDim;    // 128
constexpr int CB = kBwdChunk;  // 16 tokens per chunk
constexpr int kMid = 7;        // reference row of the decay factors
constexpr int kLast = CB - 1;
constexpr int kThreads = 256;
constexpr int TP = D + 8;      // bf16 pitch of 128-wide tiles: 272 B, ldmatrix conflict free
constexpr int SP = CB + 8;     // bf16 pitch of 16-wide tiles: 48 B
constexpr int GP = CB + 1;     // fp32 pitch of the 16 x 16 matrices

// Shared memory of the reverse pass for NV value columns per CTA (128, or 64
// in a two-CTA cluster).  Value-width tiles have pitch NV + 8.
template <int NV>
struct __align__(16) Smem {
  static constexpr int VP = NV + 8;
  __nv_bfloat16 S[D][VP];     // the state at the chunk start (bf16 checkpoint), this CTA's columns
  __nv_bfloat16 dSn[D][VP];   // dS' (gradient of the chunk-end state), bf16
  __nv_bfloat16 dSlo[D][VP];  // dS' - dSn, bf16: the pair carries dS' to ~2^-16
  __nv_bfloat16 q[CB][TP], k[CB][TP];       // raw inputs, every key
  __nv_bfloat16 v[CB][VP], dout[CB][VP];    // raw inputs, this CTA's value columns
  __nv_bfloat16 kt[CB][TP], qt[CB][TP], kh[CB][TP], kd[CB][TP], ks[CB][TP], qs[CB][TP];
  __nv_bfloat16 u[CB][VP], dl[CB][VP], ddl[CB][VP], du[CB][VP], ndr[CB][VP];
  __nv_bfloat16 tm[CB][SP], pm[CB][SP], dgm[CB][SP], dpm[CB][SP];
  float la[CB][D];            // log_alpha rows
  float et[CB][D];            // e^{g_r - g_m}
  float dgr[CB][D];           // dg_r
  float G[CB][GP];
  float em[D], gam[D], t1[D], t2[D];
  float beta[CB];
  float dbp[8][CB];           // row sums of R o dU per warp
  float dba[CB];              // row sums of dA o G
  // from the other CTA of a cluster (by chunk parity): its parts of dq, dk
  // and dg for this CTA's 64 keys, and of dbeta
  alignas(16) float xin[NV < D ? 2 : 1][3][CB][64];
  alignas(16) float xdb[NV < D ? 2 : 1][CB];
};

__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t a, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(a));
}

// Fragment loads of the m16n8k16 operands from bf16 tiles (pitch in elements).
// A (16 x 16 at m0, k0) from a tile stored [m][k] ...
__device__ __forceinline__ void lda(const __nv_bfloat16 *tile, int pitch, int m0, int k0, int lane,
                                    uint32_t (&a)[4]) {
  ldsm_x4(smem_u32(tile + (m0 + (lane & 15)) * pitch + k0 + (lane >> 4) * 8), a);
}
// ... or stored [k][m].
__device__ __forceinline__ void lda_t(const __nv_bfloat16 *tile, int pitch, int m0, int k0,
                                      int lane, uint32_t (&a)[4]) {
  ldsm_x4_t(smem_u32(tile + (k0 + (lane & 7) + ((lane >> 4) << 3)) * pitch + m0 +
                     ((lane >> 3) & 1) * 8),
            a);
}
// B for two n-tiles (16 x 16 at k0, n0): b[0], b[1] for columns n0 .. n0 + 7,
// b[2], b[3] for n0 + 8 .. n0 + 15; from a tile stored [n][k] ...
__device__ __forceinline__ void ldb(const __nv_bfloat16 *tile, int pitch, int n0, int k0, int lane,
                                    uint32_t (&b)[4]) {
  ldsm_x4(smem_u32(tile + (n0 + (lane & 7) + ((lane >> 4) << 3)) * pitch + k0 +
                   ((lane >> 3) & 1) * 8),
          b);
}
// ... or stored [k][n].
__device__ __forceinline__ void ldb_t(const __nv_bfloat16 *tile, int pitch, int n0, int k0,
                                      int lane, uint32_t (&b)[4]) {
  ldsm_x4_t(smem_u32(tile + (k0 + (lane & 7) + ((lane >> 3) & 1) * 8) * pitch + n0 +
                     (lane >> 4) * 8),
            b);
}
// B for NT (1 or 2) n-tiles from a tile stored [k][n]: b[2 j], b[2 j + 1] for
// columns n0 + 8 j .. + 7.  (x2: lanes 0-15 give the addresses.)
template <int NT>
__device__ __forceinline__ void ldbv_t(const __nv_bfloat16 *tile, int pitch, int n0, int k0,
                                       int lane, uint32_t (&b)[2 * NT]) {
  if constexpr (NT == 2) {
    ldb_t(tile, pitch, n0, k0, lane, b);
  } else {
    ldsm_x2_t(smem_u32(tile + (k0 + (lane & 7) + ((lane >> 3) & 1) * 8) * pitch + n0), b);
  }
}
template <int NT>
__device__ __forceinline__ void mmav(float (&c)[NT][4], const uint32_t (&a)[4],
                                     const uint32_t (&b)[2 * NT]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) mma_bf16_16x8x16(c[j], a[0], a[1], a[2], a[3], b[2 * j], b[2 * j + 1]);
}
__device__ __forceinline__ void mma2(float (&c)[2][4], const uint32_t (&a)[4],
                                     const uint32_t (&b)[4]) {
  mmav<2>(c, a, b);
}
template <int NT>
__device__ __forceinline__ void zero(float (&c)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) c[j][i] = 0.f;
}
__device__ __forceinline__ void st_bf2(__nv_bfloat16 *p, float x, float y) {
  *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(x, y);
}
// Two bf16 global stores: the gradient outputs are only element aligned.
__device__ __forceinline__ void st_bf2_g(__nv_bfloat16 *p, float x, float y) {
  p[0] = __float2bfloat16_rn(x);
  p[1] = __float2bfloat16_rn(y);
}
__device__ __forceinline__ float2 ld_bf2(const __nv_bfloat16 *p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}
// Cluster helpers: the shared-memory address of the same variable in CTA
// `rank` of the cluster, an fp32 pair stored there, and the cluster barrier.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float x) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(x) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Rows tb .. tb + n - 1, columns col0 .. col0 + 8 S8 - 1 of head h of a
// [N, H, 128] bf16 tensor into a [16][P] tile by 16-byte asynchronous copies;
// rows n .. 15 zero.
template <int P, int S8>
__device__ __forceinline__ void stage_rows(__nv_bfloat16 (*tile)[P], const __nv_bfloat16 *src,
                                           int64_t tb, int n, int h, int H, int col0, int tid) {
  for (int e = tid; e < CB * S8; e += kThreads) {
    const int r = e / S8, s8 = 8 * (e % S8);
    if (r < n) cp_async16(&tile[r][s8], src + ((tb + r) * H + h) * D + col0 + s8);
    else *reinterpret_cast<uint4 *>(&tile[r][s8]) = make_uint4(0u, 0u, 0u, 0u);
  }
}
// ... of an fp32 tensor (log_alpha) into [16][128] fp32.
__device__ __forceinline__ void stage_rows_f32(float (*tile)[D], const float *src, int64_t tb,
                                               int n, int h, int H, int tid) {
  for (int e = tid; e < CB * 32; e += kThreads) {
    const int r = e >> 5, s4 = 4 * (e & 31);
    if (r < n) cp_async16(&tile[r][s4], src + ((tb + r) * H + h) * D + s4);
    else *reinterpret_cast<float4 *>(&tile[r][s4]) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Decay factors of one key column c of a chunk from its log_alpha rows:
// g_r = cumulative sum (kept in log2 units), et_r = e^{g_r - g_m} (the one
// exponential per row, ex2 on the special-function unit, relative error below
// 2^-22), e^{g_m - g_r} = 1 / et_r, e^{g_l - g_r} = et_l / et_r,
// e^{g_r} = e^{g_m} et_r (each a product of factors within e^{+-40}).
struct ColFactors {
  float et[CB];
  float em, etl;  // e^{g_m}, e^{g_l - g_m}
};
__device__ __forceinline__ void col_factors(const float (*la)[D], int c, ColFactors &f) {
  constexpr float kLog2e = 1.4426950408889634f;
  float gr[CB];
  float acc = 0.f;
#pragma unroll
  for (int r = 0; r < CB; ++r) {
    acc = fmaf(la[r][c], kLog2e, acc);
    gr[r] = acc;
  }
  const float gm = gr[kMid];
#pragma unroll
  for (int r = 0; r < CB; ++r) f.et[r] = ex2(gr[r] - gm);
  f.em = ex2(gm);
  f.etl = f.et[kLast];
}

// The chain of block b and, in a cluster of VS = 128 / NV CTAs, the CTA's rank.
struct ChainOf {
  int seq, h, rank;
  int64_t t0, t1;
  bool ok;
};
template <int NV>
__device__ __forceinline__ ChainOf chain_of_block(const int32_t *cu, int32_t n_seqs,
                                                  int64_t n_tokens, int32_t H) {
  constexpr int VS = D / NV;
  ChainOf c;
  const int64_t u = blockIdx.x / VS;
  c.rank = (int)(blockIdx.x % VS);
  c.seq = (int)(u / H);
  c.h = (int)(u % H);
  c.t0 = cu[c.seq];
  c.t1 = cu[c.seq + 1];
  c.ok = c.t0 >= 0 && c.t1 >= c.t0 && c.t1 <= n_tokens &&
         (c.seq != 0 || (cu[0] == 0 && cu[n_seqs] == n_tokens));
  return c;
}

template <int NV>
__global__ void __launch_bounds__(kThreads, 1)
kda_bwd_chunk_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                     const __nv_bfloat16 *__restrict__ v, const float *__restrict__ la,
                     const float *__restrict__ beta, const int32_t *__restrict__ cu,
                     int32_t n_seqs, int64_t n_tokens, int32_t H,
                     const __nv_bfloat16 *__restrict__ ckpt, const __nv_bfloat16 *__restrict__ dout,
                     const float *__restrict__ d_final, __nv_bfloat16 *__restrict__ dq,
                     __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv,
                     float *__restrict__ d_la, float *__restrict__ d_beta,
                     float *__restrict__ d_init, DeviceStatus *status) {
  constexpr bool kPair = NV < D;   // two CTAs per chain (a cluster)
  constexpr int VP = Smem<NV>::VP;
  constexpr int NT = NV / 64;      // value n-tiles per warp: 2 or 1
  constexpr int NJ = NV / 8;       // value n-tiles of dS per thread
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem<NV> &sm = *reinterpret_cast<Smem<NV> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const ChainOf chn = chain_of_block<NV>(cu, n_seqs, n_tokens, H);
  if (!chn.ok) {  // both CTAs of a cluster see the same chain and leave together
    if (tid == 0) atomicCAS(&status->code, 0, 1 /* KDA_ERR_INVALID_ARG */);
    return;
  }
  const int seq = chn.seq, h = chn.h, rank = chn.rank;
  const int64_t t0 = chn.t0, t1 = chn.t1;
  const int vbase = NV * rank;  // this CTA's first value column
  const int kr0 = 16 * warp;    // this warp's key rows of dS, and its key columns
  const int nv0 = NV / 8 * warp;  // this warp's first (CTA-local) value column
  const int64_t sbase = ((int64_t)seq * H + h) * D * D;
  if constexpr (kPair) cluster_sync();  // both CTAs run before any remote store

  // dS (gradient of the state after the sequence), MMA accumulator layout:
  // ds[j] covers local value columns 8 j .. 8 j + 7 of key rows kr0 + g, + 8.
  float ds[NJ][4];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = vbase + 8 * j + 2 * t;
    ds[j][0] = ds[j][1] = ds[j][2] = ds[j][3] = 0.f;
    if (d_final) {
      const float *fa = d_final + sbase + (kr0 + g) * D + c, *fb = fa + 8 * D;
      ds[j][0] = fa[0];
      ds[j][1] = fa[1];
      ds[j][2] = fb[0];
      ds[j][3] = fb[1];
    }
  }

  const int64_t n_ch = (t1 - t0 + CB - 1) / CB;
  const int64_t slot0 = bwd_ckpt_slot_base(t0, seq, CB);
  // Inputs of chunk c arrive by asynchronous copies issued during chunk c + 1,
  // each tile as soon as chunk c + 1 has used it for the last time.
  auto chunk_len = [&](int64_t c) { return (int)(t1 - (t0 + CB * c) < CB ? t1 - (t0 + CB * c) : CB); };
  auto issue_qkl = [&](int64_t c) {
    const int64_t tb = t0 + CB * c;
    const int n = chunk_len(c);
    stage_rows<TP, 16>(sm.q, q, tb, n, h, H, 0, tid);
    stage_rows<TP, 16>(sm.k, k, tb, n, h, H, 0, tid);
    stage_rows_f32(sm.la, la, tb, n, h, H, tid);
  };
  auto issue_v = [&](int64_t c) {
    stage_rows<VP, NV / 8>(sm.v, v, t0 + CB * c, chunk_len(c), h, H, vbase, tid);
  };
  auto issue_rest = [&](int64_t c) {  // dO, beta and the state
    const int64_t tb = t0 + CB * c;
    const int n = chunk_len(c);
    stage_rows<VP, NV / 8>(sm.dout, dout, tb, n, h, H, vbase, tid);
    if (tid < CB) sm.beta[tid] = tid < n ? beta[(tb + tid) * H + h] : 0.f;
    const __nv_bfloat16 *Sg = ckpt + ((slot0 + c) * H + h) * (int64_t)(D * D) + vbase;
    for (int e = tid; e < D * (NV / 8); e += kThreads) {
      const int r = e / (NV / 8), s8 = 8 * (e % (NV / 8));
      cp_async16(&sm.S[r][s8], Sg + r * D + s8);
    }
  };
  if (n_ch > 0) {
    issue_qkl(n_ch - 1);
    issue_v(n_ch - 1);
    issue_rest(n_ch - 1);
  }
  for (int64_t ch = n_ch - 1; ch >= 0; --ch) {
    const int64_t tb = t0 + CB * ch;
    const int n = chunk_len(ch);
    const int par = (int)((n_ch - 1 - ch) & 1);
    cp_async_wait_all();
    __syncthreads();  // the chunk's inputs are in place; the previous chunk is done
    // rowsum_v(S o dS') over this CTA's value columns; dS' as a pair of bf16 tiles
    float p1a = 0.f, p1b = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int c = 8 * j + 2 * t;
      const float2 a = ld_bf2(&sm.S[kr0 + g][c]), b = ld_bf2(&sm.S[kr0 + g + 8][c]);
      p1a = fmaf(a.x, ds[j][0], fmaf(a.y, ds[j][1], p1a));
      p1b = fmaf(b.x, ds[j][2], fmaf(b.y, ds[j][3], p1b));
      const __nv_bfloat162 ha = __floats2bfloat162_rn(ds[j][0], ds[j][1]);
      const __nv_bfloat162 hb = __floats2bfloat162_rn(ds[j][2], ds[j][3]);
      *reinterpret_cast<__nv_bfloat162 *>(&sm.dSn[kr0 + g][c]) = ha;
      *reinterpret_cast<__nv_bfloat162 *>(&sm.dSn[kr0 + g + 8][c]) = hb;
      const float2 fa = __bfloat1622float2(ha), fb = __bfloat1622float2(hb);
      st_bf2(&sm.dSlo[kr0 + g][c], ds[j][0] - fa.x, ds[j][1] - fa.y);
      st_bf2(&sm.dSlo[kr0 + g + 8][c], ds[j][2] - fb.x, ds[j][3] - fb.y);
    }
    p1a += __shfl_xor_sync(0xffffffffu, p1a, 1);
    p1a += __shfl_xor_sync(0xffffffffu, p1a, 2);
    p1b += __shfl_xor_sync(0xffffffffu, p1b, 1);
    p1b += __shfl_xor_sync(0xffffffffu, p1b, 2);
    if (t == 0) {
      sm.t1[kr0 + g] = p1a;
      sm.t1[kr0 + g + 8] = p1b;
    }

    // ---- decay factors and the factor-scaled operands (thread: one key column;
    // threads 0-127 the k-derived tiles, 128-255 the q-derived ones)
    {
      const int c = tid & (D - 1);
      ColFactors f;
      col_factors(sm.la, c, f);
      if (tid < D) {
        sm.em[c] = f.em;
        sm.gam[c] = f.em * f.etl;
#pragma unroll
        for (int r = 0; r < CB; ++r) {
          const float kf = __bfloat162float(sm.k[r][c]);
          const float eh = __fdividef(1.0f, f.et[r]);
          sm.et[r][c] = f.et[r];
          sm.kt[r][c] = __float2bfloat16_rn(kf * f.et[r]);
          sm.kh[r][c] = __float2bfloat16_rn(kf * eh);
          sm.kd[r][c] = __float2bfloat16_rn(kf * (f.etl * eh));
          sm.ks[r][c] = __float2bfloat16_rn(kf * (f.em * f.et[r]));
        }
      } else {
#pragma unroll
        for (int r = 0; r < CB; ++r) {
          const float qf = __bfloat162float(sm.q[r][c]);
          sm.qt[r][c] = __float2bfloat16_rn(qf * f.et[r]);
          sm.qs[r][c] = __float2bfloat16_rn(qf * (f.em * f.et[r]));
        }
      }
    }
    __syncthreads();
    if (ch > 0) issue_qkl(ch - 1);  // q, k and log_alpha are used up

    // ---- G = Kt Kh^T (warp 0), P = tril(Qt Kh^T) (warp 1); R = V - Ks S,
    // U = Diag(beta) R (every warp, its value columns)
    if (warp < 2) {
      const __nv_bfloat16 *lhs = warp == 0 ? &sm.kt[0][0] : &sm.qt[0][0];
      float a2[2][4], b2[2][4];
      zero(a2);
      zero(b2);
#pragma unroll
      for (int kk = 0; kk < D / 16; kk += 2) {
        uint32_t a[4], b[4];
        lda(lhs, TP, 0, 16 * kk, lane, a);
        ldb(&sm.kh[0][0], TP, 0, 16 * kk, lane, b);
        mma2(a2, a, b);
        lda(lhs, TP, 0, 16 * kk + 16, lane, a);
        ldb(&sm.kh[0][0], TP, 0, 16 * kk + 16, lane, b);
        mma2(b2, a, b);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = 8 * j + 2 * t;
        if (warp == 0) {
          sm.G[g][c] = a2[j][0] + b2[j][0];
          sm.G[g][c + 1] = a2[j][1] + b2[j][1];
          sm.G[g + 8][c] = a2[j][2] + b2[j][2];
          sm.G[g + 8][c + 1] = a2[j][3] + b2[j][3];
        } else {
          st_bf2(&sm.pm[g][c], c <= g ? a2[j][0] + b2[j][0] : 0.f,
                 c + 1 <= g ? a2[j][1] + b2[j][1] : 0.f);
          st_bf2(&sm.pm[g + 8][c], c <= g + 8 ? a2[j][2] + b2[j][2] : 0.f,
                 c + 1 <= g + 8 ? a2[j][3] + b2[j][3] : 0.f);
        }
      }
    }
    float rr[NT][4];
    {
      zero(rr);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4], b[2 * NT];
        lda(&sm.ks[0][0], TP, 0, 16 * kk, lane, a);
        ldbv_t<NT>(&sm.S[0][0], VP, nv0, 16 * kk, lane, b);
        mmav<NT>(rr, a, b);
      }
      const float bg = sm.beta[g], bg8 = sm.beta[g + 8];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int c = nv0 + 8 * j + 2 * t;
        const float2 va = ld_bf2(&sm.v[g][c]), vb = ld_bf2(&sm.v[g + 8][c]);
        rr[j][0] = va.x - rr[j][0];
        rr[j][1] = va.y - rr[j][1];
        rr[j][2] = vb.x - rr[j][2];
        rr[j][3] = vb.y - rr[j][3];
        st_bf2(&sm.u[g][c], bg * rr[j][0], bg * rr[j][1]);
        st_bf2(&sm.u[g + 8][c], bg8 * rr[j][2], bg8 * rr[j][3]);
      }
    }
    __syncthreads();
    if (ch > 0) issue_v(ch - 1);  // v is used up

    // ---- T = (I + A)^{-1}, A = tril(Diag(beta) G, -1), on lanes 0-15 of warp 0
    // (lane j: column j, forward substitution over the rows), alongside
    // d delta = P^T dO + Kd dS' on every warp (its value columns; no T needed)
    if (warp == 0 && lane < CB) {
      const int j = lane;
      float tc[CB];
#pragma unroll
      for (int r = 0; r < CB; ++r) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) s = fmaf(sm.G[r][i], tc[i], s);
        tc[r] = (r == j ? 1.f : 0.f) - sm.beta[r] * s;
      }
#pragma unroll
      for (int r = 0; r < CB; ++r) sm.tm[r][j] = __float2bfloat16_rn(tc[r]);
    }
    {
      float dd[NT][4];
      zero(dd);
      uint32_t a[4], b[2 * NT];
      lda_t(&sm.pm[0][0], SP, 0, 0, lane, a);
      ldbv_t<NT>(&sm.dout[0][0], VP, nv0, 0, lane, b);
      mmav<NT>(dd, a, b);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {  // dS' as its bf16 pair: d beta is a
        lda(&sm.kd[0][0], TP, 0, 16 * kk, lane, a);  // dot product with cancellation
        ldbv_t<NT>(&sm.dSn[0][0], VP, nv0, 16 * kk, lane, b);
        mmav<NT>(dd, a, b);
        ldbv_t<NT>(&sm.dSlo[0][0], VP, nv0, 16 * kk, lane, b);
        mmav<NT>(dd, a, b);
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int c = nv0 + 8 * j + 2 * t;
        st_bf2(&sm.ddl[g][c], dd[j][0], dd[j][1]);
        st_bf2(&sm.ddl[g + 8][c], dd[j][2], dd[j][3]);
      }
    }
    __syncthreads();  // T is in place (each warp reads back only its own d delta)

    // ---- delta = T U; dU = T^T d delta, dR = Diag(beta) dU (= dv); rowsum(R o dU)
    {
      uint32_t a[4], b[2 * NT];
      float dlt[NT][4];
      zero(dlt);
      lda(&sm.tm[0][0], SP, 0, 0, lane, a);
      ldbv_t<NT>(&sm.u[0][0], VP, nv0, 0, lane, b);
      mmav<NT>(dlt, a, b);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int c = nv0 + 8 * j + 2 * t;
        st_bf2(&sm.dl[g][c], dlt[j][0], dlt[j][1]);
        st_bf2(&sm.dl[g + 8][c], dlt[j][2], dlt[j][3]);
      }
      float du[NT][4];
      zero(du);
      lda_t(&sm.tm[0][0], SP, 0, 0, lane, a);
      ldbv_t<NT>(&sm.ddl[0][0], VP, nv0, 0, lane, b);
      mmav<NT>(du, a, b);
      const float bg = sm.beta[g], bg8 = sm.beta[g + 8];
      float pa = 0.f, pb = 0.f;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int c = nv0 + 8 * j + 2 * t;
        pa = fmaf(rr[j][0], du[j][0], fmaf(rr[j][1], du[j][1], pa));
        pb = fmaf(rr[j][2], du[j][2], fmaf(rr[j][3], du[j][3], pb));
        st_bf2(&sm.du[g][c], du[j][0], du[j][1]);
        st_bf2(&sm.du[g + 8][c], du[j][2], du[j][3]);
        st_bf2(&sm.ndr[g][c], -bg * du[j][0], -bg * du[j][1]);
        st_bf2(&sm.ndr[g + 8][c], -bg8 * du[j][2], -bg8 * du[j][3]);
        if (g < n) st_bf2_g(dv + ((tb + g) * H + h) * D + vbase + c, bg * du[j][0], bg * du[j][1]);
        if (g + 8 < n)
          st_bf2_g(dv + ((tb + g + 8) * H + h) * D + vbase + c, bg8 * du[j][2], bg8 * du[j][3]);
      }
      pa += __shfl_xor_sync(0xffffffffu, pa, 1);
      pa += __shfl_xor_sync(0xffffffffu, pa, 2);
      pb += __shfl_xor_sync(0xffffffffu, pb, 1);
      pb += __shfl_xor_sync(0xffffffffu, pb, 2);
      if (t == 0) {
        sm.dbp[warp][g] = pa;
        sm.dbp[warp][g + 8] = pb;
      }
    }
    __syncthreads();

    // ---- dA, dP (warps 0, 1); dS = Diag(e^{g_l}) dS' + Qs^T dO - Ks^T dR (all)
    if (warp < 2) {
      const __nv_bfloat16 *lhs = warp == 0 ? &sm.du[0][0] : &sm.dout[0][0];
      float a2[2][4], b2[2][4];
      zero(a2);
      zero(b2);
#pragma unroll
      for (int kk = 0; kk < NV / 16; kk += 2) {
        uint32_t a[4], b[4];
        lda(lhs, VP, 0, 16 * kk, lane, a);
        ldb(&sm.dl[0][0], VP, 0, 16 * kk, lane, b);
        mma2(a2, a, b);
        lda(lhs, VP, 0, 16 * kk + 16, lane, a);
        ldb(&sm.dl[0][0], VP, 0, 16 * kk + 16, lane, b);
        mma2(b2, a, b);
      }
      if (warp == 0) {  // dA = tril(-dU delta^T, -1); dG = Diag(beta) dA; rowsum(dA o G)
        const float bg = sm.beta[g], bg8 = sm.beta[g + 8];
        float pa = 0.f, pb = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = 8 * j + 2 * t;
          const float x0 = c < g ? -(a2[j][0] + b2[j][0]) : 0.f;
          const float x1 = c + 1 < g ? -(a2[j][1] + b2[j][1]) : 0.f;
          const float x2 = c < g + 8 ? -(a2[j][2] + b2[j][2]) : 0.f;
          const float x3 = c + 1 < g + 8 ? -(a2[j][3] + b2[j][3]) : 0.f;
          pa = fmaf(x0, sm.G[g][c], fmaf(x1, sm.G[g][c + 1], pa));
          pb = fmaf(x2, sm.G[g + 8][c], fmaf(x3, sm.G[g + 8][c + 1], pb));
          st_bf2(&sm.dgm[g][c], bg * x0, bg * x1);
          st_bf2(&sm.dgm[g + 8][c], bg8 * x2, bg8 * x3);
        }
        pa += __shfl_xor_sync(0xffffffffu, pa, 1);
        pa += __shfl_xor_sync(0xffffffffu, pa, 2);
        pb += __shfl_xor_sync(0xffffffffu, pb, 1);
        pb += __shfl_xor_sync(0xffffffffu, pb, 2);
        if (t == 0) {
          sm.dba[g] = pa;
          sm.dba[g + 8] = pb;
        }
      } else {  // dP = tril(dO delta^T)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = 8 * j + 2 * t;
          st_bf2(&sm.dpm[g][c], c <= g ? a2[j][0] + b2[j][0] : 0.f,
                 c + 1 <= g ? a2[j][1] + b2[j][1] : 0.f);
          st_bf2(&sm.dpm[g + 8][c], c <= g + 8 ? a2[j][2] + b2[j][2] : 0.f,
                 c + 1 <= g + 8 ? a2[j][3] + b2[j][3] : 0.f);
        }
      }
    }
    {
      const float ga = sm.gam[kr0 + g], gb = sm.gam[kr0 + g + 8];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        ds[j][0] *= ga; ds[j][1] *= ga; ds[j][2] *= gb; ds[j][3] *= gb;
      }
      uint32_t aq[4], ak[4];
      lda_t(&sm.qs[0][0], TP, kr0, 0, lane, aq);
      lda_t(&sm.ks[0][0], TP, kr0, 0, lane, ak);
#pragma unroll
      for (int jp = 0; jp < NJ / 2; ++jp) {
        uint32_t b[4];
        ldb_t(&sm.dout[0][0], VP, 16 * jp, 0, lane, b);
        mma_bf16_16x8x16(ds[2 * jp], aq[0], aq[1], aq[2], aq[3], b[0], b[1]);
        mma_bf16_16x8x16(ds[2 * jp + 1], aq[0], aq[1], aq[2], aq[3], b[2], b[3]);
        ldb_t(&sm.ndr[0][0], VP, 16 * jp, 0, lane, b);
        mma_bf16_16x8x16(ds[2 * jp], ak[0], ak[1], ak[2], ak[3], b[0], b[1]);
        mma_bf16_16x8x16(ds[2 * jp + 1], ak[0], ak[1], ak[2], ak[3], b[2], b[3]);
      }
      // rowsum_v(S o dS)
      float p2a = 0.f, p2b = 0.f;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int c = 8 * j + 2 * t;
        const float2 a = ld_bf2(&sm.S[kr0 + g][c]), b = ld_bf2(&sm.S[kr0 + g + 8][c]);
        p2a = fmaf(a.x, ds[j][0], fmaf(a.y, ds[j][1], p2a));
        p2b = fmaf(b.x, ds[j][2], fmaf(b.y, ds[j][3], p2b));
      }
      p2a += __shfl_xor_sync(0xffffffffu, p2a, 1);
      p2a += __shfl_xor_sync(0xffffffffu, p2a, 2);
      p2b += __shfl_xor_sync(0xffffffffu, p2b, 1);
      p2b += __shfl_xor_sync(0xffffffffu, p2b, 2);
      if (t == 0) {
        sm.t2[kr0 + g] = p2a;
        sm.t2[kr0 + g + 8] = p2b;
      }
    }
    // ---- dKd = delta dS'^T, (-dR) S^T, dO S^T over this CTA's value columns
    // (keys kr0 .. kr0 + 15)
    float akd[2][4], akt[2][4], aqt[2][4];
    zero(akd);
    zero(akt);
    zero(aqt);
#pragma unroll
    for (int kk = 0; kk < NV / 16; ++kk) {
      uint32_t a[4], b[4];
      lda(&sm.dl[0][0], VP, 0, 16 * kk, lane, a);
      ldb(&sm.dSn[0][0], VP, kr0, 16 * kk, lane, b);
      mma2(akd, a, b);
      ldb(&sm.S[0][0], VP, kr0, 16 * kk, lane, b);
      lda(&sm.ndr[0][0], VP, 0, 16 * kk, lane, a);
      mma2(akt, a, b);
      lda(&sm.dout[0][0], VP, 0, 16 * kk, lane, a);
      mma2(aqt, a, b);
    }
    __syncthreads();  // dG, dP, rowsum(dA o G), t2 are in place
    if (ch > 0) issue_rest(ch - 1);  // dO, beta and the state are used up

    // ---- dKt = e^{g_m} o ((-dR) S^T) + dG Kh, dQt = e^{g_m} o (dO S^T) + dP Kh,
    // dKh = dG^T Kt + dP^T Qt; then dq, dk and dg for this warp's key columns
    // (in a cluster: this CTA's part of them)
    float dqv[2][2][2], dkv[2][2][2], dgv[2][2][2];  // [j][row half][e]
    {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = kr0 + 8 * j + 2 * t;
        const float e0 = sm.em[c], e1 = sm.em[c + 1];
        akt[j][0] *= e0; akt[j][1] *= e1; akt[j][2] *= e0; akt[j][3] *= e1;
        aqt[j][0] *= e0; aqt[j][1] *= e1; aqt[j][2] *= e0; aqt[j][3] *= e1;
      }
      float akh[2][4];
      zero(akh);
      uint32_t a[4], b[4];
      ldb_t(&sm.kh[0][0], TP, kr0, 0, lane, b);
      lda(&sm.dgm[0][0], SP, 0, 0, lane, a);
      mma2(akt, a, b);
      lda(&sm.dpm[0][0], SP, 0, 0, lane, a);
      mma2(aqt, a, b);
      ldb_t(&sm.kt[0][0], TP, kr0, 0, lane, b);
      lda_t(&sm.dgm[0][0], SP, 0, 0, lane, a);
      mma2(akh, a, b);
      ldb_t(&sm.qt[0][0], TP, kr0, 0, lane, b);
      lda_t(&sm.dpm[0][0], SP, 0, 0, lane, a);
      mma2(akh, a, b);

      float sphi[2][2], spsi[2][2], schi[2][2];  // column sums [j][e]
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = kr0 + 8 * j + 2 * t;
        const float etl0 = sm.et[kLast][c], etl1 = sm.et[kLast][c + 1];
#pragma unroll
        for (int e = 0; e < 2; ++e) sphi[j][e] = spsi[j][e] = schi[j][e] = 0.f;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {  // rows g, g + 8
          const int r = g + 8 * hr;
          // dg pairs each gradient with the bf16 operand value its product used,
          // so the terms of a product that cancel in exact arithmetic (the Gram
          // and P pairs within the chunk) cancel here too
          const float2 vkt = ld_bf2(&sm.kt[r][c]), vqt = ld_bf2(&sm.qt[r][c]);
          const float2 vkh = ld_bf2(&sm.kh[r][c]), vkd = ld_bf2(&sm.kd[r][c]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float et = sm.et[r][c + e];
            const float eh = __fdividef(1.0f, et);  // et in [e^-40, e^40]
            const float ed = (e ? etl1 : etl0) * eh;
            const float gkt = akt[j][2 * hr + e], gqt = aqt[j][2 * hr + e];
            const float gkh = akh[j][2 * hr + e], gkd = akd[j][2 * hr + e];
            dqv[j][hr][e] = gqt * et;
            dkv[j][hr][e] = gkt * et + gkh * eh + gkd * ed;
            const float phi = gkt * (e ? vkt.y : vkt.x) + gqt * (e ? vqt.y : vqt.x);
            const float psi = gkh * (e ? vkh.y : vkh.x);
            const float chi = gkd * (e ? vkd.y : vkd.x);
            sphi[j][e] += phi;
            spsi[j][e] += psi;
            schi[j][e] += chi;
            dgv[j][hr][e] = phi - psi - chi;
          }
        }
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            sphi[j][e] += __shfl_xor_sync(0xffffffffu, sphi[j][e], off);
            spsi[j][e] += __shfl_xor_sync(0xffffffffu, spsi[j][e], off);
            schi[j][e] += __shfl_xor_sync(0xffffffffu, schi[j][e], off);
          }
      if (g == kMid) {  // this lane also holds rows kMid and kLast = kMid + 8
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = kr0 + 8 * j + 2 * t + e;
            const float gt1 = sm.gam[c] * sm.t1[c];
            dgv[j][0][e] += -sphi[j][e] + spsi[j][e] + (sm.t2[c] - gt1);
            dgv[j][1][e] += schi[j][e] + gt1;
          }
      }
    }
    // ---- in a cluster: send the other CTA's keys, receive this CTA's
    const int own_half = warp >> 2;          // the key half of this warp's columns
    const bool mine = !kPair || own_half == rank;
    if constexpr (kPair) {
      if (!mine) {
        const uint32_t peer = (uint32_t)(rank ^ 1);
        const uint32_t base = cluster_addr(&sm.xin[par][0][0][0], peer);
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int r = g + 8 * hr, lc = kr0 - 64 * own_half + 8 * j + 2 * t;
            const uint32_t off = (uint32_t)((r * 64 + lc) * 4);
            st_cluster_f32x2(base + off, dqv[j][hr][0], dqv[j][hr][1]);
            st_cluster_f32x2(base + CB * 64 * 4 + off, dkv[j][hr][0], dkv[j][hr][1]);
            st_cluster_f32x2(base + 2 * CB * 64 * 4 + off, dgv[j][hr][0], dgv[j][hr][1]);
          }
      }
      if (rank == 1 && tid < CB) {  // this CTA's part of dbeta, to rank 0
        float s = sm.dba[tid];
#pragma unroll
        for (int w = 0; w < 8; ++w) s += sm.dbp[w][tid];
        st_cluster_f32(cluster_addr(&sm.xdb[par][tid], 0), s);
      }
      cluster_sync();  // every part has landed
    }
    if (mine) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = g + 8 * hr, c = kr0 + 8 * j + 2 * t;
          if constexpr (kPair) {
            const int lc = c - 64 * rank;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              dqv[j][hr][e] += sm.xin[par][0][r][lc + e];
              dkv[j][hr][e] += sm.xin[par][1][r][lc + e];
              dgv[j][hr][e] += sm.xin[par][2][r][lc + e];
            }
          }
          if (r < n) {
            st_bf2_g(dq + ((tb + r) * H + h) * D + c, dqv[j][hr][0], dqv[j][hr][1]);
            st_bf2_g(dk + ((tb + r) * H + h) * D + c, dkv[j][hr][0], dkv[j][hr][1]);
          }
          sm.dgr[r][c] = dgv[j][hr][0];
          sm.dgr[r][c + 1] = dgv[j][hr][1];
        }
    }
    __syncthreads();

    // ---- dlog_alpha: reverse cumulative sum over the chunk (this CTA's keys); dbeta
    constexpr int NK = kPair ? 64 : D;  // keys this CTA finishes
    if (tid < NK) {
      const int c = (kPair ? 64 * rank : 0) + tid;
      float dgc[CB];  // every row first: the stores then run back to back
#pragma unroll
      for (int r = 0; r < CB; ++r) dgc[r] = sm.dgr[r][c];
      float acc = 0.f;
#pragma unroll
      for (int r = CB - 1; r >= 0; --r) {
        acc += dgc[r];
        if (r < n) d_la[((tb + r) * H + h) * D + c] = acc;
      }
    } else if (tid < NK + CB && rank == 0) {
      const int r = tid - NK;
      if (r < n) {
        float s = sm.dba[r];
#pragma unroll
        for (int w = 0; w < 8; ++w) s += sm.dbp[w][r];
        if constexpr (kPair) s += sm.xdb[par][r];
        d_beta[(tb + r) * H + h] = s;
      }
    }
  }
  if (d_init) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int c = vbase + 8 * j + 2 * t;
      float *pa = d_init + sbase + (kr0 + g) * D + c, *pb = pa + 8 * D;
      pa[0] = ds[j][0];
      pa[1] = ds[j][1];
      pb[0] = ds[j][2];
      pb[1] = ds[j][3];
    }
  }
  if constexpr (kPair) cluster_sync();  // no remote store outlives either CTA
}

// Forward pass for the chunked backward: the state at every chunk start, as
// bf16 (checkpoint slot bwd_ckpt_slot_base(cu[s], s, 16) + chunk, 32 KiB per
// head; the backward pass uses the state only as a bf16 operand), by the chunk form
// above with the same bf16 operands: R = V - Ks S, delta = T Diag(beta) R,
// S' = Diag(e^{g_l}) S + Kd^T delta.  The state stays in registers as MMA
// accumulators (warp w: key rows 16 w .. 16 w + 15).  With NV = 64 two CTAs
// take a chain, 64 value columns each, independently (nothing to exchange: the
// key-side work is done by both).
template <int NV>
struct __align__(16) CkSmem {
  static constexpr int VP = NV + 8;
  __nv_bfloat16 S[D][VP];
  __nv_bfloat16 k[CB][TP], kt[CB][TP], kh[CB][TP], ks[CB][TP], kd[CB][TP];
  __nv_bfloat16 v[CB][VP], u[CB][VP], dl[CB][VP];
  __nv_bfloat16 tm[CB][SP];
  float la[CB][D];
  float G[CB][GP];
  float gam[D];
  float beta[CB];
};

template <int NV>
__global__ void __launch_bounds__(kThreads, 1)
kda_bwd_chunk_ckpt_kernel(const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                          const float *__restrict__ la, const float *__restrict__ beta,
                          const float *__restrict__ init_state, const int32_t *__restrict__ cu,
                          int32_t n_seqs, int64_t n_tokens, int32_t H,
                          __nv_bfloat16 *__restrict__ ckpt, DeviceStatus *status) {
  constexpr int VP = CkSmem<NV>::VP;
  constexpr int NT = NV / 64;
  constexpr int NJ = NV / 8;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  CkSmem<NV> &sm = *reinterpret_cast<CkSmem<NV> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const ChainOf chn = chain_of_block<NV>(cu, n_seqs, n_tokens, H);
  if (!chn.ok) {
    if (tid == 0) atomicCAS(&status->code, 0, 1 /* KDA_ERR_INVALID_ARG */);
    return;
  }
  const int seq = chn.seq, h = chn.h;
  const int64_t t0 = chn.t0, t1 = chn.t1;
  const int vbase = NV * chn.rank;
  const int kr0 = 16 * warp, nv0 = NV / 8 * warp;
  float st[NJ][4];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = vbase + 8 * j + 2 * t;
    st[j][0] = st[j][1] = st[j][2] = st[j][3] = 0.f;
    if (init_state) {
      const float *pa = init_state + ((int64_t)seq * H + h) * D * D + (kr0 + g) * D + c;
      st[j][0] = pa[0];
      st[j][1] = pa[1];
      st[j][2] = pa[8 * D];
      st[j][3] = pa[8 * D + 1];
    }
  }
  const int64_t n_ch = (t1 - t0 + CB - 1) / CB;
  const int64_t slot0 = bwd_ckpt_slot_base(t0, seq, CB);
  // inputs of chunk c + 1 are copied during chunk c, each tile after its last use
  auto chunk_len = [&](int64_t c) { return (int)(t1 - (t0 + CB * c) < CB ? t1 - (t0 + CB * c) : CB); };
  auto issue_kl = [&](int64_t c) {
    stage_rows<TP, 16>(sm.k, k, t0 + CB * c, chunk_len(c), h, H, 0, tid);
    stage_rows_f32(sm.la, la, t0 + CB * c, chunk_len(c), h, H, tid);
  };
  auto issue_v = [&](int64_t c) {
    stage_rows<VP, NV / 8>(sm.v, v, t0 + CB * c, chunk_len(c), h, H, vbase, tid);
  };
  auto load_beta = [&](int64_t c) {
    const int n = chunk_len(c);
    if (tid < CB) sm.beta[tid] = tid < n ? beta[(t0 + CB * c + tid) * H + h] : 0.f;
  };
  if (n_ch > 0) {
    issue_kl(0);
    issue_v(0);
    load_beta(0);
  }
  for (int64_t ch = 0; ch < n_ch; ++ch) {
    cp_async_wait_all();
    __syncthreads();  // the chunk's inputs are in place; the previous chunk is done
    __nv_bfloat16 *Sg = ckpt + ((slot0 + ch) * H + h) * (int64_t)(D * D) + vbase;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int c = 8 * j + 2 * t;
      const __nv_bfloat162 ha = __floats2bfloat162_rn(st[j][0], st[j][1]);
      const __nv_bfloat162 hb = __floats2bfloat162_rn(st[j][2], st[j][3]);
      *reinterpret_cast<__nv_bfloat162 *>(Sg + (kr0 + g) * D + c) = ha;
      *reinterpret_cast<__nv_bfloat162 *>(Sg + (kr0 + g + 8) * D + c) = hb;
      *reinterpret_cast<__nv_bfloat162 *>(&sm.S[kr0 + g][c]) = ha;
      *reinterpret_cast<__nv_bfloat162 *>(&sm.S[kr0 + g + 8][c]) = hb;
    }
    {  // factor-scaled k tiles (as in the backward pass): threads 0-127 Kt, Kh; 128-255 Ks, Kd
      const int c = tid & (D - 1);
      ColFactors f;
      col_factors(sm.la, c, f);
      if (tid < D) {
#pragma unroll
        for (int r = 0; r < CB; ++r) {
          const float kf = __bfloat162float(sm.k[r][c]);
          sm.kt[r][c] = __float2bfloat16_rn(kf * f.et[r]);
          sm.kh[r][c] = __float2bfloat16_rn(kf * __fdividef(1.0f, f.et[r]));
        }
      } else {
        sm.gam[c] = f.em * f.etl;
#pragma unroll
        for (int r = 0; r < CB; ++r) {
          const float kf = __bfloat162float(sm.k[r][c]);
          sm.ks[r][c] = __float2bfloat16_rn(kf * (f.em * f.et[r]));
          sm.kd[r][c] = __float2bfloat16_rn(kf * (f.etl * __fdividef(1.0f, f.et[r])));
        }
      }
    }
    __syncthreads();
    if (ch + 1 < n_ch) issue_kl(ch + 1);  // k and log_alpha are used up
    if (warp == 0) {  // G = Kt Kh^T
      float a2[2][4], b2[2][4];
      zero(a2);
      zero(b2);
#pragma unroll
      for (int kk = 0; kk < D / 16; kk += 2) {
        uint32_t a[4], b[4];
        lda(&sm.kt[0][0], TP, 0, 16 * kk, lane, a);
        ldb(&sm.kh[0][0], TP, 0, 16 * kk, lane, b);
        mma2(a2, a, b);
        lda(&sm.kt[0][0], TP, 0, 16 * kk + 16, lane, a);
        ldb(&sm.kh[0][0], TP, 0, 16 * kk + 16, lane, b);
        mma2(b2, a, b);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = 8 * j + 2 * t;
        sm.G[g][c] = a2[j][0] + b2[j][0];
        sm.G[g][c + 1] = a2[j][1] + b2[j][1];
        sm.G[g + 8][c] = a2[j][2] + b2[j][2];
        sm.G[g + 8][c + 1] = a2[j][3] + b2[j][3];
      }
    }
    {  // U = Diag(beta) (V - Ks S), this warp's value columns
      float rr[NT][4];
      zero(rr);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4], b[2 * NT];
        lda(&sm.ks[0][0], TP, 0, 16 * kk, lane, a);
        ldbv_t<NT>(&sm.S[0][0], VP, nv0, 16 * kk, lane, b);
        mmav<NT>(rr, a, b);
      }
      const float bg = sm.beta[g], bg8 = sm.beta[g + 8];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int c = nv0 + 8 * j + 2 * t;
        const float2 va = ld_bf2(&sm.v[g][c]), vb = ld_bf2(&sm.v[g + 8][c]);
        st_bf2(&sm.u[g][c], bg * (va.x - rr[j][0]), bg * (va.y - rr[j][1]));
        st_bf2(&sm.u[g + 8][c], bg8 * (vb.x - rr[j][2]), bg8 * (vb.y - rr[j][3]));
      }
    }
    __syncthreads();
    if (ch + 1 < n_ch) issue_v(ch + 1);  // v is used up
    if (warp == 0 && lane < CB) {  // T = (I + A)^{-1}, column `lane`
      const int j = lane;
      float tc[CB];
#pragma unroll
      for (int r = 0; r < CB; ++r) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) s = fmaf(sm.G[r][i], tc[i], s);
        tc[r] = (r == j ? 1.f : 0.f) - sm.beta[r] * s;
      }
#pragma unroll
      for (int r = 0; r < CB; ++r) sm.tm[r][j] = __float2bfloat16_rn(tc[r]);
    }
    __syncthreads();
    if (ch + 1 < n_ch) load_beta(ch + 1);  // beta is used up
    {  // delta = T U
      float dlt[NT][4];
      zero(dlt);
      uint32_t a[4], b[2 * NT];
      lda(&sm.tm[0][0], SP, 0, 0, lane, a);
      ldbv_t<NT>(&sm.u[0][0], VP, nv0, 0, lane, b);
      mmav<NT>(dlt, a, b);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int c = nv0 + 8 * j + 2 * t;
        st_bf2(&sm.dl[g][c], dlt[j][0], dlt[j][1]);
        st_bf2(&sm.dl[g + 8][c], dlt[j][2], dlt[j][3]);
      }
    }
    __syncthreads();
    {  // S' = Diag(e^{g_l}) S + Kd^T delta
      const float ga = sm.gam[kr0 + g], gb = sm.gam[kr0 + g + 8];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        st[j][0] *= ga; st[j][1] *= ga; st[j][2] *= gb; st[j][3] *= gb;
      }
      uint32_t a[4];
      lda_t(&sm.kd[0][0], TP, kr0, 0, lane, a);
#pragma unroll
      for (int jp = 0; jp < NJ / 2; ++jp) {
        uint32_t b[4];
        ldb_t(&sm.dl[0][0], VP, 16 * jp, 0, lane, b);
        mma_bf16_16x8x16(st[2 * jp], a[0], a[1], a[2], a[3], b[0], b[1]);
        mma_bf16_16x8x16(st[2 * jp + 1], a[0], a[1], a[2], a[3], b[2], b[3]);
      }
    }
  }
}

// Launch configuration of the reverse kernel for NV value columns per CTA
// (a cluster of D / NV CTAs per chain).
template <int NV>
struct ReverseLaunch {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  ReverseLaunch(int64_t chains, cudaStream_t stream) {
    cfg.gridDim = dim3((unsigned)(chains * (D / NV)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(Smem<NV>);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = D / NV;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = NV < D ? 1 : 0;
  }
};

template <int NV>
cudaError_t launch_reverse(const BwdArgs &a, int64_t chains, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_chunk_kernel<NV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(Smem<NV>));
  if (e != cudaSuccess) return e;
  ReverseLaunch<NV> l(chains, stream);
  return cudaLaunchKernelEx(
      &l.cfg, kda_bwd_chunk_kernel<NV>, static_cast<const __nv_bfloat16 *>(a.q),
      static_cast<const __nv_bfloat16 *>(a.k), static_cast<const __nv_bfloat16 *>(a.v),
      a.log_alpha, a.beta, a.cu_seqlens, a.n_seqs, a.n_tokens, a.H,
      reinterpret_cast<const __nv_bfloat16 *>(a.ckpt), static_cast<const __nv_bfloat16 *>(a.d_out),
      a.d_final, static_cast<__nv_bfloat16 *>(a.dq), static_cast<__nv_bfloat16 *>(a.dk),
      static_cast<__nv_bfloat16 *>(a.dv), a.d_log_alpha, a.d_beta, a.d_init, a.status);
}

template <int NV>
cudaError_t launch_pass(const BwdArgs &a, int64_t chains, cudaStream_t stream) {
  constexpr int VS = D / NV;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_chunk_ckpt_kernel<NV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(CkSmem<NV>));
  if (e != cudaSuccess) return e;
  kda_bwd_chunk_ckpt_kernel<NV><<<(unsigned)(chains * VS), kThreads, sizeof(CkSmem<NV>), stream>>>(
      static_cast<const __nv_bfloat16 *>(a.k), static_cast<const __nv_bfloat16 *>(a.v),
      a.log_alpha, a.beta, a.init_state, a.cu_seqlens, a.n_seqs, a.n_tokens, a.H,
      reinterpret_cast<__nv_bfloat16 *>(a.ckpt), a.status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_reverse<NV>(a, chains, stream);
  if (e != cudaSuccess && VS > 1) {
    // a cluster launch the device refuses (the stored states are the same for
    // both reverse kernels): one CTA per chain instead
    cudaGetLastError();
    e = launch_reverse<D>(a, chains, stream);
  }
  return e;
}

}  // namespace

size_t bwd_chunk_smem_bytes() { return sizeof(Smem<D>); }

// Two CTAs per chain (64 value columns each, a cluster) when every pair can be
// resident at once (the runtime's count of active two-CTA clusters of the
// reverse kernel); else one CTA per chain.
cudaError_t launch_bwd_chunk(const BwdArgs &a, cudaStream_t stream) {
  const int64_t chains = (int64_t)a.n_seqs * a.H;
  if (chains == 0) return cudaSuccess;
  if (chains > 0x3fffffffLL || !a.bf16 || a.ckpt_every != CB) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_chunk_kernel<D / 2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(Smem<D / 2>));
  if (e != cudaSuccess) return e;
  ReverseLaunch<D / 2> l(chains, stream);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kda_bwd_chunk_kernel<D / 2>, &l.cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    clusters = 0;
  }
  if (chains <= clusters) return launch_pass<D / 2>(a, chains, stream);
  return launch_pass<D>(a, chains, stream);
}

}  // namespace kda
