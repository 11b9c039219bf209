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
// chain is cut into four blocks of 32 value columns, one CTA each (8 warps).
// Lane l of warp w holds value columns 2 (l mod 16) and 2 (l mod 16) + 1 of key
// rows 16 w + 8 floor(l / 16) .. + 7: 16 state values per thread.  Column sums
// over the 128 key rows are in-thread over 8 rows, one shuffle between the
// half-warps and a shared-memory sum over the warps; row sums over the 32
// columns are in-thread over a column pair and a transposing butterfly over the
// 16 lanes of a half-warp.  dv and the initial-state gradient belong to one
// block; dq, dk, dlog_alpha and dbeta are sums over all value columns, added
// across the four blocks with fp32 atomics (so their last bits depend on the
// order of those four additions).
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
constexpr int kRows = 8;          // key rows per thread (two value columns each)
constexpr int kGroup = 4;         // tokens whose X a CTA keeps at a time

__device__ __forceinline__ int64_t ckpt_base(int64_t cu_s, int64_t s, int every) {
  return bwd_ckpt_slot_base(cu_s, s, every);
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

// 16-byte asynchronous copy global -> shared (L2 only), and its group fences.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Raw inputs of up to kGroup tokens as they sit in HBM, copied asynchronously
// one group ahead: per token the q, k and log_alpha rows, then the CTA's
// 32-column blocks of v and d_out (q, d_out unused by the forward sweep).
template <bool BF16>
struct RawLayout {
  static constexpr int kEsz = BF16 ? 2 : 4;
  static constexpr int kQ = 0, kK = D * kEsz, kLa = 2 * D * kEsz, kV = kLa + 4 * D,
                       kDo = kV + kCols * kEsz, kTok = kDo + kCols * kEsz;
  // 16-byte pieces per token: q, k, log_alpha rows, v and d_out blocks
  static constexpr int kRowPieces = D * kEsz / 16, kLaPieces = D * 4 / 16,
                       kBlkPieces = kCols * kEsz / 16;
  static constexpr int kPieces = 2 * kRowPieces + kLaPieces + 2 * kBlkPieces;
};
static_assert(RawLayout<true>::kTok % 16 == 0 && RawLayout<false>::kTok % 16 == 0,
              "raw token rows keep 16-byte alignment");
constexpr int kRawBytes = kGroup * RawLayout<false>::kTok;  // the larger (fp32) layout

// Issues (every thread) the copies of tokens tb .. tb + n - 1 of head h, value
// block cb into raw; with_q also their q and d_out.  One commit group.
template <bool BF16>
__device__ void prefetch_tokens(uint8_t *raw, int64_t tb, int n, int h, int H, int cb,
                                bool with_q, const void *q, const void *k, const void *v,
                                const float *la, const void *dout) {
  using L = RawLayout<BF16>;
  for (int e = threadIdx.x; e < n * L::kPieces; e += kThreads) {
    const int i = e / L::kPieces;
    int r = e % L::kPieces;
    const int64_t row = (tb + i) * H + h;  // token row of the [N, H, 128] tensors
    uint8_t *dst = raw + i * L::kTok;
    const uint8_t *src = nullptr;
    if (r < L::kRowPieces) {
      if (with_q) src = static_cast<const uint8_t *>(q) + row * D * L::kEsz + 16 * r;
      dst += L::kQ + 16 * r;
    } else if ((r -= L::kRowPieces) < L::kRowPieces) {
      src = static_cast<const uint8_t *>(k) + row * D * L::kEsz + 16 * r;
      dst += L::kK + 16 * r;
    } else if ((r -= L::kRowPieces) < L::kLaPieces) {
      src = reinterpret_cast<const uint8_t *>(la + row * D) + 16 * r;
      dst += L::kLa + 16 * r;
    } else if ((r -= L::kLaPieces) < L::kBlkPieces) {
      src = static_cast<const uint8_t *>(v) + (row * D + cb * kCols) * L::kEsz + 16 * r;
      dst += L::kV + 16 * r;
    } else {
      r -= L::kBlkPieces;
      if (with_q) src = static_cast<const uint8_t *>(dout) + (row * D + cb * kCols) * L::kEsz + 16 * r;
      dst += L::kDo + 16 * r;
    }
    if (src) cp_async16(dst, src);
  }
  cp_async_commit();
}

template <bool BF16>
__device__ __forceinline__ float raw_elem(const uint8_t *p, int c) {
  if constexpr (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[c]);
  else return reinterpret_cast<const float *>(p)[c];
}

// The landed raw inputs of n tokens into st (alpha = e^{log_alpha}); the betas
// come from the threads that loaded them (thread i: token i).
template <bool BF16>
__device__ void convert_tokens(Stage &st, const uint8_t *raw, int n, bool with_q, float my_beta) {
  using L = RawLayout<BF16>;
  for (int e = threadIdx.x; e < n * D; e += kThreads) {
    const int i = e / D, c = e % D;
    const uint8_t *t = raw + i * L::kTok;
    st.q[i][c] = with_q ? raw_elem<BF16>(t + L::kQ, c) : 0.f;
    st.k[i][c] = raw_elem<BF16>(t + L::kK, c);
    st.alpha[i][c] = expf(reinterpret_cast<const float *>(t + L::kLa)[c]);
  }
  for (int e = threadIdx.x; e < n * kCols; e += kThreads) {
    const int i = e / kCols, c = e % kCols;
    const uint8_t *t = raw + i * L::kTok;
    st.v[i][c] = raw_elem<BF16>(t + L::kV, c);
    st.dout[i][c] = with_q ? raw_elem<BF16>(t + L::kDo, c) : 0.f;
  }
  if (threadIdx.x < n) st.beta[threadIdx.x] = my_beta;
}

// The per-warp column partial sums, in two buffers used in turn (rp counts the
// uses): a buffer is rewritten only two uses later, after a barrier every
// thread passes once it has read it, so one barrier per use suffices.
using Red = float[2][kThreads / 32][kCols];

// One forward token on this thread's 16 state values (rows r0 + j, value
// columns ca, ca + 1 of the block); the decayed state X and the per-column p, d
// of those two columns are returned.
__device__ __forceinline__ void fwd_token(float (&s)[kRows][2], float (&x)[kRows][2], float2 &p,
                                          float2 &d, const Stage &st, int i, int r0, int ca,
                                          int lane, int warp, Red &red, uint32_t &rp) {
  float pa = 0.f, pb = 0.f;
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    const float al = st.alpha[i][r0 + j], kr = st.k[i][r0 + j];
    x[j][0] = al * s[j][0];
    x[j][1] = al * s[j][1];
    pa = fmaf(x[j][0], kr, pa);
    pb = fmaf(x[j][1], kr, pb);
  }
  pa += __shfl_xor_sync(0xffffffffu, pa, 16);  // the other 8 rows of this warp's 16
  pb += __shfl_xor_sync(0xffffffffu, pb, 16);
  float (&rb)[kThreads / 32][kCols] = red[rp++ & 1u];
  if (lane < 16) *reinterpret_cast<float2 *>(&rb[warp][ca]) = make_float2(pa, pb);
  __syncthreads();
  p = make_float2(0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const float2 v2 = *reinterpret_cast<const float2 *>(&rb[w][ca]);
    p.x += v2.x;
    p.y += v2.y;
  }
  d = make_float2(st.beta[i] * (st.v[i][ca] - p.x), st.beta[i] * (st.v[i][ca + 1] - p.y));
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    const float kr = st.k[i][r0 + j];
    s[j][0] = fmaf(kr, d.x, x[j][0]);
    s[j][1] = fmaf(kr, d.y, x[j][1]);
  }
}

// Sum of v[j] over the 16 lanes of a half-warp, for each of the 8 rows j:
// after three halving exchanges lane L holds one row, row_of(L), summed over 8
// lanes, and the last exchange completes it (lanes 2m and 2m + 1 hold the same
// row).  The exchanges stay inside each half-warp.
__device__ __forceinline__ float row_sum(const float (&v)[kRows], int lane) {
  float a[4];
  {
    const bool hi = lane & 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float mine = hi ? v[4 + j] : v[j], give = hi ? v[j] : v[4 + j];
      a[j] = mine + __shfl_xor_sync(0xffffffffu, give, 8);
    }
  }
  float b[2];
  {
    const bool hi = lane & 4;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float mine = hi ? a[2 + j] : a[j], give = hi ? a[j] : a[2 + j];
      b[j] = mine + __shfl_xor_sync(0xffffffffu, give, 4);
    }
  }
  const bool hi = lane & 2;
  const float e = (hi ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, hi ? b[0] : b[1], 2);
  return e + __shfl_xor_sync(0xffffffffu, e, 1);
}
__device__ __forceinline__ int row_of(int lane) {
  return 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
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

// Forward pass: the state before every `every`-th token, per block of columns.
template <bool BF16>
__global__ void __launch_bounds__(kThreads, 2)
kda_bwd_ckpt_kernel(const void *__restrict__ k, const void *__restrict__ v,
                    const float *__restrict__ la, const float *__restrict__ beta,
                    const float *__restrict__ init_state, const int32_t *__restrict__ cu,
                    int32_t n_seqs, int64_t n_tokens, int32_t H, int every,
                    float *__restrict__ ckpt, DeviceStatus *status) {
  __shared__ Stage st;
  __shared__ Red red;
  uint32_t rp = 0;
  __shared__ __align__(16) uint8_t raw[kRawBytes];
  const Chain c = chain_of(cu, n_seqs, n_tokens, H);
  if (!c.ok) {
    if (threadIdx.x == 0) atomicCAS(&status->code, 0, 1 /* KDA_ERR_INVALID_ARG */);
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ca = 2 * (lane & 15), r0 = 16 * warp + kRows * (lane >> 4);
  const int col = c.cb * kCols + ca;
  const int64_t sbase = ((int64_t)c.seq * H + c.h) * D * D;
  float s[kRows][2], x[kRows][2];
#pragma unroll
  for (int j = 0; j < kRows; ++j)
#pragma unroll
    for (int z = 0; z < 2; ++z) s[j][z] = init_state ? init_state[sbase + (r0 + j) * D + col + z] : 0.f;
  const int64_t base = ckpt_base(c.t0, c.seq, every);
  // the inputs of each group are copied while the group before it runs
  auto group_len = [&](int64_t tb) { return (int)(c.t1 - tb < kGroup ? c.t1 - tb : kGroup); };
  float nbeta = 0.f;
  auto prefetch = [&](int64_t tb) {
    const int n = group_len(tb);
    prefetch_tokens<BF16>(raw, tb, n, c.h, H, c.cb, false, nullptr, k, v, la, nullptr);
    if (threadIdx.x < n) nbeta = beta[(tb + threadIdx.x) * H + c.h];
  };
  if (c.t0 < c.t1) prefetch(c.t0);
  for (int64_t tb = c.t0; tb < c.t1; tb += kGroup) {
    const int n = group_len(tb);
    cp_async_wait_all();
    __syncthreads();  // the group's copies landed; the previous group's stage is consumed
    convert_tokens<BF16>(st, raw, n, false, nbeta);
    __syncthreads();  // st ready, raw free
    if (tb + kGroup < c.t1) prefetch(tb + kGroup);
    for (int i = 0; i < n; ++i) {
      const int64_t t = tb + i;
      if ((t - c.t0) % every == 0) {
        float *dst = ckpt + ((base + (t - c.t0) / every) * H + c.h) * D * D;
#pragma unroll
        for (int j = 0; j < kRows; ++j)
          *reinterpret_cast<float2 *>(dst + (r0 + j) * D + col) = make_float2(s[j][0], s[j][1]);
      }
      float2 p, d;
      fwd_token(s, x, p, d, st, i, r0, ca, lane, warp, red, rp);
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
  __shared__ Stage st, st_rec;  // the group's inputs; a recomputed earlier group's
  __shared__ Red red;
  uint32_t rp = 0;
  __shared__ float s_p[kGroup][kCols], s_d[kGroup][kCols];
  __shared__ __align__(16) float ckbuf[D][kCols];  // the block's stored state, this CTA's columns
  __shared__ __align__(16) uint8_t raw[kRawBytes];
  const Chain c = chain_of(cu, n_seqs, n_tokens, H);
  if (!c.ok) return;  // recorded by the forward pass
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ca = 2 * (lane & 15), r0 = 16 * warp + kRows * (lane >> 4);
  const int col = c.cb * kCols + ca;
  const int64_t sbase = ((int64_t)c.seq * H + c.h) * D * D;
  float ds[kRows][2];
#pragma unroll
  for (int j = 0; j < kRows; ++j)
#pragma unroll
    for (int z = 0; z < 2; ++z) ds[j][z] = d_final ? d_final[sbase + (r0 + j) * D + col + z] : 0.f;
  const int64_t base = ckpt_base(c.t0, c.seq, every);
  const int64_t len = c.t1 - c.t0;
  const int64_t n_ck = (len + every - 1) / every;
  // Work items (block blk of `every` tokens, group g of kGroup tokens in it), in
  // reverse.  Each item's stored state and own inputs are copied while the item
  // before it runs; the inputs of the groups it recomputes are loaded in place.
  auto block_end = [&](int64_t blk) {
    const int64_t e = c.t0 + (blk + 1) * every;
    return e < c.t1 ? e : c.t1;
  };
  auto groups_of = [&](int64_t blk) {
    return (int)((block_end(blk) - (c.t0 + blk * every) + kGroup - 1) / kGroup);
  };
  float nbeta = 0.f;
  auto prefetch = [&](int64_t blk, int g) {
    const float *src = ckpt + ((base + blk) * H + c.h) * D * D + c.cb * kCols;
    for (int e = threadIdx.x; e < D * (kCols / 4); e += kThreads) {
      const int row = e / (kCols / 4), q4 = e % (kCols / 4);
      cp_async16(&ckbuf[row][4 * q4], src + row * D + 4 * q4);
    }
    const int64_t gb = c.t0 + blk * every + (int64_t)g * kGroup;
    const int64_t e = block_end(blk);
    const int n = (int)(e - gb < kGroup ? e - gb : kGroup);
    prefetch_tokens<BF16>(raw, gb, n, c.h, H, c.cb, true, q, k, v, la, dout);
    if (threadIdx.x < n) nbeta = beta[(gb + threadIdx.x) * H + c.h];
  };
  if (n_ck > 0) prefetch(n_ck - 1, groups_of(n_ck - 1) - 1);
  for (int64_t blk = n_ck - 1; blk >= 0; --blk) {
    const int64_t a = c.t0 + blk * every;
    const int64_t e = block_end(blk);
    const int n_groups = groups_of(blk);
    for (int g = n_groups - 1; g >= 0; --g) {
      const int64_t gb = a + (int64_t)g * kGroup;
      const int n = (int)(e - gb < kGroup ? e - gb : kGroup);
      // the item's copies have landed: the state before token a, the group's inputs
      cp_async_wait_all();
      __syncthreads();
      float s[kRows][2], x[kRows][2];
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        const float2 v2 = *reinterpret_cast<const float2 *>(&ckbuf[r0 + j][ca]);
        s[j][0] = v2.x;
        s[j][1] = v2.y;
      }
      convert_tokens<BF16>(st, raw, n, true, nbeta);
      __syncthreads();  // ckbuf and raw are free; st is ready
      if (g > 0) prefetch(blk, g - 1);
      else if (blk > 0) prefetch(blk - 1, groups_of(blk - 1) - 1);
      // forward to the group's first token
      for (int64_t tb = a; tb < gb; tb += kGroup) {
        __syncthreads();
        stage_tokens<BF16>(st_rec, tb, kGroup, c.h, H, c.cb, nullptr, k, v, la, beta, nullptr);
        __syncthreads();
        for (int i = 0; i < kGroup; ++i) {
          float2 p, d;
          fwd_token(s, x, p, d, st_rec, i, r0, ca, lane, warp, red, rp);
        }
      }
      // the group's tokens: X, p and d kept
      for (int i = 0; i < n; ++i) {
        float2 p, d;
        fwd_token(s, x, p, d, st, i, r0, ca, lane, warp, red, rp);
#pragma unroll
        for (int j = 0; j < kRows; ++j)
          *reinterpret_cast<float2 *>(&xs[(i * D + r0 + j) * kCols + ca]) = make_float2(x[j][0], x[j][1]);
        if (warp == 0 && lane < 16) {
          *reinterpret_cast<float2 *>(&s_p[i][ca]) = p;
          *reinterpret_cast<float2 *>(&s_d[i][ca]) = d;
        }
      }
      __syncthreads();
      // ... in reverse
      for (int i = n - 1; i >= 0; --i) {
        const int64_t t = gb + i;
        const int64_t trow = (t * H + c.h) * D;
        const float2 p = *reinterpret_cast<const float2 *>(&s_p[i][ca]);
        const float2 d = *reinterpret_cast<const float2 *>(&s_d[i][ca]);
        const float b = st.beta[i];
        const float2 dov = make_float2(st.dout[i][ca], st.dout[i][ca + 1]);
        float cq[kRows], ck[kRows], cl[kRows], xa[kRows], xb[kRows];
        float pa = 0.f, pb = 0.f;
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const int r = r0 + j;
          const float2 xv = *reinterpret_cast<const float2 *>(&xs[(i * D + r) * kCols + ca]);
          const float kr = st.k[i][r], qr = st.q[i][r];
          // S_t do (row sums: dq), over this thread's two columns
          cq[j] = fmaf(fmaf(kr, d.x, xv.x), dov.x, fmaf(kr, d.y, xv.y) * dov.y);
          ds[j][0] = fmaf(qr, dov.x, ds[j][0]);          // dS += q do^T
          ds[j][1] = fmaf(qr, dov.y, ds[j][1]);
          pa = fmaf(ds[j][0], kr, pa);                   // dd = dS^T k (column sums)
          pb = fmaf(ds[j][1], kr, pb);
          xa[j] = xv.x;                                  // X, kept for the next pass
          xb[j] = xv.y;
        }
        pa += __shfl_xor_sync(0xffffffffu, pa, 16);
        pb += __shfl_xor_sync(0xffffffffu, pb, 16);
        float (&rb)[kThreads / 32][kCols] = red[rp++ & 1u];
        if (lane < 16) *reinterpret_cast<float2 *>(&rb[warp][ca]) = make_float2(pa, pb);
        __syncthreads();
        float2 dd = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
          const float2 v2 = *reinterpret_cast<const float2 *>(&rb[w][ca]);
          dd.x += v2.x;
          dd.y += v2.y;
        }
        const float2 dp = make_float2(-b * dd.x, -b * dd.y);
        if (warp == 0) {
          if (lane < 16) {
            if constexpr (BF16) {  // (dv is only element-aligned: two scalar stores)
              static_cast<__nv_bfloat16 *>(dv_out)[trow + col] = __float2bfloat16_rn(b * dd.x);
              static_cast<__nv_bfloat16 *>(dv_out)[trow + col + 1] = __float2bfloat16_rn(b * dd.y);
            } else {
              static_cast<float *>(dv_out)[trow + col] = b * dd.x;
              static_cast<float *>(dv_out)[trow + col + 1] = b * dd.y;
            }
          }
          // (both half-warps hold the same column pairs: sum within one half)
          float db = dd.x * (st.v[i][ca] - p.x) + dd.y * (st.v[i][ca + 1] - p.y);
#pragma unroll
          for (int off = 8; off > 0; off >>= 1) db += __shfl_xor_sync(0xffffffffu, db, off);
          if (lane == 0) atomicAdd(dbeta + t * H + c.h, db);
        }
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const int r = r0 + j;
          const float kr = st.k[i][r], al = st.alpha[i][r];
          const float dx0 = fmaf(kr, dp.x, ds[j][0]);     // dX = dS + k dp^T
          const float dx1 = fmaf(kr, dp.y, ds[j][1]);
          ck[j] = fmaf(ds[j][0], d.x, fmaf(xa[j], dp.x, fmaf(ds[j][1], d.y, xb[j] * dp.y)));  // dk: dS d + X dp
          cl[j] = fmaf(dx0, xa[j], dx1 * xb[j]);          // dlog_alpha: dX o X
          ds[j][0] = al * dx0;                             // dS_{t-1} = Diag(alpha) dX
          ds[j][1] = al * dx1;
        }
        const float sq = row_sum(cq, lane), sk = row_sum(ck, lane), sl = row_sum(cl, lane);
        if ((lane & 1) == 0) {
          const int r = r0 + row_of(lane);
          atomicAdd(dq_acc + trow + r, sq);
          atomicAdd(dk_acc + trow + r, sk);
          atomicAdd(dla + trow + r, sl);
        }
      }
    }
  }
  if (d_init) {
#pragma unroll
    for (int j = 0; j < kRows; ++j)
#pragma unroll
      for (int z = 0; z < 2; ++z) d_init[sbase + (r0 + j) * D + col + z] = ds[j][z];
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
  if (a.chunked) {
    if (!a.bf16 || a.ckpt_every != kBwdChunk) return cudaErrorInvalidValue;
    return launch_bwd_chunk(a, stream);  // its own checkpoint pass, then the chunks
  }
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
