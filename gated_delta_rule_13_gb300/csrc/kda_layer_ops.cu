// The per-token operations either side of the KDA recurrence, each one HBM pass.
//
// Before the recurrence ("Kimi K3: 架构、训练与系统全景解析", section 4.2.3; "Kimi K3"
// study notes, section 3-2 "2) Kimi Delta Attention"): a short causal
// convolution (kernel size 4) of q, k and v within each sequence, Swish, and an
// L2 normalisation of q and k; beta = sigmoid(b) and the lower-bounded decay
// log_alpha = -5 sigmoid(a) (全景解析 sections 2.1 and 4.2.5).  After it
// (全景解析 section 4.2.6): head-wise RMSNorm of the recurrent output times a
// sigmoid output gate whose logits come from the full-rank projection.
//   conv:    y[t] = sum_j w[j] x[t - 3 + j], zero before the sequence start
//   swish:   x sigmoid(x)
//   l2norm:  x / sqrt(sum_c x^2 + 1e-6)
//   rmsnorm: o / sqrt(mean_c o^2 + 1e-5) * gamma[c]
//
// Lane l of a warp owns channels 4l .. 4l + 3 of one (token, head) row, so both
// per-token reductions over the 128 channels are warp shuffles.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int D = kHeadDim;
constexpr int kWarps = 8;
constexpr int kTokensPerCta = 64;
constexpr int kConv = 4;
constexpr float kL2Eps = 1e-6f;
constexpr float kRmsEps = 1e-5f;
constexpr float kDecayBound = -5.0f;

template <bool BF16>
__device__ __forceinline__ float4 ld4(const void *p, int64_t i) {
  if constexpr (BF16) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p) + i);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
    return make_float4(a.x, a.y, b.x, b.y);
  } else {
    return *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
  }
}

template <bool BF16>
__device__ __forceinline__ void st4(void *p, int64_t i, float4 x) {
  if constexpr (BF16) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
    uint2 raw;
    raw.x = *reinterpret_cast<const uint32_t *>(&lo);
    raw.y = *reinterpret_cast<const uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p) + i) = raw;
  } else {
    *reinterpret_cast<float4 *>(static_cast<float *>(p) + i) = x;
  }
}

// sigmoid through the fast exponential and the approximate divide (relative
// error ~1e-6, far below the bf16 rounding of q, k, v and within the fp32 gate
// tolerance); 1 + e^-x = inf for very negative x gives exactly 0.
__device__ __forceinline__ float sigmoidf(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// The taps of channels c0 .. c0 + 3 of head h from one [H, d, 4] weight tensor.
__device__ __forceinline__ void load_taps(float4 (&w)[4], const float *wt, int h, int c0) {
  const float4 *wv = reinterpret_cast<const float4 *>(wt + ((int64_t)h * D + c0) * kConv);
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = wv[i];
}

__device__ __forceinline__ float4 scale4(float4 x, float s) {
  return make_float4(x.x * s, x.y * s, x.z * s, x.w * s);
}

// Four channels of one row as loaded: packed bf16 pairs or fp32.
template <bool BF16> struct Raw4;
template <> struct Raw4<true> { using type = uint2; };
template <> struct Raw4<false> { using type = float4; };
template <bool BF16> using raw4_t = typename Raw4<BF16>::type;

template <bool BF16>
__device__ __forceinline__ raw4_t<BF16> ld_raw(const void *p, int64_t i) {
  if constexpr (BF16)
    return *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p) + i);
  else
    return *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
}

template <bool BF16> __device__ __forceinline__ raw4_t<BF16> raw_zero() {
  if constexpr (BF16) return make_uint2(0u, 0u);
  else return make_float4(0.f, 0.f, 0.f, 0.f);
}

template <bool BF16> __device__ __forceinline__ float4 to_f4(raw4_t<BF16> r) {
  if constexpr (BF16) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
  } else {
    return r;
  }
}

__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_float(float x) { return x; }
template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ float from_float<float>(float x) { return x; }

// Index of the sequence holding token t: the last s < n_seqs with cu[s] <= t.
__device__ __forceinline__ int sequence_of(const int32_t *cu, int32_t n_seqs, int64_t t) {
  int lo = 0, hi = n_seqs;  // invariant: answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// Convolution of rows x0 .. x3 (tokens t-3 .. t) with taps w (w[i]: the four
// taps of channel c0 + i, oldest first), then Swish.
__device__ __forceinline__ float4 conv_swish(float4 x0, float4 x1, float4 x2, float4 x3,
                                             const float4 (&w)[4]) {
  float4 y;
  y.x = w[0].x * x0.x + w[0].y * x1.x + w[0].z * x2.x + w[0].w * x3.x;
  y.y = w[1].x * x0.y + w[1].y * x1.y + w[1].z * x2.y + w[1].w * x3.y;
  y.z = w[2].x * x0.z + w[2].y * x1.z + w[2].z * x2.z + w[2].w * x3.z;
  y.w = w[3].x * x0.w + w[3].y * x1.w + w[3].z * x2.w + w[3].w * x3.w;
  y.x *= sigmoidf(y.x);
  y.y *= sigmoidf(y.y);
  y.z *= sigmoidf(y.z);
  y.w *= sigmoidf(y.w);
  return y;
}

// Work split: blockIdx.z picks the output (0 q, 1 k, 2 v, 3 the gates), the
// CTA's kWarps warps take kWarps consecutive heads (one 2 KB bf16 span per
// token), and each warp walks kRunTokens consecutive tokens.  For q, k, v the
// warp slides a window of the three previous raw rows through registers and
// loads the next kGroup rows while it works on the current ones, so each input
// row is read once, plus a three-row halo per run.
constexpr int kRunTokens = 128;

template <bool BF16, bool kWindow>
__global__ void __launch_bounds__(32 * kWarps, 4)
kda_prep_kernel(const void *__restrict__ q_raw, const void *__restrict__ k_raw,
                const void *__restrict__ v_raw, const float *__restrict__ conv_w,
                const float *__restrict__ a_logit, const float *__restrict__ b_logit,
                const int32_t *__restrict__ cu_seqlens, int32_t n_seqs, int64_t n_tokens,
                int32_t H, void *__restrict__ q, void *__restrict__ k, void *__restrict__ v,
                float *__restrict__ log_alpha, float *__restrict__ beta,
                const void *__restrict__ win_in) {
  constexpr int kGroup = BF16 ? 4 : 2;  // rows in flight per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kWarps + warp;
  if (h >= H) return;
  const int c0 = 4 * lane;
  const int64_t t0 = (int64_t)blockIdx.x * kRunTokens;
  const int64_t t_end = t0 + kRunTokens < n_tokens ? t0 + kRunTokens : n_tokens;
  auto row_of = [&](int64_t t) { return (t * H + h) * D + c0; };

  if (blockIdx.z == 3) {  // gates: log_alpha = -5 sigmoid(a), beta = sigmoid(b)
    for (int64_t tb = t0 + lane; tb < t_end; tb += 32) beta[tb * H + h] = sigmoidf(b_logit[tb * H + h]);
    const int64_t rs = (int64_t)H * D;
    const float *ain = a_logit + row_of(t0);
    float *aout = log_alpha + row_of(t0);
    const int n_run = (int)(t_end - t0);
    for (int ig = 0; ig < n_run; ig += 4) {
      float4 g[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (ig + i < n_run) g[i] = *reinterpret_cast<const float4 *>(ain + i * rs);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (ig + i < n_run)
          *reinterpret_cast<float4 *>(aout + i * rs) =
              make_float4(kDecayBound * sigmoidf(g[i].x), kDecayBound * sigmoidf(g[i].y),
                          kDecayBound * sigmoidf(g[i].z), kDecayBound * sigmoidf(g[i].w));
      ain += 4 * rs;
      aout += 4 * rs;
    }
    return;
  }

  const int z = blockIdx.z;
  const void *x = z == 0 ? q_raw : (z == 1 ? k_raw : v_raw);
  void *y = z == 0 ? q : (z == 1 ? k : v);
  const bool normalise = z < 2;
  float4 w[4];
  load_taps(w, conv_w + (int64_t)z * H * D * kConv, h, c0);

  // sequence bookkeeping (token indices fit int32, like cu_seqlens): ts = first
  // token of the current sequence, nxt = the start of the next one
  int s = sequence_of(cu_seqlens, n_seqs, t0);
  int32_t ts = cu_seqlens[s];
  int32_t nxt = s + 1 < n_seqs ? cu_seqlens[s + 1] : INT32_MAX;

  // element pointers to this lane's channels of token t0, advanced token by token
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, float>::type;
  const int64_t rs = (int64_t)H * D;  // elements between consecutive tokens
  const elem_t *xin = static_cast<const elem_t *>(x) + row_of(t0);
  elem_t *yout = static_cast<elem_t *>(y) + row_of(t0);
  raw4_t<BF16> w0, w1, w2;  // raw rows t-3, t-2, t-1 (zero before token 0)
  w0 = t0 >= 3 ? ld_raw<BF16>(xin - 3 * rs, 0) : raw_zero<BF16>();
  w1 = t0 >= 2 ? ld_raw<BF16>(xin - 2 * rs, 0) : raw_zero<BF16>();
  w2 = t0 >= 1 ? ld_raw<BF16>(xin - rs, 0) : raw_zero<BF16>();
  raw4_t<BF16> cur[kGroup], ahead[kGroup];
  const int n_run = (int)(t_end - t0);
#pragma unroll
  for (int i = 0; i < kGroup; ++i) {
    cur[i] = i < n_run ? ld_raw<BF16>(xin, 0) : raw_zero<BF16>();
    xin += rs;
  }
  for (int ig = 0; ig < n_run; ig += kGroup) {
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {  // xin points at token t0 + ig + kGroup + i
      ahead[i] = ig + kGroup + i < n_run ? ld_raw<BF16>(xin, 0) : raw_zero<BF16>();
      xin += rs;
    }
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      if (ig + i >= n_run) break;
      const int32_t t = (int32_t)t0 + ig + i;
      while (t >= nxt) {  // crossed into a later sequence (warp-uniform)
        ++s;
        ts = nxt;
        nxt = s + 1 < n_seqs ? cu_seqlens[s + 1] : INT32_MAX;
      }
      const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 x0, x1, x2;
      if constexpr (!kWindow) {  // zeros before the sequence start
        const int32_t start = ts < t ? ts : t;
        x0 = t - 3 >= start ? to_f4<BF16>(w0) : zero;
        x1 = t - 2 >= start ? to_f4<BF16>(w1) : zero;
        x2 = t - 1 >= start ? to_f4<BF16>(w2) : zero;
      } else {
        x0 = to_f4<BF16>(w0);
        x1 = to_f4<BF16>(w1);
        x2 = to_f4<BF16>(w2);
        if (t - 3 < ts) {
          // taps before the sequence start read the carried window (rows oldest
          // first: tap j of token ts + u is window row u + j), or zeros
          const int u = t - ts;
          auto tap = [&](int j, float4 x) -> float4 {
            if (t - 3 + j >= ts) return x;
            if (win_in == nullptr) return zero;
            return to_f4<BF16>(ld_raw<BF16>(win_in, (((int64_t)s * 3 + z) * 3 + (u + j)) * rs +
                                                        (int64_t)h * D + c0));
          };
          x0 = tap(0, x0);
          x1 = tap(1, x1);
          x2 = tap(2, x2);
        }
      }
      float4 o = conv_swish(x0, x1, x2, to_f4<BF16>(cur[i]), w);
      if (normalise)
        o = scale4(o, rsqrtf(warp_sum(o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w) + kL2Eps));
      st4<BF16>(yout, 0, o);
      yout += rs;
      w0 = w1;
      w1 = w2;
      w2 = cur[i];
    }
#pragma unroll
    for (int i = 0; i < kGroup; ++i) cur[i] = ahead[i];
  }
}

template <bool BF16>
__global__ void __launch_bounds__(32 * kWarps)
kda_post_kernel(const void *__restrict__ o, const void *__restrict__ g,
                const float *__restrict__ gamma, int64_t n_tokens, int32_t H,
                void *__restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, c0 = 4 * lane;
  const float4 gm = *reinterpret_cast<const float4 *>(gamma + c0);
  // two tokens per step, so each warp has four rows in flight
  for (int i = warp; i < kTokensPerCta; i += 2 * kWarps) {
    const int64_t ta = (int64_t)blockIdx.x * kTokensPerCta + i, tb = ta + kWarps;
    if (ta >= n_tokens) break;
    const bool has_b = tb < n_tokens;
    const int64_t ra = (ta * H + h) * D + c0, rb = (tb * H + h) * D + c0;
    const float4 oa = ld4<BF16>(o, ra), ga = ld4<BF16>(g, ra);
    float4 ob = oa, gb = ga;
    if (has_b) { ob = ld4<BF16>(o, rb); gb = ld4<BF16>(g, rb); }
    const float sa = warp_sum(oa.x * oa.x + oa.y * oa.y + oa.z * oa.z + oa.w * oa.w);
    const float sb = warp_sum(ob.x * ob.x + ob.y * ob.y + ob.z * ob.z + ob.w * ob.w);
    const float na = rsqrtf(sa * (1.0f / D) + kRmsEps), nb = rsqrtf(sb * (1.0f / D) + kRmsEps);
    st4<BF16>(out, ra,
              make_float4(oa.x * na * gm.x * sigmoidf(ga.x), oa.y * na * gm.y * sigmoidf(ga.y),
                          oa.z * na * gm.z * sigmoidf(ga.z), oa.w * na * gm.w * sigmoidf(ga.w)));
    if (has_b)
      st4<BF16>(out, rb,
                make_float4(ob.x * nb * gm.x * sigmoidf(gb.x), ob.y * nb * gm.y * sigmoidf(gb.y),
                            ob.z * nb * gm.z * sigmoidf(gb.z), ob.w * nb * gm.w * sigmoidf(gb.w)));
  }
}

// The carried window after a prep call: per sequence s and tensor z (q, k, v),
// the three raw rows before the token after the call, oldest first: the
// sequence's last three rows, or for a shorter one the newest rows of the
// window it started from (zeros without one) followed by all of its rows.
// Every lane reads its three rows before it writes any, so the window may be
// updated in place; a malformed device cu_seqlens gives zeros, never an
// out-of-range access.
template <bool BF16>
__global__ void __launch_bounds__(32 * kWarps)
kda_conv_window_kernel(const void *__restrict__ q_raw, const void *__restrict__ k_raw,
                       const void *__restrict__ v_raw, const int32_t *__restrict__ cu_seqlens,
                       int32_t n_seqs, int64_t n_tokens, int32_t H, const void *win_in,
                       void *win_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x, z = blockIdx.y, h = blockIdx.z * kWarps + warp;
  if (h >= H) return;
  const int c0 = 4 * lane;
  const int64_t rs = (int64_t)H * D;
  const void *x = z == 0 ? q_raw : (z == 1 ? k_raw : v_raw);
  const int64_t a = cu_seqlens[s], e = cu_seqlens[s + 1];
  const bool ok = a >= 0 && e >= a && e <= n_tokens;
  const int64_t len = ok ? e - a : 0;
  raw4_t<BF16> row[3];
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int64_t t = e - 3 + r;  // token of window row r
    if (!ok) row[r] = raw_zero<BF16>();
    else if (t >= a) row[r] = ld_raw<BF16>(x, t * rs + (int64_t)h * D + c0);
    else if (win_in != nullptr)
      row[r] = ld_raw<BF16>(win_in, (((int64_t)s * 3 + z) * 3 + (r + len)) * rs + (int64_t)h * D + c0);
    else row[r] = raw_zero<BF16>();
  }
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int64_t i = (((int64_t)s * 3 + z) * 3 + r) * rs + (int64_t)h * D + c0;
    if constexpr (BF16) *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(win_out) + i) = row[r];
    else *reinterpret_cast<float4 *>(static_cast<float *>(win_out) + i) = row[r];
  }
}

// The whole layer between its projections, replayed over the accepted draft
// tokens of a speculative step ("Kimi K3: 架构、训练与系统全景解析", KDA state
// replay under speculative decoding: short convolution, norms, gating, the KDA
// recurrence and the output norm in one kernel over the accepted prefix, the
// state and the convolution window written back once).  Unit (b, h), tokens
// t < n_b = n_accept[b] clamped to [0, T], 8 warps, the tokens in groups of up
// to kLrGroup (three block barriers per group):
//   threads 0-127 (channel c): q and k of channel c for every token of the
//     group (window, convolution, Swish), then L2Norm over the 128 channels;
//   threads 128-255 (channel c - 128): v (window, convolution, Swish), the
//     decay alpha = e^{-5 sigmoid(a)}, the output gate sigmoid(g), and beta;
//   then every warp applies the group's tokens in order to its value columns of
//   the state held in registers (the decode step's layout), and the group's
//   output rows go through the head-wise RMSNorm times gamma times the gate
//   before they are stored.
// Nothing is read or written for a unit with no accepted token.
//
// The CTAs are persistent (two per SM) and walk the units with a stride of the
// grid.  While one unit's tokens run, bulk copies already bring the next unit's
// state, its convolution taps and window, and the raw inputs of its first
// kLrStageTok tokens into a shared-memory stage (its beta logits by 4-byte
// asynchronous copies), so a unit starts without a round trip to HBM.  The
// issuing thread waits on no load either: the accepted count of the unit after
// next is copied the same way, one unit ahead of its use.
constexpr int kLrStageTok = 4;                       // tokens whose inputs ride in the prefetch
constexpr int kLrGroup = 4;                          // tokens prepared together
constexpr uint32_t kLrTapBytes = 3 * D * kConv * 4;  // the unit's q, k, v taps
template <bool BF16>
constexpr uint32_t lr_esz() { return BF16 ? 2 : 4; }
// Staged token: q, k, v, g rows in the input type, then the fp32 decay logits.
template <bool BF16>
constexpr uint32_t lr_tok_bytes() { return 4 * D * lr_esz<BF16>() + 4 * D; }
template <bool BF16>
constexpr uint32_t lr_win_bytes() { return 9 * D * lr_esz<BF16>(); }
// Stage: state [D][D] fp32, taps [3][D][4] fp32, window [3][3][D], tokens.
constexpr uint32_t kLrOffTaps = D * D * 4, kLrOffWin = kLrOffTaps + kLrTapBytes;
template <bool BF16>
constexpr uint32_t lr_off_tok() { return kLrOffWin + lr_win_bytes<BF16>(); }
template <bool BF16>
constexpr size_t lr_stage_bytes() { return lr_off_tok<BF16>() + kLrStageTok * lr_tok_bytes<BF16>(); }
static_assert(kLrOffWin % 16 == 0 && lr_off_tok<true>() % 16 == 0 && lr_off_tok<false>() % 16 == 0,
              "bulk-copy destinations are 16-byte aligned");
constexpr uint64_t kLrWaitNs = 2000000000ull;  // bound on the stage's copy wait


template <bool BF16>
__device__ __forceinline__ float lr_elem(const uint8_t *row, int c) {
  if constexpr (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(row)[c]);
  else return reinterpret_cast<const float *>(row)[c];
}

template <bool BF16>
__global__ void __launch_bounds__(256, 2)
kda_layer_replay_kernel(float *__restrict__ state, void *__restrict__ win,
                        const void *__restrict__ q_raw, const void *__restrict__ k_raw,
                        const void *__restrict__ v_raw, const float *__restrict__ a_logit,
                        const float *__restrict__ b_logit, const void *__restrict__ g,
                        const float *__restrict__ conv_w, const float *__restrict__ gamma,
                        const int32_t *__restrict__ n_accept, int32_t T, int32_t H,
                        int64_t units, void *__restrict__ out) {
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, float>::type;
  constexpr uint32_t kEsz = lr_esz<BF16>(), kTok = lr_tok_bytes<BF16>();
  extern __shared__ __align__(128) uint8_t stage[];
  // the group's prepared tokens and raw output rows
  __shared__ __align__(16) float s_q[kLrGroup][D], s_k[kLrGroup][D], s_v[kLrGroup][D];
  __shared__ __align__(16) float s_alpha[kLrGroup][D], s_gate[kLrGroup][D], s_o[kLrGroup][D];
  __shared__ __align__(16) float s_gamma[D];
  __shared__ float s_red[kLrGroup][3][kWarps];
  __shared__ float s_beta[kLrGroup];
  __shared__ __align__(16) float s_w[3][D][kConv];           // the unit's taps of q, k, v
  __shared__ __align__(16) uint8_t s_tok[kLrStageTok * kTok];  // its first tokens' raw inputs
  __shared__ float s_blog[2][kLrStageTok];  // beta logits of the first tokens, by unit parity
  __shared__ int64_t s_cand;                 // the next unit to look at (thread 0)
  __shared__ int32_t s_cand_n;               // its accepted count, unclamped
  __shared__ __align__(8) uint64_t bar;
  __shared__ int64_t s_next;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int col = 16 * warp + 4 * (lane & 3);
  const int row0 = lane >> 2;
  const int role = tid >> 7, c = tid & (D - 1);
  const int za = role == 0 ? 0 : 2;
  const int64_t rs = (int64_t)H * D;  // elements per [H, D] row
  auto accepted = [&](int64_t u) {
    const int n = n_accept[u / H];
    return n < 0 ? 0 : (n > T ? T : n);
  };
  // thread 0: the next unit with accepted tokens from s_cand on (stride
  // gridDim.x), its stage copies issued and its first beta logits copied into
  // s_blog[slot].  The accepted count of the candidate after it is copied
  // asynchronously too, a unit ahead of its use, so that issuing the stage
  // waits on no load unless a unit without accepted tokens is skipped.
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
    const int cnt = n_u < kLrStageTok ? n_u : kLrStageTok;
    const int64_t b = u / H;
    const int h = (int)(u % H);
    const uint32_t s0 = smem_u32(stage);
    mbar_arrive_expect_tx(&bar, kLrOffWin + lr_win_bytes<BF16>() + (uint32_t)cnt * kTok);
    bulk_load(s0, state + u * (int64_t)(D * D), D * D * 4, &bar);
#pragma unroll
    for (int z = 0; z < 3; ++z)
      bulk_load(s0 + kLrOffTaps + z * (D * kConv * 4), conv_w + ((int64_t)z * H + h) * D * kConv,
                D * kConv * 4, &bar);
#pragma unroll
    for (int zr = 0; zr < 9; ++zr)
      bulk_load(s0 + kLrOffWin + zr * (D * kEsz),
                static_cast<const elem_t *>(win) + ((b * 3 + zr / 3) * 3 + zr % 3) * rs + (int64_t)h * D,
                D * kEsz, &bar);
#pragma unroll
    for (int t = 0; t < kLrStageTok; ++t) {
      if (t < cnt) {
        const int64_t row = ((b * T + t) * H + h) * D;
        const uint32_t dst = s0 + lr_off_tok<BF16>() + t * kTok;
        bulk_load(dst, static_cast<const elem_t *>(q_raw) + row, D * kEsz, &bar);
        bulk_load(dst + D * kEsz, static_cast<const elem_t *>(k_raw) + row, D * kEsz, &bar);
        bulk_load(dst + 2 * D * kEsz, static_cast<const elem_t *>(v_raw) + row, D * kEsz, &bar);
        bulk_load(dst + 3 * D * kEsz, static_cast<const elem_t *>(g) + row, D * kEsz, &bar);
        bulk_load(dst + 4 * D * kEsz, a_logit + row, D * 4, &bar);
        cp_async4(&s_blog[slot][t], b_logit + (b * T + t) * H + h);
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
  if (tid < D) s_gamma[tid] = gamma[tid];
  __syncthreads();
  int64_t u = s_next;
  uint32_t phase = 0;
  while (u < units) {
    const bool landed = mbar_wait(&bar, phase, kLrWaitNs);
    if (tid == 0) cp_async_wait_all();  // the beta logits and the next candidate's count
    if (__syncthreads_or(!landed)) {  // a copy that never lands: leave, every thread alike
      if (tid == 0) mbar_wait(&bar, phase, kLrWaitNs);  // (bounded) no copy outlives the CTA
      return;
    }
    const int slot = (int)phase;  // this unit's parity
    phase ^= 1u;
    const int64_t b = u / H;
    const int h = (int)(u % H);
    const int n = accepted(u);
    // ---- the stage into registers and the unit's own shared arrays
    float4 st[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      st[j] = *reinterpret_cast<const float4 *>(stage + 4 * ((row0 + 8 * j) * D + col));
    for (int e = tid; e < 3 * D; e += 256)
      *reinterpret_cast<float4 *>(&s_w[0][0][0] + 4 * e) =
          *reinterpret_cast<const float4 *>(stage + kLrOffTaps + 16 * e);
    float xa[3], xb[3];  // channel c's carried window rows (role 0: q and k, role 1: v)
    {
      const uint8_t *sw = stage + kLrOffWin;
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        xa[r] = lr_elem<BF16>(sw + (3 * za + r) * (D * kEsz), c);
        xb[r] = role == 0 ? lr_elem<BF16>(sw + (3 + r) * (D * kEsz), c) : 0.f;
      }
    }
    {
      const int cnt = n < kLrStageTok ? n : kLrStageTok;
      const uint4 *src = reinterpret_cast<const uint4 *>(stage + lr_off_tok<BF16>());
      for (int e = tid; e < cnt * (int)(kTok / 16); e += 256)
        reinterpret_cast<uint4 *>(s_tok)[e] = src[e];
    }
    __syncthreads();  // the stage is free for the next unit; the taps and inputs are in place
    if (tid == 0) prefetch_next(slot ^ 1);

    float *S = state + u * (int64_t)(D * D);
    for (int t0 = 0; t0 < n; t0 += kLrGroup) {
      const int gn = n - t0 < kLrGroup ? n - t0 : kLrGroup;
      if (t0 > 0) __syncthreads();  // the last group's output rows are out of the arrays
      // ---- convolution + Swish of the group's tokens, the window shifted token
      // by token; raw inputs staged for the first tokens, else from HBM
#pragma unroll
      for (int gi = 0; gi < kLrGroup; ++gi) {
        if (gi < gn) {
          const int t = t0 + gi;
          const int64_t tok = (b * T + t) * H + h;
          float ra, rb = 0.f, rg = 0.f, rl = 0.f;
          if (t < kLrStageTok) {
            const uint8_t *tb = s_tok + t * kTok;
            if (role == 0) {
              ra = lr_elem<BF16>(tb, c);
              rb = lr_elem<BF16>(tb + D * kEsz, c);
            } else {
              ra = lr_elem<BF16>(tb + 2 * D * kEsz, c);
              rg = lr_elem<BF16>(tb + 3 * D * kEsz, c);
              rl = reinterpret_cast<const float *>(tb + 4 * D * kEsz)[c];
            }
          } else {
            const int64_t row = tok * D + c;
            if (role == 0) {
              ra = to_float(static_cast<const elem_t *>(q_raw)[row]);
              rb = to_float(static_cast<const elem_t *>(k_raw)[row]);
            } else {
              ra = to_float(static_cast<const elem_t *>(v_raw)[row]);
              rl = a_logit[row];
              rg = to_float(static_cast<const elem_t *>(g)[row]);
            }
          }
          const float4 wa = *reinterpret_cast<const float4 *>(s_w[za][c]);
          float y = wa.x * xa[0] + wa.y * xa[1] + wa.z * xa[2] + wa.w * ra;
          y *= sigmoidf(y);
          xa[0] = xa[1]; xa[1] = xa[2]; xa[2] = ra;
          if (role == 0) {
            const float4 wb = *reinterpret_cast<const float4 *>(s_w[1][c]);
            float y2 = wb.x * xb[0] + wb.y * xb[1] + wb.z * xb[2] + wb.w * rb;
            y2 *= sigmoidf(y2);
            xb[0] = xb[1]; xb[1] = xb[2]; xb[2] = rb;
            // q and k before the L2Norm, and their sums of squares (warps 0-3)
            s_q[gi][c] = y;
            s_k[gi][c] = y2;
            const float sq = warp_sum(y * y), sk = warp_sum(y2 * y2);
            if (lane == 0) { s_red[gi][0][warp] = sq; s_red[gi][1][warp] = sk; }
          } else {
            s_v[gi][c] = y;
            s_alpha[gi][c] = __expf(kDecayBound * sigmoidf(rl));
            s_gate[gi][c] = sigmoidf(rg);
            if (c == 0) s_beta[gi] = sigmoidf(t < kLrStageTok ? s_blog[slot][t] : b_logit[tok]);
          }
        }
      }
      __syncthreads();
      if (role == 0) {
#pragma unroll
        for (int gi = 0; gi < kLrGroup; ++gi) {
          if (gi < gn) {
            const float nq = rsqrtf(s_red[gi][0][0] + s_red[gi][0][1] + s_red[gi][0][2] +
                                    s_red[gi][0][3] + kL2Eps);
            const float nk = rsqrtf(s_red[gi][1][0] + s_red[gi][1][1] + s_red[gi][1][2] +
                                    s_red[gi][1][3] + kL2Eps);
            s_q[gi][c] *= nq;
            s_k[gi][c] *= nk;
          }
        }
      }
      __syncthreads();
      // ---- the recurrence over the group's tokens, on this warp's value columns
      for (int gi = 0; gi < gn; ++gi) {
        const float4 vv = *reinterpret_cast<const float4 *>(&s_v[gi][col]);
        const float bt = s_beta[gi];
        const float *qg = s_q[gi], *kg = s_k[gi], *ag = s_alpha[gi];
        float pk0 = 0.f, pk1 = 0.f, pk2 = 0.f, pk3 = 0.f;
        float pq0 = 0.f, pq1 = 0.f, pq2 = 0.f, pq3 = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = row0 + 8 * j;
          const float al = ag[r], kr = kg[r], qr = qg[r];
          st[j].x *= al; st[j].y *= al; st[j].z *= al; st[j].w *= al;
          pk0 = fmaf(kr, st[j].x, pk0); pk1 = fmaf(kr, st[j].y, pk1);
          pk2 = fmaf(kr, st[j].z, pk2); pk3 = fmaf(kr, st[j].w, pk3);
          pq0 = fmaf(qr, st[j].x, pq0); pq1 = fmaf(qr, st[j].y, pq1);
          pq2 = fmaf(qr, st[j].z, pq2); pq3 = fmaf(qr, st[j].w, pq3);
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
        for (int j = 0; j < D / 32; ++j) kq = fmaf(kg[lane + 32 * j], qg[lane + 32 * j], kq);
        kq = warp_sum(kq);
        const float u0 = bt * (vv.x - pk0), u1 = bt * (vv.y - pk1);
        const float u2 = bt * (vv.z - pk2), u3 = bt * (vv.w - pk3);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float kr = kg[row0 + 8 * j];
          st[j].x = fmaf(kr, u0, st[j].x); st[j].y = fmaf(kr, u1, st[j].y);
          st[j].z = fmaf(kr, u2, st[j].z); st[j].w = fmaf(kr, u3, st[j].w);
        }
        // the raw output row and its sum of squares, for the norm below
        const float o0 = fmaf(kq, u0, pq0), o1 = fmaf(kq, u1, pq1);
        const float o2 = fmaf(kq, u2, pq2), o3 = fmaf(kq, u3, pq3);
        float ss = o0 * o0 + o1 * o1 + o2 * o2 + o3 * o3;  // lanes 0-3 hold distinct columns
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        if (row0 == 0) *reinterpret_cast<float4 *>(&s_o[gi][col]) = make_float4(o0, o1, o2, o3);
        if (lane == 0) s_red[gi][2][warp] = ss;
      }
      __syncthreads();
      // ---- head-wise RMSNorm of the group's output rows times gamma times the
      // gate (32 threads per row, four columns each)
      if (out != nullptr && tid < 32 * gn) {
        const int gi = tid >> 5, c4 = 4 * lane;
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tot += s_red[gi][2][w];
        const float nr = rsqrtf(tot * (1.0f / D) + kRmsEps);
        const float4 o = *reinterpret_cast<const float4 *>(&s_o[gi][c4]);
        const float4 gt = *reinterpret_cast<const float4 *>(&s_gate[gi][c4]);
        const float4 gm = *reinterpret_cast<const float4 *>(&s_gamma[c4]);
        st4<BF16>(out, ((b * T + t0 + gi) * H + h) * D + c4,
                  make_float4(o.x * nr * gm.x * gt.x, o.y * nr * gm.y * gt.y,
                              o.z * nr * gm.z * gt.z, o.w * nr * gm.w * gt.w));
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      __stcs(reinterpret_cast<float4 *>(S + (row0 + 8 * j) * D + col), st[j]);
    elem_t *wo = static_cast<elem_t *>(win);
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      wo[((b * 3 + za) * 3 + r) * rs + (int64_t)h * D + c] = from_float<elem_t>(xa[r]);
      if (role == 0) wo[((b * 3 + 1) * 3 + r) * rs + (int64_t)h * D + c] = from_float<elem_t>(xb[r]);
    }
    __syncthreads();  // s_next is set; the unit's shared arrays may be refilled
    u = s_next;
  }
}

}  // namespace

cudaError_t launch_prep(const void *q_raw, const void *k_raw, const void *v_raw,
                        const float *conv_w, const float *a_logit, const float *b_logit,
                        const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t H,
                        bool bf16, void *q, void *k, void *v, float *log_alpha, float *beta,
                        cudaStream_t stream) {
  if (n_tokens == 0 || H == 0) return cudaSuccess;
  const int64_t blocks = (n_tokens + kRunTokens - 1) / kRunTokens;
  if (blocks > 0x7fffffffLL || H > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)blocks, (unsigned)((H + kWarps - 1) / kWarps), 4), block(32 * kWarps);
  if (bf16)
    kda_prep_kernel<true, false><<<grid, block, 0, stream>>>(q_raw, k_raw, v_raw, conv_w, a_logit,
                                                      b_logit, cu_seqlens, n_seqs, n_tokens, H,
                                                      q, k, v, log_alpha, beta, nullptr);
  else
    kda_prep_kernel<false, false><<<grid, block, 0, stream>>>(q_raw, k_raw, v_raw, conv_w, a_logit,
                                                       b_logit, cu_seqlens, n_seqs, n_tokens, H,
                                                       q, k, v, log_alpha, beta, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_prep_window(const void *q_raw, const void *k_raw, const void *v_raw,
                               const float *conv_w, const float *a_logit, const float *b_logit,
                               const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens,
                               int32_t H, bool bf16, const void *win_in, void *win_out, void *q,
                               void *k, void *v, float *log_alpha, float *beta,
                               cudaStream_t stream) {
  if (H == 0 || n_seqs == 0) return cudaSuccess;
  if (n_tokens > 0) {
    const int64_t blocks = (n_tokens + kRunTokens - 1) / kRunTokens;
    if (blocks > 0x7fffffffLL || H > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)blocks, (unsigned)((H + kWarps - 1) / kWarps), 4);
    if (bf16)
      kda_prep_kernel<true, true><<<grid, 32 * kWarps, 0, stream>>>(
          q_raw, k_raw, v_raw, conv_w, a_logit, b_logit, cu_seqlens, n_seqs, n_tokens, H, q, k, v,
          log_alpha, beta, win_in);
    else
      kda_prep_kernel<false, true><<<grid, 32 * kWarps, 0, stream>>>(
          q_raw, k_raw, v_raw, conv_w, a_logit, b_logit, cu_seqlens, n_seqs, n_tokens, H, q, k, v,
          log_alpha, beta, win_in);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (win_out == nullptr) return cudaSuccess;
  // after the prep kernel on the same stream: an in-place window is read first
  if (n_seqs > 0x7fffffff || H > 65535 * kWarps) return cudaErrorInvalidValue;
  const dim3 wgrid((unsigned)n_seqs, 3, (unsigned)((H + kWarps - 1) / kWarps));
  if (bf16)
    kda_conv_window_kernel<true><<<wgrid, 32 * kWarps, 0, stream>>>(
        q_raw, k_raw, v_raw, cu_seqlens, n_seqs, n_tokens, H, win_in, win_out);
  else
    kda_conv_window_kernel<false><<<wgrid, 32 * kWarps, 0, stream>>>(
        q_raw, k_raw, v_raw, cu_seqlens, n_seqs, n_tokens, H, win_in, win_out);
  return cudaGetLastError();
}

cudaError_t launch_layer_replay(float *state, void *win, const void *q_raw, const void *k_raw,
                                const void *v_raw, const float *a_logit, const float *b_logit,
                                const void *g, const float *conv_w, const float *gamma,
                                const int32_t *n_accept, int32_t B, int32_t T, int32_t H,
                                bool bf16, void *out, cudaStream_t stream) {
  const int64_t units = (int64_t)B * H;
  if (units == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t ctas = units < 2 * (int64_t)sms ? units : 2 * (int64_t)sms;
  const size_t stage = bf16 ? lr_stage_bytes<true>() : lr_stage_bytes<false>();
  auto kern = bf16 ? kda_layer_replay_kernel<true> : kda_layer_replay_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stage);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)ctas, 256, stage, stream>>>(state, win, q_raw, k_raw, v_raw, a_logit, b_logit,
                                               g, conv_w, gamma, n_accept, T, H, units, out);
  return cudaGetLastError();
}

cudaError_t launch_post(const void *o, const void *g, const float *gamma, int64_t n_tokens,
                        int32_t H, bool bf16, void *out, cudaStream_t stream) {
  if (n_tokens == 0 || H == 0) return cudaSuccess;
  const int64_t blocks = (n_tokens + kTokensPerCta - 1) / kTokensPerCta;
  if (blocks > 0x7fffffffLL || H > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)blocks, (unsigned)H), block(32 * kWarps);
  if (bf16)
    kda_post_kernel<true><<<grid, block, 0, stream>>>(o, g, gamma, n_tokens, H, out);
  else
    kda_post_kernel<false><<<grid, block, 0, stream>>>(o, g, gamma, n_tokens, H, out);
  return cudaGetLastError();
}

}  // namespace kda
