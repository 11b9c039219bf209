// bf16 chunkwise KDA prefill on the 5th-generation tensor cores (tcgen05).
//
// One CTA (8 warps) carries one (sequence, head) chain through chunks of C = 64
// tokens.  The fp32 state lives in tensor memory for the whole chain; every
// dense contraction of a chunk is a tcgen05.mma (bf16 operands, fp32 TMEM
// accumulators); q, k, v and log_alpha tiles arrive by TMA with a 128-byte
// swizzle, prefetched one chunk ahead.
//
// Chunk algebra ("Kimi K3: 架构、训练与系统全景解析", section 4.2.4: state passed
// between chunks, lower-triangular matrix work inside, output = pre-chunk-state
// term + intra-chunk causal term; UT-transform form of the solve), with g_r the
// within-chunk cumulative log-decay per key channel and S the incoming state:
//   A = strict_lower(Diag(beta) [k_r . k_i e^{g_r - g_i}]),  T = (I + A)^{-1}
//   T' = T Diag(beta),  U = T' V,  W = T' (K o e^{g})
//   Delta = U - W S,  O = (Q o e^{g}) S + P Delta,  P = lower_incl([q_r . k_i e^{g_r - g_i}])
//   S <- Diag(e^{g_C}) S + (K o e^{g_C - g})^T Delta
//
// Decay factorisation on tensor cores.  The ratio e^{g_r - g_i} is split as
// e^{g_r - R} e^{R - g_i} with one reference R per 16-token column tile b: R =
// ref_b = cumulative log-decay at the end of tile b.  Because log_alpha >= -5,
// a 16-token tile spans at most 80 in log-decay, so for i in tile b
// e^{ref_b - g_i} is in [e^-80, 1] and for rows r of tile b e^{g_r - ref_b} is
// in [1, e^80]; rows of later tiles give factors <= 1 ("Kimi K3: 架构、训练与系统
// 全景解析", section 4.2.5: a 16-token tile's cumulative log-decay lies in
// (-80, 0), its reciprocal within e^80, so diagonal and off-diagonal tiles both
// run as dense tensor-core matmuls).  Every factor is representable in bf16 and
// fp32, and a factor only underflows where the exact product is below e^-87.
// Row factors are built from E_r = e^{g_r - start(tile(r))} (in [e^-80, 1]) times
// one per-(tile, channel) constant, so each element costs two exponentials.
//
// TMEM orientation: the state is held transposed (S^T: lane = value index n,
// column = key index c), so every state-side product is an M = 128 MMA with
// the bf16 copy of S^T (or Delta^T) as a TMEM A operand:
//   U^T  = V^T T'^T           (A = V, smem MN-major;  B = T', K-major)
//   W^T  = Kt^T T'^T          (A = Kt, smem MN-major)
//   O^T  = S^T Qt^T           (A = bf16 S^T in TMEM;  B = Qt, K-major)
//   D^T  = U^T - S^T W^T      (accumulate, B = -W, MN-major)
//   O^T += Delta^T P^T        (A = bf16 Delta^T in TMEM; B = P, K-major)
//   S^T += Delta^T Kdec       (B = Kdec, MN-major), after S^T <- S^T Diag(e^{g_C})
// The Gram and P matrices are 4 MMAs of M = 128 (rows: 64 key rows then 64
// query rows of one factor version), N = 16 (one column tile), K = 128.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int D = kHeadDim;  // 128
constexpr int C = kChunk;    // 64
constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on any single wait: 2 s
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory map (byte offsets from a 1024-byte aligned base).  Operand
// tiles use 128-byte rows with the 128-byte swizzle; a "K-major tile of R rows"
// stores columns 0-63 as R rows of 128 B, then columns 64-127 likewise.
constexpr uint32_t SM_Q = 0;                  // q chunk (TMA), 64 rows
constexpr uint32_t SM_K = SM_Q + 16384;       // k chunk (TMA), 64 rows
constexpr uint32_t SM_V = SM_K + 16384;       // v chunk (TMA), 64 rows
constexpr uint32_t SM_LA = SM_V + 16384;      // log_alpha fp32 [64][128]; then [Kt; Qt], 128 rows
constexpr uint32_t SM_VX = SM_LA + 32768;     // factor version buffer X, 128 rows; then fp32 A
constexpr uint32_t SM_VY = SM_VX + 32768;     // factor version buffer Y, 128 rows; then fp32 T
constexpr uint32_t SM_KHAT = SM_VY + 32768;   // K o e^{ref_b - g}, 64 rows
constexpr uint32_t SM_KDEC = SM_KHAT + 16384; // K o e^{g_C - g}, 64 rows
constexpr uint32_t SM_TMAT = SM_KDEC + 16384; // T' = T Diag(beta), [64 r][64 i]
constexpr uint32_t SM_PMAT = SM_TMAT + 8192;  // P, [64 r][64 i]
constexpr uint32_t SM_WMAT = SM_PMAT + 8192;  // -W, stored [128 c][64 r]
constexpr uint32_t SM_MISC = SM_WMAT + 16384;

constexpr int AP = 68;  // pitch (floats) of the fp32 64 x 64 matrices in SM_VX / SM_VY

struct Misc {
  float beta[C];
  float gammaC[D];
  float tot[4][D];
  uint64_t bar_qk, bar_la, bar_v;                        // TMA arrivals
  uint64_t bar_vx, bar_vy, bar_gp, bar_wu, bar_m1, bar_m2, bar_fin;  // MMA completions
  uint32_t tmem_base;
  int abort;
  uint32_t tma_issued[3], tma_waited[3];  // per TMA barrier: phases issued / consumed
};

constexpr uint32_t SMEM_BYTES = SM_MISC + sizeof(Misc) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(64 * AP * 4 + 3 * 256 * 4 <= 32768, "fp32 matrices fit a version buffer");

// TMEM columns (fp32 cells).
constexpr uint32_t TM_S = 0;     // S^T, 128 columns
constexpr uint32_t TM_AS = 128;  // bf16 S^T (A operand), 64 columns
constexpr uint32_t TM_U = 192;   // U^T, then Delta^T (fp32), 64 columns
constexpr uint32_t TM_O = 256;   // O^T, 64 columns
constexpr uint32_t TM_GP = 320;  // [Gram; P] rows x 64 column-tile columns
constexpr uint32_t TM_W = 384;   // W^T, 64 columns
constexpr uint32_t TM_AD = 448;  // bf16 Delta^T (A operand), 32 columns
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_GP = idesc_bf16(128, 16, false, false);
constexpr uint32_t ID_UW = idesc_bf16(128, 64, true, false);
constexpr uint32_t ID_KK64 = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_KM64 = idesc_bf16(128, 64, false, true);
constexpr uint32_t ID_KM128 = idesc_bf16(128, 128, false, true);

enum { TMA_QK = 0, TMA_LA = 1, TMA_V = 2 };

__device__ __forceinline__ void cta_sync() {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ void record_status(DeviceStatus *st, int code, int detail, int chain, int chunk) {
  if (atomicCAS(&st->code, 0, code) == 0) {
    st->detail = detail;
    st->chain = chain;
    st->chunk = chunk;
  }
}

// Byte offset of the bf16 pair (row, c..c+1), c even, in a K-major tile whose
// 64-column halves hold `rows` rows each.
__device__ __forceinline__ uint32_t kmaj_off(uint32_t rows, int row, int c) {
  return (uint32_t)(c >> 6) * rows * 128u + sw128_offset(row, (uint32_t)(c & 63) * 2u);
}

__device__ __forceinline__ float2 ld_pair(const uint8_t *tile, uint32_t rows, int row, int c) {
  return unpack_bf16x2(*reinterpret_cast<const uint32_t *>(tile + kmaj_off(rows, row, c)));
}

__device__ __forceinline__ void st_pair(uint8_t *tile, uint32_t rows, int row, int c, float x,
                                        float y) {
  *reinterpret_cast<uint32_t *>(tile + kmaj_off(rows, row, c)) = pack_bf16x2(x, y);
}

struct Ctx {
  uint8_t *smem;
  Misc *m;
  DeviceStatus *status;
  int chain;
};

// Bounded mbarrier wait; on timeout records KDA_ERR_TIMEOUT and raises the abort
// flag.  The flag is only tested right after a CTA-wide barrier, so every thread
// leaves the chunk loop at the same point.
__device__ bool wait_bar(const Ctx &x, uint64_t *bar, uint32_t parity, int where, int chunk) {
  if (mbar_wait(bar, parity, kWaitNs)) return true;
  record_status(x.status, KDA_ERR_TIMEOUT, where, x.chain, chunk);
  atomicExch(&x.m->abort, 1);
  return false;
}

__device__ __forceinline__ uint64_t kdesc(const uint8_t *tile_base, uint32_t byte_off) {
  return sdesc_sw128(smem_u32(tile_base) + byte_off, 16, 1024);
}
__device__ __forceinline__ uint64_t mndesc(const uint8_t *tile_base, uint32_t byte_off,
                                           uint32_t lbo) {
  return sdesc_sw128(smem_u32(tile_base) + byte_off, lbo, 1024);
}

__global__ void __launch_bounds__(kThreads, 1)
kda_chunk_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_la, const float *__restrict__ beta,
                        const float *__restrict__ init_state,
                        const int32_t *__restrict__ cu_seqlens, int32_t n_seqs, int64_t n_tokens,
                        int32_t H, __nv_bfloat16 *__restrict__ out,
                        float *__restrict__ final_state, DeviceStatus *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Misc &m = *reinterpret_cast<Misc *>(smem + SM_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chain = blockIdx.x;
  const int seq = chain / H, h = chain % H;
  const Ctx cx{smem, &m, status, chain};

  const int64_t t0 = cu_seqlens[seq], t1 = cu_seqlens[seq + 1];
  if (t0 < 0 || t1 < t0 || t1 > n_tokens ||
      (chain == 0 && (cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != n_tokens))) {
    if (tid == 0) record_status(status, KDA_ERR_INVALID_ARG, 1, chain, -1);
    return;
  }
  const int64_t len = t1 - t0;
  const int n_chunks = (int)((len + C - 1) / C);

  if (tid == 0) {
    mbar_init(&m.bar_qk, 1); mbar_init(&m.bar_la, 1); mbar_init(&m.bar_v, 1);
    mbar_init(&m.bar_vx, 1); mbar_init(&m.bar_vy, 1); mbar_init(&m.bar_gp, 1);
    mbar_init(&m.bar_wu, 1); mbar_init(&m.bar_m1, 1); mbar_init(&m.bar_m2, 1);
    mbar_init(&m.bar_fin, 1);
    fence_mbarrier_init();
    m.abort = 0;
    for (int i = 0; i < 3; ++i) m.tma_issued[i] = m.tma_waited[i] = 0;
  }
  if (warp == 0) {
    tmem_alloc(&m.tmem_base, TM_COLS);
    tmem_relinquish();
  }
  cta_sync();
  const uint32_t tm = m.tmem_base;
  const int q4 = warp & 3, hf = warp >> 2;     // TMEM lane quadrant, column half
  const uint32_t lane_base = 32u * q4;

  // Issues the TMA loads of chunk `ci` (thread 0 only).
  auto issue_qk = [&](int ci) {
    const int32_t tb = (int32_t)(t0 + (int64_t)C * ci);
    mbar_arrive_expect_tx(&m.bar_qk, 2 * 16384);
    tma_load_3d(smem + SM_Q, &tm_q, &m.bar_qk, 0, h, tb);
    tma_load_3d(smem + SM_Q + 8192, &tm_q, &m.bar_qk, 64, h, tb);
    tma_load_3d(smem + SM_K, &tm_k, &m.bar_qk, 0, h, tb);
    tma_load_3d(smem + SM_K + 8192, &tm_k, &m.bar_qk, 64, h, tb);
    m.tma_issued[TMA_QK]++;
  };
  auto issue_la = [&](int ci) {
    const int32_t tb = (int32_t)(t0 + (int64_t)C * ci);
    mbar_arrive_expect_tx(&m.bar_la, 32768);
    tma_load_3d(smem + SM_LA, &tm_la, &m.bar_la, 0, h, tb);
    m.tma_issued[TMA_LA]++;
  };
  auto issue_v = [&](int ci) {
    const int32_t tb = (int32_t)(t0 + (int64_t)C * ci);
    mbar_arrive_expect_tx(&m.bar_v, 16384);
    tma_load_3d(smem + SM_V, &tm_v, &m.bar_v, 0, h, tb);
    tma_load_3d(smem + SM_V + 8192, &tm_v, &m.bar_v, 64, h, tb);
    m.tma_issued[TMA_V]++;
  };

  if (tid == 0 && n_chunks > 0) {
    prefetch_tensormap(&tm_q); prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v); prefetch_tensormap(&tm_la);
    issue_qk(0); issue_la(0); issue_v(0);
  }

  // ---- initial state -> S^T in TMEM (thread: lane n, 64 key columns of its half)
  const int64_t sbase = ((int64_t)seq * H + h) * D * D;
  {
    const int n = lane_base + lane;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const int c0 = 64 * hf + 32 * part;
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        r[j] = __float_as_uint(init_state ? init_state[sbase + (int64_t)(c0 + j) * D + n] : 0.f);
      tmem_st32(tmem_addr(tm, lane_base, TM_S + c0), r);
    }
    tmem_st_wait();
  }
  cta_sync();

  bool failed = false;
  for (int ci = 0; ci < n_chunks && !failed; ++ci) {
    const uint32_t par = (uint32_t)(ci & 1);
    const int64_t tb = t0 + (int64_t)C * ci;
    const int nv = (int)((len - (int64_t)C * ci) < C ? (len - (int64_t)C * ci) : C);
    const bool has_next = ci + 1 < n_chunks;

    // ================= phase 1: decay factors and operand tiles (all threads)
    const bool ok_qk = wait_bar(cx, &m.bar_qk, par, 10, ci);
    const bool ok_la = wait_bar(cx, &m.bar_la, par, 11, ci);
    const int a = tid >> 6, cp = tid & 63, c = 2 * cp;
    float L0[16], L1[16];
    if (ok_qk && ok_la) {
      const float *la = reinterpret_cast<const float *>(smem + SM_LA);
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int row = 16 * a + j;
        float2 x = *reinterpret_cast<const float2 *>(la + row * D + c);
        if (row >= nv) x = make_float2(0.f, 0.f);
        s0 = fmaf(x.x, kLog2e, s0);
        s1 = fmaf(x.y, kLog2e, s1);
        L0[j] = s0;
        L1[j] = s1;
      }
      m.tot[a][c] = s0;
      m.tot[a][c + 1] = s1;
    }
    if (tid < C) m.beta[tid] = tid < nv ? beta[(tb + tid) * H + h] : 0.f;
    if (tid == 0) {
      if (ok_qk) m.tma_waited[TMA_QK]++;
      if (ok_la) m.tma_waited[TMA_LA]++;
    }
    cta_sync();
    if (m.abort) { failed = true; break; }

    // Tile starts st[b] and ends rf[b] of the cumulative log2-decay, channels c, c+1.
    float st0[4], st1[4], rf0[4], rf1[4];
    {
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        st0[b] = acc0; st1[b] = acc1;
        acc0 += m.tot[b][c]; acc1 += m.tot[b][c + 1];
        rf0[b] = acc0; rf1[b] = acc1;
      }
    }
    const float sa0 = a == 0 ? st0[0] : a == 1 ? st0[1] : a == 2 ? st0[2] : st0[3];
    const float sa1 = a == 0 ? st1[0] : a == 1 ? st1[1] : a == 2 ? st1[2] : st1[3];
    const float ra0 = a == 0 ? rf0[0] : a == 1 ? rf0[1] : a == 2 ? rf0[2] : rf0[3];
    const float ra1 = a == 0 ? rf1[0] : a == 1 ? rf1[1] : a == 2 ? rf1[2] : rf1[3];
    const float gC0 = rf0[3], gC1 = rf1[3];
    const float tot0 = ra0 - sa0, tot1 = ra1 - sa1;

    // E_r = 2^{L_r} (row side, relative to the tile start); Ec_r = 2^{tot - L_r}.
    float E0[16], E1[16];
    {
      uint8_t *khat = smem + SM_KHAT, *kdec = smem + SM_KDEC, *stack = smem + SM_LA;
      const float fd0 = ex2(gC0 - ra0), fd1 = ex2(gC1 - ra1);   // e^{g_C - ref_a}
      const float fs0 = ex2(sa0), fs1 = ex2(sa1);               // e^{start_a}
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int row = 16 * a + j;
        E0[j] = ex2(L0[j]);
        E1[j] = ex2(L1[j]);
        const float ec0 = ex2(tot0 - L0[j]), ec1 = ex2(tot1 - L1[j]);
        const float2 kk = ld_pair(smem + SM_K, 64, row, c);
        const float2 qq = ld_pair(smem + SM_Q, 64, row, c);
        st_pair(khat, 64, row, c, kk.x * ec0, kk.y * ec1);
        st_pair(kdec, 64, row, c, kk.x * (ec0 * fd0), kk.y * (ec1 * fd1));
        const float e0 = E0[j] * fs0, e1 = E1[j] * fs1;          // e^{g_r}
        st_pair(stack, 128, row, c, kk.x * e0, kk.y * e1);
        st_pair(stack, 128, 64 + row, c, qq.x * e0, qq.y * e1);
      }
      if (a == 0) { m.gammaC[c] = ex2(gC0); m.gammaC[c + 1] = ex2(gC1); }
    }
    // Factor version b: rows of tiles a >= b scaled by e^{g_r - ref_b}.
    auto build_version = [&](uint8_t *buf, int b) {
      const float rb0 = b == 0 ? rf0[0] : b == 1 ? rf0[1] : b == 2 ? rf0[2] : rf0[3];
      const float rb1 = b == 0 ? rf1[0] : b == 1 ? rf1[1] : b == 2 ? rf1[2] : rf1[3];
      const float f0 = ex2(sa0 - rb0), f1 = ex2(sa1 - rb1);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int row = 16 * a + j;
        const float2 kk = ld_pair(smem + SM_K, 64, row, c);
        const float2 qq = ld_pair(smem + SM_Q, 64, row, c);
        const float e0 = E0[j] * f0, e1 = E1[j] * f1;
        st_pair(buf, 128, row, c, kk.x * e0, kk.y * e1);
        st_pair(buf, 128, 64 + row, c, qq.x * e0, qq.y * e1);
      }
    };
    auto issue_gp = [&](const uint8_t *buf, int b) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t ad = kdesc(buf, (ks >> 2) * 16384u + (ks & 3) * 32u);
        const uint64_t bd = kdesc(smem + SM_KHAT, (ks >> 2) * 8192u + 2048u * b + (ks & 3) * 32u);
        umma_ss(tm + TM_GP + 16 * b, ad, bd, ID_GP, ks > 0 ? 1u : 0u);
      }
    };
    build_version(smem + SM_VX, 0);
    fence_proxy_async_smem();
    cta_sync();
    if (tid == 0) { issue_gp(smem + SM_VX, 0); umma_commit(&m.bar_vx); }
    if (a >= 1) build_version(smem + SM_VY, 1);
    fence_proxy_async_smem();
    cta_sync();
    if (tid == 0) { issue_gp(smem + SM_VY, 1); umma_commit(&m.bar_vy); }
    wait_bar(cx, &m.bar_vx, par, 20, ci);
    if (a >= 2) build_version(smem + SM_VX, 2);
    fence_proxy_async_smem();
    cta_sync();
    if (m.abort) { failed = true; break; }
    if (tid == 0) issue_gp(smem + SM_VX, 2);
    wait_bar(cx, &m.bar_vy, par, 21, ci);
    if (a >= 3) build_version(smem + SM_VY, 3);
    fence_proxy_async_smem();
    cta_sync();
    if (m.abort) { failed = true; break; }
    if (tid == 0) {
      issue_gp(smem + SM_VY, 3);
      umma_commit(&m.bar_gp);
      if (has_next) issue_qk(ci + 1);   // q, k tiles are no longer read
    }

    // ================= phase 2: A (fp32, for the solve) and P (bf16 operand)
    wait_bar(cx, &m.bar_gp, par, 22, ci);
    tc_fence_after();
    {
      uint32_t r[32];
      tmem_ld32(tmem_addr(tm, lane_base, TM_GP + 32 * hf), r);
      tmem_ld_wait(r);
      if (q4 < 2) {
        const int row = 32 * q4 + lane;
        const float br = m.beta[row];
        float *amat = reinterpret_cast<float *>(smem + SM_VX);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int i = 32 * hf + j;
          amat[row * AP + i] = i < row ? br * __uint_as_float(r[j]) : 0.f;
        }
      } else {
        const int row = 32 * (q4 - 2) + lane;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t w[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int j = 8 * g + 2 * t, i = 32 * hf + j;
            const float lo = i <= row ? __uint_as_float(r[j]) : 0.f;
            const float hi = i + 1 <= row ? __uint_as_float(r[j + 1]) : 0.f;
            w[t] = pack_bf16x2(lo, hi);
          }
          st_shared_v4(smem_u32(smem + SM_PMAT) + sw128_offset(row, (32 * hf + 8 * g) * 2),
                       w[0], w[1], w[2], w[3]);
        }
      }
    }
    cta_sync();
    if (m.abort) { failed = true; break; }

    // ================= phase 3: T = (I + A)^{-1}, blocked by 16 x 16 tiles
    {
      const float *amat = reinterpret_cast<const float *>(smem + SM_VX);
      float *tinv = reinterpret_cast<float *>(smem + SM_VY);
      float *xb = tinv + 64 * AP;
      if (warp < 4 && lane < 16) {  // diagonal blocks by forward substitution
        const int a0 = 16 * warp, j = lane;
        float tcol[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float acc = 0.f;
#pragma unroll
          for (int mm = 0; mm < r; ++mm) acc = fmaf(amat[(a0 + r) * AP + a0 + mm], tcol[mm], acc);
          tcol[r] = (j == r) ? 1.f : ((j < r) ? -acc : 0.f);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) tinv[(a0 + r) * AP + a0 + j] = tcol[r];
      }
      __syncthreads();
      // Off-diagonal blocks by distance d = a - b:
      //   T_ab = -T_aa * sum_{m=b}^{a-1} A_am T_mb
#pragma unroll 1
      for (int d = 1; d < 4; ++d) {
        const int nblk = 4 - d;
        for (int e = tid; e < nblk * 256; e += kThreads) {
          const int blk = e >> 8, r = (e >> 4) & 15, jj = e & 15;
          const int ab = d + blk, bb = blk;
          float acc = 0.f;
          for (int mm = bb; mm < ab; ++mm)
#pragma unroll
            for (int l = 0; l < 16; ++l)
              acc = fmaf(amat[(16 * ab + r) * AP + 16 * mm + l],
                         tinv[(16 * mm + l) * AP + 16 * bb + jj], acc);
          xb[blk * 256 + r * 16 + jj] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nblk * 256; e += kThreads) {
          const int blk = e >> 8, r = (e >> 4) & 15, jj = e & 15;
          const int ab = d + blk, bb = blk;
          float acc = 0.f;
#pragma unroll
          for (int l = 0; l < 16; ++l)
            acc = fmaf(tinv[(16 * ab + r) * AP + 16 * ab + l], xb[blk * 256 + l * 16 + jj], acc);
          tinv[(16 * ab + r) * AP + 16 * bb + jj] = -acc;
        }
        __syncthreads();
      }
      // T' = T Diag(beta) -> bf16, K-major [r][i]; upper triangle zero.
      {
        const int row = tid >> 2, qd = tid & 3;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t w[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int i0 = 16 * qd + 8 * half + 2 * t;
            const float lo = i0 <= row ? tinv[row * AP + i0] * m.beta[i0] : 0.f;
            const float hi = i0 + 1 <= row ? tinv[row * AP + i0 + 1] * m.beta[i0 + 1] : 0.f;
            w[t] = pack_bf16x2(lo, hi);
          }
          st_shared_v4(smem_u32(smem + SM_TMAT) + sw128_offset(row, (16 * qd + 8 * half) * 2),
                       w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
    }

    // ================= phase 4: S pass (scale by e^{g_C}, bf16 copy as A operand)
    {
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int c0 = 64 * hf + 32 * part;
        uint32_t s[32];
        tmem_ld32(tmem_addr(tm, lane_base, TM_S + c0), s);
        tmem_ld_wait(s);
        uint32_t ab[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const float f0 = __uint_as_float(s[2 * jj]), f1 = __uint_as_float(s[2 * jj + 1]);
          ab[jj] = pack_bf16x2(f0, f1);
          s[2 * jj] = __float_as_uint(f0 * m.gammaC[c0 + 2 * jj]);
          s[2 * jj + 1] = __float_as_uint(f1 * m.gammaC[c0 + 2 * jj + 1]);
        }
        tmem_st32(tmem_addr(tm, lane_base, TM_S + c0), s);
        tmem_st16(tmem_addr(tm, lane_base, TM_AS + c0 / 2), ab);
      }
      tmem_st_wait();
    }
    cta_sync();
    if (tid == 0) {
      if (wait_bar(cx, &m.bar_v, par, 12, ci)) {
        m.tma_waited[TMA_V]++;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {   // U^T = V^T T'^T ; W^T = Kt^T T'^T
          const uint64_t bd = kdesc(smem + SM_TMAT, ks * 32u);
          umma_ss(tm + TM_U, mndesc(smem + SM_V, ks * 2048u, 8192), bd, ID_UW, ks > 0);
          umma_ss(tm + TM_W, mndesc(smem + SM_LA, ks * 2048u, 16384), bd, ID_UW, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {   // O^T = S^T Qt^T
          const uint64_t bd = kdesc(smem + SM_LA, 64u * 128u + (ks >> 2) * 16384u + (ks & 3) * 32u);
          umma_ts(tm + TM_O, tm + TM_AS + 8 * ks, bd, ID_KK64, ks > 0);
        }
        umma_commit(&m.bar_wu);
      }
    }

    // ================= phase 5: -W -> smem; Delta^T = U^T - S^T W^T
    wait_bar(cx, &m.bar_wu, par, 23, ci);
    tc_fence_after();
    if (tid == 0 && has_next) { issue_v(ci + 1); issue_la(ci + 1); }
    {
      uint32_t r[32];
      tmem_ld32(tmem_addr(tm, lane_base, TM_W + 32 * hf), r);
      tmem_ld_wait(r);
      const int crow = lane_base + lane;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          w[t] = pack_bf16x2(-__uint_as_float(r[8 * g + 2 * t]), -__uint_as_float(r[8 * g + 2 * t + 1]));
        st_shared_v4(smem_u32(smem + SM_WMAT) + sw128_offset(crow, (32 * hf + 8 * g) * 2), w[0],
                     w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
    }
    cta_sync();
    if (m.abort) { failed = true; break; }
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_ts(tm + TM_U, tm + TM_AS + 8 * ks, mndesc(smem + SM_WMAT, ks * 2048u, 8192), ID_KM64, 1u);
      umma_commit(&m.bar_m1);
    }

    // ================= phase 6: bf16 Delta^T; O^T += Delta^T P^T; S^T += Delta^T Kdec
    wait_bar(cx, &m.bar_m1, par, 24, ci);
    tc_fence_after();
    {
      uint32_t r[32];
      tmem_ld32(tmem_addr(tm, lane_base, TM_U + 32 * hf), r);
      tmem_ld_wait(r);
      uint32_t ab[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj)
        ab[jj] = pack_bf16x2(__uint_as_float(r[2 * jj]), __uint_as_float(r[2 * jj + 1]));
      tmem_st16(tmem_addr(tm, lane_base, TM_AD + 16 * hf), ab);
      tmem_st_wait();
    }
    cta_sync();
    if (m.abort) { failed = true; break; }
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        umma_ts(tm + TM_O, tm + TM_AD + 8 * ks, kdesc(smem + SM_PMAT, ks * 32u), ID_KK64, 1u);
        umma_ts(tm + TM_S, tm + TM_AD + 8 * ks, mndesc(smem + SM_KDEC, ks * 2048u, 8192),
                ID_KM128, 1u);
      }
      umma_commit(&m.bar_m2);
    }

    // ================= phase 7: output rows of this chunk
    wait_bar(cx, &m.bar_m2, par, 25, ci);
    tc_fence_after();
    {
      uint32_t r[32];
      tmem_ld32(tmem_addr(tm, lane_base, TM_O + 32 * hf), r);
      tmem_ld_wait(r);
      const int n = lane_base + lane;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int rr = 32 * hf + j;
        if (rr < nv) out[((tb + rr) * H + h) * D + n] = __float2bfloat16_rn(__uint_as_float(r[j]));
      }
    }
  }

  cta_sync();
  if (!failed && !m.abort) {
    if (final_state) {
      const int n = lane_base + lane;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int c0 = 64 * hf + 32 * part;
        uint32_t r[32];
        tmem_ld32(tmem_addr(tm, lane_base, TM_S + c0), r);
        tmem_ld_wait(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) final_state[sbase + (int64_t)(c0 + j) * D + n] = __uint_as_float(r[j]);
      }
    }
  } else if (tid == 0) {
    // Drain what is still in flight (bounded), so no copy or MMA outlives the CTA.
    umma_commit(&m.bar_fin);
    mbar_wait(&m.bar_fin, 0, kWaitNs);
    uint64_t *bars[3] = {&m.bar_qk, &m.bar_la, &m.bar_v};
    for (int i = 0; i < 3; ++i)
      if (m.tma_issued[i] > m.tma_waited[i]) mbar_wait(bars[i], m.tma_waited[i] & 1u, kWaitNs);
  }
  cta_sync();
  if (warp == 0) tmem_dealloc(tm, TM_COLS);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// 3-D map over a token-major [N, H, 128] tensor: box = (box_x channels, 1 head, 64 tokens).
bool make_map(CUtensorMap *map, const void *base, CUtensorMapDataType dt, uint32_t esz, int64_t N,
              int32_t H, uint32_t box_x, CUtensorMapSwizzle sw) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)N};
  const cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)H * D * esz};
  const cuuint32_t box[3] = {box_x, 1, (cuuint32_t)C};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_fwd_bf16_tc(const ChunkArgs &a, cudaStream_t stream) {
  const int64_t chains = (int64_t)a.n_seqs * a.H;
  if (chains == 0) return cudaSuccess;
  if (chains > 0x7fffffffLL || a.n_tokens > 0x7fffffffLL - C) return cudaErrorInvalidValue;
  if (!encode_fn()) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv, mla;
  memset(&mq, 0, sizeof(mq)); memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv)); memset(&mla, 0, sizeof(mla));
  if (a.n_tokens > 0) {
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_map(&mq, a.q, bf, 2, a.n_tokens, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mk, a.k, bf, 2, a.n_tokens, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mv, a.v, bf, 2, a.n_tokens, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mla, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.n_tokens, a.H, 128,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(kda_chunk_fwd_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kda_chunk_fwd_tc_kernel<<<(unsigned)chains, kThreads, SMEM_BYTES, stream>>>(
      mq, mk, mv, mla, a.beta, a.init_state, a.cu_seqlens, a.n_seqs, a.n_tokens, a.H,
      static_cast<__nv_bfloat16 *>(a.out), a.final_state, a.status);
  return cudaGetLastError();
}

}  // namespace kda
