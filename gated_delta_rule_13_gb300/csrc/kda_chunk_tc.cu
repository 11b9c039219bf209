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
// Decay factorisation on tensor cores.  With 16-token tiles a, b and per-channel
// tile starts st_a / ends ref_b of the cumulative log-decay,
//   e^{g_r - g_i} = e^{g_r - st_a} * e^{st_a - ref_b} * e^{ref_b - g_i}
// for row r in tile a >= b and column i in tile b.  Because log_alpha >= -5 a
// tile spans at most 80 in log-decay ("Kimi K3: 架构、训练与系统全景解析",
// section 4.2.5: the cumulative log-decay of a 16-token tile lies in (-80, 0)
// and its reciprocal within e^80, so diagonal and off-diagonal tiles both run
// as dense tensor-core matmuls): the row factor is in [e^-80, 1], the column
// factor e^{st_a - g_i} = e^{st_a - ref_b} e^{ref_b - g_i} is at most e^80 (a = b)
// or 1 (a > b), and a factor underflows only where the exact product is below
// e^-87.  So one row operand [K o E; Q o E] (E_r = e^{g_r - st_a}) serves every
// block, and the column operand holds one 16-row block per tile pair (a, b),
// a >= b: the Gram and P matrices of a chunk are 8 MMAs of M = 128 (64 key
// rows, 64 query rows), N = 160 (10 blocks), K = 16 each.
//
// TMEM orientation: the state is held transposed (S^T: lane = value index n,
// column = key index c), so every state-side product is an M = 128 MMA:
//   U^T  = V^T T'^T                 (A = V, smem MN-major;  B = T', K-major)
//   W^T  = Kt^T T'^T                (A = Kt, smem MN-major)
//   [O^T | D^T] = S^T [Qt; -W]^T    (A = bf16 S^T in TMEM; D^T accumulates onto U^T)
//   S^T += Delta^T Kdec, O^T += Delta^T P^T   (A = bf16 Delta^T in TMEM),
//                                    after S^T <- S^T Diag(e^{g_C})
// where D = Delta = U - W S.  32 tcgen05.mma instructions per chunk.  The
// triangular solve (warps 0-3) overlaps the previous chunk's output stores
// (warps 4-7), and the next chunk's decay prefix overlaps the state MMAs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

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
constexpr uint32_t SM_Q = 0;                    // q chunk (TMA), 64 rows; then output staging
constexpr uint32_t SM_K = SM_Q + 16384;         // k chunk (TMA), 64 rows
constexpr uint32_t SM_V = SM_K + 16384;         // v chunk (TMA), 64 rows
constexpr uint32_t SM_LA = SM_V + 16384;        // log_alpha fp32 [64][128]
constexpr uint32_t SM_GA = SM_LA + 32768;       // Gram rows [K o E; Q o E], 128 rows; then A^T fp32
constexpr uint32_t SM_GB = SM_GA + 32768;       // Gram columns, 160 rows; then T fp32, X, T'
constexpr uint32_t SM_STACK = SM_GB + 40960;    // [Qt; Kt -> -W], 128 rows
constexpr uint32_t SM_KDEC = SM_STACK + 32768;  // K o e^{g_C - g}, 64 rows (MN-major operand)
constexpr uint32_t SM_PMAT = SM_KDEC + 16384;   // P, K-major [64 r][64 i]
constexpr uint32_t SM_TMAT = SM_PMAT + 8192;    // T' = T Diag(beta), K-major [64 r][64 i]
constexpr uint32_t SM_MISC = SM_TMAT + 8192;

constexpr uint32_t GB_ROWS = 160;
constexpr uint32_t OFF_TINV = 0;               // inside SM_GB, after the Gram MMAs
constexpr uint32_t OFF_XBUF = 64 * 72 * 4;   // 4 blocks of 16 x XP fp32
constexpr int FP = 72;  // pitch (floats) of the fp32 64 x 64 matrices of the solve
constexpr int XP = 24;  // pitch (floats) of the 16 x 16 intermediate blocks


struct Misc {
  float beta[2][C];           // beta of the current chunk and the prefetched next one
  float tot[4][D];            // per-tile total log2-decay
  float gamma[D];             // Gamma_C = e^{g_C} per key channel
  uint64_t bar_qk, bar_la, bar_v;               // TMA arrivals
  uint64_t bar_gp, bar_wu, bar_m1, bar_m2, bar_fin;  // MMA completions
  uint32_t tmem_base;
  int abort;
  uint32_t tma_issued[3], tma_waited[3];  // per TMA barrier: phases issued / consumed
};

constexpr uint32_t SMEM_BYTES = SM_MISC + sizeof(Misc);
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(64 * FP * 4 <= 32768, "A^T fits SM_GA");
static_assert(OFF_XBUF + 4 * 16 * XP * 4 <= 40960, "T and X blocks fit SM_GB");

// TMEM columns (fp32 cells).
constexpr uint32_t TM_S = 0;     // S^T, 128 columns
constexpr uint32_t TM_O = 128;   // O^T, 64 columns       } O+M1 writes [O^T | U^T]
constexpr uint32_t TM_U = 192;   // U^T, then Delta^T (fp32), 64 columns
constexpr uint32_t TM_AS = 256;  // bf16 S^T (A operand), 64 columns
constexpr uint32_t TM_AD = 320;  // bf16 Delta^T (A operand), 32 columns
constexpr uint32_t TM_GP = 352;  // [Gram; P] rows x 160 block columns
constexpr uint32_t TM_W = 352;   // W^T, 64 columns (after the Gram/P epilogue)
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_GP = idesc_bf16(128, GB_ROWS, false, false);
constexpr uint32_t ID_UW = idesc_bf16(128, 64, true, false);
constexpr uint32_t ID_OM1 = idesc_bf16(128, 128, false, false);
constexpr uint32_t ID_KM128 = idesc_bf16(128, 128, false, true);
constexpr uint32_t ID_KK64 = idesc_bf16(128, 64, false, false);

enum { TMA_QK = 0, TMA_LA = 1, TMA_V = 2 };

// Optional per-phase cycle stamps of chain 0 (profiling builds only).
#ifdef KDA_PHASE_PROFILE
__device__ long long g_phase_clock[4096 * 16];
#define PHASE_MARK(i)                                                                    \
  do {                                                                                   \
    if (tid == 0 && chain == 0 && ci < 4096) g_phase_clock[ci * 16 + (i)] = clock64();  \
  } while (0)
#else
#define PHASE_MARK(i) \
  do {                \
  } while (0)
#endif

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

// 8 consecutive fp32 from shared memory (16-byte aligned).
__device__ __forceinline__ void ld8(float (&v)[8], const float *p) {
  const float4 a = *reinterpret_cast<const float4 *>(p);
  const float4 b = *reinterpret_cast<const float4 *>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void unpack8(float (&v)[8], uint4 u) {
  const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y);
  const float2 c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  v[4] = c.x; v[5] = c.y; v[6] = d.x; v[7] = d.y;
}

// Stores x[i] * f[i] (i < 8) as 8 bf16 at a shared address.
__device__ __forceinline__ void st8_scaled(uint32_t saddr, const float (&x)[8],
                                           const float (&f)[8]) {
  st_shared_v4(saddr, pack_bf16x2(x[0] * f[0], x[1] * f[1]), pack_bf16x2(x[2] * f[2], x[3] * f[3]),
               pack_bf16x2(x[4] * f[4], x[5] * f[5]), pack_bf16x2(x[6] * f[6], x[7] * f[7]));
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

// Block column index of tile pair (a, b), a >= b, in the Gram column operand.
__host__ __device__ constexpr int blk(int a, int b) { return a * (a + 1) / 2 + b; }

__global__ void __launch_bounds__(kThreads, 1)
kda_chunk_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_la, const float *__restrict__ beta,
                        const float *__restrict__ init_state,
                        const int32_t *__restrict__ cu_seqlens, int32_t n_seqs, int64_t n_tokens,
                        int32_t H, __nv_bfloat16 *__restrict__ out,
                        float *__restrict__ final_state, DeviceStatus *status) {
  // Indexing the __shared__ array directly (no integer round trip) keeps every
  // access a shared-memory instruction.  The 128-byte swizzle atoms need a
  // 1024-byte aligned base, checked below.
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc &m = *reinterpret_cast<Misc *>(smem + SM_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chain = blockIdx.x;
  const int seq = chain / H, h = chain % H;
  const Ctx cx{smem, &m, status, chain};
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {
    if (tid == 0) record_status(status, KDA_ERR_UNSUPPORTED, 2, chain, -1);
    return;
  }

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
    mbar_init(&m.bar_gp, 1); mbar_init(&m.bar_wu, 1); mbar_init(&m.bar_m1, 1);
    mbar_init(&m.bar_m2, 1); mbar_init(&m.bar_fin, 1);
    fence_mbarrier_init();
    m.abort = 0;
    for (int i = 0; i < 3; ++i) m.tma_issued[i] = m.tma_waited[i] = 0;
  }
  if (warp == 0) {
    tmem_alloc(&m.tmem_base, TM_COLS);
    tmem_relinquish();
  }
  // P and T' blocks above the diagonal are never written: zero both tiles once.
  for (int e = tid; e < 2 * 8192 / 16; e += kThreads) st_shared_v4(sb + SM_PMAT + 16 * e, 0, 0, 0, 0);
  if (tid < C) m.beta[0][tid] = (n_chunks > 0 && tid < len) ? beta[(t0 + tid) * H + h] : 0.f;
  cta_sync();
  const uint32_t tm = m.tmem_base;
  const int q4 = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half
  const uint32_t lane_base = 32u * q4;

  // TMA loads of chunk `ci` (thread 0 only).
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

  // ---- initial state -> S^T in TMEM (thread: lane n, 64 key columns of its half); O^T = 0
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
    uint32_t z[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) z[j] = 0u;
    tmem_st32(tmem_addr(tm, lane_base, TM_O + 32 * hf), z);
    tmem_st_wait();
  }
  cta_sync();

  // Writes the output rows of a finished chunk (warps 4-7 only): O^T (TMEM) ->
  // bf16 staging in the q tile (free between the operand build and the next q
  // load) -> coalesced 16-byte stores; clears O^T for the next chunk.
  auto flush_output = [&](int64_t otb, int onv) {
    __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(smem + SM_Q);
    const int n = lane_base + lane;
    uint32_t z[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) z[j] = 0u;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      uint32_t r[32];
      tmem_ld32(tmem_addr(tm, lane_base, TM_O + 32 * part), r);
      tmem_ld_wait(r);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        stg[(32 * part + j) * D + n] = __float2bfloat16_rn(__uint_as_float(r[j]));
      tmem_st32(tmem_addr(tm, lane_base, TM_O + 32 * part), z);
    }
    tmem_st_wait();
    named_sync(2, 128);
    const uint4 *s4 = reinterpret_cast<const uint4 *>(smem + SM_Q);
    const int t = tid - 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = t + 128 * j;  // 16-byte chunk: row e / 16, column chunk e % 16
      const int rr = e >> 4;
      if (rr < onv) {
        uint4 *dst = reinterpret_cast<uint4 *>(out + ((otb + rr) * H + h) * D) + (e & 15);
        *dst = s4[e];
      }
    }
  };

  // Tile-local prefix of the log2-decay of chunk `ci` into registers; thread
  // (tile ta, channel pair cp) owns rows 16 ta .. 16 ta + 15 of channels cc, cc+1.
  const int ta = tid >> 6, cp = tid & 63, cc = 2 * cp;
  const uint32_t hsel = (uint32_t)(cc >> 6), cb = (uint32_t)(cc & 63) * 2u;
  uint32_t swzk[8];   // swizzled byte offset of channel pair cc in a row with row % 8 == k
#pragma unroll
  for (int k = 0; k < 8; ++k) swzk[k] = ((((cb >> 4) ^ (uint32_t)k) << 4) | (cb & 15u));
  float L0[16], L1[16];
  float beta_next = 0.f;
  auto scan = [&](int ci) -> bool {
    const uint32_t par = (uint32_t)(ci & 1);
    const int64_t tb = t0 + (int64_t)C * ci;
    const int nv = (int)((len - (int64_t)C * ci) < C ? (len - (int64_t)C * ci) : C);
    const bool ok_la = wait_bar(cx, &m.bar_la, par, 11, ci);
    if (ci + 1 < n_chunks && tid < C) {   // prefetch the following chunk's beta
      const int64_t len_next = len - (int64_t)C * (ci + 1);
      beta_next = tid < len_next ? beta[(tb + C + tid) * H + h] : 0.f;
    }
    const float2 *la = reinterpret_cast<const float2 *>(smem + SM_LA);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int row = 16 * ta + j;
      float2 x = la[row * (D / 2) + cp];
      if (row >= nv) x = make_float2(0.f, 0.f);
      s0 = fmaf(x.x, kLog2e, s0);
      s1 = fmaf(x.y, kLog2e, s1);
      L0[j] = s0;
      L1[j] = s1;
    }
    *reinterpret_cast<float2 *>(&m.tot[ta][cc]) = make_float2(s0, s1);
    if (tid == 0 && ok_la) m.tma_waited[TMA_LA]++;
    return ok_la;
  };

  bool failed = false;
  int64_t prev_tb = 0;
  int prev_nv = 0;
  if (n_chunks > 0) scan(0);
  for (int ci = 0; ci < n_chunks && !failed; ++ci) {
    const uint32_t par = (uint32_t)(ci & 1);
    const int64_t tb = t0 + (int64_t)C * ci;
    const int nv = (int)((len - (int64_t)C * ci) < C ? (len - (int64_t)C * ci) : C);
    const bool has_next = ci + 1 < n_chunks;
    const float *bcur = m.beta[ci & 1];
    PHASE_MARK(0);
    if (ci > 0) {   // Kdec / P of the previous chunk consumed, its state final
      wait_bar(cx, &m.bar_m2, par ^ 1u, 25, ci - 1);
      tc_fence_after();
    }
    cta_sync();     // tile totals of this chunk visible
    PHASE_MARK(1);
    if (m.abort) { failed = true; break; }
    if (tid == 0 && ci == 0 && n_chunks > 1) issue_la(1);   // log_alpha tile scanned

    // ================= phase 2: every operand tile of the chunk in one pass
    {
      const bool ok_qk = wait_bar(cx, &m.bar_qk, par, 10, ci);
      if (tid == 0 && ok_qk) m.tma_waited[TMA_QK]++;
      float st0[4], st1[4], rf0[4], rf1[4];   // tile starts / ends, channels c, c+1
      {
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const float2 t = *reinterpret_cast<const float2 *>(&m.tot[b][cc]);
          st0[b] = acc0; st1[b] = acc1;
          acc0 += t.x; acc1 += t.y;
          rf0[b] = acc0; rf1[b] = acc1;
        }
      }
      const float sa0 = ta == 0 ? st0[0] : ta == 1 ? st0[1] : ta == 2 ? st0[2] : st0[3];
      const float sa1 = ta == 0 ? st1[0] : ta == 1 ? st1[1] : ta == 2 ? st1[2] : st1[3];
      const float ra0 = ta == 0 ? rf0[0] : ta == 1 ? rf0[1] : ta == 2 ? rf0[2] : rf0[3];
      const float ra1 = ta == 0 ? rf1[0] : ta == 1 ? rf1[1] : ta == 2 ? rf1[2] : rf1[3];
      const float tot0 = ra0 - sa0, tot1 = ra1 - sa1;
      // column-block factors F[a2][ta] = 2^{st_a2 - ref_ta}, a2 = ta..3
      float fb0[4], fb1[4];
#pragma unroll
      for (int a2 = 0; a2 < 4; ++a2) {
        fb0[a2] = ex2(st0[a2] - ra0);
        fb1[a2] = ex2(st1[a2] - ra1);
      }
      const float fs0 = ex2(sa0), fs1 = ex2(sa1);                 // e^{st_a}
      const float fd0 = ex2(rf0[3] - ra0), fd1 = ex2(rf1[3] - ra1);  // e^{g_C - ref_a}
      if (ta == 0) {
        m.gamma[cc] = ex2(rf0[3]);
        m.gamma[cc + 1] = ex2(rf1[3]);
      }
      // Row-tile bases (column half of cc, first row of tile ta); element (row
      // 16 ta + j) sits j * 128 + swzk[j & 7] bytes further (128-byte swizzle).
      const uint32_t r0 = 16u * ta * 128u, h64 = hsel * 8192u, h128 = hsel * 16384u;
      const uint32_t bK = sb + SM_K + h64 + r0, bQ = sb + SM_Q + h64 + r0;
      const uint32_t bGA = sb + SM_GA + h128 + r0, bST = sb + SM_STACK + h128 + r0;
      const uint32_t bKD = sb + SM_KDEC + h64 + r0;
      const uint32_t bGB = sb + SM_GB + hsel * (GB_ROWS * 128u) + r0;
      uint32_t kraw[16], qraw[16];   // all k, q pairs of this thread, loaded up front
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        kraw[j] = ld_shared_b32(bK + (uint32_t)j * 128u + swzk[j & 7]);
        qraw[j] = ld_shared_b32(bQ + (uint32_t)j * 128u + swzk[j & 7]);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t o = (uint32_t)j * 128u + swzk[j & 7];
        const float2 kk = unpack_bf16x2(kraw[j]);
        const float2 qq = unpack_bf16x2(qraw[j]);
        const float e0 = ex2(L0[j]), e1 = ex2(L1[j]);                    // e^{g_r - st_a}
        const float ec0 = ex2(tot0 - L0[j]), ec1 = ex2(tot1 - L1[j]);    // e^{ref_a - g_r}
        st_shared_b32(bGA + o, pack_bf16x2(kk.x * e0, kk.y * e1));
        st_shared_b32(bGA + 8192u + o, pack_bf16x2(qq.x * e0, qq.y * e1));
        const float kc0 = kk.x * ec0, kc1 = kk.y * ec1;
#pragma unroll
        for (int a2 = 0; a2 < 4; ++a2) {   // block (a2, ta) of the column operand, row j
          if (a2 < ta) continue;
          st_shared_b32(bGB + 16u * blk(a2, 0) * 128u + o,
                        pack_bf16x2(kc0 * fb0[a2], kc1 * fb1[a2]));
        }
        const float g0 = e0 * fs0, g1 = e1 * fs1;                        // e^{g_r}
        st_shared_b32(bST + o, pack_bf16x2(qq.x * g0, qq.y * g1));
        st_shared_b32(bST + 8192u + o, pack_bf16x2(kk.x * g0, kk.y * g1));
        st_shared_b32(bKD + o, pack_bf16x2(kc0 * fd0, kc1 * fd1));
      }
    }
    fence_proxy_async_smem();
    if (tid < C && has_next) m.beta[(ci + 1) & 1][tid] = beta_next;
    cta_sync();
    PHASE_MARK(2);
    if (m.abort) { failed = true; break; }
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t ad = kdesc(smem + SM_GA, (ks >> 2) * 16384u + (ks & 3) * 32u);
        const uint64_t bd = kdesc(smem + SM_GB, (ks >> 2) * (GB_ROWS * 128u) + (ks & 3) * 32u);
        umma_ss(tm + TM_GP, ad, bd, ID_GP, ks > 0 ? 1u : 0u);
      }
      umma_commit(&m.bar_gp);
    }

    // ================= phase 3 (while the Gram MMAs run): S pass, previous output
    {
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int c0 = 64 * hf + 32 * part;
        uint32_t s[32];
        tmem_ld32(tmem_addr(tm, lane_base, TM_S + c0), s);
        tmem_ld_wait(s);
        uint32_t ab[16];
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          float gv[8];
          ld8(gv, &m.gamma[c0 + 8 * q8]);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = 8 * q8 + 2 * jj;
            const float f0 = __uint_as_float(s[j]), f1 = __uint_as_float(s[j + 1]);
            ab[4 * q8 + jj] = pack_bf16x2(f0, f1);
            s[j] = __float_as_uint(f0 * gv[2 * jj]);
            s[j + 1] = __float_as_uint(f1 * gv[2 * jj + 1]);
          }
        }
        tmem_st32(tmem_addr(tm, lane_base, TM_S + c0), s);
        tmem_st16(tmem_addr(tm, lane_base, TM_AS + c0 / 2), ab);
      }
      tmem_st_wait();
    }
    // ================= phase 4: A^T (fp32, for the solve) and P (bf16, K-major [r][i])
    wait_bar(cx, &m.bar_gp, par, 22, ci);
    tc_fence_after();
    PHASE_MARK(3);
    {
      // Quadrant rows: 32 (q4 & 1) + lane; block columns of tiles {0,1} are [0, 48),
      // of tiles {2,3} are [48, 160); the two warps of a quadrant split them.
      const int row = 32 * (q4 & 1) + lane;
      const int rta = row >> 4;
      const bool gram = q4 < 2;
      const float br = bcur[row];
      float *amatT = reinterpret_cast<float *>(smem + SM_GA);
      const int nld = (q4 & 1) ? 2 : 1;
      const int col_first = (q4 & 1) ? 32 + 64 * hf : 32 * hf;
      for (int li = 0; li < nld; ++li) {
        const int col0 = col_first + 32 * li;
        uint32_t v[32];
        tmem_ld32(tmem_addr(tm, lane_base, TM_GP + col0), v);
        tmem_ld_wait(v);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int bk = (col0 >> 4) + half;    // block index of these 16 columns
          const int ba = bk >= 6 ? 3 : bk >= 3 ? 2 : bk >= 1 ? 1 : 0;
          const int bb = bk - ba * (ba + 1) / 2;
          if (ba != rta) continue;
          if (gram) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int i = 16 * bb + jj;
              amatT[i * FP + row] = i < row ? br * __uint_as_float(v[16 * half + jj]) : 0.f;
            }
          } else {
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
              uint32_t w[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int j = 8 * g8 + 2 * t, i = 16 * bb + j;
                const float lo = i <= row ? __uint_as_float(v[16 * half + j]) : 0.f;
                const float hi = i + 1 <= row ? __uint_as_float(v[16 * half + j + 1]) : 0.f;
                w[t] = pack_bf16x2(lo, hi);
              }
              st_shared_v4(sb + SM_PMAT + sw128_offset(row, (16 * bb + 8 * g8) * 2), w[0], w[1],
                           w[2], w[3]);
            }
          }
        }
      }
    }
    fence_proxy_async_smem();
    cta_sync();
    PHASE_MARK(4);
    if (m.abort) { failed = true; break; }

    // ================= phase 5: T = (I + A)^{-1} (warps 0-3) while warps 4-7 write
    // the previous chunk's output.
    const float *amatT = reinterpret_cast<const float *>(smem + SM_GA);   // A^T, [i][r]
    float *tinv = reinterpret_cast<float *>(smem + SM_GB + OFF_TINV);     // T, [r][i]
    if (warp < 4) {
      float *xbuf = reinterpret_cast<float *>(smem + SM_GB + OFF_XBUF);
      if (warp < 2) {
        // Diagonal blocks by column-oriented forward substitution: lane owns
        // column j of block a; after step m, t[m] is final and is eliminated
        // from every later row.
        const int a = 2 * warp + (lane >> 4), j = lane & 15, b0 = 16 * a;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) t[r] = (r == j) ? 1.f : 0.f;
        float col[16], nxt[16];   // column mc of the block, and the next one in flight
        ld8(*reinterpret_cast<float(*)[8]>(col), amatT + b0 * FP + b0);
        ld8(*reinterpret_cast<float(*)[8]>(col + 8), amatT + b0 * FP + b0 + 8);
#pragma unroll
        for (int mc = 0; mc < 15; ++mc) {
          if (mc + 1 < 15) {
            ld8(*reinterpret_cast<float(*)[8]>(nxt), amatT + (b0 + mc + 1) * FP + b0);
            ld8(*reinterpret_cast<float(*)[8]>(nxt + 8), amatT + (b0 + mc + 1) * FP + b0 + 8);
          }
          const float tmv = t[mc];
#pragma unroll
          for (int r = mc + 1; r < 16; ++r) t[r] = fmaf(-col[r], tmv, t[r]);
#pragma unroll
          for (int r = 0; r < 16; ++r) col[r] = nxt[r];
        }
        // T (fp32, for the block recursion) and T' = T Diag(beta) (bf16 MMA operand;
        // the block's upper triangle is zero because t[r] = 0 for r < j).
        const float bj = bcur[b0 + j];
        __nv_bfloat16 *tp = reinterpret_cast<__nv_bfloat16 *>(smem + SM_TMAT);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          tinv[(b0 + r) * FP + b0 + j] = t[r];
          tp[sw128_offset(b0 + r, (b0 + j) * 2) >> 1] = __float2bfloat16_rn(t[r] * bj);
        }
      }
      named_sync(1, 128);
      // Off-diagonal blocks, block-recursive: 16 -> 32 (blocks (1,0), (3,2)), then
      // 32 -> 64 (blocks (2,0), (2,1), (3,0), (3,1)), TF32 warp MMAs.
      const int g = lane >> 2, t4 = lane & 3;
      // acc (+)= A_{ab} T_{mb} with A from A^T (column-major, pitch FP) ...
      auto mul_AT = [&](float (&acc)[2][4], int ab, int mb, int tcol) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int kc = 16 * mb + 8 * kk;
          const uint32_t a0 = to_tf32(amatT[(kc + t4) * FP + 16 * ab + g]);
          const uint32_t a1 = to_tf32(amatT[(kc + t4) * FP + 16 * ab + g + 8]);
          const uint32_t a2 = to_tf32(amatT[(kc + t4 + 4) * FP + 16 * ab + g]);
          const uint32_t a3 = to_tf32(amatT[(kc + t4 + 4) * FP + 16 * ab + g + 8]);
          const float *b0p = tinv + (kc + t4) * FP + tcol + g;
          const float *b1p = tinv + (kc + t4 + 4) * FP + tcol + g;
          mma_tf32_16x8x8(acc[0], a0, a1, a2, a3, to_tf32(b0p[0]), to_tf32(b1p[0]));
          mma_tf32_16x8x8(acc[1], a0, a1, a2, a3, to_tf32(b0p[8]), to_tf32(b1p[8]));
        }
      };
      // ... and acc (+)= T_{ar} X with T row-major (pitch FP), X a 16 x 16 block (pitch XP).
      auto mul_TX = [&](float (&acc)[2][4], int ar, int ac, const float *x) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const float *tp = tinv + (16 * ar) * FP + 16 * ac + 8 * kk;
          const uint32_t a0 = to_tf32(tp[g * FP + t4]);
          const uint32_t a1 = to_tf32(tp[(g + 8) * FP + t4]);
          const uint32_t a2 = to_tf32(tp[g * FP + t4 + 4]);
          const uint32_t a3 = to_tf32(tp[(g + 8) * FP + t4 + 4]);
          const float *x0 = x + (8 * kk + t4) * XP + g;
          const float *x1 = x + (8 * kk + t4 + 4) * XP + g;
          mma_tf32_16x8x8(acc[0], a0, a1, a2, a3, to_tf32(x0[0]), to_tf32(x1[0]));
          mma_tf32_16x8x8(acc[1], a0, a1, a2, a3, to_tf32(x0[8]), to_tf32(x1[8]));
        }
      };
      auto store_blk = [&](float *dst, int pitch, const float (&acc)[2][4], float sgn) {
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
          dst[g * pitch + 8 * nh + 2 * t4] = sgn * acc[nh][0];
          dst[g * pitch + 8 * nh + 2 * t4 + 1] = sgn * acc[nh][1];
          dst[(g + 8) * pitch + 8 * nh + 2 * t4] = sgn * acc[nh][2];
          dst[(g + 8) * pitch + 8 * nh + 2 * t4 + 1] = sgn * acc[nh][3];
        }
      };
      // Final block T_ab: fp32 into T, and T' = T Diag(beta) as bf16 pairs.
      auto store_T = [&](int ab, int bb, const float (&acc)[2][4]) {
        store_blk(tinv + (16 * ab) * FP + 16 * bb, FP, acc, -1.f);
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
          const int col = 16 * bb + 8 * nh + 2 * t4;
          const float b0v = bcur[col], b1v = bcur[col + 1];
          const uint32_t lo = pack_bf16x2(-acc[nh][0] * b0v, -acc[nh][1] * b1v);
          const uint32_t hi = pack_bf16x2(-acc[nh][2] * b0v, -acc[nh][3] * b1v);
          *reinterpret_cast<uint32_t *>(smem + SM_TMAT + sw128_offset(16 * ab + g, col * 2)) = lo;
          *reinterpret_cast<uint32_t *>(smem + SM_TMAT + sw128_offset(16 * ab + g + 8, col * 2)) = hi;
        }
      };
      float *xw = xbuf + warp * 16 * XP;
      if (warp < 2) {   // level 16 -> 32: block (1,0) on warp 0, (3,2) on warp 1
        const int ab = 2 * warp + 1, bb = 2 * warp;
        float acc[2][4] = {};
        mul_AT(acc, ab, bb, 16 * bb);                 // X = A_ab T_bb
        store_blk(xw, XP, acc, 1.f);
        __syncwarp();
        float o[2][4] = {};
        mul_TX(o, ab, ab, xw);                        // T_ab = -T_aa X
        store_T(ab, bb, o);
      }
      named_sync(1, 128);
      {                 // level 32 -> 64: warp w -> block (2 + w/2, w%2)
        const int ab = 2 + (warp >> 1), bb = warp & 1;
        float acc[2][4] = {};
        // X_{ab} = A_{ab,0:2} T_{0:2, bb} = sum_{m=bb}^{1} A_{ab,m} T_{m,bb}
        for (int mb = bb; mb < 2; ++mb) mul_AT(acc, ab, mb, 16 * bb);
        store_blk(xw, XP, acc, 1.f);
        named_sync(1, 128);
        // T_{ab} = -sum_{k=2}^{ab} T_{ab,k} X_{k,bb}
        float o[2][4] = {};
        for (int k = 2; k <= ab; ++k) mul_TX(o, ab, k, xbuf + (2 * (k - 2) + bb) * 16 * XP);
        store_T(ab, bb, o);
      }
      fence_proxy_async_smem();   // T' is an MMA operand
    } else {
      if (ci > 0) flush_output(prev_tb, prev_nv);
      named_sync(2, 128);   // output staging (q tile) read by warps 4-7
      if (tid == 128 && has_next) issue_qk(ci + 1);
    }
    __syncthreads();
    PHASE_MARK(5);

    fence_proxy_async_smem();
    cta_sync();
    PHASE_MARK(6);
    if (tid == 0) {
      if (wait_bar(cx, &m.bar_v, par, 12, ci)) {
        m.tma_waited[TMA_V]++;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {   // U^T = V^T T'^T ; W^T = Kt^T T'^T, interleaved
          const uint64_t bd = kdesc(smem + SM_TMAT, ks * 32u);
          umma_ss(tm + TM_U, mndesc(smem + SM_V, ks * 2048u, 8192), bd, ID_UW, ks > 0);
          umma_ss(tm + TM_W, mndesc(smem + SM_STACK, 64u * 128u + ks * 2048u, 16384), bd, ID_UW,
                  ks > 0);
        }
        umma_commit(&m.bar_wu);
      }
    }

    // ================= phase 6: -W -> stack rows 64.. (K-major); [O^T | D^T] = S^T [Qt; -W]^T
    wait_bar(cx, &m.bar_wu, par, 23, ci);
    tc_fence_after();
    PHASE_MARK(7);
    if (tid == 128 && has_next) issue_v(ci + 1);
    {
      uint32_t r[32];
      tmem_ld32(tmem_addr(tm, lane_base, TM_W + 32 * hf), r);
      tmem_ld_wait(r);
      const int c = lane_base + lane;   // key channel of this lane; W^T columns are rows r
      const uint32_t cbyte = (uint32_t)(c & 63) * 2u;
      const uint32_t base = sb + SM_STACK + (uint32_t)(c >> 6) * 16384u + (64u + 32u * hf) * 128u;
      uint32_t sw[8];   // swizzled byte offset of channel c in a row with row % 8 == k
#pragma unroll
      for (int k = 0; k < 8; ++k) sw[k] = ((((cbyte >> 4) ^ (uint32_t)k) << 4) | (cbyte & 15u));
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const __nv_bfloat16 w = __float2bfloat16_rn(-__uint_as_float(r[j]));
        st_shared_b16(base + (uint32_t)j * 128u + sw[j & 7], *reinterpret_cast<const uint16_t *>(&w));
      }
      fence_proxy_async_smem();
    }
    cta_sync();
    PHASE_MARK(8);
    if (m.abort) { failed = true; break; }
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_ts(tm + TM_O, tm + TM_AS + 8 * ks,
                kdesc(smem + SM_STACK, (ks >> 2) * 16384u + (ks & 3) * 32u), ID_OM1, 1u);
      umma_commit(&m.bar_m1);
    }
    // next chunk's decay prefix while the MMAs run
    if (has_next) scan(ci + 1);
    PHASE_MARK(9);

    // ================= phase 7: bf16 Delta^T; S^T += Delta^T Kdec; O^T += Delta^T P^T
    wait_bar(cx, &m.bar_m1, par, 24, ci);
    tc_fence_after();
    PHASE_MARK(10);
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
    PHASE_MARK(11);
    if (m.abort) { failed = true; break; }
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        umma_ts(tm + TM_S, tm + TM_AD + 8 * ks, mndesc(smem + SM_KDEC, ks * 2048u, 8192),
                ID_KM128, 1u);
        umma_ts(tm + TM_O, tm + TM_AD + 8 * ks, kdesc(smem + SM_PMAT, ks * 32u), ID_KK64, 1u);
      }
      umma_commit(&m.bar_m2);
      if (ci + 2 < n_chunks) issue_la(ci + 2);   // the next chunk's tile was scanned above
    }
    prev_tb = tb;
    prev_nv = nv;
  }

  // ---- the last chunk's output and the final state
  if (!failed && n_chunks > 0) {
    wait_bar(cx, &m.bar_m2, (uint32_t)((n_chunks - 1) & 1), 26, n_chunks - 1);
    tc_fence_after();
    if (warp >= 4) flush_output(prev_tb, prev_nv);
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
        for (int j = 0; j < 32; ++j)
          final_state[sbase + (int64_t)(c0 + j) * D + n] = __uint_as_float(r[j]);
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

#ifdef KDA_PHASE_PROFILE
extern "C" int kda_debug_phase_clock(long long *host, int n) {
  return cudaMemcpyFromSymbol(host, g_phase_clock, sizeof(long long) * n) == cudaSuccess ? 0 : 4;
}
#endif

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
