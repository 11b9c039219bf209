// bf16 chunkwise KDA prefill on the 5th-generation tensor cores (tcgen05).
//
// One CTA carries one (sequence, head) chain through chunks of C = 64 tokens.
// Eight compute warps do the CUDA-core work; a ninth warp issues every TMA load
// and every tcgen05.mma, so no compute warp ever blocks on an MMA issue.  The
// fp32 state lives in tensor memory for the whole chain; every dense
// contraction of a chunk is a tcgen05.mma (bf16 operands, fp32 accumulators).
//
// Chunk algebra ("Kimi K3: 架构、训练与系统全景解析", section 4.2.4: state passed
// between chunks, lower-triangular matrix work inside, output = pre-chunk-state
// term + intra-chunk causal term; UT-transform form of the solve), with g_r the
// within-chunk cumulative log-decay per key channel and S the incoming state:
//   A = strict_lower(Diag(beta) [k_r . k_i e^{g_r - g_i}]),  T = (I + A)^{-1}
//   T' = T Diag(beta),  Kt = K o e^{g},  Qt = Q o e^{g},  Y = Kt S
//   Delta = T' (V - Y),  O = Qt S + P Delta,  P = lower_incl([q_r . k_i e^{g_r - g_i}])
//   S <- Diag(e^{g_C}) S + (K o e^{g_C - g})^T Delta
// (Delta = T'V - T'Kt S is the usual U - W S with U = T'V and W = T'Kt, taken
// in the other association so that W never has to be formed.)
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
//   O^T = S^T Qt^T,  Y^T = S^T Kt^T      (A = bf16 S^T in TMEM)
//   Delta^T = (V - Y)^T T'^T              (A = bf16 (V - Y)^T in TMEM)
//   S^T += Delta^T Kdec,  O^T += Delta^T P^T   (A = bf16 Delta^T in TMEM),
//                                    after S^T <- S^T Diag(e^{g_C})
// The products with the lower-triangular T' and P skip the zero blocks: K step
// s only touches output columns r >= 16 s.
//
// Pipeline.  O^T is double-buffered in TMEM and Kdec in shared memory, so the
// next chunk's operand build overlaps this chunk's state MMAs, and the triangular
// solve (warps 0-3) overlaps the previous chunk's output stores, the O+Y MMAs and
// the (V - Y) pass (warps 4-7).  The build writes the Gram operands first, so the
// Gram MMAs of chunk c+1 run under the rest of its build.
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
constexpr int kComputeWarps = 8;                   // warpgroups 0 and 1
constexpr int kMmaWarp = kComputeWarps;            // warp 8: TMA + MMA issue (warps 9-11 idle)
constexpr int kThreads = 32 * (kComputeWarps + 4);  // 384: three whole warpgroups
// Register split (setmaxnreg): the launch gives every thread 65536 / 384 = 168;
// the issue warpgroup returns most of its share to the compute warpgroups.
constexpr uint32_t kLaunchRegs = 168, kComputeRegs = 208, kIssueRegs = 88;
static_assert(256 * kComputeRegs + 128 * kIssueRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on any single wait: 2 s
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory map (byte offsets from a 1024-byte aligned base).  Operand
// tiles use 128-byte rows with the 128-byte swizzle; a "K-major tile of R rows"
// stores columns 0-63 as R rows of 128 B, then columns 64-127 likewise.
constexpr uint32_t SM_Q = 0;                    // q chunk (TMA), 64 rows
constexpr uint32_t SM_K = SM_Q + 16384;         // k chunk (TMA), 64 rows
constexpr uint32_t SM_V = SM_K + 16384;         // v chunk (TMA), [64 r][128 n] bf16, unswizzled
constexpr uint32_t SM_LA = SM_V + 16384;        // log_alpha fp32 [64][128]; then tile totals
constexpr uint32_t SM_GA = SM_LA + 32768;       // Gram rows, 128 rows; then A fp32
constexpr uint32_t SM_GB = SM_GA + 32768;       // Gram columns, 160 rows; then T, X, T'
constexpr uint32_t SM_STACK = SM_GB + 40960;    // [Qt; Kt], 128 rows
constexpr uint32_t SM_KDEC = SM_STACK + 32768;  // 2 x (K o e^{g_C - g}), 64 rows (MN-major)
constexpr uint32_t SM_PMAT = SM_KDEC + 32768;   // P, K-major [64 r][64 i]
constexpr uint32_t SM_MISC = SM_PMAT + 8192;

constexpr uint32_t GB_ROWS = 160;
constexpr int FP = 72;  // pitch (floats) of the fp32 64 x 64 T of the solve
constexpr int FA = 68;  // pitch (floats) of A: rows 16 B aligned, 4-word bank steps
constexpr int XP = 24;  // pitch (floats) of the 16 x 16 intermediate blocks
constexpr uint32_t OFF_TINV = 0;                     // inside SM_GB, after the Gram MMAs
constexpr uint32_t OFF_XBUF = 64 * FP * 4;           // 4 blocks of 16 x XP fp32
constexpr uint32_t OFF_TMAT = OFF_XBUF + 4 * 16 * XP * 4;  // T' = T Diag(beta), K-major
constexpr uint32_t SM_TMAT = SM_GB + OFF_TMAT;

// A chunk a helper CTA has claimed (written by its issue thread).
struct HelpClaim {
  int32_t valid, chain, chunk, tb, nv, head;
};

struct Misc {
  float beta[2][C];  // beta of the chunk in flight and of the next one
  float gamma[D];    // Gamma_C = e^{g_C} per key channel
  uint64_t bar_qk, bar_la, bar_v;                     // TMA arrivals
  uint64_t bar_gp, bar_m1, bar_u, bar_m2, bar_fin;    // MMA completions
  uint64_t bar_gops;            // Gram operands of the chunk built (one arrival per warp)
  uint64_t bar_build, bar_om, bar_t1, bar_t, bar_ny, bar_ad;  // operands ready (one arrival per warp)
  uint64_t bar_plan;            // the issue thread has planned the next chunk
  uint64_t bar_pka, bar_pkb;    // package copies: [Gamma, Qt; Kt, Kdec] and [T', P]
  uint64_t bar_wb;              // helper: the package has been read out of shared memory
  uint32_t tmem_base;
  int abort;
  int test_chunk;               // chunk whose Gram-operand arrival a test withholds (-1: none)
  uint64_t wait_ns;             // bound on any single wait of this CTA
  int32_t plan[2];              // chain CTA: 1 if that chunk's package comes from a helper
  HelpClaim claim[2];           // helper CTA: the chunk being built / the next one
  // Per copy barrier (TMA_*): phase index + 1 of the last phase that carried a
  // real copy (0: none), so an aborting CTA can wait for it before exiting.
  uint32_t last_copy[5];
  // Last, so that the fields before keep their offsets: inserted among the
  // barriers above it slowed the plain schedule by 2 % (layout only).
  uint64_t bar_stg;             // chain with helpers: the staged output rows have been read
};
constexpr uint32_t SMEM_BYTES = SM_MISC + sizeof(Misc);
constexpr uint32_t SM_BETA = SM_MISC + offsetof(Misc, beta);
constexpr uint32_t SM_GAMMA = SM_MISC + offsetof(Misc, gamma);
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(64 * FA * 4 <= 32768, "A fits SM_GA");
static_assert(OFF_TMAT % 1024 == 0 && OFF_TMAT + 8192 <= 40960, "T, X and T' fit SM_GB");

// TMEM columns (fp32 cells).
constexpr uint32_t TM_S = 0;     // S^T, 128 columns
constexpr uint32_t TM_AS = 128;  // bf16 S^T (A operand), 64 columns
constexpr uint32_t TM_O = 192;   // O^T, 2 x 64 columns (chunk parity)
constexpr uint32_t TM_GP = 320;  // [Gram; P] rows x 160 block columns, then:
constexpr uint32_t TM_Y = TM_GP;        //   Y^T fp32, 64 columns
constexpr uint32_t TM_NY = TM_GP + 64;  //   bf16 (V - Y)^T (A operand), 32 columns
constexpr uint32_t TM_AD = TM_GP + 64;  //   bf16 Delta^T (A operand), after (V - Y)^T is consumed
constexpr uint32_t TM_D = TM_GP + 96;   //   Delta^T fp32, 64 columns
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_GP = idesc_bf16(128, GB_ROWS, false, false);
constexpr uint32_t ID_N64 = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_KM128 = idesc_bf16(128, 128, false, true);
constexpr uint32_t ID_N32 = idesc_bf16(128, 32, false, false);
constexpr uint32_t ID_N16 = idesc_bf16(128, 16, false, false);
// Triangle-trimmed products: K step s writes output columns 16 s .. 63.
__host__ __device__ constexpr uint32_t id_tri(int s, bool a_mn) {
  return idesc_bf16(128, 64 - 16 * s, a_mn, false);
}

enum { TMA_QK = 0, TMA_LA = 1, TMA_V = 2, TMA_PKA = 3, TMA_PKB = 4 };

// Package layout (byte offsets in a helper ring slot): shared-memory images.
constexpr uint32_t PKG_STACK = 0, PKG_KDEC = 32768, PKG_TMAT = 49152, PKG_PMAT = 57344,
                   PKG_GAMMA = 65536;
static_assert(PKG_GAMMA + 512 == kHelpPackageBytes, "package layout");
constexpr int kHelpMaxSeqs = 16384 / 8;  // sequence table of a helper (in its v buffer)
constexpr uint64_t kHelpIdleNs = 200000000ull;  // a helper with nothing to claim for 0.2 s stops

// Optional per-phase cycle stamps of chain 0 (profiling builds only), 64 slots
// per chunk: thread 0 uses slots 0-15, thread 128 slots 16-23, the MMA thread
// slots 24-31, thread 96 (warp 3) slots 32-39, thread 224 (warp 7) slots 40-47.
#ifdef KDA_PHASE_PROFILE
__device__ long long g_phase_clock[4096 * 64];
#define PHASE_STAMP(t, i)                                                                \
  do {                                                                                   \
    if (tid == (t) && chain == 0 && ci < 4096) g_phase_clock[ci * 64 + (i)] = clock64(); \
  } while (0)
// Records a value (not a clock) in slot i of chain 0's chunk.
#define PHASE_VALUE(t, i, v)                                                       \
  do {                                                                             \
    if (tid == (t) && chain == 0 && ci < 4096) g_phase_clock[ci * 64 + (i)] = (v); \
  } while (0)
#else
#define PHASE_STAMP(t, i) \
  do {                    \
  } while (0)
#define PHASE_VALUE(t, i, v) \
  do {                       \
  } while (0)
#endif
#define PHASE_MARK(i) PHASE_STAMP(0, i)
#define PHASE_MARK_W4(i) PHASE_STAMP(128, 16 + (i))
#define PHASE_MARK_MMA(i) PHASE_STAMP(32 * kMmaWarp, 24 + (i))
#define PHASE_MARK_W3(i) PHASE_STAMP(96, 32 + (i))
#define PHASE_MARK_W7(i) PHASE_STAMP(224, 40 + (i))

// CTA-wide barrier of all 288 threads, ordered with the tcgen05 operations.
__device__ __forceinline__ void cta_sync() {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// Compute-warp barrier that also decides, identically for all 256 threads,
// whether the CTA is aborting: each thread contributes the flag as it read it
// and every thread receives the OR.  (The issue thread may raise the flag at any
// moment, so a plain read after the barrier could differ between threads.)
__device__ __forceinline__ bool compute_sync_abort(const int *abort_flag) {
  const uint32_t mine = *reinterpret_cast<const volatile int *>(abort_flag) != 0 ? 1u : 0u;
  uint32_t any;
  tc_fence_before();
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(any)
      : "r"(mine), "n"(32 * kComputeWarps)
      : "memory");
  tc_fence_after();
  return any != 0;
}

// One arrival per warp on an "operands ready" barrier: every lane has already
// fenced its own shared-memory / TMEM writes; the warp barrier orders them
// before lane 0's release-arrive.
__device__ __forceinline__ void warp_arrive(uint64_t *bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
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

// Bounded mbarrier wait (kWaitNs, or a test's shorter bound); on timeout records
// KDA_ERR_TIMEOUT and raises the abort flag.  Compute warps test the flag only
// through compute_sync_abort, so they all leave the chunk loop at the same point;
// the MMA thread leaves its loop at the failed wait.
__device__ bool wait_bar(const Ctx &x, uint64_t *bar, uint32_t parity, int where, int chunk,
                         bool poll = false) {
  const uint64_t limit = *reinterpret_cast<const volatile uint64_t *>(&x.m->wait_ns);
  if (poll ? mbar_wait_poll(bar, parity, limit) : mbar_wait(bar, parity, limit)) return true;
  record_status(x.status, KDA_ERR_TIMEOUT, where, x.chain, chunk);
  atomicExch(&x.m->abort, 1);
  return false;
}

// 8 consecutive fp32 from a 16-byte aligned shared address.
__device__ __forceinline__ void lds8(float (&v)[8], uint32_t saddr) {
  const float4 a = ld_shared_f32x4(saddr);
  const float4 b = ld_shared_f32x4(saddr + 16u);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Block column index of tile pair (a, b), a >= b, in the Gram column operand.
__host__ __device__ constexpr int blk(int a, int b) { return a * (a + 1) / 2 + b; }

// Kernel variants.  kModeHelp adds helper CTAs (and the chain CTAs' side of
// their protocol); kModeTransitions is the first pass of the in-device split of
// long sequences: block b < chains runs chain b from a zero state (its
// final state is the segment's B), the block after the chains that carries b runs the same chain
// as a transition (state I, v = 0: its final state is the segment's transition
// matrix M), and neither writes outputs.  Each mode compiles its branches away
// in the others, which keeps the plain path as fast as before (the runtime
// checks alone cost about 10 % on a 96-chain prefill).
constexpr int kModePlain = 0, kModeHelp = 1, kModeTransitions = 2;
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
kda_chunk_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_la,
                        const __grid_constant__ CUtensorMap tm_o, const float *__restrict__ beta,
                        const float *__restrict__ init_state,
                        const int32_t *__restrict__ cu_seqlens, int32_t n_seqs, int64_t n_tokens,
                        int32_t H, __nv_bfloat16 *__restrict__ out,
                        float *__restrict__ final_state, DeviceStatus *status,
                        const HelpRing help, float *__restrict__ final_state_m,
                        const int32_t *__restrict__ seq_order,
                        const __grid_constant__ CUtensorMap tm_om,
                        __nv_bfloat16 *__restrict__ out_m, const int write_out,
                        const int split_k, TestControl *test_control) {
  // Indexing the __shared__ array directly (no integer round trip) keeps every
  // access a shared-memory instruction.  The 128-byte swizzle atoms need a
  // 1024-byte aligned base, checked below.
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc &m = *reinterpret_cast<Misc *>(smem + SM_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // First pass of a split: blocks [0, n_seqs H) are the zero-start runs of the
  // chains, the rest the transition runs, of every chain or, with split_k >= 2,
  // of every chain but those of each sequence's first segment (sequences of
  // split_k segments; a zero initial state needs no M_0).
  const bool transition = kMode == kModeTransitions && (int64_t)blockIdx.x >= (int64_t)n_seqs * H;
  int slot = (int)blockIdx.x;
  if (transition) {
    const int i = (int)(blockIdx.x - n_seqs * H);
    slot = split_k >= 2 ? i + (i / ((split_k - 1) * H) + 1) * H : i;
  }
  // Blocks past the chains are helpers (only when the call has a helper ring).
  const bool helping = kMode == kModeHelp && help.ring != nullptr;
  const bool helper = helping && slot >= help.n_chains;
  // With seq_order, block slots take the sequences longest first (every head of
  // a sequence in turn), so the longest chains do not start last.
  const int seq = (seq_order && !helper) ? seq_order[slot / H] : slot / H, h = slot % H;
  const int chain = helper ? slot : seq * H + h;
  const Ctx cx{smem, &m, status, chain};
  const uint32_t sb = smem_u32(smem);
  // A chain CTA that stops early tells the helpers to leave its chunks alone.
  auto chain_done = [&]() {
    if (helping && !helper && tid == 0) {
      st_relaxed_gpu(help.cons_pos + chain, 0x7fffffff);
      atomicAdd(help.finished, 1);
    }
  };
  if (sb & 1023u) {
    if (tid == 0) record_status(status, KDA_ERR_UNSUPPORTED, 2, chain, -1);
    chain_done();
    return;
  }

  int64_t t0 = 0, len = 0;
  if (!helper) {
    const int64_t a = cu_seqlens[seq], b = cu_seqlens[seq + 1];
    if (a < 0 || b < a || b > n_tokens ||
        (chain == 0 && (cu_seqlens[0] != 0 || cu_seqlens[n_seqs] != n_tokens))) {
      if (tid == 0) record_status(status, KDA_ERR_INVALID_ARG, 1, chain, -1);
      chain_done();
      return;
    }
    t0 = a;
    len = b - a;
  }
  const int n_chunks = (int)((len + C - 1) / C);

  if (tid == 0) {
    mbar_init(&m.bar_qk, 1); mbar_init(&m.bar_la, 1); mbar_init(&m.bar_v, 1);
    mbar_init(&m.bar_gp, 1); mbar_init(&m.bar_m1, 1); mbar_init(&m.bar_u, 1);
    mbar_init(&m.bar_m2, 1); mbar_init(&m.bar_fin, 1);
    mbar_init(&m.bar_gops, kComputeWarps);
    mbar_init(&m.bar_build, kComputeWarps); mbar_init(&m.bar_om, kComputeWarps);
    mbar_init(&m.bar_t1, kComputeWarps / 2); mbar_init(&m.bar_t, kComputeWarps / 2);
    mbar_init(&m.bar_ny, kComputeWarps / 2);
    mbar_init(&m.bar_ad, kComputeWarps);
    mbar_init(&m.bar_plan, 1); mbar_init(&m.bar_pka, 1); mbar_init(&m.bar_pkb, 1);
    mbar_init(&m.bar_wb, 1); mbar_init(&m.bar_stg, 1);
    fence_mbarrier_init();
    m.abort = 0;
    for (int i = 0; i < 5; ++i) m.last_copy[i] = 0;
    m.test_chunk = -1;
    m.wait_ns = kWaitNs;
    if (kMode == kModePlain && test_control != nullptr && !helper) {
      const volatile TestControl *c = test_control;
      if (c->magic0 == kTestMagic0 && c->magic1 == kTestMagic1 && c->chain == chain) {
        m.test_chunk = c->chunk;
        m.wait_ns = 1000ull * c->wait_us;
        test_control->magic0 = 0;   // one shot
        test_control->magic1 = 0;
      }
    }
  }
  if (warp == 0) {
    tmem_alloc(&m.tmem_base, TM_COLS);
    tmem_relinquish();
  }
  float beta_pref = 0.f;   // beta of the chunk after the one being built (threads < C)
  if (tid < C && !helper) {
    st_shared_f32(sb + SM_BETA + 4u * tid, (n_chunks > 0 && tid < len) ? beta[(t0 + tid) * H + h] : 0.f);
    beta_pref = (n_chunks > 1 && tid < len - C) ? beta[(t0 + C + tid) * H + h] : 0.f;
  }
  cta_sync();
  const uint32_t tm = m.tmem_base;
  const int test_chunk = kMode == kModePlain ? m.test_chunk : -1;

  if (warp >= kComputeWarps) {
    // ===================== TMA + MMA issue (one thread) =====================
    setmaxnreg_dec<kIssueRegs>();
    // Copies of a chunk's q, k, log_alpha and v tiles: `phase` is the chunk's
    // index in this CTA's sequence of chunks, `hd` the head, `tb` the first token.
    auto issue_qk = [&](int phase, int hd, int32_t tb) {
      mbar_arrive_expect_tx(&m.bar_qk, 2 * 16384);
      tma_load_3d(smem + SM_Q, &tm_q, &m.bar_qk, 0, hd, tb);
      tma_load_3d(smem + SM_Q + 8192, &tm_q, &m.bar_qk, 64, hd, tb);
      tma_load_3d(smem + SM_K, &tm_k, &m.bar_qk, 0, hd, tb);
      tma_load_3d(smem + SM_K + 8192, &tm_k, &m.bar_qk, 64, hd, tb);
      m.last_copy[TMA_QK] = (uint32_t)phase + 1u;
    };
    auto issue_la = [&](int phase, int hd, int32_t tb) {
      mbar_arrive_expect_tx(&m.bar_la, 32768);
      tma_load_3d(smem + SM_LA, &tm_la, &m.bar_la, 0, hd, tb);
      m.last_copy[TMA_LA] = (uint32_t)phase + 1u;
    };
    auto issue_v = [&](int phase, int hd, int32_t tb) {
      mbar_arrive_expect_tx(&m.bar_v, 16384);
      tma_load_3d(smem + SM_V, &tm_v, &m.bar_v, 0, hd, tb);
      m.last_copy[TMA_V] = (uint32_t)phase + 1u;
    };
    auto tok = [&](int ci) { return (int32_t)(t0 + (int64_t)C * ci); };
    // The Gram / P MMAs of the chunk whose operands were just built.  Their
    // accumulator columns also hold the previous chunk's bf16 Delta^T, so the
    // caller has waited for the previous M2 group.
    auto issue_gram = [&](uint32_t sa, uint32_t tmb) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t ad = sdesc_sw128(sa + SM_GA + (ks >> 2) * 16384u + (ks & 3) * 32u, 16, 1024);
        const uint64_t bd =
            sdesc_sw128(sa + SM_GB + (ks >> 2) * (GB_ROWS * 128u) + (ks & 3) * 32u, 16, 1024);
        umma_ss(tmb + TM_GP, ad, bd, ID_GP, ks > 0 ? 1u : 0u);
      }
      umma_commit(&m.bar_gp);
    };
    if (warp == kMmaWarp && lane == 0 && helper) {
      // ---- helper: claim a chunk well ahead of its chain CTA, build it, publish it
      const int hid = chain - help.n_chains, n_help = (int)gridDim.x - help.n_chains;
      int rr = (int)((int64_t)hid * help.n_chains / n_help);  // spread the starting chains
      // Claims the lowest chunk of some chain in [pos + kHelpLead, pos + kHelpSlots - 1]
      // (pos: the chunk its chain CTA has started) into m.claim[slot], together with
      // its ring slot: a slot is written by one helper at a time (busy word), so a
      // late writer can never mix into a newer package.  Returns false when nothing
      // is claimable: at once unless `wait`, else once every chain CTA has finished
      // or nothing was claimable for kHelpIdleNs.
      // Sequence table (start, length; length 0 for a malformed entry) in the v
      // buffer, which a helper never uses: the claim scans read no global memory
      // but the chain positions and claim counters.
      int32_t *tab = reinterpret_cast<int32_t *>(smem + SM_V);
      const int n_tab = help.n_chains / H;
      for (int sq = 0; sq < n_tab; ++sq) {
        const int64_t a = cu_seqlens[sq], b = cu_seqlens[sq + 1];
        const bool ok = a >= 0 && b >= a && b <= n_tokens;
        tab[2 * sq] = ok ? (int32_t)a : 0;
        tab[2 * sq + 1] = ok ? (int32_t)(b - a) : 0;
      }
      auto claim = [&](int slot, bool wait) -> bool {
        HelpClaim &cl = m.claim[slot];
        cl.valid = 0;
        const uint64_t idle0 = global_timer_ns();
        for (;;) {
          for (int k = 0; k < help.n_chains; ++k) {
            const int hc = rr;
            rr = rr + 1 == help.n_chains ? 0 : rr + 1;
            const int sq = hc / H;
            const int64_t a = tab[2 * sq], b = a + tab[2 * sq + 1];
            const int64_t nch = (b - a + C - 1) / C;
            if (nch <= 0) continue;
            const int64_t pos = ld_relaxed_gpu(help.cons_pos + hc);
            const int64_t lo = pos + kHelpLead;
            const int64_t hi = pos + kHelpSlots - 1 < nch - 1 ? pos + kHelpSlots - 1 : nch - 1;
            if (lo > hi) continue;
            int o = ld_relaxed_gpu(help.next_claim + hc);
            for (;;) {
              const int64_t want = o > lo ? o : lo;
              if (want > hi) break;
              const int prev = atomicCAS(help.next_claim + hc, o, (int)want + 1);
              if (prev == o) {
                // The chunk is ours; so must its slot be (else its chain computes it).
                int32_t *bz = help.busy + (size_t)hc * kHelpSlots + want % kHelpSlots;
                if (atomicCAS(bz, 0, (int)want + 1) != 0) break;
                __threadfence();  // the slot's last writer is done before we write
                cl.chain = hc;
                cl.chunk = (int)want;
                cl.tb = (int32_t)(a + C * want);
                cl.nv = (int)(b - (a + C * want) < C ? b - (a + C * want) : C);
                cl.head = hc % H;
                cl.valid = 1;
                return true;
              }
              o = prev;
            }
          }
          if (!wait || ld_relaxed_gpu(help.finished) >= help.n_chains) return false;
          if (global_timer_ns() - idle0 > kHelpIdleNs) return false;
          __nanosleep(1000);
        }
      };
      prefetch_tensormap(&tm_q); prefetch_tensormap(&tm_k); prefetch_tensormap(&tm_la);
      auto load_claim = [&](int phase) {
        const HelpClaim &c = m.claim[phase & 1];
        issue_la(phase, c.head, c.tb);
        issue_qk(phase, c.head, c.tb);
      };
      int n_published = 0;
      bool have = claim(0, true);
      mbar_arrive(&m.bar_plan);
      if (have) load_claim(0);
      for (int j = 0; have; ++j) {
        const uint32_t par = (uint32_t)(j & 1);
        uint32_t sa = sb, tmb = tm;
        asm volatile("" : "+r"(sa), "+r"(tmb));
        if (!wait_bar(cx, &m.bar_build, par, 60, j)) break;
        if (*reinterpret_cast<volatile int *>(&m.abort)) break;
        tc_fence_after();
        issue_gram(sa, tmb);
        // One pass for the next claim now, so its tiles load during this chunk
        // (the build has consumed q, k and log_alpha); if nothing is claimable
        // yet, claim again, waiting, only after this chunk is published.
        bool next = claim((j + 1) & 1, false);
        if (next) {
          mbar_arrive(&m.bar_plan);
          load_claim(j + 1);
        }
        // The package: P after the A/P epilogue, T' after the solve.
        if (!wait_bar(cx, &m.bar_om, par, 61, j)) break;
        if (!wait_bar(cx, &m.bar_t, par, 62, j)) break;
        const HelpClaim &cl = m.claim[par];
        const size_t si = (size_t)cl.chain * kHelpSlots + cl.chunk % kHelpSlots;
        // Written only while its chain CTA has not reached the chunk yet.
        if (ld_relaxed_gpu(help.cons_pos + cl.chain) < cl.chunk - 1) {
          unsigned char *slot = help.ring + si * kHelpSlotStride;
          fence_proxy_async_global();  // after the slot claim, before the async writes
          bulk_store(slot + PKG_STACK, sa + SM_STACK, 32768);
          bulk_store(slot + PKG_KDEC, sa + SM_KDEC, 16384);
          bulk_store(slot + PKG_TMAT, sa + SM_TMAT, 8192);
          bulk_store(slot + PKG_PMAT, sa + SM_PMAT, 8192);
          bulk_store(slot + PKG_GAMMA, sa + SM_GAMMA, 512);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(&m.bar_wb);  // the compute warps may build the next chunk
          bulk_wait_all();
          fence_proxy_async_global();  // the package's writes before the flag that publishes it
          st_release_gpu(help.flag + si, cl.chunk + 1);
          ++n_published;
        } else {
          mbar_arrive(&m.bar_wb);
        }
        __threadfence();
        st_release_gpu(help.busy + si, 0);  // the slot may take a later chunk
        if (!next) {
          next = claim((j + 1) & 1, true);
          mbar_arrive(&m.bar_plan);
          if (next) load_claim(j + 1);
        }
        have = next;
      }
      bulk_wait_all();
      if (n_published) atomicAdd(&status->help_published, n_published);
    } else if (warp == kMmaWarp && lane == 0 && n_chunks > 0) {
      // The issue thread polls its barriers (its reaction time is on the chain's
      // critical path), except beside helper CTAs, where suspending waits are faster.
      constexpr bool kPoll = kMode != kModeHelp;
      // A ready package of chunk ci sits in ring slot ci % kHelpSlots of this chain.
      unsigned char *my_ring =
          helping ? help.ring + (size_t)chain * kHelpSlots * kHelpSlotStride : nullptr;
      const int32_t *my_flag = helping ? help.flag + (size_t)chain * kHelpSlots : nullptr;
      auto slot_of = [&](int ci) { return my_ring + (size_t)(ci % kHelpSlots) * kHelpSlotStride; };
      prefetch_tensormap(&tm_q); prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v); prefetch_tensormap(&tm_la); prefetch_tensormap(&tm_o);
      issue_la(0, h, tok(0)); issue_qk(0, h, tok(0)); issue_v(0, h, tok(0));
      bool helped_cur = false;  // chunk ci comes from a helper's package
      int n_used = 0;           // packages used
      for (int ci = 0; ci < n_chunks; ++ci) {
        const uint32_t par = (uint32_t)(ci & 1);
        const bool has_next = ci + 1 < n_chunks;
        // Opaque per-iteration copies of the shared-memory and TMEM bases: the
        // descriptors below are rebuilt at each use instead of being hoisted out
        // of the loop into (many) registers.
        uint32_t sa = sb, tmb = tm;
        asm volatile("" : "+r"(sa), "+r"(tmb));
        auto kd = [&](uint32_t off) { return sdesc_sw128(sa + off, 16, 1024); };
        auto mnd = [&](uint32_t off, uint32_t lbo) { return sdesc_sw128(sa + off, lbo, 1024); };
        const uint32_t to = tmb + TM_O + 64u * (uint32_t)(ci & 1);
        if (!wait_bar(cx, &m.bar_gops, par, 30, ci, kPoll)) break;
        if (*reinterpret_cast<volatile int *>(&m.abort)) break;  // no new copies once aborting
        PHASE_MARK_MMA(0);
        if (ci > 0 && !wait_bar(cx, &m.bar_m2, par ^ 1u, 36, ci - 1, kPoll)) break;
        tc_fence_after();
        if (helped_cur) {
          // T' and P of the package: the previous chunk's Delta and M2 MMAs have
          // read theirs.  One phase of bar_gp per chunk either way.
          mbar_arrive_expect_tx(&m.bar_pkb, 16384);
          bulk_load(sa + SM_TMAT, slot_of(ci) + PKG_TMAT, 8192, &m.bar_pkb);
          bulk_load(sa + SM_PMAT, slot_of(ci) + PKG_PMAT, 8192, &m.bar_pkb);
          m.last_copy[TMA_PKB] = (uint32_t)ci + 1u;
          mbar_arrive(&m.bar_gp);
        } else {
          issue_gram(sa, tmb);
          mbar_arrive(&m.bar_pkb);
        }
        PHASE_MARK_MMA(5);
        // Plan the next chunk: a helper's package if one is ready (its q, k and
        // log_alpha tiles are then never loaded), else its own tiles.
        const bool helped_next = has_next && helping && ci + 1 >= kHelpLead &&
                                 ld_acquire_gpu(my_flag + (ci + 1) % kHelpSlots) == ci + 2;
        if (has_next) {
          if (helped_next) {
            fence_proxy_async_global();  // the package's writes before the copies that read it
            mbar_arrive(&m.bar_la);
            mbar_arrive(&m.bar_qk);
            ++n_used;
          } else {
            issue_la(ci + 1, h, tok(ci + 1));
            issue_qk(ci + 1, h, tok(ci + 1));
          }
          if (helping) {
            m.plan[(ci + 1) & 1] = helped_next ? 1 : 0;
            mbar_arrive(&m.bar_plan);
          }
          PHASE_STAMP(32 * kMmaWarp, 51);
        }
        // [O^T | Y^T] = S^T [Qt; Kt]^T
        if (!wait_bar(cx, &m.bar_om, par, 31, ci, kPoll)) break;
        if (!wait_bar(cx, &m.bar_build, par, 40, ci, kPoll)) break;  // [Qt; Kt] and Kdec of the chunk
        PHASE_MARK_MMA(1);
        if (helped_cur && !wait_bar(cx, &m.bar_pka, par ^ 1u, 38, ci, kPoll)) break;
        if (has_next) {
          // Gamma of the next chunk (this chunk's state pass has read Gamma); the
          // phase's byte count covers the two copies issued after the (V - Y) pass.
          if (helped_next) {
            mbar_arrive_expect_tx(&m.bar_pka, 512 + 32768 + 16384);
            bulk_load(sa + SM_GAMMA, slot_of(ci + 1) + PKG_GAMMA, 512, &m.bar_pka);
            m.last_copy[TMA_PKA] = (uint32_t)ci + 1u;
          } else {
            mbar_arrive(&m.bar_pka);
          }
        }
        tc_fence_after();
        // Y first: only it gates the (V - Y) pass; O follows in the same pipe
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = SM_STACK + (ks >> 2) * 16384u + (ks & 3) * 32u;
          umma_ts(tmb + TM_Y, tmb + TM_AS + 8u * ks, kd(off + 8192u), ID_N64, ks > 0 ? 1u : 0u);
        }
        umma_commit(&m.bar_m1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = SM_STACK + (ks >> 2) * 16384u + (ks & 3) * 32u;
          umma_ts(to, tmb + TM_AS + 8u * ks, kd(off), ID_N64, ks > 0 ? 1u : 0u);
        }
        PHASE_MARK_MMA(6);
        // Delta^T = (V - Y)^T T'^T, K step s covering tokens 16 s .. 16 s + 15 and
        // writing only output columns r >= 16 s (T' is lower triangular).  Output
        // columns 0-31 and K steps 2, 3 need only the diagonal and 16 -> 32 blocks
        // of T' and are issued as soon as those exist; the two remaining products
        // wait for the 32 -> 64 blocks.
        if (!wait_bar(cx, &m.bar_ny, par, 33, ci, kPoll)) break;
        PHASE_MARK_MMA(3);
        if (has_next) issue_v(ci + 1, h, tok(ci + 1));   // the (V - Y) pass has read this chunk's v tile
        if (!wait_bar(cx, &m.bar_t1, par, 37, ci, kPoll)) break;
        if (helped_cur && !wait_bar(cx, &m.bar_pkb, par, 39, ci, kPoll)) break;
        tc_fence_after();
        umma_ts(tmb + TM_D, tmb + TM_NY, kd(SM_TMAT), ID_N32, 0u);                       // r 0-31, s 0
        umma_ts(tmb + TM_D + 16u, tmb + TM_NY + 8u, kd(SM_TMAT + 16u * 128u + 32u), ID_N16,
                1u);                                                                   // r 16-31, s 1
        umma_ts(tmb + TM_D + 32u, tmb + TM_NY + 16u, kd(SM_TMAT + 32u * 128u + 64u), ID_N32,
                0u);                                                                   // r 32-63, s 2
        umma_ts(tmb + TM_D + 48u, tmb + TM_NY + 24u, kd(SM_TMAT + 48u * 128u + 96u), ID_N16,
                1u);                                                                   // r 48-63, s 3
        if (!wait_bar(cx, &m.bar_t, par, 32, ci, kPoll)) break;
        PHASE_MARK_MMA(2);
        tc_fence_after();
        umma_ts(tmb + TM_D + 32u, tmb + TM_NY, kd(SM_TMAT + 32u * 128u), ID_N32, 1u);        // r 32-63, s 0
        umma_ts(tmb + TM_D + 32u, tmb + TM_NY + 8u, kd(SM_TMAT + 32u * 128u + 32u), ID_N32,
                1u);                                                                   // r 32-63, s 1
        umma_commit(&m.bar_u);
        if (helped_next) {
          // [Qt; Kt] of the next chunk once every MMA up to this chunk's Delta has
          // completed (its O MMAs read the stack), and its Kdec once the staged
          // output stores have read the Kdec buffer they share.
          if (!wait_bar(cx, &m.bar_u, par, 46, ci, kPoll)) break;
          bulk_load(sa + SM_STACK, slot_of(ci + 1) + PKG_STACK, 32768, &m.bar_pka);
          if (!wait_bar(cx, &m.bar_stg, par, 47, ci, kPoll)) break;
          bulk_load(sa + SM_KDEC + 16384u * (uint32_t)((ci + 1) & 1), slot_of(ci + 1) + PKG_KDEC,
                    16384, &m.bar_pka);
        }
        // S^T += Delta^T Kdec ; O^T += Delta^T P^T
        if (!wait_bar(cx, &m.bar_ad, par, 35, ci, kPoll)) break;
        PHASE_MARK_MMA(4);
        tc_fence_after();
        const uint32_t kdec = SM_KDEC + 16384u * (uint32_t)(ci & 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          umma_ts(tmb + TM_S, tmb + TM_AD + 8u * ks, mnd(kdec + ks * 2048u, 8192), ID_KM128, 1u);
          umma_ts(to + 16u * ks, tmb + TM_AD + 8u * ks, kd(SM_PMAT + ks * 2048u + ks * 32u),
                  id_tri(ks, false), 1u);
        }
        umma_commit(&m.bar_m2);
        PHASE_MARK_MMA(7);
        helped_cur = helped_next;
      }
      if (n_used) atomicAdd(&status->help_consumed, n_used);
    }
    __syncwarp();
  } else {
    // ===================== compute warps 0-7 =====================
    setmaxnreg_inc<kComputeRegs>();
    const int q4 = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half
    const uint32_t lane_base = 32u * q4;
    const int64_t sbase = ((int64_t)seq * H + h) * D * D;

    // ---- initial state -> S^T in TMEM (thread: lane n, 64 key columns of its half)
    if (!helper) {
      const int n = lane_base + lane;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int c0 = 64 * hf + 32 * part;
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          r[j] = __float_as_uint(transition ? (c0 + j == n ? 1.f : 0.f)
                                 : init_state ? init_state[sbase + (int64_t)(c0 + j) * D + n]
                                              : 0.f);
        tmem_st32(tmem_addr(tm, lane_base, TM_S + c0), r);
      }
      tmem_st_wait();
    }

    // Writes the output rows of a finished chunk (warps 4-7): O^T (TMEM) -> bf16
    // rows [r][n] staged in an idle Kdec buffer -> one TMA store of the whole
    // 64 x 128 tile (issued by thread 128, which later waits for its read), or,
    // for a sequence's ragged last chunk, 16-byte stores of the valid rows.
    // (a transition run writes its outputs, M_t^T q_t, to out_m)
    auto flush_output = [&](int64_t otb, int onv, uint32_t ocol, uint32_t stg_off) {
      if (kMode == kModeTransitions && !write_out) return;  // warp-uniform (warps 4-7)
      const CUtensorMap *omap = transition ? &tm_om : &tm_o;
      __nv_bfloat16 *optr = transition ? out_m : out;
      const int n = lane_base + lane;
      const uint32_t stg = sb + stg_off;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tm, lane_base, ocol + 32u * part), r);
        tmem_ld_wait(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const __nv_bfloat16 o = __float2bfloat16_rn(__uint_as_float(r[j]));
          st_shared_b16(stg + (uint32_t)(32 * part + j) * 256u + 2u * n,
                        *reinterpret_cast<const uint16_t *>(&o));
        }
      }
      fence_proxy_async_smem();
      named_sync(3, 128);
      if (onv == C) {
        if (tid == 128) {
          tma_store_3d(omap, smem + stg_off, 0, h, (int32_t)otb);
          bulk_commit();
        }
      } else {
        for (int e = tid - 128; e < onv * 16; e += 128) {   // row e / 16, 16-byte chunk e % 16
          const int row = e >> 4, ch = e & 15;
          *reinterpret_cast<uint4 *>(optr + ((otb + row) * H + h) * D + 8 * ch) =
              ld_shared_v4(stg + (uint32_t)row * 256u + 16u * ch);
        }
      }
    };

    // Thread (tile ta, channel pair cp) owns rows 16 ta .. 16 ta + 15 of key
    // channels cc, cc + 1 in the decay prefix and the operand build.
    const int ta = tid >> 6, cp = tid & 63, cc = 2 * cp;
    const uint32_t hsel = (uint32_t)(cc >> 6), cb = (uint32_t)(cc & 63) * 2u;
    uint32_t swzk[8];  // swizzled byte offset of channel pair cc in a row with row % 8 == k
#pragma unroll
    for (int k = 0; k < 8; ++k) swzk[k] = ((((cb >> 4) ^ (uint32_t)k) << 4) | (cb & 15u));
    const uint32_t sla = sb + SM_LA;  // log_alpha tile [64][128] fp32, then the tile totals

    // Decay prefix and every operand tile of a chunk of nv valid rows, whose
    // q, k and log_alpha tiles are phase `par` of their barriers (ci: the chunk's
    // index in this CTA's sequence), with Kdec into the buffer at kdec_off;
    // false if the CTA aborts.  The chunk's beta must already be in shared memory.
    auto build_tiles = [&](int ci, uint32_t par, int nv, uint32_t kdec_off) -> bool {
      // tile-local prefix of the log2-decay
      wait_bar(cx, &m.bar_la, par, 11, ci);
      float L0[16], L1[16];
      {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int row = 16 * ta + j;
          float2 x = ld_shared_f32x2(sla + 4u * (row * D + cc));
          if (row >= nv) x = make_float2(0.f, 0.f);
          s0 = fmaf(x.x, kLog2e, s0);
          s1 = fmaf(x.y, kLog2e, s1);
          L0[j] = s0;
          L1[j] = s1;
        }
        // tile totals, written over this thread's own (already read) first row
        st_shared_f32x2(sla + 4u * ((16 * ta) * D + cc), s0, s1);
      }
      if (compute_sync_abort(&m.abort)) return false;
      PHASE_MARK(9);
      wait_bar(cx, &m.bar_qk, par, 10, ci);
      PHASE_MARK(14);
      float st0[4], st1[4], rf0[4], rf1[4];  // tile starts / ends, channels cc, cc + 1
      {
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const float2 t = ld_shared_f32x2(sla + 4u * ((16 * b) * D + cc));
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
      uint32_t fb2[4];
#pragma unroll
      for (int a2 = 0; a2 < 4; ++a2) fb2[a2] = pack_bf16x2(ex2(st0[a2] - ra0), ex2(st1[a2] - ra1));
      const float fs0 = ex2(sa0), fs1 = ex2(sa1);
      const uint32_t fd2 = pack_bf16x2(ex2(rf0[3] - ra0), ex2(rf1[3] - ra1));
      if (ta == 0) {
        st_shared_f32x2(sb + SM_GAMMA + 4u * cc, ex2(rf0[3]), ex2(rf1[3]));
      }
      const uint32_t r0 = 16u * ta * 128u, h64 = hsel * 8192u, h128 = hsel * 16384u;
      const uint32_t bK = sb + SM_K + h64 + r0, bQ = sb + SM_Q + h64 + r0;
      const uint32_t bGA = sb + SM_GA + h128 + 2u * r0, bST = sb + SM_STACK + h128 + r0;
      const uint32_t bKD = sb + kdec_off + h64 + r0;
      const uint32_t bGB = sb + SM_GB + hsel * (GB_ROWS * 128u) + r0;
      uint32_t kraw[16], qraw[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        kraw[j] = ld_shared_b32(bK + (uint32_t)j * 128u + swzk[j & 7]);
        qraw[j] = ld_shared_b32(bQ + (uint32_t)j * 128u + swzk[j & 7]);
      }
      // The Gram operands first, so that the Gram / P MMAs run under the rest
      // of the build; the factors the rest needs stay packed in registers.
      uint32_t g2s[16], kc2s[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t o = (uint32_t)j * 128u + swzk[j & 7];
        const uint32_t k2 = kraw[j], q2 = qraw[j];
        const float e0 = ex2(L0[j]), e1 = ex2(L1[j]);
        const uint32_t e2 = pack_bf16x2(e0, e1);
        const uint32_t ec2 = pack_bf16x2(ex2(tot0 - L0[j]), ex2(tot1 - L1[j]));
        st_shared_b32(bGA + o, hmul2_bf16(k2, e2));
        st_shared_b32(bGA + 2048u + o, hmul2_bf16(q2, e2));
        const uint32_t kc2 = hmul2_bf16(k2, ec2);
#pragma unroll
        for (int a2 = 0; a2 < 4; ++a2) {
          if (a2 < ta) continue;
          st_shared_b32(bGB + 16u * blk(a2, 0) * 128u + o, hmul2_bf16(kc2, fb2[a2]));
        }
        g2s[j] = pack_bf16x2(e0 * fs0, e1 * fs1);
        kc2s[j] = kc2;
      }
      fence_proxy_async_smem();
      // (a test may withhold warp 0's arrival, so that the issue thread's wait
      // on these operands gives up)
      if (kMode != kModePlain || !(warp == 0 && ci == test_chunk)) warp_arrive(&m.bar_gops, lane);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t o = (uint32_t)j * 128u + swzk[j & 7];
        st_shared_b32(bST + o, hmul2_bf16(qraw[j], g2s[j]));
        st_shared_b32(bST + 8192u + o, hmul2_bf16(kraw[j], g2s[j]));
        st_shared_b32(bKD + o, hmul2_bf16(kc2s[j], fd2));
      }
      PHASE_MARK(15);
      PHASE_MARK_W7(2);
      fence_proxy_async_smem();
      warp_arrive(&m.bar_build, lane);
      return true;
    };
    // Chain CTA: beta of chunk ci into its buffer and the next chunk's prefetched.
    auto chain_beta = [&](int ci) {
      if (tid < C && ci > 0) {
        const int64_t tb = t0 + (int64_t)C * ci;
        st_shared_f32(sb + SM_BETA + 4u * ((ci & 1) * C + tid), beta_pref);
        const int64_t rem = len - (int64_t)C * (ci + 1);
        beta_pref = (ci + 1 < n_chunks && tid < rem) ? beta[(tb + C + tid) * H + h] : 0.f;
      }
    };
    auto chunk_rows = [&](int ci) {
      return (int)((len - (int64_t)C * ci) < C ? (len - (int64_t)C * ci) : C);
    };
    auto scan_build = [&](int ci) -> bool {
      chain_beta(ci);
      return build_tiles(ci, (uint32_t)(ci & 1), chunk_rows(ci), SM_KDEC + 16384u * (uint32_t)(ci & 1));
    };

    // Gram / P accumulators -> A (fp32 row-major, for the solve) and P (bf16, K-major
    // [r][i]), with the chunk's beta at sbeta.  Quadrant q4 holds row tile a = q4:
    // lanes 0-15 key rows, 16-31 query rows.
    auto ap_epilogue = [&](uint32_t sbeta, int ci) {
      {
        // Warps 0-3 take blocks b = 0, 1 of their row tile, warps 4-7 blocks 2, 3
        // (b <= a): adjacent block columns, so one TMEM load per warp.
        const int a = q4, j = lane & 15, r = 16 * a + j;
        const bool isq = lane >= 16;
        const float br = ld_shared_f32(sbeta + 4u * r);
        const uint32_t sat = sb + SM_GA;  // A = Diag(beta) G, fp32 [r][i], pitch FA
        const int b0 = 2 * hf, nb = a + 1 - b0 < 2 ? a + 1 - b0 : 2;  // warp-uniform
        uint32_t v[32];
        auto block = [&](int b, int off) {
          if (!isq) {   // entries i >= r of A are never read by the solve
#pragma unroll
            for (int q4v = 0; q4v < 4; ++q4v)
              st_shared_v4(sat + 4u * (r * FA + 16 * b + 4 * q4v),
                           __float_as_uint(br * __uint_as_float(v[off + 4 * q4v])),
                           __float_as_uint(br * __uint_as_float(v[off + 4 * q4v + 1])),
                           __float_as_uint(br * __uint_as_float(v[off + 4 * q4v + 2])),
                           __float_as_uint(br * __uint_as_float(v[off + 4 * q4v + 3])));
          } else {
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
              uint32_t w[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int jj = 8 * g8 + 2 * t, i = 16 * b + jj;
                const float lo = i <= r ? __uint_as_float(v[off + jj]) : 0.f;
                const float hi = i + 1 <= r ? __uint_as_float(v[off + jj + 1]) : 0.f;
                w[t] = pack_bf16x2(lo, hi);
              }
              st_shared_v4(sb + SM_PMAT + sw128_offset(r, (16 * b + 8 * g8) * 2), w[0], w[1],
                           w[2], w[3]);
            }
          }
        };
        const uint32_t src = tmem_addr(tm, lane_base, TM_GP + 16u * blk(a, b0));
        if (nb == 2) {
          tmem_ld32(src, v);
          tmem_ld_wait(v);
          PHASE_MARK_W3(3);
          block(b0, 0);
          PHASE_MARK_W3(4);
          block(b0 + 1, 16);
        } else if (nb == 1) {
          uint32_t w[16];
          tmem_ld16(src, w);
          tmem_ld_wait(w);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = w[i];
          block(b0, 0);
        }
      }
    };

    // T = (I + A)^{-1} and T' = T Diag(beta) from A (warps 0-3), beta at sbeta;
    // arrives on bar_t1 once the diagonal and 16 -> 32 blocks of T' exist and on
    // bar_t when all of T' does.
    auto solve_T = [&](uint32_t sbeta, int ci) {
      // ---- T = (I + A)^{-1} and T' = T Diag(beta) (warps 0-3)
      const uint32_t sat = sb + SM_GA;                // A, fp32 [r][i], pitch FA
      const uint32_t stv = sb + SM_GB + OFF_TINV;     // T, fp32 [r][i], pitch FP
      const uint32_t sxb = sb + SM_GB + OFF_XBUF;     // 4 blocks of 16 x XP fp32
      if (warp < 2) {
        // Diagonal 16 x 16 blocks by forward substitution over the rows: lane
        // owns column j of block a; t[r] = [r = j] - sum_{i<r} A[r][i] t[i],
        // accumulated in i order so only the last product waits for t[r - 1].
        // Rows of A stream through a ring, three rows ahead.
        const int a = 2 * warp + (lane >> 4), j = lane & 15, b0 = 16 * a;
        float t[16];
        float rbuf[4][16];
#pragma unroll
        for (int p = 0; p < 3; ++p) {
          lds8(*reinterpret_cast<float(*)[8]>(rbuf[p]), sat + 4u * ((b0 + p) * FA + b0));
          lds8(*reinterpret_cast<float(*)[8]>(rbuf[p] + 8), sat + 4u * ((b0 + p) * FA + b0 + 8));
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          if (r + 3 < 16) {
            float *nb = rbuf[(r + 3) & 3];
            lds8(*reinterpret_cast<float(*)[8]>(nb), sat + 4u * ((b0 + r + 3) * FA + b0));
            lds8(*reinterpret_cast<float(*)[8]>(nb + 8), sat + 4u * ((b0 + r + 3) * FA + b0 + 8));
          }
          const float *row = rbuf[r & 3];
          float sacc = 0.f;
#pragma unroll
          for (int i = 0; i < r; ++i) sacc = fmaf(row[i], t[i], sacc);
          t[r] = (r == j ? 1.f : 0.f) - sacc;
        }
        // T (fp32, for the block recursion) and T' = T Diag(beta) (bf16 MMA operand;
        // the block's upper triangle is zero because t[r] = 0 for r < j).
        const float bj = ld_shared_f32(sbeta + 4u * (b0 + j));
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          st_shared_f32(stv + 4u * ((b0 + r) * FP + b0 + j), t[r]);
          const __nv_bfloat16 tb16 = __float2bfloat16_rn(t[r] * bj);
          st_shared_b16(sb + SM_TMAT + sw128_offset(b0 + r, (b0 + j) * 2),
                        *reinterpret_cast<const uint16_t *>(&tb16));
        }
      }
      PHASE_MARK(11);
      __syncwarp();   // the 16 -> 32 level of a warp reads only that warp's diagonal blocks
      // Off-diagonal blocks, block-recursive: 16 -> 32 (blocks (1,0), (3,2)), then
      // 32 -> 64 (blocks (2,0), (2,1), (3,0), (3,1)), TF32 warp MMAs.
      const int g = lane >> 2, t4 = lane & 3;
      // acc (+)= A_{ab} T_{mb} with A row-major (pitch FA) ...
      auto mul_AT = [&](float (&acc)[2][4], int ab, int mb, int tcol) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int kc = 16 * mb + 8 * kk;
          const uint32_t a0 = to_tf32(ld_shared_f32(sat + 4u * ((16 * ab + g) * FA + kc + t4)));
          const uint32_t a1 = to_tf32(ld_shared_f32(sat + 4u * ((16 * ab + g + 8) * FA + kc + t4)));
          const uint32_t a2 = to_tf32(ld_shared_f32(sat + 4u * ((16 * ab + g) * FA + kc + t4 + 4)));
          const uint32_t a3 = to_tf32(ld_shared_f32(sat + 4u * ((16 * ab + g + 8) * FA + kc + t4 + 4)));
          const uint32_t b0p = stv + 4u * ((kc + t4) * FP + tcol + g);
          const uint32_t b1p = stv + 4u * ((kc + t4 + 4) * FP + tcol + g);
          mma_tf32_16x8x8(acc[0], a0, a1, a2, a3, to_tf32(ld_shared_f32(b0p)),
                          to_tf32(ld_shared_f32(b1p)));
          mma_tf32_16x8x8(acc[1], a0, a1, a2, a3, to_tf32(ld_shared_f32(b0p + 32u)),
                          to_tf32(ld_shared_f32(b1p + 32u)));
        }
      };
      // ... and acc (+)= T_{ar} X with T row-major (pitch FP), X a 16 x 16 block (pitch XP).
      auto mul_TX = [&](float (&acc)[2][4], int ar, int ac, uint32_t x) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint32_t tq = stv + 4u * ((16 * ar) * FP + 16 * ac + 8 * kk);
          const uint32_t a0 = to_tf32(ld_shared_f32(tq + 4u * (g * FP + t4)));
          const uint32_t a1 = to_tf32(ld_shared_f32(tq + 4u * ((g + 8) * FP + t4)));
          const uint32_t a2 = to_tf32(ld_shared_f32(tq + 4u * (g * FP + t4 + 4)));
          const uint32_t a3 = to_tf32(ld_shared_f32(tq + 4u * ((g + 8) * FP + t4 + 4)));
          const uint32_t x0 = x + 4u * ((8 * kk + t4) * XP + g);
          const uint32_t x1 = x + 4u * ((8 * kk + t4 + 4) * XP + g);
          mma_tf32_16x8x8(acc[0], a0, a1, a2, a3, to_tf32(ld_shared_f32(x0)),
                          to_tf32(ld_shared_f32(x1)));
          mma_tf32_16x8x8(acc[1], a0, a1, a2, a3, to_tf32(ld_shared_f32(x0 + 32u)),
                          to_tf32(ld_shared_f32(x1 + 32u)));
        }
      };
      auto store_blk = [&](uint32_t dst, int pitch, const float (&acc)[2][4], float sgn) {
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
          st_shared_f32x2(dst + 4u * (g * pitch + 8 * nh + 2 * t4), sgn * acc[nh][0],
                          sgn * acc[nh][1]);
          st_shared_f32x2(dst + 4u * ((g + 8) * pitch + 8 * nh + 2 * t4), sgn * acc[nh][2],
                          sgn * acc[nh][3]);
        }
      };
      // Final block T_ab: fp32 into T, and T' = T Diag(beta) as bf16 pairs.
      auto store_T = [&](int ab, int bb, const float (&acc)[2][4]) {
        store_blk(stv + 4u * ((16 * ab) * FP + 16 * bb), FP, acc, -1.f);
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
          const int col = 16 * bb + 8 * nh + 2 * t4;
          const float2 bv = ld_shared_f32x2(sbeta + 4u * col);
          const float b0v = bv.x, b1v = bv.y;
          const uint32_t lo = pack_bf16x2(-acc[nh][0] * b0v, -acc[nh][1] * b1v);
          const uint32_t hi = pack_bf16x2(-acc[nh][2] * b0v, -acc[nh][3] * b1v);
          st_shared_b32(sb + SM_TMAT + sw128_offset(16 * ab + g, col * 2), lo);
          st_shared_b32(sb + SM_TMAT + sw128_offset(16 * ab + g + 8, col * 2), hi);
        }
      };
      const uint32_t xw = sxb + 4u * (warp * 16 * XP);
      if (warp < 2) {  // level 16 -> 32: block (1,0) on warp 0, (3,2) on warp 1
        const int ab = 2 * warp + 1, bb = 2 * warp;
        float acc[2][4] = {};
        mul_AT(acc, ab, bb, 16 * bb);  // X = A_ab T_bb
        store_blk(xw, XP, acc, 1.f);
        __syncwarp();
        float o[2][4] = {};
        mul_TX(o, ab, ab, xw);  // T_ab = -T_aa X
        store_T(ab, bb, o);
      }
      PHASE_MARK(12);
      named_sync(2, 128);
      fence_proxy_async_smem();   // diagonal and 16 -> 32 blocks of T' are MMA operands
      warp_arrive(&m.bar_t1, lane);
      {  // level 32 -> 64: warp w -> block (2 + w/2, w%2)
        const int ab = 2 + (warp >> 1), bb = warp & 1;
        float acc[2][4] = {};
        // X_{ab} = A_{ab,0:2} T_{0:2, bb} = sum_{m=bb}^{1} A_{ab,m} T_{m,bb}
        for (int mb = bb; mb < 2; ++mb) mul_AT(acc, ab, mb, 16 * bb);
        store_blk(xw, XP, acc, 1.f);
        PHASE_MARK(13);
        named_sync(2, 128);
        // T_{ab} = -sum_{k=2}^{ab} T_{ab,k} X_{k,bb}
        float o[2][4] = {};
        for (int k = 2; k <= ab; ++k) mul_TX(o, ab, k, sxb + 4u * ((2 * (k - 2) + bb) * 16 * XP));
        store_T(ab, bb, o);
      }
      PHASE_MARK_W3(2);
      fence_proxy_async_smem();  // T' is an MMA operand
      warp_arrive(&m.bar_t, lane);
      PHASE_MARK(5);
    };

    bool failed = false;
    int64_t prev_tb = 0;
    int prev_nv = 0;
    bool helped = false;  // this chunk's package comes from a helper
    if (!helper && n_chunks > 0 && !scan_build(0)) failed = true;
    for (int ci = 0; ci < n_chunks && !failed; ++ci) {
      const uint32_t par = (uint32_t)(ci & 1);
      const int64_t tb = t0 + (int64_t)C * ci;
      const int nv = (int)((len - (int64_t)C * ci) < C ? (len - (int64_t)C * ci) : C);
      const uint32_t sbeta = sb + SM_BETA + 4u * C * (uint32_t)(ci & 1);  // this chunk's beta
      if (helping && tid == 0) st_relaxed_gpu(help.cons_pos + chain, ci);
      PHASE_MARK(0);
      PHASE_VALUE(0, 50, helped ? 1 : 0);
      if (ci > 0) {  // the previous chunk's state update and output are final
        wait_bar(cx, &m.bar_m2, par ^ 1u, 25, ci - 1);
        tc_fence_after();
      }
      // Gamma, beta and the operand tiles of this chunk visible
      if (compute_sync_abort(&m.abort)) { failed = true; break; }
      PHASE_MARK(1);
      if (helped) wait_bar(cx, &m.bar_pka, par ^ 1u, 43, ci);  // Gamma, [Qt; Kt], Kdec of the package

      // ---- S^T <- S^T Diag(Gamma_C); bf16 pre-chunk S^T as the A operand
      {
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const int c0 = 64 * hf + 32 * part;
          uint32_t s[32];
          tmem_ld32(tmem_addr(tm, lane_base, TM_S + c0), s);
          tmem_ld_wait(s);
          if (part == 0) PHASE_MARK_W3(5);
          uint32_t ab[16];
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            float gv[8];
            lds8(gv, sb + SM_GAMMA + 4u * (c0 + 8 * q8));
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
      PHASE_MARK(2);

      if (!helped) {
        wait_bar(cx, &m.bar_gp, par, 22, ci);
        tc_fence_after();
        PHASE_MARK(3);
        PHASE_MARK_W3(0);
        ap_epilogue(sbeta, ci);
      }
      PHASE_MARK(10);
      PHASE_MARK_W3(1);
      PHASE_MARK_W7(0);
      if (!helped) fence_proxy_async_smem();
      tc_fence_before();
      warp_arrive(&m.bar_om, lane);  // S^T operand ready, Gram columns free: O+M1 may start
      // A visible to the solve warps
      if (compute_sync_abort(&m.abort)) { failed = true; break; }
      PHASE_MARK(4);

      if (warp < 4) {
        if (helped) {  // T' of the package
          wait_bar(cx, &m.bar_pkb, par, 44, ci);
          warp_arrive(&m.bar_t1, lane);
          warp_arrive(&m.bar_t, lane);
        } else {
          solve_T(sbeta, ci);
        }
      } else {
        // ---- the previous chunk's output rows (while the O+Y MMAs run), then
        // (V - Y)^T as a bf16 A operand (warps 4-7; lane n of quadrant q4 is value
        // channel n).  Staging: the Kdec buffer of chunks ci - 1 and ci + 1, idle
        // until the next build.
        PHASE_MARK_W4(0);
        if (ci > 0)
          flush_output(prev_tb, prev_nv, TM_O + 64u * (par ^ 1u), SM_KDEC + 16384u * (par ^ 1u));
        PHASE_MARK_W4(1);
        wait_bar(cx, &m.bar_m1, par, 24, ci);
        tc_fence_after();
        wait_bar(cx, &m.bar_v, par, 12, ci);
        PHASE_MARK_W4(2);
        {
          const uint32_t vb = sb + SM_V + 2u * (lane_base + lane);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            uint32_t y[32];
            tmem_ld32(tmem_addr(tm, lane_base, TM_Y + 32u * part), y);
            tmem_ld_wait(y);
            uint32_t p[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const uint32_t row = 32u * part + 2u * jj;
              // a transition run has v = 0
              const float v0 =
                  transition ? 0.f : __uint_as_float(ld_shared_u16(vb + row * 256u) << 16);
              const float v1 =
                  transition ? 0.f : __uint_as_float(ld_shared_u16(vb + (row + 1u) * 256u) << 16);
              p[jj] = pack_bf16x2(v0 - __uint_as_float(y[2 * jj]), v1 - __uint_as_float(y[2 * jj + 1]));
            }
            tmem_st16(tmem_addr(tm, lane_base, TM_NY + 16u * part), p);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        // The staged output stores must have read the Kdec buffer before anything
        // reuses it: the next build (after barriers thread 128 joins only past
        // this wait) or, with helpers, a package copy (issued on bar_stg).
        warp_arrive(&m.bar_ny, lane);
        if (tid == 128) {
          bulk_wait_read_all();
          if (helping) mbar_arrive(&m.bar_stg);
        }
        PHASE_MARK_W4(3);
        PHASE_MARK_W7(1);
      }

      // ---- bf16 Delta^T, the A operand of the state and output updates
      wait_bar(cx, &m.bar_u, par, 23, ci);
      tc_fence_after();
      PHASE_MARK(6);
      {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tm, lane_base, TM_D + 32u * hf), r);
        tmem_ld_wait(r);
        uint32_t ab[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          ab[jj] = pack_bf16x2(__uint_as_float(r[2 * jj]), __uint_as_float(r[2 * jj + 1]));
        tmem_st16(tmem_addr(tm, lane_base, TM_AD + 16u * hf), ab);
        tmem_st_wait();
      }
      tc_fence_before();
      warp_arrive(&m.bar_ad, lane);
      PHASE_MARK(7);
      prev_tb = tb;
      prev_nv = nv;
      // ---- the next chunk's operand tiles, while the state MMAs run, unless a
      // helper's package of it is on its way
      if (ci + 1 < n_chunks) {
        if (helping) {
          wait_bar(cx, &m.bar_plan, par, 45, ci);
          PHASE_STAMP(0, 52);
          if (compute_sync_abort(&m.abort)) { failed = true; break; }
          helped = m.plan[(ci + 1) & 1] != 0;
        }
        if (helped) {
          chain_beta(ci + 1);
          warp_arrive(&m.bar_gops, lane);
          warp_arrive(&m.bar_build, lane);
        } else if (!scan_build(ci + 1)) {
          failed = true;
          break;
        }
      }
      PHASE_MARK(8);
    }
    chain_done();

    // ---- helper CTA: operand build, Gram / P and solve of each claimed chunk
    for (int j = 0; helper && !failed; ++j) {
      const uint32_t par = (uint32_t)(j & 1);
      wait_bar(cx, &m.bar_plan, par, 63, j);
      if (compute_sync_abort(&m.abort)) break;
      const HelpClaim cl = m.claim[par];
      if (!cl.valid) break;
      if (j > 0) wait_bar(cx, &m.bar_wb, par ^ 1u, 64, j);  // the last package is out of smem
      const uint32_t sbeta = sb + SM_BETA + 4u * C * par;
      if (tid < C)
        st_shared_f32(sbeta + 4u * tid,
                      tid < cl.nv ? beta[((int64_t)cl.tb + tid) * H + cl.head] : 0.f);
      if (!build_tiles(j, par, cl.nv, SM_KDEC)) break;
      wait_bar(cx, &m.bar_gp, par, 65, j);
      tc_fence_after();
      ap_epilogue(sbeta, j);
      fence_proxy_async_smem();
      tc_fence_before();
      warp_arrive(&m.bar_om, lane);
      if (compute_sync_abort(&m.abort)) break;
      if (warp < 4) solve_T(sbeta, j);
    }

    // ---- the last chunk's output and the final state
    if (!failed && n_chunks > 0) {
      wait_bar(cx, &m.bar_m2, (uint32_t)((n_chunks - 1) & 1), 26, n_chunks - 1);
      tc_fence_after();
      if (warp >= 4) {
          flush_output(prev_tb, prev_nv, TM_O + 64u * (uint32_t)((n_chunks - 1) & 1), SM_KDEC);
        if (tid == 128) bulk_wait_all();
      }
    }
    const bool aborted = compute_sync_abort(&m.abort);
    if (!helper && !failed && !aborted && final_state) {
      const int n = lane_base + lane;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int c0 = 64 * hf + 32 * part;
        uint32_t r[32];
        tmem_ld32(tmem_addr(tm, lane_base, TM_S + c0), r);
        tmem_ld_wait(r);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          (transition ? final_state_m : final_state)[sbase + (int64_t)(c0 + j) * D + n] =
              __uint_as_float(r[j]);
      }
    }
    if (tid == 128) bulk_wait_all();  // no output store outlives the CTA, on any path
  }

  // ---- teardown (all warps)
  cta_sync();
  if (warp == kMmaWarp && lane == 0 && m.abort) {
    // Drain what is still in flight (bounded), so no copy or MMA outlives the CTA:
    // the MMAs, then the last phase that carried a copy on each copy barrier (a
    // barrier's phases complete in order).
    umma_commit(&m.bar_fin);
    mbar_wait(&m.bar_fin, 0, kWaitNs);
    uint64_t *bars[5] = {&m.bar_qk, &m.bar_la, &m.bar_v, &m.bar_pka, &m.bar_pkb};
    for (int i = 0; i < 5; ++i)
      if (m.last_copy[i]) mbar_wait(bars[i], (m.last_copy[i] - 1u) & 1u, kWaitNs);
    bulk_wait_all();
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

// order[r] = the sequence of rank r by length, longest first (ties by index).
// Lengths come from a device cu_seqlens that may be malformed: the ranks are a
// permutation of 0 .. n_seqs - 1 whatever the values.
__global__ void kda_seq_order_kernel(const int32_t *__restrict__ cu, int32_t n_seqs,
                                     int32_t *__restrict__ order) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n_seqs) return;
  const int64_t len = (int64_t)cu[s + 1] - cu[s];
  int rank = 0;
  for (int t = 0; t < n_seqs; ++t) {
    const int64_t lt = (int64_t)cu[t + 1] - cu[t];
    rank += (lt > len || (lt == len && t < s)) ? 1 : 0;
  }
  order[rank] = s;
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
  CUtensorMap mq, mk, mv, mla, mo, mom;
  memset(&mq, 0, sizeof(mq)); memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv)); memset(&mla, 0, sizeof(mla)); memset(&mo, 0, sizeof(mo));
  memset(&mom, 0, sizeof(mom));
  if (a.n_tokens > 0) {
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_map(&mq, a.q, bf, 2, a.n_tokens, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mk, a.k, bf, 2, a.n_tokens, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mv, a.v, bf, 2, a.n_tokens, a.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mla, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.n_tokens, a.H, 128,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mo, a.out, bf, 2, a.n_tokens, a.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        (a.out_m && !make_map(&mom, a.out_m, bf, 2, a.n_tokens, a.H, 128,
                              CU_TENSOR_MAP_SWIZZLE_NONE)))
      return cudaErrorInvalidValue;
  }
  HelpRing help;
  memset(&help, 0, sizeof(help));
  int32_t n_help = 0;
  if (a.mode == ChunkArgs::kPlain && a.help_ws && a.n_help > 0 && a.n_tokens > 0 && a.n_seqs <= kHelpMaxSeqs) {
    int32_t *hdr = reinterpret_cast<int32_t *>(a.help_ws);
    help.cons_pos = hdr;
    help.next_claim = hdr + chains;
    help.flag = hdr + 2 * chains;
    help.busy = hdr + (2 + kHelpSlots) * chains;
    help.finished = hdr + (2 + 2 * kHelpSlots) * chains;
    help.ring = a.help_ws + help_header_bytes(chains);
    help.n_chains = (int32_t)chains;
    n_help = a.n_help;
  }
  const bool transitions = a.mode == ChunkArgs::kTransitions;
  if (transitions) n_help = 0;
  if (transitions && (!a.final_state || !a.final_state_m)) return cudaErrorInvalidValue;
  auto kernel = transitions ? kda_chunk_fwd_tc_kernel<kModeTransitions>
                : n_help > 0 ? kda_chunk_fwd_tc_kernel<kModeHelp>
                             : kda_chunk_fwd_tc_kernel<kModePlain>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // The setmaxnreg split assumes the launch allocation it was sized for; with a
  // smaller one the compute warpgroups' .inc could never be satisfied.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  if ((uint32_t)fa.numRegs < kLaunchRegs) return cudaErrorNotSupported;
  // longest sequences first (plain launches of more than one sequence)
  const int32_t *seq_order = nullptr;
  if (a.seq_order && a.n_seqs > 1 && !transitions && n_help == 0) {
    kda_seq_order_kernel<<<(a.n_seqs + 255) / 256, 256, 0, stream>>>(a.cu_seqlens, a.n_seqs,
                                                                     a.seq_order);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    seq_order = a.seq_order;
  }
  const int64_t m_runs = a.split_skip_k >= 2 ? chains / a.split_skip_k * (a.split_skip_k - 1) : chains;
  const int64_t blocks = transitions ? chains + m_runs : chains + n_help;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  kernel<<<(unsigned)blocks, kThreads, SMEM_BYTES, stream>>>(
      mq, mk, mv, mla, mo, a.beta, a.init_state, a.cu_seqlens, a.n_seqs, a.n_tokens, a.H,
      static_cast<__nv_bfloat16 *>(a.out), a.final_state, a.status, help, a.final_state_m,
      seq_order, transitions && a.out_m ? mom : mo,
      static_cast<__nv_bfloat16 *>(transitions && a.out_m ? a.out_m : a.out),
      transitions ? (a.write_out ? 1 : 0) : 1, transitions ? a.split_skip_k : 0,
      (!transitions && n_help == 0) ? a.test_control : nullptr);
  return cudaGetLastError();
}

}  // namespace kda
