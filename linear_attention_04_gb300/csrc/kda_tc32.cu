// kda_tc32.cu -- tcgen05/TMEM path of the KDA chunked forward pass with the
// state recurrence stepped over 32-token super-chunks (bf16 q, k, v, theta,
// beta; dk = dv = 128; fp32 state; fp32 or bf16 out).
//
// The operation ("Kimi K3 Deep Dive", section "Core Innovation 1"):
//   S_t = (I - b_t k_t k_t^T) Diag(e^{g_t}) S_{t-1} + b_t k_t v_t^T,  o_t = S_t^T q_t,
// with the bounded log-decay g_t = g_min * sigmoid(theta_t) ("Architecture Deep
// Dive ...", sec. 3.2 eq. 1; "Kimi K3 Deep Dive", section "The Design").
//
// Chunking.  The pages' unit is the 16-token chunk: with g >= g_min = -5, no
// decay factor measured from a point inside or at the edge of a 16-token chunk
// exceeds e^{80}, finite in bf16 and fp32 ("Kimi K3 Deep Dive", sections "The
// Problem" and "The Design").  Here two consecutive 16-token chunks form one
// 32-token super-chunk whose decay factors are all anchored at the boundary
// between the two chunks: every token lies at most 16 tokens from that
// anchor, so every factor stays within [e^{-80}, e^{80}] and the whole 32 x 32
// decayed Gram tile of the super-chunk -- both chunks' diagonal tiles and the
// tile between them -- is ONE dense tensor-core product, with no
// position-by-position path.  The state S then advances once per 32 tokens.
//
// Per super-chunk (Gam = cumulative log-decay from the super-chunk start,
// mid = Gam at the anchor (after token 15), end = Gam after token 31):
//   LK = K e^{Gam-mid}, LQ = Q e^{Gam-mid}, R = K e^{mid-Gam}     (|factors| <= e^{80})
//   A  = strict_lower(Diag(b) LK R^T)   P = strict_lower(LQ R^T)   [= the decayed
//        K K^T and Q K^T tiles: (LK R^T)_{rs} = sum_c k_rc k_sc e^{Gam_rc - Gam_sc}]
//   T  = (I + A)^{-1},  Tb = T Diag(b)
//   Kt = K e^{Gam}, Qt = Q e^{Gam}, KhC = K e^{end-Gam}              (all <= 1)
//   W  = Tb Kt,  U = Tb V - W S,  O = Qt S + P U + Diag(q_t . k_t) U
//   S <- Diag(e^{end}) S + KhC^T U
// (the chunk-parallel WY form of the recurrence; the diagonal of Qt Kh^T is
// q_t . k_t exactly, applied in fp32).
//
// Precision plan (each choice measured against the fp64 oracle): the Gram tile
// in tf32 (operands rounded to 10-bit mantissas, not bf16's 7), P and U as
// bf16 high/low pairs in P U and U's low part in the state update, KhC as a
// high/low pair in the last update (the returned state), everything else bf16
// operands with fp32 accumulation; optionally (kSplitS) S^T as a high/low pair
// in the read-out products too.
//
// Warp roles (512 threads, four warpgroups; one CTA per (sequence, head)):
//   warps 0..3   state group: thread = value channel dv (TMEM lane).  The fp32
//                state row S^T[dv][0..127] lives in registers for the whole
//                sequence.  Thread 0 issues the chain's products
//                  [U | O] += S^T [-W | Qt]^T             (M=128, N=64, K=128)
//                  dS^T     = U^T KhC  (U high and low)  (M=128, N=128, K=32)
//                and the group turns U into its high/low pair, folds
//                S <- S e^{end} + dS in fp32 and writes the bf16 copy of S^T
//                (the next A operand) into TMEM.  Nothing else sits on this
//                sequential path.
//   warps 4..7   gate group: the gate and cumulative sums in fp32, every
//                decayed operand, V^T into TMEM, the q.k diagonal; warp 5
//                issues the Gram product [LK; LQ] R^T as a tf32 tcgen05.mma
//                (M = 128, N = 32, K = 128).
//   warps 8..11  solver group: TMA producer (warp 11, two super-chunks ahead,
//                plus L2 prefetch further on); reads A and P from TMEM,
//                inverts I + A in fp32 (two 16 x 16 forward substitutions and
//                the coupling tile), writes Tb and P as a high/low pair,
//                issues W^T = Kt^T Tb^T (M = 128, N = 32, K = 32), writes -W,
//                and issues [U' | 0] = V^T [Tb | 0]^T (N = 64, K = 32), the
//                start of the state group's accumulator.
//   warps 12..15 output group: issues O += U^T P^T (U and P high/low, N = 32,
//                K = 32) and stores the outputs O + (q.k) U.
// The gate and solver groups run up to two super-chunks ahead of the state
// group (double-buffered operand sets), the output group one behind it.
//
// Every wait is bounded: a wait that runs out sets the CTA's abort flag and the
// device status word (KDA_ERR_DEVICE_TIMEOUT); every role then leaves its loop,
// outstanding TMA loads and MMAs are drained and the TMEM is released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kda_device.cuh"
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int C = kChunk;      // 16: the pages' chunk (decay-bound unit)
constexpr int CS = 2 * C;      // 32: tokens per state step
constexpr int D = 128;         // dk = dv
constexpr int kThreads = 512;  // four warpgroups
constexpr int NST = 2;         // TMA ring stages (one super-chunk each)
constexpr int kPrefetch = 4;   // super-chunks prefetched into L2 beyond the ring
constexpr int NDQ = 4;         // q.k ring slots (gate group -> output group)
constexpr uint64_t kWaitNs = 2000000000ull;  // default limit of every wait: 2 s
// e^x is evaluated as 2^(x log2 e) with the hardware base-2 exponential: the
// gate works in the log2 domain throughout (G2 = G * log2 e).
constexpr float kLog2e = 1.4426950408889634f;

// Registers per thread of each warpgroup after setmaxnreg (launch: 128).  The
// sum over the four groups must not exceed the launch allocation; the host
// checks the compiled launch count before the first launch.
constexpr int kLaunchRegs = 128;
constexpr int kStateRegs = 184, kGateRegs = 160, kSolverRegs = 104, kOutRegs = 64;
static_assert((kStateRegs + kGateRegs + kSolverRegs + kOutRegs) * 128 <= kLaunchRegs * kThreads,
              "register split exceeds the launch allocation");

// ---------------------------------------------------------------- tensor memory (512 columns)
constexpr uint32_t TM_X = 0;       // 2 buffers x [U (32) | O (32)] fp32; U becomes bf16 hi|lo in place
constexpr uint32_t TM_DS = 128;    // dS^T fp32, 128 columns
constexpr uint32_t TM_SHI = 256;   // bf16 S^T high part (A operand), 64 columns
constexpr uint32_t TM_SLO = 320;   // bf16 S^T low part, 64 columns
constexpr uint32_t TM_GRAM = 384;  // [LK; LQ] R^T fp32, 32 columns (lanes 0..63)
constexpr uint32_t TM_WT = 416;    // W^T fp32, 32 columns
constexpr uint32_t TM_VT = 448;    // 2 buffers x 16 columns of bf16 V^T (A operand)
constexpr uint32_t TM_COLS = 512;
static_assert(TM_VT + 32 <= TM_COLS, "tensor memory budget");
// U in its buffer after the conversion, per 16-token K step kk: high part in
// columns 16 kk .. 16 kk + 7, low part in 16 kk + 8 .. 16 kk + 15.

// ---------------------------------------------------------------- shared memory (1024-aligned base)
constexpr uint32_t TILE = CS * D * 2;                // 8192: a 32 x 128 bf16 tile
constexpr uint32_t STAGE = 4 * TILE;                 // q, k, theta, v of one super-chunk (TMA)
constexpr uint32_t SM_RING = 0;
constexpr uint32_t SM_GL = SM_RING + NST * STAGE;    // [LK; LQ] fp32, SW128, 4 atoms x 64 rows x 128 B
constexpr uint32_t GL_ATOM = 64 * 128;
constexpr uint32_t SM_GR = SM_GL + 4 * GL_ATOM;      // R fp32, SW128, 4 atoms x 32 rows x 128 B
constexpr uint32_t GR_ATOM = 32 * 128;               // (also absorbs the M = 128 reads of GL's atom 3)
constexpr uint32_t SM_KT = SM_GR + 4 * GR_ATOM;      // 2 x Kt^T [128 dk x 32 tok] bf16, no swizzle
constexpr uint32_t KT_BYTES = D * CS * 2;            // 8192
constexpr uint32_t SM_KCL = SM_KT + 2 * KT_BYTES;    // KhC^T low part (last super-chunk only)
constexpr uint32_t SM_CH = SM_KCL + KT_BYTES;        // 2 operand sets
// operand set (offsets inside one set)
constexpr uint32_t CH_BX = 0;                        // [-W; Qt] [64 x 128] bf16, SW128, 2 atoms x 8 KB
constexpr uint32_t CH_KC = CH_BX + 2 * 64 * 128;     // KhC^T [128 x 32] bf16, no swizzle
constexpr uint32_t CH_TB = CH_KC + KT_BYTES;         // [Tb; 0] [64 x 32] bf16, no swizzle
constexpr uint32_t CH_PH = CH_TB + 64 * CS * 2;      // P high [32 x 32] bf16, no swizzle
constexpr uint32_t CH_PL = CH_PH + CS * CS * 2;      // P low
constexpr uint32_t CH_EG = CH_PL + CS * CS * 2;      // e^{end} fp32 [128]
constexpr uint32_t CH_BYTES = (CH_EG + D * 4 + 1023) / 1024 * 1024;
constexpr uint32_t SM_DQ = SM_CH + 2 * CH_BYTES;     // NDQ x q.k partial sums fp32 [4 warps][16 tokens]
constexpr uint32_t DQ_BYTES = 4 * C * 4;
constexpr uint32_t SM_AF = SM_DQ + NDQ * DQ_BYTES;   // A (b-scaled) fp32 [32][33]
constexpr uint32_t AF_LD = 33;
constexpr uint32_t SM_TF = SM_AF + CS * AF_LD * 4;   // T fp32 [32][33]
constexpr uint32_t SM_X10 = SM_TF + CS * AF_LD * 4;  // A10 T00 fp32 [16][17]
constexpr uint32_t SM_BETA = SM_X10 + C * 17 * 4;    // beta fp32 [32]
constexpr uint32_t SM_XCH = SM_BETA + CS * 4;        // chunk totals: 2 halves x 64 channel pairs x f32x2
constexpr uint32_t SM_BARS = SM_XCH + 2 * 64 * 8;
// barrier indices
constexpr int B_FULL = 0;         // [NST] TMA -> gate group
constexpr int B_EMPTY = 2;        // [NST] gate group has read the stage -> producer
constexpr int B_GRAM = 4;         // Gram product done (commit) -> solver, gate
constexpr int B_GREAD = 5;        // solver has read the Gram accumulator (2 arrivals)
constexpr int B_WDONE = 6;        // W^T product done (commit) -> solver
constexpr int B_UP = 7;           // [2] [U' | 0] product done (commit) -> state
constexpr int B_READY = 9;        // [2] operand set complete (gate + solver: 2 arrivals)
constexpr int B_X = 11;           // [U | O] products done -> state
constexpr int B_DS = 12;          // dS product done -> state
constexpr int B_UCONV = 13;       // U high/low written -> output group
constexpr int B_PU = 14;          // P U product done -> output group
constexpr int B_FREE = 15;        // [2] operand set consumed: state commit + state arrive +
                                  //     output commit + solver commit (4 arrivals)
constexpr int B_XFREE = 17;       // [2] output group has read X buffer b -> solver (U' of b + 2)
constexpr int B_DQFREE = 19;      // [NDQ] output group has read q.k slot -> gate
constexpr int B_DRAIN = 23;       // [4] final drains of the four issuers
constexpr int NBARS = 27;
constexpr uint32_t SM_MISC = SM_BARS + NBARS * 8;  // tmem base, abort flag, job flags
constexpr uint32_t SM_RANK = SM_MISC + 16;         // chain-order scratch
constexpr uint32_t SM_TOTAL = SM_RANK + (kMaxRankedSeqsDev + 1) * 4;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;   // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(SM_GL % 1024 == 0 && SM_GR % 1024 == 0 && SM_CH % 1024 == 0 && CH_BYTES % 1024 == 0,
              "SW128 tiles must be 1024-aligned");

// named barriers (id 0 is __syncthreads)
constexpr uint32_t NB_STATE = 1, NB_GATE = 2, NB_SOLVER = 3, NB_OUT = 4;

// Byte offset of (row, col) in a K-major SW128 tile of bf16 with `rows` rows:
// 64 channels per 128-byte row, 16-byte chunks XOR-swizzled by (row & 7).
__device__ __forceinline__ uint32_t sw128_bf16(int row, int col, int rows) {
  return (uint32_t)((col >> 6) * rows * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                    (col & 7) * 2);
}
// Same for fp32 (tf32 operands): 32 channels per 128-byte row.
__device__ __forceinline__ uint32_t sw128_f32(int row, int col, int rows) {
  return (uint32_t)((col >> 5) * rows * 128 + row * 128 + ((((col & 31) >> 2) ^ (row & 7)) << 4) +
                    (col & 3) * 4);
}
// Byte offset of (row, k) in a K-major tile without swizzle made of 8 x 16-byte
// core matrices: 8-row groups 128 B apart, 8-element K groups `kstride` apart.
__device__ __forceinline__ uint32_t core_off(int row, int k, uint32_t kstride) {
  return (uint32_t)((k >> 3) * kstride + (row >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// tcgen05.mma instruction descriptor, kind::tf32: fp32 accumulator, tf32 A and
// B (both K-major), M x N.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
KDA_DEV void mma_ss_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// fp32 -> tf32 with round-to-nearest (ties away from zero), kept in an fp32
// container with the low 13 mantissa bits zero.  The tf32 product reads only
// the top 19 bits of each operand (the rest is dropped, i.e. truncated), so
// the operands are rounded here first.
KDA_DEV f32x2 tf32_rna2(f32x2 v) {
  uint32_t a, b;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(a) : "f"(f2lo(v)));
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(b) : "f"(f2hi(v)));
  return (uint64_t)a | ((uint64_t)b << 32);
}
KDA_DEV void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   (uint64_t)map),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

template <int N>
__device__ __forceinline__ void set_regs() {
  if constexpr (N > kLaunchRegs)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
  else if constexpr (N < kLaunchRegs)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

struct Tc32Args {
  const SegJob* jobs;  // per-CTA work units (segmented launches), or null
  uint64_t wait_ns;    // limit of every bounded wait
  const __nv_bfloat16* beta;
  float g_min;
  int gate;
  const float* init_state;
  void* out;
  float* final_state;
  const int32_t* cu_seqlens;
  int N, H, T;
  int* status;
  float* dbg;          // stage dump of the first CTA (test hook), or null
  int dbg_nsc;         // super-chunks dumped
};

// Stage dump layout per super-chunk (floats): A [32][32] (beta-scaled, strictly
// lower), P [32][32] (strictly lower), T [32][32], W [32][128], U [32][128],
// e^{end} [128], q.k [32].
constexpr int DBG_A = 0, DBG_P = 1024, DBG_T = 2048, DBG_W = 3072, DBG_U = 3072 + 4096,
              DBG_EG = 3072 + 8192, DBG_QK = DBG_EG + 128, DBG_STRIDE = DBG_QK + 32;
static_assert(DBG_STRIDE == kTc32DumpFloats, "stage dump layout");

// Optional event trace of the first CTA (compile with -DKDA_TRACE): wall-clock
// time of each pipeline event per super-chunk, read back with
// kda_debug_trace_read_tc32.
constexpr int kTraceUnits = 256;
#ifdef KDA_TRACE
__device__ unsigned long long g_kda_trace_tc32[kTraceUnits * 32];
#define KTRACE(n, k)                                                                                \
  do {                                                                                              \
    if (blockIdx.x == 0 && (n) < kTraceUnits) g_kda_trace_tc32[(n) * 32 + (k)] = globaltimer_ns(); \
  } while (0)
#else
#define KTRACE(n, k) \
  do {               \
  } while (0)
#endif

__device__ __forceinline__ void fail(volatile int* abort, int* status) {
  *abort = 1;
  atomicExch(status, KDA_ERR_DEVICE_TIMEOUT);
}

__device__ __forceinline__ uint32_t tm_lane(int q4) { return (uint32_t)(q4 * 32) << 16; }

// bf16 high/low pair of two fp32 values: hi = bf16(x), lo = bf16(x - hi)
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(x0, x1);
  const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&hi);
  lo = pack_bf16x2(x0 - __low2float(hb), x1 - __high2float(hb));
}

template <bool kOutBf16, bool kSplitS>
__global__ void __launch_bounds__(kThreads, 1)
    kda_fwd_tc32_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_th,
                        const __grid_constant__ CUtensorMap tm_v, const Tc32Args args) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // keep the pointer arithmetic on the shared array itself (shared address space)
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = (uint64_t*)(sm + SM_BARS);
  uint32_t* tmem_slot = (uint32_t*)(sm + SM_MISC);
  volatile int* abort = (volatile int*)(sm + SM_MISC + 4);
  volatile int* sflags = (volatile int*)(sm + SM_MISC + 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(sm);

  // the work unit: a whole (sequence, head) chain, or one segment job
  Chain ch;
  int flags = 0;
  const float* init_state = args.init_state;
  float* final_state = args.final_state;
  int64_t soff = 0;  // element offset of this chain's state in init/final
  if (args.jobs) {
    const SegJob jb = args.jobs[blockIdx.x];
    ch.seq = 0;
    ch.head = jb.head;
    ch.t0 = jb.t0;
    ch.t1 = jb.t1;
    flags = jb.flags;
    init_state = jb.init;
    final_state = jb.final_state;
  } else {
    ch = chain_for_block(blockIdx.x, args.H, args.N, args.T, args.cu_seqlens, (int*)(sm + SM_RANK));
    if (!ch.valid) {
      // malformed packing table: report it and store nothing
      if (tid == 0) atomicExch(args.status, KDA_ERR_BAD_SEQLENS);
      return;
    }
    soff = ((int64_t)ch.seq * args.H + ch.head) * D * D;
  }
  const int h = ch.head;
  const int H = args.H;
  const int L = (int)(ch.t1 - ch.t0);
  const int nsc = (L + CS - 1) / CS;  // 32-token super-chunks
  float* dbg = (args.dbg && blockIdx.x == 0) ? args.dbg : nullptr;

  if (tid == 0) {
    for (int i = 0; i < NBARS; ++i) {
      uint32_t cnt = 1;
      if (i == B_GREAD || i == B_READY || i == B_READY + 1) cnt = 2;
      if (i == B_FREE || i == B_FREE + 1) cnt = 4;
      mbar_init(&bars[i], cnt);
    }
    *abort = 0;
    *sflags = flags;
    fence_mbar_init();
  }
  // the zero half of both [Tb; 0] tiles: rows 32..63 are bytes [512, 1024) of
  // every 1024-byte K group
  for (int e = tid; e < 2 * 4 * 128; e += kThreads) {
    const int set = e >> 9, kg = (e >> 7) & 3, w = e & 127;
    *(uint32_t*)(sm + SM_CH + set * CH_BYTES + CH_TB + kg * 1024 + 512 + w * 4) = 0u;
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_slot, TM_COLS);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 12) {
    // ================================================================ output group
    set_regs<kOutRegs>();
    const int q4 = warp & 3;
    const int dv = 32 * q4 + lane;
    const bool issuer = tid == 384;
    const bool no_out = *sflags & kJobNoOut;
    bool bad = false;
    for (int n = 0; n < nsc; ++n) {
      const int b = n & 1;
      const uint32_t css = sbase + SM_CH + b * CH_BYTES;
      const uint32_t ua = tmem + TM_X + 64 * b;  // U (high/low per K step), O at + 32
      if (issuer) {
        // O += U^T P^T once U's high/low pair is written
        const bool ok = mbar_wait(&bars[B_UCONV], n & 1, abort, args.wait_ns);
        tc_fence_after();
        if (ok) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t ph = sdesc_noswz(css + CH_PH + kk * 1024, 512, 128);
            const uint64_t pl = sdesc_noswz(css + CH_PL + kk * 1024, 512, 128);
            mma_ts(ua + 32, ua + 16 * kk, ph, idesc_bf16_f32(128, 32), 1);
            mma_ts(ua + 32, ua + 16 * kk + 8, ph, idesc_bf16_f32(128, 32), 1);
            mma_ts(ua + 32, ua + 16 * kk, pl, idesc_bf16_f32(128, 32), 1);
          }
          mma_commit(&bars[B_PU]);
          mma_commit(&bars[B_FREE + b]);
        } else {
          bad = true;
        }
      }
      bad |= !__all_sync(0xffffffffu, mbar_wait(&bars[B_PU], n & 1, abort, args.wait_ns));
      if (bar_sync_or(NB_OUT, 128, bad || *abort)) {
        bad = true;
        break;
      }
      if (issuer) KTRACE(n, 5);
      tc_fence_after();
      // ---- outputs of super-chunk n: O + (q.k) U, U = high + low, 16 tokens at a time
      const float* dqp = (const float*)(sm + SM_DQ + (n % NDQ) * DQ_BYTES);
      const int nvalid = no_out ? 0 : min(CS, L - n * CS);
      const int64_t row0 = ch.t0 + (int64_t)n * CS;
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        uint32_t o[16], u[16];
        tmem_ld_x16(tmem + tm_lane(q4) + TM_X + 64 * b + 32 + 16 * hc, o);
        tmem_ld_x16(tmem + tm_lane(q4) + TM_X + 64 * b + 16 * hc, u);
        tmem_wait_ld();
        if (issuer && hc == 0) KTRACE(n, 24);
        if (issuer && hc == 1) KTRACE(n, 25);
#pragma unroll
        for (int tt = 0; tt < C; ++tt) {
          const int t = C * hc + tt;
          const uint32_t hw = u[tt >> 1], lw = u[8 + (tt >> 1)];
          const float uh = __uint_as_float((tt & 1) ? (hw & 0xffff0000u) : (hw << 16));
          const float ul = __uint_as_float((tt & 1) ? (lw & 0xffff0000u) : (lw << 16));
          const float qk = dqp[(2 * hc) * C + tt] + dqp[(2 * hc + 1) * C + tt];
          const float val = __uint_as_float(o[tt]) + qk * (uh + ul);
          if (t < nvalid) {
            const int64_t idx = ((row0 + t) * H + h) * D + dv;
            if constexpr (kOutBf16)
              ((__nv_bfloat16*)args.out)[idx] = __float2bfloat16_rn(val);
            else
              ((float*)args.out)[idx] = val;
          }
          if (dbg && n < args.dbg_nsc && dv == 0) dbg[n * DBG_STRIDE + DBG_QK + t] = qk;
        }
      }
      tc_fence_before();
      if (bar_sync_or(NB_OUT, 128, bad || *abort)) {
        bad = true;
        break;
      }
      if (issuer) {
        KTRACE(n, 6);
        mbar_arrive(&bars[B_XFREE + b]);
        mbar_arrive(&bars[B_DQFREE + n % NDQ]);
      }
    }
    if (bad) fail(abort, args.status);
    if (issuer) {
      mma_commit(&bars[B_DRAIN + 3]);
      mbar_wait_drain(&bars[B_DRAIN + 3], 0, args.wait_ns);
    }
  } else if (warp >= 8) {
    // ================================================================ solver group
    set_regs<kSolverRegs>();
    const int vt = tid - 256, q4 = warp & 3;
    const bool issuer = vt == 0;
    const bool producer = vt == 96;  // warp 11, lane 0
    const bool zero_v = *sflags & kJobZeroV;
    float* Af = (float*)(sm + SM_AF);
    float* Tf = (float*)(sm + SM_TF);
    float* X10 = (float*)(sm + SM_X10);
    float* betas = (float*)(sm + SM_BETA);
    auto load = [&](int m) {
      const int s = m % NST;
      mbar_arrive_expect_tx(&bars[B_FULL + s], zero_v ? 3 * TILE : STAGE);
      unsigned char* st = sm + SM_RING + s * STAGE;
      const int row = (int)(ch.t0 + (int64_t)m * CS);
      tma_load_3d(st + 0 * TILE, &tm_q, 0, h, row, &bars[B_FULL + s]);
      tma_load_3d(st + 1 * TILE, &tm_k, 0, h, row, &bars[B_FULL + s]);
      tma_load_3d(st + 2 * TILE, &tm_th, 0, h, row, &bars[B_FULL + s]);
      if (!zero_v) tma_load_3d(st + 3 * TILE, &tm_v, 0, h, row, &bars[B_FULL + s]);
    };
    auto prefetch = [&](int m) {
      const int row = (int)(ch.t0 + (int64_t)m * CS);
      tma_prefetch_3d(&tm_q, 0, h, row);
      tma_prefetch_3d(&tm_k, 0, h, row);
      tma_prefetch_3d(&tm_th, 0, h, row);
      if (!zero_v) tma_prefetch_3d(&tm_v, 0, h, row);
    };
    int issued = 0;  // super-chunks loaded so far (the producer's count)
    if (producer && nsc > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_th);
      prefetch_tmap(&tm_v);
      for (; issued < NST && issued < nsc; ++issued) load(issued);
      for (int m = NST; m < NST + kPrefetch && m < nsc; ++m) prefetch(m);
    }
    bool bad = false;
    for (int n = 0; n < nsc; ++n) {
      const int b = n & 1;
      unsigned char* cs = sm + SM_CH + b * CH_BYTES;
      const uint32_t css = sbase + SM_CH + b * CH_BYTES;
      const int nvalid = min(CS, L - n * CS);
      if (producer && n + NST < nsc) {
        // the gate group has read super-chunk n's stage: load n + NST into it
        if (mbar_wait(&bars[B_EMPTY + n % NST], (n / NST) & 1, abort, args.wait_ns)) {
          load(n + NST);
          issued = n + NST + 1;
          if (n + NST + kPrefetch < nsc) prefetch(n + NST + kPrefetch);
        } else {
          bad = true;
        }
      }
      // beta of the super-chunk, issued before the waits
      float beta_l = 0.0f;
      if (q4 == 0 && lane < nvalid)
        beta_l = __bfloat162float(args.beta[(ch.t0 + (int64_t)n * CS + lane) * H + h]);
      bad |= !__all_sync(0xffffffffu, mbar_wait(&bars[B_GRAM], n & 1, abort, args.wait_ns));
      if (issuer) KTRACE(n, 11);
      if (n >= 2)
        bad |= !__all_sync(0xffffffffu,
                           mbar_wait(&bars[B_FREE + b], ((n >> 1) - 1) & 1, abort, args.wait_ns));
      tc_fence_after();
      if (q4 <= 1) {
        // lanes 0..31 of the Gram accumulator hold the LK rows (-> A), lanes
        // 32..63 the LQ rows (-> P)
        uint32_t raw[32];
        tmem_ld_x32(tmem + tm_lane(q4) + TM_GRAM, raw);
        tmem_wait_ld();
        if (issuer) KTRACE(n, 26);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_GREAD]);
        const int r = lane;
        if (q4 == 0) {
          betas[r] = beta_l;
#pragma unroll
          for (int s = 0; s < CS; ++s) Af[r * AF_LD + s] = (s < r) ? beta_l * __uint_as_float(raw[s]) : 0.0f;
          if (dbg && n < args.dbg_nsc) {
#pragma unroll
            for (int s = 0; s < CS; ++s) dbg[n * DBG_STRIDE + DBG_A + r * CS + s] = Af[r * AF_LD + s];
          }
        } else {
          // strictly lower P as a bf16 high/low pair; the diagonal q_t . k_t is
          // applied exactly by the output group
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const int s0 = 8 * c8 + 2 * p;
              const float x0 = s0 < r ? __uint_as_float(raw[s0]) : 0.0f;
              const float x1 = s0 + 1 < r ? __uint_as_float(raw[s0 + 1]) : 0.0f;
              split_pair(x0, x1, hi[p], lo[p]);
              if (dbg && n < args.dbg_nsc) {
                dbg[n * DBG_STRIDE + DBG_P + r * CS + s0] = x0;
                dbg[n * DBG_STRIDE + DBG_P + r * CS + s0 + 1] = x1;
              }
            }
            *(uint4*)(cs + CH_PH + core_off(r, 8 * c8, 512)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *(uint4*)(cs + CH_PL + core_off(r, 8 * c8, 512)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
      }
      if (bar_sync_or(NB_SOLVER, 128, bad || *abort)) {
        bad = true;
        break;
      }
      if (issuer) KTRACE(n, 28);
      // ---- T = (I + A)^{-1}: the two 16 x 16 diagonal blocks by forward
      // substitution (lane j < 16: column j of T00; lane 16 + j: column j of T11)
      if (q4 == 0) {
        const int j = lane & 15, off = lane & 16;
        float t[C];
#pragma unroll
        for (int i = 0; i < C; ++i) t[i] = (i == j) ? 1.0f : 0.0f;
#pragma unroll
        for (int i = 1; i < C; ++i) {
          float acc0 = 0.0f, acc1 = 0.0f;
          const float* arow = Af + (off + i) * AF_LD + off;
#pragma unroll
          for (int m = 0; m < i; m += 2) {
            acc0 = fmaf(arow[m], t[m], acc0);
            if (m + 1 < i) acc1 = fmaf(arow[m + 1], t[m + 1], acc1);
          }
          if (i > j) t[i] = -(acc0 + acc1);
        }
#pragma unroll
        for (int i = 0; i < C; ++i) Tf[(off + i) * AF_LD + off + j] = t[i];
        if (issuer) KTRACE(n, 27);
      }
      if (bar_sync_or(NB_SOLVER, 128, bad || *abort)) {
        bad = true;
        break;
      }
      if (issuer) KTRACE(n, 12);
      // ---- coupling tile T10 = -T11 (A10 T00): thread -> row i, columns j0, j0+1
      {
        const int i = vt >> 3, j0 = (vt & 7) * 2;
        float x0 = 0.0f, x1 = 0.0f;
#pragma unroll
        for (int m = 0; m < C; ++m) {
          const float a = Af[(C + i) * AF_LD + m];
          x0 = fmaf(a, Tf[m * AF_LD + j0], x0);
          x1 = fmaf(a, Tf[m * AF_LD + j0 + 1], x1);
        }
        X10[i * 17 + j0] = x0;
        X10[i * 17 + j0 + 1] = x1;
      }
      if (bar_sync_or(NB_SOLVER, 128, bad || *abort)) {
        bad = true;
        break;
      }
      {
        const int i = vt >> 3, j0 = (vt & 7) * 2;
        float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
        for (int m = 0; m < C; ++m) {
          const float tt = (m <= i) ? Tf[(C + i) * AF_LD + C + m] : 0.0f;
          y0 = fmaf(tt, X10[m * 17 + j0], y0);
          y1 = fmaf(tt, X10[m * 17 + j0 + 1], y1);
        }
        Tf[(C + i) * AF_LD + j0] = -y0;
        Tf[(C + i) * AF_LD + j0 + 1] = -y1;
      }
      if (bar_sync_or(NB_SOLVER, 128, bad || *abort)) {
        bad = true;
        break;
      }
      // ---- Tb = T Diag(beta) (bf16): thread -> row t, 8 columns
      {
        const int t = vt >> 2, c8 = vt & 3;
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int s0 = 8 * c8 + 2 * p;
          const float a0 = (s0 <= t) ? Tf[t * AF_LD + s0] * betas[s0] : 0.0f;
          const float a1 = (s0 + 1 <= t) ? Tf[t * AF_LD + s0 + 1] * betas[s0 + 1] : 0.0f;
          w[p] = pack_bf16x2(a0, a1);
          if (dbg && n < args.dbg_nsc) {
            dbg[n * DBG_STRIDE + DBG_T + t * CS + s0] = (s0 <= t) ? Tf[t * AF_LD + s0] : 0.0f;
            dbg[n * DBG_STRIDE + DBG_T + t * CS + s0 + 1] = (s0 + 1 <= t) ? Tf[t * AF_LD + s0 + 1] : 0.0f;
          }
        }
        *(uint4*)(cs + CH_TB + core_off(t, 8 * c8, 1024)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      if (bar_sync_or(NB_SOLVER, 128, bad || *abort)) {
        bad = true;
        break;
      }
      // ---- W^T = Kt^T Tb^T (M = 128 key channels, N = 32, K = 32), and the
      // start of the state group's accumulator [U' | 0] = V^T [Tb | 0]^T into X
      // buffer b once the output group has read that buffer's previous use
      if (issuer) {
        KTRACE(n, 13);
        tc_fence_after();
        const uint32_t kt = sbase + SM_KT + b * KT_BYTES;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          mma_ss(tmem + TM_WT, sdesc_noswz(kt + kk * 4096, 2048, 128),
                 sdesc_noswz(css + CH_TB + kk * 2048, 1024, 128), idesc_bf16_f32(128, 32), kk > 0);
        mma_commit(&bars[B_WDONE]);
        if (n < 2 || mbar_wait(&bars[B_XFREE + b], ((n >> 1) - 1) & 1, abort, args.wait_ns)) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_ts(tmem + TM_X + 64 * b, tmem + TM_VT + 16 * b + 8 * kk,
                   sdesc_noswz(css + CH_TB + kk * 2048, 1024, 128), idesc_bf16_f32(128, 64), kk > 0);
          mma_commit(&bars[B_UP + b]);
          mma_commit(&bars[B_FREE + b]);
        } else {
          bad = true;
        }
      }
      bad |= !__all_sync(0xffffffffu, mbar_wait(&bars[B_WDONE], n & 1, abort, args.wait_ns));
      if (issuer) KTRACE(n, 14);
      tc_fence_after();
      {
        // -W into rows 0..31 of the [-W; Qt] tile: thread = key channel dk
        const int dk = 32 * q4 + lane;
        uint32_t raw[32];
        tmem_ld_x32(tmem + tm_lane(q4) + TM_WT, raw);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < CS; ++t) {
          *(__nv_bfloat16*)(cs + CH_BX + sw128_bf16(t, dk, 64)) = __float2bfloat16_rn(-__uint_as_float(raw[t]));
          if (dbg && n < args.dbg_nsc) dbg[n * DBG_STRIDE + DBG_W + t * D + dk] = __uint_as_float(raw[t]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (bar_sync_or(NB_SOLVER, 128, bad || *abort)) {
        bad = true;
        break;
      }
      if (issuer) {
        mbar_arrive(&bars[B_READY + b]);
        KTRACE(n, 15);
      }
    }
    if (bad) fail(abort, args.status);
    if (issuer) {
      mma_commit(&bars[B_DRAIN + 2]);
      mbar_wait_drain(&bars[B_DRAIN + 2], 0, args.wait_ns);
    }
    if (producer) {
      // every load still in flight lands before the CTA releases its memory
      // (the latest load of each stage; a completed phase returns at once)
      for (int m = issued - NST > 0 ? issued - NST : 0; m < issued; ++m)
        mbar_wait_drain(&bars[B_FULL + m % NST], (m / NST) & 1, args.wait_ns);
    }
  } else if (warp >= 4) {
    // ================================================================ gate group
    set_regs<kGateRegs>();
    const int gt = tid - 128;
    const int hf = gt >> 6;        // chunk of the super-chunk: tokens 16 hf .. 16 hf + 15
    const int cp = gt & 63;        // channel pair: channels 2 cp, 2 cp + 1
    const int q4 = warp & 3;       // TMEM lane quarter (V^T)
    const bool arriver = gt == 0;  // stage release and operand hand-off
    const bool gram_issuer = gt == 32;  // warp 5, lane 0
    const bool zero_v = *sflags & kJobZeroV;
    const bool log_decay = args.gate == KDA_GATE_LOG_DECAY;
    f32x2* xch = (f32x2*)(sm + SM_XCH);
    const f32x2 kL2 = f2(kLog2e, kLog2e);
    const f32x2 kC2 = f2(-kLog2e, -kLog2e);
    const f32x2 kC1 = f2(args.g_min * kLog2e, args.g_min * kLog2e);
    const f32x2 kOne = f2(1.0f, 1.0f);
    const f32x2 kZero = 0ull;
    bool bad = false;
    for (int n = 0; n < nsc; ++n) {
      const int b = n & 1;
      unsigned char* cs = sm + SM_CH + b * CH_BYTES;
      const int nvalid = min(CS, L - n * CS);
      const bool last = n + 1 == nsc;
      unsigned char* st = sm + SM_RING + (n % NST) * STAGE;
      bad |= !__all_sync(0xffffffffu, mbar_wait(&bars[B_FULL + n % NST], (n / NST) & 1, abort, args.wait_ns));
      if (n >= 1)  // the Gram operands of the previous super-chunk have been consumed
        bad |= !__all_sync(0xffffffffu, mbar_wait(&bars[B_GRAM], (n - 1) & 1, abort, args.wait_ns));
      if (n >= 2)  // this operand set's previous contents have been consumed
        bad |= !__all_sync(0xffffffffu,
                           mbar_wait(&bars[B_FREE + b], ((n >> 1) - 1) & 1, abort, args.wait_ns));
      if (n >= NDQ)  // the q.k slot's previous contents have been read
        bad |= !__all_sync(0xffffffffu, mbar_wait(&bars[B_DQFREE + n % NDQ], ((n / NDQ) - 1) & 1,
                                                  abort, args.wait_ns));
      if (arriver) KTRACE(n, 7);
      if (nvalid < CS) {
        // rows past the end of the sequence become neutral: q = k = v = 0 and
        // g = 0 (theta = -inf for the sigmoid gate, 0 for a given log-decay)
        for (int e = gt; e < (CS - nvalid) * 16; e += 128) {
          const int row = nvalid + (e >> 4), c16 = e & 15;
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          const uint32_t tf = log_decay ? 0u : 0xff80ff80u;
          *(uint4*)(st + 0 * TILE + row * 256 + c16 * 16) = z;
          *(uint4*)(st + 1 * TILE + row * 256 + c16 * 16) = z;
          *(uint4*)(st + 2 * TILE + row * 256 + c16 * 16) = make_uint4(tf, tf, tf, tf);
          *(uint4*)(st + 3 * TILE + row * 256 + c16 * 16) = z;
        }
      }
      if (bar_sync_or(NB_GATE, 128, bad || *abort)) {
        bad = true;
        break;
      }
      // ---- gate and in-chunk cumulative sums (log2 domain), two channels per thread
      const uint32_t* sq = (const uint32_t*)(st + 0 * TILE) + C * hf * 64;
      const uint32_t* sk = (const uint32_t*)(st + 1 * TILE) + C * hf * 64;
      const uint32_t* sth = (const uint32_t*)(st + 2 * TILE) + C * hf * 64;
      f32x2 Gl[C];
      f32x2 G2 = kZero;
#pragma unroll
      for (int t = 0; t < C; ++t) {
        const f32x2 th = bf2_to_f2(sth[t * 64 + cp]);
        f32x2 g2;
        if (log_decay) {
          g2 = mul2(th, kL2);
        } else {
          const f32x2 x = mul2(th, kC2);
          const f32x2 d = add2(f2(ex2_approx(f2lo(x)), ex2_approx(f2hi(x))), kOne);
          g2 = mul2(f2(rcp_approx(f2lo(d)), rcp_approx(f2hi(d))), kC1);
        }
        G2 = add2(G2, g2);
        Gl[t] = G2;
      }
      xch[hf * 64 + cp] = G2;  // this chunk's total
      if (bar_sync_or(NB_GATE, 128, bad || *abort)) {
        bad = true;
        break;
      }
      if (arriver) KTRACE(n, 8);
      const f32x2 T0 = xch[cp], T1 = xch[64 + cp];  // totals of chunk 0 (= mid) and chunk 1
      // per-channel constants: e^{mid} and e^{end - mid}
      const f32x2 cM = f2(ex2_approx(f2lo(T0)), ex2_approx(f2hi(T0)));
      const f32x2 cE = f2(ex2_approx(f2lo(T1)), ex2_approx(f2hi(T1)));
      const f32x2 xoff = hf ? kZero : f2(-f2lo(T0), -f2hi(T0));  // Gam - mid = Gl + xoff
      uint32_t ktr[2][4], kcr[2][4], kcl[2][4];
      float dq[C];
#pragma unroll
      for (int t = 0; t < C; ++t) {
        const int r = C * hf + t;  // token row in the super-chunk
        const f32x2 x = add2(Gl[t], xoff);
        const f32x2 eL = f2(ex2_approx(f2lo(x)), ex2_approx(f2hi(x)));     // e^{Gam - mid}
        const f32x2 eR = f2(ex2_approx(-f2lo(x)), ex2_approx(-f2hi(x)));   // e^{mid - Gam}
        const f32x2 eG = mul2(eL, cM);                                      // e^{Gam}
        const f32x2 eK = mul2(eR, cE);                                      // e^{end - Gam}
        const f32x2 k = bf2_to_f2(sk[t * 64 + cp]), q = bf2_to_f2(sq[t * 64 + cp]);
        *(f32x2*)(sm + SM_GL + sw128_f32(r, 2 * cp, 64)) = tf32_rna2(mul2(k, eL));
        *(f32x2*)(sm + SM_GL + sw128_f32(CS + r, 2 * cp, 64)) = tf32_rna2(mul2(q, eL));
        *(f32x2*)(sm + SM_GR + sw128_f32(r, 2 * cp, 32)) = tf32_rna2(mul2(k, eR));
        *(uint32_t*)(cs + CH_BX + sw128_bf16(CS + r, 2 * cp, 64)) = f2_to_bf2(mul2(q, eG));
        const f32x2 kc = mul2(k, eK);
        const uint32_t ktw = f2_to_bf2(mul2(k, eG)), kcw = f2_to_bf2(kc);
        // transpose: gather 8 tokens of each channel into one 16-byte row
        const int p = (t & 7) >> 1;
        if (t & 1) {
          ktr[0][p] = __byte_perm(ktr[0][p], ktw, 0x5410);
          ktr[1][p] = __byte_perm(ktr[1][p], ktw, 0x7610);
          kcr[0][p] = __byte_perm(kcr[0][p], kcw, 0x5410);
          kcr[1][p] = __byte_perm(kcr[1][p], kcw, 0x7610);
        } else {
          ktr[0][p] = ktw & 0xffffu;
          ktr[1][p] = ktw >> 16;
          kcr[0][p] = kcw & 0xffffu;
          kcr[1][p] = kcw >> 16;
        }
        if (last) {
          const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&kcw);
          const uint32_t lw = pack_bf16x2(f2lo(kc) - __low2float(hb), f2hi(kc) - __high2float(hb));
          if (t & 1) {
            kcl[0][p] = __byte_perm(kcl[0][p], lw, 0x5410);
            kcl[1][p] = __byte_perm(kcl[1][p], lw, 0x7610);
          } else {
            kcl[0][p] = lw & 0xffffu;
            kcl[1][p] = lw >> 16;
          }
        }
        if ((t & 7) == 7) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t o = core_off(2 * cp + e, r - 7, 2048);
            *(uint4*)(sm + SM_KT + b * KT_BYTES + o) = make_uint4(ktr[e][0], ktr[e][1], ktr[e][2], ktr[e][3]);
            *(uint4*)(cs + CH_KC + o) = make_uint4(kcr[e][0], kcr[e][1], kcr[e][2], kcr[e][3]);
            if (last) *(uint4*)(sm + SM_KCL + o) = make_uint4(kcl[e][0], kcl[e][1], kcl[e][2], kcl[e][3]);
          }
        }
        const f32x2 qk = mul2(q, k);
        dq[t] = f2lo(qk) + f2hi(qk);
        if (arriver && t == 7) KTRACE(n, 16);
      }
      if (arriver) KTRACE(n, 17);
      if (hf == 0) {
        const f32x2 eE = mul2(cM, cE);  // e^{end}
        *(f32x2*)(cs + CH_EG + 8 * cp) = eE;
        if (dbg && n < args.dbg_nsc) {
          dbg[n * DBG_STRIDE + DBG_EG + 2 * cp] = f2lo(eE);
          dbg[n * DBG_STRIDE + DBG_EG + 2 * cp + 1] = f2hi(eE);
        }
      }
      {
        // q_t . k_t over this warp's 64 channels: transpose-reduce the 16
        // partial sums over the 32 lanes; lane l ends with token (l >> 1) & 15
        float v8[8], v4[4], v2[2], v1;
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          v8[j] = (b4 ? dq[j + 8] : dq[j]) + __shfl_xor_sync(0xffffffffu, b4 ? dq[j] : dq[j + 8], 16);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          v4[j] = (b3 ? v8[j + 4] : v8[j]) + __shfl_xor_sync(0xffffffffu, b3 ? v8[j] : v8[j + 4], 8);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          v2[j] = (b2 ? v4[j + 2] : v4[j]) + __shfl_xor_sync(0xffffffffu, b2 ? v4[j] : v4[j + 2], 4);
        v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        if ((lane & 1) == 0)
          ((float*)(sm + SM_DQ + (n % NDQ) * DQ_BYTES))[(warp - 4) * C + ((lane >> 1) & 15)] = v1;
      }
      if (arriver) KTRACE(n, 18);
      // ---- V^T into tensor memory: TMEM lane = value channel 32 q4 + lane,
      // 32 tokens packed two per 32-bit column
      {
        const int dv = 32 * q4 + lane;
        const unsigned short* sv = (const unsigned short*)(st + 3 * TILE);
        uint32_t w[16];
#pragma unroll
        for (int p = 0; p < 16; ++p) {
          const uint32_t v0 = (!zero_v && 2 * p < nvalid) ? (uint32_t)sv[(2 * p) * D + dv] : 0u;
          const uint32_t v1 = (!zero_v && 2 * p + 1 < nvalid) ? (uint32_t)sv[(2 * p + 1) * D + dv] : 0u;
          w[p] = v0 | (v1 << 16);
        }
        if (arriver) KTRACE(n, 19);
        tmem_st_x16(tmem + tm_lane(q4) + TM_VT + 16 * b, w);
        tmem_wait_st();
        if (arriver) KTRACE(n, 20);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (bar_sync_or(NB_GATE, 128, bad || *abort)) {
        bad = true;
        break;
      }
      if (arriver) {
        KTRACE(n, 9);
        mbar_arrive(&bars[B_EMPTY + n % NST]);  // the stage may be refilled
        // (a test job can withhold its first hand-off: the state group's
        // bounded wait then runs out and reports KDA_ERR_DEVICE_TIMEOUT)
        if (!(n == 0 && (*sflags & kJobTestWithholdFirst))) mbar_arrive(&bars[B_READY + b]);
      }
      if (gram_issuer) {
        // the Gram accumulator of the previous super-chunk has been read out
        if (n >= 1 && !mbar_wait(&bars[B_GREAD], (n - 1) & 1, abort, args.wait_ns)) bad = true;
        tc_fence_after();
        const uint32_t gl = sbase + SM_GL, gr = sbase + SM_GR;
#pragma unroll
        for (int kk = 0; kk < D / 8; ++kk)
          mma_ss_tf32(tmem + TM_GRAM, sdesc_sw128(gl + (kk >> 2) * GL_ATOM + (kk & 3) * 32),
                      sdesc_sw128(gr + (kk >> 2) * GR_ATOM + (kk & 3) * 32), idesc_tf32_f32(128, 32),
                      kk > 0);
        mma_commit(&bars[B_GRAM]);
        KTRACE(n, 10);
      }
    }
    if (bad) fail(abort, args.status);
    if (gram_issuer) {
      mma_commit(&bars[B_DRAIN + 1]);
      mbar_wait_drain(&bars[B_DRAIN + 1], 0, args.wait_ns);
    }
  } else {
    // ================================================================ state group
    set_regs<kStateRegs>();
    const int dv = tid;  // value channel = TMEM lane
    const uint32_t lb = tm_lane(warp);
    const bool issuer = tid == 0;
    const bool identity = flags & kJobIdentityInit;
    float S[D];  // S^T[dv][dk]
#pragma unroll
    for (int i = 0; i < D; ++i)
      S[i] = init_state ? init_state[soff + (int64_t)i * D + dv] : ((identity && i == dv) ? 1.0f : 0.0f);
    bool bad = false;
    // bf16 copy of S^T (high and, if split, low part) into TMEM
    auto write_sbf = [&](int blk) {
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int p = 0; p < 16; ++p) {
        if constexpr (kSplitS)
          split_pair(S[32 * blk + 2 * p], S[32 * blk + 2 * p + 1], hi[p], lo[p]);
        else
          hi[p] = pack_bf16x2(S[32 * blk + 2 * p], S[32 * blk + 2 * p + 1]);
      }
      tmem_st_x16(tmem + lb + TM_SHI + 16 * blk, hi);
      if constexpr (kSplitS) tmem_st_x16(tmem + lb + TM_SLO + 16 * blk, lo);
    };
    // [U | O] += S^T [-W | Qt]^T of super-chunk m into buffer m & 1, on top of
    // the [U' | 0] the solver group started there
    auto issue_x = [&](int m) -> bool {
      const int bb = m & 1;
      if (!mbar_wait(&bars[B_READY + bb], (m >> 1) & 1, abort, args.wait_ns)) return false;
      if (!mbar_wait(&bars[B_UP + bb], (m >> 1) & 1, abort, args.wait_ns)) return false;
      tc_fence_after();
      const uint32_t css = sbase + SM_CH + bb * CH_BYTES;
      const uint32_t dx = tmem + TM_X + 64 * bb;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t bx = sdesc_sw128(css + CH_BX + (kk >> 2) * 8192 + (kk & 3) * 32);
        mma_ts(dx, tmem + TM_SHI + 8 * kk, bx, idesc_bf16_f32(128, 64), 1);
        if constexpr (kSplitS) mma_ts(dx, tmem + TM_SLO + 8 * kk, bx, idesc_bf16_f32(128, 64), 1);
      }
      mma_commit(&bars[B_X]);
      return true;
    };
    if (nsc > 0) {
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) write_sbf(blk);
      tmem_wait_st();
      tc_fence_before();
      if (bar_sync_or(NB_STATE, 128, *abort)) bad = true;
      if (!bad && issuer && !issue_x(0)) fail(abort, args.status);
    }
    for (int n = 0; n < nsc && !bad; ++n) {
      const int b = n & 1;
      const bool last = n + 1 == nsc;
      const unsigned char* cs = sm + SM_CH + b * CH_BYTES;
      const uint32_t css = sbase + SM_CH + b * CH_BYTES;
      const uint32_t xu = tmem + lb + TM_X + 64 * b;
      // ---- U = U' - W S (fp32), then in place as bf16 high/low per K step
      bad |= !__all_sync(0xffffffffu, mbar_wait(&bars[B_X], n & 1, abort, args.wait_ns));
      if (issuer) KTRACE(n, 0);
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t u[16], w[16];
        tmem_ld_x16(xu + 16 * kk, u);
        tmem_wait_ld();
        if (issuer && kk == 0) KTRACE(n, 21);
#pragma unroll
        for (int p = 0; p < 8; ++p)
          split_pair(__uint_as_float(u[2 * p]), __uint_as_float(u[2 * p + 1]), w[p], w[8 + p]);
        if (dbg && n < args.dbg_nsc) {
#pragma unroll
          for (int t = 0; t < C; ++t) dbg[n * DBG_STRIDE + DBG_U + (C * kk + t) * D + dv] = __uint_as_float(u[t]);
        }
        tmem_st_x16(xu + 16 * kk, w);
      }
      tmem_wait_st();
      tc_fence_before();
      if (bar_sync_or(NB_STATE, 128, bad || *abort)) {
        bad = true;
        break;
      }
      if (issuer) {
        KTRACE(n, 1);
        tc_fence_after();
        const uint32_t ua = tmem + TM_X + 64 * b;
        const uint32_t kc = css + CH_KC, kcl = sbase + SM_KCL;
        // dS^T = U^T KhC (U high and low; KhC low in the last super-chunk)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint64_t bk = sdesc_noswz(kc + kk * 4096, 2048, 128);
          mma_ts(tmem + TM_DS, ua + 16 * kk, bk, idesc_bf16_f32(128, 128), kk > 0);
          mma_ts(tmem + TM_DS, ua + 16 * kk + 8, bk, idesc_bf16_f32(128, 128), 1);
          if (last)
            mma_ts(tmem + TM_DS, ua + 16 * kk, sdesc_noswz(kcl + kk * 4096, 2048, 128),
                   idesc_bf16_f32(128, 128), 1);
        }
        mma_commit(&bars[B_DS]);
        mma_commit(&bars[B_FREE + b]);
        mbar_arrive(&bars[B_UCONV]);  // the output group may issue P U on U's pair
      }
      // ---- S <- S e^{end} + dS, and its bf16 copy for the next super-chunk
      bad |= !__all_sync(0xffffffffu, mbar_wait(&bars[B_DS], n & 1, abort, args.wait_ns));
      if (issuer) KTRACE(n, 2);
      tc_fence_after();
      {
        const float4* eg = (const float4*)(cs + CH_EG);
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t ds[32];
          tmem_ld_x32(tmem + lb + TM_DS + 32 * blk, ds);
          tmem_wait_ld();
          if (issuer && blk == 0) KTRACE(n, 22);
          if (issuer && blk == 3) KTRACE(n, 23);
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 e = eg[8 * blk + i4];  // shared-memory broadcast
            const int i = 32 * blk + 4 * i4;
            S[i + 0] = fmaf(S[i + 0], e.x, __uint_as_float(ds[4 * i4 + 0]));
            S[i + 1] = fmaf(S[i + 1], e.y, __uint_as_float(ds[4 * i4 + 1]));
            S[i + 2] = fmaf(S[i + 2], e.z, __uint_as_float(ds[4 * i4 + 2]));
            S[i + 3] = fmaf(S[i + 3], e.w, __uint_as_float(ds[4 * i4 + 3]));
          }
          if (!last) write_sbf(blk);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      if (bar_sync_or(NB_STATE, 128, bad || *abort)) {
        bad = true;
        break;
      }
      if (issuer) {
        mbar_arrive(&bars[B_FREE + b]);  // e^{end} read by the whole group
        KTRACE(n, 3);
        if (!last && !issue_x(n + 1)) fail(abort, args.status);
        KTRACE(n, 4);
      }
    }
    if (bad) fail(abort, args.status);
    if (!bad && final_state) {
#pragma unroll
      for (int i = 0; i < D; ++i) final_state[soff + (int64_t)i * D + dv] = S[i];
    }
    if (issuer) {
      mma_commit(&bars[B_DRAIN]);
      mbar_wait_drain(&bars[B_DRAIN], 0, args.wait_ns);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, TM_COLS);
  }
}

template <bool kOutBf16, bool kSplitS>
cudaError_t prepare_kernel() {
  const void* fn = (const void*)kda_fwd_tc32_kernel<kOutBf16, kSplitS>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc can only draw on the registers the block was launched
  // with: a split above the compiled launch allocation would wait forever
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

// Per-device one-time kernel set-up (the shared-memory attribute applies to
// the current device's context only).
constexpr int kMaxDevices = 64;
std::once_flag g_prep_once[kMaxDevices];
cudaError_t g_prep_err[kMaxDevices];

cudaError_t prepare_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_prep_once[dev], [dev]() {
    cudaError_t e = prepare_kernel<false, false>();
    if (e == cudaSuccess) e = prepare_kernel<true, false>();
    if (e == cudaSuccess) e = prepare_kernel<false, true>();
    if (e == cudaSuccess) e = prepare_kernel<true, true>();
    g_prep_err[dev] = e;
  });
  return g_prep_err[dev];
}

}  // namespace

bool tc32_supported(int dtype, int dk, int dv) {
  return dtype == KDA_DTYPE_BF16 && dk == D && dv == D;
}

int launch_tc32_jobs(const FwdParams& p, const SegJob* jobs, int njobs, cudaStream_t stream,
                     uint64_t wait_ns, bool split_s, float* dbg, int dbg_nsc) {
  if (!tc32_supported(p.dtype, p.dk, p.dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
  const int64_t tokens = p.cu_seqlens ? (int64_t)p.T : (int64_t)p.N * p.T;
  if (tokens <= 0) {
    // nothing to load; a tensor map needs a nonzero extent, so use the SIMT
    // kernel, which handles empty sequences with no loads
    return launch_simt(p, stream);
  }
  if (tokens > INT32_MAX) return KDA_ERR_INVALID_ARG;
  CUtensorMap mq, mk, mth, mv;
  if (!encode_token_rows(&mq, p.q, p.H, tokens, CS) || !encode_token_rows(&mk, p.k, p.H, tokens, CS) ||
      !encode_token_rows(&mth, p.theta, p.H, tokens, CS) || !encode_token_rows(&mv, p.v, p.H, tokens, CS))
    return KDA_ERR_CUDA;
  if (prepare_device() != cudaSuccess) return KDA_ERR_LAUNCH;
  Tc32Args a;
  a.jobs = jobs;
  a.wait_ns = wait_ns ? wait_ns : kWaitNs;
  a.beta = (const __nv_bfloat16*)p.beta;
  a.g_min = p.g_min;
  a.gate = p.gate;
  a.init_state = p.init_state;
  a.out = p.out;
  a.final_state = p.final_state;
  a.cu_seqlens = p.cu_seqlens;
  a.N = p.N;
  a.H = p.H;
  a.T = p.T;
  a.status = status_word_device_ptr();
  a.dbg = dbg;
  a.dbg_nsc = dbg_nsc;
  if (!a.status) return KDA_ERR_CUDA;
  const unsigned grid = jobs ? (unsigned)njobs : (unsigned)(p.N * p.H);
  if (grid == 0) return KDA_OK;
  const bool ob = p.out_dtype == KDA_DTYPE_BF16;
  if (ob && split_s)
    kda_fwd_tc32_kernel<true, true><<<grid, kThreads, SMEM_BYTES, stream>>>(mq, mk, mth, mv, a);
  else if (ob)
    kda_fwd_tc32_kernel<true, false><<<grid, kThreads, SMEM_BYTES, stream>>>(mq, mk, mth, mv, a);
  else if (split_s)
    kda_fwd_tc32_kernel<false, true><<<grid, kThreads, SMEM_BYTES, stream>>>(mq, mk, mth, mv, a);
  else
    kda_fwd_tc32_kernel<false, false><<<grid, kThreads, SMEM_BYTES, stream>>>(mq, mk, mth, mv, a);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // namespace kda

#ifdef KDA_TRACE
extern "C" KDA_API int kda_debug_trace_read_tc32(void* dst, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(dst, kda::g_kda_trace_tc32, bytes);
}
#endif
