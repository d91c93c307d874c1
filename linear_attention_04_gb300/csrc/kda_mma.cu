// kda_mma.cu -- register-resident tensor-core path of the KDA chunked forward
// pass (bf16 q, k, v, theta, beta; dk = dv = 128; fp32 state; fp32 or bf16 out).
//
// The recurrence S_t = (I - b_t k_t k_t^T) Diag(e^{g_t}) S_{t-1} + b_t k_t v_t^T,
// o_t = S_t^T q_t ("Kimi K3 Deep Dive", section "Core Innovation 1") acts on
// every value channel (column of S) separately: column j of S depends only on
// k, g, b and column j of V.  So the dv = 128 value channels are split over
// four warps, 32 each, and each warp carries its 128 x 32 slice of S in fp32
// registers through the whole sequence, with no exchange between warps.
//
// Per 16-token chunk n (G = inclusive in-chunk cumulative log-decay,
// Kt = K e^{G}, Qt = Q e^{G}, Kh = K e^{-G}, KhC = K e^{G_C - G}; every factor
// lies in [e^{-80}, e^{80}] for g >= g_min = -5, "Kimi K3 Deep Dive", section
// "The Design"):
//
//   A  = strict_lower(Diag(b) Kt Kh^T)      P = strict_lower(Qt Kh^T)
//   Tb = (I + A)^{-1} Diag(b)               W = Tb Kt
//   U  = Tb V - W S                         O = Qt S + P U + Diag(q_t . k_t) U
//   S <- Diag(e^{G_C}) S + KhC^T U
//
// Warp roles (256 threads, one warp of each role per SM sub-partition):
//   warps 0..3  state warps: warp w owns value channels 32w .. 32w+31.  Per
//               chunk, with S^T (value channel x key channel) as the A operand
//               taken straight from the fp32 accumulator registers (bf16 pairs):
//                 [U | O] = [V^T Tb^T | 0] + S^T [-W | Qt]^T      (K = 128)
//                 O      += U^T P^T (U and P as bf16 high/low pairs) + (q.k) U
//                 S^T    <- S^T Diag(e^{G_C}) + U^T KhC           (K = 16)
//               then the warp writes its outputs and releases the chunk slot.
//   warps 4..7  intra warps: warp 4+i runs chunks i, i+4, i+8, ...; each
//               loads its chunk with TMA (q, k, theta, v into a private stage,
//               refilled with its next chunk as soon as the stage is read),
//               computes the gate (g = g_min * sigmoid(theta)), the cumulative
//               sums and the decayed operands in fp32, the chunk products A, P
//               and W = Tb Kt with mma.sync, the triangular inverse by forward
//               substitution, and fills a chunk slot for the state warps.
//
// All products are mma.sync m16n8k16 (bf16 operands, fp32 accumulation).
// The chain of dependent products per chunk is short (a few dozen
// instructions per warp between hand-offs) and every operand of the state
// products stays in registers, which is what the sequential recurrence needs:
// its speed is set by the latency of each step, not by tensor throughput.
//
// The diagonal of Qt Kh^T is q_t . k_t exactly (the decay factors cancel), so
// it is taken in fp32 from the bf16 inputs and applied to U in fp32.
//
// A CTA runs one whole (sequence, head) chain; or, in a segmented launch, one
// job of a table (token range, head, initial and final state, and options: v
// taken as zero, no outputs, identity initial state), which is how the
// segment-parallel forward obtains each segment's linear part and local
// state; or, in the wrapped schedule, one equal window of chunk steps over the
// chains laid end to end.  The wrapped schedule serves fixed-length batches
// with more chains than CTAs that can be resident at once: one chain per CTA
// would leave SMs idle in the last wave (256 chains on 152 SMs take two full
// chain times), while equal windows of ceil(chains * chunks / CTAs) steps
// (McNaughton's wrap-around rule) take 1.68.  A chain cut by a window boundary
// runs its first chunks at the start of the later window and the rest at the
// end of the earlier one; the fp32 state is handed over exactly, through the
// chain's final-state slot and a release/acquire flag per state warp.  The
// CTAs are launched cooperatively (all resident), and every wait is bounded.
// The gate is g_min * sigmoid(theta), or theta itself as a given log-decay.
//
// Every wait is bounded: a wait that runs out sets the CTA's abort flag and the
// device status word (KDA_ERR_DEVICE_TIMEOUT); every role then leaves its loop
// and the TMA loads still in flight are drained before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kda_device.cuh"
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int C = kChunk;  // 16
constexpr int D = 128;     // dk = dv
constexpr int kStateWarps = 4;
constexpr int kDvPerWarp = D / kStateWarps;  // value channels per state warp
constexpr int kMT = kDvPerWarp / 16;          // m16 tiles per state warp
static_assert(kMT >= 1 && kMT * 16 * kStateWarps == D, "state warp split");
constexpr int kIntraWarps = 4;
constexpr int kThreads = 32 * (kStateWarps + kIntraWarps);
// Per-thread registers of each role after setmaxnreg (0: every warp keeps the
// launch allocation).  The split must fit the launch allocation; the host
// checks it against the compiled register count before the first launch.
constexpr int kStateRegs = 0, kIntraRegs = 0;
constexpr uint64_t kWaitNs = 2000000000ull;  // default limit of every wait: 2 s
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- shared memory
constexpr uint32_t ROW = D * 2;       // 256 bytes: one 128-channel bf16 row
constexpr uint32_t TILE = C * ROW;    // 4096: a 16 x 128 bf16 tile
constexpr uint32_t STAGE = 4 * TILE;  // q, k, theta, v of one chunk (TMA, unswizzled)

// chunk slot, written by one intra warp and read by the four state warps
constexpr uint32_t SL_XB = 0;                 // [32][128] bf16: rows 0..15 Kt, then -W; 16..31 Qt
constexpr uint32_t SL_KC = SL_XB + 2 * TILE;  // [16][128] bf16 KhC (token-major)
constexpr uint32_t SL_V = SL_KC + TILE;       // [16][128] bf16 V (rows past the end zeroed)
constexpr uint32_t SL_TB = SL_V + TILE;       // [16][16] bf16 Tb
constexpr uint32_t SL_P = SL_TB + 512;        // [16][16] bf16 strictly lower P (high part)
constexpr uint32_t SL_PL = SL_P + 512;        // [16][16] bf16 low part of P
constexpr uint32_t SL_EGC = SL_PL + 512;      // [128] fp32 e^{G_C}
constexpr uint32_t SL_DC = SL_EGC + 512;      // [16] fp32 q_t . k_t
constexpr uint32_t SLOT_BYTES = SL_DC + 128;

constexpr uint32_t AB_BYTES = C * C * 4;       // [16][16] fp32 A of one intra warp
constexpr uint32_t GA_ROWS = 32 * kIntraWarps;  // tcgen05 Gram operand: [Kt; Qt] of each intra warp
constexpr uint32_t GA_BYTES = GA_ROWS * D * 2;  // 32 KB, 128-byte swizzled, two 64-channel halves
constexpr uint32_t GA_HALF = GA_ROWS * 128;     // bytes of one 64-channel half
constexpr uint32_t GB_HALF = C * 128;           // the same for a [16][128] Kh operand
constexpr int kTmemCols = 16 * kIntraWarps;     // [16 rows of A | 16 rows of P] x 16 columns per warp

// Shared-memory layout.  kTc: the intra products A and P are tcgen05.mma
// (operands in 128-byte-swizzled tiles, results in tensor memory), which
// takes a 32 KB operand tile; the chain-order scratch, used only before the
// main loops, then lies inside that tile.  Otherwise A and P are warp-level
// mma.sync over the XOR-swizzled tiles.
template <bool kTc>
struct Lay {
  static constexpr int kSlots = 6;                           // chunk slots between the roles
  static constexpr uint32_t RING = 0;                        // kIntraWarps x STAGE
  static constexpr uint32_t KH = RING + kIntraWarps * STAGE; // kIntraWarps x [16][128] bf16 Kh
  static constexpr uint32_t GA = KH + kIntraWarps * TILE;    // [Kt; Qt] operand (kTc only)
  static constexpr uint32_t AB = GA + (kTc ? GA_BYTES : 0);  // kIntraWarps x [16][16] fp32 A
  static constexpr uint32_t SLOTS = AB + kIntraWarps * AB_BYTES;
  static constexpr uint32_t BARS = SLOTS + kSlots * SLOT_BYTES;
  static constexpr int B_FULL = 0;                           // [kIntraWarps] TMA -> intra warp
  static constexpr int B_READY = kIntraWarps;                // [kSlots] intra warp -> state warps
  static constexpr int B_FREE = B_READY + kSlots;            // [kSlots] state warps (4 arrivals)
  static constexpr int B_GRAM = B_FREE + kSlots;             // [kIntraWarps] Gram product done
  static constexpr int NBARS = B_GRAM + (kTc ? kIntraWarps : 0);
  // abort, job flags, tensor memory address (16 bytes), then the CTA's chunk
  // schedule (64 bytes)
  static constexpr uint32_t MISC = BARS + NBARS * 8;
  static constexpr uint32_t SCHED = MISC + 16;
  static constexpr uint32_t RANK = kTc ? GA : MISC + 80;     // chain-order scratch
  static constexpr uint32_t TOTAL = kTc ? MISC + 80 : RANK + (kMaxRankedSeqsDev + 1) * 4;
  static constexpr uint32_t BYTES = TOTAL + (kTc ? 1024 : 128);  // + alignment slack
  static_assert(BYTES <= 232448, "shared memory budget");
  static_assert(SLOT_BYTES % 128 == 0 && SLOTS % 128 == 0, "slot alignment");
  static_assert(KH % 1024 == 0 && GA % 1024 == 0, "swizzled operand tiles on 1024-byte boundaries");
  static_assert(!kTc || (kMaxRankedSeqsDev + 1) * 4 <= GA_BYTES, "chain-order scratch fits the tile");
  static_assert(MISC % 8 == 0, "schedule alignment");
};

// Byte offset of (row, col) in a tile of 256-byte rows (128 bf16 channels)
// whose 16-byte chunks are XOR-swizzled by row: eight consecutive rows of one
// chunk column fall in distinct banks (conflict-free ldmatrix).
__device__ __forceinline__ uint32_t sw256(int row, int col) {
  const int c = col >> 3;
  return (uint32_t)(row * 256 + (((c ^ row) & 7) | (c & 8)) * 16 + (col & 7) * 2);
}
// Same for 16 x 16 bf16 tiles (32-byte rows): chunk XOR (row / 4).
__device__ __forceinline__ uint32_t sw32(int row, int col) {
  return (uint32_t)(row * 32 + (((col >> 3) ^ (row >> 2)) & 1) * 16 + (col & 7) * 2);
}

// Byte offset of (row, col) in a tcgen05 operand tile of 128 bf16 channels per
// row, K-major with the 128-byte swizzle: two 64-channel halves of
// `half_bytes` each, rows of 128 bytes (8-row atoms of 1024 bytes), the
// 16-byte pieces of row r XOR-permuted by r mod 8.
__device__ __forceinline__ uint32_t sw128(int row, int col, uint32_t half_bytes) {
  const int c = col & 63;
  return (uint32_t)((col >> 6) * half_bytes + row * 128 + ((((c >> 3) ^ row) & 7) << 4) +
                    (c & 7) * 2);
}

// D += A B with mma.sync m16n8k16, bf16 operands, fp32 accumulators (a pure
// register operation: not volatile, so the compiler may schedule it freely).
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Register count of every thread at launch (the full file divided evenly) and
// the per-role adjustment away from it.
constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8 > 255 ? 255 : (65536 / kThreads) / 8 * 8;
template <int N>
__device__ __forceinline__ void set_regs() {
  if constexpr (N > kLaunchRegs)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
  else if constexpr (N < kLaunchRegs)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Largest -G2_C (log2 domain) of a chunk that the dense tile takes: e^{-G}
// up to 2^126 stays finite in bf16 and fp32.  The bounded gate never gets
// near it (-G_C <= 80, i.e. -G2_C <= 115.4).
constexpr float kFallbackLog2 = 126.0f;

// The position-wise form of one chunk's intra tiles, for chunks whose decay
// is too steep for the dense product (the pages contrast it with the bounded
// gate: "Kimi K3 Deep Dive", sections "The Problem" and "The Design").  Every
// factor is formed per pair of positions, e^{G_r - G_s} <= 1 for s < r, so
// nothing overflows:
//   A_rs = b_r sum_c k_rc k_sc e^{G_rc - G_sc},   P_rs = sum_c q_rc k_sc e^{G_rc - G_sc}
//   KhC_t = k_t e^{G_C - G_t}
// One warp per chunk; lane l holds channels 4l .. 4l+3 (as in the dense phase
// A).  The gate is recomputed from theta in the stage; the 120 pairs are
// summed over the lane's channels and then over the warp, 16 pairs at a
// time.  Writes the beta-scaled strictly lower A (fp32, 16 x 16 at `ab`), P as
// a bf16 high/low pair and KhC into the chunk slot, replacing what the dense
// phase A left there.
__device__ __forceinline__ void position_wise_tiles(const unsigned char* st, unsigned char* sl, float* ab,
                                                 int lane, float beta_l, bool log_decay, float g_min,
                                                 f32x2 GC0, f32x2 GC1) {
  const uint2* sk = (const uint2*)(st + 1 * TILE);
  const uint2* sq = (const uint2*)(st + 0 * TILE);
  const uint2* sth = (const uint2*)(st + 2 * TILE);
  const f32x2 kL2 = f2(kLog2e, kLog2e);
  const f32x2 kC2 = f2(-kLog2e, -kLog2e);
  const f32x2 kC1 = f2(g_min * kLog2e, g_min * kLog2e);
  const f32x2 kOne = f2(1.0f, 1.0f);
  // the gate and the in-chunk cumulative sums again (log2 domain)
  f32x2 Gl[C][2];
  f32x2 G0 = 0ull, G1 = 0ull;
#pragma unroll
  for (int t = 0; t < C; ++t) {
    const uint2 thw = sth[t * 32 + lane];
    f32x2 g0, g1;
    if (log_decay) {
      g0 = mul2(bf2_to_f2(thw.x), kL2);
      g1 = mul2(bf2_to_f2(thw.y), kL2);
    } else {
      const f32x2 x0 = mul2(bf2_to_f2(thw.x), kC2), x1 = mul2(bf2_to_f2(thw.y), kC2);
      const f32x2 d0 = add2(f2(ex2_approx(f2lo(x0)), ex2_approx(f2hi(x0))), kOne);
      const f32x2 d1 = add2(f2(ex2_approx(f2lo(x1)), ex2_approx(f2hi(x1))), kOne);
      g0 = mul2(f2(rcp_approx(f2lo(d0)), rcp_approx(f2hi(d0))), kC1);
      g1 = mul2(f2(rcp_approx(f2lo(d1)), rcp_approx(f2hi(d1))), kC1);
    }
    G0 = add2(G0, g0);
    G1 = add2(G1, g1);
    Gl[t][0] = G0;
    Gl[t][1] = G1;
  }
  // KhC_t = k_t e^{G_C - G_t}
#pragma unroll
  for (int t = 0; t < C; ++t) {
    const uint2 kw = sk[t * 32 + lane];
    const f32x2 x0 = add2(GC0, f2(-f2lo(Gl[t][0]), -f2hi(Gl[t][0])));
    const f32x2 x1 = add2(GC1, f2(-f2lo(Gl[t][1]), -f2hi(Gl[t][1])));
    const f32x2 e0 = f2(ex2_approx(f2lo(x0)), ex2_approx(f2hi(x0)));
    const f32x2 e1 = f2(ex2_approx(f2lo(x1)), ex2_approx(f2hi(x1)));
    *(uint2*)(sl + SL_KC + sw256(t, 4 * lane)) =
        make_uint2(f2_to_bf2(mul2(bf2_to_f2(kw.x), e0)), f2_to_bf2(mul2(bf2_to_f2(kw.y), e1)));
  }
  // zero the tiles (their upper parts stay zero)
#pragma unroll
  for (int i = 0; i < 8; ++i) ab[8 * lane + i] = 0.0f;
  *(uint4*)(sl + SL_P + 16 * lane) = make_uint4(0u, 0u, 0u, 0u);
  *(uint4*)(sl + SL_PL + 16 * lane) = make_uint4(0u, 0u, 0u, 0u);
  __syncwarp();
  // the 120 pairs s < r, 16 at a time: lane partial sums over its channels,
  // then a transpose-reduce over the warp (lane l ends with pair (l >> 1) & 15
  // of the batch)
  float pa[16], pp[16];
  int np = 0;
#pragma unroll
  for (int r = 1; r < C; ++r) {
    const uint2 kr = sk[r * 32 + lane], qr = sq[r * 32 + lane];
    const f32x2 kr0 = bf2_to_f2(kr.x), kr1 = bf2_to_f2(kr.y);
    const f32x2 qr0 = bf2_to_f2(qr.x), qr1 = bf2_to_f2(qr.y);
#pragma unroll
    for (int s2 = 0; s2 < r; ++s2) {
      const uint2 ks = sk[s2 * 32 + lane];
      const f32x2 x0 = add2(Gl[r][0], f2(-f2lo(Gl[s2][0]), -f2hi(Gl[s2][0])));
      const f32x2 x1 = add2(Gl[r][1], f2(-f2lo(Gl[s2][1]), -f2hi(Gl[s2][1])));
      const f32x2 e0 = mul2(f2(ex2_approx(f2lo(x0)), ex2_approx(f2hi(x0))), bf2_to_f2(ks.x));
      const f32x2 e1 = mul2(f2(ex2_approx(f2lo(x1)), ex2_approx(f2hi(x1))), bf2_to_f2(ks.y));
      const f32x2 a = fma2(kr1, e1, mul2(kr0, e0));
      const f32x2 pq = fma2(qr1, e1, mul2(qr0, e0));
      pa[np & 15] = f2lo(a) + f2hi(a);
      pp[np & 15] = f2lo(pq) + f2hi(pq);
      ++np;
      if ((np & 15) == 0 || np == C * (C - 1) / 2) {
        // pad a short last batch
#pragma unroll
        for (int z = 0; z < 16; ++z)
          if (z >= ((np - 1) & 15) + 1) pa[z] = pp[z] = 0.0f;
        float sa[8], sp[8], ta[4], tp[4], ua[2], up[2], va, vp;
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          sa[j] = (b4 ? pa[j + 8] : pa[j]) + __shfl_xor_sync(0xffffffffu, b4 ? pa[j] : pa[j + 8], 16);
          sp[j] = (b4 ? pp[j + 8] : pp[j]) + __shfl_xor_sync(0xffffffffu, b4 ? pp[j] : pp[j + 8], 16);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ta[j] = (b3 ? sa[j + 4] : sa[j]) + __shfl_xor_sync(0xffffffffu, b3 ? sa[j] : sa[j + 4], 8);
          tp[j] = (b3 ? sp[j + 4] : sp[j]) + __shfl_xor_sync(0xffffffffu, b3 ? sp[j] : sp[j + 4], 8);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          ua[j] = (b2 ? ta[j + 2] : ta[j]) + __shfl_xor_sync(0xffffffffu, b2 ? ta[j] : ta[j + 2], 4);
          up[j] = (b2 ? tp[j + 2] : tp[j]) + __shfl_xor_sync(0xffffffffu, b2 ? tp[j] : tp[j + 2], 4);
        }
        va = (b1 ? ua[1] : ua[0]) + __shfl_xor_sync(0xffffffffu, b1 ? ua[0] : ua[1], 2);
        vp = (b1 ? up[1] : up[0]) + __shfl_xor_sync(0xffffffffu, b1 ? up[0] : up[1], 2);
        va += __shfl_xor_sync(0xffffffffu, va, 1);
        vp += __shfl_xor_sync(0xffffffffu, vp, 1);
        // this lane's pair index, and its (r, s) position
        const int idx = ((np - 1) & ~15) + ((lane >> 1) & 15);
        int pr = 1, base = 0;
        while (base + pr <= idx) {
          base += pr;
          ++pr;
        }
        const int ps = idx - base;
        const float br = __shfl_sync(0xffffffffu, beta_l, pr & 15);
        if ((lane & 1) == 0 && idx < np) {
          ab[pr * C + ps] = br * va;
          const __nv_bfloat16 hi = __float2bfloat16_rn(vp);
          *(__nv_bfloat16*)(sl + SL_P + sw32(pr, ps)) = hi;
          *(__nv_bfloat16*)(sl + SL_PL + sw32(pr, ps)) = __float2bfloat16_rn(vp - __bfloat162float(hi));
        }
      }
    }
  }
}

struct MmaArgs {
  const SegJob* jobs;  // per-CTA work units (segmented launches), or null
  uint64_t wait_ns;    // limit of every bounded wait
  // Wrapped schedule (kWrap launches: fixed-length batches with more chains
  // than resident CTAs): CTA b runs chunk steps [b wrap_cap, (b + 1) wrap_cap)
  // of the chains laid end to end; a chain cut by a window boundary hands its
  // state over through its final_state slot, announced by a per-warp flag set
  // to `epoch`.
  int wrap_cap;
  uint32_t epoch;
  uint32_t* hflags;  // [grid + 1][kStateWarps] handoff flags of this launch
  const __nv_bfloat16* beta;
  float g_min;
  int gate;
  const float* init_state;
  void* out;
  int out_bf16;
  float* final_state;
  const int32_t* cu_seqlens;
  int N, H, T;
  int* status;
};

// The chunk steps 0 .. nsteps-1 of one CTA.
// Unwrapped: chunks 0 .. nsteps-1 of one chain (first token row `row`, head
// `head`, `len` tokens).
// Wrapped: positions [w0, w0 + nsteps) of the N H chains of p chunks each laid
// end to end (chain c = sequence c / H, head c mod H, T tokens from row
// (c / H) T).  A chain cut by the window's start runs its first `a` chunks
// here, at the start, and the rest at the end of the previous CTA's window; a
// chain cut by the window's end runs its last `y` chunks here, at the end,
// from the state that the next CTA hands over after running its first
// chunks.  With every window at least p long, the first part of a cut chain
// ends (a chunk-steps into the later window) well before its second part
// starts (p - a chunk-steps before the earlier window's end), so the hand-over
// costs no waiting (McNaughton's wrap-around rule, with each cut chain's two
// parts in the order the recurrence needs).
struct Sched {
  int wrap, nsteps;
  int64_t row;   // unwrapped
  int64_t soff;  // unwrapped: element offset of the chain's states in init/final
  int head, len;
  int w0, a, y, p, H, T;  // wrapped
};

static_assert(sizeof(Sched) <= 64, "the schedule's shared-memory slot");

// One chain's run of consecutive steps starting at step n.
struct Piece {
  int64_t chain;     // chain index (wrapped); its states sit at chain * D * D
  int64_t row;       // token row of the chain's first token
  int head, len;     // head; tokens of the chain
  int nc0, steps;    // chunk of the chain at the piece's first step; steps
  bool from_handoff;  // start state handed over by the next CTA
  bool to_handoff;    // end state handed over to the previous CTA
};

__device__ __forceinline__ int sched_chain(const volatile Sched& s, int n, int& nc) {
  int c;
  if (n < s.a) {
    c = s.w0 / s.p;
    nc = n;
  } else if (n < s.nsteps - s.y) {
    const int v = s.w0 + n;
    c = v / s.p;
    nc = v - c * s.p;
  } else {
    c = (s.w0 + s.nsteps) / s.p;
    nc = n - s.nsteps + s.p;
  }
  return c;
}

// The chunk at one step, as an intra warp walks the schedule.
struct Cursor {
  int64_t row;  // token row of the chunk's first token
  int head;
  int rem;      // tokens of the chain from this chunk on (valid rows: min(C, rem))
  int pend;     // first step after the piece that holds this step
};

__device__ __forceinline__ Cursor cursor_at(const volatile Sched& s, int n) {
  Cursor k;
  if (!s.wrap) {
    k.row = s.row + (int64_t)n * C;
    k.head = s.head;
    k.rem = s.len - n * C;
    k.pend = s.nsteps;
    return k;
  }
  int nc;
  const int c = sched_chain(s, n, nc);
  const int seq = c / s.H;
  k.head = c - seq * s.H;
  k.row = (int64_t)seq * s.T + (int64_t)nc * C;
  k.rem = s.T - nc * C;
  if (n < s.a)
    k.pend = s.a;
  else if (n < s.nsteps - s.y)
    k.pend = n - nc + s.p;
  else
    k.pend = s.nsteps;
  return k;
}

// The cursor `step` steps after the cursor k of step n: the same chain while
// the piece lasts (no division), else looked up afresh.
__device__ __forceinline__ Cursor cursor_next(const volatile Sched& s, const Cursor& k, int n,
                                              int step) {
  if (n + step < k.pend) {
    Cursor r = k;
    r.row += (int64_t)step * C;
    r.rem -= step * C;
    return r;
  }
  return cursor_at(s, n + step);
}

template <bool kMayWrap>
__device__ __forceinline__ Piece sched_piece(const volatile Sched& s, int n) {
  Piece pc;
  pc.from_handoff = pc.to_handoff = false;
  if (!kMayWrap || !s.wrap) {
    pc.chain = 0;
    pc.row = s.row;
    pc.head = s.head;
    pc.len = s.len;
    pc.nc0 = 0;
    pc.steps = s.nsteps;
    return pc;
  }
  int nc;
  const int c = sched_chain(s, n, nc);
  pc.nc0 = nc;
  if (n < s.a) {
    pc.steps = s.a;
    pc.to_handoff = true;
  } else if (n < s.nsteps - s.y) {
    pc.steps = s.p;
  } else {
    pc.steps = s.y;
    pc.from_handoff = true;
  }
  const int seq = c / s.H;
  pc.chain = c;
  pc.head = c - seq * s.H;
  pc.row = (int64_t)seq * s.T;
  pc.len = s.T;
  return pc;
}

// Acquire / release accesses of the hand-over flags (gpu scope).
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Waits until *f == want; gives up after limit_ns or once *abort is set.
__device__ __forceinline__ bool wait_flag(const uint32_t* f, uint32_t want, const volatile int* abort,
                                          uint64_t limit_ns) {
  if (ld_acquire_u32(f) == want) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(256);
    if (ld_acquire_u32(f) == want) return true;
    if ((i & 15) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

// Optional event trace of the first CTA (compile with -DKDA_TRACE): wall-clock
// time of each pipeline event per chunk, read back with kda_debug_trace_read_mma.
constexpr int kTraceChunks = 512;
#ifdef KDA_TRACE
__device__ unsigned long long g_kda_trace_mma[kTraceChunks * 16];
#define KTRACE(n, k)                                                                              \
  do {                                                                                            \
    if (blockIdx.x == 0 && (n) < kTraceChunks) g_kda_trace_mma[(n) * 16 + (k)] = globaltimer_ns(); \
  } while (0)
#define KTRACE_CLK(n, k)                                                               \
  do {                                                                                 \
    if (blockIdx.x == 0 && (n) < kTraceChunks) g_kda_trace_mma[(n) * 16 + (k)] = clock64(); \
  } while (0)
#else
#define KTRACE(n, k) \
  do {               \
  } while (0)
#define KTRACE_CLK(n, k) \
  do {                   \
  } while (0)
#endif

__device__ __forceinline__ void fail(volatile int* abort, int* status) {
  *abort = 1;
  atomicExch(status, KDA_ERR_DEVICE_TIMEOUT);
}

// kFallback: compile the position-wise fallback for chunks whose decay is too
// steep for the dense tile (only a given, unbounded log-decay can produce
// them; the bounded gate's kernel carries no such code)
// The CTA's work unit (template parameter kMode): one whole chain
// (kModeChain), one job of a table (kModeJobs, the segmented forward and the
// failure-test hook: the job options are compiled in only here), or one
// window of the wrapped schedule (kModeWrap).
constexpr int kModeChain = 0, kModeJobs = 1, kModeWrap = 2;

template <bool kOutBf16, bool kFallback, bool kTc, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    kda_fwd_mma_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_th,
                       const __grid_constant__ CUtensorMap tm_v, const MmaArgs args) {
  using Ly = Lay<kTc>;
  constexpr bool kWrap = kMode == kModeWrap;
  constexpr bool kJobs = kMode == kModeJobs;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // pointer arithmetic on the shared array itself keeps the shared address
  // space visible to the compiler (32-bit shared addressing); the swizzled
  // tcgen05 operand tiles want a 1024-byte aligned base
  constexpr uint32_t kAlign = kTc ? 1024u : 128u;
  unsigned char* sm = smem_raw + ((kAlign - (smem_u32(smem_raw) & (kAlign - 1u))) & (kAlign - 1u));
  uint64_t* bars = (uint64_t*)(sm + Ly::BARS);
  volatile int* abort = (volatile int*)(sm + Ly::MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // fragment coordinates of mma.sync (g: row group, q: column pair) and of
  // ldmatrix.x4 (mi: which 8x8 matrix this lane addresses, rr: its row)
  const int g = lane >> 2, q = lane & 3, mi = lane >> 3, rr = lane & 7;

  // the work unit: a whole (sequence, head) chain, one segment job, or one
  // window of the wrapped schedule.  (The wrapped instantiation tests the
  // schedule at run time, as one flag it cannot fold: its register allocation
  // then measures faster than with the choice folded in.)
  const bool wrap_rt = kWrap && args.wrap_cap > 0;
  Chain ch;
  int flags = 0;
  const float* init_state = args.init_state;
  float* final_state = args.final_state;
  int64_t soff = 0;  // element offset of this chain's state in init/final
  if (kJobs) {
    const SegJob jb = args.jobs[blockIdx.x];
    ch.seq = 0;
    ch.head = jb.head;
    ch.t0 = jb.t0;
    ch.t1 = jb.t1;
    flags = jb.flags;
    init_state = jb.init;
    final_state = jb.final_state;
  } else if (wrap_rt) {
    ch.seq = ch.head = 0;
    ch.t0 = ch.t1 = 0;
    ch.valid = true;
  } else {
    ch = chain_for_block(blockIdx.x, args.H, args.N, args.T, args.cu_seqlens, (int*)(sm + Ly::RANK));
    if (!ch.valid) {
      // malformed packing table: report it and store nothing
      if (tid == 0) atomicExch(args.status, KDA_ERR_BAD_SEQLENS);
      return;
    }
    soff = ((int64_t)ch.seq * args.H + ch.head) * D * D;
  }
  // options read back from shared memory where they are used (keeps them out
  // of the register budget of the main loops)
  volatile int* sflags = (volatile int*)(sm + Ly::MISC + 4);
  const int H = args.H;
  // the CTA's chunk schedule, kept in shared memory and read where it is used
  // (out of the register budget of the main loops)
  volatile Sched& sc = *(volatile Sched*)(sm + Ly::SCHED);
  int nsteps;
  if (tid == 0) {
    Sched s = {};
    s.wrap = wrap_rt;
    if (wrap_rt) {
      s.p = (args.T + C - 1) / C;
      s.H = args.H;
      s.T = args.T;
      const int total = args.N * args.H * s.p;  // below 2^31 (checked by the host)
      s.w0 = (int)blockIdx.x * args.wrap_cap;
      s.nsteps = min(args.wrap_cap, total - s.w0);
      const int x = s.w0 % s.p;
      s.a = x ? s.p - x : 0;
      const int w1 = s.w0 + s.nsteps;
      s.y = w1 < total ? w1 % s.p : 0;
    } else {
      s.row = ch.t0;
      s.soff = soff;
      s.head = ch.head;
      s.len = (int)(ch.t1 - ch.t0);
      s.nsteps = (s.len + C - 1) / C;
    }
    sc.wrap = s.wrap;
    sc.nsteps = s.nsteps;
    sc.row = s.row;
    sc.soff = s.soff;
    sc.head = s.head;
    sc.len = s.len;
    sc.w0 = s.w0;
    sc.a = s.a;
    sc.y = s.y;
    sc.p = s.p;
    sc.H = s.H;
    sc.T = s.T;
  }

  if constexpr (kTc) {
    // tensor memory for the intra products: 16 columns per intra warp
    if (warp == kStateWarps) tmem_alloc((uint32_t*)(sm + Ly::MISC + 8), kTmemCols);
  }
  if (tid == 0) {
    for (int i = 0; i < Ly::NBARS; ++i)
      mbar_init(&bars[i], (i >= Ly::B_FREE && i < Ly::B_GRAM) ? kStateWarps : 1);
    *abort = 0;
    *sflags = flags;
    fence_mbar_init();
  }
  if constexpr (kTc) tc_fence_before();
  __syncthreads();
  if constexpr (kTc) tc_fence_after();
  const uint32_t sbase = smem_u32(sm);
  nsteps = sc.nsteps;

  if (warp >= kStateWarps) {
    // ================================================================ intra warps
    if constexpr (kIntraRegs > 0) set_regs<kIntraRegs>();
    const int iw = warp - kStateWarps;
    unsigned char* st = sm + Ly::RING + iw * STAGE;
    const uint32_t khs = sbase + Ly::KH + iw * TILE;
    unsigned char* kh = sm + Ly::KH + iw * TILE;
    float* ab = (float*)(sm + Ly::AB + iw * AB_BYTES);
    uint64_t* full = &bars[Ly::B_FULL + iw];
    const bool zero_v = kJobs && (*sflags & kJobZeroV);
    // one chain per CTA: chunk m of the chain (its length and chunk count
    // kept as values of this chain, which the loop below can see through)
    const int Lc = (int)(ch.t1 - ch.t0);
    const int nloop = kWrap ? nsteps : (Lc + C - 1) / C;
    auto load = [&](int m) {
      mbar_arrive_expect_tx(full, zero_v ? 3 * TILE : STAGE);
      const int row = (int)(ch.t0 + (int64_t)m * C);
      tma_load_3d(st + 0 * TILE, &tm_q, 0, ch.head, row, full);
      tma_load_3d(st + 1 * TILE, &tm_k, 0, ch.head, row, full);
      tma_load_3d(st + 2 * TILE, &tm_th, 0, ch.head, row, full);
      if (!zero_v) tma_load_3d(st + 3 * TILE, &tm_v, 0, ch.head, row, full);
    };
    // wrapped schedule: the chunk at a cursor
    auto load_at = [&](const Cursor& km) {
      mbar_arrive_expect_tx(full, zero_v ? 3 * TILE : STAGE);
      const int row = (int)km.row;
      tma_load_3d(st + 0 * TILE, &tm_q, 0, km.head, row, full);
      tma_load_3d(st + 1 * TILE, &tm_k, 0, km.head, row, full);
      tma_load_3d(st + 2 * TILE, &tm_th, 0, km.head, row, full);
      if (!zero_v) tma_load_3d(st + 3 * TILE, &tm_v, 0, km.head, row, full);
    };
    Cursor cur;  // wrapped schedule: the chunk of this warp's current step
    if constexpr (kWrap) cur = cursor_at(sc, iw);
    int issued = 0, consumed = 0;
    int gram_issued = 0, gram_waited = 0;  // tcgen05 Gram products of this warp
    uint32_t tmem = 0;
    if constexpr (kTc) tmem = *(volatile uint32_t*)(sm + Ly::MISC + 8);
    if (lane == 0 && iw < nloop) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_th);
      prefetch_tmap(&tm_v);
      if constexpr (kWrap)
        load_at(cur);
      else
        load(iw);
    }
    if (iw < nloop) issued = 1;
    bool bad = false;
    const bool log_decay = args.gate == KDA_GATE_LOG_DECAY;  // theta holds g itself
    const f32x2 kL2 = f2(kLog2e, kLog2e);
    const f32x2 kC2 = f2(-kLog2e, -kLog2e);
    const f32x2 kC1 = f2(args.g_min * kLog2e, args.g_min * kLog2e);
    const f32x2 kOne = f2(1.0f, 1.0f);
    const f32x2 kZero = 0ull;
    for (int n = iw; n < nloop; n += kIntraWarps) {
      const int slot = n % Ly::kSlots;
      int64_t crow;  // token row of the chunk's first token
      int h, nvalid;
      if constexpr (kWrap) {
        crow = cur.row;
        h = cur.head;
        nvalid = min(C, cur.rem);
      } else {
        crow = ch.t0 + (int64_t)n * C;
        h = ch.head;
        nvalid = min(C, Lc - n * C);
      }
      unsigned char* sl = sm + Ly::SLOTS + slot * SLOT_BYTES;
      const uint32_t sls = sbase + Ly::SLOTS + slot * SLOT_BYTES;
      // beta of the chunk (lane t holds beta_t), issued before the waits
      float beta_l = 0.0f;
      if (lane < nvalid) {
        if constexpr (kWrap)
          beta_l = __bfloat162float(args.beta[(crow + lane) * H + h]);
        else
          beta_l = __bfloat162float(args.beta[(ch.t0 + (int64_t)n * C + lane) * H + h]);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(full, consumed & 1, abort, args.wait_ns))) {
        bad = true;
        break;
      }
      ++consumed;
      if (lane == 0) KTRACE(n, 5);
      if (n >= Ly::kSlots &&
          !__all_sync(0xffffffffu, mbar_wait(&bars[Ly::B_FREE + slot], ((n / Ly::kSlots) - 1) & 1,
                                             abort, args.wait_ns))) {
        bad = true;
        break;
      }
      if (lane == 0) KTRACE(n, 6);
      if (nvalid < C) {
        // rows past the end of the sequence (the next sequence's tokens, or the
        // zero fill past the tensor) become neutral: q = k = v = 0 and g = 0 (no
        // decay, no contribution): theta = -inf for the sigmoid gate, 0 when
        // theta is the log-decay itself
        for (int e = lane; e < (C - nvalid) * 16; e += 32) {
          const int row = nvalid + (e >> 4), c16 = e & 15;
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          const uint32_t tf = log_decay ? 0u : 0xff80ff80u;
          const uint4 ninf = make_uint4(tf, tf, tf, tf);
          *(uint4*)(st + 0 * TILE + row * 256 + c16 * 16) = z;
          *(uint4*)(st + 1 * TILE + row * 256 + c16 * 16) = z;
          *(uint4*)(st + 2 * TILE + row * 256 + c16 * 16) = ninf;
          *(uint4*)(st + 3 * TILE + row * 256 + c16 * 16) = z;
        }
        __syncwarp();
      }
      // ---- phase A: gate, cumulative sums, decayed operands.  Lane l holds
      // channels 4l .. 4l+3 of every token of the chunk.
      const uint2* sq = (const uint2*)(st + 0 * TILE);
      const uint2* sk = (const uint2*)(st + 1 * TILE);
      const uint2* sth = (const uint2*)(st + 2 * TILE);
      f32x2 G0 = kZero, G1 = kZero;  // log2-domain cumulative log-decay
      f32x2 khr[C][2];               // Kh in fp32, for KhC once G_C is known
      float dq[C];                   // partial q_t . k_t over this lane's channels
#pragma unroll
      for (int t = 0; t < C; ++t) {
        const uint2 thw = sth[t * 32 + lane], kw = sk[t * 32 + lane], qw = sq[t * 32 + lane];
        const f32x2 k0 = bf2_to_f2(kw.x), k1 = bf2_to_f2(kw.y);
        const f32x2 q0 = bf2_to_f2(qw.x), q1 = bf2_to_f2(qw.y);
        const f32x2 x0 = mul2(bf2_to_f2(thw.x), kC2), x1 = mul2(bf2_to_f2(thw.y), kC2);
        const f32x2 d0 = add2(f2(ex2_approx(f2lo(x0)), ex2_approx(f2hi(x0))), kOne);
        const f32x2 d1 = add2(f2(ex2_approx(f2lo(x1)), ex2_approx(f2hi(x1))), kOne);
        const f32x2 g0 = log_decay ? mul2(bf2_to_f2(thw.x), kL2)
                                   : mul2(f2(rcp_approx(f2lo(d0)), rcp_approx(f2hi(d0))), kC1);
        const f32x2 g1 = log_decay ? mul2(bf2_to_f2(thw.y), kL2)
                                   : mul2(f2(rcp_approx(f2lo(d1)), rcp_approx(f2hi(d1))), kC1);
        G0 = add2(G0, g0);
        G1 = add2(G1, g1);
        const f32x2 e0 = f2(ex2_approx(f2lo(G0)), ex2_approx(f2hi(G0)));
        const f32x2 e1 = f2(ex2_approx(f2lo(G1)), ex2_approx(f2hi(G1)));
        const f32x2 r0 = f2(ex2_approx(-f2lo(G0)), ex2_approx(-f2hi(G0)));
        const f32x2 r1 = f2(ex2_approx(-f2lo(G1)), ex2_approx(-f2hi(G1)));
        const f32x2 kh0 = mul2(k0, r0), kh1 = mul2(k1, r1);
        const uint2 ktw = make_uint2(f2_to_bf2(mul2(k0, e0)), f2_to_bf2(mul2(k1, e1)));
        const uint2 qtw = make_uint2(f2_to_bf2(mul2(q0, e0)), f2_to_bf2(mul2(q1, e1)));
        const uint2 khw = make_uint2(f2_to_bf2(kh0), f2_to_bf2(kh1));
        *(uint2*)(sl + SL_XB + sw256(t, 4 * lane)) = ktw;
        *(uint2*)(sl + SL_XB + sw256(16 + t, 4 * lane)) = qtw;
        if constexpr (kTc) {
          // the tensor-core operands: [Kt; Qt] in this warp's 32 rows of the
          // shared A tile, Kh as this warp's B tile
          *(uint2*)(sm + Ly::GA + sw128(32 * iw + t, 4 * lane, GA_HALF)) = ktw;
          *(uint2*)(sm + Ly::GA + sw128(32 * iw + 16 + t, 4 * lane, GA_HALF)) = qtw;
          *(uint2*)(kh + sw128(t, 4 * lane, GB_HALF)) = khw;
        } else {
          *(uint2*)(kh + sw256(t, 4 * lane)) = khw;
        }
        khr[t][0] = kh0;
        khr[t][1] = kh1;
        const f32x2 qk = fma2(q1, k1, mul2(q0, k0));
        dq[t] = f2lo(qk) + f2hi(qk);
      }
      {
        const f32x2 c0 = f2(ex2_approx(f2lo(G0)), ex2_approx(f2hi(G0)));
        const f32x2 c1 = f2(ex2_approx(f2lo(G1)), ex2_approx(f2hi(G1)));
        *(float4*)(sl + SL_EGC + 16 * lane) = make_float4(f2lo(c0), f2hi(c0), f2lo(c1), f2hi(c1));
#pragma unroll
        for (int t = 0; t < C; ++t)
          *(uint2*)(sl + SL_KC + sw256(t, 4 * lane)) =
              make_uint2(f2_to_bf2(mul2(khr[t][0], c0)), f2_to_bf2(mul2(khr[t][1], c1)));
      }
      if constexpr (kTc) {
        // the Gram product A, P starts now and overlaps the work below
        fence_proxy_async_smem();  // the operand writes above, for the tensor core
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t ga = sbase + Ly::GA, gb = khs;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + 16 * iw, sdesc_sw128(ga + (kk >> 2) * GA_HALF + (kk & 3) * 32),
                   sdesc_sw128(gb + (kk >> 2) * GB_HALF + (kk & 3) * 32), idesc_bf16_f32(128, C),
                   kk > 0);
          mma_commit(&bars[Ly::B_GRAM + iw]);
        }
        ++gram_issued;
      }
      // V into the slot (swizzled)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i, row = e >> 4, c16 = e & 15;
        *(uint4*)(sl + SL_V + row * 256 + (((c16 ^ row) & 7) | (c16 & 8)) * 16) =
            zero_v ? make_uint4(0u, 0u, 0u, 0u) : *(const uint4*)(st + 3 * TILE + row * 256 + c16 * 16);
      }
      // q_t . k_t: transpose-reduce the 16 per-lane partial sums over the warp;
      // lane l ends with token (l >> 1) & 15
      {
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
        if ((lane & 1) == 0) ((float*)(sl + SL_DC))[(lane >> 1) & 15] = v1;
      }
      // Position-wise fallback: a chunk whose cumulative log-decay reaches
      // -G2_C > kFallbackLog2 (only possible with a given, unbounded log-decay)
      // would overflow e^{-G} in the dense tile; its A, P and KhC are formed
      // from per-pair factors e^{G_r - G_s} instead (position_wise_tiles).
      const float gmin_c = fminf(fminf(f2lo(G0), f2hi(G0)), fminf(f2lo(G1), f2hi(G1)));
      const bool fallback = kFallback && __any_sync(0xffffffffu, !(gmin_c >= -kFallbackLog2));
      // every lane has consumed its reads of the stage: refill it with this
      // warp's next chunk (a fallback chunk reads the stage once more first)
      __syncwarp();
      if (lane == 0) KTRACE(n, 7);
      auto refill = [&]() {
        if (n + kIntraWarps < nloop) {
          // the stage was only read (every value loaded from it has been used
          // by now, and __syncwarp orders the lanes' reads before this point),
          // so the copy that overwrites it needs no proxy fence
          if constexpr (kWrap) {
            // from here on the cursor is at this warp's next step
            cur = cursor_next(sc, cur, n, kIntraWarps);
            if (lane == 0) load_at(cur);
          } else {
            if (lane == 0) load(n + kIntraWarps);
          }
          ++issued;
        }
      };
      if constexpr (kFallback) {
        if (fallback) {
          position_wise_tiles(st, sl, ab, lane, beta_l, log_decay, args.g_min, G0, G1);
          __syncwarp();
        }
      }
      refill();
      // ---- phase B: A = Kt Kh^T and P = Qt Kh^T (M = N = 16, K = 128)
      if constexpr (kTc) {
        // One M = 128 tcgen05.mma per 16 channels of K, issued by lane 0 after
        // phase A: rows 32 iw .. 32 iw + 31 of the shared A tile are this
        // warp's [Kt; Qt] (the other rows belong to the other intra warps and
        // land in tensor memory lanes this warp never reads), B is this warp's
        // Kh, and the 16 result columns are this warp's own.  Waited for in
        // every chunk (the next chunk's operands overwrite the tiles it
        // reads); a position-wise chunk ignores its result.
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[Ly::B_GRAM + iw], (gram_issued - 1) & 1, abort,
                                               args.wait_ns))) {
          bad = true;
          break;
        }
        ++gram_waited;
        tc_fence_after();
        if (!fallback) {
        // lane l reads row 32 iw + l of the result: row l of A (l < 16) or row
        // l - 16 of P, 16 columns
        uint32_t dr[C];
        tmem_ld_x16(tmem + ((uint32_t)(32 * iw) << 16) + 16 * iw, dr);
        tmem_wait_ld();
        if (lane < C) {
          // strictly lower, scaled by beta of the row's token
          const int r = lane;
#pragma unroll
          for (int s4 = 0; s4 < C; s4 += 4)
            *(float4*)(ab + r * C + s4) = make_float4(
                s4 < r ? beta_l * __uint_as_float(dr[s4]) : 0.0f,
                s4 + 1 < r ? beta_l * __uint_as_float(dr[s4 + 1]) : 0.0f,
                s4 + 2 < r ? beta_l * __uint_as_float(dr[s4 + 2]) : 0.0f,
                s4 + 3 < r ? beta_l * __uint_as_float(dr[s4 + 3]) : 0.0f);
        } else {
          // strictly lower P as a bf16 high/low pair
          const int r = lane - C;
          uint32_t hw[C / 2], lw[C / 2];
#pragma unroll
          for (int s2 = 0; s2 < C; s2 += 2) {
            const float p0 = s2 < r ? __uint_as_float(dr[s2]) : 0.0f;
            const float p1 = s2 + 1 < r ? __uint_as_float(dr[s2 + 1]) : 0.0f;
            const uint32_t hi = pack_bf16x2(p0, p1);
            const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&hi);
            hw[s2 / 2] = hi;
            lw[s2 / 2] = pack_bf16x2(p0 - __low2float(hb), p1 - __high2float(hb));
          }
          *(uint4*)(sl + SL_P + sw32(r, 0)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *(uint4*)(sl + SL_P + sw32(r, 8)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          *(uint4*)(sl + SL_PL + sw32(r, 0)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          *(uint4*)(sl + SL_PL + sw32(r, 8)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        }
        // the tensor-memory read is complete before this warp's next product
        tc_fence_before();
        }
      } else if (!fallback) {
      float accA[2][4], accP[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) accA[j][c] = accP[j][c] = 0.0f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t akt[4], aqt[4], b[4];
        ldmatrix_x4(sls + SL_XB + sw256(rr + 8 * (mi & 1), 16 * kk + 8 * (mi >> 1)), akt[0], akt[1],
                    akt[2], akt[3]);
        ldmatrix_x4(sls + SL_XB + sw256(16 + rr + 8 * (mi & 1), 16 * kk + 8 * (mi >> 1)), aqt[0],
                    aqt[1], aqt[2], aqt[3]);
        ldmatrix_x4(khs + sw256(rr + 8 * (mi >> 1), 16 * kk + 8 * (mi & 1)), b[0], b[1], b[2], b[3]);
        mma16816(accA[0], akt, b[0], b[1]);
        mma16816(accA[1], akt, b[2], b[3]);
        mma16816(accP[0], aqt, b[0], b[1]);
        mma16816(accP[1], aqt, b[2], b[3]);
      }
      {
        const float br0 = __shfl_sync(0xffffffffu, beta_l, g);
        const float br1 = __shfl_sync(0xffffffffu, beta_l, g + 8);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int s0 = 8 * j + 2 * q;
          // rows g and g + 8; columns s0, s0 + 1; strictly lower parts only
          *(float2*)(ab + g * C + s0) =
              make_float2(s0 < g ? br0 * accA[j][0] : 0.0f, s0 + 1 < g ? br0 * accA[j][1] : 0.0f);
          *(float2*)(ab + (g + 8) * C + s0) = make_float2(
              s0 < g + 8 ? br1 * accA[j][2] : 0.0f, s0 + 1 < g + 8 ? br1 * accA[j][3] : 0.0f);
          // P as a bf16 high/low pair (P's rounding is the largest single
          // error source of the outputs)
          const float p0 = s0 < g ? accP[j][0] : 0.0f, p1 = s0 + 1 < g ? accP[j][1] : 0.0f;
          const float p2 = s0 < g + 8 ? accP[j][2] : 0.0f, p3 = s0 + 1 < g + 8 ? accP[j][3] : 0.0f;
          const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
          const __nv_bfloat162 b01 = *reinterpret_cast<const __nv_bfloat162*>(&h01);
          const __nv_bfloat162 b23 = *reinterpret_cast<const __nv_bfloat162*>(&h23);
          *(uint32_t*)(sl + SL_P + sw32(g, s0)) = h01;
          *(uint32_t*)(sl + SL_P + sw32(g + 8, s0)) = h23;
          *(uint32_t*)(sl + SL_PL + sw32(g, s0)) =
              pack_bf16x2(p0 - __low2float(b01), p1 - __high2float(b01));
          *(uint32_t*)(sl + SL_PL + sw32(g + 8, s0)) =
              pack_bf16x2(p2 - __low2float(b23), p3 - __high2float(b23));
        }
      }
      }  // mma.sync phase B
      __syncwarp();
      if (lane == 0) KTRACE(n, 8);
      if (lane < C) {
        // column j of (I + A)^{-1} by forward substitution, scaled by beta_j
        const int j = lane;
        float t[C];
#pragma unroll
        for (int i = 0; i < C; ++i) t[i] = (i == j) ? 1.0f : 0.0f;
#pragma unroll
        for (int i = 1; i < C; ++i) {
          float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
          for (int m4 = 0; m4 < i; m4 += 4) {
            const float4 a4 = *(const float4*)(ab + i * C + m4);
            acc0 = fmaf(a4.x, t[m4], acc0);
            if (m4 + 1 < i) acc1 = fmaf(a4.y, t[m4 + 1], acc1);
            if (m4 + 2 < i) acc0 = fmaf(a4.z, t[m4 + 2], acc0);
            if (m4 + 3 < i) acc1 = fmaf(a4.w, t[m4 + 3], acc1);
          }
          if (i > j) t[i] = -(acc0 + acc1);
        }
#pragma unroll
        for (int i = 0; i < C; ++i)
          *(__nv_bfloat16*)(sl + SL_TB + sw32(i, j)) = __float2bfloat16_rn(t[i] * beta_l);
      }
      __syncwarp();
      if (lane == 0) KTRACE(n, 9);
      // W = Tb Kt (M = 16, N = 128, K = 16); -W then replaces Kt in the slot
      {
        uint32_t atb[4];
        ldmatrix_x4(sls + SL_TB + sw32(rr + 8 * (mi & 1), 8 * (mi >> 1)), atb[0], atb[1], atb[2],
                    atb[3]);
        float accW[D / 8][4];
#pragma unroll
        for (int p = 0; p < D / 16; ++p) {
          uint32_t b[4];
          ldmatrix_x4_trans(sls + SL_XB + sw256(rr + 8 * (mi & 1), 16 * p + 8 * (mi >> 1)), b[0],
                            b[1], b[2], b[3]);
#pragma unroll
          for (int c = 0; c < 4; ++c) accW[2 * p][c] = accW[2 * p + 1][c] = 0.0f;
          mma16816(accW[2 * p], atb, b[0], b[1]);
          mma16816(accW[2 * p + 1], atb, b[2], b[3]);
        }
        __syncwarp();  // all reads of Kt are done before -W overwrites it
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
          *(uint32_t*)(sl + SL_XB + sw256(g, 8 * nt + 2 * q)) =
              pack_bf16x2(-accW[nt][0], -accW[nt][1]);
          *(uint32_t*)(sl + SL_XB + sw256(g + 8, 8 * nt + 2 * q)) =
              pack_bf16x2(-accW[nt][2], -accW[nt][3]);
        }
      }
      __syncwarp();
      // (a test job can withhold its first hand-off: the state warps' bounded
      // wait then runs out and reports KDA_ERR_DEVICE_TIMEOUT)
      if (lane == 0 && !(kJobs && n == 0 && (*sflags & kJobTestWithholdFirst))) {
        mbar_arrive(&bars[Ly::B_READY + slot]);
        KTRACE(n, 10);
      }
    }
    if (bad) fail(abort, args.status);
    // a refill issued for a chunk this warp never waited for is drained
    // before the CTA releases its shared memory
    if (lane == 0 && issued > consumed) mbar_wait_drain(full, consumed & 1, args.wait_ns);
    if constexpr (kTc) {
      // every product of this warp has completed before the tensor memory is
      // released (a bounded wait, as everywhere)
      if (gram_issued > gram_waited)
        mbar_wait_drain(&bars[Ly::B_GRAM + iw], (gram_issued - 1) & 1, args.wait_ns);
      __syncwarp();
      tc_fence_before();
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kIntraWarps) : "memory");  // the four intra warps
      tc_fence_after();
      if (iw == 0) tmem_dealloc(tmem, kTmemCols);
    }
  } else {
    // ================================================================ state warps
    if constexpr (kStateRegs > 0) set_regs<kStateRegs>();
    const int sw = warp;
    const bool identity = kJobs && (flags & kJobIdentityInit);
    // S[m][nt][c]: S^T element (value channel 32 sw + 16 m + g + 8 (c >> 1),
    // key channel 8 nt + 2 q + (c & 1)) -- the m16n8 accumulator layout
    float S[kMT][D / 8][4];
    bool bad = false;
    int n = 0;  // chunk step of this CTA
    // one piece per chain this CTA runs (the first piece runs even with no
    // steps: an empty chain's end state is its start state)
    for (int piece = 0; piece == 0 || n < nsteps; ++piece) {
      const Piece pc = sched_piece<kWrap>(sc, n);
      // the chain's states in init/final: one chain per CTA reads its offset
      // back from shared memory here and after the piece, so that no offset
      // stays live through the chunk loop
      int64_t psoff;
      float* fsp_w = nullptr;  // wrapped instantiation: the end state
      bool to_handoff = false;
      if constexpr (kWrap) {
        psoff = wrap_rt ? pc.chain * D * D : soff;
        fsp_w = final_state ? final_state + psoff : nullptr;
        to_handoff = pc.to_handoff;
      } else {
        psoff = sc.soff;
      }
      if (kWrap && pc.from_handoff) {
        // the start state is handed over by the next CTA, which runs this
        // chain's first chunks: wait for this warp's flag, then read its value
        // channels from the chain's final-state slot
        const uint32_t* f = args.hflags + ((int)blockIdx.x + 1) * kStateWarps + sw;
        const bool ok = lane == 0 ? wait_flag(f, args.epoch, abort, args.wait_ns) : true;
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          bad = true;
          break;
        }
        __syncwarp();
        if (ld_acquire_u32(f) != args.epoch) {
          bad = true;
          break;
        }
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
          for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int dv = kDvPerWarp * sw + 16 * m + g + 8 * (c >> 1), dk = 8 * nt + 2 * q + (c & 1);
              S[m][nt][c] = __ldcg(final_state + psoff + (int64_t)dk * D + dv);
            }
      } else {
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
          for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int dv = kDvPerWarp * sw + 16 * m + g + 8 * (c >> 1), dk = 8 * nt + 2 * q + (c & 1);
              S[m][nt][c] = init_state ? init_state[psoff + (int64_t)dk * D + dv]
                                       : (identity && dk == dv ? 1.0f : 0.0f);
            }
      }
    const int pend = n + pc.steps;
    // running over the piece's chunks: the chain's tokens from this chunk on,
    // and the element offset of this chunk's first output row (this lane's
    // first value channel)
    int rem = pc.len - pc.nc0 * C;
    int64_t rowbase = ((pc.row + (int64_t)pc.nc0 * C) * H + pc.head) * D + kDvPerWarp * sw + g;
    for (; n < pend; ++n, rem -= C, rowbase += (int64_t)C * H * D) {
      const int slot = n % Ly::kSlots;
      const unsigned char* sl = sm + Ly::SLOTS + slot * SLOT_BYTES;
      const uint32_t sls = sbase + Ly::SLOTS + slot * SLOT_BYTES;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&bars[Ly::B_READY + slot], (n / Ly::kSlots) & 1, abort, args.wait_ns))) {
        bad = true;
        break;
      }
      if (tid == 0) {
        KTRACE(n, 0);
        KTRACE_CLK(n, 15);
      }
      // ---- [U' | 0] = V^T Tb^T
      float accU[kMT][2][4], accO[kMT][2][4];
      {
        uint32_t tb[4];
        ldmatrix_x4(sls + SL_TB + sw32(rr + 8 * (mi >> 1), 8 * (mi & 1)), tb[0], tb[1], tb[2], tb[3]);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
          uint32_t a[4];
          ldmatrix_x4_trans(sls + SL_V + sw256(rr + 8 * (mi >> 1), kDvPerWarp * sw + 16 * m + 8 * (mi & 1)),
                            a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) accU[m][j][c] = accO[m][j][c] = 0.0f;
          mma16816(accU[m][0], a, tb[0], tb[1]);
          mma16816(accU[m][1], a, tb[2], tb[3]);
        }
      }
      // ---- [U | O] += S^T [-W | Qt]^T; S is rounded to bf16 for the product
      // and then scaled by e^{G_C} in place
      const float* egc = (const float*)(sl + SL_EGC);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t bw[4], bq[4];
        ldmatrix_x4(sls + SL_XB + sw256(rr + 8 * (mi >> 1), 16 * kk + 8 * (mi & 1)), bw[0], bw[1],
                    bw[2], bw[3]);
        ldmatrix_x4(sls + SL_XB + sw256(16 + rr + 8 * (mi >> 1), 16 * kk + 8 * (mi & 1)), bq[0],
                    bq[1], bq[2], bq[3]);
        const float2 e0 = *(const float2*)(egc + 16 * kk + 2 * q);
        const float2 e1 = *(const float2*)(egc + 16 * kk + 8 + 2 * q);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
          float* s0 = S[m][2 * kk];
          float* s1 = S[m][2 * kk + 1];
          const uint32_t a[4] = {pack_bf16x2(s0[0], s0[1]), pack_bf16x2(s0[2], s0[3]),
                                 pack_bf16x2(s1[0], s1[1]), pack_bf16x2(s1[2], s1[3])};
          {
            // the decay as packed multiplies on the accumulator pairs
            const f32x2 ev0 = f2(e0.x, e0.y), ev1 = f2(e1.x, e1.y);
            f32x2 p0 = mul2(f2(s0[0], s0[1]), ev0), p1 = mul2(f2(s0[2], s0[3]), ev0);
            f32x2 p2 = mul2(f2(s1[0], s1[1]), ev1), p3 = mul2(f2(s1[2], s1[3]), ev1);
            s0[0] = f2lo(p0);
            s0[1] = f2hi(p0);
            s0[2] = f2lo(p1);
            s0[3] = f2hi(p1);
            s1[0] = f2lo(p2);
            s1[1] = f2hi(p2);
            s1[2] = f2lo(p3);
            s1[3] = f2hi(p3);
          }
          mma16816(accU[m][0], a, bw[0], bw[1]);
          mma16816(accU[m][1], a, bw[2], bw[3]);
          mma16816(accO[m][0], a, bq[0], bq[1]);
          mma16816(accO[m][1], a, bq[2], bq[3]);
        }
      }
      // ---- U as a bf16 high/low pair of A fragments
      uint32_t uh[kMT][4], ul[kMT][4];
#pragma unroll
      for (int m = 0; m < kMT; ++m)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const float x0 = accU[m][j][2 * p], x1 = accU[m][j][2 * p + 1];
            const uint32_t hi = pack_bf16x2(x0, x1);
            const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&hi);
            uh[m][2 * j + p] = hi;
            ul[m][2 * j + p] = pack_bf16x2(x0 - __low2float(hb), x1 - __high2float(hb));
          }
      if (tid == 0) KTRACE(n, 2);
      // ---- O += U^T P^T
      {
        uint32_t pb[4];
        ldmatrix_x4(sls + SL_P + sw32(rr + 8 * (mi >> 1), 8 * (mi & 1)), pb[0], pb[1], pb[2], pb[3]);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
          mma16816(accO[m][0], uh[m], pb[0], pb[1]);
          mma16816(accO[m][1], uh[m], pb[2], pb[3]);
          mma16816(accO[m][0], ul[m], pb[0], pb[1]);
          mma16816(accO[m][1], ul[m], pb[2], pb[3]);
        }
        ldmatrix_x4(sls + SL_PL + sw32(rr + 8 * (mi >> 1), 8 * (mi & 1)), pb[0], pb[1], pb[2], pb[3]);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
          mma16816(accO[m][0], uh[m], pb[0], pb[1]);
          mma16816(accO[m][1], uh[m], pb[2], pb[3]);
        }
      }
      // ---- S^T += U^T KhC (K = 16).  Inside the sequence U enters as bf16:
      // the outputs do not see the difference (they sum over 128 key
      // channels and every chunk decays the state), but the final state is
      // returned element by element, so the last chunk adds the low part too.
#pragma unroll
      for (int p = 0; p < D / 16; ++p) {
        uint32_t b[4];
        ldmatrix_x4_trans(sls + SL_KC + sw256(rr + 8 * (mi & 1), 16 * p + 8 * (mi >> 1)), b[0], b[1],
                          b[2], b[3]);
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
          mma16816(S[m][2 * p], uh[m], b[0], b[1]);
          mma16816(S[m][2 * p + 1], uh[m], b[2], b[3]);
        }
      }
      if (rem <= C) {  // the chain's last chunk
#pragma unroll
        for (int p = 0; p < D / 16; ++p) {
          uint32_t b[4];
          ldmatrix_x4_trans(sls + SL_KC + sw256(rr + 8 * (mi & 1), 16 * p + 8 * (mi >> 1)), b[0],
                            b[1], b[2], b[3]);
#pragma unroll
          for (int m = 0; m < kMT; ++m) {
            mma16816(S[m][2 * p], ul[m], b[0], b[1]);
            mma16816(S[m][2 * p + 1], ul[m], b[2], b[3]);
          }
        }
      }
      if (tid == 0) KTRACE(n, 3);
      // ---- outputs of the chunk: O + Diag(q.k) U (after the state products
      // are issued, so that the tensor pipe works while the stores go out)
      {
        const float* dc = (const float*)(sl + SL_DC);
        const float2 dc0 = *(const float2*)(dc + 2 * q), dc1 = *(const float2*)(dc + 8 + 2 * q);
        const int nvalid = (kJobs && (*sflags & kJobNoOut)) ? 0 : min(C, rem);
        {
        // the four token rows this lane writes (j, c & 1), as element offsets of
        // its first channel; the channels then differ by constants
        int64_t rowoff[2][2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            rowoff[j][e] = rowbase + (int64_t)((8 * j + 2 * q + e) * H) * D;
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int r = 8 * j + 2 * q + (c & 1);
              const float dcr = j ? ((c & 1) ? dc1.y : dc1.x) : ((c & 1) ? dc0.y : dc0.x);
              const float o = accO[m][j][c] + dcr * accU[m][j][c];
              if (r < nvalid) {
                const int64_t idx = rowoff[j][c & 1] + 16 * m + 8 * (c >> 1);
                if constexpr (kOutBf16)
                  ((__nv_bfloat16*)args.out)[idx] = __float2bfloat16_rn(o);
                else
                  ((float*)args.out)[idx] = o;
              }
            }
        }
      }
      // the slot's reads are all consumed (their values fed the products above)
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[Ly::B_FREE + slot]);
      if (tid == 0) KTRACE(n, 4);
    }
      if (bad) break;
      float* const fsp =
          kWrap ? fsp_w : (final_state ? final_state + (int64_t)sc.soff : nullptr);  // end state
      if (fsp) {
        // the end state: the chain's final state, or the hand-over of its
        // first chunks' state to the previous CTA (through the same slot)
#pragma unroll
        for (int m = 0; m < kMT; ++m)
#pragma unroll
          for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int dv = kDvPerWarp * sw + 16 * m + g + 8 * (c >> 1), dk = 8 * nt + 2 * q + (c & 1);
              fsp[(int64_t)dk * D + dv] = S[m][nt][c];
            }
        if (to_handoff) {
          __threadfence();  // this lane's part of the state, before the flag
          __syncwarp();
          if (lane == 0) st_release_u32(args.hflags + (int)blockIdx.x * kStateWarps + sw, args.epoch);
        }
      }
    }
    if (bad) fail(abort, args.status);
  }
}

constexpr int kMaxAttrDevices = 64;
std::once_flag g_attr_once[kMaxAttrDevices];
cudaError_t g_attr_err[kMaxAttrDevices];
// The kernel's instantiations, indexed by f = out_bf16 + 2 fallback + 4 tc_gram
// (one chain per CTA: f < 8; one job per CTA: 8 + that) or 16 + out_bf16 +
// 2 fallback (wrapped schedule, mma.sync intra products).
constexpr int kInstances = 20;
template <int kMode>
constexpr void fill_instances(const void** fns) {
  fns[0] = (const void*)kda_fwd_mma_kernel<false, false, false, kMode>;
  fns[1] = (const void*)kda_fwd_mma_kernel<true, false, false, kMode>;
  fns[2] = (const void*)kda_fwd_mma_kernel<false, true, false, kMode>;
  fns[3] = (const void*)kda_fwd_mma_kernel<true, true, false, kMode>;
  if constexpr (kMode != kModeWrap) {
    fns[4] = (const void*)kda_fwd_mma_kernel<false, false, true, kMode>;
    fns[5] = (const void*)kda_fwd_mma_kernel<true, false, true, kMode>;
    fns[6] = (const void*)kda_fwd_mma_kernel<false, true, true, kMode>;
    fns[7] = (const void*)kda_fwd_mma_kernel<true, true, true, kMode>;
  }
}
const void* instance(int f) {
  static const void* fns[kInstances] = {};
  static std::once_flag once;
  std::call_once(once, []() {
    fill_instances<kModeChain>(fns);
    fill_instances<kModeJobs>(fns + 8);
    fill_instances<kModeWrap>(fns + 16);
  });
  return fns[f];
}
size_t instance_smem(int f) {
  return (f < 16 && (f & 4)) ? Lay<true>::BYTES : Lay<false>::BYTES;
}

// per device: CTAs of each instantiation that can be resident at once (0: no
// cooperative launch, so no wrapped schedule)
int g_coresident[kMaxAttrDevices][kInstances];

// Hand-over flags of the wrapped schedule: a ring of regions, one region per
// launch (chosen by the launch's epoch), so that launches in flight at the
// same time on one device use distinct flags unless kHandoffRing of them
// overlap.  A flag holds the epoch of the launch that set it last; launches
// count their epochs from 1, so the zero-initialised array holds none.
constexpr int kHandoffRing = 64;
constexpr int kMaxHandoffCtas = 512;
__device__ uint32_t g_fwd_handoff[kHandoffRing][(kMaxHandoffCtas + 1) * kStateWarps];
std::atomic<uint32_t> g_epoch{0};

}  // namespace

bool mma_supported(int dtype, int dk, int dv) {
  return dtype == KDA_DTYPE_BF16 && dk == D && dv == D;
}

int launch_mma_jobs(const FwdParams& p, const SegJob* jobs, int njobs, cudaStream_t stream,
                    uint64_t wait_ns, bool tc_gram) {
  if (!mma_supported(p.dtype, p.dk, p.dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
  const int64_t tokens = p.cu_seqlens ? (int64_t)p.T : (int64_t)p.N * p.T;
  if (tokens <= 0) {
    // nothing to load; a tensor map needs a nonzero extent, so use the SIMT
    // kernel, which handles empty sequences with no loads
    return launch_simt(p, stream);
  }
  if (tokens > INT32_MAX) return KDA_ERR_INVALID_ARG;
  CUtensorMap mq, mk, mth, mv;
  if (!encode_token_rows(&mq, p.q, p.H, tokens) || !encode_token_rows(&mk, p.k, p.H, tokens) ||
      !encode_token_rows(&mth, p.theta, p.H, tokens) || !encode_token_rows(&mv, p.v, p.H, tokens))
    return KDA_ERR_CUDA;
  // the shared-memory attribute applies to the current device's context only:
  // set it once per device
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxAttrDevices) return KDA_ERR_CUDA;
  std::call_once(g_attr_once[dev], [dev]() {
    cudaError_t err = cudaSuccess;
    for (int f = 0; f < kInstances; ++f) {
      const void* fn = instance(f);
      const int bytes = (int)instance_smem(f);
      if (err == cudaSuccess)
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      g_coresident[dev][f] = 0;
      if (err == cudaSuccess) {
        int coop = 0, nsm = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, (size_t)bytes) ==
                cudaSuccess) {
          if (coop) g_coresident[dev][f] = nsm * per_sm;
        } else {
          cudaGetLastError();  // a failed query only turns the wrapped schedule off
        }
      }
      if (kStateRegs > 0 && err == cudaSuccess) {
        // setmaxnreg.inc can only draw on the registers the block was launched
        // with: a split above the compiled launch allocation would wait forever
        cudaFuncAttributes fa;
        err = cudaFuncGetAttributes(&fa, fn);
        if (err == cudaSuccess &&
            kStateWarps * kStateRegs + kIntraWarps * kIntraRegs > fa.numRegs * (kThreads / 32))
          err = cudaErrorInvalidConfiguration;
      }
    }
    g_attr_err[dev] = err;
  });
  if (g_attr_err[dev] != cudaSuccess) return KDA_ERR_LAUNCH;
  MmaArgs a;
  a.jobs = jobs;
  a.beta = (const __nv_bfloat16*)p.beta;
  a.g_min = p.g_min;
  a.gate = p.gate;
  a.init_state = p.init_state;
  a.out = p.out;
  a.out_bf16 = p.out_dtype == KDA_DTYPE_BF16;
  a.final_state = p.final_state;
  a.cu_seqlens = p.cu_seqlens;
  a.N = p.N;
  a.H = p.H;
  a.T = p.T;
  a.status = status_word_device_ptr();
  a.wait_ns = wait_ns ? wait_ns : kWaitNs;
  if (!a.status) return KDA_ERR_CUDA;
  unsigned grid = jobs ? (unsigned)njobs : (unsigned)(p.N * p.H);
  if (grid == 0) return KDA_OK;
  const bool fb = p.gate == KDA_GATE_LOG_DECAY;
  // the instantiation (see instance())
  int f = (a.out_bf16 ? 1 : 0) + (fb ? 2 : 0) + (tc_gram ? 4 : 0) + (jobs ? 8 : 0);
  // Wrapped schedule: a fixed-length batch with more chains than CTAs that can
  // be resident at once (and not a multiple of that count) would leave SMs idle
  // in its last wave; instead, `resident` CTAs share the chains' chunks evenly
  // (the cut chains hand their state over through their final-state slots, so
  // the caller's final_state is needed).  All CTAs wait on one another's
  // flags, so they are launched cooperatively (all resident at once).  The
  // schedule is compiled for the mma.sync intra products only.
  bool wrap = false;
  a.wrap_cap = 0;
  a.epoch = 0;
  a.hflags = nullptr;
  const int fw = 16 + (a.out_bf16 ? 1 : 0) + (fb ? 2 : 0);
  const int resident = g_coresident[dev][fw];
  if (!jobs && !tc_gram && !p.cu_seqlens && p.final_state && resident > 0) {
    const int64_t chains = (int64_t)p.N * p.H;
    const int64_t pch = ((int64_t)p.T + C - 1) / C;
    const int64_t total = chains * pch;
    if (chains > resident && chains % resident != 0 && total < INT32_MAX) {
      const int64_t cap = (total + resident - 1) / resident;  // > pch: chains > resident
      const int64_t wgrid = (total + cap - 1) / cap;
      void* base = nullptr;
      if (wgrid <= kMaxHandoffCtas && cudaGetSymbolAddress(&base, g_fwd_handoff) == cudaSuccess) {
        uint32_t e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
        if (e == 0) e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
        wrap = true;
        f = fw;
        a.wrap_cap = (int)cap;
        a.epoch = e;
        a.hflags = (uint32_t*)base + (size_t)(e % kHandoffRing) * (kMaxHandoffCtas + 1) * kStateWarps;
        grid = (unsigned)wgrid;
      }
    }
  }
  void* kargs[5] = {(void*)&mq, (void*)&mk, (void*)&mth, (void*)&mv, (void*)&a};
  const size_t smem = instance_smem(f);
  const cudaError_t le =
      wrap ? cudaLaunchCooperativeKernel(instance(f), dim3(grid), dim3(kThreads), kargs, smem, stream)
           : cudaLaunchKernel(instance(f), dim3(grid), dim3(kThreads), kargs, smem, stream);
  if (le != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_LAUNCH;
  }
  return KDA_OK;
}

int launch_mma(const FwdParams& p, cudaStream_t stream, bool tc_gram) {
  return launch_mma_jobs(p, nullptr, 0, stream, 0, tc_gram);
}

}  // namespace kda

#ifdef KDA_TRACE
extern "C" KDA_API int kda_debug_trace_read_mma(void* dst, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(dst, kda::g_kda_trace_mma, bytes);
}
#endif
