// kda_tc.cu -- fused tcgen05/TMEM tensor-core path of the KDA chunked forward
// pass (bf16 q, k, v, theta, beta; dk = dv = 128; fp32 state; fp32 or bf16 out).
//
// One CTA runs one (sequence, head) chain from its first 16-token chunk to its
// last.  The fp32 state S (dk x dv) never leaves the SM: it lives in tensor
// memory transposed (TMEM lane = value channel dv, column = key channel dk),
// next to a bf16 copy that feeds the tensor core as the A operand.
//
// Per chunk n (C = 16 tokens; G = inclusive in-chunk cumulative log-decay,
// Kt = K e^{G}, Kh = K e^{-G}, Qt = Q e^{G}, KhC = K e^{G_C - G}; with
// g >= g_min = -5 every factor is at most e^{80}, finite in bf16 -- the bound
// of "Architecture Deep Dive ...", sec. 3.2 and "Kimi K3 Deep Dive", section
// "The Design" -- so the diagonal tile takes the same dense product path as
// every other tile):
//
//   A   = strict_lower(Diag(beta) Kt Kh^T)      P = strict_lower(Qt Kh^T)
//   Tb  = (I + A)^{-1} Diag(beta)               W = Tb Kt
//   U   = Tb V - W S                            O = Qt S + P U + Diag(q_t . k_t) U
//   S  <- Diag(e^{G_C}) S + KhC^T U
//
// The diagonal of Qt Kh^T is q_t . k_t exactly (the decay factors cancel), so
// it is taken in fp32 from the bf16 inputs and applied to U in fp32; every
// other product uses bf16 operands with fp32 accumulation, U as a bf16
// high/low pair.  (The outputs are heavy-tailed -- max |o| is ~15x RMS -- and
// the largest ones are dominated by the token's own term, which this keeps in
// fp32.)
//
// Warp roles (256 threads, two warps per SM sub-partition):
//   warps 0..3   state group: the sequential chain.  One elected lane issues
//                the chain's tcgen05.mma; hand-offs inside the group are named
//                barriers.  Per chunk: U readout, state/output products,
//                state pass (bf16 copy first, then the fp32 state scaled by
//                e^{G_C} of the next chunk), outputs, final state.
//                Warp 0 owns the TMEM allocation.
//   warps 4..7   intra group: TMA loads of q, k, theta, v tiles into a 4-stage
//                ring (one lane refills a stage as soon as the group has
//                consumed it); gate g = g_min*sigmoid(theta), cumulative sum
//                and decayed operands in fp32 (two channels per thread, packed
//                f32x2 arithmetic), V^T into TMEM, q.k diagonals; one lane
//                issues the A/P product of four chunks (M = 128 rows =
//                [Kt_c; Qt_c] for c = 0..3, N = 64 = Kh of the four chunks);
//                then per chunk the triangular inverse (fp32 forward
//                substitution), Tb, P and W = Tb Kt (warp-level mma.sync).
//
// Tensor-core products per chunk (M = 128 = dv lanes, K-major operands):
//   [U' | 0]   = V^T [Tb | 0]^T          (A = V^T in TMEM, N = 32, K = 16)
//   [U  | O]  += S^T [-W | Qt]^T         (A = bf16 S^T in TMEM, N = 32, K = 128,
//                                         two accumulators of K = 64 each)
//   S^T       += U^T KhC                 (A = bf16 U^T hi and lo, N = 128, K = 16)
//   O         += U^T P^T                 (N = 16, K = 16)
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

constexpr int C = kChunk;                    // 16
constexpr int D = 128;                       // dk = dv
constexpr int NS = 4;                        // TMA ring stages (one chunk each)
constexpr int NSLOT = 8;                     // per-chunk operand slots (two groups)
constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait
constexpr float kLog2e = 1.4426950408889634f;

// tensor memory columns (512 allocated)
constexpr uint32_t TM_S = 0;      // fp32 dS^T = (KhC^T U)^T of a chunk, 128 columns
constexpr uint32_t TM_SBF = 128;  // bf16 S^T (A operand), 64 columns
constexpr uint32_t TM_AP = 192;   // A/P tiles of a group of 4 chunks, 64 columns
constexpr uint32_t TM_UA = 256;   // [U | O] accumulator A (K = 0..63), 2 buffers x 32
constexpr uint32_t TM_UB = 320;   // [U | O] accumulator B (K = 64..127), 2 buffers x 32
constexpr uint32_t TM_UBF = 384;  // bf16 U^T (A operand): high 8 columns, low 8 columns
constexpr uint32_t TM_VT = 400;   // bf16 V^T (A operand), NSLOT buffers x 8 columns
constexpr uint32_t TM_COLS = 512;
static_assert(TM_VT + 8 * NSLOT <= TM_COLS, "tensor memory budget");

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t TILE = C * D * 2;                     // 4096: one 16 x 128 bf16 tile
constexpr uint32_t SM_RING = 0;                          // NS x {q, k, theta, v}
constexpr uint32_t SM_GA = SM_RING + NS * 4 * TILE;      // 2 x [128 x 128] bf16, SW128
constexpr uint32_t GA_BYTES = 128 * D * 2;
constexpr uint32_t SM_GB = SM_GA + 2 * GA_BYTES;         // [64 x 128] bf16, SW128
constexpr uint32_t GB_BYTES = 64 * D * 2;
constexpr uint32_t SM_KC = SM_GB + GB_BYTES;             // NSLOT x [128 x 16] bf16
constexpr uint32_t SM_P = SM_KC + NSLOT * TILE;          // NSLOT x [16 x 16] bf16
constexpr uint32_t SM_TB = SM_P + NSLOT * 512;           // NSLOT x [32 x 16] bf16
constexpr uint32_t SM_EGC = SM_TB + NSLOT * 1024;        // NSLOT x 128 fp32
constexpr uint32_t SM_BETA = SM_EGC + NSLOT * D * 4;     // NSLOT x 16 fp32
constexpr uint32_t SM_DIAG = SM_BETA + NSLOT * C * 4;    // NSLOT x 16 fp32 (q_t . k_t)
constexpr uint32_t SM_DPART = SM_DIAG + NSLOT * C * 4;   // 4 warps x 16 fp32 partial sums
constexpr uint32_t SM_XCH = SM_DPART + 4 * C * 4;        // 2 halves x 64 channel pairs x f32x2
constexpr uint32_t SM_ABUF = SM_XCH + 2 * 64 * 8;        // 4 warps x [16 x 17] fp32
constexpr uint32_t SM_BARS = SM_ABUF + 4 * C * 17 * 4;   // mbarriers
constexpr int NBARS = 48;
constexpr uint32_t SM_MISC = SM_BARS + NBARS * 8;        // tmem base, abort flag
constexpr uint32_t SM_RANK = SM_MISC + 16;               // chain-order scratch
constexpr uint32_t SM_TOTAL = SM_RANK + (kMaxRankedSeqsDev + 1) * 4;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;         // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(SM_GA % 1024 == 0 && SM_GB % 1024 == 0, "SW128 tiles must be 1024-aligned");

// barrier indices
constexpr int B_FULL = 0;     // [NS]    TMA -> intra
constexpr int B_GATE = 8;     // [NSLOT] intra phase A of chunk n done -> state group
constexpr int B_CHUNK = 16;   // [NSLOT] intra phase B of chunk n done -> state issuer
constexpr int B_GFREE = 24;   // [2]     state issuer: group's products done -> intra
constexpr int B_APDONE = 26;  //         A/P product done -> intra
constexpr int B_X = 27;       //         [U | O] products of chunk n done -> state group
constexpr int B_SO = 28;      //         state and output products of chunk n done
constexpr int B_DRAIN = 29;   //         state issuer final drain
constexpr int B_DRAIN2 = 30;  //         intra issuer final drain

// named barriers
constexpr uint32_t NB_INTRA = 1, NB_STATE = 2;

// byte offset of element (row, col) in a SW128 K-major tile with `rows` rows
__device__ __forceinline__ uint32_t sw128(int row, int col, int rows) {
  return (uint32_t)((col >> 6) * rows * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                    (col & 7) * 2);
}

struct TcArgs {
  const __nv_bfloat16* beta;
  float g_min;
  const float* init_state;
  void* out;
  int out_bf16;
  float* final_state;
  const int32_t* cu_seqlens;
  int N, H, T;
  int* status;
};

// Optional event trace of the first CTA (compile with -DKDA_TRACE): wall-clock
// time of each pipeline event per chunk, read back with kda_debug_trace_read.
constexpr int kTraceChunks = 512;
static_assert(kTraceChunks > 0, "trace size");
#ifdef KDA_TRACE
__device__ unsigned long long g_kda_trace[kTraceChunks * 16];
#define KTRACE(n, k)                                                                          \
  do {                                                                                        \
    if (blockIdx.x == 0 && (n) < kTraceChunks) g_kda_trace[(n) * 16 + (k)] = globaltimer_ns(); \
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

__global__ void __launch_bounds__(kThreads, 1)
    kda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_th,
                      const __grid_constant__ CUtensorMap tm_v, const TcArgs args) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + SM_BARS);
  uint32_t* tmem_slot = (uint32_t*)(sm + SM_MISC);
  volatile int* abort = (volatile int*)(sm + SM_MISC + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const Chain ch = chain_for_block(blockIdx.x, args.H, args.N, args.T, args.cu_seqlens,
                                   (int*)(sm + SM_RANK));
  const int h = ch.head;
  const int H = args.H;
  const int L = (int)(ch.t1 - ch.t0);
  const int nchunks = (L + C - 1) / C;
  const int ngroups = (nchunks + 3) / 4;

  if (tid == 0) {
    for (int i = 0; i < NBARS; ++i) mbar_init(&bars[i], 1);
    *abort = 0;
    fence_mbar_init();
  }
  // zero rows 16..31 of every Tb tile (the zero half of [Tb | 0]): per slot and
  // k-group, bytes [256, 512) of the 512-byte k-group block
  for (int e = tid; e < NSLOT * 128; e += kThreads) {
    const int slot = e >> 7, kg = (e >> 6) & 1, w = e & 63;
    *(uint32_t*)(sm + SM_TB + slot * 1024 + kg * 512 + 256 + w * 4) = 0u;
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
  const uint32_t sbase = smem_u32(sm);

  if (warp >= 4) {
    // ================================================================ intra group
    const int it = tid - 128;         // 0..127
    const int q4 = warp & 3;          // TMEM lane quarter of this warp
    const int wq = warp - 4;          // warp index inside the group
    const int hf = wq >> 1;           // token half of this warp: rows 8hf .. 8hf+7
    const int cp = 32 * (wq & 1) + lane;  // channel pair: channels 2cp, 2cp+1
    const f32x2 kC2 = f2(-kLog2e, -kLog2e);
    const f32x2 kC1 = f2(args.g_min * kLog2e, args.g_min * kLog2e);
    const f32x2 kOne = f2(1.0f, 1.0f);
    const f32x2 kZero = 0ull;
    f32x2* xch = (f32x2*)(sm + SM_XCH);      // per-half cumulative-sum totals
    float* dpart = (float*)(sm + SM_DPART);  // per-warp q.k partial sums of a chunk
    // TMA loads of chunk m into ring stage m % NS (issued by one lane)
    auto load_chunk = [&](int m) {
      const int s = m % NS;
      mbar_arrive_expect_tx(&bars[B_FULL + s], 4 * TILE);
      KTRACE(m, 0);
      unsigned char* st = sm + SM_RING + s * 4 * TILE;
      const int row = (int)(ch.t0 + (int64_t)m * C);
      tma_load_3d(st + 0 * TILE, &tm_q, 0, h, row, &bars[B_FULL + s]);
      tma_load_3d(st + 1 * TILE, &tm_k, 0, h, row, &bars[B_FULL + s]);
      tma_load_3d(st + 2 * TILE, &tm_th, 0, h, row, &bars[B_FULL + s]);
      tma_load_3d(st + 3 * TILE, &tm_v, 0, h, row, &bars[B_FULL + s]);
    };
    int issued = 0;
    if (it == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_th);
      prefetch_tmap(&tm_v);
      for (; issued < NS && issued < nchunks; ++issued) load_chunk(issued);
    }
    bool bad = false;
    for (int g = 0; g < ngroups; ++g) {
      const int gb = g & 1;
      unsigned char* GA = sm + SM_GA + gb * GA_BYTES;
      if (g >= 2 && !bad && !mbar_wait(&bars[B_GFREE + gb], ((g >> 1) - 1) & 1, abort, kWaitNs))
        bad = true;
      // ---- phase A: gate, cumulative sum, decayed operands of the group's chunks.
      // Warps 0,1 of the group take tokens 0..7, warps 2,3 tokens 8..15; each
      // warp covers 64 channels (a full 128-byte row span: conflict-free).
      bool stop = false;
      for (int cc = 0; cc < 4; ++cc) {
        const int n = 4 * g + cc;
        if (n >= nchunks) break;
        const int s = n % NS, slot = n % NSLOT;
        const int nvalid = min(C, L - n * C);
        // beta of this chunk: the global load is issued first so that its
        // latency hides behind the rest of phase A
        unsigned short beta_r = 0;
        if (it < nvalid)
          beta_r = reinterpret_cast<const unsigned short*>(args.beta)[(ch.t0 + (int64_t)n * C + it) * H + h];
        if (!bad && !mbar_wait(&bars[B_FULL + s], (n / NS) & 1, abort, kWaitNs)) bad = true;
        if (it == 0) KTRACE(n, 1);
        const unsigned char* st = sm + SM_RING + s * 4 * TILE;
        const uint32_t* sq = (const uint32_t*)(st + 0 * TILE);
        const uint32_t* sk = (const uint32_t*)(st + 1 * TILE);
        const uint32_t* sth = (const uint32_t*)(st + 2 * TILE);
        const unsigned short* sv = (const unsigned short*)(st + 3 * TILE);
        f32x2 Gr[8], kr[8], qr[8];
        f32x2 G2 = kZero;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 8 * hf + i;
          const bool valid = r < nvalid;
          const f32x2 th = bf2_to_f2(sth[r * 64 + cp]);
          kr[i] = valid ? bf2_to_f2(sk[r * 64 + cp]) : kZero;
          qr[i] = valid ? bf2_to_f2(sq[r * 64 + cp]) : kZero;
          const f32x2 x = mul2(th, kC2);
          const f32x2 den = add2(f2(ex2_approx(f2lo(x)), ex2_approx(f2hi(x))), kOne);
          const f32x2 g2 = mul2(f2(rcp_approx(f2lo(den)), rcp_approx(f2hi(den))), kC1);
          G2 = add2(G2, valid ? g2 : kZero);  // log2-domain cumulative log-decay
          Gr[i] = G2;
        }
        // exchange the half totals: the second half adds the first half's total,
        // both need the chunk total
        xch[hf * 64 + cp] = G2;
        if (bar_sync_or(NB_INTRA, 128, bad || *abort)) {
          stop = true;
          break;
        }
        if (it == 0) KTRACE(n, 9);
        const f32x2 other = xch[(1 - hf) * 64 + cp];
        if (hf) {
#pragma unroll
          for (int i = 0; i < 8; ++i) Gr[i] = add2(Gr[i], other);
        }
        const f32x2 GT = add2(G2, other);  // chunk total (same in both halves)
        const f32x2 eGC = f2(ex2_approx(f2lo(GT)), ex2_approx(f2hi(GT)));
        uint32_t kc0[4], kc1[4];
        float dq[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 8 * hf + i;
          const f32x2 eg = f2(ex2_approx(f2lo(Gr[i])), ex2_approx(f2hi(Gr[i])));
          const f32x2 emg = f2(ex2_approx(-f2lo(Gr[i])), ex2_approx(-f2hi(Gr[i])));
          const f32x2 kt = mul2(kr[i], eg), qt = mul2(qr[i], eg), kh = mul2(kr[i], emg);
          *(uint32_t*)(GA + sw128(32 * cc + r, 2 * cp, 128)) = f2_to_bf2(kt);
          *(uint32_t*)(GA + sw128(32 * cc + 16 + r, 2 * cp, 128)) = f2_to_bf2(qt);
          *(uint32_t*)(sm + SM_GB + sw128(16 * cc + r, 2 * cp, 64)) = f2_to_bf2(kh);
          const f32x2 khc = mul2(kh, eGC);
          if (i & 1) {
            kc0[i >> 1] = pack_bf16x2(__uint_as_float(kc0[i >> 1]), f2lo(khc));
            kc1[i >> 1] = pack_bf16x2(__uint_as_float(kc1[i >> 1]), f2hi(khc));
          } else {
            kc0[i >> 1] = __float_as_uint(f2lo(khc));
            kc1[i >> 1] = __float_as_uint(f2hi(khc));
          }
          const f32x2 qk = mul2(qr[i], kr[i]);
          dq[i] = f2lo(qk) + f2hi(qk);
        }
        {
          // KhC^T tile: row = key channel, 16 tokens along K (no swizzle);
          // this thread holds channels 2cp, 2cp+1 and tokens 8hf .. 8hf+7
          unsigned char* kc = sm + SM_KC + slot * TILE + hf * 2048;
          const int c0 = 2 * cp, c1 = 2 * cp + 1;
          *(uint4*)(kc + (c0 & 7) * 16 + (c0 >> 3) * 128) = make_uint4(kc0[0], kc0[1], kc0[2], kc0[3]);
          *(uint4*)(kc + (c1 & 7) * 16 + (c1 >> 3) * 128) = make_uint4(kc1[0], kc1[1], kc1[2], kc1[3]);
          if (hf == 0)
            *(float2*)(sm + SM_EGC + slot * D * 4 + c0 * 4) = make_float2(f2lo(eGC), f2hi(eGC));
        }
        {
          // q_t . k_t over this warp's 64 channels: reduce 8 rows over the 32
          // lanes, one row per group of four lanes
          const int b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
          float v4[4], v2[2], v1;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float send = b4 ? dq[j] : dq[j + 4];
            const float keep = b4 ? dq[j + 4] : dq[j];
            v4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float send = b3 ? v4[j] : v4[j + 2];
            const float keep = b3 ? v4[j + 2] : v4[j];
            v2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
          }
          {
            const float send = b2 ? v2[0] : v2[1];
            const float keep = b2 ? v2[1] : v2[0];
            v1 = keep + __shfl_xor_sync(0xffffffffu, send, 4);
          }
          v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
          v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
          if ((lane & 3) == 0) dpart[wq * C + 8 * hf + 4 * b4 + 2 * b3 + b2] = v1;
        }
        if (it < C) ((unsigned short*)(sm + SM_BETA + slot * C * 4))[it] = beta_r;
        {
          // V^T into tensor memory: TMEM lane = value channel 32*q4 + lane,
          // 16 tokens packed two per 32-bit column
          const int dv = 32 * q4 + lane;
          uint32_t w[8];
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const uint32_t v0 = (2 * p < nvalid) ? (uint32_t)sv[(2 * p) * D + dv] : 0u;
            const uint32_t v1 = (2 * p + 1 < nvalid) ? (uint32_t)sv[(2 * p + 1) * D + dv] : 0u;
            w[p] = v0 | (v1 << 16);
          }
          __syncwarp();
          tmem_st_x8(tmem + ((uint32_t)(q4 * 32) << 16) + TM_VT + 8 * slot, w);
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (it == 0) KTRACE(n, 14);
        if (bar_sync_or(NB_INTRA, 128, bad || *abort)) {
          stop = true;
          break;
        }
        if (wq == 0) {
          // q.k of each token: the two half-warps' partial sums
          if (lane < C) {
            const int w0 = 2 * (lane >> 3);
            ((float*)(sm + SM_DIAG + slot * C * 4))[lane] = dpart[w0 * C + lane] + dpart[(w0 + 1) * C + lane];
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bars[B_GATE + slot]);
            KTRACE(n, 2);
            if (n + NS < nchunks) {
              // the whole group has consumed stage s: refill it
              load_chunk(n + NS);
              issued = n + NS + 1;
            }
            KTRACE(n, 15);
          }
        }
      }
      if (stop) break;
      // ---- the group's A/P tiles in one product, issued by one lane
      if (it == 0) {
        tc_fence_after();
        const uint32_t ga = sbase + SM_GA + gb * GA_BYTES, gbb = sbase + SM_GB;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint64_t a = sdesc_sw128(ga + (kk >> 2) * (128 * 128) + (kk & 3) * 32);
          uint64_t b = sdesc_sw128(gbb + (kk >> 2) * (64 * 128) + (kk & 3) * 32);
          mma_ss(tmem + TM_AP, a, b, idesc_bf16_f32(128, 64), kk > 0);
        }
        mma_commit(&bars[B_APDONE]);
        KTRACE(4 * g, 11);
      }
      // ---- phase B: this warp's chunk of the group (lane quarter q4 holds its A/P rows)
      const int n = 4 * g + q4;
      if (n < nchunks) {
        const int slot = n % NSLOT;
        if (!bad && !mbar_wait(&bars[B_APDONE], g & 1, abort, kWaitNs)) bad = true;
        if (lane == 0) KTRACE(n, 3);
        __syncwarp();
        tc_fence_after();
        uint32_t raw[16];
        tmem_ld_x16(tmem + ((uint32_t)(q4 * 32) << 16) + TM_AP + 16 * q4, raw);
        tmem_wait_ld();
        float* Ab = (float*)(sm + SM_ABUF) + q4 * (C * 17);
        const __nv_bfloat16* bet = (const __nv_bfloat16*)(sm + SM_BETA + slot * C * 4);
        unsigned char* Pt = sm + SM_P + slot * 512;
        unsigned char* Tb = sm + SM_TB + slot * 1024;
        if (lane < 16) {
          const int i = lane;
          const float bi = __bfloat162float(bet[i]);
#pragma unroll
          for (int j = 0; j < C; ++j) Ab[i * 17 + j] = (j < i) ? bi * __uint_as_float(raw[j]) : 0.0f;
        } else {
          // strictly lower P (the diagonal is applied exactly by the state group)
          const int i = lane - 16;
          uint32_t w[8];
#pragma unroll
          for (int p = 0; p < 8; ++p)
            w[p] = pack_bf16x2((2 * p < i) ? __uint_as_float(raw[2 * p]) : 0.0f,
                               (2 * p + 1 < i) ? __uint_as_float(raw[2 * p + 1]) : 0.0f);
          unsigned char* pr = Pt + (i & 7) * 16 + (i >> 3) * 128;
          *(uint4*)(pr) = make_uint4(w[0], w[1], w[2], w[3]);
          *(uint4*)(pr + 256) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        __syncwarp();
        if (lane < 16) {
          // column j of (I + A)^{-1} by forward substitution, then scaled by beta_j
          const int j = lane;
          float t[C];
#pragma unroll
          for (int i = 0; i < C; ++i) t[i] = (i == j) ? 1.0f : 0.0f;
#pragma unroll
          for (int i = 1; i < C; ++i) {
            float acc0 = 0.0f, acc1 = 0.0f;  // two partial sums: shorter dependency chain
#pragma unroll
            for (int m = 0; m < i; m += 2) {
              acc0 = fmaf(Ab[i * 17 + m], t[m], acc0);
              if (m + 1 < i) acc1 = fmaf(Ab[i * 17 + m + 1], t[m + 1], acc1);
            }
            if (i > j) t[i] = -(acc0 + acc1);
          }
          const float bj = __bfloat162float(bet[j]);
#pragma unroll
          for (int i = 0; i < C; ++i)
            *(__nv_bfloat16*)(Tb + (i & 7) * 16 + (i >> 3) * 128 + (j >> 3) * 512 + (j & 7) * 2) =
                __float2bfloat16_rn(t[i] * bj);
        }
        __syncwarp();
        // W = Tb Kt (16 x 128) with mma.sync; -W overwrites the Kt rows of this chunk
        {
          const uint32_t tb_s = smem_u32(Tb);
          const int mi = lane >> 3, rr = lane & 7;
          uint32_t afr[4];
          ldmatrix_x4(tb_s + (mi & 1) * 128 + (mi >> 1) * 512 + rr * 16, afr[0], afr[1], afr[2],
                      afr[3]);
          const uint32_t ga_s = smem_u32(GA);
#pragma unroll
          for (int grp = 0; grp < 4; ++grp) {
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
              for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
              const int nt = 4 * grp + 2 * pr;
              const int tok = (mi & 1) * 8 + rr;
              const int R = 32 * q4 + tok;
              const int col = 8 * (nt + (mi >> 1));
              uint32_t b0, b1, b2, b3;
              ldmatrix_x4_trans(ga_s + sw128(R, col, 128), b0, b1, b2, b3);
              mma_bf16_16816(acc[2 * pr], afr, b0, b1);
              mma_bf16_16816(acc[2 * pr + 1], afr, b2, b3);
            }
#pragma unroll
            for (int t4 = 0; t4 < 4; ++t4) {
              const int col = 8 * (4 * grp + t4) + 2 * (lane & 3);
#pragma unroll
              for (int hf2 = 0; hf2 < 2; ++hf2) {
                const int R = 32 * q4 + (lane >> 2) + 8 * hf2;
                *(uint32_t*)(GA + sw128(R, col, 128)) =
                    pack_bf16x2(-acc[t4][2 * hf2], -acc[t4][2 * hf2 + 1]);
              }
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[B_CHUNK + slot]);
          KTRACE(n, 4);
        }
      }
    }
    if (bad) fail(abort, args.status);
    if (it == 0) {
      // drain the A/P products this group issued, and every TMA load in flight
      mma_commit(&bars[B_DRAIN2]);
      mbar_wait_drain(&bars[B_DRAIN2], 0, kWaitNs);
      for (int m = issued - NS < 0 ? 0 : issued - NS; m < issued; ++m)
        mbar_wait_drain(&bars[B_FULL + m % NS], (m / NS) & 1, kWaitNs);
    }
  } else {
    // ================================================================ state group
    const int q4 = warp & 3;
    const int dv = q4 * 32 + lane;
    const uint32_t lb = (uint32_t)(q4 * 32) << 16;
    const bool issuer = (tid == 0);
    const int64_t soff = ((int64_t)ch.seq * H + h) * D * D;
    bool bad = false;
    if (nchunks > 0) {
      // The fp32 state row of this thread (value channel dv, key channels 0..127)
      // lives in registers; TMEM holds its bf16 copy (the A operand of the
      // state products) and receives dS = U^T KhC from the tensor core.
      float S[D];
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_GATE + 0], 0, abort, kWaitNs))) bad = true;
#pragma unroll
      for (int i = 0; i < D; ++i)
        S[i] = args.init_state ? args.init_state[soff + (int64_t)i * D + dv] : 0.0f;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        uint32_t b16[16];
#pragma unroll
        for (int p = 0; p < 16; ++p) b16[p] = pack_bf16x2(S[32 * blk + 2 * p], S[32 * blk + 2 * p + 1]);
        tmem_st_x16(tmem + lb + TM_SBF + 16 * blk, b16);
      }
      tmem_wait_st();
      tc_fence_before();

      // issue the [U' | 0] and [U | O] products of chunk m into buffer m & 1
      auto issue_x = [&](int m) -> bool {
        const int slot = m % NSLOT, b = m & 1, cc = m & 3, g = m >> 2;
        if (!mbar_wait(&bars[B_CHUNK + slot], (m / NSLOT) & 1, abort, kWaitNs)) return false;
        KTRACE(m, 10);
        tc_fence_after();
        const uint32_t ua = tmem + TM_UA + 32 * b, ub = tmem + TM_UB + 32 * b;
        mma_ts(ua, tmem + TM_VT + 8 * slot, sdesc_noswz(sbase + SM_TB + slot * 1024, 512, 128),
               idesc_bf16_f32(128, 32), 0);
        const uint32_t ga = sbase + SM_GA + (g & 1) * GA_BYTES + cc * 32 * 128;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // accumulator A: K = 0..63 (k-atom 0); accumulator B: K = 64..127 (k-atom 1)
          mma_ts(ua, tmem + TM_SBF + 8 * kk, sdesc_sw128(ga + kk * 32), idesc_bf16_f32(128, 32), 1);
          mma_ts(ub, tmem + TM_SBF + 8 * (kk + 4), sdesc_sw128(ga + 128 * 128 + kk * 32),
                 idesc_bf16_f32(128, 32), kk > 0);
        }
        mma_commit(&bars[B_X]);
        return true;
      };

      if (bar_sync_or(NB_STATE, 128, bad || *abort)) bad = true;
      if (!bad && issuer && !issue_x(0)) fail(abort, args.status);

      for (int n = 0; n < nchunks && !bad; ++n) {
        const int b = n & 1, slot = n % NSLOT;
        const uint32_t ua = tmem + lb + TM_UA + 32 * b, ub = tmem + lb + TM_UB + 32 * b;
        // ---- U = U' - W S (two partial accumulators), as bf16 high/low for the products
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_X], n & 1, abort, kWaitNs))) bad = true;
        if (issuer) KTRACE(n, 5);
        tc_fence_after();
        {
          uint32_t ra[16], rb[16], w[16];
          tmem_ld_x16(ua, ra);
          tmem_ld_x16(ub, rb);
          tmem_wait_ld();
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const float x0 = __uint_as_float(ra[2 * p]) + __uint_as_float(rb[2 * p]);
            const float x1 = __uint_as_float(ra[2 * p + 1]) + __uint_as_float(rb[2 * p + 1]);
            w[p] = pack_bf16x2(x0, x1);
            const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&w[p]);
            w[8 + p] = pack_bf16x2(x0 - __low2float(hb), x1 - __high2float(hb));
          }
          tmem_st_x16(tmem + lb + TM_UBF, w);
          tmem_wait_st();
        }
        tc_fence_before();
        if (bar_sync_or(NB_STATE, 128, bad || *abort)) {
          bad = true;
          break;
        }
        if (issuer) {
          KTRACE(n, 6);
          tc_fence_after();
          const uint64_t kc = sdesc_noswz(sbase + SM_KC + slot * TILE, 2048, 128);
          const uint64_t pp = sdesc_noswz(sbase + SM_P + slot * 512, 256, 128);
          mma_ts(tmem + TM_S, tmem + TM_UBF, kc, idesc_bf16_f32(128, 128), 0);
          mma_ts(tmem + TM_UA + 32 * b + 16, tmem + TM_UBF, pp, idesc_bf16_f32(128, 16), 1);
          mma_ts(tmem + TM_S, tmem + TM_UBF + 8, kc, idesc_bf16_f32(128, 128), 1);
          mma_ts(tmem + TM_UA + 32 * b + 16, tmem + TM_UBF + 8, pp, idesc_bf16_f32(128, 16), 1);
          mma_commit(&bars[B_SO]);
        }
        // e^{G_C} of this chunk; its slot is recycled only after the group's
        // release, which follows this chunk's outputs
        const float4* eg = (const float4*)(sm + SM_EGC + slot * D * 4);
        // ---- wait for dS = U^T KhC, then S <- e^{G_C} S + dS and its bf16 copy
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_SO], n & 1, abort, kWaitNs))) {
          bad = true;
          break;
        }
        if (issuer) KTRACE(n, 7);
        tc_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t ds[64];
          tmem_ld_x32(tmem + lb + TM_S + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&ds[0]));
          tmem_ld_x32(tmem + lb + TM_S + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&ds[32]));
          tmem_wait_ld();
#pragma unroll
          for (int i4 = 0; i4 < 16; ++i4) {
            const float4 e = eg[16 * half + i4];  // shared-memory broadcast
            const int i = 64 * half + 4 * i4;
            S[i + 0] = fmaf(S[i + 0], e.x, __uint_as_float(ds[4 * i4 + 0]));
            S[i + 1] = fmaf(S[i + 1], e.y, __uint_as_float(ds[4 * i4 + 1]));
            S[i + 2] = fmaf(S[i + 2], e.z, __uint_as_float(ds[4 * i4 + 2]));
            S[i + 3] = fmaf(S[i + 3], e.w, __uint_as_float(ds[4 * i4 + 3]));
          }
          if (n + 1 < nchunks) {
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
              uint32_t b16[16];
              const int i0 = 64 * half + 32 * blk;
#pragma unroll
              for (int p = 0; p < 16; ++p) b16[p] = pack_bf16x2(S[i0 + 2 * p], S[i0 + 2 * p + 1]);
              tmem_st_x16(tmem + lb + TM_SBF + 32 * half + 16 * blk, b16);
            }
          }
        }
        if (n + 1 < nchunks) {
          tmem_wait_st();
          tc_fence_before();
          if (bar_sync_or(NB_STATE, 128, bad || *abort)) {
            bad = true;
            break;
          }
          if (issuer) {
            KTRACE(n, 8);
            // the previous group's slots may be recycled: its outputs are done
            if ((n & 3) == 0 && n > 0) mma_commit(&bars[B_GFREE + (((n >> 2) - 1) & 1)]);
            if (!issue_x(n + 1)) fail(abort, args.status);
            KTRACE(n + 1, 13);
          }
        }
        // ---- outputs of chunk n: O = [Qt S]_A + [Qt S]_B + P U + (q.k) U, with U
        // re-read from its accumulators and q.k from the intra group's partial sums
        {
          uint32_t oa[16], ob[16], ra[16], rb[16];
          tmem_ld_x16(ua + 16, oa);
          tmem_ld_x16(ub + 16, ob);
          tmem_ld_x16(ua, ra);
          tmem_ld_x16(ub, rb);
          const float4* dp4 = (const float4*)(sm + SM_DIAG + slot * C * 4);
          float Dc[16];
#pragma unroll
          for (int t4 = 0; t4 < 4; ++t4) {
            const float4 a0 = dp4[t4];
            Dc[4 * t4 + 0] = a0.x;
            Dc[4 * t4 + 1] = a0.y;
            Dc[4 * t4 + 2] = a0.z;
            Dc[4 * t4 + 3] = a0.w;
          }
          tmem_wait_ld();
          float Uc[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) Uc[t] = __uint_as_float(ra[t]) + __uint_as_float(rb[t]);
          const int nvalid = min(C, L - n * C);
          const int64_t row0 = ch.t0 + (int64_t)n * C;
          if (args.out_bf16) {
            __nv_bfloat16* out = (__nv_bfloat16*)args.out;
#pragma unroll
            for (int i = 0; i < C; ++i)
              if (i < nvalid)
                out[((row0 + i) * H + h) * D + dv] = __float2bfloat16_rn(
                    __uint_as_float(oa[i]) + __uint_as_float(ob[i]) + Dc[i] * Uc[i]);
          } else {
            float* out = (float*)args.out;
#pragma unroll
            for (int i = 0; i < C; ++i)
              if (i < nvalid)
                out[((row0 + i) * H + h) * D + dv] =
                    __uint_as_float(oa[i]) + __uint_as_float(ob[i]) + Dc[i] * Uc[i];
          }
          if (issuer) KTRACE(n, 12);
        }
      }
      if (issuer) mma_commit(&bars[B_GFREE + (((nchunks - 1) >> 2) & 1)]);
      if (!bad && args.final_state) {
#pragma unroll
        for (int i = 0; i < D; ++i) args.final_state[soff + (int64_t)i * D + dv] = S[i];
      }
      if (bad) fail(abort, args.status);
      if (issuer) {
        mma_commit(&bars[B_DRAIN]);
        mbar_wait_drain(&bars[B_DRAIN], 0, kWaitNs);
      }
    } else if (args.final_state) {
      // empty sequence: the final state is the initial state
      for (int i = 0; i < D; ++i)
        args.final_state[soff + (int64_t)i * D + dv] =
            args.init_state ? args.init_state[soff + (int64_t)i * D + dv] : 0.0f;
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

}  // namespace

bool tc_supported(int dtype, int dk, int dv) {
  return dtype == KDA_DTYPE_BF16 && dk == D && dv == D;
}

int launch_tc(const FwdParams& p, cudaStream_t stream) {
  if (!tc_supported(p.dtype, p.dk, p.dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
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
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, []() {
    attr_err = cudaFuncSetAttribute(kda_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return KDA_ERR_LAUNCH;
  TcArgs a;
  a.beta = (const __nv_bfloat16*)p.beta;
  a.g_min = p.g_min;
  a.init_state = p.init_state;
  a.out = p.out;
  a.out_bf16 = p.out_dtype == KDA_DTYPE_BF16;
  a.final_state = p.final_state;
  a.cu_seqlens = p.cu_seqlens;
  a.N = p.N;
  a.H = p.H;
  a.T = p.T;
  a.status = status_word_device_ptr();
  if (!a.status) return KDA_ERR_CUDA;
  kda_fwd_tc_kernel<<<(unsigned)(p.N * p.H), kThreads, SMEM_BYTES, stream>>>(mq, mk, mth, mv, a);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // namespace kda

#ifdef KDA_TRACE
extern "C" KDA_API int kda_debug_trace_read(void* dst, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(dst, kda::g_kda_trace, bytes);
}
#endif
