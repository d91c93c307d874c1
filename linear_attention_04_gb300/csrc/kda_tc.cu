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
//   A   = strict_lower(Diag(beta) Kt Kh^T)      P = lower_incl_diag(Qt Kh^T)
//   Tb  = (I + A)^{-1} Diag(beta)               W = Tb Kt
//   U   = Tb V - W S                            O = Qt S + P U
//   S  <- Diag(e^{G_C}) S + KhC^T U
//
// Warp roles (320 threads):
//   warp 0        TMA producer: q, k, theta, v tiles of each chunk into a
//                 2-stage ring (one lane); owns the TMEM allocation.
//   warp 1        tcgen05.mma issuer (one lane).
//   warps 2..5    "intra": gate g = g_min*sigmoid(theta) and cumulative sum in
//                 fp32, the decayed bf16 operands, V^T into TMEM; then per
//                 chunk the triangular inverse (fp32 forward substitution),
//                 Tb, P, and W = Tb Kt (warp-level mma.sync, 16x128x16).
//                 The A/P tiles of four chunks come from ONE tcgen05 MMA
//                 (M = 128 rows = [Kt_c; Qt_c] for c = 0..3, N = 64 = Kh of the
//                 four chunks); each chunk keeps its own 16 x 16 diagonal block.
//   warps 6..9    "state": U readout, the per-chunk state pass (bf16 copy for
//                 the next chunk's products, fp32 state scaled by e^{G_C}),
//                 output and final-state stores.
//
// Tensor-core products per chunk (M = 128 = dv lanes, K-major operands):
//   [U' | 0]  = V^T [Tb | 0]^T           (A = V^T in TMEM, N = 32, K = 16)
//   [U  | O] += S^T [-W | Qt]^T          (A = bf16 S^T in TMEM, N = 32, K = 128)
//   S^T      += U^T KhC                  (A = bf16 U^T in TMEM, N = 128, K = 16)
//   O        += U^T P^T                  (N = 16, K = 16)
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

constexpr int C = kChunk;                 // 16
constexpr int D = 128;                    // dk = dv
constexpr int NS = 2;                     // TMA ring stages (one chunk each)
constexpr int NSLOT = 8;                  // per-chunk operand slots (two groups)
constexpr int kThreads = 320;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait

// tensor memory columns (512 allocated)
constexpr uint32_t TM_S = 0;      // fp32 S^T, 128 columns
constexpr uint32_t TM_SBF = 128;  // bf16 S^T (A operand), 64 columns
constexpr uint32_t TM_AP = 192;   // A/P tiles of a group of 4 chunks, 64 columns
constexpr uint32_t TM_UO = 256;   // [U | O] accumulators, 2 buffers x 32 columns
constexpr uint32_t TM_UBF = 320;  // bf16 U^T (A operand): high part 8 columns, low part 8
constexpr uint32_t TM_VT = 336;   // bf16 V^T (A operand), NSLOT buffers x 8 columns
constexpr uint32_t TM_COLS = 512;
static_assert(TM_VT + 8 * NSLOT <= TM_COLS, "tensor memory budget");

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t TILE = C * D * 2;                       // 4096: one 16 x 128 bf16 tile
constexpr uint32_t SM_RING = 0;                            // NS x {q, k, theta, v}
constexpr uint32_t SM_GA = SM_RING + NS * 4 * TILE;        // 2 x [128 x 128] bf16, SW128
constexpr uint32_t GA_BYTES = 128 * D * 2;
constexpr uint32_t SM_GAL = SM_GA + 2 * GA_BYTES;          // [128 x 128] bf16 low parts
constexpr uint32_t SM_GB = SM_GAL + GA_BYTES;              // [64 x 128] bf16, SW128
constexpr uint32_t GB_BYTES = 64 * D * 2;
constexpr uint32_t SM_GBL = SM_GB + GB_BYTES;              // [64 x 128] bf16 low parts
constexpr uint32_t SM_KC = SM_GBL + GB_BYTES;              // NSLOT x [128 x 16] bf16
constexpr uint32_t SM_P = SM_KC + NSLOT * TILE;            // NSLOT x 2 x [16 x 16] bf16 (hi, lo)
constexpr uint32_t SM_TB = SM_P + NSLOT * 1024;            // NSLOT x [32 x 16] bf16
constexpr uint32_t SM_EGC = SM_TB + NSLOT * 1024;          // NSLOT x 128 fp32
constexpr uint32_t SM_BETA = SM_EGC + NSLOT * D * 4;       // NSLOT x 16 fp32
constexpr uint32_t SM_ABUF = SM_BETA + NSLOT * C * 4;      // 4 warps x [16 x 17] fp32
constexpr uint32_t SM_BARS = SM_ABUF + 4 * C * 17 * 4;     // mbarriers
constexpr int NBARS = 40;
constexpr uint32_t SM_MISC = SM_BARS + NBARS * 8;          // tmem base, abort flag
constexpr uint32_t SM_RANK = SM_MISC + 16;                 // chain-order scratch
constexpr uint32_t SM_TOTAL = SM_RANK + (kMaxRankedSeqsDev + 1) * 4;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;           // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(SM_GA % 1024 == 0 && SM_GAL % 1024 == 0 && SM_GB % 1024 == 0 && SM_GBL % 1024 == 0,
              "SW128 tiles must be 1024-aligned");

// barrier indices
constexpr int B_FULL = 0;          // [NS]  TMA -> intra
constexpr int B_EMPTY = 4;         // [NS]  intra -> TMA
constexpr int B_GATE = 8;          // [8]   intra (gate/operands of chunk n) -> state warps
constexpr int B_CHUNK = 16;        // [8]   intra (W, Tb, P of chunk n) -> MMA
constexpr int B_OPS = 24;          // [2]   intra (operands of a group) -> MMA (A/P product)
constexpr int B_GFREE = 26;        // [2]   MMA (group done) -> intra
constexpr int B_APDONE = 30;       //       MMA (A/P product done) -> intra
constexpr int B_UREADY = 31;       //       MMA (U, O products done) -> state warps
constexpr int B_UBF = 32;          //       state warps (bf16 U^T written) -> MMA
constexpr int B_SODONE = 33;       //       MMA (state and output products done) -> state warps
constexpr int B_STATE = 34;        //       state warps (state pass done) -> MMA
constexpr int B_DRAIN = 35;        //       MMA final drain

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
#ifdef KDA_TRACE
__device__ unsigned long long g_kda_trace[kTraceChunks * 16];
#define KTRACE(n, k)                                                   \
  do {                                                                 \
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
    for (int i = 0; i < NBARS; ++i) {
      uint32_t cnt = 1;
      if (i == B_UBF || i == B_STATE) cnt = 4;
      mbar_init(&bars[i], cnt);
    }
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
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_th);
      prefetch_tmap(&tm_v);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int n = 0; n < nchunks; ++n) {
        const int s = n % NS;
        if (n >= NS && !mbar_wait(&bars[B_EMPTY + s], ((n / NS) - 1) & 1, abort, kWaitNs)) {
          fail(abort, args.status);
          break;
        }
        mbar_arrive_expect_tx(&bars[B_FULL + s], 4 * TILE);
        KTRACE(n, 0);
        unsigned char* st = sm + SM_RING + s * 4 * TILE;
        const int row = (int)(ch.t0 + (int64_t)n * C);
        tma_load_3d(st + 0 * TILE, &tm_q, 0, h, row, &bars[B_FULL + s]);
        tma_load_3d(st + 1 * TILE, &tm_k, 0, h, row, &bars[B_FULL + s]);
        tma_load_3d(st + 2 * TILE, &tm_th, 0, h, row, &bars[B_FULL + s]);
        tma_load_3d(st + 3 * TILE, &tm_v, 0, h, row, &bars[B_FULL + s]);
        issued = n + 1;
      }
      // drain: every issued load has landed before the CTA may exit
      for (int n = issued - NS < 0 ? 0 : issued - NS; n < issued; ++n)
        mbar_wait_drain(&bars[B_FULL + n % NS], (n / NS) & 1, kWaitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nchunks > 0) {
      const uint32_t sbase = smem_u32(sm);
      int ap_next = 0;
      // A/P tiles of group g: [Kt;Qt] Kh^T with the P rows to ~16-bit precision:
      // hi*hi + hi*lo + lo*hi, every product accumulated in fp32
      auto issue_ap = [&](int g) {
        const uint32_t ga = sbase + SM_GA + (g & 1) * GA_BYTES, gal = sbase + SM_GAL;
        const uint32_t gb = sbase + SM_GB, gbl = sbase + SM_GBL;
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
          const uint32_t aa = pass == 2 ? gal : ga, bb = pass == 1 ? gbl : gb;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            uint64_t a = sdesc_sw128(aa + (kk >> 2) * (128 * 128) + (kk & 3) * 32);
            uint64_t b = sdesc_sw128(bb + (kk >> 2) * (64 * 128) + (kk & 3) * 32);
            mma_ss(tmem + TM_AP, a, b, idesc_bf16_f32(128, 64), (pass > 0) || (kk > 0));
          }
        }
        mma_commit(&bars[B_APDONE]);
      };
      auto try_issue_ap = [&]() {
        if (ap_next < ngroups && mbar_try_wait(&bars[B_OPS + (ap_next & 1)], (ap_next >> 1) & 1)) {
          tc_fence_after();
          issue_ap(ap_next);
          KTRACE(4 * ap_next, 15);
          ++ap_next;
        }
      };
      // wait that keeps issuing the next group's A/P product while it waits
      auto wait_poll = [&](uint64_t* bar, uint32_t parity) -> bool {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 0;; ++it) {
          if (mbar_try_wait(bar, parity)) return true;
          try_issue_ap();
          if ((it & 31u) == 31u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitNs) return false;
          }
        }
      };
      bool ok = true;
      for (int n = 0; n < nchunks && ok; ++n) {
        const int g = n >> 2, cc = n & 3, slot = n % NSLOT, buf = n & 1;
        while (ap_next <= g) {
          if (!mbar_wait(&bars[B_OPS + (ap_next & 1)], (ap_next >> 1) & 1, abort, kWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_ap(ap_next);
          KTRACE(4 * ap_next, 15);
          ++ap_next;
        }
        if (!ok) break;
        if (!wait_poll(&bars[B_CHUNK + slot], (n / NSLOT) & 1)) { ok = false; break; }
        KTRACE(n, 5);
        tc_fence_after();
        const uint32_t uo = tmem + TM_UO + 32 * buf;
        // [U' | 0] = V^T [Tb | 0]^T
        mma_ts(uo, tmem + TM_VT + 8 * slot, sdesc_noswz(sbase + SM_TB + slot * 1024, 512, 128),
               idesc_bf16_f32(128, 32), 0);
        if (!wait_poll(&bars[B_STATE], n & 1)) { ok = false; break; }
        KTRACE(n, 6);
        tc_fence_after();
        // [U | O] += S^T [-W | Qt]^T
        const uint32_t ga = sbase + SM_GA + (g & 1) * GA_BYTES + cc * 32 * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint64_t b = sdesc_sw128(ga + (kk >> 2) * (128 * 128) + (kk & 3) * 32);
          mma_ts(uo, tmem + TM_SBF + 8 * kk, b, idesc_bf16_f32(128, 32), 1);
        }
        mma_commit(&bars[B_UREADY]);
        KTRACE(n, 7);
        if (!wait_poll(&bars[B_UBF], n & 1)) { ok = false; break; }
        KTRACE(n, 8);
        tc_fence_after();
        // S^T += (U_hi + U_lo)^T KhC ;  O += U^T P^T as hi*hi + hi*lo + lo*hi
        {
          const uint64_t kc = sdesc_noswz(sbase + SM_KC + slot * TILE, 2048, 128);
          const uint64_t ph = sdesc_noswz(sbase + SM_P + slot * 1024, 256, 128);
          const uint64_t pl = sdesc_noswz(sbase + SM_P + slot * 1024 + 512, 256, 128);
          mma_ts(tmem + TM_S, tmem + TM_UBF, kc, idesc_bf16_f32(128, 128), 1);
          mma_ts(tmem + TM_S, tmem + TM_UBF + 8, kc, idesc_bf16_f32(128, 128), 1);
          mma_ts(uo + 16, tmem + TM_UBF, ph, idesc_bf16_f32(128, 16), 1);
          mma_ts(uo + 16, tmem + TM_UBF, pl, idesc_bf16_f32(128, 16), 1);
          mma_ts(uo + 16, tmem + TM_UBF + 8, ph, idesc_bf16_f32(128, 16), 1);
        }
        mma_commit(&bars[B_SODONE]);
        KTRACE(n, 9);
        if (cc == 3 || n == nchunks - 1) mma_commit(&bars[B_GFREE + (g & 1)]);
      }
      if (!ok) fail(abort, args.status);
      // drain every MMA this thread issued
      mma_commit(&bars[B_DRAIN]);
      mbar_wait_drain(&bars[B_DRAIN], 0, kWaitNs);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ intra warps
    const int it = tid - 64;          // 0..127: key/value channel of this thread in phase A
    const int q4 = warp & 3;          // TMEM lane quarter of this warp
    const int dvq = q4 * 32 + lane;   // value channel this thread moves into V^T
    bool bad = false;
    for (int g = 0; g < ngroups; ++g) {
      const int gb = g & 1;
      unsigned char* GA = sm + SM_GA + gb * GA_BYTES;
      if (g >= 2 && !bad && !mbar_wait(&bars[B_GFREE + gb], ((g >> 1) - 1) & 1, abort, kWaitNs))
        bad = true;
      // ---- phase A: gate, cumulative sum, decayed operands of the group's chunks
      bool stop = false;
      for (int cc = 0; cc < 4; ++cc) {
        const int n = 4 * g + cc;
        if (n >= nchunks) break;
        const int s = n % NS, slot = n % NSLOT;
        if (!bad && !mbar_wait(&bars[B_FULL + s], (n / NS) & 1, abort, kWaitNs)) bad = true;
        if (it == 0) KTRACE(n, 1);
        const int nvalid = min(C, L - n * C);
        const unsigned char* st = sm + SM_RING + s * 4 * TILE;
        const __nv_bfloat16* sq = (const __nv_bfloat16*)(st + 0 * TILE);
        const __nv_bfloat16* sk = (const __nv_bfloat16*)(st + 1 * TILE);
        const __nv_bfloat16* sth = (const __nv_bfloat16*)(st + 2 * TILE);
        const __nv_bfloat16* sv = (const __nv_bfloat16*)(st + 3 * TILE);
        float G = 0.0f, Gr[C], kr[C];
#pragma unroll
        for (int r = 0; r < C; ++r) {
          const bool valid = r < nvalid;
          const float th = __bfloat162float(sth[r * D + it]);
          const float kv = valid ? __bfloat162float(sk[r * D + it]) : 0.0f;
          const float qv = valid ? __bfloat162float(sq[r * D + it]) : 0.0f;
          const float gg = valid ? args.g_min * (1.0f / (1.0f + __expf(-th))) : 0.0f;
          G += gg;
          Gr[r] = G;
          kr[r] = kv;
          const float eg = __expf(G), emg = __expf(-G);
          const float xk = kv * eg, xq = qv * eg, xh = kv * emg;
          const __nv_bfloat16 hk = __float2bfloat16_rn(xk), hq = __float2bfloat16_rn(xq),
                              hh = __float2bfloat16_rn(xh);
          const uint32_t oa = sw128(32 * cc + r, it, 128), oq = sw128(32 * cc + 16 + r, it, 128);
          const uint32_t ob = sw128(16 * cc + r, it, 64);
          *(__nv_bfloat16*)(GA + oa) = hk;
          *(__nv_bfloat16*)(GA + oq) = hq;
          *(__nv_bfloat16*)(sm + SM_GAL + oa) = __float2bfloat16_rn(xk - __bfloat162float(hk));
          *(__nv_bfloat16*)(sm + SM_GAL + oq) = __float2bfloat16_rn(xq - __bfloat162float(hq));
          *(__nv_bfloat16*)(sm + SM_GB + ob) = hh;
          *(__nv_bfloat16*)(sm + SM_GBL + ob) = __float2bfloat16_rn(xh - __bfloat162float(hh));
        }
        {
          // KhC^T tile: row = key channel, 16 tokens along K (no swizzle)
          uint32_t w[8];
#pragma unroll
          for (int p = 0; p < 8; ++p)
            w[p] = pack_bf16x2(kr[2 * p] * __expf(G - Gr[2 * p]),
                               kr[2 * p + 1] * __expf(G - Gr[2 * p + 1]));
          unsigned char* kc = sm + SM_KC + slot * TILE + (it & 7) * 16 + (it >> 3) * 128;
          *(uint4*)(kc) = make_uint4(w[0], w[1], w[2], w[3]);
          *(uint4*)(kc + 2048) = make_uint4(w[4], w[5], w[6], w[7]);
          ((float*)(sm + SM_EGC + slot * D * 4))[it] = __expf(G);
        }
        if (it < C) {
          const float b = it < nvalid ? __bfloat162float(args.beta[(ch.t0 + (int64_t)n * C + it) * H + h])
                                      : 0.0f;
          ((float*)(sm + SM_BETA + slot * C * 4))[it] = b;
        }
        {
          // V^T into tensor memory: lane = value channel, 16 tokens packed in 8 columns
          __syncwarp();
          uint32_t w[8];
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            float v0 = (2 * p < nvalid) ? __bfloat162float(sv[(2 * p) * D + dvq]) : 0.0f;
            float v1 = (2 * p + 1 < nvalid) ? __bfloat162float(sv[(2 * p + 1) * D + dvq]) : 0.0f;
            w[p] = pack_bf16x2(v0, v1);
          }
          tmem_st_x8(tmem + ((uint32_t)(q4 * 32) << 16) + TM_VT + 8 * slot, w);
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (bar_sync_or(1, 128, bad || *abort)) { stop = true; break; }
        if (it == 0) {
          mbar_arrive(&bars[B_EMPTY + s]);
          mbar_arrive(&bars[B_GATE + slot]);
          KTRACE(n, 2);
        }
      }
      if (stop) break;
      if (it == 0) mbar_arrive(&bars[B_OPS + gb]);

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
        const float* bet = (const float*)(sm + SM_BETA + slot * C * 4);
        unsigned char* Pt = sm + SM_P + slot * 1024;
        unsigned char* Tb = sm + SM_TB + slot * 1024;
        if (lane < 16) {
          const int i = lane;
          const float bi = bet[i];
#pragma unroll
          for (int j = 0; j < C; ++j) Ab[i * 17 + j] = (j < i) ? bi * __uint_as_float(raw[j]) : 0.0f;
        } else {
          const int i = lane - 16;
          // P row i, split into a bf16 high part and a bf16 low part
          uint32_t wh[8], wl[8];
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const float x0 = (2 * p <= i) ? __uint_as_float(raw[2 * p]) : 0.0f;
            const float x1 = (2 * p + 1 <= i) ? __uint_as_float(raw[2 * p + 1]) : 0.0f;
            wh[p] = pack_bf16x2(x0, x1);
            const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&wh[p]);
            wl[p] = pack_bf16x2(x0 - __low2float(hb), x1 - __high2float(hb));
          }
          unsigned char* pr = Pt + (i & 7) * 16 + (i >> 3) * 128;
          *(uint4*)(pr) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
          *(uint4*)(pr + 256) = make_uint4(wh[4], wh[5], wh[6], wh[7]);
          *(uint4*)(pr + 512) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
          *(uint4*)(pr + 768) = make_uint4(wl[4], wl[5], wl[6], wl[7]);
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
            float acc = 0.0f;
#pragma unroll
            for (int m = 0; m < i; ++m) acc += Ab[i * 17 + m] * t[m];
            if (i > j) t[i] = -acc;
          }
          const float bj = bet[j];
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
              for (int hf = 0; hf < 2; ++hf) {
                const int R = 32 * q4 + (lane >> 2) + 8 * hf;
                *(uint32_t*)(GA + sw128(R, col, 128)) =
                    pack_bf16x2(-acc[t4][2 * hf], -acc[t4][2 * hf + 1]);
              }
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_CHUNK + slot]);
        if (lane == 0) KTRACE(n, 4);
      }
    }
    if (bad) fail(abort, args.status);
  } else {
    // ------------------------------------------------------------ state warps
    const int q4 = warp & 3;
    const int dv = q4 * 32 + lane;
    const uint32_t lb = (uint32_t)(q4 * 32) << 16;
    const int64_t soff = ((int64_t)ch.seq * H + h) * D * D;
    bool ok = true;
    if (nchunks > 0) {
      // initial state: bf16 copy and fp32 scaled by e^{G_C} of chunk 0
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_GATE + 0], 0, abort, kWaitNs));
      const float* eg0 = (const float*)(sm + SM_EGC);
#pragma unroll 1
      for (int blk = 0; blk < 4 && ok; ++blk) {
        uint32_t f[32], b[16];
#pragma unroll
        for (int p = 0; p < 16; ++p) {
          const int i0 = 32 * blk + 2 * p;
          const float s0 = args.init_state ? args.init_state[soff + (int64_t)i0 * D + dv] : 0.0f;
          const float s1 = args.init_state ? args.init_state[soff + (int64_t)(i0 + 1) * D + dv] : 0.0f;
          b[p] = pack_bf16x2(s0, s1);
          f[2 * p] = __float_as_uint(s0 * eg0[i0]);
          f[2 * p + 1] = __float_as_uint(s1 * eg0[i0 + 1]);
        }
        tmem_st_x16(tmem + lb + TM_SBF + 16 * blk, b);
        tmem_st_x32(tmem + lb + TM_S + 32 * blk, f);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_STATE]);
      for (int n = 0; n < nchunks && ok; ++n) {
        const int buf = n & 1;
        const uint32_t uo = tmem + lb + TM_UO + 32 * buf;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_UREADY], n & 1, abort, kWaitNs))) {
          ok = false;
          break;
        }
        if (lane == 0 && q4 == 2) KTRACE(n, 10);
        tc_fence_after();
        {
          // U^T as bf16 high part (columns 0..7) and low part (columns 8..15)
          uint32_t u[16], w[16];
          tmem_ld_x16(uo, u);
          tmem_wait_ld();
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const float x0 = __uint_as_float(u[2 * p]), x1 = __uint_as_float(u[2 * p + 1]);
            w[p] = pack_bf16x2(x0, x1);
            const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&w[p]);
            w[8 + p] = pack_bf16x2(x0 - __low2float(hb), x1 - __high2float(hb));
          }
          tmem_st_x16(tmem + lb + TM_UBF, w);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_UBF]);
        if (lane == 0 && q4 == 2) KTRACE(n, 11);
        __syncwarp();
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_SODONE], n & 1, abort, kWaitNs))) {
          ok = false;
          break;
        }
        if (lane == 0 && q4 == 2) KTRACE(n, 12);
        tc_fence_after();
        if (n + 1 < nchunks) {
          const int nslot = (n + 1) % NSLOT;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&bars[B_GATE + nslot], ((n + 1) / NSLOT) & 1, abort, kWaitNs))) {
            ok = false;
            break;
          }
          const float* eg = (const float*)(sm + SM_EGC + nslot * D * 4);
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
            uint32_t f[32], b[16];
            tmem_ld_x32(tmem + lb + TM_S + 32 * blk, f);
            tmem_wait_ld();
#pragma unroll
            for (int p = 0; p < 16; ++p)
              b[p] = pack_bf16x2(__uint_as_float(f[2 * p]), __uint_as_float(f[2 * p + 1]));
            tmem_st_x16(tmem + lb + TM_SBF + 16 * blk, b);
            const float4* eg4 = (const float4*)(eg + 32 * blk);
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 e = eg4[i4];
              f[4 * i4 + 0] = __float_as_uint(__uint_as_float(f[4 * i4 + 0]) * e.x);
              f[4 * i4 + 1] = __float_as_uint(__uint_as_float(f[4 * i4 + 1]) * e.y);
              f[4 * i4 + 2] = __float_as_uint(__uint_as_float(f[4 * i4 + 2]) * e.z);
              f[4 * i4 + 3] = __float_as_uint(__uint_as_float(f[4 * i4 + 3]) * e.w);
            }
            tmem_st_x32(tmem + lb + TM_S + 32 * blk, f);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[B_STATE]);
          if (lane == 0 && q4 == 2) KTRACE(n, 13);
          __syncwarp();
        }
        // output rows of this chunk
        {
          uint32_t o[16];
          tmem_ld_x16(uo + 16, o);
          tmem_wait_ld();
          const int nvalid = min(C, L - n * C);
          if (lane == 0 && q4 == 2) KTRACE(n, 14);
          const int64_t row0 = ch.t0 + (int64_t)n * C;
          if (args.out_bf16) {
            __nv_bfloat16* out = (__nv_bfloat16*)args.out;
#pragma unroll
            for (int i = 0; i < C; ++i)
              if (i < nvalid) out[((row0 + i) * H + h) * D + dv] = __float2bfloat16_rn(__uint_as_float(o[i]));
          } else {
            float* out = (float*)args.out;
#pragma unroll
            for (int i = 0; i < C; ++i)
              if (i < nvalid) out[((row0 + i) * H + h) * D + dv] = __uint_as_float(o[i]);
          }
        }
      }
      if (ok && args.final_state) {
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t f[32];
          tmem_ld_x32(tmem + lb + TM_S + 32 * blk, f);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            args.final_state[soff + (int64_t)(32 * blk + i) * D + dv] = __uint_as_float(f[i]);
        }
      }
      if (!ok) fail(abort, args.status);
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

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// [tokens, H, 128] bf16 -> boxes of 16 tokens x 128 channels of one head
bool encode_rows(CUtensorMap* m, const void* base, int H, int64_t tokens) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  if (!encode_rows(&mq, p.q, p.H, tokens) || !encode_rows(&mk, p.k, p.H, tokens) ||
      !encode_rows(&mth, p.theta, p.H, tokens) || !encode_rows(&mv, p.v, p.H, tokens))
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
