// kda_bwd.cu -- backward pass of KDA in chunked (WY) form, fp32 on CUDA cores.
//
// Forward, per (sequence, head) and 16-token chunk ("Kimi K3 Deep Dive",
// section "Core Innovation 1"; gate of "Architecture Deep Dive", sec. 3.2),
// with the inclusive in-chunk cumulative log-decay G, Kt = K e^{G},
// Qt = Q e^{G}, Kh = K e^{-G}, KhC = K e^{G_C - G}, ec = e^{G_C}:
//   Ab = strict_lower(Kt Kh^T),  M = (I + Diag(b) Ab)^{-1},  Tb = M Diag(b)
//   Pi = lower_incl_diag(Qt Kh^T)
//   R = V - Kt S,  U = Tb R,  O = Qt S + Pi U,  S' = Diag(ec) S + KhC^T U
// Reverse-mode differentiation of these steps, with dO the output gradient
// and dS' the gradient w.r.t. the chunk's end state:
//   dU = Pi^T dO + KhC dS'            dR = Tb^T dU        dV = dR
//   dS = Diag(ec) dS' + Qt^T dO - Kt^T dR                (carried backwards)
//   dTb = lower_incl_diag(dU R^T)     dPi = lower_incl_diag(dO U^T)
//   dQt = dO S^T + dPi Kh             dKhC = U dS'^T      dec = rowsum(dS' * S)
//   (the diagonal of dPi goes straight to dq_t += dPi_tt k_t, dk_t += dPi_tt q_t:
//   Pi_tt = q_t . k_t has no decay factor, and its shares of dG cancel exactly)
//   dA = -strict_lower(M^T (dTb Diag(b)) M^T)
//   db_j = sum_i M_ij dTb_ij + sum_l dA_jl Ab_jl
//   dKt = -dR S^T + Diag(b) dA Kh     dKh = dPi^T Qt + (Diag(b) dA)^T Kt
//   dK = dKt e^{G} + dKh e^{-G} + dKhC e^{G_C - G},   dQ = dQt e^{G}
//   dG = dKt Kt + dQt Qt - dKh Kh - dKhC KhC (elementwise),
//   dG_C = colsum(dKhC KhC) + dec ec,   dg_t = sum_{s >= t} dG_s + dG_C,
//   (summed as sum_{s >= t} (dG_s + dKhC_s KhC_s) + sum_{s < t} dKhC_s KhC_s + dec ec),
//   dtheta = dg g_min sigmoid(theta) sigmoid(-theta)   (dg for a given log-decay).
//
// One persistent launch (kda_bwd_kernel) over a caller workspace, its CTAs
// taking items from a work queue:
//   1. two recurrences per chain (independent of each other): the forward
//      recurrence, writing the state at the start of every chunk and R, U of
//      every chunk; and the reverse recurrence of dS, writing dS' and dU of
//      every chunk, and dV;
//   2. one item per chunk: every other gradient from S, dS', dU, R, U and the
//      chunk's inputs, once both recurrences of its chain are done.
// The recurrences carry their 128 x 128 state in registers with a copy in
// shared memory for the products that contract over it, and stage the next
// chunk's inputs in shared memory with cp.async while the current chunk
// computes.  Both recurrences are warp-specialised: four warps form the next
// chunk's operands while the other four run the current chunk's state
// products.  Every product is an fp32 FMA over shared-memory operands.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_device.cuh"
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = kChunk;             // 16
constexpr int D = 128;                // dk = dv
constexpr int LD = D + 4;             // row stride (floats) of 16 x 128 tiles and of the state
constexpr int LS = 20;                // row stride of 16 x 16 matrices
constexpr int kThreads = 256;
constexpr int TILE_F = C * LD;        // floats of a token tile
constexpr int STATE_F = D * LD;       // floats of the padded state
constexpr int SM16_F = C * LS;        // floats of a 16 x 16 matrix
constexpr size_t kStateF = (size_t)D * D;  // floats of one state in the workspace
static_assert(5 * SM16_F <= 4 * TILE_F, "inverse scratch fits the partial-sum tiles");

struct BwdDev {
  const void* q;
  const void* k;
  const void* v;
  const void* theta;
  const void* beta;
  float g_min;
  int log_decay;
  const float* init_state;
  const float* d_out;
  const float* d_final;
  float* dq;
  float* dk;
  float* dv;
  float* dtheta;
  float* dbeta;
  float* d_init;
  float* ws_S;   // [chain][chunk][128][128] state at each chunk start
  float* ws_dS;  // [chain][chunk][128][128] gradient w.r.t. each chunk's end state
  float* ws_dU;  // [chain][chunk][16][128]
  float* ws_RU;  // [chain][chunk][2][16][128]: R = V - Kt S and U = Tb R of each chunk
  unsigned long long* q_next;  // work-queue position (zeroed before the launch)
  int* q_done;                 // [chain] recurrences of the chain finished (0, 1 or 2)
  int* status;                 // device status word
  uint64_t wait_ns;            // limit of a gradient item's wait for its chain
  int H, T, nch;
};

// d0 += a * b0 and d1 += a * b1 as one packed instruction: two IEEE fp32
// fused multiply-adds, bit-identical to two fmaf calls, in one issue slot.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a, float b0, float b1) {
  asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %2};\n mov.b64 pb, {%3, %4};\n"
      " mov.b64 pd, {%0, %1};\n fma.rn.f32x2 pd, pa, pb, pd;\n mov.b64 {%0, %1}, pd;\n}"
      : "+f"(d0), "+f"(d1)
      : "f"(a), "f"(b0), "f"(b1));
}
// d0 += a0 * b0 and d1 += a1 * b1 as one packed instruction.
__device__ __forceinline__ void ffma2v(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n"
      " mov.b64 pd, {%0, %1};\n fma.rn.f32x2 pd, pa, pb, pd;\n mov.b64 {%0, %1}, pd;\n}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// acc[m][t] += sum_{k0 <= k < k1} A(m0 + m, k) B(k, col(t)), operands in shared
// memory.  A: A[m * lda + k] (AMK) or A[k * lda + m].  B: BKN -> B[k * ldb +
// col] with col(t) = n0 + (t / 4) * nstride + t % 4 (groups of four adjacent
// columns); else B[col * ldb + k] with col(t) = n0 + t * nstride.  k runs in
// steps of four (float4 loads along the contiguous dimension).
template <int TM, int TN, bool AMK, bool BKN>
__device__ __forceinline__ void gemm_acc(float (&acc)[TM][TN], const float* A, int lda, int m0,
                                         const float* B, int ldb, int n0, int nstride, int k0,
                                         int k1) {
  static_assert(AMK || TM % 4 == 0, "k-major A needs TM % 4 == 0");
  static_assert(!BKN || TN % 4 == 0, "k-major B needs TN % 4 == 0");
  static_assert(TN % 2 == 0, "column pairs");
  for (int k = k0; k < k1; k += 4) {
    float a[TM][4], b[4][TN];
    if constexpr (AMK) {
#pragma unroll
      for (int m = 0; m < TM; ++m) {
        const float4 x = *(const float4*)(A + (m0 + m) * lda + k);
        a[m][0] = x.x;
        a[m][1] = x.y;
        a[m][2] = x.z;
        a[m][3] = x.w;
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int m4 = 0; m4 < TM; m4 += 4) {
          const float4 x = *(const float4*)(A + (k + kk) * lda + m0 + m4);
          a[m4][kk] = x.x;
          a[m4 + 1][kk] = x.y;
          a[m4 + 2][kk] = x.z;
          a[m4 + 3][kk] = x.w;
        }
    }
    if constexpr (BKN) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int g4 = 0; g4 < TN / 4; ++g4) {
          const float4 x = *(const float4*)(B + (k + kk) * ldb + n0 + g4 * nstride);
          b[kk][4 * g4] = x.x;
          b[kk][4 * g4 + 1] = x.y;
          b[kk][4 * g4 + 2] = x.z;
          b[kk][4 * g4 + 3] = x.w;
        }
    } else {
#pragma unroll
      for (int t = 0; t < TN; ++t) {
        const float4 x = *(const float4*)(B + (n0 + t * nstride) * ldb + k);
        b[0][t] = x.x;
        b[1][t] = x.y;
        b[2][t] = x.z;
        b[3][t] = x.w;
      }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int m = 0; m < TM; ++m)
#pragma unroll
        for (int t = 0; t < TN; t += 2) {
          if constexpr (BKN) {
            // column pairs straight from the float4 loads of B: one packed
            // instruction per pair
            ffma2(acc[m][t], acc[m][t + 1], a[m][kk], b[kk][t], b[kk][t + 1]);
          } else {
            // columns from separate loads would need packing: scalar FMAs
            acc[m][t] = fmaf(a[m][kk], b[kk][t], acc[m][t]);
            acc[m][t + 1] = fmaf(a[m][kk], b[kk][t + 1], acc[m][t + 1]);
          }
        }
  }
}

// Partial sums of a 16 x 128 product with K = 128 split four ways:
// part[ks][m][n] = sum_{32 ks <= k < 32 ks + 32} A[m][k] B(k, n).  A is a
// token tile (row-major, k contiguous).  B is the padded 128 x 128 state,
// read as B[k][n] (BKN) or B[n][k].
template <bool BKN>
__device__ __forceinline__ void part16(const float* A, const float* B, float* part) {
  const int tid = threadIdx.x, ng = tid & 31, mg = (tid >> 5) & 1, ks = tid >> 6;
  float acc[8][4];
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[m][t] = 0.0f;
  if constexpr (BKN) {
    gemm_acc<8, 4, true, true>(acc, A, LD, 8 * mg, B, LD, 4 * ng, 0, 32 * ks, 32 * ks + 32);
#pragma unroll
    for (int m = 0; m < 8; ++m)
      *(float4*)(part + (ks * C + 8 * mg + m) * LD + 4 * ng) =
          make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
  } else {
    gemm_acc<8, 4, true, false>(acc, A, LD, 8 * mg, B, LD, ng, 32, 32 * ks, 32 * ks + 32);
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
      for (int t = 0; t < 4; ++t) part[(ks * C + 8 * mg + m) * LD + ng + 32 * t] = acc[m][t];
  }
}

// Partial sums of a 32 x 128 product X B^T (K = 128 split two ways); X is 32
// token rows (row-major), B the padded state read as B[n][k].
__device__ __forceinline__ void part32_nk(const float* X, const float* B, float* part) {
  const int tid = threadIdx.x, ng = tid & 31, mg = (tid >> 5) & 3, ks = tid >> 7;
  float acc[8][4];
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[m][t] = 0.0f;
  gemm_acc<8, 4, true, false>(acc, X, LD, 8 * mg, B, LD, ng, 32, 64 * ks, 64 * ks + 64);
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int t = 0; t < 4; ++t) part[(ks * 2 * C + 8 * mg + m) * LD + ng + 32 * t] = acc[m][t];
}

// out[m][n] = base[m][n] + sign * sum_s part[s][m][n] over an M x 128 tile
// (base may be null; out may alias base or part[0]).
template <int M, int KS>
__device__ __forceinline__ void reduce_parts(const float* part, float* out, const float* base,
                                             float sign) {
  for (int e = threadIdx.x; e < M * (D / 4); e += kThreads) {
    const int m = e >> 5, n = (e & 31) * 4;
    float4 s = *(const float4*)(part + m * LD + n);
#pragma unroll
    for (int ks = 1; ks < KS; ++ks) {
      const float4 x = *(const float4*)(part + (ks * M + m) * LD + n);
      s.x += x.x;
      s.y += x.y;
      s.z += x.z;
      s.w += x.w;
    }
    float4 r = base ? *(const float4*)(base + m * LD + n) : make_float4(0.f, 0.f, 0.f, 0.f);
    r.x = fmaf(sign, s.x, r.x);
    r.y = fmaf(sign, s.y, r.y);
    r.z = fmaf(sign, s.z, r.z);
    r.w = fmaf(sign, s.w, r.w);
    *(float4*)(out + m * LD + n) = r;
  }
}

// out = sign * A B (or out += sign * A B when ACC) for a 16 x 16 matrix A
// (row stride LS) and a 16 x 128 token tile B.
template <bool ACC>
__device__ __forceinline__ void small16(const float* A, const float* B, float* out, float sign) {
  const int tid = threadIdx.x, ng = tid & 31, mg = tid >> 5;
  float acc[2][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[m][t] = 0.0f;
  gemm_acc<2, 4, true, true>(acc, A, LS, 2 * mg, B, LD, 4 * ng, 0, 0, C);
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    float4* o = (float4*)(out + (2 * mg + m) * LD + 4 * ng);
    float4 r = ACC ? *o : make_float4(0.f, 0.f, 0.f, 0.f);
    r.x = fmaf(sign, acc[m][0], r.x);
    r.y = fmaf(sign, acc[m][1], r.y);
    r.z = fmaf(sign, acc[m][2], r.z);
    r.w = fmaf(sign, acc[m][3], r.w);
    *o = r;
  }
}

// sum_k X[m][k] Y[n][k] over the 128 channels of two token tiles, in four
// independent partial sums (k mod 4) added at the end.
__device__ __forceinline__ float dot128(const float* X, int m, const float* Y, int n) {
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const float* x = X + m * LD;
  const float* y = Y + n * LD;
#pragma unroll 8
  for (int k = 0; k < D; k += 4) {
    const float4 a = *(const float4*)(x + k), b = *(const float4*)(y + k);
    ffma2v(acc[0], acc[1], a.x, a.y, b.x, b.y);
    ffma2v(acc[2], acc[3], a.z, a.w, b.z, b.w);
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// The chunk's operands in two passes over all threads.  Element (t, c) of
// theta is th0[t * rs + c], and so on for k, q and v: rows of the global
// tensors (rs = H * D) or of a staged copy in shared memory (rs = D).
//   pass 1 (thread -> channel c = tid % 128, tokens 8 (tid / 128) .. + 7):
//     every load of the chunk, the gate g, its derivative factor dg and the
//     per-token factors e^{g} and 1 / e^{g}; V is written, and the raw k and q
//     wait in the KhC and Qt tiles;
//   pass 2 (threads 0..127, one channel each, sequential over the 16
//     tokens): the decay factors as running products, e^{G_t} =
//     prod_{s <= t} e^{g_s}, e^{-G_t} = prod_{s <= t} 1 / e^{g_s} and
//     e^{G_C - G_t} = prod_{s > t} e^{g_s}.  (The exponential of an fp32
//     cumulative sum would carry the sum's rounding, up to half an ulp of
//     |G| <= 80 per step, into every factor; the products stay within a few
//     ulp.)
// Thread 128 + t (t < 16) passes beta_t in bval.  Rows past the sequence end
// are neutral (q = k = v = 0, g = 0, beta = 0).  Null outputs are skipped.
// Kt is written times ksign; EGt receives e^{g}.  Contains a __syncthreads:
// every thread of the CTA calls it.
template <typename Tin>
__device__ __forceinline__ void load_chunk(const Tin* th0, const Tin* k0, const Tin* q0,
                                           const Tin* v0, int64_t rs, float bval, float g_min,
                                           int log_decay, int nvalid, float* Qt, float* Kt,
                                           float ksign, float* Kh, float* KhC, float* EGt,
                                           float* dgt, float* ec, float* bt, float* V) {
  constexpr int CH = C / 2;
  const int tid = threadIdx.x;
  if (tid < 2 * D) {
    const int c = tid & (D - 1), tb = (tid >> 7) * CH;
    float xr[CH], kr[CH], qr[CH], vr[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int t = tb + i;
      const bool ok = t < nvalid;
      xr[i] = ok ? to_f32(th0[t * rs + c]) : 0.0f;
      kr[i] = ok ? to_f32(k0[t * rs + c]) : 0.0f;
      qr[i] = (ok && Qt) ? to_f32(q0[t * rs + c]) : 0.0f;
      vr[i] = (ok && V) ? to_f32(v0[t * rs + c]) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int t = tb + i;
      float g = 0.0f, dg = 0.0f;
      if (t < nvalid) {
        if (log_decay) {
          g = xr[i];
          dg = 1.0f;
        } else {
          // sigmoid(x) and sigmoid(-x) from one exponential of -|x|: both
          // keep full relative precision (neither is formed as 1 - the other)
          const float x = xr[i];
          const float e = expf(-fabsf(x));
          const float big = 1.0f / (1.0f + e), small = e * big;
          const float sp = x >= 0.0f ? big : small, sn = x >= 0.0f ? small : big;
          g = g_min * sp;
          dg = g_min * sp * sn;
        }
      }
      const float eg = expf(g);
      Kt[t * LD + c] = eg;
      Kh[t * LD + c] = 1.0f / eg;
      KhC[t * LD + c] = kr[i];
      if (Qt) Qt[t * LD + c] = qr[i];
      if (V) V[t * LD + c] = vr[i];
      if (EGt) EGt[t * LD + c] = eg;
      if (dgt) dgt[t * LD + c] = dg;
    }
  }
  __syncthreads();
  if (tid < D) {
    const int c = tid;
    float kr[C], egr[C];
    float E = 1.0f, Ei = 1.0f;
#pragma unroll
    for (int t = 0; t < C; ++t) {
      kr[t] = KhC[t * LD + c];
      const float eg = Kt[t * LD + c];
      E *= eg;
      Ei *= Kh[t * LD + c];
      egr[t] = eg;
      Kt[t * LD + c] = ksign * kr[t] * E;
      Kh[t * LD + c] = kr[t] * Ei;
      if (Qt) Qt[t * LD + c] *= E;
    }
    ec[c] = E;
    float P = 1.0f;
#pragma unroll
    for (int t = C - 1; t >= 0; --t) {
      KhC[t * LD + c] = kr[t] * P;
      P *= egr[t];
    }
  } else if (tid < D + C) {
    bt[tid - D] = bval;
  }
}

// beta_t of the chunk for thread 128 + t (t < 16), zero elsewhere.
template <typename Tin>
__device__ __forceinline__ float load_beta(const BwdDev& a, int64_t row0, int h, int nvalid) {
  const int t = (int)threadIdx.x - D;
  return (t >= 0 && t < nvalid) ? to_f32(((const Tin*)a.beta)[(row0 + t) * a.H + h]) : 0.0f;
}

// Asynchronous 16-byte copy global -> shared (zero-filled when !valid; the
// source address is then not read).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Waits until at most one of this thread's committed copy groups is pending.
__device__ __forceinline__ void cp_async_wait_one_pending() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// M = (I + N)^{-1} with N = Diag(b) Ab strictly lower, Tb = M Diag(b), and the
// transpose of Tb when asked.  N is nilpotent (N^16 = 0), so
//   (I + N)^{-1} = (I - N)(I + N^2)(I + N^4)(I + N^8),
// four rounds of 16 x 16 products instead of sixteen sequential substitution
// steps: every thread (i, j) = (tid / 16, tid % 16) forms entry (i, j) of each
// product.  `scratch` holds five 16 x 16 matrices.  Contains __syncthreads:
// every thread of the CTA calls it; M, Tb and TbT are complete after the
// caller's next barrier.
__device__ __forceinline__ void wy_inverse(const float* Ab, const float* bt, float* M, float* Tb,
                                           float* TbT, float* scratch) {
  const int i = threadIdx.x >> 4, j = threadIdx.x & 15;
  const int ij = i * LS + j;
  float* B0 = scratch;
  float* B1 = B0 + SM16_F;
  float* B2 = B1 + SM16_F;
  float* B3 = B2 + SM16_F;
  float* B4 = B3 + SM16_F;
  // B0 = N, B1 = I - N
  const float n = j < i ? bt[i] * Ab[ij] : 0.0f;
  B0[ij] = n;
  B1[ij] = (i == j ? 1.0f : 0.0f) - n;
  __syncthreads();
  // B2 = N^2
  {
    float x = 0.0f;
#pragma unroll
    for (int l = 0; l < C; ++l) x = fmaf(B0[i * LS + l], B0[l * LS + j], x);
    B2[ij] = x;
  }
  __syncthreads();
  // B3 = (I - N)(I + N^2), B4 = N^4
  {
    float q = B1[ij], x = 0.0f;
#pragma unroll
    for (int l = 0; l < C; ++l) {
      q = fmaf(B1[i * LS + l], B2[l * LS + j], q);
      x = fmaf(B2[i * LS + l], B2[l * LS + j], x);
    }
    B3[ij] = q;
    B4[ij] = x;
  }
  __syncthreads();
  // B1 = B3 (I + N^4), B0 = N^8
  {
    float q = B3[ij], x = 0.0f;
#pragma unroll
    for (int l = 0; l < C; ++l) {
      q = fmaf(B3[i * LS + l], B4[l * LS + j], q);
      x = fmaf(B4[i * LS + l], B4[l * LS + j], x);
    }
    B1[ij] = q;
    B0[ij] = x;
  }
  __syncthreads();
  // M = B1 (I + N^8)
  float q = B1[ij];
#pragma unroll
  for (int l = 0; l < C; ++l) q = fmaf(B1[i * LS + l], B0[l * LS + j], q);
  const float bj = bt[j];
  M[ij] = q;
  Tb[ij] = q * bj;
  if (TbT) TbT[j * LS + i] = q * bj;
}

// Thread tile of the register-resident 128 x 128 state: element [i][4 g + c]
// is row 8 ig + i, column 64 g + 4 jg + c (ig = tid / 16, jg = tid % 16).
__device__ __forceinline__ void state_store(const float (&st)[8][8], float* dst, int ld) {
  const int ig = threadIdx.x >> 4, jg = threadIdx.x & 15;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int g = 0; g < 2; ++g)
      *(float4*)(dst + (size_t)(8 * ig + i) * ld + 64 * g + 4 * jg) =
          make_float4(st[i][4 * g], st[i][4 * g + 1], st[i][4 * g + 2], st[i][4 * g + 3]);
}

// The same tile from a dense 128 x 128 state in global memory (zero if null).
__device__ __forceinline__ void state_load(float (&st)[8][8], const float* src) {
  const int ig = threadIdx.x >> 4, jg = threadIdx.x & 15;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const float4 x = src ? *(const float4*)(src + (size_t)(8 * ig + i) * D + 64 * g + 4 * jg)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      st[i][4 * g] = x.x;
      st[i][4 * g + 1] = x.y;
      st[i][4 * g + 2] = x.z;
      st[i][4 * g + 3] = x.w;
    }
}

// ------------------------------------------------------- forward recurrence
// Warp-specialised: warps 0..3 (the state group) carry S and run the products
// that need it; warps 4..7 (the prep group) form the next chunk's operands --
// gate, decay factors, decayed tiles, Ab and the inverse -- meanwhile, into
// one of two buffers.  The groups hand buffers over through named barriers
// (arrive by one group, sync by the other, 256 threads each); each group also
// has its own 128-thread barrier.
constexpr int kGroup = kThreads / 2;
constexpr int BAR_SG = 1, BAR_PG = 2, BAR_READY = 3, BAR_FREE = 5;  // READY/FREE: + buffer
__device__ __forceinline__ void bar_group(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kGroup) : "memory");
}
__device__ __forceinline__ void bar_sync_all(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kThreads) : "memory");
}
__device__ __forceinline__ void bar_arrive_all(int id) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "n"(kThreads) : "memory");
}

// One chunk's operands on the 128 threads of the prep group, one channel per
// thread, sequential over the tokens: the same per-element arithmetic as
// load_chunk (the gradient kernel forms the same factors).
template <typename Tin>
__device__ __forceinline__ void prep_chunk(const Tin* th0, const Tin* k0, const Tin* v0,
                                           float bval, float g_min, int log_decay, int nvalid,
                                           float* Kt, float* Kh, float* KhC, float* ec, float* bt,
                                           float* V, int gt) {
  const int c = gt;
  float xr[C], kr[C], vr[C], egr[C];
#pragma unroll
  for (int t = 0; t < C; ++t) {
    const bool ok = t < nvalid;
    xr[t] = ok ? to_f32(th0[t * D + c]) : 0.0f;
    kr[t] = ok ? to_f32(k0[t * D + c]) : 0.0f;
    vr[t] = ok ? to_f32(v0[t * D + c]) : 0.0f;
  }
  float E = 1.0f, Ei = 1.0f;
#pragma unroll
  for (int t = 0; t < C; ++t) {
    float g = 0.0f;
    if (t < nvalid) {
      if (log_decay) {
        g = xr[t];
      } else {
        const float x = xr[t];
        const float e = expf(-fabsf(x));
        const float big = 1.0f / (1.0f + e), small = e * big;
        g = g_min * (x >= 0.0f ? big : small);
      }
    }
    const float eg = expf(g);
    E *= eg;
    Ei *= 1.0f / eg;
    egr[t] = eg;
    Kt[t * LD + c] = kr[t] * E;
    Kh[t * LD + c] = kr[t] * Ei;
    V[t * LD + c] = vr[t];
  }
  ec[c] = E;
  float P = 1.0f;
#pragma unroll
  for (int t = C - 1; t >= 0; --t) {
    KhC[t * LD + c] = kr[t] * P;
    P *= egr[t];
  }
  if (gt < C) bt[gt] = bval;
}

// (I + Diag(b) Ab)^{-1} as in wy_inverse, on the 128 threads of one group
// (two entries per thread: rows i and i + 8 of column j), with that group's
// barrier between the rounds.  M and Tb are complete after the group's next
// barrier.
__device__ __forceinline__ void wy_inverse_group(const float* Ab, const float* bt, float* M,
                                                 float* Tb, float* TbT, float* scratch, int gt,
                                                 int bar) {
  const int i0 = gt >> 4, j = gt & 15;
  float* B0 = scratch;
  float* B1 = B0 + SM16_F;
  float* B2 = B1 + SM16_F;
  float* B3 = B2 + SM16_F;
  float* B4 = B3 + SM16_F;
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int i = i0 + 8 * h2, ij = i * LS + j;
    const float n = j < i ? bt[i] * Ab[ij] : 0.0f;
    B0[ij] = n;
    B1[ij] = (i == j ? 1.0f : 0.0f) - n;
  }
  bar_group(bar);
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int i = i0 + 8 * h2;
    float x = 0.0f;
#pragma unroll
    for (int l = 0; l < C; ++l) x = fmaf(B0[i * LS + l], B0[l * LS + j], x);
    B2[i * LS + j] = x;
  }
  bar_group(bar);
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int i = i0 + 8 * h2, ij = i * LS + j;
    float q = B1[ij], x = 0.0f;
#pragma unroll
    for (int l = 0; l < C; ++l) {
      q = fmaf(B1[i * LS + l], B2[l * LS + j], q);
      x = fmaf(B2[i * LS + l], B2[l * LS + j], x);
    }
    B3[ij] = q;
    B4[ij] = x;
  }
  bar_group(bar);
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int i = i0 + 8 * h2, ij = i * LS + j;
    float q = B3[ij], x = 0.0f;
#pragma unroll
    for (int l = 0; l < C; ++l) {
      q = fmaf(B3[i * LS + l], B4[l * LS + j], q);
      x = fmaf(B4[i * LS + l], B4[l * LS + j], x);
    }
    B1[ij] = q;
    B0[ij] = x;
  }
  bar_group(bar);
  const float bj = bt[j];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int i = i0 + 8 * h2, ij = i * LS + j;
    float q = B1[ij];
#pragma unroll
    for (int l = 0; l < C; ++l) q = fmaf(B1[i * LS + l], B0[l * LS + j], q);
    M[ij] = q;
    Tb[ij] = q * bj;
    if (TbT) TbT[j * LS + i] = q * bj;
  }
}

// The state group's register tile of the 128 x 128 state: element [i][c] of
// st is row 8 ig + i, column 32 (c / 4) + 4 jg + c % 4 (ig = gt / 8, jg = gt % 8).
__device__ __forceinline__ void group_state_store(const float (&st)[8][16], float* dst, int ld,
                                                  int gt) {
  const int ig = gt >> 3, jg = gt & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int g = 0; g < 4; ++g)
      *(float4*)(dst + (size_t)(8 * ig + i) * ld + 32 * g + 4 * jg) =
          make_float4(st[i][4 * g], st[i][4 * g + 1], st[i][4 * g + 2], st[i][4 * g + 3]);
}
__device__ __forceinline__ void group_state_load(float (&st)[8][16], const float* src, int gt) {
  const int ig = gt >> 3, jg = gt & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float4 x = src ? *(const float4*)(src + (size_t)(8 * ig + i) * D + 32 * g + 4 * jg)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      st[i][4 * g] = x.x;
      st[i][4 * g + 1] = x.y;
      st[i][4 * g + 2] = x.z;
      st[i][4 * g + 3] = x.w;
    }
}
// Rows row0 .. row0 + 15 of head h of a [tokens, H, D] tensor into a dense
// [16][D] shared tile with cp.async, issued by the 128 threads of one group.
template <typename T>
__device__ __forceinline__ void stage_rows_group(const T* g, T* s, const BwdDev& a, int64_t row0,
                                                 int h, int nvalid, int gt) {
  constexpr int kUnits = (int)(D * sizeof(T) / 16);
  constexpr int kElems = (int)(16 / sizeof(T));
  const T* g0 = g + (row0 * a.H + h) * D;
  for (int u = gt; u < C * kUnits; u += kGroup) {
    const int t = u / kUnits, o = (u % kUnits) * kElems;
    const bool ok = t < nvalid;
    cp_async16(s + t * D + o, (ok ? g0 + (int64_t)t * a.H * D : g0) + o, ok);
  }
}

constexpr int BUF_F = 3 * TILE_F + SM16_F + D + C;  // one prep buffer: Kt, KhC, V/R, Tb, e^{G_C}, beta
static_assert(BUF_F % 4 == 0, "prep buffers on 16-byte boundaries");

template <typename Tin>
__device__ __forceinline__ void states_chain(const BwdDev& a, int64_t chain) {
  extern __shared__ __align__(16) float smf[];
  float* S = smf;                       // the state group's copy of S for Kt S
  float* buf = S + STATE_F;             // two prep buffers
  float* Kh = buf + 2 * BUF_F;          // prep group: Kh, Ab, M, inverse scratch
  float* Ab = Kh + TILE_F;
  float* M = Ab + SM16_F;
  float* scr = M + SM16_F;
  float* U = scr + 5 * SM16_F;          // state group: U and the partial sums of Kt S
  float* part = U + TILE_F;
  Tin* sth = (Tin*)(part + 2 * TILE_F);  // prep group: staged theta, k, v of the next chunk
  Tin* sk = sth + C * D;
  Tin* sv = sk + C * D;
  const int tid = threadIdx.x;
  const bool state_group = tid < kGroup;
  const int gt = state_group ? tid : tid - kGroup;
  const int64_t b = chain / a.H;
  const int h = (int)(chain - b * a.H);
  auto Ktb = [&](int s_) { return buf + s_ * BUF_F; };
  auto KhCb = [&](int s_) { return buf + s_ * BUF_F + TILE_F; };
  auto Vb = [&](int s_) { return buf + s_ * BUF_F + 2 * TILE_F; };
  auto Tbb = [&](int s_) { return buf + s_ * BUF_F + 3 * TILE_F; };
  auto ecb = [&](int s_) { return buf + s_ * BUF_F + 3 * TILE_F + SM16_F; };
  auto btb = [&](int s_) { return buf + s_ * BUF_F + 3 * TILE_F + SM16_F + D; };

  if (!state_group) {
    // ---------------- prep group: chunk n's operands, Ab and the inverse
    auto stage = [&](int n) -> float {  // issue chunk n's copies; returns its beta for this thread
      const int nv = min(C, a.T - n * C);
      const int64_t r0 = b * a.T + (int64_t)n * C;
      stage_rows_group((const Tin*)a.theta, sth, a, r0, h, nv, gt);
      stage_rows_group((const Tin*)a.k, sk, a, r0, h, nv, gt);
      stage_rows_group((const Tin*)a.v, sv, a, r0, h, nv, gt);
      cp_async_commit();
      return load_beta<Tin>(a, r0, h, nv);  // thread kGroup + t holds beta_t
    };
    float bnext = stage(0);
    for (int n = 0; n < a.nch; ++n) {
      const int bs = n & 1;
      const int nvalid = min(C, a.T - n * C);
      if (n >= 2) bar_sync_all(BAR_FREE + bs);  // the state group is done with chunk n - 2
      cp_async_wait_all();
      bar_group(BAR_PG);  // the staged chunk is complete
      prep_chunk<Tin>(sth, sk, sv, bnext, a.g_min, a.log_decay, nvalid, Ktb(bs), Kh, KhCb(bs),
                      ecb(bs), btb(bs), Vb(bs), gt);
      bar_group(BAR_PG);  // the staging reads are done and the tiles complete
      if (n + 1 < a.nch) bnext = stage(n + 1);
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int e = gt + kGroup * e2, m = e >> 4, nn = e & 15;
        Ab[m * LS + nn] = nn < m ? dot128(Ktb(bs), m, Kh, nn) : 0.0f;
      }
      bar_group(BAR_PG);
      wy_inverse_group(Ab, btb(bs), M, Tbb(bs), nullptr, scr, gt, BAR_PG);
      bar_arrive_all(BAR_READY + bs);  // buffer bs holds chunk n
    }
    return;
  }

  // ---------------- state group: S in registers (an 8 x 16 tile per thread)
  float* Sw = a.ws_S + (size_t)chain * a.nch * kStateF;
  float* RUw = a.ws_RU + (size_t)chain * a.nch * 2 * C * D;
  float st[8][16];
  group_state_load(st, a.init_state ? a.init_state + chain * kStateF : nullptr, gt);
  for (int n = 0; n < a.nch; ++n) {
    const int bs = n & 1;
    float* Kt = Ktb(bs);
    float* V = Vb(bs);
    group_state_store(st, Sw + (size_t)n * kStateF, D, gt);
    group_state_store(st, S, LD, gt);
    bar_sync_all(BAR_READY + bs);  // chunk n's operands are ready; S is visible to the group
    {
      // Kt S as two partial sums over 64 key channels each
      const int ng = gt & 31, mg = (gt >> 5) & 1, ks = gt >> 6;
      float acc[8][4];
#pragma unroll
      for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[m][t] = 0.0f;
      gemm_acc<8, 4, true, true>(acc, Kt, LD, 8 * mg, S, LD, 4 * ng, 0, 64 * ks, 64 * ks + 64);
#pragma unroll
      for (int m = 0; m < 8; ++m)
        *(float4*)(part + (ks * C + 8 * mg + m) * LD + 4 * ng) =
            make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    }
    bar_group(BAR_SG);
    for (int e = gt; e < C * D / 4; e += kGroup) {  // R = V - Kt S, in place of V
      const int m = e >> 5, nn = (e & 31) * 4;
      const float4 p0 = *(const float4*)(part + m * LD + nn);
      const float4 p1 = *(const float4*)(part + (C + m) * LD + nn);
      float4 r = *(const float4*)(V + m * LD + nn);
      r.x = fmaf(-1.0f, p0.x + p1.x, r.x);
      r.y = fmaf(-1.0f, p0.y + p1.y, r.y);
      r.z = fmaf(-1.0f, p0.z + p1.z, r.z);
      r.w = fmaf(-1.0f, p0.w + p1.w, r.w);
      *(float4*)(V + m * LD + nn) = r;
    }
    bar_group(BAR_SG);
    {
      // U = Tb R: rows 4 mg .. 4 mg + 3, columns 4 ng .. 4 ng + 3
      const int ng = gt & 31, mg = gt >> 5;
      float acc[4][4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[m][t] = 0.0f;
      gemm_acc<4, 4, true, true>(acc, Tbb(bs), LS, 4 * mg, V, LD, 4 * ng, 0, 0, C);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        *(float4*)(U + (4 * mg + m) * LD + 4 * ng) = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    }
    bar_group(BAR_SG);
    // R and U of the chunk for the gradient kernel
    for (int e = gt; e < 2 * C * D / 4; e += kGroup) {
      const int t = (e >> 5) & (C - 1), c = (e & 31) * 4;
      const float* src = (e < C * D / 4 ? V : U) + t * LD + c;
      *(float4*)(RUw + (size_t)n * 2 * C * D + (e >> 5) * D + c) = *(const float4*)src;
    }
    if (n + 1 < a.nch) {
      // S' = Diag(ec) S + KhC^T U (the last chunk's end state is not needed)
      const int ig = gt >> 3, jg = gt & 7;
      const float* ec = ecb(bs);
      const float* KhC = KhCb(bs);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float e = ec[8 * ig + i];
#pragma unroll
        for (int j = 0; j < 16; ++j) st[i][j] *= e;
      }
#pragma unroll 4
      for (int k = 0; k < C; ++k) {
        const float4 a0 = *(const float4*)(KhC + k * LD + 8 * ig);
        const float4 a1 = *(const float4*)(KhC + k * LD + 8 * ig + 4);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float4 bv = *(const float4*)(U + k * LD + 32 * g + 4 * jg);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            ffma2(st[i][4 * g], st[i][4 * g + 1], av[i], bv.x, bv.y);
            ffma2(st[i][4 * g + 2], st[i][4 * g + 3], av[i], bv.z, bv.w);
          }
        }
      }
    }
    // buffer bs may take chunk n + 2 (the prep group waits for this only then)
    if (n + 2 < a.nch) bar_arrive_all(BAR_FREE + bs);
  }
}

// ------------------------------------------------------- reverse recurrence
// Warp-specialised like the forward recurrence: the prep group forms chunk n's
// operands -- Qt, -Kt, Kh, KhC, dO, Ab, Pi^T, the inverse and Pi^T dO, none of
// which needs dS -- while the state group runs chunk n + 1's products with dS.

// The reverse recurrence's per-channel operands (prep group, one channel per
// thread): Qt = Q e^{G}, -Kt, Kh, KhC and e^{G_C} by the products of
// prep_chunk, and the chunk's d_out rows from the staged copy.
template <typename Tin>
__device__ __forceinline__ void prep_chunk_rev(const Tin* th0, const Tin* k0, const Tin* q0,
                                               const float* sdo, float bval, float g_min,
                                               int log_decay, int nvalid, float* Qt, float* mKt,
                                               float* Kh, float* KhC, float* dO, float* ec,
                                               float* bt, int gt) {
  const int c = gt;
  float xr[C], kr[C], qr[C], egr[C];
#pragma unroll
  for (int t = 0; t < C; ++t) {
    const bool ok = t < nvalid;
    xr[t] = ok ? to_f32(th0[t * D + c]) : 0.0f;
    kr[t] = ok ? to_f32(k0[t * D + c]) : 0.0f;
    qr[t] = ok ? to_f32(q0[t * D + c]) : 0.0f;
  }
  float E = 1.0f, Ei = 1.0f;
#pragma unroll
  for (int t = 0; t < C; ++t) {
    float g = 0.0f;
    if (t < nvalid) {
      if (log_decay) {
        g = xr[t];
      } else {
        const float x = xr[t];
        const float e = expf(-fabsf(x));
        const float big = 1.0f / (1.0f + e), small = e * big;
        g = g_min * (x >= 0.0f ? big : small);
      }
    }
    const float eg = expf(g);
    E *= eg;
    Ei *= 1.0f / eg;
    egr[t] = eg;
    Qt[t * LD + c] = qr[t] * E;
    mKt[t * LD + c] = -(kr[t] * E);
    Kh[t * LD + c] = kr[t] * Ei;
    dO[t * LD + c] = sdo[t * D + c];
  }
  ec[c] = E;
  float P = 1.0f;
#pragma unroll
  for (int t = C - 1; t >= 0; --t) {
    KhC[t * LD + c] = kr[t] * P;
    P *= egr[t];
  }
  if (gt < C) bt[gt] = bval;
}

// one prep buffer of the reverse recurrence: [Qt; -Kt], [dO; dR], KhC, dU,
// Tb^T, e^{G_C}, beta
constexpr int BUF_R = 6 * TILE_F + SM16_F + D + C;
static_assert(BUF_R % 4 == 0, "prep buffers on 16-byte boundaries");

template <typename Tin>
__device__ __forceinline__ void reverse_chain(const BwdDev& a, int64_t chain) {
  extern __shared__ __align__(16) float smf[];
  float* dS = smf;                       // the state group's copy of dS' for KhC dS'
  float* buf = dS + STATE_F;             // two prep buffers
  float* Kh = buf + 2 * BUF_R;           // prep group: Kh, Ab, Pi^T, M, Tb, inverse scratch
  float* Ab = Kh + TILE_F;
  float* PiT = Ab + SM16_F;
  float* M = PiT + SM16_F;
  float* Tb = M + SM16_F;
  float* scr = Tb + SM16_F;
  float* sdo = scr + 5 * SM16_F;         // prep group: staged d_out, theta, k, q of the next chunk
  Tin* sth = (Tin*)(sdo + C * D);
  Tin* sk = sth + C * D;
  Tin* sq = sk + C * D;
  const int tid = threadIdx.x;
  const bool state_group = tid < kGroup;
  const int gt = state_group ? tid : tid - kGroup;
  const int64_t b = chain / a.H;
  const int h = (int)(chain - b * a.H);
  auto Qtb = [&](int s_) { return buf + s_ * BUF_R; };                 // then -Kt
  auto dOb = [&](int s_) { return buf + s_ * BUF_R + 2 * TILE_F; };    // then dR
  auto KhCb = [&](int s_) { return buf + s_ * BUF_R + 4 * TILE_F; };
  auto dUb = [&](int s_) { return buf + s_ * BUF_R + 5 * TILE_F; };
  auto TbTb = [&](int s_) { return buf + s_ * BUF_R + 6 * TILE_F; };
  auto ecb = [&](int s_) { return buf + s_ * BUF_R + 6 * TILE_F + SM16_F; };
  auto btb = [&](int s_) { return buf + s_ * BUF_R + 6 * TILE_F + SM16_F + D; };

  if (!state_group) {
    // ---------------- prep group, chunks from the last to the first
    auto stage = [&](int n) -> float {  // issue chunk n's copies; returns its beta for this thread
      const int nv = min(C, a.T - n * C);
      const int64_t r0 = b * a.T + (int64_t)n * C;
      stage_rows_group(a.d_out, sdo, a, r0, h, nv, gt);
      stage_rows_group((const Tin*)a.theta, sth, a, r0, h, nv, gt);
      stage_rows_group((const Tin*)a.k, sk, a, r0, h, nv, gt);
      stage_rows_group((const Tin*)a.q, sq, a, r0, h, nv, gt);
      cp_async_commit();
      return load_beta<Tin>(a, r0, h, nv);  // thread kGroup + t holds beta_t
    };
    float bnext = stage(a.nch - 1);
    for (int i = 0; i < a.nch; ++i) {
      const int n = a.nch - 1 - i, bs = i & 1;
      const int nvalid = min(C, a.T - n * C);
      float* Qt = Qtb(bs);
      float* dO = dOb(bs);
      if (i >= 2) bar_sync_all(BAR_FREE + bs);  // the state group is done with chunk n + 2
      cp_async_wait_all();
      bar_group(BAR_PG);  // the staged chunk is complete
      prep_chunk_rev<Tin>(sth, sk, sq, sdo, bnext, a.g_min, a.log_decay, nvalid, Qt, Qt + TILE_F, Kh,
                          KhCb(bs), dO, ecb(bs), btb(bs), gt);
      bar_group(BAR_PG);  // the staging reads are done and the tiles complete
      if (n > 0) bnext = stage(n - 1);
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int e = gt + kGroup * e2, m = e >> 4, nn = e & 15;
        Ab[m * LS + nn] = nn < m ? -dot128(Qt + TILE_F, m, Kh, nn) : 0.0f;
        PiT[nn * LS + m] = nn <= m ? dot128(Qt, m, Kh, nn) : 0.0f;
      }
      bar_group(BAR_PG);
      {
        // Pi^T dO, the part of dU that does not involve dS'
        const int ng = gt & 31, mg = gt >> 5;
        float acc[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int t = 0; t < 4; ++t) acc[m][t] = 0.0f;
        gemm_acc<4, 4, true, true>(acc, PiT, LS, 4 * mg, dO, LD, 4 * ng, 0, 0, C);
        float* dU = dUb(bs);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          *(float4*)(dU + (4 * mg + m) * LD + 4 * ng) =
              make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
      }
      wy_inverse_group(Ab, btb(bs), M, Tb, TbTb(bs), scr, gt, BAR_PG);
      bar_arrive_all(BAR_READY + bs);  // buffer bs holds chunk n
    }
    return;
  }

  // ---------------- state group: dS in registers (an 8 x 16 tile per thread)
  float* dSw = a.ws_dS + (size_t)chain * a.nch * kStateF;
  float* dUw = a.ws_dU + (size_t)chain * a.nch * C * D;
  float st[8][16];
  group_state_load(st, a.d_final ? a.d_final + chain * kStateF : nullptr, gt);
  for (int i = 0; i < a.nch; ++i) {
    const int n = a.nch - 1 - i, bs = i & 1;
    const int t0 = n * C, nvalid = min(C, a.T - t0);
    const int64_t row0 = b * a.T + t0;
    float* dU = dUb(bs);
    float* dR = dOb(bs) + TILE_F;
    group_state_store(st, dSw + (size_t)n * kStateF, D, gt);
    group_state_store(st, dS, LD, gt);
    bar_sync_all(BAR_READY + bs);  // chunk n's operands are ready; dS' is visible to the group
    const int ng = gt & 31, mg = gt >> 5;
    {
      // dU = Pi^T dO + KhC dS'
      float acc[4][4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[m][t] = 0.0f;
      gemm_acc<4, 4, true, true>(acc, KhCb(bs), LD, 4 * mg, dS, LD, 4 * ng, 0, 0, D);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float4* o = (float4*)(dU + (4 * mg + m) * LD + 4 * ng);
        float4 r = *o;
        r.x = fmaf(1.0f, acc[m][0], r.x);
        r.y = fmaf(1.0f, acc[m][1], r.y);
        r.z = fmaf(1.0f, acc[m][2], r.z);
        r.w = fmaf(1.0f, acc[m][3], r.w);
        *o = r;
      }
    }
    bar_group(BAR_SG);
    for (int e = gt; e < C * D / 4; e += kGroup) {
      const int t = e >> 5, c = (e & 31) * 4;
      *(float4*)(dUw + (size_t)n * C * D + t * D + c) = *(const float4*)(dU + t * LD + c);
    }
    {
      // dR = Tb^T dU
      float acc[4][4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[m][t] = 0.0f;
      gemm_acc<4, 4, true, true>(acc, TbTb(bs), LS, 4 * mg, dU, LD, 4 * ng, 0, 0, C);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        *(float4*)(dR + (4 * mg + m) * LD + 4 * ng) =
            make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    }
    bar_group(BAR_SG);
    for (int e = gt; e < C * D; e += kGroup) {
      const int t = e >> 7, c = e & (D - 1);
      if (t < nvalid) a.dv[((row0 + t) * a.H + h) * D + c] = dR[t * LD + c];
    }
    {
      // dS = Diag(ec) dS' + [Qt; -Kt]^T [dO; dR]
      const int ig = gt >> 3, jg = gt & 7;
      const float* ec = ecb(bs);
      const float* A = Qtb(bs);
      const float* B = dOb(bs);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float e = ec[8 * ig + r];
#pragma unroll
        for (int j = 0; j < 16; ++j) st[r][j] *= e;
      }
#pragma unroll 4
      for (int k = 0; k < 2 * C; ++k) {
        const float4 a0 = *(const float4*)(A + k * LD + 8 * ig);
        const float4 a1 = *(const float4*)(A + k * LD + 8 * ig + 4);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float4 bv = *(const float4*)(B + k * LD + 32 * g + 4 * jg);
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            ffma2(st[r][4 * g], st[r][4 * g + 1], av[r], bv.x, bv.y);
            ffma2(st[r][4 * g + 2], st[r][4 * g + 3], av[r], bv.z, bv.w);
          }
        }
      }
    }
    // buffer bs may take chunk n - 2 (the prep group waits for this only then)
    if (i + 2 < a.nch) bar_arrive_all(BAR_FREE + bs);
  }
  if (a.d_init) group_state_store(st, a.d_init + chain * kStateF, D, gt);
}

// The two recurrences of every chain are independent of each other: items
// 0 .. chains-1 of the work queue run the reverse recurrence (the longer one
// per chunk), items chains .. 2 chains-1 the forward one.
template <typename Tin>
__device__ __forceinline__ void recurrence_item(const BwdDev& a, int64_t chains, int64_t item) {
  if (item < chains)
    reverse_chain<Tin>(a, item);
  else
    states_chain<Tin>(a, item - chains);
}

// ------------------------------------------------------ per-chunk gradients
// Every gradient of chunk n of one chain, item = chain * nch + n.
template <typename Tin>
__device__ __forceinline__ void grads_chunk(const BwdDev& a, int64_t item) {
  extern __shared__ __align__(16) float smf[];
  float* S = smf;  // S, then dS'
  float* Qt = S + STATE_F;
  float* Kt = Qt + TILE_F;
  float* Kh = Kt + TILE_F;
  float* KhC = Kh + TILE_F;
  float* EGt = KhC + TILE_F;  // e^{g} per token and channel
  float* dgt = EGt + TILE_F;
  float* U = dgt + TILE_F;
  float* X = U + TILE_F;  // [dO; -dR], then [dQt; dKt]
  float* dKh = X + 2 * TILE_F;
  float* V = dKh + TILE_F;  // V, then R, then row partials of dec
  float* dU = V + TILE_F;   // dU, then dKhC
  float* part = dU + TILE_F;  // 4 tiles
  float* Ab = part + 4 * TILE_F;
  float* Pi = Ab + SM16_F;
  float* M = Pi + SM16_F;
  float* Tb = M + SM16_F;
  float* TbT = Tb + SM16_F;
  float* dTb = TbT + SM16_F;  // dTb, then dA
  float* dPi = dTb + SM16_F;
  float* dPiT = dPi + SM16_F;
  float* dAb = dPiT + SM16_F;
  float* dAbT = dAb + SM16_F;
  float* Y = dAbT + SM16_F;
  float* ec = Y + SM16_F;
  float* dec = ec + D;
  float* bt = dec + D;
  float* dbt = bt + C;
  float* dpd = dbt + C;  // diagonal of dPi
  const int tid = threadIdx.x, ig = tid >> 4, jg = tid & 15;
  const int64_t chain = item / a.nch;
  const int n = (int)(item - chain * a.nch);
  const int64_t b = chain / a.H;
  const int h = (int)(chain - b * a.H);
  const int t0 = n * C, nvalid = min(C, a.T - t0);
  const int64_t row0 = b * a.T + t0;
  const size_t cidx = (size_t)chain * a.nch + n;
  const float* Sg = a.ws_S + cidx * kStateF;
  const float* dSg = a.ws_dS + cidx * kStateF;
  const float* dUg = a.ws_dU + cidx * C * D;
  const float* RUg = a.ws_RU + cidx * 2 * C * D;

  // Asynchronous copies straight into shared memory, in two groups: the
  // chunk's d_out rows, dU, R and U (first needed after the inverse), and,
  // once the chunk's inputs are loaded, S (first needed by [dO; -dR] S^T,
  // after every product that does not involve it).
  {
    const float* dO0 = a.d_out + (row0 * a.H + h) * D;
    for (int u = tid; u < C * D / 4; u += kThreads) {
      const int t = u >> 5, c = (u & 31) * 4;
      const bool ok = t < nvalid;  // d_out rows past the sequence end read as zero
      cp_async16(X + t * LD + c, dO0 + (ok ? (int64_t)t * a.H * D : 0) + c, ok);
      cp_async16(dU + t * LD + c, dUg + t * D + c, true);
    }
    for (int u = tid; u < 2 * C * D / 4; u += kThreads) {
      const int r = u >> 5, c = (u & 31) * 4;  // rows 0..15 R (into the V tile), 16..31 U
      cp_async16((r < C ? V : U) + (r & (C - 1)) * LD + c, RUg + r * D + c, true);
    }
    cp_async_commit();
  }
  // ---- the chunk's inputs: gate, decay factors and decayed operands
  {
    const int64_t g0 = (row0 * a.H + h) * D;
    load_chunk<Tin>((const Tin*)a.theta + g0, (const Tin*)a.k + g0, (const Tin*)a.q + g0,
                    (const Tin*)a.v + g0, (int64_t)a.H * D, load_beta<Tin>(a, row0, h, nvalid),
                    a.g_min, a.log_decay, nvalid, Qt, Kt, 1.0f, Kh, KhC, EGt, dgt, ec, bt, nullptr);
  }
  // S (the second copy group), issued after the chunk's own loads
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int e = tid + i * kThreads;
    cp_async16(S + (e >> 5) * LD + (e & 31) * 4, Sg + (size_t)(e >> 5) * D + (e & 31) * 4, true);
  }
  cp_async_commit();
  // this thread's tile of dS' (registers), loaded now so that its latency
  // overlaps the products before its first use
  float d[8][8];
  state_load(d, dSg);
  __syncthreads();
  {
    const int m = tid >> 4, nn = tid & 15;
    Ab[m * LS + nn] = nn < m ? dot128(Kt, m, Kh, nn) : 0.0f;
    Pi[m * LS + nn] = nn <= m ? dot128(Qt, m, Kh, nn) : 0.0f;
  }
  __syncthreads();
  wy_inverse(Ab, bt, M, Tb, TbT, part);  // (the partial sums' tiles are free here)
  cp_async_wait_one_pending();
  __syncthreads();  // d_out, dU, R and U have arrived
  small16<false>(TbT, dU, X + TILE_F, -1.0f);  // -dR = -Tb^T dU
  __syncthreads();
  {
    // dTb = lower_incl(dU R^T); dPi = lower_incl(dO U^T), its strictly lower
    // part kept as a matrix and its diagonal apart (dpd): the diagonal of Pi is
    // q_t . k_t, free of the decay, so its share of dq and dk is taken from q and
    // k directly and it has no share in dG
    const int m = tid >> 4, nn = tid & 15;
    dTb[m * LS + nn] = nn <= m ? dot128(dU, m, V, nn) : 0.0f;
    const float p = nn <= m ? dot128(X, m, U, nn) : 0.0f;
    dPi[m * LS + nn] = nn < m ? p : 0.0f;
    dPiT[nn * LS + m] = nn < m ? p : 0.0f;
    if (nn == m) dpd[m] = p;
  }
  cp_async_wait_all();
  __syncthreads();  // S has arrived
  part32_nk(X, S, part);  // [dO; -dR] S^T
  __syncthreads();
  {
    // Y = (dTb Diag(b)) M^T; db (first part) = column sums of M * dTb
    const int i = tid >> 4, j = tid & 15;
    float y = 0.0f;
#pragma unroll
    for (int l = 0; l < C; ++l) y = fmaf(dTb[i * LS + l] * bt[l], M[j * LS + l], y);
    Y[i * LS + j] = y;
    if (tid < C) {
      float s = 0.0f;
#pragma unroll
      for (int r = 0; r < C; ++r) s = fmaf(M[r * LS + tid], dTb[r * LS + tid], s);
      dbt[tid] = s;
    }
  }
  reduce_parts<2 * C, 2>(part, X, nullptr, 1.0f);  // [dQt; dKt], the S^T parts
  {
    // dec_i = sum_j dS'_ij S_ij: row partials of this thread's tile
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float s = 0.0f;
#pragma unroll
      for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          s = fmaf(d[i][4 * g + c], S[(8 * ig + i) * LD + 64 * g + 4 * jg + c], s);
      V[jg * LD + 8 * ig + i] = s;
    }
  }
  __syncthreads();
  state_store(d, S, LD);  // S is no longer needed: dS' takes its place
  {
    // dA = -strict_lower(M^T Y) (kept in dTb's place), dAb = Diag(b) dA
    const int i = tid >> 4, j = tid & 15;
    float s = 0.0f;
#pragma unroll
    for (int l = 0; l < C; ++l) s = fmaf(M[l * LS + i], Y[l * LS + j], s);
    const float dA = i > j ? -s : 0.0f;
    dTb[i * LS + j] = dA;
    dAb[i * LS + j] = bt[i] * dA;
    dAbT[j * LS + i] = bt[i] * dA;
  }
  if (tid < D) {
    float s = 0.0f;
#pragma unroll
    for (int r = 0; r < 16; ++r) s += V[r * LD + tid];
    dec[tid] = s;
  }
  __syncthreads();
  part16<false>(U, S, part);  // U dS'^T
  if (tid < C) {
    float s = dbt[tid];
#pragma unroll
    for (int l = 0; l < C; ++l) s = fmaf(dTb[tid * LS + l], Ab[tid * LS + l], s);
    dbt[tid] = s;
  }
  small16<true>(dPi, Kh, X, 1.0f);           // dQt += dPi Kh (strictly lower dPi)
  small16<true>(dAb, Kh, X + TILE_F, 1.0f);  // dKt += Diag(b) dA Kh
  small16<false>(dPiT, Qt, dKh, 1.0f);       // dKh = dPi^T Qt (strictly lower dPi)
  __syncthreads();
  small16<true>(dAbT, Kt, dKh, 1.0f);           // dKh += (Diag(b) dA)^T Kt
  reduce_parts<C, 4>(part, dU, nullptr, 1.0f);  // dKhC
  __syncthreads();
  // ---- per channel: dK, dQ, dG and the reverse cumulative sum.  The KhC
  // terms enter dg_s as -sum_{t >= s} dKhC_t KhC_t (through dG_t) plus
  // sum_t dKhC_t KhC_t (through dG_C); they are summed in the equal closed
  // form sum_{t < s} dKhC_t KhC_t, which avoids cancelling two large sums when
  // the last tokens' terms dominate (fast decay).
  // Two threads per channel: thread (c, half) takes tokens 8 half .. 8 half + 7.
  // The running products and sums that cross the two halves go through
  // shared memory (the dead partial-sum tiles), each formed in the order of
  // one sequential pass, so the results equal that pass bit for bit.
  constexpr int CH = C / 2;
  const int c = tid & (D - 1), hf = tid >> 7, tb = hf * CH;
  float* xs = part;  // [5][D]: E and e^{-G} after token 7, prefix sum, suffix product, suffix sum
  float egl[CH], dG[CH];
  {
    float run = 0.0f;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int t = tb + i;
      egl[i] = EGt[t * LD + c];
      const float dqt = X[t * LD + c], dkt = X[(C + t) * LD + c];
      dG[i] = dkt * Kt[t * LD + c] + dqt * Qt[t * LD + c] - dKh[t * LD + c] * Kh[t * LD + c];
      run = fmaf(dU[t * LD + c], KhC[t * LD + c], run);
    }
    if (hf == 0) {
      float E = 1.0f, Ei = 1.0f;
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        E *= egl[i];
        Ei *= 1.0f / egl[i];
      }
      xs[c] = E;
      xs[D + c] = Ei;
      xs[2 * D + c] = run;
    } else {
      float P = 1.0f, acc = 0.0f;
#pragma unroll
      for (int i = CH - 1; i >= 0; --i) {
        P *= egl[i];
        acc += dG[i];
      }
      xs[3 * D + c] = P;
      xs[4 * D + c] = acc;
    }
  }
  __syncthreads();
  {
    float E = hf ? xs[c] : 1.0f, Ei = hf ? xs[D + c] : 1.0f, run = hf ? xs[2 * D + c] : 0.0f;
    float P = hf ? 1.0f : xs[3 * D + c], acc = hf ? 0.0f : xs[4 * D + c];
    float sfx[CH];  // e^{G_C - G_t}
#pragma unroll
    for (int i = CH - 1; i >= 0; --i) {
      sfx[i] = P;
      P *= egl[i];
    }
    float qr[CH], kr[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int t = tb + i;
      const int64_t o = ((row0 + t) * a.H + h) * D + c;
      qr[i] = t < nvalid ? to_f32(((const Tin*)a.q)[o]) : 0.0f;
      kr[i] = t < nvalid ? to_f32(((const Tin*)a.k)[o]) : 0.0f;
    }
    float pre[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int t = tb + i;
      E *= egl[i];
      Ei *= 1.0f / egl[i];
      const float dqt = X[t * LD + c], dkt = X[(C + t) * LD + c];
      const float dkh = dKh[t * LD + c], dkhc = dU[t * LD + c];
      pre[i] = run;  // sum_{u < t} dKhC_u KhC_u
      run = fmaf(dkhc, KhC[t * LD + c], run);
      if (t < nvalid) {
        const int64_t o = ((row0 + t) * a.H + h) * D + c;
        a.dq[o] = fmaf(dpd[t], kr[i], dqt * E);
        a.dk[o] = fmaf(dpd[t], qr[i], dkt * E + dkh * Ei + dkhc * sfx[i]);
      }
    }
    const float dec_ec = dec[c] * ec[c];
#pragma unroll
    for (int i = CH - 1; i >= 0; --i) {
      const int t = tb + i;
      acc += dG[i];
      if (t < nvalid)
        a.dtheta[((row0 + t) * a.H + h) * D + c] = (acc + pre[i] + dec_ec) * dgt[t * LD + c];
    }
  }
  if (tid < nvalid) a.dbeta[(row0 + tid) * a.H + h] = dbt[tid];
}

// Bytes of the work queue at the end of the workspace: the queue position
// (256 bytes, for alignment), then one int per chain, rounded up to 256 bytes.
constexpr size_t queue_bytes(int64_t chains) {
  return 256 + ((size_t)chains * sizeof(int) + 255) / 256 * 256;
}

// Waits until *f >= want (acquire); gives up after limit_ns.
__device__ __forceinline__ bool wait_count(const int* f, int want, uint64_t limit_ns) {
  auto ld = [](const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
  };
  if (ld(f) >= want) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    __nanosleep(1000);
    if (ld(f) >= want) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > limit_ns) return false;
  }
}

// The whole backward pass as one persistent launch over a work queue (one CTA
// per SM).  A CTA takes the next item from a counter in the workspace: first
// the 2 x chains recurrences (reverse ones first: the longest first), then the
// chains * nch per-chunk gradient items, chain by chain.  A gradient item
// needs both recurrences of its chain: it waits for the chain's count of
// finished recurrences to reach 2.  Every recurrence item is taken before any
// gradient item, and only by a running CTA, so the waits always end; meanwhile
// the SMs that the recurrences' last wave leaves idle already run the
// gradients of the chains that are done (a separate gradient launch would
// start only after the last recurrence).  A wait that runs out (bounded by
// wait_ns) records KDA_ERR_DEVICE_TIMEOUT and skips the item.
template <typename Tin>
__global__ void __launch_bounds__(kThreads, 1) kda_bwd_kernel(const BwdDev a, int64_t chains) {
  __shared__ long long s_item;
  __shared__ int s_ok;
  const int64_t items = 2 * chains + chains * a.nch;
  for (;;) {
    if (threadIdx.x == 0) s_item = (long long)atomicAdd(a.q_next, 1ull);
    __syncthreads();
    const int64_t item = s_item;
    if (item >= items) break;
    if (item < 2 * chains) {
      recurrence_item<Tin>(a, chains, item);
      cp_async_wait_all();
      __threadfence();  // this thread's workspace writes, before the count
      __syncthreads();
      if (threadIdx.x == 0) atomicAdd(a.q_done + (item < chains ? item : item - chains), 1);
    } else {
      const int64_t g = item - 2 * chains;
      if (threadIdx.x == 0) {
        s_ok = wait_count(a.q_done + g / a.nch, 2, a.wait_ns);
        if (!s_ok) atomicExch(a.status, KDA_ERR_DEVICE_TIMEOUT);
      }
      __syncthreads();
      if (s_ok) grads_chunk<Tin>(a, g);
      cp_async_wait_all();
    }
    __syncthreads();  // the item's shared memory and s_item are free again
  }
}

template <typename Tin>
constexpr size_t smem_states() {
  return (size_t)(STATE_F + 2 * BUF_F + TILE_F + 7 * SM16_F + TILE_F + 2 * TILE_F) * 4 +
         3 * C * D * sizeof(Tin);
}
template <typename Tin>
constexpr size_t smem_reverse() {
  return (size_t)(STATE_F + 2 * BUF_R + TILE_F + 9 * SM16_F + C * D) * 4 + 3 * C * D * sizeof(Tin);
}
constexpr size_t kSmemGrads = (size_t)(STATE_F + 16 * TILE_F + 11 * SM16_F + 2 * D + 3 * C) * 4;
static_assert(kSmemGrads <= 232448 && smem_reverse<float>() <= 232448 &&
                  smem_states<float>() <= 232448,
              "shared memory budget");

template <typename Tin>
int launch_bwd_t(const BwdDev& d, int64_t chains, cudaStream_t stream) {
  constexpr size_t kSmemRec =
      smem_states<Tin>() > smem_reverse<Tin>() ? smem_states<Tin>() : smem_reverse<Tin>();
  constexpr size_t kSmem = kSmemRec > kSmemGrads ? kSmemRec : kSmemGrads;
  const void* fn = (const void*)kda_bwd_kernel<Tin>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) !=
      cudaSuccess)
    return KDA_ERR_LAUNCH;
  int dev = 0, nsm = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, kSmem) != cudaSuccess ||
      nsm <= 0 || per_sm <= 0)
    return KDA_ERR_LAUNCH;
  const int64_t items = 2 * chains + chains * d.nch;
  const int64_t grid = items < (int64_t)nsm * per_sm ? items : (int64_t)nsm * per_sm;
  // the queue position and the per-chain counts start at zero
  if (cudaMemsetAsync(d.q_next, 0, queue_bytes(chains), stream) != cudaSuccess) return KDA_ERR_CUDA;
  kda_bwd_kernel<Tin><<<(unsigned)grid, kThreads, kSmem, stream>>>(d, chains);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // namespace

size_t bwd_workspace_size(int B, int H, int T) {
  const size_t nch = ((size_t)T + C - 1) / C;
  return (size_t)B * H * nch * (2 * kStateF + (size_t)3 * C * D) * sizeof(float) +
         queue_bytes((int64_t)B * H);
}

// (dk = dv = 128 is checked by the caller)
int launch_bwd(const BwdParams& p, cudaStream_t stream) {
  const int64_t chains = (int64_t)p.B * p.H;
  if (chains == 0 || p.T == 0) return KDA_OK;
  const int nch = (p.T + C - 1) / C;
  if (chains * nch > (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
  BwdDev d;
  d.q = p.q;
  d.k = p.k;
  d.v = p.v;
  d.theta = p.theta;
  d.beta = p.beta;
  d.g_min = p.g_min;
  d.log_decay = p.gate == KDA_GATE_LOG_DECAY;
  d.init_state = p.init_state;
  d.d_out = p.d_out;
  d.d_final = p.d_final;
  d.dq = p.dq;
  d.dk = p.dk;
  d.dv = p.dv;
  d.dtheta = p.dtheta;
  d.dbeta = p.dbeta;
  d.d_init = p.d_init;
  d.ws_S = (float*)p.workspace;
  d.ws_dS = d.ws_S + (size_t)chains * nch * kStateF;
  d.ws_dU = d.ws_dS + (size_t)chains * nch * kStateF;
  d.ws_RU = d.ws_dU + (size_t)chains * nch * C * D;
  d.q_next = (unsigned long long*)(d.ws_RU + (size_t)chains * nch * 2 * C * D);
  d.q_done = (int*)((unsigned char*)d.q_next + 256);
  d.status = status_word_device_ptr();
  if (!d.status) return KDA_ERR_CUDA;
  // a gradient item may wait for a whole recurrence of its chain (about 10 us
  // per chunk): 2 s plus 50 us per chunk
  d.wait_ns = 2000000000ull + (uint64_t)nch * 50000ull;
  d.H = p.H;
  d.T = p.T;
  d.nch = nch;
  if (p.dtype == KDA_DTYPE_F32) return launch_bwd_t<float>(d, chains, stream);
  return launch_bwd_t<__nv_bfloat16>(d, chains, stream);
}

}  // namespace kda
