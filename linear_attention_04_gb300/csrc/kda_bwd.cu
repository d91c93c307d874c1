// kda_bwd.cu -- backward pass of the KDA recurrence (gradients of the forward
// pass w.r.t. q, k, v, theta, beta and the initial state), fp32 on CUDA cores.
//
// Forward ("Kimi K3 Deep Dive", section "Core Innovation 1"; gate of
// "Architecture Deep Dive", sec. 3.2), per (sequence, head), token t:
//   X = Diag(e^{g}) S_{t-1},  u = beta (v - X^T k),  S_t = X + k u^T,  o = S_t^T q.
// Reverse pass with L = dL/dS_t (the gradient flowing back from later tokens
// plus q do^T from this token's output):
//   dq = S_t do,  kL = L^T k,  dv = beta kL,  dbeta = kL . (v - X^T k),
//   dk = L u - beta X kL,  dX = L - beta k kL^T,  dg_i = sum_j dX_ij X_ij,
//   dtheta = dg * g_min sigmoid(theta) (1 - sigmoid(theta))  (or dg for a given
//   log-decay),  L <- Diag(e^{g}) dX  (the gradient w.r.t. S_{t-1}).
//
// One CTA per chain, 256 threads in a 16 x 16 grid; thread (r, c) holds the
// 8 x 8 tiles [8r, 8r+8) x [8c, 8c+8) of S and L in registers.  Row and column
// sums go through shared memory (16 partials per row or column).  States
// before each token come from a two-level recomputation over the caller's
// workspace: the state every kBlock tokens (forward pass), then, per block in
// reverse order, the kBlock states of the block.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_device.cuh"
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int D = 128;         // dk = dv
constexpr int TT = 8;          // tile edge per thread
constexpr int NT = D / TT;     // 16 tiles per edge
constexpr int kThreads = NT * NT;
constexpr int kBlock = 64;     // tokens per recomputation block
constexpr size_t kState = (size_t)D * D;  // floats per state

struct BwdShared {
  float q[D], k[D], e[D], dgate[D];  // token vectors (e = e^{g}, dgate = dg/dtheta)
  float v[D], dout[D];
  float colp[NT][D];   // column partial sums (one per tile row)
  float rowp[NT][D];   // row partial sums (one per tile column)
  float vec[3][D];     // reduced vectors: u, kL, kL * (v - X^T k)
  float beta;
};

template <typename Tin>
__device__ __forceinline__ void load_token(BwdShared& sh, const Tin* q, const Tin* k, const Tin* v,
                                           const Tin* theta, const Tin* beta, const float* dout,
                                           int64_t row, float g_min, int gate, int tid) {
  if (tid < D) {
    const float th = to_f32(theta[row * D + tid]);
    float g, dg;
    if (gate == KDA_GATE_LOG_DECAY) {
      g = th;
      dg = 1.0f;
    } else {
      const float s = 1.0f / (1.0f + expf(-th));
      g = g_min * s;
      dg = g_min * s * (1.0f - s);
    }
    sh.e[tid] = expf(g);
    sh.dgate[tid] = dg;
    sh.q[tid] = to_f32(q[row * D + tid]);
    sh.k[tid] = to_f32(k[row * D + tid]);
  } else {
    const int j = tid - D;
    sh.v[j] = to_f32(v[row * D + j]);
    sh.dout[j] = dout ? dout[row * D + j] : 0.0f;
  }
  if (tid == 0) sh.beta = to_f32(beta[row]);
}

// S <- X + k u^T with X = Diag(e) S, u = beta (v - X^T k); tile form.
__device__ __forceinline__ void fwd_step(BwdShared& sh, float (&S)[TT][TT], int r, int c, int tid) {
#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int b = 0; b < TT; ++b) S[a][b] *= sh.e[TT * r + a];
  // column sums of k_i X_ij
#pragma unroll
  for (int b = 0; b < TT; ++b) {
    float p = 0.0f;
#pragma unroll
    for (int a = 0; a < TT; ++a) p = fmaf(sh.k[TT * r + a], S[a][b], p);
    sh.colp[r][TT * c + b] = p;
  }
  __syncthreads();
  if (tid < D) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < NT; ++i) s += sh.colp[i][tid];
    sh.vec[0][tid] = sh.beta * (sh.v[tid] - s);  // u
  }
  __syncthreads();
#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int b = 0; b < TT; ++b) S[a][b] = fmaf(sh.k[TT * r + a], sh.vec[0][TT * c + b], S[a][b]);
}

__device__ __forceinline__ void load_tile(float (&S)[TT][TT], const float* src, int r, int c) {
#pragma unroll
  for (int a = 0; a < TT; ++a) {
    const float4* p = (const float4*)(src + (size_t)(TT * r + a) * D + TT * c);
    const float4 x = p[0], y = p[1];
    S[a][0] = x.x; S[a][1] = x.y; S[a][2] = x.z; S[a][3] = x.w;
    S[a][4] = y.x; S[a][5] = y.y; S[a][6] = y.z; S[a][7] = y.w;
  }
}

__device__ __forceinline__ void store_tile(const float (&S)[TT][TT], float* dst, int r, int c) {
#pragma unroll
  for (int a = 0; a < TT; ++a) {
    float4* p = (float4*)(dst + (size_t)(TT * r + a) * D + TT * c);
    p[0] = make_float4(S[a][0], S[a][1], S[a][2], S[a][3]);
    p[1] = make_float4(S[a][4], S[a][5], S[a][6], S[a][7]);
  }
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads, 1)
    kda_bwd_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                   const Tin* __restrict__ theta, const Tin* __restrict__ beta, float g_min, int gate,
                   const float* __restrict__ init_state, const float* __restrict__ d_out,
                   const float* __restrict__ d_final, float* __restrict__ dq,
                   float* __restrict__ dk, float* __restrict__ dv, float* __restrict__ dtheta,
                   float* __restrict__ dbeta, float* __restrict__ d_init, float* __restrict__ ws,
                   int H, int T) {
  __shared__ BwdShared sh;
  const int tid = threadIdx.x, r = tid / NT, c = tid % NT;
  const int64_t chain = blockIdx.x;  // sequence * H + head
  const int64_t b = chain / H, h = chain - b * H;
  const int nblk = (T + kBlock - 1) / kBlock;
  float* ckpt = ws + (size_t)chain * (size_t)(nblk + kBlock) * kState;  // nblk states
  float* blk = ckpt + (size_t)nblk * kState;                            // kBlock states
  auto row_of = [&](int t) { return (b * T + t) * H + h; };

  // ---- forward pass: the state at the start of every block
  float S[TT][TT];
  if (init_state)
    load_tile(S, init_state + chain * kState, r, c);
  else
#pragma unroll
    for (int a = 0; a < TT; ++a)
#pragma unroll
      for (int bb = 0; bb < TT; ++bb) S[a][bb] = 0.0f;
  for (int t = 0; t < T; ++t) {
    if (t % kBlock == 0) store_tile(S, ckpt + (size_t)(t / kBlock) * kState, r, c);
    __syncthreads();
    load_token(sh, q, k, v, theta, beta, d_out, row_of(t), g_min, gate, tid);
    __syncthreads();
    fwd_step(sh, S, r, c, tid);
  }

  // ---- reverse pass
  float L[TT][TT];
  if (d_final)
    load_tile(L, d_final + chain * kState, r, c);
  else
#pragma unroll
    for (int a = 0; a < TT; ++a)
#pragma unroll
      for (int bb = 0; bb < TT; ++bb) L[a][bb] = 0.0f;
  for (int blkI = nblk - 1; blkI >= 0; --blkI) {
    const int t0 = blkI * kBlock, t1 = min(T, t0 + kBlock);
    // the states before each token of the block
    __syncthreads();
    load_tile(S, ckpt + (size_t)blkI * kState, r, c);
    for (int t = t0; t < t1; ++t) {
      store_tile(S, blk + (size_t)(t - t0) * kState, r, c);
      __syncthreads();
      load_token(sh, q, k, v, theta, beta, d_out, row_of(t), g_min, gate, tid);
      __syncthreads();
      fwd_step(sh, S, r, c, tid);
    }
    __syncthreads();
    for (int t = t1 - 1; t >= t0; --t) {
      load_token(sh, q, k, v, theta, beta, d_out, row_of(t), g_min, gate, tid);
      __syncthreads();
      float X[TT][TT];
      load_tile(X, blk + (size_t)(t - t0) * kState, r, c);
#pragma unroll
      for (int a = 0; a < TT; ++a)
#pragma unroll
        for (int bb = 0; bb < TT; ++bb) X[a][bb] *= sh.e[TT * r + a];
      // column sums: k^T X and (with L += q do^T first) k^T L
#pragma unroll
      for (int a = 0; a < TT; ++a)
#pragma unroll
        for (int bb = 0; bb < TT; ++bb)
          L[a][bb] = fmaf(sh.q[TT * r + a], sh.dout[TT * c + bb], L[a][bb]);
#pragma unroll
      for (int bb = 0; bb < TT; ++bb) {
        float px = 0.0f, pl = 0.0f;
#pragma unroll
        for (int a = 0; a < TT; ++a) {
          px = fmaf(sh.k[TT * r + a], X[a][bb], px);
          pl = fmaf(sh.k[TT * r + a], L[a][bb], pl);
        }
        sh.colp[r][TT * c + bb] = px;
        sh.rowp[r][TT * c + bb] = pl;  // (a second column-sum buffer)
      }
      __syncthreads();
      if (tid < D) {
        float sx = 0.0f, sl = 0.0f;
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          sx += sh.colp[i][tid];
          sl += sh.rowp[i][tid];
        }
        const float w = sh.v[tid] - sx;        // v - X^T k
        sh.vec[0][tid] = sh.beta * w;          // u
        sh.vec[1][tid] = sl;                   // kL = L^T k
        sh.vec[2][tid] = sl * w;               // terms of dbeta
        dv[row_of(t) * D + tid] = sh.beta * sl;
      }
      __syncthreads();
      // row sums: dq = S_t do = X do + k (u . do); dk = L u - beta X kL;
      // dg = sum_j dX_ij X_ij with dX = L - beta k kL^T
#pragma unroll
      for (int a = 0; a < TT; ++a) {
        float pq = 0.0f, pk = 0.0f, pg = 0.0f;
        const float ki = sh.k[TT * r + a];
#pragma unroll
        for (int bb = 0; bb < TT; ++bb) {
          const int j = TT * c + bb;
          const float u = sh.vec[0][j], kl = sh.vec[1][j], dO = sh.dout[j];
          const float st = fmaf(ki, u, X[a][bb]);  // S_t
          pq = fmaf(st, dO, pq);
          pk = fmaf(L[a][bb], u, pk);
          pk = fmaf(-sh.beta * X[a][bb], kl, pk);
          const float dX = fmaf(-sh.beta * ki, kl, L[a][bb]);
          pg = fmaf(dX, X[a][bb], pg);
          L[a][bb] = sh.e[TT * r + a] * dX;  // gradient w.r.t. S_{t-1}
        }
        sh.colp[c][TT * r + a] = pq;  // row partials, indexed [tile column][row]
        sh.rowp[c][TT * r + a] = pk;
        X[a][0] = pg;                 // the dg partial of row a (X[a][.] is done)
      }
      __syncthreads();
      if (tid < D) {
        float sq = 0.0f, sk = 0.0f;
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          sq += sh.colp[i][tid];
          sk += sh.rowp[i][tid];
        }
        const int64_t o = row_of(t) * D + tid;
        dq[o] = sq;
        dk[o] = sk;
      }
      __syncthreads();
#pragma unroll
      for (int a = 0; a < TT; ++a) sh.colp[c][TT * r + a] = X[a][0];
      __syncthreads();
      if (tid < D) {
        float sg = 0.0f;
#pragma unroll
        for (int i = 0; i < NT; ++i) sg += sh.colp[i][tid];
        dtheta[row_of(t) * D + tid] = sg * sh.dgate[tid];
      }
      if (tid >= D && tid < D + 32) {
        // dbeta = sum_j kL_j (v_j - X^T k)_j: one warp
        const int l = tid - D;
        float s = 0.0f;
        for (int j = l; j < D; j += 32) s += sh.vec[2][j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (l == 0) dbeta[row_of(t)] = s;
      }
      __syncthreads();
    }
  }
  if (d_init) store_tile(L, d_init + chain * kState, r, c);
}

}  // namespace

size_t bwd_workspace_size(int B, int H, int T) {
  const int nblk = (T + kBlock - 1) / kBlock;
  return (size_t)B * H * (size_t)(nblk + kBlock) * kState * sizeof(float);
}

// (dk = dv = 128 is checked by the caller)
int launch_bwd(const BwdParams& p, cudaStream_t stream) {
  const unsigned grid = (unsigned)((int64_t)p.B * p.H);
  if (grid == 0 || p.T == 0) return KDA_OK;
  if (p.dtype == KDA_DTYPE_F32) {
    kda_bwd_kernel<float><<<grid, kThreads, 0, stream>>>(
        (const float*)p.q, (const float*)p.k, (const float*)p.v, (const float*)p.theta,
        (const float*)p.beta, p.g_min, p.gate, p.init_state, p.d_out, p.d_final, p.dq, p.dk, p.dv,
        p.dtheta, p.dbeta, p.d_init, (float*)p.workspace, p.H, p.T);
  } else {
    kda_bwd_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
        (const __nv_bfloat16*)p.q, (const __nv_bfloat16*)p.k, (const __nv_bfloat16*)p.v,
        (const __nv_bfloat16*)p.theta, (const __nv_bfloat16*)p.beta, p.g_min, p.gate, p.init_state,
        p.d_out, p.d_final, p.dq, p.dk, p.dv, p.dtheta, p.dbeta, p.d_init, (float*)p.workspace, p.H,
        p.T);
  }
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // namespace kda
