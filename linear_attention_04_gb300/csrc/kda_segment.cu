// kda_segment.cu -- segment-parallel forward pass for batches of few, long
// sequences (more SMs than (sequence, head) chains).
//
// The recurrence S_t = (I - b_t k_t k_t^T) Diag(e^{g_t}) S_{t-1} + b_t k_t v_t^T
// ("Kimi K3 Deep Dive", section "Core Innovation 1") is affine in the state, so
// over any token segment s
//
//     S_end = Phi_s S_start + S_loc_s,
//
// where S_loc_s is the end state of the segment run from a zero state and
// Phi_s (dk x dk) the end state of the segment run with v = 0 from the
// identity (column independence makes the identity's columns the basis of the
// linear part).  Each chain is cut into P segments of whole 16-token chunks:
//
//   launch 1 (one CTA per job): segment 0 in full from the caller's initial
//            state (outputs, end state = start of segment 1); segments
//            1 .. P-2 from zero without outputs (S_loc); the same segments
//            with v = 0 from the identity without outputs (Phi);
//   combine: S_start(s + 1) = Phi_s S_start(s) + S_loc_s, s = 1 .. P-2 (fp32);
//   launch 2: segments 1 .. P-1 in full from their start states (outputs; the
//            last one writes the caller's final state).
//
// Work per chain grows by about (2P - 3) / P segment-lengths, run in parallel
// on otherwise idle SMs.  All scratch lives in a caller-provided workspace
// (kda_segmented_workspace_size).  Segments are whole 32-token units, the
// state step of the tcgen05 kernel (two 16-token chunks).
//
// Segment 0 may be longer than the others.  Launch 1 holds segment 0 of every
// chain and two jobs for each of segments 1 .. P-2, launch 2 one job for each
// of segments 1 .. P-1, and each launch takes as long as its busiest SM: with
// more jobs than SMs, the jobs after the first wave wait for SMs to free up.
// A segment 0 of twice the others' length runs beside the first wave of the
// short jobs of launch 1 and lets the rest of them follow on the same SMs:
// e.g. 32 chains, P = 5, 152 SMs: equal segments take 2 + 1 waves of L/5
// (0.6 L), a first segment of 2 L/6 takes 2 L/6 + L/6 (0.5 L).  The plan
// picks whichever of the two splits a list-scheduling model of the launches
// (jobs in launch order on the device's SMs) finishes first.
#include <cuda_runtime.h>
#include <stdint.h>

#include <functional>
#include <queue>
#include <vector>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int D = 128;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct SegPlan {
  int P;           // segments per chain (effective)
  int64_t L0tok;   // tokens of segment 0
  int64_t Ltok;    // tokens of segments 1 .. P-1 (whole units; the last may be shorter)
  int64_t NH;      // chains
  size_t off_jobs1, off_jobs2, off_sst, off_sloc, off_phi, total;
};

constexpr int kSegUnit = 2 * kChunk;  // tokens per segmentation unit

// Time (in units) until `sms` SMs have run jobs of the given lengths, each job
// starting on the first SM to become free, in order.
int64_t list_schedule(const std::vector<int64_t>& jobs, int sms) {
  std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> free_at;
  for (int i = 0; i < sms; ++i) free_at.push(0);
  int64_t end = 0;
  for (int64_t len : jobs) {
    const int64_t t = free_at.top() + len;
    free_at.pop();
    free_at.push(t);
    if (t > end) end = t;
  }
  return end;
}

// Model of the two launches for segment 0 of u0 units and the others of u
// units (the last one what is left of n units).
int64_t model_time(int64_t NH, int P, int64_t n, int64_t u0, int64_t u, int sms) {
  std::vector<int64_t> j1, j2;
  j1.assign((size_t)NH, u0);
  j1.insert(j1.end(), (size_t)(NH * 2 * (P - 2)), u);
  for (int s = 1; s <= P - 1; ++s) {
    const int64_t len = s < P - 1 ? u : n - u0 - (int64_t)(P - 2) * u;
    j2.insert(j2.end(), (size_t)NH, len);
  }
  return list_schedule(j1, sms) + list_schedule(j2, sms);
}

// sms > 0: choose segment 0's length by the model above (else equal segments).
SegPlan plan(int B, int H, int T, int segments, int sms = 0) {
  SegPlan s;
  const int64_t nchunks = ((int64_t)T + kSegUnit - 1) / kSegUnit;
  int P = segments < 1 ? 1 : segments;
  if (P > nchunks) P = (int)(nchunks > 0 ? nchunks : 1);
  const int64_t per = (nchunks + P - 1) / P;  // chunks per segment
  P = (int)((nchunks + per - 1) / per);       // no empty segment
  s.P = P;
  s.L0tok = per * kSegUnit;
  s.Ltok = per * kSegUnit;
  s.NH = (int64_t)B * H;
  if (sms > 0 && P >= 3 && s.NH * 3 * P <= 200000) {
    // segment 0 twice as long as the others, if the last segment keeps some
    // tokens and the model says it finishes first
    const int64_t u = (nchunks + P) / (P + 1);
    if (2 * u + (int64_t)(P - 2) * u < nchunks &&
        model_time(s.NH, P, nchunks, 2 * u, u, sms) < model_time(s.NH, P, nchunks, per, per, sms)) {
      s.L0tok = 2 * u * kSegUnit;
      s.Ltok = u * kSegUnit;
    }
  }
  const int64_t n1 = s.NH * (P >= 2 ? 2 * P - 3 : 0);
  const int64_t n2 = s.NH * (P - 1);
  const size_t st = (size_t)D * D * sizeof(float);
  s.off_jobs1 = 0;
  s.off_jobs2 = align_up(s.off_jobs1 + (size_t)n1 * sizeof(SegJob));
  s.off_sst = align_up(s.off_jobs2 + (size_t)n2 * sizeof(SegJob));
  s.off_sloc = align_up(s.off_sst + (size_t)(s.NH * (P - 1)) * st);
  s.off_phi = align_up(s.off_sloc + (size_t)(s.NH * (P > 2 ? P - 2 : 0)) * st);
  s.total = align_up(s.off_phi + (size_t)(s.NH * (P > 2 ? P - 2 : 0)) * st);
  return s;
}

// Fills both job tables (one thread per chain).
__global__ void seg_setup_kernel(SegJob* jobs1, SegJob* jobs2, float* sst, float* sloc, float* phi,
                                 const float* init, float* fin, int64_t NH, int H, int64_t T,
                                 int P, int64_t L0tok, int64_t Ltok) {
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= NH) return;
  const int64_t b = c / H;
  const int h = (int)(c - b * H);
  const int64_t base = b * T;
  const size_t st = (size_t)D * D;
  // segment s: tokens [start(s), start(s + 1)), start(s) = L0tok + (s - 1) Ltok
  auto seg = [&](int s, SegJob& j) {
    const int64_t a = s == 0 ? 0 : L0tok + (int64_t)(s - 1) * Ltok;
    const int64_t e = L0tok + (int64_t)s * Ltok;
    j.t0 = base + a;
    j.t1 = base + (e < T ? e : T);
    j.head = h;
  };
  // launch 1: segment 0 in full; segments 1 .. P-2 local and transition
  SegJob j;
  seg(0, j);
  j.flags = 0;
  j.init = init ? init + c * st : nullptr;
  j.final_state = sst + (size_t)(c * (P - 1)) * st;
  jobs1[c] = j;
  for (int s = 1; s <= P - 2; ++s) {
    seg(s, j);
    j.flags = kJobNoOut;
    j.init = nullptr;
    j.final_state = sloc + (size_t)(c * (P - 2) + (s - 1)) * st;
    jobs1[NH * s + c] = j;
    j.flags = kJobZeroV | kJobNoOut | kJobIdentityInit;
    j.final_state = phi + (size_t)(c * (P - 2) + (s - 1)) * st;
    jobs1[NH * (P - 1 + s - 1) + c] = j;
  }
  // launch 2: segments 1 .. P-1 in full from their start states
  for (int s = 1; s <= P - 1; ++s) {
    seg(s, j);
    j.flags = 0;
    j.init = sst + (size_t)(c * (P - 1) + (s - 1)) * st;
    j.final_state = (s == P - 1 && fin) ? fin + c * st : nullptr;
    jobs2[NH * (s - 1) + c] = j;
  }
}

// S_start(s + 1) = Phi_s S_start(s) + S_loc_s for every chain, in fp32: block
// (chain, 16-row tile), thread = value column.
__global__ void __launch_bounds__(D) seg_combine_kernel(float* sst, const float* sloc, const float* phi,
                                                         int P, int s) {
  const int64_t c = blockIdx.x;
  const int i0 = blockIdx.y * 16, j = threadIdx.x;
  const size_t st = (size_t)D * D;
  const float* prev = sst + (size_t)(c * (P - 1) + (s - 1)) * st;
  const float* ph = phi + (size_t)(c * (P - 2) + (s - 1)) * st;
  const float* lo = sloc + (size_t)(c * (P - 2) + (s - 1)) * st;
  float* nxt = sst + (size_t)(c * (P - 1) + s) * st;
  float acc[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) acc[r] = lo[(size_t)(i0 + r) * D + j];
  for (int kk = 0; kk < D; ++kk) {
    const float p = prev[(size_t)kk * D + j];
#pragma unroll
    for (int r = 0; r < 16; ++r) acc[r] = fmaf(ph[(size_t)(i0 + r) * D + kk], p, acc[r]);
  }
#pragma unroll
  for (int r = 0; r < 16; ++r) nxt[(size_t)(i0 + r) * D + j] = acc[r];
}

}  // namespace

size_t segmented_workspace_size(int B, int H, int T, int segments) {
  return plan(B, H, T, segments).total;
}

int launch_segmented(const FwdParams& p, int segments, void* ws, size_t ws_bytes,
                     cudaStream_t stream, int kernel) {
  if ((int64_t)p.N * p.T > (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
  const bool mma = kernel == KDA_PATH_MMA;
  const bool split_s = kernel == KDA_PATH_TC_SPLIT;
  auto run_jobs = [&](const FwdParams& q, const SegJob* jobs, int njobs) {
    return mma ? launch_mma_jobs(q, jobs, njobs, stream)
               : launch_tc32_jobs(q, jobs, njobs, stream, 0, split_s);
  };
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KDA_ERR_CUDA;
  const SegPlan pl = plan(p.N, p.H, p.T, segments, sms);
  if (pl.P < 2) return mma ? launch_mma(p, stream) : launch_tc32_jobs(p, nullptr, 0, stream, 0, split_s);
  if (!ws || ws_bytes < pl.total) return KDA_ERR_INVALID_ARG;
  unsigned char* w = (unsigned char*)ws;
  SegJob* jobs1 = (SegJob*)(w + pl.off_jobs1);
  SegJob* jobs2 = (SegJob*)(w + pl.off_jobs2);
  float* sst = (float*)(w + pl.off_sst);
  float* sloc = (float*)(w + pl.off_sloc);
  float* phi = (float*)(w + pl.off_phi);
  seg_setup_kernel<<<(unsigned)((pl.NH + 127) / 128), 128, 0, stream>>>(
      jobs1, jobs2, sst, sloc, phi, p.init_state, p.final_state, pl.NH, p.H, p.T, pl.P, pl.L0tok,
      pl.Ltok);
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_LAUNCH;
  // the kernels see the batch as one packed sequence of B * T tokens
  FwdParams q = p;
  q.T = (int)((int64_t)p.N * p.T);
  q.N = 1;
  q.cu_seqlens = nullptr;
  int rc = run_jobs(q, jobs1, (int)(pl.NH * (2 * pl.P - 3)));
  if (rc != KDA_OK) return rc;
  for (int s = 1; s <= pl.P - 2; ++s) {
    seg_combine_kernel<<<dim3((unsigned)pl.NH, D / 16), D, 0, stream>>>(sst, sloc, phi, pl.P, s);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_LAUNCH;
  }
  return run_jobs(q, jobs2, (int)(pl.NH * (pl.P - 1)));
}

}  // namespace kda

// Test hook: the segment plan of a call on a device with `sms` SMs (0: equal
// segments), as out[0] = segments, out[1] = tokens of segment 0, out[2] =
// tokens of each later segment (the last may be shorter).
extern "C" KDA_API int kda_debug_segment_plan(int B, int H, int T, int segments, int sms,
                                              int64_t* out) {
  if (!out || B <= 0 || H <= 0 || T < 0 || sms < 0) return KDA_ERR_INVALID_ARG;
  const kda::SegPlan pl = kda::plan(B, H, T, segments, sms);
  out[0] = pl.P;
  out[1] = pl.L0tok;
  out[2] = pl.Ltok;
  return KDA_OK;
}
