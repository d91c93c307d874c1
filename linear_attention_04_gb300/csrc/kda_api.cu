// kda_api.cu -- the C ABI of libkda.so: argument checks, path choice, launch.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kda.h"
#include "kda_internal.cuh"

namespace kda {

// Per-device status word: kernels that give up on a bounded wait store
// KDA_ERR_DEVICE_TIMEOUT here.  Static device memory, one word per device.
__device__ int g_status_word = 0;

int* status_word_device_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

namespace {

constexpr int kMaxDevices = 64;
std::once_flag g_dev_once[kMaxDevices];
int g_dev_ok[kMaxDevices];  // 1 = compute capability 10.3, 0 = other, -1 = query failed

int check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return KDA_ERR_CUDA;
  if (dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED_DEVICE;
  std::call_once(g_dev_once[dev], [dev]() {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      g_dev_ok[dev] = -1;
      return;
    }
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : 0;
  });
  if (g_dev_ok[dev] < 0) return KDA_ERR_CUDA;
  return g_dev_ok[dev] ? KDA_OK : KDA_ERR_UNSUPPORTED_DEVICE;
}

bool shape_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate(const kda_fwd_args* a) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (a->B <= 0 || a->H <= 0 || a->T < 0) return KDA_ERR_INVALID_ARG;
  // token tensors may be empty (null) only when there are no tokens
  if (a->T > 0 && (!a->q || !a->k || !a->v || !a->theta || !a->beta || !a->out))
    return KDA_ERR_INVALID_ARG;
  if (a->gate != KDA_GATE_SIGMOID && a->gate != KDA_GATE_LOG_DECAY) return KDA_ERR_INVALID_ARG;
  if (a->gate == KDA_GATE_SIGMOID && (!(a->g_min < 0.0f) || a->g_min != a->g_min))
    return KDA_ERR_INVALID_ARG;
  if (a->dtype != KDA_DTYPE_BF16 && a->dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
  if (a->out_dtype != KDA_DTYPE_BF16 && a->out_dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
  if (a->dtype == KDA_DTYPE_F32 && a->out_dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
  if (a->path != KDA_PATH_AUTO && a->path != KDA_PATH_SIMT && a->path != KDA_PATH_TC &&
      a->path != KDA_PATH_MMA && a->path != KDA_PATH_TC_SPLIT && a->path != KDA_PATH_MMA_TC)
    return KDA_ERR_INVALID_ARG;
  if (!shape_ok(a->dk) || !shape_ok(a->dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
  // sizes must fit the 32-bit grid and 64-bit offsets used by the kernels
  const int64_t chains = (int64_t)a->B * a->H;
  if (chains > (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (!a->cu_seqlens && (int64_t)a->B * a->T > ((int64_t)1 << 40)) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {a->q, a->k, a->v, a->theta, a->beta, a->out, a->init_state,
                        a->final_state, a->cu_seqlens};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
  return KDA_OK;
}

}  // namespace
}  // namespace kda

extern "C" {

KDA_API int kda_select_path(int dtype, int dk, int dv) {
  if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
  if (!kda::shape_ok(dk) || !kda::shape_ok(dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
  return kda::mma_supported(dtype, dk, dv) ? KDA_PATH_MMA : KDA_PATH_SIMT;
}

KDA_API size_t kda_chunk_fwd_workspace_size(int, int, int, int, int) { return 0; }

KDA_API int kda_chunk_fwd_ex(const kda_fwd_args* a, cudaStream_t stream) {
  int rc = kda::validate(a);
  if (rc != KDA_OK) return rc;
  int path = a->path;
  if (path == KDA_PATH_AUTO) path = kda_select_path(a->dtype, a->dk, a->dv);
  if ((path == KDA_PATH_TC || path == KDA_PATH_TC_SPLIT) && !kda::tc32_supported(a->dtype, a->dk, a->dv))
    return KDA_ERR_UNSUPPORTED_SHAPE;
  if ((path == KDA_PATH_MMA || path == KDA_PATH_MMA_TC) && !kda::mma_supported(a->dtype, a->dk, a->dv))
    return KDA_ERR_UNSUPPORTED_SHAPE;
  rc = kda::check_device();
  if (rc != KDA_OK) return rc;
  const bool empty = a->T == 0;
  kda::FwdParams p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.theta = a->theta;
  p.beta = a->beta;
  p.g_min = a->g_min;
  p.init_state = a->init_state;
  p.out = a->out;
  p.final_state = a->final_state;
  p.cu_seqlens = a->cu_seqlens;
  p.N = a->B;
  p.H = a->H;
  p.T = a->T;
  p.dk = a->dk;
  p.dv = a->dv;
  p.dtype = a->dtype;
  p.out_dtype = a->out_dtype;
  p.gate = a->gate;
  if (empty && !a->cu_seqlens) {
    // no tokens: the final state is the initial state
    if (a->final_state) {
      size_t bytes = (size_t)a->B * a->H * a->dk * a->dv * sizeof(float);
      cudaError_t e = a->init_state
                          ? cudaMemcpyAsync(a->final_state, a->init_state, bytes,
                                            cudaMemcpyDeviceToDevice, stream)
                          : cudaMemsetAsync(a->final_state, 0, bytes, stream);
      if (e != cudaSuccess) return KDA_ERR_CUDA;
    }
    return KDA_OK;
  }
  if (path == KDA_PATH_TC || path == KDA_PATH_TC_SPLIT)
    return kda::launch_tc32_jobs(p, nullptr, 0, stream, 0, path == KDA_PATH_TC_SPLIT);
  if (path == KDA_PATH_MMA || path == KDA_PATH_MMA_TC)
    return kda::launch_mma(p, stream, path == KDA_PATH_MMA_TC);
  return kda::launch_simt(p, stream);
}

KDA_API int kda_chunk_fwd(const void* q, const void* k, const void* v, const void* theta,
                          const void* beta, float g_min, const float* init_state, float* out,
                          float* final_state, const int32_t* cu_seqlens, int B, int H, int T,
                          int dk, int dv, cudaStream_t stream) {
  kda_fwd_args a{q, k, v, theta, beta, g_min, init_state, out, final_state, cu_seqlens,
                 B, H, T, dk, dv, KDA_DTYPE_BF16, KDA_DTYPE_F32, KDA_PATH_AUTO, KDA_GATE_SIGMOID};
  return kda_chunk_fwd_ex(&a, stream);
}

KDA_API int kda_chunk_fwd_f32(const float* q, const float* k, const float* v, const float* theta,
                              const float* beta, float g_min, const float* init_state, float* out,
                              float* final_state, const int32_t* cu_seqlens, int B, int H, int T,
                              int dk, int dv, cudaStream_t stream) {
  kda_fwd_args a{q, k, v, theta, beta, g_min, init_state, out, final_state, cu_seqlens,
                 B, H, T, dk, dv, KDA_DTYPE_F32, KDA_DTYPE_F32, KDA_PATH_SIMT, KDA_GATE_SIGMOID};
  return kda_chunk_fwd_ex(&a, stream);
}

KDA_API size_t kda_segmented_workspace_size(int B, int H, int T, int dk, int dv, int segments) {
  if (B <= 0 || H <= 0 || T < 0 || dk != 128 || dv != 128 || segments < 1) return 0;
  return kda::segmented_workspace_size(B, H, T, segments);
}

KDA_API int kda_chunk_fwd_segmented(const kda_fwd_args* a, int segments, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  int rc = kda::validate(a);
  if (rc != KDA_OK) return rc;
  if (a->dtype != KDA_DTYPE_BF16 || a->dk != 128 || a->dv != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
  if (a->cu_seqlens || segments < 1) return KDA_ERR_INVALID_ARG;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return KDA_ERR_MISALIGNED;
  if (segments > 1 && a->T > 0 &&
      (!workspace || workspace_bytes < kda::segmented_workspace_size(a->B, a->H, a->T, segments)))
    return KDA_ERR_INVALID_ARG;
  if ((int64_t)a->B * a->T > (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
  // the kernel: the register-resident one for KDA_PATH_MMA, else tcgen05
  const int kernel = (a->path == KDA_PATH_MMA || a->path == KDA_PATH_TC_SPLIT) ? a->path : KDA_PATH_TC;
  if (a->T == 0) {
    kda_fwd_args b = *a;
    b.path = kernel;
    return kda_chunk_fwd_ex(&b, stream);
  }
  rc = kda::check_device();
  if (rc != KDA_OK) return rc;
  kda::FwdParams p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.theta = a->theta;
  p.beta = a->beta;
  p.g_min = a->g_min;
  p.init_state = a->init_state;
  p.out = a->out;
  p.final_state = a->final_state;
  p.cu_seqlens = nullptr;
  p.N = a->B;
  p.H = a->H;
  p.T = a->T;
  p.dk = a->dk;
  p.dv = a->dv;
  p.dtype = a->dtype;
  p.out_dtype = a->out_dtype;
  p.gate = a->gate;
  return kda::launch_segmented(p, segments, workspace, workspace_bytes, stream, kernel);
}

KDA_API int kda_chunk_fwd_segmented_noalloc(const kda_fwd_args* a, int segments,
                                            cudaStream_t stream) {
  int rc = kda::validate(a);
  if (rc != KDA_OK) return rc;
  if (a->dtype != KDA_DTYPE_BF16 || a->dk != 128 || a->dv != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
  if (a->cu_seqlens || segments < 1) return KDA_ERR_INVALID_ARG;
  if ((int64_t)a->B * a->T > (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
  const size_t need = a->T > 0 ? kda::segmented_workspace_size(a->B, a->H, a->T, segments) : 0;
  if (need > kda::kNoallocScratchBytes) return KDA_ERR_SCRATCH_TOO_SMALL;
  rc = kda::check_device();
  if (rc != KDA_OK) return rc;
  void* scratch = kda::noalloc_scratch();
  if (!scratch) return KDA_ERR_CUDA;
  return kda_chunk_fwd_segmented(a, segments, scratch, kda::kNoallocScratchBytes, stream);
}

KDA_API size_t kda_chunk_bwd_workspace_size(int B, int H, int T, int dk, int dv) {
  if (B <= 0 || H <= 0 || T < 0 || dk != 128 || dv != 128) return 0;
  return kda::bwd_workspace_size(B, H, T);
}

KDA_API int kda_chunk_bwd(const kda_bwd_args* a, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (a->B <= 0 || a->H <= 0 || a->T < 0) return KDA_ERR_INVALID_ARG;
  if (a->dtype != KDA_DTYPE_BF16 && a->dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
  if (a->gate != KDA_GATE_SIGMOID && a->gate != KDA_GATE_LOG_DECAY) return KDA_ERR_INVALID_ARG;
  if (a->gate == KDA_GATE_SIGMOID && (!(a->g_min < 0.0f) || a->g_min != a->g_min))
    return KDA_ERR_INVALID_ARG;
  if (a->dk_dim != 128 || a->dv_dim != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)a->B * a->H > (int64_t)INT32_MAX || (int64_t)a->B * a->T > ((int64_t)1 << 40))
    return KDA_ERR_INVALID_ARG;
  if (a->T > 0 && (!a->q || !a->k || !a->v || !a->theta || !a->beta || !a->d_out || !a->dq ||
                   !a->dk || !a->dv || !a->dtheta || !a->dbeta))
    return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {a->q, a->k, a->v, a->theta, a->beta, a->init_state, a->d_out, a->d_final,
                        a->dq, a->dk, a->dv, a->dtheta, a->dbeta, a->d_init, workspace};
  for (const void* p : ptrs)
    if (p && !kda::aligned16(p)) return KDA_ERR_MISALIGNED;
  const size_t need = kda::bwd_workspace_size(a->B, a->H, a->T);
  if (a->T > 0 && (!workspace || workspace_bytes < need)) return KDA_ERR_INVALID_ARG;
  const int rc = kda::check_device();
  if (rc != KDA_OK) return rc;
  if (a->T == 0) {
    // no tokens: the initial state's gradient is the final state's
    if (a->d_init) {
      const size_t bytes = (size_t)a->B * a->H * 128 * 128 * sizeof(float);
      const cudaError_t e = a->d_final ? cudaMemcpyAsync(a->d_init, a->d_final, bytes,
                                                         cudaMemcpyDeviceToDevice, stream)
                                       : cudaMemsetAsync(a->d_init, 0, bytes, stream);
      if (e != cudaSuccess) return KDA_ERR_CUDA;
    }
    return KDA_OK;
  }
  kda::BwdParams p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.theta = a->theta;
  p.beta = a->beta;
  p.g_min = a->g_min;
  p.gate = a->gate;
  p.init_state = a->init_state;
  p.d_out = a->d_out;
  p.d_final = a->d_final;
  p.dq = a->dq;
  p.dk = a->dk;
  p.dv = a->dv;
  p.dtheta = a->dtheta;
  p.dbeta = a->dbeta;
  p.d_init = a->d_init;
  p.workspace = workspace;
  p.B = a->B;
  p.H = a->H;
  p.T = a->T;
  p.dtype = a->dtype;
  return kda::launch_bwd(p, stream);
}

KDA_API int kda_selftest_withheld_handoff(const kda_fwd_args* a, long long wait_limit_ns,
                                          void* workspace, size_t workspace_bytes,
                                          cudaStream_t stream) {
  int rc = kda::validate(a);
  if (rc != KDA_OK) return rc;
  if (a->dtype != KDA_DTYPE_BF16 || a->dk != 128 || a->dv != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
  if (a->cu_seqlens || a->T < 16 || wait_limit_ns <= 0) return KDA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < sizeof(kda::SegJob)) return KDA_ERR_INVALID_ARG;
  if (!kda::aligned16(workspace)) return KDA_ERR_MISALIGNED;
  rc = kda::check_device();
  if (rc != KDA_OK) return rc;
  kda::SegJob job;
  job.t0 = 0;
  job.t1 = a->T;
  job.head = 0;
  job.flags = kda::kJobTestWithholdFirst;
  job.init = a->init_state;
  job.final_state = a->final_state;
  if (cudaMemcpyAsync(workspace, &job, sizeof(job), cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  kda::FwdParams p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.theta = a->theta;
  p.beta = a->beta;
  p.g_min = a->g_min;
  p.init_state = a->init_state;
  p.out = a->out;
  p.final_state = a->final_state;
  p.cu_seqlens = nullptr;
  p.N = 1;
  p.H = a->H;
  p.T = (int)((int64_t)a->B * a->T);
  p.dk = a->dk;
  p.dv = a->dv;
  p.dtype = a->dtype;
  p.out_dtype = a->out_dtype;
  p.gate = a->gate;
  // the job table lives in device memory the copy above fills, in stream order
  const kda::SegJob* jobs = (const kda::SegJob*)workspace;
  if (a->path == KDA_PATH_MMA || a->path == KDA_PATH_MMA_TC)
    return kda::launch_mma_jobs(p, jobs, 1, stream, (uint64_t)wait_limit_ns,
                                a->path == KDA_PATH_MMA_TC);
  return kda::launch_tc32_jobs(p, jobs, 1, stream, (uint64_t)wait_limit_ns, a->path == KDA_PATH_TC_SPLIT);
}

KDA_API int kda_debug_fwd_stages(const kda_fwd_args* a, float* dump, int nsc, cudaStream_t stream) {
  int rc = kda::validate(a);
  if (rc != KDA_OK) return rc;
  if (a->dtype != KDA_DTYPE_BF16 || a->dk != 128 || a->dv != 128) return KDA_ERR_UNSUPPORTED_SHAPE;
  if (a->T <= 0 || nsc < 1 || !dump) return KDA_ERR_INVALID_ARG;
  if (!kda::aligned16(dump)) return KDA_ERR_MISALIGNED;
  rc = kda::check_device();
  if (rc != KDA_OK) return rc;
  kda::FwdParams p;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.theta = a->theta;
  p.beta = a->beta;
  p.g_min = a->g_min;
  p.init_state = a->init_state;
  p.out = a->out;
  p.final_state = a->final_state;
  p.cu_seqlens = a->cu_seqlens;
  p.N = a->B;
  p.H = a->H;
  p.T = a->T;
  p.dk = a->dk;
  p.dv = a->dv;
  p.dtype = a->dtype;
  p.out_dtype = a->out_dtype;
  p.gate = a->gate;
  return kda::launch_tc32_jobs(p, nullptr, 0, stream, 0, a->path == KDA_PATH_TC_SPLIT, dump, nsc);
}

KDA_API int kda_debug_stage_floats(void) { return kda::kTc32DumpFloats; }

KDA_API int kda_decode_step(const void* q, const void* k, const void* v, const void* theta,
                            const void* beta, float g_min, float* state, float* out, int N, int H,
                            int dk, int dv, int dtype, cudaStream_t stream) {
  if (N < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
  if (!(g_min < 0.0f) || g_min != g_min) return KDA_ERR_INVALID_ARG;
  if (!kda::shape_ok(dk) || !kda::shape_ok(dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)N * H > (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (N > 0 && (!q || !k || !v || !theta || !beta || !state || !out)) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, theta, beta, state, out};
  for (const void* p : ptrs)
    if (p && !kda::aligned16(p)) return KDA_ERR_MISALIGNED;
  if (N == 0) return KDA_OK;
  const int rc = kda::check_device();
  if (rc != KDA_OK) return rc;
  kda::DecodeParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.theta = theta;
  p.beta = beta;
  p.g_min = g_min;
  p.state = state;
  p.out = out;
  p.N = N;
  p.H = H;
  p.dk = dk;
  p.dv = dv;
  p.dtype = dtype;
  return kda::launch_decode(p, stream);
}

KDA_API int kda_device_status(int clear) {
  int* p = kda::status_word_device_ptr();
  if (!p) return KDA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
  if (clear) {
    int z = 0;
    if (cudaMemcpy(p, &z, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return KDA_ERR_CUDA;
  }
  return v;
}

KDA_API const char* kda_strerror(int code) {
  switch (code) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case KDA_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3";
    case KDA_ERR_LAUNCH: return "kernel launch failed";
    case KDA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case KDA_ERR_CUDA: return "CUDA runtime error";
    case KDA_ERR_UNSUPPORTED_SHAPE: return "unsupported (dtype, dk, dv) for this kernel path";
    case KDA_ERR_SCRATCH_TOO_SMALL: return "the library's scratch area cannot hold this call";
    case KDA_ERR_BAD_SEQLENS: return "cu_seqlens is not a valid packing of the tokens";
    default: return "unknown status code";
  }
}

KDA_API int kda_version(void) { return 200; }

}  // extern "C"
