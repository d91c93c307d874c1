// Internal declarations shared by the translation units of libkda.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Chunk length of the chunk-parallel form ("Kimi K3 Deep Dive", section "The
// Problem": a 16-token chunk matches the tensor-core GEMM granularity).
constexpr int kChunk = 16;

// Validated launch parameters shared by the kernel paths.
struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* theta;
  const void* beta;
  float g_min;
  const float* init_state;
  void* out;
  float* final_state;
  const int32_t* cu_seqlens;  // device, or nullptr for fixed length
  int N;                      // sequences (B for fixed length)
  int H, T, dk, dv;
  int dtype;                  // KDA_DTYPE_* of q, k, v, theta, beta
  int out_dtype;              // KDA_DTYPE_* of out
  int gate;                   // KDA_GATE_*
};

// Validated parameters of one decode step (one token per sequence and head).
struct DecodeParams {
  const void* q;      // [N, H, dk]
  const void* k;      // [N, H, dk]
  const void* v;      // [N, H, dv]
  const void* theta;  // [N, H, dk]
  const void* beta;   // [N, H]
  float g_min;
  float* state;       // [N, H, dk, dv] fp32, read and overwritten
  float* out;         // [N, H, dv] fp32
  int N, H, dk, dv;
  int dtype;          // KDA_DTYPE_* of q, k, v, theta, beta
};

int launch_decode(const DecodeParams& p, cudaStream_t stream);

// Validated parameters of the backward pass (fixed-length batches, dk = dv = 128).
struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* theta;
  const void* beta;
  float g_min;
  int gate;
  const float* init_state;  // [B, H, dk, dv] or null
  const float* d_out;       // [B, T, H, dv]
  const float* d_final;     // [B, H, dk, dv] or null
  float* dq;                // [B, T, H, dk]
  float* dk;
  float* dv;                // [B, T, H, dv]
  float* dtheta;            // [B, T, H, dk]
  float* dbeta;             // [B, T, H]
  float* d_init;            // [B, H, dk, dv] or null
  void* workspace;
  int B, H, T;
  int dtype;
};
size_t bwd_workspace_size(int B, int H, int T);
int launch_bwd(const BwdParams& p, cudaStream_t stream);

// Device status word of the current device (bounded waits write it).
int* status_word_device_ptr();

int launch_simt(const FwdParams& p, cudaStream_t stream);
// tc_gram: the intra-chunk products A and P as tcgen05.mma into tensor memory
// (otherwise warp-level mma.sync); everything else is the same kernel.
int launch_mma(const FwdParams& p, cudaStream_t stream, bool tc_gram = false);

// One CTA of a segmented launch of the register-resident kernel: a token range
// of one head, with its own initial/final state and options.
constexpr int kJobZeroV = 1;          // V is taken as zero (the state's linear part)
constexpr int kJobNoOut = 2;          // no output stores
constexpr int kJobIdentityInit = 4;   // initial state = identity (dk = dv), init ignored
constexpr int kJobTestWithholdFirst = 8;  // test only: the first chunk's hand-off is never made
struct SegJob {
  int64_t t0, t1;          // token rows [t0, t1) of the packed [tokens, H, .] tensors
  int head;
  int flags;               // kJob* bits
  const float* init;       // [dk][dv] initial state, or null (zero / identity)
  float* final_state;      // [dk][dv] end state, or null
};
// Launches one CTA per job over the packed token axis (p.T = total tokens);
// wait_ns = 0 keeps the default limit of the bounded waits.
int launch_mma_jobs(const FwdParams& p, const SegJob* jobs, int njobs, cudaStream_t stream,
                    uint64_t wait_ns = 0, bool tc_gram = false);

// tcgen05/TMEM path with 32-token state steps (kda_tc32.cu): one CTA per job
// (jobs != null) or per (sequence, head) chain.  `split_s` keeps the state's
// bf16 copy as a high/low pair in the read-out products; `dbg` (test hook,
// may be null) receives the stage dump of the first CTA for its first
// `dbg_nsc` 32-token super-chunks (kTc32DumpFloats floats each).
bool tc32_supported(int dtype, int dk, int dv);
int launch_tc32_jobs(const FwdParams& p, const SegJob* jobs, int njobs, cudaStream_t stream,
                     uint64_t wait_ns, bool split_s, float* dbg = nullptr, int dbg_nsc = 0);
constexpr int kTc32DumpFloats = 3072 + 8192 + 128 + 32;

// Segment-parallel forward (fixed-length batches, bf16, dk = dv = 128): the
// scratch it needs and the launch sequence over a caller-provided workspace.
size_t segmented_workspace_size(int B, int H, int T, int segments);

// The library's own scratch area for kda_chunk_fwd_segmented_noalloc (one per
// device, part of the library image); null if its address cannot be found.
constexpr size_t kNoallocScratchBytes = (size_t)KDA_NOALLOC_SCRATCH_BYTES;
void* noalloc_scratch();
// kernel: KDA_PATH_MMA (register-resident), KDA_PATH_TC or KDA_PATH_TC_SPLIT.
int launch_segmented(const FwdParams& p, int segments, void* ws, size_t ws_bytes,
                     cudaStream_t stream, int kernel);
bool mma_supported(int dtype, int dk, int dv);

// TMA map over a [tokens][H][128] bf16 tensor whose boxes are `box_rows`
// tokens (16: one chunk; 32: two) x 128 channels of one head (unswizzled,
// out-of-range rows read 0).  False if the driver's encoder is unavailable or
// rejects the arguments.
bool encode_token_rows(CUtensorMap* m, const void* base, int H, int64_t tokens,
                       int box_rows = kChunk);

// Rank-ordered chain lookup for packed variable-length batches: blockIdx.x = r * H + h
// runs the r-th longest sequence first (longest-processing-time order).  For
// fixed-length batches the order is the natural one.  Small enough to inline
// in each kernel; all threads of the block must call it.
constexpr int kMaxRankedSeqs = 4096;

}  // namespace kda
