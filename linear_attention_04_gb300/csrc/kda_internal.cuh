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

// Device status word of the current device (bounded waits write it).
int* status_word_device_ptr();

int launch_simt(const FwdParams& p, cudaStream_t stream);
int launch_tc(const FwdParams& p, cudaStream_t stream);
bool tc_supported(int dtype, int dk, int dv);
int launch_mma(const FwdParams& p, cudaStream_t stream);
bool mma_supported(int dtype, int dk, int dv);

// TMA map over a [tokens][H][128] bf16 tensor whose boxes are one chunk of 16
// tokens x 128 channels of one head (unswizzled, out-of-range rows read 0).
// False if the driver's encoder is unavailable or rejects the arguments.
bool encode_token_rows(CUtensorMap* m, const void* base, int H, int64_t tokens);

// Rank-ordered chain lookup for packed variable-length batches: blockIdx.x = r * H + h
// runs the r-th longest sequence first (longest-processing-time order).  For
// fixed-length batches the order is the natural one.  Small enough to inline
// in each kernel; all threads of the block must call it.
constexpr int kMaxRankedSeqs = 4096;

}  // namespace kda
