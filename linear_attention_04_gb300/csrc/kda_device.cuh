// Small device helpers shared by the kernels of libkda.so.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {

constexpr int kMaxRankedSeqsDev = 512;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Work item of one CTA: the token range [t0, t1) of one (sequence, head) pair
// and the row index base used for the [., H, .] layouts.
struct Chain {
  int seq;      // sequence index (state index)
  int head;
  int64_t t0;   // first token row (absolute, in the flattened B*T token axis)
  int64_t t1;   // one past the last
  bool valid;   // false: the packing table is malformed (the CTA must store nothing)
};

// Maps a chain rank to (sequence, head).  For packed variable-length batches
// of at most kMaxRankedSeqsDev sequences, rank r runs the r-th longest
// sequence (ties by index), so that the block scheduler, which hands out
// blocks roughly in index order, starts the longest chains first.  Every
// thread of the block must call this (it uses __syncthreads and `scratch`, an
// int array of kMaxRankedSeqsDev + 1 entries in shared memory).
// The packing table is checked where it is used: cu_seqlens[0] = 0,
// cu_seqlens[N] = T and 0 <= t0 <= t1 <= T for this block's sequence; a block
// whose check fails gets valid = false and an empty token range.
__device__ __forceinline__ Chain chain_for_block(int rank_flat, int H, int N, int T,
                                                 const int32_t* cu_seqlens, int* scratch) {
  Chain c;
  int r = rank_flat / H;
  c.head = rank_flat - r * H;
  c.valid = true;
  if (cu_seqlens == nullptr) {
    c.seq = r;
    c.t0 = (int64_t)r * T;
    c.t1 = c.t0 + T;
    return c;
  }
  if (N <= kMaxRankedSeqsDev) {
    int* lens = scratch;
    for (int s = threadIdx.x; s < N; s += blockDim.x) lens[s] = cu_seqlens[s + 1] - cu_seqlens[s];
    __syncthreads();
    for (int s = threadIdx.x; s < N; s += blockDim.x) {
      int ls = lens[s], rank = 0;
      for (int o = 0; o < N; ++o) {
        int lo = lens[o];
        rank += (lo > ls) || (lo == ls && o < s);
      }
      if (rank == r) scratch[kMaxRankedSeqsDev] = s;
    }
    __syncthreads();
    r = scratch[kMaxRankedSeqsDev];
    __syncthreads();
  }
  c.seq = r;
  const int32_t a = cu_seqlens[r], b = cu_seqlens[r + 1];
  c.valid = cu_seqlens[0] == 0 && cu_seqlens[N] == T && 0 <= a && a <= b && b <= T;
  c.t0 = c.valid ? a : 0;
  c.t1 = c.valid ? b : 0;
  return c;
}

}  // namespace kda
