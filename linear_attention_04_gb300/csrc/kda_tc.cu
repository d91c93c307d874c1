// kda_tc.cu -- tcgen05/TMEM tensor-core path (bf16, dk = dv = 128).
#include "kda_internal.cuh"

namespace kda {

bool tc_supported(int dtype, int dk, int dv) { return false; }

int launch_tc(const FwdParams& p, cudaStream_t stream) { return KDA_ERR_UNSUPPORTED_SHAPE; }

}  // namespace kda
