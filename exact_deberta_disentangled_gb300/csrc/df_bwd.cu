// df_bwd.cu -- tensor-core backward (placeholder until the tcgen05 kernels land).
#include "df_common.cuh"
namespace df {
int launch_bwd_tc(const ProblemDev&, const Workspace&, df_dtype, const void*, const void*, const void*,
                  const void*, const void*, const float*, const void*, void*, void*, void*, void*, void*,
                  cudaStream_t) {
    return (int)cudaErrorNotSupported;
}
}  // namespace df
