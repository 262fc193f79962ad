// df_fwd.cu -- tensor-core forward (placeholder until the tcgen05 kernel lands).
#include "df_common.cuh"
namespace df {
int launch_fwd_tc(const ProblemDev&, const Workspace&, df_dtype, const void*, const void*, const void*,
                  const void*, const void*, void*, float*, cudaStream_t) {
    return (int)cudaErrorNotSupported;
}
}  // namespace df
