// df_bwd_dq.cu -- instantiates the dQ kernel (rows = queries) of df_bwd_kernel.cuh for
// every head dim, storage type and dropout setting (one translation unit per
// kernel keeps the build parallel).
#include "df_bwd_kernel.cuh"

namespace df {

int launch_bwd_dq(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* r1, const void* r2, const void* c1,
         const void* c2, void* Gbuf, int Rp, float* acc1, void* acc2,
         const float* lse, cudaStream_t st) {
#define DF_ONE(D_, BF_, DR_) launch_one<D_, BF_, 1, DR_>(p, ws, r1, r2, c1, c2, Gbuf, Rp, acc1, acc2, lse, st)
#define DF_DT(D_, DR_) (dt == DF_BF16 ? DF_ONE(D_, true, DR_) : DF_ONE(D_, false, DR_))
#define DF_DROP(D_) (p.dropout ? DF_DT(D_, true) : DF_DT(D_, false))
    switch (p.D) {
        case 32: return DF_DROP(32);
        case 64: return DF_DROP(64);
        case 128: return DF_DROP(128);
    }
#undef DF_DROP
#undef DF_DT
#undef DF_ONE
    return (int)cudaErrorInvalidValue;
}

}  // namespace df
