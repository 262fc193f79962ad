// df_noalloc.cu -- a forward entry point that allocates nothing, for callers
// that cannot allocate device memory.
//
// df_attn_fwd needs a small workspace (error word, relative-index table,
// per-token relative dot products).  Some callers cannot provide one: code
// that runs inside a host framework that owns every byte of device memory
// (a plugin or custom operator of an inference server, whose arena it may not
// grow), or latency-critical loops where cudaMalloc's implicit device-wide
// synchronisation is not acceptable.  df_attn_fwd_noalloc runs the same
// forward with its workspace in a file-scope __device__ array instead.
//
// The array is a static allocation of the library module: every GPU that
// loads the library holds kNoAllocScratchBytes of device memory until the
// process exits.  Host code cannot use the array's name as a device address,
// so the first call on each device, with that device current, looks the
// address up with cudaGetSymbolAddress and caches it.
#include <mutex>

#include "df_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_fwd_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];   // device address of g_fwd_scratch, per device ordinal

}  // namespace

extern "C" df_status df_attn_fwd_noalloc(const df_attn_params* p, const void* q, const void* k, const void* v,
                                          const void* qr, const void* kr, void* out, float* lse,
                                          df_stream_t stream) {
    const size_t need = df_attn_workspace_size(p, 0);
    if (need == 0)   // invalid or unsupported parameters: report the precise code
        return df_attn_fwd(p, q, k, v, qr, kr, out, lse, nullptr, 0, stream);
    if (need > kNoAllocScratchBytes) return DF_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DF_ERR_CUDA;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        scratch = g_scratch_addr[dev];
        if (!scratch) {
            if (cudaGetSymbolAddress(&scratch, g_fwd_scratch) != cudaSuccess || !scratch) {
                cudaGetLastError();
                return DF_ERR_CUDA;
            }
            g_scratch_addr[dev] = scratch;
        }
    }
    // the error word at the start of the workspace is cleared by df_attn_fwd;
    // every other scratch byte it reads is written earlier in the same call
    return df_attn_fwd(p, q, k, v, qr, kr, out, lse, scratch, kNoAllocScratchBytes, stream);
}

extern "C" df_status df_attn_fwd_noalloc_device_error(df_stream_t stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DF_ERR_CUDA;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        scratch = g_scratch_addr[dev];
    }
    // no call on this device yet: nothing can have failed
    if (!scratch) return DF_OK;
    return df_get_device_error(scratch, stream);
}
