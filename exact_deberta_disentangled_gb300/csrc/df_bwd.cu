// df_bwd.cu -- the backward pass: clears the diagonal-sum buffers G / G',
// stores the band bias (df_bias.cu), runs the dQ kernel and the dK/dV kernel
// (df_bwd_kernel.cuh), each followed by the half of the relative-position
// gradients (df_rel.cu) that needs only its own diagonal sums.
//
// "DisentangledFlash" (section "Hugging Face usage") splits the fused
// backward into a dQ kernel and a dK/dV kernel; section "Performance" counts
// the relative-position gradients.
//
// The dQ and dK/dV kernels read the same inputs and write disjoint outputs,
// so they run concurrently: dQ and its relative-gradient half on a side
// stream forked from the caller's stream and joined back at the end.  Each kernel
// is 128-row CTAs over (sequence, head) pairs -- at the L = 8192 workload
// 1,536 CTAs, ten full waves on 152 SMs and a 16-CTA tail -- and running the
// two together lets one kernel's tail overlap the other's waves.
#include <mutex>

#include "df_internal.h"

namespace df {
namespace {

constexpr int kMaxDevices = 64;

// Side stream and fork / join events of each device, created on first use
// with that device current.  The fork / join pair is shared by every call on
// the device, so one call's record-and-wait sequence holds `g_mu`.
std::mutex g_mu;
bool g_tried[kMaxDevices];
cudaStream_t g_side[kMaxDevices];
cudaEvent_t g_fork[kMaxDevices], g_join[kMaxDevices];

bool side_stream(int dev, cudaStream_t& side, cudaEvent_t& fork, cudaEvent_t& join) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    if (!g_tried[dev]) {
        g_tried[dev] = true;
        if (cudaStreamCreateWithFlags(&g_side[dev], cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&g_fork[dev], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&g_join[dev], cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            g_side[dev] = nullptr;
        }
    }
    if (!g_side[dev]) return false;
    side = g_side[dev];
    fork = g_fork[dev];
    join = g_join[dev];
    return true;
}

}  // namespace

int launch_bwd_tc(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* q, const void* k,
                  const void* v, const void* qr, const void* kr, const float* lse, const void* dout, void* dq,
                  void* dk, void* dv, void* dqr, void* dkr, cudaStream_t st, const BwdHook* hook) {
    if (p.D != 32 && p.D != 64 && p.D != 128) return (int)cudaErrorInvalidValue;
    const int Rp = ws.Rp;
    const size_t gbytes = (size_t)p.T * p.H * Rp * 2;
    // G (the dQ kernel's) is cleared before the fork, G' (the dK/dV kernel's)
    // after it, while the dQ kernel starts
    cudaError_t ce = cudaMemsetAsync(ws.G, 0, gbytes, st);
    if (ce != cudaSuccess) return (int)ce;
    // the relative-position bias of every band block, read by both kernels
    // (unless the forward saved it)
    int e = p.saved_bias ? 0 : launch_band_bias(p, ws, dt, q, k, qr, kr, st);
    if (e) return e;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        cudaStream_t side = nullptr;
        cudaEvent_t fork = nullptr, join = nullptr;
        bool conc = side_stream(dev, side, fork, join);
        if (conc && (cudaEventRecord(fork, st) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess)) {
            cudaGetLastError();
            conc = false;   // both kernels on the caller's stream instead
        }
        // dQ kernel: rows = queries (Q, dO), columns = keys (K, V); then the
        // relative-position gradients that need only its G (dQ, dKr), while
        // the dK/dV kernel still runs
        const cudaStream_t sq = conc ? side : st;
        e = launch_bwd_dq(p, ws, dt, q, dout, k, v, ws.G, Rp, ws.acc32a, nullptr, lse, sq);
        if (!e) e = launch_rel_tc(p, ws, dt, Rp, 0, q, kr, dq, dkr, sq, hook);
        if (conc) cudaEventRecord(join, side);
        // dK/dV kernel: rows = keys (K, V), columns = queries (Q, dO); then dK,
        // dQr.  Launched after the dQ kernel has been handed to the side
        // stream, so that the dQ kernel, the shorter of the two, takes the SMs
        // first and the dK/dV kernel's waves fill in behind it.
        if (!e && (ce = cudaMemsetAsync(ws.Gp, 0, gbytes, st)) != cudaSuccess) e = (int)ce;
        if (!e) e = launch_bwd_dkv(p, ws, dt, k, v, q, dout, ws.Gp, Rp, ws.acc32b, dv, lse, st);
        if (!e && hook) hook->fn(hook->ctx, 0, st);   // dV is final
        if (!e) e = launch_rel_tc(p, ws, dt, Rp, 1, k, qr, dk, dqr, st, hook);
        // the caller's stream continues only after the side stream's work too
        if (conc && cudaStreamWaitEvent(st, join, 0) != cudaSuccess && !e) e = (int)cudaErrorUnknown;
    }
    return e;
}

}  // namespace df
