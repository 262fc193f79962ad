// df_bwd.cu -- the backward pass: the row terms and biases (df_aux.cu),
// clears the diagonal-sum buffers G / G', stores the band bias (df_bias.cu)
// unless the forward saved it, runs the dQ kernel and the dK/dV kernel
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

// Side stream and its events of each device (fork, inputs ready, join),
// created on first use with that device current.  The events are shared by
// every call on the device, so one call's record-and-wait sequence holds
// `g_mu`.
std::mutex g_mu;
bool g_tried[kMaxDevices];
cudaStream_t g_side[kMaxDevices];
cudaEvent_t g_ev[kMaxDevices][3];

struct Side {
    cudaStream_t st = nullptr;
    cudaEvent_t fork = nullptr, ready = nullptr, join = nullptr;
};

bool side_stream(int dev, Side& s) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    if (!g_tried[dev]) {
        g_tried[dev] = true;
        bool good = cudaStreamCreateWithFlags(&g_side[dev], cudaStreamNonBlocking) == cudaSuccess;
        for (int i = 0; i < 3 && good; ++i)
            good = cudaEventCreateWithFlags(&g_ev[dev][i], cudaEventDisableTiming) == cudaSuccess;
        if (!good) {
            cudaGetLastError();
            g_side[dev] = nullptr;
        }
    }
    if (!g_side[dev]) return false;
    s.st = g_side[dev];
    s.fork = g_ev[dev][0];
    s.ready = g_ev[dev][1];
    s.join = g_ev[dev][2];
    return true;
}

}  // namespace

int launch_bwd_tc(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* q, const void* k,
                  const void* v, const void* qr, const void* kr, const void* out, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, void* dqr, void* dkr, cudaStream_t st,
                  const BwdHook* hook) {
    if (p.D != 32 && p.D != 64 && p.D != 128) return (int)cudaErrorInvalidValue;
    const int Rp = ws.Rp;
    const size_t gbytes = (size_t)p.T * p.H * Rp * 2;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    Side side;
    bool conc = side_stream(dev, side);
    if (conc && (cudaEventRecord(side.fork, st) != cudaSuccess ||
                 cudaStreamWaitEvent(side.st, side.fork, 0) != cudaSuccess)) {
        cudaGetLastError();
        conc = false;   // everything on the caller's stream instead
    }
    const cudaStream_t sq = conc ? side.st : st;
    // G (the dQ kernel's) is cleared on the side stream while the caller's
    // stream computes the row terms Dl, the row / column biases of saturated
    // tiles and, unless the forward saved it, the band bias
    cudaError_t ce = cudaMemsetAsync(ws.G, 0, gbytes, sq);
    int e = (int)ce;
    if (!e) e = launch_rowterm(p, dt, out, dout, ws.rowterm, st);
    if (!e) e = launch_relbias(p, dt, q, k, qr, kr, ws.relb, st);
    if (!e && !p.saved_bias) e = launch_band_bias(p, ws, dt, q, k, qr, kr, st);
    if (!e && conc && (cudaEventRecord(side.ready, st) != cudaSuccess ||
                       cudaStreamWaitEvent(side.st, side.ready, 0) != cudaSuccess))
        e = (int)cudaErrorUnknown;
    if (e) {
        // the side stream holds nothing the caller's stream has not waited for
        if (conc && cudaEventRecord(side.join, side.st) == cudaSuccess) cudaStreamWaitEvent(st, side.join, 0);
        return e;
    }
    // dQ kernel: rows = queries (Q, dO), columns = keys (K, V); then the
    // relative-position gradients that need only its G (dQ, dKr), while
    // the dK/dV kernel still runs
    e = launch_bwd_dq(p, ws, dt, q, dout, k, v, ws.G, Rp, ws.acc32a, nullptr, lse, sq);
    if (!e) e = launch_rel_tc(p, ws, dt, Rp, 0, q, kr, dq, dkr, sq, hook);
    if (conc) cudaEventRecord(side.join, side.st);
    // dK/dV kernel: rows = keys (K, V), columns = queries (Q, dO); then dK,
    // dQr.  Launched after the dQ kernel has been handed to the side stream,
    // so that the dQ kernel, the shorter of the two, takes the SMs first and
    // the dK/dV kernel's waves fill in behind it; G' is cleared meanwhile.
    if (!e && (ce = cudaMemsetAsync(ws.Gp, 0, gbytes, st)) != cudaSuccess) e = (int)ce;
    if (!e) e = launch_bwd_dkv(p, ws, dt, k, v, q, dout, ws.Gp, Rp, ws.acc32b, dv, lse, st);
    if (!e && hook) hook->fn(hook->ctx, 0, st);   // dV is final
    if (!e) e = launch_rel_tc(p, ws, dt, Rp, 1, k, qr, dk, dqr, st, hook);
    // the caller's stream continues only after the side stream's work too
    if (conc && cudaStreamWaitEvent(st, side.join, 0) != cudaSuccess && !e) e = (int)cudaErrorUnknown;
    return e;
}

}  // namespace df
