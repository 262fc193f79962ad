// df_common.cuh -- device-side building blocks shared by the kernels of
// libdfattn: relative-position bucketing, Philox4x32-10, bounded mbarrier
// waits, TMA bulk-tensor copies and the tcgen05 (5th-generation tensor core,
// tensor memory) instructions, all as inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "df_internal.h"

#define DF_DEV __device__ __forceinline__

namespace df {

// ------------------------------------------------------------- indexing

// DeBERTa log bucketing of a relative position r (the formula is stated in
// df_attn.h).  The logarithms run in fp64, so the integer result does not
// depend on fp32 rounding of the ratio.
DF_DEV int bucket_of(int r, int nb, int mp) {
    if (nb <= 0 || mp <= 0) return r;
    const int mid = nb / 2;
    const int a = r < 0 ? -r : r;
    if (a <= mid) return r;
    const double x = log((double)a / (double)mid) / log((double)(mp - 1) / (double)mid) * (double)(mid - 1);
    const int b = mid + (int)ceil(x);
    return r < 0 ? -b : b;
}

DF_DEV int delta_of(int r, int span, int nb, int mp) {
    int d = bucket_of(r, nb, mp) + span;
    d = d < 0 ? 0 : d;
    return d > 2 * span - 1 ? 2 * span - 1 : d;
}

// Sequence geometry: first token and length of sequence b.
DF_DEV void seq_range(const ProblemDev& p, int b, int& t0, int& n) {
    if (p.cu) {
        t0 = __ldg(p.cu + b);
        n = __ldg(p.cu + b + 1) - t0;
    } else {
        t0 = b * p.L;
        n = p.L;
    }
}

// seq_range plus a bounds check: a sequence whose offsets fall outside
// [0, T] or whose length exceeds L is treated as empty (the check kernel has
// recorded the error), so no kernel ever indexes outside its buffers.
DF_DEV bool seq_ok(const ProblemDev& p, int b, int& t0, int& n) {
    seq_range(p, b, t0, n);
    if (n < 0 || n > p.L || t0 < 0 || t0 + n > p.T) {
        n = 0;
        return false;
    }
    return true;
}

// Index of the LSE / row-term entry of (sequence b, head h, position i).
DF_DEV size_t lse_index(const ProblemDev& p, int b, int h, int t0, int i) {
    return p.cu ? (size_t)h * p.T + (size_t)(t0 + i) : ((size_t)b * p.H + h) * (size_t)p.L + (size_t)i;
}

// ---------------------------------------------------------------- Philox

// Philox4x32 with 10 rounds (Salmon et al., SC'11): words 0 and 2 are
// multiplied by the two Philox multipliers, the high halves are mixed into
// words 1 and 3 with the round key, and the key advances by the two Weyl
// increments after every round.
DF_DEV uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// The four keep bits of keys 4*(j>>2) .. 4*(j>>2)+3 for query i of
// (sequence b, head h), as bits 0..3.
DF_DEV uint32_t keep_bits4(const ProblemDev& p, int b, int h, int i, int jq) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)jq, (uint32_t)i, (uint32_t)(b * p.H + h), p.philox_offset),
                                  p.seed_lo, p.seed_hi);
    if (p.keep_all) return 0xFu;
    return (uint32_t)(w.x < p.keep_thr) | ((uint32_t)(w.y < p.keep_thr) << 1) |
           ((uint32_t)(w.z < p.keep_thr) << 2) | ((uint32_t)(w.w < p.keep_thr) << 3);
}

// ------------------------------------------------------------ error word

DF_DEV void raise_error(int* word, int code) {
    if (word) atomicCAS(word, 0, code);
}

// Index checks of a checked build (compiled with DF_CHECKED): an index x
// outside [lo, hi) records DF_ERR_DEVICE_CHECK in the error word and is
// clamped into the range, so the access stays inside its buffer (no trap,
// no fault).  Without DF_CHECKED the check is empty and the code is that of
// the plain build.
#ifdef DF_CHECKED
#define DF_CLAMP_CHECK(x, lo, hi, err)                     \
    do {                                                   \
        if ((x) < (lo) || (x) >= (hi)) {                   \
            raise_error((err), DF_ERR_DEVICE_CHECK);       \
            (x) = (x) < (lo) ? (lo) : (hi) - 1;            \
        }                                                  \
    } while (0)
#else
#define DF_CLAMP_CHECK(x, lo, hi, err) \
    do {                               \
    } while (0)
#endif

DF_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// --------------------------------------------------------------- smem / mbarrier

DF_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// The dynamic shared-memory block rounded up to a 1024-byte boundary (the
// TMA swizzle atoms and the MMA descriptors need it).  The offset is added to
// the __shared__ array itself, so that every pointer derived from the result
// is still known to address shared memory and plain C++ accesses through it
// compile to shared-memory instructions (a round trip through an integer
// leaves the compiler only generic addressing).
DF_DEV uint8_t* smem_align1024(uint8_t* raw) { return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u); }

DF_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

DF_DEV void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

DF_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

DF_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// One bounded probe of an mbarrier phase: the waiting thread may be
// suspended for a system-dependent time while the phase is incomplete.  (A
// suspend-time hint of 20 us was measured slower: the backward pair took
// ~1 % longer, its waiters resuming later after the phase completed.)
DF_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The bounded-wait context of one CTA: the device error word, the CTA-wide
// abort flag (shared memory) and the limits.  A wait gives up once BOTH
// limit_ns have passed on the global timer AND min_probes probes have failed
// (a jump of the global timer alone, as a profiler's clock resynchronisation
// can cause, does not end a wait that is about to succeed; a real hang still
// ends, after at most max(limit, min_probes probes)).  On give-up
// the error word records DF_ERR_TIMEOUT and the abort flag is set, so that
// every other role of the CTA stops waiting too.
struct WaitCtx {
    int* err;
    volatile int* abort;
    unsigned long long limit_ns;
    uint32_t min_probes;
};

DF_DEV WaitCtx wait_ctx(const ProblemDev& p, int* abort_flag_smem) {
    WaitCtx w;
    w.err = p.err;
    w.abort = abort_flag_smem;
    w.limit_ns = p.wait_ns;
    w.min_probes = p.wait_probes;
    return w;
}

// Non-blocking probe of an mbarrier phase (no suspension).
DF_DEV bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

DF_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
    // a phase that has already completed costs one plain probe
    if (mbar_test_wait(bar, parity)) return true;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 7u) == 0) {
            if (*w.abort) return false;
            if (it >= w.min_probes && globaltimer_ns() - t0 > w.limit_ns) {
                raise_error(w.err, DF_ERR_TIMEOUT);
                *w.abort = 1;
                return false;
            }
        }
    }
}

// mbar_wait taken by a whole warp with one outcome for every lane, so that
// warp-collective tcgen05 instructions after it never run divergent.
DF_DEV bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, w));
}

// Wait at exit for this thread's own asynchronous work (a tensor copy in
// flight, the last MMAs) to land, bounded by time only: it ignores the abort
// flag, so that a CTA that gave up still never leaves a copy writing into
// shared memory, or an MMA into tensor memory, after it has released them.
DF_DEV bool mbar_drain(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Pin a register value at this point of the program: the empty volatile asm
// "redefines" it, so arithmetic on a value loaded early cannot be hoisted
// above (and stall right after) the load.  Emits no instruction.
// Read-only loads whose results are used a tile later (prefetches).  Written
// as volatile asm they are issued where they stand: the compiler may move an
// ordinary read-only load down to its first use, and the prefetch would then
// wait on a fresh load.
DF_DEV float ld_early(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
DF_DEV int ld_early(const int32_t* p) {
    int v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
DF_DEV int ld_early(const uint8_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return (int)v;
}

DF_DEV void pin(float& x) { asm volatile("" : "+f"(x)); }
DF_DEV void pin(int& x) { asm volatile("" : "+r"(x)); }

// Named barrier among `nthreads` threads (a multiple of 32).
DF_DEV void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------- TMA

DF_DEV void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)m) : "memory");
}

DF_DEV void tma_load_2d(void* smem_dst, const CUtensorMap* m, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(smem_dst)),
        "l"((uint64_t)m), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

DF_DEV void tma_load_3d(void* smem_dst, const CUtensorMap* m, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"((uint64_t)m), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- tcgen05

// Shared-memory matrix descriptor (tcgen05 form): start address, leading-
// and stride-dimension byte offsets (all >> 4), descriptor version 1 and the
// swizzle mode (0 none, 2 128B, 4 64B, 6 32B).
DF_DEV uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)(swz & 7u) << 61);
}

// Instruction descriptor of kind::f16 with fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

DF_DEV void tc_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
DF_DEV void tc_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
DF_DEV void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
DF_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DF_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]
DF_DEV void tc_mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
DF_DEV void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-collective forms: the whole warp executes them (its control flow
// warp-uniform) and elect.sync picks the one lane that issues the MMA or the
// commit.  Issued this way an MMA costs about its tensor-pipe time (64 cycles
// for 128 x 128 x 16); issued from a single-lane branch it cost 2-4x more.
DF_DEV void tc_mma_ss_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
DF_DEV void tc_mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
DF_DEV void tc_commit_w(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05.mma of this
// thread have completed.
DF_DEV void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

DF_DEV void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
DF_DEV void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (base lane + t), columns col .. col+31.
DF_DEV void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Same as tc_ld32, into 32 consecutive elements of a register array.
DF_DEV void tc_ld32p(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

DF_DEV void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Same as tc_ld16, into 16 consecutive elements of a register array.
DF_DEV void tc_ld16p(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

DF_DEV void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

DF_DEV void tc_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Keep bits of the 32 keys j0 .. j0+31 (j0 a multiple of 4) for query i, as
// bits 0..31; one Philox call per 4 keys, in a rolled loop.
DF_DEV uint32_t keep_bits32_row(const ProblemDev& p, int b, int h, int i, int j0) {
    uint32_t k = 0;
#pragma unroll 1
    for (int q = 0; q < 8; ++q) k |= keep_bits4(p, b, h, i, (j0 >> 2) + q) << (4 * q);
    return k;
}

// Keep bits of the 32 queries i0 .. i0+31 for key j, as bits 0..31.  A
// warp-collective call: every lane of the warp calls it, and the four lanes
// of each quad hold the four keys of one Philox output (j & 3 == lane & 3,
// the same j >> 2).  One Philox call yields one query's bits for all four
// keys, so each lane of a quad draws 8 of the 32 queries (i0 + a + 4m for
// lane a = lane & 3, m = 0..7) and the quad exchanges them:
//   V_a bit (4m + k) = keep(i0 + a + 4m, key k of the quad)
//   lane a' returns sum_a ((V_a >> a') & 0x11111111) << a.
DF_DEV uint32_t keep_bits32_col(const ProblemDev& p, int b, int h, int i0, int j) {
    const int lane = threadIdx.x & 31, a = lane & 3;
    uint32_t v = 0;
#pragma unroll 1
    for (int m = 0; m < 8; ++m) v |= keep_bits4(p, b, h, i0 + a + 4 * m, j >> 2) << (4 * m);
    uint32_t k = 0;
#pragma unroll
    for (int src = 0; src < 4; ++src) {
        const uint32_t vs = __shfl_sync(0xffffffffu, v, (lane & ~3) | src);
        k |= ((vs >> a) & 0x11111111u) << src;
    }
    return k;
}

// Pack two fp32 into one 32-bit word of 16-bit values: `lo` in bits 0..15.
template <bool BF16>
DF_DEV uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if (BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed fp32 arithmetic (f32x2: one instruction does the work of two,
// each lane rounded exactly as the scalar instruction would round it).
DF_DEV void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0, float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
DF_DEV void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
DF_DEV void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// max(a, b, c) in one instruction
DF_DEV float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

DF_DEV float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace df
