// qdq_device.cuh -- PTX wrappers and bounded waits shared by the sm_103a kernels.
//
// Every wait in this library is bounded: mbarrier waits and inter-CTA counter
// waits give up after a wall-clock limit (read from %globaltimer), record
// QDQ_ERR_TIMEOUT in the calling translation unit's status word and return
// false, so a kernel always terminates. No __trap, no device assert.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "qdq.h"

#define QDQ_DEV __device__ __forceinline__

namespace qdq {

// Wall-clock limit of one bounded wait (about 2 s).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

QDQ_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

QDQ_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

QDQ_DEV int load_volatile(const int *p) { return *(const volatile int *)p; }

QDQ_DEV void record_status(int *status, int code) { atomicCAS(status, 0, code); }

// Device-side index and alignment checks of debug builds (-DQDQ_DEBUG), the
// stand-in for a memory checker: a failed check records QDQ_ERR_BOUNDS in the
// kernel's status word and yields false, and the caller skips the access (never
// a trap). Release builds compile every check to true.
#ifdef QDQ_DEBUG
#define QDQ_CHECK(status, cond) ((cond) ? true : (::qdq::record_status((status), QDQ_ERR_BOUNDS), false))
#else
#define QDQ_CHECK(status, cond) true
#endif

// ---- mbarrier ----------------------------------------------------------------
QDQ_DEV void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
QDQ_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
QDQ_DEV void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
QDQ_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// The suspend-time hint lets the hardware park the waiting warp (so it takes no
// issue slots) until the phase completes or about `kSuspendNs` pass.
constexpr uint32_t kSuspendNs = 20000;
QDQ_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase (no suspend): the cheap first look of a wait
// whose phase has usually completed already.
QDQ_DEV bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
QDQ_DEV bool mbar_wait(uint32_t bar, uint32_t parity, int *status) {
    if (mbar_test_wait(bar, parity)) return true;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (load_volatile(status) != 0) return false;  // another wait already failed
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                record_status(status, QDQ_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait that keeps polling (no suspension): for the level handshakes,
// where the waiter has nothing else to do and reacting late costs the whole GPU.
QDQ_DEV bool mbar_wait_spin(uint32_t bar, uint32_t parity, int *status) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((i & 255) == 0) {
            if (load_volatile(status) != 0) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                record_status(status, QDQ_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// ---- bulk copy global -> shared (1-D, non-tensor, no multicast) -----------------
// dst, src 16-byte aligned; bytes a multiple of 16. Completion is signalled as
// transaction bytes on the mbarrier.
QDQ_DEV void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// L2 policy for data read exactly once (the weight stream): evict first, so it
// does not push out data that is reused (activations, outputs).
QDQ_DEV uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
QDQ_DEV void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// ---- inter-CTA counters ---------------------------------------------------------
QDQ_DEV unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *ctr >= target (wrap-around safe).
QDQ_DEV bool wait_counter(const unsigned *ctr, unsigned target, int *status, uint64_t limit_ns) {
    if ((int)(ld_acquire_gpu(ctr) - target) >= 0) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if ((int)(ld_acquire_gpu(ctr) - target) >= 0) return true;
        if ((i & 15) == 0) {
            if (load_volatile(status) != 0) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                record_status(status, QDQ_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// ---- named barriers (consumer warps only) ----------------------------------------
QDQ_DEV void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- shared-memory loads ---------------------------------------------------------
QDQ_DEV uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
QDQ_DEV uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
QDQ_DEV float4 lds128f(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}
QDQ_DEV float ldsf(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}

// n consecutive 32-bit words starting at a 2-byte-aligned shared address:
// loads the covering 4-byte-aligned words and realigns with funnel shifts.
template <int N>
QDQ_DEV void lds_words_a2(uint32_t a, uint32_t (&out)[N]) {
    const uint32_t base = a & ~3u, sh = (a & 3u) * 8u;
    uint32_t w[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) w[i] = lds32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

// ---- packed fp32x2 arithmetic (Blackwell f32x2 forms) -------------------------------
QDQ_DEV uint64_t pack2(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
QDQ_DEV float lo_of(uint64_t v) { return __uint_as_float((uint32_t)v); }
QDQ_DEV float hi_of(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
QDQ_DEV uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
QDQ_DEV uint64_t fsub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
QDQ_DEV uint64_t bits2(uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | lo; }

// (v & MASK) | 0x4B000000 in one LOP3. Written as C, the mask-then-or costs two
// ALU-pipe instructions per weight, and the ALU pipe (half the FMA pipe's rate)
// is what bounds the batch-1 nibble loops.
template <uint32_t MASK>
QDQ_DEV uint32_t mask_magic(uint32_t v) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "n"(MASK), "n"(0x4B000000));
    return d;
}

// fp16 bit pattern -> fp32 (exact; the conversion the format's scales need).
QDQ_DEV float half_bits_to_float(uint32_t h16) { return __half2float(__ushort_as_half((unsigned short)h16)); }

}  // namespace qdq
