// common.cuh -- pieces shared by the library's kernels: the device status word,
// bounded mbarrier waits, and the 4-D tensor coordinate order of the two
// layouts.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace attn {

// Status codes written to the device status word (the same values as the
// C ABI's attn_status_t).
constexpr unsigned kStatusTimeout = 4;
constexpr unsigned kStatusDeviceBounds = 6;

// Wait-site ids reported with a timeout (which wait gave up).
enum WaitSite : unsigned {
    kSiteMmaQ = 1,
    kSiteMmaPoll = 2,
    kSiteProducerEmpty = 3,
    kSiteSoftmaxS = 4,
    kSiteSoftmaxO = 5,
    kSiteEpilogueO = 6,
    kSiteDrain = 7,
    kSiteDecodeFull = 8,
    kSiteDecodeEmpty = 9,
    kSiteSelftest = 10,
    kSiteDecodeTable = 11,
    kSiteVarlenOffsets = 12,
    kSitePagedTable = 13,
    kSiteSoftmaxV = 14,
    kSiteAppendSlot = 15,
    kSiteDecodeSeqlen = 16,
    kSiteProducerQ = 17,
    kSiteEpilogueSlot = 18,
    kSiteItem = 19,
    kSiteStoreCmd = 20,
};

// First error wins; the site is informative only.
__device__ __forceinline__ void report_status(unsigned *status, unsigned code, unsigned site) {
    if (atomicCAS(status, 0u, code) == 0u) atomicExch(status + 1, site);
}

struct WaitCtx {
    volatile int *abort_flag;  // CTA-wide "give up" flag in shared memory
    unsigned *status;          // device status word [code, site]
    uint64_t budget_ns;        // time budget of one wait
};

// Wait for the phase of `bar` with the given parity.  Gives up (returns false)
// when another thread of the CTA has raised the abort flag, or when the budget
// runs out, in which case it raises the flag and records a timeout.
// Both waits are inlined: a kernel whose warpgroups run under different
// setmaxnreg register budgets must not share an out-of-line device function
// between them.
static __device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, const WaitCtx &w, unsigned site) {
    if (ptx::mbar_try(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try(bar, parity)) return true;
        if (*w.abort_flag) return false;
        if ((it & 15u) == 0 && ptx::globaltimer() - t0 > w.budget_ns) {
            *w.abort_flag = 1;
            report_status(w.status, kStatusTimeout, site);
            return false;
        }
    }
}

// Wait by polling with the non-blocking test (the issuing threads, whose
// reaction time is on the critical path).
static __device__ __forceinline__ bool wait_spin(uint64_t *bar, uint32_t parity, const WaitCtx &w, unsigned site) {
    if (ptx::mbar_test(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_test(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*w.abort_flag) return false;
            if (ptx::globaltimer() - t0 > w.budget_ns) {
                *w.abort_flag = 1;
                report_status(w.status, kStatusTimeout, site);
                return false;
            }
        }
    }
}

// Wait for completion of an operation this thread itself started (a copy or
// an MMA in flight), ignoring the abort flag: used on the way out so that no
// asynchronous write into shared or tensor memory outlives the CTA.  Still
// bounded by the budget.
static __device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity, const WaitCtx &w) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 0;; ++it) {
        if (ptx::mbar_try(bar, parity)) return true;
        if ((it & 15u) == 0 && ptx::globaltimer() - t0 > w.budget_ns) {
            report_status(w.status, kStatusTimeout, kSiteDrain);
            return false;
        }
    }
}

// Tensor maps over q/k/v/out are 4-D with dims ordered as the memory is:
// BSHD -> {d, H, S, B}; BHSD -> {d, S, H, B}.  This returns the coordinate
// vector for (c = d offset, h, s, b).
struct Coord4 {
    int c0, c1, c2, c3;
};

__device__ __forceinline__ Coord4 coord4(bool bhsd, int c, int h, int s, int b) {
    return bhsd ? Coord4{c, s, h, b} : Coord4{c, h, s, b};
}

// ---------------------------------------------------------------------------
// Rounding of fp32 results to the bf16 output: the three modes the MoonMath
// HIP kernel page measures its bf16 output in (benchmark section).
enum RoundMode : int {
    kRoundRTNE = 0,  // to nearest, ties to even
    kRoundRTNA = 1,  // to nearest, ties away from zero
    kRoundRTZ = 2,   // toward zero
};

// Ties-away rounding on the bit pattern: adding half a bf16 unit (0x8000) to
// the magnitude bits carries into the kept 16 bits exactly when the dropped
// part is at least half a unit; a carry out of the significand moves the
// exponent, and past the largest finite bf16 it reaches infinity.
static __device__ __forceinline__ uint32_t bf16_bits_rna(float x) {
    const uint32_t u = __float_as_uint(x);
    const uint32_t mag = u & 0x7fffffffu;
    if (mag > 0x7f800000u) return (u >> 16) | 0x40u;  // NaN stays a quiet NaN
    return ((mag + 0x8000u) >> 16) | ((u >> 16) & 0x8000u);
}

// Two fp32 values to packed bf16 (lo in the low half) in the given mode.
static __device__ __forceinline__ uint32_t pack_bf16x2_mode(float lo, float hi, int mode) {
    if (mode == kRoundRTZ) return ptx::pack_bf16x2_rz(lo, hi);
    if (mode == kRoundRTNA) return bf16_bits_rna(lo) | (bf16_bits_rna(hi) << 16);
    return ptx::pack_bf16x2(lo, hi);
}

static __device__ __forceinline__ uint16_t bf16_bits_mode(float x, int mode) {
    return (uint16_t)(pack_bf16x2_mode(x, 0.f, mode) & 0xffffu);
}

}  // namespace attn
