// selftest.cu -- one 128x128x128 bf16 product through exactly the operand
// layouts, descriptors and instruction forms the attention kernel uses, so a
// layout mistake shows up in isolation.
//   mode 0: C = A B^T, A and B K-major in shared memory (the Q K^T form);
//   mode 1: C = A B,   A in tensor memory, B N-major in shared memory (the P V form).
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "prefill_tc.h"

namespace attn {
namespace st {

constexpr uint32_t HALF = 16384;
constexpr uint32_t SMEM_BYTES = 1024 + 4 * HALF + 64;

__global__ void __launch_bounds__(128, 1)
    selftest_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                    const uint32_t *__restrict__ a_words, float *__restrict__ c, int mode, unsigned *status,
                    uint64_t budget_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
    uint8_t *sa = base;
    uint8_t *sb = base + 2 * HALF;
    uint64_t *bar_load = reinterpret_cast<uint64_t *>(base + 4 * HALF);
    uint64_t *bar_mma = bar_load + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_mma + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_load, 1);
        ptx::mbar_init(bar_mma, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) ptx::tmem_alloc(tmem_slot, 256);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, status, budget_ns};

    if (mode == 1) {
        // Row i of A into tensor-memory lane i, columns 128..191 (bf16 pairs).
        const uint32_t t_a = tmem + ((uint32_t)(warp * 32) << 16) + 128;
        const int i = threadIdx.x;
#pragma unroll 1
        for (int ch = 0; ch < 2; ++ch) {
            uint32_t w[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) w[q] = a_words[i * 64 + ch * 32 + q];
            ptx::tmem_st32(t_a + ch * 32, w);
        }
        ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    __syncthreads();

    if (threadIdx.x == 0) {
        ptx::tc_fence_after();
        const uint64_t pol = ptx::policy_evict_first();
        if (mode == 0) {
            ptx::mbar_arrive_expect_tx(bar_load, 4 * HALF);
            ptx::tma_load_4d(sa, &ma, bar_load, 0, 0, 0, 0, pol);
            ptx::tma_load_4d(sa + HALF, &ma, bar_load, 64, 0, 0, 0, pol);
        } else {
            ptx::mbar_arrive_expect_tx(bar_load, 2 * HALF);
        }
        ptx::tma_load_4d(sb, &mb, bar_load, 0, 0, 0, 0, pol);
        ptx::tma_load_4d(sb + HALF, &mb, bar_load, 64, 0, 0, 0, pol);
        if (wait_bounded(bar_load, 0, wc, kSiteSelftest)) {
            ptx::tc_fence_after();
            const uint32_t a_addr = ptx::smem_addr(sa), b_addr = ptx::smem_addr(sb);
            if (mode == 0) {
                const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
                    ptx::umma_ss(tmem, ptx::desc_kmajor_sw128(a_addr + off), ptx::desc_kmajor_sw128(b_addr + off),
                                 idesc, kk > 0);
                }
            } else {
                const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    ptx::umma_ts(tmem, tmem + 128 + kk * 8, ptx::desc_mnmajor_sw128(b_addr + kk * 2048, HALF), idesc,
                                 kk > 0);
            }
        }
        ptx::umma_commit(bar_mma);
        drain_wait(bar_mma, 0, wc);
        // The loads must also be complete before the CTA can exit.
        drain_wait(bar_load, 0, wc);
    }
    __syncthreads();
    ptx::tc_fence_after();
    if (!*abort_flag) {
        const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
        const int i = threadIdx.x;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
            uint32_t w[32];
            ptx::tmem_ld32(t_row + ch * 32, w);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) c[i * 128 + ch * 32 + q] = __uint_as_float(w[q]);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 256);
    }
}

}  // namespace st

cudaError_t launch_selftest_umma(const CUtensorMap &ma, const CUtensorMap &mb, const void *a, float *c, int mode,
                                 unsigned *status, uint64_t budget_ns, cudaStream_t stream) {
    cudaError_t e =
        cudaFuncSetAttribute(st::selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    st::selftest_kernel<<<1, 128, st::SMEM_BYTES, stream>>>(ma, mb, static_cast<const uint32_t *>(a), c, mode,
                                                            status, budget_ns);
    return cudaGetLastError();
}

}  // namespace attn
