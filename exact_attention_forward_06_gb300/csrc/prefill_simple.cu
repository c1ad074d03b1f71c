// prefill_simple.cu -- the plain SIMT form of the same attention: one warp per
// query row, each lane owning 4 of the 128 head-dim elements, keys visited one
// at a time with the online-softmax update of "FlashAttention-4 中的 IO 感知块
// 分块策略" (m' = max(m, s), l' = l exp(m - m') + exp(s - m')).  No tensor
// cores, no shared memory staging: a debugging cross-check for the tensor-core
// kernel, never a fallback for it.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "prefill_tc.h"

namespace attn {
namespace g0 {

constexpr int WARPS = 4;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ int64_t offset(bool bhsd, int b, int s, int h, int S, int H) {
    return bhsd ? (((int64_t)b * H + h) * S + s) * 128 : (((int64_t)b * S + s) * H + h) * 128;
}

__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&x)[4]) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
}

__global__ void __launch_bounds__(WARPS * 32)
    simple_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                  const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *__restrict__ out, const PrefillParams p) {
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * WARPS + (threadIdx.x >> 5);
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    if (i >= p.Sq) return;
    const int g = h / p.G;
    const bool bhsd = p.bhsd != 0;
    float qf[4];
    load4(q + offset(bhsd, b, i, h, p.Sq, p.Hq) + lane * 4, qf);
#pragma unroll
    for (int e = 0; e < 4; ++e) qf[e] *= p.scale_log2;
    const int last = p.causal ? min(p.Sk - 1, i + p.Sk - p.Sq) : p.Sk - 1;
    float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j <= last; ++j) {
        float kf[4], vf[4];
        load4(k + offset(bhsd, b, j, g, p.Sk, p.Hkv) + lane * 4, kf);
        float dot = qf[0] * kf[0] + qf[1] * kf[1] + qf[2] * kf[2] + qf[3] * kf[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        const float m_new = fmaxf(m, dot);
        const float corr = ptx::ex2(m - m_new);  // m = -inf on the first key -> 0
        const float pj = ptx::ex2(dot - m_new);
        load4(v + offset(bhsd, b, j, g, p.Sk, p.Hkv) + lane * 4, vf);
        l = l * corr + pj;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = acc[e] * corr + pj * vf[e];
        m = m_new;
    }
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    __nv_bfloat16 *o = out + offset(bhsd, b, i, h, p.Sq, p.Hq) + lane * 4;
    uint2 packed;
    packed.x = ptx::pack_bf16x2(l > 0.f ? acc[0] * inv : 0.f, l > 0.f ? acc[1] * inv : 0.f);
    packed.y = ptx::pack_bf16x2(l > 0.f ? acc[2] * inv : 0.f, l > 0.f ? acc[3] * inv : 0.f);
    *reinterpret_cast<uint2 *>(o) = packed;
    if (lane == 0 && p.lse != nullptr)
        p.lse[((int64_t)b * p.Hq + h) * p.Sq + i] = l > 0.f ? (m + ptx::lg2(l)) * LN2 : -INFINITY;
}

}  // namespace g0

cudaError_t launch_prefill_simple(const void *q, const void *k, const void *v, void *out, float *lse,
                                  const PrefillParams &p0, cudaStream_t stream) {
    PrefillParams p = p0;
    p.lse = lse;
    dim3 grid((p.Sq + g0::WARPS - 1) / g0::WARPS, p.Hq, p.B);
    g0::simple_kernel<<<grid, g0::WARPS * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), static_cast<__nv_bfloat16 *>(out), p);
    return cudaGetLastError();
}

}  // namespace attn
