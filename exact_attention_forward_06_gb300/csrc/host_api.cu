// host_api.cu -- attn_fwd_host: the forward pass from and to host memory.
//
// The inputs are copied to a caller-provided device workspace, the forward
// kernel runs there, and the outputs are copied back, all asynchronously and
// in batch chunks on three helper streams (copy in, compute, copy out) so that
// the copies of one chunk overlap the compute of another:
//
//   copy-in  stream:  Q,K,V[c0]  Q,K,V[c1]  Q,K,V[c2] ...
//   compute  stream:             fwd[c0]    fwd[c1]   ...
//   copy-out stream:                        O,lse[c0] O,lse[c1] ...
//
// Events tie the helper streams to the caller's stream at both ends, so the
// call is ordered like any other work on `stream`.  The helper streams and
// events are created once per device and kept; nothing is allocated per call.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 8;

struct HostStreams {
    bool ready = false;
    cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in_done[kMaxChunks] = {}, comp_done[kMaxChunks] = {};
};

std::mutex g_host_mu;
HostStreams g_host[kMaxDevices];

bool host_streams(int dev, HostStreams **hs) {
    HostStreams &h = g_host[dev];
    if (!h.ready) {
        const unsigned ev_flags = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&h.comp, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&h.start, ev_flags) != cudaSuccess ||
            cudaEventCreateWithFlags(&h.done, ev_flags) != cudaSuccess)
            return false;
        for (int c = 0; c < kMaxChunks; ++c)
            if (cudaEventCreateWithFlags(&h.in_done[c], ev_flags) != cudaSuccess ||
                cudaEventCreateWithFlags(&h.comp_done[c], ev_flags) != cudaSuccess)
                return false;
        h.ready = true;
    }
    *hs = &h;
    return true;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Byte sizes of one batch of q (and out), k (and v) and lse.
struct BatchBytes {
    size_t q, kv, lse;
};

BatchBytes batch_bytes(int Hq, int Hkv, int Sq, int Sk, int d) {
    return {(size_t)Sq * Hq * d * 2, (size_t)Sk * Hkv * d * 2, (size_t)Hq * Sq * 4};
}

}  // namespace

extern "C" {

size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int d) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || d != 128 || Hq % Hkv != 0) return 0;
    const BatchBytes bb = batch_bytes(Hq, Hkv, Sq, Sk, d);
    // q, out, k, v and lse for the whole batch, each 256-byte aligned
    return 2 * align256(bb.q * B) + 2 * align256(bb.kv * B) + align256(bb.lse * B);
}

attn_status_t attn_fwd_host(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq,
                            int Hkv, int Sq, int Sk, int d, int layout, int causal, float scale, int round_mode,
                            void *workspace, size_t workspace_bytes, void *stream) {
    if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
    // Everything attn_fwd would reject is rejected here too, before any copy.
    if (layout != ATTN_LAYOUT_BSHD && layout != ATTN_LAYOUT_BHSD) return ATTN_ERR_INVALID_ARG;
    if (!(scale >= 0.f) || scale == INFINITY) return ATTN_ERR_INVALID_ARG;
    if (round_mode != ATTN_ROUND_RTNE && round_mode != ATTN_ROUND_RTNA && round_mode != ATTN_ROUND_RTZ)
        return ATTN_ERR_INVALID_ARG;
    if ((int64_t)B * Sq * Hq > (int64_t)1 << 31 || (int64_t)B * Sk * Hkv > (int64_t)1 << 31) return ATTN_ERR_INVALID_ARG;
    const size_t need = attn_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, d);
    if (need == 0) return d != 128 && d > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return ATTN_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    const BatchBytes bb = batch_bytes(Hq, Hkv, Sq, Sk, d);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *q_d = ws;
    uint8_t *o_d = q_d + align256(bb.q * B);
    uint8_t *k_d = o_d + align256(bb.q * B);
    uint8_t *v_d = k_d + align256(bb.kv * B);
    uint8_t *l_d = v_d + align256(bb.kv * B);
    // Batch chunks: both layouts keep one batch contiguous (BSHD [b][s][h][d],
    // BHSD [b][h][s][d]), and lse is [b][h][s].
    const int n_chunks = B < kMaxChunks ? B : kMaxChunks;
    const int per = (B + n_chunks - 1) / n_chunks;
    std::lock_guard<std::mutex> lock(g_host_mu);
    HostStreams *hs = nullptr;
    if (!host_streams(dev, &hs)) return ATTN_ERR_CUDA;
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    if (cudaEventRecord(hs->start, user) != cudaSuccess || cudaStreamWaitEvent(hs->in, hs->start, 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
    // The copy-out stream also writes `out`/`lse` only after earlier work on
    // the caller's stream: make it wait too.
    if (cudaStreamWaitEvent(hs->out, hs->start, 0) != cudaSuccess) return ATTN_ERR_CUDA;
    for (int c = 0, b0 = 0; b0 < B; ++c, b0 += per) {
        const int nb = (B - b0) < per ? (B - b0) : per;
        const size_t qo = bb.q * b0, ko = bb.kv * b0, lo = bb.lse * b0;
        const char *qh = static_cast<const char *>(q), *kh = static_cast<const char *>(k);
        const char *vh = static_cast<const char *>(v);
        if (cudaMemcpyAsync(q_d + qo, qh + qo, bb.q * nb, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
            cudaMemcpyAsync(k_d + ko, kh + ko, bb.kv * nb, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
            cudaMemcpyAsync(v_d + ko, vh + ko, bb.kv * nb, cudaMemcpyHostToDevice, hs->in) != cudaSuccess ||
            cudaEventRecord(hs->in_done[c], hs->in) != cudaSuccess)
            return ATTN_ERR_CUDA;
        if (cudaStreamWaitEvent(hs->comp, hs->in_done[c], 0) != cudaSuccess) return ATTN_ERR_CUDA;
        attn_status_t st = attn_fwd_rounded(q_d + qo, k_d + ko, v_d + ko, o_d + qo,
                                            lse ? reinterpret_cast<float *>(l_d + lo) : nullptr, nb, Hq, Hkv, Sq,
                                            Sk, d, layout, causal, scale, round_mode, hs->comp);
        if (st != ATTN_OK) return st;
        if (cudaEventRecord(hs->comp_done[c], hs->comp) != cudaSuccess ||
            cudaStreamWaitEvent(hs->out, hs->comp_done[c], 0) != cudaSuccess)
            return ATTN_ERR_CUDA;
        if (cudaMemcpyAsync(static_cast<char *>(out) + qo, o_d + qo, bb.q * nb, cudaMemcpyDeviceToHost, hs->out) !=
            cudaSuccess)
            return ATTN_ERR_CUDA;
        if (lse && cudaMemcpyAsync(reinterpret_cast<char *>(lse) + lo, l_d + lo, bb.lse * nb, cudaMemcpyDeviceToHost,
                                   hs->out) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    if (cudaEventRecord(hs->done, hs->out) != cudaSuccess || cudaStreamWaitEvent(user, hs->done, 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

}  // extern "C"
