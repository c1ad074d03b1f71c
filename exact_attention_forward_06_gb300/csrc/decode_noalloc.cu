// decode_noalloc.cu -- attn_decode_paged_noalloc: the paged decode step for
// callers that cannot allocate device memory.
//
// attn_decode_paged needs a caller-provided workspace for its split partials.
// Some callers have no way to provide one: a host framework whose operator
// interface hands a kernel only its input and output buffers and offers no
// allocator or workspace hook, or an engine that has reserved all of HBM up
// front for its own pools and forbids any further cudaMalloc (which would also
// synchronise the device in the middle of a latency-critical loop).  For them
// the partials live in a fixed device array that belongs to the library.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds ATTN_DECODE_NOALLOC_SCRATCH_BYTES of it until the process
// exits.  In host code its name is only a host-side stand-in, not a device
// address, so its real address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed to the kernels.
// That lookup happens inside the first call made on each device; make that
// first call before any stream capture.
//
// Every call shares the one array and it keeps the previous call's contents.
// Nothing in it has to start at zero: every split writes all of its partial
// entries (an empty split writes zeros and -inf) before the merge reads them.
// Calls that overlap on the GPU (for example on two streams without ordering
// between them) race on the array and must be avoided.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"

static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[ATTN_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
attn_status_t scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return ATTN_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_decode_paged_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                                   const int32_t *block_table, const int32_t *seqlens, void *out,
                                                   float *lse, int B, int Hq, int Hkv, int d, int page_size,
                                                   int num_pages, int max_blocks_per_seq, float scale,
                                                   void *stream) {
    const size_t need = attn_decode_workspace_bytes(B, Hq, d, max_blocks_per_seq);
    if (need > (size_t)ATTN_DECODE_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
    void *scratch = nullptr;
    // Arguments are validated by attn_decode_paged; look the scratch up only
    // for calls that can reach the device.
    if (need > 0) {
        attn_status_t st = scratch_on_current_device(&scratch);
        if (st != ATTN_OK) return st;
    }
    return attn_decode_paged(q, k_pages, v_pages, block_table, seqlens, out, lse, B, Hq, Hkv, d, page_size,
                             num_pages, max_blocks_per_seq, scale, scratch, (size_t)ATTN_DECODE_NOALLOC_SCRATCH_BYTES,
                             stream);
}
