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
// That lookup happens inside the first call made in each CUDA context (the
// runtime's primary context of a device, or any other context the caller
// makes current); make that first call before any stream capture.  The
// address is remembered under the context's unique id, so a context created
// later (after cudaDeviceReset, say) gets its own lookup and never a stale
// address.
//
// Every call shares the one array and it keeps the previous call's contents.
// Nothing in it has to start at zero: every split writes all of its partial
// entries (an empty split writes zeros and -inf) before the merge reads them.
// Calls that overlap on the GPU (for example on two streams without ordering
// between them) race on the array and must be avoided.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "api_internal.h"
#include "attn.h"

static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[ATTN_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxContexts = 64;

struct ScratchEntry {
    unsigned long long ctx_id;
    void *ptr;
};

std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxContexts] = {};
int g_scratch_used = 0;
int g_scratch_next = 0;  // slot replaced next once the table is full
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

// Unique id of the calling thread's current context, or false when there is
// none (or the driver cannot say).
bool current_context_id(unsigned long long *id) {
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context, looked up with
// cudaGetSymbolAddress the first time a context asks and remembered under its id.
attn_status_t scratch_in_current_context(void **out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_ctx_current == nullptr || g_ctx_id == nullptr) {
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &r1) != cudaSuccess ||
            r1 != cudaDriverEntryPointSuccess || f1 == nullptr ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &r2) != cudaSuccess ||
            r2 != cudaDriverEntryPointSuccess || f2 == nullptr)
            return ATTN_ERR_CUDA;
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
        g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
    }
    unsigned long long id = 0;
    if (current_context_id(&id)) {
        for (int i = 0; i < g_scratch_used; ++i)
            if (g_scratch[i].ctx_id == id) {
                *out = g_scratch[i].ptr;
                return ATTN_OK;
            }
    }
    // First call in this context (or no context yet: the lookup makes the
    // device's primary context current).
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_noalloc_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ERR_CUDA;
    if (!current_context_id(&id)) return ATTN_ERR_CUDA;
    int slot = g_scratch_used;
    if (slot < kMaxContexts) {
        ++g_scratch_used;
    } else {
        slot = g_scratch_next;
        g_scratch_next = (g_scratch_next + 1) % kMaxContexts;
    }
    g_scratch[slot] = ScratchEntry{id, ptr};
    *out = ptr;
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_decode_paged_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                                   const int32_t *block_table, const int32_t *seqlens, void *out,
                                                   float *lse, int B, int Hq, int Hkv, int d, int page_size,
                                                   int num_pages, int max_blocks_per_seq, float scale,
                                                   void *stream) {
    // The same argument checks as attn_decode_paged first, so that a bad call
    // gets the same status whatever its size; only then the array's limit.
    attn_status_t st = attn::check_decode_args(q, k_pages, v_pages, block_table, seqlens, out, lse, B, Hq, Hkv, d,
                                               page_size, num_pages, max_blocks_per_seq, scale);
    if (st != ATTN_OK) return st;
    const size_t need = attn_decode_workspace_bytes(B, Hq, d, max_blocks_per_seq);
    if (need > (size_t)ATTN_DECODE_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((st = scratch_in_current_context(&scratch)) != ATTN_OK) return st;
    return attn_decode_paged(q, k_pages, v_pages, block_table, seqlens, out, lse, B, Hq, Hkv, d, page_size,
                             num_pages, max_blocks_per_seq, scale, scratch, (size_t)ATTN_DECODE_NOALLOC_SCRATCH_BYTES,
                             stream);
}
