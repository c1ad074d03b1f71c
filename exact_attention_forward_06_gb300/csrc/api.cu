// api.cu -- the C ABI (include/attn.h): argument validation, TMA tensor-map
// encoding, the per-device status word, and kernel launches on the caller's
// stream.  Nothing here allocates device memory.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "attn.h"
#include "api_internal.h"
#include "prefill_tc.h"

// Device status word: [0] = first error code recorded, [1] = wait/check site.
__device__ unsigned int g_attn_status[2];

// Work counters of the prefill launches whose CTAs claim items as they free up:
// each launch takes the next pair (next item, CTAs done) round robin, and its
// last CTA sets the pair back to zero.  Launches in flight at the same time on
// one device therefore need distinct pairs: up to kSchedPairs of them.
constexpr int kSchedPairs = 256;
__device__ unsigned int g_prefill_sched[kSchedPairs][2];

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultBudgetNs = 2000000000ull;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    unsigned *status = nullptr;
    unsigned *sched = nullptr;  // g_prefill_sched on this device
    void *workspace = nullptr;  // caller-owned, for attn_fwd's tail split
    size_t workspace_bytes = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint64_t> g_budget{kDefaultBudgetNs};
std::atomic<int> g_inject{0};
std::atomic<unsigned> g_sched_next{0};

// The counter pair for the next prefill launch on the device.
unsigned *next_sched(const DeviceInfo *di) {
    return di->sched + 2 * (g_sched_next.fetch_add(1, std::memory_order_relaxed) % kSchedPairs);
}

attn_status_t device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        // The kernels are built for sm_103a only.
        d.supported = (major == 10 && minor == 3);
        d.sm_count = sms;
        if (d.supported) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_attn_status) != cudaSuccess) return ATTN_ERR_CUDA;
            d.status = static_cast<unsigned *>(ptr);
            if (cudaMemset(d.status, 0, 2 * sizeof(unsigned)) != cudaSuccess) return ATTN_ERR_CUDA;
            if (cudaGetSymbolAddress(&ptr, g_prefill_sched) != cudaSuccess) return ATTN_ERR_CUDA;
            d.sched = static_cast<unsigned *>(ptr);
        }
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return ATTN_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    if (!d.supported) return ATTN_ERR_UNSUPPORTED;
    *out = &d;
    return ATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t budget() { return g_budget.load(std::memory_order_relaxed); }

// 4-D bf16 map over a dense BSHD ([B][S][H][d], dims {d,H,S,B}) or BHSD
// ([B][H][S][d], dims {d,S,H,B}) tensor; box = 64 head-dim elements (128 B,
// 128-byte swizzle) x `rows` sequence positions x `heads` heads.  With one
// head the box is `rows` rows of one head; with G heads and 128 / G rows it
// is a head-packed Q or O tile, whose 128 rows land in shared memory as
// (position, head) pairs, head fastest in BSHD (position fastest in BHSD).
bool make_map_4d(CUtensorMap *m, const void *ptr, bool bhsd, int B, int S, int H, int d, int rows, int heads = 1) {
    const cuuint64_t e = 2;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
    if (bhsd) {
        dims[0] = d; dims[1] = S; dims[2] = H; dims[3] = B;
        strides[0] = (cuuint64_t)d * e;
        strides[1] = (cuuint64_t)S * d * e;
        strides[2] = (cuuint64_t)H * S * d * e;
        box[0] = 64; box[1] = rows; box[2] = heads; box[3] = 1;
    } else {
        dims[0] = d; dims[1] = H; dims[2] = S; dims[3] = B;
        strides[0] = (cuuint64_t)d * e;
        strides[1] = (cuuint64_t)H * d * e;
        strides[2] = (cuuint64_t)S * H * d * e;
        box[0] = 64; box[1] = heads; box[2] = rows; box[3] = 1;
    }
    const cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Page-pool map (paged prefill and decode): one box holds whole 16-row pages
// of one KV head, both 64-column halves, ordered in shared memory as
// [8-row group][half][8 rows][64 columns] (1 KiB per 8-row half, 128-byte
// swizzle), so a 128-row tile is 8 boxes of 4 KiB (or one box of 16 row
// groups for 8 consecutive pages).  Dims, innermost first: 64 columns, 8 rows
// (stride Hkv*d*2), 2 halves (stride 128 B), row groups of 8 (stride
// 8*Hkv*d*2), KV head (stride d*2).
bool make_map_pool_groups(CUtensorMap *m, const void *ptr, int num_pages, int Hkv, int d, int groups) {
    const cuuint64_t e = 2, row = (cuuint64_t)Hkv * d * e;
    cuuint64_t dims[5] = {64, 8, 2, (cuuint64_t)num_pages * 2, (cuuint64_t)Hkv};
    cuuint64_t strides[4] = {row, 64 * e, 8 * row, (cuuint64_t)d * e};
    cuuint32_t box[5] = {64, 8, 2, (cuuint32_t)groups, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

attn_status_t check_fwd_args(const void *q, const void *k, const void *v, const void *out, const float *lse,
                             int B, int Hq, int Hkv, int Sq, int Sk, int d, int layout, float scale) {
    if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (layout != ATTN_LAYOUT_BSHD && layout != ATTN_LAYOUT_BHSD) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    // Tensor-map extents are 32-bit; element counts must fit the kernels' 64-bit indexing.
    if ((int64_t)B * Sq * Hq > (int64_t)1 << 31 || (int64_t)B * Sk * Hkv > (int64_t)1 << 31)
        return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

bool valid_round_mode(int m) { return m == ATTN_ROUND_RTNE || m == ATTN_ROUND_RTNA || m == ATTN_ROUND_RTZ; }

attn_status_t fill_prefill_params(attn::PrefillParams *p, const DeviceInfo *di, float *lse, int B, int Hq,
                                  int Hkv, int Sq, int Sk, int layout, int causal, float scale) {
    p->B = B;
    p->Hq = Hq;
    p->Hkv = Hkv;
    p->Sq = Sq;
    p->Sk = Sk;
    p->G = Hq / Hkv;
    p->causal = causal ? 1 : 0;
    p->bhsd = layout == ATTN_LAYOUT_BHSD ? 1 : 0;
    p->scale_log2 = (float)((double)scale * 1.4426950408889634);
    p->lse = lse;
    p->n_m = (Sq + 127) / 128;
    p->pair_heads = (p->G % 2 == 0) ? 1 : 0;
    // GQA Q-head packing: a Q tile holds 128 / G positions of all G heads of
    // a KV group, so one K/V tile staged in shared memory serves every head
    // of the group, and short query lengths still fill the tile's 128 rows.
    // Possible when G divides 128 (dense launches; the packed-batch entry
    // points turn it off).  Used when it pads fewer rows than head pairing:
    // a unit then covers 2 * 128 / G positions instead of 128 (or 256).  On
    // long sequences, where neither pads, the two measure the same within
    // half a percent (pairing ahead), so a tie keeps pairing.
    {
        const bool can_pack = p->G >= 2 && 128 % p->G == 0;
        const int span_pack = can_pack ? 2 * (128 / p->G) : 0;
        const int span_pair = p->pair_heads ? 128 : 256;
        const int64_t pad_pack = can_pack ? (int64_t)span_pack * ((Sq + span_pack - 1) / span_pack) - Sq : 0;
        const int64_t pad_pair = (int64_t)span_pair * ((Sq + span_pair - 1) / span_pair) - Sq;
        p->pack_heads = (can_pack && pad_pack < pad_pair) ? 1 : 0;
    }
    p->pack_pos = p->pack_heads ? 128 / p->G : 0;
    p->n_pk = p->pack_heads ? (Sq + 2 * p->pack_pos - 1) / (2 * p->pack_pos) : 0;
    p->status = di->status;
    p->budget_ns = budget();
    p->inject = 0;
    p->round_mode = ATTN_ROUND_RTNE;
    p->n_full_units = attn::prefill_num_units(*p);
    p->n_items = p->n_full_units;
    p->sched = next_sched(di);
    // Non-causal units all have the same length, so ordering them by batch and
    // KV head costs no balance; it keeps the units that read the same K/V
    // together, which pays once the K/V of all heads exceed L2.
    p->kv_major = (!causal && (double)B * Hkv * Sk * 128 * 4 > 64.0 * (1 << 20)) ? 1 : 0;
    p->seq_group = 0;
    // L2 prefetch of the next wave's Q for short non-causal units (few K/V tiles).
    p->prefetch_ahead = (!causal && Sk <= 1024) ? di->sm_count : 0;
    p->split_units = 0;
    p->split_parts = 1;
    p->ws_o = nullptr;
    p->ws_lse = nullptr;
    p->cu_q = nullptr;
    p->cu_k = nullptr;
    p->total_q = 0;
    p->total_k = 0;
    p->out = nullptr;
    p->block_table = nullptr;
    p->seqlens_k = nullptr;
    p->max_blocks = 0;
    p->num_pages = 0;
    return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_fwd_rounded(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq,
                               int Hkv, int Sq, int Sk, int d, int layout, int causal, float scale, int round_mode,
                               void *stream) {
    attn_status_t st = check_fwd_args(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, d, layout, scale);
    if (st != ATTN_OK) return st;
    if (!valid_round_mode(round_mode)) return ATTN_ERR_INVALID_ARG;
    DeviceInfo *di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    attn::PrefillParams p;
    fill_prefill_params(&p, di, lse, B, Hq, Hkv, Sq, Sk, layout, causal, scale);
    p.round_mode = round_mode;
    p.inject = g_inject.exchange(0);
    const bool bhsd = p.bhsd != 0;
    // Q and O boxes: one head x 128 positions, or with head packing the
    // group's G heads x 128 / G positions.
    const int q_rows = p.pack_heads ? p.pack_pos : 128, q_heads = p.pack_heads ? p.G : 1;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map_4d(&mq, q, bhsd, B, Sq, Hq, d, q_rows, q_heads) || !make_map_4d(&mk, k, bhsd, B, Sk, Hkv, d, 128) ||
        !make_map_4d(&mv, v, bhsd, B, Sk, Hkv, d, 128) || !make_map_4d(&mo, out, bhsd, B, Sq, Hq, d, q_rows, q_heads))
        return ATTN_ERR_CUDA;
    const int units = attn::prefill_num_units(p);
    int ctas = units;
    {
        // Tail split, when the shape calls for one and the caller has set a
        // large enough workspace on this device; otherwise whole units only.
        int su = 0, parts = 1;
        const size_t need = attn::prefill_split_plan(p, di->sm_count, &su, &parts);
        std::lock_guard<std::mutex> lock(g_mu);
        if (su > 0 && di->workspace != nullptr && di->workspace_bytes >= need) {
            const size_t rows = (size_t)su * 256;
            size_t o_bytes = rows * parts * 128 * 4;
            o_bytes = (o_bytes + 255) & ~(size_t)255;
            p.n_full_units = units - su;
            p.split_units = su;
            p.split_parts = parts;
            p.ws_o = static_cast<float *>(di->workspace);
            p.ws_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(di->workspace) + o_bytes);
            ctas = p.n_full_units + su * parts;
        }
    }
    p.n_items = ctas;
    if (attn::launch_prefill(mq, mk, mv, mo, mk, mv, p, attn::prefill_grid(p.n_items, di->sm_count),
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (attn::launch_prefill_merge(out, p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq, int Hkv,
                       int Sq, int Sk, int d, int layout, int causal, float scale, void *stream) {
    return attn_fwd_rounded(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, d, layout, causal, scale, ATTN_ROUND_RTNE,
                            stream);
}

attn_status_t attn_fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int B, int Hq, int Hkv,
                              int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d, int causal,
                              float scale, int round_mode, void *stream) {
    if (!cu_seqlens_q || !cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
        return ATTN_ERR_INVALID_ARG;
    // The packed tensors are checked as one dense [1][total][H][d] batch.
    attn_status_t st = check_fwd_args(q, k, v, out, lse, 1, Hq, Hkv, total_q, total_k, d, ATTN_LAYOUT_BSHD, scale);
    if (st != ATTN_OK) return st;
    if (B < 1 || max_seqlen_q < 1 || max_seqlen_k < 1 || max_seqlen_q > total_q || max_seqlen_k > total_k)
        return ATTN_ERR_INVALID_ARG;
    if (!valid_round_mode(round_mode)) return ATTN_ERR_INVALID_ARG;
    DeviceInfo *di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    attn::PrefillParams p;
    fill_prefill_params(&p, di, lse, B, Hq, Hkv, max_seqlen_q, max_seqlen_k, ATTN_LAYOUT_BSHD, causal, scale);
    p.round_mode = round_mode;
    p.cu_q = cu_seqlens_q;
    p.prefetch_ahead = 0;  // (dense coordinates only)
    p.pack_heads = 0;      // (dense launches only)
    p.cu_k = cu_seqlens_k;
    // Keys much longer than queries (chunks against a context): K/V-first order.
    p.kv_major = max_seqlen_k >= 2 * max_seqlen_q ? 1 : 0;
    // Self-attention batches: sequences in groups of about 160 MB of K/V at
    // the longest length, row block first within a group (the causal balance
    // of row block first, with the K/V of only a few sequences in use at
    // once).  On the 16-sequence workload: groups of 5 run 4% faster than one
    // group of all 16 and move 1.49 GB from DRAM instead of 5.65 GB (floor
    // 1.41 GB); groups of 3 and of 1 gave 1.41 and 1.36 GB at +3% and -1.5%.
    if (!p.kv_major) {
        const double kv_seq = (double)max_seqlen_k * Hkv * 128 * 2 * 2;
        const int grp = (int)(160.0 * (1 << 20) / kv_seq);
        p.seq_group = grp < 1 ? 1 : (grp >= B ? 0 : grp);
    }
    p.total_q = total_q;
    p.total_k = total_k;
    p.out = out;
    p.inject = g_inject.exchange(0);
    const int64_t units = p.pair_heads ? (int64_t)B * Hkv * (p.G / 2) * p.n_m : (int64_t)B * Hq * ((p.n_m + 1) / 2);
    if (units > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
    p.n_full_units = (int)units;
    p.n_items = (int)units;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map_4d(&mq, q, false, 1, total_q, Hq, d, 128) || !make_map_4d(&mk, k, false, 1, total_k, Hkv, d, 128) ||
        !make_map_4d(&mv, v, false, 1, total_k, Hkv, d, 128) || !make_map_4d(&mo, out, false, 1, total_q, Hq, d, 128))
        return ATTN_ERR_CUDA;
    if (attn::launch_prefill(mq, mk, mv, mo, mk, mv, p, attn::prefill_grid(p.n_items, di->sm_count),
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status_t attn_fwd_paged(const void *q, const void *k_pages, const void *v_pages, const int32_t *block_table,
                             const int32_t *seqlens_k, const int32_t *cu_seqlens_q, void *out, float *lse, int B,
                             int Hq, int Hkv, int total_q, int max_seqlen_q, int d, int page_size, int num_pages,
                             int max_blocks_per_seq, int causal, float scale, int round_mode, void *stream) {
    if (!block_table || !seqlens_k || !cu_seqlens_q) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seqlens_k) & 3u) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u))
        return ATTN_ERR_INVALID_ARG;
    if (num_pages < 1 || max_blocks_per_seq < 1 || (int64_t)num_pages * 16 > 0x7fffffff ||
        (int64_t)max_blocks_per_seq * 16 > 0x7fffffff)
        return ATTN_ERR_INVALID_ARG;
    // q, out: one dense [1][total_q][Hq][d] batch; the pools as [1][16P][Hkv][d].
    attn_status_t st = check_fwd_args(q, k_pages, v_pages, out, lse, 1, Hq, Hkv, total_q, num_pages * 16, d,
                                      ATTN_LAYOUT_BSHD, scale);
    if (st != ATTN_OK) return st;
    if (page_size != 16) return ATTN_ERR_UNSUPPORTED;
    if (B < 1 || max_seqlen_q < 1 || max_seqlen_q > total_q) return ATTN_ERR_INVALID_ARG;
    if (!valid_round_mode(round_mode)) return ATTN_ERR_INVALID_ARG;
    DeviceInfo *di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    attn::PrefillParams p;
    fill_prefill_params(&p, di, lse, B, Hq, Hkv, max_seqlen_q, max_blocks_per_seq * 16, ATTN_LAYOUT_BSHD, causal,
                        scale);
    p.round_mode = round_mode;
    p.cu_q = cu_seqlens_q;
    p.prefetch_ahead = 0;  // (dense coordinates only)
    p.pack_heads = 0;      // (dense launches only)
    p.total_q = total_q;
    p.out = out;
    p.block_table = block_table;
    p.kv_major = 1;  // chunks against a cache: K/V-first order
    p.seqlens_k = seqlens_k;
    p.max_blocks = max_blocks_per_seq;
    p.num_pages = num_pages;
    p.inject = g_inject.exchange(0);
    const int64_t units = p.pair_heads ? (int64_t)B * Hkv * (p.G / 2) * p.n_m : (int64_t)B * Hq * ((p.n_m + 1) / 2);
    if (units > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
    p.n_full_units = (int)units;
    p.n_items = (int)units;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map_4d(&mq, q, false, 1, total_q, Hq, d, 128) || !make_map_pool_groups(&mk, k_pages, num_pages, Hkv, d, 2) ||
        !make_map_pool_groups(&mv, v_pages, num_pages, Hkv, d, 2) || !make_map_4d(&mo, out, false, 1, total_q, Hq, d, 128))
        return ATTN_ERR_CUDA;
    CUtensorMap mk8, mv8;
    if (!make_map_pool_groups(&mk8, k_pages, num_pages, Hkv, d, 16) ||
        !make_map_pool_groups(&mv8, v_pages, num_pages, Hkv, d, 16))
        return ATTN_ERR_CUDA;
    if (attn::launch_prefill(mq, mk, mv, mo, mk8, mv8, p, attn::prefill_grid(p.n_items, di->sm_count),
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

size_t attn_fwd_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || d != 128 || Hq % Hkv != 0) return 0;
    DeviceInfo *di = nullptr;
    if (device_info(&di) != ATTN_OK) return 0;
    attn::PrefillParams p;
    fill_prefill_params(&p, di, nullptr, B, Hq, Hkv, Sq, Sk, ATTN_LAYOUT_BSHD, causal, 1.0f);
    int su = 0, parts = 1;
    return attn::prefill_split_plan(p, di->sm_count, &su, &parts);
}

attn_status_t attn_set_workspace(void *ptr, size_t bytes) {
    if (ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & 255u)) return ATTN_ERR_INVALID_ARG;
    DeviceInfo *di = nullptr;
    attn_status_t st = device_info(&di);
    if (st != ATTN_OK) return st;
    std::lock_guard<std::mutex> lock(g_mu);
    di->workspace = ptr;
    di->workspace_bytes = ptr != nullptr ? bytes : 0;
    return ATTN_OK;
}

attn_status_t attn_fwd_simple(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq,
                              int Hkv, int Sq, int Sk, int d, int layout, int causal, float scale, void *stream) {
    attn_status_t st = check_fwd_args(q, k, v, out, lse, B, Hq, Hkv, Sq, Sk, d, layout, scale);
    if (st != ATTN_OK) return st;
    DeviceInfo *di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    if (B > 65535 || Hq > 65535) return ATTN_ERR_INVALID_ARG;
    attn::PrefillParams p;
    fill_prefill_params(&p, di, lse, B, Hq, Hkv, Sq, Sk, layout, causal, scale);
    if (attn::launch_prefill_simple(q, k, v, out, lse, p, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

size_t attn_decode_workspace_bytes(int B, int Hq, int d, int max_blocks_per_seq) {
    if (B < 1 || Hq < 1 || d != 128 || max_blocks_per_seq < 1) return 0;
    int ns = 1, pps = 1;
    attn::decode_split_plan(B, Hq, max_blocks_per_seq, &ns, &pps);
    const size_t nsplit = (size_t)ns;
    const size_t rows = (size_t)B * Hq;
    // o_part [rows][nsplit][d] fp32, then lse_part [rows][nsplit] fp32, each 256-B aligned.
    size_t o_bytes = rows * nsplit * d * 4;
    o_bytes = (o_bytes + 255) & ~(size_t)255;
    size_t l_bytes = rows * nsplit * 4;
    l_bytes = (l_bytes + 255) & ~(size_t)255;
    return o_bytes + l_bytes;
}

}  // extern "C"

namespace attn {

// The argument checks of a decode step other than its workspace (pointers,
// alignment, shapes, scale), shared by the entry points that take a
// workspace and the one that does not.
attn_status_t check_decode_args(const void *q, const void *k_pages, const void *v_pages, const int32_t *block_table,
                                const int32_t *seqlens, const void *out, const float *lse, int B, int Hq, int Hkv,
                                int d, int page_size, int num_pages, int max_blocks_per_seq, float scale) {
    if (!q || !k_pages || !v_pages || !block_table || !seqlens || !out) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out)) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seqlens) & 3u))
        return ATTN_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || num_pages < 1 || max_blocks_per_seq < 1) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || B > 65535) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
    if (d != 128 || page_size != 16) return ATTN_ERR_UNSUPPORTED;
    if ((int64_t)num_pages * 16 > ((int64_t)1 << 31) - 1) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

}  // namespace attn

extern "C" {

static attn_status_t decode_impl(const void *q, const void *k_new, const void *v_new, const void *k_pages,
                                 const void *v_pages, const int32_t *block_table, const int32_t *seqlens, void *out,
                                 float *lse, int B, int Hq, int Hkv, int d, int page_size, int num_pages,
                                 int max_blocks_per_seq, float scale, void *workspace, size_t workspace_bytes,
                                 void *stream) {
    attn_status_t st = attn::check_decode_args(q, k_pages, v_pages, block_table, seqlens, out, lse, B, Hq, Hkv, d,
                                               page_size, num_pages, max_blocks_per_seq, scale);
    if (st != ATTN_OK) return st;
    const size_t need = attn_decode_workspace_bytes(B, Hq, d, max_blocks_per_seq);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return ATTN_ERR_WORKSPACE;
    DeviceInfo *di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    CUtensorMap mk, mv;
    // One box per page and tensor: two 8-row groups, the layout the decode's
    // ldmatrix reads expect.
    if (!make_map_pool_groups(&mk, k_pages, num_pages, Hkv, d, 2) ||
        !make_map_pool_groups(&mv, v_pages, num_pages, Hkv, d, 2))
        return ATTN_ERR_CUDA;
    attn::DecodeParams p;
    p.q = q;
    p.block_table = block_table;
    p.seqlens = seqlens;
    p.out = out;
    p.lse = lse;
    attn::decode_split_plan(B, Hq, max_blocks_per_seq, &p.nsplit, &p.pages_per_split);
    const size_t rows = (size_t)B * Hq;
    size_t o_bytes = rows * p.nsplit * d * 4;
    o_bytes = (o_bytes + 255) & ~(size_t)255;
    p.o_part = static_cast<float *>(workspace);
    p.lse_part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + o_bytes);
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.num_pages = num_pages;
    p.max_blocks = max_blocks_per_seq;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.status = di->status;
    p.budget_ns = budget();
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_pool = const_cast<void *>(k_pages);
    p.v_pool = const_cast<void *>(v_pages);
    if (attn::launch_decode(mk, mv, p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status_t attn_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                                const int32_t *block_table, const int32_t *seqlens, void *out, float *lse, int B,
                                int Hq, int Hkv, int d, int page_size, int num_pages, int max_blocks_per_seq,
                                float scale, void *workspace, size_t workspace_bytes, void *stream) {
    return decode_impl(q, nullptr, nullptr, k_pages, v_pages, block_table, seqlens, out, lse, B, Hq, Hkv, d,
                       page_size, num_pages, max_blocks_per_seq, scale, workspace, workspace_bytes, stream);
}

attn_status_t attn_decode_paged_append(const void *q, const void *k_new, const void *v_new, void *k_pages,
                                       void *v_pages, const int32_t *block_table, const int32_t *seqlens, void *out,
                                       float *lse, int B, int Hq, int Hkv, int d, int page_size, int num_pages,
                                       int max_blocks_per_seq, float scale, void *workspace, size_t workspace_bytes,
                                       void *stream) {
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return ATTN_ERR_INVALID_ARG;
    return decode_impl(q, k_new, v_new, k_pages, v_pages, block_table, seqlens, out, lse, B, Hq, Hkv, d, page_size,
                       num_pages, max_blocks_per_seq, scale, workspace, workspace_bytes, stream);
}

attn_status_t attn_lse_merge(const float *o_parts, const float *lse_parts, void *out, float *lse, int rows,
                             int nsplit, int d, int round_mode, void *stream) {
    if (!o_parts || !lse_parts || !out) return ATTN_ERR_INVALID_ARG;
    if (!valid_round_mode(round_mode)) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(o_parts) & 3u) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
        !aligned16(out) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return ATTN_ERR_INVALID_ARG;
    if (rows < 1 || nsplit < 1) return ATTN_ERR_INVALID_ARG;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    attn_status_t st;
    DeviceInfo *di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    if (attn::launch_lse_merge(o_parts, lse_parts, out, lse, rows, nsplit, round_mode,
                               static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

attn_status_t attn_get_device_status(void *stream, int *site) {
    DeviceInfo *di = nullptr;
    attn_status_t st = device_info(&di);
    if (st != ATTN_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned h[2] = {0, 0};
    if (cudaMemcpy(h, di->status, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    if (h[0] != 0 && cudaMemset(di->status, 0, sizeof h) != cudaSuccess) return ATTN_ERR_CUDA;
    if (site) *site = (int)h[1];
    return static_cast<attn_status_t>(h[0]);
}

attn_status_t attn_set_wait_budget_ns(uint64_t ns) {
    g_budget.store(ns == 0 ? kDefaultBudgetNs : ns, std::memory_order_relaxed);
    return ATTN_OK;
}

attn_status_t attn_debug_inject(int mode) {
    if (mode < 0 || mode > 1) return ATTN_ERR_INVALID_ARG;
    g_inject.store(mode);
    return ATTN_OK;
}

attn_status_t attn_selftest_umma(const void *a, const void *b, float *c, int mode, void *stream) {
    if (!a || !b || !c || !aligned16(a) || !aligned16(b) || !aligned16(c)) return ATTN_ERR_INVALID_ARG;
    if (mode != 0 && mode != 1) return ATTN_ERR_INVALID_ARG;
    attn_status_t st;
    DeviceInfo *di = nullptr;
    if ((st = device_info(&di)) != ATTN_OK) return st;
    CUtensorMap ma, mb;
    // Treat each [128][128] matrix as a one-head BSHD tensor with 128 rows.
    if (!make_map_4d(&ma, a, false, 1, 128, 1, 128, 128) || !make_map_4d(&mb, b, false, 1, 128, 1, 128, 128))
        return ATTN_ERR_CUDA;
    if (attn::launch_selftest_umma(ma, mb, a, c, mode, di->status, budget(), static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

const char *attn_status_string(attn_status_t s) {
    switch (s) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
        case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
        case ATTN_ERR_DEVICE_BOUNDS: return "ATTN_ERR_DEVICE_BOUNDS";
    }
    return "ATTN_ERR_UNKNOWN";
}

int attn_version(void) { return 100; }

}  // extern "C"
