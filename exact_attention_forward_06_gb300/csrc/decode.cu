// decode.cu -- paged-KV decode split over the keys, and the log-sum-exp merge.
//
// The cache is the paged layout of the ROCm port page ("Vendor-Agnostic 多查询
// 推理优化": 16-token pages, an int32 block_table per sequence); the split over
// the keys with a merge of the partial results is the Flash-Decoding style
// tail split of the MoonMath HIP kernel page.  Decode reads every K/V byte
// once and does ~4 flops per byte, so it is bound by HBM bandwidth.
//
// Split kernel: one CTA per (group of up to 4 query heads sharing a KV head,
// split, sequence); when a KV group has more heads, its head groups are
// adjacent in the grid so that their reads of the same pages meet in L2.  The
// CTAs are small (one producer warp and four consumer warps) so three of them
// share an SM.  The producer lane gathers the split's pages with one TMA box
// per page and tensor into an 8-page shared-memory ring.  A box is the page's
// 16 rows of one KV head in two 8-row groups, each as two 64-column halves of
// 128-byte rows with the 128-byte swizzle (the layout of the paged prefill's
// tiles), so that 8 consecutive rows at one column chunk sit in 8 distinct
// bank groups.
//
// Consumer warp w takes pages w, w + 4, ...: four page streams.  A page is two
// warp-level tensor-core products (mma.sync m16n8k16, bf16 in, fp32 out), the
// 16 tokens of the page as M:
//   S^T = K Q^T   (16 tokens x 8 head columns, k = the 128 head-dim elements;
//                  K straight from shared memory with ldmatrix, Q^T held in
//                  registers, columns past the CTA's heads zero),
//   O^T += V^T P^T (8 m-tiles of 16 head-dim elements x 8 head columns,
//                  k = the 16 tokens; V^T by transposing ldmatrix).
// A lane's fragment columns are the same two heads in both products, so the
// online softmax (running max, rescale, row sum) needs no data movement
// beyond the max over the page's tokens; P goes from the S^T fragment to the
// B operand of the second product with one 8x8 transpose (movmatrix) per
// 8 tokens.  Measured on 32 sequences of 1024 to 8192 tokens (Hq=32,
// Hkv=8), the same loop with the page math left out runs at 0.91 of the copy
// bandwidth, and the earlier CUDA-core form (bf16 -> fp32 unpacking and
// packed FMAs) at 0.78: the unpacking, not the memory system, held decode
// below the roofline.
//
// P is rounded to bf16 for the second product (as in the prefill).  The
// running max is raised whenever a page's max exceeds it, so the largest key
// of a row has P = 1 exactly and a dominant key keeps its weight.  At the end
// the page streams are merged in shared memory and the split writes its
// normalised partial output and log-sum-exp; the merge kernel then combines
// the splits in a fixed order.
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "prefill_tc.h"

namespace attn {
namespace dec {

constexpr int PAGE = 16;
constexpr int D = 128;
constexpr int NCW = 4;   // consumer warps = page streams
constexpr int NST = 8;   // pages in flight per CTA
// Page i goes to slot i % NST and to consumer warp i % NCW.  With NST a
// multiple of NCW every slot has one consumer warp, which waits on the slot's
// phases in order; otherwise a warp could wait on parity r of a slot whose
// phase r - 1 is still open, and a parity wait on the phase two back returns
// at once.
static_assert(NST % NCW == 0, "each ring slot must have a single consumer warp");
constexpr int GH_MAX = 4;
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr uint32_t PAGE_BYTES = PAGE * D * 2;        // one tensor, one KV head: 4 KiB
constexpr uint32_t STAGE_BYTES = 2 * PAGE_BYTES;     // K + V
constexpr uint32_t SMEM_STAGES = NST * STAGE_BYTES;  // 64 KiB
// Page box layout: row r, 16-byte chunk c (of 16) at
// (r / 8) * GROUP_BYTES + (c / 8) * HALF_BYTES + (r % 8) * 128 + ((c % 8) ^ (r % 8)) * 16.
constexpr uint32_t GROUP_BYTES = 2048;
constexpr uint32_t HALF_BYTES = 1024;
constexpr uint32_t SMEM_MERGE = NCW * GH_MAX * (D + 2) * 4;
constexpr uint32_t SMEM_MISC = 1536;
constexpr uint32_t SMEM_ALIGN = 1024;  // the 128-byte swizzle repeats every 1 KiB
constexpr uint32_t SMEM_BYTES = SMEM_ALIGN + SMEM_STAGES + SMEM_MERGE + SMEM_MISC;
constexpr int MAX_PAGES_PER_SPLIT = 256;
constexpr int TARGET_SPLIT_CTAS = 2048;  // split CTAs the plan aims for (assuming four heads per CTA)
// barriers, per-stage flags, the abort flag and the split's page ids
static_assert(2 * NST * 8 + (NST + 4 + MAX_PAGES_PER_SPLIT) * 4 <= SMEM_MISC, "misc shared area too small");
static_assert(3 * (SMEM_BYTES + 1024) <= 233472, "three CTAs must share an SM");
constexpr float LN2 = 0.6931471805599453f;
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// GH query heads per CTA (1, 2 or 4, all of one KV head): head columns
// 0 .. GH-1 of the 8-wide MMA tiles.
template <int GH>
__global__ void __launch_bounds__(NTHREADS, 3)
    split_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                 const DecodeParams p) {
    static_assert(GH >= 1 && GH <= GH_MAX, "heads per CTA");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    uint8_t *base = smem_raw + ((SMEM_ALIGN - (raw & (SMEM_ALIGN - 1))) & (SMEM_ALIGN - 1));
    float *merge = reinterpret_cast<float *>(base + SMEM_STAGES);
    uint64_t *full = reinterpret_cast<uint64_t *>(base + SMEM_STAGES + SMEM_MERGE);
    uint64_t *empty = full + NST;
    int *stage_bad = reinterpret_cast<int *>(empty + NST);
    volatile int *abort_flag = stage_bad + NST;
    int *split_pages = stage_bad + NST + 4;  // physical page ids of this split (<= MAX_PAGES_PER_SPLIT)

    const int split = blockIdx.y;
    const int h0 = blockIdx.x * GH;
    const int b = blockIdx.z;
    const int g = h0 / p.G;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int L_raw = p.seqlens[b];
    // A length outside [0, 16 * max_blocks] is reported, and the sequence is
    // skipped: its rows get O = 0 and lse = -inf, and nothing is appended.
    const bool bad_len = L_raw < 0 || L_raw > p.max_blocks * PAGE;
    if (bad_len && threadIdx.x == 0 && split == 0 && blockIdx.x == 0)
        report_status(p.status, kStatusDeviceBounds, kSiteDecodeSeqlen);
    const int L = bad_len ? 0 : L_raw;
    const int npages = (L + PAGE - 1) / PAGE;
    const int page0 = split * p.pages_per_split;
    const int np = max(0, min(p.pages_per_split, npages - page0));
    const int64_t row0 = (int64_t)b * p.Hq + h0;  // first (b, h) row of this CTA
    // With a fused append, split 0 also attends to the new token (position L).
    const bool new_token = p.k_new != nullptr && split == 0 && !bad_len;
    // The producer warp starts the split's block-table reads at once, for the
    // entries of the split that lie within the table row, so that their
    // latency overlaps the length check and the set-up; the first np of
    // them are used.
    constexpr int TAB = MAX_PAGES_PER_SPLIT / 32;
    int tab[TAB];
    if (warp == NCW) {
        const int lim = min(p.pages_per_split, p.max_blocks - page0);
        const int32_t *row = p.block_table + (int64_t)b * p.max_blocks + page0;
#pragma unroll
        for (int q = 0; q < TAB; ++q) tab[q] = lane + 32 * q < lim ? row[lane + 32 * q] : -1;
    }

    if (np == 0 && !new_token) {  // nothing to attend to in this split
        for (int i = threadIdx.x; i < GH * D; i += NTHREADS)
            p.o_part[((row0 + i / D) * p.nsplit + split) * D + (i % D)] = 0.f;
        if (threadIdx.x < GH) p.lse_part[(row0 + threadIdx.x) * p.nsplit + split] = -INFINITY;
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            ptx::mbar_init(full + s, 1);
            ptx::mbar_init(empty + s, 1);
            stage_bad[s] = 0;
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const WaitCtx wc{abort_flag, p.status, p.budget_ns};

    if (warp == NCW) {
        // ---------------- producer
        // The whole warp puts the split's block-table entries (read at entry)
        // into shared memory, so the copy-issuing lane never waits on a
        // global load per page.
#pragma unroll
        for (int q = 0; q < TAB; ++q)
            if (lane + 32 * q < np) split_pages[lane + 32 * q] = tab[q];
        if (new_token && h0 % p.G == 0) {
            // Fused append: one CTA per (sequence, KV head) writes the new
            // token's K and V rows (256 B each) into slot L % 16 of page
            // block_table[b][L / 16].  Another split may be reading that page
            // right now, but position L lies past the L keys it attends to, so
            // whichever value it reads there is masked out.
            const int64_t slot_page = L_raw >= 0 && L_raw < p.max_blocks * PAGE
                                          ? p.block_table[(int64_t)b * p.max_blocks + L_raw / PAGE]
                                          : -1;
            if (slot_page < 0 || slot_page >= p.num_pages) {
                if (lane == 0) report_status(p.status, kStatusDeviceBounds, kSiteAppendSlot);
            } else {
                const int64_t off = ((slot_page * PAGE + L_raw % PAGE) * p.Hkv + g) * D;
                const int64_t src = ((int64_t)b * p.Hkv + g) * D;
                const bool is_v = lane >= 16;
                const uint4 *from = reinterpret_cast<const uint4 *>(
                    static_cast<const __nv_bfloat16 *>(is_v ? p.v_new : p.k_new) + src);
                uint4 *to = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(is_v ? p.v_pool : p.k_pool) + off);
                to[lane & 15] = from[lane & 15];
            }
        }
        __syncwarp();
        if (lane == 0) {
            ptx::prefetch_tensormap(&map_k);
            ptx::prefetch_tensormap(&map_v);
            // Each cache page is read once per step: evict-first keeps the
            // stream from pushing other work's data out of L2.
            const uint64_t pol = ptx::policy_evict_first();
            int issued = 0;
            for (int i = 0; i < np; ++i) {
                const int slot = i % NST;
                const int round = i / NST;
                if (round > 0 && !wait_bounded(empty + slot, (round - 1) & 1, wc, kSiteDecodeEmpty)) break;
                const int phys = split_pages[i];
                uint8_t *dst = base + slot * STAGE_BYTES;
                if (phys < 0 || phys >= p.num_pages) {
                    report_status(p.status, kStatusDeviceBounds, kSiteDecodeTable);
                    stage_bad[slot] = 1;
                    ptx::mbar_arrive(full + slot);
                } else {
                    stage_bad[slot] = 0;
                    // one box per tensor: 8-row groups 2 phys and 2 phys + 1 of KV head g
                    ptx::mbar_arrive_expect_tx(full + slot, STAGE_BYTES);
                    ptx::tma_load_5d_hint(dst, &map_k, full + slot, 0, 0, 0, phys * 2, g, pol);
                    ptx::tma_load_5d_hint(dst + PAGE_BYTES, &map_v, full + slot, 0, 0, 0, phys * 2, g, pol);
                }
                ++issued;
            }
            for (int i = max(0, issued - NST); i < issued; ++i) drain_wait(full + i % NST, (i / NST) & 1, wc);
        }
        __syncwarp();
    } else {
        // ---------------- consumers: warp w takes pages w, w + NCW, ...
        // Fragment coordinates: r4 is the row group (a token of S^T, a
        // head-dim row of O^T), c4 the column pair (heads 2 c4 and 2 c4 + 1).
        const int r4 = lane >> 2;
        const int c4 = lane & 3;
        // ldmatrix row addresses: lanes 8 i .. 8 i + 7 give the 8 rows of
        // matrix i.  K (S^T's A operand, 16 tokens x 16 head-dim elements per
        // k step): matrix i is tokens 8 (i & 1) .., chunk 2 ks + (i >> 1).
        // V (O^T's A operand through the transpose, 16 head-dim elements x 16
        // tokens per m-tile): matrix i is tokens 8 (i >> 1) .., chunk
        // 2 mt + (i & 1).  Row rr = lane % 8 of a matrix is token rr of its
        // 8-row group, so its swizzle phase is rr.
        const int mat = lane >> 3, rr = lane & 7;
        const uint32_t k_row = (uint32_t)(mat & 1) * GROUP_BYTES + rr * 128;
        const uint32_t k_x = (uint32_t)((mat >> 1) ^ rr);
        const uint32_t v_row = (uint32_t)(mat >> 1) * GROUP_BYTES + rr * 128;
        const uint32_t v_x = (uint32_t)((mat & 1) ^ rr);
        // Q^T as the B operand: head r4 (zero past the CTA's heads), head-dim
        // elements 16 ks + 2 c4 (+1) and 16 ks + 8 + 2 c4 (+1).
        uint32_t qb[8][2];
        {
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(p.q) + (row0 + r4) * (D / 2);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qb[ks][0] = r4 < GH ? qrow[ks * 8 + c4] : 0u;
                qb[ks][1] = r4 < GH ? qrow[ks * 8 + 4 + c4] : 0u;
            }
        }
        const float sl2 = p.scale_log2;
        // Running max (log2 units) and partial row sum of heads 2 c4, 2 c4 + 1,
        // and O^T: acc[mt] = rows 16 mt + r4 and 16 mt + r4 + 8, those heads.
        float m[2] = {-INFINITY, -INFINITY};
        float lsum[2] = {0.f, 0.f};
        float acc[8][4];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

        // Raise the running max of the lane's heads to mn0 / mn1 when any lane
        // of the warp needs it (so the branch is uniform), rescaling the sums.
        auto raise_max = [&](float mn0, float mn1) {
            if (__any_sync(0xffffffffu, mn0 > m[0] || mn1 > m[1])) {
                const float a0 = mn0 == -INFINITY ? 1.f : ptx::ex2(m[0] - mn0);  // m = -inf: 0
                const float a1 = mn1 == -INFINITY ? 1.f : ptx::ex2(m[1] - mn1);
                lsum[0] *= a0;
                lsum[1] *= a1;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    acc[mt][0] *= a0;
                    acc[mt][1] *= a1;
                    acc[mt][2] *= a0;
                    acc[mt][3] *= a1;
                }
                m[0] = mn0;
                m[1] = mn1;
            }
        };

        for (int i = warp; i < np; i += NCW) {
            const int slot = i % NST;
            if (!wait_bounded(full + slot, (i / NST) & 1, wc, kSiteDecodeFull)) break;
            // A page whose block-table entry could not be read holds nothing of
            // the sequence: it is skipped.
            if (stage_bad[slot] == 0) {
                const uint32_t ks_addr = ptx::smem_addr(base + slot * STAGE_BYTES);
                const uint32_t vs_addr = ks_addr + PAGE_BYTES;
                const int nvalid = L - (page0 + i) * PAGE;  // tokens of the sequence in this page (>= 1)
                // A page whose 16 slots all hold keys of the sequence needs no
                // masking: it takes a copy of the page step without the selects.
                auto page_step = [&](auto full_tag) {
                    constexpr bool FULL = decltype(full_tag)::value;
                    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        uint32_t a[4];
                        ptx::ldsm_x4(ks_addr + k_row + (ks >> 2) * HALF_BYTES + (((2u * (ks & 3)) ^ k_x) << 4), a);
                        ptx::mma_bf16_16816(s, a, qb[ks][0], qb[ks][1]);
                    }
                    // s[0], s[1]: token r4, heads 2 c4, 2 c4 + 1; s[2], s[3]: token r4 + 8.
#pragma unroll
                    for (int j = 0; j < 4; ++j) s[j] *= sl2;
                    if (!FULL) {
                        // Slots past the sequence end hold arbitrary bits: select, not add.
                        if (r4 >= nvalid) s[0] = s[1] = -INFINITY;
                        if (r4 + 8 >= nvalid) s[2] = s[3] = -INFINITY;
                    }
                    float pm0 = fmaxf(s[0], s[2]), pm1 = fmaxf(s[1], s[3]);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, off));
                        pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, off));
                    }
                    raise_max(fmaxf(m[0], pm0), fmaxf(m[1], pm1));
                    const float ms0 = m[0] == -INFINITY ? 0.f : m[0];
                    const float ms1 = m[1] == -INFINITY ? 0.f : m[1];
                    // P rounded to bf16 for the product only; the row sum (and
                    // with it the log-sum-exp) adds the fp32 values.
                    const float p0 = ptx::ex2(s[0] - ms0), p1 = ptx::ex2(s[1] - ms1);
                    const float p2 = ptx::ex2(s[2] - ms0), p3 = ptx::ex2(s[3] - ms1);
                    lsum[0] += p0 + p2;
                    lsum[1] += p1 + p3;
                    const uint32_t p_lo = ptx::pack_bf16x2(p0, p1);
                    const uint32_t p_hi = ptx::pack_bf16x2(p2, p3);
                    // P^T as the B operand: tokens 2 c4 (+1) and 8 + 2 c4 (+1), head r4.
                    const uint32_t pb0 = ptx::movmatrix_trans(p_lo);
                    const uint32_t pb1 = ptx::movmatrix_trans(p_hi);
                    // The V^T fragment holds tokens 2 c4, 2 c4 + 1 (a[0], a[1]) and
                    // those + 8 (a[2], a[3]); past the end P is 0 but 0 * NaN is
                    // NaN, so there V is zeroed.
                    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
                    if (!FULL) {
                        keep_lo = (2 * c4 < nvalid ? 0x0000ffffu : 0u) | (2 * c4 + 1 < nvalid ? 0xffff0000u : 0u);
                        keep_hi = (2 * c4 + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * c4 + 9 < nvalid ? 0xffff0000u : 0u);
                    }
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        uint32_t a[4];
                        ptx::ldsm_x4_trans(vs_addr + v_row + (mt >> 2) * HALF_BYTES + (((2u * (mt & 3)) ^ v_x) << 4),
                                           a);
                        if (!FULL) {
                            a[0] &= keep_lo;
                            a[1] &= keep_lo;
                            a[2] &= keep_hi;
                            a[3] &= keep_hi;
                        }
                        ptx::mma_bf16_16816(acc[mt], a, pb0, pb1);
                    }
                };
                if (nvalid >= PAGE)
                    page_step(std::true_type{});
                else
                    page_step(std::false_type{});
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty + slot);
        }
        if (new_token && warp == 0) {
            // The appended token, read from k_new / v_new rather than the
            // cache.  Lane l forms the partial dot products of head-dim
            // elements 4 l .. 4 l + 3 for every head, reduced over the warp;
            // the token is added to the sums once (by the lanes of row group 0).
            const int64_t src = ((int64_t)b * p.Hkv + g) * D;
            const __nv_bfloat16 *kn = static_cast<const __nv_bfloat16 *>(p.k_new) + src;
            const __nv_bfloat16 *vn = static_cast<const __nv_bfloat16 *>(p.v_new) + src;
            const uint2 ku = reinterpret_cast<const uint2 *>(kn)[lane];
            float sh0 = 0.f, sh1 = 0.f;  // scores of heads 2 c4, 2 c4 + 1 (0 past the CTA's heads)
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const uint2 qu = reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p.q) +
                                                                 (row0 + h) * D)[lane];
                float dot = bf16_lo(qu.x) * bf16_lo(ku.x);
                dot = fmaf(bf16_hi(qu.x), bf16_hi(ku.x), dot);
                dot = fmaf(bf16_lo(qu.y), bf16_lo(ku.y), dot);
                dot = fmaf(bf16_hi(qu.y), bf16_hi(ku.y), dot);
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
                if (h == 2 * c4) sh0 = dot * sl2;
                if (h == 2 * c4 + 1) sh1 = dot * sl2;
            }
            raise_max(fmaxf(m[0], sh0), fmaxf(m[1], sh1));
            const float e0 = ptx::ex2(sh0 - m[0]);
            const float e1 = ptx::ex2(sh1 - m[1]);
            if (r4 == 0) {
                lsum[0] += e0;
                lsum[1] += e1;
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const float va = __bfloat162float(vn[16 * mt + r4]);
                const float vb = __bfloat162float(vn[16 * mt + r4 + 8]);
                acc[mt][0] = fmaf(e0, va, acc[mt][0]);
                acc[mt][1] = fmaf(e1, va, acc[mt][1]);
                acc[mt][2] = fmaf(e0, vb, acc[mt][2]);
                acc[mt][3] = fmaf(e1, vb, acc[mt][3]);
            }
        }
        // Row sums over the 16 token rows of the fragments (row groups r4).
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            lsum[0] += __shfl_xor_sync(0xffffffffu, lsum[0], off);
            lsum[1] += __shfl_xor_sync(0xffffffffu, lsum[1], off);
        }
        // merge scratch row of (page stream, head): warp * GH + head
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int h = 2 * c4 + j;
            if (h < GH) {
                float *row = merge + (warp * GH + h) * (D + 2);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    row[16 * mt + r4] = acc[mt][j];
                    row[16 * mt + r4 + 8] = acc[mt][2 + j];
                }
                if (r4 == 0) {
                    row[D] = m[j];
                    row[D + 1] = lsum[j];
                }
            }
        }
    }
    __syncthreads();
    // The merge kernel may be scheduled now; it waits for this grid to finish.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (*abort_flag) return;
    // Merge the page streams: thread = head-dim element, loop over heads.
    if (threadIdx.x < D) {
        const int e = threadIdx.x;
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NCW; ++w) M = fmaxf(M, merge[(w * GH + h) * (D + 2) + D]);
            float Ls = 0.f, o = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < NCW; ++w) {
                    const float *row = merge + (w * GH + h) * (D + 2);
                    const float f = ptx::ex2(row[D] - M);  // -inf -> 0
                    Ls += row[D + 1] * f;
                    o += row[e] * f;
                }
            }
            const int64_t r = row0 + h;
            p.o_part[(r * p.nsplit + split) * D + e] = Ls > 0.f ? o / Ls : 0.f;
            if (e == 0) p.lse_part[r * p.nsplit + split] = Ls > 0.f ? (M + ptx::lg2(Ls)) * LN2 : -INFINITY;
        }
    }
}

// One CTA per row, one thread per head-dim element; splits merged in order.
__global__ void __launch_bounds__(D) merge_kernel(const float *__restrict__ o_parts,
                                                  const float *__restrict__ lse_parts,
                                                  uint16_t *__restrict__ out, float *__restrict__ lse,
                                                  int nsplit, int round_mode) {
    // Launched as a programmatic dependent of the split kernel: wait here
    // until that grid has completed and its partials are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t r = blockIdx.x;
    const int e = threadIdx.x;
    const float *ls = lse_parts + r * nsplit;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ls[s]);
    float total = 0.f, o = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < nsplit; ++s) {
            const float w = ptx::ex2((ls[s] - M) * LOG2E);
            total += w;
            o = fmaf(w, o_parts[(r * nsplit + s) * D + e], o);
        }
    }
    out[r * D + e] = bf16_bits_mode(total > 0.f ? o / total : 0.f, round_mode);
    if (e == 0 && lse != nullptr) lse[r] = total > 0.f ? M + ptx::lg2(total) * LN2 : -INFINITY;
}

}  // namespace dec

// Key-split plan, a pure function of the shape: aim for about
// TARGET_SPLIT_CTAS split CTAs (B * Hq / 4 head groups times the split count),
// so that few sequences still fill the GPU and many do not pay for a merge per
// small split; 16 .. 256 pages per split.
void decode_split_plan(int B, int Hq, int max_blocks, int *nsplit, int *pages_per_split) {
    const long groups = (long)B * ((Hq + 3) / 4);
    long want = (dec::TARGET_SPLIT_CTAS + groups - 1) / groups;
    if (want < 1) want = 1;
    long pps = (max_blocks + want - 1) / want;
    if (pps < 16) pps = 16;
    if (pps > dec::MAX_PAGES_PER_SPLIT) pps = dec::MAX_PAGES_PER_SPLIT;
    *pages_per_split = (int)pps;
    *nsplit = (int)((max_blocks + pps - 1) / pps);
}

cudaError_t launch_decode(const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                          cudaStream_t stream) {
    // Heads per CTA: 4, 2 or 1, the largest dividing the group size.
    const int GH = (p.G % 4 == 0) ? 4 : (p.G % 2 == 0) ? 2 : 1;
    dim3 grid(p.Hq / GH, p.nsplit, p.B);
    const int smem = (int)dec::SMEM_BYTES;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(dec::split_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(dec::split_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(dec::split_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        // Three CTAs of ~74 KiB per SM need the largest shared-memory carveout.
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(dec::split_kernel<4>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(dec::split_kernel<2>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(dec::split_kernel<1>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    if (GH == 4)
        dec::split_kernel<4><<<grid, dec::NTHREADS, smem, stream>>>(mk, mv, p);
    else if (GH == 2)
        dec::split_kernel<2><<<grid, dec::NTHREADS, smem, stream>>>(mk, mv, p);
    else
        dec::split_kernel<1><<<grid, dec::NTHREADS, smem, stream>>>(mk, mv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_lse_merge(p.o_part, p.lse_part, p.out, p.lse, p.B * p.Hq, p.nsplit, kRoundRTNE, stream);
}

cudaError_t launch_lse_merge(const float *o_parts, const float *lse_parts, void *out, float *lse, int rows,
                             int nsplit, int round_mode, cudaStream_t stream) {
    // Programmatic dependent launch: the merge CTAs are scheduled while the
    // previous kernel on the stream finishes and wait (griddepcontrol.wait)
    // for its results, so the launch gap between the two is hidden.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3(dec::D);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dec::merge_kernel, o_parts, lse_parts, static_cast<uint16_t *>(out), lse, nsplit,
                              round_mode);
}

}  // namespace attn
