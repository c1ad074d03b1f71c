// decode.cu -- paged-KV decode split over the keys, and the log-sum-exp merge.
//
// The cache is the paged layout of the ROCm port page ("Vendor-Agnostic 多查询
// 推理优化": 16-token pages, an int32 block_table per sequence); the split over
// the keys with a merge of the partial results is the Flash-Decoding style
// tail split of the MoonMath HIP kernel page.  Decode reads every K/V byte
// once and does ~4 flops per byte, so it is bound by HBM bandwidth and runs on
// the CUDA cores; the tensor cores would only add a reshape.
//
// Split kernel: one CTA per (group of up to 4 query heads sharing a KV head,
// split, sequence); when a KV group has more heads, its head groups are
// adjacent in the grid so that their reads of the same pages meet in L2.  The
// CTAs are small (one producer warp and four consumer warps, about 128
// registers a thread) so three of them share an SM.  The producer lane gathers
// the split's pages with one 3-D TMA copy per page and tensor (the 16 rows of
// one KV head in a page are 2 KiB apart in the pool) into an 8-page
// shared-memory ring.  A consumer warp handles at most 2 heads; with 4 heads
// two warps read each staged page (one per head pair), so the four warps form
// two page streams that take pages alternately (four streams of one warp with
// 1 or 2 heads).  In a warp, lane (tg, ds) =
// (lane/8, lane%8) owns head-dim elements [8 ds, 8 ds + 8) and
// [64 + 8 ds, 64 + 8 ds + 8) of tokens tg, tg+4, tg+8, tg+12 of the page (two
// 16-byte chunks, so the eight lanes of a token read one 256-byte row without
// bank conflicts).  Dot products are reduced over the 8 lanes of a token with
// three shuffles, the page max over the token groups with two more, and each
// warp keeps its own running max / sum / accumulator (online softmax, with the
// max moved only past a 2^8 growth).  At the end the page streams are merged in
// shared memory and the split writes its normalised partial output and
// log-sum-exp.  The merge kernel then combines the splits in a fixed order.
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
constexpr int NCW = 4;   // consumer warps
constexpr int NST = 8;   // pages in flight per CTA
constexpr int GH_MAX = 2;
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr uint32_t PAGE_BYTES = PAGE * D * 2;        // one tensor, one KV head: 4 KiB
constexpr uint32_t STAGE_BYTES = 2 * PAGE_BYTES;     // K + V
constexpr uint32_t SMEM_STAGES = NST * STAGE_BYTES;  // 64 KiB
constexpr uint32_t SMEM_MERGE = NCW * GH_MAX * (D + 2) * 4;
constexpr uint32_t SMEM_MISC = 1536;
constexpr uint32_t SMEM_ALIGN = 1024;
constexpr uint32_t SMEM_BYTES = SMEM_ALIGN + SMEM_STAGES + SMEM_MERGE + SMEM_MISC;
constexpr int MAX_PAGES_PER_SPLIT = 256;
constexpr int TARGET_SPLIT_CTAS = 2048;  // split CTAs the plan aims for (assuming four heads per CTA)
// barriers, per-stage flags, the abort flag and the split's page ids
static_assert(2 * NST * 8 + (NST + 4 + MAX_PAGES_PER_SPLIT) * 4 <= SMEM_MISC, "misc shared area too small");
constexpr float RESCALE_LOG2 = 8.0f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float LOG2E = 1.4426950408889634f;

// Eight bf16 values (one 16-byte chunk) as four fp32 pairs, in element order.
__device__ __forceinline__ void bf16x8_to_float2(const uint4 &u, float2 *x) {
    x[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
    x[1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    x[2] = make_float2(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u));
    x[3] = make_float2(__uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
}

__device__ __forceinline__ void bf16x8_to_float(const uint4 &u, float *x) {
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16);
    x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16);
    x[7] = __uint_as_float(u.w & 0xffff0000u);
}

// GH query heads per CTA (1, 2 or 4, all of one KV head).  Each consumer warp
// handles HG <= 2 of them, so the NHG = GH / HG warps of a "page stream" read
// every staged page together and the page is fetched once for all GH heads.
template <int GH>
__global__ void __launch_bounds__(NTHREADS, 3)
    split_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                 const DecodeParams p) {
    constexpr int HG = GH >= 2 ? 2 : 1;    // heads per consumer warp
    constexpr int NHG = GH / HG;           // warps reading each page
    constexpr int STREAMS = NCW / NHG;     // pages consumed in parallel
    static_assert(STREAMS * GH <= NCW * GH_MAX, "merge scratch too small");
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

    if (np == 0 && !new_token) {  // nothing to attend to in this split
        for (int i = threadIdx.x; i < GH * D; i += NTHREADS)
            p.o_part[((row0 + i / D) * p.nsplit + split) * D + (i % D)] = 0.f;
        if (threadIdx.x < GH) p.lse_part[(row0 + threadIdx.x) * p.nsplit + split] = -INFINITY;
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            ptx::mbar_init(full + s, 1);
            ptx::mbar_init(empty + s, NHG);
            stage_bad[s] = 0;
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const WaitCtx wc{abort_flag, p.status, p.budget_ns};

    if (warp == NCW) {
        // ---------------- producer
        // The whole warp reads the split's block-table entries in one go, so
        // the copy-issuing lane never waits on a global load per page.
        for (int k = lane; k < np; k += 32) split_pages[k] = p.block_table[(int64_t)b * p.max_blocks + page0 + k];
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
                    ptx::mbar_arrive_expect_tx(full + slot, STAGE_BYTES);
                    ptx::tma_load_3d_hint(dst, &map_k, full + slot, 0, g, phys * PAGE, pol);
                    ptx::tma_load_3d_hint(dst + PAGE_BYTES, &map_v, full + slot, 0, g, phys * PAGE, pol);
                }
                ++issued;
            }
            for (int i = max(0, issued - NST); i < issued; ++i) drain_wait(full + i % NST, (i / NST) & 1, wc);
        }
        __syncwarp();
    } else {
        // ---------------- consumers
        const int tg = lane >> 3;  // token group
        const int ds = lane & 7;   // head-dim chunks ds and 8 + ds
        const int hg = warp % NHG;       // this warp's heads: hg * HG .. hg * HG + HG - 1
        const int stream = warp / NHG;   // this warp's pages: stream, stream + STREAMS, ...
        const int64_t wrow0 = row0 + hg * HG;
        // Dot products and the P V accumulation run on fp32 pairs (packed
        // FFMA2): element pairs (2i, 2i+1) of the lane's 16 head-dim elements.
        float2 qf[HG][8];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
            const uint4 *qp = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.q) +
                                                              (wrow0 + h) * D);
            bf16x8_to_float2(qp[ds], qf[h]);
            bf16x8_to_float2(qp[8 + ds], qf[h] + 4);
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[h][e] = __fmul2_rn(qf[h][e], sc2);
        }
        float m[HG], lsum[HG], msub[HG];  // msub: m, or 0 while m is -inf
        float2 acc[HG][8];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
            m[h] = -INFINITY;
            msub[h] = 0.f;
            lsum[h] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] = make_float2(0.f, 0.f);
        }
        for (int i = stream; i < np; i += STREAMS) {
            const int slot = i % NST;
            if (!wait_bounded(full + slot, (i / NST) & 1, wc, kSiteDecodeFull)) break;
            const uint8_t *ks = base + slot * STAGE_BYTES;
            const uint8_t *vs = ks + PAGE_BYTES;
            const bool bad = stage_bad[slot] != 0;
            const int tok0 = (page0 + i) * PAGE;
            // A page whose 16 slots all hold keys of the sequence needs no
            // masking: it takes a copy of the page step without the selects.
            auto page_step = [&](auto full_tag) {
                constexpr bool FULL = decltype(full_tag)::value;
                float sc[4][HG];
#pragma unroll
                for (int ps = 0; ps < 4; ++ps) {
                    const int t = ps * 4 + tg;
                    const uint4 *kp = reinterpret_cast<const uint4 *>(ks + t * (D * 2));
                    float2 kf[8];
                    bf16x8_to_float2(kp[ds], kf);
                    bf16x8_to_float2(kp[8 + ds], kf + 4);
#pragma unroll
                    for (int h = 0; h < HG; ++h) {
                        float2 d2 = __fmul2_rn(qf[h][0], kf[0]);
#pragma unroll
                        for (int e = 1; e < 8; ++e) d2 = __ffma2_rn(qf[h][e], kf[e], d2);
                        float dot = d2.x + d2.y;
                        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
                        dot += __shfl_xor_sync(0xffffffffu, dot, 4);
                        sc[ps][h] = (FULL || (!bad && tok0 + t < L)) ? dot : -INFINITY;
                    }
                }
                float pr[4][HG];
#pragma unroll
                for (int h = 0; h < HG; ++h) {
                    float pm = ptx::max3(sc[0][h], sc[1][h], fmaxf(sc[2][h], sc[3][h]));
                    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
                    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
                    if (pm > m[h] + RESCALE_LOG2) {  // warp-uniform
                        const float alpha = ptx::ex2(m[h] - pm);
                        lsum[h] *= alpha;
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[h][e] = __fmul2_rn(acc[h][e], make_float2(alpha, alpha));
                        m[h] = pm;
                        msub[h] = pm;
                    }
#pragma unroll
                    for (int ps = 0; ps < 4; ++ps) {
                        // a masked score (-inf) gives ex2(-inf) = 0 with no select
                        pr[ps][h] = ptx::ex2(sc[ps][h] - msub[h]);
                        lsum[h] += pr[ps][h];
                    }
                }
                // Slots past the sequence end (and pages that could not be
                // read) hold arbitrary bits: their P is 0, but 0 * NaN is NaN,
                // so on such a page the V of invalid tokens is replaced by 0.
#pragma unroll
                for (int ps = 0; ps < 4; ++ps) {
                    const int t = ps * 4 + tg;
                    const uint4 *vp = reinterpret_cast<const uint4 *>(vs + t * (D * 2));
                    float2 vf[8];
                    bf16x8_to_float2(vp[ds], vf);
                    bf16x8_to_float2(vp[8 + ds], vf + 4);
                    if (!FULL && (bad || tok0 + t >= L)) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) vf[e] = make_float2(0.f, 0.f);
                    }
#pragma unroll
                    for (int h = 0; h < HG; ++h) {
                        const float2 p2 = make_float2(pr[ps][h], pr[ps][h]);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[h][e] = __ffma2_rn(p2, vf[e], acc[h][e]);
                    }
                }
            };
            if (!bad && tok0 + PAGE <= L)
                page_step(std::true_type{});
            else
                page_step(std::false_type{});
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty + slot);
        }
        if (new_token && stream == 0) {
            // The appended token, read from k_new / v_new rather than the
            // cache: every token group computes the same score and only
            // group 0 adds the token to its sums.
            const int64_t src = ((int64_t)b * p.Hkv + g) * D;
            const uint4 *kn = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.k_new) + src);
            const uint4 *vn = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.v_new) + src);
            float2 kf[8], vf[8];
            bf16x8_to_float2(kn[ds], kf);
            bf16x8_to_float2(kn[8 + ds], kf + 4);
            bf16x8_to_float2(vn[ds], vf);
            bf16x8_to_float2(vn[8 + ds], vf + 4);
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                float2 d2 = __fmul2_rn(qf[h][0], kf[0]);
#pragma unroll
                for (int e = 1; e < 8; ++e) d2 = __ffma2_rn(qf[h][e], kf[e], d2);
                float sc = d2.x + d2.y;
                sc += __shfl_xor_sync(0xffffffffu, sc, 1);
                sc += __shfl_xor_sync(0xffffffffu, sc, 2);
                sc += __shfl_xor_sync(0xffffffffu, sc, 4);
                if (sc > m[h] + RESCALE_LOG2) {  // warp-uniform
                    const float alpha = ptx::ex2(m[h] - sc);
                    lsum[h] *= alpha;
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[h][e] = __fmul2_rn(acc[h][e], make_float2(alpha, alpha));
                    m[h] = sc;
                }
                const float pr = tg == 0 ? ptx::ex2(sc - m[h]) : 0.f;
                lsum[h] += pr;
                const float2 p2 = make_float2(pr, pr);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] = __ffma2_rn(p2, vf[e], acc[h][e]);
            }
        }
        // Sum the four token groups (lanes 8 and 16 apart share a slice).
#pragma unroll
        for (int h = 0; h < HG; ++h) {
            lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], 8);
            lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], 16);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, 8);
                acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, 8);
                acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, 16);
                acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, 16);
            }
        }
        // merge scratch row of (page stream, head): stream * GH + head
        float *mw = merge + (stream * GH + hg * HG) * (D + 2);
#pragma unroll
        for (int h = 0; h < HG; ++h) {
            float *row = mw + h * (D + 2);
            if (tg == 0) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    row[ds * 8 + 2 * e] = acc[h][e].x;
                    row[ds * 8 + 2 * e + 1] = acc[h][e].y;
                    row[64 + ds * 8 + 2 * e] = acc[h][4 + e].x;
                    row[64 + ds * 8 + 2 * e + 1] = acc[h][4 + e].y;
                }
            }
            if (lane == 0) {
                row[D] = m[h];
                row[D + 1] = lsum[h];
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
            for (int w = 0; w < STREAMS; ++w) M = fmaxf(M, merge[(w * GH + h) * (D + 2) + D]);
            float Ls = 0.f, o = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < STREAMS; ++w) {
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
