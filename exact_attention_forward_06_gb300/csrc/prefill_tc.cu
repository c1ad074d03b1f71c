// prefill_tc.cu -- fused exact attention forward on sm_103a tensor cores.
//
// O = softmax(Q K^T * scale [+ causal mask]) V and the per-row log-sum-exp,
// with the IO-aware tiling of "FlashAttention-4 中的 IO 感知块分块策略": Q is cut
// into 128-row blocks, K/V stream through shared memory in 128-key tiles, and
// each row keeps a running max m and running sum l (m' = max(m, m_new),
// l' = l exp(m - m') + l_new) while the output accumulator is rescaled, so the
// Sq x Sk score matrix never reaches HBM.  Tiles entirely above the causal
// diagonal are never loaded or computed (the upper-triangle skip of the
// reverse-engineering page, 观点一).
//
// A work unit is two 128-row Q tiles (256 rows: two heads of one KV group at
// the same positions when the group size is even, else two adjacent position
// blocks of one head), so every K/V tile that is loaded serves 256 query
// rows.  The grid has at most one CTA per SM; each CTA takes units from the
// list (longest first where lengths differ) as it frees up, and every barrier
// phase runs on across its units, so the next unit's Q, K and V load while
// the current unit finishes.  Warp roles (384 threads, three
// warpgroups):
//   warp 0      TMA producer: per unit the two Q tiles (each once the previous
//               unit's last S product has read its buffer), then K_j / V_j
//               into a 5-slot ring of 32 KiB slots (full/empty mbarrier
//               pairs), then two ring slots that the softmax groups use to
//               stage the unit's output tiles for their TMA stores;
//   warp 1      TMEM allocator and tcgen05 MMA issuer for Q tile 0 (one lane);
//   warp 2      tcgen05 MMA issuer for Q tile 1 (one lane);
//   warp 3      idle (it completes warpgroup 0, which gives up registers);
//   warps 4-7   softmax warpgroup for Q tile 0 (one thread per row);
//   warps 8-11  softmax warpgroup for Q tile 1.
// setmaxnreg moves registers from warpgroup 0 (80 each) to the softmax
// warpgroups (208 each), which hold a whole 128-column score row.
// Tensor memory (512 columns): one fp32 score buffer S that the two tiles use
// in turn, a bf16 probability buffer P_t per tile (64 columns of packed
// pairs, read by the P V product straight from tensor memory) and an fp32
// output accumulator O_t per tile.  Each tile has its own issuing thread,
// which issues S_t(j+1) then PV_t(j) for every K/V tile j; the score tiles
// alternate through the shared S buffer (S_0(j), S_1(j), S_0(j+1), ...), each
// issued as soon as the other tile's softmax has loaded the previous one.
// While one tile's softmax runs the tensor core works on the other tile's
// products (the two-group alternation of the MoonMath page, realised as two
// Q tiles instead of two wave groups), and since an issuing thread is held
// while its products execute, two of them keep the tensor core fed across
// each other's waits.
//
// Softmax: scores are scaled into the log2 domain (scale * log2 e folded into
// one FFMA) and exponentiated with ex2.approx.  A row's running max is only
// moved (and O rescaled) when the new tile's max exceeds it by more than
// 2^8, or when the new maximum would carry more than half of the row's sum so
// far; otherwise the stale max is kept, which is exact because m and l stay
// consistent and P <= 256 is representable.  The second condition is for
// accuracy: P goes to the tensor core rounded to bf16 (8 significant bits), so
// a key that dominates its row must get P = 1 exactly (its score is the
// running max), or the rounding of two dominant keys whose V rows cancel
// shows in O.  On unit-normal scores it fires on about 1 warp-tile in 10^4.
// The rescale, when needed, is done by the softmax warp itself on its own 32
// rows of O in tensor memory, after the previous P V product has completed.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "prefill_tc.h"

namespace attn {
namespace g1 {

constexpr int BM = 128;          // rows per Q tile
constexpr int BN = 128;          // keys per K/V tile
constexpr int D = 128;           // head dim
constexpr int NSLOT = 5;         // K/V ring slots
constexpr uint32_t TILE_BYTES = BM * D * 2;  // 32 KiB (128 rows x 256 B)
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;  // one 64-column half (128 B rows, 128-B swizzle)
// Paged K/V tiles are laid out by 8-row group: [16 groups][2 halves][8 rows]
// [128 B], so one page (two groups, both halves) is one contiguous 4 KiB box.
// Row r, half h of such a tile is at (r / 8) * 2048 + h * 1024 + (r % 8) * 128.
constexpr uint32_t PAGE_BOX_BYTES = 4096;
constexpr uint32_t PG_GROUP_BYTES = 2048;  // one 8-row group, both halves
constexpr uint32_t PG_HALF_BYTES = 1024;   // one 8-row group, one half
constexpr int NUM_THREADS = 384;  // three warpgroups
constexpr uint32_t REGS_CONTROL = 80;   // warpgroup 0: producer, MMA issuer
constexpr uint32_t REGS_SOFTMAX = 208;  // warpgroups 1-2: softmax
// setmaxnreg hands registers between warpgroups within the launch budget
// (384 threads x 168): 128 x 80 + 256 x 208 <= 384 x 168.
static_assert(128 * REGS_CONTROL + 256 * REGS_SOFTMAX <= NUM_THREADS * 168, "register split exceeds the launch budget");
constexpr uint32_t SMEM_Q0 = 0;
constexpr uint32_t SMEM_Q1 = TILE_BYTES;
constexpr uint32_t SMEM_SLOTS = 2 * TILE_BYTES;
constexpr uint32_t SMEM_TILES = SMEM_SLOTS + NSLOT * TILE_BYTES;
// Work items handed from the producer to the other roles through a small
// ring in shared memory.
constexpr int ITEM_RING = 4;
// Roles that read each handed-out unit: the two MMA issuing threads and the
// eight softmax warps.
constexpr uint32_t ITEM_READERS = 2 + 8;
// q_full[2], q_free[2], kv_full[NSLOT], kv_empty[NSLOT], s_full[2], s_free[2],
// p_full[2], o_full[2], fin, item_full[ITEM_RING], item_empty[ITEM_RING],
// stage_ready[2], stage_taken[2]
constexpr int NBARS = 2 + 2 + 2 * NSLOT + 2 + 2 + 2 + 2 + 1 + 2 * ITEM_RING + 2 + 2;
constexpr uint32_t SMEM_MISC = 768;
constexpr uint32_t SMEM_ALIGN = 1024;
constexpr float RESCALE_LOG2 = 8.0f;  // move the running max past a 2^8 growth (and see softmax_wg)
constexpr float LN2 = 0.6931471805599453f;

static_assert(NBARS * 8 + 8 + 64 * ITEM_RING + 2 * 32 <= SMEM_MISC, "barrier area too small");

constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(128, 128, 0, 0);   // Q K^T: both K-major
constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(128, 128, 0, 1);  // P V: V is N(d)-major

// Tensor-memory columns: one S buffer shared by the two tiles in turn, a bf16
// P buffer per tile (64 columns of packed pairs) and an fp32 O accumulator per
// tile.  P never aliases an S that a later product writes.
constexpr uint32_t TM_S = 0;
constexpr uint32_t TM_P0 = 128;
constexpr uint32_t TM_O0 = 256;
__device__ __forceinline__ uint32_t tm_p(int t) { return TM_P0 + 64 * t; }
__device__ __forceinline__ uint32_t tm_o(int t) { return TM_O0 + 128 * t; }

struct SmemLayout {
    uint8_t *base;
    uint64_t *bars;
    // q_full(t): Q tile t of the current unit has landed; q_free(t): the
    // unit's last S product has read it (one phase per unit each).
    __device__ uint64_t *q_full(int t) const { return bars + t; }
    __device__ uint64_t *q_free(int t) const { return bars + 2 + t; }
    __device__ uint64_t *kv_full(int s) const { return bars + 4 + s; }
    __device__ uint64_t *kv_empty(int s) const { return bars + 4 + NSLOT + s; }
    __device__ uint64_t *s_full(int t) const { return bars + 4 + 2 * NSLOT + t; }
    // s_free(t): phase g completes when softmax group t has loaded its score tile g.
    __device__ uint64_t *s_free(int t) const { return bars + 6 + 2 * NSLOT + t; }
    __device__ uint64_t *p_full(int t) const { return bars + 8 + 2 * NSLOT + t; }
    __device__ uint64_t *o_full(int t) const { return bars + 10 + 2 * NSLOT + t; }
    __device__ uint64_t *fin() const { return bars + 12 + 2 * NSLOT; }
    // item_full(i): entry i of the item ring holds the next item; item_empty(i):
    // every reader has taken it.
    __device__ uint64_t *item_full(int i) const { return bars + 13 + 2 * NSLOT + i; }
    __device__ uint64_t *item_empty(int i) const { return bars + 13 + 2 * NSLOT + ITEM_RING + i; }
    // stage_ready(t): softmax group t has written a store command for its
    // output tile; stage_taken(t): the store lane has read it.
    __device__ uint64_t *stage_ready(int t) const { return bars + 13 + 2 * NSLOT + 2 * ITEM_RING + t; }
    __device__ uint64_t *stage_taken(int t) const { return bars + 15 + 2 * NSLOT + 2 * ITEM_RING + t; }
    __device__ uint32_t *tmem_slot() const { return reinterpret_cast<uint32_t *>(bars + NBARS); }
    __device__ volatile int *abort_flag() const { return reinterpret_cast<volatile int *>(bars + NBARS) + 1; }
    // Entry i of the item ring: a decoded unit (16 ints), 8-byte aligned.
    __device__ volatile int *item_ring(int i) const {
        return reinterpret_cast<volatile int *>(bars + NBARS + 1) + 16 * i;
    }
    // Store command of tile t: kind (0: no more, 1: store), ring slot, the box's
    // four coordinates (first 64-column half).
    __device__ volatile int *stage_cmd(int t) const {
        return reinterpret_cast<volatile int *>(bars + NBARS + 1) + 16 * ITEM_RING + 8 * t;
    }
    __device__ uint8_t *q_tile(int t) const { return base + (t ? SMEM_Q1 : SMEM_Q0); }
    // Ring slot s: a K or V tile, or a tile's output staging area.
    __device__ uint8_t *slot(int s) const { return base + SMEM_SLOTS + s * TILE_BYTES; }
};

// Which two (head, first row) tiles a unit covers, and its K/V tile count.
struct Unit {
    int b, g;
    int h[2];
    int s0[2];
    int n_kv;    // K/V tiles this CTA processes
    int j_lo;    // first K/V tile (absolute)
    int part;    // key-range part of a split unit, -1 for a whole unit
    int ws_row;  // first workspace row of a split unit (256 rows per unit)
    int Sq, Sk;  // lengths of this unit's sequence (a packed batch: its own)
    int q0, k0;  // first row of the sequence in q and in k, v (0 when dense)
    int tb;      // batch coordinate of the TMA boxes (0 in a packed batch)
};

// K/V tile count of a unit from its rows and its sequence's lengths: every
// tile for a non-causal unit; for a causal one, up to the tile holding the
// last key its lowest row may see (bottom-right alignment).
__host__ __device__ __forceinline__ void unit_kv_range(const PrefillParams &p, Unit &w) {
    const int n_full = (w.Sk + BN - 1) / BN;
    if (p.causal) {
        const int span = p.pack_heads ? p.pack_pos : BM;  // positions a tile covers
        int last_row = w.s0[0] + span - 1;
        if (w.s0[1] < w.Sq) last_row = last_row > w.s0[1] + span - 1 ? last_row : w.s0[1] + span - 1;
        last_row = last_row < w.Sq - 1 ? last_row : w.Sq - 1;
        const int lim = last_row + w.Sk - w.Sq;  // last visible key of the lowest row
        w.n_kv = lim < 0 ? 0 : (n_full < lim / BN + 1 ? n_full : lim / BN + 1);
    } else {
        w.n_kv = n_full;
    }
}

// Heads, rows and K/V tile count of work unit u (two 128-row Q tiles).
__host__ __device__ __forceinline__ Unit unit_coords(const PrefillParams &p, int u) {
    Unit w;
    int m_step;
    // Row block first (all heads of the longest row blocks, then the next)
    // balances the causal work.  Sequence and KV head first (longest row
    // blocks first within) runs the units that read the same K/V at the same
    // time, which pays when the keys of all heads exceed L2 and every row
    // block reads a long context (non-causal launches, whose units are all
    // alike, and chunks against a cache); the host chooses.
    const bool kv_major = p.kv_major != 0;
    if (p.pack_heads) {
        // Both tiles hold every head of KV group g, at positions
        // [s, s + pack_pos) and [s + pack_pos, s + 2 pack_pos).
        int bg;
        if (kv_major) {
            bg = u / p.n_pk;
            m_step = u % p.n_pk;
        } else {
            const int per = p.B * p.Hkv;
            m_step = u / per;
            bg = u % per;
        }
        w.b = bg / p.Hkv;
        w.g = bg % p.Hkv;
        const int mb = p.causal ? (p.n_pk - 1 - m_step) : m_step;  // causal: longest units first
        w.h[0] = w.h[1] = w.g * p.G;
        w.s0[0] = mb * 2 * p.pack_pos;
        w.s0[1] = w.s0[0] + p.pack_pos;
    } else if (p.pair_heads) {
        const int pairs = p.G / 2;
        int r;
        if (p.seq_group > 0) {
            // Sequences in groups of seq_group, row block first within a group
            // (longest row blocks of the group's sequences first), the groups
            // one after another: the K/V in use at once is one group's.
            const int per_seq = p.Hkv * pairs;              // units of one sequence per row-block step
            const int per_group = p.seq_group * per_seq * p.n_m;
            const int grp = u / per_group;
            r = u % per_group;
            const int nseq = min(p.seq_group, p.B - grp * p.seq_group);
            m_step = r / (nseq * per_seq);
            r = (grp * p.seq_group) * per_seq + r % (nseq * per_seq);  // (b, g, pair) index
        } else if (kv_major) {
            const int bg = u / (p.n_m * pairs);
            r = u % (p.n_m * pairs);
            m_step = r / pairs;
            r = bg * pairs + r % pairs;  // (b, g, pair) index
        } else {
            const int per = p.B * p.Hkv * pairs;
            m_step = u / per;
            r = u % per;
        }
        w.b = r / (p.Hkv * pairs);
        r %= p.Hkv * pairs;
        w.g = r / pairs;
        const int pr = r % pairs;
        const int mb = p.causal ? (p.n_m - 1 - m_step) : m_step;  // causal: longest units first
        w.h[0] = w.g * p.G + 2 * pr;
        w.h[1] = w.h[0] + 1;
        w.s0[0] = w.s0[1] = mb * BM;
    } else {
        const int per = p.B * p.Hq;
        const int n_mp = (p.n_m + 1) / 2;
        m_step = kv_major ? u % n_mp : u / per;
        int r = kv_major ? u / n_mp : u % per;
        if (p.seq_group > 0) {  // as above, one head per unit
            const int per_group = p.seq_group * p.Hq * n_mp;
            const int grp = u / per_group;
            const int rr = u % per_group;
            const int nseq = min(p.seq_group, p.B - grp * p.seq_group);
            m_step = rr / (nseq * p.Hq);
            r = grp * p.seq_group * p.Hq + rr % (nseq * p.Hq);
        }
        w.b = r / p.Hq;
        const int h = r % p.Hq;
        w.g = h / p.G;
        const int mp = p.causal ? (n_mp - 1 - m_step) : m_step;
        w.h[0] = w.h[1] = h;
        w.s0[0] = mp * 2 * BM;
        w.s0[1] = mp * 2 * BM + BM;
    }
    w.Sq = p.Sq;
    w.Sk = p.Sk;
    w.q0 = 0;
    w.k0 = 0;
    w.tb = w.b;
    unit_kv_range(p, w);
    w.j_lo = 0;
    w.part = -1;
    w.ws_row = 0;
    return w;
}

// The unit (and key range) of work item `it`, for each kind of launch.
// kDense: items past the whole units are the parts of the tail units,
// part-major within a unit.  kPacked / kPaged: the unit's rows and keys are
// those of its sequence; offsets that are out of order or out of range, or
// lengths past the stated maxima, are reported and the unit does nothing.
enum LaunchKind : int { kDense = 0, kPacked = 1, kPaged = 2 };

template <int KIND>
__device__ __forceinline__ Unit decode_unit(const PrefillParams &p, int it) {
    if (KIND == kPaged) {
        // Query chunk of sequence w.b against its paged cache.
        Unit w = unit_coords(p, it);
        const int q0 = p.cu_q[w.b], q1 = p.cu_q[w.b + 1];
        const int Lk = p.seqlens_k[w.b];
        const bool bad = q0 < 0 || q1 < q0 || q1 > p.total_q || q1 - q0 > p.Sq || Lk < 0 || Lk > p.max_blocks * 16;
        if (bad) report_status(p.status, kStatusDeviceBounds, kSiteVarlenOffsets);
        w.Sq = bad ? 0 : q1 - q0;
        w.Sk = bad ? 0 : Lk;
        w.q0 = bad ? 0 : q0;
        w.k0 = 0;
        w.tb = 0;
        unit_kv_range(p, w);
        return w;
    }
    if (KIND == kPacked) {
        Unit w = unit_coords(p, it);
        const int q0 = p.cu_q[w.b], q1 = p.cu_q[w.b + 1];
        const int k0 = p.cu_k[w.b], k1 = p.cu_k[w.b + 1];
        const bool bad = q0 < 0 || q1 < q0 || q1 > p.total_q || k0 < 0 || k1 < k0 || k1 > p.total_k ||
                         q1 - q0 > p.Sq || k1 - k0 > p.Sk;
        if (bad) report_status(p.status, kStatusDeviceBounds, kSiteVarlenOffsets);
        w.Sq = bad ? 0 : q1 - q0;
        w.Sk = bad ? 0 : k1 - k0;
        w.q0 = bad ? 0 : q0;
        w.k0 = bad ? 0 : k0;
        w.tb = 0;
        unit_kv_range(p, w);
        return w;
    }
    if (it < p.n_full_units) return unit_coords(p, it);
    const int v = it - p.n_full_units;
    const int su = v / p.split_parts;
    const int part = v % p.split_parts;
    Unit w = unit_coords(p, p.n_full_units + su);
    const int lo = part * w.n_kv / p.split_parts;
    const int hi = (part + 1) * w.n_kv / p.split_parts;
    w.j_lo = lo;
    w.n_kv = hi - lo;
    w.part = part;
    w.ws_row = su * 2 * BM;
    return w;
}

// ------------------------------------------------------------------ work items

// Work items are handed out dynamically: CTA c starts with item c, and each
// CTA that finishes one takes the next unclaimed item from a counter shared
// by the launch (p.sched[0], counting from gridDim.x), so the CTAs work
// through the list in order, each taking the next item as soon as it is free
// -- the order the hardware would dispatch one CTA per item in, without a
// CTA launch per item.  The producer thread claims the items and hands them
// to the other roles through the item ring; -1 ends the list.  With one CTA
// per item no counter is used.
__device__ __forceinline__ int claim_item(const PrefillParams &p) {
    if ((int)gridDim.x >= p.n_items) return -1;
    const int it = (int)gridDim.x + (int)atomicAdd(p.sched, 1u);
    return it < p.n_items ? it : -1;
}

// The next unit this CTA works on: the first item (this CTA's own first one,
// or claimed) whose rows do not all lie past their sequence's end (packed
// batches size their item list by the longest sequence); n_kv = -1 when the
// list is used up.  Only the producer thread calls this: it decodes each item
// once and hands the decoded unit to the other roles.
// Given item `it` whose rows lie past its sequence's end, the first item after
// it that may have rows, when the item list is ordered by sequence and KV head
// (kv_major): such items are contiguous within their (sequence, KV group)
// block -- its first items for a causal launch (longest row blocks first), its
// last ones otherwise.  Without that order, the next item.
__device__ __forceinline__ int next_candidate(const PrefillParams &p, int it, int seq_len) {
    if (!p.kv_major) return it + 1;
    const int step = p.pair_heads ? p.G / 2 : 1;              // items per row-block step
    const int steps = p.pair_heads ? p.n_m : (p.n_m + 1) / 2;   // row-block steps per block
    const int rows_per_step = p.pair_heads ? BM : 2 * BM;
    const int per = step * steps;
    const int start = it - it % per;
    const int valid = (seq_len + rows_per_step - 1) / rows_per_step;  // steps with rows
    const int target = p.causal ? start + (steps - valid) * step : start + per;
    return target > it + 1 ? target : it + 1;
}

template <int KIND>
__device__ __forceinline__ Unit next_unit(const PrefillParams &p, bool first) {
    for (int it = first ? ((int)blockIdx.x < p.n_items ? (int)blockIdx.x : -1) : claim_item(p); it >= 0;
         it = claim_item(p)) {
        const Unit w = decode_unit<KIND>(p, it);
        if (w.s0[0] < w.Sq) return w;
        // Move the shared counter past the rest of this run of empty items
        // (they would only be claimed and skipped one by one).
        const int nx = KIND == kDense ? it + 1 : next_candidate(p, it, w.Sq);
        if (nx > it + 1 && (int)gridDim.x < p.n_items) atomicMax(p.sched, (unsigned)max(0, nx - (int)gridDim.x));
    }
    Unit end{};
    end.n_kv = -1;
    return end;
}

// Producer side: put unit w (n_kv = -1: end of the list) into ring entry
// u % ITEM_RING for the readers.
__device__ __forceinline__ bool publish_unit(const SmemLayout &sm, const WaitCtx &wc, int u, const Unit &w) {
    const int e = u % ITEM_RING;
    if (u >= ITEM_RING && !wait_bounded(sm.item_empty(e), (uint32_t)(((u / ITEM_RING) - 1) & 1), wc, kSiteItem))
        return false;
    volatile int *d = sm.item_ring(e);
    d[0] = w.b; d[1] = w.g; d[2] = w.h[0]; d[3] = w.h[1]; d[4] = w.s0[0]; d[5] = w.s0[1]; d[6] = w.n_kv;
    d[7] = w.j_lo; d[8] = w.part; d[9] = w.ws_row; d[10] = w.Sq; d[11] = w.Sk; d[12] = w.q0; d[13] = w.k0;
    d[14] = w.tb;
    ptx::mbar_arrive(sm.item_full(e));  // release: the writes above are seen by whoever sees the phase
    return true;
}

// Reader side (every lane of a reading warp): unit u of this CTA.  Returns
// false when the CTA is giving up; w.n_kv = -1 marks the end of the list.
// The caller hands the entry back (item_empty) once every lane has read it.
__device__ __forceinline__ bool read_unit(const SmemLayout &sm, const WaitCtx &wc, int u, bool spin, Unit &w) {
    const int e = u % ITEM_RING;
    const uint32_t par = (uint32_t)((u / ITEM_RING) & 1);
    if (!(spin ? wait_spin(sm.item_full(e), par, wc, kSiteItem) : wait_bounded(sm.item_full(e), par, wc, kSiteItem)))
        return false;
    const volatile int *d = sm.item_ring(e);
    w.b = d[0]; w.g = d[1]; w.h[0] = d[2]; w.h[1] = d[3]; w.s0[0] = d[4]; w.s0[1] = d[5]; w.n_kv = d[6];
    w.j_lo = d[7]; w.part = d[8]; w.ws_row = d[9]; w.Sq = d[10]; w.Sk = d[11]; w.q0 = d[12]; w.k0 = d[13];
    w.tb = d[14];
    return true;
}

// Ring items of a unit: its K/V tiles, then one output staging slot per Q tile.
__device__ __forceinline__ int ring_items(const Unit &w) { return 2 * w.n_kv + 2; }

// ------------------------------------------------------------------ producer

__device__ __forceinline__ void load_tile(const CUtensorMap *map, uint8_t *dst, uint64_t *bar, bool bhsd, int h,
                                          int s, int b, uint64_t pol) {
    const Coord4 lo = coord4(bhsd, 0, h, s, b);
    const Coord4 hi = coord4(bhsd, 64, h, s, b);
    ptx::tma_load_4d(dst, map, bar, lo.c0, lo.c1, lo.c2, lo.c3, pol);
    ptx::tma_load_4d(dst + HALF_BYTES, map, bar, hi.c0, hi.c1, hi.c2, hi.c3, pol);
}

// L2 prefetch of the Q tiles of this CTA's next unit (short units spend much
// of their time loading Q: start it early so it is in L2 when wanted).
__device__ __forceinline__ void prefetch_q(const PrefillParams &p, const CUtensorMap *mq, const Unit &w) {
    if (w.n_kv < 0) return;
    for (int t = 0; t < 2; ++t) {
        const Coord4 lo = coord4(p.bhsd, 0, t ? w.h[1] : w.h[0], w.q0 + (t ? w.s0[1] : w.s0[0]), w.tb);
        const Coord4 hi = coord4(p.bhsd, 64, t ? w.h[1] : w.h[0], w.q0 + (t ? w.s0[1] : w.s0[0]), w.tb);
        ptx::tma_prefetch_4d(mq, lo.c0, lo.c1, lo.c2, lo.c3);
        ptx::tma_prefetch_4d(mq, hi.c0, hi.c1, hi.c2, hi.c3);
    }
}

// Dense and packed K/V (one lane).  Per unit: hand it to the other roles,
// load the two Q tiles, each once the previous unit's last S product has
// read its buffer (q_free), find the next unit while they load, then the K/V
// tiles into the ring, then the two output staging slots (a plain arrive on
// the slot's full barrier once the slot is empty: the softmax group fills it
// and empties it again after its output store has read it).
template <int KIND>
__device__ void producer(const PrefillParams &p, const SmemLayout &sm, const WaitCtx &wc, const CUtensorMap *mq,
                         const CUtensorMap *mk, const CUtensorMap *mv) {
    if (p.inject == 1) return;  // fault injection: issue nothing
    const uint64_t pol_q = ptx::policy_evict_first();
    const uint64_t pol_kv = ptx::policy_evict_last();
    int n = 0;                 // ring items issued
    int qn[2] = {0, 0};        // Q loads issued per tile
    int u = 0;                 // units handed out
    bool ok = true;
    Unit w = next_unit<KIND>(p, true);
    while (ok && w.n_kv >= 0) {
        Unit nx;
        nx.n_kv = -1;
        if (!publish_unit(sm, wc, u++, w)) {
            ok = false;
            break;
        }
        // Q tiles, each once the previous unit's last S product has read its
        // buffer; then the next unit (its claim and offsets) while they load.
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (qn[t] > 0 && !wait_bounded(sm.q_free(t), (qn[t] - 1) & 1, wc, kSiteProducerQ)) {
                ok = false;
                break;
            }
            ptx::mbar_arrive_expect_tx(sm.q_full(t), TILE_BYTES);
            load_tile(mq, sm.q_tile(t), sm.q_full(t), p.bhsd, t ? w.h[1] : w.h[0], w.q0 + (t ? w.s0[1] : w.s0[0]),
                      w.tb, pol_q);
            ++qn[t];
        }
        if (!ok) break;
        nx = next_unit<KIND>(p, false);
        if (p.prefetch_ahead > 0) prefetch_q(p, mq, nx);
        const int total = ring_items(w);
        for (int i = 0; i < total; ++i) {
            const int slot = n % NSLOT;
            if (n >= NSLOT && !wait_bounded(sm.kv_empty(slot), ((n / NSLOT) - 1) & 1, wc, kSiteProducerEmpty)) {
                ok = false;
                break;
            }
            if (i < 2 * w.n_kv) {
                ptx::mbar_arrive_expect_tx(sm.kv_full(slot), TILE_BYTES);
                load_tile((i & 1) ? mv : mk, sm.slot(slot), sm.kv_full(slot), p.bhsd, w.g,
                          w.k0 + (w.j_lo + (i >> 1)) * BN, w.tb, pol_kv);
            } else {
                ptx::mbar_arrive(sm.kv_full(slot));  // an output staging slot
            }
            ++n;
        }
        w = nx;
    }
    if (ok) publish_unit(sm, wc, u, w);  // end of the list (n_kv = -1)
    // On the way out make sure no copy is still writing into shared memory.
    for (int t = 0; t < 2; ++t)
        if (qn[t] > 0) drain_wait(sm.q_full(t), (qn[t] - 1) & 1, wc);
    for (int i = max(0, n - NSLOT); i < n; ++i) drain_wait(sm.kv_full(i % NSLOT), (i / NSLOT) & 1, wc);
}

// Paged K/V: the whole warp 0 produces.  A K/V tile is 8 pages; lane i < 8
// reads table entry i of the tile and issues the one 4 KiB box (16 rows, both
// 64-column halves) of page i, so the table loads and the 16 copies of a tile
// pair go out in parallel instead of one after another from a single lane.
// Lane 0 arms each barrier before any lane issues into it, finds and hands
// out the units, loads Q and hands out the staging slots as the dense
// producer does.  Pages past the
// sequence's last one, and bad entries (reported), get a row past the pool:
// the copy then fills zeros.  When the tile's 8 pages are consecutive in the
// pool (an engine that hands a sequence pages in order), lane 0 loads the
// tile with one 128-row box of the run maps mk8/mv8 instead.
__device__ void producer_paged(const PrefillParams &p, const SmemLayout &sm, const WaitCtx &wc, int lane,
                               const CUtensorMap *mq, const CUtensorMap *mk, const CUtensorMap *mv,
                               const CUtensorMap *mk8, const CUtensorMap *mv8) {
    if (p.inject == 1) return;
    const uint64_t pol_q = ptx::policy_evict_first();
    const uint64_t pol_kv = ptx::policy_evict_last();
    int n = 0;            // ring items issued
    int qn[2] = {0, 0};   // Q loads issued per tile (lane 0)
    int u = 0;            // units handed out (lane 0)
    bool ok = true;
    // Lane 0 finds and publishes each unit; the other lanes read it back from
    // the item ring.
    Unit w;
    w.n_kv = -1;
    if (lane == 0) w = next_unit<kPaged>(p, true);
    while (ok) {
        if (lane == 0) ok = publish_unit(sm, wc, u, w);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        __syncwarp();
        if (lane != 0) {
            const volatile int *d = sm.item_ring(u % ITEM_RING);
            w.b = d[0]; w.g = d[1]; w.h[0] = d[2]; w.h[1] = d[3]; w.s0[0] = d[4]; w.s0[1] = d[5]; w.n_kv = d[6];
            w.j_lo = d[7]; w.Sq = d[10]; w.Sk = d[11]; w.q0 = d[12]; w.tb = d[14];
        }
        ++u;
        if (w.n_kv < 0) break;  // end of the list
        Unit nx;  // (lane 0)
        nx.n_kv = -1;
        const int total = 2 * w.n_kv;
        const int n_pages = (w.Sk + 15) / 16;
        const int *row = p.block_table + (int64_t)w.b * p.max_blocks;
        int page_row = p.num_pages * 16;  // this lane's page of the current tile (lanes < 8)
        bool run = false;                 // the current tile's pages are one run in the pool
        // Block-table entries are read one tile ahead (lanes < 8: one page
        // each), so a load's latency never sits between a free slot and the
        // tile's copies; the first tile's are read before the Q loads.
        auto table_entry = [&](int jt) -> int {
            const int page = (w.j_lo + jt) * (BN / 16) + lane;
            return page < n_pages ? row[page] : -1;
        };
        int next_phys = -1;
        if (lane < BN / 16 && total > 0) next_phys = table_entry(0);
        if (lane == 0) {
            for (int t = 0; t < 2 && ok; ++t) {
                if (qn[t] > 0 && !wait_bounded(sm.q_free(t), (qn[t] - 1) & 1, wc, kSiteProducerQ)) {
                    ok = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(sm.q_full(t), TILE_BYTES);
                load_tile(mq, sm.q_tile(t), sm.q_full(t), p.bhsd, t ? w.h[1] : w.h[0],
                          w.q0 + (t ? w.s0[1] : w.s0[0]), w.tb, pol_q);
                ++qn[t];
            }
            if (ok) nx = next_unit<kPaged>(p, false);  // the next unit while this one's Q loads
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
            ok = false;
            break;
        }
        for (int i = 0; i < total + 2; ++i) {
            const int slot = n % NSLOT;
            if (i < total && (i & 1) == 0 && lane < BN / 16) {
                const int page = (w.j_lo + (i >> 1)) * (BN / 16) + lane;
                const int phys = next_phys;
                if ((i >> 1) + 1 < w.n_kv) next_phys = table_entry((i >> 1) + 1);
                const bool ok_page = phys >= 0 && phys < p.num_pages;
                if (!ok_page && page < n_pages) report_status(p.status, kStatusDeviceBounds, kSitePagedTable);
                page_row = ok_page ? phys * 16 : p.num_pages * 16;
            }
            bool got = true;
            if (lane == 0) {
                got = n < NSLOT || wait_bounded(sm.kv_empty(slot), ((n / NSLOT) - 1) & 1, wc, kSiteProducerEmpty);
                if (got) {
                    if (i < total)
                        ptx::mbar_arrive_expect_tx(sm.kv_full(slot), TILE_BYTES);
                    else
                        ptx::mbar_arrive(sm.kv_full(slot));  // an output staging slot
                }
            }
            if (!__shfl_sync(0xffffffffu, got, 0)) {
                ok = false;
                break;
            }
            if (i < total) {
                if ((i & 1) == 0) {
                    // (after the slot wait, which the table loads overlap)
                    const int first = __shfl_sync(0xffffffffu, page_row, 0);
                    const bool in_run =
                        lane >= BN / 16 || (page_row == first + 16 * lane && first < p.num_pages * 16);
                    run = __all_sync(0xffffffffu, in_run);
                }
                // The pool maps are in 8-row groups (see the paged tile layout):
                // a page is one 4 KiB box at group page_row / 8, a run one box of 16.
                if (run) {
                    if (lane == 0)
                        ptx::tma_load_5d_hint(sm.slot(slot), (i & 1) ? mv8 : mk8, sm.kv_full(slot), 0, 0, 0,
                                              page_row / 8, w.g, pol_kv);
                } else if (lane < BN / 16) {
                    ptx::tma_load_5d_hint(sm.slot(slot) + lane * PAGE_BOX_BYTES, (i & 1) ? mv : mk, sm.kv_full(slot),
                                          0, 0, 0, page_row / 8, w.g, pol_kv);
                }
            }
            ++n;
        }
        if (lane == 0) w = nx;
    }
    // On the way out make sure no copy is still writing into shared memory.
    if (lane == 0) {
        for (int t = 0; t < 2; ++t)
            if (qn[t] > 0) drain_wait(sm.q_full(t), (qn[t] - 1) & 1, wc);
        for (int i = max(0, n - NSLOT); i < n; ++i) drain_wait(sm.kv_full(i % NSLOT), (i / NSLOT) & 1, wc);
    }
}

// ------------------------------------------------------------------ MMA issuer

// The issue path is kept to a few integer operations per MMA: each operand
// descriptor is built once per tile and every k-step adds a compile-time
// offset (the start-address field is the low 14 bits, and no step carries out
// of it), so an issuing thread keeps up with the tensor core.
// PAGED: K and V tiles in the 8-row-group layout of the page-pool loads.
template <bool PAGED>
__device__ __forceinline__ void issue_s(uint32_t tmem_s, uint64_t q_desc, uint64_t k_desc) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t qoff = (uint64_t)(((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4);
        const uint64_t koff =
            PAGED ? (uint64_t)(((kk >> 2) * PG_HALF_BYTES + (kk & 3) * 32) >> 4) : qoff;
        ptx::umma_ss(tmem_s, q_desc + qoff, k_desc + koff, IDESC_S, kk > 0);
    }
}

template <bool PAGED>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t v_desc, uint32_t accumulate) {
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
        // 16 keys per step: 8 packed bf16x2 columns of P, 16 rows (2 x 8-row atoms) of V.
        const uint32_t step = PAGED ? 2 * PG_GROUP_BYTES : 2048;
        ptx::umma_ts(tmem_o, tmem_p + kk * 8, v_desc + (uint64_t)((kk * step) >> 4), IDESC_PV,
                     kk > 0 ? 1u : accumulate);
    }
}

// One issuing thread per tile (stream t), in the order
//   S_t(0), then for every K/V tile j:  S_t(j+1), PV_t(j)
// for each unit in turn.  The score tiles go through one shared S buffer in
// the order S_0(0), S_1(0), S_0(1), S_1(1), ... counted across the CTA's
// units (g below is that running index): each is issued once the softmax that
// consumed the one before (the other tile's) has loaded it.  Each group has
// its own s_free barrier: S_1(g) waits for phase g of s_free(0), S_0(g) for
// phase g-1 of s_free(1).  (A single barrier for both would let a stream that
// runs ahead pass on the parity of a phase two back.)
// An issuing thread is held while its products execute, and a P V product
// waits for its tile's whole softmax; with one stream per tile, neither holds
// up the other tile's products, and one thread's waits and commits overlap
// the other's products.
//   S_t(j)  needs Q_t, K_j and the other group's s_free;
//   PV_t(j) needs P_t(j) (p_full[t]) and V_j.
// A ring slot takes one release per stream (a commit after the stream's
// product that reads it).  After a unit's last S product the stream commits
// q_free[t]: once that product has completed, Q_t may be replaced by the next
// unit's, while this unit's last softmax, P V and output still run.
template <int T, bool PAGED>
__device__ void mma_stream(const PrefillParams &p, const SmemLayout &sm, const WaitCtx &wc, uint32_t tmem_base) {
    const uint64_t q_desc = ptx::desc_kmajor_sw128(ptx::smem_addr(sm.q_tile(T)));
    const uint32_t slot0 = ptx::smem_addr(sm.slot(0));
    auto slot_of = [](int n) { return n % NSLOT; };
    auto par_of = [](int n) { return (uint32_t)((n / NSLOT) & 1); };
    int nb = 0;  // ring number of the unit's first K/V item
    int g0 = 0;  // running index of the unit's first S / P V product
    for (int u = 0;; ++u) {
        Unit w;
        if (!read_unit(sm, wc, u, true, w)) return;  // giving up
        ptx::mbar_arrive(sm.item_empty(u % ITEM_RING));
        if (w.n_kv < 0) return;  // end of the list
        if (!wait_spin(sm.q_full(T), (uint32_t)(u & 1), wc, kSiteMmaQ)) return;
        ptx::tc_fence_after();
        // A tile wholly past its sequence's end (the second tile of a unit whose
        // rows all fit in the first: a short query with packed heads, or the odd
        // last row block) keeps the barrier protocol -- its S and P V products
        // are "done" at once and its ring slots released -- without any MMA.
        const bool dead = (T == 0 ? w.s0[0] : w.s0[1]) >= w.Sq;

        auto do_s = [&](int j) -> bool {
            const int g = g0 + j;
            const int item = nb + 2 * j;  // ring item holding K_j
            // the score tile before this one: S_0(g) for S_1(g), S_1(g-1) for S_0(g)
            const int prev = T == 1 ? g : g - 1;
            if (prev >= 0 && !wait_spin(sm.s_free(1 - T), (uint32_t)(prev & 1), wc, kSiteMmaPoll)) return false;
            if (!wait_spin(sm.kv_full(slot_of(item)), par_of(item), wc, kSiteMmaPoll)) return false;
            ptx::tc_fence_after();
            const uint32_t k_addr = slot0 + slot_of(item) * TILE_BYTES;
            // K-major, 128-byte swizzle; 8-row atoms 1 KiB apart, or 2 KiB in the paged layout
            const uint64_t k_desc = PAGED ? ptx::smem_desc(k_addr, 16, PG_GROUP_BYTES, ptx::kLayoutSwizzle128B)
                                          : ptx::desc_kmajor_sw128(k_addr);
            issue_s<PAGED>(tmem_base + TM_S, q_desc, k_desc);
            ptx::umma_commit(sm.s_full(T));
            ptx::umma_commit(sm.kv_empty(slot_of(item)));  // this stream is done with K_j
            if (j == w.n_kv - 1) ptx::umma_commit(sm.q_free(T));  // ... and with Q_t
            return true;
        };
        auto do_pv = [&](int j) -> bool {
            const int item = nb + 2 * j + 1;  // ring item holding V_j
            if (!wait_spin(sm.p_full(T), (uint32_t)((g0 + j) & 1), wc, kSiteMmaPoll)) return false;
            if (!wait_spin(sm.kv_full(slot_of(item)), par_of(item), wc, kSiteMmaPoll)) return false;
            ptx::tc_fence_after();
            const uint32_t v_addr = slot0 + slot_of(item) * TILE_BYTES;
            // MN-major, 128-byte swizzle: the two 64-column halves HALF_BYTES apart
            // and 8-key atoms 1 KiB apart, or 1 KiB and 2 KiB in the paged layout
            const uint64_t v_desc = PAGED ? ptx::smem_desc(v_addr, PG_HALF_BYTES, PG_GROUP_BYTES, ptx::kLayoutSwizzle128B)
                                          : ptx::desc_mnmajor_sw128(v_addr, HALF_BYTES);
            issue_pv<PAGED>(tmem_base + tm_o(T), tmem_base + tm_p(T), v_desc, j > 0 ? 1u : 0u);
            ptx::umma_commit(sm.o_full(T));
            ptx::umma_commit(sm.kv_empty(slot_of(item)));  // this stream is done with V_j
            return true;
        };

        // A dead tile's turns: the same waits, in the same order, then plain
        // arrivals (no products to wait for).  Waiting for each K/V item too
        // keeps its release counting for the item in the slot, so it never
        // runs ahead of the ring.
        auto dead_s = [&](int j) -> bool {
            const int g = g0 + j;
            const int item = nb + 2 * j;
            const int prev = T == 1 ? g : g - 1;
            if (prev >= 0 && !wait_spin(sm.s_free(1 - T), (uint32_t)(prev & 1), wc, kSiteMmaPoll)) return false;
            if (!wait_spin(sm.kv_full(slot_of(item)), par_of(item), wc, kSiteMmaPoll)) return false;
            ptx::mbar_arrive(sm.s_full(T));
            ptx::mbar_arrive(sm.kv_empty(slot_of(item)));
            if (j == w.n_kv - 1) ptx::mbar_arrive(sm.q_free(T));
            return true;
        };
        auto dead_pv = [&](int j) -> bool {
            const int item = nb + 2 * j + 1;
            if (!wait_spin(sm.p_full(T), (uint32_t)((g0 + j) & 1), wc, kSiteMmaPoll)) return false;
            if (!wait_spin(sm.kv_full(slot_of(item)), par_of(item), wc, kSiteMmaPoll)) return false;
            ptx::mbar_arrive(sm.o_full(T));
            ptx::mbar_arrive(sm.kv_empty(slot_of(item)));
            return true;
        };

        if (w.n_kv == 0) {
            ptx::umma_commit(sm.q_free(T));  // nothing to multiply: Q_t is free at once
        } else if (dead) {
            if (!dead_s(0)) return;
            for (int j = 0; j < w.n_kv; ++j) {
                if (j + 1 < w.n_kv && !dead_s(j + 1)) return;
                if (!dead_pv(j)) return;
            }
        } else {
            if (!do_s(0)) return;
            for (int j = 0; j < w.n_kv; ++j) {
                if (j + 1 < w.n_kv && !do_s(j + 1)) return;
                if (!do_pv(j)) return;
            }
        }
        nb += ring_items(w);
        g0 += w.n_kv;
    }
}

// ------------------------------------------------------------------ softmax / epilogue

// Row max of 128 scores: four independent chains of three-input max.
__device__ __forceinline__ float row_max(const float2 (&s)[64]) {
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 64; i += 4) {
        m0 = ptx::max3(m0, s[i].x, s[i].y);
        m1 = ptx::max3(m1, s[i + 1].x, s[i + 1].y);
        m2 = ptx::max3(m2, s[i + 2].x, s[i + 2].y);
        m3 = ptx::max3(m3, s[i + 3].x, s[i + 3].y);
    }
    return ptx::max3(m0, m1, fmaxf(m2, m3));
}

// P = exp2(s * scale_log2 - m_sub) for 128 scores, packed to bf16 pairs;
// returns the fp32 row sum.  Pairs go through the packed fp32 FMA/ADD, the
// sum through four independent accumulators.  MASKED: columns past the row's
// last visible key become exactly 0.
template <bool MASKED>
__device__ __forceinline__ float softmax_tile(const float2 (&s)[64], uint32_t (&pk)[64], float scale_log2,
                                              float m_sub, int kbase, int lim_row) {
    const float2 c2 = make_float2(scale_log2, scale_log2);
    const float2 n2 = make_float2(-m_sub, -m_sub);
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        const float2 t = __ffma2_rn(s[i], c2, n2);
        float2 pp = make_float2(ptx::ex2(t.x), ptx::ex2(t.y));
        if (MASKED) {
            pp.x = (kbase + 2 * i <= lim_row) ? pp.x : 0.f;
            pp.y = (kbase + 2 * i + 1 <= lim_row) ? pp.y : 0.f;
        }
        acc[i & 3] = __fadd2_rn(acc[i & 3], pp);
        pk[i] = ptx::pack_bf16x2(pp.x, pp.y);
    }
    const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
    return a.x + a.y;
}

// Output stores of tile t, one lane of an otherwise idle control warp: for
// each command of softmax group t, the TMA store of the staged tile (both
// 64-column halves), then, once the store has read the slot, the slot goes
// back to the ring.  The group itself moves on to its next unit as soon as the
// command is written, so the store's read of shared memory is off the path
// from one unit's last P to the next unit's first S.
__device__ void store_lane(const SmemLayout &sm, const WaitCtx &wc, int t, const CUtensorMap *mo) {
    // O is written once and not read again here: evict-first, so its dirty
    // lines leave L2 early instead of crowding out K/V and later work.
    const uint64_t pol_o = ptx::policy_evict_first();
    for (int n = 0;; ++n) {
        if (!wait_bounded(sm.stage_ready(t), (uint32_t)(n & 1), wc, kSiteStoreCmd)) return;
        volatile int *cmd = sm.stage_cmd(t);
        const int kind = cmd[0], slot = cmd[1];
        const int c0 = cmd[2], c1 = cmd[3], c2 = cmd[4], c3 = cmd[5];
        ptx::mbar_arrive(sm.stage_taken(t));
        if (kind == 0) return;  // the group has no more tiles
        const uint8_t *stage = sm.slot(slot);
        ptx::tma_store_4d_hint(mo, stage, c0, c1, c2, c3, pol_o);
        ptx::tma_store_4d_hint(mo, stage + HALF_BYTES, c0 + 64, c1, c2, c3, pol_o);
        ptx::bulk_commit_group();
        ptx::bulk_wait_group_read0();
        // one arrival for each of the two streams that release K/V slots
        ptx::mbar_arrive_cnt(sm.kv_empty(slot), 2);
    }
}

// Hand a barrier one arrival for the whole warp once every lane's tensor-memory
// accesses are complete.
__device__ __forceinline__ void warp_arrive(uint64_t *bar, int lane) {
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar);
}

template <int KIND>
__device__ void softmax_wg(const PrefillParams &p, const SmemLayout &sm, const WaitCtx &wc, uint32_t tmem_base,
                           int t, int quarter, int lane, const CUtensorMap *mo) {
    constexpr bool PACKED = KIND != kDense;  // per-sequence offsets: packed batches and paged caches
    constexpr bool PAGED = KIND == kPaged;
    const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lanes = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tS = lanes + TM_S;     // shared score buffer
    const uint32_t tP = lanes + tm_p(t);  // this tile's bf16 P
    const uint32_t tO = lanes + tm_o(t);  // this tile's O accumulator
    const float sl2 = p.scale_log2;
    int nb = 0;  // ring number of the unit's first K/V item
    int g0 = 0;  // running index of the unit's first score tile
    const bool leader = quarter == 0 && lane == 0;
    int n_cmd = 0;  // store commands handed to this tile's store lane
    // The leader writes command n_cmd once the store lane has read the one
    // before (kind 0: no more tiles).
    auto send_cmd = [&](int kind, int slot, const Coord4 &c) -> bool {
        if (n_cmd > 0 && !wait_bounded(sm.stage_taken(t), (uint32_t)((n_cmd - 1) & 1), wc, kSiteStoreCmd))
            return false;
        volatile int *cmd = sm.stage_cmd(t);
        cmd[0] = kind;
        cmd[1] = slot;
        cmd[2] = c.c0;
        cmd[3] = c.c1;
        cmd[4] = c.c2;
        cmd[5] = c.c3;
        ++n_cmd;
        ptx::mbar_arrive(sm.stage_ready(t));
        return true;
    };
    for (int u = 0;; ++u) {
        Unit w;
        const bool got = read_unit(sm, wc, u, false, w);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sm.item_empty(u % ITEM_RING));
        if (!got || w.n_kv < 0) break;  // giving up, or the end of the list (every warp of the group alike)
        // Selects, not a runtime index: an indexed Unit array would live in local memory.
        const int s0 = t ? w.s0[1] : w.s0[0];
        const int h0 = t ? w.h[1] : w.h[0];
        // This thread's row: position `pos` of head `head` (with head packing
        // the tile holds every head of the group at fewer positions).
        int pos = s0 + r, head = h0;
        if (!PACKED && p.pack_heads) {
            const int hr = p.bhsd ? r / p.pack_pos : r % p.G;
            pos = s0 + (p.bhsd ? r % p.pack_pos : r / p.G);
            head = h0 + hr;
        }
        // A tile wholly past the sequence's end computes nothing (its MMA
        // stream issues no products either) and stores nothing.
        const bool dead = s0 >= w.Sq;
        const int lim_row = p.causal ? min(pos + w.Sk - w.Sq, w.Sk - 1) : w.Sk - 1;
        // the tile's first position is its smallest
        const int lim_tile = p.causal ? min(s0 + w.Sk - w.Sq, w.Sk - 1) : w.Sk - 1;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;

        // No rows of the sequence: pass the score and P turns on.  The wait for
        // P V(g-1) stays, as on the live path: it keeps this group from
        // completing p_full(g+1) before the MMA stream has waited for p_full(g)
        // (the stream issues S(g+1) first), which would make that parity wait
        // miss its phase.
        for (int j = 0; dead && j < w.n_kv; ++j) {
            const int g = g0 + j;
            if (!wait_bounded(sm.s_full(t), (uint32_t)(g & 1), wc, kSiteSoftmaxS)) {
                ok = false;
                break;
            }
            warp_arrive(sm.s_free(t), lane);
            if (j > 0 && !wait_bounded(sm.o_full(t), (uint32_t)((g - 1) & 1), wc, kSiteSoftmaxO)) {
                ok = false;
                break;
            }
            warp_arrive(sm.p_full(t), lane);
        }
        for (int j = 0; !dead && j < w.n_kv; ++j) {
            const int g = g0 + j;
            if (!wait_bounded(sm.s_full(t), (uint32_t)(g & 1), wc, kSiteSoftmaxS)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            float2 s[64];
            {
                uint32_t a[32], b[32], c[32], d[32];
                ptx::tmem_ld32(tS + 0, a);
                ptx::tmem_ld32(tS + 32, b);
                ptx::tmem_ld32(tS + 64, c);
                ptx::tmem_ld32(tS + 96, d);
                ptx::tmem_wait_ld();
                // The scores are in registers: release the shared S buffer so the
                // other tile's next Q K^T can start while this tile's softmax runs.
                warp_arrive(sm.s_free(t), lane);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    s[i] = make_float2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
                    s[16 + i] = make_float2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
                    s[32 + i] = make_float2(__uint_as_float(c[2 * i]), __uint_as_float(c[2 * i + 1]));
                    s[48 + i] = make_float2(__uint_as_float(d[2 * i]), __uint_as_float(d[2 * i + 1]));
                }
            }
            const int kbase = (w.j_lo + j) * BN;  // absolute first key of this tile
            const bool masked = kbase + BN - 1 > lim_tile;
            float mx;
            if (masked) {
                // Scores of keys the row may not see take no part in the max.
                float2 sm2[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    sm2[i].x = (kbase + 2 * i <= lim_row) ? s[i].x : -INFINITY;
                    sm2[i].y = (kbase + 2 * i + 1 <= lim_row) ? s[i].y : -INFINITY;
                }
                mx = row_max(sm2);
            } else {
                mx = row_max(s);
            }
            const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * sl2;
            bool need = false;
            float m_new = m_tile;
            if (j > 0) {
                // Past a 2^8 growth, or a new maximum whose P = 2^(m_tile - m_run)
                // would exceed half of the running sum l_run.
                need = m_tile > m_run + RESCALE_LOG2 || (m_tile > m_run && m_tile - m_run > ptx::lg2(l_run) - 1.0f);
                m_new = need ? m_tile : m_run;
            }
            const float alpha = need ? ptx::ex2(m_run - m_new) : 1.f;
            const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
            uint32_t pk[64];
            const float rowsum = masked ? softmax_tile<true>(s, pk, sl2, m_sub, kbase, lim_row)
                                        : softmax_tile<false>(s, pk, sl2, m_sub, kbase, lim_row);
            // P_t(g-1) and O_t are read / written by PV_t(g-1): wait for it before
            // overwriting P_t or rescaling O_t (normally it finished long ago).
            // The previous unit's last P V was waited for by its epilogue.
            if (j > 0) {
                if (!wait_bounded(sm.o_full(t), (uint32_t)((g - 1) & 1), wc, kSiteSoftmaxO)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
            }
            {
                uint32_t lo[32], hi[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    lo[i] = pk[i];
                    hi[i] = pk[32 + i];
                }
                ptx::tmem_st32(tP + 0, lo);
                ptx::tmem_st32(tP + 32, hi);
            }
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                // O still holds the sum over tiles < j scaled by the old max:
                // rescale this warp's 32 rows in place, 64 columns per round trip
                // (two loads in flight per wait).
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
                for (int ch = 0; ch < 4; ch += 2) {
                    uint32_t o[32], o2[32];
                    ptx::tmem_ld32(tO + ch * 32, o);
                    ptx::tmem_ld32(tO + ch * 32 + 32, o2);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 v =
                            __fmul2_rn(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), a2);
                        o[2 * i] = __float_as_uint(v.x);
                        o[2 * i + 1] = __float_as_uint(v.y);
                        const float2 v2 =
                            __fmul2_rn(make_float2(__uint_as_float(o2[2 * i]), __uint_as_float(o2[2 * i + 1])), a2);
                        o2[2 * i] = __float_as_uint(v2.x);
                        o2[2 * i + 1] = __float_as_uint(v2.y);
                    }
                    ptx::tmem_st32(tO + ch * 32, o);
                    ptx::tmem_st32(tO + ch * 32 + 32, o2);
                }
            }
            ptx::tmem_wait_st();
            l_run = l_run * alpha + rowsum;
            m_run = m_new;
            if (PACKED && kbase + BN > w.Sk) {
                // Last tile of a packed or paged sequence: the V rows past its end
                // hold other data (the next sequence's rows, or whatever a page's
                // unused slots contain).  Their P is 0, but 0 * NaN is NaN, so each
                // group zeroes those rows in shared memory once the tile has
                // landed, before releasing its P (the two streams' P V products
                // are not ordered; both groups write the same zeros).
                const int item = nb + 2 * j + 1;
                uint8_t *vt = sm.slot(item % NSLOT);
                if (!wait_bounded(sm.kv_full(item % NSLOT), (uint32_t)((item / NSLOT) & 1), wc, kSiteSoftmaxV)) {
                    ok = false;
                    break;
                }
                if (kbase + r >= w.Sk) {
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    // row r, both halves (dense or paged tile layout)
                    uint8_t *h0 = PAGED ? vt + (r >> 3) * PG_GROUP_BYTES + (r & 7) * 128 : vt + r * 128;
                    uint8_t *h1 = h0 + (PAGED ? PG_HALF_BYTES : HALF_BYTES);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        reinterpret_cast<uint4 *>(h0)[c] = z;
                        reinterpret_cast<uint4 *>(h1)[c] = z;
                    }
                }
                ptx::fence_proxy_async_smem();
            }
            warp_arrive(sm.p_full(t), lane);
        }

        // Epilogue: O / l -> bf16 into this tile's output staging slot of the
        // ring, then a TMA store from there.  Every warp of the group reaches
        // the group barrier once per unit, whether or not it gave up on a wait,
        // and the barrier ANDs everyone's "all well" so that the whole group
        // takes the same decision to go on or to stop.
        if (ok && w.n_kv > 0) ok = wait_bounded(sm.o_full(t), (uint32_t)((g0 + w.n_kv - 1) & 1), wc, kSiteEpilogueO);
        const int o_item = nb + 2 * w.n_kv + t;
        uint8_t *stage = sm.slot(o_item % NSLOT);
        if (ok) ok = wait_bounded(sm.kv_full(o_item % NSLOT), (uint32_t)((o_item / NSLOT) & 1), wc, kSiteEpilogueSlot);
        if (!PACKED && ok && w.part >= 0) {
            // A key-range part of a split unit: its O (normalised within the range)
            // and log-sum-exp go to the workspace in fp32 for the merge kernel.
            ptx::tc_fence_after();
            const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
            const int64_t row = w.ws_row + t * BM + r;
            float4 *dst = reinterpret_cast<float4 *>(p.ws_o + (row * p.split_parts + w.part) * D);
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t o[32];
                ptx::tmem_ld32(tO + ch * 32, o);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float4 x = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                           __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
                    if (!(l_run > 0.f)) x = make_float4(0.f, 0.f, 0.f, 0.f);
                    dst[ch * 8 + i] = x;
                }
            }
            p.ws_lse[row * p.split_parts + w.part] = l_run > 0.f ? (m_run + ptx::lg2(l_run)) * LN2 : -INFINITY;
        } else if (ok && !dead) {
            ptx::tc_fence_after();
            const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t o[32];
                ptx::tmem_ld32(tO + ch * 32, o);
                ptx::tmem_wait_ld();
                uint32_t wv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float2 x = __fmul2_rn(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])),
                                          make_float2(inv, inv));
                    if (!(l_run > 0.f)) x = make_float2(0.f, 0.f);
                    wv[i] = pack_bf16x2_mode(x.x, x.y, p.round_mode);
                }
                // 32 columns = 64 bytes = four 16-byte chunks of the 128-B swizzled row.
                uint8_t *rowp = stage + (ch >> 1) * HALF_BYTES + r * 128;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int cc = (ch & 1) * 4 + kk;
                    *reinterpret_cast<uint4 *>(rowp + ((cc ^ (r & 7)) << 4)) =
                        make_uint4(wv[4 * kk], wv[4 * kk + 1], wv[4 * kk + 2], wv[4 * kk + 3]);
                }
            }
            if (p.lse != nullptr && pos < w.Sq) {
                const float lse = l_run > 0.f ? (m_run + ptx::lg2(l_run)) * LN2 : -INFINITY;
                const int64_t li = PACKED ? (int64_t)head * p.total_q + w.q0 + pos
                                          : ((int64_t)w.b * p.Hq + head) * p.Sq + pos;
                p.lse[li] = lse;
            }
        }
        ptx::tc_fence_before();
        ptx::fence_proxy_async_smem();
        if (!ptx::named_bar_and(1 + t, 128, ok && !*wc.abort_flag)) break;
        bool handed = false;  // the store lane releases the slot
        if (PACKED && s0 + BM > w.Sq) {
            // Last row block of a packed sequence: a full box would spill into the
            // next sequence's rows, so each thread stores its own row (if valid)
            // from the swizzled staging tile; the group then waits for all rows
            // before the slot is handed back.
            if (pos < w.Sq) {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) +
                                                       ((int64_t)(w.q0 + pos) * p.Hq + head) * D);
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    dst[c] = *reinterpret_cast<const uint4 *>(stage + (c >> 3) * HALF_BYTES + r * 128 +
                                                               (((c & 7) ^ (r & 7)) << 4));
            }
            ptx::named_bar_sync(1 + t, 128);
        } else if (leader && s0 < w.Sq && (PACKED || w.part < 0)) {
            // The TMA store goes to the store lane (with head packing the
            // output map's box covers the group's heads).  The staged rows were
            // made visible to the async proxy before the group barrier.
            handed = send_cmd(1, o_item % NSLOT, coord4(p.bhsd, 0, h0, w.q0 + s0, w.tb));
        }
        // Otherwise the slot is free again now (one arrival for each of the two
        // streams that release K/V slots).
        if (leader && !handed) ptx::mbar_arrive_cnt(sm.kv_empty(o_item % NSLOT), 2);
        nb += ring_items(w);
        g0 += w.n_kv;
    }
    if (leader) send_cmd(0, 0, Coord4{0, 0, 0, 0});  // the store lane stops (if it still waits)
}

// ------------------------------------------------------------------ kernel

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                   const __grid_constant__ CUtensorMap map_k8, const __grid_constant__ CUtensorMap map_v8,
                   const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    SmemLayout sm;
    sm.base = smem_raw + ((SMEM_ALIGN - (raw & (SMEM_ALIGN - 1))) & (SMEM_ALIGN - 1));
    sm.bars = reinterpret_cast<uint64_t *>(sm.base + SMEM_TILES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(sm.q_full(t), 1);
            ptx::mbar_init(sm.q_free(t), 1);  // one commit by the tile's issuing stream
        }
        for (int s = 0; s < NSLOT; ++s) {
            ptx::mbar_init(sm.kv_full(s), 1);
            ptx::mbar_init(sm.kv_empty(s), 2);  // one release per issuing stream (or a staging slot's 2)
        }
        // Softmax-side barriers take one arrival per warp (lane 0, after the
        // warp's tcgen05 fence and __syncwarp).
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(sm.s_full(t), 1);
            ptx::mbar_init(sm.p_full(t), 4);
            ptx::mbar_init(sm.o_full(t), 1);
            ptx::mbar_init(sm.s_free(t), 4);
        }
        ptx::mbar_init(sm.fin(), 2);  // one commit per issuing stream
        for (int i = 0; i < ITEM_RING; ++i) {
            ptx::mbar_init(sm.item_full(i), 1);
            ptx::mbar_init(sm.item_empty(i), ITEM_READERS);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(sm.stage_ready(t), 1);
            ptx::mbar_init(sm.stage_taken(t), 1);
        }
        *sm.abort_flag() = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&map_q);
        ptx::prefetch_tensormap(&map_k);
        ptx::prefetch_tensormap(&map_v);
        ptx::prefetch_tensormap(&map_o);
    }
    if (warp == 1) {
        ptx::tmem_alloc(sm.tmem_slot(), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot();
    const WaitCtx wc{sm.abort_flag(), p.status, p.budget_ns};

    if (warp < 4) {
        ptx::setmaxnreg_dec<REGS_CONTROL>();
        if (warp == 0) {
            if (KIND == kPaged)
                producer_paged(p, sm, wc, lane, &map_q, &map_k, &map_v, &map_k8, &map_v8);
            else if (lane == 0)
                producer<KIND>(p, sm, wc, &map_q, &map_k, &map_v);
        } else if (warp == 3) {
            if (lane < 2) store_lane(sm, wc, lane, &map_o);
        } else if (warp == 1 || warp == 2) {
            if (lane == 0) {
                if (warp == 1)
                    mma_stream<0, KIND == kPaged>(p, sm, wc, tmem_base);
                else
                    mma_stream<1, KIND == kPaged>(p, sm, wc, tmem_base);
                // Whatever happened, wait until every product issued (by
                // either stream) has completed before tensor memory is released.
                ptx::umma_commit(sm.fin());
                drain_wait(sm.fin(), 0, wc);
            }
        }
        __syncwarp();
    } else {
        ptx::setmaxnreg_inc<REGS_SOFTMAX>();
        const int t = (warp - 4) >> 2;
        softmax_wg<KIND>(p, sm, wc, tmem_base, t, warp & 3, lane, &map_o);
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // A dependent merge kernel may be scheduled now; it waits for this grid.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, 512);
    }
    if (threadIdx.x == 0 && (int)gridDim.x < p.n_items) {
        // The last CTA to finish (every producer has stopped claiming by then)
        // returns the launch's counter to zero for the next launch that uses it.
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
        }
    }
}

}  // namespace g1

int prefill_smem_bytes() { return (int)(g1::SMEM_TILES + g1::SMEM_MISC + g1::SMEM_ALIGN); }

cudaError_t launch_prefill(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                           const CUtensorMap &mo, const CUtensorMap &mk8, const CUtensorMap &mv8,
                           const PrefillParams &p, int num_ctas, cudaStream_t stream) {
    const int smem = prefill_smem_bytes();
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(g1::prefill_kernel<g1::kDense>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(g1::prefill_kernel<g1::kPacked>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(g1::prefill_kernel<g1::kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    // One instantiation per kind of launch, each with only its own paths.
    if (p.block_table != nullptr)
        g1::prefill_kernel<g1::kPaged><<<num_ctas, g1::NUM_THREADS, smem, stream>>>(mq, mk, mv, mo, mk8, mv8, p);
    else if (p.cu_q != nullptr)
        g1::prefill_kernel<g1::kPacked><<<num_ctas, g1::NUM_THREADS, smem, stream>>>(mq, mk, mv, mo, mk8, mv8, p);
    else
        g1::prefill_kernel<g1::kDense><<<num_ctas, g1::NUM_THREADS, smem, stream>>>(mq, mk, mv, mo, mk8, mv8, p);
    return cudaGetLastError();
}

int prefill_grid(int n_items, int num_sms) { return n_items < num_sms ? n_items : num_sms; }

int prefill_num_units(const PrefillParams &p) {
    if (p.pack_heads) return p.B * p.Hkv * p.n_pk;
    if (p.pair_heads) return p.B * p.Hkv * (p.G / 2) * p.n_m;
    return p.B * p.Hq * ((p.n_m + 1) / 2);
}

// Tail split (the Flash-Decoding style split of the MoonMath page, applied to
// the prefill's last wave).  CTAs are dispatched in index order and one fits
// per SM, so the last units % num_sms units run as a partial final wave.
// When every unit has the same length (non-causal) and that wave would leave
// SMs idle, each of those units is cut into parts key ranges (at least 4 K/V
// tiles each) so that the last wave fills the SMs.  Causal launches run
// longest units first and end on short units, so they are left whole.
size_t prefill_split_plan(const PrefillParams &p, int num_sms, int *split_units, int *split_parts) {
    *split_units = 0;
    *split_parts = 1;
    const int units = prefill_num_units(p);
    const int n_kv = (p.Sk + g1::BN - 1) / g1::BN;
    if (p.causal || num_sms < 2 || n_kv < 8) return 0;
    const int tail = units % num_sms;
    if (tail == 0) return 0;
    int parts = num_sms / tail;
    if (parts > n_kv / 4) parts = n_kv / 4;
    if (parts < 2) return 0;
    *split_units = tail;
    *split_parts = parts;
    const size_t rows = (size_t)tail * 2 * g1::BM;
    size_t o_bytes = rows * parts * g1::D * 4;
    o_bytes = (o_bytes + 255) & ~(size_t)255;
    size_t l_bytes = rows * parts * 4;
    l_bytes = (l_bytes + 255) & ~(size_t)255;
    return o_bytes + l_bytes;
}

namespace g1 {

// One CTA per row of the split units, one thread per head-dim element: merge
// the key-range partials in part order (deterministic) and write the row of O
// in q's layout, rounded to bf16, and its log-sum-exp.
__global__ void __launch_bounds__(D) merge_kernel(__nv_bfloat16 *__restrict__ out, const PrefillParams p) {
    // Launched as a programmatic dependent of the prefill kernel: wait here
    // until that grid has completed and its partials are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int row = blockIdx.x;  // within the split units
    const int su = row / (2 * BM);
    const int t = (row / BM) & 1;
    const int r = row % BM;
    const Unit w = unit_coords(p, p.n_full_units + su);
    int s = (t ? w.s0[1] : w.s0[0]) + r;
    int h = t ? w.h[1] : w.h[0];
    if (p.pack_heads) {  // row r of a packed tile: its position and head
        s = (t ? w.s0[1] : w.s0[0]) + (p.bhsd ? r % p.pack_pos : r / p.G);
        h += p.bhsd ? r / p.pack_pos : r % p.G;
    }
    if (s >= p.Sq) return;
    const int e = threadIdx.x;
    const float *ls = p.ws_lse + (int64_t)row * p.split_parts;
    float M = -INFINITY;
    for (int k = 0; k < p.split_parts; ++k) M = fmaxf(M, ls[k]);
    float total = 0.f, o = 0.f;
    if (M != -INFINITY) {
        for (int k = 0; k < p.split_parts; ++k) {
            const float wk = ptx::ex2((ls[k] - M) * 1.4426950408889634f);
            total += wk;
            o = fmaf(wk, p.ws_o[((int64_t)row * p.split_parts + k) * D + e], o);
        }
    }
    const int64_t off = p.bhsd ? (((int64_t)w.b * p.Hq + h) * p.Sq + s) * D : (((int64_t)w.b * p.Sq + s) * p.Hq + h) * D;
    reinterpret_cast<uint16_t *>(out)[off + e] = bf16_bits_mode(total > 0.f ? o / total : 0.f, p.round_mode);
    if (e == 0 && p.lse != nullptr)
        p.lse[((int64_t)w.b * p.Hq + h) * p.Sq + s] = total > 0.f ? M + ptx::lg2(total) * LN2 : -INFINITY;
}

}  // namespace g1

cudaError_t launch_prefill_merge(void *out, const PrefillParams &p, cudaStream_t stream) {
    if (p.split_units == 0) return cudaSuccess;
    // Programmatic dependent launch (see launch_lse_merge): the merge CTAs are
    // scheduled while the prefill's last CTAs finish.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.split_units * 2 * g1::BM));
    cfg.blockDim = dim3(g1::D);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, g1::merge_kernel, static_cast<__nv_bfloat16 *>(out), p);
}

}  // namespace attn
