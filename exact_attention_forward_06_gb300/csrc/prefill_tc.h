// prefill_tc.h -- host-side interface of the tensor-core prefill kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

struct PrefillParams {
    int B, Hq, Hkv, Sq, Sk;  // a packed batch: Sq, Sk = the largest sequence lengths
    int G;             // Hq / Hkv
    int causal;        // bottom-right causal mask
    int bhsd;          // 1: tensors are [B][H][S][d]; 0: [B][S][H][d]
    float scale_log2;  // softmax scale * log2(e)
    float *lse;        // [B][Hq][Sq] or nullptr
    int n_m;           // ceil(Sq / 128)
    int pair_heads;    // 1: a unit is two heads of one KV group at the same rows
    int pack_heads;    // 1: a Q tile is pack_pos positions x all G heads of one KV group
                       //    (row r: position r / G, head r % G in BSHD; head r / pack_pos,
                       //    position r % pack_pos in BHSD); dense launches only
    int pack_pos;      // 128 / G when packing
    int n_pk;          // units per (batch, KV group) when packing: ceil(Sq / (2 * pack_pos))
    unsigned *status;  // device status word [code, site]
    uint64_t budget_ns;
    int inject;        // 1: producer issues nothing (fault-injection test)
    int round_mode;    // RoundMode of the bf16 output (epilogue and merge)
    // Tail split: units [0, n_full_units) run whole; each of the following
    // split_units units is cut into split_parts key ranges, one CTA each, whose
    // fp32 partials go to ws_o [split_units*256][split_parts][128] and
    // ws_lse [split_units*256][split_parts] and are merged afterwards.
    int prefetch_ahead;  // > 0: L2-prefetch the Q tiles of a CTA's next unit (or of the
                         // unit this many items ahead when every CTA has one unit)
    int n_items;         // work items: whole units, then the parts of split units; with
                         // fewer CTAs than items each CTA claims the next free item
    unsigned *sched;     // [2] device counters of this launch: next item, CTAs done (both
                         // zero at launch; the last CTA resets them)
    int n_full_units;
    int kv_major;        // 1: units ordered by sequence and KV head (see unit_coords)
    int seq_group;       // > 0 (with kv_major = 0): sequences taken seq_group at a time,
                         // row block first within each group (see unit_coords)
    int split_units;
    int split_parts;
    float *ws_o;
    float *ws_lse;
    // Packed variable-length batch (cu_q == nullptr for a dense batch):
    // sequence b owns rows cu_q[b] .. cu_q[b+1]-1 of q [total_q][Hq][d] and
    // cu_k[b] .. cu_k[b+1]-1 of k, v [total_k][Hkv][d]; lse is [Hq][total_q].
    // Partial last row blocks are stored row by row through out.
    const int *cu_q;
    const int *cu_k;
    int total_q, total_k;
    void *out;
    // Paged K/V (block_table == nullptr: K and V are tensors): sequence b has
    // seqlens_k[b] keys, key t in slot t % 16 of page block_table[b][t / 16]
    // of the pools [num_pages][16][Hkv][d]; the maps for K and V are then 5-D
    // maps over the pools (see make_map_pool_groups) with one whole page of
    // one KV head per box.  Queries are packed as above (cu_q); cu_k is unused.
    const int *block_table;
    const int *seqlens_k;
    int max_blocks, num_pages;
};

int prefill_smem_bytes();
int prefill_num_units(const PrefillParams &p);
// Grid for n_items work items on a device with num_sms SMs: one CTA per SM,
// each looping over its items, when there are more items than SMs.
int prefill_grid(int n_items, int num_sms);
// mk8/mv8: paged K/V only, the same pool maps with 128-row boxes (a run of 8
// consecutive pages); pass mk/mv otherwise.  num_ctas <= p.n_items: with
// fewer CTAs than items each CTA loops over its items (persistent grid).
cudaError_t launch_prefill(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                           const CUtensorMap &mo, const CUtensorMap &mk8, const CUtensorMap &mv8,
                           const PrefillParams &p, int num_ctas, cudaStream_t stream);
// Merge of the tail-split partials into out (q's layout) and lse.
cudaError_t launch_prefill_merge(void *out, const PrefillParams &p, cudaStream_t stream);
// Tail-split plan for a shape on a device with num_sms SMs: split_units and
// split_parts (0 / 1 when no split is worth it) and the workspace it needs.
size_t prefill_split_plan(const PrefillParams &p, int num_sms, int *split_units, int *split_parts);

// Plain SIMT kernel, one warp per query row (debugging cross-check).
cudaError_t launch_prefill_simple(const void *q, const void *k, const void *v, void *out, float *lse,
                                  const PrefillParams &p, cudaStream_t stream);

// Paged decode: split kernel + log-sum-exp merge.
struct DecodeParams {
    const void *q;            // [B][Hq][d] bf16
    const int32_t *block_table;
    const int32_t *seqlens;
    void *out;                // [B][Hq][d] bf16
    float *lse;               // [B][Hq] or nullptr
    float *o_part;            // [B*Hq][nsplit][d] fp32
    float *lse_part;          // [B*Hq][nsplit] fp32
    int B, Hq, Hkv, G, num_pages, max_blocks, nsplit, pages_per_split;
    float scale_log2;
    unsigned *status;
    uint64_t budget_ns;
    // Fused append (k_new == nullptr: none): the token k_new/v_new [B][Hkv][d]
    // is written at position seqlens[b] of the pools and attended to as well.
    const void *k_new;
    const void *v_new;
    void *k_pool;
    void *v_pool;
};

void decode_split_plan(int B, int Hq, int max_blocks, int *nsplit, int *pages_per_split);
cudaError_t launch_decode(const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                          cudaStream_t stream);
cudaError_t launch_lse_merge(const float *o_parts, const float *lse_parts, void *out, float *lse, int rows,
                             int nsplit, int round_mode, cudaStream_t stream);

// Tensor-core layout self-test.
cudaError_t launch_selftest_umma(const CUtensorMap &ma, const CUtensorMap &mb, const void *a, float *c, int mode,
                                 unsigned *status, uint64_t budget_ns, cudaStream_t stream);

}  // namespace attn
