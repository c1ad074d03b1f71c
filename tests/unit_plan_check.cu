// unit_plan_check.cu -- host-side checks of the prefill work-unit plan and the
// key-split plans, against brute force.  Compiled by tests/test_unit_plan.py
// with nvcc (the kernels are compiled too but never launched) and run on the
// CPU.  Exits 0 when every check passes; prints the first failure otherwise.
//
//   1. unit_coords is a bijection onto the (batch, head, 128-row block) tiles
//      of a launch, in both orders (row block first, and sequence and KV
//      head first), for even and odd group sizes, causal or not;
//   2. a causal unit's K/V tile count is the number of 128-key tiles up to the
//      last key its lowest row may see (bottom-right alignment), and every
//      tile of a non-causal unit;
//   3. the tail-split plan cuts the partial last wave into parts of at least
//      4 K/V tiles that fill it, only for non-causal launches;
//   4. the decode split plan covers every page with 16 to 256 pages a split;
//   5. with GQA head packing, the units cover every (batch, head, position)
//      of a launch exactly once, a tile holding the 128 / G positions of all
//      G heads of one KV group, and a causal unit's K/V tile count is again
//      the brute-force count for its last position.
#include <cstdio>
#include <cstdlib>
#include <set>
#include <tuple>
#include <vector>

#include "../exact_attention_forward_06_gb300/csrc/prefill_tc.cu"
#include "../exact_attention_forward_06_gb300/csrc/decode.cu"

static int failures = 0;
#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            if (failures++ < 10) {                        \
                std::printf("FAIL %s:%d: ", __FILE__, __LINE__); \
                std::printf(__VA_ARGS__);                 \
                std::printf("\n");                        \
            }                                             \
        }                                                 \
    } while (0)

static attn::PrefillParams params(int B, int Hq, int Hkv, int Sq, int Sk, bool causal, int kv_major) {
    attn::PrefillParams p{};
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Sq = Sq;
    p.Sk = Sk;
    p.G = Hq / Hkv;
    p.causal = causal ? 1 : 0;
    p.n_m = (Sq + 127) / 128;
    p.pair_heads = p.G % 2 == 0 ? 1 : 0;
    p.kv_major = kv_major;
    p.split_parts = 1;
    p.n_full_units = attn::prefill_num_units(p);
    p.n_items = p.n_full_units;
    return p;
}

// Brute-force K/V tile count of a causal unit: tiles up to the last key the
// unit's lowest (largest-index) valid row may see.
static int brute_n_kv(const attn::PrefillParams &p, int s_lo, int s_hi) {
    const int n_full = (p.Sk + 127) / 128;
    if (!p.causal) return n_full;
    int last_row = -1;
    for (int s = s_lo; s < s_hi && s < p.Sq; ++s) last_row = s;
    const int last_key = last_row + p.Sk - p.Sq;
    if (last_row < 0 || last_key < 0) return 0;
    const int t = last_key / 128 + 1;
    return t < n_full ? t : n_full;
}

static void check_units(int B, int Hq, int Hkv, int Sq, int Sk, bool causal, int kv_major, int seq_group = 0) {
    attn::PrefillParams p = params(B, Hq, Hkv, Sq, Sk, causal, kv_major);
    p.seq_group = seq_group;
    const int units = attn::prefill_num_units(p);
    std::set<std::tuple<int, int, int>> seen;  // (b, head, row block)
    for (int u = 0; u < units; ++u) {
        const attn::g1::Unit w = attn::g1::unit_coords(p, u);
        CHECK(w.b >= 0 && w.b < B, "unit %d: batch %d", u, w.b);
        CHECK(w.g == w.h[0] / p.G && w.g == w.h[1] / p.G, "unit %d: heads %d %d not of group %d", u, w.h[0],
              w.h[1], w.g);
        int lo = 1 << 30, hi = -1;
        for (int t = 0; t < 2; ++t) {
            if (w.s0[t] >= Sq) continue;  // second tile of an odd last pair
            CHECK(w.s0[t] % 128 == 0, "unit %d: row %d", u, w.s0[t]);
            const auto key = std::make_tuple(w.b, w.h[t], w.s0[t] / 128);
            CHECK(seen.insert(key).second, "unit %d: tile (b %d, h %d, block %d) twice", u, w.b, w.h[t],
                  w.s0[t] / 128);
            lo = w.s0[t] < lo ? w.s0[t] : lo;
            hi = w.s0[t] + 128 > hi ? w.s0[t] + 128 : hi;
        }
        // both tiles of a unit share its K/V range: check against the larger rows
        CHECK(w.n_kv == brute_n_kv(p, lo, hi), "unit %d (causal %d, Sq %d, Sk %d): n_kv %d, expected %d", u,
              (int)causal, Sq, Sk, w.n_kv, brute_n_kv(p, lo, hi));
    }
    const size_t tiles = (size_t)B * Hq * p.n_m;
    CHECK(seen.size() == tiles, "B %d Hq %d Hkv %d Sq %d: %zu tiles covered of %zu", B, Hq, Hkv, Sq, seen.size(),
          tiles);
}

static void check_packed_units(int B, int Hq, int Hkv, int Sq, int Sk, bool causal, int kv_major) {
    attn::PrefillParams p = params(B, Hq, Hkv, Sq, Sk, causal, kv_major);
    p.pack_heads = 1;
    p.pack_pos = 128 / p.G;
    p.n_pk = (Sq + 2 * p.pack_pos - 1) / (2 * p.pack_pos);
    const int units = attn::prefill_num_units(p);
    const int P = p.pack_pos;
    std::set<std::tuple<int, int, int>> seen;  // (b, head, position)
    for (int u = 0; u < units; ++u) {
        const attn::g1::Unit w = attn::g1::unit_coords(p, u);
        CHECK(w.b >= 0 && w.b < B && w.g >= 0 && w.g < Hkv, "packed unit %d: batch %d group %d", u, w.b, w.g);
        CHECK(w.h[0] == w.g * p.G && w.h[1] == w.g * p.G, "packed unit %d: first heads %d %d", u, w.h[0], w.h[1]);
        CHECK(w.s0[1] == w.s0[0] + P, "packed unit %d: tiles at %d and %d", u, w.s0[0], w.s0[1]);
        int lo = 1 << 30, hi = -1;
        for (int t = 0; t < 2; ++t)
            for (int r = 0; r < 128; ++r) {  // row r of tile t, in the BSHD order (head fastest)
                const int pos = w.s0[t] + r / p.G, head = w.h[t] + r % p.G;
                if (pos >= Sq) continue;
                CHECK(seen.insert(std::make_tuple(w.b, head, pos)).second, "packed unit %d: (b %d, h %d, s %d) twice",
                      u, w.b, head, pos);
                lo = pos < lo ? pos : lo;
                hi = pos + 1 > hi ? pos + 1 : hi;
            }
        if (hi > lo)
            CHECK(w.n_kv == brute_n_kv(p, lo, hi), "packed unit %d (causal %d, Sq %d, Sk %d): n_kv %d, expected %d",
                  u, (int)causal, Sq, Sk, w.n_kv, brute_n_kv(p, lo, hi));
    }
    CHECK(seen.size() == (size_t)B * Hq * Sq, "packed B %d Hq %d Hkv %d Sq %d: %zu rows covered of %zu", B, Hq, Hkv,
          Sq, seen.size(), (size_t)B * Hq * Sq);
}

static void check_split_plan(int B, int Hq, int Hkv, int Sq, int Sk, bool causal, int sms) {
    const attn::PrefillParams p = params(B, Hq, Hkv, Sq, Sk, causal, 0);
    int su = -1, parts = -1;
    const size_t bytes = attn::prefill_split_plan(p, sms, &su, &parts);
    const int units = attn::prefill_num_units(p);
    const int n_kv = (Sk + 127) / 128;
    if (su == 0) {
        CHECK(parts == 1 && bytes == 0, "no split but parts %d bytes %zu", parts, bytes);
        return;
    }
    CHECK(!causal, "causal launch split");
    CHECK(su == units % sms, "split units %d, tail %d", su, units % sms);
    CHECK(parts >= 2 && n_kv / parts >= 4, "parts %d for %d tiles", parts, n_kv);
    CHECK(su * parts <= sms, "tail of %d x %d parts overfills %d SMs", su, parts, sms);
    CHECK(bytes >= (size_t)su * 256 * parts * 129 * 4, "workspace %zu too small", bytes);
}

static void check_decode_plan(int B, int Hq, int max_blocks) {
    int ns = 0, pps = 0;
    attn::decode_split_plan(B, Hq, max_blocks, &ns, &pps);
    CHECK(pps >= 16 && pps <= 256, "pages per split %d", pps);
    CHECK((long)ns * pps >= max_blocks && (long)(ns - 1) * pps < max_blocks, "%d splits of %d for %d pages", ns,
          pps, max_blocks);
}

int main() {
    const bool tf[2] = {false, true};
    for (bool causal : tf)
        for (int kv_major = 0; kv_major < 2; ++kv_major) {
            check_units(4, 32, 8, 4096, 4096, causal, kv_major);  // GQA, paired heads
            check_units(1, 32, 1, 1000, 1000, causal, kv_major);  // MQA, ragged last block
            check_units(2, 12, 12, 1000, 700, causal, kv_major);  // G = 1: pairs of row blocks, odd n_m
            check_units(3, 6, 2, 300, 520, causal, kv_major);     // G = 3, Sk > Sq
            check_units(2, 8, 2, 520, 130, causal, kv_major);     // Sk < Sq: rows that see no key
            check_units(5, 2, 1, 1, 1, causal, kv_major);         // single rows and keys
            check_units(2, 4, 4, 129, 129, causal, kv_major);
            if (kv_major == 0)
                for (int sg : {1, 2, 3, 5}) {  // sequences in groups, the last group shorter
                    check_units(7, 32, 8, 1000, 1000, causal, 0, sg);
                    check_units(5, 3, 1, 700, 900, causal, 0, sg);
                }
            check_packed_units(4, 32, 8, 4096, 4096, causal, kv_major);  // G = 4: 32 positions a tile
            check_packed_units(1, 32, 1, 1000, 1000, causal, kv_major);  // MQA: 4 positions a tile
            check_packed_units(3, 16, 8, 97, 300, causal, kv_major);     // G = 2, ragged, Sk > Sq
            check_packed_units(2, 64, 8, 5, 33, causal, kv_major);       // G = 8, a few queries
            check_packed_units(2, 16, 2, 300, 100, causal, kv_major);    // Sk < Sq: rows that see no key
        }
    for (int sms : {132, 148, 152})
        for (bool causal : tf) {
            check_split_plan(sms + 8, 1, 1, 256, 2048, causal, sms);
            check_split_plan(sms + 8, 2, 1, 256, 1024, causal, sms);
            check_split_plan(2, 12, 12, 32760, 32760, causal, sms);
            check_split_plan(2, 12, 12, 32760, 512, causal, sms);
            check_split_plan(4, 32, 8, 4096, 4096, causal, sms);
        }
    for (int B : {1, 2, 3, 32, 100})
        for (int Hq : {1, 4, 8, 32, 64})
            for (int mb : {1, 15, 16, 17, 64, 512, 513, 4096}) check_decode_plan(B, Hq, mb);
    if (failures) {
        std::printf("%d check(s) failed\n", failures);
        return 1;
    }
    std::printf("unit plan: all checks passed\n");
    return 0;
}
