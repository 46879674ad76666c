// plan.cuh -- the work plan of the tensor-core decode attention, built on the
// device from req_idx / seq_lens / topk_idx (no host reads, so the call stays
// graph safe), and its layout inside the caller's workspace.
//
//   group  a run of consecutive query rows of one request (at most gmax rows):
//          the draft tokens of a verification row, which share every K/V page
//   pair   (group, kv head): its block list is the union of the blocks its
//          rows selected, ascending, each with the mask of rows that selected
//          it and its page id (blocks whose page lies outside the pool are
//          dropped here).  When every kv head shares one selection the list
//          is built once per group.
//   unit   a contiguous chunk of a pair's block list: the work item of one CTA;
//          a pair split over several units leaves per-unit partials (running
//          max, sum, unnormalised output) that the last unit to finish merges.
//          Units are full chunks of `chunk` blocks plus one remainder per
//          pair; the table lists the full chunks first, then the remainders by
//          decreasing size (longest work is claimed first)
//
// Two launches build it: the list kernel (one warp per list) writes the block
// lists, their lengths and the group starts; the unit kernel cuts the lists
// into the unit table on one CTA while its other CTAs convert the queries.
#pragma once

#include <stdint.h>

#include "spd_internal.cuh"

namespace spd {

struct PlanHeader {
    int32_t status;        // bit 0: an attention wait timed out
    int32_t n_groups;
    int32_t n_pairs;
    int32_t n_units;
    int32_t chunk;         // blocks per unit
    int32_t partial_rows;  // partial rows in use
    int32_t gmax;
    int32_t next_unit;     // work counter of the attention kernel (units claimed so far)
    int32_t reserved[56];
};
static_assert(sizeof(PlanHeader) == 256, "header is one 256-byte line");

struct PlanEntry {
    int32_t page;
    uint16_t block;
    uint16_t mask;  // bit j: row j of the group selected the block
};

// Everything a CTA needs about its work item, in one 32-byte record.
struct PlanUnit {
    int32_t entry;      // first block-list entry (index into the entry array)
    int32_t count;      // entries
    int32_t part_row;   // first partial row, -1 when the pair is not split
    int32_t pair;       // group * Hkv + kv head
    int32_t t0;         // first query row of the group
    int16_t nt;         // rows in the group
    int16_t h;          // kv head
    int32_t part_base;  // first partial row of the pair's first unit
    int32_t n_split;    // units of the pair
};
static_assert(sizeof(PlanUnit) == 32, "unit record is 32 bytes");

constexpr int kPlanThreads = 512;
constexpr int kPlanMaxT = 4096;   // query rows the one-CTA planner handles
constexpr int kPlanMaxNB = 256;   // page-table capacity of the fast path
constexpr int kUnitExtra = 8192;
constexpr int kPartialStride = 4; // floats after the D output values: max, sum, pad
constexpr int kQueryTerms = 3;    // E4M3 terms per query element (12 significant bits)

// Byte layout of the workspace for capacities (T, Hq, Hkv, D, NB).
struct PlanLayout {
    size_t header, gstart, lcount, lists, units, counters, partials, qterms, cfac, total;
    int64_t unit_cap, rows_cap, pair_cap;

    __host__ __device__ static size_t align(size_t x) { return (x + 255) / 256 * 256; }

    PlanLayout() = default;

    __host__ __device__ PlanLayout(int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t NB) {
        pair_cap = T * Hkv;
        unit_cap = pair_cap + kUnitExtra;
        rows_cap = 2 * T * Hq + 16384;
        size_t off = 0;
        header = off;   off += align(sizeof(PlanHeader));
        gstart = off;   off += align(sizeof(int32_t) * (size_t)(T + 1));
        lcount = off;   off += align(sizeof(int32_t) * (size_t)(pair_cap > 0 ? pair_cap : 1));
        lists = off;    off += align(sizeof(PlanEntry) * (size_t)(pair_cap > 0 ? pair_cap : 1) * (size_t)NB);
        units = off;    off += align(sizeof(PlanUnit) * (size_t)unit_cap);
        counters = off; off += align(sizeof(int32_t) * (size_t)(pair_cap > 0 ? pair_cap : 1));
        partials = off; off += align(sizeof(float) * (size_t)rows_cap * (size_t)(D + kPartialStride));
        qterms = off;   off += align((size_t)kQueryTerms * (size_t)(T > 0 ? T : 1) * (size_t)Hq * (size_t)D);
        cfac = off;     off += align(sizeof(float) * (size_t)(T > 0 ? T : 1) * (size_t)Hq);
        total = off;
    }
};

struct PlanArgs {
    const int32_t *ri;
    int64_t ri_s0;
    const int32_t *sl;
    int64_t sl_s0;
    const int32_t *bt;
    int64_t bt_s0, bt_s1;
    const int32_t *tk;  // nullptr: dense
    int64_t tk_s0, tk_s1, tk_s2;
    int32_t T, R, NB, K, Hkv, G, gmax;
    int32_t heads_built;  // block lists per group: 1 when every kv head shares the selection, else Hkv
    int32_t list_ctas;    // CTAs of the list kernel
    int64_t P;
    int32_t num_ctas;
    char *ws;
    PlanLayout lay;
    // query conversion (the other CTAs of the unit launch)
    const void *q;
    int64_t q_s0, q_s1, q_s2;
    int32_t q_dt, Hq;
    float zscale;  // sm_scale * k_scale * log2(e)
};

// Fills heads_built and list_ctas for the call; false when the planner's
// shared memory cannot hold its per-row state (the fast path is then not
// taken).
bool plan_configure(PlanArgs *a);

// The two launches (programmatic stream serialisation: each waits for the
// previous kernel of the stream before touching memory and lets the next one
// start its prologue early).  The unit kernel's CTAs from 1 on write each
// query row as E4M3 terms (qterms[term][t][hq][d], with the row scaled by a
// power of two into [128, 256); two terms for bf16 queries, three otherwise)
// and its logit factor cfac[t][hq] = zscale / scale.
cudaError_t launch_prepare(const PlanArgs &a, int conv_ctas, cudaStream_t stream);

}  // namespace spd
