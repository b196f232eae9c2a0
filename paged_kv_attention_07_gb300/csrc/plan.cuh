// plan.cuh -- workspace layout and work lists of one pka_paged_attn_forward.
//
// The planner kernel turns the device metadata (query_start_loc, seq_lens)
// into work lists; the compute kernels are persistent and pull units from
// those lists through atomic counters, so no host round trip is needed.
//
//   decode:  pairs (request, split) of `dec_split_len` keys each; a unit is a
//            pair times one KV head (GQA) or one head group (MLA).
//   prefill/extend: items (request, pair of query tiles, slot); slot 0 is the new
//            tokens over their own keys (causal), slot c >= 1 is context chunk
//            c - 1 (the pages' chunked-context loop, run as independent
//            items); a unit is an item times one query head. Items are
//            sorted by cost, heaviest first.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace pka {

constexpr int kMaxRequests = 4096;     // planner keeps per-request metadata in smem
constexpr int kDecodeMinSplit = 256;   // fewest keys per GQA decode split
constexpr int kFaBlockM = 128;         // query rows per prefill/extend query tile (TMEM lanes)
constexpr int kFaItemTiles = 2;        // query tiles per prefill/extend item
constexpr int kFaItemRows = kFaBlockM * kFaItemTiles;
constexpr int kFaBlockN = 128;         // keys per prefill/extend tile (cost unit)
constexpr int kCostBuckets = 1024;

struct PlanHeader {
    int32_t err;            // device error word (PKA_DEVERR_*), offset 0 of the workspace
    int32_t dec_split_len;  // keys per decode split
    int32_t dec_num_pairs;
    int32_t fa_num_items;
    int32_t dec_counter;    // dynamic-scheduling counters, zeroed by the planner
    int32_t fa_counter;
    int32_t ext_rows;
    int32_t reserved[57];
};
static_assert(sizeof(PlanHeader) == 256, "plan header is one 256-byte line");

struct Layout {
    size_t off_dec_pairs, off_dec_first, off_dec_nsplit, off_fa_items, off_ext_base;
    size_t off_dec_part_o, off_dec_part_lse, off_ext_part_o, off_ext_part_lse;
    // 8-bit cache with extends: the extends' context gathered as bf16 code
    // values, ctx_nblk blocks of 128 rows per extend, and its block table
    size_t off_ctx_k, off_ctx_v, off_ctx_bt;
    size_t total;
    int dec_pair_cap, fa_item_cap, ext_row_cap, dec_target_units, ctx_nblk;
};

struct PlanParams {
    const int32_t* qsl;
    const int32_t* seq_lens;
    int num_decodes, num_extends, num_prefills, num_tokens;
    int max_query_len, max_seq_len, max_blocks_per_req, block_size, chunk;
    int dec_units_per_pair;  // kv heads (GQA) or head groups (MLA) per pair
    int dec_target_units;
    int dec_min_split;       // fewest keys per decode split
    int dec_split_align;     // split length is a multiple of this (the kernel's key tile)
    int dec_pair_cap, fa_item_cap, ext_row_cap;
    PlanHeader* hdr;
    int2* dec_pairs;
    int32_t* dec_first;
    int32_t* dec_nsplit;
    int4* fa_items;      // (request, pair of query tiles, slot, cost)
    // 1: the kernel before this one is the same call's cache write, launched
    // to let the planner start at once (the planner reads no cache). The
    // planner then waits for it before finishing, so the kernels that depend
    // on the plan also see the written cache.
    int after_cache_write;
    int32_t* ext_base;   // per extend request: first partial row
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace pka
