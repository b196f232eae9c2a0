// params.cuh -- launch parameter blocks of the attention kernels, shared by
// the kernels and the host code that fills them (api.cu).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include <cuda.h>

#include "plan.cuh"

namespace pka {

struct DecodeGqaParams {
    const __nv_bfloat16* q;        // [T, Hq, D]
    const __nv_bfloat16* k_cache;  // [nb, Hkv, bs, D]
    const __nv_bfloat16* v_cache;
    const uint8_t* k8;             // the same caches as E4M3 codes (8-bit cache kernel)
    const uint8_t* v8;
    float v_scale;                 // 8-bit cache: value of one V code unit (the output's factor)
    const int32_t* block_table;
    const int32_t* seq_lens;
    const PlanHeader* hdr;
    int32_t* counter;
    int32_t* err;
    const int2* pairs;
    const int32_t* nsplit;
    float* part_o;
    float* part_lse;
    __nv_bfloat16* out;
    float* lse;
    int64_t num_blocks;
    int max_blocks, Hq, Hkv, G, bs;
    float scale_log2;
};

struct DecodeMlaParams {
    const __nv_bfloat16* q;   // [T, Hq, 576]
    const __nv_bfloat16* kv;  // [nb, bs, 576]
    const int32_t* block_table;
    const int32_t* seq_lens;
    const PlanHeader* hdr;
    int32_t* counter;
    int32_t* err;
    const int2* pairs;
    const int32_t* nsplit;
    float* part_o;
    float* part_lse;
    __nv_bfloat16* out;
    float* lse;
    int64_t num_blocks;
    int max_blocks, Hq, bs, groups;  // groups = Hq / (8 * NW)
    int cache_rows;                  // num_blocks * bs (a row index past the cache)
    float scale_log2;
};

struct FaParams {
    const __nv_bfloat16* q;      // [T, Hq, D]
    const __nv_bfloat16* k_new;  // [T, Hkv, D]
    const __nv_bfloat16* v_new;
    const __nv_bfloat16* k_cache;  // [nb, Hkv, bs, D]
    const __nv_bfloat16* v_cache;
    const int32_t* block_table;
    const int32_t* qsl;
    const int32_t* seq_lens;
    const PlanHeader* hdr;
    int32_t* counter;
    int32_t* err;
    const int4* items;
    const int32_t* ext_base;
    float* ext_o;
    float* ext_lse;
    __nv_bfloat16* out;
    float* lse;
    int64_t num_blocks;
    int max_blocks, Hq, Hkv, G, bs, chunk, num_decodes, num_extends;
    int out_v8;  // out is 32-byte aligned: rows go out in 32-byte stores
    int bt_row0;  // request of block_table's first row (context chunks only read the table)
    float scale_log2;
    // context chunks (slots >= 1): score scale and output factor. The plain
    // bf16 cache: scale_log2 and 1. A gathered 8-bit cache holds the codes'
    // values: scale_log2 * k_scale and v_scale.
    float ctx_scale_log2, ctx_v_scale;
};

// Gather of the extends' context out of an 8-bit cache into a compact bf16
// cache (ctx_dequant.cu).
struct CtxDequantParams {
    const uint8_t* k8;  // [num_blocks, Hkv, bs, d] E4M3 codes
    const uint8_t* v8;  // [num_blocks, Hkv, bs, dv]
    const int32_t* block_table;
    const int32_t* qsl;
    const int32_t* seq_lens;
    __nv_bfloat16* kc;  // [num_extends * nblk, Hkv, 128, d]
    __nv_bfloat16* vc;  // [num_extends * nblk, Hkv, 128, dv]
    int32_t* bt_c;      // [num_extends, nblk]
    int32_t* err;
    int64_t num_blocks;
    int max_blocks, num_decodes, num_extends, Hkv, bs, d, dv, nblk;
};

struct DecodeReduceParams {
    const PlanHeader* hdr;
    const int32_t* dec_first;
    const int32_t* dec_nsplit;
    const float* part_o;
    const float* part_lse;
    __nv_bfloat16* out;
    float* lse;
    int num_decodes, Hq, dv;
};

struct ExtendReduceParams {
    const PlanHeader* hdr;
    const int32_t* qsl;
    const int32_t* seq_lens;
    const int32_t* ext_base;
    const float* part_o;
    const float* part_lse;
    __nv_bfloat16* out;
    float* lse;
    int num_decodes, num_extends, Hq, dv, chunk;
};

struct FaMaps {
    CUtensorMap q;     // [T, Hq, D]  box {64, 1, 128}
    CUtensorMap knew;  // [T, Hkv, D] box {64, 1, 128}
    CUtensorMap vnew;
    CUtensorMap kc;    // [nb * Hkv * bs, D] box {64, min(bs, 128)}
    CUtensorMap vc;
};

}  // namespace pka
