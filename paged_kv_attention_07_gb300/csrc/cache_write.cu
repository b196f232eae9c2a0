// cache_write.cu -- reshape_and_cache: scatter the new tokens' K/V rows into
// their cache slots ("Beyond porting", unified backends, stage 1 "save
// key/value into the KV cache"; the ROCm path's reshape_and_cache_flush).
//
// Cache layout [num_blocks, num_kv_heads, block_size, head_dim]: a
// (block, kv head) pair is one contiguous block_size x head_dim tile, which
// is what the attention kernels fetch with one TMA box per 16 rows.
//
// One warp copies one (token, kv head) row of K and of V with 16-byte
// vector loads/stores: 8 bf16 per lane, i.e. 256 elements per warp step.
// HBM-bound: reads and writes 2 * T * Hkv * d * 2 bytes (K and V).
#include "common.cuh"

namespace pka {

struct CacheWriteParams {
    const uint4* k;
    const uint4* v;
    const int64_t* slots;
    uint4* k_cache;
    uint4* v_cache;
    int64_t num_tokens, num_slots;
    int num_kv_heads, block_size;
    int k_vecs, v_vecs;  // head_dim / 8, head_dim_v / 8
    int32_t* err;
};

__global__ void __launch_bounds__(256) cache_write_kernel(CacheWriteParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t rows = p.num_tokens * p.num_kv_heads;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = warp; row < rows; row += nwarps) {
        const int64_t t = row / p.num_kv_heads;
        const int h = (int)(row - t * p.num_kv_heads);
        const int64_t slot = __ldg(p.slots + t);
        if (slot < 0) continue;
        if (slot >= p.num_slots) {
            if (lane == 0) set_error(p.err, PKA_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / p.block_size;
        const int64_t off = slot - blk * p.block_size;
        const int64_t dst_row = (blk * p.num_kv_heads + h) * p.block_size + off;
        const uint4* ks = p.k + row * p.k_vecs;
        uint4* kd = p.k_cache + dst_row * p.k_vecs;
        for (int i = lane; i < p.k_vecs; i += 32) kd[i] = __ldcs(ks + i);
        if (p.v) {
            const uint4* vs = p.v + row * p.v_vecs;
            uint4* vd = p.v_cache + dst_row * p.v_vecs;
            for (int i = lane; i < p.v_vecs; i += 32) vd[i] = __ldcs(vs + i);
        }
    }
}

cudaError_t launch_cache_write(const void* k, const void* v, const int64_t* slots, int64_t T,
                               int Hkv, int d, int dv, void* k_cache, void* v_cache,
                               int64_t num_blocks, int bs, int32_t* err, int num_sms,
                               cudaStream_t stream) {
    CacheWriteParams p;
    p.k = static_cast<const uint4*>(k);
    p.v = static_cast<const uint4*>(v);
    p.slots = slots;
    p.k_cache = static_cast<uint4*>(k_cache);
    p.v_cache = static_cast<uint4*>(v_cache);
    p.num_tokens = T;
    p.num_slots = num_blocks * bs;
    p.num_kv_heads = Hkv;
    p.block_size = bs;
    p.k_vecs = d / 8;
    p.v_vecs = v ? dv / 8 : 0;
    p.err = err;
    const int64_t rows = T * Hkv;
    const int64_t warps_needed = rows;
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = (int64_t)num_sms * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cache_write_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pka
