// cache_write.cu -- reshape_and_cache: scatter the new tokens' K/V rows into
// their cache slots ("Beyond porting", unified backends, stage 1 "save
// key/value into the KV cache"; the ROCm path's reshape_and_cache_flush).
//
// Cache layout [num_blocks, num_kv_heads, block_size, head_dim]: a
// (block, kv head) pair is one contiguous block_size x head_dim tile, which
// is what the attention kernels fetch with one TMA box per 16 rows.
//
// A warp moves kRows (token, kv head) rows per step: lane i copies the i-th
// 16-byte piece of the row's K then V (so d = 128 is one piece per lane for
// K and V together). The slot index and the row's data are loaded together
// (only the store address depends on the slot) and all kRows rows are loaded
// before any is stored, so a warp keeps kRows x 512 bytes in flight instead
// of waiting out two dependent round trips per row. HBM-bound: reads and
// writes T * Hkv * (d + dv) * 2 bytes each.
//
// The 8-bit variant stores E4M3 codes: x / scale rounded to the nearest code
// (ties to even) with finite values beyond 448 saturated, the division and
// the rounding both taken from float32 (the division is IEEE round to nearest).
#include <type_traits>

#include "common.cuh"

namespace pka {

namespace {

constexpr int kCwRows = 4;       // rows per warp step
constexpr int kCwMaxPieces = 4;  // 16-byte pieces per lane per row (K + V <= 128 pieces = 1024 bf16)

struct CacheWriteParams {
    const uint4* k;
    const uint4* v;
    const int64_t* slots;
    void* k_cache;
    void* v_cache;
    int64_t num_tokens, num_slots;
    int num_kv_heads, block_size;
    int k_vecs, v_vecs;  // head_dim / 8, head_dim_v / 8 (16-byte pieces of bf16 input)
    float k_scale, v_scale;  // 8-bit cache: one code unit of K / V
    int32_t* err;
};

// Four floats -> four E4M3 codes (x / s, RN-even, saturating), lowest first.
PKA_DEVICE uint32_t quantize4(float a, float b, float c, float d, float s) {
    uint32_t lo, hi;
    const float qa = __fdiv_rn(a, s), qb = __fdiv_rn(b, s), qc = __fdiv_rn(c, s), qd = __fdiv_rn(d, s);
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}" : "=r"(lo) : "f"(qa), "f"(qb));
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}" : "=r"(hi) : "f"(qc), "f"(qd));
    return lo | (hi << 16);
}

PKA_DEVICE uint2 quantize8(uint4 x, float s) {
    uint2 r;
    r.x = quantize4(bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y), s);
    r.y = quantize4(bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w), s);
    return r;
}

template <bool kFp8, int kCwPieces>
__global__ void __launch_bounds__(256) cache_write_kernel(CacheWriteParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t rows = p.num_tokens * p.num_kv_heads;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int nv = p.k_vecs + p.v_vecs;
    for (int64_t r0 = warp * kCwRows; r0 < rows; r0 += nwarps * kCwRows) {
        int64_t slot[kCwRows];
        uint4 val[kCwRows][kCwPieces];
#pragma unroll
        for (int i = 0; i < kCwRows; ++i) {
            const int64_t row = r0 + i;
            const bool in = row < rows;
            slot[i] = in ? __ldg(p.slots + row / p.num_kv_heads) : -1;
#pragma unroll
            for (int j = 0; j < kCwPieces; ++j) {
                const int c = lane + 32 * j;
                if (in && c < nv)
                    val[i][j] = c < p.k_vecs ? __ldcs(p.k + row * p.k_vecs + c) : __ldcs(p.v + row * p.v_vecs + (c - p.k_vecs));
            }
        }
#pragma unroll
        for (int i = 0; i < kCwRows; ++i) {
            const int64_t row = r0 + i;
            const int64_t s = slot[i];
            if (row >= rows || s < 0) continue;
            if (s >= p.num_slots) {
                if (lane == 0) set_error(p.err, PKA_DEVERR_SLOT);
                continue;
            }
            const int64_t t = row / p.num_kv_heads;
            const int h = (int)(row - t * p.num_kv_heads);
            const int64_t blk = s / p.block_size;
            const int64_t dst_row = (blk * p.num_kv_heads + h) * p.block_size + (s - blk * p.block_size);
#pragma unroll
            for (int j = 0; j < kCwPieces; ++j) {
                const int c = lane + 32 * j;
                if (c >= nv) continue;
                const bool is_k = c < p.k_vecs;
                const int cc = is_k ? c : c - p.k_vecs;
                const int vecs = is_k ? p.k_vecs : p.v_vecs;
                if (kFp8) {
                    uint2* dst = static_cast<uint2*>(is_k ? p.k_cache : p.v_cache) + dst_row * vecs + cc;
                    *dst = quantize8(val[i][j], is_k ? p.k_scale : p.v_scale);
                } else {
                    uint4* dst = static_cast<uint4*>(is_k ? p.k_cache : p.v_cache) + dst_row * vecs + cc;
                    *dst = val[i][j];
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_cache_write(const void* k, const void* v, const int64_t* slots, int64_t T, int Hkv, int d,
                               int dv, void* k_cache, void* v_cache, int64_t num_blocks, int bs, int32_t* err,
                               int num_sms, cudaStream_t stream, bool fp8, float k_scale, float v_scale) {
    CacheWriteParams p;
    p.k = static_cast<const uint4*>(k);
    p.v = static_cast<const uint4*>(v);
    p.slots = slots;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.num_tokens = T;
    p.num_slots = num_blocks * bs;
    p.num_kv_heads = Hkv;
    p.block_size = bs;
    p.k_vecs = d / 8;
    p.v_vecs = v ? dv / 8 : 0;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.err = err;
    const int pieces = (p.k_vecs + p.v_vecs + 31) / 32;  // per lane per row
    if (pieces > kCwMaxPieces) return cudaErrorInvalidValue;
    const int64_t rows = T * Hkv;
    int64_t blocks = (rows + 8 * kCwRows - 1) / (8 * kCwRows);
    const int64_t cap = (int64_t)num_sms * 8;  // 8 blocks of 8 warps fill an SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    auto go = [&](auto fp8_c, auto pieces_c) {
        cache_write_kernel<decltype(fp8_c)::value, decltype(pieces_c)::value><<<(unsigned)blocks, 256, 0, stream>>>(p);
    };
    using T_ = std::true_type;
    using F_ = std::false_type;
    using P1 = std::integral_constant<int, 1>;
    using P2 = std::integral_constant<int, 2>;
    using P4 = std::integral_constant<int, 4>;
    if (fp8) {
        if (pieces == 1) go(T_{}, P1{});
        else if (pieces == 2) go(T_{}, P2{});
        else go(T_{}, P4{});
    } else {
        if (pieces == 1) go(F_{}, P1{});
        else if (pieces == 2) go(F_{}, P2{});
        else go(F_{}, P4{});
    }
    return cudaGetLastError();
}

}  // namespace pka
