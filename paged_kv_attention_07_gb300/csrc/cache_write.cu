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

// Rows per warp step: enough 16-byte pieces per lane in flight to cover the
// load latency (one piece per lane per row at d = dv = 128).
template <int kCwPieces>
constexpr int cw_rows() {
    return kCwPieces == 1 ? 8 : 4;
}

// kWide: 64-bit row and slot arithmetic, only when T * Hkv or the slot count
// reaches 2^31 (64-bit division by a runtime divisor is a long software
// sequence; the 32-bit one is a few instructions).
template <bool kFp8, int kCwPieces, bool kWide>
__global__ void __launch_bounds__(256) cache_write_kernel(CacheWriteParams p) {
    using Idx = typename std::conditional<kWide, int64_t, uint32_t>::type;
    constexpr int kRows = cw_rows<kCwPieces>();
    // a forward step's planner may start now: it reads no cache
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const Idx warp = (Idx)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const Idx rows = (Idx)(p.num_tokens * p.num_kv_heads);
    const Idx nwarps = (Idx)gridDim.x * (blockDim.x >> 5);
    const Idx hkv = (Idx)p.num_kv_heads, bs = (Idx)p.block_size;
    const int nv = p.k_vecs + p.v_vecs;
    for (Idx r0 = warp * kRows; r0 < rows; r0 += nwarps * kRows) {
        int64_t slot[kRows];
        uint4 val[kRows][kCwPieces];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const Idx row = r0 + i;
            const bool in = row < rows;
            slot[i] = in ? __ldg(p.slots + row / hkv) : -1;
#pragma unroll
            for (int j = 0; j < kCwPieces; ++j) {
                const int c = lane + 32 * j;
                if (in && c < nv)
                    val[i][j] = c < p.k_vecs ? __ldcs(p.k + (int64_t)row * p.k_vecs + c)
                                             : __ldcs(p.v + (int64_t)row * p.v_vecs + (c - p.k_vecs));
            }
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const Idx row = r0 + i;
            const int64_t s64 = slot[i];
            if (row >= rows || s64 < 0) continue;
            if (s64 >= p.num_slots) {
                if (lane == 0) set_error(p.err, PKA_DEVERR_SLOT);
                continue;
            }
            const Idx s = (Idx)s64;  // < num_slots, which fits Idx
            const Idx t = row / hkv;
            const Idx h = row - t * hkv;
            const Idx blk = s / bs;
            const int64_t dst_row = ((int64_t)blk * hkv + h) * bs + (s - blk * bs);
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

// Resident CTAs per SM of one instantiation (the grid is sized to one full
// wave: the grid-stride loop then needs no second, partial wave).
template <typename K>
int cw_blocks_per_sm(K kern) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 256, 0) != cudaSuccess || n < 1) n = 1;
    return n;
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
    const bool wide = rows >= ((int64_t)1 << 31) || p.num_slots >= ((int64_t)1 << 31);
    auto go = [&](auto fp8_c, auto pieces_c, auto wide_c) {
        constexpr bool F = decltype(fp8_c)::value, W = decltype(wide_c)::value;
        constexpr int P = decltype(pieces_c)::value;
        auto kern = cache_write_kernel<F, P, W>;
        static const int per_sm = cw_blocks_per_sm(kern);  // one value per instantiation
        const int64_t need = (rows + 8 * cw_rows<P>() - 1) / (8 * cw_rows<P>());
        int64_t blocks = std::min<int64_t>(need, (int64_t)num_sms * per_sm);
        if (blocks < 1) blocks = 1;
        kern<<<(unsigned)blocks, 256, 0, stream>>>(p);
    };
    using T_ = std::true_type;
    using F_ = std::false_type;
    using P1 = std::integral_constant<int, 1>;
    using P2 = std::integral_constant<int, 2>;
    using P4 = std::integral_constant<int, 4>;
    auto by_pieces = [&](auto fp8_c, auto wide_c) {
        if (pieces == 1) go(fp8_c, P1{}, wide_c);
        else if (pieces == 2) go(fp8_c, P2{}, wide_c);
        else go(fp8_c, P4{}, wide_c);
    };
    if (fp8) {
        if (wide) by_pieces(T_{}, T_{});
        else by_pieces(T_{}, F_{});
    } else {
        if (wide) by_pieces(F_{}, T_{});
        else by_pieces(F_{}, F_{});
    }
    return cudaGetLastError();
}

}  // namespace pka
