// ctx_dequant.cu -- the context gather of an 8-bit cache for the extend
// path ("Beyond porting", absorbed / non-absorbed recipe: the prefill
// listing's gather_and_maybe_dequant_cache step before each context chunk's
// attention).
//
// The extend requests' cached positions are copied out of the paged 8-bit
// cache (E4M3 codes, [num_blocks, Hkv, bs, d]) into a compact bf16 cache in
// the workspace, [num_extends * nblk, Hkv, 128, d]: extend i's position pos
// lands in compact block i * nblk + pos / 128, row pos % 128, and the compact
// block table row i is i * nblk + j. The prefill/extend kernel then reads its
// context chunks from there with 128-key TMA boxes. The copy holds the codes'
// values (exact in bf16: 3 mantissa bits, exponents 2^-9 .. 2^8), not
// value x scale: the scales are applied by the attention kernel to the
// context chunks' scores and outputs, so no rounding is added.
//
// One CTA per (extend, compact block, kv head): 128 rows x (d + dv) codes
// in, twice the bytes out, 16 codes per thread step. HBM-bound.
#include "common.cuh"
#include "params.cuh"

namespace pka {

namespace {

constexpr int kCdRows = 128;  // rows of a compact block
constexpr int kCdThreads = 256;

// f16 pair -> two floats
PKA_DEVICE float2 f16x2_to_f32x2(uint32_t h) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
    return make_float2(lo, hi);
}

// four codes -> four bf16 values (two pairs)
PKA_DEVICE uint2 codes4_to_bf16(uint32_t w) {
    const float2 a = f16x2_to_f32x2(e4m3x2_to_f16x2(w & 0xffffu));
    const float2 b = f16x2_to_f32x2(e4m3x2_to_f16x2(w >> 16));
    return make_uint2(pack_bf16(a.x, a.y), pack_bf16(b.x, b.y));
}

__global__ void __launch_bounds__(kCdThreads) ctx_dequant_kernel(CtxDequantParams p) {
    // launched after the planner (which clears the error word this kernel may set)
    grid_dep_wait();
    const int i = blockIdx.y;  // extend
    const int j = (int)(blockIdx.x / p.Hkv), h = (int)(blockIdx.x % p.Hkv);
    const int r = p.num_decodes + i;
    if (h == 0 && threadIdx.x == 0) p.bt_c[(int64_t)i * p.nblk + j] = i * p.nblk + j;
    // context length, clamped to what the compact cache holds (bad metadata
    // is the planner's to report; nothing is written out of range)
    int ctx = p.seq_lens[r] - (p.qsl[r + 1] - p.qsl[r]);
    ctx = max(0, min(ctx, p.nblk * kCdRows));
    const int row0 = j * kCdRows;
    const int nrows = min(kCdRows, ctx - row0);
    if (nrows <= 0) return;
    const int kp = p.d / 16, vp = p.dv / 16, pieces = kp + vp;  // 16-code pieces per row
    const int32_t* bt = p.block_table + (int64_t)r * p.max_blocks;
    const int64_t dst_blk = ((int64_t)i * p.nblk + j) * p.Hkv + h;
    for (int q = threadIdx.x; q < nrows * pieces; q += kCdThreads) {
        const int row = q / pieces, pc = q - row * pieces;
        const int pos = row0 + row;
        int blk = __ldg(bt + pos / p.bs);
        if (blk < 0 || blk >= p.num_blocks) {
            set_error(p.err, PKA_DEVERR_BLOCK_ID);
            continue;
        }
        const int64_t src_row = ((int64_t)blk * p.Hkv + h) * p.bs + pos % p.bs;
        const int64_t dst_row = dst_blk * kCdRows + row;
        const bool is_k = pc < kp;
        const int c = is_k ? pc : pc - kp;
        const int width = is_k ? p.d : p.dv;
        const uint4 w = __ldcs(reinterpret_cast<const uint4*>((is_k ? p.k8 : p.v8) + src_row * width) + c);
        const uint2 a = codes4_to_bf16(w.x), b = codes4_to_bf16(w.y), cc = codes4_to_bf16(w.z),
                    d = codes4_to_bf16(w.w);
        uint4* dst = reinterpret_cast<uint4*>((is_k ? p.kc : p.vc) + dst_row * width) + 2 * c;
        dst[0] = make_uint4(a.x, a.y, b.x, b.y);
        dst[1] = make_uint4(cc.x, cc.y, d.x, d.y);
    }
}

}  // namespace

cudaError_t launch_ctx_dequant(const CtxDequantParams& p, cudaStream_t stream) {
    if (p.num_extends <= 0) return cudaSuccess;
    const dim3 grid((unsigned)(p.nblk * p.Hkv), (unsigned)p.num_extends);
    return launch_dependent(ctx_dequant_kernel, grid, dim3(kCdThreads), 0, stream, p);
}

}  // namespace pka
