// merge.cu -- the LSE merge ("Beyond porting", extend path: every chunk
// yields an output and an LSE, which captures the softmax denominator and
// lets the chunks be merged stably, the higher-scoring chunk dominating).
//
// For partial results (o_i, lse_i) over disjoint key sets:
//     m = max_i lse_i,  w_i = exp(lse_i - m)
//     o = sum_i w_i o_i / sum_i w_i,   lse = m + log(sum_i w_i)
// Three kernels use it: the two-input public merge, the decode split-KV
// reduction, and the extend reduction (new-token stage + context chunks).
// All are HBM-bound streaming kernels.
#include "common.cuh"
#include "params.cuh"
#include "plan.cuh"

namespace pka {

// ------------------------------------------------------------ public merge
template <bool kBf16>
__global__ void __launch_bounds__(256) merge_pair_kernel(void* out, float* out_lse, const void* a,
                                                         const float* a_lse, const void* b,
                                                         const float* b_lse, int64_t rows, int dv) {
    const int vec = kBf16 ? 8 : 4;
    const int per_row = dv / vec;
    const int64_t total = rows * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / per_row;
        const int c = (int)(i - row * per_row);
        const float la = a_lse[row], lb = b_lse[row];
        const float m = fmaxf(la, lb);
        float wa, wb, inv;
        if (m == -INFINITY) {
            wa = wb = 0.f;
            inv = 0.f;
        } else {
            wa = __expf(la - m);
            wb = __expf(lb - m);
            inv = 1.f / (wa + wb);
        }
        if (kBf16) {
            const uint4 x = reinterpret_cast<const uint4*>(a)[i];
            const uint4 y = reinterpret_cast<const uint4*>(b)[i];
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = (wa * bf16_lo(xs[j]) + wb * bf16_lo(ys[j])) * inv;
                const float hi = (wa * bf16_hi(xs[j]) + wb * bf16_hi(ys[j])) * inv;
                o[j] = pack_bf16(lo, hi);
            }
            reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            const float4 x = reinterpret_cast<const float4*>(a)[i];
            const float4 y = reinterpret_cast<const float4*>(b)[i];
            float4 o;
            o.x = (wa * x.x + wb * y.x) * inv;
            o.y = (wa * x.y + wb * y.y) * inv;
            o.z = (wa * x.z + wb * y.z) * inv;
            o.w = (wa * x.w + wb * y.w) * inv;
            reinterpret_cast<float4*>(out)[i] = o;
        }
        if (out_lse && c == 0) out_lse[row] = (m == -INFINITY) ? -INFINITY : m + __logf(wa + wb);
    }
}

cudaError_t launch_merge_pair(void* out, float* out_lse, const void* a, const float* a_lse,
                              const void* b, const float* b_lse, int64_t rows, int dv, int io_dtype,
                              int num_sms, cudaStream_t stream) {
    const int vec = io_dtype ? 8 : 4;
    const int64_t total = rows * (dv / vec);
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    if (blocks < 1) blocks = 1;
    if (io_dtype)
        merge_pair_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(out, out_lse, a, a_lse, b,
                                                                       b_lse, rows, dv);
    else
        merge_pair_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(out, out_lse, a, a_lse, b,
                                                                        b_lse, rows, dv);
    return cudaGetLastError();
}

// ------------------------------------------------- multi-way row merge
// One warp merges n partial rows (row stride `stride` floats between
// partials) into one bf16 output row and its lse. dv is 64 or a multiple of 128.
// Lane i holds partial i's lse (n <= 32 in one pass); its weight goes to the
// other lanes by shuffles, and each lane's loads of the n partial pieces are
// issued four at a time, so the merge costs about 1 + n / 4 memory round trips
// (rows of at most kSmallMerge partials take the one-round-trip path below).
// w[j] with a runtime j in 0..3, without indexing a register array
PKA_DEVICE float pick4(const float (&w)[4], int j) {
    return j == 0 ? w[0] : (j == 1 ? w[1] : (j == 2 ? w[2] : w[3]));
}

// Up to kSmallMerge partials: the LSEs and the first 128-dim chunk of every
// partial are loaded together before any weight is known, so a row of up to
// 128 dims costs one memory round trip (plus one per further 128 dims).
// Summation order is the partials' order, as in the general path.
constexpr int kSmallMerge = 8;

PKA_DEVICE void merge_rows_warp_small(const float* part_o, const float* part_lse, int n, int64_t stride_rows,
                                      int dv, __nv_bfloat16* out_row, float* lse_out) {
    const int lane = threadIdx.x & 31;
    auto load_chunk = [&](int c0, float4 (&x)[kSmallMerge]) {
        const int c = c0 + lane * 4;
#pragma unroll
        for (int k = 0; k < kSmallMerge; ++k)
            x[k] = (k < n && c < dv) ? *reinterpret_cast<const float4*>(part_o + (int64_t)k * stride_rows * dv + c)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    const float l_mine = lane < n ? part_lse[(int64_t)lane * stride_rows] : -INFINITY;
    float4 x[kSmallMerge];
    load_chunk(0, x);
    float m = l_mine;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float w_mine = (m == -INFINITY || l_mine == -INFINITY) ? 0.f : __expf(l_mine - m);
    float wsum = w_mine;
#pragma unroll
    for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    float w[kSmallMerge];
#pragma unroll
    for (int k = 0; k < kSmallMerge; ++k) w[k] = __shfl_sync(0xffffffffu, w_mine, k);  // 0 past n
    for (int c0 = 0; c0 < dv; c0 += 128) {
        if (c0 > 0) load_chunk(c0, x);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kSmallMerge; ++k) {
            acc.x += w[k] * x[k].x;
            acc.y += w[k] * x[k].y;
            acc.z += w[k] * x[k].z;
            acc.w += w[k] * x[k].w;
        }
        const int c = c0 + lane * 4;
        if (c < dv) {
            uint2 o;
            o.x = pack_bf16(acc.x * inv, acc.y * inv);
            o.y = pack_bf16(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(out_row + c) = o;
        }
    }
    if (lane == 0 && lse_out) *lse_out = (wsum > 0.f) ? m + __logf(wsum) : -INFINITY;
}

PKA_DEVICE void merge_rows_warp(const float* part_o, const float* part_lse, int n, int64_t stride_rows,
                                int dv, __nv_bfloat16* out_row, float* lse_out) {
    if (n <= kSmallMerge) {
        merge_rows_warp_small(part_o, part_lse, n, stride_rows, dv, out_row, lse_out);
        return;
    }
    const int lane = threadIdx.x & 31;
    float m = -INFINITY;
    float l_mine[4];  // lse of partials lane, lane + 32, ... (n <= 128 kept in registers)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = lane + 32 * j;
        l_mine[j] = i < n ? part_lse[(int64_t)i * stride_rows] : -INFINITY;
        m = fmaxf(m, l_mine[j]);
    }
    for (int i = lane + 128; i < n; i += 32) m = fmaxf(m, part_lse[(int64_t)i * stride_rows]);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float w_mine[4], wsum = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        w_mine[j] = (m == -INFINITY || l_mine[j] == -INFINITY) ? 0.f : __expf(l_mine[j] - m);
        wsum += w_mine[j];
    }
    for (int i = lane + 128; i < n; i += 32) {
        const float l = part_lse[(int64_t)i * stride_rows];
        wsum += (m == -INFINITY) ? 0.f : __expf(l - m);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    // every lane runs every iteration (the weights come by shuffles); lanes
    // past dv (dv = 64) only skip their loads and stores
    for (int c0 = 0; c0 < dv; c0 += 128) {
        const int c = c0 + lane * 4;
        const bool active = c < dv;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int i = 0;
        for (; i + 4 <= n; i += 4) {  // four partials' loads in flight at once
            float4 x[4];
            float w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[k] = active ? *reinterpret_cast<const float4*>(part_o + (int64_t)(i + k) * stride_rows * dv + c)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
                const int ii = i + k;
                const float wl = __shfl_sync(0xffffffffu, pick4(w_mine, (ii >> 5) & 3), ii & 31);
                w[k] = ii < 128 ? wl
                                : ((m == -INFINITY) ? 0.f : __expf(part_lse[(int64_t)ii * stride_rows] - m));
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc.x += w[k] * x[k].x;
                acc.y += w[k] * x[k].y;
                acc.z += w[k] * x[k].z;
                acc.w += w[k] * x[k].w;
            }
        }
        for (; i < n; ++i) {
            const float4 x = active ? *reinterpret_cast<const float4*>(part_o + (int64_t)i * stride_rows * dv + c)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            const float wl = __shfl_sync(0xffffffffu, pick4(w_mine, (i >> 5) & 3), i & 31);
            const float w = i < 128 ? wl : ((m == -INFINITY) ? 0.f : __expf(part_lse[(int64_t)i * stride_rows] - m));
            acc.x += w * x.x;
            acc.y += w * x.y;
            acc.z += w * x.z;
            acc.w += w * x.w;
        }
        if (active) {
            uint2 o;
            o.x = pack_bf16(acc.x * inv, acc.y * inv);
            o.y = pack_bf16(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(out_row + c) = o;
        }
    }
    if (lane == 0 && lse_out) *lse_out = (wsum > 0.f) ? m + __logf(wsum) : -INFINITY;
}

// Decode split-KV reduction: request r with n > 1 splits; its partials are
// rows (dec_first[r] + s) * Hq + h.

__global__ void __launch_bounds__(256, 4) decode_reduce_kernel(DecodeReduceParams p) {
    grid_dep_wait();
    if (p.hdr->dec_num_pairs == 0) return;
    const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t total = (int64_t)p.num_decodes * p.Hq;
    for (int64_t w = warp; w < total; w += (int64_t)gridDim.x * 8) {
        const int r = (int)(w / p.Hq), h = (int)(w - (int64_t)r * p.Hq);
        const int n = p.dec_nsplit[r];
        if (n <= 1) continue;  // written directly by the decode kernel
        const int64_t row0 = (int64_t)p.dec_first[r] * p.Hq + h;
        // token index of decode request r is r (one new token each)
        merge_rows_warp(p.part_o + row0 * p.dv, p.part_lse + row0, n, p.Hq, p.dv,
                        p.out + ((int64_t)r * p.Hq + h) * p.dv, p.lse ? p.lse + (int64_t)r * p.Hq + h : nullptr);
    }
}

cudaError_t launch_decode_reduce(const DecodeReduceParams& p, int num_sms, cudaStream_t stream) {
    int64_t blocks = ((int64_t)p.num_decodes * p.Hq + 7) / 8;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    if (blocks < 1) blocks = 1;
    return launch_dependent(decode_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, p);
}

// Extend reduction: token i of extend request r has nslot = 1 + chunks
// partials at rows (ext_base[r] + slot * qlen + i) * Hq + h.

__global__ void __launch_bounds__(256, 4) extend_reduce_kernel(ExtendReduceParams p) {
    grid_dep_wait();
    if (p.hdr->fa_num_items == 0) return;
    const int nd = p.num_decodes, ne = p.num_extends;
    const int t0 = p.qsl[nd], t1 = p.qsl[nd + ne];
    const int64_t total = (int64_t)(t1 - t0) * p.Hq;
    const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    for (int64_t w = warp; w < total; w += (int64_t)gridDim.x * 8) {
        const int t = t0 + (int)(w / p.Hq);
        const int h = (int)(w % p.Hq);
        int lo = nd, hi = nd + ne - 1;  // request owning token t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.qsl[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        const int r = lo;
        const int ql = p.qsl[r + 1] - p.qsl[r];
        const int ctx = p.seq_lens[r] - ql;
        const int nslot = 1 + (ctx + p.chunk - 1) / p.chunk;
        const int i = t - p.qsl[r];
        const int64_t row0 = ((int64_t)p.ext_base[r - nd] + i) * p.Hq + h;
        merge_rows_warp(p.part_o + row0 * p.dv, p.part_lse + row0, nslot, (int64_t)ql * p.Hq, p.dv,
                        p.out + ((int64_t)t * p.Hq + h) * p.dv, p.lse ? p.lse + (int64_t)t * p.Hq + h : nullptr);
    }
}

cudaError_t launch_extend_reduce(const ExtendReduceParams& p, int ext_tokens_bound, int num_sms,
                                 cudaStream_t stream) {
    int64_t blocks = ((int64_t)ext_tokens_bound * p.Hq + 7) / 8;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    if (blocks < 1) blocks = 1;
    return launch_dependent(extend_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, p);
}

}  // namespace pka
