// fa_fwd.cu -- varlen prefill and the extend path's pieces
// ("Beyond porting", section "Three-path processing explained"):
//   prefill: new sequences, causal, Q/K/V in the [num_tokens, heads, dim]
//            layout (the pages' flash_attn_varlen_func);
//   extend:  stage 1, the new tokens over their own keys (causal, bottom-right
//            aligned: new token i sees new keys 0..i), and stage 2, every
//            context chunk of `chunk` cached keys (no mask, all context
//            precedes the new tokens), each emitting (O, LSE) for the merge.
// The pages gather each context chunk into a contiguous buffer first
// (cp_mha_gather_cache); here the tile loads walk the block table directly,
// and the chunk loop is a grid dimension: every (query tile, chunk) is an
// independent work item, merged afterwards by the extend reduction.
//
// Work unit: (request, 64-row query tile, slot) x query head, slot 0 = new
// keys, slot c >= 1 = context chunk c - 1; persistent CTAs pull units from
// the planner's cost-sorted list. Flash-attention style: Q tile resident,
// K/V tiles of 64 keys double-buffered with cp.async, S and O accumulated in
// fp32 by m16n8k16 bf16 MMAs, online softmax in the log2 domain.
#include "common.cuh"
#include "params.cuh"
#include "plan.cuh"

namespace pka {

constexpr int kFaWarps = 4;
constexpr int kFaThreads = kFaWarps * 32;
constexpr int BM = kFaBlockM;  // 64 query rows: 16 per warp
constexpr int BN = kFaBlockN;  // 64 keys per tile


template <int D>
struct FaSmem {
    static constexpr int kQBytes = BM * D * 2;
    static constexpr int kKVBytes = BN * D * 2;
    static constexpr int kBytes = kQBytes + 4 * kKVBytes + 1024;
};

// [D/64 segments][rows][128 B], 128-byte swizzled; `rows` rows per segment.
template <int ROWS>
PKA_DEVICE uint32_t fa_off(int row, int c) {
    return sw128((uint32_t)((c >> 3) * ROWS + row), (uint32_t)(c & 7));
}

template <int D>
__global__ void __launch_bounds__(kFaThreads, 2) fa_fwd_kernel(const FaParams p) {
    using S = FaSmem<D>;
    constexpr int kC = D / 8;       // 16-byte chunks per row
    constexpr int kKS = D / 16;     // k-steps over the head dim
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t q_s = smem_u32(smem);
    const uint32_t kv_s = q_s + S::kQBytes;  // stage st: K at kv_s + 2*st*kKV, V after it
    __shared__ int s_unit;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int num_units = p.hdr->fa_num_items * p.Hq;

    for (;;) {
        if (tid == 0) s_unit = atomicAdd(p.counter, 1);
        __syncthreads();
        const int unit = s_unit;
        __syncthreads();
        if (unit >= num_units) break;
        const int4 it = p.items[unit / p.Hq];
        const int h = unit % p.Hq, g = h / p.G;
        const int r = it.x, qt = it.y, slot = it.z;
        const int q0 = p.qsl[r];
        const int qlen = p.qsl[r + 1] - q0;
        const int ctx = p.seq_lens[r] - qlen;
        const int row0 = qt * BM;                 // first query row (within the request)
        const int rows = min(BM, qlen - row0);
        // key space of this slot
        int kbeg, kend;
        if (slot == 0) {
            kbeg = 0;
            kend = min(qlen, row0 + BM);  // new keys 0 .. last row of the tile
        } else {
            kbeg = (slot - 1) * p.chunk;
            kend = min(ctx, kbeg + p.chunk);
        }
        const int nkt = (kend - kbeg + BN - 1) / BN;
        const int32_t* bt = p.block_table + (int64_t)r * p.max_blocks;

        auto load_kv = [&](int kt, int st) {
            const uint32_t kd = kv_s + 2 * st * S::kKVBytes, vd = kd + S::kKVBytes;
            for (int ci = tid; ci < BN * kC; ci += kFaThreads) {
                const int kr = ci / kC, c = ci % kC;
                const int j = kbeg + kt * BN + kr;
                const bool ok = j < kend;
                const __nv_bfloat16 *ks, *vs;
                if (slot == 0) {
                    const int64_t row = ((int64_t)(q0 + (ok ? j : 0))) * p.Hkv + g;
                    ks = p.k_new + row * D + c * 8;
                    vs = p.v_new + row * D + c * 8;
                } else {
                    int blk = ok ? __ldg(bt + j / p.bs) : 0;
                    if (blk < 0 || blk >= p.num_blocks) {
                        set_error(p.err, PKA_DEVERR_BLOCK_ID);
                        blk = 0;
                    }
                    const int64_t row = ((int64_t)blk * p.Hkv + g) * p.bs + (ok ? j % p.bs : 0);
                    ks = p.k_cache + row * D + c * 8;
                    vs = p.v_cache + row * D + c * 8;
                }
                cp_async_16_zfill(kd + fa_off<BN>(kr, c), ks, ok);
                cp_async_16_zfill(vd + fa_off<BN>(kr, c), vs, ok);
            }
        };

        // Q tile + first K/V tile
        for (int ci = tid; ci < BM * kC; ci += kFaThreads) {
            const int qr = ci / kC, c = ci % kC;
            const bool ok = qr < rows;
            const __nv_bfloat16* src = p.q + ((int64_t)(q0 + row0 + (ok ? qr : 0)) * p.Hq + h) * D + c * 8;
            cp_async_16_zfill(q_s + fa_off<BM>(qr, c), src, ok);
        }
        load_kv(0, 0);
        cp_async_commit();

        float o[D / 8][4];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        uint32_t qa[kKS][4];
        const int qi0 = row0 + warp * 16 + (lane >> 2);  // this thread's rows: qi0, qi0 + 8

        for (int kt = 0; kt < nkt; ++kt) {
            if (kt + 1 < nkt) load_kv(kt + 1, (kt + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
            __syncthreads();
            if (kt == 0) {
                const int mi = lane >> 3;
#pragma unroll
                for (int ks = 0; ks < kKS; ++ks)
                    ldsm_x4(q_s + fa_off<BM>(warp * 16 + (mi & 1) * 8 + (lane & 7), ks * 2 + (mi >> 1)),
                            qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
            }
            const uint32_t kb = kv_s + 2 * (kt & 1) * S::kKVBytes, vb = kb + S::kKVBytes;
            float s[BN / 8][4];
#pragma unroll
            for (int i = 0; i < BN / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
            {
                const int mi = lane >> 3;
#pragma unroll
                for (int np = 0; np < BN / 16; ++np)
#pragma unroll
                    for (int ks = 0; ks < kKS; ++ks) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kb + fa_off<BN>(np * 16 + (mi >> 1) * 8 + (lane & 7), ks * 2 + (mi & 1)), b0, b1, b2, b3);
                        mma_bf16(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                        mma_bf16(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
                    }
            }
            // mask + online softmax (rows qi0, qi0 + 8)
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int jj = kbeg + kt * BN + nt * 8 + (lane & 3) * 2 + (e & 1);
                    const int qi = qi0 + (e >> 1) * 8;
                    const bool ok = jj < kend && (slot != 0 || jj <= qi);
                    const float x = ok ? s[nt][e] * p.scale_log2 : -INFINITY;
                    s[nt][e] = x;
                    mx[e >> 1] = fmaxf(mx[e >> 1], x);
                }
            float alpha[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
                mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
                const float mn = fmaxf(m[rr], mx[rr]);
                // mn is finite: key 0 of the first tile is visible to every row
                alpha[rr] = fast_exp2(m[rr] - mn);
                m[rr] = mn;
                l[rr] *= alpha[rr];
            }
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                o[i][0] *= alpha[0];
                o[i][1] *= alpha[0];
                o[i][2] *= alpha[1];
                o[i][3] *= alpha[1];
            }
            uint32_t pa[BN / 16][4];
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt) {
                const float p0 = fast_exp2(s[nt][0] - m[0]), p1 = fast_exp2(s[nt][1] - m[0]);
                const float p2 = fast_exp2(s[nt][2] - m[1]), p3 = fast_exp2(s[nt][3] - m[1]);
                l[0] += p0 + p1;
                l[1] += p2 + p3;
                pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
                pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
            }
            {
                const int mi = lane >> 3;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
#pragma unroll
                    for (int dp = 0; dp < D / 16; ++dp) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(vb + fa_off<BN>(kk * 16 + (mi & 1) * 8 + (lane & 7), dp * 2 + (mi >> 1)), b0, b1, b2, b3);
                        mma_bf16(o[2 * dp], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
                        mma_bf16(o[2 * dp + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
                    }
            }
            __syncthreads();  // stage (kt & 1) is refilled next iteration
        }
        cp_async_wait<0>();

        // finalize and store
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 1);
            l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 2);
        }
        const bool final_out = (slot == 0 && ctx == 0);
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int qi = qi0 + rr * 8;
            if (qi >= qlen) continue;
            const float inv = 1.f / l[rr];
            const float lse_nat = (m[rr] + __log2f(l[rr])) * 0.69314718055994531f;
            if (final_out) {
                __nv_bfloat16* dst = p.out + ((int64_t)(q0 + qi) * p.Hq + h) * D;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt)
                    *reinterpret_cast<uint32_t*>(dst + nt * 8 + (lane & 3) * 2) =
                        pack_bf16(o[nt][rr * 2] * inv, o[nt][rr * 2 + 1] * inv);
                if (p.lse && (lane & 3) == 0) p.lse[(int64_t)(q0 + qi) * p.Hq + h] = lse_nat;
            } else {
                const int64_t prow =
                    ((int64_t)p.ext_base[r - p.num_decodes] + (int64_t)slot * qlen + qi) * p.Hq + h;
                float* dst = p.ext_o + prow * D;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt)
                    *reinterpret_cast<float2*>(dst + nt * 8 + (lane & 3) * 2) =
                        make_float2(o[nt][rr * 2] * inv, o[nt][rr * 2 + 1] * inv);
                if ((lane & 3) == 0) p.ext_lse[prow] = lse_nat;
            }
        }
    }
}

template <int D>
static cudaError_t launch_fa_d(const FaParams& p, int num_sms, cudaStream_t stream) {
    auto kern = fa_fwd_kernel<D>;
    const int smem = FaSmem<D>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFaThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    kern<<<num_sms * per_sm, kFaThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fa_fwd(const FaParams& p, int head_dim, int num_sms, cudaStream_t stream) {
    if (head_dim == 128) return launch_fa_d<128>(p, num_sms, stream);
    if (head_dim == 64) return launch_fa_d<64>(p, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pka
