// decode_mla.cu -- absorbed multi-head latent attention decode
// ("vLLM AMD ROCm Attention Backends Optimization", section "The hybrid
// processing strategy": decode runs specialised MLA kernels directly on the
// compressed 576-dim latent; on ROCm that is the asm mla_decode_fwd).
//
// Every token has one 576-dim latent row shared by all query heads; the
// score uses all 576 dims and the value is the row's first 512 dims:
//     s_j = scale * <q_h, c_j[0:576]>,   o_h = sum_j softmax(s)_j c_j[0:512].
// Cache layout [num_blocks, block_size, 576] bf16 (num_kv_heads == 1).
//
// Work unit: (decode request, key split, group of 64 query heads). A
// producer warp streams 16-key latent tiles (18 KB) through a 4-stage ring
// with 2-D TMA boxes through the block table (cp.async below block size 8);
// 8 compute warps each own 8 heads and run, per tile,
//     S^T[16 keys x 8 heads] = C[16 x 576] . Q^T        (36 m16n8k16 steps)
//     O^T[512 x 8 heads]    += C[:, :512]^T . P^T        (32 m16n8k16 steps)
// with the online softmax over keys in registers. Each warp covers all keys
// of the split for its heads, so no cross-warp merge is needed.
#include "common.cuh"
#include "params.cuh"
#include "plan.cuh"

namespace pka {

constexpr int kMlaD = 576, kMlaDv = 512;
constexpr int kMlaSeg = kMlaD / 64;  // 9 swizzle segments of 64 dims
constexpr int kMlaStages = 4;
constexpr int kMlaTile = 16;
constexpr int kMlaTileBytes = kMlaTile * kMlaD * 2;  // 18 KB


template <int NW>
struct MlaSmem {
    static constexpr int kQBytes = NW * 8 * kMlaD * 2;
    static constexpr int kRingBytes = kMlaStages * kMlaTileBytes;
    static constexpr int kBytes = kQBytes + kRingBytes + 1024 + 256;
};

PKA_DEVICE uint32_t mla_tile_off(int tr, int c) {  // [9 segs][16 rows][128 B]
    return sw128((uint32_t)((c >> 3) * kMlaTile + tr), (uint32_t)(c & 7));
}

template <int NW, bool kTma>
__global__ void __launch_bounds__((NW + 1) * 32, 1)
    decode_mla_kernel(const __grid_constant__ CUtensorMap kvmap, const DecodeMlaParams p) {
    grid_dep_wait();
    using S = MlaSmem<NW>;
    constexpr int HG = NW * 8;  // heads per CTA
    constexpr int kThreads = (NW + 1) * 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem + S::kQBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + S::kRingBytes);
    uint64_t* empty = full + kMlaStages;
    __shared__ int s_unit;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool producer = warp == NW;
    const int num_units = p.hdr->dec_num_pairs * p.groups;
    if (num_units == 0) return;
    const int L = p.hdr->dec_split_len;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kMlaStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        fence_barrier_init();
        s_abort = 0;
        if (kTma) tma_prefetch_desc(&kvmap);
    }
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    uint32_t ld_it = 0, cs_it = 0;  // producer: tiles issued; consumers: tiles consumed
    bool alive = true;

    for (;;) {
        if (threadIdx.x == 0) s_unit = s_abort ? num_units : atomicAdd(p.counter, 1);
        __syncthreads();
        const int unit = s_unit;
        __syncthreads();
        if (unit >= num_units) break;
        const int pair = unit / p.groups, grp = unit - pair * p.groups;
        const int2 rs = p.pairs[pair];
        const int r = rs.x;
        const int slen = p.seq_lens[r];
        const int k0 = rs.y * L;
        const int k1 = min(k0 + L, slen);
        const int ntiles = (k1 - k0 + kMlaTile - 1) / kMlaTile;
        const int h0 = grp * HG;

        if (producer) {
            const int32_t* bt = p.block_table + (int64_t)r * p.max_blocks;
            for (int j = 0; j < ntiles && alive; ++j) {
                const int stage = ld_it % kMlaStages;
                if (ld_it >= (uint32_t)kMlaStages) {
                    if (!mbar_wait(&empty[stage], ((ld_it / kMlaStages) - 1) & 1, p.err)) {
                        alive = false;
                        s_abort = 1;
                        break;
                    }
                }
                uint8_t* dst = ring + stage * kMlaTileBytes;
                const int tb = k0 + j * kMlaTile;
                const int valid = min(kMlaTile, k1 - tb);
                if (kTma && valid == kMlaTile) {
                    if (lane == 0) {
                        fence_proxy_async_smem();
                        const int boxr = p.bs < kMlaTile ? p.bs : kMlaTile;
                        const int nsub = kMlaTile / boxr;
                        mbar_arrive_expect_tx(&full[stage], (uint32_t)(kMlaTileBytes));
                        for (int sb = 0; sb < nsub; ++sb) {
                            const int pos = tb + sb * boxr;
                            int blk = __ldg(bt + pos / p.bs);
                            if (blk < 0 || blk >= p.num_blocks) {
                                set_error(p.err, PKA_DEVERR_BLOCK_ID);
                                blk = 0;
                            }
                            const int row = blk * p.bs + (pos % p.bs);
                            for (int sg = 0; sg < kMlaSeg; ++sg)
                                tma_load_2d(dst + (sg * kMlaTile + sb * boxr) * 128, &kvmap, &full[stage],
                                            sg * 64, row, pol);
                        }
                    }
                    __syncwarp();
                } else {
                    // small blocks, or the last (partial) tile: 16-byte copies
                    // with rows past the end filled with zeros, so no NaN from
                    // unused slots reaches the value product.
                    const uint32_t base = smem_u32(dst);
                    for (int ci = lane; ci < kMlaTile * (kMlaD / 8); ci += 32) {
                        const int tr = ci / (kMlaD / 8), c = ci % (kMlaD / 8);
                        const int pos = tb + tr;
                        const bool ok = pos < k1;
                        int blk = ok ? __ldg(bt + pos / p.bs) : 0;
                        if (blk < 0 || blk >= p.num_blocks) {
                            set_error(p.err, PKA_DEVERR_BLOCK_ID);
                            blk = 0;
                        }
                        const int64_t row = (int64_t)blk * p.bs + (ok ? pos % p.bs : 0);
                        cp_async_16_zfill(base + mla_tile_off(tr, c), p.kv + row * kMlaD + c * 8, ok);
                    }
                    // each lane's copies count on the barrier; lane 0's plain
                    // arrive is the phase's one expected arrival
                    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(&full[stage]))
                                 : "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[stage]);
                }
                ++ld_it;
            }
        } else {
            // Q of this head group -> smem [9 segs][HG rows][128 B]
            {
                const uint32_t qs = smem_u32(smem);
                for (int ci = threadIdx.x; ci < HG * (kMlaD / 8); ci += NW * 32) {
                    const int hr = ci / (kMlaD / 8), c = ci % (kMlaD / 8);
                    cp_async_16(qs + sw128((uint32_t)((c >> 3) * HG + hr), (uint32_t)(c & 7)),
                                p.q + ((int64_t)r * p.Hq + h0 + hr) * kMlaD + c * 8);
                }
                cp_async_commit();
                cp_async_wait<0>();
            }
            asm volatile("bar.sync 1, %0;" ::"n"(NW * 32));  // Q visible to all compute warps
            const uint32_t qs = smem_u32(smem);
            float o[kMlaDv / 16][4];
#pragma unroll
            for (int i = 0; i < kMlaDv / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
            const int mi = lane >> 3;
            for (int j = 0; j < ntiles; ++j) {
                if (!alive) break;
                const int stage = cs_it % kMlaStages;
                if (!mbar_wait(&full[stage], (cs_it / kMlaStages) & 1, p.err)) {
                    alive = false;
                    s_abort = 1;
                    break;
                }
                ++cs_it;
                uint8_t* tile = ring + stage * kMlaTileBytes;
                const int tb = k0 + j * kMlaTile;
                const int valid = min(kMlaTile, k1 - tb);
                const uint32_t tbase = smem_u32(tile);
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int ks = 0; ks < kMlaD / 16; ++ks) {
                    uint32_t a0, a1, a2, a3, b0, b1;
                    ldsm_x4(tbase + mla_tile_off((mi & 1) * 8 + (lane & 7), ks * 2 + (mi >> 1)), a0, a1, a2, a3);
                    const int c = ks * 2 + ((lane >> 3) & 1);
                    ldsm_x2(qs + sw128((uint32_t)((c >> 3) * HG + warp * 8 + (lane & 7)), (uint32_t)(c & 7)), b0, b1);
                    mma_bf16(sc, a0, a1, a2, a3, b0, b1);
                }
                const bool v0 = (lane >> 2) < valid, v1 = (lane >> 2) + 8 < valid;
                float x[4];
                x[0] = v0 ? sc[0] * p.scale_log2 : -INFINITY;
                x[1] = v0 ? sc[1] * p.scale_log2 : -INFINITY;
                x[2] = v1 ? sc[2] * p.scale_log2 : -INFINITY;
                x[3] = v1 ? sc[3] * p.scale_log2 : -INFINITY;
                float alpha[2], pr[4];
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    float mx = fmaxf(x[hc], x[hc + 2]);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float mn = fmaxf(m[hc], mx);
                    alpha[hc] = fast_exp2(m[hc] - mn);
                    m[hc] = mn;
                    pr[hc] = fast_exp2(x[hc] - mn);
                    pr[hc + 2] = fast_exp2(x[hc + 2] - mn);
                    l[hc] = l[hc] * alpha[hc] + pr[hc] + pr[hc + 2];
                }
                const uint32_t pb0 = movmatrix_t(pack_bf16(pr[0], pr[1]));
                const uint32_t pb1 = movmatrix_t(pack_bf16(pr[2], pr[3]));
#pragma unroll
                for (int mt = 0; mt < kMlaDv / 16; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(tbase + mla_tile_off((mi >> 1) * 8 + (lane & 7), mt * 2 + (mi & 1)), a0, a1, a2, a3);
                    o[mt][0] *= alpha[0];
                    o[mt][1] *= alpha[1];
                    o[mt][2] *= alpha[0];
                    o[mt][3] *= alpha[1];
                    mma_bf16(o[mt], a0, a1, a2, a3, pb0, pb1);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
            }
            // finalize this warp's 8 heads
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                l[hc] += __shfl_xor_sync(0xffffffffu, l[hc], 4);
                l[hc] += __shfl_xor_sync(0xffffffffu, l[hc], 8);
                l[hc] += __shfl_xor_sync(0xffffffffu, l[hc], 16);
            }
            const bool direct = p.nsplit[r] == 1;
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                const int h = h0 + warp * 8 + (lane & 3) * 2 + hc;
                const float inv = 1.f / l[hc];
                const float lse_nat = (m[hc] + __log2f(l[hc])) * 0.69314718055994531f;
                if (direct) {
                    __nv_bfloat16* dst = p.out + ((int64_t)r * p.Hq + h) * kMlaDv + (lane >> 2);
#pragma unroll
                    for (int mt = 0; mt < kMlaDv / 16; ++mt) {
                        dst[mt * 16] = __float2bfloat16_rn(o[mt][hc] * inv);
                        dst[mt * 16 + 8] = __float2bfloat16_rn(o[mt][hc + 2] * inv);
                    }
                    if (p.lse && lane < 4) p.lse[(int64_t)r * p.Hq + h] = lse_nat;
                } else {
                    const int64_t row = (int64_t)pair * p.Hq + h;
                    float* dst = p.part_o + row * kMlaDv + (lane >> 2);
#pragma unroll
                    for (int mt = 0; mt < kMlaDv / 16; ++mt) {
                        dst[mt * 16] = o[mt][hc] * inv;
                        dst[mt * 16 + 8] = o[mt][hc + 2] * inv;
                    }
                    if (lane < 4) p.part_lse[row] = lse_nat;
                }
            }
        }
        __syncthreads();  // Q smem and the ring are reused by the next unit
    }
    if (producer && !alive) {
        // drain: wait (bounded) for the last tile issued into each stage
        for (uint32_t t = ld_it > (uint32_t)kMlaStages ? ld_it - kMlaStages : 0u; t < ld_it; ++t)
            mbar_wait(&full[t % kMlaStages], (t / kMlaStages) & 1, p.err);
    }
}

template <int NW, bool kTma>
static cudaError_t launch_mla(const CUtensorMap& map, const DecodeMlaParams& p, int num_sms,
                             cudaStream_t stream) {
    auto kern = decode_mla_kernel<NW, kTma>;
    const int smem = MlaSmem<NW>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, (NW + 1) * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    return launch_dependent(kern, dim3(num_sms * per_sm), dim3((NW + 1) * 32), smem, stream, map, p);
}

cudaError_t launch_decode_mla(const CUtensorMap& map, const DecodeMlaParams& p, bool tma, int num_sms,
                              cudaStream_t stream) {
    const int hg = p.Hq >= 64 ? 64 : p.Hq;
    if (hg == 64) return tma ? launch_mla<8, true>(map, p, num_sms, stream) : launch_mla<8, false>(map, p, num_sms, stream);
    if (hg == 32) return tma ? launch_mla<4, true>(map, p, num_sms, stream) : launch_mla<4, false>(map, p, num_sms, stream);
    if (hg == 16) return tma ? launch_mla<2, true>(map, p, num_sms, stream) : launch_mla<2, false>(map, p, num_sms, stream);
    return cudaErrorInvalidValue;
}

int decode_mla_heads_per_cta(int Hq) { return Hq >= 64 ? 64 : Hq; }

}  // namespace pka
