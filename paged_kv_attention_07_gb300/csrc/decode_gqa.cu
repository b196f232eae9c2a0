// decode_gqa.cu -- memory-bound split-KV paged decode for grouped-query
// attention (the pages' decode path: "each decode step loads the whole KV
// cache from memory to produce one token; the bottleneck is memory
// bandwidth", served on ROCm by pa_fwd_asm; "Beyond porting", section
// "Three-path processing explained", decode path).
//
// Work unit: (decode request r, key split s, kv head g). The planner cuts
// every request's keys [0, seq_len) into splits of `dec_split_len` keys; a
// persistent CTA pulls units from an atomic counter. The G = Hq / Hkv query
// heads of kv head g share every K/V tile.
//
// Data movement: the cache is [num_blocks, Hkv, bs, d] bf16, so 16 keys of
// one (block, kv head) are one contiguous 16 x d tile. Each warp owns a ring
// of kStages tiles; lane 0 fetches a tile with 2-D TMA boxes of 64 columns x
// 16 rows (128-byte swizzle) straight through the block table, so the
// gather costs no extra pass. Block sizes below 8 use 16-byte cp.async
// copies into the same swizzled layout.
//
// Math per 16-key tile, per warp (bf16 tensor cores, fp32 accumulate):
//   S^T[16 keys x 8 heads] = K[16 x d] . Q^T[d x 8]       (m16n8k16, A = K)
//   online softmax over keys per head (warp shuffles), P^T -> bf16
//   O^T[d x 8 heads]     += V^T[d x 16] . P^T[16 x 8]      (A = V^T via ldmatrix.trans)
// The 8 heads of a group fill the MMA's n = 8 exactly; movmatrix turns the
// S^T accumulator fragment into the P^T operand fragment in registers.
// Warps' partial (m, l, O) merge in shared memory; a request with one split
// writes bf16 out + lse directly, otherwise fp32 partials for the reduce.
#include "common.cuh"
#include "params.cuh"
#include "plan.cuh"

namespace pka {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecStages = 3;  // tiles in flight per warp
constexpr int kTile = 16;      // keys per tile


template <int D>
struct DecGqaSmem {
    static constexpr int kTileBytes = kTile * D * 2;        // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;       // K + V
    static constexpr int kRingBytes = kDecWarps * kDecStages * kStageBytes;
    static constexpr int kBytes = kRingBytes + 1024 /*align*/ + 64 * 8 /*barriers*/;
};

// Smem offset of row `tr` (0..15), 16-byte chunk `c` (0..D/8-1) of a tile
// stored as [D/64 segments][16 rows][128 B], 128-byte swizzled.
template <int D>
PKA_DEVICE uint32_t tile_off(int tr, int c) {
    return sw128((uint32_t)((c >> 3) * kTile + tr), (uint32_t)(c & 7));
}

template <int D, int NT, bool kTma>
__global__ void __launch_bounds__(kDecThreads, 2)
    decode_gqa_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const DecodeGqaParams p) {
    grid_dep_wait();
    using S = DecGqaSmem<D>;
    constexpr int kSeg = D / 64;
    constexpr int kKSteps = D / 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kRingBytes);
    __shared__ int s_unit;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_units = p.hdr->dec_num_pairs * p.Hkv;
    if (num_units == 0) return;
    const int L = p.hdr->dec_split_len;

    uint64_t* full = bars + warp * kDecStages;
    if (lane == 0) {
        for (int s = 0; s < kDecStages; ++s) mbar_init(&full[s], kTma ? 1 : 32);
        fence_barrier_init();
    }
    if (threadIdx.x == 0) {
        s_abort = 0;
        if (kTma) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
        }
    }
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    uint8_t* ring = smem + warp * kDecStages * S::kStageBytes;
    uint32_t ld_it = 0, cs_it = 0;  // tiles issued / consumed by this warp (all units)
    bool alive = true;  // false once a wait of this warp timed out

    for (;;) {
        if (threadIdx.x == 0) s_unit = s_abort ? num_units : atomicAdd(p.counter, 1);
        __syncthreads();
        const int unit = s_unit;
        __syncthreads();
        if (unit >= num_units) {
            grid_dep_launch();  // out of work: the split reduction may start launching
            break;
        }
        const int pair = unit / p.Hkv, g = unit - pair * p.Hkv;
        const int2 rs = p.pairs[pair];
        const int r = rs.x, split = rs.y;
        const int slen = p.seq_lens[r];
        const int k0 = split * L;
        const int k1 = min(k0 + L, slen);
        const int ntiles = (k1 - k0 + kTile - 1) / kTile;
        const int my_n = ntiles > warp ? (ntiles - warp + kDecWarps - 1) / kDecWarps : 0;
        const int32_t* bt = p.block_table + (int64_t)r * p.max_blocks;

        // Q^T fragments (B operand): heads g*G + n, n < G; zero beyond G.
        uint32_t qf[NT][kKSteps][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hh = nt * 8 + (lane >> 2);
            const bool ok = hh < p.G;
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                p.q + ((int64_t)r * p.Hq + g * p.G + (ok ? hh : 0)) * D);
#pragma unroll
            for (int ks = 0; ks < kKSteps; ++ks) {
                qf[nt][ks][0] = ok ? __ldg(qrow + ks * 8 + (lane & 3)) : 0u;
                qf[nt][ks][1] = ok ? __ldg(qrow + ks * 8 + 4 + (lane & 3)) : 0u;
            }
        }

        // issue the loads of this warp's j-th tile into stage (ld_it % kDecStages)
        auto issue = [&](int j) {
            const int stage = ld_it % kDecStages;
            uint8_t* kdst = ring + stage * S::kStageBytes;
            uint8_t* vdst = kdst + S::kTileBytes;
            const int tb = k0 + (warp + j * kDecWarps) * kTile;
            if constexpr (kTma) {
                if (lane == 0) {
                    fence_proxy_async_smem();
                    const int boxr = p.bs < kTile ? p.bs : kTile;
                    const int nsub = kTile / boxr;
                    int nbox = 0;
                    for (int sb = 0; sb < nsub; ++sb)
                        if (tb + sb * boxr < k1) ++nbox;
                    mbar_arrive_expect_tx(&full[stage], (uint32_t)(2 * nbox * kSeg * boxr * 128));
                    for (int sb = 0; sb < nbox; ++sb) {
                        const int pos = tb + sb * boxr;
                        int blk = __ldg(bt + pos / p.bs);
                        if (blk < 0 || blk >= p.num_blocks) {
                            set_error(p.err, PKA_DEVERR_BLOCK_ID);
                            blk = 0;
                        }
                        const int row = (blk * p.Hkv + g) * p.bs + (pos % p.bs);
#pragma unroll
                        for (int sg = 0; sg < kSeg; ++sg) {
                            const int off = (sg * kTile + sb * boxr) * 128;
                            tma_load_2d(kdst + off, &kmap, &full[stage], sg * 64, row, pol);
                            tma_load_2d(vdst + off, &vmap, &full[stage], sg * 64, row, pol);
                        }
                    }
                }
            } else {
                constexpr int kChunks = kTile * D / 8;  // 16-byte chunks per tile
                const uint32_t kbase = smem_u32(kdst), vbase = smem_u32(vdst);
                for (int ci = lane; ci < kChunks; ci += 32) {
                    const int tr = ci / (D / 8), c = ci % (D / 8);
                    const int pos = tb + tr;
                    if (pos >= k1) continue;
                    int blk = __ldg(bt + pos / p.bs);
                    if (blk < 0 || blk >= p.num_blocks) {
                        set_error(p.err, PKA_DEVERR_BLOCK_ID);
                        blk = 0;
                    }
                    const int64_t row = ((int64_t)blk * p.Hkv + g) * p.bs + (pos % p.bs);
                    cp_async_16(kbase + tile_off<D>(tr, c), p.k_cache + row * D + c * 8);
                    cp_async_16(vbase + tile_off<D>(tr, c), p.v_cache + row * D + c * 8);
                }
                cp_async_arrive_noinc(&full[stage]);
            }
            ++ld_it;
        };

        float o[kKSteps][NT][4];
        float m[NT][2], l[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m[nt][0] = m[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < kKSteps; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
        }

        const int npro = my_n < kDecStages ? my_n : kDecStages;
        if (alive)
            for (int j = 0; j < npro; ++j) issue(j);

        for (int j = 0; j < my_n; ++j) {
            if (!alive) continue;  // after a timeout: no waits, no reads, no new copies
            const int stage = cs_it % kDecStages;
            const uint32_t parity = (cs_it / kDecStages) & 1;
            if (!mbar_wait(&full[stage], parity, p.err)) {
                alive = false;
                s_abort = 1;
                continue;
            }
            ++cs_it;
            uint8_t* kt = ring + stage * S::kStageBytes;
            uint8_t* vt = kt + S::kTileBytes;
            const int tb = k0 + (warp + j * kDecWarps) * kTile;
            const int valid = min(kTile, k1 - tb);
            if (valid < kTile) {  // zero V rows past the end (they may hold NaN)
                for (int ci = lane; ci < (kTile - valid) * (D / 8); ci += 32) {
                    const int tr = valid + ci / (D / 8), c = ci % (D / 8);
                    *reinterpret_cast<uint4*>(vt + tile_off<D>(tr, c)) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            const uint32_t kb = smem_u32(kt), vb = smem_u32(vt);

            // S^T = K . Q^T
            float sc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
            {
                const int mi = lane >> 3;
                const int tr = (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int ks = 0; ks < kKSteps; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(kb + tile_off<D>(tr, ks * 2 + (mi >> 1)), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16(sc[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
                }
            }
            // mask keys past the end, scale into log2 domain
            const bool v0 = (lane >> 2) < valid, v1 = (lane >> 2) + 8 < valid;
            uint32_t pb[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float x[4];
                x[0] = v0 ? sc[nt][0] * p.scale_log2 : -INFINITY;
                x[1] = v0 ? sc[nt][1] * p.scale_log2 : -INFINITY;
                x[2] = v1 ? sc[nt][2] * p.scale_log2 : -INFINITY;
                x[3] = v1 ? sc[nt][3] * p.scale_log2 : -INFINITY;
                float alpha[2], pr[4];
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    float mx = fmaxf(x[hc], x[hc + 2]);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float mn = fmaxf(m[nt][hc], mx);  // finite: key 0 of the tile is valid
                    alpha[hc] = fast_exp2(m[nt][hc] - mn);
                    m[nt][hc] = mn;
                    pr[hc] = fast_exp2(x[hc] - mn);
                    pr[hc + 2] = fast_exp2(x[hc + 2] - mn);
                    l[nt][hc] = l[nt][hc] * alpha[hc] + pr[hc] + pr[hc + 2];
                }
#pragma unroll
                for (int mt = 0; mt < kKSteps; ++mt) {
                    o[mt][nt][0] *= alpha[0];
                    o[mt][nt][1] *= alpha[1];
                    o[mt][nt][2] *= alpha[0];
                    o[mt][nt][3] *= alpha[1];
                }
                pb[nt][0] = movmatrix_t(pack_bf16(pr[0], pr[1]));  // keys 0-7
                pb[nt][1] = movmatrix_t(pack_bf16(pr[2], pr[3]));  // keys 8-15
            }
            // O^T += V^T . P^T
            {
                const int mi = lane >> 3;
                const int tr = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
                for (int mt = 0; mt < kKSteps; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(vb + tile_off<D>(tr, mt * 2 + (mi & 1)), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
            }
            __syncwarp();
            if (j + kDecStages < my_n) issue(j + kDecStages);
        }

        // ---- merge the warps' partials in smem (the ring is idle now)
        __syncthreads();
        constexpr int kH = NT * 8;
        float* cm = reinterpret_cast<float*>(smem);          // [warps][kH]
        float* cl = cm + kDecWarps * kH;                     // [warps][kH]
        float* co = cl + kDecWarps * kH;                     // [warps][kH][D]
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                float lt = l[nt][hc];
                lt += __shfl_xor_sync(0xffffffffu, lt, 4);
                lt += __shfl_xor_sync(0xffffffffu, lt, 8);
                lt += __shfl_xor_sync(0xffffffffu, lt, 16);
                const int hh = nt * 8 + (lane & 3) * 2 + hc;
                if (lane < 4) {
                    cm[warp * kH + hh] = m[nt][hc];
                    cl[warp * kH + hh] = lt;
                }
#pragma unroll
                for (int mt = 0; mt < kKSteps; ++mt) {
                    co[(warp * kH + hh) * D + mt * 16 + (lane >> 2)] = o[mt][nt][hc];
                    co[(warp * kH + hh) * D + mt * 16 + (lane >> 2) + 8] = o[mt][nt][hc + 2];
                }
            }
        __syncthreads();
        const bool direct = p.nsplit[r] == 1;
        for (int it = threadIdx.x; it < p.G * (D / 4); it += kDecThreads) {
            const int hh = it / (D / 4), c4 = (it % (D / 4)) * 4;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, cm[w * kH + hh]);
            float Ls = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) {
                const float mw = cm[w * kH + hh];
                const float wt = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
                Ls += wt * cl[w * kH + hh];
                const float4 x = *reinterpret_cast<const float4*>(co + (w * kH + hh) * D + c4);
                acc.x += wt * x.x;
                acc.y += wt * x.y;
                acc.z += wt * x.z;
                acc.w += wt * x.w;
            }
            const float inv = 1.f / Ls;
            const float lse_nat = (M + __log2f(Ls)) * 0.69314718055994531f;
            const int h = g * p.G + hh;
            if (direct) {
                uint2 v;
                v.x = pack_bf16(acc.x * inv, acc.y * inv);
                v.y = pack_bf16(acc.z * inv, acc.w * inv);
                *reinterpret_cast<uint2*>(p.out + ((int64_t)r * p.Hq + h) * D + c4) = v;
                if (p.lse && c4 == 0) p.lse[(int64_t)r * p.Hq + h] = lse_nat;
            } else {
                const int64_t row = (int64_t)pair * p.Hq + h;
                *reinterpret_cast<float4*>(p.part_o + row * D + c4) =
                    make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                if (c4 == 0) p.part_lse[row] = lse_nat;
            }
        }
        // next unit's TMA writes land after these generic smem accesses
        __syncthreads();
    }
    // A warp that gave up may still have copies in flight; wait (bounded)
    // for every tile it issued and never consumed, so none outlives the CTA.
    while (cs_it < ld_it) {
        const int stage = cs_it % kDecStages;
        mbar_wait(&full[stage], (cs_it / kDecStages) & 1, p.err);
        ++cs_it;
    }
}

template <int D, int NT, bool kTma>
static cudaError_t launch_one(const CUtensorMap& km, const CUtensorMap& vm, const DecodeGqaParams& p,
                              int num_sms, cudaStream_t stream) {
    auto kern = decode_gqa_kernel<D, NT, kTma>;
    const int smem = DecGqaSmem<D>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    return launch_dependent(kern, dim3(num_sms * per_sm), dim3(kDecThreads), smem, stream, km, vm, p);
}

cudaError_t launch_decode_gqa(const CUtensorMap& km, const CUtensorMap& vm, const DecodeGqaParams& p,
                              int head_dim, bool tma, int num_sms, cudaStream_t stream) {
    const bool nt2 = p.G > 8;
    if (head_dim == 128) {
        if (tma) return nt2 ? launch_one<128, 2, true>(km, vm, p, num_sms, stream)
                            : launch_one<128, 1, true>(km, vm, p, num_sms, stream);
        return nt2 ? launch_one<128, 2, false>(km, vm, p, num_sms, stream)
                   : launch_one<128, 1, false>(km, vm, p, num_sms, stream);
    }
    if (head_dim == 64) {
        if (tma) return nt2 ? launch_one<64, 2, true>(km, vm, p, num_sms, stream)
                            : launch_one<64, 1, true>(km, vm, p, num_sms, stream);
        return nt2 ? launch_one<64, 2, false>(km, vm, p, num_sms, stream)
                   : launch_one<64, 1, false>(km, vm, p, num_sms, stream);
    }
    return cudaErrorInvalidValue;
}

// Units a launch should be split into for good balance (used by the planner
// and the workspace sizing): ~24 units per resident CTA.
// Work units the planner aims at (it sizes the split length from them). A unit
// runs on a whole CTA here, with a per-unit merge of its warps: fewer, longer
// units amortise it (measured on the 256-request decode workload: 24 per SM
// 0.360 ms, 48 per SM 0.370 ms, 72 per SM 0.390 ms; 16-24 per SM flat).
int decode_gqa_target_units(int num_sms) { return num_sms * 24; }

}  // namespace pka
