// decode_gqa_fp8.cu -- the split-KV GQA decode over an 8-bit KV cache
// (FP8 E4M3 codes with one scale per tensor for K and one for V), the cache
// the pages dequantise while gathering it ("Beyond porting", absorbed /
// non-absorbed recipe, the prefill listing's gather_and_maybe_dequant_cache
// step). Decode is bound by the cache bytes it streams, so an 8-bit cache
// halves its time; the codes are widened on the fly, never written back.
//
// Work unit (request, split, kv head), as in decode_gqa.cu, but a whole unit
// belongs to one warp: each warp takes units from the planner's counter on
// its own, streams the unit's 16-key tiles through a private ring loaded by
// TMA straight through the block table, and writes the unit's result from
// registers -- no shared-memory merge and no block-wide barrier, so a warp
// never waits for another. The ring runs across unit boundaries: the warp
// knows its next unit one unit ahead and starts loading its tiles while the
// current unit's last tiles are consumed. (With half the bytes per key, the
// per-unit costs of the bf16 kernel's CTA-wide units would no longer hide
// behind the stream.) Head dim 128. How the MMA fragments are built:
//
//   * Every E4M3 value is exactly an f16 value (4-bit exponent, 3-bit
//     mantissa, subnormals down to 2^-9), so the tensor-core products run on
//     f16 operands: cvt.rn.f16x2.e4m3x2 widens two codes per instruction.
//     q (bf16) is converted to f16 once per unit (exact for 2^-14 <= |q| <
//     65504; the call requires |q| < 65504), P is packed as f16.
//   * The scales come out of the sums: the score scale becomes
//     scale * k_scale, and the merged output is multiplied by v_scale.
//   * S^T = K . Q^T: a dot product does not care in which order its terms
//     are summed, so lane (c = lane % 4) takes dims [32c, 32c + 32) of its two
//     key rows with two 16-byte loads, and k-step ks uses dims 32c + 4ks ..
//     +3; q's fragments follow the same order.
//   * O^T += V^T . P^T contracts over keys while a V row holds dims: lane
//     (r = lane / 4, c) reads dims [16r, 16r + 16) of its four keys (2c, 2c+1,
//     8+2c, 9+2c) with one 16-byte load each and transposes 4 x 4 byte blocks
//     with prmt; O^T row r of m-tile 2p then holds dim 16r + 4p, row r + 8
//     dim 16r + 4p + 1, and m-tile 2p + 1 dims 16r + 4p + 2 and + 3.
// Tiles are 16 rows x 128 bytes in the 128-byte swizzle, so both access
// patterns read 8 distinct 16-byte columns per quarter warp (no bank
// conflicts).
#include "common.cuh"
#include "params.cuh"
#include "plan.cuh"

namespace pka {

namespace {

constexpr int kF8Warps = 4;
constexpr int kF8Threads = kF8Warps * 32;
constexpr int kF8Tile = 16;            // keys per tile
constexpr int kF8D = 128;              // head dim (bytes per cache row)
constexpr int kF8TileBytes = kF8Tile * kF8D;       // 2 KB
constexpr int kF8StageBytes = 2 * kF8TileBytes;    // K + V

// Per head-group width NT (8 query heads per 8-wide MMA column block): tiles
// in flight per warp and CTAs per SM. One group (G <= 8) keeps 16 warps per
// SM (four 48 KB CTAs, registers capped at 128) so the warps' dependent MMA /
// softmax chains hide each other; two groups need more registers per thread.
template <int NT>
struct F8Cfg {
    static constexpr int kStages = NT == 1 ? 3 : 6;
    static constexpr int kMinBlocks = NT == 1 ? 4 : 2;
    static constexpr int kRingBytes = kF8Warps * kStages * kF8StageBytes;
    static constexpr int kSmem = kRingBytes + 1024 + 64 * 8;
};

PKA_DEVICE uint32_t e4m3_lo(uint32_t w) { return e4m3x2_to_f16x2(w & 0xffffu); }
PKA_DEVICE uint32_t e4m3_hi(uint32_t w) { return e4m3x2_to_f16x2(w >> 16); }

// bf16 pair -> f16 pair (finite results saturate at the f16 maximum).
PKA_DEVICE uint32_t bf16x2_to_f16x2(uint32_t w) {
    uint32_t d;
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

PKA_DEVICE uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
PKA_DEVICE void mma_f16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

PKA_DEVICE uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

}  // namespace

// One decode work unit as a warp sees it. blk[0] / blk[1]: validated block
// ids of the unit's TMA boxes `lane` and 32 + lane (a box is min(bs, 16) rows
// of one block), loaded when the unit is fetched, so issuing a tile's loads
// only shuffles them out of registers.
struct F8Unit {
    int unit, pair, g, r, k0, k1, ntiles;  // unit < 0: none
    int blk[2];
};

PKA_DEVICE int f8_block_id(const DecodeGqaParams& p, const int32_t* bt, int pos) {
    int blk = __ldg(bt + pos / p.bs);
    if (blk < 0 || blk >= p.num_blocks) {
        set_error(p.err, PKA_DEVERR_BLOCK_ID);
        blk = 0;
    }
    return blk;
}

// Call with the whole warp (the unit index is warp-uniform).
PKA_DEVICE F8Unit f8_unit(const DecodeGqaParams& p, int u, int num_units, int L, int lane) {
    F8Unit U;
    U.unit = -1;
    U.ntiles = 0;
    U.blk[0] = U.blk[1] = 0;
    if (u < 0 || u >= num_units) return U;
    U.unit = u;
    U.pair = u / p.Hkv;
    U.g = u - U.pair * p.Hkv;
    const int2 rs = p.pairs[U.pair];
    U.r = rs.x;
    U.k0 = rs.y * L;
    U.k1 = min(U.k0 + L, p.seq_lens[U.r]);
    U.ntiles = U.k1 > U.k0 ? (U.k1 - U.k0 + kF8Tile - 1) / kF8Tile : 0;
    if (p.bs >= 8) {
        const int boxr = p.bs < kF8Tile ? p.bs : kF8Tile;
        const int32_t* bt = p.block_table + (int64_t)U.r * p.max_blocks;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int pos = U.k0 + (32 * i + lane) * boxr;
            if (pos < U.k1) U.blk[i] = f8_block_id(p, bt, pos);
        }
    }
    return U;
}

template <int NT, bool kTma>
__global__ void __launch_bounds__(kF8Threads, F8Cfg<NT>::kMinBlocks)
    decode_gqa_fp8_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const DecodeGqaParams p) {
    grid_dep_wait();
    constexpr int kKSteps = kF8D / 16;
    constexpr int kF8Stages = F8Cfg<NT>::kStages;
    constexpr int kF8RingBytes = F8Cfg<NT>::kRingBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kF8RingBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c4 = lane & 3, r8 = lane >> 2;
    const int num_units = p.hdr->dec_num_pairs * p.Hkv;
    if (num_units == 0) return;
    const int L = p.hdr->dec_split_len;

    uint64_t* full = bars + warp * kF8Stages;
    if (lane == 0) {
        for (int s = 0; s < kF8Stages; ++s) mbar_init(&full[s], kTma ? 1 : 32);
        fence_barrier_init();
        if (kTma && warp == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
        }
    }
    __syncwarp();
    // From here on every warp runs on its own: it takes whole units from the
    // counter and never synchronises with the other warps.
    const uint64_t pol = policy_evict_first();
    uint8_t* ring = smem + warp * kF8Stages * kF8StageBytes;
    uint32_t ld_it = 0, cs_it = 0;  // tiles issued / consumed by this warp

    auto fetch = [&]() -> F8Unit {
        int u = 0;
        if (lane == 0) u = atomicAdd(p.counter, 1);
        u = __shfl_sync(0xffffffffu, u, 0);
        return f8_unit(p, u, num_units, L, lane);
    };
    F8Unit cur = fetch();
    F8Unit nxt = cur.unit >= 0 ? fetch() : cur;
    // load cursor: tile `lt` of cur (lw == 0) or of nxt (lw == 1)
    int lw = 0, lt = 0;

    // issue the next tile along the cursor into stage ld_it % kF8Stages;
    // false when nothing can be issued yet (next unit not known or none)
    auto issue_next = [&]() -> bool {
        if (lw == 0 && lt >= cur.ntiles) {
            lw = 1;
            lt = 0;
        }
        // the cursor's unit, field by field (a reference to one of two structs
        // would put both in local memory)
        F8Unit U;
        U.unit = lw ? nxt.unit : cur.unit;
        U.ntiles = lw ? nxt.ntiles : cur.ntiles;
        U.g = lw ? nxt.g : cur.g;
        U.r = lw ? nxt.r : cur.r;
        U.k0 = lw ? nxt.k0 : cur.k0;
        U.k1 = lw ? nxt.k1 : cur.k1;
        U.blk[0] = lw ? nxt.blk[0] : cur.blk[0];
        U.blk[1] = lw ? nxt.blk[1] : cur.blk[1];
        if (U.unit < 0 || lt >= U.ntiles) return false;
        const int stage = ld_it % kF8Stages;
        uint8_t* kdst = ring + stage * kF8StageBytes;
        uint8_t* vdst = kdst + kF8TileBytes;
        const int tb = U.k0 + lt * kF8Tile;
        const int32_t* bt = p.block_table + (int64_t)U.r * p.max_blocks;
        if constexpr (kTma) {
            const int boxr = p.bs < kF8Tile ? p.bs : kF8Tile;
            const int nsub = kF8Tile / boxr;  // 1 or 2 boxes per tile
            // the tile's block ids: from the unit's registers (boxes < 64), else loaded
            const int b0 = lt * nsub, b1 = b0 + nsub - 1;  // the tile's first and last box
            int blk, blk1;
            if (b1 < 64) {
                blk = __shfl_sync(0xffffffffu, b0 < 32 ? U.blk[0] : U.blk[1], b0 & 31);
                blk1 = __shfl_sync(0xffffffffu, b1 < 32 ? U.blk[0] : U.blk[1], b1 & 31);
            } else {
                blk = lane == 0 ? f8_block_id(p, bt, tb) : 0;
                blk1 = (lane == 0 && nsub > 1 && tb + boxr < U.k1) ? f8_block_id(p, bt, tb + boxr) : 0;
            }
            if (lane == 0) {
                fence_proxy_async_smem();
                const int nbox = (nsub > 1 && tb + boxr < U.k1) ? 2 : 1;
                mbar_arrive_expect_tx(&full[stage], (uint32_t)(2 * nbox * boxr * kF8D));
                for (int sb = 0; sb < nbox; ++sb) {
                    const int ps = tb + sb * boxr;
                    const int row = ((sb ? blk1 : blk) * p.Hkv + U.g) * p.bs + (ps % p.bs);
                    tma_load_2d(kdst + sb * boxr * kF8D, &kmap, &full[stage], 0, row, pol);
                    tma_load_2d(vdst + sb * boxr * kF8D, &vmap, &full[stage], 0, row, pol);
                }
            }
            __syncwarp();
        } else {
            // 16-byte copies into the same swizzled layout: 16 rows x 8 pieces
            const uint32_t kbase = smem_u32(kdst), vbase = smem_u32(vdst);
            for (int ci = lane; ci < kF8Tile * 8; ci += 32) {
                const int tr = ci >> 3, c = ci & 7;
                const int pos = tb + tr;
                if (pos >= U.k1) continue;
                int blk = __ldg(bt + pos / p.bs);
                if (blk < 0 || blk >= p.num_blocks) {
                    set_error(p.err, PKA_DEVERR_BLOCK_ID);
                    blk = 0;
                }
                const int64_t row = ((int64_t)blk * p.Hkv + U.g) * p.bs + (pos % p.bs);
                cp_async_16(kbase + sw128(tr, c), p.k8 + row * kF8D + c * 16);
                cp_async_16(vbase + sw128(tr, c), p.v8 + row * kF8D + c * 16);
            }
            cp_async_arrive_noinc(&full[stage]);
        }
        ++ld_it;
        ++lt;
        return true;
    };

    bool alive = true;  // false once a wait timed out: stop issuing and consuming
    while (alive && cur.unit >= 0) {
        while (ld_it - cs_it < (uint32_t)kF8Stages && issue_next()) {
        }
        const int r = cur.r, g = cur.g;

        // Q^T fragments (B operand, f16): head g*G + n (n = lane / 4), k-step ks
        // holds dims 32c + 4ks .. +3; zero beyond G.
        uint32_t qf[NT][kKSteps][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hh = nt * 8 + r8;
            const bool ok = hh < p.G;
            const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((int64_t)r * p.Hq + g * p.G + (ok ? hh : 0)) * kF8D +
                                                               32 * c4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // 8 dims = two k-steps per 16-byte load
                const uint4 v = ok ? __ldg(qrow + j) : make_uint4(0, 0, 0, 0);
                qf[nt][2 * j][0] = bf16x2_to_f16x2(v.x);
                qf[nt][2 * j][1] = bf16x2_to_f16x2(v.y);
                qf[nt][2 * j + 1][0] = bf16x2_to_f16x2(v.z);
                qf[nt][2 * j + 1][1] = bf16x2_to_f16x2(v.w);
            }
        }

        float o[kKSteps][NT][4];
        float m[NT][2], l[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m[nt][0] = m[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < kKSteps; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
        }

        for (int t = 0; t < cur.ntiles; ++t) {
            const int stage = cs_it % kF8Stages;
            if (!mbar_wait_warp(&full[stage], (cs_it / kF8Stages) & 1, p.err)) {
                alive = false;
                break;
            }
            ++cs_it;
            uint8_t* kt = ring + stage * kF8StageBytes;
            uint8_t* vt = kt + kF8TileBytes;
            const int tb = cur.k0 + t * kF8Tile;
            const int valid = min(kF8Tile, cur.k1 - tb);
            if (valid < kF8Tile) {  // zero V rows past the end (stale bytes may decode to NaN)
                for (int ci = lane; ci < (kF8Tile - valid) * 8; ci += 32) {
                    const int tr = valid + (ci >> 3);
                    *reinterpret_cast<uint4*>(vt + sw128(tr, ci & 7)) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            const uint32_t kb = smem_u32(kt), vb = smem_u32(vt);

            // S^T = K . Q^T: rows r8 and r8 + 8, dims [32c, 32c + 32) as two 16-byte pieces each
            float sc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int jc = 0; jc < 2; ++jc) {
                const uint4 lo = lds128(kb + sw128(r8, 2 * c4 + jc));
                const uint4 hi = lds128(kb + sw128(r8 + 8, 2 * c4 + jc));
                const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w}, wh[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ks = 4 * jc + i;
                    const uint32_t a0 = e4m3_lo(wl[i]), a1 = e4m3_lo(wh[i]);
                    const uint32_t a2 = e4m3_hi(wl[i]), a3 = e4m3_hi(wh[i]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_f16(sc[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
                }
            }
            // V fragments of this tile: keys 2c, 2c+1, 8+2c, 9+2c; dims [16 r8, 16 r8 + 16)
            const uint4 w0 = lds128(vb + sw128(2 * c4, r8));
            const uint4 w1 = lds128(vb + sw128(2 * c4 + 1, r8));
            const uint4 w2 = lds128(vb + sw128(8 + 2 * c4, r8));
            const uint4 w3 = lds128(vb + sw128(9 + 2 * c4, r8));

            // mask keys past the end, scale into log2 domain (k_scale folded in)
            const bool v0 = r8 < valid, v1 = r8 + 8 < valid;
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
                if (alpha[0] != 1.f || alpha[1] != 1.f) {  // the running max moved: rescale O
#pragma unroll
                    for (int mt = 0; mt < kKSteps; ++mt) {
                        o[mt][nt][0] *= alpha[0];
                        o[mt][nt][1] *= alpha[1];
                        o[mt][nt][2] *= alpha[0];
                        o[mt][nt][3] *= alpha[1];
                    }
                }
                pb[nt][0] = movmatrix_t(pack_f16(pr[0], pr[1]));  // keys 0-7
                pb[nt][1] = movmatrix_t(pack_f16(pr[2], pr[3]));  // keys 8-15
            }
            // O^T += V^T . P^T
            {
                const uint32_t k0w[4] = {w0.x, w0.y, w0.z, w0.w}, k1w[4] = {w1.x, w1.y, w1.z, w1.w};
                const uint32_t k2w[4] = {w2.x, w2.y, w2.z, w2.w}, k3w[4] = {w3.x, w3.y, w3.z, w3.w};
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    // 4 keys x 4 dims: pair the keys' bytes per dim
                    const uint32_t x01 = __byte_perm(k0w[pp], k1w[pp], 0x5140);  // dims +0, +1
                    const uint32_t x23 = __byte_perm(k2w[pp], k3w[pp], 0x5140);
                    const uint32_t y01 = __byte_perm(k0w[pp], k1w[pp], 0x7362);  // dims +2, +3
                    const uint32_t y23 = __byte_perm(k2w[pp], k3w[pp], 0x7362);
                    {
                        const uint32_t a0 = e4m3_lo(x01), a1 = e4m3_hi(x01), a2 = e4m3_lo(x23), a3 = e4m3_hi(x23);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma_f16(o[2 * pp][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                    }
                    {
                        const uint32_t a0 = e4m3_lo(y01), a1 = e4m3_hi(y01), a2 = e4m3_lo(y23), a3 = e4m3_hi(y23);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_f16(o[2 * pp + 1][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                    }
                }
            }
            // every lane's reads of the stage are in registers and used: refill it
            __syncwarp();
            issue_next();
        }
        if (!alive) break;

        // ---- the unit's result straight from registers: O / l (times v_scale)
        // per head, bf16 to out when the request has one split, else fp32 partials
        const bool direct = p.nsplit[r] == 1;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                float lt_ = l[nt][hc];
                lt_ += __shfl_xor_sync(0xffffffffu, lt_, 4);
                lt_ += __shfl_xor_sync(0xffffffffu, lt_, 8);
                lt_ += __shfl_xor_sync(0xffffffffu, lt_, 16);
                const int hh = nt * 8 + c4 * 2 + hc;
                if (hh >= p.G) continue;
                const int h = g * p.G + hh;
                const float inv = p.v_scale / lt_;  // the value codes' scale comes out of the sum
                const float lse_nat = (m[nt][hc] + __log2f(lt_)) * 0.69314718055994531f;
                // m-tile 2pp row r8 = dim 16 r8 + 4pp, row r8 + 8 = +1; m-tile 2pp+1: +2, +3
                if (direct) {
                    __nv_bfloat16* dst = p.out + ((int64_t)r * p.Hq + h) * kF8D + 16 * r8;
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp)
                        *reinterpret_cast<uint2*>(dst + 4 * pp) =
                            make_uint2(pack_bf16(o[2 * pp][nt][hc] * inv, o[2 * pp][nt][hc + 2] * inv),
                                       pack_bf16(o[2 * pp + 1][nt][hc] * inv, o[2 * pp + 1][nt][hc + 2] * inv));
                    if (p.lse && r8 == 0) p.lse[(int64_t)r * p.Hq + h] = lse_nat;
                } else {
                    const int64_t row = (int64_t)cur.pair * p.Hq + h;
                    float* dst = p.part_o + row * kF8D + 16 * r8;
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp)
                        *reinterpret_cast<float4*>(dst + 4 * pp) =
                            make_float4(o[2 * pp][nt][hc] * inv, o[2 * pp][nt][hc + 2] * inv,
                                        o[2 * pp + 1][nt][hc] * inv, o[2 * pp + 1][nt][hc + 2] * inv);
                    if (r8 == 0) p.part_lse[row] = lse_nat;
                }
            }
        // next unit: the one already being loaded; look one further ahead
        // (every tile of the old unit was issued; the cursor is in nxt, or at
        // the old unit's end if it has not stepped over yet: then at nxt's start)
        cur = nxt;
        if (lw == 0) lt = 0;
        lw = 0;
        nxt = cur.unit >= 0 ? fetch() : cur;
    }
    grid_dep_launch();  // out of work: the split reduction may start launching
    // No copy may outlive the CTA: wait (bounded) for every tile issued and
    // never consumed (after a timeout, or loads of units nobody ran).
    while (cs_it < ld_it) {
        mbar_wait_warp(&full[cs_it % kF8Stages], (cs_it / kF8Stages) & 1, p.err);
        ++cs_it;
    }
}

template <int NT, bool kTma>
static cudaError_t launch_fp8(const CUtensorMap& km, const CUtensorMap& vm, const DecodeGqaParams& p, int num_sms,
                              cudaStream_t stream) {
    auto kern = decode_gqa_fp8_kernel<NT, kTma>;
    constexpr int kF8Smem = F8Cfg<NT>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8Smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kF8Threads, kF8Smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    return launch_dependent(kern, dim3(num_sms * per_sm), dim3(kF8Threads), kF8Smem, stream, km, vm, p);
}

cudaError_t launch_decode_gqa_fp8(const CUtensorMap& km, const CUtensorMap& vm, const DecodeGqaParams& p, bool tma,
                                  int num_sms, cudaStream_t stream) {
    const bool nt2 = p.G > 8;
    if (tma) return nt2 ? launch_fp8<2, true>(km, vm, p, num_sms, stream) : launch_fp8<1, true>(km, vm, p, num_sms, stream);
    return nt2 ? launch_fp8<2, false>(km, vm, p, num_sms, stream) : launch_fp8<1, false>(km, vm, p, num_sms, stream);
}

// Work units for the 8-bit kernel: one warp owns a unit, so more units than the
// CTA-wide bf16 kernel balance the warps better (measured on the 256-request
// decode workload: 48 per SM 0.229 ms, 72 per SM 0.218 ms, 96 per SM 0.215 ms,
// 128 per SM 0.224 ms as the splits reach their minimum length).
int decode_gqa_fp8_target_units(int num_sms) { return num_sms * 72; }

}  // namespace pka
