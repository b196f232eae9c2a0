// fa_fwd.cu -- varlen prefill and the extend path's pieces on the 5th-gen
// tensor cores ("Beyond porting", section "Three-path processing explained"):
//   prefill: new sequences, causal, Q/K/V in the [num_tokens, heads, dim]
//            layout (served on ROCm by flash_attn_varlen_func);
//   extend:  stage 1, the new tokens over their own keys (causal, bottom-right
//            aligned: new token i sees new keys 0..i), and stage 2, every
//            context chunk of `chunk` cached keys (no mask: all context
//            precedes the new tokens), each emitting (O, LSE) for the merge.
// The pages gather each context chunk into a contiguous buffer first
// (cp_mha_gather_cache); here TMA boxes walk the block table directly, and
// the chunk loop is a grid dimension: every (query tile, chunk) is an
// independent work item, merged afterwards by the extend reduction.
//
// Work unit: (request, 128-row query tile, slot) x query head, slot 0 = new
// keys, slot c >= 1 = context chunk c - 1. Persistent CTAs (one per SM) walk
// the planner's cost-sorted unit list round-robin. Per CTA, 8 warps:
//   warps 0, 6 TMA producers: warp 0 the Q tile (double-buffered) and K
//            tiles of 128 keys, warp 6 the V tiles, each into a 2-stage ring
//            (block sizes below 8 use cp.async copies);
//   warp 1   tensor-memory owner; one thread issues S = Q K^T into one of
//            two TMEM S buffers (128 fp32 columns each), running ahead;
//   warp 7   one thread issues O += P V into the TMEM O accumulator
//            (head_dim fp32 columns) as soon as each P is written;
//   warps 2-5 softmax warpgroup, one thread per query row (= TMEM lane):
//            reads its S row, masks, keeps the running max and sum in
//            registers, writes P (bf16 pairs) into one of two TMEM P buffers
//            (the P . V product takes its A operand from TMEM), rescales its
//            O row in TMEM only when the max grew by more than 2^8
//            (otherwise the stale max is kept: P stays <= 2^8), and finally
//            reads O, divides by the sum and stores out (+ LSE).
// TMEM holds S0, S1, O, P0, P1 (512 columns). Q, S and P are
// double-buffered: while the softmax works on tile j the tensor core
// computes S_{j+1} and O += P_{j-1} V_{j-1}, and the next unit's Q loads
// during the current one. Every barrier that could complete twice before
// its waiter looks exists per buffer, so mbarrier phase parities never alias.
#include "common.cuh"
#include "params.cuh"
#include "plan.cuh"
#include "tcgen05.cuh"

namespace pka {

constexpr int kFaThreads = 256;
constexpr int BM = kFaBlockM;  // 128 query rows per unit
constexpr int BN = kFaBlockN;  // 128 keys per tile
static_assert(BM == 128 && BN == 128, "tile shape is fixed by the TMEM lane count");

template <int D>
struct FaCfg {
    static constexpr int kChunks = D / 64;                // 64-wide swizzle chunks per row
    static constexpr int kChunkBytes = 128 * 128;         // 128 rows x 128 B
    static constexpr int kQBytes = kChunks * kChunkBytes;
    static constexpr int kKVBytes = kChunks * kChunkBytes;  // one K or V tile
    static constexpr int kOffQ = 0;                        // two Q buffers
    static constexpr int kOffK = kOffQ + 2 * kQBytes;
    static constexpr int kOffV = kOffK + 2 * kKVBytes;
    static constexpr int kOffBar = kOffV + 2 * kKVBytes;
    static constexpr int kSmem = kOffBar + 256 + 1024;
    // TMEM columns: S0, S1 (fp32 128 each), O (fp32 D), P0, P1 (bf16x2, 64 each)
    static constexpr uint32_t kColS = 0, kColO = 256, kColP = 384, kTmemCols = 512;
};

struct FaUnit {
    int r, slot, h, g, q0, qlen, ctx, row0;
    int kb0, ntiles, c0, c1;  // first tile's key base, tiles, visible keys [c0, c1)
};

PKA_DEVICE FaUnit fa_unit(const FaParams& p, int u) {
    FaUnit U;
    const int4 it = p.items[u / p.Hq];
    U.h = u % p.Hq;
    U.g = U.h / p.G;
    U.r = it.x;
    U.slot = it.z;
    U.q0 = p.qsl[U.r];
    U.qlen = p.qsl[U.r + 1] - U.q0;
    U.ctx = p.seq_lens[U.r] - U.qlen;
    U.row0 = it.y * BM;
    if (U.slot == 0) {
        U.c0 = 0;
        U.c1 = min(U.qlen, U.row0 + BM);
        U.kb0 = 0;
    } else {
        U.c0 = (U.slot - 1) * p.chunk;
        U.c1 = min(U.ctx, U.c0 + p.chunk);
        U.kb0 = (U.c0 / BN) * BN;
    }
    U.ntiles = (U.c1 - U.kb0 + BN - 1) / BN;
    return U;
}

// Block id of lane `b`'s block in the context tile starting at key kb
// (lanes past the tile's valid blocks get 0); one parallel load per warp.
PKA_DEVICE int tile_block_id(const FaParams& p, const int32_t* bt, int kb, int c1, int lane) {
    const int nblk = BN / p.bs;
    const int pos = kb + lane * p.bs;
    if (lane >= nblk || pos >= c1) return 0;
    int blk = __ldg(bt + pos / p.bs);
    if (blk < 0 || blk >= p.num_blocks) {
        set_error(p.err, PKA_DEVERR_BLOCK_ID);
        blk = 0;
    }
    return blk;
}

template <int D>
__global__ void __launch_bounds__(kFaThreads, 1) fa_fwd_kernel(const __grid_constant__ FaMaps maps, const FaParams p) {
    using C = FaCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* q_full = bars + 0;    // [2] per Q buffer
    uint64_t* q_empty = bars + 2;   // [2]
    uint64_t* k_full = bars + 4;    // [2] per K stage
    uint64_t* k_empty = bars + 6;   // [2]
    uint64_t* v_full = bars + 8;    // [2] per V stage
    uint64_t* v_empty = bars + 10;  // [2]
    uint64_t* s_full = bars + 12;   // [2] per S buffer
    uint64_t* s_free = bars + 14;   // [2]
    uint64_t* p_full = bars + 16;   // [2] per P buffer
    uint64_t* pv_done = bars + 18;  // [2] per P buffer: the P . V that read it is done
    uint64_t* o_free = bars + 20;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_units = p.hdr->fa_num_items * p.Hq;
    if (num_units == 0) return;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 4);
            mbar_init(&p_full[i], 4);
            mbar_init(&pv_done[i], 1);
        }
        mbar_init(o_free, 4);
        fence_barrier_init();
        s_abort = 0;
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.knew);
        tma_prefetch_desc(&maps.vnew);
        tma_prefetch_desc(&maps.kc);
        tma_prefetch_desc(&maps.vc);
    }
    if (warp == 1) tmem_alloc(&s_tmem, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s_tmem;
    const uint32_t sm_base = smem_u32(smem);

    if (warp == 0 || warp == 6) {
        // ------------------------------------------------------------ producers
        // warp 0 loads Q and K tiles, warp 6 loads V tiles (so a V load that
        // waits for an older P . V never delays the next K). K/V lines stay
        // in L2 with normal priority: every context chunk is read by all the
        // query heads of its KV head and all query tiles of its request.
        const int which = warp == 0 ? 0 : 1;  // 0 = K (+ Q), 1 = V
        const uint64_t pol_kv = policy_evict_normal();
        const uint64_t pol_q = policy_evict_last();
        const bool ctx_tma = p.bs >= 8;
        uint32_t kv_it = 0, q_it = 0;
        uint32_t last_k[2] = {0, 0}, last_v[2] = {0, 0};  // phase + 1 of the last copy per stage (0 = none)
        FaUnit Un = blockIdx.x < num_units ? fa_unit(p, blockIdx.x) : FaUnit{};
        for (int u = blockIdx.x; u < num_units && !s_abort; u += gridDim.x, ++q_it) {
            const FaUnit U = Un;
            if (u + (int)gridDim.x < num_units) Un = fa_unit(p, u + gridDim.x);  // prefetch
            const int qb = q_it & 1;
            if (which == 0 && q_it >= 2 && !mbar_wait(&q_empty[qb], ((q_it >> 1) - 1) & 1, p.err)) {
                s_abort = 1;
                break;
            }
            if (which == 0 && lane == 0) {
                mbar_arrive_expect_tx(&q_full[qb], C::kQBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(smem + C::kOffQ + qb * C::kQBytes + c * C::kChunkBytes, &maps.q, &q_full[qb], c * 64,
                                U.h, U.q0 + U.row0, pol_q);
            }
            const int32_t* bt = p.block_table + (int64_t)U.r * p.max_blocks;
            const bool paged_tma = U.slot != 0 && ctx_tma;
            int blk_next = paged_tma ? tile_block_id(p, bt, U.kb0, U.c1, lane) : 0;
            bool ok = true;
            for (int t = 0; t < U.ntiles && ok; ++t, ++kv_it) {
                const int st = kv_it & 1;
                const uint32_t n = kv_it >> 1;
                const int kb = U.kb0 + t * BN;
                const int blk_mine = blk_next;  // block ids of this tile, one per lane
                if (paged_tma && t + 1 < U.ntiles) blk_next = tile_block_id(p, bt, kb + BN, U.c1, lane);
                {
                    uint64_t* full = which ? &v_full[st] : &k_full[st];
                    uint64_t* empty = which ? &v_empty[st] : &k_empty[st];
                    if (n > 0 && !mbar_wait(empty, (n - 1) & 1, p.err)) {
                        s_abort = 1;
                        ok = false;
                        continue;
                    }
                    uint8_t* dst = smem + (which ? C::kOffV : C::kOffK) + st * C::kKVBytes;
                    if (U.slot == 0) {
                        if (lane == 0) {
                            mbar_arrive_expect_tx(full, C::kKVBytes);
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_3d(dst + c * C::kChunkBytes, which ? &maps.vnew : &maps.knew, full, c * 64,
                                            U.g, U.q0 + kb, pol_kv);
                        }
                    } else if (ctx_tma) {
                        // one lane per block issues that block's boxes (in parallel)
                        const int bs = p.bs;
                        const int nvalid = min(BN / bs, (U.c1 - kb + bs - 1) / bs);
                        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(nvalid * C::kChunks * bs * 128));
                        __syncwarp();
                        if (lane < nvalid) {
                            const int row = (blk_mine * p.Hkv + U.g) * bs;
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_2d(dst + c * C::kChunkBytes + lane * bs * 128, which ? &maps.vc : &maps.kc,
                                            full, c * 64, row, pol_kv);
                        }
                    } else {
                        // small blocks: 16-byte copies, rows past the chunk end zero-filled
                        const uint32_t dbase = smem_u32(dst);
                        const __nv_bfloat16* src_base = which ? p.v_cache : p.k_cache;
                        for (int ci = lane; ci < BN * (D / 8); ci += 32) {
                            const int row = ci / (D / 8), c = ci % (D / 8);
                            const int pos = kb + row;
                            const bool valid = pos < U.c1;
                            int blk = valid ? __ldg(bt + pos / p.bs) : 0;
                            if (blk < 0 || blk >= p.num_blocks) {
                                set_error(p.err, PKA_DEVERR_BLOCK_ID);
                                blk = 0;
                            }
                            const int64_t grow = ((int64_t)blk * p.Hkv + U.g) * p.bs + (valid ? pos % p.bs : 0);
                            cp_async_16_zfill(dbase + (c >> 3) * C::kChunkBytes + sw128(row, c & 7),
                                              src_base + grow * D + c * 8, valid);
                        }
                        asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(full)) : "memory");
                        __syncwarp();
                        if (lane == 0) mbar_arrive(full);
                    }
                    if (which) last_v[st] = n + 1;
                    else last_k[st] = n + 1;
                }
            }
            if (!ok) break;
        }
        // no copy may outlive the CTA: wait (bounded) for the last one per stage
        for (int st = 0; st < 2; ++st) {
            if (last_k[st]) mbar_wait(&k_full[st], (last_k[st] - 1) & 1, p.err);
            if (last_v[st]) mbar_wait(&v_full[st], (last_v[st] - 1) & 1, p.err);
        }
        if (which == 0)
            for (uint32_t k = q_it > 2 ? q_it - 2 : 0; k < q_it; ++k) mbar_wait(&q_full[k & 1], (k >> 1) & 1, p.err);
    } else if (warp == 1 || warp == 7) {
        // ------------------------------------------------------------ MMA issuers
        // warp 1 streams S = Q K^T ahead of the softmax (gated only by a free S
        // buffer and the K tile); warp 7 issues O += P V as each P lands. Each
        // thread commits only its own MMAs.
        if (lane == 0 && warp == 1) {
            constexpr uint32_t idesc_qk = umma_idesc_bf16(128, 128, 0, 0);
            const uint32_t q_s = sm_base + C::kOffQ, k_s = sm_base + C::kOffK;
            uint32_t kv_it = 0, s_it = 0, q_it = 0;
            bool ok = true;
            FaUnit Un = blockIdx.x < num_units ? fa_unit(p, blockIdx.x) : FaUnit{};
            for (int u = blockIdx.x; u < num_units && ok && !s_abort; u += gridDim.x, ++q_it) {
                const FaUnit U = Un;
                if (u + (int)gridDim.x < num_units) Un = fa_unit(p, u + gridDim.x);
                const int qb = q_it & 1;
                if (!mbar_wait(&q_full[qb], (q_it >> 1) & 1, p.err)) {
                    ok = false;
                    break;
                }
                for (int t = 0; t < U.ntiles; ++t, ++kv_it) {
                    const int st = kv_it & 1;
                    const int b = s_it & 1;
                    if (!mbar_wait(&k_full[st], (kv_it >> 1) & 1, p.err)) { ok = false; break; }
                    if (s_it >= 2 && !mbar_wait(&s_free[b], ((s_it >> 1) - 1) & 1, p.err)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
                        umma_bf16(tbase + C::kColS + b * 128, umma_desc_sw128(q_s + qb * C::kQBytes + off, 16, 1024),
                                  umma_desc_sw128(k_s + st * C::kKVBytes + off, 16, 1024), idesc_qk,
                                  ks > 0 ? 1u : 0u);
                    }
                    umma_commit(&s_full[b]);
                    umma_commit(&k_empty[st]);
                    if (t == U.ntiles - 1) umma_commit(&q_empty[qb]);
                    ++s_it;
                }
            }
            if (!ok) s_abort = 1;
            if (s_it > 0) mbar_wait(&s_full[(s_it - 1) & 1], ((s_it - 1) >> 1) & 1, p.err);
        } else if (lane == 0 && warp == 7) {
            constexpr uint32_t idesc_pv = umma_idesc_bf16(128, D, 0, 1);
            const uint32_t v_s = sm_base + C::kOffV;
            uint32_t kv_it = 0, pv_it = 0, q_it = 0;
            bool ok = true;
            FaUnit Un = blockIdx.x < num_units ? fa_unit(p, blockIdx.x) : FaUnit{};
            for (int u = blockIdx.x; u < num_units && ok && !s_abort; u += gridDim.x, ++q_it) {
                const FaUnit U = Un;
                if (u + (int)gridDim.x < num_units) Un = fa_unit(p, u + gridDim.x);
                for (int t = 0; t < U.ntiles; ++t, ++kv_it) {
                    const int vs = kv_it & 1;
                    const int pb = pv_it & 1;
                    if (!mbar_wait(&p_full[pb], (pv_it >> 1) & 1, p.err)) { ok = false; break; }
                    if (!mbar_wait(&v_full[vs], (kv_it >> 1) & 1, p.err)) { ok = false; break; }
                    // the first product of a unit overwrites O: the previous unit's O must be read
                    if (t == 0 && q_it > 0 && !mbar_wait(o_free, (q_it - 1) & 1, p.err)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint64_t bdesc = umma_desc_sw128(v_s + vs * C::kKVBytes + kk * 2048, C::kChunkBytes, 1024);
                        umma_bf16_ts(tbase + C::kColO, tbase + C::kColP + pb * 64 + kk * 8, bdesc, idesc_pv,
                                     (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(&pv_done[pb]);
                    umma_commit(&v_empty[vs]);
                    ++pv_it;
                }
            }
            if (!ok) s_abort = 1;
            // let every issued MMA finish before the CTA can exit
            if (pv_it > 0) mbar_wait(&pv_done[(pv_it - 1) & 1], ((pv_it - 1) >> 1) & 1, p.err);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroup
        const int row = 32 * (warp & 3) + lane;  // TMEM lane = query row of the tile
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const int wg_tid = threadIdx.x - 64;
        const float sl2 = p.scale_log2;
        uint32_t s_it = 0, kv_it = 0;
        uint32_t p_it = 0;      // P buffers written (global)
        uint32_t pv_seen = 0;   // P . V completions waited for (global, in order)
        // wait until the P . V that used write number `k` (global) is done
        auto wait_pv = [&](uint32_t k) -> bool {
            while (pv_seen <= k) {
                if (!mbar_wait(&pv_done[pv_seen & 1], (pv_seen >> 1) & 1, p.err)) return false;
                ++pv_seen;
            }
            return true;
        };
        FaUnit Un = blockIdx.x < num_units ? fa_unit(p, blockIdx.x) : FaUnit{};
        for (int u = blockIdx.x; u < num_units && !s_abort; u += gridDim.x) {
            const FaUnit U = Un;
            if (u + (int)gridDim.x < num_units) Un = fa_unit(p, u + gridDim.x);
            const int qi = U.row0 + row;  // query index within the request's new tokens
            float m_used = -INFINITY, l = 0.f;
            bool ok = true;
            const uint32_t kv_base = kv_it;
            for (int t = 0; t < U.ntiles; ++t) {
                const int b = s_it & 1;
                if (!mbar_wait(&s_full[b], (s_it >> 1) & 1, p.err)) { ok = false; break; }
                tc_fence_after();
                float s[BN];
                {
                    uint32_t r0[32], r1[32], r2[32], r3[32];
                    const uint32_t ta = tbase + lane_off + C::kColS + b * 128;
                    tmem_ld32(ta, r0);
                    tmem_ld32(ta + 32, r1);
                    tmem_ld32(ta + 64, r2);
                    tmem_ld32(ta + 96, r3);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        s[i] = __uint_as_float(r0[i]);
                        s[32 + i] = __uint_as_float(r1[i]);
                        s[64 + i] = __uint_as_float(r2[i]);
                        s[96 + i] = __uint_as_float(r3[i]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[b]);
                ++s_it;
                // mask (raw scores), row max
                const int kb = U.kb0 + t * BN;
                const bool edge = (U.slot == 0) ? (kb + BN - 1 > U.row0 || kb + BN > U.c1)
                                                : (kb < U.c0 || kb + BN > U.c1);
                if (edge) {
                    const int lo = U.c0 - kb;  // visible columns: [lo, hi)
                    const int hi = ((U.slot == 0) ? min(qi + 1, U.c1) : U.c1) - kb;
#pragma unroll
                    for (int i = 0; i < BN; ++i) s[i] = (i >= lo && i < hi) ? s[i] : -INFINITY;
                }
                // row max as a tree over 8 independent chains
                float mxv[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mxv[k] = s[k];
#pragma unroll
                for (int i = 8; i < BN; i += 8)
#pragma unroll
                    for (int k = 0; k < 8; ++k) mxv[k] = fmaxf(mxv[k], s[i + k]);
                const float mx = fmaxf(fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])),
                                       fmaxf(fmaxf(mxv[4], mxv[5]), fmaxf(mxv[6], mxv[7])));
                const float m_new = fmaxf(m_used, mx * sl2);
                bool rescale = false;
                float alpha = 1.f;
                if (t == 0) {
                    m_used = m_new;
                } else if (m_new > m_used + 8.f) {
                    alpha = fast_exp2(m_used - m_new);
                    rescale = true;
                    l *= alpha;
                    m_used = m_new;
                }
                // P = exp2(scale * s - m_used), kept packed in registers
                uint32_t pk[BN / 2];
                float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < BN; i += 2) {
                    const float e0 = fast_exp2(fmaf(s[i], sl2, -m_used));
                    const float e1 = fast_exp2(fmaf(s[i + 1], sl2, -m_used));
                    ls[(i >> 1) & 7] += e0 + e1;
                    pk[i / 2] = pack_bf16(e0, e1);
                }
                l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                // O may be rescaled only once the previous P . V is done
                if (rescale) {
                    if (!wait_pv(p_it - 1)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tbase + lane_off + C::kColO + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(tbase + lane_off + C::kColO + c * 32, r);
                    }
                    tmem_wait_st();
                }
                // last tile of a context chunk: value rows past the chunk end may
                // hold anything (other positions, NaN-poisoned slots): zero them
                if (U.slot != 0 && kb + BN > U.c1) {
                    const uint32_t vi = kv_base + t;
                    if (!mbar_wait(&v_full[vi & 1], (vi >> 1) & 1, p.err)) { ok = false; break; }
                    const int valid = U.c1 - kb;
                    uint8_t* vt = smem + C::kOffV + (vi & 1) * C::kKVBytes;
                    for (int ci = wg_tid; ci < (BN - valid) * (D / 8); ci += 128) {
                        const int vr = valid + ci / (D / 8), c = ci % (D / 8);
                        *reinterpret_cast<uint4*>(vt + (c >> 3) * C::kChunkBytes + sw128(vr, c & 7)) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                // P buffer p_it & 1 (TMEM) was last read by P . V number p_it - 2
                if (p_it >= 2 && !wait_pv(p_it - 2)) { ok = false; break; }
                {
                    const uint32_t pa = tbase + lane_off + C::kColP + (p_it & 1) * 64;
                    uint32_t h0[32], h1[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        h0[i] = pk[i];
                        h1[i] = pk[32 + i];
                    }
                    tmem_st32(pa, h0);
                    tmem_st32(pa + 32, h1);
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[p_it & 1]);
                ++p_it;
            }
            kv_it = kv_base + U.ntiles;
            if (!ok) {
                s_abort = 1;
                break;
            }
            // ---- epilogue: O row / l once the unit's last P . V is done
            if (!wait_pv(p_it - 1)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            float o[D];
            {
                uint32_t r[D / 32][32];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) tmem_ld32(tbase + lane_off + C::kColO + c * 32, r[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < D / 32; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[c * 32 + i] = __uint_as_float(r[c][i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            if (qi < U.qlen) {
                const float inv = 1.f / l;
                const float lse_nat = (m_used + __log2f(l)) * 0.69314718055994531f;
                if (U.slot == 0 && U.ctx == 0) {
                    __nv_bfloat16* dst = p.out + ((int64_t)(U.q0 + qi) * p.Hq + U.h) * D;
#pragma unroll
                    for (int c = 0; c < D / 8; ++c) {
                        uint4 v;
                        v.x = pack_bf16(o[c * 8 + 0] * inv, o[c * 8 + 1] * inv);
                        v.y = pack_bf16(o[c * 8 + 2] * inv, o[c * 8 + 3] * inv);
                        v.z = pack_bf16(o[c * 8 + 4] * inv, o[c * 8 + 5] * inv);
                        v.w = pack_bf16(o[c * 8 + 6] * inv, o[c * 8 + 7] * inv);
                        *reinterpret_cast<uint4*>(dst + c * 8) = v;
                    }
                    if (p.lse) p.lse[(int64_t)(U.q0 + qi) * p.Hq + U.h] = lse_nat;
                } else {
                    const int64_t prow =
                        ((int64_t)p.ext_base[U.r - p.num_decodes] + (int64_t)U.slot * U.qlen + qi) * p.Hq + U.h;
                    float* dst = p.ext_o + prow * D;
#pragma unroll
                    for (int c = 0; c < D / 4; ++c)
                        *reinterpret_cast<float4*>(dst + c * 4) =
                            make_float4(o[c * 4] * inv, o[c * 4 + 1] * inv, o[c * 4 + 2] * inv, o[c * 4 + 3] * inv);
                    p.ext_lse[prow] = lse_nat;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, C::kTmemCols);
    }
}

template <int D>
static cudaError_t launch_fa_d(const FaMaps& maps, const FaParams& p, int num_sms, cudaStream_t stream) {
    auto kern = fa_fwd_kernel<D>;
    const int smem = FaCfg<D>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<num_sms, kFaThreads, smem, stream>>>(maps, p);
    return cudaGetLastError();
}

cudaError_t launch_fa_fwd(const FaMaps& maps, const FaParams& p, int head_dim, int num_sms, cudaStream_t stream) {
    if (head_dim == 128) return launch_fa_d<128>(maps, p, num_sms, stream);
    if (head_dim == 64) return launch_fa_d<64>(maps, p, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pka
