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
// the chunk loop is a grid dimension: every (query tiles, chunk) is an
// independent work item, merged afterwards by the extend reduction.
//
// Work unit: (request, two adjacent 128-row query tiles, slot) x query head,
// slot 0 = new keys, slot c >= 1 = context chunk c - 1. Persistent CTAs (one
// per SM) walk the planner's cost-sorted unit list round-robin. Per CTA, 12
// warps:
//   warp 0   TMA producer of the K tiles of 128 keys (2-stage ring);
//   warp 2   the same for the V tiles, and the unit's two Q tiles (block
//            sizes below 8 use cp.async copies for K and V);
//   warp 1   tensor-memory owner; one thread issues S_k = Q_k K^T for both
//            query tiles k of every K tile;
//   warp 3   one thread issues O_k += P_k V (A operand P_k read from TMEM),
//            keys 0..63 first when the softmax signals that half early;
//   warps 4-7, 8-11: softmax warpgroup k owns query tile k, one thread per
//            query row (= TMEM lane), with its own S_k, running max and sum
//            and O_k. It reads its S row in 64-column halves: once when the
//            tile needs no mask and its scores stay within the rescale margin
//            of the running max, else twice (row max, then exponentials; the
//            row never sits in registers whole); writes P as bf16 pairs over
//            the S_k columns it has already consumed, rescales O_k only
//            when its max grew by more than 2^8 (otherwise the stale max is
//            kept: P stays <= 2^8; warp-uniform, tcgen05.ld/st being
//            warp-collective), and ends the unit on its own: O_k / l to out
//            (+ LSE) or to the extend partials.
// Both query tiles consume every K and V tile once from shared memory, and
// the two warpgroups' exponentials overlap each other's waits. TMEM holds S0,
// S1 (128 fp32 columns each) and O0, O1 (head_dim fp32 columns each): 512
// columns. The S_k = Q_k K^T that refills S_k waits for the P_k . V that read
// P_k, so a warpgroup that sees its S tile may also touch O_k freely. Every
// barrier belongs to one buffer or one warpgroup and cannot complete twice
// before its waiter looks, so mbarrier phase parities never alias.
#include <type_traits>

#include "common.cuh"
#include "params.cuh"
#include "plan.cuh"
#include "tcgen05.cuh"

namespace pka {

constexpr int kFaThreads = 384;
constexpr int kFaRegsLaunch = 168, kFaRegsIssue = 80, kFaRegsSoftmax = 208;
static_assert(128 * kFaRegsIssue + 256 * kFaRegsSoftmax <= kFaThreads * kFaRegsLaunch, "register split");
constexpr int BM = kFaBlockM;  // 128 query rows per query tile
constexpr int BN = kFaBlockN;  // 128 keys per tile
static_assert(BM == 128 && BN == 128 && kFaItemTiles == 2, "tile shape is fixed by the TMEM lane count");

// D: q/k head dim; DV: value head dim (192 / 128 for the pages' non-absorbed
// MLA prefill, where K carries the 64 rope dims V does not).
template <int D, int DV>
struct FaCfg {
    static constexpr int kChunks = D / 64;                 // 64-wide swizzle chunks per q/k row
    static constexpr int kVChunks = DV / 64;               // ... per v row
    static constexpr int kChunkBytes = 128 * 128;          // 128 rows x 128 B
    static constexpr int kQBytes = kChunks * kChunkBytes;  // one query tile
    static constexpr int kKBytes = kChunks * kChunkBytes;  // one K tile
    static constexpr int kVBytes = kVChunks * kChunkBytes;  // one V tile
    // V ring depth: two stages, or one where two would not fit next to the
    // two query tiles and the two K stages (D = 192: 96 + 96 + 32 KB)
    static constexpr int kVStages = (2 * kQBytes + 2 * kKBytes + 2 * kVBytes + 1280 <= 232448) ? 2 : 1;
    static constexpr int kOffQ = 0;                         // the unit's two query tiles
    static constexpr int kOffK = kOffQ + 2 * kQBytes;
    static constexpr int kOffV = kOffK + 2 * kKBytes;
    static constexpr int kOffBar = kOffV + kVStages * kVBytes;
    static constexpr int kSmem = kOffBar + 256 + 1024;
    static_assert(kSmem <= 232448, "shared memory");
    // TMEM columns: S0, S1 (fp32 128 each; P_k overwrites the first 64 columns
    // of S_k as bf16 pairs), O0, O1 (fp32 DV each)
    static constexpr uint32_t kColS = 0, kColO = 256, kTmemCols = 512;
    static_assert(kColO + 2 * DV <= kTmemCols, "tensor memory");
};

struct FaUnit {
    int r, slot, h, g, q0, qlen, ctx, row0;  // row0: first row of query tile 0
    int kb0, c0, c1, nkv;                     // first tile's key base, visible keys [c0, c1), key tiles
    int c1k[2], ntk[2];                       // per query tile: end of its visible keys, its key tiles (0: no rows)
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
    U.row0 = it.y * kFaItemRows;
    if (U.slot == 0) {
        U.c0 = 0;
        U.kb0 = 0;
        for (int k = 0; k < 2; ++k) {
            const int rk = U.row0 + k * BM;
            U.c1k[k] = rk < U.qlen ? min(U.qlen, rk + BM) : 0;
        }
        U.c1 = max(U.c1k[0], U.c1k[1]);
    } else {
        U.c0 = (U.slot - 1) * p.chunk;
        U.c1 = min(U.ctx, U.c0 + p.chunk);
        U.kb0 = (U.c0 / BN) * BN;
        for (int k = 0; k < 2; ++k) U.c1k[k] = U.row0 + k * BM < U.qlen ? U.c1 : 0;
    }
    for (int k = 0; k < 2; ++k) U.ntk[k] = U.c1k[k] > 0 ? (U.c1k[k] - U.kb0 + BN - 1) / BN : 0;
    U.nkv = max(U.ntk[0], U.ntk[1]);
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

// kCtxScaled: the context chunks carry their own score scale and output
// factor (a gathered 8-bit cache); otherwise every slot uses scale_log2.
template <int D, int DV, bool kCtxScaled>
__global__ void __launch_bounds__(kFaThreads, 1) fa_fwd_kernel(const __grid_constant__ FaMaps maps, const FaParams p) {
    grid_dep_wait();
    using C = FaCfg<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* q_full = bars + 0;     // the unit's query tiles landed
    uint64_t* q_empty = bars + 1;    // the unit's last S product is done
    uint64_t* k_full = bars + 2;     // [2] per K stage
    uint64_t* k_empty = bars + 4;    // [2]
    uint64_t* v_full = bars + 6;     // [2] per V stage
    uint64_t* v_empty = bars + 8;    // [2]
    uint64_t* s_full = bars + 10;    // [2] per softmax warpgroup: its S tile is in TMEM
    uint64_t* p_full = bars + 12;    // [2] its P is in TMEM (4 warp arrivals)
    uint64_t* pv_done = bars + 14;   // [2] the P . V that read its P is done
    uint64_t* o_free = bars + 16;    // [2] its epilogue has read O_k (4 warp arrivals)
    uint64_t* p_half = bars + 18;    // [2] the first half of its P (keys 0..63) is in TMEM (4 warp arrivals)
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    // Key tiles (global count) after which the S issuer has issued query tile
    // 0's next S: the P . V issuer lets query tile 1's product of tile g go
    // only once this exceeds g, so the tensor pipe runs P_0 V, S_0 (next),
    // P_1 V, S_1 (next) and warpgroup 0 never queues behind warpgroup 1.
    __shared__ volatile int s_qk0_next;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_units = p.hdr->fa_num_items * p.Hq;
    if (num_units == 0) return;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&p_half[i], 4);
            mbar_init(&pv_done[i], 1);
            mbar_init(&o_free[i], 4);
        }
        fence_barrier_init();
        s_abort = 0;
        s_qk0_next = 0;
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
    // Registers by role (the launch gives every thread kFaRegsLaunch): the copy
    // and MMA-issuing warpgroup drops to kFaRegsIssue, the two softmax
    // warpgroups take what it frees (128 * 80 + 256 * 208 <= 384 * 168).

    if (warp < 4) {
        setmaxnreg_dec<kFaRegsIssue>();
        if (warp == 0 || warp == 2) {
            // ------------------------------------------------------------ producers
            // warp 0 loads K tiles, warp 2 the query tiles and V tiles (so a V load
            // that waits for an older P . V never delays the next K). K/V lines
            // stay in L2 with normal priority: every context chunk is read by all
            // the query heads of its KV head and all query tiles of its request.
            const int which = warp == 0 ? 0 : 1;  // 0 = K, 1 = V (+ Q)
            const uint64_t pol_kv = policy_evict_normal();
            const uint64_t pol_q = policy_evict_last();
            const bool ctx_tma = p.bs >= 8;
            uint32_t kv_it = 0, q_it = 0;
            uint32_t last[2] = {0, 0};  // phase + 1 of the last copy per stage (0 = none)
            FaUnit Un = blockIdx.x < num_units ? fa_unit(p, blockIdx.x) : FaUnit{};
            for (int u = blockIdx.x; u < num_units && !warp_flag(s_abort); u += gridDim.x, ++q_it) {
                const FaUnit U = Un;
                if (u + (int)gridDim.x < num_units) Un = fa_unit(p, u + gridDim.x);  // prefetch
                if (which == 1) {
                    // the previous unit's S products are done with the query tiles
                    if (q_it > 0 && !mbar_wait_warp(q_empty, (q_it - 1) & 1, p.err)) {
                        s_abort = 1;
                        break;
                    }
                    if (lane == 0) {
                        const int nq = U.ntk[1] > 0 ? 2 : 1;
                        mbar_arrive_expect_tx(q_full, (uint32_t)(nq * C::kQBytes));
                        for (int k = 0; k < nq; ++k)
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_3d(smem + C::kOffQ + k * C::kQBytes + c * C::kChunkBytes, &maps.q, q_full,
                                            c * 64, U.h, U.q0 + U.row0 + k * BM, pol_q);
                    }
                }
                const int32_t* bt = U.slot != 0 ? p.block_table + (int64_t)(U.r - p.bt_row0) * p.max_blocks : p.block_table;
                const bool paged_tma = U.slot != 0 && ctx_tma;
                int blk_next = paged_tma ? tile_block_id(p, bt, U.kb0, U.c1, lane) : 0;
                bool ok = true;
                const int nstage = which ? C::kVStages : 2;
                const int nchunk = which ? C::kVChunks : C::kChunks;
                const int width = which ? DV : D;  // elements per row
                for (int t = 0; t < U.nkv && ok; ++t, ++kv_it) {
                    const int st = (int)(kv_it % nstage);
                    const uint32_t n = kv_it / nstage;
                    const int kb = U.kb0 + t * BN;
                    const int blk_mine = blk_next;  // block ids of this tile, one per lane
                    if (paged_tma && t + 1 < U.nkv) blk_next = tile_block_id(p, bt, kb + BN, U.c1, lane);
                    uint64_t* full = which ? &v_full[st] : &k_full[st];
                    uint64_t* empty = which ? &v_empty[st] : &k_empty[st];
                    if (n > 0 && !mbar_wait_warp(empty, (n - 1) & 1, p.err)) {
                        s_abort = 1;
                        ok = false;
                        continue;
                    }
                    uint8_t* dst = smem + (which ? C::kOffV + st * C::kVBytes : C::kOffK + st * C::kKBytes);
                    if (U.slot == 0) {
                        if (lane == 0) {
                            mbar_arrive_expect_tx(full, (uint32_t)(nchunk * C::kChunkBytes));
                            for (int c = 0; c < nchunk; ++c)
                                tma_load_3d(dst + c * C::kChunkBytes, which ? &maps.vnew : &maps.knew, full, c * 64, U.g,
                                            U.q0 + kb, pol_kv);
                        }
                    } else if (ctx_tma) {
                        // one lane per block issues that block's boxes (in parallel)
                        const int bs = p.bs;
                        const int nvalid = min(BN / bs, (U.c1 - kb + bs - 1) / bs);
                        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(nvalid * nchunk * bs * 128));
                        __syncwarp();
                        if (lane < nvalid) {
                            const int row = (blk_mine * p.Hkv + U.g) * bs;
                            for (int c = 0; c < nchunk; ++c)
                                tma_load_2d(dst + c * C::kChunkBytes + lane * bs * 128, which ? &maps.vc : &maps.kc, full,
                                            c * 64, row, pol_kv);
                        }
                    } else {
                        // small blocks: 16-byte copies, rows past the chunk end zero-filled
                        const uint32_t dbase = smem_u32(dst);
                        const __nv_bfloat16* src_base = which ? p.v_cache : p.k_cache;
                        for (int ci = lane; ci < BN * (width / 8); ci += 32) {
                            const int row = ci / (width / 8), c = ci % (width / 8);
                            const int pos = kb + row;
                            const bool valid = pos < U.c1;
                            int blk = valid ? __ldg(bt + pos / p.bs) : 0;
                            if (blk < 0 || blk >= p.num_blocks) {
                                set_error(p.err, PKA_DEVERR_BLOCK_ID);
                                blk = 0;
                            }
                            const int64_t grow = ((int64_t)blk * p.Hkv + U.g) * p.bs + (valid ? pos % p.bs : 0);
                            cp_async_16_zfill(dbase + (c >> 3) * C::kChunkBytes + sw128(row, c & 7),
                                              src_base + grow * width + c * 8, valid);
                        }
                        asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(full)) : "memory");
                        __syncwarp();
                        if (lane == 0) mbar_arrive(full);
                    }
                    last[st] = n + 1;
                }
                if (!ok) break;
            }
            // no copy may outlive the CTA: wait (bounded) for the last one per stage
            for (int st = 0; st < (which ? C::kVStages : 2); ++st)
                if (last[st]) mbar_wait_warp(which ? &v_full[st] : &k_full[st], (last[st] - 1) & 1, p.err);
            if (which == 1 && q_it > 0) mbar_wait_warp(q_full, (q_it - 1) & 1, p.err);
        } else {  // warps 1 and 3
            // ------------------------------------------------------------ MMA issuers
            // warp 1 issues S_k = Q_k K^T for both query tiles of every K tile, each
            // once the previous P_k . V (which read P_k out of S_k's columns) is
            // done; warp 3 issues O_k += P_k V as each P_k lands. Each thread
            // commits only its own MMAs.
            if (lane == 0 && warp == 1) {
                constexpr uint32_t idesc_qk = umma_idesc_bf16(128, 128, 0, 0);
                const uint32_t q_s = sm_base + C::kOffQ, k_s = sm_base + C::kOffK;
                uint32_t kv_it = 0, q_it = 0;
                uint32_t nq[2] = {0, 0};  // products issued into S_k
                bool ok = true;
                FaUnit Un = blockIdx.x < num_units ? fa_unit(p, blockIdx.x) : FaUnit{};
                for (int u = blockIdx.x; u < num_units && ok && !s_abort; u += gridDim.x, ++q_it) {
                    const FaUnit U = Un;
                    if (u + (int)gridDim.x < num_units) Un = fa_unit(p, u + gridDim.x);
                    if (!mbar_wait(q_full, q_it & 1, p.err)) {
                        ok = false;
                        break;
                    }
                    for (int t = 0; t < U.nkv; ++t, ++kv_it) {
                        const int st = kv_it & 1;
                        if (!mbar_wait(&k_full[st], (kv_it >> 1) & 1, p.err)) { ok = false; break; }
                        // query tile 0 has no S of this tile: tile 1's product of the
                        // previous tile may go now (its next S below waits for it)
                        if (t > 0 && t >= U.ntk[0]) s_qk0_next = (int)kv_it;
                        for (int k = 0; k < 2; ++k) {
                            if (t >= U.ntk[k]) continue;
                            if (nq[k] > 0 && !mbar_wait(&pv_done[k], (nq[k] - 1) & 1, p.err)) { ok = false; break; }
                            tc_fence_after();
    #pragma unroll
                            for (int ks = 0; ks < D / 16; ++ks) {
                                const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
                                umma_bf16(tbase + C::kColS + k * 128,
                                          umma_desc_sw128(q_s + k * C::kQBytes + off, 16, 1024),
                                          umma_desc_sw128(k_s + st * C::kKBytes + off, 16, 1024), idesc_qk,
                                          ks > 0 ? 1u : 0u);
                            }
                            umma_commit(&s_full[k]);
                            ++nq[k];
                            // query tile 0's S of this tile is issued: query tile 1's
                            // product of the previous tile may go
                            if (k == 0 && t > 0) s_qk0_next = (int)kv_it;
                        }
                        if (!ok) break;
                        umma_commit(&k_empty[st]);
                        if (t == U.nkv - 1) umma_commit(q_empty);
                    }
                    if (ok) s_qk0_next = (int)kv_it;  // the unit's last tile: nothing of query tile 0 follows
                }
                if (!ok) s_abort = 1;
                for (int k = 0; k < 2; ++k)
                    if (nq[k] > 0) mbar_wait(&s_full[k], (nq[k] - 1) & 1, p.err);
            } else if (lane == 0 && warp == 3) {
                constexpr uint32_t idesc_pv = umma_idesc_bf16(128, DV, 0, 1);
                const uint32_t v_s = sm_base + C::kOffV;
                uint32_t kv_it = 0;
                uint32_t np[2] = {0, 0};  // products issued from P_k
                uint32_t uo[2] = {0, 0};  // earlier units in which warpgroup k had rows (one epilogue each)
                bool ok = true;
                FaUnit Un = blockIdx.x < num_units ? fa_unit(p, blockIdx.x) : FaUnit{};
                for (int u = blockIdx.x; u < num_units && ok && !s_abort; u += gridDim.x) {
                    const FaUnit U = Un;
                    if (u + (int)gridDim.x < num_units) Un = fa_unit(p, u + gridDim.x);
                    for (int t = 0; t < U.nkv; ++t, ++kv_it) {
                        const int vs = (int)(kv_it % C::kVStages);
                        if (!mbar_wait(&v_full[vs], (kv_it / C::kVStages) & 1, p.err)) { ok = false; break; }
                        for (int k = 0; k < 2; ++k) {
                            if (t >= U.ntk[k]) continue;
                            if (k == 1 && !wait_counter(s_qk0_next, (int)kv_it + 1, p.err)) { ok = false; break; }
                            // keys 0..63 of P may be stored before the rest (the softmax's
                            // one-pass tiles signal them early): their half of the product
                            // goes first
                            for (int hh = 0; hh < 2 && ok; ++hh) {
                                if (!mbar_wait(hh ? &p_full[k] : &p_half[k], np[k] & 1, p.err)) { ok = false; break; }
                                // a unit's first product overwrites O_k: its previous epilogue must have read it
                                if (hh == 0 && t == 0 && uo[k] > 0 && !mbar_wait(&o_free[k], (uo[k] - 1) & 1, p.err)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
    #pragma unroll
                                for (int kq = 0; kq < BN / 32; ++kq) {
                                    const int kk = hh * (BN / 32) + kq;
                                    const uint64_t bdesc =
                                        umma_desc_sw128(v_s + vs * C::kVBytes + kk * 2048, C::kChunkBytes, 1024);
                                    umma_bf16_ts(tbase + C::kColO + k * DV, tbase + C::kColS + k * 128 + kk * 8, bdesc,
                                                 idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
                                }
                            }
                            if (!ok) break;
                            umma_commit(&pv_done[k]);
                            ++np[k];
                        }
                        if (!ok) break;
                        umma_commit(&v_empty[vs]);
                    }
                    for (int k = 0; k < 2; ++k)
                        if (U.ntk[k] > 0) ++uo[k];
                }
                if (!ok) s_abort = 1;
                // let every issued MMA finish before the CTA can exit
                for (int k = 0; k < 2; ++k)
                    if (np[k] > 0) mbar_wait(&pv_done[k], (np[k] - 1) & 1, p.err);
            }
        }
    } else {
        setmaxnreg_inc<kFaRegsSoftmax>();
        // ------------------------------------------------------------ softmax warpgroups
        const int k = warp >= 8 ? 1 : 0;        // this warpgroup's query tile
        const int row = 32 * (warp & 3) + lane;  // TMEM lane = query row of the tile
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const int wg_tid = threadIdx.x - 128 * (k + 1);
        const uint32_t tS = tbase + lane_off + C::kColS + k * 128;
        const uint32_t tO = tbase + lane_off + C::kColO + k * DV;
        uint32_t n_s = 0;  // S tiles of this warpgroup (all units)
        uint32_t kv_it = 0;
        for (int u = blockIdx.x; u < num_units && !warp_flag(s_abort); u += gridDim.x) {
            const FaUnit U = fa_unit(p, u);  // the softmax waits for S anyway: no prefetch
            const uint32_t kv_base = kv_it;
            kv_it += U.nkv;
            const int ntk = k ? U.ntk[1] : U.ntk[0];
            if (ntk == 0) continue;  // no rows of this unit in this warpgroup's query tile
            const int row0 = U.row0 + k * BM;
            const int qi = row0 + row;  // query index within the request's new tokens
            const int c1 = k ? U.c1k[1] : U.c1k[0];
            const float sl2 = (kCtxScaled && U.slot != 0) ? p.ctx_scale_log2 : p.scale_log2;
            float m_used = -INFINITY, l = 0.f;
            bool ok = true;
            for (int t = 0; t < ntk; ++t) {
                if (!mbar_wait_warp(&s_full[k], n_s & 1, p.err)) { ok = false; break; }
                tc_fence_after();
                const int kb = U.kb0 + t * BN;
                const bool edge = (U.slot == 0) ? (kb + BN - 1 > row0 || kb + BN > c1) : (kb < U.c0 || kb + BN > c1);
                const int lo = U.c0 - kb;  // visible columns: [lo, hi)
                const int hi = ((U.slot == 0) ? min(qi + 1, c1) : c1) - kb;
                // General body, two passes over the row of S_k (held in registers).
                // Pass 1: row max of the raw scores (8 independent chains). Pass 2:
                // P = exp2(scale * s - m_used) as bf16 pairs, written over S_k's
                // already-read columns (keys 64h.. land in columns 32h..). Specialised on whether the
                // tile needs a mask at all (a per-element mask costs ALU issue
                // slots on every tile otherwise).
                float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                bool rescale = false;
                float alpha = 1.f;
                // exponentials of 64 scores (one TMEM round trip) into bf16 pairs
                auto exp_half = [&](const uint32_t (&r)[64], uint32_t (&pk)[32], float m_off, auto masked_c, int h) {
                    constexpr bool kMasked = decltype(masked_c)::value;
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        float v0 = __uint_as_float(r[i]);
                        float v1 = __uint_as_float(r[i + 1]);
                        if (kMasked) {
                            if ((unsigned)(64 * h + i - lo) >= (unsigned)(hi - lo)) v0 = -INFINITY;
                            if ((unsigned)(64 * h + i + 1 - lo) >= (unsigned)(hi - lo)) v1 = -INFINITY;
                        }
                        float x0, x1;
                        fma2_bcast(x0, x1, v0, v1, sl2, -m_off);
                        const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
                        const int j = (i >> 1) & 3;
                        add2(ls[2 * j], ls[2 * j + 1], e0, e1);
                        pk[i / 2] = pack_bf16(e0, e1);
                    }
                };
                auto max_half = [&](const uint32_t (&r)[64], float (&mxv)[8], auto masked_c, int h) {
                    constexpr bool kMasked = decltype(masked_c)::value;
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        float v0 = __uint_as_float(r[i]);
                        float v1 = __uint_as_float(r[i + 1]);
                        if (kMasked) {
                            if ((unsigned)(64 * h + i - lo) >= (unsigned)(hi - lo)) v0 = -INFINITY;
                            if ((unsigned)(64 * h + i + 1 - lo) >= (unsigned)(hi - lo)) v1 = -INFINITY;
                        }
                        mxv[(i >> 1) & 7] = fmax3f(mxv[(i >> 1) & 7], v0, v1);
                    }
                };
                auto reduce8 = [](const float (&mxv)[8]) {
                    return fmaxf(fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])),
                                 fmaxf(fmaxf(mxv[4], mxv[5]), fmaxf(mxv[6], mxv[7])));
                };
                auto tile_body = [&](auto masked_c) {
                    // the whole row of S_k in one TMEM round trip, kept in registers
                    // for both passes
                    uint32_t r0[64], r1[64];
                    tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(r0));
                    tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(r0 + 32));
                    tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(r1));
                    tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(r1 + 32));
                    tmem_wait_ld();
                    float mxv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) mxv[j] = -INFINITY;
                    max_half(r0, mxv, masked_c, 0);
                    max_half(r1, mxv, masked_c, 1);
                    const float m_new = fmaxf(m_used, reduce8(mxv) * sl2);
                    if (t == 0) {
                        m_used = m_new;
                    } else if (m_new > m_used + 8.f) {
                        alpha = fast_exp2(m_used - m_new);
                        rescale = true;
                        l *= alpha;
                        m_used = m_new;
                    }
                    const float m_off = m_used == -INFINITY ? 0.f : m_used;
                    uint32_t pk[32];
                    // keys 64h.. land in P columns 32h.. (S columns already read)
                    exp_half(r0, pk, m_off, masked_c, 0);
                    tmem_st32(tS, *reinterpret_cast<const uint32_t(*)[32]>(pk));
                    exp_half(r1, pk, m_off, masked_c, 1);
                    tmem_st32(tS + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk));
                };
                // Common case, one pass: an unmasked tile after the row's first,
                // whose scores stay within the lazy-rescale margin of m_used, gets
                // its exponentials straight after the row max. When a row of the
                // warp needs more, nothing has been written yet and the general
                // body runs from the start (the choice is warp-uniform because
                // tcgen05.ld/st are warp-collective).
                auto tile_fast = [&]() -> bool {
                    // both halves of S_k come in one TMEM round trip (the softmax
                    // warpgroups have the registers for it)
                    uint32_t r0[64], r1[64];
                    tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(r0));
                    tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(r0 + 32));
                    tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(r1));
                    tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(r1 + 32));
                    tmem_wait_ld();
                    float mxv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) mxv[j] = -INFINITY;
                    max_half(r0, mxv, std::false_type{}, 0);
                    max_half(r1, mxv, std::false_type{}, 1);
                    if (__any_sync(0xffffffffu, reduce8(mxv) * sl2 > m_used + 8.f)) return false;
                    uint32_t pk[32];
                    exp_half(r0, pk, m_used, std::false_type{}, 0);
                    tmem_st32(tS, pk);  // keys 0..63 -> P columns 0..31 (S columns 0..127 were read)
                    // their half of P . V may start while the rest is computed (no
                    // rescale on this path, and no value rows to zero: both need a mask)
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_half[k]);
                    exp_half(r1, pk, m_used, std::false_type{}, 1);
                    tmem_st32(tS + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk));
                    return true;
                };
                bool done = false;
                if (!edge && t > 0) {
                    done = tile_fast();
                    if (!done) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) ls[j] = 0.f;
                    }
                }
                if (!done) {
                    if (edge) tile_body(std::true_type{});
                    else tile_body(std::false_type{});
                }
                l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                // O_k's previous product finished before this S tile was computed.
                // tcgen05.ld/st are warp-collective (.sync.aligned): the whole warp
                // takes this branch if any of its rows needs the rescale (alpha
                // stays 1 for the others)
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int c = 0; c < DV / 16; ++c) {
                        uint32_t r[16];
                        tmem_ld16(tO + c * 16, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st16(tO + c * 16, r);
                    }
                }
                tmem_wait_st();
                // last tile of a context chunk: value rows past the chunk end may
                // hold anything (other positions, NaN-poisoned slots): zero them.
                // Warpgroup 0 does it (it reads every tile of a context chunk);
                // warpgroup 1's product of the same tile is issued after 0's.
                if (k == 0 && U.slot != 0 && kb + BN > U.c1) {
                    const uint32_t vi = kv_base + t;
                    if (!mbar_wait_warp(&v_full[vi % C::kVStages], (vi / C::kVStages) & 1, p.err)) { ok = false; break; }
                    const int valid = U.c1 - kb;
                    uint8_t* vt = smem + C::kOffV + (vi % C::kVStages) * C::kVBytes;
                    for (int ci = wg_tid; ci < (BN - valid) * (DV / 8); ci += 128) {
                        const int vr = valid + ci / (DV / 8), c = ci % (DV / 8);
                        *reinterpret_cast<uint4*>(vt + (c >> 3) * C::kChunkBytes + sw128(vr, c & 7)) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();  // the tensor core reads these rows through the async proxy
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (!done) mbar_arrive(&p_half[k]);
                    mbar_arrive(&p_full[k]);
                }
                ++n_s;
            }
            if (!ok) {
                s_abort = 1;
                break;
            }
            // ---- epilogue: O_k row / l once this warpgroup's last P . V is done
            if (!mbar_wait_warp(&pv_done[k], (n_s - 1) & 1, p.err)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const bool write = qi < U.qlen;
            const bool final_out = U.slot == 0 && U.ctx == 0;
            const int64_t orow = final_out ? ((int64_t)(U.q0 + qi) * p.Hq + U.h)
                                           : (((int64_t)p.ext_base[U.r - p.num_decodes] + (int64_t)U.slot * U.qlen + qi) *
                                                  p.Hq + U.h);
            const float inv = ((kCtxScaled && U.slot != 0) ? p.ctx_v_scale : 1.f) / l;
            // 64 columns per TMEM round trip; each thread writes its own row,
            // 32 bytes (one whole sector) per store where the output allows
#pragma unroll 1
            for (int c = 0; c < DV / 64; ++c) {
                uint32_t r[64];
                tmem_ld32(tO + c * 64, *reinterpret_cast<uint32_t(*)[32]>(r));
                tmem_ld32(tO + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
                tmem_wait_ld();
                if (write) {
                    if (final_out) {
                        __nv_bfloat16* dst = p.out + orow * DV + c * 64;
                        uint32_t pk[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            pk[j] = pack_bf16(__uint_as_float(r[2 * j]) * inv, __uint_as_float(r[2 * j + 1]) * inv);
                        if (p.out_v8) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                st_global_v8(dst + j * 16, pk[8 * j], pk[8 * j + 1], pk[8 * j + 2], pk[8 * j + 3],
                                             pk[8 * j + 4], pk[8 * j + 5], pk[8 * j + 6], pk[8 * j + 7]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                *reinterpret_cast<uint4*>(dst + j * 8) =
                                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        }
                    } else {
                        float* dst = p.ext_o + orow * DV + c * 64;  // workspace: 256-byte aligned rows
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_global_v8(dst + j * 8, __float_as_uint(__uint_as_float(r[8 * j]) * inv),
                                         __float_as_uint(__uint_as_float(r[8 * j + 1]) * inv),
                                         __float_as_uint(__uint_as_float(r[8 * j + 2]) * inv),
                                         __float_as_uint(__uint_as_float(r[8 * j + 3]) * inv),
                                         __float_as_uint(__uint_as_float(r[8 * j + 4]) * inv),
                                         __float_as_uint(__uint_as_float(r[8 * j + 5]) * inv),
                                         __float_as_uint(__uint_as_float(r[8 * j + 6]) * inv),
                                         __float_as_uint(__uint_as_float(r[8 * j + 7]) * inv));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[k]);
            if (write) {
                const float lse_nat = (m_used + __log2f(l)) * 0.69314718055994531f;
                if (final_out) {
                    if (p.lse) p.lse[orow] = lse_nat;
                } else {
                    p.ext_lse[orow] = lse_nat;
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

template <int D, int DV, bool kCtxScaled = false>
static cudaError_t launch_fa_d(const FaMaps& maps, const FaParams& p, int num_sms, cudaStream_t stream) {
    auto kern = fa_fwd_kernel<D, DV, kCtxScaled>;
    const int smem = FaCfg<D, DV>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(num_sms), dim3(kFaThreads), smem, stream, maps, p);
}

cudaError_t launch_fa_fwd(const FaMaps& maps, const FaParams& p, int head_dim, int head_dim_v, int num_sms,
                          cudaStream_t stream) {
    const bool scaled = p.ctx_scale_log2 != p.scale_log2 || p.ctx_v_scale != 1.f;
    if (head_dim == 128 && head_dim_v == 128)
        return scaled ? launch_fa_d<128, 128, true>(maps, p, num_sms, stream)
                      : launch_fa_d<128, 128>(maps, p, num_sms, stream);
    if (scaled) return cudaErrorInvalidValue;  // scaled context chunks: head dim 128 only
    if (head_dim == 64 && head_dim_v == 64) return launch_fa_d<64, 64>(maps, p, num_sms, stream);
    if (head_dim == 192 && head_dim_v == 128) return launch_fa_d<192, 128>(maps, p, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pka
