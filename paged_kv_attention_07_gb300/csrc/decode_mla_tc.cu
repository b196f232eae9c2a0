// decode_mla_tc.cu -- absorbed MLA decode on the 5th-generation tensor cores
// ("vLLM AMD ROCm Attention Backends Optimization", section "The hybrid
// processing strategy": decode works directly on the compressed 576-dim
// latent; the value is the latent's first 512 dims), for groups of 128
// query heads.
//
// Per key j one latent row c_j serves every head:
//     s_hj = scale * <q_h, c_j[0:576]>,   o_h = sum_j softmax_j(s_h) c_j[0:512].
// The 128 heads are the MMA's M (one TMEM lane each). Their fp32 output
// (128 x 512) alone would fill a whole SM's tensor memory, so a work unit is
// (request split, head group, value half): the two halves of a split run on
// two CTAs that compute the same scores (identical arithmetic, so identical
// softmax statistics) and each accumulate 256 value dims. They are adjacent
// in the unit order, so the second read of every latent tile hits L2.
//
// Tensor memory (512 columns, lane = head):
//     [0, 128)   S   two buffers of fp32 scores of a 64-key tile; the
//                    softmax writes that tile's P (bf16 pairs, the A operand
//                    of O += P . V) over the first 32 columns of its buffer
//     [128, 256) Qt  bf16 pairs of q[:, 0:256], the A operand of the first
//                    16 k-steps of S (no shared-memory traffic for them)
//     [256, 512) O   fp32, this unit's 256 value dims
// With two S buffers the scores of the next tile are issued right after the
// current tile's, while the softmax works on the current one: a buffer is
// reused once the P . V that read its P has completed.
// Shared memory: q[:, 256:576] (80 KB, the A operand of the last 20 k-steps)
// and a 2-stage ring of 64-key latent tiles (72 KB each), loaded with TMA
// boxes of 64 dims x min(block size, 64) rows walked through the block table;
// below block size 8, and for a split's last, partial tile, TMA gathers of
// four latent rows x 64 dims each (rows past the split's end are read at an
// out-of-range row, which TMA fills with zeros).
//
// Persistent CTAs, one per SM, allocate tensor memory once and take units
// from an atomic counter; warp 0 publishes each unit index to the other roles
// through a 2-slot ring in shared memory. Warps: 0 producer of q and the
// score-only chunks, 6 producer of the value chunks, 1 tensor-memory owner +
// MMA issuer (one elected lane issues), 2-5 softmax (one thread per head):
// S row -> online softmax (the O rescale is lazy: only when the max grew by
// more than 2^8) -> P into TMEM; at the end of a unit O / l goes to out, or
// to the fp32 split partials + LSE that the decode reduction merges.
// Per tile t the issuer runs S(t) part 1, O += P(t-1) . V(t-1), S(t) part 2;
// the commit after S(t) part 2 thus also covers the P . V before it, so the
// softmax may rescale O as soon as it sees S(t).
#include <type_traits>

#include "common.cuh"
#include "params.cuh"
#include "plan.cuh"
#include "tcgen05.cuh"

namespace pka {

constexpr int kMtThreads = 224;
constexpr int kMtTile = 64;                       // keys per tile (the N of S)
constexpr int kMtD = 576, kMtDv = 512, kMtHalf = 256;
constexpr int kMtQtDims = 256;                    // q dims held in TMEM
constexpr int kMtChunk = kMtTile * 128;           // one 64-dim column chunk of a tile (8 KB)
constexpr int kMtTileBytes = 9 * kMtChunk;        // 72 KB
constexpr int kMtQsChunk = 128 * 128;             // 128 heads x 64 dims
constexpr int kMtQsChunks = (kMtD - kMtQtDims) / 64;
constexpr int kMtQsBytes = kMtQsChunks * kMtQsChunk;  // q[:, 256:576]
constexpr int kMtOffQ = 0;
constexpr int kMtOffKV = kMtQsBytes;
constexpr int kMtOffBar = kMtOffKV + 2 * kMtTileBytes;
constexpr int kMtSmem = kMtOffBar + 256 + 1024;
constexpr uint32_t kMtColS = 0, kMtColQ = 128, kMtColO = 256, kMtCols = 512;  // S buffer b at kMtColS + 64 b
static_assert(kMtSmem <= 227 * 1024, "shared memory");
static_assert(kMtColQ + kMtQtDims / 2 == kMtColO && kMtColS + 2 * kMtTile == kMtColQ, "tensor memory columns");

struct MlaTcUnit {
    int pair, grp, half, r, k0, k1, ntiles;
};

PKA_DEVICE MlaTcUnit mla_tc_unit(const DecodeMlaParams& p, int u, int L) {
    MlaTcUnit U;
    const int upp = 2 * p.groups;
    U.pair = u / upp;
    const int rem = u - U.pair * upp;
    U.grp = rem >> 1;
    U.half = rem & 1;
    const int2 rs = p.pairs[U.pair];
    U.r = rs.x;
    U.k0 = rs.y * L;
    U.k1 = min(U.k0 + L, p.seq_lens[U.r]);
    U.ntiles = (U.k1 - U.k0 + kMtTile - 1) / kMtTile;
    return U;
}

// A unit the kernel can run without touching memory it does not own.
PKA_DEVICE bool mla_tc_unit_ok(const DecodeMlaParams& p, const MlaTcUnit& U) {
    return U.r >= 0 && U.k0 >= 0 && U.k1 > U.k0 && U.grp < p.groups;
}

__global__ void __launch_bounds__(kMtThreads, 1)
    decode_mla_tc_kernel(const __grid_constant__ CUtensorMap kvmap, const __grid_constant__ CUtensorMap qmap,
                         const __grid_constant__ CUtensorMap gmap, const DecodeMlaParams p) {
    grid_dep_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kMtOffBar);
    // A latent stage is two parts with their own barriers: the value chunks
    // this unit's P . V reads, and the other (score-only) chunks, which are
    // free again as soon as the first part of S has read them.
    uint64_t* kv_full = bars + 0;     // [2] score-only chunks landed
    uint64_t* kv_empty = bars + 2;    // [2] score-only chunks read by S
    uint64_t* kv_full_v = bars + 16;  // [2] value chunks landed
    uint64_t* u_full = bars + 4;     // [2] unit ring slot written
    uint64_t* u_empty = bars + 6;    // [2] unit ring slot read by the issuer, the value producer and the 4 softmax warps
    uint64_t* q_full = bars + 8;     // q[:, 256:576] landed in shared memory
    uint64_t* q_empty = bars + 9;    // the unit's last S product is done (Q free again)
    uint64_t* qt_ready = bars + 10;  // q[:, 0:256] written to TMEM (4 warps)
    uint64_t* s_full = bars + 11;    // a tile's S complete (and the P . V issued before its part 2)
    uint64_t* p_full = bars + 13;    // 4 warps wrote P (and rescaled O)
    // [2] the P . V of the tiles using S buffer b complete: b is free again,
    // and so are the value chunks of stage b (a tile's stage and S buffer are
    // both its index in this CTA's tile sequence, mod 2)
    uint64_t* pv_buf = bars + 20;
    uint64_t* o_full = bars + 22;    // a unit's last P . V complete
    uint64_t* o_free = bars + 15;    // 4 warps read O
    __shared__ uint32_t s_tmem;
    __shared__ int s_unit[2];
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_units = p.hdr->dec_num_pairs * 2 * p.groups;
    if (num_units == 0) return;
    const int L = p.hdr->dec_split_len;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
            mbar_init(&kv_full_v[i], 1);
            mbar_init(&u_full[i], 1);
            mbar_init(&u_empty[i], 6);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(qt_ready, 4);
        mbar_init(s_full, 1);
        mbar_init(p_full, 4);
        mbar_init(&pv_buf[0], 1);
        mbar_init(&pv_buf[1], 1);
        mbar_init(o_full, 1);
        mbar_init(o_free, 4);
        fence_barrier_init();
        s_abort = 0;
        tma_prefetch_desc(&kvmap);
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&gmap);
    }
    if (warp == 1) tmem_alloc(&s_tmem, kMtCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s_tmem;
    const uint32_t sm_base = smem_u32(smem);

    // Next unit index from the ring (every consumer reads each slot once).
    auto take_unit = [&](uint32_t i, bool arrive, int* u) -> bool {
        const int slot = i & 1;
        if (!mbar_wait_warp(&u_full[slot], (i >> 1) & 1, p.err)) return false;
        *u = s_unit[slot];
        __syncwarp();
        if (arrive) mbar_arrive(&u_empty[slot]);
        return true;
    };

    if (warp == 0 || warp == 6) {
        // ------------------------------------------------------------ producers
        // warp 0 takes the units and loads q[:, 256:576] and the score-only
        // part of each stage; warp 6 loads the value part, so neither part of
        // a stage waits behind the other's free slot.
        const int part = warp == 6 ? 1 : 0;
        const uint64_t pol = policy_evict_normal();  // the other value half re-reads each tile
        const bool use_tma = p.bs >= 8;
        uint32_t kv_it = 0, q_it = 0;
        uint32_t last[2] = {0, 0};  // phase + 1 of this part's last copy per stage (0 = none)
        int stage_half0 = -1, stage_half1 = -1;  // value half of the unit that last used stage 0 / 1
        for (uint32_t i = 0; !warp_flag(s_abort); ++i) {
            int u = 0;
            if (part == 0) {
                const int slot = i & 1;
                if (i >= 2 && !mbar_wait_warp(&u_empty[slot], ((i >> 1) - 1) & 1, p.err)) {
                    s_abort = 1;
                    break;
                }
                if (lane == 0) u = atomicAdd(p.counter, 1);
                u = __shfl_sync(0xffffffffu, u, 0);
                if (u >= num_units) u = -1;
                if (lane == 0) {
                    s_unit[slot] = u;
                    mbar_arrive(&u_full[slot]);
                }
                __syncwarp();
            } else if (!take_unit(i, lane == 0, &u)) {
                s_abort = 1;
                break;
            }
            if (u < 0) break;
            const MlaTcUnit U = mla_tc_unit(p, u, L);
            if (!mla_tc_unit_ok(p, U)) {
                if (part == 0 && lane == 0) set_error(p.err, PKA_DEVERR_CAPACITY);
                continue;
            }
            if (part == 0) {
                if (q_it > 0 && !mbar_wait_warp(q_empty, (q_it - 1) & 1, p.err)) {
                    s_abort = 1;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(q_full, kMtQsBytes);
                    for (int c = 0; c < kMtQsChunks; ++c)
                        tma_load_3d(smem + kMtOffQ + c * kMtQsChunk, &qmap, q_full, kMtQtDims + c * 64, U.grp * 128,
                                    U.r, pol);
                }
                ++q_it;
            }
            const int32_t* bt = p.block_table + (int64_t)U.r * p.max_blocks;
            // validated block id of key position `pos` of this request
            auto block_of = [&](int pos) -> int {
                int blk = __ldg(bt + pos / p.bs);
                if (blk < 0 || blk >= p.num_blocks) {
                    set_error(p.err, PKA_DEVERR_BLOCK_ID);
                    blk = 0;
                }
                return blk;
            };
            bool ok = true;
            const uint32_t vmask = U.half ? 0xF0u : 0x0Fu;  // chunks holding this half's value dims
            // this part's chunks in order (gather path: a warp step takes two of
            // them, one per half warp); entries past the count are -1
            const uint32_t my_mask = part ? vmask : (0x1FFu & ~vmask);
            int cl[6];
            {
                uint32_t m = my_mask;
#pragma unroll
                for (int j = 0; j < 6; ++j) {
                    cl[j] = m ? __ffs(m) - 1 : -1;
                    m &= m - 1;
                }
            }
            for (int t = 0; t < U.ntiles; ++t, ++kv_it) {
                const int st = kv_it & 1;
                const uint32_t n = kv_it >> 1;
                uint8_t* dst = smem + kMtOffKV + st * kMtTileBytes;
                const int tb = U.k0 + t * kMtTile;
                const int valid = min(kMtTile, U.k1 - tb);
                const bool tma = use_tma && valid == kMtTile;
                // gather path: lanes l and l + 16 take rows 4l .. 4l + 3 of the tile
                int grow[4] = {0, 0, 0, 0};
                if (!tma) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int pos = tb + 4 * (lane & 15) + k;
                        grow[k] = pos < U.k1 ? block_of(pos) * p.bs + (pos % p.bs) : p.cache_rows;  // out of range: zeros
                    }
                }
                // part 0: the score-only chunks, part 1: the value chunks
                {
                    uint64_t* empty = part ? &pv_buf[st] : &kv_empty[st];
                    uint64_t* full = part ? &kv_full_v[st] : &kv_full[st];
                    const uint32_t cmask = part ? vmask : (0x1FFu & ~vmask);
                    if (n > 0 && !mbar_wait_warp(empty, (n - 1) & 1, p.err)) {
                        ok = false;
                        break;
                    }
                    // The parts are split by the unit's value half. After a unit of the
                    // other half, this unit's score-only chunks are that unit's value
                    // chunks, free only once its P . V has read them. (The value part
                    // needs no such wait: its release comes after the previous tile's
                    // whole S, score-only chunks included.)
                    if (part == 0 && n > 0 && (st ? stage_half1 : stage_half0) != U.half &&
                        !mbar_wait_warp(&pv_buf[st], (n - 1) & 1, p.err)) {
                        ok = false;
                        break;
                    }
                    if (st) stage_half1 = U.half;
                    else stage_half0 = U.half;
                    if (tma) {
                        const int rows = p.bs < kMtTile ? p.bs : kMtTile;  // rows per box
                        const int nbox = kMtTile / rows;
                        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(__popc(cmask) * kMtChunk));
                        __syncwarp();
                        if (lane < nbox) {  // one lane per box, in parallel
                            const int pos = tb + lane * rows;
                            const int row = block_of(pos) * p.bs + (pos % p.bs);
                            for (int c = 0; c < 9; ++c)
                                if ((cmask >> c) & 1)
                                    tma_load_2d(dst + c * kMtChunk + lane * rows * 128, &kvmap, full, c * 64, row, pol);
                        }
                    } else {
                        // TMA gathers, 4 rows x 64 dims per instruction, all 32 lanes in
                        // parallel (two chunks per warp step); every chunk's bytes arrive
                        // (rows past the end as zeros)
                        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(__popc(cmask) * kMtChunk));
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 6; j += 2) {
                            const int c = lane < 16 ? cl[j] : cl[j + 1];
                            if (c >= 0)
                                tma_gather4(dst + c * kMtChunk + (lane & 15) * 4 * 128, &gmap, full, c * 64, grow[0],
                                            grow[1], grow[2], grow[3]);
                        }
                    }
                }
                if (!ok) break;
                last[st] = n + 1;
            }
            if (!ok) {
                s_abort = 1;
                break;
            }
        }
        // no copy may outlive the CTA: wait (bounded) for the last one per stage
        for (int st = 0; st < 2; ++st)
            if (last[st]) mbar_wait_warp(part ? &kv_full_v[st] : &kv_full[st], (last[st] - 1) & 1, p.err);
        if (q_it > 0) mbar_wait_warp(q_full, (q_it - 1) & 1, p.err);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop (waits, counters and descriptors are
        // warp-uniform) and one elected lane issues each MMA and commit.
        constexpr uint32_t idesc_s = umma_idesc_bf16(128, kMtTile, 0, 0);
        constexpr uint32_t idesc_o = umma_idesc_bf16(128, kMtHalf, 0, 1);
        const uint32_t q_s = sm_base + kMtOffQ, kv_s = sm_base + kMtOffKV;
        uint32_t kv_it = 0, s_it = 0, pv_it = 0, q_it = 0;
        uint32_t pv_last = 0;  // tile (S counter) of the last P . V issued
        bool ok = true;
        // S = q . C^T over all 576 dims, in two parts: the score-only chunks
        // first (their stage part is released right after), then the value
        // chunks. k-steps over q[:, 0:256] take A from TMEM, the rest from
        // shared memory. The chunk sets are fixed per value half, so each part
        // is straight-line code.
        auto issue_s_part = [&](uint32_t kvi, uint32_t tS, auto half_c, auto part_c) {
            constexpr int H = decltype(half_c)::value, PART = decltype(part_c)::value;
            constexpr int first_c = H ? 0 : 4;  // first chunk of part 0: it starts the accumulation
            const uint32_t kv = kv_s + (kvi & 1) * kMtTileBytes;
#pragma unroll
            for (int c = 0; c < 9; ++c) {
                const bool vchunk = H ? (c >= 4 && c < 8) : (c < 4);
                if (vchunk != (PART == 1)) continue;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int ks = 4 * c + kk;
                    const uint64_t bdesc = umma_desc_sw128(kv + c * kMtChunk + kk * 32, 16, 1024);
                    const uint32_t acc = (PART == 0 && c == first_c && kk == 0) ? 0u : 1u;
                    if (c < kMtQtDims / 64)
                        umma_bf16_ts_w(tS, tbase + kMtColQ + ks * 8, bdesc, idesc_s, acc);
                    else
                        umma_bf16_w(tS, umma_desc_sw128(q_s + (c - kMtQtDims / 64) * kMtQsChunk + kk * 32, 16, 1024),
                                    bdesc, idesc_s, acc);
                }
            }
        };
        // O(half) += P . C[:, half*256 .. +256), P in the first 32 columns of
        // S buffer b; the commit on pv_buf[b] frees that buffer
        auto issue_o = [&](uint32_t kvi, int half, bool first, uint32_t b) -> bool {
            if (!mbar_wait_warp(p_full, pv_it & 1, p.err)) return false;
            // a unit's first product overwrites O: the previous unit's O must have been read
            if (first && q_it > 1 && !mbar_wait_warp(o_free, (q_it - 2) & 1, p.err)) return false;
            tc_fence_after();
            const uint32_t v = kv_s + (kvi & 1) * kMtTileBytes + half * 4 * kMtChunk;
#pragma unroll
            for (int kk = 0; kk < kMtTile / 16; ++kk)
                umma_bf16_ts_w(tbase + kMtColO, tbase + kMtColS + b * kMtTile + kk * 8,
                               umma_desc_sw128(v + kk * 16 * 128, kMtChunk, 1024), idesc_o, (!first || kk > 0) ? 1u : 0u);
            umma_commit_w(&pv_buf[b]);  // b == kvi & 1: also frees the stage's value chunks
            ++pv_it;
            pv_last = s_it - 1;
            return true;
        };
        for (uint32_t i = 0; ok && !warp_flag(s_abort); ++i) {
            int u = 0;
            if (!take_unit(i, lane == 0, &u)) {
                ok = false;
                break;
            }
            if (u < 0) break;
            const MlaTcUnit U = mla_tc_unit(p, u, L);
            if (!mla_tc_unit_ok(p, U)) continue;
            ++q_it;  // units started (1-based below)
            if (!mbar_wait_warp(q_full, (q_it - 1) & 1, p.err) || !mbar_wait_warp(qt_ready, (q_it - 1) & 1, p.err)) {
                ok = false;
                break;
            }
            const uint32_t kv_base = kv_it;
            bool next_landed = false;  // the next tile's score-only chunks were seen complete
            for (int t = 0; t < U.ntiles; ++t, ++kv_it) {
                const int st = kv_it & 1;
                const uint32_t b = s_it & 1;  // S buffer of this tile
                const uint32_t tS = tbase + kMtColS + b * kMtTile;
                if (!next_landed && !mbar_wait_warp(&kv_full[st], (kv_it >> 1) & 1, p.err)) { ok = false; break; }
                next_landed = false;
                // buffer b last held the P of tile s_it - 2: its P . V must be done
                if (s_it >= 2 && !mbar_wait_warp(&pv_buf[b], ((s_it >> 1) - 1) & 1, p.err)) { ok = false; break; }
                tc_fence_after();
                if (U.half) issue_s_part(kv_it, tS, std::integral_constant<int, 1>{}, std::integral_constant<int, 0>{});
                else issue_s_part(kv_it, tS, std::integral_constant<int, 0>{}, std::integral_constant<int, 0>{});
                umma_commit_w(&kv_empty[st]);  // score-only chunks free once read
                // O += P . V of the previous tile goes between the two parts of
                // S: its value chunks are then released a whole S part earlier
                if (t > 0 && !issue_o(kv_it - 1, U.half, t == 1, b ^ 1u)) { ok = false; break; }
                // look (without blocking) at the next tile's score-only chunks now,
                // while MMAs are queued, instead of waiting for them after part 2
                if (t + 1 < U.ntiles)
                    next_landed = __all_sync(0xffffffffu, mbar_test_wait(&kv_full[st ^ 1], ((kv_it + 1) >> 1) & 1));
                if (!mbar_wait_warp(&kv_full_v[st], (kv_it >> 1) & 1, p.err)) { ok = false; break; }
                tc_fence_after();
                if (U.half) issue_s_part(kv_it, tS, std::integral_constant<int, 1>{}, std::integral_constant<int, 1>{});
                else issue_s_part(kv_it, tS, std::integral_constant<int, 0>{}, std::integral_constant<int, 1>{});
                umma_commit_w(s_full);
                ++s_it;
                if (t == U.ntiles - 1) umma_commit_w(q_empty);
            }
            if (ok && !issue_o(kv_base + U.ntiles - 1, U.half, U.ntiles == 1, (s_it - 1) & 1u)) ok = false;
            if (ok) umma_commit_w(o_full);
        }
        if (!ok) s_abort = 1;
        // let every issued MMA finish before the CTA can exit: the last P . V
        // (its buffer's earlier phases were all waited for above) covers them
        if (pv_it > 0) mbar_wait_warp(&pv_buf[pv_last & 1], (pv_last >> 1) & 1, p.err);
    } else if (warp <= 5) {
        // ------------------------------------------------------------ softmax (one thread per head)
        const int hl = 32 * (warp & 3) + lane;  // head within the group = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tQ = tbase + lane_off + kMtColQ, tO = tbase + lane_off + kMtColO;
        const float sl2 = p.scale_log2;
        uint32_t s_it = 0, o_seen = 0;
        for (uint32_t i = 0; !warp_flag(s_abort); ++i) {
            int u = 0;
            if (!take_unit(i, lane == 0, &u)) {
                s_abort = 1;
                break;
            }
            if (u < 0) break;
            const MlaTcUnit U = mla_tc_unit(p, u, L);
            if (!mla_tc_unit_ok(p, U)) continue;
            const int h = U.grp * 128 + hl;
            // q[h, 0:256] -> TMEM. The previous unit's last S product, the
            // only reader of these columns, is done: this warp saw its S.
            {
                const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((int64_t)U.r * p.Hq + h) * kMtD);
#pragma unroll 1
                for (int c = 0; c < kMtQtDims / 64; ++c) {  // 64 dims = 32 columns per step
                    uint32_t r[32];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint4 v = __ldg(qrow + c * 8 + k);
                        r[4 * k] = v.x;
                        r[4 * k + 1] = v.y;
                        r[4 * k + 2] = v.z;
                        r[4 * k + 3] = v.w;
                    }
                    tmem_st32(tQ + c * 32, r);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(qt_ready);
            }
            float m_used = -INFINITY, l = 0.f;
            bool ok = true;
            for (int t = 0; t < U.ntiles; ++t) {
                if (!mbar_wait_warp(s_full, s_it & 1, p.err)) { ok = false; break; }
                tc_fence_after();
                // this tile's S buffer; its P goes over the first 32 columns
                const uint32_t tS = tbase + lane_off + kMtColS + (s_it & 1) * kMtTile;
                float s[kMtTile];
                {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tS, r0);
                    tmem_ld32(tS + 32, r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        s[k] = __uint_as_float(r0[k]);
                        s[32 + k] = __uint_as_float(r1[k]);
                    }
                }
                ++s_it;
                const int valid = min(kMtTile, U.k1 - (U.k0 + t * kMtTile));
                if (valid < kMtTile) {
#pragma unroll
                    for (int k = 0; k < kMtTile; ++k) s[k] = k < valid ? s[k] : -INFINITY;
                }
                // row max with three-input max (two scores per instruction), 8 chains
                float mv[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mv[k] = fmaxf(s[k], s[8 + k]);
                static_assert(kMtTile % 16 == 0, "tile");
#pragma unroll
                for (int k = 16; k < kMtTile; k += 16)
#pragma unroll
                    for (int j = 0; j < 8; ++j) mv[j] = fmax3f(mv[j], s[k + j], s[k + 8 + j]);
                const float mx = fmaxf(fmaxf(fmaxf(mv[0], mv[1]), fmaxf(mv[2], mv[3])),
                                       fmaxf(fmaxf(mv[4], mv[5]), fmaxf(mv[6], mv[7])));
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
                uint32_t pk[kMtTile / 2];
                float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k = 0; k < kMtTile; k += 2) {  // packed fp32 FMA and add: two scores per instruction
                    float x0, x1;
                    fma2_bcast(x0, x1, s[k], s[k + 1], sl2, -m_used);
                    const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
                    const int j = (k >> 1) & 3;
                    add2(ls[2 * j], ls[2 * j + 1], e0, e1);
                    pk[k / 2] = pack_bf16(e0, e1);
                }
                l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                // O is free to rescale: the P . V of the previous tile was
                // issued before this tile's S part 2, whose commit we waited for
                // tcgen05.ld/st are warp-collective (.sync.aligned): the whole warp
                // takes this branch if any of its heads needs the rescale (alpha
                // stays 1 for the others)
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int c = 0; c < kMtHalf / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tO + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
                        tmem_st32(tO + c * 32, r);
                    }
                }
                tmem_st32(tS, pk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
            }
            if (!ok) {
                s_abort = 1;
                break;
            }
            if (!mbar_wait_warp(o_full, o_seen & 1, p.err)) {
                s_abort = 1;
                break;
            }
            ++o_seen;
            tc_fence_after();
            // ---- epilogue: this half's 256 value dims of O / l
            const bool direct = p.nsplit[U.r] == 1;
            const float inv = 1.f / l;
            const int64_t orow = direct ? ((int64_t)U.r * p.Hq + h) : ((int64_t)U.pair * p.Hq + h);
#pragma unroll 1
            for (int c = 0; c < kMtHalf / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tO + c * 32, r);
                tmem_wait_ld();
                const int d0 = U.half * kMtHalf + c * 32;
                if (direct) {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kMtDv + d0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_uint4(pack_bf16(__uint_as_float(r[8 * k]) * inv, __uint_as_float(r[8 * k + 1]) * inv),
                                            pack_bf16(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv),
                                            pack_bf16(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv),
                                            pack_bf16(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv));
                } else {
                    float4* dst = reinterpret_cast<float4*>(p.part_o + orow * kMtDv + d0);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                                             __uint_as_float(r[4 * k + 2]) * inv, __uint_as_float(r[4 * k + 3]) * inv);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            if (U.half == 0) {
                const float lse_nat = (m_used + __log2f(l)) * 0.69314718055994531f;
                if (direct) {
                    if (p.lse) p.lse[orow] = lse_nat;
                } else {
                    p.part_lse[orow] = lse_nat;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kMtCols);
    }
}

bool decode_mla_tc_supported(int Hq) { return Hq > 0 && Hq % 128 == 0; }

cudaError_t launch_decode_mla_tc(const CUtensorMap& kvmap, const CUtensorMap& qmap, const CUtensorMap& gmap,
                                 const DecodeMlaParams& p, int num_sms, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(decode_mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMtSmem);
    if (e != cudaSuccess) return e;
    return launch_dependent(decode_mla_tc_kernel, dim3(num_sms), dim3(kMtThreads), kMtSmem, stream, kvmap, qmap, gmap,
                            p);
}

}  // namespace pka
