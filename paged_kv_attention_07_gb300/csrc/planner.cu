// planner.cu -- validation of the batch metadata and the step's work lists.
//
// Classification follows the model runner's reorder with threshold 1
// ("Beyond porting", "Key innovations" item 2): a request with one new token
// is a decode, one with cached context and more new tokens an extend, one
// without context a prefill, and the batch must come as
// [decode : extend : prefill]. Any violation sets an error bit and leaves all
// work lists empty, so the compute kernels then touch nothing.
#include "common.cuh"
#include "plan.cuh"

namespace pka {

// Exclusive prefix sum of count(i) over i in [0, n), spread over the whole
// block: each thread takes a contiguous run of indices, the runs' totals are
// scanned with warp shuffles and one shared-memory pass. emit(i, first, count)
// is called once per index with its exclusive offset. Returns the total to
// every thread. All threads must call it (it synchronises the block); `scan`
// holds at least 33 ints. Counts and the total must fit an int.
template <typename CountF, typename EmitF>
__device__ int scan_ranges(int n, int32_t* scan, CountF count, EmitF emit) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + nthr - 1) / nthr;
    const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
    int local = 0;
    for (int i = i0; i < i1; ++i) local += count(i);
    int incl = local;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = nthr >> 5;
        int w = lane < nw ? scan[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += v;
        }
        if (lane < nw) scan[lane] = wi - w;  // exclusive offset of each warp
        if (lane == 31) scan[32] = wi;       // total (lanes past nw added 0)
    }
    __syncthreads();
    int off = scan[warp] + incl - local;
    for (int i = i0; i < i1; ++i) {
        const int c = count(i);
        emit(i, off, c);
        off += c;
    }
    const int total = scan[32];
    __syncthreads();  // `scan` may be reused by the next call
    return total;
}

__device__ __forceinline__ void plan_body(const PlanParams& p) {
    __shared__ int32_t s_qlen[kMaxRequests];
    __shared__ int32_t s_slen[kMaxRequests];
    __shared__ int32_t s_hist[kCostBuckets];
    __shared__ int32_t s_err;
    __shared__ unsigned long long s_dec_keys;
    __shared__ unsigned long long s_wsum[32];
    __shared__ int32_t s_split;
    __shared__ int32_t s_scan[33];

    // the compute kernels are launched as dependents of this one: let them
    // start (they wait for this grid to finish before reading the plan)
    grid_dep_launch();
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int nd = p.num_decodes, ne = p.num_extends;
    const int B = nd + ne + p.num_prefills;
    if (tid == 0) {
        s_err = 0;
        s_dec_keys = 0ull;
        p.hdr->err = 0;  // this call's device error word starts clean
    }
    for (int i = tid; i < kCostBuckets; i += nthr) s_hist[i] = 0;
    __syncthreads();

    // ---- load + validate
    int err = 0;
    unsigned long long dec_keys = 0;
    for (int r = tid; r < B; r += nthr) {
        const int a = p.qsl[r], b = p.qsl[r + 1], s = p.seq_lens[r];
        const int ql = b - a;
        s_qlen[r] = ql;
        s_slen[r] = s;
        if (r == 0 && a != 0) err |= PKA_DEVERR_QUERY_START_LOC;
        if (ql < 1) err |= PKA_DEVERR_QUERY_START_LOC;
        if (s < ql || s > p.max_seq_len) err |= PKA_DEVERR_SEQ_LEN;
        if (ql > p.max_query_len) err |= PKA_DEVERR_QUERY_LEN;
        if ((long long)s > (long long)p.max_blocks_per_req * p.block_size) err |= PKA_DEVERR_BLOCK_TABLE;
        const int ctx = s - ql;
        if (r < nd) {
            if (ql != 1) err |= PKA_DEVERR_ORDER;
            dec_keys += (unsigned long long)(s > 0 ? s : 0);
        } else if (r < nd + ne) {
            if (ctx < 1) err |= PKA_DEVERR_ORDER;  // one new token here takes the extend path
        } else if (ctx != 0) {
            err |= PKA_DEVERR_ORDER;
        }
    }
    if (tid == 0 && p.qsl[B] != p.num_tokens) err |= PKA_DEVERR_QUERY_START_LOC;
    // block-wide OR of the error bits and sum of the decode keys: warp
    // shuffles, then one pass over the warps' results (no shared atomics on the
    // 64-bit sum)
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        err |= __shfl_xor_sync(0xffffffffu, err, o);
        dec_keys += __shfl_xor_sync(0xffffffffu, dec_keys, o);
    }
    if ((tid & 31) == 0) {
        s_wsum[tid >> 5] = dec_keys;
        if (err) atomicOr(&s_err, err);
    }
    __syncthreads();
    if (tid == 0) {
        unsigned long long t = 0;
        for (int w = 0; w < (nthr >> 5); ++w) t += s_wsum[w];
        s_dec_keys = t;
    }
    __syncthreads();

    if (s_err) {
        if (tid == 0) {
            atomicOr(&p.hdr->err, s_err);
            p.hdr->dec_split_len = 0;
            p.hdr->dec_num_pairs = 0;
            p.hdr->fa_num_items = 0;
            p.hdr->dec_counter = 0;
            p.hdr->fa_counter = 0;
            p.hdr->ext_rows = 0;
        }
        return;
    }

    // ---- decode split length (one thread), then every request's first pair
    // and first extend partial row by block-wide prefix sums
    if (tid == 0) {
        int L = p.dec_min_split;
        if (nd > 0) {
            const unsigned long long units = s_dec_keys * (unsigned long long)p.dec_units_per_pair;
            unsigned long long want = (units + p.dec_target_units - 1) / (unsigned long long)p.dec_target_units;
            const unsigned long long a = (unsigned long long)p.dec_split_align;
            want = (want + a - 1) / a * a;
            if (want > (unsigned long long)L) L = (int)(want > (1ull << 30) ? (1ull << 30) : want);
        }
        s_split = L;
    }
    __syncthreads();
    const int L = s_split;
    // decode request r has ceil(seq_len / L) splits
    const int pairs = scan_ranges(nd, s_scan, [&](int r) { return (s_slen[r] + L - 1) / L; },
                                  [&](int r, int first, int n) {
                                      p.dec_first[r] = first;
                                      p.dec_nsplit[r] = n;
                                  });
    // extend request r has qlen * (1 + chunks) partial rows
    const int rows = scan_ranges(ne, s_scan,
                                 [&](int i) {
                                     const int r = nd + i;
                                     const int ctx = s_slen[r] - s_qlen[r];
                                     return s_qlen[r] * (1 + (ctx + p.chunk - 1) / p.chunk);
                                 },
                                 [&](int i, int first, int) { p.ext_base[i] = first; });
    if (pairs > p.dec_pair_cap || rows > p.ext_row_cap) {
        if (tid == 0) {
            atomicOr(&p.hdr->err, PKA_DEVERR_CAPACITY);
            p.hdr->dec_num_pairs = 0;
            p.hdr->fa_num_items = 0;
            p.hdr->dec_counter = 0;
            p.hdr->fa_counter = 0;
        }
        return;
    }
    // decode pairs (request, split)
    for (int r = tid; r < nd; r += nthr) {
        const int n = (s_slen[r] + L - 1) / L;
        const int base = p.dec_first[r];
        for (int s = 0; s < n; ++s) p.dec_pairs[base + s] = make_int2(r, s);
    }

    // ---- prefill / extend items. A group is one (request, slot): all query
    // tiles that read the same keys, taken two by two as items. Groups are counting-sorted by the cost of
    // their heaviest tile (heaviest first) and keep their tiles contiguous, so
    // the CTAs that share a context chunk stream it through L2 together.
    auto group_cost = [&](int r, int slot) -> int {
        const int ql = s_qlen[r];
        int keys;
        if (slot == 0) {
            keys = ql;  // the last query tile sees all new keys
        } else {
            const int ctx = s_slen[r] - ql;
            keys = min(p.chunk, ctx - (slot - 1) * p.chunk);
        }
        const int c = (keys + kFaBlockN - 1) / kFaBlockN;
        return min(c, kCostBuckets - 1);
    };
    for (int r = nd + tid; r < B; r += nthr) {
        const int ql = s_qlen[r];
        const int ctx = s_slen[r] - ql;
        const int nqt = (ql + kFaItemRows - 1) / kFaItemRows;  // items (query-tile pairs)
        const int nslot = (r < nd + ne) ? 1 + (ctx + p.chunk - 1) / p.chunk : 1;
        for (int s = 0; s < nslot; ++s) atomicAdd(&s_hist[group_cost(r, s)], nqt);
    }
    __syncthreads();
    // bucket offsets in descending cost: an exclusive scan over the reversed histogram
    const int n_items = scan_ranges(kCostBuckets, s_scan, [&](int i) { return s_hist[kCostBuckets - 1 - i]; },
                                    [&](int i, int first, int) { s_hist[kCostBuckets - 1 - i] = first; });
    if (n_items > p.fa_item_cap) {
        if (tid == 0) {
            atomicOr(&p.hdr->err, PKA_DEVERR_CAPACITY);
            p.hdr->dec_num_pairs = 0;
            p.hdr->fa_num_items = 0;
            p.hdr->dec_counter = 0;
            p.hdr->fa_counter = 0;
        }
        return;
    }
    for (int r = nd + tid; r < B; r += nthr) {
        const int ql = s_qlen[r];
        const int ctx = s_slen[r] - ql;
        const int nqt = (ql + kFaItemRows - 1) / kFaItemRows;  // items (query-tile pairs)
        const int nslot = (r < nd + ne) ? 1 + (ctx + p.chunk - 1) / p.chunk : 1;
        for (int s = 0; s < nslot; ++s) {
            const int c = group_cost(r, s);
            const int pos = atomicAdd(&s_hist[c], nqt);
            // causal groups: heaviest (last) item first
            for (int qt = 0; qt < nqt; ++qt) p.fa_items[pos + qt] = make_int4(r, s == 0 ? nqt - 1 - qt : qt, s, c);
        }
    }
    if (tid == 0) {
        p.hdr->dec_split_len = L;
        p.hdr->dec_num_pairs = pairs;
        p.hdr->fa_num_items = n_items;
        p.hdr->dec_counter = 0;
        p.hdr->fa_counter = 0;
        p.hdr->ext_rows = rows;
    }
}

__global__ void __launch_bounds__(1024) planner_kernel(PlanParams p) {
    plan_body(p);
    if (p.after_cache_write) grid_dep_wait();  // finish only after the cache write
}

cudaError_t launch_planner(const PlanParams& p, cudaStream_t stream) {
    if (p.after_cache_write) return launch_dependent(planner_kernel, dim3(1), dim3(1024), 0, stream, p);
    planner_kernel<<<1, 1024, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pka
