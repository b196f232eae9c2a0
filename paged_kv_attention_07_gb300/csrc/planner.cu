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

__global__ void __launch_bounds__(1024) planner_kernel(PlanParams p) {
    __shared__ int32_t s_qlen[kMaxRequests];
    __shared__ int32_t s_slen[kMaxRequests];
    __shared__ int32_t s_hist[kCostBuckets];
    __shared__ int32_t s_err;
    __shared__ unsigned long long s_dec_keys;
    __shared__ int32_t s_split, s_pairs, s_items, s_rows;

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int nd = p.num_decodes, ne = p.num_extends;
    const int B = nd + ne + p.num_prefills;
    if (tid == 0) {
        s_err = 0;
        s_dec_keys = 0ull;
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
    if (err) atomicOr(&s_err, err);
    if (dec_keys) atomicAdd(&s_dec_keys, dec_keys);
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

    // ---- decode split length and pair offsets (serial scan over smem)
    if (tid == 0) {
        int L = p.dec_min_split;
        if (nd > 0) {
            const unsigned long long units = s_dec_keys * (unsigned long long)p.dec_units_per_pair;
            unsigned long long want = (units + p.dec_target_units - 1) / (unsigned long long)p.dec_target_units;
            const unsigned long long a = (unsigned long long)p.dec_split_align;
            want = (want + a - 1) / a * a;
            if (want > (unsigned long long)L) L = (int)(want > (1ull << 30) ? (1ull << 30) : want);
        }
        int pairs = 0;
        for (int r = 0; r < nd; ++r) {
            const int n = (s_slen[r] + L - 1) / L;
            p.dec_first[r] = pairs;
            p.dec_nsplit[r] = n;
            pairs += n;
        }
        int rows = 0;
        for (int r = nd; r < nd + ne; ++r) {
            const int ctx = s_slen[r] - s_qlen[r];
            const int nslot = 1 + (ctx + p.chunk - 1) / p.chunk;
            p.ext_base[r - nd] = rows;
            rows += s_qlen[r] * nslot;
        }
        s_split = L;
        s_pairs = pairs;
        s_rows = rows;
    }
    __syncthreads();
    const int L = s_split;
    if (s_pairs > p.dec_pair_cap || s_rows > p.ext_row_cap) {
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
    if (tid == 0) {
        int acc = 0;
        for (int c = kCostBuckets - 1; c >= 0; --c) {  // descending cost
            const int n = s_hist[c];
            s_hist[c] = acc;
            acc += n;
        }
        s_items = acc;
    }
    __syncthreads();
    const int n_items = s_items;
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
        p.hdr->dec_num_pairs = s_pairs;
        p.hdr->fa_num_items = n_items;
        p.hdr->dec_counter = 0;
        p.hdr->fa_counter = 0;
        p.hdr->ext_rows = s_rows;
    }
}

cudaError_t launch_planner(const PlanParams& p, cudaStream_t stream) {
    planner_kernel<<<1, 1024, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pka
