// reorder.cu -- batch ordering for the forward pass: the host classification
// of requests into [decode : extend : prefill] ("Beyond porting", section
// "Key innovations", batch reordering; the decode threshold is 1 new token)
// and a device row gather that moves token and request rows into and out of
// that order.
#include <algorithm>
#include <vector>

#include "common.cuh"

namespace pka {

// dst row i = src row idx[i]; V = 16, 4 or 1 bytes per copy, rows of
// `vecs` copies: a grid-stride loop over (row, copy) pairs, consecutive
// threads on consecutive copies of a row (coalesced). I is the index type of
// that loop: 32-bit while the total fits (a cheaper division), else 64-bit.
template <typename V, typename I>
__global__ void gather_rows_kernel(V* __restrict__ dst, const V* __restrict__ src, const int32_t* __restrict__ idx,
                                   I num_rows, int64_t src_rows, I vecs, int32_t* err) {
    const I total = num_rows * vecs;
    for (I e = (I)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (I)gridDim.x * blockDim.x) {
        const I row = e / vecs, c = e - row * vecs;
        const int32_t s = __ldg(idx + row);
        if (s < 0 || s >= src_rows) {
            dst[e] = V{};
            if (c == 0) set_error(err, PKA_DEVERR_INDEX);
            continue;
        }
        dst[e] = src[(int64_t)s * vecs + c];
    }
}

struct alignas(16) V16 {
    uint4 v;
};
struct V1 {
    uint8_t v;
};

cudaError_t launch_gather_rows(void* dst, const void* src, const int32_t* idx, int64_t num_rows, int64_t src_rows,
                               int64_t row_bytes, int32_t* err, int num_sms, cudaStream_t stream) {
    if (num_rows == 0) return cudaSuccess;
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src);
    auto go = [&](auto tag, int bytes) -> cudaError_t {
        using V = decltype(tag);
        const int64_t vecs = row_bytes / bytes;
        const int64_t total = num_rows * vecs;
        const int threads = 256;
        const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((total + threads - 1) / threads,
                                                                       (int64_t)num_sms * 8));
        if (total < ((int64_t)1 << 31))
            gather_rows_kernel<V, uint32_t><<<blocks, threads, 0, stream>>>(
                static_cast<V*>(dst), static_cast<const V*>(src), idx, (uint32_t)num_rows, src_rows,
                (uint32_t)vecs, err);
        else
            gather_rows_kernel<V, int64_t><<<blocks, threads, 0, stream>>>(
                static_cast<V*>(dst), static_cast<const V*>(src), idx, num_rows, src_rows, vecs, err);
        return cudaGetLastError();
    };
    if (row_bytes % 16 == 0 && (a & 15) == 0) return go(V16{}, 16);
    if (row_bytes % 4 == 0 && (a & 3) == 0) return go(uint32_t{}, 4);
    return go(V1{}, 1);
}

}  // namespace pka

extern "C" {

pka_status pka_batch_order(int num_reqs, const int32_t* query_lens, const int32_t* ctx_lens, int32_t* req_order,
                           int32_t* qsl_ordered, int32_t* token_src, int32_t* token_dst, int32_t* counts) {
    if (num_reqs < 1 || !query_lens || !ctx_lens || !req_order || !qsl_ordered || !counts) return PKA_ERR_INVALID_ARG;
    int64_t T = 0;
    for (int r = 0; r < num_reqs; ++r) {
        if (query_lens[r] < 1 || ctx_lens[r] < 0) return PKA_ERR_INVALID_ARG;
        T += query_lens[r];
        if (T > INT32_MAX) return PKA_ERR_INVALID_ARG;
    }
    // class of a request: 0 decode (one new token), 1 extend, 2 prefill
    auto cls = [&](int r) { return query_lens[r] == 1 ? 0 : (ctx_lens[r] > 0 ? 1 : 2); };
    std::vector<int32_t> qsl(num_reqs + 1, 0);
    for (int r = 0; r < num_reqs; ++r) qsl[r + 1] = qsl[r] + query_lens[r];
    int n = 0;
    for (int c = 0; c < 3; ++c) {
        int cnt = 0;
        for (int r = 0; r < num_reqs; ++r)
            if (cls(r) == c) {
                req_order[n++] = r;
                ++cnt;
            }
        counts[c] = cnt;
    }
    qsl_ordered[0] = 0;
    for (int i = 0; i < num_reqs; ++i) {
        const int r = req_order[i];
        qsl_ordered[i + 1] = qsl_ordered[i] + query_lens[r];
        for (int k = 0; k < query_lens[r]; ++k) {
            const int32_t j = qsl_ordered[i] + k, t = qsl[r] + k;
            if (token_src) token_src[j] = t;
            if (token_dst) token_dst[t] = j;
        }
    }
    return PKA_OK;
}

}  // extern "C"
