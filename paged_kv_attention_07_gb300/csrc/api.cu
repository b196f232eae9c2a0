// api.cu -- host side of the C ABI (include/pka.h): argument validation,
// workspace layout, TMA descriptor encoding and the launch sequence of one
// step. Everything is asynchronous on the caller's stream; nothing here
// allocates device memory.
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "params.cuh"
#include "plan.cuh"

namespace pka {

// kernels (defined in the other translation units)
cudaError_t launch_planner(const PlanParams& p, cudaStream_t stream);
cudaError_t launch_cache_write(const void* k, const void* v, const int64_t* slots, int64_t T, int Hkv,
                               int d, int dv, void* k_cache, void* v_cache, int64_t num_blocks, int bs,
                               int32_t* err, int num_sms, cudaStream_t stream, bool fp8, float k_scale,
                               float v_scale);
cudaError_t launch_decode_gqa_fp8(const CUtensorMap& km, const CUtensorMap& vm, const DecodeGqaParams& p, bool tma,
                                  int num_sms, cudaStream_t stream);
cudaError_t launch_merge_pair(void* out, float* out_lse, const void* a, const float* a_lse, const void* b,
                              const float* b_lse, int64_t rows, int dv, int io_dtype, int num_sms,
                              cudaStream_t stream);

cudaError_t launch_decode_gqa(const CUtensorMap& km, const CUtensorMap& vm, const DecodeGqaParams& p,
                              int head_dim, bool tma, int num_sms, cudaStream_t stream);
cudaError_t launch_decode_mla(const CUtensorMap& map, const DecodeMlaParams& p, bool tma, int num_sms,
                              cudaStream_t stream);
cudaError_t launch_fa_fwd(const FaMaps& maps, const FaParams& p, int head_dim, int head_dim_v, int num_sms,
                          cudaStream_t stream);
cudaError_t launch_decode_reduce(const DecodeReduceParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_gather_rows(void* dst, const void* src, const int32_t* idx, int64_t num_rows, int64_t src_rows,
                               int64_t row_bytes, int32_t* err, int num_sms, cudaStream_t stream);
cudaError_t launch_extend_reduce(const ExtendReduceParams& p, int ext_tokens_bound, int num_sms,
                                 cudaStream_t stream);
cudaError_t launch_ctx_dequant(const CtxDequantParams& p, cudaStream_t stream);
int decode_gqa_target_units(int num_sms);
int decode_gqa_fp8_target_units(int num_sms);
int decode_mla_heads_per_cta(int Hq);
bool decode_mla_tc_supported(int Hq);
cudaError_t launch_decode_mla_tc(const CUtensorMap& kvmap, const CUtensorMap& qmap, const CUtensorMap& gmap,
                                 const DecodeMlaParams& p, int num_sms, cudaStream_t stream);

// MLA decode units per (request, split): on the tensor-core kernel two value
// halves per group of 128 heads, otherwise one unit per 64-head group.
static int mla_units_per_pair(int Hq) {
    return decode_mla_tc_supported(Hq) ? 2 * (Hq / 128) : Hq / decode_mla_heads_per_cta(Hq);
}

namespace {

constexpr int kMlaMinSplit = 1024;

int device_sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D bf16 view [rows, cols] (row-major, dense) read in boxes of
// 64 columns x box_rows rows with the 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte view [rows, 128] (8-bit cache rows of 128 codes) read in boxes
// of 128 bytes x box_rows rows with the 128-byte swizzle.
bool encode_rows_u8(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 view of a token-major tensor [T, H, D] read in boxes of 64
// columns x `box_heads` heads x 1 token (128-byte swizzle): one box gives 64
// dims of a run of consecutive heads of one token.
bool encode_heads(CUtensorMap* map, const void* base, uint64_t T, uint64_t H, uint64_t D, uint32_t box_heads) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {D, H, T};
    cuuint64_t strides[2] = {D * 2, H * D * 2};
    cuuint32_t box[3] = {64, box_heads, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 view of a token-major tensor [T, H, D] read in boxes of
// 64 columns x 1 head x 128 tokens (128-byte swizzle): one box gives 128
// consecutive tokens of one head, 128 bytes per token.
bool encode_tokens(CUtensorMap* map, const void* base, uint64_t T, uint64_t H, uint64_t D) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {D, H, T};
    cuuint64_t strides[2] = {D * 2, H * D * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

struct Hints {
    int nd, ne, np, T, Hq, Hkv, d, dv, maxq, maxs, chunk;
    bool mla;
    bool fp8 = false;  // 8-bit cache: the extends' context is gathered into the workspace
};

constexpr int kCtxRows = 128;  // rows of a gathered context block

// Returns false if the hints are not a shape this build supports.
bool compute_layout(const Hints& h, int num_sms, Layout* L) {
    std::memset(L, 0, sizeof(*L));
    size_t off = sizeof(PlanHeader);
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align256(off + bytes);
        return o;
    };
    const int upp = h.mla ? mla_units_per_pair(h.Hq) : h.Hkv;
    L->dec_target_units = h.mla  ? num_sms * 4
                          : h.fp8 ? decode_gqa_fp8_target_units(num_sms)
                                  : decode_gqa_target_units(num_sms);
    if (L->dec_target_units < 1) L->dec_target_units = 1;
    const int64_t pair_cap = h.nd > 0 ? (int64_t)L->dec_target_units / upp + h.nd + 1 : 0;
    int64_t item_cap = 0, row_cap = 0;
    if (h.ne + h.np > 0) {
        const int64_t t_nd = (int64_t)h.T - h.nd;
        const int64_t smax = h.ne > 0 ? 1 + ceil_div(std::max(0, h.maxs - 2), h.chunk) : 1;
        item_cap = (ceil_div(t_nd, kFaBlockM) + h.ne + h.np) * smax;
        if (h.ne > 0) row_cap = std::min<int64_t>(t_nd - h.np, (int64_t)h.ne * h.maxq) * smax;
        if (row_cap < 0) row_cap = 0;
    }
    if (pair_cap > INT32_MAX / 4 || item_cap > INT32_MAX / 4 || row_cap > INT32_MAX / 4) return false;
    L->dec_pair_cap = (int)pair_cap;
    L->fa_item_cap = (int)item_cap;
    L->ext_row_cap = (int)row_cap;
    L->off_dec_pairs = take(sizeof(int2) * (size_t)pair_cap);
    L->off_dec_first = take(sizeof(int32_t) * (size_t)h.nd);
    L->off_dec_nsplit = take(sizeof(int32_t) * (size_t)h.nd);
    L->off_fa_items = take(sizeof(int4) * (size_t)item_cap);
    L->off_ext_base = take(sizeof(int32_t) * (size_t)h.ne);
    L->off_dec_part_o = take(sizeof(float) * (size_t)pair_cap * h.Hq * h.dv);
    L->off_dec_part_lse = take(sizeof(float) * (size_t)pair_cap * h.Hq);
    L->off_ext_part_o = take(sizeof(float) * (size_t)row_cap * h.Hq * h.dv);
    L->off_ext_part_lse = take(sizeof(float) * (size_t)row_cap * h.Hq);
    if (h.fp8 && h.ne > 0) {
        // every extend's context fits ceil(max_seq_len / 128) blocks
        const int64_t nblk = (h.maxs + kCtxRows - 1) / kCtxRows;
        const int64_t rows = (int64_t)h.ne * nblk * kCtxRows * h.Hkv;
        if (nblk > INT32_MAX / 4 || (int64_t)h.ne * nblk > INT32_MAX / 4 || rows >= (int64_t)INT32_MAX) return false;
        L->ctx_nblk = (int)nblk;
        L->off_ctx_k = take(sizeof(uint16_t) * (size_t)rows * h.d);
        L->off_ctx_v = take(sizeof(uint16_t) * (size_t)rows * h.dv);
        L->off_ctx_bt = take(sizeof(int32_t) * (size_t)h.ne * nblk);
    }
    L->total = off;
    return true;
}

pka_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA; }

// ---- kernel timers (benchmarking aid)
constexpr int kTimerSlots = 4096;
struct KernelTimer {
    bool on = false;
    int launches = 0;
    int timed = 0;
    cudaEvent_t ev[2 * kTimerSlots] = {};
};
KernelTimer g_timers[PKA_KERNEL_COUNT];
std::mutex g_timer_mu;

// Records the start event of a timed launch; returns the slot or -1.
int timer_begin(int kernel, cudaStream_t st) {
    KernelTimer& t = g_timers[kernel];
    if (!t.on) return -1;
    std::lock_guard<std::mutex> lock(g_timer_mu);
    ++t.launches;
    if (t.timed >= kTimerSlots) return -1;
    const int slot = t.timed;
    for (int i = 0; i < 2; ++i)
        if (!t.ev[2 * slot + i] && cudaEventCreate(&t.ev[2 * slot + i]) != cudaSuccess) return -1;
    if (cudaEventRecord(t.ev[2 * slot], st) != cudaSuccess) return -1;
    return slot;
}

void timer_end(int kernel, int slot, cudaStream_t st) {
    if (slot < 0) return;
    KernelTimer& t = g_timers[kernel];
    std::lock_guard<std::mutex> lock(g_timer_mu);
    if (cudaEventRecord(t.ev[2 * slot + 1], st) == cudaSuccess) t.timed = slot + 1;
}

// Runs `launch` bracketed by the timer of `kernel` (when enabled).
template <typename F>
cudaError_t timed(int kernel, cudaStream_t st, F&& launch) {
    const int slot = timer_begin(kernel, st);
    const cudaError_t e = launch();
    timer_end(kernel, slot, st);
    return e;
}

// ---- scratch of pka_paged_decode_noalloc: a fixed device array, no allocation
__device__ __align__(256) uint8_t g_noalloc_scratch[PKA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current (host code cannot use the symbol's
// host-side name as a device pointer).
uint8_t* noalloc_scratch() {
    static std::mutex mu;
    static uint8_t* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev] = static_cast<uint8_t*>(p);
    }
    return addr[dev];
}

}  // namespace
}  // namespace pka

using namespace pka;

namespace pka {

__device__ int32_t g_selftest_err;

// One warp waits on an mbarrier that only it can complete (arrive != 0) or
// that nothing completes (arrive == 0: the bounded wait runs out).
__global__ void selftest_wait_kernel(int arrive, uint64_t limit_ns, int32_t* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    __syncwarp();
    const bool ok = mbar_wait_limit(&bar, 0, threadIdx.x == 0 ? err : nullptr, limit_ns);
    __syncwarp();
    (void)__all_sync(0xffffffffu, ok);
}

}  // namespace pka

extern "C" {

const char* pka_status_string(pka_status s) {
    switch (s) {
        case PKA_OK: return "ok";
        case PKA_ERR_INVALID_ARG: return "invalid argument";
        case PKA_ERR_UNSUPPORTED: return "unsupported shape";
        case PKA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case PKA_ERR_CUDA: return "CUDA error";
        case PKA_ERR_DEVICE_METADATA: return "device metadata error";
    }
    return "unknown status";
}

pka_status pka_cache_write(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                           int num_kv_heads, int head_dim, int head_dim_v, void* k_cache, void* v_cache,
                           int64_t num_blocks, int block_size, int32_t* error_word, void* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || block_size <= 0)
        return PKA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKA_OK;
    if (!k || !slot_mapping || !k_cache) return PKA_ERR_INVALID_ARG;
    if ((v == nullptr) != (v_cache == nullptr)) return PKA_ERR_INVALID_ARG;
    if (head_dim % 8 != 0 || (v && (head_dim_v <= 0 || head_dim_v % 8 != 0))) return PKA_ERR_UNSUPPORTED;
    if (!aligned(k, 16) || !aligned(k_cache, 16) || (v && (!aligned(v, 16) || !aligned(v_cache, 16))) ||
        !aligned(slot_mapping, 8))
        return PKA_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return PKA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(timed(PKA_KERNEL_CACHE_WRITE, st, [&] {
        return launch_cache_write(k, v, slot_mapping, num_tokens, num_kv_heads, head_dim, head_dim_v, k_cache,
                                  v_cache, num_blocks, block_size, error_word, sms, st, false, 1.f, 1.f);
    }));
}

pka_status pka_cache_write_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                               int num_kv_heads, int head_dim, int head_dim_v, void* k_cache, void* v_cache,
                               int64_t num_blocks, int block_size, float k_scale, float v_scale, int32_t* error_word,
                               void* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim_v <= 0 || num_blocks <= 0 ||
        block_size <= 0)
        return PKA_ERR_INVALID_ARG;
    if (!std::isfinite(k_scale) || !(k_scale > 0.f) || !std::isfinite(v_scale) || !(v_scale > 0.f))
        return PKA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKA_ERR_INVALID_ARG;
    if (head_dim % 8 != 0 || head_dim_v % 8 != 0 || (head_dim + head_dim_v) / 8 > 128) return PKA_ERR_UNSUPPORTED;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8) || (error_word && !aligned(error_word, 4)))
        return PKA_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return PKA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(timed(PKA_KERNEL_CACHE_WRITE, st, [&] {
        return launch_cache_write(k, v, slot_mapping, num_tokens, num_kv_heads, head_dim, head_dim_v, k_cache,
                                  v_cache, num_blocks, block_size, error_word, sms, st, true, k_scale, v_scale);
    }));
}

static pka_status check_shape(int nd, int ne, int np, int T, int Hq, int Hkv, int d, int dv, int maxq,
                              int maxs, int chunk, bool mla, bool* is_mla) {
    if (nd < 0 || ne < 0 || np < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || maxq <= 0 || maxs <= 0)
        return PKA_ERR_INVALID_ARG;
    const int B = nd + ne + np;
    if (B > kMaxRequests) return PKA_ERR_UNSUPPORTED;
    // every request owns at least one new token (an extend may hold just one:
    // the single-path routing puts decodes there); the planner checks the real lengths
    if ((int64_t)T < (int64_t)nd + ne + np) return PKA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return PKA_ERR_INVALID_ARG;
    if (maxs < maxq) return PKA_ERR_INVALID_ARG;
    if (chunk < 16) return PKA_ERR_INVALID_ARG;
    if (mla) {
        if (!(d == 576 && dv == 512 && Hkv == 1)) return PKA_ERR_UNSUPPORTED;
        if (!(Hq == 16 || Hq == 32 || Hq % 64 == 0)) return PKA_ERR_UNSUPPORTED;
        if (ne + np > 0) return PKA_ERR_UNSUPPORTED;
    } else {
        // (192, 128): the non-absorbed MLA prefill/extend (K = 128 nope + 64 rope
        // dims, V = 128); the split-KV decode has no kernel for it
        const bool nonabsorbed = d == 192 && dv == 128;
        if (!(((d == 64 || d == 128) && dv == d) || nonabsorbed)) return PKA_ERR_UNSUPPORTED;
        if (nonabsorbed && nd > 0) return PKA_ERR_UNSUPPORTED;
        if (Hq / Hkv > 16) return PKA_ERR_UNSUPPORTED;
    }
    *is_mla = mla;
    return PKA_OK;
}

size_t pka_workspace_size(int num_decodes, int num_extends, int num_prefills, int num_tokens, int num_q_heads,
                          int num_kv_heads, int head_dim, int head_dim_v, int max_query_len, int max_seq_len,
                          int context_chunk_tokens) {
    const bool mla = head_dim == 576;
    bool is_mla = false;
    if (check_shape(num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads, head_dim,
                    head_dim_v, max_query_len, max_seq_len, context_chunk_tokens, mla, &is_mla) != PKA_OK)
        return 0;
    const int sms = device_sm_count();
    if (sms <= 0) return 0;
    Hints h{num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads, head_dim,
            head_dim_v, max_query_len, max_seq_len, context_chunk_tokens, is_mla};
    Layout L;
    if (!compute_layout(h, sms, &L)) return 0;
    return L.total;
}

size_t pka_workspace_size_fp8(int num_decodes, int num_extends, int num_prefills, int num_tokens,
                              int num_q_heads, int num_kv_heads, int head_dim, int head_dim_v, int max_query_len,
                              int max_seq_len, int context_chunk_tokens) {
    if (head_dim != 128 || head_dim_v != 128) return 0;  // the 8-bit kernels' head dims
    bool is_mla = false;
    if (check_shape(num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads, head_dim,
                    head_dim_v, max_query_len, max_seq_len, context_chunk_tokens, false, &is_mla) != PKA_OK)
        return 0;
    const int sms = device_sm_count();
    if (sms <= 0) return 0;
    Hints h{num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads, head_dim,
            head_dim_v, max_query_len, max_seq_len, context_chunk_tokens, false};
    h.fp8 = true;
    Layout L;
    if (!compute_layout(h, sms, &L)) return 0;
    return L.total;
}

}  // extern "C"

namespace {

// The cache's element format: bf16, or E4M3 codes with one scale per tensor.
struct CacheFormat {
    bool fp8;
    float k_scale, v_scale;
};

pka_status forward_impl(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                        const void* v_cache, const int32_t* block_table, int max_blocks_per_req,
                        const int32_t* query_start_loc, const int32_t* seq_lens, int num_decodes, int num_extends,
                        int num_prefills, int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                        int head_dim_v, int64_t num_blocks, int block_size, float scale, int context_chunk_tokens,
                        int max_query_len, int max_seq_len, void* out, float* lse, void* workspace,
                        size_t workspace_bytes, void* stream, const CacheFormat& cf,
                        const int64_t* slot_mapping = nullptr, int32_t* cache_error_word = nullptr) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int B = num_decodes + num_extends + num_prefills;
    if (B == 0 && num_tokens == 0) return PKA_OK;
    // ---- host validation: nothing is launched on failure
    const bool mla = v_cache == nullptr;
    bool is_mla = false;
    pka_status sc = check_shape(num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads,
                                head_dim, head_dim_v, max_query_len, max_seq_len, context_chunk_tokens, mla,
                                &is_mla);
    if (sc != PKA_OK) return sc;
    if (cf.fp8) {
        // the 8-bit cache: GQA decode-only batches of head dim 128
        if (is_mla || head_dim != 128 || head_dim_v != 128) return PKA_ERR_UNSUPPORTED;
        if (!std::isfinite(cf.k_scale) || !(cf.k_scale > 0.f) || !std::isfinite(cf.v_scale) || !(cf.v_scale > 0.f))
            return PKA_ERR_INVALID_ARG;
    }
    if (B < 1) return PKA_ERR_INVALID_ARG;
    if (!q || !k_cache || !block_table || !query_start_loc || !seq_lens || !out || !workspace)
        return PKA_ERR_INVALID_ARG;
    if (num_extends + num_prefills > 0 && (!k_new || !v_new)) return PKA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || (v_cache && !aligned(v_cache, 16)) || !aligned(out, 16) ||
        !aligned(workspace, 256) || (k_new && !aligned(k_new, 16)) || (v_new && !aligned(v_new, 16)) ||
        (lse && !aligned(lse, 4)))
        return PKA_ERR_INVALID_ARG;
    if (max_blocks_per_req <= 0 || num_blocks <= 0 || !pow2(block_size) || block_size > 128)
        return block_size > 128 || !pow2(block_size) ? PKA_ERR_UNSUPPORTED : PKA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return PKA_ERR_INVALID_ARG;  // masking and the row max assume scale > 0
    const bool fused_write = slot_mapping != nullptr && num_tokens > 0;
    if (fused_write) {  // the step's own cache write: the new tokens' K/V into their slots
        if (!k_new || (v_cache != nullptr) != (v_new != nullptr)) return PKA_ERR_INVALID_ARG;
        if (!aligned(slot_mapping, 8) || (cache_error_word && !aligned(cache_error_word, 4))) return PKA_ERR_INVALID_ARG;
        if (head_dim % 8 != 0 || head_dim_v % 8 != 0) return PKA_ERR_UNSUPPORTED;
    }
    const int64_t cache_rows = num_blocks * num_kv_heads * (int64_t)block_size;
    if (cache_rows >= (int64_t)INT32_MAX) return PKA_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_req * block_size < max_seq_len) return PKA_ERR_INVALID_ARG;

    const int sms = device_sm_count();
    if (sms <= 0) return PKA_ERR_CUDA;
    Hints h{num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads, head_dim, head_dim_v,
            max_query_len, max_seq_len, context_chunk_tokens, is_mla};
    h.fp8 = cf.fp8;
    Layout L;
    if (!compute_layout(h, sms, &L)) return PKA_ERR_UNSUPPORTED;
    if (workspace_bytes < L.total) return PKA_ERR_WORKSPACE_TOO_SMALL;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
    cudaError_t e = cudaSuccess;  // (the planner clears the header's error word itself)

    // ---- plan
    PlanParams pp;
    pp.qsl = query_start_loc;
    pp.seq_lens = seq_lens;
    pp.num_decodes = num_decodes;
    pp.num_extends = num_extends;
    pp.num_prefills = num_prefills;
    pp.num_tokens = num_tokens;
    pp.max_query_len = max_query_len;
    pp.max_seq_len = max_seq_len;
    pp.max_blocks_per_req = max_blocks_per_req;
    pp.block_size = block_size;
    pp.chunk = context_chunk_tokens;
    pp.dec_units_per_pair = is_mla ? mla_units_per_pair(num_q_heads) : num_kv_heads;
    pp.dec_target_units = L.dec_target_units;
    pp.dec_min_split = is_mla ? kMlaMinSplit : kDecodeMinSplit;
    // the tensor-core MLA kernel reads 64-key tiles whose TMA boxes must start on block rows
    pp.dec_split_align = (is_mla && decode_mla_tc_supported(num_q_heads)) ? 64 : 16;
    pp.dec_pair_cap = L.dec_pair_cap;
    pp.fa_item_cap = L.fa_item_cap;
    pp.ext_row_cap = L.ext_row_cap;
    pp.hdr = hdr;
    pp.dec_pairs = reinterpret_cast<int2*>(ws + L.off_dec_pairs);
    pp.dec_first = reinterpret_cast<int32_t*>(ws + L.off_dec_first);
    pp.dec_nsplit = reinterpret_cast<int32_t*>(ws + L.off_dec_nsplit);
    pp.fa_items = reinterpret_cast<int4*>(ws + L.off_fa_items);
    pp.ext_base = reinterpret_cast<int32_t*>(ws + L.off_ext_base);
    pp.after_cache_write = fused_write ? 1 : 0;
    if (fused_write) {
        // launched first; the planner, which reads no cache, overlaps it and
        // waits for it before the kernels that read the cache may start
        if ((e = timed(PKA_KERNEL_CACHE_WRITE, st, [&] {
                 return launch_cache_write(k_new, v_new, slot_mapping, num_tokens, num_kv_heads, head_dim,
                                           is_mla ? 0 : head_dim_v, const_cast<void*>(k_cache),
                                           const_cast<void*>(v_cache), num_blocks, block_size, cache_error_word, sms,
                                           st, cf.fp8, cf.k_scale, cf.v_scale);
             })) != cudaSuccess)
            return PKA_ERR_CUDA;
    }
    if ((e = timed(PKA_KERNEL_PLANNER, st, [&] { return launch_planner(pp, st); })) != cudaSuccess)
        return PKA_ERR_CUDA;

    // ---- 8-bit cache with extends: gather their context as bf16 code values
    // (after the planner, which clears the error word this kernel may set)
    const bool gathered = cf.fp8 && num_extends > 0;
    CtxDequantParams cd;
    std::memset(&cd, 0, sizeof(cd));
    if (gathered) {
        cd.k8 = static_cast<const uint8_t*>(k_cache);
        cd.v8 = static_cast<const uint8_t*>(v_cache);
        cd.block_table = block_table;
        cd.qsl = query_start_loc;
        cd.seq_lens = seq_lens;
        cd.kc = reinterpret_cast<__nv_bfloat16*>(ws + L.off_ctx_k);
        cd.vc = reinterpret_cast<__nv_bfloat16*>(ws + L.off_ctx_v);
        cd.bt_c = reinterpret_cast<int32_t*>(ws + L.off_ctx_bt);
        cd.err = &hdr->err;
        cd.num_blocks = num_blocks;
        cd.max_blocks = max_blocks_per_req;
        cd.num_decodes = num_decodes;
        cd.num_extends = num_extends;
        cd.Hkv = num_kv_heads;
        cd.bs = block_size;
        cd.d = head_dim;
        cd.dv = head_dim_v;
        cd.nblk = L.ctx_nblk;
        if ((e = timed(PKA_KERNEL_CTX_DEQUANT, st, [&] { return launch_ctx_dequant(cd, st); })) != cudaSuccess)
            return PKA_ERR_CUDA;
    }

    const float scale_log2 = scale * 1.4426950408889634f;
    auto* outb = static_cast<__nv_bfloat16*>(out);
    float* dec_po = reinterpret_cast<float*>(ws + L.off_dec_part_o);
    float* dec_pl = reinterpret_cast<float*>(ws + L.off_dec_part_lse);

    // ---- decode slice
    if (num_decodes > 0) {
        const bool tma = block_size >= 8;
        if (is_mla) {
            const bool tc = decode_mla_tc_supported(num_q_heads);
            CUtensorMap map, qmap, gmap;
            std::memset(&map, 0, sizeof(map));
            std::memset(&qmap, 0, sizeof(qmap));
            std::memset(&gmap, 0, sizeof(gmap));
            if (tma && !encode_rows(&map, k_cache, (uint64_t)cache_rows, 576,
                                    (uint32_t)std::min(block_size, tc ? 64 : 16)))
                return PKA_ERR_CUDA;
            if (tc && !encode_heads(&qmap, q, (uint64_t)num_tokens, (uint64_t)num_q_heads, 576, 128))
                return PKA_ERR_CUDA;
            // one-row boxes for the tensor-core kernel's row gathers
            if (tc && !encode_rows(&gmap, k_cache, (uint64_t)cache_rows, 576, 1)) return PKA_ERR_CUDA;
            DecodeMlaParams dp;
            dp.q = static_cast<const __nv_bfloat16*>(q);
            dp.kv = static_cast<const __nv_bfloat16*>(k_cache);
            dp.block_table = block_table;
            dp.seq_lens = seq_lens;
            dp.hdr = hdr;
            dp.counter = &hdr->dec_counter;
            dp.err = &hdr->err;
            dp.pairs = pp.dec_pairs;
            dp.nsplit = pp.dec_nsplit;
            dp.part_o = dec_po;
            dp.part_lse = dec_pl;
            dp.out = outb;
            dp.lse = lse;
            dp.num_blocks = num_blocks;
            dp.max_blocks = max_blocks_per_req;
            dp.Hq = num_q_heads;
            dp.bs = block_size;
            dp.groups = tc ? num_q_heads / 128 : num_q_heads / decode_mla_heads_per_cta(num_q_heads);
            dp.cache_rows = (int)cache_rows;
            dp.scale_log2 = scale_log2;
            if ((e = timed(PKA_KERNEL_DECODE, st, [&] {
                     return tc ? launch_decode_mla_tc(map, qmap, gmap, dp, sms, st)
                               : launch_decode_mla(map, dp, tma, sms, st);
                 })) != cudaSuccess)
                return PKA_ERR_CUDA;
        } else {
            CUtensorMap km, vm;
            std::memset(&km, 0, sizeof(km));
            std::memset(&vm, 0, sizeof(vm));
            if (tma) {
                const uint32_t br = (uint32_t)std::min(block_size, 16);
                const bool ok = cf.fp8 ? (encode_rows_u8(&km, k_cache, (uint64_t)cache_rows, br) &&
                                          encode_rows_u8(&vm, v_cache, (uint64_t)cache_rows, br))
                                       : (encode_rows(&km, k_cache, (uint64_t)cache_rows, head_dim, br) &&
                                          encode_rows(&vm, v_cache, (uint64_t)cache_rows, head_dim, br));
                if (!ok) return PKA_ERR_CUDA;
            }
            DecodeGqaParams dp;
            dp.q = static_cast<const __nv_bfloat16*>(q);
            dp.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
            dp.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
            dp.k8 = static_cast<const uint8_t*>(k_cache);
            dp.v8 = static_cast<const uint8_t*>(v_cache);
            dp.v_scale = cf.fp8 ? cf.v_scale : 1.f;
            dp.block_table = block_table;
            dp.seq_lens = seq_lens;
            dp.hdr = hdr;
            dp.counter = &hdr->dec_counter;
            dp.err = &hdr->err;
            dp.pairs = pp.dec_pairs;
            dp.nsplit = pp.dec_nsplit;
            dp.part_o = dec_po;
            dp.part_lse = dec_pl;
            dp.out = outb;
            dp.lse = lse;
            dp.num_blocks = num_blocks;
            dp.max_blocks = max_blocks_per_req;
            dp.Hq = num_q_heads;
            dp.Hkv = num_kv_heads;
            dp.G = num_q_heads / num_kv_heads;
            dp.bs = block_size;
            // 8-bit cache: a score is scale * k_scale * <q, code>
            dp.scale_log2 = cf.fp8 ? scale_log2 * cf.k_scale : scale_log2;
            if ((e = timed(PKA_KERNEL_DECODE, st, [&] {
                     return cf.fp8 ? launch_decode_gqa_fp8(km, vm, dp, tma, sms, st)
                                   : launch_decode_gqa(km, vm, dp, head_dim, tma, sms, st);
                 })) != cudaSuccess)
                return PKA_ERR_CUDA;
        }
        DecodeReduceParams rp;
        rp.hdr = hdr;
        rp.dec_first = pp.dec_first;
        rp.dec_nsplit = pp.dec_nsplit;
        rp.part_o = dec_po;
        rp.part_lse = dec_pl;
        rp.out = outb;
        rp.lse = lse;
        rp.num_decodes = num_decodes;
        rp.Hq = num_q_heads;
        rp.dv = head_dim_v;
        if ((e = timed(PKA_KERNEL_DECODE_REDUCE, st, [&] { return launch_decode_reduce(rp, sms, st); })) !=
            cudaSuccess)
            return PKA_ERR_CUDA;
    }

    // ---- prefill + extend slices
    if (num_extends + num_prefills > 0) {
        FaParams fp;
        fp.q = static_cast<const __nv_bfloat16*>(q);
        fp.k_new = static_cast<const __nv_bfloat16*>(k_new);
        fp.v_new = static_cast<const __nv_bfloat16*>(v_new);
        // context chunks: the cache itself, or the gathered bf16 copy of an 8-bit cache
        const void* kc = gathered ? static_cast<const void*>(cd.kc) : k_cache;
        const void* vc = gathered ? static_cast<const void*>(cd.vc) : v_cache;
        const int ctx_bs = gathered ? kCtxRows : block_size;
        const int64_t ctx_blocks = gathered ? (int64_t)num_extends * L.ctx_nblk : num_blocks;
        fp.k_cache = static_cast<const __nv_bfloat16*>(kc);
        fp.v_cache = static_cast<const __nv_bfloat16*>(vc);
        fp.block_table = gathered ? cd.bt_c : block_table;
        fp.bt_row0 = gathered ? num_decodes : 0;
        fp.qsl = query_start_loc;
        fp.seq_lens = seq_lens;
        fp.hdr = hdr;
        fp.counter = &hdr->fa_counter;
        fp.err = &hdr->err;
        fp.items = pp.fa_items;
        fp.ext_base = pp.ext_base;
        fp.ext_o = reinterpret_cast<float*>(ws + L.off_ext_part_o);
        fp.ext_lse = reinterpret_cast<float*>(ws + L.off_ext_part_lse);
        fp.out = outb;
        fp.out_v8 = aligned(outb, 32) ? 1 : 0;
        fp.lse = lse;
        fp.num_blocks = ctx_blocks;
        fp.max_blocks = gathered ? L.ctx_nblk : max_blocks_per_req;
        fp.Hq = num_q_heads;
        fp.Hkv = num_kv_heads;
        fp.G = num_q_heads / num_kv_heads;
        fp.bs = ctx_bs;
        fp.chunk = context_chunk_tokens;
        fp.num_decodes = num_decodes;
        fp.num_extends = num_extends;
        fp.scale_log2 = scale_log2;
        // an 8-bit cache's scales apply to the context chunks only
        fp.ctx_scale_log2 = cf.fp8 ? scale_log2 * cf.k_scale : scale_log2;
        fp.ctx_v_scale = cf.fp8 ? cf.v_scale : 1.f;
        FaMaps maps;
        std::memset(&maps, 0, sizeof(maps));
        if (!encode_tokens(&maps.q, q, (uint64_t)num_tokens, num_q_heads, head_dim) ||
            !encode_tokens(&maps.knew, k_new, (uint64_t)num_tokens, num_kv_heads, head_dim) ||
            !encode_tokens(&maps.vnew, v_new, (uint64_t)num_tokens, num_kv_heads, head_dim_v))
            return PKA_ERR_CUDA;
        if (ctx_bs >= 8) {
            const uint32_t br = (uint32_t)std::min(ctx_bs, 128);
            const uint64_t rows = (uint64_t)ctx_blocks * num_kv_heads * ctx_bs;
            if (!encode_rows(&maps.kc, kc, rows, head_dim, br) || !encode_rows(&maps.vc, vc, rows, head_dim_v, br))
                return PKA_ERR_CUDA;
        }
        if ((e = timed(PKA_KERNEL_PREFILL_EXTEND, st,
                       [&] { return launch_fa_fwd(maps, fp, head_dim, head_dim_v, sms, st); })) != cudaSuccess)
            return PKA_ERR_CUDA;
        if (num_extends > 0) {
            ExtendReduceParams xp;
            xp.hdr = hdr;
            xp.qsl = query_start_loc;
            xp.seq_lens = seq_lens;
            xp.ext_base = pp.ext_base;
            xp.part_o = fp.ext_o;
            xp.part_lse = fp.ext_lse;
            xp.out = outb;
            xp.lse = lse;
            xp.num_decodes = num_decodes;
            xp.num_extends = num_extends;
            xp.Hq = num_q_heads;
            xp.dv = head_dim_v;
            xp.chunk = context_chunk_tokens;
            const int ext_tokens_bound = std::min(num_tokens - num_decodes - num_prefills,
                                                  num_extends * max_query_len);
            if ((e = timed(PKA_KERNEL_EXTEND_REDUCE, st,
                           [&] { return launch_extend_reduce(xp, ext_tokens_bound, sms, st); })) != cudaSuccess)
                return PKA_ERR_CUDA;
        }
    }
    return PKA_OK;
}

}  // namespace

extern "C" {

pka_status pka_paged_attn_forward(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                                  const void* v_cache, const int32_t* block_table, int max_blocks_per_req,
                                  const int32_t* query_start_loc, const int32_t* seq_lens, int num_decodes,
                                  int num_extends, int num_prefills, int num_tokens, int num_q_heads,
                                  int num_kv_heads, int head_dim, int head_dim_v, int64_t num_blocks,
                                  int block_size, float scale, int context_chunk_tokens, int max_query_len,
                                  int max_seq_len, void* out, float* lse, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    return forward_impl(q, k_new, v_new, k_cache, v_cache, block_table, max_blocks_per_req, query_start_loc,
                        seq_lens, num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads,
                        head_dim, head_dim_v, num_blocks, block_size, scale, context_chunk_tokens, max_query_len,
                        max_seq_len, out, lse, workspace, workspace_bytes, stream, CacheFormat{false, 1.f, 1.f});
}

pka_status pka_paged_attn_forward_fp8(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                                      const void* v_cache, const int32_t* block_table, int max_blocks_per_req,
                                      const int32_t* query_start_loc, const int32_t* seq_lens, int num_decodes,
                                      int num_extends, int num_prefills, int num_tokens, int num_q_heads,
                                      int num_kv_heads, int head_dim, int head_dim_v, int64_t num_blocks,
                                      int block_size, float scale, float k_scale, float v_scale,
                                      int context_chunk_tokens, int max_query_len, int max_seq_len, void* out,
                                      float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    return forward_impl(q, k_new, v_new, k_cache, v_cache, block_table, max_blocks_per_req, query_start_loc,
                        seq_lens, num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads,
                        head_dim, head_dim_v, num_blocks, block_size, scale, context_chunk_tokens, max_query_len,
                        max_seq_len, out, lse, workspace, workspace_bytes, stream,
                        CacheFormat{true, k_scale, v_scale});
}

pka_status pka_paged_attn_step(const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                               void* k_cache, void* v_cache, const int32_t* block_table, int max_blocks_per_req,
                               const int32_t* query_start_loc, const int32_t* seq_lens, int num_decodes,
                               int num_extends, int num_prefills, int num_tokens, int num_q_heads, int num_kv_heads,
                               int head_dim, int head_dim_v, int64_t num_blocks, int block_size, float scale,
                               int context_chunk_tokens, int max_query_len, int max_seq_len, void* out, float* lse,
                               int32_t* cache_error_word, void* workspace, size_t workspace_bytes, void* stream) {
    if (!slot_mapping) return PKA_ERR_INVALID_ARG;
    return forward_impl(q, k_new, v_new, k_cache, v_cache, block_table, max_blocks_per_req, query_start_loc,
                        seq_lens, num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads,
                        head_dim, head_dim_v, num_blocks, block_size, scale, context_chunk_tokens, max_query_len,
                        max_seq_len, out, lse, workspace, workspace_bytes, stream, CacheFormat{false, 1.f, 1.f},
                        slot_mapping, cache_error_word);
}

pka_status pka_paged_attn_step_fp8(const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                   void* k_cache, void* v_cache, const int32_t* block_table, int max_blocks_per_req,
                                   const int32_t* query_start_loc, const int32_t* seq_lens, int num_decodes,
                                   int num_extends, int num_prefills, int num_tokens, int num_q_heads,
                                   int num_kv_heads, int head_dim, int head_dim_v, int64_t num_blocks,
                                   int block_size, float scale, float k_scale, float v_scale,
                                   int context_chunk_tokens, int max_query_len, int max_seq_len, void* out,
                                   float* lse, int32_t* cache_error_word, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    if (!slot_mapping) return PKA_ERR_INVALID_ARG;
    return forward_impl(q, k_new, v_new, k_cache, v_cache, block_table, max_blocks_per_req, query_start_loc,
                        seq_lens, num_decodes, num_extends, num_prefills, num_tokens, num_q_heads, num_kv_heads,
                        head_dim, head_dim_v, num_blocks, block_size, scale, context_chunk_tokens, max_query_len,
                        max_seq_len, out, lse, workspace, workspace_bytes, stream, CacheFormat{true, k_scale, v_scale},
                        slot_mapping, cache_error_word);
}

pka_status pka_merge_attn_states(void* out, float* out_lse, const void* prefix_out, const float* prefix_lse,
                                 const void* suffix_out, const float* suffix_lse, int64_t num_rows, int head_dim,
                                 int io_dtype, void* stream) {
    if (num_rows < 0 || head_dim <= 0 || (io_dtype != 0 && io_dtype != 1)) return PKA_ERR_INVALID_ARG;
    if (num_rows == 0) return PKA_OK;
    if (!out || !prefix_out || !prefix_lse || !suffix_out || !suffix_lse) return PKA_ERR_INVALID_ARG;
    if (head_dim % (io_dtype ? 8 : 4) != 0) return PKA_ERR_UNSUPPORTED;
    if (!aligned(out, 16) || !aligned(prefix_out, 16) || !aligned(suffix_out, 16) || !aligned(prefix_lse, 4) ||
        !aligned(suffix_lse, 4) || (out_lse && !aligned(out_lse, 4)))
        return PKA_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return PKA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(timed(PKA_KERNEL_MERGE, st, [&] {
        return launch_merge_pair(out, out_lse, prefix_out, prefix_lse, suffix_out, suffix_lse, num_rows, head_dim,
                                 io_dtype, sms, st);
    }));
}

pka_status pka_gather_rows(void* dst, const void* src, const int32_t* index, int64_t num_rows, int64_t src_rows,
                           int64_t row_bytes, int32_t* error_word, void* stream) {
    if (!dst || !src || !index || num_rows < 0 || src_rows < 0 || row_bytes < 1) return PKA_ERR_INVALID_ARG;
    if (num_rows > INT64_MAX / row_bytes || src_rows > INT64_MAX / row_bytes) return PKA_ERR_INVALID_ARG;
    if (error_word && !aligned(error_word, 4)) return PKA_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return PKA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(timed(PKA_KERNEL_GATHER, st, [&] {
        return launch_gather_rows(dst, src, index, num_rows, src_rows, row_bytes, error_word, sms, st);
    }));
}

pka_status pka_paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_table, int max_blocks_per_req,
                                    const int32_t* query_start_loc, const int32_t* seq_lens, int num_decodes,
                                    int num_q_heads, int num_kv_heads, int head_dim, int64_t num_blocks,
                                    int block_size, float scale, int max_seq_len, void* out, float* lse,
                                    int32_t* error_word, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (num_decodes < 1) return num_decodes == 0 ? PKA_OK : PKA_ERR_INVALID_ARG;
    bool is_mla = false;
    pka_status sc = check_shape(num_decodes, 0, 0, num_decodes, num_q_heads, num_kv_heads, head_dim, head_dim,
                                1, max_seq_len, 16, false, &is_mla);
    if (sc != PKA_OK) return sc;
    if (!q || !k_cache || !v_cache || !block_table || !query_start_loc || !seq_lens || !out)
        return PKA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        (lse && !aligned(lse, 4)) || (error_word && !aligned(error_word, 4)))
        return PKA_ERR_INVALID_ARG;
    if (max_blocks_per_req <= 0 || num_blocks <= 0 || !pow2(block_size) || block_size > 128)
        return block_size > 128 || !pow2(block_size) ? PKA_ERR_UNSUPPORTED : PKA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return PKA_ERR_INVALID_ARG;  // masking and the row max assume scale > 0
    const int64_t cache_rows = num_blocks * num_kv_heads * (int64_t)block_size;
    if (cache_rows >= (int64_t)INT32_MAX) return PKA_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks_per_req * block_size < max_seq_len) return PKA_ERR_INVALID_ARG;

    // Scratch layout inside the fixed array: header, pairs, per-request
    // split index, then the split partials. The number of split pairs is
    // capped so everything fits; a batch that cannot fit is rejected.
    const int Hq = num_q_heads, dv = head_dim, nd = num_decodes;
    const size_t per_pair = sizeof(int2) + (size_t)Hq * dv * sizeof(float) + (size_t)Hq * sizeof(float);
    const size_t fixed = sizeof(PlanHeader) + 2 * align256((size_t)nd * sizeof(int32_t)) + 5 * 256;
    if (fixed >= PKA_NOALLOC_SCRATCH_BYTES) return PKA_ERR_WORKSPACE_TOO_SMALL;
    const int64_t cap = (int64_t)((PKA_NOALLOC_SCRATCH_BYTES - fixed) / per_pair);
    if (cap < (int64_t)nd + 2) return PKA_ERR_WORKSPACE_TOO_SMALL;
    const int sms = device_sm_count();
    if (sms <= 0) return PKA_ERR_CUDA;
    int64_t target = std::min<int64_t>(decode_gqa_target_units(sms), (cap - nd - 1) * (int64_t)num_kv_heads);
    if (target < num_kv_heads) return PKA_ERR_WORKSPACE_TOO_SMALL;
    const int pair_cap = (int)(target / num_kv_heads + nd + 1);
    size_t off = sizeof(PlanHeader);
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align256(off + bytes);
        return o;
    };
    const size_t off_pairs = take(sizeof(int2) * (size_t)pair_cap);
    const size_t off_first = take(sizeof(int32_t) * (size_t)nd);
    const size_t off_nsplit = take(sizeof(int32_t) * (size_t)nd);
    const size_t off_po = take(sizeof(float) * (size_t)pair_cap * Hq * dv);
    const size_t off_pl = take(sizeof(float) * (size_t)pair_cap * Hq);
    if (off > PKA_NOALLOC_SCRATCH_BYTES) return PKA_ERR_WORKSPACE_TOO_SMALL;

    uint8_t* ws = noalloc_scratch();
    if (!ws) return PKA_ERR_CUDA;
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
    // the header (error word, counters) must start at zero on every call
    if (cudaMemsetAsync(hdr, 0, sizeof(PlanHeader), st) != cudaSuccess) return PKA_ERR_CUDA;

    PlanParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.qsl = query_start_loc;
    pp.seq_lens = seq_lens;
    pp.num_decodes = nd;
    pp.num_tokens = nd;
    pp.max_query_len = 1;
    pp.max_seq_len = max_seq_len;
    pp.max_blocks_per_req = max_blocks_per_req;
    pp.block_size = block_size;
    pp.chunk = 16;
    pp.dec_units_per_pair = num_kv_heads;
    pp.dec_target_units = (int)target;
    pp.dec_min_split = kDecodeMinSplit;
    // the tensor-core MLA kernel reads 64-key tiles whose TMA boxes must start on block rows
    pp.dec_split_align = (is_mla && decode_mla_tc_supported(num_q_heads)) ? 64 : 16;
    pp.dec_pair_cap = pair_cap;
    pp.hdr = hdr;
    pp.dec_pairs = reinterpret_cast<int2*>(ws + off_pairs);
    pp.dec_first = reinterpret_cast<int32_t*>(ws + off_first);
    pp.dec_nsplit = reinterpret_cast<int32_t*>(ws + off_nsplit);
    if (launch_planner(pp, st) != cudaSuccess) return PKA_ERR_CUDA;

    const bool tma = block_size >= 8;
    CUtensorMap km, vm;
    std::memset(&km, 0, sizeof(km));
    std::memset(&vm, 0, sizeof(vm));
    if (tma) {
        const uint32_t br = (uint32_t)std::min(block_size, 16);
        if (!encode_rows(&km, k_cache, (uint64_t)cache_rows, head_dim, br) ||
            !encode_rows(&vm, v_cache, (uint64_t)cache_rows, head_dim, br))
            return PKA_ERR_CUDA;
    }
    auto* outb = static_cast<__nv_bfloat16*>(out);
    float* po = reinterpret_cast<float*>(ws + off_po);
    float* pl = reinterpret_cast<float*>(ws + off_pl);
    DecodeGqaParams dp;
    dp.q = static_cast<const __nv_bfloat16*>(q);
    dp.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
    dp.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
    dp.k8 = nullptr;
    dp.v8 = nullptr;
    dp.v_scale = 1.f;
    dp.block_table = block_table;
    dp.seq_lens = seq_lens;
    dp.hdr = hdr;
    dp.counter = &hdr->dec_counter;
    dp.err = &hdr->err;
    dp.pairs = pp.dec_pairs;
    dp.nsplit = pp.dec_nsplit;
    dp.part_o = po;
    dp.part_lse = pl;
    dp.out = outb;
    dp.lse = lse;
    dp.num_blocks = num_blocks;
    dp.max_blocks = max_blocks_per_req;
    dp.Hq = Hq;
    dp.Hkv = num_kv_heads;
    dp.G = Hq / num_kv_heads;
    dp.bs = block_size;
    dp.scale_log2 = scale * 1.4426950408889634f;
    if (launch_decode_gqa(km, vm, dp, head_dim, tma, sms, st) != cudaSuccess) return PKA_ERR_CUDA;
    DecodeReduceParams rp;
    rp.hdr = hdr;
    rp.dec_first = pp.dec_first;
    rp.dec_nsplit = pp.dec_nsplit;
    rp.part_o = po;
    rp.part_lse = pl;
    rp.out = outb;
    rp.lse = lse;
    rp.num_decodes = nd;
    rp.Hq = Hq;
    rp.dv = dv;
    if (launch_decode_reduce(rp, sms, st) != cudaSuccess) return PKA_ERR_CUDA;
    if (error_word &&
        cudaMemcpyAsync(error_word, &hdr->err, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return PKA_ERR_CUDA;
    return PKA_OK;
}

pka_status pka_kernel_timer(int kernel, int enable) {
    if (kernel < 0 || kernel >= PKA_KERNEL_COUNT) return PKA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_timer_mu);
    KernelTimer& t = g_timers[kernel];
    t.on = enable != 0;
    t.launches = 0;
    t.timed = 0;
    return PKA_OK;
}

pka_status pka_kernel_timer_read(int kernel, double* total_ms, int* launches, int* timed_out) {
    if (kernel < 0 || kernel >= PKA_KERNEL_COUNT) return PKA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_timer_mu);
    KernelTimer& t = g_timers[kernel];
    double sum = 0.0;
    for (int i = 0; i < t.timed; ++i) {
        if (cudaEventSynchronize(t.ev[2 * i + 1]) != cudaSuccess) return PKA_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess) return PKA_ERR_CUDA;
        sum += ms;
    }
    if (total_ms) *total_ms = sum;
    if (launches) *launches = t.launches;
    if (timed_out) *timed_out = t.timed;
    return PKA_OK;
}

pka_status pka_selftest_wait(int arrive, uint32_t limit_us, int32_t* code_out, void* stream) {
    if (!code_out || limit_us < 1 || limit_us > 2000000u) return PKA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t* d_err = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d_err), pka::g_selftest_err) != cudaSuccess) return PKA_ERR_CUDA;
    if (cudaMemsetAsync(d_err, 0, sizeof(int32_t), st) != cudaSuccess) return PKA_ERR_CUDA;
    pka::selftest_wait_kernel<<<1, 32, 0, st>>>(arrive, (uint64_t)limit_us * 1000ull, d_err);
    if (cudaGetLastError() != cudaSuccess) return PKA_ERR_CUDA;
    int32_t code = 0;
    if (cudaMemcpyAsync(&code, d_err, sizeof(code), cudaMemcpyDeviceToHost, st) != cudaSuccess) return PKA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PKA_ERR_CUDA;
    *code_out = code;
    return PKA_OK;
}

pka_status pka_get_error(const void* workspace, int32_t* code_out, void* stream) {
    if (!workspace) return PKA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t code = 0;
    if (cudaMemcpyAsync(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return PKA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PKA_ERR_CUDA;
    if (code_out) *code_out = code;
    return code ? PKA_ERR_DEVICE_METADATA : PKA_OK;
}

}  // extern "C"
