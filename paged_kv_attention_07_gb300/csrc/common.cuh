// common.cuh -- device helpers shared by the kernels of libpka.so (sm_103a).
//
// Inline PTX for the pieces the kernels are built from: bounded mbarrier
// waits (the waiting thread sleeps), TMA tile loads, cp.async with mbarrier completion,
// ldmatrix/movmatrix, bf16 tensor-core MMA, and bf16 packing.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pka.h"

#define PKA_DEVICE __device__ __forceinline__

namespace pka {

// A wait on an mbarrier gives up after this many nanoseconds of spinning,
// records PKA_DEVERR_TIMEOUT and lets the kernel finish without touching
// the stage it waited for. Nothing here should ever take a millisecond.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
// Longest single suspension inside an mbarrier wait (the thread wakes as soon
// as the phase completes; this only bounds how late a timeout is noticed).
constexpr uint32_t kSuspendNs = 1000000u;  // 1 ms

PKA_DEVICE uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

PKA_DEVICE uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

PKA_DEVICE void set_error(int32_t* err, int32_t bits) {
    if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------- mbarrier
PKA_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

PKA_DEVICE void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

PKA_DEVICE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

PKA_DEVICE void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Blocking probe: the thread is suspended (it takes no issue slots) until the
// phase completes or about `suspend_ns` pass, whichever comes first.
PKA_DEVICE bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

PKA_DEVICE bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of `bar`. Returns false (and sets the
// timeout bit) if the phase did not complete within kWaitLimitNs.
PKA_DEVICE bool mbar_wait_limit(uint64_t* bar, uint32_t parity, int32_t* err, uint64_t limit_ns) {
    if (mbar_test_wait(bar, parity)) return true;  // non-blocking fast path
    // A waiting thread sleeps inside try_wait instead of spinning: a spinning
    // warp would take issue slots from the warps of the same scheduler that
    // have work (the softmax warps share schedulers with the copy and MMA
    // warps, and with each other).
    const uint64_t t0 = global_timer_ns();
    const uint32_t nap = limit_ns < kSuspendNs ? (uint32_t)limit_ns : kSuspendNs;
    for (;;) {
        if (mbar_try_wait(bar, parity, nap)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            set_error(err, PKA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

PKA_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err) {
    return mbar_wait_limit(bar, parity, err, kWaitLimitNs);
}

// Bounded wait until a monotonic shared-memory counter reaches `target`
// (written by another thread of the CTA). Returns false (and sets the
// timeout bit) if it did not within kWaitLimitNs.
PKA_DEVICE bool wait_counter(const volatile int& counter, int target, int32_t* err) {
    if (counter >= target) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (counter >= target) return true;
        if ((i & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
            set_error(err, PKA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Full-warp forms: every lane of the warp gets the same answer, so a timeout
// or an abort can never split a warp at a later warp-synchronous point
// (__syncwarp, shuffles, .sync.aligned instructions). Call with all 32 lanes.
PKA_DEVICE bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int32_t* err) {
    const bool ok = mbar_wait(bar, parity, err);
    return __all_sync(0xffffffffu, ok);
}
PKA_DEVICE bool warp_flag(const volatile int& flag) { return __any_sync(0xffffffffu, flag != 0); }

// Generic-proxy accesses to shared memory made before this fence are ordered
// before later async-proxy (TMA / tensor core) accesses.
PKA_DEVICE void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
PKA_DEVICE void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tile load: box at (x = c0 elements, y = c1 rows) into smem, completion
// counted in bytes on `bar`.
PKA_DEVICE void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

PKA_DEVICE void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                            int c2, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
        "l"(policy)
        : "memory");
}

// Four rows of a 2-D map gathered into consecutive 128-byte rows of shared
// memory: rows r0..r3 (any order, any rows; an out-of-range row reads the
// fill value, zeros), columns [c0, c0 + box width). The map's box is one row
// high (the gather form's requirement).
PKA_DEVICE void tma_gather4(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int r0, int r1, int r2,
                            int r3) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
        : "memory");
}

// L2 prefetch of a tile (no shared memory, no completion tracking).
PKA_DEVICE void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// L2 prefetch of `bytes` (a multiple of 16) from a 16-byte aligned address.
PKA_DEVICE void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
                 : "memory");
}

PKA_DEVICE void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

PKA_DEVICE uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

PKA_DEVICE uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

PKA_DEVICE uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- cp.async
PKA_DEVICE void cp_async_16(uint32_t smem_addr, const void* gptr) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr), "l"(gptr) : "memory");
}

// 16-byte copy that writes zeros instead when `valid` is false.
PKA_DEVICE void cp_async_16_zfill(uint32_t smem_addr, const void* gptr, bool valid) {
    const uint32_t n = valid ? 16u : 0u;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr), "l"(gptr), "r"(n)
                 : "memory");
}

// Arrive on `bar` once all of this thread's earlier cp.async copies land
// (does not add to the expected count: the barrier counts one per thread).
PKA_DEVICE void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

PKA_DEVICE void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
PKA_DEVICE void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- warp MMA
PKA_DEVICE void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

PKA_DEVICE void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

PKA_DEVICE void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

PKA_DEVICE void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// Transpose an 8x8 b16 matrix held in the m8n8 fragment layout.
PKA_DEVICE uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
PKA_DEVICE void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> bf16x2 (round to nearest even); `lo` lands in the low half.
// Two E4M3 codes (low byte -> low half) to an f16 pair; exact (every E4M3
// value is an f16 value).
PKA_DEVICE uint32_t e4m3x2_to_f16x2(uint32_t x16) {
    uint32_t d;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(d) : "r"(x16));
    return d;
}

PKA_DEVICE uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

PKA_DEVICE float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
PKA_DEVICE float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// One 32-byte global store (sm_100 and later); p must be 32-byte aligned.
PKA_DEVICE void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4, uint32_t a5,
                             uint32_t a6, uint32_t a7) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2),
                 "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}

// max(a, b, c) in one instruction (three-input max, sm_100 and later).
PKA_DEVICE float fmax3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (d0, d1) = (a0 * b + c, a1 * b + c): one packed fp32 FMA, each lane rounded
// like fmaf.
PKA_DEVICE void fma2_bcast(float& d0, float& d1, float a0, float a1, float b, float c) {
    asm("{\n\t.reg .b64 x, y, z, w;\n\t"
        "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\tmov.b64 z, {%5, %5};\n\t"
        "fma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (s0, s1) += (a0, a1): one packed fp32 add.
PKA_DEVICE void add2(float& s0, float& s1, float a0, float a1) {
    asm("{\n\t.reg .b64 x, y;\n\t"
        "mov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
        "add.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "f"(a0), "f"(a1));
}

PKA_DEVICE float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- register split
// A warpgroup's register budget changes by role: every warp of the warpgroup
// executes the same instruction; increases draw on what decreases released
// from the block's launch allocation.
template <int kRegs>
PKA_DEVICE void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <int kRegs>
PKA_DEVICE void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// ---------------------------------------------------------------- dependent launches
// The forward pass is a chain of kernels on one stream. Each kernel after the
// planner is launched as a programmatic dependent (launch_dependent below):
// it may start while its predecessor still runs, and waits here, before it
// touches anything, until the predecessor has completed and its writes are
// visible. Every such kernel calls this first, so each completion implies its
// predecessors' too.
PKA_DEVICE void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream start launching (its grid_dep_wait still
// waits for this whole grid to finish).
PKA_DEVICE void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Byte offset of 16-byte chunk `c` (0..7) of 128-byte row `row` inside a
// tile written with the 128-byte swizzle (TMA CU_TENSOR_MAP_SWIZZLE_128B
// with a 1024-byte aligned base): chunks are XOR-ed with row % 8.
PKA_DEVICE uint32_t sw128(uint32_t row, uint32_t c) { return row * 128u + ((c ^ (row & 7u)) << 4); }

#ifdef __CUDACC__
// Launch `kern` as a programmatic dependent of the previous work on `stream`
// (see grid_dep_wait: the kernel must call it before reading its inputs).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                    Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
#endif

}  // namespace pka
