// Device helpers shared by the kernels: mbarrier + bulk-copy staging,
// ldmatrix / mma.sync fragments, bf16 splitting, bounded waits.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"

namespace pkv {

// ---------------------------------------------------------------- smem / mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Longest time any spin-wait of the library waits before it gives up.
constexpr uint64_t WAIT_NS = 1000000000ull;

// Wait for phase `parity` of `bar` to complete, giving up after `limit_ns`
// of polling (each try_wait itself suspends for a short while).  On give-up
// the device status word records a timeout and false is returned.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int *status,
                                                  uint64_t limit_ns = WAIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i >= 64) {
            __nanosleep(64);
            if ((i & 63) == 0 && global_ns() - t0 > limit_ns) break;
        }
    }
    if (status) atomicOr(status + STATUS_TIMEOUT, 1);
    return false;
}

// One contiguous global -> shared bulk copy (TMA bulk engine), completion
// signalled as transaction bytes on `bar`.  Addresses 16-byte aligned, bytes
// a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same copy with an L2 eviction-priority policy (see l2_evict_first).
__device__ __forceinline__ void bulk_g2s_hint(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 policy for bytes read exactly once: first in line for eviction.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Ask L2 to fetch `bytes` (multiple of 16) at a 16-byte aligned global
// address; no completion is tracked and nothing is written to the SM.
__device__ __forceinline__ void prefetch_l2(const void *src_gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

// Order this thread's earlier generic-proxy accesses to global memory
// before its later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Atomic add with release and acquire semantics at GPU scope: writes that
// happen before it (a CTA barrier included) are visible to whoever later
// acquires the location, and writes released to the location before it are
// visible after it.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Order this thread's earlier generic-proxy accesses to shared memory before
// its later async-proxy (bulk copy) writes there.
__device__ __forceinline__ void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its memory is visible / let the next grid start early.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- tensor-core fragments

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x1(uint32_t addr, uint32_t &r0) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x1.shared.b16 {%0}, [%1];" : "=r"(r0) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A (16x16 bf16, row) * B (16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma16816(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A (16x8 bf16, row) * B (8x8 bf16, col) + D.
__device__ __forceinline__ void mma1688(float *d, uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

// The same two shapes with fp16 operands (fp32 accumulate).
__device__ __forceinline__ void mma16816_f16(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma1688_f16(float *d, uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

// Pack two floats into fp16x2 (round to nearest even); `lo` goes to the low half.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Pack two floats into bf16x2 (round to nearest even); `lo` goes to the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float bf16_lo_to_f32(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Split a pair of fp32 values into bf16 high parts and bf16 residuals, so that
// x ~= hi + lo to about 2^-16 relative: the high parts feed rows 0-7 and the
// residuals rows 8-15 of one m16 tile, and the two result rows are summed.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - bf16_lo_to_f32(hi), x1 - bf16_hi_to_f32(hi));
}

// fp16 counterpart of split_bf16 (about 22 bits carried by hi + lo).
__device__ __forceinline__ void split_f16(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack_f16(x0, x1);
    const float2 h = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
    lo = pack_f16(x0 - h.x, x1 - h.y);
}

// INT4 codes -> fp16x2 tensor-core operands.  An fp16 with biased exponent
// 25 (bit pattern 0x6400 = 1024) has a unit-spaced mantissa, so OR-ing a
// nibble n into mantissa bits 0-3 gives exactly 1024 + n and into bits 4-7
// exactly 1024 + 16 n; subtracting 1032, or multiplying by 1/16 and adding
// -72, leaves the code n - 8 exactly.  Each form converts two nibbles, one per
// 16-bit half of the word.
__device__ __forceinline__ uint32_t q4_pair_lo(uint32_t x) {  // nibbles at bits 0-3 and 16-19
    const uint32_t t = (x & 0x000F000Fu) | 0x64006400u, bias = 0x64086408u;  // 1032, 1032
    uint32_t h;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(t), "r"(bias));
    return h;
}
__device__ __forceinline__ uint32_t q4_pair_hi(uint32_t x) {  // nibbles at bits 4-7 and 20-23
    const uint32_t t = (x & 0x00F000F0u) | 0x64006400u, k = 0x2C002C00u, b = 0xD480D480u;  // 1/16, -72
    uint32_t h;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(h) : "r"(t), "r"(k), "r"(b));
    return h;
}
// Register r (0..3) of a word of an INT4 operand stream: nibbles r and r + 4.
__device__ __forceinline__ uint32_t q4_reg(uint32_t w, int r) {
    const uint32_t x = w >> ((r & 2) << 2);
    return (r & 1) ? q4_pair_hi(x) : q4_pair_lo(x);
}

// a * b as an fp16x2 high part and its exact residual (the fused multiply-add
// of a, b and -hi; exact unless the residual is subnormal).
__device__ __forceinline__ void mul_split_f16(uint32_t a, uint32_t b, uint32_t &hi, uint32_t &lo) {
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(a), "r"(b));
    const uint32_t nhi = hi ^ 0x80008000u;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(a), "r"(b), "r"(nhi));
}

// Operand traits of the tensor-core path: bf16 (stored factors and dense
// rows) or fp16 (INT4 codes, exact in fp16, against fp16 split operands).
template <bool H16>
struct Ops;
template <>
struct Ops<false> {
    static __device__ __forceinline__ void mma(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
        mma16816(d, a0, a1, a2, a3, b0, b1);
    }
    static __device__ __forceinline__ void mma8(float *d, uint32_t a0, uint32_t a1, uint32_t b0) {
        mma1688(d, a0, a1, b0);
    }
    static __device__ __forceinline__ void split(float x0, float x1, uint32_t &hi, uint32_t &lo) {
        split_bf16(x0, x1, hi, lo);
    }
};
template <>
struct Ops<true> {
    static __device__ __forceinline__ void mma(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
        mma16816_f16(d, a0, a1, a2, a3, b0, b1);
    }
    static __device__ __forceinline__ void mma8(float *d, uint32_t a0, uint32_t a1, uint32_t b0) {
        mma1688_f16(d, a0, a1, b0);
    }
    static __device__ __forceinline__ void split(float x0, float x1, uint32_t &hi, uint32_t &lo) {
        split_f16(x0, x1, hi, lo);
    }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ float from_f32(float x) { return x; }
};
template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// Element (row, col) of a swizzled tile with rows of `cols` elements of type T.
template <typename T>
__device__ __forceinline__ T *swz_ptr(void *base, int row, int col, int cols) {
    return reinterpret_cast<T *>(reinterpret_cast<char *>(base) +
                                 swz_offset(row, col * (int)sizeof(T), cols * (int)sizeof(T)));
}
template <typename T>
__device__ __forceinline__ const T *swz_ptr(const void *base, int row, int col, int cols) {
    return reinterpret_cast<const T *>(reinterpret_cast<const char *>(base) +
                                       swz_offset(row, col * (int)sizeof(T), cols * (int)sizeof(T)));
}

}  // namespace pkv
