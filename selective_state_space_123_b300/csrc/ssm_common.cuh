// ssm_common.cuh -- device helpers shared by the selective-scan kernels
// (inline PTX for sm_103a: packed f32x2 arithmetic, MUFU exp2/log2/rcp,
// mbarrier waits with a time limit, TMA tile loads).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/ssm_scan.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a (Blackwell) only"
#endif

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ----------------------------------------------------------------- MUFU ---
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// --------------------------------------------------- packed f32x2 math ---
// A pair of fp32 values in one 64-bit register; one instruction does both.
typedef unsigned long long f2;

__device__ __forceinline__ f2 pk(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk(f2 r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// exp2 of both halves (two MUFU operations)
__device__ __forceinline__ f2 ex2x2(f2 x) {
    float lo, hi;
    upk(x, lo, hi);
    return pk(ex2(lo), ex2(hi));
}

// 2^x to about one fp32 ulp, on the FMA pipe, for the fp32-input path where
// the MUFU's ~2^-22 relative error would compound over long decay products.
// Range reduction x = n + f with n = round(x), |f| <= 1/2 (exact in fp32),
// then 2^f = sum_k (f ln 2)^k / k! to k = 7 (truncation < 6e-9 relative),
// then n is added to the exponent field.  x is clamped to [-125, 127]; below
// -125 the true value is under 2^-125 and the result stays a normal number.
__device__ __forceinline__ float exp2_accurate(float x) {
    x = fminf(fmaxf(x, -125.0f), 127.0f);
    const int n = __float2int_rn(x);
    const float f = x - (float)n;
    float p = 1.5252733804059840e-05f;            // ln2^7 / 7!
    p = fmaf(p, f, 1.5403530393381606e-04f);      // ln2^6 / 6!
    p = fmaf(p, f, 1.3333558146428443e-03f);      // ln2^5 / 5!
    p = fmaf(p, f, 9.6181291076284770e-03f);      // ln2^4 / 4!
    p = fmaf(p, f, 5.5504108664821580e-02f);      // ln2^3 / 3!
    p = fmaf(p, f, 2.4022650695910070e-01f);      // ln2^2 / 2!
    p = fmaf(p, f, 6.9314718055994530e-01f);      // ln2
    p = fmaf(p, f, 1.0f);
    return __int_as_float(__float_as_int(p) + (n << 23));
}
// 2^x - 1 with a small relative error for every x (the forgetting rate of a
// decay 2^x close to 1 keeps its own digits instead of those of 1).  With x =
// n + f as in exp2_accurate: (2^f - 1) / f = sum_{k>=1} ln2^k f^(k-1) / k! to
// k = 8 (truncation < 1e-9 relative), 2^f - 1 = f times that, and for n != 0
// 2^x - 1 = 2^n (2^f - 1) + (2^n - 1), where 2^n - 1 is exact for |n| <= 24
// and the two terms do not cancel.
__device__ __forceinline__ float exp2m1_accurate(float x) {
    x = fminf(fmaxf(x, -125.0f), 127.0f);
    const int n = __float2int_rn(x);
    const float f = x - (float)n;
    float q = 1.3215486790144307e-06f;            // ln2^8 / 8!
    q = fmaf(q, f, 1.5252733804059840e-05f);      // ln2^7 / 7!
    q = fmaf(q, f, 1.5403530393381606e-04f);      // ln2^6 / 6!
    q = fmaf(q, f, 1.3333558146428443e-03f);      // ln2^5 / 5!
    q = fmaf(q, f, 9.6181291076284770e-03f);      // ln2^4 / 4!
    q = fmaf(q, f, 5.5504108664821580e-02f);      // ln2^3 / 3!
    q = fmaf(q, f, 2.4022650695910070e-01f);      // ln2^2 / 2!
    q = fmaf(q, f, 6.9314718055994530e-01f);      // ln2
    const float em1f = f * q;
    if (n == 0) return em1f;
    const float p = __int_as_float((n + 127) << 23);   // 2^n, -125 <= n <= 127
    return fmaf(p, em1f, p - 1.0f);
}

// log2(1 + e) for 0 <= e <= 1 on the FMA pipe, to a few fp32 ulps: with
// s = e / (2 + e) (0 <= s <= 1/3), ln(1 + e) = 2 atanh(s) = 2 (s + s^3/3 +
// s^5/5 + ...), summed to s^17 (truncation < 2e-9 relative at s = 1/3).
__device__ __forceinline__ float log2_1p_accurate(float e) {
    const float s = __fdiv_rn(e, 2.0f + e);
    const float s2 = s * s;
    float p = 1.0f / 17.0f;
    p = fmaf(p, s2, 1.0f / 15.0f);
    p = fmaf(p, s2, 1.0f / 13.0f);
    p = fmaf(p, s2, 1.0f / 11.0f);
    p = fmaf(p, s2, 1.0f / 9.0f);
    p = fmaf(p, s2, 1.0f / 7.0f);
    p = fmaf(p, s2, 1.0f / 5.0f);
    p = fmaf(p, s2, 1.0f / 3.0f);
    p = fmaf(p, s2, 1.0f);
    return (2.0f * kLog2e) * (s * p);
}

__device__ __forceinline__ f2 exp2_accurate_x2(f2 x) {
    float lo, hi;
    upk(x, lo, hi);
    return pk(exp2_accurate(lo), exp2_accurate(hi));
}

// softplus in log2 units: for x = (delta_raw + bias) * log2(e) return
// log2(1 + 2^x) = delta / ln 2.
//  ACCURATE (fp32 inputs): max(x, 0) + log2(1 + 2^-|x|), both the power and
//  the logarithm on the FMA pipe (exp2_accurate, log2_1p_accurate), so that
//  delta keeps fp32-level relative accuracy down to the smallest steps (the
//  MUFU lg2's absolute error near 1 would dominate small results); 0 below
//  x = -126, where delta / ln2 < 2^-126.
//  fast (bf16 inputs): max(x, lg2(1 + e)) with e = 2^min(x, 64), except for
//  e < 1/64, where 1 + e loses e's low bits to rounding and the lg2's
//  absolute error near 1 would be a large relative error of a tiny delta
//  (the long-memory regime): there log2(1 + e) = log2(e) (e - e^2/2 + ...)
//  truncated after the quadratic term (relative error < e^2/3 < 8.2e-5).
template <bool ACCURATE>
__device__ __forceinline__ float softplus2(float x) {
    if (ACCURATE) {
        if (x < -126.0f) return 0.0f;
        return fmaxf(x, 0.0f) + log2_1p_accurate(exp2_accurate(-fabsf(x)));
    } else {
        const float e = ex2(fminf(x, 64.0f));
        const float series = e * fmaf(e, -0.5f * kLog2e, kLog2e);
        return e < 0.015625f ? series : fmaxf(x, lg2(1.0f + e));
    }
}


// ------------------------------------------------------- element types ---
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kBytes = 4;
    __device__ __forceinline__ static float to_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
};

// two bf16 packed in a 32-bit word -> two floats (exact widening)
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// two floats -> packed bf16 pair, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ----------------------------------------------------------- time base ---
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Record a device-side error in the status word (first error wins).
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ mbarrier ---
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Wait for phase `parity` of `bar` to complete, giving up after `limit_ns`
// nanoseconds or `spin_limit` polls, whichever comes first (spin_limit 0 means
// the default cap of 2^28 polls, so the wait ends even if the clock stalls).
// Returns false on timeout; the caller records SSM_ERR_TIMEOUT.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                          int64_t spin_limit = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const int64_t cap = spin_limit > 0 ? spin_limit : (int64_t(1) << 28);
    const uint64_t t0 = globaltimer_ns();
    for (int64_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i >= cap) return false;
        if ((i & 63) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ----------------------------------------------------------------- TMA ---
// 2-D tiled load of box {x, y} into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
// 1-D bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(smem_dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// 2-D tiled store of box {x, y} from shared memory (bulk-group completion).
// The writing threads order their shared-memory stores before it with
// fence_proxy_async() and a barrier.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* smem_src, int32_t x,
                                             int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(tmap), "r"(smem_u32(smem_src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N committed bulk groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until at most N committed bulk groups are incomplete (writes visible)
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA)
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// named barrier `id` over `count` threads (a multiple of 32)
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// First 1024-byte aligned address of the dynamic shared-memory window (the
// 128-byte TMA swizzle repeats every 1024 bytes).  The offset is added to the
// __shared__ array itself so that the compiler keeps shared-memory
// addressing for every access derived from the result.
__device__ __forceinline__ uint8_t* align_smem_1024(uint8_t* smem_dyn) {
    return smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
}

// Byte offset of element (row r, column byte cb) inside a tile whose rows are
// 128 bytes long and were written by TMA with the 128-byte swizzle: the
// 16-byte chunk index is XORed with the row index modulo 8 (tile base
// 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(uint32_t r, uint32_t cb) {
    return r * 128u + ((((cb >> 4) ^ r) & 7u) << 4) + (cb & 15u);
}

}  // namespace ssm
