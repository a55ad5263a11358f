// ssm_step.cu -- the single-token recurrent update (decode), state in place:
//   step_dec16 (N = 16, whole 128-channel tiles), step_tma (whole 64-channel
//   tiles), step_pipe and step_kernel, and the dispatch between them.
#include "ssm_common.cuh"
#include "ssm_kernels.cuh"
#include "ssm_internal.h"

namespace ssm {

// ---------------------------------------------------------------- step ---
// One thread per (b, d, group of S states); GT = ceil(N / S) threads per
// channel.  The step reads the state once and writes it once, so it is bound
// by the state's HBM traffic: each thread keeps S * 4 bytes of state loads in
// flight (S = 16 at N = 16, 64 bytes), issued before any arithmetic.
template <typename TIN>
__device__ __forceinline__ void load_vec4_in(const TIN* p, float (&v)[4]) {
    if constexpr (sizeof(TIN) == 2) {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
    } else {
        const float4 w = *reinterpret_cast<const float4*>(p);
        v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    }
}

template <typename TIN, typename TOUT, int S, int GT>
__global__ void __launch_bounds__(256) step_kernel(const StepParams p) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = gid / GT;   // b * D + d
    const int g = (int)(gid % GT);
    const bool ok = row < p.Bt * p.D;
    const int64_t r = ok ? row : 0;
    const int64_t b = r / p.D, d = r % p.D;
    const int N = p.N;
    const int n0 = g * S;
    const TIN* u = static_cast<const TIN*>(p.u);
    const TIN* dr = static_cast<const TIN*>(p.dr);
    const TIN* Bv = static_cast<const TIN*>(p.B) + b * N;
    const TIN* Cv = static_cast<const TIN*>(p.C) + b * N;
    const float* Ad = p.A + d * N;
    float* st = p.state + r * N;
    // vector loads need 16-byte (state, A) and 8/16-byte (B, C) aligned rows
    const bool vec = (N % 4) == 0 && n0 + S <= N;

    float hv[S], av[S], bv[S], cv[S];
    if (vec) {
#pragma unroll
        for (int q = 0; q < S; q += 4) {
            const float4 h4 = *reinterpret_cast<const float4*>(st + n0 + q);
            hv[q] = h4.x; hv[q + 1] = h4.y; hv[q + 2] = h4.z; hv[q + 3] = h4.w;
        }
#pragma unroll
        for (int q = 0; q < S; q += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(Ad + n0 + q);
            av[q] = a4.x; av[q + 1] = a4.y; av[q + 2] = a4.z; av[q + 3] = a4.w;
            float t4[4];
            load_vec4_in<TIN>(Bv + n0 + q, t4);
            bv[q] = t4[0]; bv[q + 1] = t4[1]; bv[q + 2] = t4[2]; bv[q + 3] = t4[3];
            load_vec4_in<TIN>(Cv + n0 + q, t4);
            cv[q] = t4[0]; cv[q + 1] = t4[1]; cv[q + 2] = t4[2]; cv[q + 3] = t4[3];
        }
    } else {
#pragma unroll
        for (int q = 0; q < S; ++q) {
            const bool in = ok && n0 + q < N;
            hv[q] = in ? st[n0 + q] : 0.0f;
            av[q] = in ? Ad[n0 + q] : 0.0f;
            bv[q] = in ? Elem<TIN>::to_f(Bv[n0 + q]) : 0.0f;
            cv[q] = in ? Elem<TIN>::to_f(Cv[n0 + q]) : 0.0f;
        }
    }
    const float uu = Elem<TIN>::to_f(u[r]);
    const float x = fmaf(Elem<TIN>::to_f(dr[r]), kLog2e, p.bias ? p.bias[d] * kLog2e : 0.0f);
    const float d2 = softplus2<sizeof(TIN) == 4>(x);
    const float du = d2 * uu * kLn2;   // delta * u

    float acc = 0.0f;
#pragma unroll
    for (int q = 0; q < S; ++q) {
        const float a = sizeof(TIN) == 4 ? exp2_accurate(d2 * av[q]) : ex2(d2 * av[q]);
        hv[q] = fmaf(a, hv[q], du * bv[q]);
        acc = fmaf(cv[q], hv[q], acc);
    }
    if (ok) {
        if (vec) {
#pragma unroll
            for (int q = 0; q < S; q += 4)
                *reinterpret_cast<float4*>(st + n0 + q) =
                    make_float4(hv[q], hv[q + 1], hv[q + 2], hv[q + 3]);
        } else {
#pragma unroll
            for (int q = 0; q < S; ++q)
                if (n0 + q < N) st[n0 + q] = hv[q];
        }
    }
#pragma unroll
    for (int o = 1; o < GT; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (ok && g == 0) {
        float v = acc + (p.Dv ? p.Dv[d] * uu : 0.0f);
        if (p.z) {
            const float zq = Elem<TIN>::to_f(static_cast<const TIN*>(p.z)[r]);
            v *= zq * rcp(1.0f + ex2(-kLog2e * zq));
        }
        if (sizeof(TOUT) == 2)
            static_cast<__nv_bfloat16*>(p.y)[r] = __float2bfloat16_rn(v);
        else
            static_cast<float*>(p.y)[r] = v;
    }
}

// Pipelined step for state sizes that are a multiple of 4 (the usual case):
// each of the 256 threads owns one 16-byte quad of states of one channel per
// tile of 256 / (N/4) channels; tiles are taken grid-stride and the states of
// the next kStepDepth tiles are already on their way into shared memory
// (cp.async, 16 bytes per thread, no registers held), so each SM keeps
// ~kStepDepth * 4 KB * CTAs of state loads in flight.  The per-channel inputs
// of the next tile are loaded one tile ahead into registers.
constexpr int kStepDepth = 6;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int K>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory"); }

template <typename TIN, typename TOUT, int QPR>
__global__ void __launch_bounds__(256) step_pipe_kernel(const StepParams p) {
    constexpr int RPT = 256 / QPR;                    // channels (rows) per tile
    __shared__ __align__(16) float4 ring[kStepDepth][256];
    const int tid = threadIdx.x;
    const int N = p.N;                                // = 4 * QPR
    const int64_t rows = p.Bt * p.D;
    const int64_t ntiles = (rows + RPT - 1) / RPT;
    const int k = tid % QPR;                          // this thread's quad of the row
    const int lr = tid / QPR;                         // row within the tile
    const TIN* u = static_cast<const TIN*>(p.u);
    const TIN* dr = static_cast<const TIN*>(p.dr);
    const TIN* zz = static_cast<const TIN*>(p.z);
    const TIN* Bv = static_cast<const TIN*>(p.B);
    const TIN* Cv = static_cast<const TIN*>(p.C);

    auto issue = [&](int64_t tile, int slot) {
        const int64_t r = tile * RPT + lr;
        const bool valid = tile < ntiles && r < rows;
        cp_async16(smem_u32(&ring[slot][tid]), p.state + (valid ? r : 0) * N + 4 * k, valid);
        // the tile's per-channel inputs (u, delta_raw, z: one line each) are
        // pulled into L2 as far ahead as its states
        if (tid < 3 && tile < ntiles) {
            const TIN* src = tid == 0 ? u : tid == 1 ? dr : zz;
            if (src) prefetch_l2(src + tile * RPT);
        }
    };
    // per-row inputs of one tile, loaded into registers one tile ahead
    struct Row {
        float u, x2, z, a[4], b[4], c[4], dd, bias;
    };
    auto load_row = [&](int64_t tile, Row& w) {
        const int64_t r0 = tile * RPT + lr;
        const bool valid = tile < ntiles && r0 < rows;
        const int64_t r = valid ? r0 : 0;
        const int64_t b = r / p.D, d = r % p.D;
        w.u = Elem<TIN>::to_f(u[r]);
        w.bias = p.bias ? p.bias[d] : 0.0f;
        w.x2 = Elem<TIN>::to_f(dr[r]);
        w.z = zz ? Elem<TIN>::to_f(zz[r]) : 0.0f;
        w.dd = p.Dv ? p.Dv[d] : 0.0f;
        const float4 a4 = *reinterpret_cast<const float4*>(p.A + d * N + 4 * k);
        w.a[0] = a4.x; w.a[1] = a4.y; w.a[2] = a4.z; w.a[3] = a4.w;
        load_vec4_in<TIN>(Bv + b * N + 4 * k, w.b);
        load_vec4_in<TIN>(Cv + b * N + 4 * k, w.c);
    };

    int64_t tile = blockIdx.x;
#pragma unroll
    for (int j = 0; j < kStepDepth; ++j) {
        issue(tile + (int64_t)j * gridDim.x, j);
        cp_async_commit();
    }
    Row cur, nxt;
    load_row(tile, cur);
    for (int jt = 0; tile < ntiles; ++jt, tile += gridDim.x) {
        const int slot = jt % kStepDepth;
        // refill the slot read in the previous iteration (long complete) with
        // the tile kStepDepth - 1 ahead; one commit per iteration keeps the
        // group count regular, so waiting for all but the newest
        // kStepDepth - 1 groups guarantees this tile has landed
        if (jt > 0)
            issue(tile + (int64_t)(kStepDepth - 1) * gridDim.x, (jt - 1) % kStepDepth);
        cp_async_commit();
        load_row(tile + gridDim.x, nxt);
        cp_async_wait<kStepDepth - 1>();
        const float4 h4 = ring[slot][tid];            // this thread's own 16 bytes

        const int64_t r = tile * RPT + lr;
        const bool ok = r < rows;
        const float x = fmaf(cur.x2, kLog2e, cur.bias * kLog2e);
        const float d2 = softplus2<sizeof(TIN) == 4>(x);
        const float du = d2 * cur.u * kLn2;   // delta * u
        float hv[4] = {h4.x, h4.y, h4.z, h4.w};
        float acc = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float a = sizeof(TIN) == 4 ? exp2_accurate(d2 * cur.a[q]) : ex2(d2 * cur.a[q]);
            hv[q] = fmaf(a, hv[q], du * cur.b[q]);
            acc = fmaf(cur.c[q], hv[q], acc);
        }
        if (ok) *reinterpret_cast<float4*>(p.state + r * N + 4 * k) = make_float4(hv[0], hv[1], hv[2], hv[3]);
#pragma unroll
        for (int o = 1; o < QPR; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (ok && k == 0) {
            float v = fmaf(cur.dd, cur.u, acc);
            if (p.z) v *= cur.z * rcp(1.0f + ex2(-kLog2e * cur.z));
            if (sizeof(TOUT) == 2)
                static_cast<__nv_bfloat16*>(p.y)[r] = __float2bfloat16_rn(v);
            else
                static_cast<float*>(p.y)[r] = v;
        }
        cur = nxt;
    }
    cp_async_wait<0>();
}

// Streaming step for 64-channel tiles (D a multiple of 64 so a tile lies in
// one batch row; N a multiple of 4, N <= 32).  One producer warp moves
// everything a tile needs into an 8-slot shared-memory ring with bulk copies
// -- the states (64 * N * 4 bytes), u, delta_raw and z of the 64 channels,
// their rows of A, their bias and D skip, and the batch row's B and C -- so
// the 8 consumer warps issue no global load at all: thread (row, quad) owns
// 16 bytes of state, updates them and stores them straight back.  Tiles are
// taken grid-stride.
constexpr int kStepRows = 64;
constexpr int kStepSlots = 8;

template <typename TIN, int QPR>
struct StepSlot {
    float4 st[kStepRows * QPR];               // states
    float4 a[kStepRows * QPR];                // rows of A
    float bias[kStepRows], dsk[kStepRows];    // delta bias, D skip
    TIN in[3][kStepRows];                     // u, delta_raw, z
    TIN bc[2][32];                            // B, C of the batch row (N <= 32)
};

template <typename TIN, typename TOUT, int QPR>
__global__ void __launch_bounds__(32 * (8 * QPR / 4 + 1), 1) step_tma_kernel(const StepParams p) {
    constexpr int CONS = kStepRows * QPR;     // consumer threads (one 16-byte quad each)
    constexpr int NW = CONS / 32;             // consumer warps
    constexpr int N = 4 * QPR;
    extern __shared__ uint8_t smem_dyn[];
    StepSlot<TIN, QPR>* ring = reinterpret_cast<StepSlot<TIN, QPR>*>(align_smem_1024(smem_dyn));
    __shared__ __align__(8) uint64_t full_bar[kStepSlots];
    __shared__ __align__(8) uint64_t empty_bar[kStepSlots];
    const int tid = threadIdx.x;
    const int rows = (int)(p.Bt * p.D);       // < 2^31 (checked by the caller)
    const int D = (int)p.D;
    const int ntiles = rows / kStepRows;
    if (tid == 0) {
        for (int s = 0; s < kStepSlots; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const TIN* zz = static_cast<const TIN*>(p.z);

    if (tid >= CONS) {                        // ---------------- producer warp
        if (tid != CONS) return;
        const TIN* u = static_cast<const TIN*>(p.u);
        const TIN* dr = static_cast<const TIN*>(p.dr);
        const TIN* Bv = static_cast<const TIN*>(p.B);
        const TIN* Cv = static_cast<const TIN*>(p.C);
        int j = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
            const int s = j % kStepSlots;
            if (j >= kStepSlots &&
                !mbar_wait(&empty_bar[s], (uint32_t)(((j / kStepSlots) - 1) & 1), kDefaultTimeoutNs)) {
                set_status(p.status, SSM_ERR_TIMEOUT);
                return;                       // the consumers time out on their own waits
            }
            const int r0 = tile * kStepRows;
            const int b = r0 / D, d0 = r0 - b * D;
            constexpr uint32_t sb = kStepRows * N * 4, ib = kStepRows * sizeof(TIN);
            constexpr uint32_t fb = kStepRows * 4, bcb = N * sizeof(TIN) < 16 ? 16 : N * sizeof(TIN);
            const uint32_t bytes = 2 * sb + (zz ? 3 : 2) * ib + (p.bias ? fb : 0) + (p.Dv ? fb : 0) +
                                   2 * bcb;
            mbar_arrive_expect_tx(&full_bar[s], bytes);
            bulk_load(ring[s].st, p.state + (size_t)r0 * N, sb, &full_bar[s]);
            bulk_load(ring[s].a, p.A + (size_t)d0 * N, sb, &full_bar[s]);
            bulk_load(ring[s].in[0], u + r0, ib, &full_bar[s]);
            bulk_load(ring[s].in[1], dr + r0, ib, &full_bar[s]);
            if (zz) bulk_load(ring[s].in[2], zz + r0, ib, &full_bar[s]);
            if (p.bias) bulk_load(ring[s].bias, p.bias + d0, fb, &full_bar[s]);
            if (p.Dv) bulk_load(ring[s].dsk, p.Dv + d0, fb, &full_bar[s]);
            bulk_load(ring[s].bc[0], Bv + (size_t)b * N, bcb, &full_bar[s]);
            bulk_load(ring[s].bc[1], Cv + (size_t)b * N, bcb, &full_bar[s]);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    const int lane = tid & 31;
    const int k = tid % QPR;                  // quad of the row
    const int lr = tid / QPR;                 // row of the tile
    int j = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
        const int s = j % kStepSlots;
        if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], (uint32_t)((j / kStepSlots) & 1), kDefaultTimeoutNs))) {
            if (lane == 0) set_status(p.status, SSM_ERR_TIMEOUT);
            return;                           // bounded wait expired: nothing more is written
        }
        const StepSlot<TIN, QPR>& sl = ring[s];
        const float4 h4 = sl.st[tid];
        const float4 a4 = sl.a[tid];
        float bq[4], cq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            bq[q] = Elem<TIN>::to_f(sl.bc[0][4 * k + q]);
            cq[q] = Elem<TIN>::to_f(sl.bc[1][4 * k + q]);
        }
        const float uu = Elem<TIN>::to_f(sl.in[0][lr]);
        const float dv = Elem<TIN>::to_f(sl.in[1][lr]);
        const float zv = zz ? Elem<TIN>::to_f(sl.in[2][lr]) : 0.0f;
        const float bias = p.bias ? sl.bias[lr] : 0.0f;
        const float Dd = p.Dv ? sl.dsk[lr] : 0.0f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);   // the slot's contents are in registers

        const float x = fmaf(dv, kLog2e, bias * kLog2e);
        const float d2 = softplus2<sizeof(TIN) == 4>(x);
        const float du = d2 * uu * kLn2;   // delta * u
        float hv[4] = {h4.x, h4.y, h4.z, h4.w};
        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
        float acc = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float a = sizeof(TIN) == 4 ? exp2_accurate(d2 * av[q]) : ex2(d2 * av[q]);
            hv[q] = fmaf(a, hv[q], du * bq[q]);
            acc = fmaf(cq[q], hv[q], acc);
        }
        const int r = tile * kStepRows + lr;
        *reinterpret_cast<float4*>(p.state + (size_t)r * N + 4 * k) = make_float4(hv[0], hv[1], hv[2], hv[3]);
#pragma unroll
        for (int o = 1; o < QPR; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (k == 0) {
            float v = fmaf(Dd, uu, acc);
            if (zz) v *= zv * rcp(1.0f + ex2(-kLog2e * zv));
            if (sizeof(TOUT) == 2)
                static_cast<__nv_bfloat16*>(p.y)[r] = __float2bfloat16_rn(v);
            else
                static_cast<float*>(p.y)[r] = v;
        }
    }
}

template <typename TIN, typename TOUT, int QPR>
static cudaError_t launch_step_tma(const StepParams& p, cudaStream_t st) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    auto kern = step_tma_kernel<TIN, TOUT, QPR>;
    const size_t smem = kStepSlots * sizeof(StepSlot<TIN, QPR>) + 1024;
    static bool attr[64] = {};
    static int per_sm[64] = {};
    if (dev >= 0 && dev < 64 && !attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, 32 * (8 * QPR / 4 + 1), smem) !=
                cudaSuccess || nb < 1)
            nb = 1;
        cudaGetLastError();
        per_sm[dev] = nb;
        attr[dev] = true;
    }
    const int nb = (dev >= 0 && dev < 64) ? per_sm[dev] : 1;
    const int64_t ntiles = p.Bt * p.D / kStepRows;
    int64_t grid = (int64_t)sms * nb;
    if (grid > ntiles) grid = ntiles;
    kern<<<(unsigned)grid, 32 * (8 * QPR / 4 + 1), smem, st>>>(p);
    return cudaGetLastError();
}

// Decode step for N = 16 and D a multiple of 128: one thread per channel.
// A producer warp moves each 128-channel tile into a ring of 3 slots (56 KB,
// so that four CTAs share an SM: more resident warps beat deeper rings,
// measured 32.9 us per step against 34.3 us with 6 slots and 2 CTAs per SM,
// 36.9 us with 2 slots): the states and the rows
// of A as 2-D TMA tiles with the 64-byte swizzle (a thread reads its 64-byte
// row as four 16-byte chunks; the swizzle spreads the 32 lanes' chunks over
// all banks), u, delta_raw, z, bias, D skip and the batch row's B and C as
// bulk copies.  4 consumer warps do the per-channel work once per channel
// and write the new states into the slot in place; one thread then stores
// the tile with a TMA tile store (whole 32-byte sectors, where per-thread
// stores of 64-byte rows would write half sectors) and releases the slot
// once that store has read it.
constexpr int kDecRows = 128;
constexpr int kDecSlots = 3;

template <typename TIN>
struct __align__(1024) DecSlot {
    float st[kDecRows * 16];                  // 64-byte rows, 64-byte swizzle
    float a[kDecRows * 16];
    float bias[kDecRows], dsk[kDecRows];
    TIN in[3][kDecRows];                      // u, delta_raw, z
    TIN bc[2][16];                            // B, C of the batch row
};

// 16-byte chunk q of row r of a 64-byte-row tile written by TMA with the
// 64-byte swizzle (chunk bits XOR address bits 7-8, i.e. (r >> 1) & 3)
__device__ __forceinline__ float4 ld_swz64(const float* tile, int r, int q) {
    return *reinterpret_cast<const float4*>(tile + r * 16 + 4 * (q ^ ((r >> 1) & 3)));
}

template <typename TIN, typename TOUT>
__global__ void __launch_bounds__(160, 2) step_dec16_kernel(const StepParams p,
                                                           const __grid_constant__ CUtensorMap tm_st,
                                                           const __grid_constant__ CUtensorMap tm_a) {
    extern __shared__ uint8_t smem_dyn[];
    DecSlot<TIN>* ring = reinterpret_cast<DecSlot<TIN>*>(align_smem_1024(smem_dyn));
    __shared__ __align__(8) uint64_t full_bar[kDecSlots];
    __shared__ __align__(8) uint64_t empty_bar[kDecSlots];
    __shared__ int dead;                      // a consumer warp's wait expired
    const int tid = threadIdx.x;
    const int rows = (int)(p.Bt * p.D);       // < 2^31 (checked by the caller)
    const int D = (int)p.D;
    const int ntiles = rows / kDecRows;
    if (tid == 0) {
        for (int s = 0; s < kDecSlots; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        dead = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const TIN* zz = static_cast<const TIN*>(p.z);

    if (tid >= 128) {                         // ---------------- producer warp
        if (tid != 128) return;
        prefetch_tmap(&tm_st);
        prefetch_tmap(&tm_a);
        const TIN* u = static_cast<const TIN*>(p.u);
        const TIN* dr = static_cast<const TIN*>(p.dr);
        const TIN* Bv = static_cast<const TIN*>(p.B);
        const TIN* Cv = static_cast<const TIN*>(p.C);
        int j = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
            const int s = j % kDecSlots;
            if (j >= kDecSlots &&
                !mbar_wait(&empty_bar[s], (uint32_t)(((j / kDecSlots) - 1) & 1), kDefaultTimeoutNs)) {
                set_status(p.status, SSM_ERR_TIMEOUT);
                return;                       // the consumers time out on their own waits
            }
            const int r0 = tile * kDecRows;
            const int b = r0 / D, d0 = r0 - b * D;
            constexpr uint32_t tb = kDecRows * 64, ib = kDecRows * sizeof(TIN), fb = kDecRows * 4;
            constexpr uint32_t bcb = 16 * sizeof(TIN);
            const uint32_t bytes = 2 * tb + (zz ? 3 : 2) * ib + (p.bias ? fb : 0) + (p.Dv ? fb : 0) + 2 * bcb;
            DecSlot<TIN>& sl = ring[s];
            mbar_arrive_expect_tx(&full_bar[s], bytes);
            tma_load_2d(sl.st, &tm_st, &full_bar[s], 0, r0);
            tma_load_2d(sl.a, &tm_a, &full_bar[s], 0, d0);
            bulk_load(sl.in[0], u + r0, ib, &full_bar[s]);
            bulk_load(sl.in[1], dr + r0, ib, &full_bar[s]);
            if (zz) bulk_load(sl.in[2], zz + r0, ib, &full_bar[s]);
            if (p.bias) bulk_load(sl.bias, p.bias + d0, fb, &full_bar[s]);
            if (p.Dv) bulk_load(sl.dsk, p.Dv + d0, fb, &full_bar[s]);
            bulk_load(sl.bc[0], Bv + (size_t)b * 16, bcb, &full_bar[s]);
            bulk_load(sl.bc[1], Cv + (size_t)b * 16, bcb, &full_bar[s]);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    // Every consumer warp reaches the per-tile barrier even when its wait
    // expired, so that the barrier always completes; the flag then ends the
    // loop for all of them.
    int j = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
        const int s = j % kDecSlots;
        DecSlot<TIN>& sl = ring[s];
        if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], (uint32_t)((j / kDecSlots) & 1), kDefaultTimeoutNs))) {
            if ((tid & 31) == 0) set_status(p.status, SSM_ERR_TIMEOUT);
            dead = 1;
            named_bar_sync(1, 128);
            break;
        }
        float hv[16], av[16], bq[16], cq[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 h4 = ld_swz64(sl.st, tid, q);
            const float4 a4 = ld_swz64(sl.a, tid, q);
            hv[4 * q] = h4.x; hv[4 * q + 1] = h4.y; hv[4 * q + 2] = h4.z; hv[4 * q + 3] = h4.w;
            av[4 * q] = a4.x; av[4 * q + 1] = a4.y; av[4 * q + 2] = a4.z; av[4 * q + 3] = a4.w;
            float t4[4];
            load_vec4_in<TIN>(&sl.bc[0][4 * q], t4);
            bq[4 * q] = t4[0]; bq[4 * q + 1] = t4[1]; bq[4 * q + 2] = t4[2]; bq[4 * q + 3] = t4[3];
            load_vec4_in<TIN>(&sl.bc[1][4 * q], t4);
            cq[4 * q] = t4[0]; cq[4 * q + 1] = t4[1]; cq[4 * q + 2] = t4[2]; cq[4 * q + 3] = t4[3];
        }
        const float uu = Elem<TIN>::to_f(sl.in[0][tid]);
        const float dv = Elem<TIN>::to_f(sl.in[1][tid]);
        const float zv = zz ? Elem<TIN>::to_f(sl.in[2][tid]) : 0.0f;
        const float bias = p.bias ? sl.bias[tid] : 0.0f;
        const float Dd = p.Dv ? sl.dsk[tid] : 0.0f;

        const float x = fmaf(dv, kLog2e, bias * kLog2e);
        const float d2 = softplus2<sizeof(TIN) == 4>(x);
        const float du = d2 * uu * kLn2;   // delta * u
        float acc = 0.0f;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float a = sizeof(TIN) == 4 ? exp2_accurate(d2 * av[q]) : ex2(d2 * av[q]);
            hv[q] = fmaf(a, hv[q], du * bq[q]);
            acc = fmaf(cq[q], hv[q], acc);
        }
        const int r = tile * kDecRows + tid;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4*>(sl.st + tid * 16 + 4 * (q ^ ((tid >> 1) & 3))) =
                make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
        fence_proxy_async();
        named_bar_sync(1, 128);
        if (dead) break;
        if (tid == 0) {
            tma_store_2d(&tm_st, sl.st, 0, tile * kDecRows);
            bulk_commit();
            bulk_wait_read<1>();              // the previous tile's store has read its slot
            if (j > 0) mbar_arrive(&empty_bar[(j - 1) % kDecSlots]);
        }
        float v = fmaf(Dd, uu, acc);
        if (zz) v *= zv * rcp(1.0f + ex2(-kLog2e * zv));
        if (sizeof(TOUT) == 2)
            static_cast<__nv_bfloat16*>(p.y)[r] = __float2bfloat16_rn(v);
        else
            static_cast<float*>(p.y)[r] = v;
    }
    if (tid == 0) bulk_wait<0>();             // the tile stores finish before the CTA exits
}

template <typename TIN, typename TOUT>
static cudaError_t launch_step_dec16(const StepParams& p, const CUtensorMap& tm_st,
                                     const CUtensorMap& tm_a, cudaStream_t st) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    auto kern = step_dec16_kernel<TIN, TOUT>;
    const size_t smem = kDecSlots * sizeof(DecSlot<TIN>) + 1024;
    static bool attr[64] = {};
    static int per_sm[64] = {};
    if (dev >= 0 && dev < 64 && !attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, 160, smem) != cudaSuccess || nb < 1)
            nb = 1;
        cudaGetLastError();
        per_sm[dev] = nb;
        attr[dev] = true;
    }
    const int nb = (dev >= 0 && dev < 64) ? per_sm[dev] : 1;
    const int64_t ntiles = p.Bt * p.D / kDecRows;
    int64_t grid = (int64_t)sms * nb;
    if (grid > ntiles) grid = ntiles;
    kern<<<(unsigned)grid, 160, smem, st>>>(p, tm_st, tm_a);
    return cudaGetLastError();
}

cudaError_t launch_step_dec16_any(int tin, int tout, const StepParams& p, const CUtensorMap& tm_st,
                                  const CUtensorMap& tm_a, cudaStream_t st) {
    if (tin == SSM_BF16)
        return tout == SSM_BF16 ? launch_step_dec16<__nv_bfloat16, __nv_bfloat16>(p, tm_st, tm_a, st)
                                : launch_step_dec16<__nv_bfloat16, float>(p, tm_st, tm_a, st);
    return tout == SSM_BF16 ? launch_step_dec16<float, __nv_bfloat16>(p, tm_st, tm_a, st)
                            : launch_step_dec16<float, float>(p, tm_st, tm_a, st);
}

template <typename TIN, typename TOUT, int QPR>
static cudaError_t launch_step_pipe(const StepParams& p, cudaStream_t st) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    const int64_t rows = p.Bt * p.D;
    const int64_t ntiles = (rows + (256 / QPR) - 1) / (256 / QPR);
    static int per_sm[64] = {};
    if (dev >= 0 && dev < 64 && per_sm[dev] == 0) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, step_pipe_kernel<TIN, TOUT, QPR>, 256, 0) !=
                cudaSuccess || nb < 1)
            nb = 4;
        cudaGetLastError();
        per_sm[dev] = nb;
    }
    const int nb = (dev >= 0 && dev < 64) ? per_sm[dev] : 4;
    int64_t grid = (int64_t)sms * nb;                 // every CTA resident at once
    if (grid > ntiles) grid = ntiles;
    step_pipe_kernel<TIN, TOUT, QPR><<<(unsigned)grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename TIN, typename TOUT, int S, int GT>
static cudaError_t launch_step_s(const StepParams& p, cudaStream_t st) {
    const int64_t threads = p.Bt * p.D * GT;
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    step_kernel<TIN, TOUT, S, GT><<<blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename TIN, typename TOUT>
static cudaError_t launch_step_t(const StepParams& p, cudaStream_t st) {
    // whole 64-channel tiles inside one batch row: the bulk-copy stream
    if (p.D % kStepRows == 0 && p.Bt * p.D < (int64_t(1) << 31)) {
        if (p.N == 16) return launch_step_tma<TIN, TOUT, 4>(p, st);
        if (p.N == 8) return launch_step_tma<TIN, TOUT, 2>(p, st);
        if (p.N == 32) return launch_step_tma<TIN, TOUT, 8>(p, st);
    }
    // state sizes 4, 8, 16, 32 otherwise: the cp.async pipeline
    if (p.N == 16) return launch_step_pipe<TIN, TOUT, 4>(p, st);
    if (p.N == 8) return launch_step_pipe<TIN, TOUT, 2>(p, st);
    if (p.N == 32) return launch_step_pipe<TIN, TOUT, 8>(p, st);
    if (p.N == 4) return launch_step_pipe<TIN, TOUT, 1>(p, st);
    // otherwise: S states per thread (a multiple of 4 when N allows vector
    // loads), GT threads per channel (a power of two, for the shuffle reduction)
    if (p.N <= 4) return launch_step_s<TIN, TOUT, 4, 1>(p, st);
    if (p.N <= 8) return launch_step_s<TIN, TOUT, 8, 1>(p, st);
    if (p.N <= 16) return launch_step_s<TIN, TOUT, 16, 1>(p, st);
    if (p.N <= 32) return launch_step_s<TIN, TOUT, 16, 2>(p, st);
    return launch_step_s<TIN, TOUT, 16, 4>(p, st);
}

cudaError_t launch_step(int tin, int tout, const StepParams& p, cudaStream_t st) {
    if (tin == SSM_BF16)
        return tout == SSM_BF16 ? launch_step_t<__nv_bfloat16, __nv_bfloat16>(p, st)
                                : launch_step_t<__nv_bfloat16, float>(p, st);
    return tout == SSM_BF16 ? launch_step_t<float, __nv_bfloat16>(p, st)
                            : launch_step_t<float, float>(p, st);
}
}  // namespace ssm
