// ssm_internal.h -- launchers shared between the C-ABI layer and the kernel
// translation units.  Internal to libssmscan.so.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ssm_kernels.cuh"

namespace ssm {

// Tensor maps of one forward launch: raw tiles of u, delta_raw, z (unused
// entries zeroed) and the prepared B/C tile.
struct FwdMaps {
    CUtensorMap u, dr, z, bc;
    CUtensorMap ya;   // the bidirectional scan's left-to-right pass: the other direction's output
};

// Forward kernel launch for padded state size NP (4, 8, 16, 32, 64), NT
// threads per channel and `warps` compute warps per CTA, with `smem` bytes of
// dynamic shared memory.  tin/tout are ssm_dtype values.
cudaError_t launch_fwd_np4(int NT, int tin, int tout, bool summary, bool tma_raw,
                           const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                           size_t smem, cudaStream_t st);
cudaError_t launch_fwd_np8(int NT, int tin, int tout, bool summary, bool tma_raw,
                           const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                           size_t smem, cudaStream_t st);
cudaError_t launch_fwd_np16(int NT, int tin, int tout, bool summary, bool tma_raw,
                            const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                            size_t smem, cudaStream_t st);
// The forward with the conv prologue, padded state size 16, TMA tiles.
cudaError_t launch_fwd_conv_np16(int NT, int tin, int tout, bool summary, const FwdParams& p,
                                 const FwdMaps& m, dim3 grid, int warps, size_t smem, cudaStream_t st);
// The forward over packed sequences (restarts at cu_seqlens), padded state
// size 16, TMA tiles, with or without the conv prologue.
cudaError_t launch_fwd_varlen_np16(int NT, int tin, int tout, bool summary, bool conv,
                                   const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                                   size_t smem, cudaStream_t st);
// The bidirectional scan's two passes, padded state size 16, TMA tiles:
// dir 1 = right to left (fp32 gated output into p.y), dir 2 = left to right
// adding p.yadd; summary = the right-to-left segment summaries (pass 1 of the
// segmented plan; the left-to-right one is the plain forward's).
cudaError_t launch_fwd_bidir_np16(int NT, int tin, int tout, int dir, bool summary,
                                  const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                                  size_t smem, cudaStream_t st);
cudaError_t launch_fwd_np32(int NT, int tin, int tout, bool summary, bool tma_raw,
                            const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                            size_t smem, cudaStream_t st);
cudaError_t launch_fwd_np64(int NT, int tin, int tout, bool summary, bool tma_raw,
                            const FwdParams& p, const FwdMaps& m, dim3 grid, int warps,
                            size_t smem, cudaStream_t st);

// The NT values each NP supports.
int fwd_supported_nt(int NP, int* out, int cap);

// Tensor maps of one backward call: raw tiles of u, delta_raw, z, dy, the
// fp32 per-token tile written by the forward sweep, and the B/C tile.
struct BwdMaps {
    CUtensorMap u, dr, z, dy, phi, bc;
};

// Launch shape of one backward call: grid, compute warps per CTA, ring
// depths and dynamic shared memory of the two sweeps.
struct BwdLaunch {
    dim3 grid;               // z = segments (1 without the segmented plan)
    int warps;
    int stages_f, stages_r;
    size_t smem_f, smem_r;
    int stages_l = 2;        // segmented plan: the adjoint summary's ring and shared memory
    size_t smem_l = 0;
};

// Backward (forward sweep, then reverse sweep) for padded state size NP
// (8, 16, 32, 64) and NT threads per channel.
cudaError_t launch_bwd_np8(int NT, int tin, int tout, bool tma, const BwdParams& p,
                           const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st);
cudaError_t launch_bwd_np16(int NT, int tin, int tout, bool tma, const BwdParams& p,
                            const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st);
cudaError_t launch_bwd_np32(int NT, int tin, int tout, bool tma, const BwdParams& p,
                            const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st);
cudaError_t launch_bwd_np64(int NT, int tin, int tout, bool tma, const BwdParams& p,
                            const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st);
// the same over packed sequences (p.cu_seqlens, p.nseq): padded state size 16,
// two or four threads per channel, 16-byte token rows (TMA tiles)
cudaError_t launch_bwd_varlen_np16(int NT, int tin, int tout, const BwdParams& p,
                                   const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st);

// The segmented backward for padded state size 16, 16-byte token rows and
// two or four threads per channel: part 0 = the adjoint summary of segments
// 1 .. nseg-1 (grid z = nseg - 1), part 1 = the forward sweep with the
// tangent sums, part 2 = the reverse sweep (both grid z = nseg).
cudaError_t launch_bwd_seg_np16(int NT, int tin, int tout, int part, const BwdParams& p,
                                const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st);
// the same over packed sequences (p.cu_seqlens, p.nseq)
cudaError_t launch_bwd_seg_varlen_np16(int NT, int tin, int tout, int part, const BwdParams& p,
                                       const BwdMaps& m, const BwdLaunch& lc, cudaStream_t st);
// The backward fed by the conv prologue (both sweeps form u from x; p.u is
// the branch input x, p.conv_w/conv_b/conv_k as in FwdParams), padded state
// size 16, 16-byte token rows, whole rows; and the prologue's reverse mode:
// dx (tout), dconv_w, dconv_b (both accumulated with atomics; zeroed by the
// host) from the sweeps' du.  The sweeps write ddelta_raw and dz as tout and
// du in fp32 (p.du: an fp32 buffer).
cudaError_t launch_bwd_conv_np16(int NT, int tin, int tout, const BwdParams& p, const BwdMaps& m,
                                 const BwdLaunch& lc, cudaStream_t st);
cudaError_t launch_conv_bwd(int tin, int tout, int64_t Bt, int64_t D, int64_t L, int K,
                            const void* x, const float* conv_w, const float* conv_b,
                            const float* du, void* dx, float* dconv_w, float* dconv_b,
                            cudaStream_t st);
// The dA terms of the tangent flowing into each segment from the ones before
// (see ssm_aux.cu); after the forward sweep of the segmented backward.
cudaError_t launch_tangent_carry(int64_t Bt, int64_t D, int N, int NP, int nseg, const float* A,
                                 const float* sumd, const float* mend, const float* gp, float* dA,
                                 cudaStream_t st);

cudaError_t launch_prep_bc(int tin, int64_t Bt, int N, int NP, int64_t L, const void* B,
                           const void* C, float* out, int* status, cudaStream_t st);
// Tail search of the segmented plan (see ssm_aux.cu): per (segment, batch
// row, channel tile) the first chunk pass 1 needs; per saturated channel a
// marker in sumd.  Segments 0 .. nseg-2.
cudaError_t launch_tail(int tin, const FwdParams& p, int CH, unsigned tiles, int* tstart, float* sumd,
                        cudaStream_t st);
// Head search of the segmented backward (see ssm_aux.cu): per (segment,
// batch row, channel tile) the chunk after the last one the adjoint summary
// needs; per saturated channel a marker in sumd.  Segments 1 .. nseg-1.
cudaError_t launch_head(int tin, const BwdParams& p, int CH, unsigned tiles, int* kstop, float* sumd,
                        cudaStream_t st);
cudaError_t launch_carry(int64_t Bt, int64_t D, int N, int NP, int nseg, const float* A,
                         const float* h0, const float* hloc, const float* sumd, float* hin,
                         cudaStream_t st, bool reverse = false);
// Packed sequences: checks cu_seqlens (0 = c_0 <= c_1 <= ... <= c_nseq = L,
// else SSM_ERR_SEQLENS in the status word) and writes the final state of
// every empty sequence (its h0, or zero).  After prep_bc, which clears the
// status word.
cudaError_t launch_varlen_prep(const int* cu, int nseq, int64_t L, int64_t per_seq, const float* h0,
                               float* hL, int* status, cudaStream_t st);
cudaError_t launch_step(int tin, int tout, const StepParams& p, cudaStream_t st);
// Decode step for N = 16 and D a multiple of 128 (one thread per channel, 2-D
// TMA tiles of the states and of A given by tm_st (rows = batch*dim) and tm_a
// (rows = dim), 16 fp32 columns, 64-byte swizzle, box 16 x 128).
cudaError_t launch_step_dec16_any(int tin, int tout, const StepParams& p, const CUtensorMap& tm_st,
                                  const CUtensorMap& tm_a, cudaStream_t st);
cudaError_t launch_expired_wait(int* status, int64_t spin_limit, cudaStream_t st);

// the bidirectional backward (ssm_flip.cu)
cudaError_t launch_flip_rows(int dtype, const void* in, void* out, int64_t rows, int64_t L,
                             cudaStream_t st);
cudaError_t launch_bidir_combine(int tout, int64_t rows, int64_t L, const float* du1,
                                 const float* du2, const float* dz1, const float* dz2,
                                 const float* ddr1, const float* ddr2, void* du, void* dz,
                                 void* ddr, void* ddr_r, cudaStream_t st);
cudaError_t launch_fold_status(int* outer, const int* inner, cudaStream_t st);

}  // namespace ssm
