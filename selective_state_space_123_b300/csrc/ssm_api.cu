// ssm_api.cu -- the C ABI of libssmscan.so (declared in include/ssm_scan.h):
// argument validation, planning of the forward launch, TMA descriptors,
// workspace layout, status word.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/ssm_scan.h"
#include "ssm_internal.h"

using namespace ssm;

namespace {

constexpr size_t kHeaderBytes = 256;   // status word at offset 0

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int dtype_bytes(int32_t t) { return t == SSM_BF16 ? 2 : 4; }

bool valid_dtype(int32_t t) { return t == SSM_F32 || t == SSM_BF16; }

// multiply with overflow check (all operands >= 0)
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

int padded_state(int64_t N) {
    if (N <= 4) return 4;
    if (N <= 8) return 8;
    if (N <= 16) return 16;
    if (N <= 32) return 32;
    return 64;
}

// A CUDA call failed: clear the (non-sticky) error state so the caller's next
// CUDA call does not see it, and report SSM_ERR_CUDA.
int cuda_fail() {
    cudaGetLastError();
    return SSM_ERR_CUDA;
}

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::atoi(v);
}

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 148; }
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 148;
    }
    return sms > 0 ? sms : 148;
}

int shape_check(const ssm_shape* s) {
    if (!s) return SSM_ERR_NULL;
    if (s->batch < 0 || s->dim < 0 || s->seqlen < 0) return SSM_ERR_SHAPE;
    if (s->dstate < 1 || s->dstate > 64) return SSM_ERR_SHAPE;
    if (!valid_dtype(s->in_dtype) || !valid_dtype(s->out_dtype)) return SSM_ERR_DTYPE;
    int64_t bd, bdl, bl;
    if (!mul_ok(s->batch, s->dim, &bd) || !mul_ok(bd, s->seqlen, &bdl) ||
        !mul_ok(s->batch, s->seqlen, &bl))
        return SSM_ERR_SHAPE;
    int64_t tmp;
    if (!mul_ok(bdl, 8, &tmp) || !mul_ok(bd, 64 * 8, &tmp) || !mul_ok(bl, 128 * 4, &tmp))
        return SSM_ERR_SHAPE;
    // TMA coordinates are 32-bit: rows of (batch*dim) and (batch*seqlen);
    // the batch index is a grid dimension (at most 65535)
    if (bd >= (int64_t(1) << 31) || bl >= (int64_t(1) << 31)) return SSM_ERR_UNSUPPORTED;
    if (s->batch > 65535) return SSM_ERR_UNSUPPORTED;
    return SSM_OK;
}

struct FwdPlan {
    int NP = 16, NT = 2, W = 4, CH = 64, stages = 2;
    size_t smem = 0;
    int nseg = 1;
    int64_t nchunks = 0, seg_chunks = 0;
    bool tma_raw = false;
    size_t off_bc = 0, off_hin = 0, off_hloc = 0, off_sumd = 0, off_tstart = 0, bytes = 0;
    // bidirectional scan: the right-to-left pass's prepared B/C and its gated
    // output (Bt, D, L) fp32; the left-to-right pass streams that output as a
    // fourth tile, with its own ring depth and shared memory
    size_t off_bc_r = 0, off_yrev = 0;
    int stages_ltr = 2;
    size_t smem_ltr = 0;
};

// Per-NT constants of the forward kernel, on the host.
int fwd_xy_bytes(int NT) {
    return 4 * (NT == 4 ? FwdLayout<4>::XY_FLOATS : NT == 2 ? FwdLayout<2>::XY_FLOATS
                                                           : FwdLayout<1>::XY_FLOATS);
}
int fwd_max_warps(int NT) { return NT == 4 ? FwdLayout<4>::kMaxWarps : FwdLayout<2>::kMaxWarps; }
int fwd_min_blocks(int NT) { return NT == 4 ? FwdLayout<4>::kMinBlocks : FwdLayout<2>::kMinBlocks; }
// registers per thread the launch bounds allow (65536 / (threads * min blocks))
int fwd_reg_cap(int NT) {
    const int threads = 32 * (fwd_max_warps(NT) + 1);
    int r = 65536 / (threads * fwd_min_blocks(NT));
    r = r > 255 ? 255 : r;
    return r & ~7;
}

// Relative cost of one state update per NT, against the per-SM rates below
// (measured with NT = 2): at the Mamba-1.4B shape 4 lanes per channel ran
// 1.5x slower than 2, and one lane per channel (4 warps, 128 channels per
// SM) 1.23x slower; the rates of one-lane warps at higher warp counts are not
// measured, so NT = 1 is taken only where NT = 2 does not apply.
double fwd_nt_cost(int NT) { return NT == 4 ? 1.5 : NT == 1 ? 1.3 : 1.0; }

// Relative throughput of one SM running `w` compute warps of the scan
// (channel-tokens per unit time), measured on the B300 with 2 lanes per
// channel: one warp per sub-partition up to 4 warps, then the sub-partitions
// holding two warps set the pace (5 warps are no faster than 4).
double fwd_sm_rate(int w) {
    static const double rate[9] = {0.0, 0.268, 0.536, 0.804, 1.071, 1.071, 1.179, 1.382, 1.396};
    if (w <= 0) return rate[1];
    return w <= 8 ? rate[w] : rate[8];
}

// Time model of one launch: `ctas` CTAs of W compute warps, each doing `work`
// units; an SM runs up to `cps` CTAs at once.  The busiest SM sets the time.
double fwd_launch_cost(int64_t ctas, int sms, int cps, int W, double work) {
    if (ctas <= 0) return 0.0;
    const int64_t k = (ctas + sms - 1) / sms;          // CTAs on the busiest SM
    const int64_t res = k < cps ? k : cps;            // resident together
    const int64_t waves = (k + res - 1) / res;
    return (double)waves * (double)res * work / fwd_sm_rate((int)(res * W));
}

// The backward sweeps' time model: one CTA per SM, full throughput from
// about 6 compute warps.
double bwd_launch_cost(int64_t ctas, int sms, int W, double work) {
    if (ctas <= 0) return 0.0;
    const int64_t waves = (ctas + sms - 1) / sms;
    double sat = (double)W / 6.0;
    if (sat > 1.0) sat = 1.0;
    return (double)waves * work / sat;
}

FwdPlan plan_fwd(const ssm_shape& s, int sm_count, bool segments = true) {
    FwdPlan pl;
    pl.NP = padded_state(s.dstate);
    const int eb = dtype_bytes(s.in_dtype);
    pl.nchunks = (s.seqlen + kT - 1) / kT;
    pl.tma_raw = (s.seqlen * eb) % 16 == 0;
    int nts[4];
    const int cnt = fwd_supported_nt(pl.NP, nts, 4);
    const int want_nt = env_int("SSM_FWD_NT", 0);
    const int want_w = env_int("SSM_FWD_W", 0);
    const int want_seg = env_int("SSM_FWD_NSEG", 0);
    const int want_cps = env_int("SSM_FWD_CPS", 0);
    double best = -1.0;
    for (int ci = 0; ci < cnt; ++ci) {
        const int NT = nts[ci];
        if (want_nt > 0 && NT != want_nt) continue;
        for (int W = 1; W <= fwd_max_warps(NT); ++W) {
            if (want_w > 0 && W != want_w) continue;
            const int CH = W * 32 / NT;
            const int64_t tiles = (s.dim + CH - 1) / CH;
            const size_t stage = (size_t)3 * CH * kT * eb + (size_t)kT * 2 * pl.NP * 4;
            const size_t xy = (size_t)W * fwd_xy_bytes(NT);
            // CTAs per SM: threads, registers, then shared memory with >= 2 stages
            int cps = 2048 / (32 * (W + 1));
            const int by_regs = 65536 / (fwd_reg_cap(NT) * 32 * (W + 1));
            if (by_regs < cps) cps = by_regs;
            if (want_cps > 0) cps = want_cps;
            while (cps > 1 && 2 * stage + xy + 2048 > (size_t)(228 * 1024) / cps) --cps;
            if (cps < 1 || 2 * stage + xy + 2048 > (size_t)kMaxSmemPerCta) continue;
            size_t avail = (size_t)(228 * 1024) / cps - 2048;
            if (avail > (size_t)kMaxSmemPerCta - 1024) avail = (size_t)kMaxSmemPerCta - 1024;
            int stages = (int)((avail - xy) / stage);
            if (stages > 4) stages = 4;
            if (stages < 2) stages = 2;
            // segments of the sequence (two passes and a carry) when there
            // are too few channel tiles to fill the GPU
            int seg_lo = 1, seg_hi = 1;
            if (want_seg > 0 && segments) seg_lo = seg_hi = want_seg;
            else if (segments && pl.nchunks >= 16 && s.batch * tiles * 2 <= (int64_t)sm_count * cps)
                seg_hi = 64;
            const int64_t nch = pl.nchunks > 0 ? pl.nchunks : 1;   // L = 0: no chunk at all
            for (int nseg0 = seg_lo; nseg0 <= seg_hi; ++nseg0) {
                int64_t nseg = nseg0;
                if (nseg > nch / 4 && want_seg <= 0) nseg = nch / 4;
                if (nseg > nch) nseg = nch;
                if (nseg < 1) nseg = 1;
                const int64_t seg_chunks = (nch + nseg - 1) / nseg;
                nseg = (nch + seg_chunks - 1) / seg_chunks;
                const double work = (double)CH * (double)seg_chunks * fwd_nt_cost(NT);
                const int64_t ctas = s.batch * tiles;
                double cost = fwd_launch_cost(ctas * nseg, sm_count, cps, W, work);
                // pass 1 costs ~0.6 of pass 2 per chunk; with the tail search it
                // runs only the last part of each segment, about 16K tokens with
                // the usual delta range (softplus of dt in [1e-3, 1e-1]): the slowest
                // state's decay reaches 2^-40 after ~29 units of accumulated delta
                double sfrac = 0.6;
                if (pl.tma_raw) {
                    const double tail = 16384.0 / ((double)seg_chunks * kT);
                    sfrac *= tail < 1.0 ? tail : 1.0;
                }
                if (nseg > 1) cost += sfrac * fwd_launch_cost(ctas * (nseg - 1), sm_count, cps, W, work);
                // near-ties go to the plan that keeps more SMs busy: with the
                // inputs cold in L2 (a fresh batch), plans that leave SMs idle
                // measured up to 20 % slower than the model says
                const double busy = (double)(ctas * nseg < sm_count ? ctas * nseg : sm_count) / sm_count;
                cost *= 1.0 + 0.05 * (1.0 - busy);
                if (best < 0.0 || cost < best * 0.999) {
                    best = cost;
                    pl.NT = NT; pl.W = W; pl.CH = CH; pl.stages = stages;
                    pl.smem = (size_t)stages * stage + xy + 1024;
                    pl.seg_chunks = seg_chunks > 0 ? seg_chunks : 1;
                    pl.nseg = (int)nseg;
                }
            }
        }
    }
    if (best < 0.0) {   // nothing fitted the overrides: the smallest configuration
        pl.NT = nts[0]; pl.W = 1; pl.CH = 32 / pl.NT; pl.stages = 2;
        pl.smem = 2 * ((size_t)3 * pl.CH * kT * eb + (size_t)kT * 2 * pl.NP * 4) +
                  fwd_xy_bytes(pl.NT) + 1024;
        pl.seg_chunks = pl.nchunks > 0 ? pl.nchunks : 1;
        pl.nseg = 1;
    }

    size_t off = kHeaderBytes;
    pl.off_bc = off;
    off += align256((size_t)s.batch * s.seqlen * 2 * pl.NP * 4);
    if (pl.nseg > 1) {
        const size_t st = (size_t)pl.nseg * s.batch * s.dim;
        pl.off_hin = off;
        off += align256(st * pl.NP * 4);
        pl.off_hloc = off;
        off += align256(st * pl.NP * 4);
        pl.off_sumd = off;
        off += align256(st * 4);
        pl.off_tstart = off;
        off += align256((size_t)pl.nseg * s.batch * ((s.dim + pl.CH - 1) / pl.CH) * 4);
    }
    pl.bytes = off;
    if (env_int("SSM_DEBUG_PLAN", 0))
        std::fprintf(stderr, "ssm fwd plan: NP=%d NT=%d W=%d CH=%d stages=%d smem=%zu nseg=%d seg_chunks=%lld\n",
                     pl.NP, pl.NT, pl.W, pl.CH, pl.stages, pl.smem, pl.nseg, (long long)pl.seg_chunks);
    return pl;
}

// The bidirectional scan: both directions share the plan, including the
// two-pass split of a long row with few channels (each direction runs its own
// summaries and carry, the right-to-left one from the last segment down).
FwdPlan plan_fwd_bidir(const ssm_shape& s, int sm_count) {
    FwdPlan pl = plan_fwd(s, sm_count, true);
    // the left-to-right pass's stage holds an fp32 tile of the other
    // direction's output besides u, delta_raw, z and B/C
    {
        const int eb = dtype_bytes(s.in_dtype);
        const size_t stage = (size_t)3 * pl.CH * kT * eb + (size_t)kT * 2 * pl.NP * 4 +
                             (size_t)pl.CH * kT * 4;
        const size_t xy = (size_t)pl.W * fwd_xy_bytes(pl.NT);
        const size_t avail = (size_t)kMaxSmemPerCta - 1024 - xy;
        int st = (int)(avail / stage);
        if (st > 4) st = 4;
        pl.stages_ltr = st;   // < 2: refused by the caller
        pl.smem_ltr = (size_t)(st > 0 ? st : 0) * stage + xy + 1024;
    }
    size_t off = pl.bytes;
    pl.off_bc_r = off;
    off += align256((size_t)s.batch * s.seqlen * 2 * pl.NP * 4);
    pl.off_yrev = off;
    off += align256((size_t)s.batch * s.dim * s.seqlen * 4);
    pl.bytes = off;
    return pl;
}

// Backward plan: the two sweeps need the prepared B/C (state size padded to
// at least 8), one fp32 number per (batch, channel, token), the final state
// and the state at the end of every 64-token chunk.  Channel tiles of W
// compute warps, one CTA per SM, chosen like the forward's.  Long sequences
// with too few channel tiles to fill the GPU are cut into segments: the
// forward's summary pass and carry give each segment its initial state, the
// adjoint summary and a right-to-left carry the adjoint entering it from the
// right, and a carry after the forward sweep adds the dA terms of the
// tangent crossing segment boundaries.
struct BwdPlan {
    int NP = 16, NT = 2, W = 4, CH = 32;
    int stages_f = 2, stages_r = 2, stages_l = 2;
    size_t smem_f = 0, smem_r = 0, smem_l = 0;
    bool tma_raw = false;
    bool ok = false;        // a tile shape fits the shared memory
    int nseg = 1;
    int64_t seg_chunks = 0;
    int fwd_tiles = 0;      // channel tiles of the forward summary pass (segments)
    size_t off_bc = 0, off_phi = 0, off_hfin = 0, off_hck = 0, off_hprev = 0, bytes = 0;
    // segments: forward summary (initial states, end states from zero, sums
    // of delta2, tail-search starts), adjoint summary and carry, tangent sums
    size_t off_hin = 0, off_hloc = 0, off_sumd = 0, off_tstart = 0, off_lamloc = 0,
           off_lamin = 0, off_sumdr = 0, off_kstop = 0, off_gp = 0, off_mend = 0;
};

int bwd_tbuf_floats(int NT, int NP) {
    if (NT == 2) return NP == 8 ? BwdLayout<2, 8>::TBUF : NP == 16 ? BwdLayout<2, 16>::TBUF
                                                                  : BwdLayout<2, 32>::TBUF;
    return NP == 16 ? BwdLayout<4, 16>::TBUF : NP == 32 ? BwdLayout<4, 32>::TBUF
                                                        : BwdLayout<4, 64>::TBUF;
}

BwdPlan plan_bwd(const ssm_shape& s, int sm_count, bool segments = true) {
    BwdPlan pl;
    pl.NP = padded_state(s.dstate);
    if (pl.NP < 8) pl.NP = 8;
    const int eb = dtype_bytes(s.in_dtype);
    pl.tma_raw = (s.seqlen * eb) % 16 == 0;
    const int64_t nchunks = (s.seqlen + kT - 1) / kT;
    // segments are built for 9..16 states and 16-byte token rows
    const bool seg_ok = segments && pl.NP == 16 && pl.tma_raw && nchunks >= 16;
    const int nts_all[2] = {2, 4};
    int want_nt = env_int("SSM_BWD_NT", 0);
    int want_w = env_int("SSM_BWD_W", 0);
    const int want_seg = env_int("SSM_BWD_NSEG", 0);
    double best = -1.0;
    // a second search without the overrides when none of them fits
    for (int attempt = 0; attempt < 2 && best < 0.0; ++attempt) {
    if (attempt == 1) want_nt = want_w = 0;
    for (int ni = 0; ni < 2; ++ni) {
        const int NT = nts_all[ni];
        if (pl.NP == 8 && NT != 2) continue;       // G = NP / NT must be 4, 8 or 16
        if (pl.NP >= 32 && NT != 4) continue;
        if (want_nt > 0 && NT != want_nt) continue;
        for (int W = 1; W <= BwdLayout<2, 16>::kMaxWarps; ++W) {
            if (want_w > 0 && W != want_w) continue;
            const int CH = W * 32 / NT;
            const size_t raw = (size_t)CH * kT * eb, rawf = (size_t)CH * kT * 4;
            const size_t bcb = (size_t)kT * 2 * pl.NP * 4;
            const size_t fixed = (size_t)2 * W * pl.NP * kT * 4 + (size_t)W * bwd_tbuf_floats(NT, pl.NP) * 4 + 1024;
            const size_t stf = 4 * raw + bcb, str = 4 * raw + rawf + bcb;
            if (2 * str + fixed > (size_t)kMaxSmemPerCta) continue;
            const int64_t tiles = (s.dim + CH - 1) / CH;
            const int64_t ctas = s.batch * tiles;
            const double work = (double)CH * (NT == 4 ? 1.15 : 1.0);
            // segments (when the channel tiles leave SMs idle): the sweeps over
            // seg_chunks chunks each, ~4 % more work in the forward sweep, and
            // the two summary passes over all segments but one at about a
            // quarter of the sweeps' cost per chunk
            int seg_lo = 1, seg_hi = 1;
            if (seg_ok && want_seg > 0) seg_lo = seg_hi = want_seg;
            else if (seg_ok && ctas < sm_count) seg_hi = 64;
            const int64_t nch = nchunks > 0 ? nchunks : 1;   // L = 0: no chunk at all
            for (int nseg0 = seg_lo; nseg0 <= seg_hi; ++nseg0) {
            int64_t nseg = nseg0 > nch ? nch : nseg0;
            if (nseg < 1) nseg = 1;
            const int64_t seg_chunks = (nch + nseg - 1) / nseg;
            nseg = (nch + seg_chunks - 1) / seg_chunks;
            const double frac = (double)seg_chunks / (double)nch;
            double cost = bwd_launch_cost(ctas * nseg, sm_count, W, work * frac);
            if (nseg > 1)
                cost = 1.04 * cost + 0.25 * bwd_launch_cost(ctas * (nseg - 1), sm_count, W, work * frac);
            if (best < 0.0 || cost < best * 0.999) {
                best = cost;
                pl.NT = NT; pl.W = W; pl.CH = CH;
                pl.nseg = (int)nseg;
                pl.seg_chunks = seg_chunks;
                int sf = (int)(((size_t)kMaxSmemPerCta - fixed) / stf);
                int sr = (int)(((size_t)kMaxSmemPerCta - fixed) / str);
                pl.stages_f = sf > 4 ? 4 : sf;
                pl.stages_r = sr > 4 ? 4 : sr;
                pl.smem_f = (size_t)pl.stages_f * stf + fixed;
                pl.smem_r = (size_t)pl.stages_r * str + fixed;
                // the adjoint summary: the forward sweep's tiles, no buffers
                int sl = (int)(((size_t)kMaxSmemPerCta - 1024) / stf);
                pl.stages_l = sl > 4 ? 4 : sl;
                pl.smem_l = (size_t)pl.stages_l * stf + 1024;
            }
            }
        }
    }
    }
    pl.ok = best >= 0.0;
    size_t off = kHeaderBytes;
    pl.off_bc = off;
    off += align256((size_t)s.batch * s.seqlen * 2 * pl.NP * 4);
    pl.off_phi = off;
    off += align256((size_t)s.batch * s.dim * s.seqlen * 4);
    pl.off_hfin = off;
    off += align256((size_t)s.batch * s.dim * pl.NP * 4);
    pl.off_hck = off;
    off += align256((size_t)s.batch * s.dim * ((s.seqlen + kT - 1) / kT) * pl.NP * 4);
    // fp32 inputs: the state before every token (the reverse sweep forms the
    // h-dependent term of ddelta from it directly)
    pl.off_hprev = off;
    if (s.in_dtype == SSM_F32) off += align256((size_t)s.batch * s.dim * s.seqlen * pl.NP * 4);
    if (pl.nseg > 1) {
        const size_t st = (size_t)pl.nseg * s.batch * s.dim * pl.NP * 4;
        const size_t sd = (size_t)pl.nseg * s.batch * s.dim * 4;
        // the forward summary pass on the tiles of the forward's own segmented plan
        const FwdPlan fp = plan_fwd(s, sm_count, true);
        pl.fwd_tiles = (int)((s.dim + fp.CH - 1) / fp.CH);
        const int64_t bwd_tiles = (s.dim + pl.CH - 1) / pl.CH;
        pl.off_hin = off;    off += align256(st);
        pl.off_hloc = off;   off += align256(st);
        pl.off_sumd = off;   off += align256(sd);
        pl.off_tstart = off; off += align256((size_t)pl.nseg * s.batch * pl.fwd_tiles * 4);
        pl.off_lamloc = off; off += align256(st);
        pl.off_lamin = off;  off += align256(st);
        pl.off_sumdr = off;  off += align256(sd);
        pl.off_kstop = off;  off += align256((size_t)pl.nseg * s.batch * bwd_tiles * 4);
        pl.off_gp = off;     off += align256(st);
        pl.off_mend = off;   off += align256(st);
    } else {
        pl.seg_chunks = nchunks;
    }
    pl.bytes = off;
    if (env_int("SSM_DEBUG_PLAN", 0))
        std::fprintf(stderr, "ssm bwd plan: NP=%d NT=%d W=%d CH=%d stages=%d/%d/%d smem=%zu/%zu/%zu nseg=%d x %lld\n",
                     pl.NP, pl.NT, pl.W, pl.CH, pl.stages_f, pl.stages_r, pl.stages_l, pl.smem_f,
                     pl.smem_r, pl.smem_l, pl.nseg, (long long)pl.seg_chunks);
    return pl;
}

// Workspace of the bidirectional backward: the status word, one backward
// workspace (fp32 per-token outputs) reused by the two directions in turn,
// token-reversed copies of the right-to-left direction's inputs, and the
// fp32 per-token gradients of both directions before they are combined.
struct BidirBwdLayout {
    size_t off_inner = 0, inner = 0, off_u = 0, off_dr = 0, off_z = 0, off_dy = 0, off_B = 0,
           off_C = 0, off_g = 0, off_dB = 0, off_dC = 0, bytes = 0;
};
BidirBwdLayout bidir_bwd_layout(const ssm_shape& s, int sm_count) {
    BidirBwdLayout w;
    ssm_shape s32 = s;
    s32.out_dtype = SSM_F32;
    const size_t tok = (size_t)s.batch * s.dim * s.seqlen;
    const size_t bnl = (size_t)s.batch * s.dstate * s.seqlen;
    const size_t eb = s.in_dtype == SSM_BF16 ? 2 : 4;
    size_t off = kHeaderBytes;
    w.off_inner = off;
    w.inner = plan_bwd(s32, sm_count).bytes;
    off += align256(w.inner);
    w.off_u = off;  off += align256(tok * eb);
    w.off_dr = off; off += align256(tok * eb);
    w.off_z = off;  off += align256(tok * eb);
    w.off_dy = off; off += align256(tok * eb);
    w.off_B = off;  off += align256(bnl * eb);
    w.off_C = off;  off += align256(bnl * eb);
    w.off_g = off;  off += 6 * align256(tok * 4);   // du, ddr, dz of each direction
    w.off_dB = off; off += align256(bnl * 4);
    w.off_dC = off; off += align256(bnl * 4);
    w.bytes = off;
    return w;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// 2-D row-major tensor (rows x cols elements), tile box_cols x box_rows.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t cols,
              uint64_t rows, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * (cuuint64_t)esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// rows x 16 fp32 (64-byte rows), box 16 x 128, 64-byte swizzle: the decode
// step's state and A tiles
bool make_map_swz64(CUtensorMap* m, const void* base, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {16, rows};
    cuuint64_t strides[1] = {64};
    cuuint32_t box[2] = {16, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t launch_fwd(const FwdPlan& pl, int tin, int tout, bool summary, bool conv, bool varlen,
                       const FwdParams& p, const FwdMaps& m, dim3 grid, cudaStream_t st) {
    if (varlen)
        return launch_fwd_varlen_np16(pl.NT, tin, tout, summary, conv, p, m, grid, pl.W, pl.smem, st);
    if (conv) return launch_fwd_conv_np16(pl.NT, tin, tout, summary, p, m, grid, pl.W, pl.smem, st);
    switch (pl.NP) {
        case 4: return launch_fwd_np4(pl.NT, tin, tout, summary, pl.tma_raw, p, m, grid, pl.W, pl.smem, st);
        case 8: return launch_fwd_np8(pl.NT, tin, tout, summary, pl.tma_raw, p, m, grid, pl.W, pl.smem, st);
        case 16: return launch_fwd_np16(pl.NT, tin, tout, summary, pl.tma_raw, p, m, grid, pl.W, pl.smem, st);
        case 32: return launch_fwd_np32(pl.NT, tin, tout, summary, pl.tma_raw, p, m, grid, pl.W, pl.smem, st);
        default: return launch_fwd_np64(pl.NT, tin, tout, summary, pl.tma_raw, p, m, grid, pl.W, pl.smem, st);
    }
}

cudaError_t launch_bwd(const BwdPlan& pl, int tin, int tout, const BwdParams& p, const BwdMaps& m,
                       dim3 grid, cudaStream_t st) {
    BwdLaunch lc;
    lc.grid = grid;
    lc.warps = pl.W;
    lc.stages_f = pl.stages_f;
    lc.stages_r = pl.stages_r;
    lc.smem_f = pl.smem_f;
    lc.smem_r = pl.smem_r;
    switch (pl.NP) {
        case 8: return launch_bwd_np8(pl.NT, tin, tout, pl.tma_raw, p, m, lc, st);
        case 16: return launch_bwd_np16(pl.NT, tin, tout, pl.tma_raw, p, m, lc, st);
        case 32: return launch_bwd_np32(pl.NT, tin, tout, pl.tma_raw, p, m, lc, st);
        default: return launch_bwd_np64(pl.NT, tin, tout, pl.tma_raw, p, m, lc, st);
    }
}

}  // namespace

namespace ssm {
int fwd_supported_nt(int NP, int* out, int cap) {
    static const int t4[] = {1}, t8[] = {2, 1}, t16[] = {2, 4, 1}, t32[] = {4, 2}, t64[] = {4};
    const int* t = t16;
    int n = 3;
    switch (NP) {
        case 4: t = t4; n = 1; break;
        case 8: t = t8; n = 2; break;
        case 16: t = t16; n = 3; break;
        case 32: t = t32; n = 2; break;
        default: t = t64; n = 1; break;
    }
    for (int i = 0; i < n && i < cap; ++i) out[i] = t[i];
    return n < cap ? n : cap;
}
}  // namespace ssm

extern "C" {

const char* ssm_strerror(int code) {
    switch (code) {
        case SSM_OK: return "ok";
        case SSM_ERR_NULL: return "a required pointer is NULL";
        case SSM_ERR_SHAPE: return "invalid shape (negative size, dstate outside 1..64, or overflow)";
        case SSM_ERR_DTYPE: return "invalid dtype";
        case SSM_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case SSM_ERR_WORKSPACE: return "workspace missing or too small";
        case SSM_ERR_CUDA: return "a CUDA runtime call failed";
        case SSM_ERR_TIMEOUT: return "device-side bounded wait expired";
        case SSM_ERR_UNSUPPORTED: return "unsupported request";
        case SSM_ERR_SEQLENS: return "packed-sequence starts out of order or out of range";
        default: return "unknown status";
    }
}

// The backward fed by the conv prologue: the whole-row plan, then the
// sweeps' fp32 du, which the prologue's reverse mode reads.
static size_t conv_bwd_du_offset(const BwdPlan& pl) { return align256(pl.bytes); }
static size_t conv_bwd_bytes(const ssm_shape& s, int sm_count) {
    const BwdPlan pl = plan_bwd(s, sm_count, false);
    return conv_bwd_du_offset(pl) + align256((size_t)s.batch * s.dim * s.seqlen * 4);
}

size_t ssm_scan_workspace_bytes(const ssm_shape* shape, int for_backward) {
    if (shape_check(shape) != SSM_OK) return 0;
    const size_t bytes = for_backward == 4 ? conv_bwd_bytes(*shape, device_sm_count())
                         : for_backward == 3 ? bidir_bwd_layout(*shape, device_sm_count()).bytes
                         : for_backward == 2 ? plan_fwd_bidir(*shape, device_sm_count()).bytes
                         : for_backward ? plan_bwd(*shape, device_sm_count()).bytes
                                        : plan_fwd(*shape, device_sm_count()).bytes;
    return bytes < kHeaderBytes ? kHeaderBytes : bytes;
}

// The forward, with or without the conv prologue (conv_w non-null: `u` is the
// branch input x and u = silu(causal depthwise conv of x)), over whole rows
// or over packed sequences (cu_seqlens non-null).
static int scan_fwd_impl(const ssm_shape* shape, const void* u, const float* conv_w,
                         const float* conv_b, int conv_k, const int32_t* cu_seqlens, int nseq,
                         const void* delta_raw, const float* A,
                         const void* B, const void* C, const float* D, const void* z,
                         const float* delta_bias, const float* h0, void* y, float* hL,
                         void* workspace, size_t ws_bytes, ssm_stream_t stream) {
    const int sc = shape_check(shape);
    if (sc != SSM_OK) return sc;
    const ssm_shape s = *shape;
    const int64_t Bt = s.batch, Dm = s.dim, N = s.dstate, L = s.seqlen;
    const bool conv = conv_w != nullptr;
    const bool varlen = cu_seqlens != nullptr;
    const bool any_work = Bt > 0 && Dm > 0;
    if (!any_work) return SSM_OK;
    if (!A || !workspace) return !A ? SSM_ERR_NULL : SSM_ERR_WORKSPACE;
    if (L > 0 && (!u || !delta_raw || !B || !C || !y)) return SSM_ERR_NULL;
    const void* ptrs[] = {u, delta_raw, A, B, C, D, z, delta_bias, h0, y, hL, workspace, conv_w, conv_b};
    if (varlen && ((uintptr_t)cu_seqlens % 4) != 0) return SSM_ERR_ALIGN;
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const FwdPlan pl = plan_fwd(s, device_sm_count());
    // the conv prologue is built for 9..16 states and 16-byte token rows
    if ((conv || varlen) && L > 0 && (pl.NP != 16 || !pl.tma_raw)) return SSM_ERR_UNSUPPORTED;
    if (ws_bytes < pl.bytes) return SSM_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws);

    const int64_t per_seq = Bt * Dm * N;   // floats of one sequence's state (packed h0, hL)
    if (L == 0 && varlen) {
        if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return cuda_fail();
        if (launch_varlen_prep(cu_seqlens, nseq, 0, per_seq, h0, hL, status, st) != cudaSuccess)
            return cuda_fail();
        return SSM_OK;
    }
    if (L == 0) {
        if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return cuda_fail();
        if (hL) {
            const size_t bytes = (size_t)(Bt * Dm * N) * sizeof(float);
            cudaError_t e = h0 ? cudaMemcpyAsync(hL, h0, bytes, cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(hL, 0, bytes, st);
            if (e != cudaSuccess) return cuda_fail();
        }
        return SSM_OK;
    }

    float* bc = reinterpret_cast<float*>(ws + pl.off_bc);
    if (launch_prep_bc(s.in_dtype, Bt, (int)N, pl.NP, L, B, C, bc, status, st) != cudaSuccess)
        return cuda_fail();
    if (varlen && launch_varlen_prep(cu_seqlens, nseq, L, per_seq, h0, hL, status, st) != cudaSuccess)
        return cuda_fail();

    const int eb = dtype_bytes(s.in_dtype);
    const CUtensorMapDataType tdt =
        s.in_dtype == SSM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    FwdMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!make_map(&maps.bc, bc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2 * pl.NP, Bt * L, 2 * pl.NP, kT,
                  false))
        return cuda_fail();
    if (pl.tma_raw) {
        const uint32_t box_t = 128 / eb;
        if (!make_map(&maps.u, u, tdt, eb, L, Bt * Dm, box_t, pl.CH, true) ||
            !make_map(&maps.dr, delta_raw, tdt, eb, L, Bt * Dm, box_t, pl.CH, true) ||
            (z && !make_map(&maps.z, z, tdt, eb, L, Bt * Dm, box_t, pl.CH, true)))
            return cuda_fail();
    }

    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.Bt = Bt; p.D = Dm; p.L = L; p.N = (int)N;
    p.u = u; p.dr = delta_raw; p.z = z; p.A = A; p.Dv = D; p.bias = delta_bias; p.h0 = h0;
    p.bc = bc; p.y = y; p.hL = hL;
    p.seg_chunks = pl.seg_chunks;
    p.nseg = pl.nseg;
    p.stages = pl.stages;
    p.status = status;
    p.timeout_ns = kDefaultTimeoutNs;
    p.conv_w = conv_w;
    p.conv_b = conv_b;
    p.conv_k = conv_k;
    p.cu_seqlens = cu_seqlens;
    p.nseq = nseq;
    const unsigned gx = (unsigned)((Dm + pl.CH - 1) / pl.CH);

    if (pl.nseg > 1) {
        p.hin = reinterpret_cast<float*>(ws + pl.off_hin);
        p.hloc = reinterpret_cast<float*>(ws + pl.off_hloc);
        p.sumd = reinterpret_cast<float*>(ws + pl.off_sumd);
        // pass 1: summaries of every segment but the last, each from the
        // chunk the tail search finds (it needs 16-byte row loads)
        FwdParams p1 = p;
        p1.hin = nullptr;
        if (pl.tma_raw) {
            int* tstart = reinterpret_cast<int*>(ws + pl.off_tstart);
            if (launch_tail(s.in_dtype, p, pl.CH, gx, tstart, p.sumd, st) != cudaSuccess)
                return cuda_fail();
            p1.tstart = tstart;
        }
        if (launch_fwd(pl, s.in_dtype, s.out_dtype, true, conv, varlen, p1, maps,
                       dim3(gx, (unsigned)Bt, (unsigned)(pl.nseg - 1)), st) != cudaSuccess)
            return cuda_fail();
        if (launch_carry(Bt, Dm, (int)N, pl.NP, pl.nseg, A, h0, p.hloc, p.sumd, p.hin, st) !=
            cudaSuccess)
            return cuda_fail();
    }
    if (launch_fwd(pl, s.in_dtype, s.out_dtype, false, conv, varlen, p, maps,
                   dim3(gx, (unsigned)Bt, (unsigned)pl.nseg), st) != cudaSuccess)
        return cuda_fail();
    return SSM_OK;
}

int ssm_scan_fwd(const ssm_shape* shape, const void* u, const void* delta_raw, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, const float* h0, void* y, float* hL, void* workspace,
                 size_t ws_bytes, ssm_stream_t stream) {
    return scan_fwd_impl(shape, u, nullptr, nullptr, 0, nullptr, 0, delta_raw, A, B, C, D, z,
                         delta_bias, h0, y, hL, workspace, ws_bytes, stream);
}

int ssm_scan_fwd_conv(const ssm_shape* shape, const void* x, const float* conv_w,
                      const float* conv_b, int conv_k, const void* delta_raw, const float* A,
                      const void* B, const void* C, const float* D, const void* z,
                      const float* delta_bias, const float* h0, void* y, float* hL,
                      void* workspace, size_t ws_bytes, ssm_stream_t stream) {
    if (!conv_w) return SSM_ERR_NULL;
    if (conv_k < 1 || conv_k > 4) return SSM_ERR_SHAPE;
    return scan_fwd_impl(shape, x, conv_w, conv_b, conv_k, nullptr, 0, delta_raw, A, B, C, D, z,
                         delta_bias, h0, y, hL, workspace, ws_bytes, stream);
}

int ssm_scan_fwd_bidir(const ssm_shape* shape, const void* u, const void* z,
                       const void* delta_raw, const float* A, const void* B, const void* C,
                       const float* D, const float* delta_bias, const float* h0,
                       const void* delta_raw_r, const float* A_r, const void* B_r, const void* C_r,
                       const float* D_r, const float* delta_bias_r, const float* h0_r,
                       void* y, float* hL, float* hL_r, void* workspace, size_t ws_bytes,
                       ssm_stream_t stream) {
    const int sc = shape_check(shape);
    if (sc != SSM_OK) return sc;
    const ssm_shape s = *shape;
    const int64_t Bt = s.batch, Dm = s.dim, N = s.dstate, L = s.seqlen;
    if (Bt == 0 || Dm == 0) return SSM_OK;
    if (!A || !A_r) return SSM_ERR_NULL;
    if (!workspace) return SSM_ERR_WORKSPACE;
    if (L > 0 && (!u || !delta_raw || !B || !C || !delta_raw_r || !B_r || !C_r || !y))
        return SSM_ERR_NULL;
    const void* ptrs[] = {u, z, delta_raw, A, B, C, D, delta_bias, h0, delta_raw_r, A_r, B_r,
                          C_r, D_r, delta_bias_r, h0_r, y, hL, hL_r, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const FwdPlan pl = plan_fwd_bidir(s, device_sm_count());
    // built for 9..16 states and 16-byte token rows
    if (L > 0 && (pl.NP != 16 || !pl.tma_raw || pl.stages_ltr < 2)) return SSM_ERR_UNSUPPORTED;
    if (ws_bytes < pl.bytes) return SSM_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws);
    if (L == 0) {
        if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return cuda_fail();
        const size_t bytes = (size_t)(Bt * Dm * N) * sizeof(float);
        const float* h0s[2] = {h0, h0_r};
        float* hLs[2] = {hL, hL_r};
        for (int i = 0; i < 2; ++i) {
            if (!hLs[i]) continue;
            cudaError_t e = h0s[i] ? cudaMemcpyAsync(hLs[i], h0s[i], bytes, cudaMemcpyDeviceToDevice, st)
                                   : cudaMemsetAsync(hLs[i], 0, bytes, st);
            if (e != cudaSuccess) return cuda_fail();
        }
        return SSM_OK;
    }
    float* bc = reinterpret_cast<float*>(ws + pl.off_bc);
    float* bc_r = reinterpret_cast<float*>(ws + pl.off_bc_r);
    float* yrev = reinterpret_cast<float*>(ws + pl.off_yrev);
    if (launch_prep_bc(s.in_dtype, Bt, (int)N, pl.NP, L, B, C, bc, status, st) != cudaSuccess ||
        launch_prep_bc(s.in_dtype, Bt, (int)N, pl.NP, L, B_r, C_r, bc_r, nullptr, st) != cudaSuccess)
        return cuda_fail();

    const int eb = dtype_bytes(s.in_dtype);
    const CUtensorMapDataType tdt =
        s.in_dtype == SSM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const uint32_t box_t = 128 / eb;
    FwdMaps mf, mr;
    std::memset(&mf, 0, sizeof(mf));
    std::memset(&mr, 0, sizeof(mr));
    if (!make_map(&mf.bc, bc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2 * pl.NP, Bt * L, 2 * pl.NP, kT, false) ||
        !make_map(&mr.bc, bc_r, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2 * pl.NP, Bt * L, 2 * pl.NP, kT, false) ||
        !make_map(&mf.u, u, tdt, eb, L, Bt * Dm, box_t, pl.CH, true) ||
        !make_map(&mf.dr, delta_raw, tdt, eb, L, Bt * Dm, box_t, pl.CH, true) ||
        !make_map(&mr.dr, delta_raw_r, tdt, eb, L, Bt * Dm, box_t, pl.CH, true) ||
        (z && !make_map(&mf.z, z, tdt, eb, L, Bt * Dm, box_t, pl.CH, true)) ||
        !make_map(&mf.ya, yrev, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, L, Bt * Dm, 32, pl.CH, true))
        return cuda_fail();
    mr.u = mf.u;
    mr.z = mf.z;

    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.Bt = Bt; p.D = Dm; p.L = L; p.N = (int)N;
    p.u = u; p.z = z;
    p.seg_chunks = pl.seg_chunks;
    p.nseg = pl.nseg;
    p.stages = pl.stages;
    p.status = status;
    p.timeout_ns = kDefaultTimeoutNs;
    FwdParams pr = p;   // right to left: fp32 gated output into the workspace
    pr.dr = delta_raw_r; pr.A = A_r; pr.Dv = D_r; pr.bias = delta_bias_r; pr.h0 = h0_r;
    pr.bc = bc_r; pr.y = yrev; pr.hL = hL_r;
    FwdParams pf = p;   // left to right, adding it (streamed through the ring)
    pf.dr = delta_raw; pf.A = A; pf.Dv = D; pf.bias = delta_bias; pf.h0 = h0;
    pf.bc = bc; pf.y = y; pf.hL = hL; pf.yadd = yrev;
    pf.stages = pl.stages_ltr;
    const unsigned gx = (unsigned)((Dm + pl.CH - 1) / pl.CH);
    const unsigned nseg = (unsigned)pl.nseg;
    if (nseg > 1) {
        // segmented plan, right to left first: summaries of segments 1 ..
        // nseg-1 (each from a zero state at its right end), the carry from the
        // last segment down, then every segment from its initial state
        pr.hin = reinterpret_cast<float*>(ws + pl.off_hin);
        pr.hloc = reinterpret_cast<float*>(ws + pl.off_hloc);
        pr.sumd = reinterpret_cast<float*>(ws + pl.off_sumd);
        FwdParams pr1 = pr;
        pr1.hin = nullptr;
        pr1.seg0 = 1;
        if (launch_fwd_bidir_np16(pl.NT, s.in_dtype, SSM_F32, 1, true, pr1, mr, dim3(gx, (unsigned)Bt, nseg - 1),
                                  pl.W, pl.smem, st) != cudaSuccess ||
            launch_carry(Bt, Dm, (int)N, pl.NP, pl.nseg, A_r, h0_r, pr.hloc, pr.sumd, pr.hin, st,
                         true) != cudaSuccess)
            return cuda_fail();
    }
    if (launch_fwd_bidir_np16(pl.NT, s.in_dtype, SSM_F32, 1, false, pr, mr, dim3(gx, (unsigned)Bt, nseg),
                              pl.W, pl.smem, st) != cudaSuccess)
        return cuda_fail();
    if (nseg > 1) {
        // left to right: the plain forward's summaries (with its tail search) and carry
        pf.hin = pr.hin;
        pf.hloc = pr.hloc;
        pf.sumd = pr.sumd;
        FwdParams pf1 = pf;
        pf1.hin = nullptr;
        pf1.stages = pl.stages;
        int* tstart = reinterpret_cast<int*>(ws + pl.off_tstart);
        if (launch_tail(s.in_dtype, pf, pl.CH, gx, tstart, pf.sumd, st) != cudaSuccess)
            return cuda_fail();
        pf1.tstart = tstart;
        if (launch_fwd(pl, s.in_dtype, s.out_dtype, true, false, false, pf1, mf,
                       dim3(gx, (unsigned)Bt, nseg - 1), st) != cudaSuccess ||
            launch_carry(Bt, Dm, (int)N, pl.NP, pl.nseg, A, h0, pf.hloc, pf.sumd, pf.hin, st) !=
                cudaSuccess)
            return cuda_fail();
    }
    if (launch_fwd_bidir_np16(pl.NT, s.in_dtype, s.out_dtype, 2, false, pf, mf, dim3(gx, (unsigned)Bt, nseg),
                              pl.W, pl.smem_ltr, st) != cudaSuccess)
        return cuda_fail();
    return SSM_OK;
}

int ssm_scan_fwd_varlen(const ssm_shape* shape, const void* u, const int32_t* cu_seqlens, int nseq,
                        const float* conv_w, const float* conv_b, int conv_k,
                        const void* delta_raw, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* delta_bias, const float* h0,
                        void* y, float* hL, void* workspace, size_t ws_bytes,
                        ssm_stream_t stream) {
    if (!cu_seqlens) return SSM_ERR_NULL;
    if (nseq < 1) return SSM_ERR_SHAPE;
    if (conv_w && (conv_k < 1 || conv_k > 4)) return SSM_ERR_SHAPE;
    if (!conv_w) conv_k = 0;
    return scan_fwd_impl(shape, u, conv_w, conv_w ? conv_b : nullptr, conv_k, cu_seqlens, nseq,
                         delta_raw, A, B, C, D, z, delta_bias, h0, y, hL, workspace, ws_bytes,
                         stream);
}

// The conv prologue's part of a backward call: u is then the branch input x,
// and dx, dconv_w, dconv_b replace du.
struct ConvBwd {
    const float* w;
    const float* b;
    int k;
    void* dx;
    float* dw;
    float* db;
};

// The backward, over whole rows or over packed sequences (cu_seqlens non-null),
// or fed by the conv prologue (conv non-null; whole rows).
static int scan_bwd_impl(const ssm_shape* shape, const void* u, const int32_t* cu_seqlens,
                         int nseq, const void* delta_raw, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* delta_bias,
                         const float* h0, const void* dy, const float* dhL, void* du,
                         void* ddelta_raw, float* dA, float* dB, float* dC, float* dD, void* dz,
                         float* ddelta_bias, float* dh0, void* workspace, size_t ws_bytes,
                         ssm_stream_t stream, const ConvBwd* conv = nullptr) {
    const int sc = shape_check(shape);
    if (sc != SSM_OK) return sc;
    const ssm_shape s = *shape;
    const int64_t Bt = s.batch, Dm = s.dim, N = s.dstate, L = s.seqlen;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen && nseq < 1) return SSM_ERR_SHAPE;
    if (varlen && ((uintptr_t)cu_seqlens % 4) != 0) return SSM_ERR_ALIGN;
    if (Dm > 0 && !A) return SSM_ERR_NULL;
    if (Dm > 0 && !dA) return SSM_ERR_NULL;
    if (conv) {
        if (!conv->w || !conv->dw) return SSM_ERR_NULL;
        if (conv->k < 1 || conv->k > 4) return SSM_ERR_SHAPE;
        const void* cp[] = {conv->w, conv->b, conv->dx, conv->dw, conv->db};
        for (const void* q : cp)
            if (q && !aligned16(q)) return SSM_ERR_ALIGN;
        // the prologue's parameter gradients are sums: they start at zero
        cudaStream_t st0 = static_cast<cudaStream_t>(stream);
        if (Dm > 0 && (cudaMemsetAsync(conv->dw, 0, (size_t)(Dm * conv->k) * 4, st0) != cudaSuccess ||
                       (conv->db && cudaMemsetAsync(conv->db, 0, (size_t)Dm * 4, st0) != cudaSuccess)))
            return cuda_fail();
        if (L > 0 && Bt > 0 && Dm > 0 && !conv->dx) return SSM_ERR_NULL;
    }
    if (Bt == 0 || Dm == 0) {
        // nothing flows; gradients of the per-channel parameters are zero
        cudaStream_t st0 = static_cast<cudaStream_t>(stream);
        const void* ptrs0[] = {A, dA, dD, ddelta_bias};
        for (const void* q : ptrs0)
            if (q && !aligned16(q)) return SSM_ERR_ALIGN;
        if (dA && cudaMemsetAsync(dA, 0, (size_t)(Dm * N) * 4, st0) != cudaSuccess) return cuda_fail();
        if (dD && cudaMemsetAsync(dD, 0, (size_t)Dm * 4, st0) != cudaSuccess) return cuda_fail();
        if (ddelta_bias && cudaMemsetAsync(ddelta_bias, 0, (size_t)Dm * 4, st0) != cudaSuccess)
            return cuda_fail();
        if (Bt > 0 && L > 0 && dB && dC) {
            if (cudaMemsetAsync(dB, 0, (size_t)(Bt * N * L) * 4, st0) != cudaSuccess ||
                cudaMemsetAsync(dC, 0, (size_t)(Bt * N * L) * 4, st0) != cudaSuccess)
                return cuda_fail();
        }
        return SSM_OK;
    }
    if (!workspace) return SSM_ERR_WORKSPACE;
    if (L > 0 && (!u || !delta_raw || !B || !C || !dy || (!du && !conv) || !ddelta_raw || !dB || !dC))
        return SSM_ERR_NULL;
    const void* ptrs[] = {u, delta_raw, A, B, C, D, z, delta_bias, h0, dy, dhL, du, ddelta_raw,
                          dA, dB, dC, dD, dz, ddelta_bias, dh0, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int sms = device_sm_count();
    const BwdPlan pl = plan_bwd(s, sms, conv == nullptr);
    if (!pl.ok) return SSM_ERR_SHAPE;   // no channel tile fits the shared memory
    // conv prologue: built for 9..16 states and 16-byte token rows; the
    // sweeps' du goes to the workspace, after the plan's buffers
    if (conv && L > 0 && (pl.NP != 16 || !pl.tma_raw)) return SSM_ERR_UNSUPPORTED;
    if (conv && ws_bytes < conv_bwd_bytes(s, sms)) return SSM_ERR_WORKSPACE;
    if (conv) du = static_cast<uint8_t*>(workspace) + conv_bwd_du_offset(pl);
    // packed sequences: built for 9..16 states and 16-byte token rows
    if (varlen && L > 0 && (pl.NP != 16 || !pl.tma_raw)) return SSM_ERR_UNSUPPORTED;
    if (ws_bytes < pl.bytes) return SSM_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws);
    const int64_t per_seq = Bt * Dm * N;   // floats of one sequence's state (packed dhL, dh0)

    // outputs summed with atomics start at zero
    if (cudaMemsetAsync(dA, 0, (size_t)(Dm * N) * 4, st) != cudaSuccess) return cuda_fail();
    if (dD && cudaMemsetAsync(dD, 0, (size_t)Dm * 4, st) != cudaSuccess) return cuda_fail();
    if (ddelta_bias && cudaMemsetAsync(ddelta_bias, 0, (size_t)Dm * 4, st) != cudaSuccess)
        return cuda_fail();
    if (L == 0 && varlen) {
        // every packed sequence is empty: dh0[s] = dhL[s]
        if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return cuda_fail();
        if (launch_varlen_prep(cu_seqlens, nseq, 0, per_seq, dhL, dh0, status, st) != cudaSuccess)
            return cuda_fail();
        return SSM_OK;
    }
    if (L == 0) {
        // an empty sequence passes dhL straight through to dh0
        if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return cuda_fail();
        if (dh0) {
            const size_t bytes = (size_t)(Bt * Dm * N) * 4;
            cudaError_t e = dhL ? cudaMemcpyAsync(dh0, dhL, bytes, cudaMemcpyDeviceToDevice, st)
                                : cudaMemsetAsync(dh0, 0, bytes, st);
            if (e != cudaSuccess) return cuda_fail();
        }
        return SSM_OK;
    }
    if (cudaMemsetAsync(dB, 0, (size_t)(Bt * N * L) * 4, st) != cudaSuccess ||
        cudaMemsetAsync(dC, 0, (size_t)(Bt * N * L) * 4, st) != cudaSuccess)
        return cuda_fail();

    float* bc = reinterpret_cast<float*>(ws + pl.off_bc);
    if (launch_prep_bc(s.in_dtype, Bt, (int)N, pl.NP, L, B, C, bc, status, st) != cudaSuccess)
        return cuda_fail();
    // packed: check the starts; empty sequences pass dhL[s] to dh0[s]
    if (varlen && launch_varlen_prep(cu_seqlens, nseq, L, per_seq, dhL, dh0, status, st) != cudaSuccess)
        return cuda_fail();

    const int eb = dtype_bytes(s.in_dtype);
    const CUtensorMapDataType tdt =
        s.in_dtype == SSM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    float* phi = reinterpret_cast<float*>(ws + pl.off_phi);
    BwdMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!make_map(&maps.bc, bc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2 * pl.NP, Bt * L, 2 * pl.NP, kT,
                  false))
        return cuda_fail();
    if (pl.tma_raw) {
        const uint32_t box_t = 128 / eb;
        if (!make_map(&maps.u, u, tdt, eb, L, Bt * Dm, box_t, pl.CH, true) ||
            !make_map(&maps.dr, delta_raw, tdt, eb, L, Bt * Dm, box_t, pl.CH, true) ||
            (z && !make_map(&maps.z, z, tdt, eb, L, Bt * Dm, box_t, pl.CH, true)) ||
            !make_map(&maps.dy, dy, tdt, eb, L, Bt * Dm, box_t, pl.CH, true) ||
            !make_map(&maps.phi, phi, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, L, Bt * Dm, 32, pl.CH,
                      true))
            return cuda_fail();
    }

    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.Bt = Bt; p.D = Dm; p.L = L; p.N = (int)N;
    p.u = u; p.dr = delta_raw; p.z = z; p.dy = dy; p.A = A; p.Dv = D; p.bias = delta_bias;
    p.h0 = h0; p.dhL = dhL; p.bc = bc; p.phi = phi;
    p.hfin = reinterpret_cast<float*>(ws + pl.off_hfin);
    p.hck = reinterpret_cast<float*>(ws + pl.off_hck);
    p.hprev = s.in_dtype == SSM_F32 ? reinterpret_cast<float*>(ws + pl.off_hprev) : nullptr;
    p.du = du; p.ddr = ddelta_raw; p.dz = dz;
    p.dA = dA; p.dB = dB; p.dC = dC; p.dD = dD; p.dbias = ddelta_bias; p.dh0 = dh0;
    p.cu_seqlens = cu_seqlens; p.nseq = varlen ? nseq : 0;
    p.status = status;
    p.timeout_ns = kDefaultTimeoutNs;
    if (conv) {
        p.conv_w = conv->w;
        p.conv_b = conv->b;
        p.conv_k = conv->k;
    }
    const unsigned gx = (unsigned)((Dm + pl.CH - 1) / pl.CH);
    if (varlen && pl.nseg == 1) {
        BwdLaunch lc;
        lc.grid = dim3(gx, (unsigned)Bt);
        lc.warps = pl.W;
        lc.stages_f = pl.stages_f;
        lc.stages_r = pl.stages_r;
        lc.smem_f = pl.smem_f;
        lc.smem_r = pl.smem_r;
        if (launch_bwd_varlen_np16(pl.NT, s.in_dtype, s.out_dtype, p, maps, lc, st) != cudaSuccess)
            return cuda_fail();
        return SSM_OK;
    }
    if (pl.nseg > 1) {
        // segmented plan: initial states (the forward's tail search, summary
        // pass and carry, on its own tiles), the adjoint entering every
        // segment (adjoint summary, right-to-left carry), the forward sweep,
        // the tangent's dA terms across segments, the reverse sweep
        FwdPlan fp = plan_fwd(s, sms, true);
        fp.nseg = pl.nseg;
        fp.seg_chunks = pl.seg_chunks;
        FwdMaps fm;
        std::memset(&fm, 0, sizeof(fm));
        fm.bc = maps.bc;
        const uint32_t box_t = 128 / eb;
        if (!make_map(&fm.u, u, tdt, eb, L, Bt * Dm, box_t, fp.CH, true) ||
            !make_map(&fm.dr, delta_raw, tdt, eb, L, Bt * Dm, box_t, fp.CH, true) ||
            (z && !make_map(&fm.z, z, tdt, eb, L, Bt * Dm, box_t, fp.CH, true)))
            return cuda_fail();
        FwdParams pf;
        std::memset(&pf, 0, sizeof(pf));
        pf.Bt = Bt; pf.D = Dm; pf.L = L; pf.N = (int)N;
        pf.u = u; pf.dr = delta_raw; pf.z = z; pf.A = A; pf.Dv = D; pf.bias = delta_bias;
        pf.h0 = h0; pf.bc = bc;
        pf.cu_seqlens = cu_seqlens;
        pf.nseq = varlen ? nseq : 0;
        pf.seg_chunks = pl.seg_chunks;
        pf.nseg = pl.nseg;
        pf.stages = fp.stages;
        pf.status = status;
        pf.timeout_ns = kDefaultTimeoutNs;
        pf.hin = reinterpret_cast<float*>(ws + pl.off_hin);
        pf.hloc = reinterpret_cast<float*>(ws + pl.off_hloc);
        pf.sumd = reinterpret_cast<float*>(ws + pl.off_sumd);
        int* tstart = reinterpret_cast<int*>(ws + pl.off_tstart);
        const unsigned gxf = (unsigned)pl.fwd_tiles;
        FwdParams pf1 = pf;
        pf1.hin = nullptr;
        pf1.tstart = tstart;
        if (launch_tail(s.in_dtype, pf, fp.CH, gxf, tstart, pf.sumd, st) != cudaSuccess ||
            launch_fwd(fp, s.in_dtype, s.out_dtype, true, false, varlen, pf1, fm,
                       dim3(gxf, (unsigned)Bt, (unsigned)(pl.nseg - 1)), st) != cudaSuccess ||
            launch_carry(Bt, Dm, (int)N, pl.NP, pl.nseg, A, h0, pf.hloc, pf.sumd, pf.hin, st) !=
                cudaSuccess)
            return cuda_fail();

        p.seg_chunks = pl.seg_chunks;
        p.nseg = pl.nseg;
        p.hin = pf.hin;
        p.lam_loc = reinterpret_cast<float*>(ws + pl.off_lamloc);
        float* lam_in = reinterpret_cast<float*>(ws + pl.off_lamin);
        p.lam_in = lam_in;
        p.sumd = reinterpret_cast<float*>(ws + pl.off_sumdr);
        p.gp = reinterpret_cast<float*>(ws + pl.off_gp);
        p.mend = reinterpret_cast<float*>(ws + pl.off_mend);
        BwdLaunch lc;
        lc.grid = dim3(gx, (unsigned)Bt, (unsigned)pl.nseg);
        lc.warps = pl.W;
        lc.stages_f = pl.stages_f;
        lc.stages_r = pl.stages_r;
        lc.stages_l = pl.stages_l;
        lc.smem_f = pl.smem_f;
        lc.smem_r = pl.smem_r;
        lc.smem_l = pl.smem_l;
        int* kstop = reinterpret_cast<int*>(ws + pl.off_kstop);
        if (launch_head(s.in_dtype, p, pl.CH, gx, kstop, p.sumd, st) != cudaSuccess)
            return cuda_fail();
        p.kstop = kstop;
        // (the last segment's adjoint summary starts from the final-state
        // gradient itself, so the carry starts from zero)
        auto seg_part = [&](int part) {
            return varlen ? launch_bwd_seg_varlen_np16(pl.NT, s.in_dtype, s.out_dtype, part, p, maps, lc, st)
                          : launch_bwd_seg_np16(pl.NT, s.in_dtype, s.out_dtype, part, p, maps, lc, st);
        };
        if (seg_part(0) != cudaSuccess ||
            launch_carry(Bt, Dm, (int)N, pl.NP, pl.nseg, A, nullptr, p.lam_loc, p.sumd, lam_in, st,
                         true) != cudaSuccess ||
            seg_part(1) != cudaSuccess ||
            launch_tangent_carry(Bt, Dm, (int)N, pl.NP, pl.nseg, A, pf.sumd, p.mend, p.gp, dA, st) !=
                cudaSuccess ||
            seg_part(2) != cudaSuccess)
            return cuda_fail();
        return SSM_OK;
    }
    if (conv) {
        // the sweeps with u formed from x, then the prologue's reverse mode
        BwdLaunch lc;
        lc.grid = dim3(gx, (unsigned)Bt);
        lc.warps = pl.W;
        lc.stages_f = pl.stages_f;
        lc.stages_r = pl.stages_r;
        lc.smem_f = pl.smem_f;
        lc.smem_r = pl.smem_r;
        if (launch_bwd_conv_np16(pl.NT, s.in_dtype, s.out_dtype, p, maps, lc, st) != cudaSuccess ||
            launch_conv_bwd(s.in_dtype, s.out_dtype, Bt, Dm, L, conv->k, u, conv->w, conv->b,
                            static_cast<const float*>(du), conv->dx, conv->dw, conv->db, st) !=
                cudaSuccess)
            return cuda_fail();
        return SSM_OK;
    }
    if (launch_bwd(pl, s.in_dtype, s.out_dtype, p, maps, dim3(gx, (unsigned)Bt), st) != cudaSuccess)
        return cuda_fail();
    return SSM_OK;
}

int ssm_scan_bwd(const ssm_shape* shape, const void* u, const void* delta_raw, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* delta_bias, const float* h0, const void* dy, const float* dhL,
                 void* du, void* ddelta_raw, float* dA, float* dB, float* dC, float* dD,
                 void* dz, float* ddelta_bias, float* dh0, void* workspace, size_t ws_bytes,
                 ssm_stream_t stream) {
    return scan_bwd_impl(shape, u, nullptr, 0, delta_raw, A, B, C, D, z, delta_bias, h0, dy, dhL,
                         du, ddelta_raw, dA, dB, dC, dD, dz, ddelta_bias, dh0, workspace,
                         ws_bytes, stream);
}

int ssm_scan_bwd_conv(const ssm_shape* shape, const void* x, const float* conv_w,
                      const float* conv_b, int conv_k, const void* delta_raw, const float* A,
                      const void* B, const void* C, const float* D, const void* z,
                      const float* delta_bias, const float* h0, const void* dy, const float* dhL,
                      void* dx, void* ddelta_raw, float* dA, float* dB, float* dC, float* dD,
                      void* dz, float* ddelta_bias, float* dh0, float* dconv_w, float* dconv_b,
                      void* workspace, size_t ws_bytes, ssm_stream_t stream) {
    const ConvBwd cv{conv_w, conv_b, conv_k, dx, dconv_w, dconv_b};
    return scan_bwd_impl(shape, x, nullptr, 0, delta_raw, A, B, C, D, z, delta_bias, h0, dy, dhL,
                         nullptr, ddelta_raw, dA, dB, dC, dD, dz, ddelta_bias, dh0, workspace,
                         ws_bytes, stream, &cv);
}

int ssm_scan_bwd_varlen(const ssm_shape* shape, const void* u, const int32_t* cu_seqlens,
                        int nseq, const void* delta_raw, const float* A, const void* B,
                        const void* C, const float* D, const void* z, const float* delta_bias,
                        const float* h0, const void* dy, const float* dhL, void* du,
                        void* ddelta_raw, float* dA, float* dB, float* dC, float* dD, void* dz,
                        float* ddelta_bias, float* dh0, void* workspace, size_t ws_bytes,
                        ssm_stream_t stream) {
    if (!cu_seqlens) return SSM_ERR_NULL;
    return scan_bwd_impl(shape, u, cu_seqlens, nseq, delta_raw, A, B, C, D, z, delta_bias, h0,
                         dy, dhL, du, ddelta_raw, dA, dB, dC, dD, dz, ddelta_bias, dh0, workspace,
                         ws_bytes, stream);
}

int ssm_scan_bwd_bidir(const ssm_shape* shape, const void* u, const void* z,
                       const void* delta_raw, const float* A, const void* B, const void* C,
                       const float* D, const float* delta_bias, const float* h0,
                       const void* delta_raw_r, const float* A_r, const void* B_r, const void* C_r,
                       const float* D_r, const float* delta_bias_r, const float* h0_r,
                       const void* dy, const float* dhL, const float* dhL_r, void* du, void* dz,
                       void* ddelta_raw, float* dA, float* dB, float* dC, float* dD,
                       float* ddelta_bias, float* dh0, void* ddelta_raw_r, float* dA_r,
                       float* dB_r, float* dC_r, float* dD_r, float* ddelta_bias_r, float* dh0_r,
                       void* workspace, size_t ws_bytes, ssm_stream_t stream) {
    const int sc = shape_check(shape);
    if (sc != SSM_OK) return sc;
    const ssm_shape s = *shape;
    const int64_t Bt = s.batch, Dm = s.dim, N = s.dstate, L = s.seqlen;
    if (Dm > 0 && (!A || !A_r || !dA || !dA_r)) return SSM_ERR_NULL;
    if (Bt == 0 || Dm == 0) {
        // nothing flows: each direction's per-channel gradients are zero
        int rc = ssm_scan_bwd(shape, u, delta_raw, A, B, C, D, z, delta_bias, h0, dy, dhL, du,
                              ddelta_raw, dA, dB, dC, dD, dz, ddelta_bias, dh0, nullptr, 0, stream);
        if (rc != SSM_OK) return rc;
        return ssm_scan_bwd(shape, u, delta_raw_r, A_r, B_r, C_r, D_r, z, delta_bias_r, h0_r, dy,
                            dhL_r, du, ddelta_raw_r, dA_r, dB_r, dC_r, dD_r, dz, ddelta_bias_r,
                            dh0_r, nullptr, 0, stream);
    }
    if (!workspace) return SSM_ERR_WORKSPACE;
    if (L > 0 && (!u || !dy || !du || !delta_raw || !B || !C || !ddelta_raw || !dB || !dC ||
                  !delta_raw_r || !B_r || !C_r || !ddelta_raw_r || !dB_r || !dC_r))
        return SSM_ERR_NULL;
    const void* ptrs[] = {u, z, delta_raw, A, B, C, D, delta_bias, h0, delta_raw_r, A_r, B_r, C_r,
                          D_r, delta_bias_r, h0_r, dy, dhL, dhL_r, du, dz, ddelta_raw, dA, dB, dC,
                          dD, ddelta_bias, dh0, ddelta_raw_r, dA_r, dB_r, dC_r, dD_r,
                          ddelta_bias_r, dh0_r, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SSM_ERR_ALIGN;
    const BidirBwdLayout w = bidir_bwd_layout(s, device_sm_count());
    if (ws_bytes < w.bytes) return SSM_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* status = reinterpret_cast<int*>(ws);
    void* inner = ws + w.off_inner;
    const int* inner_status = reinterpret_cast<const int*>(inner);
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return cuda_fail();

    // both directions' per-token gradients in fp32 first, combined at the end
    ssm_shape s32 = s;
    s32.out_dtype = SSM_F32;
    const size_t tokb = align256((size_t)(Bt * Dm * L) * 4);
    float* g = reinterpret_cast<float*>(ws + w.off_g);
    float* du1 = g;
    float* ddr1 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(g) + tokb);
    float* dz1 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(g) + 2 * tokb);
    float* du2 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(g) + 3 * tokb);
    float* ddr2 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(g) + 4 * tokb);
    float* dz2 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(g) + 5 * tokb);
    const bool gate = z != nullptr;
    const bool want_dz = dz != nullptr;   // (zeros without a gate, as in ssm_scan_bwd)

    // left to right: the ordinary backward
    int rc = ssm_scan_bwd(&s32, u, delta_raw, A, B, C, D, z, delta_bias, h0, dy, dhL, du1, ddr1,
                          dA, dB, dC, dD, want_dz ? dz1 : nullptr, ddelta_bias, dh0, inner, w.inner,
                          stream);
    if (rc != SSM_OK) return rc;
    if (launch_fold_status(status, inner_status, st) != cudaSuccess) return cuda_fail();

    // right to left: the backward of the token-reversed sequence
    void* u_f = ws + w.off_u;
    void* dr_f = ws + w.off_dr;
    void* z_f = gate ? ws + w.off_z : nullptr;
    void* dy_f = ws + w.off_dy;
    void* B_f = ws + w.off_B;
    void* C_f = ws + w.off_C;
    const int64_t rows = Bt * Dm, brows = Bt * N;
    if (launch_flip_rows(s.in_dtype, u, u_f, rows, L, st) != cudaSuccess ||
        launch_flip_rows(s.in_dtype, delta_raw_r, dr_f, rows, L, st) != cudaSuccess ||
        (gate && launch_flip_rows(s.in_dtype, z, z_f, rows, L, st) != cudaSuccess) ||
        launch_flip_rows(s.in_dtype, dy, dy_f, rows, L, st) != cudaSuccess ||
        launch_flip_rows(s.in_dtype, B_r, B_f, brows, L, st) != cudaSuccess ||
        launch_flip_rows(s.in_dtype, C_r, C_f, brows, L, st) != cudaSuccess)
        return cuda_fail();
    float* dB_f = reinterpret_cast<float*>(ws + w.off_dB);
    float* dC_f = reinterpret_cast<float*>(ws + w.off_dC);
    rc = ssm_scan_bwd(&s32, u_f, dr_f, A_r, B_f, C_f, D_r, z_f, delta_bias_r, h0_r, dy_f, dhL_r,
                      du2, ddr2, dA_r, dB_f, dC_f, dD_r, want_dz ? dz2 : nullptr, ddelta_bias_r,
                      dh0_r, inner, w.inner, stream);
    if (rc != SSM_OK) return rc;
    if (launch_fold_status(status, inner_status, st) != cudaSuccess) return cuda_fail();

    // du, dz summed; each direction's ddelta_raw, dB, dC in token order
    if (launch_bidir_combine(s.out_dtype, rows, L, du1, du2, dz1, dz2, ddr1, ddr2, du,
                             want_dz ? dz : nullptr, ddelta_raw, ddelta_raw_r, st) != cudaSuccess ||
        launch_flip_rows(SSM_F32, dB_f, dB_r, brows, L, st) != cudaSuccess ||
        launch_flip_rows(SSM_F32, dC_f, dC_r, brows, L, st) != cudaSuccess)
        return cuda_fail();
    return SSM_OK;
}

int ssm_scan_step(int64_t batch, int64_t dim, int64_t dstate, int32_t in_dtype, int32_t out_dtype,
                  const void* u, const void* delta_raw, const float* A, const void* B,
                  const void* C, const float* D, const void* z, const float* delta_bias,
                  float* state, void* y, int* status, ssm_stream_t stream) {
    if (batch < 0 || dim < 0 || dstate < 1 || dstate > 64) return SSM_ERR_SHAPE;
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return SSM_ERR_DTYPE;
    int64_t bd, tmp;
    if (!mul_ok(batch, dim, &bd) || !mul_ok(bd, dstate * 16, &tmp)) return SSM_ERR_SHAPE;
    if (bd == 0) return SSM_OK;
    if (!u || !delta_raw || !A || !B || !C || !state || !y) return SSM_ERR_NULL;
    const void* ptrs[] = {u, delta_raw, A, B, C, D, z, delta_bias, state, y};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_ALIGN;
    if (((uintptr_t)status % 4) != 0) return SSM_ERR_ALIGN;
    StepParams p;
    p.Bt = batch; p.D = dim; p.N = (int)dstate;
    p.u = u; p.dr = delta_raw; p.z = z; p.A = A; p.Dv = D; p.bias = delta_bias;
    p.B = B; p.C = C; p.state = state; p.y = y; p.status = status;
    if (dstate == 16 && dim % 128 == 0 && bd < (int64_t(1) << 31)) {
        // whole 128-channel tiles: the state and A stream through 2-D TMA tiles
        CUtensorMap tm_st, tm_a;
        if (!make_map_swz64(&tm_st, state, (uint64_t)bd) || !make_map_swz64(&tm_a, A, (uint64_t)dim))
            return cuda_fail();
        if (launch_step_dec16_any(in_dtype, out_dtype, p, tm_st, tm_a, static_cast<cudaStream_t>(stream)) !=
            cudaSuccess)
            return cuda_fail();
        return SSM_OK;
    }
    if (launch_step(in_dtype, out_dtype, p, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return cuda_fail();
    return SSM_OK;
}

int ssm_get_status(void* workspace, ssm_stream_t stream) {
    if (!workspace) return SSM_ERR_NULL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return cuda_fail();
    if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_fail();
    if (v != SSM_OK) {
        if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return cuda_fail();
        if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_fail();
    }
    return v;
}

int ssm_debug_expired_wait(void* workspace, size_t ws_bytes, int64_t spin_limit,
                           ssm_stream_t stream) {
    if (!workspace) return SSM_ERR_NULL;
    if (ws_bytes < kHeaderBytes) return SSM_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SSM_ERR_ALIGN;
    if (spin_limit < 1) return SSM_ERR_SHAPE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* status = static_cast<int*>(workspace);
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return cuda_fail();
    if (launch_expired_wait(status, spin_limit, st) != cudaSuccess) return cuda_fail();
    return SSM_OK;
}

}  // extern "C"
