// lf_gemm_common.cuh -- device code shared by the NT GEMM kernels (single-CTA
// and CTA-pair): bounded mbarrier waits with CTA-wide abort, and the three
// epilogues that read a finished accumulator out of TMEM.
//
// Epilogue sources: "Strength reduction: fold transpose into a subsequent GEMM
// call" (the bf16 output of the traced matmul) and "Allow reductions in matmul
// epilogues" (NVIDIA/Fuser issue 2213), the fusion example: row max, exp and
// its sum, the label logit picked by comparing the column index with the
// label, and the softmax-minus-onehot output.
#pragma once
#include <cuda_bf16.h>
#include <math_constants.h>

#include "lf_internal.h"
#include "lf_ptx.cuh"

namespace lf {
namespace {

constexpr float LOG2E = 1.4426950408889634f;

// Error codes written to the device error word (first writer wins).
constexpr int ERR_PRODUCER = 0x101;   // ring slot never freed
constexpr int ERR_MMA_FULL = 0x102;   // stage never landed
constexpr int ERR_MMA_ACC = 0x103;    // accumulator never released by the epilogue
constexpr int ERR_EPI = 0x104;        // accumulator never completed
constexpr int ERR_DRAIN = 0x105;      // copies / MMAs did not finish while unwinding
constexpr int ERR_SK_FLAG = 0x106;    // a stream-K partial never arrived
constexpr int ERR_SK_SLOT = 0x107;    // a CTA's own partial write did not complete
constexpr int ERR_SK_COPY = 0x109;    // the copy of a partial into shared memory did not land
constexpr int ERR_TILE_QUEUE = 0x10A; // a claimed tile index never reached this role

// Record `code` (first writer wins), raise this CTA's abort flag and, in a
// CTA pair, the peer's (peer_abort: its shared::cluster address, 0 if none).
__device__ __forceinline__ void raise_error(const GemmParams &p, volatile int *abort_flag, int code,
                                            uint32_t peer_abort)
{
    *abort_flag = 1;
    if (peer_abort)
        st_cluster_u32(peer_abort, 1u);
    atomicCAS(p.err, 0, code);
}

// Slow path of wait_bar, out of line: poll until the phase completes, the CTA
// aborts or the time limit passes (then the error is recorded and the abort
// flag raised).
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           const GemmParams &p, int code, uint32_t peer_abort)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 15u) == 0) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                raise_error(p, abort_flag, code, peer_abort);
                return false;
            }
        }
    }
}

// Wait for phase `parity` of `bar`; false if the CTA is aborting or the time
// limit passed.  The ready case stays inline: an out-of-line call on the
// MMA-issuing thread, made every K block, measurably starves the tensor pipe.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         const GemmParams &p, int code, uint32_t peer_abort = 0)
{
    if (mbar_try_wait(bar, parity))
        return true;
    return wait_bar_slow(bar, parity, abort_flag, p, code, peer_abort);
}

// Same, used while unwinding: ignores the abort flag, keeps the time limit.
__device__ __noinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                            const GemmParams &p, uint32_t peer_abort = 0)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > p.timeout_ns) {
            raise_error(p, abort_flag, ERR_DRAIN, peer_abort);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (lower address) = lo
    return *reinterpret_cast<uint32_t *>(&h);
}

// Store 32 consecutive fp32 values as bf16 to dst[0..32), 8 at a time, keeping
// only the 8-column groups that start below `limit` columns.
__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16 *dst, const float (&f)[32], int limit)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (j * 8 < limit) {
            uint4 v;
            v.x = pack_bf16(f[8 * j + 0], f[8 * j + 1]);
            v.y = pack_bf16(f[8 * j + 2], f[8 * j + 3]);
            v.z = pack_bf16(f[8 * j + 4], f[8 * j + 5]);
            v.w = pack_bf16(f[8 * j + 6], f[8 * j + 7]);
            reinterpret_cast<uint4 *>(dst)[j] = v;
        }
    }
}

// Partial accumulators of other CTA pairs to add to this tile (stream-K
// fix-up): `count` slots starting at `slot`, `stride` floats apart.
struct PartialAdd {
    const float *slot;
    size_t stride;
    int count;
    int row;                // this thread's row within its CTA's 128 rows
    const float4 *smem0;    // if set: contributor 0's slot, already copied to shared memory
    int in_tmem;            // if set: the partials' sum is in TMEM at `tpart` (this thread's lane)
    uint32_t tpart;
};

// Read 32 accumulator columns [c, c+32) of this thread's row from TMEM and
// add the partials, in pair order.
__device__ __forceinline__ void load_chunk(uint32_t taddr, int c, const PartialAdd &pa, uint32_t (&v)[32])
{
    if (pa.in_tmem) {
        uint32_t w[32];
        tmem_ld_32x32b_x32(taddr + c, v);
        tmem_ld_32x32b_x32(pa.tpart + c, w);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(w[i]));
        return;
    }
    tmem_ld_32x32b_x32(taddr + c, v);
    tmem_wait_ld();
    for (int e = 0; e < pa.count; ++e) {
        if (e == 0 && pa.smem0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 f = pa.smem0[(c / 4 + i) * BM + pa.row];
                v[4 * i + 0] = __float_as_uint(__uint_as_float(v[4 * i + 0]) + f.x);
                v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + f.y);
                v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + f.z);
                v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + f.w);
            }
            continue;
        }
        const float4 *s4 = reinterpret_cast<const float4 *>(pa.slot + static_cast<size_t>(e) * pa.stride);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 f = __ldcg(s4 + (c / 4 + i) * BM + pa.row);
            v[4 * i + 0] = __float_as_uint(__uint_as_float(v[4 * i + 0]) + f.x);
            v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + f.y);
            v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + f.z);
            v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + f.w);
        }
    }
}

// Store columns [c0, c1) of this thread's accumulator row (fp32) into a
// stream-K slot.
__device__ __forceinline__ void epi_write_partial(uint32_t taddr, float *slot, int row, int c0 = 0, int c1 = BN)
{
    float4 *s4 = reinterpret_cast<float4 *>(slot);
#pragma unroll 1
    for (int c = c0; c < c1; c += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i)
            __stcg(s4 + (c / 4 + i) * BM + row,
                   make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                               __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
    }
}

// Claimed whole tiles (GemmParams::tile_ctl): called once per pair, by the
// pair's claiming thread, when its claiming is over (its last claim went past
// the last tile, or it is aborting).  The count is a release: the pair's
// claims precede it; the pair that completes it (an acquire) has seen every
// claim and zeroes the counter and the count for the next launch.  This runs
// while the pairs still compute their last tiles, off the launch's tail.
__device__ __forceinline__ void claims_done(unsigned *ctl, unsigned pairs)
{
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(ctl + 1) : "memory");
    if (old == pairs - 1u) {
        asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(ctl) : "memory");
        asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(ctl + 1) : "memory");
    }
}

// Bounded wait until *flag == epoch (acquire); false on abort or time-out.
__device__ __noinline__ bool wait_flag(const unsigned *flag, unsigned epoch, volatile int *abort_flag,
                                       const GemmParams &p, uint32_t peer_abort)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (ld_acquire_gpu(flag) == epoch)
            return true;
        if ((it & 15u) == 15u) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                raise_error(p, abort_flag, ERR_SK_FLAG, peer_abort);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- epilogues
// Each runs on one epilogue warp: thread `lane` owns output row `row` of the
// tile, whose accumulator row starts at TMEM address `taddr`.

// out = bf16_rn(acc)
__device__ __forceinline__ void epi_store(const GemmParams &p, uint32_t taddr, int row, int nb,
                                          const PartialAdd &pa)
{
    const bool row_ok = row < p.M;
    __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.out) + static_cast<size_t>(row) * p.N;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        if (row_ok) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                f[i] = __uint_as_float(v[i]);
            store_row32_bf16(orow + col, f, p.N - col);
        }
    }
}

// Cross-entropy statistics of one 256-column tile of row `row` ("Allow
// reductions in matmul epilogues", fusion example: the row max, exp(z - max)
// and its sum, and the label logit selected by comparing the column index
// with the label), over the tile's columns n < N:
//   mx = max_n z,  se = sum_n exp(z - mx),  zl = z[label] if the label is here.
// The running (max, sum) is rescaled chunk by chunk (32 columns at a time).
__device__ __forceinline__ void xent_tile_stats(const GemmParams &p, uint32_t taddr, int lab, int nb,
                                                const PartialAdd &pa, float &mx_out, float &se_out, float &zl,
                                                bool &have_label)
{
    const int lab_local = lab - nb * BN;
    float mx = -CUDART_INF_F, s = 0.f;
    have_label = false;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        const int nvalid = p.N - col;  // >= 8 here; only the last tile is ragged
        float cm = -CUDART_INF_F;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nvalid)
                cm = fmaxf(cm, __uint_as_float(v[i]));
        const int li = lab_local - c;
        if (static_cast<unsigned>(li) < 32u) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i == li)
                    zl = __uint_as_float(v[i]);
            have_label = true;
        }
        const float nm = fmaxf(mx, cm);
        s *= exp2f((mx - nm) * LOG2E);  // mx = -inf on the first chunk: factor 0, s is 0
        float cs = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nvalid)
                cs += exp2f((__uint_as_float(v[i]) - nm) * LOG2E);
        s += cs;
        mx = nm;
    }
    mx_out = mx;
    se_out = s;
}

// Two-pass form for the one-pass gradient kernel, which keeps the tile in
// TMEM until the row's log-sum-exp is known: pass 1 finds the tile max (and
// the label logit), pass 2 replaces each accumulator value by
// e = exp(z - tile_max) (0 past column N) and returns sum e, so the gradient
// pass needs no second exponential: grad = e * exp(tile_max - lse) - onehot.
__device__ __forceinline__ float xent_tile_max(const GemmParams &p, uint32_t taddr, int lab, int nb, float &zl,
                                               bool &have_label)
{
    const int lab_local = lab - nb * BN;
    float mx = -CUDART_INF_F;
    have_label = false;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c, v);
        tmem_wait_ld();
        const int nvalid = p.N - col;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nvalid)
                mx = fmaxf(mx, __uint_as_float(v[i]));
        const int li = lab_local - c;
        if (static_cast<unsigned>(li) < 32u) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i == li)
                    zl = __uint_as_float(v[i]);
            have_label = true;
        }
    }
    return mx;
}

__device__ __forceinline__ float xent_tile_exp_store(const GemmParams &p, uint32_t taddr, int nb, float tmax)
{
    float s = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c, v);
        tmem_wait_ld();
        const int nvalid = p.N - col;
        float cs = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float e = i < nvalid ? exp2f((__uint_as_float(v[i]) - tmax) * LOG2E) : 0.f;
            cs += e;
            v[i] = __float_as_uint(e);
        }
        s += cs;
        tmem_st_32x32b_x32(taddr + c, v);
    }
    tmem_wait_st();
    return s;
}

// grad = bf16_rn(e * scale - [n == label]) with e = exp(z - tile_max) from
// TMEM and scale = exp(tile_max - lse).
__device__ __forceinline__ void xent_grad_from_exp(const GemmParams &p, uint32_t taddr, int row, int nb, int lab,
                                                   float scale)
{
    const bool row_ok = row < p.M;
    const int lab_local = lab - nb * BN;
    __nv_bfloat16 *grow = static_cast<__nv_bfloat16 *>(p.out) + static_cast<size_t>(row) * p.N;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c, v);
        tmem_wait_ld();
        if (row_ok) {
            const int li = lab_local - c;
            float g[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                g[i] = __uint_as_float(v[i]) * scale;
                if (i == li)
                    g[i] -= 1.f;
            }
            store_row32_bf16(grow + col, g, p.N - col);
        }
    }
}

// Partials of one tile to the workspace: part_max/part_sum[row, nb] and, if
// the label falls in this tile, label_logit[row].
__device__ __forceinline__ void epi_xent_partial(const GemmParams &p, uint32_t taddr, int row, int nb,
                                                 const PartialAdd &pa)
{
    const bool row_ok = row < p.M;
    const int lab = row_ok ? p.labels[row] : -1;
    float mx, se, zl = 0.f;
    bool have_label;
    xent_tile_stats(p, taddr, lab, nb, pa, mx, se, zl, have_label);
    if (row_ok) {
        const size_t o = static_cast<size_t>(row) * p.num_n_blocks + nb;
        p.part_max[o] = mx;
        p.part_sum[o] = se;
        if (have_label && lab < p.N)
            p.label_logit[row] = zl;
    }
}

// Gradient of one tile from the accumulator ("Allow reductions in matmul
// epilogues", the yhatminusy output), given the row's max and log-sum:
//   grad = bf16_rn(exp((z - row_max) - row_logsum) - [n == label])
__device__ __forceinline__ void epi_xent_grad_rows(const GemmParams &p, uint32_t taddr, int row, int nb,
                                                   const PartialAdd &pa, float rmax, float rls)
{
    const bool row_ok = row < p.M;
    const int lab = row_ok ? p.labels[row] : -1;
    const int lab_local = lab - nb * BN;
    __nv_bfloat16 *grow = static_cast<__nv_bfloat16 *>(p.out) + static_cast<size_t>(row) * p.N;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        if (row_ok) {
            const int li = lab_local - c;
            float g[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                g[i] = exp2f(((__uint_as_float(v[i]) - rmax) - rls) * LOG2E);
                if (i == li)
                    g[i] -= 1.f;
            }
            store_row32_bf16(grow + col, g, p.N - col);
        }
    }
}

// The whole row in one tile (N <= 256): with a single N tile the row's
// reduction ("Allow reductions in matmul epilogues", fusion example: max,
// exp, sum, log-sum-exp, the label logit, softmax minus one-hot) needs no
// merge across tiles, so this epilogue writes loss[row] and, when p.out is
// set, the gradient row, with no second kernel.  Three passes over TMEM (max
// and label logit; sum of exp(z - max); gradient), partials of other CTA pairs
// (stream-K) added identically in each.
__device__ __forceinline__ void epi_xent_row(const GemmParams &p, uint32_t taddr, int row, const PartialAdd &pa)
{
    const bool row_ok = row < p.M;
    const int lab = row_ok ? p.labels[row] : -1;
    float mx = -CUDART_INF_F, zl = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN && c < p.N; c += 32) {
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        const int nvalid = p.N - c;
        const int li = lab - c;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (i < nvalid)
                mx = fmaxf(mx, __uint_as_float(v[i]));
            if (i == li)
                zl = __uint_as_float(v[i]);
        }
    }
    const float mxl = mx * LOG2E;
    float s = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN && c < p.N; c += 32) {
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        const int nvalid = p.N - c;
        float cs = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            cs += i < nvalid ? ex2_approx(fmaf(__uint_as_float(v[i]), LOG2E, -mxl)) : 0.f;
        s += cs;
    }
    const float ls = logf(s);
    const bool lab_ok = lab >= 0 && lab < p.N;
    if (row_ok)
        p.loss[row] = lab_ok ? (mx - zl) + ls : CUDART_NAN_F;
    if (!p.out)
        return;
    const float off = (mx + ls) * LOG2E;
    __nv_bfloat16 *grow = static_cast<__nv_bfloat16 *>(p.out) + static_cast<size_t>(row) * p.N;
#pragma unroll 1
    for (int c = 0; c < BN && c < p.N; c += 32) {
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        if (row_ok) {
            const int li = lab - c;
            float g[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                g[i] = ex2_approx(fmaf(__uint_as_float(v[i]), LOG2E, -off));
                if (i == li)
                    g[i] -= 1.f;
            }
            store_row32_bf16(grow + c, g, p.N - c);
        }
    }
}

// Gradient pass of the two-pass form: the row statistics come from the combine kernel.
__device__ __forceinline__ void epi_xent_grad(const GemmParams &p, uint32_t taddr, int row, int nb,
                                              const PartialAdd &pa)
{
    const bool row_ok = row < p.M;
    epi_xent_grad_rows(p, taddr, row, nb, pa, row_ok ? p.row_max[row] : 0.f, row_ok ? p.row_logsum[row] : 0.f);
}

}  // namespace
}  // namespace lf
