// lf_xent_rescale.cuh -- the second half of the cross-entropy gradient after
// the GEMM's exp epilogue, one warp per unit of work.  Included by the
// follow-up rescale kernel (pointwise.cu) and by the pair GEMM, whose
// epilogue warps rescale the rows of finished bands while later bands' MMAs
// run; both run this one routine, so a unit's bytes do not depend on which of
// them took it.
//
// Source: "Allow reductions in matmul epilogues" (NVIDIA/Fuser issue 2213),
// the fusion example's softmax-minus-onehot output and the follow-up on
// reducing a row across output tiles: the row's log-sum-exp merges the
// per-tile partials,
//   m = max_j m_j,  s = sum_j s_j exp(m_j - m),  lse = m + log s,
//   loss = lse - z[label]  (NaN for a label outside [0, N)),
// and the gradient reuses it.  The exp epilogue left e = fp16(exp(z - m_j)) in
// the gradient buffer; a unit rewrites its part of the row in place,
//   grad = bf16_rn(e * exp(m_j - lse)),
// except the label column, computed from the fp32 label logit:
//   grad[label] = bf16_rn(exp(z[label] - lse) - 1).
// Error: fp16 keeps e to 2^-11 relative, so a non-label entry p < 1/2 is off by
// at most p 2^-11 (+ 1e-6) before its bf16 rounding (<= 9.8e-4 below 1/2): under
// 1.3e-3 in all; an entry p >= 1/2 is the row's (hence its tile's) maximum,
// where e = 1 exactly, so only its bf16 rounding remains.
//
// A unit is one row and RS_SEG_TILES consecutive 256-column tiles of it (8192
// columns, 16 KiB of fp16 in and of bf16 out); units are numbered row-major,
// u = row * units_per_row + segment.  Every unit merges the row's partials
// itself (in the same order, so all units of a row agree bit for bit) and the
// unit holding tile 0 writes the loss.
#pragma once
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "lf_kernel_params.h"

namespace lf {

// tiles per unit (RS_SEG_TILES, lf_kernel_params.h): lane j holds the scale of the unit's tile j
static_assert(RS_SEG_TILES == 32, "one tile scale per lane");
constexpr int RS_UNROLL = 8;  // 16-byte loads in flight per lane (4 KiB per warp)
constexpr float RS_LOG2E = 1.4426950408889634f;

struct RescaleArgs {
    const float *part_max;     // [M, NB]: tile maxima m_j
    const float *part_sum;     // [M, NB]: sum exp(z - m_j) over the tile
    const float *label_logit;  // [M]: z[label]
    const int32_t *labels;     // [M]
    int M, N, NB;              // N % 8 == 0, NB = ceil(N / 256)
    float *loss;               // [M]
    uint4 *grad;               // [M, N / 8]: fp16 e in, bf16 gradient out
};

__device__ __forceinline__ float rs_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t rs_scale_pair(uint32_t hpair, float scale)
{
    const __half2 h = *reinterpret_cast<const __half2 *>(&hpair);
    const float2 f = __half22float2(h);
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    return *reinterpret_cast<uint32_t *>(&b);
}

// Unit (row, seg); all 32 lanes of the warp call it.  Everything the exp pass
// wrote is read through L2 (.cg), so a unit taken inside the GEMM sees the
// other CTAs' writes once their band's count has been observed.
__device__ __forceinline__ void xent_rescale_unit(const RescaleArgs &a, int row, int seg)
{
    const int lane = threadIdx.x & 31;
    const float *pm = a.part_max + static_cast<size_t>(row) * a.NB;
    const float *ps = a.part_sum + static_cast<size_t>(row) * a.NB;
    // 1. the row's merge (lane-strided, then a butterfly: the same order in
    //    every unit of the row)
    float m = -CUDART_INF_F;
    for (int j = lane; j < a.NB; j += 32)
        m = fmaxf(m, __ldcg(pm + j));
#pragma unroll
    for (int o = 16; o; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
    for (int j = lane; j < a.NB; j += 32)
        s += __ldcg(ps + j) * exp2f((__ldcg(pm + j) - m) * RS_LOG2E);
#pragma unroll
    for (int o = 16; o; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    const float ls = logf(s);
    const float lse = m + ls;
    const int lab = a.labels[row];
    const bool lab_ok = lab >= 0 && lab < a.N;
    const float zl = lab_ok ? __ldcg(a.label_logit + row) : 0.f;
    if (seg == 0 && lane == 0)
        a.loss[row] = lab_ok ? (m - zl) + ls : CUDART_NAN_F;
    // 2. lane j: the scale exp(m_j - lse) of the unit's tile j
    const float lsel = lse * RS_LOG2E;
    const int t0 = seg * RS_SEG_TILES;
    const int nt = min(RS_SEG_TILES, a.NB - t0);
    const float sc_own = lane < nt ? rs_ex2(fmaf(__ldcg(pm + t0 + lane), RS_LOG2E, -lsel)) : 0.f;
    const float g_lab = rs_ex2(fmaf(zl, RS_LOG2E, -lsel)) - 1.f;
    // 3. the unit's columns: step i is tile t0 + i, lane l its 8 columns 8l..8l+7
    uint4 *rowp = a.grad + static_cast<size_t>(row) * (a.N / 8);
    const int nv = a.N / 8;
    const int lab_v = lab_ok ? lab >> 3 : -1;
#pragma unroll 1
    for (int i0 = 0; i0 < nt; i0 += RS_UNROLL) {
        uint4 q[RS_UNROLL];
#pragma unroll
        for (int u = 0; u < RS_UNROLL; ++u) {
            const int v = (t0 + i0 + u) * 32 + lane;
            if (i0 + u < nt && v < nv)
                q[u] = __ldcg(rowp + v);
        }
#pragma unroll
        for (int u = 0; u < RS_UNROLL; ++u) {
            const float sc = __shfl_sync(0xffffffffu, sc_own, (i0 + u) & 31);
            const int v = (t0 + i0 + u) * 32 + lane;
            if (i0 + u < nt && v < nv) {
                uint4 o;
                o.x = rs_scale_pair(q[u].x, sc);
                o.y = rs_scale_pair(q[u].y, sc);
                o.z = rs_scale_pair(q[u].z, sc);
                o.w = rs_scale_pair(q[u].w, sc);
                if (v == lab_v) {  // column lab & 7 of the 8: half (lab & 1) of word (lab & 7) >> 1
                    const uint32_t gb = __bfloat16_as_ushort(__float2bfloat16_rn(g_lab));
                    const int wsel = (lab & 7) >> 1;
                    const bool hi = (lab & 1) != 0;
                    const auto patch = [&](uint32_t &word, int w) {
                        if (w == wsel)
                            word = hi ? ((word & 0xFFFFu) | (gb << 16)) : ((word & 0xFFFF0000u) | gb);
                    };
                    patch(o.x, 0);
                    patch(o.y, 1);
                    patch(o.z, 2);
                    patch(o.w, 3);
                }
                __stcs(rowp + v, o);
            }
        }
    }
}

}  // namespace lf
