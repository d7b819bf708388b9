// pointwise.cu -- the K=1 outer-product kernels and the cross-entropy combine.
//
// K=1: "Feature request: Schedule a small matmul op as a reduction (or
// pointwise) op" (NVIDIA/Fuser issue 3646) -- a matmul whose contraction has
// length 1 is a broadcast multiply: out[i,j] = a[i] * b[j].  It is pure
// store bandwidth, so the kernel writes 16 bytes per thread per step, one row
// strip per grid row, with about 16 CTAs of 256 threads per SM in total
// (measured on GB300 at 64 x 8388608: 16 per SM with plain stores reaches
// ~90 % of the copy bandwidth; 8 per SM, or evict-first stores, ~70 %).
//
// Combine: "Allow reductions in matmul epilogues" (NVIDIA/Fuser issue 2213),
// the follow-up on reducing a row across output tiles with a grid
// reduction: the per-tile (max, sum-exp) partials of a row are merged as
//   m = max_j m_j,  s = sum_j s_j * exp(m_j - m),  lse = m + log s,
// and the loss is lse - z[label].
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "lf_internal.h"
#include "lf_xent_rescale.cuh"

namespace lf {
namespace {

constexpr float LOG2E = 1.4426950408889634f;

__global__ void __launch_bounds__(256) k_matmul_k1_f32_v4(const float *__restrict__ a, const float *__restrict__ b,
                                                          float *__restrict__ out, int64_t M, int64_t N)
{
    const int64_t n4 = N >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const float4 *b4 = reinterpret_cast<const float4 *>(b);
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        const float ai = __ldg(a + i);
        float4 *orow = reinterpret_cast<float4 *>(out + i * N);
        for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n4; j += stride) {
            const float4 bv = __ldg(b4 + j);
            float4 o;
            o.x = __fmul_rn(ai, bv.x);
            o.y = __fmul_rn(ai, bv.y);
            o.z = __fmul_rn(ai, bv.z);
            o.w = __fmul_rn(ai, bv.w);
            orow[j] = o;
        }
    }
}

__global__ void __launch_bounds__(256) k_matmul_k1_f32_scalar(const float *__restrict__ a, const float *__restrict__ b,
                                                              float *__restrict__ out, int64_t M, int64_t N)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        const float ai = __ldg(a + i);
        for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < N; j += stride)
            out[i * N + j] = __fmul_rn(ai, __ldg(b + j));
    }
}

__device__ __forceinline__ uint32_t mul_pack_bf16(float xi, uint32_t wpair)
{
    const float lo = __uint_as_float(wpair << 16);
    const float hi = __uint_as_float(wpair & 0xffff0000u);
    __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(xi, lo), __fmul_rn(xi, hi));
    return *reinterpret_cast<uint32_t *>(&h);
}

// bf16 K=1 NT product: x [M,1], w [N,1] -> out [M,N], N % 8 == 0, 16-byte aligned.
__global__ void __launch_bounds__(256) k_matmul_k1_bf16_v8(const __nv_bfloat16 *__restrict__ x,
                                                           const __nv_bfloat16 *__restrict__ w,
                                                           __nv_bfloat16 *__restrict__ out, int64_t M, int64_t N)
{
    const int64_t n8 = N >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4 *w8 = reinterpret_cast<const uint4 *>(w);
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        const float xi = __bfloat162float(x[i]);
        uint4 *orow = reinterpret_cast<uint4 *>(out + i * N);
        for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n8; j += stride) {
            const uint4 wv = __ldg(w8 + j);
            uint4 o;
            o.x = mul_pack_bf16(xi, wv.x);
            o.y = mul_pack_bf16(xi, wv.y);
            o.z = mul_pack_bf16(xi, wv.z);
            o.w = mul_pack_bf16(xi, wv.w);
            orow[j] = o;
        }
    }
}

// One warp per row: merge the row's per-tile partials.
__global__ void __launch_bounds__(256) k_xent_combine(const float *__restrict__ part_max,
                                                      const float *__restrict__ part_sum,
                                                      const float *__restrict__ label_logit,
                                                      const int32_t *__restrict__ labels, int M, int N, int NB,
                                                      float *__restrict__ loss, float *__restrict__ row_max,
                                                      float *__restrict__ row_logsum)
{
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= M)
        return;
    const float *pm = part_max + static_cast<size_t>(row) * NB;
    const float *ps = part_sum + static_cast<size_t>(row) * NB;
    float m = -CUDART_INF_F;
    for (int j = lane; j < NB; j += 32)
        m = fmaxf(m, pm[j]);
#pragma unroll
    for (int o = 16; o; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
    for (int j = lane; j < NB; j += 32)
        s += ps[j] * exp2f((pm[j] - m) * LOG2E);
#pragma unroll
    for (int o = 16; o; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
        const float ls = logf(s);
        const int lab = labels[row];
        loss[row] = (lab >= 0 && lab < N) ? (m - label_logit[row]) + ls : CUDART_NAN_F;
        if (row_max) {
            row_max[row] = m;
            row_logsum[row] = ls;
        }
    }
}

// Second pass of the cross-entropy gradient after the GEMM's exp epilogue
// ("Allow reductions in matmul epilogues": the row's log-sum-exp is a
// reduction across the row's output tiles, merged here, and the gradient
// reuses it; the arithmetic is xent_rescale_unit's, lf_xent_rescale.cuh).
// Every unit the GEMM did not take: with band_done, the first band_done[b]
// units of each of the first rs_bands bands (per_band units each) were
// rescaled inside the GEMM and are skipped.  Eight warps per CTA, each taking
// every (warps in the grid)-th unit, so the loads of many units are in flight
// on every SM.
constexpr int RESCALE_THREADS = 256;
constexpr int RESCALE_MAX_CTAS = 4096;

__global__ void __launch_bounds__(RESCALE_THREADS) k_xent_rescale(const RescaleArgs a,
                                                                  const unsigned *__restrict__ band_done,
                                                                  long long per_band, int rs_bands, long long total)
{
    const long long warps = static_cast<long long>(gridDim.x) * (RESCALE_THREADS / 32);
    const int upr = rs_units_per_row(a.NB);
    for (long long u = static_cast<long long>(blockIdx.x) * (RESCALE_THREADS / 32) + (threadIdx.x >> 5); u < total;
         u += warps) {
        if (band_done) {
            const long long b = u / per_band;
            if (b < rs_bands && u - b * per_band < static_cast<long long>(__ldcg(band_done + b)))
                continue;  // done inside the GEMM
        }
        xent_rescale_unit(a, static_cast<int>(u / upr), static_cast<int>(u % upr));
    }
}

// Test hook: hold an SM's shared memory (OCCUPY_SMEM bytes, so no GEMM CTA
// fits beside it) for `ns` nanoseconds, then exit.  The wait is a fixed time
// on the global timer, so it always ends.
constexpr int OCCUPY_SMEM = 200 * 1024;

__global__ void k_occupy_sm(unsigned long long ns)
{
    extern __shared__ unsigned char occupy_smem[];
    if (threadIdx.x != 0)
        return;
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
        __nanosleep(1000);
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    } while (t - t0 < ns);
    occupy_smem[0] = 1;
}

void grid_for_rows(int64_t M, int64_t cols, int num_sms, dim3 &grid)
{
    const int64_t gy = M < 65535 ? M : 65535;
    int64_t gx = (cols + 255) / 256;
    const int64_t cap = (static_cast<int64_t>(num_sms) * 16 + gy - 1) / gy;  // ~16 CTAs per SM in total
    if (gx > cap)
        gx = cap;
    if (gx < 1)
        gx = 1;
    grid = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
}

}  // namespace

cudaError_t launch_matmul_k1_f32(const float *a, const float *b, float *out, int64_t M, int64_t N, int num_sms,
                                 cudaStream_t s)
{
    const bool vec = (N % 4 == 0) && (reinterpret_cast<uintptr_t>(b) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(out) % 16 == 0);
    dim3 grid;
    grid_for_rows(M, vec ? N / 4 : N, num_sms, grid);
    if (vec)
        k_matmul_k1_f32_v4<<<grid, 256, 0, s>>>(a, b, out, M, N);
    else
        k_matmul_k1_f32_scalar<<<grid, 256, 0, s>>>(a, b, out, M, N);
    return cudaGetLastError();
}

cudaError_t launch_matmul_k1_bf16(const void *x, const void *w, void *out, int64_t M, int64_t N, int num_sms,
                                  cudaStream_t s)
{
    dim3 grid;
    grid_for_rows(M, N / 8, num_sms, grid);
    k_matmul_k1_bf16_v8<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(x),
                                             static_cast<const __nv_bfloat16 *>(w),
                                             static_cast<__nv_bfloat16 *>(out), M, N);
    return cudaGetLastError();
}

cudaError_t launch_xent_combine(const float *part_max, const float *part_sum, const float *label_logit,
                                const int32_t *labels, int M, int N, int num_n_blocks, float *loss, float *row_max,
                                float *row_logsum, cudaStream_t s)
{
    const int rows_per_block = 8;
    const int grid = (M + rows_per_block - 1) / rows_per_block;
    k_xent_combine<<<grid, 32 * rows_per_block, 0, s>>>(part_max, part_sum, label_logit, labels, M, N,
                                                         num_n_blocks, loss, row_max, row_logsum);
    return cudaGetLastError();
}

cudaError_t launch_xent_rescale(const float *part_max, const float *part_sum, const float *label_logit,
                                const int32_t *labels, int M, int N, int num_n_blocks, float *loss, void *grad,
                                const unsigned *band_done, long long units_per_band, int rs_bands, cudaStream_t s)
{
    const RescaleArgs a = {part_max, part_sum, label_logit, labels, M, N, num_n_blocks, loss,
                           static_cast<uint4 *>(grad)};
    const long long total = static_cast<long long>(M) * rs_units_per_row(num_n_blocks);
    const long long need = (total + RESCALE_THREADS / 32 - 1) / (RESCALE_THREADS / 32);
    const int grid = static_cast<int>(need < RESCALE_MAX_CTAS ? need : RESCALE_MAX_CTAS);
    k_xent_rescale<<<grid, RESCALE_THREADS, 0, s>>>(a, band_done, units_per_band > 0 ? units_per_band : 1,
                                                     rs_bands, total);
    return cudaGetLastError();
}

cudaError_t launch_occupy_sms(int ctas, unsigned long long ns, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(k_occupy_sm, cudaFuncAttributeMaxDynamicSharedMemorySize, OCCUPY_SMEM);
    if (e != cudaSuccess)
        return e;
    k_occupy_sm<<<ctas, 32, OCCUPY_SMEM, s>>>(ns);
    return cudaGetLastError();
}

}  // namespace lf
