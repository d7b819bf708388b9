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
// reuses it).  One CTA per row:
//   1. the combine: m = max_j m_j, s = sum_j s_j exp(m_j - m), lse = m + log s,
//      loss = lse - z[label] (NaN for a label outside [0, N));
//   2. per 256-column tile j: scale_j = exp(m_j - lse) into shared memory;
//   3. the row of grad, which holds e = fp16(exp(z - m_j)), is rewritten in
//      place, 8 columns (16 bytes) per load and store:
//        grad = bf16_rn(e * scale_j),
//      except the label column, computed from the fp32 label logit:
//        grad[label] = bf16_rn(exp(z[label] - lse) - 1).
// Error: fp16 keeps e to 2^-11 relative, so a non-label entry p < 1/2 is off by
// at most p 2^-11 (+ 1e-6) before its bf16 rounding (<= 9.8e-4 below 1/2): under
// 1.3e-3 in all; an entry p >= 1/2 is the row's (hence its tile's) maximum,
// where e = 1 exactly, so only its bf16 rounding remains.  The label entry is
// computed as in the single-pass epilogues.
constexpr int RESCALE_THREADS = 256;

__device__ __forceinline__ float ex2_approx_pw(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t rescale_pair(uint32_t hpair, float scale)
{
    const __half2 h = *reinterpret_cast<const __half2 *>(&hpair);
    const float2 f = __half22float2(h);
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    return *reinterpret_cast<uint32_t *>(&b);
}

__global__ void __launch_bounds__(RESCALE_THREADS) k_xent_rescale(const float *__restrict__ part_max,
                                                                  const float *__restrict__ part_sum,
                                                                  const float *__restrict__ label_logit,
                                                                  const int32_t *__restrict__ labels, int M, int N,
                                                                  int NB, float *__restrict__ loss,
                                                                  uint4 *__restrict__ grad)
{
    extern __shared__ float scale[];  // [NB]
    __shared__ float red[RESCALE_THREADS / 32];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    for (int row = blockIdx.x; row < M; row += gridDim.x) {
        const float *pm = part_max + static_cast<size_t>(row) * NB;
        const float *ps = part_sum + static_cast<size_t>(row) * NB;
        // 1. the row's max and rescaled sum over its tiles
        float m = -CUDART_INF_F;
        for (int j = tid; j < NB; j += RESCALE_THREADS)
            m = fmaxf(m, pm[j]);
#pragma unroll
        for (int o = 16; o; o >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0)
            red[warp] = m;
        __syncthreads();
        m = red[0];
#pragma unroll
        for (int w = 1; w < RESCALE_THREADS / 32; ++w)
            m = fmaxf(m, red[w]);
        __syncthreads();
        float s = 0.f;
        for (int j = tid; j < NB; j += RESCALE_THREADS)
            s += ps[j] * exp2f((pm[j] - m) * LOG2E);
#pragma unroll
        for (int o = 16; o; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0)
            red[warp] = s;
        __syncthreads();
        s = 0.f;
#pragma unroll
        for (int w = 0; w < RESCALE_THREADS / 32; ++w)
            s += red[w];
        const float ls = logf(s);
        const float lse = m + ls;
        const int lab = labels[row];
        const bool lab_ok = lab >= 0 && lab < N;
        const float zl = lab_ok ? label_logit[row] : 0.f;
        if (tid == 0)
            loss[row] = lab_ok ? (m - zl) + ls : CUDART_NAN_F;
        // 2. per-tile scales exp(m_j - lse)
        const float lsel = lse * LOG2E;
        for (int j = tid; j < NB; j += RESCALE_THREADS)
            scale[j] = ex2_approx_pw(fmaf(pm[j], LOG2E, -lsel));
        __syncthreads();
        // 3. the row, 8 columns per step; the label column from the fp32 logit
        const float g_lab = ex2_approx_pw(fmaf(zl, LOG2E, -lsel)) - 1.f;
        uint4 *rowp = grad + static_cast<size_t>(row) * (N / 8);
        const int nv = N / 8;
        const int lab_v = lab_ok ? lab >> 3 : -1;
        constexpr int U = 4;
        for (int v0 = tid; v0 < nv; v0 += U * RESCALE_THREADS) {
            uint4 q[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * RESCALE_THREADS;
                if (v < nv)
                    q[u] = __ldcs(rowp + v);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * RESCALE_THREADS;
                if (v < nv) {
                    const float sc = scale[v >> 5];  // 256 columns = 32 vectors per tile
                    uint4 o;
                    o.x = rescale_pair(q[u].x, sc);
                    o.y = rescale_pair(q[u].y, sc);
                    o.z = rescale_pair(q[u].z, sc);
                    o.w = rescale_pair(q[u].w, sc);
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
        __syncthreads();  // scale[] and red[] are rewritten for the next row
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
                                cudaStream_t s)
{
    const size_t smem = static_cast<size_t>(num_n_blocks) * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_xent_rescale, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
    }
    const int grid = M < (1 << 30) ? M : (1 << 30);
    k_xent_rescale<<<grid, RESCALE_THREADS, smem, s>>>(part_max, part_sum, label_logit, labels, M, N, num_n_blocks,
                                                       loss, static_cast<uint4 *>(grad));
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
