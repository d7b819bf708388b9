// rope.cu -- the RoPE segment around the K=1 matmul, in one kernel.
//
// Source: "Feature request: Schedule a small matmul op as a reduction (or
// pointwise) op" (NVIDIA/Fuser issue 3646), the Mistral forward listing: the
// [64,1] x [1,4096] matmul (T19) of the inverse frequencies (T3, bf16) and the
// position ids (T4, int64), its permute to [4096,64] (T20), the two pads and
// the cat that repeat it to 128 columns (T21..T23), cosf (T24) and the cast to
// bf16 (T26).  The page notes that the matmul, sent to a library, splits this
// segment into separate kernels; here the K=1 product is a broadcast multiply
// and everything after it happens in registers: each thread computes 8
// angles of one position, already in the permuted [S, H] order, and stores
// their cosines (and sines) as bf16 to both halves of the 2H-column row.
#include <cuda_bf16.h>

#include "lf_internal.h"

namespace lf {
namespace {

constexpr int THREADS = 256;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// H % 8 == 0, inv_freq and the outputs 16-byte aligned.  Work item = (s, 8
// consecutive frequencies).
__global__ void __launch_bounds__(THREADS) k_rope_cos_sin_v8(const __nv_bfloat16 *__restrict__ inv_freq,
                                                              const int64_t *__restrict__ pos,
                                                              __nv_bfloat16 *__restrict__ cos_out,
                                                              __nv_bfloat16 *__restrict__ sin_out, int64_t H,
                                                              int64_t S)
{
    const int64_t groups = H / 8, items = S * groups;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x; it < items;
         it += static_cast<int64_t>(gridDim.x) * THREADS) {
        const int64_t s = it / groups, i0 = (it % groups) * 8;
        const float p = static_cast<float>(__ldg(pos + s));  // int64 -> fp32, round to nearest
        const uint4 f8 = __ldg(reinterpret_cast<const uint4 *>(inv_freq + i0));
        const uint32_t w[4] = {f8.x, f8.y, f8.z, f8.w};
        uint32_t c[4], sn[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a0 = __fmul_rn(__uint_as_float(w[j] << 16), p);           // T19, one fp32 multiply
            const float a1 = __fmul_rn(__uint_as_float(w[j] & 0xffff0000u), p);
            float s0, c0, s1, c1;
            sincosf(a0, &s0, &c0);
            sincosf(a1, &s1, &c1);
            c[j] = pack_bf16x2(c0, c1);
            sn[j] = pack_bf16x2(s0, s1);
        }
        const uint4 cv = make_uint4(c[0], c[1], c[2], c[3]);
        __nv_bfloat16 *crow = cos_out + s * 2 * H;
        *reinterpret_cast<uint4 *>(crow + i0) = cv;       // first half of the cat
        *reinterpret_cast<uint4 *>(crow + H + i0) = cv;   // second half
        if (sin_out) {
            const uint4 sv = make_uint4(sn[0], sn[1], sn[2], sn[3]);
            __nv_bfloat16 *srow = sin_out + s * 2 * H;
            *reinterpret_cast<uint4 *>(srow + i0) = sv;
            *reinterpret_cast<uint4 *>(srow + H + i0) = sv;
        }
    }
}

// Any H and 2-byte alignment: work item = (s, i).
__global__ void __launch_bounds__(THREADS) k_rope_cos_sin_scalar(const __nv_bfloat16 *__restrict__ inv_freq,
                                                                  const int64_t *__restrict__ pos,
                                                                  __nv_bfloat16 *__restrict__ cos_out,
                                                                  __nv_bfloat16 *__restrict__ sin_out, int64_t H,
                                                                  int64_t S)
{
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x; it < S * H;
         it += static_cast<int64_t>(gridDim.x) * THREADS) {
        const int64_t s = it / H, i = it % H;
        const float a = __fmul_rn(__bfloat162float(inv_freq[i]), static_cast<float>(pos[s]));
        float sv, cv;
        sincosf(a, &sv, &cv);
        const __nv_bfloat16 cb = __float2bfloat16_rn(cv);
        cos_out[s * 2 * H + i] = cb;
        cos_out[s * 2 * H + H + i] = cb;
        if (sin_out) {
            const __nv_bfloat16 sb = __float2bfloat16_rn(sv);
            sin_out[s * 2 * H + i] = sb;
            sin_out[s * 2 * H + H + i] = sb;
        }
    }
}

}  // namespace

cudaError_t launch_rope_cos_sin(const void *inv_freq, const int64_t *pos, void *cos_out, void *sin_out, int64_t H,
                                int64_t S, int num_sms, cudaStream_t s)
{
    const auto inv = static_cast<const __nv_bfloat16 *>(inv_freq);
    const auto co = static_cast<__nv_bfloat16 *>(cos_out);
    const auto so = static_cast<__nv_bfloat16 *>(sin_out);
    const auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool vec = H % 8 == 0 && a16(inv_freq) && a16(cos_out) && (sin_out == nullptr || a16(sin_out));
    const int64_t items = vec ? S * (H / 8) : S * H;
    int64_t blocks = (items + THREADS - 1) / THREADS;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap)
        blocks = cap;
    if (vec)
        k_rope_cos_sin_v8<<<static_cast<unsigned>(blocks), THREADS, 0, s>>>(inv, pos, co, so, H, S);
    else
        k_rope_cos_sin_scalar<<<static_cast<unsigned>(blocks), THREADS, 0, s>>>(inv, pos, co, so, H, S);
    return cudaGetLastError();
}

}  // namespace lf
