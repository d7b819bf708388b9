// lf_internal.h -- declarations shared by the translation units of
// liblayoutfold.so (not part of the public C ABI).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#ifdef LF_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

#include "lf_kernel_params.h"

namespace lf {

// Launchers (host).  Return cudaSuccess or the launch error.
cudaError_t launch_gemm_nt(int epi, const CUtensorMap &ta, const CUtensorMap &tb, const GemmParams &p,
                           int grid, cudaStream_t s);
int gemm_smem_bytes();

// CTA-pair variant (cta_group::2, 256x256 tiles; p.num_m_blocks counts
// 256-row blocks; grid even).  layout bit 0: X stored [K,M] (tensor map over
// [K rows, M columns], 64x64 boxes), else [M,K] (64-column x 128-row boxes);
// bit 1: W stored [K,N] likewise, else [N,K]; bit 2: batched (3-D tensor
// maps, batch outermost; p.batch, p.w_batched, p.ldo, p.stride_o).  Layouts
// 1..3 take the EPI_STORE and cross-entropy epilogues, batched layouts
// EPI_STORE only.  `to`: the output as a
// bf16 tensor map (2-D [M rows, N columns], row pitch p.ldo; 3-D with the
// batch outermost when batched), 32 x 32 boxes, 64-byte swizzle -- read only
// when p.tma_store is set.
cudaError_t launch_gemm_nt_pair(int epi, int layout, const CUtensorMap &ta, const CUtensorMap &tb,
                                const CUtensorMap &to, const GemmParams &p, int grid, cudaStream_t s);
int gemm_pair_smem_bytes();
int gemm_pair_max_active_clusters();

// One-pass GEMM + cross-entropy + gradient on CTA pairs (no recompute GEMM,
// no combine kernel).  Requires op_k * op_Q co-resident pairs; grid = 2 * op_k * op_Q.
// `to`: the gradient (p.out) as a 2-D bf16 map, 32 x 32 boxes, 64-byte swizzle.
// layout bit 0: X stored [K,M] (ta as for the pair kernel: 64 x 64 boxes); bit
// 1: W stored [K,N] (tb with 64 x 64 boxes; op_tile 128 or 256), else tb's box
// is op_tile / 2 rows of W [N,K].
cudaError_t launch_xent_onepass(int layout, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &to,
                                const GemmParams &p, int grid, cudaStream_t s);

cudaError_t launch_xent_combine(const float *part_max, const float *part_sum, const float *label_logit,
                                const int32_t *labels, int M, int N, int num_n_blocks, float *loss,
                                float *row_max, float *row_logsum, cudaStream_t s);

// Second pass of the cross-entropy gradient after EPI_XENT_EXP: per row, the
// combine (lse from the tile partials, loss), then grad rewritten in place
// from the fp16 e = exp(z - tile max) it holds: grad = bf16_rn(e * exp(tile
// max - lse)), the label column from the fp32 label logit.
cudaError_t launch_xent_rescale(const float *part_max, const float *part_sum, const float *label_logit,
                                const int32_t *labels, int M, int N, int num_n_blocks, float *loss, void *grad,
                                cudaStream_t s);

cudaError_t launch_matmul_k1_f32(const float *a, const float *b, float *out, int64_t M, int64_t N,
                                 int num_sms, cudaStream_t s);
cudaError_t launch_matmul_k1_bf16(const void *x, const void *w, void *out, int64_t M, int64_t N,
                                  int num_sms, cudaStream_t s);
cudaError_t launch_rope_cos_sin(const void *inv_freq, const int64_t *pos, void *cos_out, void *sin_out, int64_t H,
                                int64_t S, int num_sms, cudaStream_t s);
cudaError_t launch_fp8_cast_dual(const void *x, const float *scale, void *out, void *out_t, int64_t M, int64_t K,
                                 int num_sms, cudaStream_t s);
// Test hook: `ctas` CTAs, each holding 200 KiB of shared memory (one per SM),
// that wait `ns` nanoseconds on the global timer and exit.
cudaError_t launch_occupy_sms(int ctas, unsigned long long ns, cudaStream_t s);

// A profiling range around one entry-point call: an NVTX range named after
// the call when the library is built with LF_NVTX defined, nothing otherwise.
struct CallRange {
    explicit CallRange(const char *name)
    {
#ifdef LF_NVTX
        nvtxRangePushA(name);
#else
        (void)name;
#endif
    }
    ~CallRange()
    {
#ifdef LF_NVTX
        nvtxRangePop();
#endif
    }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

// Library state and helpers shared by the entry points of every translation
// unit (defined in api.cu).
unsigned long long wait_timeout_ns();  // device-side wait limit (lf_set_test_hooks; 2 s by default)
bool cooperative_launches();           // false after lf_set_cooperative(0)
int stall_injection();                 // 1 while lf_set_test_hooks asks for a stalled first stage
void count_launches(int n);            // adds n to the lf_launch_count total
bool debug_sync_enabled();             // LF_DEBUG_SYNC is set in the environment
// 2-D bf16 tensor [rows, K] (K contiguous) as a TMA map: boxes of 64 columns x
// box_rows rows, 128-byte swizzle, zero fill out of bounds.  False if the
// driver entry point is missing or rejects the layout.
bool make_tmap_kmajor(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, uint32_t box_rows);

}  // namespace lf
