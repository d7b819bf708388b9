// lf_internal.h -- declarations shared by the translation units of
// liblayoutfold.so (not part of the public C ABI).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#ifdef LF_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace lf {

// GEMM tile: one CTA owns a BM x BN output tile, the K loop advances BK
// columns (one 128-byte swizzle row of bf16) per pipeline stage.
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;

// Epilogues of the NT GEMM kernel.
enum Epilogue : int {
    EPI_STORE = 0,         // out = bf16_rn(acc)
    EPI_XENT_PARTIAL = 1,  // per (row, N-tile): max, sum exp(z - max); label logit
    EPI_XENT_GRAD = 2,     // grad = bf16_rn(exp(z - lse) - onehot)
    EPI_STORE_T = 3,       // swapped operands: acc = W . X^T, out[m][n] = bf16_rn(acc[n][m]) (pair kernel)
    EPI_XENT_EXP = 4,      // partials as EPI_XENT_PARTIAL, and e = exp(z - tile max) as fp16 into out (pair kernel)
    EPI_XENT_ROW = 5,      // N <= 256: the tile holds whole rows; loss (and the gradient when out is set) directly
};

struct GemmParams {
    int M, N, K;
    int num_m_blocks, num_n_blocks, num_k_blocks, num_tiles;
    void *out;                  // EPI_STORE: bf16 [M,N]; EPI_XENT_GRAD: grad bf16 [M,N]
    const int32_t *labels;      // [M]
    float *part_max;            // [M, num_n_blocks]: max_n z over the tile
    float *part_sum;            // [M, num_n_blocks]: sum_n exp(z - part_max)
    float *label_logit;         // [M]: z[m, labels[m]]
    const float *row_max;       // [M]: max over the whole row (grad pass)
    const float *row_logsum;    // [M]: log sum_n exp(z - row_max) (grad pass)
    int *err;                   // device error word
    unsigned long long timeout_ns;
    int inject;                 // test hook: 1 = CTA 0 never loads its first stage
    int l2_prefetch;            // k-blocks the L2 prefetch stream runs ahead of the loads (0 = off)
    // stream-K (pair kernel): the tiles' K iterations are split evenly over
    // the pairs; a tile split across pairs is finished by the pair holding its
    // first K block, which adds the other pairs' fp32 partials.
    int streamk;                // 1 = stream-K split, 0 = whole tiles
    unsigned epoch;             // value the flags of this launch carry
    float *sk_partials;         // [2 * pairs][128 * 256] fp32 partial accumulators
    unsigned *sk_flags;         // [2 * pairs] = epoch once the slot is written
    // one-pass cross-entropy with gradient (pair kernel): groups of op_Q pairs
    // each hold one 256-row M block (two op_tile-column tiles per pair) per round.
    float *loss;                      // [M]
    unsigned long long *round_flags;  // [2 * pairs]: (epoch << 32) | rounds published
    int op_Q, op_k, op_rounds;        // pairs per M block, M blocks per round, rounds
    int op_tile, op_ntiles;           // N-tile width (128..256, multiple of 32) and ceil(N / op_tile)
    float *op_stash;                  // [CTAs][2 halves x 32 float4 columns][128 rows] float4: a tile's exp values
    // batches of strided views (pair kernel, plain store epilogue): tile
    // index = (batch, N block, M block), M block fastest
    int batch;                        // number of batches (0 or 1: not batched)
    int x_batched, w_batched;         // 0: one X (resp. W) for every batch
    long long ldo;                    // row pitch of out in elements (N when not strided)
    long long stride_o;               // batch stride of out in elements
    // EPI_STORE_T: the MMA's N (the caller's M, rounded up to 16); 0 = BN
    int tile_n;
    // pair kernel, EPI_STORE, EPI_XENT_GRAD and EPI_XENT_EXP: 1 = the output
    // tensor map is valid and the epilogue writes through TMA stores, 0 = plain stores
    int tma_store;
    // pair kernel, whole tiles: the tile order walks bands of band_m M blocks
    // (M block fastest within a band, then the N blocks, then the next band);
    // 0 = one band of all M blocks
    int band_m;
};

// One stream-K partial slot: a CTA's 128 rows x 256 columns of fp32,
// stored as [column / 4][row][4] so each warp access is contiguous.
constexpr int SK_SLOT_FLOATS = BM * BN;

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
