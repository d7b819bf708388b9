// lf_kernel_params.h -- what the GEMM kernels are compiled from besides their
// own sources: the tile constants, the epilogue selector and the parameter
// block every launch passes by value.  Host-only declarations live in
// lf_internal.h, which includes this file.
#pragma once
#include <cstdint>

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
    // pair kernel, whole tiles: 1 = pair i starts with tile i and claims every
    // further tile from tile_ctl[0] (tile order as for band_m).  tile_ctl[1]
    // counts the pairs whose claiming is over; the pair that completes the
    // count zeroes both words, so every launch finds them zero.
    int dyn_tiles;
    unsigned *tile_ctl;
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
    // pair kernel: K blocks per stage of the operand ring (1 or 2; the ring's
    // six one-K-block slots grouped into six or three stages)
    int ksub;
    // pair kernel, MN-major operands (not batched): bit 0 / bit 1 = X's / W's
    // map is the 3-D view (64 rows, K, rows / 64) whose box brings both 64-row
    // halves of the CTA's 128 rows in one copy
    int mn3;
    // pair kernel, whole tiles: the tile order walks bands of band_m M blocks
    // (M block fastest within a band, then the N blocks, then the next band);
    // 0 = one band of all M blocks
    int band_m;
};

// One stream-K partial slot: a CTA's 128 rows x 256 columns of fp32,
// stored as [column / 4][row][4] so each warp access is contiguous.
constexpr int SK_SLOT_FLOATS = BM * BN;

}  // namespace lf
