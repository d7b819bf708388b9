// gemm_nt_tc.cu -- the NT GEMM  acc = X[M,K] · W[N,K]^T  on the sm_103a tensor
// cores, with four epilogues (bf16 store, cross-entropy partials, gradient, and
// the whole cross-entropy of rows that fit one tile).
//
// Source: "Strength reduction: fold transpose into a subsequent GEMM call"
// (lightning-thunder issue 1252), Feature/Motivation: the weight is consumed in
// its stored [N,K] layout -- both operands are K-major tiles, so the transpose
// the traced program materialises never exists.  "Allow reductions in matmul
// epilogues" (NVIDIA/Fuser issue 2213): the cross-entropy reduction runs in
// the epilogue of the same kernel, tile by tile, with a grid-level combine.
//
// Structure (one persistent CTA per SM, 192 threads):
//   warp 0      : TMA producer -- loads a 128x64 tile of X and a 256x64 tile of
//                 W per stage into a 4-deep shared-memory ring (128-byte swizzle).
//   warp 1      : owns the TMEM allocation (2 x 256 fp32 columns) and, from one
//                 lane, issues tcgen05.mma (M=128, N=256, K=16) into the current
//                 accumulator buffer; tcgen05.commit frees ring slots / hands a
//                 finished accumulator to the epilogue.
//   warps 2..5  : epilogue -- warp w reads TMEM lanes 32*(w%4).. (one output row
//                 per thread) while the MMA warp fills the other accumulator.
// Tiles are visited M-block fastest, so the CTAs that share a W tile run at
// the same time and W streams from HBM about once.
//
// Every wait is bounded (%globaltimer): a wait that passes the limit records
// an error code in the device error word, raises a CTA-wide abort flag, and
// all roles unwind -- copies in flight are waited for, issued MMAs are drained
// and TMEM is freed before the CTA exits.  No trap, no assert.
#include <atomic>

#include "lf_gemm_common.cuh"

namespace lf {
namespace {

constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;   // 16 KiB
constexpr int B_BYTES = BN * BK * 2;   // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;  // 512 = all of TMEM
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + NUM_BARS * 8 + 16;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_nt(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128B-swizzle atoms need 1024-byte alignment
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + STAGES * A_BYTES;
    const uint32_t bar0 = base + STAGES * STAGE_BYTES;
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * ACC_BUFS);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + STAGES * STAGE_BYTES + NUM_BARS * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
#define FULL_BAR(s) (bar0 + 8u * (s))
#define EMPTY_BAR(s) (bar0 + 8u * (STAGES + (s)))
#define TFULL_BAR(b) (bar0 + 8u * (2 * STAGES + (b)))
#define TEMPTY_BAR(b) (bar0 + 8u * (2 * STAGES + ACC_BUFS + (b)))

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(FULL_BAR(s), 1);
            mbar_init(EMPTY_BAR(s), 1);
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            mbar_init(TFULL_BAR(b), 1);
            mbar_init(TEMPTY_BAR(b), EPI_THREADS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s)
                armed[s] = 0;
            bool ok = true, first = true;
            // L2 prefetch cursor: walks the same (tile, k-block) sequence as the
            // loads, l2_prefetch steps ahead, so operand slices are already in
            // L2 when their shared-memory load is issued.
            int pf_tile = blockIdx.x, pf_kb = 0;
            auto prefetch_next = [&]() {
                if (pf_tile < p.num_tiles) {
                    tma_prefetch_l2_2d(&tmA, pf_kb * BK, (pf_tile % p.num_m_blocks) * BM);
                    tma_prefetch_l2_2d(&tmB, pf_kb * BK, (pf_tile / p.num_m_blocks) * BN);
                    if (++pf_kb == p.num_k_blocks) {
                        pf_kb = 0;
                        pf_tile += gridDim.x;
                    }
                }
            };
            for (int i = 0; i < p.l2_prefetch; ++i)
                prefetch_next();
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                const int mb = tile % p.num_m_blocks;
                const int nb = tile / p.num_m_blocks;
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!wait_bar(EMPTY_BAR(stage), phase ^ 1u, abort_flag, p, ERR_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    if (p.l2_prefetch > 0)
                        prefetch_next();
                    const bool skip = first && p.inject == 1 && blockIdx.x == 0;
                    first = false;
                    if (!skip) {
                        mbar_arrive_expect_tx(FULL_BAR(stage), STAGE_BYTES);
                        tma_load_2d(sA + stage * A_BYTES, &tmA, kb * BK, mb * BM, FULL_BAR(stage));
                        tma_load_2d(sB + stage * B_BYTES, &tmB, kb * BK, nb * BN, FULL_BAR(stage));
                        ++armed[stage];
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Every copy this thread issued must have landed before the CTA exits.
            for (int s = 0; s < STAGES; ++s)
                if (armed[s])
                    wait_bar_drain(FULL_BAR(s), (armed[s] - 1u) & 1u, abort_flag, p);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                if (!wait_bar(TEMPTY_BAR(acc), acc_phase ^ 1u, abort_flag, p, ERR_MMA_ACC))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!wait_bar(FULL_BAR(stage), phase, abort_flag, p, ERR_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sA + stage * A_BYTES;
                    const uint32_t b0 = sB + stage * B_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        umma_f16(d_tmem, smem_desc_k128(a0 + k * UMMA_K * 2), smem_desc_k128(b0 + k * UMMA_K * 2),
                                 IDESC, (kb | k) != 0 ? 1u : 0u);
                    umma_commit(EMPTY_BAR(stage));  // ring slot free once these MMAs have read it
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit(TFULL_BAR(acc));  // accumulator complete
                if (++acc == ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Drain: every MMA this thread issued completes before TMEM is freed.
            umma_commit(drain_bar);
            wait_bar_drain(drain_bar, 0u, abort_flag, p);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
            const int mb = tile % p.num_m_blocks;
            const int nb = tile / p.num_m_blocks;
            const bool ok = wait_bar(TFULL_BAR(acc), acc_phase, abort_flag, p, ERR_EPI);
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc_fence_after();
            const int row = mb * BM + q * 32 + lane;
            const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(q * 32) << 16);
            const PartialAdd none = {nullptr, 0, 0, 0, nullptr, 0, 0u};
            if (EPI == EPI_STORE)
                epi_store(p, taddr, row, nb, none);
            else if (EPI == EPI_XENT_PARTIAL)
                epi_xent_partial(p, taddr, row, nb, none);
            else if (EPI == EPI_XENT_ROW)
                epi_xent_row(p, taddr, row, none);
            else
                epi_xent_grad(p, taddr, row, nb, none);
            tc_fence_before();
            mbar_arrive(TEMPTY_BAR(acc));
            if (++acc == ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }
#undef FULL_BAR
#undef EMPTY_BAR
#undef TFULL_BAR
#undef TEMPTY_BAR

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int EPI>
cudaError_t set_smem_attr_once()
{
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load() & bit)
        return cudaSuccess;
    e = cudaFuncSetAttribute(k_gemm_nt<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e == cudaSuccess)
        done.fetch_or(bit);
    return e;
}

template <int EPI>
cudaError_t launch_t(const CUtensorMap &ta, const CUtensorMap &tb, const GemmParams &p, int grid, cudaStream_t s)
{
    cudaError_t e = set_smem_attr_once<EPI>();
    if (e != cudaSuccess)
        return e;
    k_gemm_nt<EPI><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(ta, tb, p);
    return cudaGetLastError();
}

}  // namespace

int gemm_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_gemm_nt(int epi, const CUtensorMap &ta, const CUtensorMap &tb, const GemmParams &p, int grid,
                           cudaStream_t s)
{
    switch (epi) {
    case EPI_STORE:
        return launch_t<EPI_STORE>(ta, tb, p, grid, s);
    case EPI_XENT_PARTIAL:
        return launch_t<EPI_XENT_PARTIAL>(ta, tb, p, grid, s);
    case EPI_XENT_GRAD:
        return launch_t<EPI_XENT_GRAD>(ta, tb, p, grid, s);
    case EPI_XENT_ROW:
        return launch_t<EPI_XENT_ROW>(ta, tb, p, grid, s);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace lf
