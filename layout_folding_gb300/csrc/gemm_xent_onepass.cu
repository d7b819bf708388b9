// gemm_xent_onepass.cu -- GEMM + row-wise cross-entropy + gradient in ONE
// pass over the tensor cores: the logits are computed once, never written to
// memory, and the gradient comes from the accumulators (one tile of each
// pair by way of a stash in L2, so its accumulator is freed early).
//
// Source: "Allow reductions in matmul epilogues" (NVIDIA/Fuser issue 2213):
// the fusion example (row max, sum-exp, log-sum-exp, label logit, and the
// softmax-minus-onehot output) and the follow-up: a row reduction across the
// tiles of a row needs a grid reduction, and when the epilogue must reuse the
// reduced value (here: the gradient needs the row's log-sum-exp) every CTA of
// a row of tiles has to be resident at once so the result can be broadcast
// back.  That is what this kernel does, one 256-row block of rows at a time.
//
// Operand layouts (template LAYOUT, as in the pair GEMM kernel): bit 0 X stored
// [K,M], bit 1 W stored [K,N] -- loaded as 64 x 64 boxes and read through
// MN-major descriptors, never transposed in memory.
//
// Schedule: CTA pairs (tcgen05 cta_group::2, M=256 x N=op_tile MMAs; op_tile
// is 256, or 128..224 for problems that fit one round of pairs) form groups of
// Q = ceil(N_tiles / 2) pairs; pair qi of a group owns N tiles 2qi and 2qi+1
// of the group's M block.  k = floor(pairs / Q) groups run side by side, so a
// round covers k M blocks; round r of group g is M block r*k + g.  The tile
// processed first in a round (order 0) goes to accumulator 0 (TMEM columns
// [0, op_tile)), the second to accumulator 1 ([256, 256 + op_tile)); the two
// W tiles alternate their order every round so the next round starts on the
// W rows L2 still holds.  Per round:
//   1. mainloop of the pair's one or two tiles (same TMA/MMA machinery as the
//      pair GEMM kernel); the first tile of a round is the previous round's
//      last, and its K blocks are walked downwards, so the first loads find
//      the slices L2 still holds (the second tiles of a round, ~136 MB at the
//      bench shape, do not all fit; ascending, almost none hit);
//   2. epilogue (8 warps; a thread owns a row, warpgroup h takes columns
//      [128h, 128h + 128) of every tile): per-(row, half tile) statistics
//      (max, sum exp(z - max), label logit) in one pass over TMEM with a
//      running max.  Tile 0's exp values go to a per-CTA stash in global
//      memory (L2) while tile 1's MMAs run, and accumulator 0 is released at
//      once, so the next round's first MMAs follow this round's last ones
//      without waiting for the merge; tile 1's stay in TMEM.  Warpgroup 1
//      hands its statistics to warpgroup 0 through shared memory, which
//      merges the pair's four per row, stores one partial per row in slot
//      [qi][row] (partial-major) and releases the CTA's flag (epoch << 32 |
//      round+1) with one cumulative release store;
//   3. one warp polls the flags of the group's Q pairs (acquire, bounded, with
//      backoff) and hands the result to the other warps through an mbarrier;
//      each warpgroup merges half of the row's Q partials (coalesced loads, 16
//      per round trip), the halves are exchanged through shared memory,
//      warpgroup 0 of the group's first pair writes loss[row];
//   4. grad = exp(z - lse) - onehot, tile 1 from TMEM (then accumulator 1 is
//      released), tile 0 from the stash, written by TMA stores of 32 x 32
//      boxes staged per warp in shared memory.
// Measured per round at 4096x32768x4096 (one GB300): two mainloops of ~24.5
// us; the group's merge and the gradient of tile 1 overlap the next round's
// first mainloop (before, with both tiles held in TMEM until the merge, ~16
// us per round ran after the last MMA with the tensor cores idle).
// The producer streams the next round's first K slices into the ring while
// the epilogue runs.  Waits only go to the same round of the same group, whose
// pairs never wait on anything later, so there is no cycle; every wait is
// bounded (2 s) and an abort is mirrored into the peer CTA.
#include <atomic>

#include "lf_gemm_common.cuh"

namespace lf {
namespace {

constexpr int OP_M = 2 * BM;  // 256 rows per pair
constexpr int OP_UMMA_K = 16;
constexpr int OP_STAGES = 6;
constexpr int OP_A_BYTES = BM * BK * 2;        // this CTA's 128 rows of X
constexpr int OP_B_BYTES = (BN / 2) * BK * 2;  // room for this CTA's op_tile / 2 (<= 128) rows of W
constexpr int OP_STAGE_BYTES = OP_A_BYTES + OP_B_BYTES;
constexpr int OP_TMEM_COLS = 2 * BN;  // tile 0: columns [0, op_tile), tile 1: [256, 256 + op_tile)
constexpr int OP_THREADS = 320;     // producer, MMA, and one epilogue warpgroup per tile
constexpr int OP_EPI_WARPS = 4;    // per warpgroup (= per tile)
constexpr int OP_NUM_BARS = 2 * OP_STAGES + 2 + 2 + 5;  // ring, tfull[2], tempty[2], drain, publish, exchange, merge, group
constexpr int OP_XCH_BYTES = 8 * BM * 4;  // (max, sum) per row: 2 half-tile statistics + 2 half merges
constexpr int OP_HALF = BN / 2;           // columns of a tile taken by one epilogue warpgroup
constexpr int OP_HCH = OP_HALF / 32;      // 32-column chunks of a half
constexpr int OP_STG_WARP_BYTES = 32 * 32 * 2;            // a warp's 32 rows x 32 bf16 gradient columns
constexpr int OP_STG_OFF =
    ((OP_STAGES * OP_STAGE_BYTES + OP_NUM_BARS * 8 + 16 + OP_XCH_BYTES + 1023) / 1024) * 1024;
constexpr int OP_SMEM_BYTES = 1024 + OP_STG_OFF + 2 * OP_EPI_WARPS * OP_STG_WARP_BYTES;
constexpr uint64_t OP_ABORT_SETTLE_NS = 100000;
// MN-major operands (LAYOUT bit 0: X stored [K,M]; bit 1: W stored [K,N]) arrive
// as 64 (M or N) x 64 (K) boxes per K slice, the next box 8 KiB further; each
// K=16 step of the MMA advances two 1024-byte atoms.
constexpr uint32_t OP_MN_BOX = 8192;
constexpr uint32_t OP_MN_KSTEP = 2 * 1024;
constexpr int ERR_OP_FLAG = 0x108;  // a group member never published its partials

// L2 eviction policy: lines written with it are evicted after other lines.
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte store with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void st_f4_hint(float4 *ptr, float4 v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w), "l"(pol)
                 : "memory");
}

struct OpWork {
    int mb, nb0, ntile;
    bool swap;  // process the pair's second tile first this round
};

// Round r of `pair`: its M block and its N tiles nb0 (and nb0 + 1 if ntile == 2).
__device__ __forceinline__ bool op_work(const GemmParams &p, int pair, int r, OpWork &w)
{
    const int grp = pair / p.op_Q;
    const int qi = pair % p.op_Q;
    w.mb = r * p.op_k + grp;
    if (w.mb >= p.num_m_blocks)
        return false;
    w.nb0 = 2 * qi;  // < op_ntiles because op_Q = ceil(op_ntiles / 2)
    w.ntile = (w.nb0 + 1 < p.op_ntiles) ? 2 : 1;
    // Alternate the order of the two tiles every round: the W rows of the tile
    // processed last are what L2 still holds, so the next round starts there.
    w.swap = (r & 1) && w.ntile == 2;
    return true;
}

// Tree max / sum of the first `n` (all when FULL) of 32 values held as bits.
template <bool FULL>
__device__ __forceinline__ float op_tree_max_bits(const uint32_t (&u)[32], int n)
{
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float lo = (FULL || i < n) ? __uint_as_float(u[i]) : -CUDART_INF_F;
        const float hi = (FULL || i + 16 < n) ? __uint_as_float(u[i + 16]) : -CUDART_INF_F;
        t[i] = fmaxf(lo, hi);
    }
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i)
            t[i] = fmaxf(t[i], t[i + w]);
    return t[0];
}

__device__ __forceinline__ float op_tree_sum_bits(const uint32_t (&u)[32])
{
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        t[i] = __uint_as_float(u[i]) + __uint_as_float(u[i + 16]);
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i)
            t[i] += t[i + w];
    return t[0];
}

// Merge n (max, sum) partials of one row, pm[j * stride], ps[j * stride] for
// j < n, into the row's max `m` and sum `s` of exp(z - m): online rescaling,
// 16 partials per batch (32 kept too many registers live).  The partials are stored partial-major, so the 32
// rows of a warp read 128 contiguous bytes per partial.
__device__ __forceinline__ float op_tree_max16(const float (&a)[16])
{
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        t[i] = fmaxf(a[i], a[i + 8]);
#pragma unroll
    for (int w = 4; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i)
            t[i] = fmaxf(t[i], t[i + w]);
    return t[0];
}

__device__ __forceinline__ float op_tree_sum16(const float (&a)[16])
{
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        t[i] = a[i] + a[i + 8];
#pragma unroll
    for (int w = 4; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i)
            t[i] += t[i + w];
    return t[0];
}

__device__ __forceinline__ void merge_row_partials(const float *pm, const float *ps, size_t stride, int n, float &m,
                                                   float &s)
{
    m = -CUDART_INF_F;
    s = 0.f;
    for (int j0 = 0; j0 < n; j0 += 16) {
        float a[16], b[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int j = j0 + i;
            a[i] = j < n ? __ldcg(pm + j * stride) : -CUDART_INF_F;
            b[i] = j < n ? __ldcg(ps + j * stride) : 0.f;
        }
        const float nm = fmaxf(m, op_tree_max16(a));
        const float nml = nm * LOG2E;
        s *= ex2_approx((m - nm) * LOG2E);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            b[i] *= ex2_approx(fmaf(a[i], LOG2E, -nml));
        s += op_tree_sum16(b);
        m = nm;
    }
}

// Makes the 32 registers of a TMEM load depend on a point after
// tcgen05.wait::ld, so no use of them is scheduled before the wait.
__device__ __forceinline__ void op_regs_after_wait(uint32_t (&v)[32])
{
    asm volatile(""
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                   "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                   "+r"(v[29]), "+r"(v[30]), "+r"(v[31]));
}

// Statistics of this thread's row of one half tile (columns [col0, lim):
// at most 128, fewer in the second half of a narrower tile or past N) in a
// single pass over TMEM
// ("Allow reductions in matmul epilogues", fusion example: row max, exp(z -
// max) and its sum, the label logit).  Chunk c is taken relative to the
// running max m_c (the max over chunks 0..c): e = exp(z - m_c) is written
// back over z, and the sum is rescaled whenever the max grows, so the tile
// is read once.  Returns the tile's max and sum of exp(z - max); cm[c] = m_c,
// from which the gradient rescales chunk c.  The next chunk's TMEM load is in
// flight while the current one is processed; max and sum are tree reductions.
// FULL: all 128 columns of the half are in [col0, lim).  With `stash` set the
// exp values go to this thread's stash slots (float4 column j of the half at
// stash[j * BM]) instead of back into TMEM, so the accumulator can be reused;
// they are written with an L2 evict-last policy, so the ~17 MB a round stashes
// stay in L2 against the W stream until the gradient reads them back (without
// it about half went to DRAM and came back: +0.5 GB of traffic per call).
template <bool FULL>
__device__ __forceinline__ void op_half_stats(int lim, uint32_t taddr, int col0, int lab, float (&cm)[OP_HCH],
                                              float &mx, float &se, float &zl, bool &have, float4 *stash)
{
    const int lab_local = lab - col0;
    mx = -CUDART_INF_F;
    se = 0.f;
    have = false;
    uint32_t v[2][32];
    tmem_ld_32x32b_x32(taddr, v[0]);
#pragma unroll
    for (int c = 0; c < OP_HCH; ++c) {
        const int nvalid = FULL ? 32 * (OP_HCH - c) : lim - (col0 + c * 32);  // <= 0 past the half's last column
        tmem_wait_ld();
        if (c + 1 < OP_HCH && nvalid > 32)
            tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>((c + 1) * 32), v[(c + 1) & 1]);
        cm[c] = mx;
        if (nvalid > 0) {
            uint32_t(&u)[32] = v[c & 1];
            op_regs_after_wait(u);
            const int li = lab_local - c * 32;
            if (static_cast<unsigned>(li) < 32u) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i == li)
                        zl = __uint_as_float(u[i]);
                have = true;
            }
            const float m_c = fmaxf(mx, op_tree_max_bits<FULL>(u, nvalid));
            const float mcl = m_c * LOG2E;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                u[i] = __float_as_uint((FULL || i < nvalid) ? ex2_approx(fmaf(__uint_as_float(u[i]), LOG2E, -mcl)) : 0.f);
            se = se * ex2_approx((mx - m_c) * LOG2E) + op_tree_sum_bits(u);
            mx = m_c;
            cm[c] = m_c;
            if (stash) {
                const uint64_t pol = policy_evict_last();
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    st_f4_hint(stash + (c * 8 + i) * BM,
                               make_float4(__uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                                           __uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3])),
                               pol);
            } else {
                tmem_st_32x32b_x32(taddr + static_cast<uint32_t>(c * 32), u);
            }
        }
    }
    if (!stash)
        tmem_wait_st();
}

// grad = bf16_rn(e * scale[c] - [n == label]) for this thread's row of one
// half tile, e = exp(z - m_c) read back from TMEM (or from the stash when
// `stash` is set), scale[c] = exp(m_c - lse).  Each 32 x 32 chunk of the
// warp is packed into its 2 KiB staging tile (16-byte pieces XOR-swizzled by
// row pair: the gradient map's 64-byte swizzle) and lane 0 writes it with a
// TMA store, which leaves out rows >= M and columns >= N.  (Double-buffering
// the TMEM loads spilled registers: 168 is the limit at 10 warps per CTA.)
__device__ __forceinline__ void op_half_grad(const GemmParams &p, const CUtensorMap *tmO, int lim, uint32_t taddr,
                                             int row0, int col0, int lab, const float (&scale)[OP_HCH], uint8_t *stg,
                                             uint32_t stg_s, const float4 *stash)
{
    const int lane = threadIdx.x & 31;
    const int lab_local = lab - col0;
#pragma unroll
    for (int c = 0; c < OP_HCH; ++c) {
        const int col = col0 + c * 32;
        const int nvalid = lim - col;  // warp-uniform
        if (nvalid > 0) {
            uint32_t u[32];
            if (stash) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 f = __ldcg(stash + (c * 8 + i) * BM);
                    u[4 * i] = __float_as_uint(f.x);
                    u[4 * i + 1] = __float_as_uint(f.y);
                    u[4 * i + 2] = __float_as_uint(f.z);
                    u[4 * i + 3] = __float_as_uint(f.w);
                }
            } else {
                tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c * 32), u);
                tmem_wait_ld();
                op_regs_after_wait(u);
            }
            const int li = lab_local - c * 32;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float g0 = __uint_as_float(u[2 * i]) * scale[c];
                float g1 = __uint_as_float(u[2 * i + 1]) * scale[c];
                if (2 * i == li)
                    g0 -= 1.f;
                if (2 * i + 1 == li)
                    g1 -= 1.f;
                pk[i] = pack_bf16(g0, g1);
            }
            // the warp's 32 x 32 chunk: row `lane`, piece j (8 columns) at
            // slot j ^ ((lane >> 1) & 3) (the TMA 64-byte swizzle); the TMA
            // store of the previous chunk must have read the buffer
            if (lane == 0)
                bulk_wait_group_read<0>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4 *>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && row0 < p.M) {
                tma_store_2d(tmO, stg_s, col, row0);
                bulk_commit_group();
            }
        }
    }
    if (lane == 0)
        bulk_wait_group_read<0>();
    __syncwarp();
}

// (m, s) <- the merge of two (max, sum of exp(z - max)) statistics; an empty
// one (max = -inf) leaves the other unchanged.
__device__ __forceinline__ void op_merge2(float &m, float &s, float m2, float s2)
{
    if (m2 == -CUDART_INF_F)
        return;
    const float nm = fmaxf(m, m2);
    s = s * ex2_approx((m - nm) * LOG2E) + s2 * ex2_approx((m2 - nm) * LOG2E);
    m = nm;
}

// Gradient of this warpgroup's half of the tile processed in order i, then
// an arrive on that tile's TMEM-empty barrier in the leader CTA -- or, for the
// stashed tile (`stash` set: its accumulator was released after the
// statistics), from the stash and without an arrive.
__device__ __forceinline__ void op_grad_release(const GemmParams &p, const CUtensorMap *tmO, const OpWork &w, int h,
                                                int i, const float (&cmi)[OP_HCH], float m, float ls, uint32_t tlane,
                                                int row0, int lab, uint8_t *stg, uint32_t stg_s, uint32_t tempty_bar,
                                                const float4 *stash)
{
    const int t = w.swap ? w.ntile - 1 - i : i;
    const int col0 = (w.nb0 + t) * p.op_tile + h * OP_HALF;
    const int lim = min(p.N, (w.nb0 + t) * p.op_tile + min(p.op_tile, (h + 1) * OP_HALF));
    float scale[OP_HCH];
#pragma unroll
    for (int c = 0; c < OP_HCH; ++c)
        scale[c] = ex2_approx(((cmi[c] - m) - ls) * LOG2E);
    if (col0 < lim)
        op_half_grad(p, tmO, lim, tlane + static_cast<uint32_t>(i * BN), row0, col0, lab, scale, stg, stg_s, stash);
    if (stash)
        return;
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive_cluster(mapa_shared(tempty_bar, 0u));
}

// Bounded wait until *flag >= target (acquire).
__device__ __noinline__ bool wait_flag64(const unsigned long long *flag, unsigned long long target,
                                         volatile int *abort_flag, const GemmParams &p, uint32_t peer_abort)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (ld_acquire_gpu_u64(flag) >= target)
            return true;
        __nanosleep(64);
        if ((it & 15u) == 15u) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                raise_error(p, abort_flag, ERR_OP_FLAG, peer_abort);
                return false;
            }
        }
    }
}

template <int LAYOUT>
__global__ void __launch_bounds__(OP_THREADS, 1)
    k_xent_onepass(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmO, const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + OP_STAGES * OP_A_BYTES;
    const uint32_t bar0 = base + OP_STAGES * OP_STAGE_BYTES;
    const uint32_t drain_bar = bar0 + 8u * (2 * OP_STAGES + 4);
    const uint32_t pub_bar = drain_bar + 8u;  // warpgroup 0 wrote the pair's merged partials
    const uint32_t xch_bar = pub_bar + 8u;    // warpgroup 1 handed over its half-tile statistics
    const uint32_t mrg_bar = xch_bar + 8u;    // both warpgroups stored their half of the row merge
    const uint32_t grp_bar = mrg_bar + 8u;    // the polling warp saw every group member's flag
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + OP_STAGES * OP_STAGE_BYTES + OP_NUM_BARS * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *xch_mx = reinterpret_cast<float *>(gbase + OP_STAGES * OP_STAGE_BYTES + OP_NUM_BARS * 8 + 16);
    float *xch_se = xch_mx + 2 * BM;  // [order i][row]
    float *mrg_mx = xch_se + 2 * BM;  // [warpgroup][row]
    float *mrg_se = mrg_mx + 2 * BM;
#define FULL_BAR(s) (bar0 + 8u * (s))
#define EMPTY_BAR(s) (bar0 + 8u * (OP_STAGES + (s)))
#define TFULL_BAR(t) (bar0 + 8u * (2 * OP_STAGES + (t)))
#define TEMPTY_BAR(t) (bar0 + 8u * (2 * OP_STAGES + 2 + (t)))

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < OP_STAGES; ++s) {
            mbar_init(FULL_BAR(s), 1);
            mbar_init(EMPTY_BAR(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(TFULL_BAR(t), 1);
            mbar_init(TEMPTY_BAR(t), 4 * OP_EPI_WARPS);  // both warpgroups of both CTAs
        }
        mbar_init(drain_bar, 1);
        mbar_init(pub_bar, OP_EPI_WARPS);
        mbar_init(xch_bar, OP_EPI_WARPS);
        mbar_init(mrg_bar, 2 * OP_EPI_WARPS);
        mbar_init(grp_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmO);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), OP_TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int *>(abort_flag)), rank ^ 1u);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed[OP_STAGES];
#pragma unroll
            for (int s = 0; s < OP_STAGES; ++s)
                armed[s] = 0;
            bool ok = true, first = true;
            // both CTAs' A (128 rows) and B (op_tile / 2 rows) boxes of a K slice
            const uint32_t stage_tx = 2u * (OP_A_BYTES + static_cast<uint32_t>(p.op_tile / 2) * BK * 2u);
            OpWork w;
            for (int r = 0; ok && r < p.op_rounds && op_work(p, pair, r, w); ++r) {
                const int arow = w.mb * OP_M + static_cast<int>(rank) * BM;
                for (int i = 0; ok && i < w.ntile; ++i) {
                    const int t = w.swap ? w.ntile - 1 - i : i;
                    const int brow = (w.nb0 + t) * p.op_tile + static_cast<int>(rank) * (p.op_tile / 2);
                    // a round's first tile is the previous round's last one: walk its K
                    // blocks downwards, so the first loads find the slices L2 still holds
                    const bool down = i == 0 && r > 0 && w.ntile == 2;
                    for (int kk = 0; kk < p.num_k_blocks; ++kk) {
                        const int kb = down ? p.num_k_blocks - 1 - kk : kk;
                        if (!wait_bar(EMPTY_BAR(stage), phase ^ 1u, abort_flag, p, ERR_PRODUCER, peer_abort)) {
                            ok = false;
                            break;
                        }
                        const uint32_t full_leader = mapa_shared(FULL_BAR(stage), 0u);
                        const bool skip = first && p.inject == 1 && blockIdx.x == 0;  // test hook
                        first = false;
                        if (!skip) {
                            if (leader) {
                                mbar_arrive_expect_tx(FULL_BAR(stage), stage_tx);
                                ++armed[stage];
                            }
                            const uint32_t a_dst = sA + stage * OP_A_BYTES, b_dst = sB + stage * OP_B_BYTES;
                            if (LAYOUT & 1) {
                                tma_load_2d_pair(a_dst, &tmA, arow, kb * BK, full_leader);
                                tma_load_2d_pair(a_dst + OP_MN_BOX, &tmA, arow + 64, kb * BK, full_leader);
                            } else {
                                tma_load_2d_pair(a_dst, &tmA, kb * BK, arow, full_leader);
                            }
                            if (LAYOUT & 2) {  // op_tile / 2 = 64 or 128 rows: one or two boxes
                                for (int bx = 0; bx < p.op_tile / 128; ++bx)
                                    tma_load_2d_pair(b_dst + bx * OP_MN_BOX, &tmB, brow + 64 * bx, kb * BK,
                                                     full_leader);
                            } else {
                                tma_load_2d_pair(b_dst, &tmB, kb * BK, brow, full_leader);
                            }
                        }
                        if (++stage == OP_STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (leader)
                for (int s = 0; s < OP_STAGES; ++s)
                    if (armed[s])
                        wait_bar_drain(FULL_BAR(s), (armed[s] - 1u) & 1u, abort_flag, p, peer_abort);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only)
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t tph[2] = {0u, 0u};
            const uint32_t idesc =
                idesc_bf16_f32_major(OP_M, static_cast<uint32_t>(p.op_tile), (LAYOUT & 1) != 0, (LAYOUT & 2) != 0);
            bool ok = true;
            OpWork w;
            for (int r = 0; ok && r < p.op_rounds && op_work(p, pair, r, w); ++r) {
                for (int i = 0; ok && i < w.ntile; ++i) {
                    // accumulator i holds the tile processed in order i
                    if (!wait_bar(TEMPTY_BAR(i), tph[i] ^ 1u, abort_flag, p, ERR_MMA_ACC, peer_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(i * BN);
                    // the stages arrive in the producer's K order (downwards for a
                    // round's first tile); the first one starts the accumulation
                    for (int kk = 0; kk < p.num_k_blocks; ++kk) {
                        if (!wait_bar(FULL_BAR(stage), phase, abort_flag, p, ERR_MMA_FULL, peer_abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = sA + stage * OP_A_BYTES;
                        const uint32_t b0 = sB + stage * OP_B_BYTES;
#pragma unroll
                        for (int k = 0; k < BK / OP_UMMA_K; ++k)
                            umma_f16_pair(d_tmem,
                                          (LAYOUT & 1) ? smem_desc_mn128(a0 + k * OP_MN_KSTEP, OP_MN_BOX)
                                                       : smem_desc_k128(a0 + k * OP_UMMA_K * 2),
                                          (LAYOUT & 2) ? smem_desc_mn128(b0 + k * OP_MN_KSTEP, OP_MN_BOX)
                                                       : smem_desc_k128(b0 + k * OP_UMMA_K * 2),
                                          idesc, (kk | k) != 0 ? 1u : 0u);
                        umma_commit_pair_mc(EMPTY_BAR(stage), 0x3);
                        if (++stage == OP_STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok)
                        break;
                    umma_commit_pair_mc(TFULL_BAR(i), 0x3);
                    tph[i] ^= 1u;
                }
            }
            umma_commit_pair_mc(drain_bar, 0x1);
            wait_bar_drain(drain_bar, 0u, abort_flag, p, peer_abort);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (both CTAs)
        // Both warpgroups work on every tile: warpgroup h (warps 2..5: h = 0,
        // warps 6..9: h = 1) takes columns [128h, 128h + 128) of each tile;
        // warp w reads TMEM lanes 32 * (w % 4) .., one row per thread.
        const int h = (warp - 2) >> 2;
        const int q = warp & 3;
        uint8_t *stg = gbase + OP_STG_OFF + (warp - 2) * OP_STG_WARP_BYTES;
        const uint32_t stg_s = base + static_cast<uint32_t>(OP_STG_OFF + (warp - 2) * OP_STG_WARP_BYTES);
        const int rloc = q * 32 + lane;
        uint32_t eph_bits = 0;  // TFULL phase of tile t in bit t
        uint32_t pub_phase = 0, xch_phase = 0, mrg_phase = 0, grp_phase = 0;
        const unsigned long long epoch_hi = static_cast<unsigned long long>(p.epoch) << 32;
        const uint32_t tlane =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * OP_HALF);
        // this thread's stash slots: the CTA's 128 x 256 fp32 region, float4
        // column j of half h at [(32 h + j) * BM + row]
        float4 *stash = reinterpret_cast<float4 *>(p.op_stash) + static_cast<size_t>(blockIdx.x) * (BM * BN / 4) +
                        static_cast<size_t>(h * 32) * BM + rloc;
        OpWork w;
        bool alive = true;
        for (int r = 0; alive && r < p.op_rounds && op_work(p, pair, r, w); ++r) {
            const int row0 = w.mb * OP_M + static_cast<int>(rank) * BM + q * 32;  // lane 0's row
            const int row = row0 + lane;
            const bool row_ok = row < p.M;
            const int qi = pair % p.op_Q;
            const int lab = row_ok ? p.labels[row] : -1;
            // 1. statistics of this half of each tile, in the order the MMAs
            //    finish them (order i = 0, 1; tile t_i); the half is left in
            //    TMEM as e = exp(z - running max) for the gradient
            float tm[2] = {-CUDART_INF_F, -CUDART_INF_F}, ts[2] = {0.f, 0.f};
            float cm[2][OP_HCH];
#pragma unroll 1
            for (int i = 0; i < w.ntile && alive; ++i) {
                const int t = w.swap ? w.ntile - 1 - i : i;
                const bool got = wait_bar(TFULL_BAR(i), (eph_bits >> i) & 1u, abort_flag, p, ERR_EPI, peer_abort);
                alive = __all_sync(0xffffffffu, got);
                if (alive) {
                    eph_bits ^= 1u << i;
                    tc_fence_after();
                    const int col0 = (w.nb0 + t) * p.op_tile + h * OP_HALF;
                    // this half's columns end at the tile's width or at N
                    const int lim = min(p.N, (w.nb0 + t) * p.op_tile + min(p.op_tile, (h + 1) * OP_HALF));
                    float zl = 0.f, cmt[OP_HCH], tmt = -CUDART_INF_F, tst = 0.f;
                    bool have = false;
                    // With two tiles, the first one's exp values go to the stash
                    // while the second tile's MMAs run, and accumulator 0 is
                    // released at once: the next round's first MMAs (into it)
                    // follow this round's last ones without waiting for the
                    // merge and the gradient.
                    const bool to_stash = i == 0 && w.ntile == 2;
                    float4 *st = to_stash ? stash : nullptr;
                    if (col0 + OP_HALF <= lim)
                        op_half_stats<true>(lim, tlane + static_cast<uint32_t>(i * BN), col0, lab, cmt, tmt, tst, zl,
                                            have, st);
                    else if (col0 < lim)
                        op_half_stats<false>(lim, tlane + static_cast<uint32_t>(i * BN), col0, lab, cmt, tmt, tst,
                                             zl, have, st);
                    if (to_stash) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive_cluster(mapa_shared(TEMPTY_BAR(0), 0u));
                    }
                    if (row_ok && have && lab < p.N)
                        p.label_logit[row] = zl;
                    // keep the results in registers named by the order index
#pragma unroll
                    for (int c = 0; c < OP_HCH; ++c) {
                        cm[0][c] = i == 0 ? cmt[c] : cm[0][c];
                        cm[1][c] = i == 0 ? cm[1][c] : cmt[c];
                    }
                    tm[0] = i == 0 ? tmt : tm[0];
                    tm[1] = i == 0 ? tm[1] : tmt;
                    ts[0] = i == 0 ? tst : ts[0];
                    ts[1] = i == 0 ? ts[1] : tst;
                }
            }
            if (!alive)
                break;
            // 2. warpgroup 1 hands its half statistics to warpgroup 0, which
            //    merges the pair's (tile, half) statistics per row, stores the
            //    partial in slot [qi][row] and publishes the CTA's flag: the
            //    mbarrier orders the lanes' stores before the one release
            //    store, which is cumulative at GPU scope (no separate fence)
            if (h == 1) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    xch_mx[i * BM + rloc] = tm[i];
                    xch_se[i * BM + rloc] = ts[i];
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(xch_bar);
            } else {
                const bool got = wait_bar(xch_bar, xch_phase, abort_flag, p, ERR_SK_SLOT, peer_abort);
                if (!__all_sync(0xffffffffu, got))
                    break;
                xch_phase ^= 1u;
                float mx = tm[0], se = ts[0];
                op_merge2(mx, se, tm[1], ts[1]);
                op_merge2(mx, se, xch_mx[rloc], xch_se[rloc]);
                op_merge2(mx, se, xch_mx[BM + rloc], xch_se[BM + rloc]);
                if (row_ok) {  // partial-major: slot [qi][row]
                    p.part_max[static_cast<size_t>(qi) * p.M + row] = mx;
                    p.part_sum[static_cast<size_t>(qi) * p.M + row] = se;
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(pub_bar);
                if (warp == 2 && lane == 0 &&
                    wait_bar(pub_bar, pub_phase, abort_flag, p, ERR_SK_SLOT, peer_abort)) {
                    st_release_gpu_u64(p.round_flags + pair * 2 + rank, epoch_hi | static_cast<unsigned>(r + 1));
                }
                pub_phase ^= 1u;
            }
            // 3. wait for the group's pairs (same CTA rank holds the same rows):
            //    one warp polls the flags (lanes in parallel, with backoff, so
            //    the flags' cache lines are not flooded while the other CTAs
            //    publish) and hands the result to the others through an
            //    mbarrier (acquire by the poller, then release/acquire at CTA
            //    scope: the partials it observed are visible to every warp)
            bool got = true;
            if (warp == 2) {
                const int first = (pair / p.op_Q) * p.op_Q;
                const unsigned long long target = epoch_hi | static_cast<unsigned>(r + 1);
                for (int j = lane; j < p.op_Q && got; j += 32)
                    got = wait_flag64(p.round_flags + (first + j) * 2 + rank, target, abort_flag, p, peer_abort);
                got = __all_sync(0xffffffffu, got);
                if (got && lane == 0)
                    mbar_arrive(grp_bar);
            }
            if (got)
                got = wait_bar(grp_bar, grp_phase, abort_flag, p, ERR_OP_FLAG, peer_abort);
            grp_phase ^= 1u;
            if (!__all_sync(0xffffffffu, got))
                break;
            __syncwarp();
            // 4. merge the row's op_Q pair partials: warpgroup h takes half of
            //    them, the two halves are exchanged through shared memory
            float m = -CUDART_INF_F, s = 0.f;
            {
                const int qh = (p.op_Q + 1) >> 1;
                const int j0 = h * qh;
                const int n = min(p.op_Q, j0 + qh) - j0;
                if (row_ok && n > 0)
                    merge_row_partials(p.part_max + static_cast<size_t>(j0) * p.M + row,
                                       p.part_sum + static_cast<size_t>(j0) * p.M + row, static_cast<size_t>(p.M), n,
                                       m, s);
                mrg_mx[h * BM + rloc] = m;
                mrg_se[h * BM + rloc] = s;
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(mrg_bar);
                const bool gm = wait_bar(mrg_bar, mrg_phase, abort_flag, p, ERR_SK_SLOT, peer_abort);
                if (!__all_sync(0xffffffffu, gm))
                    break;
                mrg_phase ^= 1u;
                op_merge2(m, s, mrg_mx[(1 - h) * BM + rloc], mrg_se[(1 - h) * BM + rloc]);
            }
            const float ls = logf(s);
            if (row_ok && h == 0 && qi == 0) {
                const int lb = p.labels[row];
                p.loss[row] = (lb >= 0 && lb < p.N) ? (m - __ldcg(p.label_logit + row)) + ls : CUDART_NAN_F;
            }
            // 5. gradient: first the tile still in TMEM (its accumulator is
            //    what the next round's second tile needs; released as soon as
            //    both warpgroups of both CTAs are done), then the stashed one
            if (w.ntile == 2) {
                op_grad_release(p, &tmO, w, h, 1, cm[1], m, ls, tlane, row0, lab, stg, stg_s, TEMPTY_BAR(1), nullptr);
                op_grad_release(p, &tmO, w, h, 0, cm[0], m, ls, tlane, row0, lab, stg, stg_s, 0u, stash);
            } else {
                op_grad_release(p, &tmO, w, h, 0, cm[0], m, ls, tlane, row0, lab, stg, stg_s, TEMPTY_BAR(0), nullptr);
            }
        }
    }
#undef FULL_BAR
#undef EMPTY_BAR
#undef TFULL_BAR
#undef TEMPTY_BAR

    if (*abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < OP_ABORT_SETTLE_NS) {
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, OP_TMEM_COLS);
    }
}

template <int LAYOUT>
cudaError_t set_onepass_smem_attr_once()
{
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load() & bit)
        return cudaSuccess;
    e = cudaFuncSetAttribute(k_xent_onepass<LAYOUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, OP_SMEM_BYTES);
    if (e == cudaSuccess)
        done.fetch_or(bit);
    return e;
}

template <int LAYOUT>
cudaError_t launch_onepass_t(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &to, const GemmParams &p,
                             int grid, cudaStream_t s)
{
    cudaError_t e = set_onepass_smem_attr_once<LAYOUT>();
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(OP_THREADS, 1, 1);
    cfg.dynamicSmemBytes = OP_SMEM_BYTES;
    cfg.stream = s;
    // Clusters of two CTAs (the tcgen05 pair), launched cooperatively: the
    // pairs of a group wait for each other's row statistics, so the whole grid
    // must be resident at once -- which a cooperative launch guarantees even
    // while other kernels hold SMs ("Allow reductions in matmul epilogues":
    // reusing the row reduction in the epilogue needs every CTA of a row of
    // tiles in the same wave, i.e. a cooperative launch).
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cooperative_launches() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k_xent_onepass<LAYOUT>, ta, tb, to, p);
}

}  // namespace

cudaError_t launch_xent_onepass(int layout, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &to,
                                const GemmParams &p, int grid, cudaStream_t s)
{
    switch (layout) {
    case 0:
        return launch_onepass_t<0>(ta, tb, to, p, grid, s);
    case 1:
        return launch_onepass_t<1>(ta, tb, to, p, grid, s);
    case 2:
        return launch_onepass_t<2>(ta, tb, to, p, grid, s);
    case 3:
        return launch_onepass_t<3>(ta, tb, to, p, grid, s);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace lf
