// gemm_nt_pair.cu -- the NT GEMM  acc = X[M,K] · W[N,K]^T  on a CTA pair
// (tcgen05 cta_group::2): one 256x256 output tile per pair of SMs.
//
// Source: "Strength reduction: fold transpose into a subsequent GEMM call"
// (lightning-thunder issue 1252), Feature/Motivation: the weight is read in
// its stored [N,K] layout as the K-major B operand -- no transpose op, no
// transposed copy.  "Allow reductions in matmul epilogues" (NVIDIA/Fuser issue
// 2213): the cross-entropy epilogues run on the finished accumulator.
//
// Other operand layouts ("fold any transpose"): X stored [K,M] and/or W
// stored [K,N] are read MN-major by the same MMAs -- the tensor core reads
// either major order from shared memory, so no operand is ever transposed in
// memory; only the TMA boxes and the shared-memory descriptors change.
//
// Why a pair: each CTA stages only its half of the tile's operands (128 rows
// of X and 128 rows of W per 64-wide K slice = 32 KiB), yet the pair's MMA
// computes a 256x256 product, so the bytes each SM must pull per FLOP drop by
// a third against a 128x256 single-CTA tile, and the same 192 KiB of shared
// memory holds a 6-deep ring instead of a 4-deep one (50% more load latency
// covered).
//
// Roles (320 threads per CTA for the plain store epilogues, 192 for the
// cross-entropy ones; cluster of 2 CTAs, rank 0 = leader):
//   warp 0 (both CTAs): TMA producer for this CTA's halves; both CTAs' copies
//            complete on the LEADER's full barrier (the leader arms it for the
//            bytes of both halves).
//   warp 1 (both CTAs): TMEM allocation (pair form); in the leader one lane
//            issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16) and commits
//            with a multicast arrive to both CTAs' barriers.
//   warps 2..9 or 2..5 (both CTAs): epilogue on this CTA's 128 accumulator
//            rows (warp w reads TMEM lanes 32 (w % 4) ..; with 8 warps each
//            takes half of a tile's columns); one lane per warp arrives on
//            the leader's accumulator-free barrier.  bf16 results (the plain
//            store and the cross-entropy gradient) are packed into 32 x 32
//            staging tiles and leave through TMA stores.  A stream-K owner's
//            idle epilogue warps sum its contributors' fp32 partials into the
//            second TMEM accumulator while its last MMAs run.
// Bounded waits everywhere; an abort raised in either CTA is mirrored into the
// peer, and both meet at a final cluster barrier before TMEM is freed.
#include <atomic>

#include <cuda_fp16.h>

#include "lf_gemm_common.cuh"

namespace lf {
namespace {

constexpr int PAIR_M = 2 * BM;          // 256 rows of X per pair tile
constexpr int PAIR_UMMA_K = 16;
// The operand ring: PAIR_STAGES slots of one K block each, grouped into
// stages of p.ksub consecutive slots (six stages of one K block, or three of
// two: one wait, eight MMAs and one commit per stage; the cross-entropy
// epilogues' whole-tile launches run 3-8 % faster so, the plain store and the
// stream-K split slower).
constexpr int PAIR_STAGES = 6;
constexpr int PAIR_A_BYTES = BM * BK * 2;          // 16 KiB: this CTA's 128 rows of X
constexpr int PAIR_B_BYTES = (BN / 2) * BK * 2;    // 16 KiB: this CTA's 128 rows of W
constexpr int PAIR_STAGE_BYTES = PAIR_A_BYTES + PAIR_B_BYTES;
constexpr int PAIR_ACC_BUFS = 2;
constexpr int PAIR_TMEM_COLS = PAIR_ACC_BUFS * BN;  // 512
constexpr int PAIR_SKC_CHUNKS = BN / 32;  // a contributor's partial arrives in 8 chunks of 32 columns
constexpr int PAIR_TQ = 16;               // ring of claimed tile indices (dynamic whole tiles)
constexpr int PAIR_NUM_BARS = 2 * PAIR_STAGES + 2 * PAIR_ACC_BUFS + 2 + PAIR_SKC_CHUNKS + PAIR_TQ;
// Per epilogue warp: two 2 KiB slots, each 32 rows x 32 bf16 columns of output
// (64-byte rows whose 16-byte pieces are XOR-swizzled by row pair -- the layout
// of a TMA 64-byte swizzle), so a TMA store can read one slot while the warp
// fills the other.  The transposed store of EPI_STORE_T uses the first 2560
// bytes as 32 rows of 80 bytes (read 16 bytes at a time without bank conflicts).
constexpr int PAIR_STG_ROW = 80;
constexpr int PAIR_STG_SLOT = 32 * 64;
constexpr int PAIR_STG_WARP_BYTES = 2 * PAIR_STG_SLOT;
static_assert(PAIR_STG_WARP_BYTES >= 32 * PAIR_STG_ROW, "transposed staging tile must fit");
// 1024-byte aligned: the swizzle pattern of a TMA store follows the address bits
// (after the barriers: 16 bytes of words -- TMEM address, abort flag -- and
// the PAIR_TQ tile-index slots)
constexpr int PAIR_STG_OFF = ((PAIR_STAGES * PAIR_STAGE_BYTES + PAIR_NUM_BARS * 8 + 16 + PAIR_TQ * 4 + 1023) / 1024) * 1024;
// Epilogue warps per CTA: the plain store epilogues use two per TMEM lane
// quarter (each takes half of the tile's columns, so the last tile's
// epilogue -- the tail of the launch -- and a stream-K partial take half as
// long); the cross-entropy epilogues reduce a whole row per thread and use one.
template <int EPI>
__host__ __device__ constexpr int pair_epi_warps()
{
    return (EPI == EPI_STORE || EPI == EPI_STORE_T) ? 8 : 4;
}
template <int EPI>
__host__ __device__ constexpr int pair_threads()
{
    return 64 + 32 * pair_epi_warps<EPI>();  // producer, MMA, epilogue warps
}
template <int EPI>
__host__ __device__ constexpr int pair_smem_bytes()
{
    return 1024 + PAIR_STG_OFF + pair_epi_warps<EPI>() * PAIR_STG_WARP_BYTES;
}
static_assert(pair_smem_bytes<EPI_STORE>() <= 232448, "shared memory per CTA");
// Operand layouts (LAYOUT bit 0: X stored [K,M], M-major; bit 1: W stored
// [K,N], N-major; bit 2: batched, 3-D tensor maps with the batch as their
// outermost coordinate).  An MN-major operand arrives as two 64 x 64 boxes per K
// slice (64 rows each, the second 8 KiB after the first) and is read through
// an MN-major descriptor; each K=16 step advances two 1024-byte atoms.
constexpr uint32_t PAIR_MN_HALF = PAIR_A_BYTES / 2;  // = PAIR_B_BYTES / 2
constexpr uint32_t PAIR_MN_KSTEP = 2 * 1024;
// An MN-major descriptor of the ring's last stage can reach up to 8 KiB past
// the ring: the barriers and the staging tiles that follow it (at least 16
// KiB) keep every such address inside the allocation.
static_assert(4 * PAIR_STG_WARP_BYTES >= 8192, "room past the ring for MN-major descriptors");
constexpr uint64_t ABORT_SETTLE_NS = 100000;  // after an abort: let copies in flight land

// A run of K blocks [kb0, kb1) of one output tile.
struct Seg {
    int tile, kb0, kb1;
};

// M block and (batch-major) N block of a tile index.  Whole tiles walk bands
// of p.band_m M blocks: within a band the M block varies fastest (the pairs
// that share a W tile run side by side, so W streams from HBM once per band)
// and the band's X rows stay in L2 while it sweeps every N block.  One band
// (band_m 0) is the plain M-block-fastest order; stream-K always uses it.
__device__ __forceinline__ void tile_coords(const GemmParams &p, int tile, int &mb, int &nbt)
{
    const int MB = p.num_m_blocks;
    const int bm = (p.band_m > 0 && p.band_m < MB && !p.streamk) ? p.band_m : MB;
    const int per_band = bm * (p.num_tiles / MB);
    const int band = tile / per_band;
    const int local = tile - band * per_band;
    const int rows = min(bm, MB - band * bm);
    mb = band * bm + local % rows;
    nbt = local / rows;
}

// The sequence of segments one pair works on.
// Whole tiles: tiles pair, pair + num_pairs, ... (M-block fastest), or with
// dyn_tiles tile pair and then the tiles the pair claims at run time:
// the leader's producer claims each further tile (num_pairs + the old value
// of the launch's tile counter) when it starts loading its current tile, and
// 2 K blocks before that tile's last load hands the claim to the pair's other
// roles -- its own MMA issuer and epilogue warps, the peer CTA's producer and
// epilogue warps -- through a ring of PAIR_TQ shared-memory slots in each
// CTA, each with an mbarrier (one arrival per entry).  The leader's own copy
// is a plain store and a local arrive; the peer's is an asynchronous store
// that completes as transaction bytes on the peer's barrier, with a relaxed
// arrive: a release at cluster scope there stalled the producer about 0.5 us
// per tile.  A claim past the last tile ends every role's sequence.  Claims
// follow the tile order, so the pairs that share a W tile start it together
// however far single pairs drift over a long launch, and faster pairs take
// more tiles.  A slot is overwritten 16 entries after it was filled, and by
// then every role has taken the entry: when the producer publishes entry
// j + 1 (during tile j) it has had the stage of entry j - 1 freed, so the MMA
// issuer (6 stages behind at most) has taken entry j - 7, the epilogue warps
// of both CTAs (two accumulator buffers behind it) entry j - 9 and the peer's
// producer (whose copies the MMA waited for) entry j - 7.
// Stream-K: the pairs form G = num_pairs / MB groups of MB pairs (MB = M
// blocks); pair m of group g works on M block m.  The V = N-tiles x K-blocks
// "column iterations" are split evenly over the groups -- group g takes
// [V*g/G, V*(g+1)/G), cut at N-tile boundaries -- so the MB pairs of a group
// walk the same K slices of the same W tile in lockstep and W is fetched from
// HBM once, while every pair gets an equal share.  Only a pair's first
// segment can start inside a tile and only its last can end inside one.
struct WorkIter {
    bool sk, dyn;
    int tile, step, ntiles, KB, MB, m;
    long long v, v_end;
    // dynamic whole tiles: this CTA's ring, whether this role claims and
    // publishes (the leader's producer), ring entries taken, the next claim
    uint32_t tq_slots = 0, tq_bars = 0;
    bool fetcher = false;
    int q = 0, claimed = 0;
    bool started = false;
    const GemmParams *pp = nullptr;
    volatile int *abort_flag = nullptr;
    uint32_t peer_abort = 0;
    __device__ WorkIter(const GemmParams &p, int pair, int num_pairs)
    {
        sk = p.streamk != 0;
        dyn = !sk && p.dyn_tiles != 0;
        KB = p.num_k_blocks;
        MB = p.num_m_blocks;
        ntiles = p.num_tiles;
        tile = pair;
        step = num_pairs;
        const int G = num_pairs / MB;
        const int g = pair / MB;
        m = pair % MB;
        const long long V = static_cast<long long>(p.num_n_blocks) * (p.batch > 1 ? p.batch : 1) * KB;
        v = V * g / G;
        v_end = V * (g + 1) / G;
    }
    // Dynamic whole tiles: the ring and this role's part in it.
    __device__ void attach(const GemmParams &p, uint32_t slots, uint32_t bars, bool claims, volatile int *abort,
                           uint32_t peer)
    {
        pp = &p;
        tq_slots = slots;
        tq_bars = bars;
        fetcher = claims;
        abort_flag = abort;
        peer_abort = peer;
    }
    // The fetcher, once per tile, at its first load: claim the pair's next
    // tile (the atomic's result is first used by publish()).
    __device__ void claim(unsigned *ctr)
    {
        claimed = step + static_cast<int>(atomicAdd(ctr, 1u));
    }
    // The fetcher, once per tile after claim(): hand the claimed tile to the
    // pair's other roles (ring entry q).
    __device__ void publish()
    {
        const uint32_t slot = tq_slots + 4u * static_cast<uint32_t>(q % PAIR_TQ);
        const uint32_t bar = tq_bars + 8u * static_cast<uint32_t>(q % PAIR_TQ);
        ++q;
        st_shared_u32(slot, static_cast<uint32_t>(claimed));
        mbar_arrive(bar);
        mbar_arrive_expect_tx_cluster_relaxed(mapa_shared(bar, 1u), 4u);
        st_async_u32(mapa_shared(slot, 1u), static_cast<uint32_t>(claimed), mapa_shared(bar, 1u));
        if (claimed >= ntiles)
            finish_claims();
    }
    // The fetcher, exactly once: this pair claims nothing more (see claims_done).
    bool claims_over = false;
    __device__ void finish_claims()
    {
        if (dyn && fetcher && !claims_over) {
            claims_over = true;
            claims_done(pp->tile_ctl, static_cast<unsigned>(step));
        }
    }
    __device__ bool next(Seg &s)
    {
        if (dyn) {
            int t = tile;  // the first tile: the pair's own index
            if (started) {
                if (fetcher) {
                    t = claimed;  // published during the previous tile
                } else {
                    const uint32_t slot = tq_slots + 4u * static_cast<uint32_t>(q % PAIR_TQ);
                    const uint32_t bar = tq_bars + 8u * static_cast<uint32_t>(q % PAIR_TQ);
                    const uint32_t parity = static_cast<uint32_t>(q / PAIR_TQ) & 1u;
                    ++q;
                    if (!wait_bar(bar, parity, abort_flag, *pp, ERR_TILE_QUEUE, peer_abort))
                        return false;
                    t = static_cast<int>(ld_shared_u32(slot));
                }
            }
            if (!started && fetcher && t >= ntiles)
                finish_claims();  // no tile at all (not planned: the grid has at most one pair per tile)
            started = true;
            if (t < 0 || t >= ntiles)  // past the last tile: the end (an index is never below 0)
                return false;
            s.tile = t;
            s.kb0 = 0;
            s.kb1 = KB;
            return true;
        }
        if (!sk) {
            if (tile >= ntiles)
                return false;
            s.tile = tile;
            s.kb0 = 0;
            s.kb1 = KB;
            tile += step;
            return true;
        }
        if (v >= v_end)
            return false;
        const int nb = static_cast<int>(v / KB);
        s.tile = m + nb * MB;
        s.kb0 = static_cast<int>(v % KB);
        const long long end = s.kb0 + (v_end - v);
        s.kb1 = end < KB ? static_cast<int>(end) : KB;
        v += s.kb1 - s.kb0;
        return true;
    }
};

// Stream-K, plain store epilogues: the sum of the contributors' partials for
// this thread's row (chunks of 32 columns [32 k0, 32 nch)), loaded from L2 and
// written into the idle accumulator buffer at `tpart` while this tile's own
// MMAs still run, so the epilogue adds it with a TMEM load.  Two chunks (16
// loads of 16 bytes) are in flight at a time.
__device__ __forceinline__ void preload_partials(const PartialAdd &pa, uint32_t tpart, int k0, int nch)
{
#pragma unroll 1
    for (int c = k0; c < nch; c += 2) {
        const bool two = c + 1 < nch;  // warp-uniform
        float v0[32], v1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v0[i] = 0.f;
            v1[i] = 0.f;
        }
#pragma unroll 1
        for (int e = 0; e < pa.count; ++e) {  // in pair order, as the fix-up adds them
            const float4 *s4 = reinterpret_cast<const float4 *>(pa.slot + static_cast<size_t>(e) * pa.stride);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 f = __ldcg(s4 + (c * 8 + i) * BM + pa.row);
                const float4 g = two ? __ldcg(s4 + ((c + 1) * 8 + i) * BM + pa.row) : make_float4(0.f, 0.f, 0.f, 0.f);
                v0[4 * i + 0] += f.x;
                v0[4 * i + 1] += f.y;
                v0[4 * i + 2] += f.z;
                v0[4 * i + 3] += f.w;
                v1[4 * i + 0] += g.x;
                v1[4 * i + 1] += g.y;
                v1[4 * i + 2] += g.z;
                v1[4 * i + 3] += g.w;
            }
        }
        uint32_t u0[32], u1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            u0[i] = __float_as_uint(v0[i]);
            u1[i] = __float_as_uint(v1[i]);
        }
        tmem_st_32x32b_x32(tpart + static_cast<uint32_t>(c * 32), u0);
        if (two)
            tmem_st_32x32b_x32(tpart + static_cast<uint32_t>((c + 1) * 32), u1);
    }
    tmem_wait_st();
}

// Stream-K: number of groups after this pair's group that hold the rest of
// `tile` (their shares start before the tile's N-tile ends).  Contributor e is
// pair (g + 1 + e) * MB + m.
__device__ __forceinline__ int sk_contributors(const GemmParams &p, int pair, int num_pairs, int tile)
{
    const int MB = p.num_m_blocks;
    const int G = num_pairs / MB;
    const long long V = static_cast<long long>(p.num_n_blocks) * (p.batch > 1 ? p.batch : 1) * p.num_k_blocks;
    const long long tile_end = static_cast<long long>(tile / MB + 1) * p.num_k_blocks;
    int n = 0;
    for (int g = pair / MB + 1; g < G && V * g / G < tile_end; ++g)
        ++n;
    return n;
}

// out = bf16_rn(acc + partials) for the warp's 32 rows of the tile (thread
// `lane` owns row row0 + lane; `out` is this batch's matrix, rows p.ldo
// elements apart).  When contributor 0's slot is being copied
// into shared memory (pa.smem0 set), chunk c first waits for its own copy
// (barrier skc0 + 8 * c/32).  Each 32-column chunk is staged in the warp's
// 2 KiB of shared memory (16-byte pieces XOR-swizzled by row pair, so writes
// and reads are conflict-free) and stored 8 rows x 64 bytes per instruction
// instead of 32 rows x 16 bytes.  Returns false if a copy wait gave up.
__device__ __forceinline__ bool pair_store(const GemmParams &p, __nv_bfloat16 *out, uint32_t taddr, int row0, int nb,
                                           int c0, int c1, const PartialAdd &pa, uint32_t skc0, uint8_t *stg,
                                           volatile int *abort_flag, uint32_t peer_abort)
{
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int c = c0; c < c1; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        if (pa.smem0) {
            const bool got = wait_bar(skc0 + 8u * static_cast<uint32_t>(c / 32), 0u, abort_flag, p, ERR_SK_COPY,
                                      peer_abort);
            if (!__all_sync(0xffffffffu, got))
                return false;
        }
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4 *>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                make_uint4(pack_bf16(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                           pack_bf16(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                           pack_bf16(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                           pack_bf16(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 8 * i + (lane >> 2);  // row of the warp's 32
            const int pc = lane & 3;            // 8-column piece
            const uint4 val = *reinterpret_cast<const uint4 *>(stg + r * 64 + ((pc ^ ((r >> 1) & 3)) << 4));
            const int grow = row0 + r;
            const int gcol = col + pc * 8;  // N % 8 == 0: a piece is all in or all out
            if (grow < p.M && gcol < p.N)
                *reinterpret_cast<uint4 *>(out + static_cast<size_t>(grow) * p.ldo + gcol) = val;
        }
        __syncwarp();
    }
    return true;
}

// TMA-store path of the epilogues: chunk k of the warp (this thread's row of
// 32 columns packed as 16 bf16 pairs) goes to staging slot k & 1 (64-byte
// rows, 16-byte pieces XOR-swizzled by row pair: the output map's 64-byte
// swizzle) and lane 0 stores the 32 x 32 box at (col, row0[, bz]); the TMA
// unit leaves out the box's rows >= M and columns >= N.  A slot is refilled
// only after the store issued from it two chunks earlier has read it.
template <bool BATCHED>
__device__ __forceinline__ void tma_store_chunk(const GemmParams &p, const CUtensorMap *tmO, uint8_t *stg,
                                                uint32_t stg_s, int k, const uint32_t (&pk)[16], int col, int row0,
                                                int bz)
{
    const int lane = threadIdx.x & 31;
    const int slot = k & 1;
    if (k >= 2) {
        if (lane == 0)
            bulk_wait_group_read<1>();
        __syncwarp();
    }
    uint8_t *buf = stg + slot * PAIR_STG_SLOT;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4 *>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    fence_proxy_async_smem();  // the generic-proxy writes before the TMA unit reads them
    __syncwarp();
    if (lane == 0 && row0 < p.M) {
        const uint32_t src = stg_s + static_cast<uint32_t>(slot * PAIR_STG_SLOT);
        if (BATCHED)
            tma_store_3d(tmO, src, col, row0, bz);
        else
            tma_store_2d(tmO, src, col, row0);
        bulk_commit_group();
    }
}

// Plain-store path (when the output map could not be encoded): the warp's 32
// x 32 chunk (this thread's row as 16 packed pairs) is staged in shared memory
// and written 8 rows x 64 bytes per instruction, rows >= M and columns >= N
// left out.
__device__ __forceinline__ void plain_store_chunk(const GemmParams &p, __nv_bfloat16 *out, uint8_t *stg,
                                                  const uint32_t (&pk)[16], int col, int row0)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4 *>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 8 * i + (lane >> 2);
        const int pc = lane & 3;
        const uint4 val = *reinterpret_cast<const uint4 *>(stg + r * 64 + ((pc ^ ((r >> 1) & 3)) << 4));
        const int grow = row0 + r;
        const int gcol = col + pc * 8;
        if (grow < p.M && gcol < p.N)
            *reinterpret_cast<uint4 *>(out + static_cast<size_t>(grow) * p.N + gcol) = val;
    }
    __syncwarp();
}

// After a tile's last chunk: every store has read its staging slot.
__device__ __forceinline__ void tma_store_drain()
{
    if ((threadIdx.x & 31) == 0)
        bulk_wait_group_read<0>();
    __syncwarp();
}

// As pair_store, with the chunks written by TMA stores (tma_store_chunk).
template <bool BATCHED>
__device__ __forceinline__ bool pair_store_tma(const GemmParams &p, const CUtensorMap *tmO, uint32_t taddr, int row0,
                                               int nb, int bz, int c0, int c1, const PartialAdd &pa, uint32_t skc0,
                                               uint8_t *stg, uint32_t stg_s, volatile int *abort_flag,
                                               uint32_t peer_abort)
{
    bool ok = true;
#pragma unroll 1
    for (int c = c0; c < c1; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        if (pa.smem0) {
            const bool got = wait_bar(skc0 + 8u * static_cast<uint32_t>(c / 32), 0u, abort_flag, p, ERR_SK_COPY,
                                      peer_abort);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
        }
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        tma_store_chunk<BATCHED>(p, tmO, stg, stg_s, (c - c0) / 32, pk, col, row0, bz);
    }
    tma_store_drain();
    return ok;
}

// Swapped operands (skinny X): the accumulator holds acc[n][m] = sum_k W[n,k]
// X[m,k] -- this thread's row is output column n = row0 + lane, its TMEM
// columns are output rows m.  Each 32 x 32 chunk is written transposed into
// the warp's staging tile (S[m][n], 80-byte rows) with 2-byte stores, then
// thread t stores output row m = col + t: 32 consecutive n, 64 bytes.
__device__ __forceinline__ bool pair_store_t(const GemmParams &p, __nv_bfloat16 *out, uint32_t taddr, int row0,
                                             int nb, int tn, int c0, int c1, const PartialAdd &pa, uint32_t skc0,
                                             uint8_t *stg, volatile int *abort_flag, uint32_t peer_abort)
{
    const int lane = threadIdx.x & 31;
    const int M_out = p.N;  // the caller's M (kernel columns)
    const int N_out = p.M;  // the caller's N (kernel rows)
#pragma unroll 1
    for (int c = c0; c < c1; c += 32) {
        const int col = nb * tn + c;
        if (col >= M_out)
            break;  // warp-uniform
        if (pa.smem0) {
            const bool got = wait_bar(skc0 + 8u * static_cast<uint32_t>(c / 32), 0u, abort_flag, p, ERR_SK_COPY,
                                      peer_abort);
            if (!__all_sync(0xffffffffu, got))
                return false;
        }
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        __nv_bfloat16 *srow = reinterpret_cast<__nv_bfloat16 *>(stg);
#pragma unroll
        for (int i = 0; i < 32; ++i)  // S[m = i][n = lane]
            srow[i * (PAIR_STG_ROW / 2) + lane] = __float2bfloat16_rn(__uint_as_float(v[i]));
        __syncwarp();
        const int m = col + lane;
        if (m < M_out) {
            const uint4 *src = reinterpret_cast<const uint4 *>(stg + lane * PAIR_STG_ROW);
            __nv_bfloat16 *dst = out + static_cast<size_t>(m) * p.ldo + row0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (row0 + 8 * j < N_out)  // N % 8 == 0: 8 columns are all in or all out
                    *reinterpret_cast<uint4 *>(dst + 8 * j) = src[j];
        }
        __syncwarp();
    }
    return true;
}

// Gradient pass of the two-pass cross-entropy ("Allow reductions in matmul
// epilogues", the softmax-minus-onehot output) for the warp's 32 rows:
// grad = bf16_rn(exp(z - row_max - row_logsum) - [n == label]) with the
// exponent as one FFMA (z * log2 e - (max + logsum) * log2 e) and ex2.approx,
// staged and stored like pair_store.  Row statistics come from the combine
// kernel; this thread owns row row0 + lane.
__device__ __forceinline__ void pair_xent_grad(const GemmParams &p, const CUtensorMap *tmO, uint32_t taddr, int row0,
                                               int nb, const PartialAdd &pa, uint8_t *stg, uint32_t stg_s)
{
    const int lane = threadIdx.x & 31;
    const int row = row0 + lane;
    const bool row_ok = row < p.M;
    const int lab = row_ok ? p.labels[row] : -1;
    const float off = row_ok ? (p.row_max[row] + p.row_logsum[row]) * LOG2E : 0.f;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        const int li = lab - col;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float g0 = ex2_approx(fmaf(__uint_as_float(v[2 * i]), LOG2E, -off));
            float g1 = ex2_approx(fmaf(__uint_as_float(v[2 * i + 1]), LOG2E, -off));
            if (2 * i == li)
                g0 -= 1.f;
            if (2 * i + 1 == li)
                g1 -= 1.f;
            pk[i] = pack_bf16(g0, g1);
        }
        if (p.tma_store)
            tma_store_chunk<false>(p, tmO, stg, stg_s, c / 32, pk, col, row0, 0);
        else
            plain_store_chunk(p, out, stg, pk, col, row0);
    }
    if (p.tma_store)
        tma_store_drain();
}

// First pass of the cross-entropy gradient without a recompute GEMM ("Allow
// reductions in matmul epilogues", fusion example: row max, exp, sum-exp and
// the label logit of the tile, and the exponentials the softmax-minus-onehot
// output is made of), for the warp's 32 rows (thread `lane` owns row row0 +
// lane): over the tile's columns n < N,
//   m_t = max_n z,  s_t = sum_n exp(z - m_t),  z[label] if the label is here,
// written to part_max / part_sum [row, nb] and label_logit[row], and
//   e = fp16_rn(exp(z - m_t))  (in [0, 1]; exactly 1 at the tile's max)
// written into the gradient buffer, which the rescale kernel later rewrites in
// place as bf16_rn(e * exp(m_t - lse)) once the row's lse is known.  Two
// passes over TMEM: the max, then the exponentials (one FFMA + ex2.approx each,
// the sum as a tree) packed two per word and stored like the gradient.
__device__ __forceinline__ void pair_xent_exp(const GemmParams &p, const CUtensorMap *tmO, uint32_t taddr, int row0,
                                              int nb, const PartialAdd &pa, uint8_t *stg, uint32_t stg_s)
{
    const int lane = threadIdx.x & 31;
    const int row = row0 + lane;
    const bool row_ok = row < p.M;
    const int lab = row_ok ? p.labels[row] : -1;
    float mx = -CUDART_INF_F, zl = 0.f;
    bool have = false;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        const int nvalid = p.N - col;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nvalid)
                mx = fmaxf(mx, __uint_as_float(v[i]));
        const int li = lab - col;
        if (static_cast<unsigned>(li) < 32u) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i == li)
                    zl = __uint_as_float(v[i]);
            have = true;
        }
    }
    const float mxl = mx * LOG2E;
    float se = 0.f;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int col = nb * BN + c;
        if (col >= p.N)
            break;  // warp-uniform
        uint32_t v[32];
        load_chunk(taddr, c, pa, v);
        const int nvalid = p.N - col;
        float e[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            e[i] = i < nvalid ? ex2_approx(fmaf(__uint_as_float(v[i]), LOG2E, -mxl)) : 0.f;
        float t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            t[i] = e[i] + e[i + 16];
#pragma unroll
        for (int w = 8; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i)
                t[i] += t[i + w];
        se += t[0];
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            __half2 h = __floats2half2_rn(e[2 * i], e[2 * i + 1]);  // .x (lower address) = column 2i
            pk[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        if (p.tma_store)
            tma_store_chunk<false>(p, tmO, stg, stg_s, c / 32, pk, col, row0, 0);
        else
            plain_store_chunk(p, out, stg, pk, col, row0);
    }
    if (p.tma_store)
        tma_store_drain();
    if (row_ok) {
        const size_t o = static_cast<size_t>(row) * p.num_n_blocks + nb;
        p.part_max[o] = mx;
        p.part_sum[o] = se;
        if (have && lab < p.N)
            p.label_logit[row] = zl;
    }
}

template <int EPI, int LAYOUT, int KSUB = 1>
__global__ void __launch_bounds__(pair_threads<EPI>(), 1)
    k_gemm_nt_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmO, const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + PAIR_STAGES * PAIR_A_BYTES;
    const uint32_t bar0 = base + PAIR_STAGES * PAIR_STAGE_BYTES;
    const uint32_t drain_bar = bar0 + 8u * (2 * PAIR_STAGES + 2 * PAIR_ACC_BUFS);
    const uint32_t skw_bar = drain_bar + 8u;  // the epilogue warps finished writing a partial
    const uint32_t skc_bar = skw_bar + 8u;    // chunk c of a contributor's partial landed: skc_bar + 8c
    const uint32_t tq_bar = skc_bar + 8u * PAIR_SKC_CHUNKS;  // ring entry in slot i published: tq_bar + 8i
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + PAIR_STAGES * PAIR_STAGE_BYTES + PAIR_NUM_BARS * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t tq_slots = smem_u32(tmem_slot + 4);  // PAIR_TQ claimed tile indices
#define FULL_BAR(s) (bar0 + 8u * (s))
#define EMPTY_BAR(s) (bar0 + 8u * (PAIR_STAGES + (s)))
#define TFULL_BAR(b) (bar0 + 8u * (2 * PAIR_STAGES + (b)))
#define TEMPTY_BAR(b) (bar0 + 8u * (2 * PAIR_STAGES + PAIR_ACC_BUFS + (b)))

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    // the MMA's N: BN, or for the swapped-operand store the caller's M rounded up to 16
    const int tn = (EPI == EPI_STORE_T && p.tile_n > 0) ? p.tile_n : BN;
    // bytes both CTAs' copies of one K slice bring: A 128 rows, B tn / 2 rows each
    const uint32_t stage_tx = 2u * (PAIR_A_BYTES + static_cast<uint32_t>(tn / 2) * BK * 2u);  // per K block
    constexpr int ksub = KSUB;  // K blocks per ring stage
    constexpr int nstages = PAIR_STAGES / KSUB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PAIR_STAGES; ++s) {
            mbar_init(FULL_BAR(s), 1);   // leader: its arrive.expect_tx + both CTAs' bytes
            mbar_init(EMPTY_BAR(s), 1);  // the leader's multicast commit
        }
        for (int b = 0; b < PAIR_ACC_BUFS; ++b) {
            mbar_init(TFULL_BAR(b), 1);                    // the leader's multicast commit
            mbar_init(TEMPTY_BAR(b), 2 * pair_epi_warps<EPI>());  // leader: one arrive per epilogue warp of each CTA
        }
        mbar_init(drain_bar, 1);
        mbar_init(skw_bar, pair_epi_warps<EPI>());
        for (int c = 0; c < PAIR_SKC_CHUNKS; ++c)
            mbar_init(skc_bar + 8u * c, 1);
        for (int i = 0; i < PAIR_TQ; ++i) {
            mbar_init(tq_bar + 8u * i, 1);       // one arrival per entry (the leader's producer)
            st_shared_u32(tq_slots + 4u * i, 0x7fffffffu);  // an unwritten slot reads as the end
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if ((EPI == EPI_STORE || EPI == EPI_XENT_GRAD || EPI == EPI_XENT_EXP) && p.tma_store)
            prefetch_tmap(&tmO);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), PAIR_TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int *>(abort_flag)), rank ^ 1u);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed[PAIR_STAGES];
#pragma unroll
            for (int s = 0; s < PAIR_STAGES; ++s)
                armed[s] = 0;
            bool ok = true, first = true;
            WorkIter it(p, pair, num_pairs);
            it.attach(p, tq_slots, tq_bar, leader, abort_flag, peer_abort);
            for (Seg g; ok && it.next(g);) {
                const int claim_kb = g.kb0, publish_kb = max(g.kb0, g.kb1 - 2);
                int mb, nbt;  // M block, batch-major N block
                tile_coords(p, g.tile, mb, nbt);
                const int bz = nbt / p.num_n_blocks;       // batch (0 unless batched)
                const int nb = nbt % p.num_n_blocks;
                const int xz = p.x_batched ? bz : 0;
                const int wz = p.w_batched ? bz : 0;
                const int arow = mb * PAIR_M + static_cast<int>(rank) * BM;
                const int brow = nb * tn + static_cast<int>(rank) * (tn / 2);
                for (int kbs = g.kb0; kbs < g.kb1; kbs += ksub) {
                    const int nsub = KSUB == 1 ? 1 : min(KSUB, g.kb1 - kbs);  // K blocks in this stage
                    if (it.dyn && leader) {
                        if (kbs == claim_kb)
                            it.claim(p.tile_ctl);
                        if (publish_kb >= kbs && publish_kb < kbs + nsub)
                            it.publish();
                    }
                    if (!wait_bar(EMPTY_BAR(stage), phase ^ 1u, abort_flag, p, ERR_PRODUCER, peer_abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_leader = mapa_shared(FULL_BAR(stage), 0u);
                    // test hook: pair 0's leader never arms its first stage, so
                    // that stage can never complete and the MMA wait runs out
                    const bool skip = first && p.inject == 1 && blockIdx.x == 0;
                    first = false;
                    if (!skip) {
                        if (leader) {
                            mbar_arrive_expect_tx(FULL_BAR(stage), stage_tx * static_cast<uint32_t>(nsub));
                            ++armed[stage];
                        }
#pragma unroll
                        for (int j = 0; j < KSUB; ++j) {
                        if (j >= nsub)
                            break;
                        const int kb = kbs + j;
                        const uint32_t slot = static_cast<uint32_t>(stage * ksub + j);
                        const uint32_t a_dst = sA + slot * PAIR_A_BYTES, b_dst = sB + slot * PAIR_B_BYTES;
                        if (LAYOUT & 4) {  // batched: the batch is the maps' third coordinate
                            if (LAYOUT & 1) {
                                tma_load_3d_pair(a_dst, &tmA, arow, kb * BK, xz, full_leader);
                                tma_load_3d_pair(a_dst + PAIR_MN_HALF, &tmA, arow + 64, kb * BK, xz, full_leader);
                            } else {
                                tma_load_3d_pair(a_dst, &tmA, kb * BK, arow, xz, full_leader);
                            }
                            if (LAYOUT & 2) {
                                tma_load_3d_pair(b_dst, &tmB, brow, kb * BK, wz, full_leader);
                                tma_load_3d_pair(b_dst + PAIR_MN_HALF, &tmB, brow + 64, kb * BK, wz, full_leader);
                            } else {
                                tma_load_3d_pair(b_dst, &tmB, kb * BK, brow, wz, full_leader);
                            }
                        } else {
                            if ((LAYOUT & 1) && (p.mn3 & 1)) {  // both 64-row halves in one copy
                                tma_load_3d_pair(a_dst, &tmA, 0, kb * BK, arow / 64, full_leader);
                            } else if (LAYOUT & 1) {
                                tma_load_2d_pair(a_dst, &tmA, arow, kb * BK, full_leader);
                                tma_load_2d_pair(a_dst + PAIR_MN_HALF, &tmA, arow + 64, kb * BK, full_leader);
                            } else {
                                tma_load_2d_pair(a_dst, &tmA, kb * BK, arow, full_leader);
                            }
                            if ((LAYOUT & 2) && (p.mn3 & 2)) {
                                tma_load_3d_pair(b_dst, &tmB, 0, kb * BK, brow / 64, full_leader);
                            } else if (LAYOUT & 2) {
                                tma_load_2d_pair(b_dst, &tmB, brow, kb * BK, full_leader);
                                tma_load_2d_pair(b_dst + PAIR_MN_HALF, &tmB, brow + 64, kb * BK, full_leader);
                            } else {
                                tma_load_2d_pair(b_dst, &tmB, kb * BK, brow, full_leader);
                            }
                        }
                        }  // the stage's K blocks
                    }
                    if (++stage == nstages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            it.finish_claims();  // if the loop ended early (an abort); once only
            if (leader)
                for (int s = 0; s < nstages; ++s)
                    if (armed[s])
                        wait_bar_drain(FULL_BAR(s), (armed[s] - 1u) & 1u, abort_flag, p, peer_abort);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only)
        if (leader && lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            WorkIter it(p, pair, num_pairs);
            it.attach(p, tq_slots, tq_bar, false, abort_flag, peer_abort);
            for (Seg g; ok && it.next(g);) {
                if (!wait_bar(TEMPTY_BAR(acc), acc_phase ^ 1u, abort_flag, p, ERR_MMA_ACC, peer_abort))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kbs = g.kb0; kbs < g.kb1; kbs += ksub) {
                    const int nsub = KSUB == 1 ? 1 : min(KSUB, g.kb1 - kbs);
                    if (!wait_bar(FULL_BAR(stage), phase, abort_flag, p, ERR_MMA_FULL, peer_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t idesc =
                        idesc_bf16_f32_major(PAIR_M, static_cast<uint32_t>(tn), (LAYOUT & 1) != 0, (LAYOUT & 2) != 0);
#pragma unroll
                    for (int j = 0; j < KSUB; ++j) {
                        if (j >= nsub)
                            break;
                        const uint32_t slot = static_cast<uint32_t>(stage * ksub + j);
                        const uint32_t a0 = sA + slot * PAIR_A_BYTES;
                        const uint32_t b0 = sB + slot * PAIR_B_BYTES;
#pragma unroll
                        for (int k = 0; k < BK / PAIR_UMMA_K; ++k) {
                            const uint64_t da = (LAYOUT & 1) ? smem_desc_mn128(a0 + k * PAIR_MN_KSTEP, PAIR_MN_HALF)
                                                             : smem_desc_k128(a0 + k * PAIR_UMMA_K * 2);
                            const uint64_t db = (LAYOUT & 2) ? smem_desc_mn128(b0 + k * PAIR_MN_KSTEP, PAIR_MN_HALF)
                                                             : smem_desc_k128(b0 + k * PAIR_UMMA_K * 2);
                            umma_f16_pair(d_tmem, da, db, idesc, (kbs != g.kb0 || j != 0 || k != 0) ? 1u : 0u);
                        }
                    }
                    umma_commit_pair_mc(EMPTY_BAR(stage), 0x3);  // both CTAs may refill this stage
                    if (++stage == nstages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit_pair_mc(TFULL_BAR(acc), 0x3);  // accumulator complete in both TMEMs
                if (++acc == PAIR_ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            umma_commit_pair_mc(drain_bar, 0x1);
            wait_bar_drain(drain_bar, 0u, abort_flag, p, peer_abort);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (both CTAs)
        // warp w reads TMEM lanes 32 * (w % 4) .., one row per thread; with 8
        // epilogue warps, warps 2..5 take the first half of the tile's 32-column
        // chunks and warps 6..9 the second half
        const int q = warp & 3;
        constexpr int kParts = pair_epi_warps<EPI>() / 4;
        const int cpart = (warp - 2) >> 2;
        const int tile_chunks = (tn + 31) / 32;
        const int part_chunks = (tile_chunks + kParts - 1) / kParts;
        const int c0 = cpart * part_chunks * 32;
        const int c1 = min(tile_chunks, (cpart + 1) * part_chunks) * 32;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t skw_phase = 0;
        WorkIter it(p, pair, num_pairs);
        it.attach(p, tq_slots, tq_bar, false, abort_flag, peer_abort);
        for (Seg g; it.next(g);) {
            int mb, nbt;  // M block, batch-major N block
            tile_coords(p, g.tile, mb, nbt);
            const int nb = nbt % p.num_n_blocks;
            const int bz = nbt / p.num_n_blocks;
            const int rloc = q * 32 + lane;
            const int row = mb * PAIR_M + static_cast<int>(rank) * BM + rloc;
            const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(q * 32) << 16);
            PartialAdd pa = {nullptr, 0, 0, rloc, nullptr, 0, 0u};
            const bool owner_split = g.kb0 == 0 && g.kb1 < p.num_k_blocks;
            const int MB = p.num_m_blocks;
            const int first = (pair / MB + 1) * MB + pair % MB;  // first contributor pair
            if (owner_split) {
                // The tile's first K blocks, the rest held by the next pairs:
                // acquire their flags while this pair's MMAs still run.
                const int n = sk_contributors(p, pair, num_pairs, g.tile);
                bool got = true;
                if (lane == 0)
                    for (int e = 0; e < n && got; ++e)
                        got = wait_flag(p.sk_flags + (first + e * MB) * 2 + rank, p.epoch, abort_flag, p,
                                        peer_abort);
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (!got)
                    break;
                pa.slot = p.sk_partials + static_cast<size_t>(first * 2 + rank) * SK_SLOT_FLOATS;
                pa.stride = static_cast<size_t>(MB) * 2 * SK_SLOT_FLOATS;
                pa.count = n;
                if ((EPI == EPI_STORE || EPI == EPI_STORE_T) && n > 0) {
                    // This is the pair's last segment, so the other
                    // accumulator buffer is idle: sum the partials into it
                    // while this tile's MMAs still run.
                    const uint32_t tpart = tmem_base + static_cast<uint32_t>((acc ^ 1) * BN) +
                                           (static_cast<uint32_t>(q * 32) << 16);
                    preload_partials(pa, tpart, c0 / 32, min(c1 / 32, (p.N - nb * tn + 31) / 32));
                    pa.in_tmem = 1;
                    pa.tpart = tpart;
                    pa.count = 0;
                }
            }
            const bool ok = wait_bar(TFULL_BAR(acc), acc_phase, abort_flag, p, ERR_EPI, peer_abort);
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc_fence_after();
            if (g.kb0 != 0) {
                // Not the tile's first K blocks: hand the partial sum to the
                // pair that owns the tile's start.
                epi_write_partial(taddr, p.sk_partials + static_cast<size_t>(pair * 2 + rank) * SK_SLOT_FLOATS, rloc, c0,
                                  c1);
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(skw_bar);
                if (warp == 2 && lane == 0 &&
                    wait_bar(skw_bar, skw_phase, abort_flag, p, ERR_SK_SLOT, peer_abort)) {
                    __threadfence();
                    st_release_gpu(p.sk_flags + pair * 2 + rank, p.epoch);
                }
                skw_phase ^= 1u;
            } else {
                // chunks of 32 columns that lie inside the matrix: only those
                // are copied, and each copy is waited for by the warps that
                // read it (none is left in flight at exit)
                const int nch = min((tn + 31) / 32, (p.N - nb * tn + 31) / 32);
                if (owner_split && pa.count > 0) {
                    // This is the pair's last segment, so its MMAs are done and
                    // the operand ring is idle: pull the first contributor's
                    // 128 KiB slot into it as 8 bulk copies of 32 columns, each
                    // on its own barrier, so the epilogue starts on the first
                    // chunk while the rest are in flight.
                    if (warp == 2 && lane == 0) {
#pragma unroll 1
                        for (int c = 0; c < nch; ++c) {
                            constexpr int CH = SK_SLOT_FLOATS / PAIR_SKC_CHUNKS;  // floats per chunk
                            mbar_arrive_expect_tx(skc_bar + 8u * c, CH * 4);
                            bulk_load_g2s(sA + static_cast<uint32_t>(c * CH * 4), pa.slot + static_cast<size_t>(c) * CH,
                                          CH * 4, skc_bar + 8u * c);
                        }
                    }
                    pa.smem0 = reinterpret_cast<const float4 *>(gbase);
                }
                bool done = true;
                if (EPI == EPI_STORE && p.tma_store)
                    done = pair_store_tma<(LAYOUT & 4) != 0>(
                        p, &tmO, taddr, row - lane, nb, bz, c0, c1, pa, skc_bar,
                        gbase + PAIR_STG_OFF + (warp - 2) * PAIR_STG_WARP_BYTES,
                        base + static_cast<uint32_t>(PAIR_STG_OFF + (warp - 2) * PAIR_STG_WARP_BYTES), abort_flag,
                        peer_abort);
                else if (EPI == EPI_STORE)
                    done = pair_store(p, static_cast<__nv_bfloat16 *>(p.out) + static_cast<size_t>(bz) * p.stride_o, taddr,
                                      row - lane, nb, c0, c1, pa, skc_bar,
                                      gbase + PAIR_STG_OFF + (warp - 2) * PAIR_STG_WARP_BYTES, abort_flag, peer_abort);
                else if (EPI == EPI_STORE_T)
                    done = pair_store_t(p, static_cast<__nv_bfloat16 *>(p.out), taddr, row - lane, nb, tn, c0, c1, pa, skc_bar,
                                        gbase + PAIR_STG_OFF + (warp - 2) * PAIR_STG_WARP_BYTES, abort_flag,
                                        peer_abort);
                else {
                    if (pa.smem0) {
                        for (int c = 0; c < nch && done; ++c)
                            done = wait_bar(skc_bar + 8u * c, 0u, abort_flag, p, ERR_SK_COPY, peer_abort);
                        done = __all_sync(0xffffffffu, done);
                    }
                    if (done) {
                        if (EPI == EPI_XENT_PARTIAL)
                            epi_xent_partial(p, taddr, row, nb, pa);
                        else if (EPI == EPI_XENT_ROW)
                            epi_xent_row(p, taddr, row, pa);
                        else if (EPI == EPI_XENT_EXP)
                            pair_xent_exp(p, &tmO, taddr, row - lane, nb, pa,
                                          gbase + PAIR_STG_OFF + (warp - 2) * PAIR_STG_WARP_BYTES,
                                          base + static_cast<uint32_t>(PAIR_STG_OFF + (warp - 2) * PAIR_STG_WARP_BYTES));
                        else
                            pair_xent_grad(p, &tmO, taddr, row - lane, nb, pa,
                                           gbase + PAIR_STG_OFF + (warp - 2) * PAIR_STG_WARP_BYTES,
                                           base + static_cast<uint32_t>(PAIR_STG_OFF + (warp - 2) * PAIR_STG_WARP_BYTES));
                    }
                }
                if (!done)
                    break;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(mapa_shared(TEMPTY_BAR(acc), 0u));
            if (++acc == PAIR_ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }
#undef FULL_BAR
#undef EMPTY_BAR
#undef TFULL_BAR
#undef TEMPTY_BAR

    if (*abort_flag) {
        // Copies this CTA issued complete on the leader's barrier, so nothing
        // here can wait for them: give them a fixed, generous time to land.
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < ABORT_SETTLE_NS) {
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer no longer touches this CTA's barriers, smem or TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, PAIR_TMEM_COLS);
    }
}

// Launch configuration: clusters of two CTAs (the tcgen05 pair).  A stream-K
// launch is also cooperative: a tile's owner waits for its contributors'
// partials, so every CTA of the grid must be resident at once, which a
// cooperative launch guarantees even while other kernels hold SMs (without it
// an owner could spin while its contributor waits for an SM the owner's
// neighbours hold).  Whole-tile launches have no cross-CTA waits.
template <int EPI>
cudaLaunchConfig_t pair_config(int grid, cudaStream_t s, cudaLaunchAttribute *attr, bool cooperative)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(pair_threads<EPI>(), 1, 1);
    cfg.dynamicSmemBytes = pair_smem_bytes<EPI>();
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cooperative ? 2 : 1;
    return cfg;
}

// The dynamic shared-memory opt-in is a per-device function attribute: set it
// once per device and kernel instead of on every launch.
template <int EPI, int LAYOUT, int KSUB>
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
    e = cudaFuncSetAttribute(k_gemm_nt_pair<EPI, LAYOUT, KSUB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair_smem_bytes<EPI>());
    if (e == cudaSuccess)
        done.fetch_or(bit);
    return e;
}

template <int EPI, int LAYOUT, int KSUB = 1>
cudaError_t launch_pair_k(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &to, const GemmParams &p,
                          int grid, cudaStream_t s)
{
    cudaError_t e = set_smem_attr_once<EPI, LAYOUT, KSUB>();
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config<EPI>(grid, s, attr, p.streamk != 0 && cooperative_launches());
    return cudaLaunchKernelEx(&cfg, k_gemm_nt_pair<EPI, LAYOUT, KSUB>, ta, tb, to, p);
}

// The cross-entropy partial and exp epilogues have a two-K-block-stage form
// (p.ksub == 2, whole tiles); every other launch uses one-K-block stages.
template <int EPI, int LAYOUT>
cudaError_t launch_pair_t(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &to, const GemmParams &p,
                          int grid, cudaStream_t s)
{
    if constexpr (EPI == EPI_XENT_PARTIAL || EPI == EPI_XENT_EXP)
        if (p.ksub == 2)
            return launch_pair_k<EPI, LAYOUT, 2>(ta, tb, to, p, grid, s);
    return launch_pair_k<EPI, LAYOUT, 1>(ta, tb, to, p, grid, s);
}

}  // namespace

int gemm_pair_smem_bytes() { return pair_smem_bytes<EPI_STORE>(); }

// Number of CTA pairs of the pair kernel that fit on the device at once.
int gemm_pair_max_active_clusters()
{
    if (cudaFuncSetAttribute(k_gemm_nt_pair<EPI_STORE, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair_smem_bytes<EPI_STORE>()) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config<EPI_STORE>(2, 0, attr, false);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_gemm_nt_pair<EPI_STORE, 0>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_gemm_nt_pair(int epi, int layout, const CUtensorMap &ta, const CUtensorMap &tb,
                                const CUtensorMap &to, const GemmParams &p, int grid, cudaStream_t s)
{
    if (layout != 0 && epi == EPI_XENT_PARTIAL) {  // the cross-entropy epilogues: layouts 1..3
        switch (layout) {
        case 1:
            return launch_pair_t<EPI_XENT_PARTIAL, 1>(ta, tb, to, p, grid, s);
        case 2:
            return launch_pair_t<EPI_XENT_PARTIAL, 2>(ta, tb, to, p, grid, s);
        case 3:
            return launch_pair_t<EPI_XENT_PARTIAL, 3>(ta, tb, to, p, grid, s);
        default:
            return cudaErrorInvalidValue;
        }
    }
    if (epi == EPI_XENT_ROW) {
        switch (layout) {
        case 0:
            return launch_pair_t<EPI_XENT_ROW, 0>(ta, tb, to, p, grid, s);
        case 1:
            return launch_pair_t<EPI_XENT_ROW, 1>(ta, tb, to, p, grid, s);
        case 2:
            return launch_pair_t<EPI_XENT_ROW, 2>(ta, tb, to, p, grid, s);
        case 3:
            return launch_pair_t<EPI_XENT_ROW, 3>(ta, tb, to, p, grid, s);
        default:
            return cudaErrorInvalidValue;
        }
    }
    if (epi == EPI_XENT_EXP) {
        switch (layout) {
        case 0:
            return launch_pair_t<EPI_XENT_EXP, 0>(ta, tb, to, p, grid, s);
        case 1:
            return launch_pair_t<EPI_XENT_EXP, 1>(ta, tb, to, p, grid, s);
        case 2:
            return launch_pair_t<EPI_XENT_EXP, 2>(ta, tb, to, p, grid, s);
        case 3:
            return launch_pair_t<EPI_XENT_EXP, 3>(ta, tb, to, p, grid, s);
        default:
            return cudaErrorInvalidValue;
        }
    }
    if (layout != 0 && epi == EPI_XENT_GRAD) {
        switch (layout) {
        case 1:
            return launch_pair_t<EPI_XENT_GRAD, 1>(ta, tb, to, p, grid, s);
        case 2:
            return launch_pair_t<EPI_XENT_GRAD, 2>(ta, tb, to, p, grid, s);
        case 3:
            return launch_pair_t<EPI_XENT_GRAD, 3>(ta, tb, to, p, grid, s);
        default:
            return cudaErrorInvalidValue;
        }
    }
    if (layout != 0) {  // other operand layouts, plain store epilogue (batched: bit 2)
        if (epi != EPI_STORE)
            return cudaErrorInvalidValue;
        switch (layout) {
        case 1:
            return launch_pair_t<EPI_STORE, 1>(ta, tb, to, p, grid, s);
        case 2:
            return launch_pair_t<EPI_STORE, 2>(ta, tb, to, p, grid, s);
        case 3:
            return launch_pair_t<EPI_STORE, 3>(ta, tb, to, p, grid, s);
        case 4:
            return launch_pair_t<EPI_STORE, 4>(ta, tb, to, p, grid, s);
        case 5:
            return launch_pair_t<EPI_STORE, 5>(ta, tb, to, p, grid, s);
        case 6:
            return launch_pair_t<EPI_STORE, 6>(ta, tb, to, p, grid, s);
        case 7:
            return launch_pair_t<EPI_STORE, 7>(ta, tb, to, p, grid, s);
        default:
            return cudaErrorInvalidValue;
        }
    }
    switch (epi) {
    case EPI_STORE:
        return launch_pair_t<EPI_STORE, 0>(ta, tb, to, p, grid, s);
    case EPI_STORE_T:
        return launch_pair_t<EPI_STORE_T, 0>(ta, tb, to, p, grid, s);
    case EPI_XENT_PARTIAL:
        return launch_pair_t<EPI_XENT_PARTIAL, 0>(ta, tb, to, p, grid, s);
    case EPI_XENT_GRAD:
        return launch_pair_t<EPI_XENT_GRAD, 0>(ta, tb, to, p, grid, s);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace lf
