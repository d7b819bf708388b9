// api.cu -- the C ABI of liblayoutfold.so: argument validation, tensor-map
// encoding, per-device state (error word, cross-entropy workspace) and the
// launch sequences.  Declarations and the contract of each call are in
// include/layoutfold.h.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "layoutfold.h"
#include "lf_internal.h"

namespace {

constexpr int MAX_DEVICES = 64;
constexpr int64_t MAX_DIM = (int64_t(1) << 31) - 1;

struct DeviceState {
    bool probed = false;
    bool arch_ok = false;
    int num_sms = 0;
    int pair_clusters = 0;    // co-resident CTA pairs of the pair kernel
    void *sk_ws = nullptr;    // stream-K partial slots + flags (fixed size, zeroed once)
    void *op_flags = nullptr; // one-pass cross-entropy: round flags (2 per pair, zeroed once), then
                              // the per-CTA stash of a tile's exp values (128 x 256 fp32 per CTA)
    unsigned sk_epoch = 0;    // last epoch handed to a launch whose CTAs wait on flags
    int *err_word = nullptr;  // device int[64]; [0] = first error code
    unsigned *tile_ctl = nullptr;  // claimed whole tiles: counter and count (GemmParams::tile_ctl), zeroed once
    void *ws = nullptr;       // cross-entropy workspace (grow-only)
    size_t ws_bytes = 0;
    // Ordering of the calls that use the workspaces above (WorkspaceOrder).
    std::mutex order_mutex;
    cudaEvent_t ws_event = nullptr;    // recorded after the last such call's launches
    cudaStream_t ws_stream = nullptr;  // the stream it was recorded on
    bool ws_recorded = false;
    // Cooperative launches of CTA-pair clusters (stream-K, one-pass
    // cross-entropy): 0 = not refused so far, -1 = the runtime refused one, so
    // schedules whose CTAs wait on each other are no longer chosen.
    std::atomic<int> coop{0};
};

std::mutex g_mutex;
DeviceState g_dev[MAX_DEVICES];
std::atomic<uint64_t> g_launches{0};
// the schedule of the last tensor-core GEMM launch:
// grid | (0 single CTA, 1 CTA pairs) << 20 | stream-K << 23 | N-tile width << 24
std::atomic<uint64_t> g_last_plan{0};
// the code of the last device-side wait that gave up, as lf_check_device_error read it
std::atomic<int> g_last_wait_code{0};
std::atomic<int> g_inject{0};
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_l2_prefetch{-1};  // -1: per-shape default
// K blocks of MMA time a stream-K split costs beyond its share of the work
constexpr double SK_FIXED_KBLOCKS = 32.0;
std::atomic<int> g_variant{-1};      // -1 auto, 1 single-CTA, 2 CTA-pair whole tiles, 3 CTA-pair stream-K,
                                     // 4 swapped operands (skinny M)
std::atomic<int> g_op_tile{0};       // one-pass cross-entropy N-tile width; 0 = automatic
std::atomic<int> g_xent_path{0};     // cross-entropy gradient: 0 auto, 1 one pass, 2 exp + rescale, 3 recompute
std::atomic<int> g_band{-1};         // whole-tile band height in M blocks: -1 auto, 0 one band, > 0 forced
// Whole tiles on pairs: -1 automatic (the fixed assignment), 0 fixed, 1 claimed
// at run time.  Claiming won while the cross-entropy launches ran one-K-block
// ring stages (8192 x 128256 x 4096 loss: 4.42 ms claimed, 4.59-4.92 ms fixed,
// whose pairs drifted apart and re-read W: 6.8-12.6 GB against 2.2 GB); with
// their two-K-block stages the fixed assignment keeps its pairs together (2.20
// GB, 4.16 ms against 4.19 ms claimed), and for the plain store at the same
// size claiming is slower (4.47 vs 4.33 ms).  Claimed tiles remain an option:
// they balance the load by themselves when other work holds some SMs.
std::atomic<int> g_tile_sched{-1};
std::atomic<int> g_coop_enable{1};   // 0: launch the CTA-waiting kernels without the cooperative attribute
// L2 bytes of X a band of whole tiles may keep while it sweeps W (the L2 is
// 129 MB, but reuse measured as if about half of it were available)
constexpr double BAND_X_BYTES = 32.0 * 1024 * 1024;
// the rescale kernel keeps one scale per 256-column tile of a row in shared memory
constexpr int64_t RESCALE_MAX_TILES = 48 * 1024;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Resolve (and on first use, set up) the current device.
lf_status current_device(DeviceState **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return LF_ERR_ARCH;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &d = g_dev[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return LF_ERR_LAUNCH;
        }
        d.arch_ok = (major == 10 && minor == 3);
        d.num_sms = sms;
        if (d.arch_ok) {
            d.pair_clusters = lf::gemm_pair_max_active_clusters();
            if (cudaMalloc(&d.err_word, 64 * sizeof(int)) != cudaSuccess ||
                cudaMemset(d.err_word, 0, 64 * sizeof(int)) != cudaSuccess ||
                cudaMalloc(&d.tile_ctl, 64 * sizeof(unsigned)) != cudaSuccess ||
                cudaMemset(d.tile_ctl, 0, 64 * sizeof(unsigned)) != cudaSuccess ||
                cudaEventCreateWithFlags(&d.ws_event, cudaEventDisableTiming) != cudaSuccess ||
                cudaDeviceSynchronize() != cudaSuccess) {
                cudaGetLastError();
                return LF_ERR_LAUNCH;
            }
        }
        d.probed = true;
    }
    if (!d.arch_ok)
        return LF_ERR_ARCH;
    *out = &d;
    return LF_OK;
}

// Grow-only workspace of the current device.  Growing frees the old block
// (cudaFree waits for the device, so no kernel still uses it).
lf_status ensure_workspace(DeviceState *d, size_t bytes, void **ws)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    if (d->ws_bytes < bytes) {
        if (d->ws) {
            cudaFree(d->ws);
            d->ws = nullptr;
            d->ws_bytes = 0;
        }
        if (cudaMalloc(&d->ws, bytes) != cudaSuccess) {
            cudaGetLastError();
            d->ws = nullptr;
            return LF_ERR_WORKSPACE;
        }
        d->ws_bytes = bytes;
    }
    *ws = d->ws;
    return LF_OK;
}

// Stream-K partial slots (2 per pair) and their flags, allocated on first use.
lf_status ensure_sk_workspace(DeviceState *d)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    if (d->sk_ws)
        return LF_OK;
    const size_t slots = static_cast<size_t>(2 * d->pair_clusters) * lf::SK_SLOT_FLOATS * sizeof(float);
    const size_t bytes = slots + static_cast<size_t>(2 * d->pair_clusters) * sizeof(unsigned);
    if (cudaMalloc(&d->sk_ws, bytes) != cudaSuccess || cudaMemset(d->sk_ws, 0, bytes) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        if (d->sk_ws)
            cudaFree(d->sk_ws);
        d->sk_ws = nullptr;
        return LF_ERR_WORKSPACE;
    }
    return LF_OK;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

unsigned next_epoch(DeviceState *d)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    unsigned e = ++d->sk_epoch;
    if (e == 0)
        e = ++d->sk_epoch;
    return e;
}

// True while `s` is being captured into a CUDA graph.  Such a call plans no
// schedule whose CTAs wait on each other's flags (stream-K, the one-pass
// cross-entropy): their flags carry a per-launch epoch, which every replay of
// the graph would repeat, so a replay could take the flags of the previous
// one for its own.  The flag-free forms (whole tiles, the exp pass and the
// rescale) replay correctly.
bool capturing(cudaStream_t s)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cs != cudaStreamCaptureStatusNone;
}

// One-pass cross-entropy workspace, allocated on first use: the round flags
// (zeroed once; every launch's flags carry a new epoch) and the stash.
size_t onepass_flag_bytes(const DeviceState *d)
{
    return round_up(static_cast<size_t>(2 * d->pair_clusters) * sizeof(unsigned long long), 256);
}

lf_status ensure_onepass_flags(DeviceState *d)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    if (d->op_flags)
        return LF_OK;
    const size_t bytes = onepass_flag_bytes(d) + static_cast<size_t>(2 * d->pair_clusters) * lf::BM * lf::BN * 4;
    if (cudaMalloc(&d->op_flags, bytes) != cudaSuccess ||
        cudaMemset(d->op_flags, 0, onepass_flag_bytes(d)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        if (d->op_flags)
            cudaFree(d->op_flags);
        d->op_flags = nullptr;
        return LF_ERR_WORKSPACE;
    }
    return LF_OK;
}

// Orders the calls that use a device's library-owned workspaces (the
// cross-entropy partials, the stream-K slots and flags, the one-pass flags and
// stash, the claimed-tile counter).  A call on a different stream than the
// previous such call first makes its stream wait for that call's launches (an
// event: no host synchronisation), and the lock, held from before the
// launch's epoch is drawn until its launches are enqueued and recorded, keeps
// host threads from interleaving -- so such launches run one after another on
// the GPU, in the order of their epochs, whatever streams and threads they
// come from.  A stream that is being captured into a graph is neither made to
// wait nor recorded (graph replays are ordered by the caller).
class WorkspaceOrder {
public:
    WorkspaceOrder(DeviceState *d, cudaStream_t s) : d_(d), s_(s), lock_(d->order_mutex)
    {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
            cudaGetLastError();
            cs = cudaStreamCaptureStatusNone;
        }
        capturing_ = cs != cudaStreamCaptureStatusNone;
        if (!capturing_ && d->ws_recorded && d->ws_stream != s && cudaStreamWaitEvent(s, d->ws_event, 0) != cudaSuccess) {
            cudaGetLastError();
            ok_ = false;
        }
    }
    WorkspaceOrder(const WorkspaceOrder &) = delete;
    WorkspaceOrder &operator=(const WorkspaceOrder &) = delete;
    bool ok() const { return ok_; }
    ~WorkspaceOrder()
    {
        if (capturing_ || !ok_)
            return;
        if (cudaEventRecord(d_->ws_event, s_) == cudaSuccess) {
            d_->ws_recorded = true;
            d_->ws_stream = s_;
        } else {
            cudaGetLastError();
        }
    }

private:
    DeviceState *d_;
    cudaStream_t s_;
    std::lock_guard<std::mutex> lock_;
    bool capturing_ = false;
    bool ok_ = true;
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// 2-D bf16 tensor [rows, K] (K contiguous), box = 64 columns x box_rows rows,
// 128-byte swizzle; out-of-range rows/columns read as zero.
bool make_tmap(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, uint32_t box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(lf::BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor stored [K, rows] (rows contiguous: an MN-major operand),
// box = 64 rows x 64 K, 128-byte swizzle; out-of-range elements read as zero.
// The same [K, rows] operand viewed as (64 rows, K, rows / 64): one box of
// (64, BK, 2) brings two consecutive 64-row halves, in the order two boxes of
// make_tmap_mn would (each half's 64 K rows of 128 bytes, then the next half).
// Needs rows to be a multiple of 64.
bool make_tmap_mn3(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows % 64 != 0)
        return false;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(rows) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(lf::BK), 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_mn(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(rows) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(lf::BK)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor: `batch` matrices `stride` elements apart, each `outer`
// rows of `inner` contiguous elements with a row pitch of `ld` elements; box
// = 64 inner x box_outer rows x 1 batch, 128-byte swizzle, zero fill.
bool make_tmap3(CUtensorMap *m, const void *ptr, int64_t inner, int64_t outer, int64_t ld, int64_t batch,
                int64_t stride, uint32_t box_outer)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer),
                                static_cast<cuuint64_t>(batch)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(stride) * 2};
    const cuuint32_t box[3] = {64, box_outer, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The output of the pair kernel's store epilogue as a bf16 tensor map: N
// columns x M rows with a row pitch of ld elements (3-D: `batch` such matrices
// `stride` elements apart, batch outermost); 32 x 32 boxes with the 64-byte
// swizzle the epilogue's staging tiles use.  Returns false if the driver
// rejects the layout (the kernel then stores without TMA).
bool make_tmap_out(CUtensorMap *m, void *ptr, int64_t M, int64_t N, int64_t ld, int64_t batch, int64_t stride,
                   bool three_d)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M),
                                static_cast<cuuint64_t>(batch)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(stride) * 2};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, three_d ? 3 : 2, ptr, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A batch of strided views (gemm_batched): row pitches and batch strides in
// elements; sw == 0 means one W for every batch.
struct BatchSpec {
    int64_t batch, ldx, sx, ldw, sw, ldo, so;
};

// Everything one GEMM launch needs: variant, tensor maps, parameters, grid.
struct GemmPlan {
    bool pair = false;
    int layout = 0;  // bit 0: X stored [K,M]; bit 1: W stored [K,N] (pair kernel only)
    DeviceState *dev = nullptr;
    CUtensorMap ta, tb;
    // MN-major operands of the pair kernel: the 3-D views (make_tmap_mn3), valid
    // for the operands whose bit is set in p.mn3; the pair kernel reads both
    // 64-row halves of a CTA's rows with one copy through them (W stored [K,N],
    // 4096^3: 89.7 -> 87.7 us; both operands MN-major 97.9 -> 91.8 us)
    CUtensorMap ta3, tb3;
    CUtensorMap to;  // output map of the pair kernel's TMA-store epilogue (set by run_gemm)
    lf::GemmParams p;
    int grid = 0;
    bool no_flags = false;  // the call is being captured into a graph (see capturing)
};

lf_status plan_gemm(DeviceState *d, const void *x, const void *w, int64_t M, int64_t N, int64_t K,
                    GemmPlan *g, int layout = 0, const BatchSpec *bs = nullptr, int tile_n = 0)
{
    // the swapped path (tile_n > 0) always runs on the pair kernel; it keeps an
    // explicit whole-tile (2) or stream-K (3) choice, else decides automatically
    const int gv = g_variant.load();
    const int variant = tile_n ? ((gv == 2 || gv == 3) ? gv : -1) : gv;
    g->dev = d;
    if (bs)
        layout |= 4;
    g->layout = layout;
    // The MN-major operand paths exist in the pair kernel only.  Skinny
    // problems (M <= 128) go to the pair kernel too when single-CTA tiles would
    // leave most SMs idle and K is long enough for the stream-K split: at
    // 64 x 5120 x 13824 that measured 53 us against 94 us for 20 single-CTA tiles.
    const int64_t tiles1 = ((M + lf::BM - 1) / lf::BM) * ((N + lf::BN - 1) / lf::BN);
    const bool skinny_split = tiles1 * 4 <= d->num_sms && (K + lf::BK - 1) / lf::BK >= 128;
    g->pair = d->pair_clusters > 0 &&
              (tile_n > 0 || layout != 0 || variant >= 2 || (variant < 0 && (M > lf::BM || skinny_split)));
    if (layout != 0 && !g->pair)
        return LF_ERR_LAUNCH;
    const int tile_m = g->pair ? 2 * lf::BM : lf::BM;
    bool ok_a, ok_b;
    int mn3 = 0;  // which operands also have the pair kernel's 3-D MN-major view
    if (bs) {
        // an operand with batch stride 0 (or a batch of 1) is one matrix: a map
        // whose batch extent is 1, read at batch coordinate 0
        const bool xb = bs->sx != 0 && bs->batch > 1, wbat = bs->sw != 0 && bs->batch > 1;
        const int64_t sx = xb ? bs->sx : ((layout & 1) ? K * bs->ldx : M * bs->ldx);
        const int64_t wb = wbat ? bs->batch : 1;
        const int64_t sw = wbat ? bs->sw : ((layout & 2) ? K * bs->ldw : N * bs->ldw);
        ok_a = (layout & 1) ? make_tmap3(&g->ta, x, M, K, bs->ldx, xb ? bs->batch : 1, sx, 64)
                            : make_tmap3(&g->ta, x, K, M, bs->ldx, xb ? bs->batch : 1, sx, lf::BM);
        ok_b = (layout & 2) ? make_tmap3(&g->tb, w, N, K, bs->ldw, wb, sw, 64)
                            : make_tmap3(&g->tb, w, K, N, bs->ldw, wb, sw, lf::BN / 2);
    } else {
        mn3 = (g->pair && (layout & 1) && make_tmap_mn3(&g->ta3, x, M, K) ? 1 : 0) |
              (g->pair && (layout & 2) && make_tmap_mn3(&g->tb3, w, N, K) ? 2 : 0);
        ok_a = (layout & 1) ? make_tmap_mn(&g->ta, x, M, K) : make_tmap(&g->ta, x, M, K, lf::BM);
        const uint32_t b_rows = tile_n ? static_cast<uint32_t>(tile_n / 2) : (g->pair ? lf::BN / 2 : lf::BN);
        ok_b = (layout & 2) ? make_tmap_mn(&g->tb, w, N, K) : make_tmap(&g->tb, w, N, K, b_rows);
    }
    if (!ok_a || !ok_b)
        return LF_ERR_LAUNCH;
    lf::GemmParams &p = g->p;
    std::memset(&p, 0, sizeof p);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_m_blocks = static_cast<int>((M + tile_m - 1) / tile_m);
    p.tile_n = tile_n;
    p.num_n_blocks = static_cast<int>((N + (tile_n ? tile_n : lf::BN) - 1) / (tile_n ? tile_n : lf::BN));
    p.num_k_blocks = static_cast<int>((K + lf::BK - 1) / lf::BK);
    const int64_t batch = bs ? bs->batch : 1;
    p.batch = static_cast<int>(batch);
    p.x_batched = bs && bs->sx && batch > 1 ? 1 : 0;
    p.w_batched = bs && bs->sw && batch > 1 ? 1 : 0;
    p.ldo = bs ? bs->ldo : N;
    p.stride_o = bs ? bs->so : 0;
    if (static_cast<int64_t>(p.num_m_blocks) * p.num_n_blocks * batch > MAX_DIM)
        return LF_ERR_SHAPE;
    p.num_tiles = static_cast<int>(p.num_m_blocks * p.num_n_blocks * batch);
    p.err = d->err_word;
    p.mn3 = mn3;
    p.timeout_ns = g_timeout_ns.load();
    p.inject = g_inject.load();
    const int pf = g_l2_prefetch.load();
    p.l2_prefetch = pf >= 0 ? pf : 0;
    if (g->pair) {
        // Whole tiles leave pairs idle when the last wave is short; then the K
        // iterations can be split evenly over all pairs instead (stream-K).
        // Stream-K groups: G groups of MB pairs (one per M block), G <= V so
        // that no pair gets an empty share -- a tile's owner waits on every
        // later group's partial, so each must write one.
        const int P = d->pair_clusters;
        const long long waves = (p.num_tiles + P - 1) / P;
        const long long V = static_cast<long long>(p.num_n_blocks) * batch * p.num_k_blocks;
        long long G = p.num_m_blocks <= P ? P / p.num_m_blocks : 0;
        if (G > V)
            G = V;
        // The split pays when it shortens each pair's run -- waves x KB K
        // blocks by whole tiles, V / G when split -- by more than its fixed
        // cost (partials written, acquired and added; owners that finish after
        // single-segment pairs), about 32 K blocks of MMA time on a GB300:
        // 768 x 5120 x 13824 (216 -> 172.8 K blocks) 71.9 -> 68.9 us, while at
        // K = 4096 (64 -> 51-61) whole tiles measured 30.4-30.9 us against
        // 33.0-37.9 us split.
        const double whole_kb = static_cast<double>(waves) * p.num_k_blocks;
        const double split_kb = G > 0 ? static_cast<double>(V) / static_cast<double>(G) : whole_kb;
        p.streamk = (G > 0 && d->coop.load() >= 0 && !g->no_flags &&
                     (variant == 3 || (variant < 0 && whole_kb - split_kb > SK_FIXED_KBLOCKS)))
                        ? 1
                        : 0;
        if (p.streamk) {
            lf_status st = ensure_sk_workspace(d);
            if (st != LF_OK)
                return st;
            p.sk_partials = static_cast<float *>(d->sk_ws);
            p.sk_flags = reinterpret_cast<unsigned *>(static_cast<char *>(d->sk_ws) + static_cast<size_t>(2 * P) *
                                                                                         lf::SK_SLOT_FLOATS *
                                                                                         sizeof(float));
            g->grid = 2 * static_cast<int>(G * p.num_m_blocks);
        } else {
            g->grid = 2 * (p.num_tiles < P ? p.num_tiles : P);
        }
    } else
        g->grid = p.num_tiles < d->num_sms ? p.num_tiles : d->num_sms;
    if (g->pair && !p.streamk) {
        // Whole tiles: bands of M blocks whose X rows stay in L2 while the band
        // sweeps every N block (W then streams from HBM once per band instead
        // of X once per wave), split evenly.
        const int MB = p.num_m_blocks;
        int band = g_band.load();
        if (band < 0) {
            const double x_bytes = static_cast<double>(tile_m) * static_cast<double>(K) * 2.0;
            band = static_cast<int>(BAND_X_BYTES / x_bytes);
            if (band < 1)
                band = 1;
            if (band >= MB) {
                band = 0;
            } else {
                const int nbands = (MB + band - 1) / band;
                band = (MB + nbands - 1) / nbands;
            }
        }
        p.band_m = band < MB ? band : 0;
        p.dyn_tiles = g_tile_sched.load() == 1 ? 1 : 0;  // claimed tiles on request
    }
    return LF_OK;
}

cudaError_t run_gemm(int epi, GemmPlan &g, cudaStream_t stream)
{
    g_last_plan.store(static_cast<uint64_t>(g.grid) | (static_cast<uint64_t>(g.pair ? 1 : 0) << 20) |
                      (static_cast<uint64_t>(g.p.streamk ? 1 : 0) << 23) |
                      (static_cast<uint64_t>(g.p.tile_n ? g.p.tile_n : lf::BN) << 24));
    if (g.p.streamk)
        g.p.epoch = next_epoch(g.dev);  // each launch's flags are distinct from every earlier one
    g.p.tile_ctl = g.dev->tile_ctl;
    // Stages of two K blocks for the cross-entropy epilogues' whole-tile
    // launches (same process, same results: 4096 x 32768 x 4096 gradient
    // 664 -> 642 us, 8192 x 128256 x 4096 loss 4.71 -> 4.33 ms); one K block
    // for the plain store and every stream-K launch (the projection:
    // 71.3 -> 79.5 us with two).
    g.p.ksub = (g.pair && !g.p.streamk && (epi == lf::EPI_XENT_PARTIAL || epi == lf::EPI_XENT_EXP)) ? 2 : 1;
    g.p.tma_store = 0;
    std::memset(&g.to, 0, sizeof g.to);
    if (g.pair && (epi == lf::EPI_STORE || epi == lf::EPI_XENT_GRAD || epi == lf::EPI_XENT_EXP) && g.p.out) {
        const bool b3 = (g.layout & 4) != 0;
        const int64_t batch = b3 ? g.p.batch : 1;
        const int64_t stride = batch > 1 ? g.p.stride_o : static_cast<int64_t>(g.p.M) * g.p.ldo;
        g.p.tma_store = make_tmap_out(&g.to, g.p.out, g.p.M, g.p.N, g.p.ldo, batch, stride, b3) ? 1 : 0;
    }
    if (!g.pair)
        return lf::launch_gemm_nt(epi, g.ta, g.tb, g.p, g.grid, stream);
    const CUtensorMap &ta = (g.p.mn3 & 1) ? g.ta3 : g.ta;
    const CUtensorMap &tb = (g.p.mn3 & 2) ? g.tb3 : g.tb;
    cudaError_t e = lf::launch_gemm_nt_pair(epi, g.layout, ta, tb, g.to, g.p, g.grid, stream);
    if (e != cudaSuccess && g.p.streamk) {
        // The stream-K split is launched cooperatively (its tile owners wait for
        // other CTAs).  If the runtime refuses that, run whole tiles, which have
        // no cross-CTA waits, and stop choosing schedules that need it.
        cudaGetLastError();
        g.p.streamk = 0;
        g.p.dyn_tiles = 0;
        g.p.ksub = (epi == lf::EPI_XENT_PARTIAL || epi == lf::EPI_XENT_EXP) ? 2 : 1;
        g.grid = 2 * (g.p.num_tiles < g.dev->pair_clusters ? g.p.num_tiles : g.dev->pair_clusters);
        g_last_plan.store((g_last_plan.load() & ~((0xfffffull) | (1ull << 23))) | static_cast<uint64_t>(g.grid));
        e = lf::launch_gemm_nt_pair(epi, g.layout, ta, tb, g.to, g.p, g.grid, stream);
        if (e == cudaSuccess)
            g.dev->coop.store(-1);
    }
    return e;
}

lf_status launched(cudaError_t e, int n)
{
    if (e != cudaSuccess)
        return LF_ERR_LAUNCH;
    g_launches.fetch_add(static_cast<uint64_t>(n));
    return LF_OK;
}

// One planned GEMM launch; a stream-K launch or one that claims its tiles at
// run time uses the workspace, so it is ordered against the other workspace
// users (WorkspaceOrder).
lf_status run_planned(int epi, GemmPlan &g, cudaStream_t stream)
{
    if (!g.p.streamk && !g.p.dyn_tiles)
        return launched(run_gemm(epi, g, stream), 1);
    WorkspaceOrder order(g.dev, stream);
    if (!order.ok())
        return LF_ERR_LAUNCH;
    return launched(run_gemm(epi, g, stream), 1);
}

}  // namespace

namespace lf {

// LF_DEBUG_SYNC (read once): after every call, synchronise its stream and read
// the device error word, so asynchronous failures surface as the call's status.
bool debug_sync_enabled()
{
    static const bool on = [] {
        const char *v = std::getenv("LF_DEBUG_SYNC");
        return v && v[0] && std::strcmp(v, "0") != 0;
    }();
    return on;
}

}  // namespace lf

extern "C" lf_status lf_check_device_error(cudaStream_t stream);

namespace {

lf_status debug_sync(lf_status st, cudaStream_t stream)
{
    if (st != LF_OK || !lf::debug_sync_enabled())
        return st;
    return lf_check_device_error(stream);
}

lf_status check_gemm_shape(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0 || M > MAX_DIM || N > MAX_DIM || K > MAX_DIM)
        return LF_ERR_SHAPE;
    // the number of output tiles must fit an int as well
    if (((M + lf::BM - 1) / lf::BM) * ((N + lf::BN - 1) / lf::BN) > MAX_DIM)
        return LF_ERR_SHAPE;
    return LF_OK;
}

}  // namespace

namespace lf {

unsigned long long wait_timeout_ns() { return g_timeout_ns.load(); }
bool cooperative_launches() { return g_coop_enable.load() != 0; }
int stall_injection() { return g_inject.load(); }
void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }
bool make_tmap_kmajor(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, uint32_t box_rows)
{
    return make_tmap(m, ptr, rows, K, box_rows);
}

}  // namespace lf

extern "C" {

static lf_status gemm_nt_call(const void *x, const void *w, void *out, int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    if (!x || !w || !out)
        return LF_ERR_NULL;
    lf_status st = check_gemm_shape(M, N, K);
    if (st != LF_OK)
        return st;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || N % 8 != 0 || (K != 1 && K % 8 != 0))
        return LF_ERR_ALIGN;
    DeviceState *d = nullptr;
    if ((st = current_device(&d)) != LF_OK)
        return st;
    if (K == 1)
        return launched(lf::launch_matmul_k1_bf16(x, w, out, M, N, d->num_sms, stream), 1);
    const int variant = g_variant.load();
    GemmPlan g;
    g.no_flags = capturing(stream);
    const int64_t tiles1 = (N + lf::BN - 1) / lf::BN;  // single-CTA tiles of a skinny X
    if (d->pair_clusters > 0 && M <= lf::BM && (variant == 4 || (variant < 0 && tiles1 * 2 < d->num_sms))) {
        // Skinny X with few output tiles: swap the operands so W's N rows fill
        // the MMA's 256-row side and X's M rows (rounded up to 16) are the MMA's
        // N -- outT = W . X^T, stored transposed -- instead of tiles whose X rows
        // are mostly zero (64 x 5120 x 13824: 39 us against 54 us stream-K and
        // 94 us single-CTA).  With enough tiles (64 x 32768 x 4096) the
        // single-CTA kernel is faster (51 vs 55 us) and keeps the call.
        if ((st = plan_gemm(d, w, x, N, M, K, &g, 0, nullptr, static_cast<int>((M + 15) / 16 * 16))) != LF_OK)
            return st;
        g.p.out = out;
        g.p.ldo = N;
        return run_planned(lf::EPI_STORE_T, g, stream);
    }
    if ((st = plan_gemm(d, x, w, M, N, K, &g)) != LF_OK)
        return st;
    g.p.out = out;
    return run_planned(lf::EPI_STORE, g, stream);
}

static lf_status gemm_layout_call(const void *x, int x_layout, const void *w, int w_layout, void *out, int64_t M, int64_t N,
                                  int64_t K, cudaStream_t stream)
{
    if (!x || !w || !out)
        return LF_ERR_NULL;
    if ((x_layout != LF_K_MAJOR && x_layout != LF_MN_MAJOR) || (w_layout != LF_K_MAJOR && w_layout != LF_MN_MAJOR))
        return LF_ERR_SHAPE;
    lf_status st = check_gemm_shape(M, N, K);
    if (st != LF_OK)
        return st;
    // row pitches must be multiples of 16 bytes: K for a K-major operand, M
    // (resp. N) for an MN-major one; out's pitch is N
    const bool x_mn = x_layout == LF_MN_MAJOR, w_mn = w_layout == LF_MN_MAJOR;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || N % 8 != 0 || (x_mn && M % 8 != 0) ||
        (K != 1 && ((!x_mn && K % 8 != 0) || (!w_mn && K % 8 != 0))))
        return LF_ERR_ALIGN;
    DeviceState *d = nullptr;
    if ((st = current_device(&d)) != LF_OK)
        return st;
    if (K == 1)  // a [M,1] / [1,M] operand is the same vector either way
        return launched(lf::launch_matmul_k1_bf16(x, w, out, M, N, d->num_sms, stream), 1);
    GemmPlan g;
    g.no_flags = capturing(stream);
    if ((st = plan_gemm(d, x, w, M, N, K, &g, (x_mn ? 1 : 0) | (w_mn ? 2 : 0))) != LF_OK)
        return st;
    g.p.out = out;
    return run_planned(lf::EPI_STORE, g, stream);
}

static lf_status gemm_batched_call(const void *x, int x_layout, int64_t ldx, int64_t stride_x, const void *w, int w_layout,
                                   int64_t ldw, int64_t stride_w, void *out, int64_t ldo, int64_t stride_o, int64_t batch,
                                   int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    if (!x || !w || !out)
        return LF_ERR_NULL;
    if ((x_layout != LF_K_MAJOR && x_layout != LF_MN_MAJOR) || (w_layout != LF_K_MAJOR && w_layout != LF_MN_MAJOR))
        return LF_ERR_SHAPE;
    lf_status st = check_gemm_shape(M, N, K);
    if (st != LF_OK)
        return st;
    const bool x_mn = x_layout == LF_MN_MAJOR, w_mn = w_layout == LF_MN_MAJOR;
    // every view lies inside its row pitch; batches of out do not overlap
    if (batch < 1 || batch > MAX_DIM || ldx < (x_mn ? M : K) || ldw < (w_mn ? N : K) || ldo < N ||
        stride_x < 0 || stride_w < 0 || (batch > 1 && stride_o < (M - 1) * ldo + N))
        return LF_ERR_SHAPE;
    // TMA and the 16-byte stores: 16-byte bases, row pitches and batch strides
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || ldx % 8 || ldw % 8 || ldo % 8 || N % 8 ||
        stride_x % 8 || stride_w % 8 || stride_o % 8)
        return LF_ERR_ALIGN;
    DeviceState *d = nullptr;
    if ((st = current_device(&d)) != LF_OK)
        return st;
    const BatchSpec bs = {batch, ldx, stride_x, ldw, stride_w, ldo, stride_o};
    GemmPlan g;
    g.no_flags = capturing(stream);
    if ((st = plan_gemm(d, x, w, M, N, K, &g, (x_mn ? 1 : 0) | (w_mn ? 2 : 0), &bs)) != LF_OK)
        return st;
    g.p.out = out;
    return run_planned(lf::EPI_STORE, g, stream);
}

}  // extern "C"

namespace {

// gemm_nt_xent with X stored [M,K] (x_mn false) or [K,M], W stored [N,K]
// (w_mn false) or [K,N].  Operands in their stored layouts are read in place
// (MN-major ones through MN-major tensor-core descriptors), by the one-pass
// gradient kernel as by the two-pass form; with an N-major W the one-pass
// N-tile width is 128 or 256.
lf_status xent_impl(const void *x, bool x_mn, const void *w, bool w_mn, const int32_t *labels, float *loss,
                    void *grad_or_null, int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    if (!x || !w || !labels || !loss)
        return LF_ERR_NULL;
    lf_status st = check_gemm_shape(M, N, K);
    if (st != LF_OK)
        return st;
    if (K == 1)
        return LF_ERR_SHAPE;
    // row pitches must be multiples of 16 bytes: K for a K-major operand, M
    // (resp. N) for an MN-major one
    if (!aligned16(x) || !aligned16(w) || !aligned4(labels) || !aligned4(loss) ||
        (grad_or_null && !aligned16(grad_or_null)) || N % 8 != 0 || (x_mn && M % 8 != 0) ||
        ((!x_mn || !w_mn) && K % 8 != 0))
        return LF_ERR_ALIGN;
    DeviceState *d = nullptr;
    if ((st = current_device(&d)) != LF_OK)
        return st;
    WorkspaceOrder order(d, stream);  // every form below uses the per-device workspace
    if (!order.ok())
        return LF_ERR_LAUNCH;
    const int layout = (x_mn ? 1 : 0) | (w_mn ? 2 : 0);
    GemmPlan g;
    g.no_flags = capturing(stream);
    if ((st = plan_gemm(d, x, w, M, N, K, &g, layout)) != LF_OK)
        return st;
    lf::GemmParams &p = g.p;
    p.labels = labels;
    if (p.num_n_blocks == 1) {
        // N <= 256: one N tile holds whole rows, so the row reduction needs
        // no merge across tiles -- loss and gradient come from one epilogue,
        // one launch, no workspace.
        p.loss = loss;
        p.out = grad_or_null;
        return launched(run_gemm(lf::EPI_XENT_ROW, g, stream), 1);
    }
    // workspace: part_max, part_sum [M, NB]; label_logit, row_max, row_logsum [M]
    const size_t part = round_up(static_cast<size_t>(M) * p.num_n_blocks * sizeof(float), 256);
    const size_t vec = round_up(static_cast<size_t>(M) * sizeof(float), 256);
    void *ws = nullptr;
    if ((st = ensure_workspace(d, 2 * part + 3 * vec, &ws)) != LF_OK)
        return st;
    char *wsb = static_cast<char *>(ws);
    p.part_max = reinterpret_cast<float *>(wsb);
    p.part_sum = reinterpret_cast<float *>(wsb + part);
    p.label_logit = reinterpret_cast<float *>(wsb + 2 * part);
    float *row_max = reinterpret_cast<float *>(wsb + 2 * part + vec);
    float *row_logsum = reinterpret_cast<float *>(wsb + 2 * part + 2 * vec);
    p.labels = labels;
    // Which gradient form: the exp pass + rescale (a GEMM writing fp16
    // exp(z - tile max) into grad, then one bandwidth-bound pass) -- the
    // automatic choice --, the one-pass kernel (on request, or when a
    // one-pass tile width is forced), or the recompute pass (single-CTA tiles,
    // or rows too wide for the rescale kernel's shared memory).
    const int path = g_xent_path.load();
    const int forced = g_op_tile.load();
    const bool exp_ok = grad_or_null && g.pair && p.num_n_blocks <= RESCALE_MAX_TILES;
    const bool try_onepass = grad_or_null && g.pair && d->coop.load() >= 0 && !g.no_flags &&
                             (path == 1 || (path == 0 && (!exp_ok || forced != 0)));
    // One pass, when a whole 256-row block of tiles (two per pair) fits on the
    // resident pairs -- no recompute GEMM and no combine kernel.  N-tile width:
    // the one with the least rounds x width (the time of a round is about
    // proportional to its tiles' width), i.e. the narrowest that keeps the
    // fewest rounds: more pairs busy, shorter MMA chains.  (4096 x 32768 x
    // 4096: 0.836 ms at 224 with 74 pairs against 0.847 ms at 256 with 64.)
    int op_tile = 0;
    long long best = 0;
    for (int wdt = 256; wdt >= 128 && try_onepass; wdt -= 32) {
        if (forced && wdt != forced)
            continue;
        if (w_mn && wdt != 256 && wdt != 128)  // an N-major W arrives in 64-row boxes per CTA half tile
            continue;
        const int nt = static_cast<int>((N + wdt - 1) / wdt);
        const int q = (nt + 1) / 2;
        if (q > d->pair_clusters)
            continue;
        int k = d->pair_clusters / q;
        if (k > p.num_m_blocks)
            k = p.num_m_blocks;
        const int rounds = (p.num_m_blocks + k - 1) / k;
        const long long cost = static_cast<long long>(rounds) * wdt;
        if (op_tile == 0 || cost < best) {
            op_tile = wdt;
            best = cost;
        }
    }
    if (op_tile > 0) {
        if ((st = ensure_onepass_flags(d)) != LF_OK)
            return st;
        CUtensorMap tb_op = g.tb;  // an N-major W: the plan's 64 x 64 boxes
        if (!w_mn && !make_tmap(&tb_op, w, N, K, static_cast<uint32_t>(op_tile / 2)))
            return LF_ERR_LAUNCH;  // a K-major W: boxes of op_tile / 2 rows (each CTA's half of a tile)
        p.streamk = 0;
        p.op_tile = op_tile;
        p.op_ntiles = static_cast<int>((N + op_tile - 1) / op_tile);
        p.op_Q = (p.op_ntiles + 1) / 2;
        p.op_k = d->pair_clusters / p.op_Q;
        if (p.op_k > p.num_m_blocks)
            p.op_k = p.num_m_blocks;
        p.op_rounds = (p.num_m_blocks + p.op_k - 1) / p.op_k;
        p.round_flags = static_cast<unsigned long long *>(d->op_flags);
        p.op_stash = reinterpret_cast<float *>(static_cast<char *>(d->op_flags) + onepass_flag_bytes(d));
        p.loss = loss;
        p.out = grad_or_null;
        p.epoch = next_epoch(d);
        CUtensorMap to;  // the gradient, written by TMA stores
        if (!make_tmap_out(&to, grad_or_null, M, N, N, 1, M * N, false))
            return LF_ERR_LAUNCH;
        if (lf::launch_xent_onepass(layout, g.ta, tb_op, to, p, 2 * p.op_k * p.op_Q, stream) == cudaSuccess)
            return launched(cudaSuccess, 1);
        // The one-pass kernel is launched cooperatively (a group's pairs wait
        // for each other); the runtime refused that, so take the two-pass
        // form below, and stop choosing schedules that need it.
        cudaGetLastError();
        d->coop.store(-1);
        if ((st = plan_gemm(d, x, w, M, N, K, &g, layout)) != LF_OK)
            return st;
        p.part_max = reinterpret_cast<float *>(wsb);
        p.part_sum = reinterpret_cast<float *>(wsb + part);
        p.label_logit = reinterpret_cast<float *>(wsb + 2 * part);
        p.labels = labels;
    }
    if (exp_ok && path != 3) {
        // exp pass: partials and e = fp16(exp(z - tile max)) into grad, then
        // the rescale kernel: lse, loss, and grad rewritten in place as bf16
        p.out = grad_or_null;
        if ((st = launched(run_gemm(lf::EPI_XENT_EXP, g, stream), 1)) != LF_OK)
            return st;
        return launched(lf::launch_xent_rescale(p.part_max, p.part_sum, p.label_logit, labels, p.M, p.N,
                                                p.num_n_blocks, loss, grad_or_null, stream),
                        1);
    }
    if ((st = launched(run_gemm(lf::EPI_XENT_PARTIAL, g, stream), 1)) != LF_OK)
        return st;
    if ((st = launched(lf::launch_xent_combine(p.part_max, p.part_sum, p.label_logit, labels, p.M, p.N,
                                               p.num_n_blocks, loss, grad_or_null ? row_max : nullptr,
                                               grad_or_null ? row_logsum : nullptr, stream),
                       1)) != LF_OK)
        return st;
    if (!grad_or_null)
        return LF_OK;
    p.out = grad_or_null;
    p.row_max = row_max;
    p.row_logsum = row_logsum;
    p.inject = 0;
    return launched(run_gemm(lf::EPI_XENT_GRAD, g, stream), 1);
}

}  // namespace

extern "C" {

static lf_status gemm_nt_xent_call(const void *x, const void *w, const int32_t *labels, float *loss, void *grad_or_null,
                                   int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    return xent_impl(x, false, w, false, labels, loss, grad_or_null, M, N, K, stream);
}

static lf_status gemm_nt_xent_layout_call(const void *x, int x_layout, const void *w, int w_layout, const int32_t *labels,
                                          float *loss, void *grad_or_null, int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    if ((x_layout != LF_K_MAJOR && x_layout != LF_MN_MAJOR) || (w_layout != LF_K_MAJOR && w_layout != LF_MN_MAJOR))
        return LF_ERR_SHAPE;
    return xent_impl(x, x_layout == LF_MN_MAJOR, w, w_layout == LF_MN_MAJOR, labels, loss, grad_or_null, M, N, K,
                     stream);
}

static lf_status matmul_k1_call(const float *a, const float *b, float *out, int64_t M, int64_t N, cudaStream_t stream)
{
    if (!a || !b || !out)
        return LF_ERR_NULL;
    if (M <= 0 || N <= 0 || M > MAX_DIM || N > MAX_DIM)
        return LF_ERR_SHAPE;
    if (!aligned4(a) || !aligned4(b) || !aligned4(out))
        return LF_ERR_ALIGN;
    DeviceState *d = nullptr;
    lf_status st = current_device(&d);
    if (st != LF_OK)
        return st;
    return launched(lf::launch_matmul_k1_f32(a, b, out, M, N, d->num_sms, stream), 1);
}

static lf_status rope_cos_sin_call(const void *inv_freq, const int64_t *positions, void *cos_out, void *sin_out_or_null,
                                   int64_t H, int64_t S, cudaStream_t stream)
{
    if (!inv_freq || !positions || !cos_out)
        return LF_ERR_NULL;
    if (H <= 0 || S <= 0 || H > MAX_DIM || S > MAX_DIM)
        return LF_ERR_SHAPE;
    const auto misaligned = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
    if (misaligned(inv_freq, 2) || misaligned(positions, 8) || misaligned(cos_out, 2) ||
        (sin_out_or_null && misaligned(sin_out_or_null, 2)))
        return LF_ERR_ALIGN;
    DeviceState *d = nullptr;
    lf_status st = current_device(&d);
    if (st != LF_OK)
        return st;
    return launched(lf::launch_rope_cos_sin(inv_freq, positions, cos_out, sin_out_or_null, H, S, d->num_sms, stream),
                    1);
}

static lf_status fp8_cast_dual_call(const void *x, const float *scale, void *out, void *out_t, int64_t M, int64_t K,
                                    cudaStream_t stream)
{
    if (!x || !scale || !out || !out_t)
        return LF_ERR_NULL;
    if (M <= 0 || K <= 0 || M > MAX_DIM || K > MAX_DIM)
        return LF_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(x) & 1u) != 0)
        return LF_ERR_ALIGN;
    DeviceState *d = nullptr;
    lf_status st = current_device(&d);
    if (st != LF_OK)
        return st;
    return launched(lf::launch_fp8_cast_dual(x, scale, out, out_t, M, K, d->num_sms, stream), 1);
}

const char *lf_status_string(lf_status s)
{
    switch (s) {
    case LF_OK: return "ok";
    case LF_ERR_NULL: return "null pointer argument";
    case LF_ERR_SHAPE: return "invalid shape";
    case LF_ERR_ALIGN: return "misaligned pointer or unsupported row pitch";
    case LF_ERR_LAUNCH: return "CUDA launch or runtime error";
    case LF_ERR_WORKSPACE: return "workspace allocation failed";
    case LF_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case LF_ERR_ARCH: return "current device is not sm_103";
    }
    return "unknown status";
}

lf_status lf_check_device_error(cudaStream_t stream)
{
    DeviceState *d = nullptr;
    lf_status st = current_device(&d);
    if (st != LF_OK)
        return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return LF_ERR_LAUNCH;
    }
    int code = 0;
    if (cudaMemcpyAsync(&code, d->err_word, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return LF_ERR_LAUNCH;
    }
    if (code == 0)
        return LF_OK;
    g_last_wait_code.store(code);
    if (cudaMemsetAsync(d->err_word, 0, sizeof(int), stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return LF_ERR_LAUNCH;
    }
    return LF_ERR_DEVICE_TIMEOUT;
}

uint64_t lf_launch_count(void) { return g_launches.load(); }

int lf_last_device_wait_code(void) { return g_last_wait_code.load(); }

void lf_last_gemm_plan(int *grid, int *cta_pairs, int *stream_k, int *tile_n)
{
    const uint64_t v = g_last_plan.load();
    if (grid)
        *grid = static_cast<int>(v & 0xfffffu);
    if (cta_pairs)
        *cta_pairs = static_cast<int>((v >> 20) & 1u);
    if (stream_k)
        *stream_k = static_cast<int>((v >> 23) & 1u);
    if (tile_n)
        *tile_n = static_cast<int>(v >> 24);
}

lf_status lf_device_query(int *num_sms, int *pair_clusters)
{
    DeviceState *d = nullptr;
    lf_status st = current_device(&d);
    if (st != LF_OK)
        return st;
    if (num_sms)
        *num_sms = d->num_sms;
    if (pair_clusters)
        *pair_clusters = d->pair_clusters;
    return LF_OK;
}

void lf_set_tuning(int l2_prefetch_kblocks, int gemm_variant)
{
    g_l2_prefetch.store(l2_prefetch_kblocks < 0 ? -1 : l2_prefetch_kblocks);
    g_variant.store(gemm_variant >= 1 && gemm_variant <= 4 ? gemm_variant : -1);
}

void lf_set_xent_grad_path(int path) { g_xent_path.store(path >= 1 && path <= 3 ? path : 0); }

void lf_set_tile_band(int m_blocks) { g_band.store(m_blocks < 0 ? -1 : m_blocks); }

void lf_set_tile_schedule(int mode) { g_tile_sched.store(mode < 0 ? -1 : (mode ? 1 : 0)); }

void lf_set_cooperative(int enable) { g_coop_enable.store(enable ? 1 : 0); }

void lf_set_onepass_tile(int width)
{
    g_op_tile.store(width >= 128 && width <= 256 && width % 32 == 0 ? width : 0);
}

lf_status lf_test_occupy_sms(int ctas, uint64_t duration_ns, cudaStream_t stream)
{
    DeviceState *d = nullptr;
    lf_status st = current_device(&d);
    if (st != LF_OK)
        return st;
    if (ctas < 1 || ctas > d->num_sms || duration_ns == 0 || duration_ns > 5000000000ull)
        return LF_ERR_SHAPE;
    return launched(lf::launch_occupy_sms(ctas, static_cast<unsigned long long>(duration_ns), stream), 1);
}

void lf_set_test_hooks(int inject_stall, uint64_t wait_timeout_ns)
{
    g_inject.store(inject_stall ? 1 : 0);
    g_timeout_ns.store(wait_timeout_ns ? wait_timeout_ns : 2000000000ull);
}

}  // extern "C"

// The exported entry points: an optional profiling range around each call and,
// with LF_DEBUG_SYNC set in the environment, a synchronising check that turns
// a device-side timeout or launch error into the call's own status.
extern "C" {

lf_status gemm_nt(const void *x, const void *w, void *out, int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    const lf::CallRange range("gemm_nt");
    return debug_sync(gemm_nt_call(x, w, out, M, N, K, stream), stream);
}

lf_status gemm_layout(const void *x, int x_layout, const void *w, int w_layout, void *out, int64_t M, int64_t N,
                      int64_t K, cudaStream_t stream)
{
    const lf::CallRange range("gemm_layout");
    return debug_sync(gemm_layout_call(x, x_layout, w, w_layout, out, M, N, K, stream), stream);
}

lf_status gemm_batched(const void *x, int x_layout, int64_t ldx, int64_t stride_x, const void *w, int w_layout,
                       int64_t ldw, int64_t stride_w, void *out, int64_t ldo, int64_t stride_o, int64_t batch,
                       int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    const lf::CallRange range("gemm_batched");
    return debug_sync(gemm_batched_call(x, x_layout, ldx, stride_x, w, w_layout, ldw, stride_w, out, ldo, stride_o,
                                        batch, M, N, K, stream),
                      stream);
}

lf_status gemm_nt_xent(const void *x, const void *w, const int32_t *labels, float *loss, void *grad_or_null,
                       int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    const lf::CallRange range("gemm_nt_xent");
    return debug_sync(gemm_nt_xent_call(x, w, labels, loss, grad_or_null, M, N, K, stream), stream);
}

lf_status gemm_nt_xent_layout(const void *x, int x_layout, const void *w, int w_layout, const int32_t *labels,
                              float *loss, void *grad_or_null, int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    const lf::CallRange range("gemm_nt_xent_layout");
    return debug_sync(
        gemm_nt_xent_layout_call(x, x_layout, w, w_layout, labels, loss, grad_or_null, M, N, K, stream), stream);
}

lf_status matmul_k1(const float *a, const float *b, float *out, int64_t M, int64_t N, cudaStream_t stream)
{
    const lf::CallRange range("matmul_k1");
    return debug_sync(matmul_k1_call(a, b, out, M, N, stream), stream);
}

lf_status rope_cos_sin(const void *inv_freq, const int64_t *positions, void *cos_out, void *sin_out_or_null,
                       int64_t H, int64_t S, cudaStream_t stream)
{
    const lf::CallRange range("rope_cos_sin");
    return debug_sync(rope_cos_sin_call(inv_freq, positions, cos_out, sin_out_or_null, H, S, stream), stream);
}

lf_status fp8_cast_dual(const void *x, const float *scale, void *out, void *out_t, int64_t M, int64_t K,
                        cudaStream_t stream)
{
    const lf::CallRange range("fp8_cast_dual");
    return debug_sync(fp8_cast_dual_call(x, scale, out, out_t, M, K, stream), stream);
}

}  // extern "C"
