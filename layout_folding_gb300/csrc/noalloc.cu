// noalloc.cu -- gemm_nt_xent_noalloc: the fused GEMM + cross-entropy of
// gemm_nt_xent with its scratch in a fixed, statically sized device array
// instead of memory the library allocates.
//
// Who needs this: callers that must not allocate device memory at call time
// -- code running while a CUDA graph is being captured (cudaMalloc/cudaFree
// are not capturable and cudaFree synchronises the device), allocators that
// own every byte of the GPU (e.g. a framework caching allocator or a serving
// engine that reserved all memory up front), and real-time paths that cannot
// afford the synchronisation a first-use cudaMalloc implies.  This entry point
// calls no cudaMalloc, cudaFree or allocating library routine.
//
// The scratch is the file-scope array below: every GPU that loads the library
// holds it (NOALLOC_SCRATCH_BYTES) until the process exits.  Host code must
// not pass the array's name to a kernel (in host code it is only a stand-in
// symbol, not a device address); the device address is looked up once per
// device with cudaGetSymbolAddress and passed to the kernels.
#include <cstring>
#include <mutex>

#include <cuda_bf16.h>

#include "layoutfold.h"
#include "lf_internal.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(32) << 20;  // 32 MiB
constexpr size_t ERR_BYTES = 256;                            // error word region at the start
constexpr int MAX_DEVICES = 64;
constexpr int64_t MAX_DIM = (int64_t(1) << 31) - 1;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

struct NoAllocDevice {
    bool ready = false;
    bool arch_ok = false;
    int num_sms = 0;
    char *scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_noalloc_mutex;
NoAllocDevice g_noalloc_dev[MAX_DEVICES];

// Set-up of the current device, done once per device by the first call made
// with that device current: architecture check and the scratch's device
// address.  Nothing is allocated.
lf_status noalloc_device(NoAllocDevice **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return LF_ERR_ARCH;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
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
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return LF_ERR_LAUNCH;
            }
            d.scratch = static_cast<char *>(p);
        }
        d.ready = true;
    }
    if (!d.arch_ok)
        return LF_ERR_ARCH;
    *out = &d;
    return LF_OK;
}

// A device-side wait that ran out makes the call's outputs NaN -- every loss
// and, when a gradient was asked for, every gradient element -- so the failure
// is visible in the output of this variant.
__global__ void k_noalloc_poison(const int *err, float *loss, int M, __nv_bfloat16 *grad, size_t grad_elems)
{
    if (*err == 0)
        return;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (size_t i = i0; i < static_cast<size_t>(M); i += stride)
        loss[i] = __int_as_float(0x7fc00000);
    for (size_t i = i0; i < grad_elems; i += stride)
        grad[i] = __ushort_as_bfloat16(static_cast<unsigned short>(0x7fc0));
}

size_t round_up256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

static lf_status noalloc_call(const void *x, const void *w, const int32_t *labels, float *loss, void *grad_or_null,
                              int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    if (!x || !w || !labels || !loss)
        return LF_ERR_NULL;
    if (M <= 0 || N <= 0 || K <= 1 || M > MAX_DIM || N > MAX_DIM || K > MAX_DIM)
        return LF_ERR_SHAPE;
    const int64_t num_m_blocks = (M + lf::BM - 1) / lf::BM;
    const int64_t num_n_blocks = (N + lf::BN - 1) / lf::BN;
    if (num_m_blocks * num_n_blocks > MAX_DIM)
        return LF_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w) & 15u) ||
        (reinterpret_cast<uintptr_t>(labels) & 3u) || (reinterpret_cast<uintptr_t>(loss) & 3u) ||
        (grad_or_null && (reinterpret_cast<uintptr_t>(grad_or_null) & 15u)) || N % 8 != 0 || K % 8 != 0)
        return LF_ERR_ALIGN;
    // scratch layout: error word | part_max, part_sum [M, NB] | label_logit, row_max, row_logsum [M]
    const size_t part = round_up256(static_cast<size_t>(M) * num_n_blocks * sizeof(float));
    const size_t vec = round_up256(static_cast<size_t>(M) * sizeof(float));
    if (ERR_BYTES + 2 * part + 3 * vec > NOALLOC_SCRATCH_BYTES)
        return LF_ERR_WORKSPACE;
    NoAllocDevice *d = nullptr;
    lf_status st = noalloc_device(&d);
    if (st != LF_OK)
        return st;

    char *s = d->scratch;
    int *err = reinterpret_cast<int *>(s);
    lf::GemmParams p;
    std::memset(&p, 0, sizeof p);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_m_blocks = static_cast<int>(num_m_blocks);
    p.num_n_blocks = static_cast<int>(num_n_blocks);
    p.num_k_blocks = static_cast<int>((K + lf::BK - 1) / lf::BK);
    p.num_tiles = p.num_m_blocks * p.num_n_blocks;
    p.err = err;
    p.timeout_ns = lf::wait_timeout_ns();
    p.inject = lf::stall_injection();  // test hook, as for the other entry points
    p.labels = labels;
    p.part_max = reinterpret_cast<float *>(s + ERR_BYTES);
    p.part_sum = reinterpret_cast<float *>(s + ERR_BYTES + part);
    p.label_logit = reinterpret_cast<float *>(s + ERR_BYTES + 2 * part);
    float *row_max = reinterpret_cast<float *>(s + ERR_BYTES + 2 * part + vec);
    float *row_logsum = reinterpret_cast<float *>(s + ERR_BYTES + 2 * part + 2 * vec);

    CUtensorMap ta, tb;
    if (!lf::make_tmap_kmajor(&ta, x, M, K, lf::BM) || !lf::make_tmap_kmajor(&tb, w, N, K, lf::BN))
        return LF_ERR_LAUNCH;
    const int grid = p.num_tiles < d->num_sms ? p.num_tiles : d->num_sms;

    // The error word keeps the previous call's value: clear it first.
    if (cudaMemsetAsync(err, 0, sizeof(int), stream) != cudaSuccess) {
        cudaGetLastError();
        return LF_ERR_LAUNCH;
    }
    if (lf::launch_gemm_nt(lf::EPI_XENT_PARTIAL, ta, tb, p, grid, stream) != cudaSuccess ||
        lf::launch_xent_combine(p.part_max, p.part_sum, p.label_logit, labels, p.M, p.N, p.num_n_blocks, loss,
                                grad_or_null ? row_max : nullptr, grad_or_null ? row_logsum : nullptr,
                                stream) != cudaSuccess)
        return LF_ERR_LAUNCH;
    lf::count_launches(2);
    if (grad_or_null) {
        p.out = grad_or_null;
        p.row_max = row_max;
        p.row_logsum = row_logsum;
        p.inject = 0;
        if (lf::launch_gemm_nt(lf::EPI_XENT_GRAD, ta, tb, p, grid, stream) != cudaSuccess)
            return LF_ERR_LAUNCH;
        lf::count_launches(1);
    }
    const size_t grad_elems = grad_or_null ? static_cast<size_t>(M) * static_cast<size_t>(N) : 0;
    const size_t work = grad_elems > static_cast<size_t>(M) ? grad_elems : static_cast<size_t>(M);
    const int pgrid = static_cast<int>((work + 255) / 256 < 1024 ? (work + 255) / 256 : 1024);
    k_noalloc_poison<<<pgrid, 256, 0, stream>>>(err, loss, p.M, static_cast<__nv_bfloat16 *>(grad_or_null),
                                                grad_elems);
    if (cudaGetLastError() != cudaSuccess)
        return LF_ERR_LAUNCH;
    lf::count_launches(1);
    return LF_OK;
}

// The exported entry point: an optional profiling range and, with
// LF_DEBUG_SYNC set, a synchronising check of this call's own error word
// (a wait that ran out returns LF_ERR_DEVICE_TIMEOUT besides the NaN outputs).
extern "C" lf_status gemm_nt_xent_noalloc(const void *x, const void *w, const int32_t *labels, float *loss,
                                          void *grad_or_null, int64_t M, int64_t N, int64_t K,
                                          cudaStream_t stream)
{
    const lf::CallRange range("gemm_nt_xent_noalloc");
    lf_status st = noalloc_call(x, w, labels, loss, grad_or_null, M, N, K, stream);
    if (st != LF_OK || !lf::debug_sync_enabled())
        return st;
    NoAllocDevice *d = nullptr;
    if ((st = noalloc_device(&d)) != LF_OK)
        return st;
    int code = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess ||
        cudaMemcpy(&code, d->scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return LF_ERR_LAUNCH;
    }
    return code ? LF_ERR_DEVICE_TIMEOUT : LF_OK;
}

