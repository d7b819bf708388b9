/*
 * layoutfold.h -- C ABI of liblayoutfold.so, the GB300 (sm_103a) library for
 * the layout-folded GEMM paths.
 *
 * Notation: X is [M,K], W is [N,K]; both are row-major with K contiguous
 * ("K-major").  All matrices are contiguous, row-major, and live in device
 * memory owned by the caller; the library never frees them and keeps no
 * reference to them after the call returns.
 *
 * Every entry point validates its arguments on the host and then enqueues its
 * kernels on `stream` (0 = the legacy default stream) and returns without
 * synchronising.  Host-checkable errors are returned immediately and nothing
 * is enqueued.  A launch failure returns LF_ERR_LAUNCH.  A device-side wait
 * that runs past its time limit is not visible at return time: it is recorded
 * in a per-device error word that lf_check_device_error() reads.
 *
 * Every compute call requires an sm_103 device (LF_ERR_ARCH otherwise).  There
 * is no CPU fallback.
 *
 * Debugging aids: with LF_DEBUG_SYNC set (to anything but "0") in the
 * environment when the library is first used, every compute call
 * synchronises its stream before returning and reports a device-side timeout
 * or a launch error as its own status.  Built with LAYOUTFOLD_NVTX=1 in the
 * build environment (the LF_NVTX macro), every call is an NVTX range named
 * after the entry point.
 */
#ifndef LAYOUTFOLD_H
#define LAYOUTFOLD_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LF_OK = 0,
    LF_ERR_NULL = 1,            /* a required pointer is NULL */
    LF_ERR_SHAPE = 2,           /* M, N or K out of range (<= 0, too large), or K=1 given to gemm_nt_xent */
    LF_ERR_ALIGN = 3,           /* a base address is not 16-byte aligned, or K % 8 != 0 (K > 1), or N % 8 != 0 */
    LF_ERR_LAUNCH = 4,          /* a CUDA launch or runtime call failed */
    LF_ERR_WORKSPACE = 5,       /* the internal workspace could not be allocated */
    LF_ERR_DEVICE_TIMEOUT = 6,  /* a device-side wait exceeded its limit (reported by lf_check_device_error) */
    LF_ERR_ARCH = 7             /* the current device is not sm_103 */
} lf_status;

/*
 * gemm_nt -- out = X · Wᵀ with the weight consumed in its stored [N,K] layout.
 *
 * Source: "Strength reduction: fold transpose into a subsequent GEMM call"
 * (lightning-thunder issue 1252), Feature: `matmul(x, weight.t())` traced as a
 * separate transpose fusion followed by a GEMM; the page asks for an "NT" GEMM
 * that skips the transpose.  Here no transpose and no transposed copy exist:
 * both operands are read K-major by the tensor-core GEMM.
 *
 *   x   : bf16 [M,K], device, row-major (any leading batch dims flattened into M)
 *   w   : bf16 [N,K], device, row-major (the stored weight)
 *   out : bf16 [M,N], device, row-major; out[m,n] = bf16_rn(sum_k x[m,k]*w[n,k]),
 *         the sum accumulated in fp32.
 *   M, N, K : 1 <= M, N, K < 2^31.  K > 1 needs K % 8 == 0 and N % 8 == 0
 *         (16-byte row pitch for the tensor copies).
 *   K == 1 is not an error: it is sent to the pointwise outer-product kernel
 *         (out[m,n] = bf16_rn(float(x[m]) * float(w[n])), exact product, one rounding),
 *         as "Feature request: Schedule a small matmul op as a reduction (or
 *         pointwise) op" (NVIDIA/Fuser issue 3646) proposes; N % 8 == 0 is still required.
 *   x, w, out must be 16-byte aligned.  out must not overlap x or w.
 * One kernel launch per call.  A skinny X (M <= 128) with few output tiles is
 * computed with the operands swapped (out^T = W . X^T on the tensor cores,
 * stored transposed).  When the output has too few 256x256 tiles to
 * keep every SM busy and K is long enough for the split to pay, the launch
 * splits the K loop across SMs (stream-K) and
 * uses a library-owned per-device workspace (about 20 MB, allocated on first
 * such call).  Such a launch is cooperative (all its CTAs resident at once, as
 * its tile owners wait for other CTAs' partial sums); if the runtime refuses
 * that, whole tiles are used.  Calls that use the workspace are ordered: a
 * call on another stream than the previous one first makes its stream wait
 * for that call (an event, no host synchronisation), so such calls from
 * several streams or host threads run one after another on the GPU.
 */
lf_status gemm_nt(const void *x, const void *w, void *out,
                  int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * gemm_nt_xent -- logits z = X · Wᵀ (fp32, never written to memory) followed by
 * the row-wise cross-entropy over N, fused into the GEMM epilogue.
 *
 * Source: "Allow reductions in matmul epilogues" (NVIDIA/Fuser issue 2213),
 * the fusion example (row max, exp, sum-exp, log-sum-exp, the label logit via
 * a one-hot compare, and the softmax-minus-onehot output), and its follow-up
 * on reducing a row across tiles by a grid reduction.
 *
 *   x, w    : as for gemm_nt (K > 1, K % 8 == 0, N % 8 == 0).
 *   labels  : int32 [M], device.  Precondition 0 <= labels[m] < N; a row whose
 *             label is outside that range gets loss NaN and a grad row without
 *             the -1 term (no ignore-index exists).
 *   loss    : fp32 [M], device; loss[m] = logsumexp_n z[m,n] - z[m,labels[m]]
 *             (per row, no mean).
 *   grad_or_null : NULL, or bf16 [M,N], device, 16-byte aligned, overlapping
 *             none of x, w, labels, loss;
 *             grad[m,n] = bf16_rn(exp(z[m,n] - lse[m]) - [n == labels[m]])
 *             (within 2e-3 of the exact value).  While the call runs the
 *             buffer may hold intermediate values (see Work).
 *             When NULL nothing of size [M,N] is written anywhere.
 * Work: for N <= 256 every row lies in one 256-column tile, so one launch
 * writes the loss (and the gradient) from the GEMM's epilogue.  Otherwise,
 * without grad, one GEMM pass writing per-(row, 256-column tile)
 * partials (max, sum-exp) and the label logit, then one combine kernel.  With
 * grad on CTA pairs (always when M > 128 or an operand is MN-major), two
 * launches: a GEMM pass whose epilogue writes
 * the partials and fp16 exp(z - tile max) into the grad buffer itself, then a
 * kernel that merges each row's partials into lse and the loss and rewrites
 * grad in place as bf16 (the logits are computed once and never stored; rows
 * longer than 12,582,912 columns take the recompute form below).  On
 * request (lf_set_xent_grad_path(1)), when a 256-row block of tiles fits on
 * the co-resident CTA pairs (two N tiles per pair: N <= 512 x pairs), ONE
 * launch computes the logits once and writes loss and gradient, the pairs of a
 * row block exchanging their row partials through flags in global memory.  On
 * single-CTA tiles (small M): the partials pass, the combine and a GEMM pass
 * that recomputes the logits and writes the gradient.
 * The one-pass kernel is launched cooperatively (every CTA resident at once);
 * if the runtime refuses that, the two-pass form runs instead.
 * Partials, flags and the one-pass kernel's stash (128 KiB per CTA) live in a
 * per-device workspace that the library allocates on first use (and grows,
 * never shrinks) and frees at unload.  Calls are ordered as for gemm_nt: one
 * on another stream than the previous workspace user waits for it on the GPU
 * (an event), so calls from several streams or threads are correct and run
 * one after another.  (A stream that is being captured into a graph is not
 * ordered against other streams.)
 */
lf_status gemm_nt_xent(const void *x, const void *w, const int32_t *labels,
                       float *loss, void *grad_or_null,
                       int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * matmul_k1 -- the degenerate K=1 matmul as a broadcast multiply.
 *
 * Source: "Feature request: Schedule a small matmul op as a reduction (or
 * pointwise) op" (NVIDIA/Fuser issue 3646): the RoPE matmul of a [64,1]
 * inverse-frequency column and a [1,4096] position row, and its rewrite as
 * broadcast, multiply, squeeze.
 *
 *   a   : fp32 [M,1], device
 *   b   : fp32 [1,N], device
 *   out : fp32 [M,N], device, row-major; out[i,j] = a[i] * b[j] (one IEEE
 *         multiply, round-to-nearest: bit-exact).  The page's permuted
 *         [N,M] result is out viewed transposed.
 *   1 <= M, N < 2^31.  No alignment requirement beyond 4 bytes.
 */
lf_status matmul_k1(const float *a, const float *b, float *out,
                    int64_t M, int64_t N, cudaStream_t stream);

/* Stored layout of a GEMM operand (gemm_layout). */
typedef enum {
    LF_K_MAJOR = 0,  /* K contiguous: X stored [M,K], W stored [N,K] */
    LF_MN_MAJOR = 1  /* M (resp. N) contiguous: X stored [K,M], W stored [K,N] */
} lf_layout;

/*
 * gemm_layout -- out = X . W^T with either operand in either stored layout,
 * no operand ever transposed in memory.
 *
 * Source: "Strength reduction: fold transpose into a subsequent GEMM call"
 * (lightning-thunder issue 1252), Feature and the remark that one of the
 * transposed layouts is served by the GEMM directly; "Allow reductions in
 * matmul epilogues" (NVIDIA/Fuser issue 2213), whose matmul scheduler maps
 * any operand layout onto one canonical (M, N, K) contraction.  Here the
 * tensor core reads an MN-major operand from shared memory as readily as a
 * K-major one, so all four combinations are one kernel, one launch.
 *
 *   x : bf16, device, 16-byte aligned; LF_K_MAJOR: [M,K] row-major
 *       (X[m,k] = x[m*K + k]); LF_MN_MAJOR: [K,M] row-major (X[m,k] = x[k*M + m],
 *       i.e. the storage of X^T, or of an [M,K] tensor with strides (1, M)).
 *   w : bf16, device, 16-byte aligned; LF_K_MAJOR: [N,K] (W[n,k] = w[n*K + k],
 *       the gemm_nt case); LF_MN_MAJOR: [K,N] (W[n,k] = w[k*N + n], the plain
 *       x @ w of a [K,N] weight).
 *   out: bf16 [M,N] row-major, out[m,n] = bf16_rn(sum_k X[m,k] * W[n,k]),
 *       fp32 accumulation (tolerance as gemm_nt).
 *   Row pitches must be multiples of 16 bytes: K % 8 == 0 for a K-major
 *   operand (K > 1), M % 8 == 0 for an MN-major X, N % 8 == 0 always.
 *   K = 1 is the broadcast product of gemm_nt (either layout is a vector).
 *   An invalid layout value returns LF_ERR_SHAPE; other errors as gemm_nt.
 *   Both K-major is exactly gemm_nt.  Like gemm_nt it may use the stream-K
 *   split and its per-device workspace, ordered across streams as gemm_nt's.
 */
lf_status gemm_layout(const void *x, int x_layout, const void *w, int w_layout, void *out,
                      int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * gemm_batched -- gemm_layout over a batch of strided views: for b < batch,
 *   out_b[m,n] = bf16_rn(sum_k X_b[m,k] * W_b[n,k])
 * where, with all offsets in elements,
 *   X_b[m,k] = x[b*stride_x + m*ldx + k]    (LF_K_MAJOR)   or x[b*stride_x + k*ldx + m] (LF_MN_MAJOR)
 *   W_b[n,k] = w[b*stride_w + n*ldw + k]    (LF_K_MAJOR)   or w[b*stride_w + k*ldw + n] (LF_MN_MAJOR)
 *   out_b[m,n] = out[b*stride_o + m*ldo + n]
 * stride_x = 0 (stride_w = 0) uses one X (one W) for every batch.
 *
 * Source: "Strength reduction: fold transpose into a subsequent GEMM call"
 * (lightning-thunder issue 1252) -- the projection's input is a view of a
 * larger tensor -- and the batched, permuted operands of the Mistral listing
 * of "Feature request: Schedule a small matmul op as a reduction (or
 * pointwise) op" (NVIDIA/Fuser issue 3646): slices, transposes and batch
 * dimensions are all folded into the operand tensor maps (one launch, no copy).
 *
 *   Row pitches: ldx >= K (K-major X) or M (MN-major X); ldw >= K or N; ldo >= N.
 *   ldx, ldw, ldo, stride_x, stride_w, stride_o and N multiples of 8 (16
 *   bytes); x, w, out 16-byte aligned (else LF_ERR_ALIGN).  batch >= 1; for
 *   batch > 1 the out matrices must not overlap (stride_o >= (M-1)*ldo + N),
 *   else LF_ERR_SHAPE.  Inputs may overlap.  Accumulation and tolerance as
 *   gemm_nt; other errors, and the rule on concurrent calls, as gemm_layout.
 */
lf_status gemm_batched(const void *x, int x_layout, int64_t ldx, int64_t stride_x,
                       const void *w, int w_layout, int64_t ldw, int64_t stride_w,
                       void *out, int64_t ldo, int64_t stride_o,
                       int64_t batch, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * gemm_nt_xent_layout -- gemm_nt_xent with either operand in either stored
 * layout, read in place (no transposed copy).
 *
 * Source: as gemm_nt_xent ("Allow reductions in matmul epilogues", NVIDIA/Fuser
 * issue 2213), whose scheduler canonicalises any operand layout of the matmul
 * to one contraction; the layouts as in gemm_layout ("Strength reduction: fold
 * transpose into a subsequent GEMM call", the transposed weight read as is).
 *
 *   x_layout : LF_K_MAJOR (x is [M,K]) or LF_MN_MAJOR (x is [K,M], M % 8 == 0)
 *   w_layout : LF_K_MAJOR (w is [N,K]) or LF_MN_MAJOR (w is [K,N])
 *   K % 8 == 0 when either operand is K-major; N % 8 == 0 always.
 *   labels, loss, grad_or_null, M, N, K and the results: as gemm_nt_xent.
 * Any other layout value: LF_ERR_SHAPE.  With two K-major operands this is
 * gemm_nt_xent.  The work is that of gemm_nt_xent in every layout (with grad
 * one launch when a row block of tiles fits the resident CTA pairs; with an
 * N-major W its N tiles are 128 or 256 wide), and its workspace rules apply.
 */
lf_status gemm_nt_xent_layout(const void *x, int x_layout, const void *w, int w_layout, const int32_t *labels,
                              float *loss, void *grad_or_null, int64_t M, int64_t N, int64_t K,
                              cudaStream_t stream);

/*
 * rope_cos_sin -- the RoPE segment around the K=1 matmul, in one kernel.
 *
 * Source: "Feature request: Schedule a small matmul op as a reduction (or
 * pointwise) op" (NVIDIA/Fuser issue 3646), the Mistral forward listing from
 * the bf16 inverse frequencies T3 and int64 position ids T4 to the bf16
 * output T26: the K=1 matmul T19 (one fp32 multiply per element), its
 * permute to [S, H] (T20), the pads and cat that repeat it to 2H columns
 * (T21..T23), cosf (T24) and the cast to bf16 (T26).  The page asks for this
 * segment to run without the matmul splitting it; here it is one launch with
 * the permuted layout written directly.
 *
 *   inv_freq : bf16 [H], device, 2-byte aligned.
 *   positions: int64 [S], device, 8-byte aligned (a batch of sequences is
 *              passed flattened).
 *   cos_out  : bf16 [S, 2H], device, row-major:
 *                angle[s,i] = fp32(float(inv_freq[i]) * float(positions[s]))
 *                cos_out[s, i] = cos_out[s, H + i] = bf16_rn(cosf(angle[s,i]))
 *              (float(int64) rounds to nearest; cosf is CUDA's, within 2
 *              fp32 ulp, so an element can differ from the bf16 rounding of
 *              the exact cosine by one bf16 ulp).
 *   sin_out  : bf16 [S, 2H] or NULL: the same with sinf -- the listing prints
 *              only the cosine branch; the segment's second [4096,128] output
 *              is taken to be the sine of the same angles.
 *   1 <= H, S < 2^31.  H % 8 == 0 with 16-byte aligned inv_freq and outputs
 *   takes the vectorised kernel; anything else the element-wise one.
 * The caller owns every buffer; nothing is allocated.  Host-side checks return
 * LF_ERR_NULL / LF_ERR_SHAPE / LF_ERR_ALIGN before anything is enqueued.
 */
lf_status rope_cos_sin(const void *inv_freq, const int64_t *positions, void *cos_out, void *sin_out_or_null,
                       int64_t H, int64_t S, cudaStream_t stream);

/*
 * fp8_cast_dual -- the float8 training cast, written in both layouts by one
 * kernel.
 *
 * Source: "Improve the Inductor generated kernel for the pattern of output1 =
 * pointwise(intput); output2 = transpose(output1)" (pytorch issue 130015),
 * Examples and "The issue in test_pattern1": the input times a scale,
 * clamped to the largest finite float8_e4m3fn magnitude (448), converted to
 * float8_e4m3fn, and returned both as is and as t().contiguous().t(), which
 * the page's compiler produced with a second kernel that re-reads the fp8
 * tensor.  Here the input is read once and both outputs are written from it.
 *
 *   x     : bf16 [M,K], device, row-major, 2-byte aligned.
 *   scale : fp32, ONE element, device (the page keeps it in a device tensor).
 *   out   : float8_e4m3fn [M,K], device, row-major:
 *             out[m*K + k] = e4m3(clamp(x[m,k] * scale, -448, 448))
 *           one fp32 multiply of the exact bf16 value, round-to-nearest-even
 *           to E4M3 (bit-exact).  A NaN input stays NaN (code 0x7F or 0xFF).
 *   out_t : float8_e4m3fn, the same values column-major, i.e. the [K,M]
 *           row-major array out_t[k*M + m] = out[m*K + k] (the storage of
 *           the page's tensor_fp8_t, whose strides are (1, M)).
 *   1 <= M, K < 2^31.  Any alignment is accepted; M % 16 == 0, K % 16 == 0
 *   and 16-byte aligned x, out and out_t take the vectorised kernel.
 * The caller owns all four buffers; nothing is allocated.  out and out_t
 * must not overlap each other or x.  Host-side checks return LF_ERR_NULL /
 * LF_ERR_SHAPE / LF_ERR_ALIGN (x odd) before anything is enqueued.
 */
lf_status fp8_cast_dual(const void *x, const float *scale, void *out, void *out_t,
                        int64_t M, int64_t K, cudaStream_t stream);

/*
 * gemm_nt_xent_noalloc -- the same computation and outputs as gemm_nt_xent,
 * for callers that cannot allocate device memory during the call.  The pages
 * have no counterpart to this entry point: it is an interface addition.
 *
 * Who needs it: code that runs while a CUDA graph is being captured (where
 * cudaMalloc/cudaFree are not allowed and cudaFree would synchronise the
 * device), programs whose allocator already owns all device memory (a
 * framework caching allocator, a serving engine that reserved the GPU up
 * front), and latency-critical paths that cannot take the device
 * synchronisation of a first-use allocation.  gemm_nt_xent allocates its
 * workspace on first use; this variant never calls cudaMalloc, cudaFree or
 * any allocating library routine.
 *
 * Scratch: a fixed 32 MiB device array inside the library (it holds the
 * per-tile partials, M * ceil(N/256) * 8 bytes, plus 12 * M bytes and an
 * error word).  Every GPU that loads the library keeps those 32 MiB until
 * the process exits.  A call whose scratch need exceeds 32 MiB returns
 * LF_ERR_WORKSPACE before anything is enqueued (for example M = 8192 with
 * N = 128256, a 128K vocabulary, fits; M = 16384 with N = 262144 does not).
 * Set-up: the first call made with a given device current looks up the
 * scratch's device address (cudaGetSymbolAddress) and checks the device;
 * make that first call before any stream capture begins.
 * Concurrency: every call shares the one scratch array, which keeps the last
 * call's contents; calls that overlap on the GPU (different streams, or
 * graphs replayed concurrently) race on it and must be serialised.
 * Device-side wait timeouts are not reported through lf_check_device_error:
 * a call whose device waits ran out writes NaN to every loss[m] and, when
 * grad_or_null is given, to every gradient element.  The wait limit and the
 * stall injection of lf_set_test_hooks apply to this entry point as well.
 * Arguments, layouts, preconditions and the other error codes are those of
 * gemm_nt_xent.
 */
lf_status gemm_nt_xent_noalloc(const void *x, const void *w, const int32_t *labels,
                               float *loss, void *grad_or_null,
                               int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *lf_status_string(lf_status status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns LF_ERR_DEVICE_TIMEOUT if any kernel of this library gave up
 * on a device-side wait since the last check (its outputs are then invalid),
 * LF_ERR_LAUNCH if the stream reports a CUDA error, LF_OK otherwise.
 */
lf_status lf_check_device_error(cudaStream_t stream);

/*
 * Which device-side wait gave up, for the last LF_ERR_DEVICE_TIMEOUT that
 * lf_check_device_error reported in this process (0: none yet).  The first
 * wait to give up in a launch records its code:
 *   0x101 an operand ring slot was never freed (TMA producer)
 *   0x102 an operand stage never landed (MMA issuer)
 *   0x103 an accumulator was never released by the epilogue (MMA issuer)
 *   0x104 an accumulator was never completed (epilogue)
 *   0x105 copies or MMAs did not finish while unwinding
 *   0x106 a stream-K partial never arrived (tile owner)
 *   0x107 a CTA's own stream-K partial write did not complete
 *   0x108 a one-pass group member never published its row statistics
 *   0x109 the copy of a stream-K partial into shared memory did not land
 *   0x10a a tile claimed at run time never reached one of the pair's roles
 */
int lf_last_device_wait_code(void);

/* Number of kernel launches this library has enqueued in this process (all devices). */
uint64_t lf_launch_count(void);

/*
 * The schedule of the last tensor-core GEMM launch in this process (gemm_nt,
 * gemm_layout, gemm_batched and the two-pass cross-entropy GEMMs; not the
 * one-pass cross-entropy kernel): its grid in CTAs, whether it ran on CTA
 * pairs (1) or single CTAs (0), whether the K loop was split over the pairs
 * (stream-K: 1), and the MMA's N-tile width.  All zero before the first such
 * launch.  Any pointer may be NULL.  Not synchronised with other threads'
 * launches; meant for tests and tuning.
 */
void lf_last_gemm_plan(int *grid, int *cta_pairs, int *stream_k, int *tile_n);

/*
 * Sets up the current device if needed and reports its SM count and how many
 * CTA pairs of the pair GEMM kernel can be resident at once (either pointer
 * may be NULL).  LF_ERR_ARCH on a device that is not sm_103.
 */
lf_status lf_device_query(int *num_sms, int *pair_clusters);

/*
 * Tuning knobs, applied to launches made after the call, on every device.
 *   l2_prefetch_kblocks: how many K blocks (64 columns each) ahead of its
 *     shared-memory loads each GEMM CTA prefetches its operand slices into
 *     L2; 0 disables it, a negative value restores the default (off).
 *   gemm_variant: 1 = single-CTA 128x256 tiles, 2 = CTA-pair 256x256 tiles
 *     (tcgen05 cta_group::2) by whole tiles, 3 = CTA-pair tiles with the K
 *     iterations split evenly over all pairs (stream-K), 4 = gemm_nt with the
 *     operands swapped (M <= 128; whole tiles or stream-K chosen
 *     automatically), anything else = automatic (swapped operands when M <=
 *     128 and N has fewer 256-column tiles than half the SMs; pairs when M >
 *     128 or a long K would leave most SMs idle; stream-K when it shortens
 *     each pair's run -- waves x K blocks by whole tiles against the split's
 *     even share -- by more than its fixed cost of about 32 K blocks).
 */
void lf_set_tuning(int l2_prefetch_kblocks, int gemm_variant);

/*
 * N-tile width of the one-pass cross-entropy-with-gradient kernel, applied to
 * later gemm_nt_xent calls with a gradient: 128, 160, 192, 224 or 256; any
 * other value restores the automatic choice (the width with the least rounds
 * x width among those whose group fits the resident pairs).  A forced width
 * whose group does not fit the resident pairs falls back to the two-pass path.
 */
void lf_set_onepass_tile(int width);

/*
 * How gemm_nt_xent / gemm_nt_xent_layout compute the gradient on CTA pairs
 * when N > 256 (for N <= 256 one launch always does it), applied to later
 * calls: 1 = the one-pass kernel when a row block of tiles
 * fits the resident pairs (else as 0), 2 = the exp pass and the rescale pass
 * (a GEMM whose epilogue writes the tile partials and fp16 exp(z - tile max)
 * into grad, then one kernel that merges each row's partials into lse and
 * loss and rewrites grad in place as bf16; the recompute form when a row has
 * more than 49,152 tiles of 256 columns), 3 = partials, combine and a second
 * GEMM pass that recomputes the logits to write the gradient; anything else =
 * automatic (the exp pass and the rescale pass unless a one-pass tile width is
 * forced).  The single-CTA kernel always uses the recompute form.
 */
void lf_set_xent_grad_path(int path);

/*
 * Order of whole output tiles on CTA pairs, applied to later launches: bands
 * of `m_blocks` 256-row blocks, each band sweeping every N block before the
 * next starts (M block fastest within a band, so the pairs sharing a W tile
 * run together).  0 = one band of all rows; a negative value restores the
 * automatic choice (the largest band whose X rows take at most 32 MiB, split
 * evenly).  Results do not depend on it.
 */
void lf_set_tile_band(int m_blocks);

/*
 * Assignment of whole output tiles to CTA pairs, applied to later launches:
 * 0 = fixed (pair i takes tiles i, i + pairs, ...); 1 = claimed at run time
 * (pair i starts with tile i, then each pair claims the next unclaimed tile
 * in the tile order from a counter in the library's workspace, so the pairs
 * that share a W tile start it together and faster pairs -- for instance
 * while other work holds some SMs -- take more tiles); a negative value
 * restores the automatic choice, the fixed assignment.  Each tile is computed
 * by one pair either way: results do not depend on it.
 */
void lf_set_tile_schedule(int mode);

/*
 * Test hooks (not for production use).  inject_stall = 1 makes the next
 * tensor-core GEMM launches skip the first operand load of CTA 0, so that
 * CTA's MMA wait never completes: the bounded wait then gives up after
 * wait_timeout_ns, records LF_ERR_DEVICE_TIMEOUT for lf_check_device_error()
 * and every CTA exits normally (no trap, the context stays usable).
 * wait_timeout_ns = 0 restores the default limit of 2 s.
 */
void lf_set_test_hooks(int inject_stall, uint64_t wait_timeout_ns);

/*
 * enable = 0: later launches of the kernels whose CTAs wait on each other (the
 * stream-K split, the one-pass cross-entropy) omit the cooperative launch
 * attribute; 1 (the default) restores it.  Meant for profilers that cannot
 * replay cooperative cluster launches (they serialise kernels anyway): the
 * kernels are the same, but nothing then guarantees that all their CTAs are
 * resident together when other work holds part of the GPU.
 */
void lf_set_cooperative(int enable);

/*
 * Test hook (not for production use): enqueues on `stream` a kernel of `ctas`
 * CTAs, each holding 200 KiB of shared memory -- one per SM, with no room
 * beside it for a GEMM CTA -- that wait `duration_ns` on the GPU's global
 * timer and exit.  It stands in for another application's kernels holding
 * part of the GPU, e.g. to check that the kernels whose CTAs wait on each
 * other (stream-K, the one-pass cross-entropy) are launched so that all their
 * CTAs are resident together.  1 <= ctas <= the SM count and
 * 0 < duration_ns <= 5 s, else LF_ERR_SHAPE.
 */
lf_status lf_test_occupy_sms(int ctas, uint64_t duration_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LAYOUTFOLD_H */
