/*
 * wqbmm — A16W4 per-group pseudo-quantized matmul by MSD (multi-step decomposition) on GB300 (sm_103a).
 *
 * The operation (WeightQuantBatchMatmulExperiment page, section 4.1, eleven steps; spec in section 4.2):
 *   inputs   x fp16 [M, K] row-major; w signed int4 [K, N]; antiquant_scale fp16 [K/G, N] row-major
 *   output   y fp16 [M, N] row-major
 *   for each row m and each K-group g of G consecutive k:
 *     A_max = max |x[m, k]| over the group
 *     tmp1 = 7.49 * x / A_max,       A1 = round(tmp1)
 *     tmp2 = (tmp1 - A1) * 14.98,    A2 = round(tmp2)
 *     tmp3 = (tmp2 - A2) * 14.98,    A3 = round(tmp3)        (each A_i in [-7, 7])
 *     Y_i[m, n] = sum over the group's k of A_i[m, k] * w[k, n]            (exact integers)
 *     Y_group = (Y1/7.49 + Y2/(7.49*14.98) + Y3/(7.49*14.98^2)) * A_max * antiquant_scale[g, n]
 *   y[m, n] = sum over the groups of Y_group, rounded once to fp16 (nearest-even).
 * The unfold runs in IEEE binary32 with the constants 7.49f and 14.98f, every operation rounded on its own and the
 * division correctly rounded; "round" is half-to-even. A group whose A_max is 0 contributes 0.
 * Per-channel quantization is the case G = K: one group spans each row, A_max is the row's maximum and
 * antiquant_scale (and the zero points of wqbmm_run_ex) have one row, [1, N].
 *
 * Weight format: the caller's int4 weights are packed two per byte along K (page section 4.3): uint8 [K/2, N], byte
 * (kk, n) holds w[2kk, n] in its low nibble and w[2kk+1, n] in its high nibble, two's complement. Before the first
 * run the weights are re-laid once (wqbmm_prepack_weight) into the library's tile layout, the way a size query plus
 * an ND-to-tiled transform precede a quantized matmul on the page "aclnnCalculateMatmulWeightSizeV2 接口详解"
 * (sections on the function prototype and on its cooperation with aclnnTransMatmulWeight).
 *
 * Conventions for every entry point:
 *   - All pointers are caller-owned. Pointers marked "device" must be device memory of the current CUDA device;
 *     the library allocates nothing and keeps no state beyond cached device attributes and one device status word
 *     per device (see wqbmm_read_device_status).
 *   - Work is enqueued asynchronously on `stream` (0 = the legacy default stream); the library never synchronizes,
 *     except wqbmm_read_device_status, which waits for `stream`.
 *   - Arguments are validated before anything is enqueued. On any error nothing is launched and outputs are
 *     untouched. Validation of sizes and pointers needs no GPU; the architecture check needs the current device to
 *     be compute capability 10.3.
 *   - Status codes follow the pattern of the page "aclnnCalculateMatmulWeightSizeV2 接口详解", section on return
 *     values (null pointer, invalid parameter and runtime/platform errors are distinct codes).
 */
#ifndef WQBMM_H
#define WQBMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define WQBMM_API __attribute__((visibility("default")))
#else
#define WQBMM_API
#endif

/* Same type as cudaStream_t, without requiring the CUDA headers. */
typedef struct CUstream_st *wqbmm_stream_t;

typedef enum {
    WQBMM_OK = 0,
    WQBMM_ERR_NULLPTR = 1,            /* a required pointer argument is null */
    WQBMM_ERR_INVALID = 2,            /* a size, alignment or workspace-size rule below is broken */
    WQBMM_ERR_UNSUPPORTED_ARCH = 3,   /* the current device is not compute capability 10.3 (GB300) */
    WQBMM_ERR_CUDA = 4,               /* a CUDA runtime call failed (no device, launch failure, ...) */
    WQBMM_ERR_DEVICE_TIMEOUT = 5,     /* a kernel gave up a bounded wait (read by wqbmm_read_device_status) */
    WQBMM_ERR_SCRATCH_LIMIT = 6       /* the shape needs more scratch than wqbmm_run_static_scratch holds */
} wqbmm_status;

/* Shape rules shared by the entry points that take (M, K, N, G):
 *   1 <= M, K, N <= 2^31 - 1;  G in {32, 64, 128}, or G == K with K % 32 == 0 (per channel);  K % G == 0;
 *   N % 8 == 0;  M * N, M * K < 2^62.
 * Alignment rules: x, antiquant_scale, y, the prepacked weights and the workspace start on 16-byte boundaries. */

/*
 * Size in bytes of the prepacked weight buffer for a K x N int4 weight. Host only; no GPU needed.
 * Layout (for reference; callers treat it as opaque): tiles of 128 output columns x 128 k, tile (nt, kb) at byte
 * offset (nt * ceil(K/128) + kb) * 8192; inside a tile, row r (column n = 128 nt + r) holds 64 bytes, byte 4q + b
 * (q = 0..15, b = 0..3) with k = 128 kb + 8q + b in the low nibble and k + 4 in the high nibble, each stored as w + 8
 * (offset binary, 0..15); padding holds w = 0. Total = ceil(N/128) * ceil(K/128) * 8192 bytes.
 * Errors: WQBMM_ERR_NULLPTR if bytes is null; WQBMM_ERR_INVALID if the shape rules fail.
 */
WQBMM_API wqbmm_status wqbmm_prepacked_weight_bytes(int64_t K, int64_t N, int64_t G, size_t *bytes);

/*
 * Re-lays packed int4 weights into the prepacked tile layout (one kernel launch on `stream`).
 *   w_packed     device, uint8 [K/2, N] as described above (read only)
 *   w_prepacked  device, wqbmm_prepacked_weight_bytes(K, N, G) bytes (written)
 * The two buffers must not overlap. Errors: NULLPTR, INVALID (shape or alignment), UNSUPPORTED_ARCH, CUDA.
 */
WQBMM_API wqbmm_status wqbmm_prepack_weight(const uint8_t *w_packed, void *w_prepacked, int64_t K, int64_t N,
                                            int64_t G, wqbmm_stream_t stream);

/*
 * The same for a weight stored transposed, [N, K] (the operator's transpose option for the weight, page 2 section
 * 5.4): w_packed_nk is uint8 [N, K/2], byte (n, kk) = w[2kk, n] in the low nibble and w[2kk+1, n] in the high
 * nibble (two's complement). The output is the same prepacked buffer wqbmm_prepack_weight makes from the [K/2, N]
 * form of the same weight. Errors as for wqbmm_prepack_weight.
 */
WQBMM_API wqbmm_status wqbmm_prepack_weight_nk(const uint8_t *w_packed_nk, void *w_prepacked, int64_t K, int64_t N,
                                               int64_t G, wqbmm_stream_t stream);

/*
 * Workspace bytes wqbmm_run needs for this shape on any GB300. Host only.
 * Every shape needs one: x is unfolded once per call into it. For M <= 2 it holds the planes of x as int8 (3 bytes
 * per element, K padded to a multiple of 128) and, per row and group, four floats of combine constants; for
 * 3 <= M < 64 the planes as the tensor cores' operand image (16, 32 or 48 rows of 128 bytes per row tile of up to 16
 * rows, up to 10 when G = 32, and per 128 k) and 128 floats of constants per row tile and group, then split-K
 * partial sums and per-tile
 * arrival counters (only shapes whose split over K is wider than one thread-block cluster need those); for M >= 64
 * the planes (3 bytes per element of x, rows padded to a multiple of 128) and the constants. Per channel it also
 * holds each row's A_max and, for M >= 3, the scale and zero-point rows repeated once per 128 k (or 64 or 32 when K
 * is not a multiple of 128).
 * It needs no initialisation: every run writes what it later reads (the unfold pre-pass also clears the split-K
 * arrival counters before the main kernel uses them), so a workspace can be reused by later runs on the same stream
 * in whatever state an earlier run left it, including a run that ended with WQBMM_ERR_DEVICE_TIMEOUT. Runs that
 * execute concurrently must use different workspaces.
 * Errors: NULLPTR if bytes is null; INVALID if the shape rules fail.
 */
WQBMM_API wqbmm_status wqbmm_workspace_bytes(int64_t M, int64_t K, int64_t N, int64_t G, size_t *bytes);

/*
 * y = MSD matmul of x with the prepacked weights and antiquant_scale (the eleven steps above), on `stream`.
 *   x                device, fp16 [M, K] row-major
 *   w_prepacked      device, output of wqbmm_prepack_weight for the same K, N, G
 *   antiquant_scale  device, fp16 [K/G, N] row-major
 *   y                device, fp16 [M, N] row-major (written; must not overlap the inputs or the workspace)
 *   workspace        device, at least wqbmm_workspace_bytes(M, K, N, G) bytes
 * The result is deterministic: split-K partial sums are reduced in a fixed order.
 * The kernel is launched with programmatic stream serialization: it may start while the kernel enqueued just before
 * it on `stream` is still finishing, and it reads w_prepacked and antiquant_scale before that kernel has ended (x is
 * read, and y and the workspace are written, only after it has ended). So w_prepacked and antiquant_scale must not be
 * written by an immediately preceding kernel that itself releases its dependents early (griddepcontrol.
 * launch_dependents); ordinary kernels, copies and memsets always complete before this kernel starts.
 * Errors: NULLPTR, INVALID (shape, alignment, workspace too small), UNSUPPORTED_ARCH, CUDA (launch failure).
 * A kernel that gives up a bounded internal wait records WQBMM_ERR_DEVICE_TIMEOUT in the device status word.
 */
WQBMM_API wqbmm_status wqbmm_run(const void *x, const void *w_prepacked, const void *antiquant_scale, void *y,
                                 int64_t M, int64_t K, int64_t N, int64_t G, void *workspace,
                                 size_t workspace_bytes, wqbmm_stream_t stream);

/*
 * wqbmm_run with the operator's two optional inputs (its V2 interface): asymmetric weights and a bias. The weight
 * of group g, column n stands for (w - zero_point[g, n]) * antiquant_scale[g, n], the dequantization convention of
 * the GatherDequantInt8 page ("数学语义") and of the RKNN matmul page (section 4.1.1.3.1), with zero points per
 * group and column like the scales. The planes of x do not change; step 9 becomes Y_i = A_i . W_g - zp S_i, S_i the
 * sum of plane i over the group, and bias[n] is added to the accumulated sum of step 11 before the fp16 rounding.
 *   zero_point  device, fp16 [K/G, N] row-major, or null (symmetric weights, as wqbmm_run)
 *   bias        device, fp16 [N], or null
 * Both start on 16-byte boundaries when given. Every other argument, the workspace size, the launch and the errors
 * are as for wqbmm_run (wqbmm_workspace_bytes does not depend on the optional inputs).
 */
WQBMM_API wqbmm_status wqbmm_run_ex(const void *x, const void *w_prepacked, const void *antiquant_scale,
                                    const void *zero_point, const void *bias, void *y, int64_t M, int64_t K,
                                    int64_t N, int64_t G, void *workspace, size_t workspace_bytes,
                                    wqbmm_stream_t stream);

/*
 * Measurement aid: one part of wqbmm_run_ex on its own, so that the main kernel can be timed without the pre-passes
 * that precede it. part 0 launches everything (the same as wqbmm_run_ex); part 1 only the pre-passes (the unfold of
 * x into the workspace, and for per-channel shapes the row maxima and repeated scale rows); part 2 only the main
 * kernel, which reads what part 1 (or an earlier run of the same shape and inputs on this workspace) left in the
 * workspace. A part-2 launch on a workspace that holds no such result gives an undefined y (but stays within the
 * buffers). Arguments, launch and errors as for wqbmm_run_ex; also INVALID for a part outside 0..2.
 */
WQBMM_API wqbmm_status wqbmm_run_part(const void *x, const void *w_prepacked, const void *antiquant_scale,
                                      const void *zero_point, const void *bias, void *y, int64_t M, int64_t K,
                                      int64_t N, int64_t G, void *workspace, size_t workspace_bytes, int part,
                                      wqbmm_stream_t stream);

/*
 * Int8 weights (W8; the weight dtype INT8 of the page "aclnnCalculateMatmulWeightSizeV2 接口详解"): the same eleven
 * steps with w an int8 [K, N] matrix in [-128, 127], optional zero points and bias as for wqbmm_run_ex.
 * Internally w = 16 hi + lo (hi = w >> 4, lo = w & 15) and every group becomes two int4 groups over the same
 * planes of x (weights hi with scale 16 s and zero point -1/2; weights lo - 8 with scale s and the caller's zero
 * point): s (16 (hi + 1/2) + lo - 8 - zp) = s (w - zp) exactly, so the int4 kernels compute the int8 product.
 * G in {32, 64, 128} only (not per channel); 2K must satisfy the shape rules; |antiquant_scale| < 4096 (16 s is
 * formed in fp16).
 *   wqbmm_prepacked_weight_bytes_w8  host only: ceil(N/128) * ceil(2K/128) * 8192 bytes (= K * N, padded)
 *   wqbmm_prepack_weight_w8          w8: device int8 [K, N] row-major -> prepacked tiles of the split weights
 *   wqbmm_workspace_bytes_w8         host only: the workspace wqbmm_run_w8 needs (the int4 problem's, plus x
 *                                    repeated per group [M, 2K] and the split scales and zero points)
 *   wqbmm_run_w8                     y [M, N] fp16; x, antiquant_scale [K/G, N], zero_point [K/G, N] (or null),
 *                                    bias [N] (or null) as for wqbmm_run_ex; workspace required
 * Errors as for wqbmm_prepack_weight / wqbmm_workspace_bytes / wqbmm_run_ex.
 */
WQBMM_API wqbmm_status wqbmm_prepacked_weight_bytes_w8(int64_t K, int64_t N, int64_t G, size_t *bytes);
WQBMM_API wqbmm_status wqbmm_prepack_weight_w8(const int8_t *w8, void *w_prepacked, int64_t K, int64_t N, int64_t G,
                                               wqbmm_stream_t stream);
WQBMM_API wqbmm_status wqbmm_workspace_bytes_w8(int64_t M, int64_t K, int64_t N, int64_t G, size_t *bytes);
WQBMM_API wqbmm_status wqbmm_run_w8(const void *x, const void *w_prepacked, const void *antiquant_scale,
                                    const void *zero_point, const void *bias, void *y, int64_t M, int64_t K,
                                    int64_t N, int64_t G, void *workspace, size_t workspace_bytes,
                                    wqbmm_stream_t stream);

/*
 * A batch of products with shared weights (the operator's batched x, BatchMatmul with one weight): for b in
 * [0, batch), y_b = MSD matmul of x_b with the weights, x_b = x + b * x_batch_stride (fp16 [M, K], row stride K) and
 * y_b = y + b * y_batch_stride (fp16 [M, N], row stride N); strides count elements. Rows are independent, so when
 * the batches are contiguous (x_batch_stride == M * K and y_batch_stride == M * N) this is one product of batch * M
 * rows; otherwise one product per batch item is enqueued on `stream`, all using the same workspace one after the
 * other. The workspace must hold wqbmm_workspace_bytes(batch * M, K, N, G) bytes when contiguous, else
 * wqbmm_workspace_bytes(M, K, N, G). zero_point and bias as for wqbmm_run_ex (may be null).
 * Errors as for wqbmm_run_ex; also INVALID for batch < 1, a stride smaller than one item, a stride that breaks the
 * 16-byte alignment of x_b or y_b, or a batch whose rows overflow the shape rules.
 */
WQBMM_API wqbmm_status wqbmm_run_batched(const void *x, const void *w_prepacked, const void *antiquant_scale,
                                         const void *zero_point, const void *bias, void *y, int64_t batch,
                                         int64_t M, int64_t K, int64_t N, int64_t G, int64_t x_batch_stride,
                                         int64_t y_batch_stride, void *workspace, size_t workspace_bytes,
                                         wqbmm_stream_t stream);

/*
 * Exposes steps 1-8 exactly as the run kernel computes them (for bit-exact checks).
 *   x       device, fp16 [M, K]
 *   planes  device, int8 [3, M, K]: plane i of row m at planes[(i * M + m) * K + k], values in [-7, 7]
 *   amax    device, float [M, K/G]: A_max of each row and group
 * Shape rules as above with N ignored. Errors: NULLPTR, INVALID, UNSUPPORTED_ARCH, CUDA.
 */
WQBMM_API wqbmm_status wqbmm_debug_unfold(const void *x, int64_t M, int64_t K, int64_t G, int8_t *planes,
                                          float *amax, wqbmm_stream_t stream);

/*
 * Exposes step 9 for one group g as the run kernel's tensor-core path computes it (for bit-exact checks): the
 * kernel wqbmm_run would pick for this M, restricted to the k-block that holds group g.
 *   y123       device, int32 [3, M, N]: Y_i[m, n] of group g at y123[(i * M + m) * N + n]
 *   workspace  device, wqbmm_workspace_bytes(M, K, N, G) bytes
 * 0 <= g < K/G; G in {32, 64, 128} (per-channel partials are not exposed: INVALID). Errors: NULLPTR, INVALID (also
 * a workspace too small), UNSUPPORTED_ARCH, CUDA.
 */
WQBMM_API wqbmm_status wqbmm_debug_group_partials(const void *x, const void *w_prepacked, int64_t M, int64_t K,
                                                  int64_t N, int64_t G, int64_t g, int32_t *y123, void *workspace,
                                                  size_t workspace_bytes, wqbmm_stream_t stream);

/*
 * Reads (and, if clear != 0, resets) the current device's status word after waiting for `stream`.
 * *code is 0 when no kernel of this library has recorded an error; otherwise it is WQBMM_ERR_DEVICE_TIMEOUT in the
 * low 8 bits and the site of the wait that gave up in bits 8-15.
 * There is one status word per device for the whole library (the first error recorded wins), not one per workspace
 * or stream: an error recorded by a run on another stream, or by another caller in the same process, is reported
 * here too, and clearing it clears it for every caller. Callers that share a device should agree on who reads and
 * clears it.
 * Errors: NULLPTR, CUDA.
 */
WQBMM_API wqbmm_status wqbmm_read_device_status(int32_t *code, int clear, wqbmm_stream_t stream);

/*
 * Runs one kernel that waits on a barrier nothing will complete, with the given limit in nanoseconds
 * (1e6 <= limit_ns <= 2e9). The kernel gives up, records WQBMM_ERR_DEVICE_TIMEOUT in the status word and returns, so
 * the bounded-wait error path can be checked without a hang. Errors: INVALID, UNSUPPORTED_ARCH, CUDA.
 */
WQBMM_API wqbmm_status wqbmm_debug_wait_timeout(int64_t limit_ns, wqbmm_stream_t stream);

/*
 * Same result as wqbmm_run, for callers that cannot allocate device memory: code whose device memory is owned by
 * another allocator (a framework's caching pool, a plugin interface that hands over only its input and output
 * buffers) and that therefore has no way to provide wqbmm_run's workspace. (The paper has no counterpart: this is
 * an interface convenience, not part of the method.)
 *   x, w_prepacked, antiquant_scale, y   as for wqbmm_run (caller-owned device memory)
 * Scratch: everything wqbmm_run keeps in its workspace (the unfolded planes of x and the per-row combine constants,
 * the split-K partial sums and arrival counters, the per-channel rows) lives in one statically sized device array of
 * 2 MiB (2097152 bytes) inside this library; every GPU that loads the library holds it until the process exits. A
 * shape whose workspace (as reported by wqbmm_workspace_bytes) exceeds that size is rejected with
 * WQBMM_ERR_SCRATCH_LIMIT before anything is launched. The planes take about 3 bytes per element of x (rows padded
 * to 16 below 64 rows and to 128 from 64 rows on); shapes of 3 to 63 rows with few column tiles also need split-K
 * partial sums, 4 bytes per output element and K-slice. wqbmm_workspace_bytes gives the exact figure. Shapes that
 * fit include M = 1 or 2 with K up to 65536 at any N, M = 8 with K = 4096 and N = 11008, and M = 128 with K = 5120
 * and N = 13824; prefill-sized products (thousands of rows) do not fit and must use wqbmm_run.
 * Set-up: the first call in each CUDA context of a device looks up the array's device address (with that device
 * current) and keeps it with the context, so a device reset, which makes a new context, leads to a new look-up; make
 * the first call on a device before any stream capture. Nothing is allocated by any call: no cudaMalloc, no cudaFree,
 * no allocating library routine. Each call launches the same kernels as wqbmm_run, which write everything they later
 * read, so the array's contents from earlier calls (of any shape) do not matter.
 * All calls share the one array: calls whose executions overlap on the GPU (different streams, or one device
 * used from several host threads without ordering) race on it and give wrong results. Order them on one stream.
 * Errors: NULLPTR, INVALID, UNSUPPORTED_ARCH, CUDA, SCRATCH_LIMIT.
 */
WQBMM_API wqbmm_status wqbmm_run_static_scratch(const void *x, const void *w_prepacked, const void *antiquant_scale,
                                                void *y, int64_t M, int64_t K, int64_t N, int64_t G,
                                                wqbmm_stream_t stream);

/* Static, human-readable name of a status code. */
WQBMM_API const char *wqbmm_status_string(wqbmm_status status);

#ifdef __cplusplus
}
#endif

#endif /* WQBMM_H */
