// C ABI of the A16W4 per-group MSD matmul for GB300 (declared and documented in include/wqbmm.h).
// Host code: argument validation (no GPU needed), planning (small-M fused kernel with split-K, or large-M pre-pass
// plus GEMM kernel), kernel launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>

#include "msd_gemm.cuh"
#include "msd_gemv.cuh"
#include "msd_kernels.cuh"
#include "wqbmm.h"

namespace wqbmm {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kPlanSms = 160;       // workspace sizing assumes at most this many SMs, so it needs no device
constexpr int kCtasPerSm = 2;       // shared memory (at most 110 KB) and TMEM allow two run CTAs per SM

// Which kernels of a product to launch (wqbmm_run_part): all of them, only the pre-passes, or only the main kernel.
constexpr int kPartAll = 0, kPartPre = 1, kPartMain = 2;

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int sms = 0;
    bool smem_set[6] = {false, false, false, false, false, false};   // small-M kernels: [zero points][NMMA / 16 - 1]
    bool gemm_smem_set = false;
    bool gemv_smem_set = false;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

// G is the group size the kernels work with. Per-channel quantization (the caller's G = K, one group of all K, above
// 128) runs as sub-groups of 128, 64 or 32 k with each row's A_max and the one scale (zero-point) row: the integer
// products and the combine are linear, so the sum over the sub-groups is the per-channel result.
struct Shape {
    int64_t M, K, N, G;
    bool pc = false;
};

// Device pointers of one product; zp and bias may be null. row_amax: per-channel A_max (else null);
// group_stride: elements between the scale rows of consecutive groups as the decode kernel reads them.
struct Operands {
    const void *x, *w, *scale, *zp, *bias;
    void *y;
    const float *row_amax = nullptr;
    int group_stride = 0;
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool group_size_ok(int64_t G) { return G == 32 || G == 64 || G == 128; }

wqbmm_status check_kng(int64_t K, int64_t N, int64_t G) {
    if (K < 1 || N < 1 || K > INT_MAX || N > INT_MAX) return WQBMM_ERR_INVALID;
    if (!group_size_ok(G) && !(G == K && K % 32 == 0)) return WQBMM_ERR_INVALID;     // groups, or per channel
    if (K % G != 0 || N % 8 != 0) return WQBMM_ERR_INVALID;
    if (ceil_div(K, kKBlock) > 65535) return WQBMM_ERR_INVALID;    // prepack grid.y
    return WQBMM_OK;
}

wqbmm_status check_shape(const Shape &s) {
    wqbmm_status st = check_kng(s.K, s.N, s.G);
    if (st != WQBMM_OK) return st;
    if (s.M < 1 || s.M > INT_MAX) return WQBMM_ERR_INVALID;
    if (s.M > (INT64_C(1) << 62) / s.N || s.M > (INT64_C(1) << 62) / s.K) return WQBMM_ERR_INVALID;
    return WQBMM_OK;
}

// The kernels' view of the caller's (M, K, N, G), after check_shape succeeded.
Shape kernel_shape(int64_t M, int64_t K, int64_t N, int64_t G) {
    Shape s{M, K, N, G};
    if (!group_size_ok(G)) {                            // G = K: per channel
        s.pc = true;
        s.G = K % 128 == 0 ? 128 : (K % 64 == 0 ? 64 : 32);
    }
    return s;
}

constexpr int64_t kLargeM = 64;     // from this many rows on: the pre-pass and the 128 x 128 tile GEMM (large-M path)
constexpr int64_t kGemvMaxM = kGemvMaxRows;   // up to this many rows: the dp4a matrix-vector path

// Small-M path: rows of x per CTA, the MMA N (three stacked planes padded to 16, 32 or 48 rows), the split over K.
// Large-M path: 128-row x 128-column tiles, no split.
struct Plan {
    bool large, gemv;
    int m_sub, m_tiles, n_tiles, kb_total, splits, nmma, reduce;
};

// Splits over K (only when the output tiles alone cannot fill the GPU): aim at two CTAs per SM. Up to 12 wanted
// slices become at most 8 cluster slices reduced on chip; more go through a global workspace.
Plan make_plan(const Shape &s, int sms) {
    Plan p{};
    p.n_tiles = static_cast<int>(ceil_div(s.N, kTileN));
    p.kb_total = static_cast<int>(ceil_div(s.K, kKBlock));
    if (s.M <= kGemvMaxM) {
        p.gemv = true;
        p.m_tiles = 1;
        p.m_sub = static_cast<int>(s.M);
        p.splits = 1;
        p.reduce = kReduceNone;
        return p;
    }
    if (s.M >= kLargeM) {
        p.large = true;
        p.m_tiles = static_cast<int>(ceil_div(s.M, kGemmTileM));
        p.m_sub = kGemmTileM;
        p.splits = 1;
        p.reduce = kReduceNone;
        return p;
    }
    // tiles of up to 16 rows (MMA N = 48); with G = 32 (four groups per k-block) at most 10 rows (N = 32), since
    // three 48-row accumulators are all that fit beside the converted weights in a CTA's 256 TMEM columns
    const int64_t max_rows = s.G == 32 ? 10 : 16;
    p.m_tiles = static_cast<int>(ceil_div(s.M, max_rows));
    p.m_sub = static_cast<int>(ceil_div(s.M, p.m_tiles));
    p.nmma = p.m_sub <= 5 ? 16 : (p.m_sub <= 10 ? 32 : 48);
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    const int64_t target = static_cast<int64_t>(kCtasPerSm) * sms;
    int64_t splits = 1;
    if (tiles < sms) splits = target / tiles;
    if (splits <= 12 && splits > kMaxClusterSplits) splits = kMaxClusterSplits;
    if (splits > p.kb_total) splits = p.kb_total;
    if (splits < 1) splits = 1;
    p.splits = static_cast<int>(splits);
    p.reduce = p.splits == 1 ? kReduceNone : (p.splits <= kMaxClusterSplits ? kReduceCluster : kReduceGlobal);
    return p;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Large-M workspace: the plane tiles [m_tiles][kb][3][16 KB], then the constants [m_tiles][K/G][128] (float4).
size_t planes_bytes(const Plan &p) { return static_cast<size_t>(p.m_tiles) * p.kb_total * 3 * kPlaneImageBytes; }
size_t consts_bytes(const Shape &s, const Plan &p) {
    return static_cast<size_t>(p.m_tiles) * (s.K / s.G) * kGemmTileM * kGemmConstRowBytes;
}

// Decode workspace: int8 planes [M][kb][384 B], then the constants [M][K/G] (float4).
size_t gemv_planes_bytes(const Shape &s, const Plan &p) {
    return static_cast<size_t>(s.M) * p.kb_total * kGemvPlaneBytes;
}

// Small-M workspace: the planes images [m_tiles][kb][NMMA x 128 B], the constants [m_tiles][K/G][128] (float), then,
// for a split over K wider than a cluster, the partial sums [splits][M][N] (float) and the arrival counters.
size_t small_planes_bytes(const Plan &p) {
    return static_cast<size_t>(p.m_tiles) * p.kb_total * p.nmma * kKBlock;
}
size_t small_consts_bytes(const Shape &s, const Plan &p) {
    return static_cast<size_t>(p.m_tiles) * (s.K / s.G) * kConstFloatsPerGroup * sizeof(float);
}

size_t path_workspace(const Shape &s, const Plan &p) {
    if (p.gemv) return align256(gemv_planes_bytes(s, p)) + align256(static_cast<size_t>(s.M) * (s.K / s.G) * 16);
    if (p.large) return align256(planes_bytes(p)) + align256(consts_bytes(s, p));
    const size_t unfolded = align256(small_planes_bytes(p)) + align256(small_consts_bytes(s, p));
    if (p.reduce != kReduceGlobal) return unfolded;
    return unfolded + align256(static_cast<size_t>(p.splits) * s.M * s.N * sizeof(float)) +
           align256(static_cast<size_t>(p.m_tiles) * p.n_tiles * sizeof(uint32_t));
}

// Per channel, after the path's own workspace: the rows' A_max (float [M]) and, for the paths that load scales as
// tiles, the scale and zero-point rows repeated once per sub-group (fp16 [K/G, N] each).
size_t scale_rep_bytes(const Shape &s) { return align256(static_cast<size_t>(s.K / s.G) * s.N * 2); }
size_t per_channel_workspace(const Shape &s, const Plan &p) {
    if (!s.pc) return 0;
    return align256(static_cast<size_t>(s.M) * sizeof(float)) + (p.gemv ? 0 : 2 * scale_rep_bytes(s));
}

size_t workspace_for(const Shape &s, const Plan &p) { return path_workspace(s, p) + per_channel_workspace(s, p); }

// ------------------------------------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool probed = false;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!probed) {
        probed = true;
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// Row-major fp16 matrix [rows, cols] with a box of box_rows x box_cols; zeros outside the matrix.
bool fp16_tensor_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int box_rows, int box_cols) {
    const EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Byte matrix of `rows` rows of `row_bytes` bytes (a multiple of 16, at most 64), boxes of box_rows whole rows,
// stored in shared memory with the 64-byte swizzle (16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3)).
bool u8_rows_tensor_map(CUtensorMap *map, const void *base, int64_t rows, int row_bytes, int box_rows) {
    const EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Current device must be compute capability 10.3; caches the SM count.
wqbmm_status current_device(int *dev_out, DeviceInfo **info_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WQBMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return WQBMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return WQBMM_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.sms = sms;
        d.probed = true;
    }
    if (!d.supported) return WQBMM_ERR_UNSUPPORTED_ARCH;
    *dev_out = dev;
    *info_out = &d;
    return WQBMM_OK;
}

template <int NMMA, bool kZp>
wqbmm_status launch_msd(const RunParams &rp, const Plan &plan, DeviceInfo *info, cudaStream_t stream) {
    constexpr int idx = (kZp ? 3 : 0) + NMMA / 16 - 1;
    using C = Cfg<NMMA>;
    // the converters check every TMEM accumulator of a k-block before its MMAs: they must all exist at once
    if (kKBlock / rp.G > C::kTmemBufs) return WQBMM_ERR_INVALID;
    const int smem = SmallLayout(C::kBTileBytes, C::kOffStages, rp.G, kZp).smem_bytes;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!info->smem_set[idx]) {
            // the limit covers every group size (G = 32 has the largest layout)
            int most = 0;
            for (int g : {32, 64, 128}) {
                const int b = SmallLayout(C::kBTileBytes, C::kOffStages, g, kZp).smem_bytes;
                most = b > most ? b : most;
            }
            if (cudaFuncSetAttribute(msd_kernel<NMMA, kZp>, cudaFuncAttributeMaxDynamicSharedMemorySize, most) !=
                cudaSuccess)
                return WQBMM_ERR_CUDA;
            info->smem_set[idx] = true;
        }
    }
    // weight tiles: 128 rows of 64 packed bytes per k-block, swizzled in shared memory; scale and zero-point tiles:
    // (128 / G) groups x 128 columns
    CUtensorMap tmap_w{}, tmap_s{}, tmap_z{};
    if (!u8_rows_tensor_map(&tmap_w, rp.w, static_cast<int64_t>(plan.n_tiles) * plan.kb_total * kTileN,
                            kKBlock / 2, kTileN))
        return WQBMM_ERR_CUDA;
    if (rp.dbg_group < 0 && !fp16_tensor_map(&tmap_s, rp.scale, rp.K / rp.G, rp.N, kKBlock / rp.G, kTileN))
        return WQBMM_ERR_CUDA;
    if (kZp && rp.dbg_group < 0 && !fp16_tensor_map(&tmap_z, rp.zp, rp.K / rp.G, rp.N, kKBlock / rp.G, kTileN))
        return WQBMM_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan.n_tiles, plan.m_tiles, rp.dbg_group >= 0 ? 1 : plan.splits);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // programmatic launch: this kernel may start while the unfold pre-pass finishes; it fetches only weights and
    // scales before griddepcontrol.wait (see msd_kernel)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = static_cast<unsigned>(plan.splits);
    cfg.attrs = attr;
    cfg.numAttrs = rp.reduce == kReduceCluster ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, msd_kernel<NMMA, kZp>, rp, tmap_w, tmap_s, tmap_z) != cudaSuccess)
        return WQBMM_ERR_CUDA;
    return WQBMM_OK;
}

template <bool kZp>
wqbmm_status launch_small_zp(const RunParams &rp, const Plan &plan, DeviceInfo *info, cudaStream_t stream) {
    switch (plan.nmma) {
        case 16: return launch_msd<16, kZp>(rp, plan, info, stream);
        case 32: return launch_msd<32, kZp>(rp, plan, info, stream);
        default: return launch_msd<48, kZp>(rp, plan, info, stream);
    }
}

// Small-M path: the unfold pre-pass writes the planes images and constants into the workspace, then the tensor-core
// kernel runs under programmatic launch.
wqbmm_status launch_small(const void *x, const float *row_amax, const RunParams &rp, const Plan &plan,
                          DeviceInfo *info, cudaStream_t stream, int part) {
    if (plan.m_tiles > 65535 || plan.splits > 65535) return WQBMM_ERR_INVALID;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.kb_total), static_cast<unsigned>(plan.m_tiles), 1);
    cfg.blockDim = dim3(static_cast<unsigned>(32 * (plan.nmma / 3)), 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int n_counters = rp.ws_count != nullptr ? plan.m_tiles * plan.n_tiles : 0;
    if (part != kPartMain &&
        cudaLaunchKernelEx(&cfg, unfold_small_kernel, static_cast<const __half *>(x), rp.M, rp.K, rp.G, plan.kb_total,
                           plan.m_sub, plan.nmma, const_cast<uint8_t *>(rp.planes), const_cast<float *>(rp.consts),
                           row_amax, rp.ws_count, n_counters) != cudaSuccess)
        return WQBMM_ERR_CUDA;
    if (part == kPartPre) return WQBMM_OK;
    // debug runs read no zero points (they expose the integer partials of the plain weights)
    return rp.zp != nullptr && rp.dbg_group < 0 ? launch_small_zp<true>(rp, plan, info, stream)
                                                : launch_small_zp<false>(rp, plan, info, stream);
}

// Large-M path: the unfold pre-pass writes plane tiles and constants into the workspace, then the GEMM kernel runs
// under programmatic launch (it fetches weights and scales while the pre-pass finishes).
wqbmm_status launch_large(const Shape &s, const Plan &plan, const Operands &op, void *workspace, int dbg_group,
                          int32_t *dbg_y123, DeviceInfo *info, cudaStream_t stream, int part) {
    if (plan.n_tiles > 65535) return WQBMM_ERR_INVALID;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!info->gemm_smem_set) {
            if (cudaFuncSetAttribute(msd_gemm_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kGemmSmemLimit) != cudaSuccess ||
                cudaFuncSetAttribute(msd_gemm_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kGemmSmemLimit) != cudaSuccess ||
                cudaFuncSetAttribute(msd_gemm_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kGemmSmemLimit) != cudaSuccess)
                return WQBMM_ERR_CUDA;
            // the kernel's register split assumes the launch allocation it was written for: with any other, a
            // warpgroup's claim could wait forever, so the kernel is not launched at all
            for (const void *fn : {reinterpret_cast<const void *>(msd_gemm_kernel<false, false>),
                                   reinterpret_cast<const void *>(msd_gemm_kernel<false, true>),
                                   reinterpret_cast<const void *>(msd_gemm_kernel<true, false>)}) {
                cudaFuncAttributes fa{};
                if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess || fa.numRegs != kGemmLaunchRegs)
                    return WQBMM_ERR_CUDA;
            }
            info->gemm_smem_set = true;
        }
    }
    const bool dbg = dbg_group >= 0;
    const bool zp = op.zp != nullptr && !dbg;
    uint8_t *planes = static_cast<uint8_t *>(workspace);
    float4 *consts = reinterpret_cast<float4 *>(planes + align256(planes_bytes(plan)));
    const dim3 ugrid(static_cast<unsigned>(plan.m_tiles * kGemmTileM / 8), static_cast<unsigned>(plan.kb_total));
    if (part != kPartMain) {
        unfold_planes_kernel<<<ugrid, 256, 0, stream>>>(static_cast<const __half *>(op.x), static_cast<int>(s.M),
                                                        static_cast<int>(s.K), static_cast<int>(s.G), plan.kb_total,
                                                        planes, consts, dbg_group >= 0 ? 1 : 0, op.row_amax);
        if (cudaPeekAtLastError() != cudaSuccess) return WQBMM_ERR_CUDA;
    }
    if (part == kPartPre) return WQBMM_OK;
    CUtensorMap tmap_s{}, tmap_z{};
    if (!dbg && !fp16_tensor_map(&tmap_s, op.scale, s.K / s.G, s.N, static_cast<int>(kKBlock / s.G), kGemmTileN))
        return WQBMM_ERR_CUDA;
    if (zp && !fp16_tensor_map(&tmap_z, op.zp, s.K / s.G, s.N, static_cast<int>(kKBlock / s.G), kGemmTileN))
        return WQBMM_ERR_CUDA;
    GemmParams gp{};
    gp.w = static_cast<const uint8_t *>(op.w);
    gp.planes = planes;
    gp.consts = consts;
    gp.bias = static_cast<const __half *>(op.bias);
    gp.y = static_cast<__half *>(op.y);
    gp.dbg_y123 = dbg_y123;
    gp.M = static_cast<int>(s.M);
    gp.K = static_cast<int>(s.K);
    gp.N = static_cast<int>(s.N);
    gp.G = static_cast<int>(s.G);
    gp.m_tiles = plan.m_tiles;
    gp.n_tiles = plan.n_tiles;
    gp.kb_total = plan.kb_total;
    gp.dbg_group = dbg_group;
    const GemmLayout L(gp.G, zp);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(plan.m_tiles, plan.n_tiles, 1);     // row tiles fastest: concurrent CTAs share weight tiles
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = dbg  ? cudaLaunchKernelEx(&cfg, msd_gemm_kernel<true, false>, gp, tmap_s, tmap_z)
                          : zp ? cudaLaunchKernelEx(&cfg, msd_gemm_kernel<false, true>, gp, tmap_s, tmap_z)
                               : cudaLaunchKernelEx(&cfg, msd_gemm_kernel<false, false>, gp, tmap_s, tmap_z);
    return e == cudaSuccess ? WQBMM_OK : WQBMM_ERR_CUDA;
}

// Decode path: the unfold of the one or two rows, then the dp4a matrix-vector kernel, both under programmatic launch
// (the GEMV kernel streams its weights while the unfold runs).
template <int MR, bool kDebug, bool kZp, int KB>
bool gemv_smem_attr() {
    return cudaFuncSetAttribute(msd_gemv_kernel<MR, kDebug, kZp, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(sizeof(GemvSmem<MR>))) == cudaSuccess;
}

wqbmm_status launch_gemv(const Shape &s, const Plan &plan, const Operands &op, void *workspace, int dbg_group,
                         int32_t *dbg_y123, DeviceInfo *info, cudaStream_t stream, int part) {
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!info->gemv_smem_set) {
            if (!gemv_smem_attr<1, false, false, 4>() || !gemv_smem_attr<1, false, true, 4>() ||
                !gemv_smem_attr<2, false, false, 4>() || !gemv_smem_attr<2, false, true, 4>() ||
                !gemv_smem_attr<1, false, false, 8>() || !gemv_smem_attr<1, false, true, 8>() ||
                !gemv_smem_attr<1, true, false, 8>() || !gemv_smem_attr<2, false, false, 8>() ||
                !gemv_smem_attr<2, false, true, 8>() || !gemv_smem_attr<2, true, false, 8>())
                return WQBMM_ERR_CUDA;
            info->gemv_smem_set = true;
        }
    }
    int8_t *planes = static_cast<int8_t *>(workspace);
    float4 *consts = reinterpret_cast<float4 *>(static_cast<uint8_t *>(workspace) +
                                                align256(gemv_planes_bytes(s, plan)));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(plan.kb_total, 4)), static_cast<unsigned>(s.M), 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (part != kPartMain &&
        cudaLaunchKernelEx(&cfg, gemv_unfold_kernel, static_cast<const __half *>(op.x), static_cast<int>(s.M),
                           static_cast<int>(s.K), static_cast<int>(s.G), plan.kb_total, planes, consts,
                           dbg_group >= 0 ? 1 : 0, op.row_amax) != cudaSuccess)
        return WQBMM_ERR_CUDA;
    if (part == kPartPre) return WQBMM_OK;
    GemvParams gp{};
    gp.w = static_cast<const uint8_t *>(op.w);
    gp.scale = static_cast<const __half *>(op.scale);
    gp.zp = static_cast<const __half *>(op.zp);
    gp.group_stride = op.group_stride;
    gp.bias = static_cast<const __half *>(op.bias);
    gp.planes = planes;
    gp.consts = consts;
    gp.y = static_cast<__half *>(op.y);
    gp.dbg_y123 = dbg_y123;
    gp.M = static_cast<int>(s.M);
    gp.K = static_cast<int>(s.K);
    gp.N = static_cast<int>(s.N);
    gp.G = static_cast<int>(s.G);
    gp.kb_total = plan.kb_total;
    gp.dbg_group = dbg_group;
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(s.N, kGemvCols)), 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    const bool dbg = dbg_group >= 0;
    const bool zp = op.zp != nullptr && !dbg;
    auto go = [&](auto kernel, size_t smem) {
        cfg.dynamicSmemBytes = smem;
        return cudaLaunchKernelEx(&cfg, kernel, gp);
    };
    // four k-blocks per warp and pass when one pass of eight warps covers all of K, eight otherwise (debug: eight)
    const bool one_pass = plan.kb_total <= kGemvWarps * 4;
    cudaError_t e;
    if (s.M == 1)
        e = dbg                 ? go(msd_gemv_kernel<1, true, false, 8>, sizeof(GemvSmem<1>))
            : zp && one_pass    ? go(msd_gemv_kernel<1, false, true, 4>, sizeof(GemvSmem<1>))
            : zp                ? go(msd_gemv_kernel<1, false, true, 8>, sizeof(GemvSmem<1>))
            : one_pass          ? go(msd_gemv_kernel<1, false, false, 4>, sizeof(GemvSmem<1>))
                                : go(msd_gemv_kernel<1, false, false, 8>, sizeof(GemvSmem<1>));
    else
        e = dbg                 ? go(msd_gemv_kernel<2, true, false, 8>, sizeof(GemvSmem<2>))
            : zp && one_pass    ? go(msd_gemv_kernel<2, false, true, 4>, sizeof(GemvSmem<2>))
            : zp                ? go(msd_gemv_kernel<2, false, true, 8>, sizeof(GemvSmem<2>))
            : one_pass          ? go(msd_gemv_kernel<2, false, false, 4>, sizeof(GemvSmem<2>))
                                : go(msd_gemv_kernel<2, false, false, 8>, sizeof(GemvSmem<2>));
    return e == cudaSuccess ? WQBMM_OK : WQBMM_ERR_CUDA;
}

// Launches one product (or, with dbg_group >= 0, the integer partials of one group) planned by `plan` on the current
// device. `workspace` holds workspace_for(shape, plan) bytes, in any state: every kernel writes what it later reads.
// Per channel: each row's A_max and (for the paths that load scale tiles) the repeated scale and zero-point rows,
// into the workspace after the path's own part, by one kernel under programmatic launch.
wqbmm_status per_channel_prep(const Shape &s, const Plan &plan, Operands *op, void *workspace, cudaStream_t stream,
                              bool launch) {
    uint8_t *base = static_cast<uint8_t *>(workspace) + path_workspace(s, plan);
    float *row_amax = reinterpret_cast<float *>(base);
    __half *scale_rep = nullptr, *zp_rep = nullptr;
    if (!plan.gemv) {
        scale_rep = reinterpret_cast<__half *>(base + align256(static_cast<size_t>(s.M) * sizeof(float)));
        if (op->zp != nullptr) zp_rep = reinterpret_cast<__half *>(reinterpret_cast<uint8_t *>(scale_rep) +
                                                                   scale_rep_bytes(s));
    }
    const int reps = static_cast<int>(s.K / s.G);
    const int copy_blocks =
        plan.gemv ? 0 : static_cast<int>(std::min<int64_t>(ceil_div(int64_t(reps) * s.N, 256), 1024));
    if (s.M + copy_blocks > INT_MAX) return WQBMM_ERR_INVALID;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(s.M + copy_blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (launch &&
        cudaLaunchKernelEx(&cfg, per_channel_prep_kernel, static_cast<const __half *>(op->x), static_cast<int>(s.M),
                           static_cast<int>(s.K), row_amax, static_cast<const __half *>(op->scale),
                           static_cast<const __half *>(op->zp), static_cast<int>(s.N), reps, scale_rep,
                           zp_rep) != cudaSuccess)
        return WQBMM_ERR_CUDA;
    op->row_amax = row_amax;
    if (!plan.gemv) {
        op->scale = scale_rep;
        if (op->zp != nullptr) op->zp = zp_rep;
    }
    op->group_stride = 0;                               // the decode kernel reads the one scale row for every group
    return WQBMM_OK;
}

wqbmm_status dispatch(const Operands &op_in, const Shape &s, const Plan &plan, void *workspace, int dbg_group,
                      int32_t *dbg_y123, DeviceInfo *info, cudaStream_t stream, int part = kPartAll) {
    Operands op = op_in;
    op.group_stride = static_cast<int>(s.N);
    if (s.pc) {
        const wqbmm_status st = per_channel_prep(s, plan, &op, workspace, stream, part != kPartMain);
        if (st != WQBMM_OK) return st;
    }
    if (plan.gemv) return launch_gemv(s, plan, op, workspace, dbg_group, dbg_y123, info, stream, part);
    if (plan.large) return launch_large(s, plan, op, workspace, dbg_group, dbg_y123, info, stream, part);
    RunParams rp{};
    rp.planes = static_cast<const uint8_t *>(workspace);
    rp.consts = reinterpret_cast<const float *>(static_cast<uint8_t *>(workspace) + align256(small_planes_bytes(plan)));
    rp.w = static_cast<const uint8_t *>(op.w);
    rp.scale = static_cast<const __half *>(op.scale);
    rp.zp = static_cast<const __half *>(op.zp);
    rp.bias = static_cast<const __half *>(op.bias);
    rp.y = static_cast<__half *>(op.y);
    rp.dbg_y123 = dbg_y123;
    if (plan.reduce == kReduceGlobal) {
        uint8_t *part = static_cast<uint8_t *>(workspace) + align256(small_planes_bytes(plan)) +
                        align256(small_consts_bytes(s, plan));
        const size_t counters_at = align256(static_cast<size_t>(plan.splits) * s.M * s.N * sizeof(float));
        rp.ws_part = reinterpret_cast<float *>(part);
        rp.ws_count = reinterpret_cast<uint32_t *>(part + counters_at);     // cleared by the unfold pre-pass
    }
    rp.M = static_cast<int>(s.M);
    rp.K = static_cast<int>(s.K);
    rp.N = static_cast<int>(s.N);
    rp.G = static_cast<int>(s.G);
    rp.m_sub = plan.m_sub;
    rp.n_tiles = plan.n_tiles;
    rp.m_tiles = plan.m_tiles;
    rp.splits = plan.splits;
    rp.kb_total = plan.kb_total;
    rp.reduce = plan.reduce;
    rp.dbg_group = dbg_group;
    return launch_small(op.x, op.row_amax, rp, plan, info, stream, part);
}

// Scratch for wqbmm_run_static_scratch: a fixed device array instead of a caller workspace. Host code must not
// pass the symbol itself to a kernel (on the host it only names a stand-in); the device address of this array is
// looked up with cudaGetSymbolAddress, with the device current, on the first call in each CUDA context of a device,
// and kept with that context: after a device reset the runtime makes a new context (and loads the module again), so
// the next call sees another context and looks the address up again.
constexpr size_t kStaticScratchBytes = size_t(2) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

struct ScratchAddress {
    CUcontext ctx = nullptr;
    void *addr = nullptr;
};
ScratchAddress g_scratch_addr[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static bool probed = false;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!probed) {
        probed = true;
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    }
    return fn;
}

// Device address of g_static_scratch on `dev` (the current device) in the current context.
wqbmm_status static_scratch_address(int dev, void **addr) {
    const CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    if (!get_ctx) return WQBMM_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return WQBMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchAddress &c = g_scratch_addr[dev];
    if (ctx == nullptr || ctx != c.ctx || c.addr == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return WQBMM_ERR_CUDA;
        if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return WQBMM_ERR_CUDA;   // the lookup made it current
        c.ctx = ctx;
        c.addr = p;
    }
    *addr = c.addr;
    return WQBMM_OK;
}

// Int8 weights run as an int4 problem with 2K rows (see prepack_w8_kernel): shape checks of both problems.
wqbmm_status check_w8(int64_t K, int64_t N, int64_t G) {
    if (!group_size_ok(G)) return WQBMM_ERR_INVALID;    // groups only: the two halves of a group need two scales
    if (K < 1 || K > INT_MAX / 2) return WQBMM_ERR_INVALID;
    const wqbmm_status st = check_kng(K, N, G);
    return st != WQBMM_OK ? st : check_kng(2 * K, N, G);
}

// Layout of the int8 path's workspace: the int4 problem's own, then x2 [M, 2K], scale2 and zp2 [2 K/G, N].
struct W8Workspace {
    size_t path, x2, scale2, total;
    W8Workspace(const Shape &s2, const Plan &plan) {
        path = workspace_for(s2, plan);
        x2 = align256(static_cast<size_t>(s2.M) * s2.K * 2);
        scale2 = align256(static_cast<size_t>(s2.K / s2.G) * s2.N * 2);
        total = path + x2 + 2 * scale2;
    }
};

wqbmm_status prepack(const uint8_t *w_packed, void *w_prepacked, int64_t K, int64_t N, int64_t G, bool nk,
                     wqbmm_stream_t stream) {
    if (!w_packed || !w_prepacked) return WQBMM_ERR_NULLPTR;
    wqbmm_status st = check_kng(K, N, G);
    if (st != WQBMM_OK) return st;
    if (!aligned16(w_prepacked)) return WQBMM_ERR_INVALID;
    int dev;
    DeviceInfo *info;
    if ((st = current_device(&dev, &info)) != WQBMM_OK) return st;
    const dim3 grid(static_cast<unsigned>(ceil_div(N, kTileN)), static_cast<unsigned>(ceil_div(K, kKBlock)));
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *out = static_cast<uint8_t *>(w_prepacked);
    const int kb_total = static_cast<int>(ceil_div(K, kKBlock));
    if (nk)
        prepack_kernel<true><<<grid, 256, 0, s>>>(w_packed, out, static_cast<int>(K), static_cast<int>(N), kb_total);
    else
        prepack_kernel<false><<<grid, 256, 0, s>>>(w_packed, out, static_cast<int>(K), static_cast<int>(N), kb_total);
    return cudaPeekAtLastError() == cudaSuccess ? WQBMM_OK : WQBMM_ERR_CUDA;
}

}  // namespace
}  // namespace wqbmm

using namespace wqbmm;

extern "C" {

const char *wqbmm_status_string(wqbmm_status status) {
    switch (status) {
        case WQBMM_OK: return "WQBMM_OK";
        case WQBMM_ERR_NULLPTR: return "WQBMM_ERR_NULLPTR: a required pointer is null";
        case WQBMM_ERR_INVALID: return "WQBMM_ERR_INVALID: size, alignment or workspace rule broken";
        case WQBMM_ERR_UNSUPPORTED_ARCH: return "WQBMM_ERR_UNSUPPORTED_ARCH: device is not compute capability 10.3";
        case WQBMM_ERR_CUDA: return "WQBMM_ERR_CUDA: a CUDA runtime call failed";
        case WQBMM_ERR_DEVICE_TIMEOUT: return "WQBMM_ERR_DEVICE_TIMEOUT: a kernel gave up a bounded wait";
        case WQBMM_ERR_SCRATCH_LIMIT:
            return "WQBMM_ERR_SCRATCH_LIMIT: the shape needs more than the 2 MiB static scratch";
    }
    return "WQBMM_ERR_UNKNOWN";
}

wqbmm_status wqbmm_prepacked_weight_bytes(int64_t K, int64_t N, int64_t G, size_t *bytes) {
    if (!bytes) return WQBMM_ERR_NULLPTR;
    const wqbmm_status st = check_kng(K, N, G);
    if (st != WQBMM_OK) return st;
    *bytes = static_cast<size_t>(ceil_div(N, kTileN)) * ceil_div(K, kKBlock) * kPackedTileBytes;
    return WQBMM_OK;
}

wqbmm_status wqbmm_prepack_weight(const uint8_t *w_packed, void *w_prepacked, int64_t K, int64_t N, int64_t G,
                                  wqbmm_stream_t stream) {
    return prepack(w_packed, w_prepacked, K, N, G, false, stream);
}

wqbmm_status wqbmm_prepack_weight_nk(const uint8_t *w_packed_nk, void *w_prepacked, int64_t K, int64_t N, int64_t G,
                                     wqbmm_stream_t stream) {
    return prepack(w_packed_nk, w_prepacked, K, N, G, true, stream);
}

wqbmm_status wqbmm_prepacked_weight_bytes_w8(int64_t K, int64_t N, int64_t G, size_t *bytes) {
    if (!bytes) return WQBMM_ERR_NULLPTR;
    const wqbmm_status st = check_w8(K, N, G);
    if (st != WQBMM_OK) return st;
    *bytes = static_cast<size_t>(ceil_div(N, kTileN)) * ceil_div(2 * K, kKBlock) * kPackedTileBytes;
    return WQBMM_OK;
}

wqbmm_status wqbmm_prepack_weight_w8(const int8_t *w8, void *w_prepacked, int64_t K, int64_t N, int64_t G,
                                     wqbmm_stream_t stream) {
    if (!w8 || !w_prepacked) return WQBMM_ERR_NULLPTR;
    wqbmm_status st = check_w8(K, N, G);
    if (st != WQBMM_OK) return st;
    if (!aligned16(w_prepacked)) return WQBMM_ERR_INVALID;
    int dev;
    DeviceInfo *info;
    if ((st = current_device(&dev, &info)) != WQBMM_OK) return st;
    const int kb2 = static_cast<int>(ceil_div(2 * K, kKBlock));
    const dim3 grid(static_cast<unsigned>(ceil_div(N, kTileN)), static_cast<unsigned>(kb2));
    prepack_w8_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        w8, static_cast<uint8_t *>(w_prepacked), static_cast<int>(K), static_cast<int>(N), static_cast<int>(G), kb2);
    return cudaPeekAtLastError() == cudaSuccess ? WQBMM_OK : WQBMM_ERR_CUDA;
}

wqbmm_status wqbmm_workspace_bytes_w8(int64_t M, int64_t K, int64_t N, int64_t G, size_t *bytes) {
    if (!bytes) return WQBMM_ERR_NULLPTR;
    wqbmm_status st = check_w8(K, N, G);
    if (st != WQBMM_OK) return st;
    if ((st = check_shape(Shape{M, 2 * K, N, G})) != WQBMM_OK) return st;
    const Shape s2 = kernel_shape(M, 2 * K, N, G);
    *bytes = W8Workspace(s2, make_plan(s2, kPlanSms)).total;
    return WQBMM_OK;
}

wqbmm_status wqbmm_run_w8(const void *x, const void *w_prepacked, const void *antiquant_scale,
                          const void *zero_point, const void *bias, void *y, int64_t M, int64_t K, int64_t N,
                          int64_t G, void *workspace, size_t workspace_bytes, wqbmm_stream_t stream) {
    if (!x || !w_prepacked || !antiquant_scale || !y) return WQBMM_ERR_NULLPTR;
    wqbmm_status st = check_w8(K, N, G);
    if (st != WQBMM_OK) return st;
    if ((st = check_shape(Shape{M, 2 * K, N, G})) != WQBMM_OK) return st;
    if (!aligned16(x) || !aligned16(w_prepacked) || !aligned16(antiquant_scale) || !aligned16(y) ||
        !aligned16(zero_point) || !aligned16(bias))
        return WQBMM_ERR_INVALID;
    if (!workspace) return WQBMM_ERR_NULLPTR;
    if (!aligned16(workspace)) return WQBMM_ERR_INVALID;
    int dev;
    DeviceInfo *info;
    if ((st = current_device(&dev, &info)) != WQBMM_OK) return st;
    const Shape s2 = kernel_shape(M, 2 * K, N, G);
    const Plan plan = make_plan(s2, info->sms < kPlanSms ? info->sms : kPlanSms);
    const W8Workspace L(s2, plan);
    if (workspace_bytes < L.total) return WQBMM_ERR_INVALID;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    __half *x2 = reinterpret_cast<__half *>(ws + L.path);
    __half *scale2 = reinterpret_cast<__half *>(ws + L.path + L.x2);
    __half *zp2 = reinterpret_cast<__half *>(ws + L.path + L.x2 + L.scale2);
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    const int64_t work = std::max<int64_t>(M * 2 * K / 8, (K / G) * N);
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(ceil_div(work, 256), 4096)), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = cs;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, w8_prep_kernel, static_cast<const __half *>(x), static_cast<int>(M),
                           static_cast<int>(K), static_cast<int>(G), static_cast<const __half *>(antiquant_scale),
                           static_cast<const __half *>(zero_point), static_cast<int>(N), x2, scale2,
                           zp2) != cudaSuccess)
        return WQBMM_ERR_CUDA;
    const Operands op{x2, w_prepacked, scale2, zp2, bias, y};
    return dispatch(op, s2, plan, workspace, -1, nullptr, info, cs);
}

wqbmm_status wqbmm_workspace_bytes(int64_t M, int64_t K, int64_t N, int64_t G, size_t *bytes) {
    if (!bytes) return WQBMM_ERR_NULLPTR;
    const wqbmm_status st = check_shape(Shape{M, K, N, G});
    if (st != WQBMM_OK) return st;
    const Shape s = kernel_shape(M, K, N, G);
    *bytes = workspace_for(s, make_plan(s, kPlanSms));
    return WQBMM_OK;
}

wqbmm_status wqbmm_run(const void *x, const void *w_prepacked, const void *antiquant_scale, void *y, int64_t M,
                       int64_t K, int64_t N, int64_t G, void *workspace, size_t workspace_bytes,
                       wqbmm_stream_t stream) {
    return wqbmm_run_ex(x, w_prepacked, antiquant_scale, nullptr, nullptr, y, M, K, N, G, workspace, workspace_bytes,
                        stream);
}

wqbmm_status wqbmm_run_ex(const void *x, const void *w_prepacked, const void *antiquant_scale,
                          const void *zero_point, const void *bias, void *y, int64_t M, int64_t K, int64_t N,
                          int64_t G, void *workspace, size_t workspace_bytes, wqbmm_stream_t stream) {
    return wqbmm_run_part(x, w_prepacked, antiquant_scale, zero_point, bias, y, M, K, N, G, workspace,
                          workspace_bytes, kPartAll, stream);
}

wqbmm_status wqbmm_run_part(const void *x, const void *w_prepacked, const void *antiquant_scale,
                            const void *zero_point, const void *bias, void *y, int64_t M, int64_t K, int64_t N,
                            int64_t G, void *workspace, size_t workspace_bytes, int part, wqbmm_stream_t stream) {
    if (!x || !w_prepacked || !antiquant_scale || !y) return WQBMM_ERR_NULLPTR;
    if (part != kPartAll && part != kPartPre && part != kPartMain) return WQBMM_ERR_INVALID;
    wqbmm_status st = check_shape(Shape{M, K, N, G});
    if (st != WQBMM_OK) return st;
    const Shape s = kernel_shape(M, K, N, G);
    if (!aligned16(x) || !aligned16(w_prepacked) || !aligned16(antiquant_scale) || !aligned16(y) ||
        !aligned16(zero_point) || !aligned16(bias))
        return WQBMM_ERR_INVALID;
    // the plan for this device never needs more workspace than wqbmm_workspace_bytes reports
    if (workspace_for(s, make_plan(s, kPlanSms)) > 0 && !workspace) return WQBMM_ERR_NULLPTR;
    if (workspace && !aligned16(workspace)) return WQBMM_ERR_INVALID;
    int dev;
    DeviceInfo *info;
    if ((st = current_device(&dev, &info)) != WQBMM_OK) return st;
    const Plan plan = make_plan(s, info->sms < kPlanSms ? info->sms : kPlanSms);
    if (workspace_bytes < workspace_for(s, plan)) return WQBMM_ERR_INVALID;
    const Operands op{x, w_prepacked, antiquant_scale, zero_point, bias, y};
    return dispatch(op, s, plan, workspace, -1, nullptr, info, reinterpret_cast<cudaStream_t>(stream), part);
}

wqbmm_status wqbmm_run_batched(const void *x, const void *w_prepacked, const void *antiquant_scale,
                               const void *zero_point, const void *bias, void *y, int64_t batch, int64_t M,
                               int64_t K, int64_t N, int64_t G, int64_t x_batch_stride, int64_t y_batch_stride,
                               void *workspace, size_t workspace_bytes, wqbmm_stream_t stream) {
    if (!x || !w_prepacked || !antiquant_scale || !y) return WQBMM_ERR_NULLPTR;
    if (batch < 1 || M < 1 || K < 1 || N < 1) return WQBMM_ERR_INVALID;
    if (M > INT64_MAX / K || M > INT64_MAX / N) return WQBMM_ERR_INVALID;
    if (x_batch_stride < M * K || y_batch_stride < M * N) return WQBMM_ERR_INVALID;
    if (x_batch_stride % 8 != 0 || y_batch_stride % 8 != 0) return WQBMM_ERR_INVALID;   // 16-byte alignment
    if (x_batch_stride == M * K && y_batch_stride == M * N) {
        if (M > INT64_MAX / batch) return WQBMM_ERR_INVALID;
        return wqbmm_run_ex(x, w_prepacked, antiquant_scale, zero_point, bias, y, batch * M, K, N, G, workspace,
                            workspace_bytes, stream);
    }
    if (batch - 1 > INT64_MAX / x_batch_stride / 2 || batch - 1 > INT64_MAX / y_batch_stride / 2)
        return WQBMM_ERR_INVALID;
    // validate the shape once before enqueuing anything
    wqbmm_status st = check_shape(Shape{M, K, N, G});
    if (st != WQBMM_OK) return st;
    for (int64_t b = 0; b < batch; ++b) {
        st = wqbmm_run_ex(static_cast<const __half *>(x) + b * x_batch_stride, w_prepacked, antiquant_scale,
                          zero_point, bias, static_cast<__half *>(y) + b * y_batch_stride, M, K, N, G, workspace,
                          workspace_bytes, stream);
        if (st != WQBMM_OK) return st;
    }
    return WQBMM_OK;
}

wqbmm_status wqbmm_run_static_scratch(const void *x, const void *w_prepacked, const void *antiquant_scale, void *y,
                                      int64_t M, int64_t K, int64_t N, int64_t G, wqbmm_stream_t stream) {
    if (!x || !w_prepacked || !antiquant_scale || !y) return WQBMM_ERR_NULLPTR;
    wqbmm_status st = check_shape(Shape{M, K, N, G});
    if (st != WQBMM_OK) return st;
    const Shape s = kernel_shape(M, K, N, G);
    if (!aligned16(x) || !aligned16(w_prepacked) || !aligned16(antiquant_scale) || !aligned16(y))
        return WQBMM_ERR_INVALID;
    int dev;
    DeviceInfo *info;
    if ((st = current_device(&dev, &info)) != WQBMM_OK) return st;
    const Plan plan = make_plan(s, info->sms < kPlanSms ? info->sms : kPlanSms);
    const size_t need = workspace_for(s, plan);
    if (need > kStaticScratchBytes) return WQBMM_ERR_SCRATCH_LIMIT;
    void *base = nullptr;
    if (need > 0 && (st = static_scratch_address(dev, &base)) != WQBMM_OK) return st;
    // the array keeps whatever the previous call (of any shape) left there; as with a caller's workspace, every
    // kernel writes what it later reads (the unfold pre-pass also clears the split-K counters)
    const Operands op{x, w_prepacked, antiquant_scale, nullptr, nullptr, y};
    return dispatch(op, s, plan, base, -1, nullptr, info, reinterpret_cast<cudaStream_t>(stream));
}

wqbmm_status wqbmm_debug_unfold(const void *x, int64_t M, int64_t K, int64_t G, int8_t *planes, float *amax,
                                wqbmm_stream_t stream) {
    if (!x || !planes || !amax) return WQBMM_ERR_NULLPTR;
    wqbmm_status st = check_shape(Shape{M, K, 8, G});
    if (st != WQBMM_OK) return st;
    const Shape s = kernel_shape(M, K, 8, G);
    if (!aligned16(x)) return WQBMM_ERR_INVALID;
    int dev;
    DeviceInfo *info;
    if ((st = current_device(&dev, &info)) != WQBMM_OK) return st;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (s.pc) {
        // per channel: amax receives each row's A_max (one group per row), which the unfold then reads
        per_channel_prep_kernel<<<static_cast<unsigned>(M), 256, 0, cs>>>(static_cast<const __half *>(x),
                                                                          static_cast<int>(M), static_cast<int>(K),
                                                                          amax, nullptr, nullptr, 8, 0, nullptr,
                                                                          nullptr);
        if (cudaPeekAtLastError() != cudaSuccess) return WQBMM_ERR_CUDA;
    }
    constexpr int kWarps = 4;
    const dim3 grid(static_cast<unsigned>(M), static_cast<unsigned>(ceil_div(ceil_div(K, kKBlock), kWarps)));
    unfold_debug_kernel<<<grid, kWarps * 32, 0, cs>>>(static_cast<const __half *>(x), static_cast<int>(M),
                                                      static_cast<int>(K), static_cast<int>(s.G), planes,
                                                      s.pc ? nullptr : amax, s.pc ? amax : nullptr);
    return cudaPeekAtLastError() == cudaSuccess ? WQBMM_OK : WQBMM_ERR_CUDA;
}

wqbmm_status wqbmm_debug_group_partials(const void *x, const void *w_prepacked, int64_t M, int64_t K, int64_t N,
                                        int64_t G, int64_t g, int32_t *y123, void *workspace, size_t workspace_bytes,
                                        wqbmm_stream_t stream) {
    if (!x || !w_prepacked || !y123) return WQBMM_ERR_NULLPTR;
    const Shape s{M, K, N, G};
    wqbmm_status st = check_shape(s);
    if (st != WQBMM_OK) return st;
    if (!group_size_ok(G)) return WQBMM_ERR_INVALID;     // per channel (G = K > 128): not exposed
    if (g < 0 || g >= K / G) return WQBMM_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w_prepacked)) return WQBMM_ERR_INVALID;
    if (workspace && !aligned16(workspace)) return WQBMM_ERR_INVALID;
    if (!workspace) return WQBMM_ERR_NULLPTR;            // every path unfolds x into the workspace
    if ((M >= kLargeM || M <= kGemvMaxM) &&              // these plans do not depend on the SM count
        workspace_bytes < workspace_for(s, make_plan(s, kPlanSms)))
        return WQBMM_ERR_INVALID;
    int dev;
    DeviceInfo *info;
    if ((st = current_device(&dev, &info)) != WQBMM_OK) return st;
    Plan plan = make_plan(s, info->sms < kPlanSms ? info->sms : kPlanSms);
    if (!plan.large && !plan.gemv) {                    // the group's own k-block only, no split
        plan.splits = 1;
        plan.reduce = kReduceNone;
    }
    if (workspace_bytes < workspace_for(s, plan)) return WQBMM_ERR_INVALID;
    const Operands op{x, w_prepacked, nullptr, nullptr, nullptr, nullptr};
    return dispatch(op, s, plan, workspace, static_cast<int>(g), y123, info, reinterpret_cast<cudaStream_t>(stream));
}

wqbmm_status wqbmm_read_device_status(int32_t *code, int clear, wqbmm_stream_t stream) {
    if (!code) return WQBMM_ERR_NULLPTR;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t host = 0;
    if (cudaMemcpyFromSymbolAsync(&host, g_status_word, sizeof(host), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return WQBMM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return WQBMM_ERR_CUDA;
    if (clear) {
        const int32_t zero = 0;
        if (cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
                cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return WQBMM_ERR_CUDA;
    }
    *code = host;
    return WQBMM_OK;
}

wqbmm_status wqbmm_debug_wait_timeout(int64_t limit_ns, wqbmm_stream_t stream) {
    if (limit_ns < 1000000 || limit_ns > 2000000000) return WQBMM_ERR_INVALID;
    int dev;
    DeviceInfo *info;
    wqbmm_status st = current_device(&dev, &info);
    if (st != WQBMM_OK) return st;
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(limit_ns));
    return cudaPeekAtLastError() == cudaSuccess ? WQBMM_OK : WQBMM_ERR_CUDA;
}

}  // extern "C"
