// Device code of the A16W4 per-group MSD matmul (WeightQuantBatchMatmulExperiment page, section 4.1).
//
// Kernels:
//   prepack_kernel      packed int4 [K/2, N] -> 128x128 tiles, output-column-major, offset-binary nibbles
//   unfold_debug_kernel steps 1-8 to global memory (int8 planes, float A_max), same arithmetic as the run kernel
//   per_channel_prep_kernel  per-channel quantization (one group of all K): each row's A_max, and the scale and
//                       zero-point rows repeated once per 128-k sub-group for the kernels that load them as tiles
//   unfold_small_kernel steps 1-8 once per (row tile, 128 k): the three planes as E4M3 bytes in the MMA's B operand
//                       image (NMMA rows x 128 k, 128-byte swizzle), and per (row, group) the combine constants
//   msd_kernel<NMMA>    steps 9-11: per CTA one 128-column tile of y, a tile of rows and a K-slice
//   wait_timeout_kernel a bounded wait that nothing completes (exercises the timeout path)
//
// The run kernel computes the swapped product D^T = W^T . A_int^T on the 5th-generation tensor core: the MMA's
// M side is 128 weight columns (so TMEM lane = output column n), its N side is the three stacked residual planes
// of the row tile (NMMA = 16, 32 or 48 stacked rows), one MMA chain per K-group restarted at every group so the
// integer partial sums stay exact in FP32. x is unfolded once by the pre-pass, not once per column tile. Roles
// inside a CTA (320 threads):
//   warp 0      TMA producer: per 128 k, a 2-D tensor copy of the packed weight tile (128 rows of 64 bytes, 64-byte
//               swizzle), bulk copies of the planes image and of the constants, and 2-D tensor copies of the scale
//               (and zero-point) tile, into a ring of load stages
//   warp 1      TMEM owner and single-thread MMA issuer (tcgen05.mma kind::f8f6f4, E4M3 x E4M3 -> F32): A = the
//               converted weights in tensor memory, B = the planes read in place in the load stage
//   warps 2-5   converters: per k-block, each thread turns its weight column's 64 packed bytes (offset binary)
//               into 128 E4M3 bytes in registers and stores them with tcgen05.st into one of two TMEM A slots
//   warps 6-9   epilogue: per K-group, TMEM -> registers, Y_i = D_i - 8 S_i folded into the combine, scale,
//               accumulate; the load stage is released once its constants and scales are read
// Split-K (when there are too few column tiles to fill the GPU): up to 8 K-slices of a tile form a thread-block
// cluster and reduce through distributed shared memory; more slices reduce through a global workspace. Either way
// the slices are summed in slice order, so the result does not depend on timing.
// Weights are stored as u = w + 8 in [0, 15] so that the int4 -> E4M3 conversion is two byte permutes and an OR;
// the MMA then yields D_i = sum A_i u = Y_i + 8 S_i with S_i = sum A_i over the group, removed in the combine.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace wqbmm {

constexpr int kTileN = 128;                          // output columns per CTA (MMA M)
constexpr int kKBlock = 128;                         // k per pipeline stage (one 128-byte E4M3 swizzle row)
constexpr int kPackedTileBytes = kTileN * kKBlock / 2;  // 8192
constexpr int kASlots = 2;                           // converted weight tiles (TMEM A operands) in flight
constexpr int kACols = kKBlock / 4;                  // TMEM columns of one converted tile: 4 E4M3 bytes per column
constexpr int kMaxTmemBufs = 8;                      // TMEM accumulators (one per K-group) in flight, at most
constexpr int kSmemBudget = 110 * 1024;              // per CTA, so that two CTAs share an SM
constexpr int kThreads = 320;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kConvWarp0 = 2;                        // warps 2-5 expand the weights
constexpr int kNumConvWarps = 4;
constexpr int kConvThreads = kNumConvWarps * 32;
constexpr int kEpiWarp0 = 6;                         // warps 6-9: the epilogue, one warp per TMEM lane quarter
constexpr int kNumEpiWarps = 4;
constexpr int kEpiThreads = kNumEpiWarps * 32;
constexpr int kEpiBarrierId = 1;                     // named barrier among the epilogue warps
constexpr int kOperandBarrier0 = 2;                  // named barriers 2, 3: converted weight slot 0, 1 ready
constexpr int kOperandThreads = kConvThreads + 32;   // the converters and the MMA warp
constexpr int kConstFloatsPerGroup = 16 * 8;          // 16 rows x {c1 c2 c3 corr, S1 S2 S3 0}

// Method constants (page section 4.1): unfold factors and the combine weights 1/7.49, 1/(7.49*14.98), ...
constexpr float kF1 = 7.49f;
constexpr float kF2 = 14.98f;
constexpr float kC1 = static_cast<float>(1.0 / 7.49);
constexpr float kC2 = static_cast<float>(1.0 / (7.49 * 14.98));
constexpr float kC3 = static_cast<float>(1.0 / (7.49 * 14.98 * 14.98));

// Wait-site ids recorded with a timeout (4 is no longer used: the MMA warps wait only on named barriers)
enum WaitSite : int {
    kSiteProducerEmpty = 1,     // a load stage to be released
    kSiteConvFull = 2,          // a load stage to land
    kSiteConvEmpty = 3,         // a converted-weight slot (or TMEM slot, large M) to be free
    kSiteTmemEmpty = 5,         // a TMEM accumulator to be read by the epilogue
    kSiteEpiOperandsEmpty = 6,  // the epilogue's constants and scales
    kSiteEpiTmemFull = 7,       // a TMEM accumulator to be written
    kSiteDebugWait = 9,
};

constexpr int kReduceNone = 0, kReduceCluster = 1, kReduceGlobal = 2;
constexpr int kMaxClusterSplits = 8;

template <int NMMA>
struct Cfg {
    static_assert(NMMA == 16 || NMMA == 32 || NMMA == 48, "MMA N must be 16, 32 or 48");
    static constexpr int kMaxM = NMMA / 3;                         // rows of x per CTA (plane stride in B rows)
    static constexpr int kRowsPerWarp = kMaxM;                     // one epilogue warp per TMEM lane quarter
    static constexpr int kBufStride = NMMA <= 16 ? 16 : (NMMA <= 32 ? 32 : 64);   // TMEM columns per buffer
    // the accumulators and the two converted-weight slots share 256 columns, so that two CTAs fit in TMEM: eight
    // buffers of 16 columns, six of 32, three of 64 (at least 1.5 k-blocks of the smallest groups)
    static constexpr int kTmemBufs = NMMA <= 16 ? 8 : (NMMA <= 32 ? 6 : 3);
    static constexpr int kAColBase = kTmemBufs * kBufStride;      // first column of the converted-weight slots
    static constexpr int kTmemCols = 256;
    static_assert(kAColBase + kASlots * kACols <= kTmemCols, "TMEM columns");
    static constexpr int kBTileBytes = NMMA * kKBlock;             // planes image of one k-block
    // fixed part of the shared memory (offsets from a 1024-byte aligned base): the cluster reduction's partial sums,
    // [splits][rows owned][128 columns] floats, whatever the cluster size (2..8)
    static constexpr int red_rows() {
        int most = 0;
        for (int sl = 2; sl <= kMaxClusterSplits; ++sl) {
            const int r = sl * ((kMaxM + sl - 1) / sl);
            most = r > most ? r : most;
        }
        return most;
    }
    static constexpr int kOffRed = 0;
    static constexpr int kOffStages = (kOffRed + red_rows() * kTileN * 4 + 1023) / 1024 * 1024;
};

// The load stages of the small-M kernel, sized by the groups per k-block (gpk = 128 / G) and by whether zero points
// are staged: packed weights (128 rows of 64 bytes, 64-byte swizzle) | planes image (NMMA x 128 B, the MMA's B operand, 1024-aligned) | constants (gpk x 16
// rows x 8 floats) | scale tile (gpk x 128 n, fp16) [| zero-point tile]. As many stages as fit in the budget that
// keeps two CTAs per SM (at least 3, at most 8), then the barriers and a few flags.
struct SmallLayout {
    int gpk, b_off, c_off, s_off, z_off, stage_bytes, p_stages, off_bar, off_misc, smem_bytes;
    __host__ __device__ SmallLayout(int b_tile_bytes, int off_stages, int G, bool zp) {
        gpk = kKBlock / G;
        b_off = kPackedTileBytes;
        c_off = b_off + b_tile_bytes;
        s_off = c_off + gpk * kConstFloatsPerGroup * 4;
        z_off = s_off + gpk * kTileN * 2;
        stage_bytes = (z_off + (zp ? gpk * kTileN * 2 : 0) + 1023) / 1024 * 1024;   // swizzled operand 1024-aligned
        const int fixed = off_stages + 1024 + 256;                 // + alignment slack, barriers, flags
        const int fit = (kSmemBudget - fixed - 16 * 8) / stage_bytes;
        p_stages = fit < 3 ? 3 : (fit > 8 ? 8 : fit);
        off_bar = off_stages + p_stages * stage_bytes;
        off_misc = off_bar + (2 * p_stages + 2 * kMaxTmemBufs + kASlots) * 8;
        smem_bytes = off_misc + 64 + 1024;                         // + alignment slack
    }
};

struct RunParams {
    const uint8_t *planes;      // [m_tiles][kb_total][NMMA x 128 B] planes images from unfold_small_kernel
    const float *consts;        // [m_tiles][K/G][8 x 16] combine constants from unfold_small_kernel
    const uint8_t *w;           // prepacked tiles
    const __half *scale;
    const __half *zp;           // [K/G, N] zero points (kernels instantiated with kZp), else null
    const __half *bias;         // [N] or null
    __half *y;
    float *ws_part;             // [splits, M, N] split-K partial sums (splits > 1)
    uint32_t *ws_count;         // [m_tiles, n_tiles] arrival counters (splits > 1)
    int32_t *dbg_y123;          // [3, M, N] integer partials of group dbg_group (debug mode), else null
    int M, K, N, G;
    int m_sub, n_tiles, m_tiles, splits, kb_total;
    int reduce;                 // kReduceNone, kReduceCluster (splits <= 8, cluster along z) or kReduceGlobal
    int dbg_group;              // -1 in normal runs
};


// ------------------------------------------------------------------------------------------------ unfold

// Steps 2-7 for four values of one group, IEEE binary32 with every operation rounded on its own (no contraction);
// rintf rounds half to even. A group whose A_max is 0 holds only zeros; dividing those by 1 gives zero planes, so no
// branch is needed.
// The quotient tmp1 = RN(RN(7.49f x) / A_max) is formed from the correctly rounded reciprocal r = RN(1/A_max),
// shared by the whole group: q0 = RN(n r), the exact residual e = n - q0 A_max (one fused multiply-add) and
// q = RN(q0 + e r), the final correction step of Markstein's division sequences (P. Markstein, "IA-64 and Elementary
// Functions", 2000). Over the whole input domain (every finite fp16 x with every fp16 A_max >= |x|, 1,007,713,278
// pairs) it was checked on the GPU to equal the IEEE quotient bit for bit; it has no branch, so the four quotients
// of a lane overlap.
__device__ __forceinline__ void msd_unfold4(const float (&x)[4], float amax, float (&a1)[4], float (&a2)[4],
                                            float (&a3)[4]) {
    const float den = amax == 0.0f ? 1.0f : amax;
    const float rcp = __frcp_rn(den);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float n = __fmul_rn(kF1, x[j]);
        const float q0 = __fmul_rn(n, rcp);
        const float t1 = __fmaf_rn(__fmaf_rn(-q0, den, n), rcp, q0);
        const float r1 = rintf(t1);
        const float t2 = __fmul_rn(__fsub_rn(t1, r1), kF2);
        const float r2 = rintf(t2);
        const float t3 = __fmul_rn(__fsub_rn(t2, r2), kF2);
        a1[j] = r1;
        a2[j] = r2;
        a3[j] = rintf(t3);
    }
}

// Four fp16 of one row starting at k (k % 4 == 0); zeros past K or for rows past M.
__device__ __forceinline__ void load_x4(const __half *x, int M, int K, int row, int k, float (&v)[4]) {
    v[0] = v[1] = v[2] = v[3] = 0.0f;
    if (row < M && k < K) {
        const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(x + static_cast<size_t>(row) * K + k));
        const __half2 h01 = *reinterpret_cast<const __half2 *>(&raw.x);
        const __half2 h23 = *reinterpret_cast<const __half2 *>(&raw.y);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        v[0] = f01.x;
        v[1] = f01.y;
        v[2] = f23.x;
        v[3] = f23.y;
    }
}

// Max of non-negative values / integer sum over the lanes that share one group: a group spans G/4 consecutive lanes
// (4 values per lane). A whole-warp group uses one redux instruction (non-negative floats order like their bits).
__device__ __forceinline__ float group_absmax(float v, int lanes_per_group) {
    if (lanes_per_group == 32) return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
    for (int off = 1; off < lanes_per_group; off <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}
__device__ __forceinline__ int group_isum(int v, int lanes_per_group) {
    if (lanes_per_group == 32) return __reduce_add_sync(0xffffffffu, v);
    for (int off = 1; off < lanes_per_group; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Byte offset of (row, k) in a K-major 128-byte-swizzled operand tile with 128-byte rows.
__device__ __forceinline__ uint32_t sw128_offset(int row, int kbyte) {
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((((kbyte >> 4) ^ (row & 7)) << 4)) +
                                 (kbyte & 15));
}

// ------------------------------------------------------------------------------------------------ int4 -> e4m3

// The tensor cores read each weight as one E4M3 byte whose bits are the offset-binary nibble u = w + 8 (0..15): the
// bytes 0..7 are the E4M3 subnormals u * 2^-9 and 8..15 the first normal binade, also u * 2^-9, so the byte stands
// for u exactly and the MMA yields 2^-9 * sum_k A_i[k] (w[k] + 8). The combine multiplies by 2^9 (folded into its
// coefficients) and subtracts 8 S_i. Turning packed nibbles into these bytes needs no table: the prepacked layout
// puts k .. k+3 in the low nibbles and k+4 .. k+7 in the high nibbles of each 32-bit word.
constexpr float kMmaUnit = 512.0f;     // 2^9: one MMA unit of the weight operand

__device__ __forceinline__ uint4 expand_nibbles16(uint2 v) {
    return make_uint4(v.x & 0x0F0F0F0Fu, (v.x >> 4) & 0x0F0F0F0Fu, v.y & 0x0F0F0F0Fu, (v.y >> 4) & 0x0F0F0F0Fu);
}

// The same for a whole tile by NT threads (NT divides 1024): chunks q = t, t + NT, ... All of a thread's packed
// chunks are read before any operand byte is written, so the loads overlap (source and destination may not be
// proven disjoint by the compiler otherwise).
template <int NT>
__device__ __forceinline__ void convert_tile(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int t) {
    constexpr int kPer = 1024 / NT;
    uint2 v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) v[j] = *reinterpret_cast<const uint2 *>(src + (t + j * NT) * 8);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int q = t + j * NT;
        const int row = q >> 3, ch = q & 7;
        *reinterpret_cast<uint4 *>(dst + (row >> 3) * 1024 + (row & 7) * 128 + ((ch ^ (row & 7)) << 4)) =
            expand_nibbles16(v[j]);
    }
}

// ------------------------------------------------------------------------------------------------ kernels

// kNK: the packed weights come as [N, K/2] (each column's K contiguous, two k per byte), else as [K/2, N].
template <bool kNK>
__global__ void prepack_kernel(const uint8_t *__restrict__ in, uint8_t *__restrict__ out, int K, int N,
                               int kb_total) {
    __shared__ uint8_t tile[kKBlock / 2][kTileN + 4];
    const int nt = blockIdx.x, kb = blockIdx.y;
    const int half_k = K / 2;
    for (int idx = threadIdx.x; idx < (kKBlock / 2) * kTileN; idx += blockDim.x) {
        // consecutive threads read consecutive bytes of the source
        const int kk = kNK ? idx % (kKBlock / 2) : idx / kTileN, c = kNK ? idx / (kKBlock / 2) : idx % kTileN;
        const int gk = kb * (kKBlock / 2) + kk, gn = nt * kTileN + c;
        uint8_t v = 0;                                               // two zero weights
        if (gk < half_k && gn < N)
            v = kNK ? in[static_cast<size_t>(gn) * half_k + gk] : in[static_cast<size_t>(gk) * N + gn];
        tile[kk][c] = static_cast<uint8_t>(v ^ 0x88u);               // w -> w + 8 in both nibbles
    }
    __syncthreads();
    // row r of the tile: byte 4q + b holds k = 8q + b (low nibble) and k + 4 (high nibble)
    uint8_t *dst = out + (static_cast<size_t>(nt) * kb_total + kb) * kPackedTileBytes;
    for (int idx = threadIdx.x; idx < kPackedTileBytes; idx += blockDim.x) {
        const int r = idx / (kKBlock / 2), j = idx % (kKBlock / 2);
        const int k0 = 8 * (j >> 2) + (j & 3), k1 = k0 + 4;
        const int lo = (tile[k0 >> 1][r] >> (4 * (k0 & 1))) & 0xF, hi = (tile[k1 >> 1][r] >> (4 * (k1 & 1))) & 0xF;
        dst[idx] = static_cast<uint8_t>(lo | (hi << 4));
    }
}

// One warp per (row, 128-k block): the same lane mapping and arithmetic as the run kernel's unfold. row_amax (per
// channel: one group of all K) replaces the group maximum when given; amax_out then has one value per row.
__global__ void unfold_debug_kernel(const __half *__restrict__ x, int M, int K, int G, int8_t *__restrict__ planes,
                                    float *__restrict__ amax_out, const float *__restrict__ row_amax) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x;
    const int kwarp = (blockIdx.y * (blockDim.x / 32) + threadIdx.x / 32) * kKBlock;
    if (kwarp >= K) return;                                          // whole warp: no lane left behind a shuffle
    const int kbase = kwarp + lane * 4;
    const bool valid = kbase < K;                                    // lanes past K compute on zeros, store nothing
    float v[4];
    load_x4(x, M, K, row, kbase, v);
    const int lpg = G < kKBlock ? G / 4 : 32;
    float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    am = group_absmax(am, lpg);
    if (row_amax != nullptr) am = row_amax[row];
    float a1[4], a2[4], a3[4];
    msd_unfold4(v, am, a1, a2, a3);
    if (!valid) return;
    const size_t plane = static_cast<size_t>(M) * K;
    const size_t base = static_cast<size_t>(row) * K + kbase;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        planes[base + j] = static_cast<int8_t>(__float2int_rn(a1[j]));
        planes[plane + base + j] = static_cast<int8_t>(__float2int_rn(a2[j]));
        planes[2 * plane + base + j] = static_cast<int8_t>(__float2int_rn(a3[j]));
    }
    if (amax_out != nullptr && (lane & (lpg - 1)) == 0) amax_out[static_cast<size_t>(row) * (K / G) + kbase / G] = am;
}

// ------------------------------------------------------------------------------------------------ int8 weights
// An int8 weight w = 16 hi + lo with hi = w >> 4 in [-8, 7] and lo = w & 15 in [0, 15]. Group g of the int8 problem
// becomes groups 2g (weights hi, scale 16 s, zero point -1/2) and 2g + 1 (weights lo - 8, scale s, zero point zp)
// of an int4 problem with 2K rows, whose x repeats each group of x twice: both groups see the same planes and A_max
// and s (16 (hi + 1/2) + (lo - 8 - zp)) = s (w - zp), so the int4 path computes the int8 product exactly.

// Prepacked int4 tiles of the split weights (2K rows) from int8 [K, N]: the layout of prepack_kernel.
__global__ void prepack_w8_kernel(const int8_t *__restrict__ w8, uint8_t *__restrict__ out, int K, int N, int G,
                                  int kb_total2) {
    const int nt = blockIdx.x, kb = blockIdx.y;
    uint8_t *dst = out + (static_cast<size_t>(nt) * kb_total2 + kb) * kPackedTileBytes;
    auto nibble = [&](int k2, int n) -> uint32_t {
        if (k2 >= 2 * K || n >= N) return 8u;                           // padding: weight 0
        const int g = k2 / (2 * G), part = (k2 / G) & 1, kk = g * G + k2 % G;
        const uint32_t b = static_cast<uint8_t>(w8[static_cast<size_t>(kk) * N + n]);
        return part == 0 ? ((b ^ 0x80u) >> 4) & 15u : b & 15u;          // hi + 8, or (lo - 8) + 8
    };
    for (int idx = threadIdx.x; idx < kPackedTileBytes; idx += blockDim.x) {
        const int r = idx / (kKBlock / 2), j = idx % (kKBlock / 2);
        const int k0 = kb * kKBlock + 8 * (j >> 2) + (j & 3);
        const int n = nt * kTileN + r;
        dst[idx] = static_cast<uint8_t>(nibble(k0, n) | (nibble(k0 + 4, n) << 4));
    }
}

// The int4 problem's x [M, 2K] (each group of x twice), scales [2 K/G, N] and zero points [2 K/G, N], into the
// workspace. Grid-stride over both tasks.
__global__ void __launch_bounds__(256) w8_prep_kernel(const __half *__restrict__ x, int M, int K, int G,
                                                      const __half *__restrict__ scale, const __half *__restrict__ zp,
                                                      int N, __half *__restrict__ x2, __half *__restrict__ scale2,
                                                      __half *__restrict__ zp2) {
    // no early release of the dependents: the main kernel fetches the scales and zero points written here before
    // it waits for its own predecessor, so it must not start before this kernel has ended
    pdl_wait();              // x may be the preceding kernel's output, which may also still read these buffers
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    // x2: 8 halves (16 bytes) at a time; G is a multiple of 32, so a piece never straddles a group
    const size_t pieces = static_cast<size_t>(M) * (2 * K) / 8;
    for (size_t i = tid; i < pieces; i += stride) {
        const size_t e = i * 8;
        const int m = static_cast<int>(e / (2 * K));
        const int k2 = static_cast<int>(e % (2 * K));
        const int g = k2 / (2 * G), kk = g * G + k2 % G;
        *reinterpret_cast<uint4 *>(x2 + e) = *reinterpret_cast<const uint4 *>(x + static_cast<size_t>(m) * K + kk);
    }
    const int Gn = K / G;
    const size_t cells = static_cast<size_t>(Gn) * N;
    for (size_t i = tid; i < cells; i += stride) {
        const int g = static_cast<int>(i / N), n = static_cast<int>(i % N);
        const __half s = scale[i];
        scale2[(2 * static_cast<size_t>(g)) * N + n] = __hmul(s, __float2half(16.0f));    // exact below 4096
        scale2[(2 * static_cast<size_t>(g) + 1) * N + n] = s;
        zp2[(2 * static_cast<size_t>(g)) * N + n] = __float2half(-0.5f);
        zp2[(2 * static_cast<size_t>(g) + 1) * N + n] = zp != nullptr ? zp[i] : __float2half(0.0f);
    }
}

// Per-channel quantization (one group spanning all of K; the kernels then work in sub-groups of gs k with the
// row's A_max). Blocks [0, M): A_max of row m = max |x[m, k]| over all k (exact: a maximum of fp16 magnitudes).
// Blocks [M, M + gridDim.x - M): scale (and zero-point) row 0 copied to rows 0 .. reps - 1 of scale_rep / zp_rep,
// for the kernels that load scales as [sub-group, column] tiles (null: not needed).
__global__ void __launch_bounds__(256) per_channel_prep_kernel(const __half *__restrict__ x, int M, int K,
                                                               float *__restrict__ row_amax,
                                                               const __half *__restrict__ scale,
                                                               const __half *__restrict__ zp, int N, int reps,
                                                               __half *__restrict__ scale_rep,
                                                               __half *__restrict__ zp_rep) {
    // no early release of the dependents: the main kernels fetch the scale rows written here before they wait for
    // their own predecessor, so they must not start before this kernel has ended
    pdl_wait();              // x may be the preceding kernel's output, which may also still read these buffers
    if (static_cast<int>(blockIdx.x) >= M) {
        if (scale_rep == nullptr) return;
        const int nb = gridDim.x - M;
        const size_t total = static_cast<size_t>(reps) * N;
        for (size_t i = static_cast<size_t>(blockIdx.x - M) * blockDim.x + threadIdx.x; i < total;
             i += static_cast<size_t>(nb) * blockDim.x) {
            const int n = static_cast<int>(i % N);
            scale_rep[i] = scale[n];
            if (zp_rep != nullptr) zp_rep[i] = zp[n];
        }
        return;
    }
    const int m = blockIdx.x;
    __shared__ float red[8];
    float am = 0.0f;
    for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
        if (k + 8 <= K) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<size_t>(m) * K + k));
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[j]));
                am = fmaxf(am, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        } else {
            for (int kk = k; kk < K; ++kk) am = fmaxf(am, fabsf(__half2float(x[static_cast<size_t>(m) * K + kk])));
        }
    }
    for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = am;
    __syncthreads();
    if (threadIdx.x == 0) {
        float r = red[0];
        for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) r = fmaxf(r, red[w]);
        row_amax[m] = r;
    }
}

__global__ void wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing arrives on this barrier: the wait must give up and record the timeout
        mbar_wait(smem_addr(&bar), 0, &abort_flag, kSiteDebugWait, limit_ns);
        mbar_arrive(smem_addr(&bar));                                // complete the phase before exit
    }
}

// Steps 1-8 for the small-M path, once per (row tile, 128-k block): block (kb, mt), one warp per row slot r of the
// tile (lane: 4 k). Plane i of row r goes to row i * max_m + r of the k-block's B operand image (E4M3, 128-byte
// swizzle, K-major); row slots past the tile's rows or past M, and the padding rows 3 max_m .. nmma - 1, hold zeros.
// Per (row, group) the constant record holds 512 c_i A_max (i = 1..3, the MMA unit folded in), the offset-binary
// correction 8 sum_i c_i A_max S_i, then the plane sums S_i (read by debug runs) and a zero: [row][8] per group.
// counters (null when the main kernel reduces without them): the split-K arrival counters of the main kernel that
// follows, cleared here by block (0, 0), so that a run needs no cleared workspace even after an earlier run gave up.
__global__ void __launch_bounds__(512) unfold_small_kernel(const __half *__restrict__ x, int M, int K, int G,
                                                           int kb_total, int m_sub, int nmma,
                                                           uint8_t *__restrict__ planes, float *__restrict__ consts,
                                                           const float *__restrict__ row_amax,
                                                           uint32_t *__restrict__ counters, int n_counters) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, r = threadIdx.x >> 5;
    const int kb = blockIdx.x, mt = blockIdx.y;
    const int max_m = nmma / 3, lpg = G / 4, Gn = K / G;
    const int m = mt * m_sub + r;
    const bool live = r < m_sub && m < M;
    // the warp's 256 bytes of x (two lines) on their way to L2 while the preceding kernel finishes
    if (live && (lane & 15) == 0 && kb * kKBlock + lane * 4 < K)
        prefetch_l2(x + static_cast<size_t>(m) * K + kb * kKBlock + lane * 4);
    pdl_wait();                  // x may be the preceding kernel's output, which may also still read the planes
    // the preceding run's main kernel has ended; this run's reads its counters only after this kernel has ended
    if (counters != nullptr && kb == 0 && mt == 0)
        for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0u;
    float v[4];
    load_x4(x, live ? M : 0, K, m, kb * kKBlock + lane * 4, v);     // a dead row slot reads zeros
    float am = group_absmax(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))), lpg);
    if (row_amax != nullptr) am = live ? row_amax[m] : 0.0f;       // per channel: the whole row's maximum
    float a1[4], a2[4], a3[4];
    msd_unfold4(v, am, a1, a2, a3);
    // plane sums of a lane (each in [-28, 28]): planes 1 and 2 packed in one word so one reduction serves both
    // (11-bit fields hold lane sums + 28, at most 32 * 56 = 1792 < 2048 over a whole-warp group), plane 3 alone
    const int p1 = __float2int_rn((a1[0] + a1[1]) + (a1[2] + a1[3])) + 28;
    const int p2 = __float2int_rn((a2[0] + a2[1]) + (a2[2] + a2[3])) + 28;
    const int packed = group_isum(p1 | (p2 << 11), lpg);
    const int sum3 = group_isum(__float2int_rn((a3[0] + a3[1]) + (a3[2] + a3[3])), lpg);
    uint8_t *img = planes + (static_cast<size_t>(mt) * kb_total + kb) * nmma * kKBlock;
    const int kbyte = lane * 4;
    *reinterpret_cast<uint32_t *>(img + sw128_offset(r, kbyte)) = e4m3x2(a1[1], a1[0]) | (e4m3x2(a1[3], a1[2]) << 16);
    *reinterpret_cast<uint32_t *>(img + sw128_offset(max_m + r, kbyte)) =
        e4m3x2(a2[1], a2[0]) | (e4m3x2(a2[3], a2[2]) << 16);
    *reinterpret_cast<uint32_t *>(img + sw128_offset(2 * max_m + r, kbyte)) =
        e4m3x2(a3[1], a3[0]) | (e4m3x2(a3[3], a3[2]) << 16);
    if (r == 0)
        for (int pr = 3 * max_m; pr < nmma; ++pr) *reinterpret_cast<uint32_t *>(img + sw128_offset(pr, kbyte)) = 0u;
    const int g = kb * (kKBlock / G) + lane / lpg;
    if ((lane & (lpg - 1)) == 0 && g < Gn) {
        const int bias = 28 * lpg;
        const float s1 = static_cast<float>((packed & 0x7FF) - bias);
        const float s2 = static_cast<float>(((packed >> 11) & 0x7FF) - bias);
        const float s3 = static_cast<float>(sum3);
        const float c1 = kC1 * am, c2 = kC2 * am, c3 = kC3 * am;
        float4 *cg = reinterpret_cast<float4 *>(consts + (static_cast<size_t>(mt) * Gn + g) * kConstFloatsPerGroup) +
                     2 * r;
        cg[0] = make_float4(kMmaUnit * c1, kMmaUnit * c2, kMmaUnit * c3,      // exact: power-of-two scaling
                            8.0f * (c1 * s1 + c2 * s2 + c3 * s3));
        cg[1] = make_float4(s1, s2, s3, 0.0f);
    }
}

// Steps 10-11 for rows H * R .. H * R + R - 1 of the tile (compile-time, so the accumulator registers are indexed
// statically) from one K-group's TMEM columns d (column i * kMaxM + m holds 2^-9 sum_k A_i[m, k] u[k, n]):
// y[m] += s_n (sum_i (512 c_i A_max) d_i - corr f_n), with corr = 8 sum_i c_i A_max S_i and f_n = 1 + zp / 8.
template <int kMaxM, int R, int H, bool kZp>
__device__ __forceinline__ void combine_rows(const uint32_t (&d)[3][16], uint32_t cg, float s_n, float f_n,
                                             int rows_valid, float (&yacc)[R]) {
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int m = H * R + rr;
        if (m < kMaxM && m < rows_valid) {
            const float4 c = lds_f128(cg + 32 * m);       // the row's record: one address for the warp
            const float d1 = __uint_as_float(d[m >> 4][m & 15]);
            const float d2 = __uint_as_float(d[(kMaxM + m) >> 4][(kMaxM + m) & 15]);
            const float d3 = __uint_as_float(d[(2 * kMaxM + m) >> 4][(2 * kMaxM + m) & 15]);
            float t = fmaf(c.x, d1, kZp ? -c.w * f_n : -c.w);
            t = fmaf(c.y, d2, t);
            t = fmaf(c.z, d3, t);
            yacc[rr] = fmaf(s_n, t, yacc[rr]);
        }
    }
}

// Debug: the integer partials Y_i = 512 d_i - 8 S_i of the same rows for group dbg_group.
template <int kMaxM, int R, int H>
__device__ __forceinline__ void debug_rows(const uint32_t (&d)[3][16], uint32_t cg, int rows_valid, int32_t *dbg,
                                           int M, int N, int m0, int n) {
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int m = H * R + rr;
        if (m < kMaxM && m < rows_valid) {
            const float4 sv = lds_f128(cg + 32 * m + 16);
            const float sp[3] = {sv.x, sv.y, sv.z};
#pragma unroll
            for (int pl = 0; pl < 3; ++pl) {
                const int col = pl * kMaxM + m;
                const float yi = kMmaUnit * __uint_as_float(d[col >> 4][col & 15]) - 8.0f * sp[pl];
                dbg[(static_cast<size_t>(pl) * M + m0 + m) * N + n] = __float2int_rn(yi);
            }
        }
    }
}

// kZp: the weights carry zero points, w - zp[g, n] being the quantized value the scale multiplies. The plane dots
// then need (8 + zp) S_i taken off instead of 8 S_i, that is the correction term times 1 + zp / 8.
// Roles: warp 0 lane 0 issues the loads, warp 1 lane 0 the MMAs; warps 2-5 (the converters) expand each k-block's
// weight tile; warps 6-9 run the epilogue, one warp per TMEM lane quarter (32 output columns) over all rows, reading
// the constants and scales in place in the load stage, as soon as each K-group's MMAs have committed. So the
// expansion of a k-block and the epilogue of an earlier one run at the same time on different warps. The converters
// hand a tile to the MMA warp through a hardware named barrier, once the tile is expanded and the MMAs that read its
// slot before, and the epilogue reads of the TMEM buffers it will use, are done. The MMA-issuing thread makes no
// ordinary shared-memory access between its MMAs (such an access waits for its MMAs in flight to finish reading
// their operands) and never gives up a wait. After a failed wait the other roles skip their work but keep every
// synchronisation (arrivals on the named barrier, waits for the MMAs' commits), so nothing can wait forever.
template <int NMMA, bool kZp>
__global__ void __launch_bounds__(kThreads, 2)
    msd_kernel(const RunParams p, const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
               const __grid_constant__ CUtensorMap tmap_z) {
    using C = Cfg<NMMA>;
    constexpr int kMaxM = C::kMaxM;
    constexpr int R = C::kRowsPerWarp;
    const SmallLayout L(C::kBTileBytes, C::kOffStages, p.G, kZp);
    const int P = L.p_stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *red_buf = reinterpret_cast<float *>(smem + C::kOffRed);
    uint8_t *p_ring = smem + C::kOffStages;
    const uint32_t bar0 = smem_addr(smem + L.off_bar);
    // barriers: full_p / empty_p  load stage landed / released (converters done with the weights, epilogue with the
    //                             constants and scales after the k-block's MMAs, which read the planes)
    //           full_t / empty_t  TMEM accumulator written by the MMAs / read by the epilogue
    //           a_free            converted weight slot (TMEM) read by the MMAs (their commit)
    // and the named barriers kOperandBarrier0 + c: converted weight slot c ready for k-block i (i % 2 == c). Before
    // the converters arrive there for k-block i they have seen a_free for k-block i - 2, committed after the MMA warp
    // passed that barrier for k-block i - 2, so no arrival can count towards an earlier phase.
    auto full_p = [&](int s) { return bar0 + 8u * s; };
    auto empty_p = [&](int s) { return bar0 + 8u * (P + s); };
    constexpr int kTmemBufs = C::kTmemBufs;
    auto full_t = [&](int b) { return bar0 + 8u * (2 * P + b); };
    auto empty_t = [&](int b) { return bar0 + 8u * (2 * P + kMaxTmemBufs + b); };
    auto a_free = [&](int c) { return bar0 + 8u * (2 * P + 2 * kMaxTmemBufs + c); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);
    int *last_flag = reinterpret_cast<int *>(smem + L.off_misc + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt = blockIdx.x, mt = blockIdx.y, sp = blockIdx.z;
    const int M = p.M, K = p.K, N = p.N, G = p.G;
    const int m0 = mt * p.m_sub;
    const int gpk = kKBlock / G;                         // groups per k-block
    const int Gn = K / G;
    const bool debug = p.dbg_group >= 0;
    int kb0, kb1;
    if (debug) {
        kb0 = p.dbg_group * G / kKBlock;
        kb1 = kb0 + 1;
    } else {
        kb0 = static_cast<int>(static_cast<int64_t>(sp) * p.kb_total / p.splits);
        kb1 = static_cast<int>(static_cast<int64_t>(sp + 1) * p.kb_total / p.splits);
    }
    const int nkb = kb1 - kb0;

    // One load stage: the k-block's packed weight tile, planes image, constants, scale tile and zero-point tile, all
    // counted on full_p(s).
    const int w_row0 = (nt * p.kb_total + kb0) * kTileN;     // first row of this CTA's weight tiles (64 bytes each)
    const int gshift = 31 - __clz(G);                  // G is 32, 64 or 128
    auto groups_in = [&](int kb) { return (min(K, (kb + 1) * kKBlock) - kb * kKBlock) >> gshift; };
    auto stage_tx = [&](int kb) {
        return static_cast<uint32_t>(kPackedTileBytes + C::kBTileBytes + groups_in(kb) * kConstFloatsPerGroup * 4 +
                                     (debug ? 0 : (kZp ? 2 : 1) * gpk * kTileN * 2));
    };
    // Weights and scales are read-only inputs of the call: they are fetched before waiting for the preceding kernel
    // on the stream. The planes and constants are the unfold pre-pass's output, fetched only after pdl_wait().
    auto issue_static = [&](int i, uint64_t stream_policy, uint64_t keep_policy) {
        const int s = i % P;
        const uint32_t dst = smem_addr(p_ring + s * L.stage_bytes);
        const int kb = kb0 + i;
        mbar_arrive_expect_tx(full_p(s), stage_tx(kb));
        tma_load_2d(dst, &tmap_w, 0, w_row0 + i * kTileN, full_p(s), stream_policy);
        if (!debug) tma_load_2d(dst + L.s_off, &tmap_s, nt * kTileN, kb * gpk, full_p(s), keep_policy);
        if (kZp && !debug) tma_load_2d(dst + L.z_off, &tmap_z, nt * kTileN, kb * gpk, full_p(s), keep_policy);
    };
    auto issue_dynamic = [&](int i, uint64_t keep_policy) {
        const int s = i % P, kb = kb0 + i;
        const uint32_t dst = smem_addr(p_ring + s * L.stage_bytes);
        bulk_g2s(dst + L.b_off, p.planes + (static_cast<size_t>(mt) * p.kb_total + kb) * C::kBTileBytes,
                 C::kBTileBytes, full_p(s), keep_policy);
        bulk_g2s(dst + L.c_off, p.consts + (static_cast<size_t>(mt) * Gn + kb * gpk) * kConstFloatsPerGroup,
                 static_cast<uint32_t>(groups_in(kb) * kConstFloatsPerGroup * 4), full_p(s), keep_policy);
    };

    // ---- set-up. Thread 0 lets the next kernel on the stream start launching, initialises the barriers and at once
    // starts the weight loads of the first ring's worth of k-blocks (the slots are free), so the memory latency
    // overlaps the rest of the set-up and, under programmatic launch, the tail of the unfold pre-pass. The planes and
    // constants of those k-blocks follow from the producer after the set-up barrier, so that no other role waits
    // for their issue.
    const int first_loads = nkb < P ? nkb : P;
    uint64_t stream_policy = 0, keep_policy = 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < P; ++s) {
            mbar_init(full_p(s), 1);
            mbar_init(empty_p(s), kNumConvWarps + kNumEpiWarps);
        }
        for (int b = 0; b < kTmemBufs; ++b) {
            mbar_init(full_t(b), 1);
            mbar_init(empty_t(b), kNumEpiWarps);
        }
        for (int c = 0; c < kASlots; ++c) mbar_init(a_free(c), 1);
        *abort_flag = 0;
        *last_flag = 0;
        mbar_fence_init();
        stream_policy = l2_policy_evict_first();    // weights: read once per call
        keep_policy = l2_policy_evict_last();       // planes, constants and scale tiles: shared by many CTAs
        pdl_launch_dependents();
        for (int i = 0; i < first_loads; ++i) issue_static(i, stream_policy, keep_policy);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kProducerWarp) {
        // ================================================================ TMA producer
        if (lane == 0) {
            pdl_wait();
            for (int i = 0; i < first_loads; ++i) issue_dynamic(i, keep_policy);
            int issued = first_loads;
            for (; issued < nkb; ++issued) {
                const int s = issued % P;
                if (!mbar_wait(empty_p(s), ((issued / P) & 1) ^ 1, abort_flag, kSiteProducerEmpty)) break;
                issue_static(issued, stream_policy, keep_policy);
                issue_dynamic(issued, keep_policy);
            }
            // no copy may still be writing shared memory when the CTA exits
            for (int j = issued > P ? issued - P : 0; j < issued; ++j) mbar_wait_drain(full_p(j % P), (j / P) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ================================================================ MMA issuer
        constexpr uint32_t idesc = idesc_e4m3_f32(NMMA);
        int j = 0;                           // CTA-local group counter
        int last_j[kTmemBufs];
        for (int b = 0; b < kTmemBufs; ++b) last_j[b] = -1;
        for (int i = 0; i < nkb; ++i) {
            const int c = i % kASlots, s = i % P;
            // the whole warp: converted tile i is ready, and so are the TMEM buffers of its groups (barrier ids stay
            // compile-time constants)
            if (c == 0) named_bar_sync(kOperandBarrier0, kOperandThreads);
            else named_bar_sync(kOperandBarrier0 + 1, kOperandThreads);
            const int ng = groups_in(kb0 + i);
            if (lane == 0) {
                tc_fence_after_sync();
                const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(C::kAColBase + c * kACols);
                const uint32_t b_base = smem_addr(p_ring + s * L.stage_bytes + L.b_off);
                for (int gg = 0; gg < ng; ++gg) {
                    const int jj = j + gg, b = jj % kTmemBufs;
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * C::kBufStride);
                    for (int ks = 0; ks < G / 32; ++ks) {
                        const uint32_t kofs = static_cast<uint32_t>(gg * G + ks * 32);
                        umma_f8f6f4_ta(d_tmem, a_tmem + kofs / 4, sdesc_kmajor_sw128(b_base + kofs), idesc,
                                       ks > 0 ? 1u : 0u);
                    }
                    umma_commit(full_t(b));
                    last_j[b] = jj;
                }
                umma_commit(a_free(c));      // slot c may be overwritten once these MMAs are done
            }
            __syncwarp();
            j += ng;
        }
        // no MMA may still be writing TMEM when it is freed, nor arrive on a barrier after the CTA exits
        if (lane == 0) {
            for (int b = 0; b < kTmemBufs; ++b)
                if (last_j[b] >= 0) mbar_wait_drain(full_t(b), (last_j[b] / kTmemBufs) & 1);
            if (nkb > 0) mbar_wait_drain(a_free((nkb - 1) % kASlots), ((nkb - 1) / kASlots) & 1);
        }
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        // ================================================================ converters: weights -> TMEM (A operand)
        const int n_local = (warp & 3) * 32 + lane;      // this thread's weight column = its TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t swz = static_cast<uint32_t>((n_local >> 1) & 3);   // the tile's 64-byte swizzle
        bool ok = true;
        int j = 0;                                       // CTA-local group counter
        for (int i = 0; i < nkb; ++i) {
            const int s = i % P, c = i % kASlots;
            if (ok) ok = mbar_wait_warp(full_p(s), (i / P) & 1, abort_flag, kSiteConvFull);
            // slot c is free once the MMAs of k-block i - 2 are done. Waited for even after a failure (bounded; the
            // MMA warp never stops issuing), so that no arrival below counts towards an earlier phase.
            const uint32_t par = ((i / kASlots) & 1) ^ 1;
            if (ok) ok = mbar_wait_warp(a_free(c), par, abort_flag, kSiteConvEmpty);
            if (!ok) {
                bool drained = true;
                if (lane == 0) drained = mbar_wait_drain(a_free(c), par);
                (void)__shfl_sync(0xffffffffu, drained ? 1 : 0, 0);
            }
            if (ok) {
                tc_fence_after_sync();                   // the slot's last MMAs (a_free) before these stores
                // the column's 64 packed bytes: word q holds k = 8q .. 8q+3 in its low nibbles and 8q+4 .. 8q+7 in
                // its high nibbles, each u = w + 8; one mask (and one shift) gives four E4M3 bytes in k order, one
                // TMEM column
                const uint32_t row = smem_addr(p_ring + s * L.stage_bytes) + static_cast<uint32_t>(n_local * 64);
                uint4 v[4];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) v[ch] = lds_u128(row + 16u * (static_cast<uint32_t>(ch) ^ swz));
                uint32_t e[32];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const uint32_t w4[4] = {v[ch].x, v[ch].y, v[ch].z, v[ch].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        e[2 * (4 * ch + q)] = w4[q] & 0x0F0F0F0Fu;
                        e[2 * (4 * ch + q) + 1] = (w4[q] >> 4) & 0x0F0F0F0Fu;
                    }
                }
                tmem_st32(tmem_base + lane_off + static_cast<uint32_t>(C::kAColBase + c * kACols), e);
                tmem_wait_st();
            }
            tc_fence_before_sync();
            // the TMEM buffers of this k-block's groups must have been read by the epilogue (their previous groups)
            // before the MMA warp issues into them; that gates the MMAs, not the expansion, so one converter warp
            // checks it after its expansion, while the others finish theirs
            const int ng = groups_in(kb0 + i);
            if (warp == kConvWarp0) {
                for (int gg = 0; gg < ng && ok; ++gg) {
                    const int jj = j + gg;
                    ok = mbar_wait_warp(empty_t(jj % kTmemBufs), ((jj / kTmemBufs) & 1) ^ 1, abort_flag,
                                        kSiteTmemEmpty);
                }
            }
            j += ng;
            __syncwarp();
            if (c == 0) named_bar_arrive(kOperandBarrier0, kOperandThreads);
            else named_bar_arrive(kOperandBarrier0 + 1, kOperandThreads);
            if (ok && lane == 0) mbar_arrive(empty_p(s));   // the packed weights are read
        }
    } else {
        // ================================================================ epilogue
        pdl_wait();                                      // outputs are written after the preceding kernel ended
        const int et = threadIdx.x - kEpiWarp0 * 32;     // 0..127
        const int quarter = warp & 3;                    // TMEM lanes this warp may read
        const int n_local = quarter * 32 + lane;
        const int n = nt * kTileN + n_local;
        const int rows_valid = min(p.m_sub, M - m0);
        float yacc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) yacc[r] = 0.0f;

        // After a failed wait the work is skipped, but the MMAs' commits are still waited for (bounded) and the
        // TMEM buffers released, so that the converters and the MMA warp go on.
        bool ok = true;
        int j = 0;
        for (int i = 0; i < nkb; ++i) {
            const int s = i % P;
            // the stage landed before its tile was converted; seen here too, for the constants and scales
            if (ok) ok = mbar_wait_warp(full_p(s), (i / P) & 1, abort_flag, kSiteEpiOperandsEmpty);
            const uint8_t *stage = p_ring + s * L.stage_bytes;
            const uint32_t cs = smem_addr(stage + L.c_off);
            const uint32_t ss = smem_addr(stage + L.s_off), zs = smem_addr(stage + L.z_off);
            const int kb = kb0 + i;
            const int ng = groups_in(kb);
            for (int gg = 0; gg < ng; ++gg, ++j) {
                const int b = j % kTmemBufs;
                const bool live = ok;
                const float s_n =
                    debug || !live ? 0.0f : __half2float(__ushort_as_half(lds_u16(ss + 2 * (gg * kTileN + n_local))));
                const float f_n =
                    kZp && !debug && live
                        ? fmaf(__half2float(__ushort_as_half(lds_u16(zs + 2 * (gg * kTileN + n_local)))), 0.125f, 1.0f)
                        : 1.0f;
                if (!mbar_wait_warp(full_t(b), (j / kTmemBufs) & 1, abort_flag, kSiteEpiTmemFull)) {
                    ok = false;
                    bool drained = true;
                    if (lane == 0) drained = mbar_wait_drain(full_t(b), (j / kTmemBufs) & 1);
                    (void)__shfl_sync(0xffffffffu, drained ? 1 : 0, 0);
                }
                if (!live || !ok) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty_t(b));
                    continue;
                }
                tc_fence_after_sync();
                uint32_t d[3][16];
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(b * C::kBufStride);
                tmem_ld16(taddr, d[0]);
                if (NMMA > 16) tmem_ld16(taddr + 16, d[1]);
                if (NMMA > 32) tmem_ld16(taddr + 32, d[2]);
                tmem_wait_ld();
                reg_fence16(d[0]);
                if (NMMA > 16) reg_fence16(d[1]);
                if (NMMA > 32) reg_fence16(d[2]);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_t(b));
                const uint32_t cg = cs + 4 * gg * kConstFloatsPerGroup;
                if (debug) {
                    if (kb * gpk + gg == p.dbg_group && n < N)
                        debug_rows<kMaxM, R, 0>(d, cg, rows_valid, p.dbg_y123, M, N, m0, n);
                    continue;
                }
                combine_rows<kMaxM, R, 0, kZp>(d, cg, s_n, f_n, rows_valid, yacc);
            }
            if (!ok) continue;
            // the k-block's MMAs have completed (its last full_t wait saw them) and its constants are read
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_p(s));
        }
        // all epilogue warps take the same path from here on (named barriers below)
        ok = !named_bar_or(kEpiBarrierId, kEpiThreads, !ok);

        if (ok && !debug) {
            const float bias_n = p.bias != nullptr && n < N ? __half2float(p.bias[n]) : 0.0f;
            if (p.reduce == kReduceNone) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int m = r;
                    if (m < rows_valid && n < N)
                        p.y[static_cast<size_t>(m0 + m) * N + n] =
                            __float2half_rn(p.bias != nullptr ? yacc[r] + bias_n : yacc[r]);
                }
            } else if (p.reduce == kReduceCluster) {
                // row m is finished by CTA m % S of the cluster: this slice stores its partial sum of the row
                // straight into that CTA's shared memory, [slice][m / S][column], summed there after the cluster
                // barrier below
                const int S = p.splits, owned = (kMaxM + S - 1) / S;
                const uint32_t red = smem_addr(red_buf);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int m = r;
                    if (m < rows_valid) {
                        const uint32_t off = static_cast<uint32_t>(((sp * owned + m / S) * kTileN + n_local) * 4);
                        st_cluster_f32(cluster_map(red + off, static_cast<uint32_t>(m % S)), yacc[r]);
                    }
                }
            } else {
                float *part = p.ws_part + static_cast<size_t>(sp) * M * N;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int m = r;
                    if (m < rows_valid && n < N) part[static_cast<size_t>(m0 + m) * N + n] = yacc[r];
                }
                __threadfence();
                named_bar_sync(kEpiBarrierId, kEpiThreads);
                if (et == 0) {
                    const uint32_t prev = atomicAdd(p.ws_count + static_cast<size_t>(mt) * p.n_tiles + nt, 1u);
                    *last_flag = (prev == static_cast<uint32_t>(p.splits - 1));
                }
                named_bar_sync(kEpiBarrierId, kEpiThreads);
                if (*last_flag) {
                    __threadfence();
                    for (int m = 0; m < rows_valid && n < N; ++m) {
                        const float *src = p.ws_part + static_cast<size_t>(m0 + m) * N + n;
                        const size_t slice = static_cast<size_t>(M) * N;
                        float acc = 0.0f;
                        for (int s0 = 0; s0 < p.splits; s0 += 8) {     // eight loads in flight, summed in order
                            float v[8];
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                v[q] = s0 + q < p.splits ? __ldcg(src + (s0 + q) * slice) : 0.0f;
#pragma unroll
                            for (int q = 0; q < 8; ++q) acc += v[q];
                        }
                        if (p.bias != nullptr) acc += bias_n;
                        p.y[static_cast<size_t>(m0 + m) * N + n] = __float2half_rn(acc);
                    }
                    if (et == 0) p.ws_count[static_cast<size_t>(mt) * p.n_tiles + nt] = 0u;
                }
            }
        }
    }

    if (p.reduce == kReduceCluster && !debug) {
        // every thread of every CTA of the cluster takes part in the barrier (warps reconverged first); after it no
        // CTA touches another's shared memory, so none has to stay for its peers
        __syncwarp();
        cluster_sync_all();                                      // all partial sums are in their owners' memory
        if (warp >= kEpiWarp0) {
            const int n_local = (warp & 3) * 32 + lane;
            const int n = nt * kTileN + n_local;
            const int rows_valid = min(p.m_sub, M - m0);
            const int S = p.splits, owned = (kMaxM + S - 1) / S;
            // CTA sp of the cluster finishes rows sp, sp + S, ...; every row sums the slices in slice order
            for (int mi = 0; mi * S + sp < rows_valid && n < N; ++mi) {
                float acc = 0.0f;
                for (int q = 0; q < S; ++q) acc += red_buf[(q * owned + mi) * kTileN + n_local];
                if (p.bias != nullptr) acc += __half2float(p.bias[n]);
                p.y[static_cast<size_t>(m0 + mi * S + sp) * N + n] = __float2half_rn(acc);
            }
        }
    }

    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace wqbmm
