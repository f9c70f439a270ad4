// Decode path of the A16W4 per-group MSD matmul (WeightQuantBatchMatmulExperiment page, section 4.1), for one or two
// rows of x: a matrix-vector product bound by reading the weights once from HBM. The three integer products
// Y_i = A_i . W_g are 4-way int8 dot products on the CUDA cores (dp4a), exact in int32.
//
//   gemv_unfold_kernel  steps 1-8 once per (row, 128 k): the three planes as int8 and, per (row, group), the combine
//                       constants {c1 A_max, c2 A_max, c3 A_max, 8 sum_i c_i A_max S_i} (debug: {S1, S2, S3, 0})
//   msd_gemv_kernel     steps 9-11 for 16 output columns over all of K per CTA: no split over K, so no reduction
//                       between CTAs. Each warp takes an eighth of the k-blocks; a lane streams 16-byte pieces of two
//                       weight rows straight into registers (issued before waiting for the unfold, so the weight
//                       stream overlaps it), widens the nibbles to bytes u = w + 8 and takes dp4a against the planes:
//                       dot_i = sum A_i u = Y_i + 8 S_i. Lanes that share a group add their dots, every lane applies
//                       the combine and the scale, and the partial sums of the lanes and warps are added in a fixed
//                       order, so the result does not depend on timing.
// Both kernels run under programmatic launch: the unfold waits for the preceding kernel before reading x, the GEMV
// kernel fetches weights and scales at once and waits for the unfold before reading the planes.
#pragma once

#include "msd_kernels.cuh"

namespace wqbmm {

constexpr int kGemvMaxRows = 2;
constexpr int kGemvCols = 16;                       // output columns per CTA
constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvKbPerPass = 8;                   // k-blocks per warp held in registers at a time
constexpr int kGemvPlaneBytes = 3 * kKBlock;        // one row, one k-block: [chunk 4][plane 3][32 bytes]

// Steps 1-8 for one row and one 128-k block per warp (lane: 4 k). Planes to [row][kb][chunk][plane][32 B] as int8,
// constants to [row][group] (float4).
__global__ void __launch_bounds__(128) gemv_unfold_kernel(const __half *__restrict__ x, int M, int K, int G,
                                                          int kb_total, int8_t *__restrict__ planes,
                                                          float4 *__restrict__ consts, int debug) {
    pdl_launch_dependents();
    pdl_wait();                                        // x may be the preceding kernel's output
    const int lane = threadIdx.x & 31;
    const int kb = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int row = blockIdx.y;
    if (kb >= kb_total) return;                        // whole warps only
    const int lpg = G / 4;
    float v[4];
    load_x4(x, M, K, row, kb * kKBlock + lane * 4, v);
    float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    am = group_absmax(am, lpg);
    float a1[4], a2[4], a3[4];
    msd_unfold4(v, am, a1, a2, a3);
    const int s1 = group_isum(__float2int_rn((a1[0] + a1[1]) + (a1[2] + a1[3])), lpg);
    const int s2 = group_isum(__float2int_rn((a2[0] + a2[1]) + (a2[2] + a2[3])), lpg);
    const int s3 = group_isum(__float2int_rn((a3[0] + a3[1]) + (a3[2] + a3[3])), lpg);
    auto pack4 = [](const float (&a)[4]) {
        return (static_cast<uint32_t>(static_cast<int>(a[0])) & 0xFFu) |
               ((static_cast<uint32_t>(static_cast<int>(a[1])) & 0xFFu) << 8) |
               ((static_cast<uint32_t>(static_cast<int>(a[2])) & 0xFFu) << 16) |
               (static_cast<uint32_t>(static_cast<int>(a[3])) << 24);
    };
    int8_t *dst = planes + (static_cast<size_t>(row) * kb_total + kb) * kGemvPlaneBytes + (lane >> 3) * 96 +
                  (lane & 7) * 4;
    *reinterpret_cast<uint32_t *>(dst) = pack4(a1);
    *reinterpret_cast<uint32_t *>(dst + 32) = pack4(a2);
    *reinterpret_cast<uint32_t *>(dst + 64) = pack4(a3);
    const int Gn = K / G;
    const int g = kb * (kKBlock / G) + lane / lpg;
    if ((lane & (lpg - 1)) == 0 && g < Gn) {
        float4 rec;
        if (debug) {
            rec = make_float4(static_cast<float>(s1), static_cast<float>(s2), static_cast<float>(s3), 0.0f);
        } else {
            const float c1 = kC1 * am, c2 = kC2 * am, c3 = kC3 * am;
            rec = make_float4(c1, c2, c3,
                              8.0f * (c1 * static_cast<float>(s1) + c2 * static_cast<float>(s2) +
                                      c3 * static_cast<float>(s3)));
        }
        consts[static_cast<size_t>(row) * Gn + g] = rec;
    }
}

struct GemvParams {
    const uint8_t *w;           // prepacked tiles
    const __half *scale;        // [K/G, N]
    const int8_t *planes;       // from gemv_unfold_kernel
    const float4 *consts;
    __half *y;
    int32_t *dbg_y123;          // debug: integer partials of group dbg_group, else null
    int M, K, N, G, kb_total, dbg_group;
};

__device__ __forceinline__ uint4 ldg_stream16(const void *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

// dp4a of the eight widened words of a 16-byte weight piece (32 k) against 32 plane bytes.
__device__ __forceinline__ int dot32(const uint4 w, const int4 pa, const int4 pb, int acc) {
    acc = __dp4a(static_cast<int>(w.x & 0x0F0F0F0Fu), pa.x, acc);
    acc = __dp4a(static_cast<int>((w.x >> 4) & 0x0F0F0F0Fu), pa.y, acc);
    acc = __dp4a(static_cast<int>(w.y & 0x0F0F0F0Fu), pa.z, acc);
    acc = __dp4a(static_cast<int>((w.y >> 4) & 0x0F0F0F0Fu), pa.w, acc);
    acc = __dp4a(static_cast<int>(w.z & 0x0F0F0F0Fu), pb.x, acc);
    acc = __dp4a(static_cast<int>((w.z >> 4) & 0x0F0F0F0Fu), pb.y, acc);
    acc = __dp4a(static_cast<int>(w.w & 0x0F0F0F0Fu), pb.z, acc);
    acc = __dp4a(static_cast<int>((w.w >> 4) & 0x0F0F0F0Fu), pb.w, acc);
    return acc;
}

// One CTA: columns [16 c, 16 c + 16) (rows r0 .. r0 + 15 of weight tile nt), all of K. Warp w: k-blocks
// [w kb_total / 8, (w + 1) kb_total / 8). Lane l: weight rows r0 + l / 4 and r0 + 8 + l / 4, 32 k at (l % 4) * 32.
template <int MR, bool kDebug>
__global__ void __launch_bounds__(kGemvThreads) msd_gemv_kernel(const GemvParams p) {
    __shared__ float red[kGemvWarps][MR][kGemvCols];
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N, K = p.K, G = p.G, kb_total = p.kb_total;
    const int Gn = K / G;
    const int col0 = blockIdx.x * kGemvCols;
    const int nt = col0 / kTileN, r0 = col0 % kTileN;
    const int chunk = lane & 3;
    const int lpg_chunks = G / 32;                     // lanes (chunks of 32 k) per group: 1, 2 or 4
    const int kbw0 = static_cast<int>(static_cast<int64_t>(warp) * kb_total / kGemvWarps);
    const int kbw1 = static_cast<int>(static_cast<int64_t>(warp + 1) * kb_total / kGemvWarps);
    const uint64_t policy = l2_policy_evict_first();
    const uint8_t *wbase = p.w + static_cast<size_t>(nt) * kb_total * kPackedTileBytes + (r0 + (lane >> 2)) * 64 +
                           chunk * 16;
    const int n_a = col0 + (lane >> 2), n_b = n_a + 8;
    float yacc[MR][2];
#pragma unroll
    for (int m = 0; m < MR; ++m) yacc[m][0] = yacc[m][1] = 0.0f;
    bool waited = false;

    for (int kp = kbw0; kp < kbw1; kp += kGemvKbPerPass) {
        const int nkb = min(kGemvKbPerPass, kbw1 - kp);
        // weights of the pass: rows a and b of each k-block, 16 bytes each, all requested before any use
        uint4 wa[kGemvKbPerPass], wb[kGemvKbPerPass];
        float sa[kGemvKbPerPass], sb[kGemvKbPerPass];
#pragma unroll
        for (int j = 0; j < kGemvKbPerPass; ++j) {
            if (j < nkb) {
                const uint8_t *src = wbase + static_cast<size_t>(kp + j) * kPackedTileBytes;
                wa[j] = ldg_stream16(src, policy);
                wb[j] = ldg_stream16(src + 8 * 64, policy);
                const int g = ((kp + j) * kKBlock + chunk * 32) / G;
                if (!kDebug) {
                    sa[j] = g < Gn && n_a < N ? __half2float(__ldg(p.scale + static_cast<size_t>(g) * N + n_a)) : 0.0f;
                    sb[j] = g < Gn && n_b < N ? __half2float(__ldg(p.scale + static_cast<size_t>(g) * N + n_b)) : 0.0f;
                }
            }
        }
        if (!waited) {
            pdl_wait();                                // the planes come from the unfold kernel
            waited = true;
        }
#pragma unroll
        for (int j = 0; j < kGemvKbPerPass; ++j) {
            if (j >= nkb) break;
            const int kb = kp + j;
            const int k0 = kb * kKBlock + chunk * 32;
            const int g = k0 / G;
            const bool live = k0 < K;                   // a ragged last k-block: chunks past K hold zeros
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                const int8_t *pl = p.planes + (static_cast<size_t>(m) * kb_total + kb) * kGemvPlaneBytes + chunk * 96;
                int da[3], db[3];
#pragma unroll
                for (int q = 0; q < 3; ++q) {
                    const int4 pa = __ldg(reinterpret_cast<const int4 *>(pl + q * 32));
                    const int4 pb = __ldg(reinterpret_cast<const int4 *>(pl + q * 32 + 16));
                    da[q] = dot32(wa[j], pa, pb, 0);
                    db[q] = dot32(wb[j], pa, pb, 0);
                }
                // lanes of one group (same weight row, consecutive chunks) add their dots
#pragma unroll
                for (int q = 0; q < 3; ++q) {
                    if (lpg_chunks >= 2) {
                        da[q] += __shfl_xor_sync(0xffffffffu, da[q], 1);
                        db[q] += __shfl_xor_sync(0xffffffffu, db[q], 1);
                    }
                    if (lpg_chunks >= 4) {
                        da[q] += __shfl_xor_sync(0xffffffffu, da[q], 2);
                        db[q] += __shfl_xor_sync(0xffffffffu, db[q], 2);
                    }
                }
                if (!live) continue;
                const float4 cr = __ldg(p.consts + static_cast<size_t>(m) * Gn + g);
                if (kDebug) {
                    // the constant record holds the plane sums: Y_i = dot_i - 8 S_i
                    if (g == p.dbg_group && (chunk & (lpg_chunks - 1)) == 0 && m < p.M) {
                        const float sv[3] = {cr.x, cr.y, cr.z};
#pragma unroll
                        for (int q = 0; q < 3; ++q) {
                            const int sq = __float2int_rn(sv[q]);
                            if (n_a < N) p.dbg_y123[(static_cast<size_t>(q) * p.M + m) * N + n_a] = da[q] - 8 * sq;
                            if (n_b < N) p.dbg_y123[(static_cast<size_t>(q) * p.M + m) * N + n_b] = db[q] - 8 * sq;
                        }
                    }
                    continue;
                }
                float ta = fmaf(cr.x, static_cast<float>(da[0]), -cr.w);
                ta = fmaf(cr.y, static_cast<float>(da[1]), ta);
                ta = fmaf(cr.z, static_cast<float>(da[2]), ta);
                float tb = fmaf(cr.x, static_cast<float>(db[0]), -cr.w);
                tb = fmaf(cr.y, static_cast<float>(db[1]), tb);
                tb = fmaf(cr.z, static_cast<float>(db[2]), tb);
                yacc[m][0] = fmaf(sa[j], ta, yacc[m][0]);
                yacc[m][1] = fmaf(sb[j], tb, yacc[m][1]);
            }
        }
    }
    if (!waited) pdl_wait();
    if constexpr (!kDebug) {
    // one value per group: the lanes of a group hold equal sums, so add one lane per group (fixed order)
#pragma unroll
    for (int m = 0; m < MR; ++m) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v = yacc[m][h];
            if (lpg_chunks == 1) v += __shfl_xor_sync(0xffffffffu, v, 1);
            if (lpg_chunks <= 2) v += __shfl_xor_sync(0xffffffffu, v, 2);
            yacc[m][h] = v;
        }
    }
    if (chunk == 0) {
#pragma unroll
        for (int m = 0; m < MR; ++m) {
            red[warp][m][lane >> 2] = yacc[m][0];
            red[warp][m][8 + (lane >> 2)] = yacc[m][1];
        }
    }
    __syncthreads();
    if (threadIdx.x < MR * kGemvCols) {
        const int m = threadIdx.x / kGemvCols, c = threadIdx.x % kGemvCols;
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < kGemvWarps; ++w) acc += red[w][m][c];
        const int n = col0 + c;
        if (m < p.M && n < N) p.y[static_cast<size_t>(m) * N + n] = __float2half_rn(acc);
    }
    }
}

}  // namespace wqbmm
