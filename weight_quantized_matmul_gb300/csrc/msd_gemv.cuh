// Decode path of the A16W4 per-group MSD matmul (WeightQuantBatchMatmulExperiment page, section 4.1), for one or two
// rows of x: a matrix-vector product bound by reading the weights once from HBM. The three integer products
// Y_i = A_i . W_g are 4-way int8 dot products on the CUDA cores (dp4a), exact in int32.
//
//   gemv_unfold_kernel  steps 1-8 once per (row, 128 k): the three planes as int8 and, per (row, group), the combine
//                       constants {c1 A_max, c2 A_max, c3 A_max, 8 sum_i c_i A_max S_i} (debug: {S1, S2, S3, 0})
//   msd_gemv_kernel     steps 9-11 for 16 output columns over all of K per CTA: no split over K, so no reduction
//                       between CTAs. Each warp takes an eighth of the k-blocks; a lane streams 16-byte pieces of two
//                       weight rows straight into registers (issued before waiting for the unfold, so the weight
//                       stream overlaps it) and takes two dp4a per 32-bit weight word and plane, of its low nibbles
//                       and of the whole word (u = w + 8 per nibble): dot_i = 16 sum A_i u = 16 (Y_i + 8 S_i).
//                       Lanes that share a group add their dots, every lane applies the combine and the scale, and
//                       the partial sums of the lanes and warps are added in a fixed order, so the result does not
//                       depend on timing.
// Both kernels run under programmatic launch: the unfold waits for the preceding kernel before reading x, the GEMV
// kernel fetches weights and scales at once and waits for the unfold before reading the planes.
#pragma once

#include "msd_kernels.cuh"

namespace wqbmm {

constexpr int kGemvMaxRows = 2;
constexpr int kGemvCols = 16;                       // output columns per CTA
constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvKbPerPass = 8;                   // k-blocks per warp held in registers at a time (at most)
constexpr int kGemvPlaneBytes = 3 * kKBlock;        // one row, one k-block: [chunk 4][plane 3][32 bytes]
constexpr float kDotUnitInv = 1.0f / 16.0f;          // the dot products come out as 16 sum_k A_i u

// Steps 1-8 for one row and one 128-k block per warp (lane: 4 k). Planes to [row][kb][chunk][plane][32 B] as int8
// (low-nibble positions as 16 A_lo - A_hi, below), constants to [row][group] (float4).
__global__ void __launch_bounds__(128) gemv_unfold_kernel(const __half *__restrict__ x, int M, int K, int G,
                                                          int kb_total, int8_t *__restrict__ planes,
                                                          float4 *__restrict__ consts, int debug,
                                                          const float *__restrict__ row_amax) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int kb = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int row = blockIdx.y;
    // the warp's 256 bytes of x (two lines) on their way to L2 while the preceding kernel finishes
    if (kb < kb_total && (lane & 15) == 0 && kb * kKBlock + lane * 4 < K)
        prefetch_l2(x + static_cast<size_t>(row) * K + kb * kKBlock + lane * 4);
    pdl_wait();                                        // x may be the preceding kernel's output
    if (kb >= kb_total) return;                        // whole warps only
    const int lpg = G / 4;
    float v[4];
    load_x4(x, M, K, row, kb * kKBlock + lane * 4, v);
    float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    am = group_absmax(am, lpg);
    if (row_amax != nullptr) am = row_amax[row];                     // per channel: the whole row's maximum
    float a1[4], a2[4], a3[4];
    msd_unfold4(v, am, a1, a2, a3);
    const int s1 = group_isum(__float2int_rn((a1[0] + a1[1]) + (a1[2] + a1[3])), lpg);
    const int s2 = group_isum(__float2int_rn((a2[0] + a2[1]) + (a2[2] + a2[3])), lpg);
    const int s3 = group_isum(__float2int_rn((a3[0] + a3[1]) + (a3[2] + a3[3])), lpg);
    // k = 8q .. 8q + 3 (even lanes) meet the low nibbles lo of a weight word w, k = 8q + 4 .. 8q + 7 (odd lanes) the
    // high nibbles hi, byte for byte. The GEMV takes two dp4a per word, of lo = w & 0x0F0F0F0F against D and of w
    // itself (lo + 16 hi per byte) against H: with D = 16 A_lo - A_hi (|D| <= 119 fits int8) and H = A_hi that is
    // sum lo (16 A_lo - A_hi) + sum (lo + 16 hi) A_hi = 16 (sum lo A_lo + sum hi A_hi), exact in int32
    auto pack4 = [lane](const float (&a)[4]) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int mine = static_cast<int>(a[j]);
            const int hi = __shfl_down_sync(0xffffffffu, mine, 1);      // the same byte of the high positions
            const int v = (lane & 1) ? mine : 16 * mine - hi;
            word |= (static_cast<uint32_t>(v) & 0xFFu) << (8 * j);
        }
        return word;
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
            rec = make_float4(c1 * kDotUnitInv, c2 * kDotUnitInv, c3 * kDotUnitInv,        // exact: 1/16
                              8.0f * (c1 * static_cast<float>(s1) + c2 * static_cast<float>(s2) +
                                      c3 * static_cast<float>(s3)));
        }
        consts[static_cast<size_t>(row) * Gn + g] = rec;
    }
}

struct GemvParams {
    const uint8_t *w;           // prepacked tiles
    const __half *scale;        // [K/G, N]
    const __half *zp;           // [K/G, N] zero points (kernel instantiated with kZp), else null
    int group_stride;           // elements between the scale (zero-point) rows of consecutive groups: N, or 0 when
                                // one row serves every sub-group (per-channel quantization)
    const __half *bias;         // [N] or null
    const int8_t *planes;       // from gemv_unfold_kernel
    const float4 *consts;
    __half *y;
    int32_t *dbg_y123;          // debug: integer partials of group dbg_group, else null
    int M, K, N, G, kb_total, dbg_group;
};

__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// 16 sum_k A[k] u[k] over a 16-byte weight piece (32 k) and its 32 plane bytes: per weight word the low nibbles
// against D = 16 A_lo - A_hi and the whole word (lo + 16 hi per byte) against A_hi (see gemv_unfold_kernel).
__device__ __forceinline__ int dot32(const uint4 w, const int4 pa, const int4 pb, int acc) {
    acc = dp4a_us(w.x & 0x0F0F0F0Fu, pa.x, acc);
    acc = dp4a_us(w.x, pa.y, acc);
    acc = dp4a_us(w.y & 0x0F0F0F0Fu, pa.z, acc);
    acc = dp4a_us(w.y, pa.w, acc);
    acc = dp4a_us(w.z & 0x0F0F0F0Fu, pb.x, acc);
    acc = dp4a_us(w.z, pb.y, acc);
    acc = dp4a_us(w.w & 0x0F0F0F0Fu, pb.z, acc);
    acc = dp4a_us(w.w, pb.w, acc);
    return acc;
}

// int -> float for |v| < 2^22 with one integer add and one float subtract (1.5 * 2^23 as the bias)
__device__ __forceinline__ float small_int_to_float(int v) {
    return __int_as_float(v + 0x4B400000) - 12582912.0f;
}

// One CTA: columns [16 c, 16 c + 16) (rows r0 .. r0 + 15 of weight tile nt), all of K, in passes of at most 64
// k-blocks. In a pass, warp w takes an eighth of the pass's k-blocks; lane l reads the adjacent weight rows
// r0 + 2 (l / 4) and r0 + 2 (l / 4) + 1, 32 k at (l % 4) * 32, so that its two columns' scales (and zero points)
// come in one 4-byte load. The pass's planes and constants are copied into shared memory in one bulk
// copy each (the planes of a k-block are read by every warp of every CTA).
constexpr int kGemvPassKb = kGemvWarps * kGemvKbPerPass;      // 64

template <int MR>
struct GemvSmem {
    int8_t planes[MR][kGemvPassKb * kGemvPlaneBytes];
    float4 consts[MR][kGemvPassKb * 4];
    float red[kGemvWarps][MR][kGemvCols];
    uint64_t bar;
    int abort_flag;
};

// kZp: the quantized weight is w - zp[g, n], so a group's dots need (8 + zp) S_i taken off instead of 8 S_i: the
// lane that applies the group's correction scales it by 1 + zp / 8.
// KB: k-blocks per warp and pass held in registers. 4 when every k-block fits in one pass of 32 (K <= 4096): the
// kernel then holds half the weight registers it would with 8 (measured: the decode shape's kernel 3.37 -> 3.20 us);
// 8 for longer K, which then takes fewer passes.
template <int MR, bool kDebug, bool kZp, int KB>
__global__ void __launch_bounds__(kGemvThreads, 2) msd_gemv_kernel(const GemvParams p) {
    static_assert(KB == 4 || KB == kGemvKbPerPass, "4 or 8 k-blocks per warp and pass");
    constexpr int kPassKb = kGemvWarps * KB;
    extern __shared__ __align__(128) uint8_t gemv_smem_raw[];
    GemvSmem<MR> &sm = *reinterpret_cast<GemvSmem<MR> *>(gemv_smem_raw);
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N, K = p.K, G = p.G, kb_total = p.kb_total;
    const int gshift = 31 - __clz(G);                  // G is 32, 64 or 128: group index = k >> gshift
    const int Gn = K >> gshift, gpk = kKBlock >> gshift;
    const int col0 = blockIdx.x * kGemvCols;
    const int nt = col0 / kTileN, r0 = col0 % kTileN;
    const int chunk = lane & 3;
    const int lpg_chunks = G / 32;                     // lanes (chunks of 32 k) per group: 1, 2 or 4
    const uint32_t bar = smem_addr(&sm.bar);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        sm.abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    const uint64_t policy = l2_policy_evict_first();
    const uint8_t *wbase = p.w + static_cast<size_t>(nt) * kb_total * kPackedTileBytes + (r0 + 2 * (lane >> 2)) * 64 +
                           chunk * 16;
    const int n_a = col0 + 2 * (lane >> 2), n_b = n_a + 1;     // N is even: n_a < N implies n_b < N
    float yacc[MR][2];
#pragma unroll
    for (int m = 0; m < MR; ++m) yacc[m][0] = yacc[m][1] = 0.0f;
    bool ok = true;

    int pass = 0;
    for (int pb = 0; pb < kb_total; pb += kPassKb, ++pass) {
        const int pn = min(kPassKb, kb_total - pb);
        const int kw0 = pb + warp * pn / kGemvWarps, kw1 = pb + (warp + 1) * pn / kGemvWarps;
        const int nkb = kw1 - kw0;
        // weights and scales of the warp's k-blocks, all requested before any use (the scales stay fp16 until
        // they are used, so no instruction waits for them here)
        uint4 wa[KB], wb[KB];
        __half2 sab[KB];                               // scales of columns a and b
        __half2 zab[KB];                               // zero points of columns a and b (first chunk lane of a group)
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            if (j < nkb) {
                const uint8_t *src = wbase + static_cast<size_t>(kw0 + j) * kPackedTileBytes;
                wa[j] = ldg_stream16(src, policy);
                wb[j] = ldg_stream16(src + 64, policy);
            }
        }
        if (threadIdx.x == 0) {
            if (pass == 0) pdl_wait();                 // the planes come from the unfold kernel
            const int groups = min((pb + pn) * gpk, Gn) - pb * gpk;
            const uint32_t bytes = static_cast<uint32_t>(MR * pn * kGemvPlaneBytes + MR * groups * 16);
            mbar_arrive_expect_tx(bar, bytes);
            const uint64_t keep = l2_policy_evict_last();   // every CTA reads the same planes
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                bulk_g2s(smem_addr(sm.planes[m]), p.planes + (static_cast<size_t>(m) * kb_total + pb) * kGemvPlaneBytes,
                         static_cast<uint32_t>(pn * kGemvPlaneBytes), bar, keep);
                bulk_g2s(smem_addr(sm.consts[m]), p.consts + static_cast<size_t>(m) * Gn + pb * gpk,
                         static_cast<uint32_t>(groups * 16), bar, keep);
            }
        }
        if (!kDebug) {
#pragma unroll
            for (int j = 0; j < KB; ++j) {
                const int g = ((kw0 + j) * kKBlock + chunk * 32) >> gshift;
                const bool in = j < nkb && g < Gn;
                const size_t row_at = static_cast<size_t>(g) * p.group_stride + n_a;
                sab[j] = in && n_a < N ? __ldg(reinterpret_cast<const __half2 *>(p.scale + row_at))
                                       : __half2(0.0f, 0.0f);
                if constexpr (kZp) {
                    const bool first = in && n_a < N && (chunk & (lpg_chunks - 1)) == 0;
                    zab[j] = first ? __ldg(reinterpret_cast<const __half2 *>(p.zp + row_at)) : __half2(0.0f, 0.0f);
                }
            }
        }
        if (pass == 0 && threadIdx.x != 0) pdl_wait();
        ok = ok && mbar_wait_warp(bar, pass & 1, &sm.abort_flag, kSiteConvFull);
        if (ok) {
#pragma unroll
            for (int j = 0; j < KB; ++j) {
                if (j >= nkb) continue;                 // (not break: the loop stays fully unrolled)
                const int kb = kw0 + j, kbl = kb - pb;
                const int k0 = kb * kKBlock + chunk * 32;
                const int g = k0 >> gshift;
                const bool live = k0 < K;               // a ragged last k-block: chunks past K hold zeros
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    const int4 *pl = reinterpret_cast<const int4 *>(sm.planes[m] + kbl * kGemvPlaneBytes + chunk * 96);
                    int da[3], db[3];
#pragma unroll
                    for (int q = 0; q < 3; ++q) {
                        const int4 pa = pl[2 * q], pbv = pl[2 * q + 1];
                        da[q] = dot32(wa[j], pa, pbv, 0);
                        db[q] = dot32(wb[j], pa, pbv, 0);
                    }
                    if (kDebug) {
                        // lanes of one group (same weight row, consecutive chunks) add their dots
#pragma unroll
                        for (int q = 0; q < 3; ++q) {
                            for (int off = 1; off < lpg_chunks; off <<= 1) {
                                da[q] += __shfl_xor_sync(0xffffffffu, da[q], off);
                                db[q] += __shfl_xor_sync(0xffffffffu, db[q], off);
                            }
                        }
                    }
                    if (!live) continue;
                    const float4 cr = sm.consts[m][g - pb * gpk];
                    if (kDebug) {
                        // the constant record holds the plane sums: Y_i = dot_i / 16 - 8 S_i
                        if (g == p.dbg_group && (chunk & (lpg_chunks - 1)) == 0 && m < p.M) {
                            const float sv[3] = {cr.x, cr.y, cr.z};
#pragma unroll
                            for (int q = 0; q < 3; ++q) {
                                const int sq = __float2int_rn(sv[q]);
                                int32_t *dst = p.dbg_y123 + (static_cast<size_t>(q) * p.M + m) * N;
                                if (n_a < N) dst[n_a] = da[q] / 16 - 8 * sq;
                                if (n_b < N) dst[n_b] = db[q] / 16 - 8 * sq;
                            }
                        }
                        continue;
                    }
                    // this lane's share of the group: c_i times its own dots; the group's first chunk also takes
                    // the offset correction (the combine is linear, the lanes are added at the end)
                    const float corr = (chunk & (lpg_chunks - 1)) == 0 ? -cr.w : 0.0f;
                    float corr_a = corr, corr_b = corr;
                    if constexpr (kZp) {
                        const float2 z = __half22float2(zab[j]);
                        corr_a = corr * fmaf(z.x, 0.125f, 1.0f);
                        corr_b = corr * fmaf(z.y, 0.125f, 1.0f);
                    }
                    float ta = fmaf(cr.x, small_int_to_float(da[0]), corr_a);
                    ta = fmaf(cr.y, small_int_to_float(da[1]), ta);
                    ta = fmaf(cr.z, small_int_to_float(da[2]), ta);
                    float tb = fmaf(cr.x, small_int_to_float(db[0]), corr_b);
                    tb = fmaf(cr.y, small_int_to_float(db[1]), tb);
                    tb = fmaf(cr.z, small_int_to_float(db[2]), tb);
                    yacc[m][0] = fmaf(__low2float(sab[j]), ta, yacc[m][0]);
                    yacc[m][1] = fmaf(__high2float(sab[j]), tb, yacc[m][1]);
                }
            }
        }
        __syncthreads();                               // the next pass overwrites the planes
    }
    if (kb_total == 0) pdl_wait();
    if constexpr (!kDebug) {
        // the four chunk lanes of a weight row hold partial sums: add them (fixed order)
#pragma unroll
        for (int m = 0; m < MR; ++m) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = yacc[m][h];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                yacc[m][h] = v;
            }
        }
        if (chunk == 0) {
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                sm.red[warp][m][2 * (lane >> 2)] = yacc[m][0];
                sm.red[warp][m][2 * (lane >> 2) + 1] = yacc[m][1];
            }
        }
        __syncthreads();
        if (ok && threadIdx.x < MR * kGemvCols) {
            const int m = threadIdx.x / kGemvCols, c = threadIdx.x % kGemvCols;
            float acc = 0.0f;
#pragma unroll
            for (int w = 0; w < kGemvWarps; ++w) acc += sm.red[w][m][c];
            const int n = col0 + c;
            if (m < p.M && n < N) {
                if (p.bias != nullptr) acc += __half2float(p.bias[n]);
                p.y[static_cast<size_t>(m) * N + n] = __float2half_rn(acc);
            }
        }
    }
    // no bulk copy may still be writing shared memory when the CTA exits
    if (threadIdx.x == 0 && !ok) mbar_wait_drain(bar, (pass - 1) & 1);
}

}  // namespace wqbmm
