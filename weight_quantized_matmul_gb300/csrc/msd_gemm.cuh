// Large-M path of the A16W4 per-group MSD matmul (WeightQuantBatchMatmulExperiment page, section 4.1).
//
// When x has many rows, unfolding x inside every column-tile CTA would repeat the same work N/128 times, so the
// path is split in two kernels:
//   unfold_planes_kernel  steps 1-8 once per (row, k): the three residual planes as E4M3 bytes, written directly in
//                         the tensor-core operand layout (128-row x 128-k tiles, 128-byte swizzle, K-major), plus
//                         per-(row, group) constants {c1 A_max, c2 A_max, c3 A_max, 8 sum_i c_i A_max S_i}
//   msd_gemm_kernel       steps 9-11 for one 128-row x 128-column output tile per CTA: the planes are the MMA's A
//                         operand (M = 128 rows of x), the int4 weights converted to E4M3 the B operand (N = 128
//                         columns); each plane of each K-group accumulates in its own 128-column TMEM slot, four
//                         slots rotating
// Roles in msd_gemm_kernel (384 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps 2-3 int4 ->
// E4M3 converters (and fp16 -> fp32 scales), warps 4-11 epilogue (two warps per TMEM lane quarter, 64 columns each,
// packed FP32x2 math). The epilogue folds the planes of a group in one at a time (T = c1 D1 - corr, T += c2 D2,
// T += c3 D3, y += scale T) and hands each plane's slot back as soon as it has read it, so the MMAs can run up to
// three planes ahead of the epilogue.
// Every wait of the MMA-issuing thread leaves the tensor pipe idle for hundreds of cycles (measured: ~700 per wait
// when it waited once per plane, against ~75 per 128 x 128 x 32 MMA), so the MMA warp waits once per K-group, on a
// hardware named barrier, for everything the group's three planes need: the converters arrive there once the weights
// are converted and the epilogue has released the group's three TMEM slots. The MMA warp never gives up a wait;
// after a failed wait the other roles skip their work but keep every arrival, in order, so nothing waits forever.
#pragma once

#include "msd_kernels.cuh"

namespace wqbmm {

constexpr int kGemmTileM = 128;
constexpr int kGemmTileN = 128;
constexpr int kGemmThreads = 384;                              // 12 warps: 3 per SM sub-partition, 168 registers
constexpr int kGemmConvWarp0 = 2;
constexpr int kGemmNumConvWarps = 2;
constexpr int kGemmEpiWarp0 = 4;
constexpr int kGemmNumEpiWarps = 8;
constexpr int kGemmBStages = 2;
constexpr int kGemmSlots = 4;                                  // TMEM accumulator slots of 128 columns
constexpr int kGemmGroupBar0 = 2;                              // named barriers 2, 3: even / odd K-group ready
constexpr int kGemmGroupBarThreads = kGemmNumConvWarps * 32 + 32;
// Registers: launched with 168 per thread (384 x 168 = 64512); warps 0-3 (producer, MMA, converters) then give up
// to 96 and the two epilogue warpgroups take 200: 128 x 96 + 256 x 200 = 63488.
constexpr int kGemmLaunchRegs = 168;
constexpr uint32_t kGemmRolesRegs = 96;
constexpr uint32_t kGemmEpiRegs = 200;
static_assert(128 * kGemmRolesRegs + (kGemmThreads - 128) * kGemmEpiRegs <= kGemmThreads * kGemmLaunchRegs,
              "register split above the launch allocation");
constexpr int kPlaneImageBytes = kGemmTileM * kKBlock;         // 16384: one plane of one k-block
constexpr int kGemmConstRowBytes = 16;                         // float4 per (row, group)
constexpr int kGemmSmemLimit = 232448;                         // opt-in shared memory per CTA on sm_103

// Shared-memory layout of msd_gemm_kernel (depends on the group size through the groups per k-block, and on whether
// zero points are staged).
struct GemmLayout {
    int gpk, const_bytes, scale_bytes, stage_bytes, p_stages;
    int off_const, off_scale, off_scale32, off_zp, off_zp32, off_p, off_b, off_bar, off_misc, smem_bytes;
    __host__ __device__ static int align(int v, int a) { return (v + a - 1) / a * a; }
    __host__ __device__ GemmLayout(int G, bool zp) {
        gpk = kKBlock / G;
        const_bytes = gpk * kGemmTileM * kGemmConstRowBytes;
        scale_bytes = gpk * kGemmTileN * 2;
        // stage: three plane images | packed weight tile | constants | scale tile (fp16, as loaded) | scale (fp32)
        //        [| zero-point tile (fp16, as loaded) | 1 + zp / 8 (fp32)]
        off_const = 3 * kPlaneImageBytes + kPackedTileBytes;
        off_scale = off_const + const_bytes;
        off_scale32 = off_scale + scale_bytes;
        off_zp = off_scale32 + 2 * scale_bytes;
        off_zp32 = off_zp + scale_bytes;
        stage_bytes = align(zp ? off_zp32 + 2 * scale_bytes : off_zp, 1024);
        off_b = 0;                                             // converted weights ring first (1024-aligned)
        off_p = kGemmBStages * (kGemmTileN * kKBlock);
        const int fixed = off_p + 1024 /*align slack*/ + 512 /*barriers and flags*/;
        p_stages = (kGemmSmemLimit - fixed) / stage_bytes;
        if (p_stages > 3) p_stages = 3;
        off_bar = off_p + p_stages * stage_bytes;
        off_misc = off_bar + 8 * (3 * 3 + kGemmBStages + 2 * kGemmSlots);
        smem_bytes = off_misc + 64 + 1024;
    }
};

struct GemmParams {
    const uint8_t *w;           // prepacked tiles
    const uint8_t *planes;      // [m_tiles][kb_total][3][16 KB] from unfold_planes_kernel
    const float4 *consts;       // [m_tiles][K/G][128 rows]
    const __half *bias;         // [N] or null
    __half *y;
    int32_t *dbg_y123;          // debug: integer partials of group dbg_group, else null
    int M, K, N, G;
    int m_tiles, n_tiles, kb_total;
    int dbg_group;              // -1 in normal runs
};

// Steps 1-8 for one row and one 128-k block per warp. Planes go to the operand images, constants to the table; rows
// past M (padding of the last 128-row tile) get zero planes and zero constants. In debug mode the constant record
// holds the plane sums {S1, S2, S3, 0} instead.
__global__ void __launch_bounds__(256) unfold_planes_kernel(const __half *__restrict__ x, int M, int K, int G,
                                                            int kb_total, uint8_t *__restrict__ planes,
                                                            float4 *__restrict__ consts, int debug,
                                                            const float *__restrict__ row_amax) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);        // row within the padded rows
    const int kb = blockIdx.y;
    const int mt = row / kGemmTileM, r = row % kGemmTileM;
    const int kbase = kb * kKBlock + lane * 4;
    const int lpg = G / 4;
    const int Gn = K / G;
    float v[4];
    load_x4(x, M, K, row, kbase, v);
    float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    am = group_absmax(am, lpg);
    if (row_amax != nullptr) am = row < M ? row_amax[row] : 0.0f;   // per channel: the whole row's maximum
    float a1[4], a2[4], a3[4];
    msd_unfold4(v, am, a1, a2, a3);
    const int s1 = group_isum(__float2int_rn((a1[0] + a1[1]) + (a1[2] + a1[3])), lpg);
    const int s2 = group_isum(__float2int_rn((a2[0] + a2[1]) + (a2[2] + a2[3])), lpg);
    const int s3 = group_isum(__float2int_rn((a3[0] + a3[1]) + (a3[2] + a3[3])), lpg);
    uint8_t *img = planes + (static_cast<size_t>(mt) * kb_total + kb) * 3 * kPlaneImageBytes;
    const uint32_t off = sw128_offset(r, lane * 4);
    *reinterpret_cast<uint32_t *>(img + off) = e4m3x2(a1[1], a1[0]) | (e4m3x2(a1[3], a1[2]) << 16);
    *reinterpret_cast<uint32_t *>(img + kPlaneImageBytes + off) = e4m3x2(a2[1], a2[0]) | (e4m3x2(a2[3], a2[2]) << 16);
    *reinterpret_cast<uint32_t *>(img + 2 * kPlaneImageBytes + off) =
        e4m3x2(a3[1], a3[0]) | (e4m3x2(a3[3], a3[2]) << 16);
    const int g = kb * (kKBlock / G) + lane / lpg;
    if ((lane & (lpg - 1)) == 0 && g < Gn) {
        float4 rec;
        if (debug) {
            rec = make_float4(static_cast<float>(s1), static_cast<float>(s2), static_cast<float>(s3), 0.0f);
        } else {
            const float c1 = kC1 * am, c2 = kC2 * am, c3 = kC3 * am;
            rec = make_float4(kMmaUnit * c1, kMmaUnit * c2, kMmaUnit * c3, 8.0f * (c1 * s1 + c2 * s2 + c3 * s3));
        }
        consts[(static_cast<size_t>(mt) * Gn + g) * kGemmTileM + r] = rec;
    }
}

__device__ __forceinline__ float2 ld_scale2(const uint8_t *p) {
    return __half22float2(*reinterpret_cast<const __half2 *>(p));
}

__device__ __forceinline__ uint32_t pack_half2(float2 v) {
    const __half2 h = __float22half2_rn(v);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// kDebug: only the k-block of group p.dbg_group runs, the constant records hold the plane sums, and the epilogue
// writes that group's integer partials instead of y.
// kZp: zero-point tiles ride with the scale tiles; the converters turn them into 1 + zp / 8, the factor of the
// offset correction when the quantized weight is w - zp (the dots then need (8 + zp) S_i taken off).
template <bool kDebug, bool kZp>
__global__ void __launch_bounds__(kGemmThreads, 1)
    msd_gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap tmap_s,
                    const __grid_constant__ CUtensorMap tmap_z) {
    const GemmLayout L(p.G, kZp);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *b_ring = smem + L.off_b;
    uint8_t *p_ring = smem + L.off_p;
    const int P = L.p_stages;
    const uint32_t bar0 = smem_addr(smem + L.off_bar);
    // barriers: full_p / empty_p  load stage landed / released (MMAs done with the planes, converters with the
    //                             weights, epilogue with constants and scales)
    //           sready            scales of the stage converted to fp32 (the epilogue's view of the stage)
    //           bfree             converted weight stage consumed by the MMAs (their commit)
    //           tfull / trel      TMEM slot written by the MMAs (their commit) / read by the epilogue
    // and the named barriers kGemmGroupBar0 + (j & 1): everything K-group j of the CTA needs is ready (the converters
    // arrive, the MMA warp waits).
    auto full_p = [&](int s) { return bar0 + 8u * s; };
    auto empty_p = [&](int s) { return bar0 + 8u * (3 + s); };
    auto sready = [&](int s) { return bar0 + 8u * (6 + s); };
    auto bfree = [&](int c) { return bar0 + 8u * (9 + c); };
    auto tfull = [&](int t) { return bar0 + 8u * (9 + kGemmBStages + t); };
    auto trel = [&](int t) { return bar0 + 8u * (9 + kGemmBStages + kGemmSlots + t); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x, nt = blockIdx.y;       // row tiles vary fastest: CTAs in flight share weight tiles
    const int K = p.K, N = p.N, G = p.G, M = p.M;
    const int gpk = L.gpk;
    const int Gn = K / G;
    const int kb0 = kDebug ? p.dbg_group * G / kKBlock : 0;
    const int nkb = kDebug ? 1 : p.kb_total;

    const int gshift = 31 - __clz(G);                  // G is 32, 64 or 128
    auto groups_in = [&](int kb) { return (min(K, (kb + 1) * kKBlock) - kb * kKBlock) >> gshift; };
    // plane-accumulation units of this CTA: three per group, unit u in TMEM slot u % kGemmSlots
    const int total_units = 3 * (kDebug ? groups_in(kb0) : Gn);
    auto stage_tx = [&](int kb) {
        return static_cast<uint32_t>(3 * kPlaneImageBytes + kPackedTileBytes + groups_in(kb) * kGemmTileM * 16 +
                                     (kDebug ? 0 : (kZp ? 2 : 1) * gpk * kGemmTileN * 2));
    };
    // read-only inputs of the call (weights, scales) may be fetched before the preceding kernel (the unfold) ends
    auto issue_static = [&](int i, uint64_t pol_stream, uint64_t pol_keep) {
        const int s = i % P, kb = kb0 + i;
        const uint32_t dst = smem_addr(p_ring + s * L.stage_bytes);
        mbar_arrive_expect_tx(full_p(s), stage_tx(kb));
        bulk_g2s(dst + 3 * kPlaneImageBytes, p.w + (static_cast<size_t>(nt) * p.kb_total + kb) * kPackedTileBytes,
                 kPackedTileBytes, full_p(s), pol_stream);
        if (!kDebug) tma_load_2d(dst + L.off_scale, &tmap_s, nt * kGemmTileN, kb * gpk, full_p(s), pol_keep);
        if (kZp && !kDebug) tma_load_2d(dst + L.off_zp, &tmap_z, nt * kGemmTileN, kb * gpk, full_p(s), pol_keep);
    };
    auto issue_dynamic = [&](int i, uint64_t pol_keep) {
        const int s = i % P, kb = kb0 + i;
        const uint32_t dst = smem_addr(p_ring + s * L.stage_bytes);
        bulk_g2s(dst, p.planes + (static_cast<size_t>(mt) * p.kb_total + kb) * 3 * kPlaneImageBytes,
                 3 * kPlaneImageBytes, full_p(s), pol_keep);
        bulk_g2s(dst + L.off_const, p.consts + (static_cast<size_t>(mt) * Gn + kb * gpk) * kGemmTileM,
                 groups_in(kb) * kGemmTileM * 16, full_p(s), pol_keep);
    };
    // named barrier of K-group j, with compile-time ids
    auto group_bar = [&](int j, bool wait) {
        if (wait) {
            if ((j & 1) == 0) named_bar_sync(kGemmGroupBar0, kGemmGroupBarThreads);
            else named_bar_sync(kGemmGroupBar0 + 1, kGemmGroupBarThreads);
        } else {
            if ((j & 1) == 0) named_bar_arrive(kGemmGroupBar0, kGemmGroupBarThreads);
            else named_bar_arrive(kGemmGroupBar0 + 1, kGemmGroupBarThreads);
        }
    };

    const int first = nkb < P ? nkb : P;
    uint64_t pol_stream = 0, pol_keep = 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < P; ++s) {
            mbar_init(full_p(s), 1);
            mbar_init(empty_p(s), 1 + kGemmNumConvWarps + kGemmNumEpiWarps);
            mbar_init(sready(s), kGemmNumConvWarps);
        }
        for (int c = 0; c < kGemmBStages; ++c) mbar_init(bfree(c), 1);
        for (int t = 0; t < kGemmSlots; ++t) {
            mbar_init(tfull(t), 1);
            mbar_init(trel(t), kGemmNumEpiWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
        pol_stream = l2_policy_evict_first();
        pol_keep = l2_policy_evict_last();
        prefetch_tensormap(&tmap_s);
        if (kZp) prefetch_tensormap(&tmap_z);
        pdl_launch_dependents();
        for (int i = 0; i < first; ++i) issue_static(i, pol_stream, pol_keep);
        pdl_wait();
        for (int i = 0; i < first; ++i) issue_dynamic(i, pol_keep);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < kGemmEpiWarp0) {
      regs_release<kGemmRolesRegs>();
      if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            int issued = first;
            for (; issued < nkb; ++issued) {
                const int s = issued % P;
                if (!mbar_wait(empty_p(s), ((issued / P) & 1) ^ 1, abort_flag, kSiteProducerEmpty)) break;
                issue_static(issued, pol_stream, pol_keep);
                issue_dynamic(issued, pol_keep);
            }
            for (int j = issued > P ? issued - P : 0; j < issued; ++j) mbar_wait_drain(full_p(j % P), (j / P) & 1);
        }
      } else if (warp == 1) {
        // ================================================================ MMA issuer (the whole warp takes the
        // named barriers, lane 0 issues)
        constexpr uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(kGemmTileN >> 3) << 17) |
                                   (static_cast<uint32_t>(kGemmTileM >> 4) << 24);
        int j = 0;                                       // K-group counter of the CTA
        for (int i = 0; i < nkb; ++i) {
            const int s = i % P, cb = i % kGemmBStages;
            const uint32_t plane_base = smem_addr(p_ring + s * L.stage_bytes);
            const uint32_t w_base = smem_addr(b_ring + cb * (kGemmTileN * kKBlock));
            const int ng = groups_in(kb0 + i);
            for (int gg = 0; gg < ng; ++gg, ++j) {
                // the weights of k-block i are converted (so its stage has landed) and the three TMEM slots of
                // group j have been read
                group_bar(j, true);
                if (lane == 0) {
                    tc_fence_after_sync();
                    for (int pl = 0; pl < 3; ++pl) {
                        const int t = (3 * j + pl) % kGemmSlots;
                        const uint32_t d = tmem_base + static_cast<uint32_t>(t * kGemmTileN);
                        for (int ks = 0; ks < G / 32; ++ks) {
                            const uint32_t kofs = static_cast<uint32_t>(gg * G + ks * 32);
                            umma_f8f6f4(d, sdesc_kmajor_sw128(plane_base + pl * kPlaneImageBytes + kofs),
                                        sdesc_kmajor_sw128(w_base + kofs), idesc, ks > 0 ? 1u : 0u);
                        }
                        umma_commit(tfull(t));
                    }
                }
                __syncwarp();
            }
            if (lane == 0) {
                umma_commit(bfree(cb));
                umma_commit(empty_p(s));
            }
            __syncwarp();
        }
        // no MMA may still be writing TMEM when it is freed, nor arrive on a barrier after the CTA exits
        if (lane == 0)
            for (int v = total_units > kGemmSlots ? total_units - kGemmSlots : 0; v < total_units; ++v)
                mbar_wait_drain(tfull(v % kGemmSlots), (v / kGemmSlots) & 1);
        __syncwarp();
      } else {
        // ================================================================ int4 -> E4M3 converters, scales to fp32
        const int ct = threadIdx.x - kGemmConvWarp0 * 32;
        constexpr int kConvThreads = kGemmNumConvWarps * 32;
        bool ok = true;
        int j = 0;                                       // K-group counter of the CTA
        for (int i = 0; i < nkb; ++i) {
            const int s = i % P, cb = i % kGemmBStages;
            if (ok) ok = mbar_wait_warp(full_p(s), (i / P) & 1, abort_flag, kSiteConvFull);
            uint8_t *stage = p_ring + s * L.stage_bytes;
            if (ok && !kDebug) {
                const __half2 *s16 = reinterpret_cast<const __half2 *>(stage + L.off_scale);
                float2 *s32 = reinterpret_cast<float2 *>(stage + L.off_scale32);
                for (int e = ct; e < gpk * kGemmTileN / 2; e += kConvThreads) s32[e] = __half22float2(s16[e]);
                if constexpr (kZp) {
                    const __half2 *z16 = reinterpret_cast<const __half2 *>(stage + L.off_zp);
                    float2 *z32 = reinterpret_cast<float2 *>(stage + L.off_zp32);
                    for (int e = ct; e < gpk * kGemmTileN / 2; e += kConvThreads) {
                        const float2 z = __half22float2(z16[e]);
                        z32[e] = make_float2(fmaf(z.x, 0.125f, 1.0f), fmaf(z.y, 0.125f, 1.0f));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sready(s));
            }
            // the weight stage is free once the MMAs of k-block i - 2 are done. Waited for even after a failure
            // (bounded; the MMA warp never stops issuing), so that this warp never arrives on a group barrier
            // twice before the MMA warp has waited there once.
            const uint32_t par = ((i / kGemmBStages) & 1) ^ 1;
            if (ok) ok = mbar_wait_warp(bfree(cb), par, abort_flag, kSiteConvEmpty);
            if (!ok) {
                bool drained = true;
                if (lane == 0) drained = mbar_wait_drain(bfree(cb), par);
                (void)__shfl_sync(0xffffffffu, drained ? 1 : 0, 0);
            }
            if (ok) {
                convert_tile<kConvThreads>(stage + 3 * kPlaneImageBytes, b_ring + cb * (kGemmTileN * kKBlock), ct);
                fence_proxy_async_smem();
            }
            __syncwarp();
            // per K-group: its three planes go to slots last used by units 3j - 4 .. 3j - 2, which the epilogue
            // releases in order. Waited for even after a failure, for the same reason as above.
            const int ng = groups_in(kb0 + i);
            for (int gg = 0; gg < ng; ++gg, ++j) {
                const int v = 3 * j - 2;
                if (v >= 0) {
                    const uint32_t vpar = (v / kGemmSlots) & 1;
                    if (ok) ok = mbar_wait_warp(trel(v % kGemmSlots), vpar, abort_flag, kSiteConvEmpty);
                    if (!ok) {
                        bool drained = true;
                        if (lane == 0) drained = mbar_wait_drain(trel(v % kGemmSlots), vpar);
                        (void)__shfl_sync(0xffffffffu, drained ? 1 : 0, 0);
                    }
                }
                group_bar(j, false);
            }
            if (ok && lane == 0) mbar_arrive(empty_p(s));
        }
      }
    } else {
        // ================================================================ epilogue
        regs_claim<kGemmEpiRegs>();
        pdl_wait();
        const int ew = warp - kGemmEpiWarp0;             // 0..7
        const int quarter = warp & 3;                    // TMEM lanes (rows) this warp may read
        const int half = ew >> 2;                        // columns [64 half, 64 half + 64) of each slot
        const int r = quarter * 32 + lane;               // row within the tile
        const int m = mt * kGemmTileM + r;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        float2 yacc[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) yacc[q] = make_float2(0.0f, 0.0f);
        bool ok = true;
        // waits for the MMAs of unit uu; after a failure it still waits (bounded, the MMA warp never stops issuing)
        // so that no release runs ahead of the MMAs it frees the slot from
        auto wait_unit = [&](int uu) {
            const int t = uu % kGemmSlots;
            const uint32_t par = (uu / kGemmSlots) & 1;
            if (ok) ok = mbar_wait_warp(tfull(t), par, abort_flag, kSiteEpiTmemFull);
            if (!ok) {
                bool drained = true;
                if (lane == 0) drained = mbar_wait_drain(tfull(t), par);
                (void)__shfl_sync(0xffffffffu, drained ? 1 : 0, 0);
            }
        };
        // 32 columns of the warp's lane quarter: two loads in flight per wait
        auto ld32 = [&](uint32_t taddr, uint32_t(&dd)[2][16]) {
            tmem_ld16(taddr, dd[0]);
            tmem_ld16(taddr + 16, dd[1]);
            tmem_wait_ld();
            reg_fence16(dd[0]);
            reg_fence16(dd[1]);
        };
        auto release_unit = [&](int uu) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(trel(uu % kGemmSlots));
        };
        int u = 0;
        for (int i = 0; i < nkb; ++i) {
            const int s = i % P, kb = kb0 + i;
            // the epilogue reads constants (landed with the stage) and fp32 scales (written by the converters)
            if (ok)
                ok = kDebug ? mbar_wait_warp(full_p(s), (i / P) & 1, abort_flag, kSiteEpiOperandsEmpty)
                            : mbar_wait_warp(sready(s), (i / P) & 1, abort_flag, kSiteEpiOperandsEmpty);
            const uint8_t *stage = p_ring + s * L.stage_bytes;
            const int ng = groups_in(kb);
            for (int gg = 0; gg < ng; ++gg, u += 3) {
                const float4 cr = ok ? lds_f128(smem_addr(stage + L.off_const) + 16 * (gg * kGemmTileM + r))
                                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (kDebug) {
                    // warp-uniform: tcgen05.ld is executed by the whole warp; rows past M only skip the stores
                    const bool here = kb * gpk + gg == p.dbg_group;
                    const float splane[3] = {cr.x, cr.y, cr.z};   // debug records hold the plane sums
#pragma unroll 1
                    for (int pl = 0; pl < 3; ++pl) {
                        const int t = (u + pl) % kGemmSlots;
                        wait_unit(u + pl);
                        if (ok && here) {
                            tc_fence_after_sync();
                            const uint32_t a = tmem_base + lane_off + static_cast<uint32_t>(t * kGemmTileN + half * 64);
#pragma unroll 1
                            for (int ch = 0; ch < 4; ++ch) {
                                uint32_t d[16];
                                tmem_ld16(a + ch * 16, d);
                                tmem_wait_ld();
                                reg_fence16(d);
                                for (int q = 0; q < 16; ++q) {
                                    const int n = nt * kGemmTileN + half * 64 + ch * 16 + q;
                                    if (m < M && n < N)
                                        p.dbg_y123[(static_cast<size_t>(pl) * M + m) * N + n] =
                                            __float2int_rn(kMmaUnit * __uint_as_float(d[q]) - 8.0f * splane[pl]);
                                }
                            }
                        }
                        release_unit(u + pl);
                    }
                    continue;
                }
                // scales (and 1 + zp / 8) of the warp's 64 columns, as 32-bit shared-window addresses
                const uint32_t srow = smem_addr(stage + L.off_scale32) + 4 * (gg * kGemmTileN + half * 64);
                const uint32_t zrow = smem_addr(stage + L.off_zp32) + 4 * (gg * kGemmTileN + half * 64);
                float2 T[32];
                // plane 1: T = c1 D1 - corr (times 1 + zp / 8 per column with zero points)
                {
                    const int t = u % kGemmSlots;
                    wait_unit(u);
                    if (ok) {
                        tc_fence_after_sync();
                        const uint32_t a = tmem_base + lane_off + static_cast<uint32_t>(t * kGemmTileN + half * 64);
                        const float2 c1 = make_float2(cr.x, cr.x), nc = make_float2(-cr.w, -cr.w);
#pragma unroll
                        for (int ch2 = 0; ch2 < 2; ++ch2) {
                          uint32_t dd[2][16];
                          ld32(a + ch2 * 32, dd);
#pragma unroll
                          for (int sub = 0; sub < 2; ++sub) {
                            const int ch = ch2 * 2 + sub;
                            const uint32_t(&d)[16] = dd[sub];
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                float4 zf = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
                                if constexpr (kZp) zf = lds_f128(zrow + 16 * (ch * 4 + q4));
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int q = q4 * 2 + h;
                                    const float2 v =
                                        make_float2(__uint_as_float(d[2 * q]), __uint_as_float(d[2 * q + 1]));
                                    float2 ncz = nc;
                                    if constexpr (kZp)
                                        ncz = __fmul2_rn(nc, h == 0 ? make_float2(zf.x, zf.y)
                                                                    : make_float2(zf.z, zf.w));
                                    T[ch * 8 + q] = __ffma2_rn(c1, v, ncz);
                                }
                            }
                          }
                        }
                    }
                    release_unit(u);
                }
                // plane 2: T += c2 D2
                {
                    const int t = (u + 1) % kGemmSlots;
                    wait_unit(u + 1);
                    if (ok) {
                        tc_fence_after_sync();
                        const uint32_t a = tmem_base + lane_off + static_cast<uint32_t>(t * kGemmTileN + half * 64);
                        const float2 c2 = make_float2(cr.y, cr.y);
#pragma unroll
                        for (int ch2 = 0; ch2 < 2; ++ch2) {
                          uint32_t dd[2][16];
                          ld32(a + ch2 * 32, dd);
#pragma unroll
                          for (int sub = 0; sub < 2; ++sub) {
                            const int ch = ch2 * 2 + sub;
                            const uint32_t(&d)[16] = dd[sub];
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                T[ch * 8 + q] = __ffma2_rn(
                                    c2, make_float2(__uint_as_float(d[2 * q]), __uint_as_float(d[2 * q + 1])),
                                    T[ch * 8 + q]);
                          }
                        }
                    }
                    release_unit(u + 1);
                }
                // plane 3: T += c3 D3, then y += scale T
                {
                    const int t = (u + 2) % kGemmSlots;
                    wait_unit(u + 2);
                    if (ok) {
                        tc_fence_after_sync();
                        const uint32_t a = tmem_base + lane_off + static_cast<uint32_t>(t * kGemmTileN + half * 64);
                        const float2 c3 = make_float2(cr.z, cr.z);
#pragma unroll
                        for (int ch2 = 0; ch2 < 2; ++ch2) {
                          uint32_t dd[2][16];
                          ld32(a + ch2 * 32, dd);
#pragma unroll
                          for (int sub = 0; sub < 2; ++sub) {
                            const int ch = ch2 * 2 + sub;
                            const uint32_t(&d)[16] = dd[sub];
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const float4 sc = lds_f128(srow + 16 * (ch * 4 + q4));   // one address: broadcast
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int q = q4 * 2 + h;
                                    const float2 v =
                                        make_float2(__uint_as_float(d[2 * q]), __uint_as_float(d[2 * q + 1]));
                                    const float2 tq = __ffma2_rn(c3, v, T[ch * 8 + q]);
                                    const float2 scv = h == 0 ? make_float2(sc.x, sc.y) : make_float2(sc.z, sc.w);
                                    yacc[ch * 8 + q] = __ffma2_rn(scv, tq, yacc[ch * 8 + q]);
                                }
                            }
                          }
                        }
                    }
                    release_unit(u + 2);
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(empty_p(s));
        }
        if (!kDebug && ok && m < M) {
            __half *yrow = p.y + static_cast<size_t>(m) * N;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const int n = nt * kGemmTileN + half * 64 + c8 * 8;
                if (n < N) {
                    if (p.bias != nullptr) {
                        // the same 8 bias values for every row of the tile (L1 hits after the first warp)
                        const uint4 braw = *reinterpret_cast<const uint4 *>(p.bias + n);
                        const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            yacc[c8 * 4 + q] = __fadd2_rn(yacc[c8 * 4 + q],
                                                          __half22float2(*reinterpret_cast<const __half2 *>(&bw[q])));
                    }
                    const uint4 o = make_uint4(pack_half2(yacc[c8 * 4 + 0]), pack_half2(yacc[c8 * 4 + 1]),
                                               pack_half2(yacc[c8 * 4 + 2]), pack_half2(yacc[c8 * 4 + 3]));
                    *reinterpret_cast<uint4 *>(yrow + n) = o;
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace wqbmm
