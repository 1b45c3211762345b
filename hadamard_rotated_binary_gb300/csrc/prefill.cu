// Tensor-core paths: Y[M][N] = per-group-scaled (+-1 W) x xt^T with tcgen05
// MMAs, bf16 operands and f32 accumulation in tensor memory.
//
// Method: the folded product of the Pulse "ARCHITECTURE-SPEC" Hadamard-fold
// section, y = W @ WHT(signs * P(x)), with W in the one-bit format of the
// "Inside the One-Bit Engine" page (first station; scale per 128 weights
// applied to each group's sum).  The rotation runs first (rotate.cu).
//
// Two modes of the same kernel:
//  * prefill (M >= 64): the B operand is xt rounded to bf16, one row per
//    token; CTA tile = 128 weight rows x BN tokens (BN = 64 up to 64 tokens,
//    else 128), tokens split over grid.y.
//  * exact (2 <= M < 64): the B operand holds, for token m, rows 4m..4m+2 =
//    the three bf16 digits hi, mid, lo of xt (hi = bf16(xt), mid =
//    bf16(xt - hi), lo = bf16(xt - hi - mid): together the f32 value) and row
//    4m+3 = 0.  Products with +-1 are exact, so summing the three digit
//    columns of D gives f32-level results.  A tile of BN rows holds BN/4
//    whole tokens.
//
// CTA tile: 128 weight rows (UMMA M = 128, one TMEM lane per row) x BN columns
// of B (UMMA N = BN).  The +-1 operand A lives in tensor memory, so shared
// memory holds only B tiles (deep enough to cover the ~1 us a copy from L2
// takes when every SM streams) and the packed bits.  Per 128-wide K-group g:
//   * warp 8 TMA-loads the B tile [BN rows][128 K] (one 3-d box: two
//     128-byte-swizzled 64-column halves); warp 14 TMA-loads the group's bits
//     [128 rows][4 words] (2 KB) into a ring that runs up to 8 groups ahead;
//   * warps 10-13 (one thread per weight row = TMEM lane) turn that row's 128
//     bits into 64 columns of bf16 pairs (+-1) and store them to the group's
//     A stage in tensor memory (tcgen05.st).  The repack stores even weights
//     in the low half-word and odd weights in the high half-word, so each
//     bf16x2 column is one shift and one XOR-mask;
//   * warp 9 waits for A, B and a free accumulator buffer (one round trip:
//     the three barriers are tested together); one elected lane issues 8
//     MMAs of K = 16 (A from tensor memory, B from shared memory) into buffer
//     g % 2, then commits to the group's "done" barrier (frees the A and B
//     stages) and the buffer's "full" barrier;
//   * warps 0-7 read the buffer back (tcgen05.ld), hand it back to the MMA
//     warp, and accumulate scale[n][g] * D into f32 registers - the per-group
//     scale promotion.  Warp w serves TMEM lanes 32*(w%4).. and the columns
//     BN/2*(w/4) .. BN/2*(w/4) + BN/2 - 1.  Scales are requested 4 groups ahead.
// Prefill grids of more than one wave run persistently: one CTA per SM takes
// tiles blockIdx.x, blockIdx.x + gridDim.x, ..., and every role counts its
// K-groups across those tiles, so the stages, barrier phases and accumulator
// buffers run on from one tile into the next (the epilogue writes a tile's y
// after its last group, while the MMAs of the next tile proceed).  The tiles
// past the last full wave, when they fill less than half of the SMs, run as a
// second launch with each tile split along K over a cluster.
// Every wait is bounded in time; on expiry the kernel stops its loops, drains
// its own copies and MMAs, frees TMEM and records a timeout in the handle's
// error word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bitlin_internal.cuh"
#include "ptx.cuh"

namespace {

using namespace bitlin_impl;

constexpr int kThreads = 480;       // 15 warps
constexpr int kEpiWarps = 8;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kExpWarp0 = 10;       // warps 10..13
constexpr int kBitsWarp = 14;
constexpr int kBitsBytes = 2048;    // one group's bits: 128 rows x 4 words
constexpr int kBitsStages = 8;      // bits run this many groups ahead of the expansion
constexpr int kACols = 64;          // one A stage: 128 lanes x 64 columns (128 bf16 per row)
constexpr int kTmemColsSM = 512;    // the SM's tensor memory (split between the CTAs an SM holds)
constexpr int kMaxSplits = 8;       // split-K clusters along grid.z (portable cluster size)

// OCC: CTAs per SM.  1: the whole tensor memory and about 200 KB of shared
// memory per CTA.  2 (64-column B tiles of the exact mode): half of each (two
// accumulator buffers and two A stages in 256 columns, five B stages, 64
// registers a thread), so that two CTAs overlap their per-group hand-offs on
// one SM: gate_up at M = 8 and 16 38.0 -> 33.0 us, attn_qkv at M = 16 (80
// tiles, split-K x3 at two per SM) 20.3 -> 19.3.  Used only where the tiles
// fill at least half of the SMs at one CTA per SM: below that (ffn_down at
// M = 16, 40 tiles) the doubled split count measured 32.1 against 25.9 us.
template <int BN, int OCC = 1>
struct Cfg {
    static constexpr int kTmemCols = kTmemColsSM / OCC;
    static constexpr int kBBytes = BN * 256;  // B tile: BN rows x 128 bf16
    static constexpr int kSmemBudget = (OCC == 1 ? 200 : 96) * 1024 - kBitsStages * kBitsBytes;
    static constexpr int kStagesB = kSmemBudget / kBBytes > 8 ? 8 : kSmemBudget / kBBytes;
    static constexpr int kStagesA = (kTmemCols - 2 * BN) / kACols > 6 ? 6 : (kTmemCols - 2 * BN) / kACols;
    static constexpr int kRing = kStagesA > kStagesB ? kStagesA : kStagesB;  // "done" barriers
    static_assert(kStagesB >= 3 && kStagesA >= 2, "pipeline depth");
};

template <int BN, int OCC>
struct __align__(8) Barriers {
    uint64_t fullB[Cfg<BN, OCC>::kStagesB];  // B tile landed (1 arrival + bytes)
    uint64_t fullA[Cfg<BN, OCC>::kStagesA];  // A stage written (128 arrivals: one thread per row)
    uint64_t done[Cfg<BN, OCC>::kRing];      // the MMAs of group g (index g % kRing) completed
    uint64_t fullBits[kBitsStages];
    uint64_t emptyBits[kBitsStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t never;  // no one arrives here: used by the stall test hook
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

template <int BN, int OCC>
constexpr int smem_bytes()
{
    return Cfg<BN, OCC>::kStagesB * Cfg<BN, OCC>::kBBytes + kBitsStages * kBitsBytes +
           (int)sizeof(Barriers<BN, OCC>) + 1024;
}

// Wait until the MMAs of group h have completed (h >= 0), through the "done"
// ring: phase h / R of barrier h % R.  A waiter never runs more than one phase
// ahead: it has already seen group h - 1 complete.
template <int R>
__device__ __forceinline__ bool wait_done(uint64_t* done, int h, volatile int* abort, long long budget)
{
    return ptx::mbar_wait_bounded(&done[h % R], (uint32_t)(h / R) & 1u, abort, budget);
}

template <int BN, bool EXACT, int OCC, bool PERSIST>
__global__ void __launch_bounds__(kThreads, OCC)
    bitlin_tc_gemm(const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_bits,
                   const PrefillParams p, int stall_test)
{
    using C = Cfg<BN, OCC>;
    constexpr int kTmemCols = C::kTmemCols;
    constexpr int SB = C::kStagesB, SA = C::kStagesA, R = C::kRing;
    constexpr int kBBytes = C::kBBytes;
    constexpr int kHalf = BN / 2;                    // columns per epilogue warp
    constexpr int kChunks = kHalf / 32;              // tcgen05.ld x32 loads per group
    constexpr int kAcc = EXACT ? kHalf / 4 : kHalf;  // accumulators per epilogue thread
    constexpr bool kNarrow = !EXACT && OCC == 2;     // 16-column reads: 32 accumulators in 64 registers
    static_assert(BN % 64 == 0 && BN <= 128, "tile width");

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* tileB = smem;                         // [stage][BN * 256 B]
    unsigned char* tileBits = tileB + SB * kBBytes;      // [bits stage][2 KB]: [row][4 words]
    auto* bar = reinterpret_cast<Barriers<BN, OCC>*>(tileBits + kBitsStages * kBitsBytes);
    volatile int* abort = &bar->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Split-K over grid.z: this CTA takes the K-groups [gbase, gbase + G).
    const int Gall = p.K / 128;
    const int gbase = (int)((long long)Gall * blockIdx.z / gridDim.z);
    const int G = (int)((long long)Gall * (blockIdx.z + 1) / gridDim.z) - gbase;
    const long long budget = p.wait_budget_ns;
    // The CTA's tiles: its grid tile, or (persistent) tiles tile_base +
    // blockIdx.x, + gridDim.x, ... of the tiles_x-wide grid of tiles.  Every
    // role runs one group counter gg over all of them (tile gg / G, K-group
    // gg % G), so stages, barrier phases and accumulator buffers carry on from
    // one tile to the next.
    const int ntiles = PERSIST ? (p.tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 1;
    const int GT = ntiles * G;
    auto tile_xy = [&](int ti, int& tn0, int& tb0) {
        if (PERSIST) {
            const int t = p.tile_base + (int)blockIdx.x + ti * (int)gridDim.x;
            const int ty = t / p.tiles_x;
            tn0 = (t - ty * p.tiles_x) * kPrefillRows;
            tb0 = ty * BN;
        } else {
            tn0 = (int)blockIdx.x * kPrefillRows;
            tb0 = (int)blockIdx.y * BN;
        }
    };
    int n0, b0;  // the first tile (the split-K finish uses it)
    tile_xy(0, n0, b0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SB; ++s) ptx::mbar_init(&bar->fullB[s], 1);
        for (int s = 0; s < SA; ++s) ptx::mbar_init(&bar->fullA[s], 128);
        for (int s = 0; s < R; ++s) ptx::mbar_init(&bar->done[s], 1);
        for (int s = 0; s < kBitsStages; ++s) {
            ptx::mbar_init(&bar->fullBits[s], 1);
            ptx::mbar_init(&bar->emptyBits[s], 128);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bar->tfull[b], 1);
            ptx::mbar_init(&bar->tempty[b], kEpiWarps * 32);
        }
        ptx::mbar_init(&bar->never, 1);
        ptx::mbar_init(&bar->drain, 1);
        bar->abort = 0;
        ptx::mbar_fence_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(&bar->tmem_base, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == kTmaWarp && lane == 0) ptx::prefetch_tmap(&tmap_b);
    if (warp == kBitsWarp && lane == 0) ptx::prefetch_tmap(&tmap_bits);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bar->tmem_base;
    const uint32_t tmemA = tmem + 2 * BN;  // A stages follow the two accumulator buffers
    // Programmatic dependent launch: the next kernel may launch once every CTA
    // of this grid has started.  Only the B loader (xt, written by the
    // rotation) and the epilogue (y) wait for the previous kernel; the bits,
    // the scales and the +-1 expansion do not depend on it.
    ptx::griddep_launch_dependents();

    if (warp == kTmaWarp) {
        if (lane == 0) {
            ptx::griddep_wait();
            // B tiles; stage g % SB is free once the MMAs of group g - SB completed.
            int issued = 0;
            for (int gg = 0; gg < GT; ++gg) {
                const int ti = gg / G, g = gg - ti * G;
                int tn0, tb0;
                tile_xy(ti, tn0, tb0);
                const int st = gg % SB;
                if (gg >= SB && !wait_done<R>(bar->done, gg - SB, abort, budget)) break;
                ptx::mbar_arrive_expect_tx(&bar->fullB[st], kBBytes);
                ptx::tma_load_3d(tileB + st * kBBytes, &tmap_b, 0, tb0, 2 * (gbase + g), &bar->fullB[st]);
                issued = gg + 1;
            }
            // Every copy this lane issued must land before the CTA may exit.
            for (int g = (issued > SB ? issued - SB : 0); g < issued; ++g) {
                volatile int no_abort = 0;
                ptx::mbar_wait_bounded(&bar->fullB[g % SB], (uint32_t)(g / SB) & 1u, &no_abort, budget);
            }
        }
    } else if (warp == kBitsWarp) {
        // Bits, up to kBitsStages groups ahead of the expansion (a warp of its
        // own: two producers in one warp would take turns).
        if (lane == 0) {
            int issued = 0;
            for (int gg = 0; gg < GT; ++gg) {
                const int ti = gg / G, g = gg - ti * G;
                int tn0, tb0;
                tile_xy(ti, tn0, tb0);
                const int sb = gg % kBitsStages;
                const uint32_t ph = (uint32_t)(gg / kBitsStages) & 1u;
                if (!ptx::mbar_wait_bounded(&bar->emptyBits[sb], ph ^ 1u, abort, budget)) break;
                ptx::mbar_arrive_expect_tx(&bar->fullBits[sb], kBitsBytes);
                ptx::tma_load_2d(tileBits + sb * kBitsBytes, &tmap_bits, (gbase + g) * 4, tn0, &bar->fullBits[sb]);
                issued = gg + 1;
            }
            for (int g = (issued > kBitsStages ? issued - kBitsStages : 0); g < issued; ++g) {
                const int sb = g % kBitsStages;
                const uint32_t ph = (uint32_t)(g / kBitsStages) & 1u;
                volatile int no_abort = 0;
                ptx::mbar_wait_bounded(&bar->fullBits[sb], ph, &no_abort, budget);
            }
        }
    } else if (warp == kMmaWarp) {
        // The whole warp runs the loop and tests the three barriers in one
        // shared-memory round trip; one elected lane issues (a lane-0 branch or
        // a one-lane loop instead of elect.sync measured 30-35% slower).
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(kPrefillRows, BN);
        const uint64_t descB = ptx::smem_desc_sw128(ptx::smem_u32(tileB));
        int issued = 0;
        for (int g = 0; g < GT; ++g) {  // g: the CTA's group counter over all its tiles
            const int sb = g % SB, sa = g % SA, buf = g & 1;
            if (!ptx::mbar_wait3_bounded(&bar->fullB[sb], (uint32_t)(g / SB) & 1u, &bar->fullA[sa],
                                         (uint32_t)(g / SA) & 1u, &bar->tempty[buf], ((uint32_t)(g >> 1) & 1u) ^ 1u,
                                         abort, budget))
                break;
            ptx::tc_fence_after();
            if (ptx::elect_one()) {
                const uint32_t d = tmem + (uint32_t)(buf * BN);
                const uint32_t a = tmemA + (uint32_t)(sa * kACols);
                // Descriptor start addresses advance in 16-byte units.
                const uint64_t db = descB + (uint64_t)((sb * kBBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t offb = (uint32_t)((kk >> 2) * (kBBytes / 2) + (kk & 3) * 32) >> 4;
                    ptx::mma_bf16_ts(d, a + 8 * kk, db + offb, idesc, kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&bar->done[g % R]);
                ptx::mma_commit(&bar->tfull[buf]);
            }
            __syncwarp();
            issued = g + 1;
        }
        // Wait for every MMA issued here before TMEM is released.
        if (issued > 0) {
            if (ptx::elect_one()) ptx::mma_commit(&bar->drain);
            __syncwarp();
            volatile int no_abort = 0;
            ptx::mbar_wait_bounded(&bar->drain, 0u, &no_abort, budget);
        }
    } else if (warp >= kExpWarp0 && warp < kExpWarp0 + 4) {
        // A warp may only reach TMEM lanes 32*(warp%4) .. +31: row = that lane.
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        for (int g = 0; g < GT; ++g) {  // g: the CTA's group counter over all its tiles
            const int sa = g % SA;
            const int sb = g % kBitsStages;
            // The group's bits (prefetched up to kBitsStages groups ahead), then a
            // free A stage: the MMAs of group g - SA have completed.
            if (!ptx::mbar_wait_bounded(&bar->fullBits[sb], (uint32_t)(g / kBitsStages) & 1u, abort, budget)) break;
            const uint4 wq = *reinterpret_cast<const uint4*>(tileBits + sb * kBitsBytes + r * 16);
            ptx::mbar_arrive(&bar->emptyBits[sb]);
            if (g >= SA && !wait_done<R>(bar->done, g - SA, abort, budget)) break;
            ptx::tc_fence_after();
            const uint32_t words[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // columns 32h .. 32h+31 = words 2h, 2h+1; column 16j + i holds weights
                // 32j + 2i (low half) and 32j + 2i + 1 (high half)
                uint32_t v[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const uint32_t W = words[2 * h + (c >> 4)];
                    v[c] = 0xBF80BF80u ^ ((W << (15 - (c & 15))) & 0x80008000u);
                }
                ptx::tmem_st32(tmemA + lane_base + (uint32_t)(sa * kACols + 32 * h), v);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar->fullA[sa]);
        }
    } else if (warp < kEpiWarps) {
        ptx::griddep_wait();
        const int q = warp & 3, half = warp >> 2;
        const int r = 32 * q + lane;
        bool ok = true;
        for (int ti = 0; ti < ntiles && ok; ++ti) {
        int tn0, tb0;
        tile_xy(ti, tn0, tb0);
        const int n = tn0 + r;
        const bool valid = n < p.N;
        // Accumulators in pairs: the exact mode sums two outputs' digit columns
        // and scales them with packed f32x2 adds and FMAs (__fadd2_rn,
        // __ffma2_rn; gate_up at M = 16: 38.8 -> 38.3 us).  The bf16 mode keeps
        // scalar FMAs: its packed pairs exceeded the 128-register budget.
        static_assert(kAcc % 2 == 0, "accumulators come in pairs");
        float2 acc2[kAcc / 2];
#pragma unroll
        for (int j = 0; j < kAcc / 2; ++j) acc2[j] = make_float2(0.f, 0.f);
        const uint16_t* srow = p.scales + (size_t)(valid ? n : 0) * Gall + gbase;
        // The row's scales, requested kSRing groups ahead.
        constexpr int kSRing = 4;
        uint16_t sring[kSRing];
#pragma unroll
        for (int u = 0; u < kSRing; ++u) sring[u] = (valid && u < G) ? __ldg(srow + u) : (uint16_t)0;
        for (int g0 = 0; g0 < G && ok; g0 += kSRing) {
#pragma unroll
            for (int u = 0; u < kSRing; ++u) {
                const int g = g0 + u;
                if (g >= G) break;
                const int gg = ti * G + g;  // the CTA's group counter
                const int buf = gg & 1;
                const uint32_t tph = (uint32_t)(gg >> 1) & 1u;
                const float s = __half2float(__ushort_as_half(sring[u]));
                sring[u] = (valid && g + kSRing < G) ? __ldg(srow + g + kSRing) : (uint16_t)0;
                uint64_t* wbar = (stall_test && gg == 0) ? &bar->never : &bar->tfull[buf];
                ok = ptx::mbar_wait_bounded(wbar, tph, abort, budget);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t taddr =
                    tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * BN + kHalf * half);
                if (kNarrow) {
                    // 16-column reads (the bf16 half-SM instance's 64 registers)
#pragma unroll
                    for (int c = 0; c < kHalf / 16; ++c) {
                        float v[16];
                        ptx::tmem_ld16(taddr + 16 * c, v);
                        ptx::tmem_wait_ld();
                        if (c == kHalf / 16 - 1) {
                            ptx::tc_fence_before();
                            ptx::mbar_arrive(&bar->tempty[buf]);
                        }
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            acc2[(16 * c + j) / 2].x = fmaf(s, v[j], acc2[(16 * c + j) / 2].x);
                            acc2[(16 * c + j) / 2].y = fmaf(s, v[j + 1], acc2[(16 * c + j) / 2].y);
                        }
                    }
                } else
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    float v[32];
                    ptx::tmem_ld32(taddr + 32 * c, v);
                    ptx::tmem_wait_ld();
                    if (c == kChunks - 1) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(&bar->tempty[buf]);
                    }
                    const float2 s2 = make_float2(s, s);
                    if (EXACT) {
#pragma unroll
                        for (int t = 0; t < 8; t += 2) {
                            const float2 d = __fadd2_rn(__fadd2_rn(make_float2(v[4 * t], v[4 * t + 4]),
                                                                   make_float2(v[4 * t + 1], v[4 * t + 5])),
                                                        make_float2(v[4 * t + 2], v[4 * t + 6]));
                            acc2[(8 * c + t) / 2] = __ffma2_rn(s2, d, acc2[(8 * c + t) / 2]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            acc2[(32 * c + j) / 2].x = fmaf(s, v[j], acc2[(32 * c + j) / 2].x);
                            acc2[(32 * c + j) / 2].y = fmaf(s, v[j + 1], acc2[(32 * c + j) / 2].y);
                        }
                    }
                }
            }
        }
        if (gridDim.z > 1) {
            // Split-K: park the partial results in the B ring (idle now: every
            // copy into it has landed and every MMA reading it has completed),
            // column c = half * kAcc + j, row r: pbuf[c * 128 + r].
            float* pbuf = reinterpret_cast<float*>(tileB);
#pragma unroll
            for (int j = 0; j < kAcc; ++j) pbuf[(half * kAcc + j) * kPrefillRows + r] = (j & 1) ? acc2[j / 2].y : acc2[j / 2].x;
        } else if (ok && valid) {
#pragma unroll
            for (int j = 0; j < kAcc; ++j) {
                const int m = EXACT ? (tb0 + half * kHalf) / 4 + j : tb0 + half * kHalf + j;
                if (m < p.M) p.y[(size_t)m * p.N + n] = (j & 1) ? acc2[j / 2].y : acc2[j / 2].x;
            }
        }
        }  // tiles
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (gridDim.z > 1) {
        // The split-K CTAs of this tile form a cluster along z.  Each sums an
        // equal share of the tile's outputs over the cluster's partials, in
        // rank order 0..S-1 (deterministic), through distributed shared
        // memory, and writes y; the second barrier keeps every CTA's shared
        // memory alive until the others have read it.
        static_assert(2 * kAcc * kPrefillRows * 4 <= C::kStagesB * kBBytes, "partials fit the B ring");
        ptx::cluster_sync();
        const int S = gridDim.z;
        const int rank = (int)ptx::cluster_ctarank();
        constexpr int E = 2 * kAcc * kPrefillRows;
        const uint32_t base = ptx::smem_u32(tileB);
        for (int e = E * rank / S + (int)threadIdx.x; e < E * (rank + 1) / S; e += kThreads) {
            float v[kMaxSplits];
#pragma unroll
            for (int j = 0; j < kMaxSplits; ++j)
                if (j < S) v[j] = ptx::ld_cluster(ptx::cluster_map(base + 4u * (uint32_t)e, j));
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxSplits; ++j)
                if (j < S) sum += v[j];
            const int c = e / kPrefillRows, r = e - c * kPrefillRows;
            const int m = EXACT ? b0 / 4 + c : b0 + c;
            const int n = n0 + r;
            if (m < p.M && n < p.N) p.y[(size_t)m * p.N + n] = sum;
        }
        ptx::cluster_sync();
    }
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && bar->abort) atomicExch(p.dev_error, kDevErrTimeout);
}

// PERSIST: the launch covers tiles tile_base .. tile_base + tile_count - 1 of
// the row-major tile grid (tile_count 0: all of them).
template <int BN, bool EXACT, int OCC = 1, bool PERSIST = false>
cudaError_t launch(const PrefillParams& p, const void* tmap, const void* tmap_bits, int stall_test,
                   cudaStream_t s, int tile_base = 0, int tile_count = 0)
{
    // Once per device (the attribute applies to the current device): the shared
    // memory size, and how many clusters of each split-K size can be resident
    // at once (max_clusters[dev][s]).
    static PerDeviceOnce once;
    static int max_clusters[kMaxDevices][kMaxSplits + 1];
    int dev = 0;
    cudaError_t ce = once.run(&dev, [](int d) {
        cudaError_t e = cudaFuncSetAttribute(bitlin_tc_gemm<BN, EXACT, OCC, PERSIST>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<BN, OCC>());
        for (int z = 2; z <= kMaxSplits && e == cudaSuccess; ++z) {
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 1;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = z;
            cudaLaunchConfig_t c = {};
            c.gridDim = dim3(1, 1, z);
            c.blockDim = dim3(kThreads);
            c.dynamicSmemBytes = smem_bytes<BN, OCC>();
            c.attrs = at;
            c.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&max_clusters[d][z], bitlin_tc_gemm<BN, EXACT, OCC, PERSIST>, &c);
        }
        return e;
    });
    if (ce != cudaSuccess) return ce;
    const int rows_b = EXACT ? 4 * p.M : p.M;
    const int gx = (p.N + kPrefillRows - 1) / kPrefillRows, gy = (rows_b + BN - 1) / BN;
    // Split K when the tiles would fill less than half of the SMs (tall-K,
    // short-N matrices at small M, e.g. 17408 -> 5120): as many splits as
    // still fit one wave, at most 8 and at least 8 K-groups each.
    int splits = 1;
    const int tiles = PERSIST && tile_count > 0 ? tile_count : gx * gy, Gall = p.K / 128;
    if (2 * tiles < OCC * p.num_sms) {
        splits = OCC * p.num_sms / tiles;
        if (splits > kMaxSplits) splits = kMaxSplits;
        if (splits > Gall / 8) splits = Gall / 8;
        // All tiles' clusters must be resident at once: one cluster more than
        // fits runs as a second wave (on 152 SMs at about 200 KB of shared
        // memory a CTA, 46 clusters of 3 fit, not 48; 28 of 5).  The query
        // reports the same counts for the two-CTAs-per-SM instance, which
        // holds twice as many (80 clusters of 3 run as one wave there: attn_qkv
        // at M = 16 19.7 us, 31.4 with the split cut to 1), hence * OCC.
        while (splits > 1 && OCC * max_clusters[dev][splits] < tiles) --splits;
        if (splits < 1) splits = 1;
    }
    const CUtensorMap tb = *static_cast<const CUtensorMap*>(tmap);
    const CUtensorMap tbits = *static_cast<const CUtensorMap*>(tmap_bits);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = splits;
    cudaLaunchConfig_t cfg = {};
    PrefillParams q = p;
    q.tiles_x = gx;
    q.tiles = tiles;
    q.tile_base = PERSIST ? tile_base : 0;
    cfg.gridDim = PERSIST ? dim3(tiles < OCC * p.num_sms ? tiles : OCC * p.num_sms, 1, splits) : dim3(gx, gy, splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes<BN, OCC>();
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = splits > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, bitlin_tc_gemm<BN, EXACT, OCC, PERSIST>, tb, tbits, q, stall_test);
}

}  // namespace

int bitlin_tc_tile_width(int M, int exact)
{
    if (!exact) return M <= 64 ? 64 : kPrefillTokens;
    return 4 * M <= 64 ? 64 : 128;
}

namespace {

// Tiles of the bf16 path, and how many of them come after the last full wave
// of num_sms when those get a launch of their own (0: one launch).
int prefill_tail(int M, int N, int num_sms, int* tiles)
{
    *tiles = ((N + kPrefillRows - 1) / kPrefillRows) * ((M + kPrefillTokens - 1) / kPrefillTokens);
    if (*tiles <= num_sms) return 0;
    const int rem = *tiles - *tiles / num_sms * num_sms;
    return 2 * rem < num_sms ? rem : 0;
}

}  // namespace

int bitlin_prefill_gemm_launches(int M, int N, int num_sms)
{
    if (bitlin_tc_tile_width(M, 0) == 64) return 1;
    int tiles = 0;
    return prefill_tail(M, N, num_sms, &tiles) > 0 ? 2 : 1;
}

cudaError_t bitlin_launch_prefill(const PrefillParams& p, const void* tmap, const void* tmap_bits,
                                  int stall_test, cudaStream_t s)
{
    if (bitlin_tc_tile_width(p.M, 0) == 64) {
        // At most 64 tokens: 64-wide tiles (the exact path's shape) instead of
        // 128-wide ones half filled with zeros; two CTAs per SM when the tiles
        // fill every SM (gate_up at M = 64 46.8 -> 34.7 us, the LM head 257.8 ->
        // 191.5, ffn_down 33.3 -> 28.0, ffn_gate 25.0 -> 23.5, attn_qkv 22.9 ->
        // 20.6; two per SM from half the SMs, as the exact path does, measured
        // slower here: ffn_gate 26.7, attn_q 25.5).
        const int tiles = (p.N + kPrefillRows - 1) / kPrefillRows;
        if (tiles >= p.num_sms) return launch<64, false, 2>(p, tmap, tmap_bits, stall_test, s);
        return launch<64, false>(p, tmap, tmap_bits, stall_test, s);
    }
    // A persistent grid (one CTA per SM looping over the tiles) when the tiles
    // need more than one wave: the next tile's loads, bits and expansion then
    // follow the last groups of the previous one without a CTA start in
    // between (prefill 173.5 -> 168.8 us, gate_up at M = 1024 317.8 -> 306.5).
    int tiles = 0;
    const int rem = prefill_tail(p.M, p.N, p.num_sms, &tiles);
    if (tiles > p.num_sms) {
        // The tiles past the last full wave would run on that many SMs while
        // the others idle.  When they fill less than half of the SMs, they
        // get a launch of their own, each split along K over a cluster (the
        // split-K finish), so that every SM takes part: prefill 165.5 ->
        // 158.5 us (1064 + 24 tiles, split 5), the MLP block at M = 1024
        // 542.6 -> 492.5 (gate_up 2128 + 48 tiles, split 2; down 304 + 16,
        // split 8).  The tail waits for the first launch (programmatic
        // dependent launch), whose CTAs all end at about the same time.
        if (rem > 0) {
            const int full = tiles - rem;
            const cudaError_t e = launch<kPrefillTokens, false, 1, true>(p, tmap, tmap_bits, stall_test, s, 0, full);
            if (e != cudaSuccess) return e;
            return launch<kPrefillTokens, false, 1, true>(p, tmap, tmap_bits, stall_test, s, full, rem);
        }
        return launch<kPrefillTokens, false, 1, true>(p, tmap, tmap_bits, stall_test, s);
    }
    return launch<kPrefillTokens, false>(p, tmap, tmap_bits, stall_test, s);
}

cudaError_t bitlin_launch_tc_exact(const PrefillParams& p, const void* tmap, const void* tmap_bits,
                                   int stall_test, cudaStream_t s)
{
    if (bitlin_tc_tile_width(p.M, 1) == 64) {
        // Two CTAs per SM when the tiles fill at least half of the SMs at one
        // CTA per SM (see Cfg).
        const int tiles = (p.N + kPrefillRows - 1) / kPrefillRows;
        if (2 * tiles >= p.num_sms) return launch<64, true, 2>(p, tmap, tmap_bits, stall_test, s);
        return launch<64, true>(p, tmap, tmap_bits, stall_test, s);
    }
    return launch<128, true>(p, tmap, tmap_bits, stall_test, s);
}
