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
//    token; CTA tile = 128 weight rows x BN tokens, tokens split over grid.y.
//  * exact (2 <= M < 64): the B operand holds, for token m, rows 4m..4m+2 =
//    the three bf16 digits hi, mid, lo of xt (hi = bf16(xt), mid =
//    bf16(xt - hi), lo = bf16(xt - hi - mid): together the f32 value) and row
//    4m+3 = 0.  Products with +-1 are exact, so summing the three digit
//    columns of D gives f32-level results.  One tile holds every token.
//
// CTA tile: 128 weight rows (UMMA M = 128, one TMEM lane per row) x BN columns
// of B (UMMA N = BN).  Per 128-wide K-group g:
//   * warp 8, lane 0 TMA-loads the B tile [BN rows][128 K] as two
//     128-byte-swizzled boxes of 64 columns; lane 1 TMA-loads the group's
//     bits [128 rows][4 words] (2 KB) into a separate ring that runs up to 8
//     groups ahead, so the expansion never waits for the B tile;
//   * warps 10-13 (one thread per weight row) expand that row's 128 bits of
//     the group into +-1 bf16 directly in the same swizzled K-major layout (TMA
//     cannot expand bits).  The repack stores even weights in the low
//     half-word and odd weights in the high half-word, so each bf16x2 pair is
//     one shift and one XOR-mask;
//   * warp 9 (one lane) issues 8 MMAs of K = 16 into TMEM accumulator
//     buffer g % 2 (overwriting it at the first), then commits to the stage's
//     "empty" barrier and the buffer's "full" barrier;
//   * warps 0-7 read the buffer back (tcgen05.ld), hand it back to the MMA
//     warp, and accumulate scale[n][g] * D into f32 registers - the per-group
//     scale promotion.  Warp w serves TMEM lanes 32*(w%4).. and the columns
//     BN/2*(w/4) .. BN/2*(w/4) + BN/2 - 1.  Scales are requested 4 groups ahead.
// Shared-memory stages keep the producers ahead of the MMAs, two TMEM buffers
// keep the MMAs one group ahead of the epilogue.  Every wait is bounded in
// time; on expiry the kernel stops its loops, drains its own copies and
// MMAs, frees TMEM and records a timeout in the handle's error word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bitlin_internal.cuh"
#include "ptx.cuh"

namespace {

using namespace bitlin_impl;

constexpr int kThreads = 448;       // 14 warps
constexpr int kEpiWarps = 8;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kExpWarp0 = 10;
constexpr int kABytes = 32768;      // A tile: 128 rows x 128 bf16
constexpr int kBitsBytes = 2048;    // one group's bits: 128 rows x 4 words
constexpr int kBitsStages = 8;      // bits run this many groups ahead of the expansion

template <int STAGES>
struct __align__(8) Barriers {
    uint64_t fullA[STAGES];
    uint64_t fullB[STAGES];
    uint64_t empty[STAGES];
    uint64_t fullBits[kBitsStages];
    uint64_t emptyBits[kBitsStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t never;     // no one arrives here: used by the stall test hook
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

template <int BN>
struct Cfg {
    static constexpr int kBBytes = BN * 256;  // B tile: BN rows x 128 bf16
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBudget = 208 * 1024 - kBitsStages * kBitsBytes;
    static constexpr int kStages = kStageBytes * 4 <= kBudget ? 4 : kStageBytes * 3 <= kBudget ? 3 : 2;
    static constexpr int kTmemCols = 2 * BN <= 128 ? 128 : 2 * BN <= 256 ? 256 : 512;
    static constexpr int kSmem =
        kStages * kStageBytes + kBitsStages * kBitsBytes + (int)sizeof(Barriers<kStages>) + 1024;
};

template <int BN, bool EXACT>
__global__ void __launch_bounds__(kThreads, 1)
    bitlin_tc_gemm(const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_bits,
                   const PrefillParams p, int stall_test)
{
    constexpr int STAGES = Cfg<BN>::kStages;
    constexpr int kBBytes = Cfg<BN>::kBBytes;
    constexpr int kHalf = BN / 2;                    // columns per epilogue warp
    constexpr int kChunks = kHalf / 32;              // tcgen05.ld x32 loads per group
    constexpr int kAcc = EXACT ? kHalf / 4 : kHalf;  // accumulators per epilogue thread
    static_assert(BN % 64 == 0 && BN <= 256, "tile width");

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* tileA = smem;                         // [stage][32 KB]
    unsigned char* tileB = smem + STAGES * kABytes;      // [stage][BN * 256 B]
    unsigned char* tileBits = tileB + STAGES * kBBytes;  // [bits stage][2 KB]: [row][4 words]
    auto* bar = reinterpret_cast<Barriers<STAGES>*>(tileBits + kBitsStages * kBitsBytes);
    volatile int* abort = &bar->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kPrefillRows;
    const int b0 = blockIdx.y * BN;  // first B row of this tile
    const int G = p.K / 128;
    const long long budget = p.wait_budget_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&bar->fullA[s], 128);
            ptx::mbar_init(&bar->fullB[s], 1);
            ptx::mbar_init(&bar->empty[s], 1);
        }
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
        ptx::tmem_alloc(&bar->tmem_base, Cfg<BN>::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == kTmaWarp && lane == 0) {
        ptx::prefetch_tmap(&tmap_b);
        ptx::prefetch_tmap(&tmap_bits);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bar->tmem_base;

    if (warp == kTmaWarp) {
        if (lane == 0) {
            // B tiles, gated by the stage's "empty" barrier (the MMAs of the
            // group STAGES back have completed).
            int issued = 0;
            for (int g = 0; g < G; ++g) {
                const int st = g % STAGES;
                const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
                if (!ptx::mbar_wait_bounded(&bar->empty[st], ph ^ 1u, abort, budget)) break;
                ptx::mbar_arrive_expect_tx(&bar->fullB[st], kBBytes);
                unsigned char* dst = tileB + st * kBBytes;
                ptx::tma_load_2d(dst, &tmap_b, g * 128, b0, &bar->fullB[st]);
                ptx::tma_load_2d(dst + kBBytes / 2, &tmap_b, g * 128 + 64, b0, &bar->fullB[st]);
                issued = g + 1;
            }
            // Every copy this lane issued must land before the CTA may exit.
            for (int g = (issued > STAGES ? issued - STAGES : 0); g < issued; ++g) {
                const int st = g % STAGES;
                const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
                volatile int no_abort = 0;
                ptx::mbar_wait_bounded(&bar->fullB[st], ph, &no_abort, budget);
            }
        } else if (lane == 1) {
            // Bits, up to kBitsStages groups ahead of the expansion.
            int issued = 0;
            for (int g = 0; g < G; ++g) {
                const int sb = g % kBitsStages;
                const uint32_t ph = (uint32_t)(g / kBitsStages) & 1u;
                if (!ptx::mbar_wait_bounded(&bar->emptyBits[sb], ph ^ 1u, abort, budget)) break;
                ptx::mbar_arrive_expect_tx(&bar->fullBits[sb], kBitsBytes);
                ptx::tma_load_2d(tileBits + sb * kBitsBytes, &tmap_bits, g * 4, n0, &bar->fullBits[sb]);
                issued = g + 1;
            }
            for (int g = (issued > kBitsStages ? issued - kBitsStages : 0); g < issued; ++g) {
                const int sb = g % kBitsStages;
                const uint32_t ph = (uint32_t)(g / kBitsStages) & 1u;
                volatile int no_abort = 0;
                ptx::mbar_wait_bounded(&bar->fullBits[sb], ph, &no_abort, budget);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(kPrefillRows, BN);
            int issued = 0;
            for (int g = 0; g < G; ++g) {
                const int st = g % STAGES;
                const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
                const int buf = g & 1;
                const uint32_t tph = (uint32_t)(g >> 1) & 1u;
                if (!ptx::mbar_wait_bounded(&bar->fullA[st], ph, abort, budget)) break;
                if (!ptx::mbar_wait_bounded(&bar->fullB[st], ph, abort, budget)) break;
                if (!ptx::mbar_wait_bounded(&bar->tempty[buf], tph ^ 1u, abort, budget)) break;
                ptx::tc_fence_after();
                const uint32_t a0 = ptx::smem_u32(tileA + st * kABytes);
                const uint32_t bb = ptx::smem_u32(tileB + st * kBBytes);
                const uint32_t d = tmem + (uint32_t)(buf * BN);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t offa = (uint32_t)((kk >> 2) * (kABytes / 2) + (kk & 3) * 32);
                    const uint32_t offb = (uint32_t)((kk >> 2) * (kBBytes / 2) + (kk & 3) * 32);
                    ptx::mma_bf16(d, ptx::smem_desc_sw128(a0 + offa), ptx::smem_desc_sw128(bb + offb),
                                  idesc, kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&bar->empty[st]);
                ptx::mma_commit(&bar->tfull[buf]);
                issued = g + 1;
            }
            // Wait for every MMA issued here before TMEM is released.
            if (issued > 0) {
                ptx::mma_commit(&bar->drain);
                volatile int no_abort = 0;
                ptx::mbar_wait_bounded(&bar->drain, 0u, &no_abort, budget);
            }
        }
    } else if (warp >= kExpWarp0) {
        const int r = (warp - kExpWarp0) * 32 + lane;  // row within the tile
        for (int g = 0; g < G; ++g) {
            const int st = g % STAGES;
            const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
            const int sb = g % kBitsStages;
            const uint32_t phb = (uint32_t)(g / kBitsStages) & 1u;
            // The group's bits (prefetched up to kBitsStages groups ahead), then a
            // free A buffer: the MMAs of the group STAGES back have completed.
            if (!ptx::mbar_wait_bounded(&bar->fullBits[sb], phb, abort, budget)) break;
            const uint4 wq = *reinterpret_cast<const uint4*>(tileBits + sb * kBitsBytes + r * 16);
            ptx::mbar_arrive(&bar->emptyBits[sb]);
            if (!ptx::mbar_wait_bounded(&bar->empty[st], ph ^ 1u, abort, budget)) break;
            unsigned char* dst = tileA + st * kABytes + r * 128;
            const uint32_t words[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                // chunk c = weights 8c .. 8c+7 of the group = pairs 4(c&3) .. 4(c&3)+3 of word c>>2
                const uint32_t W = words[c >> 2];
                uint32_t v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int i = 4 * (c & 3) + q;
                    v[q] = 0xBF80BF80u ^ ((W << (15 - i)) & 0x80008000u);
                }
                const int atom = c >> 3, cc = c & 7;
                *reinterpret_cast<uint4*>(dst + atom * (kABytes / 2) + ((cc ^ (r & 7)) << 4)) =
                    make_uint4(v[0], v[1], v[2], v[3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bar->fullA[st]);
        }
    } else {
        // Epilogue warps 0..7.
        const int q = warp & 3, half = warp >> 2;
        const int r = 32 * q + lane;
        const int n = n0 + r;
        const bool valid = n < p.N;
        float acc[kAcc];
#pragma unroll
        for (int j = 0; j < kAcc; ++j) acc[j] = 0.f;
        const uint16_t* srow = p.scales + (size_t)(valid ? n : 0) * G;
        // The row's scales, requested kSRing groups ahead (G is a multiple of 8).
        constexpr int kSRing = 4;
        uint16_t sring[kSRing];
#pragma unroll
        for (int u = 0; u < kSRing; ++u) sring[u] = valid ? __ldg(srow + u) : (uint16_t)0;
        bool ok = true;
        for (int g0 = 0; g0 < G && ok; g0 += kSRing) {
#pragma unroll
            for (int u = 0; u < kSRing; ++u) {
                const int g = g0 + u;
                const int buf = g & 1;
                const uint32_t tph = (uint32_t)(g >> 1) & 1u;
                const float s = __half2float(__ushort_as_half(sring[u]));
                sring[u] = (valid && g + kSRing < G) ? __ldg(srow + g + kSRing) : (uint16_t)0;
                uint64_t* wbar = (stall_test && g == 0) ? &bar->never : &bar->tfull[buf];
                ok = ptx::mbar_wait_bounded(wbar, tph, abort, budget);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t taddr =
                    tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * BN + kHalf * half);
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    float v[32];
                    ptx::tmem_ld32(taddr + 32 * c, v);
                    ptx::tmem_wait_ld();
                    if (c == kChunks - 1) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(&bar->tempty[buf]);
                    }
                    if (EXACT) {
#pragma unroll
                        for (int t = 0; t < 8; ++t)
                            acc[8 * c + t] = fmaf(s, (v[4 * t] + v[4 * t + 1]) + v[4 * t + 2], acc[8 * c + t]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) acc[32 * c + j] = fmaf(s, v[j], acc[32 * c + j]);
                    }
                }
            }
        }
        if (ok && valid) {
#pragma unroll
            for (int j = 0; j < kAcc; ++j) {
                const int m = EXACT ? (half * (kHalf / 4) + j) : (b0 + half * kHalf + j);
                if (m < p.M) p.y[(size_t)m * p.N + n] = acc[j];
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, Cfg<BN>::kTmemCols);
    }
    if (threadIdx.x == 0 && bar->abort) atomicExch(p.dev_error, kDevErrTimeout);
}

template <int BN, bool EXACT>
cudaError_t launch(const PrefillParams& p, const void* tmap, const void* tmap_bits, int stall_test,
                   cudaStream_t s)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(bitlin_tc_gemm<BN, EXACT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<BN>::kSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int rows_b = EXACT ? 4 * p.M : p.M;
    dim3 grid((p.N + kPrefillRows - 1) / kPrefillRows, (rows_b + BN - 1) / BN);
    bitlin_tc_gemm<BN, EXACT><<<grid, kThreads, Cfg<BN>::kSmem, s>>>(
        *static_cast<const CUtensorMap*>(tmap), *static_cast<const CUtensorMap*>(tmap_bits), p, stall_test);
    return cudaGetLastError();
}

}  // namespace

int bitlin_tc_tile_width(int M, int exact)
{
    if (!exact) return kPrefillTokens;
    const int rows = 4 * M;
    return rows <= 64 ? 64 : rows <= 128 ? 128 : rows <= 192 ? 192 : 256;
}

cudaError_t bitlin_launch_prefill(const PrefillParams& p, const void* tmap, const void* tmap_bits,
                                  int stall_test, cudaStream_t s)
{
    return launch<kPrefillTokens, false>(p, tmap, tmap_bits, stall_test, s);
}

cudaError_t bitlin_launch_tc_exact(const PrefillParams& p, const void* tmap, const void* tmap_bits,
                                   int stall_test, cudaStream_t s)
{
    switch (bitlin_tc_tile_width(p.M, 1)) {
    case 64: return launch<64, true>(p, tmap, tmap_bits, stall_test, s);
    case 128: return launch<128, true>(p, tmap, tmap_bits, stall_test, s);
    case 192: return launch<192, true>(p, tmap, tmap_bits, stall_test, s);
    default: return launch<256, true>(p, tmap, tmap_bits, stall_test, s);
    }
}
