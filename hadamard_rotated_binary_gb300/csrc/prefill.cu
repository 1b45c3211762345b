// Tensor-core path (M >= 64): Y[M][N] = per-group-scaled (+-1 W) x xt^T with
// tcgen05 MMAs, bf16 operands and f32 accumulation in tensor memory.
//
// Method: the folded product of the Pulse "ARCHITECTURE-SPEC" Hadamard-fold
// section, y = W @ WHT(signs * P(x)), with W in the one-bit format of the
// "Inside the One-Bit Engine" page (first station; scale per 128 weights
// applied to each group's sum).  The rotation runs first (rotate.cu) and
// leaves xt in bf16.
//
// CTA tile: 128 weight rows (UMMA M = 128, one TMEM lane per row) x 128
// tokens (UMMA N = 128).  Per 128-wide K-group g:
//   * warp 8 (one lane) TMA-loads the xt tile [128 tokens][128 K] as two
//     128-byte-swizzled boxes of 64 columns;
//   * warps 10-13 (one thread per weight row) expand that row's 128 bits of the
//     group into +-1 bf16 directly in the same swizzled K-major layout (TMA
//     cannot expand bits).  The prefill repack stores even weights in the low
//     half-word and odd weights in the high half-word, so each bf16x2 pair is
//     one shift and one XOR-mask;
//   * warp 9 (one lane) issues 8 MMAs of K = 16 into TMEM accumulator
//     buffer g % 2 (overwriting it at the first), then commits to the stage's
//     "empty" barrier and the buffer's "full" barrier;
//   * warps 0-7 read the buffer back (tcgen05.ld), hand it back to the MMA
//     warp, and accumulate scale[n][g] * D into f32 registers - the per-group
//     scale promotion.  Warp w serves TMEM lanes 32*(w%4).. and columns
//     64*(w/4) .. 64*(w/4)+63.
// Three shared-memory stages (64 KB each) and two TMEM buffers keep the
// producers one to two groups ahead of the MMAs and the MMAs one group ahead
// of the epilogue.  Every wait is bounded in time; on expiry the kernel stops
// its loops, drains its own copies and MMAs, frees TMEM and records
// a timeout in the handle's error word.
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
constexpr int kStageBytes = 32768;  // one operand tile: 128 rows x 128 bf16
constexpr int kTmemCols = 256;      // two f32 accumulators of 128 columns

struct __align__(8) Barriers {
    uint64_t fullA[kPrefillStages];
    uint64_t fullB[kPrefillStages];
    uint64_t empty[kPrefillStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t never;     // no one arrives here: used by the stall test hook
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr int kSmemBytes = 2 * kPrefillStages * kStageBytes + (int)sizeof(Barriers) + 1024;

__global__ void __launch_bounds__(kThreads, 1)
    bitlin_tc_gemm(const __grid_constant__ CUtensorMap tmap_xt, const PrefillParams p, int stall_test)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* tileA = smem;                                   // [stage][32 KB]
    unsigned char* tileB = smem + kPrefillStages * kStageBytes;    // [stage][32 KB]
    Barriers* bar = reinterpret_cast<Barriers*>(smem + 2 * kPrefillStages * kStageBytes);
    volatile int* abort = &bar->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kPrefillRows;
    const int m0 = blockIdx.y * kPrefillTokens;
    const int G = p.K / 128;
    const long long budget = p.wait_budget_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPrefillStages; ++s) {
            ptx::mbar_init(&bar->fullA[s], 128);
            ptx::mbar_init(&bar->fullB[s], 1);
            ptx::mbar_init(&bar->empty[s], 1);
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
    if (warp == kTmaWarp && lane == 0) ptx::prefetch_tmap(&tmap_xt);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bar->tmem_base;

    if (warp == kTmaWarp) {
        if (lane == 0) {
            int issued = 0;
            for (int g = 0; g < G; ++g) {
                const int st = g % kPrefillStages;
                const uint32_t ph = (uint32_t)(g / kPrefillStages) & 1u;
                if (!ptx::mbar_wait_bounded(&bar->empty[st], ph ^ 1u, abort, budget)) break;
                ptx::mbar_arrive_expect_tx(&bar->fullB[st], kStageBytes);
                unsigned char* dst = tileB + st * kStageBytes;
                ptx::tma_load_2d(dst, &tmap_xt, g * 128, m0, &bar->fullB[st]);
                ptx::tma_load_2d(dst + kStageBytes / 2, &tmap_xt, g * 128 + 64, m0, &bar->fullB[st]);
                issued = g + 1;
            }
            // Every copy this lane issued must land before the CTA may exit.
            for (int g = (issued > kPrefillStages ? issued - kPrefillStages : 0); g < issued; ++g) {
                const int st = g % kPrefillStages;
                const uint32_t ph = (uint32_t)(g / kPrefillStages) & 1u;
                volatile int no_abort = 0;
                ptx::mbar_wait_bounded(&bar->fullB[st], ph, &no_abort, budget);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(kPrefillRows, kPrefillTokens);
            int issued = 0;
            for (int g = 0; g < G; ++g) {
                const int st = g % kPrefillStages;
                const uint32_t ph = (uint32_t)(g / kPrefillStages) & 1u;
                const int buf = g & 1;
                const uint32_t tph = (uint32_t)(g >> 1) & 1u;
                if (!ptx::mbar_wait_bounded(&bar->fullA[st], ph, abort, budget)) break;
                if (!ptx::mbar_wait_bounded(&bar->fullB[st], ph, abort, budget)) break;
                if (!ptx::mbar_wait_bounded(&bar->tempty[buf], tph ^ 1u, abort, budget)) break;
                ptx::tc_fence_after();
                const uint32_t a0 = ptx::smem_u32(tileA + st * kStageBytes);
                const uint32_t b0 = ptx::smem_u32(tileB + st * kStageBytes);
                const uint32_t d = tmem + (uint32_t)(buf * kPrefillTokens);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)((kk >> 2) * (kStageBytes / 2) + (kk & 3) * 32);
                    ptx::mma_bf16(d, ptx::smem_desc_sw128(a0 + off), ptx::smem_desc_sw128(b0 + off),
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
        const int r = (warp - kExpWarp0) * 32 + lane;   // row within the tile
        const int n = n0 + r;
        const bool valid = n < p.N;
        const uint4* src = reinterpret_cast<const uint4*>(p.bits + (size_t)(valid ? n : 0) * (p.K / 32));
        uint4 wq = valid ? __ldg(src) : make_uint4(0, 0, 0, 0);
        for (int g = 0; g < G; ++g) {
            const int st = g % kPrefillStages;
            const uint32_t ph = (uint32_t)(g / kPrefillStages) & 1u;
            uint4 wn = make_uint4(0, 0, 0, 0);
            if (valid && g + 1 < G) wn = __ldg(src + g + 1);
            if (!ptx::mbar_wait_bounded(&bar->empty[st], ph ^ 1u, abort, budget)) break;
            unsigned char* dst = tileA + st * kStageBytes + r * 128;
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
                *reinterpret_cast<uint4*>(dst + atom * (kStageBytes / 2) + ((cc ^ (r & 7)) << 4)) =
                    make_uint4(v[0], v[1], v[2], v[3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bar->fullA[st]);
            wq = wn;
        }
    } else {
        // Epilogue warps 0..7.
        const int q = warp & 3, half = warp >> 2;
        const int r = 32 * q + lane;
        const int n = n0 + r;
        const bool valid = n < p.N;
        float acc[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = 0.f;
        const uint16_t* srow = p.scales + (size_t)(valid ? n : 0) * G;
        bool ok = true;
        for (int g = 0; g < G && ok; ++g) {
            const int buf = g & 1;
            const uint32_t tph = (uint32_t)(g >> 1) & 1u;
            const float s = valid ? __half2float(__ushort_as_half(__ldg(srow + g))) : 0.f;
            uint64_t* wbar = (stall_test && g == 0) ? &bar->never : &bar->tfull[buf];
            ok = ptx::mbar_wait_bounded(wbar, tph, abort, budget);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kPrefillTokens + 64 * half);
            float v[32];
            ptx::tmem_ld32(taddr, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = fmaf(s, v[j], acc[j]);
            ptx::tmem_ld32(taddr + 32, v);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar->tempty[buf]);
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[32 + j] = fmaf(s, v[j], acc[32 + j]);
        }
        if (ok && valid) {
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const int m = m0 + 64 * half + j;
                if (m < p.M) p.y[(size_t)m * p.N + n] = acc[j];
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && bar->abort) atomicExch(p.dev_error, kDevErrTimeout);
}

}  // namespace

cudaError_t bitlin_launch_prefill(const PrefillParams& p, const void* tmap, int stall_test,
                                  cudaStream_t s)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(bitlin_tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid((p.N + kPrefillRows - 1) / kPrefillRows, (p.M + kPrefillTokens - 1) / kPrefillTokens);
    bitlin_tc_gemm<<<grid, kThreads, kSmemBytes, s>>>(*static_cast<const CUtensorMap*>(tmap), p,
                                                      stall_test);
    return cudaGetLastError();
}
