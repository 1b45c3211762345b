// Internal declarations shared by the bitlin CUDA sources (not part of the C-ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "bitlin.h"

namespace bitlin_impl {

// ---- per-device set-up -----------------------------------------------------
// Kernel attributes (cudaFuncSetAttribute) and occupancy queries apply to the
// device that is current when they run, so the launchers set them up once per
// device ordinal, under a lock, with that device current.
constexpr int kMaxDevices = 64;

struct PerDeviceOnce {
    std::atomic<int> done[kMaxDevices] = {};
    std::mutex mu;

    // Runs fn(dev) once for the current device (again after a failure);
    // *dev receives the current device's ordinal.
    template <class F>
    cudaError_t run(int* dev, F&& fn)
    {
        cudaError_t e = cudaGetDevice(dev);
        if (e != cudaSuccess) return e;
        if (*dev < 0 || *dev >= kMaxDevices) return cudaErrorInvalidDevice;
        if (done[*dev].load(std::memory_order_acquire)) return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu);
        if (done[*dev].load(std::memory_order_relaxed)) return cudaSuccess;
        e = fn(*dev);
        if (e == cudaSuccess) done[*dev].store(1, std::memory_order_release);
        return e;
    }
};

// ---- decode layout -------------------------------------------------------
// The decode GEMV works on units of (32 rows) x (512 weights along K): a
// "tile" of one "slice".  Each slice is half of a 1024-wide transform block.
constexpr int kSlice = 512;           // weights along K per lookup table
constexpr int kTileRows = 32;         // rows per tile (one row per lane)
constexpr int kWordsPerSlice = 16;    // uint32 words of one row in one slice
constexpr int kGroupsPerSlice = 4;    // 128-weight scale groups per slice
#ifndef BITLIN_DECODE_THREADS
#define BITLIN_DECODE_THREADS 512
#endif
constexpr int kDecodeThreads = BITLIN_DECODE_THREADS;  // 16 warps per CTA, one CTA per SM
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kLutBytes = 65536;      // 64 octet tables x 256 entries x f32

// ---- prefill layout ------------------------------------------------------
constexpr int kPrefillRows = 128;     // weight rows per CTA (UMMA M)
constexpr int kPrefillTokens = 128;   // tokens per CTA (UMMA N)
constexpr int kPrefillMinM = 64;      // auto path: bf16 tensor path from this M
// Auto path: the decode GEMV up to this M (tokens two at a time, each pair
// with its own tables).  Measured against the exact tensor path: gate_up
// 5120 x 34816 at M = 6: 34.1 us against 38.3 us, at M = 8: 44.2 against 38.5;
// ffn_down 17408 x 5120 at M = 6: 23.7 against 24.7, at M = 8: 29.1 against 24.8.
constexpr int kDecodeMaxM = 6;

// Device-side error word values (bitlin_t::dev_error).
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrIndex = 2;      // a token id outside [0, N) (embedding lookup)

struct DecodeParams {
    const uint4* bits;      // [S][T][4][32] uint4 (repacked, see repack.cu)
    const uint2* scales;    // [S][T][32] uint2 (4 x fp16 per lane)
    const float* signs;     // [K]
    const float* x;         // [M][K]
    float* y;               // [M][N]
    float* partials;        // [S][M][T*32], fully rewritten by every call (scratch split-K)
    int M, N, K, S, T, perm;
    int ctas_per_slice;     // set by the launcher
    int split_q, split_r;   // set by the launcher: T = split_q * ctas_per_slice + split_r
    unsigned s_mul;         // set by the launcher: ceil(2^32 / S), for division by S in the kernel
    int pbuf_bytes;         // set by the launcher: cluster split-K partial sums per CTA (bytes)
    int cluster;            // set by the launcher: 1 = split-K summed across a thread-block cluster
    int allow_cluster;      // set by the caller: 0 keeps the split-K in the global scratch
    int swiglu;             // 1: x is [M][2K] (gate | up); the GEMV's input is silu(gate) * up
    // Greedy argmax fused into the cluster split-K finish (nullptr: none): each
    // CTA reduces the outputs it writes to one (value, index) candidate,
    // amax_cand[m * kArgmaxSlots + blockIdx.x], and the CTA that takes token m's
    // last ticket picks ids[m] and re-arms the ticket.
    int32_t* ids;           // [M]
    float2* amax_cand;      // [M][kArgmaxSlots]
    unsigned* amax_tickets; // [M], zero between calls
};

// Candidate slots per token for the argmax (at least the decode grid and the
// argmax kernel's chunk count).
constexpr int kArgmaxSlots = 256;

// Total order of the greedy pick: a NaN above every number, then the usual
// order, and among equal values the smaller index.
__device__ __forceinline__ bool argmax_better(float v, int i, float bv, int bi)
{
    const bool vn = v != v, bn = bv != bv;
    if (vn != bn) return vn;
    if (!vn && v != bv) return v > bv;
    return i < bi;
}

struct PrefillParams {
    const uint32_t* bits;   // [N][K/32], prefill bit order (see repack.cu)
    const uint16_t* scales; // [N][K/128]
    float* y;               // [M][N]
    int* dev_error;
    int M, N, K;
    int num_sms;            // for the split-K choice
    long long wait_budget_ns;
    // Set by the launcher (persistent grid): tiles along N, and the launch's
    // tiles: tiles tile_base .. tile_base + tiles - 1 of the row-major tile grid.
    int tiles_x, tiles, tile_base;
};

}  // namespace bitlin_impl

struct bitlin {
    int device = 0;
    int num_sms = 0;
    int N = 0, K = 0, perm = 0;
    int S = 0, T = 0;
    int path = BITLIN_PATH_AUTO;
    int last_cuda_error = 0;
    bitlin_status sticky = BITLIN_OK;

    // decode copy of the weights
    uint4* dbits = nullptr;
    uint2* dscales = nullptr;
    // prefill copy of the weights
    uint32_t* pbits = nullptr;
    uint16_t* pscales = nullptr;
    float* signs = nullptr;

    // scratch
    float* partials = nullptr;
    int partials_M = 0;
    void* xt = nullptr;        // bf16 [M][K] rotated activations for the prefill path
    int xt_M = 0;
    alignas(64) unsigned char tmap[128];       // TMA descriptor of xt (a CUtensorMap)
    alignas(64) unsigned char tmap_bits[128];  // TMA descriptor of the tensor-path bits
    int tmap_M = 0;
    int tmap_exact = -1;
    int* dev_error = nullptr;  // device error word [0]; [1] is create's sign check
    int* h_err = nullptr;      // pinned copy of the error word
    long long wait_budget_ns = 0;
    int stall_test = 0;
    // The device reads pageable host memory coherently through the host's page
    // tables (a hardware-coherent CPU-GPU link): bitlin_forward_host may then
    // hand the caller's buffers to the kernels as they are.
    int host_page_tables = 0;

    // MLP block (bitlin_mlp_forward on the down-projection handle): the gate and
    // up outputs [M][2K] that the down projection reads through SiLU
    float* mlp_in = nullptr;
    int mlp_M = 0;
    // bitlin_argmax without a caller buffer: the scores [M][N]
    float* logits = nullptr;
    int logits_M = 0;
    void* amax_cand = nullptr;      // per-chunk (value, index) candidates
    unsigned* amax_tickets = nullptr;  // one per token, zero between calls
    int amax_M = 0;

    // host-buffer entry point staging
    float* hx = nullptr;
    float* hy = nullptr;
    int h_M = 0;
};

// Launchers (return a cudaError_t).
cudaError_t bitlin_launch_repack_decode(const uint32_t* bits, const uint16_t* scales, int N, int K,
                                        uint4* dbits, uint2* dscales, cudaStream_t s);
cudaError_t bitlin_launch_repack_prefill(const uint32_t* bits, int N, int K, uint32_t* pbits,
                                         cudaStream_t s);
cudaError_t bitlin_launch_check_signs(const float* signs, int K, int* bad, cudaStream_t s);
cudaError_t bitlin_launch_decode(const bitlin_impl::DecodeParams& p, int num_sms, cudaStream_t s);
// Kernels one bitlin_launch_decode of p launches: 1 (cluster split-K) or 2 (GEMV, then the sum).
// *fused_argmax: 1 when that launch can also pick the argmax (p.ids), 0 otherwise.
cudaError_t bitlin_decode_kernels(const bitlin_impl::DecodeParams& p, int num_sms, int* kernels,
                                  int* fused_argmax = nullptr);
cudaError_t bitlin_launch_argmax(const float* y, int M, int N, void* cand, unsigned* tickets, int32_t* ids,
                                 cudaStream_t s);
size_t bitlin_argmax_scratch_bytes(int M);
cudaError_t bitlin_launch_embed(const uint32_t* bits, const uint16_t* scales, const float* signs,
                                const int32_t* ids, int M, int N, int K, float* out, int* dev_error,
                                cudaStream_t s);
cudaError_t bitlin_launch_rotate_bf16(const float* x, const float* signs, int M, int K, int perm,
                                      int digits, int swiglu, void* xt, cudaStream_t s);
cudaError_t bitlin_launch_prefill(const bitlin_impl::PrefillParams& p, const void* tmap,
                                  const void* tmap_bits, int stall_test, cudaStream_t s);
cudaError_t bitlin_launch_tc_exact(const bitlin_impl::PrefillParams& p, const void* tmap,
                                   const void* tmap_bits, int stall_test, cudaStream_t s);
// Rows of B per tensor-core tile: 64 or 128 tokens (bf16 path) or 64/128 digit rows (exact).
int bitlin_tc_tile_width(int M, int exact);
// GEMM launches of a bf16 tensor-path call: 2 when the tiles past the last
// full wave get a split-K launch of their own, else 1.
int bitlin_prefill_gemm_launches(int M, int N, int num_sms);
