// Embedding lookup with the inverse rotation: for token id t of ids[M],
// out[m] = signs * WHT1024(z) / 32 per block, where z is row t of the folded
// one-bit matrix dequantized (bit 1 -> +scale, 0 -> -scale, scale per 128).
// Pulse "ARCHITECTURE-SPEC", Hadamard-fold section: the embedding side of the
// fold applies the transform first and the signs after (the inverse of the
// activation order), so that a row written this way and read back through the
// activation rotation returns to the dequantized row.  Q1G128 row format of the
// "Inside the One-Bit Engine" page (station on the embedding row).
//
// One warp per (token, 1024-block).  The bits come from the handle's
// tensor-path copy ([N][K/32], each word's even weights in the low half-word
// and odd weights in the high half-word).  Lane q loads word q of the block
// (one coalesced load per warp) and its scale, and holds elements 32q + e of
// the block in registers e = 0..31; the transform is separable over the ten
// index bits, so the five stages over bits 0-4 run in registers, a padded
// shared-memory transpose gives lane q the elements 32p + q (p = 0..31), the
// five stages over bits 5-9 run in registers, and the stores are coalesced.
// No shuffles (160 per warp with the bits 0-4 stages across lanes).
// Memory-bound: K/8 + K/64 bytes read and 4K written per token.
#include <cuda_fp16.h>

#include "bitlin_internal.cuh"

namespace {

using namespace bitlin_impl;

constexpr int kEmbedWarps = 8;

// In-register butterflies over the five bits of the register index.
__device__ __forceinline__ void butterflies32(float (&v)[32])
{
#pragma unroll
    for (int st = 1; st < 32; st <<= 1) {
#pragma unroll
        for (int p = 0; p < 32; ++p) {
            if ((p & st) == 0) {
                const float a = v[p], c = v[p + st];
                v[p] = a + c;
                v[p + st] = a - c;
            }
        }
    }
}

__global__ void __launch_bounds__(32 * kEmbedWarps) bitlin_embed_rows(const uint32_t* __restrict__ bits,
                                                                     const uint16_t* __restrict__ scales,
                                                                     const float* __restrict__ signs,
                                                                     const int32_t* __restrict__ ids, int M, int N,
                                                                     int K, float* __restrict__ out, int* dev_error)
{
    __shared__ float tr[kEmbedWarps][32][33];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int B = K / 1024;
    if (gw >= (long long)M * B) return;
    const int m = (int)(gw / B), b = (int)(gw - (long long)m * B);
    float* dst = out + (size_t)m * K + (size_t)b * 1024;
    const int id = __ldg(ids + m);
    if (id < 0 || id >= N) {
#pragma unroll
        for (int p = 0; p < 32; ++p) dst[32 * p + lane] = 0.f;
        if (lane == 0) atomicExch(dev_error, kDevErrIndex);
        return;
    }
    // Word `lane` of the block: element 32 * lane + e is bit e / 2 (e even) or
    // 16 + e / 2 (e odd); its scale is group (32 * lane) / 128.
    const uint32_t w = __ldg(bits + (size_t)id * (K / 32) + b * 32 + lane);
    const float s = __half2float(__ushort_as_half(__ldg(scales + (size_t)id * (K / 128) + b * 8 + (lane >> 2))));
    const uint32_t sb = __float_as_uint(s);
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const uint32_t bit = (w >> ((e & 1) ? 16 + (e >> 1) : (e >> 1))) & 1u;
        v[e] = __uint_as_float(sb ^ ((bit ^ 1u) << 31));  // 1 -> +s, 0 -> -s
    }
    butterflies32(v);  // index bits 0-4
    float(*t)[33] = tr[wib];
#pragma unroll
    for (int e = 0; e < 32; ++e) t[lane][e] = v[e];
    __syncwarp();
#pragma unroll
    for (int p = 0; p < 32; ++p) v[p] = t[p][lane];  // element 32p + lane
    butterflies32(v);  // index bits 5-9
#pragma unroll
    for (int p = 0; p < 32; ++p) {
        const int k = b * 1024 + 32 * p + lane;
        dst[32 * p + lane] = v[p] * 0.03125f * __ldg(signs + k);
    }
}

}  // namespace

cudaError_t bitlin_launch_embed(const uint32_t* bits, const uint16_t* scales, const float* signs,
                                const int32_t* ids, int M, int N, int K, float* out, int* dev_error,
                                cudaStream_t s)
{
    const long long warps = (long long)M * (K / 1024);
    const int threads = 32 * kEmbedWarps;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    bitlin_embed_rows<<<(unsigned)blocks, threads, 0, s>>>(bits, scales, signs, ids, M, N, K, out, dev_error);
    return cudaGetLastError();
}
