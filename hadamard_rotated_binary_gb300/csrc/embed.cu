// Embedding lookup with the inverse rotation: for token id t of ids[M],
// out[m] = signs * WHT1024(z) / 32 per block, where z is row t of the folded
// one-bit matrix dequantized (bit 1 -> +scale, 0 -> -scale, scale per 128).
// Pulse "ARCHITECTURE-SPEC", Hadamard-fold section: the embedding side of the
// fold applies the transform first and the signs after (the inverse of the
// activation order), so that a row written this way and read back through the
// activation rotation returns to the dequantized row.  Q1G128 row format of the
// "Inside the One-Bit Engine" page (station on the embedding row).
//
// One warp per (token, 1024-block), as rotate.cu: lane q holds element
// 32p + q of the block for p = 0..31.  The bits come from the handle's
// tensor-path copy ([N][K/32], each word's even weights in the low half-word
// and odd weights in the high half-word), so lane q's bit of word p sits at
// position q/2 (q even) or 16 + q/2 (q odd), the same for every p: one
// broadcast load of the word per p.  Memory-bound: K/8 + K/64 bytes read and
// 4K written per token.
#include <cuda_fp16.h>

#include "bitlin_internal.cuh"

namespace {

using namespace bitlin_impl;

__global__ void __launch_bounds__(256) bitlin_embed_rows(const uint32_t* __restrict__ bits,
                                                         const uint16_t* __restrict__ scales,
                                                         const float* __restrict__ signs,
                                                         const int32_t* __restrict__ ids, int M, int N, int K,
                                                         float* __restrict__ out, int* dev_error)
{
    const int lane = threadIdx.x & 31;
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
    const uint32_t* row = bits + (size_t)id * (K / 32) + b * 32;
    const uint16_t* srow = scales + (size_t)id * (K / 128) + b * 8;
    const int pos = (lane & 1) ? 16 + (lane >> 1) : (lane >> 1);

    float v[32];
#pragma unroll
    for (int p = 0; p < 32; ++p) {
        const float s = __half2float(__ushort_as_half(__ldg(srow + (p >> 2))));
        v[p] = ((__ldg(row + p) >> pos) & 1u) ? s : -s;
    }
    // H1024 = H32 (x) H32: across lanes, then across registers.
#pragma unroll
    for (int st = 1; st < 32; st <<= 1) {
#pragma unroll
        for (int p = 0; p < 32; ++p) {
            const float o = __shfl_xor_sync(0xffffffffu, v[p], st);
            v[p] = (lane & st) ? (o - v[p]) : (v[p] + o);
        }
    }
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
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    bitlin_embed_rows<<<(unsigned)blocks, threads, 0, s>>>(bits, scales, signs, ids, M, N, K, out, dev_error);
    return cudaGetLastError();
}
