// Stand-alone activation rotation for the tensor-core paths: x f32 [M][K] ->
// xt = WHT1024(signs * P(x)) / 32 per block, stored as bf16 (round to nearest
// even).  Prefill mode: one row per token, xt [M][K].  Exact mode: four rows
// per token, [4M][K]: rows 4m, 4m+1, 4m+2 hold the digits hi = bf16(xt),
// mid = bf16(xt - hi), lo = bf16(xt - hi - mid), whose sum is the f32 value,
// and row 4m+3 is zero.  Pulse "ARCHITECTURE-SPEC", Hadamard-fold section
// (order: optional tiled->grouped permutation, x * signs, normalized
// Sylvester-Walsh transform in blocks of 1024 scaled by 1/32).
//
// One warp per (token, block): lane q holds x[32p + q] for p = 0..31 in
// registers (every load and store is a coalesced row of 32 elements).
// H1024 = H32 (x) H32: 32-point butterflies across lanes (warp shuffles) for
// each p, then 32-point butterflies across the 32 registers.  Memory-bound:
// 4 bytes read and 2 written per element.
#include <cuda_bf16.h>

#include "bitlin_internal.cuh"

namespace {

__device__ __forceinline__ int perm_source(int k)
{
    const int head = k >> 7, d = k & 127;
    const int r = head % 3, kk = head / 3;
    return d + 128 * (kk + 16 * r);
}

__global__ void __launch_bounds__(256) bitlin_rotate_bf16(const float* __restrict__ x,
                                                          const float* __restrict__ signs, int M,
                                                          int K, int perm, int digits, int swiglu,
                                                          __nv_bfloat16* __restrict__ xt)
{
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int B = K / 1024;
    if (gw >= (long long)M * B) return;
    const int m = (int)(gw / B), b = (int)(gw - (long long)m * B);
    // With swiglu set, x is [M][2K] gate | up and the input is silu(gate) * up,
    // SiLU(g) = g / (1 + e^-g) in f32 ("Inside the One-Bit Engine", MLP station).
    const float* xm = x + (size_t)m * (swiglu ? 2 * K : K);

    float v[32];
#pragma unroll
    for (int p = 0; p < 32; ++p) {
        const int k = b * 1024 + 32 * p + lane;
        const int src = perm ? perm_source(k) : k;
        float a = __ldg(xm + src);
        if (swiglu) {
            const float u = __ldg(xm + K + src);
            a = a / (1.f + expf(-a)) * u;
        }
        v[p] = a * __ldg(signs + k);
    }
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
    if (!digits) {
        __nv_bfloat16* out = xt + (size_t)m * K + (size_t)b * 1024;
#pragma unroll
        for (int p = 0; p < 32; ++p) out[32 * p + lane] = __float2bfloat16_rn(v[p] * 0.03125f);
        return;
    }
    __nv_bfloat16* out = xt + (size_t)(4 * m) * K + (size_t)b * 1024;
#pragma unroll
    for (int p = 0; p < 32; ++p) {
        const float t = v[p] * 0.03125f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(t);
        const float r1 = t - __bfloat162float(hi);  // exact
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);  // exact
        const int k = 32 * p + lane;
        out[k] = hi;
        out[(size_t)K + k] = mid;
        out[2 * (size_t)K + k] = __float2bfloat16_rn(r2);
        out[3 * (size_t)K + k] = __float2bfloat16_rn(0.f);
    }
}

}  // namespace

cudaError_t bitlin_launch_rotate_bf16(const float* x, const float* signs, int M, int K, int perm,
                                      int digits, int swiglu, void* xt, cudaStream_t s)
{
    const long long warps = (long long)M * (K / 1024);
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    bitlin_rotate_bf16<<<(unsigned)blocks, threads, 0, s>>>(x, signs, M, K, perm, digits, swiglu,
                                                           static_cast<__nv_bfloat16*>(xt));
    return cudaGetLastError();
}
