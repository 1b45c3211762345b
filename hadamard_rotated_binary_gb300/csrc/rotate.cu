// Stand-alone activation rotation for the tensor-core paths: x f32 [M][K] ->
// xt = WHT1024(signs * P(x)) / 32 per block, stored as bf16 (round to nearest
// even).  Prefill mode: one row per token, xt [M][K].  Exact mode: four rows
// per token, [4M][K]: rows 4m, 4m+1, 4m+2 hold the digits hi = bf16(xt),
// mid = bf16(xt - hi), lo = bf16(xt - hi - mid), whose sum is the f32 value,
// and row 4m+3 is zero.  Pulse "ARCHITECTURE-SPEC", Hadamard-fold section
// (order: optional tiled->grouped permutation, x * signs, normalized
// Sylvester-Walsh transform in blocks of 1024 scaled by 1/32).
//
// One warp per (token, block).  The 1024-point transform is separable over the
// ten bits of the element index, so any placement of the elements on lanes and
// registers works if each bit's butterflies pair the right values.  Vector
// variant (x 16-byte aligned): element i = 128 p + 4 q + j (p < 8, j < 4)
// sits in register 4p + j of lane q, so each lane reads 8 float4 and writes 8
// groups of 4 bf16.  Its five register bits are element bits 0-1 and 7-9; a
// padded shared-memory transpose puts element bits 2-6 in the registers for
// the other five stages and a second one restores the placement for the
// packed stores: no warp shuffles.  Scalar variant (any alignment): element
// i = 32 p + q in register p of lane q, the stages in the same bit order (so
// both variants round alike), lane bits by shuffles.  Memory-bound: 4 bytes
// read and 2 written per element (4 x 2 in the exact mode).  Five CTAs of 8
// warps per SM, so that one wave covers 1024 tokens of 5120.
#include <cuda_bf16.h>

#include "bitlin_internal.cuh"

namespace {

__device__ __forceinline__ int perm_source(int k)
{
    const int head = k >> 7, d = k & 127;
    const int r = head % 3, kk = head / 3;
    return d + 128 * (kk + 16 * r);
}

// The rotated values of one (token, block), 32 per lane, written as bf16 (one
// row) or as three digits and a zero row, one element at a time.  off(r) is
// the block offset of register r of this lane.
template <typename Off>
__device__ __forceinline__ void store_rotated(const float (&v)[32], __nv_bfloat16* out, int K, int digits,
                                              Off off)
{
    if (!digits) {
#pragma unroll
        for (int r = 0; r < 32; ++r) out[off(r)] = __float2bfloat16_rn(v[r] * 0.03125f);
        return;
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const float t = v[r] * 0.03125f;  // exact scaling by 1/32
        const __nv_bfloat16 hi = __float2bfloat16_rn(t);
        const float r1 = t - __bfloat162float(hi);  // exact
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);  // exact
        const int k = off(r);
        out[k] = hi;
        out[(size_t)K + k] = mid;
        out[2 * (size_t)K + k] = __float2bfloat16_rn(r2);
        out[3 * (size_t)K + k] = __float2bfloat16_rn(0.f);
    }
}

// The vector placement: registers 4p .. 4p+3 of lane q are the consecutive
// elements 128 p + 4 q .. + 3, stored as one 8-byte group per row.
__device__ __forceinline__ uint2 pack4(float a, float b, float c, float d)
{
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

__device__ __forceinline__ void store_rotated_vec(const float (&v)[32], __nv_bfloat16* out, int K, int digits,
                                                  int lane)
{
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float t[4], d1[4], d2[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            t[j] = v[4 * p + j] * 0.03125f;  // exact scaling by 1/32
            d1[j] = t[j] - __bfloat162float(__float2bfloat16_rn(t[j]));  // exact
            d2[j] = d1[j] - __bfloat162float(__float2bfloat16_rn(d1[j]));  // exact
        }
        uint2* o = reinterpret_cast<uint2*>(out + 128 * p + 4 * lane);
        o[0] = pack4(t[0], t[1], t[2], t[3]);  // bf16(t): the row, or the hi digit
        if (digits) {
            o[K / 4] = pack4(d1[0], d1[1], d1[2], d1[3]);      // mid = bf16(t - hi)
            o[K / 2] = pack4(d2[0], d2[1], d2[2], d2[3]);      // lo = bf16(t - hi - mid)
            o[3 * (K / 4)] = make_uint2(0u, 0u);                // zero row
        }
    }
}

// Butterflies over the register-index bits st = lo, 2 lo, .. < hi.
__device__ __forceinline__ void reg_butterflies(float (&v)[32], int lo, int hi)
{
#pragma unroll
    for (int st = lo; st < hi; st <<= 1) {
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

// Butterflies over the lane bits st = lo, 2 lo, .. < hi (warp shuffles).
__device__ __forceinline__ void lane_butterflies(float (&v)[32], int lane, int lo, int hi)
{
#pragma unroll
    for (int st = lo; st < hi; st <<= 1) {
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const float o = __shfl_xor_sync(0xffffffffu, v[r], st);
            v[r] = (lane & st) ? (o - v[r]) : (v[r] + o);
        }
    }
}

__device__ __forceinline__ float silu_times(float g, float u) { return g / (1.f + expf(-g)) * u; }

// VEC: element i = 128 p + 4 q + j in register 4p + j of lane q (x 16-byte
// aligned); otherwise element i = 32 p + q in register p.  SWIGLU: x is
// [M][2K] gate | up and the input is silu(gate) * up, SiLU(g) = g / (1 + e^-g)
// in f32 ("Inside the One-Bit Engine", MLP station).
template <bool VEC, bool SWIGLU>
__global__ void __launch_bounds__(256, 5) bitlin_rotate_bf16(const float* __restrict__ x,
                                                          const float* __restrict__ signs, int M, int K,
                                                          int perm, int digits, __nv_bfloat16* __restrict__ xt)
{
    // Programmatic dependent launch: the GEMM that reads xt may launch (and set
    // up) while this grid runs; x may come from the previous kernel, so wait for
    // it before reading.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float tr[VEC ? 8 : 1][32][33];
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int B = K / 1024;
    if (gw >= (long long)M * B) return;
    const int m = (int)(gw / B), b = (int)(gw - (long long)m * B);
    const float* xm = x + (size_t)m * (SWIGLU ? 2 * K : K);
    float v[32];
    if (VEC) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int k = b * 1024 + 128 * p + 4 * lane;
            const int src = perm ? perm_source(k) : k;  // heads move whole: src stays a multiple of 4
            float4 a = __ldg(reinterpret_cast<const float4*>(xm + src));
            if (SWIGLU) {
                const float4 u = __ldg(reinterpret_cast<const float4*>(xm + K + src));
                a = make_float4(silu_times(a.x, u.x), silu_times(a.y, u.y), silu_times(a.z, u.z),
                                silu_times(a.w, u.w));
            }
            const float4 sg = __ldg(reinterpret_cast<const float4*>(signs + k));
            v[4 * p + 0] = a.x * sg.x;
            v[4 * p + 1] = a.y * sg.y;
            v[4 * p + 2] = a.z * sg.z;
            v[4 * p + 3] = a.w * sg.w;
        }
        // All five register bits (element bits 0-1 and 7-9) in registers,
        // a transpose through shared memory, the five lane bits (element
        // bits 2-6) in registers, and the transpose back for packed stores.
        reg_butterflies(v, 1, 32);
        float(*t)[33] = tr[threadIdx.x >> 5];
#pragma unroll
        for (int r = 0; r < 32; ++r) t[lane][r] = v[r];
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 32; ++r) v[r] = t[r][lane];
        reg_butterflies(v, 1, 32);
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 32; ++r) t[r][lane] = v[r];
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 32; ++r) v[r] = t[lane][r];
        __nv_bfloat16* out = xt + (size_t)(digits ? 4 * m : m) * K + (size_t)b * 1024;
        store_rotated_vec(v, out, K, digits, lane);
        return;
    } else {
#pragma unroll
        for (int p = 0; p < 32; ++p) {
            const int k = b * 1024 + 32 * p + lane;
            const int src = perm ? perm_source(k) : k;
            float a = __ldg(xm + src);
            if (SWIGLU) a = silu_times(a, __ldg(xm + K + src));
            v[p] = a * __ldg(signs + k);
        }
    }
    // Scalar placement (element 32 p + q in register p of lane q), the stages
    // in the vector placement's order, so that both give the same roundings:
    // element bits 0-1 across lanes, 7-9 across registers, 2-4 across lanes,
    // 5-6 across registers.  The lane with the bit clear holds the low element.
    lane_butterflies(v, lane, 1, 4);
    reg_butterflies(v, 4, 32);
    lane_butterflies(v, lane, 4, 32);
    reg_butterflies(v, 1, 4);
    __nv_bfloat16* out = xt + (size_t)(digits ? 4 * m : m) * K + (size_t)b * 1024;
    store_rotated(v, out, K, digits, [lane](int r) { return 32 * r + lane; });
}

}  // namespace

cudaError_t bitlin_launch_rotate_bf16(const float* x, const float* signs, int M, int K, int perm,
                                      int digits, int swiglu, void* xt, cudaStream_t s)
{
    const long long warps = (long long)M * (K / 1024);
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(xt);
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (reinterpret_cast<uintptr_t>(signs) & 15) == 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (vec && swiglu) return cudaLaunchKernelEx(&cfg, bitlin_rotate_bf16<true, true>, x, signs, M, K, perm, digits, out);
    if (vec) return cudaLaunchKernelEx(&cfg, bitlin_rotate_bf16<true, false>, x, signs, M, K, perm, digits, out);
    if (swiglu) return cudaLaunchKernelEx(&cfg, bitlin_rotate_bf16<false, true>, x, signs, M, K, perm, digits, out);
    return cudaLaunchKernelEx(&cfg, bitlin_rotate_bf16<false, false>, x, signs, M, K, perm, digits, out);
}
