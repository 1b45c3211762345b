// Decode GEMV (M < 64): activation rotation fused into the prologue, then the
// one-bit product through shared-memory signed-sum tables.
//
// Method (what is computed) - Pulse "ARCHITECTURE-SPEC", Hadamard-fold
// section: xt = WHT1024(signs * P(x)) / 32 per 1024-block, then y = W @ xt;
// "Inside the One-Bit Engine", first station: weight = +-1 from one bit, one
// scale per 128 weights applied to the group sum.
//
// How (GB300 design):
//  * Work unit = (slice s of 512 weights along K) x (tile t of 32 rows).  A CTA
//    (16 warps, one per SM) takes a contiguous run of units, so it touches one
//    or two slices; split-K partial sums land in a scratch array and the last
//    contributor of each tile (an atomic ticket per tile) adds the slices in
//    fixed order s = 0..S-1 - deterministic results.
//  * Prologue per (token, slice): gather x (with the ssm_out permutation when
//    requested), multiply by the signs, and form the 512 outputs of the
//    1024-point transform that the slice needs: with H1024 = [[H, H], [H, -H]],
//    half h of the block is H512(x_lo + (-1)^h x_hi) / 32.  H512 = H16 (x) H32 is
//    done as 32-point butterflies across lanes (warp shuffles), a transpose
//    through shared memory, and 16-point butterflies across lanes.
//  * Table: for each of the slice's 64 octets (8 weights), the 256 possible
//    signed sums sum_i (+-1) xt_i, f32, 64 KB.  It generalises the engine page's
//    subset-sum table trick (station on the LUT kernel: sixteen answers per four
//    weights, one multiply by the scale per 128) from nibbles to bytes.
//    Entry b of the table for word w, byte j sits at byte offset
//    b*256 + 128*(j>>1) + 4*(w + 16*(j&1)), i.e. in bank w + 16*(j&1).
//  * Main loop: lane L owns row 32t + L and walks its 16 words in the order
//    w = p ^ (L & 15); lanes L >= 16 read the bytes of a word in the order
//    j ^ 1 (the repack swapped them).  So at every lookup the 32 lanes read 32
//    different banks - conflict free - and each byte costs one PRMT (which
//    builds the whole shared-memory offset from the byte and a per-lane
//    register), one LDS and one FADD.  Every 4 words (one 128-group) the
//    group sum is multiplied by its fp16 scale with one FFMA.
//  * Weights stream straight from HBM into registers with 16-byte coalesced
//    loads; each warp prefetches its next tile while it computes the current
//    one, and the first tile is requested before the prologue so that DRAM
//    latency overlaps the transform and the table build.
//  * Programmatic dependent launch: the kernel lets its successor launch at
//    once and itself waits (griddepcontrol.wait) only before it reads x or
//    writes any output; weight prefetch precedes the wait.
#include <cuda_fp16.h>

#include "bitlin_internal.cuh"

namespace {

using namespace bitlin_impl;

constexpr int kPad = 33;                               // transpose row stride (floats)
constexpr int kSmemTranspose = 16 * kPad * 4;           // 2112 B
constexpr int kSmemSlice = (kSlice + kSlice / 32) * 4;  // 528 floats
constexpr int kDecodeSmem = kLutBytes + kSmemTranspose + kSmemSlice;

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float lut_at(const unsigned char* lut, uint32_t off)
{
    return *reinterpret_cast<const float*>(lut + off);
}

// Padded index of slice position i (one spare float every 32).
__device__ __forceinline__ int xpad(int i) { return i + (i >> 5); }

__device__ __forceinline__ void load_tile(const DecodeParams& p, int s, int t, int lane, uint4 (&b)[4],
                                          uint2& sc)
{
    const size_t unit = (size_t)s * p.T + t;
    const uint4* src = p.bits + unit * 4 * 32 + lane;
#pragma unroll
    for (int q = 0; q < 4; ++q) b[q] = __ldg(src + q * 32);
    sc = __ldg(p.scales + unit * 32 + lane);
}

// Source column of grouped position k under the ssm_out permutation
// (grouped [hd, rep, nk] <- tiled [hd, nk, rep], hd = 128, nk = 16, rep = 3).
__device__ __forceinline__ int perm_source(int k)
{
    const int head = k >> 7, d = k & 127;
    const int r = head % 3, kk = head / 3;
    return d + 128 * (kk + 16 * r);
}

// Rotated activations of token m for slice s into xs (padded, 512 floats).
__device__ __forceinline__ void build_slice(const DecodeParams& p, int m, int s, float* tbuf,
                                            float* xs, int warp, int lane)
{
    const int b = s >> 1, h = s & 1;
    const int i = 32 * warp + lane;  // 0..511
    const int k0 = b * 1024 + i, k1 = k0 + 512;
    const float* xm = p.x + (size_t)m * p.K;
    const int src0 = p.perm ? perm_source(k0) : k0;
    const int src1 = p.perm ? perm_source(k1) : k1;
    const float a = __ldg(xm + src0) * __ldg(p.signs + k0);
    const float c = __ldg(xm + src1) * __ldg(p.signs + k1);
    float v = h ? (a - c) : (a + c);
    // 32-point butterflies across the lanes (natural Sylvester order).
#pragma unroll
    for (int st = 1; st < 32; st <<= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, st);
        v = (lane & st) ? (o - v) : (v + o);
    }
    tbuf[warp * kPad + lane] = v;
    __syncthreads();
    // 16-point butterflies down the columns: warp w takes columns 2w, 2w+1.
    const int col = 2 * warp + (lane >> 4), row = lane & 15;
    float z = tbuf[row * kPad + col];
#pragma unroll
    for (int st = 1; st < 16; st <<= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, z, st);
        z = (row & st) ? (o - z) : (z + o);
    }
    xs[xpad(row * 32 + col)] = z * 0.03125f;  // exact scaling by 1/32
    __syncthreads();
}

// Signed-sum tables for the slice: warp v writes entries b = 16v .. 16v+15 of
// all 64 tables; lane L writes the two tables of bank L (its word w = L & 15,
// byte parity L >> 4, byte pair jh = 0, 1).
__device__ __forceinline__ void build_tables(const float* xs, unsigned char* lut, int warp, int lane)
{
    const int w = lane & 15, jlo = lane >> 4, hnib = warp;
#pragma unroll
    for (int jh = 0; jh < 2; ++jh) {
        const int j = 2 * jh + jlo;
        const int e = 32 * w + 8 * j;
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = xs[xpad(e + i)];
        float p01[4], p23[4];
        p01[0] = -x[0] - x[1];
        p01[1] = x[0] - x[1];
        p01[2] = x[1] - x[0];
        p01[3] = x[0] + x[1];
        p23[0] = -x[2] - x[3];
        p23[1] = x[2] - x[3];
        p23[2] = x[3] - x[2];
        p23[3] = x[2] + x[3];
        const float a45 = ((hnib & 1) ? x[4] : -x[4]) + ((hnib & 2) ? x[5] : -x[5]);
        const float a67 = ((hnib & 4) ? x[6] : -x[6]) + ((hnib & 8) ? x[7] : -x[7]);
        const float hi = a45 + a67;
        unsigned char* dst = lut + (size_t)(16 * hnib) * 256 + 128 * jh + 4 * lane;
#pragma unroll
        for (int l = 0; l < 16; ++l)
            *reinterpret_cast<float*>(dst + l * 256) = (p01[l & 3] + p23[l >> 2]) + hi;
    }
}

// One tile's dot products for this lane's row: sum over the slice's 4 groups
// of scale * (sum of 16 table lookups).
__device__ __forceinline__ float tile_dot(const unsigned char* lut, const uint4 (&b)[4], uint2 sc,
                                          uint32_t base_off)
{
    const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&sc.x));
    const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(&sc.y));
    const float scl[4] = {s01.x, s01.y, s23.x, s23.y};
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint32_t wv[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
        float g0 = 0.f, g1 = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t pos = 4u * u + c;
            const uint32_t off = base_off ^ ((4u * pos) * 0x101u);
            const uint32_t wd = wv[c];
            g0 += lut_at(lut, __byte_perm(wd, off, 0x7604));
            g1 += lut_at(lut, __byte_perm(wd, off, 0x7615));
            g0 += lut_at(lut + 128, __byte_perm(wd, off, 0x7624));
            g1 += lut_at(lut + 128, __byte_perm(wd, off, 0x7635));
        }
        acc = fmaf(g0 + g1, scl[u], acc);
    }
    return acc;
}

__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(const DecodeParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* lut = smem;
    float* tbuf = reinterpret_cast<float*>(smem + kLutBytes);
    float* xs = tbuf + 16 * kPad;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long U = (long long)p.S * p.T;
    const int u0 = (int)(U * blockIdx.x / gridDim.x);
    const int u1 = (int)(U * (blockIdx.x + 1) / gridDim.x);
    const size_t npad = (size_t)p.T * kTileRows;
    // Per-lane part of every table offset: byte 0 for even bytes, byte 1 for odd.
    const uint32_t base_off = (uint32_t)(4 * (lane & 15) + 64 * (lane >> 4)) |
                              ((uint32_t)(4 * (lane & 15) + 64 * (1 - (lane >> 4))) << 8);

    pdl_launch_dependents();
    bool waited = false;

    for (int u = u0; u < u1;) {
        const int s = u / p.T;
        const int ta = u - s * p.T;
        const int tb = min(p.T, ta + (u1 - u));
        u += tb - ta;

        for (int m = 0; m < p.M; ++m) {
            int t = ta + warp;
            uint4 cb[4];
            uint2 cs = make_uint2(0, 0);
            if (t < tb) load_tile(p, s, t, lane, cb, cs);
            if (!waited) {
                pdl_wait();
                waited = true;
            }
            __syncthreads();  // the previous table is no longer read
            build_slice(p, m, s, tbuf, xs, warp, lane);
            build_tables(xs, lut, warp, lane);
            __syncthreads();
            float* part = p.partials + ((size_t)s * p.M + m) * npad;
            for (; t < tb; t += kDecodeWarps) {
                const int tn = t + kDecodeWarps;
                uint4 nb[4];
                uint2 ns = make_uint2(0, 0);
                if (tn < tb) load_tile(p, s, tn, lane, nb, ns);
                part[(size_t)t * kTileRows + lane] = tile_dot(lut, cb, cs, base_off);
                if (tn < tb) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) cb[q] = nb[q];
                    cs = ns;
                }
            }
        }

        // Publish this segment's partial sums; the last slice in for a tile
        // sums all slices of that tile in order and rearms its ticket.
        __threadfence();
        __syncwarp();
        for (int t = ta + warp; t < tb; t += kDecodeWarps) {
            unsigned prev = 0;
            if (lane == 0) prev = atomicAdd(p.counters + t, 1u);
            prev = __shfl_sync(0xffffffffu, prev, 0);
            if (prev == (unsigned)(p.S - 1)) {
                __threadfence();
                const int n = t * kTileRows + lane;
                for (int m = 0; m < p.M; ++m) {
                    float sum = 0.f;
                    for (int ss = 0; ss < p.S; ++ss)
                        sum += __ldcg(p.partials + ((size_t)ss * p.M + m) * npad + n);
                    if (n < p.N) p.y[(size_t)m * p.N + n] = sum;
                }
                if (lane == 0) p.counters[t] = 0u;
            }
        }
    }
    if (!waited) pdl_wait();
}

}  // namespace

cudaError_t bitlin_launch_decode(const DecodeParams& p, int num_sms, cudaStream_t s)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kDecodeSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const long long U = (long long)p.S * p.T;
    const int grid = (int)(U < num_sms ? U : num_sms);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = kDecodeSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel, p);
}
