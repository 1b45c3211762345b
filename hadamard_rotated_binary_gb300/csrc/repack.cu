// Load-time repacking of a folded 1-bit matrix into the layouts the kernels read.
//
// The "Inside the One-Bit Engine" page (station on the band-interleaved
// repack) copies every matrix once at load into the order its fastest decode
// kernel wants and retires the original.  bitlin does the same at
// bitlin_create: the caller's row-major bits and scales become
//
//  * the decode layout: for slice s (512 weights along K) and tile t (32
//    rows), 2048 bytes of bits as [step 0..3][lane 0..31][4 words] followed,
//    in a separate array, by 256 bytes of scales as [lane][4 x fp16].  Lane L
//    owns row 32t + L.  Its 16 words of the slice are stored in the order it
//    consumes them: position p holds word p ^ (L & 15) of the slice, and for
//    L >= 16 the two byte pairs of every word are swapped.  Its 4 scales are
//    stored in consumption order too: position u holds the scale of the
//    slice's group u ^ ((L & 15) >> 2).  This order lets the decode kernel's
//    32 lanes hit 32 different shared-memory banks on every table lookup
//    (see decode.cu) and makes every global load a coalesced 16-byte load.
//
//  * the prefill layout: row-major [N][K/32] words, but within each word the
//    16 even-indexed weights come first (bit i = weight 2i) and the 16 odd
//    ones second (bit 16 + i = weight 2i + 1), so one shift and one logic op
//    turn a weight pair into a bf16x2 of +-1 (see prefill.cu).
#include "bitlin_internal.cuh"

namespace {

using namespace bitlin_impl;

__global__ void bitlin_repack_decode(const uint32_t* __restrict__ bits,
                                     const uint16_t* __restrict__ scales, int N, int K, int T,
                                     uint4* __restrict__ dbits, uint2* __restrict__ dscales)
{
    const int S = K / kSlice;
    const long long total = (long long)S * T * 32;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= total) return;
    const int lane = (int)(gid & 31);
    const long long unit = gid >> 5;          // s * T + t
    const int s = (int)(unit / T);
    const int t = (int)(unit - (long long)s * T);
    const int n = t * kTileRows + lane;
    const int words_per_row = K / 32;
    const int groups_per_row = K / 128;
    const bool valid = n < N;
    const int x = lane & 15;

    uint32_t w[kWordsPerSlice];
#pragma unroll
    for (int p = 0; p < kWordsPerSlice; ++p) {
        uint32_t v = 0;
        if (valid) v = bits[(size_t)n * words_per_row + s * kWordsPerSlice + (p ^ x)];
        if (lane >= 16) v = __byte_perm(v, 0, 0x2301);  // swap bytes 0<->1 and 2<->3
        w[p] = v;
    }
#pragma unroll
    for (int step = 0; step < 4; ++step)
        dbits[(unit * 4 + step) * 32 + lane] =
            make_uint4(w[4 * step], w[4 * step + 1], w[4 * step + 2], w[4 * step + 3]);

    uint16_t sc[kGroupsPerSlice];
#pragma unroll
    for (int u = 0; u < kGroupsPerSlice; ++u)
        sc[u] = valid ? scales[(size_t)n * groups_per_row + s * kGroupsPerSlice + (u ^ (x >> 2))]
                      : (uint16_t)0;
    dscales[unit * 32 + lane] = make_uint2((uint32_t)sc[0] | ((uint32_t)sc[1] << 16),
                                           (uint32_t)sc[2] | ((uint32_t)sc[3] << 16));
}

// Even bits to the low half-word, odd bits to the high half-word.
__device__ __forceinline__ uint32_t unshuffle_bits(uint32_t v)
{
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        r |= ((v >> (2 * i)) & 1u) << i;
        r |= ((v >> (2 * i + 1)) & 1u) << (16 + i);
    }
    return r;
}

__global__ void bitlin_repack_tc(const uint32_t* __restrict__ bits, long long words,
                                      uint32_t* __restrict__ pbits)
{
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid < words) pbits[gid] = unshuffle_bits(bits[gid]);
}

__global__ void bitlin_check_signs(const float* __restrict__ signs, int K, int* bad)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < K) {
        const float v = signs[i];
        if (!(v == 1.0f || v == -1.0f)) atomicAdd(bad, 1);
    }
}

}  // namespace

cudaError_t bitlin_launch_repack_decode(const uint32_t* bits, const uint16_t* scales, int N, int K,
                                        uint4* dbits, uint2* dscales, cudaStream_t s)
{
    const int T = (N + kTileRows - 1) / kTileRows;
    const long long total = (long long)(K / kSlice) * T * 32;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    bitlin_repack_decode<<<(unsigned)blocks, threads, 0, s>>>(bits, scales, N, K, T, dbits, dscales);
    return cudaGetLastError();
}

cudaError_t bitlin_launch_repack_prefill(const uint32_t* bits, int N, int K, uint32_t* pbits,
                                         cudaStream_t s)
{
    const long long words = (long long)N * (K / 32);
    const int threads = 256;
    const long long blocks = (words + threads - 1) / threads;
    bitlin_repack_tc<<<(unsigned)blocks, threads, 0, s>>>(bits, words, pbits);
    return cudaGetLastError();
}

cudaError_t bitlin_launch_check_signs(const float* signs, int K, int* bad, cudaStream_t s)
{
    bitlin_check_signs<<<(K + 255) / 256, 256, 0, s>>>(signs, K, bad);
    return cudaGetLastError();
}
