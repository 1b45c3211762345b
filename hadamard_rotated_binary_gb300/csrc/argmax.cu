// Greedy token choice after the LM head: ids[m] = the smallest n with
// y[m][n] = max over n of y[m][n] (first index among equal maxima).
// "Inside the One-Bit Engine", station on the LM head: the vocabulary matrix
// (248,320 rows x 5,120, folded like the other one-bit matrices) turns the
// final hidden state into one score per token of the vocabulary; picking one
// word from the scores starts from the largest.
//
// A grid of 256 CTAs per token, each reducing one contiguous chunk of
// the row (strided coalesced reads, four loads in flight per thread; the
// scores were just written and sit in L2) to a (value, index) candidate.
// The CTA that takes a token's last ticket picks among the candidates and
// re-arms the ticket.  The order (largest value, then smallest index) is
// total, so the answer does not depend on which CTA finishes last.  A NaN
// score counts as larger than every number, so a NaN is reported rather
// than hidden.
#include "bitlin_internal.cuh"

namespace {

using bitlin_impl::argmax_better;
using bitlin_impl::kArgmaxSlots;

constexpr int kChunks = kArgmaxSlots;  // one chunk per CTA; the final pick reads one candidate per thread
constexpr int kThreadsA = 256;
static_assert(kChunks <= kThreadsA, "the final pick reads one candidate per thread");

__device__ __forceinline__ void warp_best(float& bv, int& bi)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (argmax_better(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
        }
    }
}

// Block-wide best of (bv, bi); the result is valid in thread 0.
__device__ __forceinline__ void block_best(float& bv, int& bi)
{
    __shared__ float sv[kThreadsA / 32];
    __shared__ int si[kThreadsA / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    warp_best(bv, bi);
    if (lane == 0) {
        sv[warp] = bv;
        si[warp] = bi;
    }
    __syncthreads();
    if (warp == 0) {
        bv = lane < kThreadsA / 32 ? sv[lane] : -__int_as_float(0x7f800000);
        bi = lane < kThreadsA / 32 ? si[lane] : 0x7fffffff;
        warp_best(bv, bi);
    }
}

__global__ void __launch_bounds__(kThreadsA) bitlin_argmax_rows(const float* __restrict__ y, int N,
                                                                float2* __restrict__ cand, unsigned* tickets,
                                                                int32_t* __restrict__ ids)
{
    const int m = blockIdx.y, c = blockIdx.x;
    const float* row = y + (size_t)m * N;
    const int lo = (int)((long long)N * c / kChunks), hi = (int)((long long)N * (c + 1) / kChunks);
    float bv = -__int_as_float(0x7f800000);  // -inf
    int bi = 0x7fffffff;
    for (int n0 = lo + (int)threadIdx.x; n0 < hi; n0 += 4 * kThreadsA) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int n = n0 + u * kThreadsA;
            v[u] = n < hi ? row[n] : -__int_as_float(0x7f800000);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int n = n0 + u * kThreadsA;
            if (n < hi && argmax_better(v[u], n, bv, bi)) {
                bv = v[u];
                bi = n;
            }
        }
    }
    block_best(bv, bi);
    __shared__ bool last;
    if (threadIdx.x == 0) {
        cand[(size_t)m * kChunks + c] = make_float2(bv, __int_as_float(bi));
        __threadfence();
        last = atomicAdd(tickets + m, 1u) == (unsigned)(kChunks - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    bv = -__int_as_float(0x7f800000);
    bi = 0x7fffffff;
    if (threadIdx.x < kChunks) {
        const float2 k = __ldcg(cand + (size_t)m * kChunks + threadIdx.x);
        bv = k.x;
        bi = __float_as_int(k.y);
    }
    block_best(bv, bi);
    if (threadIdx.x == 0) {
        ids[m] = bi;
        tickets[m] = 0u;  // re-armed for the next call
    }
}

}  // namespace

cudaError_t bitlin_launch_argmax(const float* y, int M, int N, void* cand, unsigned* tickets, int32_t* ids,
                                 cudaStream_t s)
{
    bitlin_argmax_rows<<<dim3(kChunks, M), kThreadsA, 0, s>>>(y, N, static_cast<float2*>(cand), tickets, ids);
    return cudaGetLastError();
}

size_t bitlin_argmax_scratch_bytes(int M) { return (size_t)M * kArgmaxSlots * sizeof(float2); }
