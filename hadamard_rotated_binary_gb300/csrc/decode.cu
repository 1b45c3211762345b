// Decode GEMV (the library's choice for M <= 6; any M when forced): activation
// rotation fused into the prologue, then the one-bit product through
// shared-memory signed-sum tables.
//
// Method (what is computed) - Pulse "ARCHITECTURE-SPEC", Hadamard-fold
// section: xt = WHT1024(signs * P(x)) / 32 per 1024-block, then y = W @ xt;
// "Inside the One-Bit Engine", first station: weight = +-1 from one bit, one
// scale per 128 weights applied to the group sum.
//
// How (GB300 design):
//  * Work unit = (slice s of 512 weights along K) x (tile t of 32 rows).  A CTA
//    (one per SM: 16 warps, or 24 with a 2-deep ring for cluster shapes of at
//    most 48 tiles per CTA) owns one slice and a contiguous range of tiles.
//    Split-K: when the S slices of a tile range fit a thread-block cluster
//    (S <= 16) and their partial sums fit shared memory, the S CTAs form a
//    cluster, keep their partials in shared memory and sum them through
//    distributed shared memory (cluster_finish; a first cluster barrier phase,
//    arrived at on entry and waited on before the first remote store, makes
//    sure every CTA of the cluster has started).  Otherwise the partials land
//    in a scratch array and a second kernel (bitlin_decode_reduce, chained by
//    programmatic dependent launch) sums every output over the slices with
//    one thread each.  Both sum in the fixed order s = 0..S-1 (deterministic).
//  * Tokens: one at a time for M = 1; two at a time otherwise (a separate
//    instance with both tables built and a 2-deep register ring, so that every
//    weight tile loaded serves two tokens).
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
//    register), one LDS and one FADD.  With M = 1 and small split-K partials
//    the table sits at a 64 KB-aligned shared address whose upper bits ride in
//    the per-lane register, so the PRMT yields the complete address and no
//    add is needed before the LDS (one instruction in four fewer).  Every 4
//    words (one 128-group) the group sum is multiplied by its fp16 scale with
//    one FFMA.
//  * Weights stream from HBM into registers with 16-byte coalesced loads
//    through a ring of 4 tiles per warp (with 16 warps that is every tile of
//    a CTA at the ffn_gate shape): the first 4 tiles are requested before the
//    wait for the previous kernel, so their latency overlaps that wait, the
//    transform and the table build; each consumed tile is replaced by the
//    warp's next one.
//  * Programmatic dependent launch: the kernel lets its successor launch after
//    its table build and itself waits (griddepcontrol.wait) only before it
//    reads x or writes any output.  Before the wait it issues what does not
//    depend on the previous kernel: the first ring of tiles, the signs, an L2
//    hint for the lines of x and, on the scratch split-K path, an L2 prefetch
//    of the first part of its weight share.
//  * Every instruction before the lookups is on a call's critical path (the
//    CTAs that start last, on SMs whose previous CTA ended last, set the
//    call's time), so the tile-range split, the partial-sum placement and the
//    cluster finish use no runtime division (the launcher passes the split
//    and ceil(2^32 / S)), and the one-token instance forms the addresses of x
//    before the wait.
#include <cuda_fp16.h>

#include "bitlin_internal.cuh"
#include "ptx.cuh"

namespace {

using namespace bitlin_impl;

constexpr int kPad = 33;                               // transpose row stride (floats)
constexpr int kSmemTranspose = 16 * kPad * 4;           // 2112 B
constexpr int kSmemSlice = (kSlice + kSlice / 32) * 4;  // 528 floats
constexpr int kDecodeSmem = kLutBytes + kSmemTranspose + kSmemSlice;
// With M >= 2 a second 64 KB table follows (tokens are taken two at a time),
// then, for the cluster split-K, the CTA's partial sums [M][tiles][32].
constexpr int kLut2Off = (kDecodeSmem + 127) & ~127;
constexpr int kPbufOff = (kDecodeSmem + 15) & ~15;  // M = 1
constexpr int kPbufOff2 = kLut2Off + kLutBytes;     // M >= 2
constexpr int kMaxClusterSlices = 16;
// Warps of the wide one-token CTA (cluster split-K with at most 48 tiles per
// CTA): two tiles per warp at most, a 2-deep register ring, 80 registers per
// thread (warps are dealt round robin to the SM's four sub-partitions of
// 16,384 registers: 6 x 32 x 80 fit, 6 x 32 x 96 do not launch).  Warps
// 0-15 run the x / transform / table prologue; all of them look up.
constexpr int kWideWarps = 24;
// Aligned-table layout (M = 1): the allocation holds a pad of up to 64 KB,
// the table at the first 64 KB-aligned shared address, and the transpose
// buffer, slice and partial sums (below the table when the pad holds them,
// above it otherwise).
constexpr int kAlRestPbuf = (kSmemTranspose + kSmemSlice + 15) & ~15;  // partial sums' offset in that block
constexpr int kAlSmemBase = 2 * kLutBytes + kAlRestPbuf;              // allocation before the partial sums
// Largest partial-sum buffer for which the aligned layout is used: beyond
// it the allocation leaves too little of the SM's storage to L1 for the
// streaming weight loads (the vocabulary matrix, 76 KB of partials, measured
// 53.4 against 45.2 us per call with the aligned layout).
constexpr int kAlMaxPbuf = 32 * 1024;
constexpr int kRowsPerWarp = 16 / kDecodeWarps;  // rows of the [16][32] transform view per warp
static_assert(kDecodeWarps == 8 || kDecodeWarps == 16, "prologue mapping assumes 8 or 16 warps");

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

// NA: loads that allocate nothing in L1 (each weight byte is read once).
// Measured per call: the one-token LM head 44.5 against 45.3 us with them; the
// two-token instance on the scratch path slower with them (ffn_down at M = 4:
// 18.8 against 18.1 us), so it keeps the plain read-only loads.
template <bool NA>
__device__ __forceinline__ void load_tile(const DecodeParams& p, int s, int t, int lane, uint4 (&b)[4],
                                          uint2& sc)
{
    const size_t unit = (size_t)s * p.T + t;
    const uint4* src = p.bits + unit * 4 * 32 + lane;
    if (NA) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(b[q].x), "=r"(b[q].y), "=r"(b[q].z), "=r"(b[q].w)
                         : "l"(src + q * 32));
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                     : "=r"(sc.x), "=r"(sc.y)
                     : "l"(p.scales + unit * 32 + lane));
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) b[q] = __ldg(src + q * 32);
        sc = __ldg(p.scales + unit * 32 + lane);
    }
}

// Source column of grouped position k under the ssm_out permutation
// (grouped [hd, rep, nk] <- tiled [hd, nk, rep], hd = 128, nk = 16, rep = 3).
__device__ __forceinline__ int perm_source(int k)
{
    const int head = k >> 7, d = k & 127;
    const int r = head % 3, kk = head / 3;
    return d + 128 * (kk + 16 * r);
}

// Rotated activations of token m for slice s, in two parts so that the
// caller can issue other loads between them.  Thread (warp w, lane q) covers
// rows p = w and p = w + 8 of the [16][32] view of the half block.
// The raw x and sign values of this thread (gather through the ssm_out
// permutation when requested); no arithmetic, so nothing waits on them yet.
// The signs belong to the handle and may be read before the wait for the
// previous kernel; x may not.
__device__ __forceinline__ void slice_load_signs(const DecodeParams& p, int s, int warp, int lane,
                                                 float (&v)[4 * kRowsPerWarp])
{
    const int b = s >> 1;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int k0 = b * 1024 + 32 * (warp + kDecodeWarps * r) + lane;  // i = 0..511
        v[4 * r + 1] = __ldg(p.signs + k0);
        v[4 * r + 3] = __ldg(p.signs + k0 + 512);
    }
}

// Input element k of token m (after the permutation).  With swiglu set, x
// holds [M][2K] gate and up values and the input is silu(gate) * up, SiLU(g)
// = g / (1 + e^-g) in f32 ("Inside the One-Bit Engine", MLP station).
__device__ __forceinline__ const float* x_source(const DecodeParams& p, int m, int k)
{
    return p.x + (size_t)m * (p.swiglu ? 2 * p.K : p.K) + (p.perm ? perm_source(k) : k);
}

__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.f + expf(-g)) * u; }

// The addresses slice_load_x reads (they do not depend on the previous
// kernel, so they can be formed before the wait for it).
__device__ __forceinline__ void slice_x_ptrs(const DecodeParams& p, int m, int s, int warp, int lane,
                                             const float* (&a)[2 * kRowsPerWarp])
{
    const int b = s >> 1;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int k0 = b * 1024 + 32 * (warp + kDecodeWarps * r) + lane;
        a[2 * r + 0] = x_source(p, m, k0);
        a[2 * r + 1] = x_source(p, m, k0 + 512);
    }
}

__device__ __forceinline__ void slice_load_x_at(const DecodeParams& p, const float* const (&a)[2 * kRowsPerWarp],
                                                float (&v)[4 * kRowsPerWarp])
{
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        if (p.swiglu) {
            v[4 * r + 0] = swiglu(__ldg(a[2 * r]), __ldg(a[2 * r] + p.K));
            v[4 * r + 2] = swiglu(__ldg(a[2 * r + 1]), __ldg(a[2 * r + 1] + p.K));
        } else {
            v[4 * r + 0] = __ldg(a[2 * r]);
            v[4 * r + 2] = __ldg(a[2 * r + 1]);
        }
    }
}

__device__ __forceinline__ void slice_load_x(const DecodeParams& p, int m, int s, int warp, int lane,
                                             float (&v)[4 * kRowsPerWarp])
{
    const int b = s >> 1;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int k0 = b * 1024 + 32 * (warp + kDecodeWarps * r) + lane;
        const float* a0 = x_source(p, m, k0);
        const float* a1 = x_source(p, m, k0 + 512);
        if (p.swiglu) {
            v[4 * r + 0] = swiglu(__ldg(a0), __ldg(a0 + p.K));
            v[4 * r + 2] = swiglu(__ldg(a1), __ldg(a1 + p.K));
        } else {
            v[4 * r + 0] = __ldg(a0);
            v[4 * r + 2] = __ldg(a1);
        }
    }
}

// A hint only: ask L2 for the lines of x this thread will read.  Issued
// before the wait it has no effect on what is read after it.
__device__ __forceinline__ void slice_prefetch_x(const DecodeParams& p, int m, int s, int warp, int lane)
{
    const int b = s >> 1;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int k0 = b * 1024 + 32 * (warp + kDecodeWarps * r) + lane;
        if (p.perm || lane == 0) {
            asm volatile("prefetch.global.L2 [%0];" ::"l"(x_source(p, m, k0)));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(x_source(p, m, k0 + 512)));
            if (p.swiglu) {
                asm volatile("prefetch.global.L2 [%0];" ::"l"(x_source(p, m, k0) + p.K));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(x_source(p, m, k0 + 512) + p.K));
            }
        }
    }
}

// slice_transform: half h of the block's 1024-point transform is
// H512(xs_lo + (-1)^h xs_hi) / 32 with H512 = H16 (x) H32.  Rows part: the
// 32-point butterflies across the lanes, into tbuf; the caller then
// synchronizes and runs the columns part (16-point butterflies across
// half-warps, x 1/32, into xs, padded, 512 floats).
__device__ __forceinline__ void slice_transform_rows(int s, const float (&v)[4 * kRowsPerWarp], float* tbuf,
                                                     int warp, int lane)
{
    const int h = s & 1;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const float a = v[4 * r + 0] * v[4 * r + 1];
        const float c = v[4 * r + 2] * v[4 * r + 3];
        float z = h ? (a - c) : (a + c);
        // 32-point butterflies across the lanes (natural Sylvester order).
#pragma unroll
        for (int st = 1; st < 32; st <<= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, z, st);
            z = (lane & st) ? (o - z) : (z + o);
        }
        tbuf[(warp + kDecodeWarps * r) * kPad + lane] = z;
    }
}

__device__ __forceinline__ void slice_transform_cols(const float* tbuf, float* xs, int warp, int lane)
{
    // 16-point butterflies down the columns: warp w takes 32 / warps columns,
    // one per half-warp and round; lane & 15 is the row.
    const int row = lane & 15;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int col = 2 * kRowsPerWarp * warp + 2 * r + (lane >> 4);
        float z = tbuf[row * kPad + col];
#pragma unroll
        for (int st = 1; st < 16; st <<= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, z, st);
            z = (row & st) ? (o - z) : (z + o);
        }
        xs[xpad(row * 32 + col)] = z * 0.03125f;  // exact scaling by 1/32
    }
}

// Signed-sum tables for the slice: warp v writes entries b = 16*hn .. 16*hn+15
// (high nibbles hn = v, v + warps, ...) of all 64 tables; lane L writes the
// two tables of bank L (its word w = L & 15, byte parity L >> 4, byte pair jh).
__device__ __forceinline__ void build_tables(const float* xs, unsigned char* lut, int warp, int lane)
{
    const int w = lane & 15, jlo = lane >> 4;
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
#pragma unroll
        for (int hh = 0; hh < kRowsPerWarp; ++hh) {
            const int hnib = warp + kDecodeWarps * hh;
            const float a45 = ((hnib & 1) ? x[4] : -x[4]) + ((hnib & 2) ? x[5] : -x[5]);
            const float a67 = ((hnib & 4) ? x[6] : -x[6]) + ((hnib & 8) ? x[7] : -x[7]);
            const float hi = a45 + a67;
            unsigned char* dst = lut + (size_t)(16 * hnib) * 256 + 128 * jh + 4 * lane;
#pragma unroll
            for (int l = 0; l < 16; ++l)
                *reinterpret_cast<float*>(dst + l * 256) = (p01[l & 3] + p23[l >> 2]) + hi;
        }
    }
}

// Table reads for byte offsets built by PRMT: lo for bytes 0-1 of a word,
// hi (128 bytes further) for bytes 2-3.  LutPlain adds the table's base;
// LutAligned receives complete shared addresses (the base's upper bits are
// in bytes 2-3 of the per-lane offset register, its lower 16 bits are zero).
struct LutPlain {
    const unsigned char* lut;
    __device__ __forceinline__ float lo(uint32_t off) const { return lut_at(lut, off); }
    __device__ __forceinline__ float hi(uint32_t off) const { return lut_at(lut + 128, off); }
};
struct LutAligned {
    __device__ __forceinline__ float lo(uint32_t a) const
    {
        float v;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
        return v;
    }
    __device__ __forceinline__ float hi(uint32_t a) const
    {
        float v;
        asm volatile("ld.shared.f32 %0, [%1+128];" : "=f"(v) : "r"(a));
        return v;
    }
};

// Dot products of two tiles for this lane's two rows, interleaved so that the
// two tiles' lookup chains are independent: per tile, the sum over the
// slice's 4 groups of scale * (sum of 16 table lookups).
template <class Lut>
__device__ __forceinline__ void tile_dot2(const Lut lut, const uint4 (&b0)[4], uint2 sc0, const uint4 (&b1)[4],
                                          uint2 sc1, uint32_t base_off, float& out0, float& out1)
{
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint32_t wa[4] = {b0[u].x, b0[u].y, b0[u].z, b0[u].w};
        const uint32_t wb[4] = {b1[u].x, b1[u].y, b1[u].z, b1[u].w};
        float ga0 = 0.f, ga1 = 0.f, gb0 = 0.f, gb1 = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t pos = 4u * u + c;
            const uint32_t off = base_off ^ ((4u * pos) * 0x101u);
            ga0 += lut.lo(__byte_perm(wa[c], off, 0x7604));
            gb0 += lut.lo(__byte_perm(wb[c], off, 0x7604));
            ga1 += lut.lo(__byte_perm(wa[c], off, 0x7615));
            gb1 += lut.lo(__byte_perm(wb[c], off, 0x7615));
            ga0 += lut.hi(__byte_perm(wa[c], off, 0x7624));
            gb0 += lut.hi(__byte_perm(wb[c], off, 0x7624));
            ga1 += lut.hi(__byte_perm(wa[c], off, 0x7635));
            gb1 += lut.hi(__byte_perm(wb[c], off, 0x7635));
        }
        const uint32_t ha = (u < 2 ? sc0.x : sc0.y) >> (16 * (u & 1));
        const uint32_t hb = (u < 2 ? sc1.x : sc1.y) >> (16 * (u & 1));
        acc0 = fmaf(ga0 + ga1, __half2float(__ushort_as_half((unsigned short)ha)), acc0);
        acc1 = fmaf(gb0 + gb1, __half2float(__ushort_as_half((unsigned short)hb)), acc1);
    }
    out0 = acc0;
    out1 = acc1;
}

// One tile (a warp's last, odd one): four independent lookup chains, half the
// work of tile_dot2, the same arithmetic per tile.
template <class Lut>
__device__ __forceinline__ void tile_dot1(const Lut lut, const uint4 (&b)[4], uint2 sc, uint32_t base_off,
                                          float& out)
{
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint32_t w[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
        float g0 = 0.f, g1 = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t pos = 4u * u + c;
            const uint32_t off = base_off ^ ((4u * pos) * 0x101u);
            g0 += lut.lo(__byte_perm(w[c], off, 0x7604));
            g1 += lut.lo(__byte_perm(w[c], off, 0x7615));
            g0 += lut.hi(__byte_perm(w[c], off, 0x7624));
            g1 += lut.hi(__byte_perm(w[c], off, 0x7635));
        }
        const float sv = __half2float(__ushort_as_half((unsigned short)((u < 2 ? sc.x : sc.y) >> (16 * (u & 1)))));
        acc = fmaf(g0 + g1, sv, acc);
    }
    out = acc;
}

// One tile against two tokens' tables: every byte's shared-memory offset is
// built once and read in both tables (the second at lut2), so each loaded
// weight tile serves two tokens.
__device__ __forceinline__ void tile_dot_two(const unsigned char* lut, const unsigned char* lut2,
                                             const uint4 (&b)[4], uint2 sc, uint32_t base_off, float& out0,
                                             float& out1)
{
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint32_t w[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
        float g0 = 0.f, g1 = 0.f, h0 = 0.f, h1 = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t pos = 4u * u + c;
            const uint32_t off = base_off ^ ((4u * pos) * 0x101u);
            const uint32_t o0 = __byte_perm(w[c], off, 0x7604), o1 = __byte_perm(w[c], off, 0x7615);
            const uint32_t o2 = __byte_perm(w[c], off, 0x7624), o3 = __byte_perm(w[c], off, 0x7635);
            g0 += lut_at(lut, o0);
            h0 += lut_at(lut2, o0);
            g1 += lut_at(lut, o1);
            h1 += lut_at(lut2, o1);
            g0 += lut_at(lut + 128, o2);
            h0 += lut_at(lut2 + 128, o2);
            g1 += lut_at(lut + 128, o3);
            h1 += lut_at(lut2 + 128, o3);
        }
        const float sv = __half2float(__ushort_as_half((unsigned short)((u < 2 ? sc.x : sc.y) >> (16 * (u & 1)))));
        acc0 = fmaf(g0 + g1, sv, acc0);
        acc1 = fmaf(h0 + h1, sv, acc1);
    }
    out0 = acc0;
    out1 = acc1;
}

// Ask L2 to fetch [p, p + bytes) from HBM (no completion tracking), in 16 KB
// pieces spread over the CTA's threads so that no warp spends long issuing.
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes, int tid)
{
    const char* c = static_cast<const char*>(p);
    constexpr size_t kPiece = 16384;
    for (size_t o = (size_t)tid * kPiece; o < bytes; o += (size_t)kDecodeThreads * kPiece) {
        const size_t n = bytes - o < kPiece ? bytes - o : kPiece;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + o), "r"((unsigned)n) : "memory");
    }
}

// Units (slice x 32-row tile, 2 KB of bits) a CTA prefetches into L2 before
// the wait: 64 units = 128 KB, 19.5 MB over 152 CTAs.
constexpr int kPrefetchUnits = 64;

// Tiles in flight per warp: the register ring of prefetched tiles (even).
#ifndef BITLIN_DECODE_RING
#define BITLIN_DECODE_RING 4
#endif
constexpr int kRing = BITLIN_DECODE_RING;

// Registers per thread: 16 warps x 128 = the SM's 65,536 (one CTA per SM).
#ifndef BITLIN_DECODE_REGS
#define BITLIN_DECODE_REGS 128
#endif
constexpr int kDecodeRegs = BITLIN_DECODE_REGS;

// Split-K across a cluster.  The cluster's tiles [ta, tb) are dealt round
// robin to its S CTAs: local tile lt belongs to CTA lt % S, slot lt / S.  Every
// CTA stores each partial sum of its slice straight into the owner's shared
// memory as it computes it (pbuf [M][S][LT][32], LT = ceil((tb - ta) / S)).
// After one cluster barrier, which makes those stores visible, each CTA sums
// its own tiles over the S slices in slice order s = 0..S-1 (the same order
// and arithmetic as the global-scratch path) from its own shared memory, and
// writes y.  Nothing reads another CTA's shared memory after the barrier, so
// no second barrier is needed before the CTAs exit.
// v / S as umulhi(v, ceil(2^32 / S)): exact for S in [2, 16] and v < 2^17 (the
// partial sums of a cluster fit 96 KB, so its tile count is below 768).
__device__ __forceinline__ int div_s(const DecodeParams& p, int v) { return (int)__umulhi((unsigned)v, p.s_mul); }
__device__ __forceinline__ int cluster_slots(const DecodeParams& p, int ntile) { return div_s(p, ntile + p.S - 1); }

// Best (value, index) over the CTA's threads in the argmax order; the result
// is valid in thread 0.  red: shared scratch of 64 words, free on entry.
__device__ __forceinline__ void cta_best(float& bv, int& bi, float* red, int threads)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = threads >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (argmax_better(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
        }
    }
    if (lane == 0) {
        red[warp] = bv;
        red[32 + warp] = __int_as_float(bi);
    }
    __syncthreads();
    if (warp == 0) {
        bv = lane < nw ? red[lane] : -__int_as_float(0x7f800000);
        bi = lane < nw ? __float_as_int(red[32 + lane]) : 0x7fffffff;
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
    __syncthreads();  // red may be written again
}

// Greedy argmax of token m, fused into the finish ("Inside the One-Bit
// Engine", LM-head station: the token with the largest score is picked).
// (bv, bi) is this thread's best over the outputs it wrote.  The CTA's best
// becomes candidate blockIdx.x of token m; the CTA that takes the token's last
// ticket picks among all candidates (the order is total, so the result does
// not depend on which CTA that is) and re-arms the ticket.  Not inlined: it
// runs once per call, and inlined it cost the lookup loop registers.
__device__ __noinline__ void finish_argmax(int32_t* ids, float2* cand, unsigned* tickets, int m, float bv, int bi,
                                           float* red, int threads)
{
    cta_best(bv, bi, red, threads);
    int* last = reinterpret_cast<int*>(red + 64);
    if (threadIdx.x == 0) {
        cand[(size_t)m * kArgmaxSlots + blockIdx.x] = make_float2(bv, __int_as_float(bi));
        __threadfence();
        *last = atomicAdd(tickets + m, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!*last) return;
    __threadfence();  // every candidate is visible
    bv = -__int_as_float(0x7f800000);
    bi = 0x7fffffff;
    for (int j = (int)threadIdx.x; j < (int)gridDim.x; j += threads) {
        const float2 c = __ldcg(cand + (size_t)m * kArgmaxSlots + j);
        if (argmax_better(c.x, __float_as_int(c.y), bv, bi)) {
            bv = c.x;
            bi = __float_as_int(c.y);
        }
    }
    cta_best(bv, bi, red, threads);
    if (threadIdx.x == 0) {
        ids[m] = bi;
        tickets[m] = 0u;  // re-armed for the next call
    }
}

// AM: the greedy argmax is fused into the finish (finish_argmax), with the
// transpose buffer of the plain-table layout (free once the tables are built)
// as its shared scratch; it is addressed here, not kept live from the
// prologue, so the lookup loop keeps its registers.
template <bool AM>
__device__ __forceinline__ void cluster_finish(const DecodeParams& p, int ta, int tb, int rank, const float* pbuf,
                                               int threads)
{
    ptx::cluster_sync();
    const int ntile = tb - ta, S = p.S, LT = cluster_slots(p, ntile);
    const int mine = ntile > rank ? div_s(p, ntile - rank + S - 1) : 0;  // tiles rank, rank + S, ...
    const int stride = LT * kTileRows;
    for (int m = 0; m < p.M; ++m) {
        float bv = -__int_as_float(0x7f800000);  // AM: this thread's best output
        int bi = 0x7fffffff;
        for (int i = (int)threadIdx.x; i < mine * kTileRows; i += threads) {
            const int slot = i >> 5, lane = i & 31;
            const float* src = pbuf + (m * S * LT + slot) * kTileRows + lane;
            // All S loads in flight at once, then the sum in slice order.
            float v[kMaxClusterSlices];
#pragma unroll
            for (int s = 0; s < kMaxClusterSlices; ++s) {
                v[s] = 0.f;
                if (s < S) v[s] = src[s * stride];
            }
            float sum = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxClusterSlices; ++s)
                if (s < S) sum += v[s];
            const int n = (ta + slot * S + rank) * kTileRows + lane;
            if (n < p.N) {
                p.y[(size_t)m * p.N + n] = sum;
                if (AM && argmax_better(sum, n, bv, bi)) {
                    bv = sum;
                    bi = n;
                }
            }
        }
        if (AM) {
            extern __shared__ __align__(128) unsigned char smem[];
            finish_argmax(p.ids, p.amax_cand, p.amax_tickets, m, bv, bi,
                          reinterpret_cast<float*>(smem + kLutBytes), threads);
        }
    }
}

// TWO: tokens are taken two at a time (M >= 2), with a 2-deep register ring so
// that both tokens' accumulators fit the register budget; M = 1 keeps the
// 4-deep ring.  AL (M = 1 only): the table at a 64 KB-aligned shared address.
// AM (cluster split-K only): the greedy argmax fused into the finish.
template <bool TWO, bool AL, int NW, bool AM = false>
__global__ void __maxnreg__(NW == kDecodeWarps ? kDecodeRegs : 80) bitlin_decode_gemv(const DecodeParams p)
{
    static_assert(!(AM && AL), "the fused argmax uses the plain-table layout");
    static_assert(NW == kDecodeWarps || (!TWO && AL), "more warps only for one token with the aligned table");
    static_assert(!(TWO && AL), "the aligned table is for one token at a time");
    constexpr int RING = TWO || NW != kDecodeWarps ? 2 : kRing;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* lut = smem;
    float* tbuf = reinterpret_cast<float*>(smem + kLutBytes);
    unsigned char* lut2 = smem + kLut2Off;  // second token's table (M >= 2)
    float* pbuf = reinterpret_cast<float*>(smem + (p.M >= 2 ? kPbufOff2 : kPbufOff));  // cluster split-K only
    uint32_t lut_hi = 0;  // AL: the table's shared address (a multiple of 64 KB)
    if (AL) {
        const uint32_t sb = ptx::smem_u32(smem);
        lut_hi = (sb + 0xFFFFu) & ~0xFFFFu;
        lut = smem + (lut_hi - sb);
        unsigned char* rest = lut_hi - sb >= (uint32_t)(kAlRestPbuf + p.pbuf_bytes) ? smem : lut + kLutBytes;
        tbuf = reinterpret_cast<float*>(rest);
        pbuf = reinterpret_cast<float*>(rest + kAlRestPbuf);
    }
    float* xs = tbuf + 16 * kPad;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool pro = NW == kDecodeWarps || warp < kDecodeWarps;  // the warps of the x / transform / table prologue
    // Cluster split-K writes into the other CTAs' shared memory: every thread
    // signals that its CTA has started, and waits for the whole cluster's
    // signal before the first of those writes (long since complete by then).
    if (p.cluster) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // Units owned by this CTA, [u0, u1) in slice-major order.  With
    // ctas_per_slice > 0 every CTA stays inside one slice (one table build);
    // otherwise (more slices than CTAs) the units are split evenly.
    int u0, u1;
    int s0;        // the slice of the CTA's first segment
    int rank = 0;  // cluster mode: this CTA's slice = its rank in the cluster
    // The T tiles of a slice are split over ctas_per_slice = ncl ranges, the
    // first split_r of them one tile longer: range c starts at
    // c * split_q + min(c, split_r).  No division in the cluster case.
    if (p.cluster) {
        // Cluster c (S consecutive blocks, one per slice) covers range c of every slice.
        const int c = (int)__umulhi(blockIdx.x, p.s_mul);  // blockIdx.x / S
        rank = (int)blockIdx.x - c * p.S;
        s0 = rank;
        u0 = rank * p.T + c * p.split_q + min(c, p.split_r);
        u1 = u0 + p.split_q + (c < p.split_r ? 1 : 0);
    } else if (p.ctas_per_slice > 0) {
        const int s = (int)blockIdx.x / p.ctas_per_slice, c = (int)blockIdx.x - s * p.ctas_per_slice;
        s0 = s;
        u0 = s * p.T + c * p.split_q + min(c, p.split_r);
        u1 = u0 + p.split_q + (c < p.split_r ? 1 : 0);
    } else {
        const long long U = (long long)p.S * p.T;
        u0 = (int)(U * blockIdx.x / gridDim.x);
        u1 = (int)(U * (blockIdx.x + 1) / gridDim.x);
        s0 = u0 / p.T;
    }
    const size_t npad = (size_t)p.T * kTileRows;
    // Per-lane part of every table offset: byte 0 for even bytes, byte 1 for odd.
    const uint32_t base_off = (uint32_t)(4 * (lane & 15) + 64 * (lane >> 4)) |
                              ((uint32_t)(4 * (lane & 15) + 64 * (1 - (lane >> 4))) << 8) | lut_hi;

    // The weights do not depend on the previous kernel.  On the scratch
    // split-K path, start streaming the first kPrefetchUnits units of this
    // CTA's share (one contiguous range of bits and one of scales) from HBM
    // into L2 before waiting for it (a prefetch of everything would evict
    // itself on matrices larger than L2).  The cluster path issues only its
    // register ring: there the extra requests measured slower (ffn_gate 6.39
    // against 6.74 us per call without them, the LM head 45.9 against 46.5).
    if (!p.cluster) {
        const int pu = min(u1 - u0, kPrefetchUnits);
        prefetch_l2(p.bits + (size_t)u0 * 128, (size_t)pu * 2048, threadIdx.x);
        prefetch_l2(p.scales + (size_t)u0 * 32, (size_t)pu * 256, (threadIdx.x + 128) % kDecodeThreads);
    }
    // Before the wait: this warp's first tiles (ta + warp + NW * j, j < RING) and
    // the signs of the first segment, whose latency then overlaps the wait, and
    // the L2 hint for x.
    uint4 rb[RING][4];
    uint2 rs[RING];
    float xv[4 * kRowsPerWarp];
    // One token: the first segment's x addressed before the wait (ffn_gate 5.69
    // -> 5.63 us; the two-token instance measured slower with it).
    const float* xptr[2 * kRowsPerWarp];
    {
        const int s = s0, ta = u0 - s * p.T, tb = min(p.T, ta + (u1 - u0));
#pragma unroll
        for (int d = 0; d < RING; ++d) {
            const int t = ta + warp + NW * d;
            if (u0 < u1 && t < tb) load_tile<!TWO>(p, s, t, lane, rb[d], rs[d]);
        }
        if (pro && u0 < u1) {
            slice_load_signs(p, s, warp, lane, xv);
            slice_prefetch_x(p, 0, s, warp, lane);
            if (!TWO) slice_x_ptrs(p, 0, s, warp, lane, xptr);
        }
    }
    pdl_wait();
    bool triggered = false;
    bool preloaded = true;  // the ring and the signs hold the first (segment, token)

    for (int u = u0; u < u1;) {
        const int s = u == u0 ? s0 : u / p.T;  // no division before the first segment's loads
        const int ta = u - s * p.T;
        const int tb = min(p.T, ta + (u1 - u));
        u += tb - ta;

        // Tokens two at a time: both tables are built, then every weight tile
        // loaded serves both tokens' lookups.
        for (int m = 0; m < p.M; m += TWO ? 2 : 1) {
            const bool two = TWO && m + 1 < p.M;
            const bool first = preloaded;
            if (!preloaded) __syncthreads();  // the previous tables and buffers are no longer read
            if (!preloaded) {
                if (pro) slice_load_signs(p, s, warp, lane, xv);
#pragma unroll
                for (int d = 0; d < RING; ++d) {
                    const int t = ta + warp + NW * d;
                    if (t < tb) load_tile<!TWO>(p, s, t, lane, rb[d], rs[d]);
                }
            }
            preloaded = false;
            float xv2[4 * kRowsPerWarp];
#pragma unroll
            for (int i = 0; i < 4 * kRowsPerWarp; ++i) xv2[i] = xv[i];  // the signs
            if (pro) {
                if (!TWO && first) slice_load_x_at(p, xptr, xv);
                else slice_load_x(p, m, s, warp, lane, xv);
                if (two) slice_load_x(p, m + 1, s, warp, lane, xv2);
                slice_transform_rows(s, xv, tbuf, warp, lane);
            }
            __syncthreads();
            if (pro) slice_transform_cols(tbuf, xs, warp, lane);
            __syncthreads();
            if (pro) build_tables(xs, lut, warp, lane);
            if (two) {
                __syncthreads();  // tbuf and xs are free again
                slice_transform_rows(s, xv2, tbuf, warp, lane);
                __syncthreads();
                slice_transform_cols(tbuf, xs, warp, lane);
                __syncthreads();
                build_tables(xs, lut2, warp, lane);
            }
            __syncthreads();
            // The next kernel may launch now: its weight prefetch then overlaps
            // this kernel's lookups rather than its latency-bound prologue.
            if (!triggered) {
                pdl_launch_dependents();
                triggered = true;
                if (p.cluster) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
            }
            // Partial sums.  Scratch path: token mm, tile t, lane ->
            // partials[s][mm][t * 32 + lane].  Cluster path: into the owner's shared
            // memory (see cluster_finish).
            const int LT = p.cluster ? cluster_slots(p, tb - ta) : 0;
            const uint32_t pbase = static_cast<uint32_t>(__cvta_generic_to_shared(pbuf));
            auto put = [&](int mm, int t, float v) {
                if (p.cluster) {
                    const int lt = t - ta;
                    // lt / S as umulhi(lt, ceil(2^32 / S)): exact for S in [2, 16], lt < 2^17
                    // (the partials of a cluster fit 96 KB, so lt < 768).
                    const int q = (int)__umulhi((unsigned)lt, p.s_mul), r = lt - q * p.S;
                    const uint32_t off = (uint32_t)((((mm * p.S) + rank) * LT + q) * kTileRows + lane);
                    ptx::st_cluster(ptx::cluster_map(pbase + 4u * off, r), v);
                } else {
                    p.partials[((size_t)s * p.M + mm) * npad + (size_t)t * kTileRows + lane] = v;
                }
            };
            for (int j0 = 0;; j0 += RING) {
                bool more = true;
#pragma unroll
                for (int d = 0; d < RING; d += 2) {
                    const int t0 = ta + warp + NW * (j0 + d);
                    const int t1 = t0 + NW;
                    if (t0 >= tb) {
                        more = false;
                        break;
                    }
                    float v0, v1 = 0.f, w0 = 0.f, w1 = 0.f;
                    if (two) {
                        tile_dot_two(lut, lut2, rb[d], rs[d], base_off, v0, w0);
                        if (t1 < tb) tile_dot_two(lut, lut2, rb[d + 1], rs[d + 1], base_off, v1, w1);
                    } else if (AL) {
                        if (t1 < tb) tile_dot2(LutAligned{}, rb[d], rs[d], rb[d + 1], rs[d + 1], base_off, v0, v1);
                        else tile_dot1(LutAligned{}, rb[d], rs[d], base_off, v0);
                    } else if (t1 < tb) {
                        tile_dot2(LutPlain{lut}, rb[d], rs[d], rb[d + 1], rs[d + 1], base_off, v0, v1);
                    } else {
                        tile_dot1(LutPlain{lut}, rb[d], rs[d], base_off, v0);
                    }
                    const int tn0 = t0 + NW * RING, tn1 = t1 + NW * RING;
                    if (tn0 < tb) load_tile<!TWO>(p, s, tn0, lane, rb[d], rs[d]);
                    if (tn1 < tb) load_tile<!TWO>(p, s, tn1, lane, rb[d + 1], rs[d + 1]);
                    put(m, t0, v0);
                    if (t1 < tb) put(m, t1, v1);
                    if (two) {
                        put(m + 1, t0, w0);
                        if (t1 < tb) put(m + 1, t1, w1);
                    }
                }
                if (!more) break;
            }
        }
        if (!AM && p.cluster) cluster_finish<false>(p, ta, tb, rank, pbuf, 32 * NW);
    }
    // The fused-argmax instance finishes after the loop, from the CTA's unit
    // range (one segment on the cluster path): with the finish inside the
    // loop it needed more than 128 registers.
    if (AM && p.cluster) {
        const int ta = u0 - s0 * p.T;
        cluster_finish<true>(p, ta, ta + (u1 - u0), rank, pbuf, 32 * NW);
    }
    if (!triggered) pdl_launch_dependents();
}

// Split-K outside a cluster: the sum of the GEMV's partials [S][M][T*32].
// Thread i owns output (m, n) = (i / N, i % N) and adds its S partials in
// slice order s = 0..S-1 (the order of the cluster path), with up to B loads
// in flight: B = 48 when S > 16 (one round at K = 17408: ffn_down 8.0 -> 7.2 us
// per call against rounds of 16), else 16 (48 registers; the wide variant's 96
// halve the occupancy, and the vocabulary matrix at M = 4, almost a million
// outputs, measured 134 against 118 us per call with it).
// The grid stays small on purpose (one output per thread): the next call's
// GEMV, launched early, needs whole SMs, and it finds them on the SMs this
// grid leaves free (160 CTAs of 32 outputs measured 10.8 against 8.0 us per
// ffn_down call).
constexpr int kReduceThreads = 128;
template <int B>
__global__ void __launch_bounds__(kReduceThreads)
    bitlin_decode_reduce(const float* __restrict__ partials, float* __restrict__ y, int M, int N, int S,
                         long long npad)
{
    constexpr int kReduceBatch = B;
    // The successor may launch at once: it reads nothing this kernel writes
    // before its own wait, which covers this whole grid.
    pdl_launch_dependents();
    pdl_wait();  // the GEMV's partials are complete and visible
    const long long i = (long long)blockIdx.x * kReduceThreads + threadIdx.x;
    if (i >= (long long)M * N) return;
    const int m = (int)(i / N), n = (int)(i - (long long)m * N);
    const float* src = partials + (size_t)m * npad + n;
    const size_t step = (size_t)M * npad;
    float sum = 0.f;
    for (int s0 = 0; s0 < S; s0 += kReduceBatch) {
        const int cnt = min(kReduceBatch, S - s0);
        float v[kReduceBatch];
#pragma unroll
        for (int j = 0; j < kReduceBatch; ++j) v[j] = j < cnt ? __ldcg(src + (size_t)(s0 + j) * step) : 0.f;
#pragma unroll
        for (int j = 0; j < kReduceBatch; ++j)
            if (j < cnt) sum += v[j];
    }
    y[(size_t)m * N + n] = sum;
}

}  // namespace

namespace {

// Cluster launches reserve up to this much shared memory for the partial
// sums (the vocabulary matrix, 248,320 rows over 13 clusters, needs 76 KB).
constexpr int kPbufBytes = 96 * 1024;

// Per device: the opt-in shared memory per block, and the clusters of S CTAs
// that one call may use, by S: the clusters that can be resident at once
// divided by the CTAs that fit on an SM, so that when two fit, the next call's
// CTAs find room beside this call's and start their weight prefetch early
// (0 = none).  Set up once per device: kernel attributes apply to the device
// that is current when they are set.
struct DecodeDevice {
    int max_smem = 0;
    int max_clusters[kMaxClusterSlices + 1] = {};
};
DecodeDevice g_decode_dev[kMaxDevices];
PerDeviceOnce g_decode_once;

int query_max_clusters(int S, int num_sms)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * (num_sms / S));
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = kPbufOff + kPbufBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0, per_sm = 0;
    if (cudaOccupancyMaxActiveClusters(&n, bitlin_decode_gemv<false, false, kDecodeWarps>, &cfg) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bitlin_decode_gemv<false, false, kDecodeWarps>, kDecodeThreads,
                                                      kPbufOff + kPbufBytes) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    if (per_sm > 1) n /= per_sm;
    return n < 1 ? 0 : n;
}

// The current device's decode set-up (kernel attributes, opt-in shared memory,
// cluster capacities), done once per device.
cudaError_t configure_decode(const DecodeDevice** out)
{
    int dev = 0;
    cudaError_t e = g_decode_once.run(&dev, [](int d) {
        DecodeDevice& c = g_decode_dev[d];
        int sms = 0;
        cudaError_t r = cudaDeviceGetAttribute(&c.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
        if (r == cudaSuccess && c.max_smem < kPbufOff2) r = cudaErrorInvalidConfiguration;
        for (auto k : {bitlin_decode_gemv<false, false, kDecodeWarps>, bitlin_decode_gemv<false, true, kDecodeWarps>,
                       bitlin_decode_gemv<false, true, kWideWarps>, bitlin_decode_gemv<true, false, kDecodeWarps>,
                       bitlin_decode_gemv<false, false, kDecodeWarps, true>,
                       bitlin_decode_gemv<true, false, kDecodeWarps, true>}) {
            if (r == cudaSuccess) r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, c.max_smem);
            if (r == cudaSuccess) r = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        }
        for (int S = 2; r == cudaSuccess && S <= kMaxClusterSlices; ++S) c.max_clusters[S] = query_max_clusters(S, sms);
        return r;
    });
    *out = e == cudaSuccess ? &g_decode_dev[dev] : nullptr;
    return e;
}

// Launch shape of one call: the grid, its shared memory, the cluster size (0 =
// split-K through the scratch and bitlin_decode_reduce), whether the table is
// 64 KB-aligned, and q's launcher fields.
struct DecodeShape {
    int grid, smem, cluster, aligned, wide;
};

DecodeShape decode_shape(const DecodeParams& p, int num_sms, const DecodeDevice& dc, DecodeParams& q)
{
    q = p;
    DecodeShape d{0, p.M >= 2 ? kPbufOff2 : kDecodeSmem, 0, 0, 0};  // two tables from M = 2
    int pbytes = 0;  // cluster split-K partial sums per CTA
    q.cluster = 0;
    q.s_mul = 0xFFFFFFFFu / (unsigned)p.S + 1u;  // ceil(2^32 / S); S = K / 512 >= 2
    // Split-K across a cluster when the slices fit one (S <= 16) and the
    // partial sums fit shared memory; else through the global scratch.
    if (p.allow_cluster && p.S <= kMaxClusterSlices) {
        const int maxc = dc.max_clusters[p.S];
        if (maxc > 0) {
            const int ncl = maxc < p.T ? maxc : p.T;
            const int lt = ((p.T + ncl - 1) / ncl + p.S - 1) / p.S;  // slots per CTA
            const long long pb = (long long)p.M * p.S * lt * kTileRows * 4;
            const int poff = p.M >= 2 ? kPbufOff2 : kPbufOff;
            if (pb <= kPbufBytes && poff + pb <= dc.max_smem) {
                q.cluster = 1;
                q.ctas_per_slice = ncl;
                d.grid = p.S * ncl;
                d.smem = poff + (int)pb;
                d.cluster = p.S;
                pbytes = (int)pb;
            }
        }
    }
    if (!q.cluster) {
        if (p.S <= num_sms) {
            q.ctas_per_slice = num_sms / p.S < p.T ? num_sms / p.S : p.T;
            d.grid = p.S * q.ctas_per_slice;
        } else {
            const long long U = (long long)p.S * p.T;
            q.ctas_per_slice = 0;
            d.grid = (int)(U < num_sms ? U : num_sms);
        }
    }
    if (q.ctas_per_slice > 0) {
        q.split_q = p.T / q.ctas_per_slice;
        q.split_r = p.T - q.split_q * q.ctas_per_slice;
    }
    // The argmax is fused into the cluster finish when every CTA has a
    // candidate slot (the plain-table instances carry it); otherwise the
    // caller runs the separate argmax kernel.
    if (!q.cluster || d.grid > kArgmaxSlots) {
        q.ids = nullptr;
        q.amax_cand = nullptr;
        q.amax_tickets = nullptr;
    }
    // One token: the aligned table when the partial sums are small (the
    // allocation covers the worst-case pad below the table).
    q.pbuf_bytes = pbytes;
    if (p.M == 1 && !q.ids && pbytes <= kAlMaxPbuf && kAlSmemBase + pbytes <= dc.max_smem) {
        d.aligned = 1;
        d.smem = kAlSmemBase + pbytes;
        // Cluster split-K with at most two tiles per warp of the wide CTA (every
        // tile in its ring): ffn_gate 5.64 -> 5.57 us.  The scratch path measured
        // slower with it (ffn_down 7.99 against 8.22 us), so it keeps 16 warps.
        if (q.cluster && q.split_q + (q.split_r > 0 ? 1 : 0) <= 2 * kWideWarps) d.wide = 1;
    }
    return d;
}

}  // namespace

cudaError_t bitlin_decode_kernels(const DecodeParams& p, int num_sms, int* kernels, int* fused_argmax)
{
    const DecodeDevice* dc = nullptr;
    cudaError_t e = configure_decode(&dc);
    if (e != cudaSuccess) return e;
    DecodeParams q;
    *kernels = decode_shape(p, num_sms, *dc, q).cluster ? 1 : 2;
    if (fused_argmax) *fused_argmax = q.ids != nullptr;
    return cudaSuccess;
}

cudaError_t bitlin_launch_decode(const DecodeParams& p, int num_sms, cudaStream_t s)
{
    const DecodeDevice* dc = nullptr;
    cudaError_t e = configure_decode(&dc);
    if (e != cudaSuccess) return e;
    DecodeParams q;
    const DecodeShape d = decode_shape(p, num_sms, *dc, q);
    const int grid = d.grid, smem = d.smem, cluster = d.cluster;

    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(d.wide ? 32 * kWideWarps : kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = cluster ? 2 : 1;
    e = q.ids      ? (p.M >= 2 ? cudaLaunchKernelEx(&cfg, bitlin_decode_gemv<true, false, kDecodeWarps, true>, q)
                                : cudaLaunchKernelEx(&cfg, bitlin_decode_gemv<false, false, kDecodeWarps, true>, q))
        : p.M >= 2 ? cudaLaunchKernelEx(&cfg, bitlin_decode_gemv<true, false, kDecodeWarps>, q)
        : d.wide    ? cudaLaunchKernelEx(&cfg, bitlin_decode_gemv<false, true, kWideWarps>, q)
        : d.aligned ? cudaLaunchKernelEx(&cfg, bitlin_decode_gemv<false, true, kDecodeWarps>, q)
                    : cudaLaunchKernelEx(&cfg, bitlin_decode_gemv<false, false, kDecodeWarps>, q);
    if (e != cudaSuccess || q.cluster) return e;
    // Scratch split-K: the sum over the slices, launched as the GEMV's dependent.
    const long long outs = (long long)p.M * p.N;
    cudaLaunchConfig_t rc = {};
    rc.gridDim = dim3((unsigned)((outs + kReduceThreads - 1) / kReduceThreads));
    rc.blockDim = dim3(kReduceThreads);
    rc.stream = s;
    rc.attrs = attr;
    rc.numAttrs = 1;
    return cudaLaunchKernelEx(&rc, p.S > 16 ? bitlin_decode_reduce<48> : bitlin_decode_reduce<16>,
                              static_cast<const float*>(p.partials), p.y, p.M, p.N, p.S, (long long)p.T * kTileRows);
}
