/*
 * bitlin - Hadamard-folded 1-bit weight matrix-vector (and matrix-matrix)
 * product for NVIDIA GB300 (sm_103a).
 *
 * What it computes, for every token row m of x[M][K]:
 *
 *   1. if the handle was created with BITLIN_PERM_SSM_TILED_TO_GROUPED, the
 *      ssm_out head permutation tiled [hd=128, nk=16, rep=3] -> grouped
 *      [hd, rep, nk]: xp[d + 128*(r + 3*k)] = x[d + 128*(k + 16*r)];
 *   2. xs = xp * signs (elementwise, signs[i] in {+1, -1});
 *   3. xt = blockwise normalized Walsh-Hadamard transform of xs in blocks of
 *      1024 (natural Sylvester order, H[i][j] = (-1)^popcount(i & j)),
 *      scaled by 1/32;
 *   4. y[m][n] = sum over groups g of 128 along K of
 *          scale[n][g] * sum_{k in g} (bit(n, k) ? +1 : -1) * xt[k],
 *      where bit(n, k) = (packed_bits[n][k >> 5] >> (k & 31)) & 1.
 *
 * Sources: steps 1-3 and their order are the activation side of the Hadamard
 * fold in the Pulse engine's "ARCHITECTURE-SPEC" page (section on the
 * Hadamard fold: optional tiled->grouped permutation, x = x * signs,
 * normalized Sylvester-Walsh transform, block 1024, scale 1/32, then
 * y = W @ x; and its ssm_out permutation paragraph).  Step 4 is the one-bit
 * Q1G128 format of the "Inside the One-Bit Engine" page (first station: one
 * bit per weight, 1 -> +1, 0 -> -1, one shared scale per 128 weights, group
 * sum then one multiply by the scale; station on the embedding row: bit k is
 * bit k&31 of word k>>5, scale index k>>7, IEEE binary16 scales).
 *
 * Paths: 1 <= M <= 6 runs the decode GEMV (f32 throughout; expected max
 * relative L2 error per token row <= 1e-5 against an exact evaluation).
 * 7 <= M < 64 runs the tensor-core path with xt split exactly into three bf16
 * digits, so the +-1 x digit products and f32 accumulation give f32-level
 * results (<= 1e-5).
 * M >= 64 runs the tensor-core path with xt rounded to bf16 (<= 1e-2).  In
 * both tensor-core paths the bits become +-1 bf16 operands of tcgen05 MMAs
 * with f32 accumulation, and each group's partial product is multiplied by
 * its scale in f32.
 *
 * Errors: every function returns a bitlin_status and never aborts or prints.
 * Threads: a handle may be used from one host thread / one stream at a time.
 */
#ifndef BITLIN_H
#define BITLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque handle owning a repacked device copy of one folded 1-bit matrix. */
typedef struct bitlin* bitlin_t;

/* A cudaStream_t (the runtime's stream type is this pointer type). */
typedef struct CUstream_st* bitlin_stream_t;

typedef enum {
    BITLIN_OK = 0,
    BITLIN_EINVAL = 1,   /* a NULL pointer, a size or flag out of range, a sign that is not +-1 */
    BITLIN_ENOMEM = 2,   /* a device or host allocation failed */
    BITLIN_ECUDA = 3,    /* a CUDA runtime call or kernel launch failed (see bitlin_cuda_error) */
    BITLIN_ETIMEOUT = 4, /* a bounded wait inside a kernel gave up; the output is not valid */
    BITLIN_EDEVICE = 5,  /* the current device is not an sm_103 GPU */
    BITLIN_ESCRATCH = 6, /* bitlin_forward_noalloc: the call needs more than its fixed scratch */
    BITLIN_EINDEX = 7    /* bitlin_embed: a token id outside [0, N) (reported by bitlin_get_error) */
} bitlin_status;

#define BITLIN_PERM_NONE 0
/* ssm_out: tiled [hd=128, nk=16, rep=3] -> grouped [hd, rep, nk]; requires K == 6144.
 * (Pulse "ARCHITECTURE-SPEC", ssm_out permutation paragraph.) */
#define BITLIN_PERM_SSM_TILED_TO_GROUPED 1

#define BITLIN_PATH_AUTO 0     /* M <= 6 -> decode GEMV, 7 <= M < 64 -> exact tensor path, M >= 64 -> prefill */
#define BITLIN_PATH_DECODE 1   /* force the f32 decode GEMV (shared-memory tables) for every M */
#define BITLIN_PATH_PREFILL 2  /* force the tcgen05 path with bf16 activations for every M */
#define BITLIN_PATH_TC_EXACT 3 /* force the tcgen05 path with activations split into three bf16
                                  digits (f32-level results) for every M */

/*
 * Create a handle for one N x K folded 1-bit matrix on the current device.
 *
 *   packed_bits  device pointer, uint32 [N][K/32], row-major; bit k of row n is
 *                bit (k & 31) of word k >> 5 (LSB first); 1 means +1, 0 means -1.
 *   scales       device pointer, IEEE binary16 bit patterns [N][K/128], row-major.
 *   signs        device pointer, float [K]; every entry exactly +1.0f or -1.0f.
 *   perm_flag    BITLIN_PERM_NONE or BITLIN_PERM_SSM_TILED_TO_GROUPED.
 *
 * Requirements: N >= 1, K a positive multiple of 1024, all three pointers
 * 16-byte aligned device memory.  The call copies and repacks its inputs into
 * memory the handle owns and synchronizes before returning, so the caller may
 * free or reuse the three arrays afterwards.
 * Errors: BITLIN_EINVAL (NULL out/pointers, N < 1, K % 1024 != 0, unknown
 * perm_flag, perm with K != 6144, a sign other than +-1), BITLIN_ENOMEM,
 * BITLIN_ECUDA, BITLIN_EDEVICE.  On error *out is set to NULL.
 */
bitlin_status bitlin_create(bitlin_t* out, int N, int K, const uint32_t* packed_bits,
                            const uint16_t* scales, const float* signs, int perm_flag);

/*
 * bitlin_create from one Q1G128 tensor in its stored form: a single array of
 * 32-bit words holding first every fp16 scale, two per word, then every sign
 * bit.  Layout ("Inside the One-Bit Engine", embedding-lookup station, and
 * its weight-format station):
 *     scale of row n, group g (sidx = n*(K/128) + g): half (sidx & 1) of word
 *         sidx >> 1, the even index in the low 16 bits;
 *     scale_words = N*K/256 (every row has K/128 scales, a multiple of 8);
 *     bit k of row n: bit (k & 31) of word scale_words + n*(K/32) + (k >> 5),
 *         1 means +1, 0 means -1.
 * The whole array is N*K*9/256 words: 720 bytes per row at K = 5120 (the
 * 248,320 x 5120 vocabulary matrix: 178,790,400 bytes).
 *
 *   qdata  device pointer to that array, 16-byte aligned (the bits then are
 *          too: scale_words*4 is a multiple of 16).
 * Everything else, including ownership (the array may be freed after the
 * call) and the errors, is as bitlin_create.
 */
bitlin_status bitlin_create_q1g128(bitlin_t* out, int N, int K, const uint32_t* qdata, const float* signs,
                                   int perm_flag);

/*
 * y[M][N] = the folded product of x[M][K] (see the top of this file).
 *
 *   x       device pointer, float [M][K], row-major, read only.
 *   y       device pointer, float [M][N], row-major, fully overwritten; must not overlap x.
 *   stream  CUDA stream the work is queued on (NULL = legacy default stream).
 *
 * Asynchronous: no host synchronization.  The first call with a new largest M
 * (and the first call of the tensor-core path) allocates scratch memory the
 * handle keeps; later calls with M at most that size allocate nothing, so they
 * may be captured in a CUDA graph.  Decode launches use programmatic
 * dependent launch: the kernel starts fetching weights while the previous
 * kernel on the stream finishes, and reads x only after it has completed.
 * Errors: BITLIN_EINVAL (NULL handle/x/y, M < 1), BITLIN_ENOMEM, BITLIN_ECUDA,
 * and the sticky BITLIN_ETIMEOUT of an earlier call (see bitlin_get_error).
 */
bitlin_status bitlin_forward(bitlin_t h, const float* x, int M, float* y, bitlin_stream_t stream);

/*
 * The same product with x and y in HOST memory; returns after the result is
 * in y_host (the stream is synchronized).  How the data moves depends on the
 * buffer and the device:
 *   - page-locked memory mapped into the device's address space (for example
 *     from cudaHostAlloc or cudaHostRegister), and any host memory on a device
 *     that reads pageable memory through the host's page tables (a coherent
 *     CPU-GPU link): the kernels read x and write y there directly, with no
 *     copy operation;
 *   - otherwise x is copied into a device buffer the handle keeps (allocated
 *     on the first call with a new largest M), the product runs there, and y
 *     is copied back.
 * x_host must not change and y_host must not be read until the call returns.
 * Errors: as bitlin_forward, plus BITLIN_ETIMEOUT from this call's kernels.
 */
bitlin_status bitlin_forward_host(bitlin_t h, const float* x_host, int M, float* y_host,
                                  bitlin_stream_t stream);

/*
 * bitlin_forward for callers that must not allocate device memory on their
 * call path: code running inside a runtime that owns every device
 * allocation (a memory pool or arena that forbids outside cudaMalloc), and
 * latency-critical loops that must never enter the allocator, since cudaMalloc
 * and cudaFree can synchronize the whole device.  bitlin_forward may grow the
 * handle's scratch on a call with a new largest M; this entry point never
 * allocates.  It has no counterpart on the pages; it is an interface choice of
 * this library.
 *
 * Computes the same y[M][N] with the f32 decode GEMV (for every M), reading
 * x and writing y (device pointers, as bitlin_forward) on `stream`.  Its
 * split-K scratch is a fixed array of bitlin_noalloc_scratch_bytes() bytes
 * (16 MiB) compiled into the library, which every GPU that loads the library
 * keeps until the process exits.  The call needs
 *     (K/512) * M * ceil(N/32) * 128  bytes
 * of it and returns BITLIN_ESCRATCH, launching nothing, when that exceeds the
 * array (for example M=1 fits up to N = 248,320 at K = 5120).
 * The first call on a device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress) and caches it: make that first call
 * before any stream capture.  Every call shares the array, which keeps the
 * previous call's contents (nothing in it needs clearing: each call writes
 * every partial sum it reads).  Calls whose kernels overlap on the GPU
 * (different streams, or several host threads) race on the array: serialize
 * them.
 * Errors: BITLIN_EINVAL (NULL handle/x/y, M < 1, current device differs from
 * the handle's), BITLIN_ESCRATCH, BITLIN_ECUDA, and the handle's sticky error.
 */
bitlin_status bitlin_forward_noalloc(bitlin_t h, const float* x, int M, float* y,
                                     bitlin_stream_t stream);

/*
 * Greedy choice after the LM head: the folded product of x (as bitlin_forward:
 * same paths and tolerances), then ids[m] = the smallest n at which y[m][n] is
 * largest (a NaN score counts as largest).
 * Source: "Inside the One-Bit Engine", station on the LM head (the folded
 * vocabulary matrix, 248,320 x 5,120, gives one score per vocabulary entry)
 * and the Pulse "ARCHITECTURE-SPEC" folded-weights table (output.weight
 * carries signs + WHT, verified by argmax match).
 *
 *   x       device pointer, float [M][K], read only.
 *   logits  device pointer, float [M][N], overwritten with the scores, or NULL:
 *           the handle then keeps the scores in a buffer of its own (allocated
 *           on the first call with a new largest M).
 *   ids     device pointer, int32 [M], overwritten.
 *
 * Asynchronous on `stream`.  When the decode GEMV sums its split-K slices
 * inside thread-block clusters (one token on the vocabulary matrix), the pick
 * is fused into that kernel's finish: each CTA reduces the scores it writes
 * to one candidate and the last CTA to finish picks; otherwise a second
 * kernel reads the scores back and picks.  The first call with a new largest
 * M allocates the candidate and ticket buffers the handle keeps (the tickets
 * are zeroed in stream order on `stream`).
 * Errors: BITLIN_EINVAL (NULL handle/x/ids, M < 1), BITLIN_ENOMEM,
 * BITLIN_ECUDA, and the handle's sticky error.
 */
bitlin_status bitlin_argmax(bitlin_t h, const float* x, int M, float* logits, int32_t* ids,
                            bitlin_stream_t stream);

/*
 * The MLP block of the model around two folded matrices:
 *
 *   y = down( silu(g) * u ),  [g | u] = gate_up(x),  silu(g) = g / (1 + e^-g),
 *
 * where gate_up is a handle of 2F rows (rows 0..F-1 the gate matrix, rows
 * F..2F-1 the up matrix, both over the K of x) and down a handle with K = F.
 * Each product is the folded product of bitlin_forward (its own signs,
 * transform and, if set, permutation); SiLU and the product with up are done
 * in f32 inside the down projection's input gather (decode prologue or
 * rotation kernel), so the F-wide middle vector is never stored.
 * Source: "Inside the One-Bit Engine", MLP station (gate and up widen 5120
 * to 17408; SiLU(gate) multiplies up elementwise, in 32-bit arithmetic; a
 * third matrix narrows 17408 back to 5120); the Pulse "ARCHITECTURE-SPEC"
 * page's folded-weights table (ffn_gate, ffn_up and ffn_down carry signs +
 * WHT).
 *
 *   x       device pointer, float [M][gate_up's K], read only.
 *   y       device pointer, float [M][down's N], fully overwritten.
 *
 * Paths and tolerances as bitlin_forward, chosen per handle.  The first call
 * with a new largest M allocates the [M][2F] gate|up buffer on `down`.
 * Errors: BITLIN_EINVAL (NULL argument, M < 1, gate_up's N != 2 * down's K,
 * handles on different devices), BITLIN_ENOMEM, BITLIN_ECUDA, and either
 * handle's sticky error.
 */
bitlin_status bitlin_mlp_forward(bitlin_t gate_up, bitlin_t down, const float* x, int M, float* y,
                                 bitlin_stream_t stream);

/*
 * Embedding lookup with the inverse rotation, on the same handle (an N x K
 * folded matrix whose rows are embeddings):
 *
 *   out[m][k] = signs[k] * xt[k],  xt = blockwise normalized Walsh-Hadamard
 *   transform (blocks of 1024, 1/32) of z, z[k] = (bit(t, k) ? +1 : -1) *
 *   scale[t][k >> 7], t = ids[m].
 *
 * Source: the Pulse "ARCHITECTURE-SPEC" page, Hadamard-fold section: the
 * embedding lookup takes the transform first and the signs second (h =
 * signs * WHT(z)), the inverse order of the activation rotation, with the
 * same normalization and blocks; the row format is the Q1G128 format of the
 * "Inside the One-Bit Engine" page (station on the embedding row).  The
 * handle's permutation flag does not apply here.
 *
 *   ids     device pointer, int32 [M], token ids.
 *   out     device pointer, float [M][K], row-major, fully overwritten.
 *   stream  CUDA stream the work is queued on.
 *
 * Asynchronous; allocates nothing.  An id outside [0, N) gives a zero row and
 * makes the next bitlin_get_error return BITLIN_EINDEX (once; not sticky).
 * Errors: BITLIN_EINVAL (NULL handle/ids/out, M < 1), BITLIN_ECUDA, and the
 * handle's sticky error.
 */
bitlin_status bitlin_embed(bitlin_t h, const int32_t* ids, int M, float* out, bitlin_stream_t stream);

/* Size in bytes of the fixed scratch array used by bitlin_forward_noalloc. */
size_t bitlin_noalloc_scratch_bytes(void);

/* Select the path used for later calls (BITLIN_PATH_*).  EINVAL on an unknown value. */
bitlin_status bitlin_set_path(bitlin_t h, int path);

/*
 * The plan of a bitlin_forward call with M tokens on this handle, without
 * running it: *path = the BITLIN_PATH_* it takes (never AUTO), *kernels = the
 * kernels it launches (decode: 1 when the split-K sums inside a thread-block
 * cluster, 2 when a second kernel sums the partials; tensor paths: the
 * rotation and the GEMM, 2, or 3 on the bf16 path when the GEMM's tiles past
 * its last full wave of SMs run as a second, split-K launch).  The first call
 * may set up the decode kernels'
 * attributes on the current device.  Errors: BITLIN_EINVAL (NULL argument,
 * M < 1), BITLIN_ECUDA.
 */
bitlin_status bitlin_plan(bitlin_t h, int M, int* path, int* kernels);

/* Longest time, in nanoseconds, that any one wait inside the tensor-core
 * kernel may take before the kernel gives up and records BITLIN_ETIMEOUT
 * (default 2e9, or the BITLIN_WAIT_BUDGET_NS environment variable at create).
 * EINVAL for ns <= 0. */
bitlin_status bitlin_set_wait_budget(bitlin_t h, long long ns);

/* Testing aid for the failure path: when on != 0, later tensor-core calls
 * make their epilogue wait on a barrier that nothing ever arrives at, so the
 * bounded wait runs out, the kernel drains and frees its resources, and
 * bitlin_get_error / bitlin_forward_host report BITLIN_ETIMEOUT.  No fault,
 * trap or hang is involved.  The timeout is sticky on the handle. */
bitlin_status bitlin_test_stall(bitlin_t h, int on);

/* Release everything the handle owns.  NULL is accepted.  Synchronizes the device. */
bitlin_status bitlin_destroy(bitlin_t h);

/*
 * Wait for the handle's queued work and report a device-side failure
 * recorded by its kernels: BITLIN_ETIMEOUT when a bounded wait gave up (stays
 * set: sticky), BITLIN_EINDEX when bitlin_embed met a token id outside [0, N)
 * (reported once, then cleared), or BITLIN_ECUDA if synchronizing failed.
 */
bitlin_status bitlin_get_error(bitlin_t h);

/* The cudaError_t value behind the last BITLIN_ECUDA of this handle (0 if none). */
int bitlin_cuda_error(bitlin_t h);

/* A static, human-readable description of a status value. */
const char* bitlin_status_string(bitlin_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int bitlin_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BITLIN_H */
