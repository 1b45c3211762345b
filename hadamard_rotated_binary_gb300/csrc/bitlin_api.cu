// C-ABI of libbitlin: handle lifetime, argument checks, scratch management
// and dispatch between the decode GEMV and the tensor-core path.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <stdlib.h>
#include <string.h>

#include <new>

#include "bitlin_internal.cuh"

using namespace bitlin_impl;

namespace {

constexpr long long kDefaultWaitBudgetNs = 2000000000LL;  // 2 s per bounded wait

bitlin_status from_cuda(bitlin_t h, cudaError_t e)
{
    if (e == cudaSuccess) return BITLIN_OK;
    if (h) h->last_cuda_error = (int)e;
    return e == cudaErrorMemoryAllocation ? BITLIN_ENOMEM : BITLIN_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
void free_dev(T*& p)
{
    if (p) cudaFree(p);
    p = nullptr;
}

void release(bitlin_t h)
{
    free_dev(h->dbits);
    free_dev(h->dscales);
    free_dev(h->pbits);
    free_dev(h->pscales);
    free_dev(h->signs);
    free_dev(h->partials);
    free_dev(h->xt);
    free_dev(h->dev_error);
    free_dev(h->hx);
    free_dev(h->hy);
    free_dev(h->mlp_in);
    free_dev(h->logits);
    free_dev(h->amax_cand);
    free_dev(h->amax_tickets);
    if (h->h_err) cudaFreeHost(h->h_err);
    h->h_err = nullptr;
}

cudaError_t ensure_partials(bitlin_t h, int M)
{
    if (h->partials && h->partials_M >= M) return cudaSuccess;
    free_dev(h->partials);
    h->partials_M = 0;
    const size_t n = (size_t)h->S * M * h->T * kTileRows;
    cudaError_t e = cudaMalloc(&h->partials, n * sizeof(float));
    if (e == cudaSuccess) h->partials_M = M;
    return e;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Rotated-activation buffer for the tensor-core paths and its TMA descriptor:
// bf16 [M][K] (prefill) or [4M][K] (exact: three digits and a zero row per token).
bitlin_status ensure_xt(bitlin_t h, int M, int exact)
{
    const int rows = exact ? 4 * M : M;
    if (!h->xt || h->xt_M < rows) {
        free_dev(h->xt);
        h->xt_M = 0;
        h->tmap_M = 0;
        cudaError_t e = cudaMalloc(&h->xt, (size_t)rows * h->K * 2);
        if (e != cudaSuccess) return from_cuda(h, e);
        h->xt_M = rows;
    }
    if (h->tmap_M != M || h->tmap_exact != exact) {
        PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
        if (!enc) return from_cuda(h, cudaErrorNotSupported);
        // Viewed as [K/64][rows][64]: one box {64, tile width, 2} is a K-group's
        // two 128-byte-swizzled halves, stacked, in a single copy.
        cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(h->K / 64)};
        cuuint64_t strides[2] = {(cuuint64_t)h->K * 2, 128};
        cuuint32_t box[3] = {64, (cuuint32_t)bitlin_tc_tile_width(M, exact), 2};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = enc(reinterpret_cast<CUtensorMap*>(h->tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                         h->xt, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return from_cuda(h, cudaErrorInvalidValue);
        h->tmap_M = M;
        h->tmap_exact = exact;
    }
    return BITLIN_OK;
}

DecodeParams decode_params(bitlin_t h, const float* x, int M, float* y, int swiglu)
{
    DecodeParams p;
    p.bits = h->dbits;
    p.scales = h->dscales;
    p.signs = h->signs;
    p.x = x;
    p.y = y;
    p.partials = h->partials;
    p.M = M;
    p.N = h->N;
    p.K = h->K;
    p.S = h->S;
    p.T = h->T;
    p.perm = h->perm;
    p.ctas_per_slice = 0;
    p.cluster = 0;
    p.allow_cluster = 1;
    p.swiglu = swiglu;
    p.ids = nullptr;
    p.amax_cand = nullptr;
    p.amax_tickets = nullptr;
    return p;
}

bitlin_status run_decode(bitlin_t h, const float* x, int M, float* y, cudaStream_t s, int swiglu = 0)
{
    // The split-K scratch only when the call sums its slices outside a cluster
    // (two kernels); the cluster path keeps its partial sums in shared memory.
    int kernels = 0;
    cudaError_t e = bitlin_decode_kernels(decode_params(h, x, M, y, swiglu), h->num_sms, &kernels);
    if (e == cudaSuccess && kernels == 2) e = ensure_partials(h, M);
    if (e != cudaSuccess) return from_cuda(h, e);
    return from_cuda(h, bitlin_launch_decode(decode_params(h, x, M, y, swiglu), h->num_sms, s));
}

bitlin_status run_tc(bitlin_t h, const float* x, int M, float* y, cudaStream_t s, int exact, int swiglu = 0)
{
    bitlin_status st = ensure_xt(h, M, exact);
    if (st != BITLIN_OK) return st;
    cudaError_t e = bitlin_launch_rotate_bf16(x, h->signs, M, h->K, h->perm, exact, swiglu, h->xt, s);
    if (e != cudaSuccess) return from_cuda(h, e);
    PrefillParams p;
    p.bits = h->pbits;
    p.scales = h->pscales;
    p.y = y;
    p.dev_error = h->dev_error;
    p.M = M;
    p.N = h->N;
    p.K = h->K;
    p.num_sms = h->num_sms;
    p.wait_budget_ns = h->wait_budget_ns;
    e = exact ? bitlin_launch_tc_exact(p, h->tmap, h->tmap_bits, h->stall_test, s)
              : bitlin_launch_prefill(p, h->tmap, h->tmap_bits, h->stall_test, s);
    return from_cuda(h, e);
}

}  // namespace

extern "C" {

int bitlin_version(void) { return 100; }

const char* bitlin_status_string(bitlin_status s)
{
    switch (s) {
    case BITLIN_OK: return "success";
    case BITLIN_EINVAL: return "invalid argument";
    case BITLIN_ENOMEM: return "out of memory";
    case BITLIN_ECUDA: return "CUDA runtime error";
    case BITLIN_ETIMEOUT: return "a bounded device wait timed out";
    case BITLIN_EDEVICE: return "the current device is not an sm_103 GPU";
    case BITLIN_ESCRATCH: return "the call needs more scratch than the fixed no-alloc array holds";
    case BITLIN_EINDEX: return "a token id is outside [0, N)";
    }
    return "unknown status";
}

bitlin_status bitlin_create(bitlin_t* out, int N, int K, const uint32_t* packed_bits,
                            const uint16_t* scales, const float* signs, int perm_flag)
{
    if (!out) return BITLIN_EINVAL;
    *out = nullptr;
    if (!packed_bits || !scales || !signs || N < 1 || K < 1024 || K % 1024 != 0) return BITLIN_EINVAL;
    if (perm_flag != BITLIN_PERM_NONE && perm_flag != BITLIN_PERM_SSM_TILED_TO_GROUPED) return BITLIN_EINVAL;
    if (perm_flag == BITLIN_PERM_SSM_TILED_TO_GROUPED && K != 6144) return BITLIN_EINVAL;
    if (!aligned16(packed_bits) || !aligned16(scales) || !aligned16(signs)) return BITLIN_EINVAL;
    if ((long long)N * (K / 32) > (1LL << 40)) return BITLIN_EINVAL;

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BITLIN_EDEVICE;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) return BITLIN_EDEVICE;

    bitlin_t h = new (std::nothrow) bitlin();
    if (!h) return BITLIN_ENOMEM;
    h->device = dev;
    h->num_sms = sms;
    if (cudaDeviceGetAttribute(&h->host_page_tables, cudaDevAttrPageableMemoryAccessUsesHostPageTables, dev) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        h->host_page_tables = 0;
    }
    h->N = N;
    h->K = K;
    h->perm = perm_flag;
    h->S = K / kSlice;
    h->T = (N + kTileRows - 1) / kTileRows;
    h->wait_budget_ns = kDefaultWaitBudgetNs;
    if (const char* env = getenv("BITLIN_WAIT_BUDGET_NS")) {
        long long v = atoll(env);
        if (v > 0) h->wait_budget_ns = v;
    }

    const size_t units = (size_t)h->S * h->T;
    const size_t words = (size_t)N * (K / 32);
    const size_t groups = (size_t)N * (K / 128);
    cudaStream_t st = nullptr;
    int* bad = nullptr;
    int bad_host = 0;
    bitlin_status status = BITLIN_OK;
    cudaError_t e = cudaSuccess;
#define BITLIN_TRY(call)                      \
    do {                                      \
        e = (call);                           \
        if (e != cudaSuccess) goto fail_cuda; \
    } while (0)
    BITLIN_TRY(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
    BITLIN_TRY(cudaMalloc(&h->dbits, units * 4 * 32 * sizeof(uint4)));
    BITLIN_TRY(cudaMalloc(&h->dscales, units * 32 * sizeof(uint2)));
    BITLIN_TRY(cudaMalloc(&h->pbits, words * sizeof(uint32_t)));
    BITLIN_TRY(cudaMalloc(&h->pscales, groups * sizeof(uint16_t)));
    BITLIN_TRY(cudaMalloc(&h->signs, (size_t)K * sizeof(float)));
    BITLIN_TRY(cudaMalloc(&h->dev_error, 2 * sizeof(int)));
    BITLIN_TRY(cudaHostAlloc(&h->h_err, sizeof(int), cudaHostAllocDefault));
    bad = h->dev_error + 1;
    BITLIN_TRY(cudaMemsetAsync(h->dev_error, 0, 2 * sizeof(int), st));
    BITLIN_TRY(cudaMemcpyAsync(h->signs, signs, (size_t)K * sizeof(float), cudaMemcpyDeviceToDevice, st));
    BITLIN_TRY(cudaMemcpyAsync(h->pscales, scales, groups * sizeof(uint16_t), cudaMemcpyDeviceToDevice, st));
    BITLIN_TRY(bitlin_launch_check_signs(h->signs, K, bad, st));
    BITLIN_TRY(bitlin_launch_repack_decode(packed_bits, scales, N, K, h->dbits, h->dscales, st));
    BITLIN_TRY(bitlin_launch_repack_prefill(packed_bits, N, K, h->pbits, st));
    BITLIN_TRY(cudaMemcpyAsync(&bad_host, bad, sizeof(int), cudaMemcpyDeviceToHost, st));
    BITLIN_TRY(cudaStreamSynchronize(st));
    cudaStreamDestroy(st);
    st = nullptr;
    {
        // Tensor-path bits as a [N][K/32] u32 tensor, read in boxes of 4 words x 128 rows.
        PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
        if (!enc) {
            e = cudaErrorNotSupported;
            goto fail_cuda;
        }
        cuuint64_t dims[2] = {(cuuint64_t)(K / 32), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)(K / 8)};
        cuuint32_t box[2] = {4, (cuuint32_t)kPrefillRows};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = enc(reinterpret_cast<CUtensorMap*>(h->tmap_bits), CU_TENSOR_MAP_DATA_TYPE_UINT32, 2,
                         h->pbits, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            e = cudaErrorInvalidValue;
            goto fail_cuda;
        }
    }
    if (bad_host != 0) {
        status = BITLIN_EINVAL;
        goto fail;
    }
    *out = h;
    return BITLIN_OK;
#undef BITLIN_TRY
fail_cuda:
    status = (e == cudaErrorMemoryAllocation) ? BITLIN_ENOMEM : BITLIN_ECUDA;
fail:
    if (st) {
        cudaStreamSynchronize(st);
        cudaStreamDestroy(st);
    }
    release(h);
    delete h;
    return status;
}

// A Q1G128 tensor as the engine stores it: the fp16 scales (two per word,
// index n*(K/128) + g, the even index in the low half) and then the bits, in
// one array of words ("Inside the One-Bit Engine", embedding station).  The
// scales take N*K/256 words; on a little-endian device the low half of a word
// is the 16-bit element at the lower address, so that prefix is the [N][K/128]
// binary16 array bitlin_create takes.
bitlin_status bitlin_create_q1g128(bitlin_t* out, int N, int K, const uint32_t* qdata, const float* signs,
                                   int perm_flag)
{
    if (!out) return BITLIN_EINVAL;
    *out = nullptr;
    if (!qdata || N < 1 || K < 1024 || K % 1024 != 0) return BITLIN_EINVAL;
    const size_t scale_words = (size_t)N * (size_t)(K / 256);
    return bitlin_create(out, N, K, qdata + scale_words, reinterpret_cast<const uint16_t*>(qdata), signs,
                         perm_flag);
}

bitlin_status bitlin_set_path(bitlin_t h, int path)
{
    if (!h || path < BITLIN_PATH_AUTO || path > BITLIN_PATH_TC_EXACT) return BITLIN_EINVAL;
    h->path = path;
    return BITLIN_OK;
}

bitlin_status bitlin_set_wait_budget(bitlin_t h, long long ns)
{
    if (!h || ns <= 0) return BITLIN_EINVAL;
    h->wait_budget_ns = ns;
    return BITLIN_OK;
}

bitlin_status bitlin_test_stall(bitlin_t h, int on)
{
    if (!h) return BITLIN_EINVAL;
    h->stall_test = on ? 1 : 0;
    return BITLIN_OK;
}

namespace {

// The handle's path for M tokens (BITLIN_PATH_AUTO resolved).
int choose_path(bitlin_t h, int M)
{
    if (h->path != BITLIN_PATH_AUTO) return h->path;
    return M >= kPrefillMinM ? BITLIN_PATH_PREFILL : M > kDecodeMaxM ? BITLIN_PATH_TC_EXACT : BITLIN_PATH_DECODE;
}

bitlin_status run_path(bitlin_t h, const float* x, int M, float* y, cudaStream_t s, int swiglu)
{
    switch (choose_path(h, M)) {
    case BITLIN_PATH_PREFILL: return run_tc(h, x, M, y, s, 0, swiglu);
    case BITLIN_PATH_TC_EXACT: return run_tc(h, x, M, y, s, 1, swiglu);
    default: return run_decode(h, x, M, y, s, swiglu);
    }
}

}  // namespace

bitlin_status bitlin_plan(bitlin_t h, int M, int* path, int* kernels)
{
    if (!h || !path || !kernels || M < 1) return BITLIN_EINVAL;
    *path = choose_path(h, M);
    if (*path != BITLIN_PATH_DECODE) {
        // the rotation into bf16, then the tensor-core GEMM (bf16 path: two
        // launches when the tiles past the last full wave are split over K)
        *kernels = 1 + (*path == BITLIN_PATH_PREFILL ? bitlin_prefill_gemm_launches(M, h->N, h->num_sms) : 1);
        return BITLIN_OK;
    }
    return from_cuda(h, bitlin_decode_kernels(decode_params(h, nullptr, M, nullptr, 0), h->num_sms, kernels));
}

bitlin_status bitlin_forward(bitlin_t h, const float* x, int M, float* y, bitlin_stream_t stream)
{
    if (!h || !x || !y || M < 1) return BITLIN_EINVAL;
    if (h->sticky != BITLIN_OK) return h->sticky;
    return run_path(h, x, M, y, reinterpret_cast<cudaStream_t>(stream), 0);
}

bitlin_status bitlin_mlp_forward(bitlin_t gate_up, bitlin_t down, const float* x, int M, float* y,
                                 bitlin_stream_t stream)
{
    if (!gate_up || !down || !x || !y || M < 1) return BITLIN_EINVAL;
    if (gate_up->N != 2 * down->K || gate_up->device != down->device) return BITLIN_EINVAL;
    if (gate_up->sticky != BITLIN_OK) return gate_up->sticky;
    if (down->sticky != BITLIN_OK) return down->sticky;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!down->mlp_in || down->mlp_M < M) {
        free_dev(down->mlp_in);
        down->mlp_M = 0;
        cudaError_t e = cudaMalloc(&down->mlp_in, (size_t)M * gate_up->N * sizeof(float));
        if (e != cudaSuccess) return from_cuda(down, e);
        down->mlp_M = M;
    }
    bitlin_status st = run_path(gate_up, x, M, down->mlp_in, s, 0);
    if (st != BITLIN_OK) return st;
    return run_path(down, down->mlp_in, M, y, s, 1);
}

// Address under which the kernels may use a host buffer directly, or nullptr
// when it has to be staged through device memory: page-locked memory mapped
// into the device's address space (its device pointer), or any host memory on
// a device that reads pageable memory through the host's page tables.
static const void* host_direct(bitlin_t h, const void* p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    if (a.type == cudaMemoryTypeUnregistered && h->host_page_tables) return p;
    return nullptr;
}

bitlin_status bitlin_forward_host(bitlin_t h, const float* x_host, int M, float* y_host,
                                  bitlin_stream_t stream)
{
    if (!h || !x_host || !y_host || M < 1) return BITLIN_EINVAL;
    if (h->sticky != BITLIN_OK) return h->sticky;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    // The kernels read x and write y in host memory where the device can reach
    // it (no copy operations); otherwise x and y pass through device buffers.
    const float* xd = static_cast<const float*>(host_direct(h, x_host));
    float* yd = static_cast<float*>(const_cast<void*>(host_direct(h, y_host)));
    if ((!xd || !yd) && (!h->hx || h->h_M < M)) {
        free_dev(h->hx);
        free_dev(h->hy);
        h->h_M = 0;
        e = cudaMalloc(&h->hx, (size_t)M * h->K * sizeof(float));
        if (e == cudaSuccess) e = cudaMalloc(&h->hy, (size_t)M * h->N * sizeof(float));
        if (e != cudaSuccess) return from_cuda(h, e);
        h->h_M = M;
    }
    if (!xd) {
        e = cudaMemcpyAsync(h->hx, x_host, (size_t)M * h->K * sizeof(float), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return from_cuda(h, e);
        xd = h->hx;
    }
    bitlin_status st = bitlin_forward(h, xd, M, yd ? yd : h->hy, stream);
    if (st != BITLIN_OK) return st;
    e = cudaSuccess;
    if (!yd) e = cudaMemcpyAsync(y_host, h->hy, (size_t)M * h->N * sizeof(float), cudaMemcpyDeviceToHost, s);
    // Only the tensor-core kernels can record a timeout (the decode GEMV has no
    // waits of its own), so the error word is read back after those alone.
    const bool tc = choose_path(h, M) != BITLIN_PATH_DECODE;
    if (e == cudaSuccess && tc) e = cudaMemcpyAsync(h->h_err, h->dev_error, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return from_cuda(h, e);
    if (tc && *h->h_err == kDevErrTimeout) h->sticky = BITLIN_ETIMEOUT;
    return h->sticky;
}

bitlin_status bitlin_get_error(bitlin_t h)
{
    if (!h) return BITLIN_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(h, e);
    int v = 0;
    e = cudaMemcpy(&v, h->dev_error, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(h, e);
    if (v == kDevErrTimeout) h->sticky = BITLIN_ETIMEOUT;
    if (v == kDevErrIndex && h->sticky == BITLIN_OK) {
        e = cudaMemset(h->dev_error, 0, sizeof(int));
        if (e != cudaSuccess) return from_cuda(h, e);
        return BITLIN_EINDEX;
    }
    return h->sticky;
}

bitlin_status bitlin_argmax(bitlin_t h, const float* x, int M, float* logits, int32_t* ids,
                            bitlin_stream_t stream)
{
    if (!h || !x || !ids || M < 1) return BITLIN_EINVAL;
    if (h->sticky != BITLIN_OK) return h->sticky;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float* y = logits;
    if (!y) {
        if (!h->logits || h->logits_M < M) {
            free_dev(h->logits);
            h->logits_M = 0;
            cudaError_t e = cudaMalloc(&h->logits, (size_t)M * h->N * sizeof(float));
            if (e != cudaSuccess) return from_cuda(h, e);
            h->logits_M = M;
        }
        y = h->logits;
    }
    if (!h->amax_cand || h->amax_M < M) {
        free_dev(h->amax_cand);
        free_dev(h->amax_tickets);
        h->amax_M = 0;
        cudaError_t e = cudaMalloc(&h->amax_cand, bitlin_argmax_scratch_bytes(M));
        if (e == cudaSuccess) e = cudaMalloc(&h->amax_tickets, (size_t)M * sizeof(unsigned));
        // Zeroed in stream order: the pick kernels on this stream see zero tickets.
        if (e == cudaSuccess) e = cudaMemsetAsync(h->amax_tickets, 0, (size_t)M * sizeof(unsigned), s);
        if (e != cudaSuccess) return from_cuda(h, e);
        h->amax_M = M;
    }
    // On the decode path with cluster split-K the GEMV picks the argmax in its
    // finish; otherwise the scores are written first and a second kernel picks.
    if (choose_path(h, M) == BITLIN_PATH_DECODE) {
        DecodeParams p = decode_params(h, x, M, y, 0);
        p.ids = ids;
        p.amax_cand = static_cast<float2*>(h->amax_cand);
        p.amax_tickets = h->amax_tickets;
        int kernels = 0, fused = 0;
        cudaError_t e = bitlin_decode_kernels(p, h->num_sms, &kernels, &fused);
        if (e == cudaSuccess && fused) return from_cuda(h, bitlin_launch_decode(p, h->num_sms, s));
        if (e != cudaSuccess) return from_cuda(h, e);
    }
    bitlin_status st = run_path(h, x, M, y, s, 0);
    if (st != BITLIN_OK) return st;
    return from_cuda(h, bitlin_launch_argmax(y, M, h->N, h->amax_cand, h->amax_tickets, ids, s));
}

bitlin_status bitlin_embed(bitlin_t h, const int32_t* ids, int M, float* out, bitlin_stream_t stream)
{
    if (!h || !ids || !out || M < 1) return BITLIN_EINVAL;
    if (h->sticky != BITLIN_OK) return h->sticky;
    return from_cuda(h, bitlin_launch_embed(h->pbits, h->pscales, h->signs, ids, M, h->N, h->K, out,
                                            h->dev_error, reinterpret_cast<cudaStream_t>(stream)));
}

int bitlin_cuda_error(bitlin_t h) { return h ? h->last_cuda_error : 0; }

bitlin_status bitlin_destroy(bitlin_t h)
{
    if (!h) return BITLIN_OK;
    cudaError_t e = cudaDeviceSynchronize();
    release(h);
    delete h;
    return e == cudaSuccess ? BITLIN_OK : BITLIN_ECUDA;
}

}  // extern "C"
