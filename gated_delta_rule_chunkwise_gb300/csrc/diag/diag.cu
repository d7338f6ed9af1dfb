// Diagnostic entry points (include/ldn_diag.h), built into their own library
// (lib/libldn_diag.so), apart from the product library libldn.so: they check,
// on tiny matrices, the building blocks the tensor-core kernels rely on --
// SWIZZLE_128B placement of TMA loads, shared-memory / instruction descriptors
// for K-major and MN-major 16-bit operands, and the TMEM row layout of M = 64
// and M = 128 accumulators -- and drive a bounded wait to its limit.  They exist
// so that tests can pin these encodings and the failure path directly.  This
// library has a status word of its own (ldn_diag_get_device_status).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../../include/ldn.h"
#include "../../../include/ldn_diag.h"
#include "../sm100_ptx.cuh"
#include "../tma_host.cuh"

namespace ldn {
// Status word of the diagnostic kernels (the same encoding as libldn's: bit
// 1 << LDN_ERR_TIMEOUT set by a kernel that abandoned a bounded wait).
__device__ int g_diag_status = 0;

namespace {
using namespace sm100;

int *status_word_ptr()
{
    static int *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_diag_status) != cudaSuccess) return nullptr;
        addr[dev] = (int *)p;
    }
    return addr[dev];
}

constexpr uint64_t kDiagTimeoutNs = 2000000000ull;   // 2 s
constexpr float kSentinel = -12345.0f;

// One MMA chain D = A * B^T over K, A [M][K], B [N][K] (row-major bf16 in
// global memory), placed in shared memory K-major or MN-major; the whole
// 128-lane x N TMEM region is dumped to D_out [128][N] after being prefilled
// with a sentinel, so a test can see which lanes the accumulator occupies.
__global__ void __launch_bounds__(128)
diag_umma_kernel(const uint16_t *__restrict__ A, const uint16_t *__restrict__ B, float *__restrict__ D,
                 int M, int N, int K, int a_mn, int b_mn, uint32_t fmt, uint32_t tmem_cols, int *status)
{
    extern __shared__ uint8_t dsmem[];
    uint8_t *base = dsmem + ((1024u - (smem_u32(dsmem) & 1023u)) & 1023u);
    uint8_t *As = base;                    // up to 128 x 128 bf16
    uint8_t *Bs = base + 32768;            // up to 256 x 128 bf16
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int e = tid; e < M * K; e += 128) {
        const int m = e / K, k = e % K;
        const uint32_t off = a_mn ? (m >> 6) * (uint32_t)K * 128u + sw128_offset(k, m & 63)
                                  : (k >> 6) * (uint32_t)M * 128u + sw128_offset(m, k & 63);
        *reinterpret_cast<uint16_t *>(As + off) = A[e];
    }
    for (int e = tid; e < N * K; e += 128) {
        const int n = e / K, k = e % K;
        const uint32_t off = b_mn ? (n >> 6) * (uint32_t)K * 128u + sw128_offset(k, n & 63)
                                  : (k >> 6) * (uint32_t)N * 128u + sw128_offset(n, k & 63);
        *reinterpret_cast<uint16_t *>(Bs + off) = B[e];
    }
    fence_proxy_async_smem();
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_s;

    float sent[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) sent[i] = kSentinel;
    for (int c = 0; c < N; c += 16) tmem_st16(tmem_addr(tbase, 32 * warp, c), sent);
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
        const uint32_t idesc = idesc_f16kind_f32(M, N, a_mn, b_mn, fmt);
        const uint32_t a0 = smem_u32(As), b0 = smem_u32(Bs);
        for (int s = 0; s < K / 16; ++s) {
            const uint64_t ad = a_mn ? mnmajor_desc(a0, K, s) : kmajor_desc(a0, M, s);
            const uint64_t bd = b_mn ? mnmajor_desc(b0, K, s) : kmajor_desc(b0, N, s);
            umma_bf16(tbase, ad, bd, idesc, s > 0);
        }
        umma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0, kDiagTimeoutNs);
    if (!ok && lane == 0) atomicOr(status, 1 << LDN_ERR_TIMEOUT);
    tc_fence_after();
    if (ok) {
        for (int c = 0; c < N; c += 16) {
            float v[16];
            tmem_ld16(tmem_addr(tbase, 32 * warp, c), v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) D[(size_t)(32 * warp + lane) * N + c + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, tmem_cols);
}

// The same chain with A (M = 128) held in TMEM instead of shared memory: row r
// of A goes to lane r as 16-bit pairs, element k in the low (k even) or high
// (k odd) half of column kAcol + k / 2, written with tcgen05.st.  D occupies
// columns [0, N); the full 128 x N region is dumped as in diag_umma_kernel.
constexpr uint32_t kAcol = 256;
__global__ void __launch_bounds__(128)
diag_umma_ts_kernel(const uint16_t *__restrict__ A, const uint16_t *__restrict__ B, float *__restrict__ D,
                    int N, int K, int b_mn, uint32_t fmt, int *status)
{
    extern __shared__ uint8_t dsmem[];
    uint8_t *Bs = dsmem + ((1024u - (smem_u32(dsmem) & 1023u)) & 1023u);   // up to 256 x 128 16-bit
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base_s;
    const int tid = threadIdx.x, warp = tid >> 5;

    for (int e = tid; e < N * K; e += 128) {
        const int n = e / K, k = e % K;
        const uint32_t off = b_mn ? (n >> 6) * (uint32_t)K * 128u + sw128_offset(k, n & 63)
                                  : (k >> 6) * (uint32_t)N * 128u + sw128_offset(n, k & 63);
        *reinterpret_cast<uint16_t *>(Bs + off) = B[e];
    }
    fence_proxy_async_smem();
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_s;
    const uint32_t lane_addr = (uint32_t)(32 * warp) << 16;

    // row tid of A -> lane tid (thread tid of warp w owns lane 32 w + lane)
    float sent[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) sent[i] = kSentinel;
    for (int c = 0; c < N; c += 16) tmem_st16(tbase + lane_addr + c, sent);
    for (int c = 0; c < K / 2; c += 16) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int k = 2 * (c + i);
            w[i] = (uint32_t)A[(size_t)tid * K + k] | ((uint32_t)A[(size_t)tid * K + k + 1] << 16);
        }
        tmem_st16u(tbase + lane_addr + kAcol + c, w);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
        const uint32_t idesc = idesc_f16kind_f32(128, N, 0, b_mn, fmt);
        const uint32_t b0 = smem_u32(Bs);
        for (int s = 0; s < K / 16; ++s) {
            const uint64_t bd = b_mn ? mnmajor_desc(b0, K, s) : kmajor_desc(b0, N, s);
            umma_ts(tbase, tbase + kAcol + 8 * s, bd, idesc, s > 0);
        }
        umma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0, kDiagTimeoutNs);
    if (!ok && (tid & 31) == 0) atomicOr(status, 1 << LDN_ERR_TIMEOUT);
    tc_fence_after();
    if (ok) {
        for (int c = 0; c < N; c += 16) {
            float v[16];
            tmem_ld16(tbase + lane_addr + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) D[(size_t)tid * N + c + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// TMA load of a 64-row x 64-column bf16 box (SWIZZLE_128B) at (row0, col0)
// of a [rows][cols] matrix, then a raw byte dump of the 8 KiB tile.
__global__ void __launch_bounds__(128)
diag_tma_kernel(const __grid_constant__ CUtensorMap map, uint8_t *__restrict__ out, int col0, int row0, int *status)
{
    __shared__ __align__(1024) uint8_t tile[8192];
    __shared__ uint64_t bar;
    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar, 8192);
        tma_load_4d(tile, &map, &bar, col0, 0, row0, 0);
    }
    const bool ok = mbar_wait(&bar, 0, kDiagTimeoutNs);
    if (!ok) {
        if (tid == 0) atomicOr(status, 1 << LDN_ERR_TIMEOUT);
        return;
    }
    for (int i = tid; i < 8192 / 16; i += 128)
        reinterpret_cast<uint4 *>(out)[i] = reinterpret_cast<const uint4 *>(tile)[i];
}

// A bounded wait on an mbarrier that nothing ever arrives on: the kernel must
// give up after `timeout_ns`, record LDN_ERR_TIMEOUT and return normally.
__global__ void diag_timeout_kernel(uint64_t timeout_ns, int *status, int *waited_ok)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, timeout_ns);   // phase 0 never completes
    if (threadIdx.x == 0) {
        *waited_ok = ok ? 1 : 0;
        if (!ok) atomicOr(status, 1 << LDN_ERR_TIMEOUT);
    }
}

}  // namespace
}  // namespace ldn

using namespace ldn;

extern "C" int ldn_diag_get_device_status(void *stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LDN_ERR_CUDA;
    int h = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_diag_status, sizeof(int)) != cudaSuccess) return LDN_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_diag_status, &zero, sizeof(int)) != cudaSuccess) return LDN_ERR_CUDA;
    if (h & (1 << LDN_ERR_TIMEOUT)) return LDN_ERR_TIMEOUT;
    return h ? LDN_ERR_CUDA : LDN_OK;
}

extern "C" int ldn_diag_wait_timeout(long long timeout_ns, int *waited_ok, void *stream)
{
    if (!waited_ok || timeout_ns < 0 || timeout_ns > 2000000000LL) return LDN_ERR_INVALID_ARG;
    int *sw = status_word_ptr();
    if (!sw) return LDN_ERR_CUDA;
    diag_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)timeout_ns, sw, waited_ok);
    return cudaGetLastError() == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

extern "C" int ldn_diag_umma(const void *A, const void *B, float *D, int M, int N, int K, int a_mn, int b_mn, int fmt,
                             void *stream)
{
    if (!A || !B || !D) return LDN_ERR_INVALID_ARG;
    if (fmt != 0 && fmt != 1) return LDN_ERR_INVALID_ARG;
    if (M != 64 && M != 128) return LDN_ERR_UNSUPPORTED;
    if (N < 16 || N > 256 || N % 16 != 0) return LDN_ERR_UNSUPPORTED;
    if (K < 16 || K > 128 || K % 16 != 0) return LDN_ERR_UNSUPPORTED;
    if ((a_mn && (M % 64 != 0 || K % 8 != 0)) || (b_mn && N % 64 != 0)) return LDN_ERR_UNSUPPORTED;
    int *sw = status_word_ptr();
    if (!sw) return LDN_ERR_CUDA;
    uint32_t cols = 32;
    while (cols < (uint32_t)N) cols <<= 1;
    const size_t smem = 32768 + 65536 + 1024;
    if (cudaFuncSetAttribute(diag_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return LDN_ERR_CUDA;
    diag_umma_kernel<<<1, 128, smem, (cudaStream_t)stream>>>((const uint16_t *)A, (const uint16_t *)B,
                                                             D, M, N, K, a_mn, b_mn, (uint32_t)fmt, cols, sw);
    return cudaGetLastError() == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

extern "C" int ldn_diag_umma_tmem_a(const void *A, const void *B, float *D, int N, int K, int b_mn, int fmt,
                                    void *stream)
{
    if (!A || !B || !D) return LDN_ERR_INVALID_ARG;
    if (fmt != 0 && fmt != 1) return LDN_ERR_INVALID_ARG;
    if (N < 16 || N > 256 || N % 16 != 0) return LDN_ERR_UNSUPPORTED;
    if (K < 32 || K > 128 || K % 32 != 0) return LDN_ERR_UNSUPPORTED;
    if (b_mn && N % 64 != 0) return LDN_ERR_UNSUPPORTED;
    int *sw = status_word_ptr();
    if (!sw) return LDN_ERR_CUDA;
    const size_t smem = 65536 + 1024;
    if (cudaFuncSetAttribute(diag_umma_ts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return LDN_ERR_CUDA;
    diag_umma_ts_kernel<<<1, 128, smem, (cudaStream_t)stream>>>((const uint16_t *)A, (const uint16_t *)B, D, N, K,
                                                                b_mn, (uint32_t)fmt, sw);
    return cudaGetLastError() == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

extern "C" int ldn_diag_tma_sw128(const void *src, void *dst, int rows, int cols, int row0, int col0, void *stream)
{
    if (!src || !dst) return LDN_ERR_INVALID_ARG;
    if (((uintptr_t)src & 15u) || rows < 1 || cols < 64 || cols % 8 != 0) return LDN_ERR_INVALID_ARG;
    if (col0 < 0 || col0 % 64 != 0 || col0 + 64 > cols || row0 < 0) return LDN_ERR_INVALID_ARG;
    int *sw = status_word_ptr();
    if (!sw) return LDN_ERR_CUDA;
    CUtensorMap map;
    if (!make_tmap_bf16_4d(&map, src, (uint64_t)cols, 1, (uint64_t)rows, 1, 64, 64)) return LDN_ERR_CUDA;
    diag_tma_kernel<<<1, 128, 0, (cudaStream_t)stream>>>(map, (uint8_t *)dst, col0, row0, sw);
    return cudaGetLastError() == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}
