// Chunkwise forward on the 5th-generation tensor cores (tcgen05, fp16
// operands, fp32 accumulators in TMEM), fp32 state, for bf16 q/k/v with
// dk = 128 and dv a multiple of 64; DeltaNet and Gated DeltaNet.
//
// Operand precision: the bf16 q/k/v tiles are converted to fp16 in shared
// memory on arrival (exact for the magnitudes of normalised activations), and
// every intermediate operand (P, T, P T, Q~, W, the state copy, U~) is
// rounded to fp16 rather than bf16: 2^-11 instead of 2^-8 relative rounding,
// which keeps the chunk result within a few 1e-3 of the exact recurrence on
// a max-error / RMS scale.  Accumulation, the inverse and the state are fp32.
// Intermediates and inputs must stay below the fp16 range (65504).
//
// Chunk algebra (exact; derived from the per-token rules of the
// linear-attention notes, Sec. 2.3-2.4, which give no chunk form).  Memory
// orientation H = S^T ([dk][dv]).  For a chunk of C = 64 rows with incoming
// state H0, scalar inclusive log-decay prefix g_r and Gamma_rj = e^{g_r - g_j}:
//   A   = strict_tril(Diag(beta) (K K^T) * Gamma)         P = tril(Q K^T * Gamma)
//   T   = (I + A)^{-1}                                      (UT / WY transform)
//   Tu  = T Diag(beta),   Tw = T Diag(beta e^{g})
//   U'  = Tu V,   W = Tw K,   Q~ = Diag(e^{g}) Q - P W
//   O   = P U' + Q~ H0
//   U   = U' - W H0,   H1 = e^{g_C} H0 + K^T Diag(e^{g_C - g}) U
// Every contraction runs as an M = 128 tcgen05.mma by stacking two 64-row
// operands that share the right-hand side:
//   MMA1  [Q ; K] K^T              -> P_raw (rows 0-63), (K K^T) (rows 64-127)
//   MMA2  [P ; I] [Tu | Tw]        -> [P Tu | P Tw], [Tu | Tw]
//   MMA3  [P Tu ; Tu] V            -> P U' (= intra-chunk output), U'
//   MMA4  [Tw ; -P Tw] K           -> W, -P W
//   MMA5  accumulate [Q~ ; -W] H0 onto MMA3's result -> O (rows 0-63), U (rows 64-127)
//   MMA6  K^T U~                   -> K^T Diag(e^{g_C - g}) U (state increment)
// Only MMA5, MMA6 and the register update of H depend on the incoming state.
// The unit-lower-triangular inverse is computed on CUDA cores in fp32 by 16x16
// blocks (diagonal blocks by substitution, off-diagonal blocks by block
// substitution).
//
// Work split: one CTA per (b, h, 64-wide slice of dv) -- value columns are
// independent (state-reduction notes, Sec. 2.5) -- with 128 threads; thread t
// owns TMEM lane t, i.e. row t of every accumulator, and row t of the fp32
// state slice H[t][0:64] in registers.  q/k/v chunk tiles arrive by TMA
// (128-byte swizzle, two stages); all other operands are written by the
// threads into swizzled shared memory.  One elected thread issues TMA and MMA.
// Every mbarrier wait is bounded in time; a timeout sets LDN_ERR_TIMEOUT in
// the status word, abandons the remaining chunks, frees TMEM and returns.
#include "ldn_internal.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace ldn {
namespace {
using namespace sm100;

constexpr int kC = 64;
constexpr int kDK = 128;
constexpr int kDVS = 64;
constexpr int kThreads = 128;
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait, far above any legitimate latency

// TMEM columns (fp32, 128 lanes).
constexpr uint32_t kColD1 = 0;      // 64
constexpr uint32_t kColDP = 64;     // 128
constexpr uint32_t kColRV = 192;    // 64
constexpr uint32_t kColDK = 256;    // 128
constexpr uint32_t kColD6 = 384;    // 64
constexpr uint32_t kTmemCols = 512;

// Shared-memory plan (bytes from a 1024-aligned base).
constexpr uint32_t kQKBytes = 2 * 16384;      // [Q;K] K-major, 2 blocks of 128 rows x 128 B
constexpr uint32_t kVBytes = 8192;            // V slice, 64 rows x 128 B
constexpr uint32_t kOffQK0 = 0;
constexpr uint32_t kOffQK1 = kOffQK0 + kQKBytes;
constexpr uint32_t kOffV0 = kOffQK1 + kQKBytes;
constexpr uint32_t kOffV1 = kOffV0 + kVBytes;
constexpr uint32_t kOffPI = kOffV1 + kVBytes;          // [P ; I] K-major 128 x 64
constexpr uint32_t kOffTT = kOffPI + 16384;            // [Tu | Tw] MN-major 64 x 128  (later [Tw ; -P Tw])
constexpr uint32_t kOffAV = kOffTT + 16384;            // [P Tu ; Tu] K-major 128 x 64
constexpr uint32_t kOffA5 = kOffAV + 16384;            // [Q~ ; -W] K-major 128 x 128
constexpr uint32_t kOffHB = kOffA5 + 32768;            // H bf16, MN-major 128 x 64
constexpr uint32_t kOffF = kOffHB + 16384;             // fp32 A [64][65] (later U~ bf16 64 x 64)
constexpr uint32_t kOffTf = kOffF + 64 * 65 * 4;       // fp32 T [64][65]
constexpr uint32_t kOffX = kOffTf + 64 * 65 * 4;       // fp32 block-inverse scratch [3][16][16]
constexpr uint32_t kOffSmall = kOffX + 3 * 256 * 4;
constexpr uint32_t kSmemBytes = kOffSmall + 2048 + 1024;   // + small arrays + alignment slack

struct Small {
    uint64_t bar_load[2];
    uint64_t bar_mma;
    uint32_t tmem_base;
    int fail;
    float beta[kC];
    float g[kC];        // inclusive log-decay prefix
    float eg[kC];       // e^{g_r}
    float egc[kC];      // e^{g_C - g_r}
    float gC;           // e^{g_C}
};

__device__ __forceinline__ void st_bf16x8(uint8_t *p, const float *v)
{
    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(v[2], v[3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[4], v[5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(v[6], v[7]);
    uint4 u;
    u.x = *reinterpret_cast<uint32_t *>(&h0);
    u.y = *reinterpret_cast<uint32_t *>(&h1);
    u.z = *reinterpret_cast<uint32_t *>(&h2);
    u.w = *reinterpret_cast<uint32_t *>(&h3);
    *reinterpret_cast<uint4 *>(p) = u;
}

__device__ __forceinline__ void st_f16x8(uint8_t *p, const float *v)
{
    __half2 h0 = __floats2half2_rn(v[0], v[1]);
    __half2 h1 = __floats2half2_rn(v[2], v[3]);
    __half2 h2 = __floats2half2_rn(v[4], v[5]);
    __half2 h3 = __floats2half2_rn(v[6], v[7]);
    uint4 u;
    u.x = *reinterpret_cast<uint32_t *>(&h0);
    u.y = *reinterpret_cast<uint32_t *>(&h1);
    u.z = *reinterpret_cast<uint32_t *>(&h2);
    u.w = *reinterpret_cast<uint32_t *>(&h3);
    *reinterpret_cast<uint4 *>(p) = u;
}

// Store 16 consecutive columns [col, col+16) of row `row` into a SWIZZLE_128B
// block of fp16 operands (col % 16 == 0, col < 64).
__device__ __forceinline__ void st_row16(uint8_t *block, int row, int col, const float *v)
{
    st_f16x8(block + sw128_offset(row, col), v);
    st_f16x8(block + sw128_offset(row, col + 8), v + 8);
}

__device__ __forceinline__ void ld_row8(const uint8_t *block, int row, int col, float *v)
{
    const uint4 u = *reinterpret_cast<const uint4 *>(block + sw128_offset(row, col));
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// In-place bf16 -> fp16 conversion of `bytes` of swizzled tile (all threads).
// Exact for |x| in [2^-14, 65504]; smaller magnitudes keep an absolute error
// below 2^-25.
__device__ __forceinline__ void tile_bf16_to_f16(uint8_t *p, int bytes, int tid)
{
    for (int o = tid * 16; o < bytes; o += kThreads * 16) {
        uint4 u = *reinterpret_cast<const uint4 *>(p + o);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162 *>(&w[i]);
            __half2 h2 = __float22half2_rn(__bfloat1622float2(b2));
            w[i] = *reinterpret_cast<uint32_t *>(&h2);
        }
        *reinterpret_cast<uint4 *>(p + o) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ beta,
                const float *__restrict__ gate, const float *S0, __nv_bfloat16 *__restrict__ out,
                float *S_final, int T, int H, int dv, int *status)
{
    extern __shared__ uint8_t dsmem[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)dsmem + 1023) & ~(uintptr_t)1023);
    Small &S = *reinterpret_cast<Small *>(sm + kOffSmall);
    float *Af = reinterpret_cast<float *>(sm + kOffF);
    float *Tf = reinterpret_cast<float *>(sm + kOffTf);
    float *Xs = reinterpret_cast<float *>(sm + kOffX);
    uint8_t *PI = sm + kOffPI, *TT = sm + kOffTT, *AV = sm + kOffAV, *A5 = sm + kOffA5, *HB = sm + kOffHB;
    uint8_t *UB = sm + kOffF;   // U~ (bf16) reuses the fp32 A buffer after the inverse

    const int tid = threadIdx.x, warp = tid >> 5;
    const int slices = dv / kDVS;
    const int unit = blockIdx.x / slices;
    const int b = unit / H, h = unit % H;
    const int n0 = (blockIdx.x % slices) * kDVS;
    const int nchunks = (T + kC - 1) / kC;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

    if (tid == 0) {
        mbar_init(&S.bar_load[0], 1);
        mbar_init(&S.bar_load[1], 1);
        mbar_init(&S.bar_mma, 1);
        fence_mbar_init();
        S.fail = 0;
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 0) {
        tmem_alloc(&S.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    // Identity rows 64..127 of [P ; I] (constant for the whole sequence).
    {
        const int r = tid - 64;
        if (r >= 0)
            for (int c = 0; c < 64; c += 16) {
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = (c + i == r) ? 1.f : 0.f;
                st_row16(PI, tid, c, v);
            }
    }
    // Incoming state: row c = tid of the slice, fp32 in registers, bf16 copy in HB.
    float Hreg[kDVS];
    {
        const float *src = S0 ? S0 + ((size_t)unit * kDK + tid) * dv + n0 : nullptr;
#pragma unroll
        for (int n = 0; n < kDVS; n += 4) {
            float4 x = src ? *reinterpret_cast<const float4 *>(src + n) : make_float4(0.f, 0.f, 0.f, 0.f);
            Hreg[n] = x.x; Hreg[n + 1] = x.y; Hreg[n + 2] = x.z; Hreg[n + 3] = x.w;
        }
#pragma unroll
        for (int n = 0; n < kDVS; n += 16) st_row16(HB, tid, n, &Hreg[n]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = S.tmem_base;

    int pending[2] = {-1, -1};   // chunk whose TMA load is in flight per stage (thread 0)
    auto issue_load = [&](int c) {
        const int st = c & 1;
        pending[st] = c;
        uint8_t *qk = sm + (st ? kOffQK1 : kOffQK0);
        uint8_t *vv = sm + (st ? kOffV1 : kOffV0);
        mbar_arrive_expect_tx(&S.bar_load[st], 2 * 16384 + 8192);
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(qk + kb * 16384, &tm_q, &S.bar_load[st], kb * 64, h, c * kC, b);
            tma_load_4d(qk + kb * 16384 + 8192, &tm_k, &S.bar_load[st], kb * 64, h, c * kC, b);
        }
        tma_load_4d(vv, &tm_v, &S.bar_load[st], n0, h, c * kC, b);
    };
    if (tid == 0) {
        issue_load(0);
        if (nchunks > 1) issue_load(1);
    }

    uint32_t mma_phase = 0;
    // Wait for the MMA commit; every thread calls it.  Returns false (in every
    // thread alike) if any thread gave up on the wait.
    auto wait_mma = [&]() -> bool {
        if (!mbar_wait(&S.bar_mma, mma_phase, kWaitNs)) S.fail = 1;
        mma_phase ^= 1u;
        tc_fence_after();
        __syncthreads();
        return S.fail == 0;
    };

    // Every operand of every MMA is fp16 (the q/k/v tiles are converted in place
    // on arrival), so no MMA mixes element types.
    const uint32_t id_n64 = idesc_f16kind_f32(128, 64, 0, 0, kMmaF16);      // K-major A, K-major B
    const uint32_t id_mn_n128 = idesc_f16kind_f32(128, 128, 0, 1, kMmaF16);  // K-major A, MN-major B
    const uint32_t id_mn_n64 = idesc_f16kind_f32(128, 64, 0, 1, kMmaF16);
    const uint32_t id_amn_n64 = idesc_f16kind_f32(128, 64, 1, 1, kMmaF16);   // MN-major A and B

    for (int c = 0; c < nchunks; ++c) {
        const int st = c & 1;
        const int t0 = c * kC;
        const int L = min(kC, T - t0);
        uint8_t *QK = sm + (st ? kOffQK1 : kOffQK0);
        uint8_t *Vt = sm + (st ? kOffV1 : kOffV0);
        const uint32_t qk_s = smem_u32(QK), k_s = qk_s + 8192, v_s = smem_u32(Vt);

        // ---- gates and beta of this chunk (tail rows: beta 0, no decay)
        if (tid < kC) {
            const size_t i = ((size_t)b * T + t0 + tid) * H + h;
            S.beta[tid] = tid < L ? beta[i] : 0.f;
            S.g[tid] = (MODE == LDN_GDN && tid < L) ? gate[i] : 0.f;
        }
        __syncthreads();
        if (MODE == LDN_GDN && tid == 0) {
            float acc = 0.f;
            for (int r = 0; r < kC; ++r) { acc += S.g[r]; S.g[r] = acc; }
            S.gC = expf(acc);
        }
        __syncthreads();
        if (tid < kC) {
            S.eg[tid] = MODE == LDN_GDN ? expf(S.g[tid]) : 1.f;
            S.egc[tid] = MODE == LDN_GDN ? expf(S.g[kC - 1] - S.g[tid]) : 1.f;
        }
        const float gC = MODE == LDN_GDN ? S.gC : 1.f;

        // ---- MMA1: [Q ; K] K^T
        if (!mbar_wait(&S.bar_load[st], (c >> 1) & 1, kWaitNs)) S.fail = 1;
        __syncthreads();
        if (S.fail) break;
        if (tid == 0) pending[st] = -1;
        tile_bf16_to_f16(QK, kQKBytes, tid);
        tile_bf16_to_f16(Vt, kVBytes, tid);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            for (int s = 0; s < kDK / 16; ++s)
                umma_bf16(tbase + kColD1, kmajor_desc(qk_s, 128, s), kmajor_desc(k_s, 128, s), id_n64, s > 0);
            umma_commit(&S.bar_mma);
        }
        if (!wait_mma()) break;

        // ---- A (fp32, for the inverse) and P (bf16 operand), gated and masked
        {
            const bool isP = tid < 64;
            const int r = isP ? tid : tid - 64;
            const float gr = S.g[r], br = S.beta[r];
            for (int j0 = 0; j0 < kC; j0 += 16) {
                float v[16];
                tmem_ld16(tbase + lane_base + kColD1 + j0, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int j = j0 + i;
                    const bool keep = isP ? (j <= r) : (j < r);
                    float x = keep ? v[i] : 0.f;
                    if (MODE == LDN_GDN && keep) x *= expf(gr - S.g[j]);
                    if (!isP) x *= br;
                    v[i] = x;
                }
                if (isP) st_row16(PI, r, j0, v);
                else
#pragma unroll
                    for (int i = 0; i < 16; ++i) Af[r * 65 + j0 + i] = v[i];
            }
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- T = (I + A)^{-1}: diagonal 16x16 blocks by column substitution
        if (tid < 64) {
            const int blk = tid >> 4, col = tid & 15, o = blk * 16;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = (r == col) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < r; ++j) acc -= Af[(o + r) * 65 + o + j] * x[j];
                x[r] = (r < col) ? 0.f : acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tf[(o + r) * 65 + o + col] = x[r];
        }
        // zero the strictly-upper blocks of T
        for (int e = tid; e < 64 * 64; e += kThreads) {
            const int r = e >> 6, j = e & 63;
            if ((j >> 4) > (r >> 4)) Tf[r * 65 + j] = 0.f;
        }
        __syncthreads();
        // off-diagonal blocks by block distance d: T_{i+d,i} = -T_{i+d,i+d} sum_k A_{i+d,k} T_{k,i}
        for (int d = 1; d < 4; ++d) {
            const int nb = 4 - d;
            for (int e = tid; e < nb * 256; e += kThreads) {
                const int i = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
                const int ro = (i + d) * 16, co = i * 16;
                float acc = 0.f;
                for (int kb = i; kb < i + d; ++kb)
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)
                        acc += Af[(ro + rr) * 65 + kb * 16 + kk] * Tf[(kb * 16 + kk) * 65 + co + cc];
                Xs[e] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nb * 256; e += kThreads) {
                const int i = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
                const int ro = (i + d) * 16, co = i * 16;
                float acc = 0.f;
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) acc -= Tf[(ro + rr) * 65 + ro + kk] * Xs[(i << 8) + kk * 16 + cc];
                Tf[(ro + rr) * 65 + co + cc] = acc;
            }
            __syncthreads();
        }

        // ---- [Tu | Tw] as the MN-major right operand of MMA2 (row j of T scaled by column factors)
        {
            const int j = tid & 63;
            const bool w = tid >= 64;
            uint8_t *blk = TT + (w ? 8192 : 0);
            for (int n0c = 0; n0c < kC; n0c += 16) {
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int n = n0c + i;
                    const float f = S.beta[n] * (w ? S.eg[n] : 1.f);
                    v[i] = Tf[j * 65 + n] * f;
                }
                st_row16(blk, j, n0c, v);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA2: [P ; I] [Tu | Tw]
        if (tid == 0) {
            tc_fence_after();
            const uint32_t pi_s = smem_u32(PI), tt_s = smem_u32(TT);
            for (int s = 0; s < kC / 16; ++s)
                umma_bf16(tbase + kColDP, kmajor_desc(pi_s, 128, s), mnmajor_desc(tt_s, 64, s), id_mn_n128, s > 0);
            umma_commit(&S.bar_mma);
        }
        if (!wait_mma()) break;

        // ---- AV = [P Tu ; Tu] (own row), AK = [Tw ; -P Tw] (rows swap halves) into TT's buffer
        {
            const bool top = tid < 64;
            const int r = tid & 63;
            for (int j0 = 0; j0 < kC; j0 += 16) {
                float v[16];
                tmem_ld16(tbase + lane_base + kColDP + j0, v);
                tmem_ld_wait();
                st_row16(AV, tid, j0, v);
            }
            __syncthreads();   // every thread has read [Tu | Tw] from TT before it is overwritten
            for (int j0 = 0; j0 < kC; j0 += 16) {
                float v[16];
                tmem_ld16(tbase + lane_base + kColDP + 64 + j0, v);
                tmem_ld_wait();
                if (top) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = -v[i];
                }
                st_row16(TT, top ? 64 + r : r, j0, v);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA3: [P Tu ; Tu] V -> RV ;  MMA4: [Tw ; -P Tw] K -> DK
        if (tid == 0) {
            tc_fence_after();
            const uint32_t av_s = smem_u32(AV), ak_s = smem_u32(TT);
            for (int s = 0; s < kC / 16; ++s)
                umma_bf16(tbase + kColRV, kmajor_desc(av_s, 128, s), mnmajor_desc(v_s, 64, s), id_mn_n64, s > 0);
            for (int s = 0; s < kC / 16; ++s)
                umma_bf16(tbase + kColDK, kmajor_desc(ak_s, 128, s), mnmajor_desc(k_s, 128, s), id_mn_n128, s > 0);
            umma_commit(&S.bar_mma);
        }
        if (!wait_mma()) break;

        // ---- A5 = [Q~ ; -W]:  rows 0-63 of DK hold W, rows 64-127 hold -P W
        {
            const bool top = tid < 64;
            const int r = tid & 63;
            const float er = S.eg[r];
            for (int c0 = 0; c0 < kDK; c0 += 16) {
                float v[16];
                tmem_ld16(tbase + lane_base + kColDK + c0, v);
                tmem_ld_wait();
                uint8_t *blk = A5 + (c0 >> 6) * 16384;
                if (top) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = -v[i];
                    st_row16(blk, 64 + r, c0 & 63, v);
                } else {
                    float qv[16];
                    const uint8_t *qblk = QK + (c0 >> 6) * 16384;
                    ld_row8(qblk, r, c0 & 63, qv);
                    ld_row8(qblk, r, (c0 & 63) + 8, qv + 8);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += er * qv[i];
                    st_row16(blk, r, c0 & 63, v);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA5 (state-dependent): RV += [Q~ ; -W] H0
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a5_s = smem_u32(A5), hb_s = smem_u32(HB);
            for (int s = 0; s < kDK / 16; ++s)
                umma_bf16(tbase + kColRV, kmajor_desc(a5_s, 128, s), mnmajor_desc(hb_s, 128, s), id_mn_n64, 1);
            umma_commit(&S.bar_mma);
        }
        if (!wait_mma()) break;

        // ---- O rows to global; U~ = Diag(e^{g_C - g}) U into UB
        {
            const bool top = tid < 64;
            const int r = tid & 63;
            const float f = S.egc[r];
            for (int n = 0; n < kDVS; n += 16) {
                float v[16];
                tmem_ld16(tbase + lane_base + kColRV + n, v);
                tmem_ld_wait();
                if (top) {
                    if (r < L) {
                        __nv_bfloat16 *dst = out + (((size_t)b * T + t0 + r) * H + h) * dv + n0 + n;
                        uint8_t tmp[32];
                        st_bf16x8(tmp, v);
                        st_bf16x8(tmp + 16, v + 8);
                        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<uint4 *>(tmp);
                        *reinterpret_cast<uint4 *>(dst + 8) = *reinterpret_cast<uint4 *>(tmp + 16);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= f;
                    st_row16(UB, r, n, v);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA6: K^T U~ -> D6
        if (tid == 0) {
            tc_fence_after();
            const uint32_t ub_s = smem_u32(UB);
            for (int s = 0; s < kC / 16; ++s)
                umma_bf16(tbase + kColD6, mnmajor_desc(k_s, 128, s), mnmajor_desc(ub_s, 64, s), id_amn_n64, s > 0);
            umma_commit(&S.bar_mma);
        }
        if (!wait_mma()) break;
        // this stage's tiles are free: prefetch chunk c + 2 into it
        if (tid == 0 && c + 2 < nchunks) issue_load(c + 2);

        // ---- H1 = e^{g_C} H0 + D6 (row tid), bf16 copy for the next chunk
#pragma unroll
        for (int n = 0; n < kDVS; n += 16) {
            float v[16];
            tmem_ld16(tbase + lane_base + kColD6 + n, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                Hreg[n + i] = gC * Hreg[n + i] + v[i];
                v[i] = Hreg[n + i];
            }
            st_row16(HB, tid, n, v);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    __syncthreads();
    if (S.fail) {
        if (tid == 0) {
            atomicOr(status, 1 << LDN_ERR_TIMEOUT);
            // Give outstanding TMA loads and MMAs a bounded chance to land
            // before the shared memory and TMEM are released.
            for (int st = 0; st < 2; ++st)
                if (pending[st] >= 0) mbar_wait(&S.bar_load[st], (pending[st] >> 1) & 1, kWaitNs);
            mbar_wait(&S.bar_mma, mma_phase ^ 1u, kWaitNs);
        }
    } else if (S_final) {
        float *dst = S_final + ((size_t)unit * kDK + tid) * dv + n0;
#pragma unroll
        for (int n = 0; n < kDVS; n += 4)
            *reinterpret_cast<float4 *>(dst + n) = make_float4(Hreg[n], Hreg[n + 1], Hreg[n + 2], Hreg[n + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

bool chunk_tc_supported(const ChunkArgs &a)
{
    return a.dtype == LDN_BF16 && a.dk == kDK && a.dv % kDVS == 0 && a.chunk == kC &&
           (a.mode == LDN_DELTANET || a.mode == LDN_GDN);
}

cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st)
{
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16_4d(&tq, a.q, kDK, a.H, a.T, a.B, 64, kC) ||
        !make_tmap_bf16_4d(&tk, a.k, kDK, a.H, a.T, a.B, 64, kC) ||
        !make_tmap_bf16_4d(&tv, a.v, a.dv, a.H, a.T, a.B, 64, kC))
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)((long long)a.B * a.H * (a.dv / kDVS));
    auto kern = a.mode == LDN_GDN ? chunk_tc_kernel<LDN_GDN> : chunk_tc_kernel<LDN_DELTANET>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, a.beta, a.gate, a.S0, (__nv_bfloat16 *)a.out, a.S_final,
                                             a.T, a.H, a.dv, a.status);
    return cudaGetLastError();
}

}  // namespace ldn
