// Chunkwise backward of DeltaNet and Gated DeltaNet (scalar decay) on the tensor cores:
// warp-level fp16 MMAs (mma.sync m16n8k16, ldmatrix operands) with fp32 accumulation, for
// bf16 inputs with dk = dv = 128 and chunks of 64 tokens.
//
// The pages state the recurrence per token (linear-attention notes, Sec. 2.3-2.4) and describe
// a first-order backward that keeps the state history, checked in fp64 (the method-sources
// page, KDA entry).  The chunk form of the derivative is derived here.  In H = S^T ([dk][dv]),
// for a chunk of rows r with incoming state H0, g the inclusive prefix of the log-decay,
// Gamma_rj = e^{g_r - g_j}, ge = e^{g}, gc = e^{g_last - g} and gamma = e^{g_last}, the forward
// is
//   A = strict_tril(Diag(beta) (K K^T * Gamma)),   T = (I + A)^-1,
//   W = T Diag(beta ge) K,   U' = T Diag(beta) V,   U = U' - W H0,
//   P = tril(Q K^T * Gamma),   O = Diag(ge) Q H0 + P U,   H_C = gamma H0 + K^T Diag(gc) U,
// and, given dO and dH_C (written dH' below), its reverse is
//   dU  = Diag(gc) K dH' + P^T dO,       dW = -dU H0^T,
//   dH0 = gamma dH' + Q^T Diag(ge) dO - W^T dU                      (the chain, kernel 1)
//   dP  = tril(dO U^T),   dT = dU Vb^T + dW Kb^T  (Vb = Diag(beta) V, Kb = Diag(beta ge) K),
//   dA  = strict_tril(-T^T dT T^T),   E' = dA * Gamma,   F = dP * Gamma,
//   dQ  = Diag(ge) dO H0^T + F K,
//   dK  = Diag(beta) E' K + E'^T Diag(beta) K + F^T Q + Diag(gc) U dH'^T + Diag(beta ge) T^T dW,
//   dV  = Diag(beta) T^T dU,
//   dbeta = rowsum(E' * K K^T) + rowsum(V * T^T dU) + ge rowsum(K * T^T dW),
//   dg  = rowsum(R) - colsum(R) + ge (rowsum(Q * dO H0^T) + beta rowsum(K * T^T dW))
//         - gc rowsum(K * U dH'^T), and at the last row also + sum(gc rowsum(K * U dH'^T))
//         + gamma sum(H0 * dH'), with R = Diag(beta) E' * K K^T + F * Q K^T;
//   the log-decay input's gradient is the reverse cumulative sum of dg within the chunk.
// (Padded rows past the end of the sequence are zero and carry no decay.)
//
// The backward is three steps after a forward pass that stores the state entering every
// chunk (the pre-solved forward kernel with chunk_states) and X = [P T ; T] of every chunk
// (the pre-solved variant's solve, whose rows 64..127 are T):
//   1. bwd_prep_kernel: one CTA per (b, h, chunk), all in parallel, forms P, -W and the two
//      chain-independent terms of the state gradient's recursion, dH0 = M dH' + Bc.
//   2. bwd_chain_kernel: one CTA per (b, h, 64-wide slice of dv) walks the chunks in reverse,
//      one product per chunk, and carries dH in fp32; it stores the dH' of every chunk.
//   3. bwd_chunk_kernel: one CTA per (b, h, chunk), all in parallel, forms every gradient of
//      the chunk from its inputs, T, P, -W, H0 and dH'.
// Arithmetic: products on fp16 operands (2^-11) with fp32 accumulation; states, gradients and
// every elementwise step in fp32.  Operands stay in fp16 range when the log-decays are not
// positive (every Gamma, ge, gc <= 1).
#include "ldn_internal.cuh"
#include "sm100_ptx.cuh"
#include "warp_mma.cuh"

namespace ldn {
namespace {
using namespace sm100;
using namespace wmma8;

constexpr int kXBytes = 16384;  // X = [P T ; T] per (b, h, chunk), the swizzled image the solve writes
constexpr int kLdO = kD + 8;    // fp32 row stride of the staged gradient rows (544 B)
constexpr uint64_t kWaitNs = 2000000000ull;   // bound of every wait (2 s)
static_assert(kStateImgLd == kLdW, "the state images are the shared-memory tiles");

// Rows of a staged fp32 [64][kLdO] tile to the token rows of a [.., H, 128] gradient tensor,
// a warp per row (32 x 16 bytes), rows past the sequence skipped.
__device__ __forceinline__ void store_rows(float *__restrict__ dst, const float *src, size_t tok0, int H, int L,
                                           int tid)
{
#pragma unroll 4
    for (int e = tid; e < kC * 32; e += kThreads) {
        const int rr = e >> 5, part = e & 31;
        if (rr < L)
            *reinterpret_cast<float4 *>(dst + (tok0 + (size_t)rr * H) * kD + 4 * part) =
                *reinterpret_cast<const float4 *>(src + rr * kLdO + 4 * part);
    }
}

// T of a chunk from the rows 64..127 of the solve's X image (128-byte swizzled K-major fp16:
// the 16-byte group p of row `row` holds columns 8 ((p ^ row) & 7) ..), copied raw to shared
// memory, as fp16 tiles of stride kLdN: T itself (optional), T Diag(s1) and (optional)
// T Diag(s2), s1 / s2 per column.
__device__ __forceinline__ void load_t(const uint8_t *Xt, __half *t, __half *t1, const float *s1, __half *t2,
                                       const float *s2, int tid)
{
    uint4 u[kC * 8 / kThreads];
#pragma unroll
    for (int i = 0; i < kC * 8 / kThreads; ++i) u[i] = reinterpret_cast<const uint4 *>(Xt)[tid + kThreads * i];
#pragma unroll
    for (int i = 0; i < kC * 8 / kThreads; ++i) {
        const int e = tid + kThreads * i, j = e >> 3, c8 = 8 * (((e & 7) ^ (64 + j)) & 7);
        const __half2 *h2 = reinterpret_cast<const __half2 *>(&u[i]);
        __half2 a[4], b2[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(h2[q]);
            a[q] = __floats2half2_rn(f.x * s1[c8 + 2 * q], f.y * s1[c8 + 2 * q + 1]);
            if (t2) b2[q] = __floats2half2_rn(f.x * s2[c8 + 2 * q], f.y * s2[c8 + 2 * q + 1]);
        }
        if (t) *reinterpret_cast<uint4 *>(t + j * kLdN + c8) = u[i];
        *reinterpret_cast<uint4 *>(t1 + j * kLdN + c8) = *reinterpret_cast<uint4 *>(a);
        if (t2) *reinterpret_cast<uint4 *>(t2 + j * kLdN + c8) = *reinterpret_cast<uint4 *>(b2);
    }
}

// Per-chunk gate data: the inclusive log-decay prefix of the chunk's rows (warp 0; rows past
// the sequence and DeltaNet add nothing), beta.
template <int MODE>
__device__ __forceinline__ void chunk_gates(const float *__restrict__ beta, const float *__restrict__ gate,
                                            size_t tok0, int H, int L, int lane, float *sbeta, float *sg)
{
    for (int rr = lane; rr < kC; rr += 32) sbeta[rr] = rr < L ? __ldg(beta + tok0 + (size_t)rr * H) : 0.f;
    float a0 = 0.f, a1 = 0.f;
    if (MODE == LDN_GDN) {
        const int r0 = 2 * lane, r1 = r0 + 1;
        a0 = r0 < L ? __ldg(gate + tok0 + (size_t)r0 * H) : 0.f;
        a1 = r1 < L ? __ldg(gate + tok0 + (size_t)r1 * H) : 0.f;
    }
    float incl = a0 + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    sg[2 * lane] = incl - a1;
    sg[2 * lane + 1] = incl;
}

// =====================================================================================
// Kernel 1: the chain-independent products of every chunk, one CTA per (b, h, chunk), all in
// parallel.  The reverse chain of the state gradient,
//   dH0 = gamma dH' + Q^T Diag(ge) dO - W^T dU,   dU = Diag(gc) K dH' + P^T dO,
// is affine in dH':  dH0 = M dH' + Bc with
//   M  = gamma I - W^T Diag(gc) K        [dk x dk],
//   Bc = (Diag(ge) Q - P W)^T dO         [dk x dv]   (Diag(ge) Q - P W is the forward's Q~),
// so the serial pass is one product per chunk.  Stored per chunk as fp16 images laid out as
// their consumers' shared-memory tiles: P [64][72] and -W [64][136] (the per-chunk kernel's
// operands), M and Bc [128][136] (the chain's).
constexpr size_t kPImg = kC * kLdN * 2;      // 9216 B
constexpr size_t kWImg = kC * kLdW * 2;      // 17408 B
constexpr size_t kMImg = kStateImgBytes;     // 34816 B, also Bc's

struct PrepSmem {
    static constexpr int q = 0;                       // Q, then Q~ [64][136] fp16
    static constexpr int k = q + kC * kLdW * 2;       // K, then Diag(gc) K
    static constexpr int dO = k + kC * kLdW * 2;      // dO
    static constexpr int tk = dO + kC * kLdW * 2;     // T Diag(beta ge) [64][72]
    static constexpr int p = tk + kC * kLdN * 2;      // T's raw rows, then P [64][72]
    static constexpr int w = p + kC * kLdN * 2;       // W [64][136]
    static constexpr int small = w + kC * kLdW * 2;   // beta, g, ge, gc, beta ge
    static constexpr int bytes = small + 5 * kC * 4;
    static_assert(2 * bytes <= 232448, "two CTAs per SM");
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 2)
bwd_prep_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                const float *__restrict__ beta, const float *__restrict__ gate,
                const __nv_bfloat16 *__restrict__ dout, const uint8_t *__restrict__ X, __half *__restrict__ Pimg,
                __half *__restrict__ Wimg, __half *__restrict__ Mimg, __half *__restrict__ Bimg, int T, int H)
{
    extern __shared__ __align__(16) uint8_t smp[];
    using SM = PrepSmem;
    __half *Qs = reinterpret_cast<__half *>(smp + SM::q), *Ks = reinterpret_cast<__half *>(smp + SM::k);
    __half *dOs = reinterpret_cast<__half *>(smp + SM::dO), *TKs = reinterpret_cast<__half *>(smp + SM::tk);
    __half *Ps = reinterpret_cast<__half *>(smp + SM::p), *Ws = reinterpret_cast<__half *>(smp + SM::w);
    float *sbeta = reinterpret_cast<float *>(smp + SM::small), *sg = sbeta + kC, *sge = sg + kC, *sgc = sge + kC;
    float *sbge = sgc + kC;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = (T + kC - 1) / kC;
    const size_t chunk = blockIdx.x;
    const int unit = blockIdx.x / nch, c = blockIdx.x % nch;
    const int b = unit / H, h = unit % H;
    const int t0 = c * kC, L = min(kC, T - t0);
    const size_t tok0 = ((size_t)b * T + t0) * H + h;

    // ---- 0: T's rows of X (raw, into P's place, cp.async); q, k, dO rows to fp16; gates
    for (int e = tid; e < kC * 8; e += kThreads)
        cp_async16(Ps + 8 * e, X + chunk * kXBytes + 8192 + 16 * e, 16u);
    cp_async_commit();
    {
        const __nv_bfloat16 *const src[3] = {q, k, dout};
        __half *const dst[3] = {Qs, Ks, dOs};
        load_tiles_f16<3>(src, dst, tok0, H, L, tid);
    }
    if (warp == 0) chunk_gates<MODE>(beta, gate, tok0, H, L, lane, sbeta, sg);
    cp_async_wait<0>();
    __syncthreads();
    for (int rr = tid; rr < kC; rr += kThreads) {
        const float gl = sg[kC - 1];
        sge[rr] = MODE == LDN_GDN ? expf(sg[rr]) : 1.f;
        sgc[rr] = MODE == LDN_GDN ? expf(gl - sg[rr]) : 1.f;
        sbge[rr] = sbeta[rr] * sge[rr];
    }
    __syncthreads();
    load_t(reinterpret_cast<const uint8_t *>(Ps), nullptr, TKs, sbge, nullptr, nullptr, tid);
    __syncthreads();
    // ---- 1: P = tril(Q K^T * Gamma); W = T Diag(beta ge) K
    {
        const Op op[1] = {{Qs, kLdW, false, Ks, kLdW, true, kD}};
        cta_mma<kC, kC>(op, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = acc_row(lane, m0, e), jj = acc_col(lane, c0, nt, e);
                    const float gm = MODE == LDN_GDN ? expf(sg[rr] - sg[jj]) : 1.f;
                    Ps[rr * kLdN + jj] = __float2half_rn(jj <= rr ? acc[nt][e] * gm : 0.f);
                }
        });
        const Op ow[1] = {{TKs, kLdN, false, Ks, kLdW, false, kC}};
        cta_mma<kC, kD>(ow, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    *reinterpret_cast<__half2 *>(Ws + rr * kLdW + cc) = __floats2half2_rn(acc[nt][e], acc[nt][e + 1]);
                }
        });
    }
    __syncthreads();
    // ---- 2: the P and -W images; Q~ = Diag(ge) Q - P W (in Q's place); Diag(gc) K (in K's place)
    {
        const uint4 *ps = reinterpret_cast<const uint4 *>(Ps);
        uint4 *pd = reinterpret_cast<uint4 *>(Pimg + chunk * (kPImg / 2));
        for (int e = tid; e < (int)(kPImg / 16); e += kThreads) pd[e] = ps[e];
        const uint4 *ws = reinterpret_cast<const uint4 *>(Ws);
        uint4 *wd = reinterpret_cast<uint4 *>(Wimg + chunk * (kWImg / 2));
        for (int e = tid; e < (int)(kWImg / 16); e += kThreads) {
            uint4 u = ws[e];
            u.x ^= 0x80008000u;   // fp16 sign bits: -W
            u.y ^= 0x80008000u;
            u.z ^= 0x80008000u;
            u.w ^= 0x80008000u;
            wd[e] = u;
        }
        const Op o1[1] = {{Ps, kLdN, false, Ws, kLdW, false, kC}};
        cta_mma<kC, kD>(o1, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    __half2 *qp = reinterpret_cast<__half2 *>(Qs + rr * kLdW + cc);
                    const float2 qv = __half22float2(*qp);
                    *qp = __floats2half2_rn(sge[rr] * qv.x - acc[nt][e], sge[rr] * qv.y - acc[nt][e + 1]);
                }
        });
        if (MODE == LDN_GDN)
            for (int e = tid; e < kC * 16; e += kThreads) {
                const int rr = e >> 4, part = e & 15;
                uint4 *kp = reinterpret_cast<uint4 *>(Ks + rr * kLdW + 8 * part);
                uint4 u = *kp;
                __half2 *h2 = reinterpret_cast<__half2 *>(&u);
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float2 f = __half22float2(h2[x]);
                    h2[x] = __floats2half2_rn(f.x * sgc[rr], f.y * sgc[rr]);
                }
                *kp = u;
            }
    }
    __syncthreads();
    // ---- 3: Bc = Q~^T dO and M = gamma I - W^T Diag(gc) K, each in two 128 x 64 halves staged
    //      in the place of T Diag(beta ge) and P (read by nobody now; one [128][72] tile) and
    //      copied to the images as 16-byte row pieces
    const float gam = MODE == LDN_GDN ? expf(sg[kC - 1]) : 1.f;
    __half *stg = TKs;
    static_assert(PrepSmem::p - PrepSmem::tk == kC * kLdN * 2 && 2 * kC * kLdN == kD * kLdN, "staging tile");
#pragma unroll 1
    for (int x = 0; x < 4; ++x) {
        const int hv = x & 1;
        const bool is_m = x >= 2;
        __half *img = (is_m ? Mimg : Bimg) + chunk * (kMImg / 2) + 64 * hv;
        const Op ob[1] = {{Qs, kLdW, true, dOs + 64 * hv, kLdW, false, kC}};
        const Op om[1] = {{Ws, kLdW, true, Ks + 64 * hv, kLdW, false, kC}};
        cta_mma<kD, 64>(is_m ? om : ob, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e), gc = cc + 64 * hv;
                    const float d0 = is_m && rr == gc ? gam : 0.f, d1 = is_m && rr == gc + 1 ? gam : 0.f;
                    *reinterpret_cast<__half2 *>(stg + rr * kLdN + cc) =
                        is_m ? __floats2half2_rn(d0 - acc[nt][e], d1 - acc[nt][e + 1])
                             : __floats2half2_rn(acc[nt][e], acc[nt][e + 1]);
                }
        });
        __syncthreads();
#pragma unroll
        for (int e = tid; e < kD * 8; e += kThreads)
            *reinterpret_cast<uint4 *>(img + (e >> 3) * kStateImgLd + 8 * (e & 7)) =
                *reinterpret_cast<const uint4 *>(stg + (e >> 3) * kLdN + 8 * (e & 7));
        __syncthreads();
    }
}

// =====================================================================================
// Kernel 2: the chain dH0 = M dH' + Bc, chunks in reverse, one CTA per (b, h, 64-wide slice
// of dv), dH in fp32 registers (the warp owns the same 16 x 16 tiles of the 128 x 64 slice
// in every chunk); M and the Bc slice of the next chunk load by cp.async under the current
// product.  The fp16 state image dHs[c] receives the dH' of chunk c (the gradient at the
// state it leaves); dS0 the gradient at S0.
struct ChainSmem {
    static constexpr int m = 0;                         // M [2][128][136] fp16 (double buffer)
    static constexpr int bc = m + 2 * kD * kLdW * 2;    // Bc slice [2][128][72]
    static constexpr int dh = bc + 2 * kD * kLdN * 2;   // dH' slice [128][72]
    static constexpr int bytes = dh + kD * kLdN * 2;
};

__device__ __forceinline__ void chain_prefetch(uint8_t *smc, int buf, const __half *__restrict__ Mimg,
                                               const __half *__restrict__ Bimg, size_t chunk, int n0, int tid)
{
    using SM = ChainSmem;
    const uint8_t *ms = reinterpret_cast<const uint8_t *>(Mimg + chunk * (kMImg / 2));
    uint8_t *md = smc + SM::m + buf * (kD * kLdW * 2);
    for (int e = tid; e < (int)(kMImg / 16); e += kThreads) cp_async16(md + 16 * e, ms + 16 * e, 16u);
    const __half *bs = Bimg + chunk * (kMImg / 2) + n0;
    __half *bd = reinterpret_cast<__half *>(smc + SM::bc + buf * (kD * kLdN * 2));
    for (int e = tid; e < kD * 8; e += kThreads)
        cp_async16(bd + (e >> 3) * kLdN + 8 * (e & 7), bs + (e >> 3) * kStateImgLd + 8 * (e & 7), 16u);
    cp_async_commit();
}

__global__ void __launch_bounds__(kThreads, 1)
bwd_chain_kernel(const __half *__restrict__ Mimg, const __half *__restrict__ Bimg,
                 const float *__restrict__ dS_final, __half *__restrict__ dHs, float *__restrict__ dS0, int T,
                 int H, int dv)
{
    extern __shared__ __align__(16) uint8_t smc[];
    using SM = ChainSmem;
    __half *dHh = reinterpret_cast<__half *>(smc + SM::dh);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slices = dv / 64, unit = blockIdx.x / slices, n0 = (blockIdx.x % slices) * 64;
    const int nch = (T + kC - 1) / kC;
    (void)H;

    // dH' of the last chunk: dS_final (or zero); tile i of this warp: rows / columns of the
    // accumulator layout (M = 128 dk rows, N = 64 columns: 32 tiles, 4 per warp)
    float dh[4][2][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int2 og = tile_origin<kD, 64>(warp, i);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int rr = acc_row(lane, og.x, e), cc = acc_col(lane, og.y, nt, e);
                dh[i][nt][e] = dS_final ? dS_final[((size_t)unit * kD + rr) * dv + n0 + cc] : 0.f;
            }
    }
    chain_prefetch(smc, (nch - 1) & 1, Mimg, Bimg, (size_t)unit * nch + nch - 1, n0, tid);
    for (int c = nch - 1; c >= 0; --c) {
        const int buf = c & 1;
        const __half *Ms = reinterpret_cast<const __half *>(smc + SM::m + buf * (kD * kLdW * 2));
        const __half *Bs = reinterpret_cast<const __half *>(smc + SM::bc + buf * (kD * kLdN * 2));
        // dH' (fp16): the product's operand and the chunk's state-gradient image
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int2 og = tile_origin<kD, 64>(warp, i);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, og.x, e), cc = acc_col(lane, og.y, nt, e);
                    *reinterpret_cast<__half2 *>(dHh + rr * kLdN + cc) = __floats2half2_rn(dh[i][nt][e], dh[i][nt][e + 1]);
                }
        }
        if (c > 0) {   // the other buffer was last read before the previous chunk's closing barrier
            chain_prefetch(smc, buf ^ 1, Mimg, Bimg, (size_t)unit * nch + c - 1, n0, tid);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        {
            __half *img = dHs + ((size_t)unit * nch + c) * (kStateImgBytes / 2) + n0;
#pragma unroll
            for (int e = tid; e < kD * 8; e += kThreads)
                *reinterpret_cast<uint4 *>(img + (e >> 3) * kStateImgLd + 8 * (e & 7)) =
                    *reinterpret_cast<const uint4 *>(dHh + (e >> 3) * kLdN + 8 * (e & 7));
        }
        // ---- dH0 = M dH' + Bc
        const Op op[1] = {{Ms, kLdW, false, dHh, kLdN, false, kD}};
        cta_mma<kD, 64>(op, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    const float2 bv = __half22float2(*reinterpret_cast<const __half2 *>(Bs + rr * kLdN + cc));
                    dh[i][nt][e] = acc[nt][e] + bv.x;
                    dh[i][nt][e + 1] = acc[nt][e + 1] + bv.y;
                }
        });
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int2 og = tile_origin<kD, 64>(warp, i);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int rr = acc_row(lane, og.x, e), cc = acc_col(lane, og.y, nt, e);
                *reinterpret_cast<float2 *>(dS0 + ((size_t)unit * kD + rr) * dv + n0 + cc) =
                    make_float2(dh[i][nt][e], dh[i][nt][e + 1]);
            }
    }
}

// =====================================================================================
// Kernel 3: every chunk's gradients, one CTA per (b, h, chunk).  Shared-memory plan (fp16
// tiles; buffers are reused once their last reader is past):
//   Q, K, V, dO [64][136] (dO's place takes dW; V and dO's together the staged dK rows),
//   H0 and dH' [128][136] (their places the staged dV and dQ rows), T, X1 = T^T dT (then
//   E = Diag(beta) E'), T Diag(beta) (then dT, then E'), P (then F) [64][72], -W (then dU)
//   and U (T's raw rows first) [64][136], small vectors.
struct ChunkSmem {
    static constexpr int q = 0;
    static constexpr int k = q + kC * kLdW * 2;
    static constexpr int v = k + kC * kLdW * 2;
    static constexpr int dO = v + kC * kLdW * 2;          // then dW
    static constexpr int h0 = dO + kC * kLdW * 2;         // [128][136]; then dV fp32 [64][136]
    static constexpr int dh = h0 + kD * kLdW * 2;         // [128][136]; then dQ fp32 [64][136]
    static constexpr int t = dh + kD * kLdW * 2;
    static constexpr int tk = t + kC * kLdN * 2;          // X1; E
    static constexpr int tv = tk + kC * kLdN * 2;         // T Diag(beta); dT; E'
    static constexpr int p = tv + kC * kLdN * 2;          // P; F
    static constexpr int w = p + kC * kLdN * 2;           // -W; dU
    static constexpr int u = w + kC * kLdW * 2;           // T's raw rows; U
    static constexpr int small = u + kC * kLdW * 2;       // beta, g, ge, gc, beta ge, 8 slots, 5 x [8][64] parts
    static constexpr int bar = small + (5 * kC + 8 + 5 * kWarps * kC) * 4;   // mbarrier of the bulk copies
    static constexpr int bytes = bar + 8;
    static_assert(bytes <= 232448, "shared memory plan exceeds 227 KB");
    static_assert(kC * kLdO * 4 <= kD * kLdW * 2 && kC * kLdO * 4 == 2 * kC * kLdW * 2,
                  "dV / dQ fit a state tile, dK the V and dO tiles");
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
bwd_chunk_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                 const __nv_bfloat16 *__restrict__ v, const float *__restrict__ beta,
                 const float *__restrict__ gate, const __nv_bfloat16 *__restrict__ dout,
                 const uint8_t *__restrict__ X, const __half *__restrict__ Hs, const __half *__restrict__ dHs,
                 const __half *__restrict__ Pimg, const __half *__restrict__ Wimg,
                 float *__restrict__ dq, float *__restrict__ dk_out, float *__restrict__ dv_out,
                 float *__restrict__ dbeta, float *__restrict__ dgate, int *status, int T, int H)
{
    extern __shared__ __align__(16) uint8_t smk[];
    using SM = ChunkSmem;
    __half *Qs = reinterpret_cast<__half *>(smk + SM::q), *Ks = reinterpret_cast<__half *>(smk + SM::k);
    __half *Vs = reinterpret_cast<__half *>(smk + SM::v), *dOs = reinterpret_cast<__half *>(smk + SM::dO);
    __half *H0s = reinterpret_cast<__half *>(smk + SM::h0), *dHh = reinterpret_cast<__half *>(smk + SM::dh);
    __half *Ts = reinterpret_cast<__half *>(smk + SM::t), *TKs = reinterpret_cast<__half *>(smk + SM::tk);
    __half *TVs = reinterpret_cast<__half *>(smk + SM::tv), *Ps = reinterpret_cast<__half *>(smk + SM::p);
    __half *Ws = reinterpret_cast<__half *>(smk + SM::w), *Us = reinterpret_cast<__half *>(smk + SM::u);
    __half *dWs = dOs, *dUs = Ws, *X1s = TKs, *dTs = TVs, *Fs = Ps, *Es = TKs, *Eps = TVs;
    float *dVo = reinterpret_cast<float *>(smk + SM::h0), *dQo = reinterpret_cast<float *>(smk + SM::dh);
    float *dKo = reinterpret_cast<float *>(smk + SM::v);
    float *sbeta = reinterpret_cast<float *>(smk + SM::small), *sg = sbeta + kC, *sge = sg + kC, *sgc = sge + kC;
    float *sbge = sgc + kC;        // beta ge
    float *red = sbge + kC;        // [8] per-warp parts of sum(H0 * dH')
    // per-warp partial sums [8][64] (each written by its own warp in program order, summed over
    // the warps in a fixed order at the end: the result does not depend on scheduling)
    float *p_dge = red + 8;        // rowsum(Q * dO H0^T) + beta rowsum(K * T^T dW)  (then times ge)
    float *p_dgc = p_dge + kWarps * kC;   // rowsum(K * U dH'^T)
    float *p_db = p_dgc + kWarps * kC;    // dbeta
    float *p_dgr = p_db + kWarps * kC;    // rowsum(R)
    float *p_dgk = p_dgr + kWarps * kC;   // -colsum(R)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *pw_dge = p_dge + warp * kC, *pw_dgc = p_dgc + warp * kC, *pw_db = p_db + warp * kC;
    float *pw_dgr = p_dgr + warp * kC, *pw_dgk = p_dgk + warp * kC;
    const int nch = (T + kC - 1) / kC;
    const int unit = blockIdx.x / nch, c = blockIdx.x % nch;
    const int b = unit / H, h = unit % H;
    const int t0 = c * kC, L = min(kC, T - t0);
    const size_t tok0 = ((size_t)b * T + t0) * H + h;

    // ---- 0: inputs.  H0 and dH' (the fp16 state images), P and -W (the prep kernel's images),
    //      all in the tiles' layout, and T's rows of X (raw, into U's place) by bulk copies;
    //      meanwhile q, k, v, dO rows to fp16 (sixteen 16-byte loads per thread in flight)
    uint64_t *bar = reinterpret_cast<uint64_t *>(smk + SM::bar);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, (uint32_t)(2 * kStateImgBytes + kPImg + kWImg) + 8192u);
        const size_t chunk = (size_t)unit * nch + c;
        bulk_load(H0s, Hs + chunk * (kStateImgBytes / 2), (uint32_t)kStateImgBytes, bar);
        bulk_load(dHh, dHs + chunk * (kStateImgBytes / 2), (uint32_t)kStateImgBytes, bar);
        bulk_load(Ps, Pimg + chunk * (kPImg / 2), (uint32_t)kPImg, bar);
        bulk_load(Ws, Wimg + chunk * (kWImg / 2), (uint32_t)kWImg, bar);
        bulk_load(Us, X + chunk * kXBytes + 8192, 8192u, bar);   // T's rows, raw
    }
    {
        const __nv_bfloat16 *const src[4] = {q, k, v, dout};
        __half *const dst[4] = {Qs, Ks, Vs, dOs};
        load_tiles_f16<4>(src, dst, tok0, H, L, tid);
    }
    if (warp == 0) chunk_gates<MODE>(beta, gate, tok0, H, L, lane, sbeta, sg);
    for (int e = tid; e < 5 * kWarps * kC; e += kThreads) p_dge[e] = 0.f;
    __syncthreads();   // (also orders the barrier's initialisation before the waits)
    if (!__syncthreads_and(mbar_wait(bar, 0, kWaitNs))) {
        // the copies did not land (in some thread's view): report, give them a last bounded
        // wait, leave the chunk (every thread, the vote being the block's)
        if (tid == 0) atomicOr(status, 1 << LDN_ERR_TIMEOUT);
        mbar_wait(bar, 0, kWaitNs / 4);
        return;
    }
    // sum(H0 * dH') (the decay gradient's gamma term) from the fp16 tiles
    float hdh = 0.f;
#pragma unroll 4
    for (int e = tid; e < kD * 16; e += kThreads) {
        const int rr = e >> 4, part = e & 15;
        const uint4 a = *reinterpret_cast<const uint4 *>(H0s + rr * kLdW + 8 * part);
        const uint4 d = *reinterpret_cast<const uint4 *>(dHh + rr * kLdW + 8 * part);
        const __half2 *a2 = reinterpret_cast<const __half2 *>(&a), *d2 = reinterpret_cast<const __half2 *>(&d);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const float2 fa = __half22float2(a2[x]), fd = __half22float2(d2[x]);
            hdh += fa.x * fd.x + fa.y * fd.y;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hdh += __shfl_xor_sync(0xffffffffu, hdh, o);
    if (lane == 0) red[warp] = hdh;
    for (int rr = tid; rr < kC; rr += kThreads) {
        const float gl = sg[kC - 1];
        sge[rr] = MODE == LDN_GDN ? expf(sg[rr]) : 1.f;
        sgc[rr] = MODE == LDN_GDN ? expf(gl - sg[rr]) : 1.f;
        sbge[rr] = sbeta[rr] * sge[rr];
    }
    __syncthreads();
    load_t(reinterpret_cast<const uint8_t *>(Us), Ts, TVs, sbeta, nullptr, nullptr, tid);
    __syncthreads();
    auto gam_of = [&](int rr, int jj) { return MODE == LDN_GDN ? expf(sg[rr] - sg[jj]) : 1.f; };

    // ---- 2: U = T Diag(beta) V + (-W) H0
    {
        const Op op[2] = {{TVs, kLdN, false, Vs, kLdW, false, kC}, {Ws, kLdW, false, H0s, kLdW, false, kD}};
        cta_mma<kC, kD>(op, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    *reinterpret_cast<__half2 *>(Us + rr * kLdW + cc) = __floats2half2_rn(acc[nt][e], acc[nt][e + 1]);
                }
        });
    }
    __syncthreads();
    // ---- 3: dU = Diag(gc) K dH' + P^T dO  (into W's place)
    {
        float kd[4][2][4];
        const Op o1[1] = {{Ks, kLdW, false, dHh, kLdW, false, kD}};
        cta_mma<kC, kD>(o1, warp, lane, [&](int i, int m0, int, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) kd[i][nt][e] = acc[nt][e] * sgc[acc_row(lane, m0, e)];
        });
        const Op o2[1] = {{Ps, kLdN, true, dOs, kLdW, false, kC}};
        cta_mma<kC, kD>(o2, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    *reinterpret_cast<__half2 *>(dUs + rr * kLdW + cc) =
                        __floats2half2_rn(kd[i][nt][e] + acc[nt][e], kd[i][nt][e + 1] + acc[nt][e + 1]);
                }
        });
    }
    __syncthreads();
    // ---- 4: dQ-hat = dO H0^T (dQ's first part, and rowsum(Q * dQ-hat)); F = tril(dO U^T) * Gamma
    float dqa[4][2][4];   // this warp's dQ tiles (M = 64, N = 128)
    {
        const Op o1[1] = {{dOs, kLdW, false, H0s, kLdW, true, kD}};
        cta_mma<kC, kD>(o1, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
            float rs[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    const float2 qv = __half22float2(*reinterpret_cast<const __half2 *>(Qs + rr * kLdW + cc));
                    rs[e >> 1] += acc[nt][e] * qv.x + acc[nt][e + 1] * qv.y;
                    dqa[i][nt][e] = acc[nt][e] * sge[rr];
                    dqa[i][nt][e + 1] = acc[nt][e + 1] * sge[rr];
                }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float s = row_quad_sum(rs[hh]);
                if ((lane & 3) == 0) pw_dge[m0 + (lane >> 2) + 8 * hh] += s;
            }
        });
        const Op o2[1] = {{dOs, kLdW, false, Us, kLdW, true, kD}};
        cta_mma<kC, kC>(o2, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = acc_row(lane, m0, e), jj = acc_col(lane, c0, nt, e);
                    Fs[rr * kLdN + jj] = __float2half_rn(jj <= rr ? acc[nt][e] * gam_of(rr, jj) : 0.f);
                }
        });
    }
    __syncthreads();
    // ---- 5: dK's part Diag(gc) U dH'^T (and rowsum(K * U dH'^T)); -dW = dU H0^T into dO's place
    float dka[4][2][4];   // this warp's dK tiles
    {
        const Op o1[1] = {{Us, kLdW, false, dHh, kLdW, true, kD}};
        cta_mma<kC, kD>(o1, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
            float rs[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    const float2 kv = __half22float2(*reinterpret_cast<const __half2 *>(Ks + rr * kLdW + cc));
                    rs[e >> 1] += acc[nt][e] * kv.x + acc[nt][e + 1] * kv.y;
                    dka[i][nt][e] = acc[nt][e] * sgc[rr];
                    dka[i][nt][e + 1] = acc[nt][e + 1] * sgc[rr];
                }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float s = row_quad_sum(rs[hh]);
                if ((lane & 3) == 0) pw_dgc[m0 + (lane >> 2) + 8 * hh] += s;
            }
        });
        const Op o2[1] = {{dUs, kLdW, false, H0s, kLdW, true, kD}};
        cta_mma<kC, kD>(o2, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    *reinterpret_cast<__half2 *>(dWs + rr * kLdW + cc) = __floats2half2_rn(-acc[nt][e], -acc[nt][e + 1]);
                }
        });
    }
    __syncthreads();
    // ---- 6: dT = dU V^T Diag(beta) + dW K^T Diag(beta ge)  (into T Diag(beta)'s place)
    {
        const Op o1[1] = {{dUs, kLdW, false, Vs, kLdW, true, kD}};
        const Op o2[1] = {{dWs, kLdW, false, Ks, kLdW, true, kD}};
        float uv[2][2][4];
        cta_mma<kC, kC>(o1, warp, lane, [&](int i, int, int, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) uv[i][nt][e] = acc[nt][e];
        });
        __syncthreads();   // T Diag(beta) (read by nothing now) is overwritten below
        cta_mma<kC, kC>(o2, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = acc_row(lane, m0, e), jj = acc_col(lane, c0, nt, e);
                    dTs[rr * kLdN + jj] =
                        __float2half_rn(uv[i][nt][e] * sbeta[jj] + acc[nt][e] * sbeta[jj] * sge[jj]);
                }
        });
    }
    __syncthreads();
    // ---- 7: X1 = T^T dT (into T Diag(beta ge)'s place), then dA = strict_tril(-X1 T^T),
    //      E' = dA * Gamma (into dT's place), E = Diag(beta) E' (into X1's place)
    {
        const Op o1[1] = {{Ts, kLdN, true, dTs, kLdN, false, kC}};
        cta_mma<kC, kC>(o1, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = acc_row(lane, m0, e), jj = acc_col(lane, c0, nt, e);
                    X1s[rr * kLdN + jj] = __float2half_rn(acc[nt][e]);
                }
        });
        __syncthreads();
        float da[2][2][4];
        const Op o2[1] = {{X1s, kLdN, false, Ts, kLdN, true, kC}};
        cta_mma<kC, kC>(o2, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = acc_row(lane, m0, e), jj = acc_col(lane, c0, nt, e);
                    da[i][nt][e] = jj < rr ? -acc[nt][e] * gam_of(rr, jj) : 0.f;
                }
        });
        __syncthreads();   // X1 and dT are read: E and E' take their places
        for (int i = 0; i < 2; ++i) {
            const int2 og = tile_origin<kC, kC>(warp, i);
            const int m0 = og.x, c0 = og.y;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = acc_row(lane, m0, e), jj = acc_col(lane, c0, nt, e);
                    Eps[rr * kLdN + jj] = __float2half_rn(da[i][nt][e]);
                    Es[rr * kLdN + jj] = __float2half_rn(da[i][nt][e] * sbeta[rr]);
                }
        }
    }
    __syncthreads();
    // ---- 8: T^T dU -> dV = Diag(beta) T^T dU (and rowsum(V * T^T dU) into dbeta);
    //      T^T dW -> dK part Diag(beta ge) T^T dW (and rowsum(K * T^T dW) into dbeta and dge)
    {
        const Op o1[1] = {{Ts, kLdN, true, dUs, kLdW, false, kC}};
        cta_mma<kC, kD>(o1, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
            float rs[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    const float2 vv = __half22float2(*reinterpret_cast<const __half2 *>(Vs + rr * kLdW + cc));
                    rs[e >> 1] += acc[nt][e] * vv.x + acc[nt][e + 1] * vv.y;
                    *reinterpret_cast<float2 *>(dVo + rr * kLdO + cc) =
                        make_float2(acc[nt][e] * sbeta[rr], acc[nt][e + 1] * sbeta[rr]);
                }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float s = row_quad_sum(rs[hh]);
                if ((lane & 3) == 0) pw_db[m0 + (lane >> 2) + 8 * hh] += s;
            }
        });
        const Op o2[1] = {{Ts, kLdN, true, dWs, kLdW, false, kC}};
        cta_mma<kC, kD>(o2, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
            float rs[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                    const float2 kv = __half22float2(*reinterpret_cast<const __half2 *>(Ks + rr * kLdW + cc));
                    rs[e >> 1] += acc[nt][e] * kv.x + acc[nt][e + 1] * kv.y;
                    dka[i][nt][e] += acc[nt][e] * sbge[rr];
                    dka[i][nt][e + 1] += acc[nt][e + 1] * sbge[rr];
                }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float s = row_quad_sum(rs[hh]);
                if ((lane & 3) == 0) {
                    const int rr = m0 + (lane >> 2) + 8 * hh;
                    pw_db[rr] += sge[rr] * s;
                    pw_dge[rr] += sbeta[rr] * s;
                }
            }
        });
    }
    __syncthreads();
    store_rows(dv_out, dVo, tok0, H, L, tid);
    // ---- 9: dQ += F K; dK += E K + E^T K + F^T Q, with E = Diag(beta) E' (both terms of A's
    //      gradient, A = strict_tril(Diag(beta) (K K^T * Gamma)), carry beta on the row side)
    {
        const Op o1[1] = {{Fs, kLdN, false, Ks, kLdW, false, kC}};
        cta_mma<kC, kD>(o1, warp, lane, [&](int i, int, int, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) dqa[i][nt][e] += acc[nt][e];
        });
        const Op o2[3] = {{Es, kLdN, false, Ks, kLdW, false, kC}, {Es, kLdN, true, Ks, kLdW, false, kC},
                          {Fs, kLdN, true, Qs, kLdW, false, kC}};
        cta_mma<kC, kD>(o2, warp, lane, [&](int i, int, int, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) dka[i][nt][e] += acc[nt][e];
        });
    }
    // dQ and dK rows of this chunk, staged (V, dW, dH' are read by nobody now) and stored whole
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int2 og = tile_origin<kC, kD>(warp, i);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int rr = acc_row(lane, og.x, e), cc = acc_col(lane, og.y, nt, e);
                *reinterpret_cast<float2 *>(dQo + rr * kLdO + cc) = make_float2(dqa[i][nt][e], dqa[i][nt][e + 1]);
                *reinterpret_cast<float2 *>(dKo + rr * kLdO + cc) = make_float2(dka[i][nt][e], dka[i][nt][e + 1]);
            }
    }
    __syncthreads();
    store_rows(dq, dQo, tok0, H, L, tid);
    store_rows(dk_out, dKo, tok0, H, L, tid);
    // ---- 10: K K^T (kept), then Q K^T with, in its epilogue, R = Diag(beta) E' * K K^T + F * Q K^T:
    //       dg += rowsum(R) - colsum(R), dbeta += rowsum(E' * K K^T)
    {
        float kk[2][2][4];
        const Op o1[1] = {{Ks, kLdW, false, Ks, kLdW, true, kD}};
        cta_mma<kC, kC>(o1, warp, lane, [&](int i, int, int, float (&acc)[2][4]) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) kk[i][nt][e] = acc[nt][e];
        });
        const Op o2[1] = {{Qs, kLdW, false, Ks, kLdW, true, kD}};
        cta_mma<kC, kC>(o2, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
            float rsum[2] = {0.f, 0.f}, bsum[2] = {0.f, 0.f}, csum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, m0, e), jj = acc_col(lane, c0, nt, e);
                    const float2 ep = __half22float2(*reinterpret_cast<const __half2 *>(Eps + rr * kLdN + jj));
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(Fs + rr * kLdN + jj));
                    const float b0 = ep.x * kk[i][nt][e], b1 = ep.y * kk[i][nt][e + 1];
                    const float r0 = sbeta[rr] * b0 + f.x * acc[nt][e], r1 = sbeta[rr] * b1 + f.y * acc[nt][e + 1];
                    rsum[e >> 1] += r0 + r1;
                    bsum[e >> 1] += b0 + b1;
                    csum[nt][0] += r0;
                    csum[nt][1] += r1;
                }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float rs = row_quad_sum(rsum[hh]), bs = row_quad_sum(bsum[hh]);
                if ((lane & 3) == 0) {
                    const int rr = m0 + (lane >> 2) + 8 * hh;
                    if (MODE == LDN_GDN) pw_dgr[rr] += rs;
                    pw_db[rr] += bs;
                }
            }
            if (MODE == LDN_GDN) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        float cs = csum[nt][x];
                        cs += __shfl_xor_sync(0xffffffffu, cs, 4);
                        cs += __shfl_xor_sync(0xffffffffu, cs, 8);
                        cs += __shfl_xor_sync(0xffffffffu, cs, 16);
                        if (lane < 4) pw_dgk[c0 + 8 * nt + 2 * lane + x] -= cs;
                    }
            }
        });
    }
    __syncthreads();
    auto sum_warps = [&](const float *part, int rr) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) acc += part[w * kC + rr];
        return acc;
    };
    if (warp == 0) {
        // dbeta; dg per row, then the log-decay input's gradient = reverse cumulative sum
        for (int rr = lane; rr < kC; rr += 32)
            if (rr < L) dbeta[tok0 + (size_t)rr * H] = sum_warps(p_db, rr);
        if (MODE == LDN_GDN) {
            float hd = 0.f;
            for (int i = 0; i < kWarps; ++i) hd += red[i];
            const float gam = expf(sg[kC - 1]);
            const int r0 = 2 * lane, r1 = r0 + 1;
            const float c0 = sum_warps(p_dgc, r0), c1 = sum_warps(p_dgc, r1);
            float d0 = sum_warps(p_dgr, r0) + sum_warps(p_dgk, r0) + sge[r0] * sum_warps(p_dge, r0) - sgc[r0] * c0;
            float d1 = sum_warps(p_dgr, r1) + sum_warps(p_dgk, r1) + sge[r1] * sum_warps(p_dge, r1) - sgc[r1] * c1;
            // the last row also carries gc's and gamma's dependence on g_last
            float gcs = sgc[r0] * c0 + sgc[r1] * c1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) gcs += __shfl_xor_sync(0xffffffffu, gcs, o);
            if (lane == 31) d1 += gcs + gam * hd;
            // reverse cumulative sum over the 64 rows (two per lane)
            float inc = d0 + d1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, inc, o);
                if (lane + o < 32) inc += y;
            }
            // inc = sum over rows >= r0 of d; row r1's suffix = inc - d0
            if (r0 < L) dgate[tok0 + (size_t)r0 * H] = inc;
            if (r1 < L) dgate[tok0 + (size_t)r1 * H] = inc - d0;
        }
    }
}

}  // namespace

bool bwd_chunk_supported(const BwdArgs &a)
{
    // q, k, v and dout are read as 16-byte rows (and through TMA descriptors by the forward pass)
    const bool a16 = (((uintptr_t)a.q | (uintptr_t)a.k | (uintptr_t)a.v | (uintptr_t)a.dout) & 15u) == 0;
    return a.dtype == LDN_BF16 && a.dk == kD && a.dv == kD && (a.mode == LDN_DELTANET || a.mode == LDN_GDN) && a16;
}

// Workspace per (b, h, chunk): the solve's X (16 KB), the state entering and the state
// gradient leaving the chunk (fp16 state images, 34 KB each), the prep kernel's P (9 KB), -W
// (17 KB), M and Bc (34 KB each); and the forward pass's output (bf16).
size_t bwd_chunk_workspace_bytes(int B, int T, int H)
{
    const size_t units = (size_t)B * H, nch = (size_t)(T + kC - 1) / kC;
    return units * nch * (kXBytes + 2 * kStateImgBytes + kPImg + kWImg + 2 * kMImg) + (size_t)B * T * H * kD * 2;
}

cudaError_t launch_backward_chunk(const BwdArgs &a, cudaStream_t s)
{
    const size_t units = (size_t)a.B * a.H, nch = (size_t)(a.T + kC - 1) / kC;
    const size_t nc = units * nch;
    uint8_t *X = reinterpret_cast<uint8_t *>(a.ws);
    __half *Hs = reinterpret_cast<__half *>(X + nc * kXBytes);
    __half *dHs = Hs + nc * (kStateImgBytes / 2);
    __half *Pimg = dHs + nc * (kStateImgBytes / 2);
    __half *Wimg = Pimg + nc * (kPImg / 2);
    __half *Mimg = Wimg + nc * (kWImg / 2);
    __half *Bimg = Mimg + nc * (kMImg / 2);
    void *out = Bimg + nc * (kMImg / 2);
    // forward: the solve and the fused kernel with the chunk states
    ChunkArgs f{a.q, a.k, a.v, a.beta, a.gate, a.S0, out, nullptr, a.B, a.T, a.H, kD, kD, kC, a.mode, a.dtype,
                status_word_ptr()};
    f.chunk_states = Hs;
    if (!f.status) return cudaErrorInvalidValue;
    cudaError_t e = launch_chunk_presolved(f, X, s);
    if (e != cudaSuccess) return e;
    auto k0 = a.mode == LDN_GDN ? bwd_prep_kernel<LDN_GDN> : bwd_prep_kernel<LDN_DELTANET>;
    auto k2 = a.mode == LDN_GDN ? bwd_chunk_kernel<LDN_GDN> : bwd_chunk_kernel<LDN_DELTANET>;
    if ((e = cudaFuncSetAttribute(k0, cudaFuncAttributeMaxDynamicSharedMemorySize, PrepSmem::bytes)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(bwd_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  ChainSmem::bytes)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, ChunkSmem::bytes)) != cudaSuccess)
        return e;
    k0<<<(unsigned)nc, kThreads, PrepSmem::bytes, s>>>(
        (const __nv_bfloat16 *)a.q, (const __nv_bfloat16 *)a.k, a.beta, a.gate, (const __nv_bfloat16 *)a.dout, X,
        Pimg, Wimg, Mimg, Bimg, a.T, a.H);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_chain_kernel<<<(unsigned)(units * (kD / 64)), kThreads, ChainSmem::bytes, s>>>(
        Mimg, Bimg, a.dS_final, dHs, a.dS0, a.T, a.H, kD);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k2<<<(unsigned)nc, kThreads, ChunkSmem::bytes, s>>>(
        (const __nv_bfloat16 *)a.q, (const __nv_bfloat16 *)a.k, (const __nv_bfloat16 *)a.v, a.beta, a.gate,
        (const __nv_bfloat16 *)a.dout, X, Hs, dHs, Pimg, Wimg, a.dq, a.dk_out, a.dv_out, a.dbeta, a.dgate, f.status,
        a.T, a.H);
    return cudaGetLastError();
}

}  // namespace ldn
