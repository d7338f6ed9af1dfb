// Residual Linear Attention (RLA) and Residual DeltaNet (RDN) forward in chunk form, on
// warp-level fp16 MMAs (mma.sync, fp32 accumulation), for bf16 inputs with dk = dv = 128.
//
// Per token ("Residual Linear Attention" reading notes, Sec. 2.2 boxed form and Sec. 2.4;
// alpha = e^gate), with the base state W and the residual state R:
//   r = Clip_[-c, c](v - W_{t-1} k),   o = alpha W_{t-1} q + gamma R_t q,
//   W_t = alpha W_{t-1} + k u^T,  u = beta v (RLA) | beta (v - alpha W_{t-1} k) (RDN),
//   R_t = alpha R_{t-1} + k w^T,  w = gamma r (RLA) | gamma (r - alpha R_{t-1} k) (RDN),
// written in the state orientation H = W^T ([dk][dv]).  The notes split the computation
// into two chunkwise stages (Sec. 2.6); the chunk form of both is derived here.  For a
// chunk of rows t with incoming states H0 (base) and HR0 (residual), g the inclusive
// prefix of the log-decays, gx = g - gate (the exclusive one), Gamma_tj = e^{g_t - g_j},
// Gamma'_tj = e^{gx_t - g_j}, and H_{t-1} = e^{gx_t} H0 + sum_{j<t} e^{gx_t - g_j} k_j u_j^T:
//   W_{t-1} k_t      -> Wk = Diag(e^{gx}) K H0 + (strict_tril(K K^T) * Gamma') U,
//   alpha W_{t-1} q_t -> Wq = Diag(e^g) Q H0 + (strict_tril(Q K^T) * Gamma) U,
//   U = Diag(beta) V (RLA) | T_beta Diag(beta) (V - Diag(e^g) K H0) (RDN), where T_beta =
//     (I + strict_tril(Diag(beta) (K K^T * Gamma)))^-1 is the delta rule's UT solve,
//   r = Clip(V - Wk),
//   w = Diag(gamma) r (RLA) | T_gamma Diag(gamma) (r - Diag(e^g) K HR0) (RDN),
//   R_t q_t -> Rq = Diag(e^g) Q HR0 + (tril(Q K^T) * Gamma) w,
//   o = Wq + Diag(gamma) Rq,
//   H_C = e^{g_C} H0 + K^T Diag(e^{g_C - g}) U,   HR_C = e^{g_C} HR0 + K^T Diag(e^{g_C - g}) w.
// (Padded rows past the end of the sequence are zero and carry no decay.)  The solves
// T_beta and T_gamma come from the pre-solved variant's solve kernel (X = [P T ; T] of every
// chunk, run with beta and with gamma), written to the workspace.
//
// Work split: one CTA of 8 warps per (b, h, 64-wide slice of dv) walks the chunks; both
// state slices stay in fp32 registers (the warp owns the same 16 x 16 tiles of the 128 x 64
// slice in every chunk) and are rounded to fp16 once per chunk as MMA operands.
#include "ldn_internal.cuh"
#include "sm100_ptx.cuh"
#include "warp_mma.cuh"

namespace ldn {
namespace {
using namespace sm100;
using namespace wmma8;

constexpr int kXBytes = 16384;   // X image per (b, h, chunk)

struct RlaSmem {
    static constexpr int q = 0;                          // Q [64][136] fp16
    static constexpr int k = q + kC * kLdW * 2;          // K
    static constexpr int v = k + kC * kLdW * 2;          // V slice [64][72]
    static constexpr int h = v + kC * kLdN * 2;          // H0 slice [128][72]
    static constexpr int hr = h + kD * kLdN * 2;         // HR0 slice
    static constexpr int mk = hr + kD * kLdN * 2;        // strict_tril(K K^T) * Gamma' [64][72]
    static constexpr int mq = mk + kC * kLdN * 2;        // strict_tril(Q K^T) * Gamma
    static constexpr int mqi = mq + kC * kLdN * 2;       // tril(Q K^T) * Gamma
    static constexpr int u = mqi + kC * kLdN * 2;        // U
    static constexpr int y = u + kC * kLdN * 2;          // RDN: Diag(beta)(V - Diag(e^g) K H0); then Diag(e^{gC-g}) U
    static constexpr int r = y + kC * kLdN * 2;          // r; RDN: Diag(gamma)(r - ..); then Diag(e^{gC-g}) w
    static constexpr int w = r + kC * kLdN * 2;          // w
    static constexpr int tb = w + kC * kLdN * 2;         // T_beta (RDN)
    static constexpr int tg = tb + kC * kLdN * 2;        // T_gamma (RDN)
    static constexpr int small = tg + kC * kLdN * 2;     // beta, gamma, g, gx, e^g, e^gx, e^{gC-g}
    // staging of the next chunk's inputs (cp.async): q, k rows (bf16 [64][128]), the v slice
    // (bf16 [64][64]), T_beta's and T_gamma's raw rows (8 KB each), gate, beta, gamma
    static constexpr int sq = small + 7 * kC * 4;
    static constexpr int sk = sq + kC * kD * 2;
    static constexpr int sv = sk + kC * kD * 2;
    static constexpr int stb = sv + kC * 64 * 2;
    static constexpr int stg = stb + 8192;
    static constexpr int sgt = stg + 8192;
    static constexpr int sbt = sgt + kC * 4;
    static constexpr int sgm = sbt + kC * 4;
    static constexpr int bytes = sgm + kC * 4;
    static_assert(bytes <= 232448, "shared memory plan exceeds 227 KB");
};

// Stage chunk c's inputs (16-byte cp.async; rows past the sequence read as zero).
template <bool DELTA>
__device__ __forceinline__ void rla_prefetch(uint8_t *sm, const __nv_bfloat16 *__restrict__ q,
                                             const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                                             const float *__restrict__ beta, const float *__restrict__ gamma,
                                             const float *__restrict__ gate, const uint8_t *__restrict__ Xb,
                                             const uint8_t *__restrict__ Xg, size_t tok0, size_t xc, int H, int L,
                                             int n0, int tid)
{
    using SM = RlaSmem;
    for (int e = tid; e < 2 * kC * 16; e += kThreads) {   // q, k: 16 groups per row
        const int which = e / (kC * 16), rr = (e / 16) % kC, part = e % 16;
        const __nv_bfloat16 *src = (which ? k : q) + (tok0 + (size_t)(rr < L ? rr : 0) * H) * kD + 8 * part;
        cp_async16(sm + (which ? SM::sk : SM::sq) + (rr * 16 + part) * 16, src, rr < L ? 16u : 0u);
    }
    for (int e = tid; e < kC * 8; e += kThreads) {        // v slice: 8 groups per row; T rows
        const int rr = e >> 3, part = e & 7;
        cp_async16(sm + SM::sv + e * 16, v + (tok0 + (size_t)(rr < L ? rr : 0) * H) * kD + n0 + 8 * part,
                   rr < L ? 16u : 0u);
        if (DELTA) {
            cp_async16(sm + SM::stb + e * 16, Xb + xc + 8192 + e * 16, 16u);
            cp_async16(sm + SM::stg + e * 16, Xg + xc + 8192 + e * 16, 16u);
        }
    }
    if (tid < kC) {
        const int rr = tid;
        const size_t o = tok0 + (size_t)(rr < L ? rr : 0) * H;
        const uint32_t n = rr < L ? 4u : 0u;
        cp_async4(sm + SM::sgt + 4 * rr, gate + o, n);
        cp_async4(sm + SM::sbt + 4 * rr, beta + o, n);
        cp_async4(sm + SM::sgm + 4 * rr, gamma + o, n);
    }
    cp_async_commit();
}

template <bool DELTA>
__global__ void __launch_bounds__(kThreads, 1)
rla_chunk_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                 const __nv_bfloat16 *__restrict__ v, const float *__restrict__ beta,
                 const float *__restrict__ gamma, const float *__restrict__ gate, float clip,
                 const float *__restrict__ S0, const float *__restrict__ R0, __nv_bfloat16 *__restrict__ out,
                 float *__restrict__ S_final, float *__restrict__ R_final, const uint8_t *__restrict__ Xb,
                 const uint8_t *__restrict__ Xg, int T, int H)
{
    extern __shared__ __align__(16) uint8_t sm[];
    using SM = RlaSmem;
    __half *Qs = reinterpret_cast<__half *>(sm + SM::q), *Ks = reinterpret_cast<__half *>(sm + SM::k);
    __half *Vs = reinterpret_cast<__half *>(sm + SM::v), *Hh = reinterpret_cast<__half *>(sm + SM::h);
    __half *HRh = reinterpret_cast<__half *>(sm + SM::hr), *Mk = reinterpret_cast<__half *>(sm + SM::mk);
    __half *Mq = reinterpret_cast<__half *>(sm + SM::mq), *Mqi = reinterpret_cast<__half *>(sm + SM::mqi);
    __half *Us = reinterpret_cast<__half *>(sm + SM::u), *Ys = reinterpret_cast<__half *>(sm + SM::y);
    __half *Rs = reinterpret_cast<__half *>(sm + SM::r), *Wsm = reinterpret_cast<__half *>(sm + SM::w);
    __half *Tb = reinterpret_cast<__half *>(sm + SM::tb), *Tg = reinterpret_cast<__half *>(sm + SM::tg);
    float *sb = reinterpret_cast<float *>(sm + SM::small), *sgm = sb + kC, *sg = sgm + kC, *sgx = sg + kC;
    float *seg = sgx + kC, *segx = seg + kC, *segc = segx + kC;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x >> 1, n0 = (blockIdx.x & 1) * 64;
    const int b = unit / H, h = unit % H;
    const int nch = (T + kC - 1) / kC;

    // the state slices (rows dk, columns n0 .. n0 + 63), fp32, tile i of this warp
    float hs[4][2][4], hrs[4][2][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int2 og = tile_origin<kD, 64>(warp, i);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const size_t o = ((size_t)unit * kD + acc_row(lane, og.x, e)) * kD + n0 + acc_col(lane, og.y, nt, e);
                hs[i][nt][e] = S0 ? S0[o] : 0.f;
                hrs[i][nt][e] = R0 ? R0[o] : 0.f;
            }
    }
    auto tok_of = [&](int c) { return ((size_t)b * T + (size_t)c * kC) * H + h; };
    rla_prefetch<DELTA>(sm, q, k, v, beta, gamma, gate, Xb, Xg, tok_of(0), (size_t)unit * nch * kXBytes, H,
                        min(kC, T), n0, tid);
    for (int c = 0; c < nch; ++c) {
        const int t0 = c * kC, L = min(kC, T - t0);
        const size_t tok0 = tok_of(c);
        cp_async_wait<0>();
        __syncthreads();
        // ---- the staged inputs: q, k rows (fp16 tiles), the v slice, T's, gates; the states
        //      as fp16 operands
        for (int e = tid; e < 2 * kC * 16; e += kThreads) {
            const int which = e / (kC * 16), rr = (e / 16) % kC, part = e % 16;
            const uint4 u = *reinterpret_cast<const uint4 *>(sm + (which ? SM::sk : SM::sq) + (rr * 16 + part) * 16);
            *reinterpret_cast<uint4 *>((which ? Ks : Qs) + rr * kLdW + 8 * part) = bf16x8_to_f16(u);
        }
        for (int e = tid; e < kC * 8; e += kThreads) {
            const int rr = e >> 3, part = e & 7;
            *reinterpret_cast<uint4 *>(Vs + rr * kLdN + 8 * part) =
                bf16x8_to_f16(*reinterpret_cast<const uint4 *>(sm + SM::sv + e * 16));
            if (DELTA) {
                const int c8 = 8 * ((part ^ (64 + rr)) & 7);
                *reinterpret_cast<uint4 *>(Tb + rr * kLdN + c8) = *reinterpret_cast<const uint4 *>(sm + SM::stb + e * 16);
                *reinterpret_cast<uint4 *>(Tg + rr * kLdN + c8) = *reinterpret_cast<const uint4 *>(sm + SM::stg + e * 16);
            }
        }
        if (warp == 0) {
            const float *gg = reinterpret_cast<const float *>(sm + SM::sgt);
            const float *gb = reinterpret_cast<const float *>(sm + SM::sbt);
            const float *gm = reinterpret_cast<const float *>(sm + SM::sgm);
            const int r0 = 2 * lane, r1 = r0 + 1;
            const float a0 = gg[r0], a1 = gg[r1];
            float incl = a0 + a1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float yv = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += yv;
            }
            const float gl = __shfl_sync(0xffffffffu, incl, 31);
            const float g0 = incl - a1, g1 = incl;
            sg[r0] = g0;
            sg[r1] = g1;
            sgx[r0] = g0 - a0;
            sgx[r1] = g1 - a1;
            seg[r0] = expf(g0);
            seg[r1] = expf(g1);
            segx[r0] = expf(g0 - a0);
            segx[r1] = expf(g1 - a1);
            segc[r0] = expf(gl - g0);
            segc[r1] = expf(gl - g1);
            sb[r0] = gb[r0];
            sb[r1] = gb[r1];
            sgm[r0] = gm[r0];
            sgm[r1] = gm[r1];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int2 og = tile_origin<kD, 64>(warp, i);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, og.x, e), cc = acc_col(lane, og.y, nt, e);
                    *reinterpret_cast<__half2 *>(Hh + rr * kLdN + cc) = __floats2half2_rn(hs[i][nt][e], hs[i][nt][e + 1]);
                    *reinterpret_cast<__half2 *>(HRh + rr * kLdN + cc) =
                        __floats2half2_rn(hrs[i][nt][e], hrs[i][nt][e + 1]);
                }
        }
        __syncthreads();
        if (c + 1 < nch)   // the staging buffer is free: the next chunk's inputs load under this chunk's products
            rla_prefetch<DELTA>(sm, q, k, v, beta, gamma, gate, Xb, Xg, tok_of(c + 1),
                                ((size_t)unit * nch + c + 1) * kXBytes, H, min(kC, T - (c + 1) * kC), n0, tid);
        // ---- A: the masked, decayed score tiles; K H0 and Q H0 (fp32, this warp's tiles)
        {
            const Op okk[1] = {{Ks, kLdW, false, Ks, kLdW, true, kD}};
            cta_mma<kC, kC>(okk, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int rr = acc_row(lane, m0, e), jj = acc_col(lane, c0, nt, e);
                        Mk[rr * kLdN + jj] = __float2half_rn(jj < rr ? acc[nt][e] * expf(sgx[rr] - sg[jj]) : 0.f);
                    }
            });
            const Op oqk[1] = {{Qs, kLdW, false, Ks, kLdW, true, kD}};
            cta_mma<kC, kC>(oqk, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int rr = acc_row(lane, m0, e), jj = acc_col(lane, c0, nt, e);
                        const float s = jj <= rr ? acc[nt][e] * expf(sg[rr] - sg[jj]) : 0.f;
                        Mq[rr * kLdN + jj] = __float2half_rn(jj < rr ? s : 0.f);
                        Mqi[rr * kLdN + jj] = __float2half_rn(s);
                    }
            });
        }
        float kh[2][2][4], qh[2][2][4];
        {
            const Op o1[1] = {{Ks, kLdW, false, Hh, kLdN, false, kD}};
            cta_mma<kC, 64>(o1, warp, lane, [&](int i, int, int, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) kh[i][nt][e] = acc[nt][e];
            });
            const Op o2[1] = {{Qs, kLdW, false, Hh, kLdN, false, kD}};
            cta_mma<kC, 64>(o2, warp, lane, [&](int i, int, int, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) qh[i][nt][e] = acc[nt][e];
            });
        }
        // ---- B: U = Diag(beta) V (RLA) | Y = Diag(beta)(V - Diag(e^g) K H0) (RDN)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int2 og = tile_origin<kC, 64>(warp, i);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int rr = acc_row(lane, og.x, e), cc = acc_col(lane, og.y, nt, e);
                    const float2 vv = __half22float2(*reinterpret_cast<const __half2 *>(Vs + rr * kLdN + cc));
                    if (DELTA)
                        *reinterpret_cast<__half2 *>(Ys + rr * kLdN + cc) =
                            __floats2half2_rn(sb[rr] * (vv.x - seg[rr] * kh[i][nt][e]),
                                              sb[rr] * (vv.y - seg[rr] * kh[i][nt][e + 1]));
                    else
                        *reinterpret_cast<__half2 *>(Us + rr * kLdN + cc) = __floats2half2_rn(sb[rr] * vv.x, sb[rr] * vv.y);
                }
        }
        __syncthreads();
        if (DELTA) {   // ---- C: U = T_beta Y
            const Op o[1] = {{Tb, kLdN, false, Ys, kLdN, false, kC}};
            cta_mma<kC, 64>(o, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                        *reinterpret_cast<__half2 *>(Us + rr * kLdN + cc) = __floats2half2_rn(acc[nt][e], acc[nt][e + 1]);
                    }
            });
            __syncthreads();
        }
        // ---- D: Wk -> r = Clip(V - Wk); Wq (kept); Diag(e^{gC-g}) U (into Y's place)
        float wq[2][2][4];
        {
            const Op o1[1] = {{Mk, kLdN, false, Us, kLdN, false, kC}};
            cta_mma<kC, 64>(o1, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                        const float2 vv = __half22float2(*reinterpret_cast<const __half2 *>(Vs + rr * kLdN + cc));
                        const float r0 = fminf(fmaxf(vv.x - (segx[rr] * kh[i][nt][e] + acc[nt][e]), -clip), clip);
                        const float r1 = fminf(fmaxf(vv.y - (segx[rr] * kh[i][nt][e + 1] + acc[nt][e + 1]), -clip), clip);
                        *reinterpret_cast<__half2 *>(Rs + rr * kLdN + cc) = __floats2half2_rn(r0, r1);
                    }
            });
            const Op o2[1] = {{Mq, kLdN, false, Us, kLdN, false, kC}};
            cta_mma<kC, 64>(o2, warp, lane, [&](int i, int m0, int, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) wq[i][nt][e] = seg[acc_row(lane, m0, e)] * qh[i][nt][e] + acc[nt][e];
            });
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int2 og = tile_origin<kC, 64>(warp, i);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int rr = acc_row(lane, og.x, e), cc = acc_col(lane, og.y, nt, e);
                        const float2 uu = __half22float2(*reinterpret_cast<const __half2 *>(Us + rr * kLdN + cc));
                        *reinterpret_cast<__half2 *>(Ys + rr * kLdN + cc) = __floats2half2_rn(segc[rr] * uu.x, segc[rr] * uu.y);
                    }
            }
        }
        __syncthreads();
        // ---- E / F / G: w = Diag(gamma) r (RLA) | T_gamma Diag(gamma)(r - Diag(e^g) K HR0) (RDN);
        //      Q HR0 (kept)
        float qhr[2][2][4];
        {
            const Op o2[1] = {{Qs, kLdW, false, HRh, kLdN, false, kD}};
            cta_mma<kC, 64>(o2, warp, lane, [&](int i, int, int, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) qhr[i][nt][e] = acc[nt][e];
            });
            if (DELTA) {
                const Op o1[1] = {{Ks, kLdW, false, HRh, kLdN, false, kD}};
                // in place over r: each thread rewrites only the elements it reads
                cta_mma<kC, 64>(o1, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; e += 2) {
                            const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                            __half2 *rp = reinterpret_cast<__half2 *>(Rs + rr * kLdN + cc);
                            const float2 rv = __half22float2(*rp);
                            *rp = __floats2half2_rn(sgm[rr] * (rv.x - seg[rr] * acc[nt][e]),
                                                    sgm[rr] * (rv.y - seg[rr] * acc[nt][e + 1]));
                        }
                });
                __syncthreads();
                const Op o3[1] = {{Tg, kLdN, false, Rs, kLdN, false, kC}};
                cta_mma<kC, 64>(o3, warp, lane, [&](int, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; e += 2) {
                            const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                            *reinterpret_cast<__half2 *>(Wsm + rr * kLdN + cc) =
                                __floats2half2_rn(acc[nt][e], acc[nt][e + 1]);
                        }
                });
            } else {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int2 og = tile_origin<kC, 64>(warp, i);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; e += 2) {
                            const int rr = acc_row(lane, og.x, e), cc = acc_col(lane, og.y, nt, e);
                            const float2 rv = __half22float2(*reinterpret_cast<const __half2 *>(Rs + rr * kLdN + cc));
                            *reinterpret_cast<__half2 *>(Wsm + rr * kLdN + cc) =
                                __floats2half2_rn(sgm[rr] * rv.x, sgm[rr] * rv.y);
                        }
                }
            }
        }
        __syncthreads();
        // ---- H: Rq, o = Wq + Diag(gamma) Rq (rows of this chunk); Diag(e^{gC-g}) w (into r's place)
        {
            const Op o1[1] = {{Mqi, kLdN, false, Wsm, kLdN, false, kC}};
            cta_mma<kC, 64>(o1, warp, lane, [&](int i, int m0, int c0, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int rr = acc_row(lane, m0, e), cc = acc_col(lane, c0, nt, e);
                        const float o0 = wq[i][nt][e] + sgm[rr] * (seg[rr] * qhr[i][nt][e] + acc[nt][e]);
                        const float o1v = wq[i][nt][e + 1] + sgm[rr] * (seg[rr] * qhr[i][nt][e + 1] + acc[nt][e + 1]);
                        if (rr < L)
                            *reinterpret_cast<__nv_bfloat162 *>(out + (tok0 + (size_t)rr * H) * kD + n0 + cc) =
                                __floats2bfloat162_rn(o0, o1v);
                    }
            });
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int2 og = tile_origin<kC, 64>(warp, i);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int rr = acc_row(lane, og.x, e), cc = acc_col(lane, og.y, nt, e);
                        const float2 ww = __half22float2(*reinterpret_cast<const __half2 *>(Wsm + rr * kLdN + cc));
                        *reinterpret_cast<__half2 *>(Rs + rr * kLdN + cc) = __floats2half2_rn(segc[rr] * ww.x, segc[rr] * ww.y);
                    }
            }
        }
        __syncthreads();
        // ---- I: H = e^{gC} H0 + K^T Diag(e^{gC-g}) U,  HR = e^{gC} HR0 + K^T Diag(e^{gC-g}) w
        {
            const float gC = expf(sg[kC - 1]);
            const Op o1[1] = {{Ks, kLdW, true, Ys, kLdN, false, kC}};
            cta_mma<kD, 64>(o1, warp, lane, [&](int i, int, int, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) hs[i][nt][e] = gC * hs[i][nt][e] + acc[nt][e];
            });
            const Op o2[1] = {{Ks, kLdW, true, Rs, kLdN, false, kC}};
            cta_mma<kD, 64>(o2, warp, lane, [&](int i, int, int, float (&acc)[2][4]) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) hrs[i][nt][e] = gC * hrs[i][nt][e] + acc[nt][e];
            });
        }
        // (the next chunk's first barrier orders these reads before its writes)
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int2 og = tile_origin<kD, 64>(warp, i);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const size_t o = ((size_t)unit * kD + acc_row(lane, og.x, e)) * kD + n0 + acc_col(lane, og.y, nt, e);
                if (S_final) *reinterpret_cast<float2 *>(S_final + o) = make_float2(hs[i][nt][e], hs[i][nt][e + 1]);
                if (R_final) *reinterpret_cast<float2 *>(R_final + o) = make_float2(hrs[i][nt][e], hrs[i][nt][e + 1]);
            }
    }
}

}  // namespace

bool rla_chunk_supported(const RlaArgs &a)
{
    const bool a16 = (((uintptr_t)a.q | (uintptr_t)a.k | (uintptr_t)a.v | (uintptr_t)a.out) & 15u) == 0;
    return a.dtype == LDN_BF16 && a.dk == kD && a.dv == kD && a.T > 0 && a16;
}

size_t rla_chunk_workspace_bytes(int B, int T, int H, int delta)
{
    if (!delta) return 0;
    return 2 * (size_t)B * H * ((T + kC - 1) / kC) * kXBytes;
}

cudaError_t launch_rla_chunk(const RlaArgs &a, void *ws, cudaStream_t s)
{
    const size_t units = (size_t)a.B * a.H, nch = (size_t)(a.T + kC - 1) / kC;
    uint8_t *Xb = reinterpret_cast<uint8_t *>(ws), *Xg = Xb ? Xb + units * nch * kXBytes : nullptr;
    cudaError_t e;
    if (a.delta) {   // the two solves: T_beta and T_gamma (Gated DeltaNet's, with the same decay)
        ChunkArgs f{a.q, a.k, a.v, a.beta, a.gate, nullptr, nullptr, nullptr, a.B, a.T, a.H, kD, kD, kC, LDN_GDN,
                    a.dtype, status_word_ptr()};
        if (!f.status) return cudaErrorInvalidValue;
        if ((e = launch_chunk_solve(f, Xb, s)) != cudaSuccess) return e;
        f.beta = a.gamma;
        if ((e = launch_chunk_solve(f, Xg, s)) != cudaSuccess) return e;
    }
    auto kern = a.delta ? rla_chunk_kernel<true> : rla_chunk_kernel<false>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RlaSmem::bytes)) != cudaSuccess)
        return e;
    kern<<<(unsigned)(units * 2), kThreads, RlaSmem::bytes, s>>>(
        (const __nv_bfloat16 *)a.q, (const __nv_bfloat16 *)a.k, (const __nv_bfloat16 *)a.v, a.beta, a.gamma, a.gate,
        a.clip, a.S0, a.R0, (__nv_bfloat16 *)a.out, a.S_final, a.R_final, Xb, Xg, a.T, a.H);
    return cudaGetLastError();
}

}  // namespace ldn
