// Residual Linear Attention (RLA) and Residual DeltaNet (RDN), forward
// ("Residual Linear Attention" reading notes, Sec. 2.2 boxed form, Sec. 2.4):
//   r_t = Clip_[-c, c](v_t - S_{t-1} k_t),   o_t = alpha_t S_{t-1} q_t + gamma_t R_t q_t
//   RLA: S_t = alpha S_{t-1} + beta v k^T,          R_t = alpha R_{t-1} + gamma r k^T
//   RDN: S_t = alpha S_{t-1}(I - beta k k^T) + beta v k^T,
//        R_t = alpha R_{t-1}(I - gamma k k^T) + gamma r k^T
// The notes compute it in two stages (Sec. 2.6) so that an existing linear-attention
// kernel serves for both states; here both states step together in one pass, so
// neither r nor the residual read leaves the chip.
//
// Work split: one CTA of 256 threads per (b, h, 32-column slice of dv); each value
// column is its own linear system (state-reduction notes, Sec. 2.5).  Lane l of warp
// w owns column l and the key rows w dk/8 + j of both states, in registers, so every
// lane of a warp reads the same rows of q and k (shared-memory broadcasts).  The
// four row sums of a token go through one float4 exchange and one barrier.  A block
// of 8 tokens' inputs is loaded into registers a block ahead and stored to the other
// of two shared buffers; k . q of each token is formed once per block.
#include "ldn_internal.cuh"

namespace ldn {
namespace {

constexpr int kBT = 256, kNW = 8, kNC = 32, kSub = 8;

// Residual Linear Attention (DELTA = false) / Residual DeltaNet (DELTA = true) in
// one pass: both states step together, token by token (Residual Linear Attention
// notes, Sec. 2.2 boxed form, Sec. 2.4).  Per token the four reads of the old
// states (S k, S q, R k, R q) are reduced over the rows in one float4 exchange:
//   r = Clip(v - S_{t-1} k),  w = gamma r (RLA) | gamma (r - alpha R_{t-1} k) (RDN)
//   R_t = alpha R_{t-1} + w k^T,   R_t q = alpha R_{t-1} q + w (k . q)
//   o = alpha S_{t-1} q + gamma R_t q
//   S_t = alpha S_{t-1} + u k^T,   u = beta v (RLA) | beta (v - alpha S_{t-1} k) (RDN)
template <int DK, typename TIn, bool DELTA>
__global__ void __launch_bounds__(kBT)
rla_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
           const float *__restrict__ beta, const float *__restrict__ gamma, const float *__restrict__ gate, float clip,
           const float *__restrict__ S0, const float *__restrict__ R0, TIn *__restrict__ out,
           float *__restrict__ S_final, float *__restrict__ R_final, int T, int H, int dv)
{
    constexpr int RPT = DK / kNW;
    constexpr int NKQ = kSub * DK / kBT;
    // buffer: q, k [kSub][DK], v [kSub][kNC], beta, gamma, alpha, k.q [kSub]
    constexpr int STG = 2 * kSub * DK + kSub * kNC + 4 * kSub;
    extern __shared__ float sm[];
    float *stg = sm;
    float4 *red = reinterpret_cast<float4 *>(sm + 2 * STG);   // [2][kNW][kNC]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, r0 = warp * RPT;
    const int slices = dv / kNC;
    const int unit = blockIdx.x / slices, sl = blockIdx.x % slices;
    const int b = unit / H, h = unit % H, col = sl * kNC + lane;
    const int nsub = (T + kSub - 1) / kSub;
    auto tok = [&](int t) { return ((size_t)b * T + t) * H + h; };

    struct Pre { float k[NKQ], q[NKQ], v, b, c, a; };
    auto pre_load = [&](int s, Pre &P) {
        const int t0 = s * kSub;
#pragma unroll
        for (int x = 0; x < NKQ; ++x) {
            const int e = tid + x * kBT, t = e / DK, r = e % DK;
            const bool ok = t0 + t < T;
            const size_t i = tok(ok ? t0 + t : 0) * DK + r;
            P.k[x] = ok ? load_in(k, i) : 0.f;
            P.q[x] = ok ? load_in(q, i) : 0.f;
        }
        const int t = tid / kNC;
        const bool ok = t0 + t < T;
        P.v = ok ? load_in(v, tok(ok ? t0 + t : 0) * dv + sl * kNC + tid % kNC) : 0.f;
        P.b = P.c = P.a = 0.f;
        if (tid < kSub && t0 + tid < T) {
            P.b = beta[tok(t0 + tid)];
            P.c = gamma[tok(t0 + tid)];
            P.a = gate[tok(t0 + tid)];
        }
    };
    auto pre_store = [&](int buf, const Pre &P) {
        float *q_ = stg + buf * STG, *k_ = q_ + kSub * DK, *v_ = k_ + kSub * DK, *s_ = v_ + kSub * kNC;
#pragma unroll
        for (int x = 0; x < NKQ; ++x) {
            q_[tid + x * kBT] = P.q[x];
            k_[tid + x * kBT] = P.k[x];
        }
        v_[tid] = P.v;
        if (tid < kSub) {
            s_[tid] = P.b;
            s_[kSub + tid] = P.c;
            s_[2 * kSub + tid] = expf(P.a);
        }
    };

    float hs[RPT], hr[RPT];   // base and residual state rows of this thread's column
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        hs[j] = S0 ? S0[((size_t)unit * DK + r0 + j) * dv + col] : 0.f;
        hr[j] = R0 ? R0[((size_t)unit * DK + r0 + j) * dv + col] : 0.f;
    }
    Pre P;
    if (nsub > 0) {
        pre_load(0, P);
        pre_store(0, P);
    }
    int par = 0;
    for (int s = 0; s < nsub; ++s) {
        __syncthreads();                        // block s staged; block s - 1 done with the other buffer
        const float *qs = stg + (s & 1) * STG, *ks = qs + kSub * DK, *vs = ks + kSub * DK;
        const float *bs = vs + kSub * kNC, *gs = bs + kSub, *as = gs + kSub;
        float *kq = const_cast<float *>(as) + kSub;
        if (warp < kSub) {                      // k . q of token `warp` of the block
            float d = 0.f;
            for (int c = lane; c < DK; c += 32) d += qs[warp * DK + c] * ks[warp * DK + c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0) kq[warp] = d;
        }
        __syncthreads();
        if (s + 1 < nsub) pre_load(s + 1, P);
        const int t0 = s * kSub;
#pragma unroll
        for (int t = 0; t < kSub; ++t) {
            // this warp's rows of k_t and q_t (16-byte aligned, contiguous): vector loads
            float kr[RPT], qr[RPT];
#pragma unroll
            for (int j = 0; j < RPT; j += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(ks + t * DK + r0 + j);
                const float4 q4 = *reinterpret_cast<const float4 *>(qs + t * DK + r0 + j);
                kr[j] = k4.x; kr[j + 1] = k4.y; kr[j + 2] = k4.z; kr[j + 3] = k4.w;
                qr[j] = q4.x; qr[j + 1] = q4.y; qr[j + 2] = q4.z; qr[j + 3] = q4.w;
            }
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                x.x += hs[j] * kr[j];
                x.y += hs[j] * qr[j];
                x.z += hr[j] * kr[j];
                x.w += hr[j] * qr[j];
            }
            float4 *rb = red + par * kNW * kNC;
            rb[warp * kNC + lane] = x;
            __syncthreads();
            x = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kNW; ++w) {
                const float4 y = rb[w * kNC + lane];
                x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
            }
            par ^= 1;
            const float a = as[t], bt = bs[t], gm = gs[t], vv = vs[t * kNC + lane];
            const float r = fminf(fmaxf(vv - x.x, -clip), clip);
            const float wr = DELTA ? gm * (r - a * x.z) : gm * r;
            const float u = DELTA ? bt * (vv - a * x.x) : bt * vv;
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                hr[j] = a * hr[j] + wr * kr[j];
                hs[j] = a * hs[j] + u * kr[j];
            }
            if (warp == 0 && t0 + t < T)
                store_out(out, tok(t0 + t) * dv + col, a * x.y + gm * (a * x.w + wr * kq[t]));
        }
        if (s + 1 < nsub) pre_store((s + 1) & 1, P);
    }
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const size_t o = ((size_t)unit * DK + r0 + j) * dv + col;
        if (S_final) S_final[o] = hs[j];
        if (R_final) R_final[o] = hr[j];
    }
}

template <int DK, typename TIn, bool DELTA>
cudaError_t go_rla(const RlaArgs &a, cudaStream_t st)
{
    constexpr size_t smem = (2 * (2 * kSub * DK + kSub * kNC + 4 * kSub) + 2 * 4 * kNW * kNC) * sizeof(float);
    const unsigned grid = (unsigned)((long long)a.B * a.H * (a.dv / kNC));
    rla_kernel<DK, TIn, DELTA><<<grid, kBT, smem, st>>>((const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v, a.beta,
                                                        a.gamma, a.gate, a.clip, a.S0, a.R0, (TIn *)a.out,
                                                        a.S_final, a.R_final, a.T, a.H, a.dv);
    return cudaGetLastError();
}

template <int DK, typename TIn>
cudaError_t rla_dk(const RlaArgs &a, cudaStream_t st)
{
    return a.delta ? go_rla<DK, TIn, true>(a, st) : go_rla<DK, TIn, false>(a, st);
}

}  // namespace

cudaError_t launch_rla(const RlaArgs &a, cudaStream_t st)
{
    if (a.dtype == LDN_BF16)
        return a.dk == 128 ? rla_dk<128, __nv_bfloat16>(a, st) : rla_dk<64, __nv_bfloat16>(a, st);
    return a.dk == 128 ? rla_dk<128, float>(a, st) : rla_dk<64, float>(a, st);
}

}  // namespace ldn
