// Token-recurrent forward for scalar decay, the two state passes of Residual
// Linear Attention / Residual DeltaNet (Residual Linear Attention notes,
// Sec. 2.2, 2.4, 2.6).  Per token, on the state H = S^T ([dk][dv]) column by
// column (each value column is its own linear system, state-reduction notes
// Sec. 2.5):
//   p = S_{t-1} k_t,  s = S_{t-1} q_t                (reads of the OLD state)
//   delta rule:  u = beta (v - alpha p),  additive:  u = beta v
//   S_t = alpha S_{t-1} + u k^T,  and S_t q_t = alpha s + u (k . q)
// PRE writes p and alpha s (fp32, the base pass); POST writes S_t q_t (the
// residual pass of the additive rule).
//
// Work split as in the backward kernel: one CTA of 256 threads per (b, h,
// 32-column slice of dv); lane l of warp w owns column l and key rows w dk/8 +
// j.  Both reads of a token are reduced over the rows together: a partial per
// warp, one exchange through a double-buffered shared array, one barrier per
// token.  A block of 8 tokens' inputs is loaded into registers a block ahead and
// stored to the other of two shared buffers.
#include "ldn_internal.cuh"

namespace ldn {
namespace {

constexpr int kBT = 256, kNW = 8, kNC = 32, kSub = 8;

template <int DK>
struct RecSmem {
    static constexpr size_t stage = 2 * kSub * DK /*q, k*/ + kSub * kNC /*v*/ + 3 * kSub /*beta, alpha, k.q*/;
    static constexpr size_t bytes = (2 * stage + 2 * 2 * kNW * kNC /*row sums, float2*/) * sizeof(float);
};

template <int DK, typename TIn, bool DELTA, bool PRE, bool POST>
__global__ void __launch_bounds__(kBT)
rec_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
           const float *__restrict__ beta, const float *__restrict__ gate, const float *__restrict__ S0,
           float *__restrict__ S_final, float *__restrict__ p_out, float *__restrict__ s_out,
           TIn *__restrict__ o_out, int T, int H, int dv)
{
    constexpr int RPT = DK / kNW;
    constexpr int NKQ = kSub * DK / kBT;
    static_assert(kSub * kNC == kBT && kSub <= kNW, "one v element per thread; one k . q per warp");
    extern __shared__ float sm[];
    float *stg = sm;
    float2 *red = reinterpret_cast<float2 *>(sm + 2 * RecSmem<DK>::stage);   // [2][kNW][kNC]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, r0 = warp * RPT;
    const int slices = dv / kNC;
    const int unit = blockIdx.x / slices, sl = blockIdx.x % slices;
    const int b = unit / H, h = unit % H, col = sl * kNC + lane;
    const int nsub = (T + kSub - 1) / kSub;
    auto tok = [&](int t) { return ((size_t)b * T + t) * H + h; };

    struct Pre { float k[NKQ], q[NKQ], v, b, a; };
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
        P.b = P.a = 0.f;
        if (tid < kSub && t0 + tid < T) {
            P.b = beta[tok(t0 + tid)];
            P.a = gate[tok(t0 + tid)];
        }
    };
    // buffer layout: q [kSub][DK], k [kSub][DK], v [kSub][kNC], beta, alpha, k.q [kSub]
    auto pre_store = [&](int buf, const Pre &P) {
        float *q_ = stg + buf * RecSmem<DK>::stage, *k_ = q_ + kSub * DK, *v_ = k_ + kSub * DK;
        float *b_ = v_ + kSub * kNC, *a_ = b_ + kSub;
#pragma unroll
        for (int x = 0; x < NKQ; ++x) {
            q_[tid + x * kBT] = P.q[x];
            k_[tid + x * kBT] = P.k[x];
        }
        v_[tid] = P.v;
        if (tid < kSub) {
            b_[tid] = P.b;
            a_[tid] = expf(P.a);
        }
    };
    // k . q of every token of a staged block (warp t: token t), after a barrier
    auto dots = [&](int buf) {
        float *q_ = stg + buf * RecSmem<DK>::stage, *k_ = q_ + kSub * DK, *kq = k_ + kSub * DK + kSub * kNC + 2 * kSub;
        if (warp < kSub) {
            float d = 0.f;
            for (int c = lane; c < DK; c += 32) d += q_[warp * DK + c] * k_[warp * DK + c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0) kq[warp] = d;
        }
    };

    float hr[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) hr[j] = S0 ? S0[((size_t)unit * DK + r0 + j) * dv + col] : 0.f;
    Pre P;
    if (nsub > 0) {
        pre_load(0, P);
        pre_store(0, P);
    }
    int par = 0;
    for (int s = 0; s < nsub; ++s) {
        __syncthreads();                        // block s staged; block s - 1 done with the other buffer
        if (POST) {
            dots(s & 1);
            __syncthreads();
        }
        const float *qs = stg + (s & 1) * RecSmem<DK>::stage, *ks = qs + kSub * DK, *vs = ks + kSub * DK;
        const float *bs = vs + kSub * kNC, *as = bs + kSub, *kq = as + kSub;
        if (s + 1 < nsub) pre_load(s + 1, P);
        const int t0 = s * kSub;
#pragma unroll
        for (int t = 0; t < kSub; ++t) {
            float pp = 0.f, ss = 0.f;
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                pp += hr[j] * ks[t * DK + r0 + j];
                ss += hr[j] * qs[t * DK + r0 + j];
            }
            float2 *rb = red + par * kNW * kNC;
            rb[warp * kNC + lane] = make_float2(pp, ss);
            __syncthreads();
            pp = ss = 0.f;
#pragma unroll
            for (int w = 0; w < kNW; ++w) {
                const float2 x = rb[w * kNC + lane];
                pp += x.x;
                ss += x.y;
            }
            par ^= 1;
            const float a = as[t], bt = bs[t];
            const float u = DELTA ? bt * (vs[t * kNC + lane] - a * pp) : bt * vs[t * kNC + lane];
#pragma unroll
            for (int j = 0; j < RPT; ++j) hr[j] = a * hr[j] + u * ks[t * DK + r0 + j];
            if (warp == 0 && t0 + t < T) {
                const size_t o = tok(t0 + t) * dv + col;
                if (PRE) {
                    p_out[o] = pp;
                    s_out[o] = a * ss;
                }
                if (POST) store_out(o_out, o, a * ss + u * kq[t]);
            }
        }
        if (s + 1 < nsub) pre_store((s + 1) & 1, P);
    }
    if (S_final)
#pragma unroll
        for (int j = 0; j < RPT; ++j) S_final[((size_t)unit * DK + r0 + j) * dv + col] = hr[j];
}

template <int DK, typename TIn, bool DELTA, bool PRE, bool POST>
cudaError_t go(const RecArgs &a, cudaStream_t st)
{
    auto kern = rec_kernel<DK, TIn, DELTA, PRE, POST>;
    const unsigned grid = (unsigned)((long long)a.B * a.H * (a.dv / kNC));
    kern<<<grid, kBT, RecSmem<DK>::bytes, st>>>((const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v, a.beta, a.gate,
                                                 a.S0, a.S_final, a.p_out, a.s_out, (TIn *)a.o_out, a.T, a.H, a.dv);
    return cudaGetLastError();
}

template <int DK, typename TIn>
cudaError_t launch_dk(const RecArgs &a, cudaStream_t st)
{
    if (a.pre) return a.delta ? go<DK, TIn, true, true, false>(a, st) : go<DK, TIn, false, true, false>(a, st);
    return a.delta ? go<DK, TIn, true, false, true>(a, st) : go<DK, TIn, false, false, true>(a, st);
}

}  // namespace

cudaError_t launch_recurrent(const RecArgs &a, cudaStream_t st)
{
    if (a.dtype == LDN_BF16)
        return a.dk == 128 ? launch_dk<128, __nv_bfloat16>(a, st) : launch_dk<64, __nv_bfloat16>(a, st);
    return a.dk == 128 ? launch_dk<128, float>(a, st) : launch_dk<64, float>(a, st);
}

}  // namespace ldn
