// Single-token recurrent decode step, fp32 state streamed once through HBM.
//
// For one token per (b, h) the step is, in memory orientation H = S^T
// ([dk][dv], fp32):
//   H' = alpha H (Gated DeltaNet) | Diag(a) H (KDA) | H (DeltaNet)
//   p  = H'^T k,  s = H'^T q                      (one pass over H')
//   r  = beta (v - p),  o = s + r (k . q)         (prediction-correction form,
//                                                   Residual Linear Attention
//                                                   notes, Sec. 1.2)
//   H  <- H' + k r^T                              (in place)
// Decay before the error follows the linear-attention notes, Sec. 2.4 Eqs.
// 15-17; the KDA decay acts on the key rows of H (Sec. 2.5, Eqs. 18-20).
// Gated DeltaNet-2 (Sec. 2.6, Eqs. 21-24) keeps the KDA decay, predicts along
// the erase direction e = b * k (p = H'^T e) and writes z = w * v:
// r = z - p, with no beta; the write direction and the read stay k and q.
//
// Work split: one CTA of 128 threads per (b, h, DVC-column slice of dv).
// Columns are independent (each value channel is its own linear system,
// state-reduction notes Sec. 2.5), so slices need no communication.  A row of
// the slice is covered by DVC/4 threads with float4 accesses; the row groups
// stride over dk and each thread keeps its float4s of H' in registers
// between the read pass and the write pass, so H is read once and written
// once.  DVC = 64 for dk = 128 (32 KiB of state per CTA, 16 float4 per
// thread); for dk = 64 the state is small enough that the whole step runs in
// under two waves of CTAs, and narrow slices (DVC = 32, 8 KiB per CTA) give more,
// finer waves whose writes overlap the next CTAs' reads (14.3 us per step
// against 15.2 us with 128-column slices, L2 flushed).
#include "ldn_internal.cuh"

namespace ldn {
namespace {

constexpr int kDecThreads = 128;

template <int DK, int DVC, typename TIn, int MODE>
__global__ void __launch_bounds__(kDecThreads)
decode_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
              const float *__restrict__ beta, const float *__restrict__ gate,
              float *__restrict__ S, TIn *__restrict__ out, int dv,
              const float *__restrict__ erase, const float *__restrict__ write)
{
    constexpr bool kG2 = MODE == LDN_GDN2;
    constexpr bool kChan = MODE == LDN_KDA || kG2;
    constexpr int TPR = DVC / 4;               // threads per row (float4 each)
    constexpr int RP = kDecThreads / TPR;      // rows per pass
    constexpr int RPT = DK / RP;               // rows held per thread
    __shared__ float qs[DK], ks[DK], as[DK], es[kG2 ? DK : 1];
    __shared__ __align__(16) float red_p[RP][DVC];
    __shared__ __align__(16) float red_s[RP][DVC];
    __shared__ __align__(16) float rs[DVC];
    __shared__ float kq_part[kDecThreads / 32];

    const int slices = dv / DVC;
    const int unit = blockIdx.x / slices;      // (b, h) pair, b * H + h
    const int col0 = (blockIdx.x % slices) * DVC;
    const int tid = threadIdx.x;

    const int cg = tid % TPR;                  // float4 column group
    const int rg = tid / TPR;                  // first row of this thread
    float *Sbase = S + (size_t)unit * DK * dv + col0 + 4 * cg;

    // Issue the state loads first: they are the stream; q/k/gates are small.
    float4 h[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i)
        h[i] = *reinterpret_cast<const float4 *>(Sbase + (size_t)(rg + i * RP) * dv);

    float kq = 0.0f;
    if (tid < DK) {
        const float qv = load_in(q, (size_t)unit * DK + tid);
        const float kv = load_in(k, (size_t)unit * DK + tid);
        qs[tid] = qv;
        ks[tid] = kv;
        if (kChan) as[tid] = expf(gate[(size_t)unit * DK + tid]);
        if (kG2) es[tid] = erase[(size_t)unit * DK + tid] * kv;
        kq = qv * kv;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
    if ((tid & 31) == 0) kq_part[tid >> 5] = kq;
    const float alpha = (MODE == LDN_GDN) ? expf(gate[unit]) : 1.0f;
    __syncthreads();

    float4 p = make_float4(0.f, 0.f, 0.f, 0.f), s = p;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = rg + i * RP;
        const float d = kChan ? as[row] : alpha;
        if (MODE != LDN_DELTANET) { h[i].x *= d; h[i].y *= d; h[i].z *= d; h[i].w *= d; }
        const float kr = kG2 ? es[row] : ks[row], qr = qs[row];
        p.x += h[i].x * kr; p.y += h[i].y * kr; p.z += h[i].z * kr; p.w += h[i].w * kr;
        s.x += h[i].x * qr; s.y += h[i].y * qr; s.z += h[i].z * qr; s.w += h[i].w * qr;
    }
    *reinterpret_cast<float4 *>(&red_p[rg][4 * cg]) = p;
    *reinterpret_cast<float4 *>(&red_s[rg][4 * cg]) = s;
    __syncthreads();

    if (tid < DVC) {
        float pp = 0.f, ss = 0.f, kqt = 0.f;
#pragma unroll
        for (int g = 0; g < RP; ++g) { pp += red_p[g][tid]; ss += red_s[g][tid]; }
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w) kqt += kq_part[w];
        const size_t vi = (size_t)unit * dv + col0 + tid;
        const float r = kG2 ? write[vi] * load_in(v, vi) - pp : beta[unit] * (load_in(v, vi) - pp);
        rs[tid] = r;
        store_out(out, vi, ss + r * kqt);
    }
    __syncthreads();

    const float4 r4 = *reinterpret_cast<const float4 *>(&rs[4 * cg]);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const float kr = ks[rg + i * RP];
        float4 o = h[i];
        o.x += kr * r4.x; o.y += kr * r4.y; o.z += kr * r4.z; o.w += kr * r4.w;
        *reinterpret_cast<float4 *>(Sbase + (size_t)(rg + i * RP) * dv) = o;
    }
}

// Several consecutive steps of the same sequences in one launch (DeltaNet, Gated DeltaNet,
// KDA): the CTA's state slice stays in registers across the steps and is read and written
// once; each step's q, k, v and gates are loaded one step ahead, in registers; q, k and the
// reductions alternate between two shared buffers, so a step takes three barriers.  Inputs
// of step s are at offset s * B * H (times the row width) of each tensor.
template <int DK, int DVC, typename TIn, int MODE>
__global__ void __launch_bounds__(kDecThreads)
decode_steps_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
                    const float *__restrict__ beta, const float *__restrict__ gate, float *__restrict__ S,
                    TIn *__restrict__ out, int dv, int nsteps, long long BH)
{
    constexpr bool kChan = MODE == LDN_KDA;
    constexpr int TPR = DVC / 4, RP = kDecThreads / TPR, RPT = DK / RP;
    __shared__ float qs[2][DK], ks[2][DK], as[2][kChan ? DK : 1];
    __shared__ __align__(16) float red_p[RP][DVC];
    __shared__ __align__(16) float red_s[RP][DVC];
    __shared__ __align__(16) float rs[DVC];
    __shared__ float kq_part[2][kDecThreads / 32];

    const int slices = dv / DVC;
    const int unit = blockIdx.x / slices, col0 = (blockIdx.x % slices) * DVC;
    const int tid = threadIdx.x, cg = tid % TPR, rg = tid / TPR;
    float *Sbase = S + (size_t)unit * DK * dv + col0 + 4 * cg;
    float4 h[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) h[i] = *reinterpret_cast<const float4 *>(Sbase + (size_t)(rg + i * RP) * dv);

    float nq = 0.f, nk = 0.f, na = 0.f, nv = 0.f, nb = 0.f, ng = 0.f;   // the next step's inputs
    auto fetch = [&](int s) {
        const size_t su = (size_t)s * BH + unit;
        if (tid < DK) {
            nq = load_in(q, su * DK + tid);
            nk = load_in(k, su * DK + tid);
            if (kChan) na = gate[su * DK + tid];
        }
        if (tid < DVC) {
            nv = load_in(v, su * dv + col0 + tid);
            nb = beta[su];
        }
        if (MODE == LDN_GDN) ng = gate[su];
    };
    fetch(0);
    for (int s = 0; s < nsteps; ++s) {
        const int buf = s & 1;
        float kq = 0.f;
        if (tid < DK) {
            qs[buf][tid] = nq;
            ks[buf][tid] = nk;
            if (kChan) as[buf][tid] = expf(na);
            kq = nq * nk;
        }
        const float cv = nv, cb = nb, alpha = MODE == LDN_GDN ? expf(ng) : 1.f;
        if (s + 1 < nsteps) fetch(s + 1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
        if ((tid & 31) == 0) kq_part[buf][tid >> 5] = kq;
        __syncthreads();

        float4 p = make_float4(0.f, 0.f, 0.f, 0.f), sq = p;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int row = rg + i * RP;
            const float d = kChan ? as[buf][row] : alpha;
            if (MODE != LDN_DELTANET) { h[i].x *= d; h[i].y *= d; h[i].z *= d; h[i].w *= d; }
            const float kr = ks[buf][row], qr = qs[buf][row];
            p.x += h[i].x * kr; p.y += h[i].y * kr; p.z += h[i].z * kr; p.w += h[i].w * kr;
            sq.x += h[i].x * qr; sq.y += h[i].y * qr; sq.z += h[i].z * qr; sq.w += h[i].w * qr;
        }
        *reinterpret_cast<float4 *>(&red_p[rg][4 * cg]) = p;
        *reinterpret_cast<float4 *>(&red_s[rg][4 * cg]) = sq;
        __syncthreads();

        if (tid < DVC) {
            float pp = 0.f, ss = 0.f, kqt = 0.f;
#pragma unroll
            for (int g = 0; g < RP; ++g) { pp += red_p[g][tid]; ss += red_s[g][tid]; }
#pragma unroll
            for (int w = 0; w < kDecThreads / 32; ++w) kqt += kq_part[buf][w];
            const float r = cb * (cv - pp);
            rs[tid] = r;
            store_out(out, ((size_t)s * BH + unit) * dv + col0 + tid, ss + r * kqt);
        }
        __syncthreads();

        const float4 r4 = *reinterpret_cast<const float4 *>(&rs[4 * cg]);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const float kr = ks[buf][rg + i * RP];
            h[i].x += kr * r4.x; h[i].y += kr * r4.y; h[i].z += kr * r4.z; h[i].w += kr * r4.w;
        }
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) *reinterpret_cast<float4 *>(Sbase + (size_t)(rg + i * RP) * dv) = h[i];
}

template <int DK, int DVC, typename TIn>
cudaError_t launch_steps_cfg(const DecodeArgs &a, int nsteps, cudaStream_t st)
{
    const unsigned grid = (unsigned)((long long)a.B * a.H * (a.dv / DVC));
    const TIn *q = (const TIn *)a.q, *k = (const TIn *)a.k, *v = (const TIn *)a.v;
    TIn *o = (TIn *)a.out;
    const long long BH = (long long)a.B * a.H;
    switch (a.mode) {
    case LDN_DELTANET:
        decode_steps_kernel<DK, DVC, TIn, LDN_DELTANET><<<grid, kDecThreads, 0, st>>>(q, k, v, a.beta, a.gate, a.S, o,
                                                                                       a.dv, nsteps, BH);
        break;
    case LDN_GDN:
        decode_steps_kernel<DK, DVC, TIn, LDN_GDN><<<grid, kDecThreads, 0, st>>>(q, k, v, a.beta, a.gate, a.S, o, a.dv,
                                                                                  nsteps, BH);
        break;
    default:
        decode_steps_kernel<DK, DVC, TIn, LDN_KDA><<<grid, kDecThreads, 0, st>>>(q, k, v, a.beta, a.gate, a.S, o, a.dv,
                                                                                  nsteps, BH);
        break;
    }
    return cudaGetLastError();
}

template <int DK, int DVC, typename TIn>
cudaError_t launch_cfg(const DecodeArgs &a, cudaStream_t st)
{
    const unsigned grid = (unsigned)((long long)a.B * a.H * (a.dv / DVC));
    const TIn *q = (const TIn *)a.q, *k = (const TIn *)a.k, *v = (const TIn *)a.v;
    TIn *o = (TIn *)a.out;
    const float *eb = a.erase, *wb = a.write;
    switch (a.mode) {
    case LDN_DELTANET:
        decode_kernel<DK, DVC, TIn, LDN_DELTANET><<<grid, kDecThreads, 0, st>>>(q, k, v, a.beta, a.gate, a.S, o, a.dv,
                                                                                 eb, wb);
        break;
    case LDN_GDN:
        decode_kernel<DK, DVC, TIn, LDN_GDN><<<grid, kDecThreads, 0, st>>>(q, k, v, a.beta, a.gate, a.S, o, a.dv, eb, wb);
        break;
    case LDN_GDN2:
        decode_kernel<DK, DVC, TIn, LDN_GDN2><<<grid, kDecThreads, 0, st>>>(q, k, v, a.beta, a.gate, a.S, o, a.dv, eb, wb);
        break;
    default:
        decode_kernel<DK, DVC, TIn, LDN_KDA><<<grid, kDecThreads, 0, st>>>(q, k, v, a.beta, a.gate, a.S, o, a.dv, eb, wb);
        break;
    }
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t st)
{
    if (a.dk == 128) return launch_cfg<128, 64, TIn>(a, st);
    return launch_cfg<64, 32, TIn>(a, st);   // dk = 64 (dv is 64 or 128)
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st)
{
    return a.dtype == LDN_BF16 ? launch_t<__nv_bfloat16>(a, st) : launch_t<float>(a, st);
}

cudaError_t launch_decode_steps(const DecodeArgs &a, int nsteps, cudaStream_t st)
{
    if (a.dtype == LDN_BF16)
        return a.dk == 128 ? launch_steps_cfg<128, 64, __nv_bfloat16>(a, nsteps, st)
                           : launch_steps_cfg<64, 32, __nv_bfloat16>(a, nsteps, st);
    return a.dk == 128 ? launch_steps_cfg<128, 64, float>(a, nsteps, st) : launch_steps_cfg<64, 32, float>(a, nsteps, st);
}

}  // namespace ldn
