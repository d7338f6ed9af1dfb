// Backward of the DeltaNet / Gated DeltaNet / KDA recurrence: gradients of
// L = sum_t <dO_t, o_t> + <dS_final, S_T> with respect to q, k, v, beta, the
// log-decay gates and the initial state, fp32 arithmetic.
//
// Per token, in memory orientation (H = S^T, [dk][dv]) and per value column i
// (the columns are independent linear systems, state-reduction notes Sec. 2.5):
//   h' = D_t h_{t-1},  p = k . h',  r = beta (v_i - p),  h_t = h' + r k,  o_i = q . h_t
// and in reverse, with g = dL/dh_t:
//   g += dO_i q                 dq  += dO_i h_t           (summed over columns)
//   dr = k . g                  dv_i = beta dr            dbeta += dr (v_i - p)
//   dp = -beta dr               dk  += r g + dp h'        (summed over columns)
//   g' = g + dp k               dgate: KDA g' * h' per key channel, GDN the sum
//   g  <- D_t g'                (so g = dL/dh_{t-1})
// (the linear-attention notes, Sec. 2.3-2.5, give the forward rules; the
// benchmark's method sources keep the whole state history for their KDA
// first-order backward, this kernel keeps every eighth state and recomputes
// the rest).
//
// Work split: one CTA of 256 threads per (b, h, 32-column slice of dv).  Lane
// l of warp w owns value column 4w + (l & 3) and the key rows 8j + (l >> 2),
// j < dk / 8, in registers: reductions over the rows (p, dr) are shuffles
// across lanes 4 apart, reductions over the columns (dq, dk, dgate, dbeta) are
// a two-step halving exchange across the 4 lanes of a row group, then
// shared-memory adds across the 8 warps, then a plain store of the slice's
// partial sums; a second kernel adds the slices.
//   Phase 1 walks the sequence forward and stores the state before every block
//   of 8 tokens (workspace).
//   Phase 2 walks the blocks in reverse: it reloads the block's checkpoint,
//   recomputes the block's decayed states h' into a shared-memory ring
//   (thread-private slots), then steps the 8 tokens backward.
#include "ldn_internal.cuh"

namespace ldn {
namespace {

constexpr int kNC = 32;     // value columns per CTA
constexpr int kBT = 256;    // threads per CTA
constexpr int kSub = 8;     // tokens per recomputed block

template <int DK>
struct BwdSmem {
    static constexpr int RPT = DK / 8;                                   // rows per thread
    static constexpr size_t ring = (size_t)kSub * RPT * kBT;            // decayed states h'
    static constexpr size_t floats = ring + 3 * kSub * DK /*q, k, a*/ + 2 * kSub * kNC /*v, dO*/ +
                                     kSub /*beta*/ + 3 * kSub * DK /*sums dq, dk, dg*/ + kSub /*sum dbeta*/;
    static constexpr size_t bytes = floats * sizeof(float);
};

// Sum of v[0..N) over the 4 lanes that differ in bits 0-1 (the 4 columns of a
// row group), by halving exchanges: on return u[0..N/4) holds the sums of rows
// j = i + (N/2) (lane & 1) + (N/4) ((lane >> 1) & 1).
template <int N>
__device__ __forceinline__ void sum_over_columns(const float (&v)[N], float (&u)[N / 4], int lane)
{
    float h[N / 2];
    const bool hi1 = lane & 1, hi2 = lane & 2;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = hi1 ? v[i] : v[i + N / 2];
        const float keep = hi1 ? v[i + N / 2] : v[i];
        h[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        const float send = hi2 ? h[i] : h[i + N / 4];
        const float keep = hi2 ? h[i + N / 4] : h[i];
        u[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
}

template <int DK, typename TIn, int MODE>
__global__ void __launch_bounds__(kBT, 1)
bwd_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
           const float *__restrict__ beta, const float *__restrict__ gate, const float *__restrict__ S0,
           const TIn *__restrict__ dout, const float *__restrict__ dSf, float *__restrict__ dv_out,
           float *__restrict__ dS0, float *__restrict__ ckpt, float *__restrict__ part, int T, int H, int dv)
{
    constexpr int RPT = DK / 8;
    constexpr int GW = MODE == LDN_KDA ? DK : (MODE == LDN_GDN ? 1 : 0);   // gate width
    extern __shared__ float smb[];
    float *ring = smb;                          // [kSub][RPT][kBT]
    float *qs = ring + BwdSmem<DK>::ring;       // [kSub][DK]
    float *ks = qs + kSub * DK;                 // [kSub][DK]
    float *as = ks + kSub * DK;                 // [kSub][DK] decay factor (GDN: [t][0])
    float *vs = as + kSub * DK;                 // [kSub][kNC]
    float *ds = vs + kSub * kNC;                // [kSub][kNC] dO
    float *bs = ds + kSub * kNC;                // [kSub]
    float *aq = bs + kSub;                      // [kSub][DK] column sums of this CTA
    float *ak = aq + kSub * DK;
    float *ag = ak + kSub * DK;
    float *ab = ag + kSub * DK;                 // [kSub]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = lane >> 2;                   // row group: rows 8 j + rg
    const int c = 4 * warp + (lane & 3);        // column within the slice
    const int slices = dv / kNC;
    const int unit = blockIdx.x / slices, sl = blockIdx.x % slices;
    const int b = unit / H, h = unit % H;
    const int col = sl * kNC + c;
    const int nsub = (T + kSub - 1) / kSub;
    const size_t N = (size_t)gridDim.x / slices * T;   // token-heads (B * H * T)
    float *myck = ckpt + (size_t)blockIdx.x * nsub * RPT * kBT;

    auto tok = [&](int t) { return ((size_t)b * T + t) * H + h; };
    // Inputs of block s into shared memory (rows past T: zero, decay 1).
    auto stage = [&](int s, bool grads) {
        const int t0 = s * kSub;
        for (int e = tid; e < kSub * DK; e += kBT) {
            const int t = e / DK, r = e % DK;
            const bool ok = t0 + t < T;
            const size_t i = tok(ok ? t0 + t : 0) * DK + r;
            ks[e] = ok ? load_in(k, i) : 0.f;
            if (grads) qs[e] = ok ? load_in(q, i) : 0.f;
            if (MODE == LDN_KDA) as[e] = ok ? expf(gate[i]) : 1.f;
        }
        for (int e = tid; e < kSub * kNC; e += kBT) {
            const int t = e / kNC, n = e % kNC;
            const bool ok = t0 + t < T;
            const size_t i = tok(ok ? t0 + t : 0) * dv + sl * kNC + n;
            vs[e] = ok ? load_in(v, i) : 0.f;
            if (grads) ds[e] = ok ? load_in(dout, i) : 0.f;
        }
        if (tid < kSub) {
            const bool ok = t0 + tid < T;
            const size_t i = tok(ok ? t0 + tid : 0);
            bs[tid] = ok ? beta[i] : 0.f;
            if (MODE == LDN_GDN) as[tid * DK] = ok ? expf(gate[i]) : 1.f;
        }
        if (grads)
            for (int e = tid; e < 3 * kSub * DK + kSub; e += kBT) aq[e] = 0.f;   // aq, ak, ag, ab
    };
    auto decay = [&](int t, int j) -> float {
        return MODE == LDN_KDA ? as[t * DK + 8 * j + rg] : (MODE == LDN_GDN ? as[t * DK] : 1.f);
    };
    // One forward token step on the thread's state rows; returns r and v - p.
    auto fwd_step = [&](int t, float (&hr)[RPT], float &r, float &e) {
        float p = 0.f;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            hr[j] *= decay(t, j);
            p += hr[j] * ks[t * DK + 8 * j + rg];
        }
        p += __shfl_xor_sync(0xffffffffu, p, 4);
        p += __shfl_xor_sync(0xffffffffu, p, 8);
        p += __shfl_xor_sync(0xffffffffu, p, 16);
        e = vs[t * kNC + c] - p;
        r = bs[t] * e;
#pragma unroll
        for (int j = 0; j < RPT; ++j) hr[j] += ks[t * DK + 8 * j + rg] * r;
    };

    // ---- phase 1: forward, checkpoint before every block
    float hr[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) hr[j] = S0 ? S0[((size_t)unit * DK + 8 * j + rg) * dv + col] : 0.f;
    for (int s = 0; s < nsub; ++s) {
        __syncthreads();
        stage(s, false);
        __syncthreads();
#pragma unroll
        for (int j = 0; j < RPT; ++j) myck[((size_t)s * RPT + j) * kBT + tid] = hr[j];
#pragma unroll
        for (int t = 0; t < kSub; ++t) {
            float r, e;
            fwd_step(t, hr, r, e);
        }
    }

    // ---- phase 2: blocks in reverse
    float g[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) g[j] = dSf ? dSf[((size_t)unit * DK + 8 * j + rg) * dv + col] : 0.f;
    float *pq = part, *pk = pq + (size_t)slices * N * DK, *pg = pk + (size_t)slices * N * DK;
    float *pb = pg + (size_t)slices * N * GW;
    for (int s = nsub - 1; s >= 0; --s) {
        const int t0 = s * kSub;
        __syncthreads();
        stage(s, true);
        __syncthreads();
#pragma unroll
        for (int j = 0; j < RPT; ++j) hr[j] = myck[((size_t)s * RPT + j) * kBT + tid];
        float rr[kSub], ee[kSub];
#pragma unroll
        for (int t = 0; t < kSub; ++t) {
            // h' of token t is the state after the decay, before the write
#pragma unroll
            for (int j = 0; j < RPT; ++j) ring[((size_t)t * RPT + j) * kBT + tid] = hr[j] * decay(t, j);
            fwd_step(t, hr, rr[t], ee[t]);
        }
#pragma unroll
        for (int t = kSub - 1; t >= 0; --t) {
            if (t0 + t >= T) continue;   // uniform over the CTA
            const float dO = ds[t * kNC + c], bt = bs[t];
            float hp[RPT], vq[RPT], vk[RPT], vg[RPT];
            float dr = 0.f;
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const int row = 8 * j + rg;
                const float kr = ks[t * DK + row];
                hp[j] = ring[((size_t)t * RPT + j) * kBT + tid];
                vq[j] = (hp[j] + kr * rr[t]) * dO;       // h_t * dO
                g[j] += qs[t * DK + row] * dO;
                dr += g[j] * kr;
            }
            dr += __shfl_xor_sync(0xffffffffu, dr, 4);
            dr += __shfl_xor_sync(0xffffffffu, dr, 8);
            dr += __shfl_xor_sync(0xffffffffu, dr, 16);
            if (rg == 0) dv_out[tok(t0 + t) * dv + col] = bt * dr;
            const float dp = -bt * dr;
            float gsum = 0.f;
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const float kr = ks[t * DK + 8 * j + rg];
                vk[j] = g[j] * rr[t] + hp[j] * dp;
                g[j] += kr * dp;                         // dL/dh'
                vg[j] = g[j] * hp[j];
                gsum += vg[j];
            }
            // column sums: dq, dk (and dgate for KDA) per row, dbeta and the GDN dgate per token
            float uq[RPT / 4], uk[RPT / 4], ug[RPT / 4];
            sum_over_columns<RPT>(vq, uq, lane);
            sum_over_columns<RPT>(vk, uk, lane);
            if (MODE == LDN_KDA) sum_over_columns<RPT>(vg, ug, lane);
            const int jo = (lane & 1) * (RPT / 2) + ((lane >> 1) & 1) * (RPT / 4);
#pragma unroll
            for (int i = 0; i < RPT / 4; ++i) {
                const int row = 8 * (jo + i) + rg;
                atomicAdd(&aq[t * DK + row], uq[i]);
                atomicAdd(&ak[t * DK + row], uk[i]);
                if (MODE == LDN_KDA) atomicAdd(&ag[t * DK + row], ug[i]);
            }
            float db = rg == 0 ? dr * ee[t] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                db += __shfl_xor_sync(0xffffffffu, db, o);
                if (MODE == LDN_GDN) gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
            }
            if (lane == 0) {
                atomicAdd(&ab[t], db);
                if (MODE == LDN_GDN) atomicAdd(&ag[t * DK], gsum);
            }
#pragma unroll
            for (int j = 0; j < RPT; ++j) g[j] *= decay(t, j);   // dL/dh_{t-1}
        }
        __syncthreads();
        // this slice's partial sums of block s
        for (int e = tid; e < kSub * DK; e += kBT) {
            const int t = e / DK, r = e % DK;
            if (t0 + t >= T) continue;
            const size_t n = tok(t0 + t);
            pq[((size_t)sl * N + n) * DK + r] = aq[e];
            pk[((size_t)sl * N + n) * DK + r] = ak[e];
            if (MODE == LDN_KDA) pg[((size_t)sl * N + n) * DK + r] = ag[e];
        }
        if (tid < kSub && t0 + tid < T) {
            const size_t n = tok(t0 + tid);
            pb[(size_t)sl * N + n] = ab[tid];
            if (MODE == LDN_GDN) pg[(size_t)sl * N + n] = ag[tid * DK];
        }
    }
#pragma unroll
    for (int j = 0; j < RPT; ++j) dS0[((size_t)unit * DK + 8 * j + rg) * dv + col] = g[j];
}

// Sum of the slices' partial sums: dq, dk [N][dk], dgate [N][gw], dbeta [N].
__global__ void bwd_reduce_kernel(const float *__restrict__ part, float *__restrict__ dq, float *__restrict__ dk,
                                  float *__restrict__ dg, float *__restrict__ db, long long N, int DK, int gw,
                                  int slices)
{
    const long long per = 2LL * DK + gw + 1;   // values per token-head
    const long long total = N * per;
    const float *pq = part, *pk = pq + (size_t)slices * N * DK, *pg = pk + (size_t)slices * N * DK;
    const float *pb = pg + (size_t)slices * N * gw;
    for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < total;
         x += (long long)gridDim.x * blockDim.x) {
        const float *src;
        float *dst;
        long long i, stride;
        if (x < N * DK) { i = x; src = pq; dst = dq; stride = N * DK; }
        else if (x < 2 * N * DK) { i = x - N * DK; src = pk; dst = dk; stride = N * DK; }
        else if (x < (2LL * DK + gw) * N) { i = x - 2 * N * DK; src = pg; dst = dg; stride = N * gw; }
        else { i = x - (2LL * DK + gw) * N; src = pb; dst = db; stride = N; }
        float s = 0.f;
        for (int sl = 0; sl < slices; ++sl) s += src[sl * stride + i];
        dst[i] = s;
    }
}

template <int DK, typename TIn, int MODE>
cudaError_t launch_mode(const BwdArgs &a, cudaStream_t st)
{
    auto kern = bwd_kernel<DK, TIn, MODE>;
    const size_t smem = BwdSmem<DK>::bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int slices = a.dv / kNC;
    const unsigned grid = (unsigned)((long long)a.B * a.H * slices);
    float *ckpt = a.ws;
    float *part = ckpt + bwd_ckpt_floats(a.B, a.T, a.H, a.dk, a.dv);
    kern<<<grid, kBT, smem, st>>>((const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v, a.beta, a.gate, a.S0,
                                  (const TIn *)a.dout, a.dS_final, a.dv_out, a.dS0, ckpt, part, a.T, a.H, a.dv);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long N = (long long)a.B * a.T * a.H;
    const int gw = MODE == LDN_KDA ? DK : (MODE == LDN_GDN ? 1 : 0);
    const long long total = N * (2LL * DK + gw + 1);
    const long long blocks = std::min<long long>((total + 255) / 256, 152LL * 16);
    bwd_reduce_kernel<<<(unsigned)blocks, 256, 0, st>>>(part, a.dq, a.dk_out, a.dgate, a.dbeta, N, DK, gw, slices);
    return cudaGetLastError();
}

template <int DK, typename TIn>
cudaError_t launch_dk(const BwdArgs &a, cudaStream_t st)
{
    switch (a.mode) {
    case LDN_DELTANET: return launch_mode<DK, TIn, LDN_DELTANET>(a, st);
    case LDN_GDN: return launch_mode<DK, TIn, LDN_GDN>(a, st);
    default: return launch_mode<DK, TIn, LDN_KDA>(a, st);
    }
}

}  // namespace

size_t bwd_ckpt_floats(int B, int T, int H, int dk, int dv)
{
    const size_t nsub = (size_t)(T + kSub - 1) / kSub;
    return (size_t)B * H * dv * nsub * dk;   // per CTA: nsub x dk x 32 (dv / 32 CTAs per head)
}

size_t bwd_workspace_bytes(int B, int T, int H, int dk, int dv, int mode)
{
    const size_t N = (size_t)B * T * H, slices = (size_t)dv / kNC;
    const size_t gw = mode == LDN_KDA ? (size_t)dk : (mode == LDN_GDN ? 1 : 0);
    return (bwd_ckpt_floats(B, T, H, dk, dv) + slices * N * (2 * (size_t)dk + gw + 1)) * sizeof(float);
}

cudaError_t launch_backward(const BwdArgs &a, cudaStream_t st)
{
    if (a.dtype == LDN_BF16)
        return a.dk == 128 ? launch_dk<128, __nv_bfloat16>(a, st) : launch_dk<64, __nv_bfloat16>(a, st);
    return a.dk == 128 ? launch_dk<128, float>(a, st) : launch_dk<64, float>(a, st);
}

}  // namespace ldn
