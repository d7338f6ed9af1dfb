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
// l of warp w owns value column l and the key rows w * dk/8 + j, j < dk/8, in
// registers, so every lane of a warp reads the same rows of q, k and the gates
// (shared-memory broadcasts).  Reductions over the rows (p, dr) are a partial
// sum per warp, one exchange through a double-buffered shared array and one
// barrier per token.  Reductions over the columns (dq, dk and the KDA gate
// gradient, per row) are a reduce-scatter across the 32 lanes of the warp that
// owns the rows, so each row has one writer and no atomics are needed; the
// scalar sums (dbeta, the GDN gate gradient) are warp sums.  Each slice stores
// its partial sums; a second kernel adds the slices.
//   Phase 1 (its own launch: small shared memory, several CTAs per SM) walks the
//   sequence forward and stores the state before every block of 8 tokens
//   (workspace).
//   Phase 2 walks the blocks in reverse: it reloads the block's checkpoint,
//   recomputes the block's decayed states h' into a shared-memory ring
//   (thread-private slots), then steps the 8 tokens backward.
#include "ldn_internal.cuh"

namespace ldn {
namespace {

constexpr int kNC = 32;     // value columns per CTA (one per lane)
constexpr int kBT = 256;    // threads per CTA
constexpr int kNW = kBT / 32;
constexpr int kSub = 8;     // tokens per recomputed block

template <int DK, int PHASE = 2>
struct BwdSmem {
    static constexpr int RPT = DK / kNW;                                 // rows per thread (and per warp)
    static constexpr size_t ring = PHASE == 2 ? (size_t)kSub * RPT * kBT : 0;   // decayed states h'
    // one block's inputs: q, k, a [kSub][DK], v, dO [kSub][kNC], beta [kSub] (two buffers)
    static constexpr size_t stage = 3 * kSub * DK + 2 * kSub * kNC + kSub;
    static constexpr size_t floats = ring + 2 * stage + 3 * kSub * DK /*sums dq, dk, dg*/ + kSub /*sum dbeta*/ +
                                     kSub * kNW /*GDN gate-gradient warp sums*/ + 2 * kNW * kNC /*row sums*/;
    static constexpr size_t bytes = floats * sizeof(float);
};

// Reduce-scatter of v[0..N) over the 32 lanes of a warp (N = 16 or 8): on
// return every lane holds the warp-wide sum of one row, row j(lane) (the lanes
// sharing a row hold the same value); see row_of.
template <int N>
__device__ __forceinline__ float sum_over_lanes(const float (&v)[N], int lane)
{
    float a[N / 2];
    const bool u16 = lane & 16;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = u16 ? v[i] : v[i + N / 2];
        const float keep = u16 ? v[i + N / 2] : v[i];
        a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float b[N / 4];
    const bool u8 = lane & 8;
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        const float send = u8 ? a[i] : a[i + N / 4];
        const float keep = u8 ? a[i + N / 4] : a[i];
        b[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float c[N / 8];
    const bool u4 = lane & 4;
#pragma unroll
    for (int i = 0; i < N / 8; ++i) {
        const float send = u4 ? b[i] : b[i + N / 8];
        const float keep = u4 ? b[i + N / 8] : b[i];
        c[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float x;
    if constexpr (N == 16) {
        const bool u2 = lane & 2;
        x = (u2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, u2 ? c[0] : c[1], 2);
        x += __shfl_xor_sync(0xffffffffu, x, 1);
    } else {
        x = c[0];
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 1);
    }
    return x;
}
// The row whose sum lane `lane` holds after sum_over_lanes<N>, and whether it
// is the lane that stores it.
template <int N>
__device__ __forceinline__ int row_of(int lane)
{
    const int j = (N / 2) * ((lane >> 4) & 1) + (N / 4) * ((lane >> 3) & 1) + (N / 8) * ((lane >> 2) & 1);
    return N == 16 ? j + ((lane >> 1) & 1) : j;
}
template <int N>
__device__ __forceinline__ bool row_writer(int lane) { return N == 16 ? (lane & 1) == 0 : (lane & 3) == 0; }

template <int DK, typename TIn, int MODE, int PHASE>
__global__ void __launch_bounds__(kBT, PHASE == 1 ? 3 : 1)
bwd_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
           const float *__restrict__ beta, const float *__restrict__ gate, const float *__restrict__ S0,
           const TIn *__restrict__ dout, const float *__restrict__ dSf, float *__restrict__ dv_out,
           float *__restrict__ dS0, float *__restrict__ ckpt, float *__restrict__ part, int T, int H, int dv)
{
    using SM = BwdSmem<DK, PHASE>;
    constexpr int RPT = SM::RPT;
    constexpr int GW = MODE == LDN_KDA ? DK : (MODE == LDN_GDN ? 1 : 0);   // gate width
    extern __shared__ float smb[];
    float *ring = smb;                          // [kSub][RPT][kBT]
    float *stg = ring + SM::ring;      // 2 x one block's inputs
    // the current block's inputs (reassigned per block):
    float *qs, *ks, *as, *vs, *ds, *bs;         // q, k [kSub][DK], decay [kSub][DK] (GDN [t][0]),
                                                // v, dO [kSub][kNC], beta [kSub]
    auto use_buffer = [&](int buf) {
        qs = stg + buf * SM::stage;
        ks = qs + kSub * DK;
        as = ks + kSub * DK;
        vs = as + kSub * DK;
        ds = vs + kSub * kNC;
        bs = ds + kSub * kNC;
    };
    float *aq = stg + 2 * SM::stage;   // [kSub][DK] column sums of this CTA
    float *ak = aq + kSub * DK;
    float *ag = ak + kSub * DK;
    float *ab = ag + kSub * DK;                 // [kSub]
    float *agw = ab + kSub;                     // [kSub][kNW] GDN gate gradient per warp
    float *red = agw + kSub * kNW;              // [2][kNW][kNC] row-sum exchange

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = warp * RPT;                  // first key row of this warp
    const int slices = dv / kNC;
    const int unit = blockIdx.x / slices, sl = blockIdx.x % slices;
    const int b = unit / H, h = unit % H;
    const int col = sl * kNC + lane;
    const int nsub = (T + kSub - 1) / kSub;
    const size_t N = (size_t)gridDim.x / slices * T;   // token-heads (B * H * T)
    float *myck = ckpt + (size_t)blockIdx.x * nsub * RPT * kBT;
    int par = 0;                                // parity of the row-sum buffer

    auto tok = [&](int t) { return ((size_t)b * T + t) * H + h; };
    // A block's inputs travel global -> registers (issued a block ahead, so their
    // latency overlaps the current block) -> shared buffer (rows past T: zero, log-decay 0).
    constexpr int NKQ = kSub * DK / kBT;        // q, k, gate elements per thread
    static_assert(kSub * kNC == kBT, "one v / dO element per thread");
    struct Pre { float k[NKQ], q[NKQ], a[NKQ], v, d, b, g; };
    auto pre_load = [&](int s, bool grads, Pre &P) {
        const int t0 = s * kSub;
#pragma unroll
        for (int x = 0; x < NKQ; ++x) {
            const int e = tid + x * kBT, t = e / DK, r = e % DK;
            const bool ok = t0 + t < T;
            const size_t i = tok(ok ? t0 + t : 0) * DK + r;
            P.k[x] = ok ? load_in(k, i) : 0.f;
            P.q[x] = grads && ok ? load_in(q, i) : 0.f;
            P.a[x] = MODE == LDN_KDA && ok ? gate[i] : 0.f;
        }
        {
            const int t = tid / kNC, n = tid % kNC;
            const bool ok = t0 + t < T;
            const size_t i = tok(ok ? t0 + t : 0) * dv + sl * kNC + n;
            P.v = ok ? load_in(v, i) : 0.f;
            P.d = grads && ok ? load_in(dout, i) : 0.f;
        }
        P.b = P.g = 0.f;
        if (tid < kSub && t0 + tid < T) {
            const size_t i = tok(t0 + tid);
            P.b = beta[i];
            if (MODE == LDN_GDN) P.g = gate[i];
        }
    };
    auto pre_store = [&](int buf, bool grads, const Pre &P) {
        float *q_ = stg + buf * SM::stage, *k_ = q_ + kSub * DK, *a_ = k_ + kSub * DK;
        float *v_ = a_ + kSub * DK, *d_ = v_ + kSub * kNC, *b_ = d_ + kSub * kNC;
#pragma unroll
        for (int x = 0; x < NKQ; ++x) {
            const int e = tid + x * kBT;
            k_[e] = P.k[x];
            if (grads) q_[e] = P.q[x];
            if (MODE == LDN_KDA) a_[e] = expf(P.a[x]);
        }
        v_[tid] = P.v;
        if (grads) d_[tid] = P.d;
        if (tid < kSub) {
            b_[tid] = P.b;
            if (MODE == LDN_GDN) a_[tid * DK] = expf(P.g);
        }
    };
    // this warp's RPT rows of a [kSub][DK] input at token t (16-byte aligned): vector loads
    auto rows = [&](const float *base, int t, float (&x)[RPT]) {
#pragma unroll
        for (int j = 0; j < RPT; j += 4) {
            const float4 v4 = *reinterpret_cast<const float4 *>(base + t * DK + r0 + j);
            x[j] = v4.x; x[j + 1] = v4.y; x[j + 2] = v4.z; x[j + 3] = v4.w;
        }
    };
    auto decays = [&](int t, float (&x)[RPT]) {
        if constexpr (MODE == LDN_KDA) {
            rows(as, t, x);
        } else {
#pragma unroll
            for (int j = 0; j < RPT; ++j) x[j] = MODE == LDN_GDN ? as[t * DK] : 1.f;
        }
    };
    // Sum over the key rows of this thread's column (all warps): one barrier.
    auto row_sum = [&](float x) -> float {
        float *rb = red + par * kNW * kNC;
        rb[warp * kNC + lane] = x;
        __syncthreads();
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kNW; ++w) s += rb[w * kNC + lane];
        par ^= 1;
        return s;
    };
    // One forward token step on the thread's state rows; returns r and v - p.
    auto fwd_step = [&](int t, float (&hr)[RPT], float &r, float &e) {
        float kr[RPT], ar[RPT];
        rows(ks, t, kr);
        decays(t, ar);
        float p = 0.f;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            hr[j] *= ar[j];
            p += hr[j] * kr[j];
        }
        p = row_sum(p);
        e = vs[t * kNC + lane] - p;
        r = bs[t] * e;
#pragma unroll
        for (int j = 0; j < RPT; ++j) hr[j] += kr[j] * r;
    };

    float hr[RPT];
    Pre P;
    if constexpr (PHASE == 1) {
    // ---- phase 1: forward, checkpoint before every block
#pragma unroll
    for (int j = 0; j < RPT; ++j) hr[j] = S0 ? S0[((size_t)unit * DK + r0 + j) * dv + col] : 0.f;
    if (nsub > 0) {
        pre_load(0, false, P);
        pre_store(0, false, P);
    }
    for (int s = 0; s < nsub; ++s) {
        __syncthreads();                        // block s staged; block s - 1 done with the other buffer
        use_buffer(s & 1);
        if (s + 1 < nsub) pre_load(s + 1, false, P);
#pragma unroll
        for (int j = 0; j < RPT; ++j) myck[((size_t)s * RPT + j) * kBT + tid] = hr[j];
#pragma unroll
        for (int t = 0; t < kSub; ++t) {
            float r, e;
            fwd_step(t, hr, r, e);
        }
        if (s + 1 < nsub) pre_store((s + 1) & 1, false, P);
    }
    } else {
    // ---- phase 2: blocks in reverse
    float g[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) g[j] = dSf ? dSf[((size_t)unit * DK + r0 + j) * dv + col] : 0.f;
    float *pq = part, *pk = pq + (size_t)slices * N * DK, *pg = pk + (size_t)slices * N * DK;
    float *pb = pg + (size_t)slices * N * GW;
    const int jrow = row_of<RPT>(lane);
    const bool writer = row_writer<RPT>(lane);
    float hn[RPT];                              // state copy of the next block to run
    if (nsub > 0) {
        pre_load(nsub - 1, true, P);
        pre_store((nsub - 1) & 1, true, P);
#pragma unroll
        for (int j = 0; j < RPT; ++j) hn[j] = myck[((size_t)(nsub - 1) * RPT + j) * kBT + tid];
    }
    for (int s = nsub - 1; s >= 0; --s) {
        const int t0 = s * kSub;
        __syncthreads();                        // block s staged; block s + 1 flushed
        use_buffer(s & 1);
#pragma unroll
        for (int j = 0; j < RPT; ++j) hr[j] = hn[j];
        if (s > 0) {
            pre_load(s - 1, true, P);
#pragma unroll
            for (int j = 0; j < RPT; ++j) hn[j] = myck[((size_t)(s - 1) * RPT + j) * kBT + tid];
        }
        float rr[kSub], ee[kSub];
#pragma unroll
        for (int t = 0; t < kSub; ++t) {
            // h' of token t is the state after the decay, before the write
            float ar[RPT];
            decays(t, ar);
#pragma unroll
            for (int j = 0; j < RPT; ++j) ring[((size_t)t * RPT + j) * kBT + tid] = hr[j] * ar[j];
            fwd_step(t, hr, rr[t], ee[t]);
        }
#pragma unroll
        for (int t = kSub - 1; t >= 0; --t) {
            if (t0 + t >= T) continue;   // uniform over the CTA
            const float dO = ds[t * kNC + lane], bt = bs[t];
            float hp[RPT], vq[RPT], vk[RPT], vg[RPT], kr[RPT], qr[RPT];
            rows(ks, t, kr);
            rows(qs, t, qr);
            float dr = 0.f;
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                hp[j] = ring[((size_t)t * RPT + j) * kBT + tid];
                vq[j] = (hp[j] + kr[j] * rr[t]) * dO;    // h_t * dO
                g[j] += qr[j] * dO;
                dr += g[j] * kr[j];
            }
            dr = row_sum(dr);
            if (warp == 0) dv_out[tok(t0 + t) * dv + col] = bt * dr;
            const float dp = -bt * dr;
            float gsum = 0.f;
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                vk[j] = g[j] * rr[t] + hp[j] * dp;
                g[j] += kr[j] * dp;                      // dL/dh'
                vg[j] = g[j] * hp[j];
                gsum += vg[j];
            }
            // column sums of this warp's rows: one writer per row
            const float sq = sum_over_lanes<RPT>(vq, lane);
            const float sk = sum_over_lanes<RPT>(vk, lane);
            if (writer) {
                aq[t * DK + r0 + jrow] = sq;
                ak[t * DK + r0 + jrow] = sk;
            }
            if (MODE == LDN_KDA) {
                const float sg = sum_over_lanes<RPT>(vg, lane);
                if (writer) ag[t * DK + r0 + jrow] = sg;
            }
            if (MODE == LDN_GDN) {
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
                if (lane == 0) agw[t * kNW + warp] = gsum;
            }
            if (warp == 0) {   // dbeta: every warp holds the same dr; warp 0 sums the columns
                float db = dr * ee[t];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) db += __shfl_xor_sync(0xffffffffu, db, o);
                if (lane == 0) ab[t] = db;
            }
            float ar[RPT];
            decays(t, ar);
#pragma unroll
            for (int j = 0; j < RPT; ++j) g[j] *= ar[j];         // dL/dh_{t-1}
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
            if (MODE == LDN_GDN) {
                float sg = 0.f;
#pragma unroll
                for (int w = 0; w < kNW; ++w) sg += agw[tid * kNW + w];
                pg[(size_t)sl * N + n] = sg;
            }
        }
        if (s > 0) pre_store((s - 1) & 1, true, P);
    }
#pragma unroll
    for (int j = 0; j < RPT; ++j) dS0[((size_t)unit * DK + r0 + j) * dv + col] = g[j];
    }
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
    const int slices = a.dv / kNC;
    const unsigned grid = (unsigned)((long long)a.B * a.H * slices);
    float *ckpt = a.ws;
    float *part = ckpt + bwd_ckpt_floats(a.B, a.T, a.H, a.dk, a.dv);
    auto k1 = bwd_kernel<DK, TIn, MODE, 1>;
    auto k2 = bwd_kernel<DK, TIn, MODE, 2>;
    cudaError_t e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdSmem<DK, 2>::bytes);
    if (e != cudaSuccess) return e;
    k1<<<grid, kBT, BwdSmem<DK, 1>::bytes, st>>>((const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v, a.beta, a.gate,
                                                  a.S0, (const TIn *)a.dout, a.dS_final, a.dv_out, a.dS0, ckpt, part,
                                                  a.T, a.H, a.dv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k2<<<grid, kBT, BwdSmem<DK, 2>::bytes, st>>>((const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v, a.beta, a.gate,
                                                  a.S0, (const TIn *)a.dout, a.dS_final, a.dv_out, a.dS0, ckpt, part,
                                                  a.T, a.H, a.dv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
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
