// The steps on either side of the chunkwise path, as HBM-streaming kernels:
//   prologue -- q, k, v through a depthwise causal short convolution and SiLU
//               (the model-zoo page: DeltaNet "causal convolution plus SiLU",
//               KDA "short convolution"; the backend notes: causal_conv1d with
//               the SiLU activation), q and k L2-normalised per head, beta =
//               sigmoid(logit), and the Mamba2-style decay gate log alpha =
//               -a softplus(z + b) (Residual Linear Attention notes, Sec. 3.2-3.4);
//   epilogue -- the gated RMSNorm of the output, per head over dv, times a
//               gain vector and SiLU of the output gate (model-zoo page, Gated
//               DeltaNet entry; the backend notes: rms_norm_gated).
//
// Each block stages its tile in shared memory with 16-byte cp.async copies
// (zero-filled outside the sequence; nothing held in registers while the bytes
// are in flight), then computes from there, so that several blocks per SM keep
// HBM busy.  Convolution: a block takes 32 tokens (16 for more than four taps) of
// a group of heads whose rows make 1 KB, and one of q, k, v -- the tile holds its
// W - 1 tokens of halo, so every input row is read once from HBM (and up to W - 1
// more times from L2) -- and a thread owns one 16-byte piece of a row (8 bf16 / 4
// fp32 channels): the W taps and SiLU in packed fp32x2 arithmetic, and for q and k
// the L2 norm as a shuffle sum over the head's threads.  The convolution kernel is
// issue-bound (ncu: 59% of issue slots at 30% occupancy before the packed form),
// so instructions per element are what the layout minimises.  Blocks are numbered
// with the head fastest, so neighbouring blocks read neighbouring rows.  The gates
// (one per (b, t, h)) ride in the convolution launch, each block taking a share
// while its tile's copies are in flight; KDA's per-channel gates, a stream as large
// as the convolutions', have a launch of their own.
// RMSNorm: a block takes 64 consecutive rows of o and the gate.  Arithmetic is
// fp32; values are stored in the tensor's dtype.
#include <algorithm>

#include "ldn_internal.cuh"
#include "sm100_ptx.cuh"

namespace ldn {
namespace {
using namespace sm100;

constexpr int kThreads = 256;
constexpr int kRun = 64;     // tokens per walker

__device__ __forceinline__ void ld4(const float *p, float *v)
{
    const float4 x = *reinterpret_cast<const float4 *>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void ld4(const __nv_bfloat16 *p, float *v)
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void st4(float *p, const float *v)
{
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void st4(__nv_bfloat16 *p, const float *v)
{
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

// The activations use CUDA's fast intrinsics (the kernels are issue-bound with
// the accurate functions); their error, a few 1e-7 relative, is far inside the
// 1e-5 (fp32) / bf16-rounding budget of the results.
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }
// log(1 + e^x); for x > 15 the correction log(1 + e^-x) is below fp32 resolution of x
__device__ __forceinline__ float softplus_f(float x) { return x > 15.f ? x : __logf(1.f + __expf(x)); }

// beta = sigmoid(logit) over nb values and, when g is given, one gate per (b, t, h):
// log alpha = -a[h] softplus(z + bias[h]).  A grid-stride loop (start, stride) with
// four independent elements per thread in flight.
struct GateArgs {
    const float *logit;
    float *beta;
    const float *z, *a, *bias;
    float *g;
    long long nb;
    int H;
};

constexpr int kGateUnroll = 4;

__device__ __forceinline__ void gates_work(const GateArgs &ga, long long start, long long stride)
{
    for (long long i0 = start; i0 < ga.nb; i0 += kGateUnroll * stride) {
        float lv[kGateUnroll];
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const long long i = i0 + u * stride;
            lv[u] = i < ga.nb ? __ldg(ga.logit + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const long long i = i0 + u * stride;
            if (i < ga.nb) ga.beta[i] = sigmoid_f(lv[u]);
        }
    }
    if (!ga.g) return;
    for (long long i0 = start; i0 < ga.nb; i0 += kGateUnroll * stride) {
        float zv[kGateUnroll];
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const long long i = i0 + u * stride;
            zv[u] = i < ga.nb ? __ldg(ga.z + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const long long i = i0 + u * stride;
            if (i >= ga.nb) continue;
            const int h = (int)(i % ga.H);
            ga.g[i] = -__ldg(ga.a + h) * softplus_f(zv[u] + __ldg(ga.bias + h));
        }
    }
}

// Up to three convolutions of one row width D in one launch (blockIdx.y picks q, k or v),
// and, when `gates` is set, the gates, spread over all the launch's blocks: y =
// silu(short_conv(x)), then (norm) divided by sqrt(sum of squares + eps) per row.  x, y
// [B][T][H][D]; w [H * D][W], tap W - 1 on the current token.
struct ConvBatch {
    const void *x[3];
    const float *w[3];
    void *y[3];
    int norm[3];
    int n;
    int gates;
    GateArgs ga;
};

// Convolution tile: kConvTok tokens (plus the W - 1 before them) of a group of
// HG = 1 KB / (D * element size) consecutive heads, so that each token row of the
// tile is 1 KB of contiguous memory, and the heads' weights.  blockIdx.x = (b, run,
// head group) with the head group fastest.  A thread owns one 16-byte piece of a head's
// row (VE channels); the D / VE threads of a head and the heads of the group make a
// walker of 64 threads, and the block's two walkers take half of the tile's tokens each,
// sliding a register window of the last WMAX input rows (one shared-memory read per
// row) through a fully unrolled token loop.
constexpr int kConvWalk = 2;
constexpr int kConvThreads = 128;
// tokens per tile: 32 for up to 4 taps, 16 for up to 8 (static shared memory stays under 48 KB)
template <int WMAX>
constexpr int conv_tok() { return WMAX <= 4 ? 32 : 16; }

template <int D, typename TIn>
constexpr int conv_heads() { return 1024 / (D * (int)sizeof(TIn)); }

template <typename TIn> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void ld(const float *p, float *v)
    {
        const float4 x = *reinterpret_cast<const float4 *>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
    static __device__ __forceinline__ void st(float *p, const float *v)
    {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void ld(const __nv_bfloat16 *p, float *v)
    {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(b[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, const float *v)
    {
        uint4 u;
        __nv_bfloat162 *b = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4 *>(p) = u;
    }
};

template <int D, int WMAX, typename TIn>
__global__ void __launch_bounds__(kConvThreads)
conv_silu_kernel(const ConvBatch cb, int B, int T, int H, int W, float eps)
{
    using V = Vec16<TIn>;
    constexpr int VE = V::N;                          // channels per thread
    constexpr int L = D / VE;                         // threads per head
    constexpr int HG = conv_heads<D, TIn>();
    static_assert(HG * L * kConvWalk == kConvThreads, "two walkers of 64 threads");
    constexpr int kConvTok = conv_tok<WMAX>();
    constexpr int kRows = kConvTok + WMAX - 1;        // tile rows: tokens t0 - (W-1) ...
    constexpr int kRowElems = HG * D;                 // one token of the head group
    constexpr int TPW = kConvTok / kConvWalk;         // tokens per walker
    __shared__ __align__(16) TIn tile[kRows * kRowElems];
    __shared__ __align__(16) float wsm[HG * D * WMAX];
    const int ts = blockIdx.y;   // selected without indexing, so that cb stays in parameter space
    const TIn *x = (const TIn *)(ts == 0 ? cb.x[0] : ts == 1 ? cb.x[1] : cb.x[2]);
    const float *w = ts == 0 ? cb.w[0] : ts == 1 ? cb.w[1] : cb.w[2];
    TIn *y = (TIn *)(ts == 0 ? cb.y[0] : ts == 1 ? cb.y[1] : cb.y[2]);
    const bool norm = (ts == 0 ? cb.norm[0] : ts == 1 ? cb.norm[1] : cb.norm[2]) != 0;
    const unsigned runs = (unsigned)(T + kConvTok - 1) / kConvTok;
    const unsigned groups = (unsigned)(H + HG - 1) / HG;
    const unsigned id = blockIdx.x;
    const int h0 = (int)(id % groups) * HG;
    const unsigned br = id / groups;
    const int t0 = (int)(br % runs) * kConvTok, b = (int)(br / runs);
    const size_t rs = (size_t)H * D;                                // elements between tokens
    const size_t base = ((size_t)b * T * H + h0) * D;              // token 0, head h0
    const int hvalid = min(HG, H - h0);
    const int tbase = t0 - (W - 1);
    for (int i = threadIdx.x; i < kRows * (kRowElems / VE); i += kConvThreads) {
        const int r = i / (kRowElems / VE), e = (i % (kRowElems / VE)) * VE;
        const int t = tbase + r;
        const bool ok = t >= 0 && t < T && e < hvalid * D;
        cp_async16(&tile[r * kRowElems + e], ok ? x + base + (size_t)t * rs + e : x, ok ? 16u : 0u);
    }
    cp_async_commit();
    // this block's share of the gates (grid-stride over every block of the launch), while the
    // tile's copies are in flight
    if (cb.gates)
        gates_work(cb.ga, ((long long)blockIdx.y * gridDim.x + blockIdx.x) * kConvThreads + threadIdx.x,
                   (long long)gridDim.x * gridDim.y * kConvThreads);
    // the group's weights (in memory W taps per channel, channels of heads h0 ..), stored tap
    // by tap: wsm[j][channel], so that a thread's VE channels of a tap are 16 / 32 contiguous bytes
    for (int c = threadIdx.x; c < hvalid * D; c += kConvThreads) {
        const float *wc = w + ((size_t)h0 * D + c) * W;
#pragma unroll
        for (int j = 0; j < WMAX; ++j)
            if (j < W) wsm[j * kRowElems + c] = __ldg(wc + j);
    }

    const int walker = threadIdx.x / (HG * L), r = threadIdx.x % (HG * L);
    const int hl = r / L, c0 = VE * (r % L), h = h0 + hl;
    const bool hok = h < H;
    cp_async_wait<0>();
    __syncthreads();
    // channel pairs in packed fp32x2 arithmetic (one instruction per pair)
    constexpr int VP = VE / 2;
    float2 wt[WMAX][VP];   // tap j multiplies tile row (output row + j)
#pragma unroll
    for (int j = 0; j < WMAX; ++j)
#pragma unroll
        for (int i = 0; i < VP; ++i) {
            const bool on = hok && j < W;
            wt[j][i] = on ? *reinterpret_cast<const float2 *>(&wsm[j * kRowElems + hl * D + c0 + 2 * i])
                          : make_float2(0.f, 0.f);
        }

    const int col = hl * D + c0, u0 = walker * TPW;
    float2 win[WMAX][VP];
#pragma unroll
    for (int j = 0; j < WMAX - 1; ++j) V::ld(&tile[(u0 + j) * kRowElems + col], reinterpret_cast<float *>(win[j]));
    TIn *yp = y + base + (size_t)(t0 + u0) * rs + col;
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
        V::ld(&tile[(u0 + u + WMAX - 1) * kRowElems + col], reinterpret_cast<float *>(win[WMAX - 1]));
        float2 acc[VP];
#pragma unroll
        for (int i = 0; i < VP; ++i) acc[i] = __fmul2_rn(wt[0][i], win[0][i]);
#pragma unroll
        for (int j = 1; j < WMAX; ++j)
#pragma unroll
            for (int i = 0; i < VP; ++i) acc[i] = __ffma2_rn(wt[j][i], win[j][i], acc[i]);
#pragma unroll
        for (int j = 0; j < WMAX - 1; ++j)
#pragma unroll
            for (int i = 0; i < VP; ++i) win[j][i] = win[j + 1][i];
        // silu(x) = x / (1 + e^-x)
#pragma unroll
        for (int i = 0; i < VP; ++i) {
            const float2 d = __fadd2_rn(make_float2(__expf(-acc[i].x), __expf(-acc[i].y)), make_float2(1.f, 1.f));
            acc[i] = __fmul2_rn(acc[i], make_float2(__fdividef(1.f, d.x), __fdividef(1.f, d.y)));
        }
        if (norm) {
            float2 s2 = __fmul2_rn(acc[0], acc[0]);
#pragma unroll
            for (int i = 1; i < VP; ++i) s2 = __ffma2_rn(acc[i], acc[i], s2);
            float ss = s2.x + s2.y;
#pragma unroll
            for (int o = L / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float sc = rsqrtf(ss + eps);
#pragma unroll
            for (int i = 0; i < VP; ++i) acc[i] = __fmul2_rn(acc[i], make_float2(sc, sc));
        }
        if (hok && t0 + u0 + u < T) V::st(yp, reinterpret_cast<const float *>(acc));
        yp += rs;
    }
}

// The gates as a kernel of their own (KDA: dk per-channel gates per (b, t, h), a stream
// as large as the convolutions' that wants every block of the GPU): as gates_work, each
// thread taking kGateUnroll independent elements.  Idx is 32-bit unless the tensors need
// more.

template <int PER4, typename Idx>
__global__ void __launch_bounds__(kThreads)
gates_kernel(const float *__restrict__ logit, float *__restrict__ beta, Idx nb, const float *__restrict__ z,
             const float *__restrict__ a, const float *__restrict__ bias, float *__restrict__ g, int H)
{
    const Idx base = (Idx)blockIdx.x * (kThreads * kGateUnroll) + threadIdx.x;
    float lv[kGateUnroll];
#pragma unroll
    for (int u = 0; u < kGateUnroll; ++u) {
        const Idx i = base + (Idx)u * kThreads;
        lv[u] = i < nb ? logit[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kGateUnroll; ++u) {
        const Idx i = base + (Idx)u * kThreads;
        if (i < nb) beta[i] = sigmoid_f(lv[u]);
    }
    if (!g) return;
    if constexpr (PER4 > 0) {
        const Idx n4 = nb * PER4;   // float4s of the per-channel gate tensor
        float4 zv[kGateUnroll];
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const Idx i = base + (Idx)u * kThreads;
            zv[u] = i < n4 ? reinterpret_cast<const float4 *>(z)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const Idx i = base + (Idx)u * kThreads;
            if (i >= n4) continue;
            const int c = 4 * (int)(i % PER4);
            const int h = (int)((i / PER4) % (Idx)H);
            const float4 bb = *reinterpret_cast<const float4 *>(bias + (size_t)h * (4 * PER4) + c);
            const float ah = a[h];
            reinterpret_cast<float4 *>(g)[i] = make_float4(-ah * softplus_f(zv[u].x + bb.x), -ah * softplus_f(zv[u].y + bb.y),
                                                           -ah * softplus_f(zv[u].z + bb.z), -ah * softplus_f(zv[u].w + bb.w));
        }
    } else {
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const Idx i = base + (Idx)u * kThreads;
            lv[u] = i < nb ? z[i] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kGateUnroll; ++u) {
            const Idx i = base + (Idx)u * kThreads;
            if (i >= nb) continue;
            const int h = (int)(i % (Idx)H);
            g[i] = -a[h] * softplus_f(lv[u] + bias[h]);
        }
    }
}

template <typename Idx>
cudaError_t gates_launch(const PrologueArgs &a, cudaStream_t st)
{
    const Idx nb = (Idx)a.B * a.T * a.H;
    const bool kda = a.mode == LDN_KDA;
    const long long work = kda ? (long long)nb * (a.dk / 4) : (long long)nb;
    const unsigned blocks = (unsigned)std::max(1LL, (work + kThreads * kGateUnroll - 1) / (kThreads * kGateUnroll));
    float *g = a.mode == LDN_DELTANET ? nullptr : a.gate;
    if (!kda) gates_kernel<0, Idx><<<blocks, kThreads, 0, st>>>(a.beta_logit, a.beta, nb, a.gate_z, a.gate_a, a.gate_b, g, a.H);
    else if (a.dk == 128) gates_kernel<32, Idx><<<blocks, kThreads, 0, st>>>(a.beta_logit, a.beta, nb, a.gate_z, a.gate_a, a.gate_b, g, a.H);
    else gates_kernel<16, Idx><<<blocks, kThreads, 0, st>>>(a.beta_logit, a.beta, nb, a.gate_z, a.gate_a, a.gate_b, g, a.H);
    return cudaGetLastError();
}

// y = o / sqrt(mean(o^2) + eps) * weight * silu(g), per row of D values; a block
// stages kRows consecutive rows of o and g in shared memory (32 KB at most).
template <int D, typename TIn>
constexpr int rms_rows() { return 32768 / (2 * D * (int)sizeof(TIn)) < kRun ? 32768 / (2 * D * (int)sizeof(TIn)) : kRun; }

template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads)
rmsnorm_gated_kernel(const TIn *__restrict__ o, const TIn *__restrict__ gt, const float *__restrict__ weight,
                     TIn *__restrict__ y, long long rows, float eps)
{
    constexpr int kVec = 16 / sizeof(TIn);
    constexpr int L = D / 4, WPW = 32 / L;
    constexpr int kRows = rms_rows<D, TIn>();
    __shared__ __align__(16) TIn so[kRows * D];
    __shared__ __align__(16) TIn sg[kRows * D];
    const long long r0 = (long long)blockIdx.x * kRows;
    for (int i = threadIdx.x; i < kRows * (D / kVec); i += kThreads) {
        const int r = i / (D / kVec), cv = (i % (D / kVec)) * kVec;
        const bool ok = r0 + r < rows;
        const size_t off = ok ? (size_t)(r0 + r) * D + cv : 0;
        cp_async16(&so[r * D + cv], o + off, ok ? 16u : 0u);
        cp_async16(&sg[r * D + cv], gt + off, ok ? 16u : 0u);
    }
    cp_async_commit();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c0 = 4 * (lane % L);
    float wv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) wv[i] = weight[c0 + i];
    cp_async_wait<0>();
    __syncthreads();
#pragma unroll 2
    for (int lr = warp * WPW + lane / L; lr < kRows; lr += (kThreads / 32) * WPW) {
        float ov[4], gv[4];
        ld4(&so[lr * D + c0], ov);
        ld4(&sg[lr * D + c0], gv);
        float ss = ov[0] * ov[0] + ov[1] * ov[1] + ov[2] * ov[2] + ov[3] * ov[3];
#pragma unroll
        for (int s = L / 2; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
        const float rs = rsqrtf(ss * (1.f / D) + eps);
        float out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) out[i] = ov[i] * rs * wv[i] * silu_f(gv[i]);
        if (r0 + lr < rows) st4(y + (size_t)(r0 + lr) * D + c0, out);
    }
}

// Convolutions of the tensors in `sel` (all of row width d) in one launch, with the gates
// when `ga` is given.
template <typename TIn>
cudaError_t conv_launch(const PrologueArgs &a, const int *sel, int n, int d, const GateArgs *ga, cudaStream_t st)
{
    const void *xs[3] = {a.q_in, a.k_in, a.v_in};
    const float *ws[3] = {a.conv_q, a.conv_k, a.conv_v};
    void *ys[3] = {a.q, a.k, a.v};
    ConvBatch cb{};
    for (int i = 0; i < n; ++i) {
        cb.x[i] = xs[sel[i]];
        cb.w[i] = ws[sel[i]];
        cb.y[i] = ys[sel[i]];
        cb.norm[i] = sel[i] < 2;   // q and k are L2-normalised
    }
    cb.n = n;
    cb.gates = ga != nullptr;
    if (ga) cb.ga = *ga;
    const int hg = 1024 / (d * (int)sizeof(TIn));   // conv_heads
    const bool w4 = a.width <= 4;
    const int tok = w4 ? conv_tok<4>() : conv_tok<8>();
    const dim3 grid((unsigned)((long long)a.B * ((a.H + hg - 1) / hg) * ((a.T + tok - 1) / tok)), (unsigned)n);
    auto go = [&](auto kern) { kern<<<grid, kConvThreads, 0, st>>>(cb, a.B, a.T, a.H, a.width, a.eps); };
    if (d == 128)
        w4 ? go(conv_silu_kernel<128, 4, TIn>) : go(conv_silu_kernel<128, 8, TIn>);
    else
        w4 ? go(conv_silu_kernel<64, 4, TIn>) : go(conv_silu_kernel<64, 8, TIn>);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const PrologueArgs &a, cudaStream_t st)
{
    if (a.T == 0) return cudaSuccess;
    const bool bf = a.dtype == LDN_BF16;
    const bool kda = a.mode == LDN_KDA;
    // one gate per (b, t, h): folded into the convolution launch; KDA's per-channel gates:
    // their own launch
    const GateArgs ga{a.beta_logit, a.beta, a.gate_z, a.gate_a, a.gate_b, a.mode == LDN_DELTANET ? nullptr : a.gate,
                      (long long)a.B * a.T * a.H, a.H};
    const GateArgs *fold = kda ? nullptr : &ga;
    cudaError_t e;
    if (a.dk == a.dv) {   // q, k, v in one launch
        const int sel[3] = {0, 1, 2};
        e = bf ? conv_launch<__nv_bfloat16>(a, sel, 3, a.dk, fold, st) : conv_launch<float>(a, sel, 3, a.dk, fold, st);
    } else {
        const int sqk[2] = {0, 1}, sv[1] = {2};
        e = bf ? conv_launch<__nv_bfloat16>(a, sqk, 2, a.dk, fold, st) : conv_launch<float>(a, sqk, 2, a.dk, fold, st);
        if (e == cudaSuccess)
            e = bf ? conv_launch<__nv_bfloat16>(a, sv, 1, a.dv, nullptr, st)
                   : conv_launch<float>(a, sv, 1, a.dv, nullptr, st);
    }
    if (e != cudaSuccess || !kda) return e;
    const long long n4 = (long long)a.B * a.T * a.H * (a.dk / 4);
    return n4 + kThreads * kGateUnroll < (1LL << 31) ? gates_launch<unsigned>(a, st)
                                                      : gates_launch<unsigned long long>(a, st);
}

cudaError_t launch_rmsnorm_gated(const RmsNormArgs &a, cudaStream_t st)
{
    const long long rows = (long long)a.B * a.T * a.H;
    if (rows == 0) return cudaSuccess;
    auto grid = [&](int per) { return (unsigned)((rows + per - 1) / per); };
    if (a.dtype == LDN_BF16) {
        const __nv_bfloat16 *o = (const __nv_bfloat16 *)a.o, *g = (const __nv_bfloat16 *)a.g;
        __nv_bfloat16 *y = (__nv_bfloat16 *)a.y;
        if (a.dv == 128) rmsnorm_gated_kernel<128, __nv_bfloat16><<<grid(rms_rows<128, __nv_bfloat16>()), kThreads, 0, st>>>(o, g, a.weight, y, rows, a.eps);
        else rmsnorm_gated_kernel<64, __nv_bfloat16><<<grid(rms_rows<64, __nv_bfloat16>()), kThreads, 0, st>>>(o, g, a.weight, y, rows, a.eps);
    } else {
        const float *o = (const float *)a.o, *g = (const float *)a.g;
        float *y = (float *)a.y;
        if (a.dv == 128) rmsnorm_gated_kernel<128, float><<<grid(rms_rows<128, float>()), kThreads, 0, st>>>(o, g, a.weight, y, rows, a.eps);
        else rmsnorm_gated_kernel<64, float><<<grid(rms_rows<64, float>()), kThreads, 0, st>>>(o, g, a.weight, y, rows, a.eps);
    }
    return cudaGetLastError();
}

}  // namespace ldn
