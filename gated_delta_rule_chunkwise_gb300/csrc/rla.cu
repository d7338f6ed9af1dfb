// Residual Linear Attention (RLA) and Residual DeltaNet (RDN), forward, in the
// two stages the Residual Linear Attention notes describe (Sec. 2.6): the base
// state first, which also yields every token's S_{t-1} k_t; then the clipped
// residuals r_t as the values of a second state of the same kind.
//   RLA: S_t = alpha S_{t-1} + beta v k^T,          R_t = alpha R_{t-1} + gamma r k^T
//   RDN: S_t = alpha S_{t-1}(I - beta k k^T) + beta v k^T,
//        R_t = alpha R_{t-1}(I - gamma k k^T) + gamma r k^T       (Sec. 2.4)
//   r_t = Clip_[-c, c](v_t - S_{t-1} k_t),   o_t = alpha_t S_{t-1} q_t + gamma_t R_t q_t
// (Sec. 2.2, the boxed form).  Stage 1 is the token-recurrent kernel writing
// the reads of the old base state (S_{t-1} k_t and alpha_t S_{t-1} q_t); the
// residual kernel clips; stage 2 is the residual state with v := r and
// beta := gamma, read after its update (the tensor-core chunk kernel for RDN when
// it takes the sizes, else the recurrent kernel); the combine kernel forms o.
#include "ldn_internal.cuh"

namespace ldn {
namespace {

template <typename TIn>
__global__ void rla_residual_kernel(const TIn *__restrict__ v, const float *__restrict__ pk, TIn *__restrict__ r,
                                    float c, long long n)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        store_out(r, i, fminf(fmaxf(load_in(v, i) - pk[i], -c), c));
}

template <typename TIn>
__global__ void rla_combine_kernel(const float *__restrict__ sq, const TIn *__restrict__ o2,
                                   const float *__restrict__ gamma, TIn *__restrict__ out, long long n, int dv)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        store_out(out, i, sq[i] + gamma[i / dv] * load_in(o2, i));
}

unsigned stream_blocks(long long n)
{
    const long long b = (n + 255) / 256;
    return (unsigned)(b < 152LL * 32 ? b : 152LL * 32);
}

template <typename TIn>
cudaError_t launch_t(const RlaArgs &a, cudaStream_t st)
{
    const long long n = (long long)a.B * a.T * a.H * a.dv;
    const size_t el = sizeof(TIn);
    uint8_t *w = (uint8_t *)a.ws;
    float *pk = (float *)w;
    float *sq = (float *)(w + rla_off(n * 4));
    TIn *r = (TIn *)(w + 2 * rla_off(n * 4));
    TIn *o2 = (TIn *)(w + 2 * rla_off(n * 4) + rla_off(n * el));
    // stage 1: base state and the reads of its old value
    RecArgs s1{a.q, a.k, a.v, a.beta, a.gate, a.S0, a.S_final, pk, sq, nullptr, a.B, a.T, a.H, a.dk, a.dv,
               a.dtype, a.delta != 0, true};
    cudaError_t e = launch_recurrent(s1, st);
    if (e != cudaSuccess) return e;
    rla_residual_kernel<TIn><<<stream_blocks(n), 256, 0, st>>>((const TIn *)a.v, pk, r, a.clip, n);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // stage 2: the residual state with values r and write strength gamma, read after its update
    ChunkArgs s2{a.q, a.k, r, a.gamma, a.gate, a.R0, o2, a.R_final, a.B, a.T, a.H, a.dk, a.dv, 64,
                 (int)LDN_GDN, a.dtype, a.status};
    if (a.delta && a.dtype == LDN_BF16 && chunk_tc_supported(s2)) {
        e = launch_chunk_tc(s2, st);
    } else {
        RecArgs r2{a.q, a.k, r, a.gamma, a.gate, a.R0, a.R_final, nullptr, nullptr, o2, a.B, a.T, a.H, a.dk, a.dv,
                   a.dtype, a.delta != 0, false};
        e = launch_recurrent(r2, st);
    }
    if (e != cudaSuccess) return e;
    rla_combine_kernel<TIn><<<stream_blocks(n), 256, 0, st>>>(sq, o2, a.gamma, (TIn *)a.out, n, a.dv);
    return cudaGetLastError();
}

}  // namespace

size_t rla_off(size_t bytes) { return (bytes + 255) / 256 * 256; }

size_t rla_workspace_bytes(int B, int T, int H, int dv, int dtype)
{
    const size_t n = (size_t)B * T * H * dv, el = dtype == LDN_BF16 ? 2 : 4;
    return 2 * rla_off(n * 4) + 2 * rla_off(n * el);
}

cudaError_t launch_rla(const RlaArgs &a, cudaStream_t st)
{
    return a.dtype == LDN_BF16 ? launch_t<__nv_bfloat16>(a, st) : launch_t<float>(a, st);
}

}  // namespace ldn
