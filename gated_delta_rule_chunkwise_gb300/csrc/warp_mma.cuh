// Warp-level fp16 tensor-core products over shared-memory tiles (mma.sync m16n8k16 with
// ldmatrix operands, fp32 accumulation) for chunks of 64 tokens and 128-wide heads, with
// the tile loaders they need.  Used by the kernels that run a chunk's dense products on
// a CTA of 8 warps: the chunkwise backward and the Residual Linear Attention chunk form.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "sm100_ptx.cuh"

namespace ldn {
namespace wmma8 {
using namespace sm100;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kLdW = kD + 8;    // fp16 row stride of 128-column tiles (272 B: ldmatrix conflict-free)
constexpr int kLdN = kC + 8;    // fp16 row stride of 64-column tiles (144 B)
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// One operand pair of a product: op(A) [M x K] times op(B) [K x N], fp16 in shared memory.
// ta: A is stored K x M (element (m, k) at a[k * lda + m]), else M x K (a[m * lda + k]);
// tb: B is stored N x K (element (k, n) at b[n * ldb + k]), else K x N (b[k * ldb + n]).
struct Op {
    const __half *a;
    int lda;
    bool ta;
    const __half *b;
    int ldb;
    bool tb;
    int K;
};

// Warp grid of an M x N product: the 8 warps as WM x WN, each owning MT x NT adjacent 16 x 16
// output tiles (a 32 x 32 block for the 64 x 128 and 128 x 64 products, 16 x 32 for 64 x 64),
// so the A fragments of a k-step serve NT tiles and the B fragments MT tiles.
template <int M, int N>
struct WarpGrid {
    static constexpr int WN = N >= 128 ? 4 : 2, WM = kWarps / WN;
    static constexpr int MT = M / 16 / WM, NT = N / 16 / WN;
    static_assert(MT >= 1 && NT >= 1 && MT * 16 * WM == M && NT * 16 * WN == N, "warp grid");
};

// Origin (m0, n0) of tile i of a warp in an M x N product (the same in every product of that shape).
template <int M, int N>
__device__ __forceinline__ int2 tile_origin(int warp, int i)
{
    using G = WarpGrid<M, N>;
    return make_int2(((warp / G::WN) * G::MT + i / G::NT) * 16, ((warp % G::WN) * G::NT + i % G::NT) * 16);
}

// Out [M x N] = sum over the ops of op(A) op(B).  Warp w computes its tiles i = 0 .. TILES-1
// (tile_origin) together, every k-step fully unrolled; then calls epi(i, m0, n0, acc) per
// tile: acc[nt][e] is the element at row m0 + g + 8 (e >> 1), column n0 + 8 nt + 2 t + (e & 1),
// with g = lane / 4, t = lane % 4 (the mma.sync accumulator layout).
template <int M, int N, int NOPS, typename Epi>
__device__ __forceinline__ void cta_mma(const Op (&ops)[NOPS], int warp, int lane, Epi &&epi)
{
    using G = WarpGrid<M, N>;
    const int r = lane & 7, j = lane >> 3;
    const int2 o0 = tile_origin<M, N>(warp, 0);
    float acc[G::MT][G::NT][2][4];
#pragma unroll
    for (int a = 0; a < G::MT; ++a)
#pragma unroll
        for (int b = 0; b < G::NT; ++b)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[a][b][e >> 2][e & 3] = 0.f;
#pragma unroll
    for (int o = 0; o < NOPS; ++o) {
        const Op &op = ops[o];
#pragma unroll 8
        for (int k0 = 0; k0 < op.K; k0 += 16) {
            uint32_t af[G::MT][4], bq[G::NT][4];
#pragma unroll
            for (int a = 0; a < G::MT; ++a) {
                const int m0 = o0.x + 16 * a;
                if (op.ta)
                    ldsm_x4_trans(af[a], op.a + (k0 + r + 8 * (j >> 1)) * op.lda + m0 + 8 * (j & 1));
                else
                    ldsm_x4(af[a], op.a + (m0 + r + 8 * (j & 1)) * op.lda + k0 + 8 * (j >> 1));
            }
#pragma unroll
            for (int b = 0; b < G::NT; ++b) {
                const int n0 = o0.y + 16 * b;
                if (op.tb)
                    ldsm_x4(bq[b], op.b + (n0 + r + 8 * (j >> 1)) * op.ldb + k0 + 8 * (j & 1));
                else
                    ldsm_x4_trans(bq[b], op.b + (k0 + r + 8 * (j & 1)) * op.ldb + n0 + 8 * (j >> 1));
            }
#pragma unroll
            for (int a = 0; a < G::MT; ++a)
#pragma unroll
                for (int b = 0; b < G::NT; ++b) {
                    mma_f16_16x8x16(acc[a][b][0], af[a], bq[b]);
                    mma_f16_16x8x16(acc[a][b][1], af[a], bq[b] + 2);
                }
        }
    }
#pragma unroll
    for (int a = 0; a < G::MT; ++a)
#pragma unroll
        for (int b = 0; b < G::NT; ++b) epi(a * G::NT + b, o0.x + 16 * a, o0.y + 16 * b, acc[a][b]);
}

// Row and column of accumulator element e of half nt in a tile at (m0, n0).
__device__ __forceinline__ int acc_row(int lane, int m0, int e) { return m0 + (lane >> 2) + 8 * (e >> 1); }
__device__ __forceinline__ int acc_col(int lane, int n0, int nt, int e) { return n0 + 8 * nt + 2 * (lane & 3) + (e & 1); }

// Sum of v over the 4 threads of an accumulator row (lanes 4 g .. 4 g + 3).
__device__ __forceinline__ float row_quad_sum(float v)
{
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

// bf16 16-byte group -> fp16 16-byte group (times s)
__device__ __forceinline__ uint4 bf16x8_to_f16(uint4 u, float s = 1.f)
{
    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
    __half2 h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b2[i]);
        h[i] = __floats2half2_rn(f.x * s, f.y * s);
    }
    return *reinterpret_cast<uint4 *>(h);
}

// Rows of bf16 tiles (128 channels: 16 groups of 16 bytes) into fp16 tiles of stride kLdW:
// NT tiles of 64 rows each, every load of the thread in flight before the first store.
template <int NT>
__device__ __forceinline__ void load_tiles_f16(const __nv_bfloat16 *const (&src)[NT], __half *const (&dst)[NT],
                                               size_t tok0, int H, int L, int tid)
{
    constexpr int kPer = NT * kC * 16 / kThreads;   // 16-byte groups per thread
    uint4 u[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = tid + kThreads * i, which = e / (kC * 16), rr = (e / 16) % kC, part = e % 16;
        u[i] = rr < L ? __ldg(reinterpret_cast<const uint4 *>(src[which] + (tok0 + (size_t)rr * H) * kD) + part)
                      : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = tid + kThreads * i, which = e / (kC * 16), rr = (e / 16) % kC, part = e % 16;
        *reinterpret_cast<uint4 *>(dst[which] + rr * kLdW + 8 * part) = bf16x8_to_f16(u[i]);
    }
}

}  // namespace wmma8
}  // namespace ldn
