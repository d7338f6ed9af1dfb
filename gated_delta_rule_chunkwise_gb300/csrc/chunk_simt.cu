// Chunkwise forward on CUDA cores in fp32 (the fp32-dtype path, and a
// cross-check for the tensor-core path with bf16 inputs).
//
// Chunk algebra (exact; derived from the per-token rules of the
// linear-attention notes, Sec. 2.3-2.5, which give no chunk form).  Memory
// orientation H = S^T ([dk][dv]).  For a chunk of C rows with incoming state
// H0, g_r = sum_{j<=r} log a_j (inclusive, per key channel; a scalar
// broadcast for Gated DeltaNet, 0 for DeltaNet), and
//   Q^ = Q * e^{g},  K^ = K * e^{g},  Kv = K * e^{-g},  K~ = K * e^{g_C - g}
// (only products K^_r . Kv_j and Q^_r . Kv_j with j <= r are used, i.e. decay
// ratios e^{g_r - g_j} <= 1; the kernel never forms e^{-g} alone):
//   A   = strict_tril(Diag(beta) K^ Kv^T)          (C x C)
//   W   = (I + A)^{-1} Diag(beta) K^               (C x dk)   UT / WY form
//   U'  = (I + A)^{-1} Diag(beta) V                (C x dv)
//   P   = tril_incl(Q^ Kv^T)                       (C x C)
//   O   = P U' + (Q^ - P W) H0                     (chunk output)
//   H1  = Diag(e^{g_C}) H0 + K~^T (U' - W H0)      (state passed on)
// Only the last two lines depend on H0; everything else is per chunk.
// Gated DeltaNet-2 (linear-attention notes, Sec. 2.6, Eqs. 21-24) has the same
// form with the erase direction e = b * k in place of beta k on the row side of
// A and in W, and the write target z = w * v in place of beta V (the write
// direction, P, O and the state update keep k); it runs the KDA path with those
// three substitutions made where the tiles are loaded.
//
// Work split: one CTA per (b, h, 32-column slice of dv); columns of H are
// independent (state-reduction notes, Sec. 2.5).  The dk-side work (A, W, P)
// is repeated per slice.  All operands live in shared memory as fp32; the
// triangular solve runs one thread per right-hand-side column.
#include "ldn_internal.cuh"

namespace ldn {
namespace {

constexpr int kC = 64;           // chunk length
constexpr int kDVS = 32;         // dv columns per CTA
constexpr int kThreads = 256;

template <int DK>
struct SimtSmem {
    static constexpr int LDK = DK + 1;   // padded row strides (bank spread)
    static constexpr int LDV = kDVS + 1;
    static constexpr int LDA = kC + 1;
    static constexpr size_t floats = 3 * (size_t)kC * LDK + (size_t)kC * LDV + (size_t)kC * LDA +
                                     (size_t)DK * LDV + 3 * DK + 2 * kC;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <int DK, typename TIn, int MODE>
__global__ void __launch_bounds__(kThreads)
chunk_simt_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
                  const float *__restrict__ beta, const float *__restrict__ gate,
                  const float *S0, TIn *__restrict__ out, float *S_final,  // S0 may alias S_final
                  int T, int H, int dv, const float *__restrict__ erase, const float *__restrict__ write)
{
    constexpr bool kG2 = MODE == LDN_GDN2;
    constexpr bool kChan = MODE == LDN_KDA || kG2;   // per-key-channel decay
    using L = SimtSmem<DK>;
    extern __shared__ float smem[];
    float *Qs = smem;                         // [C][LDK]  Q -> Q^ -> Q^ - P W
    float *Ks = Qs + kC * L::LDK;             // [C][LDK]  K -> K^ -> beta K^ -> W
    float *Kc = Ks + kC * L::LDK;             // [C][LDK]  K -> Kv = K e^{-g}
    float *Vs = Kc + kC * L::LDK;             // [C][LDV]  V -> beta V -> U' -> U
    float *Am = Vs + kC * L::LDV;             // [C][LDA]  A, then P
    float *Hs = Am + kC * L::LDA;             // [DK][LDV] state slice (fp32)
    float *gC = Hs + DK * L::LDV;             // [DK]      e^{g_C} per key channel
    float *gCl = gC + DK;                     // [DK]      g_C (KDA)
    float *gm = gCl + DK;                     // [DK]      reference g at the middle row (KDA)
    float *bs = gm + DK;                      // [C]       beta (0 on tail rows)
    float *gr = bs + kC;                      // [C]       scalar log-gate prefix (GDN)

    const int tid = threadIdx.x;
    const int slices = dv / kDVS;
    const int unit = blockIdx.x / slices;     // b * H + h
    const int b = unit / H, h = unit % H;
    const int col0 = (blockIdx.x % slices) * kDVS;

    // Initial state slice.
    for (int e = tid; e < DK * kDVS; e += kThreads) {
        const int c = e / kDVS, n = e % kDVS;
        Hs[c * L::LDV + n] = S0 ? S0[((size_t)unit * DK + c) * dv + col0 + n] : 0.0f;
    }

    for (int t0 = 0; t0 < T; t0 += kC) {
        const int Lr = min(kC, T - t0);       // valid rows of this chunk
        __syncthreads();                      // previous chunk done with smem

        // 1. Load Q, K (twice), V slice, beta; zero the tail rows.
        for (int e = tid; e < kC * DK; e += kThreads) {
            const int r = e / DK, c = e % DK;
            float qv = 0.f, kv = 0.f;
            if (r < Lr) {
                const size_t i = (((size_t)b * T + t0 + r) * H + h) * DK + c;
                qv = load_in(q, i);
                kv = load_in(k, i);
            }
            Qs[r * L::LDK + c] = qv;
            Ks[r * L::LDK + c] = (kG2 && r < Lr) ? erase[(((size_t)b * T + t0 + r) * H + h) * DK + c] * kv : kv;
            Kc[r * L::LDK + c] = kv;
        }
        for (int e = tid; e < kC * kDVS; e += kThreads) {
            const int r = e / kDVS, n = e % kDVS;
            const size_t vi = (((size_t)b * T + t0 + r) * H + h) * dv + col0 + n;
            Vs[r * L::LDV + n] = r < Lr ? (kG2 ? write[vi] * load_in(v, vi) : load_in(v, vi)) : 0.f;
        }
        if (tid < kC) bs[tid] = tid < Lr ? (kG2 ? 1.f : beta[((size_t)b * T + t0 + tid) * H + h]) : 0.f;
        if (MODE == LDN_GDN && tid == 0) {
            float g = 0.f;
            for (int r = 0; r < kC; ++r) {
                if (r < Lr) g += gate[((size_t)b * T + t0 + r) * H + h];
                gr[r] = g;
            }
        }
        __syncthreads();

        // 2. Gate prefix.  Gated DeltaNet: scalar prefix g_r (gr[]).  KDA:
        //    per-channel prefix, factored around the chunk's middle row m, so
        //    Qs = Q e^{g-m}, Ks = K e^{g-m}, Kc = K e^{m-g}; the factors of the
        //    kept (lower-triangular) products multiply to e^{g_r - g_j} <= 1
        //    while each factor stays within e^{|g_C|/2}.
        if (kChan) {
            if (tid < DK) {
                const int c = tid;
                float g = 0.f, m = 0.f;
                for (int r = 0; r < kC; ++r) {
                    if (r < Lr) g += gate[(((size_t)b * T + t0 + r) * H + h) * DK + c];
                    if (r == kC / 2 - 1) m = g;
                }
                gCl[c] = g;
                gm[c] = m;
                g = 0.f;
                for (int r = 0; r < kC; ++r) {
                    if (r < Lr) g += gate[(((size_t)b * T + t0 + r) * H + h) * DK + c];
                    const float e = expf(g - m), ei = expf(m - g);
                    Qs[r * L::LDK + c] *= e;
                    Ks[r * L::LDK + c] *= e;
                    Kc[r * L::LDK + c] *= ei;
                }
            }
        }
        __syncthreads();

        // 3. A = strict_tril(Diag(beta) K^ Kv^T); for a scalar gate the decay
        //    ratio e^{g_r - g_j} is applied exactly per entry.
        for (int e = tid; e < kC * kC; e += kThreads) {
            const int r = e / kC, j = e % kC;
            float acc = 0.f;
            if (j < r) {
                for (int c = 0; c < DK; ++c) acc += Ks[r * L::LDK + c] * Kc[j * L::LDK + c];
                acc *= bs[r];
                if (MODE == LDN_GDN) acc *= expf(gr[r] - gr[j]);
            }
            Am[r * L::LDA + j] = acc;
        }
        __syncthreads();

        // 4. Right-hand sides Diag(beta) K^ (K^ = K e^{g}, chunk-start reference)
        //    and Diag(beta) V.
        for (int e = tid; e < kC * DK; e += kThreads) {
            const int r = e / DK, c = e % DK;
            float f = bs[r];
            if (MODE == LDN_GDN) f *= expf(gr[r]);
            if (kChan) f *= expf(gm[c]);
            Ks[r * L::LDK + c] *= f;
        }
        for (int e = tid; e < kC * kDVS; e += kThreads) {
            const int r = e / kDVS, n = e % kDVS;
            Vs[r * L::LDV + n] *= bs[r];
        }
        __syncthreads();

        // 5. Forward substitution (I + A) X = R, one thread per column, in place:
        //    Ks -> W, Vs -> U'.
        if (tid < DK + kDVS) {
            float *col = tid < DK ? Ks + tid : Vs + (tid - DK);
            const int ld = tid < DK ? L::LDK : L::LDV;
            for (int r = 1; r < kC; ++r) {
                float x = col[r * ld];
                for (int j = 0; j < r; ++j) x -= Am[r * L::LDA + j] * col[j * ld];
                col[r * ld] = x;
            }
        }
        __syncthreads();

        // 6. P = tril_incl(Q^ Kv^T)  (A is dead; reuse its buffer).
        for (int e = tid; e < kC * kC; e += kThreads) {
            const int r = e / kC, j = e % kC;
            float acc = 0.f;
            if (j <= r) {
                for (int c = 0; c < DK; ++c) acc += Qs[r * L::LDK + c] * Kc[j * L::LDK + c];
                if (MODE == LDN_GDN) acc *= expf(gr[r] - gr[j]);
            }
            Am[r * L::LDA + j] = acc;
        }
        __syncthreads();

        // 6b. Re-reference: Qs -> Q^ = Q e^{g} (reads the incoming state) and
        //     Kc -> K~ = K e^{g_C - g} (writes the outgoing state); gC = e^{g_C}.
        if (MODE != LDN_DELTANET) {
            for (int e = tid; e < kC * DK; e += kThreads) {
                const int r = e / DK, c = e % DK;
                const float fq = MODE == LDN_GDN ? expf(gr[r]) : expf(gm[c]);
                const float fk = MODE == LDN_GDN ? expf(gr[kC - 1] - gr[r]) : expf(gCl[c] - gm[c]);
                Qs[r * L::LDK + c] *= fq;
                Kc[r * L::LDK + c] *= fk;
            }
        }
        if (tid < DK) gC[tid] = MODE == LDN_GDN ? expf(gr[kC - 1]) : kChan ? expf(gCl[tid]) : 1.0f;
        __syncthreads();

        // 7. Q~ = Q^ - P W  (row r only reads its own row of Q^).
        for (int e = tid; e < kC * DK; e += kThreads) {
            const int r = e / DK, c = e % DK;
            float acc = Qs[r * L::LDK + c];
            for (int j = 0; j <= r; ++j) acc -= Am[r * L::LDA + j] * Ks[j * L::LDK + c];
            Qs[r * L::LDK + c] = acc;
        }
        __syncthreads();

        // 8a. O = P U' + Q~ H0, stored for the valid rows.
        for (int e = tid; e < kC * kDVS; e += kThreads) {
            const int r = e / kDVS, n = e % kDVS;
            if (r >= Lr) continue;
            float acc = 0.f;
            for (int j = 0; j <= r; ++j) acc += Am[r * L::LDA + j] * Vs[j * L::LDV + n];
            for (int c = 0; c < DK; ++c) acc += Qs[r * L::LDK + c] * Hs[c * L::LDV + n];
            store_out(out, (((size_t)b * T + t0 + r) * H + h) * dv + col0 + n, acc);
        }
        __syncthreads();

        // 8b. U = U' - W H0.
        for (int e = tid; e < kC * kDVS; e += kThreads) {
            const int r = e / kDVS, n = e % kDVS;
            float acc = Vs[r * L::LDV + n];
            for (int c = 0; c < DK; ++c) acc -= Ks[r * L::LDK + c] * Hs[c * L::LDV + n];
            Vs[r * L::LDV + n] = acc;
        }
        __syncthreads();

        // 8c. H1 = Diag(e^{g_C}) H0 + K~^T U.
        for (int e = tid; e < DK * kDVS; e += kThreads) {
            const int c = e / kDVS, n = e % kDVS;
            float acc = gC[c] * Hs[c * L::LDV + n];
            for (int j = 0; j < kC; ++j) acc += Kc[j * L::LDK + c] * Vs[j * L::LDV + n];
            Hs[c * L::LDV + n] = acc;
        }
    }
    __syncthreads();
    if (S_final)
        for (int e = tid; e < DK * kDVS; e += kThreads) {
            const int c = e / kDVS, n = e % kDVS;
            S_final[((size_t)unit * DK + c) * dv + col0 + n] = Hs[c * L::LDV + n];
        }
}

template <int DK, typename TIn, int MODE>
cudaError_t launch_mode(const ChunkArgs &a, cudaStream_t st)
{
    auto kern = chunk_simt_kernel<DK, TIn, MODE>;
    const size_t smem = SimtSmem<DK>::bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((long long)a.B * a.H * (a.dv / kDVS));
    kern<<<grid, kThreads, smem, st>>>((const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v, a.beta,
                                       a.gate, a.S0, (TIn *)a.out, a.S_final, a.T, a.H, a.dv, a.erase,
                                       a.write);
    return cudaGetLastError();
}

template <int DK, typename TIn>
cudaError_t launch_dk(const ChunkArgs &a, cudaStream_t st)
{
    switch (a.mode) {
    case LDN_DELTANET: return launch_mode<DK, TIn, LDN_DELTANET>(a, st);
    case LDN_GDN: return launch_mode<DK, TIn, LDN_GDN>(a, st);
    case LDN_GDN2: return launch_mode<DK, TIn, LDN_GDN2>(a, st);
    default: return launch_mode<DK, TIn, LDN_KDA>(a, st);
    }
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t st)
{
    if (a.dtype == LDN_BF16)
        return a.dk == 128 ? launch_dk<128, __nv_bfloat16>(a, st) : launch_dk<64, __nv_bfloat16>(a, st);
    return a.dk == 128 ? launch_dk<128, float>(a, st) : launch_dk<64, float>(a, st);
}

}  // namespace ldn
