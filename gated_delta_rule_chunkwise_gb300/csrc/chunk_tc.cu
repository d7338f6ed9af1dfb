// Chunkwise forward on the 5th-generation tensor cores (tcgen05, fp16
// operands, fp32 accumulators in TMEM), fp32 state, for bf16 q/k/v with
// dk = 128 and dv a multiple of 64; DeltaNet and Gated DeltaNet (below), KDA
// (per-channel decay factored about the chunk's row 31, see the KDA operand
// build) and Gated DeltaNet-2 (KDA with separate erase and write gates).
//
// Chunk algebra (exact; derived from the per-token rules of the
// linear-attention notes, Sec. 2.3-2.4, which give no chunk form).  Memory
// orientation H = S^T ([dk][dv]).  For a chunk of C = 64 rows with incoming
// state H0, scalar inclusive log-decay prefix g_r and Gamma_rj = e^{g_r - g_j}:
//   A   = strict_tril(Diag(beta) (K K^T) * Gamma)         P = tril(Q K^T * Gamma)
//   T   = (I + A)^{-1}                                      (UT / WY transform)
//   Tu  = T Diag(beta),   Tw = T Diag(beta e^{g})
//   U'  = Tu V,   W = Tw K,   Q~ = Diag(e^{g}) Q - P W
//   O   = P U' + Q~ H0
//   U   = U' - W H0,   H1 = e^{g_C} H0 + K^T Diag(e^{g_C - g}) U
// Only the last two lines depend on the incoming state.
//
// Warp roles (384 threads, one CTA per (b, h, 64-wide slice of dv); value
// columns are independent, state-reduction notes Sec. 2.5):
//   * 8 PREP warps compute everything that does not depend on the state for
//     chunk c + 1 while
//   * 4 SERIAL warps run the state step of chunk c (thread = TMEM lane = row
//     of the fp32 state slice H[row][0:64], held in registers).
// Contractions (tcgen05.mma, fp16 operands, fp32 TMEM accumulators):
//   MMA1 [Q ; K] K^T            M=128  bf16 tiles as loaded  -> P_raw, K K^T
//   MMA3 [P Tu ; Tu] V          M=128                        -> P U', U'
//   MMA4 [-P Tw ; Tw] K         M=128  (double-buffered)     -> -P W, W
//   MMA5 RV += [Q~ ; -W] H0     M=128  (serial, A in TMEM)   -> O, U
//   MMA6 K^T U~                 M=128  (serial)              -> state increment
// and, inside the prep warps, P T by fp16 warp MMAs (block lower-triangular).
// Hand-offs use mbarriers: prep -> serial "chunk ready" is the commit of
// MMA3 / MMA4 itself (both accumulators double-buffered in TMEM), serial ->
// prep "accumulators read".  The serial warps form the MMA5 operand
// [Q~ ; -W] from the MMA4 accumulator and leave it in tensor memory, in place
// (they are idle most of a chunk, the prep warps are not).  Input tiles sit in
// a ring of three stages: the serial warps issue the TMA loads of chunk c + 3
// as soon as the state step of chunk c has released its tiles, so a load has
// two chunks' time to land before it is needed.  The prep warps need no wait
// for MMA3 / MMA4: the commit of the next chunk's MMA1, which they wait on
// anyway, also covers the earlier MMAs of the same issuing thread.
//
// The unit-lower-triangular inverse is blocked by 16: the diagonal blocks by
// fp32 substitution on CUDA cores, the blocks below them by block
// substitution with fp16 warp MMAs (mma.sync m16n8k16, fp32 accumulate, ldmatrix
// operands), one warp per column block.  Decay ratios are applied as row / column factors
// around the chunk's middle row (e^{g_r - m} * e^{m - g_j}), each factor within e^{60}; chunks
// whose log-decay span exceeds that use one exponential per entry instead.
//
// Operand precision: MMA1 runs on the bf16 tiles as loaded; the k and v tiles
// are then converted to fp16 in place, and every computed operand (P, T,
// P T, Q~, W, the state copy, U~) is rounded to fp16 (2^-11), which keeps the
// result within a few 1e-3 of the exact recurrence on a max-error / RMS scale.
// Inputs and intermediates must stay below the fp16 range (65504).
//
// Pair variant (DeltaNet / Gated DeltaNet, dv = 128): the two dv slices of a
// (b, h) run as a cluster of two CTAs, and the state-independent preparation,
// which the fused kernel repeats in both, is split between them by chunk
// parity.  After P6 the preparing CTA copies [P Tu ; Tu], [-P Tw ; Tw] (32 KB)
// into the peer's AV / AK with one shared::cluster bulk copy; the peer's serial
// warps convert its own k / v tiles of that chunk and issue MMA3 / MMA4 while
// MMA6 of the previous chunk runs.  AV / AK are then written by the two CTAs in
// turn, chunk by chunk: a barrier per chunk parity counts the MMA3 / MMA4
// commits of both CTAs (one multicast commit each) before either writes the
// next chunk's operands.  Waits on barriers the peer completes use the
// CTA-scope try_wait like every other wait (the arrival and the transaction
// count carry the ordering); a cluster-scope acquire in the poll loop slowed
// the whole SM.
//
// Gated DeltaNet-2 (linear-attention notes, Sec. 2.6, Eqs. 21-24) runs the KDA
// form with three substitutions where the operands are formed: the K rows of the
// [Q ; K] tile (the prediction side: A's rows and W) carry the erase direction
// b * K e^{G-m} instead of K e^{G-m}, beta is 1, and the V tile is multiplied by
// the write gate w in its fp16 conversion.  The side tile (the write direction,
// P's columns and the state update) keeps K.
//
// Every mbarrier wait is bounded in time (2 s); a timeout sets LDN_ERR_TIMEOUT
// in the status word, both roles abandon their loops, in-flight copies and
// MMAs are drained with bounded waits, TMEM is freed and the CTA returns.
#include <algorithm>
#include <cstddef>

#include "ldn_internal.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace ldn {
namespace {
using namespace sm100;

constexpr int kC = 64;
constexpr int kDK = 128;
constexpr int kDVS = 64;
constexpr int kPrepThreads = 256;
constexpr int kSerialThreads = 128;
constexpr int kThreads = kPrepThreads + kSerialThreads;
constexpr uint32_t kBarPrep = 1, kBarSerial = 2;   // named barrier ids
constexpr uint32_t kBarBuild = 3, kBarBuildIssue = 4;   // KDA operand build (warps 4-7; + issuer warp 3)
constexpr uint32_t kBarChain = 5, kBarChain2 = 6;       // levels of the block inverse (warps 0-2; 0-1)
constexpr uint32_t kBarU = 7;                           // kFed: the U rows of the serial warps (64 threads)
constexpr int kIssuerB = 64;                            // kFed: prep thread issuing MMA4 (warp 2)
constexpr int kIssuer6 = kPrepThreads + 64;             // kFed: serial thread issuing MMA6 (a U row)
constexpr int kIssuer = 96;                        // prep thread issuing every prep MMA (warp 3)
constexpr int kGateWarp = 4;                       // prep warp computing gate prefixes
constexpr uint64_t kWaitNs = 2000000000ull;        // 2 s per wait
constexpr float kMaxLogSpan = 60.f;                // factored decay limit (e^60 per factor)
constexpr float kKdaMaxSpan = 8.f;                 // KDA: fp16 factors e^{+-(G - m)} stay below e^8

// TMEM columns (fp32, 128 lanes).
// Fused kernel: D1 0 (64, MMA1), DK 64 / 192 (2 x 128, MMA4 by stage; then the
// MMA5 A operand as fp16 pairs), RV 320 (2 x 64, MMA3 / MMA5), D6 448 (64, MMA6).
// Preparation kernel of the split variant: D1 0, DK 64 (128, one buffer), RV
// 192 (2 x dv <= 2 x 128, MMA3 over the whole dv).
constexpr uint32_t kColD1 = 0;
constexpr uint32_t kColD6 = 448;
constexpr uint32_t kTmemCols = 512;
template <bool SPLIT>
__device__ __forceinline__ uint32_t col_dk(int s) { return SPLIT ? 64u : (s ? 64u : 192u); }
template <bool SPLIT>
__device__ __forceinline__ uint32_t col_rv(int s) { return SPLIT ? 192u + 128u * s : 320u + 64u * s; }

// Shared memory (bytes from a 1024-aligned base).
constexpr uint32_t kQKBytes = 2 * 16384;      // [Q;K], 2 blocks of 128 rows x 128 B
constexpr uint32_t kVBytes = 8192;            // V slice, 64 rows x 128 B
constexpr uint32_t kKBBytes = 16384;          // KDA side tile [64][128] fp16, K-major (2 blocks of 64 rows)
constexpr int kLd16 = 72;                     // fp16 row stride (144 B: ldmatrix conflict-free)
constexpr uint32_t kSmallBytes = 11264;
constexpr int kMaxStages = 3;

// KIND kFused: the fused kernel, one CTA per (b, h, 64-wide dv slice) over the whole sequence.
// KIND kSplit: the preparation kernel of the split variant, one CTA per (b, h, range of
// `cpr` chunks) over the whole dv; its serial warps write the chunk operands to `ws`.
// KIND kPair: the fused kernel with the two dv slices of a (b, h) (dv = 128) as a cluster of
// two CTAs that share the state-independent preparation: CTA r prepares chunks r, r + 2, ...
// and copies their [P Tu ; Tu], [-P Tw ; Tw] into the peer's shared memory, whose serial
// warps issue MMA3 / MMA4 for those chunks themselves (DeltaNet / Gated DeltaNet).
// KIND kPrepX and kFed: the two launches of the pre-solved variant.  kPrepX (prep warps
// only, two CTAs per SM, one CTA per (b, h, range of chunks)) runs MMA1, the operands A
// and P, the inverse T and P T, and writes X = [P T ; T] (fp16, 128 x 64, the swizzled
// K-major image of an MMA A operand, 16 KB per (b, h, chunk)) to `ws`.  kFed is the fused
// kernel whose prep warps read X instead of computing it: they scale it into AV / AK,
// convert the k / v tiles, issue MMA3 / MMA4 and form the MMA5 operand [Q~ ; -W], so
// that the serial warps only run the state step.
constexpr int kFused = 0, kSplit = 1, kPair = 2, kPrepX = 3, kFed = 4;
constexpr uint32_t kXBytes = 16384;   // X = [P T ; T] per (b, h, chunk)

struct Small {
    uint64_t bar_load[kMaxStages];   // TMA tiles of ring stage ls landed
    uint64_t bar_pmma;        // prep MMA commits
    uint64_t bar_smma;        // serial MMA commits
    uint64_t bar_s6;          // kFed: MMA6 commits (its issuer does not wait for MMA5's waiters:
                              // a barrier of its own keeps a late waiter from seeing two phases)
    uint64_t bar_ready[2];    // MMA3 / MMA4 of stage s complete (prep commit)
    uint64_t bar_rvfree[2];   // serial finished reading RV[s] and DK[s]
    uint64_t bar_drain[4];    // failure path: last commit of each MMA issuer
    uint64_t bar_kbfree[2];   // KDA: MMA6 of chunk c finished reading side tile c & 1
    uint64_t bar_dkfree[2];   // split: the epilogue has read DK of chunk c (DK has one buffer)
    uint64_t bar_stgfree[2];  // split: the workspace stores of chunk c have read their staging (AV / AK)
    uint64_t bar_recv;        // pair: the peer's [P Tu ; Tu], [-P Tw ; Tw] of a chunk landed in AV / AK
    uint64_t bar_avakread[2]; // pair: MMA3 / MMA4 of chunk c read AV / AK in both CTAs (2 arrivals)
    uint64_t bar_fin;         // pair: the last commit of both MMA issuers of both CTAs (4 arrivals)
    uint32_t tmem_base;
    int fail;
    uint32_t sent, recvd;     // pair: operand transfers issued to / consumed from the peer
    // Per-chunk gate data, slot = chunk % 3: written one chunk ahead by the gate
    // warp, read by the prep warps and (eg, egc, gC) by the serial warps.
    int exact[3];             // per-entry exponentials for this chunk
    float gC[3];              // e^{g_C}
    int kflag[3][4];          // KDA: a channel of this chunk exceeds the factored span (one word per build warp)
    alignas(16) float beta[3][kC];
    alignas(16) float g[3][kC];      // inclusive log-decay prefix
    alignas(16) float eg[3][kC];     // e^{g_r}
    alignas(16) float egc[3][kC];    // e^{g_C - g_r}
    // KDA, per key channel: e^{m}, e^{g_C - m}, e^{g_C} (m, g_C: the channel's
    // log-decay prefix at rows 31 and 63)
    alignas(16) float em[3][kDK];
    alignas(16) float egcm[3][kDK];
    alignas(16) float egC[3][kDK];
    float kxm[kDK];           // KDA build: log-decay prefix at row 31, handed from the rows 0-31 warps
    float stg_beta[2][kC];    // beta / log-gate of the next chunk, prefetched by cp.async
    float stg_gate[2][kC];
    uint64_t bar_x[2];        // kFed: X of chunk c landed in AV[c & 1]
    // Factors of MMA1's decay ratios (the operand build of A and P): last, so that
    // kFed, which does not build them, leaves them out of its shared memory.
    alignas(16) float fr[3][kC];     // e^{g_r - m}
    alignas(16) float fc[3][kC];     // e^{m - g_j}
};
static_assert(sizeof(Small) <= kSmallBytes, "Small does not fit its shared-memory slot");
constexpr uint32_t kSmallBytesFed = (offsetof(Small, fr) + 127) / 128 * 128;

// Input tiles sit in a ring (chunk c in stage c % stages): three stages for
// DeltaNet / Gated DeltaNet; two for KDA and Gated DeltaNet-2, whose two side tiles take
// the room; one [Q ; K] buffer for kPrepX (MMA1 is its only reader, so the next chunk's
// tiles load while the current chunk is solved).
template <int MODE, int KIND = kFused>
struct Layout {
    static constexpr bool kda = MODE == LDN_KDA || MODE == LDN_GDN2;   // per-channel decay
    static constexpr bool prepx = KIND == kPrepX, fed = KIND == kFed, split = KIND == kSplit;
    static constexpr int stages = prepx ? 1 : (kda ? 2 : 3);
    static constexpr uint32_t vbytes = prepx ? 0 : (split ? 2 * kVBytes : kVBytes);  // V slice (split: all of dv <= 128)
    static constexpr uint32_t qk = 0;                              // stages x [Q;K]
    static constexpr uint32_t v = qk + stages * kQKBytes;          // stages x V
    static constexpr uint32_t kb = v + stages * vbytes;            // KDA: 2 x side tile (kPrepX: 1)
    static constexpr uint32_t akc = kb + (kda ? (prepx ? 1 : 2) * kKBBytes : 0); // KDA: [I ; 0] K-major 128 x 64 (16 KB, constant)
    static constexpr uint32_t ak = akc + (kda && !prepx ? 16384 : 0);   // [-P Tw ; Tw] K-major 128 x 64 (16 KB)
    // [P Tu ; Tu] K-major 128 x 64 (16 KB).  kFed: AK, AV twice (buffer s at ak + 32 KB s);
    // kPrepX: AV stages X (KDA: AK before it, for the entry-wise path's scratch only).
    static constexpr uint32_t av = ak + (prepx && !kda ? 0 : 16384);
    static constexpr uint32_t hb = av + (fed ? 16384 + 32768 : 16384);   // H fp16, MN-major 128 x 64 (16 KB)
    static constexpr uint32_t ub = hb + (split || prepx ? 0 : 16384);    // U~ fp16, MN-major 64 x 64 (8 KB)
    static constexpr uint32_t a16 = ub + (split || prepx ? 0 : 8192);    // fp16 A [64][72]
    static constexpr uint32_t p16 = a16 + (fed ? 0 : 64 * kLd16 * 2);    // fp16 P [64][72]
    static constexpr uint32_t t16 = p16 + (fed ? 0 : 64 * kLd16 * 2);    // fp16 T [64][72]
    static constexpr uint32_t x = t16 + (fed ? 0 : 64 * kLd16 * 2);      // fp16 16x16 scratch of the block inverse [4][16][24]
    static constexpr uint32_t small = x + (fed ? 0 : 3072);
    static constexpr uint32_t bytes = small + (fed ? kSmallBytesFed : kSmallBytes) + 1024;
    static_assert(bytes <= 232448, "shared memory plan exceeds 227 KB");
    static_assert(!prepx || kda || bytes <= 232448 / 2 - 1024, "kPrepX runs two CTAs per SM (DeltaNet / GDN)");
    static_assert(small % 16 == 0 && t16 % 16 == 0 && kb % 1024 == 0 && akc % 1024 == 0 && ak % 1024 == 0 &&
                      av % 1024 == 0,
                  "buffer alignment (16 B vector accesses, 1024 B swizzled tiles)");
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b)
{
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_bf2(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 16 consecutive columns [col, col + 16) of row `row` of a SWIZZLE_128B block,
// as fp16 (col % 16 == 0, col < 64).
__device__ __forceinline__ void st_row16(uint8_t *block, int row, int col, const float *v)
{
    *reinterpret_cast<uint4 *>(block + sw128_offset(row, col)) =
        make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
    *reinterpret_cast<uint4 *>(block + sw128_offset(row, col + 8)) =
        make_uint4(pack_h2(v[8], v[9]), pack_h2(v[10], v[11]), pack_h2(v[12], v[13]), pack_h2(v[14], v[15]));
}

// 8 bf16 values of a swizzled tile (as loaded by TMA), widened to fp32.
__device__ __forceinline__ void ld_row8_bf16(const uint8_t *block, int row, int col, float *v)
{
    const uint4 u = *reinterpret_cast<const uint4 *>(block + sw128_offset(row, col));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// In-place bf16 -> fp16 conversion of a V tile (64-column blocks of 64 rows, 128-byte
// swizzle) by `n` threads, each value multiplied by the write gate w of its token and
// value channel (Gated DeltaNet-2).  wrow = w of the tile's row 0, column 0 (row stride
// ldw floats, 16-byte aligned); rows at or past `rows` are zero in the tile and stay so.
// A thread converts at most NMAX 16-byte groups (NMAX * n * 16 >= bytes); all its gate
// loads are issued before the first is used, so their latencies overlap.
template <int NMAX>
__device__ __forceinline__ void tile_v_gated_to_f16(uint8_t *p, int bytes, int t, int n, const float *wrow,
                                                    size_t ldw, int rows)
{
    float4 wv[NMAX][2];
#pragma unroll
    for (int i = 0; i < NMAX; ++i) {
        const int o = (t + i * n) * 16;
        const int blk = o >> 13, r = (o >> 7) & 63, c8 = ((((o >> 4) & 7) ^ (r & 7)) << 3) + 64 * blk;
        wv[i][0] = wv[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (o < bytes && r < rows) {
            const float4 *src = reinterpret_cast<const float4 *>(wrow + (size_t)r * ldw + c8);
            wv[i][0] = __ldg(src);
            wv[i][1] = __ldg(src + 1);
        }
    }
#pragma unroll
    for (int i = 0; i < NMAX; ++i) {
        const int o = (t + i * n) * 16;
        if (o >= bytes) break;
        const uint4 u = *reinterpret_cast<const uint4 *>(p + o);
        const float g[8] = {wv[i][0].x, wv[i][0].y, wv[i][0].z, wv[i][0].w,
                            wv[i][1].x, wv[i][1].y, wv[i][1].z, wv[i][1].w};
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&w[j]));
            w[j] = pack_h2(f.x * g[2 * j], f.y * g[2 * j + 1]);
        }
        *reinterpret_cast<uint4 *>(p + o) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// In-place bf16 -> fp16 conversion of `bytes` of a tile by `n` threads.
__device__ __forceinline__ void tile_bf16_to_f16(uint8_t *p, int bytes, int t, int n)
{
    for (int o = t * 16; o < bytes; o += n * 16) {
        uint4 u = *reinterpret_cast<const uint4 *>(p + o);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&w[i]));
            w[i] = pack_h2(f.x, f.y);
        }
        *reinterpret_cast<uint4 *>(p + o) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int MODE, int KIND>
__global__ void __launch_bounds__(KIND == kPrepX ? kPrepThreads : kThreads,
                                  KIND == kPrepX && MODE != LDN_KDA && MODE != LDN_GDN2 ? 2 : 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ beta,
                const float *__restrict__ gate, const float *S0, __nv_bfloat16 *__restrict__ out,
                float *S_final, int T, int H, int dv, int *status, uint8_t *__restrict__ ws, int cpr,
                const float *__restrict__ erase, const float *__restrict__ write, __half *__restrict__ Hs)
{
    extern __shared__ uint8_t dsmem[];
    // 1024-byte aligned base, derived by pointer arithmetic on the __shared__
    // array so that every access below stays a shared-memory access.
    uint8_t *sm = dsmem + ((1024u - (smem_u32(dsmem) & 1023u)) & 1023u);
    constexpr bool SPLIT = KIND == kSplit, PAIR = KIND == kPair;
    constexpr bool kG2 = MODE == LDN_GDN2;                 // Gated DeltaNet-2: erase / write gates
    constexpr bool kKda = MODE == LDN_KDA || kG2;          // per-key-channel decay
    static_assert(!PAIR || !kKda, "the pair kernel takes DeltaNet / Gated DeltaNet");
    constexpr bool PREPX = KIND == kPrepX, FED = KIND == kFed;
    using LY = Layout<MODE, PAIR ? kFused : KIND>;
    constexpr int kStages = LY::stages;
    Small &S = *reinterpret_cast<Small *>(sm + LY::small);
    __half *A16 = reinterpret_cast<__half *>(sm + LY::a16);
    __half *P16 = reinterpret_cast<__half *>(sm + LY::p16);
    __half *T16 = reinterpret_cast<__half *>(sm + LY::t16);
    __half *X16 = reinterpret_cast<__half *>(sm + LY::x);
    uint8_t *AK = sm + LY::ak, *AV = sm + LY::av;
    uint8_t *HB = sm + LY::hb, *UB = sm + LY::ub;
    uint8_t *KB = sm + LY::kb;   // KDA side tiles (chunk c in KB + (c & 1) * kKBBytes)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nchunks_all = (T + kC - 1) / kC;
    constexpr bool RANGES = SPLIT || PREPX;   // one CTA per (b, h, range of cpr chunks)
    const int slices = RANGES ? (nchunks_all + cpr - 1) / cpr : dv / kDVS;   // split / prep-X: chunk ranges
    const int unit = blockIdx.x / slices;
    const int b = unit / H, h = unit % H;
    const int n0 = RANGES ? 0 : (blockIdx.x % slices) * kDVS;
    // chunk c of this CTA is chunk cb + c of the sequence
    const int cb = RANGES ? (blockIdx.x % slices) * cpr : 0;
    const int nchunks = RANGES ? min(cpr, nchunks_all - cb) : nchunks_all;
    constexpr uint32_t kCols = PREPX ? 64u : kTmemCols;   // prep-X: D1 only
    const uint32_t quad = (uint32_t)(warp & 3);          // TMEM lane quadrant of this warp
    const uint32_t lane_base = (32u * quad) << 16;
    // pair: cluster rank = dv slice (blockIdx.x % 2); the peer is the other slice of (b, h)
    const int prank = PAIR ? (int)(blockIdx.x & 1) : 0;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&S.bar_load[i], 1);
        mbar_init(&S.bar_pmma, FED ? 2 : 1);   // kFed: MMA3 and MMA4 come from two threads
        mbar_init(&S.bar_smma, 1);
        mbar_init(&S.bar_s6, 1);
        mbar_init(&S.bar_ready[0], 1);
        mbar_init(&S.bar_ready[1], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&S.bar_drain[i], 1);
        mbar_init(&S.bar_rvfree[0], 1);
        mbar_init(&S.bar_rvfree[1], 1);
        mbar_init(&S.bar_kbfree[0], 1);
        mbar_init(&S.bar_kbfree[1], 1);
        mbar_init(&S.bar_dkfree[0], 1);
        mbar_init(&S.bar_dkfree[1], 1);
        mbar_init(&S.bar_stgfree[0], 1);
        mbar_init(&S.bar_stgfree[1], 1);
        mbar_init(&S.bar_recv, 1);
        mbar_init(&S.bar_avakread[0], 2);
        mbar_init(&S.bar_avakread[1], 2);
        mbar_init(&S.bar_fin, 4);
        mbar_init(&S.bar_x[0], 1);
        mbar_init(&S.bar_x[1], 1);
        fence_mbar_init();
        S.fail = 0;
        S.sent = S.recvd = 0;
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 0) {
        tmem_alloc(&S.tmem_base, kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // the peer's barriers exist before anything reaches them
    tc_fence_after();
    const uint32_t tbase = S.tmem_base;
    // prep-X: the fed kernel that follows may start its CTAs as SMs free up (it waits for
    // this grid before reading the workspace)
    if constexpr (PREPX) griddep_launch_dependents();
    int pending[kMaxStages] = {-1, -1, -1};   // chunk last loaded into ring stage ls (serial thread 0)

    if (tid < kPrepThreads) {
        // ============================== PREP ==============================
        const int pt = tid;
        const int half = pt >> 7;                  // column half handled in TMEM reads
        const int row = 32 * quad + lane;          // TMEM lane of this thread
        const bool issuer = (pt == kIssuer);
        uint32_t pphase = 0;
        // Every prep thread takes the same decision (an OR over the role's barrier),
        // whatever the serial warps write to S.fail meanwhile.
        auto prep_vote = [&](bool ok) -> bool {
            const bool bad = named_sync_or(kBarPrep, kPrepThreads, !ok || S.fail != 0);
            if (bad && pt == 0) S.fail = 1;
            return !bad;
        };
        // MMA-completion and hand-off barriers: one thread polls, the others
        // block in the role's named barrier; tcgen05 ordering follows the sync.
        auto wait_pmma = [&]() -> bool {
            const bool ok = (pt == 0) ? mbar_wait(&S.bar_pmma, pphase, kWaitNs) : true;
            pphase ^= 1u;
            const bool r = prep_vote(ok);
            tc_fence_after();
            return r;
        };
        const uint32_t id_m128_n64 = idesc_f16kind_f32(128, 64, 0, 0, kMmaBF16);   // MMA1 (bf16)
        const uint32_t id_m128_n64_mn = idesc_f16kind_f32(128, 64, 0, 1, kMmaF16); // MMA3
        const uint32_t id_m128_n128_mn = idesc_f16kind_f32(128, 128, 0, 1, kMmaF16);// MMA4
        const uint32_t id_m128_n128_amn = idesc_f16kind_f32(128, 128, 1, 0, kMmaF16);// split MMA3, dv = 128

        // beta and log-gates of chunk cc into staging slot cc & 1 (gate warp; rows
        // past T read as zero), asynchronously so the loads overlap a whole chunk.
        auto prefetch_gates = [&](int cc) {
            const int tt0 = (cb + cc) * kC, LL = min(kC, T - tt0);
            for (int r = lane; r < kC; r += 32) {
                const bool ok = r < LL;
                const size_t i = ok ? ((size_t)b * T + tt0 + r) * H + h : 0;
                if (!kG2) cp_async4(&S.stg_beta[cc & 1][r], beta + i, ok ? 4u : 0u);
                if (MODE == LDN_GDN) cp_async4(&S.stg_gate[cc & 1][r], gate + i, ok ? 4u : 0u);
            }
            cp_async_commit();
        };
        // Gated DeltaNet-2: the erase and write gate rows of chunk cc into L2 (gate warp,
        // one bulk prefetch per row and gate), well before the build and the V
        // conversion load them.
        auto prefetch_g2_rows = [&](int cc) {
            if constexpr (kG2) {
                const int tb = (cb + cc) * kC, LL = min(kC, T - tb);
                for (int r = lane; r < LL; r += 32) {
                    const size_t tok = ((size_t)b * T + tb + r) * H + h;
                    bulk_prefetch_l2(erase + tok * kDK, kDK * 4);
                    bulk_prefetch_l2(write + tok * dv + n0, (SPLIT ? dv : kDVS) * 4);
                }
            }
        };
        // Gate prefix and decay factors of chunk cc into slot cc % 3 (gate warp, two
        // rows per lane); then the staging of chunk cc + 1 is started.
        auto compute_gates = [&](int cc) {
            const int sg = cc & 1, gs = cc % 3;
            cp_async_wait<0>();          // chunk cc's staged beta / gates
            __syncwarp();
            const int r0 = 2 * lane, r1 = r0 + 1;
            const float b0 = kG2 ? 1.f : S.stg_beta[sg][r0], b1 = kG2 ? 1.f : S.stg_beta[sg][r1];
            const float a0 = MODE == LDN_GDN ? S.stg_gate[sg][r0] : 0.f;
            const float a1 = MODE == LDN_GDN ? S.stg_gate[sg][r1] : 0.f;
            __syncwarp();
            if (cc + 1 < nchunks) prefetch_gates(cc + 1);
            if (cc + 1 < nchunks) prefetch_g2_rows(cc + 1);
            float incl = a0 + a1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const float g1 = incl, g0 = incl - a1;
            const float m = __shfl_sync(0xffffffffu, g1, 15);        // g at row 31
            const float gc = __shfl_sync(0xffffffffu, g1, 31);       // g at row 63
            S.beta[gs][r0] = b0; S.beta[gs][r1] = b1;
            S.g[gs][r0] = g0; S.g[gs][r1] = g1;
            if (MODE == LDN_GDN) {
                if constexpr (!FED) {   // MMA1's factors (kFed runs no MMA1 and leaves them out)
                    S.fr[gs][r0] = expf(g0 - m); S.fr[gs][r1] = expf(g1 - m);
                    S.fc[gs][r0] = expf(m - g0); S.fc[gs][r1] = expf(m - g1);
                }
                S.eg[gs][r0] = expf(g0); S.eg[gs][r1] = expf(g1);
                S.egc[gs][r0] = expf(gc - g0); S.egc[gs][r1] = expf(gc - g1);
                if (lane == 0) {
                    S.gC[gs] = expf(gc);
                    S.exact[gs] = (-m > kMaxLogSpan || m - gc > kMaxLogSpan) ? 1 : 0;
                }
            } else {
                if constexpr (!FED) S.fr[gs][r0] = S.fr[gs][r1] = S.fc[gs][r0] = S.fc[gs][r1] = 1.f;
                S.eg[gs][r0] = S.eg[gs][r1] = 1.f;
                S.egc[gs][r0] = S.egc[gs][r1] = 1.f;
                if (lane == 0) { S.gC[gs] = 1.f; S.exact[gs] = 0; }
            }
        };
        // MMA1 [Q ; K] K^T of chunk cc on its bf16 tiles as loaded (issuer thread).
        auto issue_mma1 = [&](int cc) -> bool {
            const int ls = cc % kStages;
            if (!mbar_wait(&S.bar_load[ls], (cc / kStages) & 1, kWaitNs)) return false;
            tc_fence_after();
            const uint32_t qk = smem_u32(sm + LY::qk + ls * kQKBytes);
            for (int k = 0; k < kDK / 16; ++k)
                umma_bf16(tbase + kColD1, kmajor_desc(qk, 128, k), kmajor_desc(qk + 8192, 128, k), id_m128_n64, k > 0);
            umma_commit(&S.bar_pmma);
            return true;
        };
        auto zero_upper_avak = [&]() {
            for (int e = pt; e < 6 * 16 * 2 * 2; e += kPrepThreads) {
                const int blkid = e / 64, rem = e % 64;          // 6 blocks x 16 rows x 2 halves x 2 tiles
                // (R, i) = (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
                const int R = blkid < 3 ? 0 : (blkid < 5 ? 1 : 2);
                const int i = blkid < 3 ? blkid + 1 : (blkid < 5 ? blkid - 1 : 3);
                const int rr = 16 * R + (rem >> 2), cc = 16 * i + 8 * ((rem >> 1) & 1);
                uint8_t *dst = (rem & 1) ? AK : AV;
                *reinterpret_cast<uint4 *>(dst + sw128_offset(rr, cc)) = make_uint4(0u, 0u, 0u, 0u);
            }
        };
        // build warps: wait for the TMA tiles of chunk cc (one poll per warp)
        auto build_wait_tiles = [&](int cc) {
            const int ls = cc % kStages;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&S.bar_load[ls], (cc / kStages) & 1, kWaitNs);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) && lane == 0) S.fail = 1;
        };
        // KDA: per-channel log-decay prefix G of chunk cc and the fp16 MMA1 operands
        // (build warps 4-7, thread = key channel).  The decay ratio e^{G_r - G_j} of
        // each channel is split about row 31 (m): the tile's Q and K rows become
        // Q e^{G - m}, K e^{G - m} in place, the side tile gets K e^{m - G}, so the
        // products carry exactly the decay of every pair of rows.  If |G - m| of some
        // channel exceeds kKdaMaxSpan the chunk keeps its bf16 tiles and is formed
        // entry by entry instead (kflag).  The gate prefix does not need the tiles:
        // it is formed while they are still landing.  Warp 4 calls this after the
        // serial warps released gate slot cc % 3.
        // thread = 8 key channels (ch0..ch0+7) x 8 consecutive rows (r0..r0+7).  Build warp
        // w covers channel block w & 1 and rows 32 (w >> 1) .. + 31; in a warp, lane & 7 is
        // the channel group and lane >> 3 the row group, so the 8 lanes of each
        // shared-memory phase touch 8 different 16-byte columns of one row (no bank
        // conflict under the 128-byte swizzle).  The log-gates are loaded (into G) a phase
        // ahead of the rest, so their latency is hidden.
        // KDA side tile of chunk cc (prep-X keeps one: MMA1 is its only reader)
        auto side = [&](int cc) -> uint8_t * { return KB + (PREPX ? 0 : (cc & 1) * kKBBytes); };
        const int kw = warp - 4, kch0 = 64 * (kw & 1) + 8 * (lane & 7), krh = kw >> 1, krgl = lane >> 3;
        const int kr0 = 32 * krh + 8 * krgl;
        auto kda_load_gates = [&](int cc, float (&G)[8][8]) {
            const int tb = (cb + cc) * kC, LL = min(kC, T - tb);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = kr0 + i;
                float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
                if (r < LL) {   // rows past T: zero
                    const float4 *src =
                        reinterpret_cast<const float4 *>(gate + (((size_t)b * T + tb + r) * H + h) * kDK + kch0);
                    lo = __ldg(src);
                    hi = __ldg(src + 1);
                }
                G[i][0] = lo.x; G[i][1] = lo.y; G[i][2] = lo.z; G[i][3] = lo.w;
                G[i][4] = hi.x; G[i][5] = hi.y; G[i][6] = hi.z; G[i][7] = hi.w;
            }
        };
        auto kda_build = [&](int cc, float (&G)[8][8]) {
            const int ch0 = kch0, r0 = kr0, ls = cc % kStages, gs = cc % 3;
            // inclusive prefix over the rows: within the thread, across the 4 row groups of
            // the warp, then (rows 32-63) plus the prefix at row 31 from the other warp
#pragma unroll
            for (int i = 1; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) G[i][j] += G[i - 1][j];
            float m[8], gc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float inc = G[7][j];
#pragma unroll
                for (int o = 1; o < 4; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, inc, 8 * o);
                    if (krgl >= o) inc += y;
                }
                const float excl = inc - G[7][j];
#pragma unroll
                for (int i = 0; i < 8; ++i) G[i][j] += excl;
                gc[j] = __shfl_sync(0xffffffffu, inc, (lane & 7) + 24);   // this half's last row
            }
            if (krh == 0 && krgl == 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) S.kxm[ch0 + j] = gc[j];       // prefix at row 31
            }
            named_sync(kBarBuild, 128);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (krh == 0) {
                    m[j] = gc[j];
                } else {
                    m[j] = S.kxm[ch0 + j];
                    gc[j] += m[j];   // row 63
#pragma unroll
                    for (int i = 0; i < 8; ++i) G[i][j] += m[j];
                }
            }
            // span check, and G <- e^{G - m} (the row-side factor; formed before the wait for
            // the tiles so that it overlaps it; |G - m| <= kKdaMaxSpan whenever it is used)
            bool wide = false;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float d = G[i][j] - m[j];
                    wide |= !(fabsf(d) <= kKdaMaxSpan);   // NaN: entry-wise
                    G[i][j] = __expf(d);
                }
            const bool any = __any_sync(0xffffffffu, wide);
            if (lane == 0) S.kflag[gs][warp - 4] = any ? 1 : 0;
            named_sync(kBarBuild, 128);
            const bool exact = (S.kflag[gs][0] | S.kflag[gs][1] | S.kflag[gs][2] | S.kflag[gs][3]) != 0;
            if (krh == 1 && krgl == 0) {   // per-channel factors the serial warps apply to MMA4 / MMA6 results
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    S.egC[gs][ch0 + j] = expf(gc[j]);
                    S.em[gs][ch0 + j] = exact ? 1.f : expf(m[j]);
                    S.egcm[gs][ch0 + j] = exact ? 1.f : expf(gc[j] - m[j]);
                }
            }
            build_wait_tiles(cc);
            if (!PREPX && cc >= 2) {   // side tile cc & 1: MMA6 of chunk cc - 2 has read it
                bool ok = true;
                if (lane == 0) ok = mbar_wait(&S.bar_kbfree[cc & 1], ((cc >> 1) - 1) & 1, kWaitNs);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) && lane == 0) S.fail = 1;
            }
            if (!exact) {
                uint8_t *qk = sm + LY::qk + ls * kQKBytes + (ch0 >> 6) * 16384;
                uint8_t *kbt = side(cc) + (ch0 >> 6) * 8192;
                const int col = ch0 & 63;
                // Gated DeltaNet-2: the K rows carry b * K e^{G-m}; the erase gates of a row
                // are loaded four rows ahead of their use (rows past T: K is zero there)
                const int tb = (cb + cc) * kC, LL = min(kC, T - tb);
                const float *erow = kG2 ? erase + (((size_t)b * T + tb + r0) * H + h) * kDK + ch0 : nullptr;
                constexpr int kAhead = kG2 ? 4 : 1;
                float4 eq[kAhead][2];
                auto erase_load = [&](int i, float4 (&d)[2]) {
                    d[0] = d[1] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (kG2 && r0 + i < LL) {
                        const float4 *src = reinterpret_cast<const float4 *>(erow + (size_t)i * H * kDK);
                        d[0] = __ldg(src);
                        d[1] = __ldg(src + 1);
                    }
                };
                if constexpr (kG2) {
#pragma unroll
                    for (int i = 0; i < kAhead; ++i) erase_load(i, eq[i]);
                }
                // kFed, KDA: the K^ rows also carry beta (MMA4's A operand is X = [P T ; T] unscaled)
                float brow[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    brow[i] = FED && !kG2 && r0 + i < LL ? __ldg(beta + ((size_t)b * T + tb + r0 + i) * H + h) : 1.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = r0 + i;
                    float ep[8], en[8], eb[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {   // e^{G-m} and e^{m-G}, rounded to fp16 below
                        ep[j] = G[i][j];
                        en[j] = __fdividef(1.f, G[i][j]);
                        eb[j] = ep[j] * brow[i];
                    }
                    if constexpr (kG2) {
                        const float4 lo = eq[i % kAhead][0], hi = eq[i % kAhead][1];
                        eb[0] *= lo.x; eb[1] *= lo.y; eb[2] *= lo.z; eb[3] *= lo.w;
                        eb[4] *= hi.x; eb[5] *= hi.y; eb[6] *= hi.z; eb[7] *= hi.w;
                        if (i + kAhead < 8) erase_load(i + kAhead, eq[i % kAhead]);
                    }
                    uint4 *qp = reinterpret_cast<uint4 *>(qk + sw128_offset(r, col));
                    uint4 *kp = reinterpret_cast<uint4 *>(qk + sw128_offset(64 + r, col));
                    uint4 *bp = reinterpret_cast<uint4 *>(kbt + sw128_offset(r, col));
                    const uint4 qu = *qp, ku = *kp;
                    const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qu);
                    const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&ku);
                    uint32_t wq[4], wk[4], wb[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 qf = __bfloat1622float2(q2[u]), kf = __bfloat1622float2(k2[u]);
                        wq[u] = pack_h2(qf.x * ep[2 * u], qf.y * ep[2 * u + 1]);
                        wk[u] = pack_h2(kf.x * eb[2 * u], kf.y * eb[2 * u + 1]);
                        wb[u] = pack_h2(kf.x * en[2 * u], kf.y * en[2 * u + 1]);
                    }
                    *qp = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                    *kp = make_uint4(wk[0], wk[1], wk[2], wk[3]);
                    *bp = make_uint4(wb[0], wb[1], wb[2], wb[3]);
                }
            }
            fence_proxy_async_smem();
        };
        const uint32_t id_m128_n64_f16 = idesc_f16kind_f32(128, 64, 0, 0, kMmaF16);   // MMA1 (KDA, fp16)
        auto kda_exact = [&](int cc) -> bool {
            const int gs = cc % 3;
            return (S.kflag[gs][0] | S.kflag[gs][1] | S.kflag[gs][2] | S.kflag[gs][3]) != 0;
        };
        // KDA MMA1 [Q e^{G-m} ; K e^{G-m}] (K e^{m-G})^T (issuer, after the build);
        // the commit is made even when the chunk is formed entry by entry.
        auto kda_issue_mma1 = [&](int cc) {
            const int ls = cc % kStages;
            tc_fence_after();
            if (!kda_exact(cc)) {
                const uint32_t qk = smem_u32(sm + LY::qk + ls * kQKBytes);
                const uint32_t kbt = smem_u32(side(cc));
                for (int k = 0; k < kDK / 16; ++k)
                    umma_bf16(tbase + kColD1, kmajor_desc(qk, 128, k), kmajor_desc(kbt, 64, k), id_m128_n64_f16,
                              k > 0);
            }
            umma_commit(&S.bar_pmma);
        };
        // KDA: MMA4 runs over [Q^ ; K^] with A = [[I, -P Tw], [0, Tw]]; its first 64
        // columns, [I ; 0], are the same for every chunk
        // (kFed: [-I ; 0], its MMA4 A operand being [[-I, P T], [0, T]])
        auto init_akc = [&]() {
            uint8_t *akc = sm + LY::akc;
            const uint32_t one = FED ? 0xBC00u : 0x3C00u;   // fp16 -1 / +1
            for (int e = pt; e < 128 * 8; e += kPrepThreads) {
                const int rr = e >> 3, c8 = 8 * (e & 7);
                uint32_t w[4] = {0u, 0u, 0u, 0u};
                if (rr < 64 && rr >= c8 && rr < c8 + 8) {
                    const int j = rr - c8;   // the 1.0 sits in half j of this 16-byte group
                    w[j >> 1] = (j & 1) ? one << 16 : one;
                }
                *reinterpret_cast<uint4 *>(akc + sw128_offset(rr, c8)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        };
        // prep-X: the [Q ; K] tiles of chunk cc into the single buffer (thread 0)
        auto prepx_load = [&](int cc) {
            pending[0] = cc;
            mbar_arrive_expect_tx(&S.bar_load[0], 2 * 16384);
            uint8_t *qk = sm + LY::qk;
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_4d(qk + kb * 16384, &tm_q, &S.bar_load[0], kb * 64, h, (cb + cc) * kC, b);
                tma_load_4d(qk + kb * 16384 + 8192, &tm_k, &S.bar_load[0], kb * 64, h, (cb + cc) * kC, b);
            }
        };
        // ---- kFed: the prep warps of the pre-solved variant.  Per chunk: X = [P T ; T] of
        // the chunk (from the workspace, two chunks ahead into AV[c & 1]) stays as loaded and
        // is the A operand of MMA3 and MMA4, whose B operands take the diagonal scales (beta V;
        // Diag(beta e^{g}) K in AK[c & 1]; KDA: the build's K^ rows times beta); the k / v
        // tiles become fp16; MMA3 / MMA4 give [P U' ; U'] and [P W ; W] (KDA: [-Q~ ; W]); the
        // MMA5 operand [Q~ ; -W] is formed from MMA4's accumulator in tensor memory and its
        // arrival on bar_ready is the serial warps' "chunk ready".  GDN / DeltaNet run one
        // chunk ahead: the conversions and MMA3 / MMA4 of chunk c + 1 go in right after
        // chunk c is handed over; KDA / GDN2 keep the chunk's steps in order (their look-ahead
        // operand build waits on the side tile that MMA6 of the chunk before frees).
        auto fed_prep_loop = [&]() {
            const uint8_t *xin = ws + (size_t)unit * nchunks_all * kXBytes;
            auto akb = [&](int sb) -> uint8_t * { return AK + sb * 32768; };   // AK[sb]; AV[sb] = AK[sb] + 16 KB
            int xpend[2] = {-1, -1};   // issuer: chunk last loaded into AV[sb]
            auto load_x = [&](int cc) {
                uint64_t *bar = &S.bar_x[cc & 1];
                xpend[cc & 1] = cc;
                mbar_arrive_expect_tx(bar, kXBytes);
                bulk_load(akb(cc & 1) + 16384, xin + (size_t)cc * kXBytes, kXBytes, bar);
            };
            // the tiles and X of chunk cc landed and (cc >= 2) the serial warps released RV / DK
            // of chunk cc - 2, which MMA3 / MMA4 of chunk cc overwrite (one vote)
            auto wait_inputs = [&](int cc) -> bool {
                bool ok = true;
                if (pt == 0)
                    ok = mbar_wait(&S.bar_load[cc % kStages], (cc / kStages) & 1, kWaitNs) &&
                         mbar_wait(&S.bar_x[cc & 1], (cc >> 1) & 1, kWaitNs) &&
                         (cc < 2 || mbar_wait(&S.bar_rvfree[cc & 1], ((cc >> 1) - 1) & 1, kWaitNs));
                return prep_vote(ok);
            };
            // the operand conversions of chunk c (F2) and MMA3 / MMA4 of chunk c (F3)
            auto convert = [&](int c) {
                const int s = c & 1, ls = c % kStages, gs = c % 3;
                const int t0 = c * kC, L = min(kC, T - t0);
                uint8_t *QK = sm + LY::qk + ls * kQKBytes;
                uint8_t *Vt = sm + LY::v + ls * LY::vbytes;
                uint8_t *AKs = akb(s);
                const bool kexact = kKda && kda_exact(c);
                // ---- F2: the B operands take the diagonal scales, X stays as loaded: V rows
                //      times beta (Gated DeltaNet-2: times w), and (GDN / DeltaNet) the K tile to
                //      fp16 in place for MMA6 plus K rows times beta e^{g} into AK[s] for MMA4
                //      (KDA: the build scaled its K^ rows by beta).  One 16-byte group is 8
                //      channels of one row, so one scale per group.
                {
                    // thread pt: K groups pt + 256 j (j < 4, GDN / DeltaNet) and V groups pt + 256 j
                    // (j < 2); every load is issued before the first store
                    constexpr int kNK = kKda ? 0 : 4;
                    uint4 ku[kNK > 0 ? kNK : 1], vu[2];
#pragma unroll
                    for (int j = 0; j < kNK; ++j) {
                        const int i = pt + kPrepThreads * j;
                        ku[j] = *reinterpret_cast<const uint4 *>(QK + (i >> 9) * 16384 + 8192 + (i & 511) * 16);
                    }
#pragma unroll
                    for (int j = 0; j < 2; ++j) vu[j] = *reinterpret_cast<const uint4 *>(Vt + (pt + kPrepThreads * j) * 16);
                    float wg[2][8];   // Gated DeltaNet-2: the write gate of the V group's 8 channels
                    if constexpr (kG2) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int o = (pt + kPrepThreads * j) * 16, r = o >> 7;
                            const int c8 = 8 * (((o >> 4) ^ r) & 7);
                            float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
                            if (r < L) {
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    write + (((size_t)b * T + t0 + r) * H + h) * dv + n0 + c8);
                                lo = __ldg(src);
                                hi = __ldg(src + 1);
                            }
                            wg[j][0] = lo.x; wg[j][1] = lo.y; wg[j][2] = lo.z; wg[j][3] = lo.w;
                            wg[j][4] = hi.x; wg[j][5] = hi.y; wg[j][6] = hi.z; wg[j][7] = hi.w;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < kNK; ++j) {
                        const int i = pt + kPrepThreads * j, kb = i >> 9, o = (i & 511) * 16, r = o >> 7;
                        const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&ku[j]);
                        const float sc = S.beta[gs][r] * S.eg[gs][r];
                        uint32_t a[4], bsc[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(k2[e]);
                            a[e] = pack_h2(f.x, f.y);
                            bsc[e] = pack_h2(f.x * sc, f.y * sc);
                        }
                        *reinterpret_cast<uint4 *>(QK + kb * 16384 + 8192 + o) = make_uint4(a[0], a[1], a[2], a[3]);
                        *reinterpret_cast<uint4 *>(AKs + kb * 8192 + o) = make_uint4(bsc[0], bsc[1], bsc[2], bsc[3]);
                    }
#pragma unroll
                    for (int j = 0; j < 2; ++j) {   // beta v (Gated DeltaNet-2: w * v)
                        const int o = (pt + kPrepThreads * j) * 16, r = o >> 7;
                        const __nv_bfloat162 *v2 = reinterpret_cast<const __nv_bfloat162 *>(&vu[j]);
                        const float sc = kG2 ? 1.f : S.beta[gs][r];
                        uint32_t a[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(v2[e]);
                            a[e] = kG2 ? pack_h2(f.x * wg[j][2 * e], f.y * wg[j][2 * e + 1]) : pack_h2(f.x * sc, f.y * sc);
                        }
                        *reinterpret_cast<uint4 *>(Vt + o) = make_uint4(a[0], a[1], a[2], a[3]);
                    }
                }
                if (kexact && pt < kDK) {
                    // KDA chunk whose decay span exceeds the fp16 factors: Q^ = Q e^{G}, K^ = K e^{G}
                    // (GDN2: b * K e^{G}) in place and K~ = K e^{G_C - G} into the side tile, unfactored
                    // (thread = key channel; the build left the tiles as loaded and set e^{m} = 1)
                    const int ch = pt, col = ch & 63;
                    uint8_t *blk = QK + (ch >> 6) * 16384;
                    uint8_t *kbt = side(c) + (ch >> 6) * 8192;
                    const float *gp = gate + (((size_t)b * T + t0) * H + h) * kDK + ch;
                    float gC = 0.f;
                    for (int r = 0; r < kC; ++r)
                        if (r < L) gC += __ldg(gp + (size_t)r * H * kDK);
                    float acc = 0.f;
                    for (int r = 0; r < kC; ++r) {
                        if (r < L) acc += __ldg(gp + (size_t)r * H * kDK);
                        // (the erase gate b for Gated DeltaNet-2, beta for KDA)
                        const float bvv = r >= L ? 0.f
                                          : kG2 ? __ldg(erase + (((size_t)b * T + t0 + r) * H + h) * kDK + ch)
                                                : __ldg(beta + ((size_t)b * T + t0 + r) * H + h);
                        uint8_t *qp = blk + sw128_offset(r, col), *kp = blk + sw128_offset(64 + r, col);
                        const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(qp));
                        const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kp));
                        const float eg = expf(acc);
                        *reinterpret_cast<__half *>(qp) = __float2half_rn(qv * eg);
                        *reinterpret_cast<__half *>(kp) = __float2half_rn(bvv * kv * eg);
                        *reinterpret_cast<__half *>(kbt + sw128_offset(r, col)) = __float2half_rn(kv * expf(gC - acc));
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
            };
            auto issue_mma34 = [&](int c) {
                const int s = c & 1, ls = c % kStages;
                uint8_t *QK = sm + LY::qk + ls * kQKBytes;
                uint8_t *Vt = sm + LY::v + ls * LY::vbytes;
                uint8_t *AKs = akb(s), *AVs = akb(s) + 16384;
                const uint32_t qk_s = smem_u32(QK), v_s = smem_u32(Vt);
                // (two issuing threads: MMA3 from the issuer, MMA4 from thread kIssuerB; each
                //  commit arrives once on bar_pmma, which counts two)
                const uint32_t x_s = smem_u32(AVs), ak_s = smem_u32(AKs);
                if (issuer) {
                    tc_fence_after();
                    for (int k = 0; k < kC / 16; ++k)   // X (beta V) = [P U' ; U']
                        umma_bf16(tbase + col_rv<false>(s), kmajor_desc(x_s, 128, k), mnmajor_desc(v_s, 64, k),
                                  id_m128_n64_mn, k > 0);
                    umma_commit(&S.bar_pmma);
                } else if (pt == kIssuerB) {
                    tc_fence_after();
                    if constexpr (kKda) {   // [[-I, P T], [0, T]] [Q^ ; beta K^] = [-Q~ ; W]
                        const uint32_t akc_s = smem_u32(sm + LY::akc);
                        for (int k = 0; k < kC / 16; ++k)
                            umma_bf16(tbase + col_dk<false>(s), kmajor_desc(akc_s, 128, k),
                                      mnmajor_desc(qk_s, 128, k), id_m128_n128_mn, k > 0);
                        for (int k = 0; k < kC / 16; ++k)
                            umma_bf16(tbase + col_dk<false>(s), kmajor_desc(x_s, 128, k),
                                      mnmajor_desc(qk_s, 128, k + kC / 16), id_m128_n128_mn, 1);
                    } else {                // X (Diag(beta e^{g}) K) = [P W ; W]
                        for (int k = 0; k < kC / 16; ++k)
                            umma_bf16(tbase + col_dk<false>(s), kmajor_desc(x_s, 128, k),
                                      mnmajor_desc(ak_s, 64, k), id_m128_n128_mn, k > 0);
                    }
                    umma_commit(&S.bar_pmma);
                }
            };
            // the gates (KDA: and operands) of chunk cc, formed while MMAs run
            auto lookahead = [&](int cc) {
                if (warp == kGateWarp) compute_gates(cc);
                if (kKda && warp >= 4) {
                    float Gn[8][8];
                    kda_load_gates(cc, Gn);
                    kda_build(cc, Gn);
                }
            };
            // A5 = [Q~ ; -W] (fp16 pairs) into the first 64 columns of DK[c & 1] (F5): Q~ =
            // Diag(e^{g}) Q - P W on the top rows (KDA: -(MMA4) times e^{m} per channel), -W on
            // the bottom rows.  Warps w and w + 4 share a lane quadrant and take key channels
            // 64 (w >> 2) ..; all read before either writes (the packed columns of the second
            // half overlap the fp32 columns of the first).  Then chunk c is ready.
            auto form_a5 = [&](int c) {
                const int s = c & 1, ls = c % kStages, gs = c % 3;
                uint8_t *QK = sm + LY::qk + ls * kQKBytes;
                {
                    const int kb = warp >> 2, row = 32 * quad + lane;
                    const bool top = row < 64;
                    const float er = top ? S.eg[gs][row] : 0.f;
                    const uint32_t dk_col = tbase + lane_base + col_dk<false>(s);
                    const uint8_t *qblk = QK + kb * 16384;
                    uint32_t w[32];
                    float va[64];
#pragma unroll
                    for (int q = 0; q < 4; ++q) tmem_ld16(dk_col + 64 * kb + 16 * q, va + 16 * q);
                    tmem_ld_wait();
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int cc = 32 * hf;
                        float *v = va + cc;
                        if constexpr (kKda) {
                            const float4 *emq = reinterpret_cast<const float4 *>(&S.em[gs][64 * kb + cc]);
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 e4 = emq[q];
                                v[4 * q] *= e4.x; v[4 * q + 1] *= e4.y; v[4 * q + 2] *= e4.z; v[4 * q + 3] *= e4.w;
                            }
                        }
                        // MMA4 gave [P W ; W] (GDN / DeltaNet) or [-Q~ ; W] Diag(e^{-m}) (KDA)
                        if (!kKda && top) {
#pragma unroll
                            for (int j = 0; j < 32; j += 8) {
                                float qv[8];
                                ld_row8_bf16(qblk, row, cc + j, qv);
#pragma unroll
                                for (int i = 0; i < 8; ++i) v[j + i] = er * qv[i] - v[j + i];
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = -v[i];
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[16 * hf + i] = pack_h2(v[2 * i], v[2 * i + 1]);
                    }
                    named_sync(kBarPrep, kPrepThreads);
                    tmem_st16u(dk_col + 32 * kb, w);
                    tmem_st16u(dk_col + 32 * kb + 16, w + 16);
                    tmem_st_wait();
                }
                tc_fence_before();
                named_sync(kBarPrep, kPrepThreads);
                if (pt == 0) mbar_arrive(&S.bar_ready[s]);
            };
            if (issuer) {
                griddep_wait();   // the prep-X grid wrote the workspace (its completion and memory)
                load_x(0);
                if (nchunks > 1) load_x(1);
            }
            if (warp == kGateWarp) {
                prefetch_gates(0);
                prefetch_g2_rows(0);
                if (nchunks > 1) prefetch_g2_rows(1);
                compute_gates(0);
            }
            if constexpr (kKda) {
                init_akc();
                if (warp >= 4) {
                    float G0[8][8];
                    kda_load_gates(0, G0);
                    kda_build(0, G0);
                }
            }
            named_sync(kBarPrep, kPrepThreads);
            if constexpr (kKda) {
                for (int c = 0; c < nchunks; ++c) {
                    if (!wait_inputs(c)) break;
                    convert(c);
                    named_sync(kBarPrep, kPrepThreads);
                    issue_mma34(c);
                    if (c + 1 < nchunks) lookahead(c + 1);
                    if (!wait_pmma()) break;
                    form_a5(c);
                    if (issuer && c + 2 < nchunks) load_x(c + 2);   // MMA3 / MMA4 have read AV[c & 1]
                }
            } else {
                bool live = wait_inputs(0);
                if (live) {
                    convert(0);
                    named_sync(kBarPrep, kPrepThreads);
                    issue_mma34(0);
                    if (nchunks > 1) lookahead(1);
                }
                for (int c = 0; live && c < nchunks; ++c) {
                    if (!wait_pmma()) break;          // MMA3 / MMA4 of chunk c complete
                    form_a5(c);
                    if (issuer && c + 2 < nchunks) load_x(c + 2);   // they have read AV[c & 1]
                    if (c + 1 < nchunks) {
                        if (!wait_inputs(c + 1)) break;
                        convert(c + 1);
                        named_sync(kBarPrep, kPrepThreads);
                        issue_mma34(c + 1);
                        if (c + 2 < nchunks) lookahead(c + 2);   // slot (c + 2) % 3: chunk c - 1 released
                    }
                }
            }
            // After a failure: the X loads still in flight land before the CTA leaves
            if (issuer && S.fail)
                for (int sb = 0; sb < 2; ++sb)
                    if (xpend[sb] >= 0) mbar_wait(&S.bar_x[sb], (xpend[sb] >> 1) & 1, kWaitNs / 4);
        };
        if constexpr (FED) {
            fed_prep_loop();
        } else {
        if (PREPX && pt == 0) prepx_load(0);
        if (warp == kGateWarp) {
            prefetch_gates(0);
            prefetch_g2_rows(0);
            if (nchunks > 1) prefetch_g2_rows(1);
        }
        // The strictly-upper 16x16 blocks of T and of the top halves of AV / AK
        // (the blocks of P T above the diagonal) are zero for every chunk and
        // nothing else writes them: clear them once.
        for (int e = pt; e < 64 * 64; e += kPrepThreads) {
            const int r = e >> 6, j = e & 63;
            if ((j >> 4) > (r >> 4)) T16[r * kLd16 + j] = __float2half_rn(0.f);
        }
        zero_upper_avak();
        if constexpr (kKda && !PREPX) init_akc();
        named_sync(kBarPrep, kPrepThreads);

        // The chunks this CTA prepares: every chunk, or (pair) every other one from its
        // rank on.  Iteration c = c0 - step runs only the look-ahead part (gates,
        // operands and MMA1 of chunk c0), so that code exists once.
        constexpr int kStep = PAIR ? 2 : 1;
        const int c0 = prank;
        for (int c = c0 - kStep; c < nchunks; c += kStep) {
            const int cn = c + kStep;     // the next chunk this CTA prepares
            const bool run = c >= c0;
            const int cp = run ? c : c0;
            const int s = cp & 1, ls = cp % kStages, gs = cp % 3;
            uint8_t *QK = sm + LY::qk + ls * kQKBytes;
            uint8_t *Vt = sm + LY::v + ls * LY::vbytes;
            const uint32_t qk_s = smem_u32(QK), k_s = qk_s + 8192, v_s = smem_u32(Vt);

            const bool kexact = kKda && run && kda_exact(c);
            float Gn[8][8];   // KDA, warps 4-7: log-gates of chunk c + 1
            if (kKda && warp >= 4 && cn < nchunks) kda_load_gates(cn, Gn);
            if (run) {
            // ---- P1: MMA1 of chunk c (issued while chunk c - 1 was prepared) complete
            if (!wait_pmma()) break;
            // prep-X: MMA1 has read the tiles -- the next chunk's load into the single buffer
            // (after the entry-wise A / P of a KDA chunk, which read the tiles too)
            if (PREPX && pt == 0 && !kexact && c + 1 < nchunks) prepx_load(c + 1);

            if constexpr (kKda) {
                if (kexact) {
                    // ---- P4 (KDA, decay span beyond the fp16 factors): A and P entry by entry.
                    // AV / AK, free once MMA3 / MMA4 of chunk c - 1 completed, hold the fp32
                    // per-channel log-decay prefix G [64][128] meanwhile.
                    // (prep-X: the store of chunk c - 1's X has read AV)
                    if (PREPX && pt == 0) bulk_wait_read_all();
                    if (!prep_vote(!PREPX && pt == 0 && c >= 1
                                       ? mbar_wait(&S.bar_ready[(c - 1) & 1], ((c - 1) >> 1) & 1, kWaitNs) &&
                                             (!SPLIT || mbar_wait(&S.bar_stgfree[(c - 1) & 1], ((c - 1) >> 1) & 1,
                                                                  kWaitNs))
                                       : true))
                        break;
                    float *Gs = reinterpret_cast<float *>(AK);
                    if (pt < kDK) {
                        const int tb = (cb + c) * kC, LL = min(kC, T - tb);
                        const float *gp = gate + (((size_t)b * T + tb) * H + h) * kDK + pt;
                        float acc = 0.f;
                        for (int r = 0; r < kC; ++r) {
                            if (r < LL) acc += __ldg(gp + (size_t)r * H * kDK);
                            Gs[r * kDK + pt] = acc;
                        }
                    }
                    named_sync(kBarPrep, kPrepThreads);
                    {   // A_rj = beta_r sum_ch k_r k_j e^{G_r - G_j} (j < r); P_rj = sum_ch q_r k_j e^{G_r - G_j} (j <= r)
                        // (Gated DeltaNet-2: b_r * k_r in place of beta_r k_r)
                        const int isA = pt >> 7, r = (pt >> 1) & 63, j0 = 32 * (pt & 1);
                        const int tbe = (cb + c) * kC, LLe = min(kC, T - tbe);
                        const float *erow = kG2 && isA && r < LLe ? erase + (((size_t)b * T + tbe + r) * H + h) * kDK
                                                                  : nullptr;
                        const int jmax = isA ? r - 1 : r;
                        float acc[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc[i] = 0.f;
                        if (j0 <= jmax) {
                            for (int ch = 0; ch < kDK; ++ch) {
                                const uint8_t *blk = QK + (ch >> 6) * 16384;
                                const int col = ch & 63;
                                float xr = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                    blk + sw128_offset(isA ? 64 + r : r, col)));
                                if (kG2 && isA) xr *= erow ? __ldg(erow + ch) : 0.f;
                                const float gr = Gs[r * kDK + ch];
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    if (j0 + i <= jmax) {
                                        const float kj = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                            blk + sw128_offset(64 + j0 + i, col)));
                                        acc[i] += xr * kj * expf(gr - Gs[(j0 + i) * kDK + ch]);
                                    }
                                }
                            }
                        }
                        const float sc = isA ? S.beta[gs][r] : 1.f;
                        __half *dst = (isA ? A16 : P16) + r * kLd16 + j0;
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            *reinterpret_cast<uint32_t *>(dst + i) = pack_h2(j0 + i <= jmax ? acc[i] * sc : 0.f,
                                                                             j0 + i + 1 <= jmax ? acc[i + 1] * sc : 0.f);
                    }
                    named_sync(kBarPrep, kPrepThreads);
                    if constexpr (!PREPX) {   // (prep-X runs no MMA4 / MMA6)
                        // Q^ = Q e^{G}, K^ = K e^{G} (GDN2: b * K e^{G}) in place; K~ = K e^{G_C - G}
                        // into the side tile
                        uint8_t *kbt = KB + (c & 1) * kKBBytes;
                        const int tbe = (cb + c) * kC, LLe = min(kC, T - tbe);
                        for (int e = pt; e < kC * kDK; e += kPrepThreads) {
                            const int r = e >> 7, ch = e & 127, col = ch & 63;
                            const float bv = !kG2 ? 1.f
                                             : r < LLe ? __ldg(erase + (((size_t)b * T + tbe + r) * H + h) * kDK + ch)
                                                       : 0.f;
                            uint8_t *blk = QK + (ch >> 6) * 16384;
                            const float gv = Gs[r * kDK + ch], gcv = Gs[(kC - 1) * kDK + ch];
                            uint8_t *qp = blk + sw128_offset(r, col), *kp = blk + sw128_offset(64 + r, col);
                            const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(qp));
                            const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kp));
                            const float eg = expf(gv);
                            *reinterpret_cast<__half *>(qp) = __float2half_rn(qv * eg);
                            *reinterpret_cast<__half *>(kp) = __float2half_rn(bv * kv * eg);
                            *reinterpret_cast<__half *>(kbt + (ch >> 6) * 8192 + sw128_offset(r, col)) =
                                __float2half_rn(kv * expf(gcv - gv));
                        }
                    }
                    named_sync(kBarPrep, kPrepThreads);
                    zero_upper_avak();   // G overwrote the constant zero blocks of AV / AK
                }
            }

            // ---- P4: P and A (fp16) from MMA1, with decay factors, beta and masks
            if (!kexact) {
                const bool isP = row < 64;
                const int r = isP ? row : row - 64;
                const float frr = S.fr[gs][r] * (isP ? 1.f : S.beta[gs][r]), gr = S.g[gs][r];
                const float br = isP ? 1.f : S.beta[gs][r];
                const bool exact = MODE == LDN_GDN && S.exact[gs] != 0;
                __half *dst = (isP ? P16 : A16) + r * kLd16 + 32 * half;
                if (exact) {
                    // log-decay span too wide for the factored form: one exp per entry.  A rare
                    // path, kept compact (16 columns per pass, the pass loop not unrolled)
#pragma unroll 1
                    for (int q = 0; q < 2; ++q) {
                        float w[16];
                        tmem_ld16(tbase + lane_base + kColD1 + 32 * half + 16 * q, w);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int j = 32 * half + 16 * q + i;
                            const bool keep = isP ? (j <= r) : (j < r);
                            w[i] = keep ? w[i] * br * expf(gr - S.g[gs][j]) : 0.f;
                        }
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + 16 * q);
                        d4[0] = make_uint4(pack_h2(w[0], w[1]), pack_h2(w[2], w[3]), pack_h2(w[4], w[5]), pack_h2(w[6], w[7]));
                        d4[1] = make_uint4(pack_h2(w[8], w[9]), pack_h2(w[10], w[11]), pack_h2(w[12], w[13]),
                                           pack_h2(w[14], w[15]));
                    }
                } else {
                    float v[32];
                    tmem_ld16(tbase + lane_base + kColD1 + 32 * half, v);
                    tmem_ld16(tbase + lane_base + kColD1 + 32 * half + 16, v + 16);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int j = 32 * half + i;
                        const bool keep = isP ? (j <= r) : (j < r);
                        v[i] = keep ? (frr * v[i]) * S.fc[gs][j] : 0.f;
                    }
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        d4[q4] = make_uint4(pack_h2(v[8 * q4], v[8 * q4 + 1]), pack_h2(v[8 * q4 + 2], v[8 * q4 + 3]),
                                            pack_h2(v[8 * q4 + 4], v[8 * q4 + 5]), pack_h2(v[8 * q4 + 6], v[8 * q4 + 7]));
                }
            }
            tc_fence_before();   // D1 has been read: the next MMA1 may overwrite it
            named_sync(kBarPrep, kPrepThreads);
            if (PREPX && pt == 0 && kexact && c + 1 < nchunks) prepx_load(c + 1);

            // ---- P5: T = (I + A)^{-1}: 16x16 diagonal blocks, then block substitution
            if (pt < 64) {
                const int blk = pt >> 4, col = pt & 15, o = blk * 16;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float acc = (r == col) ? 1.f : 0.f;
                    const __half *ar = A16 + (o + r) * kLd16 + o;
#pragma unroll
                    for (int j = 0; j < r; ++j) acc -= __half2float(ar[j]) * x[j];
                    x[r] = (r < col) ? 0.f : acc;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    T16[(o + r) * kLd16 + o + col] = __float2half_rn(x[r]);
                }
            }
            else if constexpr (!PREPX) {   // the other prep threads convert the k and v tiles to fp16 meanwhile
                if constexpr (!kKda) {   // (KDA tiles stay as built; see MMA4 / MMA6)
                    tile_bf16_to_f16(QK + 8192, 8192, pt - 64, kPrepThreads - 64);           // K, block 0
                    tile_bf16_to_f16(QK + 16384 + 8192, 8192, pt - 64, kPrepThreads - 64);   // K, block 1
                }
                const int vbytes = SPLIT ? dv / kDVS * kVBytes : kVBytes;
                if constexpr (kG2) {   // z = w * v (split: dv <= 128, so 16 KB at most)
                    const int tb = (cb + c) * kC;
                    constexpr int kNV = ((SPLIT ? 2 : 1) * (int)kVBytes / 16 + kPrepThreads - 65) / (kPrepThreads - 64);
                    tile_v_gated_to_f16<kNV>(Vt, vbytes, pt - 64, kPrepThreads - 64,
                                             write + (((size_t)b * T + tb) * H + h) * dv + n0, (size_t)H * dv,
                                             min(kC, T - tb));
                } else {
                    tile_bf16_to_f16(Vt, vbytes, pt - 64, kPrepThreads - 64);
                }
            }
            named_sync(kBarPrep, kPrepThreads);
            }   // run
            // Below-diagonal blocks by halves (warps 0..2).  With T_TL, T_BR the inverses of
            // the top-left and bottom-right 32x32 diagonal blocks, T_BL = -T_BR M with
            // M = A_BL T_TL, in three levels:
            //   (1) T10 = -T11 A10 T00, T32 = -T33 A32 T22, M01 = A21 T11, M11 = A31 T11;
            //   (2) M00 = A20 T00 + A21 T10, M10 = A30 T00 + A31 T10,
            //       T21 = -T22 M01, T31 = -(T32 M01 + T33 M11);
            //   (3) T20 = -T22 M00, T30 = -(T32 M00 + T33 M10).
            // Four dependent block products on the longest path (a substitution column by
            // column has six).  Each 16x16x16 product is two m16n8k16 fp16 warp MMAs (fp32
            // accumulate) with ldmatrix operands (row-major A blocks, transposed B blocks);
            // intermediate products and M are fp16 16x16 blocks in the X scratch (4 slots,
            // row stride 24).
            if (warp < 3) {
                if (run) {
                const int g = lane >> 2, t4 = lane & 3;
                const int lr = lane & 15, lc = 8 * (lane >> 4);   // ldmatrix row / column of this lane
                auto Ab = [&](int R, int C) { return A16 + 16 * R * kLd16 + 16 * C; };
                auto Tb = [&](int R, int C) { return T16 + 16 * R * kLd16 + 16 * C; };
                auto Xb = [&](int slot) { return X16 + 16 * 24 * slot; };
                auto mma_blk = [&](float (&acc)[2][4], const __half *a, int lda, const __half *bm, int ldb) {
                    uint32_t af[4], bq[4];
                    ldsm_x4(af, a + lr * lda + lc);
                    ldsm_x4_trans(bq, bm + lr * ldb + lc);
                    mma_f16_16x8x16(acc[0], af, bq);
                    mma_f16_16x8x16(acc[1], af, bq + 2);
                };
                auto st_blk = [&](__half *dst, int ld, const float (&acc)[2][4], float sgn) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            *reinterpret_cast<uint32_t *>(dst + (g + 8 * hh) * ld + 8 * nt + 2 * t4) =
                                pack_h2(sgn * acc[nt][2 * hh], sgn * acc[nt][2 * hh + 1]);
                };
                // ---- level 1
                if (warp < 2) {   // T10 (warp 0), T32 (warp 1): X = A_{r,r-1} T_{r-1,r-1}, then -T_rr X
                    const int r = warp == 0 ? 1 : 3;
                    float acc[2][4] = {};
                    mma_blk(acc, Ab(r, r - 1), kLd16, Tb(r - 1, r - 1), kLd16);
                    st_blk(Xb(warp), 24, acc, 1.f);
                    __syncwarp();
                    float t[2][4] = {};
                    mma_blk(t, Tb(r, r), kLd16, Xb(warp), 24);
                    st_blk(Tb(r, r - 1), kLd16, t, -1.f);
                } else {          // M01 = A21 T11, M11 = A31 T11
                    float m01[2][4] = {}, m11[2][4] = {};
                    mma_blk(m01, Ab(2, 1), kLd16, Tb(1, 1), kLd16);
                    mma_blk(m11, Ab(3, 1), kLd16, Tb(1, 1), kLd16);
                    st_blk(Xb(2), 24, m01, 1.f);
                    st_blk(Xb(3), 24, m11, 1.f);
                }
                named_sync(kBarChain, 96);
                // ---- level 2
                if (warp < 2) {   // M00 (warp 0), M10 (warp 1) = A_r0 T00 + A_r1 T10, r = 2, 3
                    const int r = 2 + warp;
                    float acc[2][4] = {};
                    mma_blk(acc, Ab(r, 0), kLd16, Tb(0, 0), kLd16);
                    mma_blk(acc, Ab(r, 1), kLd16, Tb(1, 0), kLd16);
                    st_blk(Xb(warp), 24, acc, 1.f);   // over this warp's level-1 scratch
                    named_sync(kBarChain2, 64);
                    // ---- level 3: T20 = -T22 M00 (warp 0), T30 = -(T32 M00 + T33 M10) (warp 1)
                    float t[2][4] = {};
                    mma_blk(t, Tb(2 + warp, 2), kLd16, Xb(0), 24);
                    if (warp == 1) mma_blk(t, Tb(3, 3), kLd16, Xb(1), 24);
                    st_blk(Tb(2 + warp, 0), kLd16, t, -1.f);
                } else {          // T21 = -T22 M01, T31 = -(T32 M01 + T33 M11)
                    float t21[2][4] = {}, t31[2][4] = {};
                    mma_blk(t21, Tb(2, 2), kLd16, Xb(2), 24);
                    mma_blk(t31, Tb(3, 2), kLd16, Xb(2), 24);
                    mma_blk(t31, Tb(3, 3), kLd16, Xb(3), 24);
                    st_blk(Tb(2, 1), kLd16, t21, -1.f);
                    st_blk(Tb(3, 1), kLd16, t31, -1.f);
                }
                }   // run
            } else if (warp == kIssuer / 32) {
                // look-ahead: MMA1 of the next chunk into D1 (read by P4 above)
                if constexpr (kKda) {
                    named_sync(kBarBuildIssue, 160);   // operands of chunk c + 1 built
                    if (issuer && cn < nchunks) kda_issue_mma1(cn);
                } else {
                    // (pair: after P9 instead -- chunk c + 2's tiles land only once the serial
                    // warps have finished chunk c - 1)
                    if (!PAIR && issuer && cn < nchunks && !issue_mma1(cn)) S.fail = 1;
                }
            } else {
                if (warp == kGateWarp) {
                    // The serial warps have read the accumulators and gate slot of chunk
                    // c - 2 (needed before MMA3 / MMA4 of chunk c overwrite RV[s], DK[s],
                    // and before slot (c + 1) % 3 = (c - 2) % 3 is rewritten).
                    // (Split: DK has one buffer, so its chunk c - 1 must have been read too.)
                    bool ok = true;
                    if (!PREPX && c >= 2 && lane == 0) ok = mbar_wait(&S.bar_rvfree[s], ((c >> 1) - 1) & 1, kWaitNs);
                    if (SPLIT && c >= 1 && lane == 0)
                        ok = ok && mbar_wait(&S.bar_dkfree[(c - 1) & 1], ((c - 1) >> 1) & 1, kWaitNs);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok) {
                        if (lane == 0) S.fail = 1;
                    } else if (c + 1 < nchunks && c + 1 >= 0) {
                        compute_gates(c + 1);   // pair: the peer's chunk (its gates are needed here too)
                    }
                }
                if constexpr (kKda) {   // warps 4-7: KDA operands of chunk c + 1
                    if (cn < nchunks) kda_build(cn, Gn);
                    named_sync(kBarBuildIssue, 160);
                }
            }
            // MMA3 / MMA4 of chunk c - 1 have finished reading AV / AK before they are rewritten
            // (split: and the workspace stores of chunk c - 1, staged there, have read them;
            // pair: in both CTAs, since this CTA's AV / AK go to the peer's as well).
            // A timeout only marks the CTA failed; the vote at the next chunk's start takes
            // every prep thread out of the loop together.
            if (PREPX && pt == 0 && run) bulk_wait_read_all();   // the store of chunk c - 1's X has read AV
            if (!PREPX && pt == 0 && run && c >= 1) {
                bool ok;
                if constexpr (PAIR)
                    ok = mbar_wait(&S.bar_avakread[(c - 1) & 1], ((c - 1) >> 1) & 1, kWaitNs);
                else
                    ok = mbar_wait(&S.bar_ready[(c - 1) & 1], ((c - 1) >> 1) & 1, kWaitNs) &&
                         (!SPLIT || mbar_wait(&S.bar_stgfree[(c - 1) & 1], ((c - 1) >> 1) & 1, kWaitNs));
                if (!ok) S.fail = 1;
            }
            named_sync(kBarPrep, kPrepThreads);
            if (run) {

            // ---- P6: stacked operands AV = [P Tu ; Tu] and AK = [-P Tw ; Tw] (fp16, K-major).
            //      Rows 64..127 straight from T; rows 0..63 from P T by fp16 warp MMAs
            //      over 16x16 blocks, (P T)_{R,i} = sum_{k=i..R} P_{R,k} T_{k,i}.
            {
                const int j = pt & 63;           // row of T
                const int n0c = 16 * (pt >> 6);  // 16-column group
                float vu[16], vw[16];
                const uint4 *trow = reinterpret_cast<const uint4 *>(T16 + j * kLd16 + n0c);
                const float4 *bq = reinterpret_cast<const float4 *>(&S.beta[gs][n0c]);
                const float4 *eq = reinterpret_cast<const float4 *>(&S.eg[gs][n0c]);
#pragma unroll
                for (int h8 = 0; h8 < 2; ++h8) {
                    const uint4 u = trow[h8];
                    const __half2 *t2 = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const float4 bb = bq[2 * h8 + q], ee = eq[2 * h8 + q];
                        const float2 ta = __half22float2(t2[2 * q]), tb = __half22float2(t2[2 * q + 1]);
                        const int i = 8 * h8 + 4 * q;
                        if constexpr (PREPX) {   // X: T itself
                            vu[i] = ta.x; vu[i + 1] = ta.y; vu[i + 2] = tb.x; vu[i + 3] = tb.y;
                        } else {
                            vu[i] = ta.x * bb.x; vu[i + 1] = ta.y * bb.y; vu[i + 2] = tb.x * bb.z; vu[i + 3] = tb.y * bb.w;
                            vw[i] = vu[i] * ee.x; vw[i + 1] = vu[i + 1] * ee.y;
                            vw[i + 2] = vu[i + 2] * ee.z; vw[i + 3] = vu[i + 3] * ee.w;
                        }
                    }
                }
                st_row16(AV, 64 + j, n0c, vu);
                if constexpr (!PREPX) st_row16(AK, 64 + j, n0c, vw);
            }
            if (warp < 7) {
                // (R, i) output blocks per warp, balanced by k-block count (20 in all).
                const int g = lane >> 2, t4 = lane & 3;
                // block codes 4R + i for this warp (-1: none)
                int code0 = -1, code1 = -1;
                switch (warp) {
                case 0: code0 = 12; break;                  // (3,0)
                case 1: code0 = 8; break;                   // (2,0)
                case 2: code0 = 13; break;                  // (3,1)
                case 3: code0 = 4; code1 = 0; break;        // (1,0) (0,0)
                case 4: code0 = 9; code1 = 5; break;        // (2,1) (1,1)
                case 5: code0 = 14; code1 = 15; break;      // (3,2) (3,3)
                default: code0 = 10; break;                 // (2,2)
                }
#pragma unroll 1
                for (int bi = 0; bi < 2; ++bi) {
                    const int code = bi == 0 ? code0 : code1;
                    if (code < 0) break;
                    const int R = code >> 2, i = code & 3;
                    const int lr = lane & 15, lc = 8 * (lane >> 4);
                    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    for (int kb = i; kb <= R; ++kb) {
                        uint32_t a[4], bq[4];
                        ldsm_x4(a, P16 + (16 * R + lr) * kLd16 + 16 * kb + lc);
                        ldsm_x4_trans(bq, T16 + (16 * kb + lr) * kLd16 + 16 * i + lc);
                        mma_f16_16x8x16(acc[0], a, bq);
                        mma_f16_16x8x16(acc[1], a, bq + 2);
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int rr = 16 * R + g + 8 * hh, cc = 16 * i + 8 * nt + 2 * t4;
                            const float p0 = acc[nt][2 * hh], p1 = acc[nt][2 * hh + 1];
                            if constexpr (PREPX) {   // X: P T itself
                                *reinterpret_cast<uint32_t *>(AV + sw128_offset(rr, cc)) = pack_h2(p0, p1);
                            } else {
                                const float2 bb = *reinterpret_cast<const float2 *>(&S.beta[gs][cc]);
                                const float2 ee = *reinterpret_cast<const float2 *>(&S.eg[gs][cc]);
                                const float u0 = p0 * bb.x, u1 = p1 * bb.y;
                                *reinterpret_cast<uint32_t *>(AV + sw128_offset(rr, cc)) = pack_h2(u0, u1);
                                *reinterpret_cast<uint32_t *>(AK + sw128_offset(rr, cc)) = pack_h2(-u0 * ee.x, -u1 * ee.y);
                            }
                        }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarPrep, kPrepThreads);

            // ---- P9: MMA3 [P Tu ; Tu] V -> RV[s], MMA4 [-P Tw ; Tw] K -> DK[s] (the
            //      gate warp saw the serial warps release both for chunk c - 2); their
            //      commit is the serial warps' "chunk ready".
            if constexpr (PREPX) {   // X of chunk c to the workspace (its shared-memory reads are
                if (pt == 0) {        // waited for before AV is written again)
                    bulk_store(ws + ((size_t)unit * nchunks_all + cb + c) * kXBytes, AV, kXBytes);
                    bulk_commit();
                }
            } else if (issuer) {
                tc_fence_after();
                const uint32_t av_s = smem_u32(AV), ak_s = smem_u32(AK);
                if (SPLIT && dv == 2 * kDVS) {   // split, dv = 128: RV^T = V^T [P Tu ; Tu]^T (lane = dv column)
                    for (int k = 0; k < kC / 16; ++k)
                        umma_bf16(tbase + col_rv<SPLIT>(s), mnmajor_desc(v_s, 64, k), kmajor_desc(av_s, 128, k),
                                  id_m128_n128_amn, k > 0);
                } else {
                    for (int j = 0; j < (SPLIT ? dv / kDVS : 1); ++j)   // split: all of dv, 64 columns at a time
                        for (int k = 0; k < kC / 16; ++k)
                            umma_bf16(tbase + col_rv<SPLIT>(s) + 64 * j, kmajor_desc(av_s, 128, k),
                                      mnmajor_desc(v_s + j * kVBytes, 64, k), id_m128_n64_mn, k > 0);
                }
                if constexpr (kKda) {   // [[I, -P Tw], [0, Tw]] [Q^ ; K^] = [Q~ ; W]
                    const uint32_t akc_s = smem_u32(sm + LY::akc);
                    for (int k = 0; k < 2 * kC / 16; ++k)
                        umma_bf16(tbase + col_dk<SPLIT>(s), kmajor_desc(akc_s, 128, k),
                                  mnmajor_desc(qk_s, 128, k), id_m128_n128_mn, k > 0);
                } else {
                    for (int k = 0; k < kC / 16; ++k)
                        umma_bf16(tbase + col_dk<SPLIT>(s), kmajor_desc(ak_s, 128, k),
                                  mnmajor_desc(k_s, 128, k), id_m128_n128_mn, k > 0);
                }
                umma_commit(&S.bar_ready[s]);
                if constexpr (PAIR) {
                    // both CTAs learn when these MMAs have read AV / AK; the same operands go
                    // to the peer's AV / AK (its MMA3 / MMA4 of chunk c - 1 have read them)
                    umma_commit_mc(&S.bar_avakread[s], 0x3);
                    const uint32_t peer = (uint32_t)(prank ^ 1);
                    const uint32_t rbar = mapa_shared(smem_u32(&S.bar_recv), peer);
                    mbar_remote_arrive_expect_tx(rbar, 2 * 16384);
                    bulk_copy_to_peer(mapa_shared(smem_u32(AK), peer), AK, 2 * 16384, rbar);   // AK, AV adjacent
                    S.sent += 1;
                }
            }
            }   // run
            if constexpr (PAIR) {
                // MMA1 of the next chunk this CTA prepares, and its gates, into the slot of
                // chunk c - 1 (which the serial warps have finished with once its RV was read)
                if (issuer && cn < nchunks && !issue_mma1(cn)) S.fail = 1;
                if (warp == kGateWarp && cn < nchunks) {
                    bool ok = true;
                    if (c >= 1 && lane == 0) ok = mbar_wait(&S.bar_rvfree[(c - 1) & 1], ((c - 1) >> 1) & 1, kWaitNs);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok) {
                        if (lane == 0) S.fail = 1;
                    } else {
                        compute_gates(cn);
                    }
                }
            }
        }
        if (PREPX && pt == 0) bulk_wait_all();   // the workspace is complete before the CTA leaves
        }   // !FED
    } else {
        // ============================== SERIAL ==============================
        const int st = tid - kPrepThreads;   // = TMEM lane = state row
        uint32_t sphase = 0;
        auto serial_vote = [&](bool ok) -> bool {
            const bool bad = named_sync_or(kBarSerial, kSerialThreads, !ok || S.fail != 0);
            if (bad && st == 0) S.fail = 1;
            return !bad;
        };
        // MMA completion: every serial thread polls the commit barrier itself; a timeout
        // marks the CTA failed and the vote at the next chunk's start ends the loop.
        auto wait_smma = [&]() -> bool {
            if (!mbar_wait(&S.bar_smma, sphase, kWaitNs)) S.fail = 1;
            sphase ^= 1u;
            tc_fence_after();
            return true;
        };
        auto issue_load = [&](int c) {
            const int ls = c % kStages;
            uint8_t *qk = sm + LY::qk + ls * kQKBytes;
            uint8_t *vv = sm + LY::v + ls * LY::vbytes;
            pending[ls] = c;
            mbar_arrive_expect_tx(&S.bar_load[ls], 2 * 16384 + (SPLIT ? dv / kDVS : 1) * 8192);
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_4d(qk + kb * 16384, &tm_q, &S.bar_load[ls], kb * 64, h, (cb + c) * kC, b);
                tma_load_4d(qk + kb * 16384 + 8192, &tm_k, &S.bar_load[ls], kb * 64, h, (cb + c) * kC, b);
            }
            if constexpr (SPLIT) {   // all of dv, one 64-column box each
                for (int j = 0; j < dv / kDVS; ++j)
                    tma_load_4d(vv + j * kVBytes, &tm_v, &S.bar_load[ls], j * kDVS, h, (cb + c) * kC, b);
            } else {
                tma_load_4d(vv, &tm_v, &S.bar_load[ls], n0, h, (cb + c) * kC, b);
            }
        };
        if (st == 0)
            for (int c = 0; c < kStages && c < nchunks; ++c) issue_load(c);
        if constexpr (SPLIT) {
        // ---- preparation kernel: the chunk's operands of the state step go to the workspace.
        // They are staged in shared memory that is free at this point -- K~ in the chunk's
        // V tile, [Q~ ; -W] over the chunk's [Q ; K] tile (row by row, after K~ has read K),
        // [P U' ; U'] in AV / AK (until P6 of a later chunk, which waits for stgfree) -- in
        // the images the state kernel uses, and leave in three bulk copies.
        const size_t ubytes = split_unit_bytes(dv);
        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1, gs = c % 3, ls = c % kStages;
            uint8_t *QK = sm + LY::qk + ls * kQKBytes;
            uint8_t *Vt = sm + LY::v + ls * LY::vbytes;
            if (!serial_vote(st == 0 ? mbar_wait(&S.bar_ready[s], (c >> 1) & 1, kWaitNs) : true)) break;
            tc_fence_after();
            if (kStages >= 3 && st == 0 && c >= 1) {   // chunk c - 1's stores have read its tile stage
                bulk_wait_read_all();
                if (c - 1 + kStages < nchunks) issue_load(c - 1 + kStages);
            }
            uint8_t *u = ws + ((size_t)unit * nchunks_all + cb + c) * ubytes;
            const bool top = st < 64;
            // (1) DK -> [Q~ ; -W] row st in registers (packed fp16); DK is handed back at once
            uint32_t a5w[2][2][16];
            {
                const float er = top ? S.eg[gs][st] : 0.f;
                const uint32_t dk_col = tbase + lane_base + col_dk<SPLIT>(s);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    const uint8_t *qblk = QK + kb * 16384;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int cc = 32 * hf;
                        float v[32];
                        tmem_ld16(dk_col + 64 * kb + cc, v);
                        tmem_ld16(dk_col + 64 * kb + cc + 16, v + 16);
                        tmem_ld_wait();
                        if constexpr (kKda) {   // MMA4 gave [Q~ ; W] Diag(e^{-m})
                            const float4 *emq = reinterpret_cast<const float4 *>(&S.em[gs][64 * kb + cc]);
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 e4 = emq[q];
                                v[4 * q] *= e4.x; v[4 * q + 1] *= e4.y; v[4 * q + 2] *= e4.z; v[4 * q + 3] *= e4.w;
                            }
                        }
                        if (top) {
                            if constexpr (!kKda) {
#pragma unroll
                                for (int j = 0; j < 32; j += 8) {
                                    float qv[8];
                                    ld_row8_bf16(qblk, st, cc + j, qv);
#pragma unroll
                                    for (int i = 0; i < 8; ++i) v[j + i] += er * qv[i];
                                }
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = -v[i];
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) a5w[kb][hf][i] = pack_h2(v[2 * i], v[2 * i + 1]);
                    }
                }
            }
            // (2) RV -> [P U' ; U'] staged in AV / AK (one swizzled 128 x 64 block per slice); for
            //     dv = 128 its transpose, lane = dv column: block 0 = (P U')^T, block 1 = U'^T
            {
                const uint32_t rv_col = tbase + lane_base + col_rv<SPLIT>(s);
                for (int n = 0; n < dv; n += 32) {
                    float v[32];
                    tmem_ld16(rv_col + n, v);
                    tmem_ld16(rv_col + n + 16, v + 16);
                    tmem_ld_wait();
                    uint8_t *blk = AK + (n / kDVS) * 16384;   // AK, AV are adjacent
                    st_row16(blk, st, n % kDVS, v);
                    st_row16(blk, st, n % kDVS + 16, v + 16);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarSerial, kSerialThreads);
            if (warp == 8) {   // (3) warp 8: send [P U' ; U'], then give AV / AK back
                if (lane == 0) {
                    mbar_arrive(&S.bar_dkfree[s]);   // DK has been read (one buffer)
                    bulk_store(u + kSplitRvOff, AK, (uint32_t)(dv / kDVS) * 16384);
                    bulk_commit();
                    bulk_wait_read_all();
                }
                __syncwarp();
                // the staging overwrote the constant zero blocks of AV / AK: restore them
                for (int e = lane; e < 6 * 16 * 2 * 2; e += 32) {
                    const int blkid = e / 64, rem = e % 64;
                    const int R = blkid < 3 ? 0 : (blkid < 5 ? 1 : 2);
                    const int i = blkid < 3 ? blkid + 1 : (blkid < 5 ? blkid - 1 : 3);
                    const int rr = 16 * R + (rem >> 2), cc = 16 * i + 8 * ((rem >> 1) & 1);
                    *reinterpret_cast<uint4 *>(((rem & 1) ? AK : AV) + sw128_offset(rr, cc)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.bar_stgfree[s]);
            }
            // (4) K~ = K e^{g_C - g} -> V tile, 2 blocks of 64 rows (thread: row st & 63, half st >> 6)
            {
                const int r = st & 63, kb = st >> 6;
#pragma unroll
                for (int c8 = 0; c8 < 64; c8 += 8) {
                    const uint8_t *src = kKda ? KB + (c & 1) * kKBBytes + kb * 8192 + sw128_offset(r, c8)
                                              : QK + kb * 16384 + sw128_offset(64 + r, c8);
                    uint4 w = *reinterpret_cast<const uint4 *>(src);
                    uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __half22float2(*reinterpret_cast<__half2 *>(&x[i]));
                        const int ch = 64 * kb + c8 + 2 * i;
                        const float f0 = kKda ? S.egcm[gs][ch] : S.egc[gs][r];
                        const float f1 = kKda ? S.egcm[gs][ch + 1] : S.egc[gs][r];
                        x[i] = pack_h2(f.x * f0, f.y * f1);
                    }
                    *reinterpret_cast<uint4 *>(Vt + kb * 8192 + sw128_offset(r, c8)) = make_uint4(x[0], x[1], x[2], x[3]);
                }
                // e^{g_C} per key channel, straight to the workspace
                if (st >= 64) {
                    float *eg = reinterpret_cast<float *>(u + split_eg_off(dv));
                    const int ch = 2 * (st - 64);
                    *reinterpret_cast<float2 *>(eg + ch) = make_float2(kKda ? S.egC[gs][ch] : S.gC[gs],
                                                                       kKda ? S.egC[gs][ch + 1] : S.gC[gs]);
                }
            }
            named_sync(kBarSerial, kSerialThreads);   // K rows read: [Q~ ; -W] may replace them
            // (5) [Q~ ; -W] row st over row st of the [Q ; K] tile (same swizzled geometry)
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4 *>(QK + kb * 16384 + sw128_offset(st, 32 * hf + 8 * q)) =
                            make_uint4(a5w[kb][hf][4 * q], a5w[kb][hf][4 * q + 1], a5w[kb][hf][4 * q + 2],
                                       a5w[kb][hf][4 * q + 3]);
            fence_proxy_async_smem();
            named_sync(kBarSerial, kSerialThreads);
            if (st == 0) {
                bulk_store(u, QK, 32768);
                bulk_store(u + split_kt_off(dv), Vt, 16384);
                bulk_commit();
                // With three tile stages the stage is reloaded after the next chunk's vote,
                // once these stores have read it.  With two (KDA, GDN2) the chunk after next
                // must be in flight before that vote: the next chunk's MMA1 precedes this
                // chunk's "ready" there.
                if constexpr (kStages < 3) {
                    bulk_wait_read_all();
                    if (c + kStages < nchunks) issue_load(c + kStages);
                }
                // RV of chunk c and gate slot c % 3 are read (RV has two buffers)
                mbar_arrive(&S.bar_rvfree[s]);
                if (kKda) mbar_arrive(&S.bar_kbfree[c & 1]);
            }
        }
        if (st == 0) bulk_wait_all();   // the workspace is complete before the CTA leaves
        } else {
        const uint32_t id_m128_n64_mn = idesc_f16kind_f32(128, 64, 0, 1, kMmaF16);   // MMA5 (pair: and MMA3)
        const uint32_t id_m128_n64_amn = idesc_f16kind_f32(128, 64, 1, 1, kMmaF16);  // MMA6
        const uint32_t id_m128_n128_mn = idesc_f16kind_f32(128, 128, 0, 1, kMmaF16); // pair: MMA4
        // Pair: chunk cc was prepared by the peer.  Its [P Tu ; Tu], [-P Tw ; Tw] arrive
        // in AV / AK; this CTA's k and v tiles of the chunk become fp16 here (the prep
        // warps convert only their own chunks' tiles); MMA3 / MMA4 follow as the prep
        // warps would issue them, and their commit is the chunk's "ready".  RV / DK of
        // this parity were last read by chunk cc - 2, finished before chunk cc - 1.
        auto pair_service = [&](int cc) {
            const int ls2 = cc % kStages, s2 = cc & 1;
            uint8_t *QK2 = sm + LY::qk + ls2 * kQKBytes;
            uint8_t *V2 = sm + LY::v + ls2 * LY::vbytes;
            if (!mbar_wait(&S.bar_load[ls2], (cc / kStages) & 1, kWaitNs)) S.fail = 1;
            tile_bf16_to_f16(QK2 + 8192, 8192, st, kSerialThreads);           // K, block 0
            tile_bf16_to_f16(QK2 + 16384 + 8192, 8192, st, kSerialThreads);   // K, block 1
            tile_bf16_to_f16(V2, kVBytes, st, kSerialThreads);
            fence_proxy_async_smem();
            named_sync(kBarSerial, kSerialThreads);
            if (st == 0) {
                if (mbar_wait(&S.bar_recv, (cc >> 1) & 1, kWaitNs))
                    S.recvd += 1;
                else
                    S.fail = 1;
                tc_fence_after();
                const uint32_t av_s = smem_u32(AV), ak_s = smem_u32(AK);
                const uint32_t v2_s = smem_u32(V2), k2_s = smem_u32(QK2) + 8192;
                for (int k = 0; k < kC / 16; ++k)
                    umma_bf16(tbase + col_rv<SPLIT>(s2), kmajor_desc(av_s, 128, k), mnmajor_desc(v2_s, 64, k),
                              id_m128_n64_mn, k > 0);
                for (int k = 0; k < kC / 16; ++k)
                    umma_bf16(tbase + col_dk<SPLIT>(s2), kmajor_desc(ak_s, 128, k), mnmajor_desc(k2_s, 128, k),
                              id_m128_n128_mn, k > 0);
                umma_commit(&S.bar_ready[s2]);
                umma_commit_mc(&S.bar_avakread[s2], 0x3);
            }
        };

        float Hreg[kDVS];
        {
            const float *src = S0 ? S0 + ((size_t)unit * kDK + st) * dv + n0 : nullptr;
#pragma unroll
            for (int n = 0; n < kDVS; n += 4) {
                const float4 x = src ? *reinterpret_cast<const float4 *>(src + n) : make_float4(0.f, 0.f, 0.f, 0.f);
                Hreg[n] = x.x; Hreg[n + 1] = x.y; Hreg[n + 2] = x.z; Hreg[n + 3] = x.w;
            }
#pragma unroll
            for (int n = 0; n < kDVS; n += 16) st_row16(HB, st, n, &Hreg[n]);
        }
        fence_proxy_async_smem();
        named_sync(kBarSerial, kSerialThreads);
        if (PAIR && prank == 1) pair_service(0);

        // ---- S1: MMA3 / MMA4 of chunk c complete (RV[s] = [P U' ; U'], DK[s] = [-P W ; W],
        //      KDA: [Q~ ; W]).  One vote per chunk, taken at the barrier that ends the chunk
        //      before (thread 0 first waits for this chunk's ready barrier), so every thread
        //      leaves the loop at the same chunk.
        bool go = nchunks > 0 && serial_vote(st == 0 ? mbar_wait(&S.bar_ready[0], 0, kWaitNs) : true);
        for (int c = 0; go && c < nchunks; ++c) {
            const int s = c & 1, t0 = (cb + c) * kC, L = min(kC, T - t0);
            const uint8_t *QK = sm + LY::qk + (c % kStages) * kQKBytes;
            const uint32_t k_s = smem_u32(QK) + 8192;
            tc_fence_after();
            // KDA: MMA3 / MMA4 have read V, Q^ and K^, and MMA6 takes K~ from the side
            // tile: the ring stage of chunk c is free already
            if (kKda && st == 0 && c + kStages < nchunks) issue_load(c + kStages);
            const int gs = c % 3;
            const float gC = S.gC[gs];
            const bool top = st < 64;
            const float egc = top ? 0.f : S.egc[gs][st - 64];
            // the state entering this chunk, for the chunkwise backward (row st of the slice, into
            // the fp16 state image)
            if (Hs) {
                __half *dst = Hs + ((size_t)unit * nchunks + c) * (kStateImgBytes / 2) + st * kStateImgLd + n0;
#pragma unroll
                for (int n = 0; n < kDVS; n += 8) {
                    __half2 h[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) h[x] = __floats2half2_rn(Hreg[n + 2 * x], Hreg[n + 2 * x + 1]);
                    *reinterpret_cast<uint4 *>(dst + n) = *reinterpret_cast<const uint4 *>(h);
                }
            }
            // gate data of this chunk for S6, read now: the slot is released (rvfree) before S6
            const float gCr = kKda ? S.egC[gs][st] : gC;   // KDA: decay of key channel st
            // KDA: the side tile holds K e^{m-G} = K~ Diag(e^{m-G_C}) per channel, row st of D6
            const float d6s = kKda ? S.egcm[gs][st] : 1.f;

            // ---- S2: A5 = [Q~ ; -W] (row st): Q~ = Diag(e^{g}) Q - P W on the top rows
            //      (Q read from the bf16 tile as loaded; KDA: MMA4 formed Q~), -W on the
            //      bottom rows, packed as
            //      fp16 pairs into the first 64 columns of DK[s] -- the MMA5 A operand,
            //      read from tensor memory.  Each thread rewrites only columns of its own
            //      lane that it has already read.  (kFed: the prep warps formed it.)
            if constexpr (!FED) {
                const float er = top ? S.eg[gs][st] : 0.f;
                const uint32_t dk_col = tbase + lane_base + col_dk<SPLIT>(s);
#pragma unroll 1   // (code size: both roles' loops must stay in the instruction cache)
                for (int kb = 0; kb < 2; ++kb) {
                    const uint8_t *qblk = QK + kb * 16384;   // Q rows 0..63 of this column block
#pragma unroll
                    for (int cc = 0; cc < 64; cc += 32) {
                        float v[32];
                        tmem_ld16(dk_col + 64 * kb + cc, v);
                        tmem_ld16(dk_col + 64 * kb + cc + 16, v + 16);
                        tmem_ld_wait();
                        if constexpr (kKda) {
                            // KDA: the tiles hold Q e^{G-m}, K e^{G-m}, so MMA4 gave [Q~ ; W] Diag(e^{-m})
                            const float4 *emq = reinterpret_cast<const float4 *>(&S.em[gs][64 * kb + cc]);
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 e4 = emq[q];
                                v[4 * q] *= e4.x; v[4 * q + 1] *= e4.y; v[4 * q + 2] *= e4.z; v[4 * q + 3] *= e4.w;
                            }
                        }
                        if (top) {
                            if constexpr (!kKda) {   // KDA: MMA4 formed Q~ itself
#pragma unroll
                                for (int j = 0; j < 32; j += 8) {
                                    float qv[8];
                                    ld_row8_bf16(qblk, st, cc + j, qv);
#pragma unroll
                                    for (int i = 0; i < 8; ++i) v[j + i] += er * qv[i];
                                }
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = -v[i];
                        }
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = pack_h2(v[2 * i], v[2 * i + 1]);
                        tmem_st16u(dk_col + 32 * kb + cc / 2, w);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                named_sync(kBarSerial, kSerialThreads);
            }

            // ---- S3: MMA5: RV[s] += [Q~ ; -W] H0  -> O (rows 0..63), U (rows 64..127)
            if (st == 0) {
                tc_fence_after();
                const uint32_t a5_t = tbase + col_dk<SPLIT>(s), hb_s = smem_u32(HB);
                for (int k = 0; k < kDK / 16; ++k)
                    umma_ts(tbase + col_rv<SPLIT>(s), a5_t + 8 * k, mnmajor_desc(hb_s, 128, k), id_m128_n64_mn, 1);
                umma_commit(&S.bar_smma);
            }
            if (!wait_smma()) break;

            // ---- S4: O -> global (bf16); U~ = Diag(e^{g_C - g}) U -> UB
            {
                const int r = top ? st : st - 64;
                float v[kDVS];   // the whole slice row in one TMEM round trip
#pragma unroll
                for (int q = 0; q < kDVS / 16; ++q) tmem_ld16(tbase + lane_base + col_rv<SPLIT>(s) + 16 * q, v + 16 * q);
                tmem_ld_wait();
                if (top) {
                    if (r < L) {
                        uint4 *dst = reinterpret_cast<uint4 *>(out + (((size_t)b * T + t0 + r) * H + h) * dv + n0);
#pragma unroll
                        for (int q4 = 0; q4 < kDVS / 8; ++q4)
                            dst[q4] = make_uint4(pack_bf2(v[8 * q4], v[8 * q4 + 1]), pack_bf2(v[8 * q4 + 2], v[8 * q4 + 3]),
                                                 pack_bf2(v[8 * q4 + 4], v[8 * q4 + 5]),
                                                 pack_bf2(v[8 * q4 + 6], v[8 * q4 + 7]));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < kDVS; ++i) v[i] *= egc;
#pragma unroll
                    for (int n = 0; n < kDVS; n += 16) st_row16(UB, r, n, v + n);
                }
            }
            // ---- S5: MMA6: K^T U~ -> D6.  A = K^T (GDN, DeltaNet: U~ carries the decay) or
            //      K~^T (KDA, side tile).  kFed: only the U rows meet before it (one of them
            //      issues it), so the O rows' output stores overlap it.
            auto issue_mma6 = [&]() {
                tc_fence_after();
                const uint32_t ub_s = smem_u32(UB);
                const uint32_t ka_s = kKda ? smem_u32(KB + (c & 1) * kKBBytes) : k_s;
                for (int k = 0; k < kC / 16; ++k)
                    umma_bf16(tbase + kColD6, mnmajor_desc(ka_s, kKda ? 64 : 128, k), mnmajor_desc(ub_s, 64, k),
                              id_m128_n64_amn, k > 0);
                umma_commit(FED ? &S.bar_s6 : &S.bar_smma);
            };
            if constexpr (FED) {
                if (!top) {
                    fence_proxy_async_smem();
                    tc_fence_before();
                    named_sync(kBarU, kSerialThreads - 64);
                    if (st == 64) issue_mma6();
                }
                tc_fence_before();
                named_sync(kBarSerial, kSerialThreads);   // every row has read RV[s]
                if (st == 0) mbar_arrive(&S.bar_rvfree[s]);
            } else {
                fence_proxy_async_smem();
                tc_fence_before();
                named_sync(kBarSerial, kSerialThreads);
                if (st == 0) {
                    mbar_arrive(&S.bar_rvfree[s]);
                    issue_mma6();
                }
            }
            // pair: the next chunk is the peer's -- its MMA3 / MMA4 go in while MMA6 runs
            if (PAIR && c + 1 < nchunks && ((c + 1) & 1) != prank) pair_service(c + 1);
            if constexpr (FED) {
                if (!mbar_wait(&S.bar_s6, (uint32_t)(c & 1), kWaitNs)) S.fail = 1;
                tc_fence_after();
            } else {
                if (!wait_smma()) break;
            }
            if (kKda && st == 0) mbar_arrive(&S.bar_kbfree[c & 1]);
            // the tiles of chunk c are no longer read by anyone: fetch chunk c + stages into them
            if (!kKda && st == 0 && c + kStages < nchunks) issue_load(c + kStages);

            // ---- S6: H1 = e^{g_C} H0 + K^T U~ (row st), fp16 copy for the next MMA5
            {
                float v[kDVS];
#pragma unroll
                for (int q = 0; q < kDVS / 16; ++q) tmem_ld16(tbase + lane_base + kColD6 + 16 * q, v + 16 * q);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < kDVS; ++i) {
                    Hreg[i] = gCr * Hreg[i] + d6s * v[i];
                    v[i] = Hreg[i];
                }
#pragma unroll
                for (int n = 0; n < kDVS; n += 16) st_row16(HB, st, n, v + n);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            const int cn = c + 1;
            go = serial_vote(st == 0 && cn < nchunks ? mbar_wait(&S.bar_ready[cn & 1], (cn >> 1) & 1, kWaitNs) : true);
        }

        if (S.fail == 0 && S_final) {
            float *dst = S_final + ((size_t)unit * kDK + st) * dv + n0;
#pragma unroll
            for (int n = 0; n < kDVS; n += 4)
                *reinterpret_cast<float4 *>(dst + n) = make_float4(Hreg[n], Hreg[n + 1], Hreg[n + 2], Hreg[n + 3]);
        }
        }   // !SPLIT
    }

    tc_fence_before();
    __syncthreads();
    if (S.fail) {
        // Drain the in-flight MMAs of both issuers and the TMA loads (bounded)
        // before shared memory and TMEM are released: a commit tracks every
        // earlier MMA of the thread that issues it.
        if (tid == 0) atomicOr(status, 1 << LDN_ERR_TIMEOUT);
        if (tid == kIssuer || tid == kPrepThreads || (FED && (tid == kIssuerB || tid == kIssuer6))) {
            const int i = tid == kIssuer ? 0 : tid == kPrepThreads ? 1 : tid == kIssuerB ? 2 : 3;
            umma_commit(&S.bar_drain[i]);
            mbar_wait(&S.bar_drain[i], 0, kWaitNs / 4);
        }
        if (tid == (PREPX ? 0 : kPrepThreads))   // the thread that issued the tile loads
            for (int ls = 0; ls < kStages; ++ls)
                if (pending[ls] >= 0) mbar_wait(&S.bar_load[ls], (pending[ls] / kStages) & 1, kWaitNs / 4);
    }
    if constexpr (PAIR) {
        // Nothing of the peer may still be on its way here when this CTA leaves.  Each
        // MMA issuer of both CTAs ends with a commit that arrives in both: the commits of
        // an issuer arrive in order, so once all four have, so have the earlier ones on
        // bar_avakread.  Then, after a failure, an operand transfer the peer issued that
        // was never waited for.
        if (tid == kIssuer || tid == kPrepThreads) umma_commit_mc(&S.bar_fin, 0x3);
        if (tid == 0 && !mbar_wait(&S.bar_fin, 0, S.fail ? kWaitNs / 4 : kWaitNs) && !S.fail) {
            S.fail = 1;
            atomicOr(status, 1 << LDN_ERR_TIMEOUT);
        }
        __syncthreads();
        cluster_sync();
        if (tid == 0) {
            const uint32_t peer_sent = ld_shared_cluster_u32(mapa_shared(smem_u32(&S.sent), (uint32_t)(prank ^ 1)));
            if (peer_sent > S.recvd) mbar_wait(&S.bar_recv, S.recvd & 1, kWaitNs / 4);
        }
        __syncthreads();
        cluster_sync();   // the peer has read this CTA's counter
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kCols);
}

}  // namespace

bool chunk_tc_supported(const ChunkArgs &a)
{
    // KDA reads its per-channel log-gates as float4: the gate tensor must be 16-byte
    // aligned; so must Gated DeltaNet-2's erase and write gates
    const bool a16 = ((uintptr_t)a.gate & 15u) == 0;
    const bool kda_ok = a.mode == LDN_KDA && a16;
    const bool g2_ok = a.mode == LDN_GDN2 && a16 && a.erase && a.write && ((uintptr_t)a.erase & 15u) == 0 &&
                       ((uintptr_t)a.write & 15u) == 0;
    return a.dtype == LDN_BF16 && a.dk == kDK && a.dv % kDVS == 0 && a.chunk == kC &&
           (a.mode == LDN_DELTANET || a.mode == LDN_GDN || kda_ok || g2_ok);
}

int sm_count()
{
    static int sms[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms[dev] = 0;
    return sms[dev];
}

namespace {
template <int KIND>
cudaError_t launch_tc(const ChunkArgs &a, uint8_t *ws, cudaStream_t st)
{
    constexpr bool SPLIT = KIND == kSplit, PAIR = KIND == kPair, PREPX = KIND == kPrepX;
    constexpr int LK = PAIR ? kFused : KIND;   // shared-memory plan
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16_4d(&tq, a.q, kDK, a.H, a.T, a.B, 64, kC) ||
        !make_tmap_bf16_4d(&tk, a.k, kDK, a.H, a.T, a.B, 64, kC) ||
        !make_tmap_bf16_4d(&tv, a.v, a.dv, a.H, a.T, a.B, 64, kC))
        return cudaErrorInvalidValue;
    int cpr = 0;
    long long grid = (long long)a.B * a.H * (a.dv / kDVS);
    if (SPLIT || PREPX) {
        // chunk ranges per sequence so that the CTAs fill the SMs once (split: one CTA per
        // SM; prep-X: two for DeltaNet / Gated DeltaNet, whose plan takes half an SM)
        const int nchunks = (a.T + kC - 1) / kC;
        const long long heads = (long long)a.B * a.H;
        const bool kda = a.mode == LDN_KDA || a.mode == LDN_GDN2;
        const long long slots = (long long)sm_count() * (PREPX && !kda ? 2 : 1);
        long long nranges = max(1LL, min((long long)nchunks, slots > 0 ? slots / heads : 1LL));
        if (PREPX && slots > 0) {   // ranges of about the same length on every slot
            const long long per = (heads * nchunks + slots - 1) / slots;
            nranges = min((long long)nchunks, max(1LL, (nchunks + per - 1) / per));
        }
        cpr = (int)((nchunks + nranges - 1) / nranges);
        nranges = (nchunks + cpr - 1) / cpr;
        grid = heads * nranges;
    }
    auto go = [&](auto kern, uint32_t smem) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (KIND == kFed) {   // may start while the prep-X grid before it drains (see griddep_wait)
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)grid);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, a.beta, a.gate, a.S0, (__nv_bfloat16 *)a.out,
                                      a.S_final, a.T, a.H, a.dv, a.status, ws, cpr, a.erase, a.write, a.chunk_states);
        }
        if (PAIR) {   // clusters of the two dv slices of a (b, h): consecutive blocks
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)grid);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, a.beta, a.gate, a.S0, (__nv_bfloat16 *)a.out,
                                      a.S_final, a.T, a.H, a.dv, a.status, ws, cpr, a.erase, a.write, a.chunk_states);
        }
        kern<<<(unsigned)grid, PREPX ? kPrepThreads : kThreads, smem, st>>>(
            tq, tk, tv, a.beta, a.gate, a.S0, (__nv_bfloat16 *)a.out, a.S_final, a.T, a.H, a.dv, a.status, ws, cpr,
            a.erase, a.write, a.chunk_states);
        return cudaGetLastError();
    };
    if (a.mode == LDN_GDN) return go(chunk_tc_kernel<LDN_GDN, KIND>, Layout<LDN_GDN, LK>::bytes);
    if constexpr (!PAIR) {
        if (a.mode == LDN_KDA) return go(chunk_tc_kernel<LDN_KDA, KIND>, Layout<LDN_KDA, LK>::bytes);
        if (a.mode == LDN_GDN2) return go(chunk_tc_kernel<LDN_GDN2, KIND>, Layout<LDN_GDN2, LK>::bytes);
    }
    return go(chunk_tc_kernel<LDN_DELTANET, KIND>, Layout<LDN_DELTANET, LK>::bytes);
}
}  // namespace

cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st) { return launch_tc<kFused>(a, nullptr, st); }

bool chunk_pair_supported(const ChunkArgs &a)
{
    return chunk_tc_supported(a) && (a.mode == LDN_DELTANET || a.mode == LDN_GDN) && a.dv == 2 * kDVS;
}

cudaError_t launch_chunk_pair(const ChunkArgs &a, cudaStream_t st) { return launch_tc<kPair>(a, nullptr, st); }

// Which tensor-core variant is expected to be fastest: a cost model in waves of
// CTAs x chunks per CTA x measured time per chunk on GB300 --
//   fused: 10 us + waves x chunks x 4.0 us (GDN / DeltaNet) or 7.9 us (KDA);
//   pair: 10 us + waves x chunks x 5.0 us (measured: each CTA's preparation waits for
//     tiles that a third ring stage frees only late, and runs slower beside the busier
//     serial warps);
//   split: 20 us + preparation waves x chunks per range x 5.4 / 10.8 us + state waves (one
//     CTA per (b, h)) x chunks x 1.6 us (with a sequence split: 10 us + 2 x chunks per segment
//     x 1.6 us + 4 us per scan step);
//   pre-solved: 22 us + prep-X chunks per slot x 3.2 / 6.6 us (two / one CTAs per SM) +
//     waves x chunks x 2.2 / 6.3 us.
// The fused and pair kernels win when their CTAs fill the SMs once and the sequences are
// short; the pre-solved variant when many sequences fill the SMs (GDN / DeltaNet); the
// split variant when few sequences are long, or for KDA.
int chunk_tc_pick(const ChunkArgs &a, bool split_ok, bool presolved_ok)
{
    const bool pair_ok = chunk_pair_supported(a);
    const int sms = sm_count();
    if (sms <= 0) return pair_ok ? LDN_VARIANT_PAIR : LDN_VARIANT_TENSOR;
    const bool kda = a.mode == LDN_KDA || a.mode == LDN_GDN2;
    const double t_fused = kda ? 7.9 : 4.0, t_pair = 5.0, t_prep = kda ? 10.8 : 5.4, t_state = 1.6;
    const double t_px = kda ? 6.6 : 3.2, t_fed = kda ? 6.3 : 2.2;
    const long long heads = (long long)a.B * a.H, nchunks = (a.T + kC - 1) / kC;
    const long long slices = heads * (a.dv / kDVS);
    const long long waves_f = (slices + sms - 1) / sms;
    const long long nranges = std::max(1LL, std::min(nchunks, sms / heads));
    const long long cpr = (nchunks + nranges - 1) / nranges;
    const long long waves_p = (heads * ((nchunks + cpr - 1) / cpr) + sms - 1) / sms;
    const long long px_slots = (long long)sms * (kda ? 1 : 2);
    int best = LDN_VARIANT_TENSOR;
    double cost = 10.0 + (double)waves_f * nchunks * t_fused;
    if (pair_ok) {
        const double pair = 10.0 + (double)waves_f * nchunks * t_pair;
        if (pair < cost) { cost = pair; best = LDN_VARIANT_PAIR; }
    }
    if (split_ok) {
        // a sequence split runs the state recurrence twice over segments of cps chunks, with a
        // scan of 3 us per segment between (chunk_state.cu)
        const int nseg = split_segments((int)heads, (int)nchunks, a.dv);
        const double state = nseg >= 3 ? 10.0 + 2.0 * ((nchunks + nseg - 1) / nseg) * t_state + 4.0 * (nseg - 2)
                                        : (double)((heads + sms - 1) / sms) * nchunks * t_state;
        const double split = 20.0 + (double)waves_p * cpr * t_prep + state;
        if (split < cost) { cost = split; best = LDN_VARIANT_SPLIT; }
    }
    if (presolved_ok) {
        const double pre = 22.0 + (double)((heads * nchunks + px_slots - 1) / px_slots) * t_px +
                           (double)waves_f * nchunks * t_fed;
        if (pre < cost) { cost = pre; best = LDN_VARIANT_PRESOLVED; }
    }
    return best;
}

size_t presolved_workspace_bytes(int B, int T, int H)
{
    return (size_t)B * H * (size_t)((T + kC - 1) / kC) * kXBytes;
}

cudaError_t launch_chunk_presolved(const ChunkArgs &a, uint8_t *ws, cudaStream_t st)
{
    cudaError_t e = launch_tc<kPrepX>(a, ws, st);
    if (e != cudaSuccess) return e;
    return launch_tc<kFed>(a, ws, st);
}

cudaError_t launch_chunk_solve(const ChunkArgs &a, uint8_t *ws, cudaStream_t st)
{
    return launch_tc<kPrepX>(a, ws, st);
}

cudaError_t launch_chunk_split(const ChunkArgs &a, uint8_t *ws, size_t ws_bytes, cudaStream_t st)
{
    cudaError_t e = launch_tc<kSplit>(a, ws, st);
    if (e != cudaSuccess) return e;
    return launch_chunk_state(a, ws, ws_bytes, st);
}

}  // namespace ldn
