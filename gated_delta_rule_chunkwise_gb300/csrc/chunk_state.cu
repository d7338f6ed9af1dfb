// State kernel of the split variant: the chunk-to-chunk recurrence, reading
// every chunk's state-independent operands from the workspace written by the
// preparation kernel (chunk_tc_kernel<MODE, true>).
//
// With H = S^T ([dk][dv]) the incoming state of a chunk, the workspace holds
// A5 = [Q~ ; -W] (fp16, 128 x dk, swizzled K-major: the exact shared-memory
// image of the MMA A operand), RV = [P U' ; U'] (fp16, 128 x 64 per dv slice),
// K~ = K scaled by e^{g_C - g} (fp16, 64 x dk) and e^{g_C} per key channel, so
// that for every chunk (chunk algebra derived from the per-token rules of the
// linear-attention notes, Sec. 2.3-2.5):
//   [O ; U] = RV + A5 H          (one M = 128, N = dv tcgen05.mma chain: MMA5)
//   H      <- Diag(e^{g_C}) H + K~^T U                      (MMA6)
// and O (rows 0..63) is the chunk's output.
//
// chunk_state_kernel<NS>: one CTA per (b, h) over the whole dv = 64 NS, 128 threads
// per 64-wide dv slice: thread = (row of the fp32 state, dv slice), the row's slice
// held in registers.  It runs dv = 64 (NS = 1); dv = 128 runs the transposed kernel
// further below (chunk_state_t_kernel), whose epilogue work spreads over every SM
// sub-partition instead of the two that own the U rows' lanes.  The operands of a chunk land in
// a two-stage ring in two parts with a barrier each: A5 (read by MMA5 at the
// start of the chunk) and RV | K~ | e^{g_C} (read later in the chunk).  A5 of
// chunk c + 2 is loaded as soon as MMA5 of chunk c has read its slot, the rest of
// chunk c + 1 when chunk c - 1 has ended, so each part has more than a chunk step
// to land.  Every wait is bounded (2 s); a timeout sets LDN_ERR_TIMEOUT,
// in-flight work is drained with bounded waits, TMEM is freed and the CTA
// returns.
#include "ldn_internal.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace ldn {
namespace {
using namespace sm100;

constexpr int kC = 64;
constexpr int kDK = 128;
constexpr int kStages = 2;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kBar = 1;
constexpr uint32_t kBarU = 2;             // the U rows' threads: MMA6 waits only for them
constexpr int kIssuer6 = 64;

// Shared-memory plan for NS 64-wide dv slices (dv = 64 NS); a stage is the workspace's chunk
// image as it is: A5 | RV slices | K~ | e^{g_C}
template <int NS>
struct Plan {
    static constexpr int kThreads = 128 * NS;
    static constexpr int kDV = 64 * NS;
    static constexpr uint32_t kOA5 = 0, kORV = 32768, kOKT = kORV + NS * 16384, kOEG = kOKT + 16384;
    static constexpr uint32_t kTxA = 32768, kTxB = NS * 16384 + 16384 + 512;
    static constexpr uint32_t kStageBytes = (kOEG + 512 + 1023) / 1024 * 1024;
    static constexpr uint32_t kOffHB = kStages * kStageBytes;   // H fp16, MN-major: NS blocks of 128 x 64
    static constexpr uint32_t kOffUB = kOffHB + NS * 16384;     // U fp16, MN-major: NS blocks of 64 x 64
    static constexpr uint32_t kOffBars = kOffUB + NS * 8192;
    static constexpr uint32_t kSmemBytes = kOffBars + 128 + 1024;   // bars: a[2], b[2], smma, drain[2], s6
    static constexpr uint32_t kColD5 = 0, kColD6 = kDV, kTmemCols = 2 * kDV;
    static_assert(kSmemBytes <= 232448, "shared memory plan exceeds 227 KB");
    static_assert(kOKT == split_kt_off(kDV) && kOEG == split_eg_off(kDV), "stage must mirror the workspace image");
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
__device__ __forceinline__ void st_row16(uint8_t *block, int row, int col, const float *v)
{
    *reinterpret_cast<uint4 *>(block + sw128_offset(row, col)) =
        make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
    *reinterpret_cast<uint4 *>(block + sw128_offset(row, col + 8)) =
        make_uint4(pack_h2(v[8], v[9]), pack_h2(v[10], v[11]), pack_h2(v[12], v[13]), pack_h2(v[14], v[15]));
}

// Sequence split (`pass` 1 and 2; dv = 128): the chunks of each (b, h) form `nseg` segments of
// `cps` chunks.  Pass 1, per (b, h): segment 0 from S0 with its outputs (its final state is
// the state entering segment 1), and for every segment s = 1 .. nseg-2 its affine map
// H_out = M_s H_in + N_s: N_s from a zero state, M_s (dk x dk) from the identity with the U'
// term dropped, no outputs.  A scan then gives every segment its incoming state, and pass 2
// runs segments 1 .. nseg-1 from them with their outputs (the last one writes S_final).  Pass
// 0 is the whole sequence from S0.  `seg` holds, per (b, h), the states entering the segments
// and the maps: [3 nseg][dk][128] fp32 (seg_slot()).
__host__ __device__ constexpr size_t seg_slot(int unit, int nseg, int kind, int s)
{   // kind 0: state entering segment s; 1: N_s; 2: M_s
    return (((size_t)unit * 3 * nseg + (size_t)kind * nseg + s) * kDK) * 128;
}
__host__ __device__ constexpr int seg_jobs(int pass, int nseg)
{   // CTAs per (b, h)
    return pass == 0 ? 1 : pass == 1 ? 1 + 2 * (nseg - 2) : nseg - 1;
}

template <int NS>
__global__ void __launch_bounds__(Plan<NS>::kThreads, 1)
chunk_state_kernel(const uint8_t *__restrict__ ws, const float *S0, __nv_bfloat16 *__restrict__ out, float *S_final,
                   int T, int H, int *status, int pass, int nseg, int cps, float *seg)
{
    using P = Plan<NS>;
    constexpr int kThreads = P::kThreads, dv = P::kDV;
    extern __shared__ uint8_t dsmem[];
    uint8_t *sm = dsmem + ((1024u - (smem_u32(dsmem) & 1023u)) & 1023u);
    uint8_t *HB = sm + P::kOffHB, *UB = sm + P::kOffUB;
    uint64_t *full_a = reinterpret_cast<uint64_t *>(sm + P::kOffBars);   // [kStages]: A5
    uint64_t *full_b = full_a + kStages;                                 // [kStages]: RV | K~ | e^{g_C}
    uint64_t *smma = full_b + kStages;
    uint64_t *drain = smma + 1;   // [2]: one per MMA-issuing thread (0, kIssuer6)
    // MMA6 completes on a barrier of its own: its issuer does not wait for the O rows to
    // have seen MMA5's completion, and one barrier for both would let a late O-row waiter
    // see two phases pass and wait for a third
    uint64_t *s6 = drain + 2;
    __shared__ uint32_t tmem_base_s;
    __shared__ int fail;

    const int st = threadIdx.x, warp = st >> 5;
    const int r = st & 127, hf = st >> 7;   // state row (TMEM lane), dv slice
    const int n0 = hf * 64;
    const int nchunks = (T + kC - 1) / kC;
    // this CTA's job: (b, h), chunk range, initial state, whether U' and outputs count, where the
    // final state goes
    const int jobs = seg_jobs(pass, nseg);
    const int unit = blockIdx.x / jobs, j = blockIdx.x % jobs;
    int sg = 0, kind = 0;   // kind 0: a run with outputs; 1: N map; 2: M map
    if (pass == 1 && j >= 1) { sg = 1 + (j - 1) / 2; kind = 1 + (j - 1) % 2; }
    else if (pass == 2) sg = 1 + j;
    const int cs = pass == 0 ? 0 : sg * cps, ce = pass == 0 ? nchunks : min(nchunks, (sg + 1) * cps);
    const int nloc = ce - cs;
    const bool use_rv = kind != 2, write_out = kind == 0;
    const int b = unit / H, h = unit % H;
    const size_t ub = split_unit_bytes(dv);
    const uint8_t *base = ws + ((size_t)unit * nchunks + cs) * ub;   // operands of the CTA's first chunk
    const float *init = pass == 0 || (pass == 1 && sg == 0) ? (S0 ? S0 + (size_t)unit * kDK * dv : nullptr)
                        : pass == 2 ? seg + seg_slot(unit, nseg, 0, sg) : nullptr;
    float *fin = pass == 0 ? (S_final ? S_final + (size_t)unit * kDK * dv : nullptr)
                 : pass == 1 ? seg + seg_slot(unit, nseg, sg == 0 ? 0 : kind, sg == 0 ? 1 : sg)
                 : sg == nseg - 1 ? (S_final ? S_final + (size_t)unit * kDK * dv : nullptr) : nullptr;
    const uint32_t lane_base = (32u * (uint32_t)(warp & 3)) << 16;

    if (st == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_a[i], 1);
            mbar_init(&full_b[i], 1);
        }
        mbar_init(smma, 1);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        mbar_init(s6, 1);
        fence_mbar_init();
        fail = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, P::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_s;

    // chunk last loaded into each slot (thread 0)
    int pend_a[kStages] = {-1, -1}, pend_b[kStages] = {-1, -1};
    // A map (no outputs) loads only what its U rows use: the -W rows of A5 (rows 64..127 of
    // both 64-column K blocks), U' (rows 64..127 of each RV slice; none for M), K~ and e^{g_C}.
    // The rows it leaves stale feed only the O rows of its products, which it never reads.
    auto load_a = [&](int c) {
        const int s = c & 1;
        uint8_t *d = sm + s * P::kStageBytes + P::kOA5;
        const uint8_t *u = base + (size_t)c * ub;
        pend_a[s] = c;
        if (write_out) {
            mbar_arrive_expect_tx(&full_a[s], P::kTxA);
            bulk_load(d, u, P::kTxA, &full_a[s]);
        } else {
            mbar_arrive_expect_tx(&full_a[s], P::kTxA / 2);
            bulk_load(d + 8192, u + 8192, 8192, &full_a[s]);
            bulk_load(d + 16384 + 8192, u + 16384 + 8192, 8192, &full_a[s]);
        }
    };
    auto load_b = [&](int c) {
        const int s = c & 1;
        uint8_t *d = sm + s * P::kStageBytes;
        const uint8_t *u = base + (size_t)c * ub;
        pend_b[s] = c;
        if (write_out) {
            mbar_arrive_expect_tx(&full_b[s], P::kTxB);
            bulk_load(d + P::kORV, u + kSplitRvOff, P::kTxB, &full_b[s]);
        } else {
            mbar_arrive_expect_tx(&full_b[s], (use_rv ? NS * 8192 : 0) + 16384 + 512);
            if (use_rv)
                for (int q = 0; q < NS; ++q)
                    bulk_load(d + P::kORV + q * 16384 + 8192, u + kSplitRvOff + q * 16384 + 8192, 8192, &full_b[s]);
            bulk_load(d + P::kOKT, u + split_kt_off(dv), 16384 + 512, &full_b[s]);
        }
    };
    if (st == 0)
        for (int c = 0; c < kStages && c < nloc; ++c) {
            load_a(c);
            load_b(c);
        }

    auto vote = [&](bool ok) -> bool {   // same decision in every thread
        const bool bad = named_sync_or(kBar, kThreads, !ok || fail != 0);
        if (bad && st == 0) fail = 1;
        return !bad;
    };
    // MMA completion: every thread polls the commit barrier itself (no role-wide
    // barrier on this path); a timeout only marks the CTA failed, and the vote at
    // the end of the chunk takes every thread out of the loop together.
    uint32_t sphase = 0;
    auto wait_smma = [&]() {
        if (!mbar_wait(smma, sphase, kWaitNs)) fail = 1;
        sphase ^= 1u;
        tc_fence_after();
    };
    const uint32_t id_mma5 = idesc_f16kind_f32(128, dv, 0, 1, kMmaF16);   // A K-major, B MN-major
    const uint32_t id_mma6 = idesc_f16kind_f32(128, dv, 1, 1, kMmaF16);   // both MN-major

    float Hreg[64];
    {
        const float *src = init ? init + (size_t)r * dv + n0 : nullptr;
#pragma unroll
        for (int n = 0; n < 64; n += 4) {
            const float4 x = src ? *reinterpret_cast<const float4 *>(src + n) : make_float4(0.f, 0.f, 0.f, 0.f);
            Hreg[n] = x.x; Hreg[n + 1] = x.y; Hreg[n + 2] = x.z; Hreg[n + 3] = x.w;
        }
        if (kind == 2)   // M map: columns n0 .. n0 + 63 of the identity
#pragma unroll
            for (int n = 0; n < 64; ++n) Hreg[n] = r == n0 + n ? 1.f : 0.f;
#pragma unroll
        for (int n = 0; n < 64; n += 16) st_row16(HB + hf * 16384, r, n, &Hreg[n]);
    }
    fence_proxy_async_smem();
    named_sync(kBar, kThreads);

    const bool top = r < 64;
    // one vote per chunk, taken at the barrier that ends the chunk: thread 0 first waits for
    // the next chunk's A5, so every thread leaves the loop at the same chunk
    bool go = nloc > 0 && vote(st == 0 ? mbar_wait(&full_a[0], 0, kWaitNs) : true);
    for (int lc = 0; go && lc < nloc; ++lc) {   // lc: the chunk's place in the CTA's range
        const int c = cs + lc, s = lc & 1, t0 = c * kC, L = min(kC, T - t0);
        const uint32_t par = (uint32_t)(lc >> 1) & 1u;
        uint8_t *stg = sm + s * P::kStageBytes;

        // ---- MMA5: D5 = [Q~ ; -W] H
        if (st == 0) {
            tc_fence_after();
            const uint32_t a5_s = smem_u32(stg + P::kOA5), hb_s = smem_u32(HB);
            for (int k = 0; k < kDK / 16; ++k)
                umma_bf16(tbase + P::kColD5, kmajor_desc(a5_s, 128, k), mnmajor_desc(hb_s, 128, k), id_mma5, k > 0);
            umma_commit(smma);
            // the rest of chunk lc + 1 goes where chunk lc - 1's was: every reader of it was done
            // at the vote that ended chunk lc - 1 (issued behind this chunk's first product)
            if (lc >= 1 && lc + 1 < nloc) load_b(lc + 1);
        }
        wait_smma();
        // MMA5 has read this chunk's A5: chunk lc + 2's takes its slot
        if (st == 0 && lc + 2 < nloc) load_a(lc + 2);

        // ---- O = P U' + Q~ H (rows 0..63) -> out; U = U' - W H (rows 64..127) -> UB
        if (!mbar_wait(&full_b[s], par, kWaitNs)) fail = 1;
        {
            const uint8_t *rv = stg + P::kORV + hf * 16384;
            float v[64];   // the whole slice row in one TMEM round trip
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16(tbase + lane_base + P::kColD5 + n0 + 16 * q, v + 16 * q);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 8 && use_rv; ++q) {
                const uint4 w = *reinterpret_cast<const uint4 *>(rv + sw128_offset(r, 8 * q));
                const __half2 *h2 = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __half22float2(h2[i]);
                    v[8 * q + 2 * i] += f.x;
                    v[8 * q + 2 * i + 1] += f.y;
                }
            }
            if (top) {
                if (write_out && r < L) {
                    uint4 *dst = reinterpret_cast<uint4 *>(out + (((size_t)b * T + t0 + r) * H + h) * dv + n0);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_uint4(pack_bf2(v[8 * q], v[8 * q + 1]), pack_bf2(v[8 * q + 2], v[8 * q + 3]),
                                            pack_bf2(v[8 * q + 4], v[8 * q + 5]), pack_bf2(v[8 * q + 6], v[8 * q + 7]));
                }
            } else {
#pragma unroll
                for (int n = 0; n < 64; n += 16) st_row16(UB + hf * 8192, r - 64, n, v + n);
            }
        }
        // MMA6 reads U only: the U rows' threads meet without the O rows' threads,
        // whose output stores overlap MMA6
        if (!top) {
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarU, kThreads / 2);
        }

        // ---- MMA6: D6 = K~^T U
        if (st == kIssuer6) {
            tc_fence_after();
            const uint32_t kt_s = smem_u32(stg + P::kOKT), ub_s = smem_u32(UB);
            for (int k = 0; k < kC / 16; ++k)
                umma_bf16(tbase + P::kColD6, mnmajor_desc(kt_s, 64, k), mnmajor_desc(ub_s, 64, k), id_mma6, k > 0);
            umma_commit(s6);
        }
        if (!mbar_wait(s6, (uint32_t)(lc & 1), kWaitNs)) fail = 1;
        tc_fence_after();

        // ---- H <- e^{g_C} H + K~^T U (row r), fp16 copy for the next MMA5
        {
            const float g = reinterpret_cast<const float *>(stg + P::kOEG)[r];
            float v[64];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16(tbase + lane_base + P::kColD6 + n0 + 16 * q, v + 16 * q);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                Hreg[i] = g * Hreg[i] + v[i];
                v[i] = Hreg[i];
            }
#pragma unroll
            for (int n = 0; n < 64; n += 16) st_row16(HB + hf * 16384, r, n, v + n);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        const int cn = lc + 1;
        go = vote(st == 0 && cn < nloc ? mbar_wait(&full_a[cn & 1], (uint32_t)(cn >> 1) & 1u, kWaitNs) : true);
    }

    if (fail == 0 && fin) {
        float *dst = fin + (size_t)r * dv + n0;
#pragma unroll
        for (int n = 0; n < 64; n += 4)
            *reinterpret_cast<float4 *>(dst + n) = make_float4(Hreg[n], Hreg[n + 1], Hreg[n + 2], Hreg[n + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (fail && (st == 0 || st == kIssuer6)) {
        // drain: the MMAs issued by this thread, then the loads still in flight (bounded)
        const int i = st == 0 ? 0 : 1;
        if (st == 0) atomicOr(status, 1 << LDN_ERR_TIMEOUT);
        umma_commit(&drain[i]);
        mbar_wait(&drain[i], 0, kWaitNs / 4);
        if (st == 0)
            for (int s = 0; s < kStages; ++s) {
                if (pend_a[s] >= 0) mbar_wait(&full_a[s], (uint32_t)(pend_a[s] >> 1) & 1u, kWaitNs / 4);
                if (pend_b[s] >= 0) mbar_wait(&full_b[s], (uint32_t)(pend_b[s] >> 1) & 1u, kWaitNs / 4);
            }
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, P::kTmemCols);
}

// dv = 128: the same recurrence transposed, so that the lanes of tensor memory are dv columns
// and any warp may take any rows of [O ; U] (D^T = H^T [Q~ ; -W]^T, the H^T and U^T operands
// in tensor memory):
//   [O ; U]^T = RV^T + H^T A5^T       (MMA5: A = H^T in TMEM, B = the A5 image, K-major)
//   H^T      <- H^T Diag(e^{g_C}) + U^T K~   (MMA6: A = U^T in TMEM, B = the K~ image, MN-major)
// The workspace's RV part holds RV^T for dv = 128 (block 0 = (P U')^T, block 1 = U'^T, rows =
// dv columns).  256 threads: lane n = dv column, warp half hh; in the epilogue half 0 forms U^T
// (one warp on every SM sub-partition: the step's critical path) and half 1 the output, staged
// in shared memory in the output tensor's swizzled tile layout and sent by one TMA store; in the
// state update half hh holds key channels 64 hh .. 64 hh + 63 of row n of H^T.  A5 lands in a
// two-stage ring, RV^T | K~ (and e^{g_C}, in a ring of its own) in a three-stage one, each part
// loaded two chunks ahead.
struct PlanT {
    static constexpr int kThreads = 256;
    static constexpr int kAStages = 2, kBStages = 3;
    static constexpr uint32_t kA = 32768;                          // A5 image
    static constexpr uint32_t kORV = 0, kOKT = 32768;              // within a B stage
    static constexpr uint32_t kB = 49152;                          // B stage: RV^T | K~
    static constexpr uint32_t kTxB = kB + 512;                     // and e^{g_C}
    static constexpr uint32_t kOffB = kAStages * kA;
    static constexpr uint32_t kOffO = kOffB + kBStages * kB;       // output tile: 2 blocks of 64 x 64 bf16
    static constexpr uint32_t kOffEG = kOffO + 16384;              // e^{g_C}: [kBStages][128] fp32
    static constexpr uint32_t kOffBars = kOffEG + kBStages * 512;
    static constexpr uint32_t kSmemBytes = kOffBars + 128 + 1024;   // bars: a[2], b[3], smma, s6, drain[2]
    // tensor memory: D5^T, D6^T (fp32, 128 columns each), H^T (fp16 pairs, 64), U^T (fp16 pairs, 32)
    static constexpr uint32_t kColD5 = 0, kColD6 = 128, kColH = 256, kColU = 320, kTmemCols = 512;
    static_assert(kSmemBytes <= 232448, "shared memory plan exceeds 227 KB");
    static_assert(kOKT == split_kt_off(128) - kSplitRvOff && kB == split_eg_off(128) - kSplitRvOff,
                  "B stage must mirror the workspace image");
};
constexpr uint32_t kBarO = 3;   // the output half's threads: the tile is complete before its store

__device__ __forceinline__ void pack_h16(const float *v, uint32_t *w)
{
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_h2(v[2 * i], v[2 * i + 1]);
}

__global__ void __launch_bounds__(PlanT::kThreads, 1)
chunk_state_t_kernel(const __grid_constant__ CUtensorMap tm_out, const uint8_t *__restrict__ ws, const float *S0,
                     float *S_final, int T, int H, int *status, int pass, int nseg, int cps, float *seg)
{
    using P = PlanT;
    constexpr int kThreads = P::kThreads, dv = 128;
    extern __shared__ uint8_t dsmem[];
    uint8_t *sm = dsmem + ((1024u - (smem_u32(dsmem) & 1023u)) & 1023u);
    uint64_t *full_a = reinterpret_cast<uint64_t *>(sm + P::kOffBars);   // [kAStages]: A5
    uint64_t *full_b = full_a + P::kAStages;                             // [kBStages]: RV^T | K~ | e^{g_C}
    uint64_t *smma = full_b + P::kBStages;
    uint64_t *s6 = smma + 1;
    uint64_t *drain = s6 + 1;   // [2]: unused slot kept for the layout; thread 0 issues every MMA
    __shared__ uint32_t tmem_base_s;
    __shared__ int fail;

    const int st = threadIdx.x, warp = st >> 5;
    const int n = st & 127, hh = st >> 7;   // dv column (TMEM lane), warp half
    const int nchunks = (T + kC - 1) / kC;
    const int jobs = seg_jobs(pass, nseg);
    const int unit = blockIdx.x / jobs, j = blockIdx.x % jobs;
    int sg = 0, kind = 0;   // kind 0: a run with outputs; 1: N map; 2: M map
    if (pass == 1 && j >= 1) { sg = 1 + (j - 1) / 2; kind = 1 + (j - 1) % 2; }
    else if (pass == 2) sg = 1 + j;
    const int cs = pass == 0 ? 0 : sg * cps, ce = pass == 0 ? nchunks : min(nchunks, (sg + 1) * cps);
    const int nloc = ce - cs;
    const bool use_rv = kind != 2, write_out = kind == 0;
    const int b = unit / H, h = unit % H;
    const size_t ub = split_unit_bytes(dv);
    const uint8_t *base = ws + ((size_t)unit * nchunks + cs) * ub;
    const float *init = pass == 0 || (pass == 1 && sg == 0) ? (S0 ? S0 + (size_t)unit * kDK * dv : nullptr)
                        : pass == 2 ? seg + seg_slot(unit, nseg, 0, sg) : nullptr;
    float *fin = pass == 0 ? (S_final ? S_final + (size_t)unit * kDK * dv : nullptr)
                 : pass == 1 ? seg + seg_slot(unit, nseg, sg == 0 ? 0 : kind, sg == 0 ? 1 : sg)
                 : sg == nseg - 1 ? (S_final ? S_final + (size_t)unit * kDK * dv : nullptr) : nullptr;
    const uint32_t lane_base = (32u * (uint32_t)(warp & 3)) << 16;

    if (st == 0) {
        for (int i = 0; i < P::kAStages; ++i) mbar_init(&full_a[i], 1);
        for (int i = 0; i < P::kBStages; ++i) mbar_init(&full_b[i], 1);
        mbar_init(smma, 1);
        mbar_init(s6, 1);
        mbar_init(&drain[0], 1);
        fence_mbar_init();
        fail = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, P::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_s;
    const uint32_t trow = tbase + lane_base;   // this warp's lanes

    // loads are issued by kLoader (a U-half thread idle while MMA6 runs), not by the MMA issuer
    constexpr int kLoader = 96;
    int pend_a[P::kAStages] = {-1, -1}, pend_b[P::kBStages] = {-1, -1, -1};   // kLoader
    // A map (no outputs) loads only what its U rows use: the -W rows of A5 (rows 64..127 of
    // both 64-column K blocks), U'^T (RV^T block 1; none for M), K~ and e^{g_C}.  What it leaves
    // stale feeds only the O columns of its products, which it never reads.
    auto load_a = [&](int c) {
        const int s = c % P::kAStages;
        uint8_t *d = sm + s * P::kA;
        const uint8_t *u = base + (size_t)c * ub;
        pend_a[s] = c;
        if (write_out) {
            mbar_arrive_expect_tx(&full_a[s], P::kA);
            bulk_load(d, u, P::kA, &full_a[s]);
        } else {
            mbar_arrive_expect_tx(&full_a[s], P::kA / 2);
            bulk_load(d + 8192, u + 8192, 8192, &full_a[s]);
            bulk_load(d + 16384 + 8192, u + 16384 + 8192, 8192, &full_a[s]);
        }
    };
    auto load_b = [&](int c) {
        const int s = c % P::kBStages;
        uint8_t *d = sm + P::kOffB + s * P::kB;
        const uint8_t *u = base + (size_t)c * ub + kSplitRvOff;
        pend_b[s] = c;
        mbar_arrive_expect_tx(&full_b[s], write_out ? P::kTxB : (use_rv ? 16384 : 0) + 16384 + 512);
        if (write_out) {
            bulk_load(d, u, P::kB, &full_b[s]);
        } else {
            if (use_rv) bulk_load(d + 16384, u + 16384, 16384, &full_b[s]);
            bulk_load(d + P::kOKT, u + P::kOKT, 16384, &full_b[s]);
        }
        bulk_load(sm + P::kOffEG + s * 512, u + P::kB, 512, &full_b[s]);
    };
    // chunk images four ahead are pulled into L2, so that the loads into the rings meet L2
    auto prefetch = [&](int c) {
        const uint8_t *u = base + (size_t)c * ub;
        if (write_out) {
            bulk_prefetch_l2(u, (uint32_t)ub);
        } else {
            bulk_prefetch_l2(u + 8192, 8192);
            bulk_prefetch_l2(u + 16384 + 8192, 8192);
            if (use_rv) bulk_prefetch_l2(u + kSplitRvOff + 16384, 16384);
            bulk_prefetch_l2(u + kSplitRvOff + P::kOKT, 16384 + 512);
        }
    };
    if (st == kLoader) {
        for (int c = 0; c < 2 && c < nloc; ++c) {
            load_a(c);
            load_b(c);
        }
        for (int c = 2; c < 4 && c < nloc; ++c) prefetch(c);
    }

    auto vote = [&](bool ok) -> bool {   // same decision in every thread
        const bool bad = named_sync_or(kBar, kThreads, !ok || fail != 0);
        if (bad && st == 0) fail = 1;
        return !bad;
    };
    uint32_t sphase = 0;
    auto wait_smma = [&]() {
        if (!mbar_wait(smma, sphase, kWaitNs)) fail = 1;
        sphase ^= 1u;
        tc_fence_after();
    };
    const uint32_t id_mma5 = idesc_f16kind_f32(128, 128, 0, 0, kMmaF16);   // A (TMEM) K-major, B K-major
    const uint32_t id_mma6 = idesc_f16kind_f32(128, 128, 0, 1, kMmaF16);   // B MN-major

    // H^T row n, key channels 64 hh .. 64 hh + 63 (fp32, registers); fp16 copy in TMEM
    float Hreg[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        const int k = 64 * hh + i;
        Hreg[i] = kind == 2 ? (n == k ? 1.f : 0.f) : init ? init[(size_t)k * dv + n] : 0.f;
    }
    {
        uint32_t w[32];
        pack_h16(Hreg, w);
        pack_h16(Hreg + 32, w + 16);
        tmem_st16u(trow + P::kColH + 32 * hh, w);
        tmem_st16u(trow + P::kColH + 32 * hh + 16, w + 16);
        tmem_st_wait();
    }
    tc_fence_before();

    // one vote per chunk, taken at the barrier that ends the chunk: thread 0 first waits for
    // the next chunk's A5, so every thread leaves the loop at the same chunk
    bool go = nloc > 0 && vote(st == 0 ? mbar_wait(&full_a[0], 0, kWaitNs) : true);
    for (int lc = 0; go && lc < nloc; ++lc) {
        const int c = cs + lc, t0 = c * kC;
        const int sa = lc % P::kAStages, sb = lc % P::kBStages;
        const uint8_t *stb = sm + P::kOffB + sb * P::kB;

        // ---- MMA5: D5^T = H^T A5^T
        if (st == 0) {
            tc_fence_after();
            const uint32_t a5_s = smem_u32(sm + sa * P::kA);
            for (int k = 0; k < kDK / 16; ++k)
                umma_ts(tbase + P::kColD5, tbase + P::kColH + 8 * k, kmajor_desc(a5_s, 128, k), id_mma5, k > 0);
            umma_commit(smma);
        }
        // while MMA5 runs: the B part of chunk lc + 2 goes where chunk lc - 1's was (every reader
        // of it was done at the vote that ended chunk lc - 1); chunk lc + 4 into L2
        if (st == kLoader) {
            if (lc + 2 < nloc) load_b(lc + 2);
            if (lc + 4 < nloc) prefetch(lc + 4);
        }
        wait_smma();

        if (!mbar_wait(&full_b[sb], (uint32_t)(lc / P::kBStages) & 1u, kWaitNs)) fail = 1;
        {
            // half 0: U^T = U'^T - (W H)^T (columns 64..127); half 1: O^T (columns 0..63)
            const uint8_t *rv = stb + P::kORV + (hh ? 0 : 16384);
            float v[64];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16(trow + P::kColD5 + (hh ? 0 : 64) + 16 * q, v + 16 * q);
            tmem_ld_wait();
            if (use_rv) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(rv + sw128_offset(n, 8 * q));
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __half22float2(h2[i]);
                        v[8 * q + 2 * i] += f.x;
                        v[8 * q + 2 * i + 1] += f.y;
                    }
                }
            }
            if (hh == 0) {
                uint32_t w[32];
                pack_h16(v, w);
                pack_h16(v + 32, w + 16);
                tmem_st16u(trow + P::kColU, w);
                tmem_st16u(trow + P::kColU + 16, w + 16);
                tmem_st_wait();
                tc_fence_before();
                named_sync(kBarU, kThreads / 2);
                if (st == kLoader && lc + 2 < nloc) load_a(lc + 2);   // where this chunk's A5 was
                // ---- MMA6: D6^T = U^T K~
                if (st == 0) {
                    tc_fence_after();
                    const uint32_t kt_s = smem_u32(stb + P::kOKT);
                    for (int k = 0; k < kC / 16; ++k)
                        umma_ts(tbase + P::kColD6, tbase + P::kColU + 8 * k, mnmajor_desc(kt_s, 64, k), id_mma6,
                                k > 0);
                    umma_commit(s6);
                }
            } else if (write_out) {
                // column n of the 64 x 128 output tile (rows past T are not stored); the store
                // of the chunk before finished reading the tile before the vote that ended it
                uint8_t *blk = sm + P::kOffO + (n >> 6) * 8192;
#pragma unroll
                for (int t = 0; t < 64; ++t)
                    *reinterpret_cast<__nv_bfloat16 *>(blk + sw128_offset(t, n & 63)) = __float2bfloat16_rn(v[t]);
                fence_proxy_async_smem();
                named_sync(kBarO, kThreads / 2);
                if (st == 128) {
                    tma_store_4d(&tm_out, sm + P::kOffO, 0, h, t0, b);
                    tma_store_4d(&tm_out, sm + P::kOffO + 8192, 64, h, t0, b);
                    bulk_commit();
                }
            }
        }
        if (!mbar_wait(s6, (uint32_t)(lc & 1), kWaitNs)) fail = 1;
        tc_fence_after();

        // ---- H^T <- H^T Diag(e^{g_C}) + D6^T (key channels 64 hh ..), fp16 copy for the next MMA5
        {
            const float4 *eg = reinterpret_cast<const float4 *>(sm + P::kOffEG + sb * 512) + 16 * hh;
            float v[64];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16(trow + P::kColD6 + 64 * hh + 16 * q, v + 16 * q);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 g = eg[q];
                Hreg[4 * q] = g.x * Hreg[4 * q] + v[4 * q];
                Hreg[4 * q + 1] = g.y * Hreg[4 * q + 1] + v[4 * q + 1];
                Hreg[4 * q + 2] = g.z * Hreg[4 * q + 2] + v[4 * q + 2];
                Hreg[4 * q + 3] = g.w * Hreg[4 * q + 3] + v[4 * q + 3];
            }
            uint32_t w[32];
            pack_h16(Hreg, w);
            pack_h16(Hreg + 32, w + 16);
            tmem_st16u(trow + P::kColH + 32 * hh, w);
            tmem_st16u(trow + P::kColH + 32 * hh + 16, w + 16);
            tmem_st_wait();
        }
        tc_fence_before();
        if (st == 128 && write_out) bulk_wait_read_all();   // the output tile may be written again
        const int cn = lc + 1;
        go = vote(st == 0 && cn < nloc
                      ? mbar_wait(&full_a[cn % P::kAStages], (uint32_t)(cn / P::kAStages) & 1u, kWaitNs)
                      : true);
    }

    if (fail == 0 && fin)
#pragma unroll
        for (int i = 0; i < 64; ++i) fin[(size_t)(64 * hh + i) * dv + n] = Hreg[i];
    if (st == 128) bulk_wait_all();   // the output stores are done
    tc_fence_before();
    __syncthreads();
    if (fail && st == 0) {   // drain: the MMAs this thread issued (bounded)
        atomicOr(status, 1 << LDN_ERR_TIMEOUT);
        umma_commit(&drain[0]);
        mbar_wait(&drain[0], 0, kWaitNs / 4);
    }
    if (fail && st == kLoader) {   // drain: the loads still in flight (bounded)
        for (int s = 0; s < P::kAStages; ++s)
            if (pend_a[s] >= 0)
                mbar_wait(&full_a[s], (uint32_t)(pend_a[s] / P::kAStages) & 1u, kWaitNs / 4);
        for (int s = 0; s < P::kBStages; ++s)
            if (pend_b[s] >= 0)
                mbar_wait(&full_b[s], (uint32_t)(pend_b[s] / P::kBStages) & 1u, kWaitNs / 4);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, P::kTmemCols);
}

// The scan of the sequence split: seg(0, s) = M_{s-1} seg(0, s-1) + N_{s-1}, s = 2 .. nseg-1, in
// fp32.  One CTA of 256 threads per ((b, h), 16-column slice of the state): its slice of each
// state depends only on its slice of the one before, which it keeps in shared memory, so the
// CTA runs its steps alone.  The maps of the next step are copied in (cp.async) while a step
// computes.  M sits in shared memory with rows padded to 132 words: a quarter-warp's 16-byte
// reads along a row hit distinct bank groups.  Thread = (row, 8 columns).
constexpr int kScanLd = kDK + 4;
constexpr int kScanM = kDK * kScanLd;                        // floats per M buffer
constexpr int kScanSmem = (2 * kScanM + 2 * kDK * 16 + kDK * 16) * 4;   // M[2], N[2], X

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__global__ void __launch_bounds__(256) seg_scan_kernel(float *seg, int nseg)
{
    extern __shared__ __align__(16) float ssm[];
    float *Ms = ssm, *Ns = ssm + 2 * kScanM, *Xs = Ns + 2 * kDK * 16;
    const int unit = blockIdx.x >> 3, c0 = (blockIdx.x & 7) * 16, tid = threadIdx.x;
    const int r = tid & 127, cc = 8 * (tid >> 7);
    auto fetch = [&](int s, int buf) {   // M_s and this CTA's columns of N_s into buffer buf
        const float *M = seg + seg_slot(unit, nseg, 2, s), *N = seg + seg_slot(unit, nseg, 1, s);
        for (int e = tid; e < kDK * kDK / 4; e += 256)
            cp_async16(Ms + buf * kScanM + (e >> 5) * kScanLd + 4 * (e & 31), M + 4 * e);
        for (int e = tid; e < kDK * 4; e += 256)
            cp_async16(Ns + buf * kDK * 16 + 4 * e, N + (e >> 2) * 128 + c0 + 4 * (e & 3));
        cp_async_commit();
    };
    if (nseg < 3) return;
    fetch(1, 1);   // M_{s-1} is used at step s from buffer (s - 1) & 1
    {
        const float *X = seg + seg_slot(unit, nseg, 0, 1);
        for (int e = tid; e < kDK * 4; e += 256)
            reinterpret_cast<float4 *>(Xs)[e] = *reinterpret_cast<const float4 *>(X + (e >> 2) * 128 + c0 + 4 * (e & 3));
    }
    for (int s = 2; s < nseg; ++s) {
        const int buf = s & 1;   // M_{s-1} is in buffer buf ^ 1; M_s goes to buffer buf
        cp_async_wait_all();
        __syncthreads();   // M_{s-1}, N_{s-1} and X landed; the step before is done with buffer buf
        if (s + 1 < nseg) fetch(s, buf);
        const float *Mb = Ms + (buf ^ 1) * kScanM, *Nb = Ns + (buf ^ 1) * kDK * 16;
        float acc[8];
        {
            const float4 n0 = *reinterpret_cast<const float4 *>(Nb + r * 16 + cc);
            const float4 n1 = *reinterpret_cast<const float4 *>(Nb + r * 16 + cc + 4);
            acc[0] = n0.x; acc[1] = n0.y; acc[2] = n0.z; acc[3] = n0.w;
            acc[4] = n1.x; acc[5] = n1.y; acc[6] = n1.z; acc[7] = n1.w;
        }
#pragma unroll 4
        for (int kk = 0; kk < kDK; kk += 4) {
            const float4 m = *reinterpret_cast<const float4 *>(Mb + r * kScanLd + kk);
            const float mv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 x0 = *reinterpret_cast<const float4 *>(Xs + (kk + i) * 16 + cc);
                const float4 x1 = *reinterpret_cast<const float4 *>(Xs + (kk + i) * 16 + cc + 4);
                acc[0] = fmaf(mv[i], x0.x, acc[0]); acc[1] = fmaf(mv[i], x0.y, acc[1]);
                acc[2] = fmaf(mv[i], x0.z, acc[2]); acc[3] = fmaf(mv[i], x0.w, acc[3]);
                acc[4] = fmaf(mv[i], x1.x, acc[4]); acc[5] = fmaf(mv[i], x1.y, acc[5]);
                acc[6] = fmaf(mv[i], x1.z, acc[6]); acc[7] = fmaf(mv[i], x1.w, acc[7]);
            }
        }
        __syncthreads();   // every read of X is done
        *reinterpret_cast<float4 *>(Xs + r * 16 + cc) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4 *>(Xs + r * 16 + cc + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        float *Y = seg + seg_slot(unit, nseg, 0, s) + (size_t)r * 128 + c0 + cc;
        *reinterpret_cast<float4 *>(Y) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4 *>(Y + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

}  // namespace

int split_segments(int units, int nchunks, int dv)
{
    if (dv != 128 || units < 1) return 1;
    const int sms = sm_count();
    if (sms <= 0 || sms / units < 5) return 1;
    int nseg = (sms / units - 1) / 2 + 2;   // pass 1 takes 1 + 2 (nseg - 2) CTAs per (b, h): one wave
    nseg = std::min(nseg, std::min(16, nchunks / 16));
    return nseg >= 3 ? nseg : 1;
}

size_t split_seg_bytes(int units, int nchunks, int dv)
{
    const int nseg = split_segments(units, nchunks, dv);
    return nseg >= 3 ? (size_t)units * 3 * nseg * kDK * 128 * 4 : 0;
}

namespace {
template <int NS>
cudaError_t launch_state(const ChunkArgs &a, const uint8_t *ws, size_t ws_bytes, cudaStream_t st)
{
    const int units = a.B * a.H, nch = (a.T + kC - 1) / kC;
    CUtensorMap tm_out;   // dv = 128: [B][T][H][dv] bf16 in 64 x 64 tiles (128-byte swizzle)
    if (NS == 2 && !make_tmap_bf16_4d(&tm_out, a.out, 128, a.H, a.T, a.B, 64, kC)) return cudaErrorInvalidValue;
    const uint32_t smem = NS == 2 ? PlanT::kSmemBytes : Plan<1>::kSmemBytes;
    cudaError_t e = NS == 2 ? cudaFuncSetAttribute(chunk_state_t_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem)
                            : cudaFuncSetAttribute(chunk_state_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
    if (e != cudaSuccess) return e;
    auto run = [&](int pass, int nseg, int cps, float *seg) {
        const unsigned grid = (unsigned)(units * seg_jobs(pass, nseg));
        if (NS == 2)
            chunk_state_t_kernel<<<grid, PlanT::kThreads, smem, st>>>(tm_out, ws, a.S0, a.S_final, a.T, a.H,
                                                                      a.status, pass, nseg, cps, seg);
        else
            chunk_state_kernel<1><<<grid, Plan<1>::kThreads, smem, st>>>(
                ws, a.S0, (__nv_bfloat16 *)a.out, a.S_final, a.T, a.H, a.status, pass, nseg, cps, seg);
        return cudaGetLastError();
    };
    const size_t base = (size_t)units * nch * split_unit_bytes(a.dv);
    const int nseg = split_segments(units, nch, a.dv);
    if (NS == 2 && nseg >= 3 && ws_bytes >= base + split_seg_bytes(units, nch, a.dv)) {
        float *seg = reinterpret_cast<float *>(const_cast<uint8_t *>(ws) + base);
        const int cps = (nch + nseg - 1) / nseg;
        if ((e = run(1, nseg, cps, seg)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem)) !=
            cudaSuccess)
            return e;
        seg_scan_kernel<<<(unsigned)(units * 8), 256, kScanSmem, st>>>(seg, nseg);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return run(2, nseg, cps, seg);
    }
    return run(0, 1, nch, nullptr);
}
}  // namespace

cudaError_t launch_chunk_state(const ChunkArgs &a, const uint8_t *ws, size_t ws_bytes, cudaStream_t st)
{
    return a.dv == 128 ? launch_state<2>(a, ws, ws_bytes, st) : launch_state<1>(a, ws, ws_bytes, st);
}

}  // namespace ldn
