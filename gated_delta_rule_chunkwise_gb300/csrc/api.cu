// C ABI of libldn: argument validation, kernel-family dispatch, status word.
// The operations and their sources are documented in include/ldn.h.
#include "ldn_internal.cuh"

namespace ldn {
__device__ int g_status = 0;

__global__ void copy_state_kernel(const float *__restrict__ S0, float *__restrict__ S_final, long long n)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        S_final[i] = S0 ? S0[i] : 0.0f;
}

cudaError_t launch_copy_state(const float *S0, float *S_final, long long n, cudaStream_t stream)
{
    if (n == 0) return cudaSuccess;
    long long blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    copy_state_kernel<<<(unsigned)blocks, 256, 0, stream>>>(S0, S_final, n);
    return cudaGetLastError();
}
// Address of g_status on the current device, resolved once per device.
int *status_word_ptr()
{
    static int *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        addr[dev] = (int *)p;
    }
    return addr[dev];
}
}  // namespace ldn

using namespace ldn;

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
static bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }
static bool supported_dim(int d) { return d == 64 || d == 128; }

// Mode LDN_GDN2 takes erase and write gates in place of beta and has entry
// points of its own (g2 = true); the beta-gated entry points reject it.
static int validate_common(int mode, int dtype, int dk, int dv, bool g2 = false)
{
    if (g2 ? mode != LDN_GDN2 : (mode < LDN_DELTANET || mode > LDN_KDA)) return LDN_ERR_INVALID_ARG;
    if (dtype != LDN_F32 && dtype != LDN_BF16) return LDN_ERR_INVALID_ARG;
    if (dk < 1 || dv < 1) return LDN_ERR_INVALID_ARG;
    if (!supported_dim(dk) || !supported_dim(dv)) return LDN_ERR_UNSUPPORTED;
    return LDN_OK;
}

// Workspace bytes of the split variant (0: it does not take these sizes): the operand images
// (`base` true: all the variant needs) and, for long sequences, the sequence split's states and
// maps (chunk_state.cu).
// (Pointers are taken as aligned: a Gated DeltaNet-2 call gets stand-in gates here.)
static size_t split_workspace_bytes(int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                                    bool base = false)
{
    if (T < 1 || B < 1 || H < 1) return 0;
    alignas(16) static const float kAligned[4] = {0.f, 0.f, 0.f, 0.f};
    ChunkArgs a{};
    a.dk = dk; a.dv = dv; a.chunk = chunk; a.mode = mode; a.dtype = dtype; a.B = B; a.T = T; a.H = H;
    a.erase = a.write = kAligned;
    if (dtype != LDN_BF16 || !chunk_tc_supported(a)) return 0;
    const int nch = (T + chunk - 1) / chunk;
    return (size_t)B * H * (size_t)nch * split_unit_bytes(dv) + (base ? 0 : split_seg_bytes(B * H, nch, dv));
}

// Argument checks shared by the chunk entry points (everything but the
// workspace).  On LDN_OK, *tc says whether the tensor-core kernels take the call.
// Gated DeltaNet-2 (mode LDN_GDN2) passes its erase and write gates, beta unused.
static int check_chunk_args(const void *q, const void *k, const void *v, const float *beta, const float *gate,
                            const float *S0, const void *out, const float *S_final, int B, int T, int H, int dk,
                            int dv, int chunk, int mode, int dtype, int variant, bool *tc,
                            const float *erase = nullptr, const float *write = nullptr)
{
    *tc = false;
    const bool g2 = mode == LDN_GDN2;
    int st = validate_common(mode, dtype, dk, dv, g2 && erase && write);
    if (st != LDN_OK) return st;
    if (B < 1 || H < 1 || T < 0) return LDN_ERR_INVALID_ARG;
    if (variant < LDN_VARIANT_AUTO || variant > LDN_VARIANT_PRESOLVED) return LDN_ERR_INVALID_ARG;
    if (chunk != 64) return LDN_ERR_UNSUPPORTED;
    // Sizes: token-head count and state element count must stay well inside int64
    // and the grid limits.
    if ((long long)B * H > (1LL << 24)) return LDN_ERR_UNSUPPORTED;
    if ((long long)B * T * H * (dk > dv ? dk : dv) > (1LL << 40)) return LDN_ERR_UNSUPPORTED;
    if (T == 0) {
        if (S0 && !aligned16(S0)) return LDN_ERR_INVALID_ARG;
        if (S_final && !aligned16(S_final)) return LDN_ERR_INVALID_ARG;
        return LDN_OK;
    }
    if (!q || !k || !v || (!g2 && !beta) || !out) return LDN_ERR_INVALID_ARG;
    if (mode != LDN_DELTANET && !gate) return LDN_ERR_INVALID_ARG;
    if (g2 && (!aligned(erase, 4) || !aligned(write, 4))) return LDN_ERR_INVALID_ARG;
    // Tiles of q, k, v, out and the states move in 16-byte vectors (TMA,
    // float4); beta and gates are read as scalars.
    const void *vec_ptrs[] = {q, k, v, S0, out, S_final};
    for (const void *p : vec_ptrs)
        if (p && !aligned16(p)) return LDN_ERR_INVALID_ARG;
    if ((!g2 && !aligned(beta, 4)) || (gate && !aligned(gate, 4))) return LDN_ERR_INVALID_ARG;
    ChunkArgs a{};
    a.gate = mode == LDN_DELTANET ? nullptr : gate;
    a.erase = erase;
    a.write = write;
    a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk; a.mode = mode; a.dtype = dtype;
    *tc = dtype == LDN_BF16 && chunk_tc_supported(a);
    if ((variant == LDN_VARIANT_TENSOR || variant == LDN_VARIANT_SPLIT || variant == LDN_VARIANT_PAIR ||
         variant == LDN_VARIANT_PRESOLVED) && !*tc)
        return LDN_ERR_UNSUPPORTED;
    if (variant == LDN_VARIANT_PAIR && !chunk_pair_supported(a)) return LDN_ERR_UNSUPPORTED;
    return LDN_OK;
}

static int chunk_fwd_impl(const void *q, const void *k, const void *v, const float *beta, const float *gate,
                          const float *S0, void *out, float *S_final, int B, int T, int H, int dk, int dv,
                          int chunk, int mode, int dtype, int variant, void *ws, size_t ws_bytes, void *stream,
                          const float *erase = nullptr, const float *write = nullptr)
{
    bool tc = false;
    const int st = check_chunk_args(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype,
                                    variant, &tc, erase, write);
    if (st != LDN_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        if (!S_final) return LDN_OK;
        return launch_copy_state(S0, S_final, (long long)B * H * dk * dv, s) == cudaSuccess ? LDN_OK
                                                                                            : LDN_ERR_CUDA;
    }
    ChunkArgs a{q, k, v, beta, mode == LDN_DELTANET ? nullptr : gate, S0, out, S_final,
                B, T, H, dk, dv, chunk, mode, dtype, nullptr};
    a.erase = erase;
    a.write = write;
    const size_t need = tc ? split_workspace_bytes(B, T, H, dk, dv, chunk, mode, dtype, true) : 0;
    const bool ws_ok = ws && aligned(ws, 256) && need > 0 && ws_bytes >= need;
    const bool pre_ok = tc && ws && aligned(ws, 256) && ws_bytes >= presolved_workspace_bytes(B, T, H);
    if (variant == LDN_VARIANT_AUTO) variant = !tc ? LDN_VARIANT_SIMT : chunk_tc_pick(a, ws_ok, pre_ok);
    if (variant == LDN_VARIANT_SPLIT && !ws_ok) return LDN_ERR_INVALID_ARG;
    if (variant == LDN_VARIANT_PRESOLVED && !pre_ok) return LDN_ERR_INVALID_ARG;
    a.status = status_word_ptr();
    if (!a.status) return LDN_ERR_CUDA;
    cudaError_t err;
    if (variant == LDN_VARIANT_PRESOLVED) err = launch_chunk_presolved(a, (uint8_t *)ws, s);
    else if (variant == LDN_VARIANT_SPLIT) err = launch_chunk_split(a, (uint8_t *)ws, ws_bytes, s);
    else if (variant == LDN_VARIANT_PAIR) err = launch_chunk_pair(a, s);
    else if (variant == LDN_VARIANT_TENSOR) err = launch_chunk_tc(a, s);
    else err = launch_chunk_simt(a, s);
    return err == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

extern "C" int ldn_chunk_fwd_variant(const void *q, const void *k, const void *v, const float *beta,
                                     const float *gate, const float *S0, void *out, float *S_final,
                                     int B, int T, int H, int dk, int dv, int chunk, int mode,
                                     int dtype, int variant, void *stream)
{
    if (variant == LDN_VARIANT_SPLIT || variant == LDN_VARIANT_PRESOLVED)
        return LDN_ERR_INVALID_ARG;   // needs a workspace: ldn_chunk_fwd_ws
    return chunk_fwd_impl(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype, variant,
                          nullptr, 0, stream);
}

extern "C" int ldn_chunk_fwd_ws(const void *q, const void *k, const void *v, const float *beta,
                                const float *gate, const float *S0, void *out, float *S_final,
                                int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                                int variant, void *workspace, size_t workspace_bytes, void *stream)
{
    return chunk_fwd_impl(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype, variant,
                          workspace, workspace_bytes, stream);
}

// Split variant through the library's static scratch.  The call is cut into
// pieces whose workspace fits the scratch: groups of whole sequences when one
// sequence fits, else chunk-aligned runs of tokens of one sequence, the state
// carried from run to run through S_final (or, without one, a state slot at
// the top of the scratch).  Pieces run in stream order and reuse the scratch.
static int noalloc_impl(const void *q, const void *k, const void *v, const float *beta, const float *gate,
                        const float *S0, void *out, float *S_final, int B, int T, int H, int dk, int dv, int chunk,
                        int mode, int dtype, int variant, void *stream, const float *erase, const float *write)
{
    if (variant != LDN_VARIANT_AUTO && variant != LDN_VARIANT_SPLIT && variant != LDN_VARIANT_PRESOLVED)
        return chunk_fwd_impl(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype,
                              variant, nullptr, 0, stream, erase, write);
    bool tc = false;
    int st = check_chunk_args(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype,
                              variant, &tc, erase, write);
    if (st != LDN_OK) return st;
    if (T == 0 || !tc)   // state copy, or the SIMT kernel: no scratch
        return chunk_fwd_impl(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype,
                              LDN_VARIANT_AUTO, nullptr, 0, stream, erase, write);
    ChunkArgs whole{};
    whole.gate = mode == LDN_DELTANET ? nullptr : gate;
    whole.erase = erase;
    whole.write = write;
    whole.B = B; whole.T = T; whole.H = H; whole.dk = dk; whole.dv = dv; whole.chunk = chunk;
    whole.mode = mode; whole.dtype = dtype;
    const int requested = variant;
    if (variant == LDN_VARIANT_AUTO) {
        const int pick = chunk_tc_pick(whole, true, true);
        if (pick != LDN_VARIANT_SPLIT && pick != LDN_VARIANT_PRESOLVED)
            return chunk_fwd_impl(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype,
                                  pick, nullptr, 0, stream, erase, write);
        variant = pick;
    }

    // Plan: nb sequences per piece, or (nb == 0) runs of tpc chunks of one sequence.  The
    // workspace per (b, h, chunk) is the split variant's operand image or the pre-solved
    // variant's X.
    const size_t cap = kStaticScratchBytes;
    const size_t unit = variant == LDN_VARIANT_SPLIT ? split_unit_bytes(dv) : presolved_workspace_bytes(1, 64, 1);
    const long long nch = (T + chunk - 1) / chunk;
    const size_t per_seq = (size_t)H * nch * unit;
    const size_t state_elems = (size_t)H * dk * dv;
    int nb = 0;
    long long tpc = 0;
    size_t carry_bytes = 0;
    if (per_seq <= cap) {
        nb = (int)((size_t)B < cap / per_seq ? (size_t)B : cap / per_seq);
    } else {
        carry_bytes = S_final ? 0 : (state_elems * sizeof(float) + 255) / 256 * 256;
        if (carry_bytes < cap) tpc = (long long)((cap - carry_bytes) / ((size_t)H * unit));
        if (tpc == 0)   // one chunk of all heads exceeds the array: a kernel without workspace (AUTO)
            return requested != LDN_VARIANT_AUTO
                       ? LDN_ERR_UNSUPPORTED
                       : chunk_fwd_impl(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode,
                                        dtype, chunk_tc_pick(whole, false, false), nullptr, 0, stream, erase, write);
    }

    cudaStream_t s = (cudaStream_t)stream;
    uint8_t *scr = nullptr;
    size_t scr_bytes = 0;
    int dev = 0;
    st = static_scratch_acquire(s, &scr, &scr_bytes, &dev);
    if (st != LDN_OK) return st;
    const size_t el = dtype == LDN_BF16 ? 2 : 4;
    const size_t gate_w = mode == LDN_KDA || mode == LDN_GDN2 ? (size_t)dk : 1;
    // One piece: sequences b0 .. b0+np-1, tokens t0 .. t0+len-1 (t0 > 0 only when np == 1).
    auto piece = [&](int b0, int np, int t0, int len, const float *s0, float *sf, size_t ws_bytes) {
        const size_t tok = ((size_t)b0 * T + t0) * H;   // token-head offset of (b0, t0)
        if (variant == LDN_VARIANT_SPLIT)   // the operand images alone: no sequence split here
            ws_bytes = std::min(ws_bytes, (size_t)np * H * (size_t)((len + chunk - 1) / chunk) * unit);
        return chunk_fwd_impl((const uint8_t *)q + tok * dk * el, (const uint8_t *)k + tok * dk * el,
                              (const uint8_t *)v + tok * dv * el, beta ? beta + tok : nullptr,
                              gate ? gate + tok * gate_w : nullptr, s0, (uint8_t *)out + tok * dv * el, sf, np, len,
                              H, dk, dv, chunk, mode, dtype, variant, scr, ws_bytes, stream,
                              erase ? erase + tok * dk : nullptr, write ? write + tok * dv : nullptr);
    };
    st = LDN_OK;
    if (nb > 0) {
        for (int b0 = 0; b0 < B && st == LDN_OK; b0 += nb) {
            const int np = B - b0 < nb ? B - b0 : nb;
            st = piece(b0, np, 0, T, S0 ? S0 + (size_t)b0 * state_elems : nullptr,
                       S_final ? S_final + (size_t)b0 * state_elems : nullptr, cap);
        }
    } else {
        const long long run = tpc * chunk;
        for (int b = 0; b < B && st == LDN_OK; ++b) {
            float *carry = S_final ? S_final + (size_t)b * state_elems : (float *)(scr + cap - carry_bytes);
            for (long long t0 = 0; t0 < T && st == LDN_OK; t0 += run) {
                const int len = (int)(T - t0 < run ? T - t0 : run);
                const float *s0 = t0 == 0 ? (S0 ? S0 + (size_t)b * state_elems : nullptr) : carry;
                float *sf = t0 + len >= T ? (S_final ? S_final + (size_t)b * state_elems : nullptr) : carry;
                st = piece(b, 1, (int)t0, len, s0, sf, cap - carry_bytes);
            }
        }
    }
    const cudaError_t rel = static_scratch_release(s, dev);
    if (st == LDN_OK && rel != cudaSuccess) st = LDN_ERR_CUDA;
    return st;
}

extern "C" int ldn_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *beta,
                                     const float *gate, const float *S0, void *out, float *S_final,
                                     int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                                     int variant, void *stream)
{
    if (mode == LDN_GDN2) return LDN_ERR_INVALID_ARG;
    return noalloc_impl(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk, mode, dtype, variant, stream,
                        nullptr, nullptr);
}

extern "C" int ldn_chunk_fwd_select_ws(int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                                       size_t workspace_bytes)
{
    const int st = validate_common(mode, dtype, dk, dv, mode == LDN_GDN2);
    if (st != LDN_OK) return -st;
    if (chunk != 64) return -LDN_ERR_UNSUPPORTED;
    if (B < 1 || H < 1 || T < 0) return -LDN_ERR_INVALID_ARG;
    alignas(16) static const float kAligned[4] = {0.f, 0.f, 0.f, 0.f};   // stand-in gates (aligned)
    ChunkArgs a{};
    a.dk = dk; a.dv = dv; a.chunk = chunk; a.mode = mode; a.dtype = dtype; a.B = B; a.T = T; a.H = H;
    a.erase = a.write = kAligned;
    if (dtype != LDN_BF16 || !chunk_tc_supported(a)) return LDN_VARIANT_SIMT;
    const size_t need = split_workspace_bytes(B, T, H, dk, dv, chunk, mode, dtype, true);
    return chunk_tc_pick(a, need > 0 && workspace_bytes >= need,
                         T > 0 && workspace_bytes >= presolved_workspace_bytes(B, T, H));
}

extern "C" int ldn_chunk_fwd_split_segments(int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                                            size_t workspace_bytes)
{
    const int st = validate_common(mode, dtype, dk, dv, mode == LDN_GDN2);
    if (st != LDN_OK) return -st;
    if (chunk != 64) return -LDN_ERR_UNSUPPORTED;
    if (B < 1 || H < 1 || T < 0) return -LDN_ERR_INVALID_ARG;
    const size_t base = split_workspace_bytes(B, T, H, dk, dv, chunk, mode, dtype, true);
    if (base == 0) return 0;
    const int nch = (T + chunk - 1) / chunk, nseg = split_segments(B * H, nch, dv);
    return nseg >= 3 && workspace_bytes >= base + split_seg_bytes(B * H, nch, dv) ? nseg : 1;
}

extern "C" size_t ldn_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype)
{
    if (validate_common(mode, dtype, dk, dv) != LDN_OK || chunk != 64) return 0;
    return split_workspace_bytes(B, T, H, dk, dv, chunk, mode, dtype);
}

extern "C" int ldn_chunk_fwd(const void *q, const void *k, const void *v, const float *beta,
                             const float *gate, const float *S0, void *out, float *S_final,
                             int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                             void *stream)
{
    return ldn_chunk_fwd_variant(q, k, v, beta, gate, S0, out, S_final, B, T, H, dk, dv, chunk,
                                 mode, dtype, LDN_VARIANT_AUTO, stream);
}

extern "C" int ldn_chunk_fwd_select(int dk, int dv, int chunk, int mode, int dtype)
{
    const int st = validate_common(mode, dtype, dk, dv);
    if (st != LDN_OK) return -st;
    if (chunk != 64) return -LDN_ERR_UNSUPPORTED;
    ChunkArgs a{};
    a.dk = dk; a.dv = dv; a.chunk = chunk; a.mode = mode; a.dtype = dtype; a.B = 1; a.T = 1; a.H = 1;
    return (dtype == LDN_BF16 && chunk_tc_supported(a)) ? LDN_VARIANT_TENSOR : LDN_VARIANT_SIMT;
}

extern "C" int ldn_decode_step(const void *q, const void *k, const void *v, const float *beta,
                               const float *gate, float *S, void *out,
                               int B, int H, int dk, int dv, int mode, int dtype, void *stream)
{
    int st = validate_common(mode, dtype, dk, dv);
    if (st != LDN_OK) return st;
    if (B < 1 || H < 1) return LDN_ERR_INVALID_ARG;
    if ((long long)B * H > (1LL << 24)) return LDN_ERR_UNSUPPORTED;
    if (!q || !k || !v || !beta || !S || !out) return LDN_ERR_INVALID_ARG;
    if (mode != LDN_DELTANET && !gate) return LDN_ERR_INVALID_ARG;
    // The state moves in float4 rows; everything else is read element-wise.
    const uintptr_t el = dtype == LDN_BF16 ? 2 : 4;
    if (!aligned16(S)) return LDN_ERR_INVALID_ARG;
    const void *el_ptrs[] = {q, k, v, out};
    for (const void *p : el_ptrs)
        if (!aligned(p, el)) return LDN_ERR_INVALID_ARG;
    if (!aligned(beta, 4) || (gate && !aligned(gate, 4))) return LDN_ERR_INVALID_ARG;
    int *sw = status_word_ptr();
    if (!sw) return LDN_ERR_CUDA;
    DecodeArgs a{q, k, v, beta, mode == LDN_DELTANET ? nullptr : gate, S, out, B, H, dk, dv, mode, dtype, sw};
    return launch_decode(a, (cudaStream_t)stream) == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

extern "C" int ldn_decode_steps(const void *q, const void *k, const void *v, const float *beta,
                                const float *gate, float *S, void *out, int n_steps,
                                int B, int H, int dk, int dv, int mode, int dtype, void *stream)
{
    if (mode == LDN_GDN2) return LDN_ERR_UNSUPPORTED;   // its step is ldn_decode_step_gdn2
    int st = validate_common(mode, dtype, dk, dv);
    if (st != LDN_OK) return st;
    if (B < 1 || H < 1 || n_steps < 0) return LDN_ERR_INVALID_ARG;
    if ((long long)B * H > (1LL << 24) || (long long)n_steps * B * H * (dk > dv ? dk : dv) > (1LL << 40))
        return LDN_ERR_UNSUPPORTED;
    if (!S) return LDN_ERR_INVALID_ARG;
    if (n_steps == 0) return LDN_OK;
    if (!q || !k || !v || !beta || !out) return LDN_ERR_INVALID_ARG;
    if (mode != LDN_DELTANET && !gate) return LDN_ERR_INVALID_ARG;
    const uintptr_t el = dtype == LDN_BF16 ? 2 : 4;
    if (!aligned16(S)) return LDN_ERR_INVALID_ARG;
    const void *el_ptrs[] = {q, k, v, out};
    for (const void *p : el_ptrs)
        if (!aligned(p, el)) return LDN_ERR_INVALID_ARG;
    if (!aligned(beta, 4) || (gate && !aligned(gate, 4))) return LDN_ERR_INVALID_ARG;
    DecodeArgs a{q, k, v, beta, mode == LDN_DELTANET ? nullptr : gate, S, out, B, H, dk, dv, mode, dtype, nullptr};
    return launch_decode_steps(a, n_steps, (cudaStream_t)stream) == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

static bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

// Gated DeltaNet-2: the KDA checks with the erase gate b (shaped like k) and
// the write gate w (shaped like v) in place of beta; kernel choice and the
// split variant's scratch as in ldn_chunk_fwd_noalloc.
extern "C" int ldn_chunk_fwd_gdn2(const void *q, const void *k, const void *v, const float *erase,
                                  const float *write, const float *gate, const float *S0, void *out, float *S_final,
                                  int B, int T, int H, int dk, int dv, int chunk, int dtype, int variant,
                                  void *stream)
{
    if (T > 0 && (!erase || !write)) return LDN_ERR_INVALID_ARG;
    alignas(16) static const float kNone[4] = {0.f, 0.f, 0.f, 0.f};   // T = 0: no gate is read
    return noalloc_impl(q, k, v, nullptr, gate, S0, out, S_final, B, T, H, dk, dv, chunk, LDN_GDN2, dtype, variant,
                        stream, erase ? erase : kNone, write ? write : kNone);
}

extern "C" int ldn_decode_step_gdn2(const void *q, const void *k, const void *v, const float *erase,
                                    const float *write, const float *gate, float *S, void *out,
                                    int B, int H, int dk, int dv, int dtype, void *stream)
{
    int st = validate_common(LDN_KDA, dtype, dk, dv);
    if (st != LDN_OK) return st;
    if (B < 1 || H < 1) return LDN_ERR_INVALID_ARG;
    if ((long long)B * H > (1LL << 24)) return LDN_ERR_UNSUPPORTED;
    if (!q || !k || !v || !erase || !write || !gate || !S || !out) return LDN_ERR_INVALID_ARG;
    const uintptr_t el = dtype == LDN_BF16 ? 2 : 4;
    if (!aligned16(S)) return LDN_ERR_INVALID_ARG;
    const void *el_ptrs[] = {q, k, v, out};
    for (const void *p : el_ptrs)
        if (!aligned(p, el)) return LDN_ERR_INVALID_ARG;
    if (!aligned(erase, 4) || !aligned(write, 4) || !aligned(gate, 4)) return LDN_ERR_INVALID_ARG;
    int *sw = status_word_ptr();
    if (!sw) return LDN_ERR_CUDA;
    DecodeArgs a{q, k, v, nullptr, gate, S, out, B, H, dk, dv, LDN_GDN2, dtype, sw};
    a.erase = erase;
    a.write = write;
    return launch_decode(a, (cudaStream_t)stream) == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

extern "C" int ldn_prologue(const void *q_in, const void *k_in, const void *v_in, const float *conv_q,
                            const float *conv_k, const float *conv_v, int width, const float *beta_logit,
                            const float *gate_z, const float *gate_a, const float *gate_b, void *q, void *k,
                            void *v, float *beta, float *gate, int B, int T, int H, int dk, int dv, int mode,
                            int dtype, float eps, void *stream)
{
    const int st = validate_common(mode, dtype, dk, dv);
    if (st != LDN_OK) return st;
    if (B < 1 || H < 1 || T < 0 || !(eps >= 0.f) || eps > 1e30f) return LDN_ERR_INVALID_ARG;
    if (width < 1) return LDN_ERR_INVALID_ARG;
    if (width > 8) return LDN_ERR_UNSUPPORTED;
    if ((long long)B * T * H * (dk > dv ? dk : dv) > (1LL << 40)) return LDN_ERR_UNSUPPORTED;
    if (T == 0) return LDN_OK;
    const bool gated = mode != LDN_DELTANET;
    const void *must[] = {q_in, k_in, v_in, conv_q, conv_k, conv_v, beta_logit, q, k, v, beta};
    for (const void *p : must)
        if (!p) return LDN_ERR_INVALID_ARG;
    if (gated && (!gate_z || !gate_a || !gate_b || !gate)) return LDN_ERR_INVALID_ARG;
    const void *vec[] = {q_in, k_in, v_in, q, k, v};   // 16-byte rows
    for (const void *p : vec)
        if (!aligned16(p)) return LDN_ERR_INVALID_ARG;
    const void *f4[] = {conv_q, conv_k, conv_v, beta_logit, beta};
    for (const void *p : f4)
        if (!aligned(p, 4)) return LDN_ERR_INVALID_ARG;
    if (gated) {
        const bool kda = mode == LDN_KDA;   // per-channel gates move as float4
        for (const void *p : {(const void *)gate_z, (const void *)gate_b, (const void *)gate})
            if (!aligned(p, kda ? 16 : 4)) return LDN_ERR_INVALID_ARG;
        if (!aligned(gate_a, 4)) return LDN_ERR_INVALID_ARG;
    }
    const size_t el = dtype == LDN_BF16 ? 2 : 4, ntok = (size_t)B * T * H;
    const size_t nk = ntok * dk * el, nv = ntok * dv * el, nb = ntok * 4, ng = gated ? ntok * 4 * (mode == LDN_KDA ? dk : 1) : 0;
    const void *ins[] = {q_in, k_in, v_in, beta_logit, gated ? gate_z : nullptr};
    const size_t nins[] = {nk, nk, nv, nb, ng};
    const void *outs[] = {q, k, v, beta, gated ? gate : nullptr};
    const size_t nouts[] = {nk, nk, nv, nb, ng};
    for (int i = 0; i < 5; ++i)
        for (int j = 0; j < 5; ++j)
            if (overlaps(ins[i], nins[i], outs[j], nouts[j])) return LDN_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i)
        for (int j = i + 1; j < 5; ++j)
            if (overlaps(outs[i], nouts[i], outs[j], nouts[j])) return LDN_ERR_INVALID_ARG;
    PrologueArgs a{q_in, k_in, v_in, conv_q, conv_k, conv_v, beta_logit, gated ? gate_z : nullptr,
                   gated ? gate_a : nullptr, gated ? gate_b : nullptr, q, k, v, beta, gated ? gate : nullptr,
                   B, T, H, dk, dv, width, mode, dtype, eps};
    return launch_prologue(a, (cudaStream_t)stream) == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

extern "C" int ldn_rmsnorm_gated(const void *o, const void *g, const float *weight, void *y, int B, int T, int H,
                                 int dv, int dtype, float eps, void *stream)
{
    if (dtype != LDN_F32 && dtype != LDN_BF16) return LDN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 0 || dv < 1 || !(eps >= 0.f) || eps > 1e30f) return LDN_ERR_INVALID_ARG;
    if (!supported_dim(dv)) return LDN_ERR_UNSUPPORTED;
    if ((long long)B * T * H * dv > (1LL << 40)) return LDN_ERR_UNSUPPORTED;
    if (T == 0) return LDN_OK;
    if (!o || !g || !weight || !y) return LDN_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(g) || !aligned16(y) || !aligned(weight, 4)) return LDN_ERR_INVALID_ARG;
    const size_t n = (size_t)B * T * H * dv * (dtype == LDN_BF16 ? 2 : 4);
    if (overlaps(g, n, y, n)) return LDN_ERR_INVALID_ARG;   // y may replace o, not g
    if (o != y && overlaps(o, n, y, n)) return LDN_ERR_INVALID_ARG;
    RmsNormArgs a{o, g, weight, y, B, T, H, dv, dtype, eps};
    return launch_rmsnorm_gated(a, (cudaStream_t)stream) == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

// Backward of the DeltaNet / Gated DeltaNet / KDA recurrence (csrc/backward.cu).
static int check_bwd_sizes(int B, int T, int H, int dk, int dv, int mode, int dtype)
{
    const int st = validate_common(mode, dtype, dk, dv);
    if (st != LDN_OK) return st;
    if (B < 1 || H < 1 || T < 0) return LDN_ERR_INVALID_ARG;
    if ((long long)B * H * (dv / 32) > (1LL << 24)) return LDN_ERR_UNSUPPORTED;
    if ((long long)B * T * H * (2LL * dk + dv + 1) * (dv / 32) > (1LL << 40)) return LDN_ERR_UNSUPPORTED;
    return LDN_OK;
}

// The chunkwise tensor-core backward takes bf16 DeltaNet / Gated DeltaNet at dk = dv = 128;
// every other call runs the recurrent backward.
static bool bwd_chunkwise(int dk, int dv, int mode, int dtype)
{
    return dtype == LDN_BF16 && dk == 128 && dv == 128 && (mode == LDN_DELTANET || mode == LDN_GDN);
}

extern "C" size_t ldn_backward_workspace_size(int B, int T, int H, int dk, int dv, int mode, int dtype)
{
    if (check_bwd_sizes(B, T, H, dk, dv, mode, dtype) != LDN_OK) return 0;
    return bwd_chunkwise(dk, dv, mode, dtype) ? bwd_chunk_workspace_bytes(B, T, H)
                                              : bwd_workspace_bytes(B, T, H, dk, dv, mode);
}

extern "C" int ldn_backward(const void *q, const void *k, const void *v, const float *beta, const float *gate,
                            const float *S0, const void *dout, const float *dS_final, float *dq, float *dk_out,
                            float *dv_out, float *dbeta, float *dgate, float *dS0, int B, int T, int H, int dk,
                            int dv, int mode, int dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    int st = check_bwd_sizes(B, T, H, dk, dv, mode, dtype);
    if (st != LDN_OK) return st;
    if (!dS0 || !aligned(dS0, 4) || (S0 && !aligned(S0, 4)) || (dS_final && !aligned(dS_final, 4)))
        return LDN_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0)
        return launch_copy_state(dS_final, dS0, (long long)B * H * dk * dv, s) == cudaSuccess ? LDN_OK
                                                                                              : LDN_ERR_CUDA;
    const bool gated = mode != LDN_DELTANET;
    const void *must[] = {q, k, v, beta, dout, dq, dk_out, dv_out, dbeta};
    for (const void *p : must)
        if (!p) return LDN_ERR_INVALID_ARG;
    if (gated && (!gate || !dgate)) return LDN_ERR_INVALID_ARG;
    const uintptr_t el = dtype == LDN_BF16 ? 2 : 4;
    const void *elp[] = {q, k, v, dout};
    for (const void *p : elp)
        if (!aligned(p, el)) return LDN_ERR_INVALID_ARG;
    const void *f4[] = {beta, dq, dk_out, dv_out, dbeta};
    for (const void *p : f4)
        if (!aligned(p, 4)) return LDN_ERR_INVALID_ARG;
    if (gated && (!aligned(gate, 4) || !aligned(dgate, 4))) return LDN_ERR_INVALID_ARG;
    const bool chunked = bwd_chunkwise(dk, dv, mode, dtype);
    if (chunked) {   // tensors read as 16-byte rows and through TMA descriptors
        const void *a16p[] = {q, k, v, dout, dq, dk_out, dv_out};
        for (const void *p : a16p)
            if (!aligned16(p)) return LDN_ERR_INVALID_ARG;
    }
    const size_t need = chunked ? bwd_chunk_workspace_bytes(B, T, H) : bwd_workspace_bytes(B, T, H, dk, dv, mode);
    if (!workspace || !aligned(workspace, chunked ? 256 : 16) || workspace_bytes < need) return LDN_ERR_INVALID_ARG;
    BwdArgs a{q, k, v, beta, gated ? gate : nullptr, S0, dout, dS_final, dq, dk_out, dv_out, dbeta,
              gated ? dgate : nullptr, dS0, (float *)workspace, B, T, H, dk, dv, mode, dtype};
    if (chunked) return launch_backward_chunk(a, s) == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
    return launch_backward(a, s) == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

extern "C" size_t ldn_rla_fwd_workspace_size(int B, int T, int H, int dk, int dv, int delta, int dtype)
{
    if (validate_common(LDN_GDN, dtype, dk, dv) != LDN_OK || B < 1 || H < 1 || T < 1 || (delta != 0 && delta != 1))
        return 0;
    if (dtype != LDN_BF16 || dk != 128 || dv != 128) return 0;   // the chunk form's shapes
    return rla_chunk_workspace_bytes(B, T, H, delta);
}

extern "C" int ldn_rla_fwd(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                           const float *gate, float clip, const float *S0, const float *R0, void *out,
                           float *S_final, float *R_final, int B, int T, int H, int dk, int dv, int delta,
                           int dtype, void *stream)
{
    return ldn_rla_fwd_ws(q, k, v, beta, gamma, gate, clip, S0, R0, out, S_final, R_final, B, T, H, dk, dv, delta,
                          dtype, nullptr, 0, stream);
}

extern "C" int ldn_rla_fwd_ws(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                              const float *gate, float clip, const float *S0, const float *R0, void *out,
                              float *S_final, float *R_final, int B, int T, int H, int dk, int dv, int delta,
                              int dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    const int st = validate_common(LDN_GDN, dtype, dk, dv);
    if (st != LDN_OK) return st;
    if (B < 1 || H < 1 || T < 0 || (delta != 0 && delta != 1) || !(clip > 0.f)) return LDN_ERR_INVALID_ARG;
    if ((long long)B * H > (1LL << 24)) return LDN_ERR_UNSUPPORTED;
    if ((long long)B * T * H * (dk > dv ? dk : dv) > (1LL << 40)) return LDN_ERR_UNSUPPORTED;
    const void *states[] = {S0, R0, S_final, R_final};
    for (const void *p : states)
        if (p && !aligned16(p)) return LDN_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const long long ns = (long long)B * H * dk * dv;
    if (T == 0) {
        if (S_final && launch_copy_state(S0, S_final, ns, s) != cudaSuccess) return LDN_ERR_CUDA;
        if (R_final && launch_copy_state(R0, R_final, ns, s) != cudaSuccess) return LDN_ERR_CUDA;
        return LDN_OK;
    }
    const void *must[] = {q, k, v, beta, gamma, gate, out};
    for (const void *p : must)
        if (!p) return LDN_ERR_INVALID_ARG;
    const void *vec[] = {q, k, v, out};
    for (const void *p : vec)
        if (!aligned16(p)) return LDN_ERR_INVALID_ARG;
    if (!aligned(beta, 4) || !aligned(gamma, 4) || !aligned(gate, 4)) return LDN_ERR_INVALID_ARG;
    RlaArgs a{q, k, v, beta, gamma, gate, S0, R0, clip, out, S_final, R_final, B, T, H, dk, dv, delta, dtype};
    if (workspace && !aligned(workspace, 256)) return LDN_ERR_INVALID_ARG;
    // chunk form: bf16, dk = dv = 128; Residual DeltaNet also needs the workspace for its solves
    if (rla_chunk_supported(a)) {
        const size_t need = rla_chunk_workspace_bytes(B, T, H, delta);
        if (need == 0 || (workspace && workspace_bytes >= need))
            return launch_rla_chunk(a, workspace, s) == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
    }
    return launch_rla(a, s) == cudaSuccess ? LDN_OK : LDN_ERR_CUDA;
}

extern "C" int ldn_get_device_status(void *stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LDN_ERR_CUDA;
    int h = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_status, sizeof(int)) != cudaSuccess) return LDN_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return LDN_ERR_CUDA;
    if (h & (1 << LDN_ERR_TIMEOUT)) return LDN_ERR_TIMEOUT;
    return h ? LDN_ERR_CUDA : LDN_OK;
}

extern "C" const char *ldn_status_string(int status)
{
    switch (status) {
    case LDN_OK: return "ok";
    case LDN_ERR_INVALID_ARG: return "invalid argument (NULL or misaligned pointer, bad enum or size)";
    case LDN_ERR_UNSUPPORTED: return "unsupported configuration (dk/dv not in {64,128}, chunk != 64, or variant)";
    case LDN_ERR_CUDA: return "CUDA runtime or launch error";
    case LDN_ERR_TIMEOUT: return "a kernel abandoned a bounded wait; outputs are incomplete";
    default: return "unknown status";
    }
}

extern "C" int ldn_version(void) { return LDN_VERSION; }
