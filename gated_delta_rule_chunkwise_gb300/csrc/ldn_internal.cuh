// Internal declarations shared by the CUDA translation units of libldn.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <algorithm>

#include "../../include/ldn.h"

namespace ldn {

// Device status word: kernels atomically OR (1 << LDN_ERR_*) into it when they
// abandon a bounded wait.  It is a __device__ variable of api.cu (no
// allocation); api.cu resolves its address per device and hands it to the
// launchers, and ldn_get_device_status() reads and clears it.
// State image of the chunkwise backward: per (b, h, chunk) a [128][kStateImgLd] fp16 tile (row
// i = state row i, 128 values padded to 272 bytes), the layout its shared-memory tiles use, so
// one bulk copy moves a state.
constexpr int kStateImgLd = 136;
constexpr size_t kStateImgBytes = 128 * kStateImgLd * 2;

struct ChunkArgs {
    const void *q, *k, *v;
    const float *beta, *gate, *S0;
    void *out;
    float *S_final;
    int B, T, H, dk, dv, chunk, mode, dtype;
    int *status;
    const float *erase = nullptr, *write = nullptr;   // Gated DeltaNet-2: b [B][T][H][dk], w [B][T][H][dv]
    // Pre-solved tensor-core kernels (dk = dv = 128): when set, the state entering every chunk
    // as the chunkwise backward's fp16 state image (kStateImgBytes per (b, h, chunk))
    __half *chunk_states = nullptr;
};

struct DecodeArgs {
    const void *q, *k, *v;
    const float *beta, *gate;
    float *S;
    void *out;
    int B, H, dk, dv, mode, dtype;
    int *status;
    const float *erase = nullptr, *write = nullptr;   // Gated DeltaNet-2: b [B][H][dk], w [B][H][dv]
};

// Prologue / epilogue around the chunkwise path (prologue.cu).
struct PrologueArgs {
    const void *q_in, *k_in, *v_in;
    const float *conv_q, *conv_k, *conv_v;
    const float *beta_logit, *gate_z, *gate_a, *gate_b;
    void *q, *k, *v;
    float *beta, *gate;
    int B, T, H, dk, dv, width, mode, dtype;
    float eps;
};

struct RmsNormArgs {
    const void *o, *g;
    const float *weight;
    void *y;
    int B, T, H, dv, dtype;
    float eps;
};

// Split variant: workspace bytes per (b, h, chunk) -- [Q~ ; -W] (32 KiB), [P U' ; U']
// per 64-column slice of dv (16 KiB each), K~ (16 KiB), e^{g_C} per key channel
// (512 B); layout described in include/ldn.h.
__host__ __device__ constexpr size_t split_unit_bytes(int dv) { return 32768 + (size_t)(dv / 64) * 16384 + 16384 + 512; }
constexpr size_t kSplitRvOff = 32768;
__host__ __device__ constexpr size_t split_kt_off(int dv) { return 32768 + (size_t)(dv / 64) * 16384; }
__host__ __device__ constexpr size_t split_eg_off(int dv) { return split_kt_off(dv) + 16384; }

// Launchers: return cudaSuccess or the launch error.  Arguments are validated
// by the caller (api.cu).
cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t stream);
cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t stream);
bool chunk_tc_supported(const ChunkArgs &a);
// Split variant: preparation kernel (chunk_tc.cu) then state kernel (chunk_state.cu).
// ws_bytes >= the operand images (units x chunks x split_unit_bytes); with split_seg_bytes()
// more, long sequences are cut into segments that run side by side (chunk_state.cu).
cudaError_t launch_chunk_split(const ChunkArgs &a, uint8_t *ws, size_t ws_bytes, cudaStream_t stream);
cudaError_t launch_chunk_state(const ChunkArgs &a, const uint8_t *ws, size_t ws_bytes, cudaStream_t stream);
// Segments per (b, h) of the split variant's state kernel (1: no split), and the fp32 bytes
// they need beyond the operand images (0 when there is no split).
int split_segments(int units, int nchunks, int dv);
size_t split_seg_bytes(int units, int nchunks, int dv);
// Streaming multiprocessors of the current device (0 if it cannot be read).
int sm_count();
// Pre-solved variant (chunk_tc.cu): X = [P T ; T] of every chunk into the workspace
// (presolved_workspace_bytes), then the fused kernel reading it.
size_t presolved_workspace_bytes(int B, int T, int H);
cudaError_t launch_chunk_presolved(const ChunkArgs &a, uint8_t *ws, cudaStream_t stream);
// The pre-solved variant's solve alone: X = [P T ; T] of every chunk into ws (16 KB per
// (b, h, chunk), rows 64..127 are T = (I + strict_tril(Diag(beta) (K K^T * Gamma)))^-1).
cudaError_t launch_chunk_solve(const ChunkArgs &a, uint8_t *ws, cudaStream_t stream);
// fastest tensor-core LDN_VARIANT_* by a cost model, given which workspace variants can run
int chunk_tc_pick(const ChunkArgs &a, bool split_ok, bool presolved_ok);
bool chunk_pair_supported(const ChunkArgs &a);    // the cluster-pair kernel takes these arguments
cudaError_t launch_chunk_pair(const ChunkArgs &a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
// nsteps consecutive steps in one launch (DeltaNet, Gated DeltaNet, KDA); inputs [nsteps][B][H][..].
cudaError_t launch_decode_steps(const DecodeArgs &a, int nsteps, cudaStream_t stream);

// Backward of the recurrence (csrc/backward.cu).
struct BwdArgs {
    const void *q, *k, *v;
    const float *beta, *gate, *S0;
    const void *dout;
    const float *dS_final;
    float *dq, *dk_out, *dv_out, *dbeta, *dgate, *dS0;
    float *ws;   // checkpoints, then the per-slice partial sums
    int B, T, H, dk, dv, mode, dtype;
};
// Residual Linear Attention / Residual DeltaNet forward (csrc/rla.cu).
struct RlaArgs {
    const void *q, *k, *v;
    const float *beta, *gamma, *gate, *S0, *R0;
    float clip;
    void *out;
    float *S_final, *R_final;
    int B, T, H, dk, dv, delta, dtype;
};
cudaError_t launch_rla(const RlaArgs &a, cudaStream_t stream);
// Chunk form of the same (csrc/rla_chunk.cu): bf16 inputs, dk = dv = 128, 16-byte aligned
// q, k, v, out.  Residual DeltaNet needs a workspace of rla_chunk_workspace_bytes (the
// solves for beta and gamma); Residual Linear Attention none.
bool rla_chunk_supported(const RlaArgs &a);
size_t rla_chunk_workspace_bytes(int B, int T, int H, int delta);
cudaError_t launch_rla_chunk(const RlaArgs &a, void *ws, cudaStream_t stream);
// Chunkwise backward on the tensor cores (csrc/backward_chunk.cu): DeltaNet / Gated DeltaNet,
// bf16 inputs, dk = dv = 128, 16-byte aligned q, k, v, dout.
bool bwd_chunk_supported(const BwdArgs &a);
size_t bwd_chunk_workspace_bytes(int B, int T, int H);
cudaError_t launch_backward_chunk(const BwdArgs &a, cudaStream_t stream);
size_t bwd_ckpt_floats(int B, int T, int H, int dk, int dv);
size_t bwd_workspace_bytes(int B, int T, int H, int dk, int dv, int mode);
cudaError_t launch_backward(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_prologue(const PrologueArgs &a, cudaStream_t stream);
cudaError_t launch_rmsnorm_gated(const RmsNormArgs &a, cudaStream_t stream);
int *status_word_ptr();   // address of the device status word on the current device
// Library-owned split-variant scratch of ldn_chunk_fwd_noalloc (static_scratch.cu).
// acquire() locks the current device's scratch and orders `s` after its previous
// user (LDN_OK), or returns LDN_ERR_INVALID_ARG (`s` belongs to another device)
// or LDN_ERR_UNSUPPORTED (first use on the device during a stream capture);
// release() records the end of this use on `s` and unlocks.
constexpr size_t kStaticScratchBytes = (size_t)256 << 20;
int static_scratch_acquire(cudaStream_t s, uint8_t **ptr, size_t *bytes, int *device);
cudaError_t static_scratch_release(cudaStream_t s, int device);
cudaError_t launch_copy_state(const float *S0, float *S_final, long long n, cudaStream_t stream);

// Loads of q/k/v in either element type, widened to fp32.
__device__ __forceinline__ float load_in(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_in(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void store_out(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }

}  // namespace ldn
