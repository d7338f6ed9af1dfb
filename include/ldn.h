/*
 * ldn.h -- C ABI of the GB300 (sm_103a) delta-rule linear-attention library.
 *
 * Operations (math orientation: the memory S is d_v x d_k, column vectors):
 *
 *   DeltaNet   S_t = S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   Gated DN   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   KDA        S_t = S_{t-1} Diag(a_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   output     o_t = S_t q_t            (the query reads the UPDATED memory)
 *
 * as defined in "Linear Attention Architectures: Mechanisms, Trade-offs, and
 * Cross-Layer Routing" (reading notes), Sec. 2.1 Eq. 8, Sec. 2.3 Eqs. 9-10/14,
 * Sec. 2.4 Eqs. 15-17 (decay before the error), Sec. 2.5 Eqs. 18-20 (Diag(a)
 * on the key side), and in "State reduction by key/query channel pruning"
 * (reading notes), Sec. 2.1 Eqs. 1-2.  The decode step is the same rule for one
 * token, written in the prediction-correction form of the Residual Linear
 * Attention notes, Sec. 1.2.
 *
 * Entry points, in the order below:
 *   ldn_chunk_fwd, _variant, _select, _ws, _workspace_size, _select_ws, _split_segments, _noalloc
 *       the chunkwise forward and its kernel families;
 *   ldn_prologue, ldn_rmsnorm_gated     the steps on either side of it;
 *   ldn_decode_step, ldn_decode_steps                     one recurrent token;
 *   ldn_chunk_fwd_gdn2, ldn_decode_step_gdn2
 *       Gated DeltaNet-2 (separate erase and write gates, Sec. 2.6);
 *   ldn_backward, ldn_backward_workspace_size
 *       gradients of the forward;
 *   ldn_rla_fwd, ldn_rla_fwd_ws, ldn_rla_fwd_workspace_size
 *       Residual Linear Attention / Residual DeltaNet (the Residual Linear
 *       Attention notes, Sec. 2.2-2.4);
 *   ldn_get_device_status, ldn_status_string, ldn_version.
 *
 * Conventions shared by every entry point
 *   - Pointers q, k, v, beta, gate, S0, S, out, S_final are DEVICE pointers to
 *     contiguous, row-major arrays.  Alignment: ldn_chunk_fwd needs q, k, v,
 *     out, S0 and S_final 16-byte aligned (and the workspace of ldn_chunk_fwd_ws
 *     256-byte aligned); ldn_decode_step needs S 16-byte
 *     aligned and q, k, v, out aligned to their element size; beta and gate
 *     are 4-byte aligned everywhere.  The caller owns every buffer (and the
 *     workspace of the split variant); the library allocates no device memory
 *     per call (ldn_chunk_fwd_noalloc uses one static library-owned array).
 *   - Gates are natural-log decays: alpha_t = exp(gate), a_t = exp(gate[c]).
 *     A positive log-gate is accepted (it is not clamped); beta is not clamped.
 *   - q is not scaled and q, k are not normalised by the library (scale = 1).
 *   - The state is stored in memory orientation H = S^T, fp32, [B][H][dk][dv]
 *     ("K x V"), i.e. element (c, i) of head (b, h) is S[i][c].
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous.  Argument errors are detected and returned
 *     synchronously before anything is enqueued.  A launch failure returns
 *     LDN_ERR_CUDA.  Device-side faults that a kernel detects itself (a wait
 *     that ran out of its iteration limit) are recorded in a device status
 *     word and read with ldn_get_device_status().
 *   - Not thread-safe across concurrent calls that share an output buffer;
 *     otherwise re-entrant.
 */
#ifndef LDN_H
#define LDN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LDN_VERSION 7

/* LDN_GDN2 (Gated DeltaNet-2) is taken only by the *_gdn2 entry points, which
 * carry its two gates; every beta-gated entry point rejects it. */
typedef enum { LDN_DELTANET = 0, LDN_GDN = 1, LDN_KDA = 2, LDN_GDN2 = 3 } ldn_mode;

/* Element type of q, k, v and out.  beta, gate and every state are fp32. */
typedef enum { LDN_F32 = 0, LDN_BF16 = 1 } ldn_dtype;

typedef enum {
    LDN_OK = 0,
    LDN_ERR_INVALID_ARG = 1, /* NULL / misaligned pointer, bad enum, negative size */
    LDN_ERR_UNSUPPORTED = 2, /* valid but not implemented: dk/dv, chunk, variant  */
    LDN_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed              */
    LDN_ERR_TIMEOUT = 4      /* a kernel gave up on a bounded wait (device word)  */
} ldn_status;

/* Kernel family for ldn_chunk_fwd_variant. */
typedef enum {
    LDN_VARIANT_AUTO = 0,   /* bf16 -> tensor-core kernel, fp32 -> fp32 SIMT kernel */
    LDN_VARIANT_SIMT = 1,   /* fp32 CUDA-core kernel, either dtype                 */
    LDN_VARIANT_TENSOR = 2, /* tcgen05 / TMEM kernel, bf16 only                     */
    LDN_VARIANT_SPLIT = 3,  /* tcgen05, two kernels through a workspace (see below) */
    LDN_VARIANT_PAIR = 4,   /* tcgen05, two CTAs per (b, h) sharing the preparation */
    LDN_VARIANT_PRESOLVED = 5 /* tcgen05, every chunk's UT/WY solve first, through a workspace */
} ldn_variant;

/*
 * ldn_chunk_fwd -- chunkwise-parallel forward over a whole sequence.
 *
 * Computes, for every (b, h), the outputs o_t of the recurrence above for
 * t = 1..T starting from S0, and the final state S_T.  The sequence is cut
 * into chunks of `chunk` tokens; inside a chunk the recurrence is solved in
 * closed form (the UT/WY transform: a unit-lower-triangular solve with
 * (I + strict_tril(Diag(beta) K^ K~^T))), chunk outputs are formed from the
 * incoming state plus the masked, decay-weighted intra-chunk interactions,
 * and only the chunk-to-chunk state update is sequential.  The result equals
 * the token recurrence up to floating-point rounding.
 *
 *   q, k     [B][T][H][dk]  dtype        v, out [B][T][H][dv] dtype
 *   beta     [B][T][H]      fp32
 *   gate     mode GDN: [B][T][H] fp32; mode KDA: [B][T][H][dk] fp32;
 *            mode DELTANET: ignored, may be NULL
 *   S0       [B][H][dk][dv] fp32, or NULL for a zero initial state
 *   S_final  [B][H][dk][dv] fp32, or NULL to skip writing it
 *            (S_final may alias S0: every block reads its slice of S0 before
 *            it writes the same slice of S_final)
 *   B, H >= 1; T >= 0 (T = 0 only copies S0, or zeros, to S_final);
 *   dk, dv in {64, 128}; chunk == 64; mode in ldn_mode; dtype in ldn_dtype.
 * Returns LDN_OK or an error code; out and S_final are written asynchronously.
 */
int ldn_chunk_fwd(const void *q, const void *k, const void *v, const float *beta,
                  const float *gate, const float *S0, void *out, float *S_final,
                  int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                  void *stream);

/* Same as ldn_chunk_fwd with an explicit kernel family (ldn_variant).
 * The tensor-core kernel takes bf16 inputs with dk = 128, dv a multiple of 64,
 * chunk = 64, any mode; for KDA it also needs a 16-byte aligned gate tensor.
 * LDN_VARIANT_TENSOR outside these returns LDN_ERR_UNSUPPORTED.
 * LDN_VARIANT_PAIR is the same computation for DeltaNet and Gated DeltaNet with
 * dv = 128: the two 64-column halves of dv of each (b, h) run as a cluster of
 * two thread blocks that split the state-independent part of every chunk
 * between them (each prepares every other chunk and hands its operands to the
 * other through distributed shared memory); its results are bit-identical to
 * LDN_VARIANT_TENSOR.  Outside those sizes it returns LDN_ERR_UNSUPPORTED.
 * LDN_VARIANT_AUTO takes the tensor-core kernel (fused or pair, by a cost model
 * in the same units as ldn_chunk_fwd_ws's) whenever one supports the call. */
int ldn_chunk_fwd_variant(const void *q, const void *k, const void *v, const float *beta,
                          const float *gate, const float *S0, void *out, float *S_final,
                          int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                          int variant, void *stream);

/* Which kernel family LDN_VARIANT_AUTO runs for these sizes (for KDA, given a
 * 16-byte aligned gate tensor): returns LDN_VARIANT_SIMT or LDN_VARIANT_TENSOR
 * (the tensor-core family: fused or pair kernel), or -LDN_ERR_* for arguments
 * that ldn_chunk_fwd would reject.  Pure host function: touches no device. */
int ldn_chunk_fwd_select(int dk, int dv, int chunk, int mode, int dtype);

/*
 * The split variant runs the chunkwise forward as two kernels: the first forms,
 * for every chunk in parallel, everything that does not depend on the state
 * (the UT/WY transform and the intra-chunk products) and writes it to a
 * device workspace; the second runs the chunk-to-chunk state recurrence from
 * it.  It takes the same inputs as the tensor-core variant and returns the
 * same results (equal up to floating-point rounding to the fused kernel).
 *
 * Workspace contents, per (b, h, chunk), in this order (all 16-byte aligned):
 *   [Q~ ; -W] fp16, 128 x dk in the swizzled K-major layout of the state
 *   step's MMA operand (32 KiB); [P U' ; U'] fp16 per 64-column slice of dv
 *   (16 KiB each; for dv = 128 its transpose, two swizzled 128 x 64 blocks
 *   (P U')^T and U'^T with one row per dv column); K~ = K Diag-scaled by
 *   e^{g_C - g} fp16 (16 KiB); e^{g_C} per key channel fp32 (512 B).
 *
 * Sequence split: when few (b, h) are long (dv = 128, at least 48 chunks each,
 * and B*H at most a fifth of the SM count), the state recurrence of each (b, h)
 * is cut into nseg = 3 .. 16 segments that run side by side: every segment's
 * affine map H_out = M H_in + N (M dk x dk, N dk x dv, fp32) is formed from the
 * operand images, a scan gives every segment its incoming state, and the
 * segments then run again from those states with their outputs.  This takes
 * B*H*3*nseg*dk*dv*4 more bytes after the operand images (segment states and
 * maps, fp32); with only the operand images the recurrence runs unsplit.  The
 * two forms agree up to fp32 rounding of the maps.
 *
 * ldn_chunk_fwd_workspace_size: bytes of workspace the split variant needs for
 * these sizes (the operand images, plus the sequence split's states and maps
 * where it applies), or 0 when it does not take them.  Host function; whether
 * the sequence split applies depends on the SM count of the current device
 * (none when no device can be read).
 */
size_t ldn_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype);

/*
 * ldn_chunk_fwd_ws -- ldn_chunk_fwd with an explicit kernel family and a
 * caller-owned device workspace (256-byte aligned, at least
 * ldn_chunk_fwd_workspace_size bytes; its contents on entry do not matter and
 * on return are unspecified).  LDN_VARIANT_SPLIT without a large enough
 * workspace returns LDN_ERR_INVALID_ARG; LDN_VARIANT_AUTO takes the split
 * variant when it supports the call, the workspace suffices and a cost model of
 * the tensor-core variants (CTA waves x chunks x measured per-chunk times)
 * expects it to be fastest -- typically when B*H*dv/64 leaves SMs idle or needs
 * several waves -- and otherwise behaves as ldn_chunk_fwd_variant(...,
 * LDN_VARIANT_AUTO, ...).  Calls on different streams need different workspaces.
 */
int ldn_chunk_fwd_ws(const void *q, const void *k, const void *v, const float *beta,
                     const float *gate, const float *S0, void *out, float *S_final,
                     int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                     int variant, void *workspace, size_t workspace_bytes, void *stream);

/* Which kernel family ldn_chunk_fwd_ws(..., LDN_VARIANT_AUTO, ...) runs for these
 * sizes and a workspace of workspace_bytes (pointers assumed aligned; mode
 * LDN_GDN2 answers for ldn_chunk_fwd_gdn2, whose split variant has the
 * library's array, given as workspace_bytes = SIZE_MAX): returns
 * LDN_VARIANT_SIMT, LDN_VARIANT_TENSOR, LDN_VARIANT_PAIR or LDN_VARIANT_SPLIT, or -LDN_ERR_* for
 * arguments that would be rejected.  Host function; it reads the SM count of
 * the current device. */
int ldn_chunk_fwd_select_ws(int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                            size_t workspace_bytes);

/* Segments per (b, h) into which ldn_chunk_fwd_ws's split variant cuts the state
 * recurrence for these sizes and a workspace of workspace_bytes (the sequence
 * split above): nseg >= 3, or 1 when it runs unsplit (the variant then makes
 * two launches; split, four: the preparation, the segments' maps, the scan and
 * the segments' outputs).  -LDN_ERR_* for arguments ldn_chunk_fwd_ws would
 * reject, 0 when the split variant does not take these sizes.  Host function;
 * it reads the SM count of the current device. */
int ldn_chunk_fwd_split_segments(int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                                 size_t workspace_bytes);

/*
 * ldn_chunk_fwd_noalloc -- ldn_chunk_fwd_ws without a caller workspace.
 * The pages have no counterpart to this entry: it is a convenience of this
 * library for callers that cannot provide device memory.
 *
 * The split variant runs through a library-owned device array of 256 MiB per
 * device (a static __device__ array); no device memory is allocated per call.
 * The array is backed with device memory when the module holding it loads:
 * under lazy module loading (the CUDA default) at the first call on a device
 * that uses it, under CUDA_MODULE_LOADING=EAGER when the library loads, so that
 * every device the process uses then holds the 256 MiB.  ldn_chunk_fwd_gdn2's
 * split variant runs through the same array.  A call whose workspace does not
 * fit is cut into pieces that do: groups of whole sequences, or, when one
 * sequence alone needs more, runs of whole chunks of one sequence with the
 * fp32 state carried between runs in S_final (or in a slot of the array when
 * S_final is NULL).  The pieces are enqueued on `stream` one after another;
 * the result is bit-identical to that of ldn_chunk_fwd_ws with the split
 * variant and a caller workspace of the operand images alone (the same kernels
 * on the same operands; the state passes between pieces in fp32, as between
 * chunks).  The sequence split is not used here.
 *
 * The first call on a device resolves the array's address and creates an
 * event; it must not be made while `stream` is being captured into a CUDA
 * graph: such a call returns LDN_ERR_UNSUPPORTED and enqueues nothing.
 * `stream` must belong to the current device; outside a stream capture a
 * stream of another device returns LDN_ERR_INVALID_ARG.
 *
 * Arguments, layouts, alignment and error behaviour are those of
 * ldn_chunk_fwd_variant, with LDN_VARIANT_SPLIT also accepted.
 * LDN_VARIANT_AUTO runs the split variant where ldn_chunk_fwd_ws with an
 * unlimited workspace would, otherwise the fused tensor-core or the SIMT
 * kernel; LDN_VARIANT_SPLIT returns LDN_ERR_UNSUPPORTED when the call cannot
 * be cut to fit (H so large that one chunk of all heads exceeds the array).
 * LDN_VARIANT_SIMT, LDN_VARIANT_TENSOR and LDN_VARIANT_PAIR touch no scratch.
 *
 * Calls share the array: calls on different streams are ordered on the
 * device by an event the library records after each call (a host lock covers
 * the enqueue).  During stream capture that event is not used, so replays of
 * a captured graph must be ordered by the caller with other users of the
 * array.  The host lock makes the call thread-safe.
 */
int ldn_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *beta,
                          const float *gate, const float *S0, void *out, float *S_final,
                          int B, int T, int H, int dk, int dv, int chunk, int mode, int dtype,
                          int variant, void *stream);

/*
 * ldn_prologue -- the input steps before the chunkwise forward (the model-zoo
 * page's DeltaNet, KDA and Gated DeltaNet entries; the Residual Linear
 * Attention notes, Sec. 3.2-3.4 and Fig. 1; the backend notes name
 * causal_conv1d with SiLU):
 *   q = l2norm(silu(conv_q * q_in)),  k = l2norm(silu(conv_k * k_in)),
 *   v = silu(conv_v * v_in),  beta = sigmoid(beta_logit),
 *   gate = -gate_a[h] * softplus(gate_z + gate_b)          (log alpha, Mamba2 style)
 * "conv *" is a depthwise causal convolution along t of width `width` (1..8):
 * out[b,t,h,c] = sum_i w[h*d + c][width-1-i] * x[b,t-i,h,c], zero before t = 0
 * (no state carried in from an earlier call).  l2norm divides each (b,t,h) row
 * by sqrt(sum of squares + eps).  Arithmetic in fp32; outputs in `dtype`.
 *   q_in, k_in, q, k [B][T][H][dk] and v_in, v [B][T][H][dv] of `dtype`
 *   conv_q, conv_k [H*dk][width], conv_v [H*dv][width] fp32
 *   beta_logit, beta [B][T][H] fp32
 *   mode GDN: gate_z, gate [B][T][H]; gate_a, gate_b [H]
 *   mode KDA: gate_z, gate [B][T][H][dk]; gate_a [H]; gate_b [H][dk]
 *   mode DELTANET: gate_z, gate_a, gate_b and gate are ignored (may be NULL)
 * The outputs are the inputs ldn_chunk_fwd takes.  They must not overlap any
 * input or each other (LDN_ERR_INVALID_ARG).  Alignment: q/k/v in and out
 * 16-byte; KDA gate_z, gate_b and gate 16-byte; the rest 4-byte.  dk, dv in
 * {64, 128}; width > 8 returns LDN_ERR_UNSUPPORTED; eps >= 0.  Asynchronous on
 * `stream`; two kernel launches (three when dk != dv).
 */
int ldn_prologue(const void *q_in, const void *k_in, const void *v_in, const float *conv_q, const float *conv_k,
                 const float *conv_v, int width, const float *beta_logit, const float *gate_z, const float *gate_a,
                 const float *gate_b, void *q, void *k, void *v, float *beta, float *gate, int B, int T, int H,
                 int dk, int dv, int mode, int dtype, float eps, void *stream);

/*
 * ldn_rmsnorm_gated -- the output epilogue (the model-zoo page's Gated DeltaNet
 * entry: the output goes through RMSNorm, a gain and a SiLU gate; the backend
 * notes name rms_norm_gated):
 *   y = o / sqrt(mean_c o_c^2 + eps) * weight * silu(g)
 * per (b,t,h) row of dv values, fp32 arithmetic.
 *   o, g, y [B][T][H][dv] of `dtype` (16-byte aligned); weight [dv] fp32 (the
 *   gain, shared by the heads).  y may be o (in place) but must not overlap g.
 * dv in {64, 128}; eps >= 0.  Asynchronous on `stream`; one kernel launch.
 */
int ldn_rmsnorm_gated(const void *o, const void *g, const float *weight, void *y, int B, int T, int H, int dv,
                      int dtype, float eps, void *stream);

/*
 * ldn_decode_step -- one recurrent step for every (b, h), state updated in place.
 *
 * For one token per sequence it forms the decayed state S' = alpha S (GDN),
 * S Diag(a) (KDA) or S (DeltaNet), the key prediction p = S' k and the query
 * read s = S' q in one pass over the state, then r = beta (v - p),
 * o = s + r (k^T q) (the prediction-correction form) and writes
 * S <- S' + r k^T back.
 *
 *   q, k  [B][H][dk] dtype      v, out [B][H][dv] dtype
 *   beta  [B][H] fp32           gate   GDN [B][H], KDA [B][H][dk] fp32, DN ignored
 *   S     [B][H][dk][dv] fp32, read and overwritten in place
 *   B, H >= 1; dk, dv in {64, 128}.
 */
int ldn_decode_step(const void *q, const void *k, const void *v, const float *beta,
                    const float *gate, float *S, void *out,
                    int B, int H, int dk, int dv, int mode, int dtype, void *stream);

/*
 * ldn_decode_steps -- n_steps consecutive ldn_decode_step calls on the same
 * sequences in one launch (DeltaNet, Gated DeltaNet, KDA), for inputs known in
 * advance (several tokens of one sequence taken in recurrent form).  Each step is
 * the arithmetic of ldn_decode_step; the state slices stay on chip between the
 * steps, so S is read once and written once per call.
 *   q, k  [n_steps][B][H][dk] dtype     v, out [n_steps][B][H][dv] dtype
 *   beta  [n_steps][B][H] fp32          gate   GDN [n_steps][B][H], KDA
 *                                              [n_steps][B][H][dk] fp32, DN ignored
 *   S     [B][H][dk][dv] fp32, read and overwritten in place (16-byte aligned)
 *   n_steps >= 0 (0: nothing to do); B, H >= 1; dk, dv in {64, 128}.
 * LDN_ERR_UNSUPPORTED for Gated DeltaNet-2 (its step is ldn_decode_step_gdn2).
 */
int ldn_decode_steps(const void *q, const void *k, const void *v, const float *beta, const float *gate, float *S,
                     void *out, int n_steps, int B, int H, int dk, int dv, int mode, int dtype, void *stream);

/*
 * Gated DeltaNet-2 (linear-attention notes, Sec. 2.6, Eqs. 21-24): the erase
 * and the write of the delta rule get gates of their own in place of the one
 * beta, both channel-wise, on top of the KDA per-key-channel decay:
 *   S_t = S_{t-1} Diag(a_t) (I - e_t k_t^T) + z_t k_t^T,   e_t = b_t * k_t,
 *   z_t = w_t * v_t (element-wise),   o_t = S_t q_t.
 * The prediction is taken along e_t, the write goes along k_t.  With
 * b_t = beta_t 1 and w_t = beta_t 1 it is KDA.  Gate values are used as given
 * (the library applies no sigmoid to them).
 *
 * ldn_chunk_fwd_gdn2 -- chunkwise forward of that recurrence over a whole
 * sequence: the chunk form of ldn_chunk_fwd with e_t in place of beta_t k_t on
 * the prediction side (the rows of A and W) and z_t in place of beta_t v_t.
 *   q, k     [B][T][H][dk] dtype      v, out [B][T][H][dv] dtype
 *   erase    [B][T][H][dk] fp32       write  [B][T][H][dv] fp32
 *   gate     [B][T][H][dk] fp32 (log a_t)
 *   S0, S_final, B, T, H, dk, dv, chunk, dtype, T = 0 and errors as for
 *   ldn_chunk_fwd.  Alignment: q, k, v, out, S0, S_final 16-byte; erase,
 *   write, gate 4-byte.
 * `variant` and the kernel families are those of ldn_chunk_fwd_noalloc (the
 * split variant through the same library-owned array, with the same rules on
 * the first call during a stream capture and on the stream's device): the tensor-core
 * kernels take bf16 inputs with dk = 128, dv a multiple of 64 and erase, write
 * and gate 16-byte aligned (LDN_VARIANT_PAIR is not offered: it returns
 * LDN_ERR_UNSUPPORTED); LDN_VARIANT_SIMT runs the fp32 CUDA-core kernel for
 * either dtype; LDN_VARIANT_AUTO picks as for KDA.
 */
int ldn_chunk_fwd_gdn2(const void *q, const void *k, const void *v, const float *erase, const float *write,
                       const float *gate, const float *S0, void *out, float *S_final, int B, int T, int H,
                       int dk, int dv, int chunk, int dtype, int variant, void *stream);

/*
 * ldn_decode_step_gdn2 -- one Gated DeltaNet-2 step for every (b, h), state
 * updated in place: S' = S Diag(a), p = S' e, s = S' q, r = z - p,
 * o = s + r (k^T q), S <- S' + r k^T.
 *   q, k, erase, gate [B][H][dk]      v, out, write [B][H][dv]
 *   (q, k, v, out of dtype; erase, write, gate fp32 4-byte aligned)
 *   S [B][H][dk][dv] fp32 16-byte aligned; B, H >= 1; dk, dv in {64, 128}.
 */
int ldn_decode_step_gdn2(const void *q, const void *k, const void *v, const float *erase, const float *write,
                         const float *gate, float *S, void *out, int B, int H, int dk, int dv, int dtype,
                         void *stream);

/*
 * ldn_backward -- gradients of the forward recurrence (modes DeltaNet, GDN,
 * KDA) for the loss L = sum_t <dout_t, o_t> + <dS_final, S_T>, with respect to
 * q, k, v, beta, the log-decay gates and the initial state.  The pages give the
 * rules per token (linear-attention notes, Sec. 2.3-2.5) and a first-order
 * backward keeping the state history (the benchmark's method sources, KDA).
 * Two forms, both equal to the exact gradient up to rounding:
 *   * chunkwise on the tensor cores, for bf16 DeltaNet and Gated DeltaNet at
 *     dk = dv = 128: a forward pass that keeps the state entering every chunk of
 *     64 tokens, the chain of state gradients from chunk to chunk in reverse,
 *     then every chunk's gradients at once by dense products (fp16 operands,
 *     fp32 accumulation; the chunk form of the derivative is derived in
 *     csrc/backward_chunk.cu).  Every log-decay must be <= 0 for its operands
 *     to stay in fp16 range.  Four launches;
 *   * otherwise the per-token rules stepped back in reverse token order, in fp32,
 *     from copies of every eighth state taken by a forward sweep.  Three launches.
 *
 *   q, k, v, beta, gate, S0, B, T, H, dk, dv, mode, dtype as ldn_chunk_fwd
 *   (mode LDN_GDN2 is not taken: LDN_ERR_INVALID_ARG)
 *   dout      [B][T][H][dv] dtype      dS_final [B][H][dk][dv] fp32 or NULL (zero)
 * Outputs, all fp32 and all overwritten:
 *   dq, dk    [B][T][H][dk]            dv    [B][T][H][dv]      dbeta [B][T][H]
 *   dgate     the gate's shape (mode DELTANET: ignored, may be NULL)
 *   dS0       [B][H][dk][dv] (the gradient at S0, or at the zero state when S0 is NULL)
 *   workspace device memory, at least ldn_backward_workspace_size(B, T, H, dk,
 *             dv, mode, dtype) bytes, 256-byte aligned for the chunkwise form
 *             (the forward's per-chunk states and solve, the state gradients)
 *             and 16-byte aligned otherwise (state copies, then per-32-column
 *             partial sums of the dk-side gradients); contents on entry do not
 *             matter.
 * Alignment: q, k, v, dout to their element size and every fp32 array 4-byte;
 * the chunkwise form also wants q, k, v, dout, dq, dk, dv 16-byte aligned
 * (else LDN_ERR_INVALID_ARG).  T = 0 writes dS0 = dS_final (or zeros) and
 * nothing else.  Asynchronous on `stream`.
 */
int ldn_backward(const void *q, const void *k, const void *v, const float *beta, const float *gate,
                 const float *S0, const void *dout, const float *dS_final, float *dq, float *dk, float *dv,
                 float *dbeta, float *dgate, float *dS0, int B, int T, int H, int dk_dim, int dv_dim, int mode,
                 int dtype, void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace ldn_backward needs for these sizes and dtype, or 0 for
 * arguments it rejects.  Pure host function. */
size_t ldn_backward_workspace_size(int B, int T, int H, int dk, int dv, int mode, int dtype);

/*
 * ldn_rla_fwd -- Residual Linear Attention (delta = 0) or Residual DeltaNet
 * (delta = 1), forward ("Residual Linear Attention" reading notes, Sec. 2.2
 * boxed form, Sec. 2.4):
 *   r_t = Clip_[-c, c](v_t - S_{t-1} k_t)     (the previous base state, before
 *                                             its decay and write)
 *   RLA: R_t = alpha_t R_{t-1} + gamma_t r_t k_t^T,  S_t = alpha_t S_{t-1} + beta_t v_t k_t^T
 *   RDN: R_t = alpha_t R_{t-1}(I - gamma_t k_t k_t^T) + gamma_t r_t k_t^T,
 *        S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   o_t = alpha_t S_{t-1} q_t + gamma_t R_t q_t      (the UPDATED residual state)
 * Two forms.  Chunk form (bf16, dk = dv = 128; for Residual DeltaNet only with a
 * workspace, see ldn_rla_fwd_ws): the notes' two-stage computation (Sec. 2.6) in
 * chunks of 64 tokens, both states carried chunk to chunk in fp32 and every
 * product on the tensor cores (fp16 operands, fp32 accumulation); Residual
 * DeltaNet's two UT solves (for beta and for gamma) run first.  Recurrent form
 * (every other case): both states step together, token by token, in fp32.
 *   q, k [B][T][H][dk], v, out [B][T][H][dv] of dtype (16-byte aligned)
 *   beta, gamma, gate (log alpha) [B][T][H] fp32 (4-byte aligned)
 *   clip c > 0 (INFINITY: no clip)
 *   S0, R0 [B][H][dk][dv] fp32 or NULL (zeros); S_final, R_final the same
 *   shape or NULL (not written); all 16-byte aligned
 *   dk, dv in {64, 128}; T = 0 copies the initial states to the final ones.
 */
int ldn_rla_fwd(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                const float *gate, float clip, const float *S0, const float *R0, void *out, float *S_final,
                float *R_final, int B, int T, int H, int dk, int dv, int delta, int dtype, void *stream);

/* ldn_rla_fwd with a caller-owned DEVICE workspace (256-byte aligned, or NULL):
 * Residual DeltaNet takes the chunk form when workspace_bytes is at least
 * ldn_rla_fwd_workspace_size(...) (its solves, 32 KiB per (b, h, chunk)), the
 * recurrent form otherwise; everything else as ldn_rla_fwd.  The workspace is
 * written, not read, and must not be used by other work until the call's kernels
 * have finished on `stream`. */
int ldn_rla_fwd_ws(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                   const float *gate, float clip, const float *S0, const float *R0, void *out, float *S_final,
                   float *R_final, int B, int T, int H, int dk, int dv, int delta, int dtype, void *workspace,
                   size_t workspace_bytes, void *stream);

/* Bytes of workspace ldn_rla_fwd_ws uses for these sizes (0: none needed, or a
 * shape without the chunk form).  Pure host function. */
size_t ldn_rla_fwd_workspace_size(int B, int T, int H, int dk, int dv, int delta, int dtype);

/* Synchronises `stream`, then reads and clears the device status word on the
 * current device.  Returns LDN_OK, LDN_ERR_TIMEOUT (a kernel abandoned a
 * bounded wait and left its outputs incomplete) or LDN_ERR_CUDA. */
int ldn_get_device_status(void *stream);

/* Static, NUL-terminated description of a status code. */
const char *ldn_status_string(int status);

/* LDN_VERSION of the loaded library. */
int ldn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LDN_H */
