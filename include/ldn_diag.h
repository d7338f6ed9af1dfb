/*
 * ldn_diag.h -- diagnostic entry points, in a library of their own
 * (lib/libldn_diag.so, built beside libldn.so; not part of the product ABI).
 *
 * These do not compute the method; they expose, on tiny inputs, the hardware
 * building blocks the tensor-core kernels of ldn.h are made of, so that tests
 * can check each encoding against a plain matrix product, and they drive a
 * bounded wait to its limit so that tests can check the failure path.
 * Pointers are device pointers; calls are asynchronous on `stream`; argument
 * errors return synchronously (LDN_ERR_* of ldn.h); a kernel that abandons a
 * bounded wait sets LDN_ERR_TIMEOUT in this library's own status word, read
 * (and cleared) by ldn_diag_get_device_status().
 */
#ifndef LDN_DIAG_H
#define LDN_DIAG_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One tcgen05.mma chain (kind::f16, fp32 accumulate in TMEM), D = A * B^T
 * over K, with A [M][K] and B [N][K] 16-bit row-major in global memory --
 * both fp16 (fmt = 0) or both bf16 (fmt = 1) -- placed in shared memory with
 * 128-byte swizzle, K-major (a_mn / b_mn = 0) or MN-major (= 1).  The accumulator's TMEM region is prefilled with
 * -12345.0 and then dumped whole: D_out [128][N] fp32, row = TMEM lane.
 * M in {64, 128}; N in [16, 256], N % 16 == 0 (N % 64 == 0 if b_mn);
 * K in [16, 128], K % 16 == 0.
 */
int ldn_diag_umma(const void *A, const void *B, float *D_out, int M, int N, int K, int a_mn, int b_mn,
                  int fmt, void *stream);

/*
 * The same chain with A held in tensor memory (M = 128): row r of A [128][K]
 * is written to TMEM lane r as 16-bit pairs (element k in the low half of a
 * 32-bit column for even k, the high half for odd k), and tcgen05.mma reads it
 * from there; B [N][K] is staged as for ldn_diag_umma.  D_out [128][N] fp32.
 * N in [16, 256], N % 16 == 0 (N % 64 == 0 if b_mn); K in {32, 64, 96, 128}.
 */
int ldn_diag_umma_tmem_a(const void *A, const void *B, float *D_out, int N, int K, int b_mn, int fmt,
                         void *stream);

/*
 * TMA tiled load (SWIZZLE_128B, box 64 x 64) of rows [row0, row0 + 64) and
 * columns [col0, col0 + 64) of a bf16 matrix src [rows][cols]; rows past the
 * end read as zero.  The 8192 bytes of the shared-memory tile are copied to
 * dst unchanged.  src 16-byte aligned, cols % 8 == 0, col0 % 64 == 0.
 */
int ldn_diag_tma_sw128(const void *src, void *dst, int rows, int cols, int row0, int col0, void *stream);

/*
 * Failure-path check of the bounded waits every kernel uses: one CTA waits on
 * an mbarrier that nothing arrives on, gives up after timeout_ns (at most 2 s),
 * sets LDN_ERR_TIMEOUT in the status word and returns normally, leaving the
 * context usable.  *waited_ok (device int) receives 1 if the wait succeeded,
 * 0 if it timed out.
 */
int ldn_diag_wait_timeout(long long timeout_ns, int *waited_ok, void *stream);

/*
 * Synchronises `stream`, then reads and clears the diagnostic kernels' status
 * word: LDN_OK, LDN_ERR_TIMEOUT (a diagnostic kernel abandoned a bounded wait)
 * or LDN_ERR_CUDA.
 */
int ldn_diag_get_device_status(void *stream);

#ifdef __cplusplus
}
#endif
#endif /* LDN_DIAG_H */
