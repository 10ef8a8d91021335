/*
 * libkda_probe -- TEST-ONLY probes of the tcgen05 / TMA building blocks the
 * KDA kernels are made of.  Not part of the product interface (kda.h); the
 * test-suite uses them to check operand layouts, instruction descriptors and
 * the TMEM lane mapping against a host matmul.  There is no counterpart on
 * the pages: these exist only to validate this implementation.
 */
#ifndef KDA_PROBE_H
#define KDA_PROBE_H

#include <cuda_runtime_api.h>

#ifndef KDA_API
#define KDA_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One CTA computes D = (+/-) n_accum * A * B[b_row0 : b_row0 + N]^T with
 * tcgen05.mma (kind::f16, bf16 in, fp32 accumulate) over K in 16-wide steps.
 *   A : device bf16 [M][K] row-major (M = 64 or 128)
 *   B : device bf16 [NB][K] row-major, NB >= b_row0 + N, NB <= 256
 *   D : device fp32 [128][N] -- the raw accumulator, TMEM lane by column
 * Operands are placed in shared memory K-major (x_mn = 0) or MN-major
 * (x_mn = 1) with swizzle code x_sw (2 = 128B, 4 = 64B, 6 = 32B); for
 * MN-major, x_mn_blocks_contig selects which of the two strides is dense.
 * tf32 = 1 stores both operands as fp32 and runs kind::tf32 (8-wide K steps);
 * then M*K*4 <= 32 KiB and NB*K*4 <= 64 KiB, and neg_a must be 0.
 * status : device int, set to 6 when the completion wait times out.
 * Returns 0 on launch, 1 on bad arguments, 4 on a CUDA error.
 */
KDA_API int kda_probe_umma(const void* A, const void* B, float* D, int M, int N, int K, int NB,
                   int a_mn, int a_sw, int a_mn_blocks_contig, int b_mn, int b_sw,
                   int b_mn_blocks_contig, int b_row0, int neg_a, int n_accum, int tf32,
                   int* status, cudaStream_t stream);

/*
 * kda_probe_umma with one more switch: a_tmem = 1 writes A (M = 128, bf16,
 * K <= 128) into tensor memory, row m in lane m, two consecutive K elements
 * per 32-bit column (the lower half the even one), and runs the MMA with A
 * read from tensor memory (a_mn must be 0, tf32 0).  a_tmem = 0 is
 * kda_probe_umma.
 */
KDA_API int kda_probe_umma_ta(const void* A, const void* B, float* D, int M, int N, int K, int NB,
                      int a_mn, int a_sw, int a_mn_blocks_contig, int b_mn, int b_sw,
                      int b_mn_blocks_contig, int b_row0, int neg_a, int n_accum, int tf32,
                      int a_tmem, int* status, cudaStream_t stream);

/*
 * TMA-loads the 64-token x d-channel tile of head h starting at token t0
 * from src (bf16 [T][H][d]) in 64-channel boxes with 128-byte swizzle, and
 * reads it back through the K-major layout function into out (bf16 [64][d]).
 * Tokens past T read as zero.  Returns 0 / 1 / 4 as above.
 */
KDA_API int kda_probe_tma(const void* src, void* out, int T, int H, int d, int h, int t0, int* status,
                  cudaStream_t stream);

/*
 * Makes a device-side wait run out on purpose: one CTA allocates TMEM, sets
 * up an mbarrier that nothing arrives on and waits on it with the KDA
 * kernels' bounded wait, limited to limit_us microseconds (1..100000).  The
 * wait gives up, *status (device int) is set to 6 (KDA_ERR_TIMEOUT), the
 * TMEM is freed and the kernel returns.  Returns 0 / 1 / 4 as above.
 */
KDA_API int kda_probe_wait_timeout(int limit_us, int* status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif
