/*
 * w4a16_testing.h -- test and benchmark hooks of the GB300 W4A16 library.
 *
 * Not part of the stable API (w4a16.h). They change process-global choices that
 * w4a16_matmul, q4b32_gemv, nvfp4_gemv and mxfp4_gemv read on the host before each
 * launch, so they must not be called while another host thread is issuing those calls.
 * The pages have no counterpart: they exist so that tests can check every kernel at every
 * shape and the benchmark can compare the kernels.
 */
#ifndef W4A16_GB300_TESTING_H
#define W4A16_GB300_TESTING_H

#ifdef __cplusplus
extern "C" {
#endif

/* Kernel w4a16_matmul uses: 0 = chosen by M (default), 1 = the small-M GEMV kernel
 * (forced for M > 8 it runs once per block of 8 rows), 2 = the TMA + tcgen05
 * tensor-core kernel, 3 = the skinny kernel (M <= 32; needs the workspace that
 * w4a16_matmul_workspace_bytes reports for an M in the skinny range). Returns the previous
 * choice, or -1 if `kernel` is out of range (nothing changes then). */
int w4a16_testing_force_kernel(int kernel);

/* Largest M that the by-M choice sends to the GEMV kernel (default 8, its maximum). A
 * negative value only queries. Returns the previous value. */
int w4a16_testing_set_gemv_max_m(int m);

/* Range of M that the by-M choice sends to the skinny kernel when the shape fits it and the
 * workspace is large enough (default 5..32; hi at most 32). Negative values only query.
 * Returns the previous range as (lo << 8) | hi. */
int w4a16_testing_set_skinny_range(int lo, int hi);

/* Range of M for which w4a16_matmul_prepared runs the prepared-layout kernel (default
 * 32..128): smallest and largest M; values below 1 only query. Each returns the previous
 * value. */
int w4a16_testing_set_prepared_min_m(int m);
int w4a16_testing_set_prepared_max_m(int m);

/* Kernel of q4b32_gemv: 2 = TMA-staged tensor-pipe kernel (default; shapes it does not
 * take fall back to 1), 1 = CUDA-core kernel with mixed FP16 FMAs, 0 = CUDA-core kernel
 * with packed fp32 FMAs. Other values only query. Returns the previous value. */
int w4a16_testing_set_q4_variant(int v);

/* Kernel of nvfp4_gemv and mxfp4_gemv: 1 = TMA-staged tensor-pipe kernel (default; shapes
 * it does not take, K % 512 != 0 or x too long for its ring, fall back to 0), 0 = the
 * plain-load kernel. Other values only query. Returns the previous value. */
int w4a16_testing_set_fp4_variant(int v);

/* Kernel of w8a16_gemv: 1 = TMA-staged tensor-pipe kernel (default; shapes it does not take,
 * K % 512 != 0 or x too long for its ring, fall back to 0), 0 = the plain-load kernel. Other
 * values only query. Returns the previous value. */
int w4a16_testing_set_w8_variant(int v);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_GB300_TESTING_H */
