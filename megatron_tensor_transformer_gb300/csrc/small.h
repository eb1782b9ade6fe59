// Host-side interface of the fold / RMSNorm / attention stand-in kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tpx {

cudaError_t launch_reduce(const float* P, int t, int M, int d, const __nv_bfloat16* res,
                          __nv_bfloat16* y, cudaStream_t st);
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* gain, float eps, int M, int d,
                           __nv_bfloat16* out, cudaStream_t st);
// e4m3 weight shards (shard s at s * src_stride bytes, [rows, K] codes) -> bf16 codes, exactly,
// in the same per-shard layout, shards packed densely (shard s at s * rows * K elements).
cudaError_t launch_widen_e4m3(const uint8_t* src, uint64_t src_stride, int rows, int K, int t, __nv_bfloat16* dst,
                              cudaStream_t st);
// Per-token e4m3 quantisation of activations x [M][K] (row stride ldx): s[m] = absmax / 448 in
// binary32 (1 for an all-zero row), q[m][k] = e4m3 RNE satfinite of x / s[m] (binary32 divide);
// q has row stride ldq bytes.  K % 8 == 0, rows 16-byte aligned.
cudaError_t launch_quantize_fp8_per_token(const __nv_bfloat16* x, int ldx, int M, int K, uint8_t* q, int ldq,
                                          float* s, cudaStream_t st);
// x[m] = row ids[m] of the vocabulary-split table (shard ids[m] / vs, row ids[m] % vs; shard s at
// s * stride bytes, rows of d bf16), or zeros for an id outside [0, vocab).
cudaError_t launch_embed(const uint8_t* table, uint64_t stride, int vs, int t, int vocab, int d, const int32_t* ids,
                         int M, __nv_bfloat16* x, cudaStream_t st);
// RMSNorm (gain 1) as per-token factors: r[m] = 1/sqrt(mean_k x[m][k]^2 + eps), x [M, d] bf16.
cudaError_t launch_rms_factors(const __nv_bfloat16* x, float eps, int M, int d, float* r, cudaStream_t st);
// The same factors from per-(token, 32-row group) sums of squares ss [M][d / 32], summed in group order.
cudaError_t launch_rms_factors_from_ss(const float* ss, float eps, int M, int d, float* r, cudaStream_t st);
// Per-token max |x[m][k]| over k as float bits, out[m] for m < M, x [M, d] bf16 (d % 8 == 0): the split
// scales of an e4m3 decode block's input.  pdl: launched as a programmatic dependent (it waits for the
// kernel before it, and lets the block after it launch at once).
cudaError_t launch_token_absmax(const __nv_bfloat16* x, int M, int d, unsigned* out, bool pdl, cudaStream_t st);
cudaError_t launch_attn1(const __nv_bfloat16* qkv, int M, int n_q, int n_kv, int hd, int t,
                         __nv_bfloat16* o_in, cudaStream_t st);

}  // namespace tpx
