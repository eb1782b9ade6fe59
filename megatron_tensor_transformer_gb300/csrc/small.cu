// The memory-bound pieces around the two GEMM halves: the shard fold ("all-reduce"),
// RMSNorm, and the one-token attention stand-in that maps each shard's heads.
#include "common.cuh"
#include <cuda_fp8.h>

#include "small.h"

#include <algorithm>

namespace tpx {

// y = bf16( ((P_0 + P_1) + ... + P_{t-1}) + residual ): Z = sum_k Z_k of the row-parallel
// split ("Tensor Parallelism (Megatron-Style)", arunshar.com), folded in shard order so that
// every run gives the same bits.  Four outputs per thread (d % 4 == 0).
__global__ void reduce_kernel(const float* __restrict__ P, int t, size_t MN, int pstride_unused,
                              const __nv_bfloat16* __restrict__ res, __nv_bfloat16* y) {
  (void)pstride_unused;
  const size_t n4 = MN / 4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    float4 v = __ldcs(reinterpret_cast<const float4*>(P) + i);
    for (int s = 1; s < t; ++s) {
      const float4 p = __ldcs(reinterpret_cast<const float4*>(P + (size_t)s * MN) + i);
      v.x += p.x;
      v.y += p.y;
      v.z += p.z;
      v.w += p.w;
    }
    if (res) {
      const uint2 r = *reinterpret_cast<const uint2*>(res + 4 * i);
      v.x += bf16_lo(r.x);
      v.y += bf16_hi(r.x);
      v.z += bf16_lo(r.y);
      v.w += bf16_hi(r.y);
    }
    uint2 o;
    o.x = (uint32_t)f2bf(v.x) | ((uint32_t)f2bf(v.y) << 16);
    o.y = (uint32_t)f2bf(v.z) | ((uint32_t)f2bf(v.w) << 16);
    *reinterpret_cast<uint2*>(y + 4 * i) = o;
  }
}

cudaError_t launch_reduce(const float* P, int t, int M, int d, const __nv_bfloat16* res,
                          __nv_bfloat16* y, cudaStream_t st) {
  const size_t MN = (size_t)M * d;
  const size_t n4 = MN / 4;
  int blocks = (int)std::min<size_t>((n4 + 255) / 256, 152 * 8);
  if (blocks < 1) blocks = 1;
  reduce_kernel<<<blocks, 256, 0, st>>>(P, t, MN, 0, res, y);
  note_launch();
  return cudaGetLastError();
}

// RMSNorm, one CTA per token: a = x / sqrt(mean(x^2) + eps) * g.  The sum of squares is
// taken in a fixed order (per-thread strided sums, then a fixed tree) so runs repeat bitwise.
__global__ void rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gain,
                               float eps, int d, __nv_bfloat16* out) {
  __shared__ float part[32];
  const int m = blockIdx.x;
  const __nv_bfloat16* xr = x + (size_t)m * d;
  float ss = 0.f;
  for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
      ss += a * a;
      ss += b * b;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) part[0] = v;
  }
  __syncthreads();
  const float inv = 1.0f / sqrtf(part[0] / (float)d + eps);
  for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint4 gv = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);  // 1.0 pairs
    if (gain) gv = *reinterpret_cast<const uint4*>(gain + i);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w[j]) * inv * bf16_lo(gw[j]);
      const float b = bf16_hi(w[j]) * inv * bf16_hi(gw[j]);
      o[j] = (uint32_t)f2bf(a) | ((uint32_t)f2bf(b) << 16);
    }
    *reinterpret_cast<uint4*>(out + (size_t)m * d + i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* gain, float eps, int M, int d,
                           __nv_bfloat16* out, cudaStream_t st) {
  rmsnorm_kernel<<<M, 256, 0, st>>>(x, gain, eps, d, out);
  note_launch();
  return cudaGetLastError();
}

// RMSNorm as a per-token factor (the layer folds it into the next GEMM's epilogue, so the
// normalised activations are never written): one block per token, the same sum of squares as
// rmsnorm_kernel (eight values per thread per step, a shuffle tree per warp, then the warps in order).
__global__ void rms_factors_kernel(const __nv_bfloat16* __restrict__ x, float eps, int d, float* __restrict__ r) {
  __shared__ float part[32];
  const int m = blockIdx.x;
  const __nv_bfloat16* xr = x + (size_t)m * d;
  float ss = 0.f;
  for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
      ss += a * a;
      ss += b * b;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) r[m] = 1.0f / sqrtf(v / (float)d + eps);
  }
}

cudaError_t launch_rms_factors(const __nv_bfloat16* x, float eps, int M, int d, float* r, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  rms_factors_kernel<<<M, 256, 0, st>>>(x, eps, d, r);
  note_launch();
  return cudaGetLastError();
}

// One thread per token: the d / 32 partial sums of squares in group order, then the factor.
__global__ void rms_factors_from_ss_kernel(const float* __restrict__ ss, float eps, int M, int d,
                                           float* __restrict__ r) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const int g = d / 32;
  const float* row = ss + (size_t)m * g;
  float acc = 0.f;
  for (int i = 0; i < g; ++i) acc += row[i];
  r[m] = 1.0f / sqrtf(acc / (float)d + eps);
}

cudaError_t launch_rms_factors_from_ss(const float* ss, float eps, int M, int d, float* r, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  rms_factors_from_ss_kernel<<<(M + 127) / 128, 128, 0, st>>>(ss, eps, M, d, r);
  note_launch();
  return cudaGetLastError();
}

// Per-token max |x| for the hi/lo split of an e4m3 decode block (exact: a maximum does not round),
// one block per token: eight values per thread per step, a shuffle tree per warp, then the warps.
// As a programmatic dependent it first lets the block kernel after it launch (that kernel starts
// streaming weights and waits for this one before it reads the maxima), then waits for the kernel
// before it, which may have written x.
__global__ void token_absmax_kernel(const __nv_bfloat16* __restrict__ x, int d, unsigned* __restrict__ out) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float part[32];
  const int m = blockIdx.x;
  const __nv_bfloat16* xr = x + (size_t)m * d;
  float mx = 0.f;
  for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) out[m] = __float_as_uint(v);
  }
}

cudaError_t launch_token_absmax(const __nv_bfloat16* x, int M, int d, unsigned* out, bool pdl, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, token_absmax_kernel, x, d, out);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// One-token attention per shard: q head h (shard s = h / nq_s) returns the v of its kv group,
// which lives in the same shard.  qkv is shard-major [q_s | k_s | v_s]; o_in is in head order.
// Prefill with e4m3 weights: each shard is widened once per call, exactly, to the bf16 codes
// the tensor cores read (the per-channel scales stay in the GEMM epilogue), so the GEMM runs
// as a plain bf16 GEMM.  16 codes per thread: one 16-byte streaming load, two 16-byte stores.
__global__ void widen_e4m3_kernel(const uint8_t* __restrict__ src, uint64_t src_stride, size_t per_shard16,
                                  int t, __nv_bfloat16* __restrict__ dst) {
  const size_t n = per_shard16 * (size_t)t;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t s = i / per_shard16, j = i % per_shard16;
    const uint4 v = ld_stream16(src + s * src_stride + j * 16);
    const uint2 c0 = e4m3x4_to_bf16x4(v.x), c1 = e4m3x4_to_bf16x4(v.y);
    const uint2 c2 = e4m3x4_to_bf16x4(v.z), c3 = e4m3x4_to_bf16x4(v.w);
    uint4* o = reinterpret_cast<uint4*>(dst + i * 16);
    o[0] = make_uint4(c0.x, c0.y, c1.x, c1.y);
    o[1] = make_uint4(c2.x, c2.y, c3.x, c3.y);
  }
}

// One CTA per token: the row's absmax (fp32 of the bf16 values), then every code.  The division
// and the rounding are the IEEE binary32 ones the definition names (no fast reciprocal).
__global__ void quantize_tok_kernel(const __nv_bfloat16* __restrict__ x, int ldx, int K, uint8_t* __restrict__ q,
                                    int ldq, float* __restrict__ s) {
  __shared__ float wmax[32];
  const int m = blockIdx.x;
  const __nv_bfloat16* xr = x + (size_t)m * ldx;
  float amax = 0.f;
  for (int k = 8 * threadIdx.x; k < K; k += 8 * blockDim.x) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? wmax[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) wmax[0] = v;
  }
  __syncthreads();
  const float sc = wmax[0] > 0.f ? __fdiv_rn(wmax[0], 448.0f) : 1.0f;
  if (threadIdx.x == 0) s[m] = sc;
  uint8_t* qr = q + (size_t)m * ldq;
  for (int k = 8 * threadIdx.x; k < K; k += 8 * blockDim.x) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(__uint_as_float(w[i] << 16), sc), __NV_SATFINITE, __NV_E4M3);
      const uint32_t c1 =
          __nv_cvt_float_to_fp8(__fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), sc), __NV_SATFINITE, __NV_E4M3);
      o[i >> 1] |= (c0 | (c1 << 8)) << (16 * (i & 1));
    }
    *reinterpret_cast<uint2*>(qr + k) = make_uint2(o[0], o[1]);
  }
}

cudaError_t launch_quantize_fp8_per_token(const __nv_bfloat16* x, int ldx, int M, int K, uint8_t* q, int ldq,
                                          float* s, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  quantize_tok_kernel<<<M, 256, 0, st>>>(x, ldx, K, q, ldq, s);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_widen_e4m3(const uint8_t* src, uint64_t src_stride, int rows, int K, int t, __nv_bfloat16* dst,
                              cudaStream_t st) {
  const size_t per_shard16 = (size_t)rows * K / 16;
  int blocks = (int)std::min<size_t>((per_shard16 * t + 255) / 256, 152 * 16);
  if (blocks < 1) blocks = 1;
  widen_e4m3_kernel<<<blocks, 256, 0, st>>>(src, src_stride, per_shard16, t, dst);
  note_launch();
  return cudaGetLastError();
}

// Vocabulary-parallel embedding: each shard owns the ids of its range; for a token only the
// owning shard contributes a row and the others contribute zeros, so the sum over shards is
// that row, copied here directly.  One CTA per token, 16 bytes per thread per step.
__global__ void embed_kernel(const uint8_t* __restrict__ table, uint64_t stride, int vs, int t, int vocab, int d,
                             const int32_t* __restrict__ ids, __nv_bfloat16* __restrict__ x) {
  const int m = blockIdx.x;
  const int id = ids[m];
  const bool ok = id >= 0 && id < vocab && id / vs < t;
  const uint4* src = ok ? reinterpret_cast<const uint4*>(table + (size_t)(id / vs) * stride +
                                                         (size_t)(id % vs) * d * 2)
                        : nullptr;
  uint4* dst = reinterpret_cast<uint4*>(x + (size_t)m * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = ok ? src[i] : make_uint4(0, 0, 0, 0);
}

cudaError_t launch_embed(const uint8_t* table, uint64_t stride, int vs, int t, int vocab, int d, const int32_t* ids,
                         int M, __nv_bfloat16* x, cudaStream_t st) {
  embed_kernel<<<M, 128, 0, st>>>(table, stride, vs, t, vocab, d, ids, x);
  note_launch();
  return cudaGetLastError();
}

__global__ void attn1_kernel(const __nv_bfloat16* __restrict__ qkv, int M, int n_q, int n_kv, int hd,
                             int t, __nv_bfloat16* o_in) {
  const int nqs = n_q / t, nkvs = n_kv / t, group = n_q / n_kv;
  const int Qs = (nqs + 2 * nkvs) * hd, Q = Qs * t;
  const int vec_per_row = n_q * hd / 8;
  const size_t total = (size_t)M * vec_per_row;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int m = (int)(i / vec_per_row), v = (int)(i % vec_per_row);
    const int col = v * 8, h = col / hd, e = col % hd;
    const int s = h / nqs, hl = h % nqs, kvl = hl / group;
    const size_t src = (size_t)m * Q + (size_t)s * Qs + (size_t)(nqs + nkvs) * hd + kvl * hd + e;
    *reinterpret_cast<uint4*>(o_in + (size_t)m * n_q * hd + col) =
        *reinterpret_cast<const uint4*>(qkv + src);
  }
}

cudaError_t launch_attn1(const __nv_bfloat16* qkv, int M, int n_q, int n_kv, int hd, int t,
                         __nv_bfloat16* o_in, cudaStream_t st) {
  const size_t total = (size_t)M * n_q * hd / 8;
  int blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 4);
  if (blocks < 1) blocks = 1;
  attn1_kernel<<<blocks, 256, 0, st>>>(qkv, M, n_q, n_kv, hd, t, o_in);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tpx
