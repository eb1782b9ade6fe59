// Decode attention over a KV cache, head-sharded: each logical shard owns whole GQA groups (its
// q heads and the kv heads they read) and the cache of those kv heads, so attention is local
// to the shard ("local attention over this GPU's heads", scalablesystem.dev, "The
// Tensor-Parallel Shard Group"; "the KV cache splits too", vidyal.ai model-parallelism).
//
// Per sequence m (one new token each) and q head h of kv head g = h / (n_q / n_kv):
//   o[m, h] = sum_j softmax_j(q . k_j / sqrt(hd)) v_j,   j = 0 .. len[m]
// where position len[m] is the new token itself (appended first).  Three launches:
//   append   the new k, v from qkv into the cache at position len[m];
//   chunks   one CTA per (128-position chunk, sequence, kv head): TMA stages the chunk's k and
//            v rows in shared memory (128-byte swizzle); the group's q heads are the rows of
//            mma.sync tiles, so every k and v byte is read once for all of them; per head the
//            chunk's max, sum of exponentials and un-normalised p.v go to the workspace;
//   combine  per (sequence, q head): the chunks merged in chunk order (log-sum-exp), / sum.
// Every sum has a fixed order, so runs repeat bit for bit.  The pass reads the cache once
// (HBM-bound).  The probabilities enter P V rounded to bf16 (the MMA's operand type).
#include <cuda.h>

#include "attn.h"
#include "common.cuh"
#include "tc.h"
#include "tc_ptx.cuh"

namespace tpx {

namespace {

constexpr int kChunk = 128, kThreads = 128, kWarps = kThreads / 32;  // a warp per 32 positions

struct AttnGeo {
  int t, M, L, n_q, n_kv, hd;
  int nqs, nkvs, G, Qs;  // per shard: q heads, kv heads; q heads per kv head; qkv columns per shard
};

__host__ __device__ inline AttnGeo attn_geo(int t, int M, int L, int n_q, int n_kv, int hd) {
  AttnGeo g{t, M, L, n_q, n_kv, hd, n_q / t, n_kv / t, n_q / n_kv, (n_q + 2 * n_kv) / t * hd};
  return g;
}

// cache element (shard s, sequence m, local kv head gl, position j, dim 0)
__device__ __forceinline__ size_t cache_off(const AttnGeo& g, int s, int m, int gl, int j) {
  return ((((size_t)s * g.M + m) * g.nkvs + gl) * g.L + j) * g.hd;
}

// grid (M, n_kv), block hd / 8 x 2: thread (i, kv) copies 8 values of k (kv = 0) or v (kv = 1)
__global__ void append_kernel(AttnGeo g, const __nv_bfloat16* __restrict__ qkv, const int32_t* __restrict__ lens,
                              __nv_bfloat16* kc, __nv_bfloat16* vc) {
  const int m = blockIdx.x, gg = blockIdx.y, s = gg / g.nkvs, gl = gg % g.nkvs;
  const int n = lens[m];
  if (n < 0 || n >= g.L) return;
  const int i = threadIdx.x, kv = threadIdx.y;
  const size_t src = (size_t)m * g.t * g.Qs + (size_t)s * g.Qs + (size_t)(g.nqs + kv * g.nkvs + gl) * g.hd + 8 * i;
  __nv_bfloat16* dst = (kv ? vc : kc) + cache_off(g, s, m, gl, n) + 8 * i;
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(qkv + src);
}

// Partial results of chunk c for (m, gg): [G][hd] un-normalised p.v, then [G] max, [G] sum.
__device__ __forceinline__ float* part_ptr(const AttnGeo& g, float* ws, int m, int gg, int c) {
  const int nch = (g.L + kChunk - 1) / kChunk;
  const size_t per = (size_t)g.G * (g.hd + 2);
  return ws + (((size_t)m * g.n_kv + gg) * nch + c) * per;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

// Byte offset of (position r, dim k) in a chunk staged as HD/64 boxes of [kChunk rows][64 dims]
// in the 128-byte swizzle (the 16-byte chunk j of a row sits at j ^ (r & 7)).
template <int HD>
__device__ __forceinline__ uint32_t sw_off(int r, int k) {
  return (uint32_t)((k >> 6) * (kChunk * 128) + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + ((k & 7) << 1));
}

// grid (chunks, M, n_kv), 128 threads.  Tensor cores through mma.sync: the group's q heads are
// the 16 rows of the MMA (rows G.. are zero), warp w takes positions 32w .. 32w+31 of the chunk.
//   S = Q K^T (fp32), softmax pieces across the four warps through shared memory, P = exp(S -
//   max) rounded to bf16 as the A operand of O = P V (fp32), the four warps' O summed in order.
template <int HD>
__global__ void __launch_bounds__(kThreads) chunk_kernel(const __grid_constant__ CUtensorMap tmK,
                                                         const __grid_constant__ CUtensorMap tmV, AttnGeo g, float scale,
                                                         const __nv_bfloat16* __restrict__ qkv,
                                                         const int32_t* __restrict__ lens, float* ws, unsigned* err) {
  constexpr int KB = HD / 64 * kChunk * 128;  // bytes of the staged k (or v) chunk
  constexpr int QSTR = HD * 2 + 16;            // padded q row (bytes), ldmatrix without conflicts
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sm;
  uint8_t* sV = sm + KB;
  uint8_t* sQ = sm + 2 * KB;                                     // [16][QSTR]
  float* sMax = reinterpret_cast<float*>(sQ + 16 * QSTR);        // [kWarps][16]
  float* sSum = sMax + kWarps * 16;                              // [kWarps][16]
  float* red = reinterpret_cast<float*>(sK);                     // [kWarps][16][HD], after S is done
  __shared__ __align__(8) uint64_t bar;
  const int c = blockIdx.x, m = blockIdx.y, gg = blockIdx.z, s = gg / g.nkvs, gl = gg % g.nkvs;
  const int n = lens[m];
  if (n < 0 || n >= g.L) return;
  const int p0 = c * kChunk, p1 = min(p0 + kChunk, n + 1);
  if (p0 >= p1) return;
  const int np = p1 - p0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, qq = lane & 3;
  const uint32_t b = tc::smem_u32(&bar);
  if (threadIdx.x == 0) {
    tc::mbar_init(b, 1);
    tc::fence_mbar_init();
    tc::mbar_arrive_expect_tx(b, 2u * KB);
    const int row0 = (((s * g.M + m) * g.nkvs + gl) * g.L) + p0;  // rows past np are masked
#pragma unroll
    for (int bx = 0; bx < HD / 64; ++bx) {
      tc::tma_load_2d(tc::smem_u32(sK + bx * kChunk * 128), &tmK, bx * 64, row0, b);
      tc::tma_load_2d(tc::smem_u32(sV + bx * kChunk * 128), &tmV, bx * 64, row0, b);
    }
  }
  // the group's q heads as 16 bf16 rows (rows >= G zero)
  const __nv_bfloat16* qp = qkv + (size_t)m * g.t * g.Qs + (size_t)s * g.Qs + (size_t)gl * g.G * HD;
  for (int i = threadIdx.x; i < 16 * HD / 8; i += kThreads) {
    const int r = i / (HD / 8), c8 = i % (HD / 8);
    const uint4 v = r < g.G ? *reinterpret_cast<const uint4*>(qp + (size_t)r * HD + 8 * c8) : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(sQ + r * QSTR + 16 * c8) = v;
  }
  __syncthreads();
  if (!tc::mbar_wait(b, 0)) {  // bounded: a copy that never lands records the error and bails
    if (threadIdx.x == 0) atomicExch(err, 40u);
    return;
  }
  if (np < kChunk) {  // staged rows past the sequence's end may hold anything (NaN too): P V sees 0 there
    for (int i = threadIdx.x; i < (kChunk - np) * (HD / 8); i += kThreads) {
      const int r = np + i / (HD / 8), c8 = i % (HD / 8);
      *reinterpret_cast<uint4*>(sV + (c8 >> 3) * (kChunk * 128) + r * 128 + ((c8 & 7) << 4)) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
  }

  // S = Q K^T for this warp's 32 positions: 4 n-tiles of 8 positions, HD/16 k-steps
  float S[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) S[j][i] = 0.f;
  const uint32_t q_base = tc::smem_u32(sQ), k_base = tc::smem_u32(sK), v_base = tc::smem_u32(sV);
#pragma unroll
  for (int k0 = 0; k0 < HD; k0 += 32) {
    uint32_t a[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)  // two k-steps of Q: rows lane % 16, dims k0 + 16h + 8 (lane / 16)
      ldsm_x4(q_base + (lane & 15) * QSTR + (k0 + 16 * h + 8 * (lane >> 4)) * 2, a[h][0], a[h][1], a[h][2], a[h][3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = 32 * warp + 8 * j + (lane & 7);  // position row of this lane's address
      uint32_t b0, b1, b2, b3;                       // dims k0, k0+8, k0+16, k0+24
      ldsm_x4(k_base + sw_off<HD>(r, k0 + 8 * (lane >> 3)), b0, b1, b2, b3);
      mma_bf16_16816(S[j], a[0][0], a[0][1], a[0][2], a[0][3], b0, b1);
      mma_bf16_16816(S[j], a[1][0], a[1][1], a[1][2], a[1][3], b2, b3);
    }
  }
  // scale, mask positions past the chunk's end, row maxima (rows gq and gq + 8)
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int pc = 32 * warp + 8 * j + 2 * qq;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool ok = pc + (i & 1) < np;
      S[j][i] = ok ? S[j][i] * scale : -INFINITY;
    }
    mx0 = fmaxf(mx0, fmaxf(S[j][0], S[j][1]));
    mx1 = fmaxf(mx1, fmaxf(S[j][2], S[j][3]));
  }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  if (qq == 0) {
    sMax[warp * 16 + gq] = mx0;
    sMax[warp * 16 + gq + 8] = mx1;
  }
  __syncthreads();  // every warp's S is done: sK may be reused for the O reduction below
  float M0 = sMax[gq], M1 = sMax[gq + 8];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    M0 = fmaxf(M0, sMax[w * 16 + gq]);
    M1 = fmaxf(M1, sMax[w * 16 + gq + 8]);
  }
  // P = exp(S - max) (masked positions give 0), the rows' partial sums
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    S[j][0] = __expf(S[j][0] - M0);
    S[j][1] = __expf(S[j][1] - M0);
    S[j][2] = __expf(S[j][2] - M1);
    S[j][3] = __expf(S[j][3] - M1);
    l0 += S[j][0] + S[j][1];
    l1 += S[j][2] + S[j][3];
  }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  if (qq == 0) {
    sSum[warp * 16 + gq] = l0;
    sSum[warp * 16 + gq + 8] = l1;
  }
  // O = P V over this warp's 32 positions: 2 k-steps of 16 positions, HD/8 n-tiles of 8 dims
  float O[HD / 8][4];
#pragma unroll
  for (int t8 = 0; t8 < HD / 8; ++t8)
#pragma unroll
    for (int i = 0; i < 4; ++i) O[t8][i] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    // the S fragments of n-tiles 2ks and 2ks+1 are the A fragment of this k-step
    const uint32_t a0 = pack_bf16(S[2 * ks][0], S[2 * ks][1]), a1 = pack_bf16(S[2 * ks][2], S[2 * ks][3]);
    const uint32_t a2 = pack_bf16(S[2 * ks + 1][0], S[2 * ks + 1][1]), a3 = pack_bf16(S[2 * ks + 1][2], S[2 * ks + 1][3]);
    const int r = 32 * warp + 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);  // position row
#pragma unroll
    for (int t16 = 0; t16 < HD / 16; ++t16) {
      uint32_t b0, b1, b2, b3;  // (positions +0/+8) x (dims 16 t16 + 0 / + 8), transposed
      ldsm_x4_t(v_base + sw_off<HD>(r, 16 * t16 + 8 * (lane >> 4)), b0, b1, b2, b3);
      mma_bf16_16816(O[2 * t16], a0, a1, a2, a3, b0, b1);
      mma_bf16_16816(O[2 * t16 + 1], a0, a1, a2, a3, b2, b3);
    }
  }
  // the four warps' O summed in warp order; rows < G go to the workspace with max and sum
#pragma unroll
  for (int t8 = 0; t8 < HD / 8; ++t8) {
    const int d = 8 * t8 + 2 * qq;
    red[(warp * 16 + gq) * HD + d] = O[t8][0];
    red[(warp * 16 + gq) * HD + d + 1] = O[t8][1];
    red[(warp * 16 + gq + 8) * HD + d] = O[t8][2];
    red[(warp * 16 + gq + 8) * HD + d + 1] = O[t8][3];
  }
  __syncthreads();
  float* part = part_ptr(g, ws, m, gg, c);
  for (int e = threadIdx.x; e < g.G * HD; e += kThreads) {
    const int hi = e / HD, d = e % HD;
    float acc = red[hi * HD + d];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) acc += red[(w * 16 + hi) * HD + d];
    part[(size_t)hi * HD + d] = acc;
  }
  if (threadIdx.x < g.G) {
    const int hi = threadIdx.x;
    float mxa = sMax[hi], sma = 0.f;
#pragma unroll
    for (int w = 1; w < kWarps; ++w) mxa = fmaxf(mxa, sMax[w * 16 + hi]);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) sma += sSum[w * 16 + hi];
    part[(size_t)g.G * HD + hi] = mxa;
    part[(size_t)g.G * HD + g.G + hi] = sma;
  }
}

// grid (M, n_q): block HD threads, one dim each; merges the sequence's chunks in order
__global__ void combine_kernel(AttnGeo g, const int32_t* __restrict__ lens, const float* __restrict__ ws,
                               __nv_bfloat16* o_in) {
  const int m = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int s = h / g.nqs, hl = h % g.nqs, gl = hl / g.G, hi = hl % g.G, gg = s * g.nkvs + gl;
  const int n = lens[m];
  __nv_bfloat16* out = o_in + (size_t)m * g.n_q * g.hd + (size_t)h * g.hd + d;
  if (n < 0 || n >= g.L) {
    *out = __float2bfloat16_rn(0.f);
    return;
  }
  const int nch = (n + 1 + kChunk - 1) / kChunk;
  float M_all = -INFINITY;
  for (int c = 0; c < nch; ++c) M_all = fmaxf(M_all, part_ptr(g, const_cast<float*>(ws), m, gg, c)[g.G * g.hd + hi]);
  float L_all = 0.f, acc = 0.f;
  for (int c = 0; c < nch; ++c) {
    const float* pt = part_ptr(g, const_cast<float*>(ws), m, gg, c);
    const float f = __expf(pt[g.G * g.hd + hi] - M_all);
    L_all += pt[g.G * g.hd + g.G + hi] * f;
    acc += pt[(size_t)hi * g.hd + d] * f;
  }
  *out = __float2bfloat16_rn(acc / L_all);
}

}  // namespace

size_t attn_workspace_bytes(int t, int M, int L, int n_q, int n_kv, int hd) {
  const AttnGeo g = attn_geo(t, M, L, n_q, n_kv, hd);
  const size_t nch = (size_t)(L + kChunk - 1) / kChunk;
  return (size_t)M * n_kv * nch * g.G * (hd + 2) * sizeof(float);
}

bool attn_supported(int hd, int G) { return (hd == 64 || hd == 128 || hd == 256) && G >= 1 && G <= 16; }

cudaError_t launch_attn_decode(int t, int M, int L, int n_q, int n_kv, int hd, const __nv_bfloat16* qkv,
                               __nv_bfloat16* kc, __nv_bfloat16* vc, const int32_t* lens, __nv_bfloat16* o_in,
                               float* ws, unsigned* err, cudaStream_t st) {
  const AttnGeo g = attn_geo(t, M, L, n_q, n_kv, hd);
  append_kernel<<<dim3(M, n_kv), dim3(hd / 8, 2), 0, st>>>(g, qkv, lens, kc, vc);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((L + kChunk - 1) / kChunk, M, n_kv);
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tm[2];
  for (int i = 0; i < 2; ++i) {  // the cache as [t M n_kv/t L rows][hd], boxes of 128 rows x 64 dims
    const cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)t * M * (n_kv / t) * L};
    const cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kChunk}, es[2] = {1, 1};
    if (enc(&tm[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, i ? (void*)vc : (void*)kc, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const size_t smem = 1024 + 2 * (size_t)(hd / 64) * kChunk * 128 + 16 * ((size_t)hd * 2 + 16) + 2 * kWarps * 16 * 4;
  const float scale = 1.0f / sqrtf((float)hd);
  auto launch = [&](auto kernel) {
    const cudaError_t a = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (a != cudaSuccess) return a;
    kernel<<<grid, kThreads, smem, st>>>(tm[0], tm[1], g, scale, qkv, lens, ws, err);
    note_launch();
    return cudaGetLastError();
  };
  if (hd == 64) e = launch(chunk_kernel<64>);
  else if (hd == 128) e = launch(chunk_kernel<128>);
  else e = launch(chunk_kernel<256>);
  if (e != cudaSuccess) return e;
  combine_kernel<<<dim3(M, n_q), hd, 0, st>>>(g, lens, ws, o_in);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tpx
