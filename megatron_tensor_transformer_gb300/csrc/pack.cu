// Weight partition + pack (+ FP8 e4m3 per-output-channel quantisation).
//
// Column-parallel weights (W_gate/W_up, W_qkv) are split on the output dim and
// row-parallel weights (W_down, W_o) on the input dim ("ColumnParallelLinear" /
// "RowParallelLinear", scalablesystem.dev, "The Tensor-Parallel Shard Group";
// A = [A_1|...|A_t], B = [B_1;...;B_t], arunshar.com "Tensor Parallelism
// (Megatron-Style)").  Each shard is stored K-major ([out rows, in]) so that the
// forward kernels stream whole rows with 16-byte loads.  The packing is a tiled
// transpose through shared memory: reads and writes are both coalesced.
#include "common.cuh"
#include "pack.h"

namespace tpx {

// Unsharded source column (and which matrix) of packed row r of shard s.
__device__ __forceinline__ int colpar_src(const PackGeom& g, int s, int r, int* which) {
  if (g.kind == TP_W_VOCAB) {  // vocabulary id s*V_s + r (>= vocab: a padding row)
    *which = 0;
    return s * g.rows + r;
  }
  if (g.kind == TP_W_GATE_UP) {
    const int fs = g.ffn / g.t;
    const int blk = r >> 4, j = r & 15;
    *which = j >> 3;
    return s * fs + blk * 8 + (j & 7);
  }
  // QKV: [q heads of s | k heads of s | v heads of s]
  *which = 0;
  const int nqs = g.n_q / g.t, nkvs = g.n_kv / g.t, hd = g.hd;
  if (r < nqs * hd) return s * nqs * hd + r;
  r -= nqs * hd;
  if (r < nkvs * hd) return g.n_q * hd + s * nkvs * hd + r;
  r -= nkvs * hd;
  return (g.n_q + g.n_kv) * hd + s * nkvs * hd + r;
}

// Whether packed row r of shard s has a source (padding rows of the vocabulary do not).
__device__ __forceinline__ bool src_valid(const PackGeom& g, int s, int r) {
  return (g.kind != TP_W_VOCAB && g.kind != TP_W_EMBED) || s * g.rows + r < g.vocab;
}

// Map (shard s, packed row r, k) -> element of the [in, out] source.
__device__ __forceinline__ const uint16_t* src_elem(const PackGeom& g, int s, int r, int k) {
  if (g.kind == TP_W_EMBED)  // rows of the [vocab, d] table as they are
    return g.W0 + (size_t)(s * g.rows + r) * g.K + k;
  if (g.colpar) {
    int which;
    const int col = colpar_src(g, s, r, &which);
    const uint16_t* W = which ? g.W1 : g.W0;
    return W + (size_t)k * g.out_cols + col;
  }
  // row-parallel: packed [n][k] = W[s*K_s + k][n]
  return g.W0 + (size_t)(s * g.K + k) * g.out_cols + r;
}

__device__ __forceinline__ float bf16_bits_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Column absmax over the full, unsharded input dim, as float bits (non-negative floats order
// like their bit patterns).  grid: (ceil(rows/256), t, ksplit)
__device__ __forceinline__ unsigned* scale_slot(const PackGeom& g, uint8_t* packed, int s, int r) {
  return reinterpret_cast<unsigned*>(packed + (size_t)s * g.shard_stride + g.scales_offset) + r;
}

__global__ void absmax_kernel(PackGeom g, uint8_t* packed) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  const int s = blockIdx.y;
  if (r >= g.rows) return;
  const int kin = g.colpar ? g.K : g.K * g.t;   // the whole input dim of the source
  const int per = (kin + gridDim.z - 1) / gridDim.z;
  const int k0 = blockIdx.z * per, k1 = min(kin, k0 + per);
  const uint16_t* base;
  if (g.colpar) {
    int which;
    const int col = colpar_src(g, s, r, &which);
    base = (which ? g.W1 : g.W0) + col;
  } else {
    base = g.W0 + r;  // column n = r, every input row
  }
  float m = 0.f;
  for (int k = k0; k < k1; ++k) m = fmaxf(m, fabsf(bf16_bits_to_f(base[(size_t)k * g.out_cols])));
  atomicMax(scale_slot(g, packed, s, r), __float_as_uint(m));
}

// amax -> scale in place (fp32 divide, IEEE round-to-nearest); an all-zero column gets 1.
__global__ void scale_kernel(PackGeom g, uint8_t* packed) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  const int s = blockIdx.y;
  if (r >= g.rows) return;
  unsigned* slot = scale_slot(g, packed, s, r);
  const float amax = __uint_as_float(*slot);
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  *reinterpret_cast<float*>(slot) = sc;
}

// 32x32 tiled transpose of one shard block; grid (K/32, rows/32, t), block (32, 8).
template <bool FP8>
__global__ void pack_kernel(PackGeom g, uint8_t* packed) {
  __shared__ uint16_t tile[32][33];
  const int k0 = blockIdx.x * 32, r0 = blockIdx.y * 32, s = blockIdx.z;
  // read: lanes walk packed rows (source columns), warps walk k (source rows)
  for (int kk = threadIdx.y; kk < 32; kk += 8) {
    const int r = r0 + threadIdx.x, k = k0 + kk;
    uint16_t v = 0;
    if (r < g.rows && k < g.K && src_valid(g, s, r)) v = *src_elem(g, s, r, k);
    tile[kk][threadIdx.x] = v;
  }
  __syncthreads();
  uint8_t* shard = packed + (size_t)s * g.shard_stride;
  for (int rr = threadIdx.y; rr < 32; rr += 8) {
    const int r = r0 + rr, k = k0 + threadIdx.x;
    if (r >= g.rows || k >= g.K) continue;
    const uint16_t v = tile[threadIdx.x][rr];
    if (!FP8) {
      reinterpret_cast<uint16_t*>(shard)[(size_t)r * g.K + k] = v;
    } else {
      const float sc = reinterpret_cast<const float*>(shard + g.scales_offset)[r];
      const float qv = __fdiv_rn(bf16_bits_to_f(v), sc);
      shard[(size_t)r * g.K + k] = (uint8_t)__nv_cvt_float_to_fp8(qv, __NV_SATFINITE, __NV_E4M3);
    }
  }
}

cudaError_t launch_pack(const PackGeom& g, uint8_t* packed, cudaStream_t st) {
  cudaError_t e;
  if (g.fp8) {
    // the amax of each row is accumulated in the shard's own scale slot, then turned into
    // the scale in place
    for (int s = 0; s < g.t; ++s) {
      e = cudaMemsetAsync(packed + (size_t)s * g.shard_stride + g.scales_offset, 0,
                          (size_t)g.rows * 4, st);
      if (e != cudaSuccess) return e;
    }
    const int kin = g.colpar ? g.K : g.K * g.t;
    const int ksplit = kin >= 4096 ? 16 : 1;
    dim3 ga((g.rows + 255) / 256, g.t, ksplit);
    absmax_kernel<<<ga, 256, 0, st>>>(g, packed);
    note_launch();
    dim3 gs((g.rows + 255) / 256, g.t);
    scale_kernel<<<gs, 256, 0, st>>>(g, packed);
    note_launch();
  }
  dim3 blk(32, 8), grid((g.K + 31) / 32, (g.rows + 31) / 32, g.t);
  if (g.fp8)
    pack_kernel<true><<<grid, blk, 0, st>>>(g, packed);
  else
    pack_kernel<false><<<grid, blk, 0, st>>>(g, packed);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tpx
