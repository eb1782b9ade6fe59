// Weight-streaming skinny GEMM for decode-sized M (<= 64 tokens per launch).
//
// The column-parallel half (QKV, gate/up + SwiGLU) and the row-parallel half
// (o_proj, down + the shard fold) of a Megatron block ("The Tensor-Parallel Shard
// Group", scalablesystem.dev; "Tensor Parallelism (Megatron-Style)", arunshar.com)
// are both HBM-bound at decode: every weight byte is read once and used M times.
//
// Design (GB300):
//  * Each thread streams 16-byte weight vectors straight into mma.sync fragment
//    registers.  The k index inside each 32-wide chunk is permuted identically for
//    the weight and activation operands, so a 16-byte load of 8 consecutive k
//    values feeds two m16n8k16 MMAs without shared memory.
//  * Tokens sit on the MMA's M side (16 per tile, masked), weight rows on N (8 per
//    group); a warp owns R groups (8R weight rows) x all tokens over a k-range.
//  * A CTA's 8 warps split the k dimension; their partial tiles are folded in
//    shared memory in warp order (fixed, deterministic).
//  * Row-parallel: the warps of a CTA split (shard, k-range); shard partials are
//    folded left to right in shard order with the residual, either in the CTA
//    (all shards in one CTA) or by the last-arriving CTA of a tile (ticket in the
//    workspace; no CTA ever waits).  The unfused path writes the same partials
//    and runs the same fold in tp_reduce_partials, so both give identical bits.
#include "common.cuh"
#include "skinny.h"

namespace tpx {

constexpr int kWarps = 8;

template <typename WT>
struct WTraits;
template <>
struct WTraits<uint16_t> {  // bf16 weights: a chunk is 32 k values, 16 B per thread per row
  static constexpr int kChunk = 32;
};
template <>
struct WTraits<uint8_t> {  // e4m3 weights: a chunk is 64 k values, 16 B per thread per row
  static constexpr int kChunk = 64;
};

// acc[tt][r][0..3] += X[tokens of tile tt] . W[rows of group r]^T over chunks [c0, c1).
template <typename WT, int TT, int R, int U>
__device__ __forceinline__ void warp_stream(const WT* __restrict__ wrow0, int K,
                                            const __nv_bfloat16* __restrict__ x, int ldx, int M,
                                            int c0, int c1, float (&acc)[TT][R][4]) {
  constexpr int CH = WTraits<WT>::kChunk;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  // per-thread base pointers
  const WT* wp[R];
#pragma unroll
  for (int r = 0; r < R; ++r) wp[r] = wrow0 + (size_t)(r * 8 + g) * K + q * (16 / sizeof(WT));
  const __nv_bfloat16* xp[TT][2];
  bool xv[TT][2];
#pragma unroll
  for (int tt = 0; tt < TT; ++tt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int m = tt * 16 + g + h * 8;
      xv[tt][h] = m < M;
      xp[tt][h] = x + (size_t)(xv[tt][h] ? m : 0) * ldx;
    }
  }
  for (int c = c0; c < c1; c += U) {
    uint4 wv[U][R];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (c + u < c1)
          wv[u][r] = ld_stream16(wp[r] + (size_t)(c + u) * CH);
        else
          wv[u][r] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (c + u >= c1) break;
      const int kb = (c + u) * CH;
      if constexpr (sizeof(WT) == 2) {
        // thread q holds k = kb + 8q .. 8q+7 of its rows and of its tokens
        uint4 xa[TT][2];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            xa[tt][h] = xv[tt][h] ? ld_ro16(xp[tt][h] + kb + 8 * q) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int tt = 0; tt < TT; ++tt)
#pragma unroll
          for (int r = 0; r < R; ++r) {
            mma_bf16_16816(acc[tt][r], xa[tt][0].x, xa[tt][1].x, xa[tt][0].y, xa[tt][1].y,
                           wv[u][r].x, wv[u][r].y);
            mma_bf16_16816(acc[tt][r], xa[tt][0].z, xa[tt][1].z, xa[tt][0].w, xa[tt][1].w,
                           wv[u][r].z, wv[u][r].w);
          }
      } else {
        // e4m3: thread q holds k = kb + 16q .. 16q+15; four MMAs of 4 values each
        uint4 xa[TT][2][2];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < 2; ++j)
              xa[tt][h][j] = xv[tt][h] ? ld_ro16(xp[tt][h] + kb + 16 * q + 8 * j)
                                       : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t wr[4] = {wv[u][r].x, wv[u][r].y, wv[u][r].z, wv[u][r].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // bytes 4j..4j+3 of the 16: two bf16x2 operands
            uint32_t b0 = e4m3x2_to_bf16x2((uint16_t)(wr[j] & 0xFFFF));
            uint32_t b1 = e4m3x2_to_bf16x2((uint16_t)(wr[j] >> 16));
#pragma unroll
            for (int tt = 0; tt < TT; ++tt) {
              const uint4& lo0 = xa[tt][0][j >> 1];
              const uint4& lo1 = xa[tt][1][j >> 1];
              uint32_t a0 = (j & 1) ? lo0.z : lo0.x, a2 = (j & 1) ? lo0.w : lo0.y;
              uint32_t a1 = (j & 1) ? lo1.z : lo1.x, a3 = (j & 1) ? lo1.w : lo1.y;
              mma_bf16_16816(acc[tt][r], a0, a1, a2, a3, b0, b1);
            }
          }
        }
      }
    }
  }
}

// Write a warp's accumulators into red[warp][row 0..8R)[token 0..16TT).
template <int TT, int R>
__device__ __forceinline__ void stash(float* red, int warp, const float (&acc)[TT][R][4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  constexpr int MP = 16 * TT, RW = 8 * R;
  float* base = red + (size_t)warp * RW * MP;
#pragma unroll
  for (int tt = 0; tt < TT; ++tt)
#pragma unroll
    for (int r = 0; r < R; ++r) {
      int row = r * 8 + 2 * q, m = tt * 16 + g;
      base[row * MP + m] = acc[tt][r][0];
      base[(row + 1) * MP + m] = acc[tt][r][1];
      base[row * MP + m + 8] = acc[tt][r][2];
      base[(row + 1) * MP + m + 8] = acc[tt][r][3];
    }
}

// ---------------------------------------------------------------- column-parallel

template <typename WT, int TT, int R, int U>
__global__ void __launch_bounds__(kWarps * 32)
    colpar_kernel(ColparArgs a) {
  extern __shared__ float red[];
  constexpr int MP = 16 * TT, RW = 8 * R;
  const int tiles_per_shard = a.rows / RW;
  const int s = blockIdx.x / tiles_per_shard, tile = blockIdx.x % tiles_per_shard;
  const int warp = threadIdx.x >> 5;
  constexpr int CH = WTraits<WT>::kChunk;
  const int nch = a.K / CH;
  const int c0 = warp * nch / kWarps, c1 = (warp + 1) * nch / kWarps;
  const uint8_t* shard = a.w + (size_t)s * a.shard_stride;
  const WT* wrow0 = reinterpret_cast<const WT*>(shard) + (size_t)tile * RW * a.K;

  float acc[TT][R][4];
#pragma unroll
  for (int tt = 0; tt < TT; ++tt)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[tt][r][i] = 0.f;
  warp_stream<WT, TT, R, U>(wrow0, a.K, a.x, a.ldx, a.M, c0, c1, acc);
  stash<TT, R>(red, warp, acc);
  __syncthreads();

  const float* scales = (sizeof(WT) == 1) ? reinterpret_cast<const float*>(shard + a.scales_offset) +
                                                tile * RW
                                          : nullptr;
  auto folded = [&](int row, int m) {
    float v = red[row * MP + m];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) v += red[((size_t)w * RW + row) * MP + m];
    if (sizeof(WT) == 1) v = __fmul_rn(v, scales[row]);
    return v;
  };
  if (a.mode == COLPAR_SWIGLU) {
    constexpr int NF = RW / 2;  // output features of this tile
    for (int i = threadIdx.x; i < NF * a.M; i += blockDim.x) {
      const int m = i / NF, f = i % NF;
      const int grow = (f / 8) * 16 + (f % 8);
      const float gv = folded(grow, m), uv = folded(grow + 8, m);
      const float hv = silu_f(gv) * uv;
      reinterpret_cast<uint16_t*>(a.out)[(size_t)m * a.ldo + (size_t)s * (a.rows / 2) + tile * NF + f] =
          f2bf(hv);
    }
  } else {
    for (int i = threadIdx.x; i < RW * a.M; i += blockDim.x) {
      const int m = i / RW, r = i % RW;
      const float v = folded(r, m);
      const size_t o = (size_t)m * a.ldo + (size_t)s * a.rows + (size_t)tile * RW + r;
      if (a.mode == COLPAR_F32)
        reinterpret_cast<float*>(a.out)[o] = v;
      else
        reinterpret_cast<uint16_t*>(a.out)[o] = f2bf(v);
    }
  }
}

// ---------------------------------------------------------------- row-parallel

template <typename WT, int TT, int R, int U>
__global__ void __launch_bounds__(kWarps * 32)
    rowpar_kernel(RowparArgs a) {
  extern __shared__ float red[];
  __shared__ int s_last;
  constexpr int MP = 16 * TT, RW = 8 * R;
  constexpr int CH = WTraits<WT>::kChunk;
  const int tile = blockIdx.x, cs = blockIdx.y;
  const int spc = a.t / gridDim.y;  // shards in this CTA
  const int ks = kWarps / spc;      // warps (k-ranges) per shard
  const int warp = threadIdx.x >> 5;
  const int sl = warp / ks, kr = warp % ks;
  const int s = cs * spc + sl;
  const int nch = a.K / CH;
  const int c0 = kr * nch / ks, c1 = (kr + 1) * nch / ks;
  const uint8_t* shard = a.w + (size_t)s * a.shard_stride;
  const WT* wrow0 = reinterpret_cast<const WT*>(shard) + (size_t)tile * RW * a.K;

  float acc[TT][R][4];
#pragma unroll
  for (int tt = 0; tt < TT; ++tt)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[tt][r][i] = 0.f;
  warp_stream<WT, TT, R, U>(wrow0, a.K, a.x + (size_t)s * a.K, a.ldx, a.M, c0, c1, acc);
  stash<TT, R>(red, warp, acc);
  __syncthreads();

  const int n0 = tile * RW;
  // shard partial P_s[row][m]: the shard's k-ranges folded in order
  auto shard_partial = [&](int slocal, int row, int m) {
    float v = red[((size_t)(slocal * ks) * RW + row) * MP + m];
    for (int j = 1; j < ks; ++j) v += red[((size_t)(slocal * ks + j) * RW + row) * MP + m];
    if (sizeof(WT) == 1)  // __fmul_rn: never contracted into the fold's adds
      v = __fmul_rn(v, reinterpret_cast<const float*>(a.w + (size_t)(cs * spc + slocal) * a.shard_stride +
                                                      a.scales_offset)[n0 + row]);
    return v;
  };

  if (a.fold == FOLD_IN_CTA) {  // gridDim.y == 1: every shard is here
    for (int i = threadIdx.x; i < RW * a.M; i += blockDim.x) {
      const int m = i / RW, row = i % RW;
      float v = shard_partial(0, row, m);
      for (int j = 1; j < spc; ++j) v += shard_partial(j, row, m);
      const size_t o = (size_t)m * a.ldy + n0 + row;
      if (a.residual) v += __bfloat162float(a.residual[o]);
      reinterpret_cast<uint16_t*>(a.y)[o] = f2bf(v);
    }
    return;
  }
  // write this CTA's shard partials: partials[s][m][n]
  for (int i = threadIdx.x; i < RW * a.M * spc; i += blockDim.x) {
    const int sl2 = i / (RW * a.M), rem = i % (RW * a.M);
    const int m = rem / RW, row = rem % RW;
    a.partials[((size_t)(cs * spc + sl2) * a.pM + m) * a.N + n0 + row] = shard_partial(sl2, row, m);
  }
  if (a.fold == FOLD_NONE) return;
  // last-arriving CTA of this tile folds all t partials in shard order
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(&a.tickets[tile], 1u);
    s_last = (old == gridDim.y - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < RW * a.M; i += blockDim.x) {
    const int m = i / RW, row = i % RW;
    const size_t pn = (size_t)m * a.N + n0 + row;
    float v = __ldcg(a.partials + pn);
    for (int j = 1; j < a.t; ++j) v += __ldcg(a.partials + (size_t)j * a.pM * a.N + pn);
    const size_t o = (size_t)m * a.ldy + n0 + row;
    if (a.residual) v += __bfloat162float(a.residual[o]);
    reinterpret_cast<uint16_t*>(a.y)[o] = f2bf(v);
  }
  if (threadIdx.x == 0) a.tickets[tile] = 0u;
}

// ---------------------------------------------------------------- host dispatch

constexpr int kTargetCTAs = 2 * 152;  // two CTAs per SM on a 152-SM GB300 (fixed: results
                                      // must not depend on the device the call runs on)

int colpar_R(int rows, bool swiglu) {
  if (rows % 32 == 0) return 4;
  if (rows % 16 == 0) return 2;
  return swiglu ? 0 : (rows % 8 == 0 ? 1 : 0);
}

RowparPlan rowpar_plan(int N, int t) {
  RowparPlan p{0, 1, 0};
  p.R = N % 32 == 0 ? 4 : (N % 16 == 0 ? 2 : (N % 8 == 0 ? 1 : 0));
  if (p.R == 0) return p;
  p.tiles = N / (8 * p.R);
  while (p.tiles * p.S < kTargetCTAs && p.S < t) p.S *= 2;
  return p;
}

template <typename K>
static cudaError_t prep_smem(K kernel, size_t smem) {
  if (smem > 48 * 1024)
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return cudaSuccess;
}

template <typename WT, int TT, int R>
static cudaError_t colpar_go(const ColparArgs& a, cudaStream_t st) {
  constexpr int U = TT == 1 ? 4 : 2;
  const size_t smem = (size_t)kWarps * 8 * R * 16 * TT * sizeof(float);
  auto k = colpar_kernel<WT, TT, R, U>;
  cudaError_t e = prep_smem(k, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(a.rows / (8 * R) * a.t);
  k<<<grid, kWarps * 32, smem, st>>>(a);
  note_launch();
  return cudaGetLastError();
}

template <typename WT, int TT, int R>
static cudaError_t rowpar_go(const RowparArgs& a, const RowparPlan& p, cudaStream_t st) {
  constexpr int U = TT == 1 ? 4 : 2;
  const size_t smem = (size_t)kWarps * 8 * R * 16 * TT * sizeof(float);
  auto k = rowpar_kernel<WT, TT, R, U>;
  cudaError_t e = prep_smem(k, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.tiles, (unsigned)p.S);
  k<<<grid, kWarps * 32, smem, st>>>(a);
  note_launch();
  return cudaGetLastError();
}

template <typename WT, int TT>
static cudaError_t colpar_R_dispatch(const ColparArgs& a, int R, cudaStream_t st) {
  switch (R) {
    case 4: return colpar_go<WT, TT, 4>(a, st);
    case 2: return colpar_go<WT, TT, 2>(a, st);
    case 1: return colpar_go<WT, TT, 1>(a, st);
  }
  return cudaErrorInvalidValue;
}

template <typename WT, int TT>
static cudaError_t rowpar_R_dispatch(const RowparArgs& a, const RowparPlan& p, cudaStream_t st) {
  switch (p.R) {
    case 4: return rowpar_go<WT, TT, 4>(a, p, st);
    case 2: return rowpar_go<WT, TT, 2>(a, p, st);
    case 1: return rowpar_go<WT, TT, 1>(a, p, st);
  }
  return cudaErrorInvalidValue;
}

static int tt_for(int M) { return M <= 16 ? 1 : (M <= 32 ? 2 : 4); }

template <typename WT>
static cudaError_t colpar_tt(const ColparArgs& a, int R, cudaStream_t st) {
  switch (tt_for(a.M)) {
    case 1: return colpar_R_dispatch<WT, 1>(a, R, st);
    case 2: return colpar_R_dispatch<WT, 2>(a, R, st);
    default: return colpar_R_dispatch<WT, 4>(a, R, st);
  }
}

template <typename WT>
static cudaError_t rowpar_tt(const RowparArgs& a, const RowparPlan& p, cudaStream_t st) {
  switch (tt_for(a.M)) {
    case 1: return rowpar_R_dispatch<WT, 1>(a, p, st);
    case 2: return rowpar_R_dispatch<WT, 2>(a, p, st);
    default: return rowpar_R_dispatch<WT, 4>(a, p, st);
  }
}

cudaError_t launch_colpar(const ColparArgs& a, bool fp8, cudaStream_t st) {
  const int R = colpar_R(a.rows, a.mode == COLPAR_SWIGLU);
  if (R == 0 || a.M <= 0 || a.M > kSkinnyMaxM) return cudaErrorInvalidValue;
  return fp8 ? colpar_tt<uint8_t>(a, R, st) : colpar_tt<uint16_t>(a, R, st);
}

cudaError_t launch_rowpar(const RowparArgs& a, bool fp8, const RowparPlan& p, cudaStream_t st) {
  if (p.R == 0 || a.M <= 0 || a.M > kSkinnyMaxM) return cudaErrorInvalidValue;
  return fp8 ? rowpar_tt<uint8_t>(a, p, st) : rowpar_tt<uint16_t>(a, p, st);
}

}  // namespace tpx
