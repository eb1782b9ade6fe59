// TMA-fed decode kernel for e4m3 weights: the column-parallel half (QKV, gate/up + SwiGLU)
// and the row-parallel half (o_proj, down + the shard fold) of a Megatron block
// ("The Tensor-Parallel Shard Group", scalablesystem.dev; "Tensor Parallelism
// (Megatron-Style)", arunshar.com) at decode token counts, where every weight byte is read
// once and the pass is HBM-bound.
//
// Design (GB300):
//  * Work units are (shard, 128-row tile, 128-k stage), tile-major inside a shard; the
//    units are split evenly over the CTAs (two per SM), each taking a contiguous run.
//  * A producer warp keeps a ring of TMA stages full: the stage's 128 x 128 e4m3 weight box
//    (128-byte swizzle) and the matching [tokens][128] bf16 activation boxes.  The first
//    stages' weights are requested before the kernel waits for the previous launch
//    (programmatic dependent launch); activations only after.
//  * Four consumer warps own 32 weight rows each.  ldmatrix hands every lane four codes of a
//    row per 16-byte piece; they are widened to bf16 exactly in registers and multiplied on
//    the tensor cores (mma.sync m16n8k16, tokens on the M side).  The activation operand uses
//    the same k order, read once per stage and reused for the warp's four row groups.
//  * A (shard, tile) that a CTA holds whole is finished by its warps directly.  One split
//    across CTAs leaves one fp32 piece per CTA; the CTA that brings the last piece sums the
//    pieces in k order and finishes it.
//  * Finishing applies the per-row scales, then: the SwiGLU or bf16 output (column-parallel);
//    or the shard partial, and by ticket the left fold of the t partials in shard order plus
//    the residual (row-parallel), the same operations as the unfused partials + fold path.
// Every sum has a fixed order for a given GPU (the split follows the SM count).
#include <cuda.h>

#include "common.cuh"
#include "ring.h"
#include "skinny.h"
#include "tc.h"
#include "tc_ptx.cuh"

namespace tpx {

namespace {

constexpr int kRows = 128;  // weight rows per tile
constexpr int kKS = 128;    // k per stage (one e4m3 box row)
constexpr int kCW = 4;      // consumer warps, 32 rows each
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kCtasPerSm = 2;

template <int TT>  // TT tiles of 16 tokens
struct RCfg {
  static constexpr int WB = kRows * kKS;      // weight bytes of a stage
  static constexpr int XBOX = 16 * TT * 128;  // one [16 TT tokens][64 k] bf16 box
  static constexpr int ST = WB + 2 * XBOX;
  static constexpr int NS = (100 * 1024) / ST;
  static constexpr size_t SMEM = 1024 + (size_t)NS * ST + (2 * NS + 1) * 8;
  static constexpr int PF = 16 * TT;  // piece floats per lane
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ long long split_at(long long U, int nct, int i) { return U * i / nct; }
// the CTA whose run holds unit v
__device__ __forceinline__ int owner_of(long long U, int nct, long long v) {
  return (int)(((v + 1) * nct + U - 1) / U) - 1;
}

// Calls f(v) for the first unit v of every piece of the tile whose units are [ub, ub + n),
// in k order: ub, then each CTA boundary inside.
template <class F>
__device__ __forceinline__ void for_pieces(long long U, int nct, long long ub, int n, F f) {
  f(ub);
  int i = owner_of(U, nct, ub) + 1;
  long long prev = ub;
  for (; i < nct; ++i) {
    const long long b = split_at(U, nct, i);
    if (b >= ub + n) break;
    if (b != prev) {
      f(b);
      prev = b;
    }
  }
}

template <int TT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    ring_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, RingArgs a) {
  using C = RCfg<TT>;
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + (size_t)C::NS * C::ST);  // full[NS], empty[NS], consumers
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = tc::smem_u32(bars), empty0 = full0 + 8 * C::NS, cbar = empty0 + 8 * C::NS;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      tc::mbar_init(full0 + 8 * i, 1);
      tc::mbar_init(empty0 + 8 * i, kCW);
    }
    tc::mbar_init(cbar, kCW);
    tc::fence_mbar_init();
  }
  __syncthreads();
  tc::griddep_launch_dependents();
  const int tiles = a.rows / kRows, nks = a.K / kKS;
  const long long U = (long long)a.t * tiles * nks;
  const int nct = gridDim.x;
  const long long u0 = split_at(U, nct, blockIdx.x), u1 = split_at(U, nct, blockIdx.x + 1);
  if (u0 >= u1) {
    tc::griddep_wait();  // this grid ends after the one before it (the next launch relies on that)
    return;
  }
  const int nu = (int)(u1 - u0);
  auto unit_of = [&](int k) -> long long { return u0 + k; };

  if (warp == kCW) {  // producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmW);
      tc::tma_prefetch_desc(&tmX);
      const uint64_t pol = tc::l2_evict_first();  // weights stream through once
      auto load_w = [&](int k) {
        const long long u = unit_of(k);
        const int item = (int)(u / nks), ks = (int)(u % nks), s = item / tiles, rt = item % tiles;
        const uint32_t fb = full0 + 8 * (k % C::NS);
        tc::mbar_arrive_expect_tx(fb, C::ST);
        tc::tma_load_3d_hint(tc::smem_u32(ring + (size_t)(k % C::NS) * C::ST), &tmW, ks * kKS, rt * kRows, s, fb,
                             pol);
      };
      auto load_x = [&](int k) {
        const long long u = unit_of(k);
        const int item = (int)(u / nks), ks = (int)(u % nks), s = item / tiles;
        const uint32_t fb = full0 + 8 * (k % C::NS);
        const int col = (a.rowpar ? s * a.K : 0) + ks * kKS;
        const uint32_t dst = tc::smem_u32(ring + (size_t)(k % C::NS) * C::ST + C::WB);
        tc::tma_load_2d(dst, &tmX, col, 0, fb);
        tc::tma_load_2d(dst + C::XBOX, &tmX, col + 64, 0, fb);
      };
      const int pre = nu < C::NS ? nu : C::NS;
      for (int k = 0; k < pre; ++k) load_w(k);  // weights do not depend on the previous launch
      tc::griddep_wait();
      for (int k = 0; k < pre; ++k) load_x(k);
      for (int k = C::NS; k < nu; ++k) {
        if (!tc::mbar_wait(empty0 + 8 * (k % C::NS), ((k / C::NS) - 1) & 1)) {
          atomicExch(a.err, 51u);
          break;
        }
        load_w(k);
        load_x(k);
      }
    }
    return;
  }

  // consumers: warp w owns rows 32w .. 32w+31 of every tile, as four groups of 8
  tc::griddep_wait();  // before any read or write of what the previous launch touches
  const int tid = threadIdx.x, g = lane >> 2, q = lane & 3;
  uint32_t cph = 0;
  auto csync = [&]() -> bool {  // the consumer warps meet (bounded wait)
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(cbar);
    const bool ok = tc::mbar_wait(cbar, cph);
    cph ^= 1u;
    __syncwarp();
    if (!ok && lane == 0) atomicExch(a.err, 53u);
    return ok;
  };

  // Output of rows 32w.. of tile (s, rt) from its full k sum v (this warp's fragments); scl is
  // this lane's row scale (row 32w + lane).  Column-parallel: the SwiGLU or bf16 output.
  // Row-parallel: the shard partial P_s = scale . sum (the fold follows by ticket).
  auto emit = [&](int s, int rt, float (&v)[TT][4][4], float scl) {
    const int r0 = rt * kRows + 32 * warp;
    if (!a.rowpar && a.mode == COLPAR_SWIGLU) {  // groups (0, 1) and (2, 3) are [8 gate | 8 up] pairs
#pragma unroll
      for (int p = 0; p < 2; ++p) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float sg = __shfl_sync(0xffffffffu, scl, 16 * p + 2 * q + e);
          const float su = __shfl_sync(0xffffffffu, scl, 16 * p + 8 + 2 * q + e);
          const int f = (r0 + 16 * p) / 2 + 2 * q + e;
#pragma unroll
          for (int tt = 0; tt < TT; ++tt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int m = 16 * tt + g + 8 * hh;
              if (m < a.M) {
                const float gv = __fmul_rn(v[tt][2 * p][2 * hh + e], sg);
                const float uv = __fmul_rn(v[tt][2 * p + 1][2 * hh + e], su);
                reinterpret_cast<uint16_t*>(a.out)[(size_t)m * a.ldo + (size_t)s * (a.rows / 2) + f] =
                    f2bf(silu_f(gv) * uv);
              }
            }
        }
      }
      return;
    }
#pragma unroll
    for (int ng = 0; ng < 4; ++ng)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = r0 + 8 * ng + 2 * q + e;
        const float scr = __shfl_sync(0xffffffffu, scl, 8 * ng + 2 * q + e);
#pragma unroll
        for (int tt = 0; tt < TT; ++tt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int m = 16 * tt + g + 8 * hh;
            if (m >= a.M) continue;
            const float val = __fmul_rn(v[tt][ng][2 * hh + e], scr);
            if (a.rowpar)
              a.partials[((size_t)s * a.pM + m) * a.rows + r] = val;
            else
              reinterpret_cast<uint16_t*>(a.out)[(size_t)m * a.ldo + (size_t)s * a.rows + r] = f2bf(val);
          }
      }
  };
  auto scale_of = [&](int s, int rt) {  // this lane's row scale of tile (s, rt)
    return reinterpret_cast<const float*>(a.w + (size_t)s * a.shard_stride + a.scales_offset)[rt * kRows + 32 * warp +
                                                                                                lane];
  };
  // Row-tile folds this CTA wins (it brought the tile's last shard partial), done after its
  // stream; s_nmerge says whether it brought a split tile's last piece.  Thread 0 writes.
  constexpr int kMaxFolds = 64;
  __shared__ int s_nmerge, s_nfold, s_fold[kMaxFolds];
  if (tid == 0) s_nmerge = s_nfold = 0;
  // After this CTA wrote shard partial (s, rt): count it in (one thread, after the warps met).
  auto count_partial = [&](int rt) -> bool {
    if (!a.rowpar || a.mode != FOLD_TICKET) return true;
    if (!csync()) return false;  // every warp's partial writes precede the fence below
    if (tid == 0) {
      __threadfence();
      unsigned* ticket = a.counters + (size_t)a.t * tiles + rt;
      if (atomicAdd(ticket, 1u) + 1u == (unsigned)a.t) {
        *ticket = 0u;
        if (s_nfold < kMaxFolds)
          s_fold[s_nfold++] = rt;
        else
          atomicExch(a.err, 54u);  // the host keeps a launch's tiles per CTA below the list size
      }
    }
    return true;
  };

  float acc[TT][4][4];
  float scl = 0.f;  // the row scale of lane's row of the current tile
  int seg_k0 = 0;   // local index of the current piece's first unit
  if (!csync()) return;  // the list counts are set
  for (int k = 0; k < nu; ++k) {
    const long long u = unit_of(k);
    const int item = (int)(u / nks), ks = (int)(u % nks), s = item / tiles, rt = item % tiles;
    if (k == 0 || ks == 0) {
#pragma unroll
      for (int tt = 0; tt < TT; ++tt)
#pragma unroll
        for (int ng = 0; ng < 4; ++ng) acc[tt][ng][0] = acc[tt][ng][1] = acc[tt][ng][2] = acc[tt][ng][3] = 0.f;
      seg_k0 = k;
      scl = scale_of(s, rt);
    }
    const int st = k % C::NS;
    if (!tc::mbar_wait(full0 + 8 * st, (k / C::NS) & 1)) {
      if (lane == 0) atomicExch(a.err, 52u);
      return;
    }
    const uint32_t wst = tc::smem_u32(ring + (size_t)st * C::ST), xst = wst + C::WB;
#pragma unroll
    for (int c = 0; c < 2; ++c) {  // two 64-k chunks of the stage
      // activations: for MMA j, tokens g and g + 8 at k = 64c + 16j + 4q .. +3
      uint2 xa[TT][4][2];
#pragma unroll
      for (int tt = 0; tt < TT; ++tt)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int row = 16 * tt + g + 8 * hh;
            xa[tt][j][hh] = lds64(xst + c * C::XBOX + row * 128 + ((((2 * j + (q >> 1)) ^ (row & 7))) << 4) +
                                  8 * (q & 1));
          }
#pragma unroll
      for (int ng = 0; ng < 4; ++ng) {
        // weights: matrix j = 16-byte piece 4c + j of rows 32w + 8ng + (0..7); lane (g, q)
        // receives codes 64c + 16j + 4q .. +3 of row g
        uint32_t wr[4];
        const int r = 32 * warp + 8 * ng + (lane & 7);
        ldsm_x4(wst + r * 128 + ((((4 * c + (lane >> 3)) ^ (r & 7))) << 4), wr[0], wr[1], wr[2], wr[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t b0 = e4m3x2_to_bf16x2((uint16_t)(wr[j] & 0xFFFFu));  // k 4q, 4q+1 of the 16
          const uint32_t b1 = e4m3x2_to_bf16x2((uint16_t)(wr[j] >> 16));      // k 4q+2, 4q+3
#pragma unroll
          for (int tt = 0; tt < TT; ++tt)
            mma_bf16_16816(acc[tt][ng], xa[tt][j][0].x, xa[tt][j][1].x, xa[tt][j][0].y, xa[tt][j][1].y, b0, b1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(empty0 + 8 * st);  // the stage goes back to the producer

    if (ks + 1 < nks && k + 1 < nu) continue;
    // this CTA's part of tile (s, rt) ends here
    const long long pu = unit_of(seg_k0);  // the part's first unit
    if (pu % nks == 0 && ks + 1 == nks) {  // the whole tile
      emit(s, rt, acc, scl);
      if (!count_partial(rt)) return;
      continue;
    }
    // a piece: stored in this CTA's slot (0: the piece that starts its run, 1: the one that ends it)
    const int end = pu == u0 ? 0 : 1;
    float* slot = a.pieces + (((size_t)blockIdx.x * 2 + end) * kCW + warp) * 32 * C::PF + lane * C::PF;
#pragma unroll
    for (int tt = 0; tt < TT; ++tt)
#pragma unroll
      for (int ng = 0; ng < 4; ++ng)
        *reinterpret_cast<float4*>(slot + (tt * 4 + ng) * 4) =
            make_float4(acc[tt][ng][0], acc[tt][ng][1], acc[tt][ng][2], acc[tt][ng][3]);
    if (!csync()) return;  // every warp's piece writes precede the fence below
    if (tid == 0) {
      __threadfence();
      int npc = 0;
      for_pieces(U, nct, (long long)item * nks, nks, [&](long long) { ++npc; });
      s_nmerge = 0;
      if (atomicAdd(a.counters + item, 1u) + 1u == (unsigned)npc) {
        a.counters[item] = 0u;
        s_nmerge = 1;
      }
    }
    if (!csync()) return;
    if (s_nmerge) {  // this CTA brought the last piece: sum all pieces in k order, then emit
      __threadfence();
      float v[TT][4][4];
#pragma unroll
      for (int tt = 0; tt < TT; ++tt)
#pragma unroll
        for (int ng = 0; ng < 4; ++ng) v[tt][ng][0] = v[tt][ng][1] = v[tt][ng][2] = v[tt][ng][3] = 0.f;
      for_pieces(U, nct, (long long)item * nks, nks, [&](long long vb) {
        const int o = owner_of(U, nct, vb);
        const int e2 = split_at(U, nct, o) == vb ? 0 : 1;
        const float* ps = a.pieces + (((size_t)o * 2 + e2) * kCW + warp) * 32 * C::PF + lane * C::PF;
#pragma unroll
        for (int tt = 0; tt < TT; ++tt)
#pragma unroll
          for (int ng = 0; ng < 4; ++ng) {
            const float4 f = __ldcg(reinterpret_cast<const float4*>(ps + (tt * 4 + ng) * 4));
            v[tt][ng][0] += f.x;
            v[tt][ng][1] += f.y;
            v[tt][ng][2] += f.z;
            v[tt][ng][3] += f.w;
          }
      });
      emit(s, rt, v, scl);
      if (!count_partial(rt)) return;
    }
    if (!csync()) return;  // s_nmerge is read by every warp before it is written again
  }

  // After the stream: the folds this CTA won (the t shard partials of a row tile, in shard
  // order, plus the residual).
  if (!csync()) return;  // the fold list is complete
  const int nfold = s_nfold;
  for (int i = 0; i < nfold; ++i) {
    // thread -> 4 consecutive rows (float4 over the partials' rows) x every 4th token, two tokens
    // (2 x t loads) in flight at a time; the t shard partials summed in shard order + residual
    const int rt = s_fold[i], rg = tid & 31, n = rt * kRows + 4 * rg;
    __threadfence();
    const size_t sstride = (size_t)a.pM * a.rows;
    for (int m0 = tid >> 5; m0 < a.M; m0 += 8) {
      float4 pv[2][8];
      uint2 rv[2];
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        const int m = m0 + 4 * mm < a.M ? m0 + 4 * mm : m0;
        const float* p = a.partials + (size_t)m * a.rows + n;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          pv[mm][j] = j < a.t ? __ldcg(reinterpret_cast<const float4*>(p + j * sstride)) : make_float4(0, 0, 0, 0);
        rv[mm] = a.residual ? *reinterpret_cast<const uint2*>(a.residual + (size_t)m * a.ldy + n) : make_uint2(0, 0);
      }
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        const int m = m0 + 4 * mm;
        if (m >= a.M) break;
        float4 f = pv[mm][0];
#pragma unroll
        for (int j = 1; j < 8; ++j)
          if (j < a.t) {
            f.x += pv[mm][j].x;
            f.y += pv[mm][j].y;
            f.z += pv[mm][j].z;
            f.w += pv[mm][j].w;
          }
        if (a.residual) {
          f.x += __uint_as_float(rv[mm].x << 16);
          f.y += __uint_as_float(rv[mm].x & 0xFFFF0000u);
          f.z += __uint_as_float(rv[mm].y << 16);
          f.w += __uint_as_float(rv[mm].y & 0xFFFF0000u);
        }
        uint2 o;
        o.x = (uint32_t)f2bf(f.x) | ((uint32_t)f2bf(f.y) << 16);
        o.y = (uint32_t)f2bf(f.z) | ((uint32_t)f2bf(f.w) << 16);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.y) + (size_t)m * a.ldy + n) = o;
      }
    }
  }
}

int sm_count_here() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

bool ring_supported(int rows, int K, int M, int t) {
  if (rows % kRows != 0 || K % kKS != 0 || K <= 0 || rows <= 0 || M < 1 || M > kRingMaxM || t < 1 || t > 8)
    return false;
  // tiles a CTA can finish: its units / stages per tile, + 2 partly held; the fold list holds 64
  const long long U = (long long)t * (rows / kRows) * (K / kKS), nct = (long long)sm_count_here() * kCtasPerSm;
  return (U + nct - 1) / nct / (K / kKS) + 2 <= 64;
}

size_t ring_pieces_bytes(int M) {
  const int TT = M <= 16 ? 1 : 2;
  return (size_t)sm_count_here() * kCtasPerSm * 2 * kCW * 32 * 16 * TT * sizeof(float);
}

size_t ring_counter_words(int rows, int t, bool rowpar) {
  return (size_t)t * (rows / kRows) + (rowpar ? (size_t)(rows / kRows) : 0);
}

cudaError_t launch_ring(const RingArgs& a, cudaStream_t st, bool pdl) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int TT = a.M <= 16 ? 1 : 2;
  CUtensorMap tmW, tmX;
  {  // weights: [t][rows][K] bytes, boxes of 128 rows x 128 codes
    const cuuint64_t dims[3] = {(cuuint64_t)a.K, (cuuint64_t)a.rows, (cuuint64_t)a.t};
    const cuuint64_t strides[2] = {(cuuint64_t)a.K, (cuuint64_t)a.shard_stride};
    const cuuint32_t box[3] = {(cuuint32_t)kKS, (cuuint32_t)kRows, 1}, es[3] = {1, 1, 1};
    if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.w), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {  // activations: [M][ldx] bf16, boxes of 16 TT tokens x 64 k (tokens past M read zero)
    const cuuint64_t cols = (cuuint64_t)(a.rowpar ? a.K * a.t : a.K);
    const cuuint64_t dims[2] = {cols, (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {(cuuint64_t)a.ldx * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(16 * TT)}, es[2] = {1, 1};
    if (enc(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(a.x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int grid = sm_count_here() * kCtasPerSm;
  auto go = [&](auto kernel, size_t smem) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kernel, tmW, tmX, a);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
  };
  if (TT == 1) return go(ring_kernel<1>, RCfg<1>::SMEM);
  return go(ring_kernel<2>, RCfg<2>::SMEM);
}

}  // namespace tpx
