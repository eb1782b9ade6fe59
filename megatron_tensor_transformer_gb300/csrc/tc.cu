// tcgen05 weight-streaming GEMM for the column- and row-parallel linears.
//
// D[weight rows, tokens] = W_s[rows, K] * X[tokens, K]^T for one shard s: the weights are
// the MMA's A operand (128 rows per tile, K-major) and the tokens its B operand (BN per
// tile, K-major), so one kernel serves decode (BN = 16..64 tokens, weight-streaming, HBM
// bound) and prefill (BN = 256 token tiles, tensor bound).  The column split of the first
// linear and the row split of the second ("ColumnParallelLinear" / "RowParallelLinear",
// scalablesystem.dev, "The Tensor-Parallel Shard Group") only change which shard buffer
// and which activation columns a tile reads, and what the epilogue does:
//   colpar:      store D (or silu(g) * u for interleaved gate/up rows) for shard s;
//   rowpar:      per-(tile, shard) partial P_s for the separate shard fold (unfused path);
//   rowpar-chain (fused): all shards' k-blocks accumulate into one TMEM tile in shard
//                order, + residual (Z = sum_k Z_k with no partials round trip).
//
// Structure: persistent CTAs (one per SM), warp roles:
//   warps 0-3  epilogue: TMEM -> registers -> global (lane i of warp w = tile row 32w+i)
//   warp 4     producer: one thread issues TMA tensor copies into a ring of smem stages
//   warp 5     MMA: one thread issues tcgen05.mma (4 per 64-wide k-block) into a
//              double-buffered TMEM accumulator; tcgen05.commit frees stages / hands off
// Every wait is an mbarrier poll bounded in time; on expiry the kernel records an error
// word, drains what it issued, frees its TMEM and returns.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "tc.h"
#include "tc_ptx.cuh"

namespace tpx {
using namespace tc;

static __device__ unsigned g_tc_error;

constexpr int BM = 128, BK = 64;
constexpr int kProducerWarp = 4, kMmaWarp = 5;

template <int BN, bool FP8 = false, bool X8 = false>
struct TcCfg {
  static constexpr int kKB = X8 ? 128 : BK;  // k per block: 128 bytes of a K-major row either way
  static constexpr int kABytes = BM * BK * 2;            // bf16 A tile the MMA reads (SW128)
  static constexpr int kAqBytes = FP8 ? BM * BK : 0;     // e4m3 A tile as TMA brings it
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes + kAqBytes;
  static constexpr int kConvWarps = FP8 ? 8 : 0;        // converter warps for e4m3 weights
  static constexpr int kThreadsT = 192 + 32 * kConvWarps;
  static constexpr int kStages = (200 * 1024) / kStageBytes > 8 ? 8 : (200 * 1024) / kStageBytes;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int kBarBytes = 1024;  // mbarriers, flags and the stream-K share table
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kBarBytes;
};

struct Geo {  // item geometry shared by the three roles
  int n_rt, n_tt, n_items, kb_per_shard, nkb;
};

__device__ __forceinline__ Geo make_geo(const TcArgs& a, int BN, int KB) {
  Geo g;
  g.n_rt = a.rows / BM;
  g.n_tt = (a.M + BN - 1) / BN;
  g.kb_per_shard = a.K / KB;
  if (a.mode == TC_ROWPAR_CHAIN) {
    g.n_items = g.n_rt * g.n_tt;
    g.nkb = g.kb_per_shard * a.t;
  } else {
    g.n_items = g.n_rt * g.n_tt * a.t;
    g.nkb = g.kb_per_shard;
  }
  return g;
}

// item -> (shard, row tile, token tile).  Column-parallel items walk token tiles fastest (a
// weight tile is reused from L2 by concurrent CTAs); row-parallel items walk shards fastest
// (the t partials of a tile finish close together).
__device__ __forceinline__ void decode_item(const TcArgs& a, const Geo& g, int i, int& s, int& rt, int& tt) {
  if (a.mode == TC_ROWPAR_CHAIN) {
    s = 0;
    tt = i % g.n_tt;
    rt = i / g.n_tt;
  } else if (a.mode == TC_ROWPAR_SHARD) {
    s = i % a.t;
    tt = (i / a.t) % g.n_tt;
    rt = i / (a.t * g.n_tt);
  } else {
    tt = i % g.n_tt;
    rt = (i / g.n_tt) % g.n_rt;
    s = i / (g.n_tt * g.n_rt);
  }
}

// Work of one CTA: whole items strided over the grid, or (stream-K) an equal contiguous
// share of the flattened (item, k-block) space, cut into segments at item boundaries.
struct Seg {
  int item, kb_lo, kb_hi;
};

struct SegIter {
  bool sk;
  int nkb, n_items, G, item;
  long long cur, end;
  __device__ SegIter(bool streamk, const Geo& g)
      : sk(streamk), nkb(g.nkb), n_items(g.n_items), G(gridDim.x), item(blockIdx.x), cur(0), end(0) {
    if (sk) {
      const long long total = (long long)n_items * nkb;
      cur = total * blockIdx.x / G;
      end = total * (blockIdx.x + 1) / G;
    }
  }
  __device__ bool next(Seg& sg) {
    if (!sk) {
      if (item >= n_items) return false;
      sg = {item, 0, nkb};
      item += G;
      return true;
    }
    if (cur >= end) return false;
    sg.item = (int)(cur / nkb);
    sg.kb_lo = (int)(cur % nkb);
    const long long rem = end - cur;
    sg.kb_hi = rem < (long long)(nkb - sg.kb_lo) ? sg.kb_lo + (int)rem : nkb;
    cur += sg.kb_hi - sg.kb_lo;
    return true;
  }
};

// Stream-K share boundaries: shares[c] = first flattened k-block of CTA c (shares[G] = total),
// precomputed once per CTA in shared memory.  CTA owning flattened k-block x:
__device__ __forceinline__ int share_owner(const uint32_t* shares, uint32_t total, int G, uint32_t x) {
  int c = (int)((unsigned long long)x * G / total);
  while (c > 0 && shares[c] > x) --c;
  while (c + 1 < G && shares[c + 1] <= x) ++c;
  return c;
}

__device__ __forceinline__ void raise_error(unsigned code, volatile int* abort_flag) {
  atomicExch(&g_tc_error, code);
  *abort_flag = 1;
}

// e4m3 weights (streamed as e4m3, or widened to bf16 beforehand): the output channel's fp32
// scale (row p of shard s); 1 for bf16 weights.
__device__ __forceinline__ float row_scale(const TcArgs& a, int s, int p) {
  return a.scales ? a.scales[(size_t)s * a.scales_stride + p] : 1.f;
}
// FP8 x FP8: token m's activation scale (1 otherwise, and past the last token).
__device__ __forceinline__ float tok_scale(const TcArgs& a, int m) {
  return (a.tok_scales && m < a.M) ? a.tok_scales[m] : 1.f;
}

// One 16-column chunk of the accumulator for tile row p (of shard s), tokens mf..mf+15.
template <int BN>
__device__ __forceinline__ void epilogue_chunk(const TcArgs& a, int s, int p, int mf, const float (&vin)[16]) {
  float v[16];
  const float sc = row_scale(a, s, p);
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = vin[j] * sc;
  if (a.tok_scales) {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] *= tok_scale(a, mf + j);
  }
  if (a.mode == TC_COLPAR_SWIGLU) {
    // rows come as [8 gate | 8 up] blocks: the up value of row p sits 8 lanes further on
    float u[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) u[j] = __shfl_down_sync(0xffffffffu, v[j], 8);
    if ((p & 15) < 8) {
      const int f = s * (a.rows / 2) + (p >> 4) * 8 + (p & 7);
      uint16_t* o = reinterpret_cast<uint16_t*>(a.out);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (mf + j < a.M) o[(size_t)(mf + j) * a.ldo + f] = f2bf(silu_f(v[j]) * u[j]);
    }
  } else if (a.mode == TC_COLPAR_BF16 || a.mode == TC_COLPAR_F32) {
    const size_t col = (size_t)s * a.rows + p;
    if (a.ncols && col >= (size_t)a.ncols) return;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (mf + j >= a.M) break;
      const size_t o = (size_t)(mf + j) * a.ldo + col;
      if (a.mode == TC_COLPAR_F32)
        reinterpret_cast<float*>(a.out)[o] = v[j];
      else
        reinterpret_cast<uint16_t*>(a.out)[o] = f2bf(v[j]);
    }
  } else if (a.mode == TC_ROWPAR_SHARD) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (mf + j < a.M) a.partials[((size_t)s * a.pM + mf + j) * a.rows + p] = v[j];
  } else {  // TC_ROWPAR_CHAIN: the whole fold is in v already
    // all residual loads first, then the stores: y may alias the residual, so interleaving
    // them would cost one memory round trip per token
    float rv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      rv[j] = (a.residual && mf + j < a.M) ? __bfloat162float(a.residual[(size_t)(mf + j) * a.ldy + p]) : 0.f;
    uint16_t yb[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      yb[j] = f2bf(v[j] + rv[j]);
      if (mf + j < a.M) reinterpret_cast<uint16_t*>(a.y)[(size_t)(mf + j) * a.ldy + p] = yb[j];
    }
    if (a.norm_ss) {
      // the warp's 32 rows of the stored values, per token: a fixed shuffle tree
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float e = __uint_as_float((uint32_t)yb[j] << 16);
        float ss = e * e;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((threadIdx.x & 31) == 0 && mf + j < a.M) a.norm_ss[(size_t)(mf + j) * (a.rows / 32) + p / 32] = ss;
      }
    }
  }
}

// Sync of the 128 epilogue threads on an mbarrier (bounded wait).
__device__ __forceinline__ bool epi_sync(uint32_t epi_bar, int& phase, volatile int* abort_flag, unsigned code) {
  mbar_arrive(epi_bar);
  const bool ok = mbar_wait(epi_bar, phase);
  phase ^= 1;
  if (!ok) raise_error(code, abort_flag);
  return ok;
}

// Grid-wide barrier of a cooperative (all CTAs co-resident) launch: bar[0] counts arrivals,
// bar[1] is a generation number that the last arrival bumps.  Bounded wait.
__device__ bool grid_sync(unsigned* bar, volatile int* abort_flag) {
  volatile unsigned* gen = bar + 1;
  const unsigned my = *gen;  // read before arriving: it cannot change until every CTA has arrived
  __threadfence();
  if (atomicAdd(bar, 1u) == gridDim.x - 1) {
    *bar = 0u;
    __threadfence();
    atomicAdd(bar + 1, 1u);
    return true;
  }
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; *gen == my; ++i) {
    if ((i & 255u) == 0 && globaltimer_ns() - t0 > 2000000000ull) {
      raise_error(11, abort_flag);
      return false;
    }
  }
  __threadfence();
  return true;
}

// Emit one output of the item (shard s, row tile rt, token tile tt): `row` is the row inside
// the 128-row tile, `m` the token.  For SwiGLU `v` is the gate and `u` the up value.
__device__ __forceinline__ void emit(const TcArgs& a, int s, int rt, int row, int m, float v, float u) {
  const int p = rt * BM + row;
  if (a.mode == TC_COLPAR_SWIGLU) {
    const int f = s * (a.rows / 2) + (p >> 4) * 8 + (p & 7);
    reinterpret_cast<uint16_t*>(a.out)[(size_t)m * a.ldo + f] = f2bf(silu_f(v) * u);
  } else if (a.mode == TC_COLPAR_BF16 || a.mode == TC_COLPAR_F32) {
    if (a.ncols && (size_t)s * a.rows + p >= (size_t)a.ncols) return;
    const size_t o = (size_t)m * a.ldo + (size_t)s * a.rows + p;
    if (a.mode == TC_COLPAR_F32)
      reinterpret_cast<float*>(a.out)[o] = v;
    else
      reinterpret_cast<uint16_t*>(a.out)[o] = f2bf(v);
  } else if (a.mode == TC_ROWPAR_SHARD) {
    a.partials[((size_t)s * a.pM + m) * a.rows + p] = v;
  } else {
    const size_t o = (size_t)m * a.ldy + p;
    const float r = a.residual ? __bfloat162float(a.residual[o]) : 0.f;
    reinterpret_cast<uint16_t*>(a.y)[o] = f2bf(v + r);
  }
}

// Stream-K fix-up, after the grid barrier.  Every item cut across CTAs is finished by all of
// its piece owners together: owner j of np sums, in piece (k) order, the pieces' values for
// its share of the tile's eight 16-row blocks (staged through the idle pipeline smem) and
// emits those outputs.  One bulk round of loads per piece, spread over the whole grid.
template <int BN>
__device__ bool streamk_fixup(const TcArgs& a, const Geo& g, const uint32_t* shares, float* sacc,
                              uint32_t epi_bar, int& phase, volatile int* abort_flag) {
  const int G = gridDim.x, tid = threadIdx.x;  // 128 epilogue threads
  const uint32_t total = shares[G];
  SegIter segs(true, g);
  Seg sg;
  while (segs.next(sg)) {
    if (sg.kb_lo == 0 && sg.kb_hi == g.nkb) continue;  // whole item: already emitted
    const uint32_t istart = (uint32_t)sg.item * g.nkb;
    const int ca = share_owner(shares, total, G, istart), cb = share_owner(shares, total, G, istart + g.nkb - 1);
    int np = 0, j = -1;
    for (int c = ca; c <= cb; ++c)
      if (shares[c + 1] > shares[c]) {
        if (c == (int)blockIdx.x) j = np;
        ++np;
      }
    const int b0 = j * 8 / np, b1 = (j + 1) * 8 / np;
    if (b0 == b1) continue;
    const int r0 = b0 * 16, nr = (b1 - b0) * 16, n4 = nr * BN / 4;
    // running sums for this thread's float4 slots of the slice ([col][row], rows contiguous),
    // at most 8 slots (32 registers) per pass over the pieces
    constexpr int kSlotsAll = (8 * 16 * BN / 4 + 127) / 128;
    constexpr int kSlots = kSlotsAll > 8 ? 8 : kSlotsAll;
#pragma unroll 1
    for (int k0 = 0; k0 < kSlotsAll; k0 += kSlots) {
      float4 acc[kSlots];
      bool first = true;
#pragma unroll 1
      for (int c = ca; c <= cb; ++c) {
        if (shares[c + 1] == shares[c]) continue;  // empty share
        const int slot = shares[c] < istart ? 1 : 0;
        const float* src = a.pieces + ((size_t)c * 2 + slot) * BN * BM;
#pragma unroll
        for (int k = 0; k < kSlots; ++k) {
          const int e4 = tid + 128 * (k0 + k);
          if (e4 < n4) {
            const int e = e4 * 4, col = e / nr, row = e % nr;
            const float4 w = __ldcg(reinterpret_cast<const float4*>(src + (size_t)col * BM + r0 + row));
            if (first) {
              acc[k] = w;
            } else {
              acc[k].x += w.x; acc[k].y += w.y; acc[k].z += w.z; acc[k].w += w.w;
            }
          }
        }
        first = false;
      }
#pragma unroll
      for (int k = 0; k < kSlots; ++k) {
        const int e4 = tid + 128 * (k0 + k);
        if (e4 < n4) reinterpret_cast<float4*>(sacc)[e4] = acc[k];
      }
    }
    if (!epi_sync(epi_bar, phase, abort_flag, 12)) return false;
    int s, rt, tt;
    decode_item(a, g, sg.item, s, rt, tt);
    const int m0 = tt * BN;
    if (a.mode == TC_COLPAR_SWIGLU) {
      const int nf = nr / 2;  // 8 features per 16-row block
      for (int e = tid; e < nf * BN; e += 128) {
        const int col = e / nf, fl = e % nf, m = m0 + col;
        if (m >= a.M) continue;
        const int grow = (fl >> 3) * 16 + (fl & 7);
        emit(a, s, rt, r0 + grow, m, sacc[col * nr + grow] * row_scale(a, s, rt * BM + r0 + grow) * tok_scale(a, m),
             sacc[col * nr + grow + 8] * row_scale(a, s, rt * BM + r0 + grow + 8) * tok_scale(a, m));
      }
    } else {
      for (int e = tid; e < nr * BN; e += 128) {
        const int col = e / nr, row = e % nr, m = m0 + col;
        if (m < a.M)
          emit(a, s, rt, r0 + row, m, sacc[col * nr + row] * row_scale(a, s, rt * BM + r0 + row) * tok_scale(a, m), 0.f);
      }
    }
    if (!epi_sync(epi_bar, phase, abort_flag, 13)) return false;  // smem reused by the next item
  }
  return true;
}

template <int BN, bool FP8, bool X8 = false>
__global__ void __launch_bounds__(TcCfg<BN, FP8, X8>::kThreadsT, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcArgs a) {
  using C = TcCfg<BN, FP8, X8>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                                   // S x [128 rows x 64] bf16, SW128
  uint8_t* sB = smem + (size_t)S * C::kABytes;          // S x [BN rows x 64] bf16, SW128
  uint8_t* sAq = sB + (size_t)S * C::kBBytes;           // S x [128 rows x 64] e4m3 (FP8 only)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * C::kStageBytes);
  // bars: full[S], empty[S], tfull[2], tempty[2], epi, drain, qfull[S]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * S + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  int* mma_consumed = reinterpret_cast<int*>(tmem_slot + 3);
  uint32_t* shares = tmem_slot + 8;  // [gridDim.x + 1]
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S), tfull0 = smem_u32(bars + 2 * S),
                 tempty0 = smem_u32(bars + 2 * S + 2), epi_bar = smem_u32(bars + 2 * S + 4),
                 drain_bar = smem_u32(bars + 2 * S + 5), qfull0 = smem_u32(bars + 2 * S + 6);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Geo g = make_geo(a, BN, C::kKB);

  // fail fast: after a bounded wait has given up (error word set, cleared by tp_sync), later
  // launches do nothing instead of each waiting out its own timeouts
  __shared__ int s_skip;
  if (threadIdx.x == 0) s_skip = *reinterpret_cast<volatile unsigned*>(&g_tc_error) != 0u;
  __syncthreads();
  if (s_skip) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full0 + 8 * i, 1 + C::kConvWarps);  // + one arrival per converter warp
      mbar_init(empty0 + 8 * i, 1);
      mbar_init(qfull0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, 4);  // one arrival per epilogue warp
    }
    mbar_init(epi_bar, 128);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *last_flag = 0;
    *mma_consumed = 0;
    fence_mbar_init();
  }
  if (a.streamk) {  // one share boundary per thread (gridDim.x + 1 <= blockDim.x)
    const unsigned long long total = (unsigned long long)g.n_items * g.nkb;
    for (int c = threadIdx.x; c <= (int)gridDim.x; c += blockDim.x) shares[c] = (uint32_t)(total * c / gridDim.x);
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  int issued = 0;  // producer: k-blocks issued

  griddep_launch_dependents();
  if (warp == kProducerWarp) {
    if (lane == 0) {
      // The packed weights are not written by the kernel this one may overlap with (under
      // programmatic dependent launch), so the first stages' weight tiles are requested
      // before waiting on it; the activation tiles only after.
      // weights are streamed once: evict them first so L2 keeps activations and scratch
      const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
      int pre = 0, pre_xcol[S], pre_row[S];
      {
        SegIter ps(a.streamk != 0, g);
        Seg q;
        while (pre < S && ps.next(q)) {
          int s, rt, tt;
          decode_item(a, g, q.item, s, rt, tt);
          for (int kb = q.kb_lo; kb < q.kb_hi && pre < S; ++kb) {
            const int ss = a.mode == TC_ROWPAR_CHAIN ? kb / g.kb_per_shard : s;
            const int kk = a.mode == TC_ROWPAR_CHAIN ? kb % g.kb_per_shard : kb;
            pre_xcol[pre] = (a.mode >= TC_ROWPAR_SHARD ? ss * a.K : 0) + kk * C::kKB;
            pre_row[pre] = tt * BN;
            if constexpr (FP8) {  // e4m3 tile to the staging buffer, for the converter warps
              mbar_arrive_expect_tx(qfull0 + 8 * pre, C::kAqBytes);
              tma_load_3d_hint(smem_u32(sAq + (size_t)pre * C::kAqBytes), &tmA, kk * C::kKB, rt * BM, ss,
                               qfull0 + 8 * pre, pol_w);
            } else {
              mbar_expect_tx(full0 + 8 * pre, C::kABytes);  // stage `pre` is fresh: no empty wait
              tma_load_3d_hint(smem_u32(sA + (size_t)pre * C::kABytes), &tmA, kk * C::kKB, rt * BM, ss, full0 + 8 * pre,
                               pol_w);
            }
            ++pre;
          }
        }
      }
      griddep_wait();
      for (int j = 0; j < pre; ++j) {
        mbar_arrive_expect_tx(full0 + 8 * j, C::kBBytes);
        tma_load_2d_hint(smem_u32(sB + (size_t)j * C::kBBytes), &tmB, pre_xcol[j], pre_row[j], full0 + 8 * j, pol_x);
      }
      issued = pre;
      SegIter segs(a.streamk != 0, g);
      Seg sg;
      bool ok = true;
      int seq = 0;
      while (ok && !*abort_flag && segs.next(sg)) {
        int s, rt, tt;
        decode_item(a, g, sg.item, s, rt, tt);
        for (int kb = sg.kb_lo; kb < sg.kb_hi; ++kb) {
          if (seq++ < pre) continue;  // already issued above
          const int st = issued % S;
          if (!mbar_wait(empty0 + 8 * st, ((issued / S) & 1) ^ 1)) {
            raise_error(1, abort_flag);
            ok = false;
            break;
          }
          const int ss = a.mode == TC_ROWPAR_CHAIN ? kb / g.kb_per_shard : s;
          const int kk = a.mode == TC_ROWPAR_CHAIN ? kb % g.kb_per_shard : kb;
          const int xcol = (a.mode >= TC_ROWPAR_SHARD ? ss * a.K : 0) + kk * C::kKB;
          if constexpr (FP8) {
            mbar_arrive_expect_tx(qfull0 + 8 * st, C::kAqBytes);
            tma_load_3d_hint(smem_u32(sAq + (size_t)st * C::kAqBytes), &tmA, kk * C::kKB, rt * BM, ss, qfull0 + 8 * st,
                             pol_w);
            mbar_arrive_expect_tx(full0 + 8 * st, C::kBBytes);
          } else {
            mbar_arrive_expect_tx(full0 + 8 * st, C::kABytes + C::kBBytes);
            tma_load_3d_hint(smem_u32(sA + (size_t)st * C::kABytes), &tmA, kk * C::kKB, rt * BM, ss, full0 + 8 * st,
                             pol_w);
          }
          tma_load_2d_hint(smem_u32(sB + (size_t)st * C::kBBytes), &tmB, xcol, tt * BN, full0 + 8 * st, pol_x);
          ++issued;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = X8 ? idesc_e4m3(BM, BN) : idesc_bf16(BM, BN);
      int consumed = 0, it = 0;
      SegIter segs(a.streamk != 0, g);
      Seg sg;
      while (!*abort_flag && segs.next(sg)) {
        const int acc = it & 1;
        if (!mbar_wait(tempty0 + 8 * acc, ((it >> 1) & 1) ^ 1)) {
          raise_error(2, abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = sg.kb_lo; kb < sg.kb_hi; ++kb) {
          const int st = consumed % S;
          if (!mbar_wait(full0 + 8 * st, (consumed / S) & 1)) {
            raise_error(3, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ab = smem_u32(sA + (size_t)st * C::kABytes), bb = smem_u32(sB + (size_t)st * C::kBBytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 32 bytes of each row per MMA: k16 of bf16, k32 of e4m3
            if constexpr (X8)
              mma_e4m3(d, sw128_desc(ab + 32 * k), sw128_desc(bb + 32 * k), idesc, (kb > sg.kb_lo) || k != 0);
            else
              mma_bf16(d, sw128_desc(ab + 32 * k), sw128_desc(bb + 32 * k), idesc, (kb > sg.kb_lo) || k != 0);
          }
          mma_commit(empty0 + 8 * st);  // the stage is free once these MMAs have read it
          ++consumed;
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);   // accumulator ready for the epilogue
        ++it;
      }
      *mma_consumed = consumed;
      // wait for every MMA this thread issued before the TMEM can be released
      mma_commit(drain_bar);
      if (!mbar_wait(drain_bar, 0)) raise_error(4, abort_flag);
    }
  } else if (warp >= 6) {
    if constexpr (FP8) {
      // converter warps: widen each stage's e4m3 weight tile ([128 rows][64 bytes]) to bf16 in
      // the MMA's 128-byte-swizzled layout (16-byte chunk j of row r goes to chunk j ^ (r & 7)).
      // A unit is one 16-byte e4m3 chunk (row, cc) -> bf16 chunks 2cc, 2cc+1.  Each group of 8
      // lanes takes two adjacent rows x 4 chunks: its 16-byte reads cover 128 distinct bytes
      // mod 128 and so do its writes (rows r, r+1 swizzle by an even and an odd mask), so
      // neither side has bank conflicts.
      constexpr int kRowsPerWarp = BM / C::kConvWarps;
      const int cw = warp - 6, p8 = lane >> 3, q8 = lane & 7;
      const int cc = q8 & 3;
      int q = 0;
      SegIter segs(a.streamk != 0, g);
      Seg sg;
      bool ok = true;
      while (ok && !*abort_flag && segs.next(sg)) {
        for (int kb = sg.kb_lo; kb < sg.kb_hi; ++kb, ++q) {
          const int st = q % S;
          if (!__all_sync(0xffffffffu, mbar_wait(qfull0 + 8 * st, (q / S) & 1))) {
            raise_error(16, abort_flag);
            ok = false;
            break;
          }
          const uint8_t* srcs = sAq + (size_t)st * C::kAqBytes;
          uint8_t* dsts = sA + (size_t)st * C::kABytes;
          uint4 v[kRowsPerWarp / 8];
#pragma unroll
          for (int it = 0; it < kRowsPerWarp / 8; ++it) {
            const int r = kRowsPerWarp * cw + 2 * (4 * it + p8) + (q8 >> 2);
            v[it] = *reinterpret_cast<const uint4*>(srcs + r * BK + cc * 16);
          }
#pragma unroll
          for (int it = 0; it < kRowsPerWarp / 8; ++it) {
            const int r = kRowsPerWarp * cw + 2 * (4 * it + p8) + (q8 >> 2);
            const uint2 c0 = e4m3x4_to_bf16x4(v[it].x), c1 = e4m3x4_to_bf16x4(v[it].y);
            const uint2 c2 = e4m3x4_to_bf16x4(v[it].z), c3 = e4m3x4_to_bf16x4(v[it].w);
            uint8_t* dst = dsts + r * 128;
            *reinterpret_cast<uint4*>(dst + (((2 * cc) ^ (r & 7)) * 16)) = make_uint4(c0.x, c0.y, c1.x, c1.y);
            *reinterpret_cast<uint4*>(dst + (((2 * cc + 1) ^ (r & 7)) * 16)) = make_uint4(c2.x, c2.y, c3.x, c3.y);
          }
          // generic-proxy smem writes become visible to the tensor core's async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(full0 + 8 * st);
        }
      }
    }
  } else {
    // epilogue warps 0..3: every global write comes after the grids this one depends on
    griddep_wait();
    const int r = warp * 32 + lane;  // row inside the 128-row tile
    int it = 0, epi_phase = 0;
    SegIter segs(a.streamk != 0, g);
    Seg sg;
    while (segs.next(sg)) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      int s, rt, tt;
      decode_item(a, g, sg.item, s, rt, tt);
      const int acc = it & 1;
      // warp-uniform: the tcgen05.ld below is a warp-collective instruction
      if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, (it >> 1) & 1))) {
        raise_error(5, abort_flag);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(warp * 32) << 16);
      const int p = rt * BM + r;  // row of the shard's matrix
      const int m0 = tt * BN;
      const bool whole = sg.kb_lo == 0 && sg.kb_hi == g.nkb;
      float* piece = nullptr;
      if (!whole) {  // this CTA holds one piece of the item: stash it as [col][row]
        const int slot = shares[blockIdx.x] < (uint32_t)sg.item * g.nkb ? 1 : 0;
        piece = a.pieces + ((size_t)blockIdx.x * 2 + slot) * BN * BM;
      }
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        tmem_ld16(tb + c0, v);
        tmem_ld_wait();
        if (whole) {
          epilogue_chunk<BN>(a, s, p, m0 + c0, v);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) piece[(c0 + j) * BM + r] = v[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      ++it;
    }
    // stream-K: once every CTA has stored its pieces, the cut items are finished grid-wide
    if (a.streamk && !*abort_flag) {
      __threadfence();  // this thread's piece stores are visible device-wide
      bool ok = epi_sync(epi_bar, epi_phase, abort_flag, 14);
      if (ok && threadIdx.x == 0) {
        __threadfence();
        if (!grid_sync(a.item_tickets, abort_flag)) *last_flag = 1;
      }
      ok = ok && epi_sync(epi_bar, epi_phase, abort_flag, 15);
      if constexpr (BN <= kTcStreamkMaxBN)  // wider token tiles never run stream-K
        if (ok && !*last_flag)
          streamk_fixup<BN>(a, g, shares, reinterpret_cast<float*>(sA), epi_bar, epi_phase, abort_flag);
    }
  }

  __syncthreads();
  // drain: wait (bounded) for any TMA copy issued but never consumed, so that no copy
  // lands in shared memory after the CTA has exited
  if (warp == kProducerWarp && lane == 0) {
    for (int q = *mma_consumed; q < issued; ++q)
      if (!mbar_wait(full0 + 8 * (q % S), (q / S) & 1)) {
        atomicExch(&g_tc_error, 6u);
        break;
      }
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

static int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

bool tc_supported(int rows, int K, bool fp8) {
  (void)fp8;  // e4m3 weights are widened to bf16 in shared memory
  return rows % BM == 0 && K % BK == 0 && K > 0;
}

// Diagnostic: one thread waits on an mbarrier that nothing ever arrives at, with a short
// limit, and records the error word the way every bounded wait in the library does.
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  if (!mbar_wait(b, 0, limit_ns)) atomicExch(&g_tc_error, 100u);
}

cudaError_t launch_bounded_wait_selftest(int timeout_us, cudaStream_t st) {
  bounded_wait_selftest_kernel<<<1, 1, 0, st>>>((uint64_t)timeout_us * 1000ull);
  note_launch();
  return cudaGetLastError();
}

// Diagnostic: decode n e4m3 codes with the converter's routine (n a multiple of 4).
__global__ void e4m3_decode_kernel(const uint32_t* codes, uint2* out, int n4) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n4) out[i] = e4m3x4_to_bf16x4(codes[i]);
}

cudaError_t launch_e4m3_decode(const void* codes, void* out, int n, cudaStream_t st) {
  const int n4 = n / 4;
  e4m3_decode_kernel<<<(n4 + 255) / 256, 256, 0, st>>>(static_cast<const uint32_t*>(codes), static_cast<uint2*>(out), n4);
  note_launch();
  return cudaGetLastError();
}

unsigned* tc_error_word() {
  static std::mutex mu;
  static unsigned* cache[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tc_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned*>(p);
  }
  return cache[dev];
}

unsigned tc_take_device_error() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_tc_error, &z, sizeof(z));
  return v;
}

template <int BN, bool FP8, bool X8 = false>
static cudaError_t tc_go(const TcArgs& a, cudaStream_t st, bool pdl) {
  using C = TcCfg<BN, FP8, X8>;
  constexpr int KB = C::kKB;
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tmA, tmB;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.K, (cuuint64_t)a.rows, (cuuint64_t)a.t};
    // bf16, and e4m3 for the e4m3 x e4m3 MMA: 128-byte-swizzled boxes the MMA reads directly;
    // e4m3 to be widened: plain 64-byte rows that the converter warps widen into that layout
    const bool bytes = FP8 || X8;
    const cuuint64_t strides[2] = {(cuuint64_t)a.K * (bytes ? 1 : 2), (cuuint64_t)a.shard_stride};
    const cuuint32_t box[3] = {(cuuint32_t)KB, BM, 1}, es[3] = {1, 1, 1};
    if (enc(&tmA, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<uint8_t*>(a.w), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            FP8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {  // activations: bf16, or (X8) their per-token e4m3 codes, [M][ldx]; boxes of 128 bytes x BN
    const cuuint64_t dims[2] = {(cuuint64_t)a.ldx, (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {(cuuint64_t)a.ldx * (X8 ? 1 : 2)};
    const cuuint32_t box[2] = {(cuuint32_t)KB, BN}, es[2] = {1, 1};
    void* base = X8 ? static_cast<void*>(const_cast<uint8_t*>(a.xq)) : static_cast<void*>(const_cast<__nv_bfloat16*>(a.x));
    if (enc(&tmB, X8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static bool attr_set = false;  // per instantiation; set before the first launch
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(tc_kernel<BN, FP8, X8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n_rt = a.rows / BM, n_tt = (a.M + BN - 1) / BN;
  const int n_items = a.mode == TC_ROWPAR_CHAIN ? n_rt * n_tt : n_rt * n_tt * a.t;
  const int sms = sm_count() < kTcMaxGrid ? sm_count() : kTcMaxGrid;
  TcArgs b = a;
  // stream-K when the caller gave scratch for it and the tokens fit one decode tile
  const long long nkb_item = a.mode == TC_ROWPAR_CHAIN ? (long long)a.K / KB * a.t : a.K / KB;
  // stream-K only when whole items cannot fill the GPU: its cross-CTA fix-up costs more than
  // the imbalance of item-granular scheduling once every SM has at least one item
  b.streamk = a.pieces && a.item_tickets && !a.norm_ss && BN <= kTcStreamkMaxBN && n_items < sms &&
              (long long)n_items * nkb_item * kTcMaxGrid < (1ll << 32);  // share table fits 32 bits
  const long long total_kb = (long long)n_items * nkb_item;
  const int grid = b.streamk ? (total_kb < sms ? (int)total_kb : sms) : (n_items < sms ? n_items : sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreadsT);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  // stream-K CTAs meet at a grid barrier: all of them must be resident together
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = b.streamk ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, tc_kernel<BN, FP8, X8>, tmA, tmB, b);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <bool FP8, bool X8 = false>
static cudaError_t tc_bn(const TcArgs& a, cudaStream_t st, bool pdl) {
  if (a.M <= 16) return tc_go<16, FP8, X8>(a, st, pdl);
  if (a.M <= 32) return tc_go<32, FP8, X8>(a, st, pdl);
  if (a.M <= 64) return tc_go<64, FP8, X8>(a, st, pdl);
  if (a.M <= 128) return tc_go<128, FP8, X8>(a, st, pdl);
  return tc_go<256, FP8, X8>(a, st, pdl);
}

cudaError_t launch_tc(const TcArgs& a, cudaStream_t st, bool pdl) {
  if (a.x8) {  // e4m3 weights x e4m3 activations: k in whole 128-byte rows
    if (a.rows % BM != 0 || a.K % 128 != 0 || a.K <= 0 || a.M <= 0 || !a.xq) return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(a.w) | reinterpret_cast<uintptr_t>(a.xq)) & 15) return cudaErrorInvalidValue;
    return tc_bn<false, true>(a, st, pdl);
  }
  if (!tc_supported(a.rows, a.K, a.fp8 != 0) || a.M <= 0) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(a.w) | reinterpret_cast<uintptr_t>(a.x)) & 15) return cudaErrorInvalidValue;
  return a.fp8 ? tc_bn<true>(a, st, pdl) : tc_bn<false>(a, st, pdl);
}

}  // namespace tpx
