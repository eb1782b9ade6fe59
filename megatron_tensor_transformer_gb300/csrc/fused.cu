// Fused decode block: one persistent tcgen05 launch per tensor-parallel block.
//
// The block is the pages' column-parallel first linear followed by the row-parallel second
// linear whose shard partials are summed ("The Tensor-Parallel Shard Group",
// scalablesystem.dev; Y = [XA_1 ... XA_t], Z = sum_k Y_k B_k, "Tensor Parallelism
// (Megatron-Style)", arunshar.com).  For decode (M <= 64 tokens, one token tile) both
// halves are weight streams, so they run as one stream of work items in one launch:
//
//   items [0, t*n_rt1)            stage 1: (shard s, 128 packed rows) of the first linear
//                                 -> SwiGLU h, or QKV plus the one-token attention o_in
//   items [t*n_rt1, + t*n_rt2)    stage 2: (shard s, 128 output rows) of the second linear
//                                 -> fp32 partial P_s of that row tile
//
// Items are taken in that order from one atomic counter (each CTA's first item is its
// block index, so its weights start streaming before the previous kernel has finished).
// A stage-2 item of shard s needs the whole stage-1 output of shard s: its weight tiles are
// issued ahead, and its activation tiles once shard s's stage-1 count is complete (a bounded
// wait).
// The last of the t shard items of a row tile (ticket) folds the t partials in shard
// order, adds the residual and writes y: the same left fold, bit for bit, as the separate
// fold kernel.  No CTA idles while another finishes a second wave of one kernel, and no
// launch gap separates the halves or the fold.
//
// Warp roles per CTA (one CTA per SM): warps 0-3 epilogue, warp 4 weight producer (and the
// scheduler), warp 5 MMA issuer; with e4m3 weights, converter warps from warp 6 and then the
// activation producer.  Every wait is bounded in time; on expiry the kernel records the
// device error word, drains, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "fused.h"
#include "tc.h"
#include "tc_ptx.cuh"

namespace tpx {
using namespace tc;

namespace {

constexpr int FBM = 128, FBK = 64, kRing = 8;
constexpr int kProducer = 4, kMma = 5;
// sync words (all zero between launches)
constexpr int kSyncItem = 0, kSyncExit = 1, kSyncNormTiles = 2, kSyncInNorm = 3, kSyncDone = 8,
              kSyncTicket = 128;

// A pipeline stage holds kSub k-blocks of weights, brought by one TMA copy (the weights viewed as
// {k within a k-block, row, k-block, shard}), and their activation tiles, brought by one more
// (the activations viewed as {64 columns, token, 64-column chunk}).  Each SM completes TMA copies
// at a nearly fixed rate per copy, so fewer, larger copies stream faster.
// bf16 weights: two 64-wide k-blocks per stage, the 128 x 64 bf16 weight tiles (128-byte swizzle)
// the MMA reads from shared memory, with their activation tiles in the same stage.
// e4m3 weights, hi/lo activation codes (SPLIT): two 128-wide k-blocks per stage, the 128 x 128
// e4m3 tiles as TMA brings them (128-byte swizzle: 128 contiguous bytes per row; 64-byte rows at
// the weights' row stride read HBM at about half the rate) go to the MMA as they are.  The
// activation tiles travel in a ring of their own (kSB slots, a second producer warp), and four
// converter warps split each in place into the e4m3 tiles hi and lo (rows 0..BN-1 and BN..2BN-1
// of the same bytes); the MMA multiplies e4m3 x e4m3 with N = 2 BN and the epilogue adds the two
// column halves before the scales.  One MMA commit per stage frees the weight stage, and the
// activation producer learns from the same barrier that the slot is free.
// e4m3 weights, widened (TP_F_KERNEL_TC, and above 32 tokens): one 128-wide k-block per stage;
// converter warps widen the tile, exactly, to bf16 in tensor memory (one of kASlots 64-column A
// slots from column kACol0) and the MMA reads A from there.  A warp may only address one quarter
// of the TMEM lanes, so the converters come as two warps per quarter, each widening one 64-wide
// half of its 32 rows; a weight stage is free again as soon as they have read it.
// Two k-blocks per stage: the MMA-issuing thread pays a fixed cost per stage (its barrier waits
// and commits; measured alone, about 270 ns for one 16 KB k-block), which capped an SM at one
// k-block per 425 ns; a 32 KB stage spreads it over twice the bytes.
template <int BN, bool FP8, bool SPLIT = false>
struct FCfg {
  static constexpr int kKB = FP8 ? 2 * FBK : FBK;        // k per k-block
  static constexpr int kSub = (SPLIT || !FP8) ? 2 : 1;     // k-blocks per stage (1: widened e4m3)
  static constexpr int kABytes1 = FP8 ? FBM * kKB : FBM * kKB * 2;  // one k-block of weights
  static constexpr int kABytes = kABytes1 * kSub;
  static constexpr int kBSub = BN * FBK * 2;               // one 64-wide activation tile
  static constexpr int kBBytes1 = kBSub * (kKB / FBK);     // one k-block of activations
  static constexpr int kBBytes = kBBytes1 * kSub;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // activation ring (e4m3 only)
  // split: a slot is refilled only after the MMA has read it, and its tile then takes an L2 round
  // trip and the split before the MMA can use it (about two stages' time), so the ring must cover
  // that loop; the rest of the shared memory holds weight stages, whose round trip from HBM is
  // several stages long
  static constexpr int kSB = SPLIT ? (kBBytes <= 16384 ? 4 : 3) : (FP8 ? (kBBytes <= 8192 ? 8 : 4) : 0);
  static constexpr int kMaxStages = SPLIT ? 6 : (FP8 ? 10 : 8);
  // bf16 and split: no tensor-memory A slots to feed, so more of the 227 KB goes to weights in flight
  static constexpr int kRingBytes = ((FP8 && !SPLIT) ? 200 : 224) * 1024 - kSB * kBBytes;
  static constexpr int kUnitBytes = FP8 ? kABytes : kStageBytes;
  static constexpr int kStages = kRingBytes / kUnitBytes > kMaxStages ? kMaxStages : kRingBytes / kUnitBytes;
  static constexpr int kBSlots = FP8 ? kSB : kStages;  // activation tiles held in shared memory
  static constexpr int kASlots = 6, kACol0 = 128, kASlotCols = kKB / 2;
  static constexpr int kAccCols = SPLIT ? 2 * BN : BN;  // accumulator columns (hi and lo halves)
  // accumulators in flight: the next item's MMAs run while the epilogue drains the last one
  // (four measured slower than two for the hi/lo block); the widened e4m3 path keeps the rest of
  // its tensor memory for the A slots
  static constexpr int kAcc = 2;
  static constexpr int kTmemCols = (FP8 && !SPLIT) ? 512 : (kAcc * kAccCols < 32 ? 32 : kAcc * kAccCols);
  static constexpr int kConvWarps = FP8 ? (SPLIT ? 4 : 8) : 0;
  // converter warps from warp 6; e4m3: then the activation producer
  static constexpr int kProducerB = 6 + kConvWarps;
  static constexpr int kThreads = 192 + 32 * kConvWarps + (FP8 ? 32 : 0);
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kABytes + (size_t)kBSlots * kBBytes + 1024;
  static_assert(!SPLIT || (FP8 && BN % 8 == 0), "split activations: e4m3 weights, 8-token multiples");
  static_assert(!SPLIT || kSB <= kStages, "split activation slots are freed through the weight stages' barriers");
};

struct FItem {
  int stage, s, rt, nkb;
};

__device__ __forceinline__ FItem fdecode(const FusedArgs& a, int i, int kkb) {
  const int n_rt1 = a.rows1 / FBM, n1 = a.t * n_rt1, n_rt2 = a.d / FBM;
  FItem f;
  if (i < n1) {
    f.stage = 1;
    f.s = i / n_rt1;
    f.rt = i % n_rt1;
    f.nkb = a.d / kkb;
  } else {
    const int j = i - n1;
    f.stage = 2;
    f.s = j / n_rt2;
    f.rt = j % n_rt2;
    f.nkb = a.K2 / kkb;
  }
  return f;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Thread 0, after a barrier of the epilogue warps: one GPU-scope acquire-release add.  The
// release covers the stores the barrier ordered before it (the other threads' partials or y);
// the acquire lets the CTA read, after the next barrier, what the earlier arrivals released.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Generic-proxy global writes (h, o_in) are read by other CTAs' TMA (async proxy).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void raise(unsigned* err, unsigned code, volatile int* abort_flag) {
  atomicExch(err, code);
  *abort_flag = 1;
}

// Wait until shard s's stage-1 items are all done (bounded, ~2 s).
__device__ bool wait_stage1(const FusedArgs& a, int s, volatile int* abort_flag) {
  const unsigned target = (unsigned)(a.rows1 / FBM);
  const unsigned* cnt = a.sync + kSyncDone + s;
  if (ld_acquire(cnt) < target) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; ld_acquire(cnt) < target; ++i) {
      if (*abort_flag) return false;
      if ((i & 63u) == 0 && globaltimer_ns() - t0 > 2000000000ull) {
        raise(a.err, 21, abort_flag);
        return false;
      }
      __nanosleep(32);
    }
  }
  fence_proxy_async_global();
  return true;
}

// e4m3 weights: the fp32 scale of packed row p of shard s in stage 1 or 2 (1 for bf16).
__device__ __forceinline__ float wscale(const FusedArgs& a, int stage, int s, int p) {
  if (!a.fp8) return 1.f;
  const uint8_t* b = stage == 1 ? a.w1 + (size_t)s * a.stride1 + a.scales1 : a.w2 + (size_t)s * a.stride2 + a.scales2;
  return reinterpret_cast<const float*>(b)[p];
}

// Split activations: the power of two s = 2^e with mx / s in [128, 256) (e = 0 for mx = 0).  Then
// x / s = hi + lo exactly, hi the e4m3 rounding of x / s and lo that of the remainder: an 8-bit
// bf16 significand fits in the two while x / s is at least 2^-2 (smaller values lose bits below
// 2^-10 s, against a largest value of at least 2^7 s).
__device__ __forceinline__ int split_exp(float mx) {
  if (!(mx > 0.f) || mx > 3.0e38f) return 0;
  const int e = (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127 - 7;
  return e < -120 ? -120 : (e > 120 ? 120 : e);
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }
// two bf16 (the first in the low half) times inv -> (hi, lo) e4m3 pairs
__device__ __forceinline__ void split_pair(uint32_t xb, float inv, uint16_t& hi, uint16_t& lo) {
  const float y0 = bf16_lo(xb) * inv, y1 = bf16_hi(xb) * inv;
  hi = __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3);
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  lo = __nv_cvt_float2_to_fp8x2(make_float2(y0 - hf.x, y1 - hf.y), __NV_SATFINITE, __NV_E4M3);
}
// the per-(shard, token) maxima of |stage-2 input| and the per-token maxima of |x| (float bits)
__device__ __forceinline__ unsigned* hmax_of(const FusedArgs& a) { return a.sync + fused_hmax_off(a.d); }
__device__ __forceinline__ unsigned* xmax_of(const FusedArgs& a) { return fused_xmax_words(a.sync, a.d); }
// the split scale 2^e of a token from its maximum's bits
__device__ __forceinline__ int split_exp_bits(const unsigned* p) { return split_exp(__uint_as_float(__ldcg(p))); }
__device__ __forceinline__ void conv_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
// The largest |value| a warp's lanes hold for each of 16 tokens, into the shard's maxima
// (non-negative floats order like their bits).
__device__ __forceinline__ void warp_token_max(const FusedArgs& a, int s, int mf, float (&mv)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mv[j] = fmaxf(mv[j], __shfl_xor_sync(0xffffffffu, mv[j], o));
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (mf + j < a.M && mv[j] > 0.f) atomicMax(hmax_of(a) + s * kFusedMaxMWords + mf + j, __float_as_uint(mv[j]));
  }
}

// Stage-1 epilogue for one 16-token chunk of tile row p (packed row of shard s).
template <int KIND, bool SPLIT>
__device__ __forceinline__ void stage1_chunk(const FusedArgs& a, int s, int p, int mf, const float (&v)[16]) {
  if (KIND == FUSED_MLP) {
    // rows come as [8 gate | 8 up] blocks: the up value of row p sits 8 lanes further on
    float u[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) u[j] = __shfl_down_sync(0xffffffffu, v[j], 8);
    float mv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) mv[j] = 0.f;
    if ((p & 15) < 8) {
      const int ldh = a.t * (a.rows1 / 2);
      const int f = s * (a.rows1 / 2) + (p >> 4) * 8 + (p & 7);
      uint16_t* h = reinterpret_cast<uint16_t*>(a.mid);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (mf + j < a.M) {
          const uint16_t hb = f2bf(silu_f(v[j]) * u[j]);
          h[(size_t)(mf + j) * ldh + f] = hb;
          mv[j] = fabsf(__uint_as_float((uint32_t)hb << 16));
        }
    }
    if constexpr (SPLIT) warp_token_max(a, s, mf, mv);
  } else {
    // qkv column s*rows1 + p; a v row also becomes o_in for every q head of its group
    const int ldq = a.t * a.rows1, nqs = a.n_q / a.t, nkvs = a.n_kv / a.t, G = a.n_q / a.n_kv;
    const int vb = (nqs + nkvs) * a.hd;
    uint16_t* q = reinterpret_cast<uint16_t*>(a.mid);
    uint16_t* o = reinterpret_cast<uint16_t*>(a.mid2);
    const int ldo = a.n_q * a.hd;
    const bool vrow = p >= vb;
    const int j = vrow ? (p - vb) / a.hd : 0, e = vrow ? (p - vb) % a.hd : 0;
    float mv[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      mv[jj] = 0.f;
      const int m = mf + jj;
      if (m >= a.M) continue;
      const uint16_t b = f2bf(v[jj]);
      q[(size_t)m * ldq + (size_t)s * a.rows1 + p] = b;
      if (vrow) {
        for (int g = 0; g < G; ++g) o[(size_t)m * ldo + (size_t)(s * nqs + j * G + g) * a.hd + e] = b;
        mv[jj] = fabsf(__uint_as_float((uint32_t)b << 16));
      }
    }
    if constexpr (SPLIT) {
      if (__any_sync(0xffffffffu, vrow)) warp_token_max(a, s, mf, mv);  // only v rows feed o_in
    }
  }
}

// The last shard item of row tile rt folds: y = bf16(((P_0 + P_1) + ... + P_{t-1}) + residual).
// Each thread takes four rows of U tokens per step and issues all U x t loads before the
// adds, so a fold of 64 tokens costs a few L2 round trips instead of one per token group.
template <int U>
__device__ __forceinline__ void fold_tile(const FusedArgs& a, int rt) {
  const int r4 = (threadIdx.x & 31) * 4, w = threadIdx.x >> 5;
  const size_t MD = (size_t)a.M * a.d;
  for (int m0 = U * w; m0 < a.M; m0 += 4 * U) {
    float4 p[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t base = (size_t)(m0 + u) * a.d + (size_t)rt * FBM + r4;
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (m0 + u < a.M && s < a.t) p[u][s] = __ldcg(reinterpret_cast<const float4*>(a.partials + s * MD + base));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int m = m0 + u;
      if (m >= a.M) break;
      const size_t base = (size_t)m * a.d + (size_t)rt * FBM + r4;
      float4 acc = p[u][0];
#pragma unroll
      for (int s = 1; s < 8; ++s) {
        if (s < a.t) {
          acc.x += p[u][s].x;
          acc.y += p[u][s].y;
          acc.z += p[u][s].z;
          acc.w += p[u][s].w;
        }
      }
      if (a.residual) {
        const uint2 r = *reinterpret_cast<const uint2*>(a.residual + base);
        acc.x += bf16_lo(r.x);
        acc.y += bf16_hi(r.x);
        acc.z += bf16_lo(r.y);
        acc.w += bf16_hi(r.y);
      }
      uint2 o;
      o.x = (uint32_t)f2bf(acc.x) | ((uint32_t)f2bf(acc.y) << 16);
      o.y = (uint32_t)f2bf(acc.z) | ((uint32_t)f2bf(acc.w) << 16);
      *reinterpret_cast<uint2*>(a.y + base) = o;
      if (a.out_rms) {
        // this tile's share of the next block's RMSNorm: sum of squares of the stored bf16
        // values of token m, four rows per lane, then a fixed shuffle tree over the warp
        const float e0 = bf16_lo(o.x), e1 = bf16_hi(o.x), e2 = bf16_lo(o.y), e3 = bf16_hi(o.y);
        float ss = ((e0 * e0 + e1 * e1) + e2 * e2) + e3 * e3;
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, sh);
        if ((threadIdx.x & 31) == 0) a.norm_ss[(size_t)m * (a.d / FBM) + rt] = ss;
      }
    }
  }
}

// Per-token RMSNorm factor of x [M, d] (gain 1): 1/sqrt(mean(x^2) + eps), by the 128 epilogue
// threads, one warp per token, each lane eight values per step, then a fixed shuffle tree.
__device__ __forceinline__ void input_norm(const FusedArgs& a) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  for (int m = w; m < a.M; m += 4) {
    float ss = 0.f;
    const __nv_bfloat16* xr = a.x + (size_t)m * a.d;
    int k = 8 * l;
    // eight 16-byte loads in flight, then the squares in k order
    for (; k + 7 * 256 < a.d; k += 8 * 256) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = *reinterpret_cast<const uint4*>(xr + k + i * 256);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float e0 = bf16_lo(u[j]), e1 = bf16_hi(u[j]);
          ss += e0 * e0;
          ss += e1 * e1;
        }
      }
    }
    for (; k < a.d; k += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float e0 = bf16_lo(u[j]), e1 = bf16_hi(u[j]);
        ss += e0 * e0;
        ss += e1 * e1;
      }
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, sh);
    if (l == 0) a.in_scale[m] = 1.f / sqrtf(ss / (float)a.d + a.eps);
  }
}

// The activation tiles of stage j of item f: one TMA copy of kBBytes, the stage's 64-column chunks
// (kSub k-blocks) as [chunk][BN tokens][128 B] tiles.  x (stage 1) and h / o_in (stage 2) are
// viewed as {64 columns, token, chunk}; a chunk past the item's last k-block is not multiplied.
template <class C>
__device__ __forceinline__ void load_act_stage(const CUtensorMap* tmB1, const CUtensorMap* tmB2, const FusedArgs& a,
                                               const FItem& f, int j, uint32_t dst, uint32_t bar, uint64_t pol) {
  const int c0 = C::kSub * j * (C::kKB / FBK);
  if (f.stage == 1)
    tma_load_3d_hint(dst, tmB1, 0, 0, c0, bar, pol);
  else
    tma_load_3d_hint(dst, tmB2, 0, 0, f.s * (a.K2 / FBK) + c0, bar, pol);
}

template <int BN, int KIND, bool FP8, bool SPLIT>
__global__ void __launch_bounds__(FCfg<BN, FP8, SPLIT>::kThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                 const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2, FusedArgs a) {
  using C = FCfg<BN, FP8, SPLIT>;
  constexpr int kProducerB = C::kProducerB;
  constexpr int kSplitBars = SPLIT ? C::kSB : 0;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                            // S x [128 rows x 64] weights (bf16 SW128 or e4m3 SW64)
  uint8_t* sB = smem + (size_t)S * C::kABytes;   // kBSlots x [BN rows x kKB] bf16, SW128 tiles of 64
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (size_t)C::kBSlots * C::kBBytes);
  // bars: full[S], empty[S], tfull[kAcc], tempty[kAcc], ifull[kRing], iempty[kRing], drain, afull[kASlots],
  // aempty[kASlots], fullB[kSB], emptyB[kSB], (split activations) splitB[kSB]
  constexpr int kAcc = C::kAcc;
  int* ring = reinterpret_cast<int*>(bars + 2 * S + 2 * kAcc + 2 * kRing + 1 + 2 * C::kASlots + 2 * C::kSB + kSplitBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring + kRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* mma_consumed = reinterpret_cast<int*>(tmem_slot + 2);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 3);
  int* conv_consumed = reinterpret_cast<int*>(tmem_slot + 4);  // e4m3: weight stages the converters took
  volatile int* norm_last = reinterpret_cast<volatile int*>(tmem_slot + 5);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S), tfull0 = smem_u32(bars + 2 * S),
                 tempty0 = smem_u32(bars + 2 * S + kAcc), ifull0 = smem_u32(bars + 2 * S + 2 * kAcc),
                 iempty0 = smem_u32(bars + 2 * S + 2 * kAcc + kRing),
                 drain_bar = smem_u32(bars + 2 * S + 2 * kAcc + 2 * kRing),
                 afull0 = drain_bar + 8, aempty0 = drain_bar + 8 + 8 * C::kASlots,
                 fullB0 = aempty0 + 8 * C::kASlots, emptyB0 = fullB0 + 8 * C::kSB, splitB0 = emptyB0 + 8 * C::kSB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n1 = a.t * (a.rows1 / FBM), ntot = n1 + a.t * (a.d / FBM);

  // fail fast after a bounded wait has given up (the error word is cleared by tp_sync)
  __shared__ int s_skip;
  if (threadIdx.x == 0) s_skip = *reinterpret_cast<volatile unsigned*>(a.err) != 0u;
  __syncthreads();
  if (s_skip) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full0 + 8 * i, 1);
      // e4m3 widened: freed by the converters; otherwise by the MMA's commit
      mbar_init(empty0 + 8 * i, FP8 && !SPLIT ? C::kConvWarps : 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, 4);  // one arrival per epilogue warp
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(ifull0 + 8 * i, 1);
      // the MMA thread + one lane per epilogue / converter warp (+ the activation producer)
      mbar_init(iempty0 + 8 * i, 5 + C::kConvWarps + (FP8 ? 1 : 0));
    }
    mbar_init(drain_bar, 1);
    if constexpr (FP8) {
      for (int i = 0; i < C::kASlots; ++i) {
        mbar_init(afull0 + 8 * i, C::kConvWarps);  // one arrival per converter warp
        mbar_init(aempty0 + 8 * i, 1);  // tcgen05.commit after the MMAs that read the slot
      }
      for (int i = 0; i < C::kSB; ++i) {
        mbar_init(fullB0 + 8 * i, 1);
        mbar_init(emptyB0 + 8 * i, 1);  // tcgen05.commit after the MMAs that read the tile
      }
      for (int i = 0; i < kSplitBars; ++i) mbar_init(splitB0 + 8 * i, C::kConvWarps);  // split in place
    }
    *abort_flag = 0;
    *mma_consumed = 0;
    *last_flag = 0;
    *conv_consumed = 0;
    fence_mbar_init();
  }
  if (warp == kProducer && lane == 0) {
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB1);
    tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmB2);
  }
  if (warp == kMma) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  int issued = 0, issuedB = 0;  // weight stages / (e4m3) activation tiles this thread issued

  griddep_launch_dependents();
  if (warp == kProducer) {
    if (lane == 0) {
      const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
      int q = 0;  // items published
      bool ok = true;
      auto publish = [&](int id) {
        const int r = q % kRing;
        if (q >= kRing && !mbar_wait(iempty0 + 8 * r, ((q / kRing) - 1) & 1)) {
          raise(a.err, 22, abort_flag);
          ok = false;
          return;
        }
        ring[r] = id;
        mbar_arrive(ifull0 + 8 * r);
        ++q;
      };
      // the weights of stage j of item f (k-blocks kSub j ..) into ring stage st: one TMA copy of
      // kABytes (a k-block past the item's last reads as zeros and is not multiplied)
      auto load_w = [&](const FItem& f, int j, int st) {
        const uint32_t dst = smem_u32(sA + (size_t)st * C::kABytes), bar = full0 + 8 * st;
        tma_load_4d_hint(dst, f.stage == 1 ? &tmA1 : &tmA2, 0, f.rt * FBM, C::kSub * j, f.s, bar, pol_w);
      };
      auto load_x = [&](const FItem& f, int j, int st) {  // bf16: the activations of stage j into stage st
        load_act_stage<C>(&tmB1, &tmB2, a, f, j, smem_u32(sB + (size_t)st * C::kBBytes), full0 + 8 * st, pol_x);
      };
      // first item (static): its first stages of weights go out before the previous kernel ends
      int item = blockIdx.x;
      FItem f = fdecode(a, item, C::kKB);
      if constexpr (FP8) {
        // weights only: the activation tiles have a producer warp of their own.  Stage j of an
        // item holds its k-blocks kSub j .. (the last stage may hold fewer)
        auto issue_w = [&](const FItem& g, int j) {
          const int st = issued % S;
          if (!mbar_wait(empty0 + 8 * st, ((issued / S) & 1) ^ 1)) {
            raise(a.err, 23, abort_flag);
            ok = false;
            return;
          }
          mbar_arrive_expect_tx(full0 + 8 * st, C::kABytes);
          load_w(g, j, st);
          ++issued;
        };
        const int nst0 = (f.nkb + C::kSub - 1) / C::kSub;
        const int pre = nst0 < S ? nst0 : S;
        for (int j = 0; j < pre; ++j) issue_w(f, j);  // fresh stages: no wait
        griddep_wait();
        publish(item);
        for (int j = pre; ok && j < nst0; ++j) issue_w(f, j);
        while (ok && !*abort_flag) {
          item = (int)gridDim.x + (int)atomicAdd(a.sync + kSyncItem, 1u);
          if (item >= ntot) break;
          f = fdecode(a, item, C::kKB);
          publish(item);
          const int nst = (f.nkb + C::kSub - 1) / C::kSub;
          for (int j = 0; ok && j < nst; ++j) issue_w(f, j);
        }
      } else {
        // bf16: a stage holds kSub k-blocks of weights and their activation tiles (the item's last
        // stage may hold fewer)
        auto issue_ab = [&](const FItem& g, int j, int code) {  // stage j: weights and activations
          const int st = issued % S;
          if (!mbar_wait(empty0 + 8 * st, ((issued / S) & 1) ^ 1)) {
            raise(a.err, code, abort_flag);
            ok = false;
            return;
          }
          mbar_arrive_expect_tx(full0 + 8 * st, C::kABytes + C::kBBytes);
          load_w(g, j, st);
          load_x(g, j, st);
          ++issued;
        };
        const int nst0 = (f.nkb + C::kSub - 1) / C::kSub;
        const int pre = nst0 < S ? nst0 : S;
        for (int j = 0; j < pre; ++j) {
          mbar_expect_tx(full0 + 8 * j, C::kABytes);
          load_w(f, j, j);
        }
        griddep_wait();
        publish(item);
        if (ok && f.stage == 2) ok = wait_stage1(a, f.s, abort_flag);
        if (ok) {
          for (int j = 0; j < pre; ++j) {
            mbar_arrive_expect_tx(full0 + 8 * j, C::kBBytes);
            load_x(f, j, j);
          }
          issued = pre;
        }
        for (int j = pre; ok && j < nst0; ++j) issue_ab(f, j, 23);
        // then items from the shared counter, in order: stage 1 of every shard, then stage 2
        while (ok && !*abort_flag) {
          item = (int)gridDim.x + (int)atomicAdd(a.sync + kSyncItem, 1u);
          if (item >= ntot) break;
          f = fdecode(a, item, C::kKB);
          publish(item);
          if (!ok) break;
          const int nst = (f.nkb + C::kSub - 1) / C::kSub;
          int j = 0;
          if (f.stage == 2 && ld_acquire(a.sync + kSyncDone + f.s) < (unsigned)(a.rows1 / FBM)) {
            // weights ahead (their stages were freed by earlier items), then the activations
            const int la = nst < S ? nst : S;
            for (; j < la; ++j) {
              const int st = issued % S;
              if (!mbar_wait(empty0 + 8 * st, ((issued / S) & 1) ^ 1)) {
                raise(a.err, 24, abort_flag);
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(full0 + 8 * st, C::kABytes + C::kBBytes);
              load_w(f, j, st);
              ++issued;
            }
            if (ok) ok = wait_stage1(a, f.s, abort_flag);
            if (!ok) break;
            for (int i = 0; i < la; ++i) load_x(f, i, (issued - la + i) % S);
          } else if (f.stage == 2) {
            fence_proxy_async_global();
          }
          for (; ok && j < nst; ++j) issue_ab(f, j, 25);
        }
      }
      if (ok) publish(-1);
    }
  } else if (warp == kMma) {
    if (lane == 0) {
      constexpr uint32_t idesc = SPLIT ? idesc_e4m3(FBM, 2 * BN) : idesc_bf16(FBM, BN);
      int q = 0, it = 0, consumed = 0;
      while (!*abort_flag) {
        const int r = q % kRing;
        if (!mbar_wait(ifull0 + 8 * r, (q / kRing) & 1)) {
          raise(a.err, 26, abort_flag);
          break;
        }
        const int id = ring[r];
        mbar_arrive(iempty0 + 8 * r);
        ++q;
        if (id < 0) break;
        const FItem f = fdecode(a, id, C::kKB);
        const int acc = it % kAcc;
        if (!mbar_wait(tempty0 + 8 * acc, ((it / kAcc) & 1) ^ 1)) {
          raise(a.err, 27, abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * C::kAccCols);
        bool ok = true;
        if constexpr (SPLIT) {
          const int nst = (f.nkb + C::kSub - 1) / C::kSub;
          for (int j = 0; j < nst; ++j) {
            // the weight stage as it landed, and the activation tiles once split into hi | lo
            const int nsub = f.nkb - C::kSub * j < C::kSub ? f.nkb - C::kSub * j : C::kSub;
            const int st = consumed % S, sl = consumed % C::kSB;
            if (!mbar_wait(full0 + 8 * st, (consumed / S) & 1) ||
                !mbar_wait(splitB0 + 8 * sl, (consumed / C::kSB) & 1)) {
              raise(a.err, 45, abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
            // the stage's descriptors once; an offset inside the stage adds to the address field
            const uint64_t ad = sw128_desc(smem_u32(sA + (size_t)st * C::kABytes)),
                           bd = sw128_desc(smem_u32(sB + (size_t)sl * C::kBBytes));
#pragma unroll
            for (int u = 0; u < C::kSub; ++u) {
              if (u < nsub) {
#pragma unroll
                for (int k = 0; k < C::kKB / 32; ++k)
                  mma_e4m3(d, ad + desc_off(u * C::kABytes1 + 32 * k), bd + desc_off(u * C::kBBytes1 + 32 * k), idesc,
                           (j > 0) || u > 0 || k != 0);
              }
            }
            // one commit frees the weight stage and (the activation producer waits on the same
            // barrier) the activation slot
            mma_commit(empty0 + 8 * st);
            ++consumed;
          }
        } else {
          const int nst = (f.nkb + C::kSub - 1) / C::kSub;
          for (int kb = 0; kb < nst; ++kb) {
            // the activation tile: in the weight stage (bf16), or in its own ring (e4m3)
            constexpr int NB = FP8 ? C::kSB : S;
            const int st = consumed % NB;
            if (!mbar_wait((FP8 ? fullB0 : full0) + 8 * st, (consumed / NB) & 1)) {
              raise(a.err, 28, abort_flag);
              ok = false;
              break;
            }
            const uint32_t bb = smem_u32(sB + (size_t)st * C::kBBytes);
            if constexpr (FP8) {
              // the widened weight tile of this k-block waits in tensor-memory slot `slot`
              const int slot = consumed % C::kASlots;
              if (!mbar_wait(afull0 + 8 * slot, (consumed / C::kASlots) & 1)) {
                raise(a.err, 33, abort_flag);
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t at = tmem_base + (uint32_t)(C::kACol0 + C::kASlotCols * slot);
#pragma unroll
              for (int k = 0; k < C::kKB / 16; ++k)
                mma_bf16_tmem_a(d, at + 8 * k, sw128_desc(bb + (k / 4) * C::kBSub + 32 * (k % 4)), idesc,
                                (kb > 0) || k != 0);
              mma_commit(emptyB0 + 8 * st);
              mma_commit(aempty0 + 8 * slot);
            } else {
              tc_fence_after();
              const uint64_t ad = sw128_desc(smem_u32(sA + (size_t)st * C::kABytes)), bd = sw128_desc(bb);
              const int nsub = f.nkb - C::kSub * kb < C::kSub ? f.nkb - C::kSub * kb : C::kSub;
#pragma unroll
              for (int u = 0; u < C::kSub; ++u) {
                if (u < nsub) {
#pragma unroll
                  for (int k = 0; k < FBK / 16; ++k)
                    mma_bf16(d, ad + desc_off(u * C::kABytes1 + 32 * k), bd + desc_off(u * C::kBBytes1 + 32 * k), idesc,
                             (kb > 0) || u > 0 || k != 0);
                }
              }
              mma_commit(empty0 + 8 * st);
            }
            ++consumed;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
        ++it;
      }
      *mma_consumed = consumed;
      mma_commit(drain_bar);
      if (!mbar_wait(drain_bar, 0)) raise(a.err, 29, abort_flag);
    }
  } else if (warp == kProducerB) {
    if constexpr (FP8) {
      // activation producer (e4m3 weights): follows the item sequence; a stage-2 item first
      // waits (bounded) for its shard's stage-1 items
      if (lane == 0) {
        const uint64_t pol_x = l2_evict_last();
        griddep_wait();
        int q = 0;
        bool ok = true;
        while (ok) {
          const int rr = q % kRing;
          if (!mbar_wait(ifull0 + 8 * rr, (q / kRing) & 1)) {
            raise(a.err, 36, abort_flag);
            break;
          }
          const int id = ring[rr];
          mbar_arrive(iempty0 + 8 * rr);
          ++q;
          if (id < 0 || *abort_flag) break;
          const FItem f = fdecode(a, id, C::kKB);
          if (f.stage == 2 && !wait_stage1(a, f.s, abort_flag)) break;
          const int nst = (f.nkb + C::kSub - 1) / C::kSub;
          for (int j = 0; j < nst; ++j) {
            const int st = issuedB % C::kSB;
            // the slot's previous tile (stage issuedB - kSB) has been read once the MMAs of that
            // stage are done: split activations have no commit of their own, the stage's weight
            // barrier tells (it cannot complete a later phase first while kSB <= kStages)
            const bool freed =
                SPLIT ? (issuedB < C::kSB ||
                         mbar_wait(empty0 + 8 * ((issuedB - C::kSB) % S), ((issuedB - C::kSB) / S) & 1))
                      : mbar_wait(emptyB0 + 8 * st, ((issuedB / C::kSB) & 1) ^ 1);
            if (!freed) {
              raise(a.err, 37, abort_flag);
              ok = false;
              break;
            }
            const uint32_t bar = fullB0 + 8 * st;
            mbar_arrive_expect_tx(bar, C::kBBytes);
            load_act_stage<C>(&tmB1, &tmB2, a, f, j, smem_u32(sB + (size_t)st * C::kBBytes), bar, pol_x);
            ++issuedB;
          }
        }
      }
    }
  } else if (warp >= 6) {
    if constexpr (SPLIT) {
      // Split converters.  The per-token maxima of |x| were written by the kernel launched just
      // before this one (launch_token_absmax), complete once the grids this one depends on are.
      const int cw = warp - 6;
      griddep_wait();
      bool ok = true;
      // each warp splits BN/4 tokens, 8 lanes a token, lane l the 16-wide k chunk l % 8
      constexpr int NIT = BN / 16;
      const int c = lane & 7;
      int tok[NIT];
      float inv1[NIT];
#pragma unroll
      for (int it = 0; it < NIT; ++it) {
        tok[it] = cw * (BN / 4) + 4 * it + (lane >> 3);
        inv1[it] = tok[it] < a.M ? pow2f(-split_exp_bits(xmax_of(a) + tok[it])) : 1.f;
      }
      // per shard, the split exponents of this warp's tokens, once the shard's stage 1 is known done
      __shared__ signed char s_exp[8][kFusedMaxM];
      unsigned shard_seen = 0u;
      int q = 0, kq = 0;
      while (ok) {
        const int rr = q % kRing;
        if (!__all_sync(0xffffffffu, mbar_wait(ifull0 + 8 * rr, (q / kRing) & 1))) {
          raise(a.err, 46, abort_flag);
          break;
        }
        const int id = ring[rr];
        __syncwarp();
        if (lane == 0) mbar_arrive(iempty0 + 8 * rr);
        ++q;
        if (id < 0 || __any_sync(0xffffffffu, *abort_flag != 0)) break;
        const FItem f = fdecode(a, id, C::kKB);
        float inv[NIT];
        if (f.stage == 1) {
#pragma unroll
          for (int it = 0; it < NIT; ++it) inv[it] = inv1[it];
        } else {
          if (!(shard_seen >> f.s & 1u)) {
            // the shard's stage-1 items are done, so the maxima of its h (or o_in) are final
            if (!__all_sync(0xffffffffu, wait_stage1(a, f.s, abort_flag))) break;
#pragma unroll
            for (int it = 0; it < NIT; ++it)
              if (c == 0)
                s_exp[f.s][tok[it]] =
                    (signed char)(tok[it] < a.M ? split_exp_bits(hmax_of(a) + f.s * kFusedMaxMWords + tok[it]) : 0);
            shard_seen |= 1u << f.s;
            __syncwarp();
          }
#pragma unroll
          for (int it = 0; it < NIT; ++it) inv[it] = pow2f(-(int)s_exp[f.s][tok[it]]);
        }
        const int nst = (f.nkb + C::kSub - 1) / C::kSub;
        for (int j = 0; j < nst; ++j, ++kq) {
          const int sl = kq % C::kSB;
          if (!__all_sync(0xffffffffu, mbar_wait(fullB0 + 8 * sl, (kq / C::kSB) & 1))) {
            raise(a.err, 47, abort_flag);
            ok = false;
            break;
          }
          const int nsub = f.nkb - C::kSub * j < C::kSub ? f.nkb - C::kSub * j : C::kSub;
#pragma unroll
          for (int u = 0; u < C::kSub; ++u) {
            if (u >= nsub) break;
            // token m's bf16 rows (k 0..63 in the first 64-wide box, 64..127 in the second) are
            // the bytes of its e4m3 rows hi = m and lo = BN + m: read all of them, then write
            uint8_t* tile = sB + (size_t)sl * C::kBBytes + (size_t)u * C::kBBytes1;
            uint4 v0[NIT], v1[NIT];
#pragma unroll
            for (int it = 0; it < NIT; ++it) {
              const int m = tok[it], sw = m & 7, cc = 2 * (c & 3);
              const uint8_t* row = tile + (c >> 2) * C::kBSub + 128 * m;
              v0[it] = *reinterpret_cast<const uint4*>(row + 16 * (cc ^ sw));
              v1[it] = *reinterpret_cast<const uint4*>(row + 16 * ((cc + 1) ^ sw));
            }
            __syncwarp();
#pragma unroll
            for (int it = 0; it < NIT; ++it) {
              const uint32_t w[8] = {v0[it].x, v0[it].y, v0[it].z, v0[it].w, v1[it].x, v1[it].y, v1[it].z, v1[it].w};
              uint16_t hi[8], lo[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) split_pair(w[e], inv[it], hi[e], lo[e]);
              uint4 H, L;
              H.x = hi[0] | ((uint32_t)hi[1] << 16); H.y = hi[2] | ((uint32_t)hi[3] << 16);
              H.z = hi[4] | ((uint32_t)hi[5] << 16); H.w = hi[6] | ((uint32_t)hi[7] << 16);
              L.x = lo[0] | ((uint32_t)lo[1] << 16); L.y = lo[2] | ((uint32_t)lo[3] << 16);
              L.z = lo[4] | ((uint32_t)lo[5] << 16); L.w = lo[6] | ((uint32_t)lo[7] << 16);
              const int m = tok[it], off = 16 * (c ^ (m & 7));
              *reinterpret_cast<uint4*>(tile + 128 * m + off) = H;
              *reinterpret_cast<uint4*>(tile + 128 * (BN + m) + off) = L;
            }
          }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(splitB0 + 8 * sl);
        }
      }
    } else if constexpr (FP8) {
      // converter warps: warp w may address TMEM lanes 32(w%4)..+31, so it widens those rows;
      // of the two warps of a quarter, warp `sub` takes the 64-wide half `sub` of the stage's
      // 128-wide k-block.  Each thread takes one row: 64 e4m3 codes (four 16-byte chunks, which
      // the 128-byte TMA swizzle keeps bank-conflict free: logical chunk c of row r sits at
      // c ^ (r & 7)), widens them exactly to 32 bf16 pairs and stores them to its TMEM lane,
      // columns 32 sub .. 32 sub + 31 of the A slot.
      const int quarter = warp & 3, r = 32 * quarter + lane, sub = (warp - 6) >> 2;
      const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
      // software pipeline: a stage's TMEM store completes while the next stage of the same item
      // is loaded and widened; the store still pending is published (afull) after that.  Never
      // across items: the next item may wait on stage-1 work that needs this one finished.
      int pend = -1;
      auto publish_pending = [&]() {
        if (pend >= 0) {
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(afull0 + 8 * pend);
          pend = -1;
        }
      };
      int q = 0, kq = 0;
      bool ok = true;
      while (ok) {
        const int rr = q % kRing;
        if (!__all_sync(0xffffffffu, mbar_wait(ifull0 + 8 * rr, (q / kRing) & 1))) {
          raise(a.err, 34, abort_flag);
          break;
        }
        const int id = ring[rr];
        __syncwarp();
        if (lane == 0) mbar_arrive(iempty0 + 8 * rr);
        ++q;
        if (id < 0 || __any_sync(0xffffffffu, *abort_flag != 0)) break;
        const int nkb = fdecode(a, id, C::kKB).nkb;
        for (int kb = 0; kb < nkb; ++kb, ++kq) {
          const int st = kq % S, slot = kq % C::kASlots;
          if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * st, (kq / S) & 1)) ||
              !__all_sync(0xffffffffu, mbar_wait(aempty0 + 8 * slot, ((kq / C::kASlots) & 1) ^ 1))) {
            raise(a.err, 35, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* row = sA + (size_t)st * C::kABytes + r * C::kKB;
          uint32_t out[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * ((4 * sub + j) ^ (r & 7)));
            const uint2 c0 = e4m3x4_to_bf16x4(v.x), c1 = e4m3x4_to_bf16x4(v.y);
            const uint2 c2 = e4m3x4_to_bf16x4(v.z), c3 = e4m3x4_to_bf16x4(v.w);
            out[8 * j + 0] = c0.x; out[8 * j + 1] = c0.y; out[8 * j + 2] = c1.x; out[8 * j + 3] = c1.y;
            out[8 * j + 4] = c2.x; out[8 * j + 5] = c2.y; out[8 * j + 6] = c3.x; out[8 * j + 7] = c3.y;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty0 + 8 * st);  // the weight stage is read: free it
          publish_pending();
          tmem_st32(tmem_base + lane_base + (uint32_t)(C::kACol0 + C::kASlotCols * slot + 32 * sub), out);
          pend = slot;
          if (kb == nkb - 1) publish_pending();
        }
      }
      publish_pending();
      if (warp == 6 && lane == 0) *conv_consumed = kq;
    }
  } else {
    // epilogue warps 0..3: global writes only after the grids this one depends on
    griddep_wait();
    const int r = warp * 32 + lane;  // row inside the 128-row tile
    if (a.in_norm && blockIdx.x == 0) {  // the input's RMSNorm factors, published to every CTA
      input_norm(a);
      __threadfence();
      epi_bar();
      if (threadIdx.x == 0) red_release_add(a.sync + kSyncInNorm, 1u);
    }
    bool scale_ready = a.in_norm == 0;
    int q = 0, it = 0;
    while (true) {
      const int rr = q % kRing;
      if (!__all_sync(0xffffffffu, mbar_wait(ifull0 + 8 * rr, (q / kRing) & 1))) {
        raise(a.err, 30, abort_flag);
        break;
      }
      const int id = ring[rr];
      __syncwarp();
      if (lane == 0) mbar_arrive(iempty0 + 8 * rr);
      ++q;
      if (id < 0 || __any_sync(0xffffffffu, *abort_flag != 0)) break;
      const FItem f = fdecode(a, id, C::kKB);
      const int acc = it % kAcc;
      // fetched while the item's MMAs run: the row's fp32 scale (e4m3), and (split activations)
      // the first 16 tokens' scales 2^e
      const int p = f.rt * FBM + r;
      const float wsc = FP8 ? wscale(a, f.stage, f.s, p) : 1.f;
      const unsigned* split_max = nullptr;  // the maxima the item's activations were split by
      float tsc0[16];
      if constexpr (SPLIT) {
        if (f.stage == 1) {
          split_max = xmax_of(a);  // written before this launch (the epilogue has passed griddep_wait)
        } else {
          if (!__all_sync(0xffffffffu, wait_stage1(a, f.s, abort_flag))) break;
          split_max = hmax_of(a) + f.s * kFusedMaxMWords;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) tsc0[j] = j < a.M ? pow2f(split_exp_bits(split_max + j)) : 0.f;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, (it / kAcc) & 1))) {
        raise(a.err, 31, abort_flag);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + (uint32_t)(acc * C::kAccCols) + ((uint32_t)(warp * 32) << 16);
      const bool tok_scale = f.stage == 1 && a.in_scale != nullptr;
      if (tok_scale && !scale_ready) {  // wait (bounded) for CTA 0's input norm
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire(a.sync + kSyncInNorm) == 0u) {
          if (globaltimer_ns() - t0 > 2000000000ull) {
            raise(a.err, 39, abort_flag);
            break;
          }
          __nanosleep(64);
        }
        scale_ready = true;
      }
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        tmem_ld16(tb + c0, v);
        if constexpr (SPLIT) {
          float w[16];
          tmem_ld16(tb + BN + c0, w);  // the lo half
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float ts = c0 == 0 ? tsc0[j] : (c0 + j < a.M ? pow2f(split_exp_bits(split_max + c0 + j)) : 0.f);
            v[j] = ((v[j] + w[j]) * wsc) * ts;
          }
        } else {
          tmem_ld_wait();
        }
        if constexpr (FP8 && !SPLIT) {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] *= wsc;
        }
        if (tok_scale) {  // RMSNorm of the input as a per-token factor on the accumulator
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] *= __ldcg(a.in_scale + c0 + j);
        }
        if (f.stage == 1) {
          stage1_chunk<KIND, SPLIT>(a, f.s, p, c0, v);
        } else {
          float* P = a.partials + (size_t)f.s * a.M * a.d + p;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < a.M) P[(size_t)(c0 + j) * a.d] = v[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      ++it;
      // make this item's stores visible, then count it (stage 1) or take the tile's ticket (stage 2)
      if (f.stage == 1) {
        // h / o_in are read by other CTAs' TMA loads (the async proxy)
        __threadfence();
        fence_proxy_async_global();
        epi_bar();
        if (threadIdx.x == 0) red_release_add(a.sync + kSyncDone + f.s, 1u);
      } else {
        epi_bar();
        if (threadIdx.x == 0) {
          const unsigned old = atom_add_acq_rel(a.sync + kSyncTicket + f.rt, 1u);
          const int last = old == (unsigned)(a.t - 1);
          if (last) a.sync[kSyncTicket + f.rt] = 0u;  // every shard has arrived: reset for the next launch
          *last_flag = last;
        }
        epi_bar();
        if (*last_flag) {
          fold_tile<FP8 ? 2 : 3>(a, f.rt);
          if (a.out_rms) {
            // the tile whose fold comes last sums every tile's share, in tile order
            epi_bar();
            if (threadIdx.x == 0) {
              const int nt = a.d / FBM;
              const unsigned old = atom_add_acq_rel(a.sync + kSyncNormTiles, 1u);
              const int lastn = old == (unsigned)(nt - 1);
              if (lastn) a.sync[kSyncNormTiles] = 0u;
              *norm_last = lastn;
            }
            epi_bar();
            if (*norm_last && threadIdx.x < a.M) {
              const int nt = a.d / FBM;
              const float* row = a.norm_ss + (size_t)threadIdx.x * nt;
              // 16 loads in flight, then the adds in tile order
              float ss = 0.f;
              int t2 = 0;
              for (; t2 + 16 <= nt; t2 += 16) {
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = __ldcg(row + t2 + j);
#pragma unroll
                for (int j = 0; j < 16; ++j) ss += v[j];
              }
              for (; t2 < nt; ++t2) ss += __ldcg(row + t2);
              a.out_rms[threadIdx.x] = 1.f / sqrtf(ss / (float)a.d + a.eps);
            }
          }
        }
      }
    }
  }

  __syncthreads();
  // drain: wait (bounded) for any TMA copy issued but never consumed
  if (warp == kProducer && lane == 0) {
    for (int qq = FP8 && !SPLIT ? *conv_consumed : *mma_consumed; qq < issued; ++qq)
      if (!mbar_wait(full0 + 8 * (qq % S), (qq / S) & 1)) {
        atomicExch(a.err, 32u);
        break;
      }
  }
  if constexpr (FP8) {
    if (warp == kProducerB && lane == 0) {
      for (int qq = *mma_consumed; qq < issuedB; ++qq)
        if (!mbar_wait(fullB0 + 8 * (qq % C::kSB), (qq / C::kSB) & 1)) {
          atomicExch(a.err, 38u);
          break;
        }
    }
  }
  __syncthreads();
  if (warp == kMma) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
  // the last CTA out resets the scheduler words for the next launch
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.sync + kSyncExit, 1u) == gridDim.x - 1) {
      a.sync[kSyncItem] = 0u;
      a.sync[kSyncInNorm] = 0u;
      for (int s = 0; s < 8; ++s) a.sync[kSyncDone + s] = 0u;
      if (SPLIT) {
        for (int i = 0; i < 8 * kFusedMaxMWords; ++i) hmax_of(a)[i] = 0u;  // the h (or o_in) maxima
      }
      if (*reinterpret_cast<volatile unsigned*>(a.err) != 0u) {
        for (int rt = 0; rt < a.d / FBM; ++rt) a.sync[kSyncTicket + rt] = 0u;
        a.sync[kSyncNormTiles] = 0u;
      }
      a.sync[kSyncExit] = 0u;
      __threadfence();
    }
  }
}

}  // namespace

bool fused_supported(int rows1, int d, int K2, int M, int t, bool fp8) {
  const int kkb = fp8 ? 2 * FBK : FBK;  // e4m3 stages take 128-wide k-blocks
  return M > 0 && M <= kFusedMaxM && t >= 1 && t <= 8 && rows1 % FBM == 0 && rows1 > 0 && d % FBM == 0 &&
         d > 0 && d % kkb == 0 && K2 % kkb == 0 && K2 > 0 && fused_sync_words(d) <= kTcMaxStreamkItems - 64;
}

template <int BN, int KIND, bool FP8, bool SPLIT>
static cudaError_t fused_go(const FusedArgs& a, cudaStream_t st, bool pdl) {
  using C = FCfg<BN, FP8, SPLIT>;
  // weights: 128-byte box rows in the 128-byte swizzle: bf16 boxes of 64 columns the MMA reads,
  // or e4m3 boxes of 128 columns the converter warps read
  const CUtensorMapDataType wty = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle wsw = CU_TENSOR_MAP_SWIZZLE_128B;
  const cuuint64_t wes = FP8 ? 1 : 2;
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tm[4];
  const cuuint32_t es4[4] = {1, 1, 1, 1}, es3[3] = {1, 1, 1};
  // Weights as {k within a k-block, row, k-block, shard}: one copy brings a whole stage, kSub
  // consecutive k-blocks of 128 rows, as kSub 128-row tiles one after another in shared memory.
  // A TMA copy costs each SM about the same time whatever its size, so two 16 KB boxes per stage
  // capped an SM's weight stream near half of what one 32 KB copy reaches.
  {  // stage-1 weights [t][rows1][d]
    const cuuint64_t dims[4] = {(cuuint64_t)C::kKB, (cuuint64_t)a.rows1, (cuuint64_t)(a.d / C::kKB), (cuuint64_t)a.t};
    const cuuint64_t strides[3] = {(cuuint64_t)a.d * wes, (cuuint64_t)C::kKB * wes, (cuuint64_t)a.stride1};
    const cuuint32_t box[4] = {(cuuint32_t)C::kKB, FBM, (cuuint32_t)C::kSub, 1};
    if (enc(&tm[0], wty, 4, const_cast<uint8_t*>(a.w1), dims, strides, box, es4,
            CU_TENSOR_MAP_INTERLEAVE_NONE, wsw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Activations as {64 columns, token, 64-column chunk}: one copy brings a stage's chunks.
  constexpr cuuint32_t kChunks = (cuuint32_t)(C::kKB / FBK * C::kSub);
  {  // x [M, d]
    const cuuint64_t dims[3] = {(cuuint64_t)FBK, (cuuint64_t)a.M, (cuuint64_t)(a.d / FBK)};
    const cuuint64_t strides[2] = {(cuuint64_t)a.d * 2, (cuuint64_t)FBK * 2};
    const cuuint32_t box[3] = {FBK, BN, kChunks};
    if (enc(&tm[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(a.x), dims, strides, box, es3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {  // stage-2 weights [t][rows2 = d][K2]
    const cuuint64_t dims[4] = {(cuuint64_t)C::kKB, (cuuint64_t)a.d, (cuuint64_t)(a.K2 / C::kKB), (cuuint64_t)a.t};
    const cuuint64_t strides[3] = {(cuuint64_t)a.K2 * wes, (cuuint64_t)C::kKB * wes, (cuuint64_t)a.stride2};
    const cuuint32_t box[4] = {(cuuint32_t)C::kKB, FBM, (cuuint32_t)C::kSub, 1};
    if (enc(&tm[2], wty, 4, const_cast<uint8_t*>(a.w2), dims, strides, box, es4,
            CU_TENSOR_MAP_INTERLEAVE_NONE, wsw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {  // stage-2 activations [M, t*K2] (h or o_in)
    const cuuint64_t dims[3] = {(cuuint64_t)FBK, (cuuint64_t)a.M, (cuuint64_t)(a.t * a.K2 / FBK)};
    const cuuint64_t strides[2] = {(cuuint64_t)a.t * a.K2 * 2, (cuuint64_t)FBK * 2};
    const cuuint32_t box[3] = {FBK, BN, kChunks};
    if (enc(&tm[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.mid2, dims, strides, box, es3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(fused_kernel<BN, KIND, FP8, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int ntot = a.t * (a.rows1 / FBM) + a.t * (a.d / FBM);
  const int grid = ntot < sms ? ntot : sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  // No cooperative launch: it would keep this grid from starting while the previous kernel
  // drains.  CTAs do wait on one another's items, but the grid is at most one CTA per SM and
  // the only CTAs that can hold an SM are those of kernels that finish without waiting on this
  // one, so every CTA becomes resident; each wait is bounded in any case.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_kernel<BN, KIND, FP8, SPLIT>, tm[0], tm[1], tm[2], tm[3], a);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int KIND, bool FP8, bool SPLIT = false>
static cudaError_t fused_bn(const FusedArgs& a, cudaStream_t st, bool pdl) {
  if (a.M <= 16) return fused_go<16, KIND, FP8, SPLIT>(a, st, pdl);
  if (a.M <= 32) return fused_go<32, KIND, FP8, SPLIT>(a, st, pdl);
  return fused_go<64, KIND, FP8, SPLIT>(a, st, pdl);
}

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t st, bool pdl) {
  if (!fused_supported(a.rows1, a.d, a.K2, a.M, a.t, a.fp8 != 0) || !a.err || !a.sync || !a.partials)
    return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(a.w1) | reinterpret_cast<uintptr_t>(a.w2) | reinterpret_cast<uintptr_t>(a.x) |
       reinterpret_cast<uintptr_t>(a.mid2)) & 15)
    return cudaErrorInvalidValue;
  if (a.split && !a.fp8) return cudaErrorInvalidValue;
  if (a.split)
    return a.kind == FUSED_MLP ? fused_bn<FUSED_MLP, true, true>(a, st, pdl)
                               : fused_bn<FUSED_PROJ, true, true>(a, st, pdl);
  if (a.fp8) return a.kind == FUSED_MLP ? fused_bn<FUSED_MLP, true>(a, st, pdl) : fused_bn<FUSED_PROJ, true>(a, st, pdl);
  return a.kind == FUSED_MLP ? fused_bn<FUSED_MLP, false>(a, st, pdl) : fused_bn<FUSED_PROJ, false>(a, st, pdl);
}

}  // namespace tpx
