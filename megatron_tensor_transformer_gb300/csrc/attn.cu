// Decode attention over a KV cache, head-sharded: each logical shard owns whole GQA groups (its
// q heads and the kv heads they read) and the cache of those kv heads, so attention is local
// to the shard: each shard attends with its own heads (scalablesystem.dev, "The
// Tensor-Parallel Shard Group"), and the KV cache is split with them (vidyal.ai model-parallelism).
//
// Per sequence m (one new token each) and q head h of kv head g = h / (n_q / n_kv):
//   o[m, h] = sum_j softmax_j(q . k_j / sqrt(hd)) v_j,   j = 0 .. len[m]
// where position len[m] is the new token itself (appended first).  Two launches:
//   append   the new k, v from qkv into the cache at position len[m]; resets the merge
//            counters; zero output rows for lengths outside [0, L).  It lets the next launch
//            start at once (programmatic dependent launch);
//   attend   a persistent kernel, one CTA per SM.  The work is a list of units (sequence,
//            kv head, chunk of P positions), split evenly over the CTAs in order, so each
//            CTA streams a contiguous run of the cache: a producer warp keeps a ring of TMA
//            stages (k and v of one chunk, 128-byte swizzle) full while consumer warps, 16
//            positions each, run an online softmax on the tensor cores (mma.sync: the
//            group's q heads are the MMA rows, so every k and v byte is read once for all
//            of them).  Where a (sequence, kv head) ends inside a CTA's run, its warps'
//            states are merged in warp order; one split across CTAs leaves a partial
//            (un-normalised p.v, max, sum) per piece, and the CTA that finishes the last
//            piece merges the pieces in position order.  The new token's k and v are written
//            into the staged chunk from qkv, so the pass does not wait for the append: it
//            overlaps it, and waits for it only before the merge counters and at exit.
// Every sum has a fixed order for a given GPU (the split follows the SM count), so runs
// repeat bit for bit.  The pass reads the cache once (HBM-bound).  The probabilities enter
// P V rounded to bf16 (the MMA's operand type).
#include <cuda.h>

#include "attn.h"
#include "common.cuh"
#include "tc.h"
#include "tc_ptx.cuh"

namespace tpx {

namespace {

constexpr unsigned kFull = 0xffffffffu;

// positions per chunk (one ring stage) for head dim hd
__host__ __device__ constexpr int chunk_positions(int hd) { return hd == 256 ? 64 : 128; }

struct AttnGeo {
  int t, M, L, n_q, n_kv, hd;
  int nqs, nkvs, G, Qs;  // per shard: q heads, kv heads; q heads per kv head; qkv columns per shard
  int P;                 // positions per chunk
};

__host__ __device__ inline AttnGeo attn_geo(int t, int M, int L, int n_q, int n_kv, int hd) {
  AttnGeo g{t, M, L, n_q, n_kv, hd, n_q / t, n_kv / t, n_q / n_kv, (n_q + 2 * n_kv) / t * hd, chunk_positions(hd)};
  return g;
}

// Stage geometry for head dim HD: k and v of P positions staged as HD/64 boxes of [P rows][64
// dims] each; one consumer warp per 16 positions; NS stages in 192 KB.
template <int HD>
struct ACfg {
  static constexpr int P = chunk_positions(HD);
  static constexpr int CW = P / 16;  // consumer warps
  static constexpr int NT = CW * 32;
  static constexpr int BOX = P * 128;
  static constexpr int KVB = HD / 64 * BOX;
  static constexpr int STAGE = 2 * KVB;
  static constexpr int NS = (192 * 1024) / STAGE;
  static constexpr int QSTR = HD * 2 + 16;  // padded q row (bytes): ldmatrix without conflicts
  static constexpr size_t kRing = (size_t)NS * STAGE;
  static constexpr size_t kQ = 16 * QSTR;
  static constexpr size_t kML = 2 * 2 * CW * 16 * 4;  // maxima and sums, two buffers
  static constexpr size_t SMEM = 1024 + kRing + kQ + kML + (2 * NS + 1) * 8;
  static_assert((size_t)CW * 16 * HD * 4 == (size_t)STAGE, "a stage holds the warps' [16][HD] fp32 states");
};

// cache element (shard s, sequence m, local kv head gl, position j, dim 0)
__device__ __forceinline__ size_t cache_off(const AttnGeo& g, int s, int m, int gl, int j) {
  return ((((size_t)s * g.M + m) * g.nkvs + gl) * g.L + j) * g.hd;
}

// Merge counters of (m, gg), after the partials in the workspace.
__device__ __forceinline__ unsigned* counter_ptr(const AttnGeo& g, float* ws, int m, int gg) {
  const size_t nch = (size_t)(g.L + g.P - 1) / g.P;
  return reinterpret_cast<unsigned*>(ws + (size_t)g.M * g.n_kv * nch * g.G * (g.hd + 2)) + (size_t)m * g.n_kv + gg;
}

// grid (M, n_kv), block hd / 8 x 2: thread (i, kv) copies 8 values of k (kv = 0) or v (kv = 1)
__global__ void append_kernel(AttnGeo g, const __nv_bfloat16* __restrict__ qkv, const int32_t* __restrict__ lens,
                              __nv_bfloat16* kc, __nv_bfloat16* vc, float* ws, __nv_bfloat16* o_in) {
  tc::griddep_launch_dependents();
  const int m = blockIdx.x, gg = blockIdx.y, s = gg / g.nkvs, gl = gg % g.nkvs;
  const int n = lens[m];
  if (threadIdx.x == 0 && threadIdx.y == 0) *counter_ptr(g, ws, m, gg) = 0u;
  if (n < 0 || n >= g.L) {  // no attention for this sequence: its heads of this group read zero
    uint4* o = reinterpret_cast<uint4*>(o_in + (size_t)m * g.n_q * g.hd + (size_t)(s * g.nqs + gl * g.G) * g.hd);
    for (int i = threadIdx.y * blockDim.x + threadIdx.x; i < g.G * g.hd / 8; i += blockDim.x * blockDim.y)
      o[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const int i = threadIdx.x, kv = threadIdx.y;
  const size_t src = (size_t)m * g.t * g.Qs + (size_t)s * g.Qs + (size_t)(g.nqs + kv * g.nkvs + gl) * g.hd + 8 * i;
  __nv_bfloat16* dst = (kv ? vc : kc) + cache_off(g, s, m, gl, n) + 8 * i;
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(qkv + src);
}

// Partial result of the piece of (m, gg) that starts at chunk c: [G][hd] un-normalised p.v,
// then [G] max, [G] sum.
__device__ __forceinline__ float* part_ptr(const AttnGeo& g, float* ws, int m, int gg, int c) {
  const int nch = (g.L + g.P - 1) / g.P;
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

// Byte offset of (position r, dim k) in a chunk staged as HD/64 boxes of [P rows][64 dims] in
// the 128-byte swizzle (the 16-byte piece j of a row sits at j ^ (r & 7)).
template <int HD>
__device__ __forceinline__ uint32_t sw_off(int r, int k) {
  return (uint32_t)((k >> 6) * ACfg<HD>::BOX + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + ((k & 7) << 1));
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- the unit list: (sequence m, kv head gg, chunk c) over sequences whose length is in
// [0, L), sequence-major, then kv head, then chunk.  Every warp walks it alike (whole-warp
// shuffles: all 32 lanes take part).
__device__ __forceinline__ int seq_chunks(const AttnGeo& g, int n) {
  return (n >= 0 && n < g.L) ? (n + g.P) / g.P : 0;  // positions 0..n
}

__device__ long long count_units(const AttnGeo& g, const int32_t* __restrict__ lens, int lane) {
  long long tot = 0;
  for (int m0 = 0; m0 < g.M; m0 += 32) {
    int cnt = m0 + lane < g.M ? seq_chunks(g, lens[m0 + lane]) : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
    tot += cnt;
  }
  return tot * g.n_kv;
}

struct Cursor {
  int m, gg, c, nch, n;  // sequence, kv head, chunk; the sequence's chunks and length
};

// the cursor at unit u (u below the unit count)
__device__ Cursor locate(const AttnGeo& g, const int32_t* __restrict__ lens, long long u, int lane) {
  Cursor cu{0, 0, 0, 1, 0};
  long long base = 0;
  for (int m0 = 0; m0 < g.M; m0 += 32) {
    const int mm = m0 + lane;
    const int n = mm < g.M ? lens[mm] : -1;
    const int ch = seq_chunks(g, n);
    int incl = ch * g.n_kv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    const int total = __shfl_sync(kFull, incl, 31);
    if (u < base + total) {
      const int f = __ffs(__ballot_sync(kFull, base + incl > u)) - 1;
      const int inc_f = __shfl_sync(kFull, incl, f), ch_f = __shfl_sync(kFull, ch, f);
      const int n_f = __shfl_sync(kFull, n, f);
      const int off = (int)(u - (base + inc_f - ch_f * g.n_kv));
      cu.m = m0 + f;
      cu.n = n_f;
      cu.nch = ch_f;
      cu.gg = off / ch_f;
      cu.c = off % ch_f;
      return cu;
    }
    base += total;
  }
  return cu;
}

// next unit (called only when there is one)
__device__ __forceinline__ void advance(const AttnGeo& g, const int32_t* __restrict__ lens, Cursor& cu) {
  if (++cu.c < cu.nch) return;
  cu.c = 0;
  if (++cu.gg < g.n_kv) return;
  cu.gg = 0;
  do {
    ++cu.m;
    cu.n = lens[cu.m];
    cu.nch = seq_chunks(g, cu.n);
  } while (cu.nch == 0 && cu.m + 1 < g.M);
}

// CTA i of nct takes units [U i / nct, U (i + 1) / nct).
__device__ __forceinline__ long long split_at(long long U, int nct, int i) { return U * i / nct; }

// Calls f(cs) for the first chunk cs of every piece of the (sequence, kv head) whose chunk 0 is
// unit ub and which has nch chunks: chunk 0, then each CTA boundary inside, in position order.
template <class F>
__device__ __forceinline__ void for_pieces(long long U, int nct, long long ub, int nch, F f) {
  f(0);
  int i = (int)(ub * nct / U);
  while (i < nct && split_at(U, nct, i) <= ub) ++i;
  long long prev = ub;
  for (; i < nct; ++i) {
    const long long b = split_at(U, nct, i);
    if (b >= ub + nch) break;
    if (b != prev) {
      f((int)(b - ub));
      prev = b;
    }
  }
}

// grid: one CTA per SM; block: CW consumer warps + one producer warp.
template <int HD>
__global__ void __launch_bounds__(ACfg<HD>::NT + 32, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnGeo g,
                float scale, const __nv_bfloat16* __restrict__ qkv, const int32_t* __restrict__ lens, float* ws,
                __nv_bfloat16* __restrict__ o_in, unsigned* err) {
  using C = ACfg<HD>;
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = ring + C::kRing;                                   // [16][QSTR] bf16, rows >= G zero
  float* mlw = reinterpret_cast<float*>(sQ + C::kQ);               // [2][2][CW][16] warps' maxima, sums
  uint64_t* bars = reinterpret_cast<uint64_t*>(mlw + 4 * C::CW * 16);  // full[NS], empty[NS], consumers
  constexpr int kMaxPieces = 32;
  __shared__ int s_last, s_npc, s_pc[kMaxPieces];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = tc::smem_u32(bars), empty0 = full0 + 8 * C::NS, cbar = empty0 + 8 * C::NS;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      tc::mbar_init(full0 + 8 * i, 1);
      tc::mbar_init(empty0 + 8 * i, C::CW);
    }
    tc::mbar_init(cbar, C::CW);
    tc::fence_mbar_init();
  }
  __syncthreads();
  const long long U = count_units(g, lens, lane);
  const int nct = gridDim.x;
  const long long u0 = split_at(U, nct, blockIdx.x), u1 = split_at(U, nct, blockIdx.x + 1);
  if (u0 >= u1) {
    tc::griddep_wait();  // this grid ends after the append (the launch after it relies on that)
    return;
  }
  const int nu = (int)(u1 - u0);
  Cursor cu = locate(g, lens, u0, lane);

  if (warp == C::CW) {  // producer: one thread keeps the ring full
    if (lane != 0) return;
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmV);
    const uint64_t pol = tc::l2_evict_first();  // the cache streams through once
    for (int k = 0; k < nu; ++k) {
      const int st = k % C::NS;
      if (k >= C::NS && !tc::mbar_wait(empty0 + 8 * st, ((k / C::NS) - 1) & 1)) {
        atomicExch(err, 41u);
        return;
      }
      const uint32_t fb = full0 + 8 * st;
      tc::mbar_arrive_expect_tx(fb, C::STAGE);
      const int sh = cu.gg / g.nkvs, gl = cu.gg % g.nkvs;
      const int row0 = ((sh * g.M + cu.m) * g.nkvs + gl) * g.L + cu.c * C::P;  // rows past the end: masked
      const uint32_t dK = tc::smem_u32(ring + (size_t)st * C::STAGE), dV = dK + C::KVB;
#pragma unroll
      for (int bx = 0; bx < HD / 64; ++bx) {
        tc::tma_load_2d_hint(dK + bx * C::BOX, &tmK, bx * 64, row0, fb, pol);
        tc::tma_load_2d_hint(dV + bx * C::BOX, &tmV, bx * 64, row0, fb, pol);
      }
      if (k + 1 < nu) advance(g, lens, cu);
    }
    tc::griddep_wait();
    return;
  }

  // consumers: warp w takes positions 16w .. 16w+15 of every chunk
  const int tid = threadIdx.x, gq = lane >> 2, qq = lane & 3, w0 = 16 * warp;
  const uint32_t q_base = tc::smem_u32(sQ);
  uint32_t cph = 0;
  auto csync = [&]() -> bool {  // the consumer warps meet (bounded wait)
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(cbar);
    const bool ok = tc::mbar_wait(cbar, cph);
    cph ^= 1u;
    __syncwarp();
    if (!ok && lane == 0) atomicExch(err, 43u);
    return ok;
  };
  // q of a (sequence, kv head): the group's G heads as 16 rows (rows >= G zero), QV pieces a thread
  constexpr int QV = (16 * HD / 8 + C::NT - 1) / C::NT;
  uint4 qn[QV];
  auto load_q = [&](const Cursor& x) {
    const int sh = x.gg / g.nkvs, gl = x.gg % g.nkvs;
    const __nv_bfloat16* qp = qkv + (size_t)x.m * g.t * g.Qs + (size_t)sh * g.Qs + (size_t)gl * g.G * HD;
#pragma unroll
    for (int i = 0; i < QV; ++i) {
      const int idx = tid + i * C::NT, r = idx / (HD / 8), c8 = idx % (HD / 8);
      qn[i] = (idx < 16 * HD / 8 && r < g.G) ? *reinterpret_cast<const uint4*>(qp + (size_t)r * HD + 8 * c8)
                                             : make_uint4(0, 0, 0, 0);
    }
  };
  auto store_q = [&]() {
#pragma unroll
    for (int i = 0; i < QV; ++i) {
      const int idx = tid + i * C::NT, r = idx / (HD / 8), c8 = idx % (HD / 8);
      if (idx < 16 * HD / 8) *reinterpret_cast<uint4*>(sQ + r * C::QSTR + 16 * c8) = qn[i];
    }
  };
  // the new token's k and v (position n of the last chunk), for the warp that owns that row
  constexpr int NV = (2 * HD / 8 + 31) / 32;
  uint4 kvn[NV];
  auto owner = [&](const Cursor& x) { return (x.n - (x.nch - 1) * C::P) >> 4; };
  auto load_new = [&](const Cursor& x) {
    if (warp != owner(x)) return;
    const int sh = x.gg / g.nkvs, gl = x.gg % g.nkvs;
    const __nv_bfloat16* base = qkv + (size_t)x.m * g.t * g.Qs + (size_t)sh * g.Qs;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = lane + 32 * i, kv = idx / (HD / 8), c8 = idx % (HD / 8);
      if (idx < 2 * HD / 8)
        kvn[i] = *reinterpret_cast<const uint4*>(base + (size_t)(g.nqs + kv * g.nkvs + gl) * HD + 8 * c8);
    }
  };
  load_q(cu);
  load_new(cu);
  store_q();
  if (!csync()) return;

  float O[HD / 8][4];
#pragma unroll
  for (int t8 = 0; t8 < HD / 8; ++t8) O[t8][0] = O[t8][1] = O[t8][2] = O[t8][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gq and gq + 8
  int c_seg = cu.c;                                          // first chunk of the current piece
  // pieces of a split (sequence, kv head) this CTA leaves: only its first and last can be such
  int np_mine = 0, pm[2] = {0, 0}, pgg[2] = {0, 0}, pnch[2] = {0, 0};
  int sb = 0;  // which max / sum buffer the next piece end uses
  long long pub[2] = {0, 0};
  for (int k = 0; k < nu; ++k) {
    const int st = k % C::NS;
    if (!tc::mbar_wait(full0 + 8 * st, (k / C::NS) & 1)) {
      if (lane == 0) atomicExch(err, 42u);
      return;
    }
    const bool last = k + 1 == nu;
    const bool seg_end = last || cu.c + 1 == cu.nch;
    const int np = min(C::P, cu.n + 1 - cu.c * C::P);  // valid positions of this chunk
    uint8_t* stage = ring + (size_t)st * C::STAGE;
    if (cu.c + 1 == cu.nch && warp == owner(cu)) {
      // The cache row of the new token may be read before the append has written it: its
      // staged copy is replaced by the values from qkv (the ones the append writes).
      const int rn = np - 1;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int idx = lane + 32 * i, kv = idx / (HD / 8), c8 = idx % (HD / 8);
        if (idx < 2 * HD / 8)
          *reinterpret_cast<uint4*>(stage + kv * C::KVB + (c8 >> 3) * C::BOX + rn * 128 + (((c8 & 7) ^ (rn & 7)) << 4)) =
              kvn[i];
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    Cursor nx = cu;
    if (!last) advance(g, lens, nx);
    if (seg_end && !last) {  // in flight while this chunk is computed
      load_q(nx);
      load_new(nx);
    }
    if (w0 < np) {
      const uint32_t kb = tc::smem_u32(stage), vb = kb + C::KVB;
      if (np < w0 + 16) {  // staged rows past the end may hold anything (NaN too): P V must see 0
        for (int i = lane; i < (w0 + 16 - np) * (HD / 8); i += 32) {
          const int r = np + i / (HD / 8), c8 = i % (HD / 8);
          *reinterpret_cast<uint4*>(stage + C::KVB + (c8 >> 3) * C::BOX + r * 128 + ((c8 & 7) << 4)) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // ordered before the producer's next copy into this stage
        __syncwarp();
      }
      // S = Q K^T over this warp's 16 positions: 2 n-tiles of 8
      float S[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
#pragma unroll
      for (int k0 = 0; k0 < HD; k0 += 32) {
        uint32_t a[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          ldsm_x4(q_base + (lane & 15) * C::QSTR + (k0 + 16 * h + 8 * (lane >> 4)) * 2, a[h][0], a[h][1], a[h][2],
                  a[h][3]);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t b0, b1, b2, b3;  // positions w0 + 8j + (0..7) x dims k0 + 0/8/16/24
          ldsm_x4(kb + sw_off<HD>(w0 + 8 * j + (lane & 7), k0 + 8 * (lane >> 3)), b0, b1, b2, b3);
          mma_bf16_16816(S[j], a[0][0], a[0][1], a[0][2], a[0][3], b0, b1);
          mma_bf16_16816(S[j], a[1][0], a[1][1], a[1][2], a[1][3], b2, b3);
        }
      }
      // scale, mask, online softmax (position w0 is valid, so each row's new max is finite)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) S[j][i] = (w0 + 8 * j + 2 * qq + (i & 1) < np) ? S[j][i] * scale : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(S[j][0], S[j][1]));
        mx1 = fmaxf(mx1, fmaxf(S[j][2], S[j][3]));
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = __expf(m0 - mn0), al1 = __expf(m1 - mn1);  // 0 on the first chunk
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        S[j][0] = __expf(S[j][0] - mn0);
        S[j][1] = __expf(S[j][1] - mn0);
        S[j][2] = __expf(S[j][2] - mn1);
        S[j][3] = __expf(S[j][3] - mn1);
      }
      l0 = l0 * al0 + ((S[0][0] + S[0][1]) + (S[1][0] + S[1][1]));  // this lane's share; quad-summed at the end
      l1 = l1 * al1 + ((S[0][2] + S[0][3]) + (S[1][2] + S[1][3]));
#pragma unroll
      for (int t8 = 0; t8 < HD / 8; ++t8) {
        O[t8][0] *= al0;
        O[t8][1] *= al0;
        O[t8][2] *= al1;
        O[t8][3] *= al1;
      }
      // O += P V: the S fragments are the A fragment of the 16-position k-step
      const uint32_t a0 = pack_bf16(S[0][0], S[0][1]), a1 = pack_bf16(S[0][2], S[0][3]);
      const uint32_t a2 = pack_bf16(S[1][0], S[1][1]), a3 = pack_bf16(S[1][2], S[1][3]);
      const int r = w0 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int t16 = 0; t16 < HD / 16; ++t16) {
        uint32_t b0, b1, b2, b3;  // (positions +0 / +8) x (dims 16 t16 + 0 / + 8), transposed
        ldsm_x4_t(vb + sw_off<HD>(r, 16 * t16 + 8 * (lane >> 4)), b0, b1, b2, b3);
        mma_bf16_16816(O[2 * t16], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(O[2 * t16 + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    if (seg_end) {
      // The piece of (m, gg) in this CTA ends: the warps' states merge through this stage's
      // memory ([CW][16][HD] fp32 fills it exactly), then the stage goes back to the producer.
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, o);
        l1 += __shfl_xor_sync(kFull, l1, o);
      }
      // two buffers: a warp may reach the next piece end while another still reads these
      float* mw = mlw + sb * 2 * C::CW * 16;
      float* lw = mw + C::CW * 16;
      sb ^= 1;
      if (qq == 0) {
        mw[warp * 16 + gq] = m0;
        mw[warp * 16 + gq + 8] = m1;
        lw[warp * 16 + gq] = l0;
        lw[warp * 16 + gq + 8] = l1;
      }
      // every warp is past this chunk's reads of the stage and of sQ once all have arrived
      // below; the raw p.v goes to the stage first (the warps' factors are applied when summing)
      if (!csync()) return;
      float* wred = reinterpret_cast<float*>(stage) + (size_t)warp * 16 * HD;
#pragma unroll
      for (int t8 = 0; t8 < HD / 8; ++t8) {  // row r at r * HD, its 8-float groups permuted by r & 7
        const int d0 = (8 * t8) ^ ((gq & 7) << 3);
        *reinterpret_cast<float2*>(wred + gq * HD + d0 + 2 * qq) = make_float2(O[t8][0], O[t8][1]);
        *reinterpret_cast<float2*>(wred + (gq + 8) * HD + d0 + 2 * qq) = make_float2(O[t8][2], O[t8][3]);
      }
      if (!last) store_q();  // the next piece's q (sQ is free: every warp is past the csync above)
      if (!csync()) return;
      const float* red = reinterpret_cast<const float*>(stage);
      const int sh = cu.gg / g.nkvs, gl = cu.gg % g.nkvs;
      __nv_bfloat16* out = o_in + (size_t)cu.m * g.n_q * HD + (size_t)(sh * g.nqs + gl * g.G) * HD;
      const bool whole = c_seg == 0 && cu.c + 1 == cu.nch;
      float* part = whole ? nullptr : part_ptr(g, ws, cu.m, cu.gg, c_seg);
      for (int e = tid; e < g.G * HD; e += C::NT) {  // the warps' p.v, scaled to the common max, warp order
        const int hi = e / HD, d = e % HD, ds = d ^ ((hi & 7) << 3);
        float Mx = mw[hi];
#pragma unroll
        for (int w = 1; w < C::CW; ++w) Mx = fmaxf(Mx, mw[w * 16 + hi]);
        float v = 0.f, Lx = 0.f;
#pragma unroll
        for (int w = 0; w < C::CW; ++w) {
          const float f = __expf(mw[w * 16 + hi] - Mx);  // 0 for a warp with no valid position
          v += red[((size_t)w * 16 + hi) * HD + ds] * f;
          Lx += lw[w * 16 + hi] * f;
        }
        if (whole) out[e] = __float2bfloat16_rn(v / Lx);
        else part[e] = v;
      }
      if (!whole && tid < g.G) {
        float Mx = mw[tid], Lx = 0.f;
        for (int w = 1; w < C::CW; ++w) Mx = fmaxf(Mx, mw[w * 16 + tid]);
        for (int w = 0; w < C::CW; ++w) Lx += lw[w * 16 + tid] * __expf(mw[w * 16 + tid] - Mx);
        part[g.G * HD + tid] = Mx;
        part[g.G * HD + g.G + tid] = Lx;
      }
      if (!whole && np_mine < 2) {
        pm[np_mine] = cu.m;
        pgg[np_mine] = cu.gg;
        pnch[np_mine] = cu.nch;
        pub[np_mine] = u0 + k - cu.c;  // unit of chunk 0 of (m, gg)
        ++np_mine;
      }
      // The stage returns to the producer once every warp has arrived below, each after its
      // own reads of it; the generic writes to it are ordered before the next copy.
      fence_proxy_async_smem();
#pragma unroll
      for (int t8 = 0; t8 < HD / 8; ++t8) O[t8][0] = O[t8][1] = O[t8][2] = O[t8][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
      c_seg = 0;
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(empty0 + 8 * st);  // the stage goes back to the producer
    cu = nx;
  }

  // Split (sequence, kv head)s: count this CTA's pieces in (after the append has reset the
  // counters); the CTA that brings the last piece merges them all, in position order.
  tc::griddep_wait();
  if (np_mine == 0) return;
  __threadfence();
  if (!csync()) return;
  for (int i = 0; i < np_mine; ++i) {
    if (tid == 0) {
      int npc = 0;
      for_pieces(U, nct, pub[i], pnch[i], [&](int cs) {
        if (npc < kMaxPieces) s_pc[npc] = cs;
        ++npc;
      });
      s_npc = npc;
      s_last = atomicAdd(counter_ptr(g, ws, pm[i], pgg[i]), 1u) + 1u == (unsigned)npc;
    }
    if (!csync()) return;
    if (s_last) {
      __threadfence();
      const int m = pm[i], gg = pgg[i], sh = gg / g.nkvs, gl = gg % g.nkvs, npc = s_npc;
      __nv_bfloat16* out = o_in + (size_t)m * g.n_q * HD + (size_t)(sh * g.nqs + gl * g.G) * HD;
      for (int e = tid; e < g.G * HD; e += C::NT) {
        const int hi = e / HD;
        float Mx = -INFINITY, acc = 0.f, Lx = 0.f;
        auto max_of = [&](int cs) { Mx = fmaxf(Mx, __ldcg(part_ptr(g, ws, m, gg, cs) + g.G * HD + hi)); };
        auto add_of = [&](int cs) {
          const float* pc = part_ptr(g, ws, m, gg, cs);
          const float f = __expf(__ldcg(pc + g.G * HD + hi) - Mx);
          acc += __ldcg(pc + e) * f;
          Lx += __ldcg(pc + g.G * HD + g.G + hi) * f;
        };
        if (npc <= kMaxPieces) {
          for (int j = 0; j < npc; ++j) max_of(s_pc[j]);
          for (int j = 0; j < npc; ++j) add_of(s_pc[j]);
        } else {  // many CTAs on one sequence (tiny workloads): walk the boundaries again
          for_pieces(U, nct, pub[i], pnch[i], max_of);
          for_pieces(U, nct, pub[i], pnch[i], add_of);
        }
        out[e] = __float2bfloat16_rn(acc / Lx);
      }
    }
    if (!csync()) return;  // s_last, s_npc and s_pc are read before they are written again
  }
}

}  // namespace

size_t attn_workspace_bytes(int t, int M, int L, int n_q, int n_kv, int hd) {
  const AttnGeo g = attn_geo(t, M, L, n_q, n_kv, hd);
  const size_t nch = (size_t)(L + g.P - 1) / g.P;
  return (size_t)M * n_kv * nch * g.G * (hd + 2) * sizeof(float) + (size_t)M * n_kv * sizeof(unsigned);
}

bool attn_supported(int hd, int G) { return (hd == 64 || hd == 128 || hd == 256) && G >= 1 && G <= 16; }

static int sm_count_here() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

cudaError_t launch_attn_decode(int t, int M, int L, int n_q, int n_kv, int hd, const __nv_bfloat16* qkv,
                               __nv_bfloat16* kc, __nv_bfloat16* vc, const int32_t* lens, __nv_bfloat16* o_in,
                               float* ws, unsigned* err, cudaStream_t st) {
  const AttnGeo g = attn_geo(t, M, L, n_q, n_kv, hd);
  append_kernel<<<dim3(M, n_kv), dim3(hd / 8, 2), 0, st>>>(g, qkv, lens, kc, vc, ws, o_in);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tm[2];
  for (int i = 0; i < 2; ++i) {  // the cache as [t M n_kv/t L rows][hd], boxes of P rows x 64 dims
    const cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)t * M * (n_kv / t) * L};
    const cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)g.P}, es[2] = {1, 1};
    if (enc(&tm[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, i ? (void*)vc : (void*)kc, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const float scale = 1.0f / sqrtf((float)hd);
  const int grid = sm_count_here();
  auto launch = [&](auto kernel, size_t smem, int threads) {
    cudaError_t a = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (a != cudaSuccess) return a;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlaps the append
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    a = cudaLaunchKernelEx(&cfg, kernel, tm[0], tm[1], g, scale, qkv, lens, ws, o_in, err);
    note_launch();
    return a != cudaSuccess ? a : cudaGetLastError();
  };
  if (hd == 64) return launch(attn_kernel<64>, ACfg<64>::SMEM, ACfg<64>::NT + 32);
  if (hd == 128) return launch(attn_kernel<128>, ACfg<128>::SMEM, ACfg<128>::NT + 32);
  return launch(attn_kernel<256>, ACfg<256>::SMEM, ACfg<256>::NT + 32);
}

}  // namespace tpx
