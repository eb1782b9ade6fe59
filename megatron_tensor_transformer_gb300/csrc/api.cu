// C ABI of libtpx.so: argument checks, packed-weight descriptors, kernel dispatch.
// Every check runs on the host before anything is enqueued.
#include <atomic>
#include <mutex>
#include <chrono>
#include <cstring>
#include <thread>

#include "attn.h"
#include "common.cuh"
#include "fused.h"
#include "pack.h"
#include "ring.h"
#include "skinny.h"
#include "small.h"
#include "tc.h"

namespace tpx {
static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace tpx

using namespace tpx;

namespace {

constexpr uint64_t kAlign = 256;
inline uint64_t align_up(uint64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// k per chunk of the decode kernels: 32 bf16 or 64 e4m3 values (16 bytes per thread per row)
inline int k_chunk(int wtype) { return wtype == TP_FP8_E4M3 ? 64 : 32; }

tp_status check_shape(const tp_shape* sh, int kind) {
  if (!sh) return TP_ERR_INVALID_ARG;
  if (kind < TP_W_GATE_UP || kind > TP_W_EMBED) return TP_ERR_INVALID_ARG;
  if (sh->wtype != TP_BF16 && sh->wtype != TP_FP8_E4M3) return TP_ERR_INVALID_ARG;
  const int t = sh->t;
  if (t != 1 && t != 2 && t != 4 && t != 8) return TP_ERR_SHAPE;
  if (sh->d <= 0) return TP_ERR_SHAPE;
  if (sh->d % 32) return TP_ERR_ALIGN;
  if (kind == TP_W_VOCAB || kind == TP_W_EMBED) {
    if (sh->vocab <= 0) return TP_ERR_SHAPE;
    if (sh->wtype != TP_BF16) return TP_ERR_UNSUPPORTED;  // the vocabulary edges are bf16 only
    if (sh->d % 64) return TP_ERR_ALIGN;                   // 64-wide k-blocks of the lm_head GEMM
    return TP_OK;
  }
  const int kc = k_chunk(sh->wtype);
  if (kind == TP_W_GATE_UP || kind == TP_W_DOWN) {
    if (sh->ffn <= 0 || sh->ffn % t) return TP_ERR_SHAPE;
    const int fs = sh->ffn / t;
    if (fs % 8) return TP_ERR_ALIGN;                       // gate/up interleave blocks of 8
    if (kind == TP_W_GATE_UP && sh->d % kc) return TP_ERR_ALIGN;
    if (kind == TP_W_DOWN && fs % kc) return TP_ERR_ALIGN;
  } else {
    const int nq = sh->n_q_heads, nkv = sh->n_kv_heads, hd = sh->head_dim;
    if (nq <= 0 || nkv <= 0 || hd <= 0) return TP_ERR_SHAPE;
    if (nq % nkv) return TP_ERR_SHAPE;                      // GQA groups
    if (nq % t || nkv % t) return TP_ERR_SHAPE;             // t divides the q and kv heads
    if (hd % 8) return TP_ERR_ALIGN;
    if (kind == TP_W_QKV && sh->d % kc) return TP_ERR_ALIGN;
    if (kind == TP_W_O && (nq / t * hd) % kc) return TP_ERR_ALIGN;
  }
  return TP_OK;
}

void geometry(const tp_shape* sh, int kind, int64_t* rows, int64_t* K, int64_t* out_cols) {
  const int t = sh->t;
  switch (kind) {
    case TP_W_GATE_UP: *rows = 2LL * sh->ffn / t; *K = sh->d; *out_cols = sh->ffn; break;
    case TP_W_DOWN: *rows = sh->d; *K = sh->ffn / t; *out_cols = sh->d; break;
    case TP_W_QKV:
      *rows = (int64_t)(sh->n_q_heads + 2 * sh->n_kv_heads) / t * sh->head_dim;
      *K = sh->d;
      *out_cols = (int64_t)(sh->n_q_heads + 2 * sh->n_kv_heads) * sh->head_dim;
      break;
    case TP_W_VOCAB:
    case TP_W_EMBED: {
      const int64_t q = 128LL * t, vp = ((int64_t)sh->vocab + q - 1) / q * q;  // padded vocabulary
      *rows = vp / t;
      *K = sh->d;
      *out_cols = kind == TP_W_VOCAB ? sh->vocab : sh->d;
      break;
    }
    default:
      *rows = sh->d; *K = (int64_t)sh->n_q_heads / t * sh->head_dim; *out_cols = sh->d; break;
  }
}

tp_status check_desc(const tp_packed_desc* d, int kind, const void* w) {
  if (!d || !w) return TP_ERR_INVALID_ARG;
  if (!aligned16(w)) return TP_ERR_ALIGN;
  if (d->magic != TP_DESC_MAGIC || d->layout_version != TP_LAYOUT_VERSION) return TP_ERR_LAYOUT_MISMATCH;
  if (d->kind != kind) return TP_ERR_LAYOUT_MISMATCH;
  tp_packed_desc ref;
  if (tp_describe(&d->shape, kind, &ref) != TP_OK) return TP_ERR_LAYOUT_MISMATCH;
  if (ref.rows_per_shard != d->rows_per_shard || ref.k_per_shard != d->k_per_shard ||
      ref.shard_payload_bytes != d->shard_payload_bytes || ref.scales_offset != d->scales_offset ||
      ref.shard_stride_bytes != d->shard_stride_bytes || ref.total_bytes != d->total_bytes ||
      ref.wtype != d->wtype)
    return TP_ERR_LAYOUT_MISMATCH;
  return TP_OK;
}

tp_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TP_OK : TP_ERR_CUDA; }

// Workspace: shard partials of one token block [t][min(M,64)][N] fp32, then row-tile tickets.
uint64_t partials_bytes(int t, int M, int N) {
  const int mb = M < kSkinnyMaxM ? M : kSkinnyMaxM;
  return align_up((uint64_t)t * mb * N * 4);
}
uint64_t ticket_bytes(int N) { return align_up((uint64_t)(N / 8 + 1) * 4); }
// Workspace layout: [stream-K scratch][row-tile tickets][shard partials for min(M, 64) tokens].
// Everything that must persist between calls (tickets, barrier words) sits at offsets that do
// not depend on M, so calls with different M can share one workspace.
uint64_t sk_bytes() { return align_up(tc_streamk_bytes()); }

// Prefill with e4m3 weights (M > 64): room to widen the largest weight of the shape to bf16
// once per call; 0 otherwise.  It follows the partials in the workspace.
uint64_t widen_bytes(const tp_shape* sh, int M) {
  if (sh->wtype != TP_FP8_E4M3 || M <= kFusedMaxM) return 0;
  uint64_t b = 0;
  const uint64_t d = (uint64_t)sh->d;
  if (sh->ffn > 0) b = 4ull * sh->ffn * d;  // gate + up, 2 bytes each
  if (sh->n_q_heads > 0 && sh->head_dim > 0) {
    const uint64_t q = (uint64_t)(sh->n_q_heads + 2 * sh->n_kv_heads) * sh->head_dim * d * 2;
    if (q > b) b = q;
  }
  return align_up(b);
}

// FP8 x FP8 (TP_F_FP8_ACT): the quantised activations of the widest GEMM input of the block
// ([M][width] e4m3) and their per-token scales; it follows the widening scratch.
uint64_t act_width(const tp_shape* sh) {
  uint64_t w = (uint64_t)sh->d;
  if (sh->ffn > 0 && (uint64_t)sh->ffn > w) w = (uint64_t)sh->ffn;
  if (sh->n_q_heads > 0 && sh->head_dim > 0 && (uint64_t)sh->n_q_heads * sh->head_dim > w)
    w = (uint64_t)sh->n_q_heads * sh->head_dim;
  return w;
}
uint64_t act_bytes(const tp_shape* sh, int M, uint32_t flags) {
  if (!(flags & TP_F_FP8_ACT) || sh->wtype != TP_FP8_E4M3 || M <= 0) return 0;
  return align_up((uint64_t)M * act_width(sh)) + align_up((uint64_t)M * 4);
}

// RMSNorm scratch of the fused layer (per-tile sums of squares, two per-token factor arrays);
// it follows the partials in the workspace.
uint64_t norm_bytes(int d) { return align_up((uint64_t)fused_norm_words(d) * 4); }
float* norm_region(void* ws, const tp_shape& sh, int M) {
  return reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sk_bytes() + ticket_bytes(sh.d) +
                                  partials_bytes(sh.t, M, sh.d));
}

// The widening scratch of a workspace of ws_bytes, or nullptr when it does not fit.
void* widen_scratch(void* ws, size_t ws_bytes, const tp_shape& sh, int M, uint64_t need) {
  if (!ws || need == 0) return nullptr;
  const uint64_t off = sk_bytes() + ticket_bytes(sh.d) + partials_bytes(sh.t, M, sh.d) + norm_bytes(sh.d);
  if (ws_bytes < off + need) return nullptr;
  return static_cast<uint8_t*>(ws) + off;
}

// The FP8 x FP8 activation scratch of a workspace: codes, then scales; false if it does not fit.
bool act_scratch(void* ws, size_t ws_bytes, const tp_shape& sh, int M, uint32_t flags, uint8_t*& q, float*& s) {
  const uint64_t need = act_bytes(&sh, M, flags);
  if (!ws || need == 0) return false;
  const uint64_t off = sk_bytes() + ticket_bytes(sh.d) + partials_bytes(sh.t, M, sh.d) + norm_bytes(sh.d) +
                       widen_bytes(&sh, M);
  if (ws_bytes < off + need) return false;
  q = static_cast<uint8_t*>(ws) + off;
  s = reinterpret_cast<float*>(q + align_up((uint64_t)M * act_width(&sh)));
  return true;
}

}  // namespace

extern "C" {

const char* tp_status_str(tp_status s) {
  switch (s) {
    case TP_OK: return "TP_OK";
    case TP_ERR_INVALID_ARG: return "TP_ERR_INVALID_ARG";
    case TP_ERR_SHAPE: return "TP_ERR_SHAPE";
    case TP_ERR_ALIGN: return "TP_ERR_ALIGN";
    case TP_ERR_LAYOUT_MISMATCH: return "TP_ERR_LAYOUT_MISMATCH";
    case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE";
    case TP_ERR_CUDA: return "TP_ERR_CUDA";
    case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT";
    case TP_ERR_DEVICE_TIMEOUT: return "TP_ERR_DEVICE_TIMEOUT";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED";
  }
  return "TP_ERR_UNKNOWN";
}

uint64_t tp_launch_count(void) { return g_launches.load(); }

tp_status tp_describe(const tp_shape* shape, int32_t kind, tp_packed_desc* desc) {
  if (!desc) return TP_ERR_INVALID_ARG;
  tp_status st = check_shape(shape, kind);
  if (st != TP_OK) return st;
  memset(desc, 0, sizeof(*desc));
  desc->magic = TP_DESC_MAGIC;
  desc->layout_version = TP_LAYOUT_VERSION;
  desc->kind = kind;
  desc->wtype = shape->wtype;
  desc->shape = *shape;
  int64_t rows, K, oc;
  geometry(shape, kind, &rows, &K, &oc);
  desc->rows_per_shard = rows;
  desc->k_per_shard = K;
  const bool fp8 = shape->wtype == TP_FP8_E4M3;
  desc->shard_payload_bytes = (uint64_t)rows * K * (fp8 ? 1 : 2);
  desc->scales_offset = fp8 ? align_up(desc->shard_payload_bytes) : desc->shard_payload_bytes;
  desc->shard_stride_bytes = align_up(desc->scales_offset + (fp8 ? (uint64_t)rows * 4 : 0));
  desc->total_bytes = desc->shard_stride_bytes * shape->t;
  return TP_OK;
}

size_t tp_packed_bytes(const tp_shape* shape, int32_t kind) {
  tp_packed_desc d;
  return tp_describe(shape, kind, &d) == TP_OK ? (size_t)d.total_bytes : 0;
}

tp_status tp_partition_weights(const tp_shape* shape, int32_t kind, const void* W0, const void* W1,
                               void* packed, size_t packed_bytes, tp_packed_desc* desc_out,
                               void* stream) {
  tp_packed_desc d;
  tp_status st = tp_describe(shape, kind, &d);
  if (st != TP_OK) return st;
  if (!W0 || !packed || !desc_out) return TP_ERR_INVALID_ARG;
  if ((kind == TP_W_GATE_UP) != (W1 != nullptr)) return TP_ERR_INVALID_ARG;
  if (!aligned16(W0) || (W1 && !aligned16(W1)) || !aligned16(packed)) return TP_ERR_ALIGN;
  if (packed_bytes < d.total_bytes) return TP_ERR_INVALID_ARG;
  PackGeom g{};
  g.kind = kind;
  g.colpar = kind == TP_W_GATE_UP || kind == TP_W_QKV || kind == TP_W_VOCAB;
  g.vocab = shape->vocab;
  g.fp8 = shape->wtype == TP_FP8_E4M3;
  g.t = shape->t;
  int64_t rows, K, oc;
  geometry(shape, kind, &rows, &K, &oc);
  g.rows = (int)rows;
  g.K = (int)K;
  g.out_cols = (int)oc;
  g.ffn = shape->ffn;
  g.n_q = shape->n_q_heads;
  g.n_kv = shape->n_kv_heads;
  g.hd = shape->head_dim;
  g.W0 = static_cast<const uint16_t*>(W0);
  g.W1 = static_cast<const uint16_t*>(W1);
  g.shard_stride = d.shard_stride_bytes;
  g.scales_offset = d.scales_offset;
  st = cuda_status(launch_pack(g, static_cast<uint8_t*>(packed), S(stream)));
  // forwards may start reading weights before earlier work on their stream has finished
  // (programmatic dependent launch), so the packed buffer is complete when this returns
  if (st == TP_OK) st = cuda_status(cudaStreamSynchronize(S(stream)));
  if (st == TP_OK) *desc_out = d;
  return st;
}

size_t tp_workspace_bytes(const tp_shape* shape, int32_t M, uint32_t flags) {
  if (!shape || M < 0 || shape->t <= 0 || shape->d <= 0) return 0;
  return (size_t)(sk_bytes() + partials_bytes(shape->t, M, shape->d) + ticket_bytes(shape->d) +
                  norm_bytes(shape->d) + widen_bytes(shape, M) + act_bytes(shape, M, flags));
}

}  // extern "C"

// ---------------------------------------------------------------- forward paths

namespace {

using bf16 = __nv_bfloat16;

// Kernel choice: the tcgen05 GEMM where the geometry allows it and M is above the
// threshold, the mma.sync skinny kernel otherwise; flags can force either one.
constexpr int kTcMinM = 0;  // tcgen05 wherever the geometry allows: with PDL it wins the whole step
constexpr uint32_t kKernelFlags = TP_F_KERNEL_SKINNY | TP_F_KERNEL_TC;
constexpr uint32_t kFwdFlags = TP_F_UNFUSED_REDUCE | kKernelFlags | TP_F_SERIAL | TP_F_SPLIT_BLOCK | TP_F_FP8_ACT |
                               TP_F_FP8_HILO | TP_F_FOLD_NORM;

bool pick_tc(uint32_t flags, int rows, int K, bool fp8, int M) {
  if (flags & TP_F_KERNEL_SKINNY) return false;
  if (!tc_supported(rows, K, fp8)) return false;
  if (flags & TP_F_KERNEL_TC) return true;
  // e4m3 decode: the mma.sync kernels, which widen in registers, stream faster (measured, 70B
  // layer at M = 16: 215 us TMA-fed, 236 us register-direct, 292 us for the tcgen05 path)
  if (fp8 && M <= kFusedMaxM) return false;
  return M > kTcMinM;
}

bool bad_kernel_flags(uint32_t flags) { return (flags & kKernelFlags) == kKernelFlags; }

int device_sms() {  // cached per device ordinal
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Stream-K scratch of the tcgen05 kernel: [pieces][item tickets], or none.
void set_streamk(TcArgs& a, void* sk_ws) {
  if (!sk_ws) return;
  a.pieces = static_cast<float*>(sk_ws);
  a.item_tickets = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(sk_ws) + tc_streamk_bytes() -
                                               (size_t)kTcMaxStreamkItems * 4);
}

// The TMA-fed e4m3 decode kernel: e4m3 weights, 1..32 tokens, 128-row tiles, unless the
// mma.sync kernel is asked for, and only with a workspace (its piece slots go in the stream-K
// scratch, its counters in the zero-between-calls ticket words that follow it).
bool pick_ring(uint32_t flags, const tp_packed_desc* d, int rows, int K, int M, bool rowpar, const void* ws,
               size_t ws_bytes) {
  if (d->wtype != TP_FP8_E4M3 || (flags & TP_F_KERNEL_SKINNY) || !ws || d->shape.t > 8) return false;
  if (!ring_supported(rows, K, M, d->shape.t)) return false;
  if (ring_pieces_bytes(M) > sk_bytes()) return false;
  if (ring_counter_words(rows, d->shape.t, rowpar) * 4 > ticket_bytes(rowpar ? rows : d->shape.d)) return false;
  return ws_bytes >= sk_bytes() + ticket_bytes(rowpar ? rows : d->shape.d) && aligned16(ws);
}

RingArgs ring_args(const tp_packed_desc* d, const void* w, int rows, int K, const bf16* x, int ldx, int M,
                   void* ws) {
  RingArgs r{};
  r.w = static_cast<const uint8_t*>(w);
  r.shard_stride = d->shard_stride_bytes;
  r.scales_offset = d->scales_offset;
  r.rows = rows;
  r.K = K;
  r.t = d->shape.t;
  r.x = x;
  r.ldx = ldx;
  r.M = M;
  r.pieces = static_cast<float*>(ws);
  r.counters = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + sk_bytes());
  r.err = tc_error_word();
  return r;
}

// Weights of a tcgen05 launch.  e4m3 weights stream as they are (widened in shared memory by
// the kernel), except for prefill-sized M when the workspace has room: then each shard is
// widened once to bf16 codes in the scratch and the GEMM runs in bf16, with the same per-row
// scales in its epilogue (same values, same bits).  That GEMM must not start streaming its
// weights before the widening has finished, so it is launched without programmatic overlap.
tp_status tc_weights(TcArgs& a, const tp_packed_desc* d, const void* w, int M, void* ws, size_t ws_bytes,
                     cudaStream_t st, bool& pdl) {
  const bool fp8 = d->wtype == TP_FP8_E4M3;
  a.w = static_cast<const uint8_t*>(w);
  a.shard_stride = d->shard_stride_bytes;
  a.fp8 = fp8;
  a.scales_offset = d->scales_offset;
  if (fp8) {
    a.scales = reinterpret_cast<const float*>(static_cast<const uint8_t*>(w) + d->scales_offset);
    a.scales_stride = d->shard_stride_bytes / 4;
  }
  const uint64_t need = (uint64_t)d->rows_per_shard * d->k_per_shard * 2 * d->shape.t;
  void* scratch = fp8 ? widen_scratch(ws, ws_bytes, d->shape, M, widen_bytes(&d->shape, M)) : nullptr;
  if (scratch && need <= widen_bytes(&d->shape, M)) {
    if (launch_widen_e4m3(static_cast<const uint8_t*>(w), d->shard_stride_bytes, (int)d->rows_per_shard,
                          (int)d->k_per_shard, d->shape.t, static_cast<bf16*>(scratch), st) != cudaSuccess)
      return TP_ERR_CUDA;
    a.w = static_cast<const uint8_t*>(scratch);
    a.shard_stride = (uint64_t)d->rows_per_shard * d->k_per_shard * 2;
    a.fp8 = 0;
    pdl = false;
  }
  return TP_OK;
}

// FP8 x FP8 (TP_F_FP8_ACT): the e4m3 weights as they are (the MMA reads them directly), the
// activations x [M][width] quantised per token into the workspace scratch.
tp_status x8_setup(TcArgs& a, const tp_packed_desc* d, const void* w, const bf16* x, int width, int M, void* ws,
                   size_t ws_bytes, uint32_t flags, cudaStream_t st) {
  uint8_t* q = nullptr;
  float* s = nullptr;
  if (!act_scratch(ws, ws_bytes, d->shape, M, flags, q, s) || (uint64_t)width > act_width(&d->shape))
    return TP_ERR_WORKSPACE;
  if (launch_quantize_fp8_per_token(x, width, M, width, q, width, s, st) != cudaSuccess) return TP_ERR_CUDA;
  a.w = static_cast<const uint8_t*>(w);
  a.shard_stride = d->shard_stride_bytes;
  a.fp8 = 1;
  a.scales_offset = d->scales_offset;
  a.scales = reinterpret_cast<const float*>(static_cast<const uint8_t*>(w) + d->scales_offset);
  a.scales_stride = d->shard_stride_bytes / 4;
  a.x8 = 1;
  a.xq = q;
  a.tok_scales = s;
  return TP_OK;
}

// Column-parallel half over token blocks of at most 64 (skinny) or all tokens (tcgen05).
// in_scale (nullable, tcgen05 path only): per-token factors on the accumulators (a folded RMSNorm).
tp_status run_colpar(const tp_packed_desc* d, const void* w, const bf16* x, int M, void* out,
                     int mode, cudaStream_t st, uint32_t flags = 0, void* sk_ws = nullptr, size_t ws_bytes = 0,
                     const float* in_scale = nullptr) {
  const int t = d->shape.t;
  const int rows = (int)d->rows_per_shard, K = (int)d->k_per_shard;
  const int ldo = mode == COLPAR_SWIGLU ? rows / 2 * t : rows * t;
  const size_t osz = mode == COLPAR_F32 ? 4 : 2;
  if (d->wtype == TP_FP8_E4M3 && (flags & TP_F_FP8_ACT)) {  // e4m3 x e4m3 on the tensor cores
    if (rows % 128 != 0 || K % 128 != 0) return TP_ERR_UNSUPPORTED;
    TcArgs a{};
    a.mode = mode == COLPAR_SWIGLU ? TC_COLPAR_SWIGLU : (mode == COLPAR_F32 ? TC_COLPAR_F32 : TC_COLPAR_BF16);
    const tp_status xs = x8_setup(a, d, w, x, K, M, sk_ws, ws_bytes, flags, st);
    if (xs != TP_OK) return xs;
    a.t = t;
    a.rows = rows;
    a.K = K;
    a.x = x;
    a.ldx = K;
    a.M = M;
    a.out = out;
    a.ldo = ldo;
    set_streamk(a, sk_ws);
    return launch_tc(a, st, (flags & TP_F_SERIAL) == 0) == cudaSuccess ? TP_OK : TP_ERR_CUDA;
  }
  if (pick_tc(flags, rows, K, d->wtype == TP_FP8_E4M3, M)) {
    TcArgs a{};
    a.mode = mode == COLPAR_SWIGLU ? TC_COLPAR_SWIGLU : (mode == COLPAR_F32 ? TC_COLPAR_F32 : TC_COLPAR_BF16);
    bool pdl = (flags & TP_F_SERIAL) == 0;
    const tp_status ws_st = tc_weights(a, d, w, M, sk_ws, ws_bytes, st, pdl);
    if (ws_st != TP_OK) return ws_st;
    a.t = t;
    a.rows = rows;
    a.K = K;
    a.x = x;
    a.ldx = K;
    a.M = M;
    a.out = out;
    a.ldo = ldo;
    a.tok_scales = in_scale;
    set_streamk(a, sk_ws);
    return launch_tc(a, st, pdl) == cudaSuccess ? TP_OK : TP_ERR_CUDA;
  }
  if (in_scale) return TP_ERR_UNSUPPORTED;
  if ((mode == COLPAR_BF16 || mode == COLPAR_SWIGLU) &&
      pick_ring(flags, d, rows, K, M, false, sk_ws, ws_bytes)) {
    RingArgs r = ring_args(d, w, rows, K, x, K, M, sk_ws);
    if (!r.err) return TP_ERR_CUDA;
    r.rowpar = 0;
    r.mode = mode;
    r.out = out;
    r.ldo = ldo;
    return launch_ring(r, st, (flags & TP_F_SERIAL) == 0) == cudaSuccess ? TP_OK : TP_ERR_CUDA;
  }
  for (int m0 = 0; m0 < M; m0 += kSkinnyMaxM) {
    ColparArgs a{};
    a.w = static_cast<const uint8_t*>(w);
    a.shard_stride = d->shard_stride_bytes;
    a.scales_offset = d->scales_offset;
    a.rows = rows;
    a.K = K;
    a.t = t;
    a.x = x + (size_t)m0 * K;
    a.ldx = K;
    a.M = M - m0 < kSkinnyMaxM ? M - m0 : kSkinnyMaxM;
    a.out = static_cast<uint8_t*>(out) + (size_t)m0 * ldo * osz;
    a.ldo = ldo;
    a.mode = mode;
    cudaError_t e = launch_colpar(a, d->wtype == TP_FP8_E4M3, st);
    if (e != cudaSuccess) return TP_ERR_CUDA;
  }
  return TP_OK;
}

// Row-parallel half: partials_user != NULL -> write [t][M][N] partials only; otherwise fold
// (in the CTA, by ticket, or unfused through tp_reduce_partials) into y with the residual.
// norm_ss (nullable, the chained tcgen05 path only): per (token, 32-row group) sums of squares of
// the stored y, for the next RMSNorm.
tp_status run_rowpar(const tp_packed_desc* d, const void* w, const bf16* a_in, int M,
                     const bf16* res, bf16* y, float* partials_user, void* ws, size_t ws_bytes,
                     uint32_t flags, cudaStream_t st, float* norm_ss = nullptr) {
  const int t = d->shape.t;
  const int N = (int)d->rows_per_shard, K = (int)d->k_per_shard;
  const RowparPlan plan = rowpar_plan(N, t);
  if (plan.R == 0) return TP_ERR_ALIGN;
  const bool unfused = (flags & TP_F_UNFUSED_REDUCE) != 0;
  const bool x8 = d->wtype == TP_FP8_E4M3 && (flags & TP_F_FP8_ACT);
  if (x8 && (N % 128 != 0 || K % 128 != 0)) return TP_ERR_UNSUPPORTED;
  const bool tc = x8 || pick_tc(flags, N, K, d->wtype == TP_FP8_E4M3, M);
  const bool ring = !tc && pick_ring(flags, d, N, K, M, true, ws, ws_bytes);
  const bool need_ws = !partials_user && (unfused || plan.S > 1 || tc || ring);
  float* wsP = nullptr;
  unsigned* tickets = nullptr;
  void* sk_ws = nullptr;
  if (need_ws) {
    const uint64_t pb = partials_bytes(t, M, N);
    if (!ws || ws_bytes < sk_bytes() + pb + ticket_bytes(N)) return TP_ERR_WORKSPACE;
    if (!aligned16(ws)) return TP_ERR_ALIGN;
    sk_ws = ws;
    tickets = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + sk_bytes());
    wsP = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sk_bytes() + ticket_bytes(N));
  }
  if (tc) {
    TcArgs a{};
    bool pdl = (flags & TP_F_SERIAL) == 0;
    const tp_status ws_st = x8 ? x8_setup(a, d, w, a_in, K * t, M, ws, ws_bytes, flags, st)
                               : tc_weights(a, d, w, M, need_ws ? ws : nullptr, ws_bytes, st, pdl);
    if (ws_st != TP_OK) return ws_st;
    const uint8_t* xq0 = a.xq;
    const float* ts0 = a.tok_scales;
    a.t = t;
    a.rows = N;
    a.K = K;
    a.ldx = K * t;
    a.ldy = N;
    set_streamk(a, sk_ws);
    // Fused default: chain every shard's k-blocks into one accumulator (no partials round
    // trip) when its row tiles fill the GPU; otherwise (decode: few 128-row tiles) per-shard
    // items, which do fill it, then the fold kernel over the partials.
    const int tiles = N / 128 * ((M + 255) / 256), sms = device_sms();
    const bool fold_pass = !partials_user && (unfused || (M <= kSkinnyMaxM && tiles < sms && tiles * t >= sms));
    if (!fold_pass) {
      // one launch over all tokens: per-shard partials only, or every shard chained, + residual
      a.mode = partials_user ? TC_ROWPAR_SHARD : TC_ROWPAR_CHAIN;
      a.x = a_in;
      a.M = M;
      a.residual = res;
      a.y = y;
      a.partials = partials_user;
      a.pM = M;
      if (norm_ss && (partials_user || N % 32 != 0)) return TP_ERR_UNSUPPORTED;
      a.norm_ss = norm_ss;
      return launch_tc(a, st, pdl) == cudaSuccess ? TP_OK : TP_ERR_CUDA;
    }
    if (norm_ss) return TP_ERR_UNSUPPORTED;
    for (int m0 = 0; m0 < M; m0 += kSkinnyMaxM) {  // per-shard partials in the workspace
      const int mb = M - m0 < kSkinnyMaxM ? M - m0 : kSkinnyMaxM;
      a.mode = TC_ROWPAR_SHARD;
      a.x = a_in + (size_t)m0 * K * t;
      if (x8) {
        a.xq = xq0 + (size_t)m0 * K * t;
        a.tok_scales = ts0 + m0;
      }
      a.M = mb;
      a.residual = res ? res + (size_t)m0 * N : nullptr;
      a.y = y + (size_t)m0 * N;
      a.partials = wsP;
      a.pM = mb;
      // unfused: per-shard partials, then the fold kernel
      if (launch_tc(a, st, pdl) != cudaSuccess) return TP_ERR_CUDA;
      if (launch_reduce(wsP, t, mb, N, a.residual, a.y, st) != cudaSuccess) return TP_ERR_CUDA;
    }
    return TP_OK;
  }
  if (norm_ss) return TP_ERR_UNSUPPORTED;
  if (ring) {
    RingArgs r = ring_args(d, w, N, K, a_in, K * t, M, ws);
    if (!r.err) return TP_ERR_CUDA;
    r.rowpar = 1;
    r.residual = res;
    r.y = y;
    r.ldy = N;
    r.partials = partials_user ? partials_user : wsP;
    r.pM = M;
    r.mode = (partials_user || unfused) ? FOLD_NONE : FOLD_TICKET;
    if (launch_ring(r, st, (flags & TP_F_SERIAL) == 0) != cudaSuccess) return TP_ERR_CUDA;
    if (!partials_user && unfused && launch_reduce(wsP, t, M, N, res, y, st) != cudaSuccess) return TP_ERR_CUDA;
    return TP_OK;
  }
  for (int m0 = 0; m0 < M; m0 += kSkinnyMaxM) {
    const int mb = M - m0 < kSkinnyMaxM ? M - m0 : kSkinnyMaxM;
    RowparArgs a{};
    a.w = static_cast<const uint8_t*>(w);
    a.shard_stride = d->shard_stride_bytes;
    a.scales_offset = d->scales_offset;
    a.N = N;
    a.K = K;
    a.t = t;
    a.x = a_in + (size_t)m0 * K * t;
    a.ldx = K * t;
    a.M = mb;
    a.residual = res ? res + (size_t)m0 * N : nullptr;
    a.y = y ? y + (size_t)m0 * N : nullptr;
    a.ldy = N;
    a.tickets = tickets;
    if (partials_user) {
      a.partials = partials_user + (size_t)m0 * N;
      a.pM = M;
      a.fold = FOLD_NONE;
    } else if (unfused) {
      a.partials = wsP;
      a.pM = mb;
      a.fold = FOLD_NONE;
    } else {
      a.partials = wsP;
      a.pM = mb;
      a.fold = plan.S == 1 ? FOLD_IN_CTA : FOLD_TICKET;
    }
    cudaError_t e = launch_rowpar(a, d->wtype == TP_FP8_E4M3, plan, st);
    if (e != cudaSuccess) return TP_ERR_CUDA;
    if (!partials_user && unfused) {
      e = launch_reduce(wsP, t, mb, N, a.residual, a.y, st);
      if (e != cudaSuccess) return TP_ERR_CUDA;
    }
  }
  return TP_OK;
}

// Sync words of the fused block kernel: inside the stream-K ticket area, past the grid-barrier
// words that the stream-K path uses (offsets independent of M, zero between calls).
unsigned* fused_sync(void* ws) {
  return reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + tc_streamk_bytes() -
                                     (size_t)kTcMaxStreamkItems * 4) + 64;
}

// One persistent launch for the whole block (decode token counts, bf16 or e4m3 weights), unless
// the flags ask for separate launches or for the mma.sync kernels.  e4m3 blocks split the
// activations into hi/lo e4m3 codes, unless TP_F_KERNEL_TC alone asks for widened weights.
bool pick_fused(uint32_t flags, const tp_packed_desc* d1, const tp_packed_desc* d2, int M) {
  if (flags & (TP_F_UNFUSED_REDUCE | TP_F_KERNEL_SKINNY | TP_F_SPLIT_BLOCK | TP_F_FP8_ACT)) return false;
  return fused_supported((int)d1->rows_per_shard, d1->shape.d, (int)d2->k_per_shard, M, d1->shape.t,
                         d1->wtype == TP_FP8_E4M3);
}

// e4m3 decode blocks: the largest token count that runs on hi/lo activation codes by default
constexpr int kHiloDefaultMaxM = 32;

tp_status run_fused(int kind, const tp_packed_desc* d1, const void* w1, const tp_packed_desc* d2, const void* w2,
                    const bf16* x, const bf16* res, int M, bf16* y, bf16* mid, bf16* mid2, void* ws,
                    uint32_t flags, cudaStream_t st, float* in_scale = nullptr, int in_norm = 0,
                    float* out_rms = nullptr, float eps = 0.f) {
  FusedArgs a{};
  a.kind = kind;
  a.t = d1->shape.t;
  a.M = M;
  a.d = d1->shape.d;
  a.fp8 = d1->wtype == TP_FP8_E4M3;
  // hi/lo activation codes by default up to kHiloDefaultMaxM tokens; above, widening the weights
  // measured faster (70B e4m3 layer at 64 tokens: 323.6 against 385.0 us)
  a.split = a.fp8 && ((flags & TP_F_FP8_HILO) != 0 || ((flags & TP_F_KERNEL_TC) == 0 && M <= kHiloDefaultMaxM));
  a.w1 = static_cast<const uint8_t*>(w1);
  a.stride1 = d1->shard_stride_bytes;
  a.scales1 = d1->scales_offset;
  a.scales2 = d2->scales_offset;
  a.rows1 = (int)d1->rows_per_shard;
  a.w2 = static_cast<const uint8_t*>(w2);
  a.stride2 = d2->shard_stride_bytes;
  a.K2 = (int)d2->k_per_shard;
  a.x = x;
  a.mid = mid;
  a.mid2 = mid2;
  a.n_q = d1->shape.n_q_heads;
  a.n_kv = d1->shape.n_kv_heads;
  a.hd = d1->shape.head_dim;
  a.residual = res;
  a.y = y;
  a.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sk_bytes() + ticket_bytes(a.d));
  a.sync = fused_sync(ws);
  a.in_scale = in_scale;
  a.in_norm = in_norm;
  a.out_rms = out_rms;
  a.norm_ss = norm_region(ws, d1->shape, M);
  a.eps = eps;
  a.err = tc_error_word();
  if (!a.err) return TP_ERR_CUDA;
  const bool pdl = (flags & TP_F_SERIAL) == 0;
  // split activations: the input's per-token maxima, computed just before the block
  if (a.split && launch_token_absmax(x, M, a.d, fused_xmax_words(a.sync, a.d), pdl, st) != cudaSuccess)
    return TP_ERR_CUDA;
  return launch_fused(a, st, pdl) == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

bool same_block(const tp_shape& a, const tp_shape& b, bool mlp) {
  if (a.d != b.d || a.t != b.t || a.wtype != b.wtype) return false;
  if (mlp) return a.ffn == b.ffn;
  return a.n_q_heads == b.n_q_heads && a.n_kv_heads == b.n_kv_heads && a.head_dim == b.head_dim;
}

// A prefill layer asked to fold its norms (TP_F_FOLD_NORM) whose four GEMMs all run on the tcgen05
// path, with the chained row-parallel fold: the RMSNorms fold into their epilogues.
bool prefill_fold(uint32_t flags, const tp_packed_desc* q, const tp_packed_desc* o, const tp_packed_desc* gu,
                  const tp_packed_desc* dn, int M) {
  if (!(flags & TP_F_FOLD_NORM) || M <= kFusedMaxM ||
      (flags & (TP_F_FP8_ACT | TP_F_SPLIT_BLOCK | TP_F_KERNEL_SKINNY | TP_F_UNFUSED_REDUCE)))
    return false;
  if (q->shape.d % 32 != 0) return false;
  for (const tp_packed_desc* d : {q, o, gu, dn})
    if (!pick_tc(flags, (int)d->rows_per_shard, (int)d->k_per_shard, d->wtype == TP_FP8_E4M3, M)) return false;
  return true;
}

}  // namespace

extern "C" {

tp_status tp_colpar_forward(const tp_packed_desc* desc, const void* w, const void* x, int32_t M,
                            void* out, void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  if (!desc) return TP_ERR_INVALID_ARG;
  const int kind = desc->kind;
  if (kind != TP_W_GATE_UP && kind != TP_W_QKV) return TP_ERR_INVALID_ARG;
  tp_status st = check_desc(desc, kind, w);
  if (st != TP_OK) return st;
  if (M < 0 || (M > 0 && (!x || !out))) return TP_ERR_INVALID_ARG;
  if ((flags & ~(uint32_t)(TP_F_FP32_COLPAR_OUT | kKernelFlags | TP_F_SERIAL | TP_F_FP8_ACT)) || bad_kernel_flags(flags))
    return TP_ERR_INVALID_ARG;
  const bool f32 = (flags & TP_F_FP32_COLPAR_OUT) != 0;
  if (f32 && kind == TP_W_GATE_UP) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  if (!aligned16(x) || !aligned16(out)) return TP_ERR_ALIGN;
  const int mode = kind == TP_W_GATE_UP ? COLPAR_SWIGLU : (f32 ? COLPAR_F32 : COLPAR_BF16);
  void* sk_ws = nullptr;  // optional stream-K scratch: the head of a tp_workspace_bytes() workspace
  if (ws && aligned16(ws) && ws_bytes >= sk_bytes()) sk_ws = ws;
  return run_colpar(desc, w, static_cast<const bf16*>(x), M, out, mode, S(stream), flags, sk_ws,
                    sk_ws ? ws_bytes : 0);
}

tp_status tp_rowpar_partials(const tp_packed_desc* desc, const void* w, const void* a, int32_t M,
                             float* partials, void* stream) {
  if (!desc) return TP_ERR_INVALID_ARG;
  const int kind = desc->kind;
  if (kind != TP_W_DOWN && kind != TP_W_O) return TP_ERR_INVALID_ARG;
  tp_status st = check_desc(desc, kind, w);
  if (st != TP_OK) return st;
  if (M < 0 || (M > 0 && (!a || !partials))) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  if (!aligned16(a) || !aligned16(partials)) return TP_ERR_ALIGN;
  return run_rowpar(desc, w, static_cast<const bf16*>(a), M, nullptr, nullptr, partials, nullptr, 0,
                    0, S(stream));
}

tp_status tp_rowpar_forward(const tp_packed_desc* desc, const void* w, const void* a,
                            const void* residual, int32_t M, void* y, void* ws, size_t ws_bytes,
                            uint32_t flags, void* stream) {
  if (!desc) return TP_ERR_INVALID_ARG;
  const int kind = desc->kind;
  if (kind != TP_W_DOWN && kind != TP_W_O) return TP_ERR_INVALID_ARG;
  tp_status st = check_desc(desc, kind, w);
  if (st != TP_OK) return st;
  if ((flags & ~kFwdFlags) || bad_kernel_flags(flags))
    return TP_ERR_INVALID_ARG;
  if (M < 0 || (M > 0 && (!a || !y))) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  if (!aligned16(a) || !aligned16(y) || (residual && !aligned16(residual))) return TP_ERR_ALIGN;
  return run_rowpar(desc, w, static_cast<const bf16*>(a), M, static_cast<const bf16*>(residual),
                    static_cast<bf16*>(y), nullptr, ws, ws_bytes, flags, S(stream));
}

tp_status tp_reduce_partials(const float* partials, int32_t t, int32_t M, int32_t d,
                             const void* residual, void* y, void* stream) {
  if (t != 1 && t != 2 && t != 4 && t != 8) return TP_ERR_SHAPE;
  if (M < 0 || d <= 0) return TP_ERR_INVALID_ARG;
  if (M > 0 && (!partials || !y)) return TP_ERR_INVALID_ARG;
  if (d % 8) return TP_ERR_ALIGN;
  if (M == 0) return TP_OK;
  if (!aligned16(partials) || !aligned16(y) || (residual && !aligned16(residual))) return TP_ERR_ALIGN;
  return cuda_status(launch_reduce(partials, t, M, d, static_cast<const bf16*>(residual),
                                   static_cast<bf16*>(y), S(stream)));
}

tp_status tp_mlp_forward(const tp_packed_desc* gu, const void* gu_w, const tp_packed_desc* dn,
                         const void* dn_w, const void* x, const void* residual, int32_t M, void* y,
                         void* h_out, void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  tp_status st = check_desc(gu, TP_W_GATE_UP, gu_w);
  if (st != TP_OK) return st;
  st = check_desc(dn, TP_W_DOWN, dn_w);
  if (st != TP_OK) return st;
  if (!same_block(gu->shape, dn->shape, true)) return TP_ERR_LAYOUT_MISMATCH;
  if ((flags & ~kFwdFlags) || bad_kernel_flags(flags))
    return TP_ERR_INVALID_ARG;
  if (M < 0 || (M > 0 && (!x || !y || !h_out))) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  if (!aligned16(x) || !aligned16(y) || !aligned16(h_out) || (residual && !aligned16(residual)))
    return TP_ERR_ALIGN;
  if (!ws || ws_bytes < tp_workspace_bytes(&gu->shape, M, flags)) return TP_ERR_WORKSPACE;
  cudaStream_t s = S(stream);
  if (pick_fused(flags, gu, dn, M))
    return run_fused(FUSED_MLP, gu, gu_w, dn, dn_w, static_cast<const bf16*>(x), static_cast<const bf16*>(residual),
                     M, static_cast<bf16*>(y), static_cast<bf16*>(h_out), static_cast<bf16*>(h_out), ws, flags, s);
  st = run_colpar(gu, gu_w, static_cast<const bf16*>(x), M, h_out, COLPAR_SWIGLU, s, flags,
                  ws, ws_bytes);
  if (st != TP_OK) return st;
  return run_rowpar(dn, dn_w, static_cast<const bf16*>(h_out), M, static_cast<const bf16*>(residual),
                    static_cast<bf16*>(y), nullptr, ws, ws_bytes, flags, s);
}

tp_status tp_proj_forward(const tp_packed_desc* qkv, const void* qkv_w, const tp_packed_desc* o,
                          const void* o_w, const void* x, const void* residual, int32_t M, void* y,
                          void* qkv_out, void* o_in, void* ws, size_t ws_bytes, uint32_t flags,
                          void* stream) {
  tp_status st = check_desc(qkv, TP_W_QKV, qkv_w);
  if (st != TP_OK) return st;
  st = check_desc(o, TP_W_O, o_w);
  if (st != TP_OK) return st;
  if (!same_block(qkv->shape, o->shape, false)) return TP_ERR_LAYOUT_MISMATCH;
  if ((flags & ~kFwdFlags) || bad_kernel_flags(flags))
    return TP_ERR_INVALID_ARG;
  if (M < 0 || (M > 0 && (!x || !y || !qkv_out || !o_in))) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  if (!aligned16(x) || !aligned16(y) || !aligned16(qkv_out) || !aligned16(o_in) ||
      (residual && !aligned16(residual)))
    return TP_ERR_ALIGN;
  const tp_shape& sh = qkv->shape;
  if (!ws || ws_bytes < tp_workspace_bytes(&sh, M, flags)) return TP_ERR_WORKSPACE;
  cudaStream_t s = S(stream);
  if (pick_fused(flags, qkv, o, M))
    return run_fused(FUSED_PROJ, qkv, qkv_w, o, o_w, static_cast<const bf16*>(x), static_cast<const bf16*>(residual),
                     M, static_cast<bf16*>(y), static_cast<bf16*>(qkv_out), static_cast<bf16*>(o_in), ws, flags, s);
  st = run_colpar(qkv, qkv_w, static_cast<const bf16*>(x), M, qkv_out, COLPAR_BF16, s, flags,
                  ws, ws_bytes);
  if (st != TP_OK) return st;
  st = cuda_status(launch_attn1(static_cast<const bf16*>(qkv_out), M, sh.n_q_heads, sh.n_kv_heads,
                                sh.head_dim, sh.t, static_cast<bf16*>(o_in), s));
  if (st != TP_OK) return st;
  return run_rowpar(o, o_w, static_cast<const bf16*>(o_in), M, static_cast<const bf16*>(residual),
                    static_cast<bf16*>(y), nullptr, ws, ws_bytes, flags, s);
}

size_t tp_layer_scratch_bytes(const tp_shape* sh, int32_t M) {
  if (!sh || M < 0 || sh->d <= 0 || sh->head_dim <= 0 || sh->ffn <= 0) return 0;
  const uint64_t Q = (uint64_t)(sh->n_q_heads + 2 * sh->n_kv_heads) * sh->head_dim;
  const uint64_t Mu = (uint64_t)M;
  // normed input, h1, attention output, normed h1 ([M, d] each), qkv [M, Q], h [M, ffn]
  return (size_t)(4 * align_up(Mu * sh->d * 2) + align_up(Mu * Q * 2) + align_up(Mu * sh->ffn * 2));
}

tp_status tp_layer_forward(const tp_packed_desc* qkv, const void* qkv_w, const tp_packed_desc* o,
                           const void* o_w, const tp_packed_desc* gu, const void* gu_w,
                           const tp_packed_desc* dn, const void* dn_w, const void* x, int32_t M, void* y,
                           float eps, void* scratch, size_t scratch_bytes, void* ws, size_t ws_bytes,
                           uint32_t flags, void* stream) {
  if (!qkv || !o || !gu || !dn) return TP_ERR_INVALID_ARG;
  const tp_shape& sa = qkv->shape;
  const tp_shape& sm = gu->shape;
  if (sa.d != sm.d || sa.t != sm.t || sa.wtype != sm.wtype) return TP_ERR_LAYOUT_MISMATCH;
  if (M < 0 || !(eps >= 0.f) || (M > 0 && (!x || !y || !scratch))) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  tp_shape both = sa;
  both.ffn = sm.ffn;
  if (scratch_bytes < tp_layer_scratch_bytes(&both, M)) return TP_ERR_WORKSPACE;
  if (!aligned16(scratch)) return TP_ERR_ALIGN;
  const uint64_t d = sa.d, Q = (uint64_t)(sa.n_q_heads + 2 * sa.n_kv_heads) * sa.head_dim;
  uint8_t* p = static_cast<uint8_t*>(scratch);
  void* a = p;  p += align_up((uint64_t)M * d * 2);
  void* h1 = p; p += align_up((uint64_t)M * d * 2);
  void* oi = p; p += align_up((uint64_t)M * d * 2);
  void* b = p;  p += align_up((uint64_t)M * d * 2);
  void* qk = p; p += align_up((uint64_t)M * Q * 2);
  void* h = p;
  if (pick_fused(flags, qkv, o, M) && pick_fused(flags, gu, dn, M)) {
    // Decode: two launches.  RMSNorm (gain 1) scales each token by 1/sqrt(mean(x^2) + eps), a
    // per-token factor, so it multiplies the column-parallel accumulators; the attention
    // block computes its input's factors itself and, in its fold, those of h1 for the MLP
    // block (the single-GPU form of the sequence-parallel "reduce-scatter, norm, all-gather").
    tp_status st = check_desc(qkv, TP_W_QKV, qkv_w);
    if (st == TP_OK) st = check_desc(o, TP_W_O, o_w);
    if (st == TP_OK) st = check_desc(gu, TP_W_GATE_UP, gu_w);
    if (st == TP_OK) st = check_desc(dn, TP_W_DOWN, dn_w);
    if (st != TP_OK) return st;
    if (!same_block(qkv->shape, o->shape, false) || !same_block(gu->shape, dn->shape, true))
      return TP_ERR_LAYOUT_MISMATCH;
    if ((flags & ~kFwdFlags) || bad_kernel_flags(flags)) return TP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return TP_ERR_ALIGN;
    if (!ws || ws_bytes < tp_workspace_bytes(&both, M, flags)) return TP_ERR_WORKSPACE;
    if (!aligned16(ws)) return TP_ERR_ALIGN;
    float* nb = norm_region(ws, both, M) + kFusedMaxMWords * (d / 128);
    float* r_x = nb;                    // factors of x (computed by the attention block)
    float* r_h1 = nb + kFusedMaxMWords;  // factors of h1 (computed by its fold)
    cudaStream_t s = S(stream);
    st = run_fused(FUSED_PROJ, qkv, qkv_w, o, o_w, static_cast<const bf16*>(x), static_cast<const bf16*>(x), M,
                   static_cast<bf16*>(h1), static_cast<bf16*>(qk), static_cast<bf16*>(oi), ws, flags, s, r_x, 1,
                   r_h1, eps);
    if (st != TP_OK) return st;
    return run_fused(FUSED_MLP, gu, gu_w, dn, dn_w, static_cast<const bf16*>(h1), static_cast<const bf16*>(h1), M,
                     static_cast<bf16*>(y), static_cast<bf16*>(h), static_cast<bf16*>(h), ws, flags, s, r_h1, 0,
                     nullptr, eps);
  }
  if (prefill_fold(flags, qkv, o, gu, dn, M)) {
    // Prefill: the RMSNorms as per-token factors on the column-parallel GEMMs' accumulators.  The
    // factors of x come from one pass over x; the o_proj epilogue, which writes h1, also leaves
    // h1's sums of squares per 32-row group, summed in order into h1's factors.  The normalised
    // activations are never written (their room in the scratch holds the sums and the factors).
    tp_status st = check_desc(qkv, TP_W_QKV, qkv_w);
    if (st == TP_OK) st = check_desc(o, TP_W_O, o_w);
    if (st == TP_OK) st = check_desc(gu, TP_W_GATE_UP, gu_w);
    if (st == TP_OK) st = check_desc(dn, TP_W_DOWN, dn_w);
    if (st != TP_OK) return st;
    if (!same_block(qkv->shape, o->shape, false) || !same_block(gu->shape, dn->shape, true))
      return TP_ERR_LAYOUT_MISMATCH;
    if ((flags & ~kFwdFlags) || bad_kernel_flags(flags)) return TP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return TP_ERR_ALIGN;
    if (!ws || ws_bytes < tp_workspace_bytes(&both, M, flags)) return TP_ERR_WORKSPACE;
    if (!aligned16(ws)) return TP_ERR_ALIGN;
    float* ss = static_cast<float*>(a);    // [M][d / 32] sums of squares of h1
    float* r_x = static_cast<float*>(b);   // [M] factors of x, then [M] factors of h1
    float* r_h1 = r_x + align_up((uint64_t)M * 4) / 4;
    cudaStream_t s = S(stream);
    st = cuda_status(launch_rms_factors(static_cast<const bf16*>(x), eps, M, (int)d, r_x, s));
    if (st == TP_OK)
      st = run_colpar(qkv, qkv_w, static_cast<const bf16*>(x), M, qk, COLPAR_BF16, s, flags, ws, ws_bytes, r_x);
    if (st == TP_OK)
      st = cuda_status(launch_attn1(static_cast<const bf16*>(qk), M, sa.n_q_heads, sa.n_kv_heads, sa.head_dim, sa.t,
                                    static_cast<bf16*>(oi), s));
    if (st == TP_OK)
      st = run_rowpar(o, o_w, static_cast<const bf16*>(oi), M, static_cast<const bf16*>(x), static_cast<bf16*>(h1),
                      nullptr, ws, ws_bytes, flags, s, ss);
    if (st == TP_OK) st = cuda_status(launch_rms_factors_from_ss(ss, eps, M, (int)d, r_h1, s));
    if (st == TP_OK)
      st = run_colpar(gu, gu_w, static_cast<const bf16*>(h1), M, h, COLPAR_SWIGLU, s, flags, ws, ws_bytes, r_h1);
    if (st == TP_OK)
      st = run_rowpar(dn, dn_w, static_cast<const bf16*>(h), M, static_cast<const bf16*>(h1), static_cast<bf16*>(y),
                      nullptr, ws, ws_bytes, flags, s);
    return st;
  }
  tp_status st = tp_rmsnorm(x, nullptr, eps, M, (int32_t)d, a, stream);
  if (st != TP_OK) return st;
  st = tp_proj_forward(qkv, qkv_w, o, o_w, a, x, M, h1, qk, oi, ws, ws_bytes, flags, stream);
  if (st != TP_OK) return st;
  st = tp_rmsnorm(h1, nullptr, eps, M, (int32_t)d, b, stream);
  if (st != TP_OK) return st;
  return tp_mlp_forward(gu, gu_w, dn, dn_w, b, h1, M, y, h, ws, ws_bytes, flags, stream);
}

size_t tp_attn_workspace_bytes(const tp_shape* sh, int32_t M, int32_t L) {
  if (!sh || M < 0 || L <= 0 || check_shape(sh, TP_W_QKV) != TP_OK) return 0;
  return attn_workspace_bytes(sh->t, M, L, sh->n_q_heads, sh->n_kv_heads, sh->head_dim);
}

tp_status tp_attn_decode(const tp_shape* sh, const void* qkv, void* k_cache, void* v_cache, int32_t L,
                         const int32_t* lens, int32_t M, void* o_in, void* ws, size_t ws_bytes, void* stream) {
  tp_status st = check_shape(sh, TP_W_QKV);
  if (st != TP_OK) return st;
  if (M < 0 || L <= 0) return TP_ERR_INVALID_ARG;
  if (!attn_supported(sh->head_dim, sh->n_q_heads / sh->n_kv_heads)) return TP_ERR_UNSUPPORTED;
  if ((int64_t)M * sh->n_kv_heads * L >= (int64_t(1) << 31)) return TP_ERR_UNSUPPORTED;  // cache rows: int32
  if (M == 0) return TP_OK;
  if (!qkv || !k_cache || !v_cache || !lens || !o_in || !ws) return TP_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o_in) || !aligned16(ws))
    return TP_ERR_ALIGN;
  if (ws_bytes < tp_attn_workspace_bytes(sh, M, L)) return TP_ERR_WORKSPACE;
  unsigned* err = tc_error_word();
  if (!err) return TP_ERR_CUDA;
  return cuda_status(launch_attn_decode(sh->t, M, L, sh->n_q_heads, sh->n_kv_heads, sh->head_dim,
                                        static_cast<const bf16*>(qkv), static_cast<bf16*>(k_cache),
                                        static_cast<bf16*>(v_cache), lens, static_cast<bf16*>(o_in),
                                        static_cast<float*>(ws), err, S(stream)));
}

tp_status tp_quantize_fp8_per_token(const void* x, int32_t M, int32_t K, void* q, float* s, void* stream) {
  if (M < 0 || K <= 0 || K % 8 != 0) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  if (!x || !q || !s) return TP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(s)) return TP_ERR_ALIGN;
  return cuda_status(launch_quantize_fp8_per_token(static_cast<const bf16*>(x), K, M, K, static_cast<uint8_t*>(q), K,
                                                   s, S(stream)));
}

size_t tp_attn_block_workspace_bytes(const tp_shape* sh, int32_t M, int32_t L, uint32_t flags) {
  if (!sh || M < 0 || L <= 0) return 0;
  const size_t proj = tp_workspace_bytes(sh, M, flags), attn = tp_attn_workspace_bytes(sh, M, L);
  if (proj == 0 || attn == 0) return 0;
  return (size_t)align_up(proj) + attn;
}

tp_status tp_attn_block_forward(const tp_packed_desc* qkv, const void* qkv_w, const tp_packed_desc* o,
                                const void* o_w, const void* x, const void* residual, int32_t M, void* k_cache,
                                void* v_cache, int32_t L, const int32_t* lens, void* y, void* qkv_out, void* o_in,
                                void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  tp_status st = check_desc(qkv, TP_W_QKV, qkv_w);
  if (st != TP_OK) return st;
  st = check_desc(o, TP_W_O, o_w);
  if (st != TP_OK) return st;
  if (!same_block(qkv->shape, o->shape, false)) return TP_ERR_LAYOUT_MISMATCH;
  if ((flags & ~kFwdFlags) || bad_kernel_flags(flags)) return TP_ERR_INVALID_ARG;
  const tp_shape& sh = qkv->shape;
  if (M < 0 || L <= 0) return TP_ERR_INVALID_ARG;
  if (!attn_supported(sh.head_dim, sh.n_q_heads / sh.n_kv_heads)) return TP_ERR_UNSUPPORTED;
  if ((int64_t)M * sh.n_kv_heads * L >= (int64_t(1) << 31)) return TP_ERR_UNSUPPORTED;
  if (M == 0) return TP_OK;
  if (!x || !y || !qkv_out || !o_in || !k_cache || !v_cache || !lens) return TP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(qkv_out) || !aligned16(o_in) || !aligned16(k_cache) ||
      !aligned16(v_cache) || (residual && !aligned16(residual)))
    return TP_ERR_ALIGN;
  const size_t proj = align_up(tp_workspace_bytes(&sh, M, flags));
  if (!ws || ws_bytes < tp_attn_block_workspace_bytes(&sh, M, L, flags)) return TP_ERR_WORKSPACE;
  if (!aligned16(ws)) return TP_ERR_ALIGN;
  unsigned* err = tc_error_word();
  if (!err) return TP_ERR_CUDA;
  cudaStream_t s = S(stream);
  st = run_colpar(qkv, qkv_w, static_cast<const bf16*>(x), M, qkv_out, COLPAR_BF16, s, flags, ws, proj);
  if (st != TP_OK) return st;
  st = cuda_status(launch_attn_decode(sh.t, M, L, sh.n_q_heads, sh.n_kv_heads, sh.head_dim,
                                      static_cast<const bf16*>(qkv_out), static_cast<bf16*>(k_cache),
                                      static_cast<bf16*>(v_cache), lens, static_cast<bf16*>(o_in),
                                      reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + proj), err, s));
  if (st != TP_OK) return st;
  return run_rowpar(o, o_w, static_cast<const bf16*>(o_in), M, static_cast<const bf16*>(residual),
                    static_cast<bf16*>(y), nullptr, ws, proj, flags, s);
}

tp_status tp_lm_head_forward(const tp_packed_desc* desc, const void* w, const void* x, int32_t M, float* logits,
                             void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  tp_status st = check_desc(desc, TP_W_VOCAB, w);
  if (st != TP_OK) return st;
  if ((flags & ~(TP_F_SERIAL | TP_F_KERNEL_TC)) != 0) return TP_ERR_INVALID_ARG;
  if (M < 0 || (M > 0 && (!x || !logits))) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  if (!aligned16(x) || !aligned16(logits)) return TP_ERR_ALIGN;
  const int rows = (int)desc->rows_per_shard, K = (int)desc->k_per_shard;
  if (!tc_supported(rows, K, false)) return TP_ERR_UNSUPPORTED;
  TcArgs a{};
  a.mode = TC_COLPAR_F32;
  a.w = static_cast<const uint8_t*>(w);
  a.shard_stride = desc->shard_stride_bytes;
  a.t = desc->shape.t;
  a.rows = rows;
  a.K = K;
  a.x = static_cast<const bf16*>(x);
  a.ldx = K;
  a.M = M;
  a.out = logits;
  a.ldo = desc->shape.vocab;  // the shards' slices, concatenated, cut to the real ids
  a.ncols = desc->shape.vocab;
  if (ws && aligned16(ws) && ws_bytes >= sk_bytes()) set_streamk(a, ws);
  return launch_tc(a, S(stream), (flags & TP_F_SERIAL) == 0) == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

tp_status tp_embed_lookup(const tp_packed_desc* desc, const void* w, const int32_t* ids, int32_t M, void* x,
                          void* stream) {
  tp_status st = check_desc(desc, TP_W_EMBED, w);
  if (st != TP_OK) return st;
  if (M < 0 || (M > 0 && (!ids || !x))) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  if (!aligned16(x)) return TP_ERR_ALIGN;
  return cuda_status(launch_embed(static_cast<const uint8_t*>(w), desc->shard_stride_bytes,
                                  (int)desc->rows_per_shard, desc->shape.t, desc->shape.vocab, desc->shape.d, ids,
                                  M, static_cast<bf16*>(x), S(stream)));
}

tp_status tp_rmsnorm(const void* x, const void* gain, float eps, int32_t M, int32_t d, void* out,
                     void* stream) {
  if (M < 0 || d <= 0 || !(eps >= 0.f)) return TP_ERR_INVALID_ARG;
  if (M > 0 && (!x || !out)) return TP_ERR_INVALID_ARG;
  if (d % 8) return TP_ERR_ALIGN;
  if (M == 0) return TP_OK;
  if (!aligned16(x) || !aligned16(out) || (gain && !aligned16(gain))) return TP_ERR_ALIGN;
  return cuda_status(launch_rmsnorm(static_cast<const bf16*>(x), static_cast<const bf16*>(gain), eps, M,
                                    d, static_cast<bf16*>(out), S(stream)));
}

tp_status tp_sync(void* stream, int32_t timeout_ms) {
  const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
  for (;;) {
    const cudaError_t e = cudaStreamQuery(S(stream));
    if (e == cudaSuccess) break;
    if (e != cudaErrorNotReady) return TP_ERR_CUDA;
    if (std::chrono::steady_clock::now() >= deadline) return TP_ERR_TIMEOUT;
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  if (tc_take_device_error() != 0) return TP_ERR_DEVICE_TIMEOUT;
  return TP_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free row-parallel
//
// Some callers cannot allocate device memory: a plugin living inside a host framework
// whose caching allocator owns the whole device (a side cudaMalloc fragments its pool
// or is forbidden), or code on a latency-critical path where cudaMalloc's implicit
// synchronisation is not acceptable.  tp_rowpar_forward_noalloc serves them: its scratch
// (shard partials and row-tile tickets) lives in the file-scope array below, so the call
// allocates nothing.  Every GPU that loads the library holds this array until exit.

namespace {

constexpr size_t kNoallocScratchBytes = 32u << 20;  // 32 MiB
static __device__ __align__(256) unsigned char tpx_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[128] = {};  // device address of the array, per device ordinal

// Host code cannot use the array's name as a device address: resolve it once per device,
// with that device current.
tp_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return TP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, tpx_noalloc_scratch) != cudaSuccess || !p) return TP_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return TP_OK;
}

}  // namespace

extern "C" size_t tp_noalloc_scratch_capacity(void) { return kNoallocScratchBytes; }

extern "C" tp_status tp_rowpar_forward_noalloc(const tp_packed_desc* desc, const void* w, const void* a,
                                               const void* residual, int32_t M, void* y, uint32_t flags,
                                               void* stream) {
  if (!desc) return TP_ERR_INVALID_ARG;
  const int kind = desc->kind;
  if (kind != TP_W_DOWN && kind != TP_W_O) return TP_ERR_INVALID_ARG;
  tp_status st = check_desc(desc, kind, w);
  if (st != TP_OK) return st;
  if ((flags & ~kFwdFlags) || bad_kernel_flags(flags))
    return TP_ERR_INVALID_ARG;
  // the per-token e4m3 activations would need a region of their own in the array
  if (flags & TP_F_FP8_ACT) return TP_ERR_UNSUPPORTED;
  if (M < 0 || (M > 0 && (!a || !y))) return TP_ERR_INVALID_ARG;
  if (M == 0) return TP_OK;
  if (!aligned16(a) || !aligned16(y) || (residual && !aligned16(residual))) return TP_ERR_ALIGN;
  const int t = desc->shape.t, N = (int)desc->rows_per_shard;
  const uint64_t pb = partials_bytes(t, M, N), need = sk_bytes() + pb + ticket_bytes(N);
  if (need > kNoallocScratchBytes) return TP_ERR_WORKSPACE;  // beyond the static scratch
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != TP_OK) return st;
  // the tickets must start at zero; the partials are fully written before they are read
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  if (cudaMemsetAsync(sc + sk_bytes(), 0, ticket_bytes(N), S(stream)) != cudaSuccess ||
      cudaMemsetAsync(sc + tc_streamk_bytes() - (size_t)kTcMaxStreamkItems * 4, 0, (size_t)kTcMaxStreamkItems * 4,
                      S(stream)) != cudaSuccess)
    return TP_ERR_CUDA;
  return run_rowpar(desc, w, static_cast<const bf16*>(a), M, static_cast<const bf16*>(residual),
                    static_cast<bf16*>(y), nullptr, scratch, (size_t)need, flags, S(stream));
}

extern "C" tp_status tp_selftest_bounded_wait(int32_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return TP_ERR_INVALID_ARG;
  return cuda_status(launch_bounded_wait_selftest(timeout_us, S(stream)));
}

extern "C" tp_status tp_selftest_e4m3_decode(const void* codes, void* out, int32_t n, void* stream) {
  if (!codes || !out || n <= 0 || n % 4) return TP_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(out)) return TP_ERR_ALIGN;
  return cuda_status(launch_e4m3_decode(codes, out, n, S(stream)));
}
