/*
 * tpx.h -- C ABI of libtpx.so: Megatron-style tensor-parallel linear layers of a
 * Llama-style block, all t logical shards on one GB300 (sm_103a).
 *
 * The method ("The Tensor-Parallel Shard Group", scalablesystem.dev; "Tensor
 * Parallelism (Megatron-Style)", arunshar.com ch. 12; "Step 1: tensor parallelism
 * slices every layer", vidyal.ai model-parallelism):
 *   - the first linear of a block is split along its OUTPUT dim (column-parallel):
 *     shard s owns a slice of output features, needs no communication in, and
 *     applies the nonlinearity to its own slice;
 *   - the second linear is split along its INPUT dim (row-parallel): shard s
 *     produces a partial Z_s of the full output and Z = sum_s Z_s ("all-reduce").
 * Here the sum over shards is a deterministic fixed-order fp32 fold on the device:
 *     y = bf16_rne( (((Z_0 + Z_1) + Z_2) + ... + Z_{t-1}) + float(residual) ).
 *
 * Conventions for every entry point below:
 *   - Pointers are DEVICE pointers unless marked (host).  All buffers are owned by
 *     the caller; the library never allocates and never synchronises on the forward
 *     path.  Work is enqueued on `stream` (a cudaStream_t passed as void*, NULL =
 *     legacy default stream).
 *   - Matrices are row-major.  Activations are bf16 [M, features].  Unsharded
 *     weights are bf16 in the [in, out] orientation of Y = X A.
 *   - Every argument check runs on the host BEFORE any launch and returns a status;
 *     a failed check enqueues nothing.  Launch errors return TP_ERR_CUDA.
 *   - Device pointers must be 16-byte aligned (TP_ERR_ALIGN otherwise).
 *   - Not thread-safe per stream: calls that share a workspace must be ordered.
 */
#ifndef TPX_H
#define TPX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TP_OK = 0,
  TP_ERR_INVALID_ARG = 1,     /* NULL pointer, M < 0, unknown kind/flags */
  TP_ERR_SHAPE = 2,           /* t not in {1,2,4,8}, t does not divide ffn / n_kv / n_q, ... */
  TP_ERR_ALIGN = 3,           /* pointer not 16-byte aligned, or a dim not a multiple the kernels need */
  TP_ERR_LAYOUT_MISMATCH = 4, /* packed descriptor does not match the call (wrong shard layout) */
  TP_ERR_WORKSPACE = 5,       /* workspace NULL or smaller than tp_workspace_bytes() */
  TP_ERR_CUDA = 6,            /* a CUDA runtime call or launch failed */
  TP_ERR_TIMEOUT = 7,         /* tp_sync deadline passed with work still pending */
  TP_ERR_DEVICE_TIMEOUT = 8,  /* a bounded device-side wait gave up (device error word set) */
  TP_ERR_UNSUPPORTED = 9      /* a valid request this build does not implement */
} tp_status;

typedef enum { TP_BF16 = 0, TP_FP8_E4M3 = 1 } tp_wtype;

/* Which weight of the block a packed buffer holds. */
typedef enum {
  TP_W_GATE_UP = 0, /* column-parallel W_gate and W_up, [d, ffn] each */
  TP_W_DOWN = 1,    /* row-parallel W_down, [ffn, d] */
  TP_W_QKV = 2,     /* column-parallel W_qkv, [d, (n_q + 2 n_kv) * head_dim] */
  TP_W_O = 3,       /* row-parallel W_o, [n_q * head_dim, d] */
  TP_W_VOCAB = 4,   /* lm_head W, [d, vocab], column-parallel over the vocabulary (bf16 only) */
  TP_W_EMBED = 5    /* embedding table E, [vocab, d], split by vocabulary rows (bf16 only) */
} tp_wkind;

/* Model dims and the shard count.  ffn is used by GATE_UP/DOWN, the head dims by
 * QKV/O, vocab by VOCAB/EMBED.  t must be 1, 2, 4 or 8 and divide ffn, n_q and n_kv (a GQA
 * head cannot be split between shards; t > n_kv head replication is not supported).  The
 * vocabulary is padded with zero rows so that each shard holds a multiple of 128 ids:
 * vocab_padded = round_up(vocab, 128 t), V_s = vocab_padded / t ids per shard. */
typedef struct {
  int32_t d, ffn, n_q_heads, n_kv_heads, head_dim, t;
  int32_t wtype; /* tp_wtype */
  int32_t vocab;
} tp_shape;

#define TP_DESC_MAGIC 0x54505831u /* "TPX1" */
#define TP_LAYOUT_VERSION 1u

/* Host struct describing a packed weight buffer.  Shard s starts at byte
 * s * shard_stride_bytes and holds a K-major matrix [rows_per_shard, k_per_shard]
 * (one row per output feature, the nn.Linear [out, in] orientation) of bf16 or
 * e4m3 codes; for FP8, float32 scales follow at scales_offset within the shard
 * (one per row of the shard).  Packed-row order:
 *   GATE_UP: shard s holds gate/up columns [s*F_s, (s+1)*F_s), F_s = ffn/t,
 *            interleaved in blocks of 8 features: rows 16b..16b+7 = gate columns
 *            s*F_s+8b+0..7, rows 16b+8..16b+15 = up columns s*F_s+8b+0..7.
 *   QKV:     shard s holds its q heads [s*n_q/t, (s+1)*n_q/t), then its kv heads
 *            [s*n_kv/t, (s+1)*n_kv/t) of k, then the same of v (head_dim rows each);
 *            q head h uses kv head h / (n_q/n_kv), so a GQA group never straddles shards.
 *   DOWN/O:  shard s holds rows [s*K_s, (s+1)*K_s) of the [in, out] weight,
 *            transposed: element [n][k] = W[s*K_s + k][n]; FP8 scales replicated.
 *   VOCAB:   shard s holds vocabulary ids [s*V_s, (s+1)*V_s): row r = column s*V_s + r of
 *            the [d, vocab] lm_head weight, zero for padding ids (>= vocab).
 *   EMBED:   shard s holds rows [s*V_s, (s+1)*V_s) of the [vocab, d] table as they are,
 *            zero for padding ids.
 * FP8: s_n = absmax over the whole unsharded input dim of column n / 448 (fp32),
 * 1 for an all-zero column; code = e4m3 RNE satfinite(W / s_n) (fp32 divide). */
typedef struct {
  uint32_t magic, layout_version;
  int32_t kind, wtype;
  tp_shape shape;
  int64_t rows_per_shard, k_per_shard;
  uint64_t shard_payload_bytes, scales_offset, shard_stride_bytes, total_bytes;
} tp_packed_desc;

/* Flags */
#define TP_F_UNFUSED_REDUCE 0x1u  /* row-parallel: write shard partials to the workspace, then
                                     run tp_reduce_partials (same bits as the fused path) */
#define TP_F_FP32_COLPAR_OUT 0x2u /* tp_colpar_forward: write fp32 instead of bf16 */
#define TP_F_SERIAL 0x40u         /* launch every kernel only after the previous work on the stream has
                                     finished.  By default a forward's tcgen05 kernels start streaming
                                     weights while the previous kernel drains (programmatic dependent
                                     launch): packed weights must then not be written by work still in
                                     flight on the stream (tp_partition_weights returns with them
                                     complete).  Activations are always read after earlier work ends. */
#define TP_F_KERNEL_SKINNY 0x10u  /* force the mma.sync weight-streaming kernel (register-direct loads) */
#define TP_F_KERNEL_TC 0x20u      /* force the tcgen05/TMA kernels (rows % 128, K % 64); default:
                                     tcgen05 where supported, except e4m3 weights at decode token counts
                                     (M <= 64).  There a whole block (tp_mlp_forward, tp_proj_forward,
                                     tp_layer_forward; 128-row tiles, k % 128) runs as one tcgen05 launch:
                                     on hi/lo activation codes (TP_F_FP8_HILO) up to 32 tokens, widening
                                     the weights to bf16 from 33 to 64 (measured faster there); with this
                                     flag that launch widens the weights at every decode token count.  The halves on their own
                                     (tp_colpar_forward, tp_rowpar_forward, TP_F_SPLIT_BLOCK) go to the
                                     TMA-fed mma.sync kernel (M <= 32, 128-row tiles, k % 128, a workspace
                                     given; widening in registers, work split evenly over two CTAs per SM,
                                     fused and unfused folds give the same bits), else to the
                                     register-direct mma.sync kernel */
#define TP_F_FP8_ACT 0x200u       /* e4m3 weights: also quantise each GEMM's activations per token (s_m =
                                     absmax/448 over the token's whole row, e4m3 RNE satfinite, as
                                     tp_quantize_fp8_per_token) and multiply e4m3 x e4m3 on the tensor
                                     cores, both scales applied to the fp32 result.  A different numeric
                                     reading from the default (the pages give no activation scale), for
                                     prefill: the tensor rate is twice bf16's.  tcgen05 kernels, rows %
                                     128 and k % 128; the workspace grows by M x the widest activation row
                                     (tp_workspace_bytes with this flag). */
#define TP_F_FP8_HILO 0x400u      /* e4m3 weights, decode blocks (tp_mlp_forward, tp_proj_forward,
                                     tp_layer_forward; M <= 64, 128-row tiles, k % 128): one persistent
                                     tcgen05 launch per block that splits each bf16 activation exactly
                                     into two e4m3 codes (x / s = hi + lo, s a power of two per token:
                                     the token's row of x, or its shard's columns of h / o_in) and
                                     multiplies e4m3 x e4m3, the weights straight from shared memory.
                                     This is what those blocks run by default up to 32 tokens; the flag
                                     asks for it up to 64 and overrides TP_F_KERNEL_TC.  The split is exact for every activation of at
                                     least 2^-10 of its token's largest (2^-2 of the scaled range): those
                                     are multiplied as the bf16 values they are.  A smaller activation
                                     loses the bits below 2^-17 of the token's largest, so the result
                                     approximates the bf16-activation product (fp32 sums, in another
                                     order) rather than equalling it.  No effect on bf16 weights or where
                                     the one-launch block does not apply */
#define TP_F_FOLD_NORM 0x800u     /* tp_layer_forward at prefill token counts (M > 64, every GEMM on the
                                     tcgen05 path): fold both RMSNorms into the GEMMs as per-token factors
                                     on the column-parallel accumulators (x's factors from one pass over x,
                                     h1's from sums of squares the o_proj epilogue leaves), so the
                                     normalised activations are never written.  Opt-in: measured on the
                                     70B layer at M = 4096 it is slower (4.79 ms against 4.66 ms), the
                                     epilogue work costing more than the norm passes it saves.  Decode
                                     layers always fold the norms into their two block launches */
#define TP_F_SPLIT_BLOCK 0x80u    /* tp_mlp_forward / tp_proj_forward: run the two halves as separate
                                     launches.  By default a decode block (M <= 64, 128-row tiles; k %
                                     64 for bf16 weights, k % 128 for e4m3, see TP_F_FP8_HILO) runs as
                                     ONE persistent launch: the column-parallel items, then the
                                     row-parallel items, each of which waits only for its own shard's
                                     first half; the last shard of each 128-row output tile folds the t
                                     partials in shard order (for bf16 weights, the same bits as the
                                     split path) */

/* Size in bytes of the packed buffer for (shape, kind); 0 if the shape is invalid. */
size_t tp_packed_bytes(const tp_shape* shape /* host */, int32_t kind);

/* Fill *desc (host) for (shape, kind) without touching the device. */
tp_status tp_describe(const tp_shape* shape /* host */, int32_t kind, tp_packed_desc* desc /* host */);

/* Split and pack an unsharded weight for degree t (column split on the output dim for
 * GATE_UP/QKV, row split on the input dim for DOWN/O; "ColumnParallelLinear" /
 * "RowParallelLinear", scalablesystem.dev "The Tensor-Parallel Shard Group").  A set-up call,
 * not on the forward path: it is the one entry point that synchronises its stream.  W0: [in,out] bf16 (W_gate for GATE_UP);
 * W1: W_up for GATE_UP, else NULL.  packed: packed_bytes >= tp_packed_bytes().
 * Writes the layout described above; for FP8 also quantises (shape.wtype).  Fills
 * *desc_out (host).  Synchronises `stream` before returning, so the packed buffer is
 * complete (forwards may start reading it early, see TP_F_SERIAL). */
tp_status tp_partition_weights(const tp_shape* shape /* host */, int32_t kind, const void* W0,
                               const void* W1, void* packed, size_t packed_bytes,
                               tp_packed_desc* desc_out /* host */, void* stream);

/* Workspace bytes the forward calls need for M tokens (shard partials and tickets).
 * The workspace must be zero-filled once before first use; calls leave it reusable.  After a
 * call has ended in TP_ERR_DEVICE_TIMEOUT (reported by tp_sync), zero-fill it again. */
size_t tp_workspace_bytes(const tp_shape* shape /* host */, int32_t M, uint32_t flags);

/* SwiGLU MLP block: h = silu(x Wg) * (x Wu) column-parallel per shard, then
 * y = fold_s(h_s Wd_s) + residual row-parallel (scalablesystem.dev "The Tensor-Parallel Shard
 * Group": the MLP's gate and up projections column-parallel, its down projection row-parallel).
 * x, residual (nullable): [M, d] bf16; y: [M, d] bf16; h_out: [M, ffn] bf16, required: it is
 * where the column-parallel half leaves h for the row-parallel half (the library allocates
 * nothing, so the caller owns that buffer), and it holds h afterwards, shard s's columns at
 * [s*F_s, (s+1)*F_s).  M == 0 returns TP_OK with no work.  y may alias residual. */
tp_status tp_mlp_forward(const tp_packed_desc* gu /* host */, const void* gu_w,
                         const tp_packed_desc* dn /* host */, const void* dn_w, const void* x,
                         const void* residual, int32_t M, void* y, void* h_out, void* ws,
                         size_t ws_bytes, uint32_t flags, void* stream);

/* Attention sub-block: qkv = x Wqkv column-parallel (each shard owns whole heads);
 * o_in = local attention per shard; y = fold_s(o_in_s Wo_s) + residual row-parallel
 * ("TPAttentionBlock", scalablesystem.dev).  The attention core is a one-token
 * context: every q head returns the v of its kv group.  qkv_out: [M, (n_q+2n_kv)hd]
 * bf16, shard-major (shard s = [q_s | k_s | v_s]); o_in: [M, n_q*hd] bf16, required: the
 * attention output that the row-parallel o_proj reads (caller-owned, as h_out above). */
tp_status tp_proj_forward(const tp_packed_desc* qkv /* host */, const void* qkv_w,
                          const tp_packed_desc* o /* host */, const void* o_w, const void* x,
                          const void* residual, int32_t M, void* y, void* qkv_out, void* o_in,
                          void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* One pre-norm Llama layer's linear parts (the pipeline-stage stack is ten of these):
 *   a = rmsnorm(x);  h1 = x + O(attn(QKV(a)));  b = rmsnorm(h1);  y = h1 + MLP(b)
 * with RMSNorm eps, gain 1.  The four packed weights must describe one block (same d, t,
 * dtype; heads for QKV/O, ffn for GATE_UP/DOWN).  x, y: [M, d] bf16 (y may alias x).
 * scratch: tp_layer_scratch_bytes(shape, M) bytes of device memory for the activations
 * between the steps; ws as for the blocks.  With B = round_up(M*d*2, 256) the scratch holds,
 * in bf16, a [M, d] at 0, h1 [M, d] at B, the attention output [M, n_q*hd] at 2B, b [M, d] at
 * 3B, qkv [M, (n_q+2n_kv)hd] (shard-major) at 4B and h [M, ffn] at 4B + round_up(M*Q*2, 256);
 * after the call h1, the attention output, qkv and h hold this layer's values.  At decode token
 * counts the norms are folded into the two block launches (per-token factors on the
 * column-parallel accumulators) and a, b are not written; at prefill the same with
 * TP_F_FOLD_NORM. */
size_t tp_layer_scratch_bytes(const tp_shape* shape /* host */, int32_t M);
tp_status tp_layer_forward(const tp_packed_desc* qkv /* host */, const void* qkv_w,
                           const tp_packed_desc* o /* host */, const void* o_w,
                           const tp_packed_desc* gu /* host */, const void* gu_w,
                           const tp_packed_desc* dn /* host */, const void* dn_w, const void* x,
                           int32_t M, void* y, float eps, void* scratch, size_t scratch_bytes, void* ws,
                           size_t ws_bytes, uint32_t flags, void* stream);

/* The "all-reduce" on one GPU: y[m][n] = bf16_rne(((P_0 + P_1) + ... + P_{t-1})[m][n]
 * + float(residual[m][n])), a left fold in shard order (Z = sum_k Z_k, arunshar.com;
 * summation order fixed so results are reproducible).  partials: [t][M][d] fp32;
 * residual nullable [M, d] bf16; y [M, d] bf16. */
tp_status tp_reduce_partials(const float* partials, int32_t t, int32_t M, int32_t d,
                             const void* residual, void* y, void* stream);

/* Column-parallel building block ("ColumnParallelLinear.forward", scalablesystem.dev "The
 * Tensor-Parallel Shard Group"; A = [A_1 | ... | A_t], each shard's output a slice of the
 * features, arunshar.com ch. 12 "Tensor Parallelism (Megatron-Style)"):
 * out[m][s*rows + r] for every shard s and packed row r.
 * GATE_UP: out = h [M, ffn] bf16 (SwiGLU applied);  QKV: out = qkv [M, Q] bf16.
 * With TP_F_FP32_COLPAR_OUT (QKV only) out is fp32.  ws is optional (NULL, or a workspace of
 * tp_workspace_bytes(shape, M) bytes, which lets the tcgen05 kernel balance work across SMs). */
tp_status tp_colpar_forward(const tp_packed_desc* desc /* host */, const void* w, const void* x,
                            int32_t M, void* out, void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* Row-parallel building block without the fold (the shard partials Z_s of arunshar.com ch. 12
 * "Tensor Parallelism (Megatron-Style)", before their sum): partials[s][m][n] = (a_s W_s)[m][n],
 * a_s = columns [s*K_s, (s+1)*K_s) of a [M, t*K_s] bf16; partials [t][M][N] fp32. */
tp_status tp_rowpar_partials(const tp_packed_desc* desc /* host */, const void* w, const void* a,
                             int32_t M, float* partials, void* stream);

/* Row-parallel linear with its "all-reduce" ("RowParallelLinear.forward", scalablesystem.dev):
 * y[m][n] = bf16(fold_s (a_s W_s)[m][n] + residual[m][n]) for DOWN or O weights, a: [M, t*K_s]
 * bf16, residual nullable [M, N], y [M, N].  Same kernels and bits as the second half of
 * tp_mlp_forward / tp_proj_forward; ws as for those (tp_workspace_bytes). */
tp_status tp_rowpar_forward(const tp_packed_desc* desc /* host */, const void* w, const void* a,
                            const void* residual, int32_t M, void* y, void* ws, size_t ws_bytes,
                            uint32_t flags, void* stream);

/* Allocation-free variant of tp_rowpar_forward.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory, such as a plugin
 * inside a host framework whose caching allocator owns the whole device, or code on a
 * latency-critical path that cannot afford cudaMalloc's implicit synchronisation.
 * Same arguments, result and bits as tp_rowpar_forward, minus the workspace: the shard
 * partials and tickets live in one static device array of tp_noalloc_scratch_capacity()
 * bytes (32 MiB), which every GPU that loads the library holds until the process exits.
 * Requests that need more (t * min(M,64) * N * 4 bytes of partials, N/2 bytes of tickets
 * and 10.5 MB of work-balancing scratch) return TP_ERR_WORKSPACE.  The call never allocates or frees memory.  The first call on
 * each device resolves the array's device address (cudaGetSymbolAddress, with that
 * device current), so make that first call before any stream capture.  Every call on a
 * device shares the one array and leaves its contents behind (the tickets are cleared
 * at the start of each call): calls that may overlap on the GPU (other streams, other
 * threads) race and must be serialised by the caller.  TP_F_FP8_ACT is refused
 * (TP_ERR_UNSUPPORTED): its quantised activations have no room in the array.  The resolved
 * address belongs to the device's current context: after a cudaDeviceReset this entry point,
 * like the rest of the library, must not be called again in the same process. */
tp_status tp_rowpar_forward_noalloc(const tp_packed_desc* desc /* host */, const void* w, const void* a,
                                    const void* residual, int32_t M, void* y, uint32_t flags,
                                    void* stream);

/* Bytes of the static scratch array tp_rowpar_forward_noalloc uses. */
size_t tp_noalloc_scratch_capacity(void);

/* Decode attention over a KV cache, head-sharded (each shard attends with its own q heads over
 * the cache of its own kv heads, whole GQA groups: each shard attends with its own heads,
 * scalablesystem.dev "The Tensor-Parallel Shard Group", and the KV cache is split with them, vidyal.ai). 
 * One new token per sequence m: its k and v (from qkv) are first written into the cache at
 * position lens[m]; then, for q head h and its kv head g = h / (n_q / n_kv),
 *   o_in[m][h*hd + i] = bf16( sum_j softmax_j(q . k_j / sqrt(hd)) v_j[i] ),  j = 0 .. lens[m],
 * with fp32 scores, softmax and accumulation; the probabilities enter the p.v product rounded
 * to bf16, the tensor cores' operand type (no positional rotation: the pages give none).
 * qkv: [M, (n_q + 2 n_kv) hd] bf16 in the column-parallel shard-major order (tp_colpar_forward's
 * QKV output); k_cache, v_cache: [t][M][n_kv/t][L][hd] bf16 (device, caller-owned; shard s holds
 * its kv heads' cache); lens: [M] int32 (device, not modified); o_in: [M, n_q hd] bf16 (the
 * row-parallel o_proj input).  A sequence with lens[m] outside [0, L) is left out: nothing is
 * written to its cache and its o_in row is zero.  head_dim must be 64, 128 or 256, n_q / n_kv at
 * most 16 and M * n_kv * L below 2^31 (else TP_ERR_UNSUPPORTED); qkv, the caches, o_in and ws
 * 16-byte aligned (else TP_ERR_ALIGN).  Cache slots after lens[m] are never read into the result.
 * ws: tp_attn_workspace_bytes(shape, M, L) bytes, partial results per 128-position chunk and a
 * merge counter per (sequence, kv head), which the call resets itself (no zero-fill needed);
 * calls that share a ws must not overlap on the GPU.  Two kernel launches; the result is
 * bitwise the same run to run.  A staged copy that never lands sets the device error word
 * (TP_ERR_DEVICE_TIMEOUT from tp_sync). */
size_t tp_attn_workspace_bytes(const tp_shape* shape /* host */, int32_t M, int32_t L);
tp_status tp_attn_decode(const tp_shape* shape /* host */, const void* qkv, void* k_cache, void* v_cache, int32_t L,
                         const int32_t* lens, int32_t M, void* o_in, void* ws, size_t ws_bytes, void* stream);

/* The attention block of a decode step over a KV cache ("TPAttentionBlock" with a real
 * attention core, scalablesystem.dev "The Tensor-Parallel Shard Group"), in one call:
 *   qkv_out = x . Wqkv                       column-parallel, shard-major (tp_colpar_forward)
 *   cache[lens[m]] = the new k, v;  o_in = attention over positions 0..lens[m] (tp_attn_decode)
 *   y = residual + o_in . Wo                 row-parallel, shards folded in order (tp_rowpar_forward)
 * qkv, o: QKV and O descriptors of one block; x, residual (nullable), y: [M, d] bf16 (y must not
 * alias x or residual); k_cache, v_cache, L, lens as for tp_attn_decode; qkv_out [M, (n_q+2n_kv)hd]
 * and o_in [M, n_q hd]: caller's bf16 buffers that keep the step's q, k, v and attention output.
 * ws: tp_attn_block_workspace_bytes(shape, M, L, flags) bytes, zero-filled once before first use
 * (its head is the projections' workspace, its tail the attention's).  Errors as for the three
 * calls; four kernel launches for bf16 weights at decode token counts. */
size_t tp_attn_block_workspace_bytes(const tp_shape* shape /* host */, int32_t M, int32_t L, uint32_t flags);
tp_status tp_attn_block_forward(const tp_packed_desc* qkv /* host */, const void* qkv_w,
                                const tp_packed_desc* o /* host */, const void* o_w, const void* x,
                                const void* residual, int32_t M, void* k_cache, void* v_cache, int32_t L,
                                const int32_t* lens, void* y, void* qkv_out, void* o_in, void* ws,
                                size_t ws_bytes, uint32_t flags, void* stream);

/* Vocabulary-parallel lm_head (the column-parallel GEMM at the model's output edge; each shard's
 * logits are a slice of the output, so the pages' all-gather is a concatenation, scalablesystem.dev
 * "The Tensor-Parallel Shard Group"): logits[m][v] = sum_k x[m][k] W[k][v] for v < vocab, fp32
 * accumulate and output.  desc: a TP_W_VOCAB buffer; x: [M, d] bf16; logits: [M, vocab] fp32
 * (padding ids are not written).  ws optional as for tp_colpar_forward.  M == 0 is a no-op. */
tp_status tp_lm_head_forward(const tp_packed_desc* desc /* host */, const void* w, const void* x, int32_t M,
                             float* logits, void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* Vocabulary-parallel embedding lookup (the table split by vocabulary rows; each shard contributes
 * its row if the id is in its range, else zeros, and the contributions are summed, which leaves
 * exactly one row): x[m] = E[ids[m]], a zero row for an id outside [0, vocab).  desc: a
 * TP_W_EMBED buffer; ids: [M] int32 (device); x: [M, d] bf16.  M == 0 is a no-op. */
tp_status tp_embed_lookup(const tp_packed_desc* desc /* host */, const void* w, const int32_t* ids, int32_t M,
                          void* x, void* stream);

/* Per-token e4m3 quantisation of activations (the TP_F_FP8_ACT path's first step, exported for
 * exact tests): x [M, K] bf16 (device, row stride K), s[m] = absmax_k |x[m][k]| / 448 in IEEE
 * binary32 (1 for an all-zero row), q[m][k] = e4m3 RNE satfinite of x[m][k] / s[m] (binary32
 * divide).  q: [M, K] bytes; s: [M] fp32 (device).  K % 8 == 0; pointers 16-byte aligned. */
tp_status tp_quantize_fp8_per_token(const void* x, int32_t M, int32_t K, void* q, float* s, void* stream);

/* RMSNorm over the hidden dim, gain 1 (or gain [d] bf16): out = bf16(x / sqrt(mean(x^2) + eps) * g).
 * The norm that the layer applies, replicated, to its full hidden vector between the
 * reductions (arunshar.com ch. 12, "12.3.1 Sequence Parallelism for LayerNorm and Dropout"). */
tp_status tp_rmsnorm(const void* x, const void* gain, float eps, int32_t M, int32_t d, void* out,
                     void* stream);

/* Block until `stream` drains or timeout_ms passes (TP_ERR_TIMEOUT; the work keeps
 * running).  Also reports a device error word set by a bounded device-side wait
 * (TP_ERR_DEVICE_TIMEOUT) and clears it. */
tp_status tp_sync(void* stream, int32_t timeout_ms);

/* Diagnostic for the failure path: launches a one-thread kernel whose wait on a barrier that
 * nothing arrives at gives up after timeout_us (1 .. 1e6) microseconds and records the device
 * error word, exactly as the library's kernels do when a wait runs out.  The next tp_sync
 * returns TP_ERR_DEVICE_TIMEOUT and clears it; the context stays usable.  No fault, no trap. */
tp_status tp_selftest_bounded_wait(int32_t timeout_us, void* stream);

/* Diagnostic: decode n e4m3 codes (bytes, n % 4 == 0) to bf16 with the exact routine the FP8
 * weight path widens weight tiles with, so a test can compare every code with its value. */
tp_status tp_selftest_e4m3_decode(const void* codes, void* out, int32_t n, void* stream);

/* Static string for a status code. */
const char* tp_status_str(tp_status s);

/* Number of kernel launches this library has enqueued since load (for launch counting). */
uint64_t tp_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* TPX_H */
