// Host-side interface of the fused decode block kernel: one persistent tcgen05 launch runs a
// whole tensor-parallel block (column-parallel first linear, then row-parallel second linear
// with its shard fold) for up to 64 tokens.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tpx {

enum FusedKind {
  FUSED_MLP = 0,  // stage 1 = gate/up + SwiGLU -> h; stage 2 = down over h
  FUSED_PROJ = 1  // stage 1 = QKV -> qkv (+ the one-token attention into o_in); stage 2 = o_proj over o_in
};

struct FusedArgs {
  int kind;
  int t, M, d;
  // stage 1 (column-parallel): per-shard packed matrix [rows1, K1 = d]
  int fp8;                       // e4m3 weights: per-row fp32 scales at scales1 / scales2 in each shard
  const uint8_t* w1;
  uint64_t stride1, scales1;
  int rows1;
  // stage 2 (row-parallel): per-shard packed matrix [rows2 = d, K2]
  const uint8_t* w2;
  uint64_t stride2, scales2;
  int K2;
  const __nv_bfloat16* x;        // [M, d]
  __nv_bfloat16* mid;            // stage-1 output: h [M, t*rows1/2] or qkv [M, t*rows1]
  __nv_bfloat16* mid2;           // stage-2 input [M, t*K2]: h (== mid) or o_in
  int n_q, n_kv, hd;             // FUSED_PROJ head geometry (whole model)
  const __nv_bfloat16* residual; // nullable [M, d]
  __nv_bfloat16* y;              // [M, d]
  float* partials;               // [t][M][d] fp32
  unsigned* sync;                // zeroed words: item counter, exit counter, per-shard counts, tile tickets
  unsigned* err;                 // device error word (fail fast, and set when a bounded wait gives up)
  // RMSNorm (gain 1) folded into the block.  Normalising the input is a per-token factor, so it
  // multiplies the column-parallel accumulators: in_scale[m] (nullable, 64 floats).  With
  // in_norm the kernel first computes in_scale[m] = 1/sqrt(mean_k x[m][k]^2 + eps) from x.
  // out_rms (nullable, 64 floats): the fold also yields the same factor of the block's bf16
  // output y, for the next block; norm_ss: scratch of 64 x d/128 fp32.
  float* in_scale;
  int in_norm;
  float* out_rms;
  float* norm_ss;
  float eps;
  // e4m3 weights, split activations: instead of widening the weights, each activation tile is
  // split exactly into two e4m3 tiles (x / s = hi + lo, s a power of two per token: over the
  // whole row for x, over the shard's columns for h or o_in) and the MMA multiplies e4m3 x e4m3
  int split;
};

constexpr int kFusedMaxM = 64;
constexpr int kFusedMaxMWords = 64;  // per-token arrays are sized for kFusedMaxM tokens
// fp32 words of RMSNorm scratch a fused block with a folded norm needs: norm_ss, in_scale, out_rms
inline int fused_norm_words(int d) { return kFusedMaxMWords * (d / 128) + 2 * kFusedMaxMWords; }
// Sync area words: 128 + one ticket per 128-row output tile, then (split activations) the
// per-(shard, token) maxima of the stage-2 input [8][64] (zero between launches) and the
// input's per-token maxima [64] (written before each launch).
__host__ __device__ inline int fused_hmax_off(int d) { return (128 + d / 128 + 31) / 32 * 32; }
// the input's per-token maxima of |x| (float bits), written before each split-activation block by
// launch_token_absmax
__host__ __device__ inline unsigned* fused_xmax_words(unsigned* sync, int d) {
  return sync + fused_hmax_off(d) + 8 * kFusedMaxMWords;
}
inline int fused_sync_words(int d) { return fused_hmax_off(d) + 8 * kFusedMaxMWords + kFusedMaxMWords; }

// Whether the fused kernel supports this block (128-row tiles, M <= 64; 64-wide k-blocks for bf16
// weights, 128-wide for e4m3).
bool fused_supported(int rows1, int d, int K2, int M, int t, bool fp8);
cudaError_t launch_fused(const FusedArgs& a, cudaStream_t st, bool pdl);

}  // namespace tpx
