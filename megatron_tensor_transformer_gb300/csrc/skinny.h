// Host-side interface of the decode (skinny-M) kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tpx {

enum ColparMode { COLPAR_BF16 = 0, COLPAR_F32 = 1, COLPAR_SWIGLU = 2 };
enum FoldMode { FOLD_NONE = 0, FOLD_IN_CTA = 1, FOLD_TICKET = 2 };

constexpr int kSkinnyMaxM = 64;  // tokens per launch; larger M is split into blocks of 64

struct ColparArgs {
  const uint8_t* w;        // packed buffer (shard 0)
  uint64_t shard_stride;   // bytes between shards
  uint64_t scales_offset;  // FP8: byte offset of the fp32 row scales inside a shard
  int rows, K, t;          // per-shard matrix [rows, K]; t shards
  const __nv_bfloat16* x;  // [M, ldx]
  int ldx, M;
  void* out;               // [M, ldo]
  int ldo, mode;
};

struct RowparArgs {
  const uint8_t* w;
  uint64_t shard_stride, scales_offset;
  int N, K, t;             // per-shard matrix [N, K]; t shards
  const __nv_bfloat16* x;  // [M, ldx]; shard s reads columns [s*K, (s+1)*K)
  int ldx, M;
  const __nv_bfloat16* residual;  // nullable, [M, ldy]
  __nv_bfloat16* y;               // [M, ldy]
  int ldy;
  float* partials;  // [t][pM][N]
  int pM;
  unsigned* tickets;  // one per row tile, zero between launches
  int fold;
};

// Launch choices that both the fused and the unfused row-parallel paths share, so
// that they produce identical bits.
struct RowparPlan {
  int R, S, tiles;
};
RowparPlan rowpar_plan(int N, int t);
int colpar_R(int rows, bool swiglu);

cudaError_t launch_colpar(const ColparArgs& a, bool fp8, cudaStream_t st);
cudaError_t launch_rowpar(const RowparArgs& a, bool fp8, const RowparPlan& p, cudaStream_t st);

}  // namespace tpx
