// Host-side interface of the tcgen05 weight-streaming GEMM (weights on the MMA's M side).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tpx {

enum TcMode {
  TC_COLPAR_BF16 = 0,    // out[m][s*rows + r] = bf16(D)
  TC_COLPAR_F32 = 1,     // same, fp32
  TC_COLPAR_SWIGLU = 2,  // gate/up rows interleaved by 8: out[m][s*rows/2 + f] = bf16(silu(g) u)
  TC_ROWPAR_SHARD = 3,   // per-(tile, shard) item: partial P_s (folded afterwards by tp_reduce_partials)
  TC_ROWPAR_CHAIN = 4    // per-tile item: all shards' k chained in shard order in one accumulator, + residual
};

struct TcArgs {
  int mode;
  const uint8_t* w;          // packed weights, shard 0
  uint64_t shard_stride;     // bytes
  int t, rows, K;            // shards; per-shard matrix [rows, K]
  int fp8;                   // e4m3 weights in `w` (widened to bf16 in smem)
  uint64_t scales_offset;    // FP8: byte offset of the scales inside a shard
  const float* scales;       // per-row fp32 scales of shard 0 (e4m3 weights), or nullptr
  uint64_t scales_stride;    // floats from one shard's scales to the next
  const __nv_bfloat16* x;    // activations [M, ldx]
  int ldx, M;
  void* out;                 // colpar output
  int ldo;
  int ncols;                 // colpar: columns to write (0 = all); padded vocabulary ids are not
  // row-parallel
  const __nv_bfloat16* residual;  // nullable, [M, ldy]
  __nv_bfloat16* y;               // [M, ldy]
  int ldy;
  float* partials;                // [t][pM][rows]
  int pM;
  // TC_ROWPAR_CHAIN, nullable: per (token, 32-row group) sums of squares of the stored bf16 y,
  // [M][rows / 32] (the next RMSNorm's input, folded into the next GEMM as per-token factors)
  float* norm_ss;
  // stream-K (decode token tiles): pieces of items cut across CTAs are summed in k order by
  // the CTA that finishes an item last
  int streamk;
  float* pieces;                  // [grid][2][BN][128] fp32
  unsigned* item_tickets;         // one per item, zero between launches
  // FP8 x FP8 (e4m3 weights streamed as they are, activations quantised per token): xq replaces
  // x as e4m3 codes [M, ldx] (ldx in bytes) and tok_scales [M] scales each token's outputs
  int x8;
  const uint8_t* xq;
  const float* tok_scales;
};

constexpr int kTcMaxGrid = 160;          // persistent CTAs (capped so workspace sizes are fixed)
constexpr int kTcMaxStreamkItems = 4096;
constexpr int kTcStreamkMaxBN = 64;
// bytes of stream-K scratch (pieces + item tickets) for token tile BN
inline size_t tc_streamk_bytes() {
  return (size_t)kTcMaxGrid * 2 * kTcStreamkMaxBN * 128 * 4 + (size_t)kTcMaxStreamkItems * 4;
}

// Whether the tcgen05 path supports this geometry (rows % 128, K % 64, bf16 weights).
bool tc_supported(int rows, int K, bool fp8);
// pdl: launch as a programmatic dependent of the previous kernel on the stream (the weight
// tiles stream in while that kernel finishes; activations are read after it completes).
cudaError_t launch_tc(const TcArgs& a, cudaStream_t st, bool pdl);
// Diagnostic kernel whose single wait is never satisfied and gives up after timeout_us.
cudaError_t launch_bounded_wait_selftest(int timeout_us, cudaStream_t st);
// Diagnostic: the FP8 converter's e4m3 -> bf16 routine over n codes (n % 4 == 0).
cudaError_t launch_e4m3_decode(const void* codes, void* out, int n, cudaStream_t st);
// Device error word set by a bounded wait that gave up (0 = none); read and cleared.
unsigned tc_take_device_error();
// Device address of that error word on the current device (resolved once per device), for
// kernels in other translation units; nullptr if it cannot be resolved.
unsigned* tc_error_word();

// cuTensorMapEncodeTiled, resolved through the runtime's driver entry point (nullptr if absent).
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encode_fn();

}  // namespace tpx
