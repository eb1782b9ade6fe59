// Host-side interface of the TMA-fed decode kernel for e4m3 weights (M <= 32 tokens).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tpx {

constexpr int kRingMaxM = 32;

struct RingArgs {
  int rowpar;              // 0: column-parallel (mode COLPAR_BF16 / COLPAR_SWIGLU); 1: row-parallel
  int mode;                // column-parallel output mode, or row-parallel FOLD_NONE / FOLD_TICKET
  const uint8_t* w;        // packed e4m3 buffer (shard 0)
  uint64_t shard_stride;   // bytes between shards
  uint64_t scales_offset;  // byte offset of the fp32 row scales inside a shard
  int rows, K, t;          // per-shard matrix [rows, K]; t shards
  const __nv_bfloat16* x;  // [M, ldx]; row-parallel shard s reads columns [s*K, (s+1)*K)
  int ldx, M;
  void* out;               // column-parallel output [M, ldo]
  int ldo;
  const __nv_bfloat16* residual;  // row-parallel, nullable, [M, ldy]
  __nv_bfloat16* y;               // row-parallel output [M, ldy]
  int ldy;
  float* partials;    // row-parallel shard partials [t][pM][rows]
  int pM;
  float* pieces;      // stream-K piece slots: ring_pieces_bytes(M) bytes
  unsigned* counters;  // ring_counter_words(...) words, zero between launches
  unsigned* err;       // device error word (a bounded wait that gives up sets it)
};

// The geometry this kernel takes: 128-row tiles, k a multiple of 128, 1..32 tokens, t <= 8.
bool ring_supported(int rows, int K, int M, int t);
// Bytes of piece slots a launch needs (depends on the GPU's SM count).
size_t ring_pieces_bytes(int M);
// Zero-between-launches counter words a launch needs: one per (shard, row tile), plus one per
// row tile for the row-parallel fold.
size_t ring_counter_words(int rows, int t, bool rowpar);
cudaError_t launch_ring(const RingArgs& a, cudaStream_t st, bool pdl);

}  // namespace tpx
