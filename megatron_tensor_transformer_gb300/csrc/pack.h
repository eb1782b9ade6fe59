// Host-side interface of the partition/pack kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace tpx {

struct PackGeom {
  int kind;                 // tp_wkind
  bool colpar, fp8;
  int t, rows, K;           // per-shard packed matrix [rows, K]
  int out_cols;             // columns of the unsharded [in, out] source
  int ffn, n_q, n_kv, hd;
  int vocab;                // VOCAB / EMBED: real ids (rows = padded ids per shard)
  const uint16_t* W0;       // bf16 bits, [in, out]
  const uint16_t* W1;       // W_up for GATE_UP
  uint64_t shard_stride, scales_offset;
};

cudaError_t launch_pack(const PackGeom& g, uint8_t* packed, cudaStream_t st);

}  // namespace tpx
