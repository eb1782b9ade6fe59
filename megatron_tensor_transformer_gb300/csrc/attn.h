// Host-side interface of the head-sharded decode attention over a KV cache.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tpx {

// workspace bytes: fp32 per-chunk partial results, then a merge counter per (sequence, kv head)
size_t attn_workspace_bytes(int t, int M, int L, int n_q, int n_kv, int hd);
// head dim 64, 128 or 256; q heads per kv head 1..16 (the rows of one MMA tile)
bool attn_supported(int hd, int G);
// append the new k, v of qkv [M, Q] (shard-major) at position lens[m], then o_in [M, n_q hd] =
// attention over positions 0..lens[m]; caches [t][M][n_kv/t][L][hd] bf16; err: the device error
// word (set if a bounded wait gives up)
cudaError_t launch_attn_decode(int t, int M, int L, int n_q, int n_kv, int hd, const __nv_bfloat16* qkv,
                               __nv_bfloat16* kc, __nv_bfloat16* vc, const int32_t* lens, __nv_bfloat16* o_in,
                               float* ws, unsigned* err, cudaStream_t st);

}  // namespace tpx
