// Interface of the tcgen05 (5th-generation tensor core) tree-attention kernel for bf16.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_common.cuh"

namespace gt {

constexpr int ATTN_TC_KEYS = 128;  // keys per K/V tile

// True when the tcgen05 kernel handles g query heads per KV head and N tree nodes.
bool attn_tc_supported(int g, int N);

// Number of split-KV pieces to aim for: the thread-block clusters of the kernel (one per
// piece, ceil(g*N/128) CTAs each, one CTA per SM) that fit on the device at once.
int attn_tc_pieces(int g, int N);

// Runs every split-KV piece of the schedule (tiles of ATTN_TC_KEYS keys, computed in the
// kernel from `sa`) and writes the partial O / LSE rows of every piece. `pieces` bounds the
// schedule's piece count (one cluster is launched per possible piece).
int attn_tc_launch(const void *Q, const void *K, const void *V, const uint64_t *mask,
                   const SchedArgs &sa, int B, int N, int Hq, int Hkv, int Lcap, float scale,
                   const AttnWs &ws, int pieces, void *O, int32_t *err, cudaStream_t s);

}  // namespace gt
