// Top-K selection over the nodes of one CTA (one node per thread) for the prune of
// "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题" §三 / §四 How (keep the
// Bver best nodes by cumulative path score) and the static-tree prune of
// "浙江大学、阿里巴巴联手破解AI推理瓶颈" §四.
#pragma once

#include "gt_internal.cuh"

namespace gt {

// Among the candidate nodes of the CTA (thread t holds node t; key != 0 marks a
// candidate, larger key = better, see order_key), keeps the K with the largest keys, equal
// keys going to the smaller thread index. Node v is kept iff fewer than K candidates have a
// larger key, or an equal key and a smaller index: the rank rule, found in O(n) by an
// exact radix select of the K-th largest key (up to four passes of 8-bit digits through a
// shared-memory histogram) and a block scan over the nodes that tie with it. The select
// stops after the first pass whose chosen digit bucket is taken whole (its count equals
// the rank still to fill): then exactly K candidates have top bits at or above the
// bucket's, every one of them has fewer than K better keys, and every other candidate
// has at least K, so the rank rule keeps exactly those and no tie is left to break.
// s_hist: 256 ints, s_sel: 3 ints, warp_tot: 32 ints of shared scratch. Every thread of
// the CTA must call it (it synchronises), or, with nthreads > 0, every one of the first
// nthreads threads (named barrier 1; the others hold no node).
__device__ __forceinline__ bool topk_keys_keep(uint32_t key, int K, int *s_hist, int *s_sel,
                                               int *warp_tot, int nthreads = 0) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int stride = nthreads ? nthreads : (int)blockDim.x;
  int total;
  (void)block_excl_count(key != 0u, warp_tot, &total, nthreads);
  if (K <= 0) return false;
  if (total <= K) return key != 0u;
  uint32_t prefix = 0u;  // top bits of the K-th largest key fixed so far
  int kr = K;            // its rank among the keys that share those bits
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += stride) s_hist[i] = 0;
    sync_threads_n(nthreads);
    const bool match =
        key != 0u && (shift == 24 || (key >> (shift + 8)) == (prefix >> (shift + 8)));
    if (match) atomicAdd(&s_hist[(key >> shift) & 255u], 1);
    sync_threads_n(nthreads);
    if (warp == 0) {
      // lane L holds the digits 255 - 8L down to 248 - 8L: lanes run from high to low
      int c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = s_hist[255 - 8 * lane - i];
        sum += c[i];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - sum;
      if (excl < kr && incl >= kr) {  // exactly one lane: the count reaches kr in its bins
        int acc = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc + c[i] >= kr) {
            s_sel[0] = 255 - 8 * lane - i;
            s_sel[1] = kr - acc;
            s_sel[2] = c[i];
            break;
          }
          acc += c[i];
        }
      }
    }
    sync_threads_n(nthreads);
    prefix |= (uint32_t)s_sel[0] << shift;
    kr = s_sel[1];
    if (s_sel[2] == kr)  // the bucket is taken whole (the same decision in every thread)
      return key != 0u && (key >> shift) >= (prefix >> shift);
  }
  // prefix is now the K-th largest key; kr of the keys equal to it are kept
  int neq;
  const int eq_rank = block_excl_count(key != 0u && key == prefix, warp_tot, &neq, nthreads);
  return key > prefix || (key == prefix && eq_rank < kr);
}

}  // namespace gt
