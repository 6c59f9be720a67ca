// Device pieces of the vocabulary top-k shared by the top-k kernel (verify.cu) and the
// sampler, which forms the same top-k in its own pass over the logits (sample.cu): order
// keys packed with indices, warp selections, the exact per-thread-list path, the CTA's
// candidate selection and the cluster merge.
//
// Sources: "浙江大学、阿里巴巴联手破解AI推理瓶颈" §二 third gear (the table rows hold the
// target's k most likely next tokens); "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快
// 与好的单选题" §五 (greedy verification: the argmax is entry 0).
#pragma once

#include <cooperative_groups.h>
#include <math.h>
#include <stdint.h>

#include "gt_internal.cuh"

namespace gt {

namespace cg = cooperative_groups;

constexpr int TOPK_THREADS = 256;
constexpr int TOPK_CLUSTER = 8;
constexpr int TOPK_PER = 5;      // float4 per thread per chunk (a second chunk in flight)
constexpr int TOPK_CAP = 512;    // candidate buffer per CTA

__device__ __forceinline__ uint64_t pack_key(uint32_t key, int idx) {
  return ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ int unpack_idx(uint64_t p) {
  return (int)(0xFFFFFFFFu - (uint32_t)(p & 0xFFFFFFFFull));
}

// Inverse of order_key for keys of real numbers; keys 0 (empty) and 1 (NaN) give -inf,
// which makes every element a candidate.
__device__ __forceinline__ float key_floor(uint32_t k) {
  if (k <= 1u) return -INFINITY;
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Insert (nk, ni) into a list sorted by key descending. Callers scan indices in
// increasing order, so on equal keys the new element (larger index) goes below.
template <int KK>
__device__ __forceinline__ void list_insert(uint32_t (&key)[KK], int (&idx)[KK], uint32_t nk,
                                            int ni) {
#pragma unroll
  for (int j = KK - 1; j >= 0; --j) {
    if (nk > key[j]) {
      if (j > 0 && nk > key[j - 1]) {
        key[j] = key[j - 1];
        idx[j] = idx[j - 1];
      } else {
        key[j] = nk;
        idx[j] = ni;
      }
    }
  }
}

template <int KK>
__device__ __forceinline__ void consider(uint32_t (&key)[KK], int (&idx)[KK], float f, int i) {
  const uint32_t kx = order_key(f);
  if (kx > key[KK - 1]) list_insert<KK>(key, idx, kx, i);
}

// A bitonic sort of one key per lane across the warp, descending: lane r returns the
// (r+1)-th largest.
__device__ __forceinline__ uint32_t warp_sorted_desc(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool up = (lane & size) != 0;          // this block sorts ascending
      const bool lower = (lane & stride) == 0;
      v = (lower == up) ? min(v, o) : max(v, o);
    }
  }
  return v;
}

// Warp-wide max of packed (order key, inverted index) words: two single-instruction
// reductions, the key first, then the lowest index among the lanes holding that key.
__device__ __forceinline__ uint64_t warp_max_packed(uint64_t v) {
  const uint32_t hi = (uint32_t)(v >> 32);
  const uint32_t khi = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t klo = __reduce_max_sync(0xffffffffu, hi == khi ? (uint32_t)v : 0u);
  return ((uint64_t)khi << 32) | klo;
}

// KK rounds over NC unsorted candidates per lane (0 = empty); lane r returns the r-th
// best. Packed words are unique, so each round removes exactly one candidate.
template <int KK, int NC>
__device__ __forceinline__ uint64_t warp_select(uint64_t (&c)[NC]) {
  const int lane = threadIdx.x & 31;
  uint64_t out = 0;
#pragma unroll
  for (int r = 0; r < KK; ++r) {
    uint64_t my = c[0];
#pragma unroll
    for (int j = 1; j < NC; ++j) my = c[j] > my ? c[j] : my;
    const uint64_t best = warp_max_packed(my);
    if (best != 0) {
#pragma unroll
      for (int j = 0; j < NC; ++j)
        if (c[j] == best) c[j] = 0;
    }
    if (lane == r) out = best;
  }
  return out;
}

// KK rounds of a warp argmax over each lane's sorted list head; lane r gets the r-th best.
template <int KK>
__device__ __forceinline__ uint64_t warp_merge_lists(uint32_t (&key)[KK], int (&idx)[KK]) {
  const int lane = threadIdx.x & 31;
  uint64_t out = 0;
#pragma unroll
  for (int r = 0; r < KK; ++r) {
    const uint64_t my = key[0] ? pack_key(key[0], idx[0]) : 0ull;
    const uint64_t best = warp_max_packed(my);
    if (best != 0 && my == best) {
#pragma unroll
      for (int j = 0; j < KK - 1; ++j) {
        key[j] = key[j + 1];
        idx[j] = idx[j + 1];
      }
      key[KK - 1] = 0u;
      idx[KK - 1] = -1;
    }
    if (lane == r) out = best;
  }
  return out;
}

// Exact per-thread sorted lists over [b, e) of one row, merged to the CTA's top-KK in
// s_top by warp 0 (rows without 16-byte alignment, and the overflow fallback).
template <int KK>
__device__ __forceinline__ void topk_exact(const float *x, int b, int e, uint64_t *s_stage,
                                           uint64_t *s_top) {
  constexpr int NW = TOPK_THREADS / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t key[KK];
  int idx[KK];
#pragma unroll
  for (int j = 0; j < KK; ++j) key[j] = 0u, idx[j] = -1;
  for (int i = b + tid; i < e; i += TOPK_THREADS) consider<KK>(key, idx, __ldcs(x + i), i);
  const uint64_t wb = warp_merge_lists<KK>(key, idx);
  if (lane < KK) s_stage[warp * KK + lane] = wb;
  __syncthreads();
  if (warp == 0) {
    constexpr int NC = (NW * KK + 31) / 32;
    uint64_t c[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int q = lane + 32 * j;
      c[j] = q < NW * KK ? s_stage[q] : 0ull;
    }
    const uint64_t bb = warp_select<KK, NC>(c);
    if (lane < KK) s_top[lane] = bb;
  }
  __syncthreads();
}

// The CTA's top-KK of cnt <= TOPK_CAP candidates into s_top (s_top[r] = the r-th best, 0 past
// the last candidate). Up to TOPK_RANKED candidates (the usual few dozen): packed words are
// unique, so a candidate's rank is the number of candidates above it, and every thread ranks
// candidates t, t + blockDim.x, ... against all of them (broadcast shared-memory reads, no
// dependent rounds); the top KK place themselves. The ranking work grows with the square of
// the count, so larger counts go to warp 0's KK selection rounds over 8 or 16 candidates per
// lane. Every thread of the CTA calls it (it synchronises).
constexpr int TOPK_RANKED = 128;
template <int KK>
__device__ __forceinline__ void select_candidates(int cnt, const uint64_t *s_cand,
                                                  uint64_t *s_top) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (cnt <= TOPK_RANKED) {
    for (int t = tid; t < cnt; t += blockDim.x) {
      const uint64_t c = s_cand[t];
      int r0 = 0, r1 = 0;
      int j = 0;
      for (; j + 1 < cnt; j += 2) {
        r0 += s_cand[j] > c;
        r1 += s_cand[j + 1] > c;
      }
      if (j < cnt) r0 += s_cand[j] > c;
      const int r = r0 + r1;
      if (r < KK) s_top[r] = c;
    }
    if (tid < KK && tid >= cnt) s_top[tid] = 0ull;
  } else if (warp == 0) {
    uint64_t bb;
    if (cnt <= 256) {
      uint64_t c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int q = lane + 32 * j;
        c[j] = q < cnt ? s_cand[q] : 0ull;
      }
      bb = warp_select<KK, 8>(c);
    } else {
      constexpr int NC = TOPK_CAP / 32;
      uint64_t c[NC];
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        const int q = lane + 32 * j;
        c[j] = q < cnt ? s_cand[q] : 0ull;
      }
      bb = warp_select<KK, NC>(c);
    }
    if (lane < KK) s_top[lane] = bb;
  }
  __syncthreads();
}

// The CTA's top-KK (s_top) into slot crank of the cluster leader's s_clus, through
// distributed shared memory. Call it once every CTA of the cluster is known to be running.
template <int KK>
__device__ __forceinline__ void send_to_leader(cg::cluster_group &cluster, int crank,
                                               const uint64_t *s_top, uint64_t *s_clus) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == 0 && lane < KK) {
    uint64_t *leader = cluster.map_shared_rank(s_clus, 0);
    leader[crank * KK + lane] = s_top[lane];
  }
}

// The leader's warp 0 merges the CL lists of its s_clus (after a cluster barrier) and writes
// the row's top-k ids and values.
template <int KK, int CL>
__device__ __forceinline__ void leader_write(int crank, const uint64_t *s_clus, const float *x,
                                             int row, int k, int32_t *__restrict__ ids,
                                             float *__restrict__ vals) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (crank == 0 && warp == 0) {
    constexpr int NC = (CL * KK + 31) / 32;
    uint64_t c[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int q = lane + 32 * j;
      c[j] = q < CL * KK ? s_clus[q] : 0ull;
    }
    const uint64_t best = warp_select<KK, NC>(c);
    if (lane < k) {
      const int id = best ? unpack_idx(best) : -1;
      const uint32_t kb = (uint32_t)(best >> 32);
      ids[(size_t)row * k + lane] = id;
      // the order key gives the value back exactly, except for the sign of a zero and the
      // payload of a NaN: those few are read from the row
      vals[(size_t)row * k + lane] = id < 0 ? __int_as_float(0x7fc00000)
                                     : (kb == 0x80000000u || kb == 1u) ? x[id] : key_floor(kb);
    }
  }
}

}  // namespace gt
