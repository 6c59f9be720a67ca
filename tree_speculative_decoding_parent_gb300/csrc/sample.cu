// a5 at temperature T > 0: one draw per logit row from softmax(z / T).
//
// Sources: "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题" §三 (the pruned
// tree goes to tree-attention verification and rejection sampling) and §七 (rejection
// sampling keeps the target's output distribution). The tree's proposals are point masses
// (top-m children, retrieved successors); rejection sampling of point masses is the same
// distribution as one target draw per node followed by a walk into the first child that
// carries the draw, so a draw per row is all the verification needs from the logits.
//
// The draw is the Gumbel-max sample: argmax_j z_j * (1/T) + G_j with G_j = -log(-log U_j)
// (Gumbel 1954; Maddison, Tarlow, Minka 2014). U_j = ((x_j >> 9) + 0.5) * 2^-23 for a 32-bit
// word x_j built from two Philox-4x32-10 blocks (Salmon, Moraes, Dror, Shaw, SC 2011) keyed
// by the seed (see SMP_GB below). The logarithm is this file's own float32 routine, the artanh
// series after splitting off the binary exponent (Abramowitz & Stegun 4.1.27). Every
// float32 operation is an explicit round-to-nearest intrinsic, so no contraction changes
// the result and any IEEE float32 implementation of the same steps draws the same token.
//
// Design: the row is split over a cluster of CL CTAs of 256 threads; each thread owns
// units of 16 consecutive logits (four 16-byte loads when the row allows it) and one Philox
// block per unit, whose bytes mark the few candidate elements (1 in 256) that alone need
// an exact score in the usual case. The (order key, lowest index) pairs meet in warp
// shuffles, shared memory and the cluster's distributed shared memory. With one Philox
// block per 16 logits the pass is close to the bound of reading the logits once.
//
// The same pass can also form the row's top-k of the unscaled logits (the table update at
// T > 0 keeps the target's k most likely tokens): with KK > 0 every thread also filters its
// units against the top-k threshold of topk_cluster_kernel (the KK-th largest of the CTA's
// lane maxima, here over each thread's first unit), and the candidates meet through the
// same warp selection and cluster merge. The logits are then read once for both results.
#include <math.h>

#include "gt_internal.cuh"
#include "launch.cuh"
#include "sample.cuh"
#include "topk_common.cuh"

namespace gt {

constexpr int SMP_THREADS = 256;
constexpr int SMP_CLUSTER = 8;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Natural logarithm of a positive normal float: x = 2^e * m, m in [sqrt(2)/2, sqrt(2)),
// s = (m - 1) / (m + 1), log m = 2s (1 + s^2/3 + s^4/5 + s^6/7 + s^8/9).
__device__ __forceinline__ float log_artanh(float x) {
  const uint32_t bits = __float_as_uint(x);
  const uint32_t mant = bits & 0x7FFFFFu;
  const bool big = mant > 0x3504F3u;  // mantissa field of float(sqrt 2)
  const int e = (int)(bits >> 23) - 127 + (big ? 1 : 0);
  const float m = __uint_as_float(mant | (big ? 0x3F000000u : 0x3F800000u));
  const float s = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
  const float z = __fmul_rn(s, s);
  float p = 1.0f / 9.0f;
  p = __fadd_rn(__fmul_rn(p, z), 1.0f / 7.0f);
  p = __fadd_rn(__fmul_rn(p, z), 1.0f / 5.0f);
  p = __fadd_rn(__fmul_rn(p, z), 1.0f / 3.0f);
  p = __fadd_rn(__fmul_rn(p, z), 1.0f);
  const float lm = __fmul_rn(__fadd_rn(s, s), p);
  return __fadd_rn(__fmul_rn((float)e, 0.693147180559945309f), lm);
}

__device__ __forceinline__ float gumbel_of(uint32_t x) {
  const float u = __fmul_rn(__fadd_rn((float)(x >> 9), 0.5f), 1.1920928955078125e-7f);
  return -log_artanh(-log_artanh(u));
}

__device__ __forceinline__ uint64_t smp_pack(float score, int j) {
  return ((uint64_t)order_key(score) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)j);
}

__device__ __forceinline__ uint64_t smp_max(uint64_t a, uint64_t b) { return a > b ? a : b; }

// The noise word of element j of row r is x_j = (A_j << 24) | (B_j >> 8): A_j is byte
// j % 16 (little-endian, word (j % 16) / 4) of the Philox block at counter (j / 16, r, step
// low, step high), B_j word j % 4 of the block at counter (j / 4 + 2^31, r, step low, step
// high). Elements with A_j = 255 are the candidates (U_j > 0.99609, G_j > 5.5432); every other
// element has G_j <= 5.5432057 (checked over all its possible words) < SMP_GB. The best
// candidate's score is a lower bound thr of the winning score; an element with
// fl(fl(z * 1/T) + SMP_GB) below thr (in the order of the draw) scores below the winner
// (rounding is monotone), so it cannot win and neither its B word nor its logarithms are
// needed. When even the row's largest z fails that test the candidates decide the draw in
// one pass; otherwise each thread scores the elements of its part that pass it.
constexpr float SMP_GB = 5.546f;
constexpr int SMP_QCAP = 1536;  // candidate queue per CTA (expected: the part's size / 256)

// float of an order key of a number (keys 0 and 1, empty and NaN, give -inf)
__device__ __forceinline__ float smp_key_value(uint32_t k) {
  if (k <= 1u) return -INFINITY;
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

__device__ __forceinline__ uint32_t word_of(uint4 w, int i) {
  return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}

struct SmpRow {
  int row, V;
  float inv_t;
  uint32_t k0, k1, s_lo, s_hi;
  __device__ __forceinline__ uint4 block_a(int u) const {
    return philox4x32_10(make_uint4((uint32_t)u, (uint32_t)row, s_lo, s_hi), k0, k1);
  }
  __device__ __forceinline__ uint32_t byte_a(uint4 a, int e) const {
    return (word_of(a, e >> 2) >> (8 * (e & 3))) & 0xFFu;
  }
  // exact score of element j given its A byte
  __device__ __forceinline__ float score(float z, int j, uint32_t a_byte) const {
    const uint4 bw = philox4x32_10(
        make_uint4((uint32_t)(j >> 2) | 0x80000000u, (uint32_t)row, s_lo, s_hi), k0, k1);
    const uint32_t xw = (a_byte << 24) | (word_of(bw, j & 3) >> 8);
    return __fadd_rn(__fmul_rn(z, inv_t), gumbel_of(xw));
  }
  __device__ __forceinline__ bool can_reach(float z, uint32_t thr) const {
    return order_key(__fadd_rn(__fmul_rn(z, inv_t), SMP_GB)) >= thr;
  }
};

// Max of (best, zk) over the cluster: warp shuffles, the CTA's warps, then every CTA writes
// its pair into slot crank of every CTA's (s_cb, s_cz) and each CTA reduces its copy.
template <int CL>
__device__ __forceinline__ void smp_cluster_max(uint64_t &best, uint32_t &zk, uint64_t *s_warp,
                                                uint32_t *s_wz, uint64_t *s_cb, uint32_t *s_cz,
                                                cg::cluster_group &cluster, int crank) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) best = smp_max(best, __shfl_xor_sync(0xffffffffu, best, o));
  zk = __reduce_max_sync(0xffffffffu, zk);
  if (lane == 0) {
    s_warp[warp] = best;
    s_wz[warp] = zk;
  }
  __syncthreads();
  if (warp == 0) {
    uint64_t b = lane < SMP_THREADS / 32 ? s_warp[lane] : 0ull;
    uint32_t z = lane < SMP_THREADS / 32 ? s_wz[lane] : 0u;
#pragma unroll
    for (int o = 16; o; o >>= 1) b = smp_max(b, __shfl_xor_sync(0xffffffffu, b, o));
    z = __reduce_max_sync(0xffffffffu, z);
    if (lane < CL) {
      *cluster.map_shared_rank(&s_cb[crank], lane) = b;
      *cluster.map_shared_rank(&s_cz[crank], lane) = z;
    }
  }
  cluster.sync();
  best = 0ull;
  zk = 0u;
#pragma unroll
  for (int c = 0; c < CL; ++c) {
    best = smp_max(best, s_cb[c]);
    zk = max(zk, s_cz[c]);
  }
}

// bit e of the result is set iff byte e of the block is 0xFF (a zero byte of ~w, found
// four at a time)
__device__ __forceinline__ uint32_t ff_bytes(uint4 a) {
  uint32_t m = 0u;
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t n = ~w[i];
    if (((n - 0x01010101u) & ~n & 0x80808080u) != 0u)  // some byte of w is 0xFF
#pragma unroll
      for (int c = 0; c < 4; ++c) m |= ((w[i] >> (8 * c)) & 0xFFu) == 0xFFu ? 1u << (4 * i + c) : 0u;
  }
  return m;
}

// exact scores of the elements of unit u whose bits are set in mask
__device__ __forceinline__ uint64_t score_mask(const SmpRow &R, const float (&z)[16], uint4 a,
                                               int u, uint32_t mask, uint64_t best) {
  while (mask) {
    const int e = __ffs(mask) - 1;
    mask &= mask - 1u;
    float v = 0.0f;
#pragma unroll
    for (int c = 0; c < 16; ++c) v = c == e ? z[c] : v;
    const int j = 16 * u + e;
    best = smp_max(best, smp_pack(R.score(v, j, R.byte_a(a, e)), j));
  }
  return best;
}

// KK > 0: the row's top-k (k <= KK) of the unscaled logits goes to ids / vals as well.
template <int CL, int KK>
__global__ void __launch_bounds__(SMP_THREADS, 4)
sample_cluster_kernel(const float *__restrict__ logits, int row0, int V, float inv_t,
                      uint32_t k0, uint32_t k1, uint32_t step_lo, uint32_t step_hi,
                      int32_t *__restrict__ sample, int k, int32_t *__restrict__ ids,
                      float *__restrict__ vals, int32_t *err) {
  static_assert(SMP_THREADS == TOPK_THREADS, "the top-k pieces assume 256 threads");
  constexpr int KS = KK > 0 ? KK : 1;  // array sizes of the top-k state
  pdl_enter();
  __shared__ uint64_t s_warp[SMP_THREADS / 32];
  __shared__ uint32_t s_wz[SMP_THREADS / 32];
  __shared__ uint64_t s_cb[2][CL];  // one set of cluster slots per reduction
  __shared__ uint32_t s_cz[2][CL];
  __shared__ int s_qj[SMP_QCAP];    // candidates found by the streaming pass: index, logit
  __shared__ float s_qz[SMP_QCAP];
  __shared__ int s_qn;
  __shared__ uint64_t s_tcand[KK > 0 ? TOPK_CAP : 1];  // top-k candidates
  __shared__ uint64_t s_top[KS];
  __shared__ uint64_t s_clus[CL * KS];
  __shared__ uint32_t s_lmax[(SMP_THREADS / 32) * KS];
  __shared__ uint32_t s_thr;
  __shared__ int s_tcnt;
  if (threadIdx.x == 0) {
    s_qn = 0;
    s_tcnt = 0;
  }
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const SmpRow R{row0 + (int)blockIdx.y, V, inv_t, k0, k1, step_lo, step_hi};
  const float *x = logits + (size_t)R.row * V;
  const int U16 = (V + 15) >> 4;  // units of 16 logits, one A block each
  const int ub = (int)((long long)U16 * crank / CL), ue = (int)((long long)U16 * (crank + 1) / CL);
  const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  const int V4 = V >> 2;
  // the 16 logits of unit u; lanes past the row's end read as -inf and are masked out
  auto load16 = [&](int u, float (&z)[16]) {
    if (vec) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int f = 4 * u + i;
        const float4 a = f < V4 ? __ldcg(reinterpret_cast<const float4 *>(x) + f)
                                : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        z[4 * i] = a.x, z[4 * i + 1] = a.y, z[4 * i + 2] = a.z, z[4 * i + 3] = a.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) z[e] = 16 * u + e < V ? x[16 * u + e] : -INFINITY;
    }
  };
  const uint32_t tail_mask = (V & 15) ? (1u << (V & 15)) - 1u : 0xFFFFu;  // valid lanes, last unit

  // pass 1: candidates' exact scores; the largest unit maximum of the part and the largest
  // of the other units' maxima
  uint64_t best = 0ull;
  float m1 = -INFINITY, m2 = -INFINITY;
  int u1 = -1;
  float zn[16];  // the next unit's logits are in flight while this unit is examined
  if (ub + (int)threadIdx.x < ue) load16(ub + (int)threadIdx.x, zn);
  float tthr = -INFINITY;  // top-k threshold
  bool nan_seen = false;   // checked builds: a NaN logit is reported as GT_ERR_VALUE
  if constexpr (KK > 0) {
    // the KK-th largest of the CTA's lane maxima over each thread's first unit: KK distinct
    // elements lie at or above it, so nothing below reaches the CTA's top-KK
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t km = 0u;
    const int u0 = ub + (int)threadIdx.x;
    if (u0 < ue)
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (16 * u0 + e < V) km = max(km, order_key(zn[e]));
    const uint32_t sorted = warp_sorted_desc(km);
    if (lane < KK) s_lmax[warp * KK + lane] = sorted;
    __syncthreads();
    if (warp == 0) {
      constexpr int NC = ((SMP_THREADS / 32) * KS + 31) / 32;
      uint32_t v = 0u;
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        const int q = lane + 32 * j;
        if (q < (SMP_THREADS / 32) * KK) v = max(v, s_lmax[q]);
      }
      const uint32_t kth = __shfl_sync(0xffffffffu, warp_sorted_desc(v), KK - 1);
      if (lane == 0) s_thr = kth;
    }
    __syncthreads();
    tthr = key_floor(s_thr);
  }
  for (int u = ub + (int)threadIdx.x; u < ue; u += SMP_THREADS) {
    float z[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) z[e] = zn[e];
    if (u + SMP_THREADS < ue) load16(u + SMP_THREADS, zn);
    const uint4 a = R.block_a(u);
    float um = z[0];
#pragma unroll
    for (int e = 1; e < 16; ++e) um = fmaxf(um, z[e]);  // NaN never counts
    if (um > m1) {
      m2 = m1;
      m1 = um;
      u1 = u;
    } else {
      m2 = fmaxf(m2, um);
    }
    if constexpr (KK > 0) {
      // the unit's elements not below tthr (NaN included) as a bit mask, then the rare set bits
      uint32_t tm = 0u;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        if (GT_CHECK && 16 * u + e < V) nan_seen |= z[e] != z[e];
        tm |= !(z[e] < tthr) ? 1u << e : 0u;
      }
      if (u == U16 - 1) tm &= tail_mask;
      while (tm) {
        const int e = __ffs(tm) - 1;
        tm &= tm - 1u;
        float v = 0.0f;
#pragma unroll
        for (int c = 0; c < 16; ++c) v = c == e ? z[c] : v;
        const int pos = atomicAdd(&s_tcnt, 1);
        if (pos < TOPK_CAP) s_tcand[pos] = pack_key(order_key(v), 16 * u + e);
      }
    }
    uint32_t cand = ff_bytes(a);
    if (u == U16 - 1) cand &= tail_mask;
    // queue the candidates; they are scored after the pass with every lane busy
    while (cand) {
      const int e = __ffs(cand) - 1;
      cand &= cand - 1u;
      float v = 0.0f;
#pragma unroll
      for (int c = 0; c < 16; ++c) v = c == e ? z[c] : v;
      const int slot = atomicAdd(&s_qn, 1);
      if (slot < SMP_QCAP) {
        s_qj[slot] = 16 * u + e;
        s_qz[slot] = v;
      }
    }
  }
  __syncthreads();
  if constexpr (KK > 0) {
    // the CTA's top-KK: the candidates, or the exact per-thread lists after an overflow
    const int tc = s_tcnt;
    if (tc > TOPK_CAP) {
      __syncthreads();  // the buffer is reused as scratch
      topk_exact<KK>(x, 16 * ub, min(16 * ue, V), s_tcand, s_top);
    } else {
      select_candidates<KK>(tc, s_tcand, s_top);
    }
    GT_CHECKED(!nan_seen, err, GT_ERR_VALUE);
  }
  const int qn = s_qn;
  for (int i = threadIdx.x; i < min(qn, SMP_QCAP); i += SMP_THREADS)
    best = smp_max(best, smp_pack(R.score(s_qz[i], s_qj[i], 0xFFu), s_qj[i]));
  // an overflowing queue leaves candidates unscored: the +inf key below sends the cluster
  // into pass 2, where this CTA rescans its whole part
  const bool overflow = qn > SMP_QCAP;
  uint32_t zk = overflow ? order_key(INFINITY) : order_key(m1);
  // every CTA of the cluster is running after the wait: the first remote write follows it
  asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
  // the top-k lists travel with the first reduction (its cluster barrier publishes them)
  if constexpr (KK > 0) send_to_leader<KK>(cluster, crank, s_top, s_clus);
  smp_cluster_max<CL>(best, zk, s_warp, s_wz, s_cb[0], s_cz[0], cluster, crank);
  if constexpr (KK > 0) leader_write<KK, CL>(crank, s_clus, x, R.row, k, ids, vals);

  const uint32_t thr = (uint32_t)(best >> 32);
  if (R.can_reach(smp_key_value(zk), thr)) {
    // pass 2 (the same decision in every CTA): the elements that can still reach thr. When
    // no other unit's maximum can, only the unit of the part's largest logit is scored.
    const bool one = thr > 1u && !overflow && !R.can_reach(m2, thr);
    // can_reach is monotone in z: when the part's largest logit m1 cannot reach thr, no
    // element of its unit can (and with `one`, no element of the other units either)
    const int ustart = one ? (R.can_reach(m1, thr) ? u1 : -1) : ub + (int)threadIdx.x;
    for (int u = ustart; u >= 0 && u < ue; u = one ? -1 : u + SMP_THREADS) {
      float z[16];
      load16(u, z);
      // the bound SMP_GB holds for non-candidates only: after an overflow the candidates
      // that missed the queue are scored whatever their logit
      uint32_t mask = 0u;
#pragma unroll
      for (int e = 0; e < 16; ++e) mask |= R.can_reach(z[e], thr) ? 1u << e : 0u;
      uint4 a = make_uint4(0u, 0u, 0u, 0u);
      if (overflow) {
        a = R.block_a(u);
        mask |= ff_bytes(a);
      }
      if (u == U16 - 1) mask &= tail_mask;
      if (mask) best = score_mask(R, z, overflow ? a : R.block_a(u), u, mask, best);
    }
    smp_cluster_max<CL>(best, zk, s_warp, s_wz, s_cb[1], s_cz[1], cluster, crank);
  }
  if (crank == 0 && threadIdx.x == 0)
    sample[R.row] = (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
}

template <int CL, int KK>
static int sample_launch_cl(const float *logits, int r0, int nr, int V, float inv_t, uint32_t k0,
                            uint32_t k1, uint32_t s_lo, uint32_t s_hi, int32_t *sample, int k,
                            int32_t *ids, float *vals, int32_t *err, cudaStream_t s) {
  return launch_cluster(sample_cluster_kernel<CL, KK>, dim3(CL, nr), dim3(SMP_THREADS),
                        dim3(CL, 1, 1), 0, s, logits, r0, V, inv_t, k0, k1, s_lo, s_hi, sample,
                        k, ids, vals, err);
}

template <int KK>
static int sample_launch_k(const float *logits, int r0, int nr, int V, float inv_t, uint32_t k0,
                           uint32_t k1, uint32_t s_lo, uint32_t s_hi, int32_t *sample, int k,
                           int32_t *ids, float *vals, int32_t *err, int cl, cudaStream_t s) {
  switch (cl) {
    case 1: return sample_launch_cl<1, KK>(logits, r0, nr, V, inv_t, k0, k1, s_lo, s_hi, sample, k, ids, vals, err, s);
    case 2: return sample_launch_cl<2, KK>(logits, r0, nr, V, inv_t, k0, k1, s_lo, s_hi, sample, k, ids, vals, err, s);
    case 4: return sample_launch_cl<4, KK>(logits, r0, nr, V, inv_t, k0, k1, s_lo, s_hi, sample, k, ids, vals, err, s);
    default:
      return sample_launch_cl<SMP_CLUSTER, KK>(logits, r0, nr, V, inv_t, k0, k1, s_lo, s_hi, sample, k,
                                               ids, vals, err, s);
  }
}

int sample_launch(const float *logits, int rows, int V, float temperature, uint64_t seed,
                  uint64_t step, int32_t *sample, cudaStream_t s, int k, int32_t *ids,
                  float *vals, int32_t *err) {
  if (!(temperature > 0.0f) || !isfinite(temperature)) return GT_ERR_ARG;
  const float inv_t = 1.0f / temperature;  // one IEEE float division
  if (!isfinite(inv_t)) return GT_ERR_ARG;
  if (V >= (1 << 30)) return GT_ERR_SHAPE;
  // CTAs per row: the most (up to 8) for which every CTA of the launch is resident at
  // once, so no second wave of a few CTAs trails the first
  int dev = 0, sms = 148, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm,
                                                    sample_cluster_kernel<SMP_CLUSTER, 16>,
                                                    SMP_THREADS, 0) != cudaSuccess) {
    (void)cudaGetLastError();
    sms = 148;
    per_sm = 2;
  }
  const long long slots = (long long)sms * max(per_sm, 1);
  int cl = SMP_CLUSTER;
  while (cl > 1 && (long long)rows * cl > slots) cl /= 2;
  const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  const uint32_t s_lo = (uint32_t)step, s_hi = (uint32_t)(step >> 32);
  for (int r0 = 0; r0 < rows; r0 += 65535) {
    const int nr = min(65535, rows - r0);
    const int rc =
        !ids ? sample_launch_k<0>(logits, r0, nr, V, inv_t, k0, k1, s_lo, s_hi, sample, k, ids, vals, err, cl, s)
        : k <= 8 ? sample_launch_k<8>(logits, r0, nr, V, inv_t, k0, k1, s_lo, s_hi, sample, k, ids, vals, err, cl, s)
                 : sample_launch_k<16>(logits, r0, nr, V, inv_t, k0, k1, s_lo, s_hi, sample, k, ids, vals, err, cl, s);
    if (rc != GT_OK) return rc;
  }
  return GT_OK;
}

}  // namespace gt
