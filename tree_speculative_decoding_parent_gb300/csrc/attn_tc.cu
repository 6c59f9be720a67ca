// tcgen05 split-KV tree attention for bf16 Q/K/V (fp32 accumulation in tensor memory).
//
// Sources: "浙江大学、阿里巴巴联手破解AI推理瓶颈" §二 third gear (one parallel verify forward of
// the flattened tree with an ancestor mask); "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码
// 跨越快与好的单选题" §三 (tree-attention verification).
//
// One CTA = one piece of a segment (request b, KV head h, a run of 128-key tiles) for up to
// 256 query rows (two 128-row M-tiles; row r = node * g + head-in-group). Roles:
//   warp 8      TMA producer: Q once, then K(0), V(0), K(1), V(1), ... into one ring of
//               5 slots of 32 KB (evict-first). A slot is reused in load order, so a K slot
//               frees as soon as Q K^T has read it and the next V can stream in early;
//   warp 9      MMA issuer (one thread) and TMEM owner: per tile and M-tile m,
//               S_m = Q_m K^T (SMEM x SMEM), then O_m += P_m V (P from TMEM, V from SMEM),
//               each MMA waiting only for the operands it reads;
//   warps 10-11 idle (they complete the third warpgroup, which gives its registers away);
//   warps 0-3   softmax of M-tile 0, warps 4-7 softmax of M-tile 1: each thread owns one
//               query row, reads its S row from TMEM, applies the prefix/ancestor mask,
//               keeps a running max and sum, writes P (bf16) back over its S row, and at
//               the end writes the normalised partial O row and its log-sum-exp.
// 128-key tiles keep every MMA at N = 128, where one tcgen05.mma of M=128, K=16 runs at
// the tensor pipe's full rate (N = 64 loses about a third of it).
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512);
// P_m occupies the first 64 columns of S_m as bf16 pairs. MMAs issued by one thread run
// in issue order, so S_m(j+1) overwrites P_m(j) only after O_m += P_m(j) V has read it,
// and the completion of S_m(j+1) implies O_m holds every tile up to j (used for lazy
// rescaling: O is rescaled only when a row's max grows by more than 2^8).
// Cache rows past a request's length may hold anything: their scores are masked by
// predicate and their V rows are zeroed in shared memory before the P V product.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "attn_tc.cuh"
#include "gt_internal.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace gt {

namespace {

constexpr int TC_THREADS = 384;     // 8 softmax warps + producer + MMA + 2 idle warps
// Register split: launched at TC_LAUNCH_REGS per thread (the most 12 warps can hold with 3
// warps per SM sub-partition), then the producer/MMA warpgroup drops to TC_LOW_REGS and
// the two softmax warpgroups rise to TC_HIGH_REGS. 2*128*224 + 128*56 = 384*168: the split
// uses exactly the registers the CTA was launched with.
constexpr int TC_LAUNCH_REGS = 168, TC_LOW_REGS = 56, TC_HIGH_REGS = 224;
static_assert(2 * 128 * TC_HIGH_REGS + 128 * TC_LOW_REGS == TC_THREADS * TC_LAUNCH_REGS,
              "register split must match the launch budget");
constexpr int TK = ATTN_TC_KEYS;    // keys per tile (128)
constexpr int SLOTS = 5;            // ring slots, each one K or one V tile
constexpr int HALF_BYTES = 16384;   // 128 rows x 64 d x bf16 (one 128B-swizzled box)
constexpr int SLOT_BYTES = 2 * HALF_BYTES;  // one tile: 128 keys x 128 d
constexpr uint32_t TMEM_COLS = 512;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
static_assert(TK == 128, "the tile shape above assumes 128-key tiles");

struct Smem {
  // offsets from the 1024-aligned base
  static constexpr int Q = 0;                          // [2 m][2 half] x 16 KB
  static constexpr int RING = Q + 4 * HALF_BYTES;      // [SLOTS] x 32 KB
  static constexpr int BAR = RING + SLOTS * SLOT_BYTES;
  static constexpr int NBAR = 1 + 2 * SLOTS + 2 + 2 + 2 + 1;
  static constexpr int END = BAR + NBAR * 8;
};
constexpr size_t TC_SMEM = Smem::END + 1024;  // + alignment slack
static_assert(TC_SMEM <= 232448, "shared memory of one CTA");

struct Bars {
  uint64_t *q_full, *full, *empty, *s_full, *p_full, *o_done, *drain;
};

__device__ __forceinline__ Bars bars_at(uint8_t *base) {
  uint64_t *b = reinterpret_cast<uint64_t *>(base + Smem::BAR);
  Bars r;
  r.q_full = b;
  r.full = b + 1;
  r.empty = r.full + SLOTS;
  r.s_full = r.empty + SLOTS;
  r.p_full = r.s_full + 2;
  r.o_done = r.p_full + 2;
  r.drain = r.o_done + 2;
  return r;
}

// Load sequence: item 2j is K(j), item 2j+1 is V(j); item q lives in slot q % SLOTS and is
// that slot's use number q / SLOTS.
__device__ __forceinline__ int slot_of(int q) { return q % SLOTS; }
__device__ __forceinline__ uint32_t use_parity(int q) { return (uint32_t)((q / SLOTS) & 1); }

// Bounded wait that ignores the abort flag (used only while draining in-flight work).
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
  int never = 0;
  return tc::mbar_wait(bar, parity, &never);
}

__global__ void __launch_bounds__(TC_THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ CUtensorMap mapV, const uint64_t *__restrict__ mask,
               const int32_t *__restrict__ prefix_len, const int32_t *__restrict__ n_nodes,
               int N, int Hq, int Hkv, float scale, SchedArgs sa, AttnWs ws, int32_t *err) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;

  const int p = blockIdx.x;
  const int4 pc = schedule_piece(sa, p, ws, err);
  if (pc.x < 0) return;
  const int seg = pc.x, b = seg / Hkv, h = seg - b * Hkv;
  const int g = Hq / Hkv;
  const int n = n_nodes[b], P = prefix_len[b], keys = P + n;
  const int row0 = blockIdx.y * 256;          // first segment row of this CTA
  const int rows_valid = g * n - row0;        // rows of this CTA holding real queries
  if (rows_valid <= 0) return;
  const int mtiles = rows_valid > 128 ? 2 : 1;
  const int t0 = pc.y, nt = pc.z - pc.y;

  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Bars bar = bars_at(base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    abort_sh = 0;
    tc::mbar_init(bar.q_full, 1);
    for (int s = 0; s < SLOTS; ++s) {
      tc::mbar_init(bar.full + s, 1);
      tc::mbar_init(bar.empty + s, 1);
    }
    for (int m = 0; m < 2; ++m) {
      tc::mbar_init(bar.s_full + m, 1);
      tc::mbar_init(bar.p_full + m, 128);
      tc::mbar_init(bar.o_done + m, 1);
    }
    tc::mbar_init(bar.drain, 1);
    tc::fence_mbar_init();
  }
  if (warp == 9) {
    tc::tmem_alloc(&tmem_sh, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_sh;
  volatile int *abort = &abort_sh;

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(TC_LOW_REGS));
    if (warp == 8 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      tc::tma_prefetch_desc(&mapQ);
      tc::tma_prefetch_desc(&mapK);
      tc::tma_prefetch_desc(&mapV);
      const uint64_t pol_kv = tc::policy_evict_first();
      const uint64_t pol_q = tc::policy_evict_last();
      tc::mbar_expect_tx(bar.q_full, mtiles * 2 * HALF_BYTES);
      for (int m = 0; m < mtiles; ++m) {
        const int node0 = (row0 + m * 128) / g;
        for (int hf = 0; hf < 2; ++hf)
          tc::tma_load_4d(base + Smem::Q + (m * 2 + hf) * HALF_BYTES, &mapQ, bar.q_full, hf * 64,
                          0, h, b * N + node0, pol_q);
      }
      const int plane = b * Hkv + h;
      int last = -1;
      for (int q = 0; q < 2 * nt; ++q) {
        const int s = slot_of(q);
        if (q >= SLOTS && !tc::mbar_wait(bar.empty + s, use_parity(q - SLOTS), abort)) break;
        uint8_t *dst = base + Smem::RING + s * SLOT_BYTES;
        const CUtensorMap *map = (q & 1) ? &mapV : &mapK;
        const int kb = (t0 + (q >> 1)) * TK;
        tc::mbar_expect_tx(bar.full + s, SLOT_BYTES);
        for (int hf = 0; hf < 2; ++hf)
          tc::tma_load_3d(dst + hf * HALF_BYTES, map, bar.full + s, hf * 64, kb, plane, pol_kv);
        last = q;
      }
      if (*abort) {  // let every issued copy land before the CTA's shared memory goes away
        drain_wait(bar.q_full, 0);
        for (int q = (last - SLOTS + 1 > 0 ? last - SLOTS + 1 : 0); q <= last; ++q)
          drain_wait(bar.full + slot_of(q), use_parity(q));
      }
    } else if (warp == 9 && lane == 0) {
      // -------------------------------------------------------------- MMA issuer
      constexpr uint32_t idS = tc::idesc_bf16(128, TK, false, false);
      constexpr uint32_t idO = tc::idesc_bf16(128, 128, false, true);
      const uint32_t sQ = tc::smem_u32(base + Smem::Q);
      const uint32_t ring = tc::smem_u32(base + Smem::RING);
      auto issue_s = [&](int m, int s) {  // S_m = Q_m K^T over d = 128 (8 steps of 16)
        const uint32_t q0 = sQ + m * 2 * HALF_BYTES, k0 = ring + s * SLOT_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * HALF_BYTES + (kk & 3) * 32;
          tc::mma_ss(tmem + m * 128, tc::sdesc_sw128(q0 + off, 16, 1024),
                     tc::sdesc_sw128(k0 + off, 16, 1024), idS, kk > 0);
        }
      };
      bool ok = tc::mbar_wait(bar.q_full, 0, abort) &&
                tc::mbar_wait(bar.full + slot_of(0), use_parity(0), abort);
      if (ok) {
        tc::tc_fence_after();
        for (int m = 0; m < mtiles; ++m) {
          issue_s(m, slot_of(0));
          tc::mma_commit(bar.s_full + m);
        }
        tc::mma_commit(bar.empty + slot_of(0));  // K(0) is free once both S_m(0) are done
      }
      for (int j = 0; ok && j < nt; ++j) {
        const int qv = 2 * j + 1, qk = 2 * j + 2;  // V(j), K(j+1)
        const bool next = j + 1 < nt;
        if (!tc::mbar_wait(bar.full + slot_of(qv), use_parity(qv), abort)) break;
        const uint32_t v0 = ring + slot_of(qv) * SLOT_BYTES;
        for (int m = 0; m < mtiles; ++m) {
          if (!tc::mbar_wait(bar.p_full + m, j & 1, abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // O_m += P_m V over 128 keys (steps of 16)
            tc::mma_ts(tmem + 256 + m * 128, tmem + m * 128 + kk * 8,
                       tc::sdesc_sw128(v0 + kk * 2048, HALF_BYTES, 1024), idO, (j > 0) || (kk > 0));
          if (next) {
            if (m == 0 && !tc::mbar_wait(bar.full + slot_of(qk), use_parity(qk), abort)) {
              ok = false;
              break;
            }
            issue_s(m, slot_of(qk));
            tc::mma_commit(bar.s_full + m);
          }
        }
        if (!ok) break;
        tc::mma_commit(bar.empty + slot_of(qv));            // V(j) read by both P V
        if (next) tc::mma_commit(bar.empty + slot_of(qk));  // K(j+1) read by both S
      }
      if (ok)
        for (int m = 0; m < mtiles; ++m) tc::mma_commit(bar.o_done + m);
      tc::mma_commit(bar.drain);  // every MMA issued above completes before teardown
      drain_wait(bar.drain, 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(TC_HIGH_REGS));
    // ------------------------------------------------------------------- softmax
    const int m = warp >> 2;                       // M-tile of this warpgroup
    const int rl = (warp & 3) * 32 + lane;          // row within the M-tile = TMEM lane
    const int r = row0 + m * 128 + rl;              // row within the segment
    const bool active = m < mtiles;
    const bool row_ok = r < g * n;
    const uint64_t mrow = row_ok ? mask[(size_t)b * N + r / g] : 0ull;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + m * 128;
    const uint32_t tO = tmem + lane_base + 256 + m * 128;
    const float sl2 = scale * LOG2E;  // scale > 0: the max of raw scores gives the max
    float m_used = -INFINITY, l = 0.f;  // running max (log2 units) and sum of this row
    bool ok = active;
    for (int j = 0; ok && j < nt; ++j) {
      // wait results are made warp-uniform: the TMEM accesses below are warp-collective
      if (!__all_sync(0xffffffffu, tc::mbar_wait(bar.s_full + m, j & 1, abort))) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(tS + c * 32, s[c]);
      tc::tmem_wait_ld();
      const int kb = (t0 + j) * TK;
      // 8 independent partial maxima of the raw scores keep the dependent chain short
      float mxa[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mxa[a] = -INFINITY;
      if (kb + TK <= P) {  // whole tile inside the committed prefix: every key visible
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int q = 0; q < 32; ++q) mxa[q & 7] = fmaxf(mxa[q & 7], __uint_as_float(s[c][q]));
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const int key = kb + c * 32 + q;
            const bool vis =
                key < P || (key < keys && ((mrow >> (unsigned)(key - P)) & 1ull));
            if (!vis) s[c][q] = __float_as_uint(-INFINITY);
            mxa[q & 7] = fmaxf(mxa[q & 7], __uint_as_float(s[c][q]));
          }
      }
      const float mx = sl2 * fmaxf(fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])),
                                   fmaxf(fmaxf(mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7])));
      // lazy rescale: move the reference max only when it grows by more than 8 (x256)
      const bool grow = mx > m_used + 8.f;
      float alpha = 1.f;
      if (grow) {
        alpha = (m_used == -INFINITY) ? 0.f : tc::ex2_approx(m_used - mx);
        m_used = mx;
      }
      if (__any_sync(0xffffffffu, grow && j > 0)) {
        // O holds every earlier tile (S_m(j) completed after O_m += P_m(j-1) V)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(tO + c * 32, o);
          tc::tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int q = 0; q < 16; ++q)
              w[q] = __float_as_uint(__uint_as_float(o[half * 16 + q]) * alpha);
            tc::tmem_st16(tO + c * 32 + half * 16, w);
          }
        }
        tc::tmem_wait_st();
      }
      l *= alpha;
      // p = 2^(s * scale * log2 e - m); a row with no visible key so far has m = -inf and
      // every s = -inf: its p are 0 (not NaN)
      const float msub = m_used == -INFINITY ? 0.f : m_used;
      float la[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) la[a] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float p0 = tc::ex2_approx(fmaf(__uint_as_float(s[c][2 * q]), sl2, -msub));
          const float p1 = tc::ex2_approx(fmaf(__uint_as_float(s[c][2 * q + 1]), sl2, -msub));
          la[q & 7] += p0 + p1;
          pk[q] = tc::pack_bf16x2(p0, p1);
        }
        tc::tmem_st16(tS + c * 16, pk);
      }
      l += ((la[0] + la[1]) + (la[2] + la[3])) + ((la[4] + la[5]) + (la[6] + la[7]));
      tc::tmem_wait_st();
      if (m == 0 && kb + TK > keys) {
        // zero V rows past the request's length (they may hold NaN) before P V reads them
        const int qv = 2 * j + 1;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(bar.full + slot_of(qv), use_parity(qv), abort))) {
          ok = false;
          break;
        }
        uint8_t *vt = base + Smem::RING + slot_of(qv) * SLOT_BYTES;
        const int first = keys - kb > 0 ? keys - kb : 0;
        for (int e = rl; e < (TK - first) * 16; e += 128) {
          const int row = first + e / 16, chunk = e % 16;  // 2 halves x 8 chunks of 16 B
          *reinterpret_cast<uint4 *>(vt + (chunk >> 3) * HALF_BYTES + row * 128 +
                                     (chunk & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        tc::fence_proxy_async_smem();
      }
      tc::tc_fence_before();
      tc::mbar_arrive(bar.p_full + m);
    }
    if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(bar.o_done + m, 0, abort));
    if (ok) {
      tc::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float *dst = ws.opart + ((size_t)p * ws.rows_pad + r) * ATTN_D;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tO + c * 32, o);
        tc::tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 32; q += 4)
            *reinterpret_cast<float4 *>(dst + c * 32 + q) =
                make_float4(__uint_as_float(o[q]) * inv, __uint_as_float(o[q + 1]) * inv,
                            __uint_as_float(o[q + 2]) * inv, __uint_as_float(o[q + 3]) * inv);
        }
      }
      if (row_ok)
        ws.lse[(size_t)p * ws.rows_pad + r] = l > 0.f ? (m_used + log2f(l)) * LN2 : -INFINITY;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort) set_err(err, GT_ERR_TIMEOUT);
  if (warp == 9) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool encode(CUtensorMap *map, const void *ptr, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides_bytes, const cuuint32_t *box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims,
            strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attn_tc_supported(int g, int N) {
  return g >= 1 && g <= 128 && (128 % g) == 0 && g * N <= 512;
}

int attn_tc_launch(const void *Q, const void *K, const void *V, const uint64_t *mask,
                   const SchedArgs &sa, int B, int N, int Hq, int Hkv, int Lcap, float scale,
                   const AttnWs &ws, int32_t *err, cudaStream_t s) {
  const int g = Hq / Hkv;
  CUtensorMap mQ, mK, mV;
  const cuuint64_t qdims[4] = {(cuuint64_t)ATTN_D, (cuuint64_t)g, (cuuint64_t)Hkv,
                               (cuuint64_t)B * N};
  const cuuint64_t qstr[3] = {(cuuint64_t)ATTN_D * 2, (cuuint64_t)g * ATTN_D * 2,
                              (cuuint64_t)Hq * ATTN_D * 2};
  const cuuint32_t qbox[4] = {64, (cuuint32_t)g, 1, (cuuint32_t)(128 / g)};
  const cuuint64_t kdims[3] = {(cuuint64_t)ATTN_D, (cuuint64_t)Lcap, (cuuint64_t)B * Hkv};
  const cuuint64_t kstr[2] = {(cuuint64_t)ATTN_D * 2, (cuuint64_t)Lcap * ATTN_D * 2};
  const cuuint32_t kbox[3] = {64, (cuuint32_t)TK, 1};
  if (!encode_fn()) {
    note_error("cuTensorMapEncodeTiled entry point", cudaErrorNotSupported);
    return GT_ERR_CUDA;
  }
  if (!encode(&mQ, Q, 4, qdims, qstr, qbox)) {
    note_error("cuTensorMapEncodeTiled(Q)", cudaErrorInvalidValue);
    return GT_ERR_CUDA;
  }
  if (!encode(&mK, K, 3, kdims, kstr, kbox) || !encode(&mV, V, 3, kdims, kstr, kbox)) {
    note_error("cuTensorMapEncodeTiled(K/V)", cudaErrorInvalidValue);
    return GT_ERR_CUDA;
  }
  static bool attr = false;
  if (!attr) {
    // the register split above is only valid at exactly TC_LAUNCH_REGS per thread
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_tc_kernel);
    if (e != cudaSuccess) return launch_status(e, "cudaFuncGetAttributes(attn_tc_kernel)");
    if (fa.numRegs != TC_LAUNCH_REGS) {
      note_error("attn_tc_kernel register count differs from its register split",
                 cudaErrorInvalidConfiguration);
      return GT_ERR_CUDA;
    }
    e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)TC_SMEM);
    if (e != cudaSuccess) return launch_status(e, "cudaFuncSetAttribute(attn_tc_kernel)");
    attr = true;
  }
  const int row_groups = ceil_div(g * N, 256);
  return launch(attn_tc_kernel, dim3(ws.maxp, row_groups), dim3(TC_THREADS), TC_SMEM, s, mQ, mK,
                mV, mask, sa.prefix_len, sa.n_nodes, N, Hq, Hkv, scale, sa, ws, err);
}

}  // namespace gt
