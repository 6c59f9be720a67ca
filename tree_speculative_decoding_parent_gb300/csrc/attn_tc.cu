// tcgen05 split-KV tree attention for bf16 Q/K/V (fp32 accumulation in tensor memory).
//
// Sources: "浙江大学、阿里巴巴联手破解AI推理瓶颈" §二 third gear (one parallel verify forward of
// the flattened tree with an ancestor mask); "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码
// 跨越快与好的单选题" §三 (tree-attention verification).
//
// Work split. A segment (request b, KV head h) has g*N query rows (row r = node * g +
// head-in-group) and keys [0, P_b + n_b). The split-KV schedule cuts its 128-key tiles into
// pieces; one thread-block cluster of C = ceil(g*N / 128) CTAs runs one piece, CTA rank c
// owning query rows [128c, 128c + 128) as one 128-row M-tile. The CTAs of a cluster read
// the same K/V tiles: the first L CTAs (L = C rounded down to a power of two) each load
// 1/L of every tile with a cluster-multicast TMA, so every tile leaves L2 once and lands
// in all C shared memories.
//
// Roles (224 threads, one CTA per SM):
//   warp 4      TMA producer: the K/V items in consumption order, through a ring of 7
//               slots of 32 KB: K(0), K(1), K(2), V(0), K(3), V(1), ... (K runs two tiles
//               ahead of V). A slot is refilled once the MMA threads of all C CTAs released
//               its previous item (multicast tcgen05.commit). Past the first three items
//               the producer waits until this CTA's softmax threads hold their Q rows and
//               ancestor masks, so that those small loads are not queued behind the ring's
//               burst of loads at the start.
//   warp 5      Q K^T issuer (one thread) and tensor-memory owner. S(t) = Q K(t)^T goes to
//               one of two S buffers (Q from tensor memory, K from shared memory); S(j+2)
//               is issued as soon as the softmax has read S(j) into registers, so Q K^T
//               stays two tiles ahead.
//   warp 6      P V issuer (one thread): O += P(j) V(j) as soon as the softmax published
//               P(j). The two streams touch disjoint tensor and shared memory, so each
//               thread commits only its own MMAs. With one issuer, P V(j) would wait behind
//               the Q K^T(j+2) instructions (an MMA issue blocks for about the MMA's
//               execution time), and the softmax, which stores P(j+1) only after P V(j),
//               would wait with it.
//   warps 0-3   softmax: thread = query row = tensor-memory lane. First the thread copies
//               its Q row into tensor memory. Per tile: read the S row (and free its
//               buffer), mask, p = 2^(s*scale*log2e - m) with a lazily moved reference max
//               m, write P (bf16) into the P buffer once O += P(j-1) V(j-1) has read the
//               previous P, and at the end the normalised partial O row and its log-sum-exp.
// Tensor memory (512 columns): S buffers at [0,128) and [128,256), O at [256,384), Q at
// [384,448) and P at [448,512), both as bf16 pairs. Neither Q K^T nor the softmax ever
// waits for the other's previous tile, and the tensor pipe always holds the next S. Keeping
// Q out of shared memory leaves all of it to the ring and halves the shared-memory reads of
// each Q K^T step.
// Cache rows past a request's length may hold anything: their scores are masked by
// predicate and their V rows are zeroed in shared memory before the P V product.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>

#include "attn_tc.cuh"
#include "gt_internal.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace gt {

namespace {

constexpr int TC_THREADS = 224;     // 4 softmax warps + producer + two MMA issuers
constexpr int TK = ATTN_TC_KEYS;    // keys per tile (128)
constexpr int NSBUF = 2;            // S buffers in tensor memory
constexpr int KLEAD = 2;            // K tiles loaded ahead of V (= NSBUF)
constexpr int HALF_BYTES = 16384;   // 128 rows x 64 d x bf16 (one 128B-swizzled box)
constexpr int MAX_CLUSTER = 4;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = 256;
constexpr uint32_t Q_COL = 384;
constexpr uint32_t P_COL = 448;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
static_assert(TK == 128, "the tile shape above assumes 128-key tiles");
static_assert(KLEAD == NSBUF, "S(t + NSBUF) reuses the buffer of P(t)");

// Ring and barriers of one CTA; a slot holds one whole K or V tile.
struct Smem {
  static constexpr int SLOTS = 7;
  static constexpr int SLOT_BYTES = 2 * HALF_BYTES;
  // offsets from the 1024-aligned base
  static constexpr int RING = 0;
  static constexpr int BAR = RING + SLOTS * SLOT_BYTES;
  // q_full, full[SLOTS], empty[SLOTS], s_full[NSBUF], s_free[NSBUF], p_full, o_ready,
  // o_done, drain[2] (one per MMA issuer)
  static constexpr int NBAR = 1 + 2 * SLOTS + 2 * NSBUF + 5;
  static constexpr int END = BAR + NBAR * 8;
  static constexpr size_t BYTES = END + 1024;  // + alignment slack
  static_assert(BYTES + 768 <= 232448, "shared memory of one CTA (dynamic + static)");
  static_assert(128 * ATTN_D * 4 <= SLOTS * SLOT_BYTES, "partial rows are staged in the ring");
};
constexpr int RING_GATE = 3;  // ring items issued before the producer waits for q_full
// Of every 8 score pairs, this many take their exponentials from a polynomial on the FMA
// pipe and the rest from the special-function unit, whose rate (16 per SM and cycle) would
// otherwise bound the softmax of a tile.
#ifndef GT_ATTN_EX2_POLY_PAIRS
#define GT_ATTN_EX2_POLY_PAIRS 0
#endif
constexpr int EX2_POLY_PAIRS = GT_ATTN_EX2_POLY_PAIRS;

struct Bars {
  uint64_t *q_full, *full, *empty, *s_full, *s_free, *p_full, *o_ready, *o_done, *drain;
};

__device__ __forceinline__ Bars bars_at(uint8_t *base) {
  uint64_t *b = reinterpret_cast<uint64_t *>(base + Smem::BAR);
  Bars r;
  r.q_full = b;
  r.full = b + 1;
  r.empty = r.full + Smem::SLOTS;
  r.s_full = r.empty + Smem::SLOTS;
  r.s_free = r.s_full + NSBUF;
  r.p_full = r.s_free + NSBUF;
  r.o_ready = r.p_full + 1;
  r.o_done = r.o_ready + 1;
  r.drain = r.o_done + 1;
  return r;
}

// Item sequence of a piece of nt tiles, the order in which the MMA threads consume them:
// K(0..P0-1) with P0 = min(KLEAD, nt), then for j = 0..nt-1: K(j+KLEAD) while
// j+KLEAD < nt, followed by V(j). Item q sits in slot q % SLOTS as that slot's use number
// q / SLOTS. The last item is V(nt-1).
__device__ __forceinline__ int pos_v(int j, int nt) {
  const int p0 = min(KLEAD, nt), e = max(0, nt - KLEAD);
  return p0 + j + min(j + 1, e);
}
__device__ __forceinline__ int pos_k(int t, int nt) {
  const int p0 = min(KLEAD, nt);
  return t < p0 ? t : p0 + 2 * (t - KLEAD);
}
__device__ __forceinline__ void item_at(int q, int nt, bool &is_v, int &tile) {
  const int p0 = min(KLEAD, nt), e = max(0, nt - KLEAD);
  if (q < p0) {
    is_v = false;
    tile = q;
    return;
  }
  const int r = q - p0;
  if (r < 2 * e) {
    is_v = (r & 1) == 1;
    tile = (r >> 1) + (is_v ? 0 : KLEAD);
    return;
  }
  is_v = true;
  tile = e + (r - 2 * e);
}

// AND of `pred` over the four softmax warps (128 threads), through named barrier 1.
__device__ __forceinline__ int __syncthreads_and_named(bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((unsigned)pred)
      : "memory");
  return r;
}

// Bounded wait that ignores the abort flag (used only while draining in-flight work).
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
  int never = 0;
  return tc::mbar_wait(bar, parity, &never);
}

// ------------------------------------------------------------------ softmax pieces
// Q row r = node * g + head-in-group of the segment (b, h) into tensor memory at tQ (this
// warp's lanes), as 64 bf16 pairs (low half = even element), the tensor-memory layout of an
// M-tile operand; rows past the tree are zero. Returns once the stores completed.
__device__ __forceinline__ void q_row_to_tmem(const __nv_bfloat16 *__restrict__ Qg, int b, int N,
                                              int Hq, int h, int g, int r, uint32_t tQ) {
  const int node = r / g;
  uint32_t qw[64];
  if (node < N) {
    const uint4 *src = reinterpret_cast<const uint4 *>(
        Qg + (((size_t)b * N + node) * Hq + (size_t)h * g + (r - node * g)) * ATTN_D);
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      const uint4 x = __ldg(src + v);
      qw[4 * v] = x.x;
      qw[4 * v + 1] = x.y;
      qw[4 * v + 2] = x.z;
      qw[4 * v + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int v = 0; v < 64; ++v) qw[v] = 0u;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t w[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) w[q] = qw[c * 16 + q];
    tc::tmem_st16(tQ + c * 16, w);
  }
  tc::tmem_wait_st();
}

// Softmax of one tile for this thread's row: s holds the row's 128 raw scores of keys
// kb .. kb+127 (masked in place), P the committed prefix length, mrow the row's ancestor mask
// over the tree keys (no bit at or past the node count). Produces the P words (bf16 pairs)
// in pk, the factor alpha by which the running O and sum must be scaled, and updates the
// reference max m_used (log2 units) and the row sum l. `later` is true for every tile after
// the piece's first. Warp-collective (its votes keep the paths warp-uniform).
//
// p = 2^(s*scale*log2e - m_used) against a lazily moved reference max. A tile wholly inside
// the committed prefix, once the row has a finite reference, goes straight to the
// exponentials with the tile's sum as the overflow test: sum <= 2^15 = 128 * 2^8 means no p
// exceeded the lazy-rescale bound 2^8, so the result is what a max pass first would give
// (up to summation order). Otherwise (the first tile, a masked tile, or the rare growth of
// the row's max by more than 8 in log2 units) a max pass moves the reference first. Both
// cases run the same exponential loop, which keeps the code small: code that runs once per
// piece is fetched cold, at a cost that grows with its size.
__device__ __forceinline__ void softmax_tile(uint32_t (&s)[4][32], int kb, int P, uint64_t mrow,
                                             float sl2, bool later, float &m_used, float &l,
                                             float &alpha, uint32_t (&pk)[4][16]) {
  alpha = 1.f;
  if (kb + TK > P) {
    // visibility of the tile's keys as one 32-bit word per column of 32 keys: the prefix keys
    // below P, then the tree keys P + u whose bit u is set in the row's ancestor mask
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int key0 = kb + c * 32;
      const int np = min(max(P - key0, 0), 32);
      const uint32_t pre = np >= 32 ? 0xFFFFFFFFu : ((1u << np) - 1u);
      const int u0 = key0 - P;
      uint32_t tree = 0u;
      if (u0 >= 0 && u0 < 64)
        tree = (uint32_t)(mrow >> u0);
      else if (u0 < 0 && u0 > -32)
        tree = (uint32_t)(mrow << (-u0));
      const uint32_t vis = pre | tree;
#pragma unroll
      for (int q = 0; q < 32; ++q)
        if (!((vis >> q) & 1u)) s[c][q] = __float_as_uint(-INFINITY);
    }
  }
  bool need_max = __any_sync(0xffffffffu, !later || kb + TK > P || m_used == -INFINITY);
  float lt;
  for (int pass = 0;; ++pass) {
    if (need_max) {
      // 8 independent partial maxima of the raw scores keep the dependent chain short
      float mxa[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mxa[a] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int q = 0; q < 32; ++q) mxa[q & 7] = fmaxf(mxa[q & 7], __uint_as_float(s[c][q]));
      const float mx = sl2 * fmaxf(fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])),
                                   fmaxf(fmaxf(mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7])));
      // lazy rescale: move the reference max only when it grows by more than 8 (x256)
      if (mx > m_used + 8.f) {
        alpha = (m_used == -INFINITY) ? 0.f : tc::ex2_approx(m_used - mx);
        m_used = mx;
      }
    }
    // a row with no visible key so far has m = -inf and every s = -inf: its p are 0
    const float msub = m_used == -INFINITY ? 0.f : m_used;
    const uint64_t a2 = tc::f32x2_pack(sl2, sl2), c2 = tc::f32x2_pack(-msub, -msub);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        float p0, p1;
        if ((q & 7) < EX2_POLY_PAIRS) {  // this pair's exponentials on the FMA pipe
          float x0, x1;
          tc::fma_x2(__uint_as_float(s[c][2 * q]), __uint_as_float(s[c][2 * q + 1]), a2, c2, x0,
                     x1);
          p0 = tc::ex2_poly(x0);
          p1 = tc::ex2_poly(x1);
        } else {
          tc::ex2_fma_x2(__uint_as_float(s[c][2 * q]), __uint_as_float(s[c][2 * q + 1]), a2, c2,
                         p0, p1);
        }
        tc::add_x2(acc[q & 3], p0, p1);
        pk[c][q] = tc::pack_bf16x2(p0, p1);
      }
    lt = (tc::f32x2_sum(acc[0]) + tc::f32x2_sum(acc[1])) +
         (tc::f32x2_sum(acc[2]) + tc::f32x2_sum(acc[3]));
    // after a max pass every p <= 2^8 by construction; without one, the sum tests it
    // (false for inf and NaN too)
    if (need_max || pass > 0 || __all_sync(0xffffffffu, lt <= 32768.f)) break;
    need_max = true;
  }
  l = l * alpha + lt;
}

// O row (tensor memory at tO, this warp's lanes) *= alpha.
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    tc::tmem_ld32(tO + c * 32, o);
    tc::tmem_wait_ld();
    uint32_t w[16];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int q = 0; q < 16; ++q) w[q] = __float_as_uint(__uint_as_float(o[half * 16 + q]) * alpha);
      tc::tmem_st16(tO + c * 32 + half * 16, w);
    }
  }
}

// The normalised partial rows and their log-sum-exps. The rows are staged in shared memory
// (`stage`, idle once O is complete) as four boxes of 32 columns x 128 rows in the 128-byte
// swizzle of the tensor map mapO (16-byte chunk k of row r at chunk k ^ (r % 8), which keeps
// a warp's 16-byte writes free of bank conflicts), then one thread stores the four boxes with
// TMA. Rows past the tree are stored too (they lie inside the piece's padded rows and are
// never read). ok: this thread's waits all succeeded. Called by the 128 softmax threads.
__device__ __forceinline__ void write_partial(uint8_t *stage, const CUtensorMap *mapO,
                                              uint32_t tO, bool ok, float l, float m_used, int p,
                                              int row0, int rows, const AttnWs &ws) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, rl = warp * 32 + lane;
  const int r = row0 + rl;
  const bool wok = __all_sync(0xffffffffu, ok);
  if (wok) {
    tc::tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tc::tmem_ld32(tO + c * 32, o);
      tc::tmem_wait_ld();
      uint8_t *row = stage + c * (128 * 128) + rl * 128;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<float4 *>(row + ((k ^ (rl & 7)) << 4)) =
            make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                        __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
    }
    if (r < rows)
      ws.lse[(size_t)p * ws.rows_pad + r] = l > 0.f ? (m_used + log2f(l)) * LN2 : -INFINITY;
    tc::fence_proxy_async_smem();  // the staged rows are visible to the TMA engine
  }
  // the four softmax warps meet (named barrier 1, 128 threads); one thread stores the boxes
  const int wall = __syncthreads_and_named(wok);
  if (wall && threadIdx.x == 0) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      tc::tma_store_2d(mapO, stage + c * (128 * 128), c * 32, p * ws.rows_pad + row0);
    tc::bulk_commit();
    tc::bulk_wait_read_all();  // shared memory may be released once the stores have read it
  }
}

// The piece is its segment's only one, so its normalised rows are the output: each
// softmax thread scales its row by 1 / l, rounds it to bf16 and stores it (zero for nodes at
// or past n; rows past the segment's g * N are not stored). The combine of a single piece
// gives the same bits (weight exp(0) = 1, sum 1), so the combine kernel skips these rows.
// ok: this thread's waits all succeeded. Called by the 128 softmax threads.
__device__ __forceinline__ void write_final(uint32_t tO, bool ok, float l, int row0, int g,
                                            int n, int N, int Hq, int h, int b,
                                            __nv_bfloat16 *__restrict__ O) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = row0 + warp * 32 + lane;
  if (!__all_sync(0xffffffffu, ok)) return;
  const int i = r / g, hq = h * g + (r - i * g);
  const bool exists = r < g * N, live = i < n;
  const float inv = live && l > 0.f ? 1.f / l : 0.f;
  uint4 *dst = reinterpret_cast<uint4 *>(O + (((size_t)b * N + i) * Hq + hq) * ATTN_D);
  tc::tc_fence_after();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    tc::tmem_ld32(tO + c * 32, o);  // warp-collective: every lane loads
    tc::tmem_wait_ld();
    if (exists) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 v =
              __floats2bfloat162_rn(__uint_as_float(o[8 * k + 2 * e]) * inv,
                                    __uint_as_float(o[8 * k + 2 * e + 1]) * inv);
          w[e] = *reinterpret_cast<const uint32_t *>(&v);
        }
        dst[c * 4 + k] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

__global__ void __launch_bounds__(TC_THREADS, 1)
attn_tc_kernel(const __nv_bfloat16 *__restrict__ Qg, const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapO,
               uint32_t q_slice, uint32_t q_bytes, const uint64_t *__restrict__ mask,
               const int32_t *__restrict__ prefix_len, const int32_t *__restrict__ n_nodes,
               int N, int Hq, int Hkv, float scale, int C, int L, SchedArgs sa, AttnWs ws,
               __nv_bfloat16 *__restrict__ O, int32_t *err) {
  using Lay = Smem;
  constexpr int SLOTS = Lay::SLOTS, SLOT_BYTES = Lay::SLOT_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;

  const int rank = (int)tc::cluster_ctarank();
  const uint16_t all_mask = (uint16_t)((1u << C) - 1u);
  const bool multicast = C > 1;
  const int box_rows = TK / L;  // keys of each tile this CTA loads when rank < L
  uint8_t *base = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Bars bar = bars_at(base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Set-up that reads nothing the previous kernels of the stream write runs before the
  // programmatic-dependency wait, overlapping their tail: barriers, tensor memory, cluster.
  if (tid == 0) {
    abort_sh = 0;
    tc::mbar_init(bar.q_full, 128);  // every softmax thread stored its Q row
    for (int s = 0; s < SLOTS; ++s) {
      tc::mbar_init(bar.full + s, 1);
      tc::mbar_init(bar.empty + s, C);  // one release per CTA, by the thread whose MMAs read it
    }
    for (int s = 0; s < NSBUF; ++s) {
      tc::mbar_init(bar.s_full + s, 1);
      tc::mbar_init(bar.s_free + s, 128);  // every softmax thread read its S row
    }
    tc::mbar_init(bar.p_full, 128);
    tc::mbar_init(bar.o_ready, 1);
    tc::mbar_init(bar.o_done, 1);
    tc::mbar_init(bar.drain, 1);
    tc::mbar_init(bar.drain + 1, 1);
    tc::fence_mbar_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(&tmem_sh, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  // no CTA may multicast into a peer before the peer's barriers exist
  if (multicast) tc::cluster_sync_all();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_sh;
  volatile int *abort = &abort_sh;

  pdl_enter();
  // Q is read only after the schedule: each CTA asks L2 for its slice of it now, so that the
  // rows are on chip when the softmax threads load them
  if (tid == 0) {
    const uint32_t q0 = blockIdx.x * q_slice;
    if (q0 < q_bytes)
      tc::prefetch_l2_bulk(reinterpret_cast<const uint8_t *>(Qg) + q0, min(q_slice, q_bytes - q0));
  }
  // every CTA of a cluster gets the same piece, so a cluster leaves here as a whole
  const int p = blockIdx.x / C;
  int2 np;
  const int4 pc = schedule_piece(sa, p, ws, err, &np);
  if (pc.x < 0) {
    if (warp == 5) tc::tmem_dealloc(tmem, TMEM_COLS);
    return;
  }
  const int seg = pc.x, b = seg / Hkv, h = seg - b * Hkv;
  const int g = Hq / Hkv;
  const int n = np.x, P = np.y, keys = P + n;  // from the schedule: no second load
  const int row0 = rank * 128;  // first segment row of this CTA (may lie past g*n)
  const int t0 = pc.y, nt = pc.z - pc.y;
  const int total = 2 * nt;
  auto slot_of = [](int q) { return q % SLOTS; };
  auto use_parity = [](int q) { return (uint32_t)((q / SLOTS) & 1); };

  if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      tc::tma_prefetch_desc(&mapK);
      tc::tma_prefetch_desc(&mapV);
      const uint64_t pol_kv = tc::policy_evict_first();
      const int plane = b * Hkv + h;
      const bool loader = rank < L;
      for (int q = 0; q < total; ++q) {
        const int s = slot_of(q);
        if (q == RING_GATE && !tc::mbar_wait(bar.q_full, 0, abort)) break;
        if (q >= SLOTS && !tc::mbar_wait(bar.empty + s, use_parity(q - SLOTS), abort)) break;
        if (*abort) break;
        tc::mbar_expect_tx(bar.full + s, SLOT_BYTES);  // both halves of the whole tile
        if (loader) {
          bool is_v;
          int tile;
          item_at(q, nt, is_v, tile);
          const CUtensorMap *map = is_v ? &mapV : &mapK;
          const int kb = (t0 + tile) * TK + rank * box_rows;
          uint8_t *dst = base + Lay::RING + s * SLOT_BYTES + rank * box_rows * 128;
          for (int hf = 0; hf < 2; ++hf) {
            if (multicast)
              tc::tma_load_3d_mc(dst + hf * HALF_BYTES, map, bar.full + s, hf * 64, kb, plane,
                                 all_mask, pol_kv);
            else
              tc::tma_load_3d(dst + hf * HALF_BYTES, map, bar.full + s, hf * 64, kb, plane,
                              pol_kv);
          }
        }
      }
    }
  } else if (warp == 5 || warp == 6) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA issuers
      const bool qk = warp == 5;  // warp 5: Q K^T; warp 6: P V
      constexpr uint32_t idS = tc::idesc_bf16(128, TK, false, false);
      constexpr uint32_t idO = tc::idesc_bf16(128, 128, false, true);
      const uint32_t ring = tc::smem_u32(base + Lay::RING);
      // Descriptors are built once; a K step moves the start address, which sits in the
      // low 14 bits (address >> 4) and never carries out of them inside shared memory.
      const uint64_t dK = tc::sdesc_sw128(ring, 16, 1024);
      const uint64_t dV = tc::sdesc_sw128(ring, HALF_BYTES, 1024);
      // a slot's release is only sent when a later item will refill it, so every release
      // that reaches a peer is awaited by that peer's producer; it follows the issuing
      // thread's own MMAs, the ones that read the slot
      auto release = [&](int q) {
        if (q + SLOTS >= total) return;
        if (multicast)
          tc::mma_commit_mc(bar.empty + slot_of(q), all_mask);
        else
          tc::mma_commit(bar.empty + slot_of(q));
      };
      bool ok = true;
      if (qk) {
        auto issue_s = [&](int t) {  // S(t) = Q K(t)^T over d = 128 (8 steps of 16)
          const int q = pos_k(t, nt);
          if (!tc::mbar_wait(bar.full + slot_of(q), use_parity(q), abort)) return false;
          tc::tc_fence_after();
          const uint64_t b0 = dK + ((slot_of(q) * SLOT_BYTES) >> 4);
          const uint32_t dS = tmem + (uint32_t)((t % NSBUF) * 128);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = ((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4;
            tc::mma_ts(dS, tmem + Q_COL + kk * 8, b0 + off, idS, kk > 0);
          }
          tc::mma_commit(bar.s_full + t % NSBUF);
          release(q);
          return true;
        };
        ok = tc::mbar_wait(bar.q_full, 0, abort);
        for (int t = 0; ok && t < min(KLEAD, nt); ++t) ok = issue_s(t);
        // S(j+2) into the buffer of S(j) once every softmax thread has read S(j)
        for (int j = 0; ok && j + KLEAD < nt; ++j) {
          if (!tc::mbar_wait(bar.s_free + j % NSBUF, (uint32_t)((j / NSBUF) & 1), abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          ok = issue_s(j + KLEAD);
        }
      } else {
        for (int j = 0; ok && j < nt; ++j) {
          const int qv = pos_v(j, nt);
          if (!tc::mbar_wait(bar.p_full, j & 1, abort) ||
              !tc::mbar_wait(bar.full + slot_of(qv), use_parity(qv), abort)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint64_t v0 = dV + ((slot_of(qv) * SLOT_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // O += P V over 128 keys (steps of 16)
            tc::mma_ts(tmem + O_COL, tmem + P_COL + kk * 8, v0 + ((kk * 2048) >> 4), idO,
                       (j > 0) || (kk > 0));
          tc::mma_commit(bar.o_ready);
          release(qv);
        }
        if (ok) tc::mma_commit(bar.o_done);
      }
      // every MMA this thread issued completes before teardown
      uint64_t *drain = bar.drain + (qk ? 0 : 1);
      tc::mma_commit(drain);
      drain_wait(drain, 0);
    }
  } else {
    // ------------------------------------------------------------------- softmax
    const int rl = warp * 32 + lane;                // row within the M-tile = TMEM lane
    const int r = row0 + rl;                        // row within the segment
    const uint64_t mword = r < g * n ? mask[(size_t)b * N + r / g] : 0ull;
    // checked builds: a tree row's mask holds the root and the node itself, no node past n
    GT_CHECKED(r >= g * n || (((mword >> (r / g)) & 1ull) && (mword & 1ull) &&
                              (n >= 64 || (mword >> n) == 0ull)),
               err, GT_ERR_TREE);
    // keys past the request's length stay invisible whatever the word holds past node n - 1
    const uint64_t mrow = n >= 64 ? mword : (mword & ((1ull << n) - 1ull));
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + O_COL;
    const float sl2 = scale * LOG2E;  // scale > 0: the max of raw scores gives the max
    float m_used = -INFINITY, l = 0.f;  // reference max (log2 units) and sum of this row
    q_row_to_tmem(Qg, b, N, Hq, h, g, r, tmem + lane_base + Q_COL);
    asm volatile("" ::"l"(mrow));  // the mask word has arrived before the arrival below
    tc::tc_fence_before();
    tc::mbar_arrive(bar.q_full);
    bool ok = true;
    for (int j = 0; ok && j < nt; ++j) {
      const uint32_t tS = tmem + lane_base + (uint32_t)((j % NSBUF) * 128);
      // wait results are made warp-uniform: the TMEM accesses below are warp-collective
      if (!__all_sync(0xffffffffu,
                      tc::mbar_wait(bar.s_full + j % NSBUF, (uint32_t)((j / NSBUF) & 1), abort))) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(tS + c * 32, s[c]);
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      tc::mbar_arrive(bar.s_free + j % NSBUF);  // S(j) is in registers: S(j+2) may follow
      const int kb = (t0 + j) * TK;
      float alpha;
      uint32_t pk[4][16];  // P(j) as bf16 pairs, stored once the previous P is consumed
      softmax_tile(s, kb, P, mrow, sl2, j > 0, m_used, l, alpha, pk);
      // O += P(j-1) V(j-1) must have completed before O is rescaled here and before P(j)
      // overwrites P(j-1)
      if (j > 0 && !__all_sync(0xffffffffu, tc::mbar_wait(bar.o_ready, (uint32_t)((j - 1) & 1), abort))) {
        ok = false;
        break;
      }
      if (__any_sync(0xffffffffu, alpha != 1.f && j > 0)) {
        tc::tc_fence_after();
        rescale_o(tO, alpha);
      }
      const uint32_t tP = tmem + lane_base + P_COL;
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_st16(tP + c * 16, pk[c]);
      tc::tmem_wait_st();
      if (kb + TK > keys) {
        // zero V rows past the request's length (they may hold NaN) before P V reads them
        const int qv = pos_v(j, nt);
        if (!__all_sync(0xffffffffu, tc::mbar_wait(bar.full + slot_of(qv), use_parity(qv), abort))) {
          ok = false;
          break;
        }
        uint8_t *vt = base + Lay::RING + slot_of(qv) * SLOT_BYTES;
        const int first = keys - kb > 0 ? keys - kb : 0;
        for (int e = rl; e < (TK - first) * 16; e += 128) {
          const int row = first + e / 16, chunk = e % 16;  // 2 halves x 8 chunks of 16 B
          *reinterpret_cast<uint4 *>(vt + (chunk >> 3) * HALF_BYTES + row * 128 +
                                     (chunk & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        tc::fence_proxy_async_smem();
      }
      tc::tc_fence_before();
      tc::mbar_arrive(bar.p_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(bar.o_done, 0, abort));
    if (pc.w == 1)
      write_final(tO, ok, l, row0, g, n, N, Hq, h, b, O);
    else
      write_partial(base + Lay::RING, &mapO, tO, ok, l, m_used, p, row0, g * n, ws);
  }

  tc::tc_fence_before();
  __syncthreads();
  const bool aborted = *abort != 0;
  if (tid == 0 && aborted) set_err(err, GT_ERR_TIMEOUT);
  if (multicast) {
    // no CTA leaves while a peer may still multicast into it or release its slots
    tc::cluster_sync_all();
    if (aborted && tid == 0) {
      // after an abort, loads a peer issued for items this CTA never consumed may still be
      // landing: give them a millisecond (no producer of the cluster issues new ones now)
      const uint64_t t_end = tc::globaltimer() + 1000000ull;
      while (tc::globaltimer() < t_end) {
      }
    }
    __syncthreads();
  }
  if (warp == 5) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_acquire);
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
      cached.store(fn, std::memory_order_release);  // racing callers find the same pointer
    } else {
      (void)cudaGetLastError();
    }
  }
  return fn;
}

bool encode(CUtensorMap *map, const void *ptr, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides_bytes, const cuuint32_t *box,
            CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, type, rank, const_cast<void *>(ptr), dims, strides_bytes, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int cluster_of(int g, int N) { return ceil_div(g * N, 128); }
int loaders_of(int C) { return C >= 4 ? 4 : (C >= 2 ? 2 : 1); }
bool set_attributes() {
  static SmemAttr attr;
  return ensure_smem(attn_tc_kernel, (int)Smem::BYTES, attr,
                     "cudaFuncSetAttribute(attn_tc_kernel)") == GT_OK;
}

}  // namespace

bool attn_tc_supported(int g, int N) {
  // rows are placed one by one (r = node * g + head-in-group), so a node's g heads may
  // straddle two CTAs of the cluster: any g works up to four 128-row M-tiles
  return g >= 1 && N >= 1 && g * N <= 128 * MAX_CLUSTER;
}

int attn_tc_pieces(int g, int N) {
  const int C = cluster_of(g, N);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return 1;
  }
  static std::atomic<int> cache[64][MAX_CLUSTER + 1];  // zero-initialised (static)
  const int hit = cache[dev][C].load(std::memory_order_relaxed);
  if (hit > 0) return hit;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 1;
  }
  int clusters = sms / C;
  if (set_attributes()) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C * clusters);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = Smem::BYTES;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, attn_tc_kernel, &cfg) == cudaSuccess && nc > 0)
      clusters = nc < clusters ? nc : clusters;
    else
      (void)cudaGetLastError();
  }
  if (clusters < 1) clusters = 1;
  cache[dev][C].store(clusters, std::memory_order_relaxed);
  return clusters;
}

int attn_tc_launch(const void *Q, const void *K, const void *V, const uint64_t *mask,
                   const SchedArgs &sa, int B, int N, int Hq, int Hkv, int Lcap, float scale,
                   const AttnWs &ws, int pieces, void *O, int32_t *err, cudaStream_t s) {
  const int g = Hq / Hkv;
  const int C = cluster_of(g, N), L = loaders_of(C);
  CUtensorMap mK, mV;
  const cuuint64_t kdims[3] = {(cuuint64_t)ATTN_D, (cuuint64_t)Lcap, (cuuint64_t)B * Hkv};
  const cuuint64_t kstr[2] = {(cuuint64_t)ATTN_D * 2, (cuuint64_t)Lcap * ATTN_D * 2};
  const cuuint32_t kbox[3] = {64, (cuuint32_t)(TK / L), 1};
  if (!encode_fn()) {
    note_error("cuTensorMapEncodeTiled entry point", cudaErrorNotSupported);
    return GT_ERR_CUDA;
  }
  if (!encode(&mK, K, 3, kdims, kstr, kbox) || !encode(&mV, V, 3, kdims, kstr, kbox)) {
    note_error("cuTensorMapEncodeTiled(K/V)", cudaErrorInvalidValue);
    return GT_ERR_CUDA;
  }
  // the partial rows: fp32 [maxp * rows_pad][d], stored in boxes of 32 columns x 128 rows
  CUtensorMap mO;
  const cuuint64_t odims[2] = {(cuuint64_t)ATTN_D, (cuuint64_t)ws.maxp * ws.rows_pad};
  const cuuint64_t ostr[1] = {(cuuint64_t)ATTN_D * 4};
  const cuuint32_t obox[2] = {32, 128};
  if (!encode(&mO, ws.opart, 2, odims, ostr, obox, CU_TENSOR_MAP_DATA_TYPE_FLOAT32)) {
    note_error("cuTensorMapEncodeTiled(partial O)", cudaErrorInvalidValue);
    return GT_ERR_CUDA;
  }
  if (!set_attributes()) return GT_ERR_CUDA;
  // each CTA asks L2 for a slice of Q (16-byte multiples) before it computes the schedule
  const uint32_t q_bytes = (uint32_t)((size_t)B * N * Hq * ATTN_D * 2);
  const int grid = C * pieces;
  const uint32_t q_slice = max(16u, (q_bytes / grid + 15u) / 16u * 16u);
  // one cluster of C CTAs per piece; the schedule never makes more than `pieces`
  return launch_cluster(attn_tc_kernel, dim3(grid), dim3(TC_THREADS), dim3(C, 1, 1),
                        Smem::BYTES, s, (const __nv_bfloat16 *)Q, mK, mV, mO, q_slice, q_bytes,
                        mask, sa.prefix_len, sa.n_nodes, N, Hq, Hkv, scale, C, L, sa, ws,
                        (__nv_bfloat16 *)O, err);
}

}  // namespace gt
