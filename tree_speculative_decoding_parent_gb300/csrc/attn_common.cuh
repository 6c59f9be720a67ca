// Split-KV work decomposition shared by the tree-attention kernels.
//
// A "segment" is one (request b, KV head h) pair: its g*N query rows attend keys
// [0, prefix_len[b] + n_nodes[b]). Keys are cut into tiles of TK; the scheduler splits
// each segment's tiles into contiguous "pieces" of about tau tiles so that the number of
// pieces is close to the number of CTAs that fit on the GPU at once. Each piece writes a
// partial (normalised O, log-sum-exp) per query row; the combine kernel merges the pieces
// of a segment with LSE weights.
#pragma once

#include <stdint.h>

#include "gt.h"

namespace gt {

constexpr int ATTN_D = 128;        // head dimension supported by the kernels
constexpr int ATTN_MAX_N = 64;     // tree nodes per request (one mask word)
constexpr int ATTN_ROWS_PAD = 128; // partial rows are padded to a multiple of this

struct AttnWs {
  int *hdr;          // [0] number of pieces; [1] 1 if some segment's piece count is not 1
  int2 *seg;         // (first piece, piece count) per segment
  float *lse;        // [maxp][rows_pad] natural-log LSE per partial row
  float *opart;      // [maxp][rows_pad][d] normalised partial O
  int maxp, rows_pad;
};

static inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Layout of the caller's workspace; returns the bytes needed.
static inline size_t attn_ws_layout(void *base, int S, int maxp, int rows_pad, AttnWs *ws) {
  size_t off = 0;
  char *p = static_cast<char *>(base);
  const size_t o_hdr = off;
  off += align256(16 * sizeof(int));
  const size_t o_seg = off;
  off += align256((size_t)S * sizeof(int2));
  const size_t o_lse = off;
  off += align256((size_t)maxp * rows_pad * sizeof(float));
  const size_t o_opart = off;
  off += align256((size_t)maxp * rows_pad * ATTN_D * sizeof(float));
  if (ws) {
    ws->hdr = reinterpret_cast<int *>(p + o_hdr);
    ws->seg = reinterpret_cast<int2 *>(p + o_seg);
    ws->lse = reinterpret_cast<float *>(p + o_lse);
    ws->opart = reinterpret_cast<float *>(p + o_opart);
    ws->maxp = maxp;
    ws->rows_pad = rows_pad;
  }
  return off;
}

// Arguments of the split-KV schedule (all device pointers are per-request arrays).
struct SchedArgs {
  const int32_t *prefix_len, *n_nodes;
  int B, Hkv, N, Lcap, TK, G;
};

#ifdef __CUDACC__
// The split-KV schedule, computed redundantly by every CTA of an attention launch so that
// no separate scheduling kernel is needed. Segment s = (b, h) has
// tiles_s = ceil((P_b + n_b) / TK) tiles (0 for an invalid request); with a piece length
// tau it gets cnt_s = ceil(tiles_s / tau) pieces of near-equal tile counts, numbered
// consecutively over s. tau starts at ceil(sum_s tiles_s / G); when G exceeds the number
// of non-empty segments, tau is raised to the smallest value whose pieces all fit in one
// wave of G (sum_s cnt_s <= G), so that no piece waits for a second wave. Returns piece p
// as (segment, tile_begin,
// tile_end, piece count of the segment), or segment -1 when p is past the last piece, and
// (when np_out is given) the node count and prefix length of the piece's request. The CTA
// at blockIdx (0,0) also publishes (first piece, count) of every segment, the piece total
// and whether any segment has a piece count other than 1 into `ws`, and reports invalid
// requests. Every thread of the CTA must call it (it synchronises).
__device__ __forceinline__ int4 schedule_piece(const SchedArgs &a, int p, AttnWs ws,
                                               int32_t *err, int2 *np_out = nullptr) {
  constexpr int CH = 4;  // segments per thread kept in registers; more are recomputed
  __shared__ long long s_red[2][32];
  __shared__ int s_scan[32];
  __shared__ int4 s_piece;
  const int S = a.B * a.Hkv, tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nw = (nt + 31) >> 5;
  const bool publisher = blockIdx.x == 0 && blockIdx.y == 0;
  const int chunk = (S + nt - 1) / nt;
  const int c0 = min(S, tid * chunk), c1 = min(S, c0 + chunk);
  auto tiles_of = [&](int s) {
    const int b = s / a.Hkv;
    const int n = a.n_nodes[b], P = a.prefix_len[b];
    const bool ok = n >= 1 && n <= a.N && P >= 0 && (long long)P + n <= (long long)a.Lcap;
    if (!ok && publisher && (s % a.Hkv) == 0 && err) atomicCAS(err, 0, GT_ERR_RANGE);
    return ok ? (P + n + a.TK - 1) / a.TK : 0;
  };
  __shared__ int2 s_np;  // (n, P) of the piece's request
  if (S <= 32) {
    // up to 32 segments: lane l of warp 0 holds segment l. The same tau and pieces as the
    // paths below, in the least code: this runs once per CTA, its instructions fetched cold
    if (warp == 0) {
      int t = 0, n = 0, P = 0;
      if (lane < S) {
        const int b = lane / a.Hkv;
        n = a.n_nodes[b];
        P = a.prefix_len[b];
        const bool ok = n >= 1 && n <= a.N && P >= 0 && (long long)P + n <= (long long)a.Lcap;
        if (!ok && publisher && (lane % a.Hkv) == 0 && err) atomicCAS(err, 0, GT_ERR_RANGE);
        t = ok ? (P + n + a.TK - 1) / a.TK : 0;
      }
      const int T = (int)__reduce_add_sync(0xffffffffu, (unsigned)t);
      const int Sn = (int)__reduce_add_sync(0xffffffffu, (unsigned)(t > 0));
      int tau = max(1, (T + a.G - 1) / a.G);
      if (Sn > 0 && a.G > Sn) {
        int lo = tau, hi = max(tau, (T + (a.G - Sn) - 1) / (a.G - Sn));
        while (lo < hi) {
          const int mid = lo + (hi - lo) / 2;
          if ((int)__reduce_add_sync(0xffffffffu, (unsigned)((t + mid - 1) / mid)) <= a.G)
            hi = mid;
          else
            lo = mid + 1;
        }
        tau = lo;
      }
      const int cnt = (t + tau - 1) / tau;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int off = incl - cnt;
      if (lane < S) {
        if (publisher) ws.seg[lane] = make_int2(off, cnt);
        if (p >= off && p < off + cnt) {
          // piece j: tiles [ceil(t j / cnt), ceil(t (j+1) / cnt)), with
          // ceil(t j / cnt) = (t / cnt) j + ceil((t % cnt) j / cnt) in 32 bits; the longer
          // pieces come first, so the last one, which holds the masked tail tile, is short
          const int j = p - off, q = t / cnt, r = t - q * cnt;
          s_piece = make_int4(lane, q * j + (r * j + cnt - 1) / cnt,
                              q * (j + 1) + (r * (j + 1) + cnt - 1) / cnt, cnt);
          s_np = make_int2(n, P);
        }
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      const bool multi = __any_sync(0xffffffffu, lane < S && cnt != 1);
      if (lane == 0) {
        if (publisher) {
          ws.hdr[0] = total;
          ws.hdr[1] = multi ? 1 : 0;
        }
        if (p >= total) s_piece = make_int4(-1, 0, 0, 0);
      }
    }
    __syncthreads();
    if (np_out) *np_out = s_np;
    return s_piece;
  }
  if (S <= 32 * CH) {
    // few segments: warp 0 computes the whole schedule with 32-bit shuffles and reductions
    // (lane l holds segments l, l + 32, ...), the same tau and pieces as the block version
    // below, and the CTA meets it at one barrier
    if (warp == 0) {
      if (lane == 0) s_piece = make_int4(-1, 0, 0, 0);
      __syncwarp();
      int wt[CH], wn[CH], wP[CH], tsum = 0, nsum = 0;
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int s = lane + 32 * i;
        wt[i] = wn[i] = wP[i] = 0;
        if (s < S) {
          const int b = s / a.Hkv;
          const int n = a.n_nodes[b], P = a.prefix_len[b];
          const bool ok = n >= 1 && n <= a.N && P >= 0 && (long long)P + n <= (long long)a.Lcap;
          if (!ok && publisher && (s % a.Hkv) == 0 && err) atomicCAS(err, 0, GT_ERR_RANGE);
          wt[i] = ok ? (P + n + a.TK - 1) / a.TK : 0;
          wn[i] = n;
          wP[i] = P;
        }
        tsum += wt[i];
        nsum += wt[i] > 0;
      }
      const int T = (int)__reduce_add_sync(0xffffffffu, (unsigned)tsum);
      const int Sn = (int)__reduce_add_sync(0xffffffffu, (unsigned)nsum);
      int tau = max(1, (T + a.G - 1) / a.G);
      if (Sn > 0 && a.G > Sn) {
        int lo = tau, hi = max(tau, (T + (a.G - Sn) - 1) / (a.G - Sn));
        while (lo < hi) {
          const int mid = lo + (hi - lo) / 2;
          int c = 0;
#pragma unroll
          for (int i = 0; i < CH; ++i) c += (wt[i] + mid - 1) / mid;
          if ((int)__reduce_add_sync(0xffffffffu, (unsigned)c) <= a.G)
            hi = mid;
          else
            lo = mid + 1;
        }
        tau = lo;
      }
      // Piece order. With at most 32 requests, requests are taken by decreasing piece
      // length (ties: lower index), each request's KV heads in order: a launch of more
      // pieces than one wave holds then starts its longest pieces first, and the shorter
      // ones fill in behind them (largest-first list scheduling). Lane b handles request b:
      // its pieces start after those of every request whose key is larger.
      const bool by_length = a.B <= 32;
      int r_off = 0, r_cnt = 0;
      if (by_length) {
        int tb = 0;
        if (lane < a.B) {
          const int n = a.n_nodes[lane], P = a.prefix_len[lane];
          const bool ok = n >= 1 && n <= a.N && P >= 0 && (long long)P + n <= (long long)a.Lcap;
          tb = ok ? (P + n + a.TK - 1) / a.TK : 0;
        }
        r_cnt = (tb + tau - 1) / tau;
        const uint32_t len = r_cnt > 0 ? (uint32_t)((tb + r_cnt - 1) / r_cnt) : 0u;
        const uint32_t key = lane < a.B ? ((len << 5) | (uint32_t)(31 - lane)) : 0u;
        const int np = lane < a.B ? r_cnt * a.Hkv : 0;
        for (int c = 0; c < 32; ++c) {
          const uint32_t kc = __shfl_sync(0xffffffffu, key, c);
          const int nc = __shfl_sync(0xffffffffu, np, c);
          if (kc > key) r_off += nc;
        }
      }
      // pieces in segment order (segments lane + 32 i for i = 0, 1, ...) or by length
      int base = 0;
      bool multi = false;
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int s = lane + 32 * i;
        const int cnt = (wt[i] + tau - 1) / tau;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        int off = base + incl - cnt;
        if (by_length) {  // request b = s / Hkv: its offset, then h pieces of cnt each
          const int b = min(s / a.Hkv, 31), h = s - (s / a.Hkv) * a.Hkv;
          off = __shfl_sync(0xffffffffu, r_off, b) + h * cnt;
        }
        if (s < S) {
          if (publisher) ws.seg[s] = make_int2(off, cnt);
          multi = multi || cnt != 1;
          if (p >= off && p < off + cnt) {
            // tiles [ceil(t j / cnt), ceil(t (j+1) / cnt)), as above
            const int j = p - off, t = wt[i], q = t / cnt, r = t - q * cnt;
            s_piece = make_int4(s, q * j + (r * j + cnt - 1) / cnt,
                                q * (j + 1) + (r * (j + 1) + cnt - 1) / cnt, cnt);
            s_np = make_int2(wn[i], wP[i]);
          }
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      multi = __any_sync(0xffffffffu, multi);
      if (publisher && lane == 0) {
        ws.hdr[0] = base;
        ws.hdr[1] = multi ? 1 : 0;
      }
    }
    __syncthreads();
    if (np_out) *np_out = s_np;
    return s_piece;
  }
  int tl[CH];  // tiles of this thread's first CH segments
#pragma unroll
  for (int i = 0; i < CH; ++i) tl[i] = c0 + i < c1 ? tiles_of(c0 + i) : 0;
  // one barrier per sum: the scratch alternates, and the barrier of the next sum orders
  // every read of this one before the one after it writes the same half
  int sum_no = 0;
  auto block_sum = [&](long long v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    long long *red = s_red[sum_no++ & 1];
    if (lane == 0) red[warp] = v;
    __syncthreads();
    long long t = 0;
    for (int w = 0; w < nw; ++w) t += red[w];
    return t;
  };
  auto pieces_of = [&](int tau) {  // sum over this thread's segments of ceil(tiles / tau)
    long long c = 0;
#pragma unroll
    for (int i = 0; i < CH; ++i) c += (tl[i] + tau - 1) / tau;
    for (int s = c0 + CH; s < c1; ++s) c += (tiles_of(s) + tau - 1) / tau;
    return c;
  };
  if (tid == 0) s_piece = make_int4(-1, 0, 0, 0);
  // total tiles and (from bit 44 up) the number of non-empty segments in one sum
  long long local = 0;
#pragma unroll
  for (int i = 0; i < CH; ++i) local += tl[i] + ((long long)(tl[i] > 0) << 44);
  for (int s = c0 + CH; s < c1; ++s) {
    const int t = tiles_of(s);
    local += t + ((long long)(t > 0) << 44);
  }
  const long long both = block_sum(local);
  const long long T = both & ((1ll << 44) - 1);
  const long long Sn = both >> 44;
  int tau = (int)max(1ll, (T + a.G - 1) / a.G);
  if (Sn > 0 && a.G > Sn) {
    // pieces(tau) does not grow with tau, and tau = ceil(T / (G - Sn)) always fits:
    // sum_s ceil(t_s / tau) < T / tau + Sn <= G
    int lo = tau, hi = (int)max((long long)tau, (T + (a.G - Sn) - 1) / (a.G - Sn));
    while (lo < hi) {
      const int mid = lo + (hi - lo) / 2;
      if (block_sum(pieces_of(mid)) <= a.G)
        hi = mid;
      else
        lo = mid + 1;
    }
    tau = lo;
  }
  const int lp = (int)pieces_of(tau);
  int incl = lp;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int off = incl - lp, total = 0;
  for (int w = 0; w < nw; ++w) {
    off += (w < warp) ? s_scan[w] : 0;
    total += s_scan[w];
  }
  bool multi = false;
  for (int s = c0; s < c1; ++s) {
    int t = 0;
#pragma unroll
    for (int i = 0; i < CH; ++i)
      if (s == c0 + i) t = tl[i];
    if (s >= c0 + CH) t = tiles_of(s);
    const int cnt = (t + tau - 1) / tau;
    if (publisher) ws.seg[s] = make_int2(off, cnt);
    multi = multi || cnt != 1;
    if (p >= off && p < off + cnt) {
      const int j = p - off;
      s_piece = make_int4(s, (int)(((long long)t * j + cnt - 1) / cnt),
                          (int)(((long long)t * (j + 1) + cnt - 1) / cnt), cnt);
      const int b = s / a.Hkv;
      s_np = make_int2(a.n_nodes[b], a.prefix_len[b]);
    }
    off += cnt;
  }
  const int any_multi = __syncthreads_or(multi);
  if (publisher && tid == 0) {
    ws.hdr[0] = total;
    ws.hdr[1] = any_multi ? 1 : 0;
  }
  if (np_out) *np_out = s_np;
  return s_piece;
}
#endif

}  // namespace gt
