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

namespace gt {

constexpr int ATTN_D = 128;        // head dimension supported by the kernels
constexpr int ATTN_MAX_N = 64;     // tree nodes per request (one mask word)
constexpr int ATTN_ROWS_PAD = 128; // partial rows are padded to a multiple of this

struct AttnWs {
  int *hdr;          // [0] number of pieces
  int4 *pieces;      // (segment, tile_begin, tile_end, 0)
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
  const size_t o_pieces = off;
  off += align256((size_t)maxp * sizeof(int4));
  const size_t o_seg = off;
  off += align256((size_t)S * sizeof(int2));
  const size_t o_lse = off;
  off += align256((size_t)maxp * rows_pad * sizeof(float));
  const size_t o_opart = off;
  off += align256((size_t)maxp * rows_pad * ATTN_D * sizeof(float));
  if (ws) {
    ws->hdr = reinterpret_cast<int *>(p + o_hdr);
    ws->pieces = reinterpret_cast<int4 *>(p + o_pieces);
    ws->seg = reinterpret_cast<int2 *>(p + o_seg);
    ws->lse = reinterpret_cast<float *>(p + o_lse);
    ws->opart = reinterpret_cast<float *>(p + o_opart);
    ws->maxp = maxp;
    ws->rows_pad = rows_pad;
  }
  return off;
}

}  // namespace gt
