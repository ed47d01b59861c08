// decode_tiles.cuh -- pieces shared by the two tcgen05 decode kernels
// (skinny.cu: weights as the MMA's N operand from shared memory;
// decode_fp8.cu: e4m3 weights widened into tensor memory as its A operand):
// the e4m3 -> bf16 widening, and the tiling of a CTA's outputs into pieces
// of consecutive features at 16-row slots.  The tiling functions take any
// parameter struct with the fields they read (tile_cap, act, tp, fo,
// kb_total, feat_total, cs).  The tiling is host-callable as well
// (TILE_FN), so a host program can check it over whole grids.
#pragma once

#include <cstdint>

#include "tpla.h"

namespace tpla {
namespace decode {

constexpr int SK_GRAIN = 16;                // features per balance unit (column side)
constexpr int SK_MAX_BOXES = 31;            // weight boxes per stage (one per producer lane)
constexpr int SK_BN = 256;                  // outputs per row-side tile
constexpr int64_t G = TP_GATE_UP_GROUP;
static_assert(2 * G == SK_BN, "a gate/up group's rows fill one 256-row tile");

#define TILE_FN __host__ __device__ __forceinline__

TILE_FN int64_t imin(int64_t a, int64_t b) { return a < b ? a : b; }

// Byte permute (PTX prmt, default mode): result byte i is byte (sel_i & 7)
// of {a, 0}, or that byte's sign bit replicated when sel_i & 8.
__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(a), "r"(sel));
  return r;
}

// Two e4m3 codes to two bf16 values, exactly.  Each 16-bit lane of w holds a
// code in its low byte and the code's sign replicated through its high byte:
// s s s s s s s s | s e e e e m m m.  Shifted left by 4 (the low lane's top
// nibble spills into bits 0-3 of the high lane, which the mask clears) and
// masked, a lane keeps the sign at bit 15 and the code's exponent and
// mantissa at bits 7..10 and 4..6: read as bf16 that is the e4m3 value times
// 2^-120 (bf16 exponent bias 127 against e4m3's 7; a subnormal code gives the
// matching subnormal bf16).  One bf16x2 multiply by 2^120 (0x7B80) restores
// the value; no step rounds.
__device__ __forceinline__ uint32_t e4m3_lanes_to_bf16x2(uint32_t w) {
  const uint32_t bits = (w << 4) & 0x87F087F0u;
  uint32_t out;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out) : "r"(bits), "r"(0x7B807B80u));
  return out;
}

// Four e4m3 codes (code k in byte k of q) to four bf16 values: codes 0, 1 in
// lo (low half first), codes 2, 3 in hi.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t q, uint32_t& lo, uint32_t& hi) {
  lo = e4m3_lanes_to_bf16x2(prmt_b32(q, 0x9180u));  // bytes: q0, sign(q0), q1, sign(q1)
  hi = e4m3_lanes_to_bf16x2(prmt_b32(q, 0xB3A2u));  // bytes: q2, sign(q2), q3, sign(q3)
}

constexpr int SK_MAX_PIECES = 8;

// One B tile's worth of work: up to SK_MAX_PIECES pieces of consecutive
// output features, each at a 16-row slot of the tile, and the k-blocks of its
// K loop.
struct Piece {
  int shard;    // column: shard of the piece; row: unused (per k-block)
  int64_t loc;  // column: first shard-local feature; row: first output
  int c;        // features (outputs) in the piece
  int slot;     // first row of the piece in the B tile (a multiple of 16)
};
struct Tile {
  int n;        // pieces
  int rows;     // slot rows used (a multiple of 16)
  int boxes;    // weight TMA boxes per stage
  int kb0, kb1; // k-blocks [kb0, kb1) of the tile's K loop
  Piece pc[SK_MAX_PIECES];
};

// Weight boxes of a piece of c rows: whole 64-row boxes, then 16-row boxes.
TILE_FN int piece_boxes(int c) { return c / 64 + ((c % 64) + 15) / 16; }

// Box `want` (0-based) of a tile, in the order pieces, then gate/up halves,
// then rows: which piece and half, its first row within the piece, and its
// height.  Returns false when the tile has fewer boxes.
TILE_FN bool tile_box(const Tile& t, bool swiglu, int want, int& piece,
                                         int& half, int& r, int& h) {
  int b = 0;
  for (int i = 0; i < t.n; ++i)
    for (int hf = 0; hf < (swiglu ? 2 : 1); ++hf) {
      const int c = t.pc[i].c;
      for (int rr = 0; rr < c; ++b) {
        const int hh = (rr + 64 <= c) ? 64 : 16;
        if (b == want) {
          piece = i;
          half = hf;
          r = rr;
          h = hh;
          return true;
        }
        rr += hh;
      }
    }
  return false;
}

// Column side: the tile starting at global feature f of a range ending at f1;
// advances f past the features it takes.
template <class P>
TILE_FN Tile column_tile(const P& p, int64_t& f, int64_t f1) {
  const bool swiglu = p.act == TP_ACT_SWIGLU;
  const int cap = p.tile_cap;  // slot rows per tile (features for SwiGLU)
  Tile t;
  t.n = 0;
  t.rows = 0;
  t.kb0 = 0;
  t.kb1 = p.kb_total;
  t.boxes = 0;
  while (f < f1 && t.n < SK_MAX_PIECES && t.rows < cap) {
    int sh = 0;
    while (sh + 1 < p.tp && p.fo[sh + 1] <= f) ++sh;
    const int64_t loc = f - p.fo[sh];
    int64_t lim = imin(f1 - f, p.fo[sh + 1] - f);
    if (swiglu) lim = imin(lim, G - loc % G);
    const int c = (int)imin(lim, cap - t.rows);
    const int nb = piece_boxes(c) * (swiglu ? 2 : 1);
    if (t.n > 0 && t.boxes + nb > SK_MAX_BOXES) break;
    t.pc[t.n].shard = (int)sh;
    t.pc[t.n].loc = loc;
    t.pc[t.n].c = c;
    t.pc[t.n].slot = t.rows;
    ++t.n;
    t.boxes += nb;
    t.rows += (c + 15) / 16 * 16;
    f += c;
  }
  return t;
}

// Column side: CTA b of grid's feature range [f0, f1), balanced in units of
// SK_GRAIN features.
template <class P>
TILE_FN void column_range_of(const P& p, int64_t b, int64_t grid, int64_t& f0, int64_t& f1) {
  const int64_t units = (p.feat_total + SK_GRAIN - 1) / SK_GRAIN;
  const int64_t u0 = b * units / grid;
  const int64_t u1 = (b + 1) * units / grid;
  f0 = imin(u0 * SK_GRAIN, p.feat_total);
  f1 = imin(u1 * SK_GRAIN, p.feat_total);
}
template <class P>
__device__ __forceinline__ void column_range(const P& p, int64_t& f0, int64_t& f1) {
  column_range_of(p, (int64_t)blockIdx.x, (int64_t)gridDim.x, f0, f1);
}

// Row side: how the outputs are cut into tiles and each tile's K loop over a
// cluster.  Tiles of SK_BN = 256 outputs: narrower tiles measured slower per
// byte -- 128-wide tiles on the same 128 CTAs took 121 us where 256-wide
// took 84 us for the 8192 x 28672 down projection, with or without the MMAs,
// so it is the smaller stages that cost.  Clusters of cs CTAs split each
// tile's K loop: cs is a multiple of cs_unit (FP8 kernels: tp, so that each
// CTA's k-range lies inside one shard), at most cs_max, each CTA keeps at
// least one k-block (kb_unit k-blocks per cs_unit CTAs), and the tiles'
// clusters fit on the device at once: resident[cs] is how many clusters of
// cs CTAs the kernel can hold (0: not known; then sms / cs).  Clusters stay
// inside a GPC, so that is below sms / cs for cs > 2 (33 clusters of 4 on
// 148 SMs).  The largest cs that fits wins; when none fits, cs_unit.  The
// bf16 decode kernel's column side uses the same choice for its K-split
// tiles (bn features each).
struct RowTiling {
  int bn, cs;
  int64_t tiles;
};
inline RowTiling choose_row_tiling(int64_t n_out, int64_t kb_total, int64_t kb_unit, int sms,
                                   int cs_max, int cs_unit, const int* resident,
                                   int bn = SK_BN) {
  (void)kb_total;
  const int64_t tiles = (n_out + bn - 1) / bn;
  RowTiling best{bn, cs_unit, tiles};
  for (int cs = cs_unit; cs <= cs_max && cs / cs_unit <= kb_unit; cs += cs_unit) {
    int64_t fit = resident ? resident[cs] : 0;
    if (fit <= 0) fit = sms / cs;
    if (tiles <= fit) best.cs = cs;
  }
  return best;
}

// Column side with the K loop split over clusters (bf16 decode kernel, when
// the feature walk would leave each CTA too few weight rows to keep the
// tensor core's fixed cost per MMA hidden): cluster `block / cs` owns the
// features [tile * tile_cap, (tile + 1) * tile_cap) and its CTA of rank r
// the k-blocks [r * kb_total / cs, (r + 1) * kb_total / cs) of each tile that
// covers them.
template <class P>
TILE_FN void column_split_range_of(const P& p, int64_t block, int64_t& f0, int64_t& f1) {
  const int64_t tile = block / p.cs;
  f0 = imin(tile * p.tile_cap, p.feat_total);
  f1 = imin(f0 + p.tile_cap, p.feat_total);
}
template <class P>
TILE_FN void split_kb_range(const P& p, int rank, int& kb0, int& kb1) {
  kb0 = (int)((int64_t)rank * p.kb_total / p.cs);
  kb1 = (int)((int64_t)(rank + 1) * p.kb_total / p.cs);
}

// Row side: the one tile of this CTA -- its cluster's tile_cap outputs and
// its rank's share of the k-blocks.
template <class P>
TILE_FN Tile row_tile_of(const P& p, int64_t block, int rank) {
  Tile t;
  const int64_t tile = block / p.cs;
  t.n = 1;
  t.pc[0].shard = 0;
  t.pc[0].loc = tile * p.tile_cap;
  t.pc[0].c = (int)imin(p.tile_cap, p.feat_total - t.pc[0].loc);
  t.pc[0].slot = 0;
  t.rows = (t.pc[0].c + 15) / 16 * 16;
  t.boxes = piece_boxes(t.pc[0].c);
  t.kb0 = (int)((int64_t)rank * p.kb_total / p.cs);
  t.kb1 = (int)((int64_t)(rank + 1) * p.kb_total / p.cs);
  return t;
}
template <class P>
__device__ __forceinline__ Tile row_tile(const P& p, int rank) {
  return row_tile_of(p, (int64_t)blockIdx.x, rank);
}

// The e4m3 decode kernel's column side walks each tile's K loop from the
// CTA's own starting k-block, rotating through the rest, so that the CTAs do
// not all read the same k-offsets of their weight rows (rows a power-of-two
// 8 KB apart) at once: its 8-token column launch went from 93.8-95.8 to
// 90.8-91.1 us.  The rotation depends on the CTA index only, and a feature
// belongs to the same CTA for every tp, so the column side stays
// bit-identical to tp = 1.  Row sides (rows 7 KB apart per shard) measured
// 2 us slower rotated, and the bf16 decode kernel (rows 16 KB apart) no
// consistent change; both keep the plain order.
__device__ __forceinline__ int kb_rotation(int nkb, bool row) {
  return (nkb > 0 && !row) ? (int)(((unsigned)blockIdx.x * 37u) % (unsigned)nkb) : 0;
}
// k-block of iteration i (0 <= i < nkb) of a K loop [kb0, kb0 + nkb) rotated
// by rot; kb0 + nkb (past the end) for i >= nkb.
__device__ __forceinline__ int kb_at(int kb0, int nkb, int rot, int i) {
  if (i >= nkb) return kb0 + nkb;
  int j = rot + i;
  if (j >= nkb) j -= nkb;
  return kb0 + j;
}

// Loop over this CTA's tiles: the column side walks its feature range, the
// row side has one tile.  Inside the body, tile_is_last tells whether tl is
// the CTA's last tile.
#define SK_FOR_EACH_TILE(tl, ...)                                     \
  do {                                                                \
    if (p.row) {                                                      \
      const Tile tl = row_tile(p, rank);                              \
      const bool tile_is_last = true;                                 \
      (void)tile_is_last;                                             \
      __VA_ARGS__                                                     \
    } else {                                                          \
      for (int64_t f_ = f0; f_ < f1;) {                               \
        const Tile tl = column_tile(p, f_, f1);                       \
        const bool tile_is_last = f_ >= f1;                           \
        (void)tile_is_last;                                           \
        __VA_ARGS__                                                   \
      }                                                               \
    }                                                                 \
  } while (0)

}  // namespace decode
}  // namespace tpla
