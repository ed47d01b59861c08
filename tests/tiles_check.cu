// tiles_check.cu -- host program (no kernel launch) that runs the decode
// kernels' tiling (csrc/decode_tiles.cuh) over whole grids, the way the
// launchers configure it, and checks the index arithmetic the kernels rely on:
//   column side, every CTA of the grid:
//     * the CTAs' feature ranges partition [0, F) in SK_GRAIN units;
//     * a CTA's tiles cover its range in order; each piece lies inside one
//       shard and, for SwiGLU, inside one gate/up group;
//     * slots are 16-row aligned and packed; a tile's slot rows never exceed
//       the tile cap the launcher sized its stages for;
//     * the boxes tile_box enumerates are at most SK_MAX_BOXES, cover each
//       piece (and half) exactly in 64- and 16-row boxes, and land inside the
//       stage's rows; their first weight row lies inside the shard buffer;
//   column side with K split over clusters (bf16 decode kernel, when the
//   feature walk leaves fewer than 128 weight rows a CTA), every CTA:
//     * the split is chosen from the total feature count, K and the SM count
//       only (so tp = 1 takes the same one), cs >= 2 clusters all resident,
//       at least 32 k-blocks per CTA;
//     * the clusters' feature ranges partition [0, F) in tiles of 256
//       features (SwiGLU 128); ranks partition each tile's k-blocks;
//     * each CTA's tiles cover its range with the checks above, and every
//       feature's partial-sum slot (SwiGLU: gate and up) lies inside the
//       260-float row of the reduction buffer;
//   row side, every (tile, rank) of the clusters:
//     * the cluster size the launchers choose for 256-wide tiles is in range
//       (a multiple of the cluster unit, at most 8, at least one k-block per
//       CTA) and the largest whose clusters all fit on the device at once,
//       for the cluster counts measured on a B300;
//     * tiles cover [0, N) once; ranks partition the k-blocks; with tp x j
//       CTAs per cluster (the FP8 kernels) each rank's k-range lies in one
//       shard.
// Prints "ok" and exits 0, or prints the first violation and exits 1.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "decode_tiles.cuh"

using namespace tpla::decode;

struct Params {
  int tile_cap = 0, act = TP_ACT_NONE, tp = 1, cs = 1, kb_total = 1;
  int64_t feat_total = 0;
  int64_t fo[TP_MAX_TP + 1] = {};
};

static int fails = 0;
#define CHECK(cond, ...)                              \
  do {                                                \
    if (!(cond)) {                                    \
      if (fails++ == 0) {                             \
        std::printf("FAIL %s:%d: ", __FILE__, __LINE__); \
        std::printf(__VA_ARGS__);                     \
        std::printf("\n");                            \
      }                                               \
      return;                                         \
    }                                                 \
  } while (0)

static int64_t gate_up_rows(int64_t ns) { return 2 * G * ((ns + G - 1) / G); }

// A CTA's walk over its features [f0, f1): the tiles column_tile cuts.
static void walk_tiles(const Params& p, const std::vector<int64_t>& widths, bool swiglu,
                       int tile_rows, int64_t f0, int64_t f1) {
  for (int64_t f = f0; f < f1;) {
    const int64_t start = f;
    const Tile t = column_tile(p, f, f1);
    CHECK(t.n >= 1 && f > start, "no progress at feature %lld", (long long)start);
    CHECK(t.rows <= p.tile_cap, "tile rows %d > cap %d", t.rows, p.tile_cap);
    CHECK(t.boxes <= SK_MAX_BOXES, "%d boxes", t.boxes);
    int64_t g = start;
    int slot = 0, boxes = 0;
    for (int i = 0; i < t.n; ++i) {
      const Piece& pc = t.pc[i];
      CHECK(pc.slot == slot && pc.slot % 16 == 0, "piece %d slot %d, expected %d", i, pc.slot,
            slot);
      CHECK(pc.c >= 1, "empty piece");
      CHECK(p.fo[pc.shard] <= g && g < p.fo[pc.shard + 1], "piece %d in the wrong shard", i);
      CHECK(pc.loc == g - p.fo[pc.shard], "piece %d loc", i);
      CHECK(pc.loc + pc.c <= widths[pc.shard], "piece %d crosses its shard's end", i);
      if (swiglu) CHECK(pc.loc / G == (pc.loc + pc.c - 1) / G, "piece %d crosses a group", i);
      const int64_t buf_rows = swiglu ? gate_up_rows(widths[pc.shard]) : widths[pc.shard];
      // this piece's boxes, in tile_box order
      for (int half = 0; half < (swiglu ? 2 : 1); ++half) {
        int covered = 0;
        while (covered < pc.c) {
          int pi, hf, r, h;
          CHECK(tile_box(t, swiglu, boxes, pi, hf, r, h), "box %d missing", boxes);
          CHECK(pi == i && hf == half && r == covered, "box %d is (%d,%d,%d)", boxes, pi, hf, r);
          CHECK(h == 64 || h == 16, "box height %d", h);
          CHECK(pc.slot + half * t.rows + r + h <= tile_rows, "box %d leaves the stage", boxes);
          const int64_t wrow =
              (swiglu ? (pc.loc / G) * 2 * G + pc.loc % G + half * G : pc.loc) + r;
          CHECK(wrow < buf_rows, "box %d starts at weight row %lld of %lld", boxes,
                (long long)wrow, (long long)buf_rows);
          covered += h;
          ++boxes;
        }
        CHECK(covered == (pc.c + 15) / 16 * 16 || (covered >= pc.c && covered - pc.c < 16),
              "piece %d half %d covered %d rows for %d", i, half, covered, pc.c);
      }
      g += pc.c;
      slot += (pc.c + 15) / 16 * 16;
    }
    int pi, hf, r, h;
    CHECK(!tile_box(t, swiglu, boxes, pi, hf, r, h) && boxes == t.boxes, "box count %d vs %d",
          boxes, t.boxes);
    CHECK(g == f && slot == t.rows, "tile covers [%lld, %lld), advanced to %lld",
          (long long)start, (long long)g, (long long)f);
  }
}

// widths: per-shard features; swiglu; cap_features: the launcher's cap.
static void check_column(const std::vector<int64_t>& widths, bool swiglu, int64_t cap_limit,
                         int sms) {
  Params p;
  p.tp = (int)widths.size();
  p.act = swiglu ? TP_ACT_SWIGLU : TP_ACT_GELU_ERF;
  p.fo[0] = 0;
  for (int i = 0; i < p.tp; ++i) p.fo[i + 1] = p.fo[i] + widths[i];
  p.feat_total = p.fo[p.tp];
  const int64_t units = (p.feat_total + SK_GRAIN - 1) / SK_GRAIN;
  const int64_t grid = units < sms ? units : sms;
  const int64_t max_range = (units + grid - 1) / grid * SK_GRAIN;
  p.tile_cap = (int)(cap_limit < max_range ? cap_limit : max_range);
  const int tile_rows = swiglu ? 2 * p.tile_cap : p.tile_cap;  // stage rows
  int64_t expect = 0;
  for (int64_t b = 0; b < grid; ++b) {
    int64_t f0, f1;
    column_range_of(p, b, grid, f0, f1);
    CHECK(f0 == expect, "CTA %lld starts at %lld, expected %lld", (long long)b, (long long)f0,
          (long long)expect);
    CHECK(f0 % SK_GRAIN == 0 && f1 >= f0, "CTA %lld range [%lld, %lld)", (long long)b,
          (long long)f0, (long long)f1);
    expect = f1;
    walk_tiles(p, widths, swiglu, tile_rows, f0, f1);
    if (fails) return;
  }
  CHECK(expect == p.feat_total, "ranges end at %lld of %lld", (long long)expect,
        (long long)p.feat_total);
}

// n_out outputs in tiles of bn, tp shards of kbs k-blocks each, clusters of
// cs CTAs.
static void check_row(int64_t n_out, int tp, int kbs, int bn, int cs, bool one_shard_per_rank) {
  Params p;
  p.tp = tp;
  p.cs = cs;
  p.tile_cap = bn;
  p.feat_total = n_out;
  p.kb_total = kbs * tp;
  const int64_t tiles = (n_out + bn - 1) / bn;
  int64_t covered = 0;
  for (int64_t tile = 0; tile < tiles; ++tile) {
    int next_kb = 0;
    for (int rank = 0; rank < cs; ++rank) {
      const Tile t = row_tile_of(p, tile * cs + rank, rank);
      CHECK(t.n == 1 && t.pc[0].loc == tile * bn, "tile %lld loc", (long long)tile);
      CHECK(t.pc[0].c >= 1 && t.pc[0].c <= bn && t.rows <= bn, "tile %lld width",
            (long long)tile);
      CHECK(t.boxes <= SK_MAX_BOXES, "row tile boxes %d", t.boxes);
      CHECK(t.kb0 == next_kb && t.kb1 > t.kb0, "rank %d k-range [%d, %d)", rank, t.kb0, t.kb1);
      next_kb = t.kb1;
      if (one_shard_per_rank)
        CHECK(t.kb0 / kbs == (t.kb1 - 1) / kbs, "rank %d k-range [%d, %d) crosses a shard", rank,
              t.kb0, t.kb1);
      if (rank == 0) covered += t.pc[0].c;
    }
    CHECK(next_kb == p.kb_total, "ranks end at k-block %d of %d", next_kb, p.kb_total);
  }
  CHECK(covered == n_out, "tiles cover %lld of %lld outputs", (long long)covered,
        (long long)n_out);
}

// Clusters of each size (1 .. 8 CTAs, one CTA per SM) that fit on a B300's
// 148 SMs at once, as cudaOccupancyMaxActiveClusters reported them: clusters
// stay inside a GPC, so sizes above 2 lose SMs to packing.
static const int kResident[9] = {0, 148, 74, 45, 33, 26, 22, 15, 15};

// Column side with the K loop split over clusters, as the bf16 decode
// kernel's launcher sets it up: returns false when the launcher would keep
// the feature walk (cs = 1 or 128 rows a CTA or more).
static bool check_column_split(const std::vector<int64_t>& widths, bool swiglu, int kb_total,
                               int sms, RowTiling* out) {
  Params p;
  p.tp = (int)widths.size();
  p.act = swiglu ? TP_ACT_SWIGLU : TP_ACT_GELU_ERF;
  p.fo[0] = 0;
  for (int i = 0; i < p.tp; ++i) p.fo[i + 1] = p.fo[i] + widths[i];
  p.feat_total = p.fo[p.tp];
  p.kb_total = kb_total;
  const int64_t units = (p.feat_total + SK_GRAIN - 1) / SK_GRAIN;
  const int64_t grid = units < sms ? units : sms;
  const int64_t max_range = (units + grid - 1) / grid * SK_GRAIN;
  const int64_t walk_cap = 256 < max_range ? 256 : max_range;
  if ((swiglu ? 2 * walk_cap : walk_cap) >= 128) return false;
  const int wf = swiglu ? SK_BN / 2 : SK_BN;
  const RowTiling ct =
      choose_row_tiling(p.feat_total, kb_total, kb_total / 32, sms, 8, 1, kResident, wf);
  *out = ct;
  if (ct.cs < 2) return false;
  bool ok = false;
  [&] {
    CHECK(ct.tiles == (p.feat_total + wf - 1) / wf && ct.cs <= 8 && 32 * ct.cs <= kb_total &&
              ct.tiles <= kResident[ct.cs],
          "%lld tiles x %d", (long long)ct.tiles, ct.cs);
    p.cs = ct.cs;
    p.tile_cap = wf;
    const int tile_rows = swiglu ? 2 * wf : wf;
    int64_t expect = 0;
    for (int64_t tile = 0; tile < ct.tiles; ++tile) {
      int next_kb = 0;
      for (int rank = 0; rank < ct.cs; ++rank) {
        const int64_t block = tile * ct.cs + rank;
        int64_t f0, f1;
        column_split_range_of(p, block, f0, f1);
        CHECK(f0 == expect && f1 > f0 && f1 - f0 <= wf, "cluster %lld range [%lld, %lld)",
              (long long)tile, (long long)f0, (long long)f1);
        int kb0, kb1;
        split_kb_range(p, rank, kb0, kb1);
        CHECK(kb0 == next_kb && kb1 > kb0, "rank %d k-range [%d, %d)", rank, kb0, kb1);
        next_kb = kb1;
        walk_tiles(p, widths, swiglu, tile_rows, f0, f1);
        if (fails) return;
        // partial-sum slots: feature offset in the range (+ wf for up rows)
        for (int64_t f = f0; f < f1;) {
          const Tile t = column_tile(p, f, f1);
          for (int i = 0; i < t.n; ++i) {
            const int64_t fl0 = p.fo[t.pc[i].shard] + t.pc[i].loc - f0;
            CHECK(fl0 >= 0 && fl0 + t.pc[i].c <= f1 - f0, "piece slot [%lld, %lld)",
                  (long long)fl0, (long long)(fl0 + t.pc[i].c));
            CHECK(fl0 + t.pc[i].c + (swiglu ? wf : 0) <= SK_BN + 4, "beyond the buffer row");
          }
        }
        if (rank == ct.cs - 1) expect = f1;
      }
      CHECK(next_kb == kb_total, "ranks end at k-block %d of %d", next_kb, kb_total);
    }
    CHECK(expect == p.feat_total, "clusters end at %lld of %lld", (long long)expect,
          (long long)p.feat_total);
    ok = true;
  }();
  return ok;
}

// The launchers' choice for n_out outputs and tp shards of kbs k-blocks:
// bf16 kernel (cluster unit 1) and FP8 kernels (unit tp, one shard per CTA).
static void check_choice(int64_t n_out, int tp, int kbs, bool fp8, int sms, RowTiling* out) {
  const int unit = fp8 ? tp : 1;
  const int64_t kb_total = (int64_t)kbs * tp;
  const RowTiling rt =
      choose_row_tiling(n_out, kb_total, fp8 ? kbs : kb_total, sms, 8, unit, kResident);
  *out = rt;
  CHECK(rt.bn == SK_BN, "bn %d", rt.bn);
  CHECK(rt.cs % unit == 0 && rt.cs >= unit && rt.cs <= 8, "cs %d (unit %d)", rt.cs, unit);
  CHECK(rt.tiles == (n_out + rt.bn - 1) / rt.bn, "tiles %lld", (long long)rt.tiles);
  CHECK(rt.cs <= kb_total && (!fp8 || rt.cs / tp <= kbs), "cs %d for %d k-blocks", rt.cs, kbs);
  // every cluster resident at once, and no larger admissible cluster would be
  CHECK(rt.cs == unit || rt.tiles <= kResident[rt.cs], "%lld clusters of %d", (long long)rt.tiles,
        rt.cs);
  for (int c = rt.cs + unit; c <= 8 && c / unit <= (fp8 ? kbs : kb_total); c += unit)
    CHECK(rt.tiles > kResident[c], "clusters of %d would fit too (cs %d chosen)", c, rt.cs);
  check_row(n_out, tp, kbs, rt.bn, rt.cs, fp8);
}

// The down projection of the decode FFN (d_ff 28672, tp 4, d_model 8192):
// bf16 448 k-blocks of 64, FP8 56 k-blocks of 128 per shard.  Both take 32
// tiles x 4 CTAs (33 clusters of 4 fit; 26 of 5 would not).
static void check_down_projection(int sms) {
  RowTiling b, f;
  check_choice(8192, 4, 112, false, sms, &b);
  CHECK(b.cs == 4 && b.tiles == 32, "bf16 down projection %d x %d", b.bn, b.cs);
  check_choice(8192, 4, 56, true, sms, &f);
  CHECK(f.cs == 4 && f.tiles == 32, "FP8 down projection %d x %d", f.bn, f.cs);
}

int main() {
  const int sms = 148;
  // decode FFN up projection, d_ff 28672, tp 4 (7168 per shard): bf16 kernel
  // (cap 256), FP8 shared-memory mode (SwiGLU cap 128), FP8 TMEM kernel
  // (SwiGLU 256 features, plain 512 rows)
  check_column({7168, 7168, 7168, 7168}, true, 256, sms);
  check_column({7168, 7168, 7168, 7168}, true, 128, sms);
  check_column({7168, 7168, 7168, 7168}, false, 512, sms);
  // QKV of the 70B attention, tp 8: (64 + 16) heads x 128 / 8 = 1280 per shard
  check_column(std::vector<int64_t>(8, 1280), false, 256, sms);
  // the uneven tp=3 split of d_ff 28672, and small ragged test shapes
  check_column({9558, 9557, 9557}, false, 256, sms);
  check_column({5, 4}, false, 256, sms);
  check_column({300, 200, 500}, false, 256, sms);
  check_column({136, 8, 256, 40}, false, 512, sms);
  check_column({200, 200, 200}, false, 256, sms);
  check_column({576, 576}, true, 256, sms);
  check_column({1152, 1152}, true, 256, sms);
  check_column({250, 250, 250, 250}, true, 128, sms);
  check_column({1}, false, 256, sms);
  check_column({16}, true, 256, sms);
  for (int tp = 1; tp <= 8; ++tp) check_column(std::vector<int64_t>(tp, 130 * tp + 7), true, 256, sms);
  // column side with K split: the QKV projection of the 70B attention at
  // tp 4 ((64 + 16) heads x 128 / 4 = 2560 per shard, K 8192): 40 tiles of
  // 256 x 3 CTAs; small and ragged shapes; the choice equals tp = 1's
  {
    RowTiling q;
    const bool split = check_column_split(std::vector<int64_t>(4, 2560), false, 128, sms, &q);
    if (!(split && q.cs == 3 && q.tiles == 40)) {
      std::printf("FAIL: QKV split %d: %lld tiles x %d\n", (int)split, (long long)q.tiles, q.cs);
      ++fails;
    }
  }
  const std::vector<std::vector<int64_t>> split_shapes = {
      {2560, 2560, 2560, 2560}, {1025, 1025, 1025, 1025}, {5, 4}, {300, 200, 500},
      {136, 8, 256, 40}, {200, 200, 200}, {576, 576}, {250, 250, 250, 250}, {1}, {16},
      {2050, 2050}, {1000, 1000, 1000}, {3000}, {100, 100, 100, 100, 100, 100, 100, 100}};
  for (const auto& w : split_shapes)
    for (bool sw : {false, true})
      for (int kb : {1, 2, 3, 16, 63, 64, 96, 128, 448}) {
        RowTiling a, one;
        int64_t total = 0;
        for (int64_t x : w) total += x;
        const bool sa = check_column_split(w, sw, kb, sms, &a);
        const bool s1 = check_column_split({total}, sw, kb, sms, &one);
        if (sa != s1 || (sa && (a.cs != one.cs || a.tiles != one.tiles))) {
          std::printf("FAIL: split choice depends on the shards (%lld features)\n",
                      (long long)total);
          ++fails;
        }
      }
  // row side: bf16 kernel cs = min(8, 148 / tiles) (capped by the k-blocks);
  // FP8 kernels cs = tp x j
  check_row(8192, 4, 112, 256, 4, true);
  check_row(8192, 8, 56, 256, 4, false);
  check_row(300, 1, 8, 256, 8, true);
  check_row(1024, 2, 16, 256, 8, true);
  check_row(520, 4, 4, 256, 8, true);
  check_row(768, 6, 8, 256, 6, true);
  check_row(40, 3, 1, 256, 3, true);
  check_row(200, 3, 8, 256, 8, false);
  check_down_projection(sms);
  const int64_t outs[] = {1, 16, 40, 200, 300, 520, 768, 1024, 4096, 8192, 8200, 28672};
  const int kbss[] = {1, 2, 5, 8, 56, 112};
  for (int64_t n : outs)
    for (int tp = 1; tp <= 8; ++tp)
      for (int kbs : kbss) {
        RowTiling rt;
        check_choice(n, tp, kbs, false, sms, &rt);
        check_choice(n, tp, kbs, true, sms, &rt);
      }
  if (fails) {
    std::printf("%d violation(s)\n", fails);
    return 1;
  }
  std::printf("ok\n");
  return 0;
}
