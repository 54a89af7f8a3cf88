// Host-side check of the verify step's launch plan (no GPU): includes the
// step kernel's translation unit and checks, for many problem shapes, the
// invariants the kernel relies on. Prints one line per shape and "FAIL ..."
// lines for violations; exit status 1 if any.

#include "step.cu"

#include <cstdio>
#include <vector>

// The planner derives the grid, the splits, the walker and the slice
// placement from the SM count; main() sweeps it.
static int g_sms = 152;
namespace dfv {
int sm_count() { return g_sms; }
}

using dfv::StepPlan;

static int g_fail = 0;
#define CHECK(cond, ...)                                        \
  do {                                                          \
    if (!(cond)) {                                              \
      std::printf("FAIL %s: ", #cond);                          \
      std::printf(__VA_ARGS__);                                 \
      std::printf("\n");                                        \
      ++g_fail;                                                 \
    }                                                           \
  } while (0)

template <int D>
static void stage_sizes(int& tile, int& spare_b, int& kbytes, int& unit_b) {
  tile = dfv::StepSmem<D>::kTileB;
  spare_b = dfv::StepSmem<D>::kSpareStageBytes;
  kbytes = dfv::StepSmem<D>::kKBytes;
  unit_b = dfv::StepSmem<D>::kUnitStageBytes;
}

static void check(int N, int hq, int hkv, int D, int W, int cap, int V, int dt, int fmt) {
  StepPlan pl;
  const bool ok = dfv::step_plan(N, hq, hkv, D, W, cap, V, dt, true, fmt, &pl);
  char tag[160];
  std::snprintf(tag, sizeof tag, "sms=%d N=%d hq=%d hkv=%d D=%d W=%d cap=%d V=%d dt=%d fmt=%d",
                g_sms, N, hq, hkv, D, W, cap, V, dt, fmt);
  if (!ok) {
    std::printf("%s: no plan\n", tag);
    return;
  }
  int tile, spare_b, kbytes, unit_b;
  if (D == 64) stage_sizes<64>(tile, spare_b, kbytes, unit_b);
  else if (D == 128) stage_sizes<128>(tile, spare_b, kbytes, unit_b);
  else stage_sizes<256>(tile, spare_b, kbytes, unit_b);
  const int esz = dt == DFV_DTYPE_BF16 ? 2 : 4;
  CHECK(pl.grid == (g_sms < dfv::kMaxStepGrid ? g_sms : dfv::kMaxStepGrid), "%s grid %d", tag,
        pl.grid);
  CHECK(pl.rows == N * (hq / hkv), "%s rows", tag);
  CHECK(pl.n_grp == (pl.rows + 127) / 128, "%s tiles", tag);
  CHECK(pl.splits >= 1 && pl.units == hkv * pl.n_grp * pl.splits && pl.units <= pl.grid,
        "%s units %d splits %d", tag, pl.units, pl.splits);
  CHECK(pl.walker == (pl.grid > pl.units ? pl.grid - 1 : 0), "%s walker %d", tag, pl.walker);
  // the walker holds no attention unit (its merge would otherwise need a
  // barrier after the walk before its copies into sK)
  CHECK(pl.walker >= pl.units, "%s the walker %d holds an attention unit", tag, pl.walker);
  // the walker stages every argmax partial in its Q tile
  CHECK(static_cast<long>(pl.lunits) * static_cast<long>(sizeof(dfv::ArgPartial)) <= tile,
        "%s lunits %d exceed the walker's staging", tag, pl.lunits);
  if (pl.walker_local)
    CHECK(static_cast<long>(N) * hkv * 2 * dfv::kv_row_bytes(fmt, D) <= kbytes,
          "%s walker's tree rows", tag);
  if (pl.lbulk) {
    // slices are staged in rounds through the two halves of the staging area
    CHECK(pl.lper >= 1 && pl.lper <= dfv::kMaxStagedSlices / 2 &&
              2L * pl.lper * pl.lstride <= spare_b,
          "%s round of %d slices of %d bytes in halves of %d", tag, pl.lper, pl.lstride, spare_b / 2);
    CHECK(pl.lunits == N * pl.lchunks, "%s lunits", tag);
    CHECK(static_cast<long>(pl.lchunk_len) * pl.lchunks >= V, "%s slices cover the vocabulary", tag);
    CHECK((static_cast<long>(V) * esz) % 16 == 0 && (pl.lchunk_len * esz) % 16 == 0,
          "%s slice alignment", tag);
    CHECK(pl.lstride >= pl.lchunk_len * esz && pl.lstride % 16 == 0, "%s stride", tag);
    std::vector<int> seen(pl.lunits, 0);
    for (int b = 0; b < pl.grid; ++b) {
      const int s0 = pl.lslot[b] & 0xFFFF, sn = pl.lslot[b] >> 16;
      if (sn == 0) continue;
      CHECK(b != pl.walker, "%s the walker stages slices", tag);
      if (b < pl.units) {
        // a unit stages one round at entry, in the smem its tile of at most
        // 32 real rows leaves free until its dequant
        const int g = (b / pl.splits) % pl.n_grp;
        const int rows_g = pl.rows - g * 128 < 128 ? pl.rows - g * 128 : 128;
        CHECK(g == pl.n_grp - 1 && rows_g <= dfv::kLightRows, "%s unit %d (tile %d, %d rows) stages slices",
              tag, b, g, rows_g);
        CHECK(sn <= pl.lper && static_cast<long>(sn) * pl.lstride <= unit_b,
              "%s unit %d stages %d slices of %d bytes in %d", tag, b, sn, pl.lstride, unit_b);
      }
      for (int u = s0; u < s0 + sn; ++u) {
        CHECK(u >= 0 && u < pl.lunits, "%s CTA %d slice %d out of range", tag, b, u);
        if (u >= 0 && u < pl.lunits) ++seen[u];
      }
    }
    for (int u = 0; u < pl.lunits; ++u) CHECK(seen[u] == 1, "%s slice %d held %d times", tag, u, seen[u]);
  } else {
    for (int b = 0; b < pl.grid; ++b) CHECK(pl.lslot[b] == 0, "%s CTA %d stages without bulk", tag, b);
  }
  // workspace regions in order, 256-byte aligned
  const size_t groups = static_cast<size_t>(hkv) * pl.n_grp;
  CHECK(pl.ws_bar == 0 && pl.ws_arg % 256 == 0 && pl.ws_qrows % 256 == 0 && pl.ws_ml % 256 == 0 &&
            pl.ws_o % 256 == 0 && pl.ws_total % 256 == 0,
        "%s workspace alignment", tag);
  CHECK(pl.ws_arg >= (4 + 2 * groups + pl.units) * 4 &&
            pl.ws_qrows >= pl.ws_arg + static_cast<size_t>(pl.lunits) * sizeof(dfv::ArgPartial) &&
            pl.ws_ml >= pl.ws_qrows + static_cast<size_t>(N) * hkv * 2 * D * 2 &&
            pl.ws_o >= pl.ws_ml && pl.ws_total >= pl.ws_o,
        "%s workspace order", tag);
  if (pl.splits > 1) {
    // partial rows: D fp16 values + (max, sum) + padding each
    CHECK(pl.ws_total - pl.ws_o >= static_cast<size_t>(pl.units) * 128 * (D * 2 + 16),
          "%s partial sizes", tag);
    // the merge stages (rows + splits) partial rows at most in sK + sV
    const long merge_b = kbytes + 128L * D * 2;
    CHECK((128 + pl.splits) * static_cast<long>(D * 2 + 16) <= merge_b,
          "%s merge staging", tag);
  }
  std::printf("%s: grid %d units %d splits %d tiles %d lunits %d lbulk %d walker_local %d\n", tag,
              pl.grid, pl.units, pl.splits, pl.n_grp, pl.lunits, pl.lbulk, pl.walker_local);
}

int main() {
  const int heads[][2] = {{4, 1}, {8, 2}, {24, 4}, {32, 4}, {6, 6}};
  for (int sms : {100, 132, 148, 152, 160, 256, 300}) {
  g_sms = sms;
  for (int D : {64, 128, 256})
    for (const auto& h : heads)
      for (int N : {1, 9, 23, 49, 65})
        for (int W : {0, 2048})
          for (int C : {0, 4096, 61440, 131072})
            for (int V : {1, 7, 1024, 32000, 151936, 262143, 262144})
              for (int dt : {DFV_DTYPE_BF16, DFV_DTYPE_F32})
                for (int fmt : {DFV_KV_Q4_0, DFV_KV_F16})
                  check(N, h[0], h[1], D, W, C + 64 * N, V, dt, fmt);
  }
  std::printf("%s (%d failures)\n", g_fail ? "FAILED" : "ok", g_fail);
  return g_fail ? 1 : 0;
}
