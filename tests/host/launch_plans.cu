// launch_plans.cu -- host-side checks of the launch planning that
// libmla_prolog.so does before any kernel runs.  None of the functions
// called here touches the device, so this runs on a machine without a GPU.
//
//  1. decode_plan over the model shapes and several SM counts: the split-K
//     of kv_a covers `hidden` with at most one tile per CTA, the W_kvb
//     column groups of every CTA fit its box, and the shared-memory layout
//     (resident W_kvb rows, region A, reduction scratch, misc) is ordered,
//     aligned and within the 227 KB budget, with region A large enough for
//     the phase-A ring and, when W_kvb is streamed, the latent rows plus two
//     stream buffers at the largest row count.
//  2. decode_phase_b: the warp assignment of the decode kernel's phase B,
//     restated below from the kernel, computes every (m-tile, column group,
//     k16 step) of every CTA exactly once, and the cross-slice scratch index
//     stays inside the 16 KB reduction area.
//  3. The packed W_kvb layout: the owner formula finds the CTA whose column
//     range holds a group, the packing is a bijection, and pack_swizzle
//     makes the eight rows of every ldmatrix tile fall in distinct 16-byte
//     bank groups.  The packed W_kva tile (four chunks a row, chunk c at
//     c ^ ((r >> 1) & 3)) is conflict-free the same way.
//  4. The W8A8 workspace: w8_workspace_carve places every region 256-byte
//     aligned, in order, disjoint and inside w8_workspace_bytes, and the
//     small-M plan splits `hidden` into chunks of at most 512 rows.
//
// Prints one line per failure and exits 1 if any check failed.
#include <cstdio>
#include <cstdint>
#include <vector>

#include "../../mla_attention_kv_gb300/csrc/internal.h"

using namespace mla;

namespace {

int g_bad = 0;

#define CHECK(cond, ...)                \
  do {                                  \
    if (!(cond)) {                      \
      ++g_bad;                          \
      std::printf("FAIL %s: ", #cond);  \
      std::printf(__VA_ARGS__);         \
      std::printf("\n");                \
    }                                   \
  } while (0)

// Layout constants of the decode kernel (the same values as its source).
constexpr int kWarps = 8;
constexpr int kSubK = 64, kPitchWA = 80, kPitchX = 144, kPitchN = kNrmPitch;
constexpr int kSmemBudget = 227 * 1024, kRedBytes = 16384, kMiscBytes = 2048;
constexpr int kNblkA = kNa / 32;
constexpr int kVariants[3][2] = {{1, 4}, {1, 8}, {2, 8}};  // (m-tiles, column groups) per warp

int col_group_begin_ref(int c, int NG, int G) { return (int)((long long)c * NG / G); }

void check_decode_shape(int hidden, int heads, int sms) {
  DecodePlan p;
  const bool ok = decode_plan(hidden, heads, sms, &p);
  // every shape of the two model families and of the tests must plan on a
  // GB300-sized part (148..160 SMs)
  CHECK(ok, "hidden %d heads %d sms %d: no plan", hidden, heads, sms);
  if (!ok) return;
  const int NG = heads * kHeadCols / 8;
  CHECK(!p.two_per_sm, "the main plan is built for one CTA per SM");
  // the <= 32-row plan: two CTAs per SM, W_kvb slice resident, same split-K
  DecodePlan q;
  if (decode_plan_small(hidden, heads, sms, &q)) {
    CHECK(q.two_per_sm && q.tt_max == kDecodeSmallTokens, "small plan tt_max %d", q.tt_max);
    CHECK(2 * (q.smem + 1024) <= 228 * 1024, "small plan smem %zu: two CTAs do not fit", q.smem);
    CHECK(q.kpre == kRank, "small plan kpre %d", q.kpre);
    CHECK(q.KB == p.KB && q.KC == p.KC && q.ngmax == p.ngmax && q.grid == p.grid, "small plan split");
    CHECK(q.nstA * (kSubK * kPitchWA + q.tt_max * kPitchX) <= q.off_red - q.off_a, "small plan ring");
    CHECK(q.tt_max * kPitchN <= q.off_red - q.off_a, "small plan latent rows");
  } else {
    // only shapes whose W_kvb slice cannot stay resident in half the SM may go without
    CHECK(p.kpre < kRank || heads * kHeadCols / sms * 2 * kRank > 40 * 1024, "no small plan for hidden %d heads %d",
          hidden, heads);
  }
  CHECK(p.grid == sms, "grid %d", p.grid);
  CHECK(p.tt_max == 64 || p.tt_max == 128, "tt_max %d", p.tt_max);
  CHECK(p.KB % 64 == 0 && p.KB * p.KC == hidden, "KB %d KC %d hidden %d", p.KB, p.KC, hidden);
  CHECK(p.KC <= 16 && p.KC * kNblkA <= sms, "KC %d", p.KC);
  CHECK(p.ngmax * sms >= NG && (p.ngmax - 1) * sms < NG, "ngmax %d NG %d", p.ngmax, NG);
  CHECK((p.ngbox & 1) && p.ngbox >= p.ngmax && p.ngbox * 8 <= 256, "ngbox %d", p.ngbox);
  CHECK(p.kpre >= p.tt_max && p.kpre <= kRank && p.kpre % 32 == 0, "kpre %d", p.kpre);
  CHECK(p.kchunk % 32 == 0 && p.kchunk >= 32, "kchunk %d", p.kchunk);
  CHECK(p.nstA >= 2 && p.nstA <= 4, "nstA %d", p.nstA);
  const int pitchB = p.ngbox * 16;
  CHECK(p.off_wb == 0 && p.off_a >= p.kpre * pitchB && p.off_a % 1024 == 0, "off_a %d", p.off_a);
  CHECK(p.off_red > p.off_a && p.off_red % 128 == 0, "off_red %d", p.off_red);
  CHECK(p.off_misc == p.off_red + kRedBytes, "off_misc %d", p.off_misc);
  CHECK(p.smem == (size_t)p.off_misc + kMiscBytes + 1024 && p.smem <= (size_t)kSmemBudget, "smem %zu",
        p.smem);
  CHECK(p.partial_floats == (size_t)p.KC * kDecodeMaxTokens * kNa, "partial_floats %zu", p.partial_floats);
  const int regionA = p.off_red - p.off_a;
  // the phase-A ring at the plan's row count (the raw-weight stage is the
  // larger of the two stage forms)
  CHECK(p.nstA * (kSubK * kPitchWA + p.tt_max * kPitchX) <= regionA, "ring %d x stage > region A %d",
        p.nstA, regionA);
  CHECK(p.tt_max * kPitchN <= regionA, "latent rows > region A");
  if (p.kpre < kRank)
    CHECK(p.tt_max * kPitchN + 2 * kWkvbBoxRows * pitchB <= regionA, "no room for two stream buffers");

  // phase B on the tensor cores: wide slices, at most 64 rows, one CTA per
  // SM; the resident K blocks fit the W area, the 64 KB latent operand and
  // the buffer blocks fit region A, the refills have a slot-free barrier
  // each (6), and the output tile fits the W area
  const int blk = p.ngmax * 8 * 128;
  if (p.tc_b) {
    CHECK(p.tt_max <= 64 && !p.two_per_sm && p.ngmax * 8 >= 128, "tc_b plan tt %d ngmax %d", p.tt_max, p.ngmax);
    CHECK(p.tb_res >= 1 && p.tb_res <= 8 && p.tb_res * blk <= p.off_a, "tb_res %d", p.tb_res);
    CHECK(p.tb_buf >= 0 && p.tb_res + p.tb_buf <= 8 && 64 * 1024 + p.tb_buf * blk <= regionA, "tb_buf %d",
          p.tb_buf);
    CHECK(8 - p.tb_res - p.tb_buf <= 6, "refills %d", 8 - p.tb_res - p.tb_buf);
    CHECK(64 * pitchB <= p.off_a, "output tile");
  } else {
    CHECK(p.ngmax * 8 < 128 || p.tt_max > 64, "wide slice without tc_b: ngmax %d", p.ngmax);
  }
  std::printf("plan hidden %d heads %d sms %d: tt %d KC %d kpre %d off_a %d off_red %d tc_b %d res %d buf %d\n",
              hidden, heads, sms, p.tt_max, p.KC, p.kpre, p.off_a, p.off_red, (int)p.tc_b, p.tb_res, p.tb_buf);

  // phase B for every row count the plan takes
  for (int mt = 1; mt * 16 <= p.tt_max; mt *= 2) {
    int v = -1, wm = 0, ks = 0;
    const bool pb = decode_phase_b(mt, p.ngmax, &v, &wm, &ks);
    CHECK(pb, "no phase-B split mt %d ngmax %d", mt, p.ngmax);
    if (!pb) continue;
    CHECK(v >= 0 && v < 3, "variant %d", v);
    const int IM = kVariants[v][0], QM = kVariants[v][1];
    const int wn = kWarps / wm;
    CHECK(wm * IM == mt && wm * wn == kWarps && wn % ks == 0, "grid wm %d ks %d mt %d", wm, ks, mt);
    for (int cta = 0; cta < sms; ++cta) {
      const int g0 = col_group_begin_ref(cta, NG, sms), ng = col_group_begin_ref(cta + 1, NG, sms) - g0;
      CHECK(ng <= p.ngmax, "cta %d ng %d", cta, ng);
      std::vector<int> cover((size_t)mt * ng * 32, 0);
      for (int warp = 0; warp < kWarps; ++warp) {
        const int mw = warp % wm, wr = warp / wm, my = wr % ks;
        for (int q = 0; q < QM; ++q) {
          const int j = wr + q * wn;
          if (j >= ng * ks) continue;
          CHECK(j % ks == my, "item slice");
          const int gi = j / ks;
          for (int i = 0; i < IM; ++i) {
            const int m = mw + i * wm;
            CHECK(m < mt, "m-tile %d", m);
            for (int st = 0; st < 32; ++st)
              if (st % ks == my) cover[((size_t)m * ng + gi) * 32 + st]++;
            if (ks > 1) {
              const int pr = gi * mt + m;
              CHECK(((pr * ks + my) * 32 + 31) * 4 + 4 <= kRedBytes / 4, "scratch pr %d", pr);
            }
          }
        }
      }
      int wrong = 0;
      for (int x : cover) wrong += x != 1;
      CHECK(wrong == 0, "hidden %d heads %d sms %d mt %d cta %d: %d items not computed once", hidden, heads,
            sms, mt, cta, wrong);
      if (wrong) return;
    }
  }
}

void check_packing(int NG, int G) {
  std::vector<int> hit((size_t)kRank * NG, 0);
  for (int g = 0; g < NG; ++g) {
    const int c = (int)(((long long)(g + 1) * G + NG - 1) / NG) - 1;
    const int g0 = col_group_begin_ref(c, NG, G), g1 = col_group_begin_ref(c + 1, NG, G);
    CHECK(g0 <= g && g < g1, "owner NG %d G %d g %d -> cta %d", NG, G, g, c);
    const int ng = g1 - g0, j = g - g0;
    for (int r = 0; r < kRank; ++r) {
      const int jj = j ^ pack_swizzle(ng, r);
      CHECK(jj >= 0 && jj < ng, "swizzle ng %d r %d", ng, r);
      if (jj < 0 || jj >= ng) return;
      hit[(size_t)g0 * kRank + (size_t)r * ng + jj]++;
    }
  }
  int wrong = 0;
  for (int x : hit) wrong += x != 1;
  CHECK(wrong == 0, "packing NG %d G %d not a bijection (%d)", NG, G, wrong);
}

void check_swizzle_banks() {
  // chunk slot of (row r, chunk c) in a slice of ng chunks per row, mod the
  // eight 16-byte bank groups: an ldmatrix reads one chunk of eight
  // consecutive rows
  for (int ng = 1; ng <= 32; ++ng)
    for (int c = 0; c < ng; ++c)
      for (int r0 = 0; r0 < kRank; r0 += 8) {
        int used[8] = {0};
        for (int r = r0; r < r0 + 8; ++r) used[(r * ng + (c ^ pack_swizzle(ng, r))) % 8]++;
        for (int k = 0; k < 8; ++k) CHECK(used[k] == 1, "bank conflict ng %d c %d r0 %d", ng, c, r0);
      }
  for (int c = 0; c < 4; ++c)
    for (int r0 = 0; r0 < 64; r0 += 8) {
      int used[8] = {0};
      for (int r = r0; r < r0 + 8; ++r) used[(r * 4 + (c ^ ((r >> 1) & 3))) % 8]++;
      for (int k = 0; k < 8; ++k) CHECK(used[k] == 1, "W_kva tile conflict c %d r0 %d", c, r0);
    }
}

void check_w8_workspace(int hidden, int q_rank, int heads, int max_tokens, int sms) {
  const size_t bytes = w8_workspace_bytes(hidden, q_rank, heads, max_tokens, sms);
  // carve at a fake, 256-aligned base: only addresses are computed
  const uintptr_t base = (uintptr_t)1 << 40;
  W8Workspace w{};
  W8SmallPlan pl{};
  w8_workspace_carve(reinterpret_cast<void*>(base), hidden, q_rank, heads, max_tokens, sms, &w, &pl);
  const size_t T = (size_t)max_tokens;
  const size_t units = (size_t)(sms + 1 + pl.nblk_b) * 4;
  struct Region { const char* name; uintptr_t at; size_t len; } rg[] = {
      {"xh", (uintptr_t)w.xh, T * hidden * 2},
      {"sx", (uintptr_t)w.sx, T * 4},
      {"acc1", (uintptr_t)w.acc1, T * (q_rank + kNa) * 4},
      {"q1", (uintptr_t)w.q1, T * q_rank},
      {"s1", (uintptr_t)w.s1, T * 4},
      {"c1", (uintptr_t)w.c1, T * kRank},
      {"s2", (uintptr_t)w.s2, T * 4},
      {"q1h", (uintptr_t)w.q1h, T * q_rank * 2},
      {"c1h", (uintptr_t)w.c1h, T * kRank * 2},
      {"units", (uintptr_t)pl.units, units},
      {"readers", (uintptr_t)w.readers, 256},
      {"wa16", (uintptr_t)w.wa16, w.wa16 ? (size_t)hidden * w.lda * 2 : 0},
      {"wqb16", (uintptr_t)w.wqb16, w.wqb16 ? (size_t)q_rank * w.ldqb * 2 : 0},
      {"wkvb16", (uintptr_t)w.wkvb16, w.wkvb16 ? (size_t)kRank * w.ldkvb * 2 : 0},
  };
  CHECK((max_tokens >= kW8PairMinRows) == (w.wa16 != nullptr), "widened copies at max_tokens %d", max_tokens);
  CHECK(w.lda % 256 == 0 && w.ldqb % 256 == 0 && w.ldkvb % 256 == 0, "widened pitches");
  uintptr_t end = base;
  for (const Region& r : rg) {
    if (r.len == 0) continue;
    CHECK(r.at % 256 == 0, "%s not 256-byte aligned", r.name);
    CHECK(r.at >= end, "%s overlaps the region before it", r.name);
    end = r.at + r.len;
  }
  CHECK(end <= base + bytes, "regions end %zu bytes past the workspace of %zu", (size_t)(end - base - bytes),
        bytes);
  CHECK(pl.kchunk % 32 == 0 && pl.kchunk <= 512 && pl.kchunk >= 32, "kchunk %d", pl.kchunk);
  CHECK(pl.splits * pl.kchunk >= hidden && (pl.splits - 1) * pl.kchunk < hidden, "splits %d", pl.splits);
  CHECK(pl.nblk_a1 * 256 >= q_rank && pl.nblk_a == pl.nblk_a1 + (kNa + 255) / 256, "nblk_a %d", pl.nblk_a);
  CHECK(pl.nblk_b1 * 128 >= heads * (kNope + kRope) && pl.nblk_b - pl.nblk_b1 == (heads * kHeadCols + 127) / 128,
        "nblk_b %d", pl.nblk_b);
  CHECK(pl.grid_b >= 1 && pl.grid_b <= sms && pl.grid_b <= pl.nblk_b, "grid_b %d", pl.grid_b);
}

}  // namespace

int main() {
  // (hidden, heads): V2-Lite, R1, and the reduced shapes the parity tests use
  const int shapes[][2] = {{2048, 16}, {7168, 128}, {5120, 128}, {64, 1}, {192, 3},
                           {640, 5},   {2048, 128}, {7168, 16},  {128, 2}, {4096, 32}};
  for (int sms : {148, 152, 160})
    for (const auto& sh : shapes) check_decode_shape(sh[0], sh[1], sms);
  // below 64 SMs the decode kernel is not planned at all
  DecodePlan none;
  CHECK(!decode_plan(2048, 16, 32, &none), "plan with 32 SMs");
  CHECK(!decode_plan(2050, 16, 152, &none), "plan with hidden %% 64 != 0");
  for (int G : {148, 152, 160})
    for (int NG : {32, 96, 160, 512, 2048, 4096, 7, 151, 153}) check_packing(NG, G);
  check_swizzle_banks();
  for (int sms : {148, 152})
    for (int T : {1, 8, 64, 8192}) {
      check_w8_workspace(7168, 1536, 128, T, sms);
      check_w8_workspace(512, 256, 4, T, sms);
    }
  std::printf("%d failed checks\n", g_bad);
  return g_bad != 0;
}
