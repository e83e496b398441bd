// Host-side checks of the persistent launcher's stage partition and shared-memory layout (no
// GPU needed: only host functions run). The kernel's source is compiled into this program as
// it is; the test prints "ok <cases>" or the first broken property and exits non-zero.
//
// Shared-memory layout, for every kernel instance, ring depth, vectors per pass and
// activation length (multiples of 512 up to 65,536): the activation buffers start on 16 bytes
// (bulk and 16-byte copies), the mbarriers on 8, the head partials, reductions, flags, stage
// scales and slot rows on their element size, the chained record state on 8 (it holds a
// pointer); regions follow one another without overlap; every configuration pick_config
// returns fits the 227 KB budget, and it returns one whenever the shallowest ring with one
// vector per pass fits.
//
// Stage partition, for random stages of 1-3 unit sets on grids of 1 to 160 CTAs:
//   * every unit of every set is owned by exactly one item (no gap, no overlap);
//   * an item holds a non-empty unit range, except the empty item a CTA without work gets so
//     that it still takes part in a stage's grid barrier;
//   * with a barrier before the stage, every CTA's first item of the stage, and only that one,
//     carries the barrier flag;
//   * with one set per CTA (stages between barriers, when there are at least as many CTAs as
//     sets), no CTA holds units of two sets;
//   * without it, no CTA holds more than its byte share plus one unit;
//   * chained stages: CTA 0 holds exactly one item, empty, and the units go to CTAs 1..grid-1.
#include "nt_persist.cu"

#include <cstdio>
#include <random>

using nt::WorkItem;

namespace {

int fail(const char* what, int grid, int ns, int one_item, int barrier) {
  std::printf("FAIL %s (grid %d, sets %d, one_item %d, barrier %d)\n", what, grid, ns, one_item, barrier);
  return 1;
}

int check(const std::vector<nt::Unitset>& sets, int grid, bool one_item, bool barrier, bool chained) {
  const int ns = (int)sets.size();
  // one set per CTA needs at least as many CTAs (CTAs 1..grid-1 in chained stages) as sets;
  // with fewer, CTAs take contiguous byte ranges across the sets
  const bool one_set = (one_item || chained) && ns <= (chained ? grid - 1 : grid);
  std::vector<std::vector<WorkItem>> per(grid);
  per[0].push_back(WorkItem{nt::kItemTernary, 999, 0, 0, 0, 0});  // an earlier stage's item stays
  if (chained) nt::partition_stage_chained(sets, grid, 3, barrier, per);
  else nt::partition_stage(sets, grid, 3, barrier, per, one_item);
  per[0].erase(per[0].begin());
  int64_t total = 0, maxu = 0;
  for (const auto& s : sets) total += s.units * s.unit_bytes, maxu = std::max(maxu, s.unit_bytes);
  std::vector<std::vector<int>> owner(ns);
  for (int i = 0; i < ns; ++i) owner[i].assign((size_t)sets[i].units, 0);
  for (int c = 0; c < grid; ++c) {
    int flagged = 0, set_of_cta = -1;
    int64_t bytes = 0;
    for (size_t k = 0; k < per[c].size(); ++k) {
      const WorkItem& w = per[c][k];
      if (w.b0 != 3) return fail("wrong pass", grid, ns, one_item, barrier);
      if (w.flags & nt::kFlagStage) {
        ++flagged;
        if (k != 0) return fail("barrier flag not on the stage's first item", grid, ns, one_item, barrier);
      }
      if (w.begin == w.end) {
        if (!(barrier || (chained && c == 0)) || per[c].size() != 1)
          return fail("empty item where none is needed", grid, ns, one_item, barrier);
        continue;
      }
      if (w.begin > w.end || w.begin < 0) return fail("bad range", grid, ns, one_item, barrier);
      int si = -1;
      for (int i = 0; i < ns; ++i)
        if (sets[i].mat == w.mat && sets[i].kind == w.kind) si = i;
      if (si < 0 || w.end > sets[si].units) return fail("range outside its set", grid, ns, one_item, barrier);
      if (one_set && set_of_cta >= 0 && set_of_cta != si)
        return fail("a CTA holds two sets", grid, ns, one_item, barrier);
      set_of_cta = si;
      for (int64_t u = w.begin; u < w.end; ++u) ++owner[si][(size_t)u];
      bytes += (w.end - w.begin) * sets[si].unit_bytes;
    }
    if (barrier && flagged != 1) return fail("barrier flag count", grid, ns, one_item, barrier);
    if (!barrier && flagged != 0) return fail("flag without a barrier", grid, ns, one_item, barrier);
    if (chained && c == 0 && (per[0].size() != 1 || per[0][0].begin != per[0][0].end))
      return fail("chained CTA 0 holds units", grid, ns, one_item, barrier);
    if (!one_item && !chained && bytes > total / grid + maxu + 1)
      return fail("byte share exceeded", grid, ns, one_item, barrier);
  }
  for (int i = 0; i < ns; ++i)
    for (int v : owner[i])
      if (v != 1) return fail(v ? "unit owned twice" : "unit not owned", grid, ns, one_item, barrier);
  return 0;
}

template <class C>
int check_layouts(bool chained) {
  int cases = 0;
  for (int act_k = 512; act_k <= 65536; act_k += 512) {
    for (int ns = 2; ns <= nt::kMaxSlots; ++ns)
      for (int cb = 1; cb <= C::NBMAX; ++cb) {
        const nt::SmemLayout L = nt::smem_layout<C>(ns, cb, act_k);
        const int at[] = {L.ring, L.act, L.bars, L.hbest, L.red, L.abort_flag, L.chain_s, L.slot_row,
                          L.rec_state, L.total};
        for (int i = 0; i + 1 < 10; ++i)
          if (at[i + 1] < at[i]) { std::printf("FAIL layout regions out of order\n"); return -1; }
        if (L.ring != 0 || L.act % 16 || L.bars % 8 || L.hbest % (int)alignof(nt::HeadPartial) || L.red % 4 ||
            L.abort_flag % 4 || L.chain_s % 4 || L.slot_row % 4 || L.rec_state % 8) {
          std::printf("FAIL misaligned layout (ns %d, cb %d, act_k %d)\n", ns, cb, act_k);
          return -1;
        }
        if (L.act - L.ring != C::CW * ns * nt::kSlotBytes || L.bars - L.act != 2 * cb * act_k ||
            L.slot_row + C::CW * nt::kMaxSlots * 4 > L.rec_state || L.total - L.rec_state != (chained ? 32 : 0)) {
          std::printf("FAIL layout region sizes (ns %d, cb %d, act_k %d)\n", ns, cb, act_k);
          return -1;
        }
        ++cases;
      }
    for (int B = 1; B <= nt::kStepMaxBatch; ++B) {
      if ((B == 1) != (C::NBMAX == 1)) continue;
      int nslots = 0, chunk_b = 0;
      size_t smem = 0;
      const bool ok = nt::pick_config(B, act_k, &nslots, &chunk_b, &smem, chained);
      const bool any = nt::smem_layout<C>(2, 1, act_k).total <= nt::kMaxSmem;
      if (ok != any) { std::printf("FAIL pick_config at B %d, act_k %d\n", B, act_k); return -1; }
      if (ok && (smem > (size_t)nt::kMaxSmem || nslots < 2 || nslots > nt::kMaxSlots || chunk_b < 1 ||
                 chunk_b > std::min(B, C::NBMAX) || smem != (size_t)nt::smem_layout<C>(nslots, chunk_b, act_k).total)) {
        std::printf("FAIL picked configuration at B %d, act_k %d\n", B, act_k);
        return -1;
      }
      ++cases;
    }
  }
  return cases;
}

}  // namespace

int main() {
  std::mt19937_64 rng(12345);
  const int grids[] = {1, 2, 3, 7, 64, 148, 152, 160};
  const int64_t unit_bytes[] = {512, 1024, 4096, 12288, 4096 + 16};
  int cases = 0;
  for (int i = 0; i < 4; ++i) {
    const int n = i == 0 ? check_layouts<nt::Cfg1>(false) : i == 1 ? check_layouts<nt::CfgB>(false)
                : i == 2 ? check_layouts<nt::Cfg1C>(true) : check_layouts<nt::CfgBC>(true);
    if (n < 0) return 1;
    cases += n;
  }
  for (int rep = 0; rep < 300; ++rep)
    for (int grid : grids)
      for (int ns = 1; ns <= 3; ++ns) {
        std::vector<nt::Unitset> sets;
        for (int i = 0; i < ns; ++i) {
          const int64_t units = 1 + (int64_t)(rng() % (rep % 3 == 0 ? 8 : 3100));
          sets.push_back(nt::Unitset{nt::kItemTernary, 10 * rep + i, units, unit_bytes[rng() % 5]});
        }
        for (int mode = 0; mode < 5; ++mode) {
          const bool chained = mode == 4;
          if (chained && grid < 2) continue;
          const bool one_item = mode >= 2, barrier = mode % 2 == 1 || chained;
          if (check(sets, grid, one_item, barrier, chained)) return 1;
          ++cases;
        }
      }
  std::printf("ok %d\n", cases);
  return 0;
}
