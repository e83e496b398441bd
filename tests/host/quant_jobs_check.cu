// Host-side check of the persistent launcher's first-phase job placement (no GPU needed: only
// host functions run). The plan source is compiled into this program as it is; the test
// prints "ok <cases>" or the first broken property and exits non-zero.
//
// CTA c runs entries c, c + grid, c + 2 grid, ... of the placed list. Properties:
//   * the list is whole rounds of `grid` entries, and a round-trip finds every vector of every
//     job exactly once, as a one-vector job with its own x, q and s; the rest are empty;
//   * the placement is a longest-processing-time one: the most loaded CTA carries at most the
//     mean load plus one job;
//   * the 8B-shaped batch-1 step (216 inputs of 4,096 values, 36 of 12,288 and the output
//     projection's 4,096) on 152 CTAs: a CTA holds one 12,288-wide vector and nothing else,
//     or at most two 4,096-wide ones.
#include "nt_step.cu"

#include <cstdio>
#include <map>
#include <random>

namespace {

const float* fx(int64_t i) { return reinterpret_cast<const float*>(static_cast<uintptr_t>(0x10000000ull + 64 * i)); }
int8_t* fq(int64_t i) { return reinterpret_cast<int8_t*>(static_cast<uintptr_t>(0x20000000ull + 64 * i)); }
float* fs(int64_t i) { return reinterpret_cast<float*>(static_cast<uintptr_t>(0x30000000ull + 64 * i)); }

int check(const std::vector<nt::QuantJob>& jobs, int grid, bool step8b) {
  const std::vector<nt::QuantJob> out = place_quant_jobs(jobs, grid);
  if (out.size() % (size_t)grid != 0) { std::printf("FAIL not whole rounds (grid %d)\n", grid); return 1; }
  // expected vectors: (x, q, s, K) of each job's vector b
  std::map<const float*, std::pair<int, int>> want;  // x -> (K, times found)
  std::map<const float*, std::pair<int8_t*, float*>> dst;
  int64_t total = 0, max_job = 0;
  for (const nt::QuantJob& j : jobs)
    for (int b = 0; b < j.B; ++b) {
      want[j.x + (int64_t)b * j.K] = {j.K, 0};
      dst[j.x + (int64_t)b * j.K] = {j.q + (int64_t)b * j.K, j.s + b};
      total += j.K + 1024;
      max_job = std::max<int64_t>(max_job, j.K + 1024);
    }
  std::vector<int64_t> load(grid, 0);
  std::vector<int> n12(grid, 0), n4(grid, 0);
  for (size_t e = 0; e < out.size(); ++e) {
    const nt::QuantJob& j = out[e];
    const int c = (int)(e % (size_t)grid);
    if (j.B == 0) {
      if (j.x || j.q || j.s || j.K) { std::printf("FAIL empty entry not blank\n"); return 1; }
      continue;
    }
    auto it = want.find(j.x);
    if (j.B != 1 || it == want.end() || it->second.first != j.K || dst[j.x].first != j.q || dst[j.x].second != j.s) {
      std::printf("FAIL entry is not one of the jobs' vectors (grid %d)\n", grid);
      return 1;
    }
    ++it->second.second;
    load[c] += j.K + 1024;
    (j.K == 12288 ? n12 : n4)[c] += 1;
  }
  for (const auto& kv : want)
    if (kv.second.second != 1) { std::printf("FAIL a vector placed %d times\n", kv.second.second); return 1; }
  const int64_t worst = *std::max_element(load.begin(), load.end());
  if (worst > total / grid + max_job) { std::printf("FAIL load %lld above mean + one job\n", (long long)worst); return 1; }
  if (step8b)
    for (int c = 0; c < grid; ++c)
      if ((n12[c] > 0 && (n12[c] > 1 || n4[c] > 0)) || n4[c] > 2) {
        std::printf("FAIL 8B step: CTA %d holds %d wide and %d narrow vectors\n", c, n12[c], n4[c]);
        return 1;
      }
  return 0;
}

}  // namespace

int main() {
  int cases = 0;
  int64_t id = 0;
  {  // the 8B-shaped batch-1 step in projection order, then the output projection
    std::vector<nt::QuantJob> jobs;
    const int Ks[7] = {4096, 4096, 4096, 4096, 4096, 4096, 12288};
    for (int l = 0; l < 36; ++l)
      for (int k : Ks) { jobs.push_back(nt::QuantJob{fx(id), fq(id), fs(id), k, 1}); id += 1000; }
    jobs.push_back(nt::QuantJob{fx(id), fq(id), fs(id), 4096, 1});
    id += 1000;
    if (check(jobs, 152, true)) return 1;
    ++cases;
  }
  std::mt19937_64 rng(777);
  const int grids[] = {1, 2, 7, 64, 152, 160};
  for (int rep = 0; rep < 400; ++rep)
    for (int grid : grids) {
      std::vector<nt::QuantJob> jobs;
      const int n = 1 + (int)(rng() % 300);
      for (int i = 0; i < n; ++i) {
        const int K = 16 * (1 + (int)(rng() % 1024)), B = 1 + (int)(rng() % 16);
        jobs.push_back(nt::QuantJob{fx(id), fq(id), fs(id), K, B});
        id += (int64_t)K * B + 64;
      }
      if (check(jobs, grid, false)) return 1;
      ++cases;
    }
  std::printf("ok %d\n", cases);
  return 0;
}
