// Host harness for the split-KV planning helpers of csrc/plan.cuh (the
// integer part of the decode: tile prefix, even split, sequence-aligned plan,
// plan choice).  It runs on the CPU, with no GPU: stdin holds cases
// ("B G tile L_0 .. L_{B-1}" after a case count); for each case one JSON line
// reports what the helpers return, and tests/test_plan.py checks it against
// the partition invariants the decode kernels rely on.
#include <cstdio>
#include <vector>

#include "../mla_latent_kv_76_b300/csrc/plan.cuh"

using namespace mla;

static void print_list(const char* key, const std::vector<long long>& v, bool last = false) {
  std::printf("\"%s\": [", key);
  for (size_t i = 0; i < v.size(); ++i) std::printf(i ? ", %lld" : "%lld", v[i]);
  std::printf(last ? "]" : "], ");
}

int main() {
  int cases = 0;
  if (std::scanf("%d", &cases) != 1) return 1;
  for (int c = 0; c < cases; ++c) {
    int B = 0, G = 0, tile = 0;
    if (std::scanf("%d %d %d", &B, &G, &tile) != 3 || B < 1 || G < 1 || tile < 1) return 1;
    std::vector<int> L(B), pre(B + 1), W(B + 1);
    for (int b = 0; b < B; ++b)
      if (std::scanf("%d", &L[b]) != 1) return 1;
    // tile prefix (the kernels build it block-wide; here sequentially)
    pre[0] = 0;
    for (int b = 0; b < B; ++b) pre[b + 1] = pre[b] + tiles_of(L[b], tile);
    const long long T = pre[B];
    int n = 0, tmin = 0x7fffffff;
    for (int b = 0; b < B; ++b) {
      const int t = pre[b + 1] - pre[b];
      if (t > 0) {
        ++n;
        if (t < tmin) tmin = t;
      }
    }
    // entry prefix and the aligned plan's longest entry
    W[0] = 0;
    int cost = 0;
    for (int b = 0; b < B; ++b) {
      const int t = pre[b + 1] - pre[b], w = plan_entries(t, T, n, G);
      W[b + 1] = W[b] + w;
      if (w > 0 && (t + w - 1) / w > cost) cost = (t + w - 1) / w;
    }
    const long long E = W[B];
    std::vector<long long> vpre(pre.begin(), pre.end()), vW(W.begin(), W.end()), wb, wof, sot, etile, soe, eot;
    for (int g = 0; g <= G; ++g) wb.push_back(worker_begin(g, T, G));
    for (long long x = 0; x < T; ++x) {
      wof.push_back(worker_of(x, T, G));
      sot.push_back(seq_of_tile(pre.data(), B, x));
    }
    for (long long e = 0; e <= E; ++e) etile.push_back(entry_tile(pre.data(), W.data(), B, e));
    for (long long e = 0; e < E; ++e) soe.push_back(seq_of_entry(W.data(), B, e));
    for (int b = 0; b < B; ++b) {
      const int t = pre[b + 1] - pre[b], w = W[b + 1] - W[b];
      for (int tau = 0; tau < t; ++tau) eot.push_back(entry_of_tile(tau, t, w));
    }
    std::printf("{\"T\": %lld, \"n\": %d, \"cost\": %d, \"aligned\": %d, ", T, n, cost,
                prefer_aligned(cost, T, G, tmin) ? 1 : 0);
    print_list("pre", vpre);
    print_list("W", vW);
    print_list("worker_begin", wb);
    print_list("worker_of", wof);
    print_list("seq_of_tile", sot);
    print_list("entry_tile", etile);
    print_list("seq_of_entry", soe);
    print_list("entry_of_tile", eot, true);
    std::printf("}\n");
  }
  return 0;
}
