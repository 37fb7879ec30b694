// Host fuzz driver for the block allocator, built with ASan/UBSan by
// tests/test_allocator_cpp.py.  Runs a seeded random script through the C ABI
// and checks structural invariants after every call:
//   * refcount of every block == number of tables holding it;
//   * the free queue holds exactly the blocks with refcount 0, once each;
//   * each table has ceil(len / block_size) entries;
//   * a failed call changes nothing (checked via a snapshot);
//   * with prefix caching on: the number of blocks carrying a hash equals the
//     map size the stats report;
//   * with swapping on: swapped-out tables hold swap-pool ids, each once, and
//     those plus the swap pool's free count cover the swap pool exactly.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <random>
#include <vector>

#include "pa.h"

struct Snapshot {
  std::vector<int32_t> free_list, refs;
  std::map<int, std::vector<int32_t>> tables;
  std::map<int, int64_t> lens;
  std::map<int, int> swapped;
  int free_cpu = 0;
  bool operator==(const Snapshot& o) const {
    return free_list == o.free_list && refs == o.refs && tables == o.tables && lens == o.lens &&
           swapped == o.swapped && free_cpu == o.free_cpu;
  }
};

static int g_nb, g_bs, g_ncpu;

static Snapshot snap(pa_alloc* a, const std::vector<int>& live) {
  Snapshot s;
  s.free_list.resize(g_nb);
  int n = pa_alloc_free_list(a, s.free_list.data(), g_nb);
  if (n < 0) { std::printf("free_list failed\n"); std::exit(2); }
  s.free_list.resize(n);
  for (int b = 0; b < g_nb; ++b) s.refs.push_back(pa_alloc_ref(a, b));
  for (int id : live) {
    std::vector<int32_t> t(4096);
    int m = 0;
    if (pa_alloc_block_table(a, id, t.data(), (int)t.size(), &m) != PA_OK) { std::printf("table\n"); std::exit(2); }
    t.resize(m);
    s.tables[id] = t;
    int64_t len = 0;
    pa_alloc_seq_len(a, id, &len);
    s.lens[id] = len;
    s.swapped[id] = pa_alloc_is_swapped(a, id);
  }
  s.free_cpu = pa_alloc_num_free_cpu(a);
  return s;
}

static void check_invariants(const Snapshot& s) {
  std::vector<int> count(g_nb, 0), in_free(g_nb, 0), cpu_count(g_ncpu, 0);
  int on_cpu = 0;
  for (auto& kv : s.tables) {
    if ((int64_t)kv.second.size() != (s.lens.at(kv.first) + g_bs - 1) / g_bs) { std::printf("table size\n"); std::exit(3); }
    if (s.swapped.at(kv.first)) {
      for (int32_t c : kv.second) {
        if (c < 0 || c >= g_ncpu || cpu_count[c]++) { std::printf("swap id %d\n", c); std::exit(3); }
        ++on_cpu;
      }
      continue;
    }
    for (int32_t b : kv.second) count[b]++;
  }
  if (on_cpu + s.free_cpu != g_ncpu) { std::printf("swap pool %d + %d != %d\n", on_cpu, s.free_cpu, g_ncpu); std::exit(3); }
  for (int32_t b : s.free_list) {
    if (in_free[b]++) { std::printf("duplicate in free list\n"); std::exit(3); }
  }
  for (int b = 0; b < g_nb; ++b) {
    if (s.refs[b] != count[b]) { std::printf("refcount mismatch at %d\n", b); std::exit(3); }
    if ((s.refs[b] == 0) != (in_free[b] == 1)) { std::printf("free set mismatch at %d\n", b); std::exit(3); }
  }
}

int main(int argc, char** argv) {
  const int steps = argc > 1 ? std::atoi(argv[1]) : 10000;
  std::mt19937 rng(1234);
  for (int round = 0; round < 8; ++round) {
    g_nb = 4 + (int)(rng() % 60);
    const int bss[] = {1, 2, 4, 16};
    g_bs = bss[rng() % 4];
    std::vector<int32_t> order(g_nb);
    for (int i = 0; i < g_nb; ++i) order[i] = i;
    std::shuffle(order.begin(), order.end(), rng);
    pa_alloc* a = nullptr;
    if (pa_alloc_create(g_nb, g_bs, order.data(), &a) != PA_OK) return 1;
    if (round % 2 == 0 && pa_alloc_enable_prefix_caching(a) != PA_OK) return 1;
    g_ncpu = round % 4 < 2 ? 2 + (int)(rng() % 40) : 0;
    if (g_ncpu && pa_alloc_enable_swap(a, g_ncpu) != PA_OK) return 1;
    std::vector<std::vector<int32_t>> prompts(4);
    for (auto& p : prompts) {
      p.resize(1 + rng() % (4 * g_bs + 3));
      for (auto& t : p) t = (int32_t)(rng() % 3);
    }
    std::vector<int> live;
    int next = 0;
    std::vector<int32_t> slots(4096);
    for (int i = 0; i < steps / 8; ++i) {
      Snapshot before = snap(a, live);
      int op = rng() % 11, rc = PA_OK;
      int id = live.empty() ? -1 : live[rng() % live.size()];
      if (op == 0 || live.empty()) {
        rc = pa_alloc_add_seq(a, next);
        if (rc == PA_OK) live.push_back(next++);
      } else if (op <= 2) {
        rc = pa_alloc_append_slots(a, id, (int)(rng() % (3 * g_bs + 2)), slots.data());
      } else if (op == 3) {
        int64_t len = 0;
        pa_alloc_seq_len(a, id, &len);
        pa_alloc_add_seq(a, next);
        live.push_back(next);
        before = snap(a, live);
        rc = pa_alloc_share(a, next++, id, (int)(len ? rng() % (len + 1) : 0));
      } else if (op == 4) {
        int32_t pair[2];
        std::vector<int32_t> t(4096);
        int m = 0;
        pa_alloc_block_table(a, id, t.data(), 4096, &m);
        rc = pa_alloc_cow(a, id, (int)(rng() % (m + 2)) - 1, pair);
      } else if (op == 5) {
        rc = pa_alloc_free_seq(a, id);
        if (rc == PA_OK) live.erase(std::find(live.begin(), live.end(), id));
      } else if (op == 7) {
        const auto& p = prompts[rng() % prompts.size()];
        int got = -1;
        rc = pa_alloc_add_seq_cached(a, next, p.data(), (int)p.size(), rng() % 2, &got);
        if (rc == PA_OK) {
          live.push_back(next++);
          if (got < 0 || got % g_bs != 0 || got > (int)p.size() - 1) { std::printf("bad hit length\n"); return 6; }
          before = snap(a, live);
          rc = pa_alloc_append_tokens(a, next - 1, p.data() + got, (int)p.size() - got, slots.data());
        }
      } else if (op == 8) {
        std::vector<int32_t> t(rng() % (2 * g_bs + 2));
        for (auto& x : t) x = (int32_t)(rng() % 3);
        rc = pa_alloc_append_tokens(a, id, t.data(), (int)t.size(), slots.data());
      } else if (op == 9 || op == 10) {
        std::vector<int32_t> pairs(2 * 4096);
        int n = -1;
        rc = (op == 9 ? pa_alloc_swap_out : pa_alloc_swap_in)(a, id, pairs.data(), 4096, &n);
        if (rc == PA_OK) {
          const auto& t = before.tables.at(id);
          if (n != (int)t.size()) { std::printf("swap pair count\n"); return 9; }
          for (int k = 0; k < n; ++k)
            if (pairs[2 * k] != t[k]) { std::printf("swap pair source\n"); return 9; }
        }
      } else {
        rc = pa_alloc_free_seq(a, 1 << 20);  // unknown: must fail without effect
        if (rc == PA_OK) return 4;
        if (pa_alloc_ref(a, g_nb) != PA_ERR_INVALID || pa_alloc_ref(a, -1) != PA_ERR_INVALID) return 4;
      }
      Snapshot after = snap(a, live);
      if (rc != PA_OK && !(after == before)) { std::printf("failed call changed state (op %d rc %d)\n", op, rc); return 5; }
      check_invariants(after);
      pa_prefix_cache_stats pst;
      if (pa_alloc_get_prefix_cache_stats(a, &pst) != PA_OK) return 7;
      int64_t hashed = 0;
      for (int b = 0; b < g_nb; ++b) {
        int c = 0;
        if (pa_alloc_block_hash(a, b, nullptr, &c) != PA_OK) return 7;
        hashed += c;
      }
      if (hashed != pst.cached_blocks) { std::printf("hash count %lld vs map %lld\n", (long long)hashed, (long long)pst.cached_blocks); return 8; }
      if (i % 23 == 0) {
        // checkpoint: the words import into an allocator with the same state,
        // and a corrupted copy either imports or is refused, never misbehaves
        int64_t nw = 0;
        if (pa_alloc_export(a, nullptr, 0, &nw) != PA_OK || nw <= 0) return 10;
        std::vector<int64_t> w(nw);
        if (pa_alloc_export(a, w.data(), nw, &nw) != PA_OK) return 10;
        pa_alloc* c = nullptr;
        if (pa_alloc_import(w.data(), nw, &c) != PA_OK) { std::printf("import refused an export\n"); return 10; }
        if (!(snap(c, live) == after)) { std::printf("imported state differs\n"); pa_alloc_destroy(c); return 10; }
        std::vector<int64_t> w2(nw);
        int64_t nw2 = 0;
        if (pa_alloc_export(c, w2.data(), nw, &nw2) != PA_OK || nw2 != nw || w2 != w) { pa_alloc_destroy(c); return 10; }
        pa_alloc_destroy(c);
        std::vector<int64_t> x = w;
        const size_t k = (size_t)(rng() % (uint64_t)nw);
        x[k] += (int64_t)(rng() % 7) - 3;
        pa_alloc* d = nullptr;
        if (pa_alloc_import(x.data(), nw, &d) == PA_OK) pa_alloc_destroy(d);
        if (pa_alloc_import(x.data(), nw - 1, &d) == PA_OK) { std::printf("truncated words imported\n"); pa_alloc_destroy(d); return 10; }
      }
    }
    pa_alloc_destroy(a);
  }
  std::printf("ok\n");
  return 0;
}
