// tune.cpp — the autotune cache (see tune.h).
#include "tune.h"

#include <cstdio>
#include <cstdlib>
#include <fstream>
#include <map>
#include <mutex>
#include <sstream>
#include <tuple>

namespace fxtx {
namespace {

struct Entry {
  int choice = 0;
  int candidates = 0;
  double best_us = 0.0, model_us = 0.0;
};

std::mutex g_mu;
std::map<TuneKey, Entry> g_cache;
int g_mode = -1;  // -1: not yet read from the environment

int mode_locked() {
  if (g_mode < 0) {
    const char* s = getenv("FXTX_AUTOTUNE");
    g_mode = (s && s[0] == '1') ? 1 : 0;
  }
  return g_mode;
}

}  // namespace

bool TuneKey::operator<(const TuneKey& o) const {
  return std::tie(kind, elem, m, n, nnz, ld, flags, sm_count) <
         std::tie(o.kind, o.elem, o.m, o.n, o.nnz, o.ld, o.flags, o.sm_count);
}

int tune_mode() {
  std::lock_guard<std::mutex> lock(g_mu);
  return mode_locked();
}

void tune_set_mode(int mode) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_mode = mode ? 1 : 0;
}

bool tune_lookup(const TuneKey& key, int* choice) {
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_cache.find(key);
  if (it == g_cache.end()) return false;
  *choice = it->second.choice;
  return true;
}

void tune_store(const TuneKey& key, int choice, int candidates, double best_us, double model_us) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_cache[key] = Entry{choice, candidates, best_us, model_us};
}

int64_t tune_entries() {
  std::lock_guard<std::mutex> lock(g_mu);
  return (int64_t)g_cache.size();
}

void tune_clear() {
  std::lock_guard<std::mutex> lock(g_mu);
  g_cache.clear();
}

bool tune_save(const std::string& path) {
  std::lock_guard<std::mutex> lock(g_mu);
  std::ofstream f(path);
  if (!f) return false;
  f << "# kind elem m n nnz ld flags sm_count choice candidates best_us model_us\n";
  for (const auto& kv : g_cache) {
    const TuneKey& k = kv.first;
    const Entry& e = kv.second;
    char line[256];
    snprintf(line, sizeof line, "%d %d %lld %lld %lld %lld %d %d %d %d %.3f %.3f\n", k.kind, k.elem, (long long)k.m,
             (long long)k.n, (long long)k.nnz, (long long)k.ld, k.flags, k.sm_count, e.choice, e.candidates,
             e.best_us, e.model_us);
    f << line;
  }
  return (bool)f;
}

bool tune_load(const std::string& path) {
  std::ifstream f(path);
  if (!f) return false;
  std::map<TuneKey, Entry> loaded;
  std::string line;
  while (std::getline(f, line)) {
    if (line.empty() || line[0] == '#') continue;
    std::istringstream in(line);
    TuneKey k;
    Entry e;
    long long m, n, nnz, ld;
    if (!(in >> k.kind >> k.elem >> m >> n >> nnz >> ld >> k.flags >> k.sm_count >> e.choice >> e.candidates >>
          e.best_us >> e.model_us))
      return false;
    std::string rest;
    if (in >> rest) return false;
    if ((k.kind != 0 && k.kind != 1) || m < 0 || n < 0 || nnz < 0 || ld < 0 || e.choice < 0 || e.candidates < 1 ||
        e.choice >= e.candidates)
      return false;
    k.m = m; k.n = n; k.nnz = nnz; k.ld = ld;
    loaded[k] = e;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  g_cache.swap(loaded);
  return true;
}

}  // namespace fxtx
