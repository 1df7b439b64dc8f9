// tune.h — the one-shot autotune cache over the launch model's candidates.
//
// "On optimizing machine learning workloads via kernel fusion" (abstract) picks launch
// parameters with an analytical model; this cache optionally replaces the model's pick
// by the fastest of its candidate launches, timed once per call shape on the device.
// Off by default (the model alone decides); on with fxtx_autotune_set(1) or the
// environment variable FXTX_AUTOTUNE=1.
#pragma once

#include <cstdint>
#include <string>

namespace fxtx {

// The shape of one call, as far as launch parameters depend on it.
struct TuneKey {
  int kind = 0;   // 0 dense, 1 CSR
  int elem = 0;   // bytes of X's elements
  int64_t m = 0, n = 0, nnz = 0, ld = 0;
  int flags = 0;  // dense: bit 0 tensor copies possible (tile), bit 1 bulk copies possible (narrow)
  int sm_count = 0;
  bool operator<(const TuneKey& o) const;
};

int tune_mode();
void tune_set_mode(int mode);
// The cached candidate index for `key`, if any.
bool tune_lookup(const TuneKey& key, int* choice);
void tune_store(const TuneKey& key, int choice, int candidates, double best_us, double model_us);
int64_t tune_entries();
void tune_clear();
// Text file, one entry per line: kind elem m n nnz ld flags sm_count choice candidates best_us model_us.
// load() replaces the cache; false (cache unchanged) on a missing file or a malformed line.
bool tune_save(const std::string& path);
bool tune_load(const std::string& path);

}  // namespace fxtx
