// autotune.cu -- opt-in tile autotuning with a disk cache.
//
// "Add FlyDSL grouped groupwise FP8 GEMM for ROCm" (Tile selection): candidate tiles are
// timed once per shape class and the winner is persisted to disk, behind an environment
// gate, with a fixed choice when the gate is off; tuning never happens during graph
// capture.  Here the shape class of the grouped GEMM is (nextPow2(total_M), N, K, G) and
// the candidates are its two tile widths; the dense GEMM's class is (nextPow2(M), N, K,
// layout, formats) and its candidates are the SM-pair and the single-CTA kernels.
//
// The gate is BSMMA_AUTOTUNE=1 (or bsmma_autotune_configure); the cache file is
// BSMMA_AUTOTUNE_CACHE, else $XDG_CACHE_HOME/bsmma/autotune.txt, else
// $HOME/.cache/bsmma/autotune.txt.  One line per shape class: "<key> <choice>".
#include <cuda_runtime.h>
#include <sys/stat.h>

#include <cerrno>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <map>
#include <mutex>
#include <sstream>
#include <string>
#include <vector>

#include "internal.h"

namespace bsmma {
namespace {

struct Tuner {
  std::mutex mu;
  bool configured = false;
  bool enabled = false;
  std::string path;
  std::map<std::string, int> choices;

  void load_file() {
    choices.clear();
    std::ifstream in(path);
    std::string line;
    while (std::getline(in, line)) {
      const size_t sp = line.find_last_of(' ');
      if (sp == std::string::npos || sp == 0) continue;
      char* end = nullptr;
      const long v = std::strtol(line.c_str() + sp + 1, &end, 10);
      if (end == line.c_str() + sp + 1) continue;
      choices[line.substr(0, sp)] = static_cast<int>(v);
    }
  }

  // Caller holds mu.
  void configure_locked(int enable, const char* cache_path) {
    if (enable < 0) {
      const char* e = std::getenv("BSMMA_AUTOTUNE");
      enabled = e && std::strcmp(e, "0") != 0 && e[0] != '\0';
    } else {
      enabled = enable != 0;
    }
    if (cache_path && cache_path[0]) {
      path = cache_path;
    } else if (const char* p = std::getenv("BSMMA_AUTOTUNE_CACHE")) {
      path = p;
    } else if (const char* x = std::getenv("XDG_CACHE_HOME")) {
      path = std::string(x) + "/bsmma/autotune.txt";
    } else if (const char* h = std::getenv("HOME")) {
      path = std::string(h) + "/.cache/bsmma/autotune.txt";
    } else {
      path.clear();
    }
    load_file();
    configured = true;
  }

  void ensure() {
    if (!configured) configure_locked(-1, nullptr);
  }

  void store(const std::string& key, int choice) {
    choices[key] = choice;
    if (path.empty()) return;
    // create the parent directories, then append one line
    for (size_t i = 1; i < path.size(); ++i)
      if (path[i] == '/') mkdir(path.substr(0, i).c_str(), 0755);
    if (FILE* f = std::fopen(path.c_str(), "a")) {
      std::fprintf(f, "%s %d\n", key.c_str(), choice);
      std::fclose(f);
    }
  }
};

Tuner& tuner() {
  static Tuner t;
  return t;
}

bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return true;   // be conservative
  return cs != cudaStreamCaptureStatusNone;
}

}  // namespace

int64_t next_pow2(int64_t v) {
  int64_t p = 1;
  while (p < v) p <<= 1;
  return v <= 0 ? 0 : p;
}

int autotune_cached(const std::string& key) {
  Tuner& t = tuner();
  std::lock_guard<std::mutex> g(t.mu);
  t.ensure();
  if (!t.enabled) return -1;
  auto it = t.choices.find(key);
  return it == t.choices.end() ? -1 : it->second;
}

int autotune_pick(const std::string& key, const std::vector<int>& candidates, int fallback,
                  cudaStream_t stream, const std::function<bsmma_status(int)>& launch) {
  Tuner& t = tuner();
  {
    std::lock_guard<std::mutex> g(t.mu);
    t.ensure();
    if (!t.enabled) return fallback;
    auto it = t.choices.find(key);
    if (it != t.choices.end()) return it->second;
  }
  if (candidates.size() < 2 || capturing(stream)) return fallback;
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return fallback;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return fallback;
  }
  int best = fallback;
  float best_ms = 0.f;
  for (int c : candidates) {
    if (launch(c) != BSMMA_OK) continue;                  // warm-up (first-launch set-up)
    cudaEventRecord(e0, stream);
    const bsmma_status st = launch(c);
    cudaEventRecord(e1, stream);
    if (st != BSMMA_OK || cudaEventSynchronize(e1) != cudaSuccess) continue;
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    if (best_ms == 0.f || ms < best_ms) {
      best_ms = ms;
      best = c;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (best_ms > 0.f) {
    std::lock_guard<std::mutex> g(t.mu);
    t.store(key, best);
  }
  return best;
}

}  // namespace bsmma

using namespace bsmma;

extern "C" {

bsmma_status bsmma_autotune_configure(int enable, const char* cache_path) {
  if (enable < -1 || enable > 1) return BSMMA_ERR_INVALID_ARG;
  Tuner& t = tuner();
  std::lock_guard<std::mutex> g(t.mu);
  t.configure_locked(enable, cache_path);
  return BSMMA_OK;
}

int bsmma_autotune_lookup(const char* key) {
  if (!key) return -1;
  Tuner& t = tuner();
  std::lock_guard<std::mutex> g(t.mu);
  t.ensure();
  auto it = t.choices.find(key);
  return it == t.choices.end() ? -1 : it->second;
}

}  // extern "C"
