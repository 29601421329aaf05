// Launch accounting and the opt-in launch-timing facility (bn_profile_*):
// when on, every kernel this thread launches through the library is bracketed
// by a pair of CUDA events on its stream and recorded with its algorithmic
// FLOPs and bytes.
#include <vector>

#include "../../include/boostblk.h"
#include "gemm.h"

namespace bn {
namespace {

struct Rec {
  int kind, epi;
  double flops, bytes;
  cudaEvent_t a, b;
};

struct Prof {
  bool on = false;
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;  // events reused across sessions
  size_t used = 0;
  cudaEvent_t pending = nullptr;
  cudaEvent_t next_event() {
    if (used == pool.size()) {
      cudaEvent_t e = nullptr;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[used++];
  }
};

thread_local Prof g_prof;

}  // namespace

bool prof_active() { return g_prof.on; }

void prof_start(Ctx& c) {
  if (!g_prof.on) return;
  g_prof.pending = g_prof.next_event();
  if (g_prof.pending) cudaEventRecord(g_prof.pending, c.stream);
}

void note_launch(Ctx& c, int kind, int epi, double flops, double bytes) {
  ++c.launches;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess && c.err == cudaSuccess) c.err = e;
  if (!g_prof.on || g_prof.pending == nullptr) return;
  cudaEvent_t b = g_prof.next_event();
  if (b == nullptr) return;
  cudaEventRecord(b, c.stream);
  g_prof.recs.push_back(Rec{kind, epi, flops, bytes, g_prof.pending, b});
  g_prof.pending = nullptr;
}

}  // namespace bn

using namespace bn;

extern "C" bn_status bn_profile_start(void) {
  g_prof.on = true;
  g_prof.recs.clear();
  g_prof.used = 0;
  g_prof.pending = nullptr;
  return BN_OK;
}

extern "C" int bn_profile_stop(bn_launch_record* out, int max_records) {
  g_prof.on = false;
  const int n = static_cast<int>(g_prof.recs.size());
  for (int i = 0; i < n && i < max_records && out != nullptr; ++i) {
    const Rec& r = g_prof.recs[i];
    float ms = -1.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess) cudaEventElapsedTime(&ms, r.a, r.b);
    out[i].kernel = r.kind;
    out[i].epi = r.epi;
    out[i].flops = r.flops;
    out[i].bytes = r.bytes;
    out[i].ms = ms;
  }
  g_prof.recs.clear();
  g_prof.used = 0;
  return n;
}
