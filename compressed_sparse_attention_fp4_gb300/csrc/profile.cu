// profile.cu -- kernel timing records behind csa2_profile_enable / _read.
//
// Not for use while a stream is being captured into a CUDA graph: the events
// would become graph nodes.  Records are kept until the next enable.
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "profile.cuh"

namespace csa2 {
namespace prof {
namespace {

struct Rec {
  std::string kernel;
  cudaEvent_t e0, e1;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pending;      // begin events of open launches

void clear_locked() {
  for (auto& r : g_recs) {
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  g_recs.clear();
  for (auto e : g_pending)
    if (e) cudaEventDestroy(e);
  g_pending.clear();
}

}  // namespace

Token begin(cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return Token{-1};
  cudaEvent_t e;
  if (cudaEventCreate(&e) != cudaSuccess) return Token{-1};
  cudaEventRecord(e, st);
  g_pending.push_back(e);
  return Token{int(g_pending.size()) - 1};
}

void end(cudaStream_t st, const char* kernel, Token t) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || t.slot < 0 || t.slot >= int(g_pending.size()) || !g_pending[t.slot]) return;
  cudaEvent_t e1;
  if (cudaEventCreate(&e1) != cudaSuccess) return;
  cudaEventRecord(e1, st);
  g_recs.push_back(Rec{kernel, g_pending[t.slot], e1});
  g_pending[t.slot] = nullptr;
}

}  // namespace prof
}  // namespace csa2

extern "C" {

csa2_status csa2_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(csa2::prof::g_mu);
  csa2::prof::clear_locked();
  csa2::prof::g_on = on != 0;
  return CSA2_OK;
}

csa2_status csa2_profile_read(csa2_kernel_time* out, int32_t max_entries, int32_t* n_entries) {
  if (!n_entries || max_entries < 0 || (max_entries > 0 && !out)) return CSA2_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(csa2::prof::g_mu);
  std::vector<csa2_kernel_time> acc;
  for (auto& r : csa2::prof::g_recs) {
    if (cudaEventSynchronize(r.e1) != cudaSuccess) return CSA2_ERR_CUDA;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, r.e0, r.e1) != cudaSuccess) return CSA2_ERR_CUDA;
    csa2_kernel_time* slot = nullptr;
    for (auto& k : acc)
      if (r.kernel == k.name) slot = &k;
    if (!slot) {
      acc.push_back(csa2_kernel_time{});
      slot = &acc.back();
      std::strncpy(slot->name, r.kernel.c_str(), sizeof(slot->name) - 1);
    }
    slot->launches += 1;
    slot->total_ms += ms;
  }
  *n_entries = int32_t(acc.size());
  for (int32_t i = 0; i < int32_t(acc.size()) && i < max_entries; ++i) out[i] = acc[i];
  return CSA2_OK;
}

}  // extern "C"
