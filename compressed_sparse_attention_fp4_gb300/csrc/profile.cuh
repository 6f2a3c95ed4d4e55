// profile.cuh -- optional kernel timing: while enabled, every kernel launch of
// the library is bracketed with CUDA events on its stream (host side only).
#pragma once

#include <cuda_runtime.h>

namespace csa2 {
namespace prof {

struct Token {
  int slot;          // -1: profiling off
};

Token begin(cudaStream_t st);
void end(cudaStream_t st, const char* kernel, Token t);

// Brackets one launch statement.
#define CSA2_PROFILED(stream, name, launch)              \
  do {                                                   \
    ::csa2::prof::Token tok_ = ::csa2::prof::begin(stream); \
    launch;                                              \
    ::csa2::prof::end(stream, name, tok_);               \
  } while (0)

}  // namespace prof
}  // namespace csa2
