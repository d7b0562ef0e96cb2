// Launch accounting shared by the kernel launchers (see prof.cu).
#pragma once

#include <cuda_runtime.h>

namespace gdn {

void prof_begin(const char* name, cudaStream_t st);
void prof_end(cudaStream_t st);

// Brackets one kernel launch: counts it and, when timing is on, times it.
struct ProfScope {
    cudaStream_t st;
    ProfScope(const char* name, cudaStream_t s) : st(s) { prof_begin(name, s); }
    ~ProfScope() { prof_end(st); }
};

}  // namespace gdn

#define GDN_PROF_CAT2(a, b) a##b
#define GDN_PROF_CAT(a, b) GDN_PROF_CAT2(a, b)
// Use as: GDN_PROF("name", stream); kernel<<<...>>>(...);  (scope = enclosing block)
#define GDN_PROF(name, st) ::gdn::ProfScope GDN_PROF_CAT(_gdn_prof_, __LINE__)(name, st)
