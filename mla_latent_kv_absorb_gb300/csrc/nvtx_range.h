// nvtx_range.h -- NVTX ranges around the library's entry points, for profilers that show them
// (Nsight Systems, Nsight Compute's range filters).  Off unless the environment has MLA_NVTX=1
// (read once per process): when off, no NVTX function is called at all.
#pragma once
#include <nvtx3/nvToolsExt.h>

#include <cstdlib>

namespace mla {

inline bool nvtx_enabled()
{
    static const bool on = [] {
        const char* v = std::getenv("MLA_NVTX");
        return v != nullptr && v[0] == '1' && v[1] == '\0';
    }();
    return on;
}

// Scoped range named after the entry point: pushed on construction, popped on return.
class NvtxRange {
public:
    explicit NvtxRange(const char* name) : on_(nvtx_enabled())
    {
        if (on_) nvtxRangePushA(name);
    }
    ~NvtxRange()
    {
        if (on_) nvtxRangePop();
    }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;

private:
    bool on_;
};

}  // namespace mla
