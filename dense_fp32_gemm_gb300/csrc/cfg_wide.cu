// cfg_wide.cu -- instantiation of the FFMA kernel for CfgWide (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgWide, kEntryWide)
}  // namespace sgemm_gb300
