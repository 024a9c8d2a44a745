// cfg_pages.cu -- instantiation of the FFMA kernel for CfgPages (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgPages, kEntryPages)
}  // namespace sgemm_gb300
