// cfg_wide_ku8.cu -- instantiation of the FFMA kernel for CfgWideKu8 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgWideKu8, kEntryWideKu8)
}  // namespace sgemm_gb300
