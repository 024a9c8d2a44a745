// cfg_wide_bk32_ku8.cu -- instantiation of the FFMA kernel for CfgWideBk32Ku8 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgWideBk32Ku8, kEntryWideBk32Ku8)
}  // namespace sgemm_gb300
