// cfg_wide_bk32.cu -- instantiation of the FFMA kernel for CfgWideBk32 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgWideBk32, kEntryWideBk32)
}  // namespace sgemm_gb300
