// cfg_wide_bk48_ku8.cu -- instantiation of the FFMA kernel for CfgWideBk48Ku8 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgWideBk48Ku8, kEntryWideBk48Ku8)
}  // namespace sgemm_gb300
