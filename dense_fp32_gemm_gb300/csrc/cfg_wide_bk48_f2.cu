// cfg_wide_bk48_f2.cu -- instantiation of the FFMA kernel for CfgWideBk48F2 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgWideBk48F2, kEntryWideBk48F2)
}  // namespace sgemm_gb300
