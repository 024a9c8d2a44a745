// cfg_wide_bk16_f2.cu -- instantiation of the FFMA kernel for CfgWideBk16F2 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgWideBk16F2, kEntryWideBk16F2)
}  // namespace sgemm_gb300
