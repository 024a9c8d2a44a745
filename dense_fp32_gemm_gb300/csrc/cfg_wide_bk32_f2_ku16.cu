// cfg_wide_bk32_f2_ku16.cu -- instantiation of the FFMA kernel for CfgWideBk32F2Ku16 (one translation
// unit per configuration so that the library compiles in parallel). One of
// the tuned configurations: built for every operand layout.
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY_ALL_LAYOUTS(CfgWideBk32F2Ku16, kEntryWideBk32F2Ku16)
}  // namespace sgemm_gb300
