// cfg_tall.cu -- instantiation of the FFMA kernel for CfgTall (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgTall, kEntryTall)
}  // namespace sgemm_gb300
