// cfg_mini_f2_ku16.cu -- instantiation of the FFMA kernel for CfgMiniF2Ku16 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgMiniF2Ku16, kEntryMiniF2Ku16)
}  // namespace sgemm_gb300
