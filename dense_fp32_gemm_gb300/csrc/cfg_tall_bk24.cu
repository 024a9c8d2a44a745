// cfg_tall_bk24.cu -- instantiation of the FFMA kernel for CfgTallBk24 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgTallBk24, kEntryTallBk24)
}  // namespace sgemm_gb300
