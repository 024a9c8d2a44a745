// cfg_square_bk32_f2.cu -- instantiation of the FFMA kernel for CfgSquareBk32F2 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgSquareBk32F2, kEntrySquareBk32F2)
}  // namespace sgemm_gb300
