// cfg_square_bk32.cu -- instantiation of the FFMA kernel for CfgSquareBk32 (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgSquareBk32, kEntrySquareBk32)
}  // namespace sgemm_gb300
