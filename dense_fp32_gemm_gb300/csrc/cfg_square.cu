// cfg_square.cu -- instantiation of the FFMA kernel for CfgSquare (one translation
// unit per configuration so that the library compiles in parallel).
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY(CfgSquare, kEntrySquare)
}  // namespace sgemm_gb300
