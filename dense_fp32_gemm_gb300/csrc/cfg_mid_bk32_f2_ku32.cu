// cfg_mid_bk32_f2_ku32.cu -- instantiation of the FFMA kernel for CfgMidBk32F2Ku32 (one
// translation unit per configuration so that the library compiles in
// parallel). A candidate of the tuner: built for every operand layout.
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY_ALL_LAYOUTS(CfgMidBk32F2Ku32, kEntryMidBk32F2Ku32)
}  // namespace sgemm_gb300
