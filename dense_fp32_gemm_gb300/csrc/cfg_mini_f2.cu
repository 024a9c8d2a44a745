// cfg_mini_f2.cu -- instantiation of the FFMA kernel for CfgMiniF2 (one translation
// unit per configuration so that the library compiles in parallel). One of
// the tuned configurations: built for every operand layout.
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY_ALL_LAYOUTS(CfgMiniF2, kEntryMiniF2)
}  // namespace sgemm_gb300
