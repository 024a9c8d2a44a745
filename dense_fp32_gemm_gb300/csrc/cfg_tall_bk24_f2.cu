// cfg_tall_bk24_f2.cu -- instantiation of the FFMA kernel for CfgTallBk24F2 (one translation
// unit per configuration so that the library compiles in parallel). One of
// the tuned configurations: built for every operand layout.
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY_ALL_LAYOUTS(CfgTallBk24F2, kEntryTallBk24F2)
}  // namespace sgemm_gb300
