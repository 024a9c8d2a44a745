// cfg_flat_bk24_f2.cu -- instantiation of the FFMA kernel for CfgFlatBk24F2 (one translation
// unit per configuration so that the library compiles in parallel). One of
// the tuned configurations: built for every operand layout.
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY_ALL_LAYOUTS(CfgFlatBk24F2, kEntryFlatBk24F2)
}  // namespace sgemm_gb300
