// cfg_flat_bk24_f2_ku24.cu -- instantiation of the FFMA kernel for CfgFlatBk24F2Ku24 (one translation
// unit per configuration so that the library compiles in parallel). A
// candidate of the tuner: built for every operand layout.
#include "launch.cuh"

namespace sgemm_gb300 {
SGEMM_GB300_DEFINE_ENTRY_ALL_LAYOUTS(CfgFlatBk24F2Ku24, kEntryFlatBk24F2Ku24)
}  // namespace sgemm_gb300
