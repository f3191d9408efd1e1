// Instances of the persistent head-dim-128 forward (fwd_pp.cuh) for e4m3 inputs (kFp8).
#include "fwd_pp.cuh"

namespace afx {

FwdFn fwd_pp_pick_fp8(int bias, int norm) { return fwd_pp_pick<kFp8>(bias, norm); }

}  // namespace afx
