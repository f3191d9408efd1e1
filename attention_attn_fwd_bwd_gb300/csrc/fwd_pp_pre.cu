// Instances of the persistent head-dim-128 forward (fwd_pp.cuh) for RoPE kind kRopePrerotated.
#include "fwd_pp.cuh"

namespace afx {

FwdFn fwd_pp_pick_pre(int bias, int norm) { return fwd_pp_pick<kRopePrerotated, 128>(bias, norm); }

}  // namespace afx
