// Head-dim-64 instances of the persistent forward (fwd_pp.cuh) for RoPE kind kRopePrerotated.
#include "fwd_pp.cuh"

namespace afx {

FwdFn fwd_pp64_pick_pre(int bias, int norm) { return fwd_pp_pick<kRopePrerotated, 64>(bias, norm); }

}  // namespace afx
