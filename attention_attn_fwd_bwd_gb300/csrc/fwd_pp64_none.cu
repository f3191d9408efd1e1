// Head-dim-64 instances of the persistent forward (fwd_pp.cuh) for RoPE kind kRopeNone.
#include "fwd_pp.cuh"

namespace afx {

FwdFn fwd_pp64_pick_none(int bias, int norm) { return fwd_pp_pick<kRopeNone, 64>(bias, norm); }

}  // namespace afx
