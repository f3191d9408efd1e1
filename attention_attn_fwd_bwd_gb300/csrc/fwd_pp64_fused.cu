// Head-dim-64 instances of the persistent forward (fwd_pp.cuh) for RoPE kind kRopeFused.
#include "fwd_pp.cuh"

namespace afx {

FwdFn fwd_pp64_pick_fused(int bias, int norm) { return fwd_pp_pick<kRopeFused, 64>(bias, norm); }

}  // namespace afx
