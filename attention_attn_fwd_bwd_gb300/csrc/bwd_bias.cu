// Backward kernels with a bias combinator (AttnFuse paper §3.1 alibi / additive_bias, §4.4),
// compiled apart from the bias-free ones so the instances build in parallel.
#include "bwd_kernels.cuh"

namespace afx {

void select_bwd_bias_kernels(int d, int rk, int bias, BwdKernel* kv, BwdKernel* dq) {
  if (bias == 1) select_bwd_kernels<1>(d, rk, kv, dq);
  else select_bwd_kernels<2>(d, rk, kv, dq);
}

}  // namespace afx
