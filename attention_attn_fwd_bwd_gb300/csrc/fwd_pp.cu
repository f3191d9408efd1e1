// Launcher of the persistent head-dim-128 forward (kernel in fwd_pp.cuh; the instances are
// compiled per operand kind in fwd_pp_none.cu, fwd_pp_fused.cu, fwd_pp_pre.cu and
// fwd_pp_fp8.cu).
#include <algorithm>
#include <mutex>

#include "fwd_pp.cuh"

namespace afx {

FwdFn fwd_pp_pick_none(int bias, int norm);
FwdFn fwd_pp_pick_fused(int bias, int norm);
FwdFn fwd_pp_pick_pre(int bias, int norm);
FwdFn fwd_pp_pick_fp8(int bias, int norm);

size_t fwd_pp_smem_size() { return kSmem; }

namespace {

// Largest number of 2-CTA clusters of this kernel that can be resident at once on the current
// device (cached per device).
int max_clusters(FwdFn fn, int dev) {
  static std::mutex mu;
  static int cache[64] = {};
  std::lock_guard<std::mutex> lk(mu);
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = sms / 2;
  }
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

}  // namespace

cudaError_t launch_fwd_pp(FwdParams p, int rope_kind, int norm, cudaStream_t stream) {
  const int bias = p.var.bias;
  FwdFn fn = rope_kind == kRopeFused        ? fwd_pp_pick_fused(bias, norm)
             : rope_kind == kRopePrerotated ? fwd_pp_pick_pre(bias, norm)
             : rope_kind == kFp8            ? fwd_pp_pick_fp8(bias, norm)
                                            : fwd_pp_pick_none(bias, norm);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  const int g = p.Hq / p.Hkv;
  p.pp_hp = (g % 4 == 0) ? 4 : (g % 2 == 0) ? 2 : 1;
  const int tq = 4 / p.pp_hp;
  const int TQ = (p.N + kBM - 1) / kBM;
  const long long units = (long long)((TQ + tq - 1) / tq) * p.B * (p.Hq / p.pp_hp);
  if (units > 0x3fffffff) return cudaErrorInvalidValue;
  const long long cl = std::min<long long>(units, max_clusters(fn, dev));
  p.pp_clusters = static_cast<int>(std::max<long long>(cl, 1));
  fn<<<2 * p.pp_clusters, kThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace afx
