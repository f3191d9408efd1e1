// Launcher of the persistent forward (kernel in fwd_pp.cuh; the instances are compiled per
// operand kind and head dim in fwd_pp_{none,fused,pre,fp8}.cu (head dim 128) and
// fwd_pp64_{none,fused,pre}.cu (head dim 64)).
#include <algorithm>
#include <mutex>

#include "fwd_pp.cuh"

namespace afx {

FwdFn fwd_pp_pick_none(int bias, int norm);
FwdFn fwd_pp_pick_fused(int bias, int norm);
FwdFn fwd_pp_pick_pre(int bias, int norm);
FwdFn fwd_pp_pick_fp8(int bias, int norm);
FwdFn fwd_pp64_pick_none(int bias, int norm);
FwdFn fwd_pp64_pick_fused(int bias, int norm);
FwdFn fwd_pp64_pick_pre(int bias, int norm);

size_t fwd_pp_smem_size(int d) { return d == 64 ? pp_smem<64>() : pp_smem<128>(); }

namespace {

// Largest number of 2-CTA clusters of a kernel instance that can be resident at once on the
// current device (cached per device and head dim).
int max_clusters(FwdFn fn, size_t smem, int d, int dev) {
  static std::mutex mu;
  static int cache[2][64] = {};
  std::lock_guard<std::mutex> lk(mu);
  const int di = d == 64 ? 1 : 0;
  if (dev >= 0 && dev < 64 && cache[di][dev] > 0) return cache[di][dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  // at most one CTA per SM: each CTA allocates all 512 columns of its SM's tensor memory
  n = std::min(n, sms / 2);
  if (dev >= 0 && dev < 64) cache[di][dev] = n;
  return n;
}

}  // namespace

cudaError_t launch_fwd_pp(FwdParams p, int d, int rope_kind, int norm, cudaStream_t stream) {
  const int bias = p.var.bias;
  FwdFn fn = nullptr;
  if (d == 64) {
    if (rope_kind == kFp8) return cudaErrorInvalidValue;
    fn = rope_kind == kRopeFused        ? fwd_pp64_pick_fused(bias, norm)
         : rope_kind == kRopePrerotated ? fwd_pp64_pick_pre(bias, norm)
                                        : fwd_pp64_pick_none(bias, norm);
  } else {
    fn = rope_kind == kRopeFused        ? fwd_pp_pick_fused(bias, norm)
         : rope_kind == kRopePrerotated ? fwd_pp_pick_pre(bias, norm)
         : rope_kind == kFp8            ? fwd_pp_pick_fp8(bias, norm)
                                        : fwd_pp_pick_none(bias, norm);
  }
  const size_t smem = fwd_pp_smem_size(d);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  const int g = p.Hq / p.Hkv;
  p.pp_hp = (g % 4 == 0) ? 4 : (g % 2 == 0) ? 2 : 1;
  const int tq = 4 / p.pp_hp;
  const int TQ = (p.N + kBM - 1) / kBM;
  const long long units = (long long)((TQ + tq - 1) / tq) * p.B * (p.Hq / p.pp_hp);
  if (units > 0x3fffffff) return cudaErrorInvalidValue;
  const long long cl = std::min<long long>(units, max_clusters(fn, smem, d, dev));
  p.pp_clusters = static_cast<int>(std::max<long long>(cl, 1));
  fn<<<2 * p.pp_clusters, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace afx
