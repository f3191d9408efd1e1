// Backward launch (AttnFuse paper §4.4): the D = rowsum(dO * O) preprocess kernel, then the
// dK/dV and dQ kernels of bwd_kernels.cuh (bias-free instances here, bias instances in
// bwd_bias.cu).
#include "bwd_kernels.cuh"

namespace afx {

// ---------------------------------------------------------------------------------------------
// D = rowsum(dO * O)
// ---------------------------------------------------------------------------------------------
__global__ void bwd_pre_kernel(const __grid_constant__ BwdParams p) {
  const int tpr = p.d / 8;  // threads per row
  const int64_t rows = (int64_t)p.B * p.Hq * p.N;
  const int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / tpr;
  const int c = threadIdx.x % tpr;
  float acc = 0.f;
  if (row < rows) {
    const int n = static_cast<int>(row % p.N);
    const int64_t bh = row / p.N;
    const int h = static_cast<int>(bh % p.Hq);
    const int64_t b = bh / p.Hq;
    const uint4 o = *reinterpret_cast<const uint4*>(p.o + b * p.o_s[0] + h * p.o_s[1] + n * p.o_s[2] + c * 8);
    const uint4 g = *reinterpret_cast<const uint4*>(p.dout + b * p.do_s[0] + h * p.do_s[1] + n * p.do_s[2] + c * 8);
    const uint32_t* ow = reinterpret_cast<const uint32_t*>(&o);
    const uint32_t* gw = reinterpret_cast<const uint32_t*>(&g);
#pragma unroll
    for (int w = 0; w < 4; ++w)
      acc += bf16lo_to_f32(ow[w]) * bf16lo_to_f32(gw[w]) + bf16hi_to_f32(ow[w]) * bf16hi_to_f32(gw[w]);
  }
  for (int off = tpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && c == 0) p.Dvec[row] = acc;
}

// ---------------------------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------------------------
cudaError_t launch_bwd(const BwdParams& p, int rk, cudaStream_t stream) {
  const int d = p.d;
  {
    const int64_t threads = (int64_t)p.B * p.Hq * p.N * (d / 8);
    const int block = 256;
    bwd_pre_kernel<<<static_cast<int>((threads + block - 1) / block), block, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int T = (p.N + kT - 1) / kT;
  BwdKernel kv = nullptr, dq = nullptr;
  if (p.var.bias == 0) select_bwd_kernels<0>(d, rk, &kv, &dq);
  else select_bwd_bias_kernels(d, rk, p.var.bias, &kv, &dq);
  const size_t s1 = kv_smem_bytes(d), s2 = dq_smem_bytes(d);
  cudaError_t e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(dq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
  if (e != cudaSuccess) return e;
  kv<<<T * p.B * p.Hkv, kBwdThreads, s1, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dq<<<T * p.B * p.Hq, kDqThreads, s2, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace afx

