// Instances of the persistent head-dim-128 forward (fwd_pp.cuh) for e4m3 inputs (kFp8), and
// the pass that widens e4m3 V to the bf16 operand of the P V MMAs.
#include <algorithm>

#include "fwd_pp.cuh"

namespace afx {

FwdFn fwd_pp_pick_fp8(int bias, int norm) { return fwd_pp_pick<kFp8, 128>(bias, norm); }

namespace {

// out[b, h, n, :] = bf16(e4m3(v[b, h, n, :])), exactly (every e4m3 value is a bf16 value); one
// thread per 16 values (16 input bytes, 32 output bytes), rows of d values.
__global__ void widen_e4m3_kernel(const uint8_t* __restrict__ v, int64_t sb, int64_t sh, int64_t sn,
                                  uint16_t* __restrict__ out, int H, int N, int d, int64_t chunks) {
  const int cpr = d / 16;  // 16-value chunks per row
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < chunks;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = static_cast<int>(idx % cpr);
    const int64_t row = idx / cpr;  // (b * H + h) * N + n
    const int n = static_cast<int>(row % N);
    const int64_t bh = row / N;
    const int h = static_cast<int>(bh % H);
    const int64_t b = bh / H;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(v + b * sb + h * sh + (int64_t)n * sn + c * 16));
    uint4 lo, hi;
    e4m3x16_to_bf16(x, lo, hi);
    uint4* dst = reinterpret_cast<uint4*>(out + row * d + c * 16);
    __stcg(dst, lo);
    __stcg(dst + 1, hi);
  }
}

}  // namespace

cudaError_t launch_widen_e4m3(const void* v, const int64_t* strides, void* out, int B, int H, int N,
                              int d, cudaStream_t stream) {
  const int64_t chunks = static_cast<int64_t>(B) * H * N * (d / 16);
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<int64_t>((chunks + threads - 1) / threads, 152 * 16));
  widen_e4m3_kernel<<<blocks, threads, 0, stream>>>(static_cast<const uint8_t*>(v), strides[0],
                                                    strides[1], strides[2],
                                                    static_cast<uint16_t*>(out), H, N, d, chunks);
  return cudaGetLastError();
}

}  // namespace afx
