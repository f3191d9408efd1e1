// Shared device helpers: RoPE angles and rotation, kernel parameter blocks, tile constants.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace afx {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

// theta_i / (2 pi) for i < d/2, split as hi + lo (two fp32 words) so that pos * (hi + lo)
// can be reduced modulo one turn without losing the angle at large positions.
struct RopeFreqs {
  float hi[64];
  float lo[64];
};

// (cos, sin) of 2 pi * pos * (hi + lo). pos * hi is split exactly (two-product via fma), its
// integer part dropped, and the remaining fraction of a turn fed to sincospif.
__device__ __forceinline__ void rope_cossin(float pos, float hi, float lo, float* c, float* s) {
  const float prod = __fmul_rn(pos, hi);
  const float err = __fmaf_rn(pos, hi, -prod);
  const float frac = __fsub_rn(prod, rintf(prod));
  const float r = __fadd_rn(frac, __fmaf_rn(pos, lo, err));
  sincospif(__fmul_rn(2.0f, r), s, c);
}

// One RoPE pair (x_i, x_{i+d/2}) rotated by the angle whose (cos, sin) is (c, s).
// Operation order is fixed (no contraction freedom) so every kernel rotates bit-identically.
__device__ __forceinline__ void rot_pair(float xl, float xh, float c, float s, float& yl,
                                         float& yh) {
  yl = __fmaf_rn(xl, c, __fmul_rn(-xh, s));
  yh = __fmaf_rn(xh, c, __fmul_rn(xl, s));
}

// Rotate 8 consecutive pairs held as two 16-byte chunks of bf16 (lo half, hi half) with the
// (cos, sin) table entries cs[0..7]. sign = -1 applies the inverse rotation. The result is
// rounded to fp16 (OUT_F16, saturating at +-65504) or to bf16.
template <bool OUT_F16>
__device__ __forceinline__ void rot_chunk(uint4& lo, uint4& hi, const float2* __restrict__ cs,
                                          float sign = 1.0f) {
  uint32_t* L = reinterpret_cast<uint32_t*>(&lo);
  uint32_t* H = reinterpret_cast<uint32_t*>(&hi);
  const float4* c4 = reinterpret_cast<const float4*>(cs);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float4 t = __ldg(c4 + w);  // (cos, sin) of pairs 2w and 2w+1
    float yl0, yh0, yl1, yh1;
    rot_pair(bf16lo_to_f32(L[w]), bf16lo_to_f32(H[w]), t.x, sign * t.y, yl0, yh0);
    rot_pair(bf16hi_to_f32(L[w]), bf16hi_to_f32(H[w]), t.z, sign * t.w, yl1, yh1);
    if (OUT_F16) {
      L[w] = pack_f16x2_sat(yl0, yl1);
      H[w] = pack_f16x2_sat(yh0, yh1);
    } else {
      L[w] = pack_bf16x2(yl0, yl1);
      H[w] = pack_bf16x2(yh0, yh1);
    }
  }
}

// Variant descriptor as seen by the kernels (host fills it from attnfuse_variant).
struct VariantDev {
  int mask;    // 0 full, 1 causal, 2 window, 3 block-sparse
  int causal;  // effective causal flag (mask == causal or variant.causal)
  int window;
  int bs_block;
  const int32_t* bs_row_ptr;
  const int32_t* bs_col_idx;
  int bias;  // 0 none, 1 alibi, 2 additive
  int add_bias_bf16;
  const float* slopes;
  const void* add_bias;
  int64_t ab_s[4];
  uint8_t* visits;
};

constexpr int kBsMaxN = 65536;                       // block-sparse sequence limit
constexpr int kBsWords = kBsMaxN / 64 / 32;          // bit words per block row (blk 64)
constexpr int kTileWords = kBsMaxN / 128 / 32;       // bit words per kv-tile bitmap

}  // namespace afx
