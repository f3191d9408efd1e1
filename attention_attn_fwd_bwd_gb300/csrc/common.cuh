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

// Rotate 8 consecutive pairs held as two 16-byte chunks of bf16 (lo half, hi half) by the
// angles whose (cos, sin) are (c[e], s[e]). The result is rounded to fp16 (OUT_F16,
// saturating at +-65504) or to bf16.
template <bool OUT_F16>
__device__ __forceinline__ void rot_chunk_cs(uint4& lo, uint4& hi, const float (&c)[8],
                                             const float (&s)[8]) {
  uint32_t* L = reinterpret_cast<uint32_t*>(&lo);
  uint32_t* H = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float yl0, yh0, yl1, yh1;
    rot_pair(bf16lo_to_f32(L[w]), bf16lo_to_f32(H[w]), c[2 * w], s[2 * w], yl0, yh0);
    rot_pair(bf16hi_to_f32(L[w]), bf16hi_to_f32(H[w]), c[2 * w + 1], s[2 * w + 1], yl1, yh1);
    if (OUT_F16) {
      L[w] = pack_f16x2_sat(yl0, yl1);
      H[w] = pack_f16x2_sat(yh0, yh1);
    } else {
      L[w] = pack_bf16x2(yl0, yl1);
      H[w] = pack_bf16x2(yh0, yh1);
    }
  }
}

// fp16 range of the rotating modes: running per-half maximum of |x| as fp16 bits (the bit
// patterns of non-negative halves order like their values, NaN above infinity), and the status
// bit raised once a rotated value reached 65504 (cvt.rn.satfinite saturates there) or is not
// finite.
__device__ __forceinline__ uint32_t f16_absmax(uint32_t acc, uint32_t w) {
  return __vmaxu2(acc, w & 0x7FFF7FFFu);
}
__device__ __forceinline__ uint32_t f16_absmax(uint32_t acc, const uint4& w) {
  return f16_absmax(f16_absmax(f16_absmax(f16_absmax(acc, w.x), w.y), w.z), w.w);
}
__device__ __forceinline__ void report_f16_range(int* status, uint32_t acc) {
  if (status && ((acc & 0xFFFFu) >= 0x7BFFu || (acc >> 16) >= 0x7BFFu))
    atomicOr(status, kDevF16Range);
}

// Packed-pair version of rot_chunk_cs for 8 pairs with (cos, sin) held as 4 packed pairs each
// (c2[w] = (c[2w], c[2w+1])) and ns2 = -s2. Per lane it performs exactly rot_pair's
// operations, so the results are bit-identical to rot_chunk_cs.
template <bool OUT_F16>
__device__ __forceinline__ void rot_chunk_cs2(uint4& lo, uint4& hi, const uint64_t (&c2)[4],
                                              const uint64_t (&s2)[4],
                                              const uint64_t (&ns2)[4]) {
  uint32_t* L = reinterpret_cast<uint32_t*>(&lo);
  uint32_t* H = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint64_t xl = bf16x2_to_f2(L[w]), xh = bf16x2_to_f2(H[w]);
    const uint64_t yl = fma2(xl, c2[w], mul2(xh, ns2[w]));   // xl c + (-xh) s
    const uint64_t yh = fma2(xh, c2[w], mul2(xl, s2[w]));    // xh c + xl s
    if (OUT_F16) {
      L[w] = pack_f16x2_sat(f2_lo(yl), f2_hi(yl));
      H[w] = pack_f16x2_sat(f2_lo(yh), f2_hi(yh));
    } else {
      L[w] = pack_bf16x2(f2_lo(yl), f2_hi(yl));
      H[w] = pack_bf16x2(f2_lo(yh), f2_hi(yh));
    }
  }
}

// Packed angle-addition step, lane-wise identical to advance_cs8 (rot_pair on (c, s) with
// (wc, ws)); also keeps ns = -s exactly.
__device__ __forceinline__ void advance_cs2(uint64_t (&c2)[4], uint64_t (&s2)[4],
                                            uint64_t (&ns2)[4], const uint64_t (&wc2)[4],
                                            const uint64_t (&ws2)[4], const uint64_t (&nws2)[4]) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint64_t c = c2[w], s = s2[w], ns = ns2[w];
    c2[w] = fma2(c, wc2[w], mul2(s, nws2[w]));    // c wc + (-s) ws
    s2[w] = fma2(s, wc2[w], mul2(c, ws2[w]));     // s wc + c ws
    ns2[w] = fma2(ns, wc2[w], mul2(c, nws2[w]));  // -(s wc + c ws), exactly
  }
}

// Load 8 (cos, sin) table entries; sign = -1 gives the inverse rotation.
__device__ __forceinline__ void load_cs8(const float2* __restrict__ cs, float (&c)[8],
                                         float (&s)[8], float sign = 1.0f) {
  const float4* c4 = reinterpret_cast<const float4*>(cs);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float4 t = __ldg(c4 + w);
    c[2 * w] = t.x;
    s[2 * w] = sign * t.y;
    c[2 * w + 1] = t.z;
    s[2 * w + 1] = sign * t.w;
  }
}

template <bool OUT_F16>
__device__ __forceinline__ void rot_chunk(uint4& lo, uint4& hi, const float2* __restrict__ cs,
                                          float sign = 1.0f) {
  float c[8], s[8];
  load_cs8(cs, c, s, sign);
  rot_chunk_cs<OUT_F16>(lo, hi, c, s);
}

// Angle-addition step: (c, s) <- (cos, sin)(a + b) from (c, s) = (cos, sin)(a) and
// (wc, ws) = (cos, sin)(b). Same operation order as rot_pair.
__device__ __forceinline__ void advance_cs8(float (&c)[8], float (&s)[8], const float (&wc)[8],
                                            const float (&ws)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float nc, ns;
    rot_pair(c[e], s[e], wc[e], ws[e], nc, ns);
    c[e] = nc;
    s[e] = ns;
  }
}

// Rows are rotated by a recurrence inside blocks of BLK rows: with CP = d/16 chunk pairs per
// row and RG = 128 / CP row groups, row r of the block at n0 starts from the table entry of
// position n0 + (r % RG) and advances (r / RG) times by the table entry of position RG. The
// forward rotates keys in blocks of 64 (head dim 128: each CTA of a pair rotates one 64-key
// half of a tile) or 128 (head dim 64); the backward rotates Q and K tiles in blocks of 128.
// key_cs8 evaluates exactly that sequence for one row, so a kernel that rotates row by row
// reproduces the in-block recurrence bit for bit.
template <int D, int BLK>
__device__ __forceinline__ void key_cs8(const float2* __restrict__ cs, int n, int chunk,
                                        float (&c)[8], float (&s)[8]) {
  constexpr int CP = D / 16, RG = 128 / CP;
  const int n0 = n & ~(BLK - 1), r = n & (BLK - 1);
  load_cs8(cs + (size_t)(n0 + r % RG) * (D / 2) + chunk * 8, c, s);
  float wc[8], ws[8];
  load_cs8(cs + (size_t)RG * (D / 2) + chunk * 8, wc, ws);
  for (int k = 0; k < r / RG; ++k) advance_cs8(c, s, wc, ws);
}

// Query rows of a 128-row tile are rotated with a recurrence too: row r of the tile at n0
// (n0 a multiple of 128) starts from the table entry of position n0 + (r % 8) and advances
// r / 8 times by the entry of position 8, so a tile needs 9 table rows instead of 128.
// query_cs8 evaluates that sequence for chunk `chunk` (8 pairs) of row n; the forward kernels
// run the same per-pair steps while rotating their Q tiles.
template <int D>
__device__ __forceinline__ void query_cs8(const float2* __restrict__ cs, int n, int chunk,
                                          float (&c)[8], float (&s)[8]) {
  const int n0 = n & ~127, r = n & 127;
  load_cs8(cs + (size_t)(n0 + (r & 7)) * (D / 2) + chunk * 8, c, s);
  float wc[8], ws[8];
  load_cs8(cs + (size_t)8 * (D / 2) + chunk * 8, wc, ws);
  for (int k = 0; k < (r >> 3); ++k) advance_cs8(c, s, wc, ws);
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
  int norm;    // 0 softmax, 1 ReLU (relu_attention)
};

constexpr int kBsMaxN = 65536;                       // block-sparse sequence limit
constexpr int kBsWords = kBsMaxN / 64 / 32;          // bit words per block row (blk 64)
constexpr int kTileWords = kBsMaxN / 128 / 32;       // bit words per kv-tile bitmap

}  // namespace afx
