// Backward attention for sm_103a (AttnFuse paper §4.4): three kernels and no atomics.
//   bwd_pre_kernel   D_m = sum_c dO_mc O_mc                       (HBM-bound row reduction)
//   dkdv_kernel      one CTA per (key tile, kv head, batch): K' and V stay in shared memory;
//                    for every query head of the GQA group and every 64-row query tile that
//                    can see the key tile: S^T = K' Q'^T and dP^T = V dO^T (tcgen05, TMEM),
//                    then P^T = exp(S^T - L), dS^T = P^T (dP^T - D), dV += P^T dO,
//                    dK' += dS^T Q' (two TMEM buffer sets, so item i+1's S^T / dP^T overlap
//                    item i's element-wise step). Epilogue: dK = scale R_n^T dK', dV (GQA sums
//                    stay inside the CTA).
//   dq_kernel        one CTA per (query tile, head, batch): Q' and dO stay in shared memory;
//                    for every visible key tile: S = Q' K'^T, dP = dO V^T, dS = P (dP - D),
//                    dQ' += dS K' (dS double-buffered in TMEM, so the next tile's S and dP
//                    overlap this tile's element-wise step). Epilogue: dQ = scale R_m^T dQ'.
// Rotations use the (cos, sin) table; the rotated operands are rounded to bf16 (the other
// operands of these contractions are bf16). Every wait is bounded (see ptx.cuh).
//
// dkdv_kernel warp roles (12 warps): 0 TMA, 1 MMA, 4-7 element-wise (one thread per TMEM
// lane/row), 8-11 rotate Q/K tiles in shared memory. dq_kernel: see there.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace afx {

namespace {

constexpr int kBwdThreads = 384;
constexpr int kT = 128;  // tile edge (keys and queries)

// Rotate a [TR x D] bf16 tile (TR = 64 or 128 rows, 128B-swizzled panels of TR rows) in place:
// row r at position pos0 + r. Executed by 128 threads (t = 0..127): thread t owns chunk pair
// c = t % CP of rows t / CP + RG k, so it reads the (cos, sin) table once and advances the
// angle by RG positions per row (angle addition) instead of one dependent table read per row.
// The recurrence runs over blocks of 128 positions (a 64-row tile at pos0 % 128 == 64 starts
// (64 / RG) steps in), matching the pre-rotation kernel's blocks of 128 bit for bit.
// Rows at or beyond N are left untouched.
template <int D, int TR>
__device__ __forceinline__ void rotate_tile_bf16(uint8_t* tile, int pos0, int N,
                                                 const float2* __restrict__ cs, int t) {
  constexpr int CP = D / 16, RG = 128 / CP, ROWS = TR / RG;
  const int c = t % CP, rg = t / CP;
  float cc[8], ss[8], wc[8], ws[8];
  load_cs8(cs + (size_t)RG * (D / 2) + c * 8, wc, ws);
  const int p0 = min((pos0 & ~127) + rg, N - 1);
  load_cs8(cs + (size_t)p0 * (D / 2) + c * 8, cc, ss);
  for (int k = 0; k < (pos0 & 127) / RG; ++k) advance_cs8(cc, ss, wc, ws);
#pragma unroll
  for (int k = 0; k < ROWS; ++k) {
    const int row = rg + RG * k;
    if (pos0 + row < N) {
      uint32_t offl, offh;
      if (D == 128) {
        offl = sw128_offset(row, c);
        offh = offl + TR * 128;
      } else {
        offl = sw128_offset(row, c);
        offh = sw128_offset(row, c + 4);
      }
      uint4 lo = *reinterpret_cast<uint4*>(tile + offl);
      uint4 hi = *reinterpret_cast<uint4*>(tile + offh);
      rot_chunk_cs<false>(lo, hi, cc, ss);
      *reinterpret_cast<uint4*>(tile + offl) = lo;
      *reinterpret_cast<uint4*>(tile + offh) = hi;
    }
    if (k + 1 < ROWS) advance_cs8(cc, ss, wc, ws);
  }
}

// Apply scale * R_pos^T to a row of D fp32 values held in registers and store it as bf16.
template <int D, bool ROPE>
__device__ __forceinline__ void store_grad_row(float (&g)[D], float scale, int pos,
                                               const float2* __restrict__ cs,
                                               __nv_bfloat16* __restrict__ dst) {
  if (ROPE) {
#pragma unroll
    for (int i = 0; i < D / 2; ++i) {
      const float2 t = __ldg(cs + (size_t)pos * (D / 2) + i);
      float yl, yh;
      rot_pair(g[i], g[i + D / 2], t.x, -t.y, yl, yh);  // inverse rotation
      g[i] = yl;
      g[i + D / 2] = yh;
    }
  }
  uint4* out = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < D / 8; ++v) {
    uint4 w;
    w.x = pack_bf16x2(g[8 * v + 0] * scale, g[8 * v + 1] * scale);
    w.y = pack_bf16x2(g[8 * v + 2] * scale, g[8 * v + 3] * scale);
    w.z = pack_bf16x2(g[8 * v + 4] * scale, g[8 * v + 5] * scale);
    w.w = pack_bf16x2(g[8 * v + 6] * scale, g[8 * v + 7] * scale);
    out[v] = w;
  }
}

// Load a TMEM row segment of D fp32 columns (one 32x32b load per 32 columns).
template <int D>
__device__ __forceinline__ void tmem_row(uint32_t taddr, float (&g)[D]) {
#pragma unroll
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t o[32];
    tmem_ld32(taddr + ch * 32, o);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) g[ch * 32 + e] = __uint_as_float(o[e]);
  }
}

constexpr int kBq = 64;  // query rows per dK/dV item

template <int D>
struct KvCfg {
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t TILE = kT * D * 2;   // K, V: 128 rows
  static constexpr uint32_t QT = kBq * D * 2;    // Q, dO: 64 rows
  static constexpr int QST = 4;                  // Q / dO stages
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = TILE;
  static constexpr uint32_t OFF_Q = 2 * TILE;
  static constexpr uint32_t OFF_DO = OFF_Q + QST * QT;
  static constexpr uint32_t OFF_VEC = OFF_DO + QST * QT;  // per stage: L (64 f32), D (64 f32)
  static constexpr uint32_t OFF_CTL = OFF_VEC + QST * 512;
};

struct KvCtl {
  uint64_t k_full, v_full, k_ready;
  uint64_t q_full[4], do_full[4], q_ready[4], vec_full[4], stage_free[4];
  uint64_t st_full[2], p_full[2], mma_done[2], mma_final;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
struct DqCfg {
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t TILE = kT * D * 2;
  static constexpr int ST = 2;  // K/V stages
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = TILE;
  static constexpr uint32_t OFF_K = 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + ST * TILE;
  static constexpr uint32_t OFF_CTL = OFF_V + ST * TILE;
};

struct DqCtl {
  uint64_t q_full, do_full, q_ready;
  uint64_t k_full[2], v_full[2], k_ready[2], kv_free[2];
  uint64_t s_full, s_free, p_full, dq_done[2], mma_final;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kDqThreads = 512;
constexpr uint32_t kDqRegsLow = 56, kDqRegsRot = 88, kDqRegsEw = 184;
static_assert(kDqRegsLow + kDqRegsRot + 2 * kDqRegsEw <= 4 * (65536 / kDqThreads),
              "register split exceeds the registers the CTA is launched with");

__host__ __device__ constexpr size_t kv_smem_bytes(int D) {
  return 1024 + 2 * (size_t)(kT * D * 2) + 2 * 4 * (size_t)(kBq * D * 2) + 4 * 512 + sizeof(KvCtl);
}
__host__ __device__ constexpr size_t dq_smem_bytes(int D) {
  return 1024 + (2 + 2 * 2) * (size_t)(kT * D * 2) + sizeof(DqCtl);
}

// Query tiles that can see key tile j (FULL: all; causal: i >= j).
__device__ __forceinline__ int first_q_tile(const BwdParams& p, int j) { return p.causal ? j : 0; }
// Key tiles visible from query tile i.
__device__ __forceinline__ int last_k_tile(const BwdParams& p, int i, int TK) {
  return p.causal ? min(i + 1, TK) : TK;
}

}  // namespace

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
// dK, dV
// ---------------------------------------------------------------------------------------------
// Items are (query head of the GQA group, 64-row query tile). TMEM: dV [0, D), dK' [D, 2D),
// and two buffer sets b = item & 1 of S^T [256 + 64b, +64) and dP^T [384 + 64b, +64), each
// overwritten in place by P^T / dS^T (bf16). While the element-wise warps work on item i, the
// tensor cores compute S^T and dP^T of item i+1 in the other set, then dV and dK' of item i.
template <int D, int RK>
__global__ void __launch_bounds__(kBwdThreads, 1) dkdv_kernel(const __grid_constant__ BwdParams p) {
  constexpr bool ROPE = (RK == kRopeFused);      // rotate Q / K tiles on chip
  constexpr bool ROPE_OUT = (RK != kRopeNone);   // rotate dK back
  using C = KvCfg<D>;
  constexpr int QST = C::QST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  KvCtl* ctl = reinterpret_cast<KvCtl*>(smem + C::OFF_CTL);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N;
  const int TK = (N + kT - 1) / kT;
  const int TQ64 = (N + kBq - 1) / kBq;
  // Group-major order: the CTAs running together share one (b, kv head) group, so that
  // group's Q and dO (re-read by every key tile) stay in L2. Within a group, key tile 0 (the
  // most query tiles under causal masking) goes first.
  const int grp = static_cast<int>(blockIdx.x) / TK;
  const int j = static_cast<int>(blockIdx.x) % TK;
  const int b = grp / p.Hkv, kvh = grp % p.Hkv;
  const bool causal = p.causal != 0;
  const int i0 = causal ? 2 * j : 0;  // first 64-row query tile that can see key tile j
  const int nq = TQ64 - i0;           // query tiles per head
  const int g = p.g;
  const int total = g * nq;           // (head, query tile) items
  int* status = p.status;
  volatile int* abort_flag = &ctl->abort_flag;

  if (tid == 0) {
    mbar_init(&ctl->k_full, 1);
    mbar_init(&ctl->v_full, 1);
    mbar_init(&ctl->k_ready, 128);
    for (int s = 0; s < QST; ++s) {
      mbar_init(&ctl->q_full[s], 1);
      mbar_init(&ctl->do_full[s], 1);
      mbar_init(&ctl->q_ready[s], 128);
      mbar_init(&ctl->vec_full[s], 4);  // one arrival per element-wise warp
      mbar_init(&ctl->stage_free[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->st_full[s], 1);
      mbar_init(&ctl->p_full[s], 4);
      mbar_init(&ctl->mma_done[s], 1);
    }
    mbar_init(&ctl->mma_final, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  constexpr uint32_t T_DV = 0, T_DK = D, T_S = 256, T_DP = 384;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA: K, V once; then Q and dO for every (head, query tile) ----
      tma_prefetch_desc(&p.tmQ64);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      tma_prefetch_desc(&p.tmDO64);
      mbar_arrive_expect_tx(&ctl->k_full, C::TILE);
      for (int pn = 0; pn < C::PANELS; ++pn)
        tma_load_4d(smem + C::OFF_K + pn * (kT * 128), &p.tmK, &ctl->k_full, pn * 64, j * kT, kvh, b);
      mbar_arrive_expect_tx(&ctl->v_full, C::TILE);
      for (int pn = 0; pn < C::PANELS; ++pn)
        tma_load_4d(smem + C::OFF_V + pn * (kT * 128), &p.tmV, &ctl->v_full, pn * 64, j * kT, kvh, b);
      int it = 0;
      for (; it < total; ++it) {
        const int s = it % QST;
        const int h = kvh * g + it / nq, qi = i0 + it % nq;
        if (it >= QST && !mbar_wait(&ctl->stage_free[s], ((it / QST) - 1) & 1, status, abort_flag)) break;
        mbar_arrive_expect_tx(&ctl->q_full[s], C::QT);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::OFF_Q + s * C::QT + pn * (kBq * 128), &p.tmQ64, &ctl->q_full[s],
                      pn * 64, qi * kBq, h, b);
        mbar_arrive_expect_tx(&ctl->do_full[s], C::QT);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::OFF_DO + s * C::QT + pn * (kBq * 128), &p.tmDO64, &ctl->do_full[s],
                      pn * 64, qi * kBq, h, b);
      }
      mbar_wait(&ctl->k_full, 0, status, nullptr);
      mbar_wait(&ctl->v_full, 0, status, nullptr);
      for (int k = max(0, it - QST); k < it; ++k) {
        mbar_wait(&ctl->q_full[k % QST], (k / QST) & 1, status, nullptr);
        mbar_wait(&ctl->do_full[k % QST], (k / QST) & 1, status, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA ----
      constexpr uint32_t idesc_st = idesc_bf16_f32(128, kBq, 0, 0);  // S^T, dP^T: K-major
      constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);     // dV, dK': B MN-major
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
      auto issue_st = [&](int it) -> bool {  // S^T, dP^T of item it into set it & 1
        const int s = it % QST, bs = it & 1;
        const uint32_t ph = (it / QST) & 1;
        if (!mbar_wait(&ctl->q_ready[s], ph, status, abort_flag)) return false;
        if (!mbar_wait(&ctl->do_full[s], ph, status, abort_flag)) return false;
        // the set was last read by dV / dK' of item it-2
        if (it >= 2 && !mbar_wait(&ctl->mma_done[bs], ((it - 2) >> 1) & 1, status, abort_flag))
          return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * (kT * 128) + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * (kBq * 128) + (kk & 3) * 32;
          mma_ss(tmem + T_S + 64 * bs, smem_desc_sw128(sK + ko, 16, 1024),
                 smem_desc_sw128(sQ + s * C::QT + qo, 16, 1024), idesc_st, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * (kT * 128) + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * (kBq * 128) + (kk & 3) * 32;
          mma_ss(tmem + T_DP + 64 * bs, smem_desc_sw128(sV + ko, 16, 1024),
                 smem_desc_sw128(sDO + s * C::QT + qo, 16, 1024), idesc_st, kk > 0);
        }
        mma_commit(&ctl->st_full[bs]);
        return true;
      };
      auto issue_g = [&](int it) -> bool {  // dV += P^T dO ; dK' += dS^T Q'
        const int s = it % QST, bs = it & 1;
        if (!mbar_wait(&ctl->p_full[bs], (it >> 1) & 1, status, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBq / 16; ++kk) {
          mma_ts(tmem + T_DV, tmem + T_S + 64 * bs + kk * 8,
                 smem_desc_sw128(sDO + s * C::QT + kk * 2048, kBq * 128, 1024), idesc_g,
                 (it > 0 || kk > 0) ? 1u : 0u);
          mma_ts(tmem + T_DK, tmem + T_DP + 64 * bs + kk * 8,
                 smem_desc_sw128(sQ + s * C::QT + kk * 2048, kBq * 128, 1024), idesc_g,
                 (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl->mma_done[bs]);
        mma_commit(&ctl->stage_free[s]);
        return true;
      };
      bool ok = mbar_wait(&ctl->k_ready, 0, status, abort_flag) &&
                mbar_wait(&ctl->v_full, 0, status, abort_flag);
      if (ok && total > 0) ok = issue_st(0);
      for (int it = 0; ok && it < total; ++it) {
        if (it + 1 < total) ok = issue_st(it + 1);
        if (ok) ok = issue_g(it);
      }
      mma_commit(&ctl->mma_final);
      mbar_wait(&ctl->mma_final, 0, status, nullptr);
    }
  } else if (warp >= 8) {
    // ---- rotators: K once, then each Q tile ----
    const int t = tid - 256;
    if (ROPE) {
      if (mbar_wait(&ctl->k_full, 0, status, abort_flag))
        rotate_tile_bf16<D, kT>(smem + C::OFF_K, j * kT, N, p.rope_cs, t);
      fence_proxy_async_smem();
    } else {
      mbar_wait(&ctl->k_full, 0, status, abort_flag);
    }
    mbar_arrive(&ctl->k_ready);
    for (int it = 0; it < total; ++it) {
      const int s = it % QST;
      const int qi = i0 + it % nq;
      if (!mbar_wait(&ctl->q_full[s], (it / QST) & 1, status, abort_flag)) break;
      if (ROPE) {
        rotate_tile_bf16<D, kBq>(smem + C::OFF_Q + s * C::QT, qi * kBq, N, p.rope_cs, t);
        fence_proxy_async_smem();
      }
      mbar_arrive(&ctl->q_ready[s]);
    }
  } else if (warp >= 4) {
    // ---- element-wise: thread = key row n of the tile, 64 query columns per item ----
    const int r = (warp - 4) * 32 + lane;
    const int n = j * kT + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    bool ok = true;
    const float c2 = p.scale_log2;
    const float* const lse = p.lse;
    const float* const dvec = p.Dvec;
    const int Hq = p.Hq;
    for (int it = 0; it < total; ++it) {
      const int s = it % QST, bs = it & 1;
      const int h = kvh * g + it / nq, qi = i0 + it % nq;
      const int m0 = qi * kBq;
      float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC + s * 512);
      // stage L (log2 units) and D of the 64 query rows; rows past N get L = +inf (P = 0)
      {
        const int m = m0 + (r & 63);
        float v = (r < 64) ? __int_as_float(0x7f800000) : 0.f;
        if (m < N) {
          const int64_t idx = ((int64_t)b * Hq + h) * N + m;
          if (r < 64) {
            const float l = lse[idx];
            v = (l == kNegInf) ? __int_as_float(0x7f800000) : l * kLog2e;
          } else {
            v = dvec[idx];
          }
        }
        vec[r] = v;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->vec_full[s]);
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&ctl->vec_full[s], (it / QST) & 1, status, abort_flag) &&
                          mbar_wait(&ctl->st_full[bs], (it >> 1) & 1, status, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64], dr[64];
      tmem_ld32<0>(tmem + lane_off + T_S + 64 * bs, sr);
      tmem_ld32<32>(tmem + lane_off + T_S + 64 * bs + 32, sr);
      tmem_ld32<0>(tmem + lane_off + T_DP + 64 * bs, dr);
      tmem_ld32<32>(tmem + lane_off + T_DP + 64 * bs + 32, dr);
      tmem_wait_ld();
      float pr[64];
#pragma unroll
      for (int c = 0; c < 64; ++c)
        pr[c] = ex2_approx(__fmaf_rn(__uint_as_float(sr[c]), c2, -vec[c]));
      if (__builtin_expect(causal && m0 < n, 0)) {
        // causal diagonal: query m0 + c sees key n only if m0 + c >= n
#pragma unroll
        for (int c = 0; c < 64; ++c) pr[c] = (m0 + c >= n) ? pr[c] : 0.f;
      }
      uint32_t pk[32], dk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float d0 = pr[2 * c] * (__uint_as_float(dr[2 * c]) - vec[64 + 2 * c]);
        const float d1 = pr[2 * c + 1] * (__uint_as_float(dr[2 * c + 1]) - vec[64 + 2 * c + 1]);
        pk[c] = pack_bf16x2(pr[2 * c], pr[2 * c + 1]);
        dk[c] = pack_bf16x2(d0, d1);
      }
      tmem_st32<0>(tmem + lane_off + T_S + 64 * bs, pk);
      tmem_st32<0>(tmem + lane_off + T_DP + 64 * bs, dk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full[bs]);
    }
    // ---- epilogue ----
    if (ok && total > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->mma_done[(total - 1) & 1], ((total - 1) >> 1) & 1,
                                             status, abort_flag));
      tc_fence_after();
    }
    float gr[D];
    if (ok && total > 0) tmem_row<D>(tmem + lane_off + T_DV, gr);
    else
#pragma unroll
      for (int c = 0; c < D; ++c) gr[c] = 0.f;
    if (n < N)
      store_grad_row<D, false>(gr, 1.f, n, p.rope_cs,
                               p.dv + b * p.dv_s[0] + kvh * p.dv_s[1] + (int64_t)n * p.dv_s[2]);
    if (ok && total > 0) tmem_row<D>(tmem + lane_off + T_DK, gr);
    else
#pragma unroll
      for (int c = 0; c < D; ++c) gr[c] = 0.f;
    if (n < N)
      store_grad_row<D, ROPE_OUT>(gr, p.scale, n, p.rope_cs,
                                  p.dk + b * p.dk_s[0] + kvh * p.dk_s[1] + (int64_t)n * p.dk_s[2]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------------------------
// dQ
// ---------------------------------------------------------------------------------------------
// 16 warps: 0 TMA, 1 MMA, 4-11 element-wise (warps 4-7 key columns 0-63 of each tile, 8-11
// columns 64-127; one query row per thread), 12-15 rotate Q once and each K tile.
// TMEM: dQ' [0, D), S [128, 256), dP [256, 384), dS (bf16) double-buffered at [384, 448) and
// [448, 512). dS does not overwrite S, so S(j+1) and dP(j+1) are computed while the
// element-wise warps still work on tile j.
template <int D, int RK>
__global__ void __launch_bounds__(kDqThreads, 1) dq_kernel(const __grid_constant__ BwdParams p) {
  constexpr bool ROPE = (RK == kRopeFused);      // rotate Q / K tiles on chip
  constexpr bool ROPE_OUT = (RK != kRopeNone);   // rotate dQ back
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  DqCtl* ctl = reinterpret_cast<DqCtl*>(smem + C::OFF_CTL);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N;
  const int TQ = (N + kT - 1) / kT;
  const int per_i = p.B * p.Hq;
  const int i = TQ - 1 - static_cast<int>(blockIdx.x) / per_i;  // longest first
  const int rem = static_cast<int>(blockIdx.x) % per_i;
  const int b = rem / p.Hq, h = rem % p.Hq;
  const int kvh = h / p.g;
  const int nk = last_k_tile(p, i, TQ);
  int* status = p.status;
  volatile int* abort_flag = &ctl->abort_flag;

  if (tid == 0) {
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->do_full, 1);
    mbar_init(&ctl->q_ready, 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->k_ready[s], 128);
      mbar_init(&ctl->kv_free[s], 1);
      mbar_init(&ctl->dq_done[s], 1);
    }
    mbar_init(&ctl->s_full, 1);
    mbar_init(&ctl->s_free, 8);   // one arrival per element-wise warp
    mbar_init(&ctl->p_full, 8);
    mbar_init(&ctl->mma_final, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  constexpr uint32_t T_DQ = 0, T_S = 128, T_DP = 256, T_DS = 384;

  if (warp < 4) {
    setmaxnreg_dec<kDqRegsLow>();
    if (warp == 0 && lane == 0) {
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      tma_prefetch_desc(&p.tmDO);
      mbar_arrive_expect_tx(&ctl->q_full, C::TILE);
      for (int pn = 0; pn < C::PANELS; ++pn)
        tma_load_4d(smem + C::OFF_Q + pn * (kT * 128), &p.tmQ, &ctl->q_full, pn * 64, i * kT, h, b);
      mbar_arrive_expect_tx(&ctl->do_full, C::TILE);
      for (int pn = 0; pn < C::PANELS; ++pn)
        tma_load_4d(smem + C::OFF_DO + pn * (kT * 128), &p.tmDO, &ctl->do_full, pn * 64, i * kT, h, b);
      int jt = 0;
      for (; jt < nk; ++jt) {
        const int s = jt & 1;
        if (jt >= 2 && !mbar_wait(&ctl->kv_free[s], ((jt >> 1) - 1) & 1, status, abort_flag)) break;
        mbar_arrive_expect_tx(&ctl->k_full[s], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::OFF_K + s * C::TILE + pn * (kT * 128), &p.tmK, &ctl->k_full[s],
                      pn * 64, jt * kT, kvh, b);
        mbar_arrive_expect_tx(&ctl->v_full[s], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::OFF_V + s * C::TILE + pn * (kT * 128), &p.tmV, &ctl->v_full[s],
                      pn * 64, jt * kT, kvh, b);
      }
      mbar_wait(&ctl->q_full, 0, status, nullptr);
      mbar_wait(&ctl->do_full, 0, status, nullptr);
      for (int k = max(0, jt - 2); k < jt; ++k) {
        mbar_wait(&ctl->k_full[k & 1], (k >> 1) & 1, status, nullptr);
        mbar_wait(&ctl->v_full[k & 1], (k >> 1) & 1, status, nullptr);
      }
    } else if (warp == 1 && lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kT, 0, 0);  // S, dP: both K-major
      constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);   // dQ': B = K' MN-major
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      auto issue_dq = [&](int jq) -> bool {  // dQ' += dS(jq) K'(jq)
        if (!mbar_wait(&ctl->p_full, jq & 1, status, abort_flag)) return false;
        tc_fence_after();
        const int s = jq & 1;
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ts(tmem + T_DQ, tmem + T_DS + s * 64 + kk * 8,
                 smem_desc_sw128(sK + s * C::TILE + kk * 2048, kT * 128, 1024), idesc_g,
                 (jq > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&ctl->dq_done[s]);
        mma_commit(&ctl->kv_free[s]);
        return true;
      };
      bool ok = mbar_wait(&ctl->q_ready, 0, status, abort_flag) &&
                mbar_wait(&ctl->do_full, 0, status, abort_flag);
      for (int jt = 0; ok && jt < nk; ++jt) {
        const int s = jt & 1;
        const uint32_t ph = (jt >> 1) & 1;
        ok = mbar_wait(&ctl->k_ready[s], ph, status, abort_flag) &&
             mbar_wait(&ctl->v_full[s], ph, status, abort_flag);
        // S and dP of tile jt overwrite those of tile jt-1 once the element-wise warps hold them
        if (ok && jt > 0) ok = mbar_wait(&ctl->s_free, (jt - 1) & 1, status, abort_flag);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (kT * 128) + (kk & 3) * 32;
          mma_ss(tmem + T_S, smem_desc_sw128(sQ + koff, 16, 1024),
                 smem_desc_sw128(sK + s * C::TILE + koff, 16, 1024), idesc_s, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (kT * 128) + (kk & 3) * 32;
          mma_ss(tmem + T_DP, smem_desc_sw128(sDO + koff, 16, 1024),
                 smem_desc_sw128(sV + s * C::TILE + koff, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&ctl->s_full);
        if (jt > 0) ok = issue_dq(jt - 1);
      }
      if (ok && nk > 0) issue_dq(nk - 1);
      mma_commit(&ctl->mma_final);
      mbar_wait(&ctl->mma_final, 0, status, nullptr);
    }
  } else if (warp >= 12) {
    setmaxnreg_dec<kDqRegsRot>();
    const int t = tid - 384;
    if (mbar_wait(&ctl->q_full, 0, status, abort_flag) && ROPE) {
      rotate_tile_bf16<D, kT>(smem + C::OFF_Q, i * kT, N, p.rope_cs, t);
      fence_proxy_async_smem();
    }
    mbar_arrive(&ctl->q_ready);
    for (int jt = 0; jt < nk; ++jt) {
      const int s = jt & 1;
      if (!mbar_wait(&ctl->k_full[s], (jt >> 1) & 1, status, abort_flag)) break;
      if (ROPE) {
        rotate_tile_bf16<D, kT>(smem + C::OFF_K + s * C::TILE, jt * kT, N, p.rope_cs, t);
        fence_proxy_async_smem();
      }
      mbar_arrive(&ctl->k_ready[s]);
    }
  } else {
    // ---- element-wise: thread = query row m, key columns 64 hh .. 64 hh + 63 ----
    setmaxnreg_inc<kDqRegsEw>();
    const int hh = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int m = i * kT + r;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const bool causal = p.causal != 0;
    float l2 = __int_as_float(0x7f800000), dd = 0.f;
    if (m < N) {
      const float l = p.lse[((int64_t)b * p.Hq + h) * N + m];
      l2 = (l == kNegInf) ? __int_as_float(0x7f800000) : l * kLog2e;
      dd = p.Dvec[((int64_t)b * p.Hq + h) * N + m];
    }
    bool ok = true;
    const float c2 = p.scale_log2;
    for (int jt = 0; jt < nk; ++jt) {
      if (!__all_sync(0xffffffffu, mbar_wait(&ctl->s_full, jt & 1, status, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64], dr[64];
      tmem_ld32<0>(tmem + lane_off + T_S + 64 * hh, sr);
      tmem_ld32<32>(tmem + lane_off + T_S + 64 * hh + 32, sr);
      tmem_ld32<0>(tmem + lane_off + T_DP + 64 * hh, dr);
      tmem_ld32<32>(tmem + lane_off + T_DP + 64 * hh + 32, dr);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_free);
      const int k0 = jt * kT + 64 * hh;  // first key of this half
      float pr[64];
      const uint64_t c22 = f2_pack(c2, c2), nl2 = f2_pack(-l2, -l2);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const uint64_t a = fma2(f2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), c22, nl2);
        pr[2 * c] = ex2_approx(f2_lo(a));
        pr[2 * c + 1] = ex2_approx(f2_hi(a));
      }
      if (__builtin_expect((causal && jt == i) || k0 + 64 > N, 0)) {
        const int c_hi = min(causal ? m - k0 : 63, N - 1 - k0);
#pragma unroll
        for (int c = 0; c < 64; ++c) pr[c] = (c <= c_hi) ? pr[c] : 0.f;
      }
      uint32_t dk[32];
      const uint64_t ndd = f2_pack(-dd, -dd);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const uint64_t dpm = add2(f2_pack(__uint_as_float(dr[2 * c]), __uint_as_float(dr[2 * c + 1])), ndd);
        const uint64_t ds = mul2(f2_pack(pr[2 * c], pr[2 * c + 1]), dpm);
        dk[c] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
      }
      // the dS buffer of tile jt was read by dQ(jt-2)
      if (jt >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(&ctl->dq_done[jt & 1], ((jt - 2) >> 1) & 1, status, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st32<0>(tmem + lane_off + T_DS + (jt & 1) * 64 + 32 * hh, dk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full);
    }
    if (hh == 0) {
      if (ok && nk > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->dq_done[(nk - 1) & 1], ((nk - 1) >> 1) & 1,
                                               status, abort_flag));
        tc_fence_after();
      }
      float g[D];
      if (ok && nk > 0) tmem_row<D>(tmem + lane_off + T_DQ, g);
      else
#pragma unroll
        for (int c = 0; c < D; ++c) g[c] = 0.f;
      if (m < N)
        store_grad_row<D, ROPE_OUT>(g, p.scale, m, p.rope_cs,
                                    p.dq + b * p.dq_s[0] + h * p.dq_s[1] + (int64_t)m * p.dq_s[2]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
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
  void (*kv)(BwdParams) = nullptr;
  void (*dq)(BwdParams) = nullptr;
  if (d == 128) {
    kv = rk == kRopeFused ? dkdv_kernel<128, kRopeFused>
         : rk == kRopePrerotated ? dkdv_kernel<128, kRopePrerotated> : dkdv_kernel<128, kRopeNone>;
    dq = rk == kRopeFused ? dq_kernel<128, kRopeFused>
         : rk == kRopePrerotated ? dq_kernel<128, kRopePrerotated> : dq_kernel<128, kRopeNone>;
  } else {
    kv = rk == kRopeFused ? dkdv_kernel<64, kRopeFused>
         : rk == kRopePrerotated ? dkdv_kernel<64, kRopePrerotated> : dkdv_kernel<64, kRopeNone>;
    dq = rk == kRopeFused ? dq_kernel<64, kRopeFused>
         : rk == kRopePrerotated ? dq_kernel<64, kRopePrerotated> : dq_kernel<64, kRopeNone>;
  }
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
