// Backward attention kernels for sm_103a (AttnFuse paper §4.4), templated on head dim, RoPE
// mode and bias combinator; bwd.cu instantiates the bias-free kernels, bwd_bias.cu the ALiBi and
// additive-bias ones. With bwd_pre_kernel (D_m = sum_c dO_mc O_mc, bwd.cu) they form the
// paper's three-kernel backward, without atomics:
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
// Variants (paper §3.1 combinators, §4.3 "both forward and backward kernels iterate only over
// active blocks"): the mask decides which (query tile, key tile) pairs a CTA visits (causal and
// sliding-window ranges; for block-sparse layouts the dK/dV kernel scans the CSR for the query
// tiles that can see its key tile, i.e. the transposed layout, and the dQ kernel reads its own
// block rows), and partial tiles are masked per element. ALiBi and the additive bias are added
// to the recomputed scores exactly as in the forward; with an additive bias the dQ kernel also
// writes dBias = dS (fp32), including the zeros of every pair it does not visit.
//
// dkdv_kernel warp roles (12 warps): 0 TMA, 1 MMA, 4-7 element-wise (one thread per TMEM
// lane/row), 8-11 rotate Q/K tiles in shared memory. dq_kernel: see there.
#pragma once
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
  int nq_bs;                        // block-sparse: active 64-row query tiles
  uint8_t qbits[kBsMaxN / kBq];     // block-sparse: bit h set = query tile active for key
                                    // block 2j + h (64-blocks; 128-blocks set both bits)
  int16_t qlist[kBsMaxN / kBq];     // block-sparse: active query tiles, ascending
};

template <int D>
struct DqCfg {
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t TILE = kT * D * 2;
  // K stages are released by dQ (the last MMA to read K), V stages by dP, which completes a
  // whole group earlier: three K stages and two V stages fill shared memory for head dim 128.
  static constexpr int KST = 3, VST = 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = TILE;
  static constexpr uint32_t OFF_K = 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + KST * TILE;
  static constexpr uint32_t OFF_CTL = OFF_V + VST * TILE;
};

struct DqCtl {
  uint64_t q_full, do_full, q_ready;
  uint64_t k_full[3], k_ready[3], k_free[3], v_full[2], v_free[2];
  uint64_t s_full, s_free, p_full[2], dq_done[2], mma_final;
  uint32_t tmem_base;
  int abort_flag;
  uint32_t tile_bits[kTileWords];   // block-sparse: key tiles with an active block
  uint32_t row_bits[2][kBsWords];   // block-sparse (64-blocks): active block columns of the
                                    // tile's two block rows
};

constexpr int kDqThreads = 512;
constexpr uint32_t kDqRegsLow = 56, kDqRegsRot = 88, kDqRegsEw = 184;
static_assert(kDqRegsLow + kDqRegsRot + 2 * kDqRegsEw <= 4 * (65536 / kDqThreads),
              "register split exceeds the registers the CTA is launched with");

__host__ __device__ constexpr size_t kv_smem_bytes(int D) {
  return 1024 + 2 * (size_t)(kT * D * 2) + 2 * 4 * (size_t)(kBq * D * 2) + 4 * 512 + sizeof(KvCtl);
}
static_assert(1024 + 2 * 32768 + 8 * 16384 + 4 * 512 + sizeof(KvCtl) <= 232448,
              "dK/dV shared memory budget (head dim 128)");
__host__ __device__ constexpr size_t dq_smem_bytes(int D) {
  return 1024 + (2 + 3 + 2) * (size_t)(kT * D * 2) + sizeof(DqCtl);
}
static_assert(1024 + 7 * 32768 + sizeof(DqCtl) <= 232448, "dQ shared memory budget (head dim 128)");

__device__ __forceinline__ bool bit_get(const uint32_t* w, int i) {
  return (w[i >> 5] >> (i & 31)) & 1u;
}

// Key tiles [lo, hi) that 128-row query tile i can see under the causal / sliding-window
// restrictions (block-sparse layouts further thin the range).
__device__ __forceinline__ void dq_range(const BwdParams& p, int i, int TK, int& lo, int& hi) {
  const VariantDev& v = p.var;
  const int m_hi = min(i * kT + kT - 1, p.N - 1);
  lo = 0;
  hi = TK;
  if (v.causal) hi = min(hi, m_hi / kT + 1);
  if (v.mask == 2) {
    lo = max(0, i * kT - v.window + 1) / kT;
    if (!v.causal) hi = min(hi, (m_hi + v.window - 1) / kT + 1);
  }
}

// 64-row query tiles [lo, hi) that can see key tile j (keys n in [128 j, n_hi]): causal needs
// m >= n, a window of W needs m < n + W and, without causal, m > n - W.
__device__ __forceinline__ void kv_range(const BwdParams& p, int j, int TQ64, int& lo, int& hi) {
  const VariantDev& v = p.var;
  const int n_hi = min(j * kT + kT - 1, p.N - 1);
  lo = 0;
  hi = TQ64;
  if (v.causal) lo = (j * kT) / kBq;
  if (v.mask == 2) {
    hi = min(hi, (n_hi + v.window - 1) / kBq + 1);
    if (!v.causal) lo = max(0, j * kT - v.window + 1) / kBq;
  }
}

// Additive-bias element (fp32 or bf16 storage), already at its element offset.
__device__ __forceinline__ float bias_at(const VariantDev& v, int64_t off) {
  return v.add_bias_bf16
             ? __bfloat162float(static_cast<const __nv_bfloat16*>(v.add_bias)[off])
             : static_cast<const float*>(v.add_bias)[off];
}

}  // namespace

// ---------------------------------------------------------------------------------------------
// dK, dV
// ---------------------------------------------------------------------------------------------
// Items are (query head of the GQA group, 64-row query tile). TMEM: dV [0, D), dK' [D, 2D),
// and two buffer sets b = item & 1 of S^T [256 + 64b, +64) and dP^T [384 + 64b, +64), each
// overwritten in place by P^T / dS^T (bf16). While the element-wise warps work on item i, the
// tensor cores compute S^T and dP^T of item i+1 in the other set, then dV and dK' of item i.
template <int D, int RK, int BIAS>
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
  const VariantDev& var = p.var;
  const bool causal = var.causal != 0;
  const bool sparse = var.mask == 3;
  int q_lo, q_hi;  // 64-row query tiles that can see key tile j
  kv_range(p, j, TQ64, q_lo, q_hi);
  const int g = p.g;
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
  if (sparse)
    for (int q = tid; q < TQ64; q += kBwdThreads) ctl->qbits[q] = 0;
  if (warp == 1) tmem_alloc(&ctl->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  constexpr uint32_t T_DV = 0, T_DK = D, T_S = 256, T_DP = 384;

  // Items: (query head of the group, query tile). Block-sparse layouts: the transposed view of
  // the CSR, i.e. the block rows that hold key block 2j / 2j+1 (64-blocks) or j (128-blocks).
  int nq = max(0, q_hi - q_lo);
  if (sparse) {
    const int blk = var.bs_block, nbt = (N + blk - 1) / blk;
    for (int br = tid; br < nbt; br += kBwdThreads) {
      int bits = 0;
      for (int e = var.bs_row_ptr[br]; e < var.bs_row_ptr[br + 1]; ++e) {
        const int col = var.bs_col_idx[e];
        if (blk == 64) bits |= (col == 2 * j ? 1 : 0) | (col == 2 * j + 1 ? 2 : 0);
        else bits |= (col == j ? 3 : 0);
      }
      if (bits) {
        if (blk == 64) {
          ctl->qbits[br] = static_cast<uint8_t>(bits);
        } else {
          ctl->qbits[2 * br] = 3;
          if (2 * br + 1 < TQ64) ctl->qbits[2 * br + 1] = 3;
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      int cnt = 0;
      for (int base = q_lo; base < q_hi; base += 32) {
        const int qi = base + lane;
        const bool on = qi < q_hi && ctl->qbits[qi] != 0;
        const uint32_t bal = __ballot_sync(0xffffffffu, on);
        if (on) ctl->qlist[cnt + __popc(bal & ((1u << lane) - 1u))] = static_cast<int16_t>(qi);
        cnt += __popc(bal);
      }
      if (lane == 0) ctl->nq_bs = cnt;
    }
    __syncthreads();
    nq = ctl->nq_bs;
  }
  const int total = g * nq;  // (head, query tile) items
  auto qtile = [&](int idx) -> int { return sparse ? static_cast<int>(ctl->qlist[idx]) : q_lo + idx; };

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
        const int h = kvh * g + it / nq, qi = qtile(it % nq);
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
      const int qi = qtile(it % nq);
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
    const int mask_kind = var.mask, W = var.window;
    const bool bs64 = sparse && var.bs_block == 64;
    for (int it = 0; it < total; ++it) {
      const int s = it % QST, bs = it & 1;
      const int h = kvh * g + it / nq, qi = qtile(it % nq);
      const int m0 = qi * kBq;
      if (p.visits_kv && r == 0) p.visits_kv[((static_cast<int64_t>(b) * Hq + h) * TQ64 + qi) * TK + j] = 1;
      float slope2 = 0.f;
      if constexpr (BIAS == 1) slope2 = var.slopes[h] * kLog2e;
      float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC + s * 512);
      // stage L (log2 units) and D of the 64 query rows; rows past N get L = +inf (P = 0).
      // ALiBi: the column part of slope (n - m) is folded into L: L + slope * (m - m0).
      {
        const int m = m0 + (r & 63);
        float v = (r < 64) ? __int_as_float(0x7f800000) : 0.f;
        if (m < N) {
          const int64_t idx = ((int64_t)b * Hq + h) * N + m;
          if (r < 64) {
            const float l = lse[idx];
            v = (l == kNegInf) ? __int_as_float(0x7f800000) : l * kLog2e;
            if constexpr (BIAS == 1) v += slope2 * static_cast<float>(r & 63);
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
      if constexpr (BIAS == 0) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          pr[c] = ex2_approx(__fmaf_rn(__uint_as_float(sr[c]), c2, -vec[c]));
      } else if constexpr (BIAS == 1) {
        const float tn = slope2 * static_cast<float>(n - m0);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          pr[c] = ex2_approx(__fmaf_rn(__uint_as_float(sr[c]), c2, tn - vec[c]));
      } else {
        // bias[b, h, m0 + c, n]: consecutive threads read consecutive keys
        const int64_t boff = b * var.ab_s[0] + h * var.ab_s[1] + (int64_t)m0 * var.ab_s[2] +
                             (int64_t)n * var.ab_s[3];
        // Branch-free: out-of-range lanes read element 0 and drop it, so the warp never
        // diverges before the warp-collective TMEM and barrier operations below.
        const int c_end = (n < N) ? min(64, N - m0) : 0;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const bool in = c < c_end;
          const float raw = bias_at(var, in ? boff + c * var.ab_s[2] : 0);
          const float bv = in ? raw : 0.f;
          pr[c] = ex2_approx(__fmaf_rn(bv, kLog2e, __fmaf_rn(__uint_as_float(sr[c]), c2, -vec[c])));
        }
      }
      // Mask of this key row over the item's 64 queries m0 + c: causal needs c >= n - m0, a
      // window c <= n + W - 1 - m0 (and c >= n - W + 1 - m0 without causal), a 64-block layout
      // the (query tile, key block) bit.
      {
        int c_lo = causal ? n - m0 : 0, c_hi = 63;
        if (mask_kind == 2) {
          c_hi = n + W - 1 - m0;
          if (!causal) c_lo = n - W + 1 - m0;
        }
        const bool on = !bs64 || ((ctl->qbits[qi] >> (r >> 6)) & 1);
        if (__builtin_expect(c_lo > 0 || c_hi < 63 || !on, 0)) {
#pragma unroll
          for (int c = 0; c < 64; ++c) pr[c] = (on && c >= c_lo && c <= c_hi) ? pr[c] : 0.f;
        }
      }
      uint32_t pk[32], dk[32];
      __syncwarp();  // tcgen05.st below is warp-aligned: reconverge after the per-row branches
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
template <int D, int RK, int BIAS>
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
  const VariantDev& var = p.var;
  const bool sparse = var.mask == 3;
  int k_lo, k_hi;  // key tiles the query tile can see; block-sparse: those with a set bit
  dq_range(p, i, TQ, k_lo, k_hi);
  int* status = p.status;
  volatile int* abort_flag = &ctl->abort_flag;

  if (tid == 0) {
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->do_full, 1);
    mbar_init(&ctl->q_ready, 128);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_ready[s], 128);
      mbar_init(&ctl->k_free[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_free[s], 1);
      mbar_init(&ctl->dq_done[s], 1);
    }
    mbar_init(&ctl->s_full, 1);
    mbar_init(&ctl->s_free, 8);   // one arrival per element-wise warp
    // dS of tile jt: one barrier per tile parity. The element-wise warps may drift one tile
    // apart (a warp that has loaded S(jt+1) can finish it before another finishes tile jt), so
    // arrivals for consecutive tiles must not share a barrier phase.
    mbar_init(&ctl->p_full[0], 8);
    mbar_init(&ctl->p_full[1], 8);
    mbar_init(&ctl->mma_final, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (sparse) {
    for (int w = tid; w < kTileWords; w += kDqThreads) ctl->tile_bits[w] = 0;
    for (int w = tid; w < 2 * kBsWords; w += kDqThreads) (&ctl->row_bits[0][0])[w] = 0;
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  constexpr uint32_t T_DQ = 0, T_S = 128, T_DP = 256, T_DS = 384;
  if (sparse) {
    // key tiles holding an active block of this query tile's block rows
    const int blk = var.bs_block, nbt = (N + blk - 1) / blk;
    for (int rr = 0; rr < kT / blk; ++rr) {
      const int br = i * (kT / blk) + rr;
      if (br >= nbt) continue;
      for (int e = var.bs_row_ptr[br] + tid; e < var.bs_row_ptr[br + 1]; e += kDqThreads) {
        const int col = var.bs_col_idx[e];
        if (col < 0 || col >= nbt) continue;
        const int tile = col * blk / kT;
        atomicOr(&ctl->tile_bits[tile >> 5], 1u << (tile & 31));
        if (blk == 64) atomicOr(&ctl->row_bits[rr][col >> 5], 1u << (col & 31));
      }
    }
    __syncthreads();
  }
  // next visible key tile at or after jt (every role walks the same sequence)
  auto next_k = [&](int jt) -> int {
    if (sparse)
      while (jt < k_hi && !bit_get(ctl->tile_bits, jt)) ++jt;
    return jt;
  };

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
      int it = 0, iv = 0;
      for (int jt = next_k(k_lo); jt < k_hi; jt = next_k(jt + 1), ++it) {
        const int sk = it % C::KST, sv = it % C::VST;
        if (it >= C::KST && !mbar_wait(&ctl->k_free[sk], ((it / C::KST) - 1) & 1, status, abort_flag)) break;
        mbar_arrive_expect_tx(&ctl->k_full[sk], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::OFF_K + sk * C::TILE + pn * (kT * 128), &p.tmK, &ctl->k_full[sk],
                      pn * 64, jt * kT, kvh, b);
        if (it >= C::VST && !mbar_wait(&ctl->v_free[sv], ((it / C::VST) - 1) & 1, status, abort_flag)) {
          ++it;  // K(it) is in flight
          break;
        }
        mbar_arrive_expect_tx(&ctl->v_full[sv], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::OFF_V + sv * C::TILE + pn * (kT * 128), &p.tmV, &ctl->v_full[sv],
                      pn * 64, jt * kT, kvh, b);
        iv = it + 1;
      }
      mbar_wait(&ctl->q_full, 0, status, nullptr);
      mbar_wait(&ctl->do_full, 0, status, nullptr);
      for (int k = max(0, it - C::KST); k < it; ++k)
        mbar_wait(&ctl->k_full[k % C::KST], (k / C::KST) & 1, status, nullptr);
      for (int k = max(0, iv - C::VST); k < iv; ++k)
        mbar_wait(&ctl->v_full[k % C::VST], (k / C::VST) & 1, status, nullptr);
    } else if (warp == 1 && lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kT, 0, 0);  // S, dP: both K-major
      constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);   // dQ': B = K' MN-major
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      auto issue_dq = [&](int jq) {  // dQ' += dS(jq) K'(jq); dS(jq) is in TMEM
        tc_fence_after();
        const int sk = jq % C::KST;
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ts(tmem + T_DQ, tmem + T_DS + (jq & 1) * 64 + kk * 8,
                 smem_desc_sw128(sK + sk * C::TILE + kk * 2048, kT * 128, 1024), idesc_g,
                 (jq > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&ctl->dq_done[jq & 1]);
        mma_commit(&ctl->k_free[sk]);
      };
      auto issue_s = [&](int js) {  // S(js) = Q' K'(js)^T, dP(js) = dO V(js)^T
        const int sk = js % C::KST, sv = js % C::VST;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (kT * 128) + (kk & 3) * 32;
          mma_ss(tmem + T_S, smem_desc_sw128(sQ + koff, 16, 1024),
                 smem_desc_sw128(sK + sk * C::TILE + koff, 16, 1024), idesc_s, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (kT * 128) + (kk & 3) * 32;
          mma_ss(tmem + T_DP, smem_desc_sw128(sDO + koff, 16, 1024),
                 smem_desc_sw128(sV + sv * C::TILE + koff, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&ctl->s_full);
        mma_commit(&ctl->v_free[sv]);  // V is read by dP only
      };
      bool ok = mbar_wait(&ctl->q_ready, 0, status, abort_flag) &&
                mbar_wait(&ctl->do_full, 0, status, abort_flag);
      int nk = 0;  // visible key tiles (js / jq below count them, not tile indices)
      for (int kt = next_k(k_lo); kt < k_hi; kt = next_k(kt + 1)) ++nk;
      // Poll-driven issue: dQ(jq) goes as soon as its dS is in TMEM (its completion frees the
      // K/V stage of tile jq + 2), S(js) and dP(js) as soon as their tile has landed and the
      // element-wise warps hold S(js - 1) and dP(js - 1). Neither waits behind the other; dQ
      // goes first when both can. The poll is bounded like every wait.
      int js = 0, jq = 0;
      uint64_t t0 = 0;
      uint32_t idle = 0;
      while (ok && jq < nk) {
        bool moved = false;
        if (jq < js && mbar_test(&ctl->p_full[jq & 1], (jq >> 1) & 1)) {
          issue_dq(jq);
          ++jq;
          moved = true;
        } else if (js < nk) {
          const int sk = js % C::KST, sv = js % C::VST;
          if (mbar_test(&ctl->k_ready[sk], (js / C::KST) & 1) &&
              mbar_test(&ctl->v_full[sv], (js / C::VST) & 1) &&
              (js == 0 || mbar_test(&ctl->s_free, (js - 1) & 1))) {
            issue_s(js);
            ++js;
            moved = true;
          }
        }
        if (moved) {
          idle = 0;
        } else if ((++idle & 255u) == 1u) {
          const uint64_t now = globaltimer_ns();
          if (idle == 1u) t0 = now;
          if (*abort_flag) {
            ok = false;
          } else if (now - t0 > ATTNFUSE_WAIT_LIMIT_NS) {
            atomicOr(status, kDevTimeout);
            *abort_flag = 1;
            ok = false;
          }
        }
      }
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
    int it = 0;
    uint8_t* const visits = p.visits_dq;
    const int TKv = (N + kT - 1) / kT;
    for (int jt = next_k(k_lo); jt < k_hi; jt = next_k(jt + 1), ++it) {
      const int s = it % C::KST;
      if (visits && t == 0) visits[((static_cast<int64_t>(b) * p.Hq + h) * TQ + i) * TKv + jt] = 1;
      if (!mbar_wait(&ctl->k_full[s], (it / C::KST) & 1, status, abort_flag)) break;
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
    const bool causal = var.causal != 0;
    const int mask_kind = var.mask, W = var.window;
    const bool bs64 = sparse && var.bs_block == 64;
    float l2 = __int_as_float(0x7f800000), dd = 0.f;
    if (m < N) {
      const float l = p.lse[((int64_t)b * p.Hq + h) * N + m];
      l2 = (l == kNegInf) ? __int_as_float(0x7f800000) : l * kLog2e;
      dd = p.Dvec[((int64_t)b * p.Hq + h) * N + m];
    }
    float slope2 = 0.f;
    if constexpr (BIAS == 1) slope2 = var.slopes[h] * kLog2e;
    int64_t brow = 0;        // additive bias: offset of element (b, h, m, 0)
    float* dbrow = nullptr;  // additive bias: dBias row (b, h, m), or none
    const bool db_vec2 = p.db_vec2 != 0;  // rows 8-byte aligned: store dBias in pairs
    if constexpr (BIAS == 2) {
      brow = b * var.ab_s[0] + h * var.ab_s[1] + (int64_t)m * var.ab_s[2];
      if (p.dbias && m < N) dbrow = p.dbias + b * p.db_s[0] + h * p.db_s[1] + (int64_t)m * p.db_s[2];
    }
    bool ok = true;
    const float c2 = p.scale_log2;
    int jt = 0;  // visible tiles done
    for (int kt = next_k(k_lo); kt < k_hi; kt = next_k(kt + 1), ++jt) {
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
      const int k0 = kt * kT + 64 * hh;  // first key of this half
      float pr[64];
      if constexpr (BIAS == 0) {
        const uint64_t c22 = f2_pack(c2, c2), nl2 = f2_pack(-l2, -l2);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const uint64_t a = fma2(f2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), c22, nl2);
          pr[2 * c] = ex2_approx(f2_lo(a));
          pr[2 * c + 1] = ex2_approx(f2_hi(a));
        }
      } else if constexpr (BIAS == 1) {
        // slope (n - m) = slope (k0 - m) + slope c
        const float base = __fmaf_rn(slope2, static_cast<float>(k0 - m), -l2);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          pr[c] = ex2_approx(__fmaf_rn(slope2, static_cast<float>(c),
                                       __fmaf_rn(__uint_as_float(sr[c]), c2, base)));
      } else {
        // Branch-free (see the dK/dV kernel): out-of-range lanes read element 0 and drop it.
        const int c_end = (m < N) ? min(64, N - k0) : 0;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const bool in = c < c_end;
          const float raw = bias_at(var, in ? brow + (int64_t)(k0 + c) * var.ab_s[3] : 0);
          const float bv = in ? raw : 0.f;
          pr[c] = ex2_approx(__fmaf_rn(bv, kLog2e, __fmaf_rn(__uint_as_float(sr[c]), c2, -l2)));
        }
      }
      // Mask of this query row over keys k0 + c: keys past N, causal c <= m - k0, a window
      // c >= m - W + 1 - k0 (and c <= m + W - 1 - k0 without causal), a 64-block layout the
      // (block row, key block) bit.
      {
        int c_lo = 0, c_hi = min(63, N - 1 - k0);
        if (causal) c_hi = min(c_hi, m - k0);
        if (mask_kind == 2) {
          c_lo = m - W + 1 - k0;
          if (!causal) c_hi = min(c_hi, m + W - 1 - k0);
        }
        const bool on = !bs64 || bit_get(ctl->row_bits[r >> 6], 2 * kt + hh);
        if (__builtin_expect(c_lo > 0 || c_hi < 63 || !on, 0)) {
#pragma unroll
          for (int c = 0; c < 64; ++c) pr[c] = (on && c >= c_lo && c <= c_hi) ? pr[c] : 0.f;
        }
      }
      uint32_t dk[32];
      const uint64_t ndd = f2_pack(-dd, -dd);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const uint64_t dpm = add2(f2_pack(__uint_as_float(dr[2 * c]), __uint_as_float(dr[2 * c + 1])), ndd);
        const uint64_t ds = mul2(f2_pack(pr[2 * c], pr[2 * c + 1]), dpm);
        dk[c] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
        if constexpr (BIAS == 2) {
          // dBias = dS (fp32, before the bf16 rounding of the MMA operand)
          if (dbrow) {
            if (db_vec2 && k0 + 2 * c + 1 < N) {
              *reinterpret_cast<float2*>(dbrow + k0 + 2 * c) = make_float2(f2_lo(ds), f2_hi(ds));
            } else {
              if (k0 + 2 * c < N) dbrow[k0 + 2 * c] = f2_lo(ds);
              if (k0 + 2 * c + 1 < N) dbrow[k0 + 2 * c + 1] = f2_hi(ds);
            }
          }
        }
      }
      // the dS buffer of tile jt was read by dQ(jt-2); reconverge first (the dBias stores
      // above are per row)
      __syncwarp();
      if (jt >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(&ctl->dq_done[jt & 1], ((jt - 2) >> 1) & 1, status, abort_flag))) {
        ok = false;
        break;
      }
      __syncwarp();  // tcgen05.st is warp-aligned: reconverge after the per-row branches above
      tc_fence_after();
      tmem_st32<0>(tmem + lane_off + T_DS + (jt & 1) * 64 + 32 * hh, dk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full[jt & 1]);
    }
    const int nk = jt;
    if constexpr (BIAS == 2) {
      // dBias is 0 on every key tile this query tile does not visit
      if (dbrow) {
        for (int kt = 0; kt < TQ; ++kt) {
          if (kt >= k_lo && kt < k_hi && (!sparse || bit_get(ctl->tile_bits, kt))) continue;
          const int k0 = kt * kT + 64 * hh;
#pragma unroll 4
          for (int c = 0; c < 64; c += 2) {
            if (db_vec2 && k0 + c + 1 < N) {
              *reinterpret_cast<float2*>(dbrow + k0 + c) = make_float2(0.f, 0.f);
            } else {
              if (k0 + c < N) dbrow[k0 + c] = 0.f;
              if (k0 + c + 1 < N) dbrow[k0 + c + 1] = 0.f;
            }
          }
        }
      }
    }
    __syncwarp();
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


using BwdKernel = void (*)(BwdParams);

// The dK/dV and dQ kernels for a head dim, RoPE mode and bias combinator.
template <int BIAS>
inline void select_bwd_kernels(int d, int rk, BwdKernel* kv, BwdKernel* dq) {
  if (d == 128) {
    *kv = rk == kRopeFused ? dkdv_kernel<128, kRopeFused, BIAS>
          : rk == kRopePrerotated ? dkdv_kernel<128, kRopePrerotated, BIAS>
                                  : dkdv_kernel<128, kRopeNone, BIAS>;
    *dq = rk == kRopeFused ? dq_kernel<128, kRopeFused, BIAS>
          : rk == kRopePrerotated ? dq_kernel<128, kRopePrerotated, BIAS>
                                  : dq_kernel<128, kRopeNone, BIAS>;
  } else {
    *kv = rk == kRopeFused ? dkdv_kernel<64, kRopeFused, BIAS>
          : rk == kRopePrerotated ? dkdv_kernel<64, kRopePrerotated, BIAS>
                                  : dkdv_kernel<64, kRopeNone, BIAS>;
    *dq = rk == kRopeFused ? dq_kernel<64, kRopeFused, BIAS>
          : rk == kRopePrerotated ? dq_kernel<64, kRopePrerotated, BIAS>
                                  : dq_kernel<64, kRopeNone, BIAS>;
  }
}

// ALiBi (bias 1) and additive-bias (bias 2) kernels, compiled in bwd_bias.cu.
void select_bwd_bias_kernels(int d, int rk, int bias, BwdKernel* kv, BwdKernel* dq);

}  // namespace afx
