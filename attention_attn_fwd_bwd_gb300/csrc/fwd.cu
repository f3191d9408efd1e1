// Forward attention kernel for sm_103a (AttnFuse paper §4.1 fused RoPE, §2 online softmax,
// §3.1 combinators, §4.3 block skipping), plus the RoPE table and pre-rotation kernels.
//
// One CTA computes two 128-row query sub-tiles that read the same key/value head: either two
// query heads of one GQA group at the same positions (they then share every rotated K tile),
// or two consecutive query tiles of one head. Warp roles (12 warps):
//   warp 0      TMA producer: Q sub-tiles once, then K/V tiles through a ring of stages
//   warp 1      MMA issuer: S_s = Q_s K^T and O_s += P_s V with tcgen05.mma, TMEM accumulators
//   warps 2-3   K rotators (fused RoPE): rotate each K stage in shared memory in place
//   warps 4-7   softmax for sub-tile 0 (one thread per query row)
//   warps 8-11  softmax for sub-tile 1
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D, 256+2D); P_s (bf16)
// overwrites the first 64 columns of S_s. Every wait is bounded (see ptx.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace afx {

namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 384;

template <int D>
struct FwdCfg {
  static constexpr int ST = (D == 128) ? 2 : 4;          // K/V pipeline stages
  static constexpr int PANELS = D / 64;                   // 128-byte swizzle panels per row
  static constexpr uint32_t TILE = 128u * D * 2u;         // bytes of one 128-row tile
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + ST * TILE;
  static constexpr uint32_t OFF_CTL = OFF_V + ST * TILE;
};

struct FwdCtl {
  uint64_t q_full[2], q_ready[2];
  uint64_t k_full[4], k_ready[4], v_full[4], kv_empty[4];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort_flag;
  int lo[2], hi[2], valid[2], q0[2], head[2];
  uint32_t tile_bits[2][kTileWords];      // block-sparse: kv tiles active per sub-tile
  uint32_t row_bits[2][2][kBsWords];      // block-sparse (blk 64): block columns per block row
};

__host__ __device__ constexpr size_t fwd_smem_bytes(int D) {
  return 1024 + (D == 128 ? (2 + 2 * 2) : (2 + 2 * 4)) * (size_t)(128 * D * 2) + sizeof(FwdCtl);
}

__device__ __forceinline__ bool bit_get(const uint32_t* w, int i) {
  return (w[i >> 5] >> (i & 31)) & 1u;
}

__device__ __forceinline__ bool tile_active(const FwdCtl* c, const FwdParams& p, int s, int j) {
  if (!c->valid[s] || j < c->lo[s] || j >= c->hi[s]) return false;
  if (p.var.mask == 3) return bit_get(c->tile_bits[s], j);
  return true;
}

__device__ __forceinline__ int next_tile(const FwdCtl* c, const FwdParams& p, int j, int je) {
  while (j < je && !tile_active(c, p, 0, j) && !tile_active(c, p, 1, j)) ++j;
  return j;
}

// Does tile (s, j) need per-element masking? Uniform for the whole sub-tile.
__device__ __forceinline__ bool tile_needs_mask(const FwdCtl* c, const FwdParams& p, int s,
                                                int j) {
  const int k0 = j * BN, q0 = c->q0[s];
  const int m_hi = min(q0 + BM - 1, p.N - 1);
  const VariantDev& v = p.var;
  if (k0 + BN > p.N) return true;
  if (v.causal && k0 + BN - 1 > q0) return true;
  if (v.mask == 2) {
    if (k0 < m_hi - v.window + 1) return true;
    if (!v.causal && k0 + BN - 1 > q0 + v.window - 1) return true;
  }
  if (v.mask == 3 && v.bs_block == 64) {
    for (int r = 0; r < 2; ++r)
      for (int h = 0; h < 2; ++h)
        if (!bit_get(c->row_bits[s][r], 2 * j + h)) return true;
  }
  return false;
}

}  // namespace

template <int D, int RK>
__global__ void __launch_bounds__(kThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int ST = C::ST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  FwdCtl* ctl = reinterpret_cast<FwdCtl*>(smem + C::OFF_CTL);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const VariantDev& var = p.var;
  constexpr bool ROPE = (RK == kRopeFused);

  // ---------------- work unit ----------------
  const int per_t = p.B * p.pairs;
  const int t = p.num_t - 1 - static_cast<int>(blockIdx.x) / per_t;  // longest first
  const int rem = static_cast<int>(blockIdx.x) % per_t;
  const int b = rem / p.pairs, pr = rem % p.pairs;
  const int TK = (p.N + BN - 1) / BN;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      const int head = p.pair_heads ? 2 * pr + s : pr;
      const int q0 = p.pair_heads ? t * BM : (2 * t + s) * BM;
      ctl->head[s] = head;
      ctl->q0[s] = q0;
      const bool valid = q0 < p.N && head < p.Hq;
      ctl->valid[s] = valid;
      int lo = 0, hi = TK;
      const int m_hi = min(q0 + BM - 1, p.N - 1);
      if (var.causal) hi = min(hi, m_hi / BN + 1);
      if (var.mask == 2) {
        lo = max(0, q0 - var.window + 1) / BN;
        if (!var.causal) hi = min(hi, (m_hi + var.window - 1) / BN + 1);
      }
      ctl->lo[s] = lo;
      ctl->hi[s] = valid ? hi : lo;
    }
    ctl->abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->q_full[s], 1);
      mbar_init(&ctl->q_ready[s], 128);
      mbar_init(&ctl->s_full[s], 1);
      mbar_init(&ctl->p_full[s], 128);
      mbar_init(&ctl->pv_done[s], 1);
    }
    for (int s = 0; s < ST; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_ready[s], 64);
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->kv_empty[s], 1);
    }
    mbar_init(&ctl->mma_final, 1);
    fence_mbar_init();
  }
  if (var.mask == 3) {
    for (int i = tid; i < 2 * kTileWords; i += kThreads) (&ctl->tile_bits[0][0])[i] = 0;
    for (int i = tid; i < 4 * kBsWords; i += kThreads) (&ctl->row_bits[0][0][0])[i] = 0;
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (var.mask == 3) {
    // Mark active kv tiles (and, for 64-blocks, active block columns per block row).
    const int blk = var.bs_block;
    for (int s = 0; s < 2; ++s) {
      if (!ctl->valid[s]) continue;
      const int br0 = ctl->q0[s] / blk;
      const int nbr = BM / blk;  // 2 for blk 64, 1 for blk 128
      const int nb_total = (p.N + blk - 1) / blk;
      for (int r = 0; r < nbr; ++r) {
        const int br = br0 + r;
        if (br >= nb_total) continue;
        const int e0 = var.bs_row_ptr[br], e1 = var.bs_row_ptr[br + 1];
        for (int e = e0 + tid; e < e1; e += kThreads) {
          const int col = var.bs_col_idx[e];
          if (col < 0 || col >= nb_total) continue;
          const int tile = col * blk / BN;
          atomicOr(&ctl->tile_bits[s][tile >> 5], 1u << (tile & 31));
          if (blk == 64) atomicOr(&ctl->row_bits[s][r][col >> 5], 1u << (col & 31));
        }
      }
    }
    __syncthreads();
  }

  const uint32_t tmem = ctl->tmem_base;
  const int jb = min(ctl->lo[0], ctl->lo[1]);
  const int je = max(ctl->hi[0], ctl->hi[1]);
  const int kvh = ctl->head[0] / p.g;
  int* status = p.status;
  volatile int* abort_flag = &ctl->abort_flag;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      for (int s = 0; s < 2; ++s) {
        if (!ctl->valid[s]) continue;
        mbar_arrive_expect_tx(&ctl->q_full[s], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::OFF_Q + s * C::TILE + pn * (BM * 128), &p.tmQ, &ctl->q_full[s],
                      pn * 64, ctl->q0[s], ctl->head[s], b);
      }
      int i = 0;
      for (int j = next_tile(ctl, p, jb, je); j < je; j = next_tile(ctl, p, j + 1, je), ++i) {
        const int s = i % ST;
        if (i >= ST && !mbar_wait(&ctl->kv_empty[s], ((i / ST) - 1) & 1, status, abort_flag))
          break;
        mbar_arrive_expect_tx(&ctl->k_full[s], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::OFF_K + s * C::TILE + pn * (BN * 128), &p.tmK, &ctl->k_full[s],
                      pn * 64, j * BN, kvh, b);
        mbar_arrive_expect_tx(&ctl->v_full[s], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d(smem + C::OFF_V + s * C::TILE + pn * (BN * 128), &p.tmV, &ctl->v_full[s],
                      pn * 64, j * BN, kvh, b);
      }
      // Drain: make sure no copy is still landing in shared memory when the CTA exits.
      const int issued = i;
      for (int k = max(0, issued - ST); k < issued; ++k) {
        mbar_wait(&ctl->k_full[k % ST], (k / ST) & 1, status, nullptr);
        mbar_wait(&ctl->v_full[k % ST], (k / ST) & 1, status, nullptr);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f32acc(128, BN, 0, 0, RK != kRopeNone);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
      bool ok = true;
      for (int s = 0; s < 2 && ok; ++s)
        if (ctl->valid[s]) ok = mbar_wait(&ctl->q_ready[s], 0, status, abort_flag);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      const uint32_t sK = smem_u32(smem + C::OFF_K);
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      auto issue_s = [&](int s, int stage) {
        const uint32_t d_tmem = tmem + s * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
          const uint64_t ad = smem_desc_sw128(sQ + s * C::TILE + koff, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sK + stage * C::TILE + koff, 16, 1024);
          mma_ss(d_tmem, ad, bd, idesc_s, kk > 0);
        }
        mma_commit(&ctl->s_full[s]);
      };
      auto issue_pv = [&](int s, int stage, bool acc) {
        const uint32_t d_tmem = tmem + 256 + s * D;
        const uint32_t p_tmem = tmem + s * 128;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bd = smem_desc_sw128(sV + stage * C::TILE + kk * 2048, BN * 128, 1024);
          mma_ts(d_tmem, p_tmem + kk * 8, bd, idesc_o, (acc || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl->pv_done[s]);
      };
      int cnt_pv[2] = {0, 0};
      bool pv_pend[2] = {false, false};
      int j = next_tile(ctl, p, jb, je);
      if (ok && j < je) {
        ok = mbar_wait(ROPE ? &ctl->k_ready[0] : &ctl->k_full[0], 0, status, abort_flag);
        tc_fence_after();
        if (ok)
          for (int s = 0; s < 2; ++s)
            if (tile_active(ctl, p, s, j)) issue_s(s, 0);
      }
      for (int i = 0; ok && j < je; ++i) {
        const int st = i % ST;
        const int jn = next_tile(ctl, p, j + 1, je);
        const int stn = (i + 1) % ST;
        bool kready = false;
        if (!mbar_wait(&ctl->v_full[st], (i / ST) & 1, status, abort_flag)) break;
        for (int s = 0; s < 2 && ok; ++s) {
          if (tile_active(ctl, p, s, j)) {
            if (!mbar_wait(&ctl->p_full[s], cnt_pv[s] & 1, status, abort_flag)) { ok = false; break; }
            tc_fence_after();
            issue_pv(s, st, cnt_pv[s] > 0);
            ++cnt_pv[s];
            pv_pend[s] = true;
          }
          if (s == 1) mma_commit(&ctl->kv_empty[st]);
          if (jn < je && tile_active(ctl, p, s, jn)) {
            if (!kready) {
              if (!mbar_wait(ROPE ? &ctl->k_ready[stn] : &ctl->k_full[stn], ((i + 1) / ST) & 1,
                             status, abort_flag)) { ok = false; break; }
              kready = true;
            }
            if (pv_pend[s]) {
              if (!mbar_wait(&ctl->pv_done[s], (cnt_pv[s] - 1) & 1, status, abort_flag)) { ok = false; break; }
              pv_pend[s] = false;
            }
            tc_fence_after();
            issue_s(s, stn);
          }
        }
        j = jn;
      }
      // All issued MMAs must finish before TMEM is released.
      mma_commit(&ctl->mma_final);
      mbar_wait(&ctl->mma_final, 0, status, nullptr);
    }
  } else if (warp < 4) {
    // ======================= K rotators (fused RoPE) =======================
    if (ROPE) {
      const int rt = tid - 64;
      constexpr int CP = D / 16;  // chunk pairs per row
      int i = 0;
      for (int j = next_tile(ctl, p, jb, je); j < je; j = next_tile(ctl, p, j + 1, je), ++i) {
        const int st = i % ST;
        if (!mbar_wait(&ctl->k_full[st], (i / ST) & 1, status, abort_flag)) break;
        uint8_t* tile = smem + C::OFF_K + st * C::TILE;
#pragma unroll 4
        for (int it = rt; it < BN * CP; it += 64) {
          const int row = it / CP, c = it % CP;
          const int pos = j * BN + row;
          if (pos >= p.N) continue;
          uint32_t offl, offh;
          if (D == 128) {
            offl = sw128_offset(row, c);
            offh = offl + BN * 128;
          } else {
            offl = sw128_offset(row, c);
            offh = sw128_offset(row, c + 4);
          }
          uint4 lo = *reinterpret_cast<uint4*>(tile + offl);
          uint4 hi = *reinterpret_cast<uint4*>(tile + offh);
          rot_chunk<true>(lo, hi, p.rope_cs + (size_t)pos * (D / 2) + c * 8);
          *reinterpret_cast<uint4*>(tile + offl) = lo;
          *reinterpret_cast<uint4*>(tile + offh) = hi;
        }
        fence_proxy_async_smem();
        mbar_arrive(&ctl->k_ready[st]);
      }
    }
  } else {
    // ======================= softmax (one thread per query row) =======================
    const int s = (warp - 4) >> 2;
    const int wq = warp & 3;                 // TMEM lane quarter
    const int r = wq * 32 + lane;            // row within the sub-tile
    const int q0 = ctl->q0[s];
    const int m = q0 + r;
    const int head = ctl->head[s];
    const bool valid = ctl->valid[s];
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + s * 128;
    const uint32_t tO = tmem + lane_off + 256 + s * D;
    bool ok = true;
    if (valid) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->q_full[s], 0, status, abort_flag));
      if (ok && ROPE && m < p.N) {
        uint8_t* tile = smem + C::OFF_Q + s * C::TILE;
        constexpr int CP = D / 16;
#pragma unroll
        for (int c = 0; c < CP; ++c) {
          uint32_t offl, offh;
          if (D == 128) {
            offl = sw128_offset(r, c);
            offh = offl + BM * 128;
          } else {
            offl = sw128_offset(r, c);
            offh = sw128_offset(r, c + 4);
          }
          uint4 lo = *reinterpret_cast<uint4*>(tile + offl);
          uint4 hi = *reinterpret_cast<uint4*>(tile + offh);
          rot_chunk<true>(lo, hi, p.rope_cs + (size_t)m * (D / 2) + c * 8);
          *reinterpret_cast<uint4*>(tile + offl) = lo;
          *reinterpret_cast<uint4*>(tile + offh) = hi;
        }
        fence_proxy_async_smem();
      }
      mbar_arrive(&ctl->q_ready[s]);
    }
    float m_run = kNegInf, l_run = 0.f;
    int n_done = 0;
    const float scale_log2 = p.scale_log2;
    const float alibi = (var.bias == 1) ? var.slopes[head] * kLog2e : 0.f;
    const int blk_row = (var.mask == 3 && var.bs_block == 64) ? (r >> 6) : 0;
    int jlast = -1;
    for (int j = next_tile(ctl, p, jb, je); valid && ok && j < je; j = next_tile(ctl, p, j + 1, je)) {
      if (!tile_active(ctl, p, s, j)) continue;
      const int k0 = j * BN;
      // Every wait result is voted across the warp so TMEM collectives never diverge.
      if (!__all_sync(0xffffffffu, mbar_wait(&ctl->s_full[s], n_done & 1, status, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t xr[BN];
      tmem_ld32<0>(tS, xr);
      tmem_ld32<32>(tS + 32, xr);
      tmem_ld32<64>(tS + 64, xr);
      tmem_ld32<96>(tS + 96, xr);
      tmem_wait_ld();
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN; ++c) x[c] = __uint_as_float(xr[c]);
      // ---- score combinators (log2 domain) ----
      float mul = scale_log2;
      if (var.bias != 0) {
#pragma unroll
        for (int c = 0; c < BN; ++c) x[c] *= scale_log2;
        mul = 1.f;
        if (var.bias == 1) {
          const float base = alibi * static_cast<float>(k0 - m);
#pragma unroll
          for (int c = 0; c < BN; ++c) x[c] = __fmaf_rn(alibi, static_cast<float>(c), x[c] + base);
        } else {
          const int64_t rowoff = b * var.ab_s[0] + head * var.ab_s[1] + (int64_t)m * var.ab_s[2];
          if (var.add_bias_bf16) {
            const __nv_bfloat16* ab = static_cast<const __nv_bfloat16*>(var.add_bias) + rowoff;
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (k0 + c < p.N && m < p.N)
                x[c] += __bfloat162float(ab[(int64_t)(k0 + c) * var.ab_s[3]]) * kLog2e;
          } else {
            const float* ab = static_cast<const float*>(var.add_bias) + rowoff;
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (k0 + c < p.N && m < p.N) x[c] += ab[(int64_t)(k0 + c) * var.ab_s[3]] * kLog2e;
          }
        }
      }
      if (tile_needs_mask(ctl, p, s, j)) {
        int c_lo = 0, c_hi = min(BN - 1, p.N - 1 - k0);
        if (var.causal) c_hi = min(c_hi, m - k0);
        if (var.mask == 2) {
          c_lo = max(c_lo, m - var.window + 1 - k0);
          if (!var.causal) c_hi = min(c_hi, m + var.window - 1 - k0);
        }
        bool h0 = true, h1 = true;
        if (var.mask == 3 && var.bs_block == 64) {
          h0 = bit_get(ctl->row_bits[s][blk_row], 2 * j);
          h1 = bit_get(ctl->row_bits[s][blk_row], 2 * j + 1);
        }
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const bool keep = (c >= c_lo) && (c <= c_hi) && (c < 64 ? h0 : h1);
          x[c] = keep ? x[c] : kNegInf;
        }
      }
      float mx = x[0];
#pragma unroll
      for (int c = 1; c < BN; ++c) mx = fmaxf(mx, x[c]);
      mx *= mul;
      // ---- online softmax with lazy rescaling (exact after the final division) ----
      const float m_new = fmaxf(m_run, mx);
      float m_use = m_run;
      bool rescale = false;
      if (n_done == 0) {
        m_use = m_new;
      } else if (m_new > m_run + 8.0f) {
        m_use = m_new;
        rescale = true;
      }
      const float nb = (m_use == kNegInf) ? 0.f : -m_use;
      float sum = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float p0 = ex2_approx(__fmaf_rn(x[2 * c], mul, nb));
        const float p1 = ex2_approx(__fmaf_rn(x[2 * c + 1], mul, nb));
        sum += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      tmem_st32<0>(tS, pk);
      tmem_st32<32>(tS + 32, pk);
      tmem_wait_st();
      if (n_done > 0) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&ctl->pv_done[s], (n_done - 1) & 1, status, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // tcgen05.ld/st are warp-collective: rescale the whole warp's rows when any row needs
      // it (alpha = 1 for rows that do not).
      if (__any_sync(0xffffffffu, rescale)) {
        const float alpha = rescale ? ex2_approx(m_run - m_use) : 1.f;
        l_run *= alpha;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tO + ch * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + ch * 32, o);
        }
        tmem_wait_st();
      }
      l_run += sum;
      m_run = m_use;
      tc_fence_before();
      mbar_arrive(&ctl->p_full[s]);
      if (var.visits && r == 0) {
        const int TQ = (p.N + BM - 1) / BM;
        var.visits[((static_cast<int64_t>(b) * p.Hq + head) * TQ + q0 / BM) * TK + j] = 1;
      }
      ++n_done;
      jlast = j;
    }
    (void)jlast;
    // ---- epilogue: O = acc / l, LSE = ln(sum) ----
    if (valid) {
      if (ok && n_done > 0) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&ctl->pv_done[s], (n_done - 1) & 1, status, abort_flag));
        tc_fence_after();
      }
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      __nv_bfloat16* orow = p.out + b * p.o_sb + head * p.o_sh + (int64_t)m * p.o_sn;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        if (ok && n_done > 0) {
          tmem_ld32(tO + ch * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (m < p.N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[v4 * 8 + 0]) * inv, __uint_as_float(o[v4 * 8 + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[v4 * 8 + 2]) * inv, __uint_as_float(o[v4 * 8 + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[v4 * 8 + 4]) * inv, __uint_as_float(o[v4 * 8 + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[v4 * 8 + 6]) * inv, __uint_as_float(o[v4 * 8 + 7]) * inv);
            dst[v4] = w;
          }
        }
      }
      if (p.lse && m < p.N)
        p.lse[(static_cast<int64_t>(b) * p.Hq + head) * p.N + m] =
            (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : kNegInf;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------------------------
// RoPE (cos, sin) table: cs[pos * half + i] for pos < N (paper §4.1, staged per tile).
// ---------------------------------------------------------------------------------------------
__global__ void rope_table_kernel(float2* __restrict__ cs, int N, int half, RopeFreqs f) {
  const int64_t total = static_cast<int64_t>(N) * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int pos = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
    float c, s;
    rope_cossin(static_cast<float>(pos), f.hi[i], f.lo[i], &c, &s);
    cs[idx] = make_float2(c, s);
  }
}

// ---------------------------------------------------------------------------------------------
// Pre-rotation (paper Fig. 1a): out[b,h,n,:] = R_n x[b,h,n,:], out contiguous. One thread per
// (row, chunk pair); HBM-bound elementwise pass.
// ---------------------------------------------------------------------------------------------
template <bool OUT_F16>
__global__ void prerotate_kernel(const __nv_bfloat16* __restrict__ x, int64_t sb, int64_t sh,
                                 int64_t sn, __nv_bfloat16* __restrict__ out, int H, int N, int d,
                                 const float2* __restrict__ cs, int64_t rows) {
  const int cp = d / 16;
  const int64_t total = rows * cp;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = idx / cp;
    const int c = static_cast<int>(idx % cp);
    const int n = static_cast<int>(row % N);
    const int64_t bh = row / N;
    const int h = static_cast<int>(bh % H);
    const int64_t bb = bh / H;
    const __nv_bfloat16* src = x + bb * sb + h * sh + n * sn;
    uint4 lo = *reinterpret_cast<const uint4*>(src + c * 8);
    uint4 hi = *reinterpret_cast<const uint4*>(src + d / 2 + c * 8);
    rot_chunk<OUT_F16>(lo, hi, cs + (size_t)n * (d / 2) + c * 8);
    __nv_bfloat16* dst = out + row * d;
    *reinterpret_cast<uint4*>(dst + c * 8) = lo;
    *reinterpret_cast<uint4*>(dst + d / 2 + c * 8) = hi;
  }
}

// ---------------------------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------------------------
size_t fwd_smem_size(int d) { return fwd_smem_bytes(d); }

cudaError_t launch_fwd(const FwdParams& p, int d, int rope_kind, int grid, cudaStream_t stream) {
  const size_t smem = fwd_smem_bytes(d);
  void (*fn)(FwdParams) = nullptr;
  if (d == 128)
    fn = rope_kind == kRopeFused ? fwd_kernel<128, kRopeFused>
         : rope_kind == kRopePrerotated ? fwd_kernel<128, kRopePrerotated>
                                        : fwd_kernel<128, kRopeNone>;
  else
    fn = rope_kind == kRopeFused ? fwd_kernel<64, kRopeFused>
         : rope_kind == kRopePrerotated ? fwd_kernel<64, kRopePrerotated>
                                        : fwd_kernel<64, kRopeNone>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  fn<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* cs, int N, int half, const RopeFreqs& f,
                              cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(N) * half;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<int64_t>((total + threads - 1) / threads, 152 * 8));
  rope_table_kernel<<<blocks, threads, 0, stream>>>(cs, N, half, f);
  return cudaGetLastError();
}

cudaError_t launch_prerotate(const void* x, const int64_t* strides, void* out, int B, int H,
                             int N, int d, const float2* cs, bool out_f16, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(B) * H * N;
  const int64_t total = rows * (d / 16);
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<int64_t>((total + threads - 1) / threads, 152 * 16));
  auto fn = out_f16 ? prerotate_kernel<true> : prerotate_kernel<false>;
  fn<<<blocks, threads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), strides[0], strides[1], strides[2],
      static_cast<__nv_bfloat16*>(out), H, N, d, cs, rows);
  return cudaGetLastError();
}

}  // namespace afx
