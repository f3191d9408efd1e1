// Forward attention kernel for head dim 64 on sm_103a (AttnFuse paper §4.1 fused RoPE, §2
// online softmax, §3.1 combinators, §4.3 block skipping), plus the RoPE table and pre-rotation
// kernels. Head dim 128 runs on the persistent CTA-pair kernel (fwd_pp.cuh).
//
// One CTA computes two 128-row query sub-tiles that read the same key/value head: either two
// query heads of one GQA group at the same positions (they then share every rotated K tile),
// or two consecutive query tiles of one head. Warp roles (16 warps, 4 warpgroups):
//   warp 0      TMA producer: Q sub-tiles once, then K and V tiles through separate rings
//   warp 1      MMA issuer: S_s = Q_s K^T and O_s += P_s V with tcgen05.mma, TMEM accumulators
//   warps 4-7   softmax for sub-tile 0 (one thread per query row)
//   warps 8-11  softmax for sub-tile 1
//   warps 12-15 K rotators (fused RoPE): rotate each 128-key tile of K once per call (by
//               whichever CTA claims it first) into an fp16 workspace copy K' that the
//               producers load with TMA, or (short or windowed sequences) each CTA's K stages
//               in shared memory in place; (cos, sin) advance down the rows by angle addition
// Registers are re-balanced with setmaxnreg: 64 (producers), 80 (rotators), 184 (softmax).
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
constexpr int kThreads = 512;
constexpr uint32_t kRegsProducer = 64;   // warpgroup 0: TMA and MMA issue
constexpr uint32_t kRegsRotator = 80;    // warpgroup 3: K rotation
constexpr uint32_t kRegsSoftmax = 184;   // warpgroups 1, 2
static_assert(kRegsProducer + kRegsRotator + 2 * kRegsSoftmax <= 4 * (65536 / kThreads),
              "register split exceeds the registers the CTA is launched with");

template <int D>
struct FwdCfg {
  static constexpr int KST = (D == 128) ? 3 : 5;          // K stages (released after S)
  static constexpr int VST = (D == 128) ? 2 : 4;          // V stages (released after PV)
  static constexpr int PANELS = D / 64;                   // 128-byte swizzle panels per row
  static constexpr uint32_t TILE = 128u * D * 2u;         // bytes of one 128-row tile
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + KST * TILE;
  static constexpr uint32_t OFF_CTL = OFF_V + VST * TILE;
};

struct FwdCtl {
  uint64_t q_full[2], q_ready[2];
  uint64_t k_full[5], k_ready[5], k_empty[5];
  uint64_t v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort_flag;
  int lo[2], hi[2], valid[2], q0[2], head[2];
  uint32_t tile_bits[2][kTileWords];      // block-sparse: kv tiles active per sub-tile
  uint32_t row_bits[2][2][kBsWords];      // block-sparse (blk 64): block columns per block row
};

__host__ __device__ constexpr size_t fwd_smem_bytes(int D) {
  return 1024 + (D == 128 ? (2 + 3 + 2) : (2 + 5 + 4)) * (size_t)(128 * D * 2) + sizeof(FwdCtl);
}
static_assert(1024 + 7 * 32768 + sizeof(FwdCtl) <= 232448, "d=128 shared memory budget");

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
  constexpr int KST = C::KST, VST = C::VST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  FwdCtl* ctl = reinterpret_cast<FwdCtl*>(smem + C::OFF_CTL);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const VariantDev& var = p.var;
  constexpr bool ROPE = (RK == kRopeFused);
  // fused RoPE, K rotated once per call into the workspace copy K' (the host picks this when
  // K tiles are re-read by enough query tiles), else each CTA rotates its K stages in place
  const bool kshare = ROPE && p.k_rot != nullptr;

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
    for (int s = 0; s < KST; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_ready[s], 128);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
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

  if (warp < 4) {
    setmaxnreg_dec<kRegsProducer>();
    if (warp == 0 && lane == 0) {
      // ======================= TMA producer =======================
      // One SM's TMA engine completes copies in issue order at a bounded byte rate, so copies
      // are issued in the order the MMAs need them: Q, K(0), then K(i+1) ahead of V(i).
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      // Q is read once; K and V are re-read by every query tile of the group.
      const uint64_t pol_stream = l2_policy_evict_first();
      const uint64_t pol_keep = l2_policy_evict_last();
      for (int s = 0; s < 2; ++s) {
        if (!ctl->valid[s]) continue;
        mbar_arrive_expect_tx(&ctl->q_full[s], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d_hint(smem + C::OFF_Q + s * C::TILE + pn * (BM * 128), &p.tmQ,
                           &ctl->q_full[s], pn * 64, ctl->q0[s], ctl->head[s], b, pol_stream);
      }
      int ik = 0, iv = 0;
      int jk = next_tile(ctl, p, jb, je), jv = jk;
      bool go = true;
      while (go && (jk < je || jv < je)) {
        if (jk < je) {
          const int s = ik % KST;
          if (ik >= KST && !mbar_wait(&ctl->k_empty[s], ((ik / KST) - 1) & 1, status, abort_flag)) {
            go = false;
            break;
          }
          // fused RoPE: K' of tile jk, rotated once per call by whichever CTA claimed it
          if (kshare && !flag_wait(p.k_sync + (b * p.Hkv + kvh) * TK + jk, 2u, status, abort_flag)) {
            go = false;
            break;
          }
          mbar_arrive_expect_tx(&ctl->k_full[s], C::TILE);
          for (int pn = 0; pn < C::PANELS; ++pn)
            tma_load_4d_hint(smem + C::OFF_K + s * C::TILE + pn * (BN * 128), &p.tmK,
                             &ctl->k_full[s], pn * 64, jk * BN, kvh, b, pol_keep);
          ++ik;
          jk = next_tile(ctl, p, jk + 1, je);
        }
        if (jv < je && (ik >= 2 || jk >= je)) {
          const int s = iv % VST;
          if (iv >= VST && !mbar_wait(&ctl->v_empty[s], ((iv / VST) - 1) & 1, status, abort_flag)) {
            go = false;
            break;
          }
          mbar_arrive_expect_tx(&ctl->v_full[s], C::TILE);
          for (int pn = 0; pn < C::PANELS; ++pn)
            tma_load_4d_hint(smem + C::OFF_V + s * C::TILE + pn * (BN * 128), &p.tmV,
                             &ctl->v_full[s], pn * 64, jv * BN, kvh, b, pol_keep);
          ++iv;
          jv = next_tile(ctl, p, jv + 1, je);
        }
      }
      // Drain: no copy may still be landing in shared memory when the CTA exits.
      for (int k = max(0, ik - KST); k < ik; ++k)
        mbar_wait(&ctl->k_full[k % KST], (k / KST) & 1, status, nullptr);
      for (int k = max(0, iv - VST); k < iv; ++k)
        mbar_wait(&ctl->v_full[k % VST], (k / VST) & 1, status, nullptr);
    } else if (warp == 1 && lane == 0) {
      // ======================= MMA issuer =======================
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
        ok = mbar_wait((ROPE && !kshare) ? &ctl->k_ready[0] : &ctl->k_full[0], 0, status, abort_flag);
        tc_fence_after();
        if (ok) {
          for (int s = 0; s < 2; ++s)
            if (tile_active(ctl, p, s, j)) {
              issue_s(s, 0);
            }
          mma_commit(&ctl->k_empty[0]);
        }
      }
      for (int i = 0; ok && j < je; ++i) {
        const int vs = i % VST;
        const int jn = next_tile(ctl, p, j + 1, je);
        const int kn = (i + 1) % KST;
        bool kready = false;
        if (!mbar_wait(&ctl->v_full[vs], (i / VST) & 1, status, abort_flag)) break;
        for (int s = 0; s < 2 && ok; ++s) {
          if (tile_active(ctl, p, s, j)) {
            if (!mbar_wait(&ctl->p_full[s], cnt_pv[s] & 1, status, abort_flag)) { ok = false; break; }
            tc_fence_after();
            issue_pv(s, vs, cnt_pv[s] > 0);
            ++cnt_pv[s];
            pv_pend[s] = true;
          }
          if (s == 1) mma_commit(&ctl->v_empty[vs]);
          if (jn < je && tile_active(ctl, p, s, jn)) {
            if (!kready) {
              if (!mbar_wait((ROPE && !kshare) ? &ctl->k_ready[kn] : &ctl->k_full[kn],
                             ((i + 1) / KST) & 1, status, abort_flag)) {
                ok = false;
                break;
              }
              kready = true;
            }
            if (pv_pend[s]) {
              if (!mbar_wait(&ctl->pv_done[s], (cnt_pv[s] - 1) & 1, status, abort_flag)) { ok = false; break; }
              pv_pend[s] = false;
            }
            tc_fence_after();
            issue_s(s, kn);
          }
        }
        if (ok && jn < je) mma_commit(&ctl->k_empty[kn]);
        j = jn;
      }
      // All issued MMAs must finish before TMEM is released.
      mma_commit(&ctl->mma_final);
      mbar_wait(&ctl->mma_final, 0, status, nullptr);
    }
  } else if (warp >= 12) {
    // ======================= K rotators (fused RoPE) =======================
    setmaxnreg_dec<kRegsRotator>();
    if (ROPE && kshare) {
      // K' = R_n K is made once per 128-key tile and call: the four rotator warps walk this
      // CTA's tiles, warp w taking every fourth; the first warp of any CTA to claim a tile (a
      // compare-and-swap on its flag: 0 untouched, 1 claimed, 2 done) rotates it from global
      // memory into the fp16 copy in the workspace and releases the flag, and the producer
      // copies K' with TMA once the flag reads 2. A claimed tile is finished by a warp that
      // waits on nothing, and an unclaimed one by this CTA's own rotators, so no wait is
      // endless. Lane (c, rl) rotates chunk pair c (dims 8c.., D/2+8c..) of rows rg + RG k
      // of the chains rg = rl + 8i, each starting from its table entry and stepping the
      // (cos, sin) of RG positions per row (the chains of the pre-rotation pass, so K' is
      // bit-identical to its output).
      constexpr int CP = D / 16;    // chunk pairs per row
      constexpr int RG = 128 / CP;  // chains per tile; a chain holds rows rg, rg + RG, ...
      static_assert(CP == 4, "the rotator lane map assumes head dim 64");
      constexpr uint64_t kSign2 = 0x8000000080000000ull;
      const int wr = warp - 12;
      const int c = lane & 3, rl = lane >> 2;
      const int kN = p.N;
      uint64_t wc2[4], ws2[4], nws2[4];
      {
        float wc[8], ws[8];
        load_cs8(p.rope_cs + (size_t)RG * (D / 2) + c * 8, wc, ws);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          wc2[w] = f2_pack(wc[2 * w], wc[2 * w + 1]);
          ws2[w] = f2_pack(ws[2 * w], ws[2 * w + 1]);
          nws2[w] = ws2[w] ^ kSign2;
        }
      }
      const uint64_t pol_tab = l2_policy_evict_last();
      const uint64_t pol_in = l2_policy_evict_first();
      const uint64_t pol_out = l2_policy_evict_last();
      const int bh = b * p.Hkv + kvh;
      const __nv_bfloat16* src = p.k_raw + b * p.k_sb + kvh * p.k_sh;
      uint16_t* dst = p.k_rot + (int64_t)bh * kN * D;
      uint32_t f16max = 0;  // |K'| as fp16 bits, per half
      int i = 0;
      for (int j = next_tile(ctl, p, jb, je); j < je; j = next_tile(ctl, p, j + 1, je), ++i) {
        if ((i & 3) != wr) continue;
        uint32_t* flag = p.k_sync + bh * TK + j;
        uint32_t mine = 0;
        if (lane == 0 && *reinterpret_cast<volatile uint32_t*>(flag) == 0u)
          mine = atomicCAS(flag, 0u, 1u) == 0u ? 1u : 0u;
        if (!__shfl_sync(0xffffffffu, mine, 0)) continue;
        const int n0 = j * BN;
#pragma unroll 1
        for (int ci = 0; ci < RG / 8; ++ci) {
          const int rg = rl + 8 * ci;
          float4 pre[4];
          {
            const float4* t = reinterpret_cast<const float4*>(
                p.rope_cs + (size_t)min(n0 + rg, kN - 1) * (D / 2) + c * 8);
#pragma unroll
            for (int w = 0; w < 4; ++w) pre[w] = ldg_f4_hint(t + w, pol_tab);
          }
          uint4 lo[CP], hi[CP];
#pragma unroll
          for (int k = 0; k < CP; ++k) {
            const __nv_bfloat16* row = src + (int64_t)min(n0 + rg + RG * k, kN - 1) * p.k_sn + c * 8;
            lo[k] = ldg_u4_hint(row, pol_in);
            hi[k] = ldg_u4_hint(row + D / 2, pol_in);
          }
          uint64_t c2[4], s2[4], ns2[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            c2[w] = f2_pack(pre[w].x, pre[w].z);
            s2[w] = f2_pack(pre[w].y, pre[w].w);
            ns2[w] = s2[w] ^ kSign2;
          }
#pragma unroll
          for (int k = 0; k < CP; ++k) {
            rot_chunk_cs2<true>(lo[k], hi[k], c2, s2, ns2);
            f16max = f16_absmax(f16_absmax(f16max, lo[k]), hi[k]);
            if (k + 1 < CP) advance_cs2(c2, s2, ns2, wc2, ws2, nws2);
          }
#pragma unroll
          for (int k = 0; k < CP; ++k) {
            const int n = n0 + rg + RG * k;
            if (n < kN) {
              uint16_t* out = dst + (int64_t)n * D + c * 8;
              stg_u4_hint(out, lo[k], pol_out);
              stg_u4_hint(out + D / 2, hi[k], pol_out);
            }
          }
        }
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(flag, 2u);
      }
      report_f16_range(status, f16max);
    } else if (ROPE) {
      // each CTA rotates its own K stages in place after they land
      constexpr int CP = D / 16;    // chunk pairs per row
      constexpr int RG = 128 / CP;  // row groups; a thread owns rows rg, rg + RG, ...
      const int rt = tid - 384;
      const int c = rt % CP, rg = rt / CP;
      uint64_t wc2[4], ws2[4], nws2[4];
      {
        float wc[8], ws[8];
        load_cs8(p.rope_cs + (size_t)RG * (D / 2) + c * 8, wc, ws);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          wc2[w] = f2_pack(wc[2 * w], wc[2 * w + 1]);
          ws2[w] = f2_pack(ws[2 * w], ws[2 * w + 1]);
          nws2[w] = f2_pack(-ws[2 * w], -ws[2 * w + 1]);
        }
      }
      uint32_t f16max = 0;  // |K'| as fp16 bits, per half
      int i = 0;
      for (int j = next_tile(ctl, p, jb, je); j < je; j = next_tile(ctl, p, j + 1, je), ++i) {
        const int st = i % KST;
        uint64_t c2[4] = {0, 0, 0, 0}, s2[4] = {0, 0, 0, 0}, ns2[4] = {0, 0, 0, 0};
        const int pos0 = j * BN + rg;
        if (pos0 < p.N) {
          float cc[8], ss[8];
          load_cs8(p.rope_cs + (size_t)pos0 * (D / 2) + c * 8, cc, ss);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            c2[w] = f2_pack(cc[2 * w], cc[2 * w + 1]);
            s2[w] = f2_pack(ss[2 * w], ss[2 * w + 1]);
            ns2[w] = f2_pack(-ss[2 * w], -ss[2 * w + 1]);
          }
        }
        if (!mbar_wait(&ctl->k_full[st], (i / KST) & 1, status, abort_flag)) break;
        uint8_t* tile = smem + C::OFF_K + st * C::TILE;
#pragma unroll
        for (int k = 0; k < CP; ++k) {
          const int row = rg + RG * k;
          if (j * BN + row < p.N) {
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
            rot_chunk_cs2<true>(lo, hi, c2, s2, ns2);
            f16max = f16_absmax(f16_absmax(f16max, lo), hi);
            *reinterpret_cast<uint4*>(tile + offl) = lo;
            *reinterpret_cast<uint4*>(tile + offh) = hi;
          }
          if (k + 1 < CP) advance_cs2(c2, s2, ns2, wc2, ws2, nws2);
        }
        fence_proxy_async_smem();
        mbar_arrive(&ctl->k_ready[st]);
      }
      report_f16_range(status, f16max);
    }
  } else {
    // ======================= softmax (one thread per query row) =======================
    setmaxnreg_inc<kRegsSoftmax>();
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
    uint32_t qmax = 0;  // |Q'| as fp16 bits, per half (fused RoPE)
    if (valid) {
      // Rotate this sub-tile's Q in place, with coalesced table reads: a warp instruction
      // covers whole table rows (lane f holds entries 2f, 2f+1 of its row, i.e. dims 2f, 2f+1
      // and their partners d/2+2f, d/2+2f+1). The reads are issued before Q lands. Same
      // arithmetic per element as a row-per-thread rotation; rows past N are not rotated.
      constexpr int F4 = D / 4;           // float4 table entries per row
      constexpr int RPI = 32 / F4;        // rows per warp instruction
      constexpr int RPT = BM / (4 * RPI); // rows per thread: rows RPI wq + rsub + 8 k
      static_assert(4 * RPI == 8, "rows of a thread are 8 positions apart");
      const int f = lane % F4, rsub = lane / F4;
      // the query-tile recurrence (query_cs8): start at position q0 + (row % 8), step 8
      float4 cs = make_float4(0.f, 0.f, 0.f, 0.f), wstep = cs;
      if (ROPE) {
        const uint64_t pol_tab = l2_policy_evict_last();  // the table stays in L2
        const float4* tab = reinterpret_cast<const float4*>(p.rope_cs);
        cs = ldg_f4_hint(tab + (size_t)min(q0 + RPI * wq + rsub, p.N - 1) * F4 + f, pol_tab);
        wstep = ldg_f4_hint(tab + (size_t)8 * F4 + f, pol_tab);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->q_full[s], 0, status, abort_flag));
      if (ok && ROPE) {
        uint8_t* tile = smem + C::OFF_Q + s * C::TILE;
        const uint32_t within = static_cast<uint32_t>(f & 3) * 4u;
#pragma unroll
        for (int k = 0; k < RPT; ++k) {
          const int rr = RPI * wq + rsub + 4 * RPI * k;
          if (q0 + rr < p.N) {
            const uint32_t offl = sw128_offset(rr, f >> 2) + within;
            const uint32_t offh = (D == 128) ? offl + BM * 128 : sw128_offset(rr, (f >> 2) + 4) + within;
            const uint32_t l2w = *reinterpret_cast<const uint32_t*>(tile + offl);
            const uint32_t h2w = *reinterpret_cast<const uint32_t*>(tile + offh);
            float yl0, yh0, yl1, yh1;
            rot_pair(bf16lo_to_f32(l2w), bf16lo_to_f32(h2w), cs.x, cs.y, yl0, yh0);
            rot_pair(bf16hi_to_f32(l2w), bf16hi_to_f32(h2w), cs.z, cs.w, yl1, yh1);
            const uint32_t wl = pack_f16x2_sat(yl0, yl1), wh = pack_f16x2_sat(yh0, yh1);
            qmax = f16_absmax(f16_absmax(qmax, wl), wh);
            *reinterpret_cast<uint32_t*>(tile + offl) = wl;
            *reinterpret_cast<uint32_t*>(tile + offh) = wh;
          }
          if (k + 1 < RPT) {  // next row of this thread: 8 positions on (advance_cs8 order)
            float c0, s0, c1, s1;
            rot_pair(cs.x, cs.y, wstep.x, wstep.y, c0, s0);
            rot_pair(cs.z, cs.w, wstep.z, wstep.w, c1, s1);
            cs = make_float4(c0, s0, c1, s1);
          }
        }
        fence_proxy_async_smem();
        report_f16_range(status, qmax);
      }
      mbar_arrive(&ctl->q_ready[s]);
    }
    float m_run = kNegInf, l_run = 0.f;
    int n_done = 0;
    const float scale_log2 = p.scale_log2;
    const float alibi = (var.bias == 1) ? var.slopes[head] * kLog2e : 0.f;
    const int blk_row = (var.mask == 3 && var.bs_block == 64) ? (r >> 6) : 0;
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
          // Branch-free loads (lanes past the sequence end read element 0 and drop it), so the
          // warp stays converged for the warp-collective TMEM operations that follow.
          const int c_end = (m < p.N) ? min(BN, p.N - k0) : 0;
          if (var.add_bias_bf16) {
            const __nv_bfloat16* ab = static_cast<const __nv_bfloat16*>(var.add_bias);
#pragma unroll
            for (int c = 0; c < BN; ++c) {
              const float raw = __bfloat162float(ab[c < c_end ? rowoff + (int64_t)(k0 + c) * var.ab_s[3] : 0]);
              x[c] += (c < c_end ? raw : 0.f) * kLog2e;
            }
          } else {
            const float* ab = static_cast<const float*>(var.add_bias);
#pragma unroll
            for (int c = 0; c < BN; ++c) {
              const float raw = ab[c < c_end ? rowoff + (int64_t)(k0 + c) * var.ab_s[3] : 0];
              x[c] += (c < c_end ? raw : 0.f) * kLog2e;
            }
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
      // row max: 8 independent 3-input chains, then a small tree
      float mp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mp[k] = fmaxf(x[2 * k], x[2 * k + 1]);
#pragma unroll
      for (int i2 = 1; i2 < BN / 16; ++i2)
#pragma unroll
        for (int k = 0; k < 8; ++k) mp[k] = max3f(mp[k], x[16 * i2 + 2 * k], x[16 * i2 + 2 * k + 1]);
      float mx = max3f(max3f(mp[0], mp[1], mp[2]), max3f(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
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
      const uint64_t mul2v = f2_pack(mul, mul), nb2 = f2_pack(nb, nb);
      uint64_t acc2[4] = {0, 0, 0, 0};
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const uint64_t a = fma2(f2_pack(x[2 * c], x[2 * c + 1]), mul2v, nb2);
        const float p0 = ex2_approx(f2_lo(a)), p1 = ex2_approx(f2_hi(a));
        acc2[c & 3] = add2(acc2[c & 3], f2_pack(p0, p1));
        pk[c] = pack_bf16x2(p0, p1);
      }
      const uint64_t acc = add2(add2(acc2[0], acc2[1]), add2(acc2[2], acc2[3]));
      const float sum = f2_lo(acc) + f2_hi(acc);
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
    }
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
            __stcs(dst + v4, w);  // streaming store: O is not re-read
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
// Pre-rotation (paper Fig. 1a): out[b,h,n,:] = R_n x[b,h,n,:], out contiguous. HBM-bound
// elementwise pass.
//
// The (cos, sin) of a row follow the recurrence the kernels use on chip: row r of a block of
// BLK rows at n0 starts from the table entry of position n0 + r % RG and advances r / RG times
// by the entry of position RG (queries of the forward: RG = 8, BLK = 128; keys: RG = 128 / (d/16)
// in blocks of 64 or 128; RG = BLK = 1 reads every row's own entry). One thread walks one such
// chain (rows n0 + q, n0 + q + RG, ...) for one chunk pair, taking one angle-addition step per
// row, so the rotated values are bit-identical to the kernels' while the pass stays bound by
// memory rather than by recomputing the chain for every row.
// ---------------------------------------------------------------------------------------------
template <bool OUT_F16>
__global__ void prerotate_kernel(const __nv_bfloat16* __restrict__ x, int64_t sb, int64_t sh,
                                 int64_t sn, __nv_bfloat16* __restrict__ out, int H, int N, int d,
                                 const float2* __restrict__ cs, int RG, int BLK, int64_t chains,
                                 int* status) {
  const int cp = d / 16;
  const int nblk = (N + BLK - 1) / BLK;
  uint32_t f16max = 0;  // fp16 output: |x'| as fp16 bits, per half
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < chains;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = static_cast<int>(idx % cp);
    int64_t t = idx / cp;
    const int q = static_cast<int>(t % RG);
    t /= RG;
    const int blk = static_cast<int>(t % nblk);
    const int64_t bh = t / nblk;
    const int h = static_cast<int>(bh % H);
    const int64_t bb = bh / H;
    const int n0 = blk * BLK + q;
    if (n0 >= N) continue;
    float cc[8], ss[8], wc[8], ws[8];
    load_cs8(cs + (size_t)n0 * (d / 2) + c * 8, cc, ss);
    if (BLK > RG) load_cs8(cs + (size_t)RG * (d / 2) + c * 8, wc, ws);
    const __nv_bfloat16* src = x + bb * sb + h * sh + c * 8;
    __nv_bfloat16* dst = out + (bh * N) * d + c * 8;
#pragma unroll 4
    for (int n = n0; n < blk * BLK + BLK && n < N; n += RG) {
      uint4 lo = *reinterpret_cast<const uint4*>(src + n * sn);
      uint4 hi = *reinterpret_cast<const uint4*>(src + n * sn + d / 2);
      rot_chunk_cs<OUT_F16>(lo, hi, cc, ss);
      if (OUT_F16) f16max = f16_absmax(f16_absmax(f16max, lo), hi);
      *reinterpret_cast<uint4*>(dst + (int64_t)n * d) = lo;
      *reinterpret_cast<uint4*>(dst + (int64_t)n * d + d / 2) = hi;
      if (n + RG < blk * BLK + BLK) advance_cs8(cc, ss, wc, ws);
    }
  }
  if (OUT_F16) report_f16_range(status, f16max);
}

// ---------------------------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------------------------
size_t fwd_smem_size(int d) { return fwd_smem_bytes(d); }

cudaError_t launch_fwd(const FwdParams& p, int d, int rope_kind, int grid, cudaStream_t stream) {
  if (d != 64) return cudaErrorInvalidValue;  // head dim 128 runs on the CTA-pair kernel (fwd_pp.cuh)
  const size_t smem = fwd_smem_bytes(d);
  void (*fn)(FwdParams) = rope_kind == kRopeFused        ? fwd_kernel<64, kRopeFused>
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
                             int N, int d, const float2* cs, bool out_f16, int block,
                             cudaStream_t stream, int* status) {
  // the recurrence of the target kernel (see prerotate_kernel)
  const int cp = d / 16;
  int RG = 1, BLK = 1;                       // block == 0: each row's own table entry
  if (block < 0) {                           // forward queries
    RG = 8;
    BLK = 128;
  } else if (block > 0) {                    // forward keys (fp16) or backward operands (bf16)
    RG = 128 / cp;
    BLK = out_f16 ? (d == 128 ? 64 : 128) : 128;
  }
  const int64_t chains = static_cast<int64_t>(B) * H * ((N + BLK - 1) / BLK) * RG * cp;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<int64_t>((chains + threads - 1) / threads, 152 * 16));
  void (*fn)(const __nv_bfloat16*, int64_t, int64_t, int64_t, __nv_bfloat16*, int, int, int,
             const float2*, int, int, int64_t, int*) = out_f16 ? prerotate_kernel<true> : prerotate_kernel<false>;
  fn<<<blocks, threads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), strides[0], strides[1], strides[2],
      static_cast<__nv_bfloat16*>(out), H, N, d, cs, RG, BLK, chains, status);
  return cudaGetLastError();
}

}  // namespace afx

