// Persistent forward attention for head dims 128 and 64 on CTA pairs with two query slots per CTA
// (AttnFuse paper §4.1 fused RoPE, §2 online softmax, §3.1 combinators, §4.3 block skipping).
//
// A cluster of two CTAs (one per SM) walks a static list of work units. A unit is four
// 128-row query tiles that read one KV head: CTA r, slot s holds tile e = 2s + r. With a GQA
// group of at least four heads the four tiles are four heads at one position, so every K tile
// that is loaded (and, with fused RoPE, rotated) serves 512 query rows; otherwise the tiles are
// two heads at two positions or four positions of one head.
//
// Each slot is an independent online softmax over its own rows, with its own score buffer S_s
// and output accumulator O_s in tensor memory and its own P buffer in shared memory. Per kv
// tile i, slot s runs
//     S_s = Q_s K(i)    as soon as the slot's softmax has read S_s of tile i-1 into registers,
//     O_s += P_s V(i-1) once that softmax has written P_s (bf16) to shared memory,
// as M = 256 cta_group::2 MMAs (both CTAs' rows of a slot at once; each CTA supplies half of
// every K and V tile), issued by the slot's own thread: the next tile's scores are computed
// while the softmax of the current one runs. The softmax rewrites P_s only after the PV that
// read it has completed.
//
// TMEM (512 columns, same addresses in both CTAs): S_0 [0,128), S_1 [128,256), O_0 [256,384),
// O_1 [384,512).
// Warp roles (16 warps):
//   warp 0      TMA producer (Q per unit and slot, this CTA's halves of K and V tiles); also
//               forwards "K / V half landed" to the even CTA
//   warps 1, 2  MMA issuers of slot 0 / slot 1 (even CTA only)
//   warp 3      scheduler: per-unit metadata (tiles, ranges, block-sparse bitmaps) into a ring
//   warps 4-7   softmax of slot 0, warps 8-11 softmax of slot 1: one query row per thread;
//               they write O and LSE at the end of a unit
//   warps 12-15 fused RoPE: rotate each unit's Q tiles in place as they land (12-13 slot 0,
//               14-15 slot 1); the keys come rotated (K') from a pass the host launches
//               first. e4m3 inputs: V comes widened to bf16 from a pass the host launches
//               first, and the scores run on kind::f8f6f4 MMAs
// Registers: launched at 128 per thread, re-dealt with setmaxnreg to 72 (warps 0-3), 192
// (softmax) and 56 (warps 12-15); at 176 for the softmax, ptxas spilled in its loop.
// Every wait is bounded (see ptx.cuh).
#pragma once
#include <cuda.h>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace afx {

namespace {

constexpr int kBM = 128;               // query rows per slot and CTA
constexpr int kBN = 128;               // keys per kv tile (64 per CTA for K)
constexpr int kThreads = 512;
constexpr int kStMax = 4;              // largest K / V stage count
constexpr int kRing = 4;               // unit metadata entries in flight
constexpr uint32_t kPTile = kBM * kBN * 2;       // 32 KB: P of one slot, two 64-key panels
constexpr uint32_t kTmS = 0, kTmO = 256;         // + 128 * slot

// Shared-memory plan for head dim D (128 or 64). Q, K and P rows are 128-byte swizzled (one
// 64-dim panel per 128 bytes); each CTA's half of a V tile holds D/2 dims of 128 keys: 128-byte
// rows for D = 128, 64-byte rows (64-byte swizzle) for D = 64.
template <int D>
struct PPCfg {
  static constexpr int KSt = D == 128 ? 3 : 4;   // K stages (released when both slots' S are done)
  static constexpr int VSt = D == 128 ? 2 : 4;   // V stages (released when both slots' PV are done)
  static constexpr uint32_t QTile = kBM * D * 2;
  static constexpr uint32_t KHalf = 64u * D * 2u;
  static constexpr uint32_t VHalf = kBN * (D / 2) * 2u;
  static constexpr uint32_t OffQ = 0;
  static constexpr uint32_t OffP = 2 * QTile;
  static constexpr uint32_t OffK = OffP + 2 * kPTile;
  static constexpr uint32_t OffV = OffK + KSt * KHalf;
  static constexpr uint32_t OffCtl = OffV + VSt * VHalf;
  static_assert(KSt <= kStMax && VSt <= kStMax, "stage arrays");
};

constexpr uint32_t kRegsLow = 72;    // warpgroup 0: producer, issuers, scheduler
constexpr uint32_t kRegsRot = 56;     // warpgroup 3: Q rotators
constexpr uint32_t kRegsSm = 192;    // warpgroups 1, 2: softmax
static_assert(kRegsLow + kRegsRot + 2 * kRegsSm <= 4 * (65536 / kThreads),
              "register split exceeds the registers the CTA is launched with");

// One unit as every role of a CTA sees it. Tile e = 2 * slot + cta.
struct UnitMeta {
  int live;                    // 0: the cluster has no more units
  int b, kvh;
  int head[2][2], q0[2][2], qv[2][2];  // [slot][cta]; qv: the tile has rows below N
  int lo[2][2], hi[2][2];              // kv tiles the tile's rows can see (empty if !qv)
  int slo[2], shi[2];                  // union over the slot's two tiles
  int jb, je;                          // kv tiles either slot needs
  int ns[2];                           // kv tiles of each slot
  uint32_t sbits[2][kTileWords];       // block-sparse: tiles of the slot (either CTA)
  uint32_t tbits[2][kTileWords];       // block-sparse: tiles of this CTA's tile of the slot
  uint32_t rbits[2][2][kBsWords];      // block-sparse 64-blocks, this CTA: [slot][row block][col]
};

struct Ctl {
  uint64_t q_full[2], k_full[kStMax], v_full[kStMax];   // local TMA completion
  uint64_t q_empty[2], k_empty[kStMax], v_empty[kStMax];  // MMA commits (multicast to both CTAs)
  uint64_t s_full[2], o_full[2], pv_done[2];           // MMA commits (multicast)
  uint64_t q_ready[2], k_ready[kStMax], v_ready[kStMax], p_full[2], s_free[2];  // even CTA: both CTAs arrive
  uint64_t o_read[2];  // even CTA: the slot's softmax warps of both CTAs took an O phase before an empty unit
  uint64_t meta_full[kRing], meta_empty[kRing];
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort_flag;
  UnitMeta ring[kRing];
};

template <int D>
__host__ __device__ constexpr size_t pp_smem() { return 1024 + PPCfg<D>::OffCtl + sizeof(Ctl); }
static_assert(pp_smem<128>() <= 232448 && pp_smem<64>() <= 232448, "shared memory budget");

__device__ __forceinline__ bool pbit(const uint32_t* w, int i) { return (w[i >> 5] >> (i & 31)) & 1u; }

// Arrive on a barrier of the even CTA: a plain shared::cta arrive there, a shared::cluster
// arrive from the odd CTA.
__device__ __forceinline__ void arrive_leader(uint64_t* bar, int rank) {
  if (rank == 0)
    mbar_arrive(bar);
  else
    mbar_arrive_cluster(mapa_shared(smem_u32(bar), 0));
}

// Next kv tile after j that either slot of the unit needs.
__device__ __forceinline__ int next_tile(const UnitMeta& M, bool bs, int j) {
  if (!bs) return j + 1;
  for (int jj = j + 1; jj < M.je;) {
    const int w = jj >> 5;
    const uint32_t bits = (M.sbits[0][w] | M.sbits[1][w]) >> (jj & 31);
    if (bits) return jj + __ffs(bits) - 1;
    jj = (w + 1) << 5;
  }
  return M.je;
}

__device__ __forceinline__ bool slot_act(const UnitMeta& M, bool bs, int s, int j) {
  return bs ? pbit(M.sbits[s], j) : (j >= M.slo[s] && j < M.shi[s]);
}

// Work-unit decomposition. hp query heads x tq query tiles per unit (hp * tq = 4); units are
// numbered longest first (for causal masks, by descending query position) and dealt to the
// clusters in a snake order, which balances the causal triangle to within a tile or two.
struct Sched {
  int hp, tq, nt, hg;  // hp: heads per unit, tq: q tiles per unit, nt: unit rows, hg: Hq / hp
  int units, clusters;
};

__device__ __forceinline__ Sched make_sched(const FwdParams& p) {
  Sched S;
  S.hp = p.pp_hp;
  S.tq = 4 / S.hp;
  const int TQ = (p.N + kBM - 1) / kBM;
  S.nt = (TQ + S.tq - 1) / S.tq;
  S.hg = p.Hq / S.hp;
  S.units = S.nt * p.B * S.hg;
  S.clusters = p.pp_clusters;
  return S;
}

// Fill ring entry M for the k-th unit of cluster c (one warp).
__device__ void fill_meta(UnitMeta& M, const FwdParams& p, const Sched& S, int c, int k, int rank,
                          int lane) {
  const VariantDev& var = p.var;
  const int C = S.clusters;
  const long long idx = (long long)k * C + ((k & 1) ? (C - 1 - c) : c);
  if (idx >= S.units) {
    if (lane == 0) M.live = 0;
    __syncwarp();
    return;
  }
  const int per_t = p.B * S.hg;
  const int t = S.nt - 1 - static_cast<int>(idx / per_t);
  const int rem = static_cast<int>(idx % per_t);
  const int b = rem / S.hg, hg = rem % S.hg;
  const int TK = (p.N + kBN - 1) / kBN;
  const bool bs = var.mask == 3;
  if (lane == 0) {
    M.live = 1;
    M.b = b;
    M.kvh = hg * S.hp / p.g;
    int jb = TK, je = 0;
    for (int s = 0; s < 2; ++s) {
      int slo = TK, shi = 0;
      for (int r = 0; r < 2; ++r) {
        const int e = 2 * s + r;
        const int head = hg * S.hp + e % S.hp;
        const int q0 = (t * S.tq + e / S.hp) * kBM;
        const bool valid = q0 < p.N;
        int lo = 0, hi = TK;
        const int m_hi = min(q0 + kBM - 1, p.N - 1);
        if (var.causal) hi = min(hi, m_hi / kBN + 1);
        if (var.mask == 2) {
          lo = max(0, q0 - var.window + 1) / kBN;
          if (!var.causal) hi = min(hi, (m_hi + var.window - 1) / kBN + 1);
        }
        if (!valid || lo >= hi) lo = hi = 0;
        M.head[s][r] = head;
        M.q0[s][r] = q0;
        M.qv[s][r] = valid ? 1 : 0;
        M.lo[s][r] = lo;
        M.hi[s][r] = hi;
        if (lo < hi) {
          slo = min(slo, lo);
          shi = max(shi, hi);
        }
      }
      if (slo >= shi) slo = shi = 0;
      M.slo[s] = slo;
      M.shi[s] = shi;
      M.ns[s] = shi - slo;
      if (slo < shi) {
        jb = min(jb, slo);
        je = max(je, shi);
      }
    }
    M.jb = jb < je ? jb : 0;
    M.je = jb < je ? je : 0;
  }
  if (!bs) {
    __syncwarp();
    return;
  }
  // Block-sparse: tiles with an active block per query tile (both CTAs' tiles, for the
  // iteration) and, for 64-blocks, this CTA's active block columns per 64-row block.
  for (int i = lane; i < 2 * kTileWords; i += 32) {
    (&M.sbits[0][0])[i] = 0u;
    (&M.tbits[0][0])[i] = 0u;
  }
  for (int i = lane; i < 4 * kBsWords; i += 32) (&M.rbits[0][0][0])[i] = 0u;
  __syncwarp();
  const int blk = var.bs_block;
  const int nb_total = (p.N + blk - 1) / blk;
  for (int s = 0; s < 2; ++s)
    for (int r = 0; r < 2; ++r) {
      if (!M.qv[s][r]) continue;
      const int lo = M.lo[s][r], hi = M.hi[s][r];
      const int br0 = M.q0[s][r] / blk;
      for (int rr = 0; rr < kBM / blk; ++rr) {
        const int br = br0 + rr;
        if (br >= nb_total) continue;
        const int e0 = var.bs_row_ptr[br], e1 = var.bs_row_ptr[br + 1];
        for (int e = e0 + lane; e < e1; e += 32) {
          const int col = var.bs_col_idx[e];
          if (col < 0 || col >= nb_total) continue;
          const int tile = col * blk / kBN;
          if (tile < lo || tile >= hi) continue;
          atomicOr(&M.sbits[s][tile >> 5], 1u << (tile & 31));
          if (r == rank) {
            atomicOr(&M.tbits[s][tile >> 5], 1u << (tile & 31));
            if (blk == 64) atomicOr(&M.rbits[s][rr][col >> 5], 1u << (col & 31));
          }
        }
      }
    }
  __syncwarp();
  if (lane == 0) {
    int jb = -1, je = 0, n0 = 0, n1 = 0;
    for (int w = 0; w < kTileWords; ++w) {
      const uint32_t u = M.sbits[0][w] | M.sbits[1][w];
      n0 += __popc(M.sbits[0][w]);
      n1 += __popc(M.sbits[1][w]);
      if (u) {
        if (jb < 0) jb = w * 32 + __ffs(u) - 1;
        je = w * 32 + 32 - __clz(u);
      }
    }
    M.ns[0] = n0;
    M.ns[1] = n1;
    M.jb = jb < 0 ? 0 : jb;
    M.je = jb < 0 ? 0 : je;
  }
  __syncwarp();
}

}  // namespace

// RK: how the score operands are produced (kRopeNone / kRopeFused / kRopePrerotated, or
// kFp8: e4m3 Q and K used as they are; V widened to bf16 by the host's pass).
// BIAS: score bias compiled in (0 none, 1 ALiBi, 2 additive). NORM: 0 softmax, 1 ReLU
// normaliser (P = relu(s) / N, no row sum).
template <int RK, int BIAS, int NORM, int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fwd_pp_kernel(const __grid_constant__ FwdParams p) {
  using C = PPCfg<D>;
  constexpr int kD = D;
  constexpr int kKSt = C::KSt, kVSt = C::VSt;
  constexpr uint32_t kQTile = C::QTile, kKHalf = C::KHalf, kVHalf = C::VHalf;
  constexpr uint32_t kOffQ = C::OffQ, kOffP = C::OffP, kOffK = C::OffK, kOffV = C::OffV,
                     kOffCtl = C::OffCtl;
  constexpr size_t kSmem = pp_smem<D>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kOffCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const VariantDev& var = p.var;
  constexpr bool ROPE = (RK == kRopeFused);
  constexpr bool FP8 = (RK == kFp8);
  // How a slot with no tiles in a unit completes that unit's O phase (both keep one o_full
  // phase per unit, in order with the softmax's waits). With fused RoPE the issuer commits it
  // once the slot's softmax warps of both CTAs have taken the previous phase (o_read); otherwise
  // the slot's softmax warps complete it themselves. Both are correct; each instance uses the
  // one that measured faster for it.
  constexpr bool kORead = ROPE;
  const int rank = static_cast<int>(cluster_ctarank());
  const int cid = static_cast<int>(blockIdx.x) >> 1;
  const Sched S = make_sched(p);
  const bool bs = var.mask == 3;

  if (tid == 0) {
    ctl->abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->q_full[s], 1);
      mbar_init(&ctl->q_empty[s], 1);
      mbar_init(&ctl->s_full[s], 1);
      mbar_init(&ctl->o_full[s], 1);
      mbar_init(&ctl->q_ready[s], ROPE ? 4 : 8);   // the slot's 2 Q rotators (fused RoPE) or
                                                   // 4 softmax warps, both CTAs
      mbar_init(&ctl->p_full[s], 8);
      mbar_init(&ctl->s_free[s], 8);    // the slot's 4 softmax warps have read S, both CTAs
      mbar_init(&ctl->pv_done[s], 1);
      if constexpr (kORead) mbar_init(&ctl->o_read[s], 8);
    }
    for (int s = 0; s < kKSt; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 2);   // one commit per issuer
      mbar_init(&ctl->k_ready[s], 2);
    }
    for (int s = 0; s < kVSt; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 2);
      mbar_init(&ctl->v_ready[s], 2);
    }
    // ring consumers: producer, (even CTA) two issuers, (fused RoPE) four rotator warps,
    // eight softmax warps
    const int consumers = 1 + (rank == 0 ? 2 : 0) + (ROPE ? 4 : 0) + 8;
    for (int e = 0; e < kRing; ++e) {
      mbar_init(&ctl->meta_full[e], 32);
      mbar_init(&ctl->meta_empty[e], consumers);
    }
    mbar_init(&ctl->mma_final, 2);   // one commit per issuer
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctl->tmem_base, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();

  const uint32_t tmem = ctl->tmem_base;
  int* status = p.status;
  volatile int* abort_flag = &ctl->abort_flag;

  if (warp < 4) {
    setmaxnreg_dec<kRegsLow>();
    if (warp == 3) {
      // ======================= scheduler =======================
      for (int k = 0;; ++k) {
        const int e = k % kRing;
        if (k >= kRing &&
            !__all_sync(0xffffffffu, mbar_wait(&ctl->meta_empty[e], ((k / kRing) - 1) & 1, status, abort_flag)))
          break;
        UnitMeta& M = ctl->ring[e];
        fill_meta(M, p, S, cid, k, rank, lane);
        mbar_arrive(&ctl->meta_full[e]);
        if (!M.live) break;
      }
    } else if (warp == 0 && lane == 0) {
      // ======================= TMA producer and relay =======================
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      const uint64_t pol_stream = l2_policy_evict_first();
      const uint64_t pol_keep = l2_policy_evict_last();
      // Three copy streams walk the units independently, each polled and issued when its
      // buffer is free: Q per (unit, slot), K and V per kv tile. Landed K / V halves are
      // forwarded to the even CTA in load order.
      int uq = 0, sq = 0;            // next Q copy
      int uk = 0, jk = -1, ik = 0;   // next K copy: unit, tile (-1: unit not started), count
      int uv = 0, jv = -1, iv = 0;   // next V copy
      int rk = 0, rv = 0;            // K / V halves forwarded
      int urel = 0;                  // ring entries released by this thread
      bool dq = false, dk = false, dv = false;
      uint64_t t0 = 0;
      uint32_t idle = 0;
      auto meta_ready = [&](int u) {
        return mbar_test(&ctl->meta_full[u % kRing], (u / kRing) & 1);
      };
      while (true) {
        bool moved = false;
        // ---- Q ----
        if (!dq && meta_ready(uq)) {
          const UnitMeta& M = ctl->ring[uq % kRing];
          if (!M.live) {
            dq = true;
          } else if (uq == 0 || mbar_test(&ctl->q_empty[sq], (uq - 1) & 1)) {
            mbar_arrive_expect_tx(&ctl->q_full[sq], FP8 ? kQTile / 2 : kQTile);
            for (int pn = 0; pn < (FP8 ? 1 : kD / 64); ++pn)
              tma_load_4d_hint(smem + kOffQ + sq * kQTile + pn * (kBM * 128), &p.tmQ, &ctl->q_full[sq],
                               pn * 64, M.q0[sq][rank], M.head[sq][rank], M.b, pol_stream);
            if (++sq == 2) {
              sq = 0;
              ++uq;
            }
            moved = true;
          }
        }
        // ---- K ----
        if (!dk && meta_ready(uk)) {
          const UnitMeta& M = ctl->ring[uk % kRing];
          if (!M.live) {
            dk = true;
          } else {
            if (jk < 0) jk = M.jb;
            if (jk >= M.je) {
              ++uk;
              jk = -1;
              moved = true;
            } else {
              const int st = ik % kKSt;
              if (ik < kKSt || mbar_test(&ctl->k_empty[st], ((ik / kKSt) - 1) & 1)) {
                mbar_arrive_expect_tx(&ctl->k_full[st], FP8 ? kKHalf / 2 : kKHalf);
                for (int pn = 0; pn < (FP8 ? 1 : kD / 64); ++pn)
                  tma_load_4d_hint(smem + kOffK + st * kKHalf + pn * (64 * 128), &p.tmK, &ctl->k_full[st],
                                   pn * 64, jk * kBN + rank * 64, M.kvh, M.b, pol_keep);
                ++ik;
                jk = next_tile(M, bs, jk);
                moved = true;
              }
            }
          }
        }
        // ---- V (never ahead of K) ----
        if (!dv && meta_ready(uv)) {
          const UnitMeta& M = ctl->ring[uv % kRing];
          if (!M.live) {
            dv = true;
          } else {
            if (jv < 0) jv = M.jb;
            if (jv >= M.je) {
              ++uv;
              jv = -1;
              moved = true;
            } else if (iv < ik) {
              const int st = iv % kVSt;
              if (iv < kVSt || mbar_test(&ctl->v_empty[st], ((iv / kVSt) - 1) & 1)) {
                mbar_arrive_expect_tx(&ctl->v_full[st], kVHalf);
                tma_load_4d_hint(smem + kOffV + st * kVHalf, &p.tmV, &ctl->v_full[st], rank * (kD / 2),
                                 jv * kBN, M.kvh, M.b, pol_keep);
                ++iv;
                jv = next_tile(M, bs, jv);
                moved = true;
              }
            }
          }
        }
        // ---- relay ----
        if (rk < ik && mbar_test(&ctl->k_full[rk % kKSt], (rk / kKSt) & 1)) {
          arrive_leader(&ctl->k_ready[rk % kKSt], rank);
          ++rk;
          moved = true;
        }
        if (rv < iv && mbar_test(&ctl->v_full[rv % kVSt], (rv / kVSt) & 1)) {
          arrive_leader(&ctl->v_ready[rv % kVSt], rank);
          ++rv;
          moved = true;
        }
        // ---- ring entries every stream has left ----
        {
          const int umin = min(uq, min(uk, uv));
          while (urel < umin) {
            mbar_arrive(&ctl->meta_empty[urel % kRing]);
            ++urel;
          }
        }
        if (dq && dk && dv && rv == iv && rk == ik) break;
        if (moved) {
          idle = 0;
        } else {
          // nothing to do: back off briefly so the polling does not compete with the MMAs'
          // operand reads for shared memory
          __nanosleep(32);
          if ((++idle & 255u) == 1u) {
            const uint64_t now = globaltimer_ns();
            if (idle == 1u) t0 = now;
            if (*abort_flag) break;
            if (now - t0 > ATTNFUSE_WAIT_LIMIT_NS) {
              atomicOr(status, kDevTimeout);
              *abort_flag = 1;
              break;
            }
          }
        }
      }
      // Drain: no copy may still be landing in shared memory when the CTA exits.
      for (int k = max(0, ik - kKSt); k < ik; ++k)
        mbar_wait(&ctl->k_full[k % kKSt], (k / kKSt) & 1, status, nullptr);
      for (int k = max(0, iv - kVSt); k < iv; ++k)
        mbar_wait(&ctl->v_full[k % kVSt], (k / kVSt) & 1, status, nullptr);
      const int nq = 2 * uq + sq;  // Q copies issued
      for (int k = max(0, nq - 2); k < nq; ++k)
        mbar_wait(&ctl->q_full[k & 1], (k >> 1) & 1, status, nullptr);
    } else if ((warp == 1 || warp == 2) && lane == 0 && rank == 0) {
      // ======================= pair-MMA issuer of slot s =======================
      // Per kv tile i the issuer of slot s runs S_s = Q_s K(i) as soon as the slot's softmax
      // has read S_s of the tile before into registers (s_free), and then O_s += P_s V(i-1)
      // once that softmax has written P_s to shared memory (p_full). The scores of the next
      // tile are thus computed while the softmax of the current one runs. The two issuers run
      // concurrently on different SM sub-partitions, so each one's barrier waits overlap the
      // other's MMAs.
      const int s = warp - 1;
      constexpr uint32_t idesc_s = FP8 ? idesc_e4m3_f32(256, kBN) : idesc_f32acc(256, kBN, 0, 0, RK != kRopeNone);
      constexpr uint32_t idesc_o = idesc_bf16_f32(256, kD, 0, 1);
      // Descriptors as a 32-bit low word (start address >> 4, plus the leading byte offset)
      // and one shared high word; a tile's k-steps add compile-time offsets to the low word.
      // Every operand lies below 256 KB of shared memory, so the address field never carries.
      static_assert(kSmem < (1u << 18), "descriptor address field");
      constexpr uint32_t dhi = desc_sw128_hi(1024);
      const uint32_t dQ = desc_sw128_lo(smem_u32(smem + kOffQ + s * kQTile), 16);
      const uint32_t dP = desc_sw128_lo(smem_u32(smem + kOffP + s * kPTile), 16);
      const uint32_t dK0 = desc_sw128_lo(smem_u32(smem + kOffK), 16);
      const uint32_t dV0 = desc_sw128_lo(smem_u32(smem + kOffV), kVHalf);
      // V halves: D/2 dims of 128 keys, MN-major; 128-byte rows (8-key atoms of 1024 bytes) for
      // D = 128, 64-byte rows (64-byte swizzle, atoms of 512 bytes) for D = 64
      constexpr uint32_t dhi_v = kD == 128 ? desc_sw128_hi(1024) : desc_sw64_hi(512);
      constexpr uint32_t kVStep = (kD / 2) * 2 * 16;  // bytes of 16 keys
      const uint32_t tS = tmem + kTmS + 128 * s, tO = tmem + kTmO + 128 * s;
      int ik = 0;          // kv tiles walked (K and V copy index)
      int sc = 0;          // S issued (phases of s_full and s_free)
      int pvc = 0;         // PV issued (phases of p_full and pv_done)
      bool pend = false;   // a PV waits for its P
      int pend_v = 0;      // its V copy index
      bool pend_acc = false, pend_last = false;
      bool ok = true;
      // the pending PV, once its P is in shared memory and its V has landed
      auto flush_pv = [&]() {
        ok = mbar_wait_cluster(&ctl->p_full[s], pvc & 1, status, abort_flag) &&
             mbar_wait_cluster(&ctl->v_ready[pend_v % kVSt], (pend_v / kVSt) & 1, status, abort_flag);
        if (!ok) return;
        tc_fence_after();
        const int vs = pend_v % kVSt;
        const uint32_t bv = dV0 + vs * (kVHalf >> 4);
        if (pend_acc)
          mma_ss_pair_w2<1>(tO, dP, dhi, bv, dhi_v, idesc_o);
        else
          mma_ss_pair_w2<0>(tO, dP, dhi, bv, dhi_v, idesc_o);
#pragma unroll
        for (int kk = 1; kk < kBN / 16; ++kk)
          mma_ss_pair_w2<1>(tO, dP + (((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4), dhi,
                            bv + kk * (kVStep >> 4), dhi_v, idesc_o);
        mma_commit_pair(&ctl->v_empty[vs], 3);
        mma_commit_pair(&ctl->pv_done[s], 3);
        if (pend_last) mma_commit_pair(&ctl->o_full[s], 3);
        ++pvc;
        pend = false;
      };
      for (int u = 0; ok; ++u) {
        const int e = u % kRing;
        ok = mbar_wait(&ctl->meta_full[e], (u / kRing) & 1, status, abort_flag);
        if (!ok) break;
        const UnitMeta& M = ctl->ring[e];
        if (!M.live) break;
        const int jb = M.jb, je = M.je, ns = M.ns[s], slo = M.slo[s], shi = M.shi[s];
        int cnt = 0;
        bool opened = false;
        // First use of the slot in this unit: the previous unit's last PV (its softmax waits
        // for that O before this unit's epilogue), then this unit's rotated Q.
        auto open_slot = [&]() {
          if (pend) {
            flush_pv();
            if (!ok) return;
          }
          ok = mbar_wait_cluster(&ctl->q_ready[s], u & 1, status, abort_flag);
          // A slot with no tiles in this unit releases its Q buffer at once; it has no O (its
          // softmax writes zeros). With kORead the issuer completes the unit's O phase without
          // an MMA; that commit completes as soon as the previous PVs have, so it first waits
          // until the slot's softmax warps of both CTAs have taken the previous phase (o_full
          // never runs two phases ahead of a waiter).
          if (ok && ns == 0) {
            mma_commit_pair(&ctl->q_empty[s], 3);
            if constexpr (kORead) {
              if (u > 0) ok = mbar_wait_cluster(&ctl->o_read[s], (u - 1) & 1, status, abort_flag);
              if (ok) mma_commit_pair(&ctl->o_full[s], 3);
            }
          }
          opened = true;
        };
        for (int j = jb; ok && j < je; j = next_tile(M, bs, j), ++ik) {
          const bool a = bs ? pbit(M.sbits[s], j) : (j >= slo && j < shi);
          const int st = ik % kKSt;
          if (!opened) open_slot();
          if (ok && !a) {
            // no MMA of this slot reads K(ik) or V(ik): release both once they have landed.
            // The pending PV goes first: a later V copy into its stage waits for it.
            if (pend) flush_pv();
            if (ok) ok = mbar_wait_cluster(&ctl->k_ready[st], (ik / kKSt) & 1, status, abort_flag);
            if (ok) ok = mbar_wait_cluster(&ctl->v_ready[ik % kVSt], (ik / kVSt) & 1, status, abort_flag);
            if (!ok) break;
            mma_commit_pair(&ctl->v_empty[ik % kVSt], 3);
            mma_commit_pair(&ctl->k_empty[st], 3);
            continue;
          }
          // ---- waits for S(j): Q, K(j) landed, the slot's previous S read ----
          if (ok) ok = mbar_wait_cluster(&ctl->k_ready[st], (ik / kKSt) & 1, status, abort_flag);
          if (ok && sc > 0) ok = mbar_wait_cluster(&ctl->s_free[s], (sc - 1) & 1, status, abort_flag);
          if (!ok) break;
          tc_fence_after();
          {
            const uint32_t bk = dK0 + st * (kKHalf >> 4);
            if constexpr (FP8) {
              // one 128-byte panel per row: four k-steps of 32 e4m3 values (32 bytes)
              mma_ss_pair_f8_w<0>(tS, dQ, bk, dhi, idesc_s);
#pragma unroll
              for (int kk = 1; kk < kD / 32; ++kk)
                mma_ss_pair_f8_w<1>(tS, dQ + ((kk * 32) >> 4), bk + ((kk * 32) >> 4), dhi, idesc_s);
            } else {
              mma_ss_pair_w<0>(tS, dQ, bk, dhi, idesc_s);
#pragma unroll
              for (int kk = 1; kk < kD / 16; ++kk)
                mma_ss_pair_w<1>(tS, dQ + (((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4),
                                 bk + (((kk >> 2) * (64 * 128) + (kk & 3) * 32) >> 4), dhi, idesc_s);
            }
            mma_commit_pair(&ctl->s_full[s], 3);
            ++sc;
            ++cnt;
            if (cnt == ns) mma_commit_pair(&ctl->q_empty[s], 3);
          }
          mma_commit_pair(&ctl->k_empty[st], 3);
          // ---- the previous tile's PV, then this tile's becomes pending ----
          if (pend) {
            flush_pv();
            if (!ok) break;
          }
          pend = true;
          pend_v = ik;
          pend_acc = cnt > 1;
          pend_last = cnt == ns;
        }
        if (ok && !opened) open_slot();
        if (ok) mbar_arrive(&ctl->meta_empty[e]);
      }
      if (ok && pend) flush_pv();
      // All MMAs must finish before TMEM is released.
      mma_commit_pair(&ctl->mma_final, 3);
      mbar_wait(&ctl->mma_final, 0, status, nullptr);
    }
  } else if (warp >= 12) {
    // ======================= Q rotators (fused RoPE) =======================
    setmaxnreg_dec<kRegsRot>();
    if (ROPE) {
      // ---- Q rotators: Q' = R_m Q of each unit's tiles, in place in shared memory (fp16), as
      // soon as a tile lands; warps 12-13 take slot 0, warps 14-15 slot 1. Warp w2 of a slot
      // rotates the rows of the query-tile recurrence chains (query_cs8) c0 = w2 + 2i (i < 4),
      // rows c0 + 8k, each chain starting from its table entry and stepping 8 positions. Lane f
      // of a row takes dims 2f, 2f+1 and their partners D/2+2f, D/2+2f+1 (F4 = D/4 lanes per
      // row, so a warp instruction covers RPI = 32/F4 chains). K' comes from the rotation pass
      // the host launches before this kernel. ----
      constexpr int F4 = kD / 4, RPI = 32 / F4;
      const int s = (warp - 12) >> 1, w2 = (warp - 12) & 1;
      const int f = lane % F4, rsub = lane / F4;
      const int N = p.N;
      const uint64_t pol_tab = l2_policy_evict_last();
      const float4* tab = reinterpret_cast<const float4*>(p.rope_cs);
      const float4 wstep = ldg_f4_hint(tab + (size_t)8 * F4 + f, pol_tab);
      uint8_t* tile = smem + kOffQ + s * kQTile;
      const uint32_t within = static_cast<uint32_t>(f & 3) * 4u;
      uint32_t f16max = 0;  // |Q'| as fp16 bits, per half
      bool ok = true;
      for (int u = 0; ok; ++u) {
        const int e = u % kRing;
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->meta_full[e], (u / kRing) & 1, status, abort_flag));
        if (!ok) break;
        const UnitMeta& M = ctl->ring[e];
        if (!M.live) break;
        const int qq0 = M.q0[s][rank];
        const bool qvalid = M.qv[s][rank] != 0;
        float4 cs[4 / RPI];
#pragma unroll
        for (int i = 0; i < 4 / RPI; ++i)
          cs[i] = qvalid ? ldg_f4_hint(tab + (size_t)min(qq0 + w2 + 2 * (RPI * i + rsub), N - 1) * F4 + f, pol_tab)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->q_full[s], u & 1, status, abort_flag));
        if (!ok) break;
        if (qvalid) {
#pragma unroll 2
          for (int k = 0; k < kBM / 8; ++k) {
#pragma unroll
            for (int i = 0; i < 4 / RPI; ++i) {
              const int rr = w2 + 2 * (RPI * i + rsub) + 8 * k;
              if (qq0 + rr < N) {
                const uint32_t offl = sw128_offset(rr, f >> 2) + within;
                const uint32_t offh = kD == 128 ? offl + kBM * 128 : sw128_offset(rr, (f >> 2) + 4) + within;
                const uint32_t l2w = *reinterpret_cast<const uint32_t*>(tile + offl);
                const uint32_t h2w = *reinterpret_cast<const uint32_t*>(tile + offh);
                float yl0, yh0, yl1, yh1;
                rot_pair(bf16lo_to_f32(l2w), bf16lo_to_f32(h2w), cs[i].x, cs[i].y, yl0, yh0);
                rot_pair(bf16hi_to_f32(l2w), bf16hi_to_f32(h2w), cs[i].z, cs[i].w, yl1, yh1);
                const uint32_t wl = pack_f16x2_sat(yl0, yl1), wh = pack_f16x2_sat(yh0, yh1);
                f16max = f16_absmax(f16_absmax(f16max, wl), wh);
                *reinterpret_cast<uint32_t*>(tile + offl) = wl;
                *reinterpret_cast<uint32_t*>(tile + offh) = wh;
              }
              float c0f, s0f, c1f, s1f;
              rot_pair(cs[i].x, cs[i].y, wstep.x, wstep.y, c0f, s0f);
              rot_pair(cs[i].z, cs[i].w, wstep.z, wstep.w, c1f, s1f);
              cs[i] = make_float4(c0f, s0f, c1f, s1f);
            }
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          arrive_leader(&ctl->q_ready[s], rank);
          mbar_arrive(&ctl->meta_empty[e]);
        }
      }
      report_f16_range(status, f16max);
    }
  } else {
    // ======================= softmax of slot s (one query row per thread) =======================
    setmaxnreg_inc<kRegsSm>();
    const int s = (warp - 4) >> 2;
    const int wq = warp & 3;                 // TMEM lane quarter
    const int r = wq * 32 + lane;            // row within this CTA's 128 rows of the slot
    const int N = p.N;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + kTmS + 128 * s;
    const uint32_t tO = tmem + lane_off + kTmO + 128 * s;
    const float scale_u = NORM == 0 ? p.scale_log2 : p.scale;  // score units
    const float bias_u = NORM == 0 ? kLog2e : 1.f;
    const float inv_n = 1.f / static_cast<float>(N);
    const int TK = (N + kBN - 1) / kBN;
    uint8_t* const visits = var.visits;
    int sc = 0;  // S of this slot consumed (phase of s_full)
    int pc = 0;  // P of this slot written (phase of p_full; PV pc-1 completes phase pc-1 of pv_done)
    bool ok = true;
    // Q' = R_m Q of unit un in place (fp16 with fused RoPE), then the slot's MMAs may read it.
    auto prep_q = [&](const UnitMeta& Mq, int un) {
      (void)Mq;
      if (ROPE) return;  // the Q rotators wait for the tile, rotate it and signal q_ready
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->q_full[s], un & 1, status, abort_flag));
      if (!ok) return;
      __syncwarp();
      if (lane == 0) arrive_leader(&ctl->q_ready[s], rank);
    };
    {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->meta_full[0], 0, status, abort_flag));
      if (ok && ctl->ring[0].live) prep_q(ctl->ring[0], 0);
    }
    for (int u = 0; ok; ++u) {
      const int e = u % kRing;
      const UnitMeta& M = ctl->ring[e];
      if (!M.live) break;
      const int b = M.b;
      const int q0 = M.q0[s][rank], head = M.head[s][rank];
      const bool valid = M.qv[s][rank] != 0;
      const int m = q0 + r;
      const int lo_o = M.lo[s][rank], hi_o = M.hi[s][rank];
      // tiles of this CTA's query tile outside [jm_lo, jm_hi) need per-element masks
      int jm_lo = 0, jm_hi = N / kBN;
      {
        const int q_last = min(q0 + kBM - 1, N - 1);
        if (var.causal) jm_hi = min(jm_hi, q0 / kBN);
        if (var.mask == 2) {
          const int lim = q_last - var.window + 1;
          if (lim > 0) jm_lo = (lim + kBN - 1) / kBN;
          if (!var.causal) {
            const int ee = q0 + var.window - kBN;
            jm_hi = min(jm_hi, ee >= 0 ? ee / kBN + 1 : 0);
          }
        }
      }
      const bool bs64 = bs && var.bs_block == 64;
      const int blk_row = bs64 ? (r >> 6) : 0;

      // ---- kv tiles of the slot ----
      const float alibi = (BIAS == 1 && valid) ? var.slopes[head] * bias_u : 0.f;
      const int64_t ab_row = b * var.ab_s[0] + head * var.ab_s[1] + (int64_t)m * var.ab_s[2];
      float m_run = kNegInf, l_run = 0.f;  // row scale (log2 units) and sum of O's rows
      bool first = true;
      for (int j = M.jb; j < M.je; j = next_tile(M, bs, j)) {
        if (!slot_act(M, bs, s, j)) continue;
        const bool act = valid && j >= lo_o && j < hi_o && (!bs || pbit(M.tbits[s], j));
        bool h0 = true, h1 = true;  // block-sparse 64-blocks of this tile present for the row
        if (bs64) {
          h0 = pbit(M.rbits[s][blk_row], 2 * j);
          h1 = pbit(M.rbits[s][blk_row], 2 * j + 1);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&ctl->s_full[s], sc & 1, status, abort_flag))) {
          ok = false;
          break;
        }
        ++sc;
        tc_fence_after();
        uint32_t xr[128];
        tmem_ld32<0>(tS, xr);
        tmem_ld32<32>(tS + 32, xr);
        tmem_ld32<64>(tS + 64, xr);
        tmem_ld32<96>(tS + 96, xr);
        tmem_wait_ld();
        // S is in registers: the issuer may compute the next tile's S over it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(&ctl->s_free[s], rank);
        bool pv_seen = false;
        // the slot's previous PV has completed: O holds every earlier tile and the P buffer
        // may be rewritten
        auto wait_prev_pv = [&]() -> bool {
          if (pv_seen || pc == 0) return true;
          pv_seen = true;
          return __all_sync(0xffffffffu, mbar_wait(&ctl->pv_done[s], (pc - 1) & 1, status, abort_flag));
        };
        float x[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(xr[c]);
        const int k0 = j * kBN;
        // ---- score combinators (score units: log2 for softmax, natural for ReLU) ----
        float mul = scale_u;
        if constexpr (BIAS != 0) {
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] *= scale_u;
          mul = 1.f;
          if constexpr (BIAS == 1) {
            const float base = alibi * static_cast<float>(k0 - m);
#pragma unroll
            for (int c = 0; c < 128; ++c) x[c] = __fmaf_rn(alibi, static_cast<float>(c), x[c] + base);
          } else if (act) {
            // Branch-free loads (lanes past the sequence end read element 0 and drop it), so
            // the warp stays converged for the warp-collective TMEM operations that follow.
            const int c_end = (m < N) ? min(kBN, N - k0) : 0;
            if (var.add_bias_bf16) {
              const __nv_bfloat16* ab = static_cast<const __nv_bfloat16*>(var.add_bias);
#pragma unroll
              for (int c = 0; c < 128; ++c) {
                const float raw = __bfloat162float(ab[c < c_end ? ab_row + (int64_t)(k0 + c) * var.ab_s[3] : 0]);
                x[c] += (c < c_end ? raw : 0.f) * bias_u;
              }
            } else {
              const float* ab = static_cast<const float*>(var.add_bias);
#pragma unroll
              for (int c = 0; c < 128; ++c) {
                const float raw = ab[c < c_end ? ab_row + (int64_t)(k0 + c) * var.ab_s[3] : 0];
                x[c] += (c < c_end ? raw : 0.f) * bias_u;
              }
            }
          }
        }
        if (__builtin_expect(!act || !h0 || !h1 || j < jm_lo || j >= jm_hi, 0)) {
          // per-element mask (cold: sequence end, causal diagonal, window edges, holes)
          int c_lo = 0, c_hi = act ? min(kBN - 1, N - 1 - k0) : -1;
          if (var.causal) c_hi = min(c_hi, m - k0);
          if (var.mask == 2) {
            c_lo = max(c_lo, m - var.window + 1 - k0);
            if (!var.causal) c_hi = min(c_hi, m + var.window - 1 - k0);
          }
#pragma unroll
          for (int c = 0; c < 128; ++c)
            x[c] = (c >= c_lo && c <= c_hi && (c < 64 ? h0 : h1)) ? x[c] : kNegInf;
        }
        uint32_t pk[64];
        if constexpr (NORM == 1) {
          // ReLU normaliser: P = relu(s) / N
          const float f = mul * inv_n;
#pragma unroll
          for (int c = 0; c < 64; ++c)
            pk[c] = pack_bf16x2(fmaxf(x[2 * c] * f, 0.f), fmaxf(x[2 * c + 1] * f, 0.f));
        } else {
          // row max: 8 independent chains, then a small tree
          float mp[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mp[k] = fmaxf(x[2 * k], x[2 * k + 1]);
#pragma unroll
          for (int i2 = 1; i2 < 8; ++i2)
#pragma unroll
            for (int k = 0; k < 8; ++k) mp[k] = max3f(mp[k], x[16 * i2 + 2 * k], x[16 * i2 + 2 * k + 1]);
          const float mx =
              max3f(max3f(mp[0], mp[1], mp[2]), max3f(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7])) * mul;
          // O keeps its scale unless this tile exceeds it by more than 2^8 (lazy rescaling)
          const float m_new = (mx > m_run + 8.0f) ? mx : m_run;
          const bool grow = m_new > m_run && m_run != kNegInf;
          if (!first && __any_sync(0xffffffffu, grow)) {
            // O must hold the slot's previous tiles before it is rescaled
            if (!wait_prev_pv()) {
              ok = false;
              break;
            }
            const float alpha = grow ? ex2_approx(m_run - m_new) : 1.f;
#pragma unroll 1
            for (int ch = 0; ch < kD / 32; ++ch) {
              uint32_t o[32];
              tmem_ld32(tO + ch * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
              tmem_st32(tO + ch * 32, o);
            }
          }
          if (grow) l_run *= ex2_approx(m_run - m_new);
          m_run = m_new;
          const float nb = (m_new == kNegInf) ? 0.f : -m_new;
          const uint64_t mul2v = f2_pack(mul, mul), nb2 = f2_pack(nb, nb);
          uint64_t acc2[4] = {0, 0, 0, 0};
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const uint64_t a = fma2(f2_pack(x[2 * c], x[2 * c + 1]), mul2v, nb2);
            const float p0 = ex2_approx(f2_lo(a)), p1 = ex2_approx(f2_hi(a));
            acc2[c & 3] = add2(acc2[c & 3], f2_pack(p0, p1));
            pk[c] = pack_bf16x2(p0, p1);
          }
          const uint64_t acc = add2(add2(acc2[0], acc2[1]), add2(acc2[2], acc2[3]));
          l_run += f2_lo(acc) + f2_hi(acc);
        }
        first = false;
        // P (bf16) into the slot's shared-memory buffer, row r, laid out like a Q tile (two
        // 128-byte-swizzled panels of 64 keys), once the PV that read the buffer has completed
        if (!wait_prev_pv()) {
          ok = false;
          break;
        }
        {
          uint8_t* prow = smem + kOffP + s * kPTile;
#pragma unroll
          for (int q = 0; q < 16; ++q)
            *reinterpret_cast<uint4*>(prow + (q >> 3) * (kBM * 128) + sw128_offset(r, q & 7)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
        ++pc;
        fence_proxy_async_smem();
        tmem_wait_st();    // a rescaled O is in TMEM before the PV accumulates into it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(&ctl->p_full[s], rank);
        if (act && visits && r == 0) {
          const int TQ = (N + kBM - 1) / kBM;
          visits[((static_cast<int64_t>(b) * p.Hq + head) * TQ + q0 / kBM) * TK + j] = 1;
        }
      }
      if (!ok) break;
      // ---- the next unit's Q first: its copy and rotation overlap this unit's last PV, and
      // the issuer can start the next unit's S while this unit's O is written out ----
      const int en = (u + 1) % kRing;
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->meta_full[en], ((u + 1) / kRing) & 1, status, abort_flag));
      if (!ok) break;
      const bool more = ctl->ring[en].live != 0;
      if (more) {
        prep_q(ctl->ring[en], u + 1);
        if (!ok) break;
      }
      // ---- epilogue: O / l and LSE once the slot's last PV has completed ----
      const bool have = M.ns[s] > 0;
      if constexpr (!kORead) {
        if (!have) {
          // no MMA completes this unit's O phase: the slot's four warps, all past the previous
          // phase, complete it themselves
          named_bar_sync(1 + s, 128);
          if (wq == 0 && lane == 0) mbar_arrive(&ctl->o_full[s]);
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->o_full[s], u & 1, status, abort_flag));
      if (!ok) break;
      // o_read phase u: the issuer may complete an empty next unit's O phase
      if constexpr (kORead) {
        if (more && lane == 0) arrive_leader(&ctl->o_read[s], rank);
      }
      tc_fence_after();
      if (valid) {
        float inv = NORM == 1 ? 1.f : ((l_run > 0.f) ? 1.f / l_run : 0.f);
        if constexpr (FP8) inv *= p.o_scale;
        __nv_bfloat16* orow = p.out + b * p.o_sb + head * p.o_sh + (int64_t)m * p.o_sn;
#pragma unroll 1
        for (int ch = 0; ch < kD / 32; ++ch) {
          uint32_t o[32];
          if (have) {
            tmem_ld32(tO + ch * 32, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = 0u;
          }
          if (m < N) {
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
        if (NORM == 0 && p.lse && m < N)
          p.lse[(static_cast<int64_t>(b) * p.Hq + head) * N + m] =
              (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : kNegInf;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->meta_empty[e]);
      if (!more) break;
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync();  // the peer is done with this CTA's barriers and all pair MMAs have finished
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

using FwdFn = void (*)(FwdParams);

// The kernel instance for one RoPE kind, bias kind and normaliser.
template <int RK, int D>
FwdFn fwd_pp_pick(int bias, int norm) {
  if (norm == 1)
    return bias == 1 ? fwd_pp_kernel<RK, 1, 1, D> : bias == 2 ? fwd_pp_kernel<RK, 2, 1, D> : fwd_pp_kernel<RK, 0, 1, D>;
  return bias == 1 ? fwd_pp_kernel<RK, 1, 0, D> : bias == 2 ? fwd_pp_kernel<RK, 2, 0, D> : fwd_pp_kernel<RK, 0, 0, D>;
}

}  // namespace afx
