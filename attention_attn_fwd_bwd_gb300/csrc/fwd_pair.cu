// Forward attention for head dim 128 on CTA pairs (AttnFuse paper §4.1 fused RoPE, §2 online
// softmax, §3.1 combinators, §4.3 block skipping).
//
// A cluster of two CTAs (one per SM) computes a 256-row query block with tcgen05.mma
// cta_group::2 (M = 256): CTA r owns 128 query rows (heads 2p+r of one GQA group at the same
// positions, or query tiles 2t+r of one head), and of every 128-key tile it loads, rotates and
// feeds to both tensor cores only its half: keys 64r..64r+63 of K, dims 64r..64r+63 of V.
// Per SM this halves the K/V copies, the K rotation and the operand reads from shared memory
// compared with one CTA doing both halves.
//
// TMEM (512 columns, same addresses in both CTAs):
//   S[0] [0,128), S[1] [128,256)  scores of even / odd tiles, so S(i+1) is computed while
//                                 the softmax of tile i runs
//   O    [256,384)                output accumulator
//   Q'   [384,448)                rotated queries, A operand of the score MMA
//   P    [448,512)                probabilities (bf16), A operand of the PV MMA
// Warp roles (16 warps):
//   warp 0      TMA producer: Q once, then this CTA's halves of K and V tiles
//   warp 1      score MMA issuer (even CTA only): S(i) = Q' K(i)^T
//   warp 2      PV MMA issuer (even CTA only): O += P(i) V(i)
//   warp 3      relay: forwards "K / V half landed" to the even CTA (K only without fused RoPE)
//   warps 4-11  softmax, one query row per thread: warps 4-7 take the even kv tiles, warps
//               8-11 the odd ones (full 128-column rows), sharing the O accumulator
//   warps 12-15 K rotators (fused RoPE): rotate this CTA's 64 keys in shared memory
// Every wait is bounded (see ptx.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace afx {

// Optional pipeline tracing (compile with -DATTNFUSE_TRACE=<even block index>; off by default):
// both CTAs of that cluster record clock64() at pipeline events of their first 64 kv tiles,
// plus the clock right after the first cluster barrier (to align the two SMs' clocks).
#ifdef ATTNFUSE_TRACE
__device__ unsigned long long g_pair_trace[2][65][32];
#define AF_PTRACE(i, e)                                                                      \
  do {                                                                                       \
    if ((blockIdx.x >> 1) == ((ATTNFUSE_TRACE) >> 1) && (i) < 64)                             \
      g_pair_trace[blockIdx.x & 1][(i)][(e)] = clock64();                                    \
  } while (0)
#define AF_PTRACE_START()                                                                    \
  do {                                                                                       \
    if ((blockIdx.x >> 1) == ((ATTNFUSE_TRACE) >> 1))                                        \
      g_pair_trace[blockIdx.x & 1][64][0] = clock64();                                       \
  } while (0)
#else
#define AF_PTRACE_START() \
  do {                    \
  } while (0)
#define AF_PTRACE(i, e) \
  do {                  \
  } while (0)
#endif

namespace {

constexpr int kPD = 128;              // head dim
constexpr int kPBM = 128;             // query rows per CTA
constexpr int kPBN = 128;             // keys per kv tile (64 per CTA for K)
constexpr int kPThreads = 512;
constexpr int kPKSt = 6;              // K stages (released when S is done)
constexpr int kPVSt = 5;              // V stages (released when PV is done)
constexpr uint32_t kQTile = 128u * 128u * 2u;  // 32 KB: 128 rows x 128 dims
constexpr uint32_t kKHalf = 64u * 128u * 2u;   // 16 KB: 64 keys x 128 dims, 2 panels of 8 KB
constexpr uint32_t kVHalf = 128u * 64u * 2u;   // 16 KB: 128 keys x 64 dims, 1 panel
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kQTile;
constexpr uint32_t kOffV = kOffK + kPKSt * kKHalf;
constexpr uint32_t kOffCtl = kOffV + kPVSt * kVHalf;
constexpr uint32_t kTmS = 0, kTmO = 256, kTmQ = 384, kTmP = 448;

#ifndef ATTNFUSE_REGS_LOW
#define ATTNFUSE_REGS_LOW 40
#define ATTNFUSE_REGS_ROT 104
#define ATTNFUSE_REGS_SM 184
#endif
constexpr uint32_t kRegsLow = ATTNFUSE_REGS_LOW;  // warpgroup 0: TMA, MMA, relays
constexpr uint32_t kRegsRot = ATTNFUSE_REGS_ROT;  // warpgroup 3: K rotation
constexpr uint32_t kRegsSm = ATTNFUSE_REGS_SM;    // warpgroups 1, 2: softmax
static_assert(kRegsLow + kRegsRot + 2 * kRegsSm <= 4 * (65536 / kPThreads),
              "register split exceeds the registers the CTA is launched with");

struct PairCtl {
  // local TMA completion
  uint64_t q_full, k_full[kPKSt], v_full[kPVSt];
  // pair-MMA commits (multicast to both CTAs); pv_done[t] completes once per PV of a tile
  // of parity t, so each softmax warpgroup waits on consecutive phases of one barrier
  uint64_t k_empty[kPKSt], v_empty[kPVSt], s_full[2], pv_done[2], mma_final;
  // gathered from both CTAs, waited on by the MMA issuer of the even CTA
  uint64_t q_ready, k_ready[kPKSt], v_ready[kPVSt], s_free[2], p_full;
  // softmax warpgroups: O's row scale published by the owner of tile i (msync[i & 1]), and
  // the final exchange of the two partial sums (xchg)
  uint64_t msync[2], xchg;
  uint32_t tmem_base;
  int abort_flag;
  int lo[2], hi[2], valid[2], q0[2], head[2];
  int jb, je;                              // kv tiles [jb, je) either CTA needs
  int16_t nxt[kBsMaxN / kPBN + 1];         // block-sparse: next needed tile after j
  uint32_t tile_bits[2][kTileWords];
  uint32_t row_bits[2][2][kBsWords];
  float m_sh[128];         // O's row scale (log2 units)
  float red_m[2][128];     // [warpgroup][row] final scale and partial sum
  float red_l[2][128];
};

constexpr size_t kPairSmem = 1024 + kOffCtl + sizeof(PairCtl);
static_assert(kPairSmem <= 232448, "shared memory budget");

__device__ __forceinline__ bool pbit(const uint32_t* w, int i) { return (w[i >> 5] >> (i & 31)) & 1u; }

// Iteration over the kv tiles either CTA of the pair needs: every tile of [jb, je) except
// with block-sparse masks, where a per-CTA table gives the next needed tile. The loops keep
// only these few values live: the full masking rules are evaluated once per CTA (tile
// bitmaps, per-row thresholds), never per tile on the critical path.
struct TileIter {
  int jb, je;
  bool bs;
  const int16_t* nxt;
};

__device__ __forceinline__ int tile_next(const TileIter& T, int j) { return T.bs ? T.nxt[j] : j + 1; }

// Arrive on a barrier of the even CTA: a plain shared::cta arrive there, a shared::cluster
// arrive from the odd CTA.
__device__ __forceinline__ void arrive_leader(uint64_t* bar, int rank) {
  if (rank == 0)
    mbar_arrive(bar);
  else
    mbar_arrive_cluster(mapa_shared(smem_u32(bar), 0));
}

}  // namespace

// RK: how the score operands are produced (kRopeNone / kRopeFused / kRopePrerotated).
// BIAS: score bias compiled in (0 none, 1 ALiBi, 2 additive); a separate instantiation per
// kind keeps the softmax loop body small.
template <int RK, int BIAS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  PairCtl* ctl = reinterpret_cast<PairCtl*>(smem + kOffCtl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const VariantDev& var = p.var;
  constexpr bool ROPE = (RK == kRopeFused);
  const int rank = static_cast<int>(cluster_ctarank());

  // ---------------- work unit (identical in both CTAs of the pair) ----------------
  const int cid = static_cast<int>(blockIdx.x) >> 1;
  const int per_t = p.B * p.pairs;
  const int t = p.num_t - 1 - cid / per_t;  // longest first
  const int rem = cid % per_t;
  const int b = rem / p.pairs, pr = rem % p.pairs;
  const int TK = (p.N + kPBN - 1) / kPBN;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      const int head = p.pair_heads ? 2 * pr + s : pr;
      const int q0 = p.pair_heads ? t * kPBM : (2 * t + s) * kPBM;
      ctl->head[s] = head;
      ctl->q0[s] = q0;
      const bool valid = q0 < p.N && head < p.Hq;
      ctl->valid[s] = valid;
      int lo = 0, hi = TK;
      const int m_hi = min(q0 + kPBM - 1, p.N - 1);
      if (var.causal) hi = min(hi, m_hi / kPBN + 1);
      if (var.mask == 2) {
        lo = max(0, q0 - var.window + 1) / kPBN;
        if (!var.causal) hi = min(hi, (m_hi + var.window - 1) / kPBN + 1);
      }
      ctl->lo[s] = lo;
      ctl->hi[s] = valid ? hi : lo;
    }
    int jb = TK, je = 0;
    for (int s = 0; s < 2; ++s)
      if (ctl->valid[s] && ctl->lo[s] < ctl->hi[s]) {
        jb = min(jb, ctl->lo[s]);
        je = max(je, ctl->hi[s]);
      }
    ctl->jb = jb < je ? jb : 0;
    ctl->je = jb < je ? je : 0;
    ctl->abort_flag = 0;
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < kPKSt; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
      mbar_init(&ctl->k_ready[s], ROPE ? 8 : 2);
    }
    for (int s = 0; s < kPVSt; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
      mbar_init(&ctl->v_ready[s], 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->s_full[s], 1);
      mbar_init(&ctl->s_free[s], 8);   // the 4 warps of the owning warpgroup, both CTAs
      mbar_init(&ctl->pv_done[s], 1);
      mbar_init(&ctl->msync[s], 4);
    }
    mbar_init(&ctl->xchg, 8);
    mbar_init(&ctl->mma_final, 2);     // one commit per issuer
    mbar_init(&ctl->q_ready, 16);      // all 8 softmax warps, both CTAs
    mbar_init(&ctl->p_full, 8);
    fence_mbar_init();
  }
  if (var.mask == 3) {
    for (int i = tid; i < 2 * kTileWords; i += kPThreads) (&ctl->tile_bits[0][0])[i] = 0;
    for (int i = tid; i < 4 * kBsWords; i += kPThreads) (&ctl->row_bits[0][0][0])[i] = 0;
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctl->tmem_base, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  if (tid == 0) AF_PTRACE_START();

  if (var.mask == 3) {
    // Mark active kv tiles (and, for 64-blocks, active block columns per block row).
    const int blk = var.bs_block;
    for (int s = 0; s < 2; ++s) {
      if (!ctl->valid[s]) continue;
      const int br0 = ctl->q0[s] / blk;
      const int nbr = kPBM / blk;
      const int nb_total = (p.N + blk - 1) / blk;
      for (int r = 0; r < nbr; ++r) {
        const int br = br0 + r;
        if (br >= nb_total) continue;
        const int e0 = var.bs_row_ptr[br], e1 = var.bs_row_ptr[br + 1];
        for (int e = e0 + tid; e < e1; e += kPThreads) {
          const int col = var.bs_col_idx[e];
          if (col < 0 || col >= nb_total) continue;
          const int tile = col * blk / kPBN;
          atomicOr(&ctl->tile_bits[s][tile >> 5], 1u << (tile & 31));
          if (blk == 64) atomicOr(&ctl->row_bits[s][r][col >> 5], 1u << (col & 31));
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      // next-needed-tile table over [jb, je); jb moves to the first needed tile
      int nx = ctl->je;
      for (int j = ctl->je - 1; j >= ctl->jb; --j) {
        ctl->nxt[j] = static_cast<int16_t>(nx);
        bool need = false;
        for (int s = 0; s < 2; ++s)
          need |= (j >= ctl->lo[s] && j < ctl->hi[s] && pbit(ctl->tile_bits[s], j));
        if (need) nx = j;
      }
      ctl->jb = nx;
    }
    __syncthreads();
  }

  const uint32_t tmem = ctl->tmem_base;
  TileIter T;
  T.jb = ctl->jb;
  T.je = ctl->je;
  T.bs = (var.mask == 3);
  T.nxt = ctl->nxt;
  const int jb = T.jb, je = T.je;
  const int kvh = ctl->head[0] / p.g;
  int* status = p.status;
  volatile int* abort_flag = &ctl->abort_flag;

  if (warp < 4) {
    setmaxnreg_dec<kRegsLow>();
    if (warp == 0 && lane == 0) {
      // ======================= TMA producer =======================
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      const uint64_t pol_stream = l2_policy_evict_first();
      const uint64_t pol_keep = l2_policy_evict_last();
      // (cos, sin) rows this CTA reads soon: the 8 its Q rotation starts from, then per K tile
      // the 16 rows its rotators start from; pulled into L2 ahead of the reads.
      auto prefetch_rows = [&](int row0, int rows) {
        rows = min(rows, p.N - row0);
        if (ROPE && rows > 0)
          prefetch_l2_bulk(p.rope_cs + (size_t)row0 * (kPD / 2), static_cast<uint32_t>(rows) * (kPD / 2) * 8u);
      };
      if (ctl->valid[rank]) prefetch_rows(ctl->q0[rank], 8);
      if (ctl->valid[rank]) {
        mbar_arrive_expect_tx(&ctl->q_full, kQTile);
        for (int pn = 0; pn < 2; ++pn)
          tma_load_4d_hint(smem + kOffQ + pn * (kPBM * 128), &p.tmQ, &ctl->q_full, pn * 64,
                           ctl->q0[rank], ctl->head[rank], b, pol_stream);
      }
      // K and V stages are recycled by different MMAs (S and PV), so neither copy stream
      // waits for the other: the free-stage barriers are polled and whichever copy can go is
      // issued, K first (K(i+1) is needed before V(i)). The poll is bounded like every wait.
      int ik = 0, iv = 0;
      int jk = jb, jv = jk;
      uint64_t t0 = 0;
      uint32_t idle = 0;
      while (jk < je || jv < je) {
        bool moved = false;
        if (jk < je) {
          const int s = ik % kPKSt;
          if (ik < kPKSt || mbar_test(&ctl->k_empty[s], ((ik / kPKSt) - 1) & 1)) {
            AF_PTRACE(ik, 0);
            prefetch_rows(jk * kPBN + rank * 64, 16);
            mbar_arrive_expect_tx(&ctl->k_full[s], kKHalf);
            for (int pn = 0; pn < 2; ++pn)
              tma_load_4d_hint(smem + kOffK + s * kKHalf + pn * (64 * 128), &p.tmK,
                               &ctl->k_full[s], pn * 64, jk * kPBN + rank * 64, kvh, b, pol_keep);
            ++ik;
            jk = tile_next(T, jk);
            moved = true;
          }
        }
        if (jv < je && iv < ik) {
          const int s = iv % kPVSt;
          if (iv < kPVSt || mbar_test(&ctl->v_empty[s], ((iv / kPVSt) - 1) & 1)) {
            AF_PTRACE(iv, 1);
            mbar_arrive_expect_tx(&ctl->v_full[s], kVHalf);
            tma_load_4d_hint(smem + kOffV + s * kVHalf, &p.tmV, &ctl->v_full[s], rank * 64,
                             jv * kPBN, kvh, b, pol_keep);
            ++iv;
            jv = tile_next(T, jv);
            moved = true;
          }
        }
        if (moved) {
          idle = 0;
        } else if ((++idle & 255u) == 1u) {
          const uint64_t now = globaltimer_ns();
          if (idle == 1u) t0 = now;
          if (*abort_flag) break;
          if (now - t0 > ATTNFUSE_WAIT_LIMIT_NS) {
            atomicExch(status, kDevTimeout);
            *abort_flag = 1;
            break;
          }
        }
      }
      // Drain: no copy may still be landing in shared memory when the CTA exits.
      for (int k = max(0, ik - kPKSt); k < ik; ++k)
        mbar_wait(&ctl->k_full[k % kPKSt], (k / kPKSt) & 1, status, nullptr);
      for (int k = max(0, iv - kPVSt); k < iv; ++k)
        mbar_wait(&ctl->v_full[k % kPVSt], (k / kPVSt) & 1, status, nullptr);
    } else if ((warp == 1 || warp == 2) && lane == 0 && rank == 0) {
      // ======================= pair-MMA issuers =======================
      // Warp 1 issues every score MMA S(i) = Q' K(i)^T, warp 2 every O += P(i) V(i). The two
      // streams are independent (separate accumulators and operands; the softmax orders S
      // buffers, P and O through the barriers), and a thread's commits track only its own
      // MMAs. With one issuer, each wait or commit between MMA groups stalls it until its
      // queued MMAs drain and the tensor pipe idles; two issuers overlap those gaps.
      int n = 0;
      for (int j = jb; j < je; j = tile_next(T, j)) ++n;
      bool ok = mbar_wait_cluster(&ctl->q_ready, 0, status, abort_flag);
      if (warp == 1) AF_PTRACE(0, 24);
      if (warp == 1) {
        constexpr uint32_t idesc_s = idesc_f32acc(256, kPBN, 0, 0, RK != kRopeNone);
        const uint32_t sK = smem_u32(smem + kOffK);
        for (int i = 0; ok && i < n; ++i) {
          const int st = i % kPKSt, bf = i & 1;
          ok = mbar_wait_cluster(&ctl->k_ready[st], (i / kPKSt) & 1, status, abort_flag);
          AF_PTRACE(i, 4);
          if (ok && i >= 2)
            ok = mbar_wait_cluster(&ctl->s_free[bf], ((i - 2) >> 1) & 1, status, abort_flag);
          if (!ok) break;
          AF_PTRACE(i, 5);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kPD / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(
                sK + st * kKHalf + (kk >> 2) * (64 * 128) + (kk & 3) * 32, 16, 1024);
            mma_ts_pair(tmem + kTmS + bf * 128, tmem + kTmQ + kk * 8, bd, idesc_s, kk > 0);
          }
          mma_commit_pair(&ctl->s_full[bf], 3);
          mma_commit_pair(&ctl->k_empty[st], 3);
          AF_PTRACE(i, 19);
        }
      } else {
        constexpr uint32_t idesc_o = idesc_bf16_f32(256, kPD, 0, 1);
        const uint32_t sV = smem_u32(smem + kOffV);
        for (int i = 0; ok && i < n; ++i) {
          const int vs = i % kPVSt;
          ok = mbar_wait_cluster(&ctl->v_ready[vs], (i / kPVSt) & 1, status, abort_flag);
          AF_PTRACE(i, 6);
          if (ok) ok = mbar_wait_cluster(&ctl->p_full, i & 1, status, abort_flag);
          if (!ok) break;
          AF_PTRACE(i, 7);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kPBN / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(sV + vs * kVHalf + kk * 2048, kVHalf, 1024);
            mma_ts_pair(tmem + kTmO, tmem + kTmP + kk * 8, bd, idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_pair(&ctl->pv_done[i & 1], 3);
          mma_commit_pair(&ctl->v_empty[vs], 3);
          AF_PTRACE(i, 20);
        }
      }
      // All MMAs of both issuers must finish before TMEM is released.
      mma_commit_pair(&ctl->mma_final, 3);
      mbar_wait(&ctl->mma_final, 0, status, nullptr);
    } else if (warp == 3 && lane == 0) {
      // ======================= K / V relay =======================
      // Forwards "this CTA's half landed" to the even CTA in the order the MMAs consume the
      // stages: K(0), then K(i+1) and V(i). With fused RoPE the rotators forward K.
      int n = 0;
      for (int j = jb; j < je; j = tile_next(T, j)) ++n;
      bool good = true;
      for (int i = 0; good && i <= n; ++i) {
        if (!ROPE && i < n) {
          const int st = i % kPKSt;
          good = mbar_wait(&ctl->k_full[st], (i / kPKSt) & 1, status, abort_flag);
          if (good) arrive_leader(&ctl->k_ready[st], rank);
        }
        if (good && i >= 1) {
          const int st = (i - 1) % kPVSt;
          good = mbar_wait(&ctl->v_full[st], ((i - 1) / kPVSt) & 1, status, abort_flag);
          if (good) arrive_leader(&ctl->v_ready[st], rank);
        }
      }
    }
  } else if (warp >= 12) {
    // ======================= K rotators (fused RoPE) =======================
    setmaxnreg_dec<kRegsRot>();
    if (ROPE) {
      // Thread (c, rg) rotates chunk pair c of rows rg, rg+16, rg+32, rg+48 of this CTA's
      // 64-key half; the (cos, sin) of successive rows advance by the angle of 16 positions.
      const int rt = tid - 384;
      const int c = rt & 7, rg = rt >> 3;
      const int kN = p.N;
      const float2* const cs_tab = p.rope_cs;
      uint64_t wc2[4], ws2[4];  // (cos, sin) of 16 positions, pairs of dims
      {
        float wc[8], ws[8];
        load_cs8(cs_tab + (size_t)16 * (kPD / 2) + c * 8, wc, ws);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          wc2[w] = f2_pack(wc[2 * w], wc[2 * w + 1]);
          ws2[w] = f2_pack(ws[2 * w], ws[2 * w + 1]);
        }
      }
      // The first row's (cos, sin) of the next tile is read one tile ahead, from a clamped
      // (always valid) table row so the load never blocks; rows past N are not rotated.
      float4 pre[4];
      const uint64_t pol_tab = l2_policy_evict_last();  // the table stays in L2
      auto fetch = [&](int jj) {
        const int pos = min(jj * kPBN + rank * 64 + rg, kN - 1);
        const float4* src = reinterpret_cast<const float4*>(cs_tab + (size_t)pos * (kPD / 2) + c * 8);
#pragma unroll
        for (int w = 0; w < 4; ++w) pre[w] = ldg_f4_hint(src + w, pol_tab);
      };
      fetch(jb);
      int i = 0;
      for (int j = jb; j < je; j = tile_next(T, j), ++i) {
        const int st = i % kPKSt;
        const int n0 = j * kPBN + rank * 64;
        uint64_t c2[4], s2[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          c2[w] = f2_pack(pre[w].x, pre[w].z);
          s2[w] = f2_pack(pre[w].y, pre[w].w);
        }
        {
          const int jn = tile_next(T, j);
          fetch(jn < je ? jn : j);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&ctl->k_full[st], (i / kPKSt) & 1, status, abort_flag)))
          break;
        if (rt == 0) AF_PTRACE(i, 2);
        uint8_t* tile = smem + kOffK + st * kKHalf;
        // two rows at a time: both rows' chunks first, then rotate and store them
#pragma unroll
        for (int k2 = 0; k2 < 4; k2 += 2) {
          uint4 lo[2], hi[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint32_t offl = sw128_offset(rg + 16 * (k2 + k), c);
            lo[k] = *reinterpret_cast<const uint4*>(tile + offl);
            hi[k] = *reinterpret_cast<const uint4*>(tile + offl + 64 * 128);
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint64_t ns2[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) ns2[w] = s2[w] ^ 0x8000000080000000ull;
            rot_chunk_cs2<true>(lo[k], hi[k], c2, s2, ns2);
            if (k2 + k + 1 < 4) {
              uint64_t nws2[4];
#pragma unroll
              for (int w = 0; w < 4; ++w) nws2[w] = ws2[w] ^ 0x8000000080000000ull;
              advance_cs2(c2, s2, ns2, wc2, ws2, nws2);
            }
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (n0 + rg + 16 * (k2 + k) < kN) {
              const uint32_t offl = sw128_offset(rg + 16 * (k2 + k), c);
              *reinterpret_cast<uint4*>(tile + offl) = lo[k];
              *reinterpret_cast<uint4*>(tile + offl + 64 * 128) = hi[k];
            }
          }
        }
        if (rt == 0) AF_PTRACE(i, 9);
        fence_proxy_async_smem();
        __syncwarp();
        if (rt == 0) AF_PTRACE(i, 3);
        if (lane == 0) arrive_leader(&ctl->k_ready[st], rank);
      }
    }
  } else {
    // ======================= softmax (one query row per thread, one column half) ===========
    setmaxnreg_inc<kRegsSm>();
    const int h = (warp - 4) >> 2;           // key columns 64h .. 64h+63 of each tile
    const int wq = warp & 3;                 // TMEM lane quarter
    if (lane == 0 && wq == 0) AF_PTRACE(h, 26);
    const int r = wq * 32 + lane;            // row within this CTA's 128 rows
    const int s = rank;
    const int q0 = ctl->q0[s];
    const int m = q0 + r;
    const int head = ctl->head[s];
    const bool valid = ctl->valid[s] != 0;
    const int N = p.N;
    // This sub-tile's tiles: [lo_s, hi_s), minus block-sparse holes; tiles outside
    // [jm_lo, jm_hi) need per-element masks (sequence end, causal diagonal, window edges).
    const int lo_s = ctl->lo[s], hi_s = ctl->hi[s];
    const bool bs = var.mask == 3, bs64 = bs && var.bs_block == 64;
    int jm_lo = 0, jm_hi = N / kPBN;
    {
      const int q_last = min(q0 + kPBM - 1, N - 1);
      if (var.causal) jm_hi = min(jm_hi, q0 / kPBN);
      if (var.mask == 2) {
        const int lim = q_last - var.window + 1;     // first key of the last row's window
        if (lim > 0) jm_lo = (lim + kPBN - 1) / kPBN;
        if (!var.causal) {
          const int e = q0 + var.window - kPBN;      // tiles ending past the first row's window
          jm_hi = min(jm_hi, e >= 0 ? e / kPBN + 1 : 0);
        }
      }
    }
    const int vab16 = var.add_bias_bf16;
    const int64_t ab_s3 = var.ab_s[3];
    const void* add_bias = var.add_bias;
    const int64_t ab_row = b * var.ab_s[0] + head * var.ab_s[1] + (int64_t)m * var.ab_s[2];
    uint8_t* const visits = var.visits;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    bool ok = true;

    // ---- Q' = R_m Q (fp16 with fused RoPE) into TMEM: this thread writes chunk pairs
    // 4h..4h+3 of row r, i.e. dims 32h..32h+31 (columns 16h..) and 64+32h.. (columns 32+16h..)
    {
      uint32_t qlo[16], qhi[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) qlo[e] = qhi[e] = 0u;
      if (ROPE) {
        // Rotate the Q tile in place first, one row per warp instruction: softmax warp w takes
        // rows w, w + 8, ..., and lane f the table entries 2f, 2f+1 of the row (one coalesced
        // 16-byte read) and dims 2f, 2f+1 with their partners 64+2f, 64+2f+1. The table reads
        // are issued before Q lands. Same arithmetic per element as a row-per-thread rotation.
        const int sw = warp - 4;
        const uint64_t pol_tab = l2_policy_evict_last();  // the table stays in L2
        // the query-tile recurrence (query_cs8): start at position q0 + sw, step 8 positions
        const float4* tab = reinterpret_cast<const float4*>(p.rope_cs);
        float4 cs = ldg_f4_hint(tab + (size_t)min(q0 + sw, N - 1) * (kPD / 4) + lane, pol_tab);
        const float4 wstep = ldg_f4_hint(tab + (size_t)8 * (kPD / 4) + lane, pol_tab);
        if (lane == 0 && wq == 0) AF_PTRACE(h, 25);
        if (valid) ok = __all_sync(0xffffffffu, mbar_wait(&ctl->q_full, 0, status, abort_flag));
        if (lane == 0 && wq == 0) AF_PTRACE(h, 21);
        if (valid && ok) {
          uint8_t* tile = smem + kOffQ;
          const uint32_t within = static_cast<uint32_t>(lane & 3) * 4u;
#pragma unroll
          for (int k = 0; k < kPBM / 8; ++k) {
            const int rr = sw + 8 * k;
            if (q0 + rr < N) {
              const uint32_t off = sw128_offset(rr, lane >> 2) + within;
              const uint32_t l2w = *reinterpret_cast<const uint32_t*>(tile + off);
              const uint32_t h2w = *reinterpret_cast<const uint32_t*>(tile + kPBM * 128 + off);
              float yl0, yh0, yl1, yh1;
              rot_pair(bf16lo_to_f32(l2w), bf16lo_to_f32(h2w), cs.x, cs.y, yl0, yh0);
              rot_pair(bf16hi_to_f32(l2w), bf16hi_to_f32(h2w), cs.z, cs.w, yl1, yh1);
              *reinterpret_cast<uint32_t*>(tile + off) = pack_f16x2_sat(yl0, yl1);
              *reinterpret_cast<uint32_t*>(tile + kPBM * 128 + off) = pack_f16x2_sat(yh0, yh1);
            }
            if (k + 1 < kPBM / 8) {  // next row of this warp: 8 positions on (advance_cs8 order)
              float c0, s0, c1, s1;
              rot_pair(cs.x, cs.y, wstep.x, wstep.y, c0, s0);
              rot_pair(cs.z, cs.w, wstep.z, wstep.w, c1, s1);
              cs = make_float4(c0, s0, c1, s1);
            }
          }
        }
        if (lane == 0 && wq == 0) AF_PTRACE(h, 23);
        named_bar_sync(1, 256);  // the eight softmax warps: rows rotated by other warps
        if (lane == 0 && wq == 0) AF_PTRACE(h, 27);
      } else {
        if (valid) ok = __all_sync(0xffffffffu, mbar_wait(&ctl->q_full, 0, status, abort_flag));
      }
      if (valid && ok) {
        const uint8_t* tile = smem + kOffQ;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c = 4 * h + cc;
          const uint4 lo = *reinterpret_cast<const uint4*>(tile + sw128_offset(r, c));
          const uint4 hi = *reinterpret_cast<const uint4*>(tile + kPBM * 128 + sw128_offset(r, c));
          qlo[4 * cc + 0] = lo.x; qlo[4 * cc + 1] = lo.y; qlo[4 * cc + 2] = lo.z; qlo[4 * cc + 3] = lo.w;
          qhi[4 * cc + 0] = hi.x; qhi[4 * cc + 1] = hi.y; qhi[4 * cc + 2] = hi.z; qhi[4 * cc + 3] = hi.w;
        }
      }
      if (ok) {
        tmem_st16(tmem + lane_off + kTmQ + 16 * h, qlo);
        tmem_st16(tmem + lane_off + kTmQ + 32 + 16 * h, qhi);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && wq == 0) AF_PTRACE(h, 22);
        if (lane == 0) arrive_leader(&ctl->q_ready, rank);
      }
    }

    // Online softmax over alternate tiles: warpgroup h takes tiles i = h, h+2, ... with full
    // 128-column rows, so one warpgroup's exponentials overlap the other's loads, maxima and
    // stores. Both feed the single O accumulator, whose row scale m_sh[r] (log2 units) only
    // grows, and lazily (by more than 8). A tile's P is computed against this warpgroup's last
    // scale and reconciled with O's scale once the previous tile's PV has completed; the P
    // buffer and O belong to one tile at a time.
    float m_h = kNegInf, l_h = 0.f;  // this warpgroup's partial row sum and its scale
    const float scale_log2 = p.scale_log2;
    const float alibi = (BIAS == 1 && valid) ? var.slopes[head] * kLog2e : 0.f;
    const int blk_row = bs64 ? (r >> 6) : 0;
    const uint32_t tP = tmem + lane_off + kTmP;
    const uint32_t tOall = tmem + lane_off + kTmO;
    int i = 0;
    for (int j = jb; ok && j < je; j = tile_next(T, j), ++i) {
      if ((i & 1) != h) continue;
      const bool act = j >= lo_s && j < hi_s && (!bs || pbit(ctl->tile_bits[s], j));
      bool h0 = true, h1 = true;  // block-sparse 64-blocks of this tile present for the row
      if (bs64) {
        h0 = pbit(ctl->row_bits[s][blk_row], 2 * j);
        h1 = pbit(ctl->row_bits[s][blk_row], 2 * j + 1);
      }
      // Every wait result is voted across the warp so TMEM collectives never diverge.
      if (!__all_sync(0xffffffffu, mbar_wait(&ctl->s_full[h], (i >> 1) & 1, status, abort_flag))) {
        ok = false;
        break;
      }
      if (lane == 0 && wq == 0) AF_PTRACE(i, h ? 14 : 8);
      tc_fence_after();
      uint32_t xr[128];
      tmem_ld32<0>(tmem + lane_off + kTmS + h * 128, xr);
      tmem_ld32<32>(tmem + lane_off + kTmS + h * 128 + 32, xr);
      tmem_ld32<64>(tmem + lane_off + kTmS + h * 128 + 64, xr);
      tmem_ld32<96>(tmem + lane_off + kTmS + h * 128 + 96, xr);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(&ctl->s_free[h], rank);
      float x[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(xr[c]);
      const int k0 = j * kPBN;
      // ---- score combinators (log2 domain) ----
      float mul = scale_log2;
      if constexpr (BIAS != 0) {
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] *= scale_log2;
        mul = 1.f;
        if constexpr (BIAS == 1) {
          const float base = alibi * static_cast<float>(k0 - m);
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] = __fmaf_rn(alibi, static_cast<float>(c), x[c] + base);
        } else if (act) {
          // Branch-free loads (lanes past the sequence end read element 0 and drop it), so the
          // warp stays converged for the warp-collective TMEM operations that follow.
          const int c_end = (m < N) ? min(kPBN, N - k0) : 0;
          if (vab16) {
            const __nv_bfloat16* ab = static_cast<const __nv_bfloat16*>(add_bias);
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              const float raw = __bfloat162float(ab[c < c_end ? ab_row + (int64_t)(k0 + c) * ab_s3 : 0]);
              x[c] += (c < c_end ? raw : 0.f) * kLog2e;
            }
          } else {
            const float* ab = static_cast<const float*>(add_bias);
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              const float raw = ab[c < c_end ? ab_row + (int64_t)(k0 + c) * ab_s3 : 0];
              x[c] += (c < c_end ? raw : 0.f) * kLog2e;
            }
          }
        }
      }
      if (__builtin_expect(!act || !h0 || !h1 || j < jm_lo || j >= jm_hi, 0)) {
        // per-element mask (cold: sequence end, causal diagonal, window edges, holes)
        int c_lo = 0, c_hi = act ? min(kPBN - 1, N - 1 - k0) : -1;
        if (var.causal) c_hi = min(c_hi, m - k0);
        if (var.mask == 2) {
          c_lo = max(c_lo, m - var.window + 1 - k0);
          if (!var.causal) c_hi = min(c_hi, m + var.window - 1 - k0);
        }
#pragma unroll
        for (int c = 0; c < 128; ++c)
          x[c] = (c >= c_lo && c <= c_hi && (c < 64 ? h0 : h1)) ? x[c] : kNegInf;
      }
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
      // exponentials against this warpgroup's scale unless the tile exceeds it by more than 8
      const float m_base = (mx > m_h + 8.0f) ? mx : m_h;
      const float nb = (m_base == kNegInf) ? 0.f : -m_base;
      const uint64_t mul2v = f2_pack(mul, mul), nb2 = f2_pack(nb, nb);
      uint64_t acc2[4] = {0, 0, 0, 0};
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const uint64_t a = fma2(f2_pack(x[2 * c], x[2 * c + 1]), mul2v, nb2);
        const float p0 = ex2_approx(f2_lo(a)), p1 = ex2_approx(f2_hi(a));
        acc2[c & 3] = add2(acc2[c & 3], f2_pack(p0, p1));
        pk[c] = pack_bf16x2(p0, p1);
      }
      const uint64_t acc = add2(add2(acc2[0], acc2[1]), add2(acc2[2], acc2[3]));
      float sum = f2_lo(acc) + f2_hi(acc);
      if (lane == 0 && wq == 0) AF_PTRACE(i, 10 + h);
      // ---- P buffer and O become this tile's once PV(i-1) has completed ----
      float m_cur = kNegInf;  // O's row scale
      if (i > 0) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&ctl->pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, status, abort_flag) &&
                            mbar_wait(&ctl->msync[(i - 1) & 1], ((i - 1) >> 1) & 1, status, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        m_cur = ctl->m_sh[r];
      }
      const float m_fin = fmaxf(m_cur, m_base);
      if (__builtin_expect(m_base < m_fin, 0)) {
        // O is at a larger scale than this tile's exponentials: bring P down to it (rare)
        const float beta = ex2_approx(m_base - m_fin);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          pk[c] = pack_bf16x2(bf16lo_to_f32(pk[c]) * beta, bf16hi_to_f32(pk[c]) * beta);
        sum *= beta;
      }
      // tcgen05.ld/st are warp-collective: rescale O for the whole warp when any row's scale
      // grows (alpha = 1 for rows that do not)
      const bool grow = i > 0 && m_cur < m_fin;
      if (__builtin_expect(__any_sync(0xffffffffu, grow), 0)) {
        const float alpha = grow ? ex2_approx(m_cur - m_fin) : 1.f;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t o[32];
          tmem_ld32(tOall + ch * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tOall + ch * 32, o);
        }
      }
      l_h = ((m_h == m_fin || m_h == kNegInf) ? l_h : l_h * ex2_approx(m_h - m_fin)) + sum;
      m_h = m_fin;
      ctl->m_sh[r] = m_fin;
      tmem_st32<0>(tP, pk);
      tmem_st32<32>(tP + 32, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && wq == 0) AF_PTRACE(i, h ? 15 : 12);
      if (lane == 0) {
        arrive_leader(&ctl->p_full, rank);
        mbar_arrive(&ctl->msync[i & 1]);
      }
      if (act && visits && r == 0) {
        const int TQ = (N + kPBM - 1) / kPBM;
        visits[((static_cast<int64_t>(b) * p.Hq + head) * TQ + q0 / kPBM) * TK + j] = 1;
      }
    }
    const int n = i;  // kv tiles of the pair
    // ---- epilogue: wait for the last PV, combine the two partial sums, O / l, LSE ----
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1,
                                             status, abort_flag));
      tc_fence_after();
    }
    float m_fin = m_h, l_tot = l_h;
    if (ok) {
      ctl->red_m[h][r] = m_h;
      ctl->red_l[h][r] = l_h;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->xchg);
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->xchg, 0, status, abort_flag));
      if (ok) {
        const float m_o = ctl->red_m[h ^ 1][r], l_o = ctl->red_l[h ^ 1][r];
        m_fin = fmaxf(m_h, m_o);
        l_tot = (m_h == kNegInf ? 0.f : l_h * ex2_approx(m_h - m_fin)) +
                (m_o == kNegInf ? 0.f : l_o * ex2_approx(m_o - m_fin));
      }
    }
    if (valid) {
      const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
      const uint32_t tO = tOall + 64 * h;
      __nv_bfloat16* orow = p.out + b * p.o_sb + head * p.o_sh + (int64_t)m * p.o_sn + 64 * h;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t o[32];
        if (ok && n > 0) {
          tmem_ld32(tO + ch * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
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
      if (h == 0 && p.lse && m < N)
        p.lse[(static_cast<int64_t>(b) * p.Hq + head) * N + m] =
            (l_tot > 0.f) ? (m_fin + log2f(l_tot)) * kLn2 : kNegInf;
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync();  // the peer is done with this CTA's barriers and all pair MMAs have finished
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

size_t fwd_pair_smem_size() { return kPairSmem; }

}  // namespace afx

#ifdef ATTNFUSE_TRACE
// Copy the pair-kernel pipeline trace (2 CTAs x 65 rows x 32 events of clock64) to host memory.
extern "C" int attnfuse_pair_trace_read(unsigned long long* dst) {
  return (int)cudaMemcpyFromSymbol(dst, afx::g_pair_trace, sizeof(unsigned long long) * 2 * 65 * 32);
}
#endif

namespace afx {

template <int RK>
static void (*pick_pair(int bias))(FwdParams) {
  return bias == 1 ? fwd_pair_kernel<RK, 1> : bias == 2 ? fwd_pair_kernel<RK, 2> : fwd_pair_kernel<RK, 0>;
}

cudaError_t launch_fwd_pair(const FwdParams& p, int rope_kind, int clusters, cudaStream_t stream) {
  void (*fn)(FwdParams) = rope_kind == kRopeFused        ? pick_pair<kRopeFused>(p.var.bias)
                          : rope_kind == kRopePrerotated ? pick_pair<kRopePrerotated>(p.var.bias)
                                                         : pick_pair<kRopeNone>(p.var.bias);
  cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmem);
  if (e != cudaSuccess) return e;
  fn<<<2 * clusters, kPThreads, kPairSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace afx
