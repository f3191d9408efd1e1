// Split-KV decode for sm_103a (AttnFuse paper §4.2 Flash Decoding).
//
// Phase 1 (decode_kernel): one CTA per (KV chunk, key/value head, batch). The g query heads
// of the group become rows 0..g-1 of a 128-row query tile (rows g..127 are zero), rotated
// in-kernel at position q_pos. The CTA streams its chunk of the (already rotated) K cache and
// the V cache in 128-key tiles through TMA, computes S = Q K^T and O += P V with tcgen05.mma
// into TMEM, and keeps the online-softmax state (max, sum) per head in registers. It writes the
// unnormalised partial (acc, max, sum) of its chunk. The padded rows cost tensor work only;
// the kernel is bound by the HBM stream of the cache.
// Phase 2 (combine_kernel): merges the chunks of every (b, query head) through their
// log-sum-exp: O = sum_s w_s acc_s / sum_s w_s l_s with w_s = 2^(m_s - max_s m_s).
//
// Warps: 0 softmax (TMEM lanes 0-31 hold rows 0-31), 1 TMA, 2 MMA, 3 builds the query tile.
// TMEM: S double-buffered at columns [0,128) and [128,256), O at [256, 256+d).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "../../include/attnfuse.h"
#include "common.cuh"
#include "launch.h"

namespace afx {

namespace {

constexpr int kDecThreads = 128;
constexpr int kDecBN = 128;

constexpr int kDecST = 3;  // K and V stages: up to three tiles of the cache in flight

template <int D>
struct DecCfg {
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t TILE = 128u * D * 2u;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = TILE;
  static constexpr uint32_t OFF_V = OFF_K + kDecST * TILE;
  static constexpr uint32_t OFF_CTL = OFF_V + kDecST * TILE;
};

struct DecCtl {
  uint64_t q_ready, s_full[2], p_full, pv_done, mma_final;
  uint64_t k_full[kDecST], k_empty[kDecST], v_full[kDecST], v_empty[kDecST];
  uint32_t tmem_base;
  int abort_flag;
  float2 qcs[64];  // (cos, sin) of q_pos per pair: every query head sits at the same position
};

__host__ __device__ constexpr size_t dec_smem_bytes(int D) {
  return 1024 + (1 + 2 * kDecST) * (size_t)(128 * D * 2) + sizeof(DecCtl);
}
static_assert(1024 + 7 * 32768 + sizeof(DecCtl) <= 232448, "decode shared memory budget");

}  // namespace

template <int D, bool ROPE_Q>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const __grid_constant__ DecParams p) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  DecCtl* ctl = reinterpret_cast<DecCtl*>(smem + C::OFF_CTL);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int key0 = split * p.chunk;
  const int key1 = min(p.L, key0 + p.chunk);
  const int ntiles = (key1 - key0 + kDecBN - 1) / kDecBN;
  int* status = p.status;
  volatile int* abort_flag = &ctl->abort_flag;

  if (tid == 0) {
    mbar_init(&ctl->q_ready, 32);
    for (int i = 0; i < kDecST; ++i) {
      mbar_init(&ctl->k_full[i], 1);
      mbar_init(&ctl->k_empty[i], 1);
      mbar_init(&ctl->v_full[i], 1);
      mbar_init(&ctl->v_empty[i], 1);
    }
    mbar_init(&ctl->s_full[0], 1);
    mbar_init(&ctl->s_full[1], 1);
    mbar_init(&ctl->p_full, 32);
    mbar_init(&ctl->pv_done, 1);
    mbar_init(&ctl->mma_final, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  // zero the query tile (rows >= g stay zero)
  for (int i = tid; i < (int)(C::TILE / 16); i += kDecThreads)
    reinterpret_cast<uint4*>(smem + C::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 2) tmem_alloc(&ctl->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  // Launched as a programmatic dependent: the set-up above overlaps the end of the previous
  // kernel on the stream; global memory is read and written only once that kernel has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 3) {
    // ---- query tile: row h = R_{q_pos} q[b, kvh*g + h], bf16, 128B-swizzled ----
    // Every chunk of the row is loaded (read-only path) first, so the global-load latency is
    // paid once and overlaps the angle computation, not once per chunk behind a store.
    constexpr int CP = D / 16;
    const int h = lane;
    uint4 lo[CP], hi[CP];
    if (h < p.g) {
      const __nv_bfloat16* qrow = p.q + b * p.q_sb + (int64_t)(kvh * p.g + h) * p.q_sh;
#pragma unroll
      for (int c = 0; c < CP; ++c) {
        lo[c] = __ldg(reinterpret_cast<const uint4*>(qrow + c * 8));
        hi[c] = __ldg(reinterpret_cast<const uint4*>(qrow + D / 2 + c * 8));
      }
    }
    if (ROPE_Q) {
      // the D/2 angles of q_pos, computed once by the whole warp
      for (int e = lane; e < D / 2; e += 32) {
        float c, sn;
        rope_cossin(static_cast<float>(p.q_pos), p.freqs.hi[e], p.freqs.lo[e], &c, &sn);
        ctl->qcs[e] = make_float2(c, sn);
      }
      __syncwarp();
    }
    if (h < p.g) {
      uint8_t* tile = smem + C::OFF_Q;
#pragma unroll
      for (int c = 0; c < CP; ++c) {
        if (ROPE_Q) {
          float cc[8], ss[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 t = ctl->qcs[c * 8 + e];
            cc[e] = t.x;
            ss[e] = t.y;
          }
          rot_chunk_cs<false>(lo[c], hi[c], cc, ss);
        }
        uint32_t offl, offh;
        if (D == 128) {
          offl = sw128_offset(h, c);
          offh = offl + 128 * 128;
        } else {
          offl = sw128_offset(h, c);
          offh = sw128_offset(h, c + 4);
        }
        *reinterpret_cast<uint4*>(tile + offl) = lo[c];
        *reinterpret_cast<uint4*>(tile + offh) = hi[c];
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(&ctl->q_ready);
  } else if (warp == 1) {
    // ---- TMA producer: K then V of every tile of the chunk, through kDecST-deep rings ----
    if (lane == 0) {
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      const uint64_t pol = l2_policy_evict_first();  // the cache is streamed once
      int i = 0;
      for (; i < ntiles; ++i) {
        const int k0 = key0 + i * kDecBN;
        const int st = i % kDecST;
        const uint32_t ph = ((i / kDecST) - 1) & 1;
        if (i >= kDecST && !mbar_wait(&ctl->k_empty[st], ph, status, abort_flag)) break;
        mbar_arrive_expect_tx(&ctl->k_full[st], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d_hint(smem + C::OFF_K + st * C::TILE + pn * (kDecBN * 128), &p.tmK,
                           &ctl->k_full[st], pn * 64, k0, kvh, b, pol);
        if (i >= kDecST && !mbar_wait(&ctl->v_empty[st], ph, status, abort_flag)) {
          ++i;  // K(i) is in flight
          break;
        }
        mbar_arrive_expect_tx(&ctl->v_full[st], C::TILE);
        for (int pn = 0; pn < C::PANELS; ++pn)
          tma_load_4d_hint(smem + C::OFF_V + st * C::TILE + pn * (kDecBN * 128), &p.tmV,
                           &ctl->v_full[st], pn * 64, k0, kvh, b, pol);
      }
      // drain: no copy may still be landing in shared memory when the CTA exits
      for (int k = max(0, i - kDecST); k < i; ++k) {
        mbar_wait(&ctl->k_full[k % kDecST], (k / kDecST) & 1, status, nullptr);
        mbar_wait(&ctl->v_full[k % kDecST], (k / kDecST) & 1, status, nullptr);
      }
    }
  } else if (warp == 2) {
    // ---- MMA issuer ----
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kDecBN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sK = smem_u32(smem + C::OFF_K),
                     sV = smem_u32(smem + C::OFF_V);
      // S is double-buffered (columns 0 and 128); O accumulates at column 256. S(i+2) reuses
      // the buffer of tile i once PV(i) has consumed the probabilities stored there.
      auto issue_s = [&](int i) {
        const int st = i % kDecST;
        const uint32_t d_tmem = tmem + (i & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
          mma_ss(d_tmem, smem_desc_sw128(sQ + koff, 16, 1024),
                 smem_desc_sw128(sK + st * C::TILE + koff, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&ctl->s_full[i & 1]);
        mma_commit(&ctl->k_empty[st]);
      };
      bool ok = mbar_wait(&ctl->q_ready, 0, status, abort_flag);
      for (int i = 0; ok && i < 2 && i < ntiles; ++i) {
        if (!mbar_wait(&ctl->k_full[i % kDecST], (i / kDecST) & 1, status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(i);
      }
      for (int i = 0; ok && i < ntiles; ++i) {
        const int st = i % kDecST;
        if (!mbar_wait(&ctl->p_full, i & 1, status, abort_flag)) break;
        if (!mbar_wait(&ctl->v_full[st], (i / kDecST) & 1, status, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kDecBN / 16; ++kk)
          mma_ts(tmem + 256, tmem + (i & 1) * 128 + kk * 8,
                 smem_desc_sw128(sV + st * C::TILE + kk * 2048, kDecBN * 128, 1024), idesc_o,
                 (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&ctl->pv_done);
        mma_commit(&ctl->v_empty[st]);
        if (i + 2 < ntiles) {
          const int n = i + 2;
          if (!mbar_wait(&ctl->k_full[n % kDecST], (n / kDecST) & 1, status, abort_flag)) break;
          if (!mbar_wait(&ctl->pv_done, i & 1, status, abort_flag)) break;
          tc_fence_after();
          issue_s(n);
        }
      }
      mma_commit(&ctl->mma_final);
      mbar_wait(&ctl->mma_final, 0, status, nullptr);
    }
  } else {
    // ---- softmax: thread = query row (rows >= g are padding) ----
    const int r = lane;
    float m_run = kNegInf, l_run = 0.f;
    bool ok = true;
    const float c2 = p.scale_log2;
    for (int i = 0; i < ntiles; ++i) {
      const uint32_t tS = tmem + (i & 1) * 128;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&ctl->s_full[i & 1], (i >> 1) & 1, status, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t xr[kDecBN];
      tmem_ld32<0>(tS, xr);
      tmem_ld32<32>(tS + 32, xr);
      tmem_ld32<64>(tS + 64, xr);
      tmem_ld32<96>(tS + 96, xr);
      tmem_wait_ld();
      const int valid = min(kDecBN, key1 - (key0 + i * kDecBN));
      float x[kDecBN];
#pragma unroll
      for (int c = 0; c < kDecBN; ++c) x[c] = (c < valid) ? __uint_as_float(xr[c]) : kNegInf;
      float mp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mp[k] = fmaxf(x[2 * k], x[2 * k + 1]);
#pragma unroll
      for (int i2 = 1; i2 < kDecBN / 16; ++i2)
#pragma unroll
        for (int k = 0; k < 8; ++k) mp[k] = max3f(mp[k], x[16 * i2 + 2 * k], x[16 * i2 + 2 * k + 1]);
      const float mx =
          max3f(max3f(mp[0], mp[1], mp[2]), max3f(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7])) * c2;
      const float m_new = fmaxf(m_run, mx);
      float m_use = m_run;
      bool rescale = false;
      if (i == 0) {
        m_use = m_new;
      } else if (m_new > m_run + 8.0f) {
        m_use = m_new;
        rescale = true;
      }
      const float nb = (m_use == kNegInf) ? 0.f : -m_use;
      const uint64_t mul2v = f2_pack(c2, c2), nb2 = f2_pack(nb, nb);
      uint64_t acc2[4] = {0, 0, 0, 0};
      uint32_t pk[kDecBN / 2];
#pragma unroll
      for (int c = 0; c < kDecBN / 2; ++c) {
        const uint64_t a = fma2(f2_pack(x[2 * c], x[2 * c + 1]), mul2v, nb2);
        const float p0 = ex2_approx(f2_lo(a)), p1 = ex2_approx(f2_hi(a));
        acc2[c & 3] = add2(acc2[c & 3], f2_pack(p0, p1));
        pk[c] = pack_bf16x2(p0, p1);
      }
      const uint64_t acc = add2(add2(acc2[0], acc2[1]), add2(acc2[2], acc2[3]));
      tmem_st32<0>(tS, pk);
      tmem_st32<32>(tS + 32, pk);
      tmem_wait_st();
      // Only a rescale touches O, so only a rescale waits for the previous PV (PV(i) itself is
      // issued after p_full(i) and accumulates in order behind PV(i-1)).
      if (__any_sync(0xffffffffu, rescale)) {
        if (i > 0) {
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&ctl->pv_done, (i - 1) & 1, status, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const float alpha = rescale ? ex2_approx(m_run - m_use) : 1.f;
        l_run *= alpha;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tmem + 256 + ch * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tmem + 256 + ch * 32, o);
        }
        tmem_wait_st();
      }
      l_run += f2_lo(acc) + f2_hi(acc);
      m_run = m_use;
      tc_fence_before();
      mbar_arrive(&ctl->p_full);
    }
    if (ok && ntiles > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->pv_done, (ntiles - 1) & 1, status, abort_flag));
      tc_fence_after();
    }
    // ---- partials of this chunk: acc (unnormalised), max (log2 units), sum ----
    const int64_t part = ((int64_t)b * p.Hq + kvh * p.g + r) * p.splits + split;
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t o[32];
      if (ok && ntiles > 0) {
        tmem_ld32(tmem + 256 + ch * 32, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (r < p.g) {
        float4* dst = reinterpret_cast<float4*>(p.part_acc + part * D + ch * 32);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          dst[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                               __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
      }
    }
    if (r < p.g) {
      p.part_m[part] = (ok && l_run > 0.f) ? m_run : kNegInf;
      p.part_l[part] = ok ? l_run : 0.f;
    }
  }
  // Let the combine kernel launch while this grid drains (its reads wait for our completion).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

// Phase 2: one CTA per (b, query head); thread c handles output column c. The splits are read
// in parallel: thread s takes split s's (max, sum), a block reduction gives the overall max,
// the per-split weights pass through shared memory, and each column then sums its splits
// with independent loads (no chain of dependent global reads).
template <int D>
__global__ void __launch_bounds__(D) combine_kernel(const __grid_constant__ DecParams p) {
  __shared__ float w_sh[kDecMaxSplits];
  __shared__ float red[D / 32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int bh = blockIdx.x;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int c = threadIdx.x, lane = c & 31, warp = c >> 5;
  const int S = p.splits_used;
  const int64_t base = (int64_t)bh * p.splits;
  // overall max over the splits (log2 units)
  float mloc = kNegInf;
  for (int s = c; s < S; s += D) mloc = fmaxf(mloc, p.part_m[base + s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
  if (lane == 0) red[warp] = mloc;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int k = 1; k < D / 32; ++k) M = fmaxf(M, red[k]);
  __syncthreads();
  // per-split weights and their sum of row sums
  float lloc = 0.f;
  for (int s = c; s < S; s += D) {
    const float ms = p.part_m[base + s];
    const float w = (M == kNegInf || ms == kNegInf) ? 0.f : ex2_approx(ms - M);
    w_sh[s] = w;
    lloc += w * p.part_l[base + s];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, off);
  if (lane == 0) red[warp] = lloc;
  __syncthreads();
  float L = 0.f;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) L += red[k];
  // column c: sum_s w_s acc_s[c]
  float acc = 0.f;
  const float* pa = p.part_acc + base * D + c;
#pragma unroll 8
  for (int s = 0; s < S; ++s) acc += w_sh[s] * pa[(int64_t)s * D];
  const float o = (L > 0.f) ? acc / L : 0.f;
  p.out[b * p.o_sb + h * p.o_sh + c] = __float2bfloat16_rn(o);
  if (p.lse && c == 0) p.lse[bh] = (L > 0.f) ? (M + log2f(L)) * kLn2 : kNegInf;
}

size_t decode_smem_size(int d) { return dec_smem_bytes(d); }

cudaError_t launch_decode(const DecParams& p, int d, bool rope_q, cudaStream_t stream) {
  const size_t smem = dec_smem_bytes(d);
  void (*k1)(DecParams) = nullptr;
  void (*k2)(DecParams) = nullptr;
  if (d == 128) {
    k1 = rope_q ? decode_kernel<128, true> : decode_kernel<128, false>;
    k2 = combine_kernel<128>;
  } else {
    k1 = rope_q ? decode_kernel<64, true> : decode_kernel<64, false>;
    k2 = combine_kernel<64>;
  }
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launches: phase 1's set-up may overlap the previous kernel on the
  // stream, and the combine grid may start launching while phase 1 drains.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits_used, p.Hkv, p.B);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k1, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(p.B * p.Hq);
  cfg.blockDim = dim3(d);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, k2, p);
}

}  // namespace afx

// ---------------------------------------------------------------------------------------------
// Decode for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device workspace: a serving runtime whose memory is
// entirely pre-reserved by its own allocator, a host program that links this library but has
// no allocator API of its own to hand out scratch buffers, or a latency-critical path where a
// cudaMalloc (which may synchronise the device) is not allowed. For them the split-KV partial
// results live in one fixed array compiled into this library instead of in a caller buffer.
// ---------------------------------------------------------------------------------------------
namespace afx {

// Scratch for attnfuse_decode_noalloc: the partial (acc, max, sum) rows of every split. Every
// GPU that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of g_decode_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_last_error(ATTNFUSE_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_last_error(ATTNFUSE_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return set_last_error(ATTNFUSE_ERR_CUDA, cudaGetErrorString(e));
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ATTNFUSE_OK;
}
}  // namespace

}  // namespace afx

extern "C" attnfuse_status attnfuse_decode_noalloc(
    const void* q, const int64_t q_strides[3], const void* k_cache, const int64_t k_strides[4],
    const void* v_cache, const int64_t v_strides[4], void* out, const int64_t o_strides[3],
    float* lse, int B, int Hq, int Hkv, int L, int d, int q_pos, float scale, float rope_theta,
    attnfuse_rope_mode rope_mode, int num_splits, cudaStream_t stream) {
  size_t need = 0;
  attnfuse_status rc = attnfuse_decode_workspace_size(B, Hq, Hkv, L, d, num_splits, &need);
  if (rc) return rc;
  if (need > afx::kNoAllocScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "attnfuse_decode_noalloc: this problem needs %zu bytes of scratch but the built-in "
             "array holds %zu; use attnfuse_decode with a workspace or fewer splits",
             need, afx::kNoAllocScratchBytes);
    return afx::set_last_error(ATTNFUSE_ERR_WORKSPACE_TOO_SMALL, msg);
  }
  void* scratch = nullptr;
  if ((rc = afx::scratch_address(&scratch))) return rc;
  return attnfuse_decode(q, q_strides, k_cache, k_strides, v_cache, v_strides, out, o_strides, lse,
                         B, Hq, Hkv, L, d, q_pos, scale, rope_theta, rope_mode, num_splits,
                         scratch, afx::kNoAllocScratchBytes, stream);
}

