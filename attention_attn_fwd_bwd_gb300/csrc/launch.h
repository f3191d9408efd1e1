// Internal interface between the C-ABI layer (api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace afx {

struct FwdParams {
  CUtensorMap tmQ, tmK, tmV;  // bf16 [B, H, N, d] maps, 128B swizzle, box (64, 128, 1, 1)
                              // (tmK: box (64, 64, 1, 1) for head dim 128)
  const float2* rope_cs;      // (cos, sin) table [N][d/2] (fused RoPE only)
  __nv_bfloat16* out;
  int64_t o_sb, o_sh, o_sn;
  float* lse;                 // [B, Hq, N] or null
  int B, Hq, Hkv, N, g;
  int pair_heads;             // head dim 64: 1: sub-tiles are heads (2p, 2p+1) at one q tile; 0: tiles (2t, 2t+1)
  int num_t;                  // q tiles (pair_heads) or q-tile pairs
  int pairs;                  // head pairs (Hq/2) or heads (Hq)
  float scale_log2;           // scale * log2(e)
  float scale;
  int pp_hp;                  // persistent head-dim-128 forward: query heads per unit (1, 2, 4)
  int pp_clusters;            // and the number of 2-CTA clusters launched
  // persistent head-dim-128 forward with fused RoPE: K is rotated once per 64-key block into
  // k_rot (fp16 [B, Hkv, N, d], contiguous; tmK maps it), k_sync[block] = 0 untouched,
  // 1 claimed, 2 rotated (zeroed before every launch)
  const __nv_bfloat16* k_raw;
  int64_t k_sb, k_sh, k_sn;
  uint16_t* k_rot;
  uint32_t* k_sync;
  float o_scale;  // e4m3 forward: O is multiplied by V's dequantisation scale
  VariantDev var;
  int* status;
};

struct DecParams {
  CUtensorMap tmK, tmV;       // caches [B, Hkv, L, d], box (64, 128, 1, 1)
  const __nv_bfloat16* q;     // [B, Hq, d]
  int64_t q_sb, q_sh;
  __nv_bfloat16* out;         // [B, Hq, d]
  int64_t o_sb, o_sh;
  float* lse;                 // [B, Hq] or null
  float* part_acc;            // [B, Hq, splits, d]
  float* part_m;              // [B, Hq, splits] (log2 units)
  float* part_l;              // [B, Hq, splits]
  int B, Hq, Hkv, g, L, q_pos;
  int chunk;                  // keys per split (multiple of 128)
  int splits;                 // partial-buffer stride
  int splits_used;            // ceil(L / chunk)
  float scale_log2;
  RopeFreqs freqs;
  int* status;
};

struct BwdParams {
  CUtensorMap tmQ, tmK, tmV, tmDO;  // bf16 [B, H, N, d], box (64, 128, 1, 1)
  CUtensorMap tmQ64, tmDO64;        // the same Q / dO with box (64, 64, 1, 1) (dK/dV items)
  const __nv_bfloat16* o;           // forward output (for D = rowsum(dO * O))
  const __nv_bfloat16* dout;
  int64_t o_s[3], do_s[3];
  const float* lse;                 // [B, Hq, N] natural log
  float* Dvec;                      // [B, Hq, N] workspace
  __nv_bfloat16 *dq, *dk, *dv;
  int64_t dq_s[3], dk_s[3], dv_s[3];
  const float2* rope_cs;
  int B, Hq, Hkv, N, d, g;
  float scale, scale_log2;
  VariantDev var;                   // mask and bias combinators (var.causal: n <= m)
  float* dbias;                     // additive bias only: dBias [B, Hq, N, N] fp32, or null
  int64_t db_s[3];                  // its (b, h, m) element strides; the key stride is 1
  int db_vec2;                      // 1: pointer and strides allow 8-byte pair stores
  uint8_t* visits_dq;               // debug record of the dQ kernel's (q tile, key tile) pairs
  uint8_t* visits_kv;               // and of the dK/dV kernel's (64-row query item, key tile)
  int* status;
};
// rope_kind: kRopeNone, kRopeFused (Q / K tiles rotated on chip) or kRopePrerotated (tmQ /
// tmK point at pre-rotated copies); dQ and dK are rotated back unless kRopeNone.
cudaError_t launch_bwd(const BwdParams& p, int rope_kind, cudaStream_t stream);

constexpr int kDecMaxSplits = 512;  // the combine kernel merges at most this many KV chunks
size_t decode_smem_size(int d);
cudaError_t launch_decode(const DecParams& p, int d, bool rope_q, cudaStream_t stream);

size_t fwd_smem_size(int d);
// rope_kind: how the score operands were produced.
constexpr int kRopeNone = 0;        // bf16 inputs used as they are
constexpr int kRopeFused = 1;       // rotated in shared memory by the kernel, rounded to fp16
constexpr int kRopePrerotated = 2;  // rotated by the pre-rotation kernel into fp16 buffers
constexpr int kFp8 = 3;             // head-dim-128 forward: e4m3 Q and K (scores on
                                    // kind::f8f6f4), V widened once per call to bf16
// One CTA per 256 query rows (two 128-row sub-tiles); head dim 64.
cudaError_t launch_fwd(const FwdParams& p, int d, int rope_kind, int grid, cudaStream_t stream);
// Head dim 128, persistent: clusters of two CTAs walk units of four 128-row query tiles of
// one KV head (two independent softmax slots per CTA). norm: 0 softmax, 1 ReLU (P = relu(s)/N).
size_t fwd_pp_smem_size(int d);
cudaError_t launch_fwd_pp(FwdParams p, int d, int rope_kind, int norm, cudaStream_t stream);
cudaError_t launch_rope_table(float2* cs, int N, int half, const RopeFreqs& f,
                              cudaStream_t stream);
// block: 0 = rotate with the table entry of each row; -1 = the forward kernels' query-tile
// recurrence (fp16 output); otherwise the in-block key recurrence of the kernels (forward keys:
// fp16 output, blocks of 64 / 128 for head dim 128 / 64; backward Q and K: bf16 output, blocks
// of 128).
// e4m3 [B, H, N, d] (element = byte strides) -> contiguous bf16, exactly (fwd_pp_fp8.cu)
cudaError_t launch_widen_e4m3(const void* v, const int64_t* strides, void* out, int B, int H, int N,
                              int d, cudaStream_t stream);
cudaError_t launch_prerotate(const void* x, const int64_t* strides, void* out, int B, int H,
                             int N, int d, const float2* cs, bool out_f16, int block,
                             cudaStream_t stream, int* status);
cudaError_t launch_wait_timeout(uint64_t limit_ns, int* status, cudaStream_t stream);
// Record a message for attnfuse_last_error() and return code.
int set_last_error(int code, const char* msg);

}  // namespace afx
