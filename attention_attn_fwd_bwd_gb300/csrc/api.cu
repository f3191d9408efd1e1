// C-ABI layer: argument validation, workspace carving, TMA descriptor encoding and launches.
// Declarations and the meaning of every argument are in include/attnfuse.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/attnfuse.h"
#include "launch.h"

namespace afx {

// Device status word: kernels write a non-zero code here when a bounded wait gives up.
__device__ int g_status_word;

namespace {

thread_local std::string t_err;

attnfuse_status fail(attnfuse_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

attnfuse_status ok() {
  t_err.clear();
  return ATTNFUSE_OK;
}

attnfuse_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTNFUSE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------------------------
// Per-device state: status word address and the TMA descriptor encoder.
// ---------------------------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

attnfuse_status device_state(int** status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTNFUSE_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    g_status_ptr[dev] = static_cast<int*>(ptr);
  }
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return fail(ATTNFUSE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *status = g_status_ptr[dev];
  return ATTNFUSE_OK;
}

// bf16 [B, H, N, d] view with element strides; box (64, box_rows, 1, 1), 128-byte swizzle.
// box_x = 32 (64-byte rows) takes the 64-byte swizzle.
attnfuse_status encode_bhnd(CUtensorMap* m, const void* ptr, const int64_t st[4], int B, int H,
                            int N, int d, const char* name, int box_rows = 128, int box_x = 64) {
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
  cuuint32_t box[4] = {(cuuint32_t)box_x, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_x == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "%s: tensor map encode failed (CUresult %d)", name,
                (int)r);
  return ATTNFUSE_OK;
}

// e4m3 [B, H, N, d] view with element (= byte) strides; box (128, box_rows, 1, 1): one
// 128-byte swizzle row holds a whole head-dim-128 row.
attnfuse_status encode_bhnd8(CUtensorMap* m, const void* ptr, const int64_t st[4], int B, int H,
                             int N, int d, const char* name, int box_rows) {
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st[2], (cuuint64_t)st[1], (cuuint64_t)st[0]};
  cuuint32_t box[4] = {128, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "%s: tensor map encode failed (CUresult %d)", name,
                (int)r);
  return ATTNFUSE_OK;
}

// ---------------------------------------------------------------------------------------------
// Validation
// ---------------------------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attnfuse_status check_tensor(const void* p, const int64_t st[4], const char* name) {
  if (!p) return fail(ATTNFUSE_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(ATTNFUSE_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  if (!st) return fail(ATTNFUSE_ERR_INVALID_ARG, "%s strides are NULL", name);
  if (st[3] != 1) return fail(ATTNFUSE_ERR_INVALID_ARG, "%s: innermost stride must be 1", name);
  for (int i = 0; i < 3; ++i)
    if (st[i] <= 0 || (st[i] % 8) != 0)
      return fail(ATTNFUSE_ERR_INVALID_ARG,
                  "%s: stride[%d] = %lld must be a positive multiple of 8 elements", name, i,
                  (long long)st[i]);
  return ATTNFUSE_OK;
}

attnfuse_status check_shape(int B, int Hq, int Hkv, int N, int d) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "sizes must be positive (B=%d Hq=%d Hkv=%d N=%d)", B,
                Hq, Hkv, N);
  if (Hq % Hkv) return fail(ATTNFUSE_ERR_UNSUPPORTED, "Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
  if (d != 64 && d != 128) return fail(ATTNFUSE_ERR_UNSUPPORTED, "head dim %d (need 64 or 128)", d);
  return ATTNFUSE_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The table always covers at least 128 positions: the fused key rotation reads the entry of
// position 128 / (d / 16) as its per-row step.
int rope_table_rows(int N) { return N < 128 ? 128 : N; }
// Forward with fused RoPE: the rotated keys (fp16) and one flag per 64-key block (head dim 128;
// head dim 64 uses one per 128-key tile, fewer).
size_t fused_k_bytes(int B, int Hkv, int N, int d) {
  return align_up((size_t)B * Hkv * N * d * 2, 256);
}
// Head dim 64 runs on the persistent CTA-pair forward (fwd_pp.cuh) when its work units share K
// tiles across heads (an even GQA group) or are long, else on the one-CTA forward (fwd.cu).
// A pair-kernel unit is four 128-row query tiles of one KV head; with one query head per KV
// head they are four consecutive positions, whose kv ranges differ, and few units balance
// poorly over the clusters. Measured on GB300 (ms, no RoPE / fused RoPE, causal):
//   B=4 Hq=32 Hkv=8 N=4096   pairs 0.512 / 0.544   one-CTA 0.557 / 0.617
//   B=8 Hq=32 Hkv=8 N=2048   pairs 0.297 / 0.328   one-CTA 0.328 / 0.374
//   B=1 H=16 N=16384         pairs 0.935 / 0.974   one-CTA 0.984 / 1.072
//   B=2 H=16 N=4096          pairs 0.164 / 0.191   one-CTA 0.150 / 0.186
//   B=16 H=16 N=1024         pairs 0.158 / 0.203   one-CTA 0.117 / 0.151
bool d64_on_pairs(int g, int N) { return g % 2 == 0 || N >= 8192; }
// Head dim 64 (one CTA per 256 query rows, not persistent): rotating each K tile once and
// sharing it through L2 pays when many query tiles re-read it; with few readers the copy's
// latency on the first reader's path costs more than rotating K stages in place per CTA.
// Measured on GB300 (B*N = 16384, H=16, causal): in place 0.166 / 0.241 ms at N = 1024 /
// 2048, shared 0.187 / 0.239; at N = 4096 shared wins for causal, ALiBi and BigBird and
// loses for a 1024-key window (0.161 vs 0.151 ms).
bool share_rotated_k_d64(int N, const VariantDev& v) {
  if (N < 2048) return false;
  if (v.mask == 2 && v.window < 2048) return false;
  return true;
}
size_t fused_sync_bytes(int B, int Hkv, int N) {
  return align_up((size_t)B * Hkv * ((N + 63) / 64) * sizeof(uint32_t), 256);
}
size_t rope_table_bytes(int N, int d) {
  return align_up((size_t)rope_table_rows(N) * (d / 2) * sizeof(float2), 256);
}

RopeFreqs make_freqs(int d, float theta) {
  RopeFreqs f;
  memset(&f, 0, sizeof(f));
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < d / 2; ++i) {
    const double turns = std::pow((double)theta, -2.0 * i / d) / two_pi;
    f.hi[i] = (float)turns;
    f.lo[i] = (float)(turns - (double)f.hi[i]);
  }
  return f;
}

attnfuse_status to_dev_variant(const attnfuse_variant* v, int N, int Hq, VariantDev* out) {
  memset(out, 0, sizeof(*out));
  if (!v) {
    out->mask = ATTNFUSE_MASK_CAUSAL;
    out->causal = 1;
    return ATTNFUSE_OK;
  }
  if (v->mask < 0 || v->mask > 3) return fail(ATTNFUSE_ERR_INVALID_ARG, "mask kind %d", v->mask);
  out->mask = v->mask;
  out->causal = (v->mask == ATTNFUSE_MASK_CAUSAL || v->causal) ? 1 : 0;
  if (v->mask == ATTNFUSE_MASK_WINDOW) {
    if (v->window < 1) return fail(ATTNFUSE_ERR_INVALID_ARG, "window %d < 1", v->window);
    out->window = v->window;
  }
  if (v->mask == ATTNFUSE_MASK_BLOCK_SPARSE) {
    if (v->bs_block != 64 && v->bs_block != 128)
      return fail(ATTNFUSE_ERR_UNSUPPORTED, "block-sparse block %d (need 64 or 128)", v->bs_block);
    if (N > kBsMaxN)
      return fail(ATTNFUSE_ERR_UNSUPPORTED, "block-sparse needs N <= %d", kBsMaxN);
    if (!v->bs_row_ptr || !v->bs_col_idx)
      return fail(ATTNFUSE_ERR_INVALID_ARG, "block-sparse CSR pointers are NULL");
    out->bs_block = v->bs_block;
    out->bs_row_ptr = v->bs_row_ptr;
    out->bs_col_idx = v->bs_col_idx;
  }
  if (v->bias < 0 || v->bias > 2) return fail(ATTNFUSE_ERR_INVALID_ARG, "bias kind %d", v->bias);
  out->bias = v->bias;
  if (v->bias == ATTNFUSE_BIAS_ALIBI) {
    if (!v->alibi_slopes) return fail(ATTNFUSE_ERR_INVALID_ARG, "ALiBi slopes are NULL");
    out->slopes = v->alibi_slopes;
  }
  if (v->bias == ATTNFUSE_BIAS_ADDITIVE) {
    if (!v->add_bias) return fail(ATTNFUSE_ERR_INVALID_ARG, "additive bias is NULL");
    out->add_bias = v->add_bias;
    out->add_bias_bf16 = v->add_bias_is_bf16 ? 1 : 0;
    for (int i = 0; i < 4; ++i) {
      if (v->add_bias_strides[i] < 0)
        return fail(ATTNFUSE_ERR_INVALID_ARG, "negative additive-bias stride");
      out->ab_s[i] = v->add_bias_strides[i];
    }
  }
  out->visits = v->tile_visits;
  if (v->normalizer != ATTNFUSE_NORM_SOFTMAX && v->normalizer != ATTNFUSE_NORM_RELU)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "normalizer %d", v->normalizer);
  out->norm = v->normalizer;
  (void)Hq;
  return ATTNFUSE_OK;
}

}  // namespace

cudaError_t launch_wait_timeout(uint64_t limit_ns, int* status, cudaStream_t stream);

int set_last_error(int code, const char* msg) {
  return fail(code, "%s", msg);
}

}  // namespace afx

using namespace afx;

extern "C" {

const char* attnfuse_last_error(void) { return t_err.c_str(); }

int attnfuse_version(void) { return 100; }

attnfuse_status attnfuse_device_status(cudaStream_t stream, int clear, int* code) {
  if (!code) return fail(ATTNFUSE_ERR_INVALID_ARG, "code is NULL");
  int* st = nullptr;
  attnfuse_status rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, st, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  if (clear && v) {
    const int zero = 0;
    e = cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear status word");
  }
  *code = (v & kDevTimeout) ? ATTNFUSE_ERR_TIMEOUT : (v & kDevF16Range) ? ATTNFUSE_ERR_FP16_RANGE : ATTNFUSE_OK;
  return ok();
}

// ATTNFUSE_ROPE_AUTO: the faster of on-chip rotation and pre-rotation, by the crossover
// N* measured on GB300 (the paper's Rotation Calculus, §5.3; B*N = 16384 tokens, causal).
// The pre-rotation pass streams at ~5 TB/s, so it costs ~70 us per 16k-token, 32-head call.
// Head dim 64: fusion wins below N* ~ 1.85k (forward; t_prerotate / t_fused over two sweeps:
// 1.19-1.23 at N = 256, 1.04-1.08 at 1024, 0.98-1.00 at 2048) and ~ 260 (backward, which
// re-reads each K tile once per query tile). Head dim 128: the persistent forward rotates Q in
// shared memory and takes K' from a one-pass rotation of K; it wins below N* ~ 15k (1.08 at
// N = 256, 1.04 at 2048, 1.02 at 4096, 1.01 at 8192, 1.00 at 16384). The backward pre-rotates at every N.
constexpr int kAutoFusedBelowN64Fwd = 1850;
constexpr int kAutoFusedBelowN64Bwd = 258;
constexpr int kAutoFusedBelowN128Fwd = 14900;

static attnfuse_rope_mode resolve_rope(attnfuse_rope_mode m, int N, int d, bool backward) {
  if (m != ATTNFUSE_ROPE_AUTO) return m;
  if (d == 64 && N < (backward ? kAutoFusedBelowN64Bwd : kAutoFusedBelowN64Fwd))
    return ATTNFUSE_ROPE_FUSED;
  if (d == 128 && !backward && N < kAutoFusedBelowN128Fwd) return ATTNFUSE_ROPE_FUSED;
  return ATTNFUSE_ROPE_PREROTATE;
}

attnfuse_status attnfuse_rope_auto_mode(int N, int d, int backward, attnfuse_rope_mode* mode) {
  if (!mode) return fail(ATTNFUSE_ERR_INVALID_ARG, "mode is NULL");
  if (N < 1) return fail(ATTNFUSE_ERR_INVALID_ARG, "N=%d", N);
  if (d != 64 && d != 128) return fail(ATTNFUSE_ERR_UNSUPPORTED, "head dim %d (need 64 or 128)", d);
  *mode = resolve_rope(ATTNFUSE_ROPE_AUTO, N, d, backward != 0);
  return ok();
}

attnfuse_status attnfuse_fwd_workspace_size(int B, int Hq, int Hkv, int N, int d,
                                            attnfuse_rope_mode rope_mode, size_t* bytes) {
  if (!bytes) return fail(ATTNFUSE_ERR_INVALID_ARG, "bytes is NULL");
  rope_mode = resolve_rope(static_cast<attnfuse_rope_mode>(rope_mode & ~ATTNFUSE_ROPE_REUSE_TABLE),
                           N, d, false);
  attnfuse_status rc = check_shape(B, Hq, Hkv, N, d);
  if (rc) return rc;
  size_t n = 0;
  if (rope_mode == ATTNFUSE_ROPE_FUSED || rope_mode == ATTNFUSE_ROPE_PREROTATE)
    n += rope_table_bytes(N, d);
  if (rope_mode == ATTNFUSE_ROPE_PREROTATE) {
    n += align_up((size_t)B * Hq * N * d * 2, 256);
    n += align_up((size_t)B * Hkv * N * d * 2, 256);
  }
  if (rope_mode == ATTNFUSE_ROPE_FUSED) n += fused_k_bytes(B, Hkv, N, d) + fused_sync_bytes(B, Hkv, N);
  if (rope_mode < 0 || rope_mode > 2) return fail(ATTNFUSE_ERR_INVALID_ARG, "rope mode %d", rope_mode);
  *bytes = n;
  return ok();
}

attnfuse_status attnfuse_rope_prerotate(const void* x, const int64_t x_strides[4], void* out,
                                        int B, int H, int N, int d, float rope_theta,
                                        void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
  attnfuse_status rc = check_shape(B, H, H, N, d);
  if (rc) return rc;
  if ((rc = check_tensor(x, x_strides, "x"))) return rc;
  if (!out || !aligned16(out)) return fail(ATTNFUSE_ERR_INVALID_ARG, "out NULL or misaligned");
  if (!(rope_theta > 0.f) || !std::isfinite(rope_theta))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "rope_theta must be positive");
  const size_t need = rope_table_bytes(N, d);
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(ATTNFUSE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes", need);
  int* st = nullptr;
  if ((rc = device_state(&st))) return rc;
  float2* cs = static_cast<float2*>(workspace);
  cudaError_t e = launch_rope_table(cs, rope_table_rows(N), d / 2, make_freqs(d, rope_theta), stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
  e = launch_prerotate(x, x_strides, out, B, H, N, d, cs, false, 0, stream, nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "prerotate launch");
  return ok();
}

attnfuse_status attnfuse_fwd(const void* q, const int64_t q_strides[4], const void* k,
                             const int64_t k_strides[4], const void* v,
                             const int64_t v_strides[4], void* out, const int64_t o_strides[4],
                             float* lse, int B, int Hq, int Hkv, int N, int d, float scale,
                             float rope_theta, attnfuse_rope_mode rope_mode,
                             const attnfuse_variant* variant, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  const bool reuse_table = (rope_mode & ATTNFUSE_ROPE_REUSE_TABLE) != 0;
  rope_mode = resolve_rope(static_cast<attnfuse_rope_mode>(rope_mode & ~ATTNFUSE_ROPE_REUSE_TABLE),
                           N, d, false);
  attnfuse_status rc = check_shape(B, Hq, Hkv, N, d);
  if (rc) return rc;
  if ((rc = check_tensor(q, q_strides, "q"))) return rc;
  if ((rc = check_tensor(k, k_strides, "k"))) return rc;
  if ((rc = check_tensor(v, v_strides, "v"))) return rc;
  if ((rc = check_tensor(out, o_strides, "out"))) return rc;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "lse is not 4-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "scale must be positive and finite");
  if (rope_mode < 0 || rope_mode > 2) return fail(ATTNFUSE_ERR_INVALID_ARG, "rope mode %d", rope_mode);
  if (rope_mode != ATTNFUSE_ROPE_NONE && (!(rope_theta > 0.f) || !std::isfinite(rope_theta)))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "rope_theta must be positive");
  FwdParams p;
  memset(&p, 0, sizeof(p));
  if ((rc = to_dev_variant(variant, N, Hq, &p.var))) return rc;
  if (p.var.norm == ATTNFUSE_NORM_RELU) {
    if (lse) return fail(ATTNFUSE_ERR_INVALID_ARG, "relu_attention has no LSE: pass lse = NULL");
  }
  size_t need = 0;
  if ((rc = attnfuse_fwd_workspace_size(B, Hq, Hkv, N, d, rope_mode, &need))) return rc;
  if (need && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return fail(ATTNFUSE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes (got %zu)", need,
                workspace_bytes);
  int* st = nullptr;
  if ((rc = device_state(&st))) return rc;

  const void* qa = q;
  const void* ka = k;
  const int64_t* qs = q_strides;
  const int64_t* ks = k_strides;
  int64_t qs_c[4], ks_c[4];
  float2* cs = nullptr;
  if (rope_mode != ATTNFUSE_ROPE_NONE) {
    cs = static_cast<float2*>(workspace);
    if (!reuse_table) {
      cudaError_t e =
          launch_rope_table(cs, rope_table_rows(N), d / 2, make_freqs(d, rope_theta), stream);
      if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
    }
  }
  if (rope_mode == ATTNFUSE_ROPE_PREROTATE) {
    uint8_t* base = static_cast<uint8_t*>(workspace) + rope_table_bytes(N, d);
    void* qr = base;
    void* kr = base + align_up((size_t)B * Hq * N * d * 2, 256);
    cudaError_t e = launch_prerotate(q, q_strides, qr, B, Hq, N, d, cs, true, -1, stream, st);
    if (e == cudaSuccess) e = launch_prerotate(k, k_strides, kr, B, Hkv, N, d, cs, true, 1, stream, st);
    if (e != cudaSuccess) return cuda_fail(e, "prerotate launch");
    qs_c[0] = (int64_t)Hq * N * d; qs_c[1] = (int64_t)N * d; qs_c[2] = d; qs_c[3] = 1;
    ks_c[0] = (int64_t)Hkv * N * d; ks_c[1] = (int64_t)N * d; ks_c[2] = d; ks_c[3] = 1;
    qa = qr; ka = kr; qs = qs_c; ks = ks_c;
  }
  // the persistent CTA-pair forward (the only one with the ReLU normaliser)
  const bool pairs = d == 128 || p.var.norm == ATTNFUSE_NORM_RELU || d64_on_pairs(Hq / Hkv, N);
  if (rope_mode == ATTNFUSE_ROPE_FUSED && pairs) {
    // Q is rotated in the forward, per work unit in shared memory; K (1/g of Q with GQA) by
    // one pass into the workspace copy K' before it, with the forward's chains
    uint8_t* kr = static_cast<uint8_t*>(workspace) + rope_table_bytes(N, d);
    cudaError_t e = launch_prerotate(k, k_strides, kr, B, Hkv, N, d, cs, true, 1, stream, st);
    if (e != cudaSuccess) return cuda_fail(e, "K rotation launch");
    ks_c[0] = (int64_t)Hkv * N * d; ks_c[1] = (int64_t)N * d; ks_c[2] = d; ks_c[3] = 1;
    ka = kr; ks = ks_c;
  } else if (rope_mode == ATTNFUSE_ROPE_FUSED && share_rotated_k_d64(N, p.var)) {
    // K is rotated once per call inside the forward, per 64-key block (head dim 128) or
    // 128-key tile (head dim 64), by whichever CTA needs it first, into a workspace copy that
    // every CTA then loads with TMA
    uint8_t* base = static_cast<uint8_t*>(workspace) + rope_table_bytes(N, d);
    p.k_raw = static_cast<const __nv_bfloat16*>(k);
    p.k_sb = k_strides[0]; p.k_sh = k_strides[1]; p.k_sn = k_strides[2];
    p.k_rot = reinterpret_cast<uint16_t*>(base);
    p.k_sync = reinterpret_cast<uint32_t*>(base + fused_k_bytes(B, Hkv, N, d));
    cudaError_t e = cudaMemsetAsync(p.k_sync, 0, fused_sync_bytes(B, Hkv, N), stream);
    if (e != cudaSuccess) return cuda_fail(e, "k_sync reset");
    ks_c[0] = (int64_t)Hkv * N * d; ks_c[1] = (int64_t)N * d; ks_c[2] = d; ks_c[3] = 1;
    ka = p.k_rot; ks = ks_c;
  }
  if ((rc = encode_bhnd(&p.tmQ, qa, qs, B, Hq, N, d, "q"))) return rc;
  // the CTA-pair forward loads 64-key halves of K and d/2-dim halves of V
  if ((rc = encode_bhnd(&p.tmK, ka, ks, B, Hkv, N, d, "k", pairs ? 64 : 128))) return rc;
  if ((rc = encode_bhnd(&p.tmV, v, v_strides, B, Hkv, N, d, "v", 128, pairs && d == 64 ? 32 : 64))) return rc;
  p.rope_cs = cs;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.o_sb = o_strides[0]; p.o_sh = o_strides[1]; p.o_sn = o_strides[2];
  p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.g = Hq / Hkv;
  const int TQ = (N + 127) / 128;
  p.pair_heads = (p.g % 2 == 0) ? 1 : 0;
  p.num_t = p.pair_heads ? TQ : (TQ + 1) / 2;
  p.pairs = p.pair_heads ? Hq / 2 : Hq;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.scale = scale;
  p.status = st;
  const int64_t grid = (int64_t)p.num_t * B * p.pairs;
  if (grid > 0x7fffffff) return fail(ATTNFUSE_ERR_UNSUPPORTED, "problem too large (grid %lld)", (long long)grid);
  const int rk = rope_mode == ATTNFUSE_ROPE_FUSED ? kRopeFused
                 : rope_mode == ATTNFUSE_ROPE_PREROTATE ? kRopePrerotated : kRopeNone;
  cudaError_t e = pairs ? launch_fwd_pp(p, d, rk, p.var.norm, stream)
                        : launch_fwd(p, d, rk, (int)grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return ok();
}

// ---------------------------------------------------------------------------------------------
// e4m3 forward
// ---------------------------------------------------------------------------------------------
namespace {
size_t fp8_v_bytes(int B, int Hkv, int N, int d) { return align_up((size_t)B * Hkv * N * d * 2, 256); }
attnfuse_status check_tensor8(const void* p, const int64_t st[4], const char* name) {
  if (!p) return fail(ATTNFUSE_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(ATTNFUSE_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  if (!st) return fail(ATTNFUSE_ERR_INVALID_ARG, "%s strides are NULL", name);
  if (st[3] != 1) return fail(ATTNFUSE_ERR_INVALID_ARG, "%s: innermost stride must be 1", name);
  for (int i = 0; i < 3; ++i)
    if (st[i] <= 0 || (st[i] % 16) != 0)
      return fail(ATTNFUSE_ERR_INVALID_ARG,
                  "%s: stride[%d] = %lld must be a positive multiple of 16 elements", name, i,
                  (long long)st[i]);
  return ATTNFUSE_OK;
}
bool positive_finite(float x) { return x > 0.f && std::isfinite(x); }
}  // namespace

attnfuse_status attnfuse_fwd_fp8_workspace_size(int B, int Hq, int Hkv, int N, int d, size_t* bytes) {
  if (!bytes) return fail(ATTNFUSE_ERR_INVALID_ARG, "bytes is NULL");
  attnfuse_status rc = check_shape(B, Hq, Hkv, N, d);
  if (rc) return rc;
  if (d != 128) return fail(ATTNFUSE_ERR_UNSUPPORTED, "e4m3 forward needs head dim 128 (got %d)", d);
  *bytes = fp8_v_bytes(B, Hkv, N, d);
  return ok();
}

attnfuse_status attnfuse_fwd_fp8(const void* q, const int64_t q_strides[4], const void* k,
                                 const int64_t k_strides[4], const void* v,
                                 const int64_t v_strides[4], void* out, const int64_t o_strides[4],
                                 float* lse, int B, int Hq, int Hkv, int N, int d, float scale,
                                 float q_scale, float k_scale, float v_scale,
                                 const attnfuse_variant* variant, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  attnfuse_status rc = check_shape(B, Hq, Hkv, N, d);
  if (rc) return rc;
  if (d != 128) return fail(ATTNFUSE_ERR_UNSUPPORTED, "e4m3 forward needs head dim 128 (got %d)", d);
  if ((rc = check_tensor8(q, q_strides, "q"))) return rc;
  if ((rc = check_tensor8(k, k_strides, "k"))) return rc;
  if ((rc = check_tensor8(v, v_strides, "v"))) return rc;
  if ((rc = check_tensor(out, o_strides, "out"))) return rc;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "lse is not 4-byte aligned");
  if (!positive_finite(scale)) return fail(ATTNFUSE_ERR_INVALID_ARG, "scale must be positive and finite");
  if (!positive_finite(q_scale) || !positive_finite(k_scale) || !positive_finite(v_scale))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "q_scale, k_scale and v_scale must be positive and finite");
  FwdParams p;
  memset(&p, 0, sizeof(p));
  if ((rc = to_dev_variant(variant, N, Hq, &p.var))) return rc;
  if (p.var.norm == ATTNFUSE_NORM_RELU && lse)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "relu_attention has no LSE: pass lse = NULL");
  size_t need = 0;
  if ((rc = attnfuse_fwd_fp8_workspace_size(B, Hq, Hkv, N, d, &need))) return rc;
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(ATTNFUSE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes (got %zu)", need,
                workspace_bytes);
  int* st = nullptr;
  if ((rc = device_state(&st))) return rc;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  // V widened to bf16 (exact) by one pass; the P V MMAs read it like a bf16 V
  void* v_wide = base;
  cudaError_t e = launch_widen_e4m3(v, v_strides, v_wide, B, Hkv, N, d, stream);
  if (e != cudaSuccess) return cuda_fail(e, "V widening launch");
  int64_t vs_c[4] = {(int64_t)Hkv * N * d, (int64_t)N * d, d, 1};
  if ((rc = encode_bhnd8(&p.tmQ, q, q_strides, B, Hq, N, d, "q", 128))) return rc;
  if ((rc = encode_bhnd8(&p.tmK, k, k_strides, B, Hkv, N, d, "k", 64))) return rc;
  if ((rc = encode_bhnd(&p.tmV, v_wide, vs_c, B, Hkv, N, d, "v (widened)"))) return rc;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.o_sb = o_strides[0]; p.o_sh = o_strides[1]; p.o_sn = o_strides[2];
  p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.g = Hq / Hkv;
  // the dequantisation scales of q and k fold into the score scale, v's into O
  const float s_qk = scale * q_scale * k_scale;
  if (!positive_finite(s_qk)) return fail(ATTNFUSE_ERR_INVALID_ARG, "scale * q_scale * k_scale is not finite");
  p.scale_log2 = s_qk * 1.4426950408889634f;
  p.scale = s_qk;
  p.o_scale = v_scale;
  p.status = st;
  e = launch_fwd_pp(p, 128, kFp8, p.var.norm, stream);
  if (e != cudaSuccess) return cuda_fail(e, "e4m3 forward launch");
  return ok();
}

// ---------------------------------------------------------------------------------------------
// Forward on host buffers: copy-in, forward and copy-out pipelined over batch chunks
// ---------------------------------------------------------------------------------------------
namespace {
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;  // copy streams (the forward runs on the caller's)
  cudaEvent_t start = nullptr, in_done[2] = {}, fwd_done[2] = {}, out_done[2] = {};
};
std::mutex g_pipe_mu;
HostPipe g_pipe[64];

cudaError_t host_pipe(int dev, HostPipe** out) {
  HostPipe& hp = g_pipe[dev];
  if (!hp.in) {
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int i = 0; i < 2; ++i) {
      if ((e = cudaEventCreateWithFlags(&hp.in_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&hp.fwd_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&hp.out_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
  }
  *out = &hp;
  return cudaSuccess;
}

struct HostChunk {  // device bytes of one chunk of cb batch elements
  size_t q, kv, o, l, ws;
};
HostChunk host_chunk(int cb, int Hq, int Hkv, int N, int d, size_t fwd_ws) {
  HostChunk c;
  c.q = align_up((size_t)cb * Hq * N * d * 2, 256);
  c.kv = align_up((size_t)cb * Hkv * N * d * 2, 256);
  c.o = c.q;
  c.l = align_up((size_t)cb * Hq * N * 4, 256);
  c.ws = align_up(fwd_ws, 256);
  return c;
}
}  // namespace

attnfuse_status attnfuse_fwd_host_workspace_size(int B, int Hq, int Hkv, int N, int d,
                                                 attnfuse_rope_mode rope_mode, int chunk_b,
                                                 size_t* bytes) {
  if (!bytes) return fail(ATTNFUSE_ERR_INVALID_ARG, "bytes is NULL");
  attnfuse_status rc = check_shape(B, Hq, Hkv, N, d);
  if (rc) return rc;
  if (chunk_b < 1 || chunk_b > B) return fail(ATTNFUSE_ERR_INVALID_ARG, "chunk_b %d (B = %d)", chunk_b, B);
  size_t fw = 0;
  const attnfuse_rope_mode m = static_cast<attnfuse_rope_mode>(rope_mode & ~ATTNFUSE_ROPE_REUSE_TABLE);
  if ((rc = attnfuse_fwd_workspace_size(chunk_b, Hq, Hkv, N, d, m, &fw))) return rc;
  const HostChunk c = host_chunk(chunk_b, Hq, Hkv, N, d, fw);
  *bytes = 2 * (c.q + 2 * c.kv + c.o + c.l) + c.ws;
  return ok();
}

attnfuse_status attnfuse_fwd_host(const void* q, const void* k, const void* v, void* out, float* lse,
                                  int B, int Hq, int Hkv, int N, int d, float scale,
                                  float rope_theta, attnfuse_rope_mode rope_mode,
                                  const attnfuse_variant* variant, int chunk_b, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !out) return fail(ATTNFUSE_ERR_INVALID_ARG, "q, k, v and out must be host pointers");
  if (rope_mode & ATTNFUSE_ROPE_REUSE_TABLE)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "the host forward builds its own table: no REUSE_TABLE");
  size_t need = 0;
  attnfuse_status rc = attnfuse_fwd_host_workspace_size(B, Hq, Hkv, N, d, rope_mode, chunk_b, &need);
  if (rc) return rc;
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(ATTNFUSE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes (got %zu)", need,
                workspace_bytes);
  rope_mode = resolve_rope(rope_mode, N, d, false);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(ATTNFUSE_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* hp = nullptr;
  if ((e = host_pipe(dev, &hp)) != cudaSuccess) return cuda_fail(e, "host pipeline setup");
  size_t fw = 0;
  if ((rc = attnfuse_fwd_workspace_size(chunk_b, Hq, Hkv, N, d, rope_mode, &fw))) return rc;
  const HostChunk c = host_chunk(chunk_b, Hq, Hkv, N, d, fw);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* fwd_ws = base + 2 * (c.q + 2 * c.kv + c.o + c.l);
  // the copies start after what the caller queued on `stream`
  if ((e = cudaEventRecord(hp->start, stream)) != cudaSuccess) return cuda_fail(e, "event");
  cudaStreamWaitEvent(hp->in, hp->start, 0);
  cudaStreamWaitEvent(hp->out, hp->start, 0);
  const size_t q_el = (size_t)Hq * N * d, kv_el = (size_t)Hkv * N * d, l_el = (size_t)Hq * N;
  const int TQ = (N + 127) / 128;
  const int g = Hq / Hkv;
  // With one batch element per chunk, each element is also split into hs groups of KV heads
  // (contiguous in every array) until there are at least 8 chunks: the first chunk's copy-in
  // and the last chunk's forward and copy-out, which nothing overlaps, shrink with the chunk.
  int hs = 1;
  if (chunk_b == 1)
    while (B * hs < 8 && Hkv % (2 * hs) == 0) hs *= 2;
  const int nh = Hkv / hs, qh = nh * g;  // KV and query heads of a chunk
  bool table_built = false;
  for (int ci = 0; ci * chunk_b < B * hs; ++ci) {
    const int b0 = (ci / hs) * chunk_b, hg = ci % hs;
    const int cb = std::min(chunk_b, B - b0);
    const int bi = ci & 1;
    uint8_t* set = base + bi * (c.q + 2 * c.kv + c.o + c.l);
    void* dq = set;
    void* dk = set + c.q;
    void* dv = set + c.q + c.kv;
    void* dout = set + c.q + 2 * c.kv;
    float* dlse = lse ? reinterpret_cast<float*>(set + c.q + 2 * c.kv + c.o) : nullptr;
    // copy-in once the forward two chunks back has read this buffer set
    if (ci >= 2) cudaStreamWaitEvent(hp->in, hp->fwd_done[bi], 0);
    // elements before the chunk and in it (a chunk of several batch elements has hs = 1)
    const size_t q0 = (size_t)b0 * q_el + (size_t)hg * qh * N * d;
    const size_t k0 = (size_t)b0 * kv_el + (size_t)hg * nh * N * d;
    const size_t l0 = (size_t)b0 * l_el + (size_t)hg * qh * N;
    const size_t qb = (size_t)cb * qh * N * d * 2, kvb = (size_t)cb * nh * N * d * 2;
    e = cudaMemcpyAsync(dq, static_cast<const uint8_t*>(q) + q0 * 2, qb, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dk, static_cast<const uint8_t*>(k) + k0 * 2, kvb, cudaMemcpyHostToDevice, hp->in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dv, static_cast<const uint8_t*>(v) + k0 * 2, kvb, cudaMemcpyHostToDevice, hp->in);
    if (e != cudaSuccess) return cuda_fail(e, "copy-in");
    cudaEventRecord(hp->in_done[bi], hp->in);
    // the forward, once its inputs are in and this buffer set's output has been copied out
    cudaStreamWaitEvent(stream, hp->in_done[bi], 0);
    if (ci >= 2) cudaStreamWaitEvent(stream, hp->out_done[bi], 0);
    attnfuse_variant vc;
    if (variant) {
      vc = *variant;
      if (vc.bias == ATTNFUSE_BIAS_ADDITIVE && vc.add_bias)
        vc.add_bias = static_cast<const uint8_t*>(vc.add_bias) +
                      ((size_t)b0 * vc.add_bias_strides[0] + (size_t)hg * qh * vc.add_bias_strides[1]) *
                          (vc.add_bias_is_bf16 ? 2 : 4);
      if (vc.bias == ATTNFUSE_BIAS_ALIBI && vc.alibi_slopes) vc.alibi_slopes += hg * qh;
      if (vc.tile_visits) vc.tile_visits += ((size_t)b0 * Hq + (size_t)hg * qh) * TQ * TQ;
    }
    const int64_t qs[4] = {(int64_t)qh * N * d, (int64_t)N * d, d, 1};
    const int64_t ks[4] = {(int64_t)nh * N * d, (int64_t)N * d, d, 1};
    const int mode = rope_mode | ((rope_mode != ATTNFUSE_ROPE_NONE && table_built) ? ATTNFUSE_ROPE_REUSE_TABLE : 0);
    rc = attnfuse_fwd(dq, qs, dk, ks, dv, ks, dout, qs, dlse, cb, qh, nh, N, d, scale, rope_theta,
                      static_cast<attnfuse_rope_mode>(mode), variant ? &vc : nullptr, fwd_ws, c.ws,
                      stream);
    if (rc) return rc;
    table_built = true;
    cudaEventRecord(hp->fwd_done[bi], stream);
    // copy-out
    cudaStreamWaitEvent(hp->out, hp->fwd_done[bi], 0);
    e = cudaMemcpyAsync(static_cast<uint8_t*>(out) + q0 * 2, dout, qb, cudaMemcpyDeviceToHost, hp->out);
    if (e == cudaSuccess && lse)
      e = cudaMemcpyAsync(lse + l0, dlse, (size_t)cb * qh * N * 4, cudaMemcpyDeviceToHost, hp->out);
    if (e != cudaSuccess) return cuda_fail(e, "copy-out");
    cudaEventRecord(hp->out_done[bi], hp->out);
  }
  // completion on the caller's stream: every copy-out has landed
  const int nchunks = (B + chunk_b - 1) / chunk_b * hs;
  for (int i = 0; i < std::min(nchunks, 2); ++i) cudaStreamWaitEvent(stream, hp->out_done[(nchunks - 1 - i) & 1], 0);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "host forward");
  return ok();
}

attnfuse_status attnfuse_rope_table(void* table, size_t table_bytes, int N, int d,
                                    float rope_theta, cudaStream_t stream) {
  if (N <= 0 || (d != 64 && d != 128))
    return fail(ATTNFUSE_ERR_UNSUPPORTED, "rope table for N=%d d=%d", N, d);
  if (!(rope_theta > 0.f) || !std::isfinite(rope_theta))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "rope_theta must be positive");
  if (!table || !aligned16(table) || table_bytes < rope_table_bytes(N, d))
    return fail(ATTNFUSE_ERR_WORKSPACE_TOO_SMALL, "table needs %zu bytes", rope_table_bytes(N, d));
  int* st = nullptr;
  attnfuse_status rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = launch_rope_table(static_cast<float2*>(table), rope_table_rows(N), d / 2,
                                    make_freqs(d, rope_theta), stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
  return ok();
}

// ---------------------------------------------------------------------------------------------
// Backward (paper §4.4)
// ---------------------------------------------------------------------------------------------
attnfuse_status attnfuse_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d,
                                            attnfuse_rope_mode rope_mode, size_t* bytes) {
  if (!bytes) return fail(ATTNFUSE_ERR_INVALID_ARG, "bytes is NULL");
  rope_mode = resolve_rope(static_cast<attnfuse_rope_mode>(rope_mode & ~ATTNFUSE_ROPE_REUSE_TABLE),
                           N, d, true);
  attnfuse_status rc = check_shape(B, Hq, Hkv, N, d);
  if (rc) return rc;
  if (rope_mode < 0 || rope_mode > 2) return fail(ATTNFUSE_ERR_INVALID_ARG, "rope mode %d", rope_mode);
  size_t n = 0;
  if (rope_mode != ATTNFUSE_ROPE_NONE) n += rope_table_bytes(N, d);
  n += align_up((size_t)B * Hq * N * 4, 256);  // D = rowsum(dO * O)
  if (rope_mode == ATTNFUSE_ROPE_PREROTATE) {     // Q' and K' (bf16, contiguous)
    n += align_up((size_t)B * Hq * N * d * 2, 256);
    n += align_up((size_t)B * Hkv * N * d * 2, 256);
  }
  *bytes = n;
  return ok();
}

static attnfuse_status check3(const void* p, const int64_t st[4], const char* name) {
  return check_tensor(p, st, name);
}

attnfuse_status attnfuse_bwd(const void* q, const int64_t q_strides[4], const void* k,
                             const int64_t k_strides[4], const void* v,
                             const int64_t v_strides[4], const void* out,
                             const int64_t o_strides[4], const float* lse, const void* dout,
                             const int64_t do_strides[4], void* dq, const int64_t dq_strides[4],
                             void* dk, const int64_t dk_strides[4], void* dv,
                             const int64_t dv_strides[4], int B, int Hq, int Hkv, int N, int d,
                             float scale, float rope_theta, attnfuse_rope_mode rope_mode,
                             const attnfuse_variant* variant, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  const bool reuse_table = (rope_mode & ATTNFUSE_ROPE_REUSE_TABLE) != 0;
  rope_mode = resolve_rope(static_cast<attnfuse_rope_mode>(rope_mode & ~ATTNFUSE_ROPE_REUSE_TABLE),
                           N, d, true);
  attnfuse_status rc = check_shape(B, Hq, Hkv, N, d);
  if (rc) return rc;
  if ((rc = check3(q, q_strides, "q")) || (rc = check3(k, k_strides, "k")) ||
      (rc = check3(v, v_strides, "v")) || (rc = check3(out, o_strides, "out")) ||
      (rc = check3(dout, do_strides, "dout")) || (rc = check3(dq, dq_strides, "dq")) ||
      (rc = check3(dk, dk_strides, "dk")) || (rc = check3(dv, dv_strides, "dv")))
    return rc;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "lse NULL or misaligned");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "scale must be positive and finite");
  if (rope_mode < 0 || rope_mode > 2) return fail(ATTNFUSE_ERR_INVALID_ARG, "rope mode %d", rope_mode);
  if (rope_mode != ATTNFUSE_ROPE_NONE && (!(rope_theta > 0.f) || !std::isfinite(rope_theta)))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "rope_theta must be positive");
  VariantDev var;
  if ((rc = to_dev_variant(variant, N, Hq, &var))) return rc;
  if (var.norm != ATTNFUSE_NORM_SOFTMAX)
    return fail(ATTNFUSE_ERR_UNSUPPORTED, "the backward supports the softmax normaliser only");
  var.visits = nullptr;  // the tile-visit record belongs to the forward
  float* dbias = variant ? variant->dbias : nullptr;
  if (dbias) {
    if (var.bias != ATTNFUSE_BIAS_ADDITIVE)
      return fail(ATTNFUSE_ERR_INVALID_ARG, "dbias needs ATTNFUSE_BIAS_ADDITIVE");
    const int64_t* ds = variant->dbias_strides;
    if ((reinterpret_cast<uintptr_t>(dbias) & 3u) || ds[3] != 1 || ds[0] < 0 || ds[1] < 0 ||
        ds[2] < 0)
      return fail(ATTNFUSE_ERR_INVALID_ARG,
                  "dbias must be 4-byte aligned with key stride 1 and non-negative strides");
  }
  size_t need = 0;
  if ((rc = attnfuse_bwd_workspace_size(B, Hq, Hkv, N, d, rope_mode, &need))) return rc;
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(ATTNFUSE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes (got %zu)", need,
                workspace_bytes);
  int* st = nullptr;
  if ((rc = device_state(&st))) return rc;
  BwdParams p;
  memset(&p, 0, sizeof(p));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (rope_mode != ATTNFUSE_ROPE_NONE) {
    p.rope_cs = reinterpret_cast<const float2*>(ws);
    if (!reuse_table) {
      cudaError_t e = launch_rope_table(reinterpret_cast<float2*>(ws), rope_table_rows(N), d / 2,
                                        make_freqs(d, rope_theta), stream);
      if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
    }
    ws += rope_table_bytes(N, d);
  }
  p.Dvec = reinterpret_cast<float*>(ws);
  ws += align_up((size_t)B * Hq * N * 4, 256);
  const void* qa = q;
  const void* ka = k;
  const int64_t* qs = q_strides;
  const int64_t* ks = k_strides;
  int64_t qs_c[4], ks_c[4];
  if (rope_mode == ATTNFUSE_ROPE_PREROTATE) {
    // Q' and K' once, in the backward kernels' in-tile recurrence (bit-identical to FUSED)
    void* qr = ws;
    void* kr = ws + align_up((size_t)B * Hq * N * d * 2, 256);
    cudaError_t e = launch_prerotate(q, q_strides, qr, B, Hq, N, d, p.rope_cs, false, 128, stream, nullptr);
    if (e == cudaSuccess) e = launch_prerotate(k, k_strides, kr, B, Hkv, N, d, p.rope_cs, false, 128, stream, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "prerotate launch");
    qs_c[0] = (int64_t)Hq * N * d; qs_c[1] = (int64_t)N * d; qs_c[2] = d; qs_c[3] = 1;
    ks_c[0] = (int64_t)Hkv * N * d; ks_c[1] = (int64_t)N * d; ks_c[2] = d; ks_c[3] = 1;
    qa = qr; ka = kr; qs = qs_c; ks = ks_c;
  }
  if ((rc = encode_bhnd(&p.tmQ, qa, qs, B, Hq, N, d, "q"))) return rc;
  if ((rc = encode_bhnd(&p.tmK, ka, ks, B, Hkv, N, d, "k"))) return rc;
  if ((rc = encode_bhnd(&p.tmV, v, v_strides, B, Hkv, N, d, "v"))) return rc;
  if ((rc = encode_bhnd(&p.tmDO, dout, do_strides, B, Hq, N, d, "dout"))) return rc;
  if ((rc = encode_bhnd(&p.tmQ64, qa, qs, B, Hq, N, d, "q", 64))) return rc;
  if ((rc = encode_bhnd(&p.tmDO64, dout, do_strides, B, Hq, N, d, "dout", 64))) return rc;
  p.o = static_cast<const __nv_bfloat16*>(out);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  for (int i = 0; i < 3; ++i) {
    p.o_s[i] = o_strides[i];
    p.do_s[i] = do_strides[i];
    p.dq_s[i] = dq_strides[i];
    p.dk_s[i] = dk_strides[i];
    p.dv_s[i] = dv_strides[i];
  }
  p.lse = lse;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d; p.g = Hq / Hkv;
  p.var = var;
  p.dbias = dbias;
  if (variant) {
    p.visits_dq = variant->bwd_dq_visits;
    p.visits_kv = variant->bwd_dkdv_visits;
  }
  if (dbias) {
    for (int i = 0; i < 3; ++i) p.db_s[i] = variant->dbias_strides[i];
    p.db_vec2 = ((reinterpret_cast<uintptr_t>(dbias) & 7u) == 0 && p.db_s[0] % 2 == 0 &&
                 p.db_s[1] % 2 == 0 && p.db_s[2] % 2 == 0) ? 1 : 0;
  }
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = st;
  const int rk = rope_mode == ATTNFUSE_ROPE_FUSED ? kRopeFused
                 : rope_mode == ATTNFUSE_ROPE_PREROTATE ? kRopePrerotated : kRopeNone;
  cudaError_t e = launch_bwd(p, rk, stream);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return ok();
}

// ---------------------------------------------------------------------------------------------
// Decode (paper §4.2)
// ---------------------------------------------------------------------------------------------
static attnfuse_status decode_plan(int B, int Hkv, int L, int num_splits, int* splits, int* chunk) {
  if (num_splits < 0) return fail(ATTNFUSE_ERR_INVALID_ARG, "num_splits %d < 0", num_splits);
  const int tiles = (L + 127) / 128;
  int s = num_splits;
  if (s == 0) {
    // One resident CTA per SM: pick the split count with the smallest makespan
    // (waves x tiles per chunk, plus about one tile of fixed cost per wave).
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long pairs = (long long)B * Hkv;
    long long best = -1;
    for (int c = 1; c <= tiles; ++c) {
      const long long waves = (pairs * c + sms - 1) / sms;
      const long long cost = waves * ((tiles + c - 1) / c + 1);
      if (best < 0 || cost < best) {
        best = cost;
        s = c;
      }
    }
  }
  s = std::max(1, std::min(std::min(s, tiles), kDecMaxSplits));
  const int ch = ((tiles + s - 1) / s) * 128;
  *chunk = ch;
  *splits = s;
  return ATTNFUSE_OK;
}

attnfuse_status attnfuse_decode_auto_splits(int B, int Hkv, int L, int* num_splits) {
  if (!num_splits || B <= 0 || Hkv <= 0 || L <= 0)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "bad arguments");
  int chunk = 0;
  attnfuse_status rc = decode_plan(B, Hkv, L, 0, num_splits, &chunk);
  if (rc) return rc;
  return ok();
}

attnfuse_status attnfuse_decode_workspace_size(int B, int Hq, int Hkv, int L, int d,
                                               int num_splits, size_t* bytes) {
  if (!bytes) return fail(ATTNFUSE_ERR_INVALID_ARG, "bytes is NULL");
  attnfuse_status rc = check_shape(B, Hq, Hkv, L, d);
  if (rc) return rc;
  int splits = 0, chunk = 0;
  if ((rc = decode_plan(B, Hkv, L, num_splits, &splits, &chunk))) return rc;
  const size_t rows = (size_t)B * Hq * splits;
  *bytes = align_up(rows * d * 4, 256) + 2 * align_up(rows * 4, 256);
  return ok();
}

attnfuse_status attnfuse_decode(const void* q, const int64_t q_strides[3], const void* k_cache,
                                const int64_t k_strides[4], const void* v_cache,
                                const int64_t v_strides[4], void* out,
                                const int64_t o_strides[3], float* lse, int B, int Hq, int Hkv,
                                int L, int d, int q_pos, float scale, float rope_theta,
                                attnfuse_rope_mode rope_mode, int num_splits, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  attnfuse_status rc = check_shape(B, Hq, Hkv, L, d);
  if (rc) return rc;
  const int g = Hq / Hkv;
  if (g > 32) return fail(ATTNFUSE_ERR_UNSUPPORTED, "decode needs Hq / Hkv <= 32 (got %d)", g);
  if (!q || !aligned16(q) || !q_strides || q_strides[2] != 1 || q_strides[0] % 8 ||
      q_strides[1] % 8 || q_strides[0] <= 0 || q_strides[1] <= 0)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "q: NULL, misaligned or bad strides");
  if (!out || !o_strides || o_strides[2] != 1 || o_strides[0] <= 0 || o_strides[1] <= 0)
    return fail(ATTNFUSE_ERR_INVALID_ARG, "out: NULL or bad strides");
  if ((rc = check_tensor(k_cache, k_strides, "k_cache"))) return rc;
  if ((rc = check_tensor(v_cache, v_strides, "v_cache"))) return rc;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "lse is not 4-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "scale must be positive and finite");
  if (rope_mode == ATTNFUSE_ROPE_AUTO) rope_mode = ATTNFUSE_ROPE_FUSED;  // only q is rotated
  if (rope_mode != ATTNFUSE_ROPE_NONE && rope_mode != ATTNFUSE_ROPE_FUSED)
    return fail(ATTNFUSE_ERR_UNSUPPORTED, "decode rotates q only: rope_mode NONE or FUSED");
  if (rope_mode == ATTNFUSE_ROPE_FUSED && (!(rope_theta > 0.f) || !std::isfinite(rope_theta)))
    return fail(ATTNFUSE_ERR_INVALID_ARG, "rope_theta must be positive");
  if (q_pos < 0) return fail(ATTNFUSE_ERR_INVALID_ARG, "q_pos %d < 0", q_pos);
  size_t need = 0;
  if ((rc = attnfuse_decode_workspace_size(B, Hq, Hkv, L, d, num_splits, &need))) return rc;
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(ATTNFUSE_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes (got %zu)", need,
                workspace_bytes);
  int* st = nullptr;
  if ((rc = device_state(&st))) return rc;
  DecParams p;
  memset(&p, 0, sizeof(p));
  int splits = 0, chunk = 0;
  if ((rc = decode_plan(B, Hkv, L, num_splits, &splits, &chunk))) return rc;
  if ((rc = encode_bhnd(&p.tmK, k_cache, k_strides, B, Hkv, L, d, "k_cache"))) return rc;
  if ((rc = encode_bhnd(&p.tmV, v_cache, v_strides, B, Hkv, L, d, "v_cache"))) return rc;
  const size_t rows = (size_t)B * Hq * splits;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_acc = reinterpret_cast<float*>(ws);
  p.part_m = reinterpret_cast<float*>(ws + align_up(rows * d * 4, 256));
  p.part_l = reinterpret_cast<float*>(ws + align_up(rows * d * 4, 256) + align_up(rows * 4, 256));
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.q_sb = q_strides[0];
  p.q_sh = q_strides[1];
  p.out = static_cast<__nv_bfloat16*>(out);
  p.o_sb = o_strides[0];
  p.o_sh = o_strides[1];
  p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.g = g; p.L = L; p.q_pos = q_pos;
  p.chunk = chunk;
  p.splits = splits;
  p.splits_used = (L + chunk - 1) / chunk;
  p.scale_log2 = scale * 1.4426950408889634f;
  if (rope_mode == ATTNFUSE_ROPE_FUSED) p.freqs = make_freqs(d, rope_theta);
  p.status = st;
  cudaError_t e = launch_decode(p, d, rope_mode == ATTNFUSE_ROPE_FUSED, stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return ok();
}

attnfuse_status attnfuse_debug_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  int* st = nullptr;
  attnfuse_status rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = launch_wait_timeout(limit_ns, st, stream);
  if (e != cudaSuccess) return cuda_fail(e, "wait-timeout launch");
  return ok();
}

}  // extern "C"
