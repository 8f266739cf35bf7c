// C ABI: argument validation, status reporting and dispatch to the kernels. Nothing here computes
// attention; every step of the path runs in the kernels of attn_fwd.cu, attn_bwd.cu and merge.cu.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "cqsa_internal.h"
#include "sm103_ptx.cuh"

namespace cqsa {

int device_error_word(DevErr* out, int clear);  // attn_fwd.cu (owns the forward's device word)
int bwd_error_word(DevErr* out, int clear);     // attn_bwd.cu (the backward's)
int device_error_word_on(DevErr* out, cudaStream_t s);  // read on one stream; cleared when set
int bwd_error_word_on(DevErr* out, cudaStream_t s);

static thread_local char t_err[512];
static unsigned int g_timeout_ms = 0;
static int g_fault = 0;

int debug_fault() { return g_fault; }

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return CQSA_OK;
  set_error("%s: %s", what, cudaGetErrorString(e));
  if (e == cudaErrorMemoryAllocation) return CQSA_ERR_OOM;
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver || e == cudaErrorNoKernelImageForDevice ||
      e == cudaErrorInvalidDevice)
    return CQSA_ERR_DEVICE;
  return CQSA_ERR_CUDA;
}

unsigned long long timeout_ns() {
  unsigned int ms = g_timeout_ms;
  if (ms == 0) {
    const char* env = getenv("CQSA_TIMEOUT_MS");
    ms = env ? static_cast<unsigned int>(strtoul(env, nullptr, 10)) : 0;
    if (ms == 0) ms = 2000;
  }
  return static_cast<unsigned long long>(ms) * 1000000ull;
}

// Status and message of a device error word.
static int report_device_error(const DevErr& e) {
  if (e.code == 0) return CQSA_OK;
  if (e.code == kDevSmSlot) {
    set_error("a d = 128 attention CTA ran on an SM id beyond the %s (block %d): its running-sum fold was "
              "skipped, so the result is exact but chunked and monolithic results may differ by more than "
              "fp32 summation order", "running-sum slots", e.block);
    return CQSA_ERR_DEVICE;
  }
  if (e.code == kDevMisaligned) {
    set_error("the backward kernel's dynamic shared memory base is not 1024-byte aligned (block %d): its "
              "swizzled tiles need that alignment, and it stopped before computing anything", e.block);
    return CQSA_ERR_DEVICE;
  }
  set_error("device wait gave up (code %d, block %d, site %d)", e.code, e.block, e.where);
  return CQSA_ERR_TIMEOUT;
}

int check_device_error_on(cudaStream_t s) {
  DevErr e = {0, 0, 0, 0};
  int rc = device_error_word_on(&e, s);
  if (rc != CQSA_OK) return rc;
  if (e.code == 0) {
    rc = bwd_error_word_on(&e, s);
    if (rc != CQSA_OK) return rc;
  }
  return report_device_error(e);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Common checks of the problem description. Returns CQSA_OK or an error with a message set.
static int check_problem(int B, int H, long long Nq, long long Nkv, int d, float scale, int dtype, bool allow_empty_kv) {
  if (B < 1 || H < 1 || Nq < 1 || Nkv < (allow_empty_kv ? 0 : 1)) {
    set_error("sizes must be positive (B=%d H=%d Nq=%lld Nkv=%lld)", B, H, Nq, Nkv);
    return CQSA_ERR_INVALID;
  }
  if (d != 64 && d != 128) {
    set_error("head dim %d is not supported (64 or 128)", d);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (dtype != CQSA_F16 && dtype != CQSA_BF16) {
    set_error("dtype %d is not supported for Q/K/V (fp16 or bf16)", dtype);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (!isfinite(scale) || scale < 0.0f) {
    set_error("scale must be finite and >= 0 (0 selects 1/sqrt(d))");
    return CQSA_ERR_INVALID;
  }
  if (static_cast<long long>(B) * H * (Nq > Nkv ? Nq : Nkv) > (1LL << 40)) {
    set_error("problem too large");
    return CQSA_ERR_UNSUPPORTED;
  }
  return CQSA_OK;
}

static float resolve_scale(float scale, int d) { return scale == 0.0f ? 1.0f / sqrtf(static_cast<float>(d)) : scale; }

}  // namespace cqsa

using namespace cqsa;

extern "C" {

const char* cqsa_version(void) { return "0.1.0"; }

const char* cqsa_last_error(void) { return t_err; }

const char* cqsa_status_string(int status) {
  switch (status) {
    case CQSA_OK: return "CQSA_OK";
    case CQSA_ERR_INVALID: return "CQSA_ERR_INVALID";
    case CQSA_ERR_UNSUPPORTED: return "CQSA_ERR_UNSUPPORTED";
    case CQSA_ERR_CUDA: return "CQSA_ERR_CUDA";
    case CQSA_ERR_OOM: return "CQSA_ERR_OOM";
    case CQSA_ERR_TIMEOUT: return "CQSA_ERR_TIMEOUT";
    case CQSA_ERR_DEVICE: return "CQSA_ERR_DEVICE";
    default: return "CQSA_UNKNOWN_STATUS";
  }
}

void cqsa_set_timeout_ms(unsigned int ms) { g_timeout_ms = ms; }

int cqsa_debug_set_fault(int kind) {
  if (kind < 0 || kind > 2) {
    set_error("unknown fault kind %d", kind);
    return CQSA_ERR_INVALID;
  }
  g_fault = kind;
  return CQSA_OK;
}

int cqsa_device_error(int* code, int* block, int clear) {
  t_err[0] = 0;
  DevErr e;
  int rc = cuda_status(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  if (rc != CQSA_OK) return rc;
  rc = device_error_word(&e, clear);
  if (rc != CQSA_OK) return rc;
  if (e.code == 0) {
    rc = bwd_error_word(&e, clear);
    if (rc != CQSA_OK) return rc;
  }
  if (code) *code = e.code;
  if (block) *block = e.block;
  return report_device_error(e);
}

int cqsa_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H, int N, int d,
                  int causal, float scale, int dtype, cudaStream_t stream) {
  t_err[0] = 0;
  int rc = check_problem(B, H, N, N, d, scale, dtype, false);
  if (rc != CQSA_OK) return rc;
  if (!q || !k || !v || !out) {
    set_error("q, k, v and out must be non-null device pointers");
    return CQSA_ERR_INVALID;
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))) {
    set_error("q, k, v, out must be 16-byte aligned (lse 4-byte)");
    return CQSA_ERR_INVALID;
  }
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.B = B;
  a.H = H;
  a.Nq = N;
  a.Nkv = N;
  a.q_off = 0;
  a.kv_off = 0;
  a.d = d;
  a.causal = causal != 0;
  a.scale = resolve_scale(scale, d);
  a.dtype = dtype;
  a.in_layout = CQSA_LAYOUT_BHND;
  a.mode = kModeOut;
  a.out = out;
  a.lse = lse;
  a.out_layout = CQSA_LAYOUT_BHND;
  return launch_attention(a, stream);
}

int cqsa_attn_fwd_chunk(const void* q_blk, const void* k_blk, const void* v_blk, long long q_off, long long kv_off,
                        int B, int H, int Nq, int Nkv, int d, int causal, float scale, int dtype, float* O_part,
                        float* LSE_part, int accumulate, cudaStream_t stream) {
  t_err[0] = 0;
  int rc = check_problem(B, H, Nq, Nkv, d, scale, dtype, true);
  if (rc != CQSA_OK) return rc;
  if (!q_blk || !O_part || !LSE_part || (Nkv > 0 && (!k_blk || !v_blk))) {
    set_error("q_blk, O_part, LSE_part (and k_blk, v_blk when Nkv > 0) must be non-null device pointers");
    return CQSA_ERR_INVALID;
  }
  if (!aligned16(q_blk) || !aligned16(O_part) || (Nkv > 0 && (!aligned16(k_blk) || !aligned16(v_blk))) ||
      (reinterpret_cast<uintptr_t>(LSE_part) & 3u)) {
    set_error("q_blk, k_blk, v_blk, O_part must be 16-byte aligned (LSE_part 4-byte)");
    return CQSA_ERR_INVALID;
  }
  if (q_off < 0 || kv_off < 0) {
    set_error("q_off and kv_off must be >= 0");
    return CQSA_ERR_INVALID;
  }
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q_blk;
  a.k = k_blk;
  a.v = v_blk;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nkv = Nkv;
  a.q_off = q_off;
  a.kv_off = kv_off;
  a.d = d;
  a.causal = causal != 0;
  a.scale = resolve_scale(scale, d);
  a.dtype = dtype;
  a.in_layout = CQSA_LAYOUT_BHND;
  a.mode = accumulate ? kModeAccum : kModePart;
  a.o_part = O_part;
  a.lse_part = LSE_part;
  a.out_layout = CQSA_LAYOUT_BHND;
  return launch_attention(a, stream);
}

int cqsa_merge_partials(const float* const* O_parts, const float* const* LSE_parts, int n, void* out, float* lse,
                        int B, int H, int Nq, int d, int out_dtype, cudaStream_t stream) {
  t_err[0] = 0;
  if (n < 1 || n > 1024) {
    set_error("n must be in [1, 1024] (got %d)", n);
    return CQSA_ERR_INVALID;
  }
  if (!O_parts || !LSE_parts || !out) {
    set_error("O_parts, LSE_parts and out must be non-null");
    return CQSA_ERR_INVALID;
  }
  if (B < 1 || H < 1 || Nq < 1) {
    set_error("sizes must be positive");
    return CQSA_ERR_INVALID;
  }
  if (d != 64 && d != 128) {
    set_error("head dim %d is not supported (64 or 128)", d);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (out_dtype != CQSA_F16 && out_dtype != CQSA_BF16 && out_dtype != CQSA_F32) {
    set_error("out_dtype %d is not supported", out_dtype);
    return CQSA_ERR_UNSUPPORTED;
  }
  for (int i = 0; i < n; ++i) {
    if (!O_parts[i] || !LSE_parts[i] || !aligned16(O_parts[i]) || (reinterpret_cast<uintptr_t>(LSE_parts[i]) & 3u)) {
      set_error("part %d: null or misaligned pointer (O 16-byte, LSE 4-byte)", i);
      return CQSA_ERR_INVALID;
    }
  }
  if (!aligned16(out) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))) {
    set_error("out must be 16-byte aligned (lse 4-byte)");
    return CQSA_ERR_INVALID;
  }
  return launch_merge(O_parts, LSE_parts, n, out, lse, static_cast<long long>(B) * H * Nq, d, out_dtype, stream);
}

size_t cqsa_attn_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  return attention_bwd_workspace(B, H, N, d);
}

int cqsa_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                  int causal, float scale, int dtype, cudaStream_t stream) {
  t_err[0] = 0;
  int rc = check_problem(B, H, N, N, d, scale, dtype, false);
  if (rc != CQSA_OK) return rc;
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv || !workspace) {
    set_error("q, k, v, out, dout, lse, dq, dk, dv and workspace must be non-null device pointers");
    return CQSA_ERR_INVALID;
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u)) {
    set_error("q, k, v, out, dout, dq, dk, dv and workspace must be 16-byte aligned (lse 4-byte)");
    return CQSA_ERR_INVALID;
  }
  const size_t need = attention_bwd_workspace(B, H, N, d);
  if (workspace_bytes < need) {
    set_error("workspace of %zu bytes is smaller than the %zu bytes cqsa_attn_bwd_workspace_size reports",
              workspace_bytes, need);
    return CQSA_ERR_INVALID;
  }
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.workspace = workspace;
  a.B = B;
  a.H = H;
  a.Nq = N;
  a.Nkv = N;
  a.d = d;
  a.causal = causal != 0;
  a.scale = resolve_scale(scale, d);
  a.dtype = dtype;
  return launch_attention_bwd(a, stream);
}

int cqsa_attn_bwd_dvec(const void* out_blk, const void* dout_blk, float* dvec_blk, int B, int H, int Nq, int d,
                       int dtype, cudaStream_t stream) {
  t_err[0] = 0;
  int rc = check_problem(B, H, Nq, Nq, d, 0.0f, dtype, false);
  if (rc != CQSA_OK) return rc;
  if (!out_blk || !dout_blk || !dvec_blk || !aligned16(out_blk) || !aligned16(dout_blk) ||
      (reinterpret_cast<uintptr_t>(dvec_blk) & 3u)) {
    set_error("out_blk and dout_blk must be non-null 16-byte aligned device pointers, dvec_blk 4-byte aligned");
    return CQSA_ERR_INVALID;
  }
  return launch_bwd_dvec(out_blk, dout_blk, dvec_blk, static_cast<long long>(B) * H * Nq, d, dtype, stream);
}

int cqsa_attn_bwd_chunk(const void* q_blk, const void* k_blk, const void* v_blk, const void* dout_blk,
                        const float* lse_blk, const float* dvec_blk, long long q_off, long long kv_off, int B, int H,
                        int Nq, int Nkv, int d, int causal, float scale, int dtype, float* dq_acc, float* dk_acc,
                        float* dv_acc, cudaStream_t stream) {
  t_err[0] = 0;
  int rc = check_problem(B, H, Nq, Nkv, d, scale, dtype, false);
  if (rc != CQSA_OK) return rc;
  if (q_off < 0 || kv_off < 0) {
    set_error("q_off and kv_off must be >= 0");
    return CQSA_ERR_INVALID;
  }
  if (!q_blk || !k_blk || !v_blk || !dout_blk || !lse_blk || !dvec_blk || !dq_acc || !dk_acc || !dv_acc) {
    set_error("every block and accumulator pointer must be a non-null device pointer");
    return CQSA_ERR_INVALID;
  }
  if (!aligned16(q_blk) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(dout_blk) || !aligned16(dq_acc) ||
      !aligned16(dk_acc) || !aligned16(dv_acc) || (reinterpret_cast<uintptr_t>(lse_blk) & 3u) ||
      (reinterpret_cast<uintptr_t>(dvec_blk) & 3u)) {
    set_error("blocks and accumulators must be 16-byte aligned (lse_blk, dvec_blk 4-byte)");
    return CQSA_ERR_INVALID;
  }
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q_blk;
  a.k = k_blk;
  a.v = v_blk;
  a.dout = dout_blk;
  a.lse = lse_blk;
  a.dvec = dvec_blk;
  a.dq_acc = dq_acc;
  a.dk_acc = dk_acc;
  a.dv_acc = dv_acc;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nkv = Nkv;
  a.d = d;
  a.q_off = q_off;
  a.kv_off = kv_off;
  a.causal = causal != 0;
  a.scale = resolve_scale(scale, d);
  a.dtype = dtype;
  return launch_attention_bwd_chunk(a, stream);
}

int cqsa_attn_bwd_cast(const float* acc, void* out, long long n, int dtype, cudaStream_t stream) {
  t_err[0] = 0;
  if (n < 0 || (n & 3)) {
    set_error("n must be a non-negative multiple of 4 (got %lld)", n);
    return CQSA_ERR_INVALID;
  }
  if (dtype != CQSA_F16 && dtype != CQSA_BF16) {
    set_error("dtype %d is not supported (fp16 or bf16)", dtype);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (n > 0 && (!acc || !out || !aligned16(acc) || (reinterpret_cast<uintptr_t>(out) & 7u))) {
    set_error("acc must be a 16-byte aligned device pointer and out 8-byte aligned");
    return CQSA_ERR_INVALID;
  }
  return launch_bwd_cast(acc, out, n, dtype, stream);
}

}  // extern "C"
