// Chunked exact attention over device-resident Q/K/V whose fp32 accumulator lives in a fixed,
// file-scope device array instead of memory the library allocates. This is for callers that cannot
// let a library call cudaMalloc: code that runs under a framework's own memory pool or a strict
// device-memory budget, where an allocation inside the call would fail, break the budget, or
// synchronise the device at a point the caller does not control. The call allocates nothing; the
// caller passes inputs and outputs, and the scratch is the array below.
//
// The array (CQSA_STATIC_SCRATCH_BYTES) is held by every device on which this module is loaded, at
// the latest from the first call of the entry point, until the process exits. All calls share it and
// it keeps the last call's contents; nothing in it needs clearing because the first key chunk of
// every query chunk overwrites the accumulator. Calls whose work overlaps on the GPU (on different
// streams, or from different host threads without ordering) race on it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <mutex>
#include <string.h>

#include "cqsa_internal.h"

namespace cqsa {
namespace {

constexpr size_t kScratchBytes = CQSA_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

// Device address of g_static_scratch for each device (in host code the symbol's name is a host-side
// stand-in, not a device address). Filled once per device, with that device current.
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

int scratch_for_current_device(void** out) {
  int dev = 0;
  int rc = cuda_status(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc != CQSA_OK) return rc;
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device index %d out of range", dev);
    return CQSA_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    rc = cuda_status(cudaGetSymbolAddress(&p, g_static_scratch), "cudaGetSymbolAddress(static scratch)");
    if (rc != CQSA_OK) return rc;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CQSA_OK;
}

// out[g0 + g, t0 + i, :] and lse[g0 + g, t0 + i] of one query chunk of n rows for heads g0 .. g0 + gn - 1 of
// a [B*H, N, d] output (dtype) from the fp32 accumulator acc[g, i, :] and lacc[g, i].
__global__ void static_finalize_kernel(const float* __restrict__ acc, const float* __restrict__ lacc, void* out,
                                       float* lse, int gn, int n, int N, long long g0, int t0, int d, int dtype) {
  const int d4 = d / 4;
  const long long total4 = static_cast<long long>(gn) * n * d4;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total4;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long gi = e / d4;  // g * n + i
    const int c4 = static_cast<int>(e % d4);
    const int g = static_cast<int>(gi / n);
    const int i = static_cast<int>(gi % n);
    const float4 v = reinterpret_cast<const float4*>(acc)[e];
    const long long orow = (g0 + g) * N + t0 + i;
    uint2 w;
    if (dtype == CQSA_BF16) {
      __nv_bfloat162 x = __floats2bfloat162_rn(v.x, v.y), y = __floats2bfloat162_rn(v.z, v.w);
      w.x = *reinterpret_cast<uint32_t*>(&x);
      w.y = *reinterpret_cast<uint32_t*>(&y);
    } else {
      __half2 x = __floats2half2_rn(v.x, v.y), y = __floats2half2_rn(v.z, v.w);
      w.x = *reinterpret_cast<uint32_t*>(&x);
      w.y = *reinterpret_cast<uint32_t*>(&y);
    }
    reinterpret_cast<uint2*>(out)[orow * d4 + c4] = w;
    if (lse && c4 == 0) lse[orow] = lacc[gi];
  }
}

}  // namespace
}  // namespace cqsa

using namespace cqsa;

extern "C" int cqsa_attn_fwd_chunked_static(const void* q, const void* k, const void* v, void* out, float* lse,
                                            int B, int H, int N, int d, int causal, float scale, int dtype,
                                            int chunk_tokens, cudaStream_t stream) {
  if (!q || !k || !v || !out) {
    set_error("q, k, v and out must be non-null device pointers");
    return CQSA_ERR_INVALID;
  }
  if (B < 1 || H < 1 || N < 1) {
    set_error("sizes must be positive (B=%d H=%d N=%d)", B, H, N);
    return CQSA_ERR_INVALID;
  }
  if (d != 64 && d != 128) {
    set_error("head dim %d is not supported (64 or 128)", d);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (dtype != CQSA_F16 && dtype != CQSA_BF16) {
    set_error("dtype %d is not supported (fp16 or bf16)", dtype);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (!isfinite(scale) || scale < 0.0f) {
    set_error("scale must be finite and >= 0 (0 selects 1/sqrt(d))");
    return CQSA_ERR_INVALID;
  }
  if (chunk_tokens < 128 || chunk_tokens % 128 != 0) {
    set_error("chunk_tokens must be a positive multiple of 128 (got %d)", chunk_tokens);
    return CQSA_ERR_INVALID;
  }
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
  if ((mis & 15u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))) {
    set_error("q, k, v, out must be 16-byte aligned (lse 4-byte)");
    return CQSA_ERR_INVALID;
  }
  const int C = chunk_tokens < N ? chunk_tokens : ((N + 127) / 128) * 128;
  // Heads are processed in groups of G consecutive (b, h) of the [B*H, N, d] tensors, as many as the
  // scratch holds accumulators for (C x d fp32 + C fp32 each): one launch per chunk pair covers the
  // whole group. A token range of the group is a strided view (N tokens per head), which the chunk
  // kernel's tensor maps address directly.
  const size_t per_head = static_cast<size_t>(C) * (d + 1) * sizeof(float);
  if (per_head > kScratchBytes) {
    set_error("a %d-token chunk needs %zu bytes of fp32 accumulator; the static scratch holds %zu "
              "(lower chunk_tokens)", C, per_head, kScratchBytes);
    return CQSA_ERR_UNSUPPORTED;
  }
  const long long BH = static_cast<long long>(B) * H;
  const long long G = static_cast<long long>(kScratchBytes / per_head) < BH
                          ? static_cast<long long>(kScratchBytes / per_head) : BH;
  void* base = nullptr;
  int rc = scratch_for_current_device(&base);
  if (rc != CQSA_OK) return rc;
  float* acc = static_cast<float*>(base);
  const float sc = scale == 0.0f ? 1.0f / sqrtf(static_cast<float>(d)) : scale;
  const size_t es = 2;
  const int nch = (N + C - 1) / C;
  for (long long g0 = 0; g0 < BH; g0 += G) {
    const int gn = static_cast<int>(BH - g0 < G ? BH - g0 : G);
    const size_t group = static_cast<size_t>(g0) * N * d * es;
    for (int i = 0; i < nch; ++i) {
      const int qt0 = i * C;
      const int qn = N - qt0 < C ? N - qt0 : C;
      float* lacc = acc + static_cast<size_t>(gn) * qn * d;  // [gn, qn] after the [gn, qn, d] accumulator
      const int last_j = causal ? i : nch - 1;
      for (int j = 0; j <= last_j; ++j) {
        const int kt0 = j * C;
        const int kn = N - kt0 < C ? N - kt0 : C;
        AttnArgs a;
        memset(&a, 0, sizeof(a));
        a.q = static_cast<const char*>(q) + group + static_cast<size_t>(qt0) * d * es;
        a.k = static_cast<const char*>(k) + group + static_cast<size_t>(kt0) * d * es;
        a.v = static_cast<const char*>(v) + group + static_cast<size_t>(kt0) * d * es;
        a.B = 1;
        a.H = gn;
        a.Nq = qn;
        a.Nkv = kn;
        a.q_tokens_alloc = N;
        a.kv_tokens_alloc = N;
        a.q_off = qt0;
        a.kv_off = kt0;
        a.d = d;
        a.causal = causal != 0;
        a.scale = sc;
        a.dtype = dtype;
        a.in_layout = CQSA_LAYOUT_BHND;
        a.mode = (j == 0) ? kModePart : kModeAccum;  // the first key chunk overwrites the accumulator
        a.o_part = acc;
        a.lse_part = lacc;
        a.out_layout = CQSA_LAYOUT_BHND;
        rc = launch_attention(a, stream);
        if (rc != CQSA_OK) return rc;
      }
      const long long total4 = static_cast<long long>(gn) * qn * d / 4;
      const long long want = (total4 + 255) / 256;
      const int blocks = static_cast<int>(want < 4096 ? want : 4096);
      static_finalize_kernel<<<blocks, 256, 0, stream>>>(acc, lacc, out, lse, gn, qn, N, g0, qt0, d, dtype);
      rc = cuda_status(cudaGetLastError(), "static finalize launch");
      if (rc != CQSA_OK) return rc;
    }
  }
  return CQSA_OK;
}
