// Host-resident attention backward: q, k, v, out, dout and lse stay in (pinned) host memory and travel
// to the device in token chunks; every needed (query chunk, key chunk) pair runs the backward's
// chunk-pair kernel into fp32 device accumulators, and dq, dk, dv return to host memory. The pages'
// streamed backward (`stream_cqsa_backward`, "stream-cqsa 2.2.0 -> 2.2.2" diff, README list of
// explicit entry points) works subproblem by subproblem from the forward's saved lse ("stream-cqsa
// 2.2.2 -> 2.2.3" diff, stream_cqsa/oom_fallback.py, `stream_cqsa_auto` docstring).
//
// Schedule (query-outer, one stream, in order): for each query chunk, copy its q, out, dout and lse,
// form D = rowsum(dout * out) and zero its fp32 dq accumulator; for each key chunk it needs (every
// chunk, or those starting at or before the query chunk's last token when causal) copy k, v and add
// the pair into dq and into that key chunk's fp32 dk / dv accumulators; then round dq to the input
// dtype and copy it out. Once every query chunk is done, dk and dv of each key chunk follow. Device
// memory: the dk / dv accumulators of the whole sequence (2 * B*H*N*64 * 4 bytes) plus one chunk of
// each input, D, lse, the dq accumulator and an output staging buffer.
#include <math.h>
#include <string.h>

#include "cqsa_internal.h"

// Run one CUDA call only while every earlier step succeeded, keeping the first failure.
#define CQSA_STEP(expr, what)                               \
  do {                                                      \
    if (rc == CQSA_OK) rc = cuda_status((expr), (what));    \
  } while (0)

namespace cqsa {
namespace {

// A packed [B,H,n,64] device chunk into tokens [t0, t0 + n) of a [B,H,N,64] host tensor (16-bit).
cudaError_t copy_chunk_out(void* host, const void* dev, int B, int H, long long N, long long t0, int n,
                           cudaStream_t s) {
  const size_t row = static_cast<size_t>(n) * 64 * 2;
  char* dst = static_cast<char*>(host) + static_cast<size_t>(t0) * 64 * 2;
  return cudaMemcpy2DAsync(dst, static_cast<size_t>(N) * 64 * 2, dev, row, row, static_cast<size_t>(B) * H,
                           cudaMemcpyDeviceToHost, s);
}

}  // namespace
}  // namespace cqsa

using namespace cqsa;

extern "C" int cqsa_stream_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int H, long long N, int d,
                                    int causal, float scale, int dtype, long long chunk_tokens, cudaStream_t stream) {
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) {
    set_error("q, k, v, out, dout, lse, dq, dk and dv must be non-null host pointers");
    return CQSA_ERR_INVALID;
  }
  if (B < 1 || H < 1 || N < 1) {
    set_error("sizes must be positive (B=%d H=%d N=%lld)", B, H, N);
    return CQSA_ERR_INVALID;
  }
  if (d != 64) {
    set_error("the backward supports head dim 64 (got %d)", d);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (dtype != CQSA_F16 && dtype != CQSA_BF16) {
    set_error("dtype %d is not supported (fp16 or bf16)", dtype);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (chunk_tokens < 128 || chunk_tokens % 128 != 0) {
    set_error("chunk_tokens must be a positive multiple of 128 (got %lld)", chunk_tokens);
    return CQSA_ERR_INVALID;
  }
  if (!isfinite(scale) || scale < 0.0f) {
    set_error("scale must be finite and >= 0 (0 selects 1/sqrt(d))");
    return CQSA_ERR_INVALID;
  }
  const long long C = chunk_tokens < N ? chunk_tokens : N;
  if (static_cast<long long>(B) * H * C > (1LL << 31) / 64 || N > 0x7fffffffLL) {
    set_error("B*H*chunk_tokens too large for one chunk launch");
    return CQSA_ERR_UNSUPPORTED;
  }
  const int n_chunks = static_cast<int>((N + C - 1) / C);
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t chunk16 = BH * static_cast<size_t>(C) * 64 * 2;  // one 16-bit chunk
  const size_t chunk32 = BH * static_cast<size_t>(C) * 64 * 4;  // one fp32 chunk
  const size_t rows32 = BH * static_cast<size_t>(C) * 4;

  // device buffers: per-key-chunk dk / dv accumulators, then one chunk of everything else
  void* acc_kv = nullptr;
  void* stage = nullptr;
  const size_t acc_bytes = 2 * static_cast<size_t>(n_chunks) * chunk32;
  const size_t stage_bytes = 6 * chunk16 + chunk32 + 2 * rows32 + 256;
  int rc = pool_alloc(&acc_kv, acc_bytes);
  if (rc == CQSA_OK) rc = pool_alloc(&stage, stage_bytes);
  if (rc != CQSA_OK) {
    pool_free(acc_kv);
    return rc;
  }
  float* dk_acc0 = static_cast<float*>(acc_kv);
  float* dv_acc0 = dk_acc0 + static_cast<size_t>(n_chunks) * (chunk32 / 4);
  char* sp = static_cast<char*>(stage);
  void* q_c = sp;
  void* out_c = sp + chunk16;
  void* g_c = sp + 2 * chunk16;
  void* k_c = sp + 3 * chunk16;
  void* v_c = sp + 4 * chunk16;
  void* o_c = sp + 5 * chunk16;  // output staging (dtype)
  float* dq_acc = reinterpret_cast<float*>(sp + 6 * chunk16);
  float* lse_c = reinterpret_cast<float*>(sp + 6 * chunk16 + chunk32);
  float* dvec_c = reinterpret_cast<float*>(sp + 6 * chunk16 + chunk32 + rows32);

  long long bytes = 0;
  CQSA_STEP(cudaMemsetAsync(acc_kv, 0, acc_bytes, stream), "zero dk/dv accumulators");
  for (int qi = 0; qi < n_chunks && rc == CQSA_OK; ++qi) {
    const long long qs = static_cast<long long>(qi) * C;
    const int nq = static_cast<int>(N - qs < C ? N - qs : C);
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
    CQSA_STEP(copy_chunk(q_c, q, CQSA_LAYOUT_BHND, B, H, N, 64, qs, nq, h2d, stream, &bytes), "copy q");
    CQSA_STEP(copy_chunk(out_c, out, CQSA_LAYOUT_BHND, B, H, N, 64, qs, nq, h2d, stream, &bytes), "copy out");
    CQSA_STEP(copy_chunk(g_c, dout, CQSA_LAYOUT_BHND, B, H, N, 64, qs, nq, h2d, stream, &bytes), "copy dout");
    CQSA_STEP(cudaMemcpy2DAsync(lse_c, static_cast<size_t>(nq) * 4, lse + qs, static_cast<size_t>(N) * 4,
                                static_cast<size_t>(nq) * 4, BH, h2d, stream),
              "copy lse");
    if (rc == CQSA_OK) rc = launch_bwd_dvec(out_c, g_c, dvec_c, static_cast<long long>(BH) * nq, dtype, stream);
    CQSA_STEP(cudaMemsetAsync(dq_acc, 0, BH * static_cast<size_t>(nq) * 64 * 4, stream), "zero dq accumulator");
    for (int ki = 0; ki < n_chunks && rc == CQSA_OK; ++ki) {
      const long long ks = static_cast<long long>(ki) * C;
      if (causal && ks > qs + nq - 1) break;  // this and every later key chunk follow the whole query chunk
      const int nk = static_cast<int>(N - ks < C ? N - ks : C);
      CQSA_STEP(copy_chunk(k_c, k, CQSA_LAYOUT_BHND, B, H, N, 64, ks, nk, h2d, stream, &bytes), "copy k");
      CQSA_STEP(copy_chunk(v_c, v, CQSA_LAYOUT_BHND, B, H, N, 64, ks, nk, h2d, stream, &bytes), "copy v");
      if (rc != CQSA_OK) break;
      BwdArgs a;
      memset(&a, 0, sizeof(a));
      a.q = q_c;
      a.k = k_c;
      a.v = v_c;
      a.dout = g_c;
      a.lse = lse_c;
      a.dvec = dvec_c;
      a.dq_acc = dq_acc;
      a.dk_acc = dk_acc0 + static_cast<size_t>(ki) * (chunk32 / 4);
      a.dv_acc = dv_acc0 + static_cast<size_t>(ki) * (chunk32 / 4);
      a.B = B;
      a.H = H;
      a.Nq = nq;
      a.Nkv = nk;
      a.d = 64;
      a.q_off = qs;
      a.kv_off = ks;
      a.causal = causal != 0;
      a.scale = scale == 0.0f ? 0.125f : scale;  // 1/sqrt(64)
      a.dtype = dtype;
      rc = launch_attention_bwd_chunk(a, stream);
    }
    if (rc == CQSA_OK) rc = launch_bwd_cast(dq_acc, o_c, static_cast<long long>(BH) * nq * 64, dtype, stream);
    CQSA_STEP(copy_chunk_out(dq, o_c, B, H, N, qs, nq, stream), "copy dq out");
    // the staging buffer is reused by the next chunk's cast: wait for this copy
    CQSA_STEP(cudaStreamSynchronize(stream), "synchronize");
  }
  for (int ki = 0; ki < n_chunks && rc == CQSA_OK; ++ki) {
    const long long ks = static_cast<long long>(ki) * C;
    const int nk = static_cast<int>(N - ks < C ? N - ks : C);
    const long long n = static_cast<long long>(BH) * nk * 64;
    if (rc == CQSA_OK) rc = launch_bwd_cast(dk_acc0 + static_cast<size_t>(ki) * (chunk32 / 4), o_c, n, dtype, stream);
    CQSA_STEP(copy_chunk_out(dk, o_c, B, H, N, ks, nk, stream), "copy dk out");
    CQSA_STEP(cudaStreamSynchronize(stream), "synchronize");
    if (rc == CQSA_OK) rc = launch_bwd_cast(dv_acc0 + static_cast<size_t>(ki) * (chunk32 / 4), o_c, n, dtype, stream);
    CQSA_STEP(copy_chunk_out(dv, o_c, B, H, N, ks, nk, stream), "copy dv out");
    CQSA_STEP(cudaStreamSynchronize(stream), "synchronize");
  }
  // every use of the buffers is complete before they return to the pool
  cudaError_t se = cudaStreamSynchronize(stream);
  if (rc == CQSA_OK) rc = cuda_status(se, "synchronize");
  // a kernel whose bounded wait gave up leaves its gradients incomplete: report it
  if (rc == CQSA_OK) rc = check_device_error_on(stream);
  pool_free(stage);
  pool_free(acc_kv);
  return rc;
}
