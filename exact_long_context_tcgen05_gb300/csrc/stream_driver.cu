// Host-resident exact attention: Q/K/V stay in (pinned) host memory and are streamed to the device
// in token chunks while the chunk kernel merges every (Q chunk, KV chunk) pair into an fp32 device
// accumulator. The pages' engine keeps inputs on the host ("stream_from_host") and overlaps the
// per-subproblem host transfers with compute ("stream-cqsa 2.2.0 -> 2.2.2" diff, README profile
// sweep); host copies are token-major ("stream-cqsa 2.2.2 -> 2.2.3" diff, api.py `_pinned_copy`).
//
// Schedule (Q-outer): for each Q chunk i, Q_i is copied once into one of two Q buffers (the copy of
// Q_{i+1} overlaps Q_i's kernels); the KV chunks j it needs (j <= i when causal) are double-buffered
// on the same copy stream: copy(j) waits for the kernel that last used its slot, the kernel for
// (i, j) waits for copy(j). Contiguous chunks (token-major, B = 1) travel as plain copies. The first pair of a Q chunk writes the accumulator
// (partial mode), later pairs merge into it in place (accumulate mode). A finalize kernel converts
// the accumulator to the output dtype and layout; host outputs leave on a second copy stream.
// The KV order alternates direction between consecutive Q chunks (serpentine), so the chunk that
// ended one Q chunk starts the next and is not copied again.
#include <chrono>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <string.h>
#include <vector>

#include "cqsa_internal.h"

namespace cqsa {
namespace {

// out[b, h, t0 + i, :] (layout BHND, N tokens) or out[b, t0 + i, h, :] (BNHD) from acc[b, h, i, :].
// With `staged`, the destination is a packed chunk buffer (N = n, t0 = 0).
__global__ void finalize_kernel(const float* __restrict__ acc, const float* __restrict__ lse_acc, void* out,
                                float* lse_out, int B, int H, int n, long long N, long long t0, int d, int layout,
                                int dtype) {
  const long long total4 = static_cast<long long>(B) * H * n * d / 4;
  const int d4 = d / 4;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total4;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = e / d4;  // (b*H + h)*n + i
    const int c4 = static_cast<int>(e % d4);
    const int i = static_cast<int>(row % n);
    const long long bh = row / n;
    const int h = static_cast<int>(bh % H);
    const int b = static_cast<int>(bh / H);
    const float4 v = reinterpret_cast<const float4*>(acc)[e];
    const long long orow = layout == CQSA_LAYOUT_BHND ? (static_cast<long long>(b) * H + h) * N + t0 + i
                                                      : (static_cast<long long>(b) * N + t0 + i) * H + h;
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
    if (lse_out && c4 == 0) lse_out[bh * N + t0 + i] = lse_acc[row];
  }
}

// Buffers, events and streams come from the library's pool and go back to it once the streams that
// use them have drained.
struct Resources {
  std::vector<void*> dev;
  std::vector<std::pair<cudaEvent_t, bool>> events;
  cudaStream_t copy = nullptr, d2h = nullptr;
  cudaStream_t compute = nullptr;  // caller's stream: drained before buffers are returned
  bool compute_set = false;
  ~Resources() {
    if (compute_set) cudaStreamSynchronize(compute);
    if (copy) cudaStreamSynchronize(copy);
    if (d2h) cudaStreamSynchronize(d2h);
    for (void* p : dev) pool_free(p);
    for (const auto& e : events) pool_event_free(e.first, e.second);
    pool_stream_free(copy);
    pool_stream_free(d2h);
  }
};

struct Ctx {
  Resources res;
  long long bytes = 0;
  int alloc(void** p, size_t n) {
    const int r = pool_alloc(p, n);
    if (r != CQSA_OK) return r;
    res.dev.push_back(*p);
    bytes += static_cast<long long>(n);
    return CQSA_OK;
  }
  int event(cudaEvent_t* e, bool timing) {
    const int r = pool_event(e, timing);
    if (r != CQSA_OK) return r;
    res.events.push_back({*e, timing});
    return CQSA_OK;
  }
};

}  // namespace

// Copy tokens [t0, t0+n) of a tensor (layout, N tokens; host or device memory) into a packed device
// chunk buffer of the same layout ([B,H,n,d] or [B,n,H,d]).
cudaError_t copy_chunk(void* dst, const void* src, int layout, int B, int H, long long N, int d, long long t0, int n,
                       cudaMemcpyKind kind, cudaStream_t s, long long* bytes) {
  const size_t es = 2;
  size_t width, height, spitch;
  const char* base = static_cast<const char*>(src);
  if (layout == CQSA_LAYOUT_BHND) {
    width = static_cast<size_t>(n) * d * es;
    height = static_cast<size_t>(B) * H;
    spitch = static_cast<size_t>(N) * d * es;
    base += static_cast<size_t>(t0) * d * es;
  } else {
    width = static_cast<size_t>(n) * H * d * es;
    height = static_cast<size_t>(B);
    spitch = static_cast<size_t>(N) * H * d * es;
    base += static_cast<size_t>(t0) * H * d * es;
  }
  *bytes += static_cast<long long>(width * height);
  // A chunk that is one contiguous range (token-major with B = 1, or the whole sequence) goes as a
  // plain copy; the strided form only for [B,H,N,d] chunks.
  if (height == 1 || spitch == width) return cudaMemcpyAsync(dst, base, width * height, kind, s);
  return cudaMemcpy2DAsync(dst, width, base, spitch, width, height, kind, s);
}

int launch_finalize(const float* acc, const float* lse_acc, void* out, float* lse_out, int B, int H, int n,
                    long long N, long long t0, int d, int layout, int dtype, cudaStream_t stream) {
  const long long total4 = static_cast<long long>(B) * H * n * d / 4;
  long long blocks = (total4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  finalize_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(acc, lse_acc, out, lse_out, B, H, n, N, t0, d,
                                                               layout, dtype);
  return cuda_status(cudaGetLastError(), "finalize launch");
}

}  // namespace cqsa

using namespace cqsa;

extern "C" int cqsa_stream_attn_fwd(const void* q_host, const void* k_host, const void* v_host, int layout, void* out,
                                    float* lse, int out_on_host, int B, int H, long long N, int d, int causal,
                                    float scale, int dtype, long long chunk_tokens, cqsa_stream_stats* stats,
                                    cudaStream_t stream) {
  const auto t_start = std::chrono::steady_clock::now();
  if (stats) memset(stats, 0, sizeof(*stats));
  if (!q_host || !k_host || !v_host || !out) {
    set_error("q_host, k_host, v_host and out must be non-null");
    return CQSA_ERR_INVALID;
  }
  if (B < 1 || H < 1 || N < 1) {
    set_error("sizes must be positive");
    return CQSA_ERR_INVALID;
  }
  if (d != 64 && d != 128) {
    set_error("head dim %d is not supported (64 or 128)", d);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (dtype != CQSA_F16 && dtype != CQSA_BF16) {
    set_error("dtype %d is not supported", dtype);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (layout != CQSA_LAYOUT_BHND && layout != CQSA_LAYOUT_BNHD) {
    set_error("layout %d is not supported", layout);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (chunk_tokens < 128 || chunk_tokens % 128 != 0 || chunk_tokens > (1LL << 30)) {
    set_error("chunk_tokens must be a positive multiple of 128 (got %lld)", chunk_tokens);
    return CQSA_ERR_INVALID;
  }
  if (!isfinite(scale) || scale < 0.0f) {
    set_error("scale must be finite and >= 0 (0 selects 1/sqrt(d))");
    return CQSA_ERR_INVALID;
  }
  if (static_cast<long long>(B) * H * chunk_tokens > (1LL << 31) - 1) {
    set_error("B*H*chunk_tokens too large for one chunk launch");
    return CQSA_ERR_UNSUPPORTED;
  }
  const float sc = scale == 0.0f ? 1.0f / sqrtf(static_cast<float>(d)) : scale;
  const long long C = chunk_tokens < N ? chunk_tokens : ((N + 127) / 128) * 128;
  const int nch = static_cast<int>((N + C - 1) / C);
  const size_t es = 2;
  const size_t chunk_elems = static_cast<size_t>(B) * H * C * d;

  Ctx cx;
  cx.res.compute = stream;
  cx.res.compute_set = true;
  int rc = CQSA_OK;
  void *qbuf[2] = {nullptr, nullptr}, *kbuf[2] = {nullptr, nullptr}, *vbuf[2] = {nullptr, nullptr};
  void *acc = nullptr, *lacc = nullptr, *ostage = nullptr, *lstage = nullptr;
  // Q is double-buffered too (when there is more than one Q chunk), so the next Q chunk's copy does
  // not wait for the current chunk's last kernel.
  const int nqbuf = nch > 1 ? 2 : 1;
  for (int s = 0; rc == CQSA_OK && s < nqbuf; ++s) rc = cx.alloc(&qbuf[s], chunk_elems * es);
  for (int s = 0; rc == CQSA_OK && s < 2; ++s) {
    rc = cx.alloc(&kbuf[s], chunk_elems * es);
    if (rc == CQSA_OK) rc = cx.alloc(&vbuf[s], chunk_elems * es);
  }
  if (rc == CQSA_OK) rc = cx.alloc(&acc, chunk_elems * 4);
  if (rc == CQSA_OK) rc = cx.alloc(&lacc, static_cast<size_t>(B) * H * C * 4);
  if (rc == CQSA_OK && out_on_host) {
    rc = cx.alloc(&ostage, chunk_elems * es);
    if (rc == CQSA_OK && lse) rc = cx.alloc(&lstage, static_cast<size_t>(B) * H * C * 4);
  }
  if (rc != CQSA_OK) return rc;
  if ((rc = pool_stream(&cx.res.copy)) != CQSA_OK) return rc;
  if ((rc = pool_stream(&cx.res.d2h)) != CQSA_OK) return rc;

  // Events: ordering (no timing) and per-operation timing pairs.
  cudaEvent_t kv_ready[2], kv_free[2], q_ready[2], q_free[2], fin_done, d2h_done;
  for (int s = 0; s < 2; ++s) {
    if ((rc = cx.event(&kv_ready[s], false)) != CQSA_OK) return rc;
    if ((rc = cx.event(&kv_free[s], false)) != CQSA_OK) return rc;
    if ((rc = cx.event(&q_ready[s], false)) != CQSA_OK) return rc;
    if ((rc = cx.event(&q_free[s], false)) != CQSA_OK) return rc;
  }
  if ((rc = cx.event(&fin_done, false)) != CQSA_OK || (rc = cx.event(&d2h_done, false)) != CQSA_OK) return rc;
  struct Span {
    cudaEvent_t a, b;
  };
  std::vector<Span> copies, kernels;
  auto span = [&](std::vector<Span>& v, Span* out_span) -> int {
    Span sp;
    int r = cx.event(&sp.a, true);
    if (r == CQSA_OK) r = cx.event(&sp.b, true);
    if (r == CQSA_OK) {
      v.push_back(sp);
      *out_span = sp;
    }
    return r;
  };

  long long h2d_bytes = 0, d2h_bytes = 0;
  int launches = 0, pairs = 0;
  int slot_of_chunk[2] = {-1, -1};  // KV chunk index resident in each slot
  int next_slot = 0;
  bool q_free_recorded[2] = {false, false}, d2h_recorded = false;

#define CK(call, what)                                 \
  do {                                                 \
    int _r = cuda_status((call), what);                \
    if (_r != CQSA_OK) {                               \
      cudaStreamSynchronize(stream);                   \
      return _r;                                       \
    }                                                  \
  } while (0)

  for (int i = 0; i < nch; ++i) {
    const long long qt0 = static_cast<long long>(i) * C;
    const int qn = static_cast<int>(N - qt0 < C ? N - qt0 : C);
    // Q chunk i goes to buffer i % 2: the kernels of Q chunk i-2 must be done with it.
    const int qs = i % nqbuf;
    if (q_free_recorded[qs]) CK(cudaStreamWaitEvent(cx.res.copy, q_free[qs], 0), "wait q_free");
    {
      Span sp;
      if ((rc = span(copies, &sp)) != CQSA_OK) return rc;
      CK(cudaEventRecord(sp.a, cx.res.copy), "record");
      CK(copy_chunk(qbuf[qs], q_host, layout, B, H, N, d, qt0, qn, cudaMemcpyHostToDevice, cx.res.copy, &h2d_bytes), "copy Q chunk");
      CK(cudaEventRecord(sp.b, cx.res.copy), "record");
    }
    CK(cudaEventRecord(q_ready[qs], cx.res.copy), "record q_ready");
    CK(cudaStreamWaitEvent(stream, q_ready[qs], 0), "wait q_ready");
    // The accumulator is reused per Q chunk: the previous finalize must have read it (same stream),
    // and a host-side D2H of the previous staging buffer must be done before finalize overwrites it.

    const int last_j = causal ? i : nch - 1;
    const bool forward = (i % 2 == 0);
    for (int t = 0; t <= last_j; ++t) {
      const int j = forward ? t : last_j - t;
      const long long kt0 = static_cast<long long>(j) * C;
      const int kn = static_cast<int>(N - kt0 < C ? N - kt0 : C);
      int slot = -1;
      for (int s = 0; s < 2; ++s)
        if (slot_of_chunk[s] == j) slot = s;
      if (slot < 0) {
        slot = next_slot;
        next_slot ^= 1;
        if (slot_of_chunk[slot] >= 0) CK(cudaStreamWaitEvent(cx.res.copy, kv_free[slot], 0), "wait kv_free");
        Span sp;
        if ((rc = span(copies, &sp)) != CQSA_OK) return rc;
        CK(cudaEventRecord(sp.a, cx.res.copy), "record");
        CK(copy_chunk(kbuf[slot], k_host, layout, B, H, N, d, kt0, kn, cudaMemcpyHostToDevice, cx.res.copy, &h2d_bytes), "copy K chunk");
        CK(copy_chunk(vbuf[slot], v_host, layout, B, H, N, d, kt0, kn, cudaMemcpyHostToDevice, cx.res.copy, &h2d_bytes), "copy V chunk");
        CK(cudaEventRecord(sp.b, cx.res.copy), "record");
        CK(cudaEventRecord(kv_ready[slot], cx.res.copy), "record kv_ready");
        slot_of_chunk[slot] = j;
      } else {
        next_slot = slot ^ 1;  // keep the resident chunk; the other slot is the next to refill
      }
      CK(cudaStreamWaitEvent(stream, kv_ready[slot], 0), "wait kv_ready");
      AttnArgs a;
      memset(&a, 0, sizeof(a));
      a.q = qbuf[qs];
      a.k = kbuf[slot];
      a.v = vbuf[slot];
      a.B = B;
      a.H = H;
      a.Nq = qn;
      a.Nkv = kn;
      a.q_off = qt0;
      a.kv_off = kt0;
      a.d = d;
      a.causal = causal != 0;
      a.scale = sc;
      a.dtype = dtype;
      a.in_layout = layout;
      a.mode = (t == 0) ? kModePart : kModeAccum;
      a.o_part = static_cast<float*>(acc);
      a.lse_part = static_cast<float*>(lacc);
      a.out_layout = CQSA_LAYOUT_BHND;
      Span sp;
      if ((rc = span(kernels, &sp)) != CQSA_OK) return rc;
      CK(cudaEventRecord(sp.a, stream), "record");
      rc = launch_attention(a, stream);
      if (rc != CQSA_OK) {
        cudaStreamSynchronize(stream);
        return rc;
      }
      CK(cudaEventRecord(sp.b, stream), "record");
      CK(cudaEventRecord(kv_free[slot], stream), "record kv_free");
      ++launches;
      ++pairs;
    }
    CK(cudaEventRecord(q_free[qs], stream), "record q_free");
    q_free_recorded[qs] = true;

    // Finalize Q chunk i.
    if (out_on_host && d2h_recorded) CK(cudaStreamWaitEvent(stream, d2h_done, 0), "wait d2h_done");
    {
      void* dst = out_on_host ? ostage : out;
      float* ldst = out_on_host ? static_cast<float*>(lstage) : lse;
      const long long Nd = out_on_host ? qn : N;
      const long long td = out_on_host ? 0 : qt0;
      rc = launch_finalize(static_cast<float*>(acc), static_cast<float*>(lacc), dst, ldst, B, H, qn, Nd, td, d, layout,
                           dtype, stream);
      if (rc != CQSA_OK) {
        cudaStreamSynchronize(stream);
        return rc;
      }
      ++launches;
    }
    if (out_on_host) {
      CK(cudaEventRecord(fin_done, stream), "record fin_done");
      CK(cudaStreamWaitEvent(cx.res.d2h, fin_done, 0), "wait fin_done");
      size_t width, height, dpitch;
      char* obase = static_cast<char*>(out);
      if (layout == CQSA_LAYOUT_BHND) {
        width = static_cast<size_t>(qn) * d * es;
        height = static_cast<size_t>(B) * H;
        dpitch = static_cast<size_t>(N) * d * es;
        obase += static_cast<size_t>(qt0) * d * es;
      } else {
        width = static_cast<size_t>(qn) * H * d * es;
        height = static_cast<size_t>(B);
        dpitch = static_cast<size_t>(N) * H * d * es;
        obase += static_cast<size_t>(qt0) * H * d * es;
      }
      if (height == 1 || dpitch == width)
        CK(cudaMemcpyAsync(obase, ostage, width * height, cudaMemcpyDeviceToHost, cx.res.d2h), "D2H out");
      else
        CK(cudaMemcpy2DAsync(obase, dpitch, ostage, width, width, height, cudaMemcpyDeviceToHost, cx.res.d2h),
           "D2H out");
      d2h_bytes += static_cast<long long>(width * height);
      if (lse) {
        const size_t lw = static_cast<size_t>(qn) * 4;
        CK(cudaMemcpy2DAsync(lse + qt0, static_cast<size_t>(N) * 4, lstage, lw, lw, static_cast<size_t>(B) * H,
                             cudaMemcpyDeviceToHost, cx.res.d2h),
           "D2H lse");
        d2h_bytes += static_cast<long long>(lw) * B * H;
      }
      CK(cudaEventRecord(d2h_done, cx.res.d2h), "record d2h_done");
      d2h_recorded = true;
    }
  }
  CK(cudaStreamSynchronize(stream), "synchronize compute stream");
  CK(cudaStreamSynchronize(cx.res.copy), "synchronize copy stream");
  CK(cudaStreamSynchronize(cx.res.d2h), "synchronize d2h stream");
  {
    // the call's own streams have drained; read the device error words on the compute stream
    int r = check_device_error_on(stream);
    if (r != CQSA_OK) return r;
  }
#undef CK
  if (stats) {
    double h2d = 0.0, comp = 0.0, stall = 0.0;
    float ms = 0.0f;
    for (const Span& s : copies)
      if (cudaEventElapsedTime(&ms, s.a, s.b) == cudaSuccess) h2d += ms;
    for (size_t k = 0; k < kernels.size(); ++k) {
      if (cudaEventElapsedTime(&ms, kernels[k].a, kernels[k].b) == cudaSuccess) comp += ms;
      if (k > 0 && cudaEventElapsedTime(&ms, kernels[k - 1].b, kernels[k].a) == cudaSuccess && ms > 0) stall += ms;
    }
    stats->h2d_ms = h2d;
    stats->compute_ms = comp;
    stats->stall_ms = stall;
    stats->h2d_bytes = h2d_bytes;
    stats->d2h_bytes = d2h_bytes;
    stats->peak_device_bytes = cx.bytes;
    stats->n_chunks = pairs;
    stats->n_launches = launches;
    stats->wall_ms =
        std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_start).count();
  }
  return CQSA_OK;
}
