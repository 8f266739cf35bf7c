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
#include <atomic>
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
  std::vector<cudaStream_t> extra;  // further compute streams (pool)
  cudaStream_t compute = nullptr;  // caller's stream: drained before buffers are returned
  bool compute_set = false;
  ~Resources() {
    if (compute_set) cudaStreamSynchronize(compute);
    for (cudaStream_t s : extra) cudaStreamSynchronize(s);
    if (copy) cudaStreamSynchronize(copy);
    if (d2h) cudaStreamSynchronize(d2h);
    for (void* p : dev) pool_free(p);
    for (const auto& e : events) pool_event_free(e.first, e.second);
    pool_stream_free(copy);
    pool_stream_free(d2h);
    for (cudaStream_t s : extra) pool_stream_free(s);
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

// ---------------------------------------------------------------------------------------------------
// Resident inputs. When Q, K, V and the output together fit the budget (cqsa_set_stream_kv_resident_bytes;
// by default half of the device's free memory), each chunk of Q, K and V is copied once, beside the
// kernels, into full-length device tensors where it stays, and each Q chunk runs as ONE launch against
// the key prefix it sees (every key when not causal) in output mode, into its own packed segment of a
// full-size output staging buffer: no fp32 accumulator, no merge, no finalize, and no buffer is reused,
// so the copy stream never waits for a kernel. Q chunks go round-robin over up to kComputeStreams
// streams (the caller's first), so launches whose inputs have landed run side by side: a small chunk's
// launch has fewer CTAs than the GPU has SMs, and one launch's last wave overlaps the next ones.
namespace {
std::atomic<long long> g_kv_resident_bytes{-1};
}  // namespace

bool stream_resident_ok(size_t bytes) {
  const long long lim = g_kv_resident_bytes.load();
  if (lim == 0) return false;
  if (lim > 0) return static_cast<long long>(bytes) <= lim;
  size_t fr = 0, tot = 0;
  if (cudaMemGetInfo(&fr, &tot) != cudaSuccess) return false;
  return bytes <= fr / 2;
}

// Tokens [t0, t0+n) of a (layout, N tokens) tensor into the same positions of another tensor of the
// same shape (host -> device here).
cudaError_t copy_range(void* dst, const void* src, int layout, int B, int H, long long N, int d, long long t0, int n,
                       cudaMemcpyKind kind, cudaStream_t s, long long* bytes) {
  const size_t es = 2;
  size_t width, height, pitch, off;
  if (layout == CQSA_LAYOUT_BHND) {
    width = static_cast<size_t>(n) * d * es;
    height = static_cast<size_t>(B) * H;
    pitch = static_cast<size_t>(N) * d * es;
    off = static_cast<size_t>(t0) * d * es;
  } else {
    width = static_cast<size_t>(n) * H * d * es;
    height = static_cast<size_t>(B);
    pitch = static_cast<size_t>(N) * H * d * es;
    off = static_cast<size_t>(t0) * H * d * es;
  }
  *bytes += static_cast<long long>(width * height);
  if (height == 1 || pitch == width)
    return cudaMemcpyAsync(static_cast<char*>(dst) + off, static_cast<const char*>(src) + off, width * height, kind, s);
  return cudaMemcpy2DAsync(static_cast<char*>(dst) + off, pitch, static_cast<const char*>(src) + off, pitch, width,
                           height, kind, s);
}

int stream_fwd_resident(const void* q_host, const void* k_host, const void* v_host, int layout, void* out, float* lse,
                        int out_on_host, int B, int H, long long N, int d, int causal, float sc, int dtype, long long C,
                        int nch, cqsa_stream_stats* stats, cudaStream_t stream,
                        std::chrono::steady_clock::time_point t_start) {
  const size_t es = 2;
  const size_t full_elems = static_cast<size_t>(B) * H * N * d;
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
  Ctx cx;
  cx.res.compute = stream;
  cx.res.compute_set = true;
  void *qfull = nullptr, *kfull = nullptr, *vfull = nullptr, *ostage = nullptr, *lstage = nullptr;
  int rc = cx.alloc(&qfull, full_elems * es);
  if (rc == CQSA_OK) rc = cx.alloc(&kfull, full_elems * es);
  if (rc == CQSA_OK) rc = cx.alloc(&vfull, full_elems * es);
  if (rc == CQSA_OK) rc = cx.alloc(&ostage, full_elems * es);  // chunk i packed at B*H*i*C*d elements
  if (rc == CQSA_OK && lse) rc = cx.alloc(&lstage, static_cast<size_t>(B) * H * N * 4);
  if (rc != CQSA_OK) return rc;
  if ((rc = pool_stream(&cx.res.copy)) != CQSA_OK) return rc;
  if ((rc = pool_stream(&cx.res.d2h)) != CQSA_OK) return rc;
  // As many streams as it takes for the launches in flight to hold about eight CTAs per SM (a launch has
  // B*H CTAs per 256 query rows), two at least (one launch's last wave beside the next), at most eight.
  constexpr int kComputeStreams = 8;
  const long long ctas = static_cast<long long>(B) * H * ((C + 255) / 256);
  long long want = (8LL * sm_count() + ctas - 1) / ctas;
  want = want < 2 ? 2 : (want > kComputeStreams ? kComputeStreams : want);
  const int ncs = static_cast<int>(nch < want ? nch : want);
  cudaStream_t comp[kComputeStreams] = {stream};
  for (int s = 1; s < ncs; ++s) {
    if ((rc = pool_stream(&comp[s])) != CQSA_OK) return rc;
    cx.res.extra.push_back(comp[s]);
  }
  // Copies run kPrefetch chunks ahead of the launches (enqueued early, so the link never waits for the
  // host); ready[] cycles over 2 * kPrefetch events, each re-recorded only after its previous wait was
  // enqueued. k_done[] is re-recorded per chunk after the D2H stream's wait on it.
  constexpr int kPrefetch = 4;
  // With at most kDeferMax chunks, every output copy is enqueued after the last launch, behind a wait
  // for the last input copy (the two directions slow each other on the link, and the launches still
  // running then leave time for the early chunks' outputs); each chunk has its own k_done event then.
  constexpr int kDeferMax = 64;
  const bool defer = nch <= kDeferMax;
  cudaEvent_t ready[2 * kPrefetch], k_done[kDeferMax], h2d_all, start_ev, end_ev[kComputeStreams];
  for (int s = 0; s < 2 * kPrefetch; ++s)
    if ((rc = cx.event(&ready[s], false)) != CQSA_OK) return rc;
  for (int s = 0; s < (defer ? nch : kComputeStreams); ++s)
    if ((rc = cx.event(&k_done[s], false)) != CQSA_OK) return rc;
  if ((rc = cx.event(&h2d_all, false)) != CQSA_OK) return rc;
  if ((rc = cx.event(&start_ev, false)) != CQSA_OK) return rc;
  for (int s = 0; s < kComputeStreams; ++s)
    if ((rc = cx.event(&end_ev[s], false)) != CQSA_OK) return rc;
  struct Span {
    cudaEvent_t a, b;
  };
  std::vector<Span> copies, kernels;
  auto span = [&](std::vector<Span>& v, Span* sp) -> int {
    int r = cx.event(&sp->a, true);
    if (r == CQSA_OK) r = cx.event(&sp->b, true);
    if (r == CQSA_OK) v.push_back(*sp);
    return r;
  };
  long long h2d_bytes = 0, d2h_bytes = 0;
#define CK(call, what)                              \
  do {                                              \
    int _r = cuda_status((call), what);             \
    if (_r != CQSA_OK) return _r;                   \
  } while (0)
  // work the caller queued on its stream comes first on every stream of this call
  CK(cudaEventRecord(start_ev, stream), "record");
  CK(cudaStreamWaitEvent(cx.res.copy, start_ev, 0), "wait start");
  for (int s = 1; s < ncs; ++s) CK(cudaStreamWaitEvent(comp[s], start_ev, 0), "wait start");
  if (!causal) {
    // every Q chunk needs every key: K and V travel first, whole
    Span sp;
    if ((rc = span(copies, &sp)) != CQSA_OK) return rc;
    CK(cudaEventRecord(sp.a, cx.res.copy), "record");
    CK(copy_range(kfull, k_host, layout, B, H, N, d, 0, static_cast<int>(N), h2d, cx.res.copy, &h2d_bytes), "copy K");
    CK(copy_range(vfull, v_host, layout, B, H, N, d, 0, static_cast<int>(N), h2d, cx.res.copy, &h2d_bytes), "copy V");
    CK(cudaEventRecord(sp.b, cx.res.copy), "record");
  }
  // copies of chunk c: Q_c and (causal) K_c, V_c into their places; launch c needs these and every
  // earlier chunk's, which the copy stream's order gives
  auto enqueue_copies = [&](int c) -> int {
    const long long t0 = static_cast<long long>(c) * C;
    const int n = static_cast<int>(N - t0 < C ? N - t0 : C);
    Span sp;
    int r = span(copies, &sp);
    if (r != CQSA_OK) return r;
    if ((r = cuda_status(cudaEventRecord(sp.a, cx.res.copy), "record")) != CQSA_OK) return r;
    r = cuda_status(copy_range(qfull, q_host, layout, B, H, N, d, t0, n, h2d, cx.res.copy, &h2d_bytes), "copy Q");
    if (r == CQSA_OK && causal)
      r = cuda_status(copy_range(kfull, k_host, layout, B, H, N, d, t0, n, h2d, cx.res.copy, &h2d_bytes), "copy K");
    if (r == CQSA_OK && causal)
      r = cuda_status(copy_range(vfull, v_host, layout, B, H, N, d, t0, n, h2d, cx.res.copy, &h2d_bytes), "copy V");
    if (r == CQSA_OK) r = cuda_status(cudaEventRecord(sp.b, cx.res.copy), "record");
    if (r == CQSA_OK) r = cuda_status(cudaEventRecord(ready[c % (2 * kPrefetch)], cx.res.copy), "record ready");
    if (r == CQSA_OK && c == nch - 1) r = cuda_status(cudaEventRecord(h2d_all, cx.res.copy), "record");
    return r;
  };
  for (int c = 0; c < kPrefetch && c < nch; ++c)
    if ((rc = enqueue_copies(c)) != CQSA_OK) return rc;
  // the output rows (and lse) of chunk i from its staging segment, on the D2H stream after launch i
  const cudaMemcpyKind okind = out_on_host ? cudaMemcpyDeviceToHost : cudaMemcpyDeviceToDevice;
  auto enqueue_out = [&](int i, cudaEvent_t done) -> int {
    const long long qt0 = static_cast<long long>(i) * C;
    const int qn = static_cast<int>(N - qt0 < C ? N - qt0 : C);
    const char* oseg = static_cast<const char*>(ostage) + static_cast<size_t>(B) * H * qt0 * d * es;
    int r = cuda_status(cudaStreamWaitEvent(cx.res.d2h, done, 0), "wait k_done");
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
    if (r == CQSA_OK)
      r = cuda_status(height == 1 || dpitch == width
                          ? cudaMemcpyAsync(obase, oseg, width * height, okind, cx.res.d2h)
                          : cudaMemcpy2DAsync(obase, dpitch, oseg, width, width, height, okind, cx.res.d2h),
                      "copy out");
    d2h_bytes += static_cast<long long>(width * height);
    if (r == CQSA_OK && lse) {
      const size_t lw = static_cast<size_t>(qn) * 4;
      const float* lseg = static_cast<const float*>(lstage) + static_cast<size_t>(B) * H * qt0;
      r = cuda_status(cudaMemcpy2DAsync(lse + qt0, static_cast<size_t>(N) * 4, lseg, lw, lw,
                                        static_cast<size_t>(B) * H, okind, cx.res.d2h),
                      "copy lse");
      d2h_bytes += static_cast<long long>(lw) * B * H;
    }
    return r;
  };
  for (int i = 0; i < nch; ++i) {
    const int s = i % ncs;
    const long long qt0 = static_cast<long long>(i) * C;
    const int qn = static_cast<int>(N - qt0 < C ? N - qt0 : C);
    cudaStream_t cs = comp[s];
    if (i + kPrefetch < nch && (rc = enqueue_copies(i + kPrefetch)) != CQSA_OK) return rc;
    CK(cudaStreamWaitEvent(cs, ready[i % (2 * kPrefetch)], 0), "wait ready");
    // Q chunk i in place in the full tensor; its packed output segment
    const size_t qoff = layout == CQSA_LAYOUT_BHND ? static_cast<size_t>(qt0) * d * es
                                                   : static_cast<size_t>(qt0) * H * d * es;
    char* oseg = static_cast<char*>(ostage) + static_cast<size_t>(B) * H * qt0 * d * es;
    float* lseg = lse ? static_cast<float*>(lstage) + static_cast<size_t>(B) * H * qt0 : nullptr;
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.q = static_cast<char*>(qfull) + qoff;
    a.q_tokens_alloc = N;
    a.k = kfull;
    a.v = vfull;
    a.B = B;
    a.H = H;
    a.Nq = qn;
    a.Nkv = static_cast<int>(causal ? qt0 + qn : N);
    a.q_off = qt0;
    a.kv_off = 0;
    a.kv_tokens_alloc = N;
    a.d = d;
    a.causal = causal != 0;
    a.scale = sc;
    a.dtype = dtype;
    a.in_layout = layout;
    a.mode = kModeOut;
    a.out = oseg;
    a.lse = lseg;
    a.out_layout = layout;
    {
      Span sp;
      if ((rc = span(kernels, &sp)) != CQSA_OK) return rc;
      CK(cudaEventRecord(sp.a, cs), "record");
      if ((rc = launch_attention(a, cs)) != CQSA_OK) return rc;
      CK(cudaEventRecord(sp.b, cs), "record");
    }
    cudaEvent_t done = k_done[defer ? i : s];
    CK(cudaEventRecord(done, cs), "record k_done");
    if (!defer && (rc = enqueue_out(i, done)) != CQSA_OK) return rc;
  }
  if (defer) {
    CK(cudaStreamWaitEvent(cx.res.d2h, h2d_all, 0), "wait h2d_all");
    for (int i = 0; i < nch; ++i)
      if ((rc = enqueue_out(i, k_done[i])) != CQSA_OK) return rc;
  }
  // the caller's stream ends after every stream of this call
  for (int s = 1; s < ncs; ++s) {
    CK(cudaEventRecord(end_ev[s], comp[s]), "record");
    CK(cudaStreamWaitEvent(stream, end_ev[s], 0), "wait end");
  }
  for (int s = 1; s < ncs; ++s) CK(cudaStreamSynchronize(comp[s]), "synchronize compute streams");
  CK(cudaStreamSynchronize(stream), "synchronize compute stream");
  CK(cudaStreamSynchronize(cx.res.copy), "synchronize copy stream");
  CK(cudaStreamSynchronize(cx.res.d2h), "synchronize d2h stream");
#undef CK
  if ((rc = check_device_error_on(stream)) != CQSA_OK) return rc;
  if (stats) {
    double h2d_ms = 0.0, comp_ms = 0.0, stall = 0.0;
    float ms = 0.0f;
    for (const Span& s : copies)
      if (cudaEventElapsedTime(&ms, s.a, s.b) == cudaSuccess) h2d_ms += ms;
    // kernel time: the union of the launches' intervals (they overlap on two streams); stall: the gaps
    // of that union after the first launch begins
    double end_rel = 0.0;  // end of the union so far, relative to the first launch's start
    for (size_t k = 0; k < kernels.size(); ++k) {
      float a0 = 0.0f, b0 = 0.0f;
      if (cudaEventElapsedTime(&a0, kernels[0].a, kernels[k].a) != cudaSuccess) continue;
      if (cudaEventElapsedTime(&b0, kernels[0].a, kernels[k].b) != cudaSuccess) continue;
      if (k > 0 && a0 > end_rel) stall += a0 - end_rel;
      const double lo = a0 > end_rel ? a0 : end_rel;
      if (b0 > lo) comp_ms += b0 - lo;
      if (b0 > end_rel) end_rel = b0;
    }
    stats->h2d_ms = h2d_ms;
    stats->compute_ms = comp_ms;
    stats->stall_ms = stall;
    stats->h2d_bytes = h2d_bytes;
    stats->d2h_bytes = d2h_bytes;
    stats->peak_device_bytes = cx.bytes;
    stats->n_chunks = nch;
    stats->n_launches = static_cast<int>(kernels.size());
    stats->wall_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_start).count();
  }
  return CQSA_OK;
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
  // Resident inputs when they fit the budget and one head's whole K and V fit the L2 share the kernel
  // groups heads by (64 MB): a launch over the key prefix has every CTA sweep its head's keys, which
  // stay in L2 only then (4M tokens, 1 GB per head: 1,091 TFLOP/s resident against 1,145 accumulating).
  const bool kv_fits_l2 = 2.0 * static_cast<double>(N) * d * es <= 64.0 * 1024 * 1024;
  if (N <= 0x7fffffffLL && kv_fits_l2 &&
      stream_resident_ok(4 * static_cast<size_t>(B) * H * N * d * es + static_cast<size_t>(B) * H * N * 4))
    return stream_fwd_resident(q_host, k_host, v_host, layout, out, lse, out_on_host, B, H, N, d, causal, sc, dtype, C,
                               nch, stats, stream, t_start);

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

extern "C" void cqsa_set_stream_kv_resident_bytes(long long bytes) {
  g_kv_resident_bytes.store(bytes < 0 ? -1 : bytes);
}
