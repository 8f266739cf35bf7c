// Host-resident attention backward: q, k, v, out, dout and lse stay in (pinned) host memory and travel
// to the device in token chunks; every needed (query chunk, key chunk) pair runs the backward's
// chunk-pair kernel into fp32 device accumulators, and dq, dk, dv return to host memory. The pages'
// streamed backward (`stream_cqsa_backward`, "stream-cqsa 2.2.0 -> 2.2.2" diff, README list of
// explicit entry points) works subproblem by subproblem from the forward's saved lse ("stream-cqsa
// 2.2.2 -> 2.2.3" diff, stream_cqsa/oom_fallback.py, `stream_cqsa_auto` docstring).
//
// Schedule (query-outer): for each query chunk, its q, out, dout and lse are copied on a copy stream
// into one of two query-side slots (the next chunk's copies overlap this chunk's kernels), D =
// rowsum(dout * out) is formed and its fp32 dq accumulator zeroed; the key chunks it needs (every chunk,
// or those starting at or before the query chunk's last token when causal) go through two K/V slots on
// the copy stream, in alternating directions from one query chunk to the next, so the chunk that ends
// one query chunk is not copied again for the next; each pair adds into dq and into that key chunk's
// fp32 dk / dv accumulators. dq is rounded to the input dtype into one of two staging buffers and leaves
// on a second stream; once every query chunk is done, dk and dv of each key chunk follow the same way.
// Device memory: the dk / dv accumulators of the whole sequence (2 * B*H*N*d * 4 bytes) plus two slots
// of each streamed chunk. When everything fits the resident budget (stream_bwd_resident below), the
// inputs instead stay on the device once copied and each key chunk is one launch over every query.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <vector>

#include "cqsa_internal.h"

// Run one CUDA call only while every earlier step succeeded, keeping the first failure.
#define CQSA_STEP(expr, what)                               \
  do {                                                      \
    if (rc == CQSA_OK) rc = cuda_status((expr), (what));    \
  } while (0)

namespace cqsa {
namespace {

// A packed [B,H,n,d] device chunk into tokens [t0, t0 + n) of a [B,H,N,d] host tensor (16-bit).
cudaError_t copy_chunk_out(void* host, const void* dev, int B, int H, long long N, int d, long long t0, int n,
                           cudaStream_t s) {
  const size_t row = static_cast<size_t>(n) * d * 2;
  char* dst = static_cast<char*>(host) + static_cast<size_t>(t0) * d * 2;
  return cudaMemcpy2DAsync(dst, static_cast<size_t>(N) * d * 2, dev, row, row, static_cast<size_t>(B) * H,
                           cudaMemcpyDeviceToHost, s);
}

}  // namespace

// ---------------------------------------------------------------------------------------------------
// Resident inputs. When q, out, dout (whole), lse, D, the fp32 dq accumulator, every K/V chunk, the dk/dv
// accumulators and the output staging fit the budget the forward's streaming uses
// (cqsa_set_stream_kv_resident_bytes), every chunk is copied once and stays. Key chunks are visited from
// the last to the first, and the query side is copied in the same order: key chunk j needs the queries at
// or after its first key (causal), which have then all arrived. Each key chunk is one launch of the
// chunk-pair kernel over every query of the sequence (the kernel starts at the first query tile that
// sees the chunk), so a key tile's CTA walks all of its query tiles in one go. The launches go
// round-robin over up to four streams; the dq reductions are atomic, dk and dv are per chunk. Copying
// the whole query side first and then running the key chunks heaviest first measured slower on 131K
// causal tokens (856 against 875 TFLOP/s): the first launch waited for every query to arrive.
int stream_bwd_resident(const void* q, const void* k, const void* v, const void* out, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, int B, int H, long long N, int d, int causal,
                        float sc, int dtype, long long C, int n_chunks, cqsa_stream_stats* stats, cudaStream_t stream,
                        std::chrono::steady_clock::time_point t_start) {
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t full16 = BH * static_cast<size_t>(N) * d * 2, full32 = 2 * full16;
  const size_t chunk16 = BH * static_cast<size_t>(C) * d * 2, chunk32 = 2 * chunk16;
  const size_t rowsN = BH * static_cast<size_t>(N) * 4;
  std::vector<void*> bufs;
  std::vector<cudaEvent_t> events, tevents;  // ordering events, timing events
  cudaStream_t copy = nullptr, prep = nullptr, d2h = nullptr;
  constexpr int kStreams = 4;
  cudaStream_t comp[kStreams] = {stream, nullptr, nullptr, nullptr};
  long long dev_bytes = 0, bytes = 0, d2h_bytes = 0;
  int rc = CQSA_OK;
  auto alloc = [&](void** ptr, size_t n) -> int {
    const int r = pool_alloc(ptr, n);
    if (r == CQSA_OK) {
      bufs.push_back(*ptr);
      dev_bytes += static_cast<long long>(n);
    }
    return r;
  };
  auto event = [&](cudaEvent_t* e, bool timing) -> int {
    const int r = pool_event(e, timing);
    if (r == CQSA_OK) (timing ? tevents : events).push_back(*e);
    return r;
  };
  void *qf = nullptr, *of = nullptr, *gf = nullptr, *lf = nullptr, *df = nullptr, *dqf = nullptr;
  void *kvc = nullptr, *acc = nullptr, *ostage = nullptr;
  rc = alloc(&qf, full16);
  if (rc == CQSA_OK) rc = alloc(&of, full16);
  if (rc == CQSA_OK) rc = alloc(&gf, full16);
  if (rc == CQSA_OK) rc = alloc(&lf, rowsN);
  if (rc == CQSA_OK) rc = alloc(&df, rowsN);
  if (rc == CQSA_OK) rc = alloc(&dqf, full32);
  if (rc == CQSA_OK) rc = alloc(&kvc, 2 * static_cast<size_t>(n_chunks) * chunk16);   // [chunk][k | v]
  if (rc == CQSA_OK) rc = alloc(&acc, 2 * static_cast<size_t>(n_chunks) * chunk32);   // [chunk][dk | dv]
  if (rc == CQSA_OK) rc = alloc(&ostage, full16 + 2 * static_cast<size_t>(n_chunks) * chunk16);
  if (rc == CQSA_OK) rc = pool_stream(&copy);
  if (rc == CQSA_OK) rc = pool_stream(&prep);
  if (rc == CQSA_OK) rc = pool_stream(&d2h);
  const int ncs = n_chunks < kStreams ? n_chunks : kStreams;
  for (int s = 1; rc == CQSA_OK && s < ncs; ++s) rc = pool_stream(&comp[s]);
  std::vector<cudaEvent_t> prep_done(n_chunks), k_ready(n_chunks), done(n_chunks);
  cudaEvent_t start_ev = nullptr, all_done = nullptr, cast_done = nullptr;
  for (int i = 0; rc == CQSA_OK && i < n_chunks; ++i) {
    if ((rc = event(&prep_done[i], false)) == CQSA_OK && (rc = event(&k_ready[i], false)) == CQSA_OK)
      rc = event(&done[i], false);
  }
  if (rc == CQSA_OK) rc = event(&start_ev, false);
  if (rc == CQSA_OK) rc = event(&all_done, false);
  if (rc == CQSA_OK) rc = event(&cast_done, false);
  // timing spans (stats): kernels on the compute streams, copies on the copy stream
  struct Span {
    cudaEvent_t a, b;
  };
  std::vector<Span> kspans, cspans;
  auto span_begin = [&](std::vector<Span>& vsp, cudaStream_t s) {
    if (!stats || rc != CQSA_OK) return;
    Span sp{nullptr, nullptr};
    if ((rc = event(&sp.a, true)) != CQSA_OK || (rc = event(&sp.b, true)) != CQSA_OK) return;
    vsp.push_back(sp);
    rc = cuda_status(cudaEventRecord(sp.a, s), "record");
  };
  auto span_end = [&](std::vector<Span>& vsp, cudaStream_t s) {
    if (!stats || rc != CQSA_OK) return;
    rc = cuda_status(cudaEventRecord(vsp.back().b, s), "record");
  };
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
  auto fp32_rows = [&](float* dst, const float* src, long long t0, int n) -> cudaError_t {
    bytes += static_cast<long long>(BH) * n * 4;
    return cudaMemcpy2DAsync(dst + t0, static_cast<size_t>(N) * 4, src + t0, static_cast<size_t>(N) * 4,
                             static_cast<size_t>(n) * 4, BH, h2d, copy);
  };
  // the query side of chunk i (q, out, dout, lse into place) and its D
  auto query_side = [&](int i) {
    const long long t0 = static_cast<long long>(i) * C;
    const int n = static_cast<int>(N - t0 < C ? N - t0 : C);
    span_begin(cspans, copy);
    CQSA_STEP(copy_range(qf, q, CQSA_LAYOUT_BHND, B, H, N, d, t0, n, h2d, copy, &bytes), "copy q");
    CQSA_STEP(copy_range(of, out, CQSA_LAYOUT_BHND, B, H, N, d, t0, n, h2d, copy, &bytes), "copy out");
    CQSA_STEP(copy_range(gf, dout, CQSA_LAYOUT_BHND, B, H, N, d, t0, n, h2d, copy, &bytes), "copy dout");
    CQSA_STEP(fp32_rows(static_cast<float*>(lf), lse, t0, n), "copy lse");
    span_end(cspans, copy);
    CQSA_STEP(cudaEventRecord(prep_done[i], copy), "record");
    CQSA_STEP(cudaStreamWaitEvent(prep, prep_done[i], 0), "wait copy");
    if (rc == CQSA_OK)
      rc = launch_bwd_dvec_range(of, gf, static_cast<float*>(df), static_cast<long long>(BH), n, N, t0, d, dtype,
                                 prep);
    CQSA_STEP(cudaEventRecord(prep_done[i], prep), "record");
  };
  auto kv_side = [&](int j) {
    const long long t0 = static_cast<long long>(j) * C;
    const int n = static_cast<int>(N - t0 < C ? N - t0 : C);
    char* kj = static_cast<char*>(kvc) + 2 * static_cast<size_t>(j) * chunk16;
    span_begin(cspans, copy);
    CQSA_STEP(copy_chunk(kj, k, CQSA_LAYOUT_BHND, B, H, N, d, t0, n, h2d, copy, &bytes), "copy k");
    CQSA_STEP(copy_chunk(kj + chunk16, v, CQSA_LAYOUT_BHND, B, H, N, d, t0, n, h2d, copy, &bytes), "copy v");
    span_end(cspans, copy);
    CQSA_STEP(cudaEventRecord(k_ready[j], copy), "record");
  };
  CQSA_STEP(cudaEventRecord(start_ev, stream), "record");
  CQSA_STEP(cudaStreamWaitEvent(copy, start_ev, 0), "wait start");
  CQSA_STEP(cudaStreamWaitEvent(prep, start_ev, 0), "wait start");
  for (int s = 1; s < ncs; ++s) CQSA_STEP(cudaStreamWaitEvent(comp[s], start_ev, 0), "wait start");
  CQSA_STEP(cudaMemsetAsync(dqf, 0, full32, prep), "zero dq accumulator");
  CQSA_STEP(cudaMemsetAsync(acc, 0, 2 * static_cast<size_t>(n_chunks) * chunk32, prep), "zero dk/dv accumulators");
  if (!causal)
    for (int i = n_chunks - 1; i >= 0; --i) query_side(i);
  for (int j = n_chunks - 1; j >= 0 && rc == CQSA_OK; --j) {
    if (causal) query_side(j);
    kv_side(j);
    const long long t0 = static_cast<long long>(j) * C;
    const int n = static_cast<int>(N - t0 < C ? N - t0 : C);
    cudaStream_t cs = comp[(n_chunks - 1 - j) % ncs];
    // every query this key chunk meets has its D (the prep stream runs in copy order), and its K / V
    CQSA_STEP(cudaStreamWaitEvent(cs, prep_done[causal ? j : 0], 0), "wait prep");
    CQSA_STEP(cudaStreamWaitEvent(cs, k_ready[j], 0), "wait k");
    char* kj = static_cast<char*>(kvc) + 2 * static_cast<size_t>(j) * chunk16;
    float* dkj = reinterpret_cast<float*>(static_cast<char*>(acc) + 2 * static_cast<size_t>(j) * chunk32);
    BwdArgs a;
    memset(&a, 0, sizeof(a));
    a.q = qf;
    a.k = kj;
    a.v = kj + chunk16;
    a.dout = gf;
    a.lse = static_cast<const float*>(lf);
    a.dvec = static_cast<const float*>(df);
    a.dq_acc = static_cast<float*>(dqf);
    a.dk_acc = dkj;
    a.dv_acc = dkj + chunk32 / 4;
    a.B = B;
    a.H = H;
    a.Nq = static_cast<int>(N);
    a.Nkv = n;
    a.d = d;
    a.q_off = 0;
    a.kv_off = t0;
    a.causal = causal != 0;
    a.scale = sc;
    a.dtype = dtype;
    span_begin(kspans, cs);
    if (rc == CQSA_OK) rc = launch_attention_bwd_chunk(a, cs);
    // dk and dv of this chunk: rounded into their staging and sent
    char* sk = static_cast<char*>(ostage) + full16 + 2 * static_cast<size_t>(j) * chunk16;
    if (rc == CQSA_OK) rc = launch_bwd_cast(dkj, sk, static_cast<long long>(BH) * n * d, dtype, cs);
    if (rc == CQSA_OK) rc = launch_bwd_cast(dkj + chunk32 / 4, sk + chunk16, static_cast<long long>(BH) * n * d, dtype, cs);
    span_end(kspans, cs);
    CQSA_STEP(cudaEventRecord(done[j], cs), "record");
    CQSA_STEP(cudaStreamWaitEvent(d2h, done[j], 0), "wait chunk");
    CQSA_STEP(copy_chunk_out(dk, sk, B, H, N, d, t0, n, d2h), "copy dk");
    CQSA_STEP(copy_chunk_out(dv, sk + chunk16, B, H, N, d, t0, n, d2h), "copy dv");
    d2h_bytes += 2 * static_cast<long long>(BH) * n * d * 2;
  }
  // dq once every key chunk has added into it
  for (int s = 1; s < ncs; ++s) {
    CQSA_STEP(cudaEventRecord(all_done, comp[s]), "record");
    CQSA_STEP(cudaStreamWaitEvent(stream, all_done, 0), "join");
  }
  span_begin(kspans, stream);
  if (rc == CQSA_OK) rc = launch_bwd_cast(static_cast<float*>(dqf), ostage, static_cast<long long>(BH) * N * d, dtype, stream);
  span_end(kspans, stream);
  CQSA_STEP(cudaEventRecord(cast_done, stream), "record");
  CQSA_STEP(cudaStreamWaitEvent(d2h, cast_done, 0), "wait dq");
  CQSA_STEP(cudaMemcpyAsync(dq, ostage, full16, cudaMemcpyDeviceToHost, d2h), "copy dq");
  d2h_bytes += static_cast<long long>(full16);
  cudaError_t se = cudaStreamSynchronize(stream);
  if (rc == CQSA_OK) rc = cuda_status(se, "synchronize");
  for (cudaStream_t s : {copy, prep, d2h, comp[1], comp[2], comp[3]}) {
    if (!s) continue;
    se = cudaStreamSynchronize(s);
    if (rc == CQSA_OK) rc = cuda_status(se, "synchronize");
  }
  if (rc == CQSA_OK) rc = check_device_error_on(stream);
  if (rc == CQSA_OK && stats) {
    // kernel time: the union of the launches' intervals (they overlap on several streams); stall: its gaps
    double comp_ms = 0.0, h2d_ms = 0.0, stall = 0.0;
    float ms = 0.0f;
    std::vector<std::pair<double, double>> iv;
    for (const Span& s : kspans) {
      float a0 = 0.0f, b0 = 0.0f;
      if (cudaEventElapsedTime(&a0, kspans[0].a, s.a) == cudaSuccess &&
          cudaEventElapsedTime(&b0, kspans[0].a, s.b) == cudaSuccess)
        iv.push_back({a0, b0});
    }
    std::sort(iv.begin(), iv.end());
    double end_rel = iv.empty() ? 0.0 : iv[0].first;
    for (const auto& x : iv) {
      if (x.first > end_rel) stall += x.first - end_rel;
      const double lo = x.first > end_rel ? x.first : end_rel;
      if (x.second > lo) comp_ms += x.second - lo;
      if (x.second > end_rel) end_rel = x.second;
    }
    for (const Span& s : cspans)
      if (cudaEventElapsedTime(&ms, s.a, s.b) == cudaSuccess) h2d_ms += ms;
    stats->compute_ms = comp_ms;
    stats->stall_ms = stall;
    stats->h2d_ms = h2d_ms;
    stats->h2d_bytes = bytes;
    stats->d2h_bytes = d2h_bytes;
    stats->peak_device_bytes = dev_bytes;
    stats->n_chunks = n_chunks;
    stats->n_launches = static_cast<int>(kspans.size());
    stats->wall_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_start).count();
  }
  for (cudaEvent_t e : events) pool_event_free(e, false);
  for (cudaEvent_t e : tevents) pool_event_free(e, true);
  for (cudaStream_t s : {copy, prep, d2h, comp[1], comp[2], comp[3]}) pool_stream_free(s);
  for (void* b2 : bufs) pool_free(b2);
  return rc;
}

}  // namespace cqsa

using namespace cqsa;

extern "C" int cqsa_stream_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int H, long long N, int d,
                                    int causal, float scale, int dtype, long long chunk_tokens, cudaStream_t stream) {
  return cqsa_stream_attn_bwd_ex(q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, dtype, chunk_tokens,
                                 nullptr, stream);
}

extern "C" int cqsa_stream_attn_bwd_ex(const void* q, const void* k, const void* v, const void* out,
                                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int H,
                                       long long N, int d, int causal, float scale, int dtype,
                                       long long chunk_tokens, cqsa_stream_stats* stats, cudaStream_t stream) {
  const auto t_start = std::chrono::steady_clock::now();
  if (stats) memset(stats, 0, sizeof(*stats));
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) {
    set_error("q, k, v, out, dout, lse, dq, dk and dv must be non-null host pointers");
    return CQSA_ERR_INVALID;
  }
  if (B < 1 || H < 1 || N < 1) {
    set_error("sizes must be positive (B=%d H=%d N=%lld)", B, H, N);
    return CQSA_ERR_INVALID;
  }
  if (dtype != CQSA_F16 && dtype != CQSA_BF16) {
    set_error("dtype %d is not supported (fp16 or bf16)", dtype);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (d != 64 && d != 128) {
    set_error("the backward supports head dim 64 or 128 (got %d)", d);
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
  if (static_cast<long long>(B) * H * C > (1LL << 31) / d || N > 0x7fffffffLL) {
    set_error("B*H*chunk_tokens too large for one chunk launch");
    return CQSA_ERR_UNSUPPORTED;
  }
  const int n_chunks = static_cast<int>((N + C - 1) / C);
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t chunk16 = BH * static_cast<size_t>(C) * d * 2;  // one 16-bit chunk
  const size_t chunk32 = BH * static_cast<size_t>(C) * d * 4;  // one fp32 chunk
  const size_t rows32 = BH * static_cast<size_t>(C) * 4;
  const float sc = scale == 0.0f ? 1.0f / sqrtf(static_cast<float>(d)) : scale;
  {
    // resident inputs when everything fits the budget: about 14 bytes of device memory per input byte
    // of one tensor (q, out, dout, the dq accumulator, the K/V chunks, the dk/dv accumulators, staging)
    const size_t full16 = BH * static_cast<size_t>(N) * d * 2;
    const size_t need = 6 * full16 + 2 * BH * static_cast<size_t>(N) * 4 + 8 * static_cast<size_t>(n_chunks) * chunk16;
    if (N <= 0x7fffffffLL && stream_resident_ok(need))
      return stream_bwd_resident(q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, causal, sc, dtype, C, n_chunks, stats,
                                 stream, t_start);
  }

  // Device memory: the dk / dv accumulators of every key chunk, and two slots of everything that
  // streams: the query side (q, out, dout, lse, D, the dq accumulator), the key side (k, v) and the
  // output staging.
  struct QSlot {
    void *q, *out, *g;
    float *lse, *dvec, *dq;
  } qsl[2];
  struct KSlot {
    void *k, *v;
  } ksl[2];
  void* ostage[2] = {nullptr, nullptr};
  std::vector<void*> bufs;
  cudaStream_t copy = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> events;
  long long dev_bytes = 0;
  auto alloc = [&](void** ptr, size_t n) -> int {
    const int r = pool_alloc(ptr, n);
    if (r == CQSA_OK) {
      bufs.push_back(*ptr);
      dev_bytes += static_cast<long long>(n);
    }
    return r;
  };
  auto event = [&](cudaEvent_t* e) -> int {
    const int r = pool_event(e, false);
    if (r == CQSA_OK) events.push_back(*e);
    return r;
  };
  void* acc_kv = nullptr;
  const size_t acc_bytes = 2 * static_cast<size_t>(n_chunks) * chunk32;
  int rc = alloc(&acc_kv, acc_bytes);
  for (int s2 = 0; s2 < 2 && rc == CQSA_OK; ++s2) {
    void* pq = nullptr;
    rc = alloc(&pq, 3 * chunk16 + chunk32 + 2 * rows32 + 256);
    if (rc != CQSA_OK) break;
    char* c = static_cast<char*>(pq);
    qsl[s2].q = c;
    qsl[s2].out = c + chunk16;
    qsl[s2].g = c + 2 * chunk16;
    qsl[s2].dq = reinterpret_cast<float*>(c + 3 * chunk16);
    qsl[s2].lse = reinterpret_cast<float*>(c + 3 * chunk16 + chunk32);
    qsl[s2].dvec = reinterpret_cast<float*>(c + 3 * chunk16 + chunk32 + rows32);
    void* pk = nullptr;
    if (rc == CQSA_OK) rc = alloc(&pk, 2 * chunk16);
    if (rc != CQSA_OK) break;
    ksl[s2].k = pk;
    ksl[s2].v = static_cast<char*>(pk) + chunk16;
    if (rc == CQSA_OK) rc = alloc(&ostage[s2], chunk16);
  }
  if (rc == CQSA_OK) rc = pool_stream(&copy);
  if (rc == CQSA_OK) rc = pool_stream(&d2h);
  cudaEvent_t q_ready[2], q_free[2], kv_ready[2], kv_free[2], o_ready[2], o_free[2];
  bool q_free_set[2] = {false, false}, kv_free_set[2] = {false, false}, o_free_set[2] = {false, false};
  for (int s2 = 0; s2 < 2 && rc == CQSA_OK; ++s2) {
    if ((rc = event(&q_ready[s2])) == CQSA_OK && (rc = event(&q_free[s2])) == CQSA_OK &&
        (rc = event(&kv_ready[s2])) == CQSA_OK && (rc = event(&kv_free[s2])) == CQSA_OK &&
        (rc = event(&o_ready[s2])) == CQSA_OK)
      rc = event(&o_free[s2]);
  }
  // with stats: timing events around every kernel segment on `stream` and every copy group on `copy`
  struct Span {
    cudaEvent_t a, b;
  };
  std::vector<Span> kspans, cspans;
  std::vector<cudaEvent_t> tevents;
  auto tspan = [&](std::vector<Span>& v, cudaStream_t s, bool begin) {
    if (!stats || rc != CQSA_OK) return;
    if (begin) {
      Span sp{nullptr, nullptr};
      if ((rc = pool_event(&sp.a, true)) != CQSA_OK) return;
      tevents.push_back(sp.a);
      if ((rc = pool_event(&sp.b, true)) != CQSA_OK) return;
      tevents.push_back(sp.b);
      v.push_back(sp);
      rc = cuda_status(cudaEventRecord(sp.a, s), "record");
    } else {
      rc = cuda_status(cudaEventRecord(v.back().b, s), "record");
    }
  };
  long long d2h_bytes = 0;
  int n_pairs = 0, n_launches = 0;
  float* dk_acc0 = static_cast<float*>(acc_kv);
  float* dv_acc0 = dk_acc0 + static_cast<size_t>(n_chunks) * (chunk32 / 4);

  long long bytes = 0;
  int out_slot = 0;  // output staging slots alternate over every chunk written out (dq, then dk, dv)
  // A 16-bit [B,H,n,d] result into staging slot out_slot (after its previous D2H), then to host rows [t0, t0+n).
  auto write_out = [&](const float* acc, void* host, long long t0, int n) {
    const int os = out_slot;
    out_slot ^= 1;
    if (o_free_set[os]) CQSA_STEP(cudaStreamWaitEvent(stream, o_free[os], 0), "wait staging");
    tspan(kspans, stream, true);
    if (rc == CQSA_OK) rc = launch_bwd_cast(acc, ostage[os], static_cast<long long>(BH) * n * d, dtype, stream);
    tspan(kspans, stream, false);
    ++n_launches;
    d2h_bytes += static_cast<long long>(BH) * n * d * 2;
    CQSA_STEP(cudaEventRecord(o_ready[os], stream), "record");
    CQSA_STEP(cudaStreamWaitEvent(d2h, o_ready[os], 0), "wait cast");
    CQSA_STEP(copy_chunk_out(host, ostage[os], B, H, N, d, t0, n, d2h), "copy out");
    CQSA_STEP(cudaEventRecord(o_free[os], d2h), "record");
    o_free_set[os] = true;
  };

  CQSA_STEP(cudaMemsetAsync(acc_kv, 0, acc_bytes, stream), "zero dk/dv accumulators");
  int kv_chunk[2] = {-1, -1};  // key chunk resident in each K/V slot
  int next_kv = 0;
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
  for (int qi = 0; qi < n_chunks && rc == CQSA_OK; ++qi) {
    const long long qs = static_cast<long long>(qi) * C;
    const int nq = static_cast<int>(N - qs < C ? N - qs : C);
    const QSlot& Q = qsl[qi & 1];
    // the query side of chunk qi - 2 is done with this slot
    if (q_free_set[qi & 1]) CQSA_STEP(cudaStreamWaitEvent(copy, q_free[qi & 1], 0), "wait q slot");
    tspan(cspans, copy, true);
    CQSA_STEP(copy_chunk(Q.q, q, CQSA_LAYOUT_BHND, B, H, N, d, qs, nq, h2d, copy, &bytes), "copy q");
    CQSA_STEP(copy_chunk(Q.out, out, CQSA_LAYOUT_BHND, B, H, N, d, qs, nq, h2d, copy, &bytes), "copy out");
    CQSA_STEP(copy_chunk(Q.g, dout, CQSA_LAYOUT_BHND, B, H, N, d, qs, nq, h2d, copy, &bytes), "copy dout");
    CQSA_STEP(cudaMemcpy2DAsync(Q.lse, static_cast<size_t>(nq) * 4, lse + qs, static_cast<size_t>(N) * 4,
                                static_cast<size_t>(nq) * 4, BH, h2d, copy),
              "copy lse");
    bytes += static_cast<long long>(BH) * nq * 4;
    tspan(cspans, copy, false);
    CQSA_STEP(cudaEventRecord(q_ready[qi & 1], copy), "record");
    CQSA_STEP(cudaStreamWaitEvent(stream, q_ready[qi & 1], 0), "wait q");
    tspan(kspans, stream, true);
    if (rc == CQSA_OK) rc = launch_bwd_dvec(Q.out, Q.g, Q.dvec, static_cast<long long>(BH) * nq, d, dtype, stream);
    CQSA_STEP(cudaMemsetAsync(Q.dq, 0, BH * static_cast<size_t>(nq) * d * 4, stream), "zero dq accumulator");
    tspan(kspans, stream, false);
    ++n_launches;
    // key chunks this query chunk needs (every chunk, or those at or before its last token when causal),
    // in alternating directions, so the chunk that ends one query chunk starts the next one
    int last = n_chunks - 1;
    if (causal) last = static_cast<int>((qs + nq - 1) / C);
    for (int t = 0; t <= last && rc == CQSA_OK; ++t) {
      const int ki = (qi & 1) ? last - t : t;
      const long long ks = static_cast<long long>(ki) * C;
      const int nk = static_cast<int>(N - ks < C ? N - ks : C);
      int slot = kv_chunk[0] == ki ? 0 : (kv_chunk[1] == ki ? 1 : -1);
      if (slot < 0) {
        slot = next_kv;
        if (kv_free_set[slot]) CQSA_STEP(cudaStreamWaitEvent(copy, kv_free[slot], 0), "wait kv slot");
        tspan(cspans, copy, true);
        CQSA_STEP(copy_chunk(ksl[slot].k, k, CQSA_LAYOUT_BHND, B, H, N, d, ks, nk, h2d, copy, &bytes), "copy k");
        CQSA_STEP(copy_chunk(ksl[slot].v, v, CQSA_LAYOUT_BHND, B, H, N, d, ks, nk, h2d, copy, &bytes), "copy v");
        tspan(cspans, copy, false);
        CQSA_STEP(cudaEventRecord(kv_ready[slot], copy), "record");
        kv_chunk[slot] = ki;
      }
      next_kv = slot ^ 1;  // the other slot is the next to refill
      CQSA_STEP(cudaStreamWaitEvent(stream, kv_ready[slot], 0), "wait kv");
      if (rc != CQSA_OK) break;
      BwdArgs a;
      memset(&a, 0, sizeof(a));
      a.q = Q.q;
      a.k = ksl[slot].k;
      a.v = ksl[slot].v;
      a.dout = Q.g;
      a.lse = Q.lse;
      a.dvec = Q.dvec;
      a.dq_acc = Q.dq;
      a.dk_acc = dk_acc0 + static_cast<size_t>(ki) * (chunk32 / 4);
      a.dv_acc = dv_acc0 + static_cast<size_t>(ki) * (chunk32 / 4);
      a.B = B;
      a.H = H;
      a.Nq = nq;
      a.Nkv = nk;
      a.d = d;
      a.q_off = qs;
      a.kv_off = ks;
      a.causal = causal != 0;
      a.scale = sc;
      a.dtype = dtype;
      tspan(kspans, stream, true);
      if (rc == CQSA_OK) rc = launch_attention_bwd_chunk(a, stream);
      tspan(kspans, stream, false);
      ++n_pairs;
      ++n_launches;
      CQSA_STEP(cudaEventRecord(kv_free[slot], stream), "record");
      kv_free_set[slot] = true;
    }
    write_out(Q.dq, dq, qs, nq);
    CQSA_STEP(cudaEventRecord(q_free[qi & 1], stream), "record");
    q_free_set[qi & 1] = true;
  }
  for (int ki = 0; ki < n_chunks && rc == CQSA_OK; ++ki) {
    const long long ks = static_cast<long long>(ki) * C;
    const int nk = static_cast<int>(N - ks < C ? N - ks : C);
    write_out(dk_acc0 + static_cast<size_t>(ki) * (chunk32 / 4), dk, ks, nk);
    write_out(dv_acc0 + static_cast<size_t>(ki) * (chunk32 / 4), dv, ks, nk);
  }
  // every use of the buffers is complete before they return to the pool
  cudaError_t se = cudaStreamSynchronize(stream);
  if (rc == CQSA_OK) rc = cuda_status(se, "synchronize");
  if (copy) {
    se = cudaStreamSynchronize(copy);
    if (rc == CQSA_OK) rc = cuda_status(se, "synchronize copy stream");
  }
  if (d2h) {
    se = cudaStreamSynchronize(d2h);
    if (rc == CQSA_OK) rc = cuda_status(se, "synchronize output stream");
  }
  // a kernel whose bounded wait gave up leaves its gradients incomplete: report it
  if (rc == CQSA_OK) rc = check_device_error_on(stream);
  if (rc == CQSA_OK && stats) {
    double comp = 0.0, h2d = 0.0, stall = 0.0;
    float ms = 0.0f;
    for (size_t i = 0; i < kspans.size(); ++i) {
      if (cudaEventElapsedTime(&ms, kspans[i].a, kspans[i].b) == cudaSuccess) comp += ms;
      if (i > 0 && cudaEventElapsedTime(&ms, kspans[i - 1].b, kspans[i].a) == cudaSuccess && ms > 0) stall += ms;
    }
    for (const Span& s : cspans)
      if (cudaEventElapsedTime(&ms, s.a, s.b) == cudaSuccess) h2d += ms;
    stats->compute_ms = comp;
    stats->h2d_ms = h2d;
    stats->stall_ms = stall;
    stats->h2d_bytes = bytes;
    stats->d2h_bytes = d2h_bytes;
    stats->peak_device_bytes = dev_bytes;
    stats->n_chunks = n_pairs;
    stats->n_launches = n_launches;
  }
  for (cudaEvent_t e : tevents) pool_event_free(e, true);
  for (cudaEvent_t e : events) pool_event_free(e, false);
  pool_stream_free(copy);
  pool_stream_free(d2h);
  for (void* b : bufs) pool_free(b);
  if (rc == CQSA_OK && stats)
    stats->wall_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_start).count();
  return rc;
}
