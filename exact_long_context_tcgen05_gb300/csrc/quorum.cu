// Cyclic quorum-set decomposition of exact attention ("stream-cqsa 2.2.0 -> 2.2.2" diff: README and
// `autoconfig.plan`, where a configuration is (c, interest_set, itr) with c**itr subproblems and
// cost (l^2/c)^itr, l = |interest_set|; the default set is (0, 1, 3) at c = 7).
//
// Reading used here (the pages name the parameters and the costs but not the construction):
//   * the sequence is cut into T = c^itr chunks of C tokens (C a multiple of 128, the last chunk
//     ragged); chunk t has base-c digits t_0 .. t_{itr-1};
//   * subproblem s (digits s_e) owns the l^itr chunks t with t_e in s_e + D (mod c) for every e,
//     D the interest set; each subproblem therefore holds l^itr of the T chunks, and running every
//     subproblem in full would cost c^itr (l^itr C)^2 = (l^2/c)^itr N^2 score entries;
//   * D must be a perfect difference set modulo c (its l(l-1) ordered differences cover every non-zero
//     residue once, so c = l(l-1) + 1): then two chunks with digits q_e != k_e share exactly one
//     s_e, and every (query chunk, key chunk) pair meets in at least one subproblem;
//   * each needed pair (q, k) (k <= q when causal) is computed exactly once, in the subproblem whose
//     digit e is the unique shared one where q_e != k_e and q_e - D[0] where q_e = k_e; its partial
//     (O, LSE) is merged into query chunk q's fp32 accumulator, so the result is the exact attention
//     whatever the order of the subproblems.
// A subproblem needs only its own chunks on the device: the executor stages Q and K/V chunks through
// two sets of l^itr slots (the previous subproblem's chunks stay while the next ones load) and keeps
// one fp32 accumulator per query chunk on the device, or, with the host accumulator (the pages'
// `accumulate_on_gpu=False`), in pinned host memory: a query chunk's accumulator then travels with
// its Q slot (copied in when the chunk is staged, written back when the slot is reused), so device
// memory stays at the slots whatever the sequence length.
// Parallel subproblem lanes (the pages' `max_parallel`): chunk pairs of different query chunks are
// independent, so pair (q, k) runs on compute stream q mod n_par; pairs of one query chunk stay in
// one stream, in schedule order, so the accumulation order (and the result, bit for bit) does not
// depend on n_par. Small chunk pairs, whose grids do not fill the GPU, then run side by side.
#include <algorithm>
#include <chrono>
#include <math.h>
#include <string.h>
#include <vector>

#include "cqsa_internal.h"

namespace cqsa {
namespace {

constexpr int kMaxQuorumChunks = 1 << 16;  // c^itr
constexpr int kMaxWavePairsLaunch = 32;     // pairs in one multi-pair launch (launch_attention_multi)

struct Triple {
  int s, q, k;
};

bool ipow_bounded(int c, int itr, int limit, int* out) {
  long long v = 1;
  for (int e = 0; e < itr; ++e) {
    v *= c;
    if (v > limit) return false;
  }
  *out = static_cast<int>(v);
  return true;
}

// CQSA_OK if D (l distinct residues in [0, c)) is a perfect difference set modulo c.
int check_set(int c, const int* D, int l) {
  if (c < 1 || l < 1 || !D) {
    set_error("quorum set: c and l must be positive and interest_set non-null");
    return CQSA_ERR_INVALID;
  }
  if (static_cast<long long>(l) * (l - 1) + 1 != c) {
    set_error("quorum set: a perfect difference set of %d residues needs c = %d (got c = %d)", l, l * (l - 1) + 1, c);
    return CQSA_ERR_INVALID;
  }
  std::vector<int> seen(c, 0);
  for (int i = 0; i < l; ++i) {
    if (D[i] < 0 || D[i] >= c) {
      set_error("quorum set: element %d is outside [0, %d)", D[i], c);
      return CQSA_ERR_INVALID;
    }
    for (int j = 0; j < l; ++j) {
      if (i == j) continue;
      const int delta = ((D[j] - D[i]) % c + c) % c;
      if (delta == 0) {
        set_error("quorum set: repeated element %d", D[i]);
        return CQSA_ERR_INVALID;
      }
      if (++seen[delta] > 1) {
        set_error("quorum set: difference %d occurs more than once (not a perfect difference set mod %d)", delta, c);
        return CQSA_ERR_INVALID;
      }
    }
  }
  return CQSA_OK;
}

// Every needed (q, k) chunk pair with the subproblem that computes it, sorted by (s, q, k).
int build_schedule(int c, const int* D, int l, int itr, int n_chunks, bool causal, std::vector<Triple>* out) {
  int rc = check_set(c, D, l);
  if (rc != CQSA_OK) return rc;
  int T = 0;
  if (itr < 1 || !ipow_bounded(c, itr, kMaxQuorumChunks, &T)) {
    set_error("quorum depth: need itr >= 1 and c^itr <= %d", kMaxQuorumChunks);
    return CQSA_ERR_UNSUPPORTED;
  }
  if (n_chunks < 0 || n_chunks > T) {
    set_error("quorum schedule: %d non-empty chunks for %d chunk slots", n_chunks, T);
    return CQSA_ERR_INVALID;
  }
  // For a non-zero digit difference delta = k_e - q_e, the index i of the set element that q_e
  // stands at in the shared subproblem: D[j] - D[i] = delta for exactly one (i, j).
  std::vector<int> first_of(c, -1);
  for (int i = 0; i < l; ++i)
    for (int j = 0; j < l; ++j)
      if (i != j) first_of[((D[j] - D[i]) % c + c) % c] = i;
  out->clear();
  for (int q = 0; q < n_chunks; ++q) {
    const int kmax = causal ? q : n_chunks - 1;
    for (int k = 0; k <= kmax; ++k) {
      int s = 0, place = 1, qq = q, kk = k;
      for (int e = 0; e < itr; ++e) {
        const int qe = qq % c, ke = kk % c;
        qq /= c;
        kk /= c;
        const int base = (qe == ke) ? D[0] : D[first_of[((ke - qe) % c + c) % c]];
        s += (((qe - base) % c + c) % c) * place;
        place *= c;
      }
      out->push_back({s, q, k});
    }
  }
  std::stable_sort(out->begin(), out->end(), [](const Triple& a, const Triple& b) { return a.s < b.s; });
  return CQSA_OK;
}

// Device buffers, events and streams come from the library's pool and go back once the streams
// that use them have drained; the pinned host accumulator is allocated per call.
struct Resources {
  std::vector<void*> dev;
  std::vector<void*> host;  // pinned host allocations (cudaHostAlloc)
  std::vector<std::pair<cudaEvent_t, bool>> events;
  std::vector<cudaStream_t> lanes;  // extra compute streams (parallel subproblem lanes)
  cudaStream_t copy = nullptr;
  cudaStream_t compute = nullptr;
  ~Resources() {
    if (compute) cudaStreamSynchronize(compute);
    for (cudaStream_t s : lanes) cudaStreamSynchronize(s);
    if (copy) cudaStreamSynchronize(copy);
    for (void* p : dev) pool_free(p);
    for (void* p : host) cudaFreeHost(p);
    for (const auto& e : events) pool_event_free(e.first, e.second);
    for (cudaStream_t s : lanes) pool_stream_free(s);
    pool_stream_free(copy);
  }
};

}  // namespace
}  // namespace cqsa

using namespace cqsa;

extern "C" int cqsa_quorum_check(int c, const int* interest_set, int l) { return check_set(c, interest_set, l); }

extern "C" long long cqsa_quorum_schedule(int c, const int* interest_set, int l, int itr, int n_chunks, int causal,
                                          int* out, long long max_triples) {
  std::vector<Triple> tr;
  const int rc = build_schedule(c, interest_set, l, itr, n_chunks, causal != 0, &tr);
  if (rc != CQSA_OK) return rc;
  if (out) {
    if (max_triples < static_cast<long long>(tr.size())) {
      set_error("quorum schedule: %zu triples do not fit in %lld", tr.size(), max_triples);
      return CQSA_ERR_INVALID;
    }
    for (size_t i = 0; i < tr.size(); ++i) {
      out[3 * i + 0] = tr[i].s;
      out[3 * i + 1] = tr[i].q;
      out[3 * i + 2] = tr[i].k;
    }
  }
  return static_cast<long long>(tr.size());
}

extern "C" int cqsa_quorum_attn_fwd(const void* q, const void* k, const void* v, int layout, int inputs_on_host,
                                    void* out, float* lse, int out_on_host, int B, int H, long long N, int d,
                                    int causal, float scale, int dtype, int c, const int* interest_set, int l,
                                    int itr, int acc_on_host, int max_parallel, cqsa_quorum_stats* stats,
                                    cudaStream_t stream) {
  return cqsa_quorum_attn_fwd_ex(q, k, v, layout, inputs_on_host, out, lse, out_on_host, B, H, N, d, causal, scale,
                                 dtype, c, interest_set, l, itr, acc_on_host, max_parallel, CQSA_ENGINE_CLASSIC, 0,
                                 stats, stream);
}

extern "C" int cqsa_quorum_attn_fwd_ex(const void* q, const void* k, const void* v, int layout, int inputs_on_host,
                                       void* out, float* lse, int out_on_host, int B, int H, long long N, int d,
                                       int causal, float scale, int dtype, int c, const int* interest_set, int l,
                                       int itr, int acc_on_host, int max_parallel, int engine, long long wave_tokens,
                                       cqsa_quorum_stats* stats, cudaStream_t stream) {
  const auto t_start = std::chrono::steady_clock::now();
  if (stats) memset(stats, 0, sizeof(*stats));
  if (!q || !k || !v || !out) {
    set_error("q, k, v and out must be non-null");
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
  if (!isfinite(scale) || scale < 0.0f) {
    set_error("scale must be finite and >= 0 (0 selects 1/sqrt(d))");
    return CQSA_ERR_INVALID;
  }
  if (max_parallel < 1 || max_parallel > 16) {
    set_error("max_parallel must be in [1, 16] (got %d)", max_parallel);
    return CQSA_ERR_INVALID;
  }
  if (engine != CQSA_ENGINE_CLASSIC && engine != CQSA_ENGINE_WAVE) {
    set_error("engine must be CQSA_ENGINE_CLASSIC or CQSA_ENGINE_WAVE (got %d)", engine);
    return CQSA_ERR_INVALID;
  }
  if (wave_tokens < 0) {
    set_error("wave_tokens must be >= 0 (0 selects min(2^21, max(2^19, N)))");
    return CQSA_ERR_INVALID;
  }
  const bool wave = engine == CQSA_ENGINE_WAVE;
  // Device-resident inputs are read in place (each chunk is a token range of the caller's tensors, which
  // the tensor maps address with the full tensors' strides): nothing is staged, only the bookkeeping of
  // the Q slots remains (the host accumulator travels with them).
  const bool in_place = !inputs_on_host;
  int T = 0;
  if (itr < 1 || c < 1 || !ipow_bounded(c, itr, kMaxQuorumChunks, &T)) {
    set_error("quorum depth: need c >= 1, itr >= 1 and c^itr <= %d", kMaxQuorumChunks);
    return CQSA_ERR_UNSUPPORTED;
  }
  const long long per = (N + T - 1) / T;
  const long long C = ((per + 127) / 128) * 128;
  const int nne = static_cast<int>((N + C - 1) / C);  // non-empty chunks
  if (static_cast<long long>(B) * H * C > (1LL << 31) - 1) {
    set_error("B*H*chunk too large for one chunk launch");
    return CQSA_ERR_UNSUPPORTED;
  }
  std::vector<Triple> sched;
  int rc = build_schedule(c, interest_set, l, itr, nne, causal != 0, &sched);
  if (rc != CQSA_OK) return rc;
  int per_sub = 1;
  for (int e = 0; e < itr; ++e) per_sub *= l;
  const int nslots = std::min(2 * per_sub, nne);
  const float sc = scale == 0.0f ? 1.0f / sqrtf(static_cast<float>(d)) : scale;
  const size_t es = 2;
  const size_t chunk_elems = static_cast<size_t>(B) * H * C * d;
  const size_t rows = static_cast<size_t>(B) * H * C;
  const cudaMemcpyKind kind = inputs_on_host ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;

  Resources res;
  res.compute = stream;
  long long dev_bytes = 0;
  auto alloc = [&](void** p, size_t n) -> int {
    const int r = pool_alloc(p, n);
    if (r != CQSA_OK) return r;
    res.dev.push_back(*p);
    dev_bytes += static_cast<long long>(n);
    return CQSA_OK;
  };
  auto event = [&](cudaEvent_t* e, bool timing) -> int {
    const int r = pool_event(e, timing);
    if (r != CQSA_OK) return r;
    res.events.push_back({*e, timing});
    return CQSA_OK;
  };
  std::vector<void*> qs(nslots), ks(nslots), vs(nslots);
  for (int s = 0; rc == CQSA_OK && !in_place && s < nslots; ++s) {
    rc = alloc(&qs[s], chunk_elems * es);
    if (rc == CQSA_OK) rc = alloc(&ks[s], chunk_elems * es);
    if (rc == CQSA_OK) rc = alloc(&vs[s], chunk_elems * es);
  }
  // Accumulators: one per query chunk on the device, or one per Q slot on the device backed by one
  // per query chunk in pinned host memory.
  const int nacc = acc_on_host ? nslots : nne;
  void *acc = nullptr, *lacc = nullptr, *ostage = nullptr, *lstage = nullptr;
  float *hacc = nullptr, *hlacc = nullptr;
  if (rc == CQSA_OK) rc = alloc(&acc, static_cast<size_t>(nacc) * chunk_elems * 4);
  if (rc == CQSA_OK) rc = alloc(&lacc, static_cast<size_t>(nacc) * rows * 4);
  if (rc == CQSA_OK && acc_on_host) {
    void* p = nullptr;
    cudaError_t e = cudaHostAlloc(&p, static_cast<size_t>(nne) * (chunk_elems + rows) * 4, cudaHostAllocDefault);
    if (e != cudaSuccess) {
      cudaGetLastError();
      set_error("pinned host allocation of the accumulator failed: %s", cudaGetErrorString(e));
      return e == cudaErrorMemoryAllocation ? CQSA_ERR_OOM : CQSA_ERR_CUDA;
    }
    res.host.push_back(p);
    hacc = static_cast<float*>(p);
    hlacc = hacc + static_cast<size_t>(nne) * chunk_elems;
  }
  if (rc == CQSA_OK && out_on_host) {
    rc = alloc(&ostage, chunk_elems * es);
    if (rc == CQSA_OK && lse) rc = alloc(&lstage, rows * 4);
  }
  if (rc != CQSA_OK) return rc;
  if ((rc = pool_stream(&res.copy)) != CQSA_OK) return rc;
  const int npar = wave ? 1 : max_parallel;  // the wave engine runs on the caller's stream alone
  // Pairs per wave launch: the token budget in query tokens (default min(2^21, max(2^19, N))) over C,
  // and at most the launch's table size.
  const long long wt = wave_tokens > 0 ? wave_tokens : std::min(1LL << 21, std::max(1LL << 19, N));
  const size_t wave_pairs = static_cast<size_t>(std::max(1LL, std::min(static_cast<long long>(kMaxWavePairsLaunch), wt / C)));
  std::vector<cudaStream_t> lane(npar, stream);
  for (int j = 1; j < npar; ++j) {
    cudaStream_t sj = nullptr;
    if ((rc = pool_stream(&sj)) != CQSA_OK) return rc;
    res.lanes.push_back(sj);
    lane[j] = sj;
  }
  // ready: the slot's staging copy is done; free[slot * npar + j]: lane j's last kernel reading the slot.
  std::vector<cudaEvent_t> q_ready(nslots), kv_ready(nslots), q_free(nslots * npar), kv_free(nslots * npar);
  for (int s = 0; s < nslots; ++s) {
    if ((rc = event(&q_ready[s], false)) != CQSA_OK || (rc = event(&kv_ready[s], false)) != CQSA_OK) return rc;
    for (int j = 0; j < npar; ++j)
      if ((rc = event(&q_free[s * npar + j], false)) != CQSA_OK || (rc = event(&kv_free[s * npar + j], false)) != CQSA_OK)
        return rc;
  }
  cudaEvent_t joined = nullptr;
  if ((rc = event(&joined, false)) != CQSA_OK) return rc;
  struct Span {
    cudaEvent_t a, b;
  };
  std::vector<Span> copies, kernels;
  auto span = [&](std::vector<Span>& vv, Span* sp) -> int {
    int r = event(&sp->a, true);
    if (r == CQSA_OK) r = event(&sp->b, true);
    if (r == CQSA_OK) vv.push_back(*sp);
    return r;
  };
#define CK(call, what)                     \
  do {                                     \
    int _r = cuda_status((call), what);    \
    if (_r != CQSA_OK) return _r;          \
  } while (0)

  auto ntok = [&](int chunk) -> int { return static_cast<int>(std::min(C, N - static_cast<long long>(chunk) * C)); };
  struct Pool {
    std::vector<int> chunk;     // chunk held by each slot (-1: none)
    std::vector<int> last_use;  // subproblem group of the last use
    std::vector<bool> used;     // [slot * npar + lane]: a kernel of that lane has read the slot
  };
  Pool qp{std::vector<int>(nslots, -1), std::vector<int>(nslots, -1), std::vector<bool>(nslots * npar, false)};
  Pool kp = qp;
  long long copy_bytes = 0;
  int loads = 0, groups = 0, launches = 0;
  std::vector<bool> started(nne, false);
  long long acc_bytes = 0;
  // Device accumulator of query chunk qc in Q slot sq.
  auto dacc = [&](int qc, int sq) -> float* {
    return static_cast<float*>(acc) + static_cast<size_t>(acc_on_host ? sq : qc) * chunk_elems;
  };
  auto dlacc = [&](int qc, int sq) -> float* {
    return static_cast<float*>(lacc) + static_cast<size_t>(acc_on_host ? sq : qc) * rows;
  };
  // Host accumulator: copy a chunk's accumulator between its host home and a device slot.
  auto acc_copy = [&](int qc, int sq, bool to_host, cudaStream_t s) -> int {
    float* h = hacc + static_cast<size_t>(qc) * chunk_elems;
    float* hl = hlacc + static_cast<size_t>(qc) * rows;
    const size_t n = static_cast<size_t>(B) * H * ntok(qc);
    int r = cuda_status(cudaMemcpyAsync(to_host ? static_cast<void*>(h) : static_cast<void*>(dacc(qc, sq)),
                                        to_host ? static_cast<void*>(dacc(qc, sq)) : static_cast<void*>(h),
                                        n * d * 4, to_host ? cudaMemcpyDeviceToHost : cudaMemcpyHostToDevice, s),
                        "accumulator copy");
    if (r == CQSA_OK)
      r = cuda_status(cudaMemcpyAsync(to_host ? static_cast<void*>(hl) : static_cast<void*>(dlacc(qc, sq)),
                                      to_host ? static_cast<void*>(dlacc(qc, sq)) : static_cast<void*>(hl), n * 4,
                                      to_host ? cudaMemcpyDeviceToHost : cudaMemcpyHostToDevice, s),
                      "accumulator copy");
    acc_bytes += static_cast<long long>(n) * (d + 1) * 4;
    return r;
  };

  // Slot of `chunk` in `pool` (*slot), staging it on the copy stream (after the slot's previous reader)
  // if absent. `keep` lists chunks the current subproblem needs, which are never evicted.
  auto stage = [&](Pool& pool, bool is_q, int chunk, int group, const std::vector<int>& keep, int* slot) -> int {
    for (int s = 0; s < nslots; ++s)
      if (pool.chunk[s] == chunk) {
        pool.last_use[s] = group;
        *slot = s;
        return CQSA_OK;
      }
    int victim = -1;
    for (int s = 0; s < nslots; ++s) {
      if (pool.chunk[s] >= 0 && std::find(keep.begin(), keep.end(), pool.chunk[s]) != keep.end()) continue;
      if (victim < 0 || pool.chunk[s] < 0 ||
          (pool.chunk[victim] >= 0 && pool.last_use[s] < pool.last_use[victim]))
        victim = s;
      if (pool.chunk[victim] < 0) break;
    }
    if (victim < 0) {  // cannot happen: a subproblem needs at most l^itr <= nslots chunks
      set_error("quorum executor: no free chunk slot");
      return CQSA_ERR_INVALID;
    }
    int r = CQSA_OK;
    for (int j = 0; j < npar; ++j)
      if (pool.used[victim * npar + j] &&
          (r = cuda_status(cudaStreamWaitEvent(res.copy, is_q ? q_free[victim * npar + j] : kv_free[victim * npar + j], 0),
                           "wait slot")) != CQSA_OK)
        return r;
    Span sp;
    if ((r = span(copies, &sp)) != CQSA_OK) return r;
    const long long t0 = static_cast<long long>(chunk) * C;
    const int n = ntok(chunk);
    if ((r = cuda_status(cudaEventRecord(sp.a, res.copy), "record")) != CQSA_OK) return r;
    if (is_q) {
      if (acc_on_host && pool.chunk[victim] >= 0 && started[pool.chunk[victim]] &&
          (r = acc_copy(pool.chunk[victim], victim, true, res.copy)) != CQSA_OK)
        return r;
      if (!in_place)
        r = cuda_status(copy_chunk(qs[victim], q, layout, B, H, N, d, t0, n, kind, res.copy, &copy_bytes),
                        "copy Q chunk");
      if (r == CQSA_OK && acc_on_host && started[chunk]) r = acc_copy(chunk, victim, false, res.copy);
    } else if (!in_place) {
      r = cuda_status(copy_chunk(ks[victim], k, layout, B, H, N, d, t0, n, kind, res.copy, &copy_bytes), "copy K chunk");
      if (r == CQSA_OK)
        r = cuda_status(copy_chunk(vs[victim], v, layout, B, H, N, d, t0, n, kind, res.copy, &copy_bytes),
                        "copy V chunk");
    }
    if (r != CQSA_OK) return r;
    if ((r = cuda_status(cudaEventRecord(sp.b, res.copy), "record")) != CQSA_OK) return r;
    if ((r = cuda_status(cudaEventRecord(is_q ? q_ready[victim] : kv_ready[victim], res.copy), "record ready")) !=
        CQSA_OK)
      return r;
    pool.chunk[victim] = chunk;
    pool.last_use[victim] = group;
    if (!in_place || is_q) ++loads;
    *slot = victim;
    return CQSA_OK;
  };

  // Wave launches of a list of pairs (waves: see the header of cqsa_quorum_attn_fwd_ex).
  struct Pending {
    AttnArgs a;
    int sq, sk, q;
    std::vector<int> sks;  // key slots of every pair fused into this one
  };
  auto launch_waves = [&](std::vector<Pending>& group_pairs) -> int {
    int rc = CQSA_OK;
    if (in_place) {
      // Pairs of one query chunk whose key chunks are adjacent read one contiguous key range of the
      // caller's tensors: they run as one pair over the whole range. The online softmax over the
      // concatenated keys is the exact merge of the parts, and a CTA walks more key tiles for its fixed
      // cost, with fewer passes over the accumulator. The first of a chunk's pairs that runs writes the
      // accumulator (when this group starts the chunk), the rest merge into it.
      std::vector<Pending> fused;
      std::vector<int> qorder;
      for (const Pending& pd : group_pairs)
        if (std::find(qorder.begin(), qorder.end(), pd.q) == qorder.end()) qorder.push_back(pd.q);
      for (int qc : qorder) {
        std::vector<const Pending*> mine;
        bool starts = false;
        for (const Pending& pd : group_pairs)
          if (pd.q == qc) {
            mine.push_back(&pd);
            starts = starts || pd.a.mode == kModePart;
          }
        std::stable_sort(mine.begin(), mine.end(),
                         [](const Pending* x, const Pending* y) { return x->a.kv_off < y->a.kv_off; });
        bool first = true;
        for (size_t m = 0; m < mine.size();) {
          Pending f = *mine[m];
          f.sks.assign(1, mine[m]->sk);
          size_t e = m + 1;
          while (e < mine.size() && mine[e]->a.kv_off == f.a.kv_off + f.a.Nkv &&
                 static_cast<long long>(f.a.Nkv) + mine[e]->a.Nkv <= 0x7fffffffLL) {
            f.a.Nkv += mine[e]->a.Nkv;
            f.sks.push_back(mine[e]->sk);
            ++e;
          }
          f.a.mode = (first && starts) ? kModePart : kModeAccum;
          first = false;
          fused.push_back(f);
          m = e;
        }
      }
      group_pairs.swap(fused);
    }
    // Waves: one launch takes at most one pair of each query chunk (pairs of one chunk accumulate into
    // one buffer, in schedule order, wave after wave) and at most wave_pairs pairs in all. Pairs with a
    // full key chunk come first in a launch, the (lighter) diagonal pairs last.
    std::vector<int> qlist;
    std::vector<std::vector<size_t>> byq;
    for (size_t i = 0; i < group_pairs.size(); ++i) {
      const int qc = group_pairs[i].q;
      size_t pos = std::find(qlist.begin(), qlist.end(), qc) - qlist.begin();
      if (pos == qlist.size()) {
        qlist.push_back(qc);
        byq.emplace_back();
      }
      byq[pos].push_back(i);
    }
    size_t depth = 0;
    for (const auto& v_ : byq) depth = std::max(depth, v_.size());
    for (size_t w = 0; w < depth; ++w) {
      std::vector<size_t> members;
      for (const auto& v_ : byq)
        if (w < v_.size()) members.push_back(v_[w]);
      std::stable_sort(members.begin(), members.end(), [&](size_t x, size_t y) {
        const AttnArgs& ax = group_pairs[x].a;
        const AttnArgs& ay = group_pairs[y].a;
        const bool fx = !causal || ax.kv_off + ax.Nkv <= ax.q_off + 1;
        const bool fy = !causal || ay.kv_off + ay.Nkv <= ay.q_off + 1;
        if (fx != fy) return fx;
        return ax.Nkv > ay.Nkv;  // then the longest key ranges first
      });
      for (size_t m0 = 0; m0 < members.size(); m0 += wave_pairs) {
        const size_t m1 = std::min(members.size(), m0 + wave_pairs);
        std::vector<AttnArgs> batch;
        for (size_t m = m0; m < m1; ++m) {
          const Pending& pd = group_pairs[members[m]];
          CK(cudaStreamWaitEvent(stream, q_ready[pd.sq], 0), "wait q_ready");
          for (int sk : pd.sks) CK(cudaStreamWaitEvent(stream, kv_ready[sk], 0), "wait kv_ready");
          batch.push_back(pd.a);
        }
        Span sp;
        if ((rc = span(kernels, &sp)) != CQSA_OK) return rc;
        CK(cudaEventRecord(sp.a, stream), "record");
        if ((rc = launch_attention_multi(batch.data(), static_cast<int>(batch.size()), stream)) != CQSA_OK) return rc;
        CK(cudaEventRecord(sp.b, stream), "record");
        for (size_t m = m0; m < m1; ++m) {
          const Pending& pd = group_pairs[members[m]];
          CK(cudaEventRecord(q_free[pd.sq * npar], stream), "record q_free");
          qp.used[pd.sq * npar] = true;
          for (int sk : pd.sks) {
            CK(cudaEventRecord(kv_free[sk * npar], stream), "record kv_free");
            kp.used[sk * npar] = true;
          }
        }
        ++launches;
      }
    }
    group_pairs.clear();
    return CQSA_OK;
  };
  // Device-resident inputs without the host accumulator: every chunk is always at hand, so a wave may
  // take pairs of every subproblem (one launch holds the w-th pair, in schedule order, of each query chunk).
  const bool global_waves = wave && in_place && !acc_on_host;
  std::vector<Pending> group_pairs;

  size_t i0 = 0;
  while (i0 < sched.size()) {
    size_t i1 = i0;
    while (i1 < sched.size() && sched[i1].s == sched[i0].s) ++i1;
    std::vector<int> needq, needk;
    for (size_t i = i0; i < i1; ++i) {
      if (std::find(needq.begin(), needq.end(), sched[i].q) == needq.end()) needq.push_back(sched[i].q);
      if (std::find(needk.begin(), needk.end(), sched[i].k) == needk.end()) needk.push_back(sched[i].k);
    }
    // Chunk pointers: the staged slot, or the token range of the caller's device tensors.
    auto chunk_ptr = [&](const void* base, const std::vector<void*>& slots, int slot, int chunk) -> const void* {
      if (!in_place) return slots[slot];
      const long long t0 = static_cast<long long>(chunk) * C;
      const size_t off = layout == CQSA_LAYOUT_BHND ? static_cast<size_t>(t0) * d * es
                                                    : static_cast<size_t>(t0) * H * d * es;
      return static_cast<const char*>(base) + off;
    };
    for (size_t i = i0; i < i1; ++i) {
      const Triple& t = sched[i];
      int sq = -1, sk = -1;
      if ((rc = stage(qp, true, t.q, groups, needq, &sq)) != CQSA_OK) return rc;
      if ((rc = stage(kp, false, t.k, groups, needk, &sk)) != CQSA_OK) return rc;
      AttnArgs a;
      memset(&a, 0, sizeof(a));
      a.q = chunk_ptr(q, qs, sq, t.q);
      a.k = chunk_ptr(k, ks, sk, t.k);
      a.v = chunk_ptr(v, vs, sk, t.k);
      if (in_place) {
        a.q_tokens_alloc = N;
        a.kv_tokens_alloc = N;
      }
      a.B = B;
      a.H = H;
      a.Nq = ntok(t.q);
      a.Nkv = ntok(t.k);
      a.q_off = static_cast<long long>(t.q) * C;
      a.kv_off = static_cast<long long>(t.k) * C;
      a.d = d;
      a.causal = causal != 0;
      a.scale = sc;
      a.dtype = dtype;
      a.in_layout = layout;
      a.mode = started[t.q] ? kModeAccum : kModePart;
      a.o_part = dacc(t.q, sq);
      a.lse_part = dlacc(t.q, sq);
      a.out_layout = CQSA_LAYOUT_BHND;
      started[t.q] = true;
      if (wave) {
        group_pairs.push_back({a, sq, sk, t.q, {sk}});
        continue;
      }
      const int j = t.q % npar;
      cudaStream_t ls = lane[j];
      CK(cudaStreamWaitEvent(ls, q_ready[sq], 0), "wait q_ready");
      CK(cudaStreamWaitEvent(ls, kv_ready[sk], 0), "wait kv_ready");
      Span sp;
      if ((rc = span(kernels, &sp)) != CQSA_OK) return rc;
      CK(cudaEventRecord(sp.a, ls), "record");
      if ((rc = launch_attention(a, ls)) != CQSA_OK) return rc;
      CK(cudaEventRecord(sp.b, ls), "record");
      CK(cudaEventRecord(q_free[sq * npar + j], ls), "record q_free");
      CK(cudaEventRecord(kv_free[sk * npar + j], ls), "record kv_free");
      qp.used[sq * npar + j] = true;
      kp.used[sk * npar + j] = true;
      ++launches;
    }
    if (wave && !global_waves && (rc = launch_waves(group_pairs)) != CQSA_OK) return rc;
    ++groups;
    i0 = i1;
  }

  if (global_waves && (rc = launch_waves(group_pairs)) != CQSA_OK) return rc;

  // Every lane's kernels finish before the caller's stream finalizes.
  for (int j = 1; j < npar; ++j) {
    CK(cudaEventRecord(joined, lane[j]), "record join");
    CK(cudaStreamWaitEvent(stream, joined, 0), "wait join");
  }

  // Finalize every query chunk into the output (device), or through a staging buffer to the host.
  // With the host accumulator, chunks still in a Q slot are finalized from it first; every other
  // chunk's accumulator is then copied into slot 0 (stream-ordered after the previous finalize).
  std::vector<int> order, slot_of(nne, -1);
  if (acc_on_host) {
    CK(cudaStreamSynchronize(res.copy), "synchronize copy stream");
    for (int s = 0; s < nslots; ++s)
      if (qp.chunk[s] >= 0) slot_of[qp.chunk[s]] = s;
    for (int qc = 0; qc < nne; ++qc)
      if (slot_of[qc] >= 0) order.push_back(qc);
    for (int qc = 0; qc < nne; ++qc)
      if (slot_of[qc] < 0) order.push_back(qc);
  } else {
    for (int qc = 0; qc < nne; ++qc) order.push_back(qc);
  }
  for (int qc : order) {
    const int n = ntok(qc);
    const long long t0 = static_cast<long long>(qc) * C;
    int sq = slot_of[qc];
    if (acc_on_host && sq < 0) {
      sq = 0;
      if ((rc = acc_copy(qc, sq, false, stream)) != CQSA_OK) return rc;
    }
    const float* accq = dacc(qc, sq);
    const float* laccq = dlacc(qc, sq);
    if (!out_on_host) {
      if ((rc = launch_finalize(accq, laccq, out, lse, B, H, n, N, t0, d, layout, dtype, stream)) != CQSA_OK) return rc;
    } else {
      if ((rc = launch_finalize(accq, laccq, ostage, static_cast<float*>(lstage), B, H, n, n, 0, d, layout, dtype,
                                stream)) != CQSA_OK)
        return rc;
      size_t width, height, dpitch;
      char* obase = static_cast<char*>(out);
      if (layout == CQSA_LAYOUT_BHND) {
        width = static_cast<size_t>(n) * d * es;
        height = static_cast<size_t>(B) * H;
        dpitch = static_cast<size_t>(N) * d * es;
        obase += static_cast<size_t>(t0) * d * es;
      } else {
        width = static_cast<size_t>(n) * H * d * es;
        height = static_cast<size_t>(B);
        dpitch = static_cast<size_t>(N) * H * d * es;
        obase += static_cast<size_t>(t0) * H * d * es;
      }
      if (height == 1 || dpitch == width)
        CK(cudaMemcpyAsync(obase, ostage, width * height, cudaMemcpyDeviceToHost, stream), "D2H out");
      else
        CK(cudaMemcpy2DAsync(obase, dpitch, ostage, width, width, height, cudaMemcpyDeviceToHost, stream), "D2H out");
      if (lse) {
        const size_t lw = static_cast<size_t>(n) * 4;
        CK(cudaMemcpy2DAsync(lse + t0, static_cast<size_t>(N) * 4, lstage, lw, lw, static_cast<size_t>(B) * H,
                             cudaMemcpyDeviceToHost, stream),
           "D2H lse");
      }
    }
    ++launches;
  }
  CK(cudaStreamSynchronize(stream), "synchronize compute stream");
  CK(cudaStreamSynchronize(res.copy), "synchronize copy stream");
  {
    // the call's own streams have drained; read the device error words on the compute stream
    int r = check_device_error_on(stream);
    if (r != CQSA_OK) return r;
  }
#undef CK
  if (stats) {
    double cp = 0.0, comp = 0.0;
    float ms = 0.0f;
    for (const Span& s : copies)
      if (cudaEventElapsedTime(&ms, s.a, s.b) == cudaSuccess) cp += ms;
    for (const Span& s : kernels)
      if (cudaEventElapsedTime(&ms, s.a, s.b) == cudaSuccess) comp += ms;
    stats->copy_ms = cp;
    stats->compute_ms = comp;
    stats->copy_bytes = copy_bytes;
    stats->acc_host_bytes = acc_bytes;
    stats->peak_device_bytes = dev_bytes;
    stats->n_subproblems = groups;
    stats->n_pairs = static_cast<int>(sched.size());
    stats->n_chunk_loads = loads;
    stats->n_launches = launches;
    stats->chunk_tokens = C;
    stats->wall_ms =
        std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_start).count();
  }
  return CQSA_OK;
}
