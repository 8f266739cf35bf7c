/*
 * cqsa.h - exact scaled-dot-product attention forward (and its backward) on one NVIDIA GB300 (sm_103a).
 *
 * C ABI of libcqsa_gb300.so. Every pointer is owned by the caller: the library never frees or
 * keeps one after a call returns. Device calls are asynchronous and ordered on the given stream
 * (NULL = the legacy default stream); cqsa_stream_attn_fwd is synchronous. Every entry point
 * validates all arguments before it launches anything, returns a cqsa_status and never aborts the
 * process; cqsa_last_error() gives a message for the calling thread's last failure.
 *
 * What is computed (the pages do not print the formula; this is the plain reading of their
 * statement that the call is a drop-in for torch's F.scaled_dot_product_attention - "stream-cqsa
 * 2.2.0 -> 2.2.2" diff, stream_cqsa/api.py, `attention` docstring - and that it is exact):
 *   for every (b, h) and query row i, over the allowed keys A_i = { j < Nkv : not causal or
 *   kv_pos(j) <= q_pos(i) },
 *     s_ij = scale * q_i . k_j,   out_i = sum_j softmax_j(s_ij) v_j,   lse_i = ln sum_j exp(s_ij).
 *   Causal masking is top-left aligned on absolute token positions. A row with no allowed key has
 *   out = 0 and lse = -inf.
 *
 * Shapes and types: Q/K/V are fp16 or bf16, head dimension d in {64, 128} (the pages' kernels
 * cover "fp16/bf16 and head dims 64/128": "stream-cqsa 2.2.2 -> 2.2.3" diff, README). Masks,
 * dropout and grouped-query attention are not part of this ABI, as the pages' call rejects them
 * ("stream-cqsa 2.2.0 -> 2.2.2" diff, api.py `attention` docstring). scale == 0 means 1/sqrt(d),
 * the SDPA default (`scale: Optional[float] = None` in the same signature).
 *
 * Layouts: CQSA_LAYOUT_BHND is SDPA's [B, H, N, d] (contiguous). CQSA_LAYOUT_BNHD is the
 * token-major [B, N, H, d] host layout the pages' streaming engine gathers from ("stream-cqsa
 * 2.2.2 -> 2.2.3" diff, api.py `_pinned_copy`). lse / LSE arrays are always [B, H, N] fp32.
 * All device pointers must be 16-byte aligned.
 */
#ifndef CQSA_H
#define CQSA_H

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CQSA_OK = 0,
  CQSA_ERR_INVALID = -1,     /* bad argument (null pointer, size, alignment, non-finite scale) */
  CQSA_ERR_UNSUPPORTED = -2, /* valid but not implemented (d not 64/128, dtype, layout) */
  CQSA_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
  CQSA_ERR_OOM = -4,         /* a device or pinned allocation failed: the caller may re-plan */
  CQSA_ERR_TIMEOUT = -5,     /* a device-side bounded wait gave up (see cqsa_device_error) */
  CQSA_ERR_DEVICE = -6       /* no usable sm_103 device, or a device-side condition other than a wait
                                (see cqsa_device_error) */
} cqsa_status;

typedef enum { CQSA_F16 = 0, CQSA_BF16 = 1, CQSA_F32 = 2 /* outputs only */ } cqsa_dtype;
typedef enum { CQSA_LAYOUT_BHND = 0, CQSA_LAYOUT_BNHD = 1 } cqsa_layout;

/*
 * Monolithic exact attention forward ("below the memory boundary the call is the monolithic
 * kernel": "stream-cqsa 2.2.2 -> 2.2.3" diff, api.py `_run`, mono branch).
 * q, k, v: device [B,H,N,d] of `dtype`. out: device [B,H,N,d] of `dtype` (RNE from fp32).
 * lse: device [B,H,N] fp32, natural log, or NULL if not wanted.
 */
int cqsa_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
                  int N, int d, int causal, float scale, int dtype, cudaStream_t stream);

/*
 * One chunk pair of the out-of-memory decomposition: queries of a Q block against the keys of a
 * KV block, giving a normalised fp32 partial output and its LSE ("partial outputs are merged into
 * an accumulator": "stream-cqsa 2.2.0 -> 2.2.2" diff, README profile sweep; the engine returns
 * `lse`: "stream-cqsa 2.2.2 -> 2.2.3" diff, oom_fallback.py `stream_cqsa_auto`).
 * q_blk: device [B,H,Nq,d]; k_blk, v_blk: device [B,H,Nkv,d]; q_off / kv_off: absolute position
 * of token 0 of each block (causal mask: key allowed iff kv_off + j <= q_off + i). Nkv may be 0.
 * O_part: device fp32 [B,H,Nq,d]; LSE_part: device fp32 [B,H,Nq].
 * accumulate = 0: O_part/LSE_part are overwritten with this pair's result (empty rows: 0 / -inf).
 * accumulate = 1: (O_part, LSE_part) hold a running (O_acc, LSE_acc) that this pair is merged
 * into exactly, in place (initialise LSE_acc to -inf; calls on one stream are race-free).
 */
int cqsa_attn_fwd_chunk(const void* q_blk, const void* k_blk, const void* v_blk, long long q_off,
                        long long kv_off, int B, int H, int Nq, int Nkv, int d, int causal, float scale,
                        int dtype, float* O_part, float* LSE_part, int accumulate, cudaStream_t stream);

/*
 * Exact merge of n partials over disjoint key sets:
 *   M = max_k LSE_k, lse = M + ln sum_k exp(LSE_k - M), out = sum_k exp(LSE_k - lse) O_k,
 * summed in the order k = 0 .. n-1 (deterministic). All-empty rows give out = 0, lse = -inf.
 * O_parts / LSE_parts: HOST arrays of n device pointers (1 <= n <= 1024) to fp32 [B,H,Nq,d] and
 * [B,H,Nq]. out: device [B,H,Nq,d] of out_dtype (F16, BF16 or F32); lse: device fp32 or NULL.
 */
int cqsa_merge_partials(const float* const* O_parts, const float* const* LSE_parts, int n, void* out,
                        float* lse, int B, int H, int Nq, int d, int out_dtype, cudaStream_t stream);

/* Statistics of one streaming call (times in milliseconds). */
typedef struct {
  double wall_ms;        /* host clock around the whole call */
  double compute_ms;     /* sum of chunk-kernel event intervals on the compute stream (resident
                            schedule: the union of its launches' intervals, which overlap) */
  double h2d_ms;         /* sum of host-to-device copy event intervals */
  double stall_ms;       /* time the compute stream waited for a copy (event gaps) */
  long long h2d_bytes;   /* bytes copied host -> device */
  long long d2h_bytes;   /* bytes copied device -> host */
  long long peak_device_bytes; /* device memory the driver allocated */
  int n_chunks;          /* Q chunks x KV chunks processed (non-empty pairs); resident schedule: Q chunks */
  int n_launches;        /* kernels launched */
} cqsa_stream_stats;

/*
 * Out-of-memory exact attention: Q/K/V stay in pinned (or pageable) host memory in `layout` and
 * are streamed to the device in chunks of chunk_tokens (a multiple of 128): for each Q chunk (two Q
 * buffers, so the next Q chunk arrives during the current one), the
 * K/V chunks it needs are double-buffered over the host link on a copy stream while the chunk
 * kernel merges each pair into an fp32 device accumulator ("stream_from_host", with per-subproblem
 * host transfers overlapping compute: "stream-cqsa 2.2.0 -> 2.2.2" diff, README profile sweep).
 * out: [B,H,N,d] (layout BHND) or [B,N,H,d] (layout BNHD) of dtype, on the host if out_on_host
 * else on the device; lse: fp32 [B,H,N] in the same memory as out, or NULL.
 * Synchronous: returns when out, lse and *stats (may be NULL) are final. Allocates its device
 * buffers up front and frees them on every path; CQSA_ERR_OOM if they do not fit.
 */
int cqsa_stream_attn_fwd(const void* q_host, const void* k_host, const void* v_host, int layout, void* out,
                         float* lse, int out_on_host, int B, int H, long long N, int d, int causal,
                         float scale, int dtype, long long chunk_tokens, cqsa_stream_stats* stats,
                         cudaStream_t stream);

/*
 * Resident inputs for cqsa_stream_attn_fwd (and the budget of cqsa_stream_attn_bwd's resident schedule,
 * described with it). When Q, K, V and the output (4 * B*H*N*d*2 bytes, plus
 * B*H*N*4 of lse) take at most `bytes` of device memory (bytes < 0, the default: at most half of the
 * device's free memory at the call; 0: never), and one head's K and V (2*N*d*2 bytes) fit the 64 MiB
 * of L2 the kernel groups heads by (longer prefixes would have every CTA sweep keys L2 cannot hold, and
 * the accumulating schedule is faster there), each chunk is still copied from the host once, chunk by
 * chunk beside the kernels, but into full-length device tensors where it stays; each Q chunk then runs
 * as one launch over the key prefix it sees (every key when not causal) and writes its output rows
 * directly (no fp32 accumulator, no merge), which return to `out` chunk by chunk.
 * Consecutive Q chunks alternate between `stream` and a second stream of the call, so one launch's
 * last wave overlaps the next one. Every query tile then sees the same key tiles in the same order
 * as in cqsa_attn_fwd, so the results are bitwise equal to it (the accumulating schedule agrees up to
 * fp32 summation order). Process-wide setting.
 */
void cqsa_set_stream_kv_resident_bytes(long long bytes);

/* ------------------------------------------------------------------------------------------------
 * Cyclic quorum-set decomposition ("stream-cqsa 2.2.0 -> 2.2.2" diff, README and autoconfig.plan: a
 * configuration is (c, interest_set, itr) with c**itr subproblems and cost (l^2/c)^itr, l the size of
 * the interest set; the default set is (0, 1, 3) at c = 7). The pages name the parameters, not the
 * construction; the reading implemented: the sequence is cut into T = c^itr chunks (a multiple of 128
 * tokens each, the last ragged); subproblem s owns the chunks whose base-c digits t_e lie in
 * s_e + interest_set (mod c) for every digit e; interest_set must be a perfect difference set mod c;
 * every needed (query chunk, key chunk) pair (key <= query when causal) is computed in exactly one
 * subproblem containing both and merged exactly into the query chunk's accumulator.
 * ------------------------------------------------------------------------------------------------ */

/* CQSA_OK if interest_set (l residues) is a perfect difference set modulo c (its l(l-1) ordered
 * differences are the non-zero residues, each once); CQSA_ERR_INVALID (with a message) otherwise. */
int cqsa_quorum_check(int c, const int* interest_set, int l);

/* The schedule of a quorum decomposition with n_chunks non-empty chunks (<= c^itr): writes the
 * triples (subproblem, query chunk, key chunk), sorted by subproblem, into out[3*i .. 3*i+2] and
 * returns their number; out == NULL returns the number only. Host-only (no GPU). Negative status on
 * an invalid set, itr < 1, c^itr > 65536, or max_triples too small. */
long long cqsa_quorum_schedule(int c, const int* interest_set, int l, int itr, int n_chunks, int causal, int* out,
                               long long max_triples);

typedef struct {
  double wall_ms;              /* host wall time of the call */
  double compute_ms;           /* sum of attention-kernel event intervals (lanes overlap, so with
                                  max_parallel > 1 this can exceed the wall time) */
  double copy_ms;              /* sum of chunk-staging copy intervals (copy stream) */
  long long copy_bytes;        /* bytes staged (host->device or device->device) */
  long long peak_device_bytes; /* device memory the executor allocated */
  long long chunk_tokens;      /* C */
  long long acc_host_bytes;    /* accumulator bytes moved between host and device (host accumulator) */
  int n_subproblems;           /* subproblems with at least one pair */
  int n_pairs;                 /* chunk pairs computed (= kernels of attention) */
  int n_chunk_loads;           /* chunk stagings (Q and K/V counted separately) */
  int n_launches;              /* kernels launched (attention + finalize) */
} cqsa_quorum_stats;

/*
 * Exact attention through the quorum decomposition. q, k, v: [B,H,N,d] (layout BHND) or [B,N,H,d]
 * (layout BNHD), fp16/bf16, in host memory (inputs_on_host, pinned for speed) or device memory. Host
 * inputs: each subproblem's chunks are staged into two sets of l^itr device slots; device inputs are
 * read in place (a chunk is a token range of the caller's tensor). acc_on_host = 0: one fp32
 * accumulator per query chunk on the device; acc_on_host = 1 (the pages' accumulate_on_gpu=False,
 * "stream-cqsa 2.2.0 -> 2.2.2" README): the accumulators live in pinned host memory allocated by the
 * call and travel with their Q slot, so device memory is bounded by the slots. out/lse as in
 * cqsa_stream_attn_fwd (host if out_on_host). Synchronous; allocates its buffers up front and frees
 * them on every path (CQSA_ERR_OOM if they do not fit). max_parallel (1..16, the pages' max_parallel):
 * chunk pairs of different query chunks run on that many compute streams (pair (q, k) on stream
 * q mod max_parallel; stream 0 is `stream`), so small pairs fill the GPU side by side. The result
 * equals the chunked-and-merged attention with chunk size C up to fp32 rounding of the merge order,
 * and is bit-identical for every acc_on_host and max_parallel.
 */
int cqsa_quorum_attn_fwd(const void* q, const void* k, const void* v, int layout, int inputs_on_host, void* out,
                         float* lse, int out_on_host, int B, int H, long long N, int d, int causal, float scale,
                         int dtype, int c, const int* interest_set, int l, int itr, int acc_on_host,
                         int max_parallel, cqsa_quorum_stats* stats, cudaStream_t stream);

/*
 * The same decomposition with a choice of engine (the pages' classic and wave engines, "stream-cqsa
 * 2.2.0 -> 2.2.2" diff: README, peak memory of the wave engine and its wave budget, and `api.py`
 * `_pick_wave`, whose default budget is min(2M, max(512K, N)) packed tokens).
 * engine = CQSA_ENGINE_CLASSIC: one chunk-pair launch after another on max_parallel lanes (as
 *   cqsa_quorum_attn_fwd).
 * engine = CQSA_ENGINE_WAVE: the pairs of each subproblem run in waves, one multi-pair launch per wave
 *   (up to 32 pairs, at most one per query chunk, so each pair's epilogue merges into its query
 *   chunk's accumulator without a race); a wave holds at most wave_tokens query tokens (0 selects
 *   min(2^21, max(2^19, N))). Partials are merged in place by the kernel's epilogue, so no packed
 *   partial buffer is needed and the budget only caps a launch's size. max_parallel is ignored (one
 *   stream). With host inputs, pairs of a query chunk are merged in the same order as by the classic
 *   engine, so the two engines give bit-identical results.
 * Device-resident inputs (inputs_on_host = 0) are read in place by either engine; nothing is staged.
 *   The wave engine then runs the pairs of a query chunk whose key chunks are adjacent as one pair over
 *   the joined key range (the online softmax over the joined keys is the exact merge of the parts), and
 *   without a host accumulator its waves span every subproblem: a causal problem then runs one pair per
 *   query chunk over its whole key prefix, bitwise equal to cqsa_attn_fwd on the same inputs; with a
 *   host accumulator, within the fp32 merge error of the classic engine.
 */
enum { CQSA_ENGINE_CLASSIC = 0, CQSA_ENGINE_WAVE = 1 };
int cqsa_quorum_attn_fwd_ex(const void* q, const void* k, const void* v, int layout, int inputs_on_host, void* out,
                            float* lse, int out_on_host, int B, int H, long long N, int d, int causal, float scale,
                            int dtype, int c, const int* interest_set, int l, int itr, int acc_on_host,
                            int max_parallel, int engine, long long wave_tokens, cqsa_quorum_stats* stats,
                            cudaStream_t stream);

/*
 * The host-driven entry points (cqsa_stream_attn_fwd, cqsa_quorum_attn_fwd) take their device buffers,
 * events and copy streams from a per-device cache that persists across calls (allocation, stream and
 * event creation and cudaFree's device synchronisation would otherwise cost a large share of a short
 * call). Cached device memory stays allocated until this call frees everything idle (all devices);
 * an allocation that fails frees the idle buffers of its device and retries once. Returns CQSA_OK.
 * Not to be called while one of those entry points runs on another thread.
 */
int cqsa_release_cache(void);

/*
 * Attention backward: the gradients of a scalar loss with respect to q, k and v, given its gradient
 * dout with respect to the forward output. The pages name a backward that works from the forward's
 * saved per-row log-sum-exp (`stream_cqsa_backward`, "stream-cqsa 2.2.0 -> 2.2.2" diff, README list of
 * explicit entry points; "2.2.2 -> 2.2.3" diff, stream_cqsa/oom_fallback.py, `stream_cqsa_auto`
 * docstring: info["lse"] is what it needs) but print no formula; this is the chain rule through the
 * row softmax of the forward above, with P recomputed from lse:
 *   P_ij = exp(s_ij - lse_i) on A_i (0 elsewhere),  D_i = dout_i . out_i,  dP_ij = dout_i . v_j,
 *   dS_ij = P_ij (dP_ij - D_i),  dv_j = sum_i P_ij dout_i,  dk_j = scale sum_i dS_ij q_i,
 *   dq_i = scale sum_j dS_ij k_j.
 * q, k, v, out (the forward's output), dout: device [B,H,N,d], d = 64 or 128, fp16 or bf16 (dtype),
 * contiguous (layout BHND); lse: device [B,H,N] fp32 as cqsa_attn_fwd wrote it (natural log). dq, dk,
 * dv: device [B,H,N,d] in dtype, written in full. P and dS enter the tensor-core products rounded to
 * dtype; all sums are fp32. workspace: caller-owned device memory of at least
 * cqsa_attn_bwd_workspace_size(B, H, N, d) bytes (the fp32 dq accumulator and D), 16-byte aligned;
 * its contents on entry do not matter. Other head dimensions return CQSA_ERR_UNSUPPORTED.
 * Asynchronous on `stream`; allocates nothing. Runs are bitwise reproducible except dq, whose fp32
 * accumulation order across key tiles follows the atomic adds (differences of a few fp32 ulps
 * before the final rounding to dtype).
 */
size_t cqsa_attn_bwd_workspace_size(int B, int H, int N, int d);
int cqsa_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                  int causal, float scale, int dtype, cudaStream_t stream);

/*
 * The backward over chunk pairs, for problems cut the way the forward's chunk pairs cut them (the
 * pages' streamed backward, `stream_cqsa_backward`, works subproblem by subproblem). The gradient is a
 * sum over key chunks (dq) and over query chunks (dk, dv) of the same chain-rule terms, with P taken
 * against the full-row lse, so accumulating every needed pair gives the monolithic gradient up to the
 * fp32 summation order.
 *
 * cqsa_attn_bwd_dvec: D_i = dout_i . out_i (fp32) of a query chunk: out_blk, dout_blk [B,H,Nq,d]
 *   (dtype), dvec_blk [B,H,Nq] fp32. out is the forward's full output for those rows.
 * cqsa_attn_bwd_chunk: one pair. q_blk, dout_blk [B,H,Nq,d] with lse_blk (the forward's full-row lse)
 *   and dvec_blk [B,H,Nq] of the query chunk at absolute position q_off; k_blk, v_blk [B,H,Nkv,d] of
 *   the key chunk at kv_off (causal masking on absolute positions; a pair with every key after every
 *   query adds nothing). Adds scale * dS K into dq_acc [B,H,Nq,d], scale * dS^T Q into dk_acc and
 *   P^T dout into dv_acc [B,H,Nkv,d], all fp32, which the caller zeroes before its first pair and
 *   keeps until its last; pairs on one stream may share accumulators. d = 64 or 128; asynchronous;
 *   allocates nothing.
 * cqsa_attn_bwd_cast: n fp32 values (n a multiple of 4) rounded to dtype (RNE), e.g. the accumulators
 *   into dq, dk, dv.
 */
int cqsa_attn_bwd_dvec(const void* out_blk, const void* dout_blk, float* dvec_blk, int B, int H, int Nq, int d,
                       int dtype, cudaStream_t stream);
int cqsa_attn_bwd_chunk(const void* q_blk, const void* k_blk, const void* v_blk, const void* dout_blk,
                        const float* lse_blk, const float* dvec_blk, long long q_off, long long kv_off, int B, int H,
                        int Nq, int Nkv, int d, int causal, float scale, int dtype, float* dq_acc, float* dk_acc,
                        float* dv_acc, cudaStream_t stream);
int cqsa_attn_bwd_cast(const float* acc, void* out, long long n, int dtype, cudaStream_t stream);

/*
 * Host-resident backward over chunk pairs (the pages' streamed backward, `stream_cqsa_backward`): q, k,
 * v, out, dout [B,H,N,d] (d = 64 or 128, fp16/bf16, layout BHND) and lse [B,H,N] fp32 in host memory
 * (pinned for speed); dq, dk, dv [B,H,N,d] written to host memory. Query-outer over chunks of chunk_tokens (a
 * positive multiple of 128): each query chunk's q/out/dout/lse and each needed key chunk's k/v are
 * copied to the device on a copy stream, double-buffered so copies overlap the kernels, the key chunks
 * in alternating directions so consecutive query chunks share one copy; each pair runs
 * cqsa_attn_bwd_chunk's kernel on `stream`; dq leaves after its query chunk, dk and dv after the last
 * one, on a second stream. Device memory: 2 * B*H*N*d*4 bytes of dk/dv accumulators plus two slots of
 * each streamed chunk (inputs, D, lse, the dq accumulator, output staging), from the library's pool
 * (CQSA_ERR_OOM if they do not fit). Synchronous; the result equals cqsa_attn_bwd's up to the fp32
 * summation order. Returns CQSA_ERR_TIMEOUT if a kernel's bounded wait gave up.
  * When q, out, dout, lse, D, the fp32 dq accumulator, every K/V chunk and the dk/dv accumulators fit
 * the resident budget (cqsa_set_stream_kv_resident_bytes; about 14 bytes of device memory per byte of
 * one input tensor), every chunk is instead copied once and stays: key chunks go from the last to the
 * first, the query side copied in the same order, and each key chunk is one launch of the chunk-pair
 * kernel over every query it meets, the launches round-robin over up to four streams.
 */
int cqsa_stream_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int B, int H, long long N, int d, int causal,
                         float scale, int dtype, long long chunk_tokens, cudaStream_t stream);
/* The same call, filling *stats (may be NULL): compute_ms sums the event intervals of its kernel segments
 * (D and the dq zeroing of each query chunk, each pair, each output cast), h2d_ms those of its copy
 * groups, stall_ms the gaps between consecutive kernel segments, n_chunks the pairs run. On the resident
 * schedule compute_ms is the union of the kernel intervals (its launches overlap on several streams) and
 * n_chunks the key-chunk launches. */
int cqsa_stream_attn_bwd_ex(const void* q, const void* k, const void* v, const void* out, const void* dout,
                            const float* lse, void* dq, void* dk, void* dv, int B, int H, long long N, int d,
                            int causal, float scale, int dtype, long long chunk_tokens, cqsa_stream_stats* stats,
                            cudaStream_t stream);

/*
 * Size of the file-scope device array that cqsa_attn_fwd_chunked_static uses as its scratch (32 MiB).
 */
#define CQSA_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * Chunked exact attention over device-resident q, k, v ([B,H,N,d], fp16/bf16) into out ([B,H,N,d],
 * same dtype) and lse ([B,H,N] fp32, or NULL) that ALLOCATES NOTHING. It is for callers that cannot
 * let a library call cudaMalloc (code running under its own memory pool or a hard device-memory
 * budget, where an allocation inside the call would fail, exceed the budget or synchronise the device
 * at an unwanted point). The paper has no counterpart of this entry point: it is a library facility.
 * The computation is the same as cqsa_stream_attn_fwd's (key chunks of chunk_tokens merged exactly
 * into an fp32 accumulator, one query chunk and one (b, h) at a time), but the accumulator lives in
 * a fixed file-scope device array of CQSA_STATIC_SCRATCH_BYTES, held by every device on which the
 * library's module is loaded until the process exits. chunk_tokens must be a multiple of 128 with
 * chunk_tokens * (d + 1) * 4 <= CQSA_STATIC_SCRATCH_BYTES, else CQSA_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture. All calls share the array and it
 * keeps the last call's contents: calls whose work overlaps on the GPU (different streams, or host
 * threads without ordering between them) race on it. Asynchronous on `stream`.
 */
int cqsa_attn_fwd_chunked_static(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                                 int H, int N, int d, int causal, float scale, int dtype, int chunk_tokens,
                                 cudaStream_t stream);

/* Human-readable name of a status code. */
const char* cqsa_status_string(int status);

/* Message of the calling thread's last failed call ("" if none). */
const char* cqsa_last_error(void);

/*
 * Device error word written by a kernel whose bounded wait gave up (instead of hanging the GPU):
 * synchronises the device, stores the code (0 = none) and the block index, optionally clears it.
 * Returns CQSA_OK, or CQSA_ERR_TIMEOUT if a code was set. Two codes return CQSA_ERR_DEVICE instead:
 * 5, a d = 128 forward CTA that ran on an SM beyond its running-sum slots (the result is still exact),
 * and 6, a backward kernel whose dynamic shared memory base was not 1024-byte aligned (it stopped
 * before computing anything).
 */
int cqsa_device_error(int* code, int* block, int clear);

/* Device-side wait limit in milliseconds (default 2000; env CQSA_TIMEOUT_MS). */
void cqsa_set_timeout_ms(unsigned int ms);

/*
 * Test hook for the device-side bounded waits (not for production use): kind 1 makes the next
 * attention launches skip the load of key/value tile 1 in their first CTA, and kind 2 makes the next
 * backward launches skip the key/value load of their first CTA, so that CTA's waits run out after the
 * timeout; the kernel then records CQSA_ERR_TIMEOUT in its device error word, drains its own copies
 * and MMAs, frees tensor memory and returns (no trap, no hang). kind 0 turns it off.
 */
int cqsa_debug_set_fault(int kind);

/* Library version, e.g. "0.1.0". */
const char* cqsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CQSA_H */
