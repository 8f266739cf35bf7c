// Internal declarations shared by the library's translation units (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/cqsa.h"

namespace cqsa {

// Output / partial modes of the attention kernel.
enum AttnMode : int {
  kModeOut = 0,    // normalised output in the input dtype + fp32 LSE (the SDPA-shaped call)
  kModePart = 1,   // normalised fp32 partial output + fp32 LSE of one chunk pair
  kModeAccum = 2,  // merge this chunk pair's result into an fp32 (O_acc, LSE_acc) in place
};

struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  int B, H;
  int Nq, Nkv;          // tokens held in the q / kv buffers
  long long q_off;      // absolute position of q-buffer token 0 (causal mask)
  long long kv_off;     // absolute position of kv-buffer token 0
  int d;
  int causal;
  float scale;          // already resolved (0 -> 1/sqrt(d) done by the caller)
  int dtype;            // CQSA_F16 / CQSA_BF16
  int in_layout;        // layout of q/k/v buffers: CQSA_LAYOUT_BHND / CQSA_LAYOUT_BNHD
  int mode;             // AttnMode
  void* out;            // kModeOut: [B,H,Nq,d] (or [B,Nq,H,d] with out_layout) in dtype
  float* lse;           // kModeOut: [B,H,Nq]
  float* o_part;        // kModePart / kModeAccum: fp32 [B,H,Nq,d] (or token-major)
  float* lse_part;      // fp32 [B,H,Nq]
  int out_layout;       // layout of out / o_part
  long long q_tokens_alloc;   // tokens per head in the q buffer when it is a token range of a longer
                              // tensor (its strides follow this count); 0: the buffer holds Nq tokens
  long long kv_tokens_alloc;  // the same for k / v; 0: Nkv
};

// Validates nothing (the ABI layer does); encodes tensor maps and launches on `stream`.
int launch_attention(const AttnArgs& a, cudaStream_t stream);
// Up to kMaxWavePairs (32) chunk pairs in one launch (the wave engine). The pairs share B, H, d, dtype,
// causal, layouts and scale; each has its own buffers, offsets, sizes, mode (kModePart or kModeAccum)
// and accumulator. Pairs writing one accumulator must not share a launch (their epilogues would race).
int launch_attention_multi(const AttnArgs* pairs, int n, cudaStream_t stream);

// Attention backward (attn_bwd.cu), head dimension 64. The monolithic call (launch_attention_bwd) takes
// q, k, v, out, dout [B,H,N,64] with Nq = Nkv = N and offsets 0, writes dq, dk, dv, and uses
// `workspace` (attention_bwd_workspace bytes) for the fp32 dQ accumulator and D. One chunk pair
// (launch_attention_bwd_chunk) takes a query chunk (q, dout, lse, dvec: Nq rows at absolute position
// q_off) and a key chunk (k, v: Nkv rows at kv_off) and adds into dq_acc [B,H,Nq,64], dk_acc and
// dv_acc [B,H,Nkv,64] (fp32, scale applied).
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* out;
  const void* dout;
  const float* lse;
  const float* dvec;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;
  float* dk_acc;
  float* dv_acc;
  void* workspace;
  int B, H, Nq, Nkv, d;
  long long q_off, kv_off;
  int causal;
  float scale;  // resolved
  int dtype;
};
size_t attention_bwd_workspace(int B, int H, int N, int d);
int launch_attention_bwd(const BwdArgs& a, cudaStream_t stream);
int launch_attention_bwd_chunk(const BwdArgs& a, cudaStream_t stream);
// D_i = dout_i . out_i (fp32) for `rows` rows of 64 features; fp32 -> dtype for n elements (n % 4 == 0).
int launch_bwd_dvec(const void* out, const void* dout, float* dvec, long long rows, int d, int dtype,
                    cudaStream_t stream);
// Host-streaming helpers (stream_driver.cu): whether `bytes` of device memory fit the resident budget
// (cqsa_set_stream_kv_resident_bytes), and a copy of tokens [t0, t0 + n) of a (layout, N tokens) tensor
// into the same positions of another of the same shape; *bytes grows by the bytes copied.
bool stream_resident_ok(size_t bytes);
cudaError_t copy_range(void* dst, const void* src, int layout, int B, int H, long long N, int d, long long t0, int n,
                       cudaMemcpyKind kind, cudaStream_t s, long long* bytes);
// D for tokens [t0, t0 + n) of every head of [BH, N, d] out / dout, into dvec [BH, N] at the same rows.
int launch_bwd_dvec_range(const void* out, const void* dout, float* dvec, long long BH, long long n, long long N,
                          long long t0, int d, int dtype, cudaStream_t stream);
int launch_bwd_cast(const float* acc, void* out, long long n, int dtype, cudaStream_t stream);

// LSE merge of n partials (device pointer arrays passed by value).
int launch_merge(const float* const* O_parts, const float* const* LSE_parts, int n, void* out, float* lse,
                 long long rows, int d, int out_dtype, cudaStream_t stream);

// Copy tokens [t0, t0+n) of a [B,H,N,d] / [B,N,H,d] tensor (host or device) into a packed chunk buffer.
cudaError_t copy_chunk(void* dst, const void* src, int layout, int B, int H, long long N, int d, long long t0, int n,
                       cudaMemcpyKind kind, cudaStream_t s, long long* bytes);

// Normalised fp32 accumulator (acc [B,H,n,d], lse_acc [B,H,n]) -> out tokens [t0, t0+n) of an N-token
// tensor in `layout` and `dtype`, plus lse_out (may be NULL).
int launch_finalize(const float* acc, const float* lse_acc, void* out, float* lse_out, int B, int H, int n,
                    long long N, long long t0, int d, int layout, int dtype, cudaStream_t stream);

// Reusable device buffers, events and non-blocking streams (per device; csrc/pool.cu). A caller
// returns them only after all work using them has completed.
int pool_alloc(void** p, size_t n);
void pool_free(void* p);
int pool_event(cudaEvent_t* e, bool timing);
void pool_event_free(cudaEvent_t e, bool timing);
int pool_stream(cudaStream_t* s);
void pool_stream_free(cudaStream_t s);

// Set-up that belongs to one device's context (kernel function attributes, cached device attributes)
// runs once per device: bit `dev` records it. Concurrent first calls may both run the set-up, which is
// idempotent; devices numbered 64 and above repeat it on every call.
struct PerDeviceOnce {
  std::atomic<unsigned long long> bits{0};
  // true when the current device's set-up has run; *dev receives the current device (-1 on error)
  bool done(int* dev) const {
    if (cudaGetDevice(dev) != cudaSuccess) {
      *dev = -1;
      return false;
    }
    return seen(*dev);
  }
  // the bookkeeping alone: has device `dev` been marked (ids outside [0, 64) never are)
  bool seen(int dev) const { return dev >= 0 && dev < 64 && ((bits.load(std::memory_order_acquire) >> dev) & 1ull); }
  void mark(int dev) {
    if (dev >= 0 && dev < 64) bits.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
};

// The device error words (set by a kernel whose bounded wait gave up), read after the caller's own
// streams have drained: each word is copied on `s` and `s` is synchronised, so no other stream of the
// process is waited for. A set word is cleared and reported as CQSA_ERR_TIMEOUT with its code, block
// and site in the error message.
int check_device_error_on(cudaStream_t s);

// Number of SMs of the current device (cached per device; 152 if the query fails).
int sm_count();

// Status helpers
void set_error(const char* fmt, ...);
int cuda_status(cudaError_t e, const char* what);
unsigned long long timeout_ns();
int debug_fault();

}  // namespace cqsa
