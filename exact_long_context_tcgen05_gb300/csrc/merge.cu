// Exact LSE merge of n partial attention results over disjoint key sets (HBM-bound).
//
// Per row:  M = max_k LSE_k,  lse = M + ln sum_k exp(LSE_k - M),  out = sum_k exp(LSE_k - lse) O_k,
// summed in part order k = 0 .. n-1 so the result is deterministic. Rows whose parts are all empty
// (LSE = -inf) give out = 0 and lse = -inf. The pages merge subproblem outputs into an accumulator
// ("stream-cqsa 2.2.0 -> 2.2.2" diff, README profile sweep) without printing the formula; this is
// the exact combination of softmax partials that carry their log-sum-exp.
//
// Layout of the work: a group of d/4 threads owns four rows at a time; each thread owns 4 consecutive
// features and streams its float4 of every O_k for the four rows (fully coalesced: a warp reads 512
// contiguous bytes per part and row pair; four independent loads in flight per part). The LSE pass is
// spread over the group's threads and reduced with shuffles inside the group. Grid-stride over row
// groups with a grid sized to the SM count.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "cqsa_internal.h"

namespace cqsa {
namespace {

template <int MAXN>
struct PartPtrs {
  const float* o[MAXN];
  const float* l[MAXN];
};

__device__ __forceinline__ void store4(void* out, long long idx4, float4 v, int dt) {
  if (dt == CQSA_F32) {
    reinterpret_cast<float4*>(out)[idx4] = v;
  } else if (dt == CQSA_F16) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&a);
    w.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(out)[idx4] = w;
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&a);
    w.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(out)[idx4] = w;
  }
}

template <int D, int MAXN>
__global__ void __launch_bounds__(256) merge_kernel(const PartPtrs<MAXN> parts, int n, void* out, float* lse,
                                                    long long rows, int out_dtype) {
  constexpr int G = D / 4;  // threads per row (16 or 32)
  constexpr int R = 4;      // rows per group per step: R independent loads in flight per part
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int g = threadIdx.x % G;
  const long long group0 = tid / G;
  const long long ngroups = static_cast<long long>(gridDim.x) * blockDim.x / G;
  const unsigned lane = threadIdx.x & 31;
  const unsigned gmask = (G == 32) ? 0xffffffffu : (0xffffu << (lane & 16u));

  for (long long r0 = group0 * R; r0 < rows; r0 += ngroups * R) {
    long long rr[R];
#pragma unroll
    for (int u = 0; u < R; ++u) rr[u] = (r0 + u < rows) ? r0 + u : rows - 1;  // clamped rows repeat a valid one
    float m[R];
#pragma unroll
    for (int u = 0; u < R; ++u) m[u] = -INFINITY;
    for (int k = g; k < n; k += G) {
#pragma unroll
      for (int u = 0; u < R; ++u) m[u] = fmaxf(m[u], __ldg(parts.l[k] + rr[u]));
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
#pragma unroll
      for (int u = 0; u < R; ++u) m[u] = fmaxf(m[u], __shfl_xor_sync(gmask, m[u], o));
    }
    float z[R];
#pragma unroll
    for (int u = 0; u < R; ++u) z[u] = 0.0f;
    for (int k = g; k < n; k += G) {
#pragma unroll
      for (int u = 0; u < R; ++u)
        if (m[u] != -INFINITY) z[u] += expf(__ldg(parts.l[k] + rr[u]) - m[u]);
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
#pragma unroll
      for (int u = 0; u < R; ++u) z[u] += __shfl_xor_sync(gmask, z[u], o);
    }
    float L[R];
    float4 acc[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      L[u] = (m[u] != -INFINITY) ? m[u] + logf(z[u]) : -INFINITY;
      acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k = 0; k < n; ++k) {
      float lk[R];
      float4 v[R];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        lk[u] = __ldg(parts.l[k] + rr[u]);
        v[u] = __ldg(reinterpret_cast<const float4*>(parts.o[k] + rr[u] * D) + g);
      }
#pragma unroll
      for (int u = 0; u < R; ++u) {
        if (lk[u] == -INFINITY) continue;  // an empty part has weight 0 (and every part of an empty row)
        const float w = expf(lk[u] - L[u]);
        acc[u].x = fmaf(w, v[u].x, acc[u].x);
        acc[u].y = fmaf(w, v[u].y, acc[u].y);
        acc[u].z = fmaf(w, v[u].z, acc[u].z);
        acc[u].w = fmaf(w, v[u].w, acc[u].w);
      }
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
      if (r0 + u >= rows) break;
      store4(out, rr[u] * G + g, acc[u], out_dtype);
      if (lse && g == 0) lse[rr[u]] = L[u];
    }
  }
}


template <int D, int MAXN>
int launch_n(const float* const* O_parts, const float* const* LSE_parts, int n, void* out, float* lse, long long rows,
             int out_dtype, cudaStream_t stream) {
  PartPtrs<MAXN> pp;
  for (int k = 0; k < MAXN; ++k) {
    pp.o[k] = k < n ? O_parts[k] : nullptr;
    pp.l[k] = k < n ? LSE_parts[k] : nullptr;
  }
  constexpr int G = D / 4;
  const long long rows_per_block = 256 / G * 4;
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = static_cast<long long>(sm_count()) * 8;  // 8 x 256 threads resident per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  merge_kernel<D, MAXN><<<static_cast<int>(blocks), 256, 0, stream>>>(pp, n, out, lse, rows, out_dtype);
  return cuda_status(cudaGetLastError(), "merge kernel launch");
}

template <int D>
int launch_d(const float* const* O_parts, const float* const* LSE_parts, int n, void* out, float* lse, long long rows,
             int out_dtype, cudaStream_t stream) {
  if (n <= 16) return launch_n<D, 16>(O_parts, LSE_parts, n, out, lse, rows, out_dtype, stream);
  if (n <= 128) return launch_n<D, 128>(O_parts, LSE_parts, n, out, lse, rows, out_dtype, stream);
  return launch_n<D, 1024>(O_parts, LSE_parts, n, out, lse, rows, out_dtype, stream);
}

}  // namespace

int launch_merge(const float* const* O_parts, const float* const* LSE_parts, int n, void* out, float* lse,
                 long long rows, int d, int out_dtype, cudaStream_t stream) {
  if (rows == 0) return CQSA_OK;
  if (d == 64) return launch_d<64>(O_parts, LSE_parts, n, out, lse, rows, out_dtype, stream);
  return launch_d<128>(O_parts, LSE_parts, n, out, lse, rows, out_dtype, stream);
}

// SM count of the current device, cached per device.
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace cqsa
