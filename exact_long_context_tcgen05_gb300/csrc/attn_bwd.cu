// Exact attention backward on sm_103a: the gradients dQ, dK, dV of softmax(Q K^T * scale [+ causal
// mask]) V, given the upstream gradient dO, the forward output O and the forward's per-row LSE.
//
// The pages name a backward that works from the forward's saved log-sum-exp ("stream-cqsa 2.2.0 ->
// 2.2.2" diff, README list of explicit entry points, `stream_cqsa_backward`; "2.2.2 -> 2.2.3" diff,
// stream_cqsa/oom_fallback.py, `stream_cqsa_auto` docstring: info["lse"] is what it needs) but print
// no formula. This is the chain rule through the row softmax, with P recomputed from the LSE:
//   P_ij  = exp(s_ij - LSE_i),  s_ij = scale q_i . k_j   (0 where the causal mask hides j from i)
//   D_i   = dO_i . O_i          (equals sum_j P_ij dP_ij)
//   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i)
//   dV_j  = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j
//
// Kernels, in stream order:
//   bwd_dot_kernel   D_i in fp32 (eight threads per row, 16-byte loads of O and dO)
//   attn_bwd_kernel  one CTA per (key tile j of 128 keys, batch-head), heaviest key tiles first. K_j
//                    and V_j stay in shared memory; Q_i and dO_i of the query tiles that see key
//                    tile j (every i, or i >= j when causal) stream through a two-slot TMA ring.
//                    Per query tile, with the key dimension on the 128 tensor-memory lanes:
//                      S^T = K_j Q_i^T, dP^T = V_j dO_i^T         (tcgen05, fp32 in tensor memory)
//                      P^T and dS^T: one thread per key row, in registers
//                      dV_j += P^T dO_i, dK_j += dS^T Q_i         (A operand from tensor memory)
//                      dQ_i  = dS K_j                             (dS^T staged MN-major in shared memory)
//                    and the dQ tile is added into an fp32 accumulator with 16-byte atomic adds while
//                    the tensor pipe already computes the next S^T and dP^T. dK_j, dV_j are written
//                    once, after the last query tile.
//   bwd_dq_kernel    fp32 dQ accumulator -> dQ in the input dtype
// P and dS enter the MMAs rounded to the input dtype; everything else is fp32. Head dimension 64.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "cqsa_internal.h"
#include "sm103_ptx.cuh"

namespace cqsa {
namespace {

__device__ DevErr g_bwd_err;

constexpr int BT = 128;                         // keys per CTA tile, queries per step
constexpr int HD = 64;                          // head dimension
constexpr uint32_t BOX = BT * HD * 2;           // one 128 x 64 tile of 16-bit elements (16 KiB)
constexpr uint32_t OFF_K = 0, OFF_V = BOX, OFF_Q = 2 * BOX, OFF_G = 4 * BOX, OFF_DS = 6 * BOX;
constexpr uint32_t OFF_DQ = 8 * BOX;            // dQ staging: 2 slots of 128 x 64 fp32
constexpr uint32_t DQ_SLOT = BT * HD * 4;
constexpr uint32_t OFF_ROW = OFF_DQ + 2 * DQ_SLOT;  // float lse2[2][128], dd[2][128]
constexpr uint32_t OFF_BAR = OFF_ROW + 4 * BT * 4;
constexpr int NBAR = 6;                         // kv, q[2], mma1, mma2, idle
constexpr uint32_t SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;  // + slack for 1024-byte alignment
// Tensor memory: S^T (P^T over its first 64 columns), dP^T (dS^T over its first 64), dV, dK, dQ.
constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 320, COL_DQ = 384;
constexpr uint32_t TMEM_COLS = 512;
constexpr float LOG2E = 1.4426950408889634f;
constexpr int NTHR = 256;  // eight warps: two per tensor-memory lane quarter, each on half the columns

enum : int { kBwdTimeoutLoad = 1, kBwdTimeoutMMA = 3 };

struct BwdParams {
  const float* lse;       // [BH, N] natural-log LSE of the forward
  const float* dvec;      // [BH, N] D_i
  float* dq_acc;          // [BH, N, 64] fp32, zeroed; receives scale * dS K
  uint16_t* dk;           // [BH, N, 64] input dtype
  uint16_t* dv;
  int H, BH, N, n_tiles;
  float scale, scale_log2;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ void record_bwd_error(int code, int where) {
  if (atomicCAS(&g_bwd_err.code, 0, code) == 0) {
    g_bwd_err.block = blockIdx.x;
    g_bwd_err.where = where;
  }
}

// Bounded wait that returns early once another thread of the CTA has given up.
__device__ __forceinline__ bool wait_abort(uint64_t* bar, uint32_t parity, unsigned long long tmo,
                                           volatile int* abort_flag, int code, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > tmo) {
        record_bwd_error(code, where);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool elect_lane() {
  uint32_t p;
  asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}" : "=r"(p));
  return p != 0;
}

// MMAs with the accumulate flag as an immediate (issued from one elected lane of a converged warp).
template <int ACC>
__device__ __forceinline__ void mma_ss_imm(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 1;" ::"r"(d), "l"(a), "l"(b), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 0;" ::"r"(d), "l"(a), "l"(b), "r"(idesc)
                 : "memory");
}
template <int ACC>
__device__ __forceinline__ void mma_ts_imm(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d), "r"(a), "l"(b), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 0;" ::"r"(d), "r"(a), "l"(b), "r"(idesc)
                 : "memory");
}

// Generic-proxy shared-memory writes become visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Bulk tensor reduction: the shared-memory box at `src` is added (fp32) into the global tensor at
// (x, y, z); rows outside the tensor are skipped. Completion is tracked by bulk groups.
__device__ __forceinline__ void tma_reduce_add_3d(uint32_t src, const CUtensorMap* map, int x, int y, int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one bulk group still reading shared memory
__device__ __forceinline__ void bulk_wait_read_le1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_pair(float lo, float hi, int bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_pair(uint32_t w, int bf16) {
  if (bf16) return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w));
  return __half22float2(*reinterpret_cast<__half2*>(&w));
}

// S^T = K Q^T (or dP^T = V dO^T): 4 MMAs of 128 x 128 x 16, both operands K-major, 128-byte swizzle.
__device__ __forceinline__ void issue_t(uint32_t dcol, uint64_t a0, uint64_t b0, uint32_t idesc) {
  mma_ss_imm<0>(dcol, a0, b0, idesc);
#pragma unroll
  for (int ks = 1; ks < HD / 16; ++ks) mma_ss_imm<1>(dcol, a0 + ks * 2, b0 + ks * 2, idesc);
}

// dV += P^T dO, dK += dS^T Q (A from tensor memory, B MN-major) and dQ = dS K (A = dS^T staged
// MN-major in shared memory, B = K MN-major): 8 key/query steps of 16.
template <int FIRST>
__device__ __forceinline__ void issue_grads(uint32_t tmem, uint64_t dG, uint64_t dQm, uint64_t dS, uint64_t dK,
                                            uint32_t idesc_g, uint32_t idesc_q) {
#pragma unroll
  for (int ks = 0; ks < BT / 16; ++ks) {
    const uint32_t off = static_cast<uint32_t>(ks * (2048 >> 4));  // 16 rows of 128 bytes
    if (FIRST && ks == 0) {
      mma_ts_imm<0>(tmem + COL_DV, tmem + COL_S + ks * 8, dG + off, idesc_g);
      mma_ts_imm<0>(tmem + COL_DK, tmem + COL_DP + ks * 8, dQm + off, idesc_g);
    } else {
      mma_ts_imm<1>(tmem + COL_DV, tmem + COL_S + ks * 8, dG + off, idesc_g);
      mma_ts_imm<1>(tmem + COL_DK, tmem + COL_DP + ks * 8, dQm + off, idesc_g);
    }
    if (ks == 0) mma_ss_imm<0>(tmem + COL_DQ, dS + off, dK + off, idesc_q);
    else mma_ss_imm<1>(tmem + COL_DQ, dS + off, dK + off, idesc_q);
  }
}

template <int DT, bool CAUSAL>
__global__ void __launch_bounds__(NTHR, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sm + OFF_K;
  uint8_t* sV = sm + OFF_V;
  uint8_t* sQ = sm + OFF_Q;  // [2][BOX]
  uint8_t* sG = sm + OFF_G;  // [2][BOX] (dO)
  uint8_t* sdS = sm + OFF_DS;
  uint8_t* sdQ = sm + OFF_DQ;  // [2][128 x 64 fp32], two 32-float boxes each, 128-byte swizzle
  float* sLse = reinterpret_cast<float*>(sm + OFF_ROW);  // [2][128], base-2 LSE
  float* sDd = sLse + 2 * BT;                            // [2][128], D_i
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_kv = bars;
  uint64_t* bar_q = bars + 1;  // [2]
  uint64_t* bar_m1 = bars + 3;
  uint64_t* bar_m2 = bars + 4;
  uint64_t* bar_idle = bars + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3;  // tensor-memory lane quarter of this warp
  const int half = warp >> 2;    // query columns [64 half, 64 half + 64) / feature columns [32 half, +32)
  const int bh = blockIdx.x % p.BH, jt = blockIdx.x / p.BH;
  const int b = bh / p.H, h = bh % p.H;
  const int k0 = jt * BT;
  const int it0 = CAUSAL ? jt : 0;
  const int nit = p.n_tiles - it0;  // >= 1
  const unsigned long long tmo = p.timeout_ns;

  if (tid == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(&bars[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmG);
    prefetch_tensormap(&tmDQ);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  // row values (base-2 LSE, D) of a query tile, one thread per row (threads < 128); fetched one step ahead
  auto row_vals = [&](int it, float& l2, float& dd) {
    const long long i = static_cast<long long>(it0 + it) * BT + tid;
    if (tid < BT && it < nit && i < p.N) {
      l2 = p.lse[static_cast<long long>(bh) * p.N + i] * LOG2E;
      dd = p.dvec[static_cast<long long>(bh) * p.N + i];
    } else {
      l2 = INFINITY;  // P = 0 for query rows past the end
      dd = 0.0f;
    }
  };
  {
    float l2, dd;
    row_vals(0, l2, dd);
    if (tid < BT) {
      sLse[tid] = l2;
      sDd[tid] = dd;
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued_q[2] = {0, 0};  // loads issued per slot (thread 0)
  auto load_q = [&](int it) {
    const int slot = it & 1;
    const int i0 = (it0 + it) * BT;
    mbar_arrive_expect_tx(&bar_q[slot], 2 * BOX);
    tma_load_4d(sQ + slot * BOX, &tmQ, &bar_q[slot], 0, i0, h, b);
    tma_load_4d(sG + slot * BOX, &tmG, &bar_q[slot], 0, i0, h, b);
    ++issued_q[slot];
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_kv, 2 * BOX);
    tma_load_4d(sK, &tmK, bar_kv, 0, k0, h, b);
    tma_load_4d(sV, &tmV, bar_kv, 0, k0, h, b);
    load_q(0);
    if (nit > 1) load_q(1);
  }

  constexpr uint32_t IDESC_T = idesc_f16(DT, 0, 128, 128);              // S^T, dP^T
  constexpr uint32_t IDESC_G = idesc_f16(DT, 1, 128, HD);               // dV, dK
  constexpr uint32_t IDESC_Q = idesc_f16(DT, 1, 128, HD) | (1u << 15);  // dQ: A MN-major too
  const uint64_t dK_k = smem_desc_sw128(smem_u32(sK), 16, 1024);
  const uint64_t dV_k = smem_desc_sw128(smem_u32(sV), 16, 1024);
  const uint64_t dK_mn = smem_desc_sw128(smem_u32(sK), 1024, 1024);
  const uint64_t dS_mn = smem_desc_sw128(smem_u32(sdS), BOX, 1024);  // two 64-query boxes along M
  auto dQ_k = [&](int slot) { return smem_desc_sw128(smem_u32(sQ + slot * BOX), 16, 1024); };
  auto dG_k = [&](int slot) { return smem_desc_sw128(smem_u32(sG + slot * BOX), 16, 1024); };
  auto dQ_mn = [&](int slot) { return smem_desc_sw128(smem_u32(sQ + slot * BOX), 1024, 1024); };
  auto dG_mn = [&](int slot) { return smem_desc_sw128(smem_u32(sG + slot * BOX), 1024, 1024); };

  bool ok = true;
  // MMA warp (warp 0, one elected lane): S^T(it) and dP^T(it)
  auto issue_m1 = [&](int it) -> bool {
    bool w = true;
    if (elect_lane()) {
      const int slot = it & 1;
      if (it == 0) w = wait_abort(bar_kv, 0, tmo, abort_flag, kBwdTimeoutLoad, 1);
      if (w) w = wait_abort(&bar_q[slot], static_cast<uint32_t>((it >> 1) & 1), tmo, abort_flag, kBwdTimeoutLoad, 2);
      if (w) {
        tc_fence_after();
        issue_t(tmem + COL_S, dK_k, dQ_k(slot), IDESC_T);
        issue_t(tmem + COL_DP, dV_k, dG_k(slot), IDESC_T);
        tc_commit(bar_m1);
      }
    }
    __syncwarp();
    return __all_sync(0xffffffffu, w);
  };
  if (warp == 0) ok = issue_m1(0);

  const int r = quarter * 32 + lane;  // key row (tensor-memory lane) in the elementwise step, query row in the dQ step
  const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const bool key_ok = k0 + r < p.N;
  const float sl2 = p.scale_log2;
  const uint32_t ds_row = smem_u32(sdS) + static_cast<uint32_t>(half * BOX + r * 128);
  const uint32_t dq_row = smem_u32(sdQ) + static_cast<uint32_t>(half * (BT * 128) + r * 128);
  const int sw = r & 7;
  int dq_groups = 0;  // bulk reductions issued (thread 0)

  for (int it = 0; it < nit; ++it) {
    const int slot = it & 1;
    const int i0 = (it0 + it) * BT;
    float nl2, ndd;
    row_vals(it + 1, nl2, ndd);  // next tile's row values, consumed at the end of this step
    if (ok) ok = wait_abort(bar_m1, static_cast<uint32_t>(it & 1), tmo, abort_flag, kBwdTimeoutMMA, 3);
    ok = __all_sync(0xffffffffu, ok);  // the warp-collective tensor-memory accesses below run warp-uniformly
    // S^T and dP^T of this warp's 64 query columns, all read before any P^T / dS^T is written over them
    uint32_t s[64], g[64];
    if (ok) {
      tc_fence_after();
      tmem_ld32(trow + COL_S + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(trow + COL_S + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld32(trow + COL_DP + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&g[0]));
      tmem_ld32(trow + COL_DP + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&g[32]));
      tmem_wait_ld();
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&g[0]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&g[32]));
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    {
      const bool diag = CAUSAL && (i0 == k0);
      const float* lrow = sLse + slot * BT + half * 64;
      const float* drow = sDd + slot * BT + half * 64;
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {  // 32-query chunk c = 2 half + c2
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int ql = c2 * 32 + 2 * e;  // query within this half
          const int q0 = half * 64 + ql;   // query within the tile
          const float2 l2 = *reinterpret_cast<const float2*>(lrow + ql);
          const float2 dd = *reinterpret_cast<const float2*>(drow + ql);
          float p0 = ex2(fmaf(__uint_as_float(s[ql]), sl2, -l2.x));
          float p1 = ex2(fmaf(__uint_as_float(s[ql + 1]), sl2, -l2.y));
          if (!key_ok) p0 = p1 = 0.0f;
          if (diag) {
            if (r > q0) p0 = 0.0f;
            if (r > q0 + 1) p1 = 0.0f;
          }
          const float d0 = p0 * (__uint_as_float(g[ql]) - dd.x);
          const float d1 = p1 * (__uint_as_float(g[ql + 1]) - dd.y);
          pw[e] = pack_pair(p0, p1, DT);
          dw[e] = pack_pair(d0, d1, DT);
        }
        const int c = 2 * half + c2;
        tmem_st16(trow + COL_S + c * 16, pw);
        tmem_st16(trow + COL_DP + c * 16, dw);
        // dS^T row r, queries [32c, 32c+32): box `half`, 16-byte chunks c2*4 .. +3, 128-byte swizzle
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = c2 * 4 + u;
          st_shared_v4(ds_row + static_cast<uint32_t>((cc ^ sw) * 16), dw[4 * u], dw[4 * u + 1], dw[4 * u + 2],
                       dw[4 * u + 3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
    }
    // the dQ staging slot written below was last read by the reduction issued two steps ago
    if (tid == 0 && dq_groups > 0) bulk_wait_read_le1();
    tc_fence_before();
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;

    // gradients of this step, then S^T and dP^T of the next one (the tensor pipe runs them in order)
    if (warp == 0) {
      bool w = true;
      if (elect_lane()) {
        tc_fence_after();
        if (it == 0)
          issue_grads<1>(tmem, dG_mn(slot), dQ_mn(slot), dS_mn, dK_mn, IDESC_G, IDESC_Q);
        else
          issue_grads<0>(tmem, dG_mn(slot), dQ_mn(slot), dS_mn, dK_mn, IDESC_G, IDESC_Q);
        tc_commit(bar_m2);
      }
      __syncwarp();
      if (it + 1 < nit) w = issue_m1(it + 1);
      ok = w;
    }
    if (ok) ok = wait_abort(bar_m2, static_cast<uint32_t>(it & 1), tmo, abort_flag, kBwdTimeoutMMA, 4);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      // this slot's Q and dO are no longer read: fetch the tile two steps ahead into it
      if (tid == 0 && it + 2 < nit) load_q(it + 2);
      // dQ tile rows (query = tensor-memory lane), feature columns [32 half, 32 half + 32), scaled,
      // into the staging slot in the reduction's 128-byte-swizzled box layout
      uint32_t o[32];
      tmem_ld32(trow + COL_DQ + half * 32, o);
      tmem_wait_ld();
      reg_fence32(o);
      const uint32_t dst = dq_row + static_cast<uint32_t>(slot * DQ_SLOT);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_shared_v4(dst + static_cast<uint32_t>((u ^ sw) * 16), __float_as_uint(__uint_as_float(o[4 * u]) * p.scale),
                     __float_as_uint(__uint_as_float(o[4 * u + 1]) * p.scale),
                     __float_as_uint(__uint_as_float(o[4 * u + 2]) * p.scale),
                     __float_as_uint(__uint_as_float(o[4 * u + 3]) * p.scale));
      fence_proxy_async_smem();
      if (tid < BT) {
        sLse[(slot ^ 1) * BT + tid] = nl2;
        sDd[(slot ^ 1) * BT + tid] = ndd;
      }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    // add the staged dQ tile into the fp32 accumulator (rows past N are clipped by the tensor map)
    if (tid == 0) {
      const uint32_t src = smem_u32(sdQ) + static_cast<uint32_t>(slot * DQ_SLOT);
      tma_reduce_add_3d(src, &tmDQ, 0, i0, bh);
      tma_reduce_add_3d(src + BT * 128, &tmDQ, 32, i0, bh);
      bulk_commit();
      ++dq_groups;
    }
  }

  if (ok) {
    // dV_j and dK_j rows (key row = tensor-memory lane), feature columns [32 half, +32), written once
    tc_fence_after();
    uint32_t a[32], g[32];
    tmem_ld32(trow + COL_DV + half * 32, a);
    tmem_ld32(trow + COL_DK + half * 32, g);
    tmem_wait_ld();
    reg_fence32(a);
    reg_fence32(g);
    if (key_ok) {
      const long long row = static_cast<long long>(bh) * p.N + k0 + r;
      uint4* dv = reinterpret_cast<uint4*>(p.dv + row * HD + half * 32);
      uint4* dk = reinterpret_cast<uint4*>(p.dk + row * HD + half * 32);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint4 wv, wk;
        wv.x = pack_pair(__uint_as_float(a[8 * u]), __uint_as_float(a[8 * u + 1]), DT);
        wv.y = pack_pair(__uint_as_float(a[8 * u + 2]), __uint_as_float(a[8 * u + 3]), DT);
        wv.z = pack_pair(__uint_as_float(a[8 * u + 4]), __uint_as_float(a[8 * u + 5]), DT);
        wv.w = pack_pair(__uint_as_float(a[8 * u + 6]), __uint_as_float(a[8 * u + 7]), DT);
        wk.x = pack_pair(__uint_as_float(g[8 * u]) * p.scale, __uint_as_float(g[8 * u + 1]) * p.scale, DT);
        wk.y = pack_pair(__uint_as_float(g[8 * u + 2]) * p.scale, __uint_as_float(g[8 * u + 3]) * p.scale, DT);
        wk.z = pack_pair(__uint_as_float(g[8 * u + 4]) * p.scale, __uint_as_float(g[8 * u + 5]) * p.scale, DT);
        wk.w = pack_pair(__uint_as_float(g[8 * u + 6]) * p.scale, __uint_as_float(g[8 * u + 7]) * p.scale, DT);
        dv[u] = wv;
        dk[u] = wk;
      }
    }
  }

  // Drain: every issued MMA, TMA load and dQ reduction completes before tensor memory is released and
  // the CTA exits (bounded waits; on the normal path these phases are already complete).
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    if (elect_lane()) {
      tc_commit(bar_idle);
      mbar_wait_bounded(bar_idle, 0, tmo);
    }
    __syncwarp();
  }
  if (tid == 0) {
    mbar_wait_bounded(bar_kv, 0, tmo);
    for (int s2 = 0; s2 < 2; ++s2)
      if (issued_q[s2] > 0) mbar_wait_bounded(&bar_q[s2], static_cast<uint32_t>((issued_q[s2] - 1) & 1), tmo);
    bulk_wait_all();
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// D_i = dO_i . O_i in fp32: eight threads per 64-feature row, one 16-byte load of each per thread.
template <int DT>
__global__ void __launch_bounds__(256) bwd_dot_kernel(const uint4* o, const uint4* g, float* dvec, long long rows) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = t >> 3;
  float acc = 0.0f;
  if (row < rows) {
    const uint4 a = __ldg(o + t), c = __ldg(g + t);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 x = unpack_pair(aw[u], DT), y = unpack_pair(cw[u], DT);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (row < rows && (t & 7) == 0) dvec[row] = acc;
}

// fp32 dQ accumulator -> input dtype, four elements per thread.
template <int DT>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float4* acc, uint2* dq, long long n4) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 v = acc[i];
    dq[i] = make_uint2(pack_pair(v.x, v.y, DT), pack_pair(v.z, v.w, DT));
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int encode_map(CUtensorMap* m, CUtensorMapDataType type, cuuint32_t rank, const void* base, const cuuint64_t* dims,
               const cuuint64_t* strides, const cuuint32_t* box) {
  static EncodeTiledFn enc = nullptr;
  if (!enc) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      enc = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return CQSA_ERR_CUDA;
  }
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, type, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return CQSA_ERR_CUDA;
  }
  return CQSA_OK;
}

// [B,H,N,64] 16-bit tensor: dims (64, N, H, B), box (64, 128, 1, 1), 128-byte swizzle, zero fill.
int make_bhnd_map(CUtensorMap* m, const void* base, int dtype, int B, int H, int N) {
  const cuuint64_t es = 2;
  const cuuint64_t dims[4] = {HD, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {HD * es, static_cast<cuuint64_t>(N) * HD * es,
                                 static_cast<cuuint64_t>(H) * N * HD * es};
  const cuuint32_t box[4] = {64, BT, 1, 1};
  return encode_map(m, dtype == CQSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    base, dims, strides, box);
}

// fp32 dQ accumulator [BH, N, 64]: dims (64, N, BH), box (32, 128, 1) (128-byte rows), 128-byte swizzle.
int make_dq_map(CUtensorMap* m, float* base, int BH, int N) {
  const cuuint64_t dims[3] = {HD, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {HD * 4, static_cast<cuuint64_t>(N) * HD * 4};
  const cuuint32_t box[3] = {32, BT, 1};
  return encode_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box);
}

template <int DT, bool CAUSAL>
int launch_main(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mg,
                const CUtensorMap& mdq, const BwdParams& p, cudaStream_t s) {
  auto kern = attn_bwd_kernel<DT, CAUSAL>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(attention backward smem)");
    attr_done = true;
  }
  const long long grid = static_cast<long long>(p.n_tiles) * p.BH;
  kern<<<static_cast<unsigned>(grid), NTHR, SMEM_BYTES, s>>>(mq, mk, mv, mg, mdq, p);
  return cuda_status(cudaGetLastError(), "attention backward kernel launch");
}

}  // namespace

size_t attention_bwd_workspace(int B, int H, int N, int d) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t dq = (rows * d * sizeof(float) + 255) & ~size_t(255);
  return dq + rows * sizeof(float);
}

int launch_attention_bwd(const BwdArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.N;
  const long long n_tiles = (a.N + BT - 1) / BT;
  if (n_tiles * a.B * a.H > 0x7fffffffLL) {
    set_error("problem too large for one launch");
    return CQSA_ERR_UNSUPPORTED;
  }
  float* dq_acc = static_cast<float*>(a.workspace);
  float* dvec = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) +
                                         ((static_cast<size_t>(rows) * HD * sizeof(float) + 255) & ~size_t(255)));
  CUtensorMap mq, mk, mv, mg, mdq;
  int rc = make_bhnd_map(&mq, a.q, a.dtype, a.B, a.H, a.N);
  if (rc == CQSA_OK) rc = make_bhnd_map(&mk, a.k, a.dtype, a.B, a.H, a.N);
  if (rc == CQSA_OK) rc = make_bhnd_map(&mv, a.v, a.dtype, a.B, a.H, a.N);
  if (rc == CQSA_OK) rc = make_bhnd_map(&mg, a.dout, a.dtype, a.B, a.H, a.N);
  if (rc == CQSA_OK) rc = make_dq_map(&mdq, dq_acc, a.B * a.H, a.N);
  if (rc != CQSA_OK) return rc;

  // D_i, then the zeroed dQ accumulator, the main kernel and the dQ conversion
  const long long dot_threads = rows * 8;
  const unsigned dot_blocks = static_cast<unsigned>((dot_threads + 255) / 256);
  if (a.dtype == CQSA_BF16)
    bwd_dot_kernel<1><<<dot_blocks, 256, 0, stream>>>(static_cast<const uint4*>(a.out),
                                                      static_cast<const uint4*>(a.dout), dvec, rows);
  else
    bwd_dot_kernel<0><<<dot_blocks, 256, 0, stream>>>(static_cast<const uint4*>(a.out),
                                                      static_cast<const uint4*>(a.dout), dvec, rows);
  rc = cuda_status(cudaGetLastError(), "attention backward dot kernel launch");
  if (rc != CQSA_OK) return rc;
  rc = cuda_status(cudaMemsetAsync(dq_acc, 0, static_cast<size_t>(rows) * HD * sizeof(float), stream),
                   "zero dQ accumulator");
  if (rc != CQSA_OK) return rc;

  BwdParams p;
  p.lse = a.lse;
  p.dvec = dvec;
  p.dq_acc = dq_acc;
  p.dk = static_cast<uint16_t*>(a.dk);
  p.dv = static_cast<uint16_t*>(a.dv);
  p.H = a.H;
  p.BH = a.B * a.H;
  p.N = a.N;
  p.n_tiles = static_cast<int>(n_tiles);
  p.scale = a.scale;
  p.scale_log2 = a.scale * LOG2E;
  p.timeout_ns = timeout_ns();
  if (a.dtype == CQSA_BF16)
    rc = a.causal ? launch_main<1, true>(mq, mk, mv, mg, mdq, p, stream)
                  : launch_main<1, false>(mq, mk, mv, mg, mdq, p, stream);
  else
    rc = a.causal ? launch_main<0, true>(mq, mk, mv, mg, mdq, p, stream)
                  : launch_main<0, false>(mq, mk, mv, mg, mdq, p, stream);
  if (rc != CQSA_OK) return rc;

  const long long n4 = rows * HD / 4;
  const unsigned cblocks = static_cast<unsigned>(std::min<long long>((n4 + 255) / 256, 152LL * 16));
  if (a.dtype == CQSA_BF16)
    bwd_dq_kernel<1><<<cblocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(dq_acc), static_cast<uint2*>(a.dq), n4);
  else
    bwd_dq_kernel<0><<<cblocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(dq_acc), static_cast<uint2*>(a.dq), n4);
  return cuda_status(cudaGetLastError(), "attention backward dQ kernel launch");
}

int bwd_error_word(DevErr* out, int clear) {
  int rc = cuda_status(cudaMemcpyFromSymbol(out, g_bwd_err, sizeof(DevErr)), "read backward error word");
  if (rc != CQSA_OK || !clear || out->code == 0) return rc;
  DevErr z = {0, 0, 0, 0};
  return cuda_status(cudaMemcpyToSymbol(g_bwd_err, &z, sizeof(z)), "clear backward error word");
}

}  // namespace cqsa
