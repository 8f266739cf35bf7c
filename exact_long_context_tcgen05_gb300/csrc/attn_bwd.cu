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
//   bwd_dot_kernel   D_i in fp32 (d / 8 threads per row, 16-byte loads of O and dO)
//   attn_bwd_kernel  one CTA per (key tile j of 128 keys, batch-head), heaviest key tiles first. K_j
//                    and V_j stay in shared memory; Q_i and dO_i of the query tiles that see key
//                    tile j (every i, or i >= j when causal) stream through a two-slot TMA ring.
//                    Per query tile, with the key dimension on the 128 tensor-memory lanes:
//                      S^T = K_j Q_i^T, dP^T = V_j dO_i^T         (tcgen05, fp32 in tensor memory)
//                      P^T and dS^T: one thread per key row and 32 queries (d = 128: 64), in registers; P^T goes
//                                    to tensor memory, dS^T to a 128-byte-swizzled shared tile
//                      dV_j += P^T dO_i                           (A operand from tensor memory)
//                      dK_j += dS^T Q_i, dQ_i = dS K_j            (the dS^T tile read K-major / MN-major)
//                    The dQ tile is scaled, staged in shared memory and added into an fp32
//                    accumulator by TMA bulk reduce-add. S^T and dP^T of the next tile are computed
//                    while the elementwise warps work on the current one. Roles: a TMA producer warp,
//                    an MMA issuer warp (d = 64: a second one for dQ), a dQ reduction warp and four
//                    (d = 128: two) elementwise warpgroups, joined by mbarriers. dK_j, dV_j are written once, after the last
//                    query tile.
//   bwd_dq_kernel    fp32 dQ accumulator -> dQ in the input dtype
// P and dS enter the MMAs rounded to the input dtype; everything else is fp32. Head dimension 64 or 128
// (d = 128 holds one Q/dO tile instead of two, and shares tensor and shared memory between phases: see
// BwdCfg).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "cqsa_internal.h"
#include "sm103_ptx.cuh"

#ifndef CQSA_BWD_GROUP_MB
#define CQSA_BWD_GROUP_MB 48
#endif

namespace cqsa {
namespace {

__device__ DevErr g_bwd_err;

constexpr int BT = 128;                         // keys per CTA tile, queries per step
constexpr uint32_t BOX = BT * 64 * 2;           // one 128 x 64 box of 16-bit elements (16 KiB)
constexpr uint32_t TMEM_COLS = 512;
constexpr int NBAR = 17;

// Shared- and tensor-memory layout per head dimension.
// d = 64: K, V, a three-slot ring of Q and dO tiles (the tile two steps ahead loads while a step's
//   products run: with two slots its load waited for them, ~0.3 us a step), the dS^T tile, two dQ
//   staging slots of 128 x 64 fp32 and the row values (226 KiB, with no slack: the kernel checks that
//   the dynamic shared memory base is 1024-byte aligned). Tensor memory: S^T, dP^T, dV, dK, dQ and
//   P^T (16-bit pairs), 512 columns.
// d = 128: every 128-row tile is two boxes, so K, V, one Q and one dO tile and dS^T take 160 KiB; dQ
//   (128 x 128 fp32, 64 KiB) is staged over the dS^T tile and the 32 KiB behind it once the step's
//   products have read dS^T. Q and dO have their own load and release barriers (bar_q[0] / bar_q[1],
//   bar_qfree[0] / bar_qfree[1]), released after dK and after dV, so each reloads as early as it can. Tensor memory: S^T 0-127 (each warpgroup writes its P^T over the first
//   half of its own S^T columns), dP^T 128-255 (dQ is accumulated over it after dS is formed), dV
//   256-383, dK 384-511.
template <int HD>
struct BwdCfg {
  static constexpr int NSLOT = HD == 64 ? 3 : 1;          // Q/dO ring slots
  static constexpr uint32_t TILE = BOX * (HD / 64);       // one 128-row tile of Q, dO, K or V
  static constexpr uint32_t OFF_K = 0, OFF_V = TILE, OFF_Q = 2 * TILE;
  static constexpr uint32_t OFF_G = OFF_Q + NSLOT * TILE;
  static constexpr uint32_t OFF_DS = OFF_G + NSLOT * TILE;  // dS^T: two 64-query boxes
  static constexpr uint32_t OFF_DQ = OFF_DS + 2 * BOX;
  static constexpr uint32_t DQ_SLOT = BT * 64 * 4;        // d = 64: one staging slot (128 x 64 fp32)
  static constexpr uint32_t OFF_ROW = HD == 64 ? OFF_DQ + 2 * DQ_SLOT : OFF_DQ + 2 * BOX;
  // row values: per elementwise warpgroup and slot, lse2 and D of the step's 128 / NWG queries (2 KiB)
  static constexpr uint32_t OFF_BAR = OFF_ROW + 2 * 2 * 128 * 4;
  // the dynamic shared memory base is 1024-byte aligned (the kernel checks, and stops with an error if not)
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + NBAR * 8 + 16;
  static constexpr uint32_t COL_S = 0, COL_DP = 128;
  static constexpr uint32_t COL_DV = 256, COL_DK = 256 + HD;
  static constexpr uint32_t COL_DQ = HD == 64 ? 384 : 128;
  static_assert(SMEM_BYTES <= 232448, "shared memory exceeds 227 KiB");
  static_assert(COL_DK + HD <= TMEM_COLS, "tensor memory exceeds 512 columns");
  // P^T column of query k-step ks (16 queries = 8 columns of 16-bit pairs)
  static __device__ __forceinline__ uint32_t col_pt(int ks) {
    return HD == 64 ? 448u + static_cast<uint32_t>(ks) * 8u
                    : static_cast<uint32_t>((ks >> 2) * 64 + (ks & 3) * 8);
  }
};
constexpr float LOG2E = 1.4426950408889634f;
// 16 columns of 32 lanes (thread t of the warp receives lane base + t), and the matching register pin.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}
// Warp roles: warpgroup 0 = TMA producer (warp 0), MMA issuer and tensor-memory owner (warp 1), dQ
// reductions (warp 2), the dQ products' issuer at d = 64 (warp 3; idle at d = 128); then the
// elementwise warpgroups, each on an equal share of the step's 128 query columns, so each tensor-memory
// lane quarter (SM sub-partition) interleaves one warp of each: four at d = 64 (32 columns each; 640
// threads), two at d = 128 (64 each; 384 threads, whose tensor and shared memory leave no room for
// more). setmaxnreg splits the launch's registers between warpgroup 0 and the elementwise warpgroups:
// d = 64, 128 * 64 + 512 * 104 <= 640 * 96; d = 128, 128 * 152 + 256 * 176 = 384 * 168. (Two warpgroups
// at d = 64: 860 TFLOP/s on the 32K causal backward; four: 913, with 104 registers; four with 96: 888.
// At d = 128 warpgroup 0's unrolled product issue spilled below ~150 registers: 96 / 200 spilled 350
// bytes, 152 / 176 none, 960 -> 1,002 TFLOP/s on the 32K causal backward.)
template <int HD>
struct BwdThreads {
  static constexpr int NWG = HD == 64 ? 4 : 2;
  static constexpr int NTHR = 128 * (NWG + 1);
  static constexpr int LOW = HD == 64 ? 64 : 152, HIGH = HD == 64 ? 104 : 176;
  static constexpr int LAUNCH_REGS = HD == 64 ? 96 : 168;
  static_assert(128 * LOW + 128 * NWG * HIGH <= NTHR * LAUNCH_REGS, "register split exceeds the launch allocation");
};

enum : int { kBwdTimeoutLoad = 1, kBwdTimeoutMMA = 3, kBwdTimeoutSoftmax = 4 };

struct BwdParams {
  const float* lse;       // [BH, Nq] natural-log LSE of the forward (over every key of the row)
  const float* dvec;      // [BH, Nq] D_i
  float* dq_acc;          // [BH, Nq, 64] fp32; receives scale * dS K (added)
  uint16_t* dk;           // [BH, Nkv, 64] input dtype (monolithic mode: written)
  uint16_t* dv;
  float* dk_acc;          // [BH, Nkv, 64] fp32 (chunk-pair mode: scale * dS^T Q added)
  float* dv_acc;          // [BH, Nkv, 64] fp32 (chunk-pair mode: P^T dO added)
  int H, BH, Nq, Nkv, n_q_tiles;
  long long q_off, kv_off;  // absolute positions of the chunks' first query / key (causal mask)
  float scale, scale_log2;
  unsigned long long timeout_ns;
  int fault;  // test hook: 2 = block 0 never loads its key/value tile (its waits must time out cleanly)
  int head_group;  // heads whose key tiles are interleaved; the rest follow group by group
  int n_kv_tiles;
};

__device__ __forceinline__ void record_bwd_error(int code, int where) {
  if (atomicCAS(&g_bwd_err.code, 0, code) == 0) {
    g_bwd_err.block = blockIdx.x;
    g_bwd_err.where = where;
  }
}

// Bounded wait that returns early once another thread of the CTA has given up.
// (32-bit shared-window addresses for the barrier and the abort flag: fewer live registers in the
// issuer warp, which runs at 64 registers.)
__device__ __forceinline__ bool wait_abort_a(uint32_t bar, uint32_t parity, unsigned long long tmo, uint32_t abort_a,
                                             int code, int where) {
  if (mbar_try_wait_a(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait_a(bar, parity)) return true;
    if ((++spins & 15u) == 0) {
      if (ld_shared_volatile_u32(abort_a)) return false;
      if (globaltimer_ns() - t0 > tmo) {
        record_bwd_error(code, where);
        st_shared_volatile_u32(abort_a, 1u);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_abort(uint64_t* bar, uint32_t parity, unsigned long long tmo,
                                           volatile int* abort_flag, int code, int where) {
  return wait_abort_a(smem_u32(bar), parity, tmo, smem_u32(const_cast<int*>(abort_flag)), code, where);
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
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
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

// S^T = K Q^T (or dP^T = V dO^T): d/16 MMAs of 128 x 128 x 16, both operands K-major, 128-byte swizzle;
// features 64..127 of d = 128 are in each tile's second box.
template <int HD>
__device__ __forceinline__ void issue_t(uint32_t dcol, uint64_t a0, uint64_t b0, uint32_t idesc) {
  mma_ss_imm<0>(dcol, a0, b0, idesc);
#pragma unroll
  for (int ks = 1; ks < HD / 16; ++ks) {
    const uint32_t off = static_cast<uint32_t>((ks >> 2) * (BOX >> 4) + (ks & 3) * 2);
    mma_ss_imm<1>(dcol, a0 + off, b0 + off, idesc);
  }
}

// dV += P^T dO (A = P^T from tensor memory), dK += dS^T Q (A = dS^T K-major in shared memory) and
// dQ = dS K (A = the same dS^T tile read MN-major): 8 steps of 16 queries (dV, dK) or keys (dQ); the
// B operands dO, Q and K are MN-major with N = d (the second 64-feature box at the descriptor's
// leading-byte offset when d = 128).
template <int FIRST, int HD, bool DQ>
__device__ __forceinline__ void issue_grads(uint32_t tmem, uint64_t dG, uint64_t dQm, uint64_t dS_k, uint64_t dS_mn,
                                            uint64_t dK, uint32_t idesc_g, uint32_t idesc_q) {
  using C = BwdCfg<HD>;
#pragma unroll
  for (int ks = 0; ks < BT / 16; ++ks) {
    const uint32_t off = static_cast<uint32_t>(ks * (2048 >> 4));                        // 16 rows of 128 bytes
    const uint32_t koff = static_cast<uint32_t>((ks >> 2) * (BOX >> 4) + (ks & 3) * 2);  // 16 columns, K-major
    if (FIRST && ks == 0) {
      mma_ts_imm<0>(tmem + C::COL_DV, tmem + C::col_pt(ks), dG + off, idesc_g);
      mma_ss_imm<0>(tmem + C::COL_DK, dS_k + koff, dQm + off, idesc_g);
    } else {
      mma_ts_imm<1>(tmem + C::COL_DV, tmem + C::col_pt(ks), dG + off, idesc_g);
      mma_ss_imm<1>(tmem + C::COL_DK, dS_k + koff, dQm + off, idesc_g);
    }
    if (DQ) {
      if (ks == 0) mma_ss_imm<0>(tmem + C::COL_DQ, dS_mn + off, dK + off, idesc_q);
      else mma_ss_imm<1>(tmem + C::COL_DQ, dS_mn + off, dK + off, idesc_q);
    }
  }
}

// ACCUM = 0: monolithic (dK, dV written in the input dtype); ACCUM = 1: one chunk pair, dK and dV
// added into fp32 accumulators.
template <int DT, bool CAUSAL, int ACCUM, int HD>
__global__ void __launch_bounds__(BwdThreads<HD>::NTHR, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BwdCfg<HD>;
  using TH = BwdThreads<HD>;
  constexpr int NWG = TH::NWG;
  constexpr int QC = 128 / NWG;  // query columns of a warpgroup
  constexpr int CW = NWG == 4 ? 16 : 32;  // columns per tensor-memory load
  constexpr int NSLOT = C::NSLOT;
  constexpr uint32_t TILE = C::TILE;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the 128-byte swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) record_bwd_error(kDevMisaligned, 0);
    return;
  }
  uint8_t* sm = smem_raw;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint8_t* sQ = sm + C::OFF_Q;    // [NSLOT][TILE]
  uint8_t* sG = sm + C::OFF_G;    // [NSLOT][TILE] (dO)
  uint8_t* sdS = sm + C::OFF_DS;  // dS^T [128 keys][128 queries], two 64-query boxes
  // dQ staging: d = 64, two slots of 128 x 64 fp32 (two 32-float boxes each); d = 128, one 128 x 128 fp32
  // tile in four 32-float boxes over dS^T and the 32 KiB behind it
  uint8_t* sdQ = HD == 64 ? sm + C::OFF_DQ : sdS;
  float* sRow = reinterpret_cast<float*>(sm + C::OFF_ROW);  // per elementwise warp: [slot 2][lse2 | D]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* bar_kv = bars + 0;
  uint64_t* bar_q = bars + 1;       // [3] Q/dO slot loaded (d = 128: [0] Q, [1] dO)
  uint64_t* bar_qfree = bars + 4;   // [3] Q/dO slot read by every MMA (commit)
  uint64_t* bar_m1 = bars + 7;      // S^T, dP^T ready (commit)
  uint64_t* bar_m2 = bars + 8;      // dV, dK, dQ products done (commit)
  uint64_t* bar_sfree = bars + 9;   // S^T, dP^T read into registers (256 elementwise threads)
  uint64_t* bar_ready = bars + 10;  // P^T and dS^T written, previous dQ read out (256 threads)
  uint64_t* bar_staged = bars + 11; // [2] dQ staging slot written (256 threads); d = 128: slot 0 only, and it
                                    // also tells the MMA issuer that dQ has left the dP^T columns
  uint64_t* bar_dqfree = bars + 13; // [2] dQ staging slot read by its reduction
  uint64_t* bar_idle = bars + 15;   // every MMA done (commit)
  uint64_t* bar_idle3 = bars + 16;  // d = 64: every dQ product of warp 3 done (commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Key tiles of head_group heads at a time, heaviest (first) key tiles first within a group, so that the
  // fp32 dQ accumulators and the Q / dO tiles of the heads in flight stay in L2.
  const int unit = static_cast<int>(blockIdx.x);
  const int per_group = p.head_group * p.n_kv_tiles;
  const int g0 = (unit / per_group) * p.head_group;
  const int gn = min(p.head_group, p.BH - g0);
  const int ur = unit - (unit / per_group) * per_group;
  const int bh = g0 + ur % gn, jt = ur / gn;
  const int b = bh / p.H, h = bh % p.H;
  const int k0 = jt * BT;
  const int Nkv = ACCUM ? p.Nkv : p.Nq;
  // first query tile with a query at or after this key tile's first key (causal; absolute positions)
  int it0 = 0;
  if constexpr (ACCUM) {
    if (CAUSAL) {
      const long long first = p.kv_off + k0 - p.q_off - (BT - 1);
      it0 = first <= 0 ? 0 : static_cast<int>(first / BT + (first % BT != 0));
    }
  } else {
    it0 = CAUSAL ? jt : 0;
  }
  const int nit = p.n_q_tiles - it0;  // >= 1 for the monolithic call
  const unsigned long long tmo = p.timeout_ns;
  if constexpr (ACCUM) {
    if (nit <= 0) return;  // every key of this tile lies after every query of the chunk: nothing to add
  }

  if (tid == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bar_q[s], 1);
      mbar_init(&bar_qfree[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_staged[s], NWG * 128);
      mbar_init(&bar_dqfree[s], 1);
    }
    mbar_init(bar_m1, 1);
    mbar_init(bar_m2, HD == 64 ? 2 : 1);  // d = 64: dV / dK (warp 1) and dQ (warp 3) commit separately
    mbar_init(bar_sfree, NWG * 128);
    mbar_init(bar_ready, NWG * 128);
    mbar_init(bar_idle, 1);
    mbar_init(bar_idle3, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(TH::LOW));
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmG);
      int issued[3] = {0, 0, 0};
      auto load_q = [&](int it) {
        const int slot = it % NSLOT;
        mbar_arrive_expect_tx(&bar_q[slot], 2 * TILE);
#pragma unroll
        for (int x = 0; x < HD / 64; ++x) {
          tma_load_4d(sQ + slot * TILE + x * BOX, &tmQ, &bar_q[slot], x * 64, (it0 + it) * BT, h, b);
          tma_load_4d(sG + slot * TILE + x * BOX, &tmG, &bar_q[slot], x * 64, (it0 + it) * BT, h, b);
        }
        ++issued[slot];
      };
      const bool skip_kv = (p.fault == 2 && blockIdx.x == 0);  // fault injection: K/V never arrive
      if (!skip_kv) {
        mbar_arrive_expect_tx(bar_kv, 2 * TILE);
#pragma unroll
        for (int x = 0; x < HD / 64; ++x) {
          tma_load_4d(sK + x * BOX, &tmK, bar_kv, x * 64, k0, h, b);
          tma_load_4d(sV + x * BOX, &tmV, bar_kv, x * 64, k0, h, b);
        }
      }
      if constexpr (HD == 64) {
        for (int it = 0; it < NSLOT && it < nit; ++it) load_q(it);
        for (int it = 0; it + NSLOT < nit; ++it) {
          // slot it % NSLOT is free once every MMA of step it has read it
          if (!wait_abort(&bar_qfree[it % NSLOT], static_cast<uint32_t>((it / NSLOT) & 1), tmo, abort_flag,
                          kBwdTimeoutLoad, 5))
            break;
          load_q(it + NSLOT);
        }
      } else {
        // d = 128, one tile each: dO (bar_q[1]) is refilled once dV of the step has read it, Q (bar_q[0])
        // once dK has; the issuer commits the two releases separately (bar_qfree[1], bar_qfree[0])
        auto load_one = [&](int it, int which) {
          uint8_t* dst = which ? sG : sQ;
          const CUtensorMap* map = which ? &tmG : &tmQ;
          mbar_arrive_expect_tx(&bar_q[which], TILE);
#pragma unroll
          for (int x = 0; x < HD / 64; ++x)
            tma_load_4d(dst + x * BOX, map, &bar_q[which], x * 64, (it0 + it) * BT, h, b);
          ++issued[which];
        };
        if (nit > 0) {
          load_one(0, 0);
          load_one(0, 1);
        }
        for (int it = 0; it + 1 < nit; ++it) {
          if (!wait_abort(&bar_qfree[1], static_cast<uint32_t>(it & 1), tmo, abort_flag, kBwdTimeoutLoad, 5)) break;
          load_one(it + 1, 1);
          if (!wait_abort(&bar_qfree[0], static_cast<uint32_t>(it & 1), tmo, abort_flag, kBwdTimeoutLoad, 5)) break;
          load_one(it + 1, 0);
        }
      }
      // every load issued lands before the CTA exits (bounded waits)
      if (!skip_kv) mbar_wait_bounded(bar_kv, 0, tmo);
      for (int s = 0; s < 3; ++s)
        if (issued[s] > 0) mbar_wait_bounded(&bar_q[s], static_cast<uint32_t>((issued[s] - 1) & 1), tmo);
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t IDESC_T = idesc_f16(DT, 0, 128, 128);              // S^T, dP^T
      constexpr uint32_t IDESC_V = idesc_f16(DT, 1, 128, HD);               // dV: A (P^T) in TMEM, B MN-major
      constexpr uint32_t IDESC_Q = idesc_f16(DT, 1, 128, HD) | (1u << 15);  // dQ: A (dS) MN-major
      const bool leader = elect_lane();
      // descriptors, prepared by the whole warp before any issue; MN-major operands with N = d reach the
      // second 64-feature box of d = 128 through the leading-byte offset
      constexpr uint32_t LBO_MN = HD == 64 ? 1024u : BOX;
      const uint64_t dK_k = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV_k = smem_desc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dK_mn = smem_desc_sw128(smem_u32(sK), LBO_MN, 1024);
      const uint64_t dS_k = smem_desc_sw128(smem_u32(sdS), 16, 1024);     // dS^T as K-major A (M = keys)
      const uint64_t dS_mn = smem_desc_sw128(smem_u32(sdS), BOX, 1024);   // dS^T as MN-major A (M = queries)
      const uint64_t dQ0_k = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dG0_k = smem_desc_sw128(smem_u32(sG), 16, 1024);
      const uint64_t dQ0_mn = smem_desc_sw128(smem_u32(sQ), LBO_MN, 1024);
      const uint64_t dG0_mn = smem_desc_sw128(smem_u32(sG), LBO_MN, 1024);
      constexpr uint32_t SLOT16 = TILE >> 4;  // one slot in descriptor address units
      auto wait_all = [&](uint64_t* bar, uint32_t parity, int code, int where) -> bool {
        const bool w = wait_abort(bar, parity, tmo, abort_flag, code, where);
        return __all_sync(0xffffffffu, w);
      };
      auto issue_m1 = [&](int it) {
        const uint32_t so = static_cast<uint32_t>(it % NSLOT) * SLOT16;
        tc_fence_after();
        if (leader) {
          issue_t<HD>(tmem + C::COL_S, dK_k, dQ0_k + so, IDESC_T);
          issue_t<HD>(tmem + C::COL_DP, dV_k, dG0_k + so, IDESC_T);
          tc_commit(bar_m1);
        }
        __syncwarp();
      };
      auto issue_m2 = [&](int it) {
        const uint32_t so = static_cast<uint32_t>(it % NSLOT) * SLOT16;
        tc_fence_after();
        if (leader) {
          if (it == 0) issue_grads<1, HD, HD != 64>(tmem, dG0_mn + so, dQ0_mn + so, dS_k, dS_mn, dK_mn, IDESC_V, IDESC_Q);
          else issue_grads<0, HD, HD != 64>(tmem, dG0_mn + so, dQ0_mn + so, dS_k, dS_mn, dK_mn, IDESC_V, IDESC_Q);
          tc_commit(bar_m2);
          tc_commit(&bar_qfree[it % NSLOT]);
        }
        __syncwarp();
      };
      // d = 128: the three gradient products one after another, with the release of dO (after dV) and of
      // Q (after dK) committed in between, so that the producer refills each as early as possible
      auto issue_grads_128 = [&](int it) {
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < BT / 16; ++ks) {
            const uint32_t off = static_cast<uint32_t>(ks * (2048 >> 4));
            if (it == 0 && ks == 0) mma_ts_imm<0>(tmem + C::COL_DV, tmem + C::col_pt(ks), dG0_mn + off, IDESC_V);
            else mma_ts_imm<1>(tmem + C::COL_DV, tmem + C::col_pt(ks), dG0_mn + off, IDESC_V);
          }
          tc_commit(&bar_qfree[1]);
#pragma unroll
          for (int ks = 0; ks < BT / 16; ++ks) {
            const uint32_t off = static_cast<uint32_t>(ks * (2048 >> 4));
            const uint32_t koff = static_cast<uint32_t>((ks >> 2) * (BOX >> 4) + (ks & 3) * 2);
            if (it == 0 && ks == 0) mma_ss_imm<0>(tmem + C::COL_DK, dS_k + koff, dQ0_mn + off, IDESC_V);
            else mma_ss_imm<1>(tmem + C::COL_DK, dS_k + koff, dQ0_mn + off, IDESC_V);
          }
          tc_commit(&bar_qfree[0]);
#pragma unroll
          for (int ks = 0; ks < BT / 16; ++ks) {
            const uint32_t off = static_cast<uint32_t>(ks * (2048 >> 4));
            if (ks == 0) mma_ss_imm<0>(tmem + C::COL_DQ, dS_mn + off, dK_mn + off, IDESC_Q);
            else mma_ss_imm<1>(tmem + C::COL_DQ, dS_mn + off, dK_mn + off, IDESC_Q);
          }
          tc_commit(bar_m2);
        }
        __syncwarp();
      };
      auto issue_s_128 = [&]() {  // S^T of the next step, behind this thread's dV (P^T is over S^T)
        tc_fence_after();
        if (leader) issue_t<HD>(tmem + C::COL_S, dK_k, dQ0_k, IDESC_T);
        __syncwarp();
      };
      auto issue_dp_128 = [&]() {  // dP^T of the next step, over the dQ columns once dQ is staged out
        tc_fence_after();
        if (leader) {
          issue_t<HD>(tmem + C::COL_DP, dV_k, dG0_k, IDESC_T);
          tc_commit(bar_m1);
        }
        __syncwarp();
      };
      bool ok = wait_all(bar_kv, 0, kBwdTimeoutLoad, 1);
      if (ok) ok = wait_all(&bar_q[0], 0, kBwdTimeoutLoad, 2);
      if (HD == 128 && ok) ok = wait_all(&bar_q[1], 0, kBwdTimeoutLoad, 2);
      if (ok) issue_m1(0);
      for (int it = 0; ok && it < nit; ++it) {
        if constexpr (HD == 64) {
          if (it + 1 < nit) {
            // S^T / dP^T of step it are in registers: the next step's products may overwrite them
            ok = wait_all(bar_sfree, static_cast<uint32_t>(it & 1), kBwdTimeoutSoftmax, 6);
            if (ok) ok = wait_all(&bar_q[(it + 1) % NSLOT], static_cast<uint32_t>(((it + 1) / NSLOT) & 1), kBwdTimeoutLoad, 2);
            if (ok) issue_m1(it + 1);
          }
          if (ok) ok = wait_all(bar_ready, static_cast<uint32_t>(it & 1), kBwdTimeoutSoftmax, 7);
          if (ok) issue_m2(it);
        } else {
          // d = 128: the gradient products of step it first (dV reads P^T from the S^T columns before the
          // next S^T is issued behind it by this thread); the next step's S^T and dP^T once the single
          // Q/dO slot holds step it + 1 and dQ of step it has left the dP^T columns
          ok = wait_all(bar_ready, static_cast<uint32_t>(it & 1), kBwdTimeoutSoftmax, 7);
          if (ok) issue_grads_128(it);
          if (ok && it + 1 < nit) {
            ok = wait_all(&bar_q[0], static_cast<uint32_t>((it + 1) & 1), kBwdTimeoutLoad, 2);
            if (ok) issue_s_128();
            if (ok) ok = wait_all(&bar_staged[0], static_cast<uint32_t>(it & 1), kBwdTimeoutSoftmax, 10);
            if (ok) ok = wait_all(&bar_q[1], static_cast<uint32_t>((it + 1) & 1), kBwdTimeoutLoad, 2);
            if (ok) issue_dp_128();
          }
        }
      }
      if (leader) tc_commit(bar_idle);
      __syncwarp();
      mbar_wait_bounded(bar_idle, 0, tmo);
    } else if (warp == 2 && lane == 0) {
      // ---------------------------------------------------------------- dQ reductions
      for (int it = 0; it < nit; ++it) {
        const int slot = HD == 64 ? (it & 1) : 0;
        const uint32_t par = static_cast<uint32_t>(HD == 64 ? ((it >> 1) & 1) : (it & 1));
        if (!wait_abort(&bar_staged[slot], par, tmo, abort_flag, kBwdTimeoutSoftmax, 8)) break;
        const uint32_t src = smem_u32(sdQ) + static_cast<uint32_t>(slot * C::DQ_SLOT);
#pragma unroll
        for (int x = 0; x < HD / 32; ++x) tma_reduce_add_3d(src + x * (BT * 128), &tmDQ, 32 * x, (it0 + it) * BT, bh);
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(&bar_dqfree[slot]);
      }
      bulk_wait_all();
    } else if (HD == 64 && warp == 3) {
      // ---------------------------------------------------------------- dQ products (d = 64)
      // dQ = dS K of each step, issued beside warp 1's dV / dK (each issuing warp shares its sub-partition
      // with four elementwise warps, so the step's 24 small products are issued from two of them); dQ of
      // the previous step has left tensor memory once the step's P^T / dS^T hand-off has arrived
      constexpr uint32_t IDESC_Q = idesc_f16(DT, 1, 128, HD) | (1u << 15);
      const bool leader = elect_lane();
      const uint64_t dK_mn = smem_desc_sw128(smem_u32(sK), 1024u, 1024);
      const uint64_t dS_mn = smem_desc_sw128(smem_u32(sdS), BOX, 1024);
      bool ok = __all_sync(0xffffffffu, wait_abort(bar_kv, 0, tmo, abort_flag, kBwdTimeoutLoad, 1));
      for (int it = 0; ok && it < nit; ++it) {
        ok = __all_sync(0xffffffffu,
                        wait_abort(bar_ready, static_cast<uint32_t>(it & 1), tmo, abort_flag, kBwdTimeoutSoftmax, 7));
        if (!ok) break;
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < BT / 16; ++ks) {
            const uint32_t off = static_cast<uint32_t>(ks * (2048 >> 4));
            if (ks == 0) mma_ss_imm<0>(tmem + C::COL_DQ, dS_mn + off, dK_mn + off, IDESC_Q);
            else mma_ss_imm<1>(tmem + C::COL_DQ, dS_mn + off, dK_mn + off, IDESC_Q);
          }
          tc_commit(bar_m2);
        }
        __syncwarp();
      }
      if (leader) tc_commit(bar_idle3);
      __syncwarp();
      mbar_wait_bounded(bar_idle3, 0, tmo);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(TH::HIGH));
    // ------------------------------------------------------------------ elementwise warpgroups
    // warpgroup wg owns query columns [64 wg, 64 wg + 64) of each step, and feature columns
    // [d/2 wg, d/2 wg + d/2) of the dQ, dK and dV read-outs; its warp q owns tensor-memory lanes [32q, 32q + 32)
    const int wg = (warp >> 2) - 1;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row (tensor-memory lane) of P^T / dS^T; query row of dQ
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool key_ok = k0 + r < Nkv;
    const float sl2 = p.scale_log2;
    // dS^T row r, queries [QC wg, QC wg + QC): box (QC wg) / 64, 16-byte chunks from ((QC wg) % 64) / 8
    const uint32_t ds_row = smem_u32(sdS) + static_cast<uint32_t>(((wg * QC) / 64) * BOX + r * 128);
    const int ds_c0 = ((wg * QC) % 64) / 8;
    // dQ staging (d = 64): features [16 wg, 16 wg + 16) = box wg / 2, chunks from 4 (wg % 2)
    const uint32_t dq_row = smem_u32(sdQ) + static_cast<uint32_t>((NWG == 4 ? wg / 2 : wg) * (BT * 128) + r * 128);
    const int dq_c0 = NWG == 4 ? (wg % 2) * 4 : 0;
    const int sw = r & 7;
    // Row values of this warpgroup's queries ([slot][lse2 QC | D QC]): each lane fetches QC / 32 queries'
    // lse2 and D one step ahead, and every warp of the warpgroup stores the same values after its step's
    // hand-off, then reads them after a __syncwarp, so no barrier across the warpgroup is needed. A
    // warp rewrites a slot only after the products of the step before, which wait for every warp's
    // hand-off, and each warp reads the slot before its own hand-off.
    float* rows = sRow + wg * 4 * QC;
    struct RowVals {
      float l[QC / 32], d[QC / 32];
    };
    auto row_vals = [&](int it) -> RowVals {
      RowVals v;
#pragma unroll
      for (int k = 0; k < QC / 32; ++k) {
        const long long i = static_cast<long long>(it0 + it) * BT + wg * QC + k * 32 + lane;
        if (it >= nit || i >= p.Nq) {
          v.l[k] = -INFINITY;  // P = 0 for rows past the end
          v.d[k] = 0.0f;
        } else {
          const long long at = static_cast<long long>(bh) * p.Nq + i;
          v.l[k] = -(p.lse[at] * LOG2E);  // negated: the packed products below add them
          v.d[k] = -p.dvec[at];
        }
      }
      return v;
    };
    auto put_rows = [&](int slot, const RowVals& v) {
#pragma unroll
      for (int k = 0; k < QC / 32; ++k) {
        rows[slot * 2 * QC + k * 32 + lane] = v.l[k];
        rows[slot * 2 * QC + QC + k * 32 + lane] = v.d[k];
      }
      __syncwarp();
    };
    put_rows(0, row_vals(0));
    bool ok = true;
    // dQ of step it (after its products completed): scaled rows into the staging slot, then hand-off
    auto stage_dq = [&](int it) -> bool {
      const int slot = HD == 64 ? (it & 1) : 0;
      if constexpr (HD == 64) {
        bool w = true;
        if (it >= 2) w = wait_abort(&bar_dqfree[slot], static_cast<uint32_t>(((it - 2) >> 1) & 1), tmo, abort_flag,
                                    kBwdTimeoutSoftmax, 9);
        w = __all_sync(0xffffffffu, w);
        if (!w) return false;
      }
      // (d = 128: the staging area was released before this step's dS^T was written over it)
      if constexpr (NWG == 4) {
        uint32_t o[16];
        tmem_ld16(trow + C::COL_DQ + wg * 16, o);
        tmem_wait_ld();
        reg_fence16(o);
        const uint32_t dst = dq_row + static_cast<uint32_t>(slot * C::DQ_SLOT);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_shared_v4(dst + static_cast<uint32_t>(((dq_c0 + u) ^ sw) * 16),
                       __float_as_uint(__uint_as_float(o[4 * u]) * p.scale),
                       __float_as_uint(__uint_as_float(o[4 * u + 1]) * p.scale),
                       __float_as_uint(__uint_as_float(o[4 * u + 2]) * p.scale),
                       __float_as_uint(__uint_as_float(o[4 * u + 3]) * p.scale));
      } else {
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t o[32];
        tmem_ld32(trow + C::COL_DQ + wg * (HD / 2) + c * 32, o);
        tmem_wait_ld();
        reg_fence32(o);
        const uint32_t dst = HD == 64 ? dq_row + static_cast<uint32_t>(slot * C::DQ_SLOT)
                                      : smem_u32(sdQ) + static_cast<uint32_t>((2 * wg + c) * (BT * 128) + r * 128);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(dst + static_cast<uint32_t>((u ^ sw) * 16), __float_as_uint(__uint_as_float(o[4 * u]) * p.scale),
                       __float_as_uint(__uint_as_float(o[4 * u + 1]) * p.scale),
                       __float_as_uint(__uint_as_float(o[4 * u + 2]) * p.scale),
                       __float_as_uint(__uint_as_float(o[4 * u + 3]) * p.scale));
      }
      }
      fence_proxy_async_smem();
      if (HD == 128) tc_fence_before();  // dQ has left the dP^T columns the next S^T / dP^T products reuse
      mbar_arrive(&bar_staged[slot]);
      return true;
    };

    for (int it = 0; ok && it < nit; ++it) {
      const int slot = it & 1;
      const RowVals nrow = row_vals(it + 1);  // next step's row values, stored at the end of this one
      ok = wait_abort(bar_m1, static_cast<uint32_t>(it & 1), tmo, abort_flag, kBwdTimeoutMMA, 3);
      ok = __all_sync(0xffffffffu, ok);
      uint32_t pw[QC / 2], dw[QC / 2];
      if (ok) {
        tc_fence_after();
        // causal: key k0 + r hides from query i0 + q when r - q > dlt (absolute positions; |dlt| < 2^31
        // as N is an int); only tiles with dlt < 127 contain such pairs. The monolithic call has dlt = 0
        // on its diagonal tile and no other masked tile.
        int dlt = 0;
        bool diag;
        if constexpr (ACCUM) {
          dlt = static_cast<int>(p.q_off - p.kv_off) + (it0 + it) * BT - k0;
          diag = CAUSAL && dlt < BT - 1;
        } else {
          diag = CAUSAL && ((it0 + it) * BT == k0);
        }
        const float* lrow = rows + slot * 2 * QC;
        const float* drow = lrow + QC;
        // two 32-query chunks: S^T and dP^T columns in registers, then P and dS packed to 16-bit pairs;
        // S^T / dP^T are released to the next step's products once both chunks are read
#pragma unroll
        for (int c2 = 0; c2 < QC / CW; ++c2) {
          uint32_t s[CW], g[CW];
          if constexpr (CW == 16) {
            tmem_ld16(trow + C::COL_S + wg * QC + c2 * CW, s);
            tmem_ld16(trow + C::COL_DP + wg * QC + c2 * CW, g);
            tmem_wait_ld();
            reg_fence16(s);
            reg_fence16(g);
          } else {
            tmem_ld32(trow + C::COL_S + wg * QC + c2 * CW, s);
            tmem_ld32(trow + C::COL_DP + wg * QC + c2 * CW, g);
            tmem_wait_ld();
            reg_fence32(s);
            reg_fence32(g);
          }
          if (HD == 64 && c2 == QC / CW - 1) {
            tc_fence_before();
            mbar_arrive(bar_sfree);
          }
#pragma unroll
          for (int e = 0; e < CW / 2; ++e) {
            const int ql = c2 * CW + 2 * e;  // query within this warpgroup's QC
            const int q0 = wg * QC + ql;     // query within the tile
            const float2 nl = *reinterpret_cast<const float2*>(lrow + ql);  // -lse2 of the two queries
            const float2 nd = *reinterpret_cast<const float2*>(drow + ql);  // -D
            const float2 arg = __ffma2_rn(make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])),
                                          make_float2(sl2, sl2), nl);
            float p0 = ex2(arg.x);
            float p1 = ex2(arg.y);
            if (!key_ok) p0 = p1 = 0.0f;
            if (diag) {
              if constexpr (ACCUM) {
                if (r - q0 > dlt) p0 = 0.0f;
                if (r - q0 - 1 > dlt) p1 = 0.0f;
              } else {
                if (r > q0) p0 = 0.0f;
                if (r > q0 + 1) p1 = 0.0f;
              }
            }
            pw[c2 * (CW / 2) + e] = pack_pair(p0, p1, DT);
            const float2 gd =
                __fadd2_rn(make_float2(__uint_as_float(g[2 * e]), __uint_as_float(g[2 * e + 1])), nd);
            const float2 ds = __fmul2_rn(make_float2(p0, p1), gd);
            dw[c2 * (CW / 2) + e] = pack_pair(ds.x, ds.y, DT);
          }
        }
      }
      if constexpr (HD == 64) {
        // P^T and dS^T of the previous step are consumed once its products are done; its dQ is read out of
        // tensor memory while this step's P^T and dS^T go in, under one wait and one fence
        if (ok && it > 0) {
          ok = wait_abort(bar_m2, static_cast<uint32_t>((it - 1) & 1), tmo, abort_flag, kBwdTimeoutMMA, 4);
          const int qs = (it - 1) & 1;
          if (ok && it - 1 >= 2)
            ok = wait_abort(&bar_dqfree[qs], static_cast<uint32_t>(((it - 3) >> 1) & 1), tmo, abort_flag,
                            kBwdTimeoutSoftmax, 9);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after();
            uint32_t o[16];
            tmem_ld16(trow + C::COL_DQ + wg * 16, o);
            tmem_st16(trow + 448u + static_cast<uint32_t>(wg * (QC / 2)), &pw[0]);
#pragma unroll
            for (int u = 0; u < QC / 8; ++u)
              st_shared_v4(ds_row + static_cast<uint32_t>(((ds_c0 + u) ^ sw) * 16), dw[4 * u], dw[4 * u + 1],
                           dw[4 * u + 2], dw[4 * u + 3]);
            tmem_wait_ld();
            reg_fence16(o);
            const uint32_t dst = dq_row + static_cast<uint32_t>(qs * C::DQ_SLOT);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              st_shared_v4(dst + static_cast<uint32_t>(((dq_c0 + u) ^ sw) * 16),
                           __float_as_uint(__uint_as_float(o[4 * u]) * p.scale),
                           __float_as_uint(__uint_as_float(o[4 * u + 1]) * p.scale),
                           __float_as_uint(__uint_as_float(o[4 * u + 2]) * p.scale),
                           __float_as_uint(__uint_as_float(o[4 * u + 3]) * p.scale));
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar_staged[qs]);
            mbar_arrive(bar_ready);
            put_rows(slot ^ 1, nrow);
          }
          ok = __all_sync(0xffffffffu, ok);
          continue;  // this step's hand-offs are done
        }
      } else {
        // the previous step's dQ, staged over the dS^T tile, must have been read by its reduction
        if (ok && it > 0) {
          ok = wait_abort(&bar_dqfree[0], static_cast<uint32_t>((it - 1) & 1), tmo, abort_flag, kBwdTimeoutSoftmax, 9);
          ok = __all_sync(0xffffffffu, ok);
        }
      }
      if (ok) {
        // P^T (d = 128: over the first half of this warpgroup's own S^T columns, already read)
        {
          const uint32_t pt = NWG == 4 ? 448u + static_cast<uint32_t>(wg * (QC / 2)) : C::col_pt(wg * 4);
#pragma unroll
          for (int k = 0; k < QC / 32; ++k) tmem_st16(trow + pt + 16 * k, &pw[16 * k]);
        }
        // dS^T row r, this warpgroup's QC queries: QC / 8 16-byte chunks, 128-byte swizzle
#pragma unroll
        for (int u = 0; u < QC / 8; ++u)
          st_shared_v4(ds_row + static_cast<uint32_t>(((ds_c0 + u) ^ sw) * 16), dw[4 * u], dw[4 * u + 1],
                       dw[4 * u + 2], dw[4 * u + 3]);
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar_ready);
        put_rows(slot ^ 1, nrow);
      }
      if constexpr (HD == 128) {
        // this step's dQ, out of the dP^T columns before the next step's products may be issued
        if (ok) {
          ok = wait_abort(bar_m2, static_cast<uint32_t>(it & 1), tmo, abort_flag, kBwdTimeoutMMA, 4);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after();
            ok = stage_dq(it);
          }
        }
      }
      ok = __all_sync(0xffffffffu, ok);
    }
    if (HD == 64 && ok) {
      // last step: dQ, then dV_j and dK_j rows (key row = tensor-memory lane), written once
      ok = wait_abort(bar_m2, static_cast<uint32_t>((nit - 1) & 1), tmo, abort_flag, kBwdTimeoutMMA, 4);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        ok = stage_dq(nit - 1);
      }
    }
    if (NWG == 4 && ok) {
      // d = 64: features [16 wg, 16 wg + 16) of dV_j and dK_j
      const int fb = wg * 16;
      uint32_t a[16], g[16];
      tmem_ld16(trow + C::COL_DV + fb, a);
      tmem_ld16(trow + C::COL_DK + fb, g);
      tmem_wait_ld();
      reg_fence16(a);
      reg_fence16(g);
      const long long row = static_cast<long long>(bh) * Nkv + k0 + r;
      if (ACCUM && key_ok) {
        float4* dv = reinterpret_cast<float4*>(p.dv_acc + row * HD + fb);
        float4* dk = reinterpret_cast<float4*>(p.dk_acc + row * HD + fb);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          atomicAdd(dv + u, make_float4(__uint_as_float(a[4 * u]), __uint_as_float(a[4 * u + 1]),
                                        __uint_as_float(a[4 * u + 2]), __uint_as_float(a[4 * u + 3])));
          atomicAdd(dk + u, make_float4(__uint_as_float(g[4 * u]) * p.scale, __uint_as_float(g[4 * u + 1]) * p.scale,
                                        __uint_as_float(g[4 * u + 2]) * p.scale,
                                        __uint_as_float(g[4 * u + 3]) * p.scale));
        }
      } else if (!ACCUM && key_ok) {
        uint4* dv = reinterpret_cast<uint4*>(p.dv + row * HD + fb);
        uint4* dk = reinterpret_cast<uint4*>(p.dk + row * HD + fb);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
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
    for (int c = 0; NWG == 2 && c < HD / 64; ++c) {
      if (!ok) break;
      const int fb = wg * (HD / 2) + c * 32;  // first feature of this chunk
      uint32_t a[32], g[32];
      tmem_ld32(trow + C::COL_DV + fb, a);
      tmem_ld32(trow + C::COL_DK + fb, g);
      tmem_wait_ld();
      reg_fence32(a);
      reg_fence32(g);
      if (ACCUM && key_ok) {
        const long long row = static_cast<long long>(bh) * Nkv + k0 + r;
        float4* dv = reinterpret_cast<float4*>(p.dv_acc + row * HD + fb);
        float4* dk = reinterpret_cast<float4*>(p.dk_acc + row * HD + fb);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          atomicAdd(dv + u, make_float4(__uint_as_float(a[4 * u]), __uint_as_float(a[4 * u + 1]),
                                        __uint_as_float(a[4 * u + 2]), __uint_as_float(a[4 * u + 3])));
          atomicAdd(dk + u, make_float4(__uint_as_float(g[4 * u]) * p.scale, __uint_as_float(g[4 * u + 1]) * p.scale,
                                        __uint_as_float(g[4 * u + 2]) * p.scale,
                                        __uint_as_float(g[4 * u + 3]) * p.scale));
        }
      } else if (!ACCUM && key_ok) {
        const long long row = static_cast<long long>(bh) * Nkv + k0 + r;
        uint4* dv = reinterpret_cast<uint4*>(p.dv + row * HD + fb);
        uint4* dk = reinterpret_cast<uint4*>(p.dk + row * HD + fb);
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
  }
  // teardown: every role has drained its own asynchronous work (bounded waits) before this barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// D_i = dO_i . O_i in fp32: d/8 threads per row (8 for d = 64, 16 for d = 128), one 16-byte load of
// each per thread, summed across the row's threads by shuffles. Row r of the `rows` = BH * n rows is
// token t0 + r % n of head r / n of [BH, N, d] tensors (n = N, t0 = 0 for packed rows).
template <int DT, int HD>
__global__ void __launch_bounds__(256) bwd_dot_kernel(const uint4* o, const uint4* g, float* dvec, long long rows,
                                                      long long n, long long N, long long t0) {
  constexpr int TPR = HD / 8;
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = t / TPR;
  const long long frow = (row / n) * N + t0 + row % n;  // the row's index in the [BH, N] tensors
  const long long e = frow * TPR + t % TPR;            // this thread's 16-byte word
  float acc = 0.0f;
  if (row < rows) {
    const uint4 a = __ldg(o + e), c = __ldg(g + e);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 x = unpack_pair(aw[u], DT), y = unpack_pair(cw[u], DT);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int m = TPR / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (row < rows && (t % TPR) == 0) dvec[frow] = acc;
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

// [B,H,N,d] 16-bit tensor: dims (d, N, H, B), box (64, 128, 1, 1), 128-byte swizzle, zero fill.
int make_bhnd_map(CUtensorMap* m, const void* base, int dtype, int B, int H, int N, int d) {
  const cuuint64_t es = 2;
  const cuuint64_t HDd = static_cast<cuuint64_t>(d);
  const cuuint64_t dims[4] = {HDd, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {HDd * es, static_cast<cuuint64_t>(N) * HDd * es,
                                 static_cast<cuuint64_t>(H) * N * HDd * es};
  const cuuint32_t box[4] = {64, BT, 1, 1};
  return encode_map(m, dtype == CQSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    base, dims, strides, box);
}

// fp32 dQ accumulator [BH, N, d]: dims (d, N, BH), box (32, 128, 1) (128-byte rows), 128-byte swizzle.
int make_dq_map(CUtensorMap* m, float* base, int BH, int N, int d) {
  const cuuint64_t HDd = static_cast<cuuint64_t>(d);
  const cuuint64_t dims[3] = {HDd, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {HDd * 4, static_cast<cuuint64_t>(N) * HDd * 4};
  const cuuint32_t box[3] = {32, BT, 1};
  return encode_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box);
}

template <int DT, bool CAUSAL, int ACCUM, int HD>
int launch_main(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mg,
                const CUtensorMap& mdq, const BwdParams& p, int n_kv_tiles, cudaStream_t s) {
  auto kern = attn_bwd_kernel<DT, CAUSAL, ACCUM, HD>;
  constexpr uint32_t SMEM_BYTES = BwdCfg<HD>::SMEM_BYTES;
  using TH = BwdThreads<HD>;
  constexpr int NTHR = TH::NTHR;
  constexpr int BWD_REGS_LOW = TH::LOW, BWD_REGS_HIGH = TH::HIGH;
  static PerDeviceOnce attr;  // the attributes belong to each device's context
  int dev = 0;
  if (!attr.done(&dev)) {
    // setmaxnreg.inc waits until its registers are free: refuse to launch unless the launch holds the split
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncGetAttributes(attention backward)");
    if (fa.numRegs * NTHR < 128 * BWD_REGS_LOW + 128 * TH::NWG * BWD_REGS_HIGH) {
      set_error("attention backward kernel built with %d registers/thread; the register split needs %d", fa.numRegs,
                (128 * BWD_REGS_LOW + 128 * TH::NWG * BWD_REGS_HIGH + NTHR - 1) / NTHR);
      return CQSA_ERR_UNSUPPORTED;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(attention backward smem)");
    attr.mark(dev);
  }
  const long long grid = static_cast<long long>(n_kv_tiles) * p.BH;
  kern<<<static_cast<unsigned>(grid), NTHR, SMEM_BYTES, s>>>(mq, mk, mv, mg, mdq, p);
  return cuda_status(cudaGetLastError(), "attention backward kernel launch");
}

template <int ACCUM, int HD>
int dispatch_main(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mg,
                  const CUtensorMap& mdq, const BwdParams& p, int n_kv_tiles, int dtype, int causal, cudaStream_t s) {
  if (dtype == CQSA_BF16)
    return causal ? launch_main<1, true, ACCUM, HD>(mq, mk, mv, mg, mdq, p, n_kv_tiles, s)
                  : launch_main<1, false, ACCUM, HD>(mq, mk, mv, mg, mdq, p, n_kv_tiles, s);
  return causal ? launch_main<0, true, ACCUM, HD>(mq, mk, mv, mg, mdq, p, n_kv_tiles, s)
                : launch_main<0, false, ACCUM, HD>(mq, mk, mv, mg, mdq, p, n_kv_tiles, s);
}

// Maps and parameters of one launch of the main kernel (the monolithic call or one chunk pair).
int run_main(const BwdArgs& a, float* dq_acc, const float* dvec, int accum, cudaStream_t stream) {
  const long long n_q_tiles = (a.Nq + BT - 1) / BT, n_kv_tiles = (a.Nkv + BT - 1) / BT;
  if (n_kv_tiles * a.B * a.H > 0x7fffffffLL) {
    set_error("problem too large for one launch");
    return CQSA_ERR_UNSUPPORTED;
  }
  if (a.d != 64 && a.d != 128) {
    set_error("the backward supports head dim 64 or 128 (got %d)", a.d);
    return CQSA_ERR_UNSUPPORTED;
  }
  CUtensorMap mq, mk, mv, mg, mdq;
  int rc = make_bhnd_map(&mq, a.q, a.dtype, a.B, a.H, a.Nq, a.d);
  if (rc == CQSA_OK) rc = make_bhnd_map(&mk, a.k, a.dtype, a.B, a.H, a.Nkv, a.d);
  if (rc == CQSA_OK) rc = make_bhnd_map(&mv, a.v, a.dtype, a.B, a.H, a.Nkv, a.d);
  if (rc == CQSA_OK) rc = make_bhnd_map(&mg, a.dout, a.dtype, a.B, a.H, a.Nq, a.d);
  if (rc == CQSA_OK) rc = make_dq_map(&mdq, dq_acc, a.B * a.H, a.Nq, a.d);
  if (rc != CQSA_OK) return rc;
  BwdParams p;
  p.lse = a.lse;
  p.dvec = dvec;
  p.dq_acc = dq_acc;
  p.dk = static_cast<uint16_t*>(a.dk);
  p.dv = static_cast<uint16_t*>(a.dv);
  p.dk_acc = a.dk_acc;
  p.dv_acc = a.dv_acc;
  p.H = a.H;
  p.BH = a.B * a.H;
  p.Nq = a.Nq;
  p.Nkv = a.Nkv;
  p.n_q_tiles = static_cast<int>(n_q_tiles);
  p.n_kv_tiles = static_cast<int>(n_kv_tiles);
  {
    // per head: the fp32 dQ accumulator and the Q and dO rows streamed past every key tile
    const long long per_head = static_cast<long long>(a.Nq) * a.d * (4 + 2 + 2);
    const long long budget = static_cast<long long>(CQSA_BWD_GROUP_MB) << 20;
    const int BH = a.B * a.H;
    long long g = (budget <= 0 || per_head * BH <= budget) ? BH : budget / per_head;
    p.head_group = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  }
  p.q_off = a.q_off;
  p.kv_off = a.kv_off;
  p.scale = a.scale;
  p.scale_log2 = a.scale * LOG2E;
  p.timeout_ns = timeout_ns();
  p.fault = debug_fault();
  const int nkt = static_cast<int>(n_kv_tiles);
  if (a.d == 128)
    return accum ? dispatch_main<1, 128>(mq, mk, mv, mg, mdq, p, nkt, a.dtype, a.causal, stream)
                 : dispatch_main<0, 128>(mq, mk, mv, mg, mdq, p, nkt, a.dtype, a.causal, stream);
  return accum ? dispatch_main<1, 64>(mq, mk, mv, mg, mdq, p, nkt, a.dtype, a.causal, stream)
               : dispatch_main<0, 64>(mq, mk, mv, mg, mdq, p, nkt, a.dtype, a.causal, stream);
}

}  // namespace

size_t attention_bwd_workspace(int B, int H, int N, int d) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t dq = (rows * d * sizeof(float) + 255) & ~size_t(255);
  return dq + rows * sizeof(float);
}

int launch_bwd_dvec_range(const void* out, const void* dout, float* dvec, long long BH, long long n, long long N,
                          long long t0, int d, int dtype, cudaStream_t stream) {
  const long long rows = BH * n;
  if (rows <= 0) return CQSA_OK;
  const long long dot_threads = rows * (d / 8);
  const unsigned dot_blocks = static_cast<unsigned>((dot_threads + 255) / 256);
  const uint4* o = static_cast<const uint4*>(out);
  const uint4* g = static_cast<const uint4*>(dout);
  if (d == 128) {
    if (dtype == CQSA_BF16) bwd_dot_kernel<1, 128><<<dot_blocks, 256, 0, stream>>>(o, g, dvec, rows, n, N, t0);
    else bwd_dot_kernel<0, 128><<<dot_blocks, 256, 0, stream>>>(o, g, dvec, rows, n, N, t0);
  } else {
    if (dtype == CQSA_BF16) bwd_dot_kernel<1, 64><<<dot_blocks, 256, 0, stream>>>(o, g, dvec, rows, n, N, t0);
    else bwd_dot_kernel<0, 64><<<dot_blocks, 256, 0, stream>>>(o, g, dvec, rows, n, N, t0);
  }
  return cuda_status(cudaGetLastError(), "attention backward dot kernel launch");
}

int launch_bwd_dvec(const void* out, const void* dout, float* dvec, long long rows, int d, int dtype,
                    cudaStream_t stream) {
  return launch_bwd_dvec_range(out, dout, dvec, 1, rows, rows, 0, d, dtype, stream);
}

int launch_bwd_cast(const float* acc, void* out, long long n, int dtype, cudaStream_t stream) {
  const long long n4 = n / 4;
  if (n4 <= 0) return CQSA_OK;
  const unsigned cblocks = static_cast<unsigned>(std::min<long long>((n4 + 255) / 256, 152LL * 16));
  if (dtype == CQSA_BF16)
    bwd_dq_kernel<1><<<cblocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(acc), static_cast<uint2*>(out), n4);
  else
    bwd_dq_kernel<0><<<cblocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(acc), static_cast<uint2*>(out), n4);
  return cuda_status(cudaGetLastError(), "attention backward cast kernel launch");
}

int launch_attention_bwd(const BwdArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.Nq;
  float* dq_acc = static_cast<float*>(a.workspace);
  float* dvec = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) +
                                         ((static_cast<size_t>(rows) * a.d * sizeof(float) + 255) & ~size_t(255)));
  // D_i, then the zeroed dQ accumulator, the main kernel and the dQ conversion
  int rc = launch_bwd_dvec(a.out, a.dout, dvec, rows, a.d, a.dtype, stream);
  if (rc != CQSA_OK) return rc;
  rc = cuda_status(cudaMemsetAsync(dq_acc, 0, static_cast<size_t>(rows) * a.d * sizeof(float), stream),
                   "zero dQ accumulator");
  if (rc != CQSA_OK) return rc;
  rc = run_main(a, dq_acc, dvec, 0, stream);
  if (rc != CQSA_OK) return rc;
  return launch_bwd_cast(dq_acc, a.dq, rows * a.d, a.dtype, stream);
}

int launch_attention_bwd_chunk(const BwdArgs& a, cudaStream_t stream) {
  return run_main(a, a.dq_acc, a.dvec, 1, stream);
}

int bwd_error_word(DevErr* out, int clear) {
  int rc = cuda_status(cudaMemcpyFromSymbol(out, g_bwd_err, sizeof(DevErr)), "read backward error word");
  if (rc != CQSA_OK || !clear || out->code == 0) return rc;
  DevErr z = {0, 0, 0, 0};
  return cuda_status(cudaMemcpyToSymbol(g_bwd_err, &z, sizeof(z)), "clear backward error word");
}

int bwd_error_word_on(DevErr* out, cudaStream_t s) {
  int rc = cuda_status(cudaMemcpyFromSymbolAsync(out, g_bwd_err, sizeof(DevErr), 0, cudaMemcpyDeviceToHost, s),
                       "read backward error word");
  if (rc == CQSA_OK) rc = cuda_status(cudaStreamSynchronize(s), "read backward error word");
  if (rc != CQSA_OK || out->code == 0) return rc;
  static const DevErr z = {0, 0, 0, 0};
  rc = cuda_status(cudaMemcpyToSymbolAsync(g_bwd_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s),
                   "clear backward error word");
  if (rc == CQSA_OK) rc = cuda_status(cudaStreamSynchronize(s), "clear backward error word");
  return rc;
}

}  // namespace cqsa
