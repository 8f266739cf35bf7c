// Exact attention forward for sm_103a: TMA-fed, tcgen05 MMAs accumulating in tensor memory, and a
// warp-specialised online softmax between the two contractions.
//
// attn_fwd2_kernel (the one every entry point launches): one CTA computes two 128-row query tiles of
// one (batch, head) against every key tile either may see, loading each K/V tile once for both.
//   warp 0        TMA producer (one lane): both Q tiles once, then K and V tiles through a ring of
//                 STAGES shared-memory stages (mbarrier full/empty pairs, byte-counted completion).
//   warps 1, 2    MMA issuers for query tiles 0 and 1 (warp 1 also owns the tensor memory): one
//                 elected lane issues S = Q K^T (A and B from shared memory) and O += P V (P from
//                 tensor memory, V from shared memory) and commits each group to mbarriers.
//   warps 4..7,   softmax warpgroups of tiles 0 and 1, one thread per query row: tcgen05.ld of the
//   8..11         row of S, masking, row max, p = exp2(s * scale * log2 e - m_ref), row sum, P packed
//                 to 16 bits and stored with tcgen05.st; rare exact rescales of O; the fold of O into
//                 an fp32 running sum between 128-key-tile segments (d = 64); the epilogue.
//   setmaxnreg moves registers from warpgroup 0 (72 per thread) to the softmax warpgroups (216).
// Tensor memory (512 columns), fp16 d = 64: S0 | S1 | P0 | P1 | O0 | O1 at 0, 128, 256, 320, 384, 448,
// so S_t(j+1) is computed while the softmax still stores P_t(j); d = 128 and bf16 write P over S.
//
// bf16: P rounded to bf16 alone (8-bit significand) costs ~2^-9 relative per weight; P is split into
// P_hi = bf16(p) and P_lo = bf16(p - P_hi) and both are multiplied into O (as the hi/lo operand split
// of the prompt-attention kernel in the "Strata" pull request #800 does for fp16), ~2^-17 overall.
//
// Reference max: m_ref is kept as an integer in the base-2 domain and raised only when a tile's row
// max exceeds it by more than TAU, to ceil(row max). Rescales of O are then exact powers of two,
// rare, and partial results of different key splits differ only by powers of two before rounding,
// so chunked and monolithic results agree to fp32 summation-order level.
//
// The pages describe the kernels they ship as "FlashAttention-2-derived CQS forward" built for
// sm80/sm90 ("stream-cqsa 2.2.0 -> 2.2.2" diff, README); this kernel keeps the blockwise online
// softmax that defines that family and is otherwise designed for tcgen05 / TMEM / TMA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "cqsa_internal.h"
#include "sm103_ptx.cuh"

#ifndef CQSA_D128_FLUSH
#define CQSA_D128_FLUSH 32
#endif
#ifndef CQSA_KV_GROUP_MB
#define CQSA_KV_GROUP_MB 64
#endif

namespace cqsa {

__device__ DevErr g_dev_err;

// Running sums of the d = 128 attention kernel: one slot of two tiles x 128 features x 128 rows (fp32)
// per SM id. Contents need no clearing: a CTA writes its slot before it reads it.
constexpr int kOsumSlots = 256;
constexpr int kOsumSlotFloats = 2 * 128 * 128;
__device__ __align__(256) float g_osum[kOsumSlots * kOsumSlotFloats];

namespace {

constexpr int BM = 128;        // query rows per tile
constexpr int BN = 128;        // keys per tile
// m_ref is raised (to ceil of the tile's row max) whenever a tile's row max exceeds it, so every
// exponent argument is <= 0: ex2.approx is exactly covariant under integer shifts of its argument
// only while the argument keeps its sign, and the chunked and monolithic paths (whose m_ref differ
// by integers) must produce P values that differ by exact powers of two. Rescales stay rare: the
// integer m_ref moves only when the running max crosses an integer.
constexpr float TAU = 0.0f;
constexpr uint32_t TILE_BYTES = 128 * 64 * 2;  // one 128 x 64 box of 16-bit elements
constexpr uint32_t TMEM_COLS = 512;

struct KParams {
  int H, BH;
  int Nq, Nkv;
  long long q_off, kv_off;
  float scale_log2;
  int n_q_tiles;
  void* out;
  float* lse;
  float* o_part;
  float* lse_part;
  int out_layout;
  unsigned long long timeout_ns;
  unsigned timeout_us;  // the same limit in microseconds (32-bit, for the two-tile kernel's loops)
  int fault;  // test hook: 1 = block 0 never loads key tile 1 (its waits must time out cleanly)
  int mode;   // output mode of a pair in a multi-pair launch (AttnMode)
  int head_group;  // heads whose units are interleaved (the rest follow group by group); >= 1
};

// A launch over several chunk pairs at once (the wave engine): one entry per pair, with its own
// tensor maps, offsets, sizes, output mode and accumulator, and the first unit (CTA) of the pair.
constexpr int kModeMulti = 3;  // template MODE of the multi-pair kernel: each pair's mode is in its entry
constexpr int kMaxWavePairs = 32;
struct PairDesc {
  CUtensorMap q, k, v;
  long long q_off, kv_off;
  float* o_part;
  float* lse_part;
  int Nq, Nkv, n_q_tiles, mode, unit_begin;
};
struct MultiParams {
  KParams common;
  int n_pairs;
  PairDesc pair[kMaxWavePairs];
};


__device__ __forceinline__ void record_error(int code, int where) {
  if (atomicCAS(&g_dev_err.code, 0, code) == 0) {
    g_dev_err.block = blockIdx.x;
    g_dev_err.where = where;
  }
}

// Bounded wait on a 32-bit shared address with a microsecond limit that also gives up as soon as another
// role of this CTA has aborted; the waiting thread sleeps in try_wait (woken when the phase completes)
// between checks of the abort flag and the clock.
__device__ __forceinline__ bool wait_or_abort_a(uint32_t bar, uint32_t parity, uint32_t tmo_us, uint32_t abort_addr,
                                                int code, int where) {
  if (mbar_try_wait_a(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep_a(bar, parity, 1000000u)) return true;
    if (ld_shared_volatile_u32(abort_addr)) return false;
    if (globaltimer_ns() - t0 > static_cast<uint64_t>(tmo_us) * 1000ull) {
      record_error(code, where);
      st_shared_volatile_u32(abort_addr, 1u);
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^k for integer-valued k <= 0 (exact; 0 below the normal range).
__device__ __forceinline__ float exp2_int(float k) {
  int e = static_cast<int>(k);
  if (e < -126) return 0.0f;
  return __int_as_float((e + 127) << 23);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Row maximum of 128 scores: three-input max, four independent chains.
__device__ __forceinline__ float row_max128(const float (&x)[128]) {
  float m0 = x[0], m1 = x[1], m2 = x[2], m3 = x[3];
#pragma unroll
  for (int c = 4; c < 128; c += 8) {
    m0 = max3(m0, x[c], x[c + 1]);
    m1 = max3(m1, x[c + 2], x[c + 3]);
    m2 = max3(m2, x[c + 4], x[c + 5]);
    m3 = max3(m3, x[c + 6], x[c + 7]);
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// p = exp2(fl(x * scale*log2e + 192) - (192 + m_ref)) for the pair (x0, x1), with packed fp32x2
// arithmetic. The first rounding puts the argument on a grid fixed by x alone (2^-16 while the
// sum stays in [128, 256)), so the subtraction of the integer-valued 192 + m_ref is exact.
__device__ __forceinline__ float2 exp_pair(float x0, float x1, float2 sl2v, float2 ncm) {
  const float2 t = __ffma2_rn(make_float2(x0, x1), sl2v, make_float2(192.0f, 192.0f));
  const float2 r = __fadd2_rn(t, ncm);
  return make_float2(fast_exp2(r.x), fast_exp2(r.y));
}

__device__ __forceinline__ long long out_row_index(int layout, int b, int h, int H, int N, int i) {
  return layout == CQSA_LAYOUT_BHND ? (static_cast<long long>(b) * H + h) * N + i
                                    : (static_cast<long long>(b) * N + i) * H + h;
}

// MMA issue from one elected lane of a converged warp, with descriptors prepared by the whole warp
// and the accumulate flag as an immediate: measured on GB300 to issue at the tensor pipe's own rate
// (a 128x64x16 MMA every 32 cycles), while issuing from a lone thread with register-held flags costs
// ~150 cycles per MMA whatever its size.
template <int ACC>
__device__ __forceinline__ void mma_ss_i(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 1;" ::"r"(d), "l"(a), "l"(b), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 0;" ::"r"(d), "l"(a), "l"(b), "r"(idesc)
                 : "memory");
}
template <int ACC>
__device__ __forceinline__ void mma_ts_i(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d), "r"(a), "l"(b), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 0;" ::"r"(d), "r"(a), "l"(b), "r"(idesc)
                 : "memory");
}
__device__ __forceinline__ bool elect_one() {
  uint32_t p;
  asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}" : "=r"(p));
  return p != 0;
}

// S = Q K^T for one query tile: D/16 MMAs of 128x128x16 (K-major Q and K, 128-byte swizzle).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t dcol, uint64_t a0, uint64_t b0, uint32_t idesc) {
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = static_cast<uint32_t>((ks >> 2) * (TILE_BYTES >> 4) + (ks & 3) * 2);
    if (ks == 0) mma_ss_i<0>(dcol, a0 + off, b0 + off, idesc);
    else mma_ss_i<1>(dcol, a0 + off, b0 + off, idesc);
  }
}

// O += P V for one query tile: 8 MMAs of 128 x D x 16 (P from tensor memory, V MN-major); bf16 adds
// the P_lo half. FIRST: the first MMA overwrites O.
template <int D, int DT, bool FIRST>
__device__ __forceinline__ void issue_pv(uint32_t ocol, uint32_t pcol, uint64_t v0, uint32_t idesc) {
#pragma unroll
  for (int ks = 0; ks < BN / 16; ++ks) {
    const uint64_t bd = v0 + static_cast<uint32_t>(ks * (2048 >> 4));
    if (FIRST && ks == 0) mma_ts_i<0>(ocol, pcol + ks * 8, bd, idesc);
    else mma_ts_i<1>(ocol, pcol + ks * 8, bd, idesc);
    if (DT) mma_ts_i<1>(ocol, pcol + 64 + ks * 8, bd, idesc);
  }
}

// ---------------------------------------------------------------------------------------------
// Two query tiles per CTA (256 rows of one (batch, head)), two softmax warpgroups. While one
// warpgroup computes its softmax, the tensor pipe runs the other tile's MMAs, and each SM sub-
// partition has two softmax warps to interleave. K/V tiles are loaded once for both query tiles.
//   warp 0      TMA producer          warp 1      TMEM allocation + MMA issue for query tile 0
//   warp 2      MMA issue for tile 1  warp 3      idle (warpgroup 0 gives registers to the softmax)
//   warps 4..7  softmax of tile 0     warps 8..11 softmax of tile 1
// Tensor memory: S0, S1 at 0 / 128. fp16 with d = 64 keeps P apart (P0, P1 at 256 / 320, O0, O1 at
// 384 / 448), so S_t(j+1) is computed as soon as S_t(j) has been read. Otherwise (d = 128, or bf16
// whose P_hi|P_lo fills 128 columns) P_t is written over S_t and the MMA issuer waits for PV_t(j)
// to finish reading it before S_t(j+1) overwrites the columns; O0, O1 then sit at 256 / 256 + d.
// ---------------------------------------------------------------------------------------------
constexpr int NTHREADS2 = 384;
// Register split (setmaxnreg): the launch gives 384 x 168 registers; warpgroup 0 (producer, MMA issuer,
// two idle warps) drops to 72 and the two softmax warpgroups rise to 216: 128*72 + 256*216 = 384*168.
constexpr int REGS_LOW = 72, REGS_HIGH = 216;
static_assert(128 * REGS_LOW + 256 * REGS_HIGH <= NTHREADS2 * 168, "register split exceeds the launch allocation");

template <int D, int DT>
struct Cfg2 {
  static constexpr bool ALIAS = (D == 128) || (DT == 1);
  static constexpr int KSUB = D / 64;
  static constexpr int STAGES = (D == 64) ? 4 : 2;
  static constexpr uint32_t QT_BYTES = KSUB * TILE_BYTES;
  static constexpr uint32_t KV_BYTES = KSUB * TILE_BYTES;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128;
  static constexpr uint32_t COL_P0 = ALIAS ? 0u : 256u, COL_P1 = ALIAS ? 128u : 320u;
  static constexpr uint32_t COL_O0 = ALIAS ? 256u : 384u, COL_O1 = COL_O0 + D;
  static constexpr int NBARS = 1 + 3 * STAGES + 2 * 5 + 2;
  // Every FLUSH key tiles the softmax folds the tensor-memory accumulator into an fp32 running sum, so no
  // tensor-core accumulation chain exceeds FLUSH * 8 (d = 64) or FLUSH * 8 * 2 (bf16 hi/lo) MMAs. (The
  // MMA's fp32 accumulation is biased toward zero: measured relative drift -1.6e-5 after 16K keys, -6.9e-5
  // after 65K; the running sum uses RNE adds.) Chunk partials whose key ranges start at multiples of
  // FLUSH * 128 tokens then accumulate exactly the segments of the monolithic call. d = 64 keeps the
  // running sum in shared memory ([tile][feature][row], conflict-free per row); d = 128 has no shared or
  // tensor memory left for it and keeps it in global memory, one 128 KiB slot per SM (g_osum below): two
  // CTAs of this kernel never share an SM (each needs more than half of its shared and all its tensor
  // memory), so the slot of the SM a CTA runs on is its own for the CTA's lifetime.
  static constexpr int FLUSH = (D == 64) ? 128 : CQSA_D128_FLUSH;
  static constexpr bool OSUM_SMEM = (D == 64);
  static constexpr uint32_t OSUM_BYTES = OSUM_SMEM ? 2u * D * 128u * 4u : 0u;
  static constexpr uint32_t SMEM_BYTES =
      1024 + 2 * QT_BYTES + 2 * STAGES * KV_BYTES + OSUM_BYTES + NBARS * 8 + 16;
  static_assert(COL_O1 + D <= TMEM_COLS, "tensor memory layout exceeds 512 columns");
};

// The kernel body, for one work unit (a pair of query tiles of one (batch, head)); the tensor maps are
// kernel parameters (__grid_constant__), passed by reference so that TMA sees their parameter-space
// addresses.
template <int D, int DT, bool CAUSAL, int MODE>
__device__ __forceinline__ void attn_fwd2_body(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                               const KParams& p, const int unit) {
  using C = Cfg2<D, DT>;
  const int mode = (MODE == kModeMulti) ? p.mode : MODE;
  constexpr int STAGES = C::STAGES;
  constexpr int KSUB = C::KSUB;
  constexpr bool ALIAS = C::ALIAS;
  constexpr bool WARP_ARRIVE = !ALIAS && MODE != kModeMulti;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;  // tile t at sQ + t * QT_BYTES
  uint8_t* sK = sQ + 2 * C::QT_BYTES;
  uint8_t* sV = sK + STAGES * C::KV_BYTES;
  // running sum of O: shared memory (d = 64) or this SM's global slot (d = 128), [tile][feature][row]
  float* sOsum = reinterpret_cast<float*>(sV + STAGES * C::KV_BYTES);
  bool osum_ok = true;
  if (!C::OSUM_SMEM) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    osum_ok = smid < static_cast<uint32_t>(kOsumSlots);
    sOsum = g_osum + static_cast<size_t>(osum_ok ? smid : 0u) * kOsumSlotFloats;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + STAGES * C::KV_BYTES + C::OSUM_BYTES);
  uint64_t* bar_q = bars;
  uint64_t* bar_k_full = bar_q + 1;
  uint64_t* bar_v_full = bar_k_full + STAGES;
  uint64_t* bar_kv_empty = bar_v_full + STAGES;
  uint64_t* bar_s_full = bar_kv_empty + STAGES;  // [2]
  uint64_t* bar_s_free = bar_s_full + 2;         // [2] (P kept apart only)
  uint64_t* bar_p_full = bar_s_free + 2;         // [2]
  uint64_t* bar_pv_done = bar_p_full + 2;        // [2]
  uint64_t* bar_o_final = bar_pv_done + 2;       // [2] single phase each
  uint64_t* bar_mma_idle = bar_o_final + 2;     // [2] one per MMA warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma_idle + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work unit: a pair of query tiles, heaviest (latest) first.
  // Units of head_group heads at a time (heads interleaved, query-tile pairs heaviest first), so that the
  // K/V of the heads in flight stay in L2; one group of all heads when they fit.
  const int gsz = p.head_group;
  const int per_group = gsz * p.n_q_tiles;
  const int g0 = (unit / per_group) * gsz;
  const int gn = min(gsz, p.BH - g0);
  const int ur = unit - (unit / per_group) * per_group;
  const int qp = p.n_q_tiles - 1 - ur / gn;
  const int bh = g0 + ur % gn;
  const int b = bh / p.H;
  const int h = bh % p.H;
  // Per query tile: first row and number of key tiles (scalars: no runtime-indexed local arrays).
  auto tile_kv = [&](int qt0) -> int {
    const int rows = min(BM, p.Nq - qt0);
    int n = (p.Nkv + BN - 1) / BN;
    if (rows <= 0) {
      n = 0;
    } else if (CAUSAL) {
      const long long last_key = p.q_off + qt0 + rows - 1 - p.kv_off;
      n = last_key < 0 ? 0 : (last_key / BN + 1 < n ? static_cast<int>(last_key / BN + 1) : n);
    }
    return n;
  };
  const int q00 = qp * 2 * BM, q01 = q00 + BM;
  const int nkv0 = tile_kv(q00), nkv1 = tile_kv(q01);
  const int n_max = max(nkv0, nkv1);

  if (threadIdx.x == 0) {
    if (!osum_ok) record_error(kDevSmSlot, 30);  // results stay exact; only the fold is skipped
    mbar_init(bar_q, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_kv_empty[s], 2);  // one arrival per MMA warp
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_s_full[t], 1);
      // One arrival per softmax warp where P is kept apart (fp16, d = 64) in the single-pair kernel, one
      // per thread otherwise (measured: per-warp arrivals gain 1% on the 32K bench shape and 4.5% at
      // 262K tokens, and lose 4% at bf16 d = 128 and 13% in the multi-pair launch of the wave engine)
      mbar_init(&bar_s_free[t], WARP_ARRIVE ? 4 : 128);
      mbar_init(&bar_p_full[t], WARP_ARRIVE ? 4 : 128);
      mbar_init(&bar_pv_done[t], 1);
      mbar_init(&bar_o_final[t], 1);
      mbar_init(&bar_mma_idle[t], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long tmo = p.timeout_ns;
  const uint32_t tmo_us = p.timeout_us;
  const uint32_t a_abort = smem_u32(const_cast<int*>(abort_flag));
  // Each warpgroup changes its register budget at the top of its own branch and leaves through its
  // own copy of the teardown barrier, so no code runs under two different budgets.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_LOW));
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && n_max > 0) {
      mbar_arrive_expect_tx(bar_q, 2 * C::QT_BYTES);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int s = 0; s < KSUB; ++s)
          tma_load_4d(sQ + t * C::QT_BYTES + s * TILE_BYTES, &tmQ, bar_q, s * 64, t ? q01 : q00, h, b);
      int issued = 0;
      int skipped = -1;  // fault injection: the key/value tile never loaded
      for (int j = 0; j < n_max; ++j) {
        const int stage = j % STAGES;
        const uint32_t round = j / STAGES;
        if (!wait_or_abort_a(smem_u32(&bar_kv_empty[stage]), (round & 1u) ^ 1u, tmo_us, a_abort, kDevTimeoutKV, 10)) break;
        if (p.fault == 1 && blockIdx.x == 0 && j == 1) {
          skipped = j;
          issued = j + 1;
          continue;
        }
        mbar_arrive_expect_tx(&bar_k_full[stage], C::KV_BYTES);
#pragma unroll
        for (int s = 0; s < KSUB; ++s)
          tma_load_4d(sK + stage * C::KV_BYTES + s * TILE_BYTES, &tmK, &bar_k_full[stage], s * 64, j * BN, h, b);
        mbar_arrive_expect_tx(&bar_v_full[stage], C::KV_BYTES);
#pragma unroll
        for (int s = 0; s < KSUB; ++s)
          tma_load_4d(sV + stage * C::KV_BYTES + s * TILE_BYTES, &tmV, &bar_v_full[stage], s * 64, j * BN, h, b);
        issued = j + 1;
      }
      {
        // Every load issued must land before the CTA exits (bounded waits, no abort check); on the
        // normal path these phases are already complete.
        for (int j = max(0, issued - STAGES); j < issued; ++j) {
          if (j == skipped) continue;
          const int stage = j % STAGES;
          const uint32_t par = (j / STAGES) & 1u;
          mbar_wait_bounded(&bar_k_full[stage], par, tmo);
          mbar_wait_bounded(&bar_v_full[stage], par, tmo);
        }
        mbar_wait_bounded(bar_q, 0, tmo);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------------ MMA issuers
    // Warp 1 issues every MMA of query tile 0 and warp 2 every MMA of tile 1, on different SM
    // sub-partitions, each on its own schedule. Each warp runs its schedule and barrier waits
    // converged (warp-uniform values); one elected lane issues each MMA group and commit.
    const int t = warp - 1;
    const bool leader = elect_one();
    const int nkv = t ? nkv1 : nkv0;
    if (n_max > 0) {
      constexpr uint32_t IDESC_S = idesc_f16(DT, 0, 128, 128);
      constexpr uint32_t IDESC_O = idesc_f16(DT, 1, 128, D);  // N = d: one MMA covers every feature
      // Shared-memory descriptors are built once; each MMA adds a compile-time offset (16-byte units)
      // to the start-address field, which cannot carry out of its 14 bits below 256 KiB. V is MN-major:
      // 8 keys x 64 features per 1024-byte atom (SBO = 1024 along keys); the second 64-feature box of
      // d = 128 starts TILE_BYTES further (LBO).
      const uint64_t dQ = smem_desc_sw128(smem_u32(sQ + t * C::QT_BYTES), 16, 1024);
      const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = smem_desc_sw128(smem_u32(sV), D == 128 ? TILE_BYTES : 1024, 1024);
      const uint32_t col_s = tmem + (t ? C::COL_S1 : C::COL_S0);
      const uint32_t col_p = tmem + (t ? C::COL_P1 : C::COL_P0);
      const uint32_t col_o = tmem + (t ? C::COL_O1 : C::COL_O0);
      auto wait_all = [&](uint64_t* bar, uint32_t parity, int code, int where) -> bool {
        const bool w = wait_or_abort_a(smem_u32(bar), parity, tmo_us, a_abort, code, where);
        return __all_sync(0xffffffffu, w);
      };
      auto do_s = [&](int j) {
        const uint64_t b0 = dK + static_cast<uint32_t>(j % STAGES) * (C::KV_BYTES >> 4);
        tc_fence_after();
        if (leader) {
          issue_qk<D>(col_s, dQ, b0, IDESC_S);
          tc_commit(&bar_s_full[t]);
        }
        __syncwarp();
      };
      auto do_pv = [&](int j) {
        const uint64_t v0 = dV + static_cast<uint32_t>(j % STAGES) * (C::KV_BYTES >> 4);
        // O restarts at every segment start of the softmax loop (key tiles 0, FLUSH, 2 FLUSH, ...)
        const bool first = (j == 0) || (C::FLUSH > 0 && osum_ok && j % (C::FLUSH > 0 ? C::FLUSH : 1) == 0);
        const bool last = (j == nkv - 1);
        tc_fence_after();
        if (leader) {
          if (first) issue_pv<D, DT, true>(col_o, col_p, v0, IDESC_O);
          else issue_pv<D, DT, false>(col_o, col_p, v0, IDESC_O);
          tc_commit(&bar_pv_done[t]);
          if (last) tc_commit(&bar_o_final[t]);
        }
        __syncwarp();
      };
      bool ok = wait_all(bar_q, 0, kDevTimeoutQ, 11);
      if (ok && nkv > 0) {
        ok = wait_all(&bar_k_full[0], 0, kDevTimeoutKV, 12);
        if (ok) do_s(0);
      }
      for (int j = 0; ok && j < n_max; ++j) {
        const int stage = j % STAGES;
        if (j < nkv) {
          if (!ALIAS) {
            if (j + 1 < nkv) {
              ok = wait_all(&bar_k_full[(j + 1) % STAGES], ((j + 1) / STAGES) & 1u, kDevTimeoutKV, 13);
              if (ok) ok = wait_all(&bar_s_free[t], j & 1u, kDevTimeoutSoftmax, 14);
              if (ok) do_s(j + 1);
            }
            if (ok) ok = wait_all(&bar_v_full[stage], (j / STAGES) & 1u, kDevTimeoutKV, 15);
            if (ok) ok = wait_all(&bar_p_full[t], j & 1u, kDevTimeoutSoftmax, 16);
            if (ok) do_pv(j);
          } else {
            ok = wait_all(&bar_v_full[stage], (j / STAGES) & 1u, kDevTimeoutKV, 15);
            if (ok) ok = wait_all(&bar_p_full[t], j & 1u, kDevTimeoutSoftmax, 16);
            if (ok) do_pv(j);
            if (ok && j + 1 < nkv) {
              ok = wait_all(&bar_k_full[(j + 1) % STAGES], ((j + 1) / STAGES) & 1u, kDevTimeoutKV, 13);
              // P_t(j) lives in S_t's columns: S_t(j+1) is issued by this thread after PV_t(j), and MMAs
              // of one issuing thread run in issue order, so PV_t(j) reads P_t(j) before it is overwritten.
              if (ok) do_s(j + 1);
            }
          }
          // This tile's use of the K/V stage ends when its MMAs complete.
          if (ok && leader) tc_commit(&bar_kv_empty[stage]);
        } else {
          // Key tile beyond this query tile's range: it never reads the stage, but its release must
          // count toward this load's phase only; waiting for the load first keeps this warp from
          // arriving a phase early (with fewer stages than key tiles it would otherwise free a stage
          // the other warp is still reading).
          ok = wait_all(&bar_k_full[stage], (j / STAGES) & 1u, kDevTimeoutKV, 21);
          if (ok) ok = wait_all(&bar_v_full[stage], (j / STAGES) & 1u, kDevTimeoutKV, 22);
          if (ok && leader) mbar_arrive(&bar_kv_empty[stage]);
        }
        __syncwarp();
      }
      // Every MMA of this warp must be complete before tensor memory is released.
      if (leader) tc_commit(&bar_mma_idle[t]);
      __syncwarp();
      mbar_wait_bounded(&bar_mma_idle[t], 0, tmo);
    }
  }
    // ------------------------------------------------------------------ teardown (warpgroup 0)
    tc_fence_before();
    asm volatile("bar.sync 0;" ::: "memory");
    if (warp == 1) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, TMEM_COLS);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_HIGH));
    // ------------------------------------------------------------------ softmax warpgroups
    const int wg = (warp - 4) >> 2;           // query tile of this warpgroup
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;        // row within the tile
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t colS = wg ? C::COL_S1 : C::COL_S0;
    const uint32_t colP = wg ? C::COL_P1 : C::COL_P0;
    const uint32_t colO = wg ? C::COL_O1 : C::COL_O0;
    const int qt0 = wg ? q01 : q00;
    const uint32_t a_s_full = smem_u32(&bar_s_full[wg]), a_s_free = smem_u32(&bar_s_free[wg]);
    const uint32_t a_p_full = smem_u32(&bar_p_full[wg]), a_pv_done = smem_u32(&bar_pv_done[wg]);
    const int nkv = wg ? nkv1 : nkv0;
    const int qi = qt0 + r;
    // Masks in key positions relative to the key block (|positions| < 2^31): the query tile starts at
    // key position rel, this thread's row at rel + r; keys at or past p.Nkv are outside the block.
    const int rel = static_cast<int>(p.q_off + qt0 - p.kv_off);
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY;
    float l = 0.0f;
    float m_sum = -INFINITY;  // reference max of O_sum (the m_ref of its last fold); O_sum holds
                              // values scaled by 2^-m_sum and is only brought to m_ref when read
    bool ok = true;

    // Key tiles in segments of FLUSH (one segment when FLUSH = 0). Between segments, once PV_t of the
    // segment's last tile is complete, O is folded into the fp32 running sum O_sum (RNE adds) and
    // the next segment's first PV_t restarts O; O is in the current reference max, O_sum is brought
    // from m_sum to it by an exact power of two. Keeping the fold out of the per-tile loop keeps that
    // loop's code identical to the unsegmented one.
    const int SEG = (C::FLUSH > 0 && osum_ok) ? C::FLUSH : (1 << 30);
    for (int j0 = 0; ok && j0 < nkv; j0 += SEG) {
      if (j0 > 0) {
        const int j = j0;
        ok = wait_or_abort_a(a_pv_done, (j - 1) & 1u, tmo_us, a_abort, kDevTimeoutMMA, 23);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool have = j > C::FLUSH;
        const float sc = (m_sum == -INFINITY) ? 0.0f : exp2_int(m_sum - m_ref);
        if (C::OSUM_SMEM) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(trow + colO + c * 32, o);
            tmem_wait_ld();
            reg_fence32(o);
            const uint32_t os = smem_u32(sOsum) + static_cast<uint32_t>(((wg * D) * 128 + r) * 4);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const uint32_t a = os + static_cast<uint32_t>((c * 32 + e) * 128 * 4);
              const float prev = have ? ld_shared_f32(a) * sc : 0.0f;
              st_shared_f32(a, prev + __uint_as_float(o[e]));
            }
          }
        } else {
          // this thread's own row of the SM's slot, written before it is read and by this thread only:
          // every earlier value is loaded first (one round trip to L2), then O is added and stored back
          float* og = sOsum + (wg * D) * 128 + r;
          float prev[D];
#pragma unroll
          for (int e = 0; e < D; ++e) prev[e] = have ? __ldcg(og + e * 128) : 0.0f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(trow + colO + c * 32, o);
            tmem_wait_ld();
            reg_fence32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) __stcg(og + (c * 32 + e) * 128, prev[c * 32 + e] * sc + __uint_as_float(o[e]));
          }
        }
        m_sum = m_ref;
      }
      const int j1 = (nkv - j0 < SEG) ? nkv : j0 + SEG;
      for (int j = j0; j < j1; ++j) {
        ok = wait_or_abort_a(a_s_full, j & 1u, tmo_us, a_abort, kDevTimeoutMMA, 18);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(trow + colS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        if (!ALIAS) {
          tc_fence_before();
          if (WARP_ARRIVE) {
            __syncwarp();
            if (lane == 0) mbar_arrive_a(a_s_free);  // S_t may now take S_t(j+1)
          } else {
            mbar_arrive_a(a_s_free);
          }
        }

        float x[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c]);
        const int k0 = j * BN;
        const bool tail = (k0 + BN > p.Nkv);
        const bool diag = CAUSAL && (k0 + BN - 1 > rel);
        if (tail || diag) {
          int lim = p.Nkv - k0;
          if (CAUSAL) {
            const int lc = rel + r - k0 + 1;
            lim = lc < lim ? lc : lim;
          }
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) x[c] = -INFINITY;
        }
        const float tmax = row_max128(x) * sl2;
        float alpha = 1.0f;
        bool rescale = false;
        if (tmax > m_ref + TAU) {
          const float m_new = ceilf(tmax);
          if (m_ref != -INFINITY) {
            alpha = exp2_int(m_ref - m_new);
            rescale = true;
          }
          m_ref = m_new;
        }
        const float cm = 192.0f + ((m_ref == -INFINITY) ? 0.0f : m_ref);
        const float2 sl2v = make_float2(sl2, sl2), ncm = make_float2(-cm, -cm);
        float2 rs2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
        const uint32_t pbuf = trow + colP;
        if (!ALIAS) {
          // fp16, P kept apart and single-buffered: compute all of P in registers first, then wait for
          // PV_t(j-1) to have read the previous P (parity wait on phase j-1 is exact: S_t(j) was issued
          // after PV_t(j-2), and PV_t(j) waits for this thread's p_full arrival), then store it.
          uint32_t pk[64];
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float2 pp = exp_pair(x[2 * c], x[2 * c + 1], sl2v, ncm);
            rs2[c & 1] = __fadd2_rn(rs2[c & 1], pp);
            pk[c] = pack2(pp.x, pp.y, 0);
          }
          if (j > 0) {
            ok = wait_or_abort_a(a_pv_done, (j - 1) & 1u, tmo_us, a_abort, kDevTimeoutMMA, 19);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          tmem_st32(pbuf, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
          tmem_st32(pbuf + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
        } else {
          // P over S: S_t(j) is complete, and its commit covers every earlier MMA of the issuing
          // thread, PV_t(j-1) included, so P_t(j-1) has been read and O_t is settled.
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int c = c4 * 16 + e;
              const float2 pp = exp_pair(x[2 * c], x[2 * c + 1], sl2v, ncm);
              rs2[c & 1] = __fadd2_rn(rs2[c & 1], pp);
              if (DT) {
                __nv_bfloat162 h2 = __floats2bfloat162_rn(pp.x, pp.y);
                const float2 hf = __bfloat1622float2(h2);
                __nv_bfloat162 l2 = __floats2bfloat162_rn(pp.x - hf.x, pp.y - hf.y);
                hi[e] = *reinterpret_cast<uint32_t*>(&h2);
                lo[e] = *reinterpret_cast<uint32_t*>(&l2);
              } else {
                hi[e] = pack2(pp.x, pp.y, 0);
              }
            }
            tmem_st16(pbuf + c4 * 16, hi);
            if (DT) tmem_st16(pbuf + 64 + c4 * 16, lo);
          }
        }
        l = l * alpha + ((rs2[0].x + rs2[1].x) + (rs2[0].y + rs2[1].y));
        // PV_t(j-1) is complete here (waited for above, or implied by S_t(j) when P is over S).
        if (__any_sync(0xffffffffu, rescale) && j > 0) {
          // O takes the new reference max (O_sum keeps its own, m_sum).
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(trow + colO + c * 32, o);
            tmem_wait_ld();
            reg_fence32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(trow + colO + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        if (WARP_ARRIVE) {
          __syncwarp();
          if (lane == 0) mbar_arrive_a(a_p_full);
        } else {
          mbar_arrive_a(a_p_full);
        }
      }
    }

    // ---------------------------------------------------------------- epilogue
    if (ok && nkv > 0) {
      ok = wait_or_abort_a(smem_u32(&bar_o_final[wg]), 0, tmo_us, a_abort, kDevTimeoutMMA, 20);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    const bool has = (nkv > 0) && (l > 0.0f);
    const float inv_l = has ? 1.0f / l : 0.0f;
    const float lse_v = has ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
    const bool store = ok && qi < p.Nq;
    const long long row = out_row_index(p.out_layout, b, h, p.H, p.Nq, qi);
    const long long lrow = static_cast<long long>(bh) * p.Nq + qi;
    bool write = store;
    bool fresh = true;
    float wa = 0.0f, wn = 1.0f, lse_out = lse_v;
    if (mode == kModeAccum && store) {
      if (!has) {
        write = false;
      } else {
        const float la = p.lse_part[lrow];
        if (la != -INFINITY) {
          fresh = false;
          const float M = fmaxf(la, lse_v);
          const float L = M + logf(expf(la - M) + expf(lse_v - M));
          wa = expf(la - L);
          wn = expf(lse_v - L);
          lse_out = L;
        }
      }
    }
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      if (ok && nkv > 0) {
        tmem_ld32(trow + colO + c * 32, o);
        tmem_wait_ld();
        reg_fence32(o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      float v[32];
      if (C::FLUSH > 0 && osum_ok && nkv > C::FLUSH) {
        const float* os = sOsum + (wg * D + c * 32) * 128 + r;
        const float sc = (m_sum == -INFINITY) ? 0.0f : exp2_int(m_sum - m_ref);
        float prev[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) prev[e] = C::OSUM_SMEM ? os[e * 128] : __ldcg(os + e * 128);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = (prev[e] * sc + __uint_as_float(o[e])) * inv_l;
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv_l;
      }
      if (write) {
        if (mode == kModeOut) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * D + c * 32);
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            uint4 w;
            w.x = pack2(v[8 * q8 + 0], v[8 * q8 + 1], DT);
            w.y = pack2(v[8 * q8 + 2], v[8 * q8 + 3], DT);
            w.z = pack2(v[8 * q8 + 4], v[8 * q8 + 5], DT);
            w.w = pack2(v[8 * q8 + 6], v[8 * q8 + 7], DT);
            dst[q8] = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.o_part + row * D + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float4 w = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
            if (mode == kModeAccum && !fresh) {
              const float4 a = dst[q4];
              w.x = wa * a.x + wn * w.x;
              w.y = wa * a.y + wn * w.y;
              w.z = wa * a.z + wn * w.z;
              w.w = wa * a.w + wn * w.w;
            }
            dst[q4] = w;
          }
        }
      }
    }
    if (write) {
      if (mode == kModeOut) {
        if (p.lse) p.lse[lrow] = lse_v;
      } else {
        p.lse_part[lrow] = lse_out;
      }
    }

    // ------------------------------------------------------------------ teardown (softmax warpgroups)
    tc_fence_before();
    asm volatile("bar.sync 0;" ::: "memory");
  }
}

template <int D, int DT, bool CAUSAL, int MODE>
__global__ void __launch_bounds__(NTHREADS2, 1)
    attn_fwd2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const KParams p) {
  attn_fwd2_body<D, DT, CAUSAL, MODE>(tmQ, tmK, tmV, p, static_cast<int>(blockIdx.x));
}

// Several chunk pairs in one launch: CTA blockIdx.x belongs to the last pair whose first unit is at or
// before it; that pair's maps, offsets, sizes, mode and accumulator replace the single-pair parameters.
template <int D, int DT, bool CAUSAL>
__global__ void __launch_bounds__(NTHREADS2, 1) attn_fwd2_multi_kernel(const __grid_constant__ MultiParams mp) {
  const int u = static_cast<int>(blockIdx.x);
  int i = 0;
  for (int k = 1; k < mp.n_pairs; ++k)
    if (mp.pair[k].unit_begin <= u) i = k;
  const PairDesc& pd = mp.pair[i];
  KParams kp = mp.common;
  kp.q_off = pd.q_off;
  kp.kv_off = pd.kv_off;
  kp.Nq = pd.Nq;
  kp.Nkv = pd.Nkv;
  kp.n_q_tiles = pd.n_q_tiles;
  kp.o_part = pd.o_part;
  kp.lse_part = pd.lse_part;
  kp.mode = pd.mode;
  attn_fwd2_body<D, DT, CAUSAL, kModeMulti>(pd.q, pd.k, pd.v, kp, u - pd.unit_begin);
}

template <int D, int DT, bool CAUSAL, int MODE>
int launch_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, KParams kp, int Nq, int BH,
             cudaStream_t stream) {
  auto kern = attn_fwd2_kernel<D, DT, CAUSAL, MODE>;
  static PerDeviceOnce attr;  // the attributes belong to each device's context
  int dev = 0;
  if (!attr.done(&dev)) {
    // setmaxnreg.inc waits until its registers are free: the launch must hold at least the split,
    // or the softmax warpgroups would wait forever. Refuse to launch otherwise.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncGetAttributes(attention)");
    if (fa.numRegs * NTHREADS2 < 128 * REGS_LOW + 256 * REGS_HIGH) {
      set_error("attention kernel built with %d registers/thread; the register split needs %d",
                fa.numRegs, (128 * REGS_LOW + 256 * REGS_HIGH + NTHREADS2 - 1) / NTHREADS2);
      return CQSA_ERR_UNSUPPORTED;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg2<D, DT>::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(attention smem)");
    attr.mark(dev);
  }
  kp.n_q_tiles = (Nq + 2 * BM - 1) / (2 * BM);  // pairs of query tiles
  const long long grid = static_cast<long long>(kp.n_q_tiles) * BH;
  kern<<<static_cast<int>(grid), NTHREADS2, Cfg2<D, DT>::SMEM_BYTES, stream>>>(mq, mk, mv, kp);
  return cuda_status(cudaGetLastError(), "attention kernel launch");
}

template <int D, int DT>
int dispatch_mode(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const KParams& kp, int Nq,
                  int BH, int causal, int mode, cudaStream_t s) {
  if (causal) {
    if (mode == kModeOut) return launch_t<D, DT, true, kModeOut>(mq, mk, mv, kp, Nq, BH, s);
    if (mode == kModePart) return launch_t<D, DT, true, kModePart>(mq, mk, mv, kp, Nq, BH, s);
    return launch_t<D, DT, true, kModeAccum>(mq, mk, mv, kp, Nq, BH, s);
  }
  if (mode == kModeOut) return launch_t<D, DT, false, kModeOut>(mq, mk, mv, kp, Nq, BH, s);
  if (mode == kModePart) return launch_t<D, DT, false, kModePart>(mq, mk, mv, kp, Nq, BH, s);
  return launch_t<D, DT, false, kModeAccum>(mq, mk, mv, kp, Nq, BH, s);
}

// Heads per group of work units: every head when the K/V of all heads fit in half of L2 (64 MB),
// otherwise as many as do (at least one).
int head_group_for(int BH, long long Nkv, int d) {
  const long long per_head = 2LL * (Nkv > 0 ? Nkv : 1) * d * 2;
  const long long budget = static_cast<long long>(CQSA_KV_GROUP_MB) << 20;
  if (budget <= 0 || per_head * BH <= budget) return BH;
  const long long g = budget / per_head;
  return static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 4-D map over tokens [0, N) of a [B,H,Nalloc,d] (layout BHND) or [B,Nalloc,H,d] (BNHD) tensor: dims
// (d, N, H, B), box (64,128,1,1),
// 128-byte swizzle (the box row is exactly 128 bytes), zero fill outside the tensor.
int make_map(CUtensorMap* m, const void* base, int dtype, int layout, int B, int H, int N, int d, long long Nalloc) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return CQSA_ERR_CUDA;
  }
  const cuuint64_t es = 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N > 0 ? N : 1),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  // Nalloc: tokens per head in the buffer (>= N); the map covers tokens [0, N) of each head
  const cuuint64_t na = static_cast<cuuint64_t>(Nalloc > N ? Nalloc : (N > 0 ? N : 1));
  cuuint64_t strides[3];
  if (layout == CQSA_LAYOUT_BHND) {
    strides[0] = d * es;
    strides[1] = na * d * es;
    strides[2] = static_cast<cuuint64_t>(H) * na * d * es;
  } else {
    strides[0] = static_cast<cuuint64_t>(H) * d * es;
    strides[1] = d * es;
    strides[2] = na * H * d * es;
  }
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, dtype == CQSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return CQSA_ERR_CUDA;
  }
  return CQSA_OK;
}

template <int D, int DT, bool CAUSAL>
int launch_multi_t(const MultiParams& mp, int grid, cudaStream_t stream) {
  auto kern = attn_fwd2_multi_kernel<D, DT, CAUSAL>;
  static PerDeviceOnce attr;  // the attributes belong to each device's context
  int dev = 0;
  if (!attr.done(&dev)) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncGetAttributes(attention, several pairs)");
    if (fa.numRegs * NTHREADS2 < 128 * REGS_LOW + 256 * REGS_HIGH) {
      set_error("multi-pair attention kernel built with %d registers/thread; the register split needs %d",
                fa.numRegs, (128 * REGS_LOW + 256 * REGS_HIGH + NTHREADS2 - 1) / NTHREADS2);
      return CQSA_ERR_UNSUPPORTED;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg2<D, DT>::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(attention smem, several pairs)");
    attr.mark(dev);
  }
  kern<<<grid, NTHREADS2, Cfg2<D, DT>::SMEM_BYTES, stream>>>(mp);
  return cuda_status(cudaGetLastError(), "attention kernel launch (several pairs)");
}

}  // namespace

int device_error_word(DevErr* out, int clear) {
  int rc = cuda_status(cudaMemcpyFromSymbol(out, g_dev_err, sizeof(DevErr)), "read device error word");
  if (rc != CQSA_OK || !clear || out->code == 0) return rc;
  DevErr z = {0, 0, 0, 0};
  return cuda_status(cudaMemcpyToSymbol(g_dev_err, &z, sizeof(z)), "clear device error word");
}

int device_error_word_on(DevErr* out, cudaStream_t s) {
  int rc = cuda_status(cudaMemcpyFromSymbolAsync(out, g_dev_err, sizeof(DevErr), 0, cudaMemcpyDeviceToHost, s),
                       "read device error word");
  if (rc == CQSA_OK) rc = cuda_status(cudaStreamSynchronize(s), "read device error word");
  if (rc != CQSA_OK || out->code == 0) return rc;
  static const DevErr z = {0, 0, 0, 0};
  rc = cuda_status(cudaMemcpyToSymbolAsync(g_dev_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s),
                   "clear device error word");
  if (rc == CQSA_OK) rc = cuda_status(cudaStreamSynchronize(s), "clear device error word");
  return rc;
}

int launch_attention(const AttnArgs& a, cudaStream_t stream) {
  if (a.Nq <= 0) return CQSA_OK;
  CUtensorMap mq, mk, mv;
  // An empty KV block issues no loads; its maps only need a valid base, so reuse Q's.
  const void* kb = a.Nkv > 0 ? a.k : a.q;
  const void* vb = a.Nkv > 0 ? a.v : a.q;
  const int nkv_map = a.Nkv > 0 ? a.Nkv : a.Nq;
  const long long kv_alloc = a.Nkv > 0 ? a.kv_tokens_alloc : a.q_tokens_alloc;
  int rc = make_map(&mq, a.q, a.dtype, a.in_layout, a.B, a.H, a.Nq, a.d, a.q_tokens_alloc);
  if (rc == CQSA_OK) rc = make_map(&mk, kb, a.dtype, a.in_layout, a.B, a.H, nkv_map, a.d, kv_alloc);
  if (rc == CQSA_OK) rc = make_map(&mv, vb, a.dtype, a.in_layout, a.B, a.H, nkv_map, a.d, kv_alloc);
  if (rc != CQSA_OK) return rc;
  KParams kp;
  kp.H = a.H;
  kp.BH = a.B * a.H;
  kp.Nq = a.Nq;
  kp.Nkv = a.Nkv;
  kp.q_off = a.q_off;
  kp.kv_off = a.kv_off;
  kp.scale_log2 = a.scale * 1.4426950408889634f;
  kp.n_q_tiles = 0;  // set per kernel variant at launch
  kp.out = a.out;
  kp.lse = a.lse;
  kp.o_part = a.o_part;
  kp.lse_part = a.lse_part;
  kp.out_layout = a.out_layout;
  kp.timeout_ns = timeout_ns();
  kp.timeout_us = static_cast<unsigned>(kp.timeout_ns / 1000ull > 0xffffffffull ? 0xffffffffull
                                                                                : kp.timeout_ns / 1000ull + 1ull);
  kp.fault = debug_fault();
  kp.mode = a.mode;
  kp.head_group = head_group_for(kp.BH, a.Nkv, a.d);
  const long long grid = static_cast<long long>((a.Nq + BM - 1) / BM) * kp.BH;
  if (grid > 0x7fffffffLL) {
    set_error("problem too large for one launch (%lld tiles)", grid);
    return CQSA_ERR_UNSUPPORTED;
  }
  const bool c = a.causal != 0;
  if (a.d == 64) {
    return a.dtype == CQSA_BF16 ? dispatch_mode<64, 1>(mq, mk, mv, kp, a.Nq, kp.BH, c, a.mode, stream)
                                : dispatch_mode<64, 0>(mq, mk, mv, kp, a.Nq, kp.BH, c, a.mode, stream);
  }
  return a.dtype == CQSA_BF16 ? dispatch_mode<128, 1>(mq, mk, mv, kp, a.Nq, kp.BH, c, a.mode, stream)
                              : dispatch_mode<128, 0>(mq, mk, mv, kp, a.Nq, kp.BH, c, a.mode, stream);
}

int launch_attention_multi(const AttnArgs* pairs, int n, cudaStream_t stream) {
  if (n < 1 || n > kMaxWavePairs) {
    set_error("a multi-pair launch takes 1..%d chunk pairs (got %d)", kMaxWavePairs, n);
    return CQSA_ERR_INVALID;
  }
  const AttnArgs& a0 = pairs[0];
  static thread_local MultiParams mp;  // ~14 KB: kept off the stack
  memset(&mp, 0, sizeof(mp));
  KParams& kp = mp.common;
  kp.H = a0.H;
  kp.BH = a0.B * a0.H;
  kp.scale_log2 = a0.scale * 1.4426950408889634f;
  kp.out = a0.out;
  kp.lse = a0.lse;
  kp.out_layout = a0.out_layout;
  kp.timeout_ns = timeout_ns();
  kp.timeout_us = static_cast<unsigned>(kp.timeout_ns / 1000ull > 0xffffffffull ? 0xffffffffull
                                                                                : kp.timeout_ns / 1000ull + 1ull);
  kp.fault = debug_fault();
  long long max_kv = 0;
  for (int i = 0; i < n; ++i) max_kv = pairs[i].Nkv > max_kv ? pairs[i].Nkv : max_kv;
  kp.head_group = head_group_for(kp.BH, max_kv, a0.d);
  long long units = 0;
  int np = 0;
  for (int i = 0; i < n; ++i) {
    const AttnArgs& a = pairs[i];
    if (a.B != a0.B || a.H != a0.H || a.d != a0.d || a.dtype != a0.dtype || a.causal != a0.causal ||
        a.in_layout != a0.in_layout || a.out_layout != a0.out_layout || a.scale != a0.scale) {
      set_error("the pairs of a multi-pair launch must share B, H, d, dtype, causal, layouts and scale");
      return CQSA_ERR_INVALID;
    }
    if (a.mode != kModePart && a.mode != kModeAccum) {
      set_error("a multi-pair launch writes fp32 partials or accumulators (mode %d)", a.mode);
      return CQSA_ERR_INVALID;
    }
    if (a.Nq <= 0) continue;
    PairDesc& pd = mp.pair[np];
    const void* kb = a.Nkv > 0 ? a.k : a.q;
    const void* vb = a.Nkv > 0 ? a.v : a.q;
    const int nkv_map = a.Nkv > 0 ? a.Nkv : a.Nq;
    const long long kv_alloc = a.Nkv > 0 ? a.kv_tokens_alloc : a.q_tokens_alloc;
    int rc = make_map(&pd.q, a.q, a.dtype, a.in_layout, a.B, a.H, a.Nq, a.d, a.q_tokens_alloc);
    if (rc == CQSA_OK) rc = make_map(&pd.k, kb, a.dtype, a.in_layout, a.B, a.H, nkv_map, a.d, kv_alloc);
    if (rc == CQSA_OK) rc = make_map(&pd.v, vb, a.dtype, a.in_layout, a.B, a.H, nkv_map, a.d, kv_alloc);
    if (rc != CQSA_OK) return rc;
    pd.q_off = a.q_off;
    pd.kv_off = a.kv_off;
    pd.o_part = a.o_part;
    pd.lse_part = a.lse_part;
    pd.Nq = a.Nq;
    pd.Nkv = a.Nkv;
    pd.n_q_tiles = (a.Nq + 2 * BM - 1) / (2 * BM);
    pd.mode = a.mode;
    pd.unit_begin = static_cast<int>(units);
    units += static_cast<long long>(pd.n_q_tiles) * kp.BH;
    ++np;
  }
  if (np == 0) return CQSA_OK;
  if (units > 0x7fffffffLL) {
    set_error("multi-pair launch too large (%lld units)", units);
    return CQSA_ERR_UNSUPPORTED;
  }
  mp.n_pairs = np;
  const int grid = static_cast<int>(units);
  const bool c = a0.causal != 0;
  if (a0.d == 64) {
    if (a0.dtype == CQSA_BF16) return c ? launch_multi_t<64, 1, true>(mp, grid, stream) : launch_multi_t<64, 1, false>(mp, grid, stream);
    return c ? launch_multi_t<64, 0, true>(mp, grid, stream) : launch_multi_t<64, 0, false>(mp, grid, stream);
  }
  if (a0.dtype == CQSA_BF16) return c ? launch_multi_t<128, 1, true>(mp, grid, stream) : launch_multi_t<128, 1, false>(mp, grid, stream);
  return c ? launch_multi_t<128, 0, true>(mp, grid, stream) : launch_multi_t<128, 0, false>(mp, grid, stream);
}

}  // namespace cqsa
