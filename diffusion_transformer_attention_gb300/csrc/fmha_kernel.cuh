// Fused attention forward kernel for sm_103a (template; instantiated by fmha_dense.cu,
// fmha_sage_i8.cu, fmha_sage_f8.cu, fmha_qk16pv8.cu, fmha_mxfp8.cu and fmha_nvfp4.cu): TMA-staged
// Q/K/V tiles, tcgen05 MMAs accumulating S = Q K^T and O += P V in tensor memory (block-scaled for
// MXFP8 / NVFP4 Q/K), online softmax with exp2, optional SAGE dequantization, P re-quantization to
// FP8 (every recipe with E4M3 V), the Skip-Softmax tile test and the optional LSE output.
//
// The method is fixed by the pages ("TRTLLM Attention" user guide: dense BF16, SAGE, Skip-Softmax;
// "SAGE + Skip-Softmax -- API Design & Test Plan", Part 1 §4: bmm1/bmm2 scales and
// threshold = factor / seqlen). The pages give no kernel design; this one is built for GB300:
//
// CTA = 2 query tiles of 128 rows of one (batch, query head); 640 or 384 threads (Parts below).
//   warp 0       TMA producer: Q0, Q1 once, then K_j / V_j into two K and two V buffers.
//   warps 1, 2   MMA issuers, one per Q tile (one elected lane each): BMM1 S_i = Q_i K_j^T (SS),
//                BMM2 O_i += P_i V_j (V is MN-major, so no transpose). Warp 2 also allocates the 512
//                tensor-memory columns (S0 | S1 | O0 | O1) at the start and frees them at the end.
//   warp 3       stages the V scales (E4M3 V) and, in SAGE, the K-block scales of each KV tile; in
//                MXFP8 and NVFP4 the block scales of Q and of each K tile, which the issuers copy
//                into tensor memory for the block-scaled BMM1.
//   warps 4-     softmax warpgroups: two per Q tile (a thread owns one row = TMEM lane and 64 of its
//                128 columns; the halves exchange their maxima through shared memory, and one
//                named barrier per tile orders that exchange and carries the Skip-Softmax vote), or
//                one per Q tile (a thread owns the whole row: no exchange, and the per-tile costs
//                are paid once per 128 scores). Which one is a property of the recipe (Parts).
// Dense (BF16 P): each softmax part writes its packed P over the first columns of its own part of
// S, and BMM2 reads P from tensor memory (TS). The issuer runs O_i += P_i(j-1) V_{j-1}, S_i = Q_i K_j^T as
// soon as P_i(j-1) is ready, so while one tile's softmax turns S into P, the tensor cores work on
// the other tile.
// E4M3 P (SAGE, QK16PV8, MXFP8, NVFP4; 16 KB per tile): P goes to a shared-memory buffer and BMM2 is
// an SS MMA. S is free as soon as the softmax has loaded it, so the issuer computes S_i(j+1) while
// the softmax works on S_i(j); a per-tile barrier (o_done) returns P's buffer and O to the softmax
// after each BMM2. With 8- or 4-bit K tiles there is room for two P buffers per tile, and the
// softmax then waits for the previous BMM2 only before it rescales O (kDblP); SAGE with
// Skip-Softmax waits only before the next P (kLazyPv).
// MXFP8 / NVFP4: the block-scaled MMA reads its scale factors from tensor memory, and S0 | S1 | O0 | O1 leave
// no room, so the two tiles share one S buffer (S | O0 | O1 | scale factors): BMM1s alternate
// between the tiles, each issued once the other tile's softmax has loaded the previous S. The
// softmax groups then run about one BMM1 apart, and each S still lands before its softmax needs it.
//
// Numerics: logits are kept in log2 units (scaled by softmax_scale * log2 e). With BF16 P, O is
// rescaled lazily (only when the running max grows by more than 8, P then stays below 2^8); with
// E4M3 P it is rescaled eagerly so P = exp2(s - m_run) lies in [0, 1] and P * 448 re-quantizes on
// the same grid as the definition. The row sum uses the unquantized P. Skip-Softmax compares the
// tile max against the exact running max.
//
// Every wait is bounded; on expiry the kernel records a timeout in the device error word, tells
// the other roles to stop, drains its own copies and MMAs, frees tensor memory and exits. Named
// barriers are reached the same number of times on every path, so no thread waits on a peer
// that left.
#pragma once
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "ditattn_internal.h"
#include "fmha_common.cuh"
#include "sm103_ptx.cuh"

namespace ditattn {
namespace {

// Softmax warpgroups per Q tile and the launch shape they imply. Two (each thread holds 64 of a row's
// 128 columns, the two halves exchange the row max through shared memory) for dense BF16 and SAGE
// INT8 without Skip-Softmax; one (each thread holds the whole row) for the other recipes, all with an
// E4M3 P (SAGE FP8, QK16PV8, MXFP8, NVFP4, and SAGE INT8 with Skip-Softmax). Each measured faster for
// its recipes on GB300 (with one warpgroup SAGE FP8 ran 15% faster, dense 15% slower, SAGE INT8 the
// same without Skip-Softmax and slower only when that kernel had nothing to skip, which factor 0 no
// longer sends to it).
template <int QKF, int PVF, bool SKIP>
struct Parts {
  static constexpr int kNH = (PVF == PV_E4M3 && (QKF != QK_F16 || SKIP)) ? 1 : 2;
  static constexpr int kThreads = 128 + 256 * kNH;
  // launched at 65536 / kThreads registers (rounded down to a multiple of 8); warpgroup 0 (producer,
  // MMA issuers, scale stager) hands registers to the softmax warpgroups
  static constexpr int kLaunchRegs = kNH == 1 ? 168 : 96;
  static constexpr int kRegsWG0 = kNH == 1 ? 72 : 64;
  static constexpr int kRegsSoftmax = kNH == 1 ? 216 : 104;
  static_assert(128 * kRegsWG0 + 256 * kNH * kRegsSoftmax <= kThreads * kLaunchRegs, "register hand-over must fit");
  static_assert(kThreads * kLaunchRegs <= 65536, "one CTA per SM");
};
constexpr int kSlots = 4;  // ring of K/V tiles: K_j in slot 2j mod 4, V_j in slot 2j+1 mod 4

// Shared-memory layout for operand formats QKF / PVF. Two Q buffers of 32 KB (also the output
// staging), two K buffers and two V buffers sized to their tiles, and in SAGE mode two 16 KB
// buffers for the E4M3 P of the two query tiles, which BMM2 reads from shared memory.
template <int QKF, int PVF>
struct SmemLayout {
  static constexpr bool kNV = (QKF == QK_NVF4);
  static constexpr uint32_t kKTile = kNV ? 128u * 64u : 128u * 128u * ((QKF == QK_E4M3 || QKF == QK_MXF8) ? 1u : 2u);
  // block-scaled Q/K: one 32 x 16-byte scale matrix per 32-bit scale word of a row (MXFP8 1, NVFP4 2)
  static constexpr uint32_t kSfWords = kNV ? 2u : 1u;
  static constexpr uint32_t kVTile = 128u * 128u * (PVF == PV_E4M3 ? 1u : 2u);
  static constexpr bool kPInSmem = (PVF == PV_E4M3);
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKOff = 2 * 32768;
  static constexpr uint32_t kVOff = kKOff + 2 * kKTile;
  static constexpr uint32_t kPOff = kVOff + 2 * kVTile;
  // E4M3 P buffers per Q tile (16 KB each): two when the K tiles are 8- or 4-bit (the shared memory
  // then has room), so that a tile's P never waits for the BMM2 that read the previous one
  static constexpr uint32_t kPBufs = kPInSmem ? (kKTile <= 16384 ? 2u : 1u) : 0u;
  // 4 x 128 floats (SAGE K-block scales), or 4 x kSfWords x 512 bytes of K tiles' block scales
  static constexpr uint32_t kKsOff = kPOff + kPBufs * 2 * 16384;
  static constexpr uint32_t kVsOff = kKsOff + kSlots * 512 * kSfWords;     // 128 floats
  static constexpr uint32_t kXmaxOff = kVsOff + 512;        // [tile][half][parity][128] partial maxima
  static constexpr uint32_t kXlOff = kXmaxOff + 2 * 2 * 2 * 512;  // [tile][half][128] partial row sums
  static constexpr uint32_t kSfaOff = kXlOff + 2 * 2 * 512;  // block-scaled: the Q tiles' scales, 2 x kSfWords x 512 B
  static constexpr uint32_t kBarOff = kSfaOff + ((QKF == QK_MXF8 || kNV) ? 2 * 512 * kSfWords : 0);
  static constexpr uint32_t kSmemBytes = kBarOff + 512 + 1024;     // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};
constexpr float kLazyRescale = 8.0f;                         // log2 units
constexpr float kLog2_448 = 8.807354922057604f;

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[kSlots];
  uint64_t kv_empty[kSlots];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t ks_full[kSlots];
  uint64_t ks_empty[kSlots];
  uint64_t vs_full;
  uint64_t drain[2];
  uint64_t s_free[2];   // SAGE: the tile's softmax has loaded S (BMM1 of the next KV tile may overwrite it)
  uint64_t o_done[2];   // SAGE: BMM2 of the tile's latest KV tile is complete (P buffer free, O stable)
  uint64_t sfa_full;    // MXFP8 / NVFP4: the Q tiles' scale factors are in shared memory
  uint32_t tmem_base;
  int abort_flag;
  int skip_flag[2][2];  // [Q tile][KV tile parity]: 1 when that KV tile was skipped
  // SAGE with Skip-Softmax hands P of odd KV tiles to the issuer through p_full_odd (even tiles through
  // p_full): the softmax waits there only for the previous kept tile's BMM2, so over skipped tiles it
  // can run ahead of the issuer, and with one barrier it could complete tile j (skipped) and tile j + 1
  // (kept) while the issuer still waited for V_j; the issuer's parity test would then wait for tile
  // j + 2, which needs a BMM1 only the issuer can issue. With a barrier per KV-tile parity a barrier's
  // next phase is tile j + 2 itself, whose S needs that BMM1, so no phase completes twice before the
  // issuer tests it. (Every other path waits for the previous BMM2, or has the issuer's order, before
  // the next P, so one barrier per tile serves it.)
  uint64_t p_full_odd[2];
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");

// Bounds checks of computed indices, compiled only into a library built with DITATTN_BOUNDS_CHECK (a
// debug build): an index outside its buffer records DIT_E_BOUNDS in the device error word (unless a
// timeout is already recorded) and the caller skips that access. The default build compiles every
// check to `true` and its arguments away.
#ifdef DITATTN_BOUNDS_CHECK
__device__ __forceinline__ bool index_ok(int* err, long long idx, long long n) {
  if (idx >= 0 && idx < n) return true;
  atomicCAS(err, 0, kErrBounds);
  return false;
}
#define DIT_INDEX_OK(err, idx, n) ::ditattn::index_ok((err), (long long)(idx), (long long)(n))
#else
#define DIT_INDEX_OK(err, idx, n) true
#endif

__device__ __forceinline__ void record_timeout(const FmhaParams& p, Bars* bars) {
  atomicExch(p.err, kErrTimeout);
  *reinterpret_cast<volatile int*>(&bars->abort_flag) = 1;
}


// WITHHOLD (a self-test of the timeout path, its own instantiation so that the production kernels'
// code is unaffected): the producer issues no copy, so nothing is in flight when the other roles'
// bounded waits run out and they leave.
template <int QKF, int PVF, int KB, bool SKIP, bool WITHHOLD = false>
__global__ void __launch_bounds__(Parts<QKF, PVF, SKIP>::kThreads, 1)
    fmha_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FmhaParams p) {
  constexpr bool kQKScaled = (QKF == QK_F16 || QKF == QK_E4M3);  // Q/K codes with token-block scales (SAGE)
  // SAGE with Skip-Softmax: the softmax waits for the previous BMM2 only before writing P, so skipped
  // tiles skip that wait (measured faster there; the other instantiations keep a wait on every tile,
  // which measured faster for them). o_done then completes once per BMM2, and the skip flag needs a
  // slot per KV-tile parity.
  constexpr bool kLazyPv = SKIP && kQKScaled;
  // Two P buffers per tile (L::kPBufs): the softmax writes its n-th P into buffer n % 2, which BMM2
  // #(n-2) read; that BMM2 was issued before BMM1 of the current KV tile (the issuer issues BMM1(j+1)
  // before BMM2(j), and its MMAs complete in order), so S's arrival already frees the buffer and the
  // softmax waits for the previous BMM2 only before it rescales O. o_done then completes once per
  // BMM2, as with kLazyPv.
  constexpr bool kDblP = (SmemLayout<QKF, PVF>::kPBufs == 2);
  // the softmax may run ahead of the issuer over several KV tiles: P is handed over through one
  // barrier per KV-tile parity and the skip flag has a slot per parity (see p_full_odd)
  constexpr bool kRunAhead = kLazyPv || kDblP;
  // K tiles ahead: the producer loads K_{j+1} before V_j and the MMA issuer tests K_{j+1} before it
  // waits for the softmax to release S. Measured faster for every instantiation but dense BF16 with
  // Skip-Softmax, which keeps the K, V, K, V order.
  constexpr bool kKAhead = !(SKIP && PVF == PV_BF16);
  constexpr bool kMX = (QKF == QK_MXF8);         // block-scaled MXFP8 Q/K (scales applied inside BMM1)
  constexpr bool kNV = (QKF == QK_NVF4);         // block-scaled NVFP4 Q/K (and a tensor scale per Q and K)
  constexpr bool kBS = kMX || kNV;
  constexpr bool kPV8 = (PVF == PV_E4M3);        // E4M3 P and V with per-channel V scales (SAGE, QK16PV8, MXFP8)
  constexpr int kQKBytes = (QKF == QK_E4M3 || kBS) ? 1 : 2;  // NVFP4: two codes per byte, one 64-byte box per row
  constexpr int kPVBytes = (PVF == PV_E4M3) ? 1 : 2;
  constexpr uint32_t kQTileBytes = kNV ? 128u * 64u : 128u * 128u * kQKBytes;
  constexpr uint32_t kVTileBytes = 128u * 128u * kPVBytes;
  constexpr int kMma1Kind = (QKF == QK_E4M3) ? KIND_F8F6F4 : KIND_F16;
  constexpr int kMma2Kind = (PVF == PV_E4M3) ? KIND_F8F6F4 : KIND_F16;
  constexpr int kK1Steps = (kQKBytes == 1) ? 4 : 8;  // K = 128 in steps of 32 (8-bit) or 16
  // tensor-memory columns: S and O of tile i; block-scaled Q/K add, per tile, 4 columns of Q scales and
  // 4 of K scales per 32-bit scale word of a row
  constexpr uint32_t kSfWords = kNV ? 2u : 1u;
  constexpr uint32_t kColS1 = kBS ? 0 : 128, kColO0 = kBS ? 128 : 256;
  constexpr uint32_t kColSfa = 384, kColSfb = 384 + 8 * kSfWords;
  constexpr int kK2Steps = (PVF == PV_E4M3) ? 4 : 8;
  constexpr uint32_t kIdesc1 = (QKF == QK_BF16)  ? make_idesc(1, 1, 0, 0, 128, 128)
                               : (QKF == QK_F16) ? make_idesc(0, 0, 0, 0, 128, 128)
                                                 : make_idesc(0, 0, 0, 0, 128, 128);
  constexpr uint32_t kIdesc2 = (PVF == PV_BF16) ? make_idesc(1, 1, 0, 1, 128, 128) : make_idesc(0, 0, 0, 1, 128, 128);

  using L = SmemLayout<QKF, PVF>;
  using P = Parts<QKF, PVF, SKIP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBarOff);
  float* s_ks = reinterpret_cast<float*>(smem + L::kKsOff);
  float* s_vs = reinterpret_cast<float*>(smem + L::kVsOff);
  const volatile int* abort_flag = &bars->abort_flag;
  // the barrier that hands P of KV tile j of Q tile i to the issuer, and the parity of that phase
  auto p_full_bar = [&](int i, int j) { return (kRunAhead && (j & 1)) ? &bars->p_full_odd[i] : &bars->p_full[i]; };
  auto p_full_par = [&](int j) -> uint32_t { return kRunAhead ? (uint32_t)((j >> 1) & 1) : (uint32_t)(j & 1); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.y, b = blockIdx.z;
  const int hkv = hq / p.group;
  const int q0 = blockIdx.x * 256;
  const int nt = p.n_kv_tiles;
  const uint64_t budget = p.wait_budget_ns;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);  // one commit from each MMA issuer
      mbar_init(&bars->ks_full[s], 32);
      mbar_init(&bars->ks_empty[s], kBS ? 2 : 8 * P::kNH);  // SAGE: one arrival per softmax warp; block-scaled: per issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4 * P::kNH);  // one arrival per softmax warp of the tile
      if constexpr (kRunAhead) mbar_init(&bars->p_full_odd[i], 4 * P::kNH);
      mbar_init(&bars->o_full[i], 1);
    }
    mbar_init(&bars->vs_full, 32);
    mbar_init(&bars->sfa_full, 32);
    mbar_init(&bars->drain[0], 1);
    mbar_init(&bars->drain[1], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_free[i], 4 * P::kNH);  // one arrival per softmax warp of the tile
      mbar_init(&bars->o_done[i], 1);
    }
    bars->abort_flag = 0;
    bars->skip_flag[0][0] = bars->skip_flag[0][1] = bars->skip_flag[1][0] = bars->skip_flag[1][1] = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  // Launched at 96 registers per thread: warpgroup 0 (producer, MMA, allocator, scale stager)
  // hands registers to the four softmax warpgroups, which hold 64 scores per thread.
  if (warp < 4) {
  regs_dec<P::kRegsWG0>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && !WITHHOLD) {
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      int issued[kSlots] = {0, 0, 0, 0};
      bool ok = true;
      mbar_arrive_expect_tx(&bars->q_full, 2 * kQTileBytes);
      for (int i = 0; i < 2; ++i) {
        uint8_t* dst = smem + L::kQOff + i * 32768;
        if (kQKBytes == 2) {
          tma_load_4d(dst, &tm_q, &bars->q_full, 0, q0 + 128 * i, hq, b, pol_q);
          tma_load_4d(dst + 16384, &tm_q, &bars->q_full, 64, q0 + 128 * i, hq, b, pol_q);
        } else {
          tma_load_4d(dst, &tm_q, &bars->q_full, 0, q0 + 128 * i, hq, b, pol_q);
        }
      }
      // kKAhead: K_0, then K_{j+1} before V_j. BMM1(j+1) needs its K tile before BMM2(j) needs V_j, and
      // K_{j+1}'s buffer is freed first (by BMM1(j-1), which the issuer runs before BMM2(j-2), the last
      // reader of V_j's buffer), so a V buffer still in use never holds back the next K tile.
      // Otherwise K_j, V_j, K_{j+1}, ... Each slot receives its tiles in order either way.
      for (int n = 0; n <= 2 * nt && ok; ++n) {
        int j, kv;
        if constexpr (kKAhead) {
          j = (n == 0) ? 0 : ((n & 1) ? (n + 1) >> 1 : (n >> 1) - 1);
          kv = (n == 0) ? 0 : ((n & 1) ? 0 : 1);
          if (kv == 0 && j >= nt) continue;  // no K_{j+1} after the last tile
        } else {
          if (n == 2 * nt) break;
          j = n >> 1;
          kv = n & 1;
        }
        const int t = 2 * j + kv, s = t & (kSlots - 1), u = t / kSlots;
        if (!mbar_wait_bounded(&bars->kv_empty[s], (u & 1) ^ 1, budget, abort_flag)) {
          record_timeout(p, bars);
          ok = false;
          break;
        }
        uint8_t* dst = smem + (kv ? L::kVOff + (s >> 1) * L::kVTile : L::kKOff + (s >> 1) * L::kKTile);
        const CUtensorMap* map = kv ? &tm_v : &tm_k;
        const int bytes = kv ? kVTileBytes : kQTileBytes;
        const int eb = kv ? kPVBytes : kQKBytes;
        mbar_arrive_expect_tx(&bars->kv_full[s], bytes);
        if (eb == 2) {
          tma_load_4d(dst, map, &bars->kv_full[s], 0, 128 * j, hkv, b, pol_kv);
          tma_load_4d(dst + 16384, map, &bars->kv_full[s], 64, 128 * j, hkv, b, pol_kv);
        } else {
          tma_load_4d(dst, map, &bars->kv_full[s], 0, 128 * j, hkv, b, pol_kv);
        }
        ++issued[s];
      }
      if (!ok) {
        // drain: wait (bounded) for every copy this thread started before shared memory goes away
        mbar_wait_bounded(&bars->q_full, 0, budget, nullptr);
        for (int s = 0; s < kSlots; ++s)
          if (issued[s] > 0) mbar_wait_bounded(&bars->kv_full[s], (issued[s] - 1) & 1, budget, nullptr);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers, one warp per Q tile
    // Each issuer reacts only to its own tile's barriers, so one tile's P never waits while the
    // other tile's MMAs are being pushed into the (shallow) tensor-core queue. The whole warp runs
    // the loop in uniform control flow; one elected lane issues the tcgen05 instructions.
    const int i = warp - 1;
    const uint32_t leader = elect_one();
    bool ok = mbar_wait_bounded(&bars->q_full, 0, budget, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && leader) record_timeout(p, bars);
    tc_fence_after();
    const uint32_t sbase = smem_u32(smem);
    // Q/K operands: 128-byte rows with the 128-byte swizzle; NVFP4's 64-byte rows with the 64-byte one
    const uint64_t aq = kNV ? make_sdesc_sw64(sbase + L::kQOff + i * 32768, 16, 512)
                            : make_sdesc_sw128(sbase + L::kQOff + i * 32768, 16, 1024);
    const uint64_t dk0 = kNV ? make_sdesc_sw64(sbase + L::kKOff, 16, 512) : make_sdesc_sw128(sbase + L::kKOff, 16, 1024);
    const uint64_t dv0 = make_sdesc_sw128(sbase + L::kVOff, kPVBytes == 2 ? 16384 : 8192, 1024);
    const uint32_t d_s = tbase + kColS1 * i;
    const uint32_t d_o = tbase + kColO0 + 128 * i;
    const uint32_t t_sfa = tbase + kColSfa + 4 * kSfWords * i;  // block-scaled: this tile's Q scale words
    const uint32_t t_sfb = tbase + kColSfb + 4 * kSfWords * i;  // and its copy of the K tile's
    volatile int (*skip_flag)[2] = bars->skip_flag;
    auto wait = [&](uint64_t* bar, int parity) {
      return __all_sync(0xffffffffu, mbar_wait_bounded(bar, (uint32_t)parity, budget, abort_flag));
    };
    // K_j sits in K buffer j % 2 and V_j in V buffer j % 2 (ring slots 2j and 2j + 1 mod 4); the
    // descriptor start address advances in 16-byte units inside its low 14 bits.
    auto bmm1 = [&](int j) {  // S_i = Q_i K_j^T, then release K_j's slot
      const uint64_t bk = dk0 + (uint64_t)(((j & 1) * L::kKTile) >> 4);
      if constexpr (kMX) {
        // K_j's scale words into tensor memory (ordered before the MMAs below), then the four
        // 32-wide K slices, each using its byte of every Q and K scale word
        tmem_cp_32x128b_x4_if(leader, t_sfb, make_sdesc_rows16(sbase + L::kKsOff + (j & 3) * 512));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_mxf8_if(leader, d_s, aq + (uint64_t)((kk * 32) >> 4), bk + (uint64_t)((kk * 32) >> 4),
                      make_idesc_mxf8(128, 128, kk), t_sfa, t_sfb, kk > 0 ? 1u : 0u);
      } else if constexpr (kNV) {
        // two 64-wide K slices (32 bytes of packed codes each), each with its own scale word per row
        // (the four E4M3 scales of its 16-channel blocks) in its own four columns
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          tmem_cp_32x128b_x4_if(leader, t_sfb + 4 * kk,
                                make_sdesc_rows16(sbase + L::kKsOff + (j & 3) * 1024 + kk * 512));
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          mma_nvf4_if(leader, d_s, aq + (uint64_t)((kk * 32) >> 4), bk + (uint64_t)((kk * 32) >> 4),
                      make_idesc_nvf4(128, 128), t_sfa + 4 * kk, t_sfb + 4 * kk, kk > 0 ? 1u : 0u);
      } else {
#pragma unroll
        for (int kk = 0; kk < kK1Steps; ++kk) {
          const uint32_t off = (kQKBytes == 2) ? (kk >> 2) * 16384 + (kk & 3) * 32 : kk * 32;
          mma_ss_if<kMma1Kind>(leader, d_s, aq + (off >> 4), bk + (off >> 4), kIdesc1, kk > 0 ? 1u : 0u);
        }
      }
      mma_commit_if(leader, &bars->s_full[i]);
      mma_commit_if(leader, &bars->kv_empty[(2 * j) & 3]);
      if constexpr (kBS) mma_commit_if(leader, &bars->ks_empty[j & 3]);  // the scales' slot
    };
    // May S_i(j) be written? With a buffer per tile: once this tile's softmax has loaded S_i(j-1).
    // MXFP8 (one S for both tiles, BMM1s in the order Q0 Q1 Q0 Q1 ...): once the other tile's
    // softmax has loaded the S computed just before, which also orders every earlier BMM1 of this
    // issuer (and its reads of the scale columns) before the new one.
    auto s_writable = [&](int j) -> bool {
      if constexpr (kBS) {
        return (i == 0) ? (j == 0 || wait(&bars->s_free[1], (j - 1) & 1)) : wait(&bars->s_free[0], j & 1);
      } else {
        return j == 0 || wait(&bars->s_free[i], (j - 1) & 1);
      }
    };
    auto k_ready = [&](int j) -> bool {  // K_j staged (and, in MXFP8 / NVFP4, its scales)
      const int tk = 2 * j;
      if constexpr (kBS) {
        return __all_sync(0xffffffffu, mbar_wait2_bounded(&bars->kv_full[tk & 3], (tk >> 2) & 1, &bars->ks_full[j & 3],
                                                          (j >> 2) & 1, budget, abort_flag));
      } else {
        return wait(&bars->kv_full[tk & 3], (tk >> 2) & 1);
      }
    };
    if constexpr (L::kPInSmem) {
      // E4M3 P in shared memory: BMM1 of the next KV tile overwrites S as soon as the softmax has
      // loaded it, so each tile's S(j+1) is computed while its softmax turns S(j) into P(j).
      // BMM2 is an SS MMA (P K-major, V MN-major); o_done tells the softmax when P's buffer and O
      // are free again.
      const uint64_t ap = make_sdesc_sw128(sbase + L::kPOff + i * L::kPBufs * 16384, 16, 1024);
      int n2 = 0;  // BMM2s issued so far (kDblP: BMM2 #n reads P buffer n % 2)
      if constexpr (kBS) {
        // this Q tile's scale words, once, ahead of every MMA that reads them
        if (ok) ok = wait(&bars->sfa_full, 0);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (uint32_t w = 0; w < kSfWords; ++w)
            tmem_cp_32x128b_x4_if(leader, t_sfa + 4 * w,
                                  make_sdesc_rows16(sbase + L::kSfaOff + (i * kSfWords + w) * 512));
        }
      }
      if (ok) ok = k_ready(0) && s_writable(0);
      if (ok) {
        tc_fence_after();
        bmm1(0);
      }
      for (int j = 0; j < nt && ok; ++j) {
        if (j + 1 < nt) {
          // kKAhead: K first. It is normally staged already, and testing it before the wait for the
          // softmax keeps that test's latency (a barrier test costs as much as a wake-up) off the
          // hand-over of S.
          if constexpr (kKAhead) {
            ok = k_ready(j + 1) && s_writable(j + 1);
          } else {
            ok = s_writable(j + 1) && k_ready(j + 1);
          }
          if (!ok) break;
          tc_fence_after();
          bmm1(j + 1);
        }
        const int tv = 2 * j + 1;
        ok = wait(&bars->kv_full[tv & 3], (tv >> 2) & 1) && wait(p_full_bar(i, j), p_full_par(j));
        if (!ok) break;
        tc_fence_after();
        const bool skipped = SKIP && skip_flag[i][kRunAhead ? (j & 1) : 0] != 0;
        if (!skipped) {
          // (the first KV tile is never skipped, so O is initialized by BMM2 of tile 0)
          const uint64_t bv = dv0 + (uint64_t)(((j & 1) * L::kVTile) >> 4);
          const uint64_t ap_n = ap + (uint64_t)(((kDblP ? (n2 & 1) : 0) * 16384) >> 4);
          ++n2;
#pragma unroll
          for (int kk = 0; kk < kK2Steps; ++kk)
            mma_ss_if<kMma2Kind>(leader, d_o, ap_n + (uint64_t)((kk * 32) >> 4), bv + (uint64_t)((kk * 4096) >> 4),
                                 kIdesc2, (j > 0 || kk > 0) ? 1u : 0u);
        }
        // o_done: one phase per BMM2 (kLazyPv) or per KV tile
        if (!kRunAhead || !skipped) mma_commit_if(leader, &bars->o_done[i]);
        mma_commit_if(leader, &bars->kv_empty[tv & 3]);
      }
    } else {
      // P in tensor memory over S: O_i += P_i(j-1) V_{j-1} then S_i = Q_i K_j^T, once P_i(j-1) is ready.
      for (int j = 0; j <= nt && ok; ++j) {
        const int tk = 2 * j, tv = 2 * j - 1;
        if (j < nt) {
          ok = wait(&bars->kv_full[tk & 3], (tk >> 2) & 1);
          if (!ok) break;
        }
        if (j >= 1) {
          ok = wait(&bars->kv_full[tv & 3], (tv >> 2) & 1) && wait(p_full_bar(i, j - 1), p_full_par(j - 1));
          if (!ok) break;
        }
        tc_fence_after();
        if (j >= 1 && (!SKIP || skip_flag[i][0] == 0)) {
          const uint64_t bv = dv0 + (uint64_t)((((j - 1) & 1) * L::kVTile) >> 4);
#pragma unroll
          for (int kk = 0; kk < kK2Steps; ++kk) {
            const uint32_t off = (kPVBytes == 2) ? kk * 2048 : kk * 4096;
            // P (bf16, two values per column) sits in the first 64 / kNH columns of each softmax part's
            // region of S (part h at columns 128 h / kNH): K step kk reads 8 columns
            constexpr int kPerPart = kK2Steps / P::kNH;
            const uint32_t pa = d_s + (kk / kPerPart) * (128 / P::kNH) + 8 * (kk % kPerPart);
            mma_ts_if<kMma2Kind>(leader, d_o, pa, bv + (off >> 4), kIdesc2, (j > 1 || kk > 0) ? 1u : 0u);
          }
        }
        // a K/V slot is free once both issuers have committed their last use of it
        if (j >= 1) mma_commit_if(leader, &bars->kv_empty[tv & 3]);
        if (j < nt) bmm1(j);
      }
    }
    if (ok) {
      mma_commit_if(leader, &bars->o_full[i]);
    } else if (leader) {
      record_timeout(p, bars);
    }
    // drain: no MMA of this issuer may still be running when tensor memory is freed
    mma_commit_if(leader, &bars->drain[i]);
    mbar_wait_bounded(&bars->drain[i], 0, budget, nullptr);
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ scale stager (V scales; SAGE K scales)
    if constexpr (kPV8) {
      const float* vs = p.v_scale + ((size_t)b * p.Hkv + hkv) * kHeadDim;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        s_vs[lane * 4 + e] = DIT_INDEX_OK(p.err, ((long long)b * p.Hkv + hkv) * kHeadDim + lane * 4 + e,
                                          (long long)p.B * p.Hkv * kHeadDim)
                                 ? vs[lane * 4 + e]
                                 : 0.0f;
      mbar_arrive(&bars->vs_full);
    }
    if constexpr (kBS) {
      // Block-scale words of the two Q tiles once, then of every K tile through the ring. A row has
      // W = kSfWords 32-bit words (MXFP8: 4 E8M0 bytes for channels 32c..; NVFP4: 8 E4M3 bytes for
      // channels 16c.., word w covering the MMA's K slice w). Each word of a 128-row tile goes to a
      // 32 x 16-byte matrix whose row l holds that word of rows l, l+32, l+64, l+96: the tensor-memory
      // copy puts them in columns 0-3 of lane l of each lane quarter, where the MMA reads row 32c + l
      // from column c. Rows past the end get 0 (their codes are zero, as TMA fills them).
      constexpr int W = (int)kSfWords;
      // base_words / all_words: the offset of `base` in its array and the array's size, in words
      // (bounds-checked builds only)
      auto load_words = [&](const uint32_t* base, long long base_words, long long all_words, int row, int nrows,
                            uint32_t* w) {
        if (row < nrows && DIT_INDEX_OK(p.err, base_words + (long long)row * W + (W - 1), all_words)) {
          if constexpr (W == 2) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(base) + row);
            w[0] = u.x;
            w[1] = u.y;
          } else {
            w[0] = __ldg(base + row);
          }
        } else {
#pragma unroll
          for (int ww = 0; ww < W; ++ww) w[ww] = 0u;
        }
      };
      const uint32_t* qsf = reinterpret_cast<const uint32_t*>(p.q_sf) + ((size_t)b * p.Hq + hq) * p.Sq * W;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        uint32_t w[4][W];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          load_words(qsf, ((long long)b * p.Hq + hq) * p.Sq * W, (long long)p.B * p.Hq * p.Sq * W,
                     q0 + 128 * t + 32 * c + lane, p.Sq, w[c]);
#pragma unroll
        for (int ww = 0; ww < W; ++ww)
          *reinterpret_cast<uint4*>(smem + L::kSfaOff + (t * W + ww) * 512 + lane * 16) =
              make_uint4(w[0][ww], w[1][ww], w[2][ww], w[3][ww]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->sfa_full);
      const uint32_t* ksf = reinterpret_cast<const uint32_t*>(p.k_sf) + ((size_t)b * p.Hkv + hkv) * p.Skv * W;
      auto load_tile = [&](int j, uint32_t (*w)[L::kSfWords]) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          load_words(ksf, ((long long)b * p.Hkv + hkv) * p.Skv * W, (long long)p.B * p.Hkv * p.Skv * W,
                     128 * j + 32 * c + lane, j < nt ? p.Skv : 0, w[c]);
      };
      constexpr int kAhead = (W == 2) ? 2 : 4;
      uint32_t pre[kAhead][4][W];
#pragma unroll
      for (int d = 0; d < kAhead; ++d) load_tile(d, pre[d]);
      for (int j = 0; j < nt; ++j) {
        const int e = j & 3, u = j >> 2;
        const bool ok = mbar_wait_bounded(&bars->ks_empty[e], (u & 1) ^ 1, budget, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) record_timeout(p, bars);
          break;
        }
#pragma unroll
        for (int ww = 0; ww < W; ++ww)
          *reinterpret_cast<uint4*>(smem + L::kKsOff + (e * W + ww) * 512 + lane * 16) =
              make_uint4(pre[0][0][ww], pre[0][1][ww], pre[0][2][ww], pre[0][3][ww]);
        fence_proxy_async_smem();
        mbar_arrive(&bars->ks_full[e]);
#pragma unroll
        for (int d = 0; d + 1 < kAhead; ++d)
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int ww = 0; ww < W; ++ww) pre[d][c][ww] = pre[d + 1][c][ww];
        load_tile(j + kAhead, pre[kAhead - 1]);
      }
    }
    if constexpr (kQKScaled) {
      bool ok = true;
      const float* ks = p.k_scale + ((size_t)b * p.Hkv + hkv) * p.nkb;
      // A tile's 128 / KB block scales, four slots per lane (0 for slots past them and past the
      // end of K). The loads run kAhead tiles ahead of the ring, so their latency stays off the
      // softmax's path even when most tiles are skipped and the ring turns over quickly.
      auto load_tile = [&](int j, float* v) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int g = lane * 4 + q;
          const int col = 128 * j + g * KB;
          v[q] = (j < nt && g < 128 / KB && col < p.Skv &&
                  DIT_INDEX_OK(p.err, ((long long)b * p.Hkv + hkv) * p.nkb + col / KB, (long long)p.B * p.Hkv * p.nkb))
                     ? __ldg(ks + col / KB)
                     : 0.0f;
        }
      };
      constexpr int kAhead = 4;
      float pre[kAhead][4];
#pragma unroll
      for (int d = 0; d < kAhead; ++d) load_tile(d, pre[d]);
      for (int j = 0; j < nt; ++j) {
        const int e = j & 3, u = j >> 2;
        ok = mbar_wait_bounded(&bars->ks_empty[e], (u & 1) ^ 1, budget, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) record_timeout(p, bars);
          break;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (lane * 4 + q < 128 / KB) s_ks[e * 128 + lane * 4 + q] = pre[0][q];
        mbar_arrive(&bars->ks_full[e]);
#pragma unroll
        for (int d = 0; d + 1 < kAhead; ++d)
#pragma unroll
          for (int q = 0; q < 4; ++q) pre[d][q] = pre[d + 1][q];
        load_tile(j + kAhead, pre[kAhead - 1]);
      }
    }
  }
  } else {
    if constexpr (P::kNH == 2) {
      // ------------------------------------------------------------ softmax groups
      regs_inc<P::kRegsSoftmax>();
      const int g = (warp - 4) >> 2;                 // softmax warpgroup 0..3
      const int i = g >> 1;                          // Q tile within the CTA
      const int h = g & 1;                           // column half: S/O columns 64h .. 64h+63
      const int r = ((warp & 3) << 5) + lane;        // row within the tile == TMEM lane
      const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
      const uint32_t t_s = tbase + lane_base + kColS1 * i + 64 * h;
      const uint32_t t_o = tbase + lane_base + kColO0 + 128 * i + 64 * h;
      const int qrow = q0 + 128 * i + r;
      const bool row_valid = qrow < p.Sq;
      const uint32_t tile_bar = 1 + i;               // the 256 threads of this Q tile
      const uint32_t group_bar = 3 + g;              // the 128 threads of this warpgroup
      float* xmax = reinterpret_cast<float*>(smem + L::kXmaxOff);
      float* xl = reinterpret_cast<float*>(smem + L::kXlOff);
      float c = p.c_scale;
      if constexpr (kNV) c = c / (__ldg(p.q_gs) * __ldg(p.k_gs));  // BMM1 carries both tensor scales
      if constexpr (kQKScaled) {
        const float qs = (row_valid && DIT_INDEX_OK(p.err, ((long long)b * p.Hq + hq) * p.nqb + qrow / p.q_block,
                                                    (long long)p.B * p.Hq * p.nqb))
                             ? __ldg(p.q_scale + ((size_t)b * p.Hq + hq) * p.nqb + qrow / p.q_block)
                             : 0.0f;
        c = qs * p.c_scale;
      }
      float m_ex = -INFINITY, m_ref = -INFINITY, l = 0.0f;
      int nskip = 0;
      bool ok = true;
      volatile int (*skip_flag)[2] = bars->skip_flag;
      int n_pv = 0;  // kLazyPv: BMM2s issued so far for this tile (o_done completes once per BMM2)
      // Exponent weight per column group (log2 units): the row constant c, times the K block scale in
      // SAGE. KB >= 4 folds the block scale into the weight; KB == 1 multiplies first.
      constexpr int kGroups = (kQKScaled && KB >= 4) ? 64 / KB : 1;

      // One KV tile. kTailMode 0: the tile is full (the masking of columns past Skv is compiled out);
      // 1: the tile may be the ragged last one (decided at run time). The masking code, present in the
      // loop body, measured several percent slower on every tile, so the last tile runs its own copy.
      auto kv_tile = [&](int j, auto tail_mode) {
        constexpr int kTailMode = decltype(tail_mode)::value;
        float wg[kGroups];
        if (ok) {
          // S_i(j), and in SAGE the K-block scales of tile j (both tested at once, so the two waits'
          // latencies overlap)
          if constexpr (kQKScaled) {
            ok = mbar_wait2_bounded(&bars->s_full[i], j & 1, &bars->ks_full[j & 3], (j >> 2) & 1, budget, abort_flag);
          } else {
            ok = mbar_wait_bounded(&bars->s_full[i], j & 1, budget, abort_flag);
          }
          ok = __all_sync(0xffffffffu, ok);
          if (!ok && lane == 0) record_timeout(p, bars);
        }
        if (!ok) {
          // keep this tile's named barrier in step with the peer half
          if (SKIP && j > 0) {
            named_bar_and(tile_bar, 256, true);
          } else {
            named_bar_sync(tile_bar, 256);
          }
          return;
        }
        tc_fence_after();
        float2 s2[32];
        float* s = reinterpret_cast<float*>(s2);
        // S into registers. tcgen05.ld.red also returns each load's max over its columns: one load per
        // K block of 16 tokens in SAGE (the block's max, weighted by its scale below), one load of all
        // 64 columns without K-block scales. K blocks of 4 or 1 token use plain loads and take their
        // maxima below (sixteen 4-column loads measured slower than two plain ones and the max tree).
        constexpr bool kLdMax = !kQKScaled || KB == 16;
        constexpr int kLoads = (kQKScaled && KB == 16) ? 4 : 1;
        constexpr int kCols = 64 / kLoads;
        float gmax[kLoads];
        if constexpr (!kLdMax) {
          tmem_ld32(t_s, s);
          tmem_ld32(t_s + 32, s + 32);
        } else {
#pragma unroll
          for (int q = 0; q < kLoads; ++q) {
            if constexpr (kCols == 64) tmem_ldmax64(t_s, s, gmax[0]);
            else tmem_ldmax16(t_s + 16 * q, s + 16 * q, gmax[q]);
          }
        }
        tmem_ld_wait();
        if constexpr (L::kPInSmem) {
          // S is in registers: the issuer may compute the next tile's S into the same columns
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->s_free[i]);
        }
        const int nvalid = min(64, p.Skv - 128 * j - 64 * h);  // may be <= 0 for the upper half
        const bool tail = kTailMode != 0 && nvalid < 64;
        if (tail) {
          // the last KV tile: columns past Skv hold the products with TMA's zero fill; mask them (and
          // take the loads' maxima over the valid columns only)
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (k >= nvalid) s[k] = -INFINITY;
          if constexpr (kLdMax) {
#pragma unroll
            for (int q = 0; q < kLoads; ++q) {
              float m = -INFINITY;
#pragma unroll
              for (int k = 0; k < kCols; ++k) m = fmaxf(m, s[kCols * q + k]);
              gmax[q] = m;
            }
          }
        }
        float mh;  // this half's max of the weighted logits
        if constexpr (kQKScaled && KB == 1) {
          // per-column scales: multiply S by them first (64 values, not held across the wait for S)
          const int e = j & 3;
          const float2* ks2 = reinterpret_cast<const float2*>(s_ks + e * 128 + 64 * h);  // this half's scales
#pragma unroll
          for (int k = 0; k < 32; ++k) s2[k] = __fmul2_rn(s2[k], ks2[k]);
          wg[0] = c;
          mh = rowmax64(s) * c;
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->ks_empty[e]);
        } else if constexpr (kQKScaled) {
          const int e = j & 3;
          const float4* ks4 = reinterpret_cast<const float4*>(s_ks + e * 128 + (64 / KB) * h);  // this half's scales
#pragma unroll
          for (int q4 = 0; q4 < kGroups / 4; ++q4) {
            const float4 k4 = ks4[q4];
            wg[4 * q4 + 0] = k4.x * c;
            wg[4 * q4 + 1] = k4.y * c;
            wg[4 * q4 + 2] = k4.z * c;
            wg[4 * q4 + 3] = k4.w * c;
          }
          mh = -INFINITY;
#pragma unroll
          for (int q = 0; q < kGroups; ++q) {
            const float gm = kLdMax ? gmax[q] : groupmax<KB>(s + q * KB);
            mh = fmaxf(mh, gm * wg[q]);  // a NaN from -inf * 0 is ignored
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->ks_empty[e]);
        } else {
          wg[0] = c;
          mh = gmax[0] * c;  // -inf when this half has no valid column
        }
        // Publish this half's max; one barrier over both halves of the tile then orders the exchange
        // and, with Skip-Softmax, carries the vote. A row's full max is below the threshold exactly
        // when both halves' maxima are, so each half votes on its own max.
        xmax[((i * 2 + h) * 2 + (j & 1)) * 128 + r] = mh;
        bool skip_tile = false;
        if (SKIP && j > 0) {
          const bool vote = !row_valid || !ok || (mh - m_ex < p.log2_thr);
          skip_tile = named_bar_and(tile_bar, 256, vote);
        } else {
          named_bar_sync(tile_bar, 256);
        }
        if constexpr (L::kPInSmem) {
          // The previous BMM2 must be complete before P's buffer, O or the skip flag change.
          // kLazyPv: o_done completes once per BMM2, so the wait before the n-th P is on phase n - 1:
          // that phase is the only one outstanding (the one before was waited for, the next needs this
          // P), so its parity is unambiguous; a skipped tile writes neither P nor O and does not wait.
          // Otherwise o_done completes once per KV tile and is waited for on every tile, which keeps
          // the waits in step with its phases.
          if constexpr (kDblP) {
            // no wait here: the P buffer is free (see kDblP); O is waited for only before a rescale
          } else if constexpr (kLazyPv) {
            if (!skip_tile && n_pv > 0 && ok) {
              ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->o_done[i], (n_pv - 1) & 1, budget, abort_flag));
              if (!ok && lane == 0) record_timeout(p, bars);
            }
          } else {
            if (j > 0 && ok) {
              ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->o_done[i], (j - 1) & 1, budget, abort_flag));
              if (!ok && lane == 0) record_timeout(p, bars);
            }
          }
          if (!ok) return;
        }
        if (skip_tile) {
          // kLazyPv: the flag has a slot per KV-tile parity; the issuer reads tile j's slot before it
          // issues the BMM1 of tile j + 2, so this tile's write cannot overtake that read. Otherwise the
          // wait on the previous BMM2 (or, with TMEM P, the issuer's order) already orders them: one slot.
          ++nskip;
          if (r == 0 && h == 0) skip_flag[i][kRunAhead ? (j & 1) : 0] = 1;
          // TMEM P: the issuer's next BMM1 overwrites the S just loaded (with P in shared memory, S
          // was already released after its load)
          if constexpr (!kLazyPv) tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full_bar(i, j));
          return;
        }
        const float mo = xmax[((i * 2 + (h ^ 1)) * 2 + (j & 1)) * 128 + r];
        const float mt = fmaxf(mh, mo);  // identical on both halves: max is exact
        if (!ok) return;
        const float m_new = fmaxf(m_ex, mt);
        bool need;
        float alpha = 1.0f;
        if constexpr (kPV8) {
          need = m_new > m_ref;
          if (need) alpha = ex2_approx(m_ref - m_new);
          m_ref = m_new;
        } else {
          need = (m_new - m_ref) > kLazyRescale;
          if (need) {
            alpha = ex2_approx(m_ref - m_new);
            m_ref = m_new;
          }
        }
        m_ex = m_new;
        l *= alpha;
        // exponentials (two columns per packed FMA) and this half's row sum
        const float bias = kPV8 ? (m_ref - kLog2_448) : m_ref;
        const float2 nb = make_float2(-bias, -bias);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float w = wg[kGroups == 1 ? 0 : (2 * k) / (kGroups == 1 ? 64 : KB)];
          const float2 t = __ffma2_rn(s2[k], make_float2(w, w), nb);
          s2[k].x = ex2_approx(t.x);
          s2[k].y = ex2_approx(t.y);
        }
        if constexpr (kQKScaled) {
          // masked columns hold -inf; with a zero weight (zero scale) that gives NaN, so clear them
          if (tail) {
#pragma unroll
            for (int k = 0; k < 64; ++k)
              if (k >= nvalid) s[k] = 0.f;
          }
        }
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k & 3] = __fadd2_rn(acc[k & 3], s2[k]);
        l += ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
        if constexpr (PVF == PV_BF16) {
          // P over the first columns of this half of S
          uint32_t w[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) w[k] = pack_bf16x2(s[2 * k], s[2 * k + 1]);
          tmem_st32(t_s, w);
        } else {
          // E4M3 P into the tile's shared-memory buffer, laid out as a K-major operand with the
          // 128-byte swizzle: row r's 16-byte chunk ch sits at (r/8)*1024 + (r%8)*128 + (ch ^ r%8)*16.
          // This half holds chunks 4h .. 4h+3 (columns 64h .. 64h+63).
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w[k] = pack_e4m3x4(s[4 * k], s[4 * k + 1], s[4 * k + 2], s[4 * k + 3]);
          uint8_t* prow = smem + L::kPOff + (i * L::kPBufs + (kDblP ? (n_pv & 1) : 0)) * 16384 + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int ch = 4 * h + q;
            if (DIT_INDEX_OK(p.err, (prow - (smem + L::kPOff)) + ((ch ^ (r & 7)) << 4), L::kPBufs * 2 * 16384 - 15))
              *reinterpret_cast<uint4*>(prow + ((ch ^ (r & 7)) << 4)) =
                  make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
          fence_proxy_async_smem();  // visible to the tensor cores' reads
        }
        // O rescale for this half (after P, when the scores are no longer held in registers; still
        // before the arrive that lets the MMA accumulate into O)
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          if constexpr (kDblP) {
            // O must not change while the previous BMM2 still accumulates into it
            if (n_pv > 0) {
              ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->o_done[i], (n_pv - 1) & 1, budget, abort_flag));
              if (!ok && lane == 0) record_timeout(p, bars);
            }
          }
          const float2 a2 = make_float2(alpha, alpha);
          if constexpr (kQKScaled && KB >= 16) {
            // frequent (every new running max): all 64 columns with one wait. Measured faster with
            // K blocks of 16; with finer blocks the two-round form below is faster.
            float2 o[32];
            tmem_ld32(t_o, reinterpret_cast<float*>(o));
            tmem_ld32(t_o + 32, reinterpret_cast<float*>(o + 16));
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __fmul2_rn(o[k], a2);
            tmem_st32(t_o, reinterpret_cast<const uint32_t*>(o));
            tmem_st32(t_o + 32, reinterpret_cast<const uint32_t*>(o + 16));
          } else {
            // two rounds of 32 columns keep register pressure low
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
              float2 o[16];
              tmem_ld32(t_o + 32 * cc, reinterpret_cast<float*>(o));
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 16; ++k) o[k] = __fmul2_rn(o[k], a2);
              tmem_st32(t_o + 32 * cc, reinterpret_cast<const uint32_t*>(o));
            }
          }
          if constexpr (kDblP) tmem_st_wait();  // the rescaled O is in tensor memory
        }
        if constexpr (!kDblP) tmem_st_wait();
        if constexpr (SKIP) {
          if (r == 0 && h == 0) skip_flag[i][kRunAhead ? (j & 1) : 0] = 0;
        }
        ++n_pv;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full_bar(i, j));
      };
      // dense and SAGE INT8: every tile keeps the run-time tail test (a peeled last tile measured no
      // faster for SAGE INT8)
      for (int j = 0; j < nt; ++j) kv_tile(j, std::integral_constant<int, 1>{});

      // ------------------------------------------------------------ epilogue: O / l -> bf16 -> TMA store
      xl[(i * 2 + h) * 128 + r] = l;
      named_bar_sync(tile_bar, 256);
      const float l_row = xl[(i * 2 + 0) * 128 + r] + xl[(i * 2 + 1) * 128 + r];
      if (p.lse != nullptr && h == 0 && row_valid && ok) {
        // ln sum_j exp(s_j) = ln 2 * (m_ref + log2 l), with l relative to m_ref (and carrying P's 448
        // with E4M3 P); only the kept KV tiles contribute under Skip-Softmax, as to the output
        const float l_true = kPV8 ? l_row * (1.0f / 448.0f) : l_row;
        if (DIT_INDEX_OK(p.err, ((long long)b * p.Hq + hq) * p.Sq + qrow, (long long)p.B * p.Hq * p.Sq))
          p.lse[((size_t)b * p.Hq + hq) * p.Sq + qrow] = 0.69314718055994531f * (m_ref + log2f(l_true));
      }
      if (ok) {
        ok = mbar_wait_bounded(&bars->o_full[i], 0, budget, abort_flag);
        if constexpr (kPV8) ok = ok && mbar_wait_bounded(&bars->vs_full, 0, budget, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0) record_timeout(p, bars);
      }
      // Stage O in this tile's own Q buffer (32 KB reserved per tile): only this tile's issuer reads
      // it, and all of that issuer's MMAs are complete once O is final. (The K/V ring may still be
      // read by the other tile's issuer.)
      uint8_t* stage = smem + L::kQOff + i * 32768 + h * 16384;
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.0f / l_row;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          float o[32];
          tmem_ld32(t_o + 32 * cc, o);
          tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float a0 = o[2 * k] * inv_l, a1 = o[2 * k + 1] * inv_l;
            if constexpr (kPV8) {
              a0 *= s_vs[64 * h + 32 * cc + 2 * k];
              a1 *= s_vs[64 * h + 32 * cc + 2 * k + 1];
            }
            w[k] = pack_bf16x2(a0, a1);
          }
          // 128-byte swizzled staging of this half (columns 64h..64h+63): 16-byte chunk ch of row r
          // sits at r*128 + ((ch ^ (r & 7)) * 16).
          uint8_t* rowp = stage + r * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int ch = cc * 4 + q;
            if (DIT_INDEX_OK(p.err, (rowp - (smem + L::kQOff + i * 32768)) + ((ch ^ (r & 7)) << 4), 32768 - 15))
              *reinterpret_cast<uint4*>(rowp + ((ch ^ (r & 7)) << 4)) =
                  make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
        fence_proxy_async_smem();
      }
      const bool all_ok = named_bar_and(group_bar, 128, ok);
      if (all_ok && r == 0) {
        tma_store_4d(&tm_o, stage, 64 * h, q0 + 128 * i, hq, b);
        tma_store_commit();
        tma_store_wait_all0();
      }
      if (r == 0 && h == 0 && p.skip_counts != nullptr) {
        const int qt = 2 * blockIdx.x + i;
        if (qt < p.n_q_tiles && DIT_INDEX_OK(p.err, ((long long)b * p.Hq + hq) * p.n_q_tiles + qt,
                                             (long long)p.B * p.Hq * p.n_q_tiles))
          p.skip_counts[((size_t)b * p.Hq + hq) * p.n_q_tiles + qt] = nskip;
      }
    } else {
      // ------------------------------------------------------------ softmax warpgroups
      regs_inc<P::kRegsSoftmax>();
      constexpr int NH = P::kNH;                     // softmax warpgroups per Q tile
      constexpr int NC = 128 / NH;                   // columns of S per thread
      const int g = (warp - 4) >> 2;                 // softmax warpgroup
      const int i = g / NH;                          // Q tile within the CTA
      const int h = g % NH;                          // column part: S/O columns NC*h .. NC*h + NC-1
      const int r = ((warp & 3) << 5) + lane;        // row within the tile == TMEM lane
      const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
      const uint32_t t_s = tbase + lane_base + kColS1 * i + NC * h;
      const uint32_t t_o = tbase + lane_base + kColO0 + 128 * i + NC * h;
      const int qrow = q0 + 128 * i + r;
      const bool row_valid = qrow < p.Sq;
      const uint32_t tile_bar = 1 + i;               // the 128 * NH threads of this Q tile
      const uint32_t group_bar = 3 + g;              // the 128 threads of this warpgroup
      const uint32_t s_base = smem_u32(smem);
      float* xmax = reinterpret_cast<float*>(smem + L::kXmaxOff);  // [tile][part][parity][128] partial maxima
      float* xl = reinterpret_cast<float*>(smem + L::kXlOff);      // [tile][part][128] partial row sums
      float c = p.c_scale;
      if constexpr (kNV) c = c / (__ldg(p.q_gs) * __ldg(p.k_gs));  // BMM1 carries both tensor scales
      if constexpr (kQKScaled) {
        const float qs = (row_valid && DIT_INDEX_OK(p.err, ((long long)b * p.Hq + hq) * p.nqb + qrow / p.q_block,
                                                    (long long)p.B * p.Hq * p.nqb))
                             ? __ldg(p.q_scale + ((size_t)b * p.Hq + hq) * p.nqb + qrow / p.q_block)
                             : 0.0f;
        c = qs * p.c_scale;
      }
      float m_ex = -INFINITY, m_ref = -INFINITY, l = 0.0f;
      int nskip = 0;
      bool ok = true;
      volatile int (*skip_flag)[2] = bars->skip_flag;
      int n_pv = 0;  // kLazyPv: BMM2s issued so far for this tile (o_done completes once per BMM2)
      // Exponent weight per group of columns that share a K-block scale (log2 units): the row constant
      // c, times the block scale in SAGE. KB >= 4 folds the block scale into the weight; KB == 1
      // multiplies S by the column scales first.
      constexpr int kGroups = (kQKScaled && KB >= 4) ? NC / KB : 1;
      // S into registers. tcgen05.ld.red also returns each load's max over its columns: one load per
      // K block of 16 tokens in SAGE (the block's max, weighted by its scale below), loads of 64
      // columns without K-block scales. K blocks of 4 or 1 token use plain loads and take their maxima
      // below (4-column loads measured slower than plain ones and the max tree).
      constexpr bool kLdMax = !kQKScaled || KB == 16;
      constexpr int kLoads = (kQKScaled && KB == 16) ? NC / 16 : NC / 64;
      constexpr int kCols = NC / kLoads;
      // E4M3 P: this row's 128 bytes in the tile's P buffer (a K-major operand with the 128-byte
      // swizzle): 16-byte chunk ch (columns 16ch .. 16ch+15) of row r sits at
      // (r/8)*1024 + (r%8)*128 + (ch ^ r%8)*16.
      uint8_t* const p_row0 = smem + L::kPOff + i * L::kPBufs * 16384 + (r >> 3) * 1024 + (r & 7) * 128;
      const uint32_t sw = (uint32_t)(r & 7);

      // One KV tile. kTailMode 0: the tile is full (the masking of columns past Skv is compiled out);
      // 1: the tile may be the ragged last one (decided at run time). The masking code, present in the
      // loop body, measured several percent slower on every tile, so the last tile runs its own copy.
      auto kv_tile = [&](int j, auto tail_mode) {
        constexpr int kTailMode = decltype(tail_mode)::value;
        if (ok) {
          // S_i(j), and in SAGE the K-block scales of tile j (both tested at once, so the two waits'
          // latencies overlap)
          if constexpr (kQKScaled) {
            ok = mbar_wait2_bounded(&bars->s_full[i], j & 1, &bars->ks_full[j & 3], (j >> 2) & 1, budget, abort_flag);
          } else {
            ok = mbar_wait_bounded(&bars->s_full[i], j & 1, budget, abort_flag);
          }
          ok = __all_sync(0xffffffffu, ok);
          if (!ok && lane == 0) record_timeout(p, bars);
        }
        if (!ok) {
          // keep this tile's named barrier in step with the other warps
          if (SKIP && j > 0) {
            named_bar_and(tile_bar, 128 * NH, true);
          } else if (NH == 2) {
            named_bar_sync(tile_bar, 128 * NH);
          }
          return;
        }
        tc_fence_after();
        float2 s2[NC / 2];
        float* s = reinterpret_cast<float*>(s2);
        float gmax[kLoads];
        if constexpr (!kLdMax) {
#pragma unroll
          for (int q = 0; q < NC / 32; ++q) tmem_ld32(t_s + 32 * q, s + 32 * q);
        } else if constexpr (kCols == 16) {
#pragma unroll
          for (int q = 0; q < kLoads; ++q) tmem_ldmax16(t_s + 16 * q, s + 16 * q, gmax[q]);
        } else {
#pragma unroll
          for (int q = 0; q < kLoads; ++q) tmem_ldmax64(t_s + 64 * q, s + 64 * q, gmax[q]);
        }
        tmem_ld_wait();
        if constexpr (L::kPInSmem) {
          // S is in registers: the issuer may compute the next tile's S into the same columns
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->s_free[i]);
        }
        const int nvalid = min(NC, p.Skv - 128 * j - NC * h);  // may be <= 0 for the upper part
        const bool tail = kTailMode != 0 && nvalid < NC;
        if (tail) {
          // the last KV tile: columns past Skv hold the products with TMA's zero fill; mask them (and
          // take the loads' maxima over the valid columns only)
#pragma unroll
          for (int k = 0; k < NC; ++k)
            if (k >= nvalid) s[k] = -INFINITY;
          if constexpr (kLdMax) {
#pragma unroll
            for (int q = 0; q < kLoads; ++q) {
              float m = -INFINITY;
#pragma unroll
              for (int k = 0; k < kCols; ++k) m = fmaxf(m, s[kCols * q + k]);
              gmax[q] = m;
            }
          }
        }
        float wg[kGroups];
        float mh;  // this part's max of the row's weighted logits
        if constexpr (kQKScaled && KB == 1) {
          // per-column scales: multiply S by them first
          const int e = j & 3;
          const uint32_t ks = s_base + L::kKsOff + e * 512 + NC * h * 4;  // this part's scales
#pragma unroll
          for (int q = 0; q < NC / 4; ++q) {
            const float4 k4 = lds128f(ks + 16 * q);
            s2[2 * q] = __fmul2_rn(s2[2 * q], make_float2(k4.x, k4.y));
            s2[2 * q + 1] = __fmul2_rn(s2[2 * q + 1], make_float2(k4.z, k4.w));
          }
          wg[0] = c;
          mh = (NC == 128 ? rowmax128(s) : rowmax64(s)) * c;
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->ks_empty[e]);
        } else if constexpr (kQKScaled) {
          const int e = j & 3;
          const uint32_t ks = s_base + L::kKsOff + e * 512 + kGroups * h * 4;  // this part's scales
#pragma unroll
          for (int q4 = 0; q4 < kGroups / 4; ++q4) {
            const float4 k4 = lds128f(ks + 16 * q4);
            wg[4 * q4 + 0] = k4.x * c;
            wg[4 * q4 + 1] = k4.y * c;
            wg[4 * q4 + 2] = k4.z * c;
            wg[4 * q4 + 3] = k4.w * c;
          }
          mh = -INFINITY;
#pragma unroll
          for (int q = 0; q < kGroups; ++q) {
            const float gm = kLdMax ? gmax[q] : groupmax<KB>(s + q * KB);
            mh = fmaxf(mh, gm * wg[q]);  // a NaN from -inf * 0 is ignored
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->ks_empty[e]);
        } else {
          wg[0] = c;
          mh = gmax[0];
#pragma unroll
          for (int q = 1; q < kLoads; ++q) mh = fmaxf(mh, gmax[q]);
          mh *= c;  // -inf when this part has no valid column
        }
        // With two parts, each publishes its max and one barrier over the tile orders the exchange.
        // Skip-Softmax: the tile is skipped when every row's max is below the threshold (padded rows do
        // not vote; a row's max is below it exactly when every part's is, so each part votes on its
        // own); the barrier over the tile carries the vote.
        if constexpr (NH == 2) xmax[((i * 2 + h) * 2 + (j & 1)) * 128 + r] = mh;
        bool skip_tile = false;
        if (SKIP && j > 0) {
          const bool vote = !row_valid || (mh - m_ex < p.log2_thr);
          skip_tile = named_bar_and(tile_bar, 128 * NH, vote);
        } else if constexpr (NH == 2) {
          named_bar_sync(tile_bar, 128 * NH);
        }
        if constexpr (L::kPInSmem) {
          // The previous BMM2 must be complete before P's buffer, O or the skip flag change.
          // kLazyPv: o_done completes once per BMM2, so the wait before the n-th P is on phase n - 1:
          // that phase is the only one outstanding (the one before was waited for, the next needs this
          // P), so its parity is unambiguous; a skipped tile writes neither P nor O and does not wait.
          // Otherwise o_done completes once per KV tile and is waited for on every tile, which keeps
          // the waits in step with its phases.
          if constexpr (kDblP) {
            // no wait here: the P buffer is free (see kDblP); O is waited for only before a rescale
          } else if constexpr (kLazyPv) {
            if (!skip_tile && n_pv > 0) {
              ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->o_done[i], (n_pv - 1) & 1, budget, abort_flag));
              if (!ok && lane == 0) record_timeout(p, bars);
            }
          } else {
            if (j > 0) {
              ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->o_done[i], (j - 1) & 1, budget, abort_flag));
              if (!ok && lane == 0) record_timeout(p, bars);
            }
          }
          if (!ok) return;
        }
        if (skip_tile) {
          // kLazyPv: the flag has a slot per KV-tile parity; the issuer reads tile j's slot before it
          // issues the BMM1 of tile j + 2, so this tile's write cannot overtake that read. Otherwise the
          // wait on the previous BMM2 (or, with TMEM P, the issuer's order) already orders them: one slot.
          ++nskip;
          if (r == 0 && h == 0) skip_flag[i][kRunAhead ? (j & 1) : 0] = 1;
          // TMEM P: the issuer's next BMM1 overwrites the S just loaded (with P in shared memory, S
          // was already released after its load)
          if constexpr (!kLazyPv) tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full_bar(i, j));
          return;
        }
        float mt = mh;
        if constexpr (NH == 2)  // identical on both parts: max is exact
          mt = fmaxf(mh, xmax[((i * 2 + (h ^ 1)) * 2 + (j & 1)) * 128 + r]);
        const float m_new = fmaxf(m_ex, mt);
        bool need;
        float alpha = 1.0f;
        if constexpr (kPV8) {
          need = m_new > m_ref;
          if (need) alpha = ex2_approx(m_ref - m_new);
          m_ref = m_new;
        } else {
          need = (m_new - m_ref) > kLazyRescale;
          if (need) {
            alpha = ex2_approx(m_ref - m_new);
            m_ref = m_new;
          }
        }
        m_ex = m_new;
        l *= alpha;
        // exponentials (two columns per packed FMA) and this part's row sum
        const float bias = kPV8 ? (m_ref - kLog2_448) : m_ref;
        const float2 nb = make_float2(-bias, -bias);
#pragma unroll
        for (int k = 0; k < NC / 2; ++k) {
          const float w = wg[kGroups == 1 ? 0 : (2 * k) / (kGroups == 1 ? NC : KB)];
          const float2 t = __ffma2_rn(s2[k], make_float2(w, w), nb);
          s2[k].x = ex2_approx(t.x);
          s2[k].y = ex2_approx(t.y);
        }
        if constexpr (kQKScaled) {
          // masked columns hold -inf; with a zero weight (zero scale) that gives NaN, so clear them
          if (tail) {
#pragma unroll
            for (int k = 0; k < NC; ++k)
              if (k >= nvalid) s[k] = 0.f;
          }
        }
        constexpr int kAcc = NC == 128 ? 8 : 4;  // independent packed partial sums
        float2 acc[kAcc];
#pragma unroll
        for (int k = 0; k < kAcc; ++k) acc[k] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NC / 2; ++k) acc[k % kAcc] = __fadd2_rn(acc[k % kAcc], s2[k]);
#pragma unroll
        for (int k = 0; k < kAcc - 4; ++k) acc[k] = __fadd2_rn(acc[k], acc[k + 4]);
        l += ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
        if constexpr (PVF == PV_BF16) {
          // P (two bf16 values per column) over the first NC / 2 columns of this part of S
          uint32_t w[NC / 2];
#pragma unroll
          for (int k = 0; k < NC / 2; ++k) w[k] = pack_bf16x2(s[2 * k], s[2 * k + 1]);
#pragma unroll
          for (int q = 0; q < NC / 64; ++q) tmem_st32(t_s + 32 * q, w + 32 * q);
        } else {
          // E4M3 P into the tile's shared-memory buffer: this part's chunks (NC / 16 of 16 columns)
#pragma unroll
          for (int cq = 0; cq < NC / 16; ++cq) {
            const uint32_t ch = (uint32_t)((NC / 16) * h + cq);
            const float* x = s + 16 * cq;
            if (DIT_INDEX_OK(p.err, (p_row0 - (smem + L::kPOff)) + (kDblP ? (n_pv & 1) * 16384 : 0) + ((ch ^ sw) << 4),
                             L::kPBufs * 2 * 16384 - 15))
              *reinterpret_cast<uint4*>(p_row0 + (kDblP ? (n_pv & 1) * 16384 : 0) + ((ch ^ sw) << 4)) =
                  make_uint4(pack_e4m3x4(x[0], x[1], x[2], x[3]), pack_e4m3x4(x[4], x[5], x[6], x[7]),
                             pack_e4m3x4(x[8], x[9], x[10], x[11]), pack_e4m3x4(x[12], x[13], x[14], x[15]));
          }
          fence_proxy_async_smem();  // visible to the tensor cores' reads
        }
        // O rescale for this part (after P, when the scores are no longer held in registers; still
        // before the arrive that lets the MMA accumulate into O)
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          if constexpr (kDblP) {
            // O must not change while the previous BMM2 still accumulates into it
            if (n_pv > 0) {
              ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->o_done[i], (n_pv - 1) & 1, budget, abort_flag));
              if (!ok && lane == 0) record_timeout(p, bars);
            }
          }
          const float2 a2 = make_float2(alpha, alpha);
          if constexpr (NC == 128 && kBS) {
            // MXFP8 / NVFP4: the whole row in one round, S's registers being free by now (measured
            // faster for them; slower for QK16PV8 and SAGE FP8, and SAGE FP8 with K blocks of 16 spills)
            float2 o[64];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld32(t_o + 32 * q, reinterpret_cast<float*>(o + 16 * q));
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 64; ++k) o[k] = __fmul2_rn(o[k], a2);
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_st32(t_o + 32 * q, reinterpret_cast<const uint32_t*>(o + 16 * q));
          } else if constexpr (NC == 128 || (kQKScaled && KB >= 16)) {
            // rounds of 64 columns with one wait each (measured faster with K blocks of 16; with finer
            // blocks and 64 columns per thread the rounds of 32 below are faster)
#pragma unroll 1
            for (int cc = 0; cc < NC / 64; ++cc) {
              float2 o[32];
              tmem_ld32(t_o + 64 * cc, reinterpret_cast<float*>(o));
              tmem_ld32(t_o + 64 * cc + 32, reinterpret_cast<float*>(o + 16));
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __fmul2_rn(o[k], a2);
              tmem_st32(t_o + 64 * cc, reinterpret_cast<const uint32_t*>(o));
              tmem_st32(t_o + 64 * cc + 32, reinterpret_cast<const uint32_t*>(o + 16));
            }
          } else {
#pragma unroll 1
            for (int cc = 0; cc < NC / 32; ++cc) {
              float2 o[16];
              tmem_ld32(t_o + 32 * cc, reinterpret_cast<float*>(o));
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 16; ++k) o[k] = __fmul2_rn(o[k], a2);
              tmem_st32(t_o + 32 * cc, reinterpret_cast<const uint32_t*>(o));
            }
          }
          if constexpr (kDblP) tmem_st_wait();  // the rescaled O is in tensor memory
        }
        if constexpr (!kDblP) tmem_st_wait();
        if constexpr (SKIP) {
          if (r == 0 && h == 0) skip_flag[i][kRunAhead ? (j & 1) : 0] = 0;
        }
        ++n_pv;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full_bar(i, j));
      };
      if constexpr (QKF == QK_E4M3) {  // measured faster peeled for SAGE FP8; QK16PV8 and MXFP8 spilled or slowed
        for (int j = 0; j + 1 < nt; ++j) kv_tile(j, std::integral_constant<int, 0>{});
        if (nt > 0) kv_tile(nt - 1, std::integral_constant<int, 1>{});
      } else {
        for (int j = 0; j < nt; ++j) kv_tile(j, std::integral_constant<int, 1>{});
      }

      // ------------------------------------------------------------ epilogue: O / l -> bf16 -> TMA store
      float l_row = l;
      if constexpr (NH == 2) {
        xl[(i * 2 + h) * 128 + r] = l;
        named_bar_sync(tile_bar, 128 * NH);
        l_row = xl[(i * 2) * 128 + r] + xl[(i * 2 + 1) * 128 + r];
      }
      if (p.lse != nullptr && h == 0 && row_valid && ok) {
        // ln sum_j exp(s_j) = ln 2 * (m_ref + log2 l), with l relative to m_ref (and carrying P's 448
        // with E4M3 P); only the kept KV tiles contribute under Skip-Softmax, as to the output
        const float l_true = kPV8 ? l_row * (1.0f / 448.0f) : l_row;
        if (DIT_INDEX_OK(p.err, ((long long)b * p.Hq + hq) * p.Sq + qrow, (long long)p.B * p.Hq * p.Sq))
          p.lse[((size_t)b * p.Hq + hq) * p.Sq + qrow] = 0.69314718055994531f * (m_ref + log2f(l_true));
      }
      if (ok) {
        ok = mbar_wait_bounded(&bars->o_full[i], 0, budget, abort_flag);
        if constexpr (kPV8) ok = ok && mbar_wait_bounded(&bars->vs_full, 0, budget, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0) record_timeout(p, bars);
      }
      // Stage O in this tile's own Q buffer (32 KB reserved per tile: two 128-byte-swizzled halves of 64
      // columns, 16-byte chunk ch of row r at r*128 + (ch ^ r%8)*16): only this tile's issuer reads it,
      // and all of that issuer's MMAs are complete once O is final. (The K/V ring may still be read by
      // the other tile's issuer.)
      const uint32_t stage = s_base + L::kQOff + i * 32768;
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.0f / l_row;
#pragma unroll 1
        for (int cc = 0; cc < NC / 32; ++cc) {
          float o[32];
          tmem_ld32(t_o + 32 * cc, o);
          tmem_ld_wait();
          const int gc = NC * h + 32 * cc;  // the first of these 32 columns within the row
          uint32_t w[16];
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            float a[4] = {o[4 * k4] * inv_l, o[4 * k4 + 1] * inv_l, o[4 * k4 + 2] * inv_l, o[4 * k4 + 3] * inv_l};
            if constexpr (kPV8) {
              const float4 vs = lds128f(s_base + L::kVsOff + (gc + 4 * k4) * 4);
              a[0] *= vs.x;
              a[1] *= vs.y;
              a[2] *= vs.z;
              a[3] *= vs.w;
            }
            w[2 * k4] = pack_bf16x2(a[0], a[1]);
            w[2 * k4 + 1] = pack_bf16x2(a[2], a[3]);
          }
          const uint32_t rowp = stage + (gc >> 6) * 16384 + r * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t ch = (uint32_t)(((gc & 63) >> 3) + q);
            if (DIT_INDEX_OK(p.err, (long long)(rowp - stage) + ((ch ^ sw) << 4), 32768 - 15))
              sts128(rowp + ((ch ^ sw) << 4), w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
        fence_proxy_async_smem();
      }
      const bool all_ok = named_bar_and(group_bar, 128, ok);
      if (all_ok && r == 0) {
        // this warpgroup's halves of 64 columns
#pragma unroll
        for (int hh = 0; hh < 2 / NH; ++hh) {
          const int half = (2 / NH) * h + hh;
          tma_store_4d(&tm_o, smem + L::kQOff + i * 32768 + half * 16384, 64 * half, q0 + 128 * i, hq, b);
        }
        tma_store_commit();
        tma_store_wait_all0();
      }
      if (r == 0 && h == 0 && p.skip_counts != nullptr) {
        const int qt = 2 * blockIdx.x + i;
        if (qt < p.n_q_tiles && DIT_INDEX_OK(p.err, ((long long)b * p.Hq + hq) * p.n_q_tiles + qt,
                                             (long long)p.B * p.Hq * p.n_q_tiles))
          p.skip_counts[((size_t)b * p.Hq + hq) * p.n_q_tiles + qt] = nskip;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int QKF, int PVF, int KB, bool SKIP, bool WITHHOLD = false>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                       const FmhaParams& p, cudaStream_t stream) {
  // set once per device and instantiation; host threads may launch concurrently
  static std::atomic<bool> attr_set[64];
  static std::mutex attr_mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(attr_mu);
    // The register hand-over in the kernel (setmaxnreg) assumes exactly kLaunchRegs per thread at
    // launch; with fewer, the softmax warpgroups' increase could never be granted.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fmha_fwd_kernel<QKF, PVF, KB, SKIP, WITHHOLD>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != Parts<QKF, PVF, SKIP>::kLaunchRegs) return cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(fmha_fwd_kernel<QKF, PVF, KB, SKIP, WITHHOLD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SmemLayout<QKF, PVF>::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const dim3 grid((p.Sq + 255) / 256, p.Hq, p.B);
  fmha_fwd_kernel<QKF, PVF, KB, SKIP, WITHHOLD><<<grid, Parts<QKF, PVF, SKIP>::kThreads, SmemLayout<QKF, PVF>::kSmemBytes, stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace ditattn
