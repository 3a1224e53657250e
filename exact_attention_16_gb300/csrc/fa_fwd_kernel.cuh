// FlashAttention forward for sm_103a: TMA + mbarrier pipeline, tcgen05 MMAs
// accumulating in tensor memory, warp-specialised online softmax, causal tile
// skipping and a persistent longest-first scheduler.
//
// What it computes (exact attention, tile by tile with online softmax):
//   "MiniPaged-Qwen: Qwen3 Prefill FlashAttention", sections 3.1 and 4 (tile
//   recurrence m, l, alpha, O~, then O = O~ / l), section 6 (GQA head map),
//   section 13 (bottom-right causal limit); "NVIDIA闪存注意力实操" sections
//   "在线Softmax算法" (exp2 with log2(e) folded into the scale), "K循环拆分"
//   (only diagonal tiles are masked, tiles above it are skipped) and
//   "ProgramId重映射" (longest work first).
//
// One CTA per SM loops over work items. A work item is two 128-row query
// tiles that read the same keys and values: two heads of one GQA group at the
// same rows when the group size is even, else two consecutive row tiles of one
// head. Warp roles (320 threads):
//   warps 0-3  softmax + epilogue for query tile 0 (TMEM lanes 0..127)
//   warps 4-7  softmax + epilogue for query tile 1
//   warp  8    TMA producer (Q tiles, then K_j / V_j tiles into a ring)
//   warp  9    MMA issuer (one thread) and TMEM owner
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// The softmax writes P (16-bit, two per column) over the first 64 columns of
// its S region; the PV MMA reads P from TMEM and V from shared memory.
//
// Key-split items (KSPLIT) serve problems with too few row tiles to fill the
// SMs, the short-sequence case of "NVIDIA闪存注意力实操" section "自动调优"
// (large tiles leave SMs idle). A work item is then ONE 128-row query tile,
// and its two slots run the even and the odd key tiles against the same Q.
// Each slot keeps its own online-softmax state (m, l, O~); at the end the
// tile-0 warps combine the two with the rescale of "MiniPaged-Qwen: Qwen3
// Prefill FlashAttention" section 4: m = max(m0, m1), a_t = 2^(m_t - m),
// O = (a0 O~0 + a1 O~1) / (a0 l0 + a1 l1). Twice as many items, each half as
// long, and no workspace.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx_sm103.cuh"
#include "softmax_row.cuh"

namespace fa {

constexpr int kBM = 128;          // query rows per tile (MMA M)
constexpr int kBN = 128;          // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kThreads = 320;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256

enum : int { kStatusOk = 0, kStatusTimeout = 4 };

struct FwdParams {
  void* o;               // (B, Sq, Hq, D) 16-bit, element strides below, d contiguous
  long long o_sb, o_ss, o_sh;
  int d_true;            // head dimension of the tensors (<= D, a multiple of 16; the tile is zero padded)
  float* lse;            // (B, Hq, Sq) fp32 natural log, contiguous, may be null
  int B, Sq, Sk, Hq, Hkv, group;
  int causal;
  float scale_log2;      // softmax scale * log2(e); nonzero (see q_b_shift)
  int q_b_shift;         // added to the batch coordinate of every Q load: B reads
                         // Q as zeros (out of range, TMA zero fill), which is how
                         // a zero scale runs: 0 * q.k = 1 * (0 . k)
  int n_mtiles;          // ceil(Sq / 128)
  int pair_heads;        // 1: item = heads (2u, 2u+1) at one row tile
  int n_units;           // head units per batch entry
  int n_mslots;          // row-tile slots per unit
  int n_items;
  int n_kv_tiles;        // ceil(Sk / 128)
  unsigned long long timeout_ns;
  int inject_skip_load;  // test hook: index of a K/V load to drop (-1: none)
  int* status;           // device status word (first error wins)
};

template <int D>
struct Smem {
  static constexpr int kChunks = D / 64;                  // 128-byte swizzle columns
  static constexpr int kChunkBytes = 128 * 128;           // 128 rows x 128 bytes
  static constexpr int kTileBytes = kChunks * kChunkBytes;  // one Q/K/V tile
  static constexpr int kStages = (D == 128) ? 4 : 6;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kTileBytes;
  // O staging for the TMA store: one 64-column chunk (32 rows x 128 bytes per
  // warp, 4 KB) per softmax warp, 8 warps.
  static constexpr int kOStageOff = kKVOff + kStages * kTileBytes;
  static constexpr int kOStageWarpBytes = 32 * 128;
  static constexpr int kBarOff = kOStageOff + 8 * kOStageWarpBytes;
  // barriers: q_full[2] q_empty[2] kv_full[S/2] kv_empty[S/2] s_full[2]
  //           p_full[2] p_half[2] o_full[2] o_empty[2] teardown stats_full
  //           stats_empty (at most this many)
  static constexpr int kNumBars = 2 + 2 + kStages + kStages + 2 + 2 + 2 + 2 + 2 + 1 + 2;
  // Key-split items: slot 1 hands its per-row (m, l, l_corr) to the tile-0
  // warps in the O staging buffer of warp 4, which only slot 0 stores from
  // otherwise (3 x 128 floats).
  static constexpr int kStatsOff = kOStageOff + 4 * kOStageWarpBytes;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;            // slack for 1024-byte alignment
};

struct WorkItem {
  int b, hq0, hq1, kvh, r0, r1;  // rows r_t .. r_t+127 of head hq_t
  int n_kv;                       // key tiles [0, n_kv) to visit
};

// Number of 128-key tiles query rows [r0, r0+128) need (0 if none visible).
// Host code calls it too, to cost the schedule before the launch.
__host__ __device__ __forceinline__ int kv_tiles_for(const FwdParams& p, int r0) {
  if (r0 >= p.Sq) return 0;
  if (!p.causal) return p.n_kv_tiles;
  int r_last = (r0 + kBM - 1 < p.Sq - 1) ? r0 + kBM - 1 : p.Sq - 1;
  long long lim = static_cast<long long>(r_last) + (p.Sk - p.Sq) + 1;  // exclusive key bound
  if (lim <= 0) return 0;
  if (lim > p.Sk) lim = p.Sk;
  return static_cast<int>((lim + kBN - 1) / kBN);
}

// Work items are numbered longest first: row-tile slot descending (causal
// cost grows with the row index), then batch, then head unit, so the heads of
// one GQA group run side by side and share K/V through L2. Key-split items
// are single row tiles (head unit = head, slot = row tile).
template <bool KSPLIT>
__host__ __device__ __forceinline__ WorkItem decode_item(const FwdParams& p, int idx) {
  WorkItem w;
  int per_slot = p.B * p.n_units;
  int slot = p.n_mslots - 1 - idx / per_slot;
  int rem = idx % per_slot;
  w.b = rem / p.n_units;
  int unit = rem % p.n_units;
  if (KSPLIT) {
    w.hq0 = unit;
    w.hq1 = unit;
    w.r0 = slot * kBM;
    w.r1 = slot * kBM;
  } else if (p.pair_heads) {
    w.hq0 = 2 * unit;
    w.hq1 = 2 * unit + 1;
    w.r0 = slot * kBM;
    w.r1 = slot * kBM;
  } else {
    w.hq0 = unit;
    w.hq1 = unit;
    w.r0 = 2 * slot * kBM;
    w.r1 = (2 * slot + 1) * kBM;
  }
  w.kvh = w.hq0 / p.group;
  const int n0 = kv_tiles_for(p, w.r0), n1 = kv_tiles_for(p, w.r1);
  w.n_kv = n0 > n1 ? n0 : n1;
  return w;
}

// Serpentine static schedule over the longest-first order: CTA c takes item
// r*G + c on even rounds and r*G + (G-1-c) on odd rounds.
__host__ __device__ __forceinline__ int item_of_round(int round, int cta, int grid) {
  return round * grid + ((round & 1) ? (grid - 1 - cta) : cta);
}

// The first round >= r in which CTA `cta` has an item with at least one key
// tile, or -1 when it has none left.
template <bool KSPLIT>
__host__ __device__ __forceinline__ int next_round(const FwdParams& p, int r, int cta, int grid) {
  for (;; ++r) {
    if (static_cast<long long>(r) * grid >= p.n_items) return -1;
    const int idx = item_of_round(r, cta, grid);
    if (idx < p.n_items && decode_item<KSPLIT>(p, idx).n_kv > 0) return r;
  }
}

// Bounded wait on an mbarrier phase. Returns false when the CTA aborted or the
// wait ran past the time limit (which records kStatusTimeout and aborts).
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         const FwdParams& p) {
  if (ptx::mbar_test_wait(bar, parity)) return true;
  uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
        atomicCAS(p.status, kStatusOk, kStatusTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) return ptx::pack_bf16x2(lo, hi);
  else return ptx::pack_f16x2(lo, hi);
}

template <int D, bool BF16, bool KSPLIT>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
              const __grid_constant__ FwdParams p) {
  using L = Smem<D>;
  constexpr int kSlots = L::kStages / 2;   // K/V ring slots of two tiles each
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  // Row-tile pairs at D = 64: the softmax signals the first half of P (keys
  // 0..63) on its own, and the MMA thread starts P V on it while the second
  // half is computed (the P V MMAs are short there; at D = 128 the extra
  // hand-off cost more than the overlap gained).
  constexpr bool kHalfP = !KSPLIT && D == 64;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);

  const uint32_t sQ = base + L::kQOff;
  const uint32_t sKV = base + L::kKVOff;
  const uint32_t bars = base + L::kBarOff;
  const uint32_t bar_q_full = bars;                       // [2]
  const uint32_t bar_q_empty = bars + 2 * 8;              // [2]
  const uint32_t bar_kv_full = bars + 4 * 8;              // [kSlots]
  const uint32_t bar_kv_empty = bar_kv_full + kSlots * 8;  // [kSlots]
  const uint32_t bar_s_full = bar_kv_empty + kSlots * 8;   // [2]
  const uint32_t bar_p_full = bar_s_full + 2 * 8;          // [2] P (all 64 columns) written
  const uint32_t bar_p_half = bar_p_full + 2 * 8;          // [2] row-tile pairs: P columns 0..31 written
  const uint32_t bar_o_full = bar_p_full + 4 * 8;          // [2]
  const uint32_t bar_o_empty = bar_o_full + 2 * 8;         // [2]
  const uint32_t bar_teardown = bar_o_empty + 2 * 8;
  const uint32_t bar_stats_full = bar_teardown + 8;       // key-split: slot 1 state written
  const uint32_t bar_stats_empty = bar_teardown + 16;     // key-split: slot 1 state consumed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar_q_full + 8 * t, 1);
      ptx::mbar_init(bar_q_empty + 8 * t, 1);
      ptx::mbar_init(bar_s_full + 8 * t, 1);
      ptx::mbar_init(bar_p_full + 8 * t, 4);   // one arrival per softmax warp
      ptx::mbar_init(bar_p_half + 8 * t, 4);
      ptx::mbar_init(bar_o_full + 8 * t, 1);
      ptx::mbar_init(bar_o_empty + 8 * t, 128);
    }
    for (int s = 0; s < kSlots; ++s) {
      ptx::mbar_init(bar_kv_full + 8 * s, 1);
      ptx::mbar_init(bar_kv_empty + 8 * s, 1);
    }
    ptx::mbar_init(bar_teardown, 1);
    ptx::mbar_init(bar_stats_full, 128);
    ptx::mbar_init(bar_stats_empty, 128);
    *abort_flag = 0;
    ptx::fence_mbarrier_init();
  }
  if (warp == kWarpProducer && lane == 0) {
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
    ptx::prefetch_tensormap(&tm_o);
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int grid = gridDim.x;
  const int cta = blockIdx.x;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    // The K/V ring holds kSlots slots of two tiles. Each slot is filled and
    // released as a unit (one full and one empty barrier phase): per key tile
    // j the MMA thread needs V_j and K_{j+1} together, so one wait covers both.
    const uint64_t pol_kv = ptx::policy_evict_last();
    const uint64_t pol_q = ptx::policy_evict_first();
    uint32_t slot_it = 0, act = 0;
    int load_idx = 0;
    bool ok = true;
    // Fill the next slot: tile (map0, key tile j0) of (kvh0, b0) at position 0
    // and (map1, j1) of (kvh1, b1) at position 1; either map may be null.
    auto load_slot = [&](const CUtensorMap* map0, int j0, int kvh0, int b0, const CUtensorMap* map1, int j1,
                         int kvh1, int b1) -> bool {
      const uint32_t sl = slot_it % kSlots;
      const uint32_t ph = ((slot_it / kSlots) & 1u) ^ 1u;
      if (!bar_wait(bar_kv_empty + 8 * sl, ph, abort_flag, p)) return false;
      if (lane == 0 && load_idx != p.inject_skip_load) {
        ptx::mbar_arrive_expect_tx(bar_kv_full + 8 * sl, ((map0 ? 1 : 0) + (map1 ? 1 : 0)) * L::kTileBytes);
        const uint32_t dst = sKV + sl * 2 * L::kTileBytes;
        if (map0) {
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_load_4d(dst + c * L::kChunkBytes, map0, bar_kv_full + 8 * sl, c * 64, kvh0, j0 * kBN, b0,
                             pol_kv);
        }
        if (map1) {
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_load_4d(dst + L::kTileBytes + c * L::kChunkBytes, map1, bar_kv_full + 8 * sl, c * 64, kvh1,
                             j1 * kBN, b1, pol_kv);
        }
      }
      __syncwarp();
      ++slot_it;
      ++load_idx;
      return true;
    };
    auto load_q = [&](int t, int hq, int r0, int b) -> bool {
      if (!bar_wait(bar_q_empty + 8 * t, (act & 1u) ^ 1u, abort_flag, p)) return false;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar_q_full + 8 * t, L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          ptx::tma_load_4d(sQ + t * L::kTileBytes + c * L::kChunkBytes, &tm_q, bar_q_full + 8 * t, c * 64, hq, r0,
                           b + p.q_b_shift, pol_q);
      }
      __syncwarp();
      return true;
    };
    // Q tiles are read once from HBM: pull the next item's into L2 while
    // this one runs, so that its TMA load at the item boundary hits L2.
    auto prefetch_q = [&](const WorkItem& nw) {
      if (lane == 0 && p.q_b_shift == 0) {
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          ptx::tma_prefetch_l2_4d(&tm_q, c * 64, nw.hq0, nw.r0, nw.b);
          if (!KSPLIT) ptx::tma_prefetch_l2_4d(&tm_q, c * 64, nw.hq1, nw.r1, nw.b);
        }
      }
    };
    if constexpr (KSPLIT) {
      for (int round = 0; ok; ++round) {
        const int idx = item_of_round(round, cta, grid);
        if (round * grid >= p.n_items) break;
        if (idx >= p.n_items) continue;
        const WorkItem w = decode_item<KSPLIT>(p, idx);
        if (w.n_kv == 0) continue;
        const int n = w.n_kv;
        // slot t runs key tiles t, t+2, ...; n1 of them for slot 1
        const int n1 = n / 2, n0 = n - n1;
        // first slot: K_0 and K_1
        ok = load_q(0, w.hq0, w.r0, w.b) &&
             load_slot(&tm_k, 0, w.kvh, w.b, n1 > 0 ? &tm_k : nullptr, 1, w.kvh, w.b);
        const int nr = next_round<KSPLIT>(p, round + 1, cta, grid);
        if (ok && nr >= 0) prefetch_q(decode_item<KSPLIT>(p, item_of_round(nr, cta, grid)));
        // per step s, for slot 0 then slot 1: (V of its tile, K of its next tile)
        for (int st = 0; ok && st < n0; ++st) {
          ok = load_slot(&tm_v, 2 * st, w.kvh, w.b, st + 1 < n0 ? &tm_k : nullptr, 2 * st + 2, w.kvh, w.b);
          if (ok && st < n1)
            ok = load_slot(&tm_v, 2 * st + 1, w.kvh, w.b, st + 1 < n1 ? &tm_k : nullptr, 2 * st + 3, w.kvh, w.b);
        }
        ++act;
      }
    } else {
      // Row-tile pairs: the CTA's items form one stream of slots. Slot use u
      // holds (V_{j-1}, K_j) of one item, and an item's last slot holds its
      // last V together with K_0 of the CTA's next item, so that the next
      // item's first Q K^T can start as soon as this item's last P V is issued.
      int round = next_round<KSPLIT>(p, 0, cta, grid);
      bool first = true;
      while (ok && round >= 0) {
        const WorkItem w = decode_item<KSPLIT>(p, item_of_round(round, cta, grid));
        const int n = w.n_kv;
        const int nr = next_round<KSPLIT>(p, round + 1, cta, grid);
        WorkItem nw = w;
        if (nr >= 0) nw = decode_item<KSPLIT>(p, item_of_round(nr, cta, grid));
        if (first) {
          // the first slot of the stream holds K_0 alone (position 1)
          ok = load_q(0, w.hq0, w.r0, w.b) && load_slot(nullptr, 0, 0, 0, &tm_k, 0, w.kvh, w.b) &&
               load_q(1, w.hq1, w.r1, w.b);
          first = false;
        } else {
          ok = load_q(0, w.hq0, w.r0, w.b) && load_q(1, w.hq1, w.r1, w.b);
        }
        if (ok && nr >= 0) prefetch_q(nw);
        for (int j = 0; ok && j < n; ++j) {
          if (j + 1 < n)
            ok = load_slot(&tm_v, j, w.kvh, w.b, &tm_k, j + 1, w.kvh, w.b);
          else
            ok = load_slot(&tm_v, j, w.kvh, w.b, nr >= 0 ? &tm_k : nullptr, 0, nw.kvh, nw.b);
        }
        ++act;
        round = nr;
      }
    }
    if (!ok && lane == 0) {
      // Let copies already in flight land before the CTA leaves: wait (bounded)
      // for the latest phase of every slot that was filled.
      const uint64_t t0 = ptx::globaltimer_ns();
      for (uint32_t k = (slot_it > (uint32_t)kSlots ? slot_it - kSlots : 0); k < slot_it; ++k) {
        const uint32_t sl = k % kSlots, ph = (k / kSlots) & 1u;
        while (!ptx::mbar_try_wait(bar_kv_full + 8 * sl, ph) && ptx::globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // Pipe order per key tile j: P0 V_j, Q0 K_{j+1}^T, P1 V_j, Q1 K_{j+1}^T,
    // each P_t V_j as soon as the softmax has written P_t. Ring tiles are
    // numbered 2 * slot + position. Lane 0 alone runs the loop.
    //
    // On sm_103a the tensor pipe holds only a few queued MMAs, so every cycle
    // this thread spends outside tcgen05.mma issue can leave it idle. Measured
    // in isolation: a commit costs nothing, a satisfied mbarrier.test_wait 17
    // cycles, but a test_wait right behind a commit about 60. So the readiness
    // of the next P is tested between the MMAs of a group, not after its
    // commit, and the result is used when that group's turn comes.
    constexpr uint32_t idesc_s = ptx::idesc_f16(BF16, kBM, kBN, false, false);
    constexpr uint32_t idesc_o = ptx::idesc_f16(BF16, kBM, D, false, true);
    constexpr uint32_t kStageDesc = L::kTileBytes >> 4;   // descriptor units per ring tile
    constexpr int kS = D / 16;    // MMAs per S tile (over the head dimension)
    constexpr int kPV = kBN / 16; // MMAs per P V (over the keys)
    // Descriptor bases; the start-address field (bits 0..13) is advanced by
    // adding byte offsets >> 4 (shared addresses stay below 256 KB).
    const uint64_t dq0 = ptx::sdesc_sw128(sQ, 16, 1024);
    const uint64_t dq1 = ptx::sdesc_sw128(sQ + L::kTileBytes, 16, 1024);
    const uint64_t dk0 = ptx::sdesc_sw128(sKV, 16, 1024);                 // K: K-major
    const uint64_t dv0 = ptx::sdesc_sw128(sKV, L::kChunkBytes, 1024);     // V: MN-major
    uint32_t slot_it = 0, act = 0, p_phase[2] = {0u, 0u}, ph_phase[2] = {0u, 0u};
    bool ok = true;
    // S_t = Q_t K^T with K in ring tile kt, k-steps [k0, k1).
    auto issue_s = [&](int t, uint32_t kt, int k0, int k1) {
      const uint64_t a = (t && !KSPLIT) ? dq1 : dq0;   // key-split: both slots read Q tile 0
      const uint64_t bk = dk0 + kt * kStageDesc;
      const uint32_t d = tmem + (t ? kColS1 : kColS0);
#pragma unroll
      for (int ks = 0; ks < kS; ++ks) {
        if (ks < k0 || ks >= k1) continue;
        const uint32_t off = static_cast<uint32_t>(((ks / 4) * L::kChunkBytes + (ks % 4) * 32) >> 4);
        ptx::mma_ss(d, a + off, bk + off, idesc_s, ks > 0 ? 1u : 0u);
      }
    };
    // O_t (+)= P_t V with V in ring tile vt, k-steps (16 keys each) [k0, k1);
    // P from TMEM.
    auto issue_pv = [&](int t, uint32_t vt, int k0, int k1, bool first) {
      const uint64_t bv = dv0 + vt * kStageDesc;
      const uint32_t d = tmem + (t ? kColO1 : kColO0);
      const uint32_t pa = tmem + (t ? kColS1 : kColS0);
#pragma unroll
      for (int ks = 0; ks < kPV; ++ks) {
        if (ks < k0 || ks >= k1) continue;
        ptx::mma_ts(d, pa + ks * 8, bv + static_cast<uint32_t>((ks * 16 * 128) >> 4), idesc_o,
                    (first && ks == 0) ? 0u : 1u);
      }
    };
    // Wait for the next slot; returns its index in `sl`.
    auto wait_slot = [&](uint32_t& sl) -> bool {
      sl = slot_it % kSlots;
      const bool r = bar_wait(bar_kv_full + 8 * sl, (slot_it / kSlots) & 1u, abort_flag, p);
      ++slot_it;
      return r;
    };
    // P_t ready (all of it: one wait per tile, not one per half). `seen` says
    // an earlier test_wait already saw this phase complete.
    auto wait_p = [&](int t, bool seen) -> bool {
      if (!seen && !bar_wait(bar_p_full + 8 * t, p_phase[t], abort_flag, p)) return false;
      p_phase[t] ^= 1u;
      ptx::tc_fence_after();
      return true;
    };
    // Row-tile pairs: the first half of P_t (keys 0..63) ready.
    auto wait_p_half = [&](int t, bool seen) -> bool {
      if (!seen && !bar_wait(bar_p_half + 8 * t, ph_phase[t], abort_flag, p)) return false;
      ph_phase[t] ^= 1u;
      ptx::tc_fence_after();
      return true;
    };
    if (lane == 0) {
      if constexpr (KSPLIT) {
        for (int round = 0; ok; ++round) {
          const int idx = item_of_round(round, cta, grid);
          if (round * grid >= p.n_items) break;
          if (idx >= p.n_items) continue;
          const WorkItem w = decode_item<KSPLIT>(p, idx);
          if (w.n_kv == 0) continue;
          const int n = w.n_kv;
          const uint32_t par = act & 1u;
          uint32_t sl = 0;
          // Slot t runs key tiles t, t+2, ...: S_t from its first key tile,
          // then per step P_t V and the next S_t, each from a ring slot of its
          // own.
          const int n1 = n / 2, n0 = n - n1;
          // prologue: S_0 from K_0 (position 0) and S_1 from K_1 (position 1)
          if (!(ok = bar_wait(bar_q_full, par, abort_flag, p) && wait_slot(sl))) break;
          if (n1 == 0) {
            // slot 1 has no key tile: close its O phase without an MMA
            if (!(ok = bar_wait(bar_o_empty + 8, par ^ 1u, abort_flag, p))) break;
          }
          ptx::tc_fence_after();
          issue_s(0, 2 * sl, 0, kS);
          ptx::mma_commit(bar_s_full);
          if (n1 > 0) {
            issue_s(1, 2 * sl + 1, 0, kS);
            ptx::mma_commit(bar_s_full + 8);
          } else {
            ptx::mma_commit(bar_o_full + 8);
          }
          ptx::mma_commit(bar_kv_empty + 8 * sl);
          if (n0 == 1 && n1 <= 1) ptx::mma_commit(bar_q_empty);   // no S after these
          for (int sj = 0; ok && sj < n0; ++sj) {
            for (int t = 0; t < 2; ++t) {
              const int nt = t ? n1 : n0;
              if (sj >= nt) break;
              if (!(ok = wait_slot(sl))) break;
              if (sj == 0 && !(ok = bar_wait(bar_o_empty + 8 * t, par ^ 1u, abort_flag, p))) break;
              if (!(ok = wait_p(t, false))) break;
              issue_pv(t, 2 * sl, 0, kPV, sj == 0);
              if (sj + 1 < nt) {
                issue_s(t, 2 * sl + 1, 0, kS);
                ptx::mma_commit(bar_s_full + 8 * t);
                // Q's last reader: slot 1's last S when slot 1 runs as many
                // steps as slot 0, else slot 0's
                if (sj + 2 == n0 && (t == 1 || n1 < n0)) ptx::mma_commit(bar_q_empty);
              } else {
                ptx::mma_commit(bar_o_full + 8 * t);
              }
              ptx::mma_commit(bar_kv_empty + 8 * sl);
            }
          }
          ++act;
        }
      } else {
        // Row-tile pairs, the CTA's items back to back (see the producer): the
        // last group of an item issues, after P_t V_{n-1}, the next item's
        // first S_t from K_0 in the same slot.
        int round = next_round<KSPLIT>(p, 0, cta, grid);
        if (round >= 0) {
          int n = decode_item<KSPLIT>(p, item_of_round(round, cta, grid)).n_kv;
          uint32_t sl = 0;
          // prologue of the stream: S_0 = Q_0 K_0^T as soon as Q_0 and K_0
          // (position 1 of the first slot) land, then S_1
          ok = bar_wait(bar_q_full, 0, abort_flag, p) && wait_slot(sl);
          if (ok) {
            ptx::tc_fence_after();
            issue_s(0, 2 * sl + 1, 0, kS);
            ptx::mma_commit(bar_s_full);
            if (n == 1) ptx::mma_commit(bar_q_empty);
            ok = bar_wait(bar_q_full + 8, 0, abort_flag, p);
          }
          if (ok) {
            ptx::tc_fence_after();
            issue_s(1, 2 * sl + 1, 0, kS);
            ptx::mma_commit(bar_s_full + 8);
            if (n == 1) ptx::mma_commit(bar_q_empty + 8);
          }
          while (ok) {
            const uint32_t par = act & 1u;
            const int nr = next_round<KSPLIT>(p, round + 1, cta, grid);
            const int nn = nr >= 0 ? decode_item<KSPLIT>(p, item_of_round(nr, cta, grid)).n_kv : 0;
            bool seen[2] = {false, false};   // P_t's next phase already seen complete
            for (int j = 0; ok && j < n; ++j) {
              const bool more = (j + 1 < n);
              const bool last_s = (j + 2 == n);   // S_t(j+1) is the item's last use of Q_t
              // One slot holds V_j (position 0) and K_{j+1} (position 1), or
              // after the last V the next item's K_0. The MMA thread does not
              // wait for it: the tile-0 softmax checks it before it signals
              // P_0(j) (at D = 64, its first half), so that signal implies the
              // slot is full, and the tile-1 softmax releases it.
              sl = slot_it % kSlots;
              ++slot_it;
              for (int t = 0; t < 2; ++t) {
                if (j == 0 && !(ok = bar_wait(bar_o_empty + 8 * t, par ^ 1u, abort_flag, p))) break;
                // the group: P_t V_j (at D = 64 its first half as soon as the
                // softmax has written keys 0..63 of P_t, while it computes the
                // rest), then Q_t K_{j+1}^T; the next group's P (first half)
                // is tested just before the group's last MMA
                const int kv0 = kHalfP ? kPV / 2 : 0;   // P V k-steps issued before all of P_t is in
                if constexpr (kHalfP) {
                  if (!(ok = wait_p_half(t, seen[t]))) break;
                  issue_pv(t, 2 * sl, 0, kv0, j == 0);
                }
                if (!(ok = wait_p(t, kHalfP ? false : seen[t]))) break;
                const int o = 1 - t;
                const uint32_t next_p = kHalfP ? bar_p_half + 8 * o : bar_p_full + 8 * o;
                const uint32_t next_ph = kHalfP ? ph_phase[o] : p_phase[o];
                if (more) {
                  issue_pv(t, 2 * sl, kv0, kPV, kv0 == 0 && j == 0);
                  issue_s(t, 2 * sl + 1, 0, kS - 1);
                  seen[o] = ptx::mbar_test_wait(next_p, next_ph);
                  issue_s(t, 2 * sl + 1, kS - 1, kS);
                  ptx::mma_commit(bar_s_full + 8 * t);
                  if (last_s) ptx::mma_commit(bar_q_empty + 8 * t);
                } else {
                  issue_pv(t, 2 * sl, kv0, kPV - 1, kv0 == 0 && j == 0);
                  seen[o] = ptx::mbar_test_wait(next_p, next_ph);
                  issue_pv(t, 2 * sl, kPV - 1, kPV, false);
                  ptx::mma_commit(bar_o_full + 8 * t);
                  if (nr >= 0) {
                    // the next item's S_t = Q_t K_0^T, K_0 at position 1
                    if (!(ok = bar_wait(bar_q_full + 8 * t, par ^ 1u, abort_flag, p))) break;
                    ptx::tc_fence_after();
                    issue_s(t, 2 * sl + 1, 0, kS);
                    ptx::mma_commit(bar_s_full + 8 * t);
                    if (nn == 1) ptx::mma_commit(bar_q_empty + 8 * t);
                  }
                }
              }
            }
            ++act;
            if (nr < 0) break;
            round = nr;
            n = nn;
          }
        }
      }
      if (!ok) {
        // Wait (bounded) for every MMA already issued before TMEM is released.
        ptx::mma_commit(bar_teardown);
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar_teardown, 0) && ptx::globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = threadIdx.x & 127;       // TMEM lane == row of the tile
    const uint32_t lane_bits = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_bits + (t ? kColS1 : kColS0);
    const uint32_t tO = tmem + lane_bits + (t ? kColO1 : kColO0);
    const float sl2 = p.scale_log2;
    const int offset = p.Sk - p.Sq;
    uint32_t s_phase = 0, act = 0;
    // Row-tile pairs: K/V ring slot uses, counted like the producer's (an
    // item of n key tiles starts at the use that holds its K_0 and ends at
    // use0 + n, which holds its last V and the next item's K_0).
    uint32_t slot_it = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_of_round(round, cta, grid);
      if (round * grid >= p.n_items) break;
      if (idx >= p.n_items) continue;
      const WorkItem w = decode_item<KSPLIT>(p, idx);
      const int hq = t ? w.hq1 : w.hq0;
      const int r0 = t ? w.r1 : w.r0;
      const int i = r0 + row;                // query row index
      const bool row_valid = i < p.Sq;
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                      (static_cast<long long>(w.b) * p.o_sb + static_cast<long long>(i) * p.o_ss +
                       static_cast<long long>(hq) * p.o_sh) * 2;
      if (w.n_kv == 0) {
        if (row_valid && !(KSPLIT && t == 1)) {   // key-split: slot 0 owns the rows
          uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < p.d_true * 2 / 16; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
          if (p.lse) p.lse[(static_cast<long long>(w.b) * p.Hq + hq) * p.Sq + i] = -__int_as_float(0x7f800000);
        }
        continue;
      }
      // exclusive key bound of this row (no key visible when <= 0)
      int lim_abs = p.Sk;
      if (p.causal) {
        long long l2 = static_cast<long long>(i) + offset + 1;
        lim_abs = static_cast<int>(l2 < 0 ? 0 : (l2 > p.Sk ? p.Sk : l2));
      }
      // key tiles from this one on need the mask for some row of this tile
      int first_masked = p.n_kv_tiles;
      if (p.Sk % kBN) first_masked = p.n_kv_tiles - 1;
      if (p.causal) {
        long long fm = (static_cast<long long>(r0) + offset + 1) / kBN;  // first tile not fully visible to row r0
        if (static_cast<long long>(r0) + offset + 1 < 0) fm = 0;
        if (fm < first_masked) first_masked = static_cast<int>(fm);
      }
      float m_ref = -__int_as_float(0x7f800000);
      float l_exact = 0.0f, l_corr = 0.0f;
      const uint32_t use0 = slot_it;   // row-tile pairs: this item's first ring slot use
      // key-split: this slot's key tiles are t, t+2, ...
      const int n_mine = KSPLIT ? (t ? w.n_kv / 2 : w.n_kv - w.n_kv / 2) : w.n_kv;
      for (int sj = 0; sj < n_mine; ++sj) {
        const int j = KSPLIT ? 2 * sj + t : sj;   // key tile
        if (!(ok = bar_wait(bar_s_full + 8 * t, s_phase, abort_flag, p))) break;
        if constexpr (!KSPLIT) {
          // S_1(j) has completed, and with it every MMA that reads ring slot
          // use0 + j (K_0 when j = 0, beside the previous item's last V;
          // else V_{j-1} and K_j): release the slot
          if (warp == 4 && lane == 0) ptx::mbar_arrive(bar_kv_empty + 8 * ((use0 + j) % kSlots));
          // The MMA thread reads V_j and K_{j+1} (slot use0 + j + 1) as soon
          // as it sees P_0(j) (at D = 64, its first half), without a wait of
          // its own: that is signalled only after this wait (normally long
          // satisfied) has seen the slot full.
          if (warp == 0) {
            const uint32_t u = use0 + j + 1;
            bool r = true;
            if (lane == 0) r = bar_wait(bar_kv_full + 8 * (u % kSlots), (u / kSlots) & 1u, abort_flag, p);
            if (!(ok = __shfl_sync(0xffffffffu, r, 0))) break;
          }
        }
        s_phase ^= 1u;
        ptx::tc_fence_after();
        uint32_t sr[128];
        ptx::tmem_ld_32x32b_x128(tS, sr);
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        // Mask (only tiles from first_masked on) and the row's largest scaled
        // score mx * sl2; the exponents below are s * sl2 - m.
        const float mx = prepare_row(s, j >= first_masked, lim_abs - j * kBN, sl2);
        const float m_new = fmaxf(m_ref, mx * sl2);
        float alpha = 1.0f;
        const bool need = m_new > m_ref + kRescaleThreshold;
        if (need) {
          alpha = ptx::ex2_approx(m_ref - m_new);   // 0 when m_ref = -inf
          m_ref = m_new;
          l_exact *= alpha;
          l_corr *= alpha;
        }
        const float neg_m = (m_ref == -__int_as_float(0x7f800000)) ? 0.0f : -m_ref;
        const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
        const uint64_t negm2 = ptx::f2_pack(neg_m, neg_m);
        // p = 2^(s * scale * log2e - m). P is rounded to the input dtype for the
        // P V product; l_exact sums the unrounded fp32 p (it gives LSE). The
        // largest p of this tile (the element equal to the tile max) is also
        // rounded here, and its rounding error is added to l_corr, so that O is
        // normalised by the sum of the weights the MMA actually used for the
        // dominant terms: when one key dominates a row, O reproduces its value.
        uint64_t acc0 = 0, acc1 = 0;
        {
          const float pmax = ptx::ex2_approx(fmaf(mx, sl2, neg_m));
          const uint32_t pr = pack2<BF16>(pmax, 0.0f);
          float pmax_r;
          if constexpr (BF16) {
            pmax_r = __uint_as_float(pr << 16);
          } else {
            float hi_unused;
            ptx::f16x2_to_f32(pr, pmax_r, hi_unused);
          }
          l_corr += pmax_r - pmax;
        }
        auto exp_half = [&](int h, uint32_t (&pk)[32]) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int e = 64 * h + 2 * c;
            float t0, t1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[e], s[e + 1]), sl2x2, negm2), t0, t1);
            const float p0 = ptx::ex2_approx(t0), p1 = ptx::ex2_approx(t1);
            pk[c] = pack2<BF16>(p0, p1);
            if (c & 1) acc1 = ptx::f2_add(acc1, ptx::f2_pack(p0, p1));
            else acc0 = ptx::f2_add(acc0, ptx::f2_pack(p0, p1));
          }
        };
        {
          uint32_t pk[32];
          exp_half(0, pk);
          ptx::tmem_st_32x32b_x32(tS, pk);
        }
        // Rescale O~ when some row of this warp raised its reference max. The
        // previous P V of this tile completed before S of this key tile did.
        if (sj > 0 && __any_sync(0xffffffffu, need)) {
          const uint64_t a2 = ptx::f2_pack(alpha, alpha);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            ptx::tmem_ld_32x32b_x32(tO + c * 32, orr);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float x0, x1;
              ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1])), a2),
                             x0, x1);
              orr[e] = __float_as_uint(x0);
              orr[e + 1] = __float_as_uint(x1);
            }
            ptx::tmem_st_32x32b_x32(tO + c * 32, orr);
          }
        }
        if constexpr (kHalfP) {
          // keys 0..63 of P_t and any rescale of O~ are in tensor memory:
          // the MMA thread may start P_t V_j on them
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar_p_half + 8 * t);
        }
        {
          uint32_t pk[32];
          exp_half(1, pk);
          ptx::tmem_st_32x32b_x32(tS + 32, pk);
        }
        {
          float a0, a1;
          ptx::f2_unpack(ptx::f2_add(acc0, acc1), a0, a1);
          l_exact += a0 + a1;
        }
        // every lane's P stores complete, then one arrival for the warp
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_p_full + 8 * t);
      }
      if (!ok) break;
      if constexpr (KSPLIT) {
        // ---- key-split epilogue: slot 1 hands (m, l, l_corr) to slot 0, which
        // combines both slots' states and stores O and LSE
        float* stats = reinterpret_cast<float*>(base_ptr + L::kStatsOff);
        if (t == 1) {
          if (!(ok = bar_wait(bar_stats_empty, (act & 1u) ^ 1u, abort_flag, p))) break;
          stats[row] = m_ref;
          stats[kBM + row] = l_exact;
          stats[2 * kBM + row] = l_corr;
          ptx::mbar_arrive(bar_stats_full);
          ++act;
          continue;
        }
        if (!(ok = bar_wait(bar_stats_full, act & 1u, abort_flag, p))) break;
        const float m1 = stats[row], l1 = stats[kBM + row], c1 = stats[2 * kBM + row];
        ptx::mbar_arrive(bar_stats_empty);
        // a slot with a finite m saw a key (and has l >= 1); one whose m is
        // still -inf contributes nothing
        const bool seen0 = m_ref != -__int_as_float(0x7f800000), seen1 = m1 != -__int_as_float(0x7f800000);
        const float m = seen1 ? (seen0 ? fmaxf(m_ref, m1) : m1) : m_ref;
        const float a0 = seen0 ? ptx::ex2_approx(m_ref - m) : 0.0f;
        const float a1 = seen1 ? ptx::ex2_approx(m1 - m) : 0.0f;
        const float l_tot = a0 * l_exact + a1 * l1;
        const bool live = seen0 || seen1;
        const float inv_l = live ? __frcp_rn(a0 * (l_exact + l_corr) + a1 * (l1 + c1)) : 0.0f;
        const uint64_t f0 = ptx::f2_pack(a0 * inv_l, a0 * inv_l);
        const uint64_t f1 = ptx::f2_pack(a1 * inv_l, a1 * inv_l);
        const bool has1 = w.n_kv >= 2;   // slot 1 ran at least one key tile
        if (!(ok = bar_wait(bar_o_full, act & 1u, abort_flag, p) && bar_wait(bar_o_full + 8, act & 1u, abort_flag, p)))
          break;
        ptx::tc_fence_after();
        const uint32_t tO1 = tmem + lane_bits + kColO1;
        const int wrow = row & 31;
        const uint32_t stage = base + L::kOStageOff + warp * L::kOStageWarpBytes;
#pragma unroll
        for (int ch = 0; ch < L::kChunks; ++ch) {
          uint32_t x0[64], x1[64];
          ptx::tmem_ld_32x32b_x64(tO + 64 * ch, x0);
          if (has1) {
            ptx::tmem_ld_32x32b_x64(tO1 + 64 * ch, x1);
          } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) x1[c] = 0u;
          }
          if (ch == L::kChunks - 1) {
            // both accumulators are in registers: the MMA may reuse them
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_o_empty);
            ptx::mbar_arrive(bar_o_empty + 8);
          }
          uint32_t ob[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint64_t y0 = ptx::f2_pack(__uint_as_float(x0[2 * c]), __uint_as_float(x0[2 * c + 1]));
            const uint64_t y1 = ptx::f2_pack(__uint_as_float(x1[2 * c]), __uint_as_float(x1[2 * c + 1]));
            float a, b;
            ptx::f2_unpack(ptx::f2_fma(y1, f1, ptx::f2_mul(y0, f0)), a, b);
            ob[c] = pack2<BF16>(a, b);
          }
          if (lane == 0) ptx::bulk_wait_group_read0();   // the previous store has read the buffer
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            ptx::st_shared_v4(stage + wrow * 128 + ((k ^ (wrow & 7)) << 4), ob[4 * k], ob[4 * k + 1], ob[4 * k + 2],
                              ob[4 * k + 3]);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_4d(&tm_o, stage, ch * 64, hq, r0 + (warp & 3) * 32, w.b);
            ptx::bulk_commit_group();
          }
        }
        if (row_valid && p.lse) {
          const float lse = live ? (m + __log2f(l_tot)) * 0.69314718055994531f : -__int_as_float(0x7f800000);
          p.lse[(static_cast<long long>(w.b) * p.Hq + hq) * p.Sq + i] = lse;
        }
        ++act;
        continue;
      }
      // ---- epilogue: O = O~ / l, LSE = (m + log2 l) * ln 2
      if (!(ok = bar_wait(bar_o_full + 8 * t, act & 1u, abort_flag, p))) break;
      // The item's last slot use (use0 + n) also holds the next item's K_0:
      // the next item's tile-1 softmax releases it with its first S_1.
      slot_it = use0 + w.n_kv;
      ptx::tc_fence_after();
      uint32_t orr[D];
      if constexpr (D == 128) {
        ptx::tmem_ld_32x32b_x128(tO, orr);
      } else {
        ptx::tmem_ld_32x32b_x64(tO, orr);
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_o_empty + 8 * t);
      const bool live = m_ref != -__int_as_float(0x7f800000);   // some key seen: l >= 1
      const float inv_l = live ? __frcp_rn(l_exact + l_corr) : 0.0f;
      // Scale, round to the dtype and stage this warp's 32 rows one 64-column
      // chunk at a time in the 128-byte-swizzled layout of the O tensor map;
      // lane 0 stores each chunk with TMA (rows past Sq are clipped by it).
      {
        const uint64_t il2 = ptx::f2_pack(inv_l, inv_l);
        const int wrow = row & 31;
        const uint32_t stage = base + L::kOStageOff + warp * L::kOStageWarpBytes;
#pragma unroll
        for (int ch = 0; ch < L::kChunks; ++ch) {
          uint32_t ob[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float a0, a1;
            ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(orr[64 * ch + 2 * c]),
                                                    __uint_as_float(orr[64 * ch + 2 * c + 1])), il2), a0, a1);
            ob[c] = pack2<BF16>(a0, a1);
          }
          if (lane == 0) ptx::bulk_wait_group_read0();   // the previous store has read the buffer
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            ptx::st_shared_v4(stage + wrow * 128 + ((k ^ (wrow & 7)) << 4), ob[4 * k], ob[4 * k + 1], ob[4 * k + 2],
                              ob[4 * k + 3]);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_4d(&tm_o, stage, ch * 64, hq, r0 + (warp & 3) * 32, w.b);
            ptx::bulk_commit_group();
          }
        }
      }
      if (row_valid && p.lse) {
        const float lse = live ? (m_ref + __log2f(l_exact)) * 0.69314718055994531f : -__int_as_float(0x7f800000);
        p.lse[(static_cast<long long>(w.b) * p.Hq + hq) * p.Sq + i] = lse;
      }
      ++act;
    }
    if (lane == 0) ptx::bulk_wait_group0();   // every O store of this warp has completed
    __syncwarp();
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kWarpMma) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace fa
