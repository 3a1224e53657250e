// Split-KV attention, sm_103a: decode, short chunks and small prefill. One
// CTA handles one row tile of the query rows that share a KV head (the G
// heads of a GQA group times P = floor(128 / G) query positions, "MiniPaged-
// Qwen: Qwen3 Prefill FlashAttention" section 6) against one contiguous
// range of 128-key tiles (a split); the per-split results are normalised
// partial states (O_s, LSE_s) that a merge combines, or the final O when
// there is one split.
// Same arithmetic as the prefill kernel (online softmax with exp2 and the
// log2e-folded scale, bottom-right causal limit of section 13): TMA K/V
// ring, tcgen05 Q K^T into a double-buffered S in tensor memory, softmax by
// one thread per row, P V with P read from tensor memory.
//
// Warp roles (192 threads): warps 0-3 softmax + epilogue (TMEM lanes 0-127,
// row r = s_local * G + g), warp 4 TMA producer, warp 5 MMA issuer / TMEM
// owner. Grid: one CTA per (split, KV head, batch, row tile) along x, row
// tiles slowest and in descending order.
// TMEM columns: S buffer 0 [0,128), S buffer 1 [128,256), O [256, 256+D);
// D = 256 fills all 512.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx_sm103.cuh"
#include "softmax_row.cuh"

namespace fa {

struct DecodeParams {
  void* o;             // final O (B, Sq, Hq, D) 16-bit (one split), element strides below
  long long o_sb, o_ss, o_sh;
  int d_true;          // head dimension of the tensors (<= D, a multiple of 16; the tile is zero padded)
  float* lse;          // final LSE (B, Hq, Sq) or null (one split)
  float* o_part;       // (n_splits, B, Sq, Hq, D) fp32 partial O (several splits)
  float* lse_part;     // (n_splits, B, Hq, Sq) fp32 partial LSE
  int B, Sq, Sk, Hq, Hkv, G;
  int P;               // query positions per row tile: floor(128 / G)
  int n_row_tiles;     // ceil(Sq / P)
  int causal;
  float scale_log2;    // softmax scale * log2(e); nonzero (see q_b_shift)
  int q_b_shift;       // added to the batch coordinate of the Q load: B reads Q as
                       // zeros (TMA zero fill), how a zero scale runs
  int n_splits, n_kv_tiles;
  int unit_group;      // (split, KV head, batch) units whose CTAs run interleaved
  unsigned long long timeout_ns;
  int* status;
};

template <int D>
struct DecodeSmem {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  // Ring unit: a whole K or V tile, or for D = 256 half of one (K: 128 of
  // its 256 columns; V: 64 of its 128 keys), so that beside the 64 KB Q tile
  // five 32 KB units fit instead of two 64 KB tiles and each load has about
  // two MMA groups to land instead of one.
  static constexpr int kHalves = (D == 256) ? 2 : 1;
  static constexpr int kUnitBytes = kTileBytes / kHalves;
  static constexpr int kVChunkBytes = kChunkBytes / kHalves;   // one 64-column chunk of a V unit
  static constexpr int kStages = (D == 256) ? 5 : (D == 128) ? 6 : 12;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kUnitBytes;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full, pv_done, o_full, teardown
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 1 + 1 + 1 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kAlloc = kMiscOff + 16 + 1024;
};

__device__ __forceinline__ bool dec_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         const DecodeParams& p) {
  if (ptx::mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
        atomicCAS(p.status, 0, 4);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t dec_pack2(float lo, float hi) {
  if constexpr (BF16) return ptx::pack_bf16x2(lo, hi);
  else return ptx::pack_f16x2(lo, hi);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(192, 1)
fa_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ DecodeParams p) {
  using L = DecodeSmem<D>;
  constexpr int kStages = L::kStages;
  constexpr int kHalves = L::kHalves;
  constexpr uint32_t kTmemCols = 512;
  constexpr float kRescale = 8.0f;
  const float kNegInf = -__int_as_float(0x7f800000);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t sQ = base + L::kQOff;
  const uint32_t sKV = base + L::kKVOff;
  const uint32_t bar_q_full = base + L::kBarOff;
  const uint32_t bar_kv_full = bar_q_full + 8;
  const uint32_t bar_kv_empty = bar_kv_full + 8 * kStages;
  const uint32_t bar_s_full = bar_kv_empty + 8 * kStages;   // [2]
  const uint32_t bar_p_full = bar_s_full + 16;
  const uint32_t bar_pv_done = bar_p_full + 8;
  const uint32_t bar_o_full = bar_pv_done + 8;
  const uint32_t bar_teardown = bar_o_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // One linear CTA index. Units (split, KV head, batch) go in groups of
  // unit_group whose K/V fit in L2 together; within a group the unit is
  // fastest and the row tile slowest and descending: with a causal mask the
  // last row tiles have the most keys, so the longest CTAs start first and
  // the short ones fill the tail (the longest-first order of "NVIDIA闪存注意力
  // 实操" section "ProgramId重映射").
  const long long n_units = static_cast<long long>(p.n_splits) * p.Hkv * p.B;
  const long long cta = blockIdx.x;
  const long long group_ctas = static_cast<long long>(p.unit_group) * p.n_row_tiles;
  const long long g0 = (cta / group_ctas) * p.unit_group;   // first unit of this CTA's group
  const long long in_group = n_units - g0 < p.unit_group ? n_units - g0 : p.unit_group;
  const long long w_in = cta - g0 * p.n_row_tiles;
  const int rt = p.n_row_tiles - 1 - static_cast<int>(w_in / in_group);
  const int in = static_cast<int>(g0 + w_in % in_group);
  const int split = in % p.n_splits;
  const int kvh = (in / p.n_splits) % p.Hkv, b = in / (p.n_splits * p.Hkv);
  const int pos0 = rt * p.P;                                  // first query position of the tile
  const int rows_box = p.G * p.P;                              // rows the Q box fills
  // key tiles this row tile needs (bottom-right causal limit of its last row)
  int n_need = p.n_kv_tiles;
  if (p.causal) {
    const long long last = static_cast<long long>(min(pos0 + p.P, p.Sq)) - 1;
    long long lim = last + p.Sk - p.Sq + 1;
    if (lim > p.Sk) lim = p.Sk;
    n_need = lim <= 0 ? 0 : static_cast<int>((lim + 127) / 128);
  }
  const int tps = (n_need + p.n_splits - 1) / p.n_splits;
  const int t_begin = split * tps;
  const int n = max(0, min(n_need, t_begin + tps) - t_begin);

  // Rows past G * P of the Q tile are never loaded: zero them so that the
  // unused rows of S, P and O stay finite.
  for (int i = threadIdx.x; i < L::kTileBytes / 16; i += blockDim.x) {
    const int row = (i * 16 / 128) % 128;
    if (row >= rows_box) reinterpret_cast<uint4*>(base_ptr + L::kQOff)[i] = make_uint4(0, 0, 0, 0);
  }
  ptx::fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar_kv_full + 8 * s, 1);
      ptx::mbar_init(bar_kv_empty + 8 * s, 1);
    }
    ptx::mbar_init(bar_s_full, 1);
    ptx::mbar_init(bar_s_full + 8, 1);
    ptx::mbar_init(bar_p_full, 128);
    ptx::mbar_init(bar_pv_done, 1);
    ptx::mbar_init(bar_o_full, 1);
    ptx::mbar_init(bar_teardown, 1);
    *abort_flag = 0;
    ptx::fence_mbarrier_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The merge of the split results may be scheduled from now on: it waits
  // for this grid's completion before it reads anything.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    uint32_t issued = 0;
    if (n > 0 && lane == 0) {
      // K/V stay in L2 while other row tiles of the same KV head will read
      // them (prefill); in decode (one row tile) each byte is read once
      const uint64_t pol_kv = p.n_row_tiles > 1 ? ptx::policy_evict_last() : ptx::policy_evict_first();
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint32_t q_bytes = static_cast<uint32_t>(rows_box) * 128u * L::kChunks;
      ptx::mbar_arrive_expect_tx(bar_q_full, q_bytes);
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c)
        ptx::tma_load_4d(sQ + c * L::kChunkBytes, &tm_q, bar_q_full, c * 64, kvh * p.G, pos0, b + p.q_b_shift, pol_q);
      // Tiles in the order the MMA thread consumes them (each in kHalves
      // pieces): K_0, K_1, then V_0, K_2, V_1, K_3, ..., V_{n-2}, V_{n-1}
      // (S runs two key tiles ahead of P V). Loading in this order, a ring
      // unit is refilled with the next tile the MMA needs once the oldest one
      // is consumed; K_{j+2} is not queued behind V_{j+1}.
      for (int u = 0; ok && u < 2 * kHalves * n; ++u) {
        const uint32_t st = u % kStages, ph = ((u / kStages) & 1u) ^ 1u;
        if (!(ok = dec_wait(bar_kv_empty + 8 * st, ph, abort_flag, p))) break;
        ptx::mbar_arrive_expect_tx(bar_kv_full + 8 * st, L::kUnitBytes);
        const int pos = u / kHalves, h = u % kHalves;
        const int lead = n < 2 ? n : 2;                   // K tiles before the first V
        bool is_k;
        int jt;
        if (pos < lead) {
          is_k = true;
          jt = pos;
        } else {
          const int q = pos - 2;                          // -1 when n == 1
          if (q < 2 * (n - 2)) {
            is_k = (q & 1) != 0;
            jt = is_k ? q / 2 + 2 : q / 2;
          } else {
            is_k = false;
            jt = q - (n - 2);
          }
        }
        const int key0 = (t_begin + jt) * 128;
        const uint32_t dst = sKV + st * L::kUnitBytes;
        if (is_k) {
          // K: column chunks h * kChunks / kHalves ..., all 128 keys
#pragma unroll
          for (int c = 0; c < L::kChunks / kHalves; ++c)
            ptx::tma_load_4d(dst + c * L::kChunkBytes, &tm_k, bar_kv_full + 8 * st,
                             (h * L::kChunks / kHalves + c) * 64, kvh, key0, b, pol_kv);
        } else {
          // V: every column chunk of keys key0 + h * 128 / kHalves ... (the V
          // map's box is 128 / kHalves keys high)
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_load_4d(dst + c * L::kVChunkBytes, &tm_v, bar_kv_full + 8 * st, c * 64, kvh,
                             key0 + h * (128 / kHalves), b, pol_kv);
        }
        ++issued;
      }
      if (!ok) {
        const uint64_t t0 = ptx::globaltimer_ns();
        for (uint32_t k = (issued > (uint32_t)kStages ? issued - kStages : 0); k < issued; ++k)
          while (!ptx::mbar_try_wait(bar_kv_full + 8 * (k % kStages), (k / kStages) & 1u) &&
                 ptx::globaltimer_ns() - t0 < 2000000ull) {
          }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 alone runs the loop (no warp-wide waits or reconvergence
    // between MMA groups); each ring unit is waited for and released in turn.
    constexpr uint32_t idesc_s = ptx::idesc_f16(BF16, 128, 128, false, false);
    constexpr uint32_t idesc_o = ptx::idesc_f16(BF16, 128, D, false, true);
    const uint64_t dq = ptx::sdesc_sw128(sQ, 16, 1024);
    const uint64_t dk0 = ptx::sdesc_sw128(sKV, 16, 1024);
    const uint64_t dv0 = ptx::sdesc_sw128(sKV, L::kVChunkBytes, 1024);   // V: MN-major, chunk stride
    constexpr uint32_t kUnitDesc = L::kUnitBytes >> 4;
    constexpr int kS = D / 16;                  // k-steps of Q K^T (16 columns each)
    constexpr int kSU = kS / kHalves;           // ... per K unit
    constexpr int kPVU = 8 / kHalves;           // k-steps of P V (16 keys each) per V unit
    if (lane == 0 && n > 0) {
      bool ok = true;
      // Ring units are consumed in load order (see the producer): the issue
      // sequence S_0, S_1, P V_0, S_2, P V_1, ... takes the next unit each time.
      int next_u = 0;
      auto wait_unit = [&](int u) -> bool {
        return dec_wait(bar_kv_full + 8 * (u % kStages), (u / kStages) & 1u, abort_flag, p);
      };
      // S buffer jt%2 = Q K_jt^T
      auto issue_s = [&](int jt) -> bool {
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          const int u = next_u++;
          const uint32_t st = u % kStages;
          if (!wait_unit(u)) return false;
          ptx::tc_fence_after();
#pragma unroll
          for (int k = 0; k < kSU; ++k) {
            const int ks = h * kSU + k;
            const uint32_t qoff = static_cast<uint32_t>(((ks / 4) * L::kChunkBytes + (ks % 4) * 32) >> 4);
            const uint32_t koff = static_cast<uint32_t>(((k / 4) * L::kChunkBytes + (k % 4) * 32) >> 4);
            ptx::mma_ss(tmem + 128 * (jt & 1), dq + qoff, dk0 + st * kUnitDesc + koff, idesc_s, ks > 0 ? 1u : 0u);
          }
          if (h + 1 == kHalves) ptx::mma_commit(bar_s_full + 8 * (jt & 1));
          ptx::mma_commit(bar_kv_empty + 8 * st);
        }
        return true;
      };
      ok = dec_wait(bar_q_full, 0, abort_flag, p) && issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      for (int j = 0; ok && j < n; ++j) {
        if (!(ok = dec_wait(bar_p_full, j & 1, abort_flag, p))) break;
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          const int u = next_u++;
          const uint32_t vst = u % kStages;
          if (!(ok = wait_unit(u))) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int k = 0; k < kPVU; ++k) {
            const int ks = h * kPVU + k;
            ptx::mma_ts(tmem + 256, tmem + 128 * (j & 1) + ks * 8,
                        dv0 + vst * kUnitDesc + static_cast<uint32_t>((k * 16 * 128) >> 4), idesc_o,
                        (j == 0 && ks == 0) ? 0u : 1u);
          }
          if (h + 1 == kHalves) {
            ptx::mma_commit(bar_pv_done);
            if (j + 1 == n) ptx::mma_commit(bar_o_full);
          }
          ptx::mma_commit(bar_kv_empty + 8 * vst);
        }
        if (ok && j + 2 < n) ok = issue_s(j + 2);
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
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int row = threadIdx.x;                    // TMEM lane
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const bool row_valid = row < rows_box && pos0 + row / p.G < p.Sq;
    const int s_q = row_valid ? pos0 + row / p.G : 0;   // query position of this row
    const int hq = kvh * p.G + (row_valid ? row % p.G : 0);
    const float sl2 = p.scale_log2;
    int lim_abs = p.Sk;                             // exclusive key bound of this row
    if (p.causal) {
      const long long l2 = static_cast<long long>(s_q) + p.Sk - p.Sq + 1;
      lim_abs = static_cast<int>(l2 < 0 ? 0 : (l2 > p.Sk ? p.Sk : l2));
    }
    float m_ref = kNegInf, l_exact = 0.0f, l_corr = 0.0f;
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      const uint32_t tS = tmem + lane_bits + 128 * (j & 1);
      if (!(ok = dec_wait(bar_s_full + 8 * (j & 1), (j >> 1) & 1, abort_flag, p))) break;
      ptx::tc_fence_after();
      uint32_t sr[128];
      ptx::tmem_ld_32x32b_x128(tS, sr);
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      // Mask where some row of the warp has hidden keys in this tile (the
      // Sk tail, the causal limit); mx * sl2 is the row's largest scaled
      // score and the exponents below are s * sl2 - m.
      const int lim = lim_abs - (t_begin + j) * 128;
      const float mx = prepare_row(s, __any_sync(0xffffffffu, lim < 128), lim, sl2);
      const float m_new = fmaxf(m_ref, mx * sl2);
      float alpha = 1.0f;
      const bool need = m_new > m_ref + kRescale;
      if (need) {
        alpha = ptx::ex2_approx(m_ref - m_new);
        m_ref = m_new;
        l_exact *= alpha;
        l_corr *= alpha;
      }
      const float neg_m = (m_ref == kNegInf) ? 0.0f : -m_ref;
      {
        const float pmax = ptx::ex2_approx(fmaf(mx, sl2, neg_m));
        const uint32_t pr = dec_pack2<BF16>(pmax, 0.0f);
        float pmax_r, unused;
        if constexpr (BF16) pmax_r = __uint_as_float(pr << 16);
        else ptx::f16x2_to_f32(pr, pmax_r, unused);
        l_corr += pmax_r - pmax;
      }
      const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2), negm2 = ptx::f2_pack(neg_m, neg_m);
      uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int e = 64 * h + 2 * c;
          float t0, t1;
          ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[e], s[e + 1]), sl2x2, negm2), t0, t1);
          const float p0 = ptx::ex2_approx(t0), p1 = ptx::ex2_approx(t1);
          pk[c] = dec_pack2<BF16>(p0, p1);
          if (c & 1) acc1 = ptx::f2_add(acc1, ptx::f2_pack(p0, p1));
          else acc0 = ptx::f2_add(acc0, ptx::f2_pack(p0, p1));
        }
        ptx::tmem_st_32x32b_x32(tS + 32 * h, pk);
      }
      {
        float a0, a1;
        ptx::f2_unpack(ptx::f2_add(acc0, acc1), a0, a1);
        l_exact += a0 + a1;
      }
      // P V of the previous key tile must have completed before O~ is rescaled
      if (j > 0) {
        if (!(ok = dec_wait(bar_pv_done, (j - 1) & 1, abort_flag, p))) break;
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
          const uint64_t a2 = ptx::f2_pack(alpha, alpha);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            ptx::tmem_ld_32x32b_x32(tmem + lane_bits + 256 + c * 32, orr);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float x0, x1;
              ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1])), a2),
                             x0, x1);
              orr[e] = __float_as_uint(x0);
              orr[e + 1] = __float_as_uint(x1);
            }
            ptx::tmem_st_32x32b_x32(tmem + lane_bits + 256 + c * 32, orr);
          }
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar_p_full);
    }
    // ---- epilogue: O~ / l in 64-column chunks, final O or fp32 partial
    bool have_o = false;
    if (ok && n > 0) {
      if ((ok = dec_wait(bar_o_full, 0, abort_flag, p))) {
        ptx::tc_fence_after();
        have_o = true;
      }
    }
    const bool live = have_o && l_exact > 0.0f;
    const float inv_l = live ? __frcp_rn(l_exact + l_corr) : 0.0f;
    const float lse = live ? (m_ref + __log2f(l_exact)) * 0.69314718055994531f : kNegInf;
    const bool write = row_valid && (ok || n == 0);
    const long long lidx = (static_cast<long long>(b) * p.Hq + hq) * p.Sq + s_q;
    const long long rows_all = static_cast<long long>(p.B) * p.Sq * p.Hq;
    const long long orow = (static_cast<long long>(b) * p.Sq + s_q) * p.Hq + hq;
    uint16_t* ofinal = static_cast<uint16_t*>(p.o) + static_cast<long long>(b) * p.o_sb +
                       static_cast<long long>(s_q) * p.o_ss + static_cast<long long>(hq) * p.o_sh;
    float* opart = p.o_part + (split * rows_all + orow) * p.d_true;
#pragma unroll 1
    for (int c0 = 0; c0 < p.d_true; c0 += 64) {
      uint32_t oc[64];
      if (have_o) ptx::tmem_ld_32x32b_x64(tmem + lane_bits + 256 + c0, oc);   // whole warp
      if (write && p.n_splits == 1) {
        uint4* dst = reinterpret_cast<uint4*>(ofinal + c0);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (c0 + 8 * c >= p.d_true) break;
          float x[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) x[q] = live ? __uint_as_float(oc[8 * c + q]) * inv_l : 0.0f;
          dst[c] = make_uint4(dec_pack2<BF16>(x[0], x[1]), dec_pack2<BF16>(x[2], x[3]), dec_pack2<BF16>(x[4], x[5]),
                              dec_pack2<BF16>(x[6], x[7]));
        }
      } else if (write) {
        float4* dst = reinterpret_cast<float4*>(opart + c0);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (c0 + 4 * c >= p.d_true) break;
          float4 v;
          v.x = live ? __uint_as_float(oc[4 * c + 0]) * inv_l : 0.0f;
          v.y = live ? __uint_as_float(oc[4 * c + 1]) * inv_l : 0.0f;
          v.z = live ? __uint_as_float(oc[4 * c + 2]) * inv_l : 0.0f;
          v.w = live ? __uint_as_float(oc[4 * c + 3]) * inv_l : 0.0f;
          dst[c] = v;
        }
      }
      __syncwarp();
    }
    if (write) {
      if (p.n_splits == 1) {
        if (p.lse) p.lse[lidx] = lse;
      } else {
        p.lse_part[split * rows_all + lidx] = lse;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 5) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace fa
