// Host side of the split-KV path (fa_fwd_decode): argument checks, split
// selection, tensor maps, launch of fa_decode_kernel and of the merge.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/fa.h"
#include "fa_decode_kernel.cuh"
#include "fa_merge.cuh"
#include "tma_host.h"

namespace fa {
int* current_status_word();   // fa_api.cu: the per-device status word read by fa_status()
}

namespace {

constexpr int kMaxDevices = 64;

struct Plan {
  int n_tiles = 0, n_splits = 1, positions = 1, n_row_tiles = 1;
  unsigned long long o_part_bytes = 0, lse_part_bytes = 0;
  unsigned long long workspace_bytes() const { return n_splits > 1 ? o_part_bytes + lse_part_bytes : 0; }
};

// SM count of the current device, looked up once per device (calls from
// several host threads may race to look it up; they store the same value).
int device_sms() {
  static std::atomic<int> sms[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Row tiles of floor(128 / G) query positions, and splits of the key range:
// the requested number, or (num_splits <= 0) as many as keep every CTA in
// one wave on `sms` SMs (a CTA fills an SM's shared memory), since a
// partial second wave leaves most SMs idle while its CTAs stream: timed on
// GB300 decode shapes (batch 4 to 64, 4K to 64K keys) one full wave beat the
// split counts around it by 5 to 30 %. At most one split per key tile.
Plan make_plan(int B, int Sq, int Sk, int Hq, int Hkv, int D, int num_splits, int sms) {
  Plan pl;
  pl.n_tiles = (Sk + 127) / 128;
  const int G = Hkv > 0 ? Hq / Hkv : 1;
  pl.positions = G > 0 ? 128 / G : 1;
  pl.n_row_tiles = (Sq + pl.positions - 1) / pl.positions;
  int want = num_splits;
  if (want <= 0) {
    const long long units = static_cast<long long>(B) * Hkv * pl.n_row_tiles;
    const long long slots = sms > 0 ? sms : 148;
    want = static_cast<int>(units >= slots ? 1 : slots / units);
  }
  if (want > pl.n_tiles) want = pl.n_tiles;
  if (want < 1) want = 1;
  pl.n_splits = want;
  const unsigned long long rows = static_cast<unsigned long long>(B) * Sq * Hq;
  pl.o_part_bytes = static_cast<unsigned long long>(pl.n_splits) * rows * D * 4;
  pl.lse_part_bytes = (static_cast<unsigned long long>(pl.n_splits) * rows * 4 + 15) / 16 * 16;
  return pl;
}

// Checks shared by the size query and the launch (no device access).
int check_args(int B, int Sq, int Sk, int Hq, int Hkv, int D, int dtype) {
  if (B < 0 || Sq < 0 || Sk < 0 || Hq < 0 || Hkv < 0 || D < 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0 || Hq == 0) return FA_OK;
  if (D < 16 || D > 256 || D % 16 != 0) return FA_ERR_UNSUPPORTED;
  if (Hq / Hkv > 128) return FA_ERR_UNSUPPORTED;   // one query position of a whole group must fit a tile
  return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Pieces a K or V tile is loaded in (the V map's box is 128 / that keys high).
int ring_pieces(int Dk) {
  return Dk == 256 ? fa::DecodeSmem<256>::kHalves : Dk == 128 ? fa::DecodeSmem<128>::kHalves
                                                               : fa::DecodeSmem<64>::kHalves;
}

template <int D, bool BF16>
int launch_decode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const fa::DecodeParams& p,
                  dim3 grid, cudaStream_t stream) {
  static std::once_flag f[kMaxDevices];
  static cudaError_t err[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::call_once(f[dev], [&] {
    err[dev] = cudaFuncSetAttribute(fa::fa_decode_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    fa::DecodeSmem<D>::kAlloc);
  });
  if (err[dev] != cudaSuccess) return FA_ERR_CUDA;
  fa::fa_decode_kernel<D, BF16><<<grid, 192, fa::DecodeSmem<D>::kAlloc, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

unsigned long long timeout_ns() {
  static const unsigned long long ns = [] {
    const char* e = std::getenv("FA_WAIT_TIMEOUT_MS");
    const long long ms = e ? std::atoll(e) : 0;
    return static_cast<unsigned long long>(ms > 0 ? ms : 2000) * 1000000ull;
  }();
  return ns;
}

}  // namespace

namespace fa {

// Launch on a given workspace (o_part / lse_part only read when n_splits > 1).
// qs, ks, vs, os: (b, s, h) element strides (16-byte multiples, already
// checked); the workspace layout is always contiguous.
int decode_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk, int Hq,
                  int Hkv, int D, const long long* qs, const long long* ks, const long long* vs, const long long* os,
                  float scale, int causal, int dtype, int num_splits, float* o_part, float* lse_part,
                  unsigned long long workspace_bytes, cudaStream_t stream, int* status_word) {
  const bool bf16 = dtype == FA_DTYPE_BF16;
  const Plan pl = make_plan(B, Sq, Sk, Hq, Hkv, D, num_splits, device_sms());
  if (pl.n_splits > 1 && (workspace_bytes < pl.workspace_bytes() || !o_part || !lse_part)) return FA_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  // the kernel's head dimension: the smallest of 64, 128, 256 that holds D
  const int Dk = D <= 64 ? 64 : (D <= 128 ? 128 : 256);
  CUtensorMap tq, tk, tv;
  if (!encode_bshd_box(&tq, q, bf16, B, Sq, Hq, D, qs, G, pl.positions) ||
      !encode_bshd_box(&tk, k, bf16, B, Sk, Hkv, D, ks, 1, 128) ||
      !encode_bshd_box(&tv, v, bf16, B, Sk, Hkv, D, vs, 1, 128 / ring_pieces(Dk)))
    return FA_ERR_CUDA;
  DecodeParams p{};
  p.o = o;
  p.o_sb = os[0];
  p.o_ss = os[1];
  p.o_sh = os[2];
  p.d_true = D;
  p.lse = lse;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.B = B; p.Sq = Sq; p.Sk = Sk; p.Hq = Hq; p.Hkv = Hkv; p.G = G;
  p.P = pl.positions;
  p.n_row_tiles = pl.n_row_tiles;
  p.causal = causal;
  // A zero scale makes every visible score 0: it runs as scale 1 on Q read as
  // zeros (the same scores, exactly), so that the kernels always have a
  // nonzero scale to rank scores by.
  p.scale_log2 = static_cast<float>(static_cast<double>(scale == 0.0f ? 1.0f : scale) * 1.4426950408889634);
  p.q_b_shift = scale == 0.0f ? B : 0;
  p.n_splits = pl.n_splits;
  p.n_kv_tiles = pl.n_tiles;
  {
    // CTAs of units whose K/V (one split's key range) fit in 32 MiB together
    // run interleaved, so the row tiles reading them hit L2
    const long long keys = static_cast<long long>((pl.n_tiles + pl.n_splits - 1) / pl.n_splits) * 128;
    const long long unit_bytes = 2LL * keys * D * 2;
    const long long n_units = static_cast<long long>(pl.n_splits) * Hkv * B;
    const long long fit = unit_bytes > 0 ? (32LL << 20) / unit_bytes : n_units;
    p.unit_group = static_cast<int>(std::max(1LL, std::min(n_units, fit)));
  }
  p.timeout_ns = timeout_ns();
  p.status = status_word;
  const long long n_cta = static_cast<long long>(pl.n_splits) * pl.n_row_tiles * Hkv * B;
  if (n_cta > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(n_cta));
  int rc;
  if (Dk == 256)
    rc = bf16 ? launch_decode<256, true>(tq, tk, tv, p, grid, stream)
              : launch_decode<256, false>(tq, tk, tv, p, grid, stream);
  else if (Dk == 128)
    rc = bf16 ? launch_decode<128, true>(tq, tk, tv, p, grid, stream)
              : launch_decode<128, false>(tq, tk, tv, p, grid, stream);
  else
    rc = bf16 ? launch_decode<64, true>(tq, tk, tv, p, grid, stream)
              : launch_decode<64, false>(tq, tk, tv, p, grid, stream);
  if (rc != FA_OK || pl.n_splits == 1) return rc;
  return merge_f32_parts(o_part, lse_part, pl.n_splits, o, lse, B, Sq, Hq, D, dtype, stream);
}

}  // namespace fa

extern "C" int fa_decode_workspace_size(int B, int Sq, int Sk, int Hq, int Hkv, int D, int num_splits,
                                        unsigned long long* bytes) {
  if (!bytes) return FA_ERR_INVALID_ARG;
  *bytes = 0;
  const int rc = check_args(B, Sq, Sk, Hq, Hkv, D, FA_DTYPE_BF16);
  if (rc != FA_OK || B == 0 || Sq == 0 || Hq == 0 || Sk == 0) return rc;
  // the automatic split count depends on the SM count of the current device
  *bytes = make_plan(B, Sq, Sk, Hq, Hkv, D, num_splits, num_splits > 0 ? 0 : device_sms()).workspace_bytes();
  return FA_OK;
}

extern "C" int fa_decode_splits(int B, int Sq, int Sk, int Hq, int Hkv, int D, int num_splits, int num_sms,
                                int* n_splits) {
  if (!n_splits || num_sms <= 0) return FA_ERR_INVALID_ARG;
  const int rc = check_args(B, Sq, Sk, Hq, Hkv, D, FA_DTYPE_BF16);
  if (rc != FA_OK) return rc;
  if (B == 0 || Sq == 0 || Hq == 0 || Sk == 0) return FA_ERR_INVALID_ARG;
  *n_splits = make_plan(B, Sq, Sk, Hq, Hkv, D, num_splits, num_sms).n_splits;
  return FA_OK;
}

extern "C" int fa_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk,
                             int Hq, int Hkv, int D, float scale, int causal, int dtype, int num_splits,
                             void* workspace, unsigned long long workspace_bytes, fa_stream_t stream_) {
  int rc = check_args(B, Sq, Sk, Hq, Hkv, D, dtype);
  if (rc != FA_OK) return rc;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  // any finite scale, as long as scale * log2(e) is a finite float
  if (std::fabs(static_cast<double>(scale)) * 1.4426950408889634 > 3.4028234663852886e38)
    return FA_ERR_UNSUPPORTED;
  if (B == 0 || Sq == 0 || Hq == 0) return FA_OK;
  if (Sk == 0) return fa_fwd(q, k, v, o, lse, B, Sq, 0, Hq, Hkv, D, scale, causal, dtype, stream_);
  if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)) ||
      (workspace && !aligned(workspace, 16)))
    return FA_ERR_INVALID_ARG;
  int* status = fa::current_status_word();
  if (!status) return FA_ERR_CUDA;
  const Plan pl = make_plan(B, Sq, Sk, Hq, Hkv, D, num_splits, device_sms());
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = workspace ? reinterpret_cast<float*>(static_cast<char*>(workspace) + pl.o_part_bytes) : nullptr;
  const long long sq[3] = {static_cast<long long>(Sq) * Hq * D, static_cast<long long>(Hq) * D, D};
  const long long skv[3] = {static_cast<long long>(Sk) * Hkv * D, static_cast<long long>(Hkv) * D, D};
  return fa::decode_launch(q, k, v, o, lse, B, Sq, Sk, Hq, Hkv, D, sq, skv, skv, sq, scale, causal, dtype, num_splits,
                           o_part, lse_part, workspace_bytes, reinterpret_cast<cudaStream_t>(stream_), status);
}
