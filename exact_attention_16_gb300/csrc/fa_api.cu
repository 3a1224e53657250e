// Host side of the C ABI declared in include/fa.h: argument validation, TMA
// tensor-map encoding, persistent-grid sizing and the launch on the caller's
// stream. Every step of the attention itself runs in fa_fwd_kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/fa.h"
#include "fa_fwd_kernel.cuh"

namespace fa {
int decode_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk, int Hq,
                  int Hkv, int D, const long long* qs, const long long* ks, const long long* vs, const long long* os,
                  float scale, int causal, int dtype, int num_splits, float* o_part, float* lse_part,
                  unsigned long long workspace_bytes, cudaStream_t stream, int* status_word);
int* current_status_word();
}  // namespace fa

namespace {

__device__ int g_fa_status = 0;

// Sk == 0: no key is visible, so O = 0 and LSE = -inf for every row. O rows
// are (b, s, h) with element strides sb, ss, sh; each row is vec16 x 16 bytes.
__global__ void fa_fill_empty_kernel(uint4* o, long long rows, int vec16, int Sq, int Hq, long long sb, long long ss,
                                     long long sh, float* lse, long long n_lse) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < rows * vec16; i += stride) {
    const long long r = i / vec16, c = i % vec16;
    const long long h = r % Hq, s = (r / Hq) % Sq, b = r / (static_cast<long long>(Hq) * Sq);
    o[(b * sb + s * ss + h * sh) / 8 + c] = make_uint4(0, 0, 0, 0);
  }
  if (lse)
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n_lse; i += stride)
      lse[i] = -__int_as_float(0x7f800000);
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  cudaError_t init_err = cudaSuccess;
  int num_sms = 0;
  int* status = nullptr;  // address of g_fa_status on this device
};
DeviceState g_dev[kMaxDevices];

std::atomic<int> g_fault_skip_load{-1};
std::atomic<int> g_fault_timeout_ms{0};
std::atomic<int> g_schedule_mode{-1};   // -1 cost model, 0 row-tile pairs, 1 key-split

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

template <int D, bool BF16, bool KSPLIT>
cudaError_t set_smem_attr() {
  static std::once_flag f[kMaxDevices];
  static cudaError_t err[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::call_once(f[dev], [&] {
    err[dev] = cudaFuncSetAttribute(fa::fa_fwd_kernel<D, BF16, KSPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    fa::Smem<D>::kAlloc);
  });
  return err[dev];
}

DeviceState* device_state(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceState& s = g_dev[dev];
  std::call_once(s.once, [&] {
    s.init_err = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (s.init_err == cudaSuccess)
      s.init_err = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.status), g_fa_status);
  });
  if (dev_out) *dev_out = dev;
  return s.init_err == cudaSuccess ? &s : nullptr;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 4-D map over a (B, S, H, D) tensor: dims innermost first (D, H, S, B); the
// box is 64 elements (128 bytes) x 1 head x `box_rows` rows x 1 batch,
// 128-byte swizzle, zero fill outside the tensor (loads) / clipping (stores).
bool encode_bshd(CUtensorMap* map, const void* ptr, bool bf16, int B, int S, int H, int D, const long long* st,
                 int box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(B)};
  // st = element strides of (b, s, h); the map wants byte strides of (h, s, b)
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2, static_cast<cuuint64_t>(st[1]) * 2,
                                 static_cast<cuuint64_t>(st[0]) * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

unsigned long long wait_timeout_ns() {
  const int fault_ms = g_fault_timeout_ms.load();
  if (fault_ms > 0) return static_cast<unsigned long long>(fault_ms) * 1000000ull;
  static const unsigned long long env_ns = [] {
    const char* e = std::getenv("FA_WAIT_TIMEOUT_MS");
    long long ms = e ? std::atoll(e) : 0;
    return static_cast<unsigned long long>(ms > 0 ? ms : 2000) * 1000000ull;
  }();
  return env_ns;
}

template <int D, bool BF16>
int launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
           const fa::FwdParams& p, bool ksplit, int grid, cudaStream_t stream) {
  if (ksplit) {
    if (set_smem_attr<D, BF16, true>() != cudaSuccess) return FA_ERR_CUDA;
    fa::fa_fwd_kernel<D, BF16, true><<<grid, fa::kThreads, fa::Smem<D>::kAlloc, stream>>>(tq, tk, tv, to, p);
  } else {
    if (set_smem_attr<D, BF16, false>() != cudaSuccess) return FA_ERR_CUDA;
    fa::fa_fwd_kernel<D, BF16, false><<<grid, fa::kThreads, fa::Smem<D>::kAlloc, stream>>>(tq, tk, tv, to, p);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Work items of each schedule: row-tile pairs (two heads of a GQA group, or
// two row tiles of one head) or key-split single row tiles.
void set_items(fa::FwdParams& p, bool ksplit) {
  p.pair_heads = (!ksplit && p.group % 2 == 0) ? 1 : 0;
  p.n_units = p.pair_heads ? p.Hq / 2 : p.Hq;
  p.n_mslots = (ksplit || p.pair_heads) ? p.n_mtiles : (p.n_mtiles + 1) / 2;
}

// Finishing time of the busiest CTA under the static serpentine schedule, in
// key-tile steps (one step = one key tile for both slots of a CTA). A key-split
// item of n key tiles takes ceil(n / 2) steps, each 1.125 times as long as a
// row-tile-pair step (every K/V tile feeds one slot instead of two, and the
// MMA thread waits for each slot's K/V itself); every item also pays 1.25
// steps of Q load, pipeline fill and epilogue. Both constants are fitted to
// GB300 timings of 18 shapes (MHA and GQA, causal and not, 0.5K to 32K keys),
// on which the model picks the faster schedule every time and predicts the
// time ratio within 9 %.
double schedule_makespan(const fa::FwdParams& p, bool ksplit, int grid) {
  constexpr double kItemOverhead = 1.25;
  constexpr double kSplitStep = 1.125;
  const int n_items = p.n_items;
  double worst = 0.0;
  for (int cta = 0; cta < grid; ++cta) {
    double t = 0.0;
    for (int round = 0; round * grid < n_items; ++round) {
      const int idx = fa::item_of_round(round, cta, grid);
      if (idx >= n_items) continue;
      const int n = ksplit ? fa::decode_item<true>(p, idx).n_kv : fa::decode_item<false>(p, idx).n_kv;
      if (n == 0) continue;
      t += (ksplit ? kSplitStep * ((n + 1) / 2) : n) + kItemOverhead;
    }
    worst = std::max(worst, t);
  }
  return worst;
}

// Picks key-split items when the row-tile pairs would leave SMs idle: too few
// items for the grid, or a long causal tail. Large problems (many waves) keep
// the pairs, whose shared K/V tiles halve the loads per MMA.
bool use_key_split(fa::FwdParams& p, int num_sms) {
  const int mode = g_schedule_mode.load();
  if (mode == 0 || mode == 1) return mode == 1;
  set_items(p, false);
  const long long pair_items = static_cast<long long>(p.B) * p.n_units * p.n_mslots;
  if (pair_items > 4LL * num_sms) return false;
  p.n_items = static_cast<int>(pair_items);
  const double t_pair = schedule_makespan(p, false, static_cast<int>(std::min<long long>(pair_items, num_sms)));
  set_items(p, true);
  const long long split_items = static_cast<long long>(p.B) * p.n_units * p.n_mslots;
  p.n_items = static_cast<int>(split_items);
  const double t_split = schedule_makespan(p, true, static_cast<int>(std::min<long long>(split_items, num_sms)));
  return t_split < t_pair;
}

}  // namespace

namespace {

// Checks one tensor's (b, s, h) element strides (d is contiguous) and
// replaces strides of size-1 dimensions, which are never used, by the
// contiguous ones so that the tensor map accepts them.
bool normalise_strides(const long long* in, long long* out, int B, int S, int H, int D) {
  const long long natural[3] = {static_cast<long long>(S) * H * D, static_cast<long long>(H) * D, D};
  const int sizes[3] = {B, S, H};
  for (int a = 0; a < 3; ++a) {
    long long st = in[a];
    if (sizes[a] <= 1) st = natural[a];
    if (st <= 0 || st % 8 != 0) return false;                  // 16-byte multiples for the tensor map
    if (static_cast<double>(st) * 2.0 >= 1099511627776.0) return false;
    out[a] = st;
  }
  return true;
}

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk, int Hq,
             int Hkv, int D, const long long* qs_in, const long long* ks_in, const long long* vs_in,
             const long long* os_in, float scale, int causal, int dtype, fa_stream_t stream_) {
  // ---- validation (nothing is enqueued on failure)
  if (B < 0 || Sq < 0 || Sk < 0 || Hq < 0 || Hkv < 0 || D < 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  // any finite scale, as long as scale * log2(e) is a finite float
  if (std::fabs(static_cast<double>(scale)) * 1.4426950408889634 > 3.4028234663852886e38)
    return FA_ERR_UNSUPPORTED;
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0 || Hq == 0) return FA_OK;
  if (D < 16 || D > 256 || D % 16 != 0) return FA_ERR_UNSUPPORTED;
  // the kernel's head dimension: the smallest of 64, 128, 256 that holds D;
  // tensor maps carry the true D, so the padding is zero-filled on load and
  // clipped on store
  const int Dk = D <= 64 ? 64 : (D <= 128 ? 128 : 256);
  if (Dk == 256 && Hq / Hkv > 128) return FA_ERR_UNSUPPORTED;
  if (!q || !o || (Sk > 0 && (!k || !v))) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || (Sk > 0 && (!aligned(k, 16) || !aligned(v, 16))) ||
      (lse && !aligned(lse, 4)))
    return FA_ERR_INVALID_ARG;
  long long qs[3], ks[3], vs[3], os[3];
  if (!normalise_strides(qs_in, qs, B, Sq, Hq, D) || !normalise_strides(os_in, os, B, Sq, Hq, D))
    return FA_ERR_INVALID_ARG;
  if (Sk > 0 && (!normalise_strides(ks_in, ks, B, Sk, Hkv, D) || !normalise_strides(vs_in, vs, B, Sk, Hkv, D)))
    return FA_ERR_INVALID_ARG;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  DeviceState* ds = device_state(nullptr);
  if (!ds) return FA_ERR_CUDA;

  if (Sk == 0) {
    const long long rows = static_cast<long long>(B) * Sq * Hq;
    const long long n_lse = static_cast<long long>(B) * Hq * Sq;
    fa_fill_empty_kernel<<<ds->num_sms * 4, 256, 0, stream>>>(static_cast<uint4*>(o), rows, D / 8, Sq, Hq, os[0],
                                                                os[1], os[2], lse, n_lse);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }

  if (Dk == 256) {
    // Two 128-row tiles with D = 256 accumulators do not fit tensor memory:
    // the one-tile split-KV kernel runs with a single key range (no workspace).
    int* status = fa::current_status_word();
    if (!status) return FA_ERR_CUDA;
    return fa::decode_launch(q, k, v, o, lse, B, Sq, Sk, Hq, Hkv, D, qs, ks, vs, os, scale, causal, dtype, 1, nullptr,
                             nullptr, 0, stream, status);
  }

  fa::FwdParams p{};
  p.o = o;
  p.o_sb = os[0];
  p.o_ss = os[1];
  p.o_sh = os[2];
  p.d_true = D;
  p.lse = lse;
  p.B = B;
  p.Sq = Sq;
  p.Sk = Sk;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = Hq / Hkv;
  p.causal = causal;
  // A zero scale makes every visible score 0: it runs as scale 1 on Q read as
  // zeros (the same scores, exactly), so that the kernels always have a
  // nonzero scale to rank scores by.
  p.scale_log2 = static_cast<float>(static_cast<double>(scale == 0.0f ? 1.0f : scale) * 1.4426950408889634);
  p.q_b_shift = scale == 0.0f ? B : 0;
  p.n_mtiles = (Sq + fa::kBM - 1) / fa::kBM;
  p.n_kv_tiles = (Sk + fa::kBN - 1) / fa::kBN;
  // every item count below fits an int: B * Hq * ceil(Sq / 128) does
  if (static_cast<long long>(B) * Hq * p.n_mtiles > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const bool ksplit = use_key_split(p, ds->num_sms);
  set_items(p, ksplit);
  const long long items = static_cast<long long>(B) * p.n_units * p.n_mslots;
  p.n_items = static_cast<int>(items);
  p.timeout_ns = wait_timeout_ns();
  p.inject_skip_load = g_fault_skip_load.load();
  p.status = ds->status;

  const bool bf16 = dtype == FA_DTYPE_BF16;
  CUtensorMap tq, tk, tv, to;
  if (!encode_bshd(&tq, q, bf16, B, Sq, Hq, D, qs) || !encode_bshd(&tk, k, bf16, B, Sk, Hkv, D, ks) ||
      !encode_bshd(&tv, v, bf16, B, Sk, Hkv, D, vs) || !encode_bshd(&to, o, bf16, B, Sq, Hq, D, os, 32))
    return FA_ERR_CUDA;

  const int grid = static_cast<int>(std::min<long long>(items, ds->num_sms));
  if (Dk == 128) {
    return bf16 ? launch<128, true>(tq, tk, tv, to, p, ksplit, grid, stream)
                : launch<128, false>(tq, tk, tv, to, p, ksplit, grid, stream);
  }
  return bf16 ? launch<64, true>(tq, tk, tv, to, p, ksplit, grid, stream)
              : launch<64, false>(tq, tk, tv, to, p, ksplit, grid, stream);
}

}  // namespace

namespace fa {
int* current_status_word() {
  DeviceState* ds = device_state(nullptr);
  return ds ? ds->status : nullptr;
}
}  // namespace fa

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk,
                      int Hq, int Hkv, int D, float scale, int causal, int dtype, fa_stream_t stream) {
  const long long sq[3] = {static_cast<long long>(Sq) * Hq * D, static_cast<long long>(Hq) * D, D};
  const long long skv[3] = {static_cast<long long>(Sk) * Hkv * D, static_cast<long long>(Hkv) * D, D};
  return fwd_impl(q, k, v, o, lse, B, Sq, Sk, Hq, Hkv, D, sq, skv, skv, sq, scale, causal, dtype, stream);
}

extern "C" int fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq,
                              int Sk, int Hq, int Hkv, int D, const long long* q_strides,
                              const long long* k_strides, const long long* v_strides,
                              const long long* o_strides, float scale, int causal, int dtype,
                              fa_stream_t stream) {
  if (!q_strides || !k_strides || !v_strides || !o_strides) return FA_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, Sq, Sk, Hq, Hkv, D, q_strides, k_strides, v_strides, o_strides, scale, causal,
                  dtype, stream);
}

extern "C" int fa_status(fa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  DeviceState* ds = device_state(nullptr);
  if (!ds) return FA_ERR_CUDA;
  int value = 0, zero = 0;
  if (cudaMemcpy(&value, ds->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpy(ds->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  return value;
}

extern "C" const char* fa_status_string(int code) {
  switch (code) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

extern "C" int fa_version(void) { return 100; }

extern "C" int fa_fwd_schedule(int B, int Sq, int Sk, int Hq, int Hkv, int causal, int num_sms, int* key_split) {
  if (!key_split || B <= 0 || Sq <= 0 || Sk <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_sms <= 0 ||
      (causal != 0 && causal != 1))
    return FA_ERR_INVALID_ARG;
  fa::FwdParams p{};
  p.B = B;
  p.Sq = Sq;
  p.Sk = Sk;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = Hq / Hkv;
  p.causal = causal;
  p.n_mtiles = (Sq + fa::kBM - 1) / fa::kBM;
  p.n_kv_tiles = (Sk + fa::kBN - 1) / fa::kBN;
  if (static_cast<long long>(B) * Hq * p.n_mtiles > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  *key_split = use_key_split(p, num_sms) ? 1 : 0;
  return FA_OK;
}

extern "C" int fa_fwd_work_items(int B, int Sq, int Sk, int Hq, int Hkv, int causal, int key_split, int num_sms,
                                 int* items, int cap, int* n_items, int* grid) {
  if (!n_items || !grid || (cap > 0 && !items) || cap < 0 || B <= 0 || Sq <= 0 || Sk <= 0 || Hq <= 0 || Hkv <= 0 ||
      Hq % Hkv != 0 || num_sms <= 0 || (causal != 0 && causal != 1) || (key_split != 0 && key_split != 1))
    return FA_ERR_INVALID_ARG;
  fa::FwdParams p{};
  p.B = B;
  p.Sq = Sq;
  p.Sk = Sk;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.group = Hq / Hkv;
  p.causal = causal;
  p.n_mtiles = (Sq + fa::kBM - 1) / fa::kBM;
  p.n_kv_tiles = (Sk + fa::kBN - 1) / fa::kBN;
  if (static_cast<long long>(B) * Hq * p.n_mtiles > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  set_items(p, key_split == 1);
  p.n_items = static_cast<int>(static_cast<long long>(B) * p.n_units * p.n_mslots);
  const int g = std::min(p.n_items, num_sms);
  *n_items = p.n_items;
  *grid = g;
  const int n = std::min(p.n_items, cap);
  for (int idx = 0; idx < n; ++idx) {
    const fa::WorkItem w = key_split ? fa::decode_item<true>(p, idx) : fa::decode_item<false>(p, idx);
    int* it = items + 8LL * idx;
    it[0] = w.b;
    it[1] = w.hq0;
    it[2] = w.hq1;
    it[3] = w.kvh;
    it[4] = w.r0;
    it[5] = w.r1;
    it[6] = w.n_kv;
    it[7] = -1;
  }
  // the CTA that runs each item: the kernel's loop over rounds
  for (int round = 0; static_cast<long long>(round) * g < p.n_items; ++round)
    for (int cta = 0; cta < g; ++cta) {
      const int idx = fa::item_of_round(round, cta, g);
      if (idx < n) items[8LL * idx + 7] = cta;
    }
  return FA_OK;
}

extern "C" int fa_debug_set_schedule(int mode) {
  if (mode < -1 || mode > 1) return FA_ERR_INVALID_ARG;
  g_schedule_mode.store(mode);
  return FA_OK;
}

extern "C" int fa_debug_set_fault(int skip_load, int timeout_ms) {
  if (skip_load < -1) return FA_ERR_INVALID_ARG;
  g_fault_skip_load.store(skip_load);
  g_fault_timeout_ms.store(skip_load >= 0 ? timeout_ms : 0);
  return FA_OK;
}
