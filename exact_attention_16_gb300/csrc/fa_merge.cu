// Merge of attention outputs computed over disjoint key sets (context-parallel
// shards or split-KV partials): LSE = ln sum_r e^{LSE_r}, O = sum_r
// e^{LSE_r - LSE} O_r. This is the online-softmax rescale of "MiniPaged-Qwen:
// Qwen3 Prefill FlashAttention" section 4 applied to whole partial states.
// Memory bound: each thread folds eight elements of one row over the parts
// with 16-byte streaming loads and fp32 accumulation.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>

#include "../../include/fa.h"
#include "fa_merge.cuh"

namespace fa {
namespace {

// Raw 16-byte chunks of a part and their conversion to fp32 (eight 16-bit
// elements, or four fp32 elements, per chunk).
template <typename T>
struct Chunk {
  static constexpr int kElems = 16 / sizeof(T);
  __device__ static uint4 load(const T* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
  __device__ static void to_float(const uint4& v, float* x);
};
template <>
__device__ void Chunk<float>::to_float(const uint4& v, float* x) {
  x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y); x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
}
template <>
__device__ void Chunk<__nv_bfloat16>::to_float(const uint4& v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    x[2 * q] = __uint_as_float(w[q] << 16);
    x[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
  }
}
template <>
__device__ void Chunk<__half>::to_float(const uint4& v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
    x[2 * q] = f.x;
    x[2 * q + 1] = f.y;
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&a);
  } else {
    const __half2 a = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&a);
  }
}

// o_parts: (n, B, Sq, Hq, D) of TP; lse_parts: (n, B, Hq, Sq) fp32;
// o: (B, Sq, Hq, D) 16-bit; lse: (B, Hq, Sq) fp32 or null. Each thread owns
// kE consecutive elements of one row and folds the parts in groups of kGroup
// (loads of a group in flight together) with a running max (the
// online-softmax rescale). Few rows and many parts (decode of one or a few
// sequences split over the whole GPU) take kE = 4 and a deep group: four
// times the threads, and fewer dependent round trips per thread.
template <typename TP, bool OUT_BF16, typename IDX, int kE, int kGroup>
__global__ void __launch_bounds__(256, 3) merge_kernel(const TP* __restrict__ o_parts,
                                                    const float* __restrict__ lse_parts, int n_parts,
                                                    void* __restrict__ o, float* __restrict__ lse, IDX rows, IDX Sq,
                                                    IDX Hq, IDX D) {
  // Launched right behind the split-KV kernel that writes the parts, this
  // grid may start before that one has finished: wait for it (and for its
  // writes to be visible). Without a programmatic launch this returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kChunks = kE / Chunk<TP>::kElems;           // 16-byte loads per part
  static_assert(kChunks >= 1 && kE % 4 == 0, "a thread loads whole 16-byte chunks");
  const IDX per_row = D / kE;
  const IDX items = rows * per_row;
  const long long part_o = static_cast<long long>(rows) * D;
  const IDX stride = static_cast<IDX>(gridDim.x) * blockDim.x;
  for (IDX it = blockIdx.x * static_cast<IDX>(blockDim.x) + threadIdx.x; it < items; it += stride) {
    const IDX row = it / per_row;
    const IDX e = (it - row * per_row) * kE;
    const IDX bs = row / Hq, h = row - bs * Hq;        // row = (b * Sq + s) * Hq + h
    const IDX b = bs / Sq, s = bs - b * Sq;
    const IDX li = (b * Hq + h) * Sq + s;
    float m = -INFINITY, tot = 0.0f, acc[kE];
#pragma unroll
    for (int q = 0; q < kE; ++q) acc[q] = 0.0f;
    for (int r0 = 0; r0 < n_parts; r0 += kGroup) {
      float lr[kGroup];
      uint4 raw[kGroup][kChunks];
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const int r = r0 + g;
        lr[g] = (r < n_parts) ? __ldg(lse_parts + static_cast<long long>(r) * rows + li) : -INFINITY;
        const TP* src = o_parts + r * part_o + static_cast<long long>(row) * D + e;
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          raw[g][c] = (r < n_parts) ? Chunk<TP>::load(src + c * Chunk<TP>::kElems) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        if (!(lr[g] > -INFINITY)) continue;
        const float m_new = fmaxf(m, lr[g]);
        const float c = expf(m - m_new);          // 0 while m = -inf
        const float wgt = expf(lr[g] - m_new);
        tot = tot * c + wgt;
#pragma unroll
        for (int ch = 0; ch < kChunks; ++ch) {
          float x[Chunk<TP>::kElems];
          Chunk<TP>::to_float(raw[g][ch], x);
#pragma unroll
          for (int q = 0; q < Chunk<TP>::kElems; ++q) {
            float& a = acc[ch * Chunk<TP>::kElems + q];
            a = fmaf(wgt, x[q], a * c);
          }
        }
        m = m_new;
      }
    }
    const bool live = m > -INFINITY;
    const float inv = live ? 1.0f / tot : 0.0f;
    uint32_t w[kE / 2];
#pragma unroll
    for (int q = 0; q < kE / 2; ++q) w[q] = pack2<OUT_BF16>(acc[2 * q] * inv, acc[2 * q + 1] * inv);
    uint16_t* dst = static_cast<uint16_t*>(o) + static_cast<long long>(row) * D + e;
    if constexpr (kE == 4) {
      __stcs(reinterpret_cast<uint2*>(dst), make_uint2(w[0], w[1]));
    } else {
#pragma unroll
      for (int q = 0; q < kE / 8; ++q)
        __stcs(reinterpret_cast<uint4*>(dst) + q, make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
    }
    if (lse && e == 0) lse[li] = live ? m + logf(tot) : -INFINITY;
  }
}

// `after_producer`: launched with programmatic stream serialization, so that
// its CTAs are scheduled while the kernel before it (which signals
// griddepcontrol.launch_dependents) still runs; merge_kernel's first
// instruction waits for that kernel's completion.
template <typename TP, bool OUT_BF16, int kE, int kGroup>
int launch_merge_e(const TP* o_parts, const float* lse_parts, int n, void* o, float* lse, long long rows, int Sq,
                   int Hq, int D, int sms, cudaStream_t stream, bool after_producer) {
  const long long items = rows * (D / kE);
  const long long blocks_needed = (items + 255) / 256;
  const int blocks = static_cast<int>(blocks_needed < 32LL * sms ? blocks_needed : 32LL * sms);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = after_producer ? 1 : 0;
  cudaError_t e;
  if (rows * D + 256LL * blocks < 0x7fffffffLL)   // every index (and the loop bound) fits 32 bits
    e = cudaLaunchKernelEx(&cfg, merge_kernel<TP, OUT_BF16, unsigned, kE, kGroup>, o_parts, lse_parts, n, o, lse,
                           static_cast<unsigned>(rows), static_cast<unsigned>(Sq), static_cast<unsigned>(Hq),
                           static_cast<unsigned>(D));
  else
    e = cudaLaunchKernelEx(&cfg, merge_kernel<TP, OUT_BF16, long long, kE, kGroup>, o_parts, lse_parts, n, o, lse,
                           rows, static_cast<long long>(Sq), static_cast<long long>(Hq), static_cast<long long>(D));
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// `after_producer`: launched with programmatic stream serialization, so that
// its CTAs are scheduled while the kernel before it (which signals
// griddepcontrol.launch_dependents) still runs; merge_kernel's first
// instruction waits for that kernel's completion.
template <typename TP, bool OUT_BF16>
int launch_merge(const TP* o_parts, const float* lse_parts, int n, void* o, float* lse, long long rows, int Sq,
                 int Hq, int D, cudaStream_t stream, bool after_producer = false) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return FA_ERR_CUDA;
  // fp32 parts with fewer 16-element items than one 256-thread block per SM:
  // four elements per thread, eight parts in flight
  if constexpr (sizeof(TP) == 4) {
    if (rows * (D / 16) < 256LL * sms)
      return launch_merge_e<TP, OUT_BF16, 4, 8>(o_parts, lse_parts, n, o, lse, rows, Sq, Hq, D, sms, stream,
                                                after_producer);
  }
  return launch_merge_e<TP, OUT_BF16, 16, sizeof(TP) == 4 ? 2 : 4>(o_parts, lse_parts, n, o, lse, rows, Sq, Hq, D,
                                                                   sms, stream, after_producer);
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

int merge_f32_parts(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int B, int Sq,
                    int Hq, int D, int dtype, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * Sq * Hq;
  if (rows == 0) return FA_OK;
  return dtype == FA_DTYPE_BF16
             ? launch_merge<float, true>(o_parts, lse_parts, n_parts, o, lse, rows, Sq, Hq, D, stream, true)
             : launch_merge<float, false>(o_parts, lse_parts, n_parts, o, lse, rows, Sq, Hq, D, stream, true);
}

}  // namespace fa

extern "C" int fa_merge(const void* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int B, int Sq,
                        int Hq, int D, int dtype, fa_stream_t stream_) {
  if (n_parts < 1 || B < 0 || Sq < 0 || Hq < 0 || D < 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (D % 16 != 0 || D > 1024) return FA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(B) * Sq * Hq;
  if (rows == 0 || D == 0) return FA_OK;
  if (!o_parts || !lse_parts || !o) return FA_ERR_INVALID_ARG;
  if (!fa::aligned_to(o_parts, 16) || !fa::aligned_to(o, 16) || !fa::aligned_to(lse_parts, 4) ||
      (lse && !fa::aligned_to(lse, 4)))
    return FA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (dtype == FA_DTYPE_BF16)
    return fa::launch_merge<__nv_bfloat16, true>(static_cast<const __nv_bfloat16*>(o_parts), lse_parts, n_parts, o,
                                                 lse, rows, Sq, Hq, D, stream);
  return fa::launch_merge<__half, false>(static_cast<const __half*>(o_parts), lse_parts, n_parts, o, lse, rows, Sq, Hq,
                                         D, stream);
}
