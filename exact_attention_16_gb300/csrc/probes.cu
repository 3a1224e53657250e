// Single-tile probes of the hardware primitives the attention kernel is built
// on (TMA with 128-byte swizzle, tcgen05.mma with shared-memory and tensor-
// memory operands, tcgen05.ld/st), and a throughput probe of the MUFU ex2
// unit that sets the attention softmax's second roof. Test and measurement
// library: each tile probe runs one CTA on one 128-row tile so a failing
// primitive is isolated from the pipeline.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx_sm103.cuh"

namespace {

constexpr int kTile = 128 * 128 * 2;   // one 128 x 128 16-bit tile
constexpr int kChunk = 128 * 128;      // one 64-column swizzle chunk

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_rows(CUtensorMap* map, const void* ptr, bool bf16, int rows) {
  void* fnp = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return false;
  auto fn = reinterpret_cast<EncodeTiledFn>(fnp);
  // (rows, 128) row-major seen as 4-D (D=128, H=1, S=rows, B=1)
  const cuuint64_t dims[4] = {128, 1, static_cast<cuuint64_t>(rows), 1};
  const cuuint64_t strides[3] = {256, 256, static_cast<cuuint64_t>(rows) * 256};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
            const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ bool wait_bounded(uint32_t bar, uint32_t parity, int* err) {
  const uint64_t t0 = fa::ptx::globaltimer_ns();
  while (!fa::ptx::mbar_try_wait(bar, parity)) {
    if (fa::ptx::globaltimer_ns() - t0 > 1000000000ull) {
      atomicExch(err, 1);
      return false;
    }
  }
  return true;
}

// S = A B^T for 128x128 A and B (both K-major, 128-byte swizzle), fp32 out.
template <bool BF16>
__global__ void __launch_bounds__(128, 1) probe_qk_kernel(const __grid_constant__ CUtensorMap ta,
                                                          const __grid_constant__ CUtensorMap tb, float* out,
                                                          int* err) {
  extern __shared__ uint8_t raw[];
  const uint32_t raw_a = fa::ptx::smem_u32(raw);
  const uint32_t base = (raw_a + 1023u) & ~1023u;
  uint8_t* bp = raw + (base - raw_a);
  const uint32_t sA = base, sB = base + kTile, bar0 = base + 2 * kTile, bar1 = bar0 + 8;
  uint32_t* slot = reinterpret_cast<uint32_t*>(bp + 2 * kTile + 16);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    fa::ptx::mbar_init(bar0, 1);
    fa::ptx::mbar_init(bar1, 1);
    fa::ptx::fence_mbarrier_init();
  }
  if (warp == 0) {
    fa::ptx::tmem_alloc(fa::ptx::smem_u32(slot), 128);
    fa::ptx::tmem_relinquish();
  }
  fa::ptx::tc_fence_before();
  __syncthreads();
  fa::ptx::tc_fence_after();
  const uint32_t tmem = *slot;
  bool ok = true;
  if (threadIdx.x == 0) {
    const uint64_t pol = fa::ptx::policy_evict_first();
    fa::ptx::mbar_arrive_expect_tx(bar0, 2 * kTile);
    for (int c = 0; c < 2; ++c) {
      fa::ptx::tma_load_4d(sA + c * kChunk, &ta, bar0, c * 64, 0, 0, 0, pol);
      fa::ptx::tma_load_4d(sB + c * kChunk, &tb, bar0, c * 64, 0, 0, 0, pol);
    }
    ok = wait_bounded(bar0, 0, err);
    if (ok) {
      fa::ptx::tc_fence_after();
      constexpr uint32_t idesc = fa::ptx::idesc_f16(BF16, 128, 128, false, false);
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * kChunk + (ks % 4) * 32;
        fa::ptx::mma_ss(tmem, fa::ptx::sdesc_sw128(sA + off, 16, 1024), fa::ptx::sdesc_sw128(sB + off, 16, 1024),
                        idesc, ks > 0);
      }
    }
    fa::ptx::mma_commit(bar1);
  }
  __syncthreads();
  if (wait_bounded(bar1, 0, err)) {
    fa::ptx::tc_fence_after();
    uint32_t r[128];
    fa::ptx::tmem_ld_32x32b_x128(tmem + (static_cast<uint32_t>(warp * 32) << 16), r);
    const int row = threadIdx.x;
    for (int c = 0; c < 128; ++c) out[row * 128 + c] = __uint_as_float(r[c]);
  }
  fa::ptx::tc_fence_before();
  __syncthreads();
  fa::ptx::tc_fence_after();
  if (warp == 0) fa::ptx::tmem_dealloc(tmem, 128);
}

// O = P V for 128x128 P (given row-major in global, staged through TMEM as the
// A operand) and V (keys x 128, MN-major B operand via TMA), fp32 out.
template <bool BF16>
__global__ void __launch_bounds__(128, 1) probe_pv_kernel(const uint16_t* P, const __grid_constant__ CUtensorMap tv,
                                                          float* out, int* err) {
  extern __shared__ uint8_t raw[];
  const uint32_t raw_a = fa::ptx::smem_u32(raw);
  const uint32_t base = (raw_a + 1023u) & ~1023u;
  uint8_t* bp = raw + (base - raw_a);
  const uint32_t sV = base, bar0 = base + kTile, bar1 = bar0 + 8;
  uint32_t* slot = reinterpret_cast<uint32_t*>(bp + kTile + 16);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    fa::ptx::mbar_init(bar0, 1);
    fa::ptx::mbar_init(bar1, 1);
    fa::ptx::fence_mbarrier_init();
  }
  if (warp == 0) {
    fa::ptx::tmem_alloc(fa::ptx::smem_u32(slot), 256);
    fa::ptx::tmem_relinquish();
  }
  fa::ptx::tc_fence_before();
  __syncthreads();
  fa::ptx::tc_fence_after();
  const uint32_t tmem = *slot;
  if (threadIdx.x == 0) {
    fa::ptx::mbar_arrive_expect_tx(bar0, kTile);
    for (int c = 0; c < 2; ++c)
      fa::ptx::tma_load_4d(sV + c * kChunk, &tv, bar0, c * 64, 0, 0, 0, fa::ptx::policy_evict_first());
  }
  // each thread packs its row of P (keys 2c, 2c+1 -> column c) into TMEM
  {
    const int row = threadIdx.x;
    uint32_t pk[64];
    for (int c = 0; c < 64; ++c)
      pk[c] = static_cast<uint32_t>(P[row * 128 + 2 * c]) | (static_cast<uint32_t>(P[row * 128 + 2 * c + 1]) << 16);
    fa::ptx::tmem_st_32x32b_x64(tmem + (static_cast<uint32_t>(warp * 32) << 16), pk);
    fa::ptx::tmem_st_wait();
  }
  fa::ptx::tc_fence_before();
  __syncthreads();
  fa::ptx::tc_fence_after();
  if (threadIdx.x == 0) {
    if (wait_bounded(bar0, 0, err)) {
      constexpr uint32_t idesc = fa::ptx::idesc_f16(BF16, 128, 128, false, true);
      for (int ks = 0; ks < 8; ++ks)
        fa::ptx::mma_ts(tmem + 128, tmem + ks * 8, fa::ptx::sdesc_sw128(sV + ks * 16 * 128, kChunk, 1024), idesc,
                        ks > 0);
    }
    fa::ptx::mma_commit(bar1);
  }
  __syncthreads();
  if (wait_bounded(bar1, 0, err)) {
    fa::ptx::tc_fence_after();
    uint32_t r[128];
    fa::ptx::tmem_ld_32x32b_x128(tmem + 128 + (static_cast<uint32_t>(warp * 32) << 16), r);
    const int row = threadIdx.x;
    for (int c = 0; c < 128; ++c) out[row * 128 + c] = __uint_as_float(r[c]);
  }
  fa::ptx::tc_fence_before();
  __syncthreads();
  fa::ptx::tc_fence_after();
  if (warp == 0) fa::ptx::tmem_dealloc(tmem, 256);
}

template <typename K, typename... A>
int run(K kernel, int smem, cudaStream_t s, int* err, A... args) {
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 3;
  kernel<<<1, 128, smem, s>>>(args..., err);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace

// A, B: (128, 128) 16-bit row-major device arrays; out: (128, 128) fp32.
// err: device int set to 1 if a bounded wait ran out.
extern "C" int fa_probe_qk(const void* A, const void* B, float* out, int bf16, int* err, void* stream) {
  CUtensorMap ta, tb;
  if (!encode_rows(&ta, A, bf16, 128) || !encode_rows(&tb, B, bf16, 128)) return 3;
  auto s = reinterpret_cast<cudaStream_t>(stream);
  const int smem = 2 * kTile + 64 + 1024;
  return bf16 ? run(probe_qk_kernel<true>, smem, s, err, ta, tb, out)
              : run(probe_qk_kernel<false>, smem, s, err, ta, tb, out);
}

// P: (128, 128) 16-bit row-major (row = query, col = key); V: (128, 128)
// row-major (row = key, col = d); out: (128, 128) fp32.
extern "C" int fa_probe_pv(const void* P, const void* V, float* out, int bf16, int* err, void* stream) {
  CUtensorMap tv;
  if (!encode_rows(&tv, V, bf16, 128)) return 3;
  auto s = reinterpret_cast<cudaStream_t>(stream);
  const int smem = kTile + 64 + 1024;
  auto p = static_cast<const uint16_t*>(P);
  return bf16 ? run(probe_pv_kernel<true>, smem, s, err, p, tv, out)
              : run(probe_pv_kernel<false>, smem, s, err, p, tv, out);
}

namespace {

// Every thread runs 8 independent chains x <- 2^(-x) (values stay in
// (0.5, 1)), so the MUFU pipe, not the latency of one chain, bounds the time.
__global__ void __launch_bounds__(256) probe_ex2_kernel(int iters, float* sink) {
  float x[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = 0.5f + 0.01f * static_cast<float>(i + (threadIdx.x & 7));
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = fa::ptx::ex2_approx(-x[i]);
  }
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc += x[i];
  if (acc == 12345.0f) sink[0] = acc;   // keeps the chains live; never true
}

}  // namespace

// MUFU ex2 throughput of the current device: `blocks` x 256 threads x `iters`
// x 8 ex2.approx.ftz.f32 operations, timed with CUDA events on `stream`.
// *ex2_per_s receives the rate. Returns 0, or 3 on a CUDA error.
extern "C" int fa_probe_ex2_rate(int blocks, int iters, double* ex2_per_s, void* stream) {
  if (blocks <= 0 || iters <= 0 || !ex2_per_s) return 1;
  auto s = reinterpret_cast<cudaStream_t>(stream);
  float* sink = nullptr;
  cudaEvent_t e0, e1;
  if (cudaMalloc(&sink, sizeof(float)) != cudaSuccess) return 3;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    cudaFree(sink);
    return 3;
  }
  probe_ex2_kernel<<<blocks, 256, 0, s>>>(iters, sink);   // warm-up
  cudaEventRecord(e0, s);
  probe_ex2_kernel<<<blocks, 256, 0, s>>>(iters, sink);
  cudaEventRecord(e1, s);
  float ms = 0.0f;
  const bool ok = cudaEventSynchronize(e1) == cudaSuccess && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess &&
                  cudaGetLastError() == cudaSuccess && ms > 0.0f;
  if (ok) *ex2_per_s = static_cast<double>(blocks) * 256.0 * iters * 8.0 / (ms * 1e-3);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(sink);
  return ok ? 0 : 3;
}
