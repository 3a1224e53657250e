// fa_fwd_host: the forward pass for tensors that live in host memory. The
// caller gives host Q, K, V, O, LSE and one device workspace; the call splits
// the problem into chunks (batch ranges, or ranges of KV heads with their
// query heads) and pipelines, per chunk, the host-to-device copy of its Q, K
// and V, the attention kernel on it, and the device-to-host copy of its O and
// LSE, on two copy streams of the library's and the caller's stream, so that
// copies in both directions overlap the kernels of other chunks. The device copy keeps the host layout; a chunk is
// a strided view of it, computed by fa_fwd_strided.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 8;

struct HostStreams {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  cudaStream_t in = nullptr, out = nullptr;   // copy-in and copy-out streams of this device
};
HostStreams g_streams[kMaxDevices];

HostStreams* streams_for(int dev) {
  HostStreams& h = g_streams[dev];
  std::call_once(h.once, [&] {
    h.err = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking);
    if (h.err == cudaSuccess) h.err = cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking);
  });
  return h.err == cudaSuccess ? &h : nullptr;
}

struct Layout {
  long long q_bytes, kv_bytes, o_bytes, lse_bytes;
};

bool layout_of(int B, int Sq, int Sk, int Hq, int Hkv, int D, Layout* l) {
  const long long e = 2;
  l->q_bytes = static_cast<long long>(B) * Sq * Hq * D * e;
  l->kv_bytes = static_cast<long long>(B) * Sk * Hkv * D * e;
  l->o_bytes = l->q_bytes;
  l->lse_bytes = static_cast<long long>(B) * Hq * Sq * 4;
  return true;
}

// 256-byte aligned offsets of q, k, v, o, lse inside the workspace.
void offsets(const Layout& l, unsigned long long off[5], unsigned long long* total) {
  const unsigned long long sizes[5] = {static_cast<unsigned long long>(l.q_bytes),
                                       static_cast<unsigned long long>(l.kv_bytes),
                                       static_cast<unsigned long long>(l.kv_bytes),
                                       static_cast<unsigned long long>(l.o_bytes),
                                       static_cast<unsigned long long>(l.lse_bytes)};
  unsigned long long at = 0;
  for (int i = 0; i < 5; ++i) {
    off[i] = at;
    at += (sizes[i] + 255ull) & ~255ull;
  }
  *total = at;
}

// A chunk: batches [b0, b1) x KV heads [h0, h1) (query heads [h0 G, h1 G)).
struct Chunk {
  int b0, b1, h0, h1;
};

// Up to four chunks of nearly equal size, over batches when there are enough
// of them, else over KV heads (all batches at once); one chunk per 48 MiB of
// copies at most, since a small chunk's kernel leaves SMs idle and its copies
// are too short to hide anything.
int plan_chunks(int B, int Hkv, long long copy_bytes, Chunk* c) {
  const int by_size = static_cast<int>(std::max(1LL, std::min<long long>(4, copy_bytes / (48LL << 20))));
  if (B >= 2) {
    const int n = std::min({B, kMaxChunks / 2, by_size});
    for (int i = 0; i < n; ++i) c[i] = {B * i / n, B * (i + 1) / n, 0, Hkv};
    return n;
  }
  const int n = std::min({Hkv, kMaxChunks / 2, by_size});
  for (int i = 0; i < n; ++i) c[i] = {0, B, Hkv * i / n, Hkv * (i + 1) / n};
  return n;
}

// Copies the box (batches [b0, b1), rows [0, S), heads [h0, h1), D) of a
// (B, S, H, D) 16-bit tensor between host and device buffers of that layout.
cudaError_t copy_bshd(void* dst, const void* src, int b0, int b1, int S, int H, int h0, int h1, int D,
                      cudaMemcpyKind kind, cudaStream_t s) {
  const size_t row = static_cast<size_t>(H) * D * 2;                      // one (b, s) row
  const size_t off = (static_cast<size_t>(b0) * S) * row + static_cast<size_t>(h0) * D * 2;
  const size_t width = static_cast<size_t>(h1 - h0) * D * 2;
  const size_t rows = static_cast<size_t>(b1 - b0) * S;
  if (rows == 0 || width == 0) return cudaSuccess;
  if (width == row)
    return cudaMemcpyAsync(static_cast<char*>(dst) + off, static_cast<const char*>(src) + off, rows * row, kind, s);
  return cudaMemcpy2DAsync(static_cast<char*>(dst) + off, row, static_cast<const char*>(src) + off, row, width, rows,
                           kind, s);
}

}  // namespace

extern "C" int fa_fwd_host_workspace_size(int B, int Sq, int Sk, int Hq, int Hkv, int D,
                                          unsigned long long* bytes) {
  if (!bytes || B < 0 || Sq < 0 || Sk < 0 || Hq < 0 || Hkv < 0 || D < 0) return FA_ERR_INVALID_ARG;
  Layout l;
  layout_of(B, Sq, Sk, Hq, Hkv, D, &l);
  unsigned long long off[5];
  offsets(l, off, bytes);
  return FA_OK;
}

extern "C" int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk,
                           int Hq, int Hkv, int D, float scale, int causal, int dtype, void* workspace,
                           unsigned long long workspace_bytes, fa_stream_t stream_) {
  if (B < 0 || Sq < 0 || Sk < 0 || Hq < 0 || Hkv < 0 || D < 0) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0 || Hq == 0) return FA_OK;
  if (D < 16 || D > 256 || D % 16 != 0) return FA_ERR_UNSUPPORTED;
  if (!q || !o || (Sk > 0 && (!k || !v))) return FA_ERR_INVALID_ARG;
  Layout l;
  layout_of(B, Sq, Sk, Hq, Hkv, D, &l);
  unsigned long long off[5], need = 0;
  offsets(l, off, &need);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  HostStreams* hs = streams_for(dev);
  if (!hs) return FA_ERR_CUDA;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  char* ws = static_cast<char*>(workspace);
  void* dq = ws + off[0];
  void* dk = ws + off[1];
  void* dv = ws + off[2];
  void* dout = ws + off[3];
  float* dlse = reinterpret_cast<float*>(ws + off[4]);
  const int G = Hq / Hkv;
  Chunk ch[kMaxChunks];
  const int n = plan_chunks(B, Hkv, l.q_bytes + 2 * l.kv_bytes + l.o_bytes + l.lse_bytes, ch);

  // events: fork, per chunk (inputs landed, outputs computed), join
  cudaEvent_t ev[2 + 2 * kMaxChunks];
  int n_ev = 0;
  int rc = FA_OK;
  for (; n_ev < 2 + 2 * n; ++n_ev)
    if (cudaEventCreateWithFlags(&ev[n_ev], cudaEventDisableTiming) != cudaSuccess) {
      rc = FA_ERR_CUDA;
      break;
    }
  if (rc == FA_OK) {
    cudaEvent_t fork = ev[0], join = ev[1];
    const long long qs[3] = {static_cast<long long>(Sq) * Hq * D, static_cast<long long>(Hq) * D, D};
    const long long ks[3] = {static_cast<long long>(Sk) * Hkv * D, static_cast<long long>(Hkv) * D, D};
    bool ok = cudaEventRecord(fork, stream) == cudaSuccess && cudaStreamWaitEvent(hs->in, fork, 0) == cudaSuccess &&
              cudaStreamWaitEvent(hs->out, fork, 0) == cudaSuccess;
    long long lse_at = 0;   // chunk LSE blocks are packed (B_c, Hq_c, Sq) in the workspace
    for (int c = 0; ok && c < n; ++c) {
      const Chunk& x = ch[c];
      const int bc = x.b1 - x.b0, hk = x.h1 - x.h0, hq = hk * G;
      cudaEvent_t in_done = ev[2 + 2 * c], out_ready = ev[3 + 2 * c];
      // copy in
      ok = copy_bshd(dq, q, x.b0, x.b1, Sq, Hq, x.h0 * G, x.h1 * G, D, cudaMemcpyHostToDevice, hs->in) ==
               cudaSuccess &&
           (Sk == 0 ||
            (copy_bshd(dk, k, x.b0, x.b1, Sk, Hkv, x.h0, x.h1, D, cudaMemcpyHostToDevice, hs->in) == cudaSuccess &&
             copy_bshd(dv, v, x.b0, x.b1, Sk, Hkv, x.h0, x.h1, D, cudaMemcpyHostToDevice, hs->in) == cudaSuccess)) &&
           cudaEventRecord(in_done, hs->in) == cudaSuccess && cudaStreamWaitEvent(stream, in_done, 0) == cudaSuccess;
      if (!ok) break;
      // compute the chunk: strided views into the device copy
      const long long qo = (static_cast<long long>(x.b0) * Sq * Hq + static_cast<long long>(x.h0) * G) * D * 2;
      const long long ko = (static_cast<long long>(x.b0) * Sk * Hkv + x.h0) * static_cast<long long>(D) * 2;
      float* lse_c = dlse + lse_at;
      rc = fa_fwd_strided(static_cast<char*>(dq) + qo, static_cast<char*>(dk) + ko, static_cast<char*>(dv) + ko,
                          static_cast<char*>(dout) + qo, lse ? lse_c : nullptr, bc, Sq, Sk, hq, hk, D, qs, ks, ks, qs,
                          scale, causal, dtype, stream);
      if (rc != FA_OK) break;
      ok = cudaEventRecord(out_ready, stream) == cudaSuccess && cudaStreamWaitEvent(hs->out, out_ready, 0) == cudaSuccess;
      // copy out
      ok = ok && copy_bshd(o, dout, x.b0, x.b1, Sq, Hq, x.h0 * G, x.h1 * G, D, cudaMemcpyDeviceToHost, hs->out) ==
                     cudaSuccess;
      if (ok && lse) {
        const size_t width = static_cast<size_t>(hq) * Sq * 4, pitch = static_cast<size_t>(Hq) * Sq * 4;
        char* dst = reinterpret_cast<char*>(lse) + static_cast<size_t>(x.b0) * pitch +
                    static_cast<size_t>(x.h0) * G * Sq * 4;
        ok = cudaMemcpy2DAsync(dst, pitch, lse_c, width, width, bc, cudaMemcpyDeviceToHost, hs->out) == cudaSuccess;
      }
      lse_at += static_cast<long long>(bc) * hq * Sq;
    }
    // join: the caller's stream continues once every copy-out has finished
    const bool joined = cudaEventRecord(join, hs->out) == cudaSuccess && cudaStreamWaitEvent(stream, join, 0) == cudaSuccess;
    if (rc == FA_OK && (!ok || !joined)) rc = FA_ERR_CUDA;
  }
  for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);   // released once their work completes
  return rc;
}
