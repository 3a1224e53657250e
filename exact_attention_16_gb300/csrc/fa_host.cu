// fa_fwd_host: the forward pass for tensors that live in host memory. The
// caller gives host Q, K, V, O, LSE and one device workspace; the call splits
// the problem into chunks (batch ranges, or ranges of KV heads and query
// rows) and pipelines, per chunk, the host-to-device copy of its Q and of the
// K/V rows it newly needs, the attention kernel on it, and the device-to-host
// copy of its O and LSE. Copies run on two streams of the library (one per
// direction), kernels on the caller's stream and one more library stream in
// turn, so that copies in both directions overlap the kernels of other chunks
// and consecutive kernels overlap each other's tail. The device copy keeps
// the host layout; a chunk is a strided view of it, computed by
// fa_fwd_strided.
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
  cudaStream_t comp = nullptr;                 // kernels of every other chunk (the caller's stream runs the rest)
};
HostStreams g_streams[kMaxDevices];

HostStreams* streams_for(int dev) {
  HostStreams& h = g_streams[dev];
  std::call_once(h.once, [&] {
    h.err = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking);
    if (h.err == cudaSuccess) h.err = cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking);
    if (h.err == cudaSuccess) h.err = cudaStreamCreateWithFlags(&h.comp, cudaStreamNonBlocking);
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

// A chunk: batches [b0, b1) x query rows [r0, r1) x KV heads [h0, h1) (query
// heads [h0 G, h1 G)). Its kernel sees keys [0, lim); the chunk copies keys
// [k0, k1) of its batches and KV heads in (the keys the chunks of the same
// heads before it did not copy).
struct Chunk {
  int b0, b1, r0, r1, lim, k0, k1, h0, h1;
};

// Keys row i may see: all of them, or up to i + Sk - Sq (bottom-right mask).
long long visible(long long i, int Sq, int Sk, int causal) {
  if (!causal) return Sk;
  return std::max(0LL, std::min<long long>(Sk, i + Sk - Sq + 1));
}

// The chunk plan, at most one chunk per 24 MiB of copies (a small chunk's
// kernel leaves SMs idle and its copies are too short to hide anything):
//  * two or more batches: ranges of batches, each cut into up to four ranges
//    of KV heads while the size allows;
//  * one batch: up to four ranges of KV heads, each cut into up to two ranges
//    of query rows (at a 128-row tile). With a causal mask the first rows see
//    fewer keys, so the first row range copies only the keys it needs and the
//    second the rest.
// Timed end to end (GB300, pinned host tensors): on the 16K causal GQA
// workload (B = 1, 4 KV heads) heads x row halves beat chunks of rows only (1
// to 16 of them), of heads only, and finer cuts (1383 TFLOP/s against at most
// 1351); on B = 2, 8K, 8 KV heads, 2 batches x 4 head ranges gave 581 against
// 540 for 4 head ranges and 513 for 4 x 2 rows; on B = 4, 4K, 8 KV heads,
// 4 x 2 stays best (386; 4 x 4: 373, 2 x 4: 363).
int plan_chunks(int B, int Sq, int Sk, int Hkv, int causal, long long copy_bytes, Chunk* c) {
  const int by_size = static_cast<int>(std::max(1LL, std::min<long long>(kMaxChunks, copy_bytes / (24LL << 20))));
  if (B >= 2) {
    const int nb = std::min(B, by_size);
    const int nh = std::min({Hkv, 4, std::max(1, by_size / nb)});
    int n = 0;
    for (int i = 0; i < nb; ++i)
      for (int h = 0; h < nh; ++h)
        c[n++] = {B * i / nb, B * (i + 1) / nb, 0, Sq, Sk, 0, Sk, Hkv * h / nh, Hkv * (h + 1) / nh};
    return n;
  }
  const int nh = std::min({Hkv, 4, by_size});
  const int tiles = (Sq + 127) / 128;
  const int nr = std::min({2, tiles, std::max(1, by_size / nh)});
  int n = 0;
  for (int hi = 0; hi < nh; ++hi) {
    const int h0 = Hkv * hi / nh, h1 = Hkv * (hi + 1) / nh;
    int r0 = 0, kdone = 0;
    for (int i = 0; i < nr; ++i) {
      const int r1 = (i + 1 == nr) ? Sq : static_cast<int>(static_cast<long long>(tiles) * (i + 1) / nr) * 128;
      if (r1 <= r0) continue;
      const int lim = static_cast<int>(visible(r1 - 1, Sq, Sk, causal));
      const int k1 = std::max(kdone, lim);
      c[n++] = {0, B, r0, r1, lim, kdone, k1, h0, h1};
      kdone = k1;
      r0 = r1;
    }
  }
  return n;
}

// Copies the box (batches [b0, b1), rows [s0, s1), heads [h0, h1), D) of a
// (B, S, H, D) 16-bit tensor between host and device buffers of that layout:
// one block when the box is whole batches, else one 2-D copy per batch.
cudaError_t copy_box(void* dst, const void* src, int b0, int b1, int s0, int s1, int h0, int h1, int S, int H, int D,
                     cudaMemcpyKind kind, cudaStream_t s) {
  const size_t row = static_cast<size_t>(H) * D * 2;   // one (b, s) row
  if (s1 <= s0 || b1 <= b0 || h1 <= h0) return cudaSuccess;
  if (s0 == 0 && s1 == S && h0 == 0 && h1 == H) {
    const size_t off = static_cast<size_t>(b0) * S * row;
    return cudaMemcpyAsync(static_cast<char*>(dst) + off, static_cast<const char*>(src) + off,
                           static_cast<size_t>(b1 - b0) * S * row, kind, s);
  }
  for (int b = b0; b < b1; ++b) {
    const size_t off = (static_cast<size_t>(b) * S + s0) * row + static_cast<size_t>(h0) * D * 2;
    const cudaError_t e =
        cudaMemcpy2DAsync(static_cast<char*>(dst) + off, row, static_cast<const char*>(src) + off, row,
                          static_cast<size_t>(h1 - h0) * D * 2, s1 - s0, kind, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
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

extern "C" int fa_fwd_host_plan(int B, int Sq, int Sk, int Hq, int Hkv, int D, int causal, int* chunks, int cap,
                                int* n_chunks) {
  if (!n_chunks || (cap > 0 && !chunks) || cap < 0 || B <= 0 || Sq <= 0 || Sk < 0 || Hq <= 0 || Hkv <= 0 ||
      Hq % Hkv != 0 || D <= 0 || (causal != 0 && causal != 1))
    return FA_ERR_INVALID_ARG;
  Layout l;
  layout_of(B, Sq, Sk, Hq, Hkv, D, &l);
  Chunk ch[kMaxChunks];
  const int n = plan_chunks(B, Sq, Sk, Hkv, causal, l.q_bytes + 2 * l.kv_bytes + l.o_bytes + l.lse_bytes, ch);
  *n_chunks = n;
  for (int i = 0; i < n && i < cap; ++i) {
    const Chunk& x = ch[i];
    const int v[9] = {x.b0, x.b1, x.h0, x.h1, x.r0, x.r1, x.k0, x.k1, x.lim};
    for (int j = 0; j < 9; ++j) chunks[9 * i + j] = v[j];
  }
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
  Chunk ch[kMaxChunks];
  const int n = plan_chunks(B, Sq, Sk, Hkv, causal, l.q_bytes + 2 * l.kv_bytes + l.o_bytes + l.lse_bytes, ch);
  const int G = Hq / Hkv;

  // events: fork, join, per chunk (inputs landed, outputs computed)
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
              cudaStreamWaitEvent(hs->out, fork, 0) == cudaSuccess &&
              cudaStreamWaitEvent(hs->comp, fork, 0) == cudaSuccess;
    long long lse_at = 0;   // each chunk's LSE block is packed (B_c, Hq_c, rows_c) in the workspace
    for (int c = 0; ok && c < n; ++c) {
      const Chunk& x = ch[c];
      const int bc = x.b1 - x.b0, sq = x.r1 - x.r0, hk = x.h1 - x.h0, hq = hk * G;
      // Consecutive chunks' kernels alternate between two streams, so that
      // one chunk's last CTAs and the next chunk's first ones share the GPU.
      cudaStream_t cs = (c & 1) ? hs->comp : stream;
      cudaEvent_t in_done = ev[2 + 2 * c], out_ready = ev[3 + 2 * c];
      // copy in: the chunk's Q rows and the keys it newly needs
      const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
      ok = copy_box(dq, q, x.b0, x.b1, x.r0, x.r1, x.h0 * G, x.h1 * G, Sq, Hq, D, h2d, hs->in) == cudaSuccess &&
           copy_box(dk, k, x.b0, x.b1, x.k0, x.k1, x.h0, x.h1, Sk, Hkv, D, h2d, hs->in) == cudaSuccess &&
           copy_box(dv, v, x.b0, x.b1, x.k0, x.k1, x.h0, x.h1, Sk, Hkv, D, h2d, hs->in) == cudaSuccess &&
           cudaEventRecord(in_done, hs->in) == cudaSuccess && cudaStreamWaitEvent(cs, in_done, 0) == cudaSuccess;
      if (!ok) break;
      // the kernel on strided views of the device copy: rows [r0, r1) against
      // keys [0, lim), which keeps the bottom-right mask (lim - sq = r0 + Sk - Sq)
      const long long qo = ((static_cast<long long>(x.b0) * Sq + x.r0) * Hq + static_cast<long long>(x.h0) * G) * D * 2;
      const long long ko = (static_cast<long long>(x.b0) * Sk * Hkv + x.h0) * static_cast<long long>(D) * 2;
      float* lse_c = dlse + lse_at;
      rc = fa_fwd_strided(static_cast<char*>(dq) + qo, static_cast<char*>(dk) + ko, static_cast<char*>(dv) + ko,
                          static_cast<char*>(dout) + qo, lse ? lse_c : nullptr, bc, sq, x.lim, hq, hk, D, qs, ks, ks,
                          qs, scale, causal, dtype, cs);
      if (rc != FA_OK) break;
      ok = cudaEventRecord(out_ready, cs) == cudaSuccess && cudaStreamWaitEvent(hs->out, out_ready, 0) == cudaSuccess;
      // copy out: O rows, and the LSE block into its (B, Hq, Sq) place
      ok = ok && copy_box(o, dout, x.b0, x.b1, x.r0, x.r1, x.h0 * G, x.h1 * G, Sq, Hq, D, cudaMemcpyDeviceToHost,
                          hs->out) == cudaSuccess;
      for (int b = x.b0; ok && lse && b < x.b1; ++b) {
        const size_t width = static_cast<size_t>(sq) * 4;
        char* dst = reinterpret_cast<char*>(lse) + ((static_cast<size_t>(b) * Hq + static_cast<size_t>(x.h0) * G) * Sq + x.r0) * 4;
        const float* srcb = lse_c + static_cast<size_t>(b - x.b0) * hq * sq;
        ok = cudaMemcpy2DAsync(dst, static_cast<size_t>(Sq) * 4, srcb, width, width, hq, cudaMemcpyDeviceToHost,
                               hs->out) == cudaSuccess;
      }
      lse_at += static_cast<long long>(bc) * hq * sq;
    }
    // join: the caller's stream continues once every copy-out has finished
    const bool joined = cudaEventRecord(join, hs->out) == cudaSuccess && cudaStreamWaitEvent(stream, join, 0) == cudaSuccess;
    if (rc == FA_OK && (!ok || !joined)) rc = FA_ERR_CUDA;
  }
  for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);   // released once their work completes
  return rc;
}
