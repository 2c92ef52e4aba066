// Prefill from host buffers (csattn_attn_fwd_host): the inputs cross the host link,
// the attention runs, and the output crosses back, pipelined over chunks of
// (sequence, KV head) pairs on three streams per device: host-to-device copies,
// kernels, device-to-host copies.  The copies of one chunk overlap the kernels of
// its neighbours, and the two copy directions overlap each other.
//
// A (sequence b, KV head g) pair owns query heads g*rep .. g*rep+rep-1 of sequence b
// (rep = Hq / Hkv) and nothing else, so consecutive pairs are contiguous in every
// [B, H, T, d] tensor and a chunk of pairs is an attention problem of its own with
// B' = pairs, Hq' = rep, Hkv' = 1 (the grouped-query mapping of "The Transformer
// architecture", section "What else the modern decoder-only model changed").  Each
// chunk's kernel computes exactly what the whole problem's kernel computes for
// those heads.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "csattn.h"
#include "internal.h"

namespace csattn {
namespace {

constexpr int kMaxChunks = 16;
constexpr int kDefaultChunks = 16;
constexpr int kMaxDev = 64;

int hfail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int hfail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  set_last_error(buf);
  return code;
}

int hfail_cuda(cudaError_t e, const char* what) {
  return hfail(CSATTN_ERR_CUDA, "attn_fwd_host: %s: %s (%s)", what, cudaGetErrorName(e),
               cudaGetErrorString(e));
}

// Streams and events of one device, created on first use and kept for the process.
struct Pipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, cmp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in[kMaxChunks] = {};
  cudaEvent_t done[kMaxChunks] = {};
};

// Held for a whole call's enqueue: two threads sharing a device's pipe must not
// interleave their event records and waits.
std::mutex g_pipe_mu;
Pipe g_pipe[kMaxDev];

int pipe_of_device(Pipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return hfail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDev) return hfail(CSATTN_ERR_UNSUPPORTED, "attn_fwd_host: device %d", dev);
  Pipe& p = g_pipe[dev];
  if (!p.ready) {
    const unsigned sf = cudaStreamNonBlocking;
    const unsigned ef = cudaEventDisableTiming;
    if ((e = cudaStreamCreateWithFlags(&p.h2d, sf)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&p.cmp, sf)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&p.d2h, sf)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&p.start, ef)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&p.end, ef)) != cudaSuccess)
      return hfail_cuda(e, "stream/event creation");
    for (int c = 0; c < kMaxChunks; ++c)
      if ((e = cudaEventCreateWithFlags(&p.in[c], ef)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&p.done[c], ef)) != cudaSuccess)
        return hfail_cuda(e, "event creation");
    p.ready = true;
  }
  *out = &p;
  return CSATTN_OK;
}

// After a failure part-way through a call's enqueue: the caller's stream still waits
// for everything already enqueued on the internal streams (so the buffers stay in use
// until that work is done, as after a successful call), and the error code is returned.
int abandon(Pipe& p, cudaStream_t caller, int rc) {
  for (cudaStream_t s : {p.h2d, p.cmp, p.d2h})
    if (cudaEventRecord(p.end, s) == cudaSuccess) (void)cudaStreamWaitEvent(caller, p.end, 0);
  return rc;
}

size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t elem_size(int dtype) {
  return dtype == CSATTN_BF16 ? 2 : (dtype == CSATTN_F32 ? 4 : 0);
}

}  // namespace
}  // namespace csattn

using namespace csattn;

extern "C" {

size_t csattn_fwd_host_workspace_size(int B, int Hq, int Hkv, int T, int d, int dtype,
                                      float rope_base) {
  const size_t esz = elem_size(dtype);
  if (esz == 0 || B < 1 || Hq < 1 || Hkv < 1 || T < 1 || d < 1) return 0;
  const size_t qb = static_cast<size_t>(B) * Hq * T * d * esz;
  const size_t kb = static_cast<size_t>(B) * Hkv * T * d * esz;
  size_t bytes = al256(qb) + 2 * al256(kb) + al256(qb);    // q, k, v, out
  bytes += al256(static_cast<size_t>(B) * Hq * T * 4);      // lse
  bytes += al256(csattn_fwd_workspace_size(B, Hq, Hkv, T, d, dtype, rope_base));  // rotated k
  return bytes;
}

int csattn_attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* out_h, int B,
                         int Hq, int Hkv, int T, int d, int dtype, int causal, float rope_base,
                         int rope_layout, float scale, float* lse_h, int num_chunks,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (q_h == nullptr || k_h == nullptr || v_h == nullptr || out_h == nullptr)
    return hfail(CSATTN_ERR_INVALID_ARG, "attn_fwd_host: q, k, v and out must be non-null");
  if (B < 1 || Hq < 1 || Hkv < 1 || T < 1)
    return hfail(CSATTN_ERR_INVALID_ARG, "attn_fwd_host: B=%d Hq=%d Hkv=%d T=%d must be >= 1",
                 B, Hq, Hkv, T);
  if (Hq % Hkv != 0)
    return hfail(CSATTN_ERR_INVALID_ARG, "attn_fwd_host: Hq=%d is not a multiple of Hkv=%d", Hq,
                 Hkv);
  const size_t esz = elem_size(dtype);
  if (esz == 0) return hfail(CSATTN_ERR_INVALID_ARG, "attn_fwd_host: unknown dtype %d", dtype);
  if (num_chunks < 0 || num_chunks > kMaxChunks)
    return hfail(CSATTN_ERR_INVALID_ARG, "attn_fwd_host: num_chunks=%d not in [0, %d]",
                 num_chunks, kMaxChunks);
  const size_t need = csattn_fwd_host_workspace_size(B, Hq, Hkv, T, d, dtype, rope_base);
  if (workspace == nullptr || need == 0 || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
    return hfail(CSATTN_ERR_WORKSPACE,
                 "attn_fwd_host: needs a 16-byte aligned workspace of %zu bytes (got %zu)", need,
                 workspace_bytes);
  const int rep = Hq / Hkv;
  const int pairs = B * Hkv;
  int n = num_chunks > 0 ? num_chunks : kDefaultChunks;
  if (n > pairs) n = pairs;
  // every argument the kernels check, checked before any copy is enqueued (each chunk is
  // the same problem with fewer sequences)
  {
    const int rc = attn_fwd_check("attn_fwd_host", B, Hq, Hkv, T, d, dtype, causal, rope_base,
                                  rope_layout, scale);
    if (rc != CSATTN_OK) return rc;
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t qb = static_cast<size_t>(B) * Hq * T * d * esz;
  const size_t kb = static_cast<size_t>(B) * Hkv * T * d * esz;
  uint8_t* dq = ws;
  uint8_t* dk = dq + al256(qb);
  uint8_t* dv = dk + al256(kb);
  uint8_t* dout = dv + al256(kb);
  float* dlse = reinterpret_cast<float*>(dout + al256(qb));
  uint8_t* dkrot = reinterpret_cast<uint8_t*>(dlse) + al256(static_cast<size_t>(B) * Hq * T * 4);

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  Pipe* pp = nullptr;
  int rc = pipe_of_device(&pp);
  if (rc != CSATTN_OK) return rc;
  Pipe& p = *pp;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((e = cudaEventRecord(p.start, caller)) != cudaSuccess) return hfail_cuda(e, "event record");
  for (cudaStream_t s : {p.h2d, p.cmp, p.d2h})
    if ((e = cudaStreamWaitEvent(s, p.start, 0)) != cudaSuccess)
      return abandon(p, caller, hfail_cuda(e, "stream wait"));
  const size_t q_pair = static_cast<size_t>(rep) * T * d * esz;  // bytes of q (or out) per pair
  const size_t k_pair = static_cast<size_t>(T) * d * esz;        // bytes of k (or v) per pair
  const size_t l_pair = static_cast<size_t>(rep) * T * 4;        // bytes of lse per pair
  for (int c = 0; c < n; ++c) {
    const int i0 = static_cast<int>(static_cast<long long>(pairs) * c / n);
    const int i1 = static_cast<int>(static_cast<long long>(pairs) * (c + 1) / n);
    const int np = i1 - i0;
    const size_t qo = q_pair * i0, qs = q_pair * np;
    const size_t ko = k_pair * i0, ks = k_pair * np;
    const size_t lo = l_pair * i0, ls = l_pair * np;
    if ((e = cudaMemcpyAsync(dq + qo, static_cast<const uint8_t*>(q_h) + qo, qs,
                             cudaMemcpyHostToDevice, p.h2d)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dk + ko, static_cast<const uint8_t*>(k_h) + ko, ks,
                             cudaMemcpyHostToDevice, p.h2d)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dv + ko, static_cast<const uint8_t*>(v_h) + ko, ks,
                             cudaMemcpyHostToDevice, p.h2d)) != cudaSuccess ||
        (e = cudaEventRecord(p.in[c], p.h2d)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(p.cmp, p.in[c], 0)) != cudaSuccess)
      return abandon(p, caller, hfail_cuda(e, "host-to-device copy"));
    const size_t wsz = csattn_fwd_workspace_size(np, rep, 1, T, d, dtype, rope_base);
    rc = csattn_attn_fwd(dq + qo, dk + ko, dv + ko, dout + qo, np, rep, 1, T, d, dtype, causal,
                         rope_base, rope_layout, scale, lse_h != nullptr ? dlse + lo / 4 : nullptr,
                         wsz > 0 ? dkrot + ko : nullptr, wsz, p.cmp);
    if (rc != CSATTN_OK) return abandon(p, caller, rc);
    if ((e = cudaEventRecord(p.done[c], p.cmp)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(p.d2h, p.done[c], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(static_cast<uint8_t*>(out_h) + qo, dout + qo, qs,
                             cudaMemcpyDeviceToHost, p.d2h)) != cudaSuccess)
      return abandon(p, caller, hfail_cuda(e, "device-to-host copy"));
    if (lse_h != nullptr &&
        (e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse_h) + lo,
                             reinterpret_cast<uint8_t*>(dlse) + lo, ls, cudaMemcpyDeviceToHost,
                             p.d2h)) != cudaSuccess)
      return abandon(p, caller, hfail_cuda(e, "device-to-host copy (lse)"));
  }
  if ((e = cudaEventRecord(p.end, p.d2h)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(caller, p.end, 0)) != cudaSuccess)
    return abandon(p, caller, hfail_cuda(e, "final wait"));
  return CSATTN_OK;
}

size_t csattn_decode_host_workspace_size(int B, int Hq, int Hkv, int Lmax, int d,
                                         int num_splits) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || d < 1 || num_splits < 0) return 0;
  const size_t qb = static_cast<size_t>(B) * Hq * d * 2;
  const size_t cb = static_cast<size_t>(B) * Hkv * Lmax * d * 2;
  return al256(qb) + 2 * al256(cb) + al256(static_cast<size_t>(B) * 4) + al256(qb) +
         al256(csattn_decode_workspace_size(B, Hq, Lmax, d, num_splits));
}

int csattn_attn_decode_host(const void* q_h, const void* k_cache_h, const void* v_cache_h,
                            const int32_t* seq_lens_h, void* out_h, int B, int Hq, int Hkv,
                            int Lmax, int d, int dtype, float scale, int num_splits,
                            int num_chunks, void* workspace, size_t workspace_bytes,
                            void* stream) {
  const char* fn = "attn_decode_host";
  if (q_h == nullptr || k_cache_h == nullptr || v_cache_h == nullptr || seq_lens_h == nullptr ||
      out_h == nullptr)
    return hfail(CSATTN_ERR_INVALID_ARG, "%s: null pointer argument", fn);
  if (B < 1 || Lmax < 1)
    return hfail(CSATTN_ERR_INVALID_ARG, "%s: B=%d Lmax=%d must be >= 1", fn, B, Lmax);
  if (num_chunks < 0 || num_chunks > kMaxChunks)
    return hfail(CSATTN_ERR_INVALID_ARG, "%s: num_chunks=%d not in [0, %d]", fn, num_chunks,
                 kMaxChunks);
  // the lengths are read here, on the host, so they are checked here too
  int max_len = 0;
  for (int b = 0; b < B; ++b) {
    const int L = seq_lens_h[b];
    if (L < 1 || L > Lmax)
      return hfail(CSATTN_ERR_INVALID_ARG, "%s: seq_lens[%d]=%d not in [1, Lmax=%d]", fn, b, L,
                   Lmax);
    if (L > max_len) max_len = L;
  }
  int rc = attn_decode_check(fn, B, Hq, Hkv, Lmax, d, dtype, scale, max_len, num_splits);
  if (rc != CSATTN_OK) return rc;
  const size_t need = csattn_decode_host_workspace_size(B, Hq, Hkv, Lmax, d, num_splits);
  if (workspace == nullptr || need == 0 || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
    return hfail(CSATTN_ERR_WORKSPACE, "%s: needs a 16-byte aligned workspace of %zu bytes (got %zu)",
                 fn, need, workspace_bytes);
  const size_t esz = 2;
  const size_t q_seq = static_cast<size_t>(Hq) * d * esz;          // q (or out) bytes per sequence
  const size_t row = static_cast<size_t>(d) * esz;                  // one cache row
  const size_t c_head = static_cast<size_t>(Lmax) * row;            // one head's cache
  const size_t c_seq = static_cast<size_t>(Hkv) * c_head;           // one sequence's cache
  uint8_t* dq = static_cast<uint8_t*>(workspace);
  uint8_t* dk = dq + al256(q_seq * B);
  uint8_t* dv = dk + al256(c_seq * B);
  int32_t* dlens = reinterpret_cast<int32_t*>(dv + al256(c_seq * B));
  uint8_t* dout = reinterpret_cast<uint8_t*>(dlens) + al256(static_cast<size_t>(B) * 4);
  uint8_t* dpart = dout + al256(q_seq * B);
  const size_t part_bytes = csattn_decode_workspace_size(B, Hq, Lmax, d, num_splits);
  int n = num_chunks > 0 ? num_chunks : 4;
  if (n > B) n = B;

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  Pipe* pp = nullptr;
  rc = pipe_of_device(&pp);
  if (rc != CSATTN_OK) return rc;
  Pipe& p = *pp;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((e = cudaEventRecord(p.start, caller)) != cudaSuccess) return hfail_cuda(e, "event record");
  for (cudaStream_t s : {p.h2d, p.cmp, p.d2h})
    if ((e = cudaStreamWaitEvent(s, p.start, 0)) != cudaSuccess)
      return abandon(p, caller, hfail_cuda(e, "stream wait"));
  for (int c = 0; c < n; ++c) {
    const int b0 = static_cast<int>(static_cast<long long>(B) * c / n);
    const int b1 = static_cast<int>(static_cast<long long>(B) * (c + 1) / n);
    const int nb = b1 - b0;
    int chunk_max = 0;
    if ((e = cudaMemcpyAsync(dq + q_seq * b0, static_cast<const uint8_t*>(q_h) + q_seq * b0,
                             q_seq * nb, cudaMemcpyHostToDevice, p.h2d)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dlens + b0, seq_lens_h + b0, static_cast<size_t>(nb) * 4,
                             cudaMemcpyHostToDevice, p.h2d)) != cudaSuccess)
      return abandon(p, caller, hfail_cuda(e, "host-to-device copy"));
    // only the rows the decode reads: rows 0..L_b-1 of every KV head of sequence b
    for (int b = b0; b < b1; ++b) {
      const int L = seq_lens_h[b];
      if (L > chunk_max) chunk_max = L;
      const size_t off = c_seq * b;
      if ((e = cudaMemcpy2DAsync(dk + off, c_head, static_cast<const uint8_t*>(k_cache_h) + off,
                                 c_head, row * L, Hkv, cudaMemcpyHostToDevice, p.h2d)) !=
              cudaSuccess ||
          (e = cudaMemcpy2DAsync(dv + off, c_head, static_cast<const uint8_t*>(v_cache_h) + off,
                                 c_head, row * L, Hkv, cudaMemcpyHostToDevice, p.h2d)) !=
              cudaSuccess)
        return abandon(p, caller, hfail_cuda(e, "host-to-device copy (cache rows)"));
    }
    if ((e = cudaEventRecord(p.in[c], p.h2d)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(p.cmp, p.in[c], 0)) != cudaSuccess)
      return abandon(p, caller, hfail_cuda(e, "event"));
    rc = csattn_attn_decode(dq + q_seq * b0, dk + c_seq * b0, dv + c_seq * b0, dlens + b0,
                            dout + q_seq * b0, nb, Hq, Hkv, Lmax, d, dtype, scale, chunk_max,
                            num_splits, dpart, part_bytes, p.cmp);
    if (rc != CSATTN_OK) return abandon(p, caller, rc);
    if ((e = cudaEventRecord(p.done[c], p.cmp)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(p.d2h, p.done[c], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(static_cast<uint8_t*>(out_h) + q_seq * b0, dout + q_seq * b0,
                             q_seq * nb, cudaMemcpyDeviceToHost, p.d2h)) != cudaSuccess)
      return abandon(p, caller, hfail_cuda(e, "device-to-host copy"));
  }
  if ((e = cudaEventRecord(p.end, p.d2h)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(caller, p.end, 0)) != cudaSuccess)
    return abandon(p, caller, hfail_cuda(e, "final wait"));
  return CSATTN_OK;
}

}  // extern "C"
