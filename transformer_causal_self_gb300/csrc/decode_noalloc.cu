// csattn_attn_decode_noalloc: KV-cache decode for callers that cannot
// allocate device memory.  The split partials that csattn_attn_decode writes
// to a caller-provided workspace go instead to a fixed buffer in static device
// memory, defined below.  The source pages have no counterpart of this: it is
// a property of the library's interface, not of the attention method.
//
// Who needs it: code that must not call cudaMalloc at decode time, for
// example a serving loop inside a framework that owns all device memory
// through its own pool and gives plugins no allocator, or a latency-critical
// step where cudaMalloc/cudaFree would synchronise the device or could fail
// with out-of-memory half-way through a batch.
#include <cstdio>
#include <mutex>
#include <string>

#include "csattn.h"
#include "internal.h"

namespace csattn {
namespace {

// The scratch.  In host code the symbol is only a stand-in for the device
// array; its device address comes from cudaGetSymbolAddress below.  The CUDA
// runtime loads this file's module (and with it reserves these bytes on the
// device) lazily by default: on the first cudaGetSymbolAddress or the first
// launch of one of its kernels on a device, i.e. on the first call of the entry
// point there.  From then on the device holds the bytes until the process exits.
constexpr size_t kStaticScratchBytes = CSATTN_DECODE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once per
// device (with that device current) and cached.
int scratch_address(void** out, const char** why) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *why = cudaGetErrorString(e);
    return CSATTN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *why = "device index out of range";
    return CSATTN_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      *why = e != cudaSuccess ? cudaGetErrorString(e) : "null symbol address";
      return CSATTN_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return CSATTN_OK;
}

}  // namespace
}  // namespace csattn

extern "C" int csattn_attn_decode_noalloc(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* seq_lens,
                                          void* out, int B, int Hq, int Hkv, int Lmax, int d,
                                          int dtype, float scale, int max_seq_len,
                                          int num_splits, void* stream) {
  const char* fn = "attn_decode_noalloc";
  // Every argument error is reported before the first CUDA call (the scratch
  // lookup below may load the module that holds the buffer).
  int rc = csattn::attn_decode_check_ptrs(fn, q, k_cache, v_cache, seq_lens, out, B, Hq, Hkv,
                                          Lmax, d, dtype, scale, max_seq_len, num_splits);
  if (rc != CSATTN_OK) return rc;
  if (num_splits > 0) {
    // the split count the decode will use for an explicit request (64-key multiples)
    const int per = (max_seq_len + num_splits - 1) / num_splits;
    const int chunk = ((per + 63) / 64) * 64;
    const size_t splits = static_cast<size_t>((max_seq_len + chunk - 1) / chunk);
    const size_t need = static_cast<size_t>(B) * Hq * splits * (static_cast<size_t>(d) + 2) * 4;
    if (need > csattn::kStaticScratchBytes) {
      char buf[200];
      snprintf(buf, sizeof(buf),
               "%s: the split partials need %zu bytes, more than the %zu-byte static scratch "
               "(fewer splits, or csattn_attn_decode with a workspace)",
               fn, need, csattn::kStaticScratchBytes);
      csattn::set_last_error(buf);
      return CSATTN_ERR_WORKSPACE;
    }
  }
  void* scratch = nullptr;
  const char* why = "";
  rc = csattn::scratch_address(&scratch, &why);
  if (rc != CSATTN_OK) {
    csattn::set_last_error((std::string(fn) + ": static scratch lookup: " + why).c_str());
    return rc;
  }
  // The decode kernels write every partial that the merge reads in the same
  // call, so nothing in the scratch has to start at zero.
  const int st = csattn_attn_decode(q, k_cache, v_cache, seq_lens, out, B, Hq, Hkv, Lmax, d,
                                    dtype, scale, max_seq_len, num_splits, scratch,
                                    csattn::kStaticScratchBytes, stream);
  if (st == CSATTN_ERR_WORKSPACE) {
    char buf[160];
    snprintf(buf, sizeof(buf),
             "%s: the split partials exceed the %zu-byte static scratch "
             "(fewer splits or csattn_attn_decode with a workspace); ",
             fn, csattn::kStaticScratchBytes);
    csattn::set_last_error((std::string(buf) + csattn_last_error()).c_str());
  }
  return st;
}
