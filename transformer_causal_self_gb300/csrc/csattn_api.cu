// C ABI of libcsattn: argument checks, the per-device status word, TMA
// descriptor encoding, and dispatch to the kernels.  See include/csattn.h for
// the contract of every entry point.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "csattn.h"
#include "internal.h"

namespace csattn {

// One status word per device (a static device variable exists once on every
// device that loads the library).  Kernels OR bits into it; csattn_check_status
// reads and clears it.
__device__ uint32_t g_status_word;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(CSATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Device address of the status word and the SM count of the current device.
int device_info(uint32_t** status, int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(CSATTN_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_status_word);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(status word)");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
    g_status_ptr[dev] = static_cast<uint32_t*>(ptr);
    g_num_sms[dev] = sms;
  }
  *status = g_status_ptr[dev];
  *num_sms = g_num_sms[dev];
  return CSATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Page sizes of the paged caches: 16 or 32 rows (one TMA box per page), or a
// multiple of 64 rows up to 65536 (boxes of 64 or 128 rows inside a page).
bool valid_page_size(int page_size) {
  return page_size == 16 || page_size == 32 ||
         (page_size >= 64 && page_size % 64 == 0 && page_size <= 65536);
}

// theta_p = base^(-2p/d), p < d/2, split into float hi + lo (hi + lo = theta
// to about 2^-48 relative).
void rope_table(RopeTable* t, int d, double base) {
  std::memset(t, 0, sizeof(*t));
  for (int p = 0; p < d / 2 && p < 64; ++p) {
    const double th = std::pow(base, -2.0 * p / static_cast<double>(d));
    const float hi = static_cast<float>(th);
    t->hi[p] = hi;
    t->lo[p] = static_cast<float>(th - static_cast<double>(hi));
  }
}

// Largest position whose angle the kernels' Cody-Waite reduction keeps exact
// (|k| < 2^13 multiples of 2 pi for theta_0 = 1).
constexpr int kMaxRopePositions = 49152;

}  // namespace

void set_last_error(const char* msg) { g_last_error = msg; }

void* tensor_map_encoder() {
  static void* fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return p;
  }();
  return fn;
}

bool make_tmap_bf16_3d(void* tmap_out, const void* base, int d, int rows, int planes,
                       int box_rows) {
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (encode == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = encode(static_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                      const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace csattn

using namespace csattn;

extern "C" {

const char* csattn_last_error(void) { return g_last_error.c_str(); }

const char* csattn_status_str(int status) {
  switch (status) {
    case CSATTN_OK: return "CSATTN_OK";
    case CSATTN_ERR_INVALID_ARG: return "CSATTN_ERR_INVALID_ARG";
    case CSATTN_ERR_UNSUPPORTED: return "CSATTN_ERR_UNSUPPORTED";
    case CSATTN_ERR_CUDA: return "CSATTN_ERR_CUDA";
    case CSATTN_ERR_TIMEOUT: return "CSATTN_ERR_TIMEOUT";
    case CSATTN_ERR_WORKSPACE: return "CSATTN_ERR_WORKSPACE";
    case CSATTN_ERR_DEVICE_ARG: return "CSATTN_ERR_DEVICE_ARG";
    default: return "CSATTN_UNKNOWN_STATUS";
  }
}

int csattn_version(void) { return 100; }

size_t csattn_fwd_workspace_size(int B, int Hq, int Hkv, int T, int d, int dtype,
                                 float rope_base) {
  return csattn_fwd_ext_workspace_size(B, Hq, Hkv, T, T, d, dtype, rope_base);
}

size_t csattn_fwd_ext_workspace_size(int B, int Hq, int Hkv, int Tq, int Tk, int d, int dtype,
                                     float rope_base) {
  (void)Hq;
  (void)Tq;
  if (dtype != CSATTN_BF16 || !(rope_base > 0.f) || B < 1 || Hkv < 1 || Tk < 1 || d < 1) return 0;
  return static_cast<size_t>(B) * Hkv * Tk * d * 2;
}

}  // extern "C"

namespace {

// Shared by csattn_attn_fwd (Tq = Tk = T, q_offset = 0) and csattn_attn_fwd_ext.
// check_only: stop after the argument checks (the workspace is not checked) and return OK.
int attn_fwd_impl(const char* fn, const void* q, const void* k, const void* v, void* out, int B,
                  int Hq, int Hkv, int Tq, int Tk, int q_offset, int d, int dv, int dtype,
                  int causal, float rope_base, int rope_layout, float scale, float* lse,
                  void* workspace, size_t workspace_bytes, void* stream,
                  bool check_only = false) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: q, k, v and out must be non-null", fn);
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: B=%d Hq=%d Hkv=%d Tq=%d Tk=%d must be >= 1", fn, B,
                Hq, Hkv, Tq, Tk);
  if (q_offset < 0) return fail(CSATTN_ERR_INVALID_ARG, "%s: q_offset=%d < 0", fn, q_offset);
  if (Hq % Hkv != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: Hq=%d is not a multiple of Hkv=%d", fn, Hq, Hkv);
  if (dtype != CSATTN_F32 && dtype != CSATTN_BF16)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, dtype);
  if (causal != 0 && causal != 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: causal must be 0 or 1", fn);
  const bool k_prerotated = (rope_layout & CSATTN_ROPE_K_PREROTATED) != 0;
  rope_layout &= ~CSATTN_ROPE_K_PREROTATED;
  if (rope_layout != CSATTN_ROPE_SPLIT_HALF && rope_layout != CSATTN_ROPE_ADJACENT)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: unknown rope_layout %d", fn, rope_layout);
  if (!std::isfinite(rope_base) || !std::isfinite(scale))
    return fail(CSATTN_ERR_INVALID_ARG, "%s: rope_base and scale must be finite", fn);
  if (d != 16 && d != 32 && d != 64 && d != 128)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: d=%d not in {16,32,64,128}", fn, d);
  if (dv != 16 && dv != 32 && dv != 64 && dv != 128)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: dv=%d not in {16,32,64,128}", fn, dv);
  if (dtype == CSATTN_BF16 && ((d != 64 && d != 128) || (dv != 64 && dv != 128)))
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: bf16 supports d, dv in {64,128}, got %d, %d", fn, d,
                dv);
  if (Tq >= (1 << 24) || Tk >= (1 << 24) || q_offset >= (1 << 24))
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: Tq=%d, Tk=%d and q_offset=%d must be < 2^24", fn, Tq,
                Tk, q_offset);
  if (rope_base > 0.f && (q_offset + Tq > kMaxRopePositions || Tk > kMaxRopePositions))
    return fail(CSATTN_ERR_UNSUPPORTED,
                "%s: RoPE supports positions < %d (q_offset + Tq = %d, Tk = %d)", fn,
                kMaxRopePositions, q_offset + Tq, Tk);
  if (static_cast<long long>(B) * Hq > (1LL << 31) - 1)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: B*Hq too large", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(CSATTN_ERR_INVALID_ARG, "%s: q, k, v, out must be 16-byte aligned", fn);
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: lse must be 4-byte aligned", fn);
  if (check_only) return CSATTN_OK;
  const size_t need =
      k_prerotated ? 0 : csattn_fwd_ext_workspace_size(B, Hq, Hkv, Tq, Tk, d, dtype, rope_base);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return fail(CSATTN_ERR_WORKSPACE,
                "%s: needs a 16-byte aligned workspace of %zu bytes (got %zu)", fn, need,
                workspace_bytes);

  FwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Tq = Tq;
  a.Tk = Tk;
  a.q_off = q_offset;
  a.d = d;
  a.dv = dv;
  a.causal = causal;
  a.rope = rope_base > 0.f ? (rope_layout == CSATTN_ROPE_SPLIT_HALF ? 1 : 2) : 0;
  a.rope_k = (a.rope != 0 && !k_prerotated) ? 1 : 0;
  a.scale = scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  if (a.rope) rope_table(&a.theta, d, static_cast<double>(rope_base));
  int rc = device_info(&a.status, &a.num_sms);
  if (rc != CSATTN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  cudaError_t e;
  if (dtype == CSATTN_F32) {
    e = launch_fwd_f32(a, st);
    if (e != cudaSuccess) return fail_cuda(e, "attn_fwd: fp32 kernel launch");
    return CSATTN_OK;
  }
  if (tensor_map_encoder() == nullptr)
    return fail(CSATTN_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", fn);
  const void* k_eff = k;
  if (a.rope_k) {
    e = launch_rope_rotate_bf16(k, workspace, B, Hkv, Tk, d, a.rope, a.theta, st);
    if (e != cudaSuccess) return fail_cuda(e, "attn_fwd: RoPE kernel launch");
    k_eff = workspace;
  }
  e = launch_fwd_sm103a(a, k_eff, st);
  if (e != cudaSuccess) return fail_cuda(e, "attn_fwd: sm_103a kernel launch");
  return CSATTN_OK;
}

}  // namespace

int csattn::attn_fwd_check(const char* fn, int B, int Hq, int Hkv, int T, int d, int dtype,
                           int causal, float rope_base, int rope_layout, float scale) {
  alignas(16) static const uint8_t dummy[16] = {};
  void* x = const_cast<uint8_t*>(dummy);
  return attn_fwd_impl(fn, x, x, x, x, B, Hq, Hkv, T, T, 0, d, d, dtype, causal, rope_base,
                       rope_layout, scale, nullptr, nullptr, 0, nullptr, true);
}

extern "C" {

int csattn_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                    int Hkv, int T, int d, int dtype, int causal, float rope_base,
                    int rope_layout, float scale, float* lse, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return attn_fwd_impl("attn_fwd", q, k, v, out, B, Hq, Hkv, T, T, 0, d, d, dtype, causal,
                       rope_base, rope_layout, scale, lse, workspace, workspace_bytes, stream);
}

int csattn_attn_fwd_ext(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                        int Hkv, int Tq, int Tk, int q_offset, int d, int dv, int dtype,
                        int causal, float rope_base, int rope_layout, float scale, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return attn_fwd_impl("attn_fwd_ext", q, k, v, out, B, Hq, Hkv, Tq, Tk, q_offset, d,
                       dv > 0 ? dv : d, dtype, causal, rope_base, rope_layout, scale, lse,
                       workspace, workspace_bytes, stream);
}

size_t csattn_bwd_workspace_size(int B, int Hq, int Hkv, int T, int d, int dtype,
                                 float rope_base) {
  return csattn_bwd_ext_workspace_size(B, Hq, Hkv, T, T, d, dtype, rope_base);
}

size_t csattn_bwd_ext_workspace_size(int B, int Hq, int Hkv, int Tq, int Tk, int d, int dtype,
                                     float rope_base) {
  if ((dtype != CSATTN_BF16 && dtype != CSATTN_F32) || B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 ||
      Tk < 1 || d < 1)
    return 0;
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t rows = static_cast<size_t>(B) * Hq * Tq;
  const size_t esz = dtype == CSATTN_F32 ? 4 : 2;
  size_t bytes = al(rows * 4);  // rowsum(dout o out), fp32
  if (rope_base > 0.f)          // rotated q and k
    bytes += al(rows * d * esz) + al(static_cast<size_t>(B) * Hkv * Tk * d * esz);
  return bytes;
}

}  // extern "C"

namespace {

// Shared by csattn_attn_bwd (Tq = Tk = T, q_offset = 0, dv = d) and csattn_attn_bwd_ext.
int attn_bwd_impl(const char* fn, const void* q, const void* k, const void* v, const void* out,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int Hq,
                  int Hkv, int Tq, int Tk, int q_offset, int d, int d_v, int dtype, int causal,
                  float rope_base, int rope_layout, float scale, void* workspace,
                  size_t workspace_bytes, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || dout == nullptr ||
      lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: null pointer argument", fn);
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: B=%d Hq=%d Hkv=%d Tq=%d Tk=%d must be >= 1", fn, B,
                Hq, Hkv, Tq, Tk);
  if (q_offset < 0) return fail(CSATTN_ERR_INVALID_ARG, "%s: q_offset=%d < 0", fn, q_offset);
  if (Hq % Hkv != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: Hq=%d is not a multiple of Hkv=%d", fn, Hq, Hkv);
  if (dtype != CSATTN_BF16 && dtype != CSATTN_F32)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, dtype);
  if (causal != 0 && causal != 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: causal must be 0 or 1", fn);
  if ((rope_layout & CSATTN_ROPE_K_PREROTATED) != 0)
    return fail(CSATTN_ERR_UNSUPPORTED,
                "%s: the backward takes k unrotated (CSATTN_ROPE_K_PREROTATED is not accepted)",
                fn);
  if (rope_layout != CSATTN_ROPE_SPLIT_HALF && rope_layout != CSATTN_ROPE_ADJACENT)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: unknown rope_layout %d", fn, rope_layout);
  if (!std::isfinite(rope_base) || !std::isfinite(scale))
    return fail(CSATTN_ERR_INVALID_ARG, "%s: rope_base and scale must be finite", fn);
  auto width_ok = [&](int w) {
    return dtype == CSATTN_BF16 ? (w == 64 || w == 128) : (w == 16 || w == 32 || w == 64 || w == 128);
  };
  if (!width_ok(d) || !width_ok(d_v))
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: %s d=%d, dv=%d not in %s", fn,
                dtype == CSATTN_BF16 ? "bf16" : "fp32", d, d_v,
                dtype == CSATTN_BF16 ? "{64,128}" : "{16,32,64,128}");
  if (Tq >= (1 << 24) || Tk >= (1 << 24) || q_offset >= (1 << 24))
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: Tq=%d, Tk=%d and q_offset=%d must be < 2^24", fn, Tq,
                Tk, q_offset);
  if (rope_base > 0.f && (q_offset + Tq > kMaxRopePositions || Tk > kMaxRopePositions))
    return fail(CSATTN_ERR_UNSUPPORTED,
                "%s: RoPE supports positions < %d (q_offset + Tq = %d, Tk = %d)", fn,
                kMaxRopePositions, q_offset + Tq, Tk);
  if (static_cast<long long>(B) * Hq > (1LL << 31) - 1)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: B*Hq too large", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  const size_t need = csattn_bwd_ext_workspace_size(B, Hq, Hkv, Tq, Tk, d, dtype, rope_base);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return fail(CSATTN_ERR_WORKSPACE,
                "%s: needs a 16-byte aligned workspace of %zu bytes (got %zu)", fn, need,
                workspace_bytes);
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t rows = static_cast<size_t>(B) * Hq * Tq;
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  BwdArgs a{};
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.dvec = reinterpret_cast<float*>(ws);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Tq = Tq;
  a.Tk = Tk;
  a.q_off = q_offset;
  a.d = d;
  a.d_v = d_v;
  a.causal = causal;
  a.rope = rope_base > 0.f ? (rope_layout == CSATTN_ROPE_SPLIT_HALF ? 1 : 2) : 0;
  a.scale = scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  if (a.rope) rope_table(&a.theta, d, static_cast<double>(rope_base));
  uint32_t* status = nullptr;
  int num_sms = 0;
  int rc = device_info(&status, &num_sms);
  if (rc != CSATTN_OK) return rc;
  a.status = status;
  a.num_sms = num_sms;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  a.qr = q;
  a.kr = k;
  char what[64];
  if (dtype == CSATTN_F32) {
    void* qr = ws + al(rows * 4);
    void* kr = static_cast<uint8_t*>(qr) + al(rows * d * 4);
    cudaError_t e = launch_bwd_f32(a, qr, kr, st);
    std::snprintf(what, sizeof(what), "%s: fp32 kernel launch", fn);
    if (e != cudaSuccess) return fail_cuda(e, what);
    return CSATTN_OK;
  }
  if (tensor_map_encoder() == nullptr)
    return fail(CSATTN_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", fn);
  if (a.rope) {
    void* qr = ws + al(rows * 4);
    void* kr = static_cast<uint8_t*>(qr) + al(rows * d * 2);
    cudaError_t e = launch_rope_rotate_bf16(q, qr, B, Hq, Tq, d, a.rope, a.theta, st, q_offset);
    if (e == cudaSuccess) e = launch_rope_rotate_bf16(k, kr, B, Hkv, Tk, d, a.rope, a.theta, st);
    std::snprintf(what, sizeof(what), "%s: RoPE kernel launch", fn);
    if (e != cudaSuccess) return fail_cuda(e, what);
    a.qr = qr;
    a.kr = kr;
  }
  cudaError_t e = launch_bwd_bf16(a, st);
  std::snprintf(what, sizeof(what), "%s: kernel launch", fn);
  if (e != cudaSuccess) return fail_cuda(e, what);
  return CSATTN_OK;
}

}  // namespace

extern "C" {

int csattn_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                    int Hq, int Hkv, int T, int d, int dtype, int causal, float rope_base,
                    int rope_layout, float scale, void* workspace, size_t workspace_bytes,
                    void* stream) {
  return attn_bwd_impl("attn_bwd", q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, T, T, 0, d, d,
                       dtype, causal, rope_base, rope_layout, scale, workspace, workspace_bytes,
                       stream);
}

int csattn_attn_bwd_ext(const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                        int Hq, int Hkv, int Tq, int Tk, int q_offset, int d, int d_v, int dtype,
                        int causal, float rope_base, int rope_layout, float scale,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_impl("attn_bwd_ext", q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Tq, Tk,
                       q_offset, d, d_v > 0 ? d_v : d, dtype, causal, rope_base, rope_layout,
                       scale, workspace, workspace_bytes, stream);
}

int csattn_rope_rotate(const void* x, void* x_rot, int B, int H, int T, int d, int dtype,
                       float rope_base, int rope_layout, void* stream) {
  if (x == nullptr || x_rot == nullptr)
    return fail(CSATTN_ERR_INVALID_ARG, "rope_rotate: null pointer argument");
  if (B < 1 || H < 1 || T < 1)
    return fail(CSATTN_ERR_INVALID_ARG, "rope_rotate: B=%d H=%d T=%d must be >= 1", B, H, T);
  if (dtype != CSATTN_BF16 && dtype != CSATTN_F32)
    return fail(CSATTN_ERR_INVALID_ARG, "rope_rotate: unknown dtype %d", dtype);
  if (dtype == CSATTN_BF16 ? (d != 64 && d != 128) : (d != 16 && d != 32 && d != 64 && d != 128))
    return fail(CSATTN_ERR_UNSUPPORTED, "rope_rotate: d=%d", d);
  if (!(rope_base > 0.f) || !std::isfinite(rope_base))
    return fail(CSATTN_ERR_INVALID_ARG, "rope_rotate: rope_base must be finite and > 0");
  if (rope_layout != CSATTN_ROPE_SPLIT_HALF && rope_layout != CSATTN_ROPE_ADJACENT)
    return fail(CSATTN_ERR_INVALID_ARG, "rope_rotate: unknown rope_layout %d", rope_layout);
  if (T > kMaxRopePositions)
    return fail(CSATTN_ERR_UNSUPPORTED, "rope_rotate: T <= %d, got %d", kMaxRopePositions, T);
  if (!aligned16(x) || !aligned16(x_rot))
    return fail(CSATTN_ERR_INVALID_ARG, "rope_rotate: x, x_rot must be 16-byte aligned");
  const size_t bytes = static_cast<size_t>(B) * H * T * d * (dtype == CSATTN_F32 ? 4 : 2);
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(x), b0 = reinterpret_cast<uintptr_t>(x_rot);
  if (a0 < b0 + bytes && b0 < a0 + bytes)
    return fail(CSATTN_ERR_INVALID_ARG, "rope_rotate: x and x_rot overlap");
  RopeTable th;
  rope_table(&th, d, static_cast<double>(rope_base));
  const int layout = rope_layout == CSATTN_ROPE_SPLIT_HALF ? 1 : 2;
  cudaError_t e =
      dtype == CSATTN_F32
          ? launch_rope_rotate_f32(x, x_rot, B, H, T, d, layout, th,
                                   static_cast<cudaStream_t>(stream))
          : launch_rope_rotate_bf16(x, x_rot, B, H, T, d, layout, th,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "rope_rotate: kernel launch");
  return CSATTN_OK;
}

size_t csattn_decode_workspace_size(int B, int Hq, int Lmax, int d, int num_splits) {
  if (B < 1 || Hq < 1 || Lmax < 1 || d < 1 || num_splits < 0) return 0;
  const size_t splits = num_splits > 0 ? static_cast<size_t>(num_splits)
                                       : static_cast<size_t>((Lmax + 255) / 256);
  // part_o [B, Hq, S, d] then part_ml [B, Hq, S, 2], fp32
  return static_cast<size_t>(B) * Hq * splits * (static_cast<size_t>(d) + 2) * 4;
}

}  // extern "C"

namespace {

// Host-side checks shared by both decode entry points (q may be any non-null
// placeholder when the queries are produced on the device).
int decode_check(const char* fn, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* seq_lens, const void* out, int B, int Hq, int Hkv, int Lmax, int d,
                 int dtype, float scale, int max_seq_len, int num_splits,
                 bool allow_f32 = false) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seq_lens == nullptr ||
      out == nullptr)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: null pointer argument", fn);
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: B=%d Hq=%d Hkv=%d Lmax=%d must be >= 1", fn,
                B, Hq, Hkv, Lmax);
  if (Hq % Hkv != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: Hq=%d is not a multiple of Hkv=%d", fn, Hq,
                Hkv);
  if (dtype != CSATTN_BF16 && !(allow_f32 && dtype == CSATTN_F32))
    return fail(dtype == CSATTN_F32 ? CSATTN_ERR_UNSUPPORTED : CSATTN_ERR_INVALID_ARG,
                "%s: only bf16 is implemented (dtype %d)", fn, dtype);
  if (dtype == CSATTN_F32) {
    if (d != 16 && d != 32 && d != 64 && d != 128)
      return fail(CSATTN_ERR_UNSUPPORTED, "%s: fp32 d=%d not in {16,32,64,128}", fn, d);
  } else {
    if (d != 64 && d != 128) return fail(CSATTN_ERR_UNSUPPORTED, "%s: d=%d", fn, d);
    if (Hq / Hkv > 16)
      return fail(CSATTN_ERR_UNSUPPORTED, "%s: group size %d > 16", fn, Hq / Hkv);
  }
  if (max_seq_len < 1 || max_seq_len > Lmax)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: max_seq_len=%d not in [1, Lmax=%d]", fn,
                max_seq_len, Lmax);
  if (num_splits < 0) return fail(CSATTN_ERR_INVALID_ARG, "%s: num_splits < 0", fn);
  if (!std::isfinite(scale)) return fail(CSATTN_ERR_INVALID_ARG, "%s: scale not finite", fn);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  return CSATTN_OK;
}

}  // namespace

int csattn::attn_decode_check_ptrs(const char* fn, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* seq_lens, const void* out,
                                   int B, int Hq, int Hkv, int Lmax, int d, int dtype, float scale,
                                   int max_seq_len, int num_splits) {
  return decode_check(fn, q, k_cache, v_cache, seq_lens, out, B, Hq, Hkv, Lmax, d, dtype, scale,
                      max_seq_len, num_splits);
}

int csattn::attn_decode_check(const char* fn, int B, int Hq, int Hkv, int Lmax, int d,
                              int dtype, float scale, int max_seq_len, int num_splits) {
  alignas(16) static const uint8_t dummy[16] = {};
  const void* x = dummy;
  return decode_check(fn, x, x, x, reinterpret_cast<const int32_t*>(dummy), x, B, Hq, Hkv,
                      Lmax, d, dtype, scale, max_seq_len, num_splits);
}

namespace {

// Shared by csattn_attn_decode (len_add 0), csattn_attn_decode_ext (dv may differ
// from d) and csattn_attn_decode_step (len_add 1: the appended row).
int decode_impl(const char* fn, const void* q, const void* k_cache, const void* v_cache,
                const int32_t* seq_lens, int len_add, void* out, int B, int Hq, int Hkv, int Lmax,
                int d, int dtype, float scale, int max_seq_len, int num_splits, void* workspace,
                size_t workspace_bytes, void* stream, const int32_t* block_table = nullptr,
                int page_size = 0, int num_pages = 0, int max_pages = 0, int dv = 0,
                bool allow_f32 = false) {
  int rc = decode_check(fn, q, k_cache, v_cache, seq_lens, out, B, Hq, Hkv, Lmax, d, dtype, scale,
                        max_seq_len, num_splits, allow_f32);
  if (rc != CSATTN_OK) return rc;
  if (dv <= 0) dv = d;
  if (dtype == CSATTN_BF16 ? (dv != 64 && dv != 128) : dv != d)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: dv=%d", fn, dv);
  DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.seq_lens = seq_lens;
  a.len_add = len_add;
  a.block_table = block_table;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.max_pages = max_pages;
  a.out = out;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.d = d;
  a.dv = dv;
  a.scale = scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  a.max_seq_len = max_seq_len;
  int num_sms = 0;
  if (num_splits > 0) {
    const int per = (max_seq_len + num_splits - 1) / num_splits;
    a.chunk = ((per + 63) / 64) * 64;
  } else {
    rc = device_info(&a.status, &num_sms);
    if (rc != CSATTN_OK) return rc;
    // Smallest chunk (>= 256 keys) that keeps the grid at most ~32 CTAs per SM
    // (measured on the B=64, L~U[512,8192] workload: 1024-key chunks).
    a.chunk = 256;
    while (a.chunk < 4096 &&
           static_cast<long long>(B) * Hkv * ((max_seq_len + a.chunk - 1) / a.chunk) >
               32LL * num_sms)
      a.chunk *= 2;
  }
  a.n_splits = (max_seq_len + a.chunk - 1) / a.chunk;
  const size_t need = static_cast<size_t>(B) * Hq * a.n_splits * (static_cast<size_t>(dv) + 2) * 4;
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return fail(CSATTN_ERR_WORKSPACE,
                "%s: needs a 16-byte aligned workspace of %zu bytes (got %zu)", fn, need,
                workspace_bytes);
  if (a.status == nullptr) {
    rc = device_info(&a.status, &num_sms);
    if (rc != CSATTN_OK) return rc;
  }
  a.part_o = static_cast<float*>(workspace);
  a.part_ml = a.part_o + static_cast<size_t>(B) * Hq * a.n_splits * dv;
  if (dtype == CSATTN_F32) {
    cudaError_t e = launch_decode_f32(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "attn_decode: fp32 kernel launch");
    return CSATTN_OK;
  }
  if (tensor_map_encoder() == nullptr)
    return fail(CSATTN_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", fn);
  cudaError_t e = launch_decode_bf16(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "attn_decode: kernel launch");
  return CSATTN_OK;
}

}  // namespace

extern "C" {

int csattn_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* seq_lens, void* out, int B, int Hq, int Hkv, int Lmax,
                       int d, int dtype, float scale, int max_seq_len, int num_splits,
                       void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl("attn_decode", q, k_cache, v_cache, seq_lens, 0, out, B, Hq, Hkv, Lmax, d,
                     dtype, scale, max_seq_len, num_splits, workspace, workspace_bytes, stream,
                     nullptr, 0, 0, 0, 0, true);
}

int csattn_attn_decode_ext(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, void* out, int B, int Hq, int Hkv, int Lmax,
                           int d, int dv, int dtype, float scale, int max_seq_len,
                           int num_splits, void* workspace, size_t workspace_bytes,
                           void* stream) {
  return decode_impl("attn_decode_ext", q, k_cache, v_cache, seq_lens, 0, out, B, Hq, Hkv, Lmax,
                     d, dtype, scale, max_seq_len, num_splits, workspace, workspace_bytes, stream,
                     nullptr, 0, 0, 0, dv > 0 ? dv : d);
}

int csattn_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                             const int32_t* block_table, const int32_t* seq_lens, void* out, int B,
                             int Hq, int Hkv, int page_size, int num_pages, int max_pages, int d,
                             int dtype, float scale, int max_seq_len, int num_splits,
                             void* workspace, size_t workspace_bytes, void* stream) {
  const char* fn = "attn_decode_paged";
  if (block_table == nullptr)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: block_table must be non-null", fn);
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: block_table must be 4-byte aligned", fn);
  if (!valid_page_size(page_size))
    return fail(CSATTN_ERR_INVALID_ARG,
                "%s: page_size=%d must be 16, 32 or a multiple of 64 in [64, 65536]", fn,
                page_size);
  if (num_pages < 1 || max_pages < 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: num_pages=%d and max_pages=%d must be >= 1", fn,
                num_pages, max_pages);
  if (Hkv >= 1 && static_cast<long long>(num_pages) * Hkv > (1LL << 31) - 1)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: num_pages * Hkv too large", fn);
  const long long lmax = static_cast<long long>(max_pages) * page_size;
  if (lmax > (1 << 30))
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: max_pages * page_size too large", fn);
  // the logical cache of a sequence is max_pages * page_size rows long
  return decode_impl(fn, q, k_pages, v_pages, seq_lens, 0, out, B, Hq, Hkv, static_cast<int>(lmax),
                     d, dtype, scale, max_seq_len, num_splits, workspace, workspace_bytes, stream,
                     block_table, page_size, num_pages, max_pages);
}

size_t csattn_prefill_paged_workspace_size(int B, int Hkv, int page_size, int max_pages,
                                           int d) {
  if (B < 1 || Hkv < 1 || max_pages < 1 || d < 1 || page_size < 1 || page_size >= 64) return 0;
  const size_t lpad = (static_cast<size_t>(max_pages) * page_size + 127) / 128 * 128;
  const size_t pool = static_cast<size_t>(B) * Hkv * lpad * d * 2;
  return 2 * align256(pool) + align256(static_cast<size_t>(B) * 4);
}

int csattn_attn_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* block_table, const int32_t* cache_lens, void* out,
                              int B, int Hq, int Hkv, int Tq, int page_size, int num_pages,
                              int max_pages, int d, int dtype, int causal, float rope_base,
                              int rope_layout, float scale, float* lse, void* workspace,
                              size_t workspace_bytes, void* stream) {
  const char* fn = "attn_prefill_paged";
  if (q == nullptr || k_pages == nullptr || v_pages == nullptr || block_table == nullptr ||
      cache_lens == nullptr || out == nullptr)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: null pointer argument", fn);
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: B=%d Hq=%d Hkv=%d Tq=%d must be >= 1", fn, B, Hq,
                Hkv, Tq);
  if (Hq % Hkv != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: Hq=%d is not a multiple of Hkv=%d", fn, Hq, Hkv);
  if (dtype != CSATTN_BF16)
    return fail(dtype == CSATTN_F32 ? CSATTN_ERR_UNSUPPORTED : CSATTN_ERR_INVALID_ARG,
                "%s: only bf16 is implemented (dtype %d)", fn, dtype);
  if (d != 64 && d != 128) return fail(CSATTN_ERR_UNSUPPORTED, "%s: d=%d not in {64,128}", fn, d);
  if (causal != 0 && causal != 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: causal must be 0 or 1", fn);
  if (rope_layout != CSATTN_ROPE_SPLIT_HALF && rope_layout != CSATTN_ROPE_ADJACENT)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: unknown rope_layout %d", fn, rope_layout);
  if (!std::isfinite(rope_base) || !std::isfinite(scale))
    return fail(CSATTN_ERR_INVALID_ARG, "%s: rope_base and scale must be finite", fn);
  if (!valid_page_size(page_size))
    return fail(CSATTN_ERR_INVALID_ARG,
                "%s: page_size=%d must be 16, 32 or a multiple of 64 in [64, 65536]", fn,
                page_size);
  if (num_pages < 1 || max_pages < 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: num_pages=%d and max_pages=%d must be >= 1", fn,
                num_pages, max_pages);
  if (static_cast<long long>(num_pages) * Hkv > (1LL << 31) - 1)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: num_pages * Hkv too large", fn);
  const long long lmax = static_cast<long long>(max_pages) * page_size;
  if (lmax >= (1 << 24))
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: max_pages * page_size must be < 2^24", fn);
  if (Tq > lmax)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: Tq=%d exceeds max_pages * page_size = %lld", fn, Tq,
                lmax);
  if (rope_base > 0.f && lmax > kMaxRopePositions)
    return fail(CSATTN_ERR_UNSUPPORTED,
                "%s: RoPE supports positions < %d (max_pages * page_size = %lld)", fn,
                kMaxRopePositions, lmax);
  if (static_cast<long long>(B) * Hq > (1LL << 31) - 1 || B > 65535)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: B=%d too large", fn, B);
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  const size_t need = csattn_prefill_paged_workspace_size(B, Hkv, page_size, max_pages, d);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return fail(CSATTN_ERR_WORKSPACE,
                "%s: %d-row pages need a 16-byte aligned workspace of %zu bytes (got %zu)", fn,
                page_size, need, workspace_bytes);

  FwdArgs a{};
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.dv = d;
  a.Tq = Tq;
  a.Tk = Tq;
  a.q_off = 0;
  a.causal = causal;
  a.rope = rope_base > 0.f ? (rope_layout == CSATTN_ROPE_SPLIT_HALF ? 1 : 2) : 0;
  a.rope_k = 0;  // the cache holds rotated keys
  a.scale = scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  if (a.rope) rope_table(&a.theta, d, static_cast<double>(rope_base));
  a.cache_lens = cache_lens;
  a.block_table = block_table;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.max_pages = max_pages;
  int rc = device_info(&a.status, &a.num_sms);
  if (rc != CSATTN_OK) return rc;
  if (tensor_map_encoder() == nullptr)
    return fail(CSATTN_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", fn);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (need > 0) {
    // small pages: gather each sequence's rows into one page of its own first
    const int lpad = static_cast<int>((lmax + 127) / 128 * 128);
    const size_t pool = static_cast<size_t>(B) * Hkv * lpad * d * 2;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* kg = ws;
    void* vg = ws + align256(pool);
    int32_t* ident = reinterpret_cast<int32_t*>(ws + 2 * align256(pool));
    cudaError_t e = launch_gather_pages_bf16(k_pages, v_pages, block_table, cache_lens, kg, vg,
                                             ident, B, Hkv, Tq, d, page_size, num_pages,
                                             max_pages, lpad, a.status, st);
    if (e != cudaSuccess) return fail_cuda(e, "attn_prefill_paged: gather kernel launch");
    a.k = kg;
    a.v = vg;
    a.block_table = ident;
    a.page_size = lpad;
    a.num_pages = B;
    a.max_pages = 1;
  }
  cudaError_t e = launch_fwd_sm103a(a, a.k, st);
  if (e != cudaSuccess) return fail_cuda(e, "attn_prefill_paged: kernel launch");
  return CSATTN_OK;
}

size_t csattn_decode_step_workspace_size(int B, int Hq, int Lmax, int d, int num_splits) {
  const size_t part = csattn_decode_workspace_size(B, Hq, Lmax, d, num_splits);
  if (part == 0) return 0;
  return align256(part) + static_cast<size_t>(B) * Hq * d * 2;  // + the rotated queries
}

int csattn_attn_decode_step(const void* q_new, const void* k_new, const void* v_new,
                            void* k_cache, void* v_cache, const int32_t* cache_lens, void* out,
                            int B, int Hq, int Hkv, int Lmax, int d, int dtype, float rope_base,
                            int rope_layout, float scale, int max_seq_len, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream) {
  const char* fn = "attn_decode_step";
  if (q_new == nullptr || k_new == nullptr || v_new == nullptr)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: q_new, k_new and v_new must be non-null", fn);
  if (!aligned16(q_new) || !aligned16(k_new) || !aligned16(v_new))
    return fail(CSATTN_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  if (rope_layout != CSATTN_ROPE_SPLIT_HALF && rope_layout != CSATTN_ROPE_ADJACENT)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: unknown rope_layout %d", fn, rope_layout);
  if (!std::isfinite(rope_base))
    return fail(CSATTN_ERR_INVALID_ARG, "%s: rope_base must be finite", fn);
  if (rope_base > 0.f && max_seq_len > kMaxRopePositions)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: RoPE supports positions < %d, max_seq_len=%d", fn,
                kMaxRopePositions, max_seq_len);
  const size_t need = csattn_decode_step_workspace_size(B, Hq, Lmax, d, num_splits);
  if (need == 0 || workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return fail(CSATTN_ERR_WORKSPACE,
                "%s: needs a 16-byte aligned workspace of %zu bytes (got %zu)", fn, need,
                workspace_bytes);
  const size_t q_at = need - static_cast<size_t>(B) * Hq * d * 2;
  void* q_rot = static_cast<uint8_t*>(workspace) + q_at;
  // every check of the decode runs before the cache is written
  int rc = decode_check(fn, q_rot, k_cache, v_cache, cache_lens, out, B, Hq, Hkv, Lmax, d, dtype,
                        scale, max_seq_len, num_splits);
  if (rc != CSATTN_OK) return rc;
  RopeTable th{};
  const int rope = rope_base > 0.f ? (rope_layout == CSATTN_ROPE_SPLIT_HALF ? 1 : 2) : 0;
  if (rope) rope_table(&th, d, static_cast<double>(rope_base));
  uint32_t* status = nullptr;
  int num_sms = 0;
  rc = device_info(&status, &num_sms);
  if (rc != CSATTN_OK) return rc;
  cudaError_t e = launch_decode_append_bf16(q_new, k_new, v_new, k_cache, v_cache, cache_lens,
                                            q_rot, B, Hq, Hkv, Lmax, d, max_seq_len, rope, th,
                                            status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "attn_decode_step: append kernel launch");
  return decode_impl(fn, q_rot, k_cache, v_cache, cache_lens, 1, out, B, Hq, Hkv, Lmax, d, dtype,
                     scale, max_seq_len, num_splits, workspace, q_at, stream);
}

}  // extern "C"

namespace {

// Shared by the contiguous and the paged chunk append (block_table == nullptr: contiguous).
int cache_append_impl(const char* fn, const void* k_new, const void* v_new, void* k_cache,
                      void* v_cache, const int32_t* cache_lens, const int32_t* block_table, int B,
                      int Hkv, int Tn, int Lmax, int d, int page_size, int num_pages,
                      int max_pages, int dtype, float rope_base, int rope_layout, void* stream) {
  if (k_new == nullptr || v_new == nullptr || k_cache == nullptr || v_cache == nullptr ||
      cache_lens == nullptr)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  if (B < 1 || Hkv < 1 || Tn < 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: B=%d, Hkv=%d, Tn=%d must be >= 1", fn, B, Hkv, Tn);
  if (dtype != CSATTN_F32 && dtype != CSATTN_BF16)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, dtype);
  if (dtype != CSATTN_BF16)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: only bf16 is implemented (dtype %d)", fn, dtype);
  if (d != 64 && d != 128) return fail(CSATTN_ERR_UNSUPPORTED, "%s: d=%d", fn, d);
  if (rope_layout != CSATTN_ROPE_SPLIT_HALF && rope_layout != CSATTN_ROPE_ADJACENT)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: unknown rope_layout %d", fn, rope_layout);
  if (!std::isfinite(rope_base))
    return fail(CSATTN_ERR_INVALID_ARG, "%s: rope_base must be finite", fn);
  if (Lmax < Tn) return fail(CSATTN_ERR_INVALID_ARG, "%s: Tn=%d > cache rows %d", fn, Tn, Lmax);
  if (Lmax >= (1 << 30) || Tn >= (1 << 20))
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: cache rows %d or Tn=%d too large", fn, Lmax, Tn);
  if (rope_base > 0.f && Lmax > kMaxRopePositions)
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: RoPE supports positions < %d, cache rows %d", fn,
                kMaxRopePositions, Lmax);
  RopeTable th{};
  const int rope = rope_base > 0.f ? (rope_layout == CSATTN_ROPE_SPLIT_HALF ? 1 : 2) : 0;
  if (rope) rope_table(&th, d, static_cast<double>(rope_base));
  uint32_t* status = nullptr;
  int num_sms = 0;
  int rc = device_info(&status, &num_sms);
  if (rc != CSATTN_OK) return rc;
  cudaError_t e = launch_cache_append_bf16(k_new, v_new, k_cache, v_cache, cache_lens,
                                           block_table, B, Hkv, Tn, Lmax, d, page_size,
                                           num_pages, max_pages, rope, th, status,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cache append kernel launch");
  return CSATTN_OK;
}

}  // namespace

extern "C" {

int csattn_cache_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                        const int32_t* cache_lens, int B, int Hkv, int Tn, int Lmax, int d,
                        int dtype, float rope_base, int rope_layout, void* stream) {
  return cache_append_impl("cache_append", k_new, v_new, k_cache, v_cache, cache_lens, nullptr,
                           B, Hkv, Tn, Lmax, d, 0, 0, 0, dtype, rope_base, rope_layout, stream);
}

int csattn_cache_append_paged(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                              const int32_t* block_table, const int32_t* cache_lens, int B,
                              int Hkv, int Tn, int page_size, int num_pages, int max_pages, int d,
                              int dtype, float rope_base, int rope_layout, void* stream) {
  const char* fn = "cache_append_paged";
  if (block_table == nullptr)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: block_table must be non-null", fn);
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: block_table must be 4-byte aligned", fn);
  if (!valid_page_size(page_size))
    return fail(CSATTN_ERR_INVALID_ARG,
                "%s: page_size=%d must be 16, 32 or a multiple of 64 in [64, 65536]", fn,
                page_size);
  if (num_pages < 1 || max_pages < 1)
    return fail(CSATTN_ERR_INVALID_ARG, "%s: num_pages=%d and max_pages=%d must be >= 1", fn,
                num_pages, max_pages);
  if (Hkv >= 1 && static_cast<long long>(num_pages) * Hkv * page_size > (1LL << 40))
    return fail(CSATTN_ERR_UNSUPPORTED, "%s: page pool too large", fn);
  const long long lmax = static_cast<long long>(max_pages) * page_size;
  if (lmax >= (1 << 30)) return fail(CSATTN_ERR_UNSUPPORTED, "%s: max_pages * page_size too large", fn);
  return cache_append_impl(fn, k_new, v_new, k_pages, v_pages, cache_lens, block_table, B, Hkv, Tn,
                           static_cast<int>(lmax), d, page_size, num_pages, max_pages, dtype,
                           rope_base, rope_layout, stream);
}

int csattn_check_status(void* stream) {
  uint32_t* status = nullptr;
  int num_sms = 0;
  int rc = device_info(&status, &num_sms);
  if (rc != CSATTN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail_cuda(e, "check_status: stream synchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e, "check_status: read status word");
  if (word != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e, "check_status: clear status word");
  }
  if (word & kStatusTimeout)
    return fail(CSATTN_ERR_TIMEOUT, "a kernel wait ran out of time (status 0x%x)", word);
  if (word & kStatusDeviceArg)
    return fail(CSATTN_ERR_DEVICE_ARG, "a device-side argument check failed (status 0x%x)", word);
  return CSATTN_OK;
}

int csattn_selftest_bounded_wait(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000)
    return fail(CSATTN_ERR_INVALID_ARG, "selftest: limit_us=%d not in [1, 1e6]", limit_us);
  uint32_t* status = nullptr;
  int num_sms = 0;
  int rc = device_info(&status, &num_sms);
  if (rc != CSATTN_OK) return rc;
  cudaError_t e = launch_selftest_wait(status, static_cast<uint64_t>(limit_us) * 1000ull,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "selftest: launch");
  return CSATTN_OK;
}

}  // extern "C"
