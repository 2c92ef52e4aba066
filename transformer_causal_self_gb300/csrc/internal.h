// Host-side interfaces between the C-ABI layer (csattn_api.cu) and the kernel
// translation units.  Launchers validate nothing: csattn_api.cu has already
// checked every argument.  They return a cudaError_t from the launch.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace csattn {

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  int B, Hq, Hkv, d;
  int dv;            // head size of v and out (d: head size of q and k)
  int Tq, Tk;        // query rows, key rows
  int q_off;         // position of query row 0 (keys sit at 0..Tk-1)
  int causal;        // 1: key j visible to query i iff j <= q_off + i
  int rope;          // 0 none, 1 split-half, 2 adjacent (applied to q)
  int rope_k;        // 1: rotate k as well; 0: k is used as given
  float scale;       // > 0
  RopeTable theta;   // valid when rope != 0
  uint32_t* status;  // device status word
  int num_sms;
  // Paged K/V (bf16, d = dv in {64, 128}; block_table == nullptr: k, v are [B, Hkv, Tk, d]).
  // k, v are pools [num_pages, Hkv, page_size, d] of rotated keys and values; sequence
  // b has cache_lens[b] + Tq rows (Tk and q_off unused), its query row i sits at
  // cache_lens[b] + i; page_size is a multiple of 64.
  const int32_t* cache_lens;
  const int32_t* block_table;
  int page_size, num_pages, max_pages;
};

// fp32 SIMT path (d and dv each in {16,32,64,128}).
cudaError_t launch_fwd_f32(const FwdArgs& a, cudaStream_t stream);

// bf16 path: x_rot = RoPE(x) for x [B, H, T, d] bf16 (rope 1 split-half, 2 adjacent),
// row t rotated at position pos0 + t.
cudaError_t launch_rope_rotate_bf16(const void* x, void* x_rot, int B, int H, int T, int d,
                                    int rope, const RopeTable& theta, cudaStream_t stream,
                                    int pos0 = 0);
// fp32: the same rotation in fp32 with the accurate sine/cosine (bwd_f32.cu).
cudaError_t launch_rope_rotate_f32(const void* x, void* x_rot, int B, int H, int T, int d,
                                   int rope, const RopeTable& theta, cudaStream_t stream);

// bf16 tcgen05 prefill; `k_eff` is k itself or its rotated copy.  q, k have d
// and v, out dv channels (each 64 or 128): dv = 64 runs the kernel in
// fwd_sm103a.cu, dv = 128 the one in fwd_sm103a_d128.cu.
cudaError_t launch_fwd_sm103a(const FwdArgs& a, const void* k_eff, cudaStream_t stream);
cudaError_t launch_fwd_sm103a_d128(const FwdArgs& a, const void* k_eff, cudaStream_t stream);

// Backward (bf16: d, d_v in {64, 128}; fp32: d, d_v in {16, 32, 64, 128}): dq, dk, dv
// of sum(out * dout).  q [B, Hq, Tq, d], k [B, Hkv, Tk, d], v [B, Hkv, Tk, d_v], out and
// dout [B, Hq, Tq, d_v]; query row i sits at position q_off + i, key j at j.  qr, kr
// are the rotated operands of the forward (bf16; the fp32 path rotates them itself);
// dvec is fp32 scratch [B, Hq, Tq] for rowsum(dout o out); lse is the forward's
// natural-log log-sum-exp.
struct BwdArgs {
  const void* qr;
  const void* kr;
  const void* v;
  const void* out;
  const void* dout;
  const float* lse;
  float* dvec;
  void* dq;
  void* dk;
  void* dv;
  int B, Hq, Hkv, Tq, Tk, q_off, d;
  int d_v;      // head size of v, out, dout and dv
  int num_sms;  // persistent dQ kernel grid
  int causal;
  int rope;  // 0 none, 1 split-half, 2 adjacent: dq, dk are rotated back by R^T
  float scale;
  RopeTable theta;
  uint32_t* status;  // device status word (timeouts of the tcgen05 kernel)
};

cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t stream);
// fp32 backward on the SIMT cores.  a.qr, a.kr are q and k as given; with RoPE they
// are rotated into q_rot, k_rot (fp32 scratch of q's and k's sizes) first.
cudaError_t launch_bwd_f32(const BwdArgs& a, void* q_rot, void* k_rot, cudaStream_t stream);
// dK, dV on tcgen05; called by launch_bwd_bf16
cudaError_t launch_bwd_kv_tc(const BwdArgs& a, cudaStream_t stream);
// dQ on tcgen05; called by launch_bwd_bf16
cudaError_t launch_bwd_q_tc(const BwdArgs& a, cudaStream_t stream);

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* seq_lens;
  int len_add;     // sequence b has seq_lens[b] + len_add cached rows
  // paged cache (block_table != nullptr): k_cache, v_cache are [num_pages, Hkv,
  // page_size, d]; row t of sequence b is in page block_table[b * max_pages +
  // t / page_size] at offset t % page_size.  page_size is a multiple of 64.
  const int32_t* block_table;
  int page_size, num_pages, max_pages;
  void* out;
  int B, Hq, Hkv, Lmax, d;
  int dv;          // head size of v_cache and out (<= 0: d)
  float scale;
  int max_seq_len;
  int chunk;       // keys per split, multiple of 64
  int n_splits;    // ceil(max_seq_len / chunk)
  float* part_o;   // [B, Hq, n_splits, dv]
  float* part_ml;  // [B, Hq, n_splits, 2]
  uint32_t* status;
};

cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t stream);
// fp32 decode on the SIMT cores (contiguous cache, d in {16, 32, 64, 128}, dv = d);
// the partials in the same layout, m in natural-log units.
cudaError_t launch_decode_f32(const DecodeArgs& a, cudaStream_t stream);

// One decode step's cache append: for sequence b at position p = cache_lens[b],
// q_rot[b,h] = RoPE_p(q_new[b,h]) for every query head, k_cache[b,g,p] =
// RoPE_p(k_new[b,g]) and v_cache[b,g,p] = v_new[b,g] for every KV head (rope
// 0: no rotation).  A position outside [0, max_pos) sets kStatusDeviceArg in
// *status and writes nothing for that sequence.
cudaError_t launch_decode_append_bf16(const void* q_new, const void* k_new, const void* v_new,
                                      void* k_cache, void* v_cache, const int32_t* cache_lens,
                                      void* q_rot, int B, int Hq, int Hkv, int Lmax, int d,
                                      int max_pos, int rope, const RopeTable& theta,
                                      uint32_t* status, cudaStream_t stream);

cudaError_t launch_selftest_wait(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);

// Replace the calling thread's csattn_last_error() message.
void set_last_error(const char* msg);

// The argument checks of csattn_attn_fwd (all but the pointers and the workspace), with
// its return codes and error messages prefixed by fn.
int attn_fwd_check(const char* fn, int B, int Hq, int Hkv, int T, int d, int dtype, int causal,
                   float rope_base, int rope_layout, float scale);

// The host-side argument checks of the bf16 decodes (all but the pointers).
int attn_decode_check(const char* fn, int B, int Hq, int Hkv, int Lmax, int d, int dtype,
                      float scale, int max_seq_len, int num_splits);

// The same checks including the pointers (null, alignment).  Touches no CUDA state.
int attn_decode_check_ptrs(const char* fn, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* seq_lens, const void* out, int B,
                           int Hq, int Hkv, int Lmax, int d, int dtype, float scale,
                           int max_seq_len, int num_splits);

// Driver entry point for cuTensorMapEncodeTiled (nullptr if unavailable).
void* tensor_map_encoder();

// Appends Tn rotated keys and values per sequence at rows cache_lens[b] + t of
// contiguous caches [B, Hkv, Lmax, d] (block_table == nullptr) or paged caches
// [num_pages, Hkv, page_size, d] with Lmax = max_pages * page_size.
cudaError_t launch_cache_append_bf16(const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const int32_t* cache_lens,
                                     const int32_t* block_table, int B, int Hkv, int Tn, int Lmax,
                                     int d, int page_size, int num_pages, int max_pages, int rope,
                                     const RopeTable& theta, uint32_t* status,
                                     cudaStream_t stream);

// Copies rows 0..cache_lens[b]+Tq-1 of each sequence's KV heads from a paged pool
// [num_pages, Hkv, page_size, d] into page b of contiguous pools [B, Hkv, Lpad, d] and
// writes the identity block table ident[b] = b (the paged prefill over small pages).
cudaError_t launch_gather_pages_bf16(const void* k_pages, const void* v_pages,
                                     const int32_t* block_table, const int32_t* cache_lens,
                                     void* k_out, void* v_out, int32_t* ident, int B, int Hkv,
                                     int Tq, int d, int page_size, int num_pages, int max_pages,
                                     int Lpad, uint32_t* status, cudaStream_t stream);

// Raises a kernel's dynamic shared-memory limit once per device (the attribute
// lasts for the process), so repeated launches skip the driver call.
struct SmemLimitOnce {
  std::atomic<uint64_t> done{0};
  template <typename Kernel>
  cudaError_t set(Kernel* kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

// 3-D bf16 tensor map over rows of `d` elements: dims {d, rows, planes},
// box {64, box_rows, 1}, 128-byte swizzle, zero fill out of bounds.
bool make_tmap_bf16_3d(void* tmap_out, const void* base, int d, int rows, int planes,
                       int box_rows);

}  // namespace csattn
