// The cache append of one decode step: the new token of sequence b sits at
// position p = cache_lens[b] ("The Transformer architecture" (cooking-agi),
// section "Hands-on": the cache grows by one row per generated token, and the
// query at cache.pos attends to keys 0..cache.pos).  Its query and key are
// rotated at p (RoPE on q and k, never v: same page, section "Now: RoPE") and
// rounded to bf16 once, as csattn_rope_rotate rounds; the rotated key and the
// value go to row p of the caches, the rotated query to q_rot, which the
// decode kernels then read with length p + 1.
//
// One CTA per sequence; thread work item = (head, 16-channel chunk): the
// chunk's 8 (cos, sin) pairs are computed once per item.  This pass moves
// B*(Hq + 2*Hkv)*d*2*2 bytes, a few hundred KB for a whole batch: it is
// launch-latency bound, and runs before the HBM-bound decode kernels.
#include "internal.h"

namespace csattn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void rotate8(const __nv_bfloat16* src, __nv_bfloat16* dst, int d,
                                        int c, int layout, const float (&cs)[8],
                                        const float (&sn)[8]) {
  int e0, e1;
  if (layout == 1) {  // split-half: channel p with p + d/2
    e0 = 8 * c;
    e1 = d / 2 + 8 * c;
  } else {            // adjacent: channels 16c..16c+15 hold pairs 8c..8c+7
    e0 = 16 * c;
    e1 = 16 * c + 8;
  }
  const uint4 a = *reinterpret_cast<const uint4*>(src + e0);
  const uint4 b = *reinterpret_cast<const uint4*>(src + e1);
  const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
  float u[8], w[8], ou[8], ow[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    u[2 * i] = bf16lo_to_f32(wa[i]);
    u[2 * i + 1] = bf16hi_to_f32(wa[i]);
    w[2 * i] = bf16lo_to_f32(wb[i]);
    w[2 * i + 1] = bf16hi_to_f32(wb[i]);
  }
  if (layout == 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ou[i] = fmaf(u[i], cs[i], -w[i] * sn[i]);
      ow[i] = fmaf(u[i], sn[i], w[i] * cs[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ou[2 * i] = fmaf(u[2 * i], cs[i], -u[2 * i + 1] * sn[i]);
      ou[2 * i + 1] = fmaf(u[2 * i], sn[i], u[2 * i + 1] * cs[i]);
      ow[2 * i] = fmaf(w[2 * i], cs[4 + i], -w[2 * i + 1] * sn[4 + i]);
      ow[2 * i + 1] = fmaf(w[2 * i], sn[4 + i], w[2 * i + 1] * cs[4 + i]);
    }
  }
  *reinterpret_cast<uint4*>(dst + e0) = make_uint4(pack_bf16x2(ou[0], ou[1]), pack_bf16x2(ou[2], ou[3]),
                                                   pack_bf16x2(ou[4], ou[5]), pack_bf16x2(ou[6], ou[7]));
  *reinterpret_cast<uint4*>(dst + e1) = make_uint4(pack_bf16x2(ow[0], ow[1]), pack_bf16x2(ow[2], ow[3]),
                                                   pack_bf16x2(ow[4], ow[5]), pack_bf16x2(ow[6], ow[7]));
}

__global__ void __launch_bounds__(kThreads) decode_append_kernel(
    const __nv_bfloat16* __restrict__ q_new, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* __restrict__ k_cache,
    __nv_bfloat16* __restrict__ v_cache, const int32_t* __restrict__ cache_lens,
    __nv_bfloat16* __restrict__ q_rot, int Hq, int Hkv, int Lmax, int d, int max_pos, int rope,
    RopeTable theta, uint32_t* status) {
  const int b = blockIdx.x;
  const int pos = cache_lens[b];
  if (pos < 0 || pos >= max_pos) {
    if (threadIdx.x == 0) atomicOr(status, kStatusDeviceArg);
    return;
  }
  const int chunks = d / 16;
  // items: query heads, then key heads (rotated); then value heads (copied)
  const int n_rot = (Hq + Hkv) * chunks;
  const int n_all = n_rot + Hkv * (d / 8);
  for (int it = threadIdx.x; it < n_all; it += blockDim.x) {
    if (it < n_rot) {
      const int head = it / chunks, c = it - head * chunks;
      const __nv_bfloat16* src;
      __nv_bfloat16* dst;
      if (head < Hq) {
        src = q_new + (static_cast<size_t>(b) * Hq + head) * d;
        dst = q_rot + (static_cast<size_t>(b) * Hq + head) * d;
      } else {
        const int g = head - Hq;
        src = k_new + (static_cast<size_t>(b) * Hkv + g) * d;
        dst = k_cache + ((static_cast<size_t>(b) * Hkv + g) * Lmax + pos) * d;
      }
      if (rope == 0) {
        // no rotation: copy the chunk's 16 channels
        const int e = 16 * c;
        *reinterpret_cast<uint4*>(dst + e) = *reinterpret_cast<const uint4*>(src + e);
        *reinterpret_cast<uint4*>(dst + e + 8) = *reinterpret_cast<const uint4*>(src + e + 8);
        continue;
      }
      float cs[8], sn[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        rope_cos_sin<false>(pos, theta.hi[8 * c + i], theta.lo[8 * c + i], cs[i], sn[i]);
      rotate8(src, dst, d, c, rope, cs, sn);
    } else {
      const int j = it - n_rot;
      const int g = j / (d / 8), e = 8 * (j - g * (d / 8));
      *reinterpret_cast<uint4*>(v_cache + ((static_cast<size_t>(b) * Hkv + g) * Lmax + pos) * d +
                                e) =
          *reinterpret_cast<const uint4*>(v_new + (static_cast<size_t>(b) * Hkv + g) * d + e);
    }
  }
}

// Append of Tn tokens per sequence (a prefill chunk): token t of sequence b sits
// at row r = cache_lens[b] + t; its key is rotated at r and rounded to bf16, and
// key and value go to row r of the caches, contiguous ([B, Hkv, Lmax, d]) or paged
// (block_table != nullptr: [num_pages, Hkv, page_size, d], row r of sequence b in
// page block_table[b * max_pages + r / page_size] at offset r % page_size).
// HBM-bound: the chunk's keys and values are read once and written once.
//
// Every thread makes one round trip to memory: it issues all of its loads, then
// writes.  The first CTAs take key items (sequence, group of kHeadGroup KV heads,
// token, 16-channel chunk: 8 loads of 16 bytes): the 8 (cos, sin) of the chunk's
// pairs depend on the position only and are computed once for the group's heads;
// the rest copy the values, kVChunks 16-byte chunks per thread, a warp's loads
// reading 512 contiguous bytes each.  On a 1024-token chunk (33.5 MB moved) this
// takes ~10.5 us back to back, against ~8-9 us for a plain 16.8 MB device copy.
constexpr int kHeadGroup = 4;
constexpr int kVChunks = 4;
constexpr int kAppendThreads = 256;

// RoPE of one chunk's 8 pairs in place, one 32-bit word of each half at a time (the
// arithmetic of rotate8, with a few registers live): a holds channels e0.., b channels
// e1.. (see rotate8).
__device__ __forceinline__ void rotate8_inplace(uint4& a, uint4& b, int layout,
                                                const float (&cs)[8], const float (&sn)[8]) {
  uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float u0 = bf16lo_to_f32(wa[i]), u1 = bf16hi_to_f32(wa[i]);
    const float w0 = bf16lo_to_f32(wb[i]), w1 = bf16hi_to_f32(wb[i]);
    if (layout == 1) {  // pairs (u_j, w_j), j = 2i, 2i + 1
      wa[i] = pack_bf16x2(fmaf(u0, cs[2 * i], -w0 * sn[2 * i]),
                          fmaf(u1, cs[2 * i + 1], -w1 * sn[2 * i + 1]));
      wb[i] = pack_bf16x2(fmaf(u0, sn[2 * i], w0 * cs[2 * i]),
                          fmaf(u1, sn[2 * i + 1], w1 * cs[2 * i + 1]));
    } else {  // pair i = (u0, u1), pair 4 + i = (w0, w1)
      wa[i] = pack_bf16x2(fmaf(u0, cs[i], -u1 * sn[i]), fmaf(u0, sn[i], u1 * cs[i]));
      wb[i] = pack_bf16x2(fmaf(w0, cs[4 + i], -w1 * sn[4 + i]),
                          fmaf(w0, sn[4 + i], w1 * cs[4 + i]));
    }
  }
  a = make_uint4(wa[0], wa[1], wa[2], wa[3]);
  b = make_uint4(wb[0], wb[1], wb[2], wb[3]);
}

// element offset of cache row r of head g (or -1 for a page index outside the pool)
__device__ __forceinline__ long long append_row(const int32_t* block_table, int b, int g, int r,
                                                int Hkv, int Lmax, int d, int page_size,
                                                int num_pages, int max_pages) {
  if (block_table == nullptr) return ((static_cast<long long>(b) * Hkv + g) * Lmax + r) * d;
  const int page = block_table[static_cast<size_t>(b) * max_pages + r / page_size];
  if (page < 0 || page >= num_pages) return -1;
  return ((static_cast<long long>(page) * Hkv + g) * page_size + r % page_size) * d;
}

__global__ void __launch_bounds__(kAppendThreads, 3) cache_append_kernel(
    const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
    __nv_bfloat16* __restrict__ k_cache, __nv_bfloat16* __restrict__ v_cache,
    const int32_t* __restrict__ cache_lens, const int32_t* __restrict__ block_table, int B,
    int Hkv, int Tn, int Lmax, int d, int page_size, int num_pages, int max_pages, int rope,
    RopeTable theta, uint32_t* status, int k_blocks) {
  __shared__ float th_hi[64], th_lo[64];
  const int tid = static_cast<int>(threadIdx.x);
  const int half = d / 2, kchunks = d / 16;
  // the frequencies through shared memory (a kernel parameter indexed per thread is
  // read from constant memory one address at a time)
  if (rope != 0 && tid < half) {
    th_hi[tid] = theta.hi[tid];
    th_lo[tid] = theta.lo[tid];
  }
  __syncthreads();
  if (static_cast<int>(blockIdx.x) < k_blocks) {
    // ------------------------------------------------------------ key items
    // (32-bit indices: the launcher checks that B * Hkv * Tn * d / 8 < 2^31)
    const int groups = (Hkv + kHeadGroup - 1) / kHeadGroup;
    int i = static_cast<int>(blockIdx.x) * kAppendThreads + tid;
    if (i >= B * groups * Tn * kchunks) return;
    const int c = i % kchunks;
    i /= kchunks;
    const int t = i % Tn;
    i /= Tn;
    const int g0 = (i % groups) * kHeadGroup;
    const int b = i / groups;
    const int L = cache_lens[b];
    if (L < 0 || L > Lmax - Tn) {  // (no overflow: Lmax, Tn < 2^30)
      if (t == 0 && c == 0 && g0 == 0) atomicOr(status, kStatusDeviceArg);
      return;
    }
    const int pos = L + t;
    // the two 8-channel halves of the chunk's pairs (channels e0.., e1.. of rotate8)
    const int e0 = rope == 1 ? 8 * c : 16 * c, e1 = rope == 1 ? half + 8 * c : 16 * c + 8;
    uint4 lo[kHeadGroup], hi[kHeadGroup];
#pragma unroll
    for (int k = 0; k < kHeadGroup; ++k) {
      if (g0 + k < Hkv) {
        const __nv_bfloat16* src = k_new + ((static_cast<size_t>(b) * Hkv + g0 + k) * Tn + t) * d;
        lo[k] = *reinterpret_cast<const uint4*>(src + e0);
        hi[k] = *reinterpret_cast<const uint4*>(src + e1);
      }
    }
    float cs[8], sn[8];
    if (rope != 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        rope_cos_sin<false>(pos, th_hi[8 * c + j], th_lo[8 * c + j], cs[j], sn[j]);
    }
#pragma unroll
    for (int k = 0; k < kHeadGroup; ++k) {
      if (g0 + k >= Hkv) continue;
      const long long row =
          append_row(block_table, b, g0 + k, pos, Hkv, Lmax, d, page_size, num_pages, max_pages);
      if (row < 0) {
        atomicOr(status, kStatusDeviceArg);
        continue;
      }
      __nv_bfloat16* dst = k_cache + row;
      if (rope != 0) rotate8_inplace(lo[k], hi[k], rope, cs, sn);
      *reinterpret_cast<uint4*>(dst + e0) = lo[k];  // (e0 = 16c, e1 = 16c + 8 without RoPE)
      *reinterpret_cast<uint4*>(dst + e1) = hi[k];
    }
    return;
  }
  // ------------------------------------------------------------ value items
  // 16-byte chunks in v_new order ([B, Hkv, Tn, d/8]); a warp takes 32 * kVChunks
  // consecutive ones, lane l chunks l, l + 32, ...: each load instruction of the warp
  // reads 512 contiguous bytes
  const int vchunks = d / 8;
  const int n_chunks = B * Hkv * Tn * vchunks;
  const int w = ((static_cast<int>(blockIdx.x) - k_blocks) * kAppendThreads + tid) / 32;
  const int base = w * (32 * kVChunks) + (tid & 31);
  uint4 val[kVChunks];
#pragma unroll
  for (int k = 0; k < kVChunks; ++k) {
    const int ci = base + 32 * k;
    if (ci < n_chunks) val[k] = reinterpret_cast<const uint4*>(v_new)[ci];
  }
#pragma unroll
  for (int k = 0; k < kVChunks; ++k) {
    int ci = base + 32 * k;
    if (ci >= n_chunks) break;
    const int c = ci % vchunks;
    ci /= vchunks;
    const int t = ci % Tn;
    ci /= Tn;
    const int g = ci % Hkv;
    const int b = ci / Hkv;
    const int L = cache_lens[b];
    if (L < 0 || L > Lmax - Tn) continue;  // reported by the key items
    const long long row =
        append_row(block_table, b, g, L + t, Hkv, Lmax, d, page_size, num_pages, max_pages);
    if (row < 0) {
      atomicOr(status, kStatusDeviceArg);
      continue;
    }
    *reinterpret_cast<uint4*>(v_cache + row + 8 * c) = val[k];
  }
}

}  // namespace

cudaError_t launch_decode_append_bf16(const void* q_new, const void* k_new, const void* v_new,
                                      void* k_cache, void* v_cache, const int32_t* cache_lens,
                                      void* q_rot, int B, int Hq, int Hkv, int Lmax, int d,
                                      int max_pos, int rope, const RopeTable& theta,
                                      uint32_t* status, cudaStream_t stream) {
  decode_append_kernel<<<B, kThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(q_new), static_cast<const __nv_bfloat16*>(k_new),
      static_cast<const __nv_bfloat16*>(v_new), static_cast<__nv_bfloat16*>(k_cache),
      static_cast<__nv_bfloat16*>(v_cache), cache_lens, static_cast<__nv_bfloat16*>(q_rot), Hq,
      Hkv, Lmax, d, max_pos, rope, theta, status);
  return cudaGetLastError();
}

cudaError_t launch_cache_append_bf16(const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const int32_t* cache_lens,
                                     const int32_t* block_table, int B, int Hkv, int Tn, int Lmax,
                                     int d, int page_size, int num_pages, int max_pages, int rope,
                                     const RopeTable& theta, uint32_t* status,
                                     cudaStream_t stream) {
  const long long k_items = static_cast<long long>(B) * ((Hkv + kHeadGroup - 1) / kHeadGroup) *
                            Tn * (d / 16);
  const long long v_chunks = static_cast<long long>(B) * Hkv * Tn * (d / 8);
  const long long k_blocks = (k_items + kAppendThreads - 1) / kAppendThreads;
  const long long v_blocks = (v_chunks + kAppendThreads * kVChunks - 1) / (kAppendThreads * kVChunks);
  // the kernel indexes chunks with 32-bit integers (B * Hkv * Tn * d / 8 chunks of 16
  // bytes; 2^31 of them would be a 32 GB chunk)
  if (v_chunks + 32LL * kAppendThreads * kVChunks >= 0x7fffffffLL) return cudaErrorInvalidValue;
  cache_append_kernel<<<static_cast<unsigned>(k_blocks + v_blocks), kAppendThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
      static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache), cache_lens,
      block_table, B, Hkv, Tn, Lmax, d, page_size, num_pages, max_pages, rope, theta, status,
      static_cast<int>(k_blocks));
  return cudaGetLastError();
}

}  // namespace csattn
