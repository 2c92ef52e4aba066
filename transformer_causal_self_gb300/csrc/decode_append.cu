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

// rotate8 on chunks already loaded: a = channels e0.., b = channels e1.. (see rotate8)
__device__ __forceinline__ void rotate8_regs(const uint4 a, const uint4 b, __nv_bfloat16* dst, int d,
                                             int c, int layout, const float (&cs)[8],
                                             const float (&sn)[8]) {
  int e0, e1;
  if (layout == 1) {
    e0 = 8 * c;
    e1 = d / 2 + 8 * c;
  } else {
    e0 = 16 * c;
    e1 = 16 * c + 8;
  }
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
// HBM-bound: the chunk's keys and values are read once and written once.  Grid
// (B * Hkv, token ranges of kTokens): a CTA streams kTokens consecutive rows of one
// head, so its reads and (contiguous-cache) writes are four runs of kTokens * d * 2
// bytes.  Thread work items: 8 channels of a value row, 8 channel pairs of a key
// row (its 8 angles computed by the thread); every load of a thread is issued
// before its first store.
constexpr int kTokens = 32;
constexpr int kVItems = 2;  // value items per thread: 32 rows x (128 / 8) / 256
constexpr int kKItems = 1;  // key items per thread:   32 rows x (128 / 16) / 256

// element offset of cache row r of head g (or -1 for a page index outside the pool)
__device__ __forceinline__ long long append_row(const int32_t* block_table, int b, int g, int r,
                                                int Hkv, int Lmax, int d, int page_size,
                                                int num_pages, int max_pages) {
  if (block_table == nullptr) return ((static_cast<long long>(b) * Hkv + g) * Lmax + r) * d;
  const int page = block_table[static_cast<size_t>(b) * max_pages + r / page_size];
  if (page < 0 || page >= num_pages) return -1;
  return ((static_cast<long long>(page) * Hkv + g) * page_size + r % page_size) * d;
}

__global__ void __launch_bounds__(kThreads) cache_append_kernel(
    const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
    __nv_bfloat16* __restrict__ k_cache, __nv_bfloat16* __restrict__ v_cache,
    const int32_t* __restrict__ cache_lens, const int32_t* __restrict__ block_table, int Hkv,
    int Tn, int Lmax, int d, int page_size, int num_pages, int max_pages, int rope,
    RopeTable theta, uint32_t* status) {
  __shared__ float th_hi[64], th_lo[64];
  const int b = blockIdx.x / Hkv, g = blockIdx.x - b * Hkv;
  const int t0 = blockIdx.y * kTokens;
  const int nt = min(kTokens, Tn - t0);
  const int L = cache_lens[b];
  if (L < 0 || L > Lmax - Tn) {  // (no overflow: Lmax, Tn < 2^30)
    if (threadIdx.x == 0 && blockIdx.y == 0 && g == 0) atomicOr(status, kStatusDeviceArg);
    return;
  }
  const int tid = static_cast<int>(threadIdx.x), nthr = static_cast<int>(blockDim.x);
  const int half = d / 2, vchunks = d / 8, kchunks = d / 16;
  const int n_val = nt * vchunks, n_key = nt * kchunks;
  const size_t src0 = ((static_cast<size_t>(b) * Hkv + g) * Tn + t0) * d;  // row t0 of the head
  for (int vb = 0, kb = 0; vb < n_val || kb < n_key; vb += kVItems * nthr, kb += kKItems * nthr) {
    uint4 val[kVItems], klo[kKItems], khi[kKItems];
    long long vrow[kVItems], krow[kKItems];
    int kcc[kKItems], kpos[kKItems];
#pragma unroll
    for (int k = 0; k < kVItems; ++k) {
      const int it = vb + tid + k * nthr;
      vrow[k] = -2;
      if (it < n_val) {
        const int tt = it / vchunks, c = it - tt * vchunks;
        val[k] = *reinterpret_cast<const uint4*>(v_new + src0 + static_cast<size_t>(tt) * d + 8 * c);
        vrow[k] = append_row(block_table, b, g, L + t0 + tt, Hkv, Lmax, d, page_size, num_pages,
                             max_pages);
        if (vrow[k] >= 0) vrow[k] += 8 * c;
      }
    }
#pragma unroll
    for (int k = 0; k < kKItems; ++k) {
      const int it = kb + tid + k * nthr;
      krow[k] = -2;
      kcc[k] = 0;
      kpos[k] = 0;
      if (it < n_key) {
        const int tt = it / kchunks, c = it - tt * kchunks;
        const __nv_bfloat16* src = k_new + src0 + static_cast<size_t>(tt) * d;
        // the two 8-channel halves of the chunk's pairs (channels e0.., e1.. of rotate8)
        const int e0 = rope == 1 ? 8 * c : 16 * c, e1 = rope == 1 ? half + 8 * c : 16 * c + 8;
        klo[k] = *reinterpret_cast<const uint4*>(src + e0);
        khi[k] = *reinterpret_cast<const uint4*>(src + e1);
        kcc[k] = c;
        kpos[k] = L + t0 + tt;
        krow[k] = append_row(block_table, b, g, kpos[k], Hkv, Lmax, d, page_size, num_pages,
                             max_pages);
      }
    }
    if (vb == 0 && rope != 0) {
      // the frequencies through shared memory, while the loads are in flight (a kernel
      // parameter indexed per thread is read from constant memory one address at a time)
      if (tid < half) {
        th_hi[tid] = theta.hi[tid];
        th_lo[tid] = theta.lo[tid];
      }
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < kVItems; ++k) {
      if (vrow[k] >= 0)
        *reinterpret_cast<uint4*>(v_cache + vrow[k]) = val[k];
      else if (vrow[k] == -1)
        atomicOr(status, kStatusDeviceArg);
    }
#pragma unroll
    for (int k = 0; k < kKItems; ++k) {
      if (krow[k] == -1) atomicOr(status, kStatusDeviceArg);
      if (krow[k] < 0) continue;
      __nv_bfloat16* dst = k_cache + krow[k];
      const int c = kcc[k];
      if (rope == 0) {  // e0 = 16c, e1 = 16c + 8 when rope == 0
        *reinterpret_cast<uint4*>(dst + 16 * c) = klo[k];
        *reinterpret_cast<uint4*>(dst + 16 * c + 8) = khi[k];
        continue;
      }
      float cs[8], sn[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        rope_cos_sin<false>(kpos[k], th_hi[8 * c + i], th_lo[8 * c + i], cs[i], sn[i]);
      rotate8_regs(klo[k], khi[k], dst, d, c, rope, cs, sn);
    }
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
  dim3 grid(B * Hkv, (Tn + kTokens - 1) / kTokens);
  cache_append_kernel<<<grid, kThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
      static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache), cache_lens,
      block_table, Hkv, Tn, Lmax, d, page_size, num_pages, max_pages, rope, theta, status);
  return cudaGetLastError();
}

}  // namespace csattn
