// RoPE on bf16 keys, once per call: x_rot[b,h,t,:] = R_{pos0+t} x[b,h,t,:], rounded
// to bf16 (round-to-nearest-even) as the pages' apply_rope returns the input
// dtype ("The Transformer architecture" (cooking-agi), section "Now: RoPE";
// angle pos * base^(-2p/d) from "Transformer" (ai-notes), RoPE section).
//
// Each key tile is read by every query tile at or below it, so rotating keys
// inside the attention kernel would repeat the same rotation T/128 times per
// key; this bandwidth-bound pass does it once (read + write of K).  One thread
// owns 8 channel pairs of one position and applies the same 8 (cos, sin) to
// that position in up to 4 heads of the batch entry, so the angles are computed
// once per (b, t) and head group rather than once per head.
#include "internal.h"

namespace csattn {
namespace {

// x, x_rot: [B, H, T, d]; thread -> (b, head group, t, c) with c in [0, d/16): pairs
// 8c..8c+7 of position pos0 + t in the kRopeHeads heads of the group.  The thread
// issues the loads of all of its heads, then computes the 8 angles while they are in
// flight, then rotates and stores (a loop of load-rotate-store per head keeps two
// loads in flight per thread and leaves the kernel waiting on memory).
constexpr int kRopeHeads = 4;

__global__ void __launch_bounds__(256) rope_rotate_bf16_kernel(
    const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ x_rot, int B, int H, int T,
    int d, int layout, RopeTable theta, int pos0) {
  const int chunks = d / 16;
  const int groups = (H + kRopeHeads - 1) / kRopeHeads;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)B * groups * T * chunks;
  if (idx >= total) return;
  const int c = static_cast<int>(idx % chunks);
  const int t = static_cast<int>((idx / chunks) % T);
  const long long bg = idx / ((long long)chunks * T);
  const int hgrp = static_cast<int>(bg % groups);
  const int b = static_cast<int>(bg / groups);
  const int h0 = hgrp * kRopeHeads;
  // element offsets of the two 8-wide vectors this thread rotates
  int e0, e1;
  if (layout == 1) {  // split-half: channel p with p + d/2
    e0 = 8 * c;
    e1 = d / 2 + 8 * c;
  } else {  // adjacent: channels 16c..16c+15 hold pairs 8c..8c+7
    e0 = 16 * c;
    e1 = 16 * c + 8;
  }
  uint4 lo[kRopeHeads], hi[kRopeHeads];
#pragma unroll
  for (int k = 0; k < kRopeHeads; ++k) {
    if (h0 + k < H) {
      const size_t base = (((size_t)b * H + h0 + k) * (size_t)T + t) * d;
      lo[k] = __ldg(reinterpret_cast<const uint4*>(x + base + e0));
      hi[k] = __ldg(reinterpret_cast<const uint4*>(x + base + e1));
    }
  }
  float cs[8], sn[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int p = 8 * c + i;
    rope_cos_sin<false>(pos0 + t, theta.hi[p], theta.lo[p], cs[i], sn[i]);
  }
#pragma unroll
  for (int k = 0; k < kRopeHeads; ++k) {
    if (h0 + k >= H) continue;
    const size_t base = (((size_t)b * H + h0 + k) * (size_t)T + t) * d;
    // one 32-bit word of each half at a time: the pairs of word i are (u_j, w_j), j = 2i,
    // 2i + 1 (split-half), or (u0, u1) = pair i and (w0, w1) = pair 4 + i (adjacent)
    uint32_t wa[4] = {lo[k].x, lo[k].y, lo[k].z, lo[k].w};
    uint32_t wb[4] = {hi[k].x, hi[k].y, hi[k].z, hi[k].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float u0 = bf16lo_to_f32(wa[i]), u1 = bf16hi_to_f32(wa[i]);
      const float w0 = bf16lo_to_f32(wb[i]), w1 = bf16hi_to_f32(wb[i]);
      if (layout == 1) {
        wa[i] = pack_bf16x2(fmaf(u0, cs[2 * i], -w0 * sn[2 * i]),
                            fmaf(u1, cs[2 * i + 1], -w1 * sn[2 * i + 1]));
        wb[i] = pack_bf16x2(fmaf(u0, sn[2 * i], w0 * cs[2 * i]),
                            fmaf(u1, sn[2 * i + 1], w1 * cs[2 * i + 1]));
      } else {
        wa[i] = pack_bf16x2(fmaf(u0, cs[i], -u1 * sn[i]), fmaf(u0, sn[i], u1 * cs[i]));
        wb[i] = pack_bf16x2(fmaf(w0, cs[4 + i], -w1 * sn[4 + i]),
                            fmaf(w0, sn[4 + i], w1 * cs[4 + i]));
      }
    }
    *reinterpret_cast<uint4*>(x_rot + base + e0) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
    *reinterpret_cast<uint4*>(x_rot + base + e1) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
  }
}

}  // namespace

cudaError_t launch_rope_rotate_bf16(const void* x, void* x_rot, int B, int H, int T, int d,
                                    int rope, const RopeTable& theta, cudaStream_t stream,
                                    int pos0) {
  const long long total =
      (long long)B * ((H + kRopeHeads - 1) / kRopeHeads) * T * (d / 16);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  rope_rotate_bf16_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(x_rot), B, H, T, d, rope,
      theta, pos0);
  return cudaGetLastError();
}

}  // namespace csattn
