// RoPE on bf16 keys, once per call: x_rot[b,h,t,:] = R_{pos0+t} x[b,h,t,:], rounded
// to bf16 (round-to-nearest-even) as the pages' apply_rope returns the input
// dtype ("The Transformer architecture" (cooking-agi), section "Now: RoPE";
// angle pos * base^(-2p/d) from "Transformer" (ai-notes), RoPE section).
//
// Each key tile is read by every query tile at or below it, so rotating keys
// inside the attention kernel would repeat the same rotation T/128 times per
// key; this bandwidth-bound pass does it once (read + write of K).  One thread
// owns 8 channel pairs of one position and applies the same 8 (cos, sin) to
// that position in every head of the batch entry, so the angles are computed
// once per (b, t) rather than once per head.
#include "internal.h"

namespace csattn {
namespace {

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16lo_to_f32(w[i]);
    f[2 * i + 1] = bf16hi_to_f32(w[i]);
  }
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
  uint4 u;
  u.x = pack_bf16x2(f[0], f[1]);
  u.y = pack_bf16x2(f[2], f[3]);
  u.z = pack_bf16x2(f[4], f[5]);
  u.w = pack_bf16x2(f[6], f[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

// x, x_rot: [B, H, T, d]; thread -> (b, t, c) with c in [0, d/16): pairs 8c..8c+7.
__global__ void __launch_bounds__(256) rope_rotate_bf16_kernel(
    const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ x_rot, int B, int H, int T,
    int d, int layout, RopeTable theta, int pos0) {
  const int chunks = d / 16;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)B * T * chunks;
  if (idx >= total) return;
  const int c = static_cast<int>(idx % chunks);
  const int t = static_cast<int>((idx / chunks) % T);
  const int b = static_cast<int>(idx / ((long long)chunks * T));

  float cs[8], sn[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int p = 8 * c + i;
    rope_cos_sin<false>(pos0 + t, theta.hi[p], theta.lo[p], cs[i], sn[i]);
  }
  // element offsets of the two 8-wide vectors this thread rotates
  int e0, e1;
  if (layout == 1) {  // split-half: channel p with p + d/2
    e0 = 8 * c;
    e1 = d / 2 + 8 * c;
  } else {  // adjacent: channels 16c..16c+15 hold pairs 8c..8c+7
    e0 = 16 * c;
    e1 = 16 * c + 8;
  }
  for (int h = 0; h < H; ++h) {
    const size_t base = (((size_t)b * H + h) * (size_t)T + t) * d;
    float u[8], w[8], ou[8], ow[8];
    load8(x + base + e0, u);
    load8(x + base + e1, w);
    if (layout == 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ou[i] = fmaf(u[i], cs[i], -w[i] * sn[i]);
        ow[i] = fmaf(u[i], sn[i], w[i] * cs[i]);
      }
    } else {
      // pairs (u0,u1),(u2,u3),(u4,u5),(u6,u7) -> pairs 0..3; (w0,w1).. -> pairs 4..7
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ou[2 * i] = fmaf(u[2 * i], cs[i], -u[2 * i + 1] * sn[i]);
        ou[2 * i + 1] = fmaf(u[2 * i], sn[i], u[2 * i + 1] * cs[i]);
        ow[2 * i] = fmaf(w[2 * i], cs[4 + i], -w[2 * i + 1] * sn[4 + i]);
        ow[2 * i + 1] = fmaf(w[2 * i], sn[4 + i], w[2 * i + 1] * cs[4 + i]);
      }
    }
    store8(x_rot + base + e0, ou);
    store8(x_rot + base + e1, ow);
  }
}

}  // namespace

cudaError_t launch_rope_rotate_bf16(const void* x, void* x_rot, int B, int H, int T, int d,
                                    int rope, const RopeTable& theta, cudaStream_t stream,
                                    int pos0) {
  const long long total = (long long)B * T * (d / 16);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  rope_rotate_bf16_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(x_rot), B, H, T, d, rope,
      theta, pos0);
  return cudaGetLastError();
}

}  // namespace csattn
