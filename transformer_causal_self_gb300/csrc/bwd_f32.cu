// Backward of causal GQA attention for fp32 inputs on the SIMT cores (FFMA), for
// fp32 callers that need the gradients close to float64: the same math as
// bwd.cu (P = exp(S - lse), D = rowsum(dout o out), dS = P o (dout V^T - D),
// dV = P^T dout, dQ = R^T(scale dS Kr), dK = R^T(scale dS^T Qr)), one thread
// group of d/16 threads per row, 16 channels each.
//
//   rope_f32_kernel     x_rot = R x at positions 0..T-1 (accurate sine/cosine)
//   rowdot_f32_kernel   D
//   bwd_dq_f32_kernel   one CTA per (ROWS query rows, query head, batch); K and V
//                       tiles staged in shared memory; dq rotated back at the end
//   bwd_dkdv_f32_kernel one CTA per (ROWS key rows, KV head, batch); loops over the
//                       group's query heads and the query tiles that see the keys
#include "internal.h"

namespace csattn {
namespace {

constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdF32Cfg {
  static constexpr int TPR = D / 16;           // threads per row
  static constexpr int ROWS = kThreads / TPR;  // rows per CTA
  static constexpr int KT = (D == 128) ? 16 : 32;  // staged rows of the other side
};

// x_rot[row] = R_pos x[row] for rows of [B*H, T, d], pos = row % T; one thread per pair.
__global__ void __launch_bounds__(256) rope_f32_kernel(const float* __restrict__ x,
                                                       float* __restrict__ x_rot, long long rows,
                                                       int T, int d, int layout,
                                                       RopeTable theta) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int half = d / 2;
  if (idx >= rows * half) return;
  const long long r = idx / half;
  const int pair = static_cast<int>(idx - r * half);
  const int pos = static_cast<int>(r % T);
  int i, j;
  if (layout == 1) {
    i = pair;
    j = pair + half;
  } else {
    i = 2 * pair;
    j = 2 * pair + 1;
  }
  float c, s;
  rope_cos_sin<true>(pos, theta.hi[pair], theta.lo[pair], c, s);
  const float a = x[r * d + i], b = x[r * d + j];
  x_rot[r * d + i] = fmaf(a, c, -b * s);
  x_rot[r * d + j] = fmaf(a, s, b * c);
}

__global__ void __launch_bounds__(256) rowdot_f32_kernel(const float* __restrict__ dout,
                                                         const float* __restrict__ out,
                                                         float* __restrict__ dvec,
                                                         long long rows, int d) {
  const long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  float acc = 0.f;
  for (int c = 0; c < d; ++c) acc = fmaf(dout[r * d + c], out[r * d + c], acc);
  dvec[r] = acc;
}

// R^T applied in place to a row of d channels held in shared memory (thread `part`
// of the row's group owns pairs part, part + TPR, ...).
__device__ __forceinline__ void rotate_back_row(float* row, int d, int tpr, int part, int layout,
                                                int pos, const RopeTable& th) {
  for (int pair = part; pair < d / 2; pair += tpr) {
    int i, j;
    if (layout == 1) {
      i = pair;
      j = pair + d / 2;
    } else {
      i = 2 * pair;
      j = 2 * pair + 1;
    }
    float c, s;
    rope_cos_sin<true>(pos, th.hi[pair], th.lo[pair], c, s);
    const float a = row[i], b = row[j];
    row[i] = fmaf(a, c, b * s);
    row[j] = fmaf(-a, s, b * c);
  }
}

// 16 consecutive floats from 16-byte aligned shared memory.
__device__ __forceinline__ void load16(const float* src, float (&dst)[16]) {
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    const float4 t = reinterpret_cast<const float4*>(src)[c4];
    dst[4 * c4] = t.x;
    dst[4 * c4 + 1] = t.y;
    dst[4 * c4 + 2] = t.z;
    dst[4 * c4 + 3] = t.w;
  }
}

struct BwdF32Params {
  const float* qr;
  const float* kr;
  const float* v;
  const float* dout;
  const float* lse;
  const float* dvec;
  float* dq;
  float* dk;
  float* dv;
  int Hq, Hkv, T, causal, rope;
  float scale;
  RopeTable theta;
};

template <int D>
__global__ void __launch_bounds__(kThreads) bwd_dq_f32_kernel(const BwdF32Params p) {
  using C = BwdF32Cfg<D>;
  __shared__ __align__(16) float sk[C::KT * D];
  __shared__ __align__(16) float sv[C::KT * D];
  __shared__ __align__(16) float srow[C::ROWS * D];
  const int tid = threadIdx.x, row = tid / C::TPR, part = tid % C::TPR;
  const int h = blockIdx.y, b = blockIdx.z, g = h / (p.Hq / p.Hkv);
  const int q0 = blockIdx.x * C::ROWS, qi = q0 + row;
  const bool live = qi < p.T;
  const size_t qrow = (static_cast<size_t>(b) * p.Hq + h) * p.T + (live ? qi : 0);
  float q[16], o[16], acc[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    q[c] = live ? p.qr[qrow * D + part * 16 + c] : 0.f;
    o[c] = live ? p.dout[qrow * D + part * 16 + c] : 0.f;
    acc[c] = 0.f;
  }
  const float lse2 = live ? p.lse[qrow] * kLog2e : 0.f;
  const float dd = live ? p.dvec[qrow] : 0.f;
  const float* kh = p.kr + (static_cast<size_t>(b) * p.Hkv + g) * p.T * D;
  const float* vh = p.v + (static_cast<size_t>(b) * p.Hkv + g) * p.T * D;
  const int k_end = p.causal ? min(p.T, q0 + C::ROWS) : p.T;
  for (int k0 = 0; k0 < k_end; k0 += C::KT) {
    const int nk = min(C::KT, k_end - k0);
    __syncthreads();
    for (int e = tid; e < C::KT * D; e += kThreads) {
      const int r = e / D;
      sk[e] = r < nk ? kh[static_cast<size_t>(k0 + r) * D + e % D] : 0.f;
      sv[e] = r < nk ? vh[static_cast<size_t>(k0 + r) * D + e % D] : 0.f;
    }
    __syncthreads();
    for (int j = 0; j < nk; ++j) {
      float kk[16], vv[16];
      load16(sk + j * D + part * 16, kk);
      load16(sv + j * D + part * 16, vv);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        s = fmaf(q[c], kk[c], s);
        dp = fmaf(o[c], vv[c], dp);
      }
#pragma unroll
      for (int off = 1; off < C::TPR; off <<= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, off);
        dp += __shfl_xor_sync(0xffffffffu, dp, off);
      }
      const int key = k0 + j;
      if (!live || (p.causal && key > qi)) continue;
      const float pr = exp2f(fmaf(s * p.scale, kLog2e, -lse2));
      const float ds = pr * (dp - dd) * p.scale;
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[c] = fmaf(ds, kk[c], acc[c]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < 16; ++c) srow[row * D + part * 16 + c] = acc[c];
  __syncwarp();
  if (p.rope) rotate_back_row(srow + row * D, D, C::TPR, part, p.rope, qi, p.theta);
  __syncwarp();
  if (live) {
#pragma unroll
    for (int c = 0; c < 16; ++c) p.dq[qrow * D + part * 16 + c] = srow[row * D + part * 16 + c];
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) bwd_dkdv_f32_kernel(const BwdF32Params p) {
  using C = BwdF32Cfg<D>;
  __shared__ __align__(16) float sq[C::KT * D];
  __shared__ __align__(16) float so[C::KT * D];
  __shared__ float slse[C::KT];
  __shared__ float sdd[C::KT];
  __shared__ __align__(16) float srow[C::ROWS * D];
  const int tid = threadIdx.x, row = tid / C::TPR, part = tid % C::TPR;
  const int g = blockIdx.y, b = blockIdx.z, rep = p.Hq / p.Hkv;
  const int k0 = blockIdx.x * C::ROWS, kj = k0 + row;
  const bool live = kj < p.T;
  const size_t krow = (static_cast<size_t>(b) * p.Hkv + g) * p.T + (live ? kj : 0);
  float k[16], v[16], adk[16], adv[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    k[c] = live ? p.kr[krow * D + part * 16 + c] : 0.f;
    v[c] = live ? p.v[krow * D + part * 16 + c] : 0.f;
    adk[c] = 0.f;
    adv[c] = 0.f;
  }
  const int q_begin = p.causal ? k0 : 0;
  for (int hh = 0; hh < rep; ++hh) {
    const int h = g * rep + hh;
    const size_t qbase = (static_cast<size_t>(b) * p.Hq + h) * p.T;
    for (int i0 = q_begin; i0 < p.T; i0 += C::KT) {
      const int ni = min(C::KT, p.T - i0);
      __syncthreads();
      for (int e = tid; e < C::KT * D; e += kThreads) {
        const int r = e / D;
        sq[e] = r < ni ? p.qr[(qbase + i0 + r) * D + e % D] : 0.f;
        so[e] = r < ni ? p.dout[(qbase + i0 + r) * D + e % D] : 0.f;
      }
      for (int e = tid; e < C::KT; e += kThreads) {
        slse[e] = e < ni ? p.lse[qbase + i0 + e] * kLog2e : 0.f;
        sdd[e] = e < ni ? p.dvec[qbase + i0 + e] : 0.f;
      }
      __syncthreads();
      for (int i = 0; i < ni; ++i) {
        float qq[16], oo[16];
        load16(sq + i * D + part * 16, qq);
        load16(so + i * D + part * 16, oo);
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          s = fmaf(qq[c], k[c], s);
          dp = fmaf(oo[c], v[c], dp);
        }
#pragma unroll
        for (int off = 1; off < C::TPR; off <<= 1) {
          s += __shfl_xor_sync(0xffffffffu, s, off);
          dp += __shfl_xor_sync(0xffffffffu, dp, off);
        }
        const int qi = i0 + i;
        if (!live || (p.causal && kj > qi)) continue;
        const float pr = exp2f(fmaf(s * p.scale, kLog2e, -slse[i]));
        const float ds = pr * (dp - sdd[i]) * p.scale;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          adv[c] = fmaf(pr, oo[c], adv[c]);
          adk[c] = fmaf(ds, qq[c], adk[c]);
        }
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < 16; ++c) srow[row * D + part * 16 + c] = adk[c];
  __syncwarp();
  if (p.rope) rotate_back_row(srow + row * D, D, C::TPR, part, p.rope, kj, p.theta);
  __syncwarp();
  if (live) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      p.dk[krow * D + part * 16 + c] = srow[row * D + part * 16 + c];
      p.dv[krow * D + part * 16 + c] = adv[c];
    }
  }
}

template <int D>
cudaError_t launch_f32_d(const BwdF32Params& p, int B, cudaStream_t stream) {
  using C = BwdF32Cfg<D>;
  dim3 gq((p.T + C::ROWS - 1) / C::ROWS, p.Hq, B);
  bwd_dq_f32_kernel<D><<<gq, kThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 gk((p.T + C::ROWS - 1) / C::ROWS, p.Hkv, B);
  bwd_dkdv_f32_kernel<D><<<gk, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_f32(const BwdArgs& a, void* q_rot, void* k_rot, cudaStream_t stream) {
  if (a.Tq != a.Tk || a.q_off != 0) return cudaErrorInvalidValue;
  const long long qrows = static_cast<long long>(a.B) * a.Hq * a.Tq;
  const long long krows = static_cast<long long>(a.B) * a.Hkv * a.Tk;
  cudaError_t e;
  BwdF32Params p{};
  p.qr = static_cast<const float*>(a.qr);
  p.kr = static_cast<const float*>(a.kr);
  if (a.rope) {
    rope_f32_kernel<<<static_cast<unsigned>((qrows * (a.d / 2) + 255) / 256), 256, 0, stream>>>(
        static_cast<const float*>(a.qr), static_cast<float*>(q_rot), qrows, a.Tq, a.d, a.rope,
        a.theta);
    rope_f32_kernel<<<static_cast<unsigned>((krows * (a.d / 2) + 255) / 256), 256, 0, stream>>>(
        static_cast<const float*>(a.kr), static_cast<float*>(k_rot), krows, a.Tk, a.d, a.rope,
        a.theta);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.qr = static_cast<const float*>(q_rot);
    p.kr = static_cast<const float*>(k_rot);
  }
  rowdot_f32_kernel<<<static_cast<unsigned>((qrows + 255) / 256), 256, 0, stream>>>(
      static_cast<const float*>(a.dout), static_cast<const float*>(a.out), a.dvec, qrows, a.d);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  p.v = static_cast<const float*>(a.v);
  p.dout = static_cast<const float*>(a.dout);
  p.lse = a.lse;
  p.dvec = a.dvec;
  p.dq = static_cast<float*>(a.dq);
  p.dk = static_cast<float*>(a.dk);
  p.dv = static_cast<float*>(a.dv);
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.T = a.Tq;
  p.causal = a.causal;
  p.rope = a.rope;
  p.scale = a.scale;
  p.theta = a.theta;
  switch (a.d) {
    case 16: return launch_f32_d<16>(p, a.B, stream);
    case 32: return launch_f32_d<32>(p, a.B, stream);
    case 64: return launch_f32_d<64>(p, a.B, stream);
    case 128: return launch_f32_d<128>(p, a.B, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csattn
