// Backward of causal GQA attention for fp32 inputs on the SIMT cores (FFMA), for
// fp32 callers that need the gradients close to float64: the same math as
// bwd.cu (P = exp(S - lse), D = rowsum(dout o out), dS = P o (dout V^T - D),
// dV = P^T dout, dQ = R^T(scale dS Kr), dK = R^T(scale dS^T Qr)).  Head sizes d (q,
// k) and dv (v, out) each in {16, 32, 64, 128}; Tq query rows at positions
// q_off..q_off+Tq-1, Tk keys at 0..Tk-1.  A row is served by TPR = max(d, dv)/16
// threads, each holding d/TPR channels of the q/k side and dv/TPR of the v/dout side.
//
//   rope_f32_kernel     x_rot = R x at positions pos0 + t (accurate sine/cosine); also
//                       csattn_rope_rotate's fp32 path
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

template <int D, int DV>
struct BwdF32Cfg {
  static constexpr int DMAX = D > DV ? D : DV;
  static constexpr int TPR = DMAX / 16;        // threads per row
  static constexpr int ROWS = kThreads / TPR;  // rows per CTA
  static constexpr int QC = D / TPR;           // q / k channels per thread (2..16)
  static constexpr int VC = DV / TPR;          // v / dout channels per thread (2..16)
  static constexpr int KT = (DMAX == 128) ? 16 : 32;  // staged rows of the other side
};

// x_rot[row] = R_pos x[row] for rows of [B*H, T, d], pos = pos0 + row % T; one thread per pair.
__global__ void __launch_bounds__(256) rope_f32_kernel(const float* __restrict__ x,
                                                       float* __restrict__ x_rot, long long rows,
                                                       int T, int d, int layout, RopeTable theta,
                                                       int pos0) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int half = d / 2;
  if (idx >= rows * half) return;
  const long long r = idx / half;
  const int pair = static_cast<int>(idx - r * half);
  const int pos = pos0 + static_cast<int>(r % T);
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

// N consecutive floats (N = 2, 4, 8 or 16) from shared memory aligned to 4N bytes
// (N <= 4) or 16 bytes.
template <int N>
__device__ __forceinline__ void load_n(const float* src, float (&dst)[N]) {
  if constexpr (N == 2) {
    const float2 t = *reinterpret_cast<const float2*>(src);
    dst[0] = t.x;
    dst[1] = t.y;
  } else {
#pragma unroll
    for (int c4 = 0; c4 < N / 4; ++c4) {
      const float4 t = reinterpret_cast<const float4*>(src)[c4];
      dst[4 * c4] = t.x;
      dst[4 * c4 + 1] = t.y;
      dst[4 * c4 + 2] = t.z;
      dst[4 * c4 + 3] = t.w;
    }
  }
}

struct BwdF32Params {
  const float* qr;    // [B, Hq, Tq, D]
  const float* kr;    // [B, Hkv, Tk, D]
  const float* v;     // [B, Hkv, Tk, DV]
  const float* dout;  // [B, Hq, Tq, DV]
  const float* lse;
  const float* dvec;
  float* dq;
  float* dk;
  float* dv;
  int Hq, Hkv, Tq, Tk, q_off, causal, rope;
  float scale;
  RopeTable theta;
};

template <int D, int DV>
__global__ void __launch_bounds__(kThreads) bwd_dq_f32_kernel(const BwdF32Params p) {
  using C = BwdF32Cfg<D, DV>;
  constexpr int QC = C::QC, VC = C::VC;
  __shared__ __align__(16) float sk[C::KT * D];
  __shared__ __align__(16) float sv[C::KT * DV];
  __shared__ __align__(16) float srow[C::ROWS * D];
  const int tid = threadIdx.x, row = tid / C::TPR, part = tid % C::TPR;
  const int h = blockIdx.y, b = blockIdx.z, g = h / (p.Hq / p.Hkv);
  const int q0 = blockIdx.x * C::ROWS, qi = q0 + row;
  const bool live = qi < p.Tq;
  const size_t qrow = (static_cast<size_t>(b) * p.Hq + h) * p.Tq + (live ? qi : 0);
  float q[QC], o[VC], acc[QC];
#pragma unroll
  for (int c = 0; c < QC; ++c) {
    q[c] = live ? p.qr[qrow * D + part * QC + c] : 0.f;
    acc[c] = 0.f;
  }
#pragma unroll
  for (int c = 0; c < VC; ++c) o[c] = live ? p.dout[qrow * DV + part * VC + c] : 0.f;
  const float lse2 = live ? p.lse[qrow] * kLog2e : 0.f;
  const float dd = live ? p.dvec[qrow] : 0.f;
  const float* kh = p.kr + (static_cast<size_t>(b) * p.Hkv + g) * p.Tk * D;
  const float* vh = p.v + (static_cast<size_t>(b) * p.Hkv + g) * p.Tk * DV;
  // causal: keys up to the position of the CTA's last row
  const int k_end = p.causal ? min(p.Tk, p.q_off + q0 + C::ROWS) : p.Tk;
  for (int k0 = 0; k0 < k_end; k0 += C::KT) {
    const int nk = min(C::KT, k_end - k0);
    __syncthreads();
    for (int e = tid; e < C::KT * D; e += kThreads) {
      const int r = e / D;
      sk[e] = r < nk ? kh[static_cast<size_t>(k0 + r) * D + e % D] : 0.f;
    }
    for (int e = tid; e < C::KT * DV; e += kThreads) {
      const int r = e / DV;
      sv[e] = r < nk ? vh[static_cast<size_t>(k0 + r) * DV + e % DV] : 0.f;
    }
    __syncthreads();
    for (int j = 0; j < nk; ++j) {
      float kk[QC], vv[VC];
      load_n<QC>(sk + j * D + part * QC, kk);
      load_n<VC>(sv + j * DV + part * VC, vv);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int c = 0; c < QC; ++c) s = fmaf(q[c], kk[c], s);
#pragma unroll
      for (int c = 0; c < VC; ++c) dp = fmaf(o[c], vv[c], dp);
#pragma unroll
      for (int off = 1; off < C::TPR; off <<= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, off);
        dp += __shfl_xor_sync(0xffffffffu, dp, off);
      }
      const int key = k0 + j;
      if (!live || (p.causal && key > p.q_off + qi)) continue;
      const float pr = exp2f(fmaf(s * p.scale, kLog2e, -lse2));
      const float ds = pr * (dp - dd) * p.scale;
#pragma unroll
      for (int c = 0; c < QC; ++c) acc[c] = fmaf(ds, kk[c], acc[c]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < QC; ++c) srow[row * D + part * QC + c] = acc[c];
  __syncwarp();
  if (p.rope) rotate_back_row(srow + row * D, D, C::TPR, part, p.rope, p.q_off + qi, p.theta);
  __syncwarp();
  if (live) {
#pragma unroll
    for (int c = 0; c < QC; ++c) p.dq[qrow * D + part * QC + c] = srow[row * D + part * QC + c];
  }
}

template <int D, int DV>
__global__ void __launch_bounds__(kThreads) bwd_dkdv_f32_kernel(const BwdF32Params p) {
  using C = BwdF32Cfg<D, DV>;
  constexpr int QC = C::QC, VC = C::VC;
  __shared__ __align__(16) float sq[C::KT * D];
  __shared__ __align__(16) float so[C::KT * DV];
  __shared__ float slse[C::KT];
  __shared__ float sdd[C::KT];
  __shared__ __align__(16) float srow[C::ROWS * D];
  const int tid = threadIdx.x, row = tid / C::TPR, part = tid % C::TPR;
  const int g = blockIdx.y, b = blockIdx.z, rep = p.Hq / p.Hkv;
  const int k0 = blockIdx.x * C::ROWS, kj = k0 + row;
  const bool live = kj < p.Tk;
  const size_t krow = (static_cast<size_t>(b) * p.Hkv + g) * p.Tk + (live ? kj : 0);
  float k[QC], v[VC], adk[QC], adv[VC];
#pragma unroll
  for (int c = 0; c < QC; ++c) {
    k[c] = live ? p.kr[krow * D + part * QC + c] : 0.f;
    adk[c] = 0.f;
  }
#pragma unroll
  for (int c = 0; c < VC; ++c) {
    v[c] = live ? p.v[krow * DV + part * VC + c] : 0.f;
    adv[c] = 0.f;
  }
  // causal: the first query row that sees key k0 sits at position k0
  const int q_begin = p.causal ? max(0, k0 - p.q_off) : 0;
  for (int hh = 0; hh < rep; ++hh) {
    const int h = g * rep + hh;
    const size_t qbase = (static_cast<size_t>(b) * p.Hq + h) * p.Tq;
    for (int i0 = q_begin; i0 < p.Tq; i0 += C::KT) {
      const int ni = min(C::KT, p.Tq - i0);
      __syncthreads();
      for (int e = tid; e < C::KT * D; e += kThreads) {
        const int r = e / D;
        sq[e] = r < ni ? p.qr[(qbase + i0 + r) * D + e % D] : 0.f;
      }
      for (int e = tid; e < C::KT * DV; e += kThreads) {
        const int r = e / DV;
        so[e] = r < ni ? p.dout[(qbase + i0 + r) * DV + e % DV] : 0.f;
      }
      for (int e = tid; e < C::KT; e += kThreads) {
        slse[e] = e < ni ? p.lse[qbase + i0 + e] * kLog2e : 0.f;
        sdd[e] = e < ni ? p.dvec[qbase + i0 + e] : 0.f;
      }
      __syncthreads();
      for (int i = 0; i < ni; ++i) {
        float qq[QC], oo[VC];
        load_n<QC>(sq + i * D + part * QC, qq);
        load_n<VC>(so + i * DV + part * VC, oo);
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int c = 0; c < QC; ++c) s = fmaf(qq[c], k[c], s);
#pragma unroll
        for (int c = 0; c < VC; ++c) dp = fmaf(oo[c], v[c], dp);
#pragma unroll
        for (int off = 1; off < C::TPR; off <<= 1) {
          s += __shfl_xor_sync(0xffffffffu, s, off);
          dp += __shfl_xor_sync(0xffffffffu, dp, off);
        }
        const int qi = i0 + i;
        if (!live || (p.causal && kj > p.q_off + qi)) continue;
        const float pr = exp2f(fmaf(s * p.scale, kLog2e, -slse[i]));
        const float ds = pr * (dp - sdd[i]) * p.scale;
#pragma unroll
        for (int c = 0; c < VC; ++c) adv[c] = fmaf(pr, oo[c], adv[c]);
#pragma unroll
        for (int c = 0; c < QC; ++c) adk[c] = fmaf(ds, qq[c], adk[c]);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < QC; ++c) srow[row * D + part * QC + c] = adk[c];
  __syncwarp();
  if (p.rope) rotate_back_row(srow + row * D, D, C::TPR, part, p.rope, kj, p.theta);
  __syncwarp();
  if (live) {
#pragma unroll
    for (int c = 0; c < QC; ++c) p.dk[krow * D + part * QC + c] = srow[row * D + part * QC + c];
#pragma unroll
    for (int c = 0; c < VC; ++c) p.dv[krow * DV + part * VC + c] = adv[c];
  }
}

template <int D, int DV>
cudaError_t launch_f32_d(const BwdF32Params& p, int B, cudaStream_t stream) {
  using C = BwdF32Cfg<D, DV>;
  dim3 gq((p.Tq + C::ROWS - 1) / C::ROWS, p.Hq, B);
  bwd_dq_f32_kernel<D, DV><<<gq, kThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 gk((p.Tk + C::ROWS - 1) / C::ROWS, p.Hkv, B);
  bwd_dkdv_f32_kernel<D, DV><<<gk, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_f32_dv(const BwdF32Params& p, int B, int dv, cudaStream_t stream) {
  switch (dv) {
    case 16: return launch_f32_d<D, 16>(p, B, stream);
    case 32: return launch_f32_d<D, 32>(p, B, stream);
    case 64: return launch_f32_d<D, 64>(p, B, stream);
    case 128: return launch_f32_d<D, 128>(p, B, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_rope_rotate_f32(const void* x, void* x_rot, int B, int H, int T, int d,
                                   int rope, const RopeTable& theta, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * H * T;
  rope_f32_kernel<<<static_cast<unsigned>((rows * (d / 2) + 255) / 256), 256, 0, stream>>>(
      static_cast<const float*>(x), static_cast<float*>(x_rot), rows, T, d, rope, theta, 0);
  return cudaGetLastError();
}

cudaError_t launch_bwd_f32(const BwdArgs& a, void* q_rot, void* k_rot, cudaStream_t stream) {
  const long long qrows = static_cast<long long>(a.B) * a.Hq * a.Tq;
  const long long krows = static_cast<long long>(a.B) * a.Hkv * a.Tk;
  cudaError_t e;
  BwdF32Params p{};
  p.qr = static_cast<const float*>(a.qr);
  p.kr = static_cast<const float*>(a.kr);
  if (a.rope) {
    rope_f32_kernel<<<static_cast<unsigned>((qrows * (a.d / 2) + 255) / 256), 256, 0, stream>>>(
        static_cast<const float*>(a.qr), static_cast<float*>(q_rot), qrows, a.Tq, a.d, a.rope,
        a.theta, a.q_off);
    rope_f32_kernel<<<static_cast<unsigned>((krows * (a.d / 2) + 255) / 256), 256, 0, stream>>>(
        static_cast<const float*>(a.kr), static_cast<float*>(k_rot), krows, a.Tk, a.d, a.rope,
        a.theta, 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.qr = static_cast<const float*>(q_rot);
    p.kr = static_cast<const float*>(k_rot);
  }
  rowdot_f32_kernel<<<static_cast<unsigned>((qrows + 255) / 256), 256, 0, stream>>>(
      static_cast<const float*>(a.dout), static_cast<const float*>(a.out), a.dvec, qrows, a.d_v);
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
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.q_off = a.q_off;
  p.causal = a.causal;
  p.rope = a.rope;
  p.scale = a.scale;
  p.theta = a.theta;
  switch (a.d) {
    case 16: return launch_f32_dv<16>(p, a.B, a.d_v, stream);
    case 32: return launch_f32_dv<32>(p, a.B, a.d_v, stream);
    case 64: return launch_f32_dv<64>(p, a.B, a.d_v, stream);
    case 128: return launch_f32_dv<128>(p, a.B, a.d_v, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csattn
