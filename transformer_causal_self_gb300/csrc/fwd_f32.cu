// fp32 prefill attention on the SIMT cores (FFMA), for the fp32 workloads that
// must match the oracle to 1e-5: tensor-core TF32 would miss that bound.
//
// One CTA owns ROWS query rows of one (batch, q-head); max(DK, DV)/16 threads
// share a row, each with up to 16 channels of the query (DK channels) and of the
// output (DV channels: v may be narrower or wider than q and k).  K/V tiles are staged in shared memory, RoPE is
// applied there (keys) and to the staged query rows, and each row keeps an
// online softmax (running max m, running sum l, accumulator) in fp32:
//   s = q.k * scale;  m' = max(m, s);  l = l e^{m-m'} + e^{s-m'};
//   acc = acc e^{m-m'} + e^{s-m'} v.
// Keys after the query's position are skipped under the causal mask
// ("Transformer Math and Implementation Deep Dive", section "Causal Masking").
#include "internal.h"

namespace csattn {
namespace {

constexpr int kThreads = 128;

template <int DK, int DV>
struct F32Cfg {
  static constexpr int D = DK > DV ? DK : DV;
  static constexpr int TPR = D / 16;           // threads per query row
  static constexpr int ROWS = kThreads / TPR;  // query rows per CTA
  static constexpr int KT = (D == 128) ? 32 : 64;
};

__device__ __forceinline__ void rotate_row_f32(float* row, int D, int pair, int layout, int pos,
                                               const RopeTable& th) {
  int i, j;
  if (layout == 1) {
    i = pair;
    j = pair + D / 2;
  } else {
    i = 2 * pair;
    j = 2 * pair + 1;
  }
  float c, s;
  rope_cos_sin<true>(pos, th.hi[pair], th.lo[pair], c, s);
  const float a = row[i], b = row[j];
  row[i] = fmaf(a, c, -b * s);
  row[j] = fmaf(a, s, b * c);
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) fwd_f32_kernel(const float* __restrict__ q,
                                                           const float* __restrict__ k,
                                                           const float* __restrict__ v,
                                                           float* __restrict__ out,
                                                           float* __restrict__ lse, int Hq,
                                                           int Hkv, int Tq, int Tk, int q_off,
                                                           int causal, int rope,
                                                           int rope_k, float scale,
                                                           RopeTable theta) {
  using C = F32Cfg<DK, DV>;
  __shared__ float sq[C::ROWS * DK];
  __shared__ float sk[C::KT * DK];
  __shared__ float sv[C::KT * DV];

  const int tid = threadIdx.x;
  const int row = tid / C::TPR;
  const int part = tid % C::TPR;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int g = h / (Hq / Hkv);
  const int q0 = blockIdx.x * C::ROWS;
  const int qpos = q0 + row;      // row of q / out
  const int qabs = q_off + qpos;  // its position

  const float* qh = q + ((size_t)b * Hq + h) * (size_t)Tq * DK;
  const float* kh = k + ((size_t)b * Hkv + g) * (size_t)Tk * DK;
  const float* vh = v + ((size_t)b * Hkv + g) * (size_t)Tk * DV;
  const bool has_q = part * 16 < DK;  // this thread's 16 query / key channels exist
  const bool has_v = part * 16 < DV;  // this thread's 16 value / output channels exist

  for (int e = tid; e < C::ROWS * DK; e += kThreads) {
    const int r = e / DK;
    sq[e] = (q0 + r < Tq) ? qh[(size_t)(q0 + r) * DK + (e % DK)] : 0.f;
  }
  __syncthreads();
  if (rope) {
    for (int e = tid; e < C::ROWS * (DK / 2); e += kThreads) {
      const int r = e / (DK / 2);
      rotate_row_f32(sq + r * DK, DK, e % (DK / 2), rope, q_off + q0 + r, theta);
    }
    __syncthreads();
  }
  float qr[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) qr[c] = has_q ? sq[row * DK + part * 16 + c] : 0.f;

  float m = -INFINITY, l = 0.f;
  float acc[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) acc[c] = 0.f;

  const int kv_end = causal ? min(Tk, q_off + q0 + C::ROWS) : Tk;
  for (int k0 = 0; k0 < kv_end; k0 += C::KT) {
    const int nk = min(C::KT, kv_end - k0);
    __syncthreads();
    for (int e = tid; e < C::KT * DK; e += kThreads) {
      const int r = e / DK;
      sk[e] = r < nk ? kh[(size_t)(k0 + r) * DK + (e % DK)] : 0.f;
    }
    for (int e = tid; e < C::KT * DV; e += kThreads) {
      const int r = e / DV;
      sv[e] = r < nk ? vh[(size_t)(k0 + r) * DV + (e % DV)] : 0.f;
    }
    __syncthreads();
    if (rope_k) {
      for (int e = tid; e < nk * (DK / 2); e += kThreads) {
        const int r = e / (DK / 2);
        rotate_row_f32(sk + r * DK, DK, e % (DK / 2), rope, k0 + r, theta);
      }
      __syncthreads();
    }
    for (int j = 0; j < nk; ++j) {
      float dot = 0.f;
      if (has_q) {
#pragma unroll
        for (int c = 0; c < 16; ++c) dot = fmaf(qr[c], sk[j * DK + part * 16 + c], dot);
      }
#pragma unroll
      for (int off = 1; off < C::TPR; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const int key = k0 + j;
      if (causal && key > qabs) continue;
      const float s = dot * scale;
      if (s > m) {
        const float corr = expf(m - s);
        l *= corr;
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[c] *= corr;
        m = s;
      }
      const float p = expf(s - m);
      l += p;
      if (has_v) {
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[c] = fmaf(p, sv[j * DV + part * 16 + c], acc[c]);
      }
    }
  }

  if (qpos < Tq) {
    const float inv = 1.f / l;
    if (has_v) {
      float* o = out + (((size_t)b * Hq + h) * (size_t)Tq + qpos) * DV + part * 16;
#pragma unroll
      for (int c = 0; c < 16; ++c) o[c] = acc[c] * inv;
    }
    if (lse != nullptr && part == 0) lse[((size_t)b * Hq + h) * (size_t)Tq + qpos] = m + logf(l);
  }
}

template <int DK, int DV>
cudaError_t launch_d(const FwdArgs& a, cudaStream_t stream) {
  using C = F32Cfg<DK, DV>;
  dim3 grid((a.Tq + C::ROWS - 1) / C::ROWS, a.Hq, a.B);
  fwd_f32_kernel<DK, DV><<<grid, kThreads, 0, stream>>>(
      static_cast<const float*>(a.q), static_cast<const float*>(a.k),
      static_cast<const float*>(a.v), static_cast<float*>(a.out), a.lse, a.Hq, a.Hkv, a.Tq, a.Tk,
      a.q_off, a.causal, a.rope, a.rope_k, a.scale, a.theta);
  return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const FwdArgs& a, cudaStream_t stream) {
  switch (a.dv) {
    case 16: return launch_d<DK, 16>(a, stream);
    case 32: return launch_d<DK, 32>(a, stream);
    case 64: return launch_d<DK, 64>(a, stream);
    case 128: return launch_d<DK, 128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 16: return launch_dk<16>(a, stream);
    case 32: return launch_dk<32>(a, stream);
    case 64: return launch_dk<64>(a, stream);
    case 128: return launch_dk<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csattn
