// KV-cache decode for fp32 inputs on the SIMT cores (FFMA), for fp32 callers that
// want the decode close to float64: the query of sequence b sits at position L_b - 1
// and attends to cached rows 0..L_b-1 ("The Transformer architecture" (cooking-agi),
// section "Hands-on", whose incremental decode in fp32 matches the one-shot forward
// to a few 1e-7).  The same split-KV arrangement as the bf16 decode (decode.cu):
//
//   decode_f32_kernel    one CTA per (split, query head, sequence): 32-key tiles of K
//                        and V staged in shared memory, four threads per key for the
//                        score (partial dot products summed by shuffles), an online
//                        softmax in fp32 with expf, one thread per channel for P V;
//                        the split's (m, l, unnormalised o) go to the workspace
//   decode_combine_f32   m = max m_s, l = sum l_s e^(m_s - m), o = sum o_s e^(m_s - m) / l
//
// Natural-log units throughout (m is the maximum scaled score).  Rows at or beyond
// L_b are never read.  Correctness path, not a performance path: the bf16 decode is
// the one tuned for HBM bandwidth.
#include "internal.h"

namespace csattn {
namespace {

constexpr int kThreadsF = 128;
constexpr int kKeysF = 32;    // keys per staged tile
constexpr int kLanesKey = 4;  // threads per key for the dot product

template <int D>
__global__ void __launch_bounds__(kThreadsF) decode_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k_cache,
    const float* __restrict__ v_cache, const int32_t* __restrict__ seq_lens, int len_add,
    float* __restrict__ part_o, float* __restrict__ part_ml, uint32_t* status, int Hq, int Hkv,
    int Lmax, int max_seq_len, int chunk, int n_splits, float scale) {
  __shared__ float sq[D];
  __shared__ float sk[kKeysF][D + 1];  // +1: the score threads read rows, not columns
  __shared__ float sv[kKeysF][D];
  __shared__ float sp[kKeysF];
  __shared__ float s_m[1], s_f[1];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (Hq / Hkv);
  const int tid = static_cast<int>(threadIdx.x);

  const int raw = seq_lens[b];
  int L = raw > max_seq_len ? max_seq_len + 1 : raw + len_add;
  if (L < 1 || L > max_seq_len) {
    if (tid == 0 && split == 0 && h == 0) atomicOr(status, kStatusDeviceArg);
    L = L < 0 ? 0 : (L > max_seq_len ? max_seq_len : L);
  }
  const int k_begin = split * chunk;
  const int k_end = min(L, k_begin + chunk);
  if (k_begin >= k_end) return;  // the merge reads only splits that hold keys

  const size_t row = (static_cast<size_t>(b) * Hq + h) * n_splits + split;
  for (int c = tid; c < D; c += kThreadsF) sq[c] = q[(static_cast<size_t>(b) * Hq + h) * D + c];
  const float* kh = k_cache + (static_cast<size_t>(b) * Hkv + g) * Lmax * D;
  const float* vh = v_cache + (static_cast<size_t>(b) * Hkv + g) * Lmax * D;

  float m = -INFINITY, l = 0.f;  // running maximum and sum (held identically by all threads)
  float acc = 0.f;               // channel tid of the un-normalised output (tid < D)
  const int key = tid / kLanesKey, part = tid % kLanesKey;
  for (int t0 = k_begin; t0 < k_end; t0 += kKeysF) {
    const int nk = min(kKeysF, k_end - t0);
    __syncthreads();
    for (int e = tid; e < kKeysF * D; e += kThreadsF) {
      const int r = e / D, c = e % D;
      sk[r][c] = r < nk ? kh[static_cast<size_t>(t0 + r) * D + c] : 0.f;
      sv[r][c] = r < nk ? vh[static_cast<size_t>(t0 + r) * D + c] : 0.f;
    }
    __syncthreads();
    // score of key `key`: channels part, part + 4, ... summed over the key's 4 threads
    float s = 0.f;
    for (int c = part; c < D; c += kLanesKey) s = fmaf(sq[c], sk[key][c], s);
#pragma unroll
    for (int off = 1; off < kLanesKey; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    s = key < nk ? s * scale : -INFINITY;
    // the tile's maximum, the running maximum and the rescale factor, by one thread
    if (part == 0) sp[key] = s;
    __syncthreads();
    if (tid == 0) {
      float tm = -INFINITY;
      for (int r = 0; r < kKeysF; ++r) tm = fmaxf(tm, sp[r]);
      const float m_new = fmaxf(m, tm);
      s_f[0] = (m == -INFINITY) ? 0.f : expf(m - m_new);
      s_m[0] = m_new;
    }
    __syncthreads();
    const float f = s_f[0];
    m = s_m[0];
    if (part == 0) sp[key] = (key < nk) ? expf(s - m) : 0.f;
    __syncthreads();
    float lt = 0.f;
    for (int r = 0; r < kKeysF; ++r) lt += sp[r];
    l = l * f + lt;
    if (tid < D) {
      float o = acc * f;
      for (int r = 0; r < nk; ++r) o = fmaf(sp[r], sv[r][tid], o);
      acc = o;
    }
  }
  if (tid < D) part_o[row * D + tid] = acc;
  if (tid == 0) {
    part_ml[row * 2 + 0] = m;
    part_ml[row * 2 + 1] = l;
  }
}

// out[b, h, :] = merge of the splits that hold keys of sequence b (natural-log units).
__global__ void decode_combine_f32_kernel(const float* __restrict__ part_o,
                                          const float* __restrict__ part_ml,
                                          const int32_t* __restrict__ seq_lens, int len_add,
                                          float* __restrict__ out, int Hq, int n_splits,
                                          int chunk, int max_seq_len, int D) {
  const int bh = blockIdx.x;
  const int b = bh / Hq;
  const int raw = seq_lens[b];
  int L = raw > max_seq_len ? max_seq_len : raw + len_add;
  L = L < 0 ? 0 : (L > max_seq_len ? max_seq_len : L);
  const int ns = (L + chunk - 1) / chunk;
  const float* ml = part_ml + static_cast<size_t>(bh) * n_splits * 2;
  const float* po = part_o + static_cast<size_t>(bh) * n_splits * D;
  float m = -INFINITY;
  for (int s = 0; s < ns; ++s) m = fmaxf(m, ml[2 * s]);
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float acc = 0.f, l = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < ns; ++s) {
        const float ms = ml[2 * s];
        const float w = (ms == -INFINITY) ? 0.f : expf(ms - m);
        acc = fmaf(w, po[static_cast<size_t>(s) * D + c], acc);
        l = fmaf(w, ml[2 * s + 1], l);
      }
    }
    out[static_cast<size_t>(bh) * D + c] = l > 0.f ? acc / l : 0.f;
  }
}

template <int D>
cudaError_t launch_f32(const DecodeArgs& a, cudaStream_t stream) {
  dim3 grid(a.n_splits, a.Hq, a.B);
  decode_f32_kernel<D><<<grid, kThreadsF, 0, stream>>>(
      static_cast<const float*>(a.q), static_cast<const float*>(a.k_cache),
      static_cast<const float*>(a.v_cache), a.seq_lens, a.len_add, a.part_o, a.part_ml,
      a.status, a.Hq, a.Hkv, a.Lmax, a.max_seq_len, a.chunk, a.n_splits, a.scale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_f32_kernel<<<a.B * a.Hq, D < 32 ? 32 : D, 0, stream>>>(
      a.part_o, a.part_ml, a.seq_lens, a.len_add, static_cast<float*>(a.out), a.Hq, a.n_splits,
      a.chunk, a.max_seq_len, D);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_f32(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.d) {
    case 16: return launch_f32<16>(a, stream);
    case 32: return launch_f32<32>(a, stream);
    case 64: return launch_f32<64>(a, stream);
    case 128: return launch_f32<128>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace csattn
