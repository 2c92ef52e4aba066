// Backward of causal GQA attention (bf16 in / out, fp32 accumulation).  The
// gradients of sum(out * dout), written out from the forward's definition:
//
//   P   = exp(S - lse)            S = scale * Qr Kr^T  (+ the causal mask)
//   D_i = sum_c dO_ic O_ic        (the softmax Jacobian's correction)
//   dS  = P o (dO V^T - D)
//   dV  = P^T dO                  summed over the query heads of a KV group
//   dQ  = R^T (scale * dS Kr)     R = the RoPE rotation at the query's position
//   dK  = R^T (scale * dS^T Qr)   summed over the group's query heads
//
// with Qr, Kr the rotated, bf16-rounded operands of the forward ("The
// Transformer architecture" (cooking-agi), "Now: RoPE": a rotation, so its
// Jacobian transpose is the inverse rotation) and lse the forward's log-sum-exp.
//
// This file holds the row-dot kernel for D and the dispatch; the dK/dV and dQ
// kernels (tcgen05, d and d_v each 64 or 128) are in bwd_tc.cu: two kernels, no atomics,
// S and dP recomputed in both (FlashAttention-2's split, which trades two extra
// GEMMs per tile pair for no global atomics).
#include "internal.h"

namespace csattn {
namespace {

// D[row] = sum_c dO[row, c] O[row, c] (fp32).  A row is d/8 lanes, each with one
// 16-byte load of dO and of O (d in {64, 128, 256}: 4, 2 or 1 rows per warp), the
// partial sums reduced over the row's lanes with shuffles.
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const __nv_bfloat16* __restrict__ dout,
                                                         const __nv_bfloat16* __restrict__ out,
                                                         float* __restrict__ dvec, long long rows,
                                                         int d) {
  const int lpr = d / 8;  // lanes per row
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = t / lpr;
  const int c = static_cast<int>(t % lpr) * 8;
  float sum = 0.f;
  if (row < rows) {
    const uint4 wa = __ldg(reinterpret_cast<const uint4*>(dout + row * d + c));
    const uint4 wo = __ldg(reinterpret_cast<const uint4*>(out + row * d + c));
    const uint32_t a4[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t o4[4] = {wo.x, wo.y, wo.z, wo.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sum = fmaf(bf16lo_to_f32(a4[e]), bf16lo_to_f32(o4[e]), sum);
      sum = fmaf(bf16hi_to_f32(a4[e]), bf16hi_to_f32(o4[e]), sum);
    }
  }
  for (int off = lpr / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (row < rows && (threadIdx.x & (lpr - 1)) == 0) dvec[row] = sum;
}

}  // namespace

cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t stream) {
  if ((a.d != 64 && a.d != 128) || (a.d_v != 64 && a.d_v != 128)) return cudaErrorInvalidValue;
  // D = rowsum(dout o out) over the d_v channels, then the two tcgen05 kernels (bwd_tc.cu)
  const long long rows = static_cast<long long>(a.B) * a.Hq * a.Tq;
  bwd_rowdot_kernel<<<static_cast<unsigned>((rows * (a.d_v / 8) + 255) / 256), 256, 0,
                      stream>>>(static_cast<const __nv_bfloat16*>(a.dout),
                                static_cast<const __nv_bfloat16*>(a.out), a.dvec, rows, a.d_v);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_bwd_kv_tc(a, stream);
  if (e != cudaSuccess) return e;
  return launch_bwd_q_tc(a, stream);
}

}  // namespace csattn
