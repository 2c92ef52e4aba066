// Backward of causal GQA attention (bf16 in / out, fp32 accumulation) on the
// mma.sync tensor-core path (m16n8k16, bf16 operands).  The gradients of
// sum(out * dout), written out from the forward's definition:
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
// d = 128 runs the tcgen05 kernels of bwd_tc.cu; this file holds the row-dot
// kernel for D and the mma.sync kernels used for d = 64.  Two kernels, no atomics:
//   bwd_dkdv_kernel  one CTA per (64 keys, KV head, batch): loops over the
//                    group's query heads and the query tiles that see the keys;
//                    dK and dV stay in registers (warp w owns keys 16w..16w+15).
//   bwd_dq_kernel    one CTA per (64 queries, query head, batch): loops over
//                    the visible key tiles; dQ stays in registers.
// S and dP are recomputed in both (FlashAttention-2's split, which trades two
// extra GEMMs per tile pair for no global atomics).  Tiles move global ->
// shared with cp.async into a 128-byte-swizzled layout read by ldmatrix, two
// stages, one __syncthreads per tile.
#include "internal.h"

namespace csattn {
namespace {

constexpr int kTile = 64;  // rows per Q / dO / K / V tile
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// 16-byte global -> shared copy; src_bytes 0 writes zeros (rows past the end)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// byte offset of 16-byte chunk cc (8 channels) of row r in a 64-row tile kept as
// 128-byte-swizzled 64-channel column blocks
__device__ __forceinline__ uint32_t toff(int r, int cc) {
  return static_cast<uint32_t>((cc >> 3) * (kTile * 128) + r * 128 +
                               (((cc & 7) ^ (r & 7)) << 4));
}

// rows [r0, r0 + 64) of a [rows, D] bf16 matrix into a swizzled tile; rows >= n_rows
// are zero-filled
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const __nv_bfloat16* src, int r0,
                                          int n_rows) {
  constexpr int kChunks = kTile * D / 8;
  for (int e = threadIdx.x; e < kChunks; e += kThreads) {
    const int r = e / (D / 8), cc = e - r * (D / 8);
    const bool ok = r0 + r < n_rows;
    const __nv_bfloat16* g = src + static_cast<size_t>(ok ? r0 + r : 0) * D + cc * 8;
    cp_async16(dst + toff(r, cc), g, ok ? 16 : 0);
  }
}

// 64 fp32 values src[r0 .. r0+63] (0 past n) into shared memory
__device__ __forceinline__ void load_vec(uint32_t dst, const float* src, int r0, int n) {
  if (threadIdx.x < kTile / 4) {
    const int e = threadIdx.x * 4;
    const float* g = src + r0 + e;
    if (r0 + e + 4 <= n && (reinterpret_cast<uintptr_t>(g) & 15u) == 0) {
      cp_async16(dst + e * 4, g, 16);
    } else {
      // ragged end or a row start that is not 16-byte aligned: plain loads
      float t[4];
      for (int i = 0; i < 4; ++i) t[i] = (r0 + e + i < n) ? g[i] : 0.f;
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(dst + e * 4), "f"(t[0]),
                   "f"(t[1]), "f"(t[2]), "f"(t[3])
                   : "memory");
    }
  }
}

// R^T applied to pairs held in the accumulator fragments of one row half
// (e in {0,1}: row r0; e in {2,3}: row r0 + 8) at position pos.
template <int D>
__device__ __forceinline__ void rope_transpose_rows(float (&acc)[D / 8][4], int rope, int pos0,
                                                    int pos1, const RopeTable& th, int cq) {
  if (rope == 1) {  // split-half: channel p with p + D/2 (n-tile nt with nt + D/16)
#pragma unroll
    for (int nt = 0; nt < D / 16; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int p = 8 * nt + cq + (e & 1);
        float c, s;
        rope_cos_sin<false>((e < 2) ? pos0 : pos1, th.hi[p], th.lo[p], c, s);
        const float a = acc[nt][e], b = acc[nt + D / 16][e];
        acc[nt][e] = fmaf(a, c, b * s);
        acc[nt + D / 16][e] = fmaf(-a, s, b * c);
      }
  } else if (rope == 2) {  // adjacent: channels (2p, 2p+1) = one register pair
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int p = (8 * nt + cq) >> 1;
        float c, s;
        rope_cos_sin<false>(h ? pos1 : pos0, th.hi[p], th.lo[p], c, s);
        const float a = acc[nt][2 * h], b = acc[nt][2 * h + 1];
        acc[nt][2 * h] = fmaf(a, c, b * s);
        acc[nt][2 * h + 1] = fmaf(-a, s, b * c);
      }
  }
}

struct BwdParams {
  const __nv_bfloat16* qr;    // rotated q [B, Hq, Tq, D]
  const __nv_bfloat16* kr;    // rotated k [B, Hkv, Tk, D]
  const __nv_bfloat16* v;     // [B, Hkv, Tk, D]
  const __nv_bfloat16* dout;  // [B, Hq, Tq, D]
  const float* lse;           // [B, Hq, Tq], natural log
  const float* dvec;          // D = rowsum(dO o O) [B, Hq, Tq]
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int Hq, Hkv, Tq, Tk, q_off, causal, rope;
  float scale, sl2;           // sl2 = scale * log2(e)
  RopeTable theta;
};

// ---------------------------------------------------------------- dK, dV
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  constexpr int TB = kTile * D * 2;  // bytes per tile
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sK = smem_u32(smem), sV = sK + TB;
  const uint32_t sQ0 = sK + 2 * TB, sO0 = sK + 4 * TB;  // two stages each
  const uint32_t sL0 = sK + 6 * TB;                     // [2 stages][lse2 64 | D 64] fp32
  const float* fL = reinterpret_cast<const float*>(smem + 6 * TB);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = lane >> 2, cq = 2 * (lane & 3), mi = lane >> 3;
  const int k0 = blockIdx.x * kTile, g = blockIdx.y, b = blockIdx.z;
  const int rep = p.Hq / p.Hkv;
  const size_t kvbase = (static_cast<size_t>(b) * p.Hkv + g) * p.Tk;

  load_tile<D>(sK, p.kr + kvbase * D, k0, p.Tk);
  load_tile<D>(sV, p.v + kvbase * D, k0, p.Tk);
  cp_async_commit();

  int i_begin = 0;
  if (p.causal) i_begin = max(0, (k0 - p.q_off) / kTile);
  const int n_qt = (p.Tq + kTile - 1) / kTile;
  const int per_head = max(0, n_qt - i_begin);
  const int n_it = rep * per_head;

  auto issue = [&](int it, int st) {
    const int h = g * rep + it / per_head;
    const int q0 = (i_begin + it % per_head) * kTile;
    const size_t qbase = (static_cast<size_t>(b) * p.Hq + h) * p.Tq;
    load_tile<D>(sQ0 + st * TB, p.qr + qbase * D, q0, p.Tq);
    load_tile<D>(sO0 + st * TB, p.dout + qbase * D, q0, p.Tq);
    load_vec(sL0 + st * 512, p.lse + qbase, q0, p.Tq);
    load_vec(sL0 + st * 512 + 256, p.dvec + qbase, q0, p.Tq);
  };
  if (n_it > 0) issue(0, 0);
  cp_async_commit();

  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[n][e] = dv[n][e] = 0.f;

  const int key_r0 = k0 + 16 * warp + r0;  // keys of this thread's two fragment rows
  const int key_r1 = key_r0 + 8;
  const int arow = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);  // A-fragment row address

  for (int it = 0; it < n_it; ++it) {
    const int st = it & 1;
    if (it + 1 < n_it) issue(it + 1, st ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t sQ = sQ0 + st * TB, sO = sO0 + st * TB;
    const float* lse2 = fL + st * 128;  // natural-log lse, converted below
    const float* dvv = lse2 + 64;
    const int q0 = (i_begin + it % per_head) * kTile;

    // S^T = Kr Qr^T: 16 keys x 64 queries per warp
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sK + toff(arow, 2 * kk + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sQ + toff(16 * np + (lane & 7) + 8 * (mi >> 1), 2 * kk + (mi & 1)), b0, b1, b2,
                b3);
        mma_bf16(s[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    // P^T = exp(S - lse), masked
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qi = 8 * nt + cq + (e & 1);
        const int q = q0 + qi;
        const int key = (e < 2) ? key_r0 : key_r1;
        const bool ok = q < p.Tq && key < p.Tk && (!p.causal || key <= p.q_off + q);
        s[nt][e] = ok ? exp2f(fmaf(s[nt][e], p.sl2, -lse2[qi] * kLog2e)) : 0.f;
      }
    // dV += P^T dO
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
      const uint32_t a0 = pack_bf16x2(s[2 * kk2][0], s[2 * kk2][1]);
      const uint32_t a1 = pack_bf16x2(s[2 * kk2][2], s[2 * kk2][3]);
      const uint32_t a2 = pack_bf16x2(s[2 * kk2 + 1][0], s[2 * kk2 + 1][1]);
      const uint32_t a3 = pack_bf16x2(s[2 * kk2 + 1][2], s[2 * kk2 + 1][3]);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sO + toff(16 * kk2 + (lane & 7) + 8 * (mi & 1), 2 * np + (mi >> 1)), b0, b1,
                  b2, b3);
        mma_bf16(dv[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(dv[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    // dP^T = V dO^T, then dS^T = P^T o (dP^T - D)
    float dp[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) dp[n][0] = dp[n][1] = dp[n][2] = dp[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sV + toff(arow, 2 * kk + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sO + toff(16 * np + (lane & 7) + 8 * (mi >> 1), 2 * kk + (mi & 1)), b0, b1, b2,
                b3);
        mma_bf16(dp[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(dp[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] *= dp[nt][e] - dvv[8 * nt + cq + (e & 1)];
    // dK += dS^T Qr
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
      const uint32_t a0 = pack_bf16x2(s[2 * kk2][0], s[2 * kk2][1]);
      const uint32_t a1 = pack_bf16x2(s[2 * kk2][2], s[2 * kk2][3]);
      const uint32_t a2 = pack_bf16x2(s[2 * kk2 + 1][0], s[2 * kk2 + 1][1]);
      const uint32_t a3 = pack_bf16x2(s[2 * kk2 + 1][2], s[2 * kk2 + 1][3]);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sQ + toff(16 * kk2 + (lane & 7) + 8 * (mi & 1), 2 * np + (mi >> 1)), b0, b1,
                  b2, b3);
        mma_bf16(dk[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(dk[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();  // this stage is refilled by the next iteration's prefetch
  }
  cp_async_wait<0>();

  // epilogue: dK = R^T (scale dK), dV as is; keys past Tk are not stored
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[n][e] *= p.scale;
  rope_transpose_rows<D>(dk, p.rope, key_r0, key_r1, p.theta, cq);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int key = h ? key_r1 : key_r0;
    if (key >= p.Tk) continue;
    __nv_bfloat16* dkr = p.dk + (kvbase + key) * D;
    __nv_bfloat16* dvr = p.dv + (kvbase + key) * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      *reinterpret_cast<uint32_t*>(dkr + 8 * nt + cq) = pack_bf16x2(dk[nt][2 * h], dk[nt][2 * h + 1]);
      *reinterpret_cast<uint32_t*>(dvr + 8 * nt + cq) = pack_bf16x2(dv[nt][2 * h], dv[nt][2 * h + 1]);
    }
  }
}

// ---------------------------------------------------------------- dQ
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  constexpr int TB = kTile * D * 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem), sO = sQ + TB;
  const uint32_t sK0 = sQ + 2 * TB, sV0 = sQ + 4 * TB;  // two stages each

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = lane >> 2, cq = 2 * (lane & 3), mi = lane >> 3;
  const int q0 = blockIdx.x * kTile, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (p.Hq / p.Hkv);
  const size_t qbase = (static_cast<size_t>(b) * p.Hq + h) * p.Tq;
  const size_t kvbase = (static_cast<size_t>(b) * p.Hkv + g) * p.Tk;

  load_tile<D>(sQ, p.qr + qbase * D, q0, p.Tq);
  load_tile<D>(sO, p.dout + qbase * D, q0, p.Tq);
  cp_async_commit();
  const int n_kt_all = (p.Tk + kTile - 1) / kTile;
  int n_kt = n_kt_all;
  if (p.causal) n_kt = min(n_kt_all, (p.q_off + min(q0 + kTile, p.Tq) - 1) / kTile + 1);
  load_tile<D>(sK0, p.kr + kvbase * D, 0, p.Tk);
  load_tile<D>(sV0, p.v + kvbase * D, 0, p.Tk);
  cp_async_commit();

  const int row_r0 = q0 + 16 * warp + r0, row_r1 = row_r0 + 8;
  float lse2[2], dvv[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int r = hh ? row_r1 : row_r0;
    lse2[hh] = r < p.Tq ? p.lse[qbase + r] * kLog2e : 0.f;
    dvv[hh] = r < p.Tq ? p.dvec[qbase + r] : 0.f;
  }
  cp_async_wait<1>();
  __syncthreads();
  // A fragments of Qr and dO for this warp's 16 rows
  uint32_t qa[D / 16][4], oa[D / 16][4];
  const int arow = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    ldsm_x4(sQ + toff(arow, 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    ldsm_x4(sO + toff(arow, 2 * kk + (lane >> 4)), oa[kk][0], oa[kk][1], oa[kk][2], oa[kk][3]);
  }

  float acc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

  for (int j = 0; j < n_kt; ++j) {
    const int st = j & 1;
    if (j + 1 < n_kt) {
      load_tile<D>(sK0 + (st ^ 1) * TB, p.kr + kvbase * D, (j + 1) * kTile, p.Tk);
      load_tile<D>(sV0 + (st ^ 1) * TB, p.v + kvbase * D, (j + 1) * kTile, p.Tk);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t sK = sK0 + st * TB, sV = sV0 + st * TB;
    // S = Qr Kr^T and dP = dO V^T: 16 rows x 64 keys per warp
    float s[8][4], dp[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[n][e] = dp[n][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        const uint32_t off = toff(16 * np + (lane & 7) + 8 * (mi >> 1), 2 * kk + (mi & 1));
        ldsm_x4(sK + off, b0, b1, b2, b3);
        mma_bf16(s[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma_bf16(s[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        ldsm_x4(sV + off, b0, b1, b2, b3);
        mma_bf16(dp[2 * np], oa[kk][0], oa[kk][1], oa[kk][2], oa[kk][3], b0, b1);
        mma_bf16(dp[2 * np + 1], oa[kk][0], oa[kk][1], oa[kk][2], oa[kk][3], b2, b3);
      }
    // dS = P o (dP - D), P = exp(S - lse), masked
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = j * kTile + 8 * nt + cq + (e & 1);
        const int row = (e < 2) ? row_r0 : row_r1;
        const bool ok = row < p.Tq && key < p.Tk && (!p.causal || key <= p.q_off + row);
        const float pr = ok ? exp2f(fmaf(s[nt][e], p.sl2, -lse2[e >> 1])) : 0.f;
        s[nt][e] = pr * (dp[nt][e] - dvv[e >> 1]);
      }
    // dQ += dS Kr
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
      const uint32_t a0 = pack_bf16x2(s[2 * kk2][0], s[2 * kk2][1]);
      const uint32_t a1 = pack_bf16x2(s[2 * kk2][2], s[2 * kk2][3]);
      const uint32_t a2 = pack_bf16x2(s[2 * kk2 + 1][0], s[2 * kk2 + 1][1]);
      const uint32_t a3 = pack_bf16x2(s[2 * kk2 + 1][2], s[2 * kk2 + 1][3]);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sK + toff(16 * kk2 + (lane & 7) + 8 * (mi & 1), 2 * np + (mi >> 1)), b0, b1,
                  b2, b3);
        mma_bf16(acc[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[n][e] *= p.scale;
  rope_transpose_rows<D>(acc, p.rope, p.q_off + row_r0, p.q_off + row_r1, p.theta, cq);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int row = hh ? row_r1 : row_r0;
    if (row >= p.Tq) continue;
    __nv_bfloat16* dqr = p.dq + (qbase + row) * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
      *reinterpret_cast<uint32_t*>(dqr + 8 * nt + cq) =
          pack_bf16x2(acc[nt][2 * hh], acc[nt][2 * hh + 1]);
  }
}

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

template <int D>
cudaError_t launch_d(const BwdArgs& a, cudaStream_t stream) {
  BwdParams p{};
  p.qr = static_cast<const __nv_bfloat16*>(a.qr);
  p.kr = static_cast<const __nv_bfloat16*>(a.kr);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
  p.dout = static_cast<const __nv_bfloat16*>(a.dout);
  p.lse = a.lse;
  p.dvec = a.dvec;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.q_off = a.q_off;
  p.causal = a.causal;
  p.rope = a.rope;
  p.scale = a.scale;
  p.sl2 = a.scale * kLog2e;
  p.theta = a.theta;

  const long long rows = static_cast<long long>(a.B) * a.Hq * a.Tq;
  bwd_rowdot_kernel<<<static_cast<unsigned>((rows * (D / 8) + 255) / 256), 256, 0, stream>>>(
      p.dout, static_cast<const __nv_bfloat16*>(a.out), a.dvec, rows, D);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  constexpr int TB = kTile * D * 2;
  const int smem_kv = 6 * TB + 1024;
  const int smem_q = 6 * TB;
  e = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_kv);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q);
  if (e != cudaSuccess) return e;
  dim3 gkv((a.Tk + kTile - 1) / kTile, a.Hkv, a.B);
  bwd_dkdv_kernel<D><<<gkv, kThreads, smem_kv, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 gq((a.Tq + kTile - 1) / kTile, a.Hq, a.B);
  bwd_dq_kernel<D><<<gq, kThreads, smem_q, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_d<64>(a, stream);
  if (a.d != 128 || a.Tq != a.Tk || a.q_off != 0) return cudaErrorInvalidValue;
  // d = 128: D = rowsum(dout o out), then the two tcgen05 kernels (bwd_tc.cu)
  const long long rows = static_cast<long long>(a.B) * a.Hq * a.Tq;
  bwd_rowdot_kernel<<<static_cast<unsigned>((rows * (128 / 8) + 255) / 256), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.dout), static_cast<const __nv_bfloat16*>(a.out), a.dvec,
      rows, 128);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_bwd_kv_tc(a, stream);
  if (e != cudaSuccess) return e;
  return launch_bwd_q_tc(a, stream);
}

}  // namespace csattn
