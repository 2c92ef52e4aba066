// dK and dV of the attention backward on tcgen05 (the math and the split into a
// dK/dV kernel and a dQ kernel are described in bwd.cu).  Head sizes: d (q, k) and
// dv (v, out) each 64 or 128; Tq query rows at positions q_off..q_off+Tq-1 and Tk
// keys at 0..Tk-1 (query i sees key j iff j <= q_off + i when causal).
//
// One CTA per (128 keys, KV head, batch); it walks the query heads of the KV
// group and, for each, the 128-row query tiles that see the keys.  Per tile:
//
//   S^T  = Kr Qr^T          M=128 keys, N=128 queries, K=d      (SS, TMEM cols [0,128))
//   dP^T = V dO^T           M=128 keys, N=128 queries, K=dv     (SS, cols [128,256))
//   P^T  = exp(scale*S^T - lse)   dS^T = P^T o (dP^T - D)      (softmax warpgroups)
//   dV  += P^T dO           M=128 keys, N=dv channels, K=128 queries (SS, cols [256,256+dv))
//   dK  += dS^T Qr          M=128 keys, N=d channels               (TS, cols [384,384+d))
//
// P^T (bf16) goes to shared memory (K-major, 128-byte swizzle) and feeds dV as
// the A operand, so the S^T columns are free as soon as the softmax warps have
// read them and S^T of the next tile overlaps this tile's softmax; dS^T (bf16)
// is written back into TMEM over the dP^T columns and feeds dK from there.
// Warps 0-3 handle queries 0-63 of the tile, warps 4-7 queries 64-127 (thread =
// key row = TMEM lane); warp 8 loads (TMA for Qr and dO, plain loads for lse and
// D); warp 9 allocates TMEM and issues the MMAs in the order dV(it), S^T(it+1),
// dK(it), dP^T(it+1): dK(it) frees the dS^T columns for dP^T(it+1).
//
// Every wait is bounded (2 s) and sets the status word's timeout bit; no named
// barriers, so a warp that gives up just leaves its loop.
#include "internal.h"

namespace csattn {
namespace {

constexpr int BK = 128;  // keys per CTA
constexpr int BQ = 128;  // queries per tile
constexpr int kThreads = 384;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int NSQ = 2;  // Q / dO stages
constexpr int BLOCK = BQ * 128;         // one 64-channel column block of a 128-row tile
constexpr int PTILE = BK * BQ * 2;      // the P^T tile, 32 KB
constexpr int VEC = 2 * BQ * 4;         // lse and D of one tile, fp32
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 100000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t IDESC_SS = idesc_bf16_f32(128, 128, 0, 0);  // both K-major (S^T, dP^T, S, dP)

// Head-size dependent sizes (d = D, dv = DV, each 64 or 128): a Q or K tile is D/64
// and a V or dO tile DV/64 column blocks of 128 rows; dK and dQ are N = D, dV an
// N = DV product, with B read MN-major.
template <int D, int DV>
struct BwdCfg {
  static_assert((D == 64 || D == 128) && (DV == 64 || DV == 128), "head sizes 64 or 128");
  static constexpr int TILE_QK = BQ * D * 2;   // a Q or K tile
  static constexpr int TILE_VO = BQ * DV * 2;  // a V or dO tile
  static constexpr int SMEM_DATA = (1 + NSQ) * (TILE_QK + TILE_VO) + PTILE + NSQ * VEC;
  static constexpr int SMEM_BYTES = SMEM_DATA + 256;
  static constexpr uint32_t IDESC_DK = idesc_bf16_f32(128, D, 0, 1);   // A K-major, B MN-major
  static constexpr uint32_t IDESC_DV = idesc_bf16_f32(128, DV, 0, 1);
};

struct KvParams {
  const float* lse;   // [B, Hq, Tq], natural log
  const float* dvec;  // [B, Hq, Tq]
  __nv_bfloat16* dk;  // [B, Hkv, Tk, D]
  __nv_bfloat16* dv;  // [B, Hkv, Tk, DV]
  uint32_t* status;
  int Hq, Hkv, Tq, Tk, q_off, causal, rope;
  float scale, sl2;
  RopeTable theta;
};

// First 128-row query tile holding a query that sees key k0 (causal: the tile's last
// row sits at or after k0).
__device__ __forceinline__ int first_query_tile(int k0, int q_off, int causal) {
  if (!causal) return 0;
  const int num = k0 - q_off - (BQ - 1);
  return num > 0 ? (num + BQ - 1) / BQ : 0;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status) {
  const bool ok = mbar_wait(bar, parity, abort, status, kWaitNs);
  return __all_sync(0xffffffffu, ok) != 0;
}

// packed bf16 column of queries 16kk..16kk+15 inside a P^T or dS^T region
__device__ __forceinline__ uint32_t packed_col(int kk) {
  return static_cast<uint32_t>(kk < 4 ? 8 * kk : 64 + 8 * (kk - 4));
}

template <int D, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_tc_kernel(const __grid_constant__ KvParams p, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_do) {
  using C = BwdCfg<D, DV>;
  constexpr int TQK = C::TILE_QK, TVO = C::TILE_VO;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sK = smem;
  uint8_t* sV = smem + TQK;
  uint8_t* sQ = sV + TVO;                        // [NSQ] Qr tiles
  uint8_t* sO = sQ + NSQ * TQK;                  // [NSQ] dO tiles
  uint8_t* sP = sO + NSQ * TVO;                  // P^T: rows = keys, queries contiguous
  float* sVec = reinterpret_cast<float*>(sP + PTILE);  // [NSQ][lse | D]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::SMEM_DATA);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;   // [NSQ]: Qr and dO tiles (TMA bytes)
  uint64_t* q_empty = bars + 3;  // [NSQ]
  uint64_t* s_full = bars + 5;   // S^T in TMEM
  uint64_t* p_full = bars + 6;   // P^T written (8 warps)
  uint64_t* ds_full = bars + 7;  // dS^T written (8 warps)
  uint64_t* acc_full = bars + 8; // dK, dV complete
  uint64_t* teardown = bars + 9;
  uint64_t* dp_full = bars + 10; // dP^T in TMEM
  uint64_t* vec_full = bars + 11; // [NSQ]: lse and D of the tile stored by the load warp
  uint64_t* s_free = bars + 13;   // S^T read by the softmax warps (8 warps)
  uint64_t* dv_done = bars + 14;  // dV(it) complete: the P^T tile may be rewritten
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusDeviceArg);
    return;
  }
  // grid (Hkv, B, key tiles): blocks launch in index order, so z runs slowest and the
  // key tiles with the most query tiles to visit (the first ones, causally) go first
  const int kt = blockIdx.z;
  const int k0 = kt * BK, g = blockIdx.x, b = blockIdx.y;
  const int rep = p.Hq / p.Hkv;
  const int n_qt = (p.Tq + BQ - 1) / BQ;
  const int i_begin = first_query_tile(k0, p.q_off, p.causal);  // query tiles that see these keys
  const int per_head = n_qt > i_begin ? n_qt - i_begin : 0;
  const int n_it = rep * per_head;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NSQ; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
      mbar_init(&vec_full[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 8);
    mbar_init(ds_full, 8);
    mbar_init(s_free, 8);
    mbar_init(dv_done, 1);
    mbar_init(acc_full, 1);
    mbar_init(teardown, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ loads (whole warp)
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(kv_full, TQK + TVO);
      const int zk = b * p.Hkv + g;
      for (int kb = 0; kb < D / 64; ++kb) tma_load_3d(sK + kb * BLOCK, &tm_k, kv_full, kb * 64, k0, zk);
      for (int kb = 0; kb < DV / 64; ++kb) tma_load_3d(sV + kb * BLOCK, &tm_v, kv_full, kb * 64, k0, zk);
    }
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % NSQ, use = it / NSQ;
      if (use > 0 && !warp_wait(&q_empty[st], (use - 1) & 1, abort_flag, p.status)) break;
      const int h = g * rep + it / per_head;
      const int q0 = (i_begin + it % per_head) * BQ;
      const int zq = b * p.Hq + h;
      if (lane == 0) {
        mbar_arrive_expect_tx(&q_full[st], TQK + TVO);
        for (int kb = 0; kb < D / 64; ++kb)
          tma_load_3d(sQ + st * TQK + kb * BLOCK, &tm_q, &q_full[st], kb * 64, q0, zq);
        for (int kb = 0; kb < DV / 64; ++kb)
          tma_load_3d(sO + st * TVO + kb * BLOCK, &tm_do, &q_full[st], kb * 64, q0, zq);
      }
      float* vec = sVec + st * 2 * BQ;
      const size_t rb = static_cast<size_t>(zq) * p.Tq;
      // all loads before the shared-memory stores, so that their latencies overlap
      float lv[BQ / 32], dvl[BQ / 32];
#pragma unroll
      for (int i = 0; i < BQ / 32; ++i) {
        const int q = q0 + lane + 32 * i;
        lv[i] = q < p.Tq ? __ldg(p.lse + rb + q) : 0.f;
        dvl[i] = q < p.Tq ? __ldg(p.dvec + rb + q) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < BQ / 32; ++i) {
        vec[lane + 32 * i] = lv[i] * kLog2e;
        vec[BQ + lane + 32 * i] = dvl[i];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&vec_full[st]);
      ++issued;
    }
    if (lane == 0 && *abort_flag) {
      mbar_wait(kv_full, 0, nullptr, p.status, kDrainNs);
      const int first = issued > NSQ ? issued - NSQ : 0;
      for (int t = first; t < issued; ++t)
        mbar_wait(&q_full[t % NSQ], (t / NSQ) & 1, nullptr, p.status, kDrainNs);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (!ok) return false;
        ok = mbar_wait(bar, parity, abort_flag, p.status, kWaitNs);
        tc_fence_after();
        return ok;
      };
      const uint32_t k_s = smem_u32(sK), v_s = smem_u32(sV);
      wait(kv_full, 0);  // also when there is nothing to do: the loads must land first
      auto q_tile = [&](int it) { return smem_u32(sQ + (it % NSQ) * TQK); };
      auto o_tile = [&](int it) { return smem_u32(sO + (it % NSQ) * TVO); };
      auto issue_st = [&](int it) {  // S^T = Kr Qr^T
        const uint32_t q_s = q_tile(it);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((kk >> 2) * BLOCK + (kk & 3) * 32);
          umma_ss(tmem, smem_desc_sw128(k_s + off, 16, 1024), smem_desc_sw128(q_s + off, 16, 1024),
                  IDESC_SS, kk > 0 ? 1u : 0u);
        }
        tc_commit(s_full);
      };
      auto issue_dpt = [&](int it) {  // dP^T = V dO^T
        const uint32_t o_s = o_tile(it);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((kk >> 2) * BLOCK + (kk & 3) * 32);
          umma_ss(tmem + 128u, smem_desc_sw128(v_s + off, 16, 1024),
                  smem_desc_sw128(o_s + off, 16, 1024), IDESC_SS, kk > 0 ? 1u : 0u);
        }
        tc_commit(dp_full);
      };
      // Order per tile: dV(it), S^T(it+1), dK(it), dP^T(it+1).  S^T(it+1) runs two
      // products ahead of dV(it+1), which needs the softmax warps' P^T(it+1); and it
      // comes after dV(it) so that the Q/dO stage of tile it+1, freed when dK(it-1)
      // completes, has the time of dP^T(it) and dV(it) to land before the MMA thread
      // waits for it.  dK(it) frees the dS^T columns for dP^T(it+1).
      if (n_it > 0 && wait(&q_full[0], 0)) {
        issue_st(0);
        issue_dpt(0);
      }
      const uint32_t p_s = smem_u32(sP);
      for (int it = 0; it < n_it && ok; ++it) {
        const uint32_t q_s = q_tile(it), o_s = o_tile(it);
        const bool next = it + 1 < n_it;
        if (!wait(p_full, it & 1)) break;
        // dV += P^T dO: A = P^T (shared memory, K-major), B = dO (rows = queries,
        // channels contiguous)
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((kk >> 2) * BLOCK + (kk & 3) * 32);
          umma_ss(tmem + 256u, smem_desc_sw128(p_s + off, 16, 1024),
                  smem_desc_sw128(o_s + 2048u * kk, BLOCK, 1024), C::IDESC_DV,
                  (it > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(dv_done);
        if (next) {
          if (!wait(s_free, it & 1)) break;
          if (!wait(&q_full[(it + 1) % NSQ], ((it + 1) / NSQ) & 1)) break;
          issue_st(it + 1);
        }
        if (!wait(ds_full, it & 1)) break;
        // dK += dS^T Qr
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          umma_ts(tmem + 384u, tmem + 128u + packed_col(kk),
                  smem_desc_sw128(q_s + 2048u * kk, BLOCK, 1024), C::IDESC_DK,
                  (it > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&q_empty[it % NSQ]);
        if (next) issue_dpt(it + 1);
      }
      tc_commit(acc_full);
      tc_commit(teardown);
      mbar_wait(teardown, 0, nullptr, p.status, kDrainNs);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ P^T, dS^T; epilogue
    const int x = warp >> 2;                 // query half of the tile
    const int row = threadIdx.x & 127;       // key row = TMEM lane
    const int key = k0 + row;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(64 * x);
    const uint32_t tD = tmem + lane_off + 128u + static_cast<uint32_t>(64 * x);
    // this thread's row of P^T: 64 queries = one 128-byte row of column block x
    uint8_t* const prow = sP + x * BLOCK + row * 128;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % NSQ;
      const int q0 = (i_begin + it % per_head) * BQ + 64 * x;  // first query of this half
      if (!warp_wait(s_full, it & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // lse and D of this tile were stored by the load warp before its vec_full arrival
      if (!warp_wait(&vec_full[st], (it / NSQ) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const float* lse2 = sVec + st * 2 * BQ + 64 * x;
      const float* dv = lse2 + BQ;
      float pt[64];
      {
        uint32_t r[64];
        tmem_ld64_sync(tS, r);
        // S^T(it) is in registers: the MMA warp may write S^T(it+1)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
        // every (key, query) of this warpgroup's half tile is visible: no per-element test
        const bool all_vis =
            q0 + 63 < p.Tq && k0 + BK <= p.Tk && (!p.causal || p.q_off + q0 >= k0 + BK - 1);
        if (all_vis) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            pt[c] = ex2_approx(fmaf(__uint_as_float(r[c]), p.sl2, -lse2[c]));
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int q = q0 + c;
            const bool vis = q < p.Tq && key < p.Tk && (!p.causal || key <= p.q_off + q);
            pt[c] = vis ? ex2_approx(fmaf(__uint_as_float(r[c]), p.sl2, -lse2[c])) : 0.f;
          }
        }
      }
      // the P^T tile is free once dV(it-1) has completed
      if (it > 0 && !warp_wait(dv_done, (it - 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) =
            make_uint4(pack_bf16x2(pt[8 * c], pt[8 * c + 1]), pack_bf16x2(pt[8 * c + 2], pt[8 * c + 3]),
                       pack_bf16x2(pt[8 * c + 4], pt[8 * c + 5]),
                       pack_bf16x2(pt[8 * c + 6], pt[8 * c + 7]));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      if (!warp_wait(dp_full, it & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t r[32], pk[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tmem_ld32_sync(tD + 32u * h, r);
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int c = 2 * t;
            const float d0 = pt[32 * h + c] * (__uint_as_float(r[c]) - dv[32 * h + c]);
            const float d1 = pt[32 * h + c + 1] * (__uint_as_float(r[c + 1]) - dv[32 * h + c + 1]);
            pk[t] = pack_bf16x2(d0, d1);
          }
          tmem_st16(tD + 16u * h, pk);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    // epilogue: warps 0-3 write dV (W = DV channels), warps 4-7 dK = R^T (scale dK)
    // (W = D); channels in 32-column chunks 32c and W/2 + 32c so that split-half RoPE
    // pairs (i, i + d/2) meet
    if (ok && (n_it == 0 || warp_wait(acc_full, 0, abort_flag, p.status))) {
      tc_fence_after();
      const int W = x ? D : DV;
      const uint32_t tacc = tmem + lane_off + (x ? 384u : 256u);
      __nv_bfloat16* dst = (x ? p.dk : p.dv) +
                           (static_cast<size_t>(b * p.Hkv + g) * p.Tk + (key < p.Tk ? key : 0)) * W;
#pragma unroll 1
      for (int c = 0; c < W / 64; ++c) {
        float a0[32], a1[32];
        {
          uint32_t r[32];
          tmem_ld32_sync(tacc + 32u * c, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) a0[e] = n_it > 0 ? __uint_as_float(r[e]) : 0.f;
          tmem_ld32_sync(tacc + static_cast<uint32_t>(W / 2) + 32u * c, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) a1[e] = n_it > 0 ? __uint_as_float(r[e]) : 0.f;
        }
        if (x == 1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            a0[e] *= p.scale;
            a1[e] *= p.scale;
          }
          if (p.rope == 1) {  // pair (i, i + d/2), i = 32c + e
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              float cs, sn;
              rope_cos_sin<false>(key, p.theta.hi[32 * c + e], p.theta.lo[32 * c + e], cs, sn);
              const float u = a0[e], w = a1[e];
              a0[e] = fmaf(u, cs, w * sn);
              a1[e] = fmaf(-u, sn, w * cs);
            }
          } else if (p.rope == 2) {  // pairs (2i, 2i + 1) inside each chunk
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              float cs, sn;
              rope_cos_sin<false>(key, p.theta.hi[16 * c + t], p.theta.lo[16 * c + t], cs, sn);
              float u = a0[2 * t], w = a0[2 * t + 1];
              a0[2 * t] = fmaf(u, cs, w * sn);
              a0[2 * t + 1] = fmaf(-u, sn, w * cs);
              rope_cos_sin<false>(key, p.theta.hi[D / 4 + 16 * c + t],
                                  p.theta.lo[D / 4 + 16 * c + t], cs, sn);
              u = a1[2 * t];
              w = a1[2 * t + 1];
              a1[2 * t] = fmaf(u, cs, w * sn);
              a1[2 * t + 1] = fmaf(-u, sn, w * cs);
            }
          }
        }
        if (key < p.Tk) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            reinterpret_cast<uint4*>(dst + 32 * c)[v4] =
                make_uint4(pack_bf16x2(a0[8 * v4], a0[8 * v4 + 1]),
                           pack_bf16x2(a0[8 * v4 + 2], a0[8 * v4 + 3]),
                           pack_bf16x2(a0[8 * v4 + 4], a0[8 * v4 + 5]),
                           pack_bf16x2(a0[8 * v4 + 6], a0[8 * v4 + 7]));
            reinterpret_cast<uint4*>(dst + W / 2 + 32 * c)[v4] =
                make_uint4(pack_bf16x2(a1[8 * v4], a1[8 * v4 + 1]),
                           pack_bf16x2(a1[8 * v4 + 2], a1[8 * v4 + 3]),
                           pack_bf16x2(a1[8 * v4 + 4], a1[8 * v4 + 5]),
                           pack_bf16x2(a1[8 * v4 + 6], a1[8 * v4 + 7]));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// dQ, persistent: one CTA per SM walks work items (128 queries of one
// query head), longest first (causally the last query tiles), in rounds of
// gridDim.x items with alternating direction.  Per item, per key tile j:
//   S  = Qr Kr_j^T, dP = dO V_j^T   (SS, TMEM columns [0,128) and [128,256))
//   dS = exp(scale*S - lse) o (dP - D)  (thread = query row; warps 0-3 keys 0-63,
//                                        warps 4-7 keys 64-127), bf16 into dP's columns
//   dQ += dS Kr_j                   (TS, B = Kr_j with channels contiguous)
// into one of two accumulators ([256,384) for even items, [384,512) for odd ones),
// so the next item's products start while warps 12-15 drain the finished dQ
// (R^T, scale, store).  K_j and V_j arrive by TMA through rings that run across
// items, three stages for K (read by S and dQ) and two for V (read by dP only), so
// the load into a freed stage has about a tile's products of time to land; S(g+1) is
// issued as soon as the softmax warps have read S(g) (g counts key tiles over all
// items of the CTA), dP(g+1) follows dQ(g).
constexpr int NSK = 3;
constexpr int NSV = 2;
constexpr int kThreadsQ = 512;
constexpr int kWarpEpiQ = 12;       // warps 12-15: dQ epilogue (TMEM lane quadrants 0-3)
constexpr int kRegsSoftmaxQ = 152;  // 2*128*152 + 128*96 + 128*112 = 65536 = 512 * 128
constexpr int kRegsCtlQ = 96;
constexpr int kRegsEpiQ = 112;

// Shared memory of the dQ kernel: Q and dO of the item, NSK K and NSV V stages.
template <int D, int DV>
struct BwdQSmem {
  static constexpr int DATA = (1 + NSK) * BwdCfg<D, DV>::TILE_QK + (1 + NSV) * BwdCfg<D, DV>::TILE_VO;
  static_assert(DATA + 256 <= 227 * 1024, "dQ kernel shared memory");
};

struct QParams {
  const float* lse;   // [B, Hq, Tq]
  const float* dvec;  // [B, Hq, Tq]
  __nv_bfloat16* dq;  // [B, Hq, Tq, D]
  uint32_t* status;
  int B, Hq, Hkv, Tq, Tk, q_off, causal, rope, n_items;
  float scale, sl2;
  RopeTable theta;
};

struct QItem {
  int qt, b, h, n_it;
};

// i-th item of this CTA: rounds of gridDim.x items, alternating direction
__device__ __forceinline__ int q_item_index(int i) {
  const int G = gridDim.x, c = blockIdx.x;
  return i * G + ((i & 1) ? (G - 1 - c) : c);
}

__device__ __forceinline__ QItem q_item(const QParams& p, int u) {
  const int n_qtiles = (p.Tq + BQ - 1) / BQ;
  const int n_kt = (p.Tk + BK - 1) / BK;
  const int per = p.B * p.Hq;
  const int r = u / per, rem = u - r * per;
  QItem it;
  it.qt = p.causal ? n_qtiles - 1 - r : r;
  it.b = rem / p.Hq;
  it.h = rem - it.b * p.Hq;
  // causal: key tiles up to the one holding the position of the tile's last row
  const int last = p.q_off + min(it.qt * BQ + BQ, p.Tq) - 1;
  it.n_it = p.causal ? min(n_kt, last / BK + 1) : n_kt;
  return it;
}

template <int N>
__device__ __forceinline__ void q_regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void q_regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int D, int DV>
__global__ void __launch_bounds__(kThreadsQ, 1)
    bwd_q_tc_kernel(const __grid_constant__ QParams p, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do) {
  using C = BwdCfg<D, DV>;
  constexpr int TQK = C::TILE_QK, TVO = C::TILE_VO;
  constexpr int Q_SMEM_DATA = BwdQSmem<D, DV>::DATA;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sO = smem + TQK;
  uint8_t* sK = sO + TVO;        // [NSK] K tiles
  uint8_t* sV = sK + NSK * TQK;  // [NSV] V tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Q_SMEM_DATA);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;   // the item's last S and dP completed
  uint64_t* k_full = bars + 2;    // [NSK]
  uint64_t* k_empty = bars + 5;   // [NSK]: S and dQ of the stage's tile completed
  uint64_t* v_full = bars + 8;    // [NSV]
  uint64_t* v_empty = bars + 10;  // [NSV]: dP of the stage's tile completed
  uint64_t* s_full = bars + 12;
  uint64_t* s_free = bars + 13;   // 8 warps: S(g) read
  uint64_t* dp_full = bars + 14;
  uint64_t* ds_full = bars + 15;  // 8 warps
  uint64_t* acc_full = bars + 16;   // [2] dQ accumulator complete
  uint64_t* acc_empty = bars + 18;  // [2] 4 epilogue warps have read it
  uint64_t* teardown = bars + 20;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 21);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusDeviceArg);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 8);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 8);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
    }
    mbar_init(teardown, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8 && warp < kWarpEpiQ) {
   q_regs_dec<kRegsCtlQ>();
   if (warp == kWarpProducer) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      bool ok = true;
      int g = 0, k_issued = 0, v_issued = 0, items = 0;
      for (int i = 0; ok; ++i) {
        const int u = q_item_index(i);
        if (u >= p.n_items) break;
        const QItem it = q_item(p, u);
        const int zq = it.b * p.Hq + it.h, zk = it.b * p.Hkv + it.h / (p.Hq / p.Hkv);
        if (i > 0 && !mbar_wait(q_empty, (i - 1) & 1, abort_flag, p.status, kWaitNs)) break;
        mbar_arrive_expect_tx(q_full, TQK + TVO);
        for (int kb = 0; kb < D / 64; ++kb)
          tma_load_3d(sQ + kb * BLOCK, &tm_q, q_full, kb * 64, it.qt * BQ, zq);
        for (int kb = 0; kb < DV / 64; ++kb)
          tma_load_3d(sO + kb * BLOCK, &tm_do, q_full, kb * 64, it.qt * BQ, zq);
        ++items;
        for (int j = 0; j < it.n_it; ++j, ++g) {
          const int sk = g % NSK, uk = g / NSK;
          if (uk > 0 && !mbar_wait(&k_empty[sk], (uk - 1) & 1, abort_flag, p.status, kWaitNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&k_full[sk], TQK);
          for (int kb = 0; kb < D / 64; ++kb)
            tma_load_3d(sK + sk * TQK + kb * BLOCK, &tm_k, &k_full[sk], kb * 64, j * BK, zk);
          ++k_issued;
          const int sv = g % NSV, uv = g / NSV;
          if (uv > 0 && !mbar_wait(&v_empty[sv], (uv - 1) & 1, abort_flag, p.status, kWaitNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[sv], TVO);
          for (int kb = 0; kb < DV / 64; ++kb)
            tma_load_3d(sV + sv * TVO + kb * BLOCK, &tm_v, &v_full[sv], kb * 64, j * BK, zk);
          ++v_issued;
        }
      }
      if (*abort_flag) {
        if (items > 0) mbar_wait(q_full, (items - 1) & 1, nullptr, p.status, kDrainNs);
        for (int t = k_issued > NSK ? k_issued - NSK : 0; t < k_issued; ++t)
          mbar_wait(&k_full[t % NSK], (t / NSK) & 1, nullptr, p.status, kDrainNs);
        for (int t = v_issued > NSV ? v_issued - NSV : 0; t < v_issued; ++t)
          mbar_wait(&v_full[t % NSV], (t / NSV) & 1, nullptr, p.status, kDrainNs);
      }
    }
   } else if (warp == kWarpMma) {
    if (lane == 0) {
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (!ok) return false;
        ok = mbar_wait(bar, parity, abort_flag, p.status, kWaitNs);
        tc_fence_after();
        return ok;
      };
      const uint32_t q_s = smem_u32(sQ), o_s = smem_u32(sO);
      auto k_tile = [&](int g) { return smem_u32(sK + (g % NSK) * TQK); };
      auto v_tile = [&](int g) { return smem_u32(sV + (g % NSV) * TVO); };
      auto issue_s = [&](int g) {  // S = Qr Kr^T
        const uint32_t k_s = k_tile(g);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((kk >> 2) * BLOCK + (kk & 3) * 32);
          umma_ss(tmem, smem_desc_sw128(q_s + off, 16, 1024), smem_desc_sw128(k_s + off, 16, 1024),
                  IDESC_SS, kk > 0 ? 1u : 0u);
        }
        tc_commit(s_full);
      };
      auto issue_dp = [&](int g) {  // dP = dO V^T, then V's stage is released
        const uint32_t v_s = v_tile(g);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((kk >> 2) * BLOCK + (kk & 3) * 32);
          umma_ss(tmem + 128u, smem_desc_sw128(o_s + off, 16, 1024),
                  smem_desc_sw128(v_s + off, 16, 1024), IDESC_SS, kk > 0 ? 1u : 0u);
        }
        tc_commit(dp_full);
        tc_commit(&v_empty[g % NSV]);
      };
      int g = 0;
      for (int i = 0; ok; ++i) {
        const int u = q_item_index(i);
        if (u >= p.n_items) break;
        const QItem it = q_item(p, u);
        const int ab = i & 1;
        const uint32_t t_acc = tmem + 256u + 128u * static_cast<uint32_t>(ab);
        // S(g), dP(g) of the item's first key tile: its Q and dO, the S columns read
        // (s_free of the previous tile), the dP columns consumed (dQ issued before)
        if (!wait(q_full, i & 1)) break;
        if (g > 0 && !wait(s_free, (g - 1) & 1)) break;
        if (!wait(&k_full[g % NSK], (g / NSK) & 1)) break;
        issue_s(g);
        if (!wait(&v_full[g % NSV], (g / NSV) & 1)) break;
        issue_dp(g);
        if (it.n_it == 1) tc_commit(q_empty);
        for (int j = 0; j < it.n_it && ok; ++j, ++g) {
          const bool next = j + 1 < it.n_it;
          if (next) {
            if (!wait(s_free, g & 1)) break;
            if (!wait(&k_full[(g + 1) % NSK], ((g + 1) / NSK) & 1)) break;
            issue_s(g + 1);
          }
          if (!wait(ds_full, g & 1)) break;
          // the accumulator's previous item (i - 2) has been read by the epilogue warps
          if (j == 0 && i >= 2 && !wait(&acc_empty[ab], ((i >> 1) - 1) & 1)) break;
          // dQ += dS Kr: A = dS (TMEM, over dP), B = Kr as (channels x keys)
          const uint32_t k_s = k_tile(g);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_ts(t_acc, tmem + 128u + packed_col(kk), smem_desc_sw128(k_s + 2048u * kk, BLOCK, 1024),
                    C::IDESC_DK, (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&k_empty[g % NSK]);
          if (next) {
            if (!wait(&v_full[(g + 1) % NSV], ((g + 1) / NSV) & 1)) break;
            issue_dp(g + 1);
            if (j + 2 == it.n_it) tc_commit(q_empty);  // S and dP of the last key tile issued
          } else {
            tc_commit(&acc_full[ab]);
          }
        }
      }
      tc_commit(teardown);
      mbar_wait(teardown, 0, nullptr, p.status, kDrainNs);
    }
    __syncwarp();
   }
  } else if (warp < 8) {
    q_regs_inc<kRegsSoftmaxQ>();
    const int x = warp >> 2;              // key half of the tile
    const int row = threadIdx.x & 127;    // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(64 * x);
    const uint32_t tD = tmem + lane_off + 128u + static_cast<uint32_t>(64 * x);
    bool ok = true;
    int g = 0;
    for (int i = 0; ok; ++i) {
      const int u = q_item_index(i);
      if (u >= p.n_items) break;
      const QItem it = q_item(p, u);
      const int q0 = it.qt * BQ, q = q0 + row;
      const size_t rb = static_cast<size_t>(it.b * p.Hq + it.h) * p.Tq;
      const float lse2 = q < p.Tq ? p.lse[rb + q] * kLog2e : 0.f;
      const float dq_d = q < p.Tq ? p.dvec[rb + q] : 0.f;
      for (int j = 0; j < it.n_it; ++j, ++g) {
        if (!warp_wait(s_full, g & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kb0 = j * BK + 64 * x;  // first key of this half
        uint32_t rs[64];
        tmem_ld64_sync(tS, rs);
        // S(g) is in registers: the MMA warp may overwrite it with S(g+1)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
        // P = exp(S - lse) while dP(g) is still being computed
        float pr[64];
        // every (query, key) of this warpgroup's half tile is visible: no per-element test
        const bool all_vis =
            kb0 + 63 < p.Tk && q0 + BQ <= p.Tq && (!p.causal || kb0 + 63 <= p.q_off + q0);
        if (all_vis) {
#pragma unroll
          for (int c = 0; c < 64; ++c) pr[c] = ex2_approx(fmaf(__uint_as_float(rs[c]), p.sl2, -lse2));
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int key = kb0 + c;
            const bool vis = q < p.Tq && key < p.Tk && (!p.causal || key <= p.q_off + q);
            pr[c] = vis ? ex2_approx(fmaf(__uint_as_float(rs[c]), p.sl2, -lse2)) : 0.f;
          }
        }
        if (!warp_wait(dp_full, g & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t pk[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t rd[32];
          tmem_ld32_sync(tD + 32u * hh, rd);
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int c = 2 * t;
            pk[16 * hh + t] = pack_bf16x2(pr[32 * hh + c] * (__uint_as_float(rd[c]) - dq_d),
                                          pr[32 * hh + c + 1] * (__uint_as_float(rd[c + 1]) - dq_d));
          }
        }
        tmem_st32(tD, pk);  // dS over dP (this half's 64 keys, packed into 32 columns)
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full);
      }
    }
  } else {
    // ------------------------------------------------------------ dQ epilogue (warps 12-15)
    // thread = query row; dQ = R^T (scale dQ) with split-half pairs (i, i + d/2) taken
    // as column chunks (32c + e, d/2 + 32c + e)
    q_regs_dec<kRegsEpiQ>();
    const int row = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    for (int i = 0;; ++i) {
      const int u = q_item_index(i);
      if (u >= p.n_items) break;
      const QItem it = q_item(p, u);
      const int ab = i & 1;
      const int q = it.qt * BQ + row;
      const int qpos = p.q_off + q;  // RoPE position of the row
      if (!warp_wait(&acc_full[ab], (i >> 1) & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t t_acc = tmem + lane_off + 256u + 128u * static_cast<uint32_t>(ab);
      __nv_bfloat16* dst = p.dq + (static_cast<size_t>(it.b * p.Hq + it.h) * p.Tq + q) * D;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        float a0[32], a1[32];
        {
          uint32_t r[32];
          tmem_ld32_sync(t_acc + 32u * c, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) a0[e] = __uint_as_float(r[e]) * p.scale;
          tmem_ld32_sync(t_acc + static_cast<uint32_t>(D / 2) + 32u * c, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) a1[e] = __uint_as_float(r[e]) * p.scale;
        }
        if (p.rope == 1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float cs, sn;
            rope_cos_sin<false>(qpos, p.theta.hi[32 * c + e], p.theta.lo[32 * c + e], cs, sn);
            const float u0 = a0[e], w = a1[e];
            a0[e] = fmaf(u0, cs, w * sn);
            a1[e] = fmaf(-u0, sn, w * cs);
          }
        } else if (p.rope == 2) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float cs, sn;
            rope_cos_sin<false>(qpos, p.theta.hi[16 * c + t], p.theta.lo[16 * c + t], cs, sn);
            float u0 = a0[2 * t], w = a0[2 * t + 1];
            a0[2 * t] = fmaf(u0, cs, w * sn);
            a0[2 * t + 1] = fmaf(-u0, sn, w * cs);
            rope_cos_sin<false>(qpos, p.theta.hi[D / 4 + 16 * c + t],
                                p.theta.lo[D / 4 + 16 * c + t], cs, sn);
            u0 = a1[2 * t];
            w = a1[2 * t + 1];
            a1[2 * t] = fmaf(u0, cs, w * sn);
            a1[2 * t + 1] = fmaf(-u0, sn, w * cs);
          }
        }
        if (q < p.Tq) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            reinterpret_cast<uint4*>(dst + 32 * c)[v4] =
                make_uint4(pack_bf16x2(a0[8 * v4], a0[8 * v4 + 1]),
                           pack_bf16x2(a0[8 * v4 + 2], a0[8 * v4 + 3]),
                           pack_bf16x2(a0[8 * v4 + 4], a0[8 * v4 + 5]),
                           pack_bf16x2(a0[8 * v4 + 6], a0[8 * v4 + 7]));
            reinterpret_cast<uint4*>(dst + D / 2 + 32 * c)[v4] =
                make_uint4(pack_bf16x2(a1[8 * v4], a1[8 * v4 + 1]),
                           pack_bf16x2(a1[8 * v4 + 2], a1[8 * v4 + 3]),
                           pack_bf16x2(a1[8 * v4 + 4], a1[8 * v4 + 5]),
                           pack_bf16x2(a1[8 * v4 + 6], a1[8 * v4 + 7]));
          }
        }
      }
      // the accumulator may take the item after next
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D, int DV>
cudaError_t launch_kv_d(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D, DV>;
  KvParams p{};
  p.lse = a.lse;
  p.dvec = a.dvec;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.status = a.status;
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
  alignas(64) CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_bf16_3d(&tq, a.qr, D, a.Tq, a.B * a.Hq, BQ) ||
      !make_tmap_bf16_3d(&tk, a.kr, D, a.Tk, a.B * a.Hkv, BK) ||
      !make_tmap_bf16_3d(&tv, a.v, DV, a.Tk, a.B * a.Hkv, BK) ||
      !make_tmap_bf16_3d(&tdo, a.dout, DV, a.Tq, a.B * a.Hq, BQ))
    return cudaErrorInvalidValue;
  static SmemLimitOnce smem_limit;
  cudaError_t e = smem_limit.set(bwd_kv_tc_kernel<D, DV>, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(a.Hkv, a.B, (a.Tk + BK - 1) / BK);
  bwd_kv_tc_kernel<D, DV><<<grid, kThreads, C::SMEM_BYTES, stream>>>(p, tq, tk, tv, tdo);
  return cudaGetLastError();
}

cudaError_t launch_bwd_kv_tc(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 64 && a.d_v == 64) return launch_kv_d<64, 64>(a, stream);
  if (a.d == 64 && a.d_v == 128) return launch_kv_d<64, 128>(a, stream);
  if (a.d == 128 && a.d_v == 64) return launch_kv_d<128, 64>(a, stream);
  if (a.d == 128 && a.d_v == 128) return launch_kv_d<128, 128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace csattn

namespace csattn {

template <int D, int DV>
cudaError_t launch_q_d(const BwdArgs& a, cudaStream_t stream) {
  constexpr int smem_bytes = BwdQSmem<D, DV>::DATA + 256;
  QParams p{};
  p.lse = a.lse;
  p.dvec = a.dvec;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.status = a.status;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.q_off = a.q_off;
  p.causal = a.causal;
  p.rope = a.rope;
  p.n_items = a.B * a.Hq * ((a.Tq + BQ - 1) / BQ);
  p.scale = a.scale;
  p.sl2 = a.scale * kLog2e;
  p.theta = a.theta;
  alignas(64) CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_bf16_3d(&tq, a.qr, D, a.Tq, a.B * a.Hq, BQ) ||
      !make_tmap_bf16_3d(&tk, a.kr, D, a.Tk, a.B * a.Hkv, BK) ||
      !make_tmap_bf16_3d(&tv, a.v, DV, a.Tk, a.B * a.Hkv, BK) ||
      !make_tmap_bf16_3d(&tdo, a.dout, DV, a.Tq, a.B * a.Hq, BQ))
    return cudaErrorInvalidValue;
  static SmemLimitOnce smem_limit;
  cudaError_t e = smem_limit.set(bwd_q_tc_kernel<D, DV>, smem_bytes);
  if (e != cudaSuccess) return e;
  const int sms = a.num_sms > 0 ? a.num_sms : 1;
  const int grid = p.n_items < sms ? p.n_items : sms;
  bwd_q_tc_kernel<D, DV><<<grid, kThreadsQ, smem_bytes, stream>>>(p, tq, tk, tv, tdo);
  return cudaGetLastError();
}

cudaError_t launch_bwd_q_tc(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 64 && a.d_v == 64) return launch_q_d<64, 64>(a, stream);
  if (a.d == 64 && a.d_v == 128) return launch_q_d<64, 128>(a, stream);
  if (a.d == 128 && a.d_v == 64) return launch_q_d<128, 64>(a, stream);
  if (a.d == 128 && a.d_v == 128) return launch_q_d<128, 128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace csattn
