// KV-cache decode, bf16, one new query per sequence: split-KV partials plus a
// log-sum-exp merge.  The query of sequence b sits at position L_b - 1 and
// attends to cached rows 0..L_b-1 ("The Transformer architecture"
// (cooking-agi), section "Hands-on": with a cache the query position is
// cache.pos and the keys run from 0 to cache.pos).  The whole cost is reading
// K and V once: 2 * n_kv * d_head * L * sizeof(bf16) bytes per sequence, the
// pages' KV-cache formula with one layer (same page, section "What else the
// modern decoder-only model changed").  Keys have d channels and values dv
// (each 64 or 128; "Scaled dot-product attention" lets the widths differ).
//
// Grid (split, kv_head, batch).  One CTA reads a chunk of one sequence's K/V
// rows once for all the query heads of the KV head's group:
//   warp 4      TMA producer: 64-row K and V tiles into a 3-stage ring
//   warps 0-3   16 keys each per tile:  S = Q K^T and O += P V on the tensor
//               cores (mma.sync m16n8k16; rows = the group's query heads,
//               padded to 16), online softmax in fp32 between the two.
// The per-CTA result (running max m, sum l, un-normalised O, log2 units) is
// written to the workspace; decode_combine_kernel merges the splits:
//   m = max_s m_s,  l = sum_s l_s 2^(m_s - m),  o = sum_s o_s 2^(m_s - m) / l.
// Cache rows at or beyond L_b are never used: scores of those keys are set to
// -inf and the V rows of the final tile are zeroed in shared memory before
// the second MMA (the cache past L_b may hold anything, NaN included).
#include "internal.h"

namespace csattn {
namespace {

constexpr int KT = 64;  // keys per tile
constexpr int NS = 3;   // ring stages
constexpr int kComputeWarps = 4;
constexpr int kThreads = 32 * (kComputeWarps + 1);
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 100000000ull;
constexpr float kRescaleThreshold = 8.0f;

template <int D, int DV>
struct DCfg {
  static constexpr int KBK = D / 64;                // 64-column blocks of a K tile
  static constexpr int KBV = DV / 64;               // ... of a V tile
  static constexpr int BLOCK_BYTES = KT * 128;      // one 64-column block of a 64-row tile
  static constexpr int K_BYTES = KT * D * 2;        // K tile
  static constexpr int V_BYTES = KT * DV * 2;       // V tile
  static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;
  static constexpr int SMEM_BYTES = NS * STAGE_BYTES + 1024 + 1024;
  static_assert(4 * 16 * DV * 4 <= NS * STAGE_BYTES, "per-warp results fit in the ring");
};

struct DParams {
  const __nv_bfloat16* q;
  const int32_t* seq_lens;
  int len_add;
  const int32_t* block_table;  // paged cache, or nullptr
  int page_size, num_pages, max_pages;
  int box_rows;                // paged: rows per TMA box (min(64, page_size))
  float* part_o;
  float* part_ml;
  uint32_t* status;
  int B, Hq, Hkv, Lmax, rep, max_seq_len, chunk, n_splits;
  float scale_log2;
};

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

// shared-memory byte offset of 16-byte chunk `cc` (8 channels) of row r of a
// 64-row tile stored as 128-byte-swizzled column blocks (TMA SWIZZLE_128B)
__device__ __forceinline__ uint32_t tile_off(int r, int cc) {
  return static_cast<uint32_t>((cc >> 3) * (KT * 128) + r * 128 + (((cc & 7) ^ (r & 7)) << 4));
}

template <int D, int DV>
__global__ void __launch_bounds__(kThreads)
    decode_bf16_kernel(const __grid_constant__ DParams p, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v) {
  using C = DCfg<D, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * C::STAGE_BYTES);
  uint64_t* empty = full + NS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NS);
  float* s_ml = reinterpret_cast<float*>(smem + NS * C::STAGE_BYTES + 256);  // [4 warps][16][2]

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int raw = p.seq_lens[b];  // (no overflow in raw + len_add past max_seq_len)
  int L = raw > p.max_seq_len ? p.max_seq_len + 1 : raw + p.len_add;
  if (L < 1 || L > p.max_seq_len) {
    if (threadIdx.x == 0 && split == 0 && kvh == 0) atomicOr(p.status, kStatusDeviceArg);
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
  }
  // let the merge kernel (launched with programmatic dependent launch) be
  // scheduled as soon as every CTA of this grid has started; it still waits
  // for this grid to finish before it reads the partials
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int k_begin = split * p.chunk;
  const int k_end = min(L, k_begin + p.chunk);
  if (k_begin >= k_end) return;  // the merge reads only splits that hold keys
  const int ntiles = (k_end - k_begin + KT - 1) / KT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kComputeWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // ------------------------------------------------------------ producer
    if (p.block_table != nullptr && p.box_rows < KT) {
      // pages of 16 or 32 rows: 4 or 2 boxes per tile, one per lane, so that their
      // table reads and copies are issued side by side; lane 0 waits and arms the
      // stage's barrier before the other lanes' copies (ordered by __syncwarp)
      if (lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      const int nbox = KT / p.box_rows;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % NS, use = t / NS;
        int okw = 1;
        if (lane == 0) {
          if (use > 0 && !ctl_wait(&empty[s], (use - 1) & 1, abort_flag, p.status, kWaitNs))
            okw = 0;
          else
            mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        }
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) break;
        __syncwarp();
        if (lane < nbox) {
          uint8_t* kdst = smem + s * C::STAGE_BYTES;
          uint8_t* vdst = kdst + C::K_BYTES;
          const int r0 = lane * p.box_rows, tr = k_begin + t * KT + r0;
          int plane = p.num_pages * p.Hkv, prow = 0;
          if (tr < L) {
            const int page =
                p.block_table[static_cast<size_t>(b) * p.max_pages + tr / p.page_size];
            if (page >= 0 && page < p.num_pages)
              plane = page * p.Hkv + kvh;
            else
              atomicOr(p.status, kStatusDeviceArg);
            prow = tr % p.page_size;
          }
          for (int kb = 0; kb < C::KBK; ++kb)
            tma_load_3d(kdst + kb * C::BLOCK_BYTES + r0 * 128, &tm_k, &full[s], kb * 64, prow,
                        plane);
          for (int kb = 0; kb < C::KBV; ++kb)
            tma_load_3d(vdst + kb * C::BLOCK_BYTES + r0 * 128, &tm_v, &full[s], kb * 64, prow,
                        plane);
        }
        __syncwarp();
        ++issued;
      }
      if (lane == 0 && *abort_flag) {
        const int first = issued > NS ? issued - NS : 0;
        for (int t = first; t < issued; ++t)
          mbar_wait(&full[t % NS], (t / NS) & 1, nullptr, p.status, kDrainNs);
      }
      return;
    }
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int z = b * p.Hkv + kvh;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % NS, use = t / NS;
        if (use > 0 && !ctl_wait(&empty[s], (use - 1) & 1, abort_flag, p.status, kWaitNs)) break;
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        uint8_t* kdst = smem + s * C::STAGE_BYTES;
        uint8_t* vdst = kdst + C::K_BYTES;
        const int row = k_begin + t * KT;
        if (p.block_table == nullptr) {
          for (int kb = 0; kb < C::KBK; ++kb)
            tma_load_3d(kdst + kb * C::BLOCK_BYTES, &tm_k, &full[s], kb * 64, row, z);
          for (int kb = 0; kb < C::KBV; ++kb)
            tma_load_3d(vdst + kb * C::BLOCK_BYTES, &tm_v, &full[s], kb * 64, row, z);
        } else {
          // paged: boxes of box_rows rows (64, or the page size when it is 16 or 32)
          // never cross a page; a box past the sequence, or a page index outside the
          // pool (reported), reads zeros (its plane coordinate is past the tensor map)
          for (int r0 = 0; r0 < KT; r0 += p.box_rows) {
            const int tr = row + r0;
            int plane = p.num_pages * p.Hkv, prow = 0;
            if (tr < L) {
              const int page =
                  p.block_table[static_cast<size_t>(b) * p.max_pages + tr / p.page_size];
              if (page >= 0 && page < p.num_pages)
                plane = page * p.Hkv + kvh;
              else
                atomicOr(p.status, kStatusDeviceArg);
              prow = tr % p.page_size;
            }
            for (int kb = 0; kb < C::KBK; ++kb)
              tma_load_3d(kdst + kb * C::BLOCK_BYTES + r0 * 128, &tm_k, &full[s], kb * 64, prow,
                          plane);
            for (int kb = 0; kb < C::KBV; ++kb)
              tma_load_3d(vdst + kb * C::BLOCK_BYTES + r0 * 128, &tm_v, &full[s], kb * 64, prow,
                          plane);
          }
        }
        ++issued;
      }
      if (*abort_flag) {
        const int first = issued > NS ? issued - NS : 0;
        for (int t = first; t < issued; ++t)
          mbar_wait(&full[t % NS], (t / NS) & 1, nullptr, p.status, kDrainNs);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- compute warps
  const int r0 = lane >> 2;        // fragment rows r0 and r0 + 8 = query heads of the group
  const int cq = 2 * (lane & 3);   // fragment column pair
  const __nv_bfloat16* qg = p.q + (static_cast<size_t>(b) * p.Hq + kvh * p.rep) * D;
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(qg + static_cast<size_t>(r0) * D);
    const uint32_t* q8 = reinterpret_cast<const uint32_t*>(qg + static_cast<size_t>(r0 + 8) * D);
    qa[kk][0] = (r0 < p.rep) ? q0[(16 * kk + cq) >> 1] : 0u;
    qa[kk][1] = (r0 + 8 < p.rep) ? q8[(16 * kk + cq) >> 1] : 0u;
    qa[kk][2] = (r0 < p.rep) ? q0[(16 * kk + 8 + cq) >> 1] : 0u;
    qa[kk][3] = (r0 + 8 < p.rep) ? q8[(16 * kk + 8 + cq) >> 1] : 0u;
  }

  float o[DV / 8][4];
#pragma unroll
  for (int n = 0; n < DV / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_used[2] = {-INFINITY, -INFINITY};  // rows r0, r0 + 8
  float l_part[2] = {0.f, 0.f};
  const float sl2 = p.scale_log2;
  const uint32_t smem_base = smem_u32(smem);

  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % NS;
    if (!mbar_wait(&full[s], (t / NS) & 1, abort_flag, p.status, kWaitNs)) {
      ok = false;
      break;
    }
    const uint32_t kbase = smem_base + s * C::STAGE_BYTES;
    const uint32_t vbase = kbase + C::K_BYTES;
    const int key0 = k_begin + t * KT + 16 * warp;  // first key of this warp's slice
    const int nvalid = k_end - key0;                // keys of the slice that exist (may be <= 0)

    // S = Q K^T for 16 keys (two n-tiles of 8)
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3;  // which 8x8 matrix this lane addresses
      const int kr = 16 * warp + (lane & 7) + 8 * (mi >> 1);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + tile_off(kr, 2 * kk + (mi & 1)), b0, b1, b2, b3);
        mma_bf16(sc[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma_bf16(sc[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
      }
    }
    // mask keys past the end of the split, scale to log2 units, row max
    float x[2][4];
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = 8 * nt + cq + (e & 1);
        const float v = (key < nvalid) ? sc[nt][e] * sl2 : -INFINITY;
        x[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
    }
    float f[2] = {1.f, 1.f};
    bool need = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float m_new = fmaxf(m_used[h], mx[h]);
      if (m_new > m_used[h] + kRescaleThreshold) {
        f[h] = ex2_approx(m_used[h] - m_new);  // 0 when m_used was -inf
        m_used[h] = m_new;
        need = true;
      }
    }
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int n = 0; n < DV / 8; ++n) {
        o[n][0] *= f[0];
        o[n][1] *= f[0];
        o[n][2] *= f[1];
        o[n][3] *= f[1];
      }
      l_part[0] *= f[0];
      l_part[1] *= f[1];
    }
    float pr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mu = m_used[e >> 1];
        const float v = (mu == -INFINITY) ? 0.f : ex2_approx(x[nt][e] - mu);
        pr[nt][e] = v;
        l_part[e >> 1] += v;
      }
    const uint32_t pa0 = pack_bf16x2(pr[0][0], pr[0][1]);
    const uint32_t pa1 = pack_bf16x2(pr[0][2], pr[0][3]);
    const uint32_t pa2 = pack_bf16x2(pr[1][0], pr[1][1]);
    const uint32_t pa3 = pack_bf16x2(pr[1][2], pr[1][3]);

    // V rows past the end of the sequence may hold anything: zero them
    const bool zeroed = nvalid < 16;
    if (zeroed) {
      uint8_t* vtile = smem + s * C::STAGE_BYTES + C::K_BYTES;
      const int first = nvalid < 0 ? 0 : nvalid;
      for (int e = lane; e < 16 * (DV / 8); e += 32) {
        const int rr = e / (DV / 8), cc = e % (DV / 8);
        if (rr >= first)
          *reinterpret_cast<uint4*>(vtile + tile_off(16 * warp + rr, cc)) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    // O += P V for 16 keys: 8-channel n-tiles in pairs
    {
      const int mi = lane >> 3;
      const int vr = 16 * warp + (lane & 7) + 8 * (mi & 1);
#pragma unroll
      for (int np = 0; np < DV / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + tile_off(vr, 2 * np + (mi >> 1)), b0, b1, b2, b3);
        mma_bf16(o[2 * np], pa0, pa1, pa2, pa3, b0, b1);
        mma_bf16(o[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
    }
    if (zeroed) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // sum l over the four lanes of a row
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_part[h] += __shfl_xor_sync(0xffffffffu, l_part[h], 1);
    l_part[h] += __shfl_xor_sync(0xffffffffu, l_part[h], 2);
  }
  // all tiles consumed: the ring is free to hold the per-warp results
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kComputeWarps) : "memory");
  if (!ok || *abort_flag) return;
  float* s_o = reinterpret_cast<float*>(smem);  // [4 warps][16 rows][DV]
  if ((lane & 3) == 0) {
    s_ml[(warp * 16 + r0) * 2 + 0] = m_used[0];
    s_ml[(warp * 16 + r0) * 2 + 1] = l_part[0];
    s_ml[(warp * 16 + r0 + 8) * 2 + 0] = m_used[1];
    s_ml[(warp * 16 + r0 + 8) * 2 + 1] = l_part[1];
  }
#pragma unroll
  for (int n = 0; n < DV / 8; ++n) {
    const int c = 8 * n + cq;
    s_o[(warp * 16 + r0) * DV + c] = o[n][0];
    s_o[(warp * 16 + r0) * DV + c + 1] = o[n][1];
    s_o[(warp * 16 + r0 + 8) * DV + c] = o[n][2];
    s_o[(warp * 16 + r0 + 8) * DV + c + 1] = o[n][3];
  }
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kComputeWarps) : "memory");
  // merge the four warps; write this split's partial for each head of the group
  for (int e = threadIdx.x; e < p.rep * DV; e += 32 * kComputeWarps) {
    const int r = e / DV, c = e % DV;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) m = fmaxf(m, s_ml[(w * 16 + r) * 2]);
    float acc = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) {
      const float mw = s_ml[(w * 16 + r) * 2];
      const float fw = (mw == -INFINITY) ? 0.f : ex2_approx(mw - m);
      acc += fw * s_o[(w * 16 + r) * DV + c];
      l += fw * s_ml[(w * 16 + r) * 2 + 1];
    }
    const size_t row = (static_cast<size_t>(b) * p.Hq + kvh * p.rep + r) * p.n_splits + split;
    p.part_o[row * DV + c] = acc;
    if (c == 0) {
      p.part_ml[row * 2 + 0] = m;
      p.part_ml[row * 2 + 1] = l;
    }
  }
}

// out[b, h, :] = merge of the splits that hold keys of sequence b (D = the value width).
__global__ void decode_combine_kernel(const float* __restrict__ part_o,
                                      const float* __restrict__ part_ml,
                                      const int32_t* __restrict__ seq_lens, int len_add,
                                      __nv_bfloat16* __restrict__ out, int Hq, int n_splits,
                                      int chunk, int max_seq_len, int D) {
  // wait until the split kernel has finished and its partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
        const float f = (ms == -INFINITY) ? 0.f : ex2_approx(ms - m);
        acc += f * po[static_cast<size_t>(s) * D + c];
        l += f * ml[2 * s + 1];
      }
    }
    out[static_cast<size_t>(bh) * D + c] = __float2bfloat16_rn(l > 0.f ? acc / l : 0.f);
  }
}

template <int D, int DV>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t stream) {
  using C = DCfg<D, DV>;
  DParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.seq_lens = a.seq_lens;
  p.len_add = a.len_add;
  p.block_table = a.block_table;
  p.page_size = a.page_size;
  p.num_pages = a.num_pages;
  p.max_pages = a.max_pages;
  p.box_rows = a.page_size > 0 && a.page_size < KT ? a.page_size : KT;
  p.part_o = a.part_o;
  p.part_ml = a.part_ml;
  p.status = a.status;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Lmax = a.Lmax;
  p.rep = a.Hq / a.Hkv;
  p.max_seq_len = a.max_seq_len;
  p.chunk = a.chunk;
  p.n_splits = a.n_splits;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);

  alignas(64) CUtensorMap tk, tv;
  const int rows = a.block_table != nullptr ? a.page_size : a.Lmax;
  const int planes = a.block_table != nullptr ? a.num_pages * a.Hkv : a.B * a.Hkv;
  const int box = a.block_table != nullptr ? p.box_rows : KT;
  if (!make_tmap_bf16_3d(&tk, a.k_cache, D, rows, planes, box) ||
      !make_tmap_bf16_3d(&tv, a.v_cache, DV, rows, planes, box))
    return cudaErrorInvalidValue;
  static SmemLimitOnce smem_limit;
  cudaError_t e = smem_limit.set(decode_bf16_kernel<D, DV>, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_splits, a.Hkv, a.B);
  decode_bf16_kernel<D, DV><<<grid, kThreads, C::SMEM_BYTES, stream>>>(p, tk, tv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.Hq, 1, 1);
  cfg.blockDim = dim3(DV, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel, static_cast<const float*>(a.part_o),
                            static_cast<const float*>(a.part_ml), a.seq_lens, a.len_add,
                            static_cast<__nv_bfloat16*>(a.out), a.Hq, a.n_splits, a.chunk,
                            a.max_seq_len, DV);
}

}  // namespace

cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t stream) {
  const int dv = a.dv > 0 ? a.dv : a.d;
  if (a.d == 64 && dv == 64) return launch_d<64, 64>(a, stream);
  if (a.d == 64 && dv == 128) return launch_d<64, 128>(a, stream);
  if (a.d == 128 && dv == 64) return launch_d<128, 64>(a, stream);
  if (a.d == 128 && dv == 128) return launch_d<128, 128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace csattn
